"""CPU checks of the GPU parity helper (tests/parity.py): a selection that reproduces the
oracle's passes, and each kind of mistake the helper exists to catch is rejected -- a
changed CSR row of a VS head, pooled scores off by more than the stated bound, a PE pair
dropped far from the cut, a PE row without its diagonal."""
import numpy as np
import pytest

from tests import parity as P
from workloads import get
from workloads.planted import generate


@pytest.fixture(scope="module")
def tiny():
    w = get("tiny_n4k")
    g = generate(w)
    return w, g, P.oracle_select(w, g, threads=2)


def _fake_gpu_selection(w, osel):
    nb = w.n_blocks
    sel = dict(route_vs=np.zeros(w.hq, np.uint8), c_struct=np.zeros(w.hq, np.float32),
               p_v=np.zeros((w.hq, nb), np.float32), p_s=np.zeros((w.hq, nb), np.float32),
               sel_v=np.zeros((w.hq, nb), np.uint8), sel_s=np.zeros((w.hq, nb), np.uint8))
    for h, o in osel.items():
        sel["route_vs"][h] = o["route_vs"]
        sel["c_struct"][h] = o["c_struct"]
        if o["route_vs"]:
            sel["p_v"][h], sel["p_s"][h] = o["p_v"], o["p_s"]
            sel["sel_v"][h, o["S_v"]] = 1
            sel["sel_s"][h, o["S_s"]] = 1
    sel["row_ptr"], sel["col"] = P.csr_from_masks([osel[h]["mask"] for h in range(w.hq)], nb)
    return sel


def _with_mask(w, osel, h, mask):
    masks = [osel[x]["mask"] if x != h else mask for x in range(w.hq)]
    return P.csr_from_masks(masks, w.n_blocks)


def test_helper_accepts_the_oracle_selection(tiny):
    w, g, osel = tiny
    rep = P.compare_selection(w, _fake_gpu_selection(w, osel), osel, g=g)
    assert rep["vs_heads"] == 1 and rep["pe_heads"] == 1 and rep["mask_differs"] == []
    assert rep["rows_checked"] == 2 * w.n_blocks


def test_helper_rejects_a_changed_vs_row(tiny):
    w, g, osel = tiny
    sel = _fake_gpu_selection(w, osel)
    m = osel[0]["mask"].copy()
    I = w.n_blocks - 1
    K = int(np.nonzero(m[I, 1:I])[0][0]) + 1      # a selected block that is neither 0 nor I
    m[I, K] = False
    sel["row_ptr"], sel["col"] = _with_mask(w, osel, 0, m)
    with pytest.raises(AssertionError, match="VS CSR rows"):
        P.compare_selection(w, sel, osel, g=g)


def test_helper_rejects_pooled_score_error(tiny):
    w, g, osel = tiny
    sel = _fake_gpu_selection(w, osel)
    sel["p_v"][0] *= np.float32(1 + 5 * P.MAX_P_REL)
    with pytest.raises(AssertionError, match="pooled score error"):
        P.compare_selection(w, sel, osel, g=g)


def test_helper_rejects_pe_pair_far_from_cut(tiny):
    w, g, osel = tiny
    sel = _fake_gpu_selection(w, osel)
    o = osel[1]
    m = o["mask"].copy()
    v = np.where(np.tril(m, -1), o["v"], 0)
    I, K = np.unravel_index(int(np.argmax(v)), v.shape)   # the largest selected off-diagonal v
    assert I != K and v[I, K] > 2 * o["v_star"]
    m[I, K] = False
    sel["row_ptr"], sel["col"] = _with_mask(w, osel, 1, m)
    with pytest.raises(AssertionError, match="PE pair"):
        P.compare_selection(w, sel, osel, g=g)


def test_helper_rejects_pe_row_without_diagonal(tiny):
    w, g, osel = tiny
    o = osel[1]
    rescued = o["rescued_rows"]
    assert rescued.size                    # the last row of the diffuse head is rescued
    m = o["mask"].copy()
    m[rescued[-1], rescued[-1]] = False
    m[rescued[-1], 0] = True               # keep the row non-empty
    sel = _fake_gpu_selection(w, osel)
    sel["row_ptr"], sel["col"] = _with_mask(w, osel, 1, m)
    with pytest.raises(AssertionError):
        P.compare_selection(w, sel, osel, g=g)


def test_near_threshold_counts_grow_with_the_band(tiny):
    """The oracle-side band counts (the reference for crisp_stats' near_* fields) are
    monotone in the band width and count the diffuse head's ties around its cut value."""
    w, g, osel = tiny
    a = P.near_threshold_counts(w, osel, 1e-4)
    b = P.near_threshold_counts(w, osel)
    c = P.near_threshold_counts(w, osel, 1e-1)
    for k in a:
        assert 0 <= a[k] <= b[k] <= c[k]
    assert c["near_pe_pairs"] > b["near_pe_pairs"] > 0

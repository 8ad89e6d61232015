"""CPU checks of the GPU parity helper (tests/parity.py).

A selection that reproduces the oracle's passes, and each kind of mistake the helper
exists to catch is rejected:
- VS heads: a changed CSR row; a block dropped from the block set far from the floor, with
  the CSR rows following it; pooled scores off by more than the stated bound;
- routing: a route flipped far from tau; a C_struct error;
- PE heads: a pair dropped far from the cut; a pair added below it; a row without its
  diagonal;
- outputs: errors beyond the output tolerances.
"""
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


def test_helper_rejects_a_route_flipped_far_from_tau(tiny):
    w, g, osel = tiny
    assert abs(osel[0]["c_struct"] - w.tau_proxy) > 10 * P.TOL_REL * w.tau_proxy
    sel = _fake_gpu_selection(w, osel)
    sel["route_vs"][0] = 0
    with pytest.raises(AssertionError, match="route differs"):
        P.compare_selection(w, sel, osel, g=g)


def test_helper_rejects_c_struct_error(tiny):
    w, g, osel = tiny
    sel = _fake_gpu_selection(w, osel)
    sel["c_struct"][1] += np.float32(1e-3)
    with pytest.raises(AssertionError, match="C_struct"):
        P.compare_selection(w, sel, osel, g=g)


def test_helper_rejects_a_vs_block_dropped_far_from_the_floor(tiny):
    """The GPU's own block set loses a block scored far above alpha * mu, and its CSR rows
    follow that set (so the union rule holds): the block-set comparison must catch it."""
    w, g, osel = tiny
    o = osel[0]
    thr = w.alpha * o["mu_v"]
    kth = P._kth_largest(o["p_v"], o["k_v"])      # the padding's reference score
    far = [J for J in o["S_v"] if o["p_v"][J] > 2 * thr and J not in (0, w.n_blocks - 1)
           and abs(o["p_v"][J] - kth) > 10 * P.TOL_REL * kth]
    assert far
    sel = _fake_gpu_selection(w, osel)
    sel["sel_v"][0, far[0]] = 0
    m = P.O.vs_block_mask(np.nonzero(sel["sel_v"][0])[0], np.nonzero(sel["sel_s"][0])[0],
                          w.n_blocks)
    sel["row_ptr"], sel["col"] = _with_mask(w, osel, 0, m)
    with pytest.raises(AssertionError, match="differs"):
        P.compare_selection(w, sel, osel, g=g)


def test_helper_rejects_an_extra_pe_pair_below_the_cut(tiny):
    w, g, osel = tiny
    o = osel[1]
    m = o["mask"].copy()
    v = np.where(np.tril(~m), o["v"], np.inf)
    I, K = np.unravel_index(int(np.argmin(v)), v.shape)   # the smallest unselected v
    assert abs(v[I, K] - o["v_star"]) > 10 * P.TOL_REL * o["v_star"]
    m[I, K] = True
    sel = _fake_gpu_selection(w, osel)
    sel["row_ptr"], sel["col"] = _with_mask(w, osel, 1, m)
    with pytest.raises(AssertionError, match="PE pair"):
        P.compare_selection(w, sel, osel, g=g)


def test_output_tolerances():
    """compare_outputs holds max abs 2e-2, mean abs 2e-3 and relative RMS 1e-2."""
    ref = np.random.default_rng(3).standard_normal((256, 128)) / np.sqrt(128)
    P.compare_outputs(ref + 5e-4, ref, "small uniform error passes")
    one = ref.copy()
    one[7, 9] += 3e-2
    with pytest.raises(AssertionError, match="max abs"):
        P.compare_outputs(one, ref, "one large error")
    with pytest.raises(AssertionError):
        P.compare_outputs(ref + 3e-3, ref, "mean error")
    with pytest.raises(AssertionError):
        P.compare_outputs(ref * 1.05, ref, "relative error")

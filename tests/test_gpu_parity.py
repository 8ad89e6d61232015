"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Every workload is seeded and synthetic (workloads/).  Selections (routes, VS block sets,
PE pair sets, CSR rows) must be bit-exact up to counted near-threshold items; outputs on
the oracle's own index set must be within max abs 2e-2 / mean abs 2e-3 (tests/parity.py).
"""
import numpy as np
import pytest

from tests.parity import (REPORTS, TOL_REL, compare_outputs, compare_selection,
                          csr_from_masks, gpu_masks, near_threshold_counts, oracle_outputs,
                          oracle_select, to_device)
from workloads import get
from workloads.configs import Workload
from workloads.planted import generate, random_qkv

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dsp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dynamic_sparse_prefill_gb300 as d
    return d


def _cfg(dsp, w, flags=0):
    if w.vs_floor == "median":
        flags |= dsp.FLAG_MEDIAN_FLOOR
    if w.vs_rule == "gamma":
        flags |= dsp.FLAG_VS_GAMMA_CUMSUM
    return dsp.default_cfg(alpha=w.alpha, gamma=w.gamma, tau_proxy=w.tau_proxy,
                           k_min_tokens=w.k_min_tokens, w_sink=w.w_sink, w_local=w.w_local,
                           flags=flags)


def _rows(blocks, B=128):
    return np.concatenate([np.arange(I * B, (I + 1) * B) for I in blocks])


def run_parity(dsp, w, g, sample=None, seed=0, flags=0, report=None):
    """Full selection parity, then output parity on the oracle's index set.

    sample: None for every query block of every head, else (n_heads, n_blocks) drawn
    with `seed`.
    """
    nb = w.n_blocks
    q, k, v = to_device(g["q"]), to_device(g["k"]), to_device(g["v"])
    dims = dsp.make_dims(1, w.n, w.hq, w.hkv)
    ctx = dsp.Context(dims)
    cfg = _cfg(dsp, w, flags=flags)
    o = torch.empty_like(q)
    ctx.prefill(dims, q, k, v, cfg, o)
    assert ctx.sync_status() == 0
    sel = ctx.selection_get(dims)
    force = None
    if flags & dsp.FLAG_FORCE_VS:
        force = "vs"
    if flags & dsp.FLAG_FORCE_PE:
        force = "pe"
    osel = oracle_select(w, g) if force is None else _oracle_forced(w, g, force)
    rep = compare_selection(w, sel, osel, g=g)
    # near-threshold counts made on the device against the oracle's, the band edges widened
    # by 3% for the scores' own rounding differences
    dev = ctx.stats(dims)
    rep.update({k: dev[k] for k in ("near_routes", "near_vs_blocks", "near_pe_pairs")})
    # (alpha = 0 puts the VS threshold at 0, and gamma = 1 leaves it to rounding whether the
    # PE scores reach gamma at all: both are left out)
    if w.alpha > 0 and w.gamma < 1 and rep["route_mismatch_exempt"] == 0:
        lo = near_threshold_counts(w, osel, TOL_REL * 0.97)
        hi = near_threshold_counts(w, osel, TOL_REL * 1.03)
        for key in lo:
            assert lo[key] <= dev[key] <= hi[key], (key, dev[key], lo[key], hi[key])

    if sample is None:
        blocks = {h: list(range(nb)) for h in range(w.hq)}
    else:
        rng = np.random.default_rng(seed)
        hs = rng.choice(w.hq, size=min(sample[0], w.hq), replace=False)
        blocks = {int(h): sorted(set(rng.choice(nb, size=min(sample[1], nb), replace=False).tolist())
                                 | {nb - 1}) for h in hs}
    ref = oracle_outputs(w, g, osel, blocks)

    # (1) the CUDA attention on the oracle's index set
    rp, col = csr_from_masks([osel[h]["mask"] for h in range(w.hq)], nb)
    ctx.selection_set(dims, rp, col)
    o2 = torch.empty_like(q)
    ctx.attend(dims, q, k, v, o2)
    assert ctx.sync_status() == 0
    got = o2.float().cpu().numpy()
    worst = [0.0, 0.0, 0.0]
    for h, bl in blocks.items():
        r = compare_outputs(got[h][_rows(bl)], ref[h], f"attend on oracle S, head {h}")
        worst = [max(a, b) for a, b in zip(worst, r)]
    rep["attend_max_abs"], rep["attend_mean_abs"], rep["attend_rel_rms"] = worst

    # (2) crisp_prefill's own output for every sampled head: against the rows above where
    # the GPU selection equals the oracle's, else against the oracle's attention on the
    # GPU's own selection (which compare_selection has validated item by item)
    got_p = o.float().cpu().numpy()
    gmask = gpu_masks(sel, w.hq, nb)
    differ = {h: bl for h, bl in blocks.items() if h in rep["mask_differs"]}
    ref_g = oracle_outputs(w, g, {h: {"mask": gmask[h]} for h in differ}, differ) if differ else {}
    for h, bl in blocks.items():
        if h not in differ:
            assert np.array_equal(gmask[h], np.tril(osel[h]["mask"])), h
        compare_outputs(got_p[h][_rows(bl)], ref_g[h] if h in differ else ref[h],
                        f"prefill, head {h}")
    rep["prefill_heads_compared"] = len(blocks)
    rep["prefill_heads_on_gpu_selection"] = len(differ)
    ctx.close()
    REPORTS.append((f"{w.name} n={w.n} hq={w.hq} alpha={w.alpha} flags={flags:#x}", dict(rep)))
    if report is not None:
        report.update(rep)
    return rep, sel, osel


def _oracle_forced(w, g, force):
    from oracle import crisp_oracle as O
    params = O.workload_params(w)
    out = {}
    for h in range(w.hq):
        qh = O.bf16_bits_to_f64(g["q"][h])
        kh = O.bf16_bits_to_f64(g["k"][h // w.group])
        out[h] = O.crisp_select_head(qh, kh, force=force, **params)
    return out


def test_tiny_full(dsp):
    w = get("tiny_n4k")
    rep, sel, osel = run_parity(dsp, w, generate(w))
    assert sel["route_vs"].tolist() == [1, 0]
    print("tiny_n4k", rep)


@pytest.mark.parametrize("n,hq,hkv,seed", [(128, 2, 1, 1), (256, 2, 2, 2), (384, 4, 2, 3),
                                          (1152, 3, 1, 4), (2176, 2, 1, 5)])
def test_edge_shapes_random(dsp, n, hq, hkv, seed):
    """Ragged small shapes (N_b = 1, 2, 3, 9, 17) on unplanted inputs, both routes forced."""
    g = random_qkv(n, hq, hkv, 128, seed, scale=3.0)
    w = Workload("edge", n=n, hq=hq, hkv=hkv, seed=seed)
    for flags in (dsp.FLAG_FORCE_VS, dsp.FLAG_FORCE_PE, 0):
        run_parity(dsp, w, g, flags=flags)


@pytest.mark.parametrize("n,hq,hkv,seed", [(512, 2, 1, 6), (16896, 2, 1, 7)])
def test_edge_shapes_clipped_prob_stores(dsp, n, hq, hkv, seed):
    """N_b = 4 and 132 (N_b % 4 == 0, so the PE probabilities leave through TMA stores whose
    boxes run past the last row and key: the copy must clip them), both routes forced;
    full selection parity, outputs on sampled query blocks."""
    g = random_qkv(n, hq, hkv, 128, seed, scale=3.0)
    w = Workload("edge_tma", n=n, hq=hq, hkv=hkv, seed=seed)
    for flags in (dsp.FLAG_FORCE_PE, 0):
        run_parity(dsp, w, g, sample=(hq, 6), seed=seed, flags=flags)


def test_prefill_graph_replay_matches_eager(dsp):
    """CRISP_FLAG_GRAPH_REPLAY: the captured graph reproduces the eager crisp_prefill bit for
    bit (output and selection), repeated calls replay it, and a new output pointer or a new
    cfg is captured again."""
    w = get("llama8b_n32k")
    g = generate(w, q_heads=range(8), kv_heads=range(2))
    w = w.with_params(hq=8, hkv=2)
    q, k, v = to_device(g["q"]), to_device(g["k"]), to_device(g["v"])
    dims = dsp.make_dims(1, w.n, w.hq, w.hkv)
    ctx = dsp.Context(dims)

    def run(wl, flags, o):
        ctx.prefill(dims, q, k, v, _cfg(dsp, wl, flags=flags), o)
        torch.cuda.synchronize()
        assert ctx.sync_status() == 0
        return ctx.selection_get(dims)

    def same_sel(a, b):
        assert a.keys() == b.keys()
        for key in a:
            assert np.array_equal(np.asarray(a[key]), np.asarray(b[key])), key

    o_e = torch.empty_like(q)
    sel_e = run(w, 0, o_e)
    o_g = torch.full_like(q, 7.0)
    for _ in range(3):  # capture, then two replays
        sel_g = run(w, dsp.FLAG_GRAPH_REPLAY, o_g)
        assert torch.equal(o_e, o_g)
        same_sel(sel_e, sel_g)
    o_g2 = torch.zeros_like(q)
    run(w, dsp.FLAG_GRAPH_REPLAY, o_g2)
    assert torch.equal(o_e, o_g2)
    w2 = w.with_params(alpha=2.0, gamma=0.9)
    o_e2, o_g3 = torch.empty_like(q), torch.zeros_like(q)
    sel_e2 = run(w2, 0, o_e2)
    sel_g3 = run(w2, dsp.FLAG_GRAPH_REPLAY, o_g3)
    assert torch.equal(o_e2, o_g3)
    same_sel(sel_e2, sel_g3)
    assert not torch.equal(o_e, o_e2)
    ctx.close()


@pytest.mark.parametrize("alpha,kmin,gamma", [(0.0, 0, 0.5), (1.25, 0, 0.95), (1.0, 4096, 1.0),
                                              (3.0, 256, 0.99)])
def test_parameter_edges(dsp, alpha, kmin, gamma):
    w = get("tiny_n4k").with_params(alpha=alpha, k_min_tokens=kmin, gamma=gamma)
    run_parity(dsp, w, generate(w))


def test_llama_n32k_full(dsp):
    w = get("llama8b_n32k")
    rep, sel, osel = run_parity(dsp, w, generate(w))
    assert rep["vs_heads"] + rep["pe_heads"] + rep["route_mismatch_exempt"] == w.hq
    print("llama8b_n32k", rep)


def test_dense_matches_oracle_and_sdpa(dsp):
    """crisp_dense vs the oracle's dense causal attention (all blocks) on sampled rows, and
    against torch's SDPA (a library cross-check) on every row."""
    w = get("llama8b_n32k")
    g = generate(w, q_heads=range(8), kv_heads=range(2))
    w = w.with_params(hq=8, hkv=2, pe_heads=())
    q, k, v = to_device(g["q"]), to_device(g["k"]), to_device(g["v"])
    dims = dsp.make_dims(1, w.n, w.hq, w.hkv)
    ctx = dsp.Context(dims)
    o = torch.empty_like(q)
    ctx.dense(dims, q, k, v, o)
    assert ctx.sync_status() == 0
    assert ctx.attend_info() == 0   # no row of these inputs needs the rescue pass
    from oracle import crisp_oracle as O
    nb = w.n_blocks
    full = np.tril(np.ones((nb, nb), bool))
    got = o.float().cpu().numpy()
    for h in (0, 5):
        qh = O.bf16_bits_to_f64(g["q"][h])
        kh = O.bf16_bits_to_f64(g["k"][h // 4])
        vh = O.bf16_bits_to_f64(g["v"][h // 4])
        bl = [0, 1, 77, nb - 1]
        ref = O.block_sparse_attention(qh, kh, vh, full, 128, bl)
        compare_outputs(got[h][_rows(bl)], ref, f"dense head {h}")
    kk = k.repeat_interleave(4, dim=0)[None]
    vv = v.repeat_interleave(4, dim=0)[None]
    sd = torch.nn.functional.scaled_dot_product_attention(q[None], kk, vv, is_causal=True)[0]
    d = (sd.float() - o.float()).abs()
    assert float(d.max()) < 2e-2 and float(d.mean()) < 2e-3
    ctx.close()


def test_rescue_pass_recomputes_overflowing_rows(dsp):
    """The attention kernel exponentiates a row against one reference, the larger of the
    exact row maxima of its two first key blocks.  Three query rows of block 5 and one key
    of block 3 share a component of 30 (logit ~115 log2-units above the reference), which
    would overflow: the item must go to the rescue pass (running maxima) and still match
    the oracle's exact softmax, through crisp_dense and through a hand-set sparse
    selection; a selection without block 3 needs no rescue."""
    from oracle import crisp_oracle as O
    from workloads.planted import f32_to_bf16_bits
    n, hq, hkv = 1024, 2, 1
    nb = n // 128
    g = random_qkv(n, hq, hkv, 128, seed=41, scale=4.0)
    q, k, v = g["q"].copy(), g["k"].copy(), g["v"]
    big = f32_to_bf16_bits(np.float32([30.0]))[0]
    for r in (5 * 128 + 3, 5 * 128 + 64, 5 * 128 + 127):
        q[0, r, :] = 0
        q[0, r, 1] = big
    k[0, 3 * 128 + 7, :] = 0
    k[0, 3 * 128 + 7, 1] = big
    dq, dk, dv = to_device(q), to_device(k), to_device(v)
    dims = dsp.make_dims(1, n, hq, hkv)
    ctx = dsp.Context(dims)
    qf = [O.bf16_bits_to_f64(q[h]) for h in range(hq)]
    kf, vf = O.bf16_bits_to_f64(k[0]), O.bf16_bits_to_f64(v[0])

    o = torch.empty_like(dq)
    ctx.dense(dims, dq, dk, dv, o)
    assert ctx.sync_status() == 0
    assert ctx.attend_info() == 1
    got = o.float().cpu().numpy()
    full = np.tril(np.ones((nb, nb), bool))
    for h in range(hq):
        ref = O.block_sparse_attention(qf[h], kf, vf, full, 128, list(range(nb)))
        compare_outputs(got[h], ref, f"dense with rescue, head {h}")

    for with_key, rescued in ((True, 1), (False, 0)):
        masks = [np.eye(nb, dtype=bool) for _ in range(hq)]
        masks[0][:, 0] = True
        masks[0][5, 1] = True          # blocks 0 and 1 are the row's first blocks
        if with_key:
            masks[0][5, 3] = True      # third block: above the reference by ~110 log2-units
        rp, col = csr_from_masks(masks, nb)
        ctx.selection_set(dims, rp, col)
        o2 = torch.empty_like(dq)
        ctx.attend(dims, dq, dk, dv, o2)
        assert ctx.sync_status() == 0
        assert ctx.attend_info() == rescued
        got = o2.float().cpu().numpy()
        for h in range(hq):
            ref = O.block_sparse_attention(qf[h], kf, vf, np.tril(masks[h]), 128, list(range(nb)))
            compare_outputs(got[h], ref, f"sparse with_key={with_key}, head {h}")
    ctx.close()


@pytest.mark.parametrize("n,row,keys", [(4096, 30, 13), (65536, 486, 195)])
def test_pe_tie_ranks_exact_on_zero_queries(dsp, n, row, keys):
    """Queries of zeros make every pooled score 0, so row I of the PE triangle holds I + 1
    equal values v = 1/((I+1) N_b): each row carries 1/N_b of the mass and ties decide the
    cut.  gamma = 0.95: rows 0..row-1 are taken whole (row = floor(0.95 N_b)) and the rest of
    the mass, 0.95 - row/N_b, comes from the first ceil((0.95 - row/N_b) N_b (row+1)) keys of
    row `row` in flat order (tie ranks across the head), plus the forced diagonals.
    N_b = 32 (13 keys of row 30) runs the one-kernel cut of short sequences, N_b = 512 (195
    keys of row 486) the multi-kernel radix select.  The GPU's index set must equal the
    oracle's and this closed form exactly (no exemption)."""
    hq, hkv = 2, 1
    nb = n // 128
    assert row == int(0.95 * nb) and keys == int(np.ceil((0.95 - row / nb) * nb * (row + 1)))
    g = random_qkv(n, hq, hkv, 128, seed=81, scale=3.0)
    g["q"][:] = 0
    w = Workload("zero_q", n=n, hq=hq, hkv=hkv, seed=81)
    rep, sel, osel = run_parity(dsp, w, g, flags=dsp.FLAG_FORCE_PE,
                                sample=None if nb <= 64 else (2, 8), seed=3)
    expect = np.tril(np.ones((nb, nb), bool))
    expect[row:] = False
    expect[row, :keys] = True
    expect[np.arange(row, nb), np.arange(row, nb)] = True
    gm = gpu_masks(sel, hq, nb)
    for h in range(hq):
        assert np.array_equal(np.tril(osel[h]["mask"]), expect), h
        assert np.array_equal(gm[h], expect), h
    assert rep["pe_pair_exempt"] == 0


@pytest.mark.parametrize("n,hq,hkv,seed", [(4096, 4, 2, 71), (4736, 4, 1, 72)])
def test_attend_random_index_sets(dsp, n, hq, hkv, seed):
    """crisp_attend on arbitrary caller-supplied index sets (crisp_selection_set): per row a
    random non-empty subset of [0, I] whose density ranges from one block to every block,
    the diagonal block included or not, N_b = 32 and a ragged 37; every query block of
    every head against the oracle's exact attention on the same sets."""
    from oracle import crisp_oracle as O
    nb = n // 128
    g = random_qkv(n, hq, hkv, 128, seed, scale=3.0)
    rng = np.random.default_rng(seed)
    masks = []
    for h in range(hq):
        m = np.zeros((nb, nb), bool)
        for I in range(nb):
            p = rng.choice([0.0, 0.15, 0.5, 1.0])
            row = rng.random(I + 1) < p
            if rng.random() < 0.7:
                row[I] = True
            if not row.any():
                row[rng.integers(0, I + 1)] = True
            m[I, : I + 1] = row
        masks.append(m)
    assert any(not masks[h][I, I] for h in range(hq) for I in range(1, nb))
    q, k, v = to_device(g["q"]), to_device(g["k"]), to_device(g["v"])
    dims = dsp.make_dims(1, n, hq, hkv)
    ctx = dsp.Context(dims)
    rp, col = csr_from_masks(masks, nb)
    ctx.selection_set(dims, rp, col)
    o = torch.empty_like(q)
    ctx.attend(dims, q, k, v, o)
    assert ctx.sync_status() == 0
    got = o.float().cpu().numpy()
    grp = hq // hkv
    for h in range(hq):
        ref = O.block_sparse_attention(O.bf16_bits_to_f64(g["q"][h]),
                                       O.bf16_bits_to_f64(g["k"][h // grp]),
                                       O.bf16_bits_to_f64(g["v"][h // grp]), masks[h], 128,
                                       list(range(nb)))
        compare_outputs(got[h], ref, f"random index sets, head {h}")
    ctx.close()


@pytest.mark.parametrize("name", ["tiny_n4k", "llama8b_n32k"])
def test_prefill_host_matches_device_path(dsp, name):
    """crisp_prefill_host (host buffers, chunked by KV-head groups, copies overlapped)
    gives the device path's output: the heads are independent, so per-chunk selection and
    attention are the same computation (up to the attention's summation order)."""
    w = get(name)
    g = generate(w)
    q, k, v = to_device(g["q"]), to_device(g["k"]), to_device(g["v"])
    dims = dsp.make_dims(1, w.n, w.hq, w.hkv)
    ctx = dsp.Context(dims)
    cfg = _cfg(dsp, w)
    o = torch.empty_like(q)
    ctx.prefill(dims, q, k, v, cfg, o)
    assert ctx.sync_status() == 0
    ref = o.float().cpu().numpy().astype(np.float64)
    t = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
    qh, kh, vh = t(g["q"]), t(g["k"]), t(g["v"])
    oh = torch.zeros(o.shape, dtype=torch.bfloat16).pin_memory()
    q2, k2, v2, o2 = (torch.empty_like(x) for x in (q, k, v, o))
    ctx.prefill_host(dims, qh, kh, vh, cfg, oh, q2, k2, v2, o2)
    assert ctx.sync_status() == 0
    got = oh.float().numpy()
    for h in range(w.hq):
        compare_outputs(got[h], ref[h], f"prefill_host vs prefill, head {h}")
    with pytest.raises(dsp.CrispError):   # the call leaves no selection behind
        ctx.attend(dims, q, k, v, o)
    ctx.close()


def test_prefill_host_batch_two_uneven_chunks(dsp):
    """crisp_prefill_host with batch 2 and 4 KV heads per entry (8 flattened KV heads) at
    32k: the chunks hold 3, 3 and 2 KV heads, so the second spans both batch entries in the
    flattened layout and the last is smaller; the output must match the device path."""
    n, hq, hkv = 32768, 8, 4
    g = random_qkv(n, 2 * hq, 2 * hkv, 128, seed=57, scale=3.0)
    q, k, v = to_device(g["q"]), to_device(g["k"]), to_device(g["v"])
    dims = dsp.make_dims(2, n, hq, hkv)
    ctx = dsp.Context(dims)
    cfg = dsp.default_cfg()
    o = torch.empty_like(q)
    ctx.prefill(dims, q, k, v, cfg, o)
    assert ctx.sync_status() == 0
    ref = o.float().cpu().numpy().astype(np.float64)
    t = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
    qh, kh, vh = t(g["q"]), t(g["k"]), t(g["v"])
    oh = torch.zeros(o.shape, dtype=torch.bfloat16).pin_memory()
    q2, k2, v2, o2 = (torch.empty_like(x) for x in (q, k, v, o))
    ctx.prefill_host(dims, qh, kh, vh, cfg, oh, q2, k2, v2, o2)
    assert ctx.sync_status() == 0
    got = oh.float().numpy()
    for h in range(2 * hq):
        compare_outputs(got[h], ref[h], f"prefill_host batch 2, head {h}")
    ctx.close()


def test_prefill_host_single_head_end_chunks(dsp):
    """At 64k with 4 query heads per KV head, chunks hold one KV head and the first and
    last groups are split into one query head per chunk (K/V uploaded with the group's
    first head): the output must still match the device path."""
    n, hq, hkv = 65536, 8, 2
    g = random_qkv(n, hq, hkv, 128, seed=61, scale=3.0)
    q, k, v = to_device(g["q"]), to_device(g["k"]), to_device(g["v"])
    dims = dsp.make_dims(1, n, hq, hkv)
    ctx = dsp.Context(dims)
    cfg = dsp.default_cfg()
    o = torch.empty_like(q)
    ctx.prefill(dims, q, k, v, cfg, o)
    assert ctx.sync_status() == 0
    ref = o.float().cpu().numpy().astype(np.float64)
    t = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
    qh, kh, vh = t(g["q"]), t(g["k"]), t(g["v"])
    oh = torch.zeros(o.shape, dtype=torch.bfloat16).pin_memory()
    q2, k2, v2, o2 = (torch.empty_like(x) for x in (q, k, v, o))
    ctx.prefill_host(dims, qh, kh, vh, cfg, oh, q2, k2, v2, o2)
    assert ctx.sync_status() == 0
    got = oh.float().numpy()
    for h in range(hq):
        compare_outputs(got[h], ref[h], f"prefill_host single-head chunks, head {h}")
    ctx.close()


def test_timeout_is_reported_and_context_recovers(dsp):
    """A dropped barrier arrive makes a bounded wait run out: the kernel exits, the host
    reads CRISP_ERR_TIMEOUT, and the next call on the same context succeeds."""
    w = get("tiny_n4k")
    g = generate(w)
    q, k, v = to_device(g["q"]), to_device(g["k"]), to_device(g["v"])
    dims = dsp.make_dims(1, w.n, w.hq, w.hkv)
    ctx = dsp.Context(dims)
    o = torch.empty_like(q)
    ctx.set_debug(dsp.DEBUG_DROP_ARRIVE)
    ctx.dense(dims, q, k, v, o)
    assert ctx.sync_status() == 5  # CRISP_ERR_TIMEOUT
    ctx.set_debug(0)
    ctx.dense(dims, q, k, v, o)
    assert ctx.sync_status() == 0
    ref = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], v[None], is_causal=True)[0]
    assert float((ref.float() - o.float()).abs().max()) < 2e-2
    ctx.close()


def test_api_errors(dsp):
    w = get("tiny_n4k")
    g = generate(w)
    q, k, v = to_device(g["q"]), to_device(g["k"]), to_device(g["v"])
    dims = dsp.make_dims(1, w.n, w.hq, w.hkv)
    ctx = dsp.Context(dims)
    o = torch.empty_like(q)
    with pytest.raises(dsp.CrispError) as e:
        ctx.attend(dims, q, k, v, o)
    assert e.value.status == 7
    big = dsp.make_dims(1, 2 * w.n, w.hq, w.hkv)
    with pytest.raises(dsp.CrispError) as e:
        ctx.dense(big, q, k, v, o)
    assert e.value.status == 1
    nb = w.n_blocks
    rp = np.arange(w.hq * nb + 1, dtype=np.int64)
    bad = np.tile(np.arange(nb, dtype=np.int32) + 1, w.hq)  # key block I+1 > I
    with pytest.raises(dsp.CrispError) as e:
        ctx.selection_set(dims, rp, bad)
    assert e.value.status == 1
    cfg = dsp.default_cfg(gamma=0.0)
    with pytest.raises(dsp.CrispError) as e:
        ctx.select(dims, q, k, cfg)
    assert e.value.status == 1
    ctx.close()


@pytest.mark.parametrize("name", ["llama8b_n128k_a1", "llama8b_n128k_a125", "qwen7b_n128k"])
def test_n128k_sampled(dsp, name):
    w = get(name)
    rep, _, _ = run_parity(dsp, w, generate(w), sample=(8, 16), seed=7)
    print(name, rep)


def test_llama_n512k_sampled_and_dense(dsp):
    w = get("llama8b_n512k")
    g = generate(w)
    rep, _, osel = run_parity(dsp, w, g, sample=(8, 16), seed=11)
    print("llama8b_n512k", rep)
    # dense on the same inputs, sampled rows against the oracle
    q, k, v = to_device(g["q"]), to_device(g["k"]), to_device(g["v"])
    dims = dsp.make_dims(1, w.n, w.hq, w.hkv)
    ctx = dsp.Context(dims)
    o = torch.empty_like(q)
    ctx.dense(dims, q, k, v, o)
    assert ctx.sync_status() == 0
    assert ctx.attend_info() == 0   # no row of these inputs needs the rescue pass
    from oracle import crisp_oracle as O
    nb = w.n_blocks
    full = np.tril(np.ones((nb, nb), bool))
    got = o[[0, 31]].float().cpu().numpy()
    for i, h in enumerate((0, 31)):
        qh = O.bf16_bits_to_f64(g["q"][h])
        kh = O.bf16_bits_to_f64(g["k"][h // w.group])
        vh = O.bf16_bits_to_f64(g["v"][h // w.group])
        bl = [3, nb // 2, nb - 1]
        ref = O.block_sparse_attention(qh, kh, vh, full, 128, bl)
        compare_outputs(got[i][_rows(bl)], ref, f"dense 512k head {h}")
    ctx.close()


def test_max_length_n1m(dsp):
    """The longest supported sequence (n = 2^20, N_b = 8192: the VS selection's shared-memory
    sort at its size limit, an 8192 x 8192 PE triangle), one VS-planted and one PE head:
    full selection parity, outputs on sampled query blocks."""
    w = Workload("max_n1m", n=1 << 20, hq=2, hkv=1, seed=2024, sink_scale=4.0,
                 needles=("fixed", 6), pe_heads=(1,))
    rep, sel, _ = run_parity(dsp, w, generate(w), sample=(2, 3), seed=5)
    assert rep["vs_heads"] + rep["pe_heads"] == 2
    print("max_n1m", rep)


@pytest.mark.parametrize("name,sample", [("llama8b_n8k", None), ("llama8b_n16k", None),
                                         ("llama8b_n64k", (8, 16)), ("llama8b_n256k", (8, 16))])
def test_sweep_lengths(dsp, name, sample):
    """The other lengths of the latency sweep hold the same parity bar."""
    w = get(name)
    rep, _, _ = run_parity(dsp, w, generate(w), sample=sample, seed=3)
    print(name, rep)


@pytest.mark.parametrize("name", ["tiny_n4k", "llama8b_n32k"])
@pytest.mark.parametrize("variant", [dict(vs_floor="median"), dict(vs_rule="gamma")])
def test_vs_variants(dsp, name, variant):
    """Median noise floor and FlexPrefill's gamma-cumsum VS budget (the Abl.1 rule) hold
    the same parity bar as the page's rule."""
    w = get(name).with_params(**variant)
    rep, sel, osel = run_parity(dsp, w, generate(w), sample=None if name == "tiny_n4k" else (8, 8),
                                seed=5)
    print(name, variant, rep)


@pytest.mark.parametrize("name", ["tiny_n4k", "llama8b_n32k", "qwen7b_n128k"])
def test_jsd_routing_diagnostic(dsp, name):
    """crisp_jsd (FlexPrefill's JSD signal) against the oracle: D_JS per head within
    1e-4 + 1e-3 relative, JSD routes equal except within 1e-3 relative of tau_jsd."""
    from oracle import crisp_oracle as O
    w = get(name)
    g = generate(w)
    q, k = to_device(g["q"]), to_device(g["k"])
    dims = dsp.make_dims(1, w.n, w.hq, w.hkv)
    ctx = dsp.Context(dims)
    ctx.select(dims, q, k, _cfg(dsp, w))
    tau = 0.1
    d_js = torch.zeros(w.hq, dtype=torch.float32, device="cuda")
    route = torch.zeros(w.hq, dtype=torch.uint8, device="cuda")
    ctx.jsd(dims, q, k, tau, d_js, route)
    assert ctx.sync_status() == 0
    sel = ctx.selection_get(dims, with_csr=False)
    dj, rt = d_js.cpu().numpy(), route.cpu().numpy()
    agree = 0
    for h in range(w.hq):
        qh = O.bf16_bits_to_f64(g["q"][h])
        kh = O.bf16_bits_to_f64(g["k"][h // w.group])
        ref = O.jsd_route(qh, kh, w.B, w.b, tau)
        assert abs(dj[h] - ref["d_js"]) <= 1e-4 + 1e-3 * ref["d_js"], (h, dj[h], ref["d_js"])
        if bool(rt[h]) != ref["route_vs"]:
            assert abs(ref["d_js"] - tau) <= 1e-3 * tau
        agree += int(bool(rt[h]) == bool(sel["route_vs"][h]))
    print(name, "JSD/C_struct route agreement", agree, "/", w.hq, "D_JS", np.round(dj, 4).tolist())
    with pytest.raises(dsp.CrispError):   # p_v must come from crisp_select, not selection_set
        nb = w.n_blocks
        rp = np.arange(w.hq * nb + 1, dtype=np.int64)
        ctx.selection_set(dims, rp, np.tile(np.arange(nb, dtype=np.int32), w.hq))
        ctx.jsd(dims, q, k, tau, d_js, route)
    ctx.close()


def test_batch_two_matches_flattened_heads(dsp):
    """batch = 2 with (hq, hkv) = (4, 2) addresses the same heads and KV heads as batch = 1
    with (8, 4): routes, selections and outputs must be bit-identical; the flattened case
    also holds oracle parity."""
    w = Workload("batch_flat", n=4096, hq=8, hkv=4, seed=77, pe_heads=(1, 6),
                 needles=("uniform", 2, 6))
    g = generate(w)
    run_parity(dsp, w, g)
    q, k, v = to_device(g["q"]), to_device(g["k"]), to_device(g["v"])
    outs, sels = [], []
    for dims in (dsp.make_dims(1, w.n, 8, 4), dsp.make_dims(2, w.n, 4, 2)):
        ctx = dsp.Context(dims)
        o = torch.empty_like(q)
        ctx.prefill(dims, q, k, v, _cfg(dsp, w), o)
        assert ctx.sync_status() == 0
        sels.append(ctx.selection_get(dims))
        outs.append(o.clone())
        ctx.close()
    for key in ("route_vs", "c_struct", "sel_v", "sel_s", "row_ptr", "col"):
        assert np.array_equal(sels[0][key], sels[1][key]), key
    assert torch.equal(outs[0], outs[1])


def test_batch_two_matches_flattened_heads_multi_kernel(dsp):
    """The same check at 64k (N_b = 512, above the one-CTA limit): the PE radix passes, tie
    counts and masks walk the device-built list of PE heads, which with batch = 2 holds heads
    of both entries; routes, selections and outputs must match the flattened layout bit for
    bit, and the flattened case holds sampled oracle parity."""
    w = Workload("batch_flat_64k", n=65536, hq=8, hkv=4, seed=78, pe_heads=(1, 6),
                 needles=("uniform", 2, 6))
    g = generate(w)
    run_parity(dsp, w, g, sample=(4, 6), seed=3)
    q, k, v = to_device(g["q"]), to_device(g["k"]), to_device(g["v"])
    outs, sels = [], []
    for dims in (dsp.make_dims(1, w.n, 8, 4), dsp.make_dims(2, w.n, 4, 2)):
        ctx = dsp.Context(dims)
        o = torch.empty_like(q)
        ctx.prefill(dims, q, k, v, _cfg(dsp, w), o)
        assert ctx.sync_status() == 0
        sels.append(ctx.selection_get(dims))
        outs.append(o.clone())
        ctx.close()
    assert sels[0]["route_vs"].tolist().count(0) == 2  # one PE head in each batch entry
    for key in ("route_vs", "c_struct", "sel_v", "sel_s", "row_ptr", "col"):
        assert np.array_equal(sels[0][key], sels[1][key]), key
    assert torch.equal(outs[0], outs[1])


def test_repeated_selections_reset_their_state(dsp):
    """One context, selections with different PE head sets in a row at 64k (the multi-kernel
    PE path): every head forced PE, the planted routes, every head forced VS, the planted
    routes again.  Each must equal what a fresh context selects on the same inputs bit for
    bit: the PE head list, the radix state, the histograms and the near counts are rebuilt
    on every call."""
    w = Workload("repeat_64k", n=65536, hq=8, hkv=4, seed=79, pe_heads=(2, 5),
                 needles=("uniform", 2, 6))
    g = generate(w)
    q, k = to_device(g["q"]), to_device(g["k"])
    dims = dsp.make_dims(1, w.n, w.hq, w.hkv)
    keys = ("route_vs", "c_struct", "sel_v", "sel_s", "counts", "row_ptr", "col")

    def fresh(flags):
        c = dsp.Context(dims)
        c.select(dims, q, k, _cfg(dsp, w, flags=flags))
        assert c.sync_status() == 0
        out = c.selection_get(dims), c.stats(dims)
        c.close()
        return out

    ref = {f: fresh(f) for f in (dsp.FLAG_FORCE_PE, 0, dsp.FLAG_FORCE_VS)}
    ctx = dsp.Context(dims)
    for flags in (dsp.FLAG_FORCE_PE, 0, dsp.FLAG_FORCE_VS, 0):
        ctx.select(dims, q, k, _cfg(dsp, w, flags=flags))
        assert ctx.sync_status() == 0
        sel, st = ctx.selection_get(dims), ctx.stats(dims)
        rsel, rst = ref[flags]
        for key in keys:
            assert np.array_equal(sel[key], rsel[key]), (flags, key)
        assert st == rst, flags
    ctx.close()

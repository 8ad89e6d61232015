"""Pins of the fp64 CPU oracle against what the CRISP page and mathematics fix.

Each test ties an oracle function to something other than itself: a closed form, a
special case that reduces to a library routine, brute force on tiny inputs, or a worked
example under tests/golden/.  Sections cited are those of the analysis page "CRISP:
Cliff-awaRe Input-adaptive Sparse Prefilling with Structural-Mass-Motivated Routing"
(paper.rainbus.top).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import crisp_oracle as O
from workloads import get
from workloads.planted import generate

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ---------------------------------------------------------------- attention (step 4)
@pytest.mark.parametrize("n,d,B", [(512, 16, 128), (384, 128, 128), (256, 32, 32)])
def test_all_blocks_equals_dense_causal_sdpa(n, d, B):
    """Special case -> library: with every block K <= I selected, A(Q,K,V,S) is dense
    causal softmax attention ("Prerequisites": prefill and sparse attention)."""
    q, k, v = (_rand((n, d), s) for s in (1, 2, 3))
    nb = n // B
    mask = np.tril(np.ones((nb, nb), dtype=bool))
    got = O.block_sparse_attention(q, k, v, mask, B)
    t = lambda a: torch.from_numpy(a)[None, None]
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True)
    np.testing.assert_allclose(got, ref[0, 0].numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_block_sparse_attention_bruteforce_full_matrix(seed):
    """Brute force: the page's formula Softmax(QK^T/sqrt(d) + M_S) V written as one n x n
    matrix with M_S = -inf outside the selected blocks and above the diagonal."""
    n, d, B = 256, 16, 32
    nb = n // B
    rng = np.random.default_rng(seed)
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    mask = np.tril(rng.random((nb, nb)) < 0.4)
    mask[np.arange(nb), np.arange(nb)] = True
    got = O.block_sparse_attention(q, k, v, mask, B)
    ii, jj = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    allowed = mask[ii // B, jj // B] & (jj <= ii)
    logits = q @ k.T / math.sqrt(d)
    logits[~allowed] = -np.inf
    w = np.exp(logits - logits.max(axis=1, keepdims=True))
    ref = (w / w.sum(axis=1, keepdims=True)) @ v
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    # sampled blocks give the same rows
    blocks = [nb - 1, 2, 0]
    part = O.block_sparse_attention(q, k, v, mask, B, blocks)
    rows = np.concatenate([np.arange(I * B, (I + 1) * B) for I in blocks])
    np.testing.assert_allclose(part, ref[rows], rtol=0, atol=1e-12)


def test_attention_per_token_loop_tiny():
    """Brute force with scalar loops on a tiny case (n=16, B=4)."""
    n, d, B = 16, 3, 4
    rng = np.random.default_rng(7)
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    mask = np.array([[1, 0, 0, 0], [0, 1, 0, 0], [1, 0, 1, 0], [0, 1, 1, 1]], dtype=bool)
    got = O.block_sparse_attention(q, k, v, mask, B)
    for i in range(n):
        keys = [j for j in range(i + 1) if mask[i // B, j // B]]
        s = [sum(q[i, t] * k[j, t] for t in range(d)) / math.sqrt(d) for j in keys]
        mx = max(s)
        e = [math.exp(x - mx) for x in s]
        z = sum(e)
        ref = [sum(e[a] / z * v[j, t] for a, j in enumerate(keys)) for t in range(d)]
        np.testing.assert_allclose(got[i], ref, rtol=0, atol=1e-13)


# ---------------------------------------------------------------- PatSearch (step 1)
@pytest.mark.parametrize("n,b", [(1024, 128), (256, 128), (128, 128)])
def test_proxy_uniform_logits_closed_form(n, b):
    """Q = 0 makes every visible logit 0, so A_hat[r, j] = 1/(p_r+1) for j <= p_r (causal
    proxy), and a_v, a_s and C_struct have closed forms."""
    d = 16
    q = np.zeros((n, d))
    k = _rand((n, d), 5)
    a = O.proxy_attention(q, k, b)
    pos = n - b + np.arange(b)
    for r in (0, b // 2, b - 1):
        np.testing.assert_allclose(a[r, : pos[r] + 1], 1.0 / (pos[r] + 1), rtol=1e-14)
        assert np.all(a[r, pos[r] + 1:] == 0)
    j = np.arange(n)
    av_ref = np.array([sum(1.0 / (p + 1) for p in pos if p >= jj) for jj in j]) / b
    np.testing.assert_allclose(O.vertical_score(a), av_ref, rtol=1e-13)
    # the slash score at offset delta sums the same reciprocals over rows with p_r >= delta
    np.testing.assert_allclose(O.slash_score(a), av_ref, rtol=1e-13)
    ws, wl = 128, 128
    anchors = [jj for jj in j if jj < ws or jj >= n - wl]
    c_ref = sum(sum(1.0 / (p + 1) for p in pos if p >= jj) for jj in anchors) / b
    assert abs(O.c_struct_from_av(O.vertical_score(a), ws, wl) - c_ref) < 1e-13


@pytest.mark.parametrize("n,k,delta", [(4096, 6, 12.0), (32768, 40, 9.5), (2048, 1, 3.0)])
def test_mass_cliff_epsilon_closed_form(n, k, delta):
    """Mass cliff ("Core method", innovation 2): one softmax row with k signal logits
    Delta and n-k zero logits gives each background token e^-D/(k + (n-k)e^-D).  Planted
    with d = 2: signal keys (sqrt(2), 0), background keys 0, queries (Delta, 0)."""
    d, b, B = 2, 128, 128
    kk = np.zeros((n, d))
    sig = np.arange(100, 100 + k)                  # all visible to every proxy row
    kk[sig, 0] = math.sqrt(2.0)
    q = np.zeros((n, d))
    q[:, 0] = delta
    a = O.proxy_attention(q, kk, b)
    for r in (0, 77, b - 1):
        nr = n - b + r + 1                          # keys visible to proxy row r
        eps = O.mass_cliff_epsilon(nr, k, delta)
        e = math.exp(-delta)
        assert abs(eps - e / (k + (nr - k) * e)) <= 1e-15 * eps
        bg = np.setdiff1d(np.arange(nr), sig)
        np.testing.assert_allclose(a[r, bg], eps, rtol=1e-13)
        np.testing.assert_allclose(a[r, sig], eps * math.exp(delta), rtol=1e-13)
    # a background block's pooled vertical mass is the row average of B * eps_r
    p_v = O.block_pool(O.vertical_score(a), B)
    J = (n - b) // B - 1
    assert J * B > sig[-1]
    eps_rows = [O.mass_cliff_epsilon(n - b + r + 1, k, delta) for r in range(b)]
    assert abs(p_v[J] - B * np.mean(eps_rows)) <= 1e-13 * p_v[J]


@pytest.mark.parametrize("k,delta,gamma", [(4, 8.0, 0.95), (16, 6.0, 0.9)])
def test_gamma_cumsum_garbage_grows_linearly(k, delta, gamma):
    """N_garbage ("Core method"): when the signal holds k*eps_s < gamma of the mass, the
    gamma-cumsum takes every signal token plus ceil((gamma - k eps_s)/eps) background
    tokens, a number linear in n."""
    counts = []
    for n in (2000, 4000, 8000, 16000):
        e = math.exp(-delta)
        z = k + (n - k) * e
        eps_s, eps = 1.0 / z, e / z
        assert k * eps_s < gamma
        vals = np.full(n, eps)
        vals[:k] = eps_s
        sel = O.gamma_cut(vals, gamma)
        expect = k + math.ceil((gamma - k * eps_s) / eps)
        assert sel.size == expect
        assert set(range(k)) <= set(sel.tolist())
        counts.append(sel.size - k)
    ratios = np.array(counts[1:]) / np.array(counts[:-1])
    assert np.all(ratios > 1.8)                   # ~2x per doubling of n


def test_slash_and_vertical_index_direction():
    """Hand-built A_hat: every proxy row puts all its mass on key p_r - delta0.  Then the
    slash score is 1 at delta0 only (delta = query minus key position) and the vertical
    score is 1/b on each of those keys."""
    n, b, delta0 = 1024, 128, 37
    a = np.zeros((b, n))
    pos = n - b + np.arange(b)
    a[np.arange(b), pos - delta0] = 1.0
    a_s = O.slash_score(a)
    assert a_s[delta0] == 1.0 and np.count_nonzero(a_s) == 1
    a_v = O.vertical_score(a)
    np.testing.assert_allclose(a_v[pos - delta0], 1.0 / b)
    assert np.count_nonzero(a_v) == b


def test_scores_sum_to_one_and_anchor_slice():
    """sum(a_v) = sum(a_s) = 1; C_struct equals the anchor-slice sum of A_hat taken
    directly from the b x n map ("Core method" step 1)."""
    w = get("tiny_n4k")
    g = generate(w)
    for h in range(w.hq):
        q = O.bf16_bits_to_f64(g["q"][h])
        k = O.bf16_bits_to_f64(g["k"][h // w.group])
        a = O.proxy_attention(q, k, w.b)
        a_v, a_s = O.vertical_score(a), O.slash_score(a)
        assert abs(a_v.sum() - 1) < 1e-12 and abs(a_s.sum() - 1) < 1e-12
        direct = (a[:, : w.w_sink].sum() + a[:, w.n - w.w_local:].sum()) / w.b
        assert abs(O.c_struct_from_av(a_v, w.w_sink, w.w_local) - direct) < 1e-12


def test_noise_floor_closed_form_from_c_struct():
    """With w_sink = w_local = B, r_v = 1 - p_v[0] - p_v[N_b-1] = 1 - C_struct, so
    mu_v = max(1 - C_struct, 0)/(N_b - 2)."""
    w = get("tiny_n4k")
    g = generate(w)
    q = O.bf16_bits_to_f64(g["q"][0])
    k = O.bf16_bits_to_f64(g["k"][0])
    res = O.crisp_select_head(q, k, **O.workload_params(w))
    nb = w.n_blocks
    assert abs(res["mu_v"] - max(1 - res["c_struct"], 0) / (nb - 2)) < 1e-15
    assert O.noise_floor(np.array([0.3, 0.7])) == 0.0


# ---------------------------------------------------------------- VSIndex (step 2)
def test_vs_select_worked_example():
    fx = json.load(open(os.path.join(GOLD, "vs_select_worked.json")))
    p = np.array(fx["p"])
    mu = O.noise_floor(p)
    assert abs(mu - fx["mu"]) < 1e-15
    for case in fx["cases"]:
        S, c, kd = O.select_above_floor(p, case["alpha"], mu, case["kmin_blocks"])
        assert c == case["count_above"]
        assert S.tolist() == case["selected"]


def test_vs_block_mask_worked_example():
    fx = json.load(open(os.path.join(GOLD, "vs_block_mask_worked.json")))
    m = O.vs_block_mask(np.array(fx["S_v"]), np.array(fx["S_s"]), fx["n_blocks"])
    rows = [np.nonzero(m[I])[0].tolist() for I in range(fx["n_blocks"])]
    assert rows == fx["rows"]


def test_vs_select_threshold_is_strict():
    """Algorithm 3 keeps the blocks strictly above alpha * mu_d.  With binary-exact scores
    the four non-anchor blocks sit exactly on the floor (r = 1 - 1/4 - 1/4 = 1/2,
    mu = r / 4 = 1/8, alpha = 1): only the two anchor blocks pass."""
    p = np.array([0.25, 0.125, 0.125, 0.125, 0.125, 0.25])
    mu = O.noise_floor(p)
    assert mu == 0.125
    S, c, kd = O.select_above_floor(p, 1.0, mu, 1)
    assert (S.tolist(), c, kd) == ([0, 5], 2, 2)
    # k_min pads with the largest remaining blocks, ties to the lower index
    S, c, kd = O.select_above_floor(p, 1.0, mu, 3)
    assert (S.tolist(), c, kd) == ([0, 1, 5], 2, 3)


def test_noise_floor_clamps_at_zero():
    """Algorithm 3's floor is max(1 - p_d[0] - p_d[N_b-1], 0) / (N_b - 2): when the anchor
    blocks' scores sum past 1 (here by 2^-50, all values binary-exact) the floor is 0, and
    blocks with score 0 are not above it."""
    p = np.array([0.75, 0.0, 0.0, 0.25 + 2.0 ** -50])
    assert O.noise_floor(p) == 0.0
    S, c, kd = O.select_above_floor(p, 1.0, O.noise_floor(p), 0)
    assert (S.tolist(), c, kd) == ([0, 3], 2, 2)


def test_kmin_blocks():
    """"Method step details": k_min = 1024 tokens is 8 blocks of B = 128.  Reading for
    other values: at least k_min tokens, i.e. ceil(k_min / B) blocks."""
    assert O.kmin_blocks(1024, 128) == 8
    assert O.kmin_blocks(1000, 128) == 8
    assert O.kmin_blocks(1025, 128) == 9
    assert O.kmin_blocks(0, 128) == 0


@pytest.mark.parametrize("seed", range(6))
def test_vs_select_bruteforce_and_invariants(seed):
    """Brute force over all k-subsets of a tiny N_b: the selection is a maximum-mass
    k_d-subset; it contains every block above the floor; |S| >= min(k_min, N_b)."""
    rng = np.random.default_rng(seed)
    nb = 9
    p = rng.dirichlet(np.full(nb, 0.5))
    mu = O.noise_floor(p)
    for alpha in (0.0, 0.5, 1.0, 1.25, 3.0):
        for kmb in (0, 2, 4, 8, 12):
            S, c, kd = O.select_above_floor(p, alpha, mu, kmb)
            assert len(S) == kd == min(max(c, kmb), nb)
            above = set(np.nonzero(p > alpha * mu)[0].tolist())
            assert above <= set(S.tolist())
            best = max(sum(p[list(T)]) for T in itertools.combinations(range(nb), kd))
            assert abs(p[S].sum() - best) < 1e-15
            if alpha == 0.0:
                assert set(np.nonzero(p > 0)[0].tolist()) <= set(S.tolist())


# ---------------------------------------------------------------- PEIndex (step 3)
@pytest.mark.parametrize("seed", range(5))
def test_gamma_cut_bruteforce(seed):
    """Brute force over all subsets: the gamma-cut returns a set of minimum cardinality
    whose mass reaches gamma, and among those one of maximum mass."""
    rng = np.random.default_rng(100 + seed)
    vals = rng.dirichlet(np.ones(7))
    for gamma in (0.3, 0.6, 0.9, 0.95):
        sel = O.gamma_cut(vals, gamma)
        assert vals[sel].sum() >= gamma
        kmin = min(len(T) for r in range(1, 8) for T in itertools.combinations(range(7), r)
                   if vals[list(T)].sum() >= gamma)
        assert sel.size == kmin
        best = max(vals[list(T)].sum() for T in itertools.combinations(range(7), kmin))
        assert abs(vals[sel].sum() - best) < 1e-15
        # dropping the smallest selected item falls below gamma
        assert vals[sel].sum() - vals[sel].min() < gamma


def test_gamma_cut_stops_when_the_sum_reaches_gamma():
    """"Prerequisites", cumulative coverage: the smallest prefix (largest first) whose sum is
    >= gamma.  Binary-exact values reach gamma = 3/4 exactly after two items."""
    vals = np.array([0.125, 0.5, 0.125, 0.25])
    assert O.gamma_cut(vals, 0.75).tolist() == [1, 3]
    assert O.gamma_cut(vals, 0.75 + 2.0 ** -40).tolist() == [0, 1, 3]


def test_route_at_threshold_is_vs():
    """Algorithm 2 routes a head VS iff C_struct >= tau_proxy: with tau equal to the head's
    own C_struct the head is VS, with the next larger double it is PE."""
    w = get("tiny_n4k")
    g = generate(w)
    q = O.bf16_bits_to_f64(g["q"][0])
    k = O.bf16_bits_to_f64(g["k"][0])
    params = O.workload_params(w)
    c = O.crisp_select_head(q, k, **params)["c_struct"]
    params["tau_proxy"] = c
    assert O.crisp_select_head(q, k, **params)["route_vs"]
    params["tau_proxy"] = float(np.nextafter(c, np.inf))
    assert not O.crisp_select_head(q, k, **params)["route_vs"]


def test_gamma_one_selects_everything():
    vals = np.random.default_rng(3).dirichlet(np.ones(50))
    assert O.gamma_cut(vals, 1.0).size == 50


def test_pe_uniform_pooled_scores_closed_form():
    """Q = 0: pooled logits are all 0, so A_bar[I, K] = 1/(I+1) and v = 1/((I+1) N_b).
    N_b = 12, gamma = 0.9: rows 0..9 hold 10/12 of the mass; row 10's pairs weigh
    1/132 each and 9 of them bring the sum to >= 0.9 (8.8 needed).  Ties inside a row go
    to the lower key block, and row 11 is rescued with its diagonal."""
    nb, B, d = 12, 16, 8
    q = np.zeros((nb * B, d))
    k = _rand((nb * B, d), 11)
    pe = O.pe_index(q, k, B, 0.9)
    I = np.arange(nb)
    np.testing.assert_allclose(pe["a_bar"][I, 0], 1.0 / (I + 1), rtol=1e-15)
    exp = np.zeros((nb, nb), dtype=bool)
    for r in range(10):
        exp[r, : r + 1] = True
    exp[10, :9] = True
    exp[I, I] = True
    assert np.array_equal(pe["mask"], exp)
    assert pe["rescued_rows"].tolist() == [11]
    assert pe["n_selected"] == 55 + 9


def test_pe_scores_normalised():
    w = get("tiny_n4k")
    g = generate(w)
    q = O.bf16_bits_to_f64(g["q"][1])
    k = O.bf16_bits_to_f64(g["k"][1])
    pe = O.pe_index(q, k, w.B, w.gamma)
    nb = w.n_blocks
    np.testing.assert_allclose(pe["a_bar"].sum(axis=1), 1.0, rtol=1e-14)
    assert abs(pe["v"].sum() - 1.0) < 1e-13
    assert np.all(pe["v"][np.triu_indices(nb, 1)] == 0)
    sel = pe["v"][pe["mask"]]
    assert pe["v"][pe["v"] >= pe["v_star"]].sum() >= w.gamma - 1e-12
    assert sel.size >= pe["n_selected"]


# ---------------------------------------------------------------- whole algorithm
def test_planted_tiny_routes_and_end_to_end_bruteforce():
    """Planted tiny workload: head 0 (sink + needles) routes VS with its needle blocks
    selected, head 1 (diffuse) routes PE; the outputs match the full-matrix formula."""
    w = get("tiny_n4k")
    g = generate(w)
    params = O.workload_params(w)
    for h in range(w.hq):
        q = O.bf16_bits_to_f64(g["q"][h])
        k = O.bf16_bits_to_f64(g["k"][h // w.group])
        v = O.bf16_bits_to_f64(g["v"][h // w.group])
        res = O.crisp_head(q, k, v, blocks=[0, 5, w.n_blocks - 1], **params)
        if h == 0:
            assert res["route_vs"] and res["c_struct"] > 0.5
            assert set(g["params"]["needles"][0].tolist()) <= set(res["S_v"].tolist())
        else:
            assert not res["route_vs"] and res["c_struct"] < w.tau_proxy
        mask = res["mask"]
        B = w.B
        for bi, I in enumerate([0, 5, w.n_blocks - 1]):
            rows = np.arange(I * B, (I + 1) * B)
            allowed = mask[I, np.arange(w.n) // B][None, :] & (np.arange(w.n)[None, :] <= rows[:, None])
            logits = q[rows] @ k.T / math.sqrt(w.d)
            logits[~allowed] = -np.inf
            e = np.exp(logits - logits.max(axis=1, keepdims=True))
            ref = (e / e.sum(axis=1, keepdims=True)) @ v
            np.testing.assert_allclose(res["out"][bi * B:(bi + 1) * B], ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- VS variants (NEXT rows)
def test_vs_variants_worked_example():
    """Median noise floor and the gamma-cumsum VS budget against a hand-worked example."""
    fx = json.load(open(os.path.join(GOLD, "vs_variants_worked.json")))
    p = np.array(fx["p"])
    assert abs(O.noise_floor_median(p) - fx["median"]) < 1e-15
    assert abs(O.noise_floor(p) - fx["mean"]) < 1e-15
    for case in fx["median_floor_cases"]:
        S, _, _ = O.select_above_floor(p, case["alpha"], O.noise_floor_median(p), case["kmin_blocks"])
        assert S.tolist() == case["selected"]
    for case in fx["gamma_cases"]:
        S, cut, kd = O.select_gamma_cumsum(p, case["gamma"], case["kmin_blocks"])
        assert cut == case["cut"] and S.tolist() == case["selected"]


@pytest.mark.parametrize("seed", range(4))
def test_median_floor_bruteforce(seed):
    """The median floor is the middle order statistic of the non-anchor scores (counted
    directly): as many scores lie at or below it as at or above it."""
    rng = np.random.default_rng(200 + seed)
    for nb in (3, 4, 9, 10, 33):
        p = rng.dirichlet(np.ones(nb))
        mid = O.noise_floor_median(p)
        inner = p[1:nb - 1]
        assert np.count_nonzero(inner <= mid) >= (nb - 2 + 1) // 2
        assert np.count_nonzero(inner >= mid) >= (nb - 2 + 1) // 2
        if (nb - 2) % 2 == 1:
            assert mid in inner
    assert O.noise_floor_median(np.array([0.4, 0.6])) == 0.0


# ---------------------------------------------------------------- JSD routing (NEXT row)
def test_js_divergence_closed_forms():
    """D_JS = 0 for equal distributions; ln 2 for disjoint supports; a two-point closed
    form for x = (1, 0), y = (1/2, 1/2): 1/2 ln(4/3) + 1/4 ln(2/3) + 1/4 ln 2."""
    x = np.array([0.2, 0.3, 0.5])
    assert abs(O.js_divergence(x, x)) < 1e-16
    assert abs(O.js_divergence(np.array([1.0, 0, 0, 0]), np.array([0, 0, 0.5, 0.5])) - math.log(2)) < 1e-15
    ref = 0.5 * math.log(4 / 3) + 0.25 * math.log(2 / 3) + 0.25 * math.log(2)
    assert abs(O.js_divergence(np.array([1.0, 0.0]), np.array([0.5, 0.5])) - ref) < 1e-15
    rng = np.random.default_rng(9)
    for _ in range(5):
        a, b = rng.dirichlet(np.ones(7)), rng.dirichlet(np.ones(7))
        dj = O.js_divergence(a, b)
        assert 0 <= dj <= math.log(2) and abs(dj - O.js_divergence(b, a)) < 1e-15


def test_pooled_estimate_special_cases():
    """Q = 0 gives a uniform a_bar; keys constant within each block and a query equal to
    the block-J key give the softmax of the block dot products (closed form)."""
    n, d, B, b = 1024, 8, 128, 128
    k = np.random.default_rng(4).standard_normal((n, d))
    np.testing.assert_allclose(O.pooled_estimate(np.zeros((n, d)), k, B, b), 1.0 / (n // B),
                               rtol=1e-15)
    nb = n // B
    kb = np.random.default_rng(5).standard_normal((nb, d))
    kc = np.repeat(kb, B, axis=0)
    q = np.tile(kb[3], (n, 1))
    z = kb @ kb[3] / math.sqrt(d)
    ref = np.exp(z - z.max()) / np.exp(z - z.max()).sum()
    np.testing.assert_allclose(O.pooled_estimate(q, kc, B, b), ref, rtol=1e-13)


# ---------------------------------------------------------------- worked examples (PE, JSD)
def _pe_worked_inputs(fx):
    """Block-structured Q and K of the PE worked example: the key block means are e_K and
    the query block means a_I with a_I[K] = 2 ln w[I][K] (K <= I), 2 ln 1000 (K > I); rows
    inside a block differ by +-0.5 / +-0.25 along another axis, so only a block *mean*
    gives those vectors."""
    nb, B, d = len(fx["w"]), fx["B"], fx["d"]
    c = np.array([0.5, -0.5, 0.25, -0.25])
    assert B == c.size and d == nb
    k = np.zeros((nb * B, d))
    q = np.zeros((nb * B, d))
    for blk in range(nb):
        a = np.full(d, 2 * math.log(1000.0))
        a[: blk + 1] = [2 * math.log(x) for x in fx["w"][blk]]
        for r in range(B):
            k[blk * B + r, blk] = 1.0
            k[blk * B + r, (blk + 1) % d] += c[r]
            q[blk * B + r] = a
            q[blk * B + r, (blk + 2) % d] += c[r]
    return q, k


def test_pe_index_worked_example():
    """PEIndex ("Method step details" step 3; Algorithm 4) on a case worked by hand in
    tests/golden/pe_index_worked.json: block-mean pooling, the 1/sqrt(d) scale, the causal
    block softmax, v = A_bar / N_b, the gamma-cumsum cut with flat-index ties, and the
    diagonal rescue of an emptied row."""
    from fractions import Fraction
    fx = json.load(open(os.path.join(GOLD, "pe_index_worked.json")))
    q, k = _pe_worked_inputs(fx)
    nb = len(fx["w"])
    # closed form of A_bar from the weights (exact fractions), and the fixture's copy
    exact = np.zeros((nb, nb))
    for I, row in enumerate(fx["w"]):
        for K, x in enumerate(row):
            exact[I, K] = float(Fraction(x, sum(row)))
    np.testing.assert_array_equal(exact, np.array(fx["a_bar"], dtype=float))
    for case in fx["cases"]:
        pe = O.pe_index(q, k, fx["B"], case["gamma"])
        np.testing.assert_allclose(pe["a_bar"], exact, rtol=0, atol=1e-13)
        np.testing.assert_allclose(pe["v"], exact / nb, rtol=0, atol=1e-13)
        rows = [np.nonzero(pe["mask"][I])[0].tolist() for I in range(nb)]
        assert rows == case["rows"], case["gamma"]
        assert pe["n_selected"] == case["n_selected"]
        assert abs(pe["v_star"] - case["v_star"]) < 1e-13
        assert pe["rescued_rows"].tolist() == case["rescued_rows"]


def test_jsd_route_worked_example():
    """FlexPrefill's JSD routing ("Prerequisites", JSD) on a two-block case worked by hand
    in tests/golden/jsd_route_worked.json: a_hat is the causal proxy attention averaged over
    its rows and pooled by key block (the vertical score, not the slash score), a_bar the
    softmax of the mean proxy query against the key block means, D_JS in nats."""
    from fractions import Fraction
    fx = json.load(open(os.path.join(GOLD, "jsd_route_worked.json")))
    n, B, b, d = fx["n"], fx["B"], fx["b"], fx["d"]
    w = fx["w_proxy"]
    k = np.zeros((n, d))
    k[:B, 0] = 1.0
    k[B:, 1] = 1.0
    q = np.zeros((n, d))
    q[: n - b, 0] = 2 * math.log(50.0)
    for r in range(b):
        q[n - b + r, 0] = 2 * math.log(w[r])
    # closed forms: Z_r = 4 w_r + r + 1; a_hat[0] = sum_r w_r / Z_r; a_bar from 72^(1/4)
    a_hat0 = sum(Fraction(wr, 4 * wr + r + 1) for r, wr in enumerate(w))
    a_hat = np.array([float(a_hat0), float(1 - a_hat0)])
    g = math.prod(w) ** 0.25
    a_bar = np.array([g / (g + 1), 1 / (g + 1)])
    m = 0.5 * (a_hat + a_bar)
    d_js = 0.5 * sum(a_hat * np.log(a_hat / m)) + 0.5 * sum(a_bar * np.log(a_bar / m))
    np.testing.assert_allclose(a_hat, fx["a_hat"], rtol=1e-15)
    np.testing.assert_allclose(a_bar, fx["a_bar"], rtol=1e-15)
    assert abs(d_js - fx["d_js"]) < 1e-15
    for case in fx["route_cases"]:
        res = O.jsd_route(q, k, B, b, case["tau"])
        np.testing.assert_allclose(res["a_hat"], a_hat, rtol=1e-13)
        np.testing.assert_allclose(res["a_bar"], a_bar, rtol=1e-13)
        assert abs(res["d_js"] - d_js) < 1e-14
        assert res["route_vs"] == case["route_vs"]

"""Plain, slow CPU oracle (numpy float64) of the CRISP sparse-prefill path.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the benchmark's
CPU-baseline leg may import this module; the product path (the CUDA library and its
Python binding) never does, and this module imports nothing from it.

Source: the analysis page "CRISP: Cliff-awaRe Input-adaptive Sparse Prefilling with
Structural-Mass-Motivated Routing" (paper.rainbus.top/paper/2609.01925).  Citations
below name that page's sections:
  [Prereq]   "Prerequisites" (attention sinks; prefill and sparse attention, the
             formula A(Q,K,V,S) = Softmax(QK^T/sqrt(d) + M_S) V; the gamma-cumsum rule)
  [Core]     "Core method" (PatSearch, C_struct routing, the mass cliff and epsilon)
  [Steps]    "Method step details" (Algorithm 1, steps 1-4 and the default parameters)
  [Alg2] [Alg3] [Alg4]  the descriptions of Algorithms 2 (PatSearch), 3 (VSIndex) and
             4 (PEIndex) under "Figures and tables"

Everything is computed in float64 from the exact bf16 inputs.  Where the page leaves a
point open (the "Method step details" prose and the Algorithm 3 and 4 descriptions name
an operation without fixing its normalisation, direction or tie order), the plainest
reading consistent with the rest of the page is taken and marked "Reading:" beside the
step it affects.

Every function here is pinned by tests in tests/test_oracle_pins.py against closed
forms, special cases, brute force or a worked example; none is "parity unpinned".
"""
import math

import numpy as np

NEG_INF = -np.inf


def bf16_bits_to_f64(u16) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns (uint16) to float64."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def _softmax_rows(logits: np.ndarray) -> np.ndarray:
    m = np.max(logits, axis=-1, keepdims=True)
    e = np.exp(logits - m)
    return e / np.sum(e, axis=-1, keepdims=True)


# --------------------------------------------------------------------------------------
# Step 1: PatSearch proxy attention [Core] step 1, [Steps] step 1, [Alg2]
# --------------------------------------------------------------------------------------
def proxy_attention(q: np.ndarray, k: np.ndarray, b: int) -> np.ndarray:
    """A_hat = Softmax(Q_hat K^T / sqrt(d)) with Q_hat = Q[-b:]  -> [b, n].

    Reading: the proxy softmax is causal, i.e. proxy row r (absolute position n-b+r)
    sees keys j <= n-b+r, as every workload is causal prefill [Prereq].
    """
    n, d = k.shape
    q_hat = q[n - b:]
    logits = (q_hat @ k.T) / math.sqrt(d)
    pos = n - b + np.arange(b)
    logits[np.arange(n)[None, :] > pos[:, None]] = NEG_INF
    return _softmax_rows(logits)


def vertical_score(a_hat: np.ndarray) -> np.ndarray:
    """a_v[j] = (1/b) sum_r A_hat[r, j]: the column mean [Alg3]."""
    return a_hat.sum(axis=0) / a_hat.shape[0]


def slash_score(a_hat: np.ndarray) -> np.ndarray:
    """a_s[delta] = (1/b) sum_r A_hat[r, p_r - delta], p_r = n-b+r  [Alg3].

    Reading: delta is query position minus key position (delta = 0 is the main
    diagonal), and the diagonal "mean" divides by b like the column mean, so that
    sum(a_s) = sum(a_v) = 1.  Terms with p_r - delta < 0 are absent.
    """
    b, n = a_hat.shape
    a_s = np.zeros(n)
    for r in range(b):
        p = n - b + r
        a_s[: p + 1] += a_hat[r, p::-1]
    return a_s / b


def anchor_set(n: int, w_sink: int, w_local: int) -> np.ndarray:
    """S_anchor: the first w_sink and the last w_local key positions (their union)."""
    idx = np.zeros(n, dtype=bool)
    idx[: min(w_sink, n)] = True
    idx[max(n - w_local, 0):] = True
    return idx


def c_struct_from_av(a_v: np.ndarray, w_sink: int, w_local: int) -> float:
    """C_struct = (1/b) sum_i sum_{j in S_anchor} A_hat[i, j] = sum_{j in S_anchor} a_v[j]
    [Core] step 1, [Alg2]."""
    return float(a_v[anchor_set(a_v.shape[0], w_sink, w_local)].sum())


def route_is_vs(c_struct: float, tau_proxy: float) -> bool:
    """VS iff C_struct >= tau_proxy, else PE [Core] step 1, [Alg2]."""
    return bool(c_struct >= tau_proxy)


# --------------------------------------------------------------------------------------
# Step 2: VSIndex, the sink-aware noise floor [Steps] step 2, [Alg3], [Core] innovation 2
# --------------------------------------------------------------------------------------
def block_pool(score: np.ndarray, B: int) -> np.ndarray:
    """p_d[J] = sum of score over block J.  Reading: pooling is a sum (so sum(p_d) = 1,
    which the floor r_d = 1 - p_d[0] - p_d[N_b-1] presumes)."""
    return score.reshape(-1, B).sum(axis=1)


def noise_floor(p: np.ndarray) -> float:
    """mu_d = max(1 - p_d[0] - p_d[N_b-1], 0) / (N_b - 2)  [Alg3].

    Reading: with N_b <= 2 there is no non-anchor block; mu = 0 (every block passes).
    """
    nb = p.shape[0]
    if nb <= 2:
        return 0.0
    r = max(1.0 - p[0] - p[nb - 1], 0.0)
    return r / (nb - 2)


def noise_floor_median(p: np.ndarray) -> float:
    """Variant floor: the median of the non-anchor block scores p_d[1..N_b-2] instead of
    their mean ("Limitations" item 6 and "Weaknesses" item 4: the mean floor can be lifted
    by one dominant block; the median variant changes accuracy by about 0.7 pp).

    Reading: the median of an even count is the mean of the two middle values; with
    N_b <= 2 there is no non-anchor block and mu = 0, as for the mean floor.
    """
    nb = p.shape[0]
    if nb <= 2:
        return 0.0
    return float(np.median(p[1:nb - 1]))


def topk_desc(p: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest values, ties broken toward the lower index; sorted."""
    order = np.lexsort((np.arange(p.shape[0]), -p))
    return np.sort(order[:k])


def select_above_floor(p: np.ndarray, alpha: float, mu: float, kmin_blocks: int):
    """Blocks with p_d[J] > alpha*mu_d, their count clipped to [k_min, N_b]  [Alg3].

    Reading: the clip keeps the top-k_d blocks by p_d, k_d = clip(c_d, k_min, N_b);
    when c_d >= k_min that is exactly {J: p_d[J] > alpha*mu_d}.
    Returns (sorted block indices, c_d, k_d).
    """
    nb = p.shape[0]
    c = int(np.count_nonzero(p > alpha * mu))
    kd = min(max(c, kmin_blocks), nb)
    return topk_desc(p, kd), c, kd


def select_gamma_cumsum(p: np.ndarray, gamma: float, kmin_blocks: int):
    """FlexPrefill's VS budget as the page describes it ("Prerequisites", cumulative
    coverage; "Novelty" and Table 5, ablation Abl.1 = C_struct routing with this rule):
    the smallest set of blocks, largest first, whose scores reach gamma, padded to the
    minimum budget k_min.  Returns (sorted block indices, cut size, k_d)."""
    nb = p.shape[0]
    cut = gamma_cut(p, gamma).size
    kd = min(max(cut, kmin_blocks), nb)
    return topk_desc(p, kd), cut, kd


def kmin_blocks(k_min_tokens: int, B: int) -> int:
    """k_min of 1024 tokens is 8 blocks of 128 per direction [Steps]."""
    return -(-k_min_tokens // B)


def vs_index(a_hat: np.ndarray, B: int, alpha: float, k_min_tokens: int, floor: str = "mean",
             vs_rule: str = "floor", gamma: float = 0.95) -> dict:
    """Algorithm 3: vertical and slash scores, pooled, floored and selected.

    floor="median" uses noise_floor_median; vs_rule="gamma" replaces the floor rule by the
    gamma-cumsum budget (select_gamma_cumsum), mu is then still reported.
    """
    a_v = vertical_score(a_hat)
    a_s = slash_score(a_hat)
    p_v = block_pool(a_v, B)
    p_s = block_pool(a_s, B)
    kmb = kmin_blocks(k_min_tokens, B)
    fl = noise_floor_median if floor == "median" else noise_floor
    mu_v, mu_s = fl(p_v), fl(p_s)
    if vs_rule == "gamma":
        S_v, c_v, k_v = select_gamma_cumsum(p_v, gamma, kmb)
        S_s, c_s, k_s = select_gamma_cumsum(p_s, gamma, kmb)
    else:
        S_v, c_v, k_v = select_above_floor(p_v, alpha, mu_v, kmb)
        S_s, c_s, k_s = select_above_floor(p_s, alpha, mu_s, kmb)
    return dict(a_v=a_v, a_s=a_s, p_v=p_v, p_s=p_s, mu_v=mu_v, mu_s=mu_s,
                S_v=S_v, S_s=S_s, c_v=c_v, c_s=c_s, k_v=k_v, k_s=k_s, kmin_blocks=kmb)


def vs_block_mask(S_v: np.ndarray, S_s: np.ndarray, nb: int) -> np.ndarray:
    """Key blocks per query block for a VS head: S_v u S_s u {0, N_b-1}  [Alg3].

    Reading: a vertical block K is a key block (kept for query blocks I >= K); a slash
    block J is the block diagonal at distance J (key block I-J for query block I); the
    two anchors are the sink (key block 0) and the local window, i.e. the diagonal key
    block I of every query block (slash block 0; vertical block N_b-1 is the last query
    block's diagonal).  Returns a bool [N_b, N_b] lower-triangular mask.
    """
    m = np.zeros((nb, nb), dtype=bool)
    I = np.arange(nb)
    for K in S_v:
        m[K:, K] = True
    for J in S_s:
        rows = I[I >= J]
        m[rows, rows - J] = True
    m[:, 0] = True
    m[I, I] = True
    return np.tril(m)


# --------------------------------------------------------------------------------------
# Step 3: PEIndex, pooled estimate and gamma-cumsum [Steps] step 3, [Alg4], [Prereq]
# --------------------------------------------------------------------------------------
def block_mean(x: np.ndarray, B: int) -> np.ndarray:
    """Mean of each block of B rows -> [N_b, d]."""
    n, d = x.shape
    return x.reshape(n // B, B, d).mean(axis=1)


def gamma_cut(values: np.ndarray, gamma: float) -> np.ndarray:
    """The smallest set of items whose values sum to >= gamma, taken largest first.

    Accumulate the scores sorted in descending order (ties: lower index first) and stop
    at the first prefix whose running sum reaches gamma [Prereq] (the cumulative
    coverage rule) and [Alg4].  If the whole sum stays below gamma every item is taken.
    Returns the selected indices, sorted.
    """
    order = np.lexsort((np.arange(values.shape[0]), -values))
    csum = np.cumsum(values[order])
    hit = np.nonzero(csum >= gamma)[0]
    cnt = int(hit[0]) + 1 if hit.size else values.shape[0]
    return np.sort(order[:cnt])


def pe_index(q: np.ndarray, k: np.ndarray, B: int, gamma: float) -> dict:
    """Algorithm 4: pool all queries and keys by block, causal block softmax, normalise,
    flatten, gamma-cumsum.

    Reading: A_bar[I, K] = softmax over K <= I of (Qbar_I . Kbar_K / sqrt(d)) (block
    means; the diagonal pair uses the full-block means); "normalise" divides by N_b so
    the flattened scores v sum to 1; pairs are flattened with index I*N_b + K (ties in
    v go to the lower flat index).  A query block left with no pair by the cut gets its
    diagonal pair (I, I) so that its output is defined ("rescued").
    """
    n, d = q.shape
    nb = n // B
    qb, kb = block_mean(q, B), block_mean(k, B)
    logits = (qb @ kb.T) / math.sqrt(d)
    tri = np.tril(np.ones((nb, nb), dtype=bool))
    logits[~tri] = NEG_INF
    a_bar = _softmax_rows(logits)
    v_full = a_bar / nb
    I, K = np.nonzero(tri)                 # row-major: flat index I*nb+K increasing
    v = v_full[I, K]
    sel = gamma_cut(v, gamma)
    mask = np.zeros((nb, nb), dtype=bool)
    mask[I[sel], K[sel]] = True
    v_star = float(v[sel].min()) if sel.size else float("inf")
    empty_rows = ~mask.any(axis=1)
    mask[np.arange(nb), np.arange(nb)] = True
    return dict(a_bar=a_bar, v=v_full, mask=mask, v_star=v_star, n_selected=int(sel.size),
                rescued_rows=np.nonzero(empty_rows)[0])


# --------------------------------------------------------------------------------------
# Step 4: exact attention over the selected blocks [Prereq] A(Q,K,V,S), [Steps] step 4
# --------------------------------------------------------------------------------------
def block_sparse_attention(q, k, v, mask: np.ndarray, B: int, blocks=None) -> np.ndarray:
    """O_i = sum_{j in S(i), j <= i} softmax_j(q_i . k_j / sqrt(d)) v_j, where S(i) is the
    union of the key blocks mask[I] of i's query block I; token-causal within blocks.

    Returns the output rows of the requested query blocks ([len(blocks)*B, d]).
    """
    n, d = q.shape
    nb = n // B
    blocks = range(nb) if blocks is None else blocks
    out = []
    for I in blocks:
        kb = np.nonzero(mask[I, : I + 1])[0]
        keys = (kb[:, None] * B + np.arange(B)[None, :]).reshape(-1)
        qi = q[I * B:(I + 1) * B]
        logits = (qi @ k[keys].T) / math.sqrt(d)
        qpos = I * B + np.arange(B)
        logits[keys[None, :] > qpos[:, None]] = NEG_INF
        out.append(_softmax_rows(logits) @ v[keys])
    return np.concatenate(out, axis=0) if out else np.zeros((0, d))


# --------------------------------------------------------------------------------------
# Algorithm 1 per head [Steps], [Alg1 under "Figures and tables"]
# --------------------------------------------------------------------------------------
def crisp_select_head(q, k, B=128, b=128, w_sink=128, w_local=128, tau_proxy=0.2,
                      alpha=1.0, gamma=0.95, k_min_tokens=1024, force=None, floor="mean",
                      vs_rule="floor") -> dict:
    """PatSearch -> VSIndex or PEIndex for one query head (fp64 inputs [n, d]).

    force: None, "vs" or "pe" overrides the route (the C_struct value is still computed).
    floor / vs_rule: the median-floor and gamma-cumsum VS variants (see vs_index).
    """
    n = k.shape[0]
    nb = n // B
    a_hat = proxy_attention(q, k, b)
    a_v = vertical_score(a_hat)
    c = c_struct_from_av(a_v, w_sink, w_local)
    is_vs = route_is_vs(c, tau_proxy) if force is None else (force == "vs")
    res = dict(c_struct=c, route_vs=is_vs, n_blocks=nb)
    if is_vs:
        vs = vs_index(a_hat, B, alpha, k_min_tokens, floor=floor, vs_rule=vs_rule, gamma=gamma)
        res.update(vs)
        res["mask"] = vs_block_mask(vs["S_v"], vs["S_s"], nb)
    else:
        pe = pe_index(q, k, B, gamma)
        res.update(pe)
    return res


def crisp_head(q, k, v, blocks=None, **params) -> dict:
    """Selection plus attention output rows for one head."""
    sel = crisp_select_head(q, k, **params)
    sel["out"] = block_sparse_attention(q, k, v, sel["mask"], params.get("B", 128), blocks)
    return sel


def workload_params(w) -> dict:
    """The method parameters of a workload description (B, b, windows, tau, alpha, ...)."""
    return dict(B=w.B, b=w.b, w_sink=w.w_sink, w_local=w.w_local, tau_proxy=w.tau_proxy,
                alpha=w.alpha, gamma=w.gamma, k_min_tokens=w.k_min_tokens,
                floor=getattr(w, "vs_floor", "mean"), vs_rule=getattr(w, "vs_rule", "floor"))


def kl_divergence(x: np.ndarray, y: np.ndarray) -> float:
    """KL(x || y) = sum x log(x / y) in nats, with 0 log 0 = 0."""
    nz = x > 0
    return float(np.sum(x[nz] * np.log(x[nz] / y[nz])))


def js_divergence(x: np.ndarray, y: np.ndarray) -> float:
    """D_JS = 1/2 KL(x || m) + 1/2 KL(y || m), m = (x + y)/2  ("Prerequisites", JSD)."""
    m = 0.5 * (x + y)
    return 0.5 * kl_divergence(x, m) + 0.5 * kl_divergence(y, m)


def pooled_estimate(q: np.ndarray, k: np.ndarray, B: int, b: int) -> np.ndarray:
    """a_bar, the "pool first, then softmax" distribution over key blocks ("Prerequisites",
    JSD): the mean of the last b queries against the block means of the keys, softmax over
    the N_b blocks.  Reading: the pooled query stands for the last query block, which sees
    every key block; the logits are scaled by 1/sqrt(d) like the attention's."""
    n, d = k.shape
    qbar = q[n - b:].mean(axis=0)
    logits = block_mean(k, B) @ qbar / math.sqrt(d)
    return _softmax_rows(logits[None, :])[0]


def jsd_route(q: np.ndarray, k: np.ndarray, B: int, b: int, tau_jsd: float) -> dict:
    """FlexPrefill's JSD routing, the signal C_struct replaces ("Prerequisites", JSD;
    "Motivation"): a_hat = the proxy attention averaged over its b queries and pooled by
    key block (p_v), a_bar = pooled_estimate; VS iff D_JS(a_hat, a_bar) >= tau_jsd."""
    p_v = block_pool(vertical_score(proxy_attention(q, k, b)), B)
    a_bar = pooled_estimate(q, k, B, b)
    dj = js_divergence(p_v, a_bar)
    return dict(d_js=dj, route_vs=bool(dj >= tau_jsd), a_hat=p_v, a_bar=a_bar)


def mass_cliff_epsilon(n: int, k: int, delta: float) -> float:
    """Background-token mass of one softmax row with k signal logits delta and n-k zero
    logits: e^-delta / (k + (n-k) e^-delta)  [Core] innovation 2."""
    e = math.exp(-delta)
    return e / (k + (n - k) * e)

"""Plants mistakes in a copy of the oracle and checks that its pins catch each one.

A pin that still passes when the oracle computes something else pins nothing.  Each case
rewrites one step of a fresh copy of oracle/crisp_oracle.py, built from its source text
(the oracle itself is never modified), points the pin tests at the copy, and requires at
least one of the pins named for that step to fail.  The unmodified copy must pass the
same pins, so a broken harness cannot pass for a caught mistake.  Sections cited are those
of the analysis page "CRISP: Cliff-awaRe Input-adaptive Sparse Prefilling with
Structural-Mass-Motivated Routing" (paper.rainbus.top).
"""
import pathlib
import types

import pytest

from oracle import crisp_oracle as O

import tests.test_oracle_pins as pins

SRC = pathlib.Path(O.__file__).read_text()


def _copy(text):
    mod = types.ModuleType("crisp_oracle_copy")
    mod.__file__ = O.__file__
    exec(compile(text, O.__file__, "exec"), mod.__dict__)
    return mod


def _pin(name, *args):
    return (name, args)


# (case, text in the oracle, replacement, pins that must catch it)
MUTATIONS = [
    # "Figures and tables", Algorithm 4: pooled logits scaled by 1/sqrt(d)
    ("pe_index without 1/sqrt(d)",
     "    logits = (qb @ kb.T) / math.sqrt(d)\n", "    logits = (qb @ kb.T)\n",
     [_pin("test_pe_index_worked_example")]),
    # Algorithm 4: queries pooled by block mean
    ("pe_index pools Q by sum",
     "    qb, kb = block_mean(q, B), block_mean(k, B)\n",
     "    qb, kb = block_mean(q, B) * B, block_mean(k, B)\n",
     [_pin("test_pe_index_worked_example")]),
    # Algorithm 4: normalise by N_b
    ("pe_index without the 1/N_b normalisation",
     "    v_full = a_bar / nb\n", "    v_full = a_bar\n",
     [_pin("test_pe_index_worked_example"), _pin("test_pe_scores_normalised")]),
    # reading: an emptied query row gets its diagonal pair
    ("pe_index without the diagonal rescue",
     "    mask[np.arange(nb), np.arange(nb)] = True\n", "",
     [_pin("test_pe_index_worked_example")]),
    # "Prerequisites", JSD: a_hat is the row-averaged proxy attention pooled by key block
    ("jsd_route on the slash score",
     "    p_v = block_pool(vertical_score(proxy_attention(q, k, b)), B)\n",
     "    p_v = block_pool(slash_score(proxy_attention(q, k, b)), B)\n",
     [_pin("test_jsd_route_worked_example")]),
    # "Prerequisites", cumulative coverage: ties of the gamma cut go to the lower index
    ("gamma_cut ties to the higher index",
     "    order = np.lexsort((np.arange(values.shape[0]), -values))\n",
     "    order = np.lexsort((-np.arange(values.shape[0]), -values))\n",
     [_pin("test_gamma_cut_bruteforce", s) for s in range(5)]
     + [_pin("test_pe_index_worked_example")]),
    # "Core method" step 1: the proxy softmax is causal
    ("proxy_attention not causal",
     "    logits[np.arange(n)[None, :] > pos[:, None]] = NEG_INF\n", "",
     [_pin("test_proxy_uniform_logits_closed_form", 1024, 128),
      _pin("test_slash_and_vertical_index_direction")]),
    # Algorithm 3: the slash score indexes by query minus key position
    ("slash_score indexed by key position",
     "        a_s[: p + 1] += a_hat[r, p::-1]\n", "        a_s[: p + 1] += a_hat[r, : p + 1]\n",
     [_pin("test_slash_and_vertical_index_direction"),
      _pin("test_proxy_uniform_logits_closed_form", 1024, 128)]),
    # Algorithm 3: the noise floor excludes the two anchor blocks
    ("noise_floor over all blocks",
     "    return r / (nb - 2)\n", "    return r / nb\n",
     [_pin("test_vs_select_worked_example"), _pin("test_noise_floor_closed_form_from_c_struct")]),
    # Algorithm 3: blocks strictly above alpha * mu
    ("select_above_floor with >=",
     "    c = int(np.count_nonzero(p > alpha * mu))\n",
     "    c = int(np.count_nonzero(p >= alpha * mu))\n",
     [_pin("test_vs_select_threshold_is_strict"), _pin("test_vs_select_worked_example")]),
    # Algorithm 2: VS iff C_struct >= tau_proxy
    ("route with > instead of >=",
     "    return bool(c_struct >= tau_proxy)", "    return bool(c_struct > tau_proxy)",
     [_pin("test_route_at_threshold_is_vs")]),
    # Algorithm 3: the floor is clamped at zero
    ("noise_floor without the clamp at zero",
     "    r = max(1.0 - p[0] - p[nb - 1], 0.0)", "    r = 1.0 - p[0] - p[nb - 1]",
     [_pin("test_noise_floor_clamps_at_zero")]),
    # reading: k_min tokens are at least ceil(k_min / B) blocks
    ("kmin_blocks rounded down",
     "    return -(-k_min_tokens // B)", "    return k_min_tokens // B",
     [_pin("test_kmin_blocks")]),
    # "Prerequisites", cumulative coverage: stop when the sum reaches gamma (>=)
    ("gamma_cut needs the sum above gamma",
     "    hit = np.nonzero(csum >= gamma)[0]", "    hit = np.nonzero(csum > gamma)[0]",
     [_pin("test_gamma_cut_stops_when_the_sum_reaches_gamma")]),
    # "Core method" step 1: S_anchor is the first w_sink and the last w_local keys
    ("anchor set without the local window",
     "    idx[max(n - w_local, 0):] = True\n", "",
     [_pin("test_scores_sum_to_one_and_anchor_slice"),
      _pin("test_proxy_uniform_logits_closed_form", 1024, 128)]),
    ("anchor set without the sink",
     "    idx[: min(w_sink, n)] = True\n", "",
     [_pin("test_scores_sum_to_one_and_anchor_slice"),
      _pin("test_proxy_uniform_logits_closed_form", 1024, 128)]),
    # Algorithm 3: the vertical score is the column mean
    ("vertical_score as a column sum",
     "    return a_hat.sum(axis=0) / a_hat.shape[0]", "    return a_hat.sum(axis=0)",
     [_pin("test_proxy_uniform_logits_closed_form", 1024, 128)]),
    # reading: the diagonal mean divides by b
    ("slash_score divided by n",
     "    return a_s / b\n", "    return a_s / n\n",
     [_pin("test_slash_and_vertical_index_direction"),
      _pin("test_scores_sum_to_one_and_anchor_slice")]),
    # reading: block pooling is a sum
    ("block_pool as a mean",
     "    return score.reshape(-1, B).sum(axis=1)", "    return score.reshape(-1, B).mean(axis=1)",
     [_pin("test_mass_cliff_epsilon_closed_form", 4096, 6, 12.0),
      _pin("test_noise_floor_closed_form_from_c_struct")]),
    # Algorithm 3: the count is clipped to [k_min, N_b]
    ("select_above_floor without the N_b clip",
     "    kd = min(max(c, kmin_blocks), nb)\n    return topk_desc(p, kd), c, kd",
     "    kd = max(c, kmin_blocks)\n    return topk_desc(p, kd), c, kd",
     [_pin("test_vs_select_bruteforce_and_invariants", s) for s in range(6)]),
    # reading: top-k padding ties go to the lower block index
    ("topk_desc ties to the higher index",
     "    order = np.lexsort((np.arange(p.shape[0]), -p))",
     "    order = np.lexsort((-np.arange(p.shape[0]), -p))",
     [_pin("test_vs_select_threshold_is_strict"), _pin("test_vs_select_worked_example")]),
    # Algorithm 3: the union keeps key block 0 and the diagonal of every query block
    ("vs_block_mask without the sink column",
     "    m[:, 0] = True\n", "",
     [_pin("test_vs_block_mask_worked_example")]),
    ("vs_block_mask slash block read forward",
     "        m[rows, rows - J] = True", "        m[rows, np.minimum(rows + J, nb - 1)] = True",
     [_pin("test_vs_block_mask_worked_example")]),
    # "Limitations" item 6: the median floor is over the non-anchor blocks
    ("noise_floor_median over all blocks",
     "    return float(np.median(p[1:nb - 1]))", "    return float(np.median(p))",
     [_pin("test_median_floor_bruteforce", s) for s in range(4)]),
    # Abl.1: the gamma-cumsum budget is padded to k_min
    ("select_gamma_cumsum without k_min",
     "    kd = min(max(cut, kmin_blocks), nb)", "    kd = cut",
     [_pin("test_vs_variants_worked_example")]),
    # "Algorithm 4": the PE block softmax is causal
    ("pe_index without the causal block mask",
     "    logits[~tri] = NEG_INF\n", "",
     [_pin("test_pe_uniform_pooled_scores_closed_form")]),
    # "Prerequisites", JSD: m = (x + y) / 2, logs in nats; a_bar from the last b queries
    ("js_divergence against max(x, y)",
     "    m = 0.5 * (x + y)", "    m = np.maximum(x, y)",
     [_pin("test_js_divergence_closed_forms")]),
    ("kl_divergence in bits",
     "    return float(np.sum(x[nz] * np.log(x[nz] / y[nz])))",
     "    return float(np.sum(x[nz] * np.log2(x[nz] / y[nz])))",
     [_pin("test_js_divergence_closed_forms")]),
    ("pooled_estimate over all queries",
     "    qbar = q[n - b:].mean(axis=0)", "    qbar = q.mean(axis=0)",
     [_pin("test_jsd_route_worked_example")]),
    ("pooled_estimate without 1/sqrt(d)",
     "    logits = block_mean(k, B) @ qbar / math.sqrt(d)", "    logits = block_mean(k, B) @ qbar",
     [_pin("test_pooled_estimate_special_cases")]),
    # "Core method" step 1: the proxy queries are the last b rows
    ("proxy_attention on the first b rows",
     "    q_hat = q[n - b:]", "    q_hat = q[:b]",
     [_pin("test_jsd_route_worked_example")]),
    # "Prerequisites", A(Q,K,V,S): token-causal inside the diagonal block
    ("block_sparse_attention not causal inside a block",
     "        logits[keys[None, :] > qpos[:, None]] = NEG_INF\n", "",
     [_pin("test_all_blocks_equals_dense_causal_sdpa", 512, 16, 128)]),
    # "Prerequisites", A(Q,K,V,S): attention logits scaled by 1/sqrt(d)
    ("block_sparse_attention without 1/sqrt(d)",
     "        logits = (qi @ k[keys].T) / math.sqrt(d)\n", "        logits = (qi @ k[keys].T)\n",
     [_pin("test_all_blocks_equals_dense_causal_sdpa", 512, 16, 128)]),
]


def _run(mod, pin_list, monkeypatch):
    """Runs the pins against `mod`; returns the names of those that failed."""
    monkeypatch.setattr(pins, "O", mod)
    failed = []
    for name, args in pin_list:
        try:
            getattr(pins, name)(*args)
        except AssertionError:
            failed.append(name)
    return failed


@pytest.mark.parametrize("case,old,new,pin_list", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(case, old, new, pin_list, monkeypatch):
    assert SRC.count(old) == 1, f"{case}: the text to replace is not in the oracle once"
    assert _run(_copy(SRC), pin_list, monkeypatch) == [], f"{case}: the unmodified copy fails"
    failed = _run(_copy(SRC.replace(old, new)), pin_list, monkeypatch)
    assert failed, f"{case}: no pin caught the planted mistake"

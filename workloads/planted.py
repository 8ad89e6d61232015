"""Seeded planted Q/K/V generator (synthetic stand-in for real-model activations).

The CRISP analysis page ("CRISP: Cliff-awaRe Input-adaptive Sparse Prefilling with
Structural-Mass-Motivated Routing", paper.rainbus.top) measures on real Llama/Qwen
activations. Those are not available, so every workload here is synthetic, seeded, and
planted with the structures the page describes (section "Prerequisites", attention
sinks and the VS/PE dichotomy; section "Core method", the mass cliff):

* base entries of Q, K and V are N(0,1)/sqrt(d);
* dimension 0 is the shared sink direction u.  With sigma = d**0.25, adding a*sigma*e to
  a query and c*sigma*e to a key adds exactly a*c to the logit q.k/sqrt(d), so the
  sink (all VS queries and keys 0..127 scaled by s) adds s*s logits (16 for s=4,
  25 for s=5);
* dimensions 1..7 carry needles: query head slot r of a KV group gets +4*sigma*e_{1+r},
  and the keys of each of its needle blocks get +3*sigma*e_{1+r} (+12 logits).  Needle
  blocks are distinct, uniform in [2, N_b-3];
* dimensions 64..127 carry a locality term: 32 rotary pairs with seeded frequencies
  omega_m ~ U(0, pi/256]; query i and key j get sqrt(L/M)*sigma*(cos, sin)(omega_m*pos),
  which adds (L/M) * sum_m cos(omega_m (i-j)) logits: L=2 at i=j, a main lobe of a
  few hundred tokens and a small far-field ripple;
* diffuse (PE-planted) query heads have all planted dimensions zero and dimensions
  8..63 drawn N(0, sigma_q^2) with sigma_q = 0.3*d/sqrt(56), i.e. logit std 0.3.

Values are produced in float32 and rounded to bfloat16 (round to nearest even) exactly
once; the bf16 bit patterns (uint16) are what both the oracle and the GPU path consume.
Every (tensor, head) pair draws from its own seed stream, so any head can be generated
alone and the result does not depend on the thread count.

This module holds no arithmetic of the method: it only makes inputs.
"""
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .configs import Workload

_T_Q, _T_K, _T_V, _T_PARAM = 1, 2, 3, 4
_LOC_PAIRS = 32          # M
_LOC_GAIN = 2.0          # L
_LOC_DIM0 = 64
_PE_DIM0, _PE_DIM1 = 8, 64


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(w: Workload, tid: int, head: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, tid, head])))


def plant_params(w: Workload) -> dict:
    """Per-head needle blocks and per-group locality frequencies (seeded)."""
    g = w.group
    nb = w.n_blocks
    pe = set(w.pe_heads)
    needles = {}
    for h in range(w.hq):
        if h in pe:
            needles[h] = np.zeros(0, dtype=np.int64)
            continue
        r = _rng(w, _T_PARAM, h)
        if w.needles[0] == "fixed":
            cnt = int(w.needles[1])
        else:
            cnt = int(r.integers(w.needles[1], w.needles[2] + 1))
        lo, hi = 2, nb - 3
        avail = max(hi - lo + 1, 0)
        cnt = min(cnt, avail)
        needles[h] = np.sort(r.choice(np.arange(lo, hi + 1), size=cnt, replace=False)) if cnt else \
            np.zeros(0, dtype=np.int64)
    omega = {}
    for hk in range(w.hkv):
        r = _rng(w, _T_PARAM, 10_000 + hk)
        omega[hk] = (1.0 - r.random(_LOC_PAIRS)) * (math.pi / 256.0)
    assert g <= 7, "needle directions use dims 1..7"
    return {"needles": needles, "omega": omega}


def _locality(w: Workload, omega: np.ndarray) -> np.ndarray:
    """[n, 64] float32 rotary locality rows (cos, sin interleaved per pair)."""
    sigma = w.d ** 0.25
    c = math.sqrt(_LOC_GAIN / _LOC_PAIRS) * sigma
    pos = np.arange(w.n, dtype=np.float64)[:, None]
    ang = pos * omega[None, :]
    out = np.empty((w.n, 2 * _LOC_PAIRS), dtype=np.float64)
    out[:, 0::2] = c * np.cos(ang)
    out[:, 1::2] = c * np.sin(ang)
    return out.astype(np.float32)


def _base(w: Workload, tid: int, head: int) -> np.ndarray:
    a = np.empty((w.n, w.d), dtype=np.float32)
    _rng(w, tid, head).standard_normal(out=a, dtype=np.float32)
    a *= np.float32(1.0 / math.sqrt(w.d))
    return a


def gen_q_head(w: Workload, h: int, params: dict = None, loc_cache: dict = None) -> np.ndarray:
    params = params or plant_params(w)
    sigma = np.float32(w.d ** 0.25)
    if h in set(w.pe_heads):
        q = np.zeros((w.n, w.d), dtype=np.float32)
        sq = 0.3 * w.d / math.sqrt(_PE_DIM1 - _PE_DIM0)
        z = np.empty((w.n, _PE_DIM1 - _PE_DIM0), dtype=np.float32)
        _rng(w, _T_Q, h).standard_normal(out=z, dtype=np.float32)
        q[:, _PE_DIM0:_PE_DIM1] = z * np.float32(sq)
        return f32_to_bf16_bits(q)
    q = _base(w, _T_Q, h)
    hk, slot = h // w.group, h % w.group
    q[:, 0] += np.float32(w.sink_scale) * sigma
    q[:, 1 + slot] += np.float32(4.0) * sigma
    loc = (loc_cache or {}).get(hk)
    if loc is None:
        loc = _locality(w, params["omega"][hk])
    q[:, _LOC_DIM0:] += loc
    return f32_to_bf16_bits(q)


def gen_k_head(w: Workload, hk: int, params: dict = None, loc_cache: dict = None) -> np.ndarray:
    params = params or plant_params(w)
    sigma = np.float32(w.d ** 0.25)
    k = _base(w, _T_K, hk)
    k[: min(128, w.n), 0] += np.float32(w.sink_scale) * sigma
    for slot in range(w.group):
        h = hk * w.group + slot
        for blk in params["needles"][h]:
            k[blk * w.B:(blk + 1) * w.B, 1 + slot] += np.float32(3.0) * sigma
    loc = (loc_cache or {}).get(hk)
    if loc is None:
        loc = _locality(w, params["omega"][hk])
    k[:, _LOC_DIM0:] += loc
    return f32_to_bf16_bits(k)


def gen_v_head(w: Workload, hk: int) -> np.ndarray:
    return f32_to_bf16_bits(_base(w, _T_V, hk))


def generate(w: Workload, q_heads=None, kv_heads=None, threads: int = None) -> dict:
    """Generate bf16 bit patterns.

    Returns {"q": [len(q_heads), n, d] uint16, "k": [len(kv_heads), n, d], "v": ...,
    "q_heads", "kv_heads", "params"}.  Defaults: all heads.
    """
    q_heads = list(range(w.hq)) if q_heads is None else list(q_heads)
    kv_heads = list(range(w.hkv)) if kv_heads is None else list(kv_heads)
    params = plant_params(w)
    threads = threads or min(32, os.cpu_count() or 1)
    q = np.empty((len(q_heads), w.n, w.d), dtype=np.uint16)
    k = np.empty((len(kv_heads), w.n, w.d), dtype=np.uint16)
    v = np.empty((len(kv_heads), w.n, w.d), dtype=np.uint16)
    need_loc = sorted({h // w.group for h in q_heads} | set(kv_heads))
    with ThreadPoolExecutor(threads) as ex:
        locs = dict(zip(need_loc, ex.map(lambda hk: _locality(w, params["omega"][hk]), need_loc)))

        def fq(i):
            q[i] = gen_q_head(w, q_heads[i], params, locs)

        def fk(i):
            k[i] = gen_k_head(w, kv_heads[i], params, locs)

        def fv(i):
            v[i] = gen_v_head(w, kv_heads[i])

        futs = [ex.submit(fq, i) for i in range(len(q_heads))]
        futs += [ex.submit(fk, i) for i in range(len(kv_heads))]
        futs += [ex.submit(fv, i) for i in range(len(kv_heads))]
        for f in futs:
            f.result()
    return {"q": q, "k": k, "v": v, "q_heads": q_heads, "kv_heads": kv_heads, "params": params}


def random_qkv(n: int, hq: int, hkv: int, d: int, seed: int, scale: float = 1.0) -> dict:
    """Unplanted N(0, scale^2/d) inputs (bf16 bits), for edge-case tests."""
    r = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 99])))

    def mk(h):
        a = r.standard_normal((h, n, d), dtype=np.float32) * np.float32(scale / math.sqrt(d))
        return f32_to_bf16_bits(a)

    return {"q": mk(hq), "k": mk(hkv), "v": mk(hkv)}

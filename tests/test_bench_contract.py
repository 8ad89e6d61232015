"""The bench's reference arm (the fp64 oracle on the host cores) prints one JSON line with
the keys the measurement contract asks for; checked on CPU on the smallest workload."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
         "tiny_n4k", "--steps", "1", "--warmup", "3", "--ref-budget", "2"],
        capture_output=True, text=True, timeout=600, cwd=ROOT, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["higher_is_better"] is False and d["unit"] == "ms/layer"
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny_n4k"
    assert d["config"]["vs_variant"] == "none"   # the GPU arm's config carries the same keys
    assert d["value"] > 0 and d["ms_per_step"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["sample"] and "VS" in cb["sample"] and "PE" in cb["sample"]


def test_algorithmic_flops_counts_causal_token_pairs():
    """The roofline's numerator: every causal (query, key) token pair of a selected block
    pair costs one d-long dot product for Q K^T and one d-long multiply-add row for P V,
    i.e. 4d FLOP ("Prerequisites", A(Q,K,V,S) = Softmax(QK^T/sqrt(d) + M_S) V, causal).
    Brute force over a random lower-triangular block mask that keeps every diagonal."""
    import numpy as np
    import bench
    B, D, nb = bench.B, bench.D, 6
    rng = np.random.default_rng(5)
    mask = np.tril(rng.random((nb, nb)) < 0.5)
    mask[np.arange(nb), np.arange(nb)] = True
    tok = np.arange(nb * B)
    blk = tok // B
    pairs = (tok[None, :] <= tok[:, None]) & mask[blk[:, None], blk[None, :]]
    brute = 4.0 * D * int(pairs.sum())
    assert bench.algorithmic_flops(int(mask.sum()), nb) == brute

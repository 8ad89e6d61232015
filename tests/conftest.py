import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running (large workloads)")


def pytest_terminal_summary(terminalreporter):
    """Per-workload parity reports of the GPU tests (exempt counts, worst errors)."""
    try:
        from tests.parity import REPORTS
    except Exception:  # noqa: BLE001 - the CPU-only environment may lack the GPU modules
        return
    if not REPORTS:
        return
    keys = ("heads", "vs_heads", "pe_heads", "route_mismatch_exempt", "vs_block_exempt",
            "max_vs_exempt_head", "pe_pair_exempt", "max_pe_exempt_head", "max_p_err",
            "max_cstruct_err", "attend_max_abs", "attend_mean_abs", "attend_rel_rms",
            "prefill_heads_compared", "prefill_heads_on_gpu_selection", "near_routes",
            "near_vs_blocks", "near_pe_pairs")
    terminalreporter.section("parity reports")
    for name, rep in REPORTS:
        parts = []
        for k in keys:
            if k in rep:
                v = rep[k]
                parts.append(f"{k}={v:.3g}" if isinstance(v, float) else f"{k}={v}")
        terminalreporter.write_line(f"{name}: " + " ".join(parts))

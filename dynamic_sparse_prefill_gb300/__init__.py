"""GB300 (sm_103a) CRISP sparse-prefill attention: a C-ABI CUDA library and its binding.

The library (libcrisp.so, built from csrc/ by ``build.py``) implements the whole path:
PatSearch proxy attention and C_struct routing, VS and PE index selection, and the
block-sparse exact attention, plus a dense causal kernel.  Importing this package loads
the library and fails if it has not been built; there is no fallback path.
"""
from ._lib import (  # noqa: F401
    DEBUG_DROP_ARRIVE, FLAG_FORCE_PE, FLAG_FORCE_VS, FLAG_GRAPH_REPLAY, FLAG_MEDIAN_FLOOR,
    FLAG_VS_GAMMA_CUMSUM, Cfg, Context, CrispError, Dims, LIB_PATH,
    default_cfg, lib, make_dims, prefill_launches,
)

lib()

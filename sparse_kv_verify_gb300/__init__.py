"""GB300 (sm_103a) sparse-verification hot path of Dustin.

The work is done by ``libdustin.so`` (hand-written CUDA kernels behind the C
ABI of ``include/dustin.h``); this package is a thin ctypes binding over it.
"""
from . import binding  # noqa: F401
from .binding import (  # noqa: F401
    DustinError, Params, Signal, VerifyLayer, Workspace, StepCall, AppendCall, workspace, workspace_bytes,
    check, version, lib, kv_view, dustin_score, dustin_select, dustin_verify_attn,
    dense_verify_attn, dustin_kv_append, dustin_compact_kv, dustin_verify_step, dustin_score_noalloc,
    noalloc_check, wait_selftest, verify_split, split_units,
    EXPORTS, LIB_PATH,
    DEV_INDEX, DEV_NAN, DEV_APPEND, DEV_TIMEOUT, DEV_SEQLEN)

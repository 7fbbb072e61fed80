"""ctypes loader for libcoda.so with the argument types of every entry point
declared in include/coda.h. Loading fails loudly if the library is missing:
there is no fallback implementation."""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, Structure, c_char_p, c_double, c_float, c_int, c_size_t, c_uint64, c_void_p

# CODA_LIBRARY names another build of the same library to load instead (the
# checked build, libcoda_checked.so, next to this file).
LIB_PATH = os.environ.get("CODA_LIBRARY") or os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcoda.so")

P = c_void_p  # any device pointer (bf16 / fp32 / int32) or stream handle
I = c_int



class CodaBlock(Structure):
    """coda_block_t: descriptor of one period of the block-level chain (field
    order and types as in include/coda.h)."""
    _fields_ = [
        ("M", c_int), ("d", c_int), ("F", c_int), ("head_dim", c_int), ("rope_cols", c_int), ("S", c_int),
        ("eps", c_float), ("cos_tab", P), ("sin_tab", P),
        ("P", P), ("x", P), ("O", P), ("Wd", P), ("gamma1", P), ("Wqkv", P), ("Wo", P), ("gamma2", P), ("Wgu", P),
        ("h1", P), ("h1g", P), ("h2", P), ("h2g", P), ("gu", P), ("r1", P), ("r2", P),
        ("qkv", P), ("a", P),
        ("dqkv", P), ("gh", P), ("Wdn", P),
        ("dh1", P), ("dh2", P), ("dO", P), ("dWd", P), ("dWqkv", P), ("dWo", P), ("dWgu", P),
        ("dgamma1", P), ("dgamma2", P),
        ("dgur", P), ("dqr", P), ("s1", P), ("s2", P),
        ("workspace", P),
    ]


BLK = POINTER(CodaBlock)

# name -> (restype, argtypes); mirrors include/coda.h
SIGNATURES = {
    "coda_last_error": (c_char_p, []),
    "coda_init": (I, [I]),
    "coda_device_status": (I, [I]),
    "coda_set_wait_timeout_ns": (I, [c_uint64]),
    "coda_set_cta_group": (I, [I]),
    "coda_set_stream_k": (I, [I]),
    "coda_test_inject_missing_load": (I, []),
    "coda_num_col_tiles": (I, [I]),
    "coda_num_row_tiles": (I, [I]),
    "coda_gemm": (I, [I, I, I, P, I, I, P, I, I, P, I, P]),
    "coda_gemm_res_rmsprep": (I, [I, I, I, P, P, P, P, P, P, P, P]),
    "coda_rms_reduce": (I, [I, I, I, P, c_float, P, P]),
    "coda_gemm_rowscale": (I, [I, I, I, P, P, P, P, P]),
    "coda_gemm_swiglu": (I, [I, I, I, P, P, P, P, P]),
    "coda_gemm_swiglu_bwd": (I, [I, I, I, P, P, P, P, P]),
    "coda_rope_tables": (I, [I, I, c_double, P, P, P]),
    "coda_gemm_rope": (I, [I, I, I, P, P, P, P, I, I, I, P, P]),
    "coda_gemm_rope_bwd": (I, [I, I, I, P, P, P, P, I, I, I, P, P]),
    "coda_gemm_ce_lse": (I, [I, I, I, P, P, P, P, P, P, P, P]),
    "coda_ce_reduce": (I, [I, I, P, P, P, P, P, P, P, P, P]),
    "coda_gemm_ce_bwd": (I, [I, I, I, P, P, P, P, c_float, P, P]),
    "coda_gemm_rowdot": (I, [I, I, I, P, P, P, P, P, P, P, P]),
    "coda_rowdot_reduce": (I, [I, I, I, P, P, P]),
    "coda_gemm_rmsnorm_bwd": (I, [I, I, I, P, P, P, P, P, P, P, P, P]),
    "coda_colsum_reduce": (I, [I, I, P, P, P]),
    "coda_unfused_add": (I, [I, I, P, P, P, P]),
    "coda_unfused_rmsnorm": (I, [I, I, P, P, c_float, P, P, P]),
    "coda_unfused_rowscale": (I, [I, I, P, P, P, P]),
    "coda_unfused_swiglu": (I, [I, I, P, P, P]),
    "coda_unfused_swiglu_bwd": (I, [I, I, P, P, P, P]),
    "coda_unfused_rope": (I, [I, I, P, P, I, I, I, P, P]),
    "coda_unfused_rope_bwd": (I, [I, I, P, P, I, I, I, P, P]),
    "coda_unfused_ce_fwd": (I, [I, I, P, P, P, P, P, P, P]),
    "coda_unfused_ce_bwd": (I, [I, I, P, P, P, c_float, P, P]),
    "coda_unfused_rowdot": (I, [I, I, I, P, P, P, P]),
    "coda_unfused_rmsnorm_bwd": (I, [I, I, P, P, P, P, P, P, P]),
    "coda_gemm_rowscale_rope": (I, [I, I, I, P, P, P, P, P, I, I, I, P, P]),
    "coda_gemm_rowscale_swiglu": (I, [I, I, I, P, P, P, P, P, P]),
    "coda_gemm_swiglu_bwd_rowdot": (I, [I, I, I, P, P, P, P, P, P, P]),
    "coda_gemm_rmsnorm_bwd_res": (I, [I, I, I, P, P, P, P, P, P, P, P, P, P]),
    "coda_rope_bwd_rowdot": (I, [I, I, P, P, P, P, P, I, I, I, I, P, P, P]),
    "coda_gemm_fp8": (I, [I, I, I, P, P, c_float, P, P]),
    "coda_gemm_rope_fp8": (I, [I, I, I, P, P, c_float, P, P, I, I, I, P, P]),
    "coda_gemm_swiglu_fp8": (I, [I, I, I, P, P, c_float, P, P, P]),
    "coda_gemm_ce_lse_fp8": (I, [I, I, I, P, P, c_float, P, P, P, P, P, P]),
    "coda_gemm_ce_bwd_fp8": (I, [I, I, I, P, P, c_float, P, P, c_float, P, P]),
    "coda_block_workspace_bytes": (c_size_t, [I, I, I, I]),
    "coda_block_fwd": (I, [BLK, P]),
    "coda_block_fwd_noalloc": (I, [BLK, P]),
    "coda_block_bwd": (I, [BLK, P]),
    "coda_block_fwd_unfused": (I, [BLK, P]),
    "coda_block_bwd_unfused": (I, [BLK, P]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libcoda.so (once) and set every entry point's signature."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{os.path.basename(path)} not found at {path}: build it with "
            "`python -m gemm_epilogue_transformer_gb300.build_lib` (add --checked for the checked build; "
            "needs nvcc for sm_103a)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib

"""ctypes declarations of libdsa_rr.so (see include/dsa_rr.h). No computation happens here."""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa_rr.so")

c_int, c_i64, c_sz, c_f, c_vp, c_u32p = (ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                                         ctypes.c_float, ctypes.c_void_p,
                                         ctypes.POINTER(ctypes.c_uint32))
c_vpp, c_i64p = ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_int64)

# name -> (restype, argtypes), in header order
SIGNATURES = {
    "dsa_last_error_string": (ctypes.c_char_p, []),
    "dsa_version": (c_int, []),
    "dsa_read_device_errors": (c_int, [c_u32p]),
    "dsa_selftest_bounded_wait": (c_int, [c_i64, c_vp]),
    "dsa_probe_row_gather": (c_int, [c_vp, c_i64, c_vp, c_int, c_int, c_int, c_int, c_vp, c_vp]),
    "dsa_rr_shard_len": (c_i64, [c_i64, c_int, c_int]),
    "dsa_rr_split_metadata": (c_int, [c_vp, c_int, c_i64, c_int, c_int, c_vp, c_vp, c_vp, c_vp,
                                      c_vp, c_vp, c_i64, c_vp]),
    "dsa_rr_split_decode_metadata": (c_int, [c_vp, c_vp, c_int, c_i64, c_int, c_int, c_vp, c_vp,
                                             c_vp, c_vp, c_vp, c_vp, c_i64, c_vp]),
    "dsa_rr_rerange": (c_int, [c_vp, c_vp, c_i64, c_int, c_i64, c_i64, c_vp]),
    "dsa_rr_rerange_multi": (c_int, [c_vpp, c_vpp, c_i64p, c_int, c_i64, c_int, c_i64, c_vp]),
    "dsa_rr_rerange_paged": (c_int, [c_vp, c_vp, c_i64, c_i64, c_int, c_i64, c_i64, c_vp, c_int,
                                     c_vp, c_int, c_int, c_vp]),
    "dsa_rr_cache_local_paged": (c_int, [c_vp, c_vp, c_i64, c_i64, c_int, c_int, c_i64, c_vp,
                                         c_int, c_vp, c_int, c_int, c_vp]),
    "dsa_indexer_topk_workspace_size": (c_sz, [c_i64, c_int, c_int]),
    "dsa_score_row_stride": (c_i64, [c_int]),
    "dsa_indexer_scores": (c_int, [c_vp, c_vp, c_vp, c_i64, c_vp, c_int, c_vp, c_vp, c_i64, c_int,
                                   c_int, c_int, c_vp, c_int, c_int, c_vp, c_i64, c_vp, c_sz,
                                   c_vp]),
    "dsa_topk_select": (c_int, [c_vp, c_i64, c_vp, c_i64, c_int, c_int, c_vp, c_vp]),
    "dsa_indexer_topk": (c_int, [c_vp, c_vp, c_vp, c_i64, c_vp, c_int, c_vp, c_vp, c_i64, c_int,
                                 c_int, c_int, c_int, c_vp, c_int, c_int, c_vp, c_vp, c_sz, c_vp]),
    "dsa_indexer_topk_noalloc": (c_int, [c_vp, c_vp, c_vp, c_i64, c_vp, c_int, c_vp, c_vp, c_i64,
                                         c_int, c_int, c_int, c_int, c_vp, c_int, c_int, c_vp,
                                         c_vp]),
    "dsa_quantize_fp8_rows": (c_int, [c_vp, c_i64, c_int, c_vp, c_vp, c_vp]),
    "dsa_quantize_fp8_latent": (c_int, [c_vp, c_i64, c_vp, c_vp]),
    "dsa_dequantize_fp8_latent": (c_int, [c_vp, c_i64, c_vp, c_vp]),
    "dsa_indexer_scores_fp8": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_vp, c_int, c_vp,
                                       c_vp, c_i64, c_int, c_int, c_int, c_vp, c_int, c_int, c_vp,
                                       c_i64, c_vp, c_sz, c_vp]),
    "dsa_indexer_topk_fp8": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_vp, c_int, c_vp, c_vp,
                                     c_i64, c_int, c_int, c_int, c_int, c_vp, c_int, c_int, c_vp,
                                     c_vp, c_sz, c_vp]),
    "dsa_sparse_mla": (c_int, [c_vp, c_vp, c_i64, c_vp, c_int, c_vp, c_vp, c_i64, c_int, c_int,
                               c_int, c_int, c_f, c_vp, c_int, c_int, c_vp, c_vp, c_vp]),
    "dsa_sparse_mla_workspace_size": (c_sz, [c_i64]),
    "dsa_sparse_mla_balanced": (c_int, [c_vp, c_vp, c_i64, c_vp, c_int, c_vp, c_vp, c_vp, c_i64,
                                        c_int, c_int, c_int, c_int, c_f, c_vp, c_int, c_int, c_vp,
                                        c_vp, c_vp, c_sz, c_vp]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library once. Raises if it has not been built: there is no fallback path."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; "
                "g.build()' or python deepseek_v3_sparse_round_gb300/build.py)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib

"""ctypes declarations of the C ABI in include/dsa_idx.h (same names).

Argument marshalling only.  Loading fails loudly when libdsa_idx.so has not
been built; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

# DSA_IDX_LIB selects another build of the same ABI (e.g. the checked build,
# libdsa_idx_checked.so); by default the in-tree product library.
LIB_PATH = os.environ.get("DSA_IDX_LIB") or os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdsa_idx.so")

# dsa_status_t
DSA_OK = 0
DSA_ERR_INVALID_ARG = 1
DSA_ERR_UNSUPPORTED = 2
DSA_ERR_CUDA = 3
DSA_ERR_WORKSPACE = 4
DSA_ERR_TIMEOUT = 5
DSA_ERR_BOUNDS = 6
# dsa_dtype_t
DSA_DTYPE_F32 = 0
DSA_DTYPE_BF16 = 1
# dsa_precision_t
DSA_PREC_BF16 = 0
DSA_PREC_MXFP8 = 1
DSA_PREC_FP8 = 2
# dsa_mx_scale_rule_t
DSA_MX_SCALE_NOSAT = 0
DSA_MX_SCALE_FLOOR = 1
# flags
DSA_FLAG_DETERMINISTIC = 0x1
DSA_FLAG_SORT_BY_SCORE = 0x2
DSA_FLAG_KPOOL_TAIL = 0x4
DSA_FLAG_COMPRESSED_KEYS = 0x8

_c_int, _c_i64, _c_f, _c_size, _vp = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

# name -> (restype, argtypes); every pointer is passed as an integer address
SIGNATURES = {
    "dsa_idx_version": (_c_int, []),
    "dsa_idx_last_error": (ctypes.c_char_p, []),
    "dsa_idx_status_string": (ctypes.c_char_p, [_c_int]),
    "dsa_idx_workspace_size": (_c_size, [_c_int] * 7 + [_c_int]),
    "dsa_idx_output_width": (_c_int, [_c_int, _c_int, _c_int]),
    "dsa_idx_preprocess": (_c_int, [_vp, _vp, _c_int, _vp, _vp, _c_f, _vp, _c_int, _c_int, _c_int,
                                    _c_int, _c_int, _c_int, _c_f, _c_int, _c_int, _c_int, _c_int,
                                    _vp, _vp, _vp, _vp, _vp]),
    "dsa_idx_quantize_mxfp8": (_c_int, [_vp, _c_int, _c_i64, _c_int, _c_int, _vp, _vp, _vp]),
    "dsa_idx_quantize_fp8_rows": (_c_int, [_vp, _c_int, _c_i64, _c_int, _c_int, _vp, _vp, _vp]),
    "dsa_idx_kpool_compress": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                        _vp, _vp, _vp]),
    "dsa_idx_score_topk": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_f, _vp, _c_int, _c_int,
                                    _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _vp,
                                    _vp, _vp, _vp, _vp, _c_size, _vp]),
    "dsa_idx_score_topk_kv": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_f, _vp, _vp, _c_int, _c_int,
                                       _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                       _vp, _vp, _vp, _vp, _c_size, _vp]),
    "dsa_idx_score_topk_noalloc": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_f, _vp, _c_int, _c_int,
                                            _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _vp,
                                            _vp, _vp, _vp, _vp]),
    "dsa_idx_score_topk_noalloc_status": (_c_int, [_vp, ctypes.POINTER(_c_int)]),
    "dsa_idx_read_status": (_c_int, [_vp, _vp, ctypes.POINTER(_c_int)]),
    "dsa_idx_debug_mma_tile": (_c_int, [_vp, _vp, _c_i64, _c_i64, _vp, _vp, _c_i64, _c_i64, _c_int,
                                        _c_int, _c_int, _vp, _vp, _c_size, _vp]),
    # test hooks (not in the public header)
    "dsa_idx_test_set_timeout_ns": (None, [ctypes.c_ulonglong]),
    "dsa_idx_test_set_fault_inject": (None, [_c_int]),
}

_lib = None


def load() -> ctypes.CDLL:
    """Load libdsa_idx.so and declare every entry point.  Raises if missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is not built; run `python -m sparse_attention_indexer_dsa_gb300.build_lib` "
            "(or __graft_entry__.build()) first.  There is no fallback implementation.")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def __getattr__(name):
    if name in SIGNATURES:
        return getattr(load(), name)
    raise AttributeError(name)

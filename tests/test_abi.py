"""The C-ABI library builds, loads without a GPU and exports every entry
point include/dsa_idx.h declares; host-only functions and host-side argument
checks behave as documented.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

from sparse_attention_indexer_dsa_gb300 import _abi, build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return _abi.load()


def _declared():
    src = "".join(open(os.path.join(ROOT, "include", h)).read() for h in ("dsa_idx.h", "dsa_idx_testing.h"))
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_idx_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
        assert n in _abi.SIGNATURES, f"binding lacks {n}"


def test_host_only_functions(lib):
    assert lib.dsa_idx_version() >= 100
    assert lib.dsa_idx_status_string(5) == b"DSA_ERR_TIMEOUT"
    assert lib.dsa_idx_output_width(2048, 1, 0) == 2048
    assert lib.dsa_idx_output_width(2048, 4, _abi.DSA_FLAG_KPOOL_TAIL) == 2051
    assert lib.dsa_idx_output_width(2048, 4, 0) == 2048
    ws = lib.dsa_idx_workspace_size(32768, 1, 32768, 64, 128, 2048, 1, _abi.DSA_PREC_MXFP8)
    assert ws >= 8 * 32768
    assert lib.dsa_idx_workspace_size(-1, 1, 0, 64, 128, 1, 1, 0) == 0
    # the 8-bit formats keep one 512-byte key-scale tile per 128 keys (plus one
    # per document) in the workspace; BF16 needs none
    args = (32768, 3, 32768, 64, 128, 2048, 1)
    bf = lib.dsa_idx_workspace_size(*args, _abi.DSA_PREC_BF16)
    mx = lib.dsa_idx_workspace_size(*args, _abi.DSA_PREC_MXFP8)
    f8 = lib.dsa_idx_workspace_size(*args, _abi.DSA_PREC_FP8)
    assert mx == f8 == bf + 512 * (32768 // 128 + 3 + 1)


def test_host_argument_checks_precede_any_cuda_call(lib):
    P = ctypes.c_void_p
    # null q -> INVALID_ARG, before the device is touched
    rc = lib.dsa_idx_score_topk(None, None, P(256), None, P(256), 0, 1.0, P(256), 1, 16, 16, 64, 128,
                                16, 0, 1, 1, None, P(256), None, None, P(256), 1 << 20, None)
    assert rc == _abi.DSA_ERR_INVALID_ARG
    assert b"null" in lib.dsa_idx_last_error()
    # unsupported head count
    rc = lib.dsa_idx_score_topk(P(256), None, P(256), None, P(256), 0, 1.0, P(256), 1, 16, 16, 3, 128,
                                16, 0, 1, 1, None, P(256), None, None, P(256), 1 << 20, None)
    assert rc == _abi.DSA_ERR_UNSUPPORTED
    # MXFP8 without scales
    rc = lib.dsa_idx_score_topk(P(256), None, P(256), None, P(256), 0, 1.0, P(256), 1, 16, 16, 64, 128,
                                16, 1, 1, 1, None, P(256), None, None, P(256), 1 << 20, None)
    assert rc == _abi.DSA_ERR_INVALID_ARG
    # workspace too small
    rc = lib.dsa_idx_score_topk(P(256), None, P(256), None, P(256), 0, 1.0, P(256), 1, 16, 16, 64, 128,
                                16, 0, 1, 1, None, P(256), None, None, P(256), 16, None)
    assert rc == _abi.DSA_ERR_WORKSPACE
    # top-k beyond the supported 4096
    rc = lib.dsa_idx_score_topk(P(256), None, P(256), None, P(256), 0, 1.0, P(256), 1, 16, 16, 64, 128,
                                4097, 0, 1, 1, None, P(256), None, None, P(256), 1 << 20, None)
    assert rc == _abi.DSA_ERR_UNSUPPORTED
    # KPool: at most 4096 pools
    rc = lib.dsa_idx_score_topk(P(256), None, P(256), None, P(256), 0, 1.0, P(256), 1, 16, 16, 64, 128,
                                4 * 4097, 0, 1, 4, P(256), P(256), None, None, P(256), 1 << 20, None)
    assert rc == _abi.DSA_ERR_UNSUPPORTED
    # the no-allocation status reader needs somewhere to put the status
    assert lib.dsa_idx_score_topk_noalloc_status(None, None) == _abi.DSA_ERR_INVALID_ARG
    # misaligned tensor
    rc = lib.dsa_idx_quantize_mxfp8(P(257), 0, 4, 128, 0, P(256), P(256), None)
    assert rc == _abi.DSA_ERR_INVALID_ARG
    rc = lib.dsa_idx_quantize_mxfp8(P(256), 0, 4, 100, 0, P(256), P(256), None)
    assert rc == _abi.DSA_ERR_INVALID_ARG
    rc = lib.dsa_idx_preprocess(P(256), P(256), 0, None, None, 1e-6, P(256), 1, 8, 8, 64, 128, 12, 1e4,
                                0, 1, 0, 0, P(256), None, P(256), None, None)
    assert rc == _abi.DSA_ERR_INVALID_ARG          # rope_dim not a multiple of 8
    rc = lib.dsa_idx_kpool_compress(P(256), 0, P(256), P(256), P(256), 1, 8, 128, 3, P(256), P(256), None)
    assert rc == _abi.DSA_ERR_UNSUPPORTED


def test_host_checks_of_the_extended_modes(lib):
    """Argument checks of the key-offset entry point, compressed keys and
    per-vector FP8, all before any CUDA call."""
    P = ctypes.c_void_p
    F = _abi.DSA_FLAG_DETERMINISTIC
    # documents with more keys than queries: cu_seqlens_k is required
    rc = lib.dsa_idx_score_topk_kv(P(256), None, P(256), None, P(256), 0, 1.0, P(256), None, 1, 8, 16, 8, 16,
                                   64, 128, 16, 0, F, P(256), None, None, P(256), 1 << 20, None)
    assert rc == _abi.DSA_ERR_INVALID_ARG
    # ... and a key length above the 16-bit index range
    rc = lib.dsa_idx_score_topk_kv(P(256), None, P(256), None, P(256), 0, 1.0, P(256), P(256), 1, 8, 16, 8,
                                   70000, 64, 128, 16, 0, F, P(256), None, None, P(256), 1 << 20, None)
    assert rc == _abi.DSA_ERR_UNSUPPORTED
    C = _abi.DSA_FLAG_COMPRESSED_KEYS
    assert lib.dsa_idx_output_width(300, 4, C) == 300
    # compressed keys: ratio range, cu_pools required, no KPool tail
    for ratio, pools, flags, want in ((1, P(256), F | C, _abi.DSA_ERR_UNSUPPORTED),
                                      (65, P(256), F | C, _abi.DSA_ERR_UNSUPPORTED),
                                      (4, None, F | C, _abi.DSA_ERR_INVALID_ARG),
                                      (4, P(256), F | C | _abi.DSA_FLAG_KPOOL_TAIL, _abi.DSA_ERR_INVALID_ARG)):
        rc = lib.dsa_idx_score_topk(P(256), None, P(256), None, P(256), 0, 1.0, P(256), 1, 16, 16, 64, 128,
                                    16, 0, flags, ratio, pools, P(256), None, None, P(256), 1 << 20, None)
        assert rc == want, (ratio, flags, rc)
    # per-vector FP8: head_dim 128 and both scale arrays
    rc = lib.dsa_idx_score_topk(P(256), None, P(256), P(256), P(256), 0, 1.0, P(256), 1, 16, 16, 64, 128,
                                16, _abi.DSA_PREC_FP8, F, 1, None, P(256), None, None, P(256), 1 << 20, None)
    assert rc == _abi.DSA_ERR_INVALID_ARG
    rc = lib.dsa_idx_score_topk(P(256), P(256), P(256), P(256), P(256), 0, 1.0, P(256), 1, 16, 16, 64, 64,
                                16, _abi.DSA_PREC_FP8, F, 1, None, P(256), None, None, P(256), 1 << 20, None)
    assert rc == _abi.DSA_ERR_UNSUPPORTED
    rc = lib.dsa_idx_quantize_fp8_rows(P(256), 0, 4, 64, 0, P(256), P(256), None)
    assert rc == _abi.DSA_ERR_UNSUPPORTED
    # ranking order ranks by the scores: topk_score is required
    rc = lib.dsa_idx_score_topk(P(256), None, P(256), None, P(256), 0, 1.0, P(256), 1, 16, 16, 64, 128,
                                16, 0, F | _abi.DSA_FLAG_SORT_BY_SCORE, 1, None, P(256), None, None, P(256),
                                1 << 20, None)
    assert rc == _abi.DSA_ERR_INVALID_ARG


def test_score_plan_fits_every_supported_shape(lib):
    """Every supported (precision, head count, top-k) has a kernel plan; the
    planner lives in C, so probe it through the host path: a valid call with
    a zero-token batch stops at device discovery, not at planning."""
    P = ctypes.c_void_p
    for prec, D in ((0, 128), (0, 64), (1, 128), (2, 128)):
        for H in (4, 8, 16, 32, 64):
            for k in ((1, 32, 256, 1024) if (prec != 0 and H == 4) else (1, 32, 256, 2048, 3000, 4096)):
                rc = lib.dsa_idx_score_topk(P(256), P(256), P(256), P(256), P(256), 0, 1.0, P(256), 1, 0, 0,
                                            H, D, k, prec, 1, 1, None, P(256), None, None, P(256), 1 << 20, None)
                assert rc in (_abi.DSA_OK, _abi.DSA_ERR_CUDA, _abi.DSA_ERR_UNSUPPORTED), (prec, D, H, k, rc)
                if rc == _abi.DSA_ERR_UNSUPPORTED:
                    assert b"no kernel configuration" not in lib.dsa_idx_last_error(), (prec, D, H, k)


def test_checked_build_exports_the_same_entry_points():
    """The checked build (-DDSA_CHECKED, device bounds checks and a NaN/Inf
    scan of the inputs) compiles, loads without a GPU, exports every declared
    entry point and reports itself by an odd version number."""
    path = build_lib.build_checked()
    chk = ctypes.CDLL(path)
    for n in _declared():
        assert hasattr(chk, n), n
    chk.dsa_idx_version.restype = ctypes.c_int
    assert chk.dsa_idx_version() % 2 == 1
    assert _abi.load().dsa_idx_version() % 2 == 0
    chk.dsa_idx_status_string.restype = ctypes.c_char_p
    assert chk.dsa_idx_status_string(_abi.DSA_ERR_BOUNDS) == b"DSA_ERR_BOUNDS"

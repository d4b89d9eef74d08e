"""The C-ABI library: it builds, loads without a GPU and exports every symbol its headers declare."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M):
            if not m.group(0).lstrip().startswith(("typedef", "#", "return")):
                names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    from vocab_cross_entropy_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_headers_declare_the_boundary():
    names = declared_functions()
    for n in ("ce_forward", "ce_backward", "ce_merge_chunks", "vce_get_status", "vce_status_string"):
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in sorted(declared_functions()) if not hasattr(lib, n)]
    assert not missing, missing


def test_host_only_calls(lib):
    lib.vce_status_string.restype = ctypes.c_char_p
    assert lib.vce_abi_version() == 1
    assert lib.vce_row_stats_floats() == 4
    assert b"label" in lib.vce_status_string(1)
    assert lib.vce_status_string(12345) == b"unknown status"


def test_argument_errors_need_no_gpu(lib):
    # checks that fail before any CUDA call: bad dtype, bad reduction, null status, ld < V
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    f = lib.ce_forward
    f.argtypes = [P, ctypes.c_int, i64, i64, i64, P, i64, ctypes.c_int, P, P, P, P, P]
    x = P(0x1000)
    assert f(x, 7, 4, 8, 8, x, -100, 2, x, x, x, x, None) == -2
    assert f(x, 1, 4, 8, 8, x, -100, 5, x, x, x, x, None) == -2
    assert f(x, 1, 4, 8, 8, x, -100, 2, x, x, x, None, None) == -1
    assert f(x, 1, 4, 8, 7, x, -100, 2, x, x, x, x, None) == -4
    assert f(x, 1, 4, 0, 8, x, -100, 2, x, x, x, x, None) == -3
    m = lib.ce_merge_chunks
    assert m(0, None, None, None, 1, 4, None, -100, 2, None, None, None, None, None, None, 1, None, None,
             None) == -8
    st = lib.vce_test_ce_fwd_stall   # the forward ring's give-up hook: its host checks
    st.argtypes = [P, i64, i64, P, P, P, P, ctypes.c_uint64, P, P]
    assert st(x, 4, 20000, x, x, x, x, 50_000_000, None, None) == -1       # null status
    assert st(x, 0, 20000, x, x, x, x, 50_000_000, x, None) == -3          # no rows
    assert st(x, 70000, 20000, x, x, x, x, 50_000_000, x, None) == -3      # beyond the folded reduction
    assert st(x, 4, 20000, x, x, x, x, 1000, x, None) == -8                # wait bound under 1 ms
    assert st(x, 4, 8000, x, x, x, x, 50_000_000, x, None) == -8           # 16 KB rows: the warp kernel


def test_linear_and_gemm_hook_argument_errors_need_no_gpu(lib):
    """linear_ce_fwd_bwd_filtered refuses a NaN, negative or infinite eps, vce_test_gemm_skip
    refuses null pointers, bad shapes and short bit rows, and vce_gemm_bf16_variant refuses pairs
    on an odd tile count, all before any CUDA call."""
    P, i64, i32, f32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    x = P(0x1000)
    f = lib.linear_ce_fwd_bwd_filtered
    f.argtypes = [P, P, i64, i64, i64, P, i64, i32, P, P, P, P, P, i32, f32, P, P, sz, P, P]
    args = lambda eps: (x, x, 16, 64, 100, x, -100, 2, x, x, x, x, x, 1, eps, None, x, 1 << 30, x, None)
    for eps in (float("nan"), -1e-3, float("inf")):
        assert f(*args(eps)) == -8, eps
    assert lib.linear_ce_workspace_bytes(i64(16), i64(60), i64(100)) == 0      # D not a multiple of 8
    g = lib.vce_test_gemm_skip
    g.argtypes = [P, P, i64, i64, i64, P, i64, P, P]
    assert g(None, x, 256, 256, 128, x, 1, x, None) == -1                        # null A
    assert g(x, x, 256, 256, 100, x, 1, x, None) == -3                           # K not a multiple of 8
    assert g(x, x, 256, 256, 8192, x, 1, x, None) == -8                          # 64 blocks need 2 words
    v = lib.vce_gemm_bf16_variant
    v.argtypes = [P, i32, P, i32, i64, i64, i64, P, i64, i32, P]
    assert v(x, 0, x, 0, 384, 256, 128, x, 256, 1, None) == -8          # 3 M tiles cannot pair
    assert v(x, 0, x, 0, 256, 256, 128, x, 256, 3, None) == -8          # pair is 0, 1 or 2
    assert v(x, 0, x, 0, 256, 256, 192, x, 256, 2, None) == -8          # 3 K blocks cannot pair up
    assert v(x, 0, x, 0, 256, 256, 128, x, 200, 1, None) == -4          # ldc < N

"""Python binding of libvce.so, the GB300 vocabulary cross-entropy library.

Argument marshalling only: every step of the computation runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (torch supplies device memory and streams);
each function passes raw pointers to the C entry point of the same name in
``include/vce.h`` and raises ``VceError`` on a non-zero return.  There is no CPU
fallback: importing works without a GPU, calling a compute entry point needs one.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = ["VceError", "lib", "library_path", "ce_forward", "ce_backward", "ce_forward_ls", "ce_backward_ls",
           "ce_forward_backward", "ce_forward_backward_ls", "ce_merge_chunks", "ce_merge_chunks_ls",
           "ce_merge_chunks_noalloc",
           "linear_ce_workspace_bytes", "linear_ce_fwd_bwd", "linear_ce_fwd_bwd_filtered", "linear_ce_fwd_bwd_timed",
           "vce_get_status", "vce_status_string", "vce_debug_checks", "vce_debug_status", "use_library",
           "restore_library",
           "vce_abi_version", "cross_entropy", "IGNORE_INDEX", "F32", "BF16", "RED"]

IGNORE_INDEX = -100
F32, BF16 = 0, 1
RED = {"none": 0, "sum": 1, "mean": 2}
ROW_STATS = 4
CHUNK_STATS = 4
_DT = {torch.float32: F32, torch.bfloat16: BF16}

library_path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libvce.so")
# the same library built with device-side index checks (build --debug-checks)
debug_library_path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libvce_debug.so")


class VceError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        msg = f"{fn} failed: {code} ({vce_status_string(code)})"
        if code == -7:   # VCE_ERR_CUDA: name the CUDA runtime result behind it
            e = _get().vce_last_cuda_error()
            msg += f"; CUDA: {e} {_get().vce_cuda_error_name(e).decode()}"
        super().__init__(msg)


def _load(path=None):
    path = path or library_path
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built: run `python -m vocab_cross_entropy_gb300.build` "
                          "(or __graft_entry__.build()) first; this library has no fallback path")
    L = ctypes.CDLL(path)
    p, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    L.vce_abi_version.restype = i32
    L.vce_status_string.argtypes = [i32]
    L.vce_status_string.restype = ctypes.c_char_p
    L.vce_row_stats_floats.restype = sz
    L.vce_get_status.argtypes = [p, p, p]
    L.vce_last_cuda_error.restype = i32
    L.vce_cuda_error_name.argtypes = [i32]
    L.vce_cuda_error_name.restype = ctypes.c_char_p
    L.vce_debug_checks.restype = i32
    L.vce_debug_status.argtypes = [p]
    L.vce_debug_status.restype = i32
    L.ce_forward.argtypes = [p, i32, i64, i64, i64, p, i64, i32, p, p, p, p, p]
    L.ce_backward.argtypes = [p, i32, i64, i64, i64, p, i64, i32, p, p, p, i32, i64, p]
    L.ce_forward_backward.argtypes = [p, i32, i64, i64, i64, p, i64, i32, p, p, p, p, p, i32, i64, p, p]
    L.ce_forward_backward_ls.argtypes = [p, i32, i64, i64, i64, p, i64, ctypes.c_float, i32, p, p, p, p, p, i32, i64,
                                         p, p]
    f32 = ctypes.c_float
    L.ce_forward_ls.argtypes = [p, i32, i64, i64, i64, p, i64, f32, i32, p, p, p, p, p]
    L.ce_backward_ls.argtypes = [p, i32, i64, i64, i64, p, i64, f32, i32, p, p, p, i32, i64, p]
    L.ce_merge_chunks.argtypes = [i32, p, p, p, i32, i64, p, i64, i32, p, p, p, p, p, p, i32, p, p, p]
    L.ce_merge_chunks_ls.argtypes = [i32, p, p, p, i32, i64, p, i64, ctypes.c_float, i32, p, p, p, p, p, p, i32, p, p,
                                     p, p]
    L.ce_merge_chunks_noalloc.argtypes = [i32, p, p, p, i32, i64, p, i64, i32, p, p, p, p, p, p, i32, p, p]
    if hasattr(L, "linear_ce_fwd_bwd"):
        L.linear_ce_workspace_bytes.argtypes = [i64, i64, i64]
        L.linear_ce_workspace_bytes.restype = sz
        L.linear_ce_fwd_bwd.argtypes = [p, p, i64, i64, i64, p, i64, i32, p, p, p, p, p, i32, p, sz, p, p]
        if hasattr(L, "linear_ce_fwd_bwd_filtered"):
            L.linear_ce_fwd_bwd_filtered.argtypes = [p, p, i64, i64, i64, p, i64, i32, p, p, p, p, p, i32, f32, p,
                                                     p, sz, p, p]
        L.linear_ce_fwd_bwd_timed.argtypes = [p, p, i64, i64, i64, p, i64, i32, p, p, p, p, p, i32, f32, p, p, sz,
                                              p, p, p, p]
        L.vce_gemm_bf16.argtypes = [p, i32, p, i32, i64, i64, i64, p, i64, p]
        L.vce_gemm_bf16.restype = i32
        L.vce_gemm_bf16_variant.argtypes = [p, i32, p, i32, i64, i64, i64, p, i64, i32, p]
        L.vce_gemm_bf16_variant.restype = i32
        L.vce_test_gemm_stall.argtypes = [p, p, i64, i64, i64, p, ctypes.c_uint64, p, p]
        L.vce_test_gemm_stall.restype = i32
        if hasattr(L, "vce_test_gemm_skip"):
            L.vce_test_gemm_skip.argtypes = [p, p, i64, i64, i64, p, i64, p, p]
            L.vce_test_gemm_skip.restype = i32
        L.vce_test_ce_fused_stall.argtypes = [p, i64, i64, p, p, p, p, p, ctypes.c_uint64, p, p]
        L.vce_test_ce_fused_stall.restype = i32
        L.vce_test_ce_fwd_stall.argtypes = [p, i64, i64, p, p, p, p, ctypes.c_uint64, p, p]
        L.vce_test_ce_fwd_stall.restype = i32
    for name in ("ce_forward", "ce_backward", "ce_forward_ls", "ce_backward_ls", "ce_forward_backward",
                 "ce_forward_backward_ls", "ce_merge_chunks_ls",
                 "ce_merge_chunks", "ce_merge_chunks_noalloc",
                 "linear_ce_fwd_bwd", "linear_ce_fwd_bwd_filtered", "linear_ce_fwd_bwd_timed",
                 "vce_get_status"):
        if hasattr(L, name):
            getattr(L, name).restype = i32
    return L


_lib = None


def _get():
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def use_library(path):
    """Route every call of this module to the library at `path` (e.g. debug_library_path, the
    build with device-side index checks); returns the previous library (None if none was
    loaded yet).  No fallback: the library must exist."""
    global _lib
    prev = _lib
    _lib = _load(path)
    return prev


def restore_library(prev):
    """Undo use_library: route calls back to `prev` (None: the default library, loaded on use)."""
    global _lib
    _lib = prev


def vce_debug_checks() -> bool:
    """Whether the library in use was built with device-side index checks."""
    return bool(_get().vce_debug_checks())


def vce_debug_status() -> int:
    """Waits for the device; the first failed index check's code since the last call, or 0."""
    out = ctypes.c_int32(0)
    _check("vce_debug_status", _get().vce_debug_status(ctypes.byref(out)))
    return int(out.value)


def __getattr__(name):   # `lib` is loaded on first use, so the build module imports without it
    if name == "lib":
        return _get()
    raise AttributeError(name)


def vce_abi_version() -> int:
    return _get().vce_abi_version()


def vce_status_string(code: int) -> str:
    return _get().vce_status_string(int(code)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, rc):
    if rc != 0:
        raise VceError(fn, rc)


def _dtype(t):
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}; use float32 or bfloat16") from None


def _ld(t):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D tensor with unit column stride")
    return t.stride(0)


def vce_get_status(status, stream=None) -> int:
    """Wait for the stream and return the device status word (0 = ok, 1 = bad label)."""
    out = ctypes.c_int32(0)
    _check("vce_get_status", _get().vce_get_status(_ptr(status), _stream(stream), ctypes.byref(out)))
    return out.value


def ce_forward(logits, labels, ignore_index=IGNORE_INDEX, reduction="mean", *, loss_rows=None, loss_out=None,
               row_stats=None, status=None, stream=None):
    """Per-row loss, reduced loss and row statistics.  Returns (loss_out, loss_rows, row_stats, status)."""
    T, V = logits.shape
    dev = logits.device
    loss_rows = torch.empty(T, dtype=torch.float32, device=dev) if loss_rows is None else loss_rows
    row_stats = torch.empty(T, ROW_STATS, dtype=torch.float32, device=dev) if row_stats is None else row_stats
    status = torch.empty(1, dtype=torch.int32, device=dev) if status is None else status
    if reduction != "none" and loss_out is None:
        loss_out = torch.empty(1, dtype=torch.float32, device=dev)
    _check("ce_forward", _get().ce_forward(_ptr(logits), _dtype(logits), T, V, _ld(logits), _ptr(labels),
                                        int(ignore_index), RED[reduction], _ptr(loss_rows), _ptr(loss_out),
                                        _ptr(row_stats), _ptr(status), _stream(stream)))
    return loss_out, loss_rows, row_stats, status


def ce_backward(logits, labels, row_stats, grad_output, ignore_index=IGNORE_INDEX, reduction="mean", *,
                grad_logits=None, grad_dtype=None, stream=None):
    """Gradient of the reduced loss w.r.t. the logits.  Returns grad_logits."""
    T, V = logits.shape
    if grad_logits is None:
        grad_logits = torch.empty(T, V, dtype=grad_dtype or logits.dtype, device=logits.device)
    _check("ce_backward", _get().ce_backward(_ptr(logits), _dtype(logits), T, V, _ld(logits), _ptr(labels),
                                          int(ignore_index), RED[reduction], _ptr(row_stats), _ptr(grad_output),
                                          _ptr(grad_logits), _dtype(grad_logits), _ld(grad_logits),
                                          _stream(stream)))
    return grad_logits


def ce_forward_ls(logits, labels, label_smoothing, ignore_index=IGNORE_INDEX, reduction="mean", *, loss_rows=None,
                  loss_out=None, row_stats=None, status=None, stream=None):
    """ce_forward with label smoothing.  Returns (loss_out, loss_rows, row_stats, status)."""
    T, V = logits.shape
    dev = logits.device
    loss_rows = torch.empty(T, dtype=torch.float32, device=dev) if loss_rows is None else loss_rows
    row_stats = torch.empty(T, ROW_STATS, dtype=torch.float32, device=dev) if row_stats is None else row_stats
    status = torch.empty(1, dtype=torch.int32, device=dev) if status is None else status
    if reduction != "none" and loss_out is None:
        loss_out = torch.empty(1, dtype=torch.float32, device=dev)
    _check("ce_forward_ls", _get().ce_forward_ls(_ptr(logits), _dtype(logits), T, V, _ld(logits), _ptr(labels),
                                              int(ignore_index), float(label_smoothing), RED[reduction],
                                              _ptr(loss_rows), _ptr(loss_out), _ptr(row_stats), _ptr(status),
                                              _stream(stream)))
    return loss_out, loss_rows, row_stats, status


def ce_backward_ls(logits, labels, row_stats, grad_output, label_smoothing, ignore_index=IGNORE_INDEX,
                   reduction="mean", *, grad_logits=None, grad_dtype=None, stream=None):
    """ce_backward with label smoothing.  Returns grad_logits."""
    T, V = logits.shape
    if grad_logits is None:
        grad_logits = torch.empty(T, V, dtype=grad_dtype or logits.dtype, device=logits.device)
    _check("ce_backward_ls", _get().ce_backward_ls(
        _ptr(logits), _dtype(logits), T, V, _ld(logits), _ptr(labels), int(ignore_index), float(label_smoothing),
        RED[reduction], _ptr(row_stats), _ptr(grad_output), _ptr(grad_logits), _dtype(grad_logits),
        _ld(grad_logits), _stream(stream)))
    return grad_logits


def ce_forward_backward(logits, labels, ignore_index=IGNORE_INDEX, reduction="mean", *, grad_output=None,
                        grad_logits=None, grad_dtype=None, loss_rows=None, loss_out=None, row_stats=None,
                        status=None, stream=None):
    """Forward and gradient in one pass.  Returns (loss_out, loss_rows, row_stats, grad_logits, status)."""
    T, V = logits.shape
    dev = logits.device
    loss_rows = torch.empty(T, dtype=torch.float32, device=dev) if loss_rows is None else loss_rows
    row_stats = torch.empty(T, ROW_STATS, dtype=torch.float32, device=dev) if row_stats is None else row_stats
    status = torch.empty(1, dtype=torch.int32, device=dev) if status is None else status
    if reduction != "none" and loss_out is None:
        loss_out = torch.empty(1, dtype=torch.float32, device=dev)
    if grad_output is None:
        grad_output = torch.ones(T if reduction == "none" else 1, dtype=torch.float32, device=dev)
    if grad_logits is None:
        grad_logits = torch.empty(T, V, dtype=grad_dtype or logits.dtype, device=dev)
    _check("ce_forward_backward", _get().ce_forward_backward(
        _ptr(logits), _dtype(logits), T, V, _ld(logits), _ptr(labels), int(ignore_index), RED[reduction],
        _ptr(grad_output), _ptr(loss_rows), _ptr(loss_out), _ptr(row_stats), _ptr(grad_logits),
        _dtype(grad_logits), _ld(grad_logits), _ptr(status), _stream(stream)))
    return loss_out, loss_rows, row_stats, grad_logits, status


def ce_forward_backward_ls(logits, labels, label_smoothing, ignore_index=IGNORE_INDEX, reduction="mean", *,
                           grad_output=None, grad_logits=None, grad_dtype=None, loss_rows=None, loss_out=None,
                           row_stats=None, status=None, stream=None):
    """ce_forward_backward with label smoothing.  Returns (loss_out, loss_rows, row_stats, grad_logits, status)."""
    T, V = logits.shape
    dev = logits.device
    loss_rows = torch.empty(T, dtype=torch.float32, device=dev) if loss_rows is None else loss_rows
    row_stats = torch.empty(T, ROW_STATS, dtype=torch.float32, device=dev) if row_stats is None else row_stats
    status = torch.empty(1, dtype=torch.int32, device=dev) if status is None else status
    if reduction != "none" and loss_out is None:
        loss_out = torch.empty(1, dtype=torch.float32, device=dev)
    if grad_output is None:
        grad_output = torch.ones(T if reduction == "none" else 1, dtype=torch.float32, device=dev)
    if grad_logits is None:
        grad_logits = torch.empty(T, V, dtype=grad_dtype or logits.dtype, device=dev)
    _check("ce_forward_backward_ls", _get().ce_forward_backward_ls(
        _ptr(logits), _dtype(logits), T, V, _ld(logits), _ptr(labels), int(ignore_index), float(label_smoothing),
        RED[reduction], _ptr(grad_output), _ptr(loss_rows), _ptr(loss_out), _ptr(row_stats), _ptr(grad_logits),
        _dtype(grad_logits), _ld(grad_logits), _ptr(status), _stream(stream)))
    return loss_out, loss_rows, row_stats, grad_logits, status

def ce_merge_chunks(chunks, labels, ignore_index=IGNORE_INDEX, reduction="mean", *, grad_output=None,
                    chunk_grads=None, grad_dtype=None, want_grad=True, loss_rows=None, loss_out=None,
                    row_stats=None, chunk_stats=None, status=None, stream=None, label_smoothing=0.0):
    """CE over column chunks (list of [T, w_c] tensors); label_smoothing > 0 calls ce_merge_chunks_ls.

    Returns (loss_out, loss_rows, row_stats, chunk_grads or None, chunk_stats [k, T, 4], status).
    """
    k = len(chunks)
    T = chunks[0].shape[0]
    dev = chunks[0].device
    dt = _dtype(chunks[0])
    if any(_dtype(c) != dt or c.shape[0] != T for c in chunks):
        raise ValueError("chunks must share dtype and row count")
    loss_rows = torch.empty(T, dtype=torch.float32, device=dev) if loss_rows is None else loss_rows
    row_stats = torch.empty(T, ROW_STATS, dtype=torch.float32, device=dev) if row_stats is None else row_stats
    chunk_stats = torch.empty(k, T, CHUNK_STATS, dtype=torch.float32, device=dev) if chunk_stats is None else chunk_stats
    status = torch.empty(1, dtype=torch.int32, device=dev) if status is None else status
    if reduction != "none" and loss_out is None:
        loss_out = torch.empty(1, dtype=torch.float32, device=dev)
    if want_grad and chunk_grads is None:
        chunk_grads = [torch.empty(T, c.shape[1], dtype=grad_dtype or c.dtype, device=dev) for c in chunks]
    if want_grad and grad_output is None:
        grad_output = torch.ones(T if reduction == "none" else 1, dtype=torch.float32, device=dev)
    P = ctypes.c_void_p * k
    I = ctypes.c_int64 * k
    in_ptrs = P(*[c.data_ptr() for c in chunks])
    widths = I(*[c.shape[1] for c in chunks])
    lds = I(*[_ld(c) for c in chunks])
    g_ptrs = P(*[g.data_ptr() for g in chunk_grads]) if want_grad else None
    g_lds = I(*[_ld(g) for g in chunk_grads]) if want_grad else None
    gdt = _dtype(chunk_grads[0]) if want_grad else F32
    if label_smoothing:
        chunk_sums = torch.empty(k, T, dtype=torch.float32, device=dev)
        _check("ce_merge_chunks_ls", _get().ce_merge_chunks_ls(
            k, in_ptrs, widths, lds, dt, T, _ptr(labels), int(ignore_index), float(label_smoothing), RED[reduction],
            _ptr(loss_rows), _ptr(loss_out), _ptr(row_stats), _ptr(grad_output), g_ptrs, g_lds, gdt,
            _ptr(chunk_stats), _ptr(chunk_sums), _ptr(status), _stream(stream)))
    else:
        _check("ce_merge_chunks", _get().ce_merge_chunks(
            k, in_ptrs, widths, lds, dt, T, _ptr(labels), int(ignore_index), RED[reduction], _ptr(loss_rows),
            _ptr(loss_out), _ptr(row_stats), _ptr(grad_output), g_ptrs, g_lds, gdt, _ptr(chunk_stats),
            _ptr(status), _stream(stream)))
    return loss_out, loss_rows, row_stats, (chunk_grads if want_grad else None), chunk_stats, status


NOALLOC_MAX_CHUNK_ROWS = 262144


def ce_merge_chunks_noalloc(chunks, labels, ignore_index=IGNORE_INDEX, reduction="mean", *, grad_output,
                            chunk_grads, loss_rows, loss_out, row_stats, status, stream=None):
    """ce_merge_chunks without a scratch workspace, for callers that cannot allocate device memory.

    Every output buffer is the caller's (this wrapper allocates nothing); chunk_grads may be
    None for a forward-only call.  The statistics go to an array the library keeps in device
    memory (k * T <= NOALLOC_MAX_CHUNK_ROWS).  Returns None; raises VceError on a non-zero return.
    """
    k = len(chunks)
    T = chunks[0].shape[0]
    dt = _dtype(chunks[0])
    P = ctypes.c_void_p * k
    I = ctypes.c_int64 * k
    in_ptrs = P(*[c.data_ptr() for c in chunks])
    widths = I(*[c.shape[1] for c in chunks])
    lds = I(*[_ld(c) for c in chunks])
    g_ptrs = P(*[g.data_ptr() for g in chunk_grads]) if chunk_grads is not None else None
    g_lds = I(*[_ld(g) for g in chunk_grads]) if chunk_grads is not None else None
    gdt = _dtype(chunk_grads[0]) if chunk_grads is not None else F32
    _check("ce_merge_chunks_noalloc", _get().ce_merge_chunks_noalloc(
        k, in_ptrs, widths, lds, dt, T, _ptr(labels), int(ignore_index), RED[reduction], _ptr(loss_rows),
        _ptr(loss_out), _ptr(row_stats), _ptr(grad_output), g_ptrs, g_lds, gdt, _ptr(status), _stream(stream)))


def vce_gemm_bf16(A, B, a_mn=False, b_mn=False, *, C=None, stream=None):
    """C = A(m,k) B(n,k) on the tensor cores; A [M,K] or [K,M] (a_mn), B [N,K] or [K,N] (b_mn), bf16."""
    M = A.shape[1] if a_mn else A.shape[0]
    K = A.shape[0] if a_mn else A.shape[1]
    N = B.shape[1] if b_mn else B.shape[0]
    if C is None:
        C = torch.empty(M, N, dtype=torch.float32, device=A.device)
    _check("vce_gemm_bf16", _get().vce_gemm_bf16(_ptr(A), int(a_mn), _ptr(B), int(b_mn), M, N, K, _ptr(C),
                                              C.stride(0), _stream(stream)))
    return C


def vce_gemm_bf16_variant(A, B, a_mn=False, b_mn=False, *, pair=0, C=None, stream=None):
    """vce_gemm_bf16 in a chosen launch form: pair 0 single CTAs, 1 CTA pairs (256-row tiles),
    2 CTA pairs with two K blocks per pipeline stage."""
    M = A.shape[1] if a_mn else A.shape[0]
    K = A.shape[0] if a_mn else A.shape[1]
    N = B.shape[1] if b_mn else B.shape[0]
    if C is None:
        C = torch.empty(M, N, dtype=torch.float32, device=A.device)
    _check("vce_gemm_bf16_variant", _get().vce_gemm_bf16_variant(
        _ptr(A), int(a_mn), _ptr(B), int(b_mn), M, N, K, _ptr(C), C.stride(0), int(pair), _stream(stream)))
    return C


def vce_test_gemm_stall(A, B, wait_ns=50_000_000, *, stream=None):
    """Run the GEMM pipeline with a stage that never completes; returns the device status word."""
    M, K = A.shape
    N = B.shape[0]
    C = torch.empty(M, N, dtype=torch.float32, device=A.device)
    status = torch.empty(1, dtype=torch.int32, device=A.device)
    _check("vce_test_gemm_stall", _get().vce_test_gemm_stall(_ptr(A), _ptr(B), M, N, K, _ptr(C), int(wait_ns),
                                                          _ptr(status), _stream(stream)))
    return vce_get_status(status, stream)


def vce_test_gemm_skip(A, B, skip_bits, *, stream=None):
    """C = A B^T over the 128-column K blocks whose bit is set for each 128-row M tile;
    skip_bits an int32 device tensor [ceil(M/128), words]."""
    M, K = A.shape
    N = B.shape[0]
    C = torch.empty(M, N, dtype=torch.float32, device=A.device)
    _check("vce_test_gemm_skip", _get().vce_test_gemm_skip(_ptr(A), _ptr(B), M, N, K, _ptr(skip_bits),
                                                        skip_bits.shape[1], _ptr(C), _stream(stream)))
    return C


def vce_test_ce_fwd_stall(logits, labels, wait_ns=50_000_000, *, stream=None):
    """Run ce_forward's stage-ring kernel with stages that never complete; returns the device
    status word (written by the kernel itself: filled with garbage first)."""
    T, V = logits.shape
    dev = logits.device
    loss_rows = torch.empty(T, dtype=torch.float32, device=dev)
    row_stats = torch.empty(T, ROW_STATS, dtype=torch.float32, device=dev)
    loss_out = torch.empty(1, dtype=torch.float32, device=dev)
    status = torch.full((1,), 0x7FFF1234, dtype=torch.int32, device=dev)
    _check("vce_test_ce_fwd_stall", _get().vce_test_ce_fwd_stall(
        _ptr(logits), T, V, _ptr(labels), _ptr(loss_rows), _ptr(row_stats), _ptr(loss_out), int(wait_ns),
        _ptr(status), _stream(stream)))
    return vce_get_status(status, stream)


def vce_test_ce_fused_stall(logits, labels, wait_ns=50_000_000, *, stream=None):
    """Run the one-pass shared-memory kernel with stages that never complete; returns the device
    status word."""
    T, V = logits.shape
    dev = logits.device
    go = torch.ones(1, dtype=torch.float32, device=dev)
    loss_rows = torch.empty(T, dtype=torch.float32, device=dev)
    row_stats = torch.empty(T, ROW_STATS, dtype=torch.float32, device=dev)
    grad = torch.empty_like(logits)
    status = torch.empty(1, dtype=torch.int32, device=dev)
    _check("vce_test_ce_fused_stall", _get().vce_test_ce_fused_stall(
        _ptr(logits), T, V, _ptr(labels), _ptr(go), _ptr(loss_rows), _ptr(row_stats), _ptr(grad), int(wait_ns),
        _ptr(status), _stream(stream)))
    return vce_get_status(status, stream)


def linear_ce_workspace_bytes(T, D, V) -> int:
    return int(_get().linear_ce_workspace_bytes(T, D, V))


def linear_ce_fwd_bwd(E, W, labels, ignore_index=IGNORE_INDEX, reduction="mean", *, grad_output=None,
                      grad_dtype=None, dE=None, dW=None, loss_rows=None, loss_out=None, workspace=None,
                      status=None, stream=None):
    """Fused linear-CE: loss of softmax(E W^T) and the gradients dE, dW.

    Returns (loss_out, loss_rows, dE, dW, status).
    """
    return _linear_ce(E, W, labels, ignore_index, reduction, grad_output, grad_dtype, dE, dW, loss_rows, loss_out,
                      workspace, status, stream, None, None)


def linear_ce_fwd_bwd_filtered(E, W, labels, filter_eps, ignore_index=IGNORE_INDEX, reduction="mean", *,
                               grad_output=None, grad_dtype=None, dE=None, dW=None, loss_rows=None, loss_out=None,
                               workspace=None, kept_blocks=None, status=None, stream=None):
    """linear_ce_fwd_bwd with gradient filtering at threshold filter_eps (128 x 128 blocks of G).

    Returns (loss_out, loss_rows, dE, dW, status, kept_blocks), kept_blocks a device int64 [1]
    with the number of blocks kept.
    """
    if kept_blocks is None:
        kept_blocks = torch.empty(1, dtype=torch.int64, device=E.device)
    out = _linear_ce(E, W, labels, ignore_index, reduction, grad_output, grad_dtype, dE, dW, loss_rows, loss_out,
                     workspace, status, stream, float(filter_eps), kept_blocks)
    return out + (kept_blocks,)


GEMM_KINDS = ("statistics", "gradient_tiles", "dW", "dE")


def linear_ce_fwd_bwd_timed(E, W, labels, filter_eps=0.0, ignore_index=IGNORE_INDEX, reduction="mean", *,
                            grad_output=None, grad_dtype=None, dE=None, dW=None, loss_rows=None, loss_out=None,
                            workspace=None, kept_blocks=None, status=None, stream=None):
    """linear_ce_fwd_bwd(_filtered) with CUDA events around each GEMM launch (blocking).

    Returns ((loss_out, loss_rows, dE, dW, status), {kind: (milliseconds, launches)}) for the
    GEMM kinds in GEMM_KINDS.
    """
    ms = (ctypes.c_float * 4)()
    n = (ctypes.c_int * 4)()
    out = _linear_ce(E, W, labels, ignore_index, reduction, grad_output, grad_dtype, dE, dW, loss_rows, loss_out,
                     workspace, status, stream, float(filter_eps), kept_blocks, timed=(ms, n))
    return out, {k: (float(ms[i]), int(n[i])) for i, k in enumerate(GEMM_KINDS)}


def _linear_ce(E, W, labels, ignore_index, reduction, grad_output, grad_dtype, dE, dW, loss_rows, loss_out,
               workspace, status, stream, filter_eps, kept_blocks, timed=None):
    T, D = E.shape
    V = W.shape[0]
    dev = E.device
    gdt = grad_dtype or E.dtype
    dE = torch.empty(T, D, dtype=gdt, device=dev) if dE is None else dE
    dW = torch.empty(V, D, dtype=gdt, device=dev) if dW is None else dW
    loss_rows = torch.empty(T, dtype=torch.float32, device=dev) if loss_rows is None else loss_rows
    if reduction != "none" and loss_out is None:
        loss_out = torch.empty(1, dtype=torch.float32, device=dev)
    if grad_output is None:
        grad_output = torch.ones(T if reduction == "none" else 1, dtype=torch.float32, device=dev)
    status = torch.empty(1, dtype=torch.int32, device=dev) if status is None else status
    need = linear_ce_workspace_bytes(T, D, V)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    if timed is not None:
        _check("linear_ce_fwd_bwd_timed", _get().linear_ce_fwd_bwd_timed(
            _ptr(E), _ptr(W), T, D, V, _ptr(labels), int(ignore_index), RED[reduction], _ptr(grad_output),
            _ptr(loss_rows), _ptr(loss_out), _ptr(dE), _ptr(dW), _dtype(dE), filter_eps, _ptr(kept_blocks),
            _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream), timed[0], timed[1]))
    elif filter_eps is None:
        _check("linear_ce_fwd_bwd", _get().linear_ce_fwd_bwd(
            _ptr(E), _ptr(W), T, D, V, _ptr(labels), int(ignore_index), RED[reduction], _ptr(grad_output),
            _ptr(loss_rows), _ptr(loss_out), _ptr(dE), _ptr(dW), _dtype(dE), _ptr(workspace), workspace.numel(),
            _ptr(status), _stream(stream)))
    else:
        _check("linear_ce_fwd_bwd_filtered", _get().linear_ce_fwd_bwd_filtered(
            _ptr(E), _ptr(W), T, D, V, _ptr(labels), int(ignore_index), RED[reduction], _ptr(grad_output),
            _ptr(loss_rows), _ptr(loss_out), _ptr(dE), _ptr(dW), _dtype(dE), filter_eps, _ptr(kept_blocks),
            _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream)))
    return loss_out, loss_rows, dE, dW, status


class _CrossEntropy(torch.autograd.Function):
    """Autograd wrapper: forward = ce_forward_ls, backward = ce_backward_ls (bf16 input is not upcast)."""

    @staticmethod
    def forward(ctx, logits, labels, ignore_index, reduction, label_smoothing):
        loss_out, loss_rows, row_stats, status = ce_forward_ls(logits, labels, label_smoothing, ignore_index,
                                                               reduction)
        ctx.save_for_backward(logits, labels, row_stats)
        ctx.ignore_index, ctx.reduction, ctx.eps = ignore_index, reduction, label_smoothing
        return loss_rows if reduction == "none" else loss_out.reshape(())

    @staticmethod
    def backward(ctx, grad):
        logits, labels, row_stats = ctx.saved_tensors
        go = grad.reshape(-1).to(torch.float32).contiguous()
        g = ce_backward_ls(logits, labels, row_stats, go, ctx.eps, ctx.ignore_index, ctx.reduction)
        return g, None, None, None, None


def cross_entropy(logits, labels, ignore_index=IGNORE_INDEX, reduction="mean", label_smoothing=0.0):
    """Collapse-safe softmax cross-entropy of [T, V] float32/bfloat16 CUDA logits with autograd."""
    return _CrossEntropy.apply(logits, labels, ignore_index, reduction, float(label_smoothing))

"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the fp64 oracle.

Nothing here computes any part of the cross-entropy: this module only draws the
logits, labels, hidden states and classifier weights of the five workloads the
library is measured and checked on, from the counter-based generator in
``vce_gen.c``.  Every matrix row is a pure function of (seed, stream, row), so a
test can regenerate just the rows it checks.

Workloads (sizes and value distributions of the pages' problems):

  tiny     T=64,    V=1000,   fp32 logits ~N(0, 3^2), 8 rows with the target
           raised to max(row)+U[20,40], 4 ignored rows
  mid      T=4096,  V=32000,  bf16 ~N(0, 2^2), 5% ignored
  pages    T=16384, V=128256, bf16 ~N(0, 2^2), 10% rows raised by U[17,50],
           1% ignored (torchtitan PR #5723, "Measured on H100, V=128256, T=16384")
  chunked  the pages' matrix cut into 8 column chunks of 16032
  linear   E [8192, 4096] ~N(0,1), W [128256, 4096] ~N(0, 0.02^2), 2% ignored;
           small case T=8191, D=128, V=32 (the Cut Cross-Entropy issue #14 toy)
  linear_peaked  the linear shapes with hidden states aligned to their targets
           (E_i = 0.5 N(0,1) + a W_{t_i}, target logit ~24 above the rest), standing in
           for a trained model's concentrated softmax
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vce_gen.c")
_LIB = os.path.join(_HERE, "libvce_gen.so")

IGNORE_INDEX = -100

# stream ids: one independent counter space per kind of draw
S_LOGITS, S_LABELS, S_PERM, S_MARGIN, S_E, S_W = 1, 2, 3, 4, 5, 6

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile vce_gen.c into libvce_gen.so next to it (plain gcc, no platform flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, f64, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.vce_gen_hash.argtypes = [u64, u64, u64]
            lib.vce_gen_hash.restype = u64
            lib.vce_gen_uniform_f64.argtypes = [u64, u64, u64, i64, f64, f64, p]
            lib.vce_gen_uniform_int.argtypes = [u64, u64, u64, i64, u64, p]
            lib.vce_gen_permutation.argtypes = [u64, u64, i64, p]
            for name in ("vce_gen_normal_rows_f32", "vce_gen_normal_rows_bf16"):
                getattr(lib, name).argtypes = [u64, u64, i64, i64, i64, i64, f64, f64, p, p, p]
            lib.vce_gen_copy_cols.argtypes = [p, i64, i64, i64, i64, i64, p, i64]
            lib.vce_gen_aligned_rows_bf16.argtypes = [u64, u64, i64, i64, i64, f64, p, p, p]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def uniform_f64(seed, stream, n, lo, hi, ctr0=0):
    out = np.empty(n, np.float64)
    _load().vce_gen_uniform_f64(seed, stream, ctr0, n, lo, hi, _ptr(out))
    return out


def uniform_int(seed, stream, n, rng, ctr0=0):
    out = np.empty(n, np.int64)
    _load().vce_gen_uniform_int(seed, stream, ctr0, n, rng, _ptr(out))
    return out


def permutation(seed, stream, n):
    out = np.empty(n, np.int64)
    _load().vce_gen_permutation(seed, stream, n, _ptr(out))
    return out


def normal_rows(seed, stream, r0, nrows, ncols, mean, std, dtype, out=None, ld=None,
                raise_col=None, raise_by=None):
    """Rows r0..r0+nrows-1 of an N(mean, std^2) [*, ncols] matrix.

    dtype 'f32' gives float32 values, 'bf16' gives the uint16 storage bits.
    """
    ld = ncols if ld is None else ld
    npdt = np.float32 if dtype == "f32" else np.uint16
    if out is None:
        out = np.empty((nrows, ld), npdt)
    assert out.dtype == npdt and out.flags.c_contiguous and out.shape[0] >= nrows
    if raise_col is not None:
        raise_col = np.ascontiguousarray(raise_col, np.int64)
        raise_by = np.ascontiguousarray(raise_by, np.float64)
    fn = _load().vce_gen_normal_rows_f32 if dtype == "f32" else _load().vce_gen_normal_rows_bf16
    fn(seed, stream, r0, nrows, ncols, ld, mean, std, _ptr(raise_col), _ptr(raise_by), _ptr(out))
    return out


def _parallel_rows(total, fn, threads=None, block=None):
    threads = threads or min(32, os.cpu_count() or 1)
    block = block or max(1, -(-total // (threads * 4)))
    starts = list(range(0, total, block))
    if len(starts) == 1 or threads == 1:
        for s in starts:
            fn(s, min(block, total - s))
        return
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda s: fn(s, min(block, total - s)), starts))


@dataclass
class CEProblem:
    """One seeded CE workload: labels and row roles are small and held; logits are drawn on demand."""
    name: str
    T: int
    V: int
    dtype: str              # 'f32' or 'bf16' storage of the logits
    seed: int
    std: float
    n_margin: int
    margin_lo: float
    margin_hi: float
    n_ignore: int
    ignore_index: int = IGNORE_INDEX
    labels: np.ndarray = field(init=False)
    margin: np.ndarray = field(init=False)       # per row: raise added to max(row), NaN if none
    margin_rows: np.ndarray = field(init=False)
    ignore_rows: np.ndarray = field(init=False)

    def __post_init__(self):
        labels = uniform_int(self.seed, S_LABELS, self.T, self.V)
        perm = permutation(self.seed, S_PERM, self.T)
        self.margin_rows = np.sort(perm[: self.n_margin])
        self.ignore_rows = np.sort(perm[self.n_margin: self.n_margin + self.n_ignore])
        self.margin = np.full(self.T, np.nan)
        if self.n_margin:
            self.margin[self.margin_rows] = uniform_f64(self.seed, S_MARGIN, self.n_margin,
                                                        self.margin_lo, self.margin_hi)
        labels[self.ignore_rows] = self.ignore_index
        self.labels = labels

    @property
    def np_dtype(self):
        return np.float32 if self.dtype == "f32" else np.uint16

    def _raise_args(self, r0, n):
        m = self.margin[r0: r0 + n]
        col = np.where(np.isnan(m), -1, self.labels[r0: r0 + n]).astype(np.int64)
        return col, np.nan_to_num(m, nan=0.0)

    def rows(self, idx) -> np.ndarray:
        """Logits storage of the given rows (float32 values or bf16 bits), shape [len(idx), V]."""
        idx = np.atleast_1d(np.asarray(idx, np.int64))
        out = np.empty((len(idx), self.V), self.np_dtype)
        for k, r in enumerate(idx):
            col, by = self._raise_args(int(r), 1)
            normal_rows(self.seed, S_LOGITS, int(r), 1, self.V, 0.0, self.std, self.dtype,
                        out=out[k: k + 1], raise_col=col, raise_by=by)
        return out

    def full(self, out: np.ndarray | None = None, threads=None) -> np.ndarray:
        """All T rows, drawn in parallel into `out` (e.g. a pinned host buffer's numpy view)."""
        if out is None:
            out = np.empty((self.T, self.V), self.np_dtype)
        assert out.shape == (self.T, self.V) and out.dtype == self.np_dtype and out.flags.c_contiguous

        def fill(r0, n):
            col, by = self._raise_args(r0, n)
            normal_rows(self.seed, S_LOGITS, r0, n, self.V, 0.0, self.std, self.dtype,
                        out=out[r0: r0 + n], raise_col=col, raise_by=by)
        _parallel_rows(self.T, fill, threads)
        return out


def copy_cols(src: np.ndarray, c0: int, w: int, out: np.ndarray | None = None, threads=None):
    """Columns [c0, c0+w) of a row-major matrix into a contiguous [rows, w] array."""
    rows = src.shape[0]
    if out is None:
        out = np.empty((rows, w), src.dtype)
    lib = _load()

    def fill(r0, n):
        lib.vce_gen_copy_cols(ctypes.c_void_p(src[r0:].ctypes.data), src.shape[1], n, c0, w,
                              src.itemsize, ctypes.c_void_p(out[r0:].ctypes.data), out.shape[1])
    _parallel_rows(rows, fill, threads)
    return out


# --- the five workloads ------------------------------------------------------------------

def tiny(seed=1001):
    return CEProblem("tiny", 64, 1000, "f32", seed, 3.0, 8, 20.0, 40.0, 4)


def mid(seed=1002):
    return CEProblem("mid", 4096, 32000, "bf16", seed, 2.0, 0, 0.0, 0.0, round(0.05 * 4096))


def pages(seed=1003):
    T = 16384
    return CEProblem("pages", T, 128256, "bf16", seed, 2.0, round(0.10 * T), 17.0, 50.0, round(0.01 * T))


CHUNKS = 8
CHUNK_WIDTH = 16032   # 8 * 16032 = 128256


def chunk_bounds(V=128256, k=CHUNKS):
    """Equal column chunks of the pages' vocabulary: list of (offset, width)."""
    w = V // k
    assert w * k == V
    return [(c * w, w) for c in range(k)]


def custom(T, V, dtype="bf16", seed=7, std=2.0, n_margin=0, margin=(17.0, 50.0), n_ignore=0):
    return CEProblem("custom", T, V, dtype, seed, std, n_margin, margin[0], margin[1], n_ignore)


@dataclass
class LinearProblem:
    """Fused linear-CE workload: E [T, D] ~N(0,1), W [V, D] ~N(0, 0.02^2), bf16, labels in [0, V).

    peak > 0 draws hidden states aligned with their targets, a stand-in for a trained model
    whose softmax is concentrated on the label: E_i = e_std * N(0, 1) + a * W_{t_i} with
    a = peak / (D * w_std^2), so the target logit sits about `peak` above the others
    (ignored rows get the noise alone).
    """
    name: str
    T: int
    D: int
    V: int
    seed: int
    n_ignore: int
    e_std: float = 1.0
    w_std: float = 0.02
    peak: float = 0.0
    ignore_index: int = IGNORE_INDEX
    labels: np.ndarray = field(init=False)
    ignore_rows: np.ndarray = field(init=False)

    def __post_init__(self):
        labels = uniform_int(self.seed, S_LABELS, self.T, self.V)
        perm = permutation(self.seed, S_PERM, self.T)
        self.ignore_rows = np.sort(perm[: self.n_ignore])
        labels[self.ignore_rows] = self.ignore_index
        self.labels = labels

    def _aligned(self, r0, n, out, W=None):
        """Rows r0..r0+n-1 of the target-aligned E (peak > 0), W the full classifier or None."""
        t = self.labels[r0: r0 + n]
        ok = (t >= 0) & (t < self.V)
        tt = np.where(ok, t, 0)
        add = np.ascontiguousarray(W[tt]) if W is not None else self.W_rows(tt)
        a = np.where(ok, self.peak / (self.D * self.w_std ** 2), 0.0).astype(np.float64)
        _load().vce_gen_aligned_rows_bf16(self.seed, S_E, r0, n, self.D, self.e_std, _ptr(add), _ptr(a),
                                          _ptr(out))
        return out

    def E_rows(self, idx):
        idx = np.atleast_1d(np.asarray(idx, np.int64))
        out = np.empty((len(idx), self.D), np.uint16)
        for k, r in enumerate(idx):
            if self.peak > 0:
                self._aligned(int(r), 1, out[k: k + 1])
            else:
                normal_rows(self.seed, S_E, int(r), 1, self.D, 0.0, self.e_std, "bf16", out=out[k: k + 1])
        return out

    def W_rows(self, idx):
        idx = np.atleast_1d(np.asarray(idx, np.int64))
        out = np.empty((len(idx), self.D), np.uint16)
        for k, r in enumerate(idx):
            normal_rows(self.seed, S_W, int(r), 1, self.D, 0.0, self.w_std, "bf16", out=out[k: k + 1])
        return out

    def E(self, out=None, threads=None, W=None):
        """All of E; with peak > 0 the classifier W (bf16 bits) is drawn first unless given."""
        out = np.empty((self.T, self.D), np.uint16) if out is None else out
        if self.peak > 0:
            W = self.W(threads=threads) if W is None else W
            _parallel_rows(self.T, lambda r0, n: self._aligned(r0, n, out[r0: r0 + n], W), threads)
            return out
        _parallel_rows(self.T, lambda r0, n: normal_rows(self.seed, S_E, r0, n, self.D, 0.0, self.e_std,
                                                         "bf16", out=out[r0: r0 + n]), threads)
        return out

    def W(self, out=None, threads=None):
        out = np.empty((self.V, self.D), np.uint16) if out is None else out
        _parallel_rows(self.V, lambda r0, n: normal_rows(self.seed, S_W, r0, n, self.D, 0.0, self.w_std,
                                                         "bf16", out=out[r0: r0 + n]), threads)
        return out


def linear(seed=1005):
    T = 8192
    return LinearProblem("linear", T, 4096, 128256, seed, round(0.02 * T))


def linear_small(seed=1005):
    T = 8191
    return LinearProblem("linear_small", T, 128, 32, seed, round(0.02 * T))


def linear_custom(T, D, V, seed=11, n_ignore=0, e_std=1.0, w_std=0.02, peak=0.0):
    return LinearProblem("linear_custom", T, D, V, seed, n_ignore, e_std, w_std, peak)


def linear_peaked(seed=1006):
    """The linear workload's shapes with target-aligned hidden states (noise std 0.5, the
    target logit ~24 above the rest): a concentrated softmax for gradient filtering."""
    T = 8192
    return LinearProblem("linear_peaked", T, 4096, 128256, seed, round(0.02 * T), 0.5, 0.02, 24.0)

"""fp64 CPU oracle for the vocabulary cross-entropy library.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check of ``__graft_entry__``
and the CPU-baseline leg of ``bench.py`` may import this module.  The library's
product path never calls it and shares no code with it: it has its own input
decoding, its own arithmetic and its own rounding helpers.

What it computes is the plain definition of softmax cross-entropy,
    loss_i = -log softmax(z_i)_{t_i},   dloss/dz_ij = c_i * (softmax(z_i)_j - [j == t_i]),
arranged the way the torchtitan page (PR #5723, "[loss] fix softmax collapse with
improved ce perf", Numerics section) arranges it, so that fp64 itself never
collapses: the target is left out of the log-sum-exp and the loss is
    loss_i = softplus(logsumexp_{j != t} z_ij - z_it) = log(1 + sum_{j != t} e^{z_ij - z_it}),
which is -log p_t exactly.  With x = L' - z_t (L' the target-excluded log-sum-exp):
    p_non_target = sigmoid(x),   p_j = exp(z_j - L') * sigmoid(x) for j != t,
    p_t - 1 = -sigmoid(x).
The page's branch between p_t - 1 and -p_non_target is an fp32 device: in fp64
both are -sigmoid(x) to ~1e-16, so the oracle takes -sigmoid(x) (stable form).

Readings where the pages leave a step open:
  * ignored rows (label == ignore_index, -100 by default) give loss 0 and gradient
    +0.0 by selection, whatever the logits hold (torchtitan page: "Ignored labels
    act as targets on no shard ... zeroed by the label mask");
  * a label outside [0, V) that is not ignore_index is an error;
  * reduction 'mean' divides by the number of non-ignored rows N (0/0 = NaN when
    N = 0, with all gradients 0); c_i = grad_output / N; 'sum' gives c_i =
    grad_output; 'none' takes a per-row grad_output;
  * the target-excluded maximum over an empty set is -inf and its sum is 0.

Vocabulary-chunked statistics follow the Megatron-core page
(core.tensor_parallel.cross_entropy: calculate_logits_max, gather_predicted_logits,
the all-reduce over the tensor-parallel group): each chunk gives its own
(max, sum-exp, target logit if it owns the target) over its non-target columns and
the merge rescales the sums to the global maximum.

The fused linear-CE follows the Cut Cross-Entropy issue #14 page
(linear_cross_entropy(e, c, targets), no bias; impl="cce_exact": no gradient
filtering): logits z = E W^T, then the CE above, then dE = G W and dW = G^T E.
The same page names gradient filtering as what "cce_exact" turns off and gives no rule for
it; linear_ce_filtered states the block rule this library takes (see there).
"""
from __future__ import annotations

import numpy as np

IGNORE_INDEX = -100


# ----------------------------------------------------------------------------------------
# input decoding (the oracle's own; the CUDA path decodes on the device)

def widen(storage: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of stored logits: 'f32' float32 values or 'bf16' uint16 bits."""
    if dtype == "f32":
        return np.asarray(storage, np.float32).astype(np.float64)
    if dtype == "bf16":
        bits = np.asarray(storage, np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


# ----------------------------------------------------------------------------------------
# scalar functions in fp64

def softplus(x):
    """log(1 + e^x), evaluated without overflow for large x and without loss for small."""
    x = np.asarray(x, np.float64)
    with np.errstate(over="ignore"):
        return np.where(x > 0, x + np.log1p(np.exp(-np.abs(x))), np.log1p(np.exp(np.minimum(x, 0.0))))


def sigmoid(x):
    """1 / (1 + e^-x) in the form that keeps relative accuracy on both tails."""
    x = np.asarray(x, np.float64)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


# ----------------------------------------------------------------------------------------
# per-row statistics and the CE forward / backward

def check_labels(labels: np.ndarray, V: int, ignore_index: int = IGNORE_INDEX) -> np.ndarray:
    """Boolean mask of valid rows; raises on a label that is neither ignored nor in [0, V)."""
    labels = np.asarray(labels, np.int64)
    valid = labels != ignore_index
    bad = valid & ((labels < 0) | (labels >= V))
    if bad.any():
        raise ValueError(f"label out of range at rows {np.nonzero(bad)[0][:8].tolist()}")
    return valid


def target_excluded_stats(z: np.ndarray, cols: np.ndarray):
    """Per row: (max over j != t of z_j, sum over j != t of e^{z_j - max}, z_t).

    `cols` holds each row's target column inside `z`, or -1 when the row's target is
    not among these columns (then every column counts and z_t is NaN).
    The maximum of an empty or all -inf set is -inf with a sum of 0.
    """
    z = np.asarray(z, np.float64)
    n, V = z.shape
    cols = np.asarray(cols, np.int64)
    owned = cols >= 0
    zm = z.copy()
    rows = np.nonzero(owned)[0]
    zt = np.full(n, np.nan)
    zt[rows] = z[rows, cols[rows]]
    zm[rows, cols[rows]] = -np.inf                      # drop the target column
    m = zm.max(axis=1) if V > 0 else np.full(n, -np.inf)
    finite = np.isfinite(m)
    s = np.zeros(n)
    with np.errstate(invalid="ignore"):
        e = np.exp(zm[finite] - m[finite, None])
    s[finite] = e.sum(axis=1)
    return m, s, zt


def ce_rows(z: np.ndarray, labels: np.ndarray, ignore_index: int = IGNORE_INDEX):
    """Row-wise forward: dict with loss, x = L' - z_t, L' (target-excluded LSE), valid mask.

    Ignored rows: loss 0, x = -inf, L' = -inf.  (torchtitan PR #5723, Numerics)
    """
    z = np.asarray(z, np.float64)
    n, V = z.shape
    valid = check_labels(labels, V, ignore_index)
    cols = np.where(valid, labels, -1)
    m, s, zt = target_excluded_stats(z, cols)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse_nt = np.where(s > 0, m + np.log(s), -np.inf)
        x = lse_nt - zt
    x = np.where(valid, x, -np.inf)
    lse_nt = np.where(valid, lse_nt, -np.inf)
    loss = np.where(valid, softplus(x), 0.0)
    return {"loss": loss, "x": x, "lse_nt": lse_nt, "zt": np.where(valid, zt, np.nan), "valid": valid,
            "max_nt": np.where(valid, m, -np.inf), "sum_nt": np.where(valid, s, 0.0)}


def row_scale(valid: np.ndarray, reduction: str, grad_output) -> np.ndarray:
    """c_i: the factor of row i's gradient for reduction 'mean', 'sum' or 'none'."""
    valid = np.asarray(valid, bool)
    if reduction == "none":
        g = np.broadcast_to(np.asarray(grad_output, np.float64), valid.shape)
        return np.where(valid, g, 0.0)
    g = float(np.asarray(grad_output, np.float64).reshape(-1)[0])
    if reduction == "sum":
        return np.where(valid, g, 0.0)
    if reduction == "mean":
        N = int(valid.sum())
        return np.where(valid, g / N, 0.0) if N else np.zeros(valid.shape)
    raise ValueError(reduction)


def reduce_loss(loss: np.ndarray, valid: np.ndarray, reduction: str):
    if reduction == "none":
        return np.asarray(loss, np.float64)
    total = float(np.sum(np.where(valid, loss, 0.0)))
    if reduction == "sum":
        return total
    N = int(np.sum(valid))
    return total / N if N else float("nan")


def ce_grad_rows(z: np.ndarray, labels: np.ndarray, fwd: dict, c: np.ndarray) -> np.ndarray:
    """grad_ij = c_i * p_ij for j != t, and c_i * (p_t - 1) = -c_i * sigmoid(x) at j = t.

    p_ij = exp(z_ij - L') * sigmoid(x) (torchtitan PR #5723: softmax minus one-hot, with the
    target entry taken from the non-target mass).  Ignored rows are +0.0 by selection.
    """
    z = np.asarray(z, np.float64)
    valid = fwd["valid"]
    p_nt = sigmoid(fwd["x"])
    L = fwd["lse_nt"]
    g = np.zeros_like(z)
    rows = np.nonzero(valid)[0]
    if len(rows):
        zr = z[rows]
        Lr = L[rows]
        fin = np.isfinite(Lr)
        p = np.zeros_like(zr)
        with np.errstate(invalid="ignore", over="ignore"):
            p[fin] = np.exp(zr[fin] - Lr[fin, None]) * p_nt[rows][fin, None]
        cr = np.asarray(c, np.float64)[rows]
        gr = cr[:, None] * p
        t = np.asarray(labels, np.int64)[rows]
        gr[np.arange(len(rows)), t] = -cr * p_nt[rows]
        g[rows] = gr
    return g


def ce(z, labels, reduction="mean", grad_output=1.0, ignore_index=IGNORE_INDEX, want_grad=True):
    """Whole CE forward (+ backward) on a small [T, V] float64 matrix.

    Returns dict: loss_rows, loss (reduced), grad (if want_grad), x, lse_nt, valid, c.
    """
    fwd = ce_rows(z, labels, ignore_index)
    out = dict(fwd)
    out["loss_rows"] = fwd["loss"]
    out["loss_out"] = reduce_loss(fwd["loss"], fwd["valid"], reduction)
    out["c"] = row_scale(fwd["valid"], reduction, grad_output)
    if want_grad:
        out["grad"] = ce_grad_rows(z, labels, fwd, out["c"])
    return out


# ----------------------------------------------------------------------------------------
# label smoothing (Megatron-core vocab_parallel_cross_entropy: label_smoothing in [0, 1))
#
# The page gives the argument and its range only.  Reading taken: the target distribution
# is the one-hot mixed with the uniform distribution over all V classes,
#     q = (1 - eps) onehot(t) + eps / V,
#     loss = -sum_j q_j log p_j = (1 - eps) (-log p_t) + eps (LSE(z) - mean_j z_j),
#     dloss/dz_j = c (p_j - q_j).
# -log p_t and p_j are taken from the collapse-safe forms above; LSE(z) over all columns is
# max(z_t, L') + softplus(-|z_t - L'|).

def ce_smoothed(z, labels, eps, reduction="mean", grad_output=1.0, ignore_index=IGNORE_INDEX, want_grad=True):
    """CE with label smoothing eps: dict with loss_rows, loss_out, grad (and the plain CE fields)."""
    z = np.asarray(z, np.float64)
    V = z.shape[1]
    out = ce(z, labels, reduction, grad_output, ignore_index, want_grad)
    valid = out["valid"]
    x, L = out["x"], out["lse_nt"]
    zt = out["zt"]
    with np.errstate(invalid="ignore", over="ignore"):
        hi = np.maximum(zt, L)
        lse_all = np.where(np.isneginf(L), zt, np.where(np.isneginf(zt), L, hi + softplus(-np.abs(x))))
        mean_z = z.mean(axis=1)
        loss = (1.0 - eps) * out["loss"] + eps * (lse_all - mean_z)
    loss = np.where(valid, loss, 0.0)
    out["loss"] = out["loss_rows"] = loss
    out["loss_out"] = reduce_loss(loss, valid, reduction)
    if want_grad:
        g = out["grad"]                     # c (p - onehot), rows of ignored labels are 0
        c = out["c"]
        shift = np.where(valid, c * eps / V, 0.0)
        g = g - shift[:, None]
        rows = np.nonzero(valid)[0]
        g[rows, np.asarray(labels, np.int64)[rows]] += c[rows] * eps
        out["grad"] = g
    return out


# ----------------------------------------------------------------------------------------
# vocabulary-chunked statistics and their merge (Megatron-core cross_entropy page)

def chunk_stats(z_chunk: np.ndarray, labels: np.ndarray, offset: int, ignore_index=IGNORE_INDEX):
    """Statistics of one column chunk covering global columns [offset, offset + width).

    Returns (m_c, s_c, owner, zt_c): the max and sum-exp over the chunk's non-target
    columns, whether the chunk holds the row's target, and the target logit if so.
    Ignored rows own nothing ("act as targets on no shard").
    """
    z_chunk = np.asarray(z_chunk, np.float64)
    w = z_chunk.shape[1]
    labels = np.asarray(labels, np.int64)
    owner = (labels != ignore_index) & (labels >= offset) & (labels < offset + w)
    cols = np.where(owner, labels - offset, -1)
    m, s, zt = target_excluded_stats(z_chunk, cols)
    return m, s, owner, zt


def merge_chunk_stats(stats, labels, V, ignore_index=IGNORE_INDEX):
    """Combine per-chunk (m_c, s_c, owner, zt_c) into the row forward of `ce_rows`.

    M = max_c m_c;  S = sum_c s_c e^{m_c - M} over chunks with m_c > -inf;  z_t from the
    single owning chunk.  The rescale to a common maximum is what an all-reduce of the
    per-rank statistics does on the Megatron-core page.
    """
    valid = check_labels(labels, V, ignore_index)
    ms = np.stack([s[0] for s in stats])
    ss = np.stack([s[1] for s in stats])
    own = np.stack([s[2] for s in stats])
    zts = np.stack([s[3] for s in stats])
    if np.any(own.sum(axis=0)[valid] != 1):
        raise ValueError("every valid row needs exactly one owning chunk")
    M = ms.max(axis=0)
    S = np.zeros_like(M)
    for c in range(ms.shape[0]):
        ok = ms[c] > -np.inf
        S[ok] += ss[c, ok] * np.exp(ms[c, ok] - M[ok])
    zt = np.where(own, zts, 0.0).sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse_nt = np.where(S > 0, M + np.log(S), -np.inf)
        x = lse_nt - zt
    x = np.where(valid, x, -np.inf)
    lse_nt = np.where(valid, lse_nt, -np.inf)
    loss = np.where(valid, softplus(x), 0.0)
    return {"loss": loss, "x": x, "lse_nt": lse_nt, "zt": np.where(valid, zt, np.nan), "valid": valid,
            "max_nt": np.where(valid, M, -np.inf), "sum_nt": np.where(valid, S, 0.0)}


def ce_chunked(chunks, offsets, labels, V, reduction="mean", grad_output=1.0, ignore_index=IGNORE_INDEX):
    """CE over logits given as column chunks; returns the merged forward and per-chunk grads."""
    stats = [chunk_stats(zc, labels, off, ignore_index) for zc, off in zip(chunks, offsets)]
    fwd = merge_chunk_stats(stats, labels, V, ignore_index)
    c = row_scale(fwd["valid"], reduction, grad_output)
    grads = []
    p_nt = sigmoid(fwd["x"])
    for zc, off in zip(chunks, offsets):
        zc = np.asarray(zc, np.float64)
        g = np.zeros_like(zc)
        rows = np.nonzero(fwd["valid"])[0]
        L = fwd["lse_nt"][rows]
        fin = np.isfinite(L)
        p = np.zeros((len(rows), zc.shape[1]))
        p[fin] = np.exp(zc[rows][fin] - L[fin, None]) * p_nt[rows][fin, None]
        gr = c[rows, None] * p
        t = np.asarray(labels, np.int64)[rows]
        mine = (t >= off) & (t < off + zc.shape[1])
        gr[np.nonzero(mine)[0], t[mine] - off] = -c[rows][mine] * p_nt[rows][mine]
        g[rows] = gr
        grads.append(g)
    out = dict(fwd)
    out.update(stats=stats, loss_rows=fwd["loss"], loss_out=reduce_loss(fwd["loss"], fwd["valid"], reduction),
               c=c, grads=grads)
    return out


# ----------------------------------------------------------------------------------------
# fused linear cross-entropy (Cut Cross-Entropy issue #14: linear_cross_entropy(e, c, targets))

def linear_logits(E: np.ndarray, W: np.ndarray) -> np.ndarray:
    """z = E W^T in float64; products of bf16 values are exact in fp64."""
    return np.asarray(E, np.float64) @ np.asarray(W, np.float64).T


def linear_ce(E, W, labels, reduction="mean", grad_output=1.0, ignore_index=IGNORE_INDEX):
    """Loss, dE = G W and dW = G^T E for the fused linear-CE, G the CE gradient of z = E W^T."""
    E = np.asarray(E, np.float64)
    W = np.asarray(W, np.float64)
    z = linear_logits(E, W)
    r = ce(z, labels, reduction, grad_output, ignore_index)
    G = r["grad"]
    r["dE"] = G @ W
    r["dW"] = G.T @ E
    r["z"] = z
    return r


def linear_ce_row_forward(E, W, labels, ignore_index=IGNORE_INDEX, block=256):
    """Row forward (loss, x, L', valid) of the linear-CE for many rows, `block` rows of z at a time."""
    E = np.asarray(E, np.float64)
    W = np.asarray(W, np.float64)
    T = E.shape[0]
    parts = []
    for r0 in range(0, T, block):
        parts.append(ce_rows(E[r0: r0 + block] @ W.T, labels[r0: r0 + block], ignore_index))
    return {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}


def linear_ce_grad_columns(E, W, labels, fwd, c, cols, ignore_index=IGNORE_INDEX):
    """G[:, cols] for all rows: the CE gradient restricted to a set of vocabulary columns."""
    E = np.asarray(E, np.float64)
    Wc = np.asarray(W, np.float64)[cols]
    z = E @ Wc.T                                       # [T, len(cols)]
    valid = fwd["valid"]
    p_nt = sigmoid(fwd["x"])
    L = fwd["lse_nt"]
    G = np.zeros_like(z)
    rows = np.nonzero(valid & np.isfinite(L))[0]
    G[rows] = np.asarray(c)[rows, None] * np.exp(z[rows] - L[rows, None]) * p_nt[rows, None]
    labels = np.asarray(labels, np.int64)
    for k, j in enumerate(cols):
        hit = np.nonzero(valid & (labels == j))[0]
        G[hit, k] = -np.asarray(c)[hit] * p_nt[hit]
    return G


# ----------------------------------------------------------------------------------------
# gradient filtering of the fused linear-CE (Cut Cross-Entropy issue #14: impl="cce_exact"
# is the variant that disables it; the page states no rule)
#
# Reading taken: G is cut into blocks of `block` rows by `block` vocabulary columns, aligned
# at row 0 and column 0 (block = 128 in the library).  A block is dropped -- its entries count
# as 0 in dE = G W and dW = G^T E -- when no valid row of it has its target among the block's
# columns and every non-target probability p_ij of its valid rows is below eps.  Kept blocks
# keep their exact entries.  The loss and the statistics are not filtered.

def filter_blocks(z, labels, eps, block=128, ignore_index=IGNORE_INDEX):
    """keep[rb, cb] for the blocks of G, with the blocks' largest non-target probability
    (0 where a block has no valid row) and whether a block holds a valid row's target."""
    z = np.asarray(z, np.float64)
    T, V = z.shape
    fwd = ce_rows(z, labels, ignore_index)
    valid = fwd["valid"]
    labels = np.asarray(labels, np.int64)
    nr, nc = -(-T // block), -(-V // block)
    pmax = np.zeros((nr, nc))
    has_t = np.zeros((nr, nc), bool)
    starts = np.arange(0, V, block)
    pnt = sigmoid(fwd["x"])
    for i in np.nonzero(valid)[0]:
        p = np.zeros(V)
        if np.isfinite(fwd["lse_nt"][i]):
            p = np.exp(z[i] - fwd["lse_nt"][i]) * pnt[i]   # p_j, j != t (collapse-safe form)
        p[labels[i]] = 0.0
        rb = i // block
        pmax[rb] = np.maximum(pmax[rb], np.maximum.reduceat(p, starts))
        has_t[rb, labels[i] // block] = True
    return has_t | (pmax >= eps), pmax, has_t


def linear_ce_filtered(E, W, labels, eps, reduction="mean", grad_output=1.0, ignore_index=IGNORE_INDEX,
                       block=128):
    """linear_ce with gradient filtering: dE and dW from G with its dropped blocks zeroed."""
    E = np.asarray(E, np.float64)
    W = np.asarray(W, np.float64)
    r = linear_ce(E, W, labels, reduction, grad_output, ignore_index)
    keep, pmax, has_t = filter_blocks(r["z"], labels, eps, block, ignore_index)
    T, V = r["z"].shape
    mask = np.repeat(np.repeat(keep, block, axis=0), block, axis=1)[:T, :V]
    Gf = np.where(mask, r["grad"], 0.0)
    r["dE"] = Gf @ W
    r["dW"] = Gf.T @ E
    r["keep"], r["block_pmax"], r["block_target"] = keep, pmax, has_t
    return r


def filter_blocks_columns(E, W, labels, fwd, cols, eps, block=128, ignore_index=IGNORE_INDEX):
    """The filter's keep decision for one column block -- `cols`, the columns of that block --
    in every row block, from the row forward `fwd` of the whole matrix (linear_ce_row_forward):
    the column-sampled form of filter_blocks, for matrices too large to form z."""
    E = np.asarray(E, np.float64)
    z = E @ np.asarray(W, np.float64)[cols].T                      # [T, len(cols)]
    labels = np.asarray(labels, np.int64)
    valid = fwd["valid"]
    L = fwd["lse_nt"]
    live = valid & np.isfinite(L)
    p = np.zeros_like(z)
    p[live] = np.exp(z[live] - L[live, None]) * sigmoid(fwd["x"][live])[:, None]
    tgt = (labels[:, None] == np.asarray(cols)[None, :]) & valid[:, None]
    p[tgt] = 0.0
    starts = np.arange(0, z.shape[0], block)
    pmax = np.maximum.reduceat(p.max(axis=1), starts)
    has_t = np.logical_or.reduceat(tgt.any(axis=1), starts)
    return has_t | (pmax >= eps), pmax, has_t

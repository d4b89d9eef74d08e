"""Pins of the gradient-filtering oracle (linear_ce_filtered, Cut Cross-Entropy issue #14:
the filtering that impl="cce_exact" turns off, with the block rule this library states).

The filtered oracle reduces to the exact linear-CE at eps = 0 and keeps exactly the blocks
holding a target once eps exceeds every probability. On tiny shapes it agrees with a brute
force written from the plain softmax definition. It moves dE and dW by no more than the
dropped entries can. Each planted mistake at the end must make one of these fail.
"""
import math

import numpy as np
import pytest

import gen
from oracle import ce_oracle as O


def _problem(T, D, V, seed, n_ignore=2, peak=0.0, e_std=1.0, w_std=0.3):
    p = gen.linear_custom(T, D, V, seed=seed, n_ignore=n_ignore, e_std=e_std, w_std=w_std, peak=peak)
    W = p.W()
    E = p.E(W=W)
    return p, O.widen(E, "bf16"), O.widen(W, "bf16")


def _brute(E, W, labels, eps, block, reduction):
    """Plain loops: p_ij = e^{z_ij} / sum_k e^{z_ik}, G_ij = c (p_ij - [j == t_i]), a block kept
    when one of its valid rows has its target in it or a non-target p_ij >= eps."""
    T, D = E.shape
    V = W.shape[0]
    valid = [int(t) != gen.IGNORE_INDEX for t in labels]
    n = sum(valid)
    c = 1.0 / n if reduction == "mean" else 1.0
    G = [[0.0] * V for _ in range(T)]
    P = [[0.0] * V for _ in range(T)]
    for i in range(T):
        if not valid[i]:
            continue
        z = [sum(float(E[i, d]) * float(W[j, d]) for d in range(D)) for j in range(V)]
        mx = max(z)
        ex = [math.exp(v - mx) for v in z]
        s = sum(ex)
        for j in range(V):
            P[i][j] = ex[j] / s
            G[i][j] = c * (P[i][j] - (1.0 if j == int(labels[i]) else 0.0))
    nr, nc = -(-T // block), -(-V // block)
    keep = [[False] * nc for _ in range(nr)]
    pmax = [[0.0] * nc for _ in range(nr)]
    for i in range(T):
        if not valid[i]:
            continue
        t = int(labels[i])
        keep[i // block][t // block] = True
        for j in range(V):
            if j != t:
                pmax[i // block][j // block] = max(pmax[i // block][j // block], P[i][j])
                if P[i][j] >= eps:
                    keep[i // block][j // block] = True
    Gf = [[G[i][j] if keep[i // block][j // block] else 0.0 for j in range(V)] for i in range(T)]
    dE = [[sum(Gf[i][j] * float(W[j, d]) for j in range(V)) for d in range(D)] for i in range(T)]
    dW = [[sum(Gf[i][j] * float(E[i, d]) for i in range(T)) for d in range(D)] for j in range(V)]
    return np.array(keep), np.array(pmax), np.array(dE), np.array(dW)


def _eps_in_a_gap(values, lo_q=0.3):
    """An eps between two block maxima at least 2% apart, near the lo_q quantile, so no block's
    decision hangs on the last bits of its probability."""
    v = np.unique(np.asarray(values)[np.asarray(values) > 0])
    start = int(lo_q * (len(v) - 1))
    for k in range(start, len(v) - 1):
        if v[k + 1] > 1.02 * v[k]:
            return math.sqrt(v[k] * v[k + 1])
    raise AssertionError("no gap between block maxima")


@pytest.mark.parametrize("block", [8, 128])
def test_eps_zero_is_the_exact_linear_ce(block):
    p, E, W = _problem(70, 12, 50, 21)
    f = O.linear_ce_filtered(E, W, p.labels, 0.0, "sum", block=block)
    r = O.linear_ce(E, W, p.labels, "sum")
    assert np.array_equal(f["dE"], r["dE"]) and np.array_equal(f["dW"], r["dW"])
    assert np.array_equal(f["loss"], r["loss"])


def test_eps_above_every_probability_keeps_only_target_blocks():
    p, E, W = _problem(64, 10, 90, 22, n_ignore=5)
    f = O.linear_ce_filtered(E, W, p.labels, 1.5, "mean", block=16)
    want = np.zeros_like(f["keep"])
    for i, t in enumerate(p.labels):
        if t != gen.IGNORE_INDEX:
            want[i // 16, t // 16] = True
    assert np.array_equal(f["keep"], want)
    assert 0 < want.sum() < want.size


@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_brute_force_on_tiny_shapes(reduction):
    p, E, W = _problem(11, 3, 14, 23, n_ignore=2, peak=5.0, e_std=1.0, w_std=0.5)
    _, pm, _, _ = _brute(E, W, p.labels, 2.0, 4, reduction)
    eps = _eps_in_a_gap(pm)
    keep, pmax, dE, dW = _brute(E, W, p.labels, eps, 4, reduction)
    f = O.linear_ce_filtered(E, W, p.labels, eps, reduction, block=4)
    assert np.array_equal(f["keep"], keep)
    assert 0 < keep.sum() < keep.size          # the rule drops some blocks and keeps others
    np.testing.assert_allclose(f["block_pmax"], pmax, rtol=1e-12, atol=0)
    np.testing.assert_allclose(f["dE"], dE, rtol=1e-10, atol=1e-15)
    np.testing.assert_allclose(f["dW"], dW, rtol=1e-10, atol=1e-15)


def test_dropped_entries_bound_the_change():
    """|dW_f - dW| <= eps sum_i |c_i| |E_id| and |dE_f - dE| <= eps |c_i| sum_v |W_vd|: every
    dropped entry is c_i p_ij with p_ij < eps."""
    p, E, W = _problem(96, 16, 300, 24, n_ignore=3, w_std=0.6)
    probe = O.linear_ce_filtered(E, W, p.labels, 2.0, "mean", block=8)
    eps = _eps_in_a_gap(probe["block_pmax"], 0.5)
    f = O.linear_ce_filtered(E, W, p.labels, eps, "mean", block=8)
    r = O.linear_ce(E, W, p.labels, "mean")
    assert 0 < f["keep"].sum() < f["keep"].size
    c = np.where(r["valid"], 1.0 / r["valid"].sum(), 0.0)
    bound_dW = eps * (np.abs(c)[:, None] * np.abs(E)).sum(0)              # [D], for every v
    bound_dE = eps * np.abs(c)[:, None] * np.abs(W).sum(0)[None, :]        # [T, D]
    assert np.all(np.abs(f["dW"] - r["dW"]) <= bound_dW[None, :] * (1 + 1e-12))
    assert np.all(np.abs(f["dE"] - r["dE"]) <= bound_dE * (1 + 1e-12))
    assert np.abs(f["dW"] - r["dW"]).max() > 0   # filtering did change something


def test_column_sampled_decisions_match_the_full_ones():
    """filter_blocks_columns (one column block at a time, from the row forward) gives the
    column of filter_blocks' keep table for every column block, ragged last block included."""
    p, E, W = _problem(100, 12, 70, 25, n_ignore=4, peak=4.0, w_std=0.5)
    fwd = O.linear_ce_row_forward(E, W, p.labels, block=32)
    z = E @ W.T
    probe, pm, _ = O.filter_blocks(z, p.labels, 2.0, block=16)
    eps = _eps_in_a_gap(pm, 0.5)
    keep, pmax, has_t = O.filter_blocks(z, p.labels, eps, block=16)
    assert 0 < keep.sum() < keep.size
    for cb in range(keep.shape[1]):
        cols = np.arange(16 * cb, min(16 * cb + 16, 70))
        k, m, h = O.filter_blocks_columns(E, W, p.labels, fwd, cols, eps, block=16)
        assert np.array_equal(k, keep[:, cb]) and np.array_equal(h, has_t[:, cb])
        np.testing.assert_allclose(m, pmax[:, cb], rtol=1e-12, atol=0)


# ---------------------------------------------------------------- planted mistakes

def _must_fail(*checks):
    for chk in checks:
        try:
            chk()
        except AssertionError:
            return
    pytest.fail("no pin caught the planted mistake")


def test_mistake_target_blocks_not_kept(monkeypatch):
    real = O.filter_blocks

    def wrong(z, labels, eps, block=128, ignore_index=O.IGNORE_INDEX):
        keep, pmax, has_t = real(z, labels, eps, block, ignore_index)
        return pmax >= eps, pmax, has_t
    monkeypatch.setattr(O, "filter_blocks", wrong)
    _must_fail(test_eps_above_every_probability_keeps_only_target_blocks)


def test_mistake_probability_without_the_sigmoid(monkeypatch):
    """p_ij taken as exp(z_ij - L') (the share among non-targets), dropping the sigma(x) factor."""
    real_sigmoid = O.sigmoid
    real = O.filter_blocks

    def wrong(z, labels, eps, block=128, ignore_index=O.IGNORE_INDEX):
        monkeypatch.setattr(O, "sigmoid", lambda x: np.ones_like(np.asarray(x, np.float64)))
        try:
            return real(z, labels, eps, block, ignore_index)
        finally:
            monkeypatch.setattr(O, "sigmoid", real_sigmoid)
    monkeypatch.setattr(O, "filter_blocks", wrong)
    _must_fail(lambda: test_brute_force_on_tiny_shapes("mean"))


def test_mistake_rows_assigned_to_the_wrong_block(monkeypatch):
    real = O.filter_blocks

    def wrong(z, labels, eps, block=128, ignore_index=O.IGNORE_INDEX):
        keep, pmax, has_t = real(np.asarray(z)[::-1], np.asarray(labels)[::-1], eps, block, ignore_index)
        return keep[::-1], pmax[::-1], has_t[::-1]
    monkeypatch.setattr(O, "filter_blocks", wrong)
    _must_fail(lambda: test_brute_force_on_tiny_shapes("sum"))


def test_mistake_mask_on_the_wrong_axis(monkeypatch):
    """The dropped-block mask applied to G transposed block-wise (row block <-> column block)."""
    real = O.filter_blocks

    def wrong(z, labels, eps, block=128, ignore_index=O.IGNORE_INDEX):
        keep, pmax, has_t = real(z, labels, eps, block, ignore_index)
        k = np.zeros_like(keep)
        n = min(keep.shape)
        k[:n, :n] = keep[:n, :n].T
        return k, pmax, has_t
    monkeypatch.setattr(O, "filter_blocks", wrong)
    _must_fail(lambda: test_brute_force_on_tiny_shapes("mean"))

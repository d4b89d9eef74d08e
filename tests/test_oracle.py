"""Pins of the fp64 oracle against things other than itself (no GPU needed).

closed forms (uniform rows, one raised target), 60-digit decimal brute force, torch's
CPU float64 cross_entropy + autograd where fp64 does not collapse, invariants, chunk
consistency, the linear-CE reducing to the CE, and the pages' stated constants.
Each is chosen so that a plausible slip in the oracle (a dropped term, a sign, an
index, a transposed operand) fails at least one of them.
"""
import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

import gen
from oracle import ce_oracle as O
from oracle import rounding as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.abs(a - b) / np.maximum(np.abs(b), 1e-300)


# ---------------------------------------------------------------- closed form P-a: uniform rows

@pytest.mark.parametrize("V", [1, 2, 3, 1000, 32000, 128256])
@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_uniform_rows_closed_form(V, reduction):
    T = 3
    z = np.full((T, V), 1.75)
    labels = np.array([0, V - 1, V // 2])
    r = O.ce(z, labels, reduction, grad_output=2.0)
    np.testing.assert_allclose(r["loss_rows"], math.log(V), rtol=1e-13, atol=0 if V > 1 else 1e-300)
    c = 2.0 / T if reduction == "mean" else 2.0
    want = np.full((T, V), c / V)
    want[np.arange(T), labels] = c * (1.0 / V - 1.0)
    np.testing.assert_allclose(r["grad"], want, rtol=1e-12, atol=1e-300)


# ---------------------------------------------------------------- closed form P-b: one raised target

@pytest.mark.parametrize("V", [2, 1000, 128256])
@pytest.mark.parametrize("m", [0.0, 5.0, 16.6, 17.0, 30.0, 50.0, 80.0])
def test_margin_row_closed_form(V, m):
    base = -0.3
    t = 7 % V
    z = np.full((1, V), base)
    z[0, t] = base + m
    r = O.ce(z, np.array([t]), "sum")
    q = (V - 1) * math.exp(-m)
    assert _rel(r["loss_rows"][0], math.log1p(q)) < 1e-13
    g = r["grad"][0]
    assert _rel(g[t], -q / (1 + q)) < 1e-13
    others = np.delete(g, t)
    np.testing.assert_allclose(others, math.exp(-m) / (1 + q), rtol=1e-12)
    assert r["loss_rows"][0] > 0 and g[t] < 0    # never collapses, even at m = 80


def test_margin_row_target_position_matters():
    """A target index read one column off would give the loss of a non-target column."""
    V, m = 50, 9.0
    z = np.zeros((1, V))
    z[0, 11] = m
    right = O.ce(z, np.array([11]), "sum")["loss_rows"][0]
    wrong = O.ce(z, np.array([12]), "sum")["loss_rows"][0]
    assert _rel(right, math.log1p((V - 1) * math.exp(-m))) < 1e-13
    assert _rel(wrong, m + math.log1p((V - 1) * math.exp(-m))) < 1e-12


# ---------------------------------------------------------------- brute force P-d (decimal, 400 digits)

def _decimal_ce(z_row, t):
    # the loss of a row with margin m is ~e^-m: at m = 700 that is 1e-304 against 1, so the
    # working precision must exceed 304 digits for ln(sum) - z_t to keep 60 of them
    getcontext().prec = 400
    zs = [Decimal(float(v)) for v in z_row]       # exact binary values
    ex = [v.exp() for v in zs]
    tot = sum(ex, Decimal(0))
    loss = tot.ln() - zs[t]
    grad = [e / tot for e in ex]
    grad[t] -= 1
    return loss, grad


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_brute_force_decimal(seed):
    rng = np.random.default_rng(seed)
    T, V = 16, 8
    z = rng.normal(0, 3, (T, V))
    labels = rng.integers(0, V, T)
    margins = [0.0, 1.0, 10.0, 16.64, 25.0, 40.0, 100.0, 300.0, 700.0]
    for i, mg in enumerate(margins):
        z[i, labels[i]] = z[i].max() + mg
    labels[len(margins)] = O.IGNORE_INDEX
    r = O.ce(z, labels, "sum")
    for i in range(T):
        if labels[i] == O.IGNORE_INDEX:
            assert r["loss_rows"][i] == 0.0 and np.all(r["grad"][i] == 0.0)
            continue
        loss, grad = _decimal_ce(z[i], labels[i])
        assert _rel(r["loss_rows"][i], float(loss)) < 1e-13, (i, r["loss_rows"][i], loss)
        np.testing.assert_allclose(r["grad"][i], [float(g) for g in grad], rtol=1e-12, atol=0)


# ---------------------------------------------------------------- library special case P-e

@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("V", [5, 1000, 32000])
def test_against_torch_float64(reduction, V):
    # torch forms p_t - 1 by subtraction, which in fp64 keeps ~1e-16 / (1 - p_t) relative
    # accuracy; margins up to 10 keep that below 1e-11, so the comparison is fair
    g = gen.custom(64, V, "f32", seed=5, std=3.0, n_margin=6, margin=(3.0, 10.0), n_ignore=5)
    z = O.widen(g.full(), "f32")
    zt = torch.tensor(z, requires_grad=True)
    lab = torch.tensor(g.labels)
    loss = torch.nn.functional.cross_entropy(zt, lab, ignore_index=O.IGNORE_INDEX, reduction=reduction)
    go = np.linspace(0.5, 1.5, 64) if reduction == "none" else 1.3
    loss.backward(torch.tensor(go) if reduction == "none" else torch.tensor(go, dtype=torch.float64))
    r = O.ce(z, g.labels, reduction, grad_output=go)
    if reduction == "none":
        # torch's logsumexp - z_t carries an absolute error of a few eps * |logits|
        np.testing.assert_allclose(r["loss_rows"], loss.detach().numpy(), rtol=1e-12, atol=1e-14)
    else:
        assert _rel(r["loss_out"], loss.item()) < 1e-12
    np.testing.assert_allclose(r["grad"], zt.grad.numpy(), rtol=1e-10, atol=1e-18)


def test_mean_with_no_valid_rows_matches_torch():
    z = np.random.default_rng(3).normal(size=(4, 9))
    labels = np.full(4, O.IGNORE_INDEX)
    r = O.ce(z, labels, "mean")
    zt = torch.tensor(z, requires_grad=True)
    loss = torch.nn.functional.cross_entropy(zt, torch.tensor(labels), ignore_index=O.IGNORE_INDEX)
    loss.backward()
    assert math.isnan(r["loss_out"]) and math.isnan(loss.item())
    assert np.all(r["grad"] == 0)
    assert np.all(np.nan_to_num(zt.grad.numpy()) == 0)


# ---------------------------------------------------------------- invariants P-c

def test_invariants_rows_sum_to_zero_and_inputs_untouched():
    g = gen.custom(128, 777, "f32", seed=9, std=4.0, n_margin=20, margin=(17.0, 60.0), n_ignore=10)
    stored = g.full()
    z = O.widen(stored, "f32")
    before = z.copy()
    r = O.ce(z, g.labels, "mean", grad_output=0.7)
    assert np.array_equal(z, before)
    rs = r["grad"].sum(axis=1)
    assert np.all(np.abs(rs) <= 1e-12 * np.maximum(np.abs(r["c"]), 1e-300) + 1e-300)
    ign = g.labels == O.IGNORE_INDEX
    assert np.all(r["grad"][ign] == 0) and np.all(r["loss_rows"][ign] == 0)
    assert np.all(np.signbit(r["grad"][ign]) == False)  # noqa: E712  (+0.0, not -0.0)
    assert np.all(r["loss_rows"][~ign] > 0)


def test_ignored_rows_with_infinities_are_exactly_zero():
    z = np.array([[np.inf, -np.inf, 3.0], [-np.inf, -np.inf, -np.inf], [1.0, 2.0, 3.0]])
    labels = np.array([O.IGNORE_INDEX, O.IGNORE_INDEX, 1])
    r = O.ce(z, labels, "mean")
    assert np.all(r["loss_rows"][:2] == 0) and np.all(r["grad"][:2] == 0)
    assert np.isfinite(r["loss_out"])


def test_non_finite_valid_rows():
    # every non-target is -inf: p_t = 1, loss 0, gradient 0; a -inf target: loss +inf, p = softmax of the rest
    z = np.array([[-np.inf, 2.0, -np.inf], [0.0, -np.inf, math.log(3.0)]])
    r = O.ce(z, np.array([1, 1]), "sum")
    assert r["loss_rows"][0] == 0.0 and np.all(r["grad"][0] == 0)
    assert r["loss_rows"][1] == np.inf
    np.testing.assert_allclose(r["grad"][1], [0.25, -1.0, 0.75], rtol=1e-15)


def test_v1_rows():
    r = O.ce(np.array([[4.0], [-2.0]]), np.array([0, 0]), "mean")
    assert np.all(r["loss_rows"] == 0) and np.all(r["grad"] == 0)


def test_invalid_label_raises():
    with pytest.raises(ValueError):
        O.ce(np.zeros((2, 4)), np.array([1, 4]), "mean")
    with pytest.raises(ValueError):
        O.ce(np.zeros((2, 4)), np.array([-1, 0]), "mean")


# ---------------------------------------------------------------- negative control P-f and the page's constant

def _naive_fp32(z_row, t):
    """The pre-fix formulation in fp32: p = softmax(z), loss = -log p_t, target gradient p_t - 1."""
    z = np.asarray(z_row, np.float32)
    e = np.exp(z - z.max())
    p_t = e[t] / np.sum(e, dtype=np.float32)
    return np.float32(-np.log(p_t)), np.float32(p_t - np.float32(1))


def _naive_fp32_loss(z_row, t):
    return _naive_fp32(z_row, t)[0]


def test_collapse_constant_from_the_pages():
    pin = json.load(open(os.path.join(GOLDEN, "pages_constants.json")))["collapse_margin"]["value"]
    onset = 24 * math.log(2)   # 1 + e^-m rounds to 1 in fp32 once e^-m < 2^-24 (half an ulp of 1)
    assert abs(onset - pin) < 0.05
    for m, collapses in [(onset - 0.05, False), (onset + 0.05, True), (30.0, True), (50.0, True)]:
        z = np.array([0.0, m], np.float32)
        naive = _naive_fp32_loss(z, 1)
        assert (naive == 0.0) == collapses, (m, naive)
        r = O.ce(z[None].astype(np.float64), np.array([1]), "sum")
        assert _rel(r["loss_rows"][0], math.log1p(math.exp(-float(np.float32(m))))) < 1e-13
        assert r["grad"][0, 1] < 0


def test_naive_fp32_collapses_on_pages_margin_rows_but_oracle_does_not():
    g = gen.custom(32, 4096, "bf16", seed=21, std=2.0, n_margin=32, margin=(17.0, 50.0))
    z = O.widen(g.full(), "bf16")
    r = O.ce(z, g.labels, "sum")
    collapsed = sum(_naive_fp32_loss(z[i], g.labels[i]) == 0.0 for i in range(32))
    assert collapsed >= 16                      # the old formulation loses most of these rows
    assert np.all(r["loss_rows"] > 0) and np.all(r["loss_rows"] < 1e-6)
    tgt = r["grad"][np.arange(32), g.labels]
    assert np.all(tgt < 0)


def test_target_branch_threshold_is_ln3():
    """p_t < 1/4 exactly when x = L' - z_t > ln 3 (the page's branch point)."""
    pin = json.load(open(os.path.join(GOLDEN, "pages_constants.json")))["target_branch_p_t"]["value"]
    for x in [math.log(3) - 1e-9, math.log(3) + 1e-9]:
        p_t = float(O.sigmoid(-x))
        assert (p_t < pin) == (x > math.log(3))


# ---------------------------------------------------------------- chunk consistency P-g

@pytest.mark.parametrize("widths", [[7, 9, 1, 15], [32], [1, 1, 30], [16, 16]])
def test_chunked_equals_unchunked(widths):
    V = sum(widths)
    g = gen.custom(40, V, "f32", seed=31, std=3.0, n_margin=8, margin=(20.0, 45.0), n_ignore=4)
    z = O.widen(g.full(), "f32")
    offs = np.cumsum([0] + widths[:-1])
    chunks = [z[:, o: o + w] for o, w in zip(offs, widths)]
    full = O.ce(z, g.labels, "mean", grad_output=1.5)
    ch = O.ce_chunked(chunks, offs, g.labels, V, "mean", grad_output=1.5)
    np.testing.assert_allclose(ch["loss_rows"], full["loss_rows"], rtol=1e-14, atol=0)
    np.testing.assert_allclose(np.concatenate(ch["grads"], axis=1), full["grad"], rtol=1e-13, atol=0)
    # the merged maximum over non-target columns is exactly the unchunked one
    v = full["valid"]
    assert np.array_equal(ch["max_nt"][v], full["max_nt"][v])
    # every valid row has exactly one owner, at the right offset
    own = np.stack([s[2] for s in ch["stats"]])
    assert np.all(own.sum(0)[v] == 1) and np.all(own.sum(0)[~v] == 0)


def test_chunk_holding_only_the_target():
    z = np.array([[0.5, 2.0, -1.0]])
    ch = O.ce_chunked([z[:, :1], z[:, 1:]], [0, 1], np.array([0]), 3, "sum")
    m0, s0, own0, zt0 = ch["stats"][0]
    assert m0[0] == -np.inf and s0[0] == 0 and own0[0] and zt0[0] == 0.5
    full = O.ce(z, np.array([0]), "sum")
    np.testing.assert_allclose(ch["loss_rows"], full["loss_rows"], rtol=1e-15)


# ---------------------------------------------------------------- linear-CE P-h and torch autograd

def test_linear_ce_reduces_to_ce_and_matches_torch():
    p = gen.linear_custom(96, 24, 40, seed=4, n_ignore=3, w_std=0.3)
    E = O.widen(p.E(), "bf16")
    W = O.widen(p.W(), "bf16")
    r = O.linear_ce(E, W, p.labels, "mean")
    z = E @ W.T
    ref = O.ce(z, p.labels, "mean")
    np.testing.assert_array_equal(r["loss_rows"], ref["loss_rows"])
    Et = torch.tensor(E, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    loss = torch.nn.functional.cross_entropy(Et @ Wt.T, torch.tensor(p.labels), ignore_index=O.IGNORE_INDEX)
    loss.backward()
    assert _rel(r["loss_out"], loss.item()) < 1e-12
    np.testing.assert_allclose(r["dE"], Et.grad.numpy(), rtol=1e-9, atol=1e-15)
    np.testing.assert_allclose(r["dW"], Wt.grad.numpy(), rtol=1e-9, atol=1e-15)
    assert r["dE"].shape == E.shape and r["dW"].shape == W.shape


def test_linear_ce_invariants():
    p = gen.linear_custom(64, 16, 12, seed=6, n_ignore=2)
    E = O.widen(p.E(), "bf16")
    W = O.widen(p.W(), "bf16")
    r = O.linear_ce(E, W, p.labels, "sum")
    # each row of G sums to 0, so the columns of dW (sum over vocabulary rows) vanish
    assert np.max(np.abs(r["dW"].sum(axis=0))) < 1e-12 * np.abs(r["dW"]).sum()
    # equal classifier rows: dE = sum_j G_ij w = 0
    W2 = np.repeat(W[:1], W.shape[0], axis=0)
    r2 = O.linear_ce(E, W2, p.labels, "sum")
    assert np.max(np.abs(r2["dE"])) < 1e-13


def test_linear_ce_sampled_helpers_agree_with_full():
    p = gen.linear_custom(50, 20, 30, seed=8, n_ignore=4)
    E = O.widen(p.E(), "bf16")
    W = O.widen(p.W(), "bf16")
    full = O.linear_ce(E, W, p.labels, "mean")
    fwd = O.linear_ce_row_forward(E, W, p.labels, block=7)
    np.testing.assert_allclose(fwd["loss"], full["loss_rows"], rtol=1e-14)
    c = O.row_scale(fwd["valid"], "mean", 1.0)
    cols = np.array([0, 5, 29, 13])
    Gc = O.linear_ce_grad_columns(E, W, p.labels, fwd, c, cols)
    np.testing.assert_allclose(Gc, full["grad"][:, cols], rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(Gc.T @ E, full["dW"][cols], rtol=1e-11, atol=1e-300)


# ---------------------------------------------------------------- rounding helper used by the graders

def test_round_bf16_matches_fp32_bit_rounding_on_fp32_values():
    rng = np.random.default_rng(0)
    f = (rng.normal(size=20000) * np.exp(rng.uniform(-60, 60, 20000))).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rne = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    got = R.bf16_bits(R.round_bf16(f.astype(np.float64)))
    assert np.array_equal(got, rne)


def test_round_bf16_is_single_rounding_from_fp64():
    # bf16 spacing above 1 is 2^-7.  1 + 2^-8 + 2^-30 lies just above the midpoint and rounds up;
    # a stop in fp32 would first drop the 2^-30, leave a tie and round down to 1
    x = 1 + 2 ** -8 + 2 ** -30
    assert R.round_bf16(x) == 1 + 2 ** -7
    assert R.round_bf16(1 + 2 ** -8) == 1.0
    assert R.bf16_ulp_distance(R.bf16_bits(R.round_bf16(np.array([1.0]))), np.array([1 + 2 ** -6]))[0] == 2

"""The error model behind the cancellation clause of the linear-CE grading (tests/test_lce_gpu),
checked on the CPU by emulating the arithmetic it describes.

  accumulation  an fp32 accumulator that adds `steps` partial sums of 16 exact products, each
                rounded to fp32 -- to nearest, or toward zero as a truncating adder would --
                stays within steps * 2^-23 * sum |t| of the exact sum;
  G split       G_hi = RNE_bf16(g), G_lo = RNE_bf16(g - G_hi) leaves |g - G_hi - G_lo| <=
                2^-16 |g| (bf16 keeps 8 significant bits: each rounding loses up to 2^-8 of its
                argument, the residual g - G_hi is at most 2^-8 |g|);
  merge         the two-sum (s = a + x, e = (a - (s - (s - a))) + (x - (s - a))) gives
                s + e = a + x exactly, so partial products merge without adding error.
"""
import numpy as np
import pytest

from oracle import rounding as R
from tests.test_lce_gpu import ACC_ULP, G_SPLIT


def _to_f32(x, toward_zero):
    """fp64 -> fp32, to nearest, or toward zero (the float32 value not above |x|)."""
    f = np.float32(x)
    if toward_zero and abs(float(f)) > abs(x):
        f = np.nextafter(f, np.float32(0.0))
    return f


def _accumulate(terms, toward_zero):
    """The tensor core's accumulation as the model reads it: each MMA step sums 16 exact
    products (exactly, then one rounding to fp32) and adds them to the fp32 accumulator (one
    rounding)."""
    acc = np.float32(0.0)
    for k in range(0, len(terms), 16):
        part = _to_f32(float(np.sum(terms[k:k + 16], dtype=np.float64)), toward_zero)
        acc = _to_f32(float(acc) + float(part), toward_zero)
    return float(acc)


@pytest.mark.parametrize("toward_zero", [False, True])
@pytest.mark.parametrize("kind", ["random signs", "same sign", "large then small", "cancelling"])
def test_blocked_fp32_accumulation_stays_within_the_bound(kind, toward_zero):
    rng = np.random.default_rng(hash(kind) % 2**32)
    K = 4096
    if kind == "random signs":
        t = rng.standard_normal(K)
    elif kind == "same sign":
        t = np.abs(rng.standard_normal(K))
    elif kind == "large then small":
        t = np.concatenate([np.full(K // 2, 1.0), np.full(K // 2, 2.0 ** -16)])
    else:
        half = np.abs(rng.standard_normal(K // 2))
        t = np.concatenate([half, -half[::-1] * (1 + 2.0 ** -20)])
    t = np.asarray(t, np.float32).astype(np.float64)   # terms that an fp32 MMA product gives
    steps = K // 16
    got = _accumulate(t, toward_zero)
    exact = float(np.sum(t, dtype=np.float64))
    bound = steps * ACC_ULP * float(np.sum(np.abs(t)))
    assert abs(got - exact) <= bound, (kind, abs(got - exact) / bound)


def test_the_bound_is_not_loose_by_orders_of_magnitude():
    """A truncating accumulator over same-sign terms uses a sizeable share of the bound: the
    model is not padded by orders of magnitude for the adversarial case."""
    rng = np.random.default_rng(3)
    t = np.abs(rng.standard_normal(16384)).astype(np.float32).astype(np.float64)
    got = _accumulate(t, True)
    share = abs(got - float(np.sum(t))) / ((len(t) // 16) * ACC_ULP * float(np.sum(np.abs(t))))
    assert 0.05 < share <= 1.0, share


def test_hi_lo_split_is_exact_to_2_pow_minus_16():
    rng = np.random.default_rng(5)
    g = (rng.standard_normal(200000) * np.exp(rng.uniform(-60, 5, 200000))).astype(np.float32).astype(np.float64)
    hi = R.round_bf16(g)
    lo = R.round_bf16(np.asarray(g - hi, np.float32).astype(np.float64))   # the residual is exact in fp32
    err = np.abs(g - hi - lo)
    assert np.all(err <= G_SPLIT * np.abs(g))
    assert np.max(err / np.abs(g)) > G_SPLIT / 4   # and it is reached within a factor 4


def test_two_sum_merge_is_exact():
    rng = np.random.default_rng(7)
    a = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32)
    s = a + x
    bp = s - a
    e = (a - (s - bp)) + (x - bp)
    assert np.array_equal(s.astype(np.float64) + e.astype(np.float64), a.astype(np.float64) + x.astype(np.float64))

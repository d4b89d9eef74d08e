"""The oracle's pins have teeth: plant a plausible mistake in the oracle, the pins must fail.

Each case monkeypatches one oracle function with a wrong variant (a dropped term, a sign,
an index, a missing rescale, a wrong divisor, a missing mask) and runs the pin tests of
test_oracle.py that should catch it.
"""
import numpy as np
import pytest

import gen
from oracle import ce_oracle as O
from tests import test_gen as TG
from tests import test_oracle as TO


def _must_fail(*checks):
    for chk in checks:
        try:
            chk()
        except (AssertionError, ValueError, IndexError):
            return
    pytest.fail("no pin caught the planted mistake")


def test_dropped_log1p_term(monkeypatch):
    monkeypatch.setattr(O, "softplus", lambda x: np.maximum(np.asarray(x, np.float64), 0.0))
    _must_fail(lambda: TO.test_margin_row_closed_form(1000, 30.0))


def test_target_left_in_the_sum(monkeypatch):
    real = O.target_excluded_stats

    def keep_target(z, cols):
        m, s, zt = real(z, np.full(len(cols), -1))
        rows = np.nonzero(np.asarray(cols) >= 0)[0]
        zt = np.full(len(cols), np.nan)
        zt[rows] = np.asarray(z, np.float64)[rows, np.asarray(cols)[rows]]
        return m, s, zt
    monkeypatch.setattr(O, "target_excluded_stats", keep_target)
    _must_fail(lambda: TO.test_uniform_rows_closed_form(1000, "sum"))


def test_sigmoid_sign_error(monkeypatch):
    monkeypatch.setattr(O, "sigmoid", lambda x: 1.0 / (1.0 + np.exp(np.asarray(x, np.float64))))
    _must_fail(lambda: TO.test_margin_row_closed_form(1000, 5.0))


def test_target_gradient_sign(monkeypatch):
    real = O.ce_grad_rows

    def flipped(z, labels, fwd, c):
        g = real(z, labels, fwd, c)
        rows = np.nonzero(fwd["valid"])[0]
        g[rows, np.asarray(labels)[rows]] *= -1
        return g
    monkeypatch.setattr(O, "ce_grad_rows", flipped)
    _must_fail(lambda: TO.test_margin_row_closed_form(2, 5.0))


def test_target_index_off_by_one(monkeypatch):
    real = O.ce_rows
    monkeypatch.setattr(O, "ce_rows", lambda z, labels, ig=O.IGNORE_INDEX: real(
        z, np.where(np.asarray(labels) == ig, ig, (np.asarray(labels) + 1) % np.asarray(z).shape[1]), ig))
    _must_fail(lambda: TO.test_margin_row_target_position_matters())


def test_mean_over_all_rows_instead_of_valid(monkeypatch):
    real = O.row_scale

    def wrong(valid, reduction, grad_output):
        if reduction == "mean":
            return np.where(valid, float(np.asarray(grad_output).reshape(-1)[0]) / len(valid), 0.0)
        return real(valid, reduction, grad_output)
    monkeypatch.setattr(O, "row_scale", wrong)
    _must_fail(lambda: TO.test_against_torch_float64("mean", 1000))


def test_ignored_rows_not_masked(monkeypatch):
    real = O.check_labels
    monkeypatch.setattr(O, "check_labels", lambda labels, V, ig=O.IGNORE_INDEX: np.ones(len(labels), bool)
                        if np.all((np.asarray(labels) == ig) | (np.asarray(labels) >= 0)) else real(labels, V, ig))
    _must_fail(lambda: TO.test_invariants_rows_sum_to_zero_and_inputs_untouched())


def test_chunk_merge_without_rescale(monkeypatch):
    real = O.merge_chunk_stats

    def no_rescale(stats, labels, V, ig=O.IGNORE_INDEX):
        flat = [(np.full_like(m, np.max([s[0] for s in stats], axis=0)), s, own, zt) for m, s, own, zt in stats]
        return real(flat, labels, V, ig)
    monkeypatch.setattr(O, "merge_chunk_stats", no_rescale)
    _must_fail(lambda: TO.test_chunked_equals_unchunked([7, 9, 1, 15]))


def test_linear_gradient_on_the_wrong_operand(monkeypatch):
    real = O.linear_ce

    def swapped(E, W, labels, reduction="mean", grad_output=1.0, ignore_index=O.IGNORE_INDEX):
        r = real(E, W, labels, reduction, grad_output, ignore_index)
        r["dE"] = r["grad"] @ np.asarray(W, np.float64)[::-1]   # classifier rows taken in the wrong order
        return r
    monkeypatch.setattr(O, "linear_ce", swapped)
    _must_fail(lambda: TO.test_linear_ce_reduces_to_ce_and_matches_torch())


def test_bf16_decoding_shift(monkeypatch):
    monkeypatch.setattr(O, "widen", lambda storage, dtype: (np.asarray(storage, np.uint16).astype(np.uint32)
                                                            << np.uint32(15)).view(np.float32).astype(np.float64)
                        if dtype == "bf16" else np.asarray(storage, np.float32).astype(np.float64))
    _must_fail(lambda: TG.test_distribution_moments())


def test_unmutated_oracle_passes_the_same_pins():
    TO.test_margin_row_closed_form(1000, 30.0)
    TO.test_uniform_rows_closed_form(1000, "sum")
    TO.test_chunked_equals_unchunked([7, 9, 1, 15])
    TO.test_against_torch_float64("mean", 1000)
    TG.test_distribution_moments()
    assert gen.tiny().T == 64

"""Tolerances of the parity tests (CUDA path vs the fp64 oracle), in one place.

  per-row loss   relative 1e-4 on every valid row; the only exemption is a row whose
                 oracle loss is below 1e-30 while the device loss is 0 or subnormal
                 (no absolute floor: a collapsed 0 must fail on a 1e-8..1e-22 loss);
                 ignored rows exactly +0.0
  fp32 gradient  |g - o| <= 1e-6 + 1e-4 |o|, and on raised-target rows the target entry
                 is nonzero and within relative 1e-4 (the absolute term alone would let
                 a collapsed target gradient pass)
  bf16 gradient  the device bits equal RNE_bf16(o), o rounded once from fp64, or one of
                 its two bf16 neighbours
  reduced loss   relative 1e-4
  linear-CE loss the same, plus a per-row slack where the logits are fp32 sums of D bf16
                 products formed on the tensor cores (tests/test_lce_gpu.z_sum_slack): a
                 row's loss moves by sigma(x) |dx|, and with a large target margin the loss
                 is ~e^x, so its relative error is the absolute error of x itself
"""
import numpy as np

from oracle import rounding as R

LOSS_RTOL = 1e-4
G32_ATOL, G32_RTOL = 1e-6, 1e-4


def check_loss_rows(got, want, valid, what="loss", slack=None):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    valid = np.asarray(valid, bool)
    assert np.all(got[~valid] == 0.0) and not np.any(np.signbit(got[~valid])), f"{what}: ignored rows not +0"
    g, w = got[valid], want[valid]
    exempt = (np.abs(w) < 1e-30) & ((g == 0) | (np.abs(g) < np.finfo(np.float32).tiny))
    if slack is not None:
        exempt |= np.abs(g - w) <= LOSS_RTOL * np.abs(w) + np.asarray(slack, np.float64)[valid]
    rel = np.abs(g - w) / np.maximum(np.abs(w), 1e-300)
    bad = (~exempt) & ~(rel <= LOSS_RTOL) & ~((g == w) & np.isinf(w))
    assert not bad.any(), (f"{what}: {bad.sum()} rows beyond rel {LOSS_RTOL}; worst rel "
                           f"{np.nanmax(np.where(bad, rel, 0)):.3e} at {np.nonzero(bad)[0][:5]}")
    return float(np.max(np.where(exempt | ~np.isfinite(rel), 0, rel))) if len(rel) else 0.0


def check_grad_f32(got, want, what="grad"):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    err = np.abs(got - want)
    tol = G32_ATOL + G32_RTOL * np.abs(want)
    bad = ~(err <= tol)
    assert not bad.any(), f"{what}: {bad.sum()} entries out of tolerance, worst {np.max(err - tol):.3e}"


def check_target_entries(got, want, what="target grad"):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert np.all(got != 0), f"{what}: collapsed (exact zero) target gradient"
    rel = np.abs(got - want) / np.abs(want)
    assert np.all(rel <= 1e-4), f"{what}: worst rel {rel.max():.3e}"


def check_grad_bf16(got_bits, want, what="grad"):
    d = R.bf16_ulp_distance(np.asarray(got_bits).view(np.uint16), want)
    bad = d > 1
    assert not bad.any(), f"{what}: {bad.sum()} entries beyond one bf16 ulp (max {d.max()})"
    return int(d.max()) if d.size else 0


def bf16_tensor_bits(t):
    """Host uint16 bits of a torch bfloat16 tensor."""
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def check_reduced(got, want, what="reduced loss", slack=0.0):
    if np.isnan(want):
        assert np.isnan(got), f"{what}: expected NaN, got {got}"
        return
    assert abs(got - want) <= LOSS_RTOL * abs(want) + slack, f"{what}: {got} vs {want}"

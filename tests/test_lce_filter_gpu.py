"""Parity of the gradient-filtered linear-CE (linear_ce_fwd_bwd_filtered through the C ABI)
with the filtered fp64 oracle (128 x 128 blocks of G dropped when they hold no target and
every non-target probability is below eps).

Hidden states aligned with their targets give a concentrated softmax, so a good share of
blocks drop.  eps is taken in a gap of at least 2% between the oracle's block maxima, so no
keep decision rests on the last bits of a probability; the count of kept blocks must then be
exact, and dE / dW are graded as the unfiltered outputs are, against the filtered oracle.
"""
import numpy as np
import pytest
import torch

import gen
from oracle import ce_oracle as O
from tests import _grading as G
from tests.test_ce_gpu import vce  # noqa: F401  (fixture)
from tests.test_lce_gpu import dev_bf16, grade_sum, host
from tests.test_oracle_filter import _eps_in_a_gap

pytestmark = pytest.mark.gpu


def _inputs(p):
    Wb = p.W()
    Eb = p.E(W=Wb)
    return Eb, Wb


def _run(vce, Eb, Wb, p, eps, reduction="mean", grad_dtype=torch.bfloat16):
    labels = torch.from_numpy(p.labels).cuda()
    E, W = dev_bf16(Eb), dev_bf16(Wb)
    lo, lr, dE, dW, st, kept = vce.linear_ce_fwd_bwd_filtered(E, W, labels, eps, reduction=reduction,
                                                              grad_dtype=grad_dtype)
    torch.cuda.synchronize()
    assert vce.vce_get_status(st) == 0
    return lo, lr, dE, dW, int(kept.item())


# T=300: odd row tiles (dE on single CTAs), ragged T and V, most rows ignored so that blocks
# without a target exist; V=20000: two vocabulary chunks, dE on CTA pairs; V=16768: a second
# chunk of 384 columns
@pytest.mark.parametrize("T,D,V,peak,reduction,n_ignore", [(300, 192, 1000, 8.0, "mean", 280),
                                                           (512, 128, 20000, 9.0, "sum", 5),
                                                           (256, 64, 16768, 7.0, "mean", 5)])
def test_filtered_matches_the_filtered_oracle(vce, T, D, V, peak, reduction, n_ignore):
    p = gen.linear_custom(T, D, V, seed=T + V, n_ignore=n_ignore, e_std=0.5, w_std=0.05, peak=peak)
    Eb, Wb = _inputs(p)
    E, W = O.widen(Eb, "bf16"), O.widen(Wb, "bf16")
    probe = O.linear_ce_filtered(E, W, p.labels, 2.0, reduction)
    eps = _eps_in_a_gap(probe["block_pmax"], 0.5)
    ref = O.linear_ce_filtered(E, W, p.labels, eps, reduction)
    keep = ref["keep"]
    assert 0 < keep.sum() < keep.size
    lo, lr, dE, dW, kept = _run(vce, Eb, Wb, p, eps, reduction)
    assert kept == int(keep.sum()), f"kept {kept} blocks, the rule keeps {int(keep.sum())}"
    G.check_loss_rows(lr.cpu().numpy(), ref["loss_rows"], ref["valid"])
    G.check_reduced(lo.item(), ref["loss_out"])
    mask = np.repeat(np.repeat(keep, 128, 0), 128, 1)[:T, :V]
    aG = np.abs(np.where(mask, ref["grad"], 0.0))
    grade_sum(host(dE), ref["dE"], aG @ np.abs(W), "dE")
    grade_sum(host(dW), ref["dW"], aG.T @ np.abs(E), "dW")


def test_fp32_gradients_and_per_row_grad_output(vce):
    p = gen.linear_custom(384, 96, 3000, seed=31, n_ignore=330, e_std=0.5, w_std=0.05, peak=8.0)
    Eb, Wb = _inputs(p)
    E, W = O.widen(Eb, "bf16"), O.widen(Wb, "bf16")
    go = np.linspace(-1.5, 2.0, p.T)
    probe = O.linear_ce_filtered(E, W, p.labels, 2.0, "none", grad_output=go)
    eps = _eps_in_a_gap(probe["block_pmax"], 0.4)
    ref = O.linear_ce_filtered(E, W, p.labels, eps, "none", grad_output=go)
    labels = torch.from_numpy(p.labels).cuda()
    lo, lr, dE, dW, st, kept = vce.linear_ce_fwd_bwd_filtered(
        dev_bf16(Eb), dev_bf16(Wb), labels, eps, reduction="none",
        grad_output=torch.from_numpy(go.astype(np.float32)).cuda(), grad_dtype=torch.float32)
    torch.cuda.synchronize()
    assert vce.vce_get_status(st) == 0
    assert int(kept.item()) == int(ref["keep"].sum())
    mask = np.repeat(np.repeat(ref["keep"], 128, 0), 128, 1)[:p.T, :p.V]
    aG = np.abs(np.where(mask, ref["grad"], 0.0))
    grade_sum(host(dE), ref["dE"], aG @ np.abs(W), "dE")
    grade_sum(host(dW), ref["dW"], aG.T @ np.abs(E), "dW")


def test_large_eps_keeps_only_target_blocks(vce):
    p = gen.linear_custom(260, 64, 2000, seed=33, n_ignore=4, w_std=0.05)
    Eb, Wb = _inputs(p)
    *_, kept = _run(vce, Eb, Wb, p, 0.9)
    want = {(i // 128, int(t) // 128) for i, t in enumerate(p.labels) if t != gen.IGNORE_INDEX}
    assert kept == len(want)


def test_eps_zero_is_the_unfiltered_call(vce):
    p = gen.linear_custom(200, 64, 700, seed=34, n_ignore=3, w_std=0.05)
    Eb, Wb = _inputs(p)
    labels = torch.from_numpy(p.labels).cuda()
    E, W = dev_bf16(Eb), dev_bf16(Wb)
    a = vce.linear_ce_fwd_bwd(E, W, labels)
    b = vce.linear_ce_fwd_bwd_filtered(E, W, labels, 0.0)
    torch.cuda.synchronize()
    assert torch.equal(a[2], b[2]) and torch.equal(a[3], b[3]) and torch.equal(a[1], b[1])
    assert int(b[5].item()) == 0


@pytest.mark.parametrize("eps", [float("nan"), -1e-3, float("inf")])
def test_invalid_eps_is_refused(vce, eps):
    p = gen.linear_custom(16, 8, 10, seed=35)
    Eb, Wb = _inputs(p)
    labels = torch.from_numpy(p.labels).cuda()
    with pytest.raises(vce.VceError):
        vce.linear_ce_fwd_bwd_filtered(dev_bf16(Eb), dev_bf16(Wb), labels, eps)

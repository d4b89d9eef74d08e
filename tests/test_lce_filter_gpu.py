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
from tests.test_lce_gpu import dev_bf16, grade_sum, host, lce_steps, z_sum_slack
from tests.test_oracle_filter import _eps_in_a_gap


def filtered_steps(T, V):
    """Accumulation steps of the filtered gradient GEMMs (dW over all of T in one launch)."""
    return lce_steps(T, V, filtered=True)


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


# T=300: odd row tiles, ragged T and V, most rows ignored so that blocks without a target
# exist; V=40000: two vocabulary chunks of the 32768-column chunking; V=33152: a second chunk
# of 384 columns
@pytest.mark.parametrize("T,D,V,peak,reduction,n_ignore", [(300, 192, 1000, 8.0, "mean", 280),
                                                           (384, 128, 40000, 9.0, "sum", 5),
                                                           (256, 64, 33152, 7.0, "mean", 5)])
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
    st = filtered_steps(p.T, p.V)
    grade_sum(host(dE), ref["dE"], aG @ np.abs(W), "dE", steps=st["dE"])
    grade_sum(host(dW), ref["dW"], aG.T @ np.abs(E), "dW", steps=st["dW"])


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
    st = filtered_steps(p.T, p.V)
    grade_sum(host(dE), ref["dE"], aG @ np.abs(W), "dE", steps=st["dE"])
    grade_sum(host(dW), ref["dW"], aG.T @ np.abs(E), "dW", steps=st["dW"])


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


def test_full_size_peaked_sampled(vce):
    """E [8192, 4096] aligned with the targets, W [128256, 4096], eps = 2^-12, the launch the
    bench times: every loss row; dE rows of two whole 128-row blocks and dW rows of two
    128-column blocks against the filtered oracle, keep decisions from z in fp64 (none of
    them within a factor 2 of eps)."""
    p = gen.linear_peaked()
    Wb = p.W()
    Eb = p.E(W=Wb)
    eps = 2.0 ** -12
    labels = torch.from_numpy(p.labels).cuda()
    lo, lr, dE, dW, st, kept = vce.linear_ce_fwd_bwd_filtered(dev_bf16(Eb), dev_bf16(Wb), labels, eps)
    torch.cuda.synchronize()
    assert vce.vce_get_status(st) == 0
    E, W = O.widen(Eb, "bf16"), O.widen(Wb, "bf16")
    fwd = O.linear_ce_row_forward(E, W, p.labels, block=512)
    # losses ~e^-21: their relative error is the absolute error of x, which the fp32 sums of
    # 4096 products forming z carry (z_t ~ 24); z_sum_slack bounds it
    slack = z_sum_slack(E, W, p.labels, fwd)
    G.check_loss_rows(lr.cpu().numpy(), fwd["loss"], fwd["valid"], "full-size loss rows", slack=slack)
    N = int(fwd["valid"].sum())
    G.check_reduced(lo.item(), float(fwd["loss"][fwd["valid"]].sum()) / N, slack=float(slack.sum()) / N)
    c = O.row_scale(fwd["valid"], "mean", 1.0)
    rng = np.random.default_rng(9)
    aW = np.abs(W)
    kept_rows = []
    for rb in (3, 41):   # dE: whole row blocks, so the keep decisions are those of the full matrix
        rows = np.arange(128 * rb, 128 * rb + 128)
        z = E[rows] @ W.T
        keep, pmax, _ = O.filter_blocks(z, p.labels[rows], eps, 128)
        assert np.all((pmax < eps / 2) | (pmax > 2 * eps))
        kept_rows.append(int(keep.sum()))
        sub = {k: v[rows] for k, v in fwd.items()}
        Gr = O.ce_grad_rows(z, p.labels[rows], sub, c[rows])
        Gf = np.where(np.repeat(keep[0], 128)[None, :p.V], Gr, 0.0)
        pick = np.sort(rng.choice(128, 24, replace=False))
        grade_sum(host(dE[torch.from_numpy(rows[pick]).cuda()]), Gf[pick] @ W, np.abs(Gf[pick]) @ aW,
                  f"full-size dE rows of block {rb}", steps=filtered_steps(p.T, p.V)["dE"])
    assert 0 < min(kept_rows) and max(kept_rows) < -(-p.V // 128)
    for cb in (int(p.labels[p.labels >= 0][0]) // 128, 7):   # a block holding a target, and block 7
        cols = np.arange(128 * cb, min(128 * cb + 128, p.V))
        keep, pmax, _ = O.filter_blocks_columns(E, W, p.labels, fwd, cols, eps, 128)
        assert np.all((pmax < eps / 2) | (pmax > 2 * eps))
        Gc = O.linear_ce_grad_columns(E, W, p.labels, fwd, c, cols)
        Gf = np.where(np.repeat(keep, 128)[:p.T, None], Gc, 0.0)
        pick = np.sort(rng.choice(len(cols), 16, replace=False))
        grade_sum(host(dW[torch.from_numpy(cols[pick]).cuda()]), Gf[:, pick].T @ E, np.abs(Gf[:, pick]).T @ np.abs(E),
                  f"full-size dW rows of column block {cb}", steps=filtered_steps(p.T, p.V)["dW"])
    assert 0 < int(kept.item()) < -(-p.T // 128) * -(-p.V // 128)


@pytest.mark.parametrize("eps", [0.0, 2.0 ** -12])
def test_all_rows_ignored(vce, eps):
    """Every label ignored: the mean is 0/0 = NaN, every loss row 0, dE = dW = 0.  Filtered, no
    block is kept, so every dW and dE tile takes the zero-accumulator epilogue, and the dE merge
    adds zero partials across both vocabulary chunks."""
    p = gen.linear_custom(256, 64, 40000, seed=36, w_std=0.05)
    Eb, Wb = _inputs(p)
    labels = torch.full((p.T,), -100, dtype=torch.int64, device="cuda")
    lo, lr, dE, dW, st, kept = vce.linear_ce_fwd_bwd_filtered(dev_bf16(Eb), dev_bf16(Wb), labels, eps)
    torch.cuda.synchronize()
    assert vce.vce_get_status(st) == 0
    assert np.isnan(lo.item()) and torch.all(lr == 0)
    assert torch.all(dE == 0) and torch.all(dW == 0)
    assert int(kept.item()) == 0

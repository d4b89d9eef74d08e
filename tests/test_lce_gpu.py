"""Parity of the fused linear-CE (linear_ce_fwd_bwd through the C ABI) with the fp64 oracle.

dE and dW are sums o = sum_k t_k of T or V products t_k = G_k X_k.  They are graded as bf16
outputs against the oracle rounded once to bf16 (one ulp).  An entry whose sum cancels (a
large condition number sum_k |t_k| / |o|) may instead be within the error the arithmetic of
the tensor-core path can carry, beta * sum_k |t_k| plus half a bf16 ulp of its own rounding:

  accumulation   each fp32 accumulator adds `steps` MMA partial sums (16 products each), one
                 rounding per addition, counted as a whole fp32 ulp (2^-23) so that a
                 truncating adder is covered: steps * 2^-23.  The partials of separate
                 launches are merged with a two-sum, so `steps` is that of one launch: dW is
                 two launches over the halves of T (steps = 2 (T / 2) / 16, G's hi and lo
                 halves both), dE one launch per 32768-column vocabulary chunk (steps =
                 2 chunk / 16); the filtered call's dW is one launch over all of T.
  G split        G enters as G_hi + G_lo, each a rounding to 8 significant bits (bf16, unit
                 roundoff 2^-8): |g - G_hi - G_lo| <= 2^-16 |g| per term.
  G evaluation   each G entry is an fp32 product of c, sigma(x) and a hardware exp2: 2^-20.

Each grading prints how many entries needed the clause, their condition numbers, and the
largest share of the bound any of them used.
"""
import numpy as np
import pytest
import torch

import gen
from oracle import ce_oracle as O
from oracle import rounding as R
from tests import _grading as G
from tests.test_ce_gpu import vce  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu

ACC_ULP = 2.0 ** -23       # one fp32 ulp per accumulation step
G_SPLIT = 2.0 ** -16       # G = G_hi + G_lo: two roundings to bf16 (2^-8 each, compounded)
G_EVAL = 2.0 ** -20        # fp32 evaluation of a G entry
CHUNK = 32768              # vocabulary columns per gradient chunk
Z_SLACK_REL = 2.0 ** -14   # fp32 tensor-core logits: 2 x (D / 16) x 2^-23 at D = 4096


def lce_steps(T, V, filtered=False):
    """Accumulation steps of one launch of each gradient GEMM (see the module docstring)."""
    t_pad = -(-T // 128) * 128
    v_pad = -(-V // 256) * 256
    return {"dW": (2 if filtered else 1) * t_pad // 16, "dE": 2 * min(v_pad, CHUNK) // 16}


def sum_bound(steps):
    """beta: |gpu - o| <= beta * sum_k |t_k| before the output's own bf16 rounding."""
    return steps * ACC_ULP + G_SPLIT + G_EVAL


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host(t):
    if t.dtype == torch.bfloat16:
        return G.bf16_tensor_bits(t)
    return t.cpu().numpy()


def _bf16_half_ulp(v):
    """Half the bf16 spacing at |v| (8 significant bits; subnormal spacing 2^-133)."""
    v = np.abs(np.asarray(v, np.float64))
    e = np.frexp(np.where(v > 0, v, 1.0))[1]
    return 0.5 * np.ldexp(1.0, np.maximum(e - 8, -133))


def grade_sum(got, want, abs_terms, what, steps):
    """bf16 bits (or fp32 values) of a GEMM output vs the fp64 oracle and its sum of |terms|.
    Returns the report line: entries beyond one ulp (bf16) or the plain fp32 tolerance, how
    many of them only the cancellation clause passes, their condition numbers, and the largest
    share of the clause's bound they used."""
    beta = sum_bound(steps)
    want = np.asarray(want, np.float64)
    abs_terms = np.asarray(abs_terms, np.float64)
    if got.dtype == np.uint16:
        d = R.bf16_ulp_distance(got, want)
        val = O.widen(got, "bf16")
        plain = d <= 1
        slack = beta * abs_terms + _bf16_half_ulp(val)
    else:
        val = got.astype(np.float64)
        plain = np.abs(val - want) <= 1e-6 + 1e-4 * np.abs(want)
        slack = beta * abs_terms
    err = np.abs(val - want)
    within = err <= slack
    ok = plain | within
    clause = ~plain & within
    cond = abs_terms / np.maximum(np.abs(want), 1e-300)
    info = (f"{what}: {np.sum(~plain)} of {plain.size} beyond the plain bar, {np.sum(clause)} passed by the "
            f"cancellation clause (beta = {beta:.3g}, {steps} accumulation steps)")
    if clause.any():
        c = cond[clause]
        info += (f", condition numbers {c.min():.3g} .. {c.max():.3g} (median {np.median(c):.3g}), "
                 f"at most {np.max(err[clause] / slack[clause]):.2f} of the bound used")
        info += f"; plain-bar entries: median condition {np.median(cond[plain]):.3g}"
    if (~ok).any():
        info += (f"; {np.sum(~ok)} FAIL, worst |err| / sum|t| {np.max((err / abs_terms)[~ok]):.3g}"
                 f" at condition {cond[~ok][:5]}")
    print(info)
    assert ok.all(), info
    return info


def z_sum_slack(E, W, labels, fwd):
    """Per-row loss slack for logits formed as fp32 sums of D products: x = L' - z_t moves by
    at most Z_SLACK_REL (sum_d |E_id W_td| + ||E_i|| max_j ||W_j||) (the first term bounds z_t's sum,
    the second, by Cauchy-Schwarz, every z_j's and so L'), and the loss by sigma(x) times that."""
    valid = fwd["valid"]
    t = np.where(valid, np.asarray(labels), 0)
    a_t = np.einsum("ij,ij->i", np.abs(E), np.abs(W[t]))
    a_nt = np.linalg.norm(E, axis=1) * np.linalg.norm(W, axis=1).max()
    return np.where(valid, Z_SLACK_REL * O.sigmoid(fwd["x"]) * (a_t + a_nt), 0.0)


def run_lce(vce, p, reduction="mean", grad_output=1.0, grad_dtype=torch.bfloat16):
    Eb, Wb = p.E(), p.W()
    E, W = dev_bf16(Eb), dev_bf16(Wb)
    labels = torch.from_numpy(p.labels).cuda()
    go = torch.empty(p.T if reduction == "none" else 1, device="cuda")
    go[:] = torch.as_tensor(grad_output, dtype=torch.float32)
    E0, W0 = E.clone(), W.clone()
    loss_out, loss_rows, dE, dW, status = vce.linear_ce_fwd_bwd(E, W, labels, reduction=reduction, grad_output=go,
                                                                grad_dtype=grad_dtype)
    torch.cuda.synchronize()
    assert vce.vce_get_status(status) == 0
    assert torch.equal(E, E0) and torch.equal(W, W0)
    return Eb, Wb, loss_out, loss_rows, dE, dW


def full_check(vce, p, reduction="mean", grad_output=1.0, grad_dtype=torch.bfloat16):
    Eb, Wb, loss_out, loss_rows, dE, dW = run_lce(vce, p, reduction, grad_output, grad_dtype)
    E, W = O.widen(Eb, "bf16"), O.widen(Wb, "bf16")
    ref = O.linear_ce(E, W, p.labels, reduction, grad_output)
    G.check_loss_rows(loss_rows.cpu().numpy(), ref["loss_rows"], ref["valid"])
    if reduction != "none":
        G.check_reduced(loss_out.item(), ref["loss_out"])
    aG = np.abs(ref["grad"])
    st = lce_steps(p.T, p.V)
    grade_sum(host(dE), ref["dE"], aG @ np.abs(W), "dE", st["dE"])
    grade_sum(host(dW), ref["dW"], aG.T @ np.abs(E), "dW", st["dW"])


def test_pages_toy_shape(vce):
    """T=8191, D=128, V=32: the Cut Cross-Entropy issue's toy, checked in full."""
    full_check(vce, gen.linear_small())


@pytest.mark.parametrize("T,D,V", [(300, 192, 1000), (128, 64, 256), (1, 8, 1), (257, 128, 513), (1024, 512, 40000)])
def test_ragged_shapes(vce, T, D, V):
    full_check(vce, gen.linear_custom(T, D, V, seed=T + V, n_ignore=min(3, T - 1)))


@pytest.mark.parametrize("reduction", ["sum", "none"])
def test_reductions(vce, reduction):
    p = gen.linear_custom(200, 128, 700, seed=3, n_ignore=5)
    full_check(vce, p, reduction, np.linspace(0.5, 2.0, 200) if reduction == "none" else 0.5)


def test_fp32_gradients(vce):
    full_check(vce, gen.linear_custom(256, 128, 3000, seed=4, n_ignore=4), grad_dtype=torch.float32)


def test_raised_targets_do_not_collapse(vce):
    """Rows whose target logit dominates: loss ~e^-m stays nonzero, exactly as the oracle."""
    p = gen.linear_custom(64, 64, 500, seed=9, w_std=0.3)
    Eb, Wb = p.E(), p.W()
    E, W = O.widen(Eb, "bf16"), O.widen(Wb, "bf16")
    # point W's target rows along E's rows: z_t = |e|^2 / 2 ~ 32, far above the other logits
    Wm = Wb.copy()
    for i in range(0, 64, 4):
        Wm[p.labels[i]] = R.bf16_bits(R.round_bf16(0.5 * E[i]))
    p.W = lambda out=None, threads=None: Wm
    full_check(vce, p, "sum")


@pytest.mark.parametrize("V", [100, 9000])   # one statistics tile per row; 36 (merged in ranges)
def test_invalid_label(vce, V):
    p = gen.linear_custom(64, 64, V, seed=2)
    p.labels = p.labels.copy()
    p.labels[5] = V
    p.labels[7] = -100
    E, W = dev_bf16(p.E()), dev_bf16(p.W())
    out = vce.linear_ce_fwd_bwd(E, W, torch.from_numpy(p.labels).cuda())
    assert vce.vce_get_status(out[4]) == 1
    assert np.isnan(out[1][5].item())
    assert out[1][7].item() == 0.0


def test_full_size_sampled(vce):
    """E [8192, 4096], W [128256, 4096]: every loss row, 128 sampled dE rows (and 4 ignored ones)
    and 128 sampled dW rows (16 of them target columns) vs fp64."""
    p = gen.linear()
    Eb, Wb, loss_out, loss_rows, dE, dW = run_lce(vce, p)
    E, W = O.widen(Eb, "bf16"), O.widen(Wb, "bf16")
    fwd = O.linear_ce_row_forward(E, W, p.labels, block=512)          # all T rows in fp64
    G.check_loss_rows(loss_rows.cpu().numpy(), fwd["loss"], fwd["valid"], "full-size loss rows")
    N = int(fwd["valid"].sum())
    G.check_reduced(loss_out.item(), float(fwd["loss"][fwd["valid"]].sum()) / N)
    c = O.row_scale(fwd["valid"], "mean", 1.0)
    rng = np.random.default_rng(5)
    aW = np.abs(W)
    # dE rows: the full gradient row of z, times W
    rows = np.unique(np.concatenate([rng.choice(p.T, 128, replace=False), p.ignore_rows[:4]]))
    z = E[rows] @ W.T
    sub = {k: v[rows] for k, v in fwd.items()}
    Gr = O.ce_grad_rows(z, p.labels[rows], sub, c[rows])
    st = lce_steps(p.T, p.V)
    grade_sum(host(dE[torch.from_numpy(rows).cuda()]), Gr @ W, np.abs(Gr) @ aW, "full-size dE rows", st["dE"])
    # dW rows: one vocabulary column of G over all T rows, times E
    targets = np.unique(p.labels[fwd["valid"]])
    cols = np.unique(np.concatenate([rng.choice(p.V, 112, replace=False), rng.choice(targets, 16, replace=False)]))
    Gc = O.linear_ce_grad_columns(E, W, p.labels, fwd, c, cols)
    grade_sum(host(dW[torch.from_numpy(cols).cuda()]), Gc.T @ E, np.abs(Gc).T @ np.abs(E), "full-size dW rows",
              st["dW"])


@pytest.mark.parametrize("seed", range(12))
def test_random_shapes(vce, seed):
    """Randomised linear-CE shapes and options against the fp64 oracle: one or many 128-row tiles
    (single CTAs or CTA pairs), D giving an odd or an even number of 64-column K blocks (one or
    two K blocks per pipeline stage), vocabularies inside one chunk or over several, each
    reduction, bf16 or fp32 gradients, ignored rows."""
    rng = np.random.default_rng(2000 + seed)
    T = int(rng.choice([1, 100, 128, 129, 256])) if rng.random() < 0.4 else int(rng.integers(257, 1300))
    D = 8 * int(rng.choice([1, 8, 16, 24, 48, int(rng.integers(1, 97))]))
    V = int(rng.choice([1, int(rng.integers(2, 600)), int(rng.integers(600, 9000)), int(rng.integers(30000, 40000)),
                        int(rng.integers(40000, 70000))]))
    reduction = str(rng.choice(["mean", "sum", "none"]))
    gdt = torch.bfloat16 if rng.random() < 0.7 else torch.float32
    n_ignore = int(rng.integers(0, max(1, T // 5)))
    go = rng.uniform(0.25, 2.0, T) if reduction == "none" else float(rng.uniform(0.25, 2.0))
    full_check(vce, gen.linear_custom(T, D, V, seed=seed, n_ignore=n_ignore), reduction, go, gdt)

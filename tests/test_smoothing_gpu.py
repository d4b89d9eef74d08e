"""Label smoothing (ce_forward_ls / ce_backward_ls) through the C ABI vs the fp64 oracle."""
import numpy as np
import pytest
import torch

import gen
from oracle import ce_oracle as O
from oracle import rounding as R
from tests import _grading as G
from tests.test_ce_gpu import to_device, vce  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


def grade_smoothed_grad(grad_t, ref, c, eps, V, labels):
    """One bf16 ulp (or the fp32 bar), except where the smoothing term cancels the softmax
    term (p_j ~ eps/V off target, 1 - p_t ~ eps (1 - 1/V) on target): there the fp32 error of
    the two terms, 4e-6 c (|p_j| + eps/V) resp. 4e-6 c (|p_t - 1| + eps), bounds the difference."""
    want = ref["grad"]
    ac = np.abs(c)[:, None]
    rel = np.abs(want / np.where(c == 0, 1, c)[:, None])
    scale = 4e-6 * ac * (rel + 2 * eps / V)
    rows = np.nonzero(ref["valid"])[0]
    t = np.asarray(labels)[rows]
    scale[rows, t] = 4e-6 * ac[rows, 0] * (rel[rows, t] + 2 * eps)
    if grad_t.dtype == torch.bfloat16:
        bits = G.bf16_tensor_bits(grad_t)
        d = R.bf16_ulp_distance(bits, want)
        ok = (d <= 1) | (np.abs(O.widen(bits, "bf16") - want) <= scale)
    else:
        got = grad_t.cpu().numpy().astype(np.float64)
        err = np.abs(got - want)
        ok = (err <= G.G32_ATOL + G.G32_RTOL * np.abs(want)) | (err <= scale)
    assert ok.all(), f"{np.sum(~ok)} entries out of tolerance"


@pytest.mark.parametrize("V", [3001, 3008])   # per-block forward; shared-memory stage ring (16-byte rows)
@pytest.mark.parametrize("eps", [0.0, 0.1, 0.5])
@pytest.mark.parametrize("dtype,reduction", [("bf16", "mean"), ("f32", "sum"), ("bf16", "none")])
def test_smoothing_parity(vce, eps, dtype, reduction, V):
    p = gen.custom(64, V, dtype, seed=71, std=2.0, n_margin=8, margin=(17.0, 50.0), n_ignore=4)
    storage = p.full()
    logits = to_device(storage, dtype)
    labels = torch.from_numpy(p.labels).cuda()
    go_np = np.linspace(0.5, 2.0, 64) if reduction == "none" else np.array([1.25])
    go = torch.from_numpy(go_np.astype(np.float32)).cuda()
    out, rows, stats, status = vce.ce_forward_ls(logits, labels, eps, reduction=reduction)
    grad = vce.ce_backward_ls(logits, labels, stats, go, eps, reduction=reduction)
    torch.cuda.synchronize()
    assert vce.vce_get_status(status) == 0
    ref = O.ce_smoothed(O.widen(storage, dtype), p.labels, eps, reduction, go_np if reduction == "none" else 1.25)
    G.check_loss_rows(rows.cpu().numpy(), ref["loss_rows"], ref["valid"])
    if reduction != "none":
        G.check_reduced(out.item(), ref["loss_out"])
    grade_smoothed_grad(grad, ref, ref["c"], eps, p.V, p.labels)
    if eps == 0.0:   # exactly the plain calls
        o2, r2, s2, st2 = vce.ce_forward(logits, labels, reduction=reduction)
        g2 = vce.ce_backward(logits, labels, s2, go, reduction=reduction)
        assert torch.equal(rows, r2) and torch.equal(stats, s2) and torch.equal(grad, g2)


@pytest.mark.parametrize("T,V,dtype", [(2000, 3008, "bf16"), (1300, 24576, "bf16"), (600, 10000, "f32")])
def test_smoothing_forward_ring_groups(vce, T, V, dtype):
    """Many rows per CTA with the row sums of label smoothing: one warp per row (6 KB rows), the
    forward ring's two consumer groups (48 KB and 40 KB rows)."""
    eps = 0.1
    p = gen.custom(T, V, dtype, seed=T + 7, std=2.0, n_margin=T // 10, margin=(17.0, 50.0), n_ignore=T // 20)
    storage = p.full()
    logits = to_device(storage, dtype)
    labels = torch.from_numpy(p.labels).cuda()
    out, rows, stats, status = vce.ce_forward_ls(logits, labels, eps, reduction="mean")
    torch.cuda.synchronize()
    assert vce.vce_get_status(status) == 0
    ref = O.ce_smoothed(O.widen(storage, dtype), p.labels, eps, "mean", 1.0)
    G.check_loss_rows(rows.cpu().numpy(), ref["loss_rows"], ref["valid"])
    G.check_reduced(out.item(), ref["loss_out"])


def test_smoothing_rejects_bad_eps(vce):
    x = torch.zeros(2, 4, device="cuda")
    lab = torch.zeros(2, dtype=torch.int64, device="cuda")
    for bad in (-0.1, 1.0, float("nan")):
        with pytest.raises(vce.VceError):
            vce.ce_forward_ls(x, lab, bad)


def test_smoothing_autograd_matches_torch_on_small_margins(vce):
    p = gen.custom(32, 500, "f32", seed=72, std=2.0, n_margin=4, margin=(3.0, 8.0), n_ignore=2)
    storage = p.full()
    logits = to_device(storage, "f32").requires_grad_(True)
    loss = vce.cross_entropy(logits, torch.from_numpy(p.labels).cuda(), label_smoothing=0.2)
    loss.backward()
    zt = torch.tensor(O.widen(storage, "f32"), requires_grad=True)
    tl = torch.nn.functional.cross_entropy(zt, torch.from_numpy(p.labels), ignore_index=-100, label_smoothing=0.2)
    tl.backward()
    assert abs(loss.item() - tl.item()) <= 1e-4 * abs(tl.item())
    np.testing.assert_allclose(logits.grad.cpu().numpy(), zt.grad.numpy(), rtol=1e-4, atol=1e-7)


def test_smoothing_pages_shape_sampled(vce):
    p = gen.pages()
    storage = p.full()
    logits = to_device(storage, "bf16")
    labels = torch.from_numpy(p.labels).cuda()
    eps = 0.1
    out, rows, stats, status = vce.ce_forward_ls(logits, labels, eps)
    grad = vce.ce_backward_ls(logits, labels, stats, torch.ones(1, device="cuda"), eps)
    torch.cuda.synchronize()
    rng = np.random.default_rng(21)
    rr = np.unique(np.concatenate([p.margin_rows[:100], rng.choice(p.T, 100, replace=False)]))
    N = int(np.sum(p.labels != p.ignore_index))
    ref = O.ce_smoothed(O.widen(storage[rr], "bf16"), p.labels[rr], eps, "sum", grad_output=1.0 / N)
    G.check_loss_rows(rows.cpu().numpy()[rr], ref["loss_rows"], ref["valid"])
    grade_smoothed_grad(grad[torch.from_numpy(rr).cuda()], ref, ref["c"], eps, p.V, p.labels[rr])


# ---- the one-pass call (ce_forward_backward_ls) -----------------------------------------------

@pytest.mark.parametrize("V", [3001, 3008, 70000])   # L2 re-read; stage ring, one CTA; 2-CTA cluster
@pytest.mark.parametrize("eps", [0.1, 0.5])
@pytest.mark.parametrize("dtype,reduction,gdt", [("bf16", "mean", None), ("f32", "sum", None),
                                                 ("bf16", "none", torch.float32)])
def test_one_pass_smoothing_parity(vce, eps, dtype, reduction, gdt, V):
    T = 32 if V > 10000 else 64
    p = gen.custom(T, V, dtype, seed=73, std=2.0, n_margin=6, margin=(17.0, 50.0), n_ignore=3)
    storage = p.full()
    logits = to_device(storage, dtype)
    labels = torch.from_numpy(p.labels).cuda()
    go_np = np.linspace(0.5, 2.0, T) if reduction == "none" else np.array([1.25])
    go = torch.from_numpy(go_np.astype(np.float32)).cuda()
    out, rows, stats, grad, status = vce.ce_forward_backward_ls(logits, labels, eps, reduction=reduction,
                                                               grad_output=go, grad_dtype=gdt)
    torch.cuda.synchronize()
    assert vce.vce_get_status(status) == 0
    ref = O.ce_smoothed(O.widen(storage, dtype), p.labels, eps, reduction, go_np if reduction == "none" else 1.25)
    G.check_loss_rows(rows.cpu().numpy(), ref["loss_rows"], ref["valid"])
    if reduction != "none":
        G.check_reduced(out.item(), ref["loss_out"])
    grade_smoothed_grad(grad, ref, ref["c"], eps, p.V, p.labels)


@pytest.mark.parametrize("V", [3001, 3008])
def test_one_pass_smoothing_zero_is_the_plain_call(vce, V):
    p = gen.custom(40, V, "bf16", seed=74, n_margin=4, n_ignore=2)
    logits = to_device(p.full(), "bf16")
    labels = torch.from_numpy(p.labels).cuda()
    a = vce.ce_forward_backward_ls(logits, labels, 0.0)
    a = tuple(x.clone() for x in a)
    b = vce.ce_forward_backward(logits, labels)
    torch.cuda.synchronize()
    for x, y in zip(a[:4], b[:4]):
        assert torch.equal(x, y)
    for bad in (-0.1, 1.0, float("nan")):
        with pytest.raises(vce.VceError):
            vce.ce_forward_backward_ls(logits, labels, bad)


def test_one_pass_smoothing_pages_shape_sampled(vce):
    p = gen.pages()
    storage = p.full()
    logits = to_device(storage, "bf16")
    labels = torch.from_numpy(p.labels).cuda()
    eps = 0.1
    out, rows, stats, grad, status = vce.ce_forward_backward_ls(logits, labels, eps)
    torch.cuda.synchronize()
    assert vce.vce_get_status(status) == 0
    rng = np.random.default_rng(22)
    rr = np.unique(np.concatenate([p.margin_rows[:100], rng.choice(p.T, 100, replace=False)]))
    N = int(np.sum(p.labels != p.ignore_index))
    ref = O.ce_smoothed(O.widen(storage[rr], "bf16"), p.labels[rr], eps, "sum", grad_output=1.0 / N)
    G.check_loss_rows(rows.cpu().numpy()[rr], ref["loss_rows"], ref["valid"])
    grade_smoothed_grad(grad[torch.from_numpy(rr).cuda()], ref, ref["c"], eps, p.V, p.labels[rr])


# ---- the chunked call (ce_merge_chunks_ls) ----------------------------------------------------

@pytest.mark.parametrize("widths", [[1000, 2001], [64] * 8, [7, 993, 1]])
@pytest.mark.parametrize("eps,dtype,reduction", [(0.1, "bf16", "mean"), (0.5, "f32", "none")])
def test_chunked_smoothing_parity(vce, widths, eps, dtype, reduction):
    V = sum(widths)
    p = gen.custom(48, V, dtype, seed=75 + V, std=2.0, n_margin=5, margin=(17.0, 50.0), n_ignore=3)
    storage = p.full()
    offs = np.cumsum([0] + list(widths[:-1]))
    chunks = [to_device(np.ascontiguousarray(storage[:, o:o + w]), dtype) for o, w in zip(offs, widths)]
    labels = torch.from_numpy(p.labels).cuda()
    go_np = np.linspace(0.5, 2.0, p.T) if reduction == "none" else np.array([0.75])
    go = torch.from_numpy(go_np.astype(np.float32)).cuda()
    out, rows, stats, grads, cstats, status = vce.ce_merge_chunks(chunks, labels, reduction=reduction,
                                                                  grad_output=go, label_smoothing=eps)
    torch.cuda.synchronize()
    assert vce.vce_get_status(status) == 0
    ref = O.ce_smoothed(O.widen(storage, dtype), p.labels, eps, reduction, go_np if reduction == "none" else 0.75)
    G.check_loss_rows(rows.cpu().numpy(), ref["loss_rows"], ref["valid"])
    if reduction != "none":
        G.check_reduced(out.item(), ref["loss_out"])
    grade_smoothed_grad(torch.cat(grads, dim=1), ref, ref["c"], eps, p.V, p.labels)


def test_chunked_smoothing_rejects_bad_eps(vce):
    chunks = [torch.zeros(2, 4, device="cuda"), torch.zeros(2, 4, device="cuda")]
    lab = torch.zeros(2, dtype=torch.int64, device="cuda")
    for bad in (-0.1, 1.0, float("nan")):
        with pytest.raises(vce.VceError):
            vce.ce_merge_chunks(chunks, lab, label_smoothing=bad)

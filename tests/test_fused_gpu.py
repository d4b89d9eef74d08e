"""ce_forward_backward (one pass) through the C ABI: parity with the oracle and bitwise
equality with ce_forward followed by ce_backward."""
import numpy as np
import pytest
import torch

import gen
from oracle import ce_oracle as O
from tests import _grading as G
from tests.test_ce_gpu import TORCH_DT, grade_grad, to_device, vce  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


def fused_vs_two_calls(vce, p, reduction="mean", grad_output=1.0, grad_dtype=None, storage=None):
    storage = p.full() if storage is None else storage
    logits = to_device(storage, p.dtype)
    labels = torch.from_numpy(p.labels).cuda()
    go = torch.empty(p.T if reduction == "none" else 1, device="cuda")
    go[:] = torch.as_tensor(grad_output, dtype=torch.float32)
    f_out, f_rows, f_stats, f_grad, f_status = vce.ce_forward_backward(logits, labels, reduction=reduction,
                                                                       grad_output=go, grad_dtype=grad_dtype)
    t_out, t_rows, t_stats, t_status = vce.ce_forward(logits, labels, reduction=reduction)
    t_grad = vce.ce_backward(logits, labels, t_stats, go, reduction=reduction, grad_dtype=grad_dtype)
    torch.cuda.synchronize()
    assert vce.vce_get_status(f_status) == 0 and vce.vce_get_status(t_status) == 0
    assert torch.equal(f_rows, t_rows) and torch.equal(f_stats, t_stats) and torch.equal(f_grad, t_grad)
    if reduction != "none":
        assert torch.equal(f_out, t_out)
    return storage, f_out, f_rows, f_grad


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("dtype,gdt", [("bf16", None), ("bf16", torch.float32), ("f32", None), ("f32", torch.bfloat16)])
def test_fused_parity(vce, reduction, dtype, gdt):
    p = gen.custom(80, 5000, dtype, seed=61, std=2.5, n_margin=10, margin=(17.0, 50.0), n_ignore=5)
    go = np.linspace(0.25, 2.0, 80) if reduction == "none" else 0.5
    storage, out, rows, grad = fused_vs_two_calls(vce, p, reduction, go, gdt)
    ref = O.ce(O.widen(storage, dtype), p.labels, reduction, go)
    G.check_loss_rows(rows.cpu().numpy(), ref["loss_rows"], ref["valid"])
    if reduction != "none":
        G.check_reduced(out.item(), ref["loss_out"])
    grade_grad(grad, ref["grad"], p.margin_rows, p.labels)


@pytest.mark.parametrize("V", [1, 7, 1001, 70000])
def test_fused_odd_sizes(vce, V):
    p = gen.custom(21, V, "bf16", seed=V + 3, n_margin=3 if V > 1 else 0, n_ignore=2)
    storage, out, rows, grad = fused_vs_two_calls(vce, p)
    ref = O.ce(O.widen(storage, "bf16"), p.labels, "mean")
    G.check_loss_rows(rows.cpu().numpy(), ref["loss_rows"], ref["valid"])
    grade_grad(grad, ref["grad"])


def test_fused_all_ignored_and_bad_label(vce):
    p = gen.custom(6, 300, "bf16", seed=5)
    logits = to_device(p.full(), "bf16")
    out = vce.ce_forward_backward(logits, torch.full((6,), -100, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert np.isnan(out[0].item()) and torch.all(out[3] == 0) and torch.all(out[1] == 0)
    lab = torch.from_numpy(p.labels).cuda()
    lab[2] = 300
    out = vce.ce_forward_backward(logits, lab)
    assert vce.vce_get_status(out[4]) == 1 and torch.all(out[3][2] == 0) and np.isnan(out[1][2].item())


def test_fused_pages_shape_equals_two_calls(vce):
    """The pages' matrix: the one-pass outputs are bitwise those of the two calls."""
    p = gen.pages()
    storage, out, rows, grad = fused_vs_two_calls(vce, p)
    rng = np.random.default_rng(3)
    rr = np.unique(np.concatenate([p.margin_rows[:200], rng.choice(p.T, 100, replace=False)]))
    z = O.widen(storage[rr], "bf16")
    fwd = O.ce_rows(z, p.labels[rr])
    N = int(np.sum(p.labels != p.ignore_index))
    want = O.ce_grad_rows(z, p.labels[rr], fwd, O.row_scale(fwd["valid"], "sum", 1.0 / N))
    G.check_loss_rows(rows.cpu().numpy()[rr], fwd["loss"], fwd["valid"])
    G.check_grad_bf16(G.bf16_tensor_bits(grad[torch.from_numpy(rr).cuda()]), want)

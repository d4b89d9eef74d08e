"""Parity of the CUDA CE forward/backward (through the C ABI) with the fp64 oracle."""
import numpy as np
import pytest
import torch

import gen
from oracle import ce_oracle as O
from oracle import rounding as R
from tests import _grading as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vce():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    import vocab_cross_entropy_gb300 as v
    return v


TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def to_device(storage, dtype):
    t = torch.from_numpy(np.ascontiguousarray(storage))
    if dtype == "bf16":
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.cuda()


def host_values(t):
    if t.dtype == torch.bfloat16:
        return O.widen(G.bf16_tensor_bits(t), "bf16")
    return t.detach().cpu().numpy().astype(np.float64)


def grade_grad(grad_t, want, rows_raised_target=None, labels=None, what="grad"):
    if grad_t.dtype == torch.bfloat16:
        G.check_grad_bf16(G.bf16_tensor_bits(grad_t), want, what)
    else:
        got = grad_t.cpu().numpy().astype(np.float64)
        G.check_grad_f32(got, want, what)
        if rows_raised_target is not None and len(rows_raised_target):
            r = rows_raised_target
            G.check_target_entries(got[r, labels[r]], want[r, labels[r]], what + " (raised targets)")


def run_ce(vce, logits, labels_np, reduction="mean", grad_output=1.0, grad_dtype=None, ignore_index=-100):
    labels = torch.from_numpy(labels_np).cuda()
    loss_out, loss_rows, stats, status = vce.ce_forward(logits, labels, ignore_index, reduction)
    T = logits.shape[0]
    go = torch.full((T,) if reduction == "none" else (1,), 0.0, dtype=torch.float32, device="cuda")
    go[:] = torch.as_tensor(grad_output, dtype=torch.float32)
    grad = vce.ce_backward(logits, labels, stats, go, ignore_index, reduction, grad_dtype=grad_dtype)
    torch.cuda.synchronize()
    return loss_out, loss_rows, stats, status, grad


def full_check(vce, p, reduction="mean", grad_output=1.0, grad_dtype=None, block=512):
    """Whole-matrix parity for a problem the oracle finishes in seconds."""
    storage = p.full()
    logits = to_device(storage, p.dtype)
    before = logits.clone()
    loss_out, loss_rows, stats, status, grad = run_ce(vce, logits, p.labels, reduction, grad_output, grad_dtype)
    assert vce.vce_get_status(status) == 0
    assert torch.equal(logits, before)   # the input is never written
    z = O.widen(storage, p.dtype)
    ref = O.ce(z, p.labels, reduction, grad_output)
    G.check_loss_rows(loss_rows.cpu().numpy(), ref["loss_rows"], ref["valid"])
    if reduction != "none":
        G.check_reduced(loss_out.item(), ref["loss_out"])
    grade_grad(grad, ref["grad"], p.margin_rows, p.labels)
    st = stats.cpu().numpy().astype(np.float64)
    v = ref["valid"]
    fin = v & np.isfinite(ref["lse_nt"])
    assert np.all(np.abs(st[fin, 0] - ref["lse_nt"][fin]) <= 1e-5 * np.maximum(1, np.abs(ref["lse_nt"][fin])))
    assert np.all(st[~v] == 0)
    return grad, stats


def test_tiny_config_full(vce):
    full_check(vce, gen.tiny())


def test_mid_config_full(vce):
    p = gen.mid()
    storage = p.full()
    logits = to_device(storage, "bf16")
    loss_out, loss_rows, stats, status, grad = run_ce(vce, logits, p.labels)
    assert vce.vce_get_status(status) == 0
    lr = loss_rows.cpu().numpy()
    gbits = G.bf16_tensor_bits(grad)
    losses = []
    for r0 in range(0, p.T, 512):
        z = O.widen(storage[r0:r0 + 512], "bf16")
        fwd = O.ce_rows(z, p.labels[r0:r0 + 512])
        c = O.row_scale(fwd["valid"], "sum", 1.0 / (p.T - p.n_ignore))
        want = O.ce_grad_rows(z, p.labels[r0:r0 + 512], fwd, c)
        G.check_loss_rows(lr[r0:r0 + 512], fwd["loss"], fwd["valid"])
        G.check_grad_bf16(gbits[r0:r0 + 512], want, f"grad rows {r0}+")
        losses.append(fwd["loss"])
    valid = p.labels != p.ignore_index
    G.check_reduced(loss_out.item(), np.concatenate(losses)[valid].sum() / valid.sum())


@pytest.mark.parametrize("reduction", ["sum", "none"])
@pytest.mark.parametrize("dtype,gdt", [("bf16", torch.float32), ("f32", torch.bfloat16), ("f32", None)])
def test_reductions_and_grad_dtypes(vce, reduction, dtype, gdt):
    p = gen.custom(96, 3000, dtype, seed=41, std=2.5, n_margin=12, margin=(17.0, 50.0), n_ignore=6)
    go = np.linspace(0.25, 2.0, 96) if reduction == "none" else 0.75
    full_check(vce, p, reduction, go, gdt)


@pytest.mark.parametrize("V", [1, 2, 3, 7, 9, 1001, 4097, 33333])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_odd_vocab_sizes(vce, V, dtype):
    p = gen.custom(19, V, dtype, seed=V, std=2.0, n_margin=3 if V > 1 else 0, n_ignore=2)
    full_check(vce, p)


def test_single_row(vce):
    full_check(vce, gen.custom(1, 5000, "bf16", seed=2, n_margin=1))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_padded_ld_and_unaligned_rows(vce, dtype):
    """A view with ld > V whose rows start off the 16-byte grid (head/tail path and scalar path)."""
    p = gen.custom(33, 1000, dtype, seed=17, n_margin=4, n_ignore=3)
    storage = p.full()
    big = np.zeros((33, 1013), storage.dtype)
    big[:, 3:1003] = storage
    base = to_device(big, dtype)
    logits = base[:, 3:1003]
    labels = torch.from_numpy(p.labels).cuda()
    loss_out, loss_rows, stats, status = vce.ce_forward(logits, labels)
    go = torch.ones(1, device="cuda")
    gbase = torch.full((33, 1011), 7.0, dtype=TORCH_DT[dtype], device="cuda")
    grad = vce.ce_backward(logits, labels, stats, go, grad_logits=gbase[:, 1:1001])
    torch.cuda.synchronize()
    ref = O.ce(O.widen(storage, dtype), p.labels, "mean")
    G.check_loss_rows(loss_rows.cpu().numpy(), ref["loss_rows"], ref["valid"])
    grade_grad(gbase[:, 1:1001], ref["grad"], p.margin_rows, p.labels)
    assert torch.all(gbase[:, :1] == 7) and torch.all(gbase[:, 1001:] == 7)   # nothing written outside


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_output_phase_differs_from_input(vce, dtype):
    p = gen.custom(17, 999, dtype, seed=18, n_margin=3, n_ignore=2)
    storage = p.full()
    logits = to_device(storage, dtype)
    labels = torch.from_numpy(p.labels).cuda()
    _, loss_rows, stats, status = vce.ce_forward(logits, labels)
    gbase = torch.full((17, 1003), 3.0, dtype=TORCH_DT[dtype], device="cuda")
    gview = gbase[:, 1:1000]
    vce.ce_backward(logits, labels, stats, torch.ones(1, device="cuda"), grad_logits=gview)
    torch.cuda.synchronize()
    ref = O.ce(O.widen(storage, dtype), p.labels, "mean")
    grade_grad(gview, ref["grad"], p.margin_rows, p.labels)
    assert torch.all(gbase[:, 0] == 3) and torch.all(gbase[:, 1000:] == 3)


def test_non_finite_rows(vce):
    z = np.array([
        [np.inf, -np.inf, 3.0, 1.0],      # ignored row holding +-inf: exactly zero
        [-np.inf, -np.inf, -np.inf, -np.inf],   # ignored
        [-np.inf, 2.0, -np.inf, -np.inf],  # every non-target -inf: loss 0, gradient 0
        [0.0, -np.inf, np.log(3.0), -np.inf],   # -inf target: loss +inf
        [1.0, -np.inf, 2.0, 0.5],
    ], np.float32)
    labels = np.array([-100, -100, 1, 1, 2])
    for dtype in ("f32", "bf16"):
        storage = z if dtype == "f32" else (z.view(np.uint32) >> 16).astype(np.uint16)
        logits = to_device(storage, dtype)
        loss_out, loss_rows, stats, status, grad = run_ce(vce, logits, labels, "sum")
        ref = O.ce(O.widen(storage, dtype), labels, "sum")
        lr = loss_rows.cpu().numpy()
        assert lr[0] == 0 and lr[1] == 0 and lr[2] == 0 and lr[3] == np.inf
        assert abs(lr[4] - ref["loss_rows"][4]) <= 1e-4 * ref["loss_rows"][4]
        g = host_values(grad)
        assert np.all(g[:3] == 0)
        if dtype == "bf16":   # the one-ulp bar of every bf16 gradient, -inf columns included
            G.check_grad_bf16(G.bf16_tensor_bits(grad)[3:], ref["grad"][3:], "non-finite rows")
        else:
            np.testing.assert_allclose(g[3:], ref["grad"][3:], rtol=1e-5, atol=1e-7)


@pytest.mark.parametrize("V", [100, 104])   # per-block kernels; shared-memory stage rings
def test_all_rows_ignored(vce, V):
    p = gen.custom(8, V, "bf16", seed=3)
    labels = np.full(8, -100)
    logits = to_device(p.full(), "bf16")
    loss_out, loss_rows, stats, status, grad = run_ce(vce, logits, labels, "mean")
    assert np.isnan(loss_out.item())
    assert torch.all(loss_rows == 0) and torch.all(grad == 0)


@pytest.mark.parametrize("V", [100, 104])
def test_invalid_label_sets_status(vce, V):
    p = gen.custom(8, V, "f32", seed=4)
    labels = p.labels.copy()
    labels[3] = V
    labels[5] = -7
    logits = to_device(p.full(), "f32")
    loss_out, loss_rows, stats, status, grad = run_ce(vce, logits, labels, "mean")
    assert vce.vce_get_status(status) == 1
    lr = loss_rows.cpu().numpy()
    assert np.isnan(lr[3]) and np.isnan(lr[5]) and np.isnan(loss_out.item())
    assert torch.all(grad[3] == 0) and torch.all(grad[5] == 0)
    # a clean call resets the status word
    _, _, _, status2, _ = run_ce(vce, logits, p.labels, "mean")
    assert vce.vce_get_status(status2) == 0


def test_host_argument_errors(vce):
    import ctypes
    lib = vce.lib
    x = torch.zeros(4, 8, device="cuda")
    lab = torch.zeros(4, dtype=torch.int64, device="cuda")
    out = torch.zeros(4, device="cuda")
    st = torch.zeros(4, 4, device="cuda")
    s = torch.zeros(1, dtype=torch.int32, device="cuda")
    P = ctypes.c_void_p
    args = lambda **kw: [P(kw.get("x", x.data_ptr())), kw.get("dt", 0), kw.get("T", 4), kw.get("V", 8),
                         kw.get("ld", 8), P(lab.data_ptr()), -100, kw.get("red", 2), P(out.data_ptr()),
                         P(out.data_ptr()), P(kw.get("st", st.data_ptr())), P(s.data_ptr()), None]
    assert lib.ce_forward(*args()) == 0
    assert lib.ce_forward(*args(dt=5)) == -2
    assert lib.ce_forward(*args(red=9)) == -2
    assert lib.ce_forward(*args(V=0)) == -3
    assert lib.ce_forward(*args(ld=7)) == -4
    assert lib.ce_forward(*args(x=x.data_ptr() + 2)) == -5
    assert lib.ce_forward(*args(st=st.data_ptr() + 4)) == -5
    assert lib.ce_forward(*args(T=1 << 62, ld=1 << 3)) == -3
    torch.cuda.synchronize()


def test_repeatable_bitwise(vce):
    p = gen.custom(64, 20000, "bf16", seed=8, n_margin=6, n_ignore=3)
    logits = to_device(p.full(), "bf16")
    a = run_ce(vce, logits, p.labels)
    b = run_ce(vce, logits, p.labels)
    for name, j in (("loss_out", 0), ("loss_rows", 1), ("row_stats", 2), ("grad", 4)):
        d = (a[j].float() - b[j].float()).abs()
        assert torch.equal(a[j], b[j]), f"{name}: {int((d > 0).sum())} entries differ, max {float(d.max())}"
    assert vce.vce_get_status(a[3]) == 0 and vce.vce_get_status(b[3]) == 0


def test_autograd_wrapper(vce):
    p = gen.custom(32, 700, "bf16", seed=9, n_margin=4, n_ignore=2)
    storage = p.full()
    logits = to_device(storage, "bf16").requires_grad_(True)
    loss = vce.cross_entropy(logits, torch.from_numpy(p.labels).cuda())
    (2.0 * loss).backward()
    ref = O.ce(O.widen(storage, "bf16"), p.labels, "mean", grad_output=2.0)
    G.check_reduced(loss.item(), ref["loss_out"])
    G.check_grad_bf16(G.bf16_tensor_bits(logits.grad), ref["grad"])


# ------------------------------------------------------------------ the pages' shape, as the bench runs it

@pytest.fixture(scope="module")
def pages_data():
    p = gen.pages()
    storage = p.full()
    return p, storage


def test_pages_shape_sampled(vce, pages_data):
    p, storage = pages_data
    logits = to_device(storage, "bf16")
    labels = torch.from_numpy(p.labels).cuda()
    loss_out, loss_rows, stats, status = vce.ce_forward(logits, labels)
    grad = vce.ce_backward(logits, labels, stats, torch.ones(1, device="cuda"))
    torch.cuda.synchronize()
    assert vce.vce_get_status(status) == 0
    rng = np.random.default_rng(0)
    valid = p.labels != p.ignore_index
    N = int(valid.sum())
    rows = np.unique(np.concatenate([p.margin_rows, rng.choice(p.T, 256, replace=False), [0, p.T - 1]]))
    lr = loss_rows.cpu().numpy()
    idx = torch.from_numpy(rows).cuda()
    gbits = G.bf16_tensor_bits(grad.index_select(0, idx))
    for k in range(0, len(rows), 256):
        rr = rows[k:k + 256]
        z = O.widen(storage[rr], "bf16")
        fwd = O.ce_rows(z, p.labels[rr])
        want = O.ce_grad_rows(z, p.labels[rr], fwd, O.row_scale(fwd["valid"], "sum", 1.0 / N))
        G.check_loss_rows(lr[rr], fwd["loss"], fwd["valid"], "pages loss")
        G.check_grad_bf16(gbits[k:k + 256], want, "pages grad")
    # ignored rows: exactly zero gradient; reduction consistent with the per-row losses
    ig = torch.from_numpy(p.ignore_rows).cuda()
    assert torch.all(grad.index_select(0, ig) == 0) and np.all(lr[p.ignore_rows] == 0)
    G.check_reduced(loss_out.item(), float(np.sum(lr[valid].astype(np.float64)) / N))
    # collapse regime: every raised-target row has a positive loss and a negative target gradient
    assert np.all(lr[p.margin_rows] > 0)
    tg = grad[torch.from_numpy(p.margin_rows).cuda(), torch.from_numpy(p.labels[p.margin_rows]).cuda()]
    assert torch.all(tg < 0)


@pytest.mark.parametrize("dtype,gdt,reduction", [("f32", torch.float32, "mean"), ("bf16", torch.float32, "none")])
def test_pages_shape_other_dtypes_sampled(vce, dtype, gdt, reduction):
    """The pages' shape with fp32 logits, and with bf16 logits, fp32 gradients and per-row losses."""
    base = gen.pages()
    p = gen.CEProblem("pages", base.T, base.V, dtype, base.seed, base.std, base.n_margin, base.margin_lo,
                      base.margin_hi, base.n_ignore)
    storage = p.full()
    logits = to_device(storage, dtype)
    labels = torch.from_numpy(p.labels).cuda()
    go_np = np.linspace(0.5, 1.5, p.T) if reduction == "none" else np.ones(1)
    go = torch.from_numpy(go_np.astype(np.float32)).cuda()
    loss_out, loss_rows, stats, status = vce.ce_forward(logits, labels, reduction=reduction)
    grad = vce.ce_backward(logits, labels, stats, go, reduction=reduction, grad_dtype=gdt)
    torch.cuda.synchronize()
    assert vce.vce_get_status(status) == 0
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([p.margin_rows[:200], rng.choice(p.T, 200, replace=False)]))
    z = O.widen(storage[rows], dtype)
    fwd = O.ce_rows(z, p.labels[rows])
    N = int(np.sum(p.labels != p.ignore_index))
    c = fwd["valid"] * (go_np[rows] if reduction == "none" else 1.0 / N)
    want = O.ce_grad_rows(z, p.labels[rows], fwd, c)
    G.check_loss_rows(loss_rows.cpu().numpy()[rows], fwd["loss"], fwd["valid"])
    got = grad[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
    G.check_grad_f32(got, want)
    raised = np.isin(rows, p.margin_rows)
    G.check_target_entries(got[raised, p.labels[rows][raised]], want[raised, p.labels[rows][raised]])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_non_target_spikes_take_the_rescale_path(vce, dtype):
    """Non-target values far above the rest (late in the row, and one early) force the forward's
    running reference to be replaced mid-row; results must still match the oracle."""
    p = gen.custom(24, 20000, dtype, seed=33, std=2.0, n_margin=4, margin=(17.0, 50.0), n_ignore=2)
    storage = p.full().copy()
    z = O.widen(storage, dtype)
    rng = np.random.default_rng(4)
    for i in range(p.T):
        if p.labels[i] == p.ignore_index:
            continue
        for bump, pos in ((30.0, 19000), (60.0, 15000), (90.0, 7), (45.0, 12345)):
            j = (pos + i) % p.V
            if j == p.labels[i]:
                continue
            z[i, j] = z[i].max() + bump + rng.uniform(0, 1)
    if dtype == "f32":
        storage = z.astype(np.float32)
    else:
        storage = R.bf16_bits(R.round_bf16(z))
    ref = O.ce(O.widen(storage, dtype), p.labels, "mean")
    logits = to_device(storage, dtype)
    loss_out, loss_rows, stats, status, grad = run_ce(vce, logits, p.labels)
    assert vce.vce_get_status(status) == 0
    G.check_loss_rows(loss_rows.cpu().numpy(), ref["loss_rows"], ref["valid"])
    G.check_reduced(loss_out.item(), ref["loss_out"])
    grade_grad(grad, ref["grad"])


# ---- ce_forward's row kernels: one warp per row (rows of at most 32 KB), the shared-memory --
# ---- stage ring (longer rows of whole 16-byte vectors; rows of two stages in two consumer groups)

@pytest.mark.parametrize("T,V,dtype,reduction", [
    (40, 8, "bf16", "mean"),          # warp per row, 16-byte rows
    (300, 4096, "f32", "none"),       # warp per row, 16 KB rows
    (200, 70000, "bf16", "sum"),      # ring: 4.3 stages per row, partial last stage
    (24, 128256, "f32", "mean"),      # ring: 15.7 stages per row, the ring wraps within a row
    (700, 16384, "bf16", "mean"),     # warp per row, exactly 32 KB
    (4000, 2000, "bf16", "mean"),     # warp per row, 26-27 rows per warp's stride
    (2000, 12000, "f32", "none"),     # ring, two groups: 1.46 stages per row, 13-14 rows per CTA
    (1300, 32768, "bf16", "sum"),     # ring, two groups: two whole stages, 8-9 rows per CTA
    (1300, 16392, "bf16", "mean"),    # ring, two groups: one whole stage and 16 bytes
])
def test_forward_ring_shapes(vce, T, V, dtype, reduction):
    p = gen.custom(T, V, dtype, seed=T + V, std=2.0, n_margin=max(1, T // 10), margin=(17.0, 50.0),
                   n_ignore=max(1, T // 20))
    full_check(vce, p, reduction, np.linspace(0.5, 1.5, T) if reduction == "none" else 1.0)


def test_forward_ring_padded_ld(vce):
    """ld = V + 8: the padding (80.0, which would dominate the sums) is never read."""
    p = gen.custom(60, 5000, "bf16", seed=9, n_margin=6, n_ignore=3)
    storage = p.full()
    wide = np.zeros((p.T, 5008), dtype=storage.dtype)
    wide[:, :5000] = storage
    wide[:, 5000:] = 0x42A0
    logits = to_device(wide, "bf16")[:, :5000]
    loss_out, loss_rows, stats, status, grad = run_ce(vce, logits, p.labels)
    assert vce.vce_get_status(status) == 0
    ref = O.ce(O.widen(storage, "bf16"), p.labels, "mean")
    G.check_loss_rows(loss_rows.cpu().numpy(), ref["loss_rows"], ref["valid"])
    G.check_reduced(loss_out.item(), ref["loss_out"])


def test_forward_ring_non_finite_and_bad_labels(vce):
    """V = 8: -inf entries, a row of all -inf non-targets, ignored and invalid labels."""
    rng = np.random.default_rng(12)
    z = rng.normal(0, 2, (6, 8)).astype(np.float32)
    z[1, :] = -np.inf
    z[1, 3] = 1.5                       # every non-target -inf: loss 0
    z[2, 5] = -np.inf                   # the target itself -inf: loss +inf
    z[4, 0] = -np.inf
    labels = np.array([2, 3, 5, -100, 7, 9])   # row 5: label 9 >= V
    for dtype in ("f32", "bf16"):
        storage = z if dtype == "f32" else (z.view(np.uint32) >> 16).astype(np.uint16)
        logits = to_device(storage, dtype)
        lab = torch.from_numpy(labels).cuda()
        loss_out, loss_rows, stats, status = vce.ce_forward(logits, lab, reduction="none")
        torch.cuda.synchronize()
        assert vce.vce_get_status(status) == 1
        lr = loss_rows.cpu().numpy()
        ref = O.ce(O.widen(storage, dtype), np.where(labels < 8, labels, -100), "none")
        assert lr[1] == 0 and lr[2] == np.inf and lr[3] == 0 and np.isnan(lr[5])
        for r in (0, 4):
            assert abs(lr[r] - ref["loss_rows"][r]) <= 1e-4 * ref["loss_rows"][r]


@pytest.mark.parametrize("T,V", [(24, 20000), (152, 17000), (300, 40000)])
def test_folded_reduction_repeats_exactly(vce, T, V):
    """Rows of the forward ring reduced in-kernel by the CTA that finishes last, with every CTA
    finishing within microseconds of the others: 40 calls into buffers refilled with NaN each
    time give the same reduced loss, bit for bit, and the oracle's value."""
    p = gen.custom(T, V, "bf16", seed=T + 1, std=2.0, n_ignore=2)
    storage = p.full()
    logits = to_device(storage, "bf16")
    labels = torch.from_numpy(p.labels).cuda()
    want = O.ce(O.widen(storage, "bf16"), p.labels, "mean")["loss_out"]
    rows = torch.empty(T, dtype=torch.float32, device="cuda")
    out = torch.empty(1, dtype=torch.float32, device="cuda")
    stats = torch.empty(T, 4, dtype=torch.float32, device="cuda")
    status = torch.empty(1, dtype=torch.int32, device="cuda")
    got = []
    for _ in range(40):
        rows.fill_(float("nan"))
        out.fill_(float("nan"))
        vce.ce_forward(logits, labels, reduction="mean", loss_rows=rows, loss_out=out, row_stats=stats, status=status)
        got.append(out.item())
        assert vce.vce_get_status(status) == 0
    assert all(g == got[0] for g in got), got
    G.check_reduced(got[0], want)


@pytest.mark.parametrize("reduction", ["mean", "none"])
def test_forward_ring_launch_slots(vce, reduction):
    """The stage ring claims rows from a per-launch slot of device words that its last CTA puts
    back to zero, and writes the status word itself.  1100 calls (more than the 1024 slots, so
    every slot is used and reused) into a status word filled with garbage and outputs filled
    with NaN each time: every call's status is 0 and its outputs equal the first call's, bit for
    bit.  A call with a bad label in the middle sets VCE_ERR_LABEL, and the next calls, which
    reuse slots after it, are clean again."""
    T, V = 400, 20000
    p = gen.custom(T, V, "bf16", seed=91, std=2.0, n_margin=10, n_ignore=40)
    logits = to_device(p.full(), "bf16")
    labels = torch.from_numpy(p.labels).cuda()
    bad_np = p.labels.copy()
    bad_np[17] = V
    bad = torch.from_numpy(bad_np).cuda()
    rows = torch.empty(T, dtype=torch.float32, device="cuda")
    out = torch.empty(1, dtype=torch.float32, device="cuda")
    stats = torch.empty(T, 4, dtype=torch.float32, device="cuda")
    status = torch.empty(1, dtype=torch.int32, device="cuda")
    first = None
    for i in range(1100):
        status.fill_(0x7FFF1234)
        rows.fill_(float("nan"))
        out.fill_(float("nan"))
        lab = bad if i == 500 else labels
        vce.ce_forward(logits, lab, reduction=reduction, loss_rows=rows, loss_out=out, row_stats=stats,
                       status=status)
        if i == 500:
            assert vce.vce_get_status(status) == 1
            assert np.isnan(rows[17].item())
            continue
        if i % 50 and i != 501:   # the status and outputs of every 50th call, and the one after the error
            continue
        assert vce.vce_get_status(status) == 0, i
        got = (rows.clone(), stats.clone(), out.clone())
        if first is None:
            first = got
            ref = O.ce(O.widen(p.full(), "bf16"), p.labels, "none")
            G.check_loss_rows(got[0].cpu().numpy(), ref["loss_rows"], ref["valid"])
        else:
            assert torch.equal(got[0], first[0]) and torch.equal(got[1], first[1]), i
            if reduction != "none":
                assert torch.equal(got[2], first[2]), i
    torch.cuda.synchronize()
    assert vce.vce_get_status(status) == 0


@pytest.mark.parametrize("V", [20000, 70000])
def test_backward_ring_launch_slots(vce, V):
    """The backward ring claims items from a per-launch slot that its last CTA puts back to zero:
    1100 calls (more than the 1024 slots) into a gradient filled with NaN every 50 calls give the
    same gradient, bit for bit, and the first one matches the oracle."""
    T = 300
    p = gen.custom(T, V, "bf16", seed=V + 3, std=2.0, n_margin=8, n_ignore=30)
    storage = p.full()
    logits = to_device(storage, "bf16")
    labels = torch.from_numpy(p.labels).cuda()
    _, _, stats, status = vce.ce_forward(logits, labels, reduction="mean")
    assert vce.vce_get_status(status) == 0
    go = torch.ones(1, device="cuda")
    grad = torch.empty_like(logits)
    first = None
    for i in range(1100):
        if i % 50 == 0:
            grad.fill_(float("nan"))
        vce.ce_backward(logits, labels, stats, go, grad_logits=grad)
        if i % 50:
            continue
        if first is None:
            first = grad.clone()
            ref = O.ce(O.widen(storage, "bf16"), p.labels, "mean")
            grade_grad(first, ref["grad"], p.margin_rows, p.labels)
        else:
            assert torch.equal(grad, first), i
    torch.cuda.synchronize()


def test_ring_launches_on_two_streams(vce):
    """Ring launches on two streams that nothing orders against each other hold different launch
    slots: 200 forward + backward pairs alternating between the streams, each on its own batch,
    give every checked result equal, bit for bit, to the batch's first, and the first matches
    the oracle."""
    T, V = 300, 20000
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    batches = []
    for seed in (5, 6):
        p = gen.custom(T, V, "bf16", seed=seed, std=2.0, n_margin=6, n_ignore=20)
        storage = p.full()
        batches.append(dict(p=p, storage=storage, logits=to_device(storage, "bf16"),
                            labels=torch.from_numpy(p.labels).cuda(),
                            rows=torch.empty(T, device="cuda"), out=torch.empty(1, device="cuda"),
                            stats=torch.empty(T, 4, device="cuda"),
                            status=torch.empty(1, dtype=torch.int32, device="cuda"),
                            go=torch.ones(1, device="cuda"),
                            grad=torch.empty(T, V, dtype=torch.bfloat16, device="cuda"), snaps=[]))
    torch.cuda.synchronize()
    for i in range(200):
        for b, s in zip(batches, streams):
            with torch.cuda.stream(s):
                vce.ce_forward(b["logits"], b["labels"], reduction="mean", loss_rows=b["rows"],
                               loss_out=b["out"], row_stats=b["stats"], status=b["status"], stream=s)
                vce.ce_backward(b["logits"], b["labels"], b["stats"], b["go"], grad_logits=b["grad"], stream=s)
                if i % 40 == 0:
                    b["snaps"].append((b["rows"].clone(), b["out"].clone(), b["grad"].clone(), b["status"].clone()))
    torch.cuda.synchronize()
    for b in batches:
        rows0, out0, grad0, st0 = b["snaps"][0]
        assert int(st0.item()) == 0
        ref = O.ce(O.widen(b["storage"], "bf16"), b["p"].labels, "mean")
        G.check_loss_rows(rows0.cpu().numpy(), ref["loss_rows"], ref["valid"])
        G.check_reduced(out0.item(), ref["loss_out"])
        grade_grad(grad0, ref["grad"], b["p"].margin_rows, b["p"].labels)
        for rows, out, grad, st in b["snaps"][1:]:
            assert int(st.item()) == 0
            assert torch.equal(rows, rows0) and torch.equal(out, out0) and torch.equal(grad, grad0)


def test_forward_ring_stall_gives_up_and_the_slot_stays_usable(vce):
    """Stages that never complete in ce_forward's stage ring (its producer announces 16 bytes more
    per stage than its copies deliver): the bounded waits give up with a code that the kernel
    itself writes into a status word filled with garbage, the call returns within seconds, and
    the next 1100 calls -- one of them on the launch slot the stalled launch held -- are correct
    with status 0."""
    import time
    T, V = 300, 20000
    p = gen.custom(T, V, "bf16", seed=29, std=2.0, n_margin=4, n_ignore=10)
    storage = p.full()
    logits = to_device(storage, "bf16")
    labels = torch.from_numpy(p.labels).cuda()
    t0 = time.time()
    st = vce.vce_test_ce_fwd_stall(logits, labels, wait_ns=50_000_000)
    assert st in (105, 106, 108, 110, 112), st
    assert "gave up" in vce.vce_status_string(st)
    assert time.time() - t0 < 60
    ref = O.ce(O.widen(storage, "bf16"), p.labels, "mean")
    rows = torch.empty(T, dtype=torch.float32, device="cuda")
    out = torch.empty(1, dtype=torch.float32, device="cuda")
    stats = torch.empty(T, 4, dtype=torch.float32, device="cuda")
    status = torch.empty(1, dtype=torch.int32, device="cuda")
    first = None
    for i in range(1100):
        vce.ce_forward(logits, labels, reduction="mean", loss_rows=rows, loss_out=out, row_stats=stats,
                       status=status)
        if i % 100 and i != 1099:
            continue
        assert vce.vce_get_status(status) == 0, i
        if first is None:
            first = (rows.clone(), out.clone())
            G.check_loss_rows(first[0].cpu().numpy(), ref["loss_rows"], ref["valid"])
            G.check_reduced(first[1].item(), ref["loss_out"])
        else:
            assert torch.equal(rows, first[0]) and torch.equal(out, first[1]), i


@pytest.mark.parametrize("V", [20000, 70000])
def test_forward_ring_first_rows_ignored(vce, V):
    """Rows 0..199 ignored: every CTA's first fixed rows (152 CTAs) are ignored ones, which the
    producer skips and the statistics warp writes as +0 losses with zero statistics; the rest
    match the oracle, the mean included."""
    T = 600
    p = gen.custom(T, V, "bf16", seed=V + 11, std=2.0, n_margin=10)
    labels = p.labels.copy()
    labels[:200] = -100
    storage = p.full()
    logits = to_device(storage, "bf16")
    lab = torch.from_numpy(labels).cuda()
    out, rows, stats, status = vce.ce_forward(logits, lab, -100, "mean")
    torch.cuda.synchronize()
    assert vce.vce_get_status(status) == 0
    ref = O.ce(O.widen(storage, "bf16"), labels, "mean")
    lr = rows.cpu().numpy()
    assert np.all(lr[:200] == 0) and np.all(stats.cpu().numpy()[:200] == 0)
    G.check_loss_rows(lr, ref["loss_rows"], ref["valid"])
    G.check_reduced(out.item(), ref["loss_out"])


def test_forward_ring_beyond_the_folded_reduction(vce):
    """65540 rows of 32 KB + 16 B: more rows than the ring reduces in-kernel, so k_ce_reduce runs
    after it.  The MEAN call's loss is the fp64 mean of the same kernel's per-row losses (its
    NONE call), its weights 1/N, and a bad label still sets the status."""
    T, V = 65540, 16392
    p = gen.custom(T, V, "bf16", seed=77, std=2.0, n_ignore=650)
    logits = to_device(p.full(), "bf16")
    labels = torch.from_numpy(p.labels).cuda()
    _, rows_none, _, st_none = vce.ce_forward(logits, labels, -100, "none")
    out, rows, stats, status = vce.ce_forward(logits, labels, -100, "mean")
    torch.cuda.synchronize()
    assert vce.vce_get_status(status) == 0 and vce.vce_get_status(st_none) == 0
    assert torch.equal(rows, rows_none)
    valid = p.labels != -100
    n = int(valid.sum())
    want = float(np.sum(rows_none.cpu().numpy().astype(np.float64)[valid])) / n
    assert abs(out.item() - want) <= 1e-6 * abs(want)
    w = stats.cpu().numpy()[:, 3]
    assert np.all(w[valid] == np.float32(1.0 / n)) and np.all(w[~valid] == 0)
    bad = p.labels.copy()
    bad[T - 1] = V
    out2, _, _, status2 = vce.ce_forward(logits, torch.from_numpy(bad).cuda(), -100, "sum")
    torch.cuda.synchronize()
    assert vce.vce_get_status(status2) == 1 and np.isnan(out2.item())


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_forward_ring_bad_labels_and_reduction(vce, reduction):
    """Rows of 40 KB (the stage ring, two consumer groups; for SUM and MEAN it also reduces the
    losses itself): ignored rows, labels below 0 and at V.  The status is VCE_ERR_LABEL, bad rows'
    losses and a reduced loss are NaN, and the valid rows match the oracle, weights included."""
    T, V = 700, 20000
    p = gen.custom(T, V, "bf16", seed=31, std=2.0, n_margin=20, margin=(17.0, 50.0), n_ignore=35)
    labels = p.labels.copy()
    bad = np.array([3, 150, 699])
    labels[bad] = [-7, V, V + 123]
    storage = p.full()
    logits = to_device(storage, "bf16")
    lab = torch.from_numpy(labels).cuda()
    loss_out, loss_rows, stats, status = vce.ce_forward(logits, lab, -100, reduction)
    torch.cuda.synchronize()
    assert vce.vce_get_status(status) == 1
    lr = loss_rows.cpu().numpy()
    assert np.all(np.isnan(lr[bad]))
    ok = labels.copy()
    ok[bad] = -100
    ref = O.ce(O.widen(storage, "bf16"), ok, "none")
    valid = ref["valid"]
    G.check_loss_rows(np.where(np.isin(np.arange(T), bad), 0.0, lr), ref["loss_rows"], valid)
    if reduction != "none":
        assert np.isnan(loss_out.item())
    st = stats.cpu().numpy()
    n_valid = int(valid.sum())
    want_w = 1.0 / n_valid if reduction == "mean" else 1.0
    assert np.all(st[valid, 3] == np.float32(want_w))
    assert np.all(st[~valid, 3] == 0)
    # the same batch without the bad labels reduces to the oracle's value, status 0
    lab2 = torch.from_numpy(ok).cuda()
    loss_out2, rows2, stats2, status2 = vce.ce_forward(logits, lab2, -100, reduction)
    torch.cuda.synchronize()
    assert vce.vce_get_status(status2) == 0
    if reduction != "none":
        G.check_reduced(loss_out2.item(), O.ce(O.widen(storage, "bf16"), ok, reduction)["loss_out"])


@pytest.mark.parametrize("dtype,gdt", [("bf16", torch.float32), ("f32", torch.bfloat16), ("bf16", torch.bfloat16)])
def test_backward_ring_padded_gradient(vce, dtype, gdt):
    """ce_backward on the stage ring into a wider gradient buffer (ld_grad = V + 8): every entry
    of the view is written, the padding is not; weight-0 rows come out +0.0."""
    p = gen.custom(70, 5000, dtype, seed=31, std=2.0, n_margin=7, margin=(17.0, 50.0), n_ignore=6)
    storage = p.full()
    logits = to_device(storage, dtype)
    labels = torch.from_numpy(p.labels).cuda()
    loss_out, loss_rows, stats, status = vce.ce_forward(logits, labels)
    gbuf = torch.full((p.T, 5008), 7.0, dtype=gdt, device="cuda")
    vce.ce_backward(logits, labels, stats, torch.full((1,), 0.5, device="cuda"), grad_logits=gbuf[:, :5000])
    torch.cuda.synchronize()
    ref = O.ce(O.widen(storage, dtype), p.labels, "mean", 0.5)
    grade_grad(gbuf[:, :5000], ref["grad"], p.margin_rows, p.labels)
    assert torch.all(gbuf[:, 5000:] == 7.0)
    ign = torch.from_numpy(p.labels == p.ignore_index).cuda()
    g = gbuf[:, :5000][ign].float()
    assert torch.all(g == 0) and not torch.any(torch.signbit(g))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_empty_batch(vce, dtype):
    """T = 0 rows through every CE entry point: the calls succeed, MEAN is 0/0 = NaN, SUM is 0,
    the status word is 0 (reading: mean over N = 0 rows, as torch)."""
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    logits = torch.empty(0, 1000, dtype=tdt, device="cuda")
    labels = torch.empty(0, dtype=torch.int64, device="cuda")
    for red, want in (("mean", None), ("sum", 0.0)):
        loss_out, loss_rows, stats, status = vce.ce_forward(logits, labels, -100, red)
        go = torch.ones(1, device="cuda")
        grad = vce.ce_backward(logits, labels, stats, go, -100, red)
        lo2, lr2, st2, g2, s2 = vce.ce_forward_backward(logits, labels, -100, red, grad_output=go)
        chunks = [torch.empty(0, 300, dtype=tdt, device="cuda"), torch.empty(0, 700, dtype=tdt, device="cuda")]
        lo3, lr3, st3, g3, cs3, s3 = vce.ce_merge_chunks(chunks, labels, -100, red, grad_output=go)
        torch.cuda.synchronize()
        for lo, s in ((loss_out, status), (lo2, s2), (lo3, s3)):
            assert vce.vce_get_status(s) == 0
            if want is None:
                assert np.isnan(lo.item())
            else:
                assert lo.item() == want
        assert grad.shape == (0, 1000) and g2.shape == (0, 1000) and [g.shape for g in g3] == [(0, 300), (0, 700)]


@pytest.mark.parametrize("seed", range(16))
def test_random_shapes(vce, seed):
    """Randomised shapes and options through the two-call path and the one-pass call: row counts
    from 1 to 700 (fewer than, about and several times the 152 CTAs), vocabularies that take the
    warp kernel, the stage ring with one or two consumer groups, the per-block kernel (not a
    multiple of 8) and clusters in the one pass; bf16 or fp32 logits and gradients, each
    reduction, ignored rows and raised targets.  Every output against the oracle."""
    rng = np.random.default_rng(1000 + seed)
    T = int(rng.choice([1, 7, 151, 152, 153])) if rng.random() < 0.4 else int(rng.integers(200, 700))
    V = int(rng.choice([int(rng.integers(2, 4000)), int(rng.integers(16001, 16400)) * 2 // 2,
                        int(rng.integers(4000, 8192)) * 8, int(rng.integers(8200, 12000)) * 8 + 3,
                        70000]))
    dtype = str(rng.choice(["bf16", "f32"]))
    gdt = [None, torch.float32, torch.bfloat16][int(rng.integers(0, 3))]
    reduction = str(rng.choice(["mean", "sum", "none"]))
    n_ignore = int(rng.integers(0, max(1, T // 4)))
    n_margin = int(rng.integers(0, max(1, T // 8)))
    p = gen.custom(T, V, dtype, seed=seed, std=2.0, n_margin=n_margin, margin=(17.0, 50.0), n_ignore=n_ignore)
    go = rng.uniform(0.25, 2.0, T) if reduction == "none" else float(rng.uniform(0.25, 2.0))
    full_check(vce, p, reduction, go, gdt)
    storage = p.full()
    logits = to_device(storage, dtype)
    labels = torch.from_numpy(p.labels).cuda()
    g = torch.empty(T if reduction == "none" else 1, device="cuda")
    g[:] = torch.as_tensor(go, dtype=torch.float32)
    out, rows, stats, grad, status = vce.ce_forward_backward(logits, labels, reduction=reduction, grad_output=g,
                                                             grad_dtype=gdt)
    torch.cuda.synchronize()
    assert vce.vce_get_status(status) == 0
    ref = O.ce(O.widen(storage, dtype), p.labels, reduction, go)
    G.check_loss_rows(rows.cpu().numpy(), ref["loss_rows"], ref["valid"])
    if reduction != "none":
        G.check_reduced(out.item(), ref["loss_out"])
    grade_grad(grad, ref["grad"], p.margin_rows, p.labels)

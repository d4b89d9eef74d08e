"""ce_forward_backward (one pass) through the C ABI: parity with the oracle and run-to-run
reproducibility, on both of its kernels.

Rows whose length and leading dimensions are multiples of 8 elements (16-byte aligned
buffers) are held in shared memory by a cluster of 1, 2, 4 or 8 CTAs (the smallest whose
column slices fit 128 KB); any other layout takes the kernel that re-reads the row from L2.
The shapes below name the path each one takes."""
import numpy as np
import pytest
import torch

import gen
from oracle import ce_oracle as O
from oracle import rounding as R
from tests import _grading as G
from tests.test_ce_gpu import TORCH_DT, grade_grad, to_device, vce  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


def fused(vce, p, reduction="mean", grad_output=1.0, grad_dtype=None, storage=None, logits=None, grad_logits=None):
    """Two calls on the same inputs: both succeed and agree bitwise.  Returns the first."""
    storage = p.full() if storage is None else storage
    logits = to_device(storage, p.dtype) if logits is None else logits
    labels = torch.from_numpy(p.labels).cuda()
    go = torch.empty(p.T if reduction == "none" else 1, device="cuda")
    go[:] = torch.as_tensor(grad_output, dtype=torch.float32)
    a = vce.ce_forward_backward(logits, labels, reduction=reduction, grad_output=go, grad_dtype=grad_dtype,
                                grad_logits=grad_logits)
    a = tuple(x.clone() if x is not None else None for x in a)
    b = vce.ce_forward_backward(logits, labels, reduction=reduction, grad_output=go, grad_dtype=grad_dtype,
                                grad_logits=grad_logits)
    torch.cuda.synchronize()
    assert vce.vce_get_status(a[4]) == 0 and vce.vce_get_status(b[4]) == 0
    for x, y in zip(a[:4], b[:4]):
        assert (x is None and y is None) or torch.equal(x, y), "one-pass outputs differ between two runs"
    return storage, a[0], a[1], a[3]


def check_against_oracle(p, storage, out, rows, grad, reduction="mean", go=1.0):
    ref = O.ce(O.widen(storage, p.dtype), p.labels, reduction, go)
    G.check_loss_rows(rows.cpu().numpy(), ref["loss_rows"], ref["valid"])
    if reduction != "none":
        G.check_reduced(out.item(), ref["loss_out"])
    grade_grad(grad, ref["grad"], p.margin_rows, p.labels)


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("dtype,gdt", [("bf16", None), ("bf16", torch.float32), ("f32", None), ("f32", torch.bfloat16)])
def test_fused_parity(vce, reduction, dtype, gdt):
    """V = 5000: shared-memory path, one CTA per row."""
    p = gen.custom(80, 5000, dtype, seed=61, std=2.5, n_margin=10, margin=(17.0, 50.0), n_ignore=5)
    go = np.linspace(0.25, 2.0, 80) if reduction == "none" else 0.5
    storage, out, rows, grad = fused(vce, p, reduction, go, gdt)
    check_against_oracle(p, storage, out, rows, grad, reduction, go)


@pytest.mark.parametrize("V", [1, 7, 1001, 4999])
def test_fused_odd_sizes(vce, V):
    """Row lengths that are not multiples of 8: the L2 re-read path."""
    p = gen.custom(21, V, "bf16", seed=V + 3, n_margin=3 if V > 1 else 0, n_ignore=2)
    storage, out, rows, grad = fused(vce, p)
    ref = O.ce(O.widen(storage, "bf16"), p.labels, "mean")
    G.check_loss_rows(rows.cpu().numpy(), ref["loss_rows"], ref["valid"])
    grade_grad(grad, ref["grad"])


@pytest.mark.parametrize("V,dtype,gdt", [
    (8, "bf16", None),                  # one CTA, one partial stage
    (70000, "bf16", None),              # 2-CTA cluster, 3 stages per slice
    (70000, "bf16", torch.float32),
    (128256, "f32", None),              # 4-CTA cluster, 4 full stages per slice
    (128256, "f32", torch.bfloat16),
    (400000, "bf16", None),             # 8-CTA cluster
])
def test_fused_cluster_sizes(vce, V, dtype, gdt):
    T = 24 if V > 100000 else 40
    p = gen.custom(T, V, dtype, seed=V % 9973 + 11, std=2.0, n_margin=6, margin=(17.0, 50.0), n_ignore=3)
    storage, out, rows, grad = fused(vce, p, "mean", 1.0, gdt)
    check_against_oracle(p, storage, out, rows, grad)


def test_fused_ring_wraps_over_many_rows(vce):
    """More rows than clusters: each CTA's stage ring wraps many times, the exchange parity
    alternates, ignored rows in between skip the ring."""
    p = gen.custom(600, 70000, "bf16", seed=77, std=2.0, n_margin=40, margin=(17.0, 50.0), n_ignore=60)
    storage, out, rows, grad = fused(vce, p, "none", np.linspace(0.5, 1.5, 600))
    check_against_oracle(p, storage, out, rows, grad, "none", np.linspace(0.5, 1.5, 600))


@pytest.mark.parametrize("T,V,dtype,reduction", [
    (2000, 5000, "bf16", "mean"),       # one CTA per row, one stage: 13-14 rows per CTA
    (600, 65536, "bf16", "none"),       # one CTA per row, four whole stages: three of the next row's beside them
    (1500, 70000, "bf16", "sum"),       # 2-CTA clusters, about 20 rows per cluster
    (300, 128256, "f32", "mean"),       # 4-CTA clusters
    (160, 400000, "bf16", "mean"),      # 8-CTA clusters, about 8 rows per cluster
])
def test_fused_many_rows_per_cta(vce, T, V, dtype, reduction):
    """Many rows per CTA or cluster, for every cluster size: the stage ring wraps many times
    and the hand-off slots, double-buffered by row parity, are rewritten many times."""
    p = gen.custom(T, V, dtype, seed=T + V, std=2.0, n_margin=T // 10, margin=(17.0, 50.0), n_ignore=T // 20)
    go = np.linspace(0.5, 1.5, T) if reduction == "none" else 1.0
    storage, out, rows, grad = fused(vce, p, reduction, go)
    check_against_oracle(p, storage, out, rows, grad, reduction, go)


@pytest.mark.parametrize("T,V", [(24, 20000), (152, 70000), (40, 128256)])
def test_folded_reduction_repeats_exactly(vce, T, V):
    """The one-pass kernel's in-kernel reduction (the CTA that finishes last sums the losses),
    every CTA finishing within microseconds of the others: 40 calls into buffers refilled with
    NaN give the same reduced loss bit for bit, and the oracle's value."""
    p = gen.custom(T, V, "bf16", seed=T + 2, std=2.0, n_ignore=2)
    storage = p.full()
    logits = to_device(storage, "bf16")
    labels = torch.from_numpy(p.labels).cuda()
    want = O.ce(O.widen(storage, "bf16"), p.labels, "mean")["loss_out"]
    go = torch.ones(1, device="cuda")
    rows = torch.empty(T, dtype=torch.float32, device="cuda")
    out = torch.empty(1, dtype=torch.float32, device="cuda")
    stats = torch.empty(T, 4, dtype=torch.float32, device="cuda")
    status = torch.empty(1, dtype=torch.int32, device="cuda")
    grad = torch.empty_like(logits)
    got = []
    for _ in range(40):
        rows.fill_(float("nan"))
        out.fill_(float("nan"))
        vce.ce_forward_backward(logits, labels, grad_output=go, grad_logits=grad, loss_rows=rows, loss_out=out,
                                row_stats=stats, status=status)
        got.append(out.item())
        assert vce.vce_get_status(status) == 0
    assert all(g == got[0] for g in got), got
    G.check_reduced(got[0], want)


@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_fused_beyond_the_folded_reduction(vce, reduction):
    """70000 rows of 16 bytes: more rows than the ring reduces in-kernel, so k_ce_count_valid runs
    before it (MEAN) and k_ce_reduce after it; checked in full against the oracle."""
    p = gen.custom(70000, 8, "bf16", seed=5, std=2.0, n_margin=700, margin=(17.0, 50.0), n_ignore=700)
    storage, out, rows, grad = fused(vce, p, reduction, 1.0)
    check_against_oracle(p, storage, out, rows, grad, reduction, 1.0)


def test_fused_padded_leading_dimensions(vce):
    """ld = V + 8 and ld_grad = V + 16 (shared-memory path): the padding is neither read into
    the statistics nor written."""
    p = gen.custom(50, 5000, "bf16", seed=8, n_margin=5, n_ignore=4)
    storage = p.full()
    wide = np.zeros((p.T, 5008), dtype=storage.dtype)
    wide[:, :5000] = storage
    wide[:, 5000:] = 0x42A0   # bf16 80.0: would dominate every row's sum if it were read
    logits = to_device(wide, "bf16")[:, :5000]
    gbuf = torch.full((p.T, 5016), 7.0, dtype=torch.bfloat16, device="cuda")
    storage, out, rows, grad = fused(vce, p, storage=storage, logits=logits, grad_logits=gbuf[:, :5000])
    check_against_oracle(p, storage, out, rows, grad)
    assert torch.all(gbuf[:, 5000:] == 7.0)


def test_fused_non_target_spikes(vce):
    """Values far above a thread's first group force the forward's rescale path."""
    p = gen.custom(64, 70000, "bf16", seed=19, std=1.0, n_ignore=2)
    z = O.widen(p.full(), "bf16")
    rng = np.random.default_rng(5)
    for r in range(p.T):
        cols = rng.choice(p.V, 6, replace=False)
        cols = cols[cols != p.labels[r]]
        z[r, cols] = rng.uniform(30.0, 60.0, len(cols))
    storage = R.bf16_bits(R.round_bf16(z))
    storage, out, rows, grad = fused(vce, p, storage=storage)
    check_against_oracle(p, storage, out, rows, grad)


@pytest.mark.parametrize("V", [300, 304])
def test_fused_all_ignored_and_bad_label(vce, V):
    p = gen.custom(6, V, "bf16", seed=5)
    logits = to_device(p.full(), "bf16")
    out = vce.ce_forward_backward(logits, torch.full((6,), -100, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert np.isnan(out[0].item()) and torch.all(out[3] == 0) and torch.all(out[1] == 0)
    lab = torch.from_numpy(p.labels).cuda()
    lab[2] = V
    out = vce.ce_forward_backward(logits, lab)
    assert vce.vce_get_status(out[4]) == 1 and torch.all(out[3][2] == 0) and np.isnan(out[1][2].item())


def test_fused_single_row(vce):
    p = gen.custom(1, 128256, "bf16", seed=2, n_margin=1, margin=(30.0, 30.0))
    storage, out, rows, grad = fused(vce, p)
    check_against_oracle(p, storage, out, rows, grad)


def test_fused_pages_shape(vce):
    """T=16384, V=128256 bf16 (2-CTA clusters): sampled rows against the oracle, including
    the collapse-regime margin rows."""
    p = gen.pages()
    storage, out, rows, grad = fused(vce, p)
    rng = np.random.default_rng(3)
    rr = np.unique(np.concatenate([p.margin_rows[:200], rng.choice(p.T, 100, replace=False)]))
    z = O.widen(storage[rr], "bf16")
    fwd = O.ce_rows(z, p.labels[rr])
    N = int(np.sum(p.labels != p.ignore_index))
    want = O.ce_grad_rows(z, p.labels[rr], fwd, O.row_scale(fwd["valid"], "sum", 1.0 / N))
    G.check_loss_rows(rows.cpu().numpy()[rr], fwd["loss"], fwd["valid"])
    G.check_grad_bf16(G.bf16_tensor_bits(grad[torch.from_numpy(rr).cuda()]), want)


@pytest.mark.parametrize("V,reduction", [(70000, "mean"), (70000, "none"), (20000, "sum")])
def test_one_pass_launch_slots(vce, V, reduction):
    """The one-pass ring claims rows from a per-launch slot of device words that its last CTA
    puts back to zero (2-CTA clusters at V = 70000: the cluster's first CTA hands each claim to
    its peer), and writes the status word itself.  1100 calls (more than the 1024 slots) into a
    status word filled with garbage and outputs filled with NaN each time: every checked call's
    status is 0 and its outputs equal the first call's, bit for bit; a call with a bad label in
    the middle sets VCE_ERR_LABEL and the calls after it are clean."""
    T = 300
    p = gen.custom(T, V, "bf16", seed=V + 5, std=2.0, n_margin=8, n_ignore=30)
    storage = p.full()
    logits = to_device(storage, "bf16")
    labels = torch.from_numpy(p.labels).cuda()
    bad_np = p.labels.copy()
    bad_np[41] = -9
    bad = torch.from_numpy(bad_np).cuda()
    go = torch.ones(T if reduction == "none" else 1, device="cuda")
    rows = torch.empty(T, dtype=torch.float32, device="cuda")
    out = torch.empty(1, dtype=torch.float32, device="cuda")
    stats = torch.empty(T, 4, dtype=torch.float32, device="cuda")
    grad = torch.empty_like(logits)
    status = torch.empty(1, dtype=torch.int32, device="cuda")
    first = None
    for i in range(1100):
        status.fill_(0x7FFF1234)
        if i % 50 == 0 or i in (500, 501):
            rows.fill_(float("nan"))
            out.fill_(float("nan"))
            grad.fill_(float("nan"))
        lab = bad if i == 500 else labels
        vce.ce_forward_backward(logits, lab, reduction=reduction, grad_output=go, grad_logits=grad, loss_rows=rows,
                                loss_out=out, row_stats=stats, status=status)
        if i == 500:
            assert vce.vce_get_status(status) == 1
            assert np.isnan(rows[41].item())
            continue
        if i % 50 and i != 501:
            continue
        assert vce.vce_get_status(status) == 0, i
        got = (rows.clone(), stats.clone(), grad.clone(), out.clone())
        if first is None:
            first = got
            check_against_oracle(p, storage, got[3], got[0], got[2], reduction)
        else:
            for x, y in zip(got[:3], first[:3]):
                assert torch.equal(x, y), i
            if reduction != "none":
                assert torch.equal(got[3], first[3]), i
    torch.cuda.synchronize()
    assert vce.vce_get_status(status) == 0


def test_stalled_ring_gives_up_and_the_context_survives(vce):
    """Stages that never complete (2-CTA clusters): the bounded waits give up with a status code,
    the kernel returns within seconds, and the next one-pass call on the same context is correct."""
    import time
    p = gen.custom(64, 70000, "bf16", seed=23, n_margin=4, n_ignore=2)
    logits = to_device(p.full(), "bf16")
    labels = torch.from_numpy(p.labels).cuda()
    t0 = time.time()
    status = vce.vce_test_ce_fused_stall(logits, labels, wait_ns=50_000_000)
    assert 105 <= status <= 109, status
    assert "gave up" in vce.vce_status_string(status)
    assert time.time() - t0 < 60
    storage, out, rows, grad = fused(vce, p)
    check_against_oracle(p, storage, out, rows, grad)

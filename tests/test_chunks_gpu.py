"""Parity of the vocabulary-chunked CE (ce_merge_chunks through the C ABI) with the oracle."""
import numpy as np
import pytest
import torch

import gen
from oracle import ce_oracle as O
from tests import _grading as G
from tests.test_ce_gpu import to_device, grade_grad, vce  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


def chunk_check(vce, p, widths, reduction="mean", grad_output=1.0):
    storage = p.full()
    offs = np.cumsum([0] + list(widths[:-1]))
    chunks_np = [np.ascontiguousarray(storage[:, o:o + w]) for o, w in zip(offs, widths)]
    chunks = [to_device(c, p.dtype) for c in chunks_np]
    labels = torch.from_numpy(p.labels).cuda()
    T = p.T
    go = torch.empty(T if reduction == "none" else 1, device="cuda")
    go[:] = torch.as_tensor(grad_output, dtype=torch.float32)
    loss_out, loss_rows, stats, grads, cstats, status = vce.ce_merge_chunks(chunks, labels, reduction=reduction,
                                                                             grad_output=go)
    torch.cuda.synchronize()
    assert vce.vce_get_status(status) == 0
    zs = [O.widen(c, p.dtype) for c in chunks_np]
    ref = O.ce_chunked(zs, offs, p.labels, sum(widths), reduction, grad_output)
    G.check_loss_rows(loss_rows.cpu().numpy(), ref["loss_rows"], ref["valid"])
    if reduction != "none":
        G.check_reduced(loss_out.item(), ref["loss_out"])
    for c, g in enumerate(grads):
        grade_grad(g, ref["grads"][c], what=f"chunk {c} grad")
    cs = cstats.cpu().numpy().astype(np.float64)
    v = ref["valid"]
    for c, (m, s, own, zt) in enumerate(ref["stats"]):
        assert np.array_equal(cs[c, :, 3] != 0, own), f"chunk {c}: owners"
        assert np.array_equal(cs[c, v, 0], m[v]), f"chunk {c}: maxima must be bit-exact"
        ok = v & (m > -np.inf)
        assert np.all(np.abs(cs[c, ok, 1] - s[ok]) <= 1e-5 * s[ok]), f"chunk {c}: sum-exp"
        assert np.array_equal(cs[c, own, 2], zt[own]), f"chunk {c}: target logit"
    return loss_rows, grads


# widths of whole 16-byte vectors in both dtypes ([1000], [64] * 16, [8] * 4, [4096, 8, 70000]) take
# the shared-memory stage ring for the chunk statistics; the others take one warp per item
@pytest.mark.parametrize("widths", [[7, 9, 1, 15], [1000], [1, 1, 998], [333, 334, 333], [64] * 16, [8] * 4,
                                    [4096, 8, 70000]])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chunks_small(vce, widths, dtype):
    p = gen.custom(50, sum(widths), dtype, seed=len(widths) * 7 + sum(widths), std=3.0, n_margin=8,
                   margin=(17.0, 50.0), n_ignore=4)
    chunk_check(vce, p, widths)


@pytest.mark.parametrize("reduction", ["sum", "none"])
def test_chunks_reductions(vce, reduction):
    p = gen.custom(40, 2000, "bf16", seed=77, n_margin=6, n_ignore=3)
    chunk_check(vce, p, [500, 700, 800], reduction, np.linspace(0.5, 1.5, 40) if reduction == "none" else 2.0)


def test_chunk_with_only_the_target(vce):
    z = np.array([[0.5, 2.0, -1.0], [3.0, 1.0, 0.0]], np.float32)
    labels = np.array([0, 2])
    chunks = [to_device(np.ascontiguousarray(z[:, :1]), "f32"), to_device(np.ascontiguousarray(z[:, 1:]), "f32")]
    out = vce.ce_merge_chunks(chunks, torch.from_numpy(labels).cuda(), reduction="sum")
    torch.cuda.synchronize()
    ref = O.ce(z.astype(np.float64), labels, "sum")
    G.check_loss_rows(out[1].cpu().numpy(), ref["loss_rows"], ref["valid"])
    cs = out[4].cpu().numpy()
    assert cs[0, 0, 0] == -np.inf and cs[0, 0, 1] == 0 and cs[0, 0, 3] == 1 and cs[0, 0, 2] == 0.5


def test_forward_only(vce):
    p = gen.custom(30, 900, "bf16", seed=5, n_margin=3, n_ignore=2)
    storage = p.full()
    chunks = [to_device(np.ascontiguousarray(storage[:, o:o + 300]), "bf16") for o in (0, 300, 600)]
    loss_out, loss_rows, stats, grads, cs, status = vce.ce_merge_chunks(chunks, torch.from_numpy(p.labels).cuda(),
                                                                        want_grad=False)
    torch.cuda.synchronize()
    assert grads is None
    ref = O.ce(O.widen(storage, "bf16"), p.labels, "mean")
    G.check_loss_rows(loss_rows.cpu().numpy(), ref["loss_rows"], ref["valid"])


def test_chunked_invalid_label(vce):
    p = gen.custom(6, 40, "f32", seed=6)
    labels = p.labels.copy()
    labels[2] = 40
    st = p.full()
    chunks = [to_device(np.ascontiguousarray(st[:, :20]), "f32"), to_device(np.ascontiguousarray(st[:, 20:]), "f32")]
    out = vce.ce_merge_chunks(chunks, torch.from_numpy(labels).cuda())
    assert vce.vce_get_status(out[5]) == 1
    assert np.isnan(out[1][2].item()) and torch.all(out[3][0][2] == 0) and torch.all(out[3][1][2] == 0)


def test_pages_chunked_matches_unchunked_and_oracle(vce):
    """The pages' matrix as 8 column chunks of 16032 in separate buffers."""
    p = gen.pages()
    storage = p.full()
    bounds = gen.chunk_bounds(p.V, gen.CHUNKS)
    chunks = [to_device(gen.copy_cols(storage, o, w), "bf16") for o, w in bounds]
    labels = torch.from_numpy(p.labels).cuda()
    loss_out, loss_rows, stats, grads, cstats, status = vce.ce_merge_chunks(chunks, labels)
    full = to_device(storage, "bf16")
    u_out, u_rows, u_stats, u_status = vce.ce_forward(full, labels)
    u_grad = vce.ce_backward(full, labels, u_stats, torch.ones(1, device="cuda"))
    torch.cuda.synchronize()
    assert vce.vce_get_status(status) == 0
    lr, ur = loss_rows.cpu().numpy(), u_rows.cpu().numpy()
    valid = p.labels != p.ignore_index
    rel = np.abs(lr[valid] - ur[valid]) / np.abs(ur[valid])
    assert rel.max() <= 1e-4, rel.max()
    assert abs(loss_out.item() - u_out.item()) <= 1e-5 * abs(u_out.item())
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([p.margin_rows[:300], rng.choice(p.T, 200, replace=False)]))
    idx = torch.from_numpy(rows).cuda()
    cat = torch.cat([g.index_select(0, idx) for g in grads], dim=1)
    ug = u_grad.index_select(0, idx)
    d = G.bf16_tensor_bits(cat).astype(np.int64) - G.bf16_tensor_bits(ug).astype(np.int64)
    assert np.abs(d).max() <= 2   # each side is within one ulp of the same rounded oracle value
    N = int(valid.sum())
    z = O.widen(storage[rows], "bf16")
    fwd = O.ce_rows(z, p.labels[rows])
    G.check_loss_rows(lr[rows], fwd["loss"], fwd["valid"])
    want = O.ce_grad_rows(z, p.labels[rows], fwd, O.row_scale(fwd["valid"], "sum", 1.0 / N))
    G.check_grad_bf16(G.bf16_tensor_bits(cat), want, "chunked grad")
    # merged global max over non-target columns equals the unchunked row max, bit for bit
    cs = cstats.cpu().numpy()
    own = cs[:, :, 3] != 0
    assert np.all(own.sum(0)[valid] == 1) and np.all(own.sum(0)[~valid] == 0)
    M = cs[:, rows, 0].max(axis=0)
    assert np.array_equal(M[fwd["valid"]].astype(np.float64), fwd["max_nt"][fwd["valid"]])


@pytest.mark.parametrize("seed", range(10))
def test_random_chunkings(vce, seed):
    """Randomised chunkings against the oracle: 1 to 16 chunks, widths that are and are not
    whole 16-byte vectors (the backward ring's items or the per-block kernel), row counts about
    and beyond the 152 CTAs, either logits dtype, each reduction, ignored rows and raised
    targets."""
    rng = np.random.default_rng(3000 + seed)
    k = int(rng.integers(1, 17))
    widths = [int(rng.choice([int(rng.integers(1, 40)), 8 * int(rng.integers(1, 600)), int(rng.integers(1, 9000))]))
              for _ in range(k)]
    T = int(rng.choice([1, 152, 153])) if rng.random() < 0.3 else int(rng.integers(100, 600))
    dtype = str(rng.choice(["bf16", "f32"]))
    reduction = str(rng.choice(["mean", "sum", "none"]))
    go = rng.uniform(0.25, 2.0, T) if reduction == "none" else float(rng.uniform(0.25, 2.0))
    p = gen.custom(T, sum(widths), dtype, seed=seed, std=2.5, n_margin=int(rng.integers(0, max(1, T // 8))),
                   margin=(17.0, 50.0), n_ignore=int(rng.integers(0, max(1, T // 5))))
    chunk_check(vce, p, widths, reduction, go)

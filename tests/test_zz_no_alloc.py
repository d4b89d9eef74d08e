"""ce_merge_chunks_noalloc: the chunked CE for callers that cannot allocate device memory.

Such callers (a host program that drives the library through its C ABI with no device
memory manager of its own, or an engine that hands all device memory to one arena at
start-up) cannot supply the chunk-statistics workspace that ce_merge_chunks takes.  The
no-allocation entry point keeps those statistics in an array the library defines in device
memory.  These tests check, through the C ABI, that it gives what ce_merge_chunks gives on
two calls in a row (the second with different data and sizes, so stale contents of the
shared array would show), and that sizes beyond its array are refused.

This file is named to be collected last: it must pass on its own in a fresh process and
after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import gen
from tests import _grading as G

pytestmark = pytest.mark.gpu


def _vce():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    import vocab_cross_entropy_gb300 as v
    return v


def _device_chunks(p, widths):
    storage = p.full()
    t = torch.from_numpy(storage.view(np.int16) if p.dtype == "bf16" else storage)
    if p.dtype == "bf16":
        t = t.view(torch.bfloat16)
    full = t.cuda()
    offs = np.cumsum([0] + list(widths[:-1]))
    return [full[:, o:o + w].contiguous() for o, w in zip(offs, widths)]


def _bf16_values(bits):
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _outputs(T, chunks, reduction):
    dev = chunks[0].device
    return dict(loss_rows=torch.full((T,), -1.0, device=dev),
                loss_out=torch.full((1,), -1.0, device=dev),
                row_stats=torch.full((T, 4), -1.0, device=dev),
                status=torch.full((1,), -7, dtype=torch.int32, device=dev),
                chunk_grads=[torch.full_like(c, 5.0) for c in chunks])


def _compare_one_call(vce, p, widths, reduction, go_value):
    chunks = _device_chunks(p, widths)
    labels = torch.from_numpy(p.labels).cuda()
    T = p.T
    go = torch.full((T if reduction == "none" else 1,), go_value, device="cuda")

    ref = vce.ce_merge_chunks(chunks, labels, reduction=reduction, grad_output=go)
    mine = _outputs(T, chunks, reduction)
    vce.ce_merge_chunks_noalloc(chunks, labels, reduction=reduction, grad_output=go, **mine)
    torch.cuda.synchronize()

    assert vce.vce_get_status(ref[5]) == 0 and vce.vce_get_status(mine["status"]) == 0
    valid = p.labels != p.ignore_index
    G.check_loss_rows(mine["loss_rows"].cpu().numpy(), ref[1].cpu().numpy().astype(np.float64), valid,
                      "no-alloc loss rows")
    if reduction != "none":
        G.check_reduced(mine["loss_out"].item(), ref[0].item(), "no-alloc reduced loss")
    rs_ref, rs = ref[2].cpu().numpy().astype(np.float64), mine["row_stats"].cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(rs, rs_ref, rtol=1e-6, atol=0)
    for c, (g_ref, g) in enumerate(zip(ref[3], mine["chunk_grads"])):
        if g.dtype == torch.bfloat16:
            G.check_grad_bf16(G.bf16_tensor_bits(g), _bf16_values(G.bf16_tensor_bits(g_ref)), f"chunk {c} gradient")
        else:
            G.check_grad_f32(g.cpu().numpy(), g_ref.cpu().numpy().astype(np.float64), f"chunk {c} gradient")


def test_noalloc_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    vce = _vce()
    # first call: 8 bf16 chunks of a 4096-row matrix, mean reduction
    p1 = gen.custom(4096, 8000, "bf16", seed=501, std=2.0, n_margin=400, margin=(17.0, 50.0), n_ignore=41)
    _compare_one_call(vce, p1, [1000] * 8, "mean", 1.0)
    # second call right after: other data, 13 fp32 chunks, k * T = 260000 (just under the
    # 262144-entry array), sum reduction
    w2 = [97, 100, 131, 64, 1, 300, 77, 90, 210, 33, 150, 8, 39]
    p2 = gen.custom(20000, sum(w2), "f32", seed=502, std=3.0, n_margin=2000, margin=(20.0, 40.0), n_ignore=200)
    _compare_one_call(vce, p2, w2, "sum", 0.5)


def test_noalloc_after_a_larger_call_with_another_chunk_count():
    """A large call, then a smaller one with a different k and T: the array still holds the
    large call's statistics in the entries past the small call's k * T, and in the same
    entries under the other [k][T] layout, so a read at a wrong stride or with a stale k or T
    would pick up values that are not this call's."""
    vce = _vce()
    w1 = [200, 200, 200, 200, 416]
    p1 = gen.custom(50000, sum(w1), "bf16", seed=503, std=2.0, n_margin=5000, margin=(17.0, 50.0), n_ignore=500)
    _compare_one_call(vce, p1, w1, "mean", 1.0)
    w2 = [300, 129, 700]
    p2 = gen.custom(3001, sum(w2), "bf16", seed=504, std=2.5, n_margin=300, margin=(20.0, 45.0), n_ignore=30)
    _compare_one_call(vce, p2, w2, "none", 0.75)


def test_noalloc_refuses_sizes_beyond_its_array():
    vce = _vce()
    lib = vce.lib
    T = vce.NOALLOC_MAX_CHUNK_ROWS // 2 + 1   # k = 2 chunks: k * T one row past the limit
    P = ctypes.c_void_p
    ptrs = (P * 2)(P(0x1000), P(0x1000))
    widths = (ctypes.c_int64 * 2)(4, 4)
    rc = lib.ce_merge_chunks_noalloc(2, ptrs, widths, widths, 1, T, P(0x1000), -100, 2, P(0x1000), P(0x1000),
                                     P(0x1000), P(0x1000), None, None, 1, P(0x1000), None)
    assert rc == -10 and "scratch" in vce.vce_status_string(rc)

"""The debug build of the library (device-side index checks; python -m
vocab_cross_entropy_gb300.build --debug-checks makes libvce_debug.so).

On valid inputs of every kernel family -- the per-block and shared-memory-ring CE forward and
backward, the chunk statistics and merge, the one-pass call on a CTA cluster and its per-block
fallback, and the tensor-core GEMMs of the linear-CE on CTA pairs and single CTAs -- no index
check fails (vce_debug_status() == 0), and every output equals the release
build's bit for bit: the checks only guard accesses, they change no arithmetic.
"""
import numpy as np
import pytest
import torch

import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_library():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from vocab_cross_entropy_gb300 import build as b
    return b.build(debug_checks=True)   # compiled on first use


def _dev(p):
    storage = p.full()
    t = torch.from_numpy(storage.view(np.int16) if p.dtype == "bf16" else storage)
    if p.dtype == "bf16":
        t = t.view(torch.bfloat16)
    return t.cuda(), torch.from_numpy(p.labels).cuda()


def _run_everything(vce):
    """Outputs of one call of each kernel family on fixed valid inputs."""
    out = []
    for T, V, dt in ((300, 4096, "bf16"), (200, 1001, "f32"), (64, 129000, "bf16")):
        p = gen.custom(T, V, dt, seed=T + V, std=2.0, n_margin=T // 10, margin=(17.0, 40.0), n_ignore=3)
        logits, labels = _dev(p)
        loss_out, loss_rows, stats, status = vce.ce_forward(logits, labels)
        grad = vce.ce_backward(logits, labels, stats, torch.ones(1, device="cuda"))
        out += [loss_out, loss_rows, stats, grad]
        out += list(vce.ce_forward_backward(logits, labels)[:4])
        k = 4
        w = V // k
        chunks = [logits[:, c * w: (c + 1) * w if c < k - 1 else V].contiguous() for c in range(k)]
        merged = vce.ce_merge_chunks(chunks, labels)
        out += [merged[0], merged[1], merged[2]] + list(merged[3])
    p = gen.linear_custom(512, 128, 1000, seed=77, n_ignore=5)
    E = torch.from_numpy(p.E().view(np.int16)).view(torch.bfloat16).cuda()
    W = torch.from_numpy(p.W().view(np.int16)).view(torch.bfloat16).cuda()
    lab = torch.from_numpy(p.labels).cuda()
    out += list(vce.linear_ce_fwd_bwd(E, W, lab)[:4])
    out += list(vce.linear_ce_fwd_bwd(E[:384], W, lab[:384])[:4])     # 3 row tiles: single CTAs
    for pair in (0, 1):
        out.append(vce.vce_gemm_bf16_variant(E, W, pair=pair))
    torch.cuda.synchronize()
    return [t.clone() for t in out]


def test_debug_build_finds_no_bad_index_and_changes_nothing(debug_library):
    import vocab_cross_entropy_gb300 as vce
    release = _run_everything(vce)
    assert not vce.vce_debug_checks()
    prev = vce.use_library(debug_library)
    try:
        assert vce.vce_debug_checks()
        assert vce.vce_debug_status() == 0
        debug = _run_everything(vce)
        assert vce.vce_debug_status() == 0, vce.vce_status_string(vce.vce_debug_status())
    finally:
        vce.restore_library(prev)
    assert len(release) == len(debug)
    for i, (a, b) in enumerate(zip(release, debug)):
        assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8)), f"output {i} differs"

"""The tensor-core GEMM building block (vce_gemm_bf16) with K-major and MN-major operands,
against a float64 matrix product of the same bf16 values."""
import numpy as np
import pytest
import torch

from oracle import ce_oracle as O
from tests.test_ce_gpu import vce  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


def _bf16(rng, shape, std=1.0):
    x = torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    return x, O.widen(bits, "bf16")


@pytest.mark.parametrize("a_mn", [False, True])
@pytest.mark.parametrize("b_mn", [False, True])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 320), (136, 264, 72), (8, 8, 8), (384, 768, 1024),
                                   (2560, 4096, 128)])
def test_gemm_layouts(vce, a_mn, b_mn, M, N, K):
    rng = np.random.default_rng(M * 7 + N + K + 2 * a_mn + b_mn)
    A, A64 = _bf16(rng, (K, M) if a_mn else (M, K))
    B, B64 = _bf16(rng, (K, N) if b_mn else (N, K), 0.05)
    C = vce.vce_gemm_bf16(A.cuda(), B.cuda(), a_mn, b_mn)
    torch.cuda.synchronize()
    Am = A64.T if a_mn else A64
    Bm = B64.T if b_mn else B64
    want = Am @ Bm.T
    bound = 2.0 ** -20 * (np.abs(Am) @ np.abs(Bm).T) + 1e-30
    err = np.abs(C.cpu().numpy().astype(np.float64) - want)
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound):.3g}"


@pytest.mark.parametrize("pair", [0, 1, 2])
@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (True, True), (False, True), (True, False)])
@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (256, 256, 128), (512, 384, 1000), (2560, 640, 1536)])
def test_gemm_variants(vce, pair, a_mn, b_mn, M, N, K):
    """The three launch forms of the GEMM -- single CTAs, CTA pairs issuing cta_group::2 MMAs,
    and pairs taking two K blocks per stage -- against a float64 product of the same bf16
    values.  The last form refuses an odd count of 64-column K blocks."""
    rng = np.random.default_rng(M + 3 * N + K + 5 * pair + 7 * a_mn + 11 * b_mn)
    A, A64 = _bf16(rng, (K, M) if a_mn else (M, K))
    B, B64 = _bf16(rng, (K, N) if b_mn else (N, K), 0.05)
    if pair == 2 and (K + 63) // 64 % 2:
        with pytest.raises(vce.VceError):
            vce.vce_gemm_bf16_variant(A.cuda(), B.cuda(), a_mn, b_mn, pair=pair)
        return
    C = vce.vce_gemm_bf16_variant(A.cuda(), B.cuda(), a_mn, b_mn, pair=pair)
    torch.cuda.synchronize()
    Am = A64.T if a_mn else A64
    Bm = B64.T if b_mn else B64
    want = Am @ Bm.T
    bound = 2.0 ** -20 * (np.abs(Am) @ np.abs(Bm).T) + 1e-30
    err = np.abs(C.cpu().numpy().astype(np.float64) - want)
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound):.3g}"


def test_pairs_and_single_ctas_agree_bitwise(vce):
    """The three launch forms accumulate each tile's K blocks in the same order: equal bits."""
    rng = np.random.default_rng(17)
    A, _ = _bf16(rng, (1024, 2048))
    B, _ = _bf16(rng, (768, 2048), 0.05)
    C1 = vce.vce_gemm_bf16_variant(A.cuda(), B.cuda(), pair=0)
    C2 = vce.vce_gemm_bf16_variant(A.cuda(), B.cuda(), pair=1)
    C3 = vce.vce_gemm_bf16_variant(A.cuda(), B.cuda(), pair=2)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
    assert torch.equal(C1, C3)


def test_gemm_variant_refuses_bad_arguments(vce):
    A = torch.zeros(384, 128, dtype=torch.bfloat16, device="cuda")   # 3 M tiles: no pairs
    B = torch.zeros(256, 128, dtype=torch.bfloat16, device="cuda")
    for pair in (1, 2, -1):
        with pytest.raises(vce.VceError):
            vce.vce_gemm_bf16_variant(A, B, pair=pair)


@pytest.mark.parametrize("M", [128, 256])   # single CTAs; a CTA pair
def test_stalled_pipeline_gives_up_and_the_context_survives(vce, M):
    """A stage that never completes: the bounded waits give up with a status code, the kernel
    returns (both CTAs of a pair), and the next GEMM on the same context is correct."""
    import time
    rng = np.random.default_rng(5)
    A, A64 = _bf16(rng, (M, 128))
    B, B64 = _bf16(rng, (512, 128), 0.05)
    Ad, Bd = A.cuda(), B.cuda()
    t0 = time.time()
    status = vce.vce_test_gemm_stall(Ad, Bd, wait_ns=50_000_000)
    assert status in (101, 102, 103, 104), status
    assert "gave up" in vce.vce_status_string(status)
    assert time.time() - t0 < 60
    C = vce.vce_gemm_bf16(Ad, Bd)
    torch.cuda.synchronize()
    want = A64 @ B64.T
    bound = 2.0 ** -20 * (np.abs(A64) @ np.abs(B64).T) + 1e-30
    assert np.all(np.abs(C.cpu().numpy().astype(np.float64) - want) <= bound)


@pytest.mark.parametrize("M,N,K", [(512, 512, 1000), (1024, 256, 4160), (384, 512, 256)])
def test_k_block_skipping(vce, M, N, K):
    """The K-block skipping gradient filtering rides on, against float64: each 128-row M tile
    adds only the 128-column K blocks whose bit is set (a ragged last block included); one tile
    keeps none (its accumulator is never written: zeros), one keeps all."""
    rng = np.random.default_rng(M + K)
    A, A64 = _bf16(rng, (M, K))
    B, B64 = _bf16(rng, (N, K), 0.05)
    tiles, nblk = -(-M // 128), -(-K // 128)
    words = -(-nblk // 32) + 1   # one spare word: rows may be longer than needed
    keep = rng.random((tiles, nblk)) < 0.4
    keep[1] = False
    keep[2] = True
    bits = np.zeros((tiles, words), np.uint32)
    for t in range(tiles):
        for b in np.nonzero(keep[t])[0]:
            bits[t, b // 32] |= np.uint32(1) << np.uint32(b % 32)
    C = vce.vce_test_gemm_skip(A.cuda(), B.cuda(), torch.from_numpy(bits.view(np.int32)).cuda())
    torch.cuda.synchronize()
    kmask = np.repeat(keep, 128, axis=1)[:, :K]                    # [tiles, K]
    Am = A64 * np.repeat(kmask, 128, axis=0)[:M]                   # dropped blocks of each tile zeroed
    want = Am @ B64.T
    bound = 2.0 ** -20 * (np.abs(Am) @ np.abs(B64).T) + 1e-30
    got = C.cpu().numpy().astype(np.float64)
    assert np.all(got[128:256] == 0.0), "a tile with no kept block must be zero"
    assert np.all(np.abs(got - want) <= bound), f"max err/bound {np.max(np.abs(got - want) / bound):.3g}"


def test_k_block_skipping_refuses_bad_arguments(vce):
    A = torch.zeros(384, 128, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(256, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(vce.VceError):
        vce.vce_test_gemm_skip(A, B, torch.zeros(3, 0, dtype=torch.int32, device="cuda"))

"""The tcgen05 projection kernel alone, through dflash_gemm_bf16, against an
fp64 matmul of the same bf16 inputs (a library primitive, not the CUDA path).

Shapes cover every activation tile width (16..256), ragged output widths and
reduction depths (TMA zero fill), several row tiles and split-K."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K,splits", [
    (1, 128, 64, 1), (16, 256, 512, 1), (5, 200, 72, 1), (17, 384, 1024, 3), (33, 1000, 520, 2),
    (64, 128, 4096, 6), (100, 130, 200, 1), (256, 256, 256, 1), (300, 640, 384, 4), (512, 1024, 2880, 1),
])
def test_gemm_bf16_matches_fp64(M, N, K, splits):
    import torch
    from block_diffusion_speculative_hidden_gb300 import gemm_bf16
    rng = np.random.default_rng(M * 7 + N + K)
    W = synth.round_to_bf16(rng.standard_normal((N, K)).astype(np.float32) * 0.05)
    X = synth.round_to_bf16(rng.standard_normal((M, K)).astype(np.float32))
    Wd = torch.from_numpy(W).cuda().bfloat16()
    Xd = torch.from_numpy(X).cuda().bfloat16()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gemm_bf16(Wd, Xd, splits=splits, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.sum(0).double().cpu().numpy()
    ref = X.astype(np.float64) @ W.astype(np.float64).T
    # fp32 accumulation of K bf16 products: error ~ sqrt(K) * 2^-24 * |terms|
    tol = 1e-5 * np.sqrt(K) * 4
    np.testing.assert_allclose(got, ref, atol=tol, rtol=1e-5)
    # each split is the sum over its own k-blocks
    used = out.shape[0]
    per = -(-((K + 63) // 64) // used)
    s0 = out[0].double().cpu().numpy()
    k1 = min(K, per * 64)
    np.testing.assert_allclose(s0, X[:, :k1].astype(np.float64) @ W[:, :k1].astype(np.float64).T, atol=tol,
                               rtol=1e-5)


@pytest.mark.parametrize("M,N,K,splits", [(16, 256, 512, 2), (17, 300, 1000, 1), (100, 384, 264, 3), (128, 128, 64, 1),
                                          (200, 640, 4096, 1),
                                          # many rows: the persistent kernel, 128-row activation tiles
                                          (2048, 5760, 2880, 1),
                                          # persistent, ragged rows, columns and depth
                                          (1000, 20000, 1000, 1), (512, 4000, 520, 1)])
def test_gemm_bf16_hi_lo_pair(M, N, K, splits):
    """Activations as an exact hi + lo pair: the product keeps ~16 bits of x.
    From 256 rows with at least a full wave of output tiles the projection
    runs on the persistent kernel (one CTA an SM over many tiles, two TMEM
    accumulators); the same check holds there."""
    import torch
    from block_diffusion_speculative_hidden_gb300 import gemm_bf16
    rng = np.random.default_rng(M + 3 * N + K)
    W = synth.round_to_bf16(rng.standard_normal((N, K)).astype(np.float32) * 0.05)
    x = rng.standard_normal((M, K)).astype(np.float32)
    hi = synth.round_to_bf16(x)
    lo = synth.round_to_bf16(x - hi)
    out = gemm_bf16(torch.from_numpy(W).cuda().bfloat16(), torch.from_numpy(hi).cuda().bfloat16(),
                    splits=splits, X_lo=torch.from_numpy(lo).cuda().bfloat16())
    got = out.sum(0).double().cpu().numpy()
    ref = (hi.astype(np.float64) + lo.astype(np.float64)) @ W.astype(np.float64).T
    np.testing.assert_allclose(got, ref, atol=4e-5 * np.sqrt(K), rtol=1e-5)
    # and against the unsplit x: the pair's error is far below bf16 rounding
    ref_x = x.astype(np.float64) @ W.astype(np.float64).T
    assert np.abs(got - ref_x).max() < 3e-4 * np.sqrt(K) * 0.05

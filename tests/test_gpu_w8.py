"""The E4M3-weight projection kernel (dflash_gemm_w8) against the oracle's
reading of the FP8 weight format: out = diag(s) . decode(codes) applied to
the exact activations (hi + lo), in fp64, on ragged shapes that reach every
tile width (16..256 activation rows), split-K, k tails shorter than a
64-wide block and weight-row counts that are not multiples of the 128-row
tile.  Each split's partial plane is checked on its own k-range."""
import numpy as np
import pytest

from oracle import dflash_oracle as O

pytestmark = pytest.mark.gpu

# (N weight rows, K, M activation rows, requested splits, hi+lo activations)
SHAPES = [
    (300, 208, 1, 1, True),       # k tail of 16 in the last block, ragged N
    (200, 1216, 3, 4, True),      # 19 k-blocks in four splits: the last split's last stage is half empty
    (517, 1344, 16, 3, True),     # BN = 16, three splits
    (1024, 4096, 37, 4, True),    # BN = 64
    (256, 512, 129, 2, True),     # BN = 128 (hi+lo)
    (130, 528, 200, 1, False),    # BN = 256 (one bf16 term)
    (6144, 4096, 16, 1, True),    # c2's QKV shape
]


def _data(N, K, M, seed):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, size=(N, K)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x00                  # no NaN codes
    scale = (rng.random(N).astype(np.float32) * 1e-3 + 1e-4).astype(np.float32)
    x = rng.standard_normal((M, K)).astype(np.float32)
    return codes, scale, x


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "N{}_K{}_M{}_s{}_{}".format(*s))
def test_w8_gemm_matches_decoded_fp64_product(shape):
    import torch
    from block_diffusion_speculative_hidden_gb300 import gemm_w8
    N, K, M, splits, lo = shape
    codes, scale, x = _data(N, K, M, seed=N * 7 + K + M)
    xt = torch.from_numpy(x)
    hi = xt.bfloat16()
    x_lo = (xt - hi.float()).bfloat16() if lo else None
    dev = torch.device("cuda")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = gemm_w8(torch.from_numpy(codes).to(dev), torch.from_numpy(scale).to(dev), hi.to(dev),
                  splits=splits, status=status, X_lo=None if x_lo is None else x_lo.to(dev))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.cpu().numpy().astype(np.float64)              # [splits_used, M, N]
    xs = hi.double().numpy() + (x_lo.double().numpy() if lo else 0.0)
    w = O.decode_e4m3(codes)                                # [N, K] fp64, exact
    n_kb = -(-K // 64)
    per = -(-n_kb // min(splits, n_kb))
    per += per & 1                                          # whole two-k-block stages per split
    assert got.shape[0] == -(-n_kb // per)
    for s in range(got.shape[0]):
        k0, k1 = s * per * 64, min(K, (s + 1) * per * 64)
        ref = (xs[:, k0:k1] @ w[:, k0:k1].T) * scale.astype(np.float64)[None, :]
        # fp32 accumulation of exact products: bound by K * 2^-23 * sum |terms|
        mag = (np.abs(xs[:, k0:k1]) @ np.abs(w[:, k0:k1]).T) * scale.astype(np.float64)[None, :]
        err = np.abs(got[s] - ref)
        assert np.all(err <= (k1 - k0) * 2.0 ** -23 * mag + 1e-30), (s, err.max(), mag.max())

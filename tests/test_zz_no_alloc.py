"""dflash_gemm_bf16_noalloc, the projection entry point for callers that
cannot allocate device memory (their HBM belongs to another allocator, or
they cannot take cudaMalloc's implicit synchronisation).  It keeps its
split-K partials in a fixed array inside the library, so it is checked here
against the regular entry point, whose partials live in caller memory.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.  Calls go straight through
the C ABI with ctypes."""
import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _inputs(M, N, K, seed, with_lo):
    import torch
    rng = np.random.default_rng(seed)
    W = synth.round_to_bf16(rng.standard_normal((N, K)).astype(np.float32) * 0.05)
    x = rng.standard_normal((M, K)).astype(np.float32)
    hi = synth.round_to_bf16(x)
    lo = synth.round_to_bf16(x - hi) if with_lo else None
    dev = lambda a: None if a is None else torch.from_numpy(a).cuda().bfloat16().contiguous()
    return dev(W), dev(hi), dev(lo)


def _regular(L, W, X, X_lo, splits):
    """The existing entry point: partials [splits_used, M, N] in caller memory, summed in split order."""
    import torch
    N, K = W.shape
    M = X.shape[0]
    n_kb = (K + 63) // 64
    want = min(splits, n_kb)
    per = (n_kb + want - 1) // want
    used = (n_kb + per - 1) // per
    part = torch.empty((used, M, N), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = ctypes.c_int(0)
    rc = L.dflash_gemm_bf16(_ptr(W), N, K, _ptr(X), _ptr(X_lo), M, _ptr(part), splits, ctypes.byref(got),
                            _ptr(status), _stream())
    assert rc == 0 and got.value == used
    acc = part[0].clone()
    for s in range(1, used):
        acc += part[s]
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return acc, used


def test_noalloc_matches_regular_entry_on_two_calls_in_a_row():
    import torch
    from block_diffusion_speculative_hidden_gb300 import _lib
    L = _lib.lib()
    # the second call reuses the shared array; the third reports device
    # errors through a status word of its own, which must stay clear
    cases = [(16, 640, 1024, 4, True, False), (33, 200, 520, 3, False, False), (64, 384, 768, 2, True, True)]
    for i, (M, N, K, splits, with_lo, own_status) in enumerate(cases):
        W, X, X_lo = _inputs(M, N, K, 100 + i, with_lo)
        ref, used = _regular(L, W, X, X_lo, splits)
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda") if own_status else None
        got = ctypes.c_int(0)
        rc = L.dflash_gemm_bf16_noalloc(_ptr(W), N, K, _ptr(X), _ptr(X_lo), M, _ptr(out), splits,
                                        ctypes.byref(got), _ptr(status), _stream())
        torch.cuda.synchronize()
        assert rc == 0 and got.value == used
        if own_status:
            assert int(status.item()) == 0
        # the tolerance of the projection tests (fp32 accumulation of K products)
        np.testing.assert_allclose(out.cpu().numpy(), ref.cpu().numpy(), atol=4e-5 * np.sqrt(K), rtol=1e-5)


def test_noalloc_rejects_requests_beyond_its_scratch():
    import torch
    from block_diffusion_speculative_hidden_gb300 import _lib
    L = _lib.lib()
    M, N, K = 256, 8192, 256          # 2 splits x 256 x 8192 floats > the 2^21 - 64 that fit
    W, X, _ = _inputs(M, N, K, 7, False)
    out = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    rc = L.dflash_gemm_bf16_noalloc(_ptr(W), N, K, _ptr(X), None, M, _ptr(out), 2, None, None, _stream())
    torch.cuda.synchronize()
    assert rc == 7                    # DFLASH_ERR_TOO_LARGE, nothing enqueued
    assert float(out.abs().max().item()) == 0.0

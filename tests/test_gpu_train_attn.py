"""Training-time block attention (dflash_block_attention) against the
oracle's per-block masked attention.

Sequences' context keys and values are seeded fp16 values written straight
into the pool's pages under a page table of the test's own (the kernel and
the oracle read the same values); blocks pick a sequence and a prefix
length at random, including the edge lengths 0, 15, 16, 17 and the whole
context.  Both attention tile shapes are covered (G = 4: 64 query rows per
kv head; G = 8: 128).  Tolerance: probabilities are rounded to fp16 for the
P.V product (relative 2^-11), so |error| <= 2^-11 * max|v| plus fp32
accumulation: 3e-3 for N(0, 1) values."""
import numpy as np
import pytest

import synth
from oracle import dflash_oracle as O

pytestmark = pytest.mark.gpu

TOL = 3e-3


def _setup(name, S, NB, seed, ramp=0.0):
    import torch
    from block_diffusion_speculative_hidden_gb300 import Drafter, weights_to_device
    cfg = synth.get_config(name).replace(n_layers=2)
    rng = np.random.default_rng(seed)
    Hkv, dh, Hq = cfg.n_kv_heads, cfg.head_dim, cfg.n_q_heads
    T = rng.integers(20, 300, size=S)
    T[0] = 16                                   # a context of exactly one page
    mpps = 20
    dr = Drafter(cfg, weights_to_device(synth.make_weights(cfg), cfg.dtype), max_batch=NB,
                 max_pages_per_seq=mpps, n_pages=S * mpps, max_rows=17, max_inject_rows=NB * 17)
    Kp, Vp = dr.pool_kv()                       # [L, pages, Hkv, 16, dh] fp16
    layer = 1
    ctx_k = [rng.standard_normal((t, Hkv, dh)) for t in T]
    ctx_v = [rng.standard_normal((t, Hkv, dh)).astype(np.float16) for t in T]
    u = rng.standard_normal((Hkv, dh))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    if ramp > 0:
        # keys grow along u with their position, so a query row's scores
        # climb by 4 ramp / sqrt(dh) nats a position (with the +4 u added to q below)
        for s in range(S):
            ctx_k[s] += ramp * np.arange(T[s])[:, None, None] * u[None]
    ctx_k = [k.astype(np.float16) for k in ctx_k]
    pt = np.full((NB, mpps), -1, np.int32)
    for s in range(S):
        n = -(-int(T[s]) // 16)
        # sequence 1: its pages in scattered order (within its own range, so no page is shared)
        pages = s * mpps + (rng.permutation(mpps)[:n] if s == 1 else np.arange(n))
        pt[s, :n] = pages
        for pos in range(int(T[s])):
            Kp[layer, int(pages[pos // 16]), :, pos % 16, :] = torch.from_numpy(ctx_k[s][pos]).cuda()
            Vp[layer, int(pages[pos // 16]), :, pos % 16, :] = torch.from_numpy(ctx_v[s][pos]).cuda()
    dr.page_table.copy_(torch.from_numpy(pt).cuda())
    sl = np.zeros(NB, np.int32)
    sl[:S] = T
    dr.seq_len.copy_(torch.from_numpy(sl).cuda())
    seq = rng.integers(0, S, size=NB).astype(np.int32)
    ctx_len = np.array([rng.integers(0, T[s] + 1) for s in seq], np.int32)
    edge = [0, 15, 16, 17]
    for j, c in enumerate(edge):
        seq[j] = 2
        ctx_len[j] = min(c, int(T[2]))
    seq[4], ctx_len[4] = 0, T[0]                 # the whole one-page context
    seq[5], ctx_len[5] = 3, T[3]                 # a whole multi-page context
    q = rng.standard_normal((NB, 16, Hq, dh)) * 2.0
    if ramp > 0:
        q += 4.0 * np.repeat(u, Hq // Hkv, axis=0)[None, None]
    q = q.astype(np.float16)
    kb = rng.standard_normal((NB, 16, Hkv, dh)).astype(np.float16)
    vb = rng.standard_normal((NB, 16, Hkv, dh)).astype(np.float16)
    torch.cuda.synchronize()
    return dr, layer, ctx_k, ctx_v, seq, ctx_len, q, kb, vb, T


# 40 blocks x 2 kv heads: fewer problems than SMs, the 8-page key blocks;
# 80 blocks: more problems than SMs (152 on a GB300), the 4-page key blocks
@pytest.mark.parametrize("NB", [40, 80])
@pytest.mark.parametrize("name", ["mini_a", "mini_b"])
def test_block_attention_matches_oracle(name, NB):
    import torch
    dr, layer, ctx_k, ctx_v, seq, ctx_len, q, kb, vb, T = _setup(name, S=5, NB=NB, seed=31)
    c = lambda a: torch.from_numpy(a).cuda()
    out = dr.block_attention(layer, c(seq), c(ctx_len), c(q), c(kb), c(vb))
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    ref = O.block_attention_train(q, kb, vb, ctx_k, ctx_v, seq, ctx_len)
    err = np.abs(out.cpu().numpy().astype(np.float64) - ref)
    assert err.max() < TOL, (err.max(), np.unravel_index(err.argmax(), err.shape))


# scores that climb about 6 nats a page: the running max passes the one P is
# taken against, by far, at most key blocks, so the O accumulator is
# rescaled over and over (in the 128-row variant, in TMEM)
@pytest.mark.parametrize("name", ["mini_a", "mini_b"])
def test_block_attention_with_a_climbing_max(name):
    import torch
    dr, layer, ctx_k, ctx_v, seq, ctx_len, q, kb, vb, T = _setup(name, S=5, NB=80, seed=33, ramp=0.75)
    c = lambda a: torch.from_numpy(a).cuda()
    out = dr.block_attention(layer, c(seq), c(ctx_len), c(q), c(kb), c(vb))
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    ref = O.block_attention_train(q, kb, vb, ctx_k, ctx_v, seq, ctx_len)
    err = np.abs(out.cpu().numpy().astype(np.float64) - ref)
    assert err.max() < TOL, (err.max(), np.unravel_index(err.argmax(), err.shape))


def test_block_attention_out_of_range_prefix_is_flagged_and_clamped():
    import torch
    from block_diffusion_speculative_hidden_gb300 import _lib
    dr, layer, ctx_k, ctx_v, seq, ctx_len, q, kb, vb, T = _setup("mini_a", S=4, NB=8, seed=32)
    ctx_len[3] = T[seq[3]] + 5                  # past the end of its sequence
    c = lambda a: torch.from_numpy(a).cuda()
    out = dr.block_attention(layer, c(seq), c(ctx_len), c(q), c(kb), c(vb))
    torch.cuda.synchronize()
    assert dr.device_status() & _lib.DEV_BAD_BLOCK
    ctx_len[3] = T[seq[3]]
    ref = O.block_attention_train(q, kb, vb, ctx_k, ctx_v, seq, ctx_len)
    assert np.abs(out.cpu().numpy().astype(np.float64) - ref).max() < TOL

"""Acceptance kernels vs the oracle on identical inputs.

Greedy: bit-exact tau and emitted tokens.  Stochastic: the same Philox
uniforms on both sides; exact except where a decision sits within 1e-5 of
its threshold (u vs p/q, or the top two race keys), which fp32 (GPU) and
fp64 (oracle) may decide differently."""
import numpy as np
import pytest

import synth
from harness import stochastic_exempt
from oracle import dflash_oracle as O

pytestmark = pytest.mark.gpu

CFG = synth.MINI_CONFIGS["mini_b"]


@pytest.fixture(scope="module")
def drafter():
    import torch
    from block_diffusion_speculative_hidden_gb300 import Drafter, weights_to_device
    cfg = CFG.replace(batch=64)
    w = synth.make_weights(cfg)
    dr = Drafter(cfg, weights_to_device(w, cfg.dtype), max_batch=256, max_pages_per_seq=4, n_pages=16)
    yield dr
    dr.close()


def test_greedy_accept_bit_exact(drafter):
    import torch
    B, K = 256, 16
    rng = np.random.default_rng(1)
    y = rng.integers(0, 3000, size=(B, K + 1)).astype(np.int32)
    d = y[:, :K].copy()
    for b in range(B):
        if b % 5 == 0:
            continue                      # full match: tau = K, bonus emitted
        i = b % K
        d[b, i] = (d[b, i] + 1) % 3000    # first mismatch at i
        d[b, i + 1:] = rng.integers(0, 3000, size=K - i - 1)
    tau, em, n = drafter.accept(0, torch.from_numpy(d).cuda(), target_tokens=torch.from_numpy(y).cuda())
    t_o, e_o, n_o = O.accept_greedy(d, y)
    np.testing.assert_array_equal(tau.cpu().numpy(), t_o)
    np.testing.assert_array_equal(em.cpu().numpy(), e_o)
    np.testing.assert_array_equal(n.cpu().numpy(), n_o)


@pytest.mark.parametrize("full_q,temp,boost", [(False, 1.0, 9.0), (False, 0.7, 7.0), (True, 1.0, 3.0),
                                                (False, 1.0, 0.0)])
def test_stochastic_accept_matches_oracle(drafter, full_q, temp, boost):
    import torch
    B, K, V = 64, 16, CFG.vocab
    cfg = CFG
    d = synth.make_draft_tokens(cfg, 11, B, K, V)
    z = synth.make_target_logits(cfg, 12, d, V, noise_std=1.0, boost=boost)
    q = synth.make_draft_probs(cfg, 13, B, K, V) if full_q else None
    if full_q:   # sampled drafts: make each draft token likely under q
        q[np.arange(B)[:, None], np.arange(K)[None, :], d] += 0.5
        q /= q.sum(-1, keepdims=True)
        q = q.astype(np.float32)
    seed, rnd = 0x1234_5678_9ABC, 7
    tau, em, n = drafter.accept(1, torch.from_numpy(d).cuda(), target_logits=torch.from_numpy(z).cuda(),
                                draft_probs=None if q is None else torch.from_numpy(q).cuda(),
                                temperature=temp, seed=seed, round=rnd)
    tau, em, n = tau.cpu().numpy(), em.cpu().numpy(), n.cpu().numpy()
    t_o, e_o, n_o = O.accept_stochastic(z, d, q, temp, seed, rnd)
    np.testing.assert_array_equal(n, tau + 1)
    mism = [b for b in range(B) if tau[b] != t_o[b] or not np.array_equal(em[b], e_o[b])]
    for b in mism:
        assert stochastic_exempt(z, d, temp, seed, rnd, b, int(min(tau[b], t_o[b])), q), (b, tau[b], t_o[b])
    assert len(mism) <= 2
    if boost >= 9:
        assert t_o.mean() > 1.0          # the case exercises long accepts


@pytest.mark.slow
@pytest.mark.parametrize("boost", [0.0, 16.0])
def test_stochastic_accept_full_vocab_c5_shape(boost):
    """The gpt-oss-120b-shaped workload's accept: 128 sequences, vocab
    201088, temperature 1, point-mass q (argmax drafts).  Target logits are
    draft-like logits (std 1.07, the random-init drafter's) plus N(0, 1)
    noise: almost every sequence rejects at position 0 (the workload's own
    path); boosted at the drafts, long accepts and bonus draws occur.  Exact
    against the oracle outside the near-threshold exemption."""
    import torch
    from block_diffusion_speculative_hidden_gb300 import Drafter, weights_to_device
    cfg = synth.CONFIGS["c5"]
    B, K, V = cfg.batch, 16, cfg.vocab
    small = cfg.replace(n_layers=1, hidden=64, n_q_heads=8, n_kv_heads=8, head_dim=64, ffn=64, n_taps=1,
                        tap_width=64, vocab=V)
    dr = Drafter(small, weights_to_device({k: v for k, v in synth.make_weights(small).items()}, "bf16"),
                 max_batch=B, max_pages_per_seq=2, n_pages=8)
    d = synth.make_draft_tokens(cfg, 21, B, K, V)
    z = synth.make_target_logits(cfg, 22, d, V, noise_std=1.0, boost=boost)
    z += 1.07 * synth.make_target_logits(cfg, 23, d, V, noise_std=1.0)
    seed, rnd = cfg.seed, 3
    tau, em, n = dr.accept(1, torch.from_numpy(d).cuda(), target_logits=torch.from_numpy(z).cuda(),
                           temperature=cfg.temperature, seed=seed, round=rnd)
    tau, em, n = tau.cpu().numpy(), em.cpu().numpy(), n.cpu().numpy()
    assert dr.device_status() == 0
    dr.close()
    t_o, e_o, n_o = O.accept_stochastic(z, d, None, cfg.temperature, seed, rnd)
    np.testing.assert_array_equal(n, tau + 1)
    mism = [b for b in range(B) if tau[b] != t_o[b] or not np.array_equal(em[b], e_o[b])]
    for b in mism:
        assert stochastic_exempt(z, d, cfg.temperature, seed, rnd, b, int(min(tau[b], t_o[b]))), (b, tau[b], t_o[b])
    assert len(mism) <= 2
    if boost:
        assert t_o.mean() > 3.0 and (t_o == K).any()       # long accepts and the bonus draw
    else:
        assert (t_o == 0).mean() > 0.9                      # the workload's early-reject path

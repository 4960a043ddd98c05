"""Acceptance kernels vs the oracle on identical inputs.

Greedy: bit-exact tau and emitted tokens.  Stochastic: the same Philox
uniforms on both sides; exact except where a decision sits within 1e-5 of
its threshold (u vs p/q, or the top two race keys), which fp32 (GPU) and
fp64 (oracle) may decide differently."""
import numpy as np
import pytest

import synth
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


def _exempt(z, d, q, temp, seed, rnd, b, i_stop):
    """True if the oracle's decision at position i_stop is within 1e-5 of a threshold."""
    K = d.shape[1]
    for i in range(min(i_stop, K - 1) + 1):
        p = O.softmax(z[b, i] / temp)
        if i < K:
            qd = 1.0 if q is None else float(q[b, i, d[b, i]])
            ratio = min(1.0, p[d[b, i]] / qd) if qd > 0 else 1.0
            u = float(O.rng_uniform(seed, rnd, b, i, 0, 0))
            if abs(u - ratio) < 1e-5:
                return True
    i = min(i_stop, K)
    p = O.softmax(z[b, i] / temp)
    if i < K:
        qq = np.zeros_like(p) if q is None else q[b, i].astype(np.float64)
        if q is None:
            qq[d[b, i]] = 1.0
        r = np.maximum(0.0, p - qq)
    else:
        r = p
    e = -np.log(O.rng_uniform(seed, rnd, b, i, 1, np.arange(p.shape[0])))
    key = np.sort(np.where(r > 0, r / e, 0.0))
    return (key[-1] - key[-2]) < 1e-5 * key[-1]


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
        assert _exempt(z, d, q, temp, seed, rnd, b, int(min(tau[b], t_o[b]))), (b, tau[b], t_o[b])
    assert len(mism) <= 2
    if boost >= 9:
        assert t_o.mean() > 1.0          # the case exercises long accepts

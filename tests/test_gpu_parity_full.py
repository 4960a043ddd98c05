"""GPU vs oracle at the full workload sizes, in the launch configuration the
benchmark times (bench.Workload: same pool, prefill chunks and per-round
inputs), on outputs the oracle can compute one by one.

- Every sequence runs on the GPU; the fp64 oracle recomputes a sample of
  them (sequences are independent: inject, draft and accept never mix
  them), and their block logits, argmax and confidences are compared with
  the stated tolerances.
- Page tables and lengths of *all* sequences are compared bit-exactly with a
  paging-only replay of the oracle's allocation rule.
- Acceptance of all sequences is compared bit-exactly with the oracle's rule
  on the GPU's drafts and the synthetic target.
"""
import numpy as np
import pytest

import synth
from harness import LOGIT_TOL, check_two_pass, compare_logits, compare_tokens, stochastic_exempt
from oracle import dflash_oracle as O

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

K = 16
# sampled sequences per workload (first, last, and one in between)
SAMPLES = {"c2": [0], "c2w8": [0], "c3": [0, 13, 31], "c4": [2], "c5": [0, 127]}


def paging_replay(cfg, lens, chunk, round_rows, mpps, n_pages):
    """The oracle's page allocation over all sequences, without K/V payload."""
    pk = O.PagedKV(1, n_pages, 1, 1, cfg.batch, mpps, cfg.page_size)
    for b in range(cfg.batch):
        for s0 in range(0, int(lens[b]), chunk):
            n = [0] * cfg.batch
            n[b] = min(chunk, int(lens[b]) - s0)
            assert pk.allocate(n)
            pk.seq_len[b] += n[b]
    for rows in round_rows:
        assert pk.allocate([int(x) for x in rows])
        pk.seq_len += np.asarray(rows, dtype=pk.seq_len.dtype)
    return pk


@pytest.mark.parametrize("name", ["c2", "c2w8", "c3", "c4", "c5"])
def test_full_size_sampled_parity(name):
    import torch
    import bench
    cfg = synth.CONFIGS[name]
    B, V = cfg.batch, cfg.vocab
    dev = torch.device("cuda", 0)
    wl = bench.Workload(cfg, 2, 0, dev, reset_every=16)
    dr = wl.dr
    chunk = min(1024, int(wl.lens.max()))
    seqs = SAMPLES[name]

    # oracle over the sampled sequences only (pool sized for them)
    pages = sum(-(-(int(wl.lens[b]) + 17 * 4) // 16) + 1 for b in seqs) + 4
    orc = O.OracleDrafter(cfg, wl.w_np, pages, wl.mpps, key_offsets=synth.make_key_offsets(cfg), seqs=seqs)
    for j, b in enumerate(seqs):
        feats = synth.make_prefill_features(cfg, b, int(wl.lens[b]))
        step = 4096
        for s0 in range(0, feats.shape[0], step):
            rows = [np.zeros((0, cfg.feat_dim), np.float32)] * len(seqs)
            rows[j] = feats[s0:s0 + step]
            assert orc.inject(rows)

    round_rows = []
    pass2_compared = 0
    n_rows = np.ones(B, np.int32)          # the bench's first round injects one row per sequence
    for rnd in range(2):
        feats_r = wl.h_feats[rnd]          # [B, 17, F] resident round inputs
        dr.inject_kv(wl.feats[rnd], torch.from_numpy(n_rows).to(dev))
        round_rows.append(n_rows.copy())
        assert orc.inject([feats_r[b, :n_rows[b]] for b in seqs])
        logits = torch.empty((B, K, V), dtype=torch.float32, device=dev)
        committed = torch.empty((B, K), dtype=torch.int32, device=dev)
        tok, conf, _, _ = dr.draft_block(B, cfg.s_passes, logits=logits, committed=committed)
        torch.cuda.synchronize()
        tok_h, conf_h = tok.cpu().numpy(), conf.cpu().numpy()
        com = committed.cpu().numpy().astype(bool)
        for j, b in enumerate(seqs):
            zg = logits[b].cpu().numpy()
            r = orc.draft(j)
            if cfg.s_passes == 1:
                compare_logits(zg, r["logits"], cfg.dtype)
                compare_tokens(tok_h[b], r["logits"])
                lc = np.log(np.maximum(conf_h[b], 1e-38))
                assert np.max(np.abs(lc - np.log(r["conf"]))) < 2 * LOGIT_TOL[cfg.dtype] + 1e-6
            else:
                # S = 2: both passes of every sampled sequence (harness.check_two_pass)
                pass2_compared += check_two_pass(orc, j, r, tok_h[b], com[b], zg, cfg)
        # acceptance of every sequence against the oracle's rule, on the
        # drafts: greedy bit-exact; stochastic (the gpt-oss-shaped workload,
        # temperature 1, point-mass q) against synthetic target logits,
        # exact outside the near-threshold exemption
        if cfg.accept == "greedy":
            y = synth.make_target_tokens(cfg, rnd, tok_h).astype(np.int32)
            tau, em, n = dr.accept(0, tok, target_tokens=torch.from_numpy(y).to(dev))
            t_o, e_o, n_o = O.accept_greedy(tok_h, y)
            np.testing.assert_array_equal(tau.cpu().numpy(), t_o)
            np.testing.assert_array_equal(em.cpu().numpy(), e_o)
        else:
            zt = synth.make_target_logits(cfg, 100 + rnd, tok_h, V, noise_std=1.0)
            tau, em, n = dr.accept(1, tok, target_logits=torch.from_numpy(zt).to(dev), temperature=cfg.temperature,
                                   seed=cfg.seed, round=rnd)
            t_o, e_o, n_o = O.accept_stochastic(zt, tok_h, None, cfg.temperature, cfg.seed, rnd)
            tg, eg = tau.cpu().numpy(), em.cpu().numpy()
            mism = [b for b in range(B) if tg[b] != t_o[b] or not np.array_equal(eg[b], e_o[b])]
            for b in mism:
                assert stochastic_exempt(zt, tok_h, cfg.temperature, cfg.seed, rnd, b, int(min(tg[b], t_o[b])))
            assert len(mism) <= 2
            n_o = np.where([b in mism for b in range(B)], tg + 1, n_o)   # the chain follows the GPU there
        np.testing.assert_array_equal(n.cpu().numpy(), n_o)
        n_rows = n_o.astype(np.int32)

    if cfg.s_passes == 2:
        assert pass2_compared == 2 * len(seqs)      # every sampled sequence, both rounds
    # paging of every sequence, bit-exact
    pk = paging_replay(cfg, wl.lens, chunk, round_rows, wl.mpps, B * wl.mpps + 8)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(dr.seq_len.cpu().numpy(), pk.seq_len)
    np.testing.assert_array_equal(dr.page_table.cpu().numpy(), pk.page_table)
    assert dr.device_status() == 0

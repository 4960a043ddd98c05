"""GPU vs oracle on workloads the oracle finishes in seconds: prefill, then
rounds of inject(tau+1 rows) -> draft -> accept, checking page tables and
lengths bit-exact, KV pages, logits and confidences within tolerance, argmax
agreement (near ties exempt), S = 2 commits, and tau / emitted bit-exact
given identical drafts."""
import numpy as np
import pytest

import synth
from oracle import dflash_oracle as O
from harness import Pair

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["c1", "mini_f32", "mini_a", "mini_b", "mini_c", "mini_d", "mini_w8", "mini_w8b"])
def test_chain_parity(name):
    import torch
    cfg = synth.get_config(name)
    if name in ("mini_b", "mini_w8b"):
        cfg = cfg.replace(weight_std=0.06)   # peaked confidences: a well-separated S = 2 commit order
    rounds = 3
    pair = Pair(cfg, rounds)
    pair.prefill()
    pair.check_cache()
    S = cfg.s_passes
    for rnd in range(rounds):
        res, tok_gpu = pair.draft_and_check(S)
        # the chain follows the oracle's drafts; both sides accept the same drafts
        d = np.stack([res[b]["tokens"] for b in range(cfg.batch)]).astype(np.int32)
        if cfg.accept == "greedy":
            y = synth.make_target_tokens(cfg, rnd, d)
            tau, em, n = pair.gpu.accept(0, torch.from_numpy(d).cuda(), target_tokens=torch.from_numpy(y).cuda())
            t_o, e_o, n_o = O.accept_greedy(d, y)
            np.testing.assert_array_equal(tau.cpu().numpy(), t_o)
            np.testing.assert_array_equal(em.cpu().numpy(), e_o)
        else:
            z = np.stack([res[b]["logits"] for b in range(cfg.batch)]).astype(np.float32)
            zt = np.concatenate([z * 4.0, np.zeros((cfg.batch, 1, cfg.vocab), np.float32)], 1)
            zt += synth.make_target_logits(cfg, 100 + rnd, d, cfg.vocab, noise_std=1.0)
            tau, em, n = pair.gpu.accept(1, torch.from_numpy(d).cuda(), target_logits=torch.from_numpy(zt).cuda(),
                                         temperature=cfg.temperature, seed=cfg.seed, round=rnd)
            t_o, e_o, n_o = O.accept_stochastic(zt, d, None, cfg.temperature, cfg.seed, rnd)
            np.testing.assert_array_equal(tau.cpu().numpy(), t_o)
            np.testing.assert_array_equal(em.cpu().numpy(), e_o)
        pair.inject_round(rnd, n_o.astype(np.int32))
        pair.check_cache()


def test_incremental_inject_equals_one_prefill():
    """Injecting a prompt in pieces writes the same bf16 K/V as one call."""
    import torch
    cfg = synth.MINI_CONFIGS["mini_a"]
    a = Pair(cfg, 2)
    a.prefill()
    b = Pair(cfg, 2, max_rows_prefill=37)     # the same prompts, 37-row chunks
    b.prefill()
    torch.cuda.synchronize()
    sl = a.gpu.seq_len.cpu().numpy()
    Ka, Va = a.gpu.pool_kv()
    Kb, Vb = b.gpu.pool_kv()
    pta, ptb = a.gpu.page_table.cpu().numpy(), b.gpu.page_table.cpu().numpy()
    for s in range(cfg.batch):
        pos = np.arange(sl[s])
        ia = torch.from_numpy(pta[s, pos // 16]).long().cuda()
        ib = torch.from_numpy(ptb[s, pos // 16]).long().cuda()
        sl_ = torch.from_numpy(pos % 16).long().cuda()
        assert torch.equal(Ka[:, ia, :, sl_, :], Kb[:, ib, :, sl_, :])
        assert torch.equal(Va[:, ia, :, sl_, :], Vb[:, ib, :, sl_, :])


def test_pool_exhaustion_changes_nothing():
    import torch
    from block_diffusion_speculative_hidden_gb300 import Drafter, weights_to_device
    cfg = synth.MINI_CONFIGS["mini_f32"]
    w = synth.make_weights(cfg)
    dr = Drafter(cfg, weights_to_device(w, cfg.dtype), max_batch=2, max_pages_per_seq=8, n_pages=5, max_rows=40,
                 max_inject_rows=80)
    F = cfg.feat_dim
    feats = torch.zeros((2, 40, F), device="cuda")
    dr.inject_kv(feats, torch.tensor([40, 20], dtype=torch.int32, device="cuda"))   # 3 + 2 pages: fits
    assert dr.device_status() == 0
    pt0 = dr.page_table.clone()
    dr.inject_kv(feats, torch.tensor([10, 0], dtype=torch.int32, device="cuda"))    # needs 1 more: none left
    assert dr.device_status() == 1
    assert torch.equal(dr.page_table, pt0)
    assert dr.seq_len.tolist() == [40, 20]
    dr.release(1)
    dr.reset()
    assert dr.device_status() == 0 and dr.seq_len.tolist() == [0, 0]
    dr.close()


@pytest.mark.parametrize("name", ["mini_b", "mini_w8b"])
def test_second_pass_lm_head_on_uncommitted_rows_only(name):
    """S = 2: the second pass runs the LM head on the K/2 uncommitted rows
    only (compacted), and a logits store puts each of them back at its block
    row; asking for the logits changes neither the drafts nor the
    confidences, bit for bit, and the stored logits of the uncommitted rows
    are the ones checked against the oracle above."""
    import torch
    cfg = synth.get_config(name).replace(weight_std=0.06)
    pair = Pair(cfg, 2)
    pair.prefill()
    dr = pair.gpu
    B = cfg.batch
    logits = torch.empty((B, 16, cfg.vocab), dtype=torch.float32, device="cuda")
    com = torch.empty((B, 16), dtype=torch.int32, device="cuda")
    tok_full, conf_full, _, _ = dr.draft_block(B, 2, logits=logits, committed=com)
    tok_c, conf_c, _, _ = dr.draft_block(B, 2)
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    assert torch.equal(tok_full, tok_c)
    assert torch.equal(conf_full, conf_c)

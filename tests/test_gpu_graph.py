"""Host-free rounds: a whole round recorded once as a CUDA graph
(dflash_graph_begin / _end) and replayed with dflash_graph_launch.

The round is: inject the previous round's tau+1 feature rows (n_rows = the
previous accept's n_emit, never read by the host), draft, the synthetic
target's verify as device work of the caller's own (torch ops on the same
stream), accept, and n_emit copied into next round's n_rows.  Round 0 runs
eagerly (it sets up the shapes' host state), later rounds are replays of one
recording.  Every round is checked against the oracle as in the eager chain
test: logits, confidences, argmax and S = 2 commits within tolerance; tau,
emitted tokens and the page tables bit-exact.  Stochastic rounds draw the
uniforms of round r through the device round counter (DFLASH_ROUND_DEVICE),
so a replay draws fresh ones."""
import numpy as np
import pytest

import synth
from harness import Pair
from oracle import dflash_oracle as O

pytestmark = pytest.mark.gpu

K = 16


@pytest.mark.parametrize("name", ["mini_a", "mini_b"])
def test_replayed_rounds_match_the_oracle(name):
    import torch
    from block_diffusion_speculative_hidden_gb300 import ROUND_DEVICE, DflashError
    cfg = synth.get_config(name)
    if name == "mini_b":
        cfg = cfg.replace(weight_std=0.06)   # peaked confidences: a well-separated S = 2 commit order
    rounds = 4
    pair = Pair(cfg, rounds + 1)
    pair.prefill()
    torch.cuda.synchronize()
    dr = pair.gpu
    B, V, F, S = cfg.batch, cfg.vocab, cfg.feat_dim, cfg.s_passes
    greedy = cfg.accept == "greedy"
    stream = torch.cuda.Stream()
    dev = torch.device("cuda")
    # fixed buffers the recorded round reads and writes
    feats = torch.zeros((B, 17, F), dtype=dr.tdtype, device=dev)
    n_rows = torch.zeros(B, dtype=torch.int32, device=dev)          # nothing new before the first draft
    tok = torch.empty((B, K), dtype=torch.int32, device=dev)
    conf = torch.empty((B, K), dtype=torch.float32, device=dev)
    logits = torch.empty((B, K, V), dtype=torch.float32, device=dev)
    com = torch.empty((B, K), dtype=torch.int32, device=dev)
    match = torch.zeros((B, K + 1), dtype=torch.bool, device=dev)
    rand = torch.zeros((B, K + 1), dtype=torch.int32, device=dev)
    y = torch.zeros((B, K + 1), dtype=torch.int32, device=dev)
    noise = torch.zeros((B, K + 1, V), dtype=torch.float32, device=dev)
    zt = torch.zeros((B, K + 1, V), dtype=torch.float32, device=dev)
    out = (torch.empty(B, dtype=torch.int32, device=dev), torch.empty((B, K + 1), dtype=torch.int32, device=dev),
           torch.empty(B, dtype=torch.int32, device=dev))

    def round_body():
        dr.inject_kv(feats, n_rows, stream=stream)
        dr.draft_block(B, S, tokens=tok, conf=conf, logits=logits, committed=com, stream=stream)
        with torch.cuda.stream(stream):
            if greedy:
                torch.where(match[:, :K], tok, rand[:, :K], out=y[:, :K])
                y[:, K].copy_(rand[:, K])
                dr.accept(0, tok, target_tokens=y, out=out, stream=stream)
            else:
                torch.mul(logits, 4.0, out=zt[:, :K])
                zt[:, K].zero_()
                zt.add_(noise)
                dr.accept(1, tok, target_logits=zt, temperature=cfg.temperature, seed=cfg.seed,
                          round=ROUND_DEVICE, out=out, stream=stream)
            n_rows.copy_(out[2])

    graph = None
    n_prev = np.zeros(B, np.int64)
    for r in range(rounds):
        fr = np.stack([synth.make_round_features(cfg, r, b, 17) for b in range(B)])
        match_h, rand_h = synth.make_target_match(cfg, r, B, K)
        noise_h = synth.make_target_logits(cfg, 100 + r, np.zeros((B, K), np.int32), V, noise_std=1.0)
        with torch.cuda.stream(stream):
            feats.copy_(torch.from_numpy(fr).to(dev).to(dr.tdtype))
            match.copy_(torch.from_numpy(match_h).to(dev))
            rand.copy_(torch.from_numpy(rand_h).to(dev))
            noise.copy_(torch.from_numpy(noise_h).to(dev))
        if r == 0:
            round_body()
        else:
            if graph is None:
                dr.graph_begin(stream=stream)
                with pytest.raises(DflashError) as e:
                    dr.device_status(stream=stream)      # a synchronising call is refused while recording
                assert e.value.code == 8
                round_body()
                graph = dr.graph_end(stream=stream)
            graph.launch(stream=stream)
        stream.synchronize()

        # the oracle takes the same round: the rows of the previous round's accepted tokens, then a draft
        assert pair.orc.inject([fr[b, :n_prev[b]] for b in range(B)])
        tok_h, conf_h = tok.cpu().numpy(), conf.cpu().numpy()
        com_h, zg = com.cpu().numpy().astype(bool), logits.cpu().numpy()
        pair.check_outputs(S, tok_h, conf_h, com_h, zg)
        if greedy:
            y_o = rand_h.copy()
            y_o[:, :K] = np.where(match_h[:, :K], tok_h, rand_h[:, :K])
            t_o, e_o, n_o = O.accept_greedy(tok_h, y_o)
        else:
            zt_o = np.concatenate([zg * np.float32(4.0), np.zeros((B, 1, V), np.float32)], 1) + noise_h
            t_o, e_o, n_o = O.accept_stochastic(zt_o, tok_h, None, cfg.temperature, cfg.seed, r)
        np.testing.assert_array_equal(out[0].cpu().numpy(), t_o)
        np.testing.assert_array_equal(out[1].cpu().numpy(), e_o)
        np.testing.assert_array_equal(out[2].cpu().numpy(), n_o)
        np.testing.assert_array_equal(n_rows.cpu().numpy(), n_o)
        n_prev = n_o
        pair.check_cache()
    graph.close()

"""Seeded synthetic inputs for the DFlash block-draft hot path.

This module is the one piece shared by the CPU oracle and the CUDA path.  It
holds the workload shapes and the seeded random draws (weights, target
features, context lengths, synthetic target tokens and logits) and nothing of
the method's arithmetic: no projection, norm, attention, argmax or acceptance
rule lives here.

Workloads follow the method's pages:
  * DFlash Guide (aifetchly blog), "Functional Verification Harness" and
    "3. Cross-Layer KV Injection": a small drafter over random weights and
    random target hidden states;
  * the named serving shapes (Qwen3-8B-shaped and gpt-oss-120b-shaped
    drafters, K = 16 block, paged KV with 16-token pages).

Draws: every tensor has its own numpy PCG64 stream derived from
(config seed, tensor id) with ``numpy.random.SeedSequence``.  Weights are
N(0, 0.02) drawn in fp32; feature rows N(0, 1) drawn in fp32.  For bf16
workloads both are rounded to the nearest bf16 (ties to even) so that the
oracle (which upcasts to fp64) and the GPU (which stores bf16) see
identical values.  Norm gains are ones.
"""
from __future__ import annotations

import concurrent.futures as _fut
import dataclasses
import os
from typing import Dict, List, Optional

import numpy as np

__all__ = [
    "DraftConfig", "CONFIGS", "MINI_CONFIGS", "get_config",
    "round_to_bf16", "bf16_bits", "make_weights", "make_ctx_lens",
    "make_prefill_features", "make_round_features", "make_key_offsets",
    "make_target_tokens", "make_target_match", "make_target_logits", "make_draft_tokens",
    "make_draft_probs", "weight_names", "quantize_e4m3_rows", "PROJECTIONS",
]


@dataclasses.dataclass(frozen=True)
class DraftConfig:
    name: str
    batch: int
    ctx_lo: int                 # context lengths are uniform integers in [ctx_lo, ctx_hi]
    ctx_hi: int
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    n_taps: int
    tap_width: int
    s_passes: int = 1           # S refinement passes (1 or 2)
    accept: str = "greedy"      # "greedy" | "stochastic"
    match_prob: float = 0.8     # synthetic target: y_i = d_i with this probability
    temperature: float = 1.0
    dtype: str = "bf16"         # "bf16" | "f32"
    rounds: int = 8
    seed: int = 1000
    block_k: int = 16
    page_size: int = 16
    rope_theta: float = 1.0e6
    rms_eps: float = 1.0e-6
    key_offset_std: float = 0.0  # >0: shared pre-RoPE key offset on even kv heads
    weight_std: float = 0.02
    weight_format: str = "bf16"  # "bf16" | "e4m3": projection weights as FP8 codes + per-row scales

    @property
    def mask_id(self) -> int:
        return self.vocab - 1

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def feat_dim(self) -> int:
        return self.n_taps * self.tap_width

    def max_ctx(self) -> int:
        """Largest context a sequence reaches over the configured rounds."""
        return self.ctx_hi + (self.block_k + 1) * (self.rounds + 1)

    def replace(self, **kw) -> "DraftConfig":
        return dataclasses.replace(self, **kw)


# The five workloads (seed = 1000 + index).  c5 does not state the draft
# hidden size or the tap count: hidden = target hidden = 2880, 3 taps.
CONFIGS: Dict[str, DraftConfig] = {
    "c1": DraftConfig("c1_tiny_f32", batch=1, ctx_lo=64, ctx_hi=64, n_layers=1,
                      hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn=688,
                      vocab=2048, n_taps=3, tap_width=256, match_prob=0.8,
                      dtype="f32", rounds=8, seed=1001),
    "c2": DraftConfig("c2_qwen3_8b_shaped", batch=1, ctx_lo=2048, ctx_hi=2048,
                      n_layers=5, hidden=4096, n_q_heads=32, n_kv_heads=8,
                      head_dim=128, ffn=12288, vocab=151936, n_taps=5,
                      tap_width=4096, match_prob=0.85, rounds=8, seed=1002),
    # c2 with FP8 (e4m3, per-row scale) projection weights: half the weight bytes
    "c2w8": DraftConfig("c2_qwen3_8b_shaped_fp8w", batch=1, ctx_lo=2048, ctx_hi=2048,
                        n_layers=5, hidden=4096, n_q_heads=32, n_kv_heads=8,
                        head_dim=128, ffn=12288, vocab=151936, n_taps=5,
                        tap_width=4096, match_prob=0.85, rounds=8, seed=1006, weight_format="e4m3"),
    "c3": DraftConfig("c3_serving_batch32", batch=32, ctx_lo=512, ctx_hi=4096,
                      n_layers=5, hidden=4096, n_q_heads=32, n_kv_heads=8,
                      head_dim=128, ffn=12288, vocab=151936, n_taps=5,
                      tap_width=4096, match_prob=0.8, rounds=32, seed=1003),
    "c4": DraftConfig("c4_long_context_32k", batch=4, ctx_lo=32768, ctx_hi=32768,
                      n_layers=3, hidden=4096, n_q_heads=32, n_kv_heads=8,
                      head_dim=128, ffn=12288, vocab=151936, n_taps=5,
                      tap_width=4096, match_prob=0.85, rounds=64, seed=1004,
                      key_offset_std=4.0),
    "c5": DraftConfig("c5_gpt_oss_120b_shaped", batch=128, ctx_lo=1024, ctx_hi=8192,
                      n_layers=3, hidden=2880, n_q_heads=64, n_kv_heads=8,
                      head_dim=64, ffn=2880, vocab=201088, n_taps=3,
                      tap_width=2880, s_passes=2, accept="stochastic",
                      temperature=1.0, rounds=8, seed=1005),
}

# Small workloads the oracle finishes in seconds.  They keep the structure of
# the full ones but are ragged on purpose: output widths and reduction depths
# that are not multiples of the GPU tiles, uneven context lengths, partial
# last pages.
MINI_CONFIGS: Dict[str, DraftConfig] = {
    # dh = 128, G = 4, S = 1, greedy
    "mini_a": DraftConfig("mini_a", batch=3, ctx_lo=5, ctx_hi=300, n_layers=2,
                          hidden=512, n_q_heads=8, n_kv_heads=2, head_dim=128,
                          ffn=1320, vocab=5000, n_taps=3, tap_width=448,
                          match_prob=0.8, rounds=3, seed=2001),
    # dh = 64, G = 8, S = 2, stochastic
    "mini_b": DraftConfig("mini_b", batch=4, ctx_lo=1, ctx_hi=200, n_layers=2,
                          hidden=384, n_q_heads=16, n_kv_heads=2, head_dim=64,
                          ffn=776, vocab=3001, n_taps=3, tap_width=384,
                          s_passes=2, accept="stochastic", rounds=3, seed=2002),
    # dh = 64, G = 1, many sequences with long contexts: few key splits per
    # (sequence, kv head), each streaming several 8-page blocks
    "mini_c": DraftConfig("mini_c", batch=12, ctx_lo=150, ctx_hi=1400, n_layers=1,
                          hidden=512, n_q_heads=8, n_kv_heads=8, head_dim=64,
                          ffn=1024, vocab=3000, n_taps=2, tap_width=512,
                          match_prob=0.8, rounds=3, seed=2004),
    # FP8 projection weights (e4m3 + per-row scales), otherwise like mini_a
    # (FP8 rows must be a multiple of 16 bytes, so ffn = 1328: still ragged
    # against the 64-wide k-blocks)
    "mini_w8": DraftConfig("mini_w8", batch=3, ctx_lo=9, ctx_hi=260, n_layers=2,
                           hidden=512, n_q_heads=8, n_kv_heads=2, head_dim=128,
                           ffn=1328, vocab=5000, n_taps=3, tap_width=448,
                           match_prob=0.8, rounds=3, seed=2005, weight_format="e4m3"),
    # FP8 projection weights with S = 2 and stochastic acceptance (dh = 64, G = 8)
    "mini_w8b": DraftConfig("mini_w8b", batch=4, ctx_lo=1, ctx_hi=200, n_layers=2,
                            hidden=384, n_q_heads=16, n_kv_heads=2, head_dim=64,
                            ffn=784, vocab=3001, n_taps=3, tap_width=384,
                            s_passes=2, accept="stochastic", rounds=3, seed=2006, weight_format="e4m3"),
    # a serving-size batch (16 sequences = 256 block rows) with a wide FFN:
    # the gate/up projection (160 tiles of 128 x 128 on 152 SMs) runs on the
    # persistent kernel, whose 8 tiles of the last, partial round are split
    # in K 8 ways (one 64-k block a segment)
    "mini_d": DraftConfig("mini_d", batch=16, ctx_lo=3, ctx_hi=120, n_layers=1,
                          hidden=512, n_q_heads=8, n_kv_heads=2, head_dim=64,
                          ffn=5120, vocab=3000, n_taps=2, tap_width=512,
                          match_prob=0.8, rounds=3, seed=2007),
    # fp32 mini: ragged, several pages, G = 2
    "mini_f32": DraftConfig("mini_f32", batch=2, ctx_lo=17, ctx_hi=90, n_layers=2,
                            hidden=192, n_q_heads=6, n_kv_heads=3, head_dim=32,
                            ffn=440, vocab=1500, n_taps=2, tap_width=160,
                            dtype="f32", rounds=3, seed=2003),
}


def get_config(name: str) -> DraftConfig:
    if name in CONFIGS:
        return CONFIGS[name]
    if name in MINI_CONFIGS:
        return MINI_CONFIGS[name]
    raise KeyError(name)


# ---------------------------------------------------------------------------
# bf16 storage format (input quantisation, not part of the method)
# ---------------------------------------------------------------------------

def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 value (ties to even); fp32 result."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    r = (u + bias) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """The upper 16 bits of bf16-representable fp32 values, as uint16."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _rng(cfg: DraftConfig, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([cfg.seed, *key])))


def _normal(cfg: DraftConfig, shape, std: float, *key: int) -> np.ndarray:
    a = _rng(cfg, *key).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    if cfg.dtype == "bf16":
        a = round_to_bf16(a)
    return a


# ---------------------------------------------------------------------------
# weights
# ---------------------------------------------------------------------------

def weight_names(cfg: DraftConfig) -> List[str]:
    names = ["w_fc", "g_fc", "embed", "g_final", "w_lm"]
    for l in range(cfg.n_layers):
        names += [f"{n}.{l}" for n in ("w_q", "w_k", "w_v", "w_o", "w_gate", "w_up",
                                       "w_down", "g_in", "g_post")]
    return names


def _weight_shape(cfg: DraftConfig, name: str):
    base = name.split(".")[0]
    d = cfg.hidden
    return {
        "w_fc": (d, cfg.feat_dim), "g_fc": (d,), "embed": (cfg.vocab, d),
        "g_final": (d,), "w_lm": (cfg.vocab, d),
        "w_q": (cfg.q_dim, d), "w_k": (cfg.kv_dim, d), "w_v": (cfg.kv_dim, d),
        "w_o": (d, cfg.q_dim), "w_gate": (cfg.ffn, d), "w_up": (cfg.ffn, d),
        "w_down": (d, cfg.ffn), "g_in": (d,), "g_post": (d,),
    }[base]


PROJECTIONS = ("w_fc", "w_lm", "w_q", "w_k", "w_v", "w_o", "w_gate", "w_up", "w_down")


def _one_weight(cfg: DraftConfig, idx: int, name: str) -> np.ndarray:
    shape = _weight_shape(cfg, name)
    if name.split(".")[0].startswith("g_"):
        return np.ones(shape, dtype=np.float32)
    return _normal(cfg, shape, cfg.weight_std, 1, idx)


def quantize_e4m3_rows(w: np.ndarray):
    """Storage format of the FP8-weight workloads (input preparation, not
    part of the method): per output row the fp32 scale s = max|w_row| / 448
    (448 = the largest E4M3 magnitude) and the E4M3 codes of w_row / s,
    rounded to nearest even by PyTorch's float8_e4m3fn cast.  Returns
    (codes uint8 [rows, cols], scales fp32 [rows]); an all-zero row gets
    scale 1 and zero codes."""
    import torch
    amax = np.abs(w).max(axis=1)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    t = torch.from_numpy(np.ascontiguousarray(w / scale[:, None], dtype=np.float32))
    codes = t.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    return codes, scale


def _one_weight_e4m3(cfg: DraftConfig, idx: int, name: str):
    shape = _weight_shape(cfg, name)
    w = _rng(cfg, 1, idx).standard_normal(size=shape, dtype=np.float32) * np.float32(cfg.weight_std)
    return quantize_e4m3_rows(w)


def make_weights(cfg: DraftConfig, threads: Optional[int] = None) -> Dict[str, np.ndarray]:
    """All drafter weights as fp32 arrays (bf16-exact values for bf16 workloads).

    Layout: every matrix is [out_features, in_features], row-major.
    Keys: w_fc, g_fc, embed, g_final, w_lm and per layer l: w_q.l, w_k.l, w_v.l,
    w_o.l, w_gate.l, w_up.l, w_down.l, g_in.l, g_post.l.  With
    weight_format "e4m3" every projection <name> (w_fc, w_lm and the per-layer
    w_q ... w_down) comes instead as "q:<name>" (E4M3 codes, uint8) and
    "s:<name>" (fp32 per-row scales) from the same N(0, std) draw
    (quantize_e4m3_rows); the embedding and the gains stay as they are.
    """
    names = weight_names(cfg)
    threads = threads or min(16, os.cpu_count() or 1)
    out: Dict[str, np.ndarray] = {}
    fp8 = cfg.weight_format == "e4m3"
    with _fut.ThreadPoolExecutor(max_workers=threads) as ex:
        futs = {}
        for i, n in enumerate(names):
            if fp8 and n.split(".")[0] in PROJECTIONS:
                futs[ex.submit(_one_weight_e4m3, cfg, i, n)] = n
            else:
                futs[ex.submit(_one_weight, cfg, i, n)] = n
        for f in futs:
            n = futs[f]
            if fp8 and n.split(".")[0] in PROJECTIONS:
                out["q:" + n], out["s:" + n] = f.result()
            else:
                out[n] = f.result()
    return out


def make_key_offsets(cfg: DraftConfig) -> Optional[np.ndarray]:
    """Shared pre-RoPE key offsets [L, Hkv, dh] (fp32), or None.

    The long-context workload peaks attention by giving every even kv head
    (the kv heads of q heads 0, 8, 16, 24 at G = 4) one seeded offset vector
    c ~ N(0, std^2) added to the injected keys at every context position.
    """
    if cfg.key_offset_std <= 0:
        return None
    c = _rng(cfg, 5).standard_normal(size=(cfg.n_layers, cfg.n_kv_heads, cfg.head_dim),
                                     dtype=np.float32) * np.float32(cfg.key_offset_std)
    c[:, 1::2, :] = 0.0
    if cfg.dtype == "bf16":
        c = round_to_bf16(c)
    return c


# ---------------------------------------------------------------------------
# context lengths and feature rows
# ---------------------------------------------------------------------------

def make_ctx_lens(cfg: DraftConfig) -> np.ndarray:
    if cfg.ctx_lo == cfg.ctx_hi:
        return np.full(cfg.batch, cfg.ctx_lo, dtype=np.int64)
    return _rng(cfg, 2).integers(cfg.ctx_lo, cfg.ctx_hi + 1, size=cfg.batch).astype(np.int64)


def make_prefill_features(cfg: DraftConfig, b: int, n_rows: int) -> np.ndarray:
    """Tapped target hidden states of sequence b's prompt: [n_rows, n_taps*tap_width].

    Taps are concatenated along the feature axis in ascending tapped-layer
    order; each element N(0, 1).
    """
    return _normal(cfg, (n_rows, cfg.feat_dim), 1.0, 3, b)


def make_round_features(cfg: DraftConfig, rnd: int, b: int, n_rows: int) -> np.ndarray:
    """Feature rows for the tau+1 tokens accepted in round ``rnd``."""
    return _normal(cfg, (n_rows, cfg.feat_dim), 1.0, 4, rnd, b)


# ---------------------------------------------------------------------------
# synthetic target side (stands in for the target model's verify pass)
# ---------------------------------------------------------------------------

def make_target_match(cfg: DraftConfig, rnd: int, B: int, K: int):
    """Coins of the synthetic target for round ``rnd``: (match [B, K+1] bool,
    rand_tok [B, K+1] int32).  Position K (the bonus position) never matches."""
    g = _rng(cfg, 6, rnd)
    match = g.random(size=(B, K + 1)) < cfg.match_prob
    match[:, K] = False
    rand_tok = g.integers(0, cfg.vocab, size=(B, K + 1)).astype(np.int32)
    return match, rand_tok


def make_target_tokens(cfg: DraftConfig, rnd: int, drafts: np.ndarray) -> np.ndarray:
    """Synthetic target greedy tokens y [B, K+1]: y_i = d_i with prob match_prob,
    else a uniform token; y_K (the bonus position, no draft) is uniform."""
    B, K = drafts.shape
    match, rand_tok = make_target_match(cfg, rnd, B, K)
    y = rand_tok.copy()
    y[:, :K] = np.where(match[:, :K], drafts, rand_tok[:, :K])
    return y.astype(np.int32)


def make_draft_tokens(cfg: DraftConfig, key: int, B: int, K: int, vocab: int) -> np.ndarray:
    return _rng(cfg, 7, key).integers(0, vocab, size=(B, K)).astype(np.int32)


def make_target_logits(cfg: DraftConfig, key: int, drafts: np.ndarray, vocab: int,
                       noise_std: float = 1.0, boost: float = 0.0) -> np.ndarray:
    """Synthetic target logits [B, K+1, V] fp32: N(0, noise_std^2), plus ``boost``
    added at each position's draft token (raises p(d_i) so that longer accepts
    occur)."""
    B, K = drafts.shape
    z = _rng(cfg, 8, key).standard_normal(size=(B, K + 1, vocab), dtype=np.float32)
    z *= np.float32(noise_std)
    if boost:
        bi = np.arange(B)[:, None]
        ki = np.arange(K)[None, :]
        z[bi, ki, drafts] += np.float32(boost)
    return z


def make_draft_probs(cfg: DraftConfig, key: int, B: int, K: int, vocab: int,
                     conc: float = 1.0) -> np.ndarray:
    """Random draft distributions q [B, K, V] fp32 (Dirichlet(conc)), rows sum to 1."""
    g = _rng(cfg, 9, key)
    q = g.gamma(conc, size=(B, K, vocab)).astype(np.float64)
    q /= q.sum(axis=-1, keepdims=True)
    return q.astype(np.float32)

"""CPU oracle for the DFlash block-draft hot path.  TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module.  The CUDA library never uses it and shares no
code with it; the two meet only through the seeded inputs of ``synth``.

Plain, slow, obviously correct: NumPy in fp64 throughout.  Inputs arrive as
the exact values the GPU receives (bf16-exact fp32 or fp32) and are upcast to
fp64; no intermediate is rounded.  Each function cites the passage it
follows.  The pages:

  P1  "DFlash Guide: Block Diffusion for Speculative Decoding" (aifetchly blog)
  P2  "DFlash: Block Diffusion for Flash Speculative Decoding" (arXiv 2602.06036
      abstract page on sciencestack: TL;DR, abstract, figure captions)
  P3  "DFlash: Diffusion Drafts the Block" (stable-lab "Parallel drafting" chapter)

Readings taken where the pages are silent (each repeated at its function):
  R1  fusion = concatenate taps -> one linear FC -> RMSNorm (eps 1e-6, gain ones)
  R2  one fused feature h feeds the K/V projections of every draft layer
  R3  no norm, bias or q/k-norm on the injected path or anywhere else
  R4  RoPE everywhere, rotate-half (NeoX) over the full head dim, theta 1e6;
      context keys rotated at their absolute position, block q/k at T_b + i
  R5  the block is K [MASK] embeddings; nothing else enters it
  R6  untied embedding and LM head, final RMSNorm before the head
  R7  block attention is unmasked: all context and all K block positions,
      scale 1/sqrt(dh), query head h uses kv head floor(h / G)
  R8  argmax ties go to the lowest vocab index
  R9  S = 2: commit the K/2 most confident positions (confidence = max softmax
      probability, ties to the lower position), re-run with their tokens
      embedded, take the other K/2 tokens from pass 2
  R10 greedy target y has K+1 entries so that tau = K emits the bonus y_K
  R11 stochastic accept with argmax drafts uses the point-mass q = delta(d_i)
  R12 randomness: Philox4x32-10, key = seed, counter = (v >> 2, i | stream<<16,
      b, round), the uniform of index v taken from output word v & 3 (four
      consecutive indices share one counter)
  R13 residual / bonus sampling by an exponential race, ties to lowest v
  R14 page allocation: FIFO free list, sequences served in index order
  R15 optional shared pre-RoPE key offset on the injected keys (workload knob)
  R17 training-time block attention (P2 Fig. 4): a block of K positions
      that starts at response position c sees the target context at
      positions [0, c) (nothing later than its own start) and all K
      positions of its own block (bidirectional, as at inference), and
      nothing of any other block (no leakage between blocks); anchors (clean
      tokens inside a block) change only the block's input embeddings, not
      the mask
  R16 FP8 weights (the Guide mentions mixed FP4/FP8 execution on Blackwell): a
      projection weight is an e4m3 code per entry and an fp32 scale per
      output row, W = diag(s) . decode(codes); the drafter's arithmetic is
      otherwise that of the bf16 workload

Pins (tests/test_oracle_pins.py, tests/test_oracle_accept_pins.py): closed
forms, textbook special cases, invariants, brute force and exact
enumeration; the stochastic acceptance (accept_stochastic, race_sample)
against an exact enumeration of the lossless rule, the rule's closed-form
per-round outcome probabilities and the race's defining frequencies.  There is no worked numeric
example on any page, so the block's logit VALUES are pinned only through
those invariants and special cases (two independent formulations of KV
injection, RoPE shift invariance, special weights that reduce a layer to the
identity, textbook attention cases).
"""
from __future__ import annotations

import collections
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

F64 = np.float64


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=F64)


# ---------------------------------------------------------------------------
# Building blocks
# ---------------------------------------------------------------------------

def rms_norm(x: np.ndarray, gain: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * gain over the last axis (R1; the drafter's
    norm type is not printed on the pages, RMSNorm is the workload's)."""
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * _f64(gain)


def rope_cos_sin(pos: np.ndarray, head_dim: int, theta: float) -> Tuple[np.ndarray, np.ndarray]:
    """Angles pos * theta^(-2i/dh), i < dh/2 (R4).  Returns cos, sin [n, dh/2]."""
    half = head_dim // 2
    inv_freq = theta ** (-(2.0 * np.arange(half, dtype=F64)) / head_dim)
    ang = _f64(pos)[:, None] * inv_freq[None, :]
    return np.cos(ang), np.sin(ang)


def apply_rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE on x [n, H, dh] at positions pos [n] (R4): element i of
    the first half and element i of the second half form one rotated pair."""
    x = _f64(x)
    dh = x.shape[-1]
    half = dh // 2
    c, s = rope_cos_sin(pos, dh, theta)
    c = c[:, None, :]
    s = s[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(t: np.ndarray) -> np.ndarray:
    """t * sigmoid(t)."""
    t = _f64(t)
    return t / (1.0 + np.exp(-t))


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """Unmasked softmax attention with grouped kv heads (R7).

    q [n_q, Hq, dh], k/v [n_k, Hkv, dh] -> o [n_q, Hq, dh].  Query head h reads
    kv head h // G.  No causal mask: block positions see every context key and
    every block key (P1: attention inside the block is bidirectional; P3 the [MASK]
    placeholders of both neighbours are visible).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    Hq, dh = q.shape[1], q.shape[2]
    G = Hq // k.shape[1]
    out = np.empty_like(q)
    for h in range(Hq):
        g = h // G
        s = q[:, h, :] @ k[:, g, :].T / np.sqrt(dh)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, g, :]
    return out


def block_attention_train(q: np.ndarray, k_blk: np.ndarray, v_blk: np.ndarray,
                          ctx_k: Sequence[np.ndarray], ctx_v: Sequence[np.ndarray],
                          seq: np.ndarray, ctx_len: np.ndarray) -> np.ndarray:
    """Training-time block attention (R17, P2 Fig. 4).

    q [NB, K, Hq, dh]; k_blk, v_blk [NB, K, Hkv, dh] (the blocks' own keys,
    positions already encoded, and values); ctx_k[s], ctx_v[s] [T_s, Hkv, dh]
    the context of sequence s.  Block j belongs to sequence seq[j] and sees
    that context's first ctx_len[j] positions and its own K keys, unmasked.
    Returns o [NB, K, Hq, dh]."""
    out = np.empty(np.shape(q), dtype=F64)
    for j in range(len(seq)):
        s, c = int(seq[j]), int(ctx_len[j])
        keys = np.concatenate([_f64(ctx_k[s])[:c], _f64(k_blk[j])], axis=0)
        vals = np.concatenate([_f64(ctx_v[s])[:c], _f64(v_blk[j])], axis=0)
        out[j] = attention(q[j], keys, vals)
    return out


# ---------------------------------------------------------------------------
# Step 1-2: feature fusion and KV injection
# ---------------------------------------------------------------------------

def fuse_features(feats: np.ndarray, w_fc: np.ndarray, g_fc: np.ndarray, eps: float) -> np.ndarray:
    """h = RMSNorm(concat(taps) . W_fc^T)   [n, d].

    P1 "2. Target Hidden-State Conditioning", H_cond = W_proj H_T; P2 Fig. 2
    ("hidden context features ... are fused").  ``feats`` already holds the taps
    concatenated in ascending layer order (R1).
    """
    u = _f64(feats) @ _f64(w_fc).T
    return rms_norm(u, g_fc, eps)


def project_kv(h: np.ndarray, w_k: np.ndarray, w_v: np.ndarray, pos: np.ndarray,
               n_kv_heads: int, theta: float,
               key_offset: Optional[np.ndarray] = None) -> Tuple[np.ndarray, np.ndarray]:
    """One draft layer's injected K, V for fused rows h [n, d] at positions pos.

    P1 "3. Cross-Layer KV Injection": K^(l) = W_K^(l) H_cond, V^(l) = W_V^(l) H_cond;
    P3 "KV Injection": the target's representations pass through the draft
    model's KV projections into its KV cache.  Keys are rotated at their
    absolute position (R4); no bias (R3) except the optional workload offset
    key_offset [Hkv, dh], added before the rotation (R15).
    """
    n = h.shape[0]
    dh = w_k.shape[0] // n_kv_heads
    k = (_f64(h) @ _f64(w_k).T).reshape(n, n_kv_heads, dh)
    if key_offset is not None:
        k = k + _f64(key_offset)[None, :, :]
    v = (_f64(h) @ _f64(w_v).T).reshape(n, n_kv_heads, dh)
    return apply_rope(k, pos, theta), v


class PagedKV:
    """Paged draft KV cache that holds only injected target context.

    P1 "Zero Redundant KV Caching" and P3 ("the drafter never builds its own
    understanding of the prompt"): only injected rows are stored; the block's
    own keys and values are never cached, so rejected drafts need no rollback.

    Pool K, V: [L, n_pages, Hkv, page, dh].  Page table [B, max_pages] (-1 =
    none).  Allocation (R14): a FIFO free list that starts 0..P-1; an append of
    n_b rows to every sequence serves b = 0..B-1 in order, and sequence b takes
    ceil((len_b + n_b)/page) - ceil(len_b/page) pages from the head of the list.
    If the total need exceeds the free count the append fails and changes
    nothing.  ``release`` returns a sequence's pages to the tail in table order.
    """

    def __init__(self, n_layers: int, n_pages: int, n_kv_heads: int, head_dim: int,
                 batch: int, max_pages_per_seq: int, page_size: int = 16,
                 initial_free: Optional[Sequence[int]] = None):
        self.L, self.P, self.H, self.dh = n_layers, n_pages, n_kv_heads, head_dim
        self.page = page_size
        self.k = np.zeros((n_layers, n_pages, n_kv_heads, page_size, head_dim), F64)
        self.v = np.zeros_like(self.k)
        self.page_table = np.full((batch, max_pages_per_seq), -1, np.int64)
        self.seq_len = np.zeros(batch, np.int64)
        order = range(n_pages) if initial_free is None else initial_free
        self.free = collections.deque(int(p) for p in order)

    def pages_needed(self, b: int, n: int) -> int:
        pg = self.page
        return -(-(int(self.seq_len[b]) + n) // pg) - (-(-int(self.seq_len[b]) // pg))

    def allocate(self, n_rows: Sequence[int]) -> bool:
        """Reserve pages for n_rows[b] new rows of every sequence (R14)."""
        need = [self.pages_needed(b, int(n)) for b, n in enumerate(n_rows)]
        if sum(need) > len(self.free):
            return False
        for b, nb in enumerate(need):
            first = -(-int(self.seq_len[b]) // self.page)
            if first + nb > self.page_table.shape[1]:
                raise ValueError("sequence exceeds max_pages_per_seq")
            for j in range(nb):
                self.page_table[b, first + j] = self.free.popleft()
        return True

    def slot(self, b: int, pos: int) -> Tuple[int, int]:
        return int(self.page_table[b, pos // self.page]), pos % self.page

    def write(self, layer: int, b: int, pos: int, k_row: np.ndarray, v_row: np.ndarray) -> None:
        p, s = self.slot(b, pos)
        self.k[layer, p, :, s, :] = k_row
        self.v[layer, p, :, s, :] = v_row

    def gather(self, layer: int, b: int) -> Tuple[np.ndarray, np.ndarray]:
        """Context keys/values of sequence b in position order: [T_b, Hkv, dh]."""
        T = int(self.seq_len[b])
        pos = np.arange(T)
        pages = self.page_table[b, pos // self.page]
        slots = pos % self.page
        return self.k[layer, pages, :, slots, :], self.v[layer, pages, :, slots, :]

    def release(self, b: int) -> None:
        n = -(-int(self.seq_len[b]) // self.page)
        for j in range(n):
            self.free.append(int(self.page_table[b, j]))
            self.page_table[b, j] = -1
        self.seq_len[b] = 0


def inject(cache: PagedKV, w: Dict[str, np.ndarray], feats: Sequence[np.ndarray], cfg,
           key_offsets: Optional[np.ndarray] = None) -> bool:
    """Append feats[b] ([n_b, n_taps*tap_width]) to every sequence b.

    Fusion (step 1) then, for every layer, injected K/V (step 2) written into
    the pages at positions seq_len[b] .. seq_len[b]+n_b-1; seq_len advances by
    n_b.  Returns False (and changes nothing) when the pool is exhausted.
    """
    n_rows = [int(f.shape[0]) for f in feats]
    if not cache.allocate(n_rows):
        return False
    for b, f in enumerate(feats):
        n = n_rows[b]
        if n == 0:
            continue
        pos = int(cache.seq_len[b]) + np.arange(n)
        h = fuse_features(f, w["w_fc"], w["g_fc"], cfg.rms_eps)
        for l in range(cfg.n_layers):
            off = None if key_offsets is None else key_offsets[l]
            k, v = project_kv(h, w[f"w_k.{l}"], w[f"w_v.{l}"], pos, cfg.n_kv_heads,
                              cfg.rope_theta, off)
            for j in range(n):
                cache.write(l, b, int(pos[j]), k[j], v[j])
        cache.seq_len[b] += n
    return True


# ---------------------------------------------------------------------------
# Steps 4-8: the K-block draft forward pass and the LM head
# ---------------------------------------------------------------------------

def draft_layer(x: np.ndarray, w: Dict[str, np.ndarray], l: int, ctx_k: np.ndarray,
                ctx_v: np.ndarray, block_pos: np.ndarray, cfg) -> np.ndarray:
    """One pre-norm draft layer over the K block rows x [K, d].

    Attention reads [injected context ; block] keys/values with no mask (R7);
    SwiGLU MLP x += (silu(m W_g^T) * (m W_u^T)) W_d^T.
    """
    K = x.shape[0]
    a = rms_norm(x, w[f"g_in.{l}"], cfg.rms_eps)
    q = (a @ _f64(w[f"w_q.{l}"]).T).reshape(K, cfg.n_q_heads, cfg.head_dim)
    k = (a @ _f64(w[f"w_k.{l}"]).T).reshape(K, cfg.n_kv_heads, cfg.head_dim)
    v = (a @ _f64(w[f"w_v.{l}"]).T).reshape(K, cfg.n_kv_heads, cfg.head_dim)
    q = apply_rope(q, block_pos, cfg.rope_theta)
    k = apply_rope(k, block_pos, cfg.rope_theta)
    keys = np.concatenate([_f64(ctx_k), k], axis=0)
    vals = np.concatenate([_f64(ctx_v), v], axis=0)
    o = attention(q, keys, vals).reshape(K, -1)
    x = x + o @ _f64(w[f"w_o.{l}"]).T
    m = rms_norm(x, w[f"g_post.{l}"], cfg.rms_eps)
    gate = m @ _f64(w[f"w_gate.{l}"]).T
    up = m @ _f64(w[f"w_up.{l}"]).T
    return x + (silu(gate) * up) @ _f64(w[f"w_down.{l}"]).T


def lm_head(x: np.ndarray, w: Dict[str, np.ndarray], cfg) -> np.ndarray:
    """z = RMSNorm_final(x) W_lm^T (R6).  [K, V]."""
    return rms_norm(x, w["g_final"], cfg.rms_eps) @ _f64(w["w_lm"]).T


def logsumexp(z: np.ndarray) -> np.ndarray:
    m = z.max(axis=-1, keepdims=True)
    return (m + np.log(np.exp(z - m).sum(axis=-1, keepdims=True)))[..., 0]


def argmax_conf(z: np.ndarray) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Greedy draft tokens (ties to lowest index, R8), confidence
    exp(max - LSE) (the max softmax probability), and LSE.  P1 eq. in "1.
    Single-Pass Block-Diffusion Drafting": x_hat = argmax D_theta(m | x, H_T)."""
    tok = np.argmax(z, axis=-1)
    lse = logsumexp(z)
    conf = np.exp(z.max(axis=-1) - lse)
    return tok, conf, lse


def block_forward(w: Dict[str, np.ndarray], ctx_kv: Sequence[Tuple[np.ndarray, np.ndarray]],
                  T: int, block_tokens: np.ndarray, cfg) -> np.ndarray:
    """Logits [K, V] of one block pass for one sequence.

    ctx_kv[l] = (K_ctx, V_ctx) [T, Hkv, dh] of layer l.  block_tokens [K] are
    embedded (R5: all [MASK] in the first pass); block position i sits at
    absolute position T + i (P1 eq.: predict m_{1:gamma} given x_{<t}).
    """
    x = _f64(w["embed"])[np.asarray(block_tokens)]
    pos = T + np.arange(len(block_tokens))
    for l in range(cfg.n_layers):
        x = draft_layer(x, w, l, ctx_kv[l][0], ctx_kv[l][1], pos, cfg)
    return lm_head(x, w, cfg)


def commit_order(conf: np.ndarray, n_commit: int) -> np.ndarray:
    """Boolean mask of the n_commit most confident positions, ties to the lower
    position (R9; P3: positions are committed most confident first)."""
    K = conf.shape[0]
    order = sorted(range(K), key=lambda i: (-float(conf[i]), i))
    mask = np.zeros(K, bool)
    mask[order[:n_commit]] = True
    return mask


def draft(w: Dict[str, np.ndarray], ctx_kv, T: int, cfg, s_passes: int = 1) -> Dict[str, np.ndarray]:
    """One DFlash draft of a K block for one sequence (P1 "1. Single-Pass
    Block-Diffusion Drafting"; P3 "The Model at a Glance": a fully masked K
    block, S refinement passes committing positions in confidence order).

    Returns tokens [K], conf [K], lse [K], logits [K, V] (for S = 2: pass-1
    rows on the committed positions, pass-2 rows elsewhere), commit [K] bool
    (all False for S = 1) and the pass-1 logits.
    """
    K = cfg.block_k
    masks = np.full(K, cfg.mask_id, np.int64)
    z1 = block_forward(w, ctx_kv, T, masks, cfg)
    tok1, conf1, lse1 = argmax_conf(z1)
    if s_passes == 1:
        return dict(tokens=tok1, conf=conf1, lse=lse1, logits=z1,
                    commit=np.zeros(K, bool), logits_pass1=z1)
    if s_passes != 2:
        raise ValueError("S must be 1 or 2")
    commit = commit_order(conf1, K // 2)
    inp = np.where(commit, tok1, cfg.mask_id)
    z2 = block_forward(w, ctx_kv, T, inp, cfg)
    tok2, conf2, lse2 = argmax_conf(z2)
    c = commit
    return dict(tokens=np.where(c, tok1, tok2), conf=np.where(c, conf1, conf2),
                lse=np.where(c, lse1, lse2), logits=np.where(c[:, None], z1, z2),
                commit=commit, logits_pass1=z1)


def dense_block_forward(w: Dict[str, np.ndarray], h_ctx: np.ndarray, ctx_pos: np.ndarray,
                        block_pos: np.ndarray, block_tokens: np.ndarray, cfg,
                        key_offsets: Optional[np.ndarray] = None) -> np.ndarray:
    """Second, page-free formulation of the same pass (pin for KV injection).

    Projects the fused context rows h_ctx with each layer's W_k/W_v and
    concatenates them in front of the block's own keys/values, all inside one
    explicit attention call, with explicit positions.  P1 eq. K^(l) = W_K^(l)
    H_cond; its toy drafter's idea of concatenating the projected context into
    the sequence, applied at the K/V level.
    """
    x = _f64(w["embed"])[np.asarray(block_tokens)]
    K = x.shape[0]
    for l in range(cfg.n_layers):
        kc = (_f64(h_ctx) @ _f64(w[f"w_k.{l}"]).T).reshape(len(ctx_pos), cfg.n_kv_heads, cfg.head_dim)
        if key_offsets is not None:
            kc = kc + _f64(key_offsets[l])[None]
        vc = (_f64(h_ctx) @ _f64(w[f"w_v.{l}"]).T).reshape(len(ctx_pos), cfg.n_kv_heads, cfg.head_dim)
        a = rms_norm(x, w[f"g_in.{l}"], cfg.rms_eps)
        q = (a @ _f64(w[f"w_q.{l}"]).T).reshape(K, cfg.n_q_heads, -1)
        kb = (a @ _f64(w[f"w_k.{l}"]).T).reshape(K, cfg.n_kv_heads, -1)
        vb = (a @ _f64(w[f"w_v.{l}"]).T).reshape(K, cfg.n_kv_heads, -1)
        all_pos = np.concatenate([ctx_pos, block_pos])
        keys = apply_rope(np.concatenate([kc, kb], 0), all_pos, cfg.rope_theta)
        vals = np.concatenate([vc, vb], 0)
        qr = apply_rope(q, block_pos, cfg.rope_theta)
        o = attention(qr, keys, vals).reshape(K, -1)
        x = x + o @ _f64(w[f"w_o.{l}"]).T
        m = rms_norm(x, w[f"g_post.{l}"], cfg.rms_eps)
        x = x + (silu(m @ _f64(w[f"w_gate.{l}"]).T) * (m @ _f64(w[f"w_up.{l}"]).T)) @ _f64(w[f"w_down.{l}"]).T
    return lm_head(x, w, cfg)


# ---------------------------------------------------------------------------
# Steps 10-11: lossless acceptance
# ---------------------------------------------------------------------------

def accept_greedy(drafts: np.ndarray, target: np.ndarray) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Greedy longest-prefix acceptance (P1 "Verification Phase": the longest
    valid prefix tau <= gamma is accepted; R10).

    drafts [B, K], target [B, K+1] (the target's greedy token at each block
    position and the bonus position).  tau_b = first i with d_i != y_i, else K.
    Emits y_0 .. y_tau (tau+1 tokens; y_i = d_i for i < tau).  Returns tau [B],
    emitted [B, K+1] (-1 padded), n_emit [B] = tau+1.
    """
    drafts = np.asarray(drafts)
    target = np.asarray(target)
    B, K = drafts.shape
    tau = np.full(B, K, np.int64)
    for b in range(B):
        for i in range(K):
            if drafts[b, i] != target[b, i]:
                tau[b] = i
                break
    emitted = np.full((B, K + 1), -1, np.int64)
    for b in range(B):
        emitted[b, :tau[b] + 1] = target[b, :tau[b] + 1]
    return tau, emitted, tau + 1


_PHILOX_M0, _PHILOX_M1 = 0xD2511F53, 0xCD9E8D57
_PHILOX_W0, _PHILOX_W1 = 0x9E3779B9, 0xBB67AE85
_M32 = 0xFFFFFFFF


def philox4x32_10(ctr: np.ndarray, key: np.ndarray) -> np.ndarray:
    """Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel random
    numbers: as easy as 1, 2, 3", SC'11).  ctr [..., 4], key [..., 2] uint32-valued.

    One round maps (c0, c1, c2, c3) with key (k0, k1) to
    (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0)); between
    rounds the key is bumped by the Weyl constants W0, W1 (mod 2^32).  The
    32x32-bit products are formed exactly on uint64 lanes.
    """
    c = np.asarray(ctr, dtype=np.uint64) & _M32
    k = np.asarray(key, dtype=np.uint64) & _M32
    c0, c1, c2, c3 = (c[..., j].copy() for j in range(4))
    k0, k1 = k[..., 0].copy(), k[..., 1].copy()
    m0, m1 = np.uint64(_PHILOX_M0), np.uint64(_PHILOX_M1)
    for r in range(10):
        p0 = m0 * c0          # < 2^64: 32x32 products fit in uint64
        p1 = m1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(_M32)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(_M32)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        if r < 9:
            k0 = (k0 + np.uint64(_PHILOX_W0)) & np.uint64(_M32)
            k1 = (k1 + np.uint64(_PHILOX_W1)) & np.uint64(_M32)
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def uniform_from_u32(x: np.ndarray) -> np.ndarray:
    """Open-interval uniform: ((x >> 9) + 1/2) * 2^-23, exactly representable
    in fp32 and fp64, in [2^-24, 1 - 2^-24]."""
    return ((np.asarray(x, dtype=np.uint64) >> np.uint64(9)).astype(F64) + 0.5) * 2.0 ** -23


STREAM_ACCEPT, STREAM_RACE = 0, 1


def rng_uniform(seed: int, rnd: int, b, i, stream: int, v) -> np.ndarray:
    """The uniform of R12: Philox4x32-10 at key (seed lo, seed hi) and
    counter (v >> 2, i | stream << 16, b, round lo), output word v & 3,
    broadcast over b, i, v."""
    b, i, v = np.broadcast_arrays(np.asarray(b, np.uint64), np.asarray(i, np.uint64),
                                  np.asarray(v, np.uint64))
    ctr = np.stack([v >> np.uint64(2), i | np.uint64(stream << 16), b,
                    np.full(b.shape, rnd & _M32, np.uint64)], axis=-1)
    key = np.broadcast_to(np.array([seed & _M32, (seed >> 32) & _M32], np.uint64), ctr.shape[:-1] + (2,))
    words = philox4x32_10(ctr, key)
    word = np.take_along_axis(words, (v & np.uint64(3)).astype(np.int64)[..., None], axis=-1)[..., 0]
    return uniform_from_u32(word)


def race_sample(r: np.ndarray, seed: int, rnd: int, b: int, i: int) -> int:
    """Draw v with probability r(v)/sum(r) by an exponential race (R13):
    argmax_v r(v)/E_v with E_v = -ln U_v, U_v the race-stream uniform at v;
    ties to the lowest v.  (min_v E_v/r(v) is exponential with rate sum(r) and
    falls on v with probability r(v)/sum(r).)"""
    V = r.shape[0]
    u = rng_uniform(seed, rnd, b, i, STREAM_RACE, np.arange(V))
    e = -np.log(u)
    key = np.where(r > 0, _f64(r) / e, -np.inf)
    return int(np.argmax(key))


def softmax(z: np.ndarray) -> np.ndarray:
    z = _f64(z)
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def accept_stochastic(target_logits: np.ndarray, drafts: np.ndarray,
                      draft_probs: Optional[np.ndarray], temperature: float,
                      seed: int, rnd: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Speculative rejection sampling (P1 "Verification Phase"; P3 "the lossless
    acceptance rule ... position by position"; the output distribution is the
    target's exactly).

    p_i = softmax(z_i / temperature) from target_logits [B, K+1, V].  For
    i = 0, 1, ...: accept d_i iff u_i < min(1, p_i(d_i) / q_i(d_i)); on the
    first reject emit a draw from norm(max(0, p_i - q_i)) and stop; if all K are
    accepted emit a draw from p_K.  draft_probs None means the point-mass q
    (R11).  A residual with zero mass (p_i = q_i) falls back to p_i.
    Returns tau [B], emitted [B, K+1] (-1 padded), n_emit [B].
    """
    z = _f64(target_logits)
    B, K1, V = z.shape
    K = K1 - 1
    drafts = np.asarray(drafts)
    tau = np.full(B, K, np.int64)
    emitted = np.full((B, K + 1), -1, np.int64)
    for b in range(B):
        for i in range(K + 1):
            p = softmax(z[b, i] / temperature)
            if i == K:
                emitted[b, K] = race_sample(p, seed, rnd, b, K)
                break
            d = int(drafts[b, i])
            if draft_probs is None:
                q = np.zeros(V)
                q[d] = 1.0
            else:
                q = _f64(draft_probs[b, i])
            u = float(rng_uniform(seed, rnd, b, i, STREAM_ACCEPT, 0))
            ratio = p[d] / q[d] if q[d] > 0 else np.inf
            if u < min(1.0, ratio):
                emitted[b, i] = d
                continue
            r = np.maximum(0.0, p - q)
            if r.sum() <= 0:
                r = p
            emitted[b, i] = race_sample(r, seed, rnd, b, i)
            tau[b] = i
            break
    return tau, emitted, tau + 1


def accept_stochastic_trials(p_rows: np.ndarray, q_rows: Optional[np.ndarray],
                             drafts: np.ndarray, seed: int, rnd: int) -> Tuple[np.ndarray, np.ndarray]:
    """The same rule as ``accept_stochastic``, vectorised over many independent
    trials for the Monte-Carlo pin.  p_rows [K+1, V] and q_rows [K, V] are
    shared by all trials; drafts [N, K]; trial n uses RNG sequence index b = n.
    Returns tau [N], emitted [N, K+1]."""
    N, K = drafts.shape
    V = p_rows.shape[1]
    p_rows = _f64(p_rows)
    alive = np.ones(N, bool)
    tau = np.full(N, K, np.int64)
    emitted = np.full((N, K + 1), -1, np.int64)
    n_idx = np.arange(N)
    vv = np.arange(V)
    for i in range(K + 1):
        idx = n_idx[alive]
        if idx.size == 0:
            break
        p = p_rows[i]
        e = -np.log(rng_uniform(seed, rnd, idx[:, None], i, STREAM_RACE, vv[None, :]))
        if i == K:
            key = np.where(p[None, :] > 0, p[None, :] / e, -np.inf)
            emitted[idx, K] = np.argmax(key, axis=1)
            break
        d = drafts[idx, i]
        if q_rows is None:
            qd = np.ones(idx.size)
            q = np.zeros((idx.size, V))
            q[np.arange(idx.size), d] = 1.0
        else:
            q = np.broadcast_to(_f64(q_rows[i]), (idx.size, V))
            qd = q[np.arange(idx.size), d]
        ratio = np.where(qd > 0, p[d] / np.where(qd > 0, qd, 1.0), np.inf)
        u = rng_uniform(seed, rnd, idx, i, STREAM_ACCEPT, 0)
        acc = u < np.minimum(1.0, ratio)
        emitted[idx[acc], i] = d[acc]
        rej = idx[~acc]
        if rej.size:
            r = np.maximum(0.0, p[None, :] - q[~acc])
            zero = r.sum(axis=1) <= 0
            r[zero] = p[None, :]
            key = np.where(r > 0, r / e[~acc], -np.inf)
            emitted[rej, i] = np.argmax(key, axis=1)
            tau[rej] = i
            alive[rej] = False
    return tau, emitted


# ---------------------------------------------------------------------------
# FP8 (e4m3) weights (R16)
# ---------------------------------------------------------------------------

def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """Values of 8-bit E4M3 codes (OCP 8-bit floating point, "FP8 E4M3"):
    sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
    holds the subnormals m/8 * 2^-6; no infinities; S.1111.111 is NaN, so the
    largest finite magnitude is 1.75 * 2^8 = 448."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7 == 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(F64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2((e - 7).astype(F64)))
    out = sign * mag
    return np.where((e == 15) & ((c & 7) == 7), np.nan, out)


def dequantize_weights(w: Dict[str, np.ndarray]) -> Dict[str, np.ndarray]:
    """A weight set whose projections are stored as e4m3 codes ("q:<name>",
    uint8 [rows, cols]) with per-row scales ("s:<name>", fp32 [rows]) ->
    the same set with "<name>" = s[:, None] * decode(codes) in fp64 (exact:
    a product of an fp32 and a 4-significant-bit value).  Other entries pass
    through."""
    out = {}
    for k, v in w.items():
        if k.startswith("q:"):
            name = k[2:]
            out[name] = _f64(w["s:" + name])[:, None] * decode_e4m3(v)
        elif not k.startswith("s:"):
            out[k] = v
    return out


# ---------------------------------------------------------------------------
# A whole round for a batch (driver used by tests and the CPU baseline)
# ---------------------------------------------------------------------------

class OracleDrafter:
    """Holds one batch's paged cache and runs inject -> draft -> accept rounds
    (P3 "each cycle becomes: one parallel draft pass proposes the block -> one
    target pass verifies it")."""

    def __init__(self, cfg, weights: Dict[str, np.ndarray], n_pages: int, max_pages_per_seq: int,
                 key_offsets: Optional[np.ndarray] = None, seqs: Optional[Sequence[int]] = None):
        self.cfg = cfg
        if any(k.startswith("q:") for k in weights):
            weights = dequantize_weights(weights)
        self.w = {k: _f64(v) for k, v in weights.items()}
        self.key_offsets = key_offsets
        B = cfg.batch if seqs is None else len(seqs)
        self.cache = PagedKV(cfg.n_layers, n_pages, cfg.n_kv_heads, cfg.head_dim, B,
                             max_pages_per_seq, cfg.page_size)

    def inject(self, feats: Sequence[np.ndarray]) -> bool:
        return inject(self.cache, self.w, feats, self.cfg, self.key_offsets)

    def ctx_kv(self, b: int):
        return [self.cache.gather(l, b) for l in range(self.cfg.n_layers)]

    def draft(self, b: int, s_passes: Optional[int] = None) -> Dict[str, np.ndarray]:
        S = self.cfg.s_passes if s_passes is None else s_passes
        return draft(self.w, self.ctx_kv(b), int(self.cache.seq_len[b]), self.cfg, S)

"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these re-types an oracle formula: each checks a closed form, a
textbook special case, a library routine, an invariant, brute force or a
published known-answer vector, chosen so that a plausible slip (a dropped
term, a wrong sign or index, a transposed operand, a swapped gate) fails.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import synth
from oracle import dflash_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tiny_cfg(**kw):
    base = dict(name="pin", batch=2, ctx_lo=3, ctx_hi=40, n_layers=2, hidden=32,
                n_q_heads=4, n_kv_heads=2, head_dim=8, ffn=24, vocab=50, n_taps=2,
                tap_width=12, dtype="f32", rounds=2, seed=77)
    base.update(kw)
    return synth.DraftConfig(**base)


def f64w(cfg):
    return {k: v.astype(np.float64) for k, v in synth.make_weights(cfg, threads=2).items()}


# ---------------------------------------------------------------- building blocks

def test_rms_norm_closed_form():
    x = np.array([[3.0, 4.0]])
    out = O.rms_norm(x, np.array([1.0, 2.0]), 0.0)
    r = math.sqrt(12.5)
    np.testing.assert_allclose(out, [[3 / r, 8 / r]], rtol=1e-15)
    c = np.full((1, 7), -0.25)
    np.testing.assert_allclose(O.rms_norm(c, np.ones(7), 1e-2), -0.25 / math.sqrt(0.0625 + 1e-2),
                               rtol=1e-14)


def test_rope_identity_at_zero_and_2x2_rotation():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((3, 2, 6))
    np.testing.assert_array_equal(O.apply_rope(x, np.zeros(3), 1e6), x)
    # dh = 2: the single pair (x0, x1) turns by angle pos (inverse frequency 1)
    v = rng.standard_normal((4, 1, 2))
    pos = np.array([0.0, 1.0, 2.5, 1000.0])
    out = O.apply_rope(v, pos, 1e6)
    for n in range(4):
        R = np.array([[math.cos(pos[n]), -math.sin(pos[n])], [math.sin(pos[n]), math.cos(pos[n])]])
        np.testing.assert_allclose(out[n, 0], R @ v[n, 0], rtol=1e-13, atol=1e-13)


def test_rope_rotate_half_pairing_dh4():
    # theta = 100, dh = 4: inverse frequencies 1 and 100^(-1/2) = 0.1; pairs are
    # (x0, x2) and (x1, x3) (rotate-half), not (x0, x1).
    x = np.array([[[1.0, 2.0, 3.0, 4.0]]])
    p = 3.0
    out = O.apply_rope(x, np.array([p]), 100.0)[0, 0]
    a0, a1 = p * 1.0, p * 0.1
    exp = [1 * math.cos(a0) - 3 * math.sin(a0), 2 * math.cos(a1) - 4 * math.sin(a1),
           3 * math.cos(a0) + 1 * math.sin(a0), 4 * math.cos(a1) + 2 * math.sin(a1)]
    np.testing.assert_allclose(out, exp, rtol=1e-14, atol=1e-14)


def test_rope_norm_and_relative_position():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 1, 64))
    k = rng.standard_normal((1, 1, 64))
    for (p, s, d) in [(5, 2, 11), (0, 400, 3000), (33000, 17, 129)]:
        qa = O.apply_rope(q, np.array([p]), 1e6)
        ka = O.apply_rope(k, np.array([s]), 1e6)
        qb = O.apply_rope(q, np.array([p + d]), 1e6)
        kb = O.apply_rope(k, np.array([s + d]), 1e6)
        assert abs(np.linalg.norm(qa) - np.linalg.norm(q)) < 1e-12
        assert abs(np.sum(qa * ka) - np.sum(qb * kb)) < 1e-10


def test_silu_library_and_odd_identity():
    t = np.linspace(-30, 30, 601)
    np.testing.assert_allclose(O.silu(t), t * scipy.special.expit(t), rtol=1e-14, atol=1e-300)
    # silu(t) - silu(-t) = t  (sigma(t) + sigma(-t) = 1)
    np.testing.assert_allclose(O.silu(t) - O.silu(-t), t, atol=1e-12)
    assert O.silu(np.array([0.0]))[0] == 0.0


def test_attention_textbook_cases():
    rng = np.random.default_rng(2)
    # identical keys: uniform weights -> mean of the values
    q = rng.standard_normal((5, 2, 8))
    k = np.repeat(rng.standard_normal((1, 2, 8)), 7, axis=0)
    v = rng.standard_normal((7, 2, 8))
    np.testing.assert_allclose(O.attention(q, k, v), np.broadcast_to(v.mean(0), (5, 2, 8)), atol=1e-13)
    # two keys: weight of key 0 = sigmoid((s0 - s1)/sqrt(dh))
    q = rng.standard_normal((1, 1, 16))
    k = rng.standard_normal((2, 1, 16))
    v = rng.standard_normal((2, 1, 16))
    s = (k[:, 0] @ q[0, 0])
    w0 = scipy.special.expit((s[0] - s[1]) / 4.0)
    np.testing.assert_allclose(O.attention(q, k, v)[0, 0], w0 * v[0, 0] + (1 - w0) * v[1, 0], atol=1e-13)
    # one dominant key
    k = rng.standard_normal((6, 1, 16)) * 0.01
    k[3] = q[0] * 1e3
    vv = rng.standard_normal((6, 1, 16))
    np.testing.assert_allclose(O.attention(q, k, vv)[0, 0], vv[3, 0], atol=1e-12)


def test_attention_gqa_equals_repeated_mha_and_key_permutation():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((4, 8, 16))
    k = rng.standard_normal((9, 2, 16))
    v = rng.standard_normal((9, 2, 16))
    gqa = O.attention(q, k, v)
    mha = O.attention(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1))
    np.testing.assert_allclose(gqa, mha, atol=1e-14)
    perm = rng.permutation(9)
    np.testing.assert_allclose(O.attention(q, k[perm], v[perm]), gqa, atol=1e-13)
    # G = 4: query heads 0-3 read kv head 0 and heads 4-7 kv head 1 (h // G,
    # not h % Hkv); perturbing kv head 1 must leave heads 0-3 untouched
    k2 = k.copy()
    k2[:, 1] += 10.0 * rng.standard_normal((9, 16))
    out2 = O.attention(q, k2, v)
    np.testing.assert_allclose(out2[:, :4], gqa[:, :4], atol=1e-14)
    assert np.abs(out2[:, 4:] - gqa[:, 4:]).max() > 1e-3


# ---------------------------------------------------------------- fusion and injection

def test_fusion_selects_a_tap_with_block_identity():
    rng = np.random.default_rng(4)
    d = 12
    feats = rng.standard_normal((5, 3 * d))
    w = np.zeros((d, 3 * d))
    w[:, d:2 * d] = np.eye(d)        # keep tap 1 only
    h = O.fuse_features(feats, w, np.ones(d), 1e-6)
    t = feats[:, d:2 * d]
    np.testing.assert_allclose(h, t / np.sqrt((t ** 2).mean(1, keepdims=True) + 1e-6), rtol=1e-13)


def test_project_kv_identity_weights():
    rng = np.random.default_rng(5)
    h = rng.standard_normal((4, 8))
    k, v = O.project_kv(h, np.eye(8), 2 * np.eye(8), np.zeros(4), 2, 1e6)
    np.testing.assert_allclose(k.reshape(4, 8), h, atol=1e-15)
    np.testing.assert_allclose(v.reshape(4, 8), 2 * h, atol=1e-15)


def _chain(cfg, w, initial_free=None, split_rounds=True, key_offsets=None):
    """Prefill + 2 rounds (ragged row counts); returns the drafter."""
    lens = synth.make_ctx_lens(cfg)
    n_pages = 64
    dr = O.OracleDrafter(cfg, w, n_pages, 16, key_offsets=key_offsets)
    if initial_free is not None:
        dr.cache = O.PagedKV(cfg.n_layers, n_pages, cfg.n_kv_heads, cfg.head_dim, cfg.batch, 16,
                             cfg.page_size, initial_free)
    pre = [synth.make_prefill_features(cfg, b, int(lens[b])) for b in range(cfg.batch)]
    extra = [[synth.make_round_features(cfg, r, b, 1 + (3 * b + 5 * r) % 17) for b in range(cfg.batch)]
             for r in range(2)]
    if split_rounds:
        assert dr.inject(pre)
        for r in range(2):
            assert dr.inject(extra[r])
    else:
        assert dr.inject([np.concatenate([pre[b], extra[0][b], extra[1][b]]) for b in range(cfg.batch)])
    return dr, pre, extra


def test_kv_injection_paged_equals_dense_concatenation():
    """KV injection == projecting the fused features with W_k/W_v and
    concatenating them into attention (P1 eq. K^(l) = W_K^(l) H_cond)."""
    cfg = tiny_cfg(key_offset_std=3.0)
    w = f64w(cfg)
    off = synth.make_key_offsets(cfg)
    dr, pre, extra = _chain(cfg, w, key_offsets=off)
    for b in range(cfg.batch):
        rows = np.concatenate([pre[b], extra[0][b], extra[1][b]])
        h = O.fuse_features(rows, w["w_fc"], w["g_fc"], cfg.rms_eps)
        T = rows.shape[0]
        assert int(dr.cache.seq_len[b]) == T
        masks = np.full(cfg.block_k, cfg.mask_id)
        dense = O.dense_block_forward(w, h, np.arange(T), T + np.arange(cfg.block_k), masks, cfg,
                                      key_offsets=off)
        paged = dr.draft(b)["logits"]
        np.testing.assert_allclose(paged, dense, rtol=0, atol=1e-12)


def test_paging_permutation_and_incremental_invariance():
    cfg = tiny_cfg()
    w = f64w(cfg)
    a, _, _ = _chain(cfg, w)
    perm = list(np.random.default_rng(6).permutation(64))
    bperm, _, _ = _chain(cfg, w, initial_free=perm)
    c, _, _ = _chain(cfg, w, split_rounds=False)
    assert not np.array_equal(a.cache.page_table, bperm.cache.page_table)
    for b in range(cfg.batch):
        za = a.draft(b)["logits"]
        np.testing.assert_array_equal(za, bperm.draft(b)["logits"])
        # one prefill of all rows vs prefill + rounds: BLAS blocks the
        # projections differently by row count, so equal to rounding only
        np.testing.assert_allclose(za, c.draft(b)["logits"], rtol=0, atol=1e-13)
        for l in range(cfg.n_layers):
            np.testing.assert_allclose(a.cache.gather(l, b)[0], c.cache.gather(l, b)[0], rtol=0, atol=1e-13)
            np.testing.assert_allclose(a.cache.gather(l, b)[1], c.cache.gather(l, b)[1], rtol=0, atol=1e-13)


def test_paging_worked_example():
    ex = json.load(open(os.path.join(GOLDEN, "paging_worked_example.json")))
    kv = O.PagedKV(1, ex["n_pages"], 1, 2, ex["batch"], ex["max_pages_per_seq"], ex["page_size"])
    for st in ex["steps"]:
        if st["op"] == "append":
            assert kv.allocate(st["n_rows"]) == st["ok"], st["why"]
            if st["ok"]:
                kv.seq_len += np.array(st["n_rows"])
        else:
            kv.release(st["b"])
        assert kv.page_table.tolist() == st["page_table"], st["why"]
        assert kv.seq_len.tolist() == st["seq_len"], st["why"]
        assert list(kv.free) == st["free"], st["why"]


def test_rope_shift_invariance_of_whole_block():
    cfg = tiny_cfg()
    w = f64w(cfg)
    rng = np.random.default_rng(7)
    h = rng.standard_normal((23, cfg.hidden))
    masks = np.full(cfg.block_k, cfg.mask_id)
    z0 = O.dense_block_forward(w, h, np.arange(23), 23 + np.arange(16), masks, cfg)
    z1 = O.dense_block_forward(w, h, 5000 + np.arange(23), 5023 + np.arange(16), masks, cfg)
    np.testing.assert_allclose(z0, z1, atol=1e-10)
    # but the block's own positions matter: without RoPE every row would be equal
    assert np.abs(z0[0] - z0[7]).max() > 1e-6


def test_layer_reduces_to_identity_and_head_closed_form():
    cfg = tiny_cfg()
    w = f64w(cfg)
    for l in range(cfg.n_layers):
        w[f"w_o.{l}"][:] = 0.0
        w[f"w_down.{l}"][:] = 0.0
    rng = np.random.default_rng(8)
    h = rng.standard_normal((10, cfg.hidden))
    z = O.dense_block_forward(w, h, np.arange(10), 10 + np.arange(16), np.full(16, cfg.mask_id), cfg)
    e = w["embed"][cfg.mask_id]
    expect = (e / np.sqrt(np.mean(e * e) + cfg.rms_eps)) @ w["w_lm"].T
    np.testing.assert_allclose(z, np.broadcast_to(expect, z.shape), atol=1e-12)


def test_zero_query_weights_make_keys_irrelevant():
    cfg = tiny_cfg()
    w = f64w(cfg)
    for l in range(cfg.n_layers):
        w[f"w_q.{l}"][:] = 0.0
    rng = np.random.default_rng(9)
    h = rng.standard_normal((10, cfg.hidden))
    args = (h, np.arange(10), 10 + np.arange(16), np.full(16, cfg.mask_id), cfg)
    z0 = O.dense_block_forward(w, *args)
    w2 = dict(w)
    for l in range(cfg.n_layers):
        w2[f"w_k.{l}"] = rng.standard_normal(w[f"w_k.{l}"].shape)
    np.testing.assert_allclose(O.dense_block_forward(w2, *args), z0, atol=1e-12)


def test_swiglu_gate_order_scalar_closed_form():
    # d = 2, F = 1, attention switched off (w_o = 0): x' = x + w_d * silu(w_g.m) * (w_u.m)
    cfg = tiny_cfg(n_layers=1, hidden=2, n_q_heads=1, n_kv_heads=1, head_dim=2, ffn=1, vocab=3)
    w = {"embed": np.array([[0.3, -1.2], [1.0, 2.0], [0.5, 0.5]]), "g_final": np.ones(2),
         "w_lm": np.eye(3, 2), "w_q.0": np.eye(2), "w_k.0": np.eye(2), "w_v.0": np.eye(2),
         "w_o.0": np.zeros((2, 2)), "w_gate.0": np.array([[0.7, -0.4]]),
         "w_up.0": np.array([[1.5, 0.25]]), "w_down.0": np.array([[2.0], [-1.0]]),
         "g_in.0": np.ones(2), "g_post.0": np.ones(2)}
    x = np.array([[0.3, -1.2]])
    out = O.draft_layer(x, w, 0, np.zeros((0, 1, 2)), np.zeros((0, 1, 2)), np.array([0]), cfg)
    r = math.sqrt((0.09 + 1.44) / 2 + cfg.rms_eps)
    m = [0.3 / r, -1.2 / r]
    g = 0.7 * m[0] - 0.4 * m[1]
    u = 1.5 * m[0] + 0.25 * m[1]
    act = g / (1 + math.exp(-g)) * u
    np.testing.assert_allclose(out[0], [0.3 + 2.0 * act, -1.2 - 1.0 * act], rtol=1e-13)


def test_empty_context_and_mask_only_block():
    cfg = tiny_cfg()
    w = f64w(cfg)
    dr = O.OracleDrafter(cfg, w, 8, 4)
    out = dr.draft(0)
    assert np.isfinite(out["logits"]).all()
    dense = O.dense_block_forward(w, np.zeros((0, cfg.hidden)), np.arange(0), np.arange(16),
                                  np.full(16, cfg.mask_id), cfg)
    np.testing.assert_allclose(out["logits"], dense, atol=1e-12)


def test_mask_semantics_logits_depend_only_on_context():
    """P3: a block position sees its neighbours' [MASK] placeholders, never
    sampled tokens; all K logits exist before any token is drawn.  At S = 1
    the logits are a function of (context rows, weights) alone."""
    cfg = tiny_cfg()
    w = f64w(cfg)
    a, _, _ = _chain(cfg, w)
    z = a.draft(0)["logits"]
    # same context, a different history of targets/drafts/RNG: identical logits
    tau, em, _ = O.accept_greedy(np.zeros((1, 16), int), np.ones((1, 17), int))
    b2, _, _ = _chain(cfg, w)
    O.accept_stochastic(np.zeros((1, 17, cfg.vocab)), np.zeros((1, 16), int), None, 1.0, 99, 3)
    np.testing.assert_array_equal(b2.draft(0)["logits"], z)
    # and the pass equals a forward whose block input is K copies of [MASK]
    T = int(a.cache.seq_len[0])
    z_direct = O.block_forward(a.w, a.ctx_kv(0), T, np.full(16, cfg.mask_id), cfg)
    np.testing.assert_array_equal(z_direct, z)


def test_argmax_confidence_closed_forms_and_library():
    # two logits: the confidence is the logistic of their gap
    for a, b in [(2.0, -1.0), (0.3, 0.1), (-5.0, -7.5)]:
        tok, conf, _ = O.argmax_conf(np.array([[a, b]]))
        assert tok[0] == 0 and math.isclose(conf[0], 1.0 / (1.0 + math.exp(b - a)), rel_tol=1e-14)
    # uniform row: 1 / V, the lowest index wins the tie
    tok, conf, lse = O.argmax_conf(np.full((1, 37), 0.25))
    assert tok[0] == 0 and math.isclose(conf[0], 1.0 / 37, rel_tol=1e-14)
    assert math.isclose(lse[0], 0.25 + math.log(37), rel_tol=1e-14)
    z = np.zeros((1, 10))
    z[0, 3] = z[0, 7] = 1.5
    assert O.argmax_conf(z)[0][0] == 3
    # against the library, including magnitudes that overflow a naive exp
    rng = np.random.default_rng(5)
    z = rng.standard_normal((6, 501)) * 4.0
    z[2] += 1000.0
    z[4] -= 800.0
    tok, conf, lse = O.argmax_conf(z)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(z, axis=-1), rtol=1e-13)
    np.testing.assert_allclose(conf, scipy.special.softmax(z, axis=-1).max(axis=-1), rtol=1e-12)
    np.testing.assert_array_equal(tok, np.argmax(scipy.special.softmax(z, axis=-1), axis=-1))
    # shifting a row changes neither the token nor the confidence
    t2, c2, l2 = O.argmax_conf(z + 123.0)
    np.testing.assert_array_equal(t2, tok)
    np.testing.assert_allclose(c2, conf, rtol=1e-12)
    np.testing.assert_allclose(l2, lse + 123.0, rtol=1e-13)


def test_lm_head_normalises_then_projects_rows():
    # W_lm = [I; 2I] (V = 2d, so a transposed operand cannot even multiply),
    # unit final gain: z = [x / rms(x), 2 x / rms(x)] per row
    cfg = tiny_cfg()
    d = cfg.hidden
    rng = np.random.default_rng(9)
    x = rng.standard_normal((3, d))
    w = {"g_final": np.ones(d), "w_lm": np.vstack([np.eye(d), 2.0 * np.eye(d)])}
    z = O.lm_head(x, w, cfg)
    xh = x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + cfg.rms_eps)
    np.testing.assert_allclose(z, np.hstack([xh, 2.0 * xh]), rtol=1e-13, atol=1e-13)


def test_two_pass_commit_rule():
    rng = np.random.default_rng(10)
    conf = rng.random(16)
    m = O.commit_order(conf, 8)
    np.testing.assert_array_equal(np.flatnonzero(m), np.sort(np.argsort(-conf, kind="stable")[:8]))
    assert O.commit_order(np.full(16, 0.5), 8).tolist() == [True] * 8 + [False] * 8
    c = np.array([0.1] * 4 + [0.9] * 12)
    assert np.flatnonzero(O.commit_order(c, 8)).tolist() == list(range(4, 12))


def test_two_pass_keeps_committed_and_equals_one_pass_when_head_prefers_mask():
    cfg = tiny_cfg(s_passes=2)
    w = f64w(cfg)
    a, _, _ = _chain(cfg, w)
    out = a.draft(0, s_passes=2)
    one = a.draft(0, s_passes=1)
    c = out["commit"]
    assert c.sum() == 8
    np.testing.assert_array_equal(out["tokens"][c], one["tokens"][c])
    np.testing.assert_array_equal(out["logits"][c], one["logits"][c])
    # pass 2 sees committed tokens: at least one uncommitted row changes
    assert np.abs(out["logits"][~c] - one["logits"][~c]).max() > 0
    # a zero LM head ties every logit: argmax takes token 0 (lowest index);
    # if token 0 embeds like [MASK], pass 2 sees pass 1's input and repeats it
    w2 = dict(a.w)
    w2["w_lm"] = np.zeros_like(w2["w_lm"])
    w2["embed"] = w2["embed"].copy()
    w2["embed"][0] = w2["embed"][cfg.mask_id]
    z1 = O.draft(w2, a.ctx_kv(0), int(a.cache.seq_len[0]), cfg, 1)
    assert (z1["tokens"] == 0).all()
    np.testing.assert_allclose(z1["conf"], 1.0 / cfg.vocab, rtol=1e-13)
    z2 = O.draft(w2, a.ctx_kv(0), int(a.cache.seq_len[0]), cfg, 2)
    np.testing.assert_array_equal(z2["logits"], z1["logits"])
    assert z2["commit"].tolist() == [True] * 8 + [False] * 8


# ---------------------------------------------------------------- acceptance

def test_greedy_accept_brute_force_all_mismatch_patterns():
    K = 10
    rng = np.random.default_rng(11)
    y = rng.integers(0, 100, size=(1 << K, K + 1))
    d = y[:, :K].copy()
    for pat in range(1 << K):
        for i in range(K):
            if pat >> i & 1:
                d[pat, i] = (y[pat, i] + 1 + i) % 100
    tau, em, n = O.accept_greedy(d, y)
    for pat in range(1 << K):
        t = K if pat == 0 else (pat & -pat).bit_length() - 1
        assert tau[pat] == t
        assert n[pat] == t + 1
        assert em[pat, :t + 1].tolist() == y[pat, :t + 1].tolist()
        assert (em[pat, t + 1:] == -1).all()


def test_greedy_chain_reproduces_target_stream():
    """Lossless greedy: the concatenated emission equals the target's own
    greedy stream whatever the drafts are."""
    rng = np.random.default_rng(12)
    Y = rng.integers(0, 1000, size=400)
    pos, out = 0, []
    while pos + 17 <= len(Y):
        d = Y[pos:pos + 16].copy()
        bad = rng.random(16) < 0.2
        d[bad] = (d[bad] + 1) % 1000
        tau, em, n = O.accept_greedy(d[None], Y[None, pos:pos + 17])
        out.extend(em[0, :n[0]].tolist())
        pos += int(n[0])
    assert out == Y[:pos].tolist()
    tau, em, n = O.accept_greedy(Y[None, :16], Y[None, :17])
    assert tau[0] == 16 and n[0] == 17 and em[0].tolist() == Y[:17].tolist()


def test_philox_known_answer_vectors():
    for line in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        w = [int(t, 16) for t in line.split()]
        out = O.philox4x32_10(np.array(w[:4], np.uint64), np.array(w[4:6], np.uint64))
        assert out.tolist() == w[6:10]


def test_uniforms_take_the_four_words_of_one_philox_block():
    """R12's index mapping: the uniforms of v = 4g .. 4g + 3 (seed, round, b,
    i, stream) are the four output words of the Philox block at counter
    (g, i | stream << 16, b, round), key (seed lo, seed hi): checked on the
    published known-answer vectors."""
    for line in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        w = [int(t, 16) for t in line.split()]
        c0, c1, c2, c3, k0, k1 = w[:6]
        seed = k0 | (k1 << 32)
        v = 4 * c0 + np.arange(4, dtype=np.uint64)
        u = O.rng_uniform(seed, c3, c2, c1 & 0xFFFF, c1 >> 16, v)
        np.testing.assert_array_equal(u, O.uniform_from_u32(np.array(w[6:10], np.uint64)))


def test_uniform_is_open_interval_and_fp32_exact():
    x = np.array([0, 1, 511, 512, 0xFFFFFFFF], np.uint64)
    u = O.uniform_from_u32(x)
    assert u[0] == 2.0 ** -24 and u[-1] == 1 - 2.0 ** -24
    assert u[1] == u[0] and u[3] > u[2]
    np.testing.assert_array_equal(u.astype(np.float32).astype(np.float64), u)


def test_exponential_race_frequencies_chi_square():
    V = 8
    rng = np.random.default_rng(13)
    p = rng.dirichlet(np.ones(V))
    N = 400_000
    _, em = O.accept_stochastic_trials(p[None], None, np.zeros((N, 0), int), seed=5, rnd=1)
    counts = np.bincount(em[:, 0], minlength=V)
    stat, pval = scipy.stats.chisquare(counts, N * p)
    assert pval > 1e-3, (counts, N * p)


def _stream_trials(p_pos, q_pos, n_trials, n_tokens, K, point_mass, seed):
    """Run rounds for n_trials independent streams until each has n_tokens.

    Target at stream position j: p_pos[j]; drafts: sampled from q_pos[j] (or
    the argmax of q_pos[j] with the point-mass q).  Returns [N, n_tokens]."""
    N = n_trials
    V = p_pos.shape[1]
    rng = np.random.default_rng(seed)
    pos = np.zeros(N, int)
    toks = np.full((N, n_tokens), -1)
    step = 0
    while (pos < n_tokens).any():
        for s in np.unique(pos[pos < n_tokens]):
            idx = np.flatnonzero(pos == s)
            rows_p = p_pos[s:s + K + 1]
            rows_q = q_pos[s:s + K]
            if point_mass:
                d = np.broadcast_to(np.argmax(rows_q, axis=1), (idx.size, K)).copy()
                qarg = None
            else:
                cum = np.cumsum(rows_q, axis=1)
                d = (rng.random((idx.size, K, 1)) > cum[None]).sum(-1)
                d = np.minimum(d, V - 1)
                qarg = rows_q
            tau, em = O.accept_stochastic_trials(rows_p, qarg, d, seed=seed, rnd=1000 + step)
            # trials of this group use RNG sequence ids 0..|idx|-1 at step `step`;
            # distinct steps give independent draws
            for j in range(K + 1):
                has = tau >= j
                tgt = pos[idx] + j
                ok = has & (tgt < n_tokens)
                toks[idx[ok], tgt[ok]] = em[ok, j]
            pos[idx] += tau + 1
            step += 1
    return toks


@pytest.mark.parametrize("point_mass", [False, True])
def test_lossless_theorem_monte_carlo(point_mass):
    """The emitted stream is distributed exactly as the target's (P1 'Exact
    Lossless'; P3 'the output distribution is the target's, exactly').
    vocab 8, K = 4, position-dependent target and draft distributions."""
    V, K, n_tok = 8, 4, 3
    rng = np.random.default_rng(14)
    P = rng.dirichlet(np.ones(V), size=n_tok + K + 1)
    Q = rng.dirichlet(np.ones(V) * 0.7, size=n_tok + K + 1)
    N = 300_000
    toks = _stream_trials(P, Q, N, n_tok, K, point_mass, seed=21 + point_mass)
    for j in range(n_tok):
        cnt = np.bincount(toks[:, j], minlength=V)
        _, pval = scipy.stats.chisquare(cnt, N * P[j])
        assert pval > 1e-3, (j, cnt / N, P[j])
    cells = toks[:, 0] * V + toks[:, 1]
    cnt = np.bincount(cells, minlength=V * V)
    expect = N * np.outer(P[0], P[1]).ravel()
    _, pval = scipy.stats.chisquare(cnt, expect)
    assert pval > 1e-3
    tv = 0.5 * np.abs(cnt / N - expect / N).sum()
    assert tv < 3 * np.sqrt(V * V / N)


def test_stochastic_accept_special_cases():
    V, K = 6, 4
    rng = np.random.default_rng(15)
    z = rng.standard_normal((3, K + 1, V))
    d = rng.integers(0, V, size=(3, K))
    # q = p: the ratio is 1 and every draft is accepted
    q = np.stack([O.softmax(z[:, i]) for i in range(K)], axis=1)
    tau, em, n = O.accept_stochastic(z, d, q, 1.0, 3, 0)
    assert (tau == K).all() and (em[:, :K] == d).all()
    # p(d_0) = 0: rejected at once, residual never returns d_0
    z2 = z.copy()
    z2[np.arange(3), 0, d[:, 0]] = -np.inf
    tau, em, n = O.accept_stochastic(z2, d, None, 1.0, 3, 0)
    assert (tau == 0).all() and (em[:, 0] != d[:, 0]).all()
    # temperature -> 0: point-mass stochastic accept equals greedy accept on argmax
    y = np.argmax(z, axis=-1)
    d3 = y[:, :K].copy()
    d3[0, 2] = (d3[0, 2] + 1) % V
    tau_s, em_s, _ = O.accept_stochastic(z, d3, None, 1e-4, 3, 0)
    tau_g, em_g, _ = O.accept_greedy(d3, y)
    np.testing.assert_array_equal(tau_s, tau_g)
    np.testing.assert_array_equal(em_s, em_g)


# ---------------------------------------------------------------- FP8 (e4m3) weights

def test_e4m3_decode_matches_the_library_cast_on_every_code():
    """All 256 codes against PyTorch's float8_e4m3fn -> float32 conversion
    (an independent implementation of the same format)."""
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    ours = O.decode_e4m3(codes)
    assert np.array_equal(np.isnan(lib), np.isnan(ours))
    ok = ~np.isnan(lib)
    np.testing.assert_array_equal(ours[ok], lib[ok])


def test_e4m3_decode_closed_forms():
    d = O.decode_e4m3
    assert d(np.uint8(0x38)) == 1.0            # exponent field 7 = bias: 2^0
    assert d(np.uint8(0xB8)) == -1.0           # sign bit
    assert d(np.uint8(0x7E)) == 448.0          # largest finite: 1.75 * 2^8
    assert d(np.uint8(0x08)) == 2.0 ** -6      # smallest normal
    assert d(np.uint8(0x01)) == 2.0 ** -9      # smallest subnormal: 1/8 * 2^-6
    assert d(np.uint8(0x07)) == 7 * 2.0 ** -9  # largest subnormal
    assert d(np.uint8(0x00)) == 0.0 and d(np.uint8(0x80)) == 0.0
    assert np.isnan(d(np.uint8(0x7F))) and np.isnan(d(np.uint8(0xFF)))
    # positive codes 0..126 are strictly increasing, and negation flips the sign bit
    pos = d(np.arange(127, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)
    np.testing.assert_array_equal(d(np.arange(128, 255, dtype=np.uint8)), -pos)


def test_dequantized_weights_scale_each_output_row():
    """W = diag(s) . decode(codes): a row scale multiplies exactly that
    output feature of x . W^T."""
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 256, size=(5, 7)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38          # no NaN codes
    s = np.array([1.0, 0.5, 2.0, 0.25, 3.0], np.float32)
    w = O.dequantize_weights({"q:w_o.0": codes, "s:w_o.0": s, "g_in.0": np.ones(7, np.float32)})
    assert set(w) == {"w_o.0", "g_in.0"}
    x = rng.standard_normal((3, 7))
    y1 = x @ O.decode_e4m3(codes).T
    np.testing.assert_allclose(x @ w["w_o.0"].T, y1 * s.astype(np.float64), rtol=1e-15, atol=0)


# ---------------------------------------------------------------- training-time block attention

def _train_attn_case(rng, S=3, NB=7, K=4, Hq=4, Hkv=2, dh=8):
    T = rng.integers(5, 30, size=S)
    ctx_k = [rng.standard_normal((t, Hkv, dh)) for t in T]
    ctx_v = [rng.standard_normal((t, Hkv, dh)) for t in T]
    seq = rng.integers(0, S, size=NB)
    ctx_len = np.array([rng.integers(0, T[s] + 1) for s in seq])
    q = rng.standard_normal((NB, K, Hq, dh))
    kb = rng.standard_normal((NB, K, Hkv, dh))
    vb = rng.standard_normal((NB, K, Hkv, dh))
    return q, kb, vb, ctx_k, ctx_v, seq, ctx_len


def test_train_attention_equals_one_dense_masked_softmax():
    """Every block at once as one attention over [all contexts ; all block
    keys] with an explicit 0 / -inf mask (a second formulation: a single
    dense score matrix, mask built from the rule, SciPy's softmax)."""
    rng = np.random.default_rng(21)
    q, kb, vb, ctx_k, ctx_v, seq, ctx_len = _train_attn_case(rng)
    NB, K, Hq, dh = q.shape
    Hkv = kb.shape[2]
    G = Hq // Hkv
    keys = np.concatenate(list(ctx_k) + [kb.reshape(NB * K, Hkv, dh)])
    vals = np.concatenate(list(ctx_v) + [vb.reshape(NB * K, Hkv, dh)])
    off = np.concatenate([[0], np.cumsum([c.shape[0] for c in ctx_k])])
    n_ctx = off[-1]
    mask = np.full((NB * K, keys.shape[0]), -np.inf)
    for j in range(NB):
        rows = slice(j * K, (j + 1) * K)
        mask[rows, off[seq[j]]:off[seq[j]] + ctx_len[j]] = 0.0
        mask[rows, n_ctx + j * K:n_ctx + (j + 1) * K] = 0.0
    qf = q.reshape(NB * K, Hq, dh)
    dense = np.empty_like(qf)
    for h in range(Hq):
        sc = qf[:, h] @ keys[:, h // G].T / math.sqrt(dh) + mask
        dense[:, h] = scipy.special.softmax(sc, axis=1) @ vals[:, h // G]
    got = O.block_attention_train(q, kb, vb, ctx_k, ctx_v, seq, ctx_len)
    np.testing.assert_allclose(got.reshape(NB * K, Hq, dh), dense, rtol=1e-12, atol=1e-12)


def test_train_attention_sees_no_other_block_and_no_later_context():
    rng = np.random.default_rng(22)
    q, kb, vb, ctx_k, ctx_v, seq, ctx_len = _train_attn_case(rng)
    base = O.block_attention_train(q, kb, vb, ctx_k, ctx_v, seq, ctx_len)
    # perturb block 0's own keys: only block 0 changes
    kb2 = kb.copy()
    kb2[0] += 1.0
    o2 = O.block_attention_train(q, kb2, vb, ctx_k, ctx_v, seq, ctx_len)
    assert not np.allclose(o2[0], base[0])
    np.testing.assert_array_equal(o2[1:], base[1:])
    # perturb every context position at or past each block's prefix of its sequence: nothing changes
    for j in range(len(seq)):
        ck = [c.copy() for c in ctx_k]
        cv = [c.copy() for c in ctx_v]
        ck[seq[j]][ctx_len[j]:] += 5.0
        cv[seq[j]][ctx_len[j]:] -= 5.0
        o3 = O.block_attention_train(q, kb, vb, ck, cv, seq, ctx_len)
        np.testing.assert_array_equal(o3[j], base[j])


def test_train_attention_reduces_to_inference_attention_and_own_block():
    """A block whose prefix is the whole context is the inference block
    attention over [context ; block]; an empty prefix attends to its own
    block only; one key and one value make the output that value."""
    rng = np.random.default_rng(23)
    q, kb, vb, ctx_k, ctx_v, seq, ctx_len = _train_attn_case(rng, NB=3)
    seq = np.array([0, 1, 2])
    full = np.array([c.shape[0] for c in ctx_k])
    o = O.block_attention_train(q, kb, vb, ctx_k, ctx_v, seq, full)
    for j in range(3):
        ref = O.attention(q[j], np.concatenate([ctx_k[j], kb[j]]), np.concatenate([ctx_v[j], vb[j]]))
        np.testing.assert_allclose(o[j], ref, rtol=0, atol=0)
    o0 = O.block_attention_train(q, kb, vb, ctx_k, ctx_v, seq, np.zeros(3, int))
    for j in range(3):
        np.testing.assert_allclose(o0[j], O.attention(q[j], kb[j], vb[j]), rtol=0, atol=0)
    # K = 1, no context: softmax over one key is 1, the output is its value
    o1 = O.block_attention_train(q[:, :1], kb[:, :1], vb[:, :1], ctx_k, ctx_v, seq, np.zeros(3, int))
    G = q.shape[2] // kb.shape[2]
    np.testing.assert_allclose(o1[:, 0], np.repeat(vb[:, 0], G, axis=1), rtol=1e-15)

"""Python face of libdflash: the same three calls as the C ABI (inject_kv,
draft_block, accept) on PyTorch-owned device memory.

PyTorch only provides memory and streams here; every step of the hot path
runs in libdflash's kernels.  Weight packing (q|k|v rows, gate|up rows, the
per-layer k|v rows of the inject projection) is a one-time layout step at
construction.
"""
from __future__ import annotations

import ctypes
from typing import Dict, Optional

import torch

from . import _lib

_DTYPES = {"bf16": (_lib.DTYPE_BF16, torch.bfloat16), "f32": (_lib.DTYPE_F32, torch.float32)}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def weights_to_device(np_weights: Dict[str, "object"], dtype: str, device="cuda") -> Dict[str, torch.Tensor]:
    """numpy fp32 arrays (values exact in the target dtype) -> device tensors.
    E4M3 projection weights ("q:<name>" uint8 codes, "s:<name>" fp32 row
    scales) keep their types."""
    tdt = _DTYPES[dtype][1]
    out = {}
    for k, v in np_weights.items():
        t = torch.from_numpy(v).to(device=device)
        out[k] = (t if k.startswith(("q:", "s:")) else t.to(tdt)).contiguous()
    return out


def gemm_bf16(W: torch.Tensor, X: torch.Tensor, splits: int = 1, status: Optional[torch.Tensor] = None,
              X_lo: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The drafter's tensor-core projection alone: returns fp32 partials
    [splits_used, M, N] with out[s] = (X + X_lo) . W^T restricted to split s's
    k-blocks (X_lo: optional second bf16 term of the activations)."""
    L = _lib.lib()
    N, K = W.shape
    M = X.shape[0]
    assert W.dtype == torch.bfloat16 and X.dtype == torch.bfloat16 and X.shape[1] == K
    assert W.is_contiguous() and X.is_contiguous()
    n_kb = (K + 63) // 64
    want = min(splits, n_kb)
    per = (n_kb + want - 1) // want
    used = (n_kb + per - 1) // per
    out = torch.empty((used, M, N), dtype=torch.float32, device=W.device)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=W.device)
    got = ctypes.c_int(0)
    _lib.check(L.dflash_gemm_bf16(_ptr(W), N, K, _ptr(X), _ptr(X_lo), M, _ptr(out), splits, ctypes.byref(got),
                                  _ptr(status), _stream(stream)), "dflash_gemm_bf16")
    assert got.value == used
    return out


def gemm_w8(W: torch.Tensor, w_scale: torch.Tensor, X: torch.Tensor, splits: int = 1,
            status: Optional[torch.Tensor] = None, X_lo: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """gemm_bf16 with E4M3 weights: W uint8 codes [N, K], w_scale fp32 [N];
    out[s] = w_scale * ((X + X_lo) . decode(W)^T over split s's k-blocks).
    Every split but the last owns an even number of 64-wide k-blocks."""
    L = _lib.lib()
    N, K = W.shape
    M = X.shape[0]
    assert W.dtype == torch.uint8 and w_scale.dtype == torch.float32 and w_scale.numel() == N
    assert X.dtype == torch.bfloat16 and X.shape[1] == K and W.is_contiguous() and X.is_contiguous()
    n_kb = (K + 63) // 64
    want = min(splits, n_kb)
    per = (n_kb + want - 1) // want
    per += per & 1                      # whole pipeline stages (two k-blocks) per split
    used = (n_kb + per - 1) // per
    out = torch.empty((used, M, N), dtype=torch.float32, device=W.device)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=W.device)
    got = ctypes.c_int(0)
    _lib.check(L.dflash_gemm_w8(_ptr(W), _ptr(w_scale), N, K, _ptr(X), _ptr(X_lo), M, _ptr(out), splits,
                                ctypes.byref(got), _ptr(status), _stream(stream)), "dflash_gemm_w8")
    assert got.value == used
    return out


def pack_gate_up(w_gate: torch.Tensor, w_up: torch.Tensor) -> torch.Tensor:
    """[128 * ceil(F/64), d]: per group of 64 features, the 64 gate rows then
    the 64 matching up rows (the last group zero-padded), so that one 128-row
    projection tile holds both halves of its SwiGLU."""
    F, d = w_gate.shape
    G = -(-F // 64)
    pad = G * 64 - F
    g = torch.cat([w_gate, w_gate.new_zeros(pad, d)]) if pad else w_gate
    u = torch.cat([w_up, w_up.new_zeros(pad, d)]) if pad else w_up
    return torch.stack([g.reshape(G, 64, d), u.reshape(G, 64, d)], 1).reshape(G * 128, d)


class RoundGraph:
    """A recorded round (dflash_graph_end); launch() replays it."""

    def __init__(self, L, handle: ctypes.c_void_p):
        self.L, self.handle = L, handle

    def launch(self, stream=None) -> None:
        _lib.check(self.L.dflash_graph_launch(self.handle, _stream(stream)), "dflash_graph_launch")

    def close(self) -> None:
        if getattr(self, "handle", None):
            self.L.dflash_graph_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Drafter:
    """One libdflash context plus the device buffers it borrows.

    shape: any object with the attributes n_layers, hidden, n_q_heads,
    n_kv_heads, head_dim, ffn, vocab, mask_id, n_taps, tap_width, rope_theta,
    rms_eps, dtype ("bf16" | "f32").
    weights: device tensors keyed w_fc, g_fc, embed, g_final, w_lm and per
    layer l: w_q.l, w_k.l, w_v.l, w_o.l, w_gate.l, w_up.l, w_down.l, g_in.l,
    g_post.l (matrices [out, in]).
    """

    def __init__(self, shape, weights: Dict[str, torch.Tensor], *, max_batch: int, max_pages_per_seq: int,
                 n_pages: int, max_rows: int = 17, max_inject_rows: Optional[int] = None,
                 key_offset: Optional[torch.Tensor] = None, device: str = "cuda"):
        self.L = _lib.lib()
        dcode, tdt = _DTYPES[shape.dtype]
        w8 = "q:w_lm" in weights  # E4M3 projection weights with per-row scales
        if w8:
            assert shape.dtype == "bf16"
            dcode = _lib.DTYPE_BF16_W8
        self.w8 = w8
        self.tdtype = tdt
        self.shape = shape
        self.device = torch.device(device)
        cfg = _lib.DflashConfig()
        for f in ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab", "mask_id",
                  "n_taps", "tap_width"):
            setattr(cfg, f, int(getattr(shape, f)))
        cfg.block_k = 16
        cfg.page_size = 16
        cfg.max_batch = max_batch
        cfg.max_pages_per_seq = max_pages_per_seq
        cfg.n_pages = n_pages
        cfg.max_rows = max_rows
        cfg.max_inject_rows = max_inject_rows if max_inject_rows is not None else max_batch * max_rows
        cfg.rope_theta = float(shape.rope_theta)
        cfg.rms_eps = float(shape.rms_eps)
        cfg.dtype = dcode
        self.cfg = cfg
        ws = self.L.dflash_workspace_size(ctypes.byref(cfg))
        pool = self.L.dflash_kv_pool_size(ctypes.byref(cfg))
        if ws == 0 or pool == 0:
            raise _lib.DflashError(2, "config rejected")
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=self.device)
        self.kv_pool = torch.empty(pool, dtype=torch.uint8, device=self.device)
        self.page_table = torch.full((max_batch, max_pages_per_seq), -1, dtype=torch.int32, device=self.device)
        self.seq_len = torch.zeros(max_batch, dtype=torch.int32, device=self.device)

        nl = shape.n_layers
        w = weights
        self._keep = []

        def keep(t, dt=tdt):
            t = t.to(device=self.device, dtype=dt).contiguous()
            self._keep.append(t)
            return t

        # projections: values (bf16 / fp32) or, for E4M3 weights, codes; their
        # row scales are packed with the same row order
        pre = "q:" if w8 else ""
        wdt = torch.uint8 if w8 else tdt

        def pw(name):
            return w[pre + name]

        def ps(name):
            return w["s:" + name].reshape(-1, 1)

        w_qkv = [keep(torch.cat([pw(f"w_q.{l}"), pw(f"w_k.{l}"), pw(f"w_v.{l}")], 0), wdt) for l in range(nl)]
        w_gu = [keep(pack_gate_up(pw(f"w_gate.{l}"), pw(f"w_up.{l}")), wdt) for l in range(nl)]
        w_kv = keep(torch.cat([torch.cat([pw(f"w_k.{l}"), pw(f"w_v.{l}")], 0) for l in range(nl)], 0), wdt)
        singles = {k: keep(w[k]) for k in ("g_fc", "embed", "g_final")}
        singles.update({k: keep(pw(k), wdt) for k in ("w_fc", "w_lm")})
        w_o = [keep(pw(f"w_o.{l}"), wdt) for l in range(nl)]
        w_dn = [keep(pw(f"w_down.{l}"), wdt) for l in range(nl)]
        g_in = [keep(w[f"g_in.{l}"]) for l in range(nl)]
        g_post = [keep(w[f"g_post.{l}"]) for l in range(nl)]
        if w8:
            f32 = torch.float32
            s_qkv = [keep(torch.cat([ps(f"w_q.{l}"), ps(f"w_k.{l}"), ps(f"w_v.{l}")], 0).reshape(-1), f32)
                     for l in range(nl)]
            s_gu = [keep(pack_gate_up(ps(f"w_gate.{l}"), ps(f"w_up.{l}")).reshape(-1), f32) for l in range(nl)]
            s_kv = keep(torch.cat([torch.cat([ps(f"w_k.{l}"), ps(f"w_v.{l}")], 0) for l in range(nl)], 0).reshape(-1),
                        f32)
            s_fc, s_lm = keep(w["s:w_fc"], f32), keep(w["s:w_lm"], f32)
            s_o = [keep(w[f"s:w_o.{l}"], f32) for l in range(nl)]
            s_dn = [keep(w[f"s:w_down.{l}"], f32) for l in range(nl)]
        self.key_offset = None
        if key_offset is not None:
            self.key_offset = key_offset.to(device=self.device, dtype=torch.float32).contiguous()

        def arr(ts):
            a = (ctypes.c_void_p * nl)(*[t.data_ptr() for t in ts])
            self._keep.append(a)
            return ctypes.cast(a, ctypes.POINTER(ctypes.c_void_p))

        wt = _lib.DflashWeights()
        wt.w_fc = singles["w_fc"].data_ptr()
        wt.g_fc = singles["g_fc"].data_ptr()
        wt.embed = singles["embed"].data_ptr()
        wt.g_final = singles["g_final"].data_ptr()
        wt.w_lm = singles["w_lm"].data_ptr()
        wt.w_kv_inject = w_kv.data_ptr()
        wt.key_offset = None if self.key_offset is None else self.key_offset.data_ptr()
        wt.w_qkv, wt.w_o, wt.w_gu, wt.w_down = arr(w_qkv), arr(w_o), arr(w_gu), arr(w_dn)
        wt.g_in, wt.g_post = arr(g_in), arr(g_post)
        if w8:
            wt.s_fc, wt.s_lm, wt.s_kv_inject = s_fc.data_ptr(), s_lm.data_ptr(), s_kv.data_ptr()
            wt.s_qkv, wt.s_o, wt.s_gu, wt.s_down = arr(s_qkv), arr(s_o), arr(s_gu), arr(s_dn)
        self._wt = wt
        ctx = ctypes.c_void_p()
        _lib.check(self.L.dflash_create(ctypes.byref(cfg), ctypes.byref(wt), _ptr(self.kv_pool), pool,
                                        _ptr(self.page_table), _ptr(self.seq_len), _ptr(self.workspace), ws,
                                        ctypes.byref(ctx)), "dflash_create")
        self.ctx = ctx

    # ------------------------------------------------------------------ cache views
    def pool_kv(self):
        """(K, V) views of the pool: [L, n_pages + max_batch, Hkv, 16, head_dim],
        fp16 for bf16 workloads and fp32 for fp32 ones.  Pages n_pages + b hold
        sequence b's draft-block keys and values of the latest pass."""
        s, c = self.shape, self.cfg
        pages = c.n_pages + c.max_batch
        n = s.n_layers * pages * s.n_kv_heads * 16 * s.head_dim
        flat = self.kv_pool.view(torch.float16 if s.dtype == "bf16" else torch.float32)
        shp = (s.n_layers, pages, s.n_kv_heads, 16, s.head_dim)
        return flat[:n].view(shp), flat[n:2 * n].view(shp)

    # ------------------------------------------------------------------ the ABI calls
    def inject_kv(self, feats: torch.Tensor, n_rows: torch.Tensor, first_seq: int = 0, stream=None) -> None:
        """feats [B, max_rows, n_taps*tap_width] (config dtype), n_rows int32 [B] on the device."""
        B, max_rows = feats.shape[0], feats.shape[1]
        assert feats.is_contiguous() and feats.dtype == self.tdtype and n_rows.dtype == torch.int32
        _lib.check(self.L.dflash_inject_kv(self.ctx, _ptr(feats), _ptr(n_rows), first_seq, B, max_rows,
                                           _stream(stream)), "dflash_inject_kv")

    def draft_block(self, B: int, S: int = 1, tokens: Optional[torch.Tensor] = None,
                    conf: Optional[torch.Tensor] = None, logits: Optional[torch.Tensor] = None,
                    committed: Optional[torch.Tensor] = None, want_conf: bool = True, stream=None):
        """Returns (tokens int32 [B,16], conf fp32 [B,16] or None, logits or None, committed or None)."""
        if tokens is None:
            tokens = torch.empty((B, 16), dtype=torch.int32, device=self.device)
        if conf is None and want_conf:
            conf = torch.empty((B, 16), dtype=torch.float32, device=self.device)
        _lib.check(self.L.dflash_draft_block(self.ctx, B, S, _ptr(tokens), _ptr(conf), _ptr(logits),
                                             _ptr(committed), _stream(stream)), "dflash_draft_block")
        return tokens, conf, logits, committed

    def accept(self, mode: int, draft_tokens: torch.Tensor, target_tokens: Optional[torch.Tensor] = None,
               target_logits: Optional[torch.Tensor] = None, draft_probs: Optional[torch.Tensor] = None,
               temperature: float = 1.0, seed: int = 0, round: int = 0, out=None, stream=None):
        """mode 0 greedy (target_tokens [B,17]), 1 stochastic (target_logits [B,17,V] fp32).
        Returns (accept_len [B], emitted [B,17], n_emit [B]) int32."""
        B = draft_tokens.shape[0]
        if out is None:
            out = (torch.empty(B, dtype=torch.int32, device=self.device),
                   torch.empty((B, 17), dtype=torch.int32, device=self.device),
                   torch.empty(B, dtype=torch.int32, device=self.device))
        tau, emitted, n_emit = out
        _lib.check(self.L.dflash_accept(self.ctx, mode, B, _ptr(draft_tokens), _ptr(target_tokens),
                                        _ptr(target_logits), _ptr(draft_probs), float(temperature),
                                        int(seed), int(round), _ptr(tau), _ptr(emitted), _ptr(n_emit),
                                        _stream(stream)), "dflash_accept")
        return tau, emitted, n_emit

    def block_attention(self, layer: int, seq: torch.Tensor, ctx_len: torch.Tensor, q: torch.Tensor,
                        k_blk: torch.Tensor, v_blk: torch.Tensor, out: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
        """Training-time block attention: NB blocks; block j sees sequence seq[j]'s
        context prefix of ctx_len[j] positions and its own 16 keys.  q fp16
        [NB, 16, Hq, dh]; k_blk, v_blk fp16 [NB, 16, Hkv, dh]; returns fp32 [NB, 16, Hq, dh]."""
        NB = q.shape[0]
        assert q.dtype == torch.float16 and k_blk.dtype == torch.float16 and v_blk.dtype == torch.float16
        assert q.is_contiguous() and k_blk.is_contiguous() and v_blk.is_contiguous()
        assert seq.dtype == torch.int32 and ctx_len.dtype == torch.int32
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=self.device)
        _lib.check(self.L.dflash_block_attention(self.ctx, layer, NB, _ptr(seq), _ptr(ctx_len), _ptr(q), _ptr(k_blk),
                                                 _ptr(v_blk), _ptr(out), _stream(stream)), "dflash_block_attention")
        return out

    def reset(self, stream=None) -> None:
        """Empty every sequence and clear the device status word."""
        _lib.check(self.L.dflash_reset(self.ctx, _stream(stream)), "dflash_reset")

    def release(self, b: int, stream=None) -> None:
        _lib.check(self.L.dflash_release(self.ctx, b, _stream(stream)), "dflash_release")

    def truncate(self, b: int, new_len: int, stream=None) -> None:
        """Shorten sequence b to new_len tokens; freed pages go to the free-list tail."""
        _lib.check(self.L.dflash_truncate(self.ctx, b, new_len, _stream(stream)), "dflash_truncate")

    # ------------------------------------------------------------------ host-free rounds
    def graph_begin(self, stream=None) -> None:
        """Start recording the stream (not the legacy default stream): calls on it,
        this library's and torch's, are recorded until graph_end."""
        _lib.check(self.L.dflash_graph_begin(self.ctx, _stream(stream)), "dflash_graph_begin")

    def graph_end(self, stream=None) -> "RoundGraph":
        """Stop recording; the recorded calls as a replayable graph."""
        g = ctypes.c_void_p()
        _lib.check(self.L.dflash_graph_end(self.ctx, _stream(stream), ctypes.byref(g)), "dflash_graph_end")
        return RoundGraph(self.L, g)

    def profile(self, enable: bool) -> None:
        """Bracket every launch with CUDA events (read with profile_read)."""
        _lib.check(self.L.dflash_profile_enable(self.ctx, 1 if enable else 0), "dflash_profile_enable")

    def profile_read(self, stream=None) -> Dict[str, tuple]:
        """{class: (total ms, launches)} since the last read; synchronises."""
        n = len(_lib.PROF_CLASSES)
        ms = (ctypes.c_float * n)()
        cnt = (ctypes.c_int * n)()
        _lib.check(self.L.dflash_profile_read(self.ctx, ms, cnt, _stream(stream)), "dflash_profile_read")
        return {k: (float(ms[i]), int(cnt[i])) for i, k in enumerate(_lib.PROF_CLASSES)}

    def device_status(self, stream=None) -> int:
        v = ctypes.c_int(0)
        _lib.check(self.L.dflash_get_status(self.ctx, ctypes.byref(v), _stream(stream)), "dflash_get_status")
        return v.value

    def close(self) -> None:
        if getattr(self, "ctx", None):
            self.L.dflash_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

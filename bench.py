#!/usr/bin/env python
"""Draft tokens/sec of the DFlash block-draft hot path on GB300.

One step = one speculative round on the GPU: KV-inject the tau+1 rows the
previous round accepted, draft a K = 16 block (S passes), and accept against
the synthetic target.  Default workload (the largest that fits one GPU): the
gpt-oss-120b-shaped drafter (3 layers, hidden 2880, 64/8 heads of 64, SwiGLU
2880, vocab 201088, 3 taps of 2880), 128 sequences with contexts uniform in
[1024, 8192], S = 2 confidence-ordered commits, stochastic rejection-sampling
accept at temperature 1 against target logits = the committing pass's draft
logits + N(0, 1) noise; random-init N(0, 0.02) bf16 weights, N(0, 1)
features (seeded, synthetic).  The other workloads (tiny fp32, Qwen3-8B-
shaped at batch 1 with bf16 and FP8 weights, the 32-sequence serving batch,
4 x 32k long context) are timed in the same run and reported under
"per_config".

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs its own replica (the path shards by
sequence; no collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

K_BLOCK = 16
METRIC = "draft tokens/sec (K=16 block pass incl. KV inject+accept); % HBM/TC roofline"
UNIT = "draft tok/s"


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="c5")
    ap.add_argument("--per-config", default="c1,c2,c2w8,c3,c4",
                    help="workloads timed after the headline one (comma list; empty: none)")
    ap.add_argument("--per-config-steps", type=int, default=100)
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-rounds", type=int, default=4, help="oracle rounds timed for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay leg")
    ap.add_argument("--sweep", action="store_true",
                    help="draft-cost sweeps (1/3/5 draft layers; projections on 1 vs 16 rows), JSON line per item")
    ap.add_argument("--reset-every", type=int, default=0,
                    help="roll each sequence back to its prompt length every N rounds "
                         "(0: the workload's stated round count)")
    ap.add_argument("--kernel", choices=["gemm", "train_attn"], default=None,
                    help="time one kernel alone on the workload's shapes (small case for profilers)")
    ap.add_argument("--small", action="store_true",
                    help="profiler case: the workload's layer shapes with 1 draft layer and a 16384 vocab")
    return ap.parse_args(argv)


# --------------------------------------------------------------------------- helpers

def load_peaks(sustained: bool = True):
    """(HBM GB/s, dense bf16 TFLOP/s, "measured" | "fallback").  The tensor
    figure is the sustained one (under the power cap) for kernels timed
    inside a seconds-long loop, the burst one for a kernel timed alone."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        burst = float(d.get("bf16_tflops", 1900.0))
        tc = float(d.get("bf16_tflops_sustained", burst)) if sustained else burst
        return float(d["hbm_gbs"]), tc, "measured"
    return 6800.0, (1700.0 if sustained else 1900.0), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling while a region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.f = None

    def __enter__(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.f is None:
            return None
        self.f.flush()
        rows = []
        for line in open(self.f.name):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5], parts[6], parts[7], parts[8]))
            except ValueError:
                continue
        os.unlink(self.f.name)
        if not rows:
            return None
        sm = [r[0] for r in rows]
        reasons = set()
        for r in rows:
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), r[2:]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return ws, rank, local


def aggregate(tokens: float, ms: float, world: int):
    """Whole-job numbers: tokens summed over ranks, time = max over ranks."""
    if world == 1:
        return tokens, ms
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([tokens], dtype=torch.float64, device=dev)
    m = torch.tensor([ms], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    dist.all_reduce(m, op=dist.ReduceOp.MAX)
    return float(t.item()), float(m.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# Per-launch DRAM traffic of the projection + LM-head launches, measured by
# ncu at full size: (profile file, the sources whose text it was taken on)
GEMM_SOURCES = ("gemm_kernel.cuh", "gemm.cu", "epilogue.cuh", "common.cuh")
TRAFFIC_PROFILES = {
    "c2_qwen3_8b_shaped": ("k_gemm_tc_c2_layer.md", GEMM_SOURCES),
    "c5_gpt_oss_120b_shaped": ("k_gemm_pers_c5_traffic.md", ("gemm_persist.cuh",) + GEMM_SOURCES),
    "c3_serving_batch32": ("gemm_traffic_c3.md", ("gemm_persist.cuh",) + GEMM_SOURCES),
    "c4_long_context_32k": ("gemm_traffic_c4.md", ("gemm_persist.cuh",) + GEMM_SOURCES),
}


def code_text(src: str) -> str:
    """C/CUDA source without its comments and with whitespace runs collapsed:
    what the fingerprint of a profiled kernel hashes, so that editing a
    comment does not void a capture."""
    import re
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def gemm_traffic(cfg):
    """DRAM bytes per projection / LM-head launch measured by ncu for this
    workload (see the profile file), or None when there is no capture for it
    or the GEMM sources changed since."""
    import hashlib
    if cfg.name not in TRAFFIC_PROFILES:
        return None
    fname, sources = TRAFFIC_PROFILES[cfg.name]
    path = os.path.join(ROOT, "profiles", fname)
    if not os.path.exists(path):
        return None
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, "block_diffusion_speculative_hidden_gb300", "csrc", f)) as fh:
            h.update(code_text(fh.read()).encode())
    fields = {}
    for line in open(path):
        if ":" in line and line.split(":")[0] in ("traffic_per_launch_bytes", "source_fingerprint"):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("source_fingerprint") != h.hexdigest()[:16]:
        return None
    return float(fields["traffic_per_launch_bytes"])


def algorithmic_bytes(cfg):
    """Bytes the hot path must move per round (B sequences), by kernel class.

    Projections: bf16 weights once + activations in (hi+lo bf16, 4 B/elem) +
    fp32 results out; the LM head's logits out where the accept reads them.
    Attention (kv_bytes): the K/V of every layer once.
    Inject: FC and K/V weights + the new rows; accept: tokens only."""
    B, d, F, V, L = cfg.batch, cfg.hidden, cfg.ffn, cfg.vocab, cfg.n_layers
    qd, kvd = cfg.q_dim, cfg.kv_dim
    M = B * K_BLOCK
    w8 = cfg.weight_format == "e4m3"
    wb = 1 if w8 else 2                       # weight bytes per entry (E4M3 codes: 1, plus a 4-byte row scale)

    def wbytes(N, Kd):
        return N * Kd * wb + (4 * N if w8 else 0)

    def proj(N, Kd, m=M):
        return wbytes(N, Kd) + m * Kd * 4 + m * N * 4

    Fp = 64 * -(-F // 64)                     # gate/up rows are packed in groups of 64
    per_layer = proj(qd + 2 * kvd, d) + proj(d, qd) + proj(2 * Fp, d) + proj(d, F)
    lm_rows = M + (cfg.s_passes - 1) * (M // 2)  # S = 2: the second LM head runs on the K/2 uncommitted rows
    return {"proj": L * per_layer * cfg.s_passes,
            # stochastic workloads also write the rows' fp32 logits (the accept reads them)
            "lm_head": wbytes(V, d) * cfg.s_passes + lm_rows * d * 4
                       + (lm_rows * V * 4 if cfg.accept == "stochastic" else 0),
            "inject_weights": wbytes(d, cfg.feat_dim) + wbytes(2 * L * kvd, d)}


def kv_bytes(cfg, ctx_len):
    """K and V of every layer read once per pass: fp16 for bf16 workloads, fp32 otherwise."""
    e = 2 if cfg.dtype == "bf16" else 4
    return cfg.n_layers * 2 * cfg.kv_dim * e * (ctx_len + K_BLOCK) * cfg.batch * cfg.s_passes


# --------------------------------------------------------------------------- GPU arm

def reset_period(cfg, reset_every: int) -> int:
    """Rounds between roll-backs to the prompt: the workload's stated round
    count (c3: 32, c4: 64, the others 8) unless given."""
    return reset_every if reset_every > 0 else cfg.rounds


class Workload:
    """The drafter on the GPU with its prompt injected and every round's
    inputs (new feature rows, synthetic target coins or noise) already in HBM.

    Stochastic workloads: the synthetic target's logits are the committing
    pass's draft logits (the draft call's logits output: pass-1 rows on the
    committed positions, pass-2 rows elsewhere) plus N(0, 1) noise, and the
    bonus row is noise alone; the noise comes from n_noise device-resident
    draws (torch's seeded generator, used cyclically)."""

    def __init__(self, cfg, rounds: int, rank: int, device, reset_every: int = 0, n_noise: int = 4):
        import torch
        from block_diffusion_speculative_hidden_gb300 import Drafter, weights_to_device
        self.torch = torch
        self.cfg = cfg
        self.dev = device
        B, F = cfg.batch, cfg.feat_dim
        t0 = time.time()
        self.w_np = synth.make_weights(cfg)
        self.t_gen = time.time() - t0
        self.lens = synth.make_ctx_lens(cfg)
        chunk = min(1024, int(self.lens.max()))
        self.period = reset_period(cfg, reset_every)
        max_ctx = int(self.lens.max()) + 17 * (self.period + 2)
        self.mpps = -(-max_ctx // 16) + 2
        n_pages = B * self.mpps + 8
        koff = synth.make_key_offsets(cfg)
        self.dr = Drafter(cfg, weights_to_device(self.w_np, cfg.dtype, device), max_batch=B,
                          max_pages_per_seq=self.mpps, n_pages=n_pages, max_rows=max(17, chunk),
                          max_inject_rows=max(B * 17, chunk),
                          key_offset=None if koff is None else torch.from_numpy(koff), device=str(device))
        tdt = self.dr.tdtype
        # prompt: every chunk staged on the device first, then the injects
        # timed alone (the prefill is reported apart from the rounds)
        calls = []
        for b in range(B):
            feats = synth.make_prefill_features(cfg, b, int(self.lens[b]))
            for s0 in range(0, feats.shape[0], chunk):
                part = feats[s0:s0 + chunk]
                buf = torch.zeros((1, chunk, F), dtype=tdt, device=device)
                buf[0, :part.shape[0]] = torch.from_numpy(part).to(device).to(tdt)
                calls.append((buf, torch.tensor([part.shape[0]], dtype=torch.int32, device=device), b))
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for buf, n, b in calls:
            self.dr.inject_kv(buf, n, first_seq=b)
        e1.record()
        torch.cuda.synchronize(device)
        self.prefill = {"ms": e0.elapsed_time(e1), "rows": int(self.lens.sum()), "calls": len(calls),
                        "rows_per_call": chunk}
        del calls
        assert self.dr.device_status() == 0
        # per-round inputs, resident
        self.rounds = rounds
        self.stochastic = cfg.accept == "stochastic"
        if self.stochastic:
            V = cfg.vocab
            self.zd = torch.empty((B, K_BLOCK, V), dtype=torch.float32, device=device)
            self.zt = torch.empty((B, K_BLOCK + 1, V), dtype=torch.float32, device=device)
            gen = torch.Generator(device=device).manual_seed(cfg.seed * 1000 + rank)
            self.noise = [torch.randn((B, K_BLOCK + 1, V), generator=gen, device=device) for _ in range(n_noise)]
        feats = np.zeros((rounds, B, 17, F), np.float32)
        match = np.zeros((rounds, B, 17), bool)
        rand = np.zeros((rounds, B, 17), np.int32)
        for r in range(rounds):
            for b in range(B):
                feats[r, b] = synth.make_round_features(cfg, 1000 * rank + r, b, 17)
            match[r], rand[r] = synth.make_target_match(cfg, 1000 * rank + r, B, K_BLOCK)
        self.h_feats = feats
        self.h_match, self.h_rand = match, rand
        self.feats = torch.from_numpy(feats).to(device).to(tdt)
        self.match = torch.from_numpy(match).to(device)
        self.y = torch.from_numpy(rand).to(device)          # bonus column stays random
        self.n_rows = torch.ones(B, dtype=torch.int32, device=device)
        self.tok = torch.empty((B, K_BLOCK), dtype=torch.int32, device=device)
        self.conf = torch.empty((B, K_BLOCK), dtype=torch.float32, device=device)
        self.acc = (torch.empty(B, dtype=torch.int32, device=device),
                    torch.empty((B, 17), dtype=torch.int32, device=device),
                    torch.empty(B, dtype=torch.int32, device=device))
        self.tau_sum = torch.zeros(B, dtype=torch.int64, device=device)
        self.target_events = None    # list of event pairs while the target's ops are timed

    def step(self, r: int, feats=None, y=None, match=None):
        """One round: inject tau+1 rows, draft, synthetic target, accept."""
        torch = self.torch
        cfg = self.cfg
        r %= self.rounds
        self.dr.inject_kv(self.feats[r] if feats is None else feats, self.n_rows)
        if self.stochastic:
            self.dr.draft_block(cfg.batch, cfg.s_passes, tokens=self.tok, conf=self.conf, logits=self.zd)
            # synthetic target verify: its logits are the draft logits plus noise
            nz = self.noise[r % len(self.noise)]
            ev = None
            if self.target_events is not None:
                ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                ev[0].record()
            torch.add(self.zd, nz[:, :K_BLOCK], out=self.zt[:, :K_BLOCK])
            self.zt[:, K_BLOCK].copy_(nz[:, K_BLOCK])
            if ev is not None:
                ev[1].record()
                self.target_events.append(ev)
            tau, em, n = self.dr.accept(1, self.tok, target_logits=self.zt, temperature=cfg.temperature,
                                        seed=cfg.seed, round=r, out=self.acc)
            self.n_rows.copy_(n)
            self.tau_sum += tau
            return
        self.dr.draft_block(cfg.batch, cfg.s_passes, tokens=self.tok, conf=self.conf)
        yy = self.y[r] if y is None else y
        mm = self.match[r] if match is None else match
        # synthetic target verify: y_i = d_i where the round's coin matched
        ev = None
        if self.target_events is not None:
            ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            ev[0].record()
        torch.where(mm[:, :K_BLOCK], self.tok, yy[:, :K_BLOCK], out=yy[:, :K_BLOCK])
        if ev is not None:
            ev[1].record()
            self.target_events.append(ev)
        tau, em, n = self.dr.accept(0, self.tok, target_tokens=yy, out=self.acc)
        self.n_rows.copy_(n)
        self.tau_sum += tau

    def maybe_reset(self, r: int):
        """After round r: roll every sequence back to its prompt at the end of
        each period of the workload's stated round count."""
        every = self.period
        if r % every == every - 1:
            for b in range(self.cfg.batch):
                self.dr.truncate(b, int(self.lens[b]))


def run_ours(args, cfg, world, rank, local, steps=None, legs=True):
    """Warm-up, then timed region A (the number: one CUDA-event pair around
    `steps` rounds, clocks sampled meanwhile) and timed region B (the same
    rounds with per-launch events per kernel class, and the synthetic
    target's ops timed on their own); with legs, the end-to-end and graph
    replay legs.  Returns the figures and the workload."""
    import torch
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    steps = args.steps if steps is None else steps
    period = reset_period(cfg, args.reset_every)
    rounds = min(64, max(16, 2 * period))
    wl = Workload(cfg, rounds, rank, device, reset_every=args.reset_every)
    stream = torch.cuda.current_stream(device)
    B = cfg.batch

    def loop(n, start):
        for i in range(n):
            wl.step(start + i)
            wl.maybe_reset(start + i)

    # warm-up
    loop(args.warmup, 0)
    torch.cuda.synchronize(device)
    assert wl.dr.device_status() == 0
    wl.tau_sum.zero_()
    # ---- timed region A: the number
    barrier(world)
    torch.cuda.synchronize(device)
    clk = ClockSampler(local)
    with clk:
        time.sleep(0.3)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        # an NVTX range marks the timed rounds (a profiler can capture them alone)
        torch.cuda.nvtx.range_push("timed_rounds")
        e0.record(stream)
        loop(steps, args.warmup)
        e1.record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1)
    barrier(world)
    mean_tau = float(wl.tau_sum.sum().item()) / (steps * B)
    tokens, ms_max = aggregate(float(steps * B * K_BLOCK), ms, world)
    value = tokens / (ms_max / 1e3)
    clocks = clk.summary()
    # ---- timed region B: same loop with per-launch events (kernel classes)
    wl.dr.profile(True)
    wl.dr.profile_read()
    wl.target_events = []
    torch.cuda.synchronize(device)
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    loop(steps, args.warmup + steps)
    f1.record(stream)
    prof = wl.dr.profile_read()
    ms_b = f0.elapsed_time(f1)
    wl.dr.profile(False)
    target_ms = sum(a.elapsed_time(b) for a, b in wl.target_events)
    wl.target_events = None
    assert wl.dr.device_status() == 0
    launches_per_step = sum(v[1] for v in prof.values()) / steps
    # ---- e2e: host buffers through the public API, copies inside the region
    e2e = run_e2e(wl, args, device) if legs and args.e2e_steps > 0 else None
    graph = None if (args.no_graph or not legs) else run_graph(wl, args, device)
    return dict(value=value, ms=ms_max, tokens=tokens, mean_tau=mean_tau, clocks=clocks, prof=prof, ms_b=ms_b,
                target_ms=target_ms, launches_per_step=launches_per_step, e2e=e2e, graph=graph, wl=wl,
                lens=wl.lens, steps=steps, period=wl.period)


def run_graph(wl, args, device):
    """The same rounds replayed as CUDA graphs (dflash_graph_*): one recording
    per round slot r mod rounds (inject, draft, the synthetic target's
    verify, accept, bookkeeping and the periodic rollback, exactly the eager
    round), then the timed region launches one graph per round."""
    import torch
    gs = torch.cuda.Stream(device)
    torch.cuda.synchronize(device)
    graphs = []
    with torch.cuda.stream(gs):
        for r in range(wl.rounds):
            wl.dr.graph_begin(stream=gs)
            wl.step(r)
            wl.maybe_reset(r)
            graphs.append(wl.dr.graph_end(stream=gs))
    n = wl.rounds
    # start from the prompts, so that the rollback schedule of the recorded
    # rounds (round index mod reset_every) applies from replay 0
    with torch.cuda.stream(gs):
        for b in range(wl.cfg.batch):
            wl.dr.truncate(b, int(wl.lens[b]), stream=gs)
    for i in range(args.warmup):
        graphs[i % n].launch(stream=gs)
    gs.synchronize()
    wl.tau_sum.zero_()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(gs)
    for i in range(args.steps):
        graphs[(args.warmup + i) % n].launch(stream=gs)
    e1.record(gs)
    gs.synchronize()
    ms = e0.elapsed_time(e1)
    assert wl.dr.device_status() == 0
    tau = float(wl.tau_sum.sum().item()) / (args.steps * wl.cfg.batch)
    for g in graphs:
        g.close()
    return {"value": args.steps * wl.cfg.batch * K_BLOCK / (ms / 1e3), "unit": UNIT,
            "ms_per_step": ms / args.steps, "steps": args.steps, "mean_tau": tau,
            "launch": "one CUDA graph per round (dflash_graph_launch), inputs resident"}


def run_e2e(wl, args, device):
    """Per step: pinned host feature rows and target coins (greedy
    workloads) -> device, the three library calls, drafts + emitted tokens +
    counts -> pinned host, then a stream sync (the caller reads its result).
    A step's inputs are copied on a stream of their own into one of two
    device buffers while the previous step computes (the copy of step i + 1
    is issued before step i's calls; a step waits for its own copy), so
    every step's host-to-device copy is inside the timed region and overlaps
    compute, as a serving loop would do it.  Timed twice: each step's calls
    issued one by one, and each step as one replay of a CUDA graph recorded
    from the same calls and the result copies (dflash_graph_*); the graph
    figure is the e2e value, the other is reported beside it."""
    torch = wl.torch
    cfg = wl.cfg
    B, F = cfg.batch, cfg.feat_dim
    n = args.e2e_steps
    h_feats = torch.from_numpy(wl.h_feats).to(wl.dr.tdtype).pin_memory()
    h_match = torch.from_numpy(wl.h_match).pin_memory()
    h_y = torch.from_numpy(wl.h_rand).pin_memory()
    d_feats = [torch.empty((B, 17, F), dtype=wl.dr.tdtype, device=device) for _ in range(2)]
    d_match = [torch.empty((B, 17), dtype=torch.bool, device=device) for _ in range(2)]
    d_y = [torch.empty((B, 17), dtype=torch.int32, device=device) for _ in range(2)]
    o_tok = torch.empty((B, K_BLOCK), dtype=torch.int32).pin_memory()
    o_em = torch.empty((B, 17), dtype=torch.int32).pin_memory()
    o_n = torch.empty((B,), dtype=torch.int32).pin_memory()
    # stochastic workloads: the synthetic target's noise stays on the device
    # (target-side state); the host supplies the round's feature rows
    h2d = d_feats[0].numel() * d_feats[0].element_size() + (0 if wl.stochastic else d_match[0].numel() + d_y[0].numel() * 4)
    d2h = o_tok.numel() * 4 + o_em.numel() * 4 + o_n.numel() * 4
    gs = torch.cuda.Stream(device)   # the library calls
    cs = torch.cuda.Stream(device)   # the input copies
    copied = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]

    def issue_copy(i):
        """Step i's inputs into the buffer of its round's parity, once the
        step that used that buffer last is done."""
        r = i % wl.rounds
        slot = r % 2
        cs.wait_event(free[slot])
        with torch.cuda.stream(cs):
            d_feats[slot].copy_(h_feats[r], non_blocking=True)
            if not wl.stochastic:
                d_match[slot].copy_(h_match[r], non_blocking=True)
                d_y[slot].copy_(h_y[r], non_blocking=True)
        copied[slot].record(cs)

    def body(r, slot):
        # the calls of round r on buffer `slot`, and the result copies
        wl.step(r, feats=d_feats[slot], y=d_y[slot], match=d_match[slot])
        wl.maybe_reset(r)
        o_tok.copy_(wl.tok, non_blocking=True)
        o_em.copy_(wl.acc[1], non_blocking=True)
        o_n.copy_(wl.acc[2], non_blocking=True)

    def restart():
        # from the prompts, so that the rollback schedule (round index mod
        # reset_every) bounds every sequence's growth
        with torch.cuda.stream(gs):
            for b in range(B):
                wl.dr.truncate(b, int(wl.lens[b]), stream=gs)
        for ev in free:
            ev.record(gs)
        gs.synchronize()

    def timed(run_round):
        restart()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(gs)
        cs.wait_event(e0)  # the first copy starts inside the region too
        issue_copy(0)
        for i in range(n):
            if i + 1 < n:
                issue_copy(i + 1)
            r = i % wl.rounds
            slot = r % 2
            gs.wait_event(copied[slot])
            run_round(r, slot)
            free[slot].record(gs)
            gs.synchronize()
        e1.record(gs)
        gs.synchronize()
        return e0.elapsed_time(e1)

    # a round's buffer is fixed by its index (its parity)
    with torch.cuda.stream(gs):
        ms_eager = timed(body)
        graphs, why = None, None
        if not args.no_graph:
            graphs = []
            try:
                for r in range(wl.rounds):
                    wl.dr.graph_begin(stream=gs)
                    try:
                        body(r, r % 2)
                    finally:
                        g = wl.dr.graph_end(stream=gs)    # ends the recording either way
                    graphs.append(g)
            except Exception as e:                         # a copy the recording refuses: eager only
                why = f"{type(e).__name__}: {e}"[:200]
                graphs = None
                gs.synchronize()
        if graphs is not None:
            ms_graph = timed(lambda r, slot: graphs[r].launch(stream=gs))
            for g in graphs:
                g.close()
    assert wl.dr.device_status() == 0
    ms = ms_graph if graphs is not None else ms_eager
    out = {"value": n * B * K_BLOCK / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
           "d2h_bytes_per_step": int(d2h), "steps": n,
           "calls": ("one CUDA graph replay per step (dflash_graph_launch, result copies inside); each step's "
                     "inputs copied on a second stream under the previous step") if graphs is not None
           else "the three library calls per step; inputs copied on a second stream under the previous step"}
    if graphs is not None:
        out["eager_value"] = n * B * K_BLOCK / (ms_eager / 1e3)
    elif why is not None:
        out["graph_unavailable"] = why
    return out


# --------------------------------------------------------------------------- oracle (CPU)

ORACLE_SEQS = 4  # sequences of a batch the CPU oracle times (sequences are independent)


def oracle_seqs(cfg):
    """The sequences the oracle times: all of a small batch, else a seeded
    sample of ORACLE_SEQS (per-sequence work is independent of the others,
    so the batch's token rate is the sample's)."""
    if cfg.batch <= ORACLE_SEQS:
        return list(range(cfg.batch))
    rng = np.random.default_rng(cfg.seed)
    return sorted(rng.choice(cfg.batch, size=ORACLE_SEQS, replace=False).tolist())


def oracle_rounds(cfg, weights, n_rounds: int, lens, seqs):
    """Time the oracle on rounds of the same workload for sequences `seqs`:
    inject tau+1 rows, draft (S passes), accept (greedy against the synthetic
    target's tokens, or stochastic against its logits = the committing
    pass's draft logits + N(0, 1) noise).  Returns (seconds per round,
    threads, mean tau)."""
    from oracle import dflash_oracle as O
    nb = len(seqs)
    ln = lens[seqs]
    mpps = -(-(int(ln.max()) + 17 * (n_rounds + 2)) // 16) + 1
    dr = O.OracleDrafter(cfg, weights, nb * mpps + 4, mpps, key_offsets=synth.make_key_offsets(cfg), seqs=seqs)
    assert dr.inject([synth.make_prefill_features(cfg, b, int(lens[b])) for b in seqs])
    n_rows = np.ones(nb, np.int64)
    taus = []
    t0 = time.perf_counter()
    for r in range(n_rounds):
        assert dr.inject([synth.make_round_features(cfg, r, b, int(n_rows[j])) for j, b in enumerate(seqs)])
        res = [dr.draft(j) for j in range(nb)]
        d = np.stack([x["tokens"] for x in res]).astype(np.int64)
        if cfg.accept == "stochastic":
            z = np.stack([x["logits"] for x in res])
            zt = np.concatenate([z, np.zeros((nb, 1, cfg.vocab))], 1)
            zt += synth.make_target_logits(cfg, 100 + r, d, cfg.vocab, noise_std=1.0)
            tau, _, n = O.accept_stochastic(zt, d, None, cfg.temperature, cfg.seed, r)
        else:
            y = synth.make_target_tokens(cfg, r, d)
            tau, _, n = O.accept_greedy(d, y)
        n_rows = n
        taus.append(tau.mean())
    dt = (time.perf_counter() - t0) / n_rounds
    return dt, os.cpu_count(), float(np.mean(taus))


def oracle_sample_text(cfg, seqs, rounds):
    part = "all" if len(seqs) == cfg.batch else f"{len(seqs)} seeded of {cfg.batch} (tok/s extrapolated: the per-sequence rate)"
    return (f"{rounds} rounds of {cfg.name}, sequences {part}, NumPy fp64, after an untimed prompt injection")


def cpu_baseline(cfg, args, weights=None):
    w = weights if weights is not None else synth.make_weights(cfg)
    lens = synth.make_ctx_lens(cfg)
    seqs = oracle_seqs(cfg)
    dt, cores, _ = oracle_rounds(cfg, w, args.cpu_rounds, lens, seqs)
    return {"value": len(seqs) * K_BLOCK / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": oracle_sample_text(cfg, seqs, args.cpu_rounds)}


def run_reference(args, cfg, world, rank):
    """The reference arm: the CPU oracle, as it stands, on this workload."""
    if rank != 0:
        return
    w = synth.make_weights(cfg)
    lens = synth.make_ctx_lens(cfg)
    seqs = oracle_seqs(cfg)
    # untimed warm-up rounds, which also size the bounded sample: about a
    # minute of timed oracle work
    warmup = max(1, args.warmup)
    dt1, cores, _ = oracle_rounds(cfg, w, warmup, lens, seqs)
    steps = max(1, min(args.steps, int(60.0 / max(dt1, 1e-3))))
    dt, cores, mean_tau = oracle_rounds(cfg, w, steps, lens, seqs)
    value = len(seqs) * K_BLOCK / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": steps, "warmup": warmup, "ms_per_step": dt * 1e3 * cfg.batch / len(seqs),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_block(cfg, lens), "mean_tau": mean_tau,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": oracle_sample_text(cfg, seqs, steps) + f" ({args.steps} requested)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_block(cfg, lens):
    """The workload, identical in both arms' lines."""
    ab = algorithmic_bytes(cfg)
    return {"workload": cfg.name, "weights": "e4m3 codes + fp32 row scales" if cfg.weight_format == "e4m3" else cfg.dtype,
            "batch": cfg.batch, "context": [int(lens.min()), int(lens.max())], "block_k": K_BLOCK,
            "s_passes": cfg.s_passes, "draft_layers": cfg.n_layers, "hidden": cfg.hidden,
            "heads": f"{cfg.n_q_heads}/{cfg.n_kv_heads}x{cfg.head_dim}", "ffn": cfg.ffn, "vocab": cfg.vocab,
            "taps": f"{cfg.n_taps}x{cfg.tap_width}", "accept": cfg.accept,
            "temperature": cfg.temperature if cfg.accept == "stochastic" else None,
            "match_prob": cfg.match_prob if cfg.accept == "greedy" else None,
            "rounds_per_prompt": cfg.rounds,
            "l2": "inputs larger than L2: every step streams all drafter weights "
                  f"({(ab['proj'] + ab['lm_head']) / 1e9:.2f} GB) from HBM"}


# --------------------------------------------------------------------------- single kernels

def run_kernel_gemm(args, cfg):
    """The gate/up projection of one draft layer alone: W [2F, d] bf16, the
    workload's B x 16 activation rows as a hi+lo pair, split-K as the
    library sizes it for the draft block (about 1.5 CTAs per SM, at most 8
    splits, at least 4 k-blocks a split)."""
    import torch
    from block_diffusion_speculative_hidden_gb300 import gemm_bf16
    N, K, M = 2 * cfg.ffn, cfg.hidden, cfg.batch * K_BLOCK
    g = torch.Generator(device="cuda").manual_seed(0)
    W = (torch.randn((N, K), device="cuda", generator=g) * 0.02).bfloat16()
    x = torch.randn((M, K), device="cuda", generator=g)
    hi = x.bfloat16()
    lo = (x - hi.float()).bfloat16()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    bn = 16
    while bn < M and bn < 128:
        bn *= 2
    n_tiles, n_kb = -(-N // 128) * -(-M // bn), -(-K // 64)
    splits = max(1, min(-(-(3 * sms // 2) // n_tiles), 8, max(1, n_kb // 4)))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        gemm_bf16(W, hi, splits=splits, X_lo=lo)
    torch.cuda.synchronize()
    times = []
    for _ in range(args.steps):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        gemm_bf16(W, hi, splits=splits, X_lo=lo)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = float(np.median(times))
    byts = N * K * 2 + M * K * 4 + M * N * 4 * splits
    flops = 2.0 * M * N * K
    hbm, tc, kind = load_peaks(sustained=False)
    print(json.dumps({"kernel": f"k_gemm_tc (gate/up, M={M} hi+lo)", "N": N, "K": K, "M": M, "splits": splits,
                      "us": ms * 1e3, "GB_per_s": byts / (ms / 1e3) / 1e9,
                      "frac_hbm": byts / (ms / 1e3) / 1e9 / hbm,
                      "TFLOP_per_s_method": flops / (ms / 1e3) / 1e12,
                      "TFLOP_per_s_issued": 2 * flops / (ms / 1e3) / 1e12, "peak": f"{kind} {hbm} GB/s, {tc} TFLOP/s"}),
          flush=True)


def _median_ms(fn, reps: int, flush) -> float:
    import torch
    times = []
    for _ in range(reps):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    return float(np.median(times))


def run_sweep(args, cfg):
    """Draft-cost sweeps on the workload's shapes.

    layers: a round (inject, draft, accept) and a draft pass alone with 1, 3
    and 5 draft layers.  rows: the drafter's projections (one layer's QKV, O,
    gate/up, down, and the LM head) on 1 activation row (one token per
    sequence, an autoregressive step) and on 16 rows (the K = 16 block), each
    from HBM (L2 flushed before every launch); one JSON line per item."""
    import torch
    from block_diffusion_speculative_hidden_gb300 import gemm_bf16
    device = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    steps = args.steps
    for L in (1, 3, 5):
        c = cfg.replace(n_layers=L, name=f"{cfg.name}_{L}layer")
        wl = Workload(c, 64, 0, device, reset_every=args.reset_every)
        for i in range(args.warmup):
            wl.step(i)
            wl.maybe_reset(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(steps):
            wl.step(args.warmup + i)
            wl.maybe_reset(args.warmup + i)
        e1.record()
        torch.cuda.synchronize()
        round_ms = e0.elapsed_time(e1) / steps
        B = c.batch
        draft_ms = _median_ms(lambda: wl.dr.draft_block(B, c.s_passes, tokens=wl.tok, conf=wl.conf), steps, flush)
        assert wl.dr.device_status() == 0
        print(json.dumps({"sweep": "draft_layers", "workload": c.name, "n_layers": L, "round_ms": round_ms,
                          "draft_pass_ms": draft_ms, "draft_tok_per_s": B * K_BLOCK / (round_ms / 1e3)}), flush=True)
        del wl
        torch.cuda.empty_cache()
    d, F, V = cfg.hidden, cfg.ffn, cfg.vocab
    qkv = (cfg.n_q_heads + 2 * cfg.n_kv_heads) * cfg.head_dim
    shapes = {"qkv": (qkv, d), "o": (d, cfg.n_q_heads * cfg.head_dim), "gate_up": (2 * F, d), "down": (d, F),
              "lm_head": (V, d)}
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    g = torch.Generator(device=device).manual_seed(0)
    tot = {1: 0.0, 16: 0.0}
    st = torch.zeros(1, dtype=torch.int32, device=device)
    for name, (N, Kd) in shapes.items():
        W = (torch.randn((N, Kd), device=device, generator=g) * 0.02).bfloat16()
        n_tiles, n_kb = -(-N // 128), -(-Kd // 64)
        splits = max(1, min(2 * sms // n_tiles, max(1, n_kb // 4)))
        row = {}
        for M in (1, 16):
            x = torch.randn((M, Kd), device=device, generator=g)
            hi = x.bfloat16()
            lo = (x - hi.float()).bfloat16()
            for _ in range(args.warmup):
                gemm_bf16(W, hi, splits=splits, X_lo=lo, status=st)
            row[M] = _median_ms(lambda: gemm_bf16(W, hi, splits=splits, X_lo=lo, status=st), steps, flush)
            tot[M] += row[M] * (cfg.n_layers if name != "lm_head" else 1)
        print(json.dumps({"sweep": "block_rows", "projection": name, "N": N, "K": Kd, "us_1_row": row[1] * 1e3,
                          "us_16_rows": row[16] * 1e3, "ratio_16_over_1": row[16] / row[1]}), flush=True)
        del W
    assert int(st.item()) == 0
    print(json.dumps({"sweep": "block_rows", "projection": f"all ({cfg.n_layers} layers + LM head)",
                      "ms_1_row": tot[1], "ms_16_rows": tot[16], "ratio_16_over_1": tot[16] / tot[1]}), flush=True)


def gemm_flops(cfg):
    """Multiply-add flops (x2) of the projections and the LM head per round:
    the method's (one product per weight and activation row) and the issued
    ones (bf16 workloads multiply the hi and the lo activation terms).  S = 2
    runs the layers twice and the second LM head on the K/2 uncommitted rows
    of each block only."""
    M, d, F, V, L = cfg.batch * K_BLOCK, cfg.hidden, cfg.ffn, cfg.vocab, cfg.n_layers
    qd, kvd = cfg.q_dim, cfg.kv_dim
    per_layer = 2 * M * d * (qd + 2 * kvd) + 2 * M * qd * d + 2 * M * d * 2 * F + 2 * M * F * d
    proj = L * per_layer * cfg.s_passes
    lm = 2 * M * d * V + (cfg.s_passes - 1) * 2 * (M // 2) * d * V
    terms = 2 if cfg.dtype == "bf16" else 1
    return {"proj": proj, "lm_head": lm, "issued_factor": terms}


def tensor_bound(cfg) -> bool:
    """The projections are tensor-bound from M = 512 activation rows up
    (weights streamed at M rows have ~M flop per byte, above GB300's ridge)."""
    return cfg.dtype == "bf16" and cfg.batch * K_BLOCK >= 512


def mean_context(res) -> float:
    """The context grows by tau + 1 per round and is rolled back to the
    prompt every `period` rounds: mean over the period."""
    return float(res["lens"].mean()) + 0.5 * res["period"] * (res["mean_tau"] + 1)


def roofline_block(cfg, res, hbm, tc, peak_kind):
    """The dominant kernel's roofline (the projections and LM head) and
    the per-class figures, from the profiled (second) timed region."""
    ab = algorithmic_bytes(cfg)
    fl = gemm_flops(cfg)
    prof = res["prof"]
    steps = res["steps"]
    B = cfg.batch
    gemm_ms = prof["proj"][0] + prof["lm_head"][0]
    gemm_launches = prof["proj"][1] + prof["lm_head"][1]
    per_class = {k: {"ms_per_step": v[0] / steps, "launches_per_step": v[1] / steps} for k, v in prof.items()}
    attn_bytes = kv_bytes(cfg, int(mean_context(res))) * steps
    if prof["attention"][0] > 0:
        per_class["attention"]["GB_per_s"] = attn_bytes / (prof["attention"][0] / 1e3) / 1e9
        per_class["attention"]["frac_hbm"] = per_class["attention"]["GB_per_s"] / hbm
    for k in ("proj", "lm_head"):
        per_class[k]["GB_per_s"] = ab[k] * steps / (prof[k][0] / 1e3) / 1e9
        per_class[k]["TFLOP_per_s_method"] = fl[k] * steps / (prof[k][0] / 1e3) / 1e12
        per_class[k]["TFLOP_per_s_issued"] = fl[k] * fl["issued_factor"] * steps / (prof[k][0] / 1e3) / 1e12
    if prof["inject"][0] > 0:
        per_class["inject"]["GB_per_s"] = ab["inject_weights"] * steps / (prof["inject"][0] / 1e3) / 1e9
        per_class["inject"]["frac_hbm"] = per_class["inject"]["GB_per_s"] / hbm
    if cfg.accept == "stochastic" and prof["accept"][0] > 0:
        # each of the tau + 1 target rows read: one pass for its softmax
        # normaliser, one for the race (fp32 logits)
        acc_bytes = B * (res["mean_tau"] + 1) * cfg.vocab * 4 * 2 * steps
        per_class["accept"]["GB_per_s"] = acc_bytes / (prof["accept"][0] / 1e3) / 1e9
        per_class["accept"]["frac_hbm"] = per_class["accept"]["GB_per_s"] / hbm
    per_class["synthetic_target"] = {"ms_per_step": res["target_ms"] / steps,
                                     "what": "torch ops that form the target's verify output; not this library's"}
    # the projections and LM head of 256 block rows and more run on the
    # persistent kernel (k_gemm_pers), fewer on the single-tile one
    kname = ("k_gemm_pers" if cfg.dtype == "bf16" and cfg.weight_format != "e4m3" and cfg.batch * K_BLOCK >= 256
             else "k_gemm_tc")
    common = {"kernel": f"{kname} (tcgen05 projections + LM head)",
              "launches_per_step": gemm_launches / steps,
              "timed_in": "second timed region of the same loop, per-launch CUDA events"}
    if tensor_bound(cfg):
        flops = (fl["proj"] + fl["lm_head"]) * steps
        achieved = flops / (gemm_ms / 1e3) / 1e12
        tf = gemm_traffic(cfg)
        roof = dict(common, bound="tensor", achieved=achieved, peak=tc, unit="TFLOP/s", frac=achieved / tc,
                    peak_kind=f"{peak_kind} bf16_tflops_sustained (kernels timed inside a seconds-long loop)",
                    flops_per_step=fl["proj"] + fl["lm_head"], traffic=tf,
                    traffic_unit=(f"bytes per launch (ncu dram read+write at full size; profiles/"
                                  f"{TRAFFIC_PROFILES[cfg.name][0]})") if tf is not None else None,
                    algorithmic_bytes_per_launch=(ab["proj"] + ab["lm_head"]) * steps / max(gemm_launches, 1),
                    issued={"achieved": achieved * fl["issued_factor"], "frac": achieved * fl["issued_factor"] / tc,
                            "what": "both bf16 activation terms (hi + lo) multiplied: twice the method's flops"})
        return roof, per_class
    gemm_bytes = (ab["proj"] + ab["lm_head"]) * steps
    achieved = gemm_bytes / (gemm_ms / 1e3) / 1e9
    roof = dict(common, bound="hbm", achieved=achieved, peak=hbm, unit="GB/s", frac=achieved / hbm,
                peak_kind=f"{peak_kind} hbm_gbs", traffic=gemm_traffic(cfg),
                traffic_unit=(f"bytes per launch (ncu dram read+write at full size; profiles/"
                              f"{TRAFFIC_PROFILES[cfg.name][0]})") if cfg.name in TRAFFIC_PROFILES else None,
                algorithmic_bytes_per_launch=(ab["proj"] + ab["lm_head"]) * steps / max(gemm_launches, 1),
                bytes_per_step=ab["proj"] + ab["lm_head"])
    return roof, per_class


def run_per_config(args, names, world, rank, local, hbm, tc, peak_kind):
    """The other workloads, each timed like the headline one (its own
    warm-up, region A with clocks, region B per kernel class), without the
    end-to-end and graph legs."""
    import torch
    out = {}
    for name in names:
        c = synth.get_config(name)
        torch.cuda.empty_cache()
        res = run_ours(args, c, world, rank, local, steps=args.per_config_steps, legs=False)
        roof, per_class = roofline_block(c, res, hbm, tc, peak_kind)
        out[name] = {"workload": c.name, "value": res["value"], "unit": UNIT,
                     "ms_per_step": res["ms"] / res["steps"], "steps": res["steps"], "warmup": args.warmup,
                     "dtype": line_dtype(c), "mean_tau": res["mean_tau"], "accept": c.accept,
                     "rounds_per_prompt": res["period"], "mean_context": mean_context(res),
                     "roofline": roof, "kernels": per_class, "clocks": res["clocks"],
                     "gpu_launches_per_step": res["launches_per_step"]}
        del res
    torch.cuda.empty_cache()
    return out


def line_dtype(cfg) -> str:
    """The arithmetic the path computes in: fp32 SIMT for fp32 workloads,
    bf16 tensor-core products (fp32 accumulation) otherwise, with E4M3
    weights widened to bf16 for the FP8-weight workloads."""
    if cfg.dtype == "f32":
        return "f32"
    return "bf16 (e4m3 weights)" if cfg.weight_format == "e4m3" else "bf16"


def run_kernel_train_attn(args, cfg):
    """Training-time block attention (Fig. 4 mask) on the workload's attention
    shape: S sequences of T context positions (seeded fp16 keys and values in
    the pool), NB blocks at seeded prefix lengths, each launch from a flushed
    L2; the oracle timed on a sample of the same blocks."""
    import torch
    from block_diffusion_speculative_hidden_gb300 import Drafter, weights_to_device
    S, T, per_seq = 4, 4096, 64
    NB = S * per_seq
    c = cfg.replace(n_layers=1, ffn=256, vocab=512, n_taps=1, tap_width=cfg.hidden, name=cfg.name + "_attn")
    Hq, Hkv, dh = c.n_q_heads, c.n_kv_heads, c.head_dim
    mpps = T // 16
    dev = torch.device("cuda", 0)
    dr = Drafter(c, weights_to_device(synth.make_weights(c), c.dtype, device=dev), max_batch=NB,
                 max_pages_per_seq=mpps, n_pages=S * mpps, max_rows=17, max_inject_rows=NB * 17)
    g = torch.Generator(device=dev).manual_seed(7)
    Kp, Vp = dr.pool_kv()
    Kp[0, :S * mpps].copy_(torch.randn(Kp[0, :S * mpps].shape, generator=g, device=dev).half())
    Vp[0, :S * mpps].copy_(torch.randn(Vp[0, :S * mpps].shape, generator=g, device=dev).half())
    pt = torch.full((NB, mpps), -1, dtype=torch.int32)
    pt[:S] = torch.arange(S * mpps, dtype=torch.int32).reshape(S, mpps)
    dr.page_table.copy_(pt)
    sl = torch.zeros(NB, dtype=torch.int32)
    sl[:S] = T
    dr.seq_len.copy_(sl)
    rng = np.random.default_rng(8)
    seq = np.repeat(np.arange(S, dtype=np.int32), per_seq)
    ctx_len = rng.integers(T // 4, T + 1, size=NB).astype(np.int32)
    q = torch.randn((NB, 16, Hq, dh), generator=g, device=dev).half()
    kb = torch.randn((NB, 16, Hkv, dh), generator=g, device=dev).half()
    vb = torch.randn((NB, 16, Hkv, dh), generator=g, device=dev).half()
    sq, cl = torch.from_numpy(seq).to(dev), torch.from_numpy(ctx_len).to(dev)
    out = torch.empty((NB, 16, Hq, dh), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(max(3, args.warmup)):
        dr.block_attention(0, sq, cl, q, kb, vb, out=out)
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    ms = _median_ms(lambda: dr.block_attention(0, sq, cl, q, kb, vb, out=out), max(10, min(args.steps, 50)), flush)
    keys = ctx_len.astype(np.float64) + 16
    flops = float(np.sum(4.0 * 16 * Hq * dh * keys))
    logical = float(np.sum(2.0 * keys * Hkv * dh * 2))           # K and V each block reads
    unique = 2.0 * S * T * Hkv * dh * 2 + 3.0 * NB * 16 * Hkv * dh * 2 + NB * 16 * Hq * dh * (2 + 4)
    hbm, tc, kind = load_peaks(sustained=False)
    # the oracle on a sample of blocks (fp64 NumPy), scaled to all NB
    from oracle import dflash_oracle as O
    Kh, Vh = Kp[0, :S * mpps].float().cpu().numpy(), Vp[0, :S * mpps].float().cpu().numpy()
    ctx_k = [Kh[s * mpps:(s + 1) * mpps].transpose(0, 2, 1, 3).reshape(T, Hkv, dh) for s in range(S)]
    ctx_v = [Vh[s * mpps:(s + 1) * mpps].transpose(0, 2, 1, 3).reshape(T, Hkv, dh) for s in range(S)]
    sample = np.arange(0, NB, NB // 8)
    t0 = time.time()
    O.block_attention_train(q[sample].float().cpu().numpy(), kb[sample].float().cpu().numpy(),
                            vb[sample].float().cpu().numpy(), ctx_k, ctx_v, seq[sample], ctx_len[sample])
    cpu_s = (time.time() - t0) * NB / len(sample)
    print(json.dumps({
        "kernel": "k_attn_mma (training-time block attention, Fig. 4 mask; dflash_block_attention)",
        "workload": f"{c.name}: {S} sequences x {T} context, {NB} blocks of 16, prefixes U[{T // 4}, {T}]",
        "heads": f"{Hq}/{Hkv}x{dh}", "us": ms * 1e3, "blocks_per_s": NB / (ms / 1e3),
        "roofline": {"bound": "tensor", "achieved": flops / (ms / 1e3) / 1e12, "peak": tc, "unit": "TFLOP/s",
                     "frac": flops / (ms / 1e3) / 1e12 / tc, "peak_kind": f"{kind} bf16_tflops (fp16 MMA, same rate)",
                     "flops_per_launch": flops},
        "kv_bytes": {"logical_per_launch": logical, "unique_per_launch": unique,
                     "logical_GB_per_s": logical / (ms / 1e3) / 1e9, "unique_frac_hbm": unique / (ms / 1e3) / 1e9 / hbm},
        "l2": "L2 flushed before every launch",
        "cpu_baseline": {"kind": "oracle", "seconds_per_launch": cpu_s, "sample": f"{len(sample)} of {NB} blocks",
                         "cores": os.cpu_count()},
    }), flush=True)


# --------------------------------------------------------------------------- main

def main(argv=None):
    args = parse_args(argv)
    cfg = synth.get_config(args.config)
    if args.small:
        cfg = cfg.replace(n_layers=1, vocab=16384, name=cfg.name + "_1layer_v16k")
    if args.kernel == "gemm":
        run_kernel_gemm(args, cfg)
        return
    if args.kernel == "train_attn":
        run_kernel_train_attn(args, cfg)
        return
    if args.sweep:
        run_sweep(args, cfg)
        return
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, cfg, world, rank)
        return
    res = run_ours(args, cfg, world, rank, local)
    if rank != 0:
        return
    hbm, tc, peak_kind = load_peaks()
    steps = args.steps
    lens = res["lens"]
    roof, per_class = roofline_block(cfg, res, hbm, tc, peak_kind)
    wl = res.pop("wl")
    w_np, prefill, stoch = wl.w_np, wl.prefill, wl.stochastic
    del wl
    per_config = None
    names = [n for n in args.per_config.split(",") if n and n != args.config]
    if names and world == 1:
        per_config = run_per_config(args, names, world, rank, local, hbm, tc, peak_kind)
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(cfg, args, w_np)
    target = ("per step, torch forms the target's logits: the draft call's logits output (pass-1 rows on the "
              "committed positions, pass-2 rows elsewhere) + N(0,1) noise from 4 device-resident draws, the bonus "
              "row noise alone; inside the region, timed as kernels.synthetic_target" if stoch else
              "per step, one torch elementwise op forms y from the drafts and the round's coins; inside the region")
    line = {
        "metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": res["ms"] / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": line_dtype(cfg),
        "data": "synthetic (seeded random-init weights, N(0,1) features)",
        "config": config_block(cfg, lens),
        "mean_tau": res["mean_tau"], "mean_context": mean_context(res), "parallelism": f"replicas x{world}",
        "synthetic_target": target,
        "roofline": roof,
        "kernels": per_class,
        "cpu_baseline": cpu,
        "accepted_tok_per_s": world * cfg.batch * (res["mean_tau"] + 1) / (res["ms"] / steps / 1e3),
        "prefill_inject": prefill,
        "e2e": res["e2e"],
        "graph": res["graph"],
        "per_config": per_config,
        "gpu_launches": int(round(res["launches_per_step"] * steps)),
        "clocks": res["clocks"],
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

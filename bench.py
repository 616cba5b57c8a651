#!/usr/bin/env python
"""Benchmark: exact verify throughput of the 4-layer hybrid stack on GB300.

A step is one full verify round of the hot path over one batch: xv_verify_block
(embedding, 4 x [RMSNorm, input GEMM, GDN verify or KV append + decode-row
attention, output GEMM, residual + RMSNorm, gate/up GEMM, SwiGLU, down GEMM,
residual + RMSNorm], LM head, argmax, acceptance) followed by the commit of
the accepted positions.  Workload: hidden 5120, 3 GDN layers (32 x 128 x 128
fp32 state) + 1 gated attention layer (24/4 heads of 256), MLP 17408, vocab
151936, k = 8 tokens per sequence, batch 1, context 2183, all inputs seeded
and synthetic.  Metric: verified tokens per second (k * B per step).

Prints one JSON line.  `--impl reference` times the CPU oracle instead.
Multi-GPU (torchrun): each rank runs its own independent sequence (weak
scaling, no collective on the data path); the job value is the sum of tokens
over the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import atexit
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "exact verify tok/s (k=8, 1 stream) per hybrid block"
UNIT = "tok/s"
WORKLOAD = ("4-layer hybrid stack (3 GDN + 1 gated attention), hidden 5120, MLP 17408, vocab 151936; "
            "verify k=8 draft tokens, batch 1, context 2183")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="xv", choices=["xv", "reference"])
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--k", type=int, default=8)
    ap.add_argument("--context", type=int, default=2183)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--lmax", type=int, default=None,
                    help="KV-cache capacity per sequence (default: enough for every step the run makes)")
    ap.add_argument("--prefill", type=int, default=None, metavar="T",
                    help="time an exact chunked prefill of T prompt tokens instead of the verify step")
    ap.add_argument("--chunk", type=int, default=None,
                    help="with --prefill: tokens per verify pass (default 64 / batch, the most one GEMM call takes)")
    ap.add_argument("--full-gdn", action="store_true",
                    help="complete GDN layers: 16 q/k heads for the 32 v heads, width-4 causal convolution, "
                         "gated output norm")
    ap.add_argument("--page-size", type=int, default=None,
                    help="paged KV cache with pages of this many positions (a multiple of 64)")
    ap.add_argument("--no-overlap", action="store_true", help="launch kernels without programmatic dependent launch")
    ap.add_argument("--no-kernel-rooflines", action="store_true", help="skip the per-kernel measurements")
    ap.add_argument("--kernel", choices=["gemm", "gdn", "attn"], default=None,
                    help="time one hot kernel alone on one workload shape (for profiler captures) instead of the step")
    ap.add_argument("--shape", default=None, help="with --kernel: gemm gdn_in|gdn_out|attn_in|attn_out|gate_up|down|"
                    "lm_head (M = --batch * --k); gdn: B = --batch; attn: context --context, B = --batch")
    ap.add_argument("--launches", type=int, default=4, help="with --kernel: launches to run")
    ap.add_argument("--speculative", type=float, default=None, metavar="ACCEPT",
                    help="run greedy speculative decoding rounds (verify k, accept, commit) with a stand-in drafter "
                         "whose drafts are right with probability ACCEPT, and report committed tokens per second")
    ap.add_argument("--tokens", type=int, default=128, help="with --speculative: tokens to emit")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 10 ms while running, each sample tagged
    with the host time it arrived."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "10", "-i", str(self.index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            atexit.register(self.__exit__)   # the sampler never outlives the bench, even on an error
        except FileNotFoundError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def wait_first(self, timeout=5.0):
        """Blocks until the sampler has produced a line (so the timed region is covered)."""
        t0 = time.time()
        while self.proc and not self.lines and time.time() - t0 < timeout:
            time.sleep(0.02)

    def __exit__(self, *a):
        if self.proc and self.proc.poll() is None:
            self.proc.terminate()
            self.proc.wait(timeout=5)

    def summary(self, t0, t1, t_load):
        """Samples of the timed region [t0, t1] (host times), and of the loaded window [t0, t_load]
        that continues it with more steps of the same workload: the median SM clock over the
        timed region's samples (over the loaded window's when a short region caught fewer than
        three), throttle reasons seen anywhere in the loaded window."""
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        timed, loaded, mx, reasons = [], [], None, set()
        for t, ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7 or not (t0 <= t <= t_load):
                continue
            try:
                f = float(parts[0])
                mx = float(parts[1])
            except ValueError:
                continue
            loaded.append(f)
            if t <= t1:
                timed.append(f)
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        use = timed if len(timed) >= 3 else loaded
        return {"sm_mhz": float(np.median(use)) if use else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(timed), "samples_loaded": len(loaded),
                "window": "timed region" if use is timed else
                          "timed region and the traced and end-to-end steps that follow it"}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ----------------------------------------------------------------- setup

def make_stack(args, device, rank=0, extra_rounds=0, w=None, wd=None, device_kv=False):
    """The 4-layer stack with its weights (the same on every rank: replicas of one model) and
    rank's own sequences (caches, GDN states and draft tokens from the rank's seed).  ``w`` / ``wd``
    reuse weights already drawn (host bits / device tensors); with ``device_kv`` the KV caches are
    drawn on the device (seeded N(0, 1), the recipe's distribution) instead of on the host, for the
    long-context timing lines."""
    import torch
    from synth import workloads
    from bit_exact_speculative_gb300.model import HybridStack, tile_weights
    from bit_exact_speculative_gb300.replicas import rank_seed

    cfg = workloads.STACK_FULL if args.full_gdn else workloads.STACK
    if w is None:
        w = workloads.weights(cfg, seed=0)
    if wd is None:
        # the GEMM weights in the tiled layout (the same bits as row-major, faster streaming)
        wd = tile_weights(cfg, {n: torch.from_numpy(a.view(np.int16)).to(device) for n, a in w.items()})
    B, k, L = args.batch, args.k, args.context
    seq = rank_seed(0, rank)
    rounds = 3 * (args.steps + args.warmup) + 8 + extra_rounds
    Lmax = L + k * rounds + 64
    if args.lmax:
        if args.lmax < Lmax:
            raise SystemExit(f"--lmax {args.lmax} is below the {Lmax} positions this run needs")
        Lmax = args.lmax
    paged = {}
    if args.page_size:
        # a pool with room for every sequence at Lmax, its pages handed out in a seeded random order
        n_pages = B * (-(-Lmax // args.page_size))
        paged = dict(page_size=args.page_size, n_pages=n_pages,
                     page_order=np.random.default_rng(seq).permutation(n_pages))
    stk = HybridStack(cfg, wd, B, k, Lmax, device=device, **paged)

    def reset():
        stk.set_context([L] * B)
        for l, kd in enumerate(cfg["kinds"]):
            if kd == 0:
                stk.state[f"{l}.state"].copy_(torch.from_numpy(workloads.gdn_state(cfg, seq, l, B)))
                if cfg.get("gdn_conv"):
                    stk.state[f"{l}.conv"].copy_(torch.from_numpy(workloads.conv_state(cfg, seq, l, B).view(np.int16)))
            elif device_kv:
                g = torch.Generator(device=device)
                g.manual_seed(seq * 1000 + l)
                for name in ("kc", "vc"):
                    c = stk.state[f"{l}.{name}"]
                    c.zero_()
                    for b in range(B):
                        c[b, :, :L].copy_(torch.randn(c[b, :, :L].shape, generator=g, device=device)
                                          .to(torch.bfloat16).view(torch.int16))
            else:
                kc, vc = workloads.kv_cache(cfg, seq, l, B, [L] * B, Lmax)
                stk.load_kv(l, torch.from_numpy(kc.view(np.int16)), torch.from_numpy(vc.view(np.int16)))

    reset()
    stk.reset = reset
    stk.wd = wd
    toks = np.stack([workloads.draft_tokens(cfg, seq, r, B, k) for r in range(rounds)])
    return cfg, w, stk, toks


def gemm_shapes(cfg, M):
    """(N, K) of every GEMM in one verify step, with its output element size."""
    H, F, V = cfg["hidden"], cfg["mlp"], cfg["vocab"]
    from bit_exact_speculative_gb300.model import gdn_in_dim
    gin = gdn_in_dim(cfg)
    ain = 2 * cfg["attn_hq"] * cfg["attn_hd"] + 2 * cfg["attn_hkv"] * cfg["attn_hd"]
    out = []
    for kd in cfg["kinds"]:
        if kd == 0:
            out += [(gin, H, 2), (H, cfg["gdn_heads"] * cfg["gdn_dv"], 2)]
        else:
            out += [(ain, H, 2), (H, cfg["attn_hq"] * cfg["attn_hd"], 2)]
        out += [(2 * F, H, 2), (H, F, 2)]
    out.append((V, H, 4))
    return out


def code_digest(path: str) -> str:
    """sha256 (16 hex digits) of a C++/CUDA source with its comments and white space removed: a
    comment edit leaves it as it is, any change to the code does not."""
    import hashlib
    import re
    src = open(path).read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return hashlib.sha256(" ".join(src.split()).encode()).hexdigest()[:16]


def traffic_ratio_from_profile(kernel_src: str):
    """ncu DRAM bytes (read + write) per algorithmic byte of the GEMM kernel, from the committed
    capture of one projection shape (profiles/traffic.json), if that capture matches this source's
    code (`code_digest`); else None.  The GEMM streams each weight once, so its traffic scales with
    the bytes it moves."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    h = code_digest(kernel_src)
    e = d.get("gemm_small_m")
    if not e or e.get("code_digest") != h:
        return None
    return float(e["ratio"])


# ------------------------------------------------------ per-kernel rooflines

def _back_to_back_ms(launch, n):
    """Device time per launch of n launches issued back to back (programmatic dependent launch
    as in the step), between two events on the launching stream."""
    import torch
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        launch(i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def kernel_rooflines(xv, device, peak):
    """The three hot kernels alone, each timed over back-to-back launches with its inputs rotated
    through more than 3x L2 (every launch reads cold data), per launch."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(0)
    out = {}

    def rnd(shape, scale=1.0, dtype=torch.bfloat16):
        return (torch.randn(shape, generator=g, device=device) * scale).to(dtype)

    def copies_for(nbytes):
        return max(2, int(np.ceil(400e6 / max(nbytes, 1))))

    def line(ms, nbytes):
        return {"us": round(ms * 1e3, 2), "bytes": nbytes, "gbs": round(nbytes / ms / 1e6, 1),
                "frac": round(nbytes / ms / 1e6 / peak, 4)}

    # small-M GEMM: every projection shape of the stack at 8 and 64 token rows, and the
    # gate/up (17408 x 5120) and down (5120 x 17408) sweep over M in {1, 2, 4, 8, 9, 16}
    gem, sweep = {}, {}
    cases = [(M, N, K, name, f32, gem) for M in (8, 64)
             for N, K, name, f32 in [(12352, 5120, "gdn_in", False), (5120, 4096, "gdn_out", False),
                                     (14336, 5120, "attn_in", False), (5120, 6144, "attn_out", False),
                                     (34816, 5120, "gate_up", False), (5120, 17408, "down", False),
                                     (151936, 5120, "lm_head", True)]]
    cases += [(M, N, K, name, False, sweep) for M in (1, 2, 4, 8, 9, 16)
              for N, K, name in [(17408, 5120, "up17408"), (5120, 17408, "down17408")]]
    W_cache = {}
    for M, N, K, name, f32, dst in cases:
        nc = copies_for(2 * N * K)
        if (N, K) not in W_cache:
            W_cache.clear()
            torch.cuda.empty_cache()
            tile = xv.tile_gate_up if name == "gate_up" else xv.tile_weight
            W_cache[(N, K)] = [tile(rnd((N, K), 0.02)) for _ in range(nc)]
        Ws = W_cache[(N, K)]
        X = rnd((M, K))
        gated = name == "gate_up"   # as in the step: the SwiGLU fused, F = N / 2 outputs
        Y = torch.empty((M, N // 2 if gated else N), dtype=torch.float32 if f32 else torch.bfloat16, device=device)
        ws = xv.workspace(max(xv.xv_gemm_workspace_size(M, N, K), 256), device=device)
        if gated:
            launch = lambda i: xv.xv_gemm_swiglu(X, Ws[i % nc], Y)
        else:
            launch = lambda i: xv.xv_gemm_small_m(X, Ws[i % nc], Y, ws)
        for i in range(nc):
            launch(i)
        ms = _back_to_back_ms(launch, 3 * nc)
        nbytes = 2 * N * K + 2 * M * K + Y.numel() * Y.element_size()
        dst[f"{name}_M{M}"] = dict(N=N, K=K, splits=xv.xv_gemm_splits(N, K), **line(ms, nbytes))
    W_cache.clear()
    torch.cuda.empty_cache()
    out["gemm_small_m"] = gem
    out["gemm_sweep"] = sweep

    # GDN verify: 32 heads of 128 x 128 fp32, k = 8 speculative steps after 1 replayed step (8 staged)
    H, D, k = 32, 128, 8
    gd = {}
    for B in (1, 8):
        state_bytes = 4 * B * H * D * D
        nc = copies_for(state_bytes)
        states = [torch.randn((B, H, D, D), generator=g, device=device) * 0.1 for _ in range(nc)]
        rows = B * k
        qkv = rnd((rows, H * 3 * D))
        gates = torch.rand((rows, 2 * H), generator=g, device=device).to(torch.bfloat16)
        st = xv.gdn_steps(qkv, qkv[:, H * D:], qkv[:, 2 * H * D:], gates, gates[:, H:], 3 * H * D, 2 * H, k)
        n = torch.ones(B, dtype=torch.int32, device=device)
        o = torch.empty((rows, H * D), dtype=torch.bfloat16, device=device)
        launch = lambda i: xv.xv_gdn_verify(states[i % nc], st, n, k, st, k, o, H * D, B, H, D, D, True)
        for i in range(nc):
            launch(i)
        ms = _back_to_back_ms(launch, 3 * nc)
        nbytes = 2 * state_bytes + 2 * (1 + k) * B * H * (3 * D + 2) + 2 * k * B * H * D
        gd[f"B{B}"] = line(ms, nbytes)
        del states
        torch.cuda.empty_cache()
    out["gdn_verify"] = gd

    # decode-row attention (split + combine): 24 q / 4 kv heads of 256, 8 rows per sequence
    Hq, Hkv, hd, R = 24, 4, 256, 8
    at = {}
    for L in (640, 2183, 131072):
        for B in (1, 8):
            Lmax = L + R
            cache_bytes = 2 * B * Hkv * Lmax * hd * 2
            nc = copies_for(cache_bytes) if L < 131072 else 1
            kcs = [rnd((B, Hkv, Lmax, hd)) for _ in range(nc)]
            vcs = [rnd((B, Hkv, Lmax, hd)) for _ in range(nc)]
            q = rnd((B * R, Hq * hd))
            outb = torch.empty((B * R, Hq * hd), dtype=torch.bfloat16, device=device)
            ctx = torch.full((B,), L, dtype=torch.int32, device=device)
            ws = xv.workspace(xv.xv_attn_workspace_size(B, R, Hq, hd, L + R - 1), device=device)
            launch = lambda i: xv.xv_attn_decode_rows(q, q.stride(0), kcs[i % nc], vcs[i % nc], ctx, R, B, Hq, Hkv, hd,
                                                      Lmax, L + R - 1, hd ** -0.5, outb, outb.stride(0), ws)
            for i in range(nc):
                launch(i)
            ms = _back_to_back_ms(launch, max(3 * nc, 5))
            nbytes = B * (4 * Hkv * (L + R - 1) * hd + 2 * 2 * R * Hq * hd)   # K+V of every visible position, q, out
            at[f"L{L}_B{B}"] = line(ms, nbytes)
            del kcs, vcs
            torch.cuda.empty_cache()
    out["attn_decode_rows"] = at
    out["timing"] = ("per launch over back-to-back launches between two CUDA events, inputs rotated through "
                     "more than 3x L2 (cold every launch)")
    return out


def gemm_chain_ms(xv, stk, cfg, M, reps, device):
    """The step's 17 projection GEMMs alone, in step order, on the stack's own weights, issued back
    to back with programmatic dependent launch as in the step (each still waits for the previous
    one before reading its activations): device time per GEMM launch.  The weights (4.4 GB) stream
    from HBM every round."""
    import torch
    from bit_exact_speculative_gb300.model import gdn_in_dim
    H, F, V = cfg["hidden"], cfg["mlp"], cfg["vocab"]
    w = stk.wd
    plan = []
    for l, kd in enumerate(cfg["kinds"]):
        inner = cfg["gdn_heads"] * cfg["gdn_dv"] if kd == 0 else cfg["attn_hq"] * cfg["attn_hd"]
        plan += [(w[f"{l}.w_in"], H, False), (w[f"{l}.w_out"], inner, False), (w[f"{l}.w_gu"], H, False),
                 (w[f"{l}.w_down"], F, False)]
    plan.append((w["lm_head"], H, True))
    g = torch.Generator(device=device)
    g.manual_seed(1)
    Xs = {K: torch.randn((M, K), generator=g, device=device).to(torch.bfloat16) for _, K, _ in plan}
    calls = []
    for W, K, f32 in plan:
        N = W.shape[0]
        gated = getattr(W, "gated", False)   # gate/up with the SwiGLU fused: F = N / 2 outputs
        Y = torch.empty((M, N // 2 if gated else N), dtype=torch.float32 if f32 else torch.bfloat16, device=device)
        ws = xv.workspace(max(xv.xv_gemm_workspace_size(M, N, K), 256), device=device)
        calls.append((Xs[K], W, Y, ws, 2 * N * K + 2 * M * K + Y.numel() * Y.element_size()))

    def launch(i):
        X, W, Y, ws, _ = calls[i % len(calls)]
        if getattr(W, "gated", False):
            xv.xv_gemm_swiglu(X, W, Y)
        else:
            xv.xv_gemm_small_m(X, W, Y, ws)
    for i in range(len(calls)):
        launch(i)
    ms = _back_to_back_ms(launch, reps * len(calls))
    return ms, sum(c[4] for c in calls) / len(calls), len(calls)


def step_line(args, device, w, wd, batch, context, steps=10, warmup=3):
    """ms per verify step and verified tok/s of one more (batch, context) configuration of the same
    stack (KV caches drawn on the device)."""
    import copy
    import torch
    a = copy.copy(args)
    a.batch, a.context, a.steps, a.warmup, a.page_size, a.lmax = batch, context, steps, warmup, None, None
    cfg, _, stk, toks = make_stack(a, device, 0, w=w, wd=wd, device_kv=True)
    tok_dev = torch.from_numpy(toks).to(device)
    k = a.k
    for i in range(warmup):
        stk.verify_commit(tok_dev[i], k)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        stk.verify_commit(tok_dev[warmup + i], k)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    del stk
    torch.cuda.empty_cache()
    return {"batch": batch, "context": context, "k": k, "steps": steps, "ms_per_step": round(ms, 4),
            "value": round(batch * k / (ms / 1e3), 1), "unit": UNIT}


# ------------------------------------------------------ one kernel alone

GEMM_SHAPES = {"gdn_in": (12352, 5120), "gdn_out": (5120, 4096), "attn_in": (14336, 5120), "attn_out": (5120, 6144),
               "gate_up": (34816, 5120), "down": (5120, 17408), "lm_head": (151936, 5120)}


def run_one_kernel(args):
    """--kernel: `launches` launches of one hot kernel on one stack shape, inputs resident (a fresh
    weight or state copy per launch up to 3 copies), for profiler captures; prints one JSON line."""
    import torch
    from bit_exact_speculative_gb300 import build
    from bit_exact_speculative_gb300 import xv
    build.build()
    device = torch.device("cuda", 0)
    g = torch.Generator(device=device)
    g.manual_seed(0)

    def rnd(shape, scale=1.0):
        return (torch.randn(shape, generator=g, device=device) * scale).to(torch.bfloat16)

    B, k, n = args.batch, args.k, args.launches
    if args.kernel == "gemm":
        N, K = GEMM_SHAPES[args.shape]
        M = B * k
        Ws = [xv.tile_weight(rnd((N, K), 0.02)) for _ in range(3)]
        X = rnd((M, K))
        Y = torch.empty((M, N), dtype=torch.float32 if args.shape == "lm_head" else torch.bfloat16, device=device)
        ws = xv.workspace(xv.xv_gemm_workspace_size(M, N, K), device=device)
        launch = lambda i: xv.xv_gemm_small_m(X, Ws[i % 3], Y, ws)
        desc = {"M": M, "N": N, "K": K}
    elif args.kernel == "gdn":
        H, D = 32, 128
        states = [torch.randn((B, H, D, D), generator=g, device=device) * 0.1 for _ in range(3)]
        qkv = rnd((B * k, H * 3 * D))
        gates = torch.rand((B * k, 2 * H), generator=g, device=device).to(torch.bfloat16)
        st = xv.gdn_steps(qkv, qkv[:, H * D:], qkv[:, 2 * H * D:], gates, gates[:, H:], 3 * H * D, 2 * H, k)
        nc = torch.ones(B, dtype=torch.int32, device=device)
        o = torch.empty((B * k, H * D), dtype=torch.bfloat16, device=device)
        launch = lambda i: xv.xv_gdn_verify(states[i % 3], st, nc, k, st, k, o, H * D, B, H, D, D, True)
        desc = {"B": B, "heads": H, "dk": D, "dv": D, "k": k}
    else:
        Hq, Hkv, hd, L = 24, 4, 256, args.context
        Lmax = max(L + k, args.lmax or 0)
        kcs = [rnd((B, Hkv, Lmax, hd)) for _ in range(2)]
        vcs = [rnd((B, Hkv, Lmax, hd)) for _ in range(2)]
        q = rnd((B * k, Hq * hd))
        out = torch.empty((B * k, Hq * hd), dtype=torch.bfloat16, device=device)
        ctx = torch.full((B,), L, dtype=torch.int32, device=device)
        ws = xv.workspace(xv.xv_attn_workspace_size(B, k, Hq, hd, L + k - 1), device=device)
        launch = lambda i: xv.xv_attn_decode_rows(q, q.stride(0), kcs[i % 2], vcs[i % 2], ctx, k, B, Hq, Hkv, hd, Lmax,
                                                  L + k - 1, hd ** -0.5, out, out.stride(0), ws)
        desc = {"B": B, "rows": k, "context": L, "hq": Hq, "hkv": Hkv, "hd": hd}
    launch(0)   # the first launch also loads the module: not timed
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(1, n):
        launch(i)
    e1.record()
    torch.cuda.synchronize()
    code = xv.xv_device_check()
    print(json.dumps({"kernel": args.kernel, "shape": args.shape, **desc, "launches": n,
                      "us_per_launch": round(e0.elapsed_time(e1) / max(n - 1, 1) * 1e3, 2),
                      "device_error_bits": code}), flush=True)


# ------------------------------------------------------- speculative rounds

def run_prefill(args):
    """Exact chunked prefill of a T-token prompt from an empty context on the 4-layer stack (verify
    passes of `chunk` tokens, every position committed, the LM head only in the last pass), timed
    with CUDA events: time to the first token and prompt tokens per second.  The caches and states
    it leaves are those of T decode steps."""
    import torch
    from synth import workloads
    from bit_exact_speculative_gb300 import build
    from bit_exact_speculative_gb300.model import HybridStack, tile_weights
    build.build()
    device = torch.device("cuda", 0)
    cfg = workloads.STACK_FULL if args.full_gdn else workloads.STACK
    w = workloads.weights(cfg, seed=0)
    wd = tile_weights(cfg, {n: torch.from_numpy(a.view(np.int16)).to(device) for n, a in w.items()})
    B, T = args.batch, args.prefill
    k = args.chunk if args.chunk else max(1, 64 // B)
    stk = HybridStack(cfg, wd, B, k, T + 64, device=device)
    prompt = torch.from_numpy(np.concatenate([workloads.draft_tokens(cfg, 0, 1000 + i % 97, B, 1) for i in range(T)],
                                             axis=1)).to(device)
    times = []
    for rep in range(2):   # the first run warms up
        stk.set_context([0] * B)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        stk.prefill(prompt, k)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3)
    t = times[-1]
    print(json.dumps({
        "metric": f"exact chunked prefill, prompt tok/s (chunks of {k}, batch {B})", "value": round(B * T / t, 1),
        "unit": "tok/s", "n_gpus": 1, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD.replace("verify k=8 draft tokens, batch 1, context 2183",
                                                f"prefill of {T} tokens from an empty context"),
                   "prompt_tokens": T, "batch": B, "chunk": k},
        "ttft_s": round(t, 4), "verify_passes": -(-T // k),
        "timing": "CUDA events around the whole prefill (second run)"}), flush=True)


def run_speculative(args):
    """Greedy speculative decoding of one sequence on the 4-layer stack: first the target's own
    greedy decode (k = 1 steps) as the reference, then rounds of verify k / accept / commit from
    the same state with drafts taken from that reference and corrupted at rate 1 - ACCEPT.  The
    emitted tokens must equal the reference exactly; the metric is committed tokens per second."""
    import torch
    from bit_exact_speculative_gb300 import build
    from bit_exact_speculative_gb300.speculative import ReplayDrafter, greedy_decode, speculative_decode
    build.build()
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    args.batch = 1
    n, k = args.tokens, args.k
    cfg, _, stk, toks = make_stack(args, device, 0, extra_rounds=(2 * n + 4 * k) // k + 1)
    first = int(toks[0, 0, 0])
    greedy_decode(stk, first, 4)                         # warm-up, then start over
    stk.reset()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ref = greedy_decode(stk, first, n)
    t_dec = time.perf_counter() - t0
    stk.reset()
    torch.cuda.synchronize()
    drafter = ReplayDrafter(ref, cfg["vocab"], args.speculative, seed=1)
    t0 = time.perf_counter()
    emitted, accepted = speculative_decode(stk, first, n, k, drafter)
    t_spec = time.perf_counter() - t0
    exact = emitted[:n] == ref[1:n + 1]
    value = len(emitted) / t_spec
    print(json.dumps({
        "metric": f"greedy speculative decode, committed tok/s (k={k}, 1 stream, draft acceptance {args.speculative})",
        "value": round(value, 1), "unit": UNIT, "n_gpus": 1, "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic", "config": {"workload": WORKLOAD.replace("verify k=8 draft tokens, batch 1",
                                                                      f"speculative rounds k={k}, batch 1"),
                                        "tokens": len(emitted), "context": args.context},
        "exact": bool(exact), "rounds": len(accepted),
        "mean_accepted_drafts": round(float(np.mean(accepted)), 3),
        "decode_tok_s": round(n / t_dec, 1), "speedup_vs_decode": round(value / (n / t_dec), 3),
        "timing": "host wall clock, one synchronisation per round (the next round's first token is read back)"}),
        flush=True)
    if not exact:
        raise SystemExit("speculative decoding diverged from the greedy decode")


# ------------------------------------------------------------ GPU arm

def run_gpu(args):
    import torch
    import torch.distributed as dist
    from bit_exact_speculative_gb300 import build
    from bit_exact_speculative_gb300 import xv
    from bit_exact_speculative_gb300.replicas import job_throughput

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if rank == 0:
        build.build()
    if world > 1:
        dist.barrier()
    xv.lib()
    xv.xv_set_overlap(not args.no_overlap)

    cfg, w_host, stk, toks = make_stack(args, device, rank)
    B, k = args.batch, args.k
    tok_dev = torch.from_numpy(toks).to(device)
    stream = torch.cuda.current_stream()
    rnd = 0

    def step(i):
        stk.verify_commit(tok_dev[i], k)

    for _ in range(args.warmup):
        step(rnd)
        rnd += 1
    xv.xv_device_check()

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- timed region: K steps on device-resident inputs
    launches0 = xv.xv_launch_count()
    clk = ClockSampler(local).__enter__()
    clk.wait_first()
    barrier()
    torch.cuda.synchronize()
    t_region0 = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step(rnd)
        rnd += 1
    e1.record(stream)
    torch.cuda.synchronize()
    t_region1 = time.time()
    barrier()
    launches = xv.xv_launch_count() - launches0
    ms = e0.elapsed_time(e1)
    value, s_max, _ = job_throughput(ms / 1e3, B * k * args.steps, device)   # all ranks' tokens / slowest
    ms_max = s_max * 1e3
    code = xv.xv_device_check()

    # ---- per-kernel durations (serialised: every launch bracketed by events, which breaks the
    # programmatic overlap; used for shares only)
    xv.xv_trace_enable(64 * args.steps)
    for _ in range(args.steps):
        step(rnd)
        rnd += 1
    torch.cuda.synchronize()
    recs = xv.xv_trace_read()
    xv.xv_trace_disable()
    per_kind = {}
    for name, tms, nb in recs:
        d = per_kind.setdefault(name, [0, 0.0, 0])
        d[0] += 1
        d[1] += tms
        d[2] += nb
    # ---- the dominant kernel as it runs in the step: the step's GEMMs back to back
    gemm_ms_per_launch, gemm_bytes_per_launch, _ = gemm_chain_ms(xv, stk, cfg, B * k, max(2, args.steps // 5), device)
    achieved = gemm_bytes_per_launch / (gemm_ms_per_launch / 1e3) / 1e9
    peak, peak_kind = peaks()
    gemm_bytes_step = sum(2 * N * K + 2 * B * k * K + B * k * N * o for N, K, o in gemm_shapes(cfg, B * k))
    traffic_ratio = traffic_ratio_from_profile(os.path.join(ROOT, "bit_exact_speculative_gb300", "csrc", "gemm.cu"))
    n_gemm = len(gemm_shapes(cfg, B * k))

    # ---- end to end through the public API: pinned host tokens in, results out, every step
    h_tok = torch.from_numpy(toks[rnd: rnd + args.steps].copy()).pin_memory()
    # the step's argmax ids and accept counts, read back in one copy (HybridStack keeps them side
    # by side: argmax [B * kmax] then n_accept [B])
    h_res = torch.empty(stk.results.shape, dtype=torch.int32).pin_memory()
    stk_results_bytes = stk.results.numel() * 4
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        # one call: the drafts copied in, verify + commit, the results copied out
        stk.step_host(h_tok[i], h_res)
        stream.synchronize()
    e2e_s = time.perf_counter() - t0
    t_loaded = time.time()
    clk.__exit__(None, None, None)
    clocks = clk.summary(t_region0, t_region1, t_loaded)
    e2e_value, _, _ = job_throughput(e2e_s, B * k * args.steps, device)
    barrier()

    rooflines, more = None, None
    if rank == 0 and world == 1 and not args.no_kernel_rooflines:
        wd = stk.wd
        del stk
        torch.cuda.empty_cache()
        more = {}
        for bb, ctx in ((1, 131072), (8, 2183), (8, 131072)):
            if (bb, ctx) != (B, args.context):
                more[f"batch{bb}_ctx{ctx}"] = step_line(args, device, w_host, wd, bb, ctx)
        del wd
        torch.cuda.empty_cache()
        rooflines = kernel_rooflines(xv, device, peak)

    out = None
    if rank == 0:
        out = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "batch_per_gpu": B, "k": k, "context": args.context,
                       "parallelism": f"replicas x{world}", "overlap": not args.no_overlap,
                       "kv_cache": f"paged, {args.page_size}-position pages" if args.page_size else "contiguous",
                       "gdn_layer": "complete (conv 4, gated norm, 16 q/k heads)" if args.full_gdn else
                                    "recurrence only (32 q/k/v heads)",
                       "weights": "GEMM weights in the tiled layout (128 x 64 tiles contiguous)",
                       "l2": "inputs larger than L2 (4.4 GB of weights per step)"},
            "gpu_launches": int(launches),
            "roofline": {"bound": "hbm", "kernel": "gemm_small_m", "achieved": round(achieved, 1),
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": (round(traffic_ratio * gemm_bytes_per_launch) if traffic_ratio else None),
                         "traffic_source": ("ncu dram bytes per algorithmic byte of the down projection (M=8) "
                                            "x this launch average" if traffic_ratio else None),
                         "algorithmic_bytes_per_launch": round(gemm_bytes_per_launch),
                         "launches_per_step": n_gemm, "ms_per_launch": round(gemm_ms_per_launch, 5),
                         "timing": "the step's GEMMs alone, back to back with programmatic launch as in the step, "
                                   "CUDA events around the chain"},
            "step_roofline": {"algorithmic_bytes": gemm_bytes_step,
                              "achieved_gbs": round(gemm_bytes_step / (ms_max / args.steps / 1e3) / 1e9, 1),
                              "frac": round(gemm_bytes_step / (ms_max / args.steps / 1e3) / 1e9 / peak, 4)},
            "kernels": {n: {"launches": v[0], "ms_total": round(v[1], 4),
                            "share": round(v[1] / max(sum(x[1] for x in per_kind.values()), 1e-9), 4)}
                        for n, v in sorted(per_kind.items(), key=lambda kv: -kv[1][1])},
            "kernels_timing": "every launch bracketed by events (serialised, no programmatic overlap): shares only",
            "more_configs": more,
            "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": int(B * k * 4),
                    "d2h_bytes_per_step": int(stk_results_bytes)},
            "clocks": clocks,
            "kernel_rooflines": rooflines,
            "device_error_bits": code,
        }
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return out, (cfg, w_host)


# ------------------------------------------------------------- CPU side

def oracle_session(args, cfg, w):
    """The oracle holding sequence 0 of the same workload (weights, caches, states, context)."""
    import oracle
    from synth import workloads
    L = args.context
    Lmax = L + 4 * (args.steps + args.warmup) + 64
    oracle.build()
    st = oracle.Stack(workloads.oracle_cfg(cfg), w, Lmax)
    for l, kd in enumerate(cfg["kinds"]):
        if kd == 0:
            st.S[l][...] = workloads.gdn_state(cfg, 0, l, 1)[0]
        else:
            kc, vc = workloads.kv_cache(cfg, 0, l, 1, [L], Lmax)
            st.kc[l][...], st.vc[l][...] = kc[0], vc[0]
    st.len = L
    toks = workloads.draft_tokens(cfg, 0, 0, 1, 4 * (args.steps + args.warmup) + 8)[0]
    return st, toks


def cores_used():
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def oracle_sample(args, cfg, w, budget_s=12.0):
    """The oracle decoding verify positions of the same workload until ~budget_s of CPU time."""
    st, toks = oracle_session(args, cfg, w)
    n, t0 = 0, time.perf_counter()
    limit = min(len(toks), st.Lmax - st.len)
    while n < limit and (n == 0 or time.perf_counter() - t0 < budget_s):
        st.decode(int(toks[n]))
        n += 1
    dt = time.perf_counter() - t0
    return {"value": round(n / dt, 4), "unit": UNIT, "cores": cores_used(), "kind": "oracle",
            "sample": f"{n} verify positions of one sequence ({n / args.k:.1f} verify steps of k = {args.k}; the "
                      f"oracle verifies by decoding them one at a time), context {args.context}, full-size "
                      f"weights; {dt:.1f} s"}


def oracle_configs(args, cfg, w):
    """The oracle on the other configurations, one bounded sample each, in the units of the GPU
    figures beside it (µs per call; positions per second for the step): the 17408-wide GEMMs at
    M = 1 and 16, GDN verify of one sequence (1 replayed and 8 speculative steps of 32 heads of
    128 x 128), the decode-row attention of one sequence (8 rows, 24 q / 4 kv heads of 256) at 640,
    2183 and 131072 positions, and the verify step at context 131072.  The oracle takes sequences
    one after another, so its batch-8 figures are 8 x the per-sequence time (its rate per position
    stays the same)."""
    import types
    import numpy as np
    import oracle
    rng = np.random.default_rng(0)

    def bf16(shape, scale=1.0):
        x = (rng.standard_normal(int(np.prod(shape)), dtype=np.float32) * scale).reshape(shape)
        return (x.view(np.uint32) >> 16).astype(np.uint16)   # truncated: the values do not matter here

    def timed(fn, reps=1):
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        return (time.perf_counter() - t0) / reps * 1e6

    out = {"cores": cores_used(), "kind": "oracle"}
    gemm = {}
    for name, (N, K) in (("up17408", (17408, 5120)), ("down17408", (5120, 17408))):
        W = bf16((N, K), 0.02)
        for M in (1, 16):
            X = bf16((M, K))
            gemm[f"{name}_M{M}"] = round(timed(lambda: oracle.gemm(X, W)), 1)
        del W
    out["gemm_sweep_us"] = gemm
    H, D, k = 32, 128, 8
    S = rng.standard_normal((H, D, D)) * 0.1
    q, kk, v = bf16((k + 1, H, D)), bf16((k + 1, H, D)), bf16((k + 1, H, D))
    beta, gate = bf16((k + 1, H)), bf16((k + 1, H))

    def gdn():
        St = S.copy()
        for t in range(k + 1):
            oracle.gdn_step_heads(St, q[t], kk[t], v[t], beta[t], gate[t], True)
    out["gdn_verify_us_per_sequence"] = round(timed(gdn), 1)
    attn = {}
    for L in (640, 2183, 131072):
        R = 8 if L < 100000 else 1   # one of the 8 rows at 131072, scaled by 8
        kc, vc = bf16((4, L + 8, 256)), bf16((4, L + 8, 256))
        qq = bf16((R, 24, 256))
        attn[f"L{L}"] = round(timed(lambda: oracle.attn_rows(qq, kc, vc, L, 256 ** -0.5)) * (8 // R), 1)
        del kc, vc
    out["attn_decode_rows_us_per_sequence"] = attn
    st, toks = oracle_session(types.SimpleNamespace(context=131072, steps=1, warmup=1), cfg, w)
    n, t0 = 0, time.perf_counter()
    while n == 0 or (n < 4 and time.perf_counter() - t0 < 5.0):
        st.decode(int(toks[n]))
        n += 1
    out["step_ctx131072"] = {"value": round(n / (time.perf_counter() - t0), 4), "unit": UNIT,
                             "sample": f"{n} verify positions of one sequence decoded one at a time"}
    out["sample"] = ("one call per GEMM shape and per attention length (at 131072 one of the 8 rows, "
                     "scaled by 8), one GDN verify, 1-4 positions of the 131072-position step")
    return out


def run_reference(args):
    """The oracle as the reference arm: each step verifies one position of the workload on the host
    cores (verify = sequential decode by definition); value = positions per second."""
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    from synth import workloads
    cfg = workloads.STACK
    w = workloads.weights(cfg, seed=0)
    st, toks = oracle_session(args, cfg, w)
    i = 0
    for _ in range(args.warmup):
        st.decode(int(toks[i]))
        i += 1
    t0 = time.perf_counter()
    for _ in range(args.steps):
        st.decode(int(toks[i]))
        i += 1
    dt = time.perf_counter() - t0
    value = args.steps / dt
    cb = {"value": round(value, 4), "unit": UNIT, "cores": cores_used(), "kind": "oracle",
          "sample": f"{args.steps} verify positions of one sequence decoded one at a time, context "
                    f"{args.context}, full-size weights; {dt:.1f} s"}
    return {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "batch_per_gpu": 1, "k": args.k, "context": args.context},
            "cpu_baseline": cb, "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    if args.kernel:
        run_one_kernel(args)
        return
    if args.speculative is not None:
        run_speculative(args)
        return
    if args.prefill:
        run_prefill(args)
        return
    if args.impl == "reference":
        out = run_reference(args)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    out, (cfg, w) = run_gpu(args)
    rank, world, _ = dist_env()
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = oracle_sample(args, cfg, w)
            out["cpu_configs"] = oracle_configs(args, cfg, w)
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Benchmark of the MoE FFN decode layer on GB300.

Default workload: the Large layer (H=7168, 512 routed experts, top-16,
F=2048, shared expert F=2048, 4-bit affine group-64 experts, 8-bit router)
decoding B=1 token per step, every expert resident in HBM.  A step is one
full pass of the layer: router GEMV + softmax/top-k + grouping, gate|up +
SwiGLU of the 16 routed experts and the shared expert, down projection and
the weighted combine.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--batch B]
                  [--impl ours|reference]

One JSON line on rank 0.  `value` is tokens/s over all ranks (each rank runs
an independent replica of the layer: the path has no cross-GPU exchange).
`--impl reference` times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer decode tokens/s + achieved HBM GB/s vs ~8 TB/s peak (B=1/4/16)"
WORKLOAD = "large-decode"
NOMINAL_HBM_GBS = 8000.0
# What the decode path computes in: activations as 16-bit fixed point (one
# power-of-two exponent per 32 inputs, per 8 for h) times the 4-bit codes,
# summed exactly in int32 by dp4a; scale/bias, SwiGLU and the combine in f32.
DTYPE = "int16 fixed-point x uint4 -> int32 (dp4a), f32 scale/bias/SwiGLU/combine"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "ffn_b1_kernel_large_decode_b1.txt")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--batch", type=int, default=1)
    p.add_argument("--pool", type=int, default=64, help="distinct hidden-state batches rotated")
    p.add_argument("--windows", type=int, default=5,
                   help="timed windows of K steps each; the value is the median window")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--experts", type=int, default=0,
                   help="shrink the routed-expert count (small layers for ncu captures only; with "
                        "--streamed-only also the slots, E/8, and the steps, --steps)")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the B=4/16 lines, e2e, per-kernel and CPU-baseline passes")
    p.add_argument("--prefill-only", action="store_true",
                   help="only the prefill-chunk measurement (mid-prefill, T=128), one JSON object")
    p.add_argument("--streamed", action="store_true",
                   help="the streamed-cache workload (4 large layers, experts in pinned host "
                        "memory, 64 HBM slots per layer, 256 B=1 steps, with and without the "
                        "router lookahead; ~51 GB of host RAM) also with --no-extras; the default "
                        "run includes it at N=1")
    p.add_argument("--no-streamed", action="store_true",
                   help="leave the streamed-cache workload out of the default run")
    p.add_argument("--streamed-only", action="store_true",
                   help="only the streamed-cache workload, one JSON object")
    p.add_argument("--mid-only", action="store_true",
                   help="only the mid-decode leg (B=1/4/16 over rotated layer copies), one JSON object")
    p.add_argument("--mid-batch", type=int, default=0,
                   help="mid-decode leg at this one batch size only (0: B = 1, 4 and 16)")
    p.add_argument("--copies", type=int, default=16,
                   help="mid-decode layer copies rotated step by step (fewer for ncu captures only)")
    p.add_argument("--rvq-only", action="store_true",
                   help="only the residual-VQ expert decode (large shape, B=1 and 4), one JSON object")
    a = p.parse_args()
    a.warmup = max(a.warmup, 3)
    return a


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [v.strip() for v in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        win = [p for t, p in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        if not win and self.samples:
            win = [min(self.samples, key=lambda s: abs(s[0] - t1))[1]]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(p[1]) for p in win if num(p[1]) is not None]
        mx = [num(p[2]) for p in win if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(win),
                "power_w_max": max((num(p[3]) or 0.0) for p in win)}


# ----------------------------------------------------------------- helpers

def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v: float, device) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def record_bytes_unpadded(H, F):
    return 3 * (F * H // 2) + 3 * (F * H // 64) * 4


def layer_step_bytes(s, B, distinct: float, with_f32: bool) -> dict:
    """Algorithmic bytes of one step: every weight byte of the distinct active
    experts, the shared expert and the router once, activations once."""
    rec, sh = record_bytes_unpadded(s.H, s.F), record_bytes_unpadded(s.H, s.Fs) if s.Fs else 0
    router = s.E * s.H + s.E * (s.H // 64) * 4
    act = B * s.H * 2 + B * s.H * (2 + (4 if with_f32 else 0)) + B * s.k * 8
    gateup_w = lambda F: 2 * (F * s.H // 2) + 2 * (F * s.H // 64) * 4
    down_w = lambda F: s.H * F // 2 + (s.H * F // 64) * 4
    pairs = B * s.k
    gateup = distinct * gateup_w(s.F) + (gateup_w(s.Fs) if s.Fs else 0) + B * s.H * 2 + \
        (pairs * s.F + B * s.Fs) * 4
    # the single-token fused kernel: every gate|up and down weight byte of
    # the step's experts once, the token in, the output out (bf16 + f32)
    fused = distinct * (gateup_w(s.F) + down_w(s.F)) + \
        ((gateup_w(s.Fs) + down_w(s.Fs)) if s.Fs else 0) + B * s.H * (2 + 2 + (4 if with_f32 else 0))
    return {"step": distinct * rec + sh + router + act, "gateup": gateup, "fused": fused}


def gpu_id_for(device_index: int) -> str:
    import torch
    try:
        p = torch.cuda.get_device_properties(device_index)
        return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
    except Exception:
        return str(device_index)


def decode_b1_code_hash() -> str:
    """sha256 (16 hex digits) of decode_b1.cu's code: '//' comments and
    blank space removed, so a comment-only edit keeps the capture valid."""
    src = os.path.join(ROOT, "quantized_routed_expert_gemv_gb300", "csrc", "decode_b1.cu")
    lines = []
    for ln in open(src, encoding="utf-8").read().splitlines():
        code = ln.split("//", 1)[0].strip()
        if code:
            lines.append(" ".join(code.split()))
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def read_traffic():
    """dram bytes per launch of the single-token fused kernel from the
    committed ncu summary, or None when the kernel source changed since the
    capture."""
    try:
        lines = open(PROFILE_SUMMARY).read().splitlines()
    except OSError:
        return None
    kv = {}
    for ln in lines:
        if ":" in ln and not ln.startswith(" "):
            k, v = ln.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("decode_b1_cu_code_sha256_16") != decode_b1_code_hash():
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------- reference arm

class _OracleSlices:
    """One token of the layer through the fp64 oracle, cut into bounded
    slices: the router, then per selected expert (and the shared expert)
    128-row blocks of its gate and up rows (SwiGLU after the last block) and
    448-row blocks of its down rows, added into the output with the routing
    weight.  Every slice is the oracle's own arithmetic (route, gemv4, silu)
    on a part of the token; a token is complete after all its slices."""

    GU_ROWS, DN_ROWS = 128, 448

    def __init__(self, orc, oracle, synth, wl, s):
        self.orc, self.oracle, self.synth, self.wl, self.s = orc, oracle, synth, wl, s
        self.L = {F: oracle.record_layout(s.H, F) for F in {s.F, s.Fs} if F}
        self.tokens_done = 0
        self.plan = []

    def _new_token(self, x_bits):
        s, orc = self.s, self.orc
        self.x_bits = x_bits
        self.x = self.synth.bf16_bits_to_float(x_bits).astype(np.float64)
        self.out = np.zeros(s.H)
        self.plan = [("route", None)]

    def _expert_slices(self, rec, F, p):
        s = self.s
        L = self.L[F]
        g = np.zeros(F)
        u = np.zeros(F)
        st = {"h": None}
        sl = []
        gc = rec[L["gate_codes"]:L["up_codes"]]
        uc = rec[L["up_codes"]:L["down_codes"]]
        dc = rec[L["down_codes"]:L["gate_sb"]]
        gs = rec[L["gate_sb"]:L["up_sb"]].view(np.uint32)
        us = rec[L["up_sb"]:L["down_sb"]].view(np.uint32)
        ds = rec[L["down_sb"]:L["bytes"]].view(np.uint32)
        H, G = s.H, s.H // 64
        for r0 in range(0, F, self.GU_ROWS):
            r1 = min(F, r0 + self.GU_ROWS)

            def gu(r0=r0, r1=r1):
                n = r1 - r0
                g[r0:r1] = self.oracle.gemv4(gc[r0 * H // 2:r1 * H // 2], gs[r0 * G:r1 * G], n, H, self.x)
                u[r0:r1] = self.oracle.gemv4(uc[r0 * H // 2:r1 * H // 2], us[r0 * G:r1 * G], n, H, self.x)
                if r1 == F:
                    st["h"] = np.array([self.oracle.silu(float(v)) for v in g]) * u
            sl.append(gu)
        Gd = F // 64
        for r0 in range(0, H, self.DN_ROWS):
            r1 = min(H, r0 + self.DN_ROWS)

            def dn(r0=r0, r1=r1):
                y = self.oracle.gemv4(dc[r0 * F // 2:r1 * F // 2], ds[r0 * Gd:r1 * Gd], r1 - r0, F, st["h"])
                self.out[r0:r1] += p * y
            sl.append(dn)
        return sl

    def prepare(self, x_bits):
        """Untimed: records the next slice needs (a new token routes first)."""
        if not self.plan:
            self._new_token(x_bits)

    def step(self):
        """Runs one slice (timed by the caller); returns True when a token finished."""
        kind, fn = self.plan.pop(0)
        if kind == "route":
            _, ids, p = self.orc.route(self.x_bits)
            work = []
            for e, pe in zip(ids, p):
                rec = self.synth.expert_record(self.wl.weight_seed, 0, int(e), self.s.H, self.s.F)
                work += self._expert_slices(rec, self.s.F, float(pe))
            if self.s.Fs:
                work += self._expert_slices(self.orc._shared, self.s.Fs, 1.0)
            self.plan = [("slice", f) for f in work]
            self._n_slices = len(self.plan) + 1
            return False
        fn()
        if not self.plan:
            self.tokens_done += 1
            return True
        return False


def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    from quantized_routed_expert_gemv_gb300 import synth

    wl = synth.WORKLOADS[WORKLOAD]
    s = wl.shape
    rc, rsb = synth.router(wl.weight_seed, 0, s.E, s.H)
    shared = synth.expert_record(wl.weight_seed, 0, s.E, s.H, s.Fs)
    orc = oracle.Layer(s.H, s.E, s.k, s.F, s.Fs, {}, shared, rc, rsb)
    B = args.batch
    sl = _OracleSlices(orc, oracle, synth, wl, s)
    tok = [0]

    def one_step():
        if not sl.plan:
            sl.prepare(synth.hidden(wl.input_seed, 1000 + (tok[0] // B) % args.pool, tok[0] % B, s.H))
            tok[0] += 1
        t0 = time.perf_counter()
        sl.step()
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        one_step()
    done0, frac0 = sl.tokens_done, _frac(sl)
    total = sum(one_step() for _ in range(args.steps))
    tokens = (sl.tokens_done - done0) + (_frac(sl) - frac0)
    value = tokens / total
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(s, B),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} timed slices (router, 128-row gate|up blocks, "
                                   f"448-row down blocks) of B={B} token(s), {tokens:.3f} tokens of "
                                   "work, single-threaded fp64 C oracle"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def _frac(sl):
    """Fraction of the current token's slices already done."""
    if not sl.plan or not hasattr(sl, "_n_slices"):
        return 0.0
    return 1.0 - len(sl.plan) / sl._n_slices


def config_dict(s, B, windows=1):
    return {"workload": f"{WORKLOAD}: H={s.H} E={s.E} top-{s.k} F={s.F} Fs={s.Fs}, "
                        f"4-bit affine group-64 experts, 8-bit router, all experts in HBM",
            "batch": B, "hidden": s.H, "experts": s.E, "top_k": s.k, "ffn": s.F,
            "shared_ffn": s.Fs,
            "l2": "inputs larger than L2: >=425 MB of distinct weights per step, hidden "
                  "states rotated over a pool of distinct batches",
            "graphs": f"{GRAPH_STEPS} consecutive steps per CUDA graph replay (the remainder "
                      "of K as one-step graphs); every step is a full layer call",
            "timing": f"{windows} timed windows of K steps; value from the median window"}


# ----------------------------------------------------------------- our arm

GRAPH_STEPS = 16  # consecutive steps captured in one CUDA graph


def time_graphs(torch, graphs, chunks, K, W, stream, world, device, windows=1):
    """W warm-up steps, then `windows` timed windows of exactly K steps each:
    K // GRAPH_STEPS replays of the multi-step graphs (rotating over the
    pool) and the remainder as single-step graphs; without multi-step graphs,
    K single-step replays.  Every window is bracketed by a barrier and a
    synchronize and timed with CUDA events on the launching stream.  Returns
    (per-window ms over all ranks (max), t0, t1)."""
    for i in range(W):
        graphs[i % len(graphs)].replay()
    torch.cuda.synchronize()
    out = []
    t_first = None
    for w in range(windows):
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        t_first = t0 if t_first is None else t_first
        with torch.cuda.stream(stream):
            e0.record(stream)
            n_multi = K // GRAPH_STEPS if chunks else 0
            for i in range(n_multi):
                chunks[(i + w) % len(chunks)].replay()
            for i in range(K - n_multi * GRAPH_STEPS):
                graphs[i % len(graphs)].replay()
            e1.record(stream)
        torch.cuda.synchronize()
        t1 = time.time()
        barrier(world)
        out.append(max_over_ranks(world, e0.elapsed_time(e1), device))
    return out, t_first, t1


def window_stats(ms_list, K):
    """Median window and the spread of the windows, per step."""
    per = sorted(m / K for m in ms_list)
    return {"ms_per_step": statistics.median(per), "windows": len(per),
            "spread_ms_per_step": [per[0], per[-1]],
            "spread_pct": 100.0 * (per[-1] - per[0]) / statistics.median(per)}


def kernel_times(torch, moe, dl, x, outs, stream, pool, n=100):
    """Per-kernel CUDA-event durations (ms) of the dispatch's kernels: the
    profiling hook records events between them and launches without
    programmatic dependent launch.  Returns the three intervals averaged."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in evs:               # torch creates the CUDA event on its first record
        e.record(stream)
    torch.cuda.synchronize()
    moe.moe_set_profile_events(dl.handle, [e.cuda_event for e in evs])
    sums = [0.0, 0.0, 0.0]
    with torch.cuda.stream(stream):
        for i in range(n + 5):
            dl.decode(x[i % pool], outs, stream.cuda_stream)
            evs[3].synchronize()
            if i >= 5:
                for j in range(3):
                    sums[j] += evs[j].elapsed_time(evs[j + 1])
    moe.moe_set_profile_events(dl.handle, None)
    return [v / n for v in sums]


def run_ours(args, world, rank, local):
    import torch

    from quantized_routed_expert_gemv_gb300 import moe, synth
    from quantized_routed_expert_gemv_gb300.device import DeviceLayer, bf16_tensor

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if args.prefill_only:
        peaks = _peaks()
        stream = torch.cuda.Stream(device)
        res = run_prefill(args, device, stream, peaks.get("hbm_gbs", 6800.0), peaks.get("bf16_tflops", 1900.0))
        if rank == 0:
            print(json.dumps({"prefill": res}), flush=True)
        return
    if args.rvq_only:
        stream = torch.cuda.Stream(device)
        res = run_rvq(args, device, stream, _peaks().get("hbm_gbs", 6800.0))
        if rank == 0:
            print(json.dumps({"rvq": res}), flush=True)
        return
    if args.mid_only:
        stream = torch.cuda.Stream(device)
        res = run_mid_decode(args, device, stream, _peaks().get("hbm_gbs", 6800.0), world)
        if rank == 0:
            print(json.dumps({"mid_decode": res}), flush=True)
        return
    if args.streamed_only:
        stream = torch.cuda.Stream(device)
        res = run_streamed(args, device, stream, _peaks().get("hbm_gbs", 6800.0))
        if rank == 0:
            print(json.dumps({"streamed": res}), flush=True)
        return
    streamed = (args.streamed or not args.no_extras) and not args.no_streamed and world == 1
    wl = synth.WORKLOADS[WORKLOAD]
    s = wl.shape
    if args.experts:
        s = synth.Shape(s.H, args.experts, s.k, s.F, s.Fs)
    batches = [args.batch] if args.no_extras else sorted({args.batch, 1, 4, 16})
    maxB = max(batches)
    # the same layer also takes 128-token prefill chunks (the large-prefill line)
    dl = DeviceLayer(s, wl.weight_seed, max_tokens=maxB if args.no_extras else max(maxB, 128), device=device)
    stream = torch.cuda.Stream(device)

    def make(B):
        xs = np.stack([np.stack([synth.hidden(wl.input_seed, 1000 + p, t, s.H) for t in range(B)])
                       for p in range(args.pool)])
        x = bf16_tensor(xs, device)
        outs = dl.outputs(B)
        graphs = []
        with torch.cuda.stream(stream):
            dl.decode(x[0], outs, stream.cuda_stream)  # warm the path before capture
        torch.cuda.synchronize()
        distinct = []
        for p in range(args.pool):
            with torch.cuda.stream(stream):
                dl.decode(x[p], outs, stream.cuda_stream)
            stream.synchronize()
            distinct.append(len(np.unique(outs[2].cpu().numpy())))
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                dl.decode(x[p], outs, stream.cuda_stream)
            graphs.append(g)
        # multi-step graphs: GRAPH_STEPS consecutive steps over consecutive
        # pool batches each, as a decode loop captures many layer calls at once
        chunks = []
        for c0 in range(0, max(1, args.pool - GRAPH_STEPS + 1), GRAPH_STEPS):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for p in range(c0, c0 + GRAPH_STEPS):
                    dl.decode(x[p % args.pool], outs, stream.cuda_stream)
            chunks.append(g)
        torch.cuda.synchronize()
        return xs, x, outs, graphs, chunks, float(np.mean(distinct))

    results = {}
    clocks = ClockSampler(gpu_id_for(local))
    clocks.start()
    time.sleep(0.3)
    main = None
    peaks = _peaks()
    peak = peaks.get("hbm_gbs", 6800.0)
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    for B in batches:
        xs, x, outs, graphs, chunks, distinct = make(B)
        K = args.steps if B == args.batch else min(args.steps, 2000)
        nwin = args.windows if B == args.batch else min(args.windows, 3)
        ms_list, t0, t1 = time_graphs(torch, graphs, chunks, K, args.warmup, stream, world, device, nwin)
        assert dl.check(stream.cuda_stream) == moe.MOE_OK, moe.last_error()
        st = window_stats(ms_list, K)
        msps = st["ms_per_step"]
        nbytes = layer_step_bytes(s, B, distinct, with_f32=True)
        r = {"tokens_per_s": B * world / (msps / 1e3), "ms_per_step": msps,
             "windows": st["windows"], "spread_ms_per_step": st["spread_ms_per_step"],
             "spread_pct": st["spread_pct"], "distinct_experts": distinct, "bytes_per_step": nbytes["step"],
             "layer_gbs": nbytes["step"] / (msps / 1e3) / 1e9,
             "gpu_launches_per_step": moe.lib().moe_decode_kernels(dl.handle, B)}
        r["layer_frac_of_8tbs"] = r["layer_gbs"] / NOMINAL_HBM_GBS
        if not args.no_extras:
            per = kernel_times(torch, moe, dl, x, outs, stream, args.pool, n=min(args.steps, 200))
            # one token: the router, then the fused gate|up + down kernel (the
            # third interval is empty); 2..16 tokens: the router, the few-token
            # fused kernel, then the combine
            fused = (B == 1 and per[2] < 0.1 * per[1]) or (2 <= B <= 16 and r["gpu_launches_per_step"] == 3)
            key = "fused" if fused else "gateup"
            kname = ("ffn_b1_kernel" if B == 1 else "ffn_bt_kernel") if fused else \
                ("gateup_b1_kernel" if B == 1 else "gateup_kernel")
            achieved = nbytes[key] / (per[1] / 1e3) / 1e9
            r["kernel_ms"] = ({"router": per[0], "ffn": per[1]} if fused and B == 1 else
                              {"router": per[0], "ffn": per[1], "combine": per[2]} if fused else
                              {"router": per[0], "gateup": per[1], "down": per[2]})
            r["kernel"] = {"name": kname, "algorithmic_bytes_per_launch": nbytes[key],
                           "achieved_gbs": achieved, "frac_of_measured_hbm": achieved / peak}
        results[B] = r
        if B == args.batch:
            main = dict(r, K=K, t0=t0, t1=t1, xs=xs, x=x, outs=outs, nbytes=nbytes)
        del graphs, chunks
    time.sleep(0.2)
    clocks.stop()
    clk = clocks.summary(main["t0"], main["t1"])

    out = {"metric": METRIC, "value": main["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": main["ms_per_step"],
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE,
           "data": "synthetic (seeded SplitMix64 layer and hidden states)",
           "config": config_dict(s, args.batch, args.windows),
           "gpu_launches": main["gpu_launches_per_step"] * args.steps * main["windows"],
           "timing": {"windows": main["windows"], "steps_per_window": main["K"],
                      "value_from": "median window", "spread_ms_per_step": main["spread_ms_per_step"],
                      "spread_pct": main["spread_pct"]},
           "clocks": clk,
           "layer": {"gbs": main["layer_gbs"], "frac_of_8tbs": main["layer_frac_of_8tbs"],
                     "bytes_per_step": main["bytes_per_step"],
                     "distinct_experts": main["distinct_experts"]},
           "by_batch": {str(b): {k: v for k, v in r.items()} for b, r in results.items()}}

    if not args.no_extras:
        B = args.batch
        kern = main["kernel"]
        fused = kern["name"] in ("ffn_b1_kernel", "ffn_bt_kernel")
        out["roofline"] = {"bound": "hbm", "kernel": kern["name"], "achieved": kern["achieved_gbs"],
                           "peak": peak, "unit": "GB/s", "frac": kern["achieved_gbs"] / peak,
                           "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                           "traffic": read_traffic() if fused and B == 1 else None,
                           "algorithmic_bytes_per_launch": kern["algorithmic_bytes_per_launch"],
                           "kernel_ms": main["kernel_ms"]}
        x, outs = main["x"], main["outs"]

        # end to end through the host-buffer entry point
        xs = main["xs"]
        hx = torch.from_numpy(xs.view(np.int16)).pin_memory()
        hob = torch.empty((B, s.H), dtype=torch.int16).pin_memory()
        hids = torch.empty((B, s.k), dtype=torch.int32).pin_memory()
        hw = torch.empty((B, s.k), dtype=torch.float32).pin_memory()
        Ke = min(args.steps, 500)
        # the caller's buffers are fixed: their addresses are taken once, as a
        # serving loop would hold them
        px = [hx[p].data_ptr() for p in range(args.pool)]
        args_out = (B, hob.data_ptr(), None, hids.data_ptr(), hw.data_ptr(), dl.ws.data_ptr(), dl.ws_bytes,
                    stream.cuda_stream)
        for i in range(args.warmup):
            moe.moe_decode_host(dl.handle, px[i % args.pool], *args_out)
        barrier(world)
        t0 = time.perf_counter()
        for i in range(Ke):
            moe.moe_decode_host(dl.handle, px[i % args.pool], *args_out)
        dt = max_over_ranks(world, time.perf_counter() - t0, device)
        out["e2e"] = {"value": B * Ke * world / dt, "unit": "tokens/s",
                      "h2d_bytes_per_step": B * s.H * 2,
                      # bf16 output, ids and weights, written by the kernels into mapped host memory
                      "d2h_bytes_per_step": B * s.H * 2 + 2 * B * s.k * 4, "steps": Ke,
                      "entry": "moe_decode_host (pinned host buffers: a kernel copies x from the layer's mapped "
                               "input buffer; the kernels write the outputs, ids and weights into its mapped "
                               "output buffer; sync per step)"}

        if rank == 0 and world == 1:
            out["cpu_baseline"] = cpu_baseline(wl, s)
        # a 128-token prefill chunk of this layer (no router offsets)
        pl = time_prefill(args, dl, s, wl.input_seed, device, stream, peak, peaks.get("bf16_tflops", 1900.0))
        out["prefill_large"] = dict({"workload": f"large-prefill: T=128 token chunks of the {WORKLOAD} layer "
                                                 f"(H={s.H} E={s.E} top-{s.k} F={s.F} Fs={s.Fs})"}, **pl)
    dl.close()
    del x, outs
    main.clear()
    torch.cuda.empty_cache()
    # the streamed cache holds ~51 GB of pinned host records per process:
    # one replica only.  It is bound by the host link, which the machine's
    # other GPUs share: the same leg has measured 79 to 135 tokens/s.
    if streamed:
        out["streamed"] = run_streamed(args, device, stream, peak)
    if not args.no_extras:
        out["mid_decode"] = run_mid_decode(args, device, stream, peak, world)
        out["prefill"] = run_prefill(args, device, stream, peak, peaks.get("bf16_tflops", 1900.0))
        out["rvq"] = run_rvq(args, device, stream, peak)
    if rank == 0:
        print(json.dumps(out), flush=True)


def _peaks() -> dict:
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except OSError:
        return {}




def run_mid_decode(args, device, stream, hbm_peak, world):
    """Decode on the mid layer (H=2048, E=128, top-8, F=768, Fs=2048) at
    B = 1, 4 and 16.  One step reads ~28.6 MB at B=1, far less than L2 (129
    MB), so consecutive steps rotate over 16 distinct copies of the
    layer (synthetic layers 0..15, 3.6 GB): a copy comes back only after the
    other fifteen steps have streamed ~430 MB (B=1) through L2, so each step
    reads its weights from HBM.  Timed like the main leg (16-step graphs, one
    step per copy, median of windows of K steps).  `--copies` lowers the
    copy count for small ncu captures."""
    import torch

    from quantized_routed_expert_gemv_gb300 import moe, synth
    from quantized_routed_expert_gemv_gb300.device import DeviceLayer, bf16_tensor

    wl = synth.WORKLOADS["mid-decode"]
    s = wl.shape
    n_copies = max(1, min(args.copies, 16))
    dls = [DeviceLayer(s, wl.weight_seed, layer=l, max_tokens=16, device=device) for l in range(n_copies)]
    out = {"workload": f"mid-decode: H={s.H} E={s.E} top-{s.k} F={s.F} Fs={s.Fs}, {n_copies} layer "
                       "copies rotated step by step (each step reads HBM, not L2)"}
    K = max(GRAPH_STEPS, min(args.steps, 1024) // GRAPH_STEPS * GRAPH_STEPS)
    for B in ((args.mid_batch,) if args.mid_batch else (1, 4, 16)):
        npool = 2 * GRAPH_STEPS
        x = bf16_tensor(np.stack([np.stack([synth.hidden(wl.input_seed, 3000 + p, t, s.H) for t in range(B)])
                                  for p in range(npool)]), device)
        outs = [d.outputs(B) for d in dls]
        distinct = []
        with torch.cuda.stream(stream):
            for p in range(npool):
                l = p % n_copies
                dls[l].decode(x[p], outs[l], stream.cuda_stream)
                stream.synchronize()
                distinct.append(len(np.unique(outs[l][2].cpu().numpy())))
        chunks = []
        for c0 in range(0, npool, GRAPH_STEPS):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for p in range(c0, c0 + GRAPH_STEPS):
                    l = p % n_copies
                    dls[l].decode(x[p], outs[l], stream.cuda_stream)
            chunks.append(g)
        torch.cuda.synchronize()
        ms_list, _, _ = time_graphs(torch, chunks, chunks, K, max(args.warmup, 3), stream, world, device,
                                    min(args.windows, 3))
        for d in dls:
            assert d.check(stream.cuda_stream) == moe.MOE_OK, moe.last_error()
        st = window_stats(ms_list, K)
        d = float(np.mean(distinct))
        nb = layer_step_bytes(s, B, d, with_f32=True)
        per = kernel_times(torch, moe, dls[0], x, outs[0], stream, npool, n=50)
        kb = nb["fused"]
        out[str(B)] = {"tokens_per_s": B * world / (st["ms_per_step"] / 1e3), "ms_per_step": st["ms_per_step"],
                       "spread_pct": st["spread_pct"], "distinct_experts": d, "bytes_per_step": nb["step"],
                       "layer_gbs": nb["step"] / (st["ms_per_step"] / 1e3) / 1e9,
                       "gpu_launches_per_step": moe.lib().moe_decode_kernels(dls[0].handle, B),
                       "kernel_ms": per, "fused_kernel_gbs": kb / (per[1] / 1e3) / 1e9,
                       "fused_kernel_frac_of_measured_hbm": kb / (per[1] / 1e3) / 1e9 / hbm_peak}
        out[str(B)]["layer_frac_of_8tbs"] = out[str(B)]["layer_gbs"] / NOMINAL_HBM_GBS
        del chunks
    for d in dls:
        d.close()
    return out


def run_prefill(args, device, stream, hbm_peak, bf16_peak):
    """Prefill chunks of the mid-prefill workload (H=2048, E=128, top-8,
    F=768, Fs=2048, per-expert logit offsets ~ N(0,1)): T=128 tokens per
    chunk on the tensor-core path, 8 distinct chunks replayed as CUDA graphs.
    Algorithmic bytes: every distinct selected expert's record, the shared
    record and the router once, plus the activations; flops: 2 x 3 x F x H
    per (token, expert) pair and 2 x 3 x Fs x H per token."""
    from quantized_routed_expert_gemv_gb300 import synth
    from quantized_routed_expert_gemv_gb300.device import DeviceLayer

    wl = synth.WORKLOADS["mid-prefill"]
    s, T = wl.shape, 128
    dl = DeviceLayer(s, wl.weight_seed, beta=synth.beta_for(wl), max_tokens=T, device=device)
    res = time_prefill(args, dl, s, wl.input_seed, device, stream, hbm_peak, bf16_peak)
    dl.close()
    res = dict({"workload": f"mid-prefill: T={T} token chunks, H={s.H} E={s.E} top-{s.k} F={s.F} Fs={s.Fs}, "
                           "per-expert logit offsets ~ N(0,1)"}, **res)
    res["l2"] = "inputs larger than L2: ~344 MB of distinct weights per chunk"
    return res


def time_prefill(args, dl, s, input_seed, device, stream, hbm_peak, bf16_peak, T=128, pool=8):
    """T-token chunks through `dl` on the tensor-core path, `pool` distinct
    chunks replayed as CUDA graphs; the chunk time, bytes, flops and the
    per-phase split (events around router + pack, gate|up, down + combine)."""
    import torch

    from quantized_routed_expert_gemv_gb300 import moe, synth
    from quantized_routed_expert_gemv_gb300.device import bf16_tensor

    xs = [bf16_tensor(np.stack([synth.hidden(input_seed, 2000 + p, t, s.H) for t in range(T)]), device)
          for p in range(pool)]
    outs = dl.outputs(T)
    graphs, distinct = [], []
    with torch.cuda.stream(stream):
        dl.prefill(xs[0], outs, stream.cuda_stream)
    torch.cuda.synchronize()
    for p in range(pool):
        with torch.cuda.stream(stream):
            dl.prefill(xs[p], outs, stream.cuda_stream)
        stream.synchronize()
        distinct.append(len(np.unique(outs[2].cpu().numpy())))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            dl.prefill(xs[p], outs, stream.cuda_stream)
        graphs.append(g)
    K = min(args.steps, 200)
    ms_list, _, _ = time_graphs(torch, graphs, [], K, args.warmup, stream, 1, device, min(args.windows, 3))
    ms = window_stats(ms_list, K)["ms_per_step"] * K
    assert dl.check(stream.cuda_stream) == moe.MOE_OK, moe.last_error()
    d = float(np.mean(distinct))
    rec = record_bytes_unpadded(s.H, s.F)
    nbytes = d * rec + record_bytes_unpadded(s.H, s.Fs) + s.E * s.H + s.E * (s.H // 64) * 4 + T * s.H * 8
    flops = 2.0 * 3 * s.F * s.H * T * s.k + 2.0 * 3 * s.Fs * s.H * T
    sec = ms / K / 1e3
    # per-phase split: events around router+pack, gate|up, down+combine
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in evs:
        e.record(stream)
    torch.cuda.synchronize()
    moe.moe_set_profile_events(dl.handle, [e.cuda_event for e in evs])
    sums = [0.0, 0.0, 0.0]
    with torch.cuda.stream(stream):
        for i in range(20):
            dl.prefill(xs[i % pool], outs, stream.cuda_stream)
            evs[3].synchronize()
            for j in range(3):
                sums[j] += evs[j].elapsed_time(evs[j + 1])
    moe.moe_set_profile_events(dl.handle, None)
    del graphs
    return {"tokens_per_s": T / sec, "ms_per_chunk": sec * 1e3, "distinct_experts": d,
            "bytes_per_chunk": nbytes, "gbs": nbytes / sec / 1e9, "frac_of_measured_hbm": nbytes / sec / 1e9 / hbm_peak,
            "tflops": flops / sec / 1e12, "frac_of_bf16_peak": flops / sec / 1e12 / bf16_peak,
            "phase_ms": {"router_pack": sums[0] / 20, "gateup": sums[1] / 20, "down_combine": sums[2] / 20}}


def h2d_bandwidth(torch, device, nbytes=1 << 30, reps=5) -> float:
    """Pinned host -> device copy bandwidth (GB/s), best of reps."""
    src = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(nbytes, dtype=torch.uint8, device=device)
    best = 0.0
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = max(best, nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9)
    del src, dst
    return best


LOOKAHEAD_RHO = 0.9   # hidden-state correlation between consecutive layers (chained inputs)
LOOKAHEAD_N = 6       # experts read ahead per token
STREAMED_COUNTS = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tests", "golden",
                               "streamed_lfu_counts.txt")
COUNT_KEYS = ("hits", "misses", "evictions", "lookahead_copies", "lookahead_hits")


def streamed_expected() -> dict:
    """{run: [[counter per COUNT_KEYS] per layer]} from the oracle's replay of
    the streamed workload (tests/golden/make_streamed_lfu_counts.py)."""
    out = {}
    try:
        for line in open(STREAMED_COUNTS):
            if line.strip() and not line.startswith("#"):
                f = [c.strip() for c in line.split("|")]
                out.setdefault(f[0], []).append([int(v) for v in f[2:]])
    except OSError:
        pass
    return out


def replay_match(expected, st) -> str:
    """'equal' when every layer's counters equal the oracle's replay."""
    if not expected:
        return "no stored replay"
    diffs = [f"layer {l} {k}: {s[k]} vs {e[i]}" for l, (s, e) in enumerate(zip(st, expected))
             for i, k in enumerate(COUNT_KEYS) if s[k] != e[i]]
    return "equal" if not diffs and len(st) == len(expected) else "differs: " + "; ".join(diffs[:4])


def streamed_shape(args):
    """(workload, shape, layers, slots, steps) of the streamed-cache leg."""
    from quantized_routed_expert_gemv_gb300 import synth
    wl = synth.WORKLOADS["large-streamed"]
    s, nl, slots, steps = wl.shape, wl.layers, 64, 256
    if args.experts:  # a reduced copy for small captures: fewer experts, slots in proportion
        s = synth.Shape(s.H, args.experts, s.k, s.F, s.Fs)
        slots = max(s.k, args.experts // 8)
        steps = min(steps, max(GRAPH_STEPS, args.steps))
    return wl, s, nl, slots, steps


def streamed_hosts(args):
    """The streamed leg's expert records in page-locked host memory, one
    tensor per layer (~51 GB at the full shape)."""
    from quantized_routed_expert_gemv_gb300.device import pinned_records
    wl, s, nl, _, _ = streamed_shape(args)
    return [pinned_records(s, wl.weight_seed, layer=l) for l in range(nl)]


def run_streamed(args, device, stream, hbm_peak, hosts=None):
    """Streamed expert cache: 4 stacked layers of the large shape, all expert
    records in pinned host memory, 64 HBM slots per layer, router offsets
    Zipf(1.1) per layer, 256 consecutive B=1 steps from a cold cache, timed
    end to end (the cache update waits on the router every layer).

    Three runs: (1) hidden states drawn independently per step and layer;
    (2) and (3) hidden states chained across layers (synth.hidden_chain,
    rho = LOOKAHEAD_RHO), without and with the router lookahead: after layer
    l's step is issued, layer l+1's router runs on layer l's hidden state on
    a stream of its own and its first LOOKAHEAD_N experts are read ahead.
    All layers share one copy stream, so lookahead copies queue behind the
    demand copies issued before them."""
    import numpy as np
    import torch

    from quantized_routed_expert_gemv_gb300 import synth
    from quantized_routed_expert_gemv_gb300.device import CachedLayer, DeviceLayer, bf16_tensor, \
        pinned_records

    wl, s, nl, slots, steps = streamed_shape(args)
    bw = h2d_bandwidth(torch, device)
    dls = []
    if hosts is None:
        hosts = streamed_hosts(args)
    for l in range(nl):
        dls.append(DeviceLayer(s, wl.weight_seed, layer=l, beta=synth.beta_for(wl, l)[:s.E], max_tokens=1,
                               device=device, resident=False))
    xs_ind = bf16_tensor(np.stack([np.stack([synth.hidden(wl.input_seed, l, t, s.H)[None] for l in range(nl)])
                                   for t in range(steps)]), device)  # [steps][layers][1][H]
    xs_chain = bf16_tensor(np.stack([synth.hidden_chain(wl.input_seed, t, s.H, nl, LOOKAHEAD_RHO)[:, None]
                                     for t in range(steps)]), device)
    outs = [d.outputs(1) for d in dls]
    copy = torch.cuda.Stream(device)
    side = torch.cuda.Stream(device)
    hbm_bytes = nl * steps * layer_step_bytes(s, 1, s.k, with_f32=True)["step"]

    def caches_new():
        cs = [CachedLayer(dls[l], hosts[l], slots) for l in range(nl)]
        for c in cs:
            c.copy_stream = copy
            c.prepare_lookahead(side.cuda_stream)
        return cs

    def run(n, caches, xs, ahead):
        with torch.cuda.stream(stream):
            for t in range(n):
                for l in range(nl):
                    caches[l].decode(xs[t, l], outs[l], stream.cuda_stream)
                    if ahead and l + 1 < nl:
                        caches[l + 1].lookahead(xs[t, l], LOOKAHEAD_N, stream=side.cuda_stream)

    expected = streamed_expected()

    def measure(xs, ahead, run_name):
        warm = caches_new()
        run(max(args.warmup, 3), warm, xs, ahead)  # kernels and copies warmed on throwaway caches
        torch.cuda.synchronize()
        for c in warm:
            c.close()
        caches = caches_new()
        torch.cuda.synchronize()
        # the cache's host logic is on every step's path: no garbage
        # collection pauses inside the timed run
        gc.collect()
        gc.disable()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        t0 = time.perf_counter()
        run(steps, caches, xs, ahead)
        e1.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        gc.enable()
        ms = e0.elapsed_time(e1)
        for d in dls:
            assert d.check(stream.cuda_stream) == 0
        for c in caches:
            assert c.check_lookahead(stream.cuda_stream) == 0
        st = [c.stats() for c in caches]
        for c in caches:
            c.close()

        def tot(key, layers=range(nl)):
            return sum(st[l][key] for l in layers)

        hits, misses = tot("hits"), tot("misses")
        h2d = tot("bytes_h2d") + tot("lookahead_bytes")
        bound_s = max(hbm_bytes / (hbm_peak * 1e9), h2d / (bw * 1e9))
        later = range(1, nl)
        return {"oracle_replay": replay_match(expected.get(run_name), st),
                "tokens_per_s": steps / (ms / 1e3), "ms_per_token": ms / steps, "wall_s": wall,
                "hit_rate": hits / max(1, hits + misses), "hits": hits, "misses": misses,
                "hit_rate_layers_1_on": tot("hits", later) / max(1, tot("hits", later) + tot("misses", later)),
                "lookahead_copies": tot("lookahead_copies"), "lookahead_hits": tot("lookahead_hits"),
                "bytes_h2d": h2d, "h2d_bytes_per_token": h2d / steps,
                "h2d_gbs_achieved": h2d / (ms / 1e3) / 1e9,
                "bound_ms_per_token": bound_s * 1e3 / steps,
                "frac_of_bound": (bound_s * 1e3 / steps) / (ms / steps)}

    base = measure(xs_ind, False, "independent")
    chained_off = measure(xs_chain, False, "chained_off")
    chained_on = measure(xs_chain, True, "chained_on")
    for d in dls:
        d.close()
    # the same layers with 3-bit residual-VQ expert records (same routers, so
    # the same ids and cache counters; a miss copies 3 bits per weight)
    dls.clear()
    hosts.clear()
    torch.cuda.synchronize()
    for l in range(nl):
        dls.append(DeviceLayer(s, wl.weight_seed, layer=l, beta=synth.beta_for(wl, l)[:s.E], max_tokens=1,
                               device=device, resident=False, rvq=True))
        hosts.append(pinned_records(s, wl.weight_seed, layer=l, rvq=True))
    outs = [d.outputs(1) for d in dls]
    hbm_bytes_4bit = hbm_bytes
    rvq_bytes = lambda F: 3 * (3 * F * s.H // 8)
    hbm_bytes = nl * steps * (s.k * rvq_bytes(s.F) + rvq_bytes(s.Fs) + s.E * s.H + s.E * (s.H // 64) * 4 +
                              s.H * 8 + s.k * 8)
    rvq_run = measure(xs_ind, False, "independent")
    for d in dls:
        d.close()
    del hosts
    res = {"workload": f"large-streamed: {nl} layers of H={s.H} E={s.E} top-{s.k} F={s.F} Fs={s.Fs}, "
                       f"{slots} HBM slots per layer, Zipf(1.1) router offsets, {steps} B=1 steps "
                       "from a cold cache",
           "h2d_gbs_probed": bw, "hbm_bytes_per_token": hbm_bytes_4bit / steps}
    res.update(base)
    res["lookahead"] = {"inputs": f"hidden states chained across layers, rho={LOOKAHEAD_RHO}",
                        "n_ahead": LOOKAHEAD_N, "off": chained_off, "on": chained_on}
    res["rvq_records"] = dict(rvq_run, records="3-bit residual-VQ experts (moe_rvq_record_layout_of), "
                                               "independent inputs", 
                              h2d_bytes_vs_4bit=rvq_run["bytes_h2d"] / max(1, base["bytes_h2d"]))
    return res


def run_rvq(args, device, stream, hbm_peak):
    """Decode on the large shape with 3-bit residual-VQ experts (WASTE page,
    section "Quantization ve doğruluk"), B = 1 and 4, timed as replays of
    CUDA graphs of GRAPH_STEPS consecutive steps like the main leg.
    Algorithmic bytes per step: the code bytes of the distinct experts and
    of the shared expert, the router, the codebooks once, the activations."""
    import numpy as np
    import torch

    from quantized_routed_expert_gemv_gb300 import moe, synth
    from quantized_routed_expert_gemv_gb300.device import DeviceLayer, bf16_tensor

    wl = synth.WORKLOADS["large-decode"]
    s = wl.shape
    if args.experts:
        s = synth.Shape(s.H, args.experts, s.k, s.F, s.Fs)
    dl = DeviceLayer(s, wl.weight_seed, max_tokens=4, device=device, rvq=True)
    rvq_bytes = lambda F: 3 * (3 * F * s.H // 8)
    router = s.E * s.H + s.E * (s.H // 64) * 4
    pool = max(GRAPH_STEPS, min(args.pool, 32))
    K = 256
    out = {"workload": f"large-decode with residual-VQ experts: H={s.H} E={s.E} top-{s.k} F={s.F} Fs={s.Fs}, "
                       "3 code bytes per 8 weights, bf16 codebooks 3 x 3 x 256 x 8",
           "gpu_launches_per_step": moe.lib().moe_decode_kernels(dl.handle, 1)}
    for B in (1, 4):
        xs = np.stack([np.stack([synth.hidden(wl.input_seed, 2000 + p, t, s.H) for t in range(B)])
                       for p in range(pool)])
        x = bf16_tensor(xs, device)
        outs = dl.outputs(B)
        distinct = []
        with torch.cuda.stream(stream):
            for p in range(pool):
                dl.decode(x[p], outs, stream.cuda_stream)
                stream.synchronize()
                distinct.append(len(np.unique(outs[2].cpu().numpy())))
        chunks = []
        for c0 in range(0, pool - GRAPH_STEPS + 1, GRAPH_STEPS):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for p in range(c0, c0 + GRAPH_STEPS):
                    dl.decode(x[p], outs, stream.cuda_stream)
            chunks.append(g)
        torch.cuda.synchronize()
        for i in range(max(args.warmup, 3)):
            chunks[i % len(chunks)].replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for i in range(K // GRAPH_STEPS):
                chunks[i % len(chunks)].replay()
            e1.record(stream)
        torch.cuda.synchronize()
        assert dl.check(stream.cuda_stream) == moe.MOE_OK, moe.last_error()
        ms = e0.elapsed_time(e1) / K
        d = float(np.mean(distinct))
        step_bytes = d * rvq_bytes(s.F) + rvq_bytes(s.Fs) + router + 3 * 3 * 256 * 8 * 2 + \
            B * s.H * (2 + 2 + 4) + B * s.k * 8
        gbs = step_bytes / (ms / 1e3) / 1e9
        # per kernel (events between launches, no programmatic dependent
        # launch): the router, gate|up, then down + combine
        per = kernel_times(torch, moe, dl, x, outs, stream, pool, n=50)
        pair_bytes = B * s.k * rvq_bytes(s.F) + B * rvq_bytes(s.Fs)  # each token reads its own experts
        out[str(B)] = {"tokens_per_s": B / (ms / 1e3), "ms_per_step": ms, "distinct_experts": d,
                       "bytes_per_step": step_bytes, "gbs": gbs, "frac_of_measured_hbm": gbs / hbm_peak,
                       "kernel_ms": {"router": per[0], "gateup": per[1], "down_combine": per[2]},
                       "expert_bytes_read": pair_bytes,
                       "expert_gbs": pair_bytes / ((per[1] + per[2]) / 1e3) / 1e9}
        del chunks
    dl.close()
    return out


def cpu_baseline(wl, s, target_s=15.0):
    import oracle
    from quantized_routed_expert_gemv_gb300 import synth
    rc, rsb = synth.router(wl.weight_seed, 0, s.E, s.H)
    shared = synth.expert_record(wl.weight_seed, 0, s.E, s.H, s.Fs)
    orc = oracle.Layer(s.H, s.E, s.k, s.F, s.Fs, {}, shared, rc, rsb)
    total, n = 0.0, 0
    while total < target_s and n < 32:
        x = synth.hidden(wl.input_seed, 1000 + n, 0, s.H)
        _, ids, _ = orc.route(x)
        for e in ids:
            if int(e) not in orc._recs:
                orc.set_record(int(e), synth.expert_record(wl.weight_seed, 0, int(e), s.H, s.F))
        t0 = time.perf_counter()
        orc.token(x)
        total += time.perf_counter() - t0
        n += 1
        for e in list(orc._recs):
            orc._recs.pop(e)
    return {"value": n / total, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} B=1 tokens of the same workload through the single-threaded fp64 C "
                      f"oracle ({total:.1f} s of CPU time; record generation untimed)"}


def main():
    args = parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

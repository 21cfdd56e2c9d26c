#!/usr/bin/env python
"""Benchmark: tensor-parallel Llama decoder layer, t ranks emulated on one GB300.

One step = one decoder layer forward (RMSNorm, column-parallel qkv + RoPE +
KV write, GQA attention, row-parallel o_proj with the fused t-way reduction,
RMSNorm, column-parallel gate_up + SiLU, row-parallel down_proj with the fused
reduction) of a decode batch: 16 sequences, each one new token attending to a
1024-token KV cache, at the Llama-3.1-8B shape (hidden 4096, 32 Q / 8 KV heads,
head_dim 128, intermediate 14336).  The headline runs t = 8 emulated ranks;
t = 1, 2, 4 are reported beside it.  Seeded synthetic weights ~N(0, 0.02),
KV cache ~N(0, 1), hidden ~N(0, 1).  Steps rotate over 4 layers with distinct
weights and caches (2 GB), so every step streams inputs far larger than L2.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on the
same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sharded-layer tokens/s at Llama-3.1-8B shape, t=1..8; % of HBM/TC roofline"
UNIT = "tokens/s"
WORKLOAD = "llama8b_decode"
LAYER_KINDS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wg", "wu", "wd")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=4000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--t", type=int, default=8)
    p.add_argument("--rotate", type=int, default=4)
    p.add_argument("--fused", type=int, default=1)
    p.add_argument("--per-t", type=int, default=1)
    p.add_argument("--cpu-baseline", type=int, default=1)
    p.add_argument("--prefill", type=int, default=1)
    p.add_argument("--configs", type=int, default=1)
    p.add_argument("--prefill-only", type=int, default=0,
                   help="profiling aid: run only the prefill section and print its JSON")
    p.add_argument("--prefill-bn", type=int, default=0,
                   help="prefill GEMMs' output-feature tile width (0: chosen per GEMM)")
    p.add_argument("--prefill-pairs", type=int, default=0,
                   help="prefill GEMMs on CTA pairs: 0 auto, 1 always, 2 never")
    p.add_argument("--cpu-budget-s", type=float, default=15.0)
    p.add_argument("--reference-budget-s", type=float, default=150.0)
    return p.parse_args()


# ---------------------------------------------------------------------------
# byte accounting (algorithmic: what the method must move once per step)
# ---------------------------------------------------------------------------
def layer_bytes(w, t):
    H, d, I = w.hidden, w.head_dim, w.intermediate
    M = w.tokens
    b = {
        "gemm_qkv": (w.n_heads + 2 * w.n_kv_heads) * d * H * 2 + M * H * 2 + M * (w.n_heads + 2 * w.n_kv_heads) * d * 2,
        "gemm_o": H * w.n_heads * d * 2 + M * w.n_heads * d * 2 + 2 * M * H * 2,
        "gemm_gate_up": 2 * I * H * 2 + M * H * 2 + M * I * 2,
        "gemm_down": H * I * 2 + M * I * 2 + 2 * M * H * 2,
        "attn_decode": w.n_seqs * w.n_kv_heads * w.ctx * d * 2 * 2 + 2 * M * w.n_heads * d * 2,
        "rmsnorm": 2 * M * H * 2 + H * 2,
    }
    # the RMSNorms move no bytes of their own in the method: h is read by the
    # GEMM after each norm anyway (counted there), and up to 32 tokens the
    # library applies the norms inside qkv / gate_up; where a norm kernel
    # runs, its bytes are an implementation cost (b["rmsnorm"] is kept for
    # that kernel's own line)
    total = sum(v for k, v in b.items() if k != "rmsnorm")
    return b, total


def measured_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None when the CUDA sources changed since that capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    d = os.path.join(ROOT, "megatron_tensor_layers_tp_gb300", "csrc")
    h = hashlib.sha256()
    for n in sorted(os.listdir(d)):
        h.update(n.encode())
        with open(os.path.join(d, n), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != rec.get("csrc_sha256"):
        return None
    k = rec.get("kernels", {}).get(kernel)
    return k["dram_bytes_per_launch"] if k else None


def max_over_ranks(x: float, world: int, device: str = "cuda") -> float:
    """The largest of every rank's x (one all-reduce; the replicas share no
    data, this only joins their clocks)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    tm = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(tm, op=dist.ReduceOp.MAX)
    return float(tm.item())


def whole_job_rate(units_per_rank: int, steps: int, ms_max: float, world: int) -> float:
    """Units per second of the whole job: every replica processes the same
    units per step, and the job takes as long as its slowest replica."""
    return world * units_per_rank * steps / (ms_max / 1e3)


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return pk.get("hbm_gbs", 6800.0), pk.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class NvmlSampler:
    """Reads the SM clock and the clock-event reasons through NVML (ctypes,
    read-only queries) every ~0.5 ms from a thread, so that even a timed
    region of a few milliseconds holds samples.  Raises OSError when NVML is
    not available (the nvidia-smi sampler is used then)."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(gpu_index, ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        mx = ctypes.c_uint(0)
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
        self.max_mhz = float(mx.value)
        self.samples = []
        self.on = False
        self.stop_flag = False
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def _run(self):
        ct, lib = self.ct, self.lib
        mhz, rs, mw = ct.c_uint(0), ct.c_ulonglong(0), ct.c_uint(0)
        while not self.stop_flag:
            if self.on:
                lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz))
                lib.nvmlDeviceGetCurrentClocksEventReasons(self.h, ct.byref(rs))
                lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw))
                self.samples.append((float(mhz.value), int(rs.value), mw.value / 1000.0))
            time.sleep(0.0005)

    def start(self):
        self.on = True

    def stop(self):
        self.on = False
        self.stop_flag = True
        self.thread.join(timeout=2)

    def summary(self, *_):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "nvml"}
        reasons = set()
        for _, r, _ in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(m for m, _, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "power_w_max": max(p for _, _, p in self.samples),
                "samples": len(self.samples), "source": "nvml, every ~0.5 ms inside the timed region"}


def clock_sampler(gpu_index: int):
    try:
        return NvmlSampler(gpu_index)
    except (OSError, AttributeError):
        return ClockSampler(gpu_index)


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:  # no nvidia-smi on this machine: no clock samples
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def start(self):
        pass

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [s for ts, s in self.samples if t0 <= ts <= t1]
        adjacent = False
        if not inside:
            near = sorted(self.samples, key=lambda x: min(abs(x[0] - t0), abs(x[0] - t1)))[:3]
            inside = [s for _, s in near]
            adjacent = True
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[1]) for s in inside if num(s[1]) is not None]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for s in inside:
            for name, v in zip(names, s[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": num(inside[0][2]), "reasons": sorted(reasons),
               "power_w_max": max((num(s[3]) or 0) for s in inside), "samples": len(inside)}
        if adjacent:
            out["sampled_adjacent"] = True
        return out


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------
def build(w, t, rotate, head=False):
    import torch
    import synth
    from megatron_tensor_layers_tp_gb300.runtime import TPModel, decode_batch, make_config
    cfg = make_config(w.hidden, w.n_heads, w.n_kv_heads, w.head_dim, w.intermediate, w.vocab,
                      rotate, t, w.rms_eps, w.rope_theta, max_positions=w.l_max)
    layers = []
    for l in range(rotate):
        shapes = synth.weight_shapes(w, l)
        L = {}
        for k in LAYER_KINDS:
            x = torch.empty(shapes[k], dtype=torch.bfloat16, device="cuda")
            if k.endswith("norm"):
                x.fill_(1.0)
            else:
                synth.fill_normal_(x, w.seed, synth.tensor_id(k, l), w.sigma_w)
            L[k] = x
        layers.append(L)
    emb = fn = lm = None
    if head:
        emb = torch.empty((w.vocab, w.hidden), dtype=torch.bfloat16, device="cuda")
        synth.fill_normal_(emb, w.seed, synth.tensor_id("embed"), w.sigma_w)
        lm = torch.empty((w.vocab, w.hidden), dtype=torch.bfloat16, device="cuda")
        synth.fill_normal_(lm, w.seed, synth.tensor_id("lm_head"), w.sigma_w)
        fn = torch.ones(w.hidden, dtype=torch.bfloat16, device="cuda")
    model = TPModel(cfg, layers, emb, fn, lm, max_tokens=w.tokens)
    del layers, emb, lm
    torch.cuda.empty_cache()
    ks, vs = [], []
    for l in range(rotate):
        k = model.alloc_kv(w.n_seqs, w.l_max)
        v = model.alloc_kv(w.n_seqs, w.l_max)
        for cache, kind in ((k, "k_cache"), (v, "v_cache")):
            for cp in range(cfg.kv_copies):
                for b in range(w.n_seqs):
                    synth.fill_normal_(cache[cp, b], w.seed, synth.tensor_id(kind, l), w.sigma_kv,
                                       start=synth.kv_logical_start(w, b, cp * cfg.kv_heads_per_rank))
        ks.append(k)
        vs.append(v)
    batch = decode_batch(w.n_seqs, w.ctx, ks, vs, w.l_max)
    h = torch.empty((w.tokens, w.hidden), dtype=torch.bfloat16, device="cuda")
    synth.fill_normal_(h, w.seed, synth.tensor_id("hidden"), w.sigma_h)
    torch.cuda.synchronize()
    return model, batch, h


def timed_steps(model, batch, h, steps, warmup, rotate, fused, stream, profile=False):
    import torch
    from megatron_tensor_layers_tp_gb300 import binding as B
    cb = batch.to_c()
    ws, nws = model.ws_args
    s = stream.cuda_stream

    def step(i):
        B.check(B.tp_layer_forward(model.handle, i % rotate, cb, h.data_ptr(), fused, ws, nws, s),
                "tp_layer_forward")
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    B.tp_profile(model.handle, profile)
    model.reset_stats()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    B.tp_profile(model.handle, False)
    ms = e0.elapsed_time(e1)
    prof = B.tp_profile_read(model.handle, s) if profile else {}
    launches = model.stats().kernel_launches
    return ms, prof, launches


def step_median_ms(model, batch, h, steps, rotate, fused, stream):
    """Median of per-step CUDA-event durations (events recorded between the
    steps on the launch stream), in a pass of its own: an event between two
    steps ends the programmatic overlap of the steps' kernels, so this pass
    stays out of the headline window."""
    import torch
    from megatron_tensor_layers_tp_gb300 import binding as B
    cb = batch.to_c()
    ws, nws = model.ws_args
    s = stream.cuda_stream
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for i in range(steps):
        B.check(B.tp_layer_forward(model.handle, i % rotate, cb, h.data_ptr(), fused, ws, nws, s),
                "tp_layer_forward")
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    return statistics.median(ev[i].elapsed_time(ev[i + 1]) for i in range(steps))


def run_ours(args, rank, world):
    import torch
    import torch.distributed as dist
    import synth
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    w = synth.WORKLOADS[WORKLOAD]
    stream = torch.cuda.Stream()
    hbm_peak, tc_peak, peak_src = read_peaks()
    with torch.cuda.stream(stream):
        model, batch, h = build(w, args.t, args.rotate)
    gpu_idx = int(os.environ.get("LOCAL_RANK", 0))
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            gpu_idx = int(vis.split(",")[gpu_idx])
        except ValueError:
            pass
    sampler = clock_sampler(gpu_idx)
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_host0 = time.time()
    sampler.start()
    ms, _, launches = timed_steps(model, batch, h, args.steps, args.warmup, args.rotate,
                                  args.fused, stream, profile=False)
    sampler.stop()
    t_host1 = time.time()
    if world > 1:
        dist.barrier()
    clocks = sampler.summary(t_host0, t_host1)
    ms = max_over_ranks(ms, world)
    med_steps = max(20, min(args.steps, 200))
    ms_med = step_median_ms(model, batch, h, med_steps, args.rotate, args.fused, stream)
    # per-kernel durations: the same steps again with two CUDA events recorded
    # around every launch on the launch stream (the brackets cost a few
    # microseconds per launch, so they stay out of the headline region)
    prof_steps = min(args.steps, 2000)
    ms_prof, prof, _ = timed_steps(model, batch, h, prof_steps, 0, args.rotate, args.fused,
                                   stream, profile=True)
    assert model.check_device(stream) == 0, "device status word set"
    ms_step = ms / args.steps
    tokens = w.tokens
    value = whole_job_rate(tokens, args.steps, ms, world)
    model_bytes_per_layer = model.model_bytes() / args.rotate

    kb, step_bytes = layer_bytes(w, args.t)
    kernels = kernel_table(prof, kb, hbm_peak)
    tot_all = sum(tot for _, tot in prof.values()) or 1.0
    for name, (n, tot) in prof.items():
        kernels[name]["share"] = round(tot / tot_all, 3)
    dom = max(prof.items(), key=lambda kv: kv[1][1])[0] if prof else None
    roofline = None
    if dom in kb:
        n, tot = prof[dom]
        avg_s = tot / n * 1e-3
        ach = kb[dom] / avg_s / 1e9
        roofline = {"kernel": dom, "bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak,
                    "unit": "GB/s", "frac": round(ach / hbm_peak, 3),
                    "traffic": measured_traffic(dom),
                    "algorithmic_bytes": kb[dom], "peak_source": peak_src}
    step_gbs = step_bytes / (ms_step * 1e-3) / 1e9

    # the same steps replayed from CUDA graphs (one per rotating layer)
    graphs = [model.capture_layer(l, batch, h, stream, fused=bool(args.fused))
              for l in range(args.rotate)]
    n_g = max(min(args.steps, 2000), 20)
    for i in range(args.warmup):
        graphs[i % args.rotate].launch(stream)
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for i in range(n_g):
        graphs[i % args.rotate].launch(stream)
    g1.record(stream)
    torch.cuda.synchronize()
    ms_graph_step = g0.elapsed_time(g1) / n_g
    for g in graphs:
        g.close()

    # every t, with the fused and the unfused reduction (the unfused one
    # materialises t fp32 partials per row-parallel op and reduces them in a
    # kernel of its own: its extra HBM cost is the measured difference)
    per_t = {}
    if args.per_t and rank == 0 and world == 1:
        n_pt = max(args.steps // 4, 20)

        def one(m_, b_, h_, tt, fused):
            ms_, _, _ = timed_steps(m_, b_, h_, n_pt, args.warmup, args.rotate, fused, stream)
            st_ = ms_ / n_pt
            _, sb_ = layer_bytes(w, tt)
            return {"ms": round(st_, 4), "tok_s": round(tokens / (st_ * 1e-3)),
                    "hbm_frac": round(sb_ / (st_ * 1e-3) / 1e9 / hbm_peak, 3)}
        for tt in (1, 2, 4, 8):
            if tt == args.t:
                m2, b2, h2 = model, batch, h
            else:
                with torch.cuda.stream(stream):
                    m2, b2, h2 = build(w, tt, args.rotate)
            per_t[str(tt)] = {"fused": one(m2, b2, h2, tt, 1), "unfused": one(m2, b2, h2, tt, 0),
                              "unfused_extra_bytes_per_row_op": 2 * tt * w.tokens * w.hidden * 4}
            if m2 is not model:
                m2.close()
                del m2, b2, h2
                torch.cuda.empty_cache()

    # end to end through the public API with host buffers: each step, the
    # library's host-buffer call brings the pinned input rows to the device,
    # runs the layer and writes the result rows back to pinned host memory
    # (kernels reading/writing host memory over NVLink-C2C where the GPU is
    # coherent with its host, volatile loads so every step fetches from host
    # memory; cudaMemcpyAsync elsewhere)
    e2e_steps = max(min(args.steps, 500), 10)
    hin = torch.empty((w.tokens, w.hidden), dtype=torch.bfloat16, pin_memory=True)
    hin.copy_(h.cpu())
    hout = torch.empty_like(hin, pin_memory=True)
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            model.layer_forward_host(i % args.rotate, batch, hin, hout, h, bool(args.fused),
                                     stream=stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    cb = batch.to_c()
    model.reset_stats()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(e2e_steps):
            model.layer_forward_host(i % args.rotate, batch, hin, hout, h, bool(args.fused),
                                     stream=stream, cbatch=cb)
        e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1), world)
    # two more kernels per step than the layer alone: the transfers ran as kernels
    e2e_launches = model.stats().kernel_launches / e2e_steps
    transfer = ("kernels reading/writing pinned host memory (NVLink-C2C)"
                if round(e2e_launches) == round(launches / (args.steps + 0.0)) + 2
                else "cudaMemcpyAsync")
    e2e = {"value": round(whole_job_rate(tokens, e2e_steps, ms_e2e, world), 1), "unit": UNIT,
           "h2d_bytes_per_step": w.tokens * w.hidden * 2, "d2h_bytes_per_step": w.tokens * w.hidden * 2,
           "steps": e2e_steps, "call": "tp_layer_forward_host", "transfer": transfer}

    cpu = None
    if args.cpu_baseline and rank == 0 and world == 1:
        cpu = cpu_baseline(w, args.t, args.cpu_budget_s)
    prefill = prefill_detail = None
    configs, configs_detail = {}, {}
    if (args.prefill or args.configs) and rank == 0 and world == 1:
        model.close()
        torch.cuda.empty_cache()
    if args.prefill and rank == 0 and world == 1:
        prefill, prefill_detail = prefill_section(stream, prefill_bn=args.prefill_bn,
                                                   prefill_pairs=args.prefill_pairs)
    if args.configs and rank == 0 and world == 1:
        for name in ("qwen32b_decode", "qwen32b_decode_kv4"):
            configs[name], configs_detail[name] = decode_layer_section(name, stream, hbm_peak)
        configs["llama8b_full"], configs_detail["llama8b_full"] = full_forward_section(stream, hbm_peak)

    model.close()
    if rank != 0:
        return
    # per-kernel tables of every section: a second JSON line on stderr
    print(json.dumps({"bench_detail": {"decode_layer_kernels": kernels, "prefill": prefill_detail,
                                       "decode_configs": configs_detail,
                                       "kernel_timing": "CUDA events around each launch on the "
                                       f"launch stream, {prof_steps} steps after the timed region "
                                       f"({ms_prof / prof_steps:.4f} ms/step with the events)"}}),
          file=sys.stderr, flush=True)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded random-init weights ~N(0,0.02), KV cache ~N(0,1), hidden ~N(0,1)",
        "config": {
            **workload_config(w, args.t),
            "fused_reduction": bool(args.fused),
            "parallelism": f"tp{args.t} emulated on 1 GPU" + (f", {world} replicas" if world > 1 else ""),
            "l2": f"inputs larger than L2: steps rotate over {args.rotate} layers with distinct "
                  f"weights and KV ({args.rotate * step_bytes / 1e9:.2f} GB)",
            "step_bytes": step_bytes, "step_gbs": round(step_gbs, 1),
            "step_hbm_frac": round(step_gbs / hbm_peak, 3),
            "ms_per_step_median": round(ms_med, 5), "median_of_steps": med_steps,
            "ms_per_step_cuda_graph": round(ms_graph_step, 5),
            "model_bytes_per_layer": int(model_bytes_per_layer),
            "kernels_per_step": round(launches / args.steps, 2),
        },
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "decode_configs": configs,
        "prefill": prefill,
        "per_t": per_t,
    }
    print(json.dumps(line), flush=True)


def kernel_table(prof, kb, hbm_peak):
    out = {}
    for name, (n, tot) in prof.items():
        avg = tot / n
        e = {"launches": n, "avg_us": round(avg * 1e3, 2)}
        if name in kb:
            e["gbs"] = round(kb[name] / (avg * 1e-3) / 1e9, 1)
            e["frac_hbm"] = round(e["gbs"] / hbm_peak, 3)
        out[name] = e
    return out


def decode_layer_section(name, stream, hbm_peak, steps=200, warmup=10):
    """One Qwen2.5-32B-shaped decoder layer in decode at t = 8: 64 sequences x
    1 token over a 2048-token KV context (8 KV heads, or 4 shared by replica
    pairs).  One layer is 1.2-1.5 GB of weights and KV, far above L2."""
    import torch
    import synth
    from megatron_tensor_layers_tp_gb300 import binding as B
    w = synth.WORKLOADS[name]
    t = 8
    with torch.cuda.stream(stream):
        model, batch, h = build(w, t, 1)
    ms, _, _ = timed_steps(model, batch, h, steps, warmup, 1, 1, stream)
    _, prof, _ = timed_steps(model, batch, h, steps // 2, 0, 1, 1, stream, profile=True)
    assert model.check_device(stream) == 0
    model.close()
    del model, batch, h
    torch.cuda.empty_cache()
    kb, step_bytes = layer_bytes(w, t)
    st = ms / steps
    compact = {"ms": round(st, 4), "tok_s": round(w.tokens / (st * 1e-3)),
               "hbm_frac": round(step_bytes / (st * 1e-3) / 1e9 / hbm_peak, 3)}
    detail = {"workload": f"Qwen2.5-32B-shaped decoder layer, decode: {w.n_seqs} sequences x 1 "
                          f"token, {w.ctx}-token KV context, {w.n_kv_heads} KV heads, t={t}",
              "step_bytes": step_bytes, **compact, "kernels": kernel_table(prof, kb, hbm_peak)}
    return compact, detail


def full_forward_section(stream, hbm_peak, reps=10, warmup=3):
    """Llama-3.1-8B-shaped full decode forward at t = 8: vocab-parallel
    embedding of 64 tokens (one per sequence), 32 layers over a 4096-token KV
    context, final RMSNorm and the vocab-parallel LM head with the logits
    gather (49 GB of weights and KV per step)."""
    import torch
    import synth
    from megatron_tensor_layers_tp_gb300 import binding as B
    w = synth.WORKLOADS["llama8b_full"]
    t = 8
    with torch.cuda.stream(stream):
        model, batch, _ = build(w, t, w.n_layers, head=True)
        ids = torch.empty(w.tokens, dtype=torch.int32, device="cuda")
        synth.fill_uniform_(ids, w.seed, synth.tensor_id("ids"), w.vocab)
        hbuf = torch.empty((w.tokens, w.hidden), dtype=torch.bfloat16, device="cuda")
        logits = torch.empty((w.n_seqs, w.vocab), dtype=torch.bfloat16, device="cuda")
        cb = batch.to_c()
    torch.cuda.synchronize()

    def run(n):
        for _ in range(n):
            model.forward(ids, batch, stream=stream, h=hbuf, logits=logits, cbatch=cb)
    run(warmup)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(reps)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    B.tp_profile(model.handle, True)
    run(2)
    B.tp_profile(model.handle, False)
    prof = B.tp_profile_read(model.handle, stream.cuda_stream)
    # the same forward replayed from one CUDA graph
    graph = model.capture_forward(ids, batch, hbuf, logits, stream, cbatch=cb)
    for _ in range(warmup):
        graph.launch(stream)
    e0.record(stream)
    for _ in range(reps):
        graph.launch(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_graph = e0.elapsed_time(e1) / reps
    graph.close()
    assert model.check_device(stream) == 0
    model.close()
    del model, batch
    torch.cuda.empty_cache()
    kb, lb = layer_bytes(w, t)
    kb = dict(kb)
    kb["gemm_lm_head"] = w.vocab * w.hidden * 2 + w.tokens * w.hidden * 2 + w.tokens * w.vocab * 2
    kb["embed"] = 2 * w.tokens * w.hidden * 2
    step_bytes = w.n_layers * lb + kb["gemm_lm_head"] + kb["embed"]  # norms: see layer_bytes
    compact = {"ms": round(ms, 4), "tok_s": round(w.tokens / (ms * 1e-3)),
               "hbm_frac": round(step_bytes / (ms * 1e-3) / 1e9 / hbm_peak, 3),
               "ms_cuda_graph": round(ms_graph, 4)}
    detail = {"workload": "Llama-3.1-8B-shaped full decode forward: 64 sequences x 1 token, "
                          "4096-token KV context, 32 layers + embedding + LM head, t=8",
              "step_bytes": step_bytes, **compact, "kernels": kernel_table(prof, kb, hbm_peak)}
    return compact, detail


def prefill_section(stream, reps=10, prefill_bn=0, prefill_pairs=0):
    """Llama-3.1-8B-shaped prefill chunk at t = 4: 8 sequences x 256 tokens
    through the vocab-parallel embedding, one decoder layer and the
    vocab-parallel LM head on each sequence's last token.  Reports every
    kernel's duration and, for the contractions, TFLOP/s against the burst
    bf16 tensor-core peak (each forward lasts under a millisecond and the
    timed loop ten of them: far from the seconds-long loop of the sustained
    figure)."""
    import torch
    import synth
    from megatron_tensor_layers_tp_gb300 import binding as B
    from megatron_tensor_layers_tp_gb300.runtime import TPModel, make_config, prefill_batch
    w = synth.WORKLOADS["llama8b_prefill"]
    t = 4
    H, d, I, V, M = w.hidden, w.head_dim, w.intermediate, w.vocab, w.tokens
    with torch.cuda.stream(stream):
        shapes = synth.weight_shapes(w, 0)
        L = {}
        for k in LAYER_KINDS:
            x = torch.empty(shapes[k], dtype=torch.bfloat16, device="cuda")
            if k.endswith("norm"):
                x.fill_(1.0)
            else:
                synth.fill_normal_(x, w.seed, synth.tensor_id(k, 0), w.sigma_w)
            L[k] = x
        emb = torch.empty((V, H), dtype=torch.bfloat16, device="cuda")
        synth.fill_normal_(emb, w.seed, synth.tensor_id("embed"), w.sigma_w)
        lm = torch.empty((V, H), dtype=torch.bfloat16, device="cuda")
        synth.fill_normal_(lm, w.seed, synth.tensor_id("lm_head"), w.sigma_w)
        fn = torch.ones(H, dtype=torch.bfloat16, device="cuda")
        cfg = make_config(H, w.n_heads, w.n_kv_heads, d, I, V, 1, t, w.rms_eps, w.rope_theta,
                          max_positions=w.l_max, prefill_bn=prefill_bn,
                          prefill_cta_pairs=prefill_pairs)
        model = TPModel(cfg, [L], emb, fn, lm, max_tokens=M, stream=stream)
        del L, emb, lm
        k = model.alloc_kv(w.n_seqs, w.l_max)
        v = model.alloc_kv(w.n_seqs, w.l_max)
        batch = prefill_batch(w.n_seqs, w.seq_len, [k], [v], w.l_max)
        ids = torch.empty(M, dtype=torch.int32, device="cuda")
        synth.fill_uniform_(ids, w.seed, synth.tensor_id("ids"), V)
        hbuf = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
        logits = torch.empty((w.n_seqs, V), dtype=torch.bfloat16, device="cuda")
        cb = batch.to_c()
    torch.cuda.synchronize()

    def run(n):
        for _ in range(n):
            model.forward(ids, batch, stream=stream, h=hbuf, logits=logits, cbatch=cb)
    run(3)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(reps)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    B.tp_profile(model.handle, True)
    run(reps)
    B.tp_profile(model.handle, False)
    prof = B.tp_profile_read(model.handle, stream.cuda_stream)
    assert model.check_device(stream) == 0
    _, tc_peak, _ = read_peaks()
    attn_flops = 0
    for _ in range(w.n_seqs):
        attn_flops += 4 * w.n_heads * d * (w.seq_len * (w.seq_len + 1) // 2)
    flops = {
        "gemm_qkv": 2 * M * H * (w.n_heads + 2 * w.n_kv_heads) * d,
        "gemm_o": 2 * M * w.n_heads * d * H,
        "gemm_gate_up": 2 * M * H * 2 * I,
        "gemm_down": 2 * M * I * H,
        "attn_prefill": attn_flops,
    }
    kern = {}
    for name, (n, tot) in prof.items():
        avg_ms = tot / n
        e = {"launches": n, "avg_us": round(avg_ms * 1e3, 2)}
        if name in flops:
            tf = flops[name] / (avg_ms * 1e-3) / 1e12
            e["tflops"] = round(tf, 1)
            e["frac_tc"] = round(tf / tc_peak, 3)
        if name == "gemm_lm_head":
            gbs = (V * H * 2) / (avg_ms * 1e-3) / 1e9
            e["gbs"] = round(gbs, 1)
        kern[name] = e
    gem = [k for k in ("gemm_qkv", "gemm_o", "gemm_gate_up", "gemm_down") if k in prof]
    g_flops = sum(flops[k] for k in gem)
    g_ms = sum(prof[k][1] / prof[k][0] for k in gem)
    model.close()
    tot = sum(p[1] for p in prof.values()) / reps
    compact = {"ms": round(ms, 4), "tok_s": round(M / (ms * 1e-3)),
               "gemm_frac_tc": round(g_flops / (g_ms * 1e-3) / 1e12 / tc_peak, 3),
               "tc_peak": tc_peak,
               **{k[5:]: kern[k]["frac_tc"] for k in gem},
               "attn_us": kern.get("attn_prefill", {}).get("avg_us"),
               "attn_share": round(prof["attn_prefill"][1] / reps / tot, 3) if "attn_prefill" in prof else None}
    detail = {"workload": "8 sequences x 256 tokens, t=4: embedding + 1 layer + LM head on the "
                          "last token of each sequence", **compact,
              "gemm_tflops": round(g_flops / (g_ms * 1e-3) / 1e12, 1), "kernels": kern}
    return compact, detail


# ---------------------------------------------------------------------------
# the CPU oracle (baseline leg and --impl reference)
# ---------------------------------------------------------------------------
def oracle_inputs(w):
    import oracle as O
    import synth
    shapes = synth.weight_shapes(w, 0)
    W = O.LayerWeights(**{k: synth.host_weight(w, k, 0, shapes[k]) for k in LAYER_KINDS})
    h = synth.host_hidden(w)
    kc = {b: synth.host_kv(w, "k_cache", 0, b) for b in range(w.n_seqs)}
    vc = {b: synth.host_kv(w, "v_cache", 0, b) for b in range(w.n_seqs)}
    dims = O.Dims(w.hidden, w.n_heads, w.n_kv_heads, w.head_dim, w.intermediate, w.vocab,
                  w.rms_eps, w.rope_theta)
    return W, h, kc, vc, dims


def oracle_step(w, t, inputs):
    import oracle as O
    W, h, kc, vc, dims = inputs
    p = O.plan(w.n_heads, w.n_kv_heads, w.intermediate, w.vocab, t)
    return O.sharded_layer_forward(h, W, O.split_cache_copies(kc, dims, p),
                                   O.split_cache_copies(vc, dims, p),
                                   O.Batch.decode(w.n_seqs, w.ctx), dims, p)


def workload_config(w, t):
    """The config keys both arms report for the decode-layer workload."""
    return {"workload": "Llama-3.1-8B-shaped decoder layer, decode: 16 sequences x 1 token, "
                        "1024-token KV context, t emulated TP ranks",
            "hidden": w.hidden, "n_heads": w.n_heads, "n_kv_heads": w.n_kv_heads,
            "head_dim": w.head_dim, "intermediate": w.intermediate, "batch": w.n_seqs,
            "ctx": w.ctx, "t": t}


def cpu_baseline(w, t, budget_s):
    inputs = oracle_inputs(w)
    oracle_step(w, t, inputs)  # warm
    n, t0 = 0, time.perf_counter()
    while True:
        oracle_step(w, t, inputs)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0))
    return {"value": round(n * w.tokens / dt, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} decode step(s) of one layer, {w.tokens} tokens, t={t} sharded emulation "
                      f"in float64 numpy ({dt:.1f} s)"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import synth
    w = synth.WORKLOADS[WORKLOAD]
    inputs = oracle_inputs(w)
    for _ in range(min(args.warmup, 2)):
        oracle_step(w, args.t, inputs)
    n, t0 = 0, time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, args.t, inputs)
        n += 1
        if time.perf_counter() - t0 >= args.reference_budget_s:
            break
    dt = time.perf_counter() - t0
    value = n * w.tokens / dt
    cores = len(os.sched_getaffinity(0))
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "steps_run": n, "warmup": args.warmup,
        "ms_per_step": round(dt / n * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded inputs)",
        "config": workload_config(w, args.t),
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{n} decode step(s) of {w.tokens} tokens (wall-time capped at "
                                   f"{args.reference_budget_s:.0f} s)"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.prefill_only:
        import torch
        stream = torch.cuda.Stream()
        print(json.dumps({"prefill": prefill_section(stream, prefill_bn=args.prefill_bn,
                                                   prefill_pairs=args.prefill_pairs)[1]}), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    run_ours(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Throughput of the routed-expert MoE layer on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one moe_layer_forward_ex call (router -> dispatch -> [condensation] ->
routed experts -> combine, with the shared experts on a second stream beside
dispatch and the routed experts) over one batch of T synthetic tokens already
resident in HBM; the single-stream moe_layer_forward is timed beside it.
Default workload: the largest layer of the five, the Llama-4-Scout-shaped bf16
layer with FarSkip-Collective wiring (T=8192, d=5120, 16 experts top-1 sigmoid,
hidden 8192, 1 shared expert of hidden 8192, external attention-partial
residual); --workload names any other.  Inputs and weights are seeded synthetic
draws (routing_expert_ffn_gb300.inputs); the weights exceed L2 and L2 is
additionally flushed (a 256 MB write) between timed steps, outside the timed
events.  Besides the K timed steps, a steady region replays the same step for
at least one second (and at least 200 steps) with its own clock samples.

Under torchrun each rank runs an independent replica on its own GPU (weak
scaling, no data-path collective); the reported time is the max over ranks.
`--impl reference` times the fp64 CPU oracle on a bounded token sample of the
same workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s on 1 GB300; expert-GEMM % of BF16 peak; dispatch GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes (read + write) of the grouped-GEMM launches of one moe_expert_ffn call, from
# one-pass ncu captures (dram__bytes_read.sum + dram__bytes_write.sum) of the pair kernel at
# the workload's full size; workloads without a capture report null.
GEMM_DRAM_BYTES = {"dsv2_lite": 1496.8e6, "llama4_scout_farskip": 6316.9e6,
                   "qwen3_30b_a3b": 1888.8e6, "luffy_condense": 808.1e6}


def load_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks (NVML, read only)
class ClockSampler:
    """Polls SM clock and clock-event reasons through NVML while the timed region runs."""
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, device_index: int):
        self.samples: list[tuple[int, int]] = []
        self.max_mhz = None
        self.ok = False
        self._stop = threading.Event()
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            uuid = os.environ.get("BENCH_GPU_UUID")
            if uuid:
                r = self.nvml.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h))
            else:
                r = self.nvml.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(self.h))
            if r != 0:
                return
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:  # 1 = SM
                self.max_mhz = int(mx.value)
            self.ok = True
        except OSError:
            pass

    def _sample(self):
        c = ctypes.c_uint()
        reasons = ctypes.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) != 0:
            return
        self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(reasons))
        self.samples.append((int(c.value), int(reasons.value)))

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(0.002)

    def start(self):
        if self.ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()

    def stop(self) -> dict:
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"]}
        self._stop.set()
        self._t.join()
        if not self.samples:
            self._sample()
        mhz = [s for s, _ in self.samples]
        mask = 0
        for _, r in self.samples:
            mask |= r
        reasons = [n for b, n in self.REASONS.items() if mask & b and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(mhz)}


# ------------------------------------------------------------------ work accounting
def work(cfg, n_condensed: int = 0, active_experts: int | None = None) -> dict:
    """Algorithmic FLOPs and bytes of one layer call (no padding rows, no re-reads).

    ffn_bytes: what the expert GEMMs must move at least -- the weights of every expert
    that received a token (active_experts, all E when not given) and of the shared
    experts, once, plus x_perm / x read, h written and read back, y / shared written.
    """
    b = 2 if cfg.dtype == "bf16" else 4
    P = cfg.T * cfg.k
    n_act = cfg.E if active_experts is None else active_experts
    ffn_bytes = ((n_act * 3 * cfg.H + cfg.n_shared * 3 * cfg.H_shared) * cfg.d * b
                 + (P - n_condensed) * (2 * cfg.d + 2 * cfg.H) * b
                 + cfg.T * cfg.n_shared * (2 * cfg.d + 2 * cfg.H_shared) * b)
    routed_flops = 6.0 * cfg.d * cfg.H * (P - n_condensed)
    shared_flops = 6.0 * cfg.d * cfg.H_shared * cfg.T * cfg.n_shared
    idx_bytes = P * 4
    dispatch_bytes = cfg.T * cfg.d * b + P * cfg.d * b + idx_bytes * 3  # x in, x_perm out, idx/perm/slot_of
    res_reads = {"none": 0, "input": 1, "external": 1, "input_plus_external": 2}[cfg.residual]
    combine_bytes = (P * cfg.d * b + cfg.T * cfg.d * b * (1 + res_reads + (1 if cfg.n_shared else 0))
                     + idx_bytes * 2)
    return dict(routed_flops=routed_flops, shared_flops=shared_flops,
                ffn_flops=routed_flops + shared_flops, ffn_bytes=ffn_bytes,
                dispatch_bytes=dispatch_bytes,
                combine_bytes=combine_bytes, router_flops=2.0 * cfg.T * cfg.d * cfg.E)


def launches_per_step(cfg, condense: bool) -> int:
    # router: bf16 layers split W_r into bf16 terms, run the tensor-core logits and the
    # top-k; fp32 layers run FMA logits and the top-k
    n = 3 if cfg.dtype == "bf16" else 2
    # dispatch: block ranks and row scatter; the (expert, 1024-pair block) count table is
    # scanned inside the scatter up to 2048 entries, by a launch of its own above that
    n += 2 + (cfg.E * -(-(cfg.T * cfg.k) // 1024) > 2048)
    bf16 = cfg.dtype == "bf16"
    if condense:
        # m-tiles, tile list, similarity GEMM (its epilogue also finds each row's earliest
        # similar row), resolve, greedy scan (the dispatch forms the row statistics of a
        # condensing layer)
        n += 5
        n += 3  # compact reps, m-tiles over representatives, gather representative rows
    elif not bf16:
        n += 1  # m-tiles (the bf16 pair GEMM reads the bucket offsets itself)
    n += 2      # routed gate/up + down GEMMs
    if cfg.n_shared:
        n += 2 + (0 if bf16 else 1)  # shared gate/up + down GEMMs (+ m-tiles for fp32)
    n += 1      # combine
    return n


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest value over all ranks (the slowest replica's step time)."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: every replica's tokens over the slowest replica's time."""
    return world * tokens_per_rank / (max_ms / 1e3)


def capture(torch, fn):
    """CUDA graph of fn() (fn launches on torch's current stream); fn runs once first."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


# ------------------------------------------------------------------ ours
def run_ours(args, rank: int, world: int, local_rank: int) -> None:
    import torch
    from routing_expert_ffn_gb300 import build as moe_build
    from routing_expert_ffn_gb300 import inputs as gen
    from routing_expert_ffn_gb300 import moe

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    moe_build.build()
    moe.lib()
    cfg = workload_config(args)
    inp = gen.make_inputs(cfg)
    C = moe.Config.from_workload(cfg)
    w, x, r = moe.upload(C, inp, device=dev)
    tau = cfg.taus[0] if cfg.taus else math.nan
    condense = tau <= 1.0
    layer = moe.Layer(C, w, condense=condense, device=dev)
    out = torch.empty((C.T, C.d), dtype=C.torch_dtype, device=dev)
    ncond = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # One layer call is captured once as a CUDA graph and replayed every step, so
    # the timed region holds device work only (no per-kernel host launch cost).
    # The step is moe_layer_forward_ex: with shared experts they run on a second
    # stream after the router, beside dispatch and the routed experts (FarSkip's
    # overlap of the routing-independent work); under FarSkip wiring (an external
    # residual stream) the partial activation r + shared is written as well.
    # (a higher-priority second stream measured best: its GEMM tiles get SMs first
    # as the dispatch kernels retire)
    aux = torch.cuda.Stream(priority=-1) if C.n_shared > 0 else None
    part = torch.empty_like(out) if C.residual in ("external", "input_plus_external") else None

    def layer_step():
        layer(x, r, tau, out=out, n_condensed_out=ncond, partial_out=part, aux_stream=aux)

    def timed_each(g, n) -> list:
        """Per-step device ms of n replays, L2 flushed before each (outside the events)."""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for i in range(n):
            flush.zero_()
            evs[i][0].record(stream)
            g.replay()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    def timed(g) -> float:
        return sum(timed_each(g, args.steps)) / args.steps

    graph = capture(torch, layer_step)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    st = moe.get_device_status()
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {moe.status_string(st)}")
    n_condensed = int(ncond.item())

    sampler = ClockSampler(local_rank)
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    ms = timed(graph)
    clocks = sampler.stop()
    barrier()
    ms = max_over_ranks(ms, world, dev)

    # Steady region: the same step replayed for >= 1 s of device time (and >= 200 steps),
    # so that a box's clock behaviour and run-to-run noise can be told apart from a change.
    n_steady = max(200, int(math.ceil(1000.0 / max(ms, 1e-3))))
    sampler2 = ClockSampler(local_rank)
    barrier()
    torch.cuda.synchronize()
    sampler2.start()
    per = timed_each(graph, n_steady)
    clocks2 = sampler2.stop()
    barrier()
    med = statistics.median(per)
    steady = {"steps": n_steady, "device_s": sum(per) / 1e3, "median_ms": med,
              "p10_ms": sorted(per)[len(per) // 10], "p90_ms": sorted(per)[(9 * len(per)) // 10],
              "median_tokens_per_s": job_tokens_per_s(C.T, world, max_over_ranks(med, world, dev)),
              "clocks": clocks2}
    if clocks2.get("sm_mhz") and clocks2.get("sm_max_mhz"):
        # the step time scaled to the maximum SM clock (time x median MHz / max MHz)
        steady["median_ms_at_max_clock"] = med * clocks2["sm_mhz"] / clocks2["sm_max_mhz"]

    # For comparison: the same layer as one moe_layer_forward call on a single stream.
    g_serial = capture(torch, lambda: layer(x, r, tau, out=out, n_condensed_out=ncond))
    for _ in range(args.warmup):
        g_serial.replay()
    torch.cuda.synchronize()
    ms_serial = max_over_ranks(timed(g_serial), world, dev)
    serial = {"ms_per_step": ms_serial, "tokens_per_s": job_tokens_per_s(C.T, world, ms_serial),
              "path": "moe_layer_forward, every kernel on one stream"}

    # The layer's backward (moe_layer_backward) on the same tokens: a seeded output
    # gradient, one CUDA graph per step, L2 flushed between steps like the forward.
    backward = None
    if C.dtype == "bf16" and not condense and not args.no_backward:
        bwd = moe.Backward(C, w, device=dev)
        g_out = torch.randn((C.T, C.d), generator=torch.Generator(device=dev).manual_seed(7),
                            device=dev).to(C.torch_dtype)
        g_bwd = capture(torch, lambda: bwd(x, g_out))
        for _ in range(args.warmup):
            g_bwd.replay()
        torch.cuda.synchronize()
        ms_b = max_over_ranks(timed(g_bwd), world, dev)
        wkb = work(C)
        b_flops = 2.0 * wkb["ffn_flops"]  # input and weight gradients: 12 d H per pair (+ shared)
        peak_b = float(load_peaks()[0].get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        backward = {"ms_per_step": ms_b, "tokens_per_s": job_tokens_per_s(C.T, world, ms_b),
                    "algorithmic_TFLOP_s": b_flops / (ms_b / 1e3) / 1e12,
                    "frac_of_bf16_peak": b_flops / (ms_b / 1e3) / 1e12 / peak_b,
                    # the call also recomputes the forward's expert GEMMs (6 d H per pair and
                    # per token and shared expert): the tensor work it actually does
                    "frac_of_bf16_peak_with_recompute":
                        (b_flops + wkb["ffn_flops"]) / (ms_b / 1e3) / 1e12 / peak_b,
                    "path": "moe_layer_backward (forward recomputed inside), CUDA graph",
                    "flops_note": "12 d H per routed pair + 12 d H_shared per token and shared "
                                  "expert; the recompute of the forward (6 d H per pair) is not counted"}
        st = moe.get_device_status()
        if st != 0:
            raise RuntimeError(f"device status after the backward: {moe.status_string(st)}")

    # experts that received at least one token (the weights a step has to stream)
    _, idx_chk, _ = moe.route(C, x, w.W_r, w.router_bias)
    active = int((torch.bincount(idx_chk.flatten().long(), minlength=C.E) > 0).sum().item())

    # per-phase breakdown (FarSkip Eq. 9 terms): the same step as separate ABI calls
    phases = phase_breakdown(args, moe, C, w, x, r, tau, flush, stream, torch)
    history = history_report(args, moe, C, w, x, tau, flush, stream, torch) if condense else None
    # the layer's outputs after all timing passes still come from the same graph
    graph.replay()
    # end to end: pinned host input -> device -> layer -> pinned host output, every step,
    # double-buffered so that one step's copies overlap its neighbours' layer calls
    def layer_on(xb, rb, ob):
        return capture(torch, lambda: layer(xb, rb, tau, out=ob, n_condensed_out=ncond,
                                            partial_out=part, aux_stream=aux))
    e2e = end_to_end(args, C, graph, layer_on, x, r, out, stream, torch, world, dev)
    st = moe.get_device_status()
    if st != 0:
        raise RuntimeError(f"device status after timing: {moe.status_string(st)}")

    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    wk = work(C, n_condensed, active_experts=active)
    ffn_s = phases["T_experts_ms"] / 1e3
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    # The expert GEMMs are bound by the tensor pipes when their arithmetic intensity is
    # above the machine's ridge (peak FLOP/s over HBM bytes/s), else by streaming the
    # weights from HBM (decode-shaped steps).
    if wk["ffn_flops"] / wk["ffn_bytes"] >= peak * 1e12 / (hbm * 1e9):
        roofline = {"bound": "tensor", "kernel": "grouped expert GEMM (moe_expert_ffn)",
                    "achieved": wk["ffn_flops"] / ffn_s / 1e12, "peak": peak, "unit": "TFLOP/s",
                    "peak_source": f"{peak_src} bf16 burst"}
    else:
        roofline = {"bound": "hbm", "kernel": "grouped expert GEMM (moe_expert_ffn), weight stream",
                    "achieved": wk["ffn_bytes"] / ffn_s / 1e9, "peak": hbm, "unit": "GB/s",
                    "peak_source": f"{peak_src} HBM copy", "bytes": wk["ffn_bytes"],
                    "active_experts": active}
    roofline["frac"] = roofline["achieved"] / roofline["peak"]
    reduced = bool(args.tokens or args.experts)
    roofline["traffic"] = None if reduced else GEMM_DRAM_BYTES.get(cfg.name)
    disp_gbs = wk["dispatch_bytes"] / (phases["T_dispatch_ms"] / 1e3) / 1e9
    comb_gbs = wk["combine_bytes"] / (phases["T_combine_ms"] / 1e3) / 1e9
    line = {
        "metric": METRIC,
        "value": job_tokens_per_s(C.T, world, ms),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": C.dtype,
        "data": "synthetic (seeded N(0,1) tokens, N(0,0.02^2) weights, router N(0,1/d)); no dataset",
        "config": {"workload": workload_desc(cfg),
                   "tokens_per_gpu": C.T, "parallelism": f"replicas x{world}",
                   "launch": "each step replays one CUDA graph of moe_layer_forward_ex"
                  + (" (shared experts on a second stream)" if aux is not None else "")
                  + (", partial activation written" if part is not None else ""),
                   "l2": "256 MB write between timed steps (outside the timed events); weights "
                         f"{(C.E * 3 * C.H + C.n_shared * 3 * C.H_shared) * C.d * 2 / 1e9:.2f} GB > L2"},
        "roofline": roofline,
        "dispatch": {"GB/s": disp_gbs, "frac_of_hbm": disp_gbs / hbm,
                     "bytes": wk["dispatch_bytes"]},
        "combine": {"GB/s": comb_gbs, "frac_of_hbm": comb_gbs / hbm, "bytes": wk["combine_bytes"]},
        "phases_ms": phases,
        "eq9": eq9_report(ms, phases),
        "serial": serial,
        "backward": backward,
        "condensed": n_condensed,
        "history": history,
        "gpu_launches": launches_per_step(C, condense) * args.steps,
        "clocks": clocks,
        "steady": steady,
        "e2e": e2e,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, inp, target_s=args.cpu_seconds)
    print(json.dumps(line), flush=True)


def phase_breakdown(args, moe, C, w, x, r, tau, flush, stream, torch) -> dict:
    """Per-phase device time of the step, each phase its own ABI call, events between them."""
    L = moe.lib()
    c = C.c()
    dev = x.device
    P = C.T * C.k
    i32, f32 = torch.int32, torch.float32
    logits = torch.empty((C.T, C.E), dtype=f32, device=dev)
    idx = torch.empty((C.T, C.k), dtype=i32, device=dev)
    gate = torch.empty((C.T, C.k), dtype=f32, device=dev)
    counts = torch.empty((C.E,), dtype=i32, device=dev)
    offsets = torch.empty((C.E + 1,), dtype=i32, device=dev)
    perm = torch.empty((P,), dtype=i32, device=dev)
    slot_of = torch.empty((C.T, C.k), dtype=i32, device=dev)
    x_perm = torch.empty((P, C.d), dtype=C.torch_dtype, device=dev)
    y_perm = torch.empty((P, C.d), dtype=C.torch_dtype, device=dev)
    so = torch.empty((C.T, C.d), dtype=C.torch_dtype, device=dev) if C.n_shared else None
    rep_of = torch.empty((P,), dtype=i32, device=dev)
    n_rep = torch.empty((C.E,), dtype=i32, device=dev)
    ncond = torch.empty((1,), dtype=i32, device=dev)
    out = torch.empty((C.T, C.d), dtype=C.torch_dtype, device=dev)
    condense = tau <= 1.0
    nr = L.moe_route_workspace_size(ctypes.byref(c))
    ws_r = torch.empty(max(nr, 1), dtype=torch.uint8, device=dev)
    nd = L.moe_dispatch_workspace_size(ctypes.byref(c))
    nc = L.moe_condense_workspace_size(ctypes.byref(c)) if condense else 0
    nf = L.moe_expert_ffn_workspace_size(ctypes.byref(c), int(condense))
    ws_d = torch.empty(max(nd, 1), dtype=torch.uint8, device=dev)
    ws_c = torch.empty(max(nc, 1), dtype=torch.uint8, device=dev)
    ws_f = torch.empty(max(nf, 1), dtype=torch.uint8, device=dev)
    wc = w.c()
    p = lambda t: None if t is None else t.data_ptr()

    def cur():
        return torch.cuda.current_stream().cuda_stream

    def ph_route():
        s = cur()
        moe._check(L.moe_route(ctypes.byref(c), p(x), p(w.W_r), p(w.router_bias), p(logits), p(idx),
                               p(gate), p(ws_r), nr, s), "route")

    def ph_dispatch():
        s = cur()
        moe._check(L.moe_dispatch(ctypes.byref(c), p(x), p(idx), p(counts), p(offsets), p(perm),
                                  p(slot_of), p(x_perm), p(ws_d), nd, s), "dispatch")

    def ph_condense():
        s = cur()
        if condense:
            moe._check(L.moe_condense(ctypes.byref(c), p(x_perm), p(offsets), tau, p(rep_of),
                                      p(n_rep), p(ncond), p(ws_c), nc, s), "condense")

    def ph_ffn():
        s = cur()
        moe._check(L.moe_expert_ffn(ctypes.byref(c), ctypes.byref(wc), p(x_perm), p(offsets),
                                    p(rep_of) if condense else None, p(x), p(y_perm), p(so),
                                    p(ws_f), nf, s), "expert_ffn")

    def ph_combine():
        s = cur()
        moe._check(L.moe_combine(ctypes.byref(c), p(y_perm), p(so), p(slot_of),
                                 p(rep_of) if condense else None, p(gate), p(x), p(r), p(out), s),
                   "combine")

    # the routed experts alone (the same call with the shared experts switched off)
    c_routed = C.c()
    c_routed.n_shared = 0
    nf_r = L.moe_expert_ffn_workspace_size(ctypes.byref(c_routed), int(condense))

    def ph_routed_only():
        s = cur()
        moe._check(L.moe_expert_ffn(ctypes.byref(c_routed), ctypes.byref(wc), p(x_perm), p(offsets),
                                    p(rep_of) if condense else None, p(x), p(y_perm), None,
                                    p(ws_f), nf_r, s), "expert_ffn (routed only)")

    fns = [ph_route, ph_dispatch, ph_condense, ph_ffn, ph_combine, ph_routed_only]
    names = ["T_gate_ms", "T_dispatch_ms", "T_condense_ms", "T_experts_ms", "T_combine_ms",
             "T_routed_ms"]
    inside = phases_inside_graph(args, torch, fns[:5], fns[5], names, flush, stream,
                                 skip=None if condense else ph_condense)
    if inside is not None:
        return inside
    graphs = [capture(torch, f) if (f is not ph_condense or condense) else None for f in fns]

    def step(evs):
        for i, g in enumerate(graphs):
            if i == len(graphs) - 1:
                flush.zero_()  # the routed-only pass starts from a cold L2 as well
            evs[2 * i].record(stream)
            if g is not None:
                g.replay()
            evs[2 * i + 1].record(stream)

    n_ev = 2 * len(graphs)
    for _ in range(max(1, args.warmup)):
        step([torch.cuda.Event(enable_timing=True) for _ in range(n_ev)])
    torch.cuda.synchronize()
    all_evs = []
    for _ in range(args.steps):
        flush.zero_()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
        step(evs)
        all_evs.append(evs)
    torch.cuda.synchronize()
    res = {n: 0.0 for n in names}
    for evs in all_evs:
        for i, n in enumerate(names):
            res[n] += evs[2 * i].elapsed_time(evs[2 * i + 1]) / len(all_evs)
    res["T_shared_ms"] = max(0.0, res["T_experts_ms"] - res["T_routed_ms"])
    res["note"] = ("each phase is one ABI call captured as a CUDA graph and replayed in layer order; "
                   "T_experts = moe_expert_ffn (routed + shared grouped GEMMs on tcgen05 and their "
                   "m-tile tables); T_routed = the same call without the shared experts; "
                   "T_shared = their difference")
    return res


def _external_event_record():
    """cuEventRecordWithFlags(event, stream, CU_EVENT_RECORD_EXTERNAL) from the driver library:
    recorded while a stream is being captured, it becomes an event-record node of the graph,
    whose timestamp can be read after each replay.  None if the driver call is unavailable."""
    try:
        cu = ctypes.CDLL("libcuda.so.1")
        f = cu.cuEventRecordWithFlags
    except (OSError, AttributeError):
        return None
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
    f.restype = ctypes.c_int
    return lambda ev, st: f(ctypes.c_void_p(ev.cuda_event), ctypes.c_void_p(st.cuda_stream), 1)


def phases_inside_graph(args, torch, step_fns, routed_fn, names, flush, stream, skip=None):
    """Phase times from events recorded inside the captured graph of the whole step (one graph:
    event, phase, event, phase, ...; the routed-only call in a graph of its own, after an L2
    flush), so that each phase's events bracket its own kernels and not the graph's launch.
    Returns None (the caller then times one graph per phase) if the events cannot be recorded
    into a graph."""
    rec = _external_event_record()
    if rec is None:
        return None
    cap = torch.cuda.Stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(step_fns) + 3)]
    for e in evs:
        e.record(stream)  # creates the events
    torch.cuda.synchronize()
    if not all(getattr(e, "cuda_event", 0) for e in evs):
        return None
    ok = [True]

    def record(e):
        if rec(e, torch.cuda.current_stream()) != 0:
            ok[0] = False

    def whole():
        record(evs[0])
        for i, f in enumerate(step_fns):
            if f is not skip:
                f()
            record(evs[i + 1])

    def routed():
        record(evs[-2])
        routed_fn()
        record(evs[-1])

    try:
        for f in step_fns + [routed_fn]:  # every ABI call once outside the capture
            if f is not skip:
                f()
        torch.cuda.synchronize()
        graphs = []
        for fn in (whole, routed):
            g = torch.cuda.CUDAGraph()
            cap.wait_stream(torch.cuda.current_stream())
            with torch.cuda.graph(g, stream=cap):
                fn()
            graphs.append(g)
        torch.cuda.synchronize()
    except Exception:  # the capture could not record the events: time one graph per phase
        return None
    if not ok[0]:
        return None
    res = {n: 0.0 for n in names}
    n_step = max(args.steps, 1)
    for it in range(max(1, args.warmup) + n_step):
        flush.zero_()
        graphs[0].replay()
        flush.zero_()
        graphs[1].replay()
        torch.cuda.synchronize()
        if it < max(1, args.warmup):
            continue
        for i in range(len(step_fns)):
            res[names[i]] += evs[i].elapsed_time(evs[i + 1]) / n_step
        res[names[-1]] += evs[-2].elapsed_time(evs[-1]) / n_step
    res["T_shared_ms"] = max(0.0, res["T_experts_ms"] - res["T_routed_ms"])
    res["note"] = ("the step's ABI calls captured as one CUDA graph with event-record nodes between "
                   "them (the events bracket each phase's own kernels, not the graph launch), "
                   "replayed after an L2 flush; T_experts = moe_expert_ffn (routed + shared grouped "
                   "GEMMs on tcgen05); T_routed = the same call without the shared experts, in a "
                   "graph of its own after another flush; T_shared = their difference")
    return res


def history_report(args, moe, C, w, x, tau, flush, stream, torch) -> dict:
    """Condensation with Luffy's historical similarity (moe_condense_hist, S1 = 0.8,
    S2 = 0.2) against plain moe_condense on the same dispatched batch: a first block (no
    record: every Gram tile needs cosines, and the classes are recorded) and a repeated block
    (the record of the same batch: tiles whose pairs all have a class skip the tensor cores).
    Each timed as one ABI call in a CUDA graph, L2 flushed before each replay."""
    dev = x.device
    _, idx, _ = moe.route(C, x, w.W_r, w.router_bias)
    d = moe.dispatch(C, x, idx)
    torch.cuda.synchronize()
    rec_a = torch.empty(moe.condense_history_bytes(C), dtype=torch.uint8, device=dev)
    rec_b = torch.empty_like(rec_a)
    outs = {}

    def plain():
        outs["plain"] = moe.condense(C, d["x_perm"], d["offsets"], tau)

    def first():
        outs["first"] = moe.condense_hist(C, d["x_perm"], d["offsets"], d["perm"], d["slot_of"],
                                          tau, 0.8, 0.2, hist_in=None, hist_out=rec_a)

    def repeat():
        outs["repeat"] = moe.condense_hist(C, d["x_perm"], d["offsets"], d["perm"], d["slot_of"],
                                           tau, 0.8, 0.2, hist_in=rec_a, hist_out=rec_b)

    res = {}
    for name, fn in (("plain", plain), ("first", first), ("repeat", repeat)):
        g = capture(torch, fn)
        for _ in range(args.warmup):
            g.replay()
        ts = []
        for _ in range(max(args.steps, 20)):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        res[f"T_condense_{name}_ms"] = statistics.median(ts)
    torch.cuda.synchronize()
    same = all(torch.equal(outs[n][0], outs["plain"][0]) for n in ("first", "repeat"))
    res.update({"tiles_first": int(outs["first"][3].item()),
                "tiles_repeat": int(outs["repeat"][3].item()),
                "condensed": int(outs["plain"][2].item()),
                "same_assignment_as_plain": bool(same),
                "note": "S1 = 0.8, S2 = 0.2; 'first' = no record yet, 'repeat' = the record of the "
                        "same batch (a block whose tokens and routing repeat the previous one's); "
                        "tiles = Gram tiles that needed tensor-core cosines"})
    return res


def eq9_report(ms_layer: float, phases: dict) -> dict:
    """FarSkip-Collective's overlap condition (review ledger, Section 4.1, Eq. 9): the
    exchange steps fit in the window the layer leaves beside the routed experts and the
    gate, T_Dispatch + T_Combine <= T_layer - T_routed - T_gate.  On one GPU the
    exchange steps are the local dispatch permutation and the combine."""
    window = ms_layer - phases["T_routed_ms"] - phases["T_gate_ms"]
    comm = phases["T_dispatch_ms"] + phases["T_combine_ms"]
    return {"T_layer_ms": ms_layer, "T_gate_ms": phases["T_gate_ms"],
            "T_routed_ms": phases["T_routed_ms"], "T_dispatch_ms": phases["T_dispatch_ms"],
            "T_combine_ms": phases["T_combine_ms"], "window_ms": window, "dispatch_plus_combine_ms": comm,
            "holds": comm <= window}


def end_to_end(args, C, graph, layer_on, x, r, out, stream, torch, world=1, dev=None) -> dict:
    """Every step: its pinned host input x (and residual) -> a device input buffer, one
    layer call (a captured graph), its whole output -> a pinned host buffer.  Two device
    buffer sets alternate: step i+1's host-to-device copy and step i-1's device-to-host
    copy run on their own streams while step i's layer runs, as a serving loop overlaps
    them.  The timed region spans the first copy in to the last copy out."""
    xh = x.cpu().pin_memory()
    rh = r.cpu().pin_memory() if r is not None else None
    bufs = [(x, r, out, graph)]
    x1, r1, o1 = torch.empty_like(x), (torch.empty_like(r) if r is not None else None), torch.empty_like(out)
    x1.copy_(x)
    if r1 is not None:
        r1.copy_(r)
    bufs.append((x1, r1, o1, layer_on(x1, r1, o1)))
    outh = [torch.empty((C.T, C.d), dtype=C.torch_dtype).pin_memory() for _ in bufs]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event() for _ in bufs] for k in ("in", "done", "out")}
    used = [False, False]

    def step(i):
        b = i % 2
        xb, rb, ob, g = bufs[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev["done"][b])  # the layer has read this buffer's last input
            xb.copy_(xh, non_blocking=True)
            if rb is not None:
                rb.copy_(rh, non_blocking=True)
            ev["in"][b].record(s_in)
        stream.wait_event(ev["in"][b])
        if used[b]:
            stream.wait_event(ev["out"][b])  # this buffer's last output has left the device
        g.replay()
        ev["done"][b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["done"][b])
            outh[b].copy_(ob, non_blocking=True)
            ev["out"][b].record(s_out)
        used[b] = True

    for i in range(max(2, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(args.steps):
        step(i)
    s_out.wait_stream(s_in)
    s_out.wait_stream(stream)
    b.record(s_out)
    torch.cuda.synchronize()
    # whole job: every rank's tokens over the slowest rank's time
    ms = max_over_ranks(a.elapsed_time(b) / args.steps, world, dev)
    h2d = xh.numel() * xh.element_size() + (rh.numel() * rh.element_size() if rh is not None else 0)
    d2h = outh[0].numel() * outh[0].element_size()
    return {"value": job_tokens_per_s(C.T, world, ms), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "path": "every step: pinned host -> device copy of its input, the layer step (CUDA "
                    "graph), device -> pinned host copy of its output; two device buffer sets, "
                    "copies on their own streams overlapping the neighbouring steps' layer calls"}


# ------------------------------------------------------------------ oracle (CPU) timing
def _oracle_call(orc, cfg, inp64, T_s):
    return orc.layer_forward(inp64["x"][:T_s], inp64["W_r"], inp64["bias"], inp64["W_gu"],
                             inp64["W_down"], inp64["Ws_gu"], inp64["Ws_down"], cfg.k, cfg.gating,
                             residual_mode=cfg.residual,
                             residual=None if inp64["residual"] is None else inp64["residual"][:T_s],
                             tau=cfg.taus[0] if cfg.taus else None)


def _as_f64(inp):
    import numpy as np
    return {k: (None if v is None else np.asarray(v, dtype=np.float64)) for k, v in inp.items()
            if k != "labels"}


def cpu_baseline(cfg, inp, target_s: float = 12.0) -> dict:
    """The oracle as it stands on this host's cores, on the workload's tokens.

    A 128-token prefix first; if that is quick, a longer prefix (up to the whole
    batch) and, if the whole batch is still quick, repeated whole-batch calls,
    until about target_s seconds of host work have been timed.
    """
    from oracle import moe_oracle as orc
    inp64 = _as_f64(inp)
    T_s = min(cfg.T, 128)
    t0 = time.perf_counter()
    _oracle_call(orc, cfg, inp64, T_s)
    dt = time.perf_counter() - t0
    if dt < target_s / 3 and T_s < cfg.T:
        T_s = min(cfg.T, max(T_s, int(T_s * target_s / max(dt, 1e-3))))
    reps, tokens, t0 = 0, 0, time.perf_counter()
    while True:
        _oracle_call(orc, cfg, inp64, T_s)
        reps += 1
        tokens += T_s
        dt = time.perf_counter() - t0
        if dt >= target_s or reps >= 50:
            break
    return {"value": tokens / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{reps} fp64 layer call(s) on the first {T_s} of {cfg.T} tokens "
                      f"({dt:.1f} s); weights pre-cast to float64"}


def workload_config(args):
    """The named workload, with --tokens / --experts overriding T and E (smaller cases of the
    same kernels for profiler captures; the bench line then names the reduced shape)."""
    from dataclasses import replace
    from routing_expert_ffn_gb300 import inputs as gen
    cfg = gen.CONFIGS[args.workload]
    if args.tokens:
        cfg = replace(cfg, T=args.tokens)
    if args.experts:
        cfg = replace(cfg, E=args.experts)
    return cfg


def workload_desc(cfg) -> str:
    """The workload named by its shape (the same string in both arms' config)."""
    tau = cfg.taus[0] if cfg.taus else math.nan
    return (f"{cfg.name}: T={cfg.T} d={cfg.d} E={cfg.E} top-{cfg.k} {cfg.gating} "
            f"H={cfg.H} shared={cfg.n_shared}x{cfg.H_shared} residual={cfg.residual}"
            + (f" tau={tau:.6f}" if tau <= 1.0 else ""))


def run_reference(args, rank: int) -> None:
    if rank != 0:
        return
    from oracle import moe_oracle as orc
    from routing_expert_ffn_gb300 import inputs as gen
    cfg = workload_config(args)
    inp64 = _as_f64(gen.make_inputs(cfg))
    # Each step is a bounded token sample, sized from one 32-token call so that the whole
    # run (warm-up and timed steps) takes about --reference-seconds of host time.
    t0 = time.perf_counter()
    _oracle_call(orc, cfg, inp64, min(cfg.T, 32))
    per_token = (time.perf_counter() - t0) / min(cfg.T, 32)
    per_step = args.reference_seconds / (args.warmup + args.steps)
    T_s = int(max(16, min(cfg.T, args.reference_tokens, per_step / max(per_token, 1e-9))))
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        _oracle_call(orc, cfg, inp64, T_s)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = T_s / (ms / 1e3)
    sample = f"first {T_s} of {cfg.T} tokens per step, fp64 oracle, weights pre-cast to float64"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_desc(cfg), "tokens_per_step": T_s},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama4_scout_farskip")
    ap.add_argument("--tokens", type=int, default=0, help="override the workload's T")
    ap.add_argument("--experts", type=int, default=0, help="override the workload's E")
    ap.add_argument("--no-backward", action="store_true", help="skip timing the layer backward")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reference-tokens", type=int, default=1024,
                    help="most tokens per reference step")
    ap.add_argument("--reference-seconds", type=float, default=150.0,
                    help="host time the whole reference run aims at")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

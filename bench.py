#!/usr/bin/env python3
"""Benchmark of the routed-expert MoE FFN with a quantized HBM expert cache.

Default workload (batch-1 decode through 48 MoE layers): hidden 2048, 512
experts, top-8, expert FFN 1152 (SwiGLU), Q4 blocks of 32; router logits with
Zipf(1.1) expert popularity under a per-layer permutation; the HBM pool holds
all experts of 40 layers and a 60% hot set (seeded from the synthetic
routing-frequency table) of the other 8; the rest is read zero-copy from
pinned host memory.  One step = one decoded token: for each of the 48 layers,
router top-k and the expert FFN (quantize, gate/up mat-vec + SwiGLU +
quantize h, down mat-vec + combine), then the promotion pass (cache_step).

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Prints one JSON line (rank 0).  `value` is whole-job tokens/s with inputs
resident in HBM; `e2e` is the same through the C ABI with the step's inputs
copied from pinned host memory and its outputs copied back inside the timed
region; `roofline` is for the fused expert-FFN layer kernel (the dominant
kernel) over the fully resident layers; `cpu_baseline` is the CPU oracle on a bounded sample.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE expert-layer tokens/s (decode, prefill); achieved GB/s vs HBM/PCIe peak"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_b1_resident")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--cpu-sample-steps", type=int, default=6)
    ap.add_argument("--prefill-steps", type=int, default=2)
    ap.add_argument("--prefill-workload", default="prefill_t4096")
    ap.add_argument("--large-decode-steps", type=int, default=16,
                    help="decode steps per batch size of the large-expert leg (0 skips the leg)")
    ap.add_argument("--q8-steps", type=int, default=64,
                    help="timed decode steps of each of the Q8_0 / Q5_0 weight-format legs (0 skips them)")
    ap.add_argument("--pool-steps", type=int, default=256,
                    help="decode tokens per run of the pool-mode / preheat leg (0 skips it)")
    ap.add_argument("--case", default=None,
                    choices=["decode_layer", "decode_layer_cold", "decode_layer_q8", "prefill_layer",
                             "prefill_layer_wide"],
                    help="small profiling case: one layer (hidden 2048, 512 experts, top-8, FFN 1152, every "
                         "expert resident, or every expert in host memory for decode_layer_cold, Q8_0 weights "
                         "for decode_layer_q8), --launches forwards at batch 1 (routed) or 4096 tokens")
    ap.add_argument("--launches", type=int, default=20)
    ap.add_argument("--lookahead-steps", type=int, default=64,
                    help="timed decode steps of each run of the decode lookahead leg (0 skips it)")
    ap.add_argument("--cold-launches", type=int, default=20,
                    help="timed batch-1 forwards of the all-cold layer leg (0 skips it)")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def over_ranks(ms_local, units_local, world, device="cuda"):
    """Replicas (one process per GPU, no data-path collective): the slowest
    rank's time and the units every rank processed, so that whole-job
    throughput = units / time.  One process: the local values."""
    if world == 1:
        return float(ms_local), float(units_local)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms_local)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    u = torch.tensor([float(units_local)], dtype=torch.float64, device=device)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def src_hash(paths):
    """Hash of source text: a path (the whole file) or (path, first line,
    end line) for the part of a file from its first marker line up to the end
    marker (a kernel and the device helpers it uses)."""
    h = hashlib.sha256()
    for p in paths:
        path, a, b = (p, None, None) if isinstance(p, str) else p
        with open(os.path.join(ROOT, path), "rb") as f:
            txt = f.read()
        if a is not None:
            i = txt.index(a.encode())
            txt = txt[i:txt.index(b.encode(), i)]
        h.update(txt)
    return h.hexdigest()[:16]


# the fused decode layer kernel: its section of kernels_decode.cu and the
# shared device header (the traffic summary is valid while these are unchanged)
DECODE_KERNEL_SRC = [("quantized_expert_cache_gb300/csrc/kernels_decode.cu",
                      "// --------------------------------------------------------------- fused layer",
                      "// --------------------------------------------------------------- hooks"),
                     "quantized_expert_cache_gb300/csrc/common.cuh"]


def read_traffic(kernel_file, key):
    """Per-launch DRAM traffic of a kernel from its committed ncu summary,
    valid only while the kernel source is unchanged since the capture."""
    p = os.path.join(ROOT, "profiles", kernel_file)
    if not os.path.exists(p):
        return None
    vals = {}
    with open(p) as f:
        for line in f:
            if ":" in line and line.startswith("bench."):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    try:
        if vals.get("bench.source_hash") != src_hash(DECODE_KERNEL_SRC):
            return None
        return float(vals[key])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------
# workload setup
# ----------------------------------------------------------------------------

def decode_workload_desc(wl):
    """The decode workload as both arms name it in `config`."""
    L, H, E, k, F = wl.n_layers, wl.hidden, wl.n_experts, wl.top_k, wl.ffn
    T = wl.phases[0][1]
    caps = [wl.layer_capacity(l) for l in range(L)]
    return (f"{wl.name}: {L} MoE layers, hidden {H}, {E} experts, top-{k}, FFN {F} SwiGLU, Q4 blocks of 32, "
            f"Zipf({wl.zipf_s}) routing, batch {T} decode, HBM pool {caps.count(E)} full layers + "
            f"{min(caps)}/{E} hot set on the rest")


def register_workload(qec, synth, ctx, wl, log):
    t0 = time.time()
    bufs = {}
    for layer in range(wl.n_layers):
        order = wl.seed_order(layer)
        cap = wl.layer_capacity(layer)
        for kind in range(3):
            rows, cols = wl.tensor_shapes[kind]
            key = (rows, cols)
            if key not in bufs:
                bufs[key] = np.empty((wl.n_experts, rows, cols // synth.BLOCK_ELEMS[wl.weight_format],
                                      synth.BLOCK_BYTES[wl.weight_format]),
                                     np.uint8)
            wl.expert_tensor(layer, kind, out=bufs[key])
            qec.register_expert_tensor(ctx, layer, kind, bufs[key], rows, cols, cap, order, cap)
    log(f"registered {3 * wl.n_layers} expert tensors in {time.time() - t0:.1f}s")


def make_inputs(wl, n_steps, T):
    X = np.empty((n_steps, wl.n_layers, T, wl.hidden), np.float32)
    LG = np.empty((n_steps, wl.n_layers, T, wl.n_experts), np.float32)
    for s in range(n_steps):
        for l in range(wl.n_layers):
            X[s, l] = wl.x(l, s, T)
            LG[s, l] = wl.logits(l, s, T)
    return X, LG


def run_ours(args):
    import torch
    import quantized_expert_cache_gb300 as qec
    import synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def log(m):
        if rank == 0:
            print(f"[bench] {m}", file=sys.stderr, flush=True)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    qec.load()
    wl = synth.WORKLOADS[args.workload]
    label, T, _ = wl.phases[0]
    if label != "decode":
        raise SystemExit("bench.py times a decode workload")
    L, H, E, k, F = wl.n_layers, wl.hidden, wl.n_experts, wl.top_k, wl.ffn
    spt = max(wl.layer_capacity(l) for l in range(L))
    stream = torch.cuda.Stream()
    ctx = qec.moe_layer_init(H, F, E, k, L, spt, T, stream=stream)
    register_workload(qec, synth, ctx, wl, log)

    S = args.warmup + args.steps
    t0 = time.time()
    Xh, LGh = make_inputs(wl, S + args.steps, T)
    log(f"inputs for {S} steps in {time.time() - t0:.1f}s")
    X = torch.from_numpy(Xh).cuda()
    LG = torch.from_numpy(LGh).cuda()
    xin = torch.empty((L, T, H), device="cuda")
    lin = torch.empty((L, T, E), device="cuda")
    idx = torch.empty((L, T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((L, T, k), device="cuda")
    y = torch.empty((L, T, H), device="cuda")
    sptr = stream.cuda_stream

    # the fully resident layers, timed as one segment inside the step graph
    # (two event nodes; the launches between them stay chained)
    resident = [l for l in range(L) if wl.layer_capacity(l) == E]
    seg = None
    if resident and resident == list(range(resident[0], resident[-1] + 1)) and not args.no_graph:
        try:
            seg = (torch.cuda.Event(enable_timing=True, external=True),
                   torch.cuda.Event(enable_timing=True, external=True))
        except TypeError:
            seg = None

    def layers(mark=False):
        # router top-k + expert FFN per layer (one launch per layer for
        # small batches: every CTA routes the tokens itself)
        for l in range(L):
            if mark and seg is not None and l == resident[0]:
                seg[0].record(stream)
            qec.moe_ffn_forward_routed(ctx, l, xin[l], lin[l], T, idx[l], w[l], y[l], sptr)
            if mark and seg is not None and l == resident[-1]:
                seg[1].record(stream)

    graph = None
    if not args.no_graph:
        # warm the kernels once, then capture the L-layer step
        with torch.cuda.stream(stream):
            xin.copy_(X[0])
            lin.copy_(LG[0])
        layers()
        stream.synchronize()
        qec.miss_drain(ctx)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            layers(mark=True)
    launches_per_step = L * (1 if T * k <= 256 else 4) + 1  # per layer + the table update kernel
    used_graph = graph is not None

    def step(s, host_io=None):
        with torch.cuda.stream(stream):
            if host_io is None:
                xin.copy_(X[s])
                lin.copy_(LG[s])
            else:
                xin.copy_(host_io[0][s], non_blocking=True)
                lin.copy_(host_io[1][s], non_blocking=True)
            if graph is not None:
                graph.replay()
            else:
                layers()
        qec.cache_step(ctx, T)
        if host_io is not None:
            with torch.cuda.stream(stream):
                host_io[2].copy_(y, non_blocking=True)

    # the clock sampler starts before the warm-up so that nvidia-smi's own
    # start-up does not fall inside the timed region
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(1.0)
    for s in range(args.warmup):
        step(s)
    stream.synchronize()
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    seg_ms, seg_n = 0.0, 0
    ev0.record(stream)
    for s in range(args.warmup, S):
        step(s)
        if seg is not None:
            # cache_step has waited for this step's forwards
            seg_ms += seg[0].elapsed_time(seg[1])
            seg_n += 1
    ev1.record(stream)
    stream.synchronize()
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    barrier()
    torch.cuda.synchronize()
    ms_max, tokens = over_ranks(ms, args.steps * T, world)
    tok_per_s = tokens / (ms_max / 1e3)
    st_main = qec.moe_stats(ctx)
    log(f"timed: {tok_per_s:.1f} tokens/s, {ms_max / args.steps:.4f} ms/step, clocks {clk}")

    # end to end: the step's inputs from pinned host memory, outputs back
    Xp = torch.from_numpy(Xh).pin_memory()   # the e2e leg's step inputs (steps S..S+K-1)
    LGp = torch.from_numpy(LGh).pin_memory()
    Yp = torch.empty((L, T, H)).pin_memory()
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(S, S + args.steps):
        step(s, host_io=(Xp, LGp, Yp))
    stream.synchronize()
    e2e_s = time.perf_counter() - t0
    barrier()
    e2e_ms, e2e_tokens = over_ranks(e2e_s * 1e3, args.steps * T, world)
    e2e_tok = e2e_tokens / (e2e_ms / 1e3)
    log(f"e2e: {e2e_tok:.1f} tokens/s")

    # roofline of the fused expert-FFN layer kernel (routing, gate/up, SwiGLU,
    # down and combine in one launch per layer) over the fully resident
    # layers: their segment of every timed step graph (CUDA events on the
    # context stream), algorithmic bytes = the weights of the experts each
    # launch uses (3 tensors) + x and y
    blob = wl.tensor_bytes(0)
    peaks, peak_src = load_peaks()
    if seg is not None and seg_n > 0:
        alg = 0
        for s in range(args.warmup, S):
            for l in resident:
                alg += len(np.unique(LGh[s, l].argsort(axis=1)[:, -k:])) * 3 * blob + 2 * T * H * 4
        n_launch = seg_n * len(resident)
        launch_us = 1e3 * seg_ms / n_launch
        achieved = alg / (seg_ms / 1e3) / 1e9
        roof_how = "segment of the timed step graph: fully resident layers, events around the segment"
    else:
        # eager pass with events around each launch (no graph)
        graph = None
        qec.moe_debug_timing(ctx, True)
        gu_ms, alg, n_launch = 0.0, 0, 0
        for s in range(args.warmup, args.warmup + min(args.steps, 32)):
            step(s)
            g_ms, _ = qec.moe_debug_timing_read(ctx, L)
            for l in resident:
                gu_ms += g_ms[l]
                alg += len(np.unique(LGh[s, l].argsort(axis=1)[:, -k:])) * 3 * blob + 2 * T * H * 4
                n_launch += 1
        qec.moe_debug_timing(ctx, False)
        launch_us = 1e3 * gu_ms / max(1, n_launch)
        achieved = alg / (gu_ms / 1e3) / 1e9
        roof_how = "eager launches, events around each launch"
    traffic = read_traffic("decode_layer_kernel_decode_b1.txt", "bench.traffic_bytes_per_launch")

    # bytes of the whole step (weights of the unique experts of every layer)
    step_bytes = 0
    for l in range(L):
        u = len(np.unique(LGh[args.warmup, l].argsort(axis=1)[:, -k:]))
        step_bytes += u * 3 * blob
    # host link: zero-copy 128-bit reads of pinned host memory and copy-engine H2D
    probe = torch.empty(2 << 30, dtype=torch.uint8).pin_memory()
    zc_gbs, ce_gbs = qec.moe_probe_host_read(probe.data_ptr(), probe.numel(), iters=5)
    del probe
    log(f"host link: zero-copy read {zc_gbs:.1f} GB/s, copy engine {ce_gbs:.1f} GB/s")
    lookahead = None
    if args.lookahead_steps > 0 and seg is not None:
        lookahead = run_lookahead_leg(args, qec, synth, torch, log, ctx, stream, resident, blob)
    out = {
        "metric": METRIC, "value": round(tok_per_s, 2), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": decode_workload_desc(wl),
                   "l2": "inputs larger than L2: ~1.5 GB of expert weights per step vs 129 MB L2",
                   "cuda_graph": used_graph, "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": "decode_layer_kernel (fused expert FFN, resident layers)",
                     "achieved": round(achieved, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "peak_source": f"{peak_src} hbm_gbs (copy)", "traffic": traffic,
                     "algorithmic_bytes_per_launch": round(alg / max(1, n_launch)),
                     "avg_launch_us": round(launch_us, 3), "launches": n_launch, "timing": roof_how},
        "step_weight_gbs": round(step_bytes / (ms_max / args.steps / 1e3) / 1e9, 1),
        "host_link": {"zero_copy_read_gbs": round(zc_gbs, 1), "copy_engine_h2d_gbs": round(ce_gbs, 1)},
        "cache": {"hits": st_main["hits"], "misses": st_main["misses"], "admissions": st_main["admissions"],
                  "evictions": st_main["evictions"], "cold_bytes": st_main["cold_bytes"]},
        "e2e": {"value": round(e2e_tok, 2), "unit": "tokens/s",
                "h2d_bytes_per_step": int(Xh[0].nbytes + LGh[0].nbytes), "d2h_bytes_per_step": int(L * T * H * 4)},
        "clocks": clk,
        "gpu_launches": launches_per_step * args.steps,
    }
    if lookahead is not None:
        out["lookahead"] = lookahead
    qec.moe_destroy(ctx)
    del X, LG, Xp, LGp
    link_peak = max(zc_gbs, ce_gbs)
    out["host_link"]["peak_gbs"] = round(link_peak, 1)
    out["host_link"]["peak_source"] = "best of the zero-copy read probe and the copy-engine H2D probe, this run"
    if args.prefill_steps > 0:
        out["prefill"] = run_prefill_leg(args, qec, synth, torch, log)
        out["roofline_tensor"] = out["prefill"]["roofline_tensor"]
    if args.cold_launches > 0:
        out["cold_layer"] = run_cold_layer_leg(args, qec, synth, torch, log, link_peak)
    if args.pool_steps > 0:
        out["pool"] = run_pool_leg(args, qec, synth, torch, log, link_peak)
        out["roofline_link"] = {"pool_per_tensor": out["pool"]["per_tensor"]["roofline_link"],
                                "all_cold_layer": out.get("cold_layer", {}).get("roofline_link")}
    if args.large_decode_steps > 0:
        out["large_expert"] = run_large_expert_leg(args, qec, synth, torch, log)
    if args.q8_steps > 0:
        out["formats"] = {"q8_0": run_format_leg(args, qec, synth, torch, log, "decode_b1_q8_resident16"),
                          "q5_0": run_format_leg(args, qec, synth, torch, log, "decode_b1_q5_resident16"),
                          "q4_k": run_format_leg(args, qec, synth, torch, log, "decode_b1_q4k_resident16"),
                          "q6_k": run_format_leg(args, qec, synth, torch, log, "decode_b1_q6k_resident16"),
                          "q5_k": run_format_leg(args, qec, synth, torch, log, "decode_b1_q5k_resident16"),
                          "q4_shared_expert": run_format_leg(args, qec, synth, torch, log,
                                                             "decode_b1_shared_resident16", shared=True)}
    if rank == 0:
        out["cpu_baseline"] = cpu_baseline(wl, args.cpu_sample_steps, T) if args.cpu_sample_steps > 0 else None
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_case(args):
    """One layer of the decode / prefill workload shape with every expert
    resident, args.launches forwards on fresh seeded inputs, each timed with
    CUDA events; the small case that profiler captures run."""
    import torch
    import quantized_expert_cache_gb300 as qec
    import synth
    qec.load()
    H, F, E, k = 2048, 1152, 512, 8
    T = 4096 if args.case.startswith("prefill_layer") else 1
    if args.case == "prefill_layer_wide":
        E = 64  # ~512 tokens per expert: every token tile of the grouped GEMM full
    cap = 0 if args.case == "decode_layer_cold" else E
    fmt = synth.FMT_Q8_0 if args.case == "decode_layer_q8" else synth.FMT_Q4
    n = max(3, args.launches)
    wl = synth.Workload("case", H, E, k, F, 1, routing="zipf", zipf_s=1.1, capacity=[cap], weight_format=fmt)
    st = torch.cuda.current_stream()
    ctx = qec.moe_layer_init(H, F, E, k, 1, E, T, stream=st.cuda_stream, weight_format=fmt)
    for kind in range(3):
        rows, cols = wl.tensor_shapes[kind]
        qec.register_expert_tensor(ctx, 0, kind, wl.expert_tensor(0, kind), rows, cols, cap, wl.seed_order(0),
                                   cap)
    xs = [torch.from_numpy(wl.x(0, s, T)).cuda() for s in range(n)]
    lgs = [torch.from_numpy(wl.logits(0, s, T)).cuda() for s in range(n)]
    idx = torch.empty((n, T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((n, T, k), device="cuda")
    y = torch.empty((T, H), device="cuda")
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    kt = []
    qec.moe_debug_timing(ctx, True)
    for s in range(n):
        evs[s][0].record(st)
        qec.moe_ffn_forward_routed(ctx, 0, xs[s], lgs[s], T, idx[s], w[s], y, st.cuda_stream)
        evs[s][1].record(st)
        gu, dn = qec.moe_debug_timing_read(ctx, 1)
        kt.append((gu[0], dn[0]))
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in evs]
    qec.moe_destroy(ctx)
    res = {"case": args.case, "tokens": T, "launches": n, "median_ms_per_forward": round(float(np.median(ms[2:])), 5),
           "median_ms_gate_up_kernel": round(float(np.median([a for a, _ in kt[2:]])), 5),
           "median_ms_down_kernel": round(float(np.median([b for _, b in kt[2:]])), 5)}
    if T > 32:
        flop_gu = 2.0 * T * k * 2 * H * F
        res["gate_up_tflops"] = round(flop_gu / (res["median_ms_gate_up_kernel"] * 1e-3) / 1e12, 1)
        res["down_tflops"] = round(flop_gu / 2 / (res["median_ms_down_kernel"] * 1e-3) / 1e12, 1)
    if cap == 0:
        # every weight byte crosses the host link
        b = float(np.median(ms[2:]))
        res["host_link_gbs"] = round(k * 3 * wl.tensor_bytes(0) / (b * 1e-3) / 1e9, 1)
    print(json.dumps(res), flush=True)


def run_lookahead_leg(args, qec, synth, torch, log, ctx, stream, resident, blob):
    """Decode lookahead prefetch on the decode model (same weights and pool
    seeding as the headline workload) with the router model's inputs
    (decode_b1_resident_router: residual stream x_l = 0.9 x_(l-1) + ..., logits
    linear in x_l): the routers of all layers registered, then
    args.lookahead_steps batch-1 decode steps (48 routed layer launches in a
    CUDA graph + the promotion pass) from the seeded cache state, lookahead
    off and on, alternated twice.  Tokens/s from CUDA events around the timed
    steps, the resident layers' segment time, and the prediction hit rate."""
    wl = synth.WORKLOADS["decode_b1_resident_router"]
    L, H, E, k = wl.n_layers, wl.hidden, wl.n_experts, wl.top_k
    T = 1
    t0 = time.time()
    for l in range(L):
        qec.moe_set_router(ctx, l, wl.router_scale * wl.router(l), wl.router_bias(l))
    W, n = args.warmup, args.lookahead_steps
    Xh, LGh = make_inputs(wl, W + n, T)
    log(f"lookahead leg: routers and {W + n} steps of inputs in {time.time() - t0:.1f}s")
    X, LG = torch.from_numpy(Xh).cuda(), torch.from_numpy(LGh).cuda()
    sp = stream.cuda_stream
    xin = torch.empty((L, T, H), device="cuda")
    lin = torch.empty((L, T, E), device="cuda")
    idx = torch.empty((L, T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((L, T, k), device="cuda")
    y = torch.empty((L, T, H), device="cuda")
    seg = (torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))

    def layers(mark=False):
        for l in range(L):
            if mark and l == resident[0]:
                seg[0].record(stream)
            qec.moe_ffn_forward_routed(ctx, l, xin[l], lin[l], T, idx[l], w[l], y[l], sp)
            if mark and l == resident[-1]:
                seg[1].record(stream)

    runs = {"off": [], "on": []}
    for mode in ("off", "on", "off", "on"):
        qec.moe_set_lookahead(ctx, mode == "on")
        with torch.cuda.stream(stream):
            xin.copy_(X[0])
            lin.copy_(LG[0])
        layers()
        stream.synchronize()
        qec.miss_drain(ctx)
        qec.moe_cache_reset(ctx, False)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            layers(mark=True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        seg_ms = 0.0
        s0 = None
        for s in range(W + n):
            if s == W:
                stream.synchronize()
                s0 = qec.moe_stats(ctx)
                e0.record(stream)
            with torch.cuda.stream(stream):
                xin.copy_(X[s])
                lin.copy_(LG[s])
                graph.replay()
            qec.cache_step(ctx, T)
            if s >= W:
                seg_ms += seg[0].elapsed_time(seg[1])
        e1.record(stream)
        stream.synchronize()
        ms = e0.elapsed_time(e1)
        s1 = qec.moe_stats(ctx)
        pred = s1["lookahead_predicted"] - s0["lookahead_predicted"]
        hits = s1["lookahead_hits"] - s0["lookahead_hits"]
        r = {"tokens_per_s": round(n * T / (ms * 1e-3), 1), "ms_per_step": round(ms / n, 4),
             "resident_layer_us": round(1e3 * seg_ms / (n * len(resident)), 3),
             "prediction_hit_rate": round(hits / pred, 4) if pred else None}
        runs[mode].append(r)
        log(f"lookahead leg, {mode}: {r}")
        del graph
    qec.moe_set_lookahead(ctx, False)
    out = {"workload": (f"{wl.name}: the headline model's weights and pool seeding; inputs from the router model "
                        f"(residual stream rho {wl.residual_rho}, logits = log popularity + "
                        f"{wl.router_scale:.4f} R_l x_l); {n} timed batch-1 decode steps per run, CUDA graph, "
                        f"promotion pass after each step, runs from the seeded state"),
           "off": runs["off"][-1], "on": runs["on"][-1],
           "tokens_per_s_runs": {m: [r["tokens_per_s"] for r in v] for m, v in runs.items()},
           "prediction": f"top-{k} of layer l+1's router on layer l's input, pool-resident weights prefetched into L2"}
    out["speedup"] = round(out["on"]["tokens_per_s"] / out["off"]["tokens_per_s"], 4)
    return out


def run_cold_layer_leg(args, qec, synth, torch, log, link_peak):
    """One layer of the decode shape (hidden 2048, 512 experts, top-8, FFN
    1152) with every expert in pinned host memory: each batch-1 routed
    forward reads its 8 experts' 3 tensors zero-copy over the host link.
    args.cold_launches forwards on fresh seeded inputs, each timed with CUDA
    events (the first two untimed); link roofline = the weight bytes of the
    experts each forward uses over its median time, against the link probe."""
    H, F, E, k, T = 2048, 1152, 512, 8, 1
    n = max(3, args.cold_launches)
    wl = synth.Workload("cold_layer", H, E, k, F, 1, routing="zipf", zipf_s=1.1, capacity=[0])
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream
    ctx = qec.moe_layer_init(H, F, E, k, 1, 1, T, stream=sp)
    for kind in range(3):
        rows, cols = wl.tensor_shapes[kind]
        qec.register_expert_tensor(ctx, 0, kind, wl.expert_tensor(0, kind), rows, cols, 0, wl.seed_order(0), 0)
    xs = [torch.from_numpy(wl.x(0, s, T)).cuda() for s in range(n)]
    lgs = [torch.from_numpy(wl.logits(0, s, T)).cuda() for s in range(n)]
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), device="cuda")
    y = torch.empty((T, H), device="cuda")
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for s in range(n):
        evs[s][0].record(stream)
        qec.moe_ffn_forward_routed(ctx, 0, xs[s], lgs[s], T, idx, w, y, sp)
        evs[s][1].record(stream)
    stream.synchronize()
    qec.miss_drain(ctx)
    qec.moe_destroy(ctx)
    ms = float(np.median([a.elapsed_time(b) for a, b in evs[2:]]))
    byts = k * 3 * wl.tensor_bytes(0)
    gbs = byts / (ms * 1e-3) / 1e9
    log(f"all-cold layer: {ms * 1e3:.1f} us per forward, {gbs:.1f} GB/s over the host link")
    return {"workload": f"one layer, hidden {H}, {E} experts, top-{k}, FFN {F}, every expert in pinned host memory, "
                        f"batch-1 routed forwards",
            "us_per_forward": round(ms * 1e3, 2),
            "roofline_link": {"bound": "host link", "achieved": round(gbs, 1), "peak": round(link_peak, 1),
                              "unit": "GB/s", "frac": round(gbs / link_peak, 4), "bytes_per_forward": byts,
                              "what": "weights of the 8 experts each forward reads zero-copy, over the median "
                                      "event time of one forward"}}


def run_pool_leg(args, qec, synth, torch, log, link_peak):
    """Shared expert pool and prefill preheat against per-tensor pools, on
    the 25%-pool model (one registration; moe_cache_reset puts the seeded
    state back before every run).  (1) decode_b1_pool25: args.pool_steps
    batch-1 decode tokens from the seeded state with a pool per tensor, with
    one pool for all layers, and with a pool per tensor plus per-layer upload
    overlap (moe_set_upload_overlap), alternated twice.  (2)
    prompt_then_decode_pool25 (same weights and seeding, the request's
    popularity drifted from the seeding table), one pool: half of the pool is
    lent to a 4096-token prompt pass, given back refilled by seed order or,
    with prefill preheat, by the prompt's use counts, then args.pool_steps
    decode tokens.  Tokens/s from CUDA events around the decode loop (forwards
    and promotion passes), hit rate from the library's counters."""
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream
    wl = synth.WORKLOADS["decode_b1_pool25"]
    wp = synth.WORKLOADS["prompt_then_decode_pool25"]
    L, H, E, k, F = wl.n_layers, wl.hidden, wl.n_experts, wl.top_k, wl.ffn
    T = wp.phases[0][1]
    spt = max(wl.layer_capacity(l) for l in range(L))
    ctx = qec.moe_layer_init(H, F, E, k, L, spt, T, stream=sp)
    register_workload(qec, synth, ctx, wl, log)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), device="cuda")
    y = torch.empty((T, H), device="cuda")

    def inputs(w_, n, phase):
        X = np.stack([np.stack([w_.x(l, s, 1, phase) for l in range(L)]) for s in range(n)])
        LG = np.stack([np.stack([w_.logits(l, s, 1, phase) for l in range(L)]) for s in range(n)])
        return torch.from_numpy(X).cuda(), torch.from_numpy(LG).cuda()

    def decode(X, LG):
        n = X.shape[0]
        torch.cuda.synchronize()
        s0 = qec.moe_stats(ctx)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s in range(n):
            for l in range(L):
                qec.moe_ffn_forward_routed(ctx, l, X[s, l], LG[s, l], 1, idx[:1], w[:1], y[:1], sp)
            qec.cache_step(ctx, 1)
        e1.record(stream)
        stream.synchronize()
        ms = e0.elapsed_time(e1)
        s1 = qec.moe_stats(ctx)
        d = {key: s1[key] - s0[key] for key in ("hits", "misses", "admissions", "evictions", "cold_bytes",
                                                 "upload_bytes")}
        # host-link roofline of the run: every byte that crossed the link
        # (zero-copy weight reads by the kernels + promotion-pass uploads)
        # over the run's time, against the link probe of this run
        link_bytes = d["cold_bytes"] + d["upload_bytes"]
        gbs = link_bytes / (ms * 1e-3) / 1e9
        return {"tokens_per_s": round(n / (ms * 1e-3), 1), "ms_per_token": round(ms / n, 4),
                "hit_rate": round(d["hits"] / max(1, d["hits"] + d["misses"]), 4), **d,
                "roofline_link": {"bound": "host link", "achieved": round(gbs, 1), "peak": round(link_peak, 1),
                                  "unit": "GB/s", "frac": round(gbs / link_peak, 4),
                                  "bytes_per_token": round(link_bytes / n),
                                  "what": "zero-copy cold weight bytes + promotion-pass upload bytes, over the "
                                          "decode loop's event time (forwards and promotion passes)"}}

    out = {"workload": (f"{wl.name}: {L} layers, hidden {H}, {E} experts, top-{k}, FFN {F}, Zipf({wl.zipf_s}) "
                        f"routing, 128/512 experts per tensor seeded, {args.pool_steps} batch-1 decode tokens "
                        f"from the seeded state per run")}
    X, LG = inputs(wl, args.pool_steps, 0)
    # one untimed run first: the first decode after registration runs slower
    # (first touches of the pinned copies), whichever pool mode it uses
    qec.moe_cache_reset(ctx, False)
    decode(X[:32], LG[:32])
    runs = {"per_tensor": [], "global": [], "per_tensor_overlap": []}
    for name in ("per_tensor", "global", "per_tensor_overlap", "per_tensor", "global", "per_tensor_overlap"):
        qec.moe_cache_reset(ctx, name == "global")
        qec.moe_set_upload_overlap(ctx, name.endswith("overlap"))
        runs[name].append(decode(X, LG))
        log(f"pool leg, {wl.name}, {name} pool: {runs[name][-1]}")
    qec.moe_set_upload_overlap(ctx, False)
    for name, r in runs.items():
        out[name] = dict(r[-1], tokens_per_s_runs=[v["tokens_per_s"] for v in r])
    del X, LG
    # prompt pass, then decode
    n_borrow = 3 * L * spt // 2
    PX = [torch.from_numpy(wp.x(l, 0, T, 0)).cuda() for l in range(L)]
    PLG = [torch.from_numpy(wp.logits(l, 0, T, 0)).cuda() for l in range(L)]
    X, LG = inputs(wp, args.pool_steps, 1)
    prompt = {}
    for name in ("seed_refill", "preheat"):
        qec.moe_cache_reset(ctx, True)
        qec.moe_set_preheat(ctx, name == "preheat")
        qec.moe_pool_borrow(ctx, n_borrow)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for l in range(L):
            qec.route_topk(ctx, PLG[l], T, E, k, idx, w, sp)
            qec.moe_ffn_forward(ctx, l, PX[l], T, idx, w, y, sp)
        e1.record(stream)
        stream.synchronize()
        qec.miss_drain(ctx)
        qec.moe_pool_return(ctx)
        r = decode(X, LG)
        r["prompt_pass_ms"] = round(e0.elapsed_time(e1), 2)
        prompt[name] = r
        log(f"pool leg, {wp.name}, {name}: {r}")
    qec.moe_destroy(ctx)
    prompt["workload"] = (f"{wp.name}: one pool for all layers (128/512 per tensor seeded), {n_borrow} of "
                          f"{3 * L * spt} blocks lent to a {T}-token prompt pass (cold experts staged through the "
                          f"lent blocks), then {args.pool_steps} decode tokens; the request's popularity ranks "
                          f"drift from the seeding table (rank noise {wp.drift} x E)")
    out["prompt_then_decode"] = prompt
    return out


def run_format_leg(args, qec, synth, torch, log, name, shared=False):
    """Q8_0, Q5_0, Q4_K, Q6_K or Q5_K expert weights (or Q4 with a shared expert per layer) on
    16 fully resident layers of the decode shape: batch-1 decode steps
    captured in a CUDA graph (router top-k, plan, gate/up and down mat-vec
    launches per layer), timed with CUDA events on the context stream;
    roofline = the weights of the experts each step uses (3 tensors; the
    shared expert counts as one more) + x and y, over the step time."""
    wl = synth.WORKLOADS[name]
    L, H, E, k, F = wl.n_layers, wl.hidden, wl.n_experts, wl.top_k, wl.ffn
    fmt_name = {synth.FMT_Q4: "Q4", synth.FMT_Q8_0: "Q8_0", synth.FMT_Q5_0: "Q5_0",
                synth.FMT_Q4_K: "Q4_K", synth.FMT_Q6_K: "Q6_K", synth.FMT_Q5_K: "Q5_K"}[wl.weight_format]
    T = 1
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream
    ctx = qec.moe_layer_init(H, F, E, k, L, E, T, stream=sp, weight_format=wl.weight_format,
                             shared_experts=int(shared))
    register_workload(qec, synth, ctx, wl, log)
    if shared:
        sw = synth.Workload("shared", H, 1, 1, F, L, seed=wl.seed + 101, weight_format=wl.weight_format)
        for l in range(L):
            for kind in range(3):
                rows, cols = sw.tensor_shapes[kind]
                qec.register_shared_expert(ctx, l, kind, sw.expert_tensor(l, kind)[0], rows, cols)
    n = args.q8_steps
    W = args.warmup
    Xh, LGh = make_inputs(wl, W + n, T)
    X, LG = torch.from_numpy(Xh).cuda(), torch.from_numpy(LGh).cuda()
    xin = torch.empty((L, T, H), device="cuda")
    lin = torch.empty((L, T, E), device="cuda")
    idx = torch.empty((L, T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((L, T, k), device="cuda")
    y = torch.empty((L, T, H), device="cuda")

    def layers():
        for l in range(L):
            qec.moe_ffn_forward_routed(ctx, l, xin[l], lin[l], T, idx[l], w[l], y[l], sp)

    with torch.cuda.stream(stream):
        xin.copy_(X[0])
        lin.copy_(LG[0])
    layers()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        layers()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for s in range(W + n):
        if s == W:
            stream.synchronize()
            e0.record(stream)
        with torch.cuda.stream(stream):
            xin.copy_(X[s])
            lin.copy_(LG[s])
            graph.replay()
    e1.record(stream)
    stream.synchronize()
    ms = e0.elapsed_time(e1) / n
    blob = wl.tensor_bytes(0)
    alg = 0
    for s in range(W, W + n):
        for l in range(L):
            alg += (len(np.unique(LGh[s, l].argsort(axis=1)[:, -k:])) + int(shared)) * 3 * blob + 2 * T * H * 4
    alg /= n
    peaks, src = load_peaks()
    gbs = alg / (ms * 1e-3) / 1e9
    qec.moe_destroy(ctx)
    what = fmt_name + (" + shared expert" if shared else "")
    log(f"{what} leg: {T / (ms * 1e-3):.1f} tokens/s through {L} resident layers, {ms * 1e3 / L:.2f} us per "
        f"layer, {gbs:.0f} GB/s")
    return {"workload": f"{wl.name}: {L} layers, hidden {H}, {E} experts, top-{k}"
                        f"{' + 1 shared expert' if shared else ''}, FFN {F}, {fmt_name} blocks of 32 "
                        f"({synth.BLOCK_BYTES[wl.weight_format]} B per {synth.BLOCK_ELEMS[wl.weight_format]}), "
                        f"every expert resident, batch-1 decode, {n} timed "
                        f"steps in a CUDA graph",
            "tokens_per_s": round(T / (ms * 1e-3), 1), "us_per_layer": round(ms * 1e3 / L, 3),
            "roofline": {"bound": "hbm",
                         "kernels": f"topk + plan + gate_up_kernel<{fmt_name}> + down_kernel<{fmt_name}> per layer",
                         "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": f"{src} hbm_gbs (copy)",
                         "algorithmic_bytes_per_step": int(alg), "traffic": None}}


def run_large_expert_leg(args, qec, synth, torch, log):
    """The large-expert workload (hidden 2880, 128 experts, top-4, FFN 2880,
    36 layers, 64 of 128 experts per tensor seeded, uniform + Zipf(0.8)
    routing): 8 slots of every tensor lent to the prompt passes, prompts of
    512, 4096 and 12288 tokens through the 36 layers (grouped GEMM; cold
    experts uploaded a layer ahead by the lookahead prefetch), the slots given
    back, then batch 1, 8 and 32 decode steps with a promotion pass after
    each (per-layer upload overlap on: the forwards are issued eagerly).  Prompt tokens/s from CUDA events around the layer loop (one warm-up
    pass of each size first); decode tokens/s from CUDA events around
    args.large_decode_steps steps."""
    wl = synth.WORKLOADS["large_expert"]
    L, H, E, k, F = wl.n_layers, wl.hidden, wl.n_experts, wl.top_k, wl.ffn
    spt = max(wl.layer_capacity(l) for l in range(L))
    T_max = max(T for label, T, _ in wl.phases)
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream
    ctx = qec.moe_layer_init(H, F, E, k, L, spt, T_max, stream=sp)
    register_workload(qec, synth, ctx, wl, log)
    qec.moe_set_lookahead(ctx, True)
    idx = torch.empty((T_max, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T_max, k), device="cuda")
    y = torch.empty((T_max, H), device="cuda")
    n_borrow = 3 * L * 8
    qec.moe_pool_borrow(ctx, n_borrow)
    out = {"workload": (f"{wl.name}: {L} layers, hidden {H}, {E} experts, top-{k}, FFN {F}, 64/128 experts per "
                        f"tensor seeded, 0.5 uniform + 0.5 Zipf(0.8) routing; {n_borrow} pool blocks lent to the "
                        f"prompt passes (lookahead prefetch on), returned before decode"),
           "prefill": {}, "decode": {}}
    peaks, _ = load_peaks()
    for phase, (label, T, _) in enumerate(wl.phases):
        if label != "prefill":
            continue
        X = [torch.from_numpy(wl.x(l, 0, T, phase)).cuda() for l in range(L)]
        LG = [torch.from_numpy(wl.logits(l, 0, T, phase)).cuda() for l in range(L)]
        torch.cuda.synchronize()
        ms = []
        for rep in range(2):  # a warm-up pass, then the timed one
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for l in range(L):
                qec.route_topk(ctx, LG[l], T, E, k, idx, w, sp)
                qec.moe_ffn_forward(ctx, l, X[l], T, idx, w, y, sp)
            e1.record(stream)
            stream.synchronize()
            qec.miss_drain(ctx)
            ms.append(e0.elapsed_time(e1))
        tfl = 2.0 * T * k * 3 * H * F * L / (ms[-1] * 1e-3) / 1e12
        out["prefill"][str(T)] = {"tokens_per_s": round(T / (ms[-1] * 1e-3), 1), "ms_per_pass": round(ms[-1], 2),
                                  "tflops": round(tfl, 1), "frac_of_bf16_peak": round(tfl / peaks["bf16_tflops"], 4)}
        log(f"large expert prefill {T}: {out['prefill'][str(T)]}")
        del X, LG
    qec.moe_pool_return(ctx)
    # decode is issued eagerly here: each layer waits only for its own uploads
    qec.moe_set_upload_overlap(ctx, True)
    n = args.large_decode_steps
    for phase, (label, T, _) in enumerate(wl.phases):
        if label != "decode":
            continue
        Xh, LGh = [], []
        for s in range(n):
            Xh.append(np.stack([wl.x(l, s, T, phase) for l in range(L)]))
            LGh.append(np.stack([wl.logits(l, s, T, phase) for l in range(L)]))
        X, LG = torch.from_numpy(np.stack(Xh)).cuda(), torch.from_numpy(np.stack(LGh)).cuda()
        s0 = qec.moe_stats(ctx)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s in range(n):
            for l in range(L):
                qec.moe_ffn_forward_routed(ctx, l, X[s, l], LG[s, l], T, idx[:T], w[:T], y[:T], sp)
            qec.cache_step(ctx, T)
        e1.record(stream)
        stream.synchronize()
        ms = e0.elapsed_time(e1)
        s1 = qec.moe_stats(ctx)
        hits, misses = s1["hits"] - s0["hits"], s1["misses"] - s0["misses"]
        out["decode"][str(T)] = {"tokens_per_s": round(n * T / (ms * 1e-3), 1), "ms_per_step": round(ms / n, 4),
                                 "hit_rate": round(hits / max(1, hits + misses), 4)}
        log(f"large expert decode batch {T}: {out['decode'][str(T)]}")
    qec.moe_destroy(ctx)
    return out


def run_prefill_leg(args, qec, synth, torch, log):
    """One prefill micro-batch through every layer of the prefill workload
    (grouped tensor-core GEMM, cold experts read zero-copy), timed with CUDA
    events after one warm-up pass."""
    wl = synth.WORKLOADS[args.prefill_workload]
    label, T, _ = wl.phases[0]
    L, H, E, k, F = wl.n_layers, wl.hidden, wl.n_experts, wl.top_k, wl.ffn
    stream = torch.cuda.Stream()
    spt = max(wl.layer_capacity(l) for l in range(L))
    ctx = qec.moe_layer_init(H, F, E, k, L, spt, T, stream=stream.cuda_stream)
    register_workload(qec, synth, ctx, wl, log)
    x = [torch.from_numpy(wl.x(l, 0, T)).cuda() for l in range(L)]
    lg = [torch.from_numpy(wl.logits(l, 0, T)).cuda() for l in range(L)]
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), device="cuda")
    y = torch.empty((T, H), device="cuda")
    sp = stream.cuda_stream

    def pass_():
        for l in range(L):
            qec.route_topk(ctx, lg[l], T, E, k, idx, w, sp)
            qec.moe_ffn_forward(ctx, l, x[l], T, idx, w, y, sp)

    def timed(gemm_events=False):
        pass_()
        stream.synchronize()
        qec.miss_drain(ctx)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        per_layer = np.zeros(L)
        gemm_ms = np.zeros((L, 2))
        total = 0.0
        qec.moe_debug_timing(ctx, gemm_events)
        for s in range(args.prefill_steps):
            with torch.cuda.stream(stream):
                e0.record()
                for l in range(L):
                    qec.route_topk(ctx, lg[l], T, E, k, idx, w, sp)
                    ev[l][0].record()
                    qec.moe_ffn_forward(ctx, l, x[l], T, idx, w, y, sp)
                    ev[l][1].record()
                e1.record()
            stream.synchronize()
            qec.miss_drain(ctx)
            total += e0.elapsed_time(e1)
            per_layer += np.array([a.elapsed_time(b) for a, b in ev])
            if gemm_events:
                gu, dn = qec.moe_debug_timing_read(ctx, L)
                gemm_ms += np.stack([gu, dn], axis=1)
        qec.moe_debug_timing(ctx, False)
        n = args.prefill_steps
        return total / n, per_layer / n, gemm_ms / n

    # cold experts read zero-copy by the GEMM's converters, then with the
    # lookahead prefetch (layer l + 1's cold experts uploaded by the copy
    # engine while layer l computes)
    ms_zc, per_layer_zc, _ = timed()
    qec.moe_set_lookahead(ctx, True)
    # the lookahead pass, with events around each layer's two GEMM kernels
    # (the per-layer times then include the event records: a few us)
    ms, per_layer, gemm_ms = timed(gemm_events=True)
    flop = 2.0 * T * k * 3 * H * F
    peaks, src = load_peaks()
    best = float(per_layer.min())
    tfl = flop / (best * 1e-3) / 1e12
    # tensor roofline of the grouped GEMM kernels alone: 2 A (2 H F) flops of
    # gate/up and 2 A F H of down per layer (A = T k assignments), over their
    # own event time, summed over the pass's layers
    gk_ms = float(gemm_ms.sum())
    gk_tfl = L * flop / (gk_ms * 1e-3) / 1e12
    peak_t = peaks.get("bf16_tflops_sustained") or peaks.get("bf16_tflops", 1900.0)
    gu_tfl = L * 2.0 * T * k * 2 * H * F / (float(gemm_ms[:, 0].sum()) * 1e-3) / 1e12
    dn_tfl = L * 2.0 * T * k * H * F / (float(gemm_ms[:, 1].sum()) * 1e-3) / 1e12
    qec.moe_destroy(ctx)
    log(f"prefill: {T / (ms * 1e-3):.0f} tokens/s through {L} layers with lookahead prefetch "
        f"({T / (ms_zc * 1e-3):.0f} with zero-copy cold reads), best layer {best:.3f} ms = {tfl:.1f} TFLOP/s")
    return {"workload": f"{wl.name}: {T} tokens, {L} layers, hidden {H}, {E} experts, top-{k}, FFN {F}, "
                        f"pool {wl.layer_capacity(0)}/{E} per layer",
            "cold_experts": "uploaded a layer ahead by the copy engine (lookahead prefetch)",
            "tokens_per_s": round(T / (ms * 1e-3), 1), "ms_per_pass": round(ms, 3),
            "layer_ms_median": round(float(np.median(per_layer)), 3),
            "zero_copy": {"tokens_per_s": round(T / (ms_zc * 1e-3), 1),
                          "layer_ms_median": round(float(np.median(per_layer_zc)), 3)},
            "gemm": {"bound": "tensor", "achieved_tflops_best_layer": round(tfl, 1),
                     "peak_tflops": peaks.get("bf16_tflops"), "unit": "TFLOP/s",
                     "frac": round(tfl / peaks.get("bf16_tflops", 1900.0), 4),
                     "note": "kind::f16 MMA on integer-valued fp16 operands (sm_103a has no tcgen05 kind::i8); "
                             "per-layer time includes quantize, sort, gather, both GEMMs and the combine"},
            "roofline_tensor": {"bound": "tensor", "kernel": "grouped GEMM kernels (gate/up + SwiGLU + h "
                                                             "quantization, down)",
                                "achieved": round(gk_tfl, 1), "peak": peak_t, "unit": "TFLOP/s",
                                "frac": round(gk_tfl / peak_t, 4),
                                "peak_source": f"{src} bf16_tflops_sustained (the GEMMs run inside a "
                                               f"{ms:.0f} ms pass; kind::f16 runs at the bf16 rate)",
                                "gate_up_tflops": round(gu_tfl, 1), "down_tflops": round(dn_tfl, 1),
                                "gemm_ms_per_layer": round(gk_ms / L, 4),
                                "flops_per_layer": flop,
                                "timing": "CUDA events around each GEMM launch on the context stream, all "
                                          f"{L} layers of the lookahead pass"}}


# ----------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# ----------------------------------------------------------------------------

def oracle_layer_token(oracle, wl, layer, step, T, cache):
    x, lg = wl.x(layer, step, T), wl.logits(layer, step, T)
    idx, w = oracle.topk(lg, wl.top_k)
    used = sorted(set(idx.ravel().tolist()))
    tens = []
    for kind in range(3):
        d = {}
        for e in used:
            key = (layer, kind, e)
            if key not in cache:
                cache[key] = wl.expert_tensor(layer, kind, e, e + 1)[0]
            d[e] = cache[key]
        tens.append(d)
    return x, idx, w, tens


def cpu_baseline(wl, n_steps, T):
    """The oracle as it stands, single-threaded, on a bounded sample: n_steps
    decode steps through all layers (weights generated outside the timing)."""
    import oracle
    cache = {}
    work = []
    for s in range(n_steps):
        for l in range(wl.n_layers):
            work.append(oracle_layer_token(oracle, wl, l, s, T, cache))
    t0 = time.perf_counter()
    for x, idx, w, (g, u, d) in work:
        oracle.layer(x, idx, w, g, u, d, wl.hidden, wl.ffn)
    dt = time.perf_counter() - t0
    return {"value": round(n_steps * T / dt, 4), "unit": "tokens/s", "cores": 1, "host_cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{n_steps} decode steps x {wl.n_layers} layers (batch {T}), single-threaded C oracle, "
                      f"{dt:.1f}s"}


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    import oracle
    import synth
    wl = synth.WORKLOADS[args.workload]
    label, T, _ = wl.phases[0]
    L = wl.n_layers
    layers = list(range(0, L, 12))  # bounded sample: 4 of the 48 layers per step
    cache = {}
    per_step = []
    for s in range(args.warmup + args.steps):
        work = [oracle_layer_token(oracle, wl, l, s, T, cache) for l in layers]
        t0 = time.perf_counter()
        for x, idx, w, (g, u, d) in work:
            oracle.layer(x, idx, w, g, u, d, wl.hidden, wl.ffn)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            per_step.append(dt)
        if len(cache) > 3 * 8 * 64:
            cache.clear()
    sample_s = float(np.mean(per_step))     # measured: the sampled layers of one step
    step_s = sample_s * L / len(layers)     # extrapolated to all layers of the step
    value = T / step_s
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sample_s * 1e3, 2),
        "ms_per_step_what": f"measured time of one step's sampled work ({len(layers)} of {L} layers, one token)",
        "ms_per_step_extrapolated": round(step_s * 1e3, 2),
        "extrapolation": f"value = tokens / (measured sample time x {L}/{len(layers)}): the oracle's layers all cost "
                         f"the same (same shapes, 8 experts each)",
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": decode_workload_desc(wl), "parallelism": "single host core (the CPU oracle)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": 1, "host_cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"each step: layers {layers} of {L} for one token, scaled by {L}/{len(layers)}"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    a = parse()
    if a.case:
        run_case(a)
    elif a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)

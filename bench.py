"""Benchmark of the batch-invariant MoE prefill path on GB300.

One step = one pass of the whole path over one prefill batch of M = 4096
tokens (16 requests of 256) through 40 layers; each layer runs:
  bi_router_gate_topk F32 router, H=2048, E=256, top-8 (logits, ids,
                      weights, margins) with the shared-expert gate dot and
                      sigmoid fused into its selection kernel
  bi_route_trace_hash per-request FNV-1a hashes, chained over the layers (on
                      a side stream: it only reads that layer's ids)
  bi_gemm_bf16        the M-invariant bf16 projection, K = N = 4096
Every layer has its own weights and its own hidden states, so a step
streams about 4 GB (inputs larger than the 129 MB L2; no flush needed).

value: tokens/s of whole steps (all ranks).  Per-part device times come from
CUDA events recorded around each call inside the timed steps; the roofline
object describes the dominant kernel.

--impl reference times the CPU oracle (the plain C reference the tests
check against) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

LAYERS, M, H, E, K_TOP = 40, 4096, 2048, 256, 8
G_N = G_K = 4096
N_REQ = 16
METRIC = "router+top-k tokens/s & M-invariant bf16 GEMM TFLOP/s, % of roofline"
WORKLOAD = ("moe-prefill block prologue: 40 layers x (F32 router H2048 E256 top8 + shared gate + "
            "route hash + bf16 projection K=N=4096), M=4096 tokens (16 requests x 256)")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6781.4), d.get("bf16_tflops", 1897.4), d.get("bf16_tflops_sustained", 1683.3), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu
# capture of the kernel as it stands, at this launch shape; None where no capture of the
# current code exists.  Reset to None whenever the kernel changes.  The router call is
# its two launches (projection + selection) captured inside the layer sequence with the
# caches as the preceding kernels left them (mean of two layers); its writes include L2
# evictions of the preceding kernels' dirty lines.
NCU_TRAFFIC = {# every kernel here gained its failure-path drains after its last capture
               # (the normal path's loads and stores are unchanged, but the counters were
               # taken on the earlier code): no figure until they are captured again
               "gemm_bf16_kernel": None,
               "moe_call": None,
               "router_call": None,
               "rmsnorm_kernel": None,
               "attn_prefill_kernel": None}


def fp32_peak(torch, dev) -> dict:
    """The FP32 FMA peak from this GPU's unit counts and its maximum SM clock:
    SMs (device properties) x 128 FP32 lanes x 2 flop x the maximum SM clock
    (nvidia-smi clocks.max.sm).  None where the clock cannot be read."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = None
    try:
        out = subprocess.run(["nvidia-smi", "-i", str(dev.index or 0), "--query-gpu=clocks.max.sm",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=20)
        mhz = float(out.stdout.strip().splitlines()[0])
    except (OSError, ValueError, IndexError, subprocess.SubprocessError):
        pass
    tflops = sms * 128 * 2 * mhz * 1e6 / 1e12 if mhz else None
    return {"tflops": tflops, "sms": sms, "sm_max_mhz": mhz,
            "source": f"derived: {sms} SMs x 128 FP32 lanes x 2 flop x {mhz} MHz (nvidia-smi clocks.max.sm)"}


class Clocks:
    """nvidia-smi sampled every 25 ms, each sample stamped by nvidia-smi
    itself; only the samples whose stamps fall inside the timed region count
    (mark() opens it, stop() closes it).  The region of a default run is
    about 0.1 s, so it holds a few samples."""

    def __init__(self, gpu_index: int):
        q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        self.t_begin = None
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={q}",
                                       "--format=csv,noheader,nounits", "-lms", "25"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.5)          # let nvidia-smi start sampling before the region opens
        except OSError:
            self.p = None

    def mark(self):
        import datetime
        self.t_begin = datetime.datetime.now()

    def stop(self, t_end=None):
        """Close the region (now, unless t_end is given) and summarise the
        samples stamped inside it."""
        import datetime
        t_end = t_end or datetime.datetime.now()
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)              # the sample that straddles the end
        self.p.terminate()
        out, _ = self.p.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
                rows.append((ts, float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        t0 = self.t_begin or t_end
        inside = [r for r in rows if t0 <= r[0] <= t_end]
        widened = False
        if not inside:               # region shorter than the sampling interval
            pad = datetime.timedelta(milliseconds=100)
            inside = [r for r in rows if t0 - pad <= r[0] <= t_end + pad]
            widened = True
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = {n for r in inside for n, v in zip(names, r[3]) if v.lower() == "active"}
        sm = [r[1] for r in inside]
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(r[2] for r in inside) if inside else None,
               "reasons": sorted(reasons), "samples": len(sm),
               "region_s": (t_end - t0).total_seconds()}
        if widened:
            out["window"] = "widened by 100 ms on each side (no sample inside the region)"
        return out


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x: float, device="cpu") -> float:
    """The maximum of x over all ranks (x itself when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_per_step: int, world_size: int, steps: int, max_seconds: float) -> float:
    """Units processed by all ranks divided by the slowest rank's time: every
    rank runs its own replica of the step (tokens shard with no collective)."""
    return units_per_rank_per_step * world_size * steps / max_seconds


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from serving_numerics_gb300 import binding as bi
    from serving_numerics_gb300 import synth

    ws, rank, local = dist_setup()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    bi.load()
    dev = torch.device("cuda", local)
    seed = 1000 + rank

    if args.moe_only:
        # the grouped expert GEMM alone (a small case for profiling): one
        # router call supplies the ids and weights
        x0 = synth.device_normal((M, H), seed * 100 + 200, 1.0, torch.float32, dev)
        w0 = synth.device_normal((E, H), seed * 100, 0.02, torch.float32, dev)
        r = bi.router_topk(x0, w0, K_TOP)
        hbm = peaks()[0]
        if rank == 0:
            print(json.dumps({"moe_expert_gemm": moe_measure(bi, synth, torch, dev, hbm, x0, r["ids"],
                                                             r["weights"], reps=args.moe_reps)}), flush=True)
        return

    # resident weights and inputs (seeded, drawn on the device)
    Wg = [synth.device_normal((E, H), seed * 100 + l, 0.02, torch.float32, dev) for l in range(LAYERS)]
    Wsg = [synth.device_normal((H,), seed * 100 + 50 + l, 0.02, torch.float32, dev) for l in range(LAYERS)]
    Bw = [synth.device_normal((G_N, G_K), seed * 100 + 100 + l, 1 / 64, torch.bfloat16, dev) for l in range(LAYERS)]
    X = [synth.device_normal((M, H), seed * 100 + 200 + l, 1.0, torch.float32, dev) for l in range(LAYERS)]
    A = [synth.device_normal((M, G_K), seed * 100 + 300 + l, 1 / 64, torch.bfloat16, dev) for l in range(LAYERS)]
    logits = torch.empty((LAYERS, M, E), dtype=torch.float32, device=dev)
    ids = torch.empty((LAYERS, M, K_TOP), dtype=torch.int32, device=dev)
    wts = torch.empty((LAYERS, M, K_TOP), dtype=torch.float32, device=dev)
    mg = torch.empty((LAYERS, M), dtype=torch.float32, device=dev)
    mu = torch.empty((LAYERS, M), dtype=torch.int32, device=dev)
    gdot = torch.empty((LAYERS, M), dtype=torch.float32, device=dev)
    gsig = torch.empty((LAYERS, M), dtype=torch.float32, device=dev)
    Cout = torch.empty((M, G_N), dtype=torch.bfloat16, device=dev)
    hashes = torch.empty((N_REQ,), dtype=torch.int64, device=dev)
    ws_router = bi.router_workspace(M, E, dev)      # caller-owned: the library allocates nothing
    offs = [i * (M // N_REQ) for i in range(N_REQ + 1)]
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    # the route hash only reads each layer's ids: it runs on a side stream,
    # ordered after that layer's router by an event, chained layer to layer
    side = torch.cuda.Stream(dev)
    ids_ready = [torch.cuda.Event() for _ in range(LAYERS)]
    # kernels per layer: the router call's (as the library plans it for this
    # M: its projection launches and the selection with the shared gate
    # fused in), then the route hash and the GEMM
    launches_per_layer = bi.router_plan(M, E)[2] + 2

    def layer(l, ev=None):
        if ev is not None:
            ev[0].record(stream)
        bi.bi_router_gate_topk(X[l], Wg[l], Wsg[l], bi.BI_F32, bi.BI_F32, M, H, E, K_TOP, logits[l], ids[l],
                               wts[l], mg[l], mu[l], gdot[l], gsig[l], workspace=ws_router, stream=sh)
        ids_ready[l].record(stream)
        if ev is not None:
            ev[1].record(stream)
        side.wait_event(ids_ready[l])
        bi.bi_route_trace_hash(ids[l], M, K_TOP, offs, None if l == 0 else hashes, hashes,
                               stream=side.cuda_stream)
        if ev is not None:
            ev[2].record(stream)
        bi.bi_gemm_bf16(A[l], Bw[l], Cout, M, G_N, G_K, G_K, G_K, G_N, stream=sh)
        if ev is not None:
            ev[3].record(stream)

    def step(evs=None):
        for l in range(LAYERS):
            layer(l, None if evs is None else evs[l])
        stream.wait_stream(side)      # the step ends when every hash is done

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0

    # --- timed region: K steps, per-call events inside, clocks sampled
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(LAYERS)]
           for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = Clocks(local)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark()
    t0.record(stream)
    for s in range(args.steps):
        step(evs[s])
    t1.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    ck = clocks.stop()
    ms = reduce_max(t0.elapsed_time(t1), dev)
    router_ms = [evs[s][l][0].elapsed_time(evs[s][l][1]) for s in range(args.steps) for l in range(LAYERS)]
    gemm_ms = [evs[s][l][2].elapsed_time(evs[s][l][3]) for s in range(args.steps) for l in range(LAYERS)]
    assert bi.bi_get_last_device_error() == 0

    # --- end to end: inputs from pinned host memory, results back to host
    pin_X = [torch.empty((M, H), dtype=torch.float32, pin_memory=True) for _ in range(LAYERS)]
    pin_A = [torch.empty((M, G_K), dtype=torch.bfloat16, pin_memory=True) for _ in range(LAYERS)]
    for l in range(LAYERS):
        pin_X[l].copy_(X[l])
        pin_A[l].copy_(A[l])
    # every layer's routing decision comes back (ids, weights, margins, gate),
    # plus the per-request route hashes; the logits and the projection output
    # stay on the device, where the next layer of a model would read them
    res = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
           for n, t in (("ids", ids), ("weights", wts), ("margin", mg), ("margin_ulps", mu),
                        ("gate_dot", gdot), ("gate_sigmoid", gsig))}
    res_h = torch.empty((N_REQ,), dtype=torch.int64, pin_memory=True)
    # inputs stream in on a copy stream ahead of the compute that needs them;
    # a layer's buffers are refilled only once the previous step's compute of
    # that layer is done with them; each layer's results go back on a second
    # copy stream as soon as that layer's router is done
    e2e_steps = max(1, min(args.steps, 5))
    copy = torch.cuda.Stream(dev)
    back = torch.cuda.Stream(dev)
    arrived = [torch.cuda.Event() for _ in range(LAYERS)]
    consumed = [torch.cuda.Event() for _ in range(LAYERS)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    for step_i in range(e2e_steps):
        for l in range(LAYERS):
            if step_i > 0:
                copy.wait_event(consumed[l])
            with torch.cuda.stream(copy):
                X[l].copy_(pin_X[l], non_blocking=True)
                A[l].copy_(pin_A[l], non_blocking=True)
            arrived[l].record(copy)
        for l in range(LAYERS):
            stream.wait_event(arrived[l])
            layer(l)
            consumed[l].record(stream)
            back.wait_event(ids_ready[l])
            with torch.cuda.stream(back):
                for n, src in (("ids", ids), ("weights", wts), ("margin", mg), ("margin_ulps", mu),
                               ("gate_dot", gdot), ("gate_sigmoid", gsig)):
                    res[n][l].copy_(src[l], non_blocking=True)
        back.wait_stream(side)
        with torch.cuda.stream(back):
            res_h.copy_(hashes, non_blocking=True)
        back.synchronize()         # this step's results are on the host
        stream.synchronize()
    e2e_s = reduce_max(time.perf_counter() - w0, dev)
    h2d = LAYERS * (M * H * 4 + M * G_K * 2)
    d2h = sum(t.numel() * t.element_size() for t in res.values()) + N_REQ * 8
    # the host link's own rate: one layer's inputs copied alone, as above
    torch.cuda.synchronize()
    c0 = time.perf_counter()
    n_probe = min(8, len(X))
    for l in range(n_probe):
        with torch.cuda.stream(copy):
            X[l].copy_(pin_X[l], non_blocking=True)
            A[l].copy_(pin_A[l], non_blocking=True)
    copy.synchronize()
    h2d_gbs = n_probe * (M * H * 4 + M * G_K * 2) / (time.perf_counter() - c0) / 1e9
    copy_bound = M * ws / (h2d / (h2d_gbs * 1e9))

    fma_tflops = fma_probe(bi, torch, dev)
    fma2_tflops = fma_probe(bi, torch, dev, packed=True)
    fp32 = fp32_peak(torch, dev)
    FP32_PEAK_TFLOPS = fp32["tflops"] or fma_tflops
    margins_bf16 = margin_histogram_bf16(torch, logits, K_TOP)
    hbm, bf16_burst, bf16_sus, src = peaks()
    value = whole_job_rate(M, ws, args.steps, ms / 1e3)
    g_avg = statistics.mean(gemm_ms) / 1e3
    r_avg = statistics.mean(router_ms) / 1e3
    g_flop = 2.0 * M * G_N * G_K
    r_flop = 2.0 * M * (E + 1) * H             # E gate rows + the shared-expert gate row
    r_bytes = 4 * (E + 1) * H + 4 * M * H + 4 * M * E + 8 * M * K_TOP + 8 * M + 8 * M
    g_bytes = 2 * (M * G_K + G_N * G_K + M * G_N)
    roof_gemm = {"bound": "tensor", "achieved": g_flop / g_avg / 1e12, "peak": bf16_sus,
                 "unit": "TFLOP/s", "frac": g_flop / g_avg / 1e12 / bf16_sus,
                 "traffic": NCU_TRAFFIC["gemm_bf16_kernel"],
                 "kernel": "gemm_bf16_kernel (one launch per call)",
                 "peak_source": f"{src} bf16 sustained (kernel timed inside a long step), of {src}",
                 "algorithmic_bytes": g_bytes}
    roof_router = {"bound": "alu", "achieved": r_flop / r_avg / 1e12, "peak": FP32_PEAK_TFLOPS,
                   "unit": "TFLOP/s", "frac": r_flop / r_avg / 1e12 / FP32_PEAK_TFLOPS,
                   "traffic": NCU_TRAFFIC["router_call"],
                   "kernel": "bi_router_gate_topk call: router_proj_persist_kernel (the persistent projection, "
                             "shared gate included) + router_select_kernel, timed as one call, so the selection "
                             "counts against the projection",
                   "algorithmic_bytes": r_bytes, "hbm_time_frac": (r_bytes / (hbm * 1e9)) / r_avg,
                   "peak_source": fp32["source"] if fp32["tflops"] else "the FMA probe (clock not readable)",
                   "fma_probe_tflops": fma_tflops, "fma_probe_packed_tflops": fma2_tflops,
                   "frac_of_fma_probe": r_flop / r_avg / 1e12 / fma_tflops}
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 router / bf16 GEMM (f32 accumulate)",
        "data": "synthetic (seeded normal draws, shapes of the pages' workloads)",
        "config": {"workload": WORKLOAD, "tokens_per_step_per_gpu": M, "layers": LAYERS,
                   "parallelism": f"replicas x{ws} (tokens sharded, no collective)",
                   "l2": "inputs larger than L2 (about 4 GB streamed per step)"},
        "parts": {
            "router_topk_tokens_per_s": M / r_avg, "router_call_us": r_avg * 1e6,
            "router_tflops": r_flop / r_avg / 1e12,
            "gemm_tflops": g_flop / g_avg / 1e12, "gemm_call_us": g_avg * 1e6,
            "gemm_frac_of_bf16_sustained": g_flop / g_avg / 1e12 / bf16_sus,
        },
        "roofline_gemm": roof_gemm,
        "roofline_router": roof_router,
        # the kernel with the larger share of the step's device time
        "roofline": roof_router if r_avg >= g_avg else roof_gemm,
        "e2e": {"value": whole_job_rate(M, ws, e2e_steps, e2e_s), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "returns": "every layer's ids, weights, margin, margin_ulps, gate dot and sigmoid, and the "
                           "16 chained route hashes; logits and projection outputs stay on the device",
                "h2d_gbs_measured": h2d_gbs, "copy_bound_tokens_per_s": copy_bound,
                "frac_of_copy_bound": whole_job_rate(M, ws, e2e_steps, e2e_s) / copy_bound},
        "gpu_launches": launches_per_layer * LAYERS * args.steps,
        "clocks": ck,
    }
    out["margins_f32_router_in_bf16_ulps"] = margins_bf16
    out["fp32_peak"] = {"derived_tflops": fp32["tflops"], "source": fp32["source"],
                        "fma_probe_tflops": fma_tflops, "fma_probe_packed_tflops": fma2_tflops}
    if not args.no_sweep:
        del X, A, Bw, Wg, Wsg, pin_X, pin_A
        torch.cuda.empty_cache()
        out["router_sweep"] = router_sweep(bi, synth, torch, dev, hbm, FP32_PEAK_TFLOPS)
        out["gemm_sweep"] = gemm_sweep(bi, synth, torch, dev, bf16_burst, bf16_sus)
        out["tie_heavy_bf16_router"] = tie_heavy_measure(bi, synth, torch, dev)
        out["mixed_prefill"] = mixed_prefill_measure(bi, synth, torch, dev)
        out["context_m_variant"] = m_variant_context(bi, synth, torch, dev)
        xs0 = synth.device_normal((M, H), seed * 100 + 200, 1.0, torch.float32, dev)
        out["moe_expert_gemm"] = moe_measure(bi, synth, torch, dev, hbm, xs0, ids[0], wts[0])
        xs = [synth.device_normal((M, H), seed * 100 + 200 + l, 1.0, torch.float32, dev) for l in range(LAYERS)]
        out["rmsnorm"] = rmsnorm_measure(bi, synth, torch, dev, hbm, xs)
        del xs
        out["attention_prefill"] = attention_measure(bi, synth, torch, dev, bf16_burst)
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_seconds)
    out["digest"] = digest(out)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws > 1:
        dist.destroy_process_group()


ROUTER_SWEEP_M = ([1, 2, 4, 8, 16, 19, 32] + list(range(35, 65)) +
                  [65, 75, 96, 128, 129, 256, 512, 1024, 2048, 4096])


def graph_time(torch, stream, fn, n, reps=3):
    """Seconds per call of fn(i) for i < n, captured once in a CUDA graph
    (so host launch cost is not timed; the calls keep their programmatic-
    dependent-launch edges) and replayed reps times between CUDA events."""
    fn_range = range(n)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in fn_range:
            fn(i)
    g.replay()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(reps):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    del g
    return a.elapsed_time(b) / 1e3 / (reps * n)


def router_sweep(bi, synth, torch, dev, hbm_gbs, fp32_tflops):
    """bi_router_topk alone (F32, H=2048, E=256, top-8, all outputs) at every M
    of ROUTER_SWEEP_M: back-to-back calls cycling through 96 gate matrices
    (192 MiB, more than L2) so every call reads its weights from HBM, in a
    CUDA graph; the per-call time is against the binding roofline
    max(bytes / HBM, flops / FP32).  floor_us: the same graph of the
    dependent-launch probe (one cluster launch that waits for its
    predecessor, reads one word and writes one), the fixed cost under any
    one-launch call."""
    pool = 96
    Ws = [synth.device_normal((E, H), 77000 + i, 0.02, torch.float32, dev) for i in range(pool)]
    res = []
    stream = torch.cuda.current_stream(dev)
    ws = bi.router_workspace(max(ROUTER_SWEEP_M), E, dev)
    for Mi in ROUTER_SWEEP_M:
        xs = [synth.device_normal((Mi, H), 78000 + i, 1.0, torch.float32, dev) for i in range(8)]
        lg = torch.empty((Mi, E), dtype=torch.float32, device=dev)
        ids = torch.empty((Mi, K_TOP), dtype=torch.int32, device=dev)
        w = torch.empty((Mi, K_TOP), dtype=torch.float32, device=dev)
        mg = torch.empty((Mi,), dtype=torch.float32, device=dev)
        mu = torch.empty((Mi,), dtype=torch.int32, device=dev)

        def call(i):
            bi.bi_router_topk(xs[i % 8], Ws[i % pool], bi.BI_F32, bi.BI_F32, Mi, H, E, K_TOP, lg, ids, w,
                              mg, mu, workspace=ws, stream=None)
        n = pool if Mi <= 1024 else pool // 2
        t = graph_time(torch, stream, call, n)
        byt = 4 * E * H + 4 * Mi * H + 4 * Mi * E + 8 * Mi * K_TOP + 8 * Mi
        flop = 2.0 * Mi * E * H
        t_hbm, t_alu = byt / (hbm_gbs * 1e9), flop / (fp32_tflops * 1e12)
        res.append({"M": Mi, "us": round(t * 1e6, 2), "launches": bi.router_plan(Mi, E)[2],
                    "bound": "hbm" if t_hbm >= t_alu else "alu",
                    "frac_binding": round(max(t_hbm, t_alu) / t, 4),
                    "frac_hbm": round((byt / t / 1e9) / hbm_gbs, 4)})
    del Ws
    a_ = torch.zeros(64, dtype=torch.float32, device=dev)
    b_ = torch.zeros(64, dtype=torch.float32, device=dev)
    floor = graph_time(torch, stream, lambda i: bi.selftest_dependent_floor(a_ if i % 2 == 0 else b_,
                                                                         b_ if i % 2 == 0 else a_), pool)
    return {"calls": res, "floor_us": round(floor * 1e6, 3),
            "note": "F32 H=2048 E=256 top-8, all outputs; 96 gate matrices cycled (192 MiB > L2), CUDA graph; "
                    "floor_us = one dependent cluster launch doing no arithmetic"}


def gemm_sweep(bi, synth, torch, dev, bf16_burst, bf16_sus):
    """bi_gemm_bf16 at every M of the projection workload (K = N = 4096,
    A, B ~ N(0,1)/64): back-to-back calls cycling 8 weight matrices and
    2 input matrices (256 MiB + 128 MiB, far more than L2), timed with
    CUDA events in a CUDA graph."""
    Ms = [1, 19, 64, 65, 75, 128, 1024, 2048, 4096, 8192]
    Bs = [synth.device_normal((G_N, G_K), 82000 + i, 1 / 64, torch.bfloat16, dev) for i in range(8)]
    As = [synth.device_normal((max(Ms), G_K), 82100 + i, 1 / 64, torch.bfloat16, dev) for i in range(2)]
    C_ = torch.empty((max(Ms), G_N), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    out = []
    for Mi in Ms:
        def call(i):
            bi.bi_gemm_bf16(As[i % 2], Bs[i % 8], C_, Mi, G_N, G_K, G_K, G_K, G_N, stream=None)
        n = 64 if Mi <= 1024 else 16
        t = graph_time(torch, stream, call, n)
        tf = 2.0 * Mi * G_N * G_K / t / 1e12
        out.append({"M": Mi, "us": round(t * 1e6, 2), "tflops": round(tf, 1),
                    "frac_sustained": round(tf / bf16_sus, 4), "frac_burst": round(tf / bf16_burst, 4)})
    del Bs, As
    return {"calls": out, "note": "K=N=4096 bf16, f32 accumulate; 8 weight matrices cycled (beyond L2), "
                                  "CUDA graph; peaks: measured bf16 sustained / burst"}


def tie_heavy_measure(bi, synth, torch, dev):
    """The tie-heavy bf16-logit router: H=2048, E=512, top-10, bf16 inputs on
    the {-1, +1} * 2^-8 grid, 48 calls of 5 tokens, each call with its own
    gate matrix (as in the pages' 48 prefill calls).  Reports the time per
    call in a CUDA graph of the 48 calls, the exact-tie count at the k
    boundary (margin_ulps == 0) over the 240 token-slots, the histogram of
    the boundary margins in bf16 ULPs, and the chained route hash of the 48
    calls' sorted id sets."""
    import numpy as np
    n_calls, n_tok, Et, kt = 48, 5, 512, 10
    xs, ws = [], []
    for c in range(n_calls):
        X, W = synth.tie_heavy_call(0, c)
        xs.append(torch.from_numpy(X.view(np.int16)).to(dev).view(torch.bfloat16))
        ws.append(torch.from_numpy(W.view(np.int16)).to(dev).view(torch.bfloat16))
    lg = torch.empty((n_calls, n_tok, Et), dtype=torch.bfloat16, device=dev)
    ids = torch.empty((n_calls, n_tok, kt), dtype=torch.int32, device=dev)
    w = torch.empty((n_calls, n_tok, kt), dtype=torch.float32, device=dev)
    mg = torch.empty((n_calls, n_tok), dtype=torch.float32, device=dev)
    mu = torch.empty((n_calls, n_tok), dtype=torch.int32, device=dev)
    h = torch.empty((1,), dtype=torch.int64, device=dev)

    def call(c):
        bi.bi_router_topk(xs[c], ws[c], bi.BI_BF16, bi.BI_BF16, n_tok, H, Et, kt, lg[c], ids[c], w[c], mg[c],
                          mu[c], stream=None)
    stream = torch.cuda.current_stream(dev)
    t = graph_time(torch, stream, call, n_calls)
    for c in range(n_calls):
        call(c)
        bi.bi_route_trace_hash(ids[c], n_tok, kt, [0, n_tok], None if c == 0 else h, h, stream=None)
    torch.cuda.synchronize()
    u = mu.flatten().cpu().numpy()
    edges = [0, 1, 2, 3, 4, 8, 16, 64, 256, 2 ** 31]
    hist = {(f"{lo}" if hi == lo + 1 else f"{lo}-{hi - 1}" if hi < 2 ** 31 else f">={lo}"):
            int(np.sum((u >= lo) & (u < hi))) for lo, hi in zip(edges[:-1], edges[1:])}
    byt = 2 * Et * H + 2 * n_tok * H + 2 * n_tok * Et + 8 * n_tok * kt + 8 * n_tok
    return {"config": "bf16 H=2048 E=512 top-10, 48 calls x 5 tokens, X, W in {-1,+1}*2^-8",
            "us_per_call": round(t * 1e6, 2), "tokens_per_s": n_tok / t,
            "frac_hbm": None, "GBps": round(byt / t / 1e9, 1),
            "slots": int(u.size), "exact_ties": int(np.sum(u == 0)), "ulp_histogram": hist,
            "chained_hash": f"{int(h.cpu().numpy().view(np.uint64)[0]):016x}"}


def margin_histogram_bf16(torch, logits, k):
    """The F32 router's boundary margins of the timed step (all 40 layers,
    4096 tokens each) with both endpoints -- the smallest selected and the
    largest rejected logit -- rounded to bf16 (nearest even) and their
    distance counted in bf16 ULPs under the sign-magnitude order.  Analysis
    of the step's outputs, outside any timed region."""
    import numpy as np
    top = torch.topk(logits.reshape(-1, logits.shape[-1]), k + 1, dim=1).values
    b = top[:, k - 1:k + 1].to(torch.bfloat16).view(torch.int16).to(torch.int32) & 0xFFFF
    o = torch.where(b >= 0x8000, -(b & 0x7FFF), b)
    d = (o[:, 0] - o[:, 1]).cpu().numpy()
    edges = [0, 1, 2, 3, 4, 8, 16, 64, 256, 2 ** 31]
    hist = {(f"{lo}" if hi == lo + 1 else f"{lo}-{hi - 1}" if hi < 2 ** 31 else f">={lo}"):
            int(np.sum((d >= lo) & (d < hi))) for lo, hi in zip(edges[:-1], edges[1:])}
    return {"tokens": int(d.size), "ulp_histogram": hist, "bf16_ties": int(np.sum(d == 0)),
            "note": "F32 router, 40 layers x 4096 tokens, both boundary logits rounded to bf16"}


def mixed_prefill_measure(bi, synth, torch, dev, reps=3):
    """The mixed prefill with a prefix cache: 16 requests of lengths U[5, 300]
    (seed 0), H = 2048, 40 layers, each running the router with the shared
    gate (E = 256, top-8), a 2048 x 2048 bf16 projection and the per-request
    route hashes, chained over the layers.  Run as a cache miss (every row,
    M = sum N) and as a suffix-only cache hit (M = sum of N mod 16, the last
    full block where that is 0; bi_prefix_split).  Reports the time per
    layer of each (a CUDA graph of the 40 layers) and whether each request's
    chained hash over its suffix rows is the same in both runs."""
    import numpy as np
    Hm, Em, km, L, blk = 2048, 256, 8, LAYERS, 16
    lens = [int(v) for v in synth.request_lengths(0)]
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(int).tolist()
    Mtot = offs[-1]
    cached, sub = bi.prefix_split(lens, blk)
    Mhit = sub[-1]
    rows_hit = np.concatenate([np.arange(offs[r] + cached[r], offs[r + 1]) for r in range(16)])
    idx_hit = torch.from_numpy(rows_hit).to(dev)
    Wg = [synth.device_normal((Em, Hm), 83000 + l, 0.02, torch.float32, dev) for l in range(L)]
    Wsg = [synth.device_normal((Hm,), 83100 + l, 0.02, torch.float32, dev) for l in range(L)]
    Bw = [synth.device_normal((Hm, Hm), 83200 + l, 1 / 64, torch.bfloat16, dev) for l in range(L)]
    Xm = [synth.device_normal((Mtot, Hm), 83300 + l, 1.0, torch.float32, dev) for l in range(L)]
    Am = [synth.device_normal((Mtot, Hm), 83400 + l, 1 / 64, torch.bfloat16, dev) for l in range(L)]
    Xh = [x.index_select(0, idx_hit).contiguous() for x in Xm]
    Ah = [a.index_select(0, idx_hit).contiguous() for a in Am]

    def make(Mr, Xs, As, ranges):
        o = {"lg": torch.empty((Mr, Em), dtype=torch.float32, device=dev),
             "ids": torch.empty((Mr, km), dtype=torch.int32, device=dev),
             "w": torch.empty((Mr, km), dtype=torch.float32, device=dev),
             "mg": torch.empty((Mr,), dtype=torch.float32, device=dev),
             "mu": torch.empty((Mr,), dtype=torch.int32, device=dev),
             "gd": torch.empty((Mr,), dtype=torch.float32, device=dev),
             "gs": torch.empty((Mr,), dtype=torch.float32, device=dev),
             "C": torch.empty((Mr, Hm), dtype=torch.bfloat16, device=dev),
             "h": torch.empty((len(ranges) - 1,), dtype=torch.int64, device=dev),
             "ws": bi.router_workspace(Mr, Em, dev)}

        def lay(l):
            bi.bi_router_gate_topk(Xs[l], Wg[l], Wsg[l], bi.BI_F32, bi.BI_F32, Mr, Hm, Em, km, o["lg"], o["ids"],
                                   o["w"], o["mg"], o["mu"], o["gd"], o["gs"], workspace=o["ws"], stream=None)
            bi.bi_route_trace_hash(o["ids"], Mr, km, ranges, None if l == 0 else o["h"], o["h"], stream=None)
            bi.bi_gemm_bf16(As[l], Bw[l], o["C"], Mr, Hm, Hm, Hm, Hm, Hm, stream=None)
        return o, lay

    miss, lay_miss = make(Mtot, Xm, Am, offs)
    hit, lay_hit = make(Mhit, Xh, Ah, sub)
    stream = torch.cuda.current_stream(dev)
    t_miss = graph_time(torch, stream, lay_miss, L, reps) * L
    t_hit = graph_time(torch, stream, lay_hit, L, reps) * L
    # invariance: per-request chained hash of the suffix rows (the rows a hit
    # recomputes), taken from the miss's ids and from the hit's
    hsub = torch.empty((16,), dtype=torch.int64, device=dev)
    for l in range(L):
        lay_miss(l)
        ids_suffix = miss["ids"].index_select(0, idx_hit).contiguous()
        bi.bi_route_trace_hash(ids_suffix, Mhit, km, sub, None if l == 0 else hsub, hsub, stream=None)
    for l in range(L):
        lay_hit(l)
    torch.cuda.synchronize()
    equal = bool(torch.equal(hsub, hit["h"]))
    return {"config": f"16 requests U[5,300] seed 0 (total {Mtot} rows; hit recomputes {Mhit}), 40 layers x "
                      "(router E=256 top-8 + shared gate + route hash + 2048x2048 bf16 projection)",
            "miss_us_per_layer": round(t_miss / L * 1e6, 2), "hit_us_per_layer": round(t_hit / L * 1e6, 2),
            "miss_tokens_per_s": Mtot / t_miss, "hit_tokens_per_s": Mhit / t_hit,
            "suffix_hashes_equal_miss_vs_hit": equal}


def digest(out) -> dict:
    """A compact restatement of the headline figures, printed last in the
    JSON line (readers that keep only the line's tail still get them)."""
    d = {"ms_per_step": round(out["ms_per_step"], 3), "tokens_per_s": round(out["value"]),
         "router_call_us_M4096": round(out["parts"]["router_call_us"], 1),
         "router_frac_fp32": round(out["roofline_router"]["frac"], 3),
         "gemm_call_us_M4096": round(out["parts"]["gemm_call_us"], 1),
         "gemm_frac_sustained": round(out["roofline_gemm"]["frac"], 3),
         "e2e_tokens_per_s": round(out["e2e"]["value"])}
    rs = out.get("router_sweep")
    if rs:
        d["router_us_by_M"] = {str(r["M"]): r["us"] for r in rs["calls"]
                               if r["M"] in (1, 4, 16, 19, 32, 48, 64, 65, 75, 128, 129, 256, 1024, 4096)}
        d["router_frac_hbm_M1_16_64"] = [r["frac_hbm"] for r in rs["calls"] if r["M"] in (1, 16, 64)]
        d["dependent_launch_floor_us"] = rs["floor_us"]
    gs = out.get("gemm_sweep")
    if gs:
        d["gemm_tflops_by_M"] = {str(r["M"]): r["tflops"] for r in gs["calls"]}
    th = out.get("tie_heavy_bf16_router")
    if th:
        d["tie_heavy"] = {"us_per_call": th["us_per_call"], "exact_ties": th["exact_ties"], "slots": th["slots"]}
    mp = out.get("mixed_prefill")
    if mp:
        d["mixed_prefill_us_per_layer"] = {"miss": mp["miss_us_per_layer"], "hit": mp["hit_us_per_layer"],
                                           "hashes_equal": mp["suffix_hashes_equal_miss_vs_hit"]}
    for key in ("moe_expert_gemm", "rmsnorm"):
        if key in out:
            d[key] = {"us": round(out[key]["us_per_call"], 1), "frac_hbm": round(out[key]["roofline"]["frac"], 3)}
    at = out.get("attention_prefill")
    if at:
        d["attention_prefill"] = {"us": round(at["us_per_call"], 1), "frac_bf16": round(at["roofline"]["frac"], 3),
                                  "long_context_frac_bf16": round(at["long_context"]["frac"], 3)}
    return d


def moe_measure(bi, synth, torch, dev, hbm_gbs, X, ids, wts, reps=10):
    """bi_moe_expert_gemm alone, on the router's own choice: the first
    layer's hidden states (rounded to bf16) through the experts it picked,
    top-8 of 256 experts of [N=1024, K=2048] bf16 (1 GiB of weights, two
    expert sets alternated so nothing stays in L2), per-slot outputs and
    the weighted combine.  Bound by HBM: every expert's weights are read."""
    En, Nn, Kn = E, 1024, H
    Ws = [synth.device_normal((En, Nn, Kn), 80000 + i, 1.0 / 64, torch.bfloat16, dev) for i in range(2)]
    xb = X.to(torch.bfloat16)
    Y = torch.empty((M, K_TOP, Nn), dtype=torch.bfloat16, device=dev)
    out = torch.empty((M, Nn), dtype=torch.bfloat16, device=dev)
    buf, n = bi.moe_workspace(M, K_TOP, En, Nn, Kn, dev)
    base = (buf.data_ptr() + 255) // 256 * 256

    def call(i):
        bi.bi_moe_expert_gemm(xb, ids, wts, Ws[i % 2], M, K_TOP, En, Nn, Kn, Y, out, base, n, stream=None)
    for i in range(4):
        call(i)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for i in range(reps):
        call(i)
    b.record()
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0
    t = a.elapsed_time(b) / 1e3 / reps
    flop = 2.0 * M * K_TOP * Nn * Kn
    byt = 2 * En * Nn * Kn + 2 * M * Kn + 8 * M * K_TOP + 2 * M * K_TOP * Nn + 2 * M * Nn
    del Ws
    return {"config": f"M={M} tokens, top-{K_TOP} of {En} experts, expert [N={Nn}, K={Kn}] bf16, "
                      "ids and weights from the step's router",
            "us_per_call": t * 1e6, "tflops": flop / t / 1e12,
            "launches_per_call": 4,
            "roofline": {"bound": "hbm", "achieved": byt / t / 1e9, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": byt / t / 1e9 / hbm_gbs, "algorithmic_bytes": byt,
                         "traffic": NCU_TRAFFIC["moe_call"]}}


def fma_probe(bi, torch, dev, packed: bool = False) -> float:
    """The FP32 FMA rate this GPU sustains, in TFLOP/s: the library's probe
    kernel (8 blocks of 256 threads per SM, 8 independent register-resident
    fused multiply-add chains per thread; packed: each chain two lanes of the
    two-wide f32 FMA instruction), timed with CUDA events on the launching
    stream; the best of five launches of about 20 ms each."""
    sink = torch.empty((8 * 1024,), dtype=torch.float32, device=dev)
    iters = 20000
    bi.selftest_fma_rate(iters, sink, packed=packed)
    best = 0.0
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        flop = bi.selftest_fma_rate(iters, sink, packed=packed)
        b.record()
        torch.cuda.synchronize()
        best = max(best, flop / (a.elapsed_time(b) / 1e3) / 1e12)
    return best


def rmsnorm_measure(bi, synth, torch, dev, hbm_gbs, Xs):
    """bi_rmsnorm alone: f32 rows of H=2048 -> bf16, M=4096, one call per
    layer's hidden states (40 different 32 MiB inputs, so each call reads
    from HBM), timed back to back.  Bound by HBM."""
    w = (1.0 + 0.1 * synth.device_normal((H,), 81000, 1.0, torch.float32, dev)).contiguous()
    y = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    r = torch.empty((M,), dtype=torch.float32, device=dev)
    for x in Xs[:4]:
        bi.bi_rmsnorm(x, w, bi.BI_F32, M, H, 1e-6, y, r)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for x in Xs:
        bi.bi_rmsnorm(x, w, bi.BI_F32, M, H, 1e-6, y, r)
    b.record()
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0
    t = a.elapsed_time(b) / 1e3 / len(Xs)
    byt = 4 * M * H + 2 * M * H + 4 * H + 4 * M
    return {"config": f"M={M}, H={H}, f32 in, bf16 out", "us_per_call": t * 1e6, "launches_per_call": 1,
            "roofline": {"bound": "hbm", "achieved": byt / t / 1e9, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": byt / t / 1e9 / hbm_gbs, "algorithmic_bytes": byt,
                         "traffic": NCU_TRAFFIC["rmsnorm_kernel"]}}


def attention_flops(q_lens, prefix, heads: int, D: int = 128) -> float:
    """Algorithmic FLOPs of causal attention: 4 D per (query, visible key,
    head) -- q.k and p.v, two flops per multiply-add; masked keys count
    nothing."""
    pairs = sum(int(n) * int(p) + int(n) * (int(n) + 1) // 2 for n, p in zip(q_lens, prefix))
    return 4.0 * D * heads * pairs


def attention_measure(bi, synth, torch, dev, bf16_peak, reps=50):
    """bi_attention_prefill alone on the prefill workload: 4096 queries in 8
    requests (five behind cached prefixes of 512 to 3072 tokens), 16 query
    heads over 2 key/value heads of dimension 128, bf16; eight input sets
    rotated, timed back to back with events on the launching stream.  Plus
    one long context (a 16384-token full prefill), where every SM stays busy
    to the end, and one request's prefix-cache hit (128 queries behind 32768
    cached tokens), which fills only 16 SMs.  Bound by the tensor cores (and
    the exponentials, which match them one to one per score)."""
    nh, nkv, D = synth.ATTN_HEADS, synth.ATTN_KV_HEADS, synth.ATTN_D
    qo, ko = synth.attention_offsets(synth.ATTN_Q_LENS, synth.ATTN_PREFIX)
    Tq, Tkv = int(qo[-1]), int(ko[-1])
    qo_l, ko_l = [int(v) for v in qo], [int(v) for v in ko]
    sets = [(synth.device_normal((Tq, nh, D), 83000 + i, 1.0, torch.bfloat16, dev),
             synth.device_normal((Tkv, nkv, D), 83100 + i, 1.0, torch.bfloat16, dev),
             synth.device_normal((Tkv, nkv, D), 83200 + i, 1.0, torch.bfloat16, dev)) for i in range(8)]
    o = torch.empty((Tq, nh, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((Tq, nh), dtype=torch.float32, device=dev)
    scale = 1.0 / math.sqrt(D)

    def timed(call, n):
        for i in range(4):
            call(i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for i in range(n):
            call(i)
        b.record()
        torch.cuda.synchronize()
        assert bi.bi_get_last_device_error() == 0
        return a.elapsed_time(b) / 1e3 / n

    t = timed(lambda i: bi.bi_attention_prefill(*sets[i % 8], len(qo_l) - 1, qo_l, ko_l, nh, nkv, D, scale, o,
                                                lse), reps)
    flop = attention_flops(synth.ATTN_Q_LENS, synth.ATTN_PREFIX, nh, D)
    del sets
    n = 16384
    ql = [synth.device_normal((n, nh, D), 83300, 1.0, torch.bfloat16, dev),
          synth.device_normal((n, nkv, D), 83301, 1.0, torch.bfloat16, dev),
          synth.device_normal((n, nkv, D), 83302, 1.0, torch.bfloat16, dev)]
    o2 = torch.empty((n, nh, D), dtype=torch.bfloat16, device=dev)
    ws2 = bi.attention_workspace([0, n], [0, n], nh, dev)
    t2 = timed(lambda i: bi.bi_attention_prefill(*ql, 1, [0, n], [0, n], nh, nkv, D, scale, o2, None, workspace=ws2),
               10)
    flop2 = attention_flops([n], [0], nh, D)
    del ql, o2, ws2
    # a prefix-cache hit of one request: 128 new queries behind 32768 cached
    # tokens (one query tile: 16 CTAs, one head each)
    pre, nq = 32768, 128
    hq = [synth.device_normal((nq, nh, D), 83400, 1.0, torch.bfloat16, dev),
          synth.device_normal((pre + nq, nkv, D), 83401, 1.0, torch.bfloat16, dev),
          synth.device_normal((pre + nq, nkv, D), 83402, 1.0, torch.bfloat16, dev)]
    o3 = torch.empty((nq, nh, D), dtype=torch.bfloat16, device=dev)
    ws3 = bi.attention_workspace([0, nq], [0, pre + nq], nh, dev)
    t3 = timed(lambda i: bi.bi_attention_prefill(*hq, 1, [0, nq], [0, pre + nq], nh, nkv, D, scale, o3, None,
                                                 workspace=ws3), 10)
    flop3 = attention_flops([nq], [pre], nh, D)
    tiles = sum((int(q) + 127) // 128 for q in synth.ATTN_Q_LENS)
    return {"config": f"{Tq} queries in {len(qo_l) - 1} requests (q_len {list(synth.ATTN_Q_LENS)}, cached prefix "
                      f"{list(synth.ATTN_PREFIX)}), {nh} query heads over {nkv} key/value heads, D={D}, bf16, "
                      "causal, lse written",
            "us_per_call": t * 1e6, "tflops": flop / t / 1e12, "algorithmic_flop": flop,
            "launches_per_call": 1, "ctas": tiles * nh // 2,
            "roofline": {"bound": "tensor", "achieved": flop / t / 1e12, "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": flop / t / 1e12 / bf16_peak, "peak_kind": "bf16 burst, of measured",
                         "traffic": NCU_TRAFFIC["attn_prefill_kernel"]},
            "long_context": {"config": f"one request, {n}-token full prefill, {nh}/{nkv} heads, D={D}",
                             "us_per_call": t2 * 1e6, "tflops": flop2 / t2 / 1e12,
                             "frac": flop2 / t2 / 1e12 / bf16_peak},
            "cache_hit_one_request": {"config": f"one request, {nq} queries behind {pre} cached tokens, "
                                                f"{nh}/{nkv} heads, D={D}: one query tile, {nh} CTAs",
                                      "us_per_call": t3 * 1e6, "tflops": flop3 / t3 / 1e12,
                                      "frac": flop3 / t3 / 1e12 / bf16_peak}}


def m_variant_context(bi, synth, torch, dev):
    """The M-variant arm the pages contrast with (context, not the product):
    stock torch.matmul in F32 with TF32 off plus torch.topk for the router,
    and torch.matmul in bf16 for the projection, on the same shapes.  For
    each op, the first M in the sweep at which row 0 of the batch stops being
    byte-identical to its M = 1 result, and the op's throughput at M = 4096."""
    torch.backends.cuda.matmul.allow_tf32 = False
    W = synth.device_normal((E, H), 79000, 0.02, torch.float32, dev)
    X = synth.device_normal((M, H), 79001, 1.0, torch.float32, dev)
    B = synth.device_normal((G_N, G_K), 79002, 1.0 / 64, torch.bfloat16, dev)
    A = synth.device_normal((8192, G_K), 79003, 1.0 / 64, torch.bfloat16, dev)
    r_sweep = [1, 2, 4, 8, 16, 19, 32] + list(range(35, 65)) + [65, 75, 96, 128, 256, 512, 1024, 2048, 4096]
    g_sweep = [1, 19, 64, 65, 75, 128, 1024, 4096, 8192]
    solo_l = torch.matmul(X[:1], W.t())
    solo_i = torch.topk(solo_l, K_TOP).indices
    first_l = first_i = first_g = None
    for Mi in r_sweep:
        lg = torch.matmul(X[:Mi], W.t())
        ids = torch.topk(lg, K_TOP).indices
        if first_l is None and not torch.equal(lg[:1].view(torch.int32), solo_l.view(torch.int32)):
            first_l = Mi
        if first_i is None and not torch.equal(ids[:1], solo_i):
            first_i = Mi
    solo_g = torch.matmul(A[:1], B.t())
    for Mi in g_sweep:
        c = torch.matmul(A[:Mi], B.t())
        if first_g is None and not torch.equal(c[:1].view(torch.int16), solo_g.view(torch.int16)):
            first_g = Mi

    def timed(fn, n=20):
        for _ in range(3):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3 / n

    t_r = timed(lambda: torch.topk(torch.matmul(X, W.t()), K_TOP))
    t_g = timed(lambda: torch.matmul(A[:M], B.t()))
    # this library's kernels in the same loop, on the same tensors
    lg = torch.empty((M, E), dtype=torch.float32, device=dev)
    ids = torch.empty((M, K_TOP), dtype=torch.int32, device=dev)
    wt = torch.empty((M, K_TOP), dtype=torch.float32, device=dev)
    Cb = torch.empty((M, G_N), dtype=torch.bfloat16, device=dev)
    wsp = bi.router_workspace(M, E, dev)
    t_r_bi = timed(lambda: bi.bi_router_topk(X, W, bi.BI_F32, bi.BI_F32, M, H, E, K_TOP, lg, ids, wt, None, None,
                                             workspace=wsp, stream=None))
    t_g_bi = timed(lambda: bi.bi_gemm_bf16(A, B, Cb, M, G_N, G_K, G_K, G_K, G_N, stream=None))
    return {"router_f32_matmul_topk": {"first_M_row0_logits_differ": first_l, "first_M_row0_ids_differ": first_i,
                                       "swept_M": r_sweep, "tokens_per_s_at_4096": M / t_r,
                                       "bi_router_topk_tokens_per_s_same_loop": M / t_r_bi},
            "gemm_bf16_matmul": {"first_M_row0_differs": first_g, "swept_M": g_sweep,
                                 "tflops_at_4096": 2.0 * M * G_N * G_K / t_g / 1e12,
                                 "bi_gemm_bf16_tflops_same_loop": 2.0 * M * G_N * G_K / t_g_bi / 1e12},
            "note": "torch.matmul (cuBLAS) with TF32 off and torch.topk on the same shapes, timed back to "
                    "back on the same (L2-warm) tensors, beside this library's calls in the same loop; "
                    "null = row 0 identical at every swept M"}


_CPU_STATE = {}


def _cpu_layer_sample(seed_stream: int, budget_s: float):
    """One worker's share of the CPU baseline: the oracle, as it stands,
    over fresh tokens through one layer (router + shared gate + route hash +
    one projection row) until budget_s of timed oracle work.  Input draws are
    outside the timed region.  Returns (tokens, seconds)."""
    from oracle import oracle as orc
    from serving_numerics_gb300 import synth
    st = _CPU_STATE
    if not st:
        orc.build()
        st["W"] = synth.router_weights(7, 0, E, H)
        st["wsg"] = synth.shared_gate_weights(7, 0, H)
        st["B"] = synth.gemm_b(7, G_N, G_K)
        st["next"] = 0
    n, spent = 0, 0.0
    while spent < budget_s:
        tok = seed_stream * 1_000_000 + st["next"]
        st["next"] += 1
        X = synth.tokens(7, 0, tok, 1, H)
        Ar = synth.gemm_a(7, 1, G_K, layer=tok)
        t = time.perf_counter()
        r = orc.router_full(X, st["W"], K_TOP, "f32")
        orc.shared_gate(X, st["wsg"])
        orc.route_hash(r["ids"])
        orc.gemm_bf16(Ar, st["B"])
        spent += time.perf_counter() - t
        n += 1
    return n, spent


class CpuBaseline:
    """The oracle timed on the host cores: on one thread, and as one
    single-threaded worker process per core of this process's affinity set
    (rows are independent, so the workers split the tokens; the oracle itself
    is unchanged).  Workers are started with spawn (this process already
    holds a CUDA context) and kept for every sample."""

    def __init__(self):
        import multiprocessing as mp
        self.affinity = sorted(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else []
        self.nproc = os.cpu_count()
        self.workers = max(1, len(self.affinity) or (self.nproc or 1))
        self.pool = mp.get_context("spawn").Pool(self.workers)
        # load the oracle and the weights in every worker before any timing
        self.pool.map(_cpu_pool_task, [(i, 0.0) for i in range(self.workers)])

    def close(self):
        self.pool.close()
        self.pool.join()

    def sample(self, single_s: float, parallel_s: float) -> dict:
        n1, t1 = _cpu_layer_sample(1_000, single_s)
        res = self.pool.map(_cpu_pool_task, [(i, parallel_s) for i in range(self.workers)])
        rate_all = sum(n / t for n, t in res if t > 0)       # tokens-through-one-layer per second
        n_all = sum(n for n, _ in res)
        return {"value": rate_all / LAYERS, "unit": "tokens/s", "cores": self.workers, "kind": "oracle",
                "single_thread_value": n1 / t1 / LAYERS,
                "affinity_cpus": len(self.affinity), "nproc": self.nproc,
                "sample": f"1 thread: {n1} tokens through 1 of the 40 layers (router+gate+hash+GEMM row) "
                          f"in {t1:.1f} s; {self.workers} worker processes (one per core of the affinity "
                          f"set, the single-threaded oracle unchanged): {n_all} tokens in about "
                          f"{parallel_s:.1f} s each; both scaled to 40 layers"}


def _cpu_pool_task(arg):
    i, budget = arg
    return _cpu_layer_sample(2_000 + i, budget)


def oracle_sweep() -> dict:
    """The oracle, single-threaded, per call over M (about 15 s): the router
    (F32, H=2048, E=256, top-8) in full at every M listed; the K=N=4096
    projection in full at every M up to 128, and as a fixed 64-row sample
    standing for any larger M (the oracle's cost is linear in the rows)."""
    from oracle import oracle as orc
    from serving_numerics_gb300 import synth
    orc.build()
    W = synth.router_weights(7, 0, E, H)
    router = {}
    for m in (1, 19, 64, 65, 75, 128, 256, 1024, 4096):
        X = synth.tokens(7, 0, 5000 + m, m, H)
        t = time.perf_counter()
        orc.router_full(X, W, K_TOP, "f32")
        router[str(m)] = m / (time.perf_counter() - t)
    B = synth.gemm_b(7, G_N, G_K)
    gemm = {}
    for m, label in ((1, "1"), (19, "19"), (64, "64"), (65, "65"), (75, "75"), (128, "128"),
                     (64, "per-row rate from a 64-row sample (any larger M)")):
        A = synth.gemm_a(7, m, G_K, layer=6000 + m)
        t = time.perf_counter()
        orc.gemm_bf16(A, B)
        gemm[label] = 2.0 * m * G_N * G_K / (time.perf_counter() - t) / 1e9
    return {"router_tokens_per_s_by_M": router, "gemm_gflops_by_M": gemm, "threads": 1}


def cpu_baseline(budget_s: float = 15.0):
    """About budget_s of host time: two thirds on one thread, the rest on all
    cores at once; then the oracle's per-call rates over M."""
    cb = CpuBaseline()
    try:
        out = cb.sample(budget_s * 2 / 3, budget_s / 3)
    finally:
        cb.close()
    out["oracle_sweep"] = oracle_sweep()
    return out


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on this host's cores
    (one single-threaded worker per core); rank 0 alone under torchrun (the
    other ranks exit without work).  Each step is a bounded sample of about
    --cpu-seconds of host time."""
    ws, rank, _ = dist_setup()
    if rank != 0:
        return
    budget = args.cpu_seconds
    cb = CpuBaseline()
    try:
        for _ in range(args.warmup):
            cb.sample(0.2, 0.2)
        vals = []
        t = time.perf_counter()
        for _ in range(args.steps):
            vals.append(cb.sample(budget * 2 / 3, budget / 3))
        total = time.perf_counter() - t
    finally:
        cb.close()
    v = statistics.mean(x["value"] for x in vals)
    last = vals[-1]
    out = {"metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "impl": "reference",
           "data": "synthetic (seeded normal draws)",
           "config": {"workload": WORKLOAD, "tokens_per_step_per_gpu": M, "layers": LAYERS},
           "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": last["cores"], "kind": "oracle",
                            "single_thread_value": statistics.mean(x["single_thread_value"] for x in vals),
                            "affinity_cpus": last["affinity_cpus"], "nproc": last["nproc"],
                            "sample": last["sample"]},
           "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_case(args):
    """One operation, called exactly three times on fresh inputs and then
    checked for device errors -- a small, fixed launch sequence for profilers
    (the third call is the one to capture):
      router:M    bi_router_topk, F32, H=2048, E=256, top-8, all outputs
      gemm:M      bi_gemm_bf16, K = N = 4096
      rmsnorm:M   bi_rmsnorm, f32 rows of H=2048 -> bf16
      attn:N      bi_attention_prefill, one N-token full prefill (default 4096),
                  16 query heads over 2 key/value heads, D=128
      attnmix     bi_attention_prefill on the benchmark's mixed prefill batch"""
    import torch

    from serving_numerics_gb300 import binding as bi
    from serving_numerics_gb300 import synth
    bi.load()
    dev = torch.device("cuda", 0)
    kind, _, m = args.case.partition(":")
    Mi = int(m or M)
    if kind == "router":
        Ws = [synth.device_normal((E, H), 90000 + i, 0.02, torch.float32, dev) for i in range(3)]
        xs = [synth.device_normal((Mi, H), 90100 + i, 1.0, torch.float32, dev) for i in range(3)]
        out = bi.router_topk(xs[0], Ws[0], K_TOP)
        ws = bi.router_workspace(Mi, E, dev)
        calls = [lambda i=i: bi.router_topk(xs[i], Ws[i], K_TOP, out=out, workspace=ws) for i in range(3)]
    elif kind == "gemm":
        Bs = [synth.device_normal((G_N, G_K), 90200 + i, 1 / 64, torch.bfloat16, dev) for i in range(3)]
        As = [synth.device_normal((Mi, G_K), 90300 + i, 1 / 64, torch.bfloat16, dev) for i in range(3)]
        Cm = torch.empty((Mi, G_N), dtype=torch.bfloat16, device=dev)
        calls = [lambda i=i: bi.gemm_bf16(As[i], Bs[i], out=Cm) for i in range(3)]
    elif kind == "rmsnorm":
        w = (1.0 + 0.1 * synth.device_normal((H,), 90400, 1.0, torch.float32, dev)).contiguous()
        xs = [synth.device_normal((Mi, H), 90500 + i, 1.0, torch.float32, dev) for i in range(3)]
        calls = [lambda i=i: bi.rmsnorm(xs[i], w, 1e-6) for i in range(3)]
    elif kind == "attn":
        nh, nkv, D = synth.ATTN_HEADS, synth.ATTN_KV_HEADS, synth.ATTN_D
        n = Mi if m else 4096
        xs = [[synth.device_normal((n, h_, D), 90600 + 3 * i + j, 1.0, torch.bfloat16, dev)
               for j, h_ in enumerate((nh, nkv, nkv))] for i in range(3)]
        o = torch.empty((n, nh, D), dtype=torch.bfloat16, device=dev)
        calls = [lambda i=i: bi.bi_attention_prefill(*xs[i], 1, [0, n], [0, n], nh, nkv, D, 1 / math.sqrt(D), o,
                                                     None) for i in range(3)]
    elif kind == "attnmix":
        nh, nkv, D = synth.ATTN_HEADS, synth.ATTN_KV_HEADS, synth.ATTN_D
        qo, ko = synth.attention_offsets(synth.ATTN_Q_LENS, synth.ATTN_PREFIX)
        qo_l, ko_l = [int(v) for v in qo], [int(v) for v in ko]
        xs = [[synth.device_normal((qo_l[-1], nh, D), 90700 + 3 * i, 1.0, torch.bfloat16, dev),
               synth.device_normal((ko_l[-1], nkv, D), 90701 + 3 * i, 1.0, torch.bfloat16, dev),
               synth.device_normal((ko_l[-1], nkv, D), 90702 + 3 * i, 1.0, torch.bfloat16, dev)] for i in range(3)]
        o = torch.empty((qo_l[-1], nh, D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((qo_l[-1], nh), dtype=torch.float32, device=dev)
        calls = [lambda i=i: bi.bi_attention_prefill(*xs[i], len(qo_l) - 1, qo_l, ko_l, nh, nkv, D,
                                                     1 / math.sqrt(D), o, lse) for i in range(3)]
    else:
        raise SystemExit(f"unknown case {args.case}")
    torch.cuda.synchronize()
    for c in calls:
        c()
    torch.cuda.synchronize()
    assert bi.bi_get_last_device_error() == 0
    print(json.dumps({"case": args.case, "calls": 3, "ok": True}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the router-only M sweep")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--moe-only", action="store_true",
                    help="measure only the grouped expert GEMM (a small case for profiling)")
    ap.add_argument("--moe-reps", type=int, default=10)
    ap.add_argument("--layers", type=int, default=LAYERS,
                    help="fewer layers for a small profiling case (the benchmark uses 40)")
    ap.add_argument("--case", default=None,
                    help="router:M, gemm:M, rmsnorm:M, attn:N or attnmix: three calls of one operation, for profiling")
    args = ap.parse_args()
    globals()["LAYERS"] = args.layers
    if args.case:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

"""Benchmark of MXFP4 MoE layer steps on GB300.

A step is one pass of the whole hot path over one batch: router logits,
top-k, segments, FP8 activation quantisation, gate/up + SwiGLU + h
quantisation, down, combine -- for every layer of the workload.  The default
workload is the largest one a single GPU holds: a stack of 8
DeepSeek-V4.1-shaped MoE layers (hidden 5120, intermediate 2304, 384 routed
experts top-6 + 1 shared each, ~58 GB resident) run back to back on 64
concurrent decode tokens with Zipf(1.1)-skewed routing and a bf16 residual
add between layers (each layer's input RMS-normalised).  The single-layer
decode, verification and prefill workloads are selectable with --workload.

Prints ONE JSON line (rank 0).  `value` is tokens/s through the workload
(all its layers) with inputs resident in HBM; each step gets fresh tokens and
the L2 is flushed between steps (outside the timed events).  `e2e` is the
same metric through the library's host-buffer entry point
(moe_stack_forward_host for a stack, moe_forward_host for one layer) with
pinned host buffers, the copies inside the timed region.
`--impl reference` times the fp64 CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from synth.workloads import WORKLOADS  # noqa: E402

DEFAULT = "v41_stack8_decode_t64_zipf"
METRIC = "MoE-layer tokens/s; decode HBM GB/s vs peak; prefill FP4 TFLOPS vs peak"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=DEFAULT, choices=sorted(WORKLOADS))
    p.add_argument("--path", type=int, default=0, help="0 auto, 1 SIMT, 2 tensor cores")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--graph", type=int, default=1, help="1: launch each step as a captured CUDA graph, 0: stream launches")
    p.add_argument("--mma-rates", action="store_true",
                   help="build and run the tensor-core MMA issue-rate microbenchmark, then exit")
    p.add_argument("--shared", default="mxfp4", choices=["mxfp4", "fp8"],
                   help="shared experts' weights: mxfp4 (as the routed bank) or fp8 (E4M3, 32 x 32 blocks)")
    p.add_argument("--act", default="fp8", choices=["fp8", "fp4"],
                   help="activation format: fp8 (the layer) or fp4 (the FP4-activation variant)")
    return p.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "src": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "src": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None
        return self

    def __exit__(self, *a):
        if self.p:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except Exception:
                self.p.kill()

    def summary(self):
        self.f.flush()
        rows = []
        try:
            for line in open(self.f.name):
                parts = [s.strip() for s in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        except Exception:
            pass
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "reasons": reasons, "samples": len(rows)}


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(v: float, pg, device) -> float:
    """The slowest rank's figure (every rank gets it); v itself on one process."""
    if pg is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return t.item()


def job_tokens_per_s(world: int, tokens: int, steps: int, total_ms: float) -> float:
    """Whole-job throughput of N replicas: every rank's tokens over the slowest rank's time."""
    return world * tokens * steps / (total_ms / 1e3)


def layer_bytes(wl, n_experts_touched: int, T: int, shared_fp8: bool = False) -> dict:
    """Algorithmic HBM bytes of one layer step and of its two FFN kernels."""
    H, I, E, k, ns = wl.hidden, wl.inter, wl.n_experts, wl.top_k, wl.n_shared
    P = T * k + ns * T
    per_mat = H * I // 2 + H * I // 32
    # a shared matrix: MXFP4 like the routed ones, or FP8 with one scale per 32 x 32 block
    sh_mat = H * I + (H // 32) * (I // 32) if shared_fp8 else per_mat
    n = n_experts_touched + ns
    up = n_experts_touched * 2 * per_mat + ns * 2 * sh_mat + T * (H + H // 32) + P * (I + I // 32)
    down = n_experts_touched * per_mat + ns * sh_mat + P * (I + I // 32) + P * H * 4
    layer = n_experts_touched * wl.expert_bytes + ns * 3 * sh_mat + E * H * 4 + E * 4 + 2 * T * H * 2
    return {"layer": layer, "ffn_up_simt": up, "ffn_down_simt": down,
            "ffn_up_mma": up, "ffn_down_mma": down}


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) as a multiple of the
# launch's algorithmic bytes, from the ncu capture summarised in
# profiles/ffn_mma_t64_e128_full.md (one layer of the 8-layer stack's shape: 64 tokens, Zipf
# routing, a 128-expert bank, 64-token tiles).  The stack's launches stream their experts the
# same way (one 64-token tile per active expert), so the traffic scales with the experts touched:
# traffic = ratio x algorithmic bytes.  Valid only for the kernel source the capture was taken on.
_TRAFFIC_SRC = ("mxfp4_expert_ffn_gb300/csrc/ffn_mma_kernel.cuh", "mxfp4_expert_ffn_gb300/csrc/ffn_mma.cu")
_TRAFFIC_SHA256 = "43238bab094a43e7bc8bd8f4ff4fe51a4d4eca07537d156305b4d70d0ff7b393"
# (dram__bytes_read.sum + dram__bytes_write.sum) / algorithmic bytes of one gate/up launch:
# 64 tokens over a 128-expert bank (stack-shaped layer, Zipf routing) and one decode token
# over a 24-expert bank; each streams the same bytes per selected expert as the full layer.
_T64_RATIO = (702.981632 + 3.166720) / 715.826688
_T1_RATIO = (88.943104 + 2.243584) / 87.758232
_TRAFFIC_RATIO = {("v41_stack8_decode_t64_zipf", "ffn_up_mma"): _T64_RATIO,
                  ("ncu_v41_e128_decode_t64_zipf", "ffn_up_mma"): _T64_RATIO,
                  ("v41_layer_decode_t1", "ffn_up_mma"): _T1_RATIO,
                  ("ncu_v41_e24_decode_t1", "ffn_up_mma"): _T1_RATIO}


def measured_traffic(workload: str, kernel: str, algorithmic_bytes: float):
    import hashlib
    try:
        h = hashlib.sha256()
        for src in _TRAFFIC_SRC:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != _TRAFFIC_SHA256:
            return None  # the kernel changed since the counters were taken
    except OSError:
        return None
    r = _TRAFFIC_RATIO.get((workload, kernel))
    return None if r is None else r * algorithmic_bytes


def layer_flops(wl, T: int) -> int:
    return (T * wl.top_k + wl.n_shared * T) * 3 * 2 * wl.hidden * wl.inter


# Block-scaled tcgen05.mma throughput of one SM at M = 128, N >= 128, in FLOP per
# SM clock cycle, as measured by the issue-rate microbenchmark (mma_rate.cu,
# `bench.py --mma-rates`; profiles/mma_issue_rates.md): 128 x 256 x K x 2 FLOP in
# 128.2 cycles, K = 32 for kind::mxf8f6f4 (FP4 weights x FP8 activations) and
# K = 64 for kind::mxf4 (FP4 x FP4).
MMA_FLOP_PER_CYCLE_SM = {"mxf8f6f4": 16362.0, "mxf4": 32724.0}


def tensor_peak_tflops(kind: str, n_sms: int, sm_mhz: float) -> float:
    """Dense peak of one block-scaled MMA kind at the given SM clock."""
    return MMA_FLOP_PER_CYCLE_SM[kind] * n_sms * sm_mhz * 1e6 / 1e12


def oracle_tokens_per_s(wl, n_tokens: int, threads: int, stream: int = 50, experts: dict | None = None):
    """Times the fp64 oracle (input norm, routing and layer, for every layer of
    the workload) on n_tokens seeded tokens.  The expert bytes the sample
    touches are generated before the clock starts (input generation, on
    parallel host threads); `experts` keeps them across calls."""
    import oracle
    import synth
    experts = {} if experts is None else experts
    x = synth.activations(wl, tokens=n_tokens, stream=stream)
    t_total = 0.0
    cur = x
    for layer in range(wl.layers):
        Wr, b = synth.router_weights(wl, layer), synth.router_bias(wl, layer)
        t0 = time.perf_counter()
        xin = oracle.rmsnorm(cur, 1e-6) if wl.rmsnorm else cur
        lg = oracle.router_logits(xin, Wr, b, threads=threads)
        idx, w = oracle.topk(lg, wl.top_k)
        t_total += time.perf_counter() - t0
        ids = [int(e) for e in np.unique(idx)] + [wl.n_experts + s for s in range(wl.n_shared)]
        missing = [e for e in ids if (layer, e) not in experts]
        experts.update({(layer, e): v for e, v in synth.host_experts(wl, layer, missing).items()})
        ex = {e: experts[(layer, e)] for e in ids[:len(ids) - wl.n_shared]}
        sh = [experts[(layer, wl.n_experts + s)] for s in range(wl.n_shared)]
        t0 = time.perf_counter()
        y, _ = oracle.moe_layer(xin, idx, w, ex, sh, wl.n_experts, wl.inter,
                                residual=cur if wl.rmsnorm else None, threads=threads)
        t_total += time.perf_counter() - t0
        cur = y
    return n_tokens / t_total, t_total


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    wl = WORKLOADS[args.workload]
    cores = os.cpu_count() or 1
    threads = min(cores, oracle.max_threads())
    # one token per thread (the oracle runs tokens in parallel), the same
    # seeded block every step so that its experts are generated once
    n_tok = max(1, threads)
    experts = {}
    for i in range(args.warmup):
        oracle_tokens_per_s(wl, 1, 1, stream=300, experts=experts)
    total_t, total_n = 0.0, 0
    for i in range(args.steps):
        _, t = oracle_tokens_per_s(wl, n_tok, threads, stream=300, experts=experts)
        total_t += t
        total_n += n_tok
    v = total_n / total_t
    sample = (f"{n_tok} seeded tokens per step (one per thread) of workload {wl.name}, through all "
              f"{wl.layers} layer(s): input norm, routing and layer, fp64 oracle")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000 * total_t / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "tokens": wl.tokens, "layers": wl.layers},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": min(threads, n_tok),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch

    import mxfp4_expert_ffn_gb300 as m
    import synth
    from synth import gpu as sg

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(dev))
        pg = dist
    wl = WORKLOADS[args.workload]
    T, H, E, k = wl.tokens, wl.hidden, wl.n_experts, wl.top_k
    nl = wl.layers
    W = [sg.device_layer(wl, l, dev) for l in range(nl)]
    if args.shared == "fp8":  # the shared experts in the FP8 (32 x 32 block) format
        for l in range(nl):
            exs = [synth.host_expert_fp8(wl, l, E + s) for s in range(wl.n_shared)]
            for mname in ("gate", "up", "down"):
                for kind in ("codes", "scales"):
                    a = np.ascontiguousarray(np.stack([e[f"{mname}_{kind}"] for e in exs]))
                    W[l][f"s_{mname}_{kind}"] = torch.from_numpy(a).to(dev)
    Ls = [m.Layer(H, wl.inter, E, k, wl.n_shared, T, W[l]) for l in range(nl)]
    for L in Ls:
        L.set_option(m.MOE_OPT_PATH, args.path)
        if args.shared == "fp8":
            L.set_shared_format(m.MOE_SHARED_FP8_B32)
        if args.act == "fp4":
            L.set_act_format(m.MOE_ACT_FP4)
    n_in = args.steps + args.warmup
    # distinct token blocks: one per step, up to 2^29 values in all (the
    # largest prefill sweeps cycle through fewer; every block is far above L2)
    n_x = max(1, min(n_in, (1 << 29) // (T * H)))
    xs = sg.bf16_tensor(synth.activations(wl, tokens=n_x * T, stream=100 + rank), dev).view(n_x, T, H)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    wt = torch.empty((T, k), dtype=torch.float32, device=dev)
    bufs = [torch.empty((T, H), dtype=torch.int16, device=dev) for _ in range(3)]
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)  # > 126 MB L2
    sink = torch.empty((), dtype=torch.uint8, device=dev)

    def flush_l2(i):
        # write a buffer 4x the L2, then read it back: the read evicts the dirty
        # lines, so their write-back happens here and not inside the next step
        flush.fill_(i & 0xFF)
        torch.amax(flush, dim=0, out=sink)
    st = torch.cuda.current_stream()

    def step(i, y_out=None):
        # one call per layer: moe_step = route + forward (for up to 64 tokens the
        # router, top-k, x codes and segments are a single launch)
        x = xs[i % n_x]
        if nl == 1:
            Ls[0].step(x, T, bufs[0] if y_out is None else y_out)
            return
        cur, xn = x, bufs[0]
        for layer in range(nl):
            nxt = bufs[1] if cur is not bufs[1] else bufs[2]
            m.moe_rmsnorm(cur, T, H, 1e-6, xn)          # normalised input of the layer
            Ls[layer].step(xn, T, nxt, residual=cur)   # x_{l+1} = x_l + layer(norm(x_l))
            cur = nxt

    run = step
    if args.graph:
        for i in range(args.warmup):
            step(i)  # first launches (attributes, lazy module load) outside capture
        torch.cuda.synchronize()
        graphs = []
        for i in range(n_in):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(i)
            graphs.append(g)
        torch.cuda.synchronize()
        run = lambda i: graphs[i].replay()  # noqa: E731

    def timed_loop(run):
        times = []
        for i in range(args.warmup):
            run(i)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        for i in range(args.warmup, n_in):
            flush_l2(i)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            run(i)
            e1.record(st)
            times.append((e0, e1))
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        return [a.elapsed_time(b) for a, b in times]

    with ClockSampler(local) as clk:
        ms = timed_loop(run)
    clocks = clk.summary()
    total_ms = max_over_ranks(sum(ms), pg, dev)
    ms_step = total_ms / args.steps
    value = job_tokens_per_s(world, T, args.steps, total_ms)

    # union of experts per step (for byte accounting), outside the timed region
    unions = []
    for i in range(args.warmup, n_in):
        if nl == 1:
            Ls[0].route(xs[i % n_x], T, idx, wt)
            torch.cuda.synchronize()
            unions.append(len(np.unique(idx.cpu().numpy())))
            continue
        # a stack: every layer's routing of its own input (the same steps again)
        cur, xn = xs[i % n_x], bufs[0]
        for layer in range(nl):
            nxt = bufs[1] if cur is not bufs[1] else bufs[2]
            m.moe_rmsnorm(cur, T, H, 1e-6, xn)
            Ls[layer].step(xn, T, nxt, residual=cur, idx=idx, w=wt)
            torch.cuda.synchronize()
            unions.append(len(np.unique(idx.cpu().numpy())))
            cur = nxt
    mean_union = float(np.mean(unions)) if unions else None

    # per-kernel times: the same loop again with the library's event timing on
    for L in Ls:
        L.set_option(m.MOE_OPT_TIMING, 1)
        L.kernel_times()
    # this library's launches in one step (every layer call records each of its launches)
    step(0)
    per_step_launches = sum(n for L in Ls for _, _, n in L.kernel_times())
    per_step_launches += nl if nl > 1 else 0  # one moe_rmsnorm launch per layer of a stack
    timed_loop(step)  # stream launches: the library's events bracket each kernel
    ktimes = {}
    for L in Ls:
        for name, kms, n in L.kernel_times():
            a = ktimes.setdefault(name, [0.0, 0])
            a[0] += kms
            a[1] += n
        L.set_option(m.MOE_OPT_TIMING, 0)
    dom = max(ktimes, key=lambda n: ktimes[n][0])
    dom_ms = ktimes[dom][0] / ktimes[dom][1]

    pk = peaks()
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_mhz = clocks.get("sm_mhz") or clocks.get("sm_max_mhz") or 2070.0
    mma_kind = "mxf4" if args.act == "fp4" else "mxf8f6f4"
    mma_peak = tensor_peak_tflops(mma_kind, n_sms, sm_mhz)
    roofline = None
    if mean_union is not None:
        b = layer_bytes(wl, mean_union, T, shared_fp8=args.shared == "fp8")
        if dom in b:
            # the dominant kernel against the bound that takes longer at peak: HBM
            # streaming of its algorithmic bytes, or its useful block-scaled MMA
            # FLOPs (gate/up: 2 of the 3 matrices) at the measured MMA rate
            kflops = layer_flops(wl, T) * (2 / 3 if "up" in dom else 1 / 3)
            t_hbm = b[dom] / (pk["hbm_gbs"] * 1e9)
            t_tensor = kflops / (mma_peak * 1e12)
            if "mma" in dom and t_tensor > t_hbm:
                ach = kflops / (dom_ms / 1e3) / 1e12
                roofline = {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": mma_peak,
                            "unit": "TFLOP/s", "frac": ach / mma_peak, "traffic": None,
                            "algorithmic_flops_per_launch": kflops, "avg_launch_ms": dom_ms,
                            "peak_src": f"measured {mma_kind} issue rate x {n_sms} SMs x median SM clock "
                                        f"{sm_mhz:.0f} MHz"}
            else:
                ach = b[dom] / (dom_ms / 1e3) / 1e9
                roofline = {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": pk["hbm_gbs"],
                            "unit": "GB/s", "frac": ach / pk["hbm_gbs"],
                            "traffic": measured_traffic(wl.name, dom, b[dom]),
                            "algorithmic_bytes_per_launch": b[dom], "avg_launch_ms": dom_ms,
                            "peak_src": pk["src"]}
        layer_gbs = nl * b["layer"] / (ms_step / 1e3) / 1e9  # all layers' bytes over the step
        if roofline is not None:
            # the whole step (every kernel of every layer) against HBM
            roofline["step"] = {"achieved_gbs": layer_gbs, "frac": layer_gbs / pk["hbm_gbs"],
                                "algorithmic_bytes_per_step": nl * b["layer"]}
    else:
        layer_gbs = None

    # end to end through the host-buffer entry point (copies inside the timed
    # region): one layer, or the whole stack in one call
    xh = torch.empty((n_x, T, H), dtype=torch.int16).pin_memory()
    xh.copy_(xs.cpu())
    yh = torch.empty((T, H), dtype=torch.int16).pin_memory()

    def host_step(i):
        if nl == 1:
            Ls[0].forward_host(xh[i % n_x], T, yh)
        else:
            m.moe_stack_forward_host(Ls, xh[i % n_x], T, 1e-6 if wl.rmsnorm else -1.0, yh)
    for i in range(args.warmup):
        host_step(i)
    tt = 0.0
    for i in range(args.warmup, n_in):
        flush_l2(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        host_step(i)
        tt += time.perf_counter() - t0
    tt = max_over_ranks(tt, pg, dev)
    e2e = {"value": world * T * args.steps / tt, "unit": "tokens/s",
           "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 2,
           "entry_point": "moe_forward_host" if nl == 1 else "moe_stack_forward_host"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        threads = min(os.cpu_count() or 1, oracle.max_threads())
        n_tok = max(1, threads)  # one token per thread
        # batches of fresh seeded tokens until ~10 s of oracle time (at most 30 batches)
        tot_t, tot_n, nb = 0.0, 0, 0
        while tot_t < 10.0 and nb < 30:
            _, t = oracle_tokens_per_s(wl, n_tok, threads, stream=400 + nb)
            tot_t += t
            tot_n += n_tok
            nb += 1
        cpu = {"value": tot_n / tot_t, "unit": "tokens/s", "cores": min(threads, n_tok), "kind": "oracle",
               "sample": f"{nb} batch(es) of {n_tok} seeded tokens of {wl.name} ({tot_n} tokens) through "
                         f"all {nl} layer(s): input norm, routing and layer, fp64 oracle, "
                         f"{tot_t:.1f} s of oracle time"}
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "fp4xfp4->f32" if args.act == "fp4" else "fp4xfp8->f32", "data": "synthetic",
                "config": {"workload": wl.name + ("_act_fp4" if args.act == "fp4" else "") +
                           ("_shared_fp8" if args.shared == "fp8" else ""), "tokens": T, "hidden": H, "inter": wl.inter,
                           "experts": E, "top_k": k, "shared": wl.n_shared, "layers": nl,
                           "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                           "launch": "cuda_graph" if args.graph else "stream",
                           "l2": "flushed between steps (512 MB write + read), " +
                                 ("fresh tokens each step" if n_x == n_in else
                                  f"{n_x} distinct token block(s) of {T * H * 2 / 1e6:.0f} MB cycled"),
                           "mean_expert_union": mean_union,
                           "input_norm": "RMS norm of each layer's input, eps 1e-6, no gain" if nl > 1 else None},
                "layer_gbs": layer_gbs,
                "kernels": {n: {"ms_per_launch": a[0] / a[1], "launches": a[1]}
                            for n, a in ktimes.items()},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": per_step_launches * args.steps, "clocks": clocks}
        if wl.tokens >= 512:
            # useful MMA work (routed + shared slots, no tile padding) against the
            # measured block-scaled MMA peaks (issue-rate microbenchmark x SMs x the
            # median SM clock of the timed loop): the FP8-activation kind the layer
            # uses, and the FP4 x FP4 kind
            tf = layer_flops(wl, T) / (ms_step / 1e3) / 1e12
            line["tflops"] = tf
            fp8 = tensor_peak_tflops("mxf8f6f4", n_sms, sm_mhz)
            fp4 = tensor_peak_tflops("mxf4", n_sms, sm_mhz)
            up_ms = ktimes.get("ffn_up_mma", [0.0, 1])
            up_tf = (2 / 3) * layer_flops(wl, T) / (up_ms[0] / up_ms[1] / 1e3) / 1e12 if up_ms[0] else None
            line["tensor"] = {"useful_tflops": tf, "peak_fp8_kind": fp8, "frac_fp8_kind": tf / fp8,
                              "peak_fp4": fp4, "frac_fp4": tf / fp4,
                              "gate_up_kernel_tflops": up_tf,
                              "gate_up_frac_fp8_kind": up_tf / fp8 if up_tf else None,
                              "gate_up_frac_fp4": up_tf / fp4 if up_tf else None,
                              "peak_src": f"measured issue rates (mma_rate.cu) x {n_sms} SMs x {sm_mhz:.0f} MHz"}
        print(json.dumps(line), flush=True)
    for L in Ls:
        L.close()
    if pg:
        pg.destroy_process_group()
    return 0


def run_mma_rates() -> int:
    """Cycles per block-scaled tcgen05.mma (no memory traffic), both kinds the
    expert GEMM uses; prints the microbenchmark's table."""
    import subprocess
    import tempfile
    src = os.path.join(ROOT, "mma_rate.cu")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "mma_rate")
        subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe, src])
        return subprocess.call([exe])


def main():
    args = parse()
    if args.mma_rates:
        return run_mma_rates()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

"""Benchmark of the small-batch NVFP4 MoE layer on GB300.

Default workload: one NVFP4 MoE layer at T = 8 tokens (H = 2048, 256 routed
experts of I = 512, sigmoid top-6, one shared expert), the configuration the
headline metric is quoted on.  A step is one full layer forward (router +
top-6 + gate/up + SiLU*up + down + combine).  L2 is kept cold by rotating the
steps over L distinct resident layers (the selected-expert bytes of one
rotation are far larger than the 126 MB L2): step k runs layer k mod L.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--tokens T] [--layers L] [--wtype nvfp4|bf16] [--stack NL]
                    [--dense proj|large] [--no-secondary] [--no-cpu-baseline]

--stack NL measures a pre-norm decoder stack of NL resident layers instead
(x <- x + MoE_l(RMSNorm(x)), one moe_stack_forward per step; the stack is far
larger than L2, so it runs cold without rotation).

9..88 tokens (BF16 weights: 9..56) run the decode kernel on chunks of at
most 8 tokens (bytes summed over the chunks).  Above that the grouped
tensor-core path runs;
the line then reports the layer's dense-equivalent TFLOP/s (router + 7 expert
MLPs per token, padding excluded) against the measured bf16 tensor peak.
--dense times the dense NVFP4 GEMV (moe_dense_gemv_nvfp4) instead.

By default the T = 8 NVFP4 line also times, in the same process and listed
under config.secondary: NVFP4 T = 1, BF16 T = 8 and T = 1, the T = 8192
grouped layer, T = 64 (chunked), and the dense GEMV on the attention
projections (T = 8 and 1) and on one large matrix.

Prints one JSON line (rank 0).  value = algorithmic bytes of all steps / time
(GB/s); the bytes of a step are the router weights + the selected and shared
experts' packed weights + x + out.  N > 1 (torchrun) runs independent
replicas, one per GPU; value sums their bytes over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

EXPERT_BYTES = {"nvfp4": 1_179_648 + 589_824,      # packed gate/up + down of one expert
                "bf16": (2 * 512 * 2048 + 2048 * 512) * 2}
ROUTER_BYTES = 256 * 2048 * 2
METRIC = "MoE layer µs and weight-read GB/s (% of HBM peak) at T=1/8, NVFP4 and BF16"


def layer_flops(T: int, n_shared: int = 1) -> int:
    """Router GEMM + (top-6 + shared) expert MLPs of T tokens (2 flops per MAC)."""
    return 2 * T * 256 * 2048 + 2 * T * (6 + n_shared) * (2 * 512 * 2048 + 2048 * 512)


def layer_bytes(T: int, n_distinct: int, n_shared: int = 1, wtype: str = "nvfp4") -> int:
    return ROUTER_BYTES + (n_distinct + n_shared) * EXPERT_BYTES[wtype] + 2 * T * 2048 * 2


# DRAM traffic of moe_layer_kernel per algorithmic byte (dram__bytes_read.sum +
# dram__bytes_write.sum over the algorithmic bytes of two captured launches at
# T = 8).  It holds only for the kernel sources it was measured on; any change
# to them makes the bench report traffic as null.
NCU_TRAFFIC = {
    # DRAM bytes read + written per algorithmic byte of the decode kernel at
    # T = 8, from one ncu capture of two launches (layers with 46 and 42
    # distinct experts: 168,418,304 bytes against 161,480,704), valid while
    # the kernel's sources hash to this value
    "sources_sha256": "e4728cf4b97467716ce9734e60dd6010695bf7df396f66a7804e0bdfd19a8a4f",
    "per_algorithmic_byte": 168_418_304 / 161_480_704,
}
KERNEL_SOURCES = ("layer.cu", "stage.cuh", "common.cuh", "kernels.cuh", "topk.cuh")


def kernel_sources_sha256() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "nvfp4_moe_decode_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.gpu)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


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
        dist.init_process_group(backend=backend)
    return world, rank, local


def reduce_max(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ---------------------------------------------------------------------------
# CPU oracle timing (the reference arm and cpu_baseline)
# ---------------------------------------------------------------------------

def oracle_sample(layers_host, x_bits, T: int, budget_s: float, wtype: str = "nvfp4"):
    """Run the fp64 oracle layer over the resident layers until budget_s.
    Returns (seconds, algorithmic bytes, layers done, threads)."""
    import oracle

    done, nbytes, t0 = 0, 0, time.perf_counter()
    while True:
        for (wr, experts, shared, nd) in layers_host:
            oracle.moe_forward(x_bits, wr, experts, 6, 512, shared)
            done += 1
            nbytes += layer_bytes(T, nd, 1, wtype)
            if time.perf_counter() - t0 >= budget_s:
                return time.perf_counter() - t0, nbytes, done, oracle.num_threads()


def host_expert(li, e: int):
    """Host copy of expert e of a synthetic layer, in the oracle's form."""
    import numpy as np
    import torch

    import oracle

    if li.wtype == 0:
        return oracle.ExpertWeights(0, li.codes13[e].cpu().numpy(), li.scales13[e].cpu().numpy(),
                                    float(li.tscale13[e]), li.codes2[e].cpu().numpy(),
                                    li.scales2[e].cpu().numpy(), float(li.tscale2[e]))
    bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)  # noqa: E731
    return oracle.ExpertWeights(1, bits(li.w13[e]), None, 1.0, bits(li.w2[e]), None, 1.0)


def host_layers_for_oracle(lis, x, n: int):
    """Host copies of the experts the oracle will select in the first n layers."""
    import numpy as np
    import torch

    import oracle

    bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)  # noqa: E731
    xb = bits(x)
    out = []
    for li in lis[:n]:
        wr = bits(li.router_w)
        idx, _ = oracle.select_topk(oracle.router_logits(xb, wr), 6)
        experts = [None] * 256
        sel = sorted(set(idx.reshape(-1).tolist()))
        for e in sel:
            experts[e] = host_expert(li, e)
        out.append((wr, experts, host_expert(li, 256), len(sel)))
    return xb, out


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--tokens", type=int, default=8)
    ap.add_argument("--layers", type=int, default=16)
    ap.add_argument("--wtype", choices=["nvfp4", "bf16"], default="nvfp4")
    ap.add_argument("--stack", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dense", choices=["proj", "large"], default=None,
                    help="time the dense NVFP4 GEMV instead: the attention projections (qkv 5120 x 2048, "
                         "o 2048 x 4096, 32 matrices) or one large matrix (16384 x 4096, --dense-mats of them)")
    ap.add_argument("--dense-mats", type=int, default=8)
    ap.add_argument("--no-secondary", action="store_true",
                    help="time only the selected workload (by default the T=8 NVFP4 line also times "
                         "NVFP4 T=1, BF16 T=8 and T=1, T=8192, T=64 and the dense GEMV)")
    args = ap.parse_args()
    assert args.warmup >= 3

    import torch

    world, rank, local = dist_setup()
    T, L, WT = args.tokens, args.layers, args.wtype
    WTI = 0 if WT == "nvfp4" else 1
    workload = (f"one {WT.upper()} MoE layer, T={T} tokens (H=2048, 256 routed experts I=512, sigmoid top-6, "
                f"1 shared expert), synthetic seeded weights")
    config = {"workload": workload, "weights": WT, "tokens": T, "hidden": 2048, "experts": 256, "top_k": 6, "inter": 512,
              "layers_rotated": L,
              "l2": f"cold: steps rotate over {L} distinct resident layers (selected bytes per rotation >> L2)"}

    if args.impl == "reference":
        if rank != 0:
            return
        from nvfp4_moe_decode_gb300 import synth

        dev = "cuda" if torch.cuda.is_available() else "cpu"
        import oracle

        oracle.build()
        nl = min(L, 4)
        lis = [synth.make_layer(s, T, wtype=WTI, device=dev) for s in range(nl)]
        x = lis[0].x
        xb, hl = host_layers_for_oracle(lis, x, nl)
        for _ in range(args.warmup if args.warmup < 4 else 3):
            oracle.moe_forward(xb, hl[0][0], hl[0][1], 6, 512, hl[0][2])
        t_tot, b_tot, n_tot = 0.0, 0, 0
        for _ in range(args.steps if args.steps <= 20 else 20):
            s, b, n, threads = oracle_sample(hl, xb, T, 0.0, WT)
            t_tot += s
            b_tot += b
            n_tot += n
        v = b_tot / t_tot / 1e9
        line = {"metric": METRIC, "value": v, "unit": "GB/s", "impl": "reference", "n_gpus": args.gpus,
                "steps": n_tot, "warmup": args.warmup, "ms_per_step": 1e3 * t_tot / n_tot,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"kind": "oracle", "value": v, "unit": "GB/s", "cores": threads,
                                 "sample": f"{n_tot} layer forwards of the fp64 C oracle, one per step"},
                "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import nvfp4_moe_decode_gb300 as m

    m.load()
    if args.stack:
        return run_stack(args, world, rank, local)
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    K, W = args.steps, args.warmup
    if args.dense:
        shapes, nm = (([(5120, 2048), (2048, 4096)], 32) if args.dense == "proj"
                      else ([(16384, 4096)], args.dense_mats))
        line = measure_dense(args, T, shapes, nm, world, dev, K, W,
                             "attention projections" if args.dense == "proj" else "one large matrix")
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    if T > chunk_limit(WT):
        line = measure_grouped(args, T, WT, world, dev, True, K, W)
    else:
        line = measure_decode(args, T, WT, L, world, dev, True, K, W)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args, T, WT, L, dev)
    if not args.no_secondary and T == 8 and WT == "nvfp4":
        # the other points of the metric, timed the same way in this process
        sec = []
        # secondary step counts: at least as many as the main line up to 2,000
        # decode steps (40 grouped steps of ~1 ms), after at least 3 warm-ups
        k2, w2 = max(min(K, 2000), 16), max(min(W, 64), 3)
        for (t2, wt2) in ((1, "nvfp4"), (8, "bf16"), (1, "bf16")):
            sec.append(secondary_entry(measure_decode(args, t2, wt2, L, world, dev, False, k2, w2)))
            torch.cuda.empty_cache()
        sec.append(secondary_entry(measure_grouped(args, 8192, "nvfp4", world, dev, False,
                                                   max(min(K, 40), 4), max(min(W, 6), 3))))
        torch.cuda.empty_cache()
        # a mid-size batch: the decode kernel on chunks of at most 8 tokens
        sec.append(secondary_entry(measure_decode(args, 64, "nvfp4", L, world, dev, False,
                                                  max(min(K, 200), 16), w2)))
        torch.cuda.empty_cache()
        # the dense GEMV on the packed layout: the attention projections of a
        # 2048-wide decoder (qkv 5120 x 2048, o 2048 x 4096), and a large matrix
        for (t2, shapes, nm, label) in ((8, [(5120, 2048), (2048, 4096)], 32, "attention projections"),
                                        (1, [(5120, 2048), (2048, 4096)], 32, "attention projections"),
                                        (8, [(16384, 4096)], 8, "one large matrix")):
            sec.append(secondary_entry(measure_dense(args, t2, shapes, nm, world, dev, k2, w2, label)))
            torch.cuda.empty_cache()
        line["config"]["secondary"] = sec
        line["gpu_launches"] += sum(e["gpu_launches"] for e in sec)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def secondary_entry(line) -> dict:
    """The summary of a measured line kept under config.secondary."""
    c = line["config"]
    return {"workload": c["workload"], "tokens": c["tokens"], "weights": c["weights"],
            "us_per_layer": c["us_per_layer"], "value": line["value"], "unit": line["unit"],
            "frac": line["roofline"]["frac"], "bound": line["roofline"]["bound"],
            "peak": line["roofline"]["peak"], "steps": line["steps"],
            "device_flag": c["device_flag"], "clocks": line["clocks"], "gpu_launches": line["gpu_launches"]}


def timed_replays(stream, graphs, local: int):
    """Replay ``graphs`` (a list of (graph, times)) between two CUDA events on
    ``stream``, after a barrier and a device synchronize.  A ~1 ms GPU sleep
    is enqueued ahead of the start event so that the host's launch latency
    of the first graph falls outside the timed span.  Returns (ms, clocks)."""
    import torch

    clocks = ClockSampler(local)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(2_000_000)
        e0.record(stream)
        for g, n in graphs:
            for _ in range(n):
                g.replay()
        e1.record(stream)
    e1.synchronize()
    clk = clocks.stop()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1), clk


def chunk_limit(WT: str) -> int:
    """The largest T the library runs as chunks of the decode kernel."""
    import nvfp4_moe_decode_gb300 as m
    return m.MAX_CHUNKED_T_BF16 if WT == "bf16" else m.MAX_CHUNKED_T


def chunks_of(T: int):
    """The library's balanced chunks of at most 8 tokens (T <= chunk_limit)."""
    n = (T + 7) // 8
    return [(T * c // n, T * (c + 1) // n) for c in range(n)]


def measure_decode(args, T: int, WT: str, L: int, world: int, dev, with_e2e: bool, K: int, W: int) -> dict:
    """One decode-path layer (T <= 8, or up to chunk_limit tokens in chunks of at
    most 8) per step, rotating over L resident layers.  The bytes of a step
    add up the chunks: each reads the router, its own selected and the
    shared experts, its x and out."""
    import torch

    import nvfp4_moe_decode_gb300 as m
    from nvfp4_moe_decode_gb300 import synth
    from nvfp4_moe_decode_gb300.layer import Bf16Layer, PackedLayer, new_workspace

    WTI = 0 if WT == "nvfp4" else 1
    stream = torch.cuda.Stream(dev)
    # ---- resident layers (seeds 0..L-1), x fixed (seed 0) ----
    packed = []
    x = synth.make_x(0, T, device=dev)
    with torch.cuda.stream(stream):
        for s in range(L):
            li = synth.make_layer(s, T, wtype=WTI, device=dev)
            packed.append(PackedLayer.from_inputs(li, stream) if WTI == 0 else Bf16Layer.from_inputs(li))
            del li
    stream.synchronize()
    # distinct routed experts per layer (from our router, outside the timed region)
    ws = new_workspace(T, dev, stream)
    nd = []
    with torch.cuda.stream(stream):
        idx = torch.empty(T, 6, dtype=torch.int32, device=dev)
        w = torch.empty(T, 6, dtype=torch.float32, device=dev)
        for pl in packed:
            m.moe_route(x, pl.router_w, T, idx, w, None, ws, stream)
            stream.synchronize()
            ih = idx.cpu().numpy()
            nd.append([len(set(ih[t0:t1].reshape(-1).tolist())) for (t0, t1) in chunks_of(T)])
    m.moe_workspace_init(ws, stream)
    out = torch.empty(T, 2048, dtype=torch.bfloat16, device=dev)

    def run_steps(k0: int, n: int):
        for k in range(k0, k0 + n):
            packed[k % L].forward(x, out, ws, stream)

    # ---- graphs: one rotation of L steps, plus the remainder ----
    def capture(n: int):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run_steps(0, n)
        return g

    run_steps(0, L)   # eager warm-up before capture
    stream.synchronize()
    g_full = capture(L)
    with torch.cuda.stream(stream):
        for _ in range(max(1, W // L)):
            g_full.replay()
        run_steps(0, W % L)
    stream.synchronize()
    rem_graph = capture(K % L) if K % L else None
    def step_bytes(k):
        return sum(layer_bytes(t1 - t0, u, 1, WT) for (t0, t1), u in zip(chunks_of(T), nd[k % L]))

    steps_bytes = sum(step_bytes(k) for k in range(K))

    barrier(world)
    graphs = [(g_full, K // L)] + ([(rem_graph, 1)] if rem_graph is not None else [])
    ms, clk = timed_replays(stream, graphs, dev.index)
    barrier(world)
    ms_max = reduce_max(ms, world)
    total_bytes = reduce_sum(float(steps_bytes), world)
    value = total_bytes / (ms_max * 1e-3) / 1e9
    us_per_layer = 1e3 * ms_max / K
    flag = m.moe_read_device_flag(ws, stream)

    peak, peak_src = peaks()
    layer_alg = steps_bytes / K
    traffic = None
    if WT == "nvfp4" and kernel_sources_sha256() == NCU_TRAFFIC["sources_sha256"]:
        traffic = layer_alg * NCU_TRAFFIC["per_algorithmic_byte"]
    workload = (f"one {WT.upper()} MoE layer, T={T} tokens (H=2048, 256 routed experts I=512, sigmoid top-6, "
                f"1 shared expert), synthetic seeded weights"
                + (f"; decode kernel on {len(chunks_of(T))} chunks of at most 8 tokens" if T > 8 else ""))
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_max / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": f"{WT} weights x bf16 activations, f32 accumulate", "data": "synthetic",
        "config": {"workload": workload, "weights": WT, "tokens": T, "hidden": 2048, "experts": 256, "top_k": 6,
                   "inter": 512, "layers_rotated": L,
                   "l2": f"cold: steps rotate over {L} distinct resident layers (selected bytes per rotation >> L2)",
                   "timing": "CUDA events on the launching stream around K graph-replayed steps; a 1 ms GPU sleep "
                             "ahead of the start event keeps host launch latency out of the span",
                   "us_per_layer": us_per_layer, "tokens_per_s": T * K / (ms_max * 1e-3),
                   "distinct_experts_per_layer": [v[0] if len(v) == 1 else v for v in nd],
                   "algorithmic_bytes_per_layer": layer_alg,
                   "hbm_frac": value / world / peak, "device_flag": flag},
        "roofline": {"bound": "hbm", "achieved": layer_alg / (us_per_layer * 1e-6) / 1e9, "peak": peak,
                     "unit": "GB/s", "frac": layer_alg / (us_per_layer * 1e-6) / 1e9 / peak,
                     "traffic": traffic, "peak_source": peak_src,
                     "kernel": "moe_layer_kernel (router, top-6, gate/up, down, combine fused; one launch per layer)"},
        "gpu_launches": K * len(chunks_of(T)),
        "clocks": clk,
    }
    if with_e2e:
        # ---- e2e: host x in, host out back, through the public C-ABI ----
        xh = x.cpu().pin_memory()
        oh = torch.empty(T, 2048, dtype=torch.bfloat16).pin_memory()
        ne = args.e2e_steps
        xd = torch.empty_like(x)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for k in range(ne):
                xd.copy_(xh, non_blocking=True)
                packed[k % L].forward(xd, out, ws, stream)
                oh.copy_(out, non_blocking=True)
                stream.synchronize()
        e2e_s = time.perf_counter() - t0
        e2e_bytes = sum(step_bytes(k) for k in range(ne))
        e2e_v = reduce_sum(e2e_bytes, world) / reduce_max(e2e_s, world) / 1e9
        line["e2e"] = {"value": e2e_v, "unit": "GB/s", "steps": ne, "h2d_bytes_per_step": T * 2048 * 2,
                       "d2h_bytes_per_step": T * 2048 * 2}
    del packed, ws
    return line


def cpu_baseline(args, T: int, WT: str, L: int, dev) -> dict:
    """The fp64 oracle on the host cores over a bounded sample of the workload."""
    from nvfp4_moe_decode_gb300 import synth

    import oracle

    oracle.build()
    WTI = 0 if WT == "nvfp4" else 1
    if T > 8:
        n_tok = 4
        li = synth.make_layer(0, T, wtype=WTI, device=dev)
        xs = li.x[:n_tok].contiguous()
        xb, hl = host_layers_for_oracle([synth.LayerInputs(**{**li.__dict__, "x": xs})], xs, 1)
        del li
        t0 = time.perf_counter()
        done = 0
        while time.perf_counter() - t0 < args.cpu_budget:
            oracle.moe_forward(xb, hl[0][0], hl[0][1], 6, 512, hl[0][2])
            done += 1
        sec = time.perf_counter() - t0
        return {"value": layer_flops(n_tok) * done / sec / 1e12, "unit": "TFLOP/s",
                "cores": oracle.num_threads(), "kind": "oracle",
                "sample": f"{done} oracle layer forwards of {n_tok} of the {T} tokens, {sec:.1f} s"}
    x = synth.make_x(0, T, device=dev)
    lis = [synth.make_layer(s, T, wtype=WTI, device=dev) for s in range(min(L, 4))]
    xb, hl = host_layers_for_oracle(lis, x, len(lis))
    del lis
    s, b, n, threads = oracle_sample(hl, xb, T, args.cpu_budget, WT)
    return {"value": b / s / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} layer forwards (T={T}) of the fp64 C oracle over {len(hl)} of the rotated layers, "
                      f"{s:.1f} s"}


def measure_grouped(args, T: int, WT: str, world: int, dev, with_e2e: bool, K: int, W: int) -> dict:
    """One layer at T > 8 tokens (the grouped tensor-core path) per step, two
    resident layers alternated."""
    import torch

    import nvfp4_moe_decode_gb300 as m
    from nvfp4_moe_decode_gb300 import synth
    from nvfp4_moe_decode_gb300.layer import Bf16Layer, PackedLayer, new_workspace

    WTI = 0 if WT == "nvfp4" else 1
    stream = torch.cuda.Stream(dev)
    L = 2
    layers = []
    with torch.cuda.stream(stream):
        for s_ in range(L):
            li = synth.make_layer(s_, T, wtype=WTI, device=dev)
            layers.append(PackedLayer.from_inputs(li, stream) if WTI == 0 else Bf16Layer.from_inputs(li))
            if s_ == 0:
                x = li.x
            del li
    ws = new_workspace(T, dev, stream)
    out = torch.empty(T, 2048, dtype=torch.bfloat16, device=dev)
    with torch.cuda.stream(stream):
        for k in range(W):
            layers[k % L].forward(x, out, ws, stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for k in range(L):
            layers[k].forward(x, out, ws, stream)
    reps = max(1, K // L)
    barrier(world)
    ms, clk = timed_replays(stream, [(g, reps)], dev.index)
    barrier(world)
    steps = reps * L
    ms_max = reduce_max(ms, world)
    fl = layer_flops(T)
    value = reduce_sum(float(fl * steps), world) / (ms_max * 1e-3) / 1e12
    us_layer = 1e3 * ms_max / steps
    flag = m.moe_read_device_flag(ws, stream)
    idx = torch.empty(T, 6, dtype=torch.int32, device=dev)
    w = torch.empty(T, 6, dtype=torch.float32, device=dev)
    m.moe_route(x, layers[0].router_w, T, idx, w, None, ws, stream)
    load = torch.bincount(idx.reshape(-1).long(), minlength=256)

    pk = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else None
    peak = float(pk["bf16_tflops_sustained"]) if pk else 1700.0
    achieved = fl / (us_layer * 1e-6) / 1e12
    workload = (f"one {WT.upper()} MoE layer, T={T} tokens (H=2048, 256 routed experts I=512, sigmoid top-6, "
                f"1 shared expert), synthetic seeded weights; grouped tcgen05 path")
    line = {
        "metric": "MoE layer TFLOP/s (% of bf16 tensor peak) at T=8192, grouped path", "value": value,
        "unit": "TFLOP/s", "n_gpus": world, "steps": steps, "warmup": W, "ms_per_step": ms_max / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("nvfp4 weights as f16 x f16 activations" if WTI == 0 else "bf16 x bf16") + ", f32 accumulate",
        "data": "synthetic",
        "config": {"workload": workload, "weights": WT, "tokens": T, "hidden": 2048, "experts": 256, "top_k": 6,
                   "inter": 512, "layers_rotated": L,
                   "l2": "cold: 2 layers of weights (>= 455 MB each) alternated, far above L2",
                   "us_per_layer": us_layer, "tokens_per_s": T / (us_layer * 1e-6), "flops_per_layer": fl,
                   "expert_load_min_max": [int(load.min()), int(load.max())], "device_flag": flag},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None,
                     "peak_source": "measured (sustained)" if pk else "fallback",
                     "kernel": "the grouped chain per layer (router GEMM, top-k, lists, gate/up, h rescale, down, "
                               "shared down + combine)"},
        "gpu_launches": steps * 8,
        "clocks": clk,
    }
    if with_e2e:
        xh = x.cpu().pin_memory()
        oh = torch.empty(T, 2048, dtype=torch.bfloat16).pin_memory()
        xd = torch.empty_like(x)
        ne = max(3, min(args.e2e_steps, 50))
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for k in range(ne):
                xd.copy_(xh, non_blocking=True)
                layers[k % L].forward(xd, out, ws, stream)
                oh.copy_(out, non_blocking=True)
                stream.synchronize()
        e2e_v = reduce_sum(float(fl * ne), world) / reduce_max(time.perf_counter() - t0, world) / 1e12
        line["e2e"] = {"value": e2e_v, "unit": "TFLOP/s", "steps": ne, "h2d_bytes_per_step": T * 2048 * 2,
                       "d2h_bytes_per_step": T * 2048 * 2}
    del layers, ws
    return line


def measure_dense(args, T: int, shapes, n_mats: int, world: int, dev, K: int, W: int, label: str) -> dict:
    """Dense NVFP4 GEMVs (moe_dense_gemv_nvfp4), one per step, over n_mats
    distinct resident matrices whose (N, K) cycle through ``shapes``; step k
    runs matrix k mod n_mats (the matrices of one rotation are far larger than
    L2).  The bytes of a step are the packed matrix + x + y."""
    import torch

    import nvfp4_moe_decode_gb300 as m
    from nvfp4_moe_decode_gb300 import synth

    stream = torch.cuda.Stream(dev)
    mats = []
    with torch.cuda.stream(stream):
        for i in range(n_mats):
            N, Kd = shapes[i % len(shapes)]
            d = synth.make_dense(1000 + i, T, N, Kd, device=dev)
            pk = torch.empty(m.moe_packed_bytes(N, Kd), dtype=torch.uint8, device=dev)
            m.moe_pack_nvfp4(d.codes, d.scales, N, Kd, m.MOE_PACK_PLAIN, 1, pk, stream)
            mats.append((N, Kd, pk, d.x.clone(), torch.empty(T, N, dtype=torch.bfloat16, device=dev)))
            del d
    stream.synchronize()
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)

    def step_bytes(N, Kd):
        return m.moe_packed_bytes(N, Kd) + 4 + T * Kd * 2 + T * N * 2

    def run_steps(n: int):
        for k in range(n):
            N, Kd, pk, xx, yy = mats[k % n_mats]
            m.moe_dense_gemv_nvfp4(xx, pk, 1.0, N, Kd, T, yy, ws, stream)

    with torch.cuda.stream(stream):
        run_steps(n_mats)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run_steps(n_mats)
    with torch.cuda.stream(stream):
        for _ in range(max(1, W // n_mats)):
            g.replay()
    stream.synchronize()
    reps = max(1, K // n_mats)
    steps = reps * n_mats
    barrier(world)
    ms, clk = timed_replays(stream, [(g, reps)], dev.index)
    barrier(world)
    ms_max = reduce_max(ms, world)
    rot_bytes = sum(step_bytes(N, Kd) for (N, Kd, _, _, _) in mats)
    alg = rot_bytes / n_mats
    value = reduce_sum(float(rot_bytes * reps), world) / (ms_max * 1e-3) / 1e9
    us = 1e3 * ms_max / steps
    flag = m.moe_read_device_flag(ws, stream)
    peak, peak_src = peaks()
    shp = ", ".join(f"{N}x{Kd}" for (N, Kd) in shapes)
    workload = (f"dense NVFP4 GEMV y = W x, T={T} tokens, W of {shp} ({label}), packed layout, "
                f"synthetic seeded weights")
    line = {
        "metric": "dense NVFP4 GEMV weight-read GB/s (% of HBM peak)", "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": steps, "warmup": W, "ms_per_step": ms_max / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4 weights x bf16 activations, f32 accumulate",
        "data": "synthetic",
        "config": {"workload": workload, "weights": "nvfp4", "tokens": T, "layers_rotated": n_mats,
                   "l2": f"cold: steps rotate over {n_mats} distinct resident matrices "
                         f"({rot_bytes / 1e6:.0f} MB, above L2)",
                   "us_per_layer": us, "algorithmic_bytes_per_step": alg, "device_flag": flag},
        "roofline": {"bound": "hbm", "achieved": alg / (us * 1e-6) / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": alg / (us * 1e-6) / 1e9 / peak, "traffic": None, "peak_source": peak_src,
                     "kernel": "dense_gemv_kernel"},
        "gpu_launches": steps,
        "clocks": clk,
    }
    del mats
    return line


def run_stack(args, world: int, rank: int, local: int):
    """A pre-norm stack of args.stack layers (seeds 0..NL-1), T tokens."""
    import torch

    import nvfp4_moe_decode_gb300 as m
    from nvfp4_moe_decode_gb300 import synth
    from nvfp4_moe_decode_gb300.layer import Bf16Layer, PackedLayer, Stack, new_stack_workspace, new_workspace

    T, NL, WT = args.tokens, args.stack, args.wtype
    WTI = 0 if WT == "nvfp4" else 1
    eps = 1e-6
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    layers = []
    with torch.cuda.stream(stream):
        for s in range(NL):
            li = synth.make_layer(s, T, wtype=WTI, device=dev)
            layers.append(PackedLayer.from_inputs(li, stream) if WTI == 0 else Bf16Layer.from_inputs(li))
            del li
    stream.synchronize()
    x0 = synth.make_x(0, T, device=dev)
    # distinct experts per layer: the stack layer by layer, routing each
    # layer's own normalised input (outside the timed region)
    nd = []
    wsl = new_workspace(T, dev, stream)
    with torch.cuda.stream(stream):
        resid, delta = x0.clone(), None
        idx = torch.empty(T, 6, dtype=torch.int32, device=dev)
        w = torch.empty(T, 6, dtype=torch.float32, device=dev)
        for lay in layers:
            out = torch.empty(T, 2048, dtype=torch.bfloat16, device=dev)
            v, xn = torch.empty_like(out), torch.empty_like(out)
            m.moe_layer_forward_prenorm(resid, delta, v, xn, eps, lay.router_w, lay.routed, lay.shared, out, T,
                                        wsl, stream)
            m.moe_route(xn, lay.router_w, T, idx, w, None, wsl, stream)
            stream.synchronize()
            nd.append(len(set(idx.cpu().reshape(-1).tolist())))
            resid, delta = v, out
    st = Stack(layers, eps)
    ws = new_stack_workspace(T, dev, stream)
    x = x0.clone()
    # per layer: the layer's weights + x and out, plus the residual stream
    # (delta read, residual written); the final add reads two and writes one
    step_bytes = sum(layer_bytes(T, n, 1, WT) + 2 * T * 2048 * 2 for n in nd) + 3 * T * 2048 * 2

    def step():
        x.copy_(x0)
        st.forward(x, ws, stream)

    K, W = args.steps, args.warmup
    with torch.cuda.stream(stream):
        for _ in range(W):
            step()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.2)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(K):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    clk = clocks.stop()
    torch.cuda.synchronize(dev)
    barrier(world)
    ms_max = reduce_max(e0.elapsed_time(e1), world)
    value = reduce_sum(float(step_bytes * K), world) / (ms_max * 1e-3) / 1e9
    us_stack = 1e3 * ms_max / K
    flag = m.moe_read_device_flag(ws, stream)

    xh = x0.cpu().pin_memory()
    oh = torch.empty(T, 2048, dtype=torch.bfloat16).pin_memory()
    ne = max(3, min(args.e2e_steps, K))
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(ne):
            x.copy_(xh, non_blocking=True)
            st.forward(x, ws, stream)
            oh.copy_(x, non_blocking=True)
            stream.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_v = reduce_sum(float(step_bytes * ne), world) / reduce_max(e2e_s, world) / 1e9

    peak, peak_src = peaks()
    workload = (f"{NL}-layer pre-norm stack of {WT.upper()} MoE layers, T={T} tokens (H=2048, 256 routed experts "
                f"I=512, sigmoid top-6, 1 shared expert), synthetic seeded weights")
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_max / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": f"{WT} weights x bf16 activations, f32 accumulate", "data": "synthetic",
        "config": {"workload": workload, "weights": WT, "tokens": T, "layers": NL, "hidden": 2048,
                   "experts": 256, "top_k": 6, "inter": 512,
                   "l2": "cold: the stack's selected weights far exceed L2",
                   "us_per_stack": us_stack, "us_per_layer": us_stack / NL,
                   "tokens_per_s": T / (us_stack * 1e-6), "distinct_experts_per_layer": nd,
                   "algorithmic_bytes_per_step": step_bytes, "hbm_frac": value / world / peak,
                   "resident_weight_bytes": sum(l.bytes_resident() for l in layers), "device_flag": flag},
        "roofline": {"bound": "hbm", "achieved": step_bytes / (us_stack * 1e-6) / 1e9, "peak": peak,
                     "unit": "GB/s", "frac": step_bytes / (us_stack * 1e-6) / 1e9 / peak, "traffic": None,
                     "peak_source": peak_src,
                     "kernel": "moe_layer_kernel x NL (pre-norm residual fused) + residual_add_kernel"},
        "e2e": {"value": e2e_v, "unit": "GB/s", "steps": ne, "h2d_bytes_per_step": T * 2048 * 2,
                "d2h_bytes_per_step": T * 2048 * 2},
        "gpu_launches": K * (NL + 1),
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()

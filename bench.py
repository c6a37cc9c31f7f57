"""Benchmark: fp9 MoE-layer decode on one GB300 (DeepSeek-V3 MoE layer, bsz 1).

A step is one MoE-layer forward (router, fused fp9 expert kernel, combine)
for one batch of synthetic tokens, on one of several resident layers in
turn, so every step streams its 446 MB of fp9 expert weights from HBM
(4 layers x 12.7 GB rotate; no weight is re-read within 3 steps, far more
than the 129 MB L2).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
  python bench.py --leg fp8_to_fp9|prefill|moe_prefill   (one side measurement alone)

Prints one JSON line (rank 0). ``--impl reference`` times the CPU oracle on
the host cores instead (one token through one whole MoE layer per step, its
expert FFNs on one worker process each). Multi-GPU runs are independent replicas (the path
has no exchange step), launched one rank per GPU by torchrun.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fp9 MoE-layer decode tok/s (bsz 1/2) & weight-stream HBM GB/s vs GB300 peak"
FP9_BYTES_PER_WEIGHT = 9.0 / 8.0


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)
    p.add_argument("--warmup", type=int, default=100)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--bsz", type=int, default=1)
    p.add_argument("--layers", type=int, default=4, help="resident layers rotated per step")
    p.add_argument("--experts", type=int, default=256,
                   help="routed experts per layer (smaller layers for profiling captures)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-extra", action="store_true", help="skip the bsz-2 / dense side runs")
    p.add_argument("--leg", choices=["fp8_to_fp9", "prefill", "moe_prefill", "stack"], default=None,
                   help="run one side measurement alone and print its record (profiling captures)")
    p.add_argument("--tokens", type=int, nargs="+", default=[1481, 4096],
                   help="prompt lengths of the moe_prefill leg")
    p.add_argument("--cpu-sample", type=str, default=None, help=argparse.SUPPRESS)
    return p.parse_args()


KERNEL_SOURCES = ("fp9_weight_expert_gb300/csrc/fp9_expert.cu", "fp9_weight_expert_gb300/csrc/fp9_device.cuh",
                  "fp9_weight_expert_gb300/csrc/fp9_plan.h")


def _profiled_traffic():
    """DRAM bytes per fused-kernel launch from the committed ncu summary, or
    None when the kernel's sources changed since that capture."""
    import hashlib
    import re
    try:
        text = open(os.path.join(ROOT, "profiles", "expert_kernel_dsv3_bsz1.md")).read()
        want = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text).group(1)
        traffic = int(re.search(r"traffic_bytes_per_launch:\s*(\d+)", text).group(1))
        h = hashlib.sha256()
        for f in KERNEL_SOURCES:
            with open(os.path.join(ROOT, f), "rb") as fh:
                h.update(fh.read())
        return traffic if h.hexdigest()[:16] == want else None
    except Exception:
        return None


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _tensor_peak():
    """Dense bf16 tensor TFLOP/s timed alone (burst), measured on this GPU
    model, else the fallback figure."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


# ------------------------------------------------------------ clock sampler

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self, t0: float, t1: float):
        """Median SM clock and active throttle reasons over samples taken
        between host times t0 and t1 (the nearest sample if none fell inside)."""
        import datetime
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[1]), float(f[2]), float(f[3]), f[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        if not inside and rows:
            inside = [min(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))]
        reasons = set()
        for r in inside:
            for n, v in zip(names, r[4]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in inside) if inside else None,
                "sm_max_mhz": inside[0][2] if inside else None,
                "power_w_max": max(r[3] for r in inside) if inside else None,
                "reasons": sorted(reasons), "samples": len(inside)}


# ------------------------------------------------------- replica plumbing

def max_over_ranks(value: float) -> float:
    """Largest value over the ranks of the default process group (the value
    itself when not distributed). Host-side only (gloo), no data-path
    collective: replicas are independent."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world: int, bsz: int, steps: int, max_elapsed_s: float) -> float:
    """Whole-job tokens/s: every rank processed bsz * steps tokens; the job
    took as long as its slowest rank."""
    return world * bsz * steps / max_elapsed_s


# ----------------------------------------------------------- native bench

def _native(args):
    import torch
    import torch.distributed as dist

    from fp9_weight_expert_gb300 import Workspace, binding, build_lib, layers, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    if rank == 0:
        build_lib.build()
    if world > 1:
        dist.barrier()
    binding.load()

    shape = synth.DSV3
    if args.experts != shape.n_experts:
        import dataclasses
        shape = dataclasses.replace(shape, n_experts=args.experts)
    H, I, bsz = shape.hidden, shape.inter, args.bsz
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if args.leg == "fp8_to_fp9":
        return {"leg": args.leg, **_convert_run(dev, _peaks()[0])}
    if args.leg == "prefill":
        return {"leg": args.leg, **_prefill_run(dev, _tensor_peak())}
    if args.leg == "stack":
        return {"leg": args.leg, **_stack_run(dev, shape)}

    def make_layer(l):
        L = layers.MoELayer(H, I, shape.n_experts, shape.n_groups, shape.topk_groups, shape.topk,
                            shape.n_shared, shape.route_scale, dev)
        kinds = (synth.ROUTED, synth.SHARED)
        L.fill(lambda b, k, m: synth.ffn_weight(shape, I, H, synth.seed_for(1000 + rank, l, kinds[b], k, m), dev),
               synth.normal((shape.n_experts, H), shape.router_std,
                            synth.seed_for(1000 + rank, l, synth.ROUTER), dev), status)
        return L

    t0 = time.time()
    Ls = [make_layer(l) for l in range(args.layers)]
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("packing failed: " + binding.status_str(int(status.item())))
    setup_s = time.time() - t0
    if args.leg == "moe_prefill":
        return {"leg": args.leg, "experts": shape.n_experts,
                **_moe_prefill_run(Ls, status, dev, shape, args.tokens)}

    n_tok = 64
    xs = synth.tokens(n_tok * bsz, H, synth.seed_for(2000 + rank, 0, synth.TOKENS), dev).view(n_tok, bsz, H)
    y = torch.empty((bsz, H), dtype=torch.float32, device=dev)
    K, W = args.steps, args.warmup
    ids = torch.empty((K, bsz, shape.topk), dtype=torch.int32, device=dev)
    ws = Workspace.for_moe(Ls[0], bsz, dev)
    stream = torch.cuda.current_stream()

    def step(i, ids_out=None):
        binding.fp9_moe_forward(Ls[i % len(Ls)], xs[i % n_tok], y, ws.tensor, status, ids_out)

    # The clock sampler starts before the warm-up, so that the GPU stays busy
    # from the warm-up into the timed region (an idle GPU takes a while to
    # come back to full speed, which a short region would measure).
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    for i in range(W):
        step(i)
    if world > 1:
        torch.cuda.synchronize()
        dist.barrier()
    # Timed region: K back-to-back steps with nothing queued between the
    # launches (an event recorded between two launches would stop the next
    # kernel from starting while the previous one finishes).
    torch.cuda.synchronize()
    t_region0 = time.time()
    start.record(stream)
    for i in range(K):
        step(W + i, ids[i])
    stop.record(stream)
    torch.cuda.synchronize()
    t_region1 = time.time()
    if world > 1:
        dist.barrier()

    # Kernel region: the same steps again, with CUDA events around every
    # launch of the fused expert kernel, for its duration.
    Kk = min(K, 2000)
    ev_k = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Kk)]
    for a, b in ev_k:  # torch creates the CUDA event on first record
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    for i in range(Kk):
        binding.fp9_profile_events(ev_k[i][0], ev_k[i][1])
        step(W + i)
    torch.cuda.synchronize()
    binding.fp9_profile_events(None, None)
    time.sleep(0.1)
    sampler.stop()
    if int(status.item()) != 0:
        raise RuntimeError("device status: " + binding.status_str(int(status.item())))

    elapsed_ms = max_over_ranks(start.elapsed_time(stop))
    kern_ms = [a.elapsed_time(b) for a, b in ev_k]

    # union of experts streamed per step: distinct routed ids + shared
    idc = ids.cpu()
    units = [len(set(idc[i].flatten().tolist())) + shape.n_shared for i in range(K)]
    unit_bytes = 3 * I * H * FP9_BYTES_PER_WEIGHT
    weight_bytes = [u * unit_bytes for u in units]
    mean_kern_s = sum(kern_ms) / Kk / 1e3
    kernel_gbs = (sum(weight_bytes[:Kk]) / Kk) / mean_kern_s / 1e9
    step_gbs = sum(weight_bytes) / (elapsed_ms / 1e3) / 1e9
    # all algorithmic bytes of a step: the fp9 weights, the fp32 router
    # weights (4 E H) and x and y (8 bsz H)
    other_bytes = 4 * shape.n_experts * H + 8 * bsz * H
    total_gbs = (sum(weight_bytes) + K * other_bytes) / (elapsed_ms / 1e3) / 1e9
    peak, peak_kind = _peaks()

    # end to end through the C ABI with host buffers: one fp9_moe_forward_host
    # call per step (H2D of x, the forward, D2H of y on the stream), then a
    # stream synchronisation so that y is on the host
    Ke = min(K, 500)
    xh = torch.empty((n_tok, bsz, H), dtype=torch.float32).pin_memory()
    xh.copy_(xs.cpu())
    yh = torch.empty((bsz, H), dtype=torch.float32).pin_memory()
    wsh = Workspace.for_moe_host(Ls[0], bsz, dev)
    # the binding's per-step form (layer, workspace and stream marshalled
    # once per layer); the host rows are views made before the loop
    fwd = [binding.host_forward_fn(L, wsh.tensor, status, stream) for L in Ls]
    xrows = [xh[j] for j in range(n_tok)]
    for i in range(3):
        fwd[i % len(Ls)](xrows[i % n_tok], yh)
        stream.synchronize()
    if world > 1:
        dist.barrier()
    t_e = time.perf_counter()
    for i in range(Ke):
        fwd[i % len(Ls)](xrows[i % n_tok], yh)
        stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t_e)

    extra = {}
    if not args.no_extra and world == 1:
        extra = _side_runs(Ls, ws, status, dev, shape)
        extra["tiny"] = _tiny_run(dev)
        extra["dense_decode"] = _dense_decode_run(dev, _peaks()[0])
        extra["fp8_to_fp9"] = _convert_run(dev, _peaks()[0])
        extra["stack12"] = _stack_run(dev, shape)
        extra["prefill"] = _prefill_run(dev, _tensor_peak())

    if rank != 0:
        return None
    value = replica_throughput(world, bsz, K, elapsed_ms / 1e3)
    clocks = sampler.summary(t_region0, t_region1)
    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "tok/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(elapsed_ms / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded N(0,0.02) weights packed to fp9 on the GPU, N(0,1) tokens)",
        "config": _workload_config(shape, bsz, len(Ls), sum(weight_bytes) / K, world),
        "roofline": {
            "bound": "hbm",
            "kernel": "fp9::expert_kernel",
            "achieved": round(kernel_gbs, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(kernel_gbs / peak, 4),
            "traffic": _profiled_traffic() if bsz == 1 else None,
            "algorithmic_bytes_per_launch": round(sum(weight_bytes) / K),
            "kernel_us": round(mean_kern_s * 1e6, 2),
            "kernel_timing": f"CUDA events around each of {Kk} fused-kernel launches, in a second pass of the "
                             "same steps (value comes from the pass with no events between launches)",
        },
        "weight_stream_gbs_per_step": round(step_gbs, 1),
        "total_gbs_per_step": round(total_gbs, 1),
        "us_per_layer": round(elapsed_ms / K * 1e3, 2),
        "e2e": {
            "value": round(replica_throughput(world, bsz, Ke, e2e_s), 2),
            "unit": "tok/s",
            "h2d_bytes_per_step": bsz * H * 4,
            "d2h_bytes_per_step": bsz * H * 4,
            "steps": Ke,
            "api": "fp9_moe_forward_host (pinned host x and y, through binding.host_forward_fn: x copied in, "
                   "y written to host memory by the last kernel) + stream synchronise, per step",
        },
        "gpu_launches": 3 * K,
        "clocks": clocks,
        "setup_s": round(setup_s, 1),
    }
    if extra:
        out["extra"] = extra
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = _cpu_baseline(mode="layer")
    return out


def _side_runs(Ls, ws, status, dev, shape):
    """The same layers at bsz 2, 5 and 8 (the pair and verify row counts):
    weight-stream GB/s of the union of touched experts, and the fused
    kernel's (expert, token) passes per step (an MoE call plans one token
    per job; the repeated passes of an expert read its rows from L2)."""
    import torch

    from fp9_weight_expert_gb300 import Workspace, binding, synth
    res = {}
    unit = 3 * shape.inter * shape.hidden * FP9_BYTES_PER_WEIGHT
    for bsz in (2, 5, 8):
        K = 400 if bsz == 2 else 200
        xs = synth.tokens(64 * bsz, shape.hidden, synth.seed_for(3000, bsz, synth.TOKENS), dev).view(64, bsz, -1)
        y = torch.empty((bsz, shape.hidden), device=dev)
        ids = torch.empty((K, bsz, shape.topk), dtype=torch.int32, device=dev)
        w2 = Workspace.for_moe(Ls[0], bsz, dev)
        for i in range(10):
            binding.fp9_moe_forward(Ls[i % len(Ls)], xs[i % 64], y, w2.tensor, status)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(K):
            binding.fp9_moe_forward(Ls[i % len(Ls)], xs[i % 64], y, w2.tensor, status, ids[i])
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        idc = ids.cpu()
        units = sum(len(set(idc[i].flatten().tolist())) + shape.n_shared for i in range(K))
        gbs = units * unit / (ms / 1e3) / 1e9
        res[f"bsz{bsz}"] = {"tok_s": round(bsz * K / (ms / 1e3), 1), "us_per_layer": round(ms / K * 1e3, 2),
                            "weight_stream_gbs": round(gbs, 1), "mean_experts": round(units / K, 2),
                            "passes": bsz * (shape.topk + shape.n_shared), "steps": K}
        del w2
    res.update(_moe_prefill_run(Ls, status, dev, shape, (1481, 4096)))
    if int(status.item()) != 0:
        raise RuntimeError("side runs status: " + binding.status_str(int(status.item())))
    return res


def _tiny_run(dev, K=2000):
    """The tiny layer (hidden 256, 8 experts top-2, 1 shared; 1 MB of fp9,
    L2-resident, so no roofline claim): tokens/s and us per layer at bsz 1."""
    import torch

    from fp9_weight_expert_gb300 import Workspace, binding, layers, synth
    shape = synth.TINY
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    L = layers.MoELayer(shape.hidden, shape.inter, shape.n_experts, shape.n_groups, shape.topk_groups, shape.topk,
                        shape.n_shared, shape.route_scale, dev)
    kinds = (synth.ROUTED, synth.SHARED)
    L.fill(lambda b, k, m: synth.ffn_weight(shape, shape.inter, shape.hidden, synth.seed_for(8100, 0, kinds[b], k, m),
                                            dev),
           synth.normal((shape.n_experts, shape.hidden), shape.router_std, synth.seed_for(8100, 0, synth.ROUTER), dev),
           status)
    xs = synth.tokens(64, shape.hidden, synth.seed_for(8200, 0, synth.TOKENS), dev).view(64, 1, -1)
    y = torch.empty((1, shape.hidden), device=dev)
    ws = Workspace.for_moe(L, 1, dev)
    for i in range(20):
        binding.fp9_moe_forward(L, xs[i % 64], y, ws.tensor, status)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(K):
        binding.fp9_moe_forward(L, xs[i % 64], y, ws.tensor, status)
    b.record()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("tiny status: " + binding.status_str(int(status.item())))
    ms = a.elapsed_time(b) / K
    return {"tok_s": round(1.0 / (ms / 1e3), 1), "us_per_layer": round(ms * 1e3, 2), "steps": K,
            "note": "995 KB of fp9: L2-resident, launch-latency bound"}


def _dense_decode_run(dev, peak, K=400):
    """The dense FFN of the model's first layers (hidden 7168, intermediate
    18432; 445.9 MB of fp9) decoded at bsz 1 and 2 with fp9_dense_ffn; two
    FFNs alternate, so every call streams its weights from HBM."""
    import torch

    from fp9_weight_expert_gb300 import FFNBank, Workspace, binding, synth
    H, I = synth.DENSE_HIDDEN, synth.DENSE_INTER
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    fs = []
    for n in range(2):
        f = FFNBank(1, I, H, dev)
        for m in range(3):
            f.pack(0, m, synth.ffn_weight(None, I, H, synth.seed_for(8300, n, synth.DENSE, 0, m), dev), status)
        fs.append(f)
    wbytes = 3 * I * H * FP9_BYTES_PER_WEIGHT
    out = {"weight_bytes": int(wbytes)}
    for bsz in (1, 2):
        xs = synth.tokens(64 * bsz, H, synth.seed_for(8400, bsz, synth.TOKENS), dev).view(64, bsz, -1)
        y = torch.empty((bsz, H), device=dev)
        ws = Workspace.for_dense(fs[0], bsz, dev)
        for i in range(10):
            binding.fp9_dense_ffn(fs[i % 2], xs[i % 64], y, ws.tensor, status)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(K):
            binding.fp9_dense_ffn(fs[i % 2], xs[i % 64], y, ws.tensor, status)
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / K
        gbs = wbytes / (ms / 1e3) / 1e9
        out[f"bsz{bsz}"] = {"tok_s": round(bsz / (ms / 1e3), 1), "us_per_call": round(ms * 1e3, 2),
                            "weight_stream_gbs": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peak, 4),
                            "steps": K}
    if int(status.item()) != 0:
        raise RuntimeError("dense status: " + binding.status_str(int(status.item())))
    del fs
    torch.cuda.empty_cache()
    return out


def _moe_prefill_run(Ls, status, dev, shape, lengths):
    """The MoE layer over a whole prompt at once (fp9_moe_prefill) for each
    prompt length, on the resident layers in turn; with the pages' long
    prompt (1481 tokens) every expert has tokens, so each call streams all
    routed and shared experts."""
    import torch

    from fp9_weight_expert_gb300 import Workspace, binding, synth
    res = {}
    for m in lengths:
        x = synth.tokens(m, shape.hidden, synth.seed_for(3100, m, synth.TOKENS), dev)
        y = torch.empty_like(x)
        wp = Workspace.for_moe_prefill(Ls[0], m, dev)
        for name, prec in (("split", binding.FP9_PREFILL_SPLIT), ("fp16", binding.FP9_PREFILL_FP16)):
            for i in range(2):
                binding.fp9_moe_prefill(Ls[i % len(Ls)], x, y, wp.tensor, status, precision=prec)
            torch.cuda.synchronize()
            K = 8
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for i in range(K):
                binding.fp9_moe_prefill(Ls[i % len(Ls)], x, y, wp.tensor, status, precision=prec)
            b.record()
            torch.cuda.synchronize()
            ms = a.elapsed_time(b) / K
            wbytes = (shape.n_experts + shape.n_shared) * 3 * shape.inter * shape.hidden * FP9_BYTES_PER_WEIGHT
            key = f"moe_prefill_m{m}" + ("" if name == "split" else "_fp16")
            res[key] = {"us_per_layer": round(ms * 1e3, 1), "tok_s": round(m / (ms / 1e3)),
                        "weight_stream_gbs": round(wbytes / (ms / 1e3) / 1e9, 1),
                        "precision": "activations as two fp16 terms (hi + lo; the default)" if name == "split"
                        else "activations as one fp16 term (opt-in)"}
        del wp
        torch.cuda.empty_cache()
    if int(status.item()) != 0:
        raise RuntimeError("moe prefill status: " + binding.status_str(int(status.item())))
    return res


def _stack_run(dev, shape, n_layers=12, K=1000):
    """The 12-layer stack of the workload: 12 distinct resident
    DeepSeek-V3 MoE layers (153 GB) with the residual + RMSNorm between
    them, h <- h + MoE_l(RMSNorm(h)); the whole stack step is captured once
    in a CUDA graph and replayed K = 1000 times (the workload's steady
    state over 1000 steps). Tokens/s through all 12 layers, for the layer
    step with the glue folded in (fp9_moe_forward_residual: three kernels a
    layer) and, under "glue", for the separate glue kernel between
    fp9_moe_forward calls (four kernels a layer)."""
    import torch

    from fp9_weight_expert_gb300 import Workspace, binding, layers, synth
    H, I = shape.hidden, shape.inter
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    Ls = []
    for l in range(n_layers):
        L = layers.MoELayer(H, I, shape.n_experts, shape.n_groups, shape.topk_groups, shape.topk,
                            shape.n_shared, shape.route_scale, dev)
        kinds = (synth.ROUTED, synth.SHARED)
        L.fill(lambda b, k, m: synth.ffn_weight(shape, I, H, synth.seed_for(7000, l, kinds[b], k, m), dev),
               synth.normal((shape.n_experts, H), shape.router_std, synth.seed_for(7000, l, synth.ROUTER), dev),
               status)
        Ls.append(L)
    out = {"layers": n_layers, "resident_gb": round(n_layers * 3 * H * I * (shape.n_experts + shape.n_shared)
                                                    * FP9_BYTES_PER_WEIGHT / 1e9, 1)}
    # bsz 2: an MTP pair (confirmed + draft token) in lockstep; bsz 5: a
    # speculative verify block of 5 rows
    for mode, bsz in (("residual", 1), ("residual", 2), ("residual", 5), ("glue", 1), ("glue", 2), ("glue", 5)):
        h0 = synth.tokens(bsz, H, synth.seed_for(7100, bsz, synth.TOKENS), dev) * 2.0
        h = h0.clone()
        x = torch.empty_like(h)
        y = torch.empty_like(h)
        ss = torch.empty((bsz, H // 16), dtype=torch.float32, device=dev)
        ids = torch.empty((n_layers, bsz, shape.topk), dtype=torch.int32, device=dev)
        ws = Workspace.for_moe(Ls[0], bsz, dev)

        def step():
            binding.fp9_residual_rmsnorm(h, None, x)
            for l, L in enumerate(Ls):
                if mode == "residual":
                    # the next layer's router weights are read into L2 meanwhile
                    # (after the last layer: the first one, the next replay's)
                    binding.fp9_moe_forward_residual(L, x if l == 0 else None, h, ss, ws.tensor, status, ids[l],
                                                     next_layer=Ls[(l + 1) % len(Ls)])
                else:
                    binding.fp9_moe_forward(L, x, y, ws.tensor, status, ids[l])
                    binding.fp9_residual_rmsnorm(h, y, x)

        step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(K):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        if int(status.item()) != 0:
            raise RuntimeError("stack status: " + binding.status_str(int(status.item())))
        ms = a.elapsed_time(b) / K
        idc = ids.cpu()
        experts = sum(len(set(idc[l].flatten().tolist())) + shape.n_shared for l in range(n_layers))
        wbytes = experts * 3 * I * H * FP9_BYTES_PER_WEIGHT
        rec = {"tok_s": round(bsz / (ms / 1e3), 1), "us_per_stack_step": round(ms * 1e3, 1),
               "us_per_layer": round(ms * 1e3 / n_layers, 2),
               "weight_stream_gbs": round(wbytes / (ms / 1e3) / 1e9, 1),
               "experts_streamed": experts, "steps": K}
        if mode == "residual":
            out[f"bsz{bsz}"] = rec
        else:
            out.setdefault("glue", {})[f"bsz{bsz}"] = rec
    del Ls
    torch.cuda.empty_cache()
    return out


def _convert_run(dev, peak):
    """fp9_from_fp8 on 24 DeepSeek-V3 expert matrices (fp8 e4m3 + 128x128
    scales -> fp9 planes): HBM GB/s of the bytes it must move (1 B read and
    1.125 B written per weight, plus the scales). The input is made like a
    block-scaled checkpoint (torch's e4m3 conversion makes the bytes)."""
    import torch

    from fp9_weight_expert_gb300 import binding
    n, rows, cols = 24, 2048, 7168
    # checkpoint-like input: N(0, 0.02) weights quantised to e4m3 with the
    # scale of each 128x128 block = its largest magnitude / 448
    g = torch.Generator(device=dev)
    g.manual_seed(4242)
    w8 = torch.empty((n * rows, cols), dtype=torch.uint8, device=dev)
    scale = torch.empty((n * rows // 128, cols // 128), dtype=torch.float32, device=dev)
    for i in range(n):
        w = torch.randn((rows, cols), generator=g, device=dev) * 0.02
        blocks = w.view(rows // 128, 128, cols // 128, 128)
        sc = blocks.abs().amax(dim=(1, 3)) / 448.0
        scale[i * rows // 128:(i + 1) * rows // 128] = sc
        q = (blocks / sc[:, None, :, None]).to(torch.float8_e4m3fn)
        w8[i * rows:(i + 1) * rows] = q.view(rows, cols).view(torch.uint8)
    body = torch.empty((n * rows, cols), dtype=torch.uint8, device=dev)
    sign = torch.empty((n * rows, cols // 8), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(3):
        binding.fp9_from_fp8(w8, scale, body, sign, status)
    torch.cuda.synchronize()
    K = 20
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(K):
        binding.fp9_from_fp8(w8, scale, body, sign, status)
    b.record()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("fp9_from_fp8 status: " + binding.status_str(int(status.item())))
    us = a.elapsed_time(b) / K * 1e3
    weights = n * rows * cols
    nbytes = weights * (1 + 1.125) + scale.numel() * 4
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"weights_per_call": weights, "us_per_call": round(us, 1), "bytes_per_call": int(nbytes),
            "gbs": round(gbs, 1), "peak": peak, "frac": round(gbs / peak, 4), "bound": "hbm",
            "inputs_vs_l2": "752 MB per call, larger than L2"}


def _prefill_run(dev, peaks):
    """fp9_ffn_prefill (the FFN over many prompt tokens on the tensor cores)
    for the pages' long prompt (1481 tokens) and a 4096-token one, through
    the dense FFN (7168 / 18432) and through DeepSeek-V3 experts (7168 /
    2048, 8 experts rotated so their 396 MB of weights exceed L2): tensor
    TFLOP/s of 2 * m * 3 * hidden * inter flops against the measured dense
    bf16 peak (fp16 runs at the bf16 rate)."""
    import torch

    from fp9_weight_expert_gb300 import FFNBank, Workspace, binding, synth
    peak, peak_src = peaks
    out = {"peak_source": peak_src}
    for name, n, H, I in (("dense_7168x18432", 1, 7168, 18432), ("expert_7168x2048", 8, 7168, 2048)):
        f = FFNBank(n, I, H, dev)
        for k in range(n):
            for m in range(3):
                f.pack(k, m, synth.ffn_weight(None, I, H, synth.seed_for(17, 0, synth.DENSE, k, m), dev))
        for m in (1481, 4096):
            x = synth.tokens(m, H, 5, dev)
            y = torch.empty_like(x)
            ws = Workspace.for_prefill(f, m, dev).tensor
            status = torch.zeros(1, dtype=torch.int32, device=dev)
            for pname, prec in (("split", binding.FP9_PREFILL_SPLIT), ("fp16", binding.FP9_PREFILL_FP16)):
                for i in range(3):
                    binding.fp9_ffn_prefill(f, x, y, ws, i % n, status, precision=prec)
                torch.cuda.synchronize()
                K = 20
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                for i in range(K):
                    binding.fp9_ffn_prefill(f, x, y, ws, i % n, status, precision=prec)
                b.record()
                torch.cuda.synchronize()
                if int(status.item()) != 0:
                    raise RuntimeError("fp9_ffn_prefill status: " + binding.status_str(int(status.item())))
                us = a.elapsed_time(b) / K * 1e3
                # useful flops of the FFN; the default precision issues twice
                # the MMAs (each weight meets the hi and the lo term)
                tf = 2.0 * m * 3 * H * I / (us * 1e-6) / 1e12
                key = f"{name}_m{m}" + ("" if pname == "split" else "_fp16")
                out[key] = {"us_per_call": round(us, 1), "tflops": round(tf, 1),
                            "tok_per_s": round(m / (us * 1e-6)), "peak_tflops": peak,
                            "frac": round(tf / peak, 4), "bound": "tensor",
                            "mma_tflops": round(tf * (2 if pname == "split" else 1), 1),
                            "dtype": "fp16 x fp9->fp16, activations as hi + lo fp16 terms" if pname == "split"
                            else "fp16 x fp9->fp16, one fp16 term per activation"}
        del f
        torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------- CPU oracle
#
# The oracle (oracle/, float64 numpy) timed on the host cores as a reported
# baseline. Each process runs numpy with one BLAS thread; "all cores" runs
# one worker process per expert FFN of the layer (the oracle's own
# dense_ffn on that expert's planes), so the FFNs of a layer run side by
# side, as many at once as there are workers.

def _cpu_baseline(mode: str, steps: int = 0, warmup: int = 0):
    """Runs the oracle timing in a fresh process (no CUDA, one BLAS thread
    per process) and returns its record."""
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[v] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-sample", f"{mode}:{steps}:{warmup}"]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=1800)
    if r.returncode != 0:
        return {"error": (r.stderr or r.stdout)[-400:]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def _expert_planes(kind: int, k: int):
    """The oracle's packed planes of one DeepSeek-V3 expert FFN, from the
    seeded fp32 draws."""
    import oracle as O
    from fp9_weight_expert_gb300 import synth
    shape = synth.DSV3
    out = []
    for m in range(3):
        body, sign, _ = O.fp9_pack(synth.ffn_weight(shape, shape.inter, shape.hidden,
                                                    synth.seed_for(5000, 0, kind, k, m)).numpy())
        out += [body, sign]
    return tuple(out)


def _expert_worker(conn, kind: int, k: int):
    """Child process: packs one expert once (not timed), then answers each
    token block x with the oracle's dense_ffn(x, planes), or ("parts", x)
    with the seconds of its two steps (decode the planes, run the FFN on
    x), until it gets None."""
    import oracle as O
    planes = _expert_planes(kind, k)
    conn.send("ready")
    while True:
        msg = conn.recv()
        if msg is None:
            break
        if isinstance(msg, tuple):
            t0 = time.perf_counter()
            dec = tuple(O.fp9_decode(planes[2 * i], planes[2 * i + 1]) for i in range(3))
            t1 = time.perf_counter()
            O.ffn(msg[1], *dec)
            conn.send((t1 - t0, time.perf_counter() - t1))
        else:
            conn.send(O.dense_ffn(msg, planes))
    conn.close()


class _ExpertPool:
    """One worker process per expert FFN (spawned: no state is shared)."""

    def __init__(self, experts):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.conns, self.procs = [], []
        for kind, k in experts:
            a, b = ctx.Pipe()
            p = ctx.Process(target=_expert_worker, args=(b, kind, k), daemon=True)
            p.start()
            self.conns.append(a)
            self.procs.append(p)
        for c in self.conns:
            assert c.recv() == "ready"

    def run(self, x):
        """Every worker's FFN of x, all at once."""
        for c in self.conns:
            c.send(x)
        return [c.recv() for c in self.conns]

    def run_one_at_a_time(self, x):
        """The same FFNs, one worker at a time (one core busy)."""
        out = []
        for c in self.conns:
            c.send(x)
            out.append(c.recv())
        return out

    def parts(self, x):
        """(decode seconds, FFN seconds) of worker 0 alone."""
        self.conns[0].send(("parts", x))
        return self.conns[0].recv()

    def close(self):
        for c in self.conns:
            c.send(None)
        for p in self.procs:
            p.join(timeout=30)


def _oracle_layer_setup():
    """One DeepSeek-V3 MoE layer at bsz 1: the router weight, one
    token, its routing (oracle) and the experts it needs."""
    import oracle as O
    from fp9_weight_expert_gb300 import synth
    shape = synth.DSV3
    wr = synth.normal((shape.n_experts, shape.hidden), shape.router_std, synth.seed_for(5000, 0, synth.ROUTER)).numpy()
    x = synth.tokens(1, shape.hidden, synth.seed_for(5000, 0, synth.TOKENS)).numpy()
    ids, w = O.route(x, wr, shape.n_groups, shape.topk_groups, shape.topk, shape.route_scale)
    experts = [(synth.ROUTED, int(e)) for e in ids[0]] + [(synth.SHARED, 0)]
    return shape, wr, x, ids, w, experts


def _layer_all_cores(pool, x, wr, shape, w, one_core=False):
    """One layer step on the pool: the oracle's routing, then the routed and
    shared expert FFNs side by side (or one at a time), added as the
    oracle's moe() adds them."""
    import oracle as O
    O.route(x, wr, shape.n_groups, shape.topk_groups, shape.topk, shape.route_scale)
    ys = pool.run_one_at_a_time(x) if one_core else pool.run(x)
    y = sum(float(wk) * yk for wk, yk in zip(w[0], ys[:-1])) + ys[-1]
    return y


def _cpu_sample_worker(spec: str):
    """Oracle timing, CPU only (see _cpu_baseline).

    mode 'layer' (the bench's cpu_baseline): the DeepSeek-V3 layer at bsz 1
    on one core (the oracle's moe() on one token, two passes) and on all
    cores (the layer's 9 expert FFNs on 9 worker processes); then the tiny
    layer (measured), the layer at bsz 2, 5 and 8 and the dense FFN (from the
    measured per-expert times, scaled to each workload's expert count).
    mode 'ref' (the reference arm): `steps` timed steps of that layer on
    all cores after `warmup` untimed ones.
    """
    import numpy as np

    import oracle as O
    from fp9_weight_expert_gb300 import synth

    mode, steps, warmup = spec.split(":")
    steps, warmup = int(steps), int(warmup)
    ncores = len(os.sched_getaffinity(0))
    shape, wr, x, ids, w, experts = _oracle_layer_setup()
    t0 = time.perf_counter()
    pool = _ExpertPool(experts)
    setup_s = time.perf_counter() - t0
    workers = len(experts)
    used = min(workers, ncores)
    try:
        if mode == "ref":
            for _ in range(warmup):
                _layer_all_cores(pool, x, wr, shape, w)
            t0 = time.perf_counter()
            for _ in range(max(steps, 1)):
                y = _layer_all_cores(pool, x, wr, shape, w)
            dt = (time.perf_counter() - t0) / max(steps, 1)
            assert np.isfinite(y).all()
            print(json.dumps({
                "value": round(1.0 / dt, 5), "unit": "tok/s", "cores": used, "host_cores": ncores,
                "kind": "oracle", "seconds_per_step": round(dt, 4), "setup_s": round(setup_s, 1),
                "sample": f"per step one token through one DeepSeek-V3 MoE layer: the oracle's routing, then its "
                          f"8 routed + 1 shared expert FFNs (fp64 numpy, one BLAS thread each) on {workers} worker "
                          f"processes side by side ({used} of {ncores} host cores busy), added as moe() adds them"}))
            return
        # all cores: the DeepSeek-V3 layer at bsz 1, two timed passes after one untimed
        _layer_all_cores(pool, x, wr, shape, w)
        t0 = time.perf_counter()
        for _ in range(2):
            y_all = _layer_all_cores(pool, x, wr, shape, w)
        t_all = (time.perf_counter() - t0) / 2
        # one core: the same layer with its FFNs one after the other
        t0 = time.perf_counter()
        y_one = _layer_all_cores(pool, x, wr, shape, w, one_core=True)
        t_one = time.perf_counter() - t0
        assert np.array_equal(y_one, y_all)
        t_dec, t_tok = pool.parts(x)
    finally:
        pool.close()
    xs8 = synth.tokens(8, shape.hidden, synth.seed_for(5000, 1, synth.TOKENS)).numpy()
    t0 = time.perf_counter()
    ids8, _ = O.route(xs8, wr, shape.n_groups, shape.topk_groups, shape.topk, shape.route_scale)
    t_route8 = time.perf_counter() - t0
    configs = {}
    # the tiny layer (hidden 256, 8 experts), measured directly (one core)
    tiny = synth.TINY

    def tiny_planes(kind, k):
        out = []
        for m in range(3):
            b, sg, _ = O.fp9_pack(synth.ffn_weight(tiny, tiny.inter, tiny.hidden,
                                                   synth.seed_for(5100, 0, kind, k, m)).numpy())
            out += [b, sg]
        return tuple(out)
    tcache = {k: tiny_planes(synth.ROUTED, k) for k in range(tiny.n_experts)}
    tsh = [tiny_planes(synth.SHARED, 0)]
    twr = synth.normal((tiny.n_experts, tiny.hidden), tiny.router_std, synth.seed_for(5100, 0, synth.ROUTER)).numpy()
    tx = synth.tokens(1, tiny.hidden, synth.seed_for(5100, 0, synth.TOKENS)).numpy()
    t0 = time.perf_counter()
    n_tiny = 50
    for _ in range(n_tiny):
        O.moe(tx, twr, lambda e: tcache[e], tsh, tiny.n_groups, tiny.topk_groups, tiny.topk, tiny.route_scale)
    t_tiny = (time.perf_counter() - t0) / n_tiny
    configs["tiny_bsz1"] = {"tok_s_1core": round(1.0 / t_tiny, 2), "measured": "directly (moe(), 50 passes)"}
    configs["dsv3_bsz1"] = {"tok_s_1core": round(1.0 / t_one, 5), "tok_s_all_cores": round(1.0 / t_all, 5),
                            "measured": "directly"}
    # the DeepSeek-V3 layer at bsz 2, 5, 8 (tokens drawn independently); the oracle decodes
    # each distinct expert once and runs one FFN per (token, expert) pair
    for bsz in (2, 5, 8):
        U = len(set(ids8[:bsz].flatten().tolist())) + shape.n_shared
        pairs = bsz * shape.topk + bsz
        t1 = t_route8 * bsz / 8 + U * t_dec + pairs * t_tok
        rounds = -(-U // ncores)
        ta = t_route8 * bsz / 8 + rounds * t_all
        configs[f"dsv3_bsz{bsz}"] = {"experts": U, "tok_s_1core": round(bsz / t1, 5),
                                     "tok_s_all_cores": round(bsz / ta, 5),
                                     "measured": "scaled from the per-expert times (decode once per expert, one "
                                                 "FFN per token and expert; all cores: one expert per core, "
                                                 "rounds of the measured all-core layer time)"}
    # the dense FFN 7168 / 18432 (18432 = 9 x 2048 rows) costs 9 expert FFNs
    for bsz in (1, 2):
        t1 = 9 * t_dec + 9 * bsz * t_tok
        configs[f"dense_bsz{bsz}"] = {"tok_s_1core": round(bsz / t1, 5),
                                      "tok_s_all_cores": round(bsz / (t_all + (bsz - 1) * t_tok), 5),
                                      "measured": "scaled: 9 x one expert's decode + FFN (one core); all cores: "
                                                  "its 9 row blocks of 2048 side by side, as the 9 expert FFNs "
                                                  "of the bsz-1 layer, plus one more token's FFN per extra token"}
    print(json.dumps({
        "value": round(1.0 / t_all, 5), "unit": "tok/s", "cores": used, "host_cores": ncores, "kind": "oracle",
        "seconds_all_cores": round(t_all, 4), "one_core": {"value": round(1.0 / t_one, 5), "cores": 1,
                                                           "seconds": round(t_one, 4)},
        "per_expert_s": {"decode": round(t_dec, 4), "ffn_one_token": round(t_tok, 4)},
        "configs": configs,
        "sample": f"one token through one DeepSeek-V3 MoE layer (oracle routing over 256 experts, 8 routed + 1 "
                  f"shared expert FFN, fp64 numpy, one BLAS thread per process): all cores = the 9 expert FFNs "
                  f"on {workers} worker processes side by side ({used} of {ncores} host cores busy, two passes); "
                  f"one core = the same FFNs one at a time (one pass)"}))


def _workload_config(shape, bsz, n_layers, bytes_per_step, world):
    """The bench line's config (both arms print the same one)."""
    return {
        "workload": f"one DeepSeek-V3 MoE layer, bsz {bsz}: hidden 7168, {shape.n_experts} routed experts "
                    f"(8 groups x {shape.n_experts // 8}, top-4 groups, top-8) + 1 shared, "
                    "intermediate 2048, fp9 weights",
        "bsz": bsz,
        "resident_layers": n_layers,
        "l2": f"inputs larger than L2: {n_layers} resident layers (12.7 GB each) rotate, each step streams "
              f"{bytes_per_step / 1e6:.1f} MB of fp9 weights",
        "parallelism": "replicas" if world > 1 else "single GPU",
    }


def _reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    from fp9_weight_expert_gb300 import synth
    rec = _cpu_baseline(mode="ref", steps=args.steps, warmup=args.warmup)
    if "error" in rec:
        return {"impl": "reference", "unavailable": "oracle run failed: " + rec["error"][-200:]}
    v = rec["value"]
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": v,
        "unit": "tok/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(rec["seconds_per_step"] * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        # the native arm's workload at bsz 1 (9 experts of 49.5 MB a step)
        "config": _workload_config(synth.DSV3, 1, args.layers,
                                   9 * 3 * 2048 * 7168 * FP9_BYTES_PER_WEIGHT, int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": rec,
        "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = _args()
    if args.cpu_sample:
        _cpu_sample_worker(args.cpu_sample)
        return
    out = _reference(args) if args.impl == "reference" else _native(args)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()

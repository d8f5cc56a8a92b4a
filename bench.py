"""Benchmark of the multi-scale deformable attention hot path on B300.

One step = one forward and one backward pass (every kernel of the path) over
the Deformable DETR encoder workload (bs=2, 4-level 100x167 pyramid, 22223
queries, 8 heads, head_dim 32, 4 points, fp32), inputs resident in HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl native|reference] [--no-cpu-baseline] [--no-e2e]

Prints ONE JSON line (rank 0).  Timing: CUDA events on the launching stream
around each kernel call of every timed step; L2 is flushed (a write of twice
the L2 size) before every step, outside the events.  Under torchrun each rank
runs its own batch (weak scaling, no data-path collective); the step time is
the max over ranks.  ``--impl reference`` times the fp64 CPU oracle on the
host cores instead (bounded sample per step).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from scale_deformable_attention_05_b300 import inputs as gen  # noqa: E402

METRIC = "MSDeformAttn fwd/bwd sampled points/s (1×B300); achieved GB/s vs HBM roofline"
FALLBACK_HBM_GBS = 6400.0
KERNEL_SOURCES = ["msda_device.cuh", "msda_forward.cuh", "msda_backward.cuh", "msda_kernels.cu"]


# --------------------------------------------------------------------- utils
def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, burst copy)"
    return FALLBACK_HBM_GBS, "fallback 6.4 TB/s"


def _kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "scale_deformable_attention_05_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _profiled_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches the sources."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")
    if not os.path.exists(path):
        return None
    rec = {}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if ":" in line:
            k, v = line.split(":", 1)
            rec[k.strip()] = v.strip()
    if rec.get("source_hash") != _kernel_source_hash():
        return None
    v = rec.get(f"{kernel}_dram_bytes_per_launch")
    return float(v) if v else None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------- reference arm
def _oracle_step(inp, wl, threads=0):
    import oracle
    args = (inp["value"], inp["spatial_shapes"], inp["level_start_index"],
            inp["sampling_locations"], inp["attention_weights"])
    oracle.forward(*args, threads=threads)
    oracle.backward(*args, inp["grad_output"], threads=threads)


def _sample_inputs(inp, wl, q_count):
    """The first q_count queries of the workload (all batches, heads, levels, points)."""
    s = dict(inp)
    for k in ("sampling_locations", "attention_weights", "grad_output"):
        s[k] = np.ascontiguousarray(inp[k][:, :q_count])
    return s


def cpu_baseline(wl, inp, budget_s=12.0, min_reps=1):
    """Time the oracle (forward + backward) on the host cores; bounded sample."""
    import oracle
    threads = oracle.max_threads()
    reps, t0 = 0, time.perf_counter()
    while True:
        _oracle_step(inp, wl)
        reps += 1
        el = time.perf_counter() - t0
        if reps >= min_reps and (el >= budget_s or el / reps * (reps + 1) > 2.5 * budget_s):
            break
    # the same oracle on one core, on the first queries only (a few seconds):
    # at least 200k samples so the per-call setup does not dominate
    per_q = wl.bs * wl.num_heads * wl.num_levels * wl.num_points
    q1 = min(wl.num_queries, max(wl.num_queries // 16, -(-200_000 // per_q)))
    sample1 = _sample_inputs(inp, wl, q1)
    t1 = time.perf_counter()
    _oracle_step(sample1, wl, threads=1)
    el1 = time.perf_counter() - t1
    pts1 = wl.bs * q1 * wl.num_heads * wl.num_levels * wl.num_points
    return {"value": wl.points * reps / el, "unit": "points/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{reps} full forward+backward pass(es) of the '{wl.name}' workload "
                      f"({wl.points} samples each), fp64 C oracle, {el:.1f} s",
            "single_core": {"value": pts1 / el1, "unit": "points/s", "cores": 1,
                            "sample": f"first {q1} of {wl.num_queries} queries ({pts1} samples), "
                                      f"forward + backward, {el1:.1f} s"}}


def run_layer(args, wl):
    """The MSDeformAttn layer (module.MSDeformAttn: four tensor-core projections
    around the fused entry points) forward + backward through autograd on the workload's
    shape: seeded random query / input features, the workload's fused reference
    points, the layer's initial parameters.  Each step is timed with CUDA events
    as the layer runs (Python and autograd included) and, unless --no-graph, as
    replays of one CUDA graph of the whole step (the line's value); L2 flushed
    before each."""
    import torch
    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    from scale_deformable_attention_05_b300.module import MSDeformAttn
    if wl.dtype not in ("f32", "bf16", "f16"):
        raise SystemExit("--path layer runs fp32, bf16 or fp16 workloads")
    torch.backends.cuda.matmul.allow_tf32 = False
    dev = torch.device("cuda", local)
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[wl.dtype]
    wl_r = rank_workload(wl, rank)
    C = wl.num_heads * wl.head_dim
    torch.manual_seed(wl_r.seed)
    layer = MSDeformAttn(C, wl.num_levels, wl.num_heads, wl.num_points).to(dev).to(tdt)
    fin = gen.make_fused_inputs(wl_r, 2)
    gcpu = torch.Generator().manual_seed(wl_r.seed)
    q = torch.randn(wl.bs, wl.num_queries, C, generator=gcpu).to(dev, tdt).requires_grad_()
    x = torch.randn(wl.bs, wl.num_keys, C, generator=gcpu).to(dev, tdt).requires_grad_()
    go = torch.randn(wl.bs, wl.num_queries, C, generator=gcpu).to(dev, tdt)
    ref = torch.from_numpy(fin["reference_points"]).to(dev, tdt)
    shapes = torch.from_numpy(fin["spatial_shapes"]).to(dev)
    lsi = torch.from_numpy(fin["level_start_index"]).to(dev)
    mask = (torch.from_numpy(gen.padding_mask(wl_r)).to(dev) if args.padding_mask else None)
    flush = torch.empty(max(2 * torch.cuda.get_device_properties(dev).L2_cache_size, 64 << 20) // 4,
                        dtype=torch.float32, device=dev)

    def step():
        for prm in layer.parameters():
            prm.grad = None
        q.grad = x.grad = None
        layer(q, ref, x, shapes, lsi, mask).backward(go)

    def timed_steps(n, run=step, sampler=None):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        torch.cuda.synchronize()
        if sampler:
            sampler.start()
        for e0, e1 in evs:
            flush.zero_()
            e0.record()
            run()
            e1.record()
        torch.cuda.synchronize()
        clocks = sampler.stop() if sampler else None
        return [e0.elapsed_time(e1) for e0, e1 in evs], clocks

    def capture():
        """The whole forward + backward as one CUDA graph (warmed up on a side
        stream first, gradients unset so that the captured backward writes them
        into the graph's own memory); replays rewrite the same gradient tensors."""
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(3):
                step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        for prm in layer.parameters():
            prm.grad = None
        q.grad = x.grad = None
        with torch.cuda.graph(graph):
            layer(q, ref, x, shapes, lsi, mask).backward(go)
        torch.cuda.synchronize()
        return graph

    use_graph = not args.no_graph

    def measure(tensor_cores, warmup, sampler=None):
        layer.tensor_core_projections = tensor_cores
        for _ in range(warmup):
            flush.zero_()
            step()
        eager, clk = timed_steps(args.steps, sampler=None if use_graph else sampler)
        if not use_graph:
            return eager, None, clk
        graph = capture()
        for _ in range(2):
            graph.replay()
        replayed, clk = timed_steps(args.steps, run=graph.replay, sampler=sampler)
        del graph
        return eager, replayed, clk

    # the same layer with torch.nn.Linear (cuBLAS) projections first, for
    # comparison; it warms up twice as long as asked (first-use costs of the
    # allocator and of each kernel module)
    compare = None
    if not args.no_projection_compare:
        cb_eager, cb_graph, _ = measure(False, 2 * args.warmup)
        compare = {"cublas_projections_ms": statistics.median(cb_graph or cb_eager),
                   "cublas_projections_eager_ms": statistics.median(cb_eager),
                   "gemm": None}
    if dist:
        dist.barrier()
    sampler = ClockSampler(local)
    tc_eager, tc_graph, clocks = measure(True, args.warmup, sampler)
    if dist:
        dist.barrier()
    if compare is not None:
        compare["gemm"] = _projection_gemm(layer.output_proj, wl.bs * wl.num_keys, dev, flush)
    ms = tc_graph or tc_eager
    ms_step = max_over_ranks(sum(ms) / len(ms), dist, dev)
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0
    cfg = _config(wl, args)
    cfg["entry_points"] = ("module.MSDeformAttn: value / offset / weight / output projections "
                           + ("(msda_linear on the tensor cores forward and for the input "
                              "gradients; weight gradients with torch (cuBLAS), bias gradients "
                              "with msda_linear_bias_grad)"
                              if wl.dtype != "f32" else
                              "(msda_linear_f32, three TF32 products on the tensor cores, "
                              "forward and for the input gradients; weight and bias "
                              "gradients with msda_linear_wgrad_f32)")
                           + " around msda_forward_fused / msda_backward_fused, autograd")
    cfg["launch"] = ("eager through autograd (Python and autograd inside the events)"
                     if not use_graph else
                     "forward + backward through autograd captured once as one CUDA graph and "
                     "replayed (the eager step is timed beside it)")
    line = {
        "metric": METRIC, "value": job_rate(wl.points, ws, ms_step), "unit": "points/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (random query / input features, initial layer parameters)",
        "config": cfg,
        "passes": {"layer": {"ms": sum(ms) / len(ms), "median_ms": statistics.median(ms),
                             "min_ms": min(ms)},
                   "layer_eager": {"ms": sum(tc_eager) / len(tc_eager),
                                   "median_ms": statistics.median(tc_eager)}},
        "projections": compare,
        "roofline": None, "clocks": clocks, "e2e": None,
        # the library's kernels per step: fused forward; grad_value (or fp32 workspace)
        # zero-fill + fused backward (+ the half-precision finalize); four projections
        # forward and four input gradients, one launch each in bf16 / fp16 and two (the
        # split of w and the GEMM) in fp32; four parameter gradients: in fp32 two
        # zero-fills and the weight-gradient kernel each, in bf16 / fp16 a zero-fill
        # and the bias column sum each
        "gpu_launches": (3 + 8 * 2 + 4 * 3 if wl.dtype == "f32" else 4 + 8 + 4 * 2) * args.steps,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def _projection_gemm(linear, rows, dev, flush, reps=20):
    """One d_model x d_model projection of `rows` tokens in the layer's dtype:
    msda_linear / msda_linear_f32 (tcgen05) against torch's F.linear (cuBLAS),
    and in fp32 the parameter gradients (msda_linear_wgrad_f32 against torch);
    CUDA events around each call, enqueued while the device sleeps, L2 flushed
    before each call."""
    import torch
    import torch.nn.functional as F
    from scale_deformable_attention_05_b300 import binding as B
    g = torch.Generator(device=dev).manual_seed(11)
    dt = linear.weight.dtype
    xg = torch.randn(rows, linear.in_features, generator=g, device=dev).to(dt)
    w, b = linear.weight.detach(), linear.bias.detach()
    bf = b.float()
    out = torch.empty(rows, linear.out_features, dtype=dt, device=dev)
    ws = torch.empty(B.msda_linear_workspace_bytes(rows, linear.in_features, linear.out_features),
                     dtype=torch.uint8, device=dev)

    def timed(fn):
        # the device sleeps while the host enqueues every rep, so that the host's
        # marshalling (15-20 us a call, more on a loaded host) stays outside the events
        for _ in range(3):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        torch.cuda.synchronize()
        torch.cuda._sleep(20_000_000)           # ~10 ms at the B300's clocks
        for e0, e1 in evs:
            flush.zero_()
            e0.record()
            fn()
            e1.record()
        torch.cuda.synchronize()
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)

    if dt != torch.float32:
        tc = timed(lambda: B.msda_linear(xg, w, bf, out=out))
    else:
        tc = timed(lambda: B.msda_linear_f32(xg, w, b, out=out, workspace=ws))
    cb = timed(lambda: F.linear(xg, w, b))
    flops = 2.0 * rows * linear.in_features * linear.out_features
    nbytes = float(xg.element_size()) * rows * (linear.in_features + linear.out_features)
    res = {"rows": rows, "in_features": linear.in_features,
           "out_features": linear.out_features,
           "tcgen05_us": tc * 1e3, "cublas_us": cb * 1e3,
           "tcgen05_tflops": flops / tc / 1e9, "tcgen05_gbs": nbytes / tc / 1e6}
    if dt == torch.float32:
        # the parameter gradients of the same projection: msda_linear_wgrad_f32
        # against torch's grad_y^T x and column sum (cuBLAS fp32 and a reduction)
        gy = torch.randn(rows, linear.out_features, generator=g, device=dev)
        gw = torch.empty_like(w)
        gb = torch.empty_like(b)
        wg = timed(lambda: B.msda_linear_wgrad_f32(gy, xg, grad_w=gw, grad_b=gb))
        wg_torch = timed(lambda: (gy.t() @ xg, gy.sum(0)))
        res.update(wgrad_tcgen05_us=wg * 1e3, wgrad_torch_us=wg_torch * 1e3)
    return res


def touched_roofline(wl, inp, passes, hbm_gbs):
    """Secondary roofline: the value (and grad_value) bytes counted over the
    distinct (b, key, m) rows the workload's samples touch with a non-zero
    weight, as counted by the oracle, instead of the whole tensor.  Matters
    where few rows are read (the decoder's 300 queries)."""
    import oracle
    rows = oracle.touched_rows(inp["spatial_shapes"], inp["level_start_index"],
                               inp["sampling_locations"], inp["attention_weights"],
                               wl.bs, wl.num_keys, wl.num_heads)
    row_bytes = wl.head_dim * wl.elem_bytes
    value = wl.bs * wl.num_keys * wl.num_heads * row_bytes
    out = {"label": "secondary: value and grad_value bytes over touched rows only",
           "touched_rows": rows, "of_rows": wl.bs * wl.num_keys * wl.num_heads}
    for name, n_value in (("forward", 1), ("backward", 2)):
        b = passes[name]["compulsory_bytes"] - n_value * (value - rows * row_bytes)
        gbs = b / (passes[name]["ms"] / 1e3) / 1e9
        out[name] = {"bytes": b, "gbs": gbs, "frac": gbs / hbm_gbs}
    return out


def run_reference(args, wl):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    import oracle
    inp = gen.make_inputs(wl)
    threads = oracle.max_threads()
    # per step: the first q queries, sized so one step takes about a second
    t0 = time.perf_counter()
    probe_q = max(1, wl.num_queries // 16)
    _oracle_step(_sample_inputs(inp, wl, probe_q), wl)
    per_q = (time.perf_counter() - t0) / probe_q
    q = int(max(1, min(wl.num_queries, 1.0 / max(per_q, 1e-9))))
    sample = _sample_inputs(inp, wl, q)
    pts = wl.bs * q * wl.num_heads * wl.num_levels * wl.num_points
    for _ in range(args.warmup):
        _oracle_step(sample, wl)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(sample, wl)
    el = time.perf_counter() - t0
    value = pts * args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "points/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(wl, args),
        "cpu_baseline": {"value": value, "unit": "points/s", "cores": threads, "kind": "oracle",
                         "sample": f"first {q} of {wl.num_queries} queries per step "
                                   f"({pts} samples), forward + backward"},
        "e2e": {"value": value, "unit": "points/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _config(wl, args):
    return {"workload": wl.name, "bs": wl.bs, "num_queries": wl.num_queries,
            "spatial_shapes": [list(s) for s in wl.spatial_shapes], "num_keys": wl.num_keys,
            "num_heads": wl.num_heads, "head_dim": wl.head_dim, "num_levels": wl.num_levels,
            "num_points": wl.num_points, "io_dtype": wl.dtype,
            "passes": "forward+backward",
            "entry_points": (f"msda_forward_fused / msda_backward_fused "
                             f"({getattr(args, 'ref_dim', 2)}-d reference points, offsets, logits)"
                             if getattr(args, "path", "plain") == "fused"
                             else "msda_forward / msda_backward"),
            "padding_mask": ("per-image top-left valid region, U[0.6, 1] of each side, image 0 "
                             "unpadded" if getattr(args, "padding_mask", False) else None),
            "launch": ("Python binding per pass" if getattr(args, "no_graph", False) else
                       "each pass captured once as a CUDA graph and replayed"),
            "l2": "flushed before every step (write of 2x L2 size, outside the timed events)",
            "parallelism": f"replicas x{args.gpus} (each rank its own batch)"}


# ------------------------------------------------------------ replica logic
def rank_workload(wl, rank):
    """The batch rank `rank` draws: every replica its own seeded inputs (weak scaling)."""
    return wl.with_(seed=wl.seed + 7919 * rank)


def max_over_ranks(x, dist=None, device=None):
    """Max of a per-rank float over all ranks (the job's time is its slowest rank)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world_size, ms):
    """Units all ranks processed per second, over the max-over-ranks time in ms."""
    return units_per_rank * world_size / (ms / 1e3)


def _e2e_pipelined(B, args, wl, fused, names, host, d, shapes, lsi, results, workspace, stream,
                   dev, dist, world):
    """The step end to end through the public API with host buffers: every step
    copies its inputs from pinned host memory to the device, runs the forward and
    the backward, and copies the output and the three gradients back.  Two
    buffer sets make it a two-deep pipeline on three streams (host -> device,
    compute, device -> host): step i+1's uploads and step i's downloads move in
    opposite directions of the link while step i computes."""
    import torch
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(x.numel() * x.element_size() for x in results)
    sets = []
    for i in range(2):
        din = d if i == 0 else {k: torch.empty_like(v) for k, v in d.items()}
        dres = results if i == 0 else tuple(torch.empty_like(x) for x in results)
        hres = tuple(torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in dres)
        sets.append((din, dres, hres))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in, ev_done, ev_copied = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def compute(din, dres):
        o, g_v, g_l, g_w = dres
        mask = din.get("key_padding_mask")
        a = (din["value"], shapes, lsi) + tuple(din[k] for k in names[1:-1])
        if fused:
            B.msda_forward_fused(*a, key_padding_mask=mask, output=o, stream=stream)
            B.msda_backward_fused(*a, din["grad_output"], key_padding_mask=mask, grad_value=g_v,
                                  grad_sampling_offsets=g_l, grad_attn_logits=g_w,
                                  reference_grad=False, workspace=workspace, stream=stream)
        else:
            B.msda_forward(*a, output=o, stream=stream)
            B.msda_backward(*a, din["grad_output"], g_v, g_l, g_w, workspace=workspace,
                            stream=stream)

    def e2e_step(i):
        b = i % 2
        din, dres, hres = sets[b]
        s_in.wait_event(ev_done[b])            # set b's inputs are free again
        with torch.cuda.stream(s_in):
            for k in host:
                din[k].copy_(host[k], non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_copied[b])        # set b's results have been read back
        compute(din, dres)
        ev_done[b].record(stream)
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            for h, x in zip(hres, dres):
                h.copy_(x, non_blocking=True)
        ev_copied[b].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = max(4, min(args.steps, 10))
    e0.record(s_in)
    for i in range(n_e2e):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, dist, dev)
    link = _link_baseline(host, sets[0][0], sets[0][1], sets[0][2], s_in, s_out, n_e2e, h2d, d2h,
                          wl.points)
    return {"value": job_rate(wl.points, world, e2e_ms), "unit": "points/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
            "link": link,
            "path": "per step: pinned host -> device copies of the inputs, msda_forward%s and "
                    "msda_backward%s through the Python API, device -> pinned host copies of the "
                    "output and the three gradients; two buffer sets, uploads / compute / "
                    "downloads on three streams" % (("_fused",) * 2 if fused else ("", ""))}


def _link_baseline(host, din, dres, hres, s_in, s_out, reps, h2d, d2h, points):
    """The same copies as one end-to-end step with no compute: the step's uploads
    alone, its downloads alone, and both at once on their two streams (one
    cudaMemcpyAsync per tensor, pinned host memory), so that e2e reads as a
    fraction of what the link moves."""
    import torch

    def up():
        with torch.cuda.stream(s_in):
            for k in host:
                din[k].copy_(host[k], non_blocking=True)

    def down():
        with torch.cuda.stream(s_out):
            for h, x in zip(hres, dres):
                h.copy_(x, non_blocking=True)

    def timed(fns, first, last):
        for fn in fns:
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(first)
        if last is not first:
            last.wait_event(a)
        for _ in range(reps):
            for fn in fns:
                fn()
        if last is not first:
            done = torch.cuda.Event()
            done.record(first)
            last.wait_event(done)
        b.record(last)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    up_ms = timed([up], s_in, s_in)
    down_ms = timed([down], s_out, s_out)
    both_ms = timed([up, down], s_in, s_out)
    return {"h2d_gbs": h2d / up_ms / 1e6, "d2h_gbs": d2h / down_ms / 1e6,
            "h2d_ms": up_ms, "d2h_ms": down_ms, "both_directions_ms": both_ms,
            "copy_only_points_per_s": points / both_ms * 1e3,
            "what": "the step's copies without compute: uploads alone, downloads alone, and "
                    "both at once on two streams"}


class _CapturedPass:
    """One pass captured as a CUDA graph with the runtime API (stream capture on
    the bench's side stream) and launched with cudaGraphLaunch: only the
    library's kernels are in the graph, and a replay enqueues nothing else."""

    def __init__(self, fn, stream):
        from cuda.bindings import runtime as cudart
        self.cudart, self.handle = cudart, cudart.cudaStream_t(stream.cuda_stream)
        mode = cudart.cudaStreamCaptureMode.cudaStreamCaptureModeThreadLocal
        self._ok(cudart.cudaStreamBeginCapture(self.handle, mode))
        try:
            fn()
        finally:
            err, graph = cudart.cudaStreamEndCapture(self.handle)
        self._ok((err,))
        err, self.exe = cudart.cudaGraphInstantiate(graph, 0)
        self._ok((err,))
        self._ok(cudart.cudaGraphDestroy(graph))

    def _ok(self, res):
        err = res[0]
        if err != self.cudart.cudaError_t.cudaSuccess:
            raise RuntimeError(f"CUDA graph capture: {err}")

    def __call__(self):
        self._ok(self.cudart.cudaGraphLaunch(self.exe, self.handle))


# -------------------------------------------------------------- native arm
def run_native(args, wl):
    import torch
    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    from scale_deformable_attention_05_b300 import binding as B

    dev = torch.device("cuda", local)
    fused = args.path == "fused"
    wl_r = rank_workload(wl, rank)
    inp = gen.make_fused_inputs(wl_r, args.ref_dim) if fused else gen.make_inputs(wl_r)
    names = (("value", "reference_points", "sampling_offsets", "attention_logits",
              "grad_output") if fused else
             ("value", "sampling_locations", "attention_weights", "grad_output"))

    def t(name):
        if wl.dtype in ("bf16", "f16"):
            tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
            return torch.from_numpy(inp[name + "_" + wl.dtype].view(np.int16).copy()).view(tdt)
        return torch.from_numpy(np.ascontiguousarray(inp[name]))

    host = {k: t(k).pin_memory() for k in names}
    if fused and args.padding_mask:
        host["key_padding_mask"] = torch.from_numpy(gen.padding_mask(wl_r)).pin_memory()
    d = {k: v.to(dev) for k, v in host.items()}
    mask = d.get("key_padding_mask")
    shapes = torch.from_numpy(inp["spatial_shapes"]).to(dev)
    lsi = torch.from_numpy(inp["level_start_index"]).to(dev)
    out = torch.empty((wl.bs, wl.num_queries, wl.num_heads * wl.head_dim), dtype=d["value"].dtype,
                      device=dev)
    gv = torch.empty_like(d["value"])
    gl = torch.empty_like(d[names[2] if fused else "sampling_locations"])
    gw = torch.empty_like(d[names[3] if fused else "attention_weights"])
    code = {"f32": B.MSDA_F32, "bf16": B.MSDA_BF16, "f16": B.MSDA_F16}[wl.dtype]
    ws_bytes = B.msda_backward_workspace_bytes(wl.bs, wl.num_keys, wl.num_heads, wl.head_dim, code)
    workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 64 << 20) // 4, dtype=torch.float32, device=dev)
    torch.cuda.synchronize(dev)
    stream = torch.cuda.Stream(dev)      # graphs cannot be captured on the legacy default stream
    torch.cuda.set_stream(stream)
    args_fwd = (d["value"], shapes, lsi) + tuple(d[k] for k in names[1:-1])

    def run_forward():
        if fused:
            B.msda_forward_fused(*args_fwd, key_padding_mask=mask, output=out, stream=stream)
        else:
            B.msda_forward(*args_fwd, output=out, stream=stream)

    def run_backward(accumulate):
        if fused:     # the encoder's reference points are constants: no reference gradient
            B.msda_backward_fused(*args_fwd, d["grad_output"], key_padding_mask=mask,
                                  grad_value=gv, grad_sampling_offsets=gl, grad_attn_logits=gw,
                                  reference_grad=False, workspace=workspace,
                                  accumulate=accumulate, stream=stream)
        else:
            B.msda_backward(*args_fwd, d["grad_output"], gv, gl, gw, workspace=workspace,
                            accumulate=accumulate, stream=stream)

    # kernels per step (ours): forward 1; backward: zero-fill 1 + main 1 (+ finalize 1 for bf16)
    launches_per_step = 3 + (1 if wl.dtype != "f32" else 0)

    def zero_grad_value():
        if wl.dtype == "f32":
            B.msda_zero_fill(gv, stream=stream)

    passes_fn = [run_forward, zero_grad_value, lambda: run_backward(wl.dtype == "f32")]

    def step(evs=None):
        for i, fn in enumerate(passes_fn):
            if evs:
                evs[i].record(stream)
            fn()
        if evs:
            evs[3].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if not args.no_graph:
        # Each pass captured once as a CUDA graph and replayed: the timed region
        # then holds the library's kernels alone, not the Python marshalling
        # between them (which exceeds the kernel time of the small workloads).
        passes_fn = [_CapturedPass(fn, stream) for fn in passes_fn]
        for _ in range(2):
            flush.zero_()
            step()
        torch.cuda.synchronize()
    if dist:
        dist.barrier()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        step(ev[i])
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()

    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    zero_ms = [e[1].elapsed_time(e[2]) for e in ev]
    bwd_ms = [e[2].elapsed_time(e[3]) for e in ev]
    step_ms = [e[0].elapsed_time(e[3]) for e in ev]
    mean = lambda xs: sum(xs) / len(xs)
    ms_step = max_over_ranks(mean(step_ms), dist, dev)

    assert B.msda_last_device_error() == 0

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = _e2e_pipelined(B, args, wl, fused, names, host, d, shapes, lsi, (out, gv, gl, gw),
                             workspace, stream, dev, dist, ws)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    hbm_gbs, peak_src = _peaks()
    if fused:
        # reference points [bs, Q, L, 2 or 4] replace nothing; offsets and logits have
        # the sizes of locations and weights
        ref_bytes = wl.bs * wl.num_queries * wl.num_levels * args.ref_dim * wl.elem_bytes
        if mask is not None:
            ref_bytes += wl.bs * wl.num_keys        # one mask byte per key
        fb = wl.compulsory_bytes(backward=False) + ref_bytes
        bb = wl.compulsory_bytes(backward=True) + ref_bytes
    else:
        fb = wl.compulsory_bytes(backward=False)
        bb = wl.compulsory_bytes(backward=True)
    passes = {
        "forward": {"kernel": "forward_kernel", "ms": mean(fwd_ms), "min_ms": min(fwd_ms),
                    "median_ms": statistics.median(fwd_ms),
                    "points_per_s": wl.points / (mean(fwd_ms) / 1e3),
                    "compulsory_bytes": fb, "gbs": fb / (mean(fwd_ms) / 1e3) / 1e9},
        "zero_fill": {"kernel": "zero_fill_kernel", "ms": mean(zero_ms)},
        "backward": {"kernel": "backward_kernel" + ("" if wl.dtype == "f32" else
                                                    " (+zero/finalize)"),
                     "ms": mean(bwd_ms), "min_ms": min(bwd_ms),
                     "median_ms": statistics.median(bwd_ms),
                     "points_per_s": wl.points / (mean(bwd_ms) / 1e3),
                     "compulsory_bytes": bb, "gbs": bb / (mean(bwd_ms) / 1e3) / 1e9},
    }
    for p in ("forward", "backward"):
        passes[p]["frac_of_measured_hbm"] = passes[p]["gbs"] / hbm_gbs
        passes[p]["frac_of_8tbs"] = passes[p]["gbs"] / 8000.0
    dom = max(("forward", "backward"), key=lambda p: passes[p]["ms"])
    kname = "forward_kernel" if dom == "forward" else "backward_kernel"
    roofline = {"bound": "hbm", "kernel": kname, "achieved": passes[dom]["gbs"],
                "peak": hbm_gbs, "unit": "GB/s", "frac": passes[dom]["gbs"] / hbm_gbs,
                "peak_source": peak_src,
                "algorithmic_bytes_per_launch": passes[dom]["compulsory_bytes"],
                # the committed captures run unmasked, with 2-d reference points
                "traffic": (None if mask is not None or (fused and args.ref_dim != 2) else
                            _profiled_traffic(wl.name, kname + ("_fused" if fused else "")))}

    line = {
        "metric": METRIC, "value": job_rate(wl.points, ws, ms_step), "unit": "points/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype, "data": "synthetic", "config": _config(wl, args),
        "roofline": roofline, "passes": passes, "gpu_launches": launches_per_step * args.steps,
        "wall_s_timed_region_incl_flush": wall, "clocks": clocks, "e2e": e2e,
    }
    if not args.no_cpu_baseline and ws == 1:
        inp0 = gen.make_inputs(wl)
        line["cpu_baseline"] = cpu_baseline(wl, inp0)
        if not fused:
            line["roofline_touched"] = touched_roofline(wl, inp0, passes, hbm_gbs)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


CEILING_PROBES = [
    # (name, probe, param, CTAs of 16 warps per SM)
    ("gather_ldg128_l1", 0, 64 << 10, 2), ("gather_ldg128_l1", 0, 64 << 10, 4),
    ("gather_ldg128_l2", 0, 64 << 20, 2), ("gather_ldg128_l2", 0, 64 << 20, 4),
    ("gather_ldg256_l1", 1, 64 << 10, 4), ("gather_ldg256_l2", 1, 64 << 20, 4),
    ("gather_lds128", 2, 0, 2), ("gather_lds128", 2, 0, 3),
    ("red_shared_f32_conflict_free", 3, 0, 2), ("red_shared_f32_4way", 3, 1, 2),
    ("red_shared_f32_stride33", 3, 2, 2), ("rmw_shared_f32_conflict_free", 5, 0, 2),
    ("red_global_v4_l2", 4, 64 << 20, 2), ("red_global_v4_l2", 4, 64 << 20, 4),
    ("gather_tma4_l2", 6, 64 << 20, 1), ("gather_tma4_l2", 6, 64 << 20, 2),
    ("gather_tma4_hbm", 6, 512 << 20, 2),
]


def run_ceiling(iters=2048):
    """On-chip ceilings of the row gathers and scatters (csrc/msda_ceiling.cu), one
    JSON line per probe: random 128-byte rows per SM clock."""
    import ctypes
    from scale_deformable_attention_05_b300 import build as lib_build
    lib = ctypes.CDLL(lib_build.build_ceiling())
    lib.msda_ceiling_run.argtypes = [ctypes.c_int, ctypes.c_longlong, ctypes.c_int, ctypes.c_int,
                                     ctypes.POINTER(ctypes.c_double)]
    lib.msda_ceiling_run.restype = ctypes.c_int
    for name, probe, param, ctas in CEILING_PROBES:
        out = (ctypes.c_double * 4)()
        rc = lib.msda_ceiling_run(probe, param, ctas, iters, out)
        if rc != 0:
            raise RuntimeError(f"ceiling probe {name} failed with CUDA error {rc}")
        print(json.dumps({"ceiling": name, "warps_per_sm": 16 * ctas, "param": param,
                          "rows_per_clk_per_sm": round(out[0], 4),
                          "bytes_per_clk_per_sm": round(out[0] * 128, 1),
                          "ms": round(out[1], 4), "sm_mhz": round(out[2], 1),
                          "rows": out[3]}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="encoder", choices=sorted(gen.WORKLOADS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--path", default="plain", choices=["plain", "fused", "layer"],
                    help="fused: msda_forward_fused / msda_backward_fused from reference "
                         "points, offsets and logits; layer: the MSDeformAttn layer with its "
                         "projections, through autograd")
    ap.add_argument("--padding-mask", action="store_true",
                    help="with --path fused: pass a key padding mask (padded image batch)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ref-dim", type=int, default=2, choices=[2, 4],
                    help="--path fused: 2-d reference points or 4-d reference boxes")
    ap.add_argument("--no-projection-compare", action="store_true",
                    help="--path layer: skip the cuBLAS-projection layer and the GEMM comparisons "
                         "(for launch lists of the library's own step)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every pass through the Python binding instead of replaying "
                         "its captured CUDA graph")
    ap.add_argument("--ceiling", action="store_true",
                    help="print the on-chip gather / scatter ceilings (one JSON line per probe) "
                         "instead of the benchmark line")
    args = ap.parse_args()
    if args.ceiling:
        return run_ceiling()
    # timing rule: at least three untimed warm-up steps
    args.warmup = max(args.warmup, 3)
    wl = gen.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, wl)
    if args.path == "layer":
        return run_layer(args, wl)
    return run_native(args, wl)


if __name__ == "__main__":
    sys.exit(main())

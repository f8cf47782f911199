"""Benchmark of the fused weight-gradient + optimizer step (one JSON line on rank 0).

A step is one pass of the whole hot path over one batch: for every linear layer of the
workload, dW = dY^T X accumulated in FP32 on chip and consumed by the optimizer in the same
kernel (weights and moments updated in place).  Default workload: the Llama-3.1-8B MLP weight
updates (gate/up 14336x4096, down 4096x14336, T = 4096 tokens, AdamW with FP32 moments at step
10), inputs seeded and synthetic, resident in HBM before timing starts.

  value       fused TFLOP/s = sum over layers of 2 T d_out d_in per step / device time per step
  unfused     the two-phase baseline (dW written to HBM, then the optimizer pass) on the same data
  e2e         the same metric with dY/X copied from pinned host memory each step and the updated
              weights copied back, through the same C-ABI calls
  roofline    the fused kernel's average launch time (CUDA events on its stream) against the
              measured dense BF16 tensor peak
  cpu_baseline  the CPU oracle timed on a bounded sample of the same workload

--impl reference times the CPU oracle as the reference arm (there is no other implementation of
this method to run).  Under torchrun every rank runs its own copy of the per-GPU work (the layers
are independent; no data-path collective), so the scaling is weak.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "backward_optimizer_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def _ncu_traffic(workload: str, opt: str, state: str):
    """DRAM bytes per launch of the fused kernel from a committed ncu summary, if it was taken
    from the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{workload}/{opt}/{state}")
    if not e or e.get("source_hash") != _kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = open(os.devnull, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        if self.out:
            self.out.close()

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------ ranks

def tensor_peak_for(peaks: dict, clocks) -> tuple:
    """The bf16 tensor peak a timed region is held to, and its key in the peaks file: the
    sustained figure (the GEMM timed in a seconds-long loop under the power cap) when the clock
    samples of the region saw the power cap, else the burst figure."""
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    if "sw_power_cap" in (clocks or {}).get("reasons", []) and "bf16_tflops_sustained" in peaks:
        return float(peaks["bf16_tflops_sustained"]), "bf16_tflops_sustained"
    return burst, "bf16_tflops"


def algorithmic_bytes(wl, opt: str, state: str, operands: str) -> int:
    """Least HBM bytes of one fused pass: per weight element W read and written (2 + 2) and each
    moment the optimizer keeps read and written (binary32 4 + 4, bf16 2 + 2, int8 1 + 1 plus a
    4-byte scale per 64 each way), plus dY and X read once (2 bytes per bf16 element, 1 per E4M3)."""
    from workloads import MOMENTS
    per_moment = {"fp32": 8.0, "bf16": 4.0, "int8": 2.0 + 8.0 / 64}[state]
    per_el = 4.0 + per_moment * sum(MOMENTS[opt])
    op = 2 if operands == "bf16" else 1
    return int(sum(l.d_out * l.d_in * per_el + wl.T * (l.d_out + l.d_in) * op for l in wl.layers))


def roofline_entry(flops, alg_bytes, launch_ms, tensor_peak, hbm_peak, traffic, hbm, tensor_src, hbm_src):
    """The fused kernel's roofline: the bound is the unit whose time at its peak is longer for the
    launch's algorithmic work -- the tensor core for its flops (TFLOP/s) or HBM for its bytes (GB/s)
    -- and `achieved` is that work over the measured launch time.  The other side is kept as
    `other` (frac of its own peak) so both can be read."""
    secs = launch_ms * 1e-3
    t_tensor = flops / (tensor_peak * 1e12)
    t_hbm = alg_bytes / (hbm_peak * 1e9)
    tensor = {"achieved": flops / secs / 1e12, "peak": tensor_peak, "unit": "TFLOP/s",
              "frac": flops / secs / 1e12 / tensor_peak, "peak_source": tensor_src}
    mem = {"achieved": alg_bytes / secs / 1e9, "peak": hbm_peak, "unit": "GB/s",
           "frac": alg_bytes / secs / 1e9 / hbm_peak, "peak_source": hbm_src}
    bound, main, other = ("tensor", tensor, mem) if t_tensor >= t_hbm else ("hbm", mem, tensor)
    return {"bound": bound, **main, "traffic": traffic, "hbm": hbm, "kernel": "forge_tile_kernel (fused)",
            "avg_launch_ms": launch_ms, "flops_per_launch": flops, "bytes_per_launch": alg_bytes,
            "other": dict(other, bound="tensor" if bound == "hbm" else "hbm")}


def max_over_ranks(values, world: int, device="cpu"):
    """Element-wise maximum of per-rank timings (the slowest rank defines the job's time).  The
    only collective of the benchmark besides barriers; no data of the path is exchanged."""
    import torch
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(flops_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Whole-job TFLOP/s under weak scaling: every rank does the same per-GPU work."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


# ------------------------------------------------------------------------------------ GPU arm

def _act_key(wl, i):
    """Activation buffer of layer i: its own for small workloads; for a many-layer sweep one dY/X
    buffer per distinct layer shape, shared by the layers of that shape."""
    l = wl.layers[i]
    return (l.d_out, l.d_in) if len(wl.layers) > 8 else i


def _make_layer(wl, i, opt, state, device, seed, act_cache, operands="bf16"):
    """One layer's W/m/v (its own) and dY/X (see _act_key): bf16, or E4M3 codes with per-tensor scales."""
    import torch
    from workloads import activations, activations_fp8, layer_state
    key = _act_key(wl, i)
    if key not in act_cache:
        if operands in ("e4m3", "e4m3-channel"):
            dyq, s_dy, xq, s_x = activations_fp8(wl, i, 1, seed, device=device,
                                                 per_channel=operands == "e4m3-channel")
            act_cache[key] = (dyq, xq, s_dy, s_x)
        else:
            act_cache[key] = activations(wl, i, 1, seed, device=device) + (1.0, 1.0)
    dy, x, s_dy, s_x = act_cache[key]
    w, m, v = layer_state(wl, i, opt, seed, device=device)
    q = None
    if state == "int8":
        l = wl.layers[i]
        n = l.d_out * l.d_in
        m = None if m is None else torch.randint(-127, 128, (l.d_out, l.d_in), dtype=torch.int8, device=device)
        v = None if v is None else torch.randint(0, 128, (l.d_out, l.d_in), dtype=torch.int8, device=device)
        q = torch.rand(2 * n // 64, device=device) * 1e-5
    elif state == "bf16":
        m = None if m is None else m.to(torch.bfloat16)
        v = None if v is None else v.to(torch.bfloat16)
    return dict(dy=dy, x=x, w=w, m=m, v=v, q=q, s_dy=s_dy, s_x=s_x)


def run_gpu(args, rank, world):
    import torch
    import backward_optimizer_gb300 as fg
    from workloads import WORKLOADS, default_hparams

    fg.build()
    fg.lib()
    dev = torch.device("cuda", torch.cuda.current_device())
    wl = WORKLOADS[args.workload]
    hp = default_hparams(args.opt)
    t_step = wl.steps[-1]
    act_cache = {}
    e4m3 = args.operands != "bf16"
    layers = [_make_layer(wl, i, args.opt, args.state, dev, 1000 * rank, act_cache, args.operands)
              for i in range(len(wl.layers))]
    stream = torch.cuda.current_stream()
    flops_step = wl.flops_per_step()

    def fused(i, L, on=None):
        on = stream if on is None else on
        if e4m3:
            fg.fused_dw_step_e4m3(L["dy"], L["x"], L["s_dy"], L["s_x"], L["w"], L["m"], L["v"], L["q"], args.opt, hp,
                                  t_step, seed=0x5EED + i, stream=on)
        else:
            fg.fused_dw_step(L["dy"], L["x"], L["w"], L["m"], L["v"], L["q"], args.opt, hp, t_step,
                             seed=0x5EED + i, stream=on)

    # bf16 operands: every layer of the step in one call (forge_fused_dw_step_layers), which runs
    # the layers that take CTA pairs together, up to 16 per launch; E4M3 operands: one call per layer
    grouped = not e4m3 and not args.per_layer_calls and len(layers) > 1
    group_args = [(L["dy"], L["x"], L["w"], L["m"], L["v"], L["q"], 0x5EED + i) for i, L in enumerate(layers)]
    calls_per_step = 1 if grouped else len(layers)

    def per_layer_pass(ev=None, on=None):
        on = stream if on is None else on
        for i, L in enumerate(layers):
            if ev is not None:
                ev[i][0].record(on)
            fused(i, L, on=on)
            if ev is not None:
                ev[i][1].record(on)

    def fused_pass(ev=None, on=None):
        on = stream if on is None else on
        if not grouped:
            return per_layer_pass(ev, on)
        if ev is not None:
            ev[0][0].record(on)
        fg.fused_dw_step_layers(group_args, args.opt, hp, t_step, stream=on)
        if ev is not None:
            ev[0][1].record(on)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---- fused, device-resident
    for _ in range(args.warmup):
        fused_pass()
    torch.cuda.synchronize()
    status = fg.sync_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = fg.launch_count()
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clocks:
        start.record(stream)
        for k in range(args.steps):
            fused_pass()
        stop.record(stream)
        torch.cuda.synchronize()
    barrier()
    launches = fg.launch_count() - launches0
    elapsed_ms = start.elapsed_time(stop)
    status = fg.sync_status()
    if status != 0:
        raise RuntimeError(f"device status {status} in the timed region")
    # the same K steps again with an event pair around every launch, for the kernel's average
    # launch duration (the roofline).  Kept out of the step timing: recording two events per launch
    # costs host time that a small layer's launch does not hide.
    per_launch = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(calls_per_step)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0.record(stream)
    for k in range(args.steps):
        fused_pass(per_launch[k])
    l1.record(stream)
    torch.cuda.synchronize()
    barrier()
    launch_ms = [a.elapsed_time(b) for step_ev in per_launch for (a, b) in step_ev]
    launch_pass_ms = l0.elapsed_time(l1) / args.steps
    if fg.sync_status() != 0:
        raise RuntimeError("device status in the per-launch timing")
    # the same step as one call per layer (one launch each), for comparison with the grouped call
    per_layer_ms = float("nan")
    if grouped:
        for _ in range(args.warmup):
            per_layer_pass()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        p0.record(stream)
        for _ in range(args.steps):
            per_layer_pass()
        p1.record(stream)
        torch.cuda.synchronize()
        per_layer_ms = p0.elapsed_time(p1) / args.steps
        if fg.sync_status() != 0:
            raise RuntimeError("device status in the per-layer timing")

    # ---- the same fused pass captured once in a CUDA graph and replayed: no host launch path per
    # layer (it matters only for small layers, whose kernels are shorter than a launch)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side), torch.cuda.graph(graph):
        fused_pass(on=torch.cuda.current_stream())
    stream.wait_stream(side)
    for _ in range(args.warmup):
        graph.replay()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    g0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    graph_ms = g0.elapsed_time(g1) / args.steps
    del graph
    if fg.sync_status() != 0:
        raise RuntimeError("device status after the graph replays")

    # ---- unfused two-phase baseline on the same data: all dW to HBM, then every optimizer pass
    dws = [torch.empty(l.d_out, l.d_in, dtype=torch.float32, device=dev) for l in wl.layers]
    torch.cuda.synchronize()
    mem0 = torch.cuda.memory_allocated()

    def unfused_pass(on=None):
        on = stream if on is None else on
        for L, dW in zip(layers, dws):
            if e4m3:
                fg.dw_gemm_e4m3(L["dy"], L["x"], L["s_dy"], L["s_x"], dW, stream=on)
            else:
                fg.dw_gemm(L["dy"], L["x"], dW, stream=on)
        for i, (L, dW) in enumerate(zip(layers, dws)):
            fg.opt_step(dW, L["w"], L["m"], L["v"], L["q"], args.opt, hp, t_step, seed=0x5EED + i, stream=on)

    for _ in range(args.warmup):
        unfused_pass()
    u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    u0.record(stream)
    for _ in range(args.steps):
        unfused_pass()
    u1.record(stream)
    torch.cuda.synchronize()
    unfused_ms = u0.elapsed_time(u1) / args.steps
    # the two-phase pass from a CUDA graph too, beside the fused pass's graph: for small layers,
    # whose kernels are shorter than a launch, the two differ most there
    ugraph = torch.cuda.CUDAGraph()
    side.wait_stream(stream)
    with torch.cuda.stream(side), torch.cuda.graph(ugraph):
        unfused_pass(on=torch.cuda.current_stream())
    stream.wait_stream(side)
    for _ in range(args.warmup):
        ugraph.replay()
    barrier()
    torch.cuda.synchronize()
    g0.record(stream)
    for _ in range(args.steps):
        ugraph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    unfused_graph_ms = g0.elapsed_time(g1) / args.steps
    del ugraph
    grad_pool_unfused = sum(d.numel() * 4 for d in dws)
    del dws
    torch.cuda.synchronize()

    # ---- end to end: dY/X from pinned host memory each step, updated W copied back
    # (one pinned host copy per distinct layer shape; every layer's dY/X is copied in each step)
    host_act = {k: (a[0].cpu().pin_memory(), a[1].cpu().pin_memory()) for k, a in act_cache.items()}
    host_in = [host_act[_act_key(wl, i)] for i in range(len(wl.layers))]
    out_by_key = {k: torch.empty((a[0].shape[1], a[1].shape[1]), dtype=torch.bfloat16).pin_memory()
                  for k, a in act_cache.items()}
    host_out = [out_by_key[_act_key(wl, i)] for i in range(len(wl.layers))]
    h2d = sum(a.numel() * a.element_size() + b.numel() * b.element_size() for a, b in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)

    # Three streams, so that copies overlap the kernels: layer i+1's inputs go up while layer i
    # computes, and layer i's updated W comes back while layer i+1 computes.  Events keep each
    # buffer's uses in order across layers and steps: an input buffer is refilled only after the
    # step that last read it (layers of one shape share a buffer in large sweeps), and W is updated
    # again only after its previous copy to the host.
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    keys = [_act_key(wl, i) for i in range(len(wl.layers))]
    consumed = {}  # buffer key -> event after the last fused step that read it
    w_read = {}    # layer -> event after its last W copy to the host

    def e2e_pass():
        for i, L in enumerate(layers):
            if keys[i] in consumed:
                up.wait_event(consumed[keys[i]])
            with torch.cuda.stream(up):
                L["dy"].copy_(host_in[i][0], non_blocking=True)
                L["x"].copy_(host_in[i][1], non_blocking=True)
            loaded = torch.cuda.Event()
            loaded.record(up)
            stream.wait_event(loaded)
            if i in w_read:
                stream.wait_event(w_read[i])
            fused(i, L)
            done = torch.cuda.Event()
            done.record(stream)
            consumed[keys[i]] = done
            down.wait_event(done)
            with torch.cuda.stream(down):
                host_out[i].copy_(L["w"], non_blocking=True)
            read = torch.cuda.Event()
            read.record(down)
            w_read[i] = read

    for _ in range(args.warmup):
        e2e_pass()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    up.wait_event(e0)  # no copy of the timed steps starts before the timer
    for _ in range(args.steps):
        e2e_pass()
    for ev in w_read.values():  # the last W copies end inside the timed region
        stream.wait_event(ev)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps

    # ---- the layer's input gradient dX = dY W (which must read W before the step replaces it),
    # alone and as the ordered layer backward (dX, then the fused step, per layer)
    dxs = [torch.empty(wl.T, l.d_in, dtype=torch.bfloat16, device=dev) for l in wl.layers]
    dx_ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in layers] for _ in range(args.steps)]

    def dx_pass(ev=None):
        for i, (L, dX) in enumerate(zip(layers, dxs)):
            if ev is not None:
                ev[i][0].record(stream)
            fg.dx_gemm(L["dy"], L["w"], dX, stream=stream)
            if ev is not None:
                ev[i][1].record(stream)

    def backward_pass():
        for i, (L, dX) in enumerate(zip(layers, dxs)):
            fg.linear_backward(L["dy"], L["x"], L["w"], L["m"], L["v"], L["q"], dX, args.opt, hp, t_step,
                               seed=0x5EED + i, stream=stream)

    timed = {"dx": float("nan"), "backward": float("nan")}
    for name, fn in () if e4m3 else (("dx", dx_pass), ("backward", backward_pass)):
        for _ in range(args.warmup):
            fn()
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        b0.record(stream)
        for k in range(args.steps):
            fn(dx_ev[k]) if name == "dx" else fn()
        b1.record(stream)
        torch.cuda.synchronize()
        timed[name] = b0.elapsed_time(b1) / args.steps
    dx_launch_ms = [] if e4m3 else [a.elapsed_time(b) for step_ev in dx_ev for (a, b) in step_ev]
    status = fg.sync_status()
    if status != 0:
        raise RuntimeError(f"device status {status} in the dX / backward timing")
    del dxs

    elapsed_ms, unfused_ms, e2e_ms, dx_ms, bwd_ms, graph_ms, unfused_graph_ms, per_layer_ms = max_over_ranks(
        [elapsed_ms, unfused_ms, e2e_ms, timed["dx"], timed["backward"], graph_ms, unfused_graph_ms, per_layer_ms],
        world, dev)
    ms_step = elapsed_ms / args.steps
    return dict(ms_step=ms_step, flops_step=flops_step, launch_ms=launch_ms, launches=launches,
                unfused_ms=unfused_ms, e2e_ms=e2e_ms, h2d=h2d, d2h=d2h, clocks=clocks.summary(),
                grad_pool_unfused=grad_pool_unfused, mem_fused=mem0, wl=wl, dx_ms=dx_ms, bwd_ms=bwd_ms, graph_ms=graph_ms,
                launch_pass_ms=launch_pass_ms, unfused_graph_ms=unfused_graph_ms, per_layer_ms=per_layer_ms,
                calls_per_step=calls_per_step, grouped=grouped,
                dx_launch_ms=dx_launch_ms)


def run_sweep(name, opt, steps, warmup, rank, world):
    """A many-layer sweep (one step = every layer once): the fused step against the two-phase
    schedule (every layer's dW to HBM, then every optimizer pass), with the peak HBM the gradients
    take in each (torch's allocator high-water mark over the step's own allocations)."""
    import torch
    import backward_optimizer_gb300 as fg
    from workloads import WORKLOADS, default_hparams
    dev = torch.device("cuda", torch.cuda.current_device())
    wl = WORKLOADS[name]
    hp = default_hparams(opt)
    t_step = wl.steps[-1]
    act_cache = {}
    layers = [_make_layer(wl, i, opt, "fp32", dev, 1000 * rank, act_cache) for i in range(len(wl.layers))]
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    group_args = [(L["dy"], L["x"], L["w"], L["m"], L["v"], None, 0x5EED + i) for i, L in enumerate(layers)]

    def fused_pass():
        fg.fused_dw_step_layers(group_args, opt, hp, t_step, stream=stream)

    def per_layer_pass():
        for i, L in enumerate(layers):
            fg.fused_dw_step(L["dy"], L["x"], L["w"], L["m"], L["v"], None, opt, hp, t_step, seed=0x5EED + i,
                             stream=stream)

    def timed(fn):
        for _ in range(warmup):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    # the sweep runs at the power cap (a step is 0.16 s of full load): one call per layer and one
    # grouped call measured within the noise of each other, so the sweep keeps one call per layer,
    # the way a backward pass hands over its layers, and times the grouped call beside it
    with ClockSampler(torch.cuda.current_device()) as clocks:
        fused_ms = timed(per_layer_pass)
    fused_pool = torch.cuda.max_memory_allocated() - base
    grouped_ms = timed(fused_pass)
    if fg.sync_status() != 0:
        raise RuntimeError("device status after the sweep's fused steps")
    torch.cuda.reset_peak_memory_stats()
    dws = [torch.empty(l.d_out, l.d_in, dtype=torch.float32, device=dev) for l in wl.layers]

    def unfused_pass():
        for L, dW in zip(layers, dws):
            fg.dw_gemm(L["dy"], L["x"], dW, stream=stream)
        for i, (L, dW) in enumerate(zip(layers, dws)):
            fg.opt_step(dW, L["w"], L["m"], L["v"], None, opt, hp, t_step, seed=0x5EED + i, stream=stream)

    unfused_ms = timed(unfused_pass)
    unfused_pool = torch.cuda.max_memory_allocated() - base
    if fg.sync_status() != 0:
        raise RuntimeError("device status after the sweep's two-phase steps")
    del dws, layers, act_cache
    torch.cuda.empty_cache()
    fused_ms, unfused_ms, grouped_ms = max_over_ranks([fused_ms, unfused_ms, grouped_ms], world, dev)
    return dict(wl=wl, fused_ms=fused_ms, unfused_ms=unfused_ms, fused_pool=fused_pool, unfused_pool=unfused_pool,
                grouped_ms=grouped_ms,
                clocks=clocks.summary(), steps=steps, warmup=warmup)


# ------------------------------------------------------------------------------------ CPU oracle

class OracleSample:
    """The CPU oracle's whole step (float64 dW, optimizer, Philox + stochastic rounding) timed on
    the first `rows` weight rows of the workload's first three layers: a bounded sample of the
    same workload.  Inputs are generated once."""

    def __init__(self, workload: str, opt: str, seed: int = 0):
        from tests.helpers import bits, f32
        from workloads import WORKLOADS, activations, default_hparams, layer_state
        self.wl = WORKLOADS[workload]
        self.opt = opt
        self.hp = default_hparams(opt)
        self.layers = []
        for i, l in enumerate(self.wl.layers[:3]):
            dy, x = activations(self.wl, i, 1, seed)
            w, m, v = layer_state(self.wl, i, opt, seed)
            self.layers.append((l, bits(dy), bits(x), bits(w), None if m is None else f32(m),
                                None if v is None else f32(v)))

    def run(self, rows: int):
        """Returns (flops done, seconds) for one sampled step of `rows` rows per layer."""
        import numpy as np
        from oracle import step as ostep
        flops, secs = 0, 0.0
        for i, (l, dyb, xb, wb, m, v) in enumerate(self.layers):
            r = min(rows, l.d_out)
            args = (np.ascontiguousarray(dyb[:, :r]), xb, np.ascontiguousarray(wb[:r]),
                    None if m is None else m[:r], None if v is None else v[:r])
            t0 = time.perf_counter()
            ostep.fused_step(self.opt, *args, self.hp, self.wl.steps[-1], 1 + i)
            secs += time.perf_counter() - t0
            flops += 2 * self.wl.T * r * l.d_in
        return flops, secs

    def whole(self, rows: int) -> bool:
        """Whether a sample of `rows` rows per layer is the workload's whole step."""
        return len(self.wl.layers) == len(self.layers) and all(rows >= l.d_out for l, *_ in self.layers)

    def describe(self, rows: int) -> str:
        """The sample in words: the rows of each sampled layer it covers."""
        if self.whole(rows):
            return f"the whole step of {self.wl.name} (every weight row of every layer)"
        parts = ", ".join(f"{min(rows, l.d_out)} of {l.d_out} rows of {l.name}" for l, *_ in self.layers)
        return f"the first weight rows of the first {len(self.layers)} layers of {self.wl.name}: {parts}"

    def rows_for(self, seconds: float) -> int:
        """Sample size (a multiple of 64 rows, 64 .. 4096) whose step takes about `seconds`."""
        f, s = self.run(64)
        return int(min(4096, max(64, 64 * int(seconds / max(s, 1e-6)))))


def blas_threads():
    """Threads numpy's BLAS runs the oracle's float64 products on: from threadpoolctl where it is
    installed, else from the OpenBLAS library numpy loaded (its get_num_threads symbol)."""
    import numpy as np
    np.ones((2, 2)) @ np.ones((2, 2))  # make sure the BLAS is loaded
    try:
        from threadpoolctl import threadpool_info
        for info in threadpool_info():
            if info.get("user_api") == "blas":
                return {"threads": int(info["num_threads"]), "library": info.get("internal_api", "blas")}
    except Exception:
        pass
    import ctypes
    try:
        with open("/proc/self/maps") as f:
            paths = sorted({l.split()[-1] for l in f if "openblas" in l.lower() and ".so" in l})
        for path in paths:
            lib = ctypes.CDLL(path)
            for sym in ("openblas_get_num_threads", "openblas_get_num_threads64_", "scipy_openblas_get_num_threads64_",
                        "scipy_openblas_get_num_threads"):
                fn = getattr(lib, sym, None)
                if fn is not None:
                    fn.restype = ctypes.c_int
                    return {"threads": int(fn()), "library": os.path.basename(path)}
    except OSError:
        pass
    return {"threads": None, "library": "unknown"}


def cpu_baseline(args):
    sample = OracleSample(args.workload, args.opt)
    rows = sample.rows_for(15.0) if args.oracle_rows <= 0 else args.oracle_rows
    flops, secs = sample.run(rows)
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "blas_threads": blas_threads(),
            "sample": f"{sample.describe(rows)} (float64 NumPy oracle, whole step incl. Philox/SR), "
                      f"{secs:.1f} s"}


# ------------------------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="forge", choices=["forge", "reference"])
    ap.add_argument("--workload", default="llama8b-mlp")
    ap.add_argument("--opt", default="adamw")
    ap.add_argument("--state", default="fp32", choices=["fp32", "int8", "bf16"])
    ap.add_argument("--operands", default="bf16", choices=["bf16", "e4m3", "e4m3-channel"],
                    help="dY/X format: bf16, or E4M3 codes with per-tensor or per-channel scales")
    ap.add_argument("--oracle-rows", type=int, default=0, help="rows per layer of the oracle sample (0: sized by time)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--per-layer-calls", action="store_true",
                    help="time the fused step as one call per layer instead of one call over all layers")
    ap.add_argument("--sweep", default="qwen14b-sweep",
                    help="many-layer sweep timed after the main workload, fused against two-phase ('none': skip)")
    ap.add_argument("--sweep-steps", type=int, default=5)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    from workloads import WORKLOADS
    wl = WORKLOADS[args.workload]
    metric = "fused dW+AdamW TFLOP/s & step ms per layer sweep vs unfused; % of BF16 tensor peak"
    config = {"workload": f"{wl.name}: {wl.description}", "opt": args.opt, "state": args.state,
              "operands": args.operands,
              "T": wl.T, "layers": [f"{l.name} {l.d_out}x{l.d_in}" for l in wl.layers[:7]],
              "n_layers": len(wl.layers), "l2": "inputs larger than L2 (W/m/v/dY/X per step >> 129 MB)"}

    if args.impl == "reference":
        if rank != 0:
            return
        t0 = time.perf_counter()
        sample = OracleSample(args.workload, args.opt)
        # whole --steps/--warmup run within ~2 minutes of oracle time
        rows = sample.rows_for(120.0 / (args.steps + args.warmup)) if args.oracle_rows <= 0 else args.oracle_rows
        vals = []
        for _ in range(args.warmup + args.steps):
            flops, secs = sample.run(rows)
            vals.append(flops / secs / 1e12)
        vals = vals[args.warmup:]
        v = statistics.median(vals)
        flops_step = wl.flops_per_step()
        line = {"impl": "reference", "metric": metric, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": flops_step / (v * 1e12) * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic",
                "config": dict(config, ms_per_step="measured on the whole step" if sample.whole(rows) else
                               "extrapolated to the full step at the oracle's measured rate"),
                "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                                 "blas_threads": blas_threads(),
                                 "sample": f"{sample.describe(rows)}, per step (float64 NumPy oracle, whole "
                                           f"step incl. Philox/SR)"},
                "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "wall_s": time.perf_counter() - t0}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    r = run_gpu(args, rank, world)
    sweep = None
    if args.sweep != "none" and args.state == "fp32" and args.operands == "bf16":
        sweep = run_sweep(args.sweep, args.opt, args.sweep_steps, max(3, min(args.warmup, 5)), rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return

    peaks, peaks_src = _peaks()
    bf16_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    tensor_peak, key = tensor_peak_for(peaks, r["clocks"])
    e4m3 = args.operands != "bf16"
    # E4M3 contractions take the FP8 peak: the measured bf16 peak times the nominal ratio 4.5 / 2.25
    peak = 2.0 * tensor_peak if e4m3 else tensor_peak
    cap_note = " (the timed region ran at the power cap)" if key == "bf16_tflops_sustained" else ""
    peak_source = (f"2 x {key} of {peaks_src} (nominal fp8/bf16 dense ratio 4.5/2.25){cap_note}" if e4m3
                   else f"{key} of {peaks_src}{cap_note}")
    n_layers = len(r["wl"].layers)
    avg_launch_ms = statistics.mean(r["launch_ms"])  # per call: the grouped call, or one layer's
    calls = r["calls_per_step"]
    flops_launch = r["flops_step"] / calls
    achieved = flops_launch / (avg_launch_ms * 1e-3) / 1e12
    value = job_throughput(r["flops_step"], world, r["ms_step"])
    # the epilogue side of the same launches: HBM bytes per launch over the same launch time
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    alg_bytes = algorithmic_bytes(r["wl"], args.opt, args.state, args.operands) / calls
    traffic = _ncu_traffic(args.workload, args.opt, args.state) if not e4m3 else None
    hbm = {"unit": "GB/s", "peak": hbm_peak, "algorithmic_bytes_per_launch": alg_bytes,
           "achieved_algorithmic": alg_bytes / (avg_launch_ms * 1e-3) / 1e9,
           "frac_algorithmic": alg_bytes / (avg_launch_ms * 1e-3) / 1e9 / hbm_peak,
           "achieved_measured": None if traffic is None else traffic / (avg_launch_ms * 1e-3) / 1e9,
           "peak_source": f"hbm_gbs of {peaks_src}"}
    line = {
        "metric": metric, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3" if e4m3 else "bf16", "data": "synthetic", "config": config,
        "calls": {"fused": "one forge_fused_dw_step_layers call per step (layers on CTA pairs run together, up to 16 "
                           "per launch)" if r["grouped"] else "one forge_fused_dw_step call per layer",
                  "launches_per_step": r["launches"] / args.steps},
        "per_layer": None if not r["grouped"] else {
            "ms_per_step": r["per_layer_ms"], "value": job_throughput(r["flops_step"], world, r["per_layer_ms"]),
            "what": "the same step as one forge_fused_dw_step call (one launch) per layer"},
        "unfused": {"ms_per_step": r["unfused_ms"], "value": job_throughput(r["flops_step"], world, r["unfused_ms"]),
                    "speedup_fused": r["unfused_ms"] / r["ms_step"],
                    "graph_ms_per_step": r["unfused_graph_ms"],
                    "graph_speedup_fused": r["unfused_graph_ms"] / r["graph_ms"]},
        "grad_pool_bytes": {"fused_hbm": 0, "unfused_hbm": r["grad_pool_unfused"],
                            "fused_on_chip": "two FP32 accumulators per SM in TMEM (at most 2 x 128x256 = 256 KiB), independent of model size"},
        "e2e": {"value": job_throughput(r["flops_step"], world, r["e2e_ms"]), "unit": "TFLOP/s",
                "ms_per_step": r["e2e_ms"], "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
        "gpu_launches": r["launches"],
        "graph": {"ms_per_step": r["graph_ms"], "value": job_throughput(r["flops_step"], world, r["graph_ms"]),
                  "unit": "TFLOP/s", "what": "the fused pass captured once in a CUDA graph and replayed"},
        "roofline": dict(roofline_entry(flops_launch, alg_bytes, avg_launch_ms, peak, hbm_peak, traffic, hbm,
                                        peak_source, f"hbm_gbs of {peaks_src}"),
                         launch_timing=f"CUDA events around each launch on its stream, over {args.steps} steps timed "
                                       f"again after the step timing ({r['launch_pass_ms']:.4f} ms per step there)"),
        "clocks": r["clocks"],
        # the layer's input gradient dX = dY W (same flops as dW) and the ordered layer backward
    }
    if r["dx_launch_ms"]:  # bf16 operands only: dX = dY W needs dY in bf16
        line["dx"] = {"ms_per_step": r["dx_ms"], "value": job_throughput(r["flops_step"], world, r["dx_ms"]),
                      "unit": "TFLOP/s", "avg_launch_ms": statistics.mean(r["dx_launch_ms"]),
                      "frac": r["flops_step"] / n_layers / (statistics.mean(r["dx_launch_ms"]) * 1e-3) / 1e12 / tensor_peak}
        line["layer_backward"] = {"ms_per_step": r["bwd_ms"],
                                  "value": job_throughput(2 * r["flops_step"], world, r["bwd_ms"]),
                                  "unit": "TFLOP/s", "what": "dX then the fused step, per layer, one stream"}
    if sweep is not None:
        sw = sweep["wl"]
        sus = float(peaks.get("bf16_tflops_sustained", bf16_peak))
        fused_v = job_throughput(sw.flops_per_step(), world, sweep["fused_ms"])
        line["sweep"] = {
            "workload": f"{sw.name}: {sw.description}", "layers": len(sw.layers), "T": sw.T, "opt": args.opt,
            "steps": sweep["steps"], "warmup": sweep["warmup"],
            "fused": {"ms_per_step": sweep["fused_ms"], "value": fused_v, "unit": "TFLOP/s",
                      "frac": fused_v / world / sus,
                      "peak": sus, "peak_source": f"bf16_tflops_sustained of {peaks_src} (a step of {len(sw.layers)} layers)",
                      "what": "one forge_fused_dw_step call per layer (280 launches)"},
            "unfused": {"ms_per_step": sweep["unfused_ms"],
                        "value": job_throughput(sw.flops_per_step(), world, sweep["unfused_ms"]), "unit": "TFLOP/s"},
            "speedup_fused": sweep["unfused_ms"] / sweep["fused_ms"],
            "grouped": {"ms_per_step": sweep["grouped_ms"],
                        "what": "the fused step as one forge_fused_dw_step_layers call (launches of up to 16 layers)"},
            "grad_pool_bytes": {"fused_hbm": sweep["fused_pool"], "unfused_hbm": sweep["unfused_pool"],
                                "what": "peak HBM allocated during the step beyond W/m/v/dY/X (torch allocator)"},
            "clocks": sweep["clocks"]}
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(args)
    print(json.dumps(line))


if __name__ == "__main__":
    main()

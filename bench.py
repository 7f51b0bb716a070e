"""Benchmark: block-sparse video attention forward on B300.

Default workload (one "step"): one va_sparse_attn_fwd call of the
Wan-2.1-1.3B-shaped radial-mask attention: B=1, 12 heads, 21x30x52 = 32,760
tokens, head_dim 128, bf16, 128-token blocks, radial mask with W0 = H*W
(29,786 of 65,536 block pairs live). The static mask is built once before
timing (it is shared by every step, layer and head). Inputs are synthetic
(seeded Fourier-mode Q/K, N(0,1) V) and resident in HBM when device timing
starts; one call touches Q+K+V+O = 403 MB, more than the 126 MB L2, so no
flush is needed between timed calls.

Metric: effective TFLOP/s over live blocks, i.e. 4 * d * (sum over live block
pairs of |I| * |J|, real tokens only) * B * heads per call, and ms per call.

--workload selects another measured workload (its own JSON line, same keys):
  lvsa_long       LVSA long horizon, 12 heads, 126x30x52 = 196,560 tokens,
                  +-2-frame window, anchor every 8th frame (step 0)
  hunyuan_radial  HunyuanVideo 720p shape, 24 heads, 33x45x80 = 118,800 tokens
  hunyuan_dense   the same with the all-ones mask on the same kernel
  svgear          one SVG-EAR step on the Wan shape: k-means of Q (256
                  clusters) and K (1,024 clusters), 10 iterations each, then
                  va_compensate_route at 15% density
  linear, mixed   linear attention (GB/s) and LinVideo's mixed attention at
                  r = 0.5 with the radial mask, on the Wan-shaped inputs
  backward        the attention backward (dq, dk, dv) of the Wan radial
                  workload: 2.5x the forward's FLOPs per call

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload NAME]
Under torchrun (N > 1) every rank runs its own copy of the workload (weak
scaling, no collective on the data path); rank 0 prints one JSON line.
--impl reference times the float64 CPU oracle (the only reference there is)
on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

D, BLOCK, BATCH = 128, 128, 1
UNIT = "TFLOP/s"
# attention workloads: grid, heads, mask kind and parameters, input seed
WORKLOADS = {
    "wan_radial": dict(T=21, H=30, W=52, heads=12, kind="radial", params={}, step=0, seed=1235,
                       desc="Wan-2.1-1.3B-shaped radial block-sparse attention forward",
                       mask="radial, W0=H*W"),
    "lvsa_long": dict(T=126, H=30, W=52, heads=12, kind="lvsa",
                      params=dict(local=2, period=8, anchor0=0, rot_stride=1), step=0,
                      seed=1237, desc="LVSA long-horizon (6x Wan frames) block-sparse attention "
                      "forward", mask="LVSA, +-2 frames + anchor every 8th frame, step 0"),
    "hunyuan_radial": dict(T=33, H=45, W=80, heads=24, kind="radial", params={}, step=0,
                           seed=1239, desc="HunyuanVideo-720p-shaped radial block-sparse "
                           "attention forward", mask="radial, W0=H*W"),
    "hunyuan_dense": dict(T=33, H=45, W=80, heads=24, kind="dense", params={}, step=0,
                          seed=1239, desc="HunyuanVideo-720p-shaped attention forward with the "
                          "all-ones mask on the same block-sparse kernel", mask="dense"),
    "wan_radial_d64": dict(T=21, H=30, W=52, heads=12, kind="radial", params={}, step=0,
                           seed=1235, d=64, desc="Wan-shaped radial block-sparse attention "
                           "forward with head_dim 64", mask="radial, W0=H*W"),
    "wan_radial_b64": dict(T=21, H=30, W=52, heads=12, kind="radial", params={}, step=0,
                           seed=1235, block=64, desc="Wan-shaped radial block-sparse attention "
                           "forward with 64-token mask blocks", mask="radial, W0=H*W, block 64"),
}
METRIC = "block-sparse attn effective TFLOP/s + ms/call at 32,760 tok; % of B300 BF16 peak"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "attn_tc_wan_radial_traffic.json")
KERNEL_SRC = os.path.join(ROOT, "linear_attention_video_fwd_b300", "csrc", "attn_tc.cuh")
# fp32 FMA roof of a B300 (148 SMs x 128 FP32 lanes x 2 FLOP at the 2,032 MHz
# maximum SM clock), the bound of the SIMT SVG-EAR kernels
FP32_FMA_PEAK_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12


def workload_metric(name, wl):
    if name == "wan_radial":
        return METRIC
    N = wl["T"] * wl["H"] * wl["W"]
    return "block-sparse attn effective TFLOP/s + ms/call at %s tok (%s); %% of B300 BF16 peak" % (
        format(N, ","), name)


def workload_config(name, wl):
    N = wl["T"] * wl["H"] * wl["W"]
    d = wl.get("d", D)
    return {"workload": wl["desc"], "B": BATCH, "heads": wl["heads"],
            "grid_THW": [wl["T"], wl["H"], wl["W"]], "tokens": N, "head_dim": d,
            "block": wl.get("block", BLOCK), "mask": wl["mask"],
            "l2": "inputs larger than L2 (Q+K+V+O = %d MB per call vs 126 MB L2), no flush"
                  % round(4 * BATCH * wl["heads"] * N * d * 2 / 1e6)}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "hbm_gbs": 6400.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock and throttle-reason sampling (every 200 ms) while active."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.samples = []
        self._proc = None
        self._t = None

    def _reader(self):
        for line in self._proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append(parts)

    def __enter__(self):
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._reader, daemon=True)
            self._t.start()
        except OSError:
            self._proc = None
        return self

    def __exit__(self, *exc):
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
            self._t.join(timeout=5)

    def summary(self):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(s[1]) for s in self.samples) if v is not None]
        smax = [v for v in (num(s[2]) for s in self.samples) if v is not None]
        reasons = sorted({self.REASONS[i] for s in self.samples for i in range(4)
                          if s[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(self.samples)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(os.environ.get("VA_BENCH_BACKEND", "nccl"))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def kernel_hash() -> str:
    with open(KERNEL_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it matches this kernel."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(PROFILE_TRAFFIC) as f:
        rec = json.load(f)
    if rec.get("kernel_sha256_16") != kernel_hash():
        return None
    return rec.get("dram_bytes_per_launch")


def threads_used() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def make_inputs(wl, seed):
    import synth
    return synth.video_qkv(BATCH, wl["heads"], wl["T"], wl["H"], wl["W"], wl.get("d", D),
                           seed=seed, dtype="bf16")


def oracle_block_mask(wl):
    from oracle import masks as OM
    kind = {"radial": OM.RADIAL, "lvsa": OM.LVSA, "dense": OM.DENSE}[wl["kind"]]
    return OM.block_mask(kind, wl["T"], wl["H"], wl["W"],
                         OM.MaskParams(block=wl.get("block", BLOCK), **wl["params"]), wl["step"])


def oracle_sample(wl, q, k, v, bm, rows):
    """Run the float64 oracle on `rows` of every head; returns (seconds, live
    FLOPs done, output rows [B, heads, R, d])."""
    from oracle import attention as OA
    N, d = q.shape[2], q.shape[3]
    blk = wl.get("block", BLOCK)
    live_keys_per_block = (bm * np.array([min(N, (b + 1) * blk) - b * blk
                                          for b in range(bm.shape[0])])[None, :]).sum(1)
    flops = 4.0 * d * float(live_keys_per_block[rows // blk].sum()) * BATCH * wl["heads"]
    t0 = time.perf_counter()
    o, _ = OA.block_sparse_attention(q, k, v, bm, blk, 1.0 / np.sqrt(d), rows=rows)
    return time.perf_counter() - t0, flops, o


def parity_record(got, want, what, max_abs=2e-2, mean_abs=2e-3, relative=False):
    """Element-wise comparison of sampled output rows with the oracle, taken
    outside the timed region. With `relative` the bars scale with the
    reference (gradients): max-abs <= max_abs * max|want|, mean-abs <=
    mean_abs * mean|want|."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.abs(got - want)
    mx, mn = float(err.max()), float(err.mean())
    bar_max = max_abs * float(np.abs(want).max()) if relative else max_abs
    bar_mean = mean_abs * float(np.abs(want).mean()) if relative else mean_abs
    return {"compared": what, "max_abs": mx, "mean_abs": mn,
            "bar": {"max_abs": bar_max, "mean_abs": bar_mean},
            "finite": bool(np.isfinite(got).all()),
            "pass": bool(np.isfinite(got).all() and mx <= bar_max and mn <= bar_mean)}


def e2e_leg(world, dev, stream, dev_in, dev_out, call, steps):
    """The same call end to end: each step copies its inputs in from pinned
    host memory and its result back out (non-blocking copies on the call's
    stream) around the call, timed with CUDA events, max over ranks.
    Returns (ms per step, host-to-device bytes, device-to-host bytes)."""
    import torch
    host_in = [x.to("cpu").pin_memory() for x in dev_in]
    host_out = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in dev_out]

    def step():
        for d_, h_ in zip(dev_in, host_in):
            d_.copy_(h_, non_blocking=True)
        call()
        for h_, d_ in zip(host_out, dev_out):
            h_.copy_(d_, non_blocking=True)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(3, min(steps, 10))
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / n
    return (ms, sum(x.numel() * x.element_size() for x in host_in),
            sum(x.numel() * x.element_size() for x in host_out))


def count_launches(call):
    """This library's kernels (namespace va) launched by one call, counted from
    the profiler's CUDA activity outside the timed region; None where the
    profiler records no kernels."""
    import torch
    try:
        from torch.profiler import ProfilerActivity, profile
        torch.cuda.synchronize()
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            call()
            torch.cuda.synchronize()
        names = [e.name for e in prof.events()
                 if e.device_type == torch.autograd.DeviceType.CUDA]
    except Exception:
        return None
    n = sum(1 for name in names if "va::" in name)
    return n if n > 0 else None


def timed_region(args, world, local, call, stream):
    """Warm-up, a >= 0.6 s pre-roll under the clock sampler, then K timed calls.

    Returns (total_ms max over ranks, per-call launch ms list, clock summary).
    """
    import torch
    for _ in range(args.warmup):
        call()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        # Keep the GPU busy with the same call for >= 0.6 s before timing, so the
        # 200 ms clock samples are all taken under this load.
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 0.6:
            for _ in range(4):
                call()
            torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("va:timed %d steps" % args.steps)
        t_begin.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            call()
            ends[i].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        time.sleep(0.25)
    barrier(world)
    total_ms = max_over_ranks(t_begin.elapsed_time(t_end), world, torch.device("cuda", local))
    return total_ms, [a.elapsed_time(b) for a, b in zip(starts, ends)], clocks.summary()


def run_ours(args, world, rank, local):
    import torch
    import linear_attention_video_fwd_b300 as va
    from oracle import attention as OA

    name = args.workload
    wl = WORKLOADS[name]
    T, H, W, heads = wl["T"], wl["H"], wl["W"], wl["heads"]
    N = T * H * W
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    q, k, v = make_inputs(wl, wl["seed"] + rank)
    qt, kt, vt = (torch.from_numpy(x).to(dev, torch.bfloat16) for x in (q, k, v))
    out = torch.empty_like(qt)
    kind = {"radial": va.RADIAL, "lvsa": va.LVSA, "dense": va.DENSE}[wl["kind"]]
    mask = va.mask_build(kind, T, H, W, block=wl.get("block", BLOCK), step=wl["step"], **wl["params"])
    flops = 4.0 * wl.get("d", D) * mask.live_pairs * BATCH * heads
    stream = torch.cuda.current_stream()

    def call():
        va.sparse_attn_fwd(qt, kt, vt, mask, out=out)

    # ---- device-timed region: inputs resident in HBM --------------------------
    total_ms, launch_ms, clocks = timed_region(args, world, local, call, stream)
    err = va.device_error()
    if err != va.OK:
        raise RuntimeError("device error in the timed region: %s" % va.status_string(err))
    ms_per_step = total_ms / args.steps
    value = world * flops * args.steps / (total_ms * 1e-3) / 1e12

    # ---- end to end through the public API with host buffers ------------------
    qh, kh, vh = (x.to("cpu").pin_memory() for x in (qt, kt, vt))
    oh = torch.empty(qh.shape, dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(3, min(args.steps, 10))

    def e2e_call():
        # host q/k/v in, host out back: va_sparse_attn_fwd_host pipelines the
        # copies of one chunk of heads with the attention of another
        va.sparse_attn_fwd_host(qh, kh, vh, mask, out=oh, stream=stream)

    for _ in range(2):
        e2e_call()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_call()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / e2e_steps
    tensor_bytes = qt.numel() * qt.element_size()

    pk, src = peaks()
    achieved = flops / (float(np.mean(launch_ms)) * 1e-3) / 1e12
    line = {
        "metric": workload_metric(name, wl), "value": round(value, 2), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Fourier-mode Q/K + N(0,0.5^2), V~N(0,1)); no weights needed",
        "config": dict(workload_config(name, wl),
                       live_blocks="%d/%d" % (mask.nnz, mask.nqb * mask.nqb),
                       parallelism="replicas: one independent workload per GPU"),
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": 3 * tensor_bytes, "d2h_bytes_per_step": tensor_bytes},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2),
                     "peak": pk["bf16_tflops"], "unit": UNIT,
                     "frac": round(achieved / pk["bf16_tflops"], 4),
                     "peak_source": "%s bf16 dense burst (MEASURED_PEAKS.json)" % src
                     if src == "measured" else "fallback 1800 TFLOP/s",
                     "frac_of_sustained": round(achieved / pk["bf16_tflops_sustained"], 4),
                     "flops_per_launch": flops, "launch_ms_mean": round(float(np.mean(launch_ms)), 4),
                     "launch_ms_min": round(float(np.min(launch_ms)), 4),
                     "traffic": profiled_traffic() if name == "wan_radial" else None,
                     "kernel": "va::attn_tc_kernel<%d, %s>" % (
                         wl.get("d", D), "true" if wl.get("block", BLOCK) == 64 else "false")},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if rank == 0:
        bm = oracle_block_mask(wl)
        full = world == 1 and not args.no_cpu_baseline
        rows = OA.sample_rows(N, wl.get("block", BLOCK), args.oracle_rows if full else 64, seed=7)
        secs, oflops, want = oracle_sample(wl, q, k, v, bm, rows)
        got = out[:, :, torch.from_numpy(rows).to(dev)].float().cpu().numpy()
        line["parity"] = parity_record(got, want, "output rows %d x %d heads vs the float64 "
                                       "oracle (last timed call)" % (len(rows), heads))
        if full:
            line["cpu_baseline"] = {"value": round(oflops / secs / 1e12, 6), "unit": UNIT,
                                    "cores": threads_used(), "kind": "oracle",
                                    "seconds": round(secs, 2),
                                    "sample": "%d seeded query rows x %d heads of the same "
                                              "workload (float64 numpy oracle, masked dense "
                                              "rows)" % (len(rows), heads)}
    mask.free()
    return line


SVG = dict(T=21, H=30, W=52, heads=12, Cq=256, Ck=1024, iters=10, density=0.15, seed=1238)


def svgear_flops(qa, ka, sel, Cq, Ck, N, iters, d=D):
    """Algorithmic FLOPs of one SVG-EAR step per stage (all heads), from the
    step's own clusters and selection."""
    heads = qa.shape[1]
    out = {"cluster_q": 2.0 * N * Cq * d * iters * heads,
           "cluster_k": 2.0 * N * Ck * d * iters * heads, "probe": 0.0, "exact": 0.0,
           "virtual": 0.0}
    for h in range(heads):
        nq = np.bincount(qa[0, h], minlength=Cq).astype(np.float64)
        nk = np.bincount(ka[0, h], minlength=Ck).astype(np.float64)
        s = sel[0, h]
        out["probe"] += 8.0 * (nq > 0).sum() * N * d          # 2 passes x (logits + values)
        out["exact"] += 4.0 * d * float((nq[:, None] * nk[None, :])[s].sum())
        virt = (~s) & (nk[None, :] > 0)
        out["virtual"] += 4.0 * d * float((nq[:, None] * virt).sum())
    return out


def run_svgear(args, world, rank, local, d=D):
    import torch
    import linear_attention_video_fwd_b300 as va
    import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    T, H, W, heads, Cq, Ck = SVG["T"], SVG["H"], SVG["W"], SVG["heads"], SVG["Cq"], SVG["Ck"]
    N = T * H * W
    q, k, v = synth.video_qkv(BATCH, heads, T, H, W, d, seed=SVG["seed"] + rank, dtype="bf16")
    qt, kt, vt = (torch.from_numpy(x).to(dev, torch.bfloat16) for x in (q, k, v))
    qinit = torch.from_numpy(synth.init_indices(BATCH, heads, N, Cq, seed=SVG["seed"])).to(dev)
    kinit = torch.from_numpy(synth.init_indices(BATCH, heads, N, Ck, seed=SVG["seed"],
                                                tensor=synth.INIT + 1)).to(dev)
    qa = torch.empty((BATCH, heads, N), dtype=torch.int32, device=dev)
    ka = torch.empty_like(qa)
    qc = torch.empty((BATCH, heads, Cq, d), dtype=torch.float32, device=dev)
    kc = torch.empty((BATCH, heads, Ck, d), dtype=torch.float32, device=dev)
    qn = torch.empty((BATCH, heads, Cq), dtype=torch.int32, device=dev)
    kn = torch.empty((BATCH, heads, Ck), dtype=torch.int32, device=dev)
    out = torch.empty_like(qt)
    sel = torch.empty((BATCH, heads, Cq, Ck), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    stage_ms = {"cluster_q": [], "cluster_k": [], "compensate_route": []}
    record = [False]

    def call():
        ev[0].record(stream)
        va.cluster(qt, Cq, SVG["iters"], qinit, qa, qc, qn)
        ev[1].record(stream)
        va.cluster(kt, Ck, SVG["iters"], kinit, ka, kc, kn)
        ev[2].record(stream)
        va.compensate_route(qt, kt, vt, qa, Cq, ka, Ck, SVG["density"], out=out, sel=sel)
        ev[3].record(stream)
        if record[0]:
            torch.cuda.synchronize()
            stage_ms["cluster_q"].append(ev[0].elapsed_time(ev[1]))
            stage_ms["cluster_k"].append(ev[1].elapsed_time(ev[2]))
            stage_ms["compensate_route"].append(ev[2].elapsed_time(ev[3]))

    total_ms, launch_ms, clocks = timed_region(args, world, local, call, stream)
    err = va.device_error()
    if err != va.OK:
        raise RuntimeError("device error in the timed region: %s" % va.status_string(err))
    # end to end: host q, k, v and the initial indices in, host output out
    e2e_ms, h2d, d2h = e2e_leg(world, dev, stream, [qt, kt, vt, qinit, kinit], [out], call,
                               args.steps)
    per_call = count_launches(call)
    record[0] = True
    for _ in range(3):
        call()
    fl = svgear_flops(qa.cpu().numpy(), ka.cpu().numpy(), sel.cpu().numpy().astype(bool), Cq, Ck,
                      N, SVG["iters"], d)
    step_flops = sum(fl.values())
    ms_per_step = total_ms / args.steps
    st = {k2: float(np.median(v2)) for k2, v2 in stage_ms.items()}
    comp_flops = fl["probe"] + fl["exact"] + fl["virtual"]
    stages = {"cluster_q": (fl["cluster_q"], st["cluster_q"]),
              "cluster_k": (fl["cluster_k"], st["cluster_k"]),
              "compensate_route": (comp_flops, st["compensate_route"])}
    pk, src = peaks()
    step_tf = step_flops / (ms_per_step * 1e-3) / 1e12
    line = {
        "metric": "SVG-EAR step (k-means Q/K + probe + routing + compensated attention) "
                  "effective TFLOP/s + ms/step at 32,760 tok" + ("" if d == D else ", head_dim %d" % d),
        "value": round(world * step_flops * args.steps / (total_ms * 1e-3) / 1e12, 3),
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 inputs, f32 arithmetic",
        "data": "synthetic (seeded Fourier-mode Q/K + N(0,0.5^2), V~N(0,1))",
        "config": {"workload": "SVG-EAR-style compensated sparse attention, Wan shape",
                   "B": BATCH, "heads": heads, "grid_THW": [T, H, W], "tokens": N,
                   "head_dim": d, "Cq": Cq, "Ck": Ck, "kmeans_iters": SVG["iters"],
                   "density": SVG["density"],
                   "parallelism": "replicas: one independent workload per GPU"},
        "stages_ms": {k2: round(v2, 3) for k2, v2 in st.items()},
        "stages_tflops": {n: round(f / (t * 1e-3) / 1e12, 2) for n, (f, t) in stages.items()},
        "flops_per_step": {k2: float(v2) for k2, v2 in fl.items()},
        # The step mixes tensor-core kernels (k-means distances, probe,
        # compensated attention) with memory-bound ones (member sums, routing,
        # gathers): its roofline is the whole step's algorithmic FLOPs against
        # the bf16 dense peak; the per-kernel split is in the ncu launch list.
        "roofline": {"bound": "tensor", "achieved": round(step_tf, 2),
                     "peak": pk["bf16_tflops"], "unit": UNIT,
                     "frac": round(step_tf / pk["bf16_tflops"], 4),
                     "peak_source": "%s bf16 dense burst" % src, "kernel": "whole SVG-EAR step",
                     "traffic": None},
        "e2e": {"value": round(world * step_flops / (e2e_ms * 1e-3) / 1e12, 3), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * per_call if per_call else None,
        "clocks": clocks,
    }
    if rank == 0:
        line.update(svgear_checks(args, world, va, q, k, v, qt, kt, vt, qa, ka, qinit, kinit,
                                  out, sel, Cq, Ck, N, d))
    return line


def svgear_checks(args, world, va, q, k, v, qt, kt, vt, qa, ka, qinit, kinit, out, sel, Cq, Ck,
                  N, d=D):
    """Outside the timed region: the step's output and routing against the
    float64 oracle (given the step's own clusters), the last k-means step
    against the oracle's argmin, and the oracle's compensated attention timed
    on the same rows as the CPU baseline."""
    import torch
    from oracle import attention as OA
    from oracle import kmeans as KM
    from oracle import svgear as S
    heads = q.shape[1]
    scale = 1.0 / np.sqrt(d)
    dev = qt.device
    err = torch.empty((BATCH, heads, Cq, Ck), dtype=torch.float32, device=dev)
    sel2 = torch.empty_like(sel)
    out2, _, _ = va.compensate_route(qt, kt, vt, qa, Cq, ka, Ck, SVG["density"], err=err, sel=sel2)
    qa9 = torch.empty_like(qa)
    qc9 = torch.empty((BATCH, heads, Cq, d), dtype=torch.float32, device=dev)
    qn9 = torch.empty((BATCH, heads, Cq), dtype=torch.int32, device=dev)
    va.cluster(qt, Cq, SVG["iters"] - 1, qinit, qa9, qc9, qn9)
    if va.device_error() != va.OK:
        raise RuntimeError("device error in the parity calls")
    # Member lists hold each cluster's tokens in ascending order, so a
    # repeated call on the same clusters is bit-identical (a pass criterion).
    same = bool(torch.equal(out2, out)) and bool(torch.equal(sel2, sel))
    qa_h, ka_h = qa.cpu().numpy(), ka.cpu().numpy()
    err_h, sel_h = err.cpu().numpy(), sel.cpu().numpy().astype(bool)
    sel2_h = sel2.cpu().numpy().astype(bool)
    rows = OA.sample_rows(N, BLOCK, 64, seed=9)
    got = out[:, :, torch.from_numpy(rows).to(dev)].float().cpu().numpy()
    want = np.empty_like(got, dtype=np.float64)
    route_exact = True
    oflops, secs = 0.0, 0.0
    for h in range(heads):
        nq, _ = S.cluster_stats(q[0, h], qa_h[0, h], Cq)
        nk, _ = S.cluster_stats(k[0, h], ka_h[0, h], Ck)
        # routing rule on the same call's own float32 errors, bit for bit
        route_exact &= bool(np.array_equal(sel2_h[0, h], S.route(err_h[0, h], nq, nk, N,
                                                                 SVG["density"])))
        t0 = time.perf_counter()
        want[0, h] = S.compensated_attention(q[0, h], k[0, h], v[0, h], qa_h[0, h], ka_h[0, h],
                                             Ck, sel_h[0, h], scale, rows=rows)
        secs += time.perf_counter() - t0
        for i in rows:
            s_row = sel_h[0, h][qa_h[0, h, i]]
            oflops += 4.0 * d * (float(s_row[ka_h[0, h]].sum()) + float((~s_row & (nk > 0)).sum()))
    rec = parity_record(got, want, "compensated output rows %d x %d heads vs the float64 oracle "
                        "on the step's clusters and selection" % (len(rows), heads))
    near = 0
    qc9_h, qa9_h = qc9.cpu().numpy().astype(np.float64), qa9.cpu().numpy()
    for h in (0, heads - 1):
        # the 10th assignment is the oracle's argmin under the GPU's 9th centroids
        d2 = KM.sq_distances(q[0, h], qc9_h[0, h])
        want_a = np.argmin(d2, axis=1)
        bad = np.nonzero(qa_h[0, h] != want_a)[0]
        gap = d2[bad, qa_h[0, h][bad]] - d2[bad, want_a[bad]]
        scl = (q[0, h][bad].astype(np.float64) ** 2).sum(1) + (qc9_h[0, h][want_a[bad]] ** 2).sum(1)
        if (gap > 1e-4 * scl).any():
            route_exact = False
        near += len(bad)
    rec.update({"routing_bit_exact": route_exact, "kmeans_near_ties_2_heads": near,
                "repeat_call_identical": same})
    rec["pass"] = bool(rec["pass"] and route_exact and same)
    extra = {"parity": rec}
    if world == 1 and not args.no_cpu_baseline:
        extra["cpu_baseline"] = {"value": round(oflops / secs / 1e12, 6), "unit": UNIT,
                                 "cores": threads_used(), "kind": "oracle",
                                 "seconds": round(secs, 2),
                                 "sample": "compensated attention (exact keys of the selected "
                                           "clusters + virtual keys) of %d query rows x %d "
                                           "heads, float64 oracle" % (len(rows), heads)}
    return extra


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm: bounded samples of the same workload per step."""
    if rank != 0:
        return None
    from oracle import attention as OA
    name = args.workload if args.workload in WORKLOADS else "wan_radial"
    wl = WORKLOADS[name]
    N = wl["T"] * wl["H"] * wl["W"]
    q, k, v = make_inputs(wl, wl["seed"])
    bm = oracle_block_mask(wl)
    per_step = args.reference_rows
    for i in range(args.warmup):
        oracle_sample(wl, q, k, v, bm, OA.sample_rows(N, wl.get("block", BLOCK), per_step,
                                                       seed=1000 + i))
    secs, fl = 0.0, 0.0
    for i in range(args.steps):
        s, f, _ = oracle_sample(wl, q, k, v, bm, OA.sample_rows(N, wl.get("block", BLOCK),
                                                                per_step, seed=2000 + i))
        secs += s
        fl += f
    value = fl / secs / 1e12
    return {
        "metric": workload_metric(name, wl), "value": round(value, 6), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded inputs as the GPU arm)", "impl": "reference",
        "config": dict(workload_config(name, wl), parallelism="single process, host cores"),
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads_used(),
                         "kind": "oracle",
                         "sample": "%d seeded query rows x %d heads per step"
                                   % (per_step, wl["heads"])},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_linear(args, world, rank, local, mixed, d=D):
    """Linear attention (or LinVideo's mixed attention, r = 0.5 with the radial
    mask) on the Wan-shaped inputs, head_dim d."""
    import torch
    import linear_attention_video_fwd_b300 as va

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = dict(WORKLOADS["wan_radial"], d=d)
    T, H, W, heads = wl["T"], wl["H"], wl["W"], wl["heads"]
    N = T * H * W
    q, k, v = make_inputs(wl, seed=1235 + rank)
    qt, kt, vt = (torch.from_numpy(x).to(dev, torch.bfloat16) for x in (q, k, v))
    out = torch.empty_like(qt)
    stream = torch.cuda.current_stream()
    r = 0.5
    mask = va.mask_build(1, T, H, W, block=128) if mixed else None  # radial

    def call():
        if mixed:
            va.mixed_attn_fwd(qt, kt, vt, mask, r, out=out)
        else:
            va.linear_attn_fwd(qt, kt, vt, out=out)

    total_ms, launch_ms, clocks = timed_region(args, world, local, call, stream)
    err = va.device_error()
    if err != va.OK:
        raise RuntimeError("device error in the timed region: %s" % va.status_string(err))
    ms_per_step = total_ms / args.steps
    call_ms = float(np.mean(launch_ms))
    e2e_ms, h2d, d2h = e2e_leg(world, dev, stream, [qt, kt, vt], [out], call, args.steps)
    per_call = count_launches(call)
    tensor_bytes = qt.numel() * qt.element_size()
    io_bytes = 4 * tensor_bytes                       # read Q, K, V; write O
    lin_flops = 4.0 * N * d * (d + 1) * BATCH * heads  # phi(K)^T [V | 1] and phi(Q) [S | z]
    pk, src = peaks()
    cfg = {"workload": ("LinVideo mixed attention r=0.5 (radial block-sparse + linear)"
                        if mixed else "linear attention forward, elu+1 feature map"),
           "B": BATCH, "heads": heads, "grid_THW": [T, H, W], "tokens": N, "head_dim": d,
           "l2": "inputs larger than L2 (Q+K+V+O = %d MB per call vs 126 MB L2), no flush"
                 % round(4 * N * d * 2 * BATCH * heads / 1e6),
           "parallelism": "replicas: one independent workload per GPU"}
    line = {"n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded Fourier-mode Q/K + N(0,0.5^2), V~N(0,1))",
            "config": cfg, "gpu_launches": args.steps * per_call if per_call else None,
            "clocks": clocks}
    if mixed:
        rp, col = mask.csr()
        blk = 128
        sizes = np.minimum(blk, N - np.arange((N + blk - 1) // blk) * blk)
        live = sum(int(sizes[i]) * int(sizes[col[rp[i]:rp[i + 1]]].sum())
                   for i in range(len(rp) - 1))
        att_flops = 4.0 * d * live * BATCH * heads
        flops = att_flops + lin_flops
        tf = flops / (call_ms * 1e-3) / 1e12
        line.update({
            "metric": "LinVideo mixed attention (r=0.5) effective TFLOP/s + ms/call at 32,760 tok"
                      + ("" if d == D else ", head_dim %d" % d),
            "value": round(world * flops * args.steps / (total_ms * 1e-3) / 1e12, 2),
            "unit": UNIT,
            "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": pk["bf16_tflops"],
                         "unit": UNIT, "frac": round(tf / pk["bf16_tflops"], 4),
                         "peak_source": "%s bf16 dense burst" % src,
                         "kernel": "whole call (attention + linear attention)", "traffic": None},
            "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
                    "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h}})
        mask.free()
    else:
        gbs = io_bytes / (call_ms * 1e-3) / 1e9
        line.update({
            "metric": "linear attention forward achieved GB/s + ms/call at 32,760 tok"
                      + ("" if d == D else ", head_dim %d" % d),
            "value": round(world * io_bytes * args.steps / (total_ms * 1e-3) / 1e9, 1),
            "unit": "GB/s",
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                         "peak_source": "%s copy bandwidth" % src,
                         "kernel": "whole call (lin_state + lin_prep + lin_out)",
                         "algorithmic_bytes": io_bytes, "flops": lin_flops, "traffic": None},
            "e2e": {"value": round(world * io_bytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                    "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h}})
    if rank == 0:
        from oracle import attention as OA
        from oracle import linear as OL
        rows = OA.sample_rows(N, BLOCK, 64, seed=10)
        got = out[:, :, torch.from_numpy(rows).to(dev)].float().cpu().numpy()
        t0 = time.perf_counter()
        if mixed:
            bm = oracle_block_mask(wl)
            want = OL.mixed_attention(q, k, v, bm, BLOCK, 1.0 / np.sqrt(d), r, rows=rows)
        else:
            want = OL.linear_attention(q, k, v, rows=rows)
        secs = time.perf_counter() - t0
        line["parity"] = parity_record(got, want, "output rows %d x %d heads vs the float64 "
                                       "oracle (last timed call)" % (len(rows), heads))
        if world == 1 and not args.no_cpu_baseline:
            if mixed:
                live_keys = (bm * np.minimum(BLOCK, N - np.arange(bm.shape[0]) * BLOCK)[None, :]).sum(1)
                oflops = (4.0 * d * float(live_keys[rows // BLOCK].sum())
                          + 4.0 * N * d * len(rows)) * BATCH * heads
                base = {"value": round(oflops / secs / 1e12, 6), "unit": UNIT}
            else:
                # the oracle's time for R rows, scaled to a whole call's rows,
                # against the call's algorithmic bytes
                full_secs = secs * N / len(rows)
                base = {"value": round(io_bytes / full_secs / 1e9, 4), "unit": "GB/s"}
            line["cpu_baseline"] = dict(base, cores=threads_used(), kind="oracle",
                                        seconds=round(secs, 2),
                                        sample="%d query rows x %d heads (float64 oracle, "
                                               "pairwise weights%s)"
                                               % (len(rows), heads,
                                                  ", plus the masked softmax rows" if mixed
                                                  else "; scaled to all rows"))
    head = {k2: line.pop(k2) for k2 in ("metric", "value", "unit")}
    return {**head, **line}


def run_bwd(args, world, rank, local):
    """The block-sparse attention backward on the Wan radial workload: one
    va_sparse_attn_bwd call per step (row preprocess, dK/dV kernel, dQ kernel),
    with out and lse from one forward call before timing."""
    import torch
    import linear_attention_video_fwd_b300 as va
    from oracle import attention as OA
    from oracle import attention_bwd as OB
    import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = WORKLOADS["wan_radial"]
    T, H, W, heads = wl["T"], wl["H"], wl["W"], wl["heads"]
    N = T * H * W
    q, k, v = make_inputs(wl, seed=1235 + rank)
    g = synth.upstream_grad(BATCH, heads, N, D, seed=1235 + rank)
    qt, kt, vt, gt = (torch.from_numpy(x).to(dev, torch.bfloat16) for x in (q, k, v, g))
    mask = va.mask_build(va.RADIAL, T, H, W, block=BLOCK)
    lse = torch.empty((BATCH, heads, N), dtype=torch.float32, device=dev)
    out, _ = va.sparse_attn_fwd(qt, kt, vt, mask, lse=lse)
    dq, dk, dv = (torch.empty_like(qt) for _ in range(3))
    fwd_flops = 4.0 * D * mask.live_pairs * BATCH * heads
    flops = 2.5 * fwd_flops          # S, dP, dV, dK, dQ: five products per live pair
    stream = torch.cuda.current_stream()

    def call():
        va.sparse_attn_bwd(qt, kt, vt, out, gt, lse, mask, dq=dq, dk=dk, dv=dv)

    total_ms, launch_ms, clocks = timed_region(args, world, local, call, stream)
    err = va.device_error()
    if err != va.OK:
        raise RuntimeError("device error in the timed region: %s" % va.status_string(err))
    ms_per_step = total_ms / args.steps
    call_ms = float(np.mean(launch_ms))

    # end to end: host q, k, v, out, dout, lse in; host dq, dk, dv out
    e2e_ms, h2d, d2h = e2e_leg(world, dev, stream, [qt, kt, vt, out, gt, lse], [dq, dk, dv],
                               call, args.steps)
    per_call = count_launches(call)

    pk, src = peaks()
    tf = flops / (call_ms * 1e-3) / 1e12
    line = {
        "metric": "block-sparse attn backward effective TFLOP/s + ms/call at 32,760 tok",
        "value": round(world * flops * args.steps / (total_ms * 1e-3) / 1e12, 2), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Fourier-mode Q/K + N(0,0.5^2), V~N(0,1), dO~N(0,1))",
        "config": dict(workload_config("wan_radial", wl),
                       workload="Wan-2.1-1.3B-shaped radial block-sparse attention backward "
                                "(dq, dk, dv from out, lse, dO)",
                       l2="inputs larger than L2 (Q+K+V+O+dO+dQ+dK+dV = 805 MB per call), "
                          "no flush",
                       parallelism="replicas: one independent workload per GPU"),
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": pk["bf16_tflops"],
                     "unit": UNIT, "frac": round(tf / pk["bf16_tflops"], 4),
                     "peak_source": "%s bf16 dense burst" % src,
                     "frac_of_sustained": round(tf / pk["bf16_tflops_sustained"], 4),
                     "flops_per_launch": flops, "launch_ms_mean": round(call_ms, 4),
                     "kernel": "whole call (bwd_prep + bwd_dkdv_tc + bwd_dq_tc)",
                     "traffic": None},
        "gpu_launches": args.steps * per_call if per_call else None,
        "clocks": clocks,
    }
    if rank == 0:
        bm = oracle_block_mask(wl)
        rows = OA.sample_rows(N, BLOCK, 64, seed=8)
        live_keys = (bm * np.minimum(BLOCK, N - np.arange(bm.shape[0]) * BLOCK)[None, :]).sum(1)
        oflops = 6.0 * D * float(live_keys[rows // BLOCK].sum()) * BATCH * heads
        t0 = time.perf_counter()
        want_dq, _, _ = OB.block_sparse_attention_grad(q, k, v, g, bm, BLOCK, 1.0 / np.sqrt(D),
                                                       rows=rows,
                                                       keys=np.array([], dtype=np.int64))
        secs = time.perf_counter() - t0
        got_dq = dq[:, :, torch.from_numpy(rows).to(dev)].float().cpu().numpy()
        line["parity"] = parity_record(got_dq, want_dq, "dq rows %d x %d heads vs the float64 "
                                       "gradient oracle (last timed call)" % (len(rows), heads),
                                       max_abs=3e-2, mean_abs=1e-2, relative=True)
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = {"value": round(oflops / secs / 1e12, 6), "unit": UNIT,
                                    "cores": threads_used(), "kind": "oracle",
                                    "seconds": round(secs, 2),
                                    "sample": "dq of %d seeded query rows x %d heads (float64 "
                                              "oracle: logits, dP and dQ products, 6*d FLOPs "
                                              "per live pair)" % (len(rows), heads)}
    mask.free()
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload",
                    choices=sorted(WORKLOADS) + ["svgear", "svgear_d64", "linear", "linear_d64", "mixed",
                                                 "mixed_d64", "backward"],
                    default="wan_radial")
    ap.add_argument("--oracle-rows", type=int, default=512,
                    help="query rows per head in the CPU-oracle baseline sample")
    ap.add_argument("--reference-rows", type=int, default=16,
                    help="query rows per head per step of the reference (oracle) arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if world != args.gpus:
        print("warning: --gpus %d but WORLD_SIZE %d" % (args.gpus, world), file=sys.stderr)
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    elif args.workload in ("svgear", "svgear_d64"):
        line = run_svgear(args, world, rank, local, 64 if args.workload == "svgear_d64" else D)
    elif args.workload in ("linear", "mixed", "linear_d64", "mixed_d64"):
        line = run_linear(args, world, rank, local, args.workload.startswith("mixed"),
                          64 if args.workload.endswith("_d64") else D)
    elif args.workload == "backward":
        line = run_bwd(args, world, rank, local)
    else:
        line = run_ours(args, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

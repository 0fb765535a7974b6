"""Benchmark: attention TFLOP/s (live-tile FLOPs) of one fwd + bwd step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl ours|reference]

One step = the whole hot path over one batch of synthetic input: the forward
kernel (O, LSE) and the three backward launches of flash_msa_bwd (D, dK/dV,
dQ), called through the C-ABI library.  FLOPs are counted on live 128 x 128 tiles only:
fwd = B * H * nnz * 4 * 128 * 128 * d, bwd = 2.5 x fwd (five products per
tile), step = 3.5 x fwd.  The default workload is B=1, H=32, N=16384,
d=128, causal (a 7B-style layer at long context); ``--config`` picks another
workload.  After the headline, ``sparse_scaling`` times the two block-sparse
workloads (causal window 1024 + strided, N=32768; causal window 4096 +
dilation, N=131072) for a few GPU-only steps each and reports their time per
live tile against the headline's.

Timing: W untimed warm-up steps, then K steps bracketed by a barrier and
cuda synchronize, CUDA events on the launching stream, max over ranks.  The
working set (Q, K, V, O, dO, dQ, dK, dV) is larger than the 129 MB L2, so no
flush is inserted between steps.  SM clocks and throttle reasons are sampled
with nvidia-smi during the timed region.  ``e2e`` repeats the step through the
same C-ABI calls with pinned HOST buffers, host<->device copies inside the
timed region.  ``cpu_baseline`` times the float64 oracle on a bounded sample of
the same workload on the host cores (rank 0 only).

Multi-GPU (torchrun): heads are independent, so each rank runs its own copy
of the per-GPU workload (weak scaling, no data-path collective); value = all
ranks' FLOPs / the slowest rank's time.

``--impl reference`` times the float64 oracle (the only reference this method
has) on the same workload and metric, each step a bounded sample of heads.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TILE = 128


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sparse-scaling", action="store_true")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return PEAKS_FALLBACK, "fallback"


def reduce_max(x: float, device) -> float:
    """Maximum of a per-rank scalar over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(step_flops: float, ms_per_step: float, world: int) -> float:
    """Whole-job TFLOP/s: every rank runs the same per-GPU work (weak scaling)."""
    return world * step_flops / (ms_per_step * 1e-3) / 1e12


def live_flops(w, nnz):
    fwd = w.B * w.H * nnz * 4.0 * TILE * TILE * w.d
    return fwd, 2.5 * fwd


# ---------------------------------------------------------------------------
# CPU oracle timing (process pool started with spawn before any GPU work)
# ---------------------------------------------------------------------------
FULL_ORACLE_MAX_N = 4096  # above this a head's (N, N) float64 matrices get too large


def mask_config(w):
    """The workload's mask for the JSON line (packed documents described, not listed)."""
    cfg = dict(w.mask)
    if w.docs is not None:
        cfg["documents"] = {"mean_tokens": w.docs[0], "seed": w.docs[1],
                            "as": "bit-packed mask" if w.docs_as == "bitmask" else "varlen offsets"}
    return cfg


def _oracle_head_job(args):
    """Oracle on one head: fwd + bwd with full materialisation for N <= 4096,
    else the row-chunked forward only."""
    from oracle import attention
    from oracle.mask import MaskSpec
    q, k, v, do, fields = args
    spec = MaskSpec(**fields)
    scale = q.shape[1] ** -0.5
    t0 = time.perf_counter()
    if q.shape[0] <= FULL_ORACLE_MAX_N:
        attention.forward_head(q, k, v, scale, spec)
        attention.backward_head(q, k, v, do, scale, spec)
    else:
        attention.forward_rows(q, k, v, scale, spec)
    return time.perf_counter() - t0


def oracle_work_fraction(w):
    """Share of the fwd+bwd step FLOPs one oracle head job performs."""
    return 1.0 if w.N <= FULL_ORACLE_MAX_N else 1.0 / 3.5


def oracle_sample_inputs(w, n_heads):
    """The first n_heads (b, h) pairs of the workload's seeded inputs (float64)."""
    from tiled_exact_attention_flash_gb300.inputs import as_f64, workload_inputs
    inp = workload_inputs(w)
    jobs = []
    for idx in range(n_heads):
        b, h = divmod(idx, w.H)
        jobs.append(tuple(as_f64(inp[n][b, :, h]) for n in ("q", "k", "v", "do")) + (w.mask_fields(),))
    return jobs


class OraclePool:
    """Spawned worker processes, one BLAS thread each."""

    def __init__(self, workers):
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        self.workers = workers
        self.pool = mp.get_context("spawn").Pool(workers)

    def time_sample(self, jobs):
        t0 = time.perf_counter()
        self.pool.map(_oracle_head_job, jobs, chunksize=1)
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


def oracle_heads_for(w, budget_s=15.0):
    """Heads per sample: enough work for the pool, bounded for long sequences."""
    per_head_s = {1: 0.01, 2: 3.5, 3: 20.0, 4: 20.0, 5: 30.0}.get(w.cid, 10.0)
    cores = os.cpu_count() or 1
    n = max(1, min(w.B * w.H, int(budget_s * cores / per_head_s)))
    return min(n, cores * 4, w.B * w.H)


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() in ("active", "1"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def sources_sha(names):
    """First 16 hex digits of the SHA-256 of the named kernel sources, concatenated."""
    h = hashlib.sha256()
    for n in names:
        path = os.path.join(ROOT, "tiled_exact_attention_flash_gb300", "csrc", n)
        if not os.path.exists(path):
            return None
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16] if names else None


def traffic_per_launch(kernel, workload_name):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel, {})
    sha = sources_sha(rec.get("sources", []))
    if not rec or sha is None or sha != rec.get("source_sha") or rec.get("workload") != workload_name:
        return None
    return rec.get("bytes_per_launch")


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
# The backward's launches, each timed on its own: (name, stage bits, the
# tensor-core FLOPs it issues per live tile in units of the forward's 4 x
# 128 x 128 x d, for the per-kernel roofline).
BWD_LAUNCHES = (("bwd_pre", "BWD_PREPROCESS", 0.0),
                ("bwd_dkdv", "BWD_DKDV", 2.0),
                ("bwd_dq", "BWD_DQ", 1.5))


class Problem:
    """One workload resident on the device: inputs, outputs, workspace, mask
    and index, and its live-tile FLOP counts."""

    def __init__(self, w, dev, api, host=None):
        import torch
        from tiled_exact_attention_flash_gb300.inputs import workload_inputs
        self.w = w
        fields = w.mask_fields()
        self.mask = api.Mask(**fields) if fields else None
        self.index = None
        if self.mask is not None and self.mask.needs_index:
            self.index = api.build_block_index(self.mask, w.N).to(dev)
            self.nnz = self.index.nnz
        else:
            nb = (w.N + TILE - 1) // TILE
            self.nnz = nb * (nb + 1) // 2 if (self.mask and self.mask.causal) else nb * nb
        self.fwd_flops, self.bwd_flops = live_flops(w, self.nnz)
        self.step_flops = self.fwd_flops + self.bwd_flops
        self.host = workload_inputs(w) if host is None else host
        self.q, self.k, self.v, self.do = (self.host[n].to(dev) for n in ("q", "k", "v", "do"))
        B, N, H, d = self.q.shape
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        self.dq, self.dk, self.dv = (torch.empty_like(self.q) for _ in range(3))
        self.ws = torch.empty(api.bwd_workspace_bytes(B, H, N, d, self.index), dtype=torch.uint8,
                              device=dev)

    def step(self, api, stream, ev=None):
        """fwd, then the backward's launches one by one; ev: events recorded
        before the forward and after every launch."""
        if ev is not None:
            ev[0].record(stream)
        api.fwd(self.q, self.k, self.v, mask=self.mask, index=self.index, out=self.o,
                lse=self.lse, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        for i, (_, bits, _) in enumerate(BWD_LAUNCHES):
            api.bwd(self.q, self.k, self.v, self.o, self.lse, self.do, mask=self.mask,
                    index=self.index, dq=self.dq, dk=self.dk, dv=self.dv, workspace=self.ws,
                    stream=stream, stages=getattr(api, bits))
            if ev is not None:
                ev[2 + i].record(stream)


def sparse_scaling(api, dev, stream, ms_per_tile_ref, ref_name, steps=5, warmup=2):
    """GPU-only fwd+bwd steps of the two block-sparse workloads: time per live
    tile (ms per step / (B * H * live tiles per head)) as a ratio to the
    headline workload's."""
    import torch
    from tiled_exact_attention_flash_gb300.inputs import WORKLOADS
    out = {"reference_workload": ref_name, "steps": steps,
           "note": "ratio = (ms per step / live tiles) / the same for the reference workload; "
                   "1.0 means time scales exactly with the live-tile count"}
    for cid in (4, 5):
        w = WORKLOADS[cid]
        prob = Problem(w, dev, api)
        for _ in range(warmup):
            prob.step(api, stream)
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            prob.step(api, stream)
        b.record(stream)
        torch.cuda.synchronize(dev)
        api.check_status(stream)
        ms = a.elapsed_time(b) / steps
        tiles = w.B * w.H * prob.nnz
        out[f"C{cid}"] = {"workload": w.name, "live_tiles": tiles, "ms_per_step": round(ms, 4),
                          "step_tflops": round(prob.step_flops / (ms * 1e-3) / 1e12, 2),
                          "ms_per_live_tile_ratio": round((ms / tiles) / ms_per_tile_ref, 4)}
        del prob
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch

    from tiled_exact_attention_flash_gb300 import api
    from tiled_exact_attention_flash_gb300.inputs import WORKLOADS

    rank, world, local = dist_env()
    w = WORKLOADS[args.config]
    peaks, peak_src = load_peaks()

    # CPU oracle pool first: spawned before any CUDA call
    pool = None
    if rank == 0 and not args.no_cpu_baseline:
        n_heads = oracle_heads_for(w)
        pool = OraclePool(min(os.cpu_count() or 1, n_heads))
        oracle_jobs = oracle_sample_inputs(w, n_heads)

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    stream = torch.cuda.current_stream(dev)

    prob = Problem(w, dev, api)
    mask, index, nnz = prob.mask, prob.index, prob.nnz
    fwd_flops, bwd_flops, step_flops = prob.fwd_flops, prob.bwd_flops, prob.step_flops
    # element-exact count beside the tile count: live (i, j) pairs per head
    # (the builder's count; closed forms for the arithmetic dense / causal lists)
    if index is not None:
        live_elems = index.live_elements
    elif mask is not None and mask.causal:
        live_elems = w.N * (w.N + 1) // 2
    else:
        live_elems = w.N * w.N
    exact_fwd_flops = w.B * w.H * live_elems * 4.0 * w.d

    host = prob.host
    q, k, v, do, o, lse = prob.q, prob.k, prob.v, prob.do, prob.o, prob.lse
    dq, dk, dv, ws = prob.dq, prob.dk, prob.dv, prob.ws
    B, N, H, d = q.shape
    n_ev = 2 + len(BWD_LAUNCHES)

    def step(ev=None):
        prob.step(api, stream, ev)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    api.check_status(stream)

    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]
    if not gpu_index.isdigit():
        gpu_index = str(local)
    clocks = ClockSampler(gpu_index)
    time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        step(evs[s])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clock_rec = clocks.stop()
    api.check_status(stream)
    total_ms = reduce_max(t_start.elapsed_time(t_end), dev)
    ms_per_step = total_ms / args.steps
    names = ["fwd"] + [name for name, _, _ in BWD_LAUNCHES]
    per_kernel = {name: sum(evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(args.steps))
                  / args.steps for i, name in enumerate(names)}

    value = job_value(step_flops, ms_per_step, world)
    fwd_tflops = fwd_flops / (per_kernel["fwd"] * 1e-3) / 1e12
    bwd_ms = sum(per_kernel[name] for name, _, _ in BWD_LAUNCHES)
    bwd_tflops = bwd_flops / (bwd_ms * 1e-3) / 1e12

    # roofline of the dominant kernel: tensor-core FLOPs it issues on live tiles
    kernel_flops = {"fwd": fwd_flops}
    kernel_flops.update({name: f * fwd_flops for name, _, f in BWD_LAUNCHES if f > 0})
    dominant = max(kernel_flops, key=lambda n: per_kernel[n])
    # the kernels are timed inside a long loop of back-to-back steps (about a
    # second and a half at the default workload), under the power cap: the
    # sustained bf16 figure is their roofline; the burst figure is reported
    # beside it (the *_pct_peak keys)
    peak = peaks["bf16_tflops"]
    peak_sus = peaks.get("bf16_tflops_sustained", peak)
    achieved = kernel_flops[dominant] / (per_kernel[dominant] * 1e-3) / 1e12
    roofline = {"kernel": dominant, "bound": "tensor", "achieved": round(achieved, 1),
                "peak": peak_sus, "unit": "TFLOP/s", "frac": round(achieved / peak_sus, 4),
                "peak_source": f"{peak_src} bf16_tflops_sustained (kernels timed inside a "
                               f"long loop of steps); frac of the burst {peak}: "
                               f"{achieved / peak:.4f}",
                "traffic": traffic_per_launch(dominant, w.name),
                "per_kernel_ms": {n: round(t, 4) for n, t in per_kernel.items()},
                "per_kernel_frac": {n: round(kernel_flops[n] / (per_kernel[n] * 1e-3) / 1e12 / peak_sus, 4)
                                    for n in kernel_flops}}

    # end to end through the same C-ABI with pinned host buffers: every step
    # copies its own Q, K, V, dO in and O, LSE, dQ, dK, dV out.  Copy-in,
    # compute and copy-out run on three streams over two buffer sets, so step
    # i's copies overlap the compute of its neighbours (a host pipeline; a
    # step's own copies still precede and follow its compute).
    e2e = None
    if not args.no_e2e:
        hq, hk, hv, hdo = (host[n].pin_memory() for n in ("q", "k", "v", "do"))
        dsets, hsets = [], []
        for _ in range(2):
            dsets.append({"q": torch.empty_like(q), "k": torch.empty_like(k),
                          "v": torch.empty_like(v), "do": torch.empty_like(do),
                          "o": torch.empty_like(o), "lse": torch.empty_like(lse),
                          "dq": torch.empty_like(dq), "dk": torch.empty_like(dk),
                          "dv": torch.empty_like(dv), "ws": torch.empty_like(ws)})
            hsets.append({"o": torch.empty_like(hq).pin_memory(),
                          "lse": torch.empty((B, H, N), dtype=torch.float32).pin_memory(),
                          "dq": torch.empty_like(hq).pin_memory(),
                          "dk": torch.empty_like(hk).pin_memory(),
                          "dv": torch.empty_like(hv).pin_memory()})
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of set j copied in
        ev_comp = [torch.cuda.Event() for _ in range(2)]  # set j computed (inputs free)
        ev_out = [torch.cuda.Event() for _ in range(2)]   # outputs of set j copied out

        def e2e_step(i):
            j = i % 2
            d, h = dsets[j], hsets[j]
            s_in.wait_event(ev_comp[j])
            with torch.cuda.stream(s_in):
                d["q"].copy_(hq, non_blocking=True)
                d["k"].copy_(hk, non_blocking=True)
                d["v"].copy_(hv, non_blocking=True)
                d["do"].copy_(hdo, non_blocking=True)
                ev_in[j].record(s_in)
            stream.wait_event(ev_in[j])
            stream.wait_event(ev_out[j])
            api.fwd(d["q"], d["k"], d["v"], mask=mask, index=index, out=d["o"], lse=d["lse"],
                    stream=stream)
            api.bwd(d["q"], d["k"], d["v"], d["o"], d["lse"], d["do"], mask=mask, index=index,
                    dq=d["dq"], dk=d["dk"], dv=d["dv"], workspace=d["ws"], stream=stream)
            ev_comp[j].record(stream)
            s_out.wait_event(ev_comp[j])
            with torch.cuda.stream(s_out):
                for n in ("o", "lse", "dq", "dk", "dv"):
                    h[n].copy_(d[n], non_blocking=True)
                ev_out[j].record(s_out)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        e_steps = max(3, min(args.steps, 20))
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(s_in)
        for i in range(e_steps):
            e2e_step(i)
        a1.record(s_out)
        torch.cuda.synchronize(dev)
        api.check_status(stream)
        e_ms = reduce_max(a0.elapsed_time(a1) / e_steps, dev)
        elem = q.numel() * q.element_size()
        kv_elem = k.numel() * k.element_size()
        e2e = {"value": round(world * step_flops / (e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
               "ms_per_step": round(e_ms, 4), "h2d_bytes_per_step": 2 * elem + 2 * kv_elem,
               "d2h_bytes_per_step": 2 * elem + 2 * kv_elem + lse.numel() * 4,
               "pipeline": "copy-in, compute, copy-out on three streams, two buffer sets"}

    # sparse workloads against the headline's time per live tile (one GPU;
    # only with the dense causal headline as the reference)
    scaling = None
    if world == 1 and args.config == 3 and not args.no_sparse_scaling:
        scaling = sparse_scaling(api, dev, stream, ms_per_step / (w.B * w.H * nnz), w.name)

    cpu_baseline = None
    if pool is not None:
        sample_s = pool.time_sample(oracle_jobs)
        pool.close()
        n_heads = len(oracle_jobs)
        frac = oracle_work_fraction(w)
        cpu_flops = step_flops * frac * n_heads / (w.B * w.H)
        what = "fwd+bwd" if frac == 1.0 else "forward only"
        cpu_baseline = {"value": cpu_flops / sample_s / 1e12, "unit": "TFLOP/s",
                        "cores": pool.workers, "kind": "oracle",
                        "sample": f"{n_heads} of {w.B * w.H} heads of the workload, float64 "
                                  f"{what}, {sample_s:.1f} s wall",
                        "cpu": cpu_model()}

    if rank == 0:
        line = {
            "metric": "attention TFLOP/s (live FLOPs, fwd+bwd step)",
            "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic: seeded N(0,1) fp32 rounded to bf16",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "mask": mask_config(w), "live_tiles_per_head": nnz, "layout": "(B,N,H,d)",
                       "l2": "no flush: working set of 8 (B,N,H,d) bf16 tensors "
                             f"= {8 * B * N * H * d * 2 / 2**20:.0f} MiB > 129 MB L2"},
            "fwd_tflops": round(fwd_tflops, 2), "bwd_tflops": round(bwd_tflops, 2),
            "fwd_pct_peak": round(100 * fwd_tflops / peak, 2),
            "bwd_pct_peak": round(100 * bwd_tflops / peak, 2),
            "step_pct_peak": round(100 * value / world / peak, 2),
            "pct_of": f"burst bf16 peak {peak} TF/s; against the sustained {peak_sus}: "
                      f"fwd {100 * fwd_tflops / peak_sus:.2f}%, bwd {100 * bwd_tflops / peak_sus:.2f}%, "
                      f"step {100 * value / world / peak_sus:.2f}%",
            "roofline": roofline, "cpu_baseline": cpu_baseline, "e2e": e2e,
            "sparse_scaling": scaling,
            "gpu_launches": (1 + len(BWD_LAUNCHES)) * args.steps, "clocks": clock_rec,
            "element_exact": {
                "live_elements_per_head": live_elems,
                "fwd_gflop": round(exact_fwd_flops / 1e9, 3),
                "fwd_tflops": round(exact_fwd_flops / (per_kernel["fwd"] * 1e-3) / 1e12, 2),
                "step_tflops": round(world * 3.5 * exact_fwd_flops / (ms_per_step * 1e-3) / 1e12, 2),
                "note": "4 d flops per live (i, j) pair in the forward, 3.5x that per step; "
                        "the headline counts whole live 128x128 tiles"},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return os.uname().machine


# ---------------------------------------------------------------------------
# reference arm: the float64 oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from tiled_exact_attention_flash_gb300.inputs import WORKLOADS
    w = WORKLOADS[args.config]
    from oracle import block_index
    from oracle.mask import MaskSpec
    fields = w.mask_fields()
    nnz = block_index.build(w.N, MaskSpec(**fields))["nnz"] \
        if any(key != "causal" for key in fields) else None
    if nnz is None:
        nb = (w.N + TILE - 1) // TILE
        nnz = nb * (nb + 1) // 2 if w.mask.get("causal") else nb * nb
    fwd_flops, bwd_flops = live_flops(w, nnz)
    step_flops = fwd_flops + bwd_flops
    n_heads = max(1, min(oracle_heads_for(w, budget_s=4.0), os.cpu_count() or 1))
    pool = OraclePool(min(os.cpu_count() or 1, n_heads))
    jobs = oracle_sample_inputs(w, n_heads)
    for _ in range(max(1, args.warmup)):
        pool.time_sample(jobs[:1])
    times = [pool.time_sample(jobs) for _ in range(args.steps)]
    pool.close()
    frac = oracle_work_fraction(w)
    sample_flops = step_flops * frac * n_heads / (w.B * w.H)
    ms = 1e3 * sum(times) / len(times)
    value = sample_flops / (ms * 1e-3) / 1e12
    line = {
        "impl": "reference", "metric": "attention TFLOP/s (live FLOPs, fwd+bwd step)",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded N(0,1) fp32 rounded to bf16",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "mask": mask_config(w)},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": pool.workers,
                         "kind": "oracle",
                         "sample": f"each step: {n_heads} of {w.B * w.H} heads, float64 "
                                   + ("fwd+bwd" if frac == 1.0 else "forward only"),
                         "cpu": cpu_model()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

"""Benchmark: serving-shaped paged decode on B300 (KV GB/s read and decode seq-steps/s).

Workload (serve256_bf16): 256 sequences, context lengths lognormal (median 500, sigma 0.8,
clipped to [16, 4096]), 32 layers, 32 query / 8 KV heads, head_dim 128, bf16 K/V, 16-token
blocks. One step = for every sequence one appended position (host allocator, pkv_append),
then for each of the 32 layers: slot-mapped write of the new K/V (pkv_reshape_and_cache) and
paged decode attention over the whole context (pkv_paged_decode). Synthetic data, random
values; every KV byte of every layer is read each step (23 GB per step, far above L2).

value        KV GB/s read = sum over layers and sequences of 2*len*Hkv*D*2 bytes / device time
             per step, inputs resident in HBM (CUDA events on the launch stream).
e2e          the same metric with the host allocator call, host->device copies of the step's
             inputs (slots, block tables, lengths, q/k/v of every layer, pinned) and the
             device->host copy of every layer's output inside the timed region.
roofline     decode launches timed alone with CUDA events inside the timed region, against the
             measured HBM copy bandwidth.
cpu_baseline the binary64 oracle (C, OpenMP) on a bounded sample of the same workload.

``--impl reference`` times the oracle (there is no other implementation of the pages' method)
on the host cores; under torchrun only rank 0 runs it.

Multi-GPU: replicas only. Each rank runs the whole workload on its own GPU; no collective is
on the data path (one barrier and one max-reduction of the timing).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

WORKLOAD = "serve256_bf16"
METRIC = "paged-decode KV GB/s read (% of B300 HBM peak); decode seq-steps/sec"
FALLBACK_HBM_GBS = 6400.0
NOMINAL_HBM_GBS = 7700.0      # B300 HBM3e datasheet figure (context beside the measured copy peak)
L2_FLUSH_BYTES = 256 << 20    # a write of this many bytes evicts the 126 MB L2
PREFILL_KERNEL = "paged_prefill_tc_kernel (tcgen05.mma, S and O in tensor memory, P as bf16 hi + lo)"


# ------------------------------------------------------------------------------------------------
# distributed plumbing (replicas)
# ------------------------------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(x: float, dist, device=None) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, dist, device=None) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------------------------------------
# clocks
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


def workload_config(name: str, world: int) -> dict:
    """The `config` object of a bench line; both arms print the same one for the same workload."""
    w = synth.workload(WORKLOAD)
    fp8 = name == "serve256_fp8"
    return {
        "workload": name,
        "description": w.description + (
            "; fp8 E4M3 pool with per-(token, head) scales (KV bytes = codes + scales)" if fp8 else ""),
        "n_seqs": w.n_seqs, "layers": w.n_layers, "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
        "head_dim": w.head_dim, "block_size": w.block_size,
        "l2": "inputs larger than L2 (every step reads all KV of 32 layers, >20 GB)",
        "parallelism": f"replicas x{world}", "partition": "balanced split (partition_tokens=0)",
    }


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def decode_traffic_record(workload: str):
    """Per-launch DRAM bytes of the decode kernel on `workload` from the committed ncu summary, if
    the kernel source it was taken on is unchanged (else None)."""
    rec = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(rec):
        return None
    with open(rec) as f:
        d = json.load(f)
    if d.get("kernel_sha256") != kernel_sha():
        return None
    return d.get("workloads", {}).get(workload)


def _strip_comments(src: str) -> str:
    """C/C++ source without // and /* */ comments, blank lines or indentation (comment edits keep
    the hash)."""
    out, i, n = [], 0, len(src)
    while i < n:
        if src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif src[i] == '"':                      # string literal (asm text): copied verbatim
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            out.append(src[i])
            i += 1
    return "\n".join(line.strip() for line in "".join(out).splitlines() if line.strip())


def kernel_sha() -> str:
    """Hash of the kernel sources' code (comments excluded): identifies the kernels ncu counters
    were taken on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_494_b300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(_strip_comments(f.read()).encode())
    return h.hexdigest()


# ------------------------------------------------------------------------------------------------
# the CUDA path
# ------------------------------------------------------------------------------------------------
class Serve:
    """Pool, caches and per-step inputs of the serving workload on one GPU."""

    def __init__(self, seed: int, n_steps: int, device, fp8: bool = False):
        import torch
        import paged_kv_cache_494_b300 as pkv
        self.torch, self.pkv = torch, pkv
        w = synth.workload(WORKLOAD)
        self.w = w
        self.fp8 = fp8
        self.L, self.n, self.Hq, self.Hkv, self.D, self.B = (w.n_layers, w.n_seqs, w.num_q_heads, w.num_kv_heads,
                                                             w.head_dim, w.block_size)
        self.lens0 = synth.lengths(w, seed)
        NB = synth.pool_blocks(w, self.lens0 + n_steps)
        self.MB = -(-(int(self.lens0.max()) + n_steps) // self.B) + 1
        self.pool = pkv.Pool(self.L, self.Hkv, self.D, self.B, NB, self.n + 1, self.MB, pkv.FP8 if fp8 else pkv.BF16,
                             initial_free_list=synth.free_list(NB, seed))
        self.seqs = [self.pool.alloc(-1, int(t))[0] for t in self.lens0]
        self.device = device
        g = torch.Generator(device=device).manual_seed(seed)
        shape = (NB, self.Hkv, self.B, self.D)
        # prefilled context: random K/V everywhere (values are data; only their bytes matter here)
        if fp8:
            kshape, vshape, sshape = self.pool.fp8_shapes()
            self.k_caches = [torch.randint(0, 0x7E, kshape, device=device, dtype=torch.uint8, generator=g)
                             for _ in range(self.L)]
            self.v_caches = [torch.randint(0, 0x7E, vshape, device=device, dtype=torch.uint8, generator=g)
                             for _ in range(self.L)]
            self.k_scales = [torch.rand(sshape, device=device, generator=g) * 0.01 for _ in range(self.L)]
            self.v_scales = [torch.rand(sshape, device=device, generator=g) * 0.01 for _ in range(self.L)]
        else:
            self.k_caches = [torch.randn(shape, device=device, dtype=torch.bfloat16, generator=g)
                             for _ in range(self.L)]
            self.v_caches = [torch.randn(shape, device=device, dtype=torch.bfloat16, generator=g)
                             for _ in range(self.L)]
        self.q = [torch.randn(self.n, self.Hq, self.D, device=device, dtype=torch.bfloat16, generator=g)
                  for _ in range(self.L)]
        self.k_new = [torch.randn(self.n, self.Hkv, self.D, device=device, dtype=torch.bfloat16, generator=g)
                      for _ in range(self.L)]
        self.v_new = [torch.randn(self.n, self.Hkv, self.D, device=device, dtype=torch.bfloat16, generator=g)
                      for _ in range(self.L)]
        self.out = [torch.empty(self.n, self.Hq, self.D, device=device, dtype=torch.float32) for _ in range(self.L)]
        self.ws = torch.empty(self.pool.decode_workspace_bytes(self.n, self.Hq, 0) // 4 + 4, device=device)
        self.stream = torch.cuda.current_stream(device)
        self.nvtx = False          # one NVTX range per layer (bench.py --nvtx)

    def plan_steps(self, n_steps: int):
        """Host allocator work for n decode steps (slot of each appended token, tables, lengths)."""
        torch = self.torch
        steps = []
        for _ in range(n_steps):
            slots, pairs = self.pool.append(self.seqs)
            assert len(pairs) == 0
            tables, lens = self.pool.block_table(self.seqs)
            steps.append((torch.from_numpy(slots).to(self.device), torch.from_numpy(tables).to(self.device),
                          torch.from_numpy(lens).to(self.device), lens.astype(np.int64)))
        return steps

    def kv_bytes(self, lens: np.ndarray) -> int:
        per_token_head = (self.D + 4) * 2 if self.fp8 else self.D * 2 * 2   # K + V (+ fp8 scales)
        return int(lens.sum()) * self.Hkv * per_token_head * self.L

    def decode(self, l, tables, lens) -> None:
        """One layer's paged decode (a single kernel launch) on the bench stream."""
        if self.fp8:
            self.pool.paged_decode_fp8(self.out[l], self.q[l], self.k_caches[l], self.v_caches[l],
                                       self.k_scales[l], self.v_scales[l], tables, lens, self.w.scale, 0, 0, self.ws,
                                       stream=self.stream)
        else:
            self.pool.paged_decode(self.out[l], self.q[l], self.k_caches[l], self.v_caches[l], tables, lens,
                                   self.w.scale, 0, self.ws, stream=self.stream)

    def run_step(self, step) -> int:
        """Enqueue one step: per layer K1 then decode. Returns the number of kernels launched."""
        slots, tables, lens, _ = step
        nvtx = self.torch.cuda.nvtx if self.nvtx else None
        for l in range(self.L):
            if nvtx:
                nvtx.range_push(f"layer {l}")
            if self.fp8:
                self.pool.reshape_and_cache_fp8(self.k_new[l], self.v_new[l], slots, self.k_caches[l],
                                                self.v_caches[l], self.k_scales[l], self.v_scales[l],
                                                stream=self.stream)
            else:
                self.pool.reshape_and_cache(self.k_new[l], self.v_new[l], slots, self.k_caches[l], self.v_caches[l],
                                            stream=self.stream)
            self.decode(l, tables, lens)
            if nvtx:
                nvtx.range_pop()
        return self.L * 2


def bench_cuda(args, world, rank, local):
    import torch
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist = init_dist(world, "nccl")
    steps_total = args.warmup + 2 * args.steps
    fp8 = args.workload == "serve256_fp8"
    s = Serve(args.seed + rank, 2 * steps_total + args.warmup + args.steps + 4, device, fp8=fp8)
    pkv = s.pkv
    plan = s.plan_steps(steps_total)
    s.nvtx = args.nvtx
    Ev = lambda: torch.cuda.Event(enable_timing=True)

    for i in range(args.warmup):
        s.run_step(plan[i])
    torch.cuda.synchronize()
    assert pkv.last_error() == pkv.OK

    # timed region 1 (`value`): K steps exactly as a user would enqueue them, nothing else inside
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    start, stop = Ev(), Ev()
    launches = 0
    with ClockSampler(local) as clocks:
        start.record(s.stream)
        for k in range(args.steps):
            launches += s.run_step(plan[args.warmup + k])
        stop.record(s.stream)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    assert pkv.last_error() == pkv.OK
    t_ms = start.elapsed_time(stop)
    t_ms_max = max_over_ranks(t_ms, dist, device)
    kv_bytes = sum(s.kv_bytes(plan[args.warmup + k][3]) for k in range(args.steps))
    kv_bytes_all = sum_over_ranks(kv_bytes, dist, device)
    seq_steps_all = sum_over_ranks(s.n * args.steps, dist, device)
    value = kv_bytes_all / (t_ms_max * 1e-3) / 1e9

    # timed region 2 (roofline): the decode calls of the next K steps, back to back on the launch
    # stream (every layer of every step, > 20 GB of KV per step), CUDA events only at the two ends:
    # the average duration of one decode launch as the kernel runs in a sequence of launches
    torch.cuda.synchronize()
    r0, r1 = Ev(), Ev()
    r0.record(s.stream)
    for k in range(args.steps):
        _, tables_k, lens_k, _ = plan[args.warmup + args.steps + k]
        for l in range(s.L):
            s.decode(l, tables_k, lens_k)
    r1.record(s.stream)
    torch.cuda.synchronize()
    assert pkv.last_error() == pkv.OK
    dec_ms = [r0.elapsed_time(r1) / (args.steps * s.L)]
    dec_bytes = sum(s.kv_bytes(plan[args.warmup + args.steps + k][3]) for k in range(args.steps))
    dec_bytes_per_launch = dec_bytes / (args.steps * s.L)
    achieved = dec_bytes_per_launch / (float(np.mean(dec_ms)) * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()

    e2e = bench_e2e(s, args, dist, device) if not fp8 else None
    traffic = decode_traffic_record(args.workload)
    clk = clocks.summary()
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_ms_max / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8e4m3" if fp8 else "bf16",
        "accumulate": "f32",
        "data": "synthetic",
        "config": workload_config(args.workload, world),
        "mean_context": float(np.mean(plan[args.warmup][3])),
        "kv_gb_per_step": round(kv_bytes / args.steps / 1e9, 3),
        "seq_steps_per_s": round(seq_steps_all / (t_ms_max * 1e-3), 1),
        "pct_of_hbm_peak": round(100.0 * value / (peak * world), 2),
        "pct_of_nominal_hbm": round(100.0 * value / (NOMINAL_HBM_GBS * world), 2),
        "roofline": {
            "bound": "hbm",
            "kernel": "paged_decode_kernel (one pkv_paged_decode call; split units merged in-kernel by log-sum-exp)",
            "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": None if traffic is None else int(traffic["bytes_per_launch_profile"] * dec_bytes_per_launch
                                                         / traffic["algorithmic_bytes_profile"]),
            "algorithmic_bytes_per_launch": int(dec_bytes_per_launch),
            "mean_launch_us": round(1e3 * float(np.mean(dec_ms)), 2),
        },
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk,
    }
    if fp8:
        line["metric"] = "paged-decode KV GB/s read (fp8 pool, codes + scales); decode seq-steps/sec"
        line.pop("e2e")
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not fp8:
        line["cpu_baseline"] = cpu_baseline(args, budget_s=args.cpu_seconds)
    if rank == 0 and world == 1 and not fp8 and not args.no_workloads:
        del s, plan
        torch.cuda.empty_cache()
        line["workloads"] = bench_workloads(args, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def bench_e2e(s: Serve, args, dist, device):
    """Same metric through the public API with host buffers, all inside the timed region: the host
    allocator call (pkv_append), host->device copies of the step's inputs from pinned memory (slots,
    block tables, lengths, and q / k / v of every layer), the kernels, and the device->host copy of
    every layer's output. Copies run on their own streams so that layer l's inputs upload while
    layer l-1 computes and layer l-2's output downloads; device and pinned staging buffers are
    double-buffered across steps (a step reuses the buffers of the step before last)."""
    torch = s.torch
    L, n = s.L, s.n
    pin = lambda t: t.cpu().pin_memory()
    hq = [pin(t) for t in s.q]
    hk = [pin(t) for t in s.k_new]
    hv = [pin(t) for t in s.v_new]
    hout = [torch.empty(n, s.Hq, s.D, dtype=torch.float32).pin_memory() for _ in range(L)]
    dq = [[torch.empty_like(t) for t in s.q] for _ in range(2)]
    dk = [[torch.empty_like(t) for t in s.k_new] for _ in range(2)]
    dv = [[torch.empty_like(t) for t in s.v_new] for _ in range(2)]
    dout = [[torch.empty_like(t) for t in s.out] for _ in range(2)]
    h_slots = [torch.empty(n, dtype=torch.int64).pin_memory() for _ in range(2)]
    h_tab = [torch.empty(n, s.MB, dtype=torch.int32).pin_memory() for _ in range(2)]
    h_len = [torch.empty(n, dtype=torch.int32).pin_memory() for _ in range(2)]
    d_slots = [torch.empty(n, dtype=torch.int64, device=device) for _ in range(2)]
    d_tab = [torch.empty(n, s.MB, dtype=torch.int32, device=device) for _ in range(2)]
    d_len = [torch.empty(n, dtype=torch.int32, device=device) for _ in range(2)]
    s_h2d, s_comp, s_d2h = torch.cuda.Stream(device), torch.cuda.Stream(device), torch.cuda.Stream(device)
    step_done = [torch.cuda.Event(), torch.cuda.Event()]
    for e in step_done:
        e.record(s_d2h)
    ev_in = [[torch.cuda.Event() for _ in range(L)] for _ in range(2)]
    ev_out = [[torch.cuda.Event() for _ in range(L)] for _ in range(2)]
    count = [0]

    def step():
        p = count[0] & 1
        count[0] += 1
        step_done[p].synchronize()    # the step before last has released parity p's buffers
        slots, pairs = s.pool.append(s.seqs)
        tables, lens = s.pool.block_table(s.seqs)
        h_slots[p].numpy()[:] = slots
        h_tab[p].numpy()[:] = tables
        h_len[p].numpy()[:] = lens
        with torch.cuda.stream(s_h2d):
            d_slots[p].copy_(h_slots[p], non_blocking=True)
            d_tab[p].copy_(h_tab[p], non_blocking=True)
            d_len[p].copy_(h_len[p], non_blocking=True)
            for l in range(L):
                dq[p][l].copy_(hq[l], non_blocking=True)
                dk[p][l].copy_(hk[l], non_blocking=True)
                dv[p][l].copy_(hv[l], non_blocking=True)
                ev_in[p][l].record(s_h2d)
        for l in range(L):
            s_comp.wait_event(ev_in[p][l])
            s.pool.reshape_and_cache(dk[p][l], dv[p][l], d_slots[p], s.k_caches[l], s.v_caches[l], stream=s_comp)
            s.pool.paged_decode(dout[p][l], dq[p][l], s.k_caches[l], s.v_caches[l], d_tab[p], d_len[p], s.w.scale,
                                0, s.ws, stream=s_comp)
            ev_out[p][l].record(s_comp)
        with torch.cuda.stream(s_d2h):
            for l in range(L):
                s_d2h.wait_event(ev_out[p][l])
                hout[l].copy_(dout[p][l], non_blocking=True)
            step_done[p].record(s_d2h)
        return lens.astype(np.int64)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    # three timed repetitions of K steps each; the median is reported (a wall-clock measurement
    # catches host hiccups of the box, which one repetition would report as the library's time)
    runs = []
    for _ in range(3):
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        kv = 0
        for _ in range(args.steps):
            kv += s.kv_bytes(step())
        torch.cuda.synchronize()
        t = time.perf_counter() - t0
        runs.append((max_over_ranks(t, dist, device), sum_over_ranks(kv, dist, device)))
    t_max, kv_all = sorted(runs, key=lambda r: r[1] / r[0])[1]
    h2d = n * 8 + n * s.MB * 4 + n * 4 + L * (hq[0].numel() * 2 + 2 * hk[0].numel() * 2)
    d2h = L * hout[0].numel() * 4
    assert s.pkv.last_error() == s.pkv.OK
    return {"value": round(kv_all / t_max / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(1e3 * t_max / args.steps, 3),
            "runs_gbps": [round(k / t / 1e9, 2) for t, k in runs],
            "timing": "wall clock (perf_counter) around K steps, device synchronised at both ends; "
                      "median of 3 repetitions"}


# ------------------------------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and --impl reference)
# ------------------------------------------------------------------------------------------------
def oracle_sample(seed: int, n_sample: int):
    """Host inputs for the oracle: the first n_sample sequences of the workload, one layer."""
    from oracle import alloc_model as am
    w = synth.workload(WORKLOAD)
    lens = synth.lengths(w, seed)[:n_sample]
    NB = int(sum(-(-int(t) // w.block_size) for t in lens))
    MB = -(-int(lens.max()) // w.block_size)
    model = am.PoolModel(NB, w.block_size, n_sample, MB, initial_free_list=synth.free_list(NB, seed))
    for t in lens:
        model.alloc(-1, int(t))
    tables, _ = model.block_table(range(n_sample))
    shape = (NB, w.num_kv_heads, w.block_size, w.head_dim)
    kc = synth.encode(synth.normal_f32(shape, seed, 11), "bf16")
    vc = synth.encode(synth.normal_f32(shape, seed, 12), "bf16")
    q = synth.encode(synth.normal_f32((n_sample, w.num_q_heads, w.head_dim), seed, 13), "bf16")
    return w, q, kc, vc, np.asarray(tables, dtype=np.int32), lens.astype(np.int32)


def time_oracle(seed: int, budget_s: float, n_sample: int = 32):
    from oracle import native
    w, q, kc, vc, tables, lens = oracle_sample(seed, n_sample)
    bytes_per_call = int(lens.sum()) * w.num_kv_heads * w.head_dim * 2 * 2
    calls, t_total, threads = 0, 0.0, 0
    while t_total < budget_s or calls == 0:
        t0 = time.perf_counter()
        _, threads = native.decode(q, kc, vc, tables, lens, w.scale, return_threads=True)
        t_total += time.perf_counter() - t0
        calls += 1
    per_call = t_total / calls
    gbs = bytes_per_call / per_call / 1e9
    seq_steps = n_sample / (per_call * w.n_layers)
    sample = (f"{n_sample} of {w.n_seqs} sequences ({int(lens.sum())} tokens), 1 of {w.n_layers} layers per call, "
              f"{calls} calls in {t_total:.1f} s; same lengths recipe, bf16 inputs, binary64 arithmetic")
    return gbs, seq_steps, threads, sample, per_call


def cpu_baseline(args, budget_s: float):
    gbs, seq_steps, threads, sample, _ = time_oracle(args.seed, budget_s)
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample,
            "seq_steps_per_s": round(seq_steps, 3), "host_cpus": len(os.sched_getaffinity(0))}


def bench_reference(args, world, rank):
    if world > 1:
        import torch.distributed as dist
        if rank != 0:
            return
    per_step_budget = max(1.0, args.cpu_seconds / max(args.steps, 1))
    # warm-up calls (untimed), then K timed steps, each one bounded oracle sample
    from oracle import native
    native.build()
    for _ in range(args.warmup):
        time_oracle(args.seed, 0.0, n_sample=8)
    gbs_list, ss_list, threads, sample = [], [], 0, ""
    t_all = 0.0
    for _ in range(args.steps):
        gbs, seq_steps, threads, sample, per_call = time_oracle(args.seed, per_step_budget)
        gbs_list.append(gbs)
        ss_list.append(seq_steps)
        t_all += per_call
    value = float(np.median(gbs_list))
    w = synth.workload(WORKLOAD)
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * t_all / args.steps * w.n_layers, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(WORKLOAD, world),
        "seq_steps_per_s": round(float(np.median(ss_list)), 3),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


class L2Flush:
    """Writes a buffer larger than L2 on the current stream (between timed launches)."""

    def __init__(self, device):
        import torch
        self.buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)

    def __call__(self):
        self.buf.fill_(1)


def time_launches(torch, fn, flush, n_iter: int, stream=None):
    """Median device time (ms) of fn() over n_iter launches, L2 flushed before each; CUDA events on
    the launch stream bracket fn() alone."""
    stream = stream or torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_iter)]
    for a, b in evs:
        flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return float(np.median([a.elapsed_time(b) for a, b in evs]))


def capture(torch, fn, n: int):
    """A CUDA graph of n calls of fn() (one direct call first, as the library asks before capture).
    Replaying it launches the same kernels without the host cost of n Python calls, so short kernels
    are timed on the device rather than by the speed of the host."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(n):
            fn()
    torch.cuda.synchronize()
    return g


def time_back_to_back(torch, fn, n_iter: int, stream=None):
    """Average device time (ms) of one fn() over n_iter launches enqueued back to back."""
    stream = stream or torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fn()
    a.record(stream)
    for _ in range(n_iter):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n_iter


def prefill_entry(args, n_iter: int = 10):
    """Causal paged prefill (prefill_bf16): every position of 16 x 2,048-token prompts is a query.
    Useful attention TFLOP/s (4 * D per (query row, attended key): q.K and p.V) against the measured
    dense bf16 tensor peak, L2 flushed before each timed launch."""
    import torch
    import paged_kv_cache_494_b300 as pkv
    w = synth.workload("prefill_bf16")
    lens = synth.lengths(w, args.seed)
    NB = synth.pool_blocks(w, lens)
    MB = -(-int(lens.max()) // w.block_size)
    pool = pkv.Pool(1, w.num_kv_heads, w.head_dim, w.block_size, NB, w.n_seqs, MB, pkv.BF16,
                    initial_free_list=synth.free_list(NB, args.seed))
    seqs = [pool.alloc(-1, int(t))[0] for t in lens]
    tables, l = pool.block_table(seqs)
    g = torch.Generator(device="cuda").manual_seed(args.seed)
    shape = (NB, w.num_kv_heads, w.block_size, w.head_dim)
    kc = torch.randn(shape, device="cuda", dtype=torch.bfloat16, generator=g)
    vc = torch.randn(shape, device="cuda", dtype=torch.bfloat16, generator=g)
    total = int(lens.sum())
    q = torch.randn(total, w.num_q_heads, w.head_dim, device="cuda", dtype=torch.bfloat16, generator=g)
    out = torch.empty(total, w.num_q_heads, w.head_dim, device="cuda")
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).cuda()
    t_tab, t_len = torch.from_numpy(tables).cuda(), torch.from_numpy(l).cuda()
    run = lambda: pool.paged_prefill(out, q, kc, vc, t_tab, t_len, cu, w.scale)
    for _ in range(max(args.warmup, 3)):
        run()
    torch.cuda.synchronize()
    flush = L2Flush("cuda")
    g1 = capture(torch, run, 1)
    t = time_launches(torch, g1.replay, flush, n_iter) * 1e-3
    assert pkv.last_error() == pkv.OK
    keys = sum(int(L) * (int(L) + 1) // 2 for L in lens)          # attended (row, key) pairs per head
    flops = 4.0 * w.head_dim * keys * w.num_q_heads
    kv_bytes = int(lens.sum()) * w.num_kv_heads * w.head_dim * 2 * 2
    peak = measured_tflops()
    tf = flops / t / 1e12
    return {"workload": "prefill_bf16", "description": w.description, "kernel": PREFILL_KERNEL,
            "ms_per_launch": round(t * 1e3, 4), "tflops": round(tf, 2), "kv_gb_per_s": round(kv_bytes / t / 1e9, 1),
            "flops_per_launch": flops,
            "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(tf / peak, 4)},
            "timing": f"median of {n_iter} launches (one-launch CUDA graph replays), L2 flushed before each"}


def measured_tflops() -> float:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"])
    return 1800.0


def bench_prefill(args):
    """The prefill line on its own (``--workload prefill_bf16``)."""
    with ClockSampler(0) as clocks:
        e = prefill_entry(args, n_iter=max(args.steps, 3))
    print(json.dumps({
        "metric": "paged-prefill causal attention TFLOP/s (useful FLOPs)", "value": e["tflops"], "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": e["ms_per_launch"],
        "higher_is_better": True, "dtype": "bf16", "accumulate": "f32", "data": "synthetic",
        "config": {"workload": "prefill_bf16", "description": e["description"], "l2": "flushed before each launch"},
        "kv_gb_per_s": e["kv_gb_per_s"], "roofline": e["roofline"], "kernel": e["kernel"],
        "clocks": clocks.summary()}), flush=True)


def decode_pool(pkv, name: str, seed: int, fp8: bool, full_pool: bool):
    """Pool, block tables and lengths of one layer of a decode workload, built by the library's
    allocator as the workload states. full_pool=False cuts the long-context workload's 80 GB pool
    to twice its pages (same scattered placement) so that an ncu capture holds a few GB."""
    w = synth.workload(name)
    lens = synth.lengths(w, seed)
    dtype = pkv.FP8 if fp8 else pkv.BF16
    if w.length_kind == "prefix":
        # one prompt forked into every child, the prompt released, each child's suffix appended:
        # the children share the prompt's blocks (the shared-prefix workload)
        NB = synth.pool_blocks(w, lens)
        MB = -(-int(lens.max()) // w.block_size) + 1
        pool = pkv.Pool(1, w.num_kv_heads, w.head_dim, w.block_size, NB, w.n_seqs + 1, MB, dtype,
                        initial_free_list=synth.free_list(NB, seed))
        root = None
        kids = []
        for op in synth.prefix_trace(w, seed):
            if op[0] == "new":
                root = pool.alloc(-1, op[1])[0]
            elif op[0] == "fork":
                kids.append(pool.fork(root))
            elif op[0] == "free":
                pool.free(root)
            elif op[2] > 0:
                pool.alloc(kids[op[1]], op[2])
        seqs = kids
    else:
        pages = sum(-(-int(t) // w.block_size) for t in lens)
        # the long-context workload's 80 GB pool is cut to twice its pages (same scattered placement
        # by a seeded permutation) so that the capture holds a few GB
        NB = synth.pool_blocks(w, lens) if (full_pool or w.pool_rule != "bytes:80e9") else 2 * pages
        MB = -(-int(lens.max()) // w.block_size) + 1
        pool = pkv.Pool(1, w.num_kv_heads, w.head_dim, w.block_size, NB, w.n_seqs, MB, dtype,
                        initial_free_list=synth.free_list(NB, seed))
        seqs = [pool.alloc(-1, int(t))[0] for t in lens]
    tables, l = pool.block_table(seqs)
    return w, pool, NB, tables, l, seqs


class DecodeProblem:
    """One layer of a decode workload on the device: pool, caches, q, tables, output, workspace."""

    def __init__(self, name: str, seed: int, fp8: bool = False, full_pool: bool = True,
                 partition_tokens=None, cascade: bool = False):
        import torch
        import paged_kv_cache_494_b300 as pkv
        self.torch, self.pkv, self.fp8 = torch, pkv, fp8
        w, pool, NB, tables, l, seqs = decode_pool(pkv, name, seed, fp8, full_pool)
        self.w, self.pool, self.NB = w, pool, NB
        g = torch.Generator(device="cuda").manual_seed(seed)
        if fp8:
            ks_, vs_, ss_ = pool.fp8_shapes()
            self.kc = torch.randint(0, 0x7E, ks_, device="cuda", dtype=torch.uint8, generator=g)
            self.vc = torch.randint(0, 0x7E, vs_, device="cuda", dtype=torch.uint8, generator=g)
            self.ksc = torch.rand(ss_, device="cuda", generator=g) * 0.01
            self.vsc = torch.rand(ss_, device="cuda", generator=g) * 0.01
        else:
            dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
            shape = (NB, w.num_kv_heads, w.block_size, w.head_dim)
            self.kc = torch.randn(shape, device="cuda", dtype=dt, generator=g)
            self.vc = torch.randn(shape, device="cuda", dtype=dt, generator=g)
        self.n = len(l)
        qdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
        self.q = torch.randn(self.n, w.num_q_heads, w.head_dim, device="cuda", dtype=qdt, generator=g)
        self.out = torch.empty(self.n, w.num_q_heads, w.head_dim, device="cuda")
        self.pt = w.partition_tokens if partition_tokens is None else partition_tokens
        # cascade: the blocks every sequence shares (the allocator's sharing structure) are attended
        # once for the batch, then merged with each sequence's private suffix
        self.cascade = cascade
        self.prefix_blocks = pool.shared_prefix_blocks(seqs) if cascade else 0
        wsb = (pool.shared_prefix_workspace_bytes(self.n, w.num_q_heads, self.prefix_blocks) if cascade
               else pool.decode_workspace_bytes(self.n, w.num_q_heads, self.pt))
        self.ws = torch.empty(wsb // 4 + 4, device="cuda")
        self.tab, self.lens = torch.from_numpy(tables).cuda(), torch.from_numpy(l).cuda()
        self.lens_host = l
        per = (w.head_dim + 4) * 2 if fp8 else w.head_dim * 2 * w.elem_bytes
        self.kv_bytes = int(l.sum()) * w.num_kv_heads * per      # logical KV bytes one launch reads
        # distinct KV bytes: every physical block a launch touches, counted once
        self.unique_bytes = len({int(b) for row, n_ in zip(tables, l) for b in row[:-(-int(n_) // w.block_size)]}) \
            * w.block_size * w.num_kv_heads * per

    def run(self):
        if self.cascade:
            self.pool.paged_decode_shared_prefix(self.out, self.q, self.kc, self.vc, self.tab, self.lens, self.w.scale,
                                                 self.prefix_blocks, self.ws)
        elif self.fp8:
            self.pool.paged_decode_fp8(self.out, self.q, self.kc, self.vc, self.ksc, self.vsc, self.tab, self.lens,
                                       self.w.scale, 0, self.pt, self.ws)
        else:
            self.pool.paged_decode(self.out, self.q, self.kc, self.vc, self.tab, self.lens, self.w.scale, self.pt,
                                   self.ws)


def decode_entry(name: str, seed: int, peak: float, flush, partition_tokens=None, n_iter: int = 20,
                 cascade: bool = False):
    """One decode workload: median of n_iter launches with L2 flushed before each (the number
    reported for every workload), and the average of n_iter launches back to back. GB/s and the
    roofline fraction use the logical KV bytes a launch reads (for the shared-prefix workload: the
    distinct blocks, each once); where the committed ncu record of the same kernel code has the
    launch's DRAM bytes, they are reported too. cascade=True runs the shared-prefix entry point."""
    import torch
    p = DecodeProblem(name, seed, partition_tokens=partition_tokens, cascade=cascade)
    for _ in range(3):
        p.run()
    torch.cuda.synchronize()
    assert p.pkv.last_error() == p.pkv.OK
    g1, gn = capture(torch, p.run, 1), capture(torch, p.run, n_iter)
    t = time_launches(torch, g1.replay, flush, n_iter)
    tb = time_back_to_back(torch, gn.replay, 1) / n_iter
    assert p.pkv.last_error() == p.pkv.OK
    gbs = p.kv_bytes / (t * 1e-3) / 1e9
    e = {"workload": name, "partition_tokens": p.pt, "n_seqs": p.n, "num_q_heads": p.w.num_q_heads,
         "num_kv_heads": p.w.num_kv_heads, "block_size": p.w.block_size, "pool_blocks": p.NB,
         "mean_context": round(float(np.mean(p.lens_host)), 1), "kv_bytes_per_launch": p.kv_bytes,
         "us_per_launch": round(1e3 * t, 2), "gb_per_s": round(gbs, 1),
         "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                      "frac": round(gbs / peak, 4)},
         "b2b_us_per_launch": round(1e3 * tb, 2), "b2b_gb_per_s": round(p.kv_bytes / (tb * 1e-3) / 1e9, 1),
         "timing": f"median of {n_iter} launches (one-launch CUDA graph replays), L2 flushed before each; "
                   f"b2b = mean of {n_iter} launches back to back in one CUDA graph (no flush)"}
    if p.w.length_kind == "prefix":
        # the children's shared prompt blocks are one set of physical pages: the bytes a launch must
        # bring from memory count each distinct block once
        ach = p.unique_bytes / (t * 1e-3) / 1e9
        e["unique_kv_bytes_per_launch"] = p.unique_bytes
        e["roofline"].update(achieved=round(ach, 1), frac=round(ach / peak, 4), achieved_logical=round(gbs, 1),
                             basis="distinct physical KV blocks a launch reads, each counted once")
    if cascade:
        e["method"] = ("cascade: blocks shared by every sequence attended once for the batch on tensor cores, "
                       "private suffixes by the decode kernel, log-sum-exp merge")
        e["prefix_blocks"] = p.prefix_blocks
    key = name if (partition_tokens is None or partition_tokens == p.w.partition_tokens) else None
    if key is not None and cascade:
        key += "_cascade"
    rec = decode_traffic_record(key) if key else None
    if rec is not None:
        e["dram_bytes_per_launch"] = int(rec["bytes_per_launch_profile"] * p.kv_bytes / rec["algorithmic_bytes_profile"])
    del p
    torch.cuda.empty_cache()
    return e


def fp8_step_entry(args, peak: float, local: int):
    """The serving step on an fp8 pool, timed like the headline value (K steps back to back on the
    launch stream, > 10 GB of codes per step), and its decode launches back to back (roofline)."""
    import torch
    device = torch.device("cuda", local)
    n_steps = 2 * args.steps + args.warmup
    s = Serve(args.seed, 2 * n_steps + 4, device, fp8=True)
    plan = s.plan_steps(n_steps)
    for i in range(args.warmup):
        s.run_step(plan[i])
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s.stream)
    for k in range(args.steps):
        s.run_step(plan[args.warmup + k])
    b.record(s.stream)
    torch.cuda.synchronize()
    t_step = a.elapsed_time(b) / args.steps
    kv = sum(s.kv_bytes(plan[args.warmup + k][3]) for k in range(args.steps)) / args.steps
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r0.record(s.stream)
    for k in range(args.steps):
        _, tab, ln, _ = plan[args.warmup + args.steps + k]
        for l in range(s.L):
            s.decode(l, tab, ln)
    r1.record(s.stream)
    torch.cuda.synchronize()
    assert s.pkv.last_error() == s.pkv.OK
    dec_ms = r0.elapsed_time(r1) / (args.steps * s.L)
    dec_bytes = sum(s.kv_bytes(plan[args.warmup + args.steps + k][3]) for k in range(args.steps)) / (args.steps * s.L)
    ach = dec_bytes / (dec_ms * 1e-3) / 1e9
    e = {"workload": "serve256_fp8", "ms_per_step": round(t_step, 4), "kv_gb_per_step": round(kv / 1e9, 3),
         "gb_per_s": round(kv / (t_step * 1e-3) / 1e9, 1),
         "seq_steps_per_s": round(s.n / (t_step * 1e-3), 1),
         "roofline": {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                      "frac": round(ach / peak, 4), "mean_launch_us": round(1e3 * dec_ms, 2),
                      "kernel": "paged_decode_kernel<Fp8Math<4,3>,128,4,false>", "traffic": None},
         "timing": f"{args.steps} steps back to back (32 layers of cache write + decode each), inputs larger "
                   "than L2; roofline = decode launches of the next steps back to back"}
    rec = decode_traffic_record("serve256_fp8")
    if rec is not None:   # ncu DRAM bytes of one decode launch, scaled to this launch's bytes
        e["roofline"]["traffic"] = int(rec["bytes_per_launch_profile"] * dec_bytes / rec["algorithmic_bytes_profile"])
    del s
    torch.cuda.empty_cache()
    return e


def bench_workloads(args, local: int):
    """Every workload of the benchmark set, one entry each (see decode_entry / fp8_step_entry /
    prefill_entry), with the clocks seen while they ran."""
    import torch
    peak, _ = measured_peaks()
    flush = L2Flush(torch.device("cuda", local))
    out = {}
    with ClockSampler(local) as clocks:
        out["tiny_f32"] = decode_entry("tiny_f32", args.seed, peak, flush)
        out["gqa5_bf16"] = decode_entry("gqa5_bf16", args.seed, peak, flush)
        out["prefix_cow_bf16"] = decode_entry("prefix_cow_bf16", args.seed, peak, flush)
        out["prefix_cow_bf16_cascade"] = decode_entry("prefix_cow_bf16", args.seed, peak, flush, cascade=True)
        out["long_split_bf16"] = decode_entry("long_split_bf16", args.seed, peak, flush)
        out["long_split_bf16_balanced"] = decode_entry("long_split_bf16", args.seed, peak, flush, partition_tokens=0)
        out["serve256_fp8"] = fp8_step_entry(args, peak, local)
        out["prefill_bf16"] = prefill_entry(args)
    out["clocks"] = clocks.summary()
    return out


def profile_decode(args):
    """Small case for ncu: one layer of a decode workload, decode x5. serve256_bf16 (default; about
    0.8 GB of bf16 KV, above L2), serve256_fp8 (the fp8 pool), gqa5_bf16, tiny_f32, prefix_cow_bf16
    (128 children sharing a 1,024-token prompt: logical bytes above DRAM bytes) or long_split_bf16
    (8 x 32,768 tokens, 512-token partitions as the workload states; pool cut to twice its pages)."""
    fp8 = args.workload == "serve256_fp8"
    name = WORKLOAD if fp8 else args.workload
    p = DecodeProblem(name, args.seed, fp8=fp8, full_pool=False, cascade=args.cascade)
    for _ in range(5):
        p.run()
    p.torch.cuda.synchronize()
    assert p.pkv.last_error() == p.pkv.OK
    print(json.dumps({"profile_decode": args.workload, "layers": 1, "kv_bytes_per_launch": p.kv_bytes, "NB": p.NB,
                      "partition_tokens": p.pt, "cascade": args.cascade}))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload entries (every other benchmark configuration) of the line")
    ap.add_argument("--nvtx", action="store_true", help="one NVTX range per layer in the timed steps")
    ap.add_argument("--workload", choices=[WORKLOAD, "serve256_fp8", "prefill_bf16", "prefix_cow_bf16",
                                           "long_split_bf16", "gqa5_bf16", "tiny_f32"], default=WORKLOAD,
                    help="serve256_bf16 (the benchmark line), serve256_fp8 (the same step on an fp8 pool) or "
                         "prefill_bf16 (causal prefill kernel line)")
    ap.add_argument("--cascade", action="store_true",
                    help="with --profile-decode --workload prefix_cow_bf16: the shared-prefix entry point")
    ap.add_argument("--profile-decode", action="store_true",
                    help="run one layer's decode 5 times (small case for ncu); prints no bench line")
    args = ap.parse_args(argv)
    if args.profile_decode:
        return profile_decode(args)
    if args.workload in ("prefix_cow_bf16", "long_split_bf16", "gqa5_bf16", "tiny_f32"):
        ap.error(f"--workload {args.workload} is a --profile-decode case (the bench line is serve256_bf16)")
    if args.workload == "prefill_bf16":
        return bench_prefill(args)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    if args.impl == "reference":
        bench_reference(args, world, rank)
    else:
        bench_cuda(args, world, rank, local)


if __name__ == "__main__":
    main()

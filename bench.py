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
        for l in range(self.L):
            if self.fp8:
                self.pool.reshape_and_cache_fp8(self.k_new[l], self.v_new[l], slots, self.k_caches[l],
                                                self.v_caches[l], self.k_scales[l], self.v_scales[l],
                                                stream=self.stream)
            else:
                self.pool.reshape_and_cache(self.k_new[l], self.v_new[l], slots, self.k_caches[l], self.v_caches[l],
                                            stream=self.stream)
            self.decode(l, tables, lens)
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
        "config": {
            "workload": args.workload,
            "description": synth.workload(WORKLOAD).description + (
                "; fp8 E4M3 pool with per-(token, head) scales (KV bytes = codes + scales)" if fp8 else ""),
            "n_seqs": s.n, "layers": s.L, "num_q_heads": s.Hq, "num_kv_heads": s.Hkv, "head_dim": s.D,
            "block_size": s.B, "mean_context": float(np.mean(plan[args.warmup][3])),
            "kv_gb_per_step": round(kv_bytes / args.steps / 1e9, 3),
            "l2": "inputs larger than L2 (every step reads all KV of 32 layers, >20 GB)",
            "parallelism": f"replicas x{world}", "partition": "balanced split (partition_tokens=0)",
        },
        "seq_steps_per_s": round(seq_steps_all / (t_ms_max * 1e-3), 1),
        "pct_of_hbm_peak": round(100.0 * value / (peak * world), 2),
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
        "config": {"workload": WORKLOAD, "description": w.description, "n_seqs": w.n_seqs, "layers": w.n_layers},
        "seq_steps_per_s": round(float(np.median(ss_list)), 3),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def bench_prefill(args):
    """Causal paged prefill (prefill_bf16): every position of 16 x 2,048-token prompts is a query.
    Reports useful attention TFLOP/s (4 * D per (query row, attended key): q.K and p.V) against the
    measured dense bf16 tensor peak, and KV bytes per launch."""
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
    for _ in range(args.warmup):
        pool.paged_prefill(out, q, kc, vc, t_tab, t_len, cu, w.scale)
    torch.cuda.synchronize()
    Ev = lambda: torch.cuda.Event(enable_timing=True)
    a, b = Ev(), Ev()
    with ClockSampler(0) as clocks:
        a.record()
        for _ in range(args.steps):
            pool.paged_prefill(out, q, kc, vc, t_tab, t_len, cu, w.scale)
        b.record()
        torch.cuda.synchronize()
    assert pkv.last_error() == pkv.OK
    t = a.elapsed_time(b) / args.steps * 1e-3
    keys = sum(int(L) * (int(L) + 1) // 2 for L in lens)          # attended (row, key) pairs per head
    flops = 4.0 * w.head_dim * keys * w.num_q_heads
    kv_bytes = int(lens.sum()) * w.num_kv_heads * w.head_dim * 2 * 2
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        peak = float(json.load(f)["bf16_tflops"])
    tf = flops / t / 1e12
    print(json.dumps({
        "metric": "paged-prefill causal attention TFLOP/s (useful FLOPs)", "value": round(tf, 2), "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 4),
        "higher_is_better": True, "dtype": "bf16", "accumulate": "f32", "data": "synthetic",
        "config": {"workload": "prefill_bf16", "description": w.description},
        "kv_gb_per_s": round(kv_bytes / t / 1e9, 1),
        "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(tf / peak, 4), "note": "mma.sync m16n8k16; P carried as bf16 hi + lo (2 mmas)"},
        "clocks": clocks.summary()}), flush=True)


def _profile_pool(pkv, args, fp8: bool):
    """Pool, block tables and lengths of the workload a --profile-decode run uses (one layer)."""
    name = {"serve256_fp8": WORKLOAD}.get(args.workload, args.workload)
    w = synth.workload(name)
    lens = synth.lengths(w, args.seed)
    dtype = pkv.FP8 if fp8 else pkv.BF16
    if w.length_kind == "prefix":
        # one prompt forked into every child, the prompt released, each child's suffix appended:
        # the children share the prompt's blocks (the shared-prefix workload)
        NB = synth.pool_blocks(w, lens)
        MB = -(-int(lens.max()) // w.block_size) + 1
        pool = pkv.Pool(1, w.num_kv_heads, w.head_dim, w.block_size, NB, w.n_seqs + 1, MB, dtype,
                        initial_free_list=synth.free_list(NB, args.seed))
        root = None
        kids = []
        for op in synth.prefix_trace(w, args.seed):
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
        NB = synth.pool_blocks(w, lens) if w.pool_rule != "bytes:80e9" else 2 * pages
        MB = -(-int(lens.max()) // w.block_size) + 1
        pool = pkv.Pool(1, w.num_kv_heads, w.head_dim, w.block_size, NB, w.n_seqs, MB, dtype,
                        initial_free_list=synth.free_list(NB, args.seed))
        seqs = [pool.alloc(-1, int(t))[0] for t in lens]
    tables, l = pool.block_table(seqs)
    return w, pool, NB, tables, l


def profile_decode(args):
    """Small case for ncu: one layer of a decode workload, decode x5. serve256_bf16 (default; about
    0.8 GB of bf16 KV, above L2), serve256_fp8 (the fp8 pool), prefix_cow_bf16 (128 children sharing
    a 1,024-token prompt: logical bytes above DRAM bytes) or long_split_bf16 (8 x 32,768 tokens,
    512-token partitions as the workload states)."""
    import torch
    import paged_kv_cache_494_b300 as pkv
    fp8 = args.workload == "serve256_fp8"
    w, pool, NB, tables, l = _profile_pool(pkv, args, fp8)
    g = torch.Generator(device="cuda").manual_seed(args.seed)
    shape = (NB, w.num_kv_heads, w.block_size, w.head_dim)
    if fp8:
        ks_, vs_, ss_ = pool.fp8_shapes()
        kc = torch.randint(0, 0x7E, ks_, device="cuda", dtype=torch.uint8, generator=g)
        vc = torch.randint(0, 0x7E, vs_, device="cuda", dtype=torch.uint8, generator=g)
        ksc = torch.rand(ss_, device="cuda", generator=g) * 0.01
        vsc = torch.rand(ss_, device="cuda", generator=g) * 0.01
    else:
        kc = torch.randn(shape, device="cuda", dtype=torch.bfloat16, generator=g)
        vc = torch.randn(shape, device="cuda", dtype=torch.bfloat16, generator=g)
    n = len(l)
    q = torch.randn(n, w.num_q_heads, w.head_dim, device="cuda", dtype=torch.bfloat16, generator=g)
    out = torch.empty(n, w.num_q_heads, w.head_dim, device="cuda")
    pt = w.partition_tokens
    ws = torch.empty(pool.decode_workspace_bytes(n, w.num_q_heads, pt) // 4 + 4, device="cuda")
    t_tab, t_len = torch.from_numpy(tables).cuda(), torch.from_numpy(l).cuda()
    for _ in range(5):
        if fp8:
            pool.paged_decode_fp8(out, q, kc, vc, ksc, vsc, t_tab, t_len, w.scale, 0, pt, ws)
        else:
            pool.paged_decode(out, q, kc, vc, t_tab, t_len, w.scale, pt, ws)
    torch.cuda.synchronize()
    assert pkv.last_error() == pkv.OK
    per = (w.head_dim + 4) * 2 if fp8 else w.head_dim * 2 * 2
    kv = int(l.sum()) * w.num_kv_heads * per
    print(json.dumps({"profile_decode": args.workload, "layers": 1, "kv_bytes_per_launch": kv, "NB": NB,
                      "partition_tokens": pt}))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=[WORKLOAD, "serve256_fp8", "prefill_bf16", "prefix_cow_bf16",
                                           "long_split_bf16"], default=WORKLOAD,
                    help="serve256_bf16 (the benchmark line), serve256_fp8 (the same step on an fp8 pool) or "
                         "prefill_bf16 (causal prefill kernel line)")
    ap.add_argument("--profile-decode", action="store_true",
                    help="run one layer's decode 5 times (small case for ncu); prints no bench line")
    args = ap.parse_args(argv)
    if args.profile_decode:
        return profile_decode(args)
    if args.workload in ("prefix_cow_bf16", "long_split_bf16"):
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

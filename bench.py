#!/usr/bin/env python
"""Benchmark of the paged decode hot path on GB300.

One step = one pass of the whole decode path over the batch: the host
allocator reserves every sequence's next slot (new block when full,
copy-on-write when shared), slots/tables go to the device, block copies run,
the new keys/values are appended, and paged decode (split-K + log-sum-exp
merge) attends over the grown contexts.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

Prints one JSON line (rank 0).  ``value`` is KV-read GB/s of whole steps
(algorithmic KV bytes: every context token's key and value row read once per
step) with the step inputs resident in HBM; ``e2e`` is the same metric with
each step's new tokens copied from pinned host memory and the output copied
back inside the timed region.  ``--impl reference`` times the CPU oracle on
a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import WORKLOADS, context_lens, free_order, pool_blocks, queries, random_pool  # noqa: E402
from workloads import normal, serving_step_tokens  # noqa: E402

DEFAULT_WORKLOAD = "long_bf16"
METRIC = "paged-decode KV-read GB/s"
UNIT = "GB/s"


def kv_bytes(ctx: np.ndarray, w, groups=None, partition_size: int = 0, elem_bytes: int | None = None) -> int:
    """Algorithmic KV bytes of one decode step: every context token's key and
    value row per KV head (``elem_bytes`` per element: the workload's, or 1
    for an E4M3 cache); with prefix groups, the tokens of a group's shared
    partitions once for the whole group."""
    ctx = np.asarray(ctx, dtype=np.int64)
    tokens = int(ctx.sum())
    for first, count, prefix in (groups or ()):
        shared = np.minimum(ctx[first:first + count], prefix // partition_size * partition_size)
        tokens -= int(shared.sum()) - int(shared.max())
    return tokens * w.num_kv_heads * w.head_dim * 2 * (w.elem_bytes if elem_bytes is None else elem_bytes)


DECODE_SOURCES = ("paged_kv_cache_216_gb300/csrc/decode_tc.cu", "paged_kv_cache_216_gb300/csrc/device_common.cuh",
                  "paged_kv_cache_216_gb300/csrc/kernels.h", "paged_kv_cache_216_gb300/csrc/block_layout.cuh")
DECODE_FP8_SOURCES = ("paged_kv_cache_216_gb300/csrc/decode_fp8.cu", "paged_kv_cache_216_gb300/csrc/device_common.cuh",
                      "paged_kv_cache_216_gb300/csrc/kernels.h")


def strip_comments(src: str) -> str:
    """C/C++ source without its comments, blank lines and runs of spaces
    (string literals are kept), so that a comment edit does not count as a
    kernel change."""
    import re

    pat = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\])*"', re.S)
    out = pat.sub(lambda m: m.group(0) if m.group(0).startswith('"') else "", src)
    return "\n".join(" ".join(line.split()) for line in out.splitlines() if line.strip())


def decode_kernel_hash(sources=DECODE_SOURCES, read=None) -> str:
    """Hash of the decode kernel's sources, comments left out: DRAM counters
    taken on another version of the kernel are not reported.  `read(rel)`
    may supply a file's text (default: the working tree)."""
    import hashlib

    h = hashlib.sha256()
    for rel in sources:
        if read is None:
            with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
                text = f.read()
        else:
            text = read(rel)
        h.update(strip_comments(text).encode("utf-8"))
    return h.hexdigest()[:16]


def decode_traffic(workload: str, fp8: bool = False):
    """DRAM bytes (read + write) of one decode-kernel launch on this workload
    from the committed ncu summary profiles/decode_dram_traffic.txt (lines:
    workload read_bytes write_bytes source_hash), or None if absent or taken
    on another version of the kernel."""
    p = os.path.join(ROOT, "profiles", "decode_dram_traffic.txt")
    if not os.path.exists(p):
        return None
    cur = decode_kernel_hash(DECODE_FP8_SOURCES if fp8 else DECODE_SOURCES)
    if fp8:
        workload = workload + "/fp8"
    with open(p) as f:
        for line in f:
            parts = line.split("#", 1)[0].split()
            if len(parts) == 4 and parts[0] == workload and parts[3] == cur:
                return int(float(parts[1]) + float(parts[2]))
    return None


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f)
    return {}


def smi_gpu_id(device: int) -> str:
    """The identifier nvidia-smi knows this process's CUDA device ``device``
    by.  nvidia-smi numbers GPUs physically and ignores CUDA_VISIBLE_DEVICES,
    so the CUDA ordinal is not it: use the device's UUID, else its PCI
    address, else the ordinal mapped through CUDA_VISIBLE_DEVICES."""
    try:
        import torch

        props = torch.cuda.get_device_properties(device)
        uuid = str(getattr(props, "uuid", "") or "")
        if uuid:
            return uuid if uuid.startswith(("GPU-", "MIG-")) else "GPU-" + uuid
        if hasattr(props, "pci_bus_id"):
            return f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
    except Exception:
        pass
    vis = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    if device < len(vis):
        return vis[device]
    return str(device)


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.proc = None
        self.path = None
        self.gpu = smi_gpu_id(device)
        exe = shutil.which("nvidia-smi")
        if exe:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen([exe, "-i", self.gpu, "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)

    def stop(self) -> dict:
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": sorted(reasons),
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
                if any(r[3].replace(".", "").isdigit() for r in rows) else None}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        import torch

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def allreduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def allreduce_sum(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def workload_for(name: str, rank: int):
    w = WORKLOADS[name]
    return w.replace(seed=w.seed + 1000 * rank) if rank else w


def _host_tokens(w, steps):
    """Per-step new tokens (q, k, v) as numpy bf16 bits / fp32."""
    return [serving_step_tokens(w, i) for i in range(steps)]


def run_ours(args, rank, world, local):
    import torch

    import paged_kv_cache_216_gb300 as pa
    from paged_kv_cache_216_gb300 import build
    from paged_kv_cache_216_gb300.prefix import populate

    build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workload_for(args.workload, rank)
    if args.partition_size is not None:
        w = w.replace(partition_size=args.partition_size)
    K, W = args.steps, args.warmup
    Kp = K + (K % 2)  # untimed pass that launches every per-step graph once (even: same buffer parity)
    # warm-up, graph warm-up, timed run, roofline warm-up, roofline run, end-to-end run
    total_steps = W + 2 + K + Kp + K + K
    ctx0 = context_lens(w)
    nb = pool_blocks(w, ctx0, extra_steps=total_steps) + w.prefix_share
    order = free_order(w, nb)

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    k_cache = to_dev(random_pool(w, nb, "k"))
    v_cache = to_dev(random_pool(w, nb, "v"))
    fp8 = args.kv_dtype == "fp8"
    kv_scales = None
    if fp8:
        # E4M3 caches: the pools are stored through the append kernel, one
        # slot per token row; new tokens are quantized the same way each step
        kv_scales = (w.std / 32.0, w.std / 32.0)
        n_, h_, b_, d_ = k_cache.shape
        slots = torch.arange(n_ * b_, dtype=torch.int64, device=dev)
        codes = []
        for src in (k_cache, v_cache):
            dst = torch.zeros(src.shape, dtype=torch.uint8, device=dev)
            codes.append(dst)
        pa.cache_append_fp8(k_cache.permute(0, 2, 1, 3).reshape(n_ * b_, h_, d_).contiguous(),
                            v_cache.permute(0, 2, 1, 3).reshape(n_ * b_, h_, d_).contiguous(), slots, codes[0],
                            codes[1], *kv_scales)
        torch.cuda.synchronize()
        del k_cache, v_cache, slots
        torch.cuda.empty_cache()
        k_cache, v_cache = codes
    alloc = pa.BlockAllocator(nb, w.block_size, order)
    pairs = populate(alloc, ctx0, w.prefix_len, w.prefix_share)
    if len(pairs):
        pa.copy_blocks(k_cache, v_cache, to_dev(pairs))
    seq_ids = np.arange(w.num_seqs)
    # the forked sequences share the prefix's whole blocks (its last, partly
    # filled block was copied by each one's first append)
    groups = None
    if w.prefix_share and not args.no_prefix_groups:
        groups = [(0, w.prefix_share, w.prefix_len // w.block_size * w.block_size)]
    if fp8:
        groups = None  # prefix groups are not supported with E4M3 caches
    eng = pa.ServingEngine(k_cache, v_cache, alloc, seq_ids, w.num_heads, w.scale,
                           int(ctx0.max()) + total_steps, w.partition_size, prefix_groups=groups,
                           kv_scales=kv_scales)
    if not eng.split:
        groups = None  # one partition per context: no shared partitions

    def step_bytes(ctx):
        return kv_bytes(ctx, w, groups, eng.partition_size, 1 if fp8 else None)

    toks = _host_tokens(w, total_steps)
    n_dev = W + 2 + K + Kp + K
    dev_toks = [tuple(to_dev(x) for x in t) for t in toks[:n_dev]]
    packed = [eng.pack_tokens(*t) for t in dev_toks]  # each step's new tokens, resident in HBM
    out = torch.empty((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.bfloat16 if fp8 else k_cache.dtype,
                      device=dev)
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = None
    if step_bytes(ctx0) < 2 * l2:
        flush = torch.empty(4 * l2 // 4, dtype=torch.int32, device=dev)
    step = 0  # steps done so far; step j decodes contexts ctx0 + j + 1

    # warm-up (eager steps; they also initialise the library's per-device state)
    for i in range(W):
        if flush is not None:
            flush.add_(1)
        eng.step(*dev_toks[step], out=out)
        step += 1
    torch.cuda.synchronize()

    # Timed run: K steps.  With graph support the main-stream part of a step
    # (append, decode, merge) replays a captured CUDA graph, one per device
    # buffer, reading the step's new tokens from staging buffers that the
    # upload stream fills while the previous step decodes; else steps run
    # eagerly.
    from paged_kv_cache_216_gb300.serving import _event, graphs_supported

    use_graphs = graphs_supported() and not args.eager
    par = eng.capture() if use_graphs else None

    def run_step(i, graphs=None, events=None):
        if use_graphs:
            eng.replay(graphs if graphs is not None else par, packed=packed[i])
        else:
            eng.step(*dev_toks[i], out=out, events=events)

    for _ in range(2):  # launch each graph once before timing
        run_step(step)
        step += 1
    torch.cuda.synchronize()
    T0 = step
    bytes_steps = [step_bytes(ctx0 + T0 + i + 1) for i in range(K)]
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    launches0 = eng.launches
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    if flush is None:
        # The GPU spins for about a millisecond first, so the region opens
        # with the first steps already queued (after that the host runs ahead
        # of the GPU); every step's device work stays inside it.
        torch.cuda._sleep(2_000_000)
        step_ev[0][0].record(stream)
        for i in range(K):
            run_step(T0 + i)
        step_ev[-1][1].record(stream)
    else:
        for i in range(K):
            flush.add_(1)
            step_ev[i][0].record(stream)
            run_step(T0 + i)
            step_ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t_wall
    launches = eng.launches - launches0
    clk = clocks.stop()
    step += K
    assert np.array_equal(eng.ctx_h.numpy(), ctx0 + step)
    if flush is None:
        t_dev = step_ev[0][0].elapsed_time(step_ev[-1][1]) / 1e3
    else:
        t_dev = sum(a.elapsed_time(b) for a, b in step_ev) / 1e3
    local_bytes = float(sum(bytes_steps))
    t_max = allreduce_max(t_dev, world)
    total_bytes = allreduce_sum(local_bytes, world)
    value = total_bytes / t_max / 1e9
    tokens_s = allreduce_sum(float(w.num_seqs * K), world) / t_max

    # Roofline run: K more steps, each replaying its own graph whose timing
    # events bracket the decode (events inside a graph add a few us per
    # step, so the timed run above goes without them); every graph is
    # launched once first.
    dec_ev = [(_event(True), _event(True)) for _ in range(K)]
    if use_graphs:
        gsteps = [eng.capture(events=dec_ev[i], parity=(step + Kp + i) % 2) for i in range(K)]
        for i in range(Kp):
            if i < K and gsteps[i].graphs[eng.k] is not None:
                run_step(step + i, gsteps[i])
            else:
                run_step(step + i)
    else:
        gsteps = [None] * K
        for i in range(Kp):
            run_step(step + i)
    step += Kp
    R0 = step
    dec_bytes = sum(step_bytes(ctx0 + R0 + i + 1) for i in range(K)) / K
    torch.cuda.synchronize()
    for i in range(K):
        run_step(R0 + i, gsteps[i], events=dec_ev[i])
    torch.cuda.synchronize()
    step += K
    t_dec = [a.elapsed_time(b) / 1e3 for a, b in dec_ev]

    # end-to-end run: host (pinned) tokens in, host output back, every step
    def host(x):
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16) if x.dtype == np.uint16 else x)
        return t.view(torch.bfloat16) if x.dtype == np.uint16 else t

    pin = [eng.pack_tokens(*(host(x) for x in t), pin=True) for t in toks[step:step + K]]
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()  # every step's output lands here
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_bytes = sum(step_bytes(ctx0 + step + i + 1) for i in range(K))
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(K):
        if flush is not None:
            flush.add_(1)
        eng.step_host(out_h=out_h, graphs=par, packed=pin[i])
    stream.wait_stream(eng.down_stream)  # the last output copy is part of the timed region
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_e2e = allreduce_max(e0.elapsed_time(e1) / 1e3, world)
    e2e_value = allreduce_sum(float(e2e_bytes), world) / t_e2e / 1e9
    h2d = pin[0].numel() * pin[0].element_size()
    d2h = out_h.numel() * out_h.element_size()

    # roofline of the decode call (main kernel + its merge), from the live events
    dec_avg = sum(t_dec) / len(t_dec)
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or 6800.0
    achieved = dec_bytes / dec_avg / 1e9
    traffic = decode_traffic(args.workload, fp8)
    status = pa.get_status()
    if status:
        raise RuntimeError(f"device status word {status:#x} after the benchmark")

    res = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(t_max / K * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3" if fp8 else w.dtype, "data": "synthetic",
        "config": {
            "workload": w.name, "batch": w.num_seqs, "query_heads": w.num_heads, "kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "block_size": w.block_size, "partition_size": eng.partition_size,
            "context_start_mean": float(ctx0.mean()), "context_start_max": int(ctx0.max()),
            "kv_bytes_per_step": int(local_bytes / K),
            "prefix_groups": groups,
            "kv_bytes_per_step_logical": int(sum(kv_bytes(ctx0 + T0 + i + 1, w, elem_bytes=1 if fp8 else None)
                                                 for i in range(K)) / K),
            "l2": ("flushed before every step" if flush is not None else
                   f"inputs larger than L2 ({local_bytes / K / 1e9:.2f} GB KV per step vs {l2 / 1e6:.0f} MB L2)"),
            "parallelism": f"replicas x{world}",
            "kv_storage": ("E4M3 codes, one scale per cache; f16 tensor-core products, f32 accumulation, bf16 q/out"
                           if fp8 else w.dtype),
            "launch": ("tables and new tokens uploaded on a side stream; append+decode+merge replayed as a "
                       "CUDA graph per device buffer" if use_graphs else "uploads on a side stream; eager launches"),
        },
        "decode_tokens_per_s": round(tokens_s, 1),
        "wall_s": round(wall, 4),
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": launches,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": ("paged_decode_fp8_kernel" if fp8 else
                                "paged_decode_tc_kernel (with shared-prefix items)" if groups
                                else "paged_decode_tc_kernel") + (" + lse_merge_kernel" if eng.split else ""),
                     "peak_source": f"{peak_src} hbm_gbs", "decode_ms": round(dec_avg * 1e3, 4),
                     "timing": f"CUDA events inside each step's graph, {K} steps after the timed run"},
        "clocks": clk,
    }
    return res, eng, w


def oracle_sample(w, budget_s: float):
    """Time the CPU oracle on a bounded sample of the workload: decode of as
    many whole sequences as fit the time budget.  Returns (GB/s, sample
    description, threads)."""
    from oracle.attention import paged_decode
    from oracle.serving import initial_state, tables_array

    ctx = context_lens(w)
    nb = pool_blocks(w, ctx) + w.prefix_share
    order = free_order(w, nb)
    alloc, _ = initial_state(w.num_seqs, w.block_size, ctx, nb, order, w.prefix_len, w.prefix_share)
    tables = tables_array(alloc, range(w.num_seqs), -(-int(ctx.max()) // w.block_size))
    kp = random_pool(w, nb, "k")
    vp = random_pool(w, nb, "v")
    q = queries(w)
    done, t, nbytes = 0, 0.0, 0
    rng = np.random.default_rng(0)
    order_s = rng.permutation(w.num_seqs)
    while t < budget_s and done < 100 * w.num_seqs:
        s = int(order_s[done % w.num_seqs])
        t0 = time.perf_counter()
        paged_decode(q, kp, vp, tables, ctx, w.scale, w.dtype, seqs=[s])
        t += time.perf_counter() - t0
        nbytes += kv_bytes(ctx[[s]], w)
        done += 1
    gbs = nbytes / t / 1e9
    desc = (f"oracle decode of {done} sequences (cycling over the {w.num_seqs} of the batch; "
            f"{nbytes / 1e6:.1f} MB of KV) in {t:.1f} s")
    return gbs, desc, t


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, rank, world):
    if rank != 0:
        return None
    if args.prefill:
        return run_reference_prefill(args, world)
    w = WORKLOADS[args.workload]
    vals = []
    desc = ""
    for _ in range(args.steps):
        gbs, desc, _ = oracle_sample(w, budget_s=max(1.0, args.ref_budget / max(1, args.steps)))
        vals.append(gbs)
    value = statistics.median(vals)
    res = {
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": w.name, "batch": w.num_seqs, "query_heads": w.num_heads,
                   "kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return res


PREFILL_SHAPE = dict(num_seqs=8, cached=512, new=512, num_heads=32, num_kv_heads=8, head_dim=128, block_size=16)


def _ragged_prefill_shape():
    """8 prompts of U[64, 2048] new tokens after U[0, 4096] cached ones
    (seeded), heads and blocks as PREFILL_SHAPE."""
    rng = np.random.default_rng(3)
    cached = [int(x) for x in rng.integers(0, 4097, size=8)]
    new = [int(x) for x in rng.integers(64, 2049, size=8)]
    return dict(PREFILL_SHAPE, cached=cached, new=new)


PREFILL_RAGGED_SHAPE = _ragged_prefill_shape()


def _prefill_shape(args):
    return PREFILL_RAGGED_SHAPE if getattr(args, "prefill_ragged", False) else PREFILL_SHAPE


def _per_seq(sh):
    S = sh["num_seqs"]
    as_list = lambda x: [int(v) for v in x] if isinstance(x, (list, tuple)) else [int(x)] * S
    return as_list(sh["cached"]), as_list(sh["new"])


def prefill_batch(seed: int = 11, **shape):
    """Seeded synthetic prefill batch: sequence s has `cached` tokens in the
    pool and `new` prompt tokens to append and attend (one value for every
    sequence, or one per sequence); shuffled tables."""
    sh = dict(PREFILL_SHAPE, **shape)
    S, H, Hkv, D, B = (sh[k] for k in ("num_seqs", "num_heads", "num_kv_heads", "head_dim", "block_size"))
    cached, new = _per_seq(sh)
    rng = np.random.default_rng(seed)
    nb = [-(-(c + n) // B) for c, n in zip(cached, new)]
    N = sum(nb) + 8
    perm = rng.permutation(N).astype(np.int32)
    tables = np.zeros((S, max(nb)), dtype=np.int32)
    slots = []
    at = 0
    for s in range(S):
        tables[s, :nb[s]] = perm[at:at + nb[s]]
        at += nb[s]
        pos = cached[s] + np.arange(new[s])
        slots.append(tables[s, pos // B] * B + pos % B)
    T = sum(new)
    return dict(q=normal((T, H, D), 1.0, "bf16", seed, 31), k=normal((T, Hkv, D), 1.0, "bf16", seed, 32),
                v=normal((T, Hkv, D), 1.0, "bf16", seed, 33), kc=normal((N, Hkv, B, D), 1.0, "bf16", seed, 34),
                vc=normal((N, Hkv, B, D), 1.0, "bf16", seed, 35), slots=np.concatenate(slots).astype(np.int64),
                tables=tables, qs=np.r_[0, np.cumsum(new)].astype(np.int32),
                ctx=np.array([c + n for c, n in zip(cached, new)], dtype=np.int32), shape=sh,
                scale=1.0 / np.sqrt(D))


def prefill_flops(b) -> float:
    """Attention FLOPs of a prefill call: each new token's query head does
    2·D flops per key for Q·Kᵀ and 2·D for P·V over its keys 0..p."""
    sh = b["shape"]
    cached, new = _per_seq(sh)
    keys = sum(n * c + n * (n + 1) // 2 for c, n in zip(cached, new))
    return float(keys) * sh["num_heads"] * sh["head_dim"] * 4


def run_prefill(args, rank, world, local):
    """One prefill call per step (append of every sequence's prompt plus its
    causal attention) on the synthetic batch; L2 flushed between steps."""
    import torch

    import paged_kv_cache_216_gb300 as pa
    from paged_kv_cache_216_gb300 import build

    build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    b = prefill_batch(seed=11 + rank, **_prefill_shape(args))
    sh = b["shape"]
    cached, new = _per_seq(sh)

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    q, k, v, kc, vc = (to_dev(b[x]) for x in ("q", "k", "v", "kc", "vc"))
    slots, qs, ctx, tables = (to_dev(b[x]) for x in ("slots", "qs", "ctx", "tables"))
    out = torch.empty_like(q)
    mql, mctx = max(new), int(b["ctx"].max())

    def call(qq=q, kk=k, vv=v, oo=out):
        pa.prefill(qq, kk, vv, slots, qs, ctx, tables, mql, mctx, b["scale"], kc, vc, out=oo)

    K, W = args.steps, args.warmup
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(4 * l2 // 4, dtype=torch.int32, device=dev)
    for _ in range(W):
        flush.add_(1)
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    for i in range(K):
        flush.add_(1)
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    t_dev = allreduce_max(sum(a.elapsed_time(z) for a, z in ev) / 1e3, world)
    flops = prefill_flops(b)
    value = allreduce_sum(flops * K, world) / t_dev / 1e12
    # end to end: inputs from pinned host memory, output back, every step
    def pin(a):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        return t.pin_memory()

    hq, hk, hv = pin(b["q"]), pin(b["k"]), pin(b["v"])
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(K):
        flush.add_(1)
        q.copy_(hq, non_blocking=True)
        k.copy_(hk, non_blocking=True)
        v.copy_(hv, non_blocking=True)
        call()
        hout.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    t_e2e = allreduce_max(e0.elapsed_time(e1) / 1e3, world)
    status = pa.get_status()
    if status:
        raise RuntimeError(f"device status word {status:#x} after the benchmark")
    peaks = measured_peaks()
    peak = peaks.get("bf16_tflops") or 1900.0
    achieved = flops * K / t_dev / 1e12  # one GPU's calls over the slowest rank's time
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
    res = {
        "metric": "prefill attention TFLOP/s", "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(t_dev / K * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "prefill_ragged_bf16" if args.prefill_ragged else "prefill_bf16", **sh,
                   "tokens_per_step": sum(new),
                   "flops_per_step": flops, "l2": "flushed before every step", "parallelism": f"replicas x{world}"},
        "prefill_tokens_per_s": round(allreduce_sum(float(sum(new) * K), world) / t_dev, 1),
        "e2e": {"value": round(allreduce_sum(flops * K, world) / t_e2e / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(hout.numel() * hout.element_size())},
        "gpu_launches": 2 * K,
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": None, "kernel": "cache_append_kernel + prefill_tc_kernel (tcgen05)",
                     "peak_source": ("measured bf16_tflops" if peaks.get("bf16_tflops") else "fallback")},
        "clocks": clk,
    }
    return res


def prefill_oracle_sample(budget_s: float, shape=None):
    """Oracle prefill on whole sequences of the bench batch for a bounded
    time: TFLOP/s of the sample."""
    from oracle.prefill import prefill as oracle_prefill

    b = prefill_batch(**(shape or PREFILL_SHAPE))
    sh = b["shape"]
    cached, new = _per_seq(sh)
    t0 = time.perf_counter()
    done = 0
    keys = 0
    while time.perf_counter() - t0 < budget_s and done < sh["num_seqs"]:
        q0, q1 = int(b["qs"][done]), int(b["qs"][done + 1])
        rows = slice(q0, q1)
        oracle_prefill(b["q"][rows], b["k"][rows], b["v"][rows], b["slots"][rows], np.array([0, q1 - q0], np.int32),
                       b["ctx"][done:done + 1], b["tables"][done:done + 1], b["kc"], b["vc"], b["scale"], "bf16")
        c, n = cached[done], new[done]
        keys += n * c + n * (n + 1) // 2
        done += 1
    t = time.perf_counter() - t0
    flops = float(keys) * sh["num_heads"] * sh["head_dim"] * 4
    return flops / t / 1e12, f"oracle prefill of {done} of the {sh['num_seqs']} sequences in {t:.1f} s"


def run_reference_prefill(args, world):
    """The reference arm of the prefill benchmark: the oracle on whole
    sequences of the same batch, a bounded sample per step, with our arm's
    metric, unit and workload."""
    vals, desc = [], ""
    for _ in range(args.steps):
        v, desc = prefill_oracle_sample(max(0.5, args.ref_budget / max(1, args.steps)), _prefill_shape(args))
        vals.append(v)
    value = statistics.median(vals)
    sh = _prefill_shape(args)
    return {
        "metric": "prefill attention TFLOP/s", "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": "prefill_ragged_bf16" if args.prefill_ragged else "prefill_bf16", **sh},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--ref-budget", type=float, default=20.0, help="seconds of oracle time in the reference arm")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--eager", action="store_true", help="launch every step's kernels eagerly (no CUDA graph)")
    ap.add_argument("--kv-dtype", choices=["native", "fp8"], default="native",
                    help="store the KV cache as the workload's type or as E4M3 codes")
    ap.add_argument("--partition-size", type=int, default=None,
                    help="split-K partition size in tokens (default: the workload's, 0 = library choice)")
    ap.add_argument("--prefill", action="store_true",
                    help="time prefill (append + causal attention of 8 x 512 new tokens after 512 cached)")
    ap.add_argument("--prefill-ragged", action="store_true",
                    help="time prefill on 8 ragged prompts (U[64, 2048] new tokens after U[0, 4096] cached)")
    ap.add_argument("--no-prefix-groups", action="store_true",
                    help="decode prefix-sharing sequences one by one (no shared-prefix kernel)")
    args = ap.parse_args()
    args.prefill = args.prefill or args.prefill_ragged
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_setup()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if args.prefill:
        res = run_prefill(args, rank, world, local)
        if rank == 0:
            val, desc = prefill_oracle_sample(min(args.cpu_budget, 15.0), _prefill_shape(args))
            res["cpu_baseline"] = {"value": round(val, 6), "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
                                   "sample": desc}
            print(json.dumps(res), flush=True)
        return
    res, eng, w = run_ours(args, rank, world, local)
    if rank == 0:
        gbs, desc, _ = oracle_sample(WORKLOADS[args.workload], args.cpu_budget)
        res["cpu_baseline"] = {"value": round(gbs, 4), "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                               "sample": desc}
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()

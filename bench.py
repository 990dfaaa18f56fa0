"""Benchmark: one decode layer step (append + paged decode attention) per step.

Default workload: Llama-3-8B heads (32 query / 8 kv heads x 128), bf16, 256
sequences with lognormal context lengths (median 1024, sigma 1, cap 8192).
One step appends one new token per sequence at its explicit position and runs
decode attention over context + 1 tokens.  The per-layer K/V (about 1.7 GB)
is far larger than the 129 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs its own
replica on its own GPU (the path shards by sequence; no collective) and the
value is the work of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode-attention achieved HBM GB/s (% of GB300 peak) and decode tokens/s"
NOMINAL_HBM_GBS = 7900.0      # GB300 HBM3e nominal bandwidth (the measured copy peak is lower)
L2_BYTES = 129e6
# workloads whose pool is near L2's size: the timed step runs every layer, each on a pool of its
# own, so L2 cannot serve one layer's cache to the next
ROTATE_LAYERS = {"qwen2.5-0.5b_gqa": 24}
# workloads whose unique K/V fit in L2: consecutive steps cycle through this many copies of the
# pools (as consecutive layers of a model would), so no step finds the previous one's data in L2
STEP_POOLS = {"llama3-8b_shared_prefix": 4}
# tokens every sequence of the workload shares in the same physical blocks
SHARED_TOKENS = {"llama3-8b_shared_prefix": 4096}
LAYERS = {"llama3-8b_batch256": 32, "llama3-8b_long_context": 32, "llama3-8b_shared_prefix": 32,
          "qwen2.5-0.5b_gqa": 24, "gpt2_tiny_f32": 12}


# ---------------------------------------------------------------------------
# distributed plumbing
# ---------------------------------------------------------------------------
def dist_init(n_gpus: int):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        if dist.get_backend() == "nccl":
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def all_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def all_sum(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------
def kv_bytes_per_token(wl, kv_dtype="bf16") -> int:
    """K+V bytes of one token (all kv heads): elements, or E4M3 codes + one fp32 scale
    per (slot, kv head) for the FP8 cache."""
    if kv_dtype == "fp8":
        return 2 * wl.num_kv_heads * (wl.head_dim + 4)
    if kv_dtype == "fp4":            # E2M1 codes + one E8M0 byte per 32 values, K and V
        return 2 * wl.num_kv_heads * (wl.head_dim // 2 + wl.head_dim // 32)
    e = 2 if wl.dtype == "bf16" else 4
    return 2 * wl.num_kv_heads * wl.head_dim * e


def decode_bytes(wl, kv_dtype="bf16") -> int:
    """Bytes one decode launch must move: each K/V element of every context once,
    q and out, the block-table entries and lengths, and the split-KV partials
    (written and read back) of sequences longer than one partition."""
    e = 2 if wl.dtype == "bf16" else 4
    L = wl.context_lens.astype(np.int64) + 1
    kv = int((L * kv_bytes_per_token(wl, kv_dtype)).sum())
    qo = 2 * wl.num_seqs * wl.num_q_heads * wl.head_dim * e
    table = int((4 * ((L + 15) // 16)).sum()) + 4 * wl.num_seqs
    pt = {"fp8": 1024, "fp4": 2048}.get(kv_dtype, 1024 if wl.head_dim == 64 else 512)
    parts = (L + pt - 1) // pt                   # split-KV partitions of each context
    multi = parts[parts > 1]
    partial = int((multi * wl.num_q_heads * (wl.head_dim + 2) * 4 * 2).sum())
    return kv + qo + table + partial


def logical_kv_bytes(wl) -> int:
    e = 2 if wl.dtype == "bf16" else 4
    return int(((wl.context_lens.astype(np.int64) + 1) * 2 * wl.num_kv_heads * wl.head_dim * e).sum())


def unique_kv_bytes(wl, shared: int) -> int:
    """K/V bytes when the shared prefix is counted once (the bytes that exist in the pool)."""
    e = 2 if wl.dtype == "bf16" else 4
    per_token = 2 * wl.num_kv_heads * wl.head_dim * e
    private = (wl.context_lens.astype(np.int64) + 1 - shared).clip(min=0).sum()
    return int((shared + private) * per_token)


def append_bytes(wl, kv_dtype="bf16") -> int:
    """New rows read, and written into the pools, plus start / cu / table reads."""
    e = 2 if wl.dtype == "bf16" else 4
    rows = wl.num_seqs * wl.num_kv_heads * wl.head_dim * e * 2   # K and V read
    return rows + wl.num_seqs * kv_bytes_per_token(wl, kv_dtype) + 12 * wl.num_seqs


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        try:
            props = torch.cuda.get_device_properties(device_index)
            uuid = str(props.uuid)
            self.gpu = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            self.gpu = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "200"]
            if self.gpu:
                cmd += ["-i", self.gpu]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# the CUDA arm
# ---------------------------------------------------------------------------
def load_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


def decode_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("pa_decode.cu", "pa_ptx.cuh", "pa_internal.h"):
        h.update(open(os.path.join(ROOT, "paged_kv_cache_207_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kv_dtype: str = "bf16"):
    """dram bytes per decode launch from a committed ncu summary, if it was taken on
    the current decode source; else None."""
    tag = "" if kv_dtype == "bf16" else kv_dtype + "_"
    path = os.path.join(ROOT, "profiles", f"decode_{tag}{workload}_dram.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        if "=" in line and not line.startswith("#"):
            k, v = line.split("=", 1)
            kv[k.strip()] = v.strip()
    if kv.get("decode_source_sha256_16") != decode_source_hash():
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class PipelinedE2E:
    """End-to-end steps through the public API.  Every step copies its inputs in from pinned
    host memory and its result back, both inside the timed region.  The inputs sit in one
    pinned buffer (256-byte aligned segments) and go over in one copy.  The copies run on a
    stream per direction into two sets of device buffers, so step i + 1's inputs load while
    step i computes and step i's result returns while step i + 1 runs (a copy in queued
    behind a copy back would wait for the compute); events order each buffer's reuse."""

    def __init__(self, srcs, out, stream):
        self.stream = stream
        offs, total = [], 0
        for t in srcs:
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256

        def views(buf):
            return tuple(buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                         for o, t in zip(offs, srcs))
        self.h_in = torch.empty(total, dtype=torch.uint8).pin_memory()
        for dst, src in zip(views(self.h_in), srcs):
            dst.copy_(src.cpu())
        self.d_in = [torch.empty(total, dtype=torch.uint8, device="cuda") for _ in range(2)]
        self.bufs = [views(b) for b in self.d_in]
        self.outs = [torch.empty_like(out) for _ in range(2)]
        self.h_outs = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        self.h2d = sum(t.numel() * t.element_size() for t in srcs)
        self.d2h = out.numel() * out.element_size()
        self.in_stream, self.back_stream = torch.cuda.Stream(), torch.cuda.Stream()
        self.loaded = [torch.cuda.Event() for _ in range(2)]     # inputs of set b are in
        self.computed = [torch.cuda.Event() for _ in range(2)]   # the step using set b is done
        self.returned = [torch.cuda.Event() for _ in range(2)]   # output b is back on the host
        self.used = [False, False]

    def step(self, i, compute):
        """compute(device_inputs, device_out) enqueues the step's kernels on self.stream."""
        b = i & 1
        with torch.cuda.stream(self.in_stream):
            if self.used[b]:
                self.in_stream.wait_event(self.computed[b])      # step i - 2 is done with set b
            self.d_in[b].copy_(self.h_in, non_blocking=True)
            self.loaded[b].record(self.in_stream)
        self.stream.wait_event(self.loaded[b])
        if self.used[b]:
            self.stream.wait_event(self.returned[b])             # output b of step i - 2 is home
        compute(self.bufs[b], self.outs[b])
        self.computed[b].record(self.stream)
        with torch.cuda.stream(self.back_stream):
            self.back_stream.wait_event(self.computed[b])
            self.h_outs[b].copy_(self.outs[b], non_blocking=True)
            self.returned[b].record(self.back_stream)
        self.used[b] = True

    def run(self, compute, warmup, steps, world=1):
        """Returns (device ms per step, max over ranks; the host's enqueue ms per step; the
        last step's output as copied back)."""
        for i in range(warmup):
            self.step(i, compute)
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.in_stream)
        self.stream.wait_event(e0)
        self.back_stream.wait_event(e0)
        th = time.perf_counter()
        for i in range(steps):
            self.step(i, compute)
        host_ms = (time.perf_counter() - th) * 1e3 / steps
        self.in_stream.wait_stream(self.stream)
        self.in_stream.wait_stream(self.back_stream)
        e1.record(self.in_stream)
        torch.cuda.synchronize()
        barrier(world)
        return all_max(e0.elapsed_time(e1), world) / steps, host_ms, self.h_outs[(steps - 1) & 1]


def run_ours(args, rank, world, local):
    import paged_kv_cache_207_gb300 as pk
    from paged_kv_cache_207_gb300 import build, workloads as W

    torch.cuda.set_device(local)
    build.build()
    pk.lib()
    kw = {}
    if args.workload == "llama3-8b_batch256":
        kw["seed"] = 210 + 1000 * rank
    if args.num_seqs:
        kw["num_seqs"] = args.num_seqs
    wl = W.WORKLOADS[args.workload](device="cuda", **kw)
    tdt = wl.torch_dtype()
    S, Hq, Hkv, D = wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    quant = args.kv_dtype if args.kv_dtype in ("fp8", "fp4") else None
    if quant and wl.dtype != "bf16":
        raise SystemExit("the quantised caches take bf16 rows")
    if quant:
        shape = (pk.fp8_pool_shape if quant == "fp8" else pk.fp4_pool_shape)(wl.num_blocks, Hkv, D)
        kp = torch.zeros(shape, dtype=torch.uint8, device="cuda")
        vp = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    else:
        shape = pk.pool_shape(wl.num_blocks, Hkv, D, tdt)
        kp = torch.zeros(shape, dtype=tdt, device="cuda")
        vp = torch.zeros(shape, dtype=tdt, device="cuda")
    append = {"fp8": pk.append_kv_fp8, "fp4": pk.append_kv_fp4}.get(quant, pk.append_kv)
    tables = torch.from_numpy(wl.block_tables).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # fill the context (untimed set-up), one append call
    seqs = [f[0] for f in wl.fill]
    ns = [f[3] for f in wl.fill]
    first, end = wl.fill[0][2], wl.fill[-1][2] + wl.fill[-1][3]
    append(kp, vp, wl.k_rows[first:end].contiguous(), wl.v_rows[first:end].contiguous(),
                 tables[torch.tensor(seqs, device="cuda")].contiguous(),
                 torch.tensor([f[1] for f in wl.fill], dtype=torch.int32, device="cuda"),
                 torch.tensor(np.concatenate([[0], np.cumsum(ns)]), dtype=torch.int32, device="cuda"),
                 err_flag=err)
    rows = torch.from_numpy(wl.new_rows).cuda()
    k_new = wl.k_rows[rows].contiguous()
    v_new = wl.v_rows[rows].contiguous()
    start = torch.from_numpy(wl.context_lens.astype(np.int32)).cuda()
    cu = torch.arange(S + 1, dtype=torch.int32, device="cuda")
    lens = start + 1
    q = wl.q.contiguous()
    out = torch.empty_like(q)
    ws = pk.decode_workspace(S, Hq, Hkv, D, wl.max_blocks)
    hint = int(lens.max().item())
    del wl.k_rows, wl.v_rows
    torch.cuda.empty_cache()
    stream = torch.cuda.current_stream()
    rot = ROTATE_LAYERS.get(args.workload, 1)
    npools = rot * STEP_POOLS.get(args.workload, 1)
    pools = [(kp, vp)] + [(kp.clone(), vp.clone()) for _ in range(npools - 1)]
    pool_bytes = 2 * npools * kp.numel() * kp.element_size()
    counter = [0]          # steps issued so far: step i, layer l uses pool (i rot + l) % npools

    shared = args.shared_prefix
    # the bf16, f32 and FP8 caches take the step as one call (the decode kernel writes the
    # new token itself, with or without a shared prefix); the FP4 path appends, then decodes
    fused = quant != "fp4"

    def append_decode(q_, kn, vn, tab_, lens_, pool, out=out, strm=stream):
        kp, vp = pools[pool]
        if quant == "fp8":
            pk.append_decode_attention_fp8(out, q_, kp, vp, kn, vn, tab_, lens_, wl.scale,
                                           workspace=ws, max_context_len_hint=hint, err_flag=err,
                                           stream=strm)
        elif shared:
            pk.append_decode_attention_shared_prefix(out, q_, kp, vp, kn, vn, tab_, lens_, wl.scale,
                                                     shared, workspace=ws,
                                                     max_context_len_hint=hint, err_flag=err,
                                                     stream=strm)
        else:
            pk.append_decode_attention(out, q_, kp, vp, kn, vn, tab_, lens_, wl.scale,
                                       workspace=ws, max_context_len_hint=hint, err_flag=err,
                                       stream=strm)

    def decode(q_, tab_, lens_, pool, out=out, strm=stream):
        kp, vp = pools[pool]
        if quant:
            dec = pk.decode_attention_fp8 if quant == "fp8" else pk.decode_attention_fp4
            dec(out, q_, kp, vp, tab_, lens_, wl.scale, workspace=ws, max_context_len_hint=hint,
                err_flag=err, stream=strm)
        elif shared:
            pk.decode_attention_shared_prefix(out, q_, kp, vp, tab_, lens_, wl.scale, shared,
                                              workspace=ws, max_context_len_hint=hint,
                                              err_flag=err, stream=strm)
        else:
            pk.decode_attention(out, q_, kp, vp, tab_, lens_, wl.scale, workspace=ws,
                                max_context_len_hint=hint, err_flag=err, stream=strm)

    def step(ev_d0=None, ev_d1=None, strm=stream):
        base = counter[0] * rot
        counter[0] += 1
        for layer in range(rot):
            pool = (base + layer) % npools
            if not fused:
                append(*pools[pool], k_new, v_new, tables, start, cu, err_flag=err, stream=strm)
            if ev_d0 is not None:
                ev_d0[layer].record(strm)
            if fused:
                append_decode(q, k_new, v_new, tables, lens, pool, strm=strm)
            else:
                decode(q, tables, lens, pool, strm=strm)
            if ev_d1 is not None:
                ev_d1[layer].record(strm)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error flag {int(err.item())} during warm-up")

    # The timed steps replay CUDA graphs of the same calls (one per phase of the pool
    # rotation), as a serving loop would, so that host launch time does not pace short steps;
    # without graph support (or with --no-graphs) they are launched directly.  The
    # shared-prefix call is always launched directly: its prefix and suffix kernels run side
    # by side through programmatic dependent launch, and replayed from a graph its step took
    # 28.4 us against 24.3 us (GB300).
    period = npools // math.gcd(rot, npools)
    graphs = []
    if not args.no_graphs and not shared:
        try:
            for j in range(period):
                counter[0] = j
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, capture_error_mode="relaxed"):
                    step(strm=None)                   # (the capture stream)
                graphs.append(g)
            for g in graphs:
                g.replay()
            torch.cuda.synchronize()
        except Exception:                             # noqa: BLE001 -- plain launches instead
            graphs = []
            torch.cuda.synchronize()
        if int(err.item()) != 0:
            raise RuntimeError(f"device error flag {int(err.item())} in the captured steps")

    def timed_step(i):
        if graphs:
            graphs[i % period].replay()
        else:
            step()

    K = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(K):
        timed_step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    # The decode call alone, for the roofline: the same K steps again with events
    # around each decode (events between the launches stop the append -> decode
    # overlap, so the step time above is taken without them).
    d0 = [[torch.cuda.Event(enable_timing=True) for _ in range(rot)] for _ in range(K)]
    d1 = [[torch.cuda.Event(enable_timing=True) for _ in range(rot)] for _ in range(K)]
    for i in range(K):
        step(d0[i], d1[i])
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms_total = t0.elapsed_time(t1)
    dec_ms = sum(a.elapsed_time(b) for ea, eb in zip(d0, d1) for a, b in zip(ea, eb)) / (K * rot)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error flag {int(err.item())} during the timed steps")

    ms_total_max = all_max(ms_total, world)
    # with a shared prefix the bytes that must move count the prefix once (it exists once in
    # the pool); the logical figure (every sequence's whole context) is reported beside it
    dbytes = decode_bytes(wl, args.kv_dtype)
    # (either path: the prefix exists once in the pool, and a kernel that reads it once per
    # sequence gets the repeats from L2)
    wl_shared = SHARED_TOKENS.get(args.workload, 0)
    if wl_shared:
        dbytes += unique_kv_bytes(wl, wl_shared) - logical_kv_bytes(wl)
    step_bytes = (dbytes + append_bytes(wl, args.kv_dtype)) * rot
    total_bytes = all_sum(float(step_bytes) * K, world)
    value = total_bytes / (ms_total_max / 1e3) / 1e9
    ms_per_step = ms_total_max / K
    layers = LAYERS.get(args.workload, 32)
    # a step covers `rot` of the model's `layers` layers
    tokens_per_s = all_sum(float(S), world) / ((layers / rot) * ms_per_step / 1e3)

    # end to end through the public API, host copies in the timed region every step
    e2e = PipelinedE2E((q, k_new, v_new, start, cu, lens, tables), out, stream)

    def e2e_compute(inp, o):
        d_q, d_k, d_v, d_start, d_cu, d_lens, d_tab = inp
        base = counter[0] * rot
        counter[0] += 1
        for layer in range(rot):
            pool = (base + layer) % npools
            if fused:
                append_decode(d_q, d_k, d_v, d_tab, d_lens, pool, o)
            else:
                append(*pools[pool], d_k, d_v, d_tab, d_start, d_cu, err_flag=err, stream=stream)
                decode(d_q, d_tab, d_lens, pool, o)
    e2e_step_ms, host_ms, h_last = e2e.run(e2e_compute, max(3, args.warmup), K, world)
    e2e_ms = e2e_step_ms * K
    e2e_value = total_bytes / (e2e_ms / 1e3) / 1e9
    h2d, d2h = e2e.h2d, e2e.d2h
    assert torch.equal(h_last, out.cpu())       # the copied-back result is the device result

    peaks = load_peaks()
    if peaks and peaks.get("hbm_gbs"):
        peak, peak_src = float(peaks["hbm_gbs"]), "measured"
    else:
        peak, peak_src = 6800.0, "fallback"
    # the timed call's algorithmic bytes: the decode's, and the append's when the decode
    # kernel writes the new token itself
    kbytes = dbytes + (append_bytes(wl, args.kv_dtype) if fused else 0)
    achieved = kbytes / (dec_ms / 1e3) / 1e9
    pt = {"fp8": 1024, "fp4": 2048}.get(args.kv_dtype, 1024 if D == 64 and not shared else 512)
    launches_per_step = ((0 if fused else 1) + 1 +
                         (1 if int(math.ceil(hint / pt)) > 1 or shared >= 512 else 0) +
                         (1 if shared >= 512 else 0)) * rot

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"fp8": "fp8_e4m3 K/V, bf16 q/out, fp32 softmax",
                  "fp4": "mxfp4 (e2m1, e8m0 per 32) K/V, bf16 q/out, fp32 softmax"}.get(quant, wl.dtype),
        "data": "synthetic",
        "config": {"workload": args.workload, "num_seqs_per_gpu": S, "num_q_heads": Hq,
                   "kv_cache": {"fp8": "fp8_e4m3 (per-slot fp32 scales)",
                                "fp4": "mxfp4 (e2m1 codes, one e8m0 scale per 32 values)"}.get(quant, wl.dtype),
                   "num_kv_heads": Hkv, "head_dim": D, "block_size": 16,
                   "context_tokens_after_append": int((wl.context_lens + 1).sum()),
                   "max_context": int(hint),
                   "step": ("%d layers x (" % rot if rot > 1 else "") +
                           (("pa_append_decode_attention_fp8" if quant == "fp8" else
                             "pa_append_decode_attention_shared_prefix" if shared else
                             "pa_append_decode_attention") +
                            " (1 token/seq appended by the decode kernel)"
                            if fused else "pa_append_kv (1 token/seq) + " +
                            {"fp8": "pa_decode_attention_fp8",
                             "fp4": "pa_decode_attention_fp4"}.get(quant, "pa_decode_attention")) +
                           (")" if rot > 1 else ""),
                   "shared_prefix_tokens": shared,
                   "layers_for_tokens_per_s": layers,
                   "layer_pools": rot,
                   "pool_sets": npools,
                   "cuda_graphs": bool(graphs),
                   "l2": ("inputs larger than L2 (K/V pools %.2f GB per GPU vs 129 MB L2%s), no flush"
                          if pool_bytes > L2_BYTES else
                          "K/V pools %.2f GB fit in the 129 MB L2%s")
                         % (pool_bytes / 1e9,
                            ", a distinct pool per layer of the step" if rot > 1 else
                            (", %d pool copies cycled over consecutive steps" % npools
                             if npools > 1 else "")),
                   "parallelism": f"replicas x{world} (sequences sharded by rank, no collective)"},
        "pct_of_peak_hbm": round(100.0 * value / peak, 2),
        "pct_of_nominal_hbm": round(100.0 * value / NOMINAL_HBM_GBS, 2),
        **({"unique_kv_bytes_per_step": unique_kv_bytes(wl, wl_shared),
            "logical_kv_bytes_per_step": logical_kv_bytes(wl),
            "logical_gbs": round(value * (step_bytes - unique_kv_bytes(wl, wl_shared) +
                                          logical_kv_bytes(wl)) / step_bytes, 1)} if wl_shared else {}),
        "tokens_per_s": round(tokens_per_s, 1),
        "roofline": {"kernel": ("pa_append_decode_attention_fp8 (main kernel with the quantising append "
                                "+ partition merge)" if fused and quant == "fp8" else
                                "pa_append_decode_attention_shared_prefix (prefix kernel, suffix kernel "
                                "with the append, partition merge)" if fused and shared else
                                "pa_append_decode_attention (main kernel with the append + partition merge)"
                                if fused else
                                {"fp8": "pa_decode_attention_fp8", "fp4": "pa_decode_attention_fp4"}.get(
                                    quant, "pa_decode_attention") + " (main kernel + partition merge)"),
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_source": f"{peak_src} hbm_gbs", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None if wl_shared else profiled_traffic(args.workload, args.kv_dtype),
                     "algorithmic_bytes_per_launch": kbytes, "avg_launch_ms": round(dec_ms, 5)},
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "ms_per_step": round(e2e_ms / K, 5),
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "host_enqueue_ms_per_step": round(host_ms, 5)},
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
    }
    return result, wl


# ---------------------------------------------------------------------------
# the CPU oracle (baseline, and the `--impl reference` arm)
# ---------------------------------------------------------------------------
class OracleSample:
    """The oracle's own pools holding the context of the first n sequences."""

    def __init__(self, wl, n):
        from oracle import oracle as orc
        self.orc = orc
        self.wl = wl
        self.n = n
        od = orc.BF16 if wl.dtype == "bf16" else orc.F32
        self.od = od
        et = np.uint16 if od == orc.BF16 else np.float32
        shape = orc.pool_shape(wl.num_blocks, wl.num_kv_heads, wl.head_dim, od)
        self.kp = np.zeros(shape, et)
        self.vp = np.zeros(shape, et)
        kr, vr = wl.k_rows_cpu, wl.v_rows_cpu
        for (s, start, first, cnt) in wl.fill:
            if s < n:
                orc.append_kv(self.kp, self.vp, kr[first:first + cnt], vr[first:first + cnt],
                              wl.block_tables[s:s + 1], np.array([start], np.int32),
                              np.array([0, cnt], np.int32), num_kv_heads=wl.num_kv_heads,
                              head_dim=wl.head_dim, num_blocks=wl.num_blocks, dtype=od)
        rows = torch.from_numpy(wl.new_rows[:n])
        self.k_new, self.v_new = kr[rows], vr[rows]
        self.q = wl.q_cpu[:n]
        self.pairs = [(s, h) for s in range(n) for h in range(wl.num_q_heads)]
        L = wl.context_lens[:n].astype(np.int64) + 1
        e = 2 if wl.dtype == "bf16" else 4
        self.bytes = int((L * 2 * wl.num_kv_heads * wl.head_dim * e).sum()) + \
            2 * n * wl.num_q_heads * wl.head_dim * e + int((4 * ((L + 15) // 16)).sum()) + \
            n * wl.num_kv_heads * wl.head_dim * e * 4

    def step(self, pool=None, threads=1):
        """One append + decode; with a thread pool the decode's (sequence, head) pairs are
        split over `threads` threads (the oracle's C calls run without the GIL)."""
        wl, orc, n = self.wl, self.orc, self.n
        if pool is not None and threads > 1:
            orc.append_kv(self.kp, self.vp, self.k_new, self.v_new, wl.block_tables[:n],
                          wl.context_lens[:n].astype(np.int32), np.arange(n + 1, dtype=np.int32),
                          num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
                          num_blocks=wl.num_blocks, dtype=self.od)
            lens = (wl.context_lens + 1).astype(np.int32)
            futs = [pool.submit(orc.decode_pairs, self.pairs[i::threads], self.q, self.kp, self.vp,
                                wl.block_tables, lens, num_q_heads=wl.num_q_heads,
                                num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
                                num_blocks=wl.num_blocks, scale=wl.scale, dtype=self.od)
                    for i in range(threads) if self.pairs[i::threads]]
            return [f.result() for f in futs]
        orc.append_kv(self.kp, self.vp, self.k_new, self.v_new, wl.block_tables[:n],
                      wl.context_lens[:n].astype(np.int32), np.arange(n + 1, dtype=np.int32),
                      num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim, num_blocks=wl.num_blocks,
                      dtype=self.od)
        return orc.decode_pairs(self.pairs, self.q, self.kp, self.vp, wl.block_tables,
                                (wl.context_lens + 1).astype(np.int32), num_q_heads=wl.num_q_heads,
                                num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
                                num_blocks=wl.num_blocks, scale=wl.scale, dtype=self.od)


def cpu_workload(name):
    """The same workload drawn on the CPU generator only for its shape; the oracle's
    numbers come from the same generator call on the GPU when one exists."""
    from paged_kv_cache_207_gb300 import workloads as W
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    wl = W.WORKLOADS[name](device=dev)
    wl.k_rows_cpu = wl.k_rows.cpu()
    wl.v_rows_cpu = wl.v_rows.cpu()
    wl.q_cpu = wl.q.cpu()
    return wl


def pick_sample(wl, target_s: float):
    """Grow the number of sequences until one oracle step takes about target_s seconds."""
    n = 1
    while True:
        smp = OracleSample(wl, n)
        t = time.perf_counter()
        smp.step()
        dt = time.perf_counter() - t
        if dt >= target_s or n >= wl.num_seqs:
            return smp, dt
        n = min(wl.num_seqs, max(n + 1, int(n * min(8.0, target_s / max(dt, 1e-3)))))


def cpu_baseline(wl, target_s=12.0):
    smp, _ = pick_sample(wl, target_s / 3)
    t = time.perf_counter()
    reps = 0
    while time.perf_counter() - t < target_s or reps == 0:
        smp.step()
        reps += 1
    dt = (time.perf_counter() - t) / reps
    res = {"value": round(smp.bytes / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": f"append + decode of the first {smp.n} of {wl.num_seqs} sequences "
                     f"(all {wl.num_q_heads} query heads), {reps} repetitions, plain C oracle, "
                     f"one thread, {dt:.2f} s per repetition"}
    cores = host_cores()
    if cores > 1:
        # the same oracle calls over all host cores, one thread per share of the pairs
        with cf.ThreadPoolExecutor(max_workers=cores) as ex:
            smp.step(ex, cores)
            t = time.perf_counter()
            reps = 0
            while time.perf_counter() - t < target_s / 2 or reps == 0:
                smp.step(ex, cores)
                reps += 1
            dt = (time.perf_counter() - t) / reps
        res["all_cores"] = {"value": round(smp.bytes / dt / 1e9, 4), "unit": "GB/s", "cores": cores,
                            "sample": f"the same sample, {reps} repetitions, decode pairs split "
                                      f"over {cores} threads"}
    return res


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, rank, world):
    if rank != 0:
        return None
    wl = cpu_workload(args.workload)
    cores = host_cores()
    # size one step so that warm-up plus timed steps take about two minutes on all host cores
    smp, dt = pick_sample(wl, max(0.005, min(1.0, 120.0 / (args.steps + args.warmup))) * cores)
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        for _ in range(args.warmup):
            smp.step(ex, cores)
        t = time.perf_counter()
        for _ in range(args.steps):
            smp.step(ex, cores)
        el = time.perf_counter() - t
    value = smp.bytes * args.steps / el / 1e9
    S = smp.n
    layers = LAYERS.get(args.workload, 32)
    ms = el * 1e3 / args.steps
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic",
        "config": {"workload": args.workload, "num_seqs_per_step": S,
                   "num_q_heads": wl.num_q_heads, "num_kv_heads": wl.num_kv_heads,
                   "head_dim": wl.head_dim, "block_size": 16,
                   "step": "oracle append + decode of a bounded sample of the workload"},
        "tokens_per_s": round(S / (layers * ms / 1e3), 3),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {S} of {wl.num_seqs} sequences per step, decode pairs "
                                   f"split over {cores} threads"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_replay(args, rank, world, local):
    """The spindle-shaped replay: every iteration of continuous batching, 12 layers of
    append + decode, timed as a whole (wall clock) and on the GPU (events)."""
    import paged_kv_cache_207_gb300 as pk
    from paged_kv_cache_207_gb300 import build, workloads as W
    from paged_kv_cache_207_gb300.replay import Replay
    torch.cuda.set_device(local)
    build.build()
    pk.lib()
    rw = W.spindle_replay(device="cuda", seed=208 + 1000 * rank)
    barrier(world)
    graphs = not args.no_graphs
    # warm-up runs on the instance that is timed, so that its graphs (one per running-batch
    # size) are captured before the timed run, as an engine captures them once
    rp = Replay(rw, device="cuda", use_graphs=graphs)
    for i in range(max(1, min(args.warmup, 3))):
        if i:
            rp.reset()
        rp.run()
    torch.cuda.synchronize()
    rp.reset(time_gpu=True)
    st = rp.run()
    barrier(world)
    wall = all_max(st.wall_s, world)
    gpu_s = all_max(st.gpu_ms / 1e3, world)
    tokens = all_sum(float(st.generated_tokens), world)
    dbytes = all_sum(float(st.decode_bytes), world)
    peaks = load_peaks() or {}
    from paged_kv_cache_207_gb300.replay import contiguous_account, paged_account
    ca, pa_ = contiguous_account(rw, max_new_tokens=192), paged_account(rw)
    return {
        "metric": METRIC, "value": round(dbytes / gpu_s / 1e9, 1), "unit": "GB/s",
        "n_gpus": world, "steps": st.iterations, "warmup": args.warmup,
        "ms_per_step": round(gpu_s * 1e3 / st.iterations, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "spindle_replay", "requests": rw.num_seqs,
                   "cow_children": rw.num_children, "layers": rw.num_layers,
                   "heads": rw.num_heads, "head_dim": rw.head_dim, "pool_slots": rw.num_blocks * 16,
                   "step": "one continuous-batching iteration: 12 x (append + decode)",
                   "cuda_graphs": graphs},
        "pct_of_peak_hbm": round(100 * dbytes / gpu_s / 1e9 / peaks.get("hbm_gbs", 6800.0), 2),
        "pct_of_nominal_hbm": round(100 * dbytes / gpu_s / 1e9 / NOMINAL_HBM_GBS, 2),
        "tokens_per_s": round(tokens / wall, 1),
        # the whole replay on the wall clock: host scheduling, block manager, the per-iteration
        # copies of tables and positions, and every launch through the public API
        "e2e": {"value": round(dbytes / wall / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(wall * 1e3 / st.iterations, 4),
                "h2d_bytes_per_step": int(st.h2d_bytes // max(1, st.iterations)),
                "d2h_bytes_per_step": 0},
        "tokens_per_s_gpu_time": round(tokens / gpu_s, 1),
        "replay": {"iterations": st.iterations, "generated_tokens": st.generated_tokens,
                   "preemptions": st.preemptions, "cow_copies": st.cow_copies,
                   "prefill_tokens": st.prefill_tokens,
                   "peak_physical_slots": st.peak_physical_slots,
                   "mean_slot_utilisation": round(st.mean_slot_utilisation, 4),
                   "wall_s": round(wall, 3), "gpu_s": round(gpu_s, 4)},
        "allocators": {
            "contiguous": {"peak_slots_held": ca.peak_slots_held,
                           "mean_slot_utilisation": round(ca.mean_slot_utilisation, 4),
                           "steps_to_drain": ca.steps_to_drain},
            "paged": {"peak_slots_held": pa_.peak_slots_held,
                      "mean_slot_utilisation": round(pa_.mean_slot_utilisation, 4),
                      "steps_to_drain": pa_.steps_to_drain}},
        "gpu_launches": st.launches,
    }


def run_prefill(args, rank, world, local):
    """Chunked prefill attention, Llama-3-8B heads: 16 sequences each append a 512-token
    chunk at a start drawn U[0, 3584] and attend causally over their whole prefix."""
    import paged_kv_cache_207_gb300 as pk
    from paged_kv_cache_207_gb300 import build, workloads as W
    torch.cuda.set_device(local)
    build.build()
    pk.lib()
    rng = np.random.default_rng(213 + 1000 * rank)
    S, n = 16, 512
    starts = rng.integers(0, 3585, size=S)
    wl = W.make_decode_workload("llama3-8b_prefill", context_lens=starts + n - 1, num_q_heads=32,
                                num_kv_heads=8, head_dim=128, dtype="bf16", seed=213 + rank,
                                device="cuda")
    shape = pk.pool_shape(wl.num_blocks, 8, 128, torch.bfloat16)
    kp = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    tables = torch.from_numpy(wl.block_tables).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # context before the chunk: positions 0 .. start-1 (set-up, untimed)
    all_rows = [torch.from_numpy(wl.logical_rows(s_)) for s_ in range(S)]
    ctx = torch.cat([r[:int(st)] for r, st in zip(all_rows, starts)]).cuda()
    chunk = torch.cat([r[int(st):int(st) + n] for r, st in zip(all_rows, starts)]).cuda()
    cu_ctx = torch.tensor(np.concatenate([[0], np.cumsum(starts)]), dtype=torch.int32, device="cuda")
    pk.append_kv(kp, vp, wl.k_rows[ctx].contiguous(), wl.v_rows[ctx].contiguous(), tables,
                 torch.zeros(S, dtype=torch.int32, device="cuda"), cu_ctx, err_flag=err)
    k_chunk, v_chunk = wl.k_rows[chunk].contiguous(), wl.v_rows[chunk].contiguous()
    del wl.k_rows, wl.v_rows
    # consecutive steps alternate between two copies of the pools (as consecutive layers
    # would), so no step finds the previous step's K/V in L2
    pools = [(kp, vp), (kp.clone(), vp.clone())]
    pool_bytes = 2 * len(pools) * kp.numel() * kp.element_size()
    counter = [0]
    g = torch.Generator(device="cuda").manual_seed(7)
    q = torch.randn(S * n, 32, 128, generator=g, device="cuda").to(torch.bfloat16)
    out = torch.empty_like(q)
    start_t = torch.from_numpy(starts.astype(np.int32)).cuda()
    cu_q = torch.arange(0, S * n + 1, n, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def next_pools():
        counter[0] += 1
        return pools[counter[0] % len(pools)]

    def step():
        kp, vp = next_pools()
        pk.append_kv(kp, vp, k_chunk, v_chunk, tables, start_t, cu_q, err_flag=err, stream=stream)
        pk.prefill_attention(out, q, kp, vp, tables, start_t, cu_q, wl.scale, max_chunk=n,
                             err_flag=err, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    K = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    t0.record(stream)
    for _ in range(K):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error flag {int(err.item())}")
    ms = t0.elapsed_time(t1) / K
    # the attention kernel alone, for the roofline (same inputs; the appends above left the
    # cache as a step leaves it)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        kp, vp = next_pools()
        pk.prefill_attention(out, q, kp, vp, tables, start_t, cu_q, wl.scale, max_chunk=n,
                             err_flag=err, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    kernel_ms = e0.elapsed_time(e1) / K

    # end to end through the public API, host copies in the timed region every step
    e2e = PipelinedE2E((q, k_chunk, v_chunk, start_t, cu_q, tables), out, stream)

    def e2e_compute(inp, o):
        d_q, d_k, d_v, d_st, d_cu, d_tab = inp
        kp, vp = next_pools()
        pk.append_kv(kp, vp, d_k, d_v, d_tab, d_st, d_cu, err_flag=err, stream=stream)
        pk.prefill_attention(o, d_q, kp, vp, d_tab, d_st, d_cu, wl.scale, max_chunk=n,
                             err_flag=err, stream=stream)
    e2e_ms, _, h_last = e2e.run(e2e_compute, args.warmup, K)
    assert torch.equal(h_last, out.cpu())
    h2d, d2h = e2e.h2d, e2e.d2h
    pos = (starts[:, None] + np.arange(n)[None, :]).astype(np.int64)   # positions of chunk rows
    flops = float(4 * 128 * 32 * (pos + 1).sum())                       # QK and PV, all heads
    peaks = load_peaks() or {}
    peak = float(peaks.get("bf16_tflops", 1900.0))
    tflops = flops / (ms / 1e3) / 1e12
    return {"metric": "chunked prefill attention TFLOP/s (bf16 tensor cores)", "value": round(tflops, 2),
            "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "llama3-8b_prefill", "num_seqs": S, "chunk_tokens": n,
                       "start_positions": "U[0, 3584]", "num_q_heads": 32, "num_kv_heads": 8,
                       "head_dim": 128, "step": "pa_append_kv (512 rows/seq) + pa_prefill_attention",
                       "l2": "two copies of the K/V pools (%.2f GB in all) alternate over consecutive "
                             "steps; the chunk's K/V tiles are re-read from L2 within a step by design"
                             % (pool_bytes / 1e9)},
            "roofline": {"kernel": "prefill_tc_kernel (tcgen05, TMEM accumulators)", "bound": "tensor",
                         "achieved": round(flops / (kernel_ms / 1e3) / 1e12, 2), "peak": peak,
                         "peak_source": "measured bf16_tflops", "unit": "TFLOP/s",
                         "frac": round(flops / (kernel_ms / 1e3) / 1e12 / peak, 4),
                         "avg_launch_ms": round(kernel_ms, 4), "flops_per_launch": flops, "traffic": None},
            "tokens_per_s": round(S * n / (ms / 1e3), 1),
            "e2e": {"value": round(flops / (e2e_ms / 1e3) / 1e12, 2), "unit": "TFLOP/s",
                    "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h)},
            "gpu_launches": 2 * K, "clocks": clk}


# Workloads measured after the headline in the same process (one GPU; each with its own timed
# region, CUDA-event roofline and clock record).  The first is the long-context split-KV case,
# the second workload the 70 %-of-HBM target names.
EXTRA_CONFIGS = [
    ("llama3-8b_long_context", {"workload": "llama3-8b_long_context"}),
    ("qwen2.5-0.5b_gqa", {"workload": "qwen2.5-0.5b_gqa"}),
    ("llama3-8b_shared_prefix", {"workload": "llama3-8b_shared_prefix"}),
    ("llama3-8b_shared_prefix+sharing", {"workload": "llama3-8b_shared_prefix",
                                          "shared_prefix": 4096}),
    ("llama3-8b_batch256+fp8", {"workload": "llama3-8b_batch256", "kv_dtype": "fp8"}),
    ("llama3-8b_long_context+fp8", {"workload": "llama3-8b_long_context", "kv_dtype": "fp8"}),
    ("llama3-8b_batch256+fp4", {"workload": "llama3-8b_batch256", "kv_dtype": "fp4"}),
    ("llama3-8b_long_context+fp4", {"workload": "llama3-8b_long_context", "kv_dtype": "fp4"}),
    ("spindle_replay", {"workload": "spindle_replay"}),
    ("llama3-8b_prefill", {"workload": "llama3-8b_prefill"}),
]
DROP_KEYS = ("metric", "n_gpus", "higher_is_better", "scaling", "vs_baseline", "data")
# Workloads whose step is short (tens of microseconds; 0.1-0.2 ms) run at least this many
# timed steps (and warm-up steps) in the default run: about 10 ms of timed work each.
MIN_CONFIG_STEPS = {"llama3-8b_shared_prefix": 100, "llama3-8b_shared_prefix+sharing": 400,
                    "llama3-8b_batch256+fp8": 60, "llama3-8b_batch256+fp4": 60,
                    "llama3-8b_long_context+fp8": 50, "llama3-8b_long_context+fp4": 50}
MIN_CONFIG_WARMUP = {"llama3-8b_shared_prefix+sharing": 20}


def run_one(args, rank, world, local):
    if args.workload == "llama3-8b_prefill":
        return run_prefill(args, rank, world, local)
    if args.workload == "spindle_replay":
        return run_replay(args, rank, world, local)
    return run_ours(args, rank, world, local)[0]


def run_extra_configs(args, rank, world, local) -> dict:
    """Every other workload, one after the other, each freed before the next.  Steps are
    capped so that the extra configs add a minute or two to the run."""
    out = {}
    for name, over in EXTRA_CONFIGS:
        sub = argparse.Namespace(**vars(args))
        sub.kv_dtype, sub.shared_prefix, sub.num_seqs = "bf16", 0, 0
        for k, v in over.items():
            setattr(sub, k, v)
        sub.steps = max(1, min(args.steps, 50))
        sub.warmup = max(3, min(args.warmup, 5))
        # short steps get enough of them for a timed region of several milliseconds
        sub.steps = max(sub.steps, MIN_CONFIG_STEPS.get(name, 0))
        sub.warmup = max(sub.warmup, MIN_CONFIG_WARMUP.get(name, 0))
        try:
            res = run_one(sub, rank, world, local)
            out[name] = {k: v for k, v in res.items() if k not in DROP_KEYS}
            out[name]["metric"] = res.get("metric")
        except Exception as e:       # one workload failing must not hide the others
            out[name] = {"error": f"{type(e).__name__}: {e}"}
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama3-8b_batch256")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graphs", action="store_true",
                    help="launch every kernel of the timed steps directly instead of replaying "
                         "CUDA graphs of them (decode workloads: one per pool-rotation phase; "
                         "replay: one per batch size)")
    ap.add_argument("--kv-dtype", choices=["bf16", "fp8", "fp4"], default="bf16",
                    help="K/V cache element type; fp8 = E4M3 codes with per-slot scales, "
                         "fp4 = MXFP4 (E2M1 codes, one E8M0 scale per 32 values)")
    ap.add_argument("--shared-prefix", type=int, default=0,
                    help="decode through pa_decode_attention_shared_prefix with this many shared "
                         "tokens (the llama3-8b_shared_prefix workload shares 4096)")
    ap.add_argument("--num-seqs", type=int, default=0,
                    help="override the workload's sequence count (smaller cases for profiling)")
    ap.add_argument("--no-configs", action="store_true",
                    help="measure the headline workload only (no `configs` entries)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local = dist_init(args.gpus)
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    if args.workload in ("llama3-8b_prefill", "spindle_replay"):
        res = run_one(args, rank, world, local)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    res, wl = run_ours(args, rank, world, local)
    del wl
    torch.cuda.empty_cache()
    # the default run (one GPU, the headline workload) also measures every other workload
    default_run = (args.workload == "llama3-8b_batch256" and args.kv_dtype == "bf16" and
                   not args.shared_prefix and not args.num_seqs)
    if world == 1 and default_run and not args.no_configs:
        res["configs"] = run_extra_configs(args, rank, world, local)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            wl_cpu = cpu_workload(args.workload)
            res["cpu_baseline"] = cpu_baseline(wl_cpu)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

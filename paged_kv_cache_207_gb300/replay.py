"""Continuous-batching replay over the paged cache (a minimal engine loop).

Drives the library the way an engine does, one iteration at a time (spindle,
"Continuous batching, and the control" and "Paging"):

1. admit waiting requests first-come-first-served while the pool has blocks for
   their context plus one token; a preempted request is recomputed (its whole
   context is appended again);
2. reserve the next slot of every running sequence through the host block
   manager; a write into a shared block yields a copy-on-write pair; when the
   pool runs dry the most recently admitted sequence is preempted;
3. per layer: append the admitted contexts, copy the copy-on-write blocks, append
   one new token per running sequence at its explicit position, and decode over
   context + 1 (spindle, "Two bugs worth recording": explicit positions and
   lengths, advanced once per iteration by this loop, never by the cache).

The synthetic "model" supplies q / k / v rows for every (sequence, layer,
position) from the workload tensors.
"""
from __future__ import annotations

import collections
import time
from dataclasses import dataclass, field

import numpy as np
import torch

from . import _native as pk

BLOCK = pk.BLOCK_SIZE


@dataclass
class ReplayStats:
    iterations: int = 0
    generated_tokens: int = 0
    preemptions: int = 0
    cow_copies: int = 0
    prefill_tokens: int = 0
    peak_physical_slots: int = 0
    slot_util_sum: float = 0.0
    decode_bytes: int = 0
    gpu_ms: float = 0.0
    wall_s: float = 0.0
    launches: int = 0
    h2d_bytes: int = 0            # host -> device copies of schedule data (tables, positions)
    per_iteration_running: list = field(default_factory=list)

    @property
    def mean_slot_utilisation(self) -> float:
        return self.slot_util_sum / max(1, self.iterations)


class Replay:
    """``device=None`` runs the host schedule alone (block manager and accounting, no
    kernels): the same admissions, preemptions and copy pairs as a device run."""

    def __init__(self, rw, device="cuda", time_gpu: bool = False, block_manager=None,
                 on_schedule=None, use_graphs: bool = False):
        self.rw = rw
        self.dev = device
        self.time_gpu = time_gpu and device is not None
        self.use_graphs = use_graphs and device is not None
        self.bm = block_manager if block_manager is not None else pk.BlockManager(rw.num_blocks)
        self.on_schedule = on_schedule
        self.max_blocks = (rw.max_len + BLOCK - 1) // BLOCK
        if device is not None:
            shape = pk.pool_shape(rw.num_blocks, rw.num_heads, rw.head_dim, torch.bfloat16)
            # fresh pools hold NaN bits: every value a decode reads must have been appended
            self.k = [torch.full(shape, float("nan"), dtype=torch.bfloat16, device=device)
                      for _ in range(rw.num_layers)]
            self.v = [torch.full(shape, float("nan"), dtype=torch.bfloat16, device=device)
                      for _ in range(rw.num_layers)]
            self.err = torch.zeros(1, dtype=torch.int32, device=device)
        if self.use_graphs:
            n = rw.num_seqs
            # fixed device buffers the captured steps read; host staging in pinned memory
            self.g_tables = torch.full((n, self.max_blocks), -1, dtype=torch.int32, device=device)
            self.g_lens = torch.zeros(n, dtype=torch.int32, device=device)
            self.g_seq = torch.zeros(n, dtype=torch.long, device=device)
            self.g_pos = torch.zeros(n, dtype=torch.long, device=device)
            self.h_tables = torch.empty_like(self.g_tables, device="cpu").pin_memory()
            self.h_lens = torch.empty_like(self.g_lens, device="cpu").pin_memory()
            self.h_seq = torch.empty_like(self.g_seq, device="cpu").pin_memory()
            self.h_pos = torch.empty_like(self.g_pos, device="cpu").pin_memory()
            self.graphs = {}          # running-batch size -> (graph, per-layer outputs)
            self.h_free = None        # event: the last staging copy has been read
        self._owns_bm = block_manager is None
        self._reset_host()

    def reset(self, time_gpu: bool | None = None) -> None:
        """Start the workload over on the same pools, buffers and captured graphs (as an
        engine keeps its graphs across batches): the schedule, the block manager and the
        statistics begin afresh.  Every value a decode reads is appended again first."""
        if not self._owns_bm:
            raise RuntimeError("reset() needs the replay's own block manager")
        if time_gpu is not None:
            self.time_gpu = time_gpu and self.dev is not None
        self.bm = pk.BlockManager(self.rw.num_blocks)
        self._reset_host()

    def _reset_host(self) -> None:
        rw = self.rw
        n = rw.num_seqs
        self.gen_done = [0] * n
        self.bm_id = [-1] * n
        self.state = ["waiting"] * n
        first_child = n - rw.num_children
        self.waiting = collections.deque([("one", i) for i in range(first_child)])
        if rw.num_children:
            self.waiting.append(("group", list(range(first_child, n))))
        self.running: list[int] = []          # admission order
        self._timed: list = []                 # (start, end) events of the timed iterations
        self.stats = ReplayStats()

    # -- host scheduling ------------------------------------------------------
    def ctx(self, i: int) -> int:
        return int(self.rw.prompt_lens[i]) + self.gen_done[i]

    def _free_blocks(self) -> int:
        return int(self.bm.stats()["free_blocks"])

    def _admit(self, prefill: list) -> None:
        while self.waiting:
            kind, who = self.waiting[0]
            if kind == "one":
                need = (self.ctx(who) + 1 + BLOCK - 1) // BLOCK
                if need > self._free_blocks():
                    return
                self.waiting.popleft()
                sid = self.bm.add_seq()
                self.bm.prepare_append(sid, 0, self.ctx(who))
                self.bm_id[who] = sid
                self.state[who] = "running"
                self.running.append(who)
                prefill.append((who, self.bm.block_table(sid, self.max_blocks), self.ctx(who), [who]))
            else:
                p = self.rw.parent_prompt
                need = (p + BLOCK - 1) // BLOCK + len(who)
                if need > self._free_blocks():
                    return
                self.waiting.popleft()
                parent = self.bm.add_seq()
                self.bm.prepare_append(parent, 0, p)
                # the parent prompt's rows are the first child's first p rows
                prefill.append((who[0], self.bm.block_table(parent, self.max_blocks), p, list(who)))
                for c in who:
                    self.bm_id[c] = self.bm.fork(parent)
                    self.state[c] = "running"
                    self.running.append(c)
                self.bm.free(parent)

    def _preempt_latest(self) -> int:
        victim = self.running.pop()
        self.bm.free(self.bm_id[victim])
        self.bm_id[victim] = -1
        self.state[victim] = "waiting"
        self.waiting.appendleft(("one", victim))
        self.stats.preemptions += 1
        return victim

    def _reserve(self) -> list:
        pairs = []
        i = 0
        while i < len(self.running):
            s = self.running[i]
            try:
                pairs += self.bm.prepare_append(self.bm_id[s], self.ctx(s), 1)
                i += 1
            except pk.PagedKVError as e:
                if e.status != 4:
                    raise
                if self._preempt_latest() == s:
                    continue        # s itself was the latest; the loop ends or moves on
        return pairs

    # -- device work ------------------------------------------------------------
    def _tables_into(self, ids: list, out: np.ndarray) -> np.ndarray:
        """The block tables of sequences `ids` into the int32 rows of `out`: one call into
        the native block manager where it offers the batch, else one per sequence."""
        if hasattr(self.bm, "block_tables"):
            return self.bm.block_tables(ids, self.max_blocks, out=out)
        out[:] = np.asarray([self.bm.block_table(i, self.max_blocks) for i in ids], np.int32)
        return out

    def _decode_kernels(self, hint: int) -> int:
        """Kernels of one pa_append_decode_attention call: the main kernel, and the
        partition merge when a context can span two partitions."""
        return 1 + (1 if hint > pk.partition_tokens(self.rw.head_dim) else 0)

    def _i32(self, a) -> torch.Tensor:
        return torch.tensor(np.asarray(a, np.int32), dtype=torch.int32, device=self.dev)

    def step(self, observer=None) -> bool:
        """One iteration.  Returns False when every request has finished."""
        if not self.running and not self.waiting:
            return False
        prefill: list = []
        self._admit(prefill)
        pairs = self._reserve()
        # a context whose every holder was preempted again in this same iteration is not
        # written: its blocks went back to the pool and may already belong to someone else
        # (a preempted sequence never emitted copy pairs here: it is always the latest
        # admitted, so it had not reserved its slot yet)
        prefill = [p for p in prefill if any(self.state[h] == "running" for h in p[3])]
        run = list(self.running)
        if not run:
            if not self.waiting:
                return False
            raise RuntimeError("a single request needs more blocks than the pool holds")
        rw = self.rw
        S = len(run)
        ctx = np.array([self.ctx(s) for s in run], np.int32)
        self.stats.cow_copies += len(pairs)
        self.stats.prefill_tokens += int(sum(p[2] for p in prefill))
        if self.on_schedule is not None:
            self.on_schedule(self, run, ctx, prefill, pairs)
        if self.dev is not None:
            self._device_work(run, ctx, prefill, pairs, observer)
        self._finish_iteration(run, ctx)
        return True

    def _capture(self, S: int):
        """One CUDA graph for an iteration with S running sequences: per layer the
        gather of the new rows and one pa_append_decode_attention (the decode kernel
        writes the new rows itself), all reading the fixed buffers above."""
        rw = self.rw
        g = torch.cuda.CUDAGraph()
        tables, lens = self.g_tables[:S], self.g_lens[:S]
        seq, pos = self.g_seq[:S], self.g_pos[:S]
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            outs = []
            for l in range(rw.num_layers):
                k_new = rw.k[seq, l, pos]
                v_new = rw.v[seq, l, pos]
                q = rw.q[seq, l, pos]
                out = torch.empty_like(q)
                pk.append_decode_attention(out, q, self.k[l], self.v[l], k_new, v_new, tables,
                                           lens, rw.scale, max_context_len_hint=rw.max_len,
                                           err_flag=self.err)
                outs.append(out)
        return g, outs

    def _device_work(self, run, ctx, prefill, pairs, observer) -> None:
        if self.use_graphs:
            return self._device_work_graph(run, ctx, prefill, pairs, observer)
        rw = self.rw
        S = len(run)
        tables = self._i32(self._tables_into([self.bm_id[s] for s in run],
                                             np.empty((S, self.max_blocks), np.int32)))
        lens = self._i32(ctx + 1)
        seq_idx = torch.tensor(run, dtype=torch.long, device=self.dev)
        pos_idx = torch.from_numpy(ctx.astype(np.int64)).to(self.dev)
        if prefill:
            pf_tables = self._i32([p[1] for p in prefill])
            pf_start = self._i32([0] * len(prefill))
            pf_cu = self._i32(np.concatenate([[0], np.cumsum([p[2] for p in prefill])]))
            pf_seq = torch.cat([torch.full((p[2],), p[0], dtype=torch.long) for p in prefill]).to(self.dev)
            pf_pos = torch.cat([torch.arange(p[2]) for p in prefill]).to(self.dev)
        pairs_t = self._i32(pairs).reshape(-1, 2) if pairs else None
        self.stats.h2d_bytes += sum(t.numel() * t.element_size()
                                    for t in (tables, lens, seq_idx, pos_idx))

        ev0 = ev1 = None
        if self.time_gpu:
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        outs = []
        for l in range(rw.num_layers):
            if prefill:
                pk.append_kv(self.k[l], self.v[l], rw.k[pf_seq, l, pf_pos].contiguous(),
                             rw.v[pf_seq, l, pf_pos].contiguous(), pf_tables, pf_start, pf_cu,
                             err_flag=self.err)
                self.stats.launches += 1
            if pairs_t is not None:
                pk.copy_block(self.k[l], self.v[l], pairs_t, err_flag=self.err)
                self.stats.launches += 1
            k_new = rw.k[seq_idx, l, pos_idx].contiguous()
            v_new = rw.v[seq_idx, l, pos_idx].contiguous()
            q = rw.q[seq_idx, l, pos_idx].contiguous()
            out = torch.empty_like(q)
            if ev0 is not None and l == 0:
                ev0.record()
            hint = int(ctx.max()) + 1
            pk.append_decode_attention(out, q, self.k[l], self.v[l], k_new, v_new, tables, lens,
                                       rw.scale, max_context_len_hint=hint, err_flag=self.err)
            self.stats.launches += self._decode_kernels(hint)
            outs.append(out)
        if ev1 is not None:
            ev1.record()
        if observer is not None:
            observer(self, run, ctx, outs)
        if ev0 is not None:
            self._timed.append((ev0, ev1))        # read after the run: no wait per iteration

    def _device_work_graph(self, run, ctx, prefill, pairs, observer) -> None:
        rw = self.rw
        S = len(run)
        # host side first: the iteration's tables and positions into the pinned staging (the
        # previous iteration's copies out of it must be done), and the admission / copy inputs
        if self.h_free is not None:
            self.h_free.synchronize()
        self._tables_into([self.bm_id[s] for s in run], self.h_tables[:S].numpy())
        self.h_lens[:S].numpy()[:] = ctx + 1
        self.h_seq[:S].numpy()[:] = np.asarray(run, np.int64)
        self.h_pos[:S].numpy()[:] = ctx.astype(np.int64)
        pf_tables = pf_start = pf_cu = pf_seq = pf_pos = None
        if prefill:
            pf_tables = self._i32([p[1] for p in prefill])
            pf_start = self._i32([0] * len(prefill))
            pf_cu = self._i32(np.concatenate([[0], np.cumsum([p[2] for p in prefill])]))
            pf_seq = torch.cat([torch.full((p[2],), p[0], dtype=torch.long) for p in prefill]).to(self.dev)
            pf_pos = torch.cat([torch.arange(p[2]) for p in prefill]).to(self.dev)
        pairs_t = self._i32(pairs).reshape(-1, 2) if pairs else None
        if S not in self.graphs:
            self.graphs[S] = self._capture(S)
        g, outs = self.graphs[S]
        # then the device work, back to back
        ev0 = ev1 = None
        if self.time_gpu:
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record()
        if prefill or pairs:       # admissions and copy-on-write copies: ordinary launches
            for l in range(rw.num_layers):
                if prefill:
                    pk.append_kv(self.k[l], self.v[l], rw.k[pf_seq, l, pf_pos].contiguous(),
                                 rw.v[pf_seq, l, pf_pos].contiguous(), pf_tables, pf_start, pf_cu,
                                 err_flag=self.err)
                    self.stats.launches += 1
                if pairs_t is not None:
                    pk.copy_block(self.k[l], self.v[l], pairs_t, err_flag=self.err)
                    self.stats.launches += 1
        for d, h in ((self.g_tables, self.h_tables), (self.g_lens, self.h_lens),
                     (self.g_seq, self.h_seq), (self.g_pos, self.h_pos)):
            d[:S].copy_(h[:S], non_blocking=True)
            self.stats.h2d_bytes += h[:S].numel() * h.element_size()
        self.h_free = torch.cuda.Event()
        self.h_free.record()
        g.replay()
        self.stats.launches += self._decode_kernels(rw.max_len) * rw.num_layers
        if ev1 is not None:
            ev1.record()
            self._timed.append((ev0, ev1))        # read after the run: no wait per iteration
        if observer is not None:
            observer(self, run, ctx, [o.clone() for o in outs])

    def _finish_iteration(self, run, ctx) -> None:
        """Accounting, then advance every running length once for the whole iteration."""
        rw = self.rw
        S = len(run)
        st = self.bm.stats()
        self.stats.peak_physical_slots = max(self.stats.peak_physical_slots, st["physical_slots"])
        held = sum(self.ctx(s) + 1 for s in run)
        if st["physical_slots"]:
            self.stats.slot_util_sum += min(1.0, held / st["physical_slots"])
        self.stats.decode_bytes += rw.num_layers * int((ctx + 1).sum()) * 2 * rw.num_heads * rw.head_dim * 2
        self.stats.iterations += 1
        self.stats.generated_tokens += S
        self.stats.per_iteration_running.append(S)
        for s in run:
            self.gen_done[s] += 1
        for s in list(self.running):
            if self.gen_done[s] >= int(rw.gen_lens[s]):
                self.bm.free(self.bm_id[s])
                self.bm_id[s] = -1
                self.state[s] = "done"
                self.running.remove(s)

    def run(self, observer=None, max_iterations: int = 100000) -> ReplayStats:
        t = time.perf_counter()
        for _ in range(max_iterations):
            if not self.step(observer):
                break
        if self.dev is None:
            self.stats.wall_s = time.perf_counter() - t
            return self.stats
        torch.cuda.synchronize()
        self.stats.wall_s = time.perf_counter() - t
        self.stats.gpu_ms += sum(a.elapsed_time(b) for a, b in self._timed)
        self._timed.clear()
        if int(self.err.item()) != 0:
            raise RuntimeError(f"device error flag {int(self.err.item())} during the replay")
        return self.stats


# ---- the control: a contiguous per-sequence allocator ------------------------------

@dataclass
class AllocatorAccount:
    peak_slots_held: int
    mean_slot_utilisation: float
    steps_to_drain: int


def contiguous_account(rw, max_new_tokens: int | None = None, slots: int | None = None) -> AllocatorAccount:
    """Replay the same requests through a contiguous allocator (spindle, "Paging": a
    contiguous buffer is sized at admission to prompt + max_new_tokens, the only bound
    known then, and held for the request's whole lifetime).  Same FCFS admission, one
    token per running request per step; a fork cannot share, so each copy-on-write
    child holds its own buffer.  Host accounting only."""
    cap = int(rw.gen_lens.max()) if max_new_tokens is None else max_new_tokens
    total = rw.num_blocks * BLOCK if slots is None else slots
    waiting = collections.deque(range(rw.num_seqs))
    running: list[int] = []
    done_gen = [0] * rw.num_seqs
    held = steps = peak = 0
    util_sum = 0.0
    while waiting or running:
        while waiting and held + int(rw.prompt_lens[waiting[0]]) + cap <= total:
            i = waiting.popleft()
            held += int(rw.prompt_lens[i]) + cap
            running.append(i)
        if not running:
            raise RuntimeError("a request does not fit the pool")
        peak = max(peak, held)
        tokens = sum(int(rw.prompt_lens[i]) + done_gen[i] + 1 for i in running)
        util_sum += tokens / held
        steps += 1
        for i in running:
            done_gen[i] += 1
        for i in list(running):
            if done_gen[i] >= int(rw.gen_lens[i]):
                running.remove(i)
                held -= int(rw.prompt_lens[i]) + cap
    return AllocatorAccount(peak, util_sum / steps, steps)


def paged_account(rw) -> AllocatorAccount:
    """The block-paged schedule of ``Replay`` run on the host alone."""
    st = Replay(rw, device=None).run()
    return AllocatorAccount(st.peak_physical_slots, st.mean_slot_utilisation, st.iterations)

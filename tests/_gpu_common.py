"""Helpers shared by the GPU parity tests: device pools filled through the library's
own append, the oracle's view of the same workload, and the tolerances.

Tolerances (written here once, used by every parity test):
  * fp32 outputs: per (sequence, query head) row, max_d |gpu - oracle| / max_d |oracle|
    <= 1e-5 (the elementwise relative error is ill-posed where the oracle is ~0);
  * bf16 outputs: max |gpu - oracle| <= 2e-2 (outputs are convex combinations of
    N(0, 1) value rows, so they are of order 1).
Append, copy and block-table indexing are compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import paged_kv_cache_207_gb300 as pk
from oracle import oracle as orc

F32_ROW_RTOL = 1e-5
BF16_ATOL = 2e-2

CANARY_BF16 = 0xFFFF          # a NaN pattern no N(0,1) draw produces
CANARY_F32 = 0x7FC00001


def odtype(wl) -> int:
    return orc.BF16 if wl.dtype == "bf16" else orc.F32


def canary_fill(t: torch.Tensor) -> torch.Tensor:
    if t.dtype == torch.bfloat16:
        t.view(torch.int16).fill_(np.int16(np.uint16(CANARY_BF16).view(np.int16)))
    else:
        t.view(torch.int32).fill_(CANARY_F32)
    return t


class DevicePools:
    """K/V pools on the GPU, filled with the workload's context through pa_append_kv."""

    def __init__(self, wl, device="cuda", canary=True):
        self.wl = wl
        shape = pk.pool_shape(wl.num_blocks, wl.num_kv_heads, wl.head_dim, wl.torch_dtype())
        alloc = torch.empty if canary else torch.zeros
        self.k = alloc(shape, dtype=wl.torch_dtype(), device=device)
        self.v = alloc(shape, dtype=wl.torch_dtype(), device=device)
        if canary:
            canary_fill(self.k)
            canary_fill(self.v)
        self.tables = torch.from_numpy(wl.block_tables).to(device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.fill_context()

    def fill_context(self):
        wl = self.wl
        if not wl.fill:
            return
        seqs = [f[0] for f in wl.fill]
        starts = [f[1] for f in wl.fill]
        first = wl.fill[0][2]
        ns = [f[3] for f in wl.fill]
        end = wl.fill[-1][2] + wl.fill[-1][3]
        assert all(wl.fill[i][2] + wl.fill[i][3] == wl.fill[i + 1][2] for i in range(len(wl.fill) - 1))
        dev = self.k.device
        tables = self.tables[torch.tensor(seqs, device=dev)].contiguous()
        cu = torch.tensor(np.concatenate([[0], np.cumsum(ns)]), dtype=torch.int32, device=dev)
        pk.append_kv(self.k, self.v, wl.k_rows[first:end].to(dev).contiguous(),
                     wl.v_rows[first:end].to(dev).contiguous(), tables,
                     torch.tensor(starts, dtype=torch.int32, device=dev), cu, err_flag=self.err)

    def step_inputs(self):
        """(k_new, v_new, start_pos, cu, context_lens after the append) for one decode step."""
        wl = self.wl
        dev = self.k.device
        rows = torch.from_numpy(wl.new_rows).to(wl.k_rows.device)
        k_new = wl.k_rows[rows].to(dev).contiguous()
        v_new = wl.v_rows[rows].to(dev).contiguous()
        start = torch.from_numpy(wl.context_lens.astype(np.int32)).to(dev)
        cu = torch.arange(wl.num_seqs + 1, dtype=torch.int32, device=dev)
        lens = start + 1
        return k_new, v_new, start, cu, lens

    def run_step(self, q=None, hint=0):
        """Append the new token of every sequence, then decode over context + 1."""
        wl = self.wl
        k_new, v_new, start, cu, lens = self.step_inputs()
        pk.append_kv(self.k, self.v, k_new, v_new, self.tables, start, cu, err_flag=self.err)
        return self.decode(lens, q=q, hint=hint)

    def run_step_one_call(self, hint=0, shared=0):
        """The same step as one pa_append_decode_attention call (with a shared prefix of
        `shared` tokens, pa_append_decode_attention_shared_prefix): the bench's bf16 step."""
        wl = self.wl
        k_new, v_new, start, cu, lens = self.step_inputs()
        q = wl.q.to(self.k.device).contiguous()
        out = torch.empty_like(q)
        ws = pk.decode_workspace(q.shape[0], wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                 self.tables.shape[1], device=self.k.device)
        if shared:
            pk.append_decode_attention_shared_prefix(out, q, self.k, self.v, k_new, v_new,
                                                     self.tables, lens, wl.scale, shared,
                                                     workspace=ws, max_context_len_hint=hint,
                                                     err_flag=self.err)
        else:
            pk.append_decode_attention(out, q, self.k, self.v, k_new, v_new, self.tables, lens,
                                       wl.scale, workspace=ws, max_context_len_hint=hint,
                                       err_flag=self.err)
        return out

    def decode(self, lens, q=None, hint=0, tables=None):
        wl = self.wl
        q = (wl.q if q is None else q).to(self.k.device).contiguous()
        tables = self.tables if tables is None else tables
        out = torch.empty_like(q)
        ws = pk.decode_workspace(q.shape[0], wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                 tables.shape[1], device=self.k.device)
        pk.decode_attention(out, q, self.k, self.v, tables, lens, wl.scale, workspace=ws,
                            max_context_len_hint=hint, err_flag=self.err)
        return out


def oracle_pools(wl):
    """The oracle's own pools for the workload (its own append), before the step's append."""
    od = odtype(wl)
    et = np.uint16 if od == orc.BF16 else np.uint32
    shape = orc.pool_shape(wl.num_blocks, wl.num_kv_heads, wl.head_dim, od)
    kp = np.full(shape, CANARY_BF16 if od == orc.BF16 else CANARY_F32, et)
    vp = np.full(shape, CANARY_BF16 if od == orc.BF16 else CANARY_F32, et)
    if od == orc.F32:
        kp, vp = kp.view(np.float32), vp.view(np.float32)
    kr, vr = wl.k_rows.cpu(), wl.v_rows.cpu()
    for (s, start, first, n) in wl.fill:
        rc = orc.append_kv(kp, vp, kr[first:first + n], vr[first:first + n],
                           wl.block_tables[s:s + 1], np.array([start], np.int32),
                           np.array([0, n], np.int32), num_kv_heads=wl.num_kv_heads,
                           head_dim=wl.head_dim, num_blocks=wl.num_blocks, dtype=od)
        assert rc == 0
    return kp, vp


def oracle_step_append(wl, kp, vp):
    od = odtype(wl)
    rows = torch.from_numpy(wl.new_rows)
    rc = orc.append_kv(kp, vp, wl.k_rows.cpu()[rows], wl.v_rows.cpu()[rows], wl.block_tables,
                       wl.context_lens.astype(np.int32), np.arange(wl.num_seqs + 1, dtype=np.int32),
                       num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
                       num_blocks=wl.num_blocks, dtype=od)
    assert rc == 0


def oracle_contig(wl, pairs, q=None, lens_after=None):
    """Oracle outputs (float64 [n][D]) for (sequence, query head) pairs, computed on
    each sequence's logical rows with no paging at all."""
    od = odtype(wl)
    q = (wl.q if q is None else q).cpu()
    kr, vr = wl.k_rows.cpu(), wl.v_rows.cpu()
    G = wl.num_q_heads // wl.num_kv_heads
    out = np.zeros((len(pairs), wl.head_dim))
    cache = {}
    for i, (s, h) in enumerate(pairs):
        if s not in cache:
            rows = torch.from_numpy(wl.logical_rows(s))
            if lens_after is not None:
                rows = rows[:int(lens_after[s])]
            cache = {s: (kr[rows].contiguous(), vr[rows].contiguous())}
        K, V = cache[s]
        out[i] = orc.decode_contig(q[s, h], K, V, h // G, num_kv_heads=wl.num_kv_heads,
                                   head_dim=wl.head_dim, scale=wl.scale, dtype=od)
    return out


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def assert_close(wl, got: np.ndarray, want: np.ndarray, what=""):
    """got, want: [..., D] float64 arrays."""
    if wl.dtype == "bf16":
        err = np.abs(got - want).max() if got.size else 0.0
        assert err <= BF16_ATOL, f"{what}: max abs error {err} > {BF16_ATOL}"
    else:
        num = np.abs(got - want).max(axis=-1)
        den = np.maximum(np.abs(want).max(axis=-1), 1e-30)
        rel = (num / den).max() if got.size else 0.0
        assert rel <= F32_ROW_RTOL, f"{what}: max row-relative error {rel} > {F32_ROW_RTOL}"


def pool_bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.view(torch.int32).cpu().numpy().view(np.uint32)


def np_bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint16) if a.dtype == np.uint16 else a.view(np.uint32)

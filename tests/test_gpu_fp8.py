"""GPU parity of the FP8 (E4M3) KV cache: quantising append and decode.

The quantised pools (codes and per-slot scales) must equal, byte for byte, the
pools the oracle builds from the same bf16 rows with its own quantisation; the
decode must match the oracle's attention over the dequantised cache within the
bf16 tolerance.  Slots past each context hold NaN codes that must not leak.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_207_gb300 as pk
from paged_kv_cache_207_gb300 import workloads as W
from _gpu_common import BF16_ATOL
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


class Fp8Pools:
    def __init__(self, wl, nan_fill=True):
        self.wl = wl
        shape = pk.fp8_pool_shape(wl.num_blocks, wl.num_kv_heads, wl.head_dim)
        self.k = torch.full(shape, 0x7F if nan_fill else 0, dtype=torch.uint8, device="cuda")
        self.v = torch.full(shape, 0x7F if nan_fill else 0, dtype=torch.uint8, device="cuda")
        self.tables = torch.from_numpy(wl.block_tables).cuda()
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        seqs = [f[0] for f in wl.fill]
        ns = [f[3] for f in wl.fill]
        first, end = wl.fill[0][2], wl.fill[-1][2] + wl.fill[-1][3]
        pk.append_kv_fp8(self.k, self.v, wl.k_rows[first:end].contiguous(),
                         wl.v_rows[first:end].contiguous(),
                         self.tables[torch.tensor(seqs, device="cuda")].contiguous(),
                         torch.tensor([f[1] for f in wl.fill], dtype=torch.int32, device="cuda"),
                         torch.tensor(np.concatenate([[0], np.cumsum(ns)]), dtype=torch.int32,
                                      device="cuda"), err_flag=self.err)

    def step(self, hint=0):
        wl = self.wl
        rows = torch.from_numpy(wl.new_rows).cuda()
        start = torch.from_numpy(wl.context_lens.astype(np.int32)).cuda()
        cu = torch.arange(wl.num_seqs + 1, dtype=torch.int32, device="cuda")
        pk.append_kv_fp8(self.k, self.v, wl.k_rows[rows].contiguous(), wl.v_rows[rows].contiguous(),
                         self.tables, start, cu, err_flag=self.err)
        return self.decode(start + 1, hint=hint)

    def step_one_call(self, hint=0):
        """The same step as one pa_append_decode_attention_fp8 call (the bench's FP8 step)."""
        wl = self.wl
        rows = torch.from_numpy(wl.new_rows).cuda()
        lens = torch.from_numpy(wl.context_lens.astype(np.int32)).cuda() + 1
        out = torch.empty_like(wl.q)
        ws = pk.decode_workspace(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                 self.tables.shape[1])
        pk.append_decode_attention_fp8(out, wl.q, self.k, self.v, wl.k_rows[rows].contiguous(),
                                       wl.v_rows[rows].contiguous(), self.tables, lens, wl.scale,
                                       workspace=ws, max_context_len_hint=hint, err_flag=self.err)
        torch.cuda.synchronize()
        return out

    def decode(self, lens, q=None, tables=None, hint=0):
        wl = self.wl
        q = wl.q if q is None else q
        tables = self.tables if tables is None else tables
        out = torch.empty_like(q)
        ws = pk.decode_workspace(q.shape[0], wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                 tables.shape[1])
        pk.decode_attention_fp8(out, q, self.k, self.v, tables, lens, wl.scale, workspace=ws,
                                max_context_len_hint=hint, err_flag=self.err)
        torch.cuda.synchronize()
        return out


def oracle_fp8_pools(wl, with_step=True):
    shape = orc.fp8_pool_shape(wl.num_blocks, wl.num_kv_heads, wl.head_dim)
    kp = np.full(shape, 0x7F, np.uint8)
    vp = np.full(shape, 0x7F, np.uint8)
    kr, vr = wl.k_rows.cpu(), wl.v_rows.cpu()
    for (s, start, first, n) in wl.fill:
        assert orc.append_kv_fp8(kp, vp, kr[first:first + n], vr[first:first + n],
                                 wl.block_tables[s:s + 1], np.array([start], np.int32),
                                 np.array([0, n], np.int32), num_kv_heads=wl.num_kv_heads,
                                 head_dim=wl.head_dim, num_blocks=wl.num_blocks) == 0
    if with_step:
        rows = torch.from_numpy(wl.new_rows)
        assert orc.append_kv_fp8(kp, vp, kr[rows], vr[rows], wl.block_tables,
                                 wl.context_lens.astype(np.int32),
                                 np.arange(wl.num_seqs + 1, dtype=np.int32),
                                 num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
                                 num_blocks=wl.num_blocks) == 0
    return kp, vp


def _oracle_out(wl, kp, vp, pairs):
    return orc.decode_fp8_pairs(pairs, wl.q.cpu(), kp, vp, wl.block_tables,
                                (wl.context_lens + 1).astype(np.int32),
                                num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
                                head_dim=wl.head_dim, num_blocks=wl.num_blocks, scale=wl.scale)


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (14, 2, 64), (12, 12, 64), (8, 1, 128)])
def test_fp8_append_bit_exact_and_decode_against_oracle(hq, hkv, d):
    lens = [1, 15, 16, 17, 100, 511, 512, 513, 1500, 2047]
    wl = W.make_decode_workload("fp8", context_lens=np.array(lens) - 1, num_q_heads=hq,
                                num_kv_heads=hkv, head_dim=d, dtype="bf16", seed=hq + d,
                                device="cuda", pool_blocks=500)
    fp = Fp8Pools(wl)
    out = fp.step()
    assert int(fp.err.item()) == 0
    kp, vp = oracle_fp8_pools(wl)
    assert np.array_equal(fp.k.cpu().numpy(), kp)
    assert np.array_equal(fp.v.cpu().numpy(), vp)
    pairs = [(s, h) for s in range(wl.num_seqs) for h in range(hq)]
    want = _oracle_out(wl, kp, vp, pairs)
    got = out.float().cpu().double().numpy().reshape(len(pairs), d)
    err = np.abs(got - want).max()
    assert err <= BF16_ATOL, err
    assert torch.isfinite(out.float()).all()


def test_fp8_batched_equals_alone_bitwise():
    wl = W.make_decode_workload("fp8b", context_lens=[5, 700, 1300, 63, 2100], num_q_heads=32,
                                num_kv_heads=8, head_dim=128, dtype="bf16", seed=4, device="cuda")
    fp = Fp8Pools(wl)
    batched = fp.step()
    lens = torch.from_numpy(wl.context_lens.astype(np.int32)).cuda() + 1
    for s in range(wl.num_seqs):
        alone = fp.decode(lens[s:s + 1], q=wl.q[s:s + 1], tables=fp.tables[s:s + 1].contiguous())
        assert torch.equal(alone[0], batched[s]), s


def test_fp8_copy_block_bit_exact():
    Hkv, D, nb = 8, 128, 20
    shape = pk.fp8_pool_shape(nb, Hkv, D)
    g = torch.Generator(device="cuda").manual_seed(5)
    kp = torch.randint(0, 255, shape, dtype=torch.uint8, device="cuda", generator=g)
    vp = torch.randint(0, 255, shape, dtype=torch.uint8, device="cuda", generator=g)
    k0, v0 = kp.clone(), vp.clone()
    pk.copy_block_fp8(kp, vp, torch.tensor([[2, 9], [19, 0]], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(kp[9], k0[2]) and torch.equal(vp[0], v0[19])
    assert torch.equal(kp[1], k0[1]) and torch.equal(vp[5], v0[5])


@pytest.mark.parametrize("one_call", [False, True])
def test_fp8_llama_batch_full_size_sampled(one_call):
    # the 256-sequence workload at full size, as append + decode and as the bench's one call
    wl = W.llama8b_batch(device="cuda")
    fp = Fp8Pools(wl, nan_fill=False)
    hint = int(wl.context_lens.max()) + 1
    out = fp.step_one_call(hint=hint) if one_call else fp.step(hint=hint)
    assert int(fp.err.item()) == 0
    rng = np.random.default_rng(8)
    seqs = sorted(set(rng.choice(wl.num_seqs, 12, replace=False).tolist()) |
                  {int(np.argmax(wl.context_lens))})
    # the oracle's own pools, only for the sampled sequences (others left unfilled)
    shape = orc.fp8_pool_shape(wl.num_blocks, wl.num_kv_heads, wl.head_dim)
    kp = np.zeros(shape, np.uint8)
    vp = np.zeros(shape, np.uint8)
    kr, vr = wl.k_rows.cpu(), wl.v_rows.cpu()
    for (s, start, first, n) in wl.fill:
        if s in seqs:
            orc.append_kv_fp8(kp, vp, kr[first:first + n], vr[first:first + n],
                              wl.block_tables[s:s + 1], np.array([start], np.int32),
                              np.array([0, n], np.int32), num_kv_heads=8, head_dim=128,
                              num_blocks=wl.num_blocks)
    rows = torch.from_numpy(wl.new_rows)
    orc.append_kv_fp8(kp, vp, kr[rows], vr[rows], wl.block_tables, wl.context_lens.astype(np.int32),
                      np.arange(wl.num_seqs + 1, dtype=np.int32), num_kv_heads=8, head_dim=128,
                      num_blocks=wl.num_blocks)
    pairs = [(s, int(rng.integers(32))) for s in seqs]
    want = _oracle_out(wl, kp, vp, pairs)
    got = np.stack([out[s, h].float().cpu().double().numpy() for s, h in pairs])
    err = np.abs(got - want).max()
    assert err <= BF16_ATOL, err

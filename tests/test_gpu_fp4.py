"""GPU parity of the block-scaled FP4 (MXFP4) cache against the oracle.

The pools the library's quantising append writes must equal the oracle append's
bytes exactly (codes, nibble order, scales; canary bytes where nothing was
written), including rows of one call that share V bytes.  Decode over the
quantised cache must match the oracle's decode of the same codes within the
bf16 tolerance of the parity tests.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_207_gb300 as pk
from paged_kv_cache_207_gb300 import workloads as W
from _gpu_common import BF16_ATOL
from oracle import oracle as orc

pytestmark = pytest.mark.gpu
CANARY = 0xFF            # codes -6 / -6 and scale byte 255 (not a scale the append writes)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_207_gb300 import build
    build.build()
    pk.lib()


class Fp4Pools:
    def __init__(self, wl, canary=True):
        self.wl = wl
        shape = pk.fp4_pool_shape(wl.num_blocks, wl.num_kv_heads, wl.head_dim)
        self.k = torch.full(shape, CANARY if canary else 0, dtype=torch.uint8, device="cuda")
        self.v = torch.full(shape, CANARY if canary else 0, dtype=torch.uint8, device="cuda")
        self.tables = torch.from_numpy(wl.block_tables).cuda()
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        seqs = [f[0] for f in wl.fill]
        ns = [f[3] for f in wl.fill]
        first, end = wl.fill[0][2], wl.fill[-1][2] + wl.fill[-1][3]
        pk.append_kv_fp4(self.k, self.v, wl.k_rows[first:end].contiguous(),
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
        pk.append_kv_fp4(self.k, self.v, wl.k_rows[rows].contiguous(), wl.v_rows[rows].contiguous(),
                         self.tables, start, cu, err_flag=self.err)
        return self.decode(start + 1, hint=hint)

    def decode(self, lens, q=None, tables=None, hint=0):
        wl = self.wl
        q = wl.q if q is None else q
        tables = self.tables if tables is None else tables
        out = torch.empty_like(q)
        ws = pk.decode_workspace(q.shape[0], wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                 tables.shape[1])
        pk.decode_attention_fp4(out, q, self.k, self.v, tables, lens, wl.scale, workspace=ws,
                                max_context_len_hint=hint, err_flag=self.err)
        torch.cuda.synchronize()
        return out


def oracle_fp4_pools(wl, seqs=None, canary=True):
    shape = orc.fp4_pool_shape(wl.num_blocks, wl.num_kv_heads, wl.head_dim)
    kp = np.full(shape, CANARY if canary else 0, np.uint8)
    vp = np.full(shape, CANARY if canary else 0, np.uint8)
    kr, vr = wl.k_rows.cpu(), wl.v_rows.cpu()
    for (s, start, first, n) in wl.fill:
        if seqs is None or s in seqs:
            assert orc.append_kv_fp4(kp, vp, kr[first:first + n], vr[first:first + n],
                                     wl.block_tables[s:s + 1], np.array([start], np.int32),
                                     np.array([0, n], np.int32), num_kv_heads=wl.num_kv_heads,
                                     head_dim=wl.head_dim, num_blocks=wl.num_blocks) == 0
    rows = torch.from_numpy(wl.new_rows)
    assert orc.append_kv_fp4(kp, vp, kr[rows], vr[rows], wl.block_tables,
                             wl.context_lens.astype(np.int32),
                             np.arange(wl.num_seqs + 1, dtype=np.int32),
                             num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
                             num_blocks=wl.num_blocks) == 0
    return kp, vp


def _oracle_out(wl, kp, vp, pairs):
    return orc.decode_fp4_pairs(pairs, wl.q.cpu(), kp, vp, wl.block_tables,
                                (wl.context_lens + 1).astype(np.int32),
                                num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
                                head_dim=wl.head_dim, num_blocks=wl.num_blocks, scale=wl.scale)


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (14, 2, 64), (12, 12, 64), (8, 1, 128)])
def test_fp4_append_bit_exact_and_decode_against_oracle(hq, hkv, d):
    lens = [1, 15, 16, 17, 100, 511, 512, 513, 2047, 2048, 2049, 4100]
    wl = W.make_decode_workload("fp4", context_lens=np.array(lens) - 1, num_q_heads=hq,
                                num_kv_heads=hkv, head_dim=d, dtype="bf16", seed=hq + d + 1,
                                device="cuda", pool_blocks=900)
    fp = Fp4Pools(wl)
    out = fp.step()
    assert int(fp.err.item()) == 0
    kp, vp = oracle_fp4_pools(wl)
    assert np.array_equal(fp.k.cpu().numpy(), kp)
    assert np.array_equal(fp.v.cpu().numpy(), vp)
    pairs = [(s, h) for s in range(wl.num_seqs) for h in range(hq)]
    want = _oracle_out(wl, kp, vp, pairs)
    got = out.float().cpu().double().numpy().reshape(len(pairs), d)
    err = np.abs(got - want).max()
    assert err <= BF16_ATOL, err
    assert torch.isfinite(out.float()).all()


def test_fp4_value_scales_spanning_many_octaves():
    # tokens whose values differ by up to 2^24 in magnitude: the per-block reference
    # exponent rises mid-partition and the outputs are rescaled; compared relative to
    # each row's size
    S, Hkv, D = 3, 2, 128
    lens = [300, 1500, 2600]
    wl = W.make_decode_workload("fp4_range", context_lens=np.array(lens) - 1, num_q_heads=8,
                                num_kv_heads=Hkv, head_dim=D, dtype="bf16", seed=17, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(18)
    mag = 2.0 ** torch.randint(-12, 13, (wl.v_rows.shape[0], Hkv, 1), generator=g, device="cuda")
    wl.v_rows = (wl.v_rows.float() * mag).to(torch.bfloat16)
    fp = Fp4Pools(wl)
    out = fp.step()
    assert int(fp.err.item()) == 0
    kp, vp = oracle_fp4_pools(wl)
    assert np.array_equal(fp.v.cpu().numpy(), vp)
    pairs = [(s, h) for s in range(S) for h in range(8)]
    want = _oracle_out(wl, kp, vp, pairs)
    got = out.float().cpu().double().numpy().reshape(len(pairs), D)
    rel = (np.abs(got - want).max(axis=1) / np.abs(want).max(axis=1)).max()
    assert rel <= BF16_ATOL, rel


def test_fp4_batched_equals_alone_bitwise():
    wl = W.make_decode_workload("fp4b", context_lens=[5, 700, 2300, 63, 4500], num_q_heads=32,
                                num_kv_heads=8, head_dim=128, dtype="bf16", seed=6, device="cuda")
    fp = Fp4Pools(wl)
    batched = fp.step()
    lens = torch.from_numpy(wl.context_lens.astype(np.int32)).cuda() + 1
    for s in range(wl.num_seqs):
        alone = fp.decode(lens[s:s + 1], q=wl.q[s:s + 1], tables=fp.tables[s:s + 1].contiguous())
        assert torch.equal(alone[0], batched[s]), s


def test_fp4_copy_block_bit_exact():
    Hkv, D, nb = 8, 128, 20
    shape = pk.fp4_pool_shape(nb, Hkv, D)
    g = torch.Generator(device="cuda").manual_seed(7)
    kp = torch.randint(0, 255, shape, dtype=torch.uint8, device="cuda", generator=g)
    vp = torch.randint(0, 255, shape, dtype=torch.uint8, device="cuda", generator=g)
    k0, v0 = kp.clone(), vp.clone()
    pk.copy_block_fp4(kp, vp, torch.tensor([[2, 9], [19, 0]], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(kp[9], k0[2]) and torch.equal(vp[0], v0[19])
    assert torch.equal(kp[1], k0[1]) and torch.equal(vp[5], v0[5])


def test_fp4_llama_batch_full_size_sampled():
    wl = W.llama8b_batch(device="cuda")
    fp = Fp4Pools(wl, canary=False)
    out = fp.step(hint=int(wl.context_lens.max()) + 1)
    assert int(fp.err.item()) == 0
    rng = np.random.default_rng(9)
    seqs = sorted(set(rng.choice(wl.num_seqs, 12, replace=False).tolist()) |
                  {int(np.argmax(wl.context_lens))})
    kp, vp = oracle_fp4_pools(wl, seqs=seqs, canary=False)
    pairs = [(s, int(rng.integers(32))) for s in seqs]
    want = _oracle_out(wl, kp, vp, pairs)
    got = np.stack([out[s, h].float().cpu().double().numpy() for s, h in pairs])
    err = np.abs(got - want).max()
    assert err <= BF16_ATOL, err

"""GPU parity: the CUDA library against the CPU oracle, through the C ABI.

Sizes span several 16-token blocks, several 512-token split-KV partitions and
ragged tails; the five named workloads run at full size with sampled outputs
checked one by one against the oracle.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_207_gb300 as pk
from paged_kv_cache_207_gb300 import workloads as W
from _gpu_common import (DevicePools, as_f64, assert_close, np_bits, oracle_contig, oracle_pools,
                         oracle_step_append, pool_bits)
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

RAGGED = [0, 1, 15, 16, 17, 100, 511, 512, 513, 1024, 1500, 2047]


def _all_pairs(wl):
    return [(s, h) for s in range(wl.num_seqs) for h in range(wl.num_q_heads)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_207_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    pk.lib()


def test_gpt2_tiny_f32_pools_bit_exact_and_outputs_within_tolerance():
    wl = W.gpt2_tiny_f32(device="cuda")
    dp = DevicePools(wl)
    kp, vp = oracle_pools(wl)
    assert np.array_equal(pool_bits(dp.k), np_bits(kp)) and np.array_equal(pool_bits(dp.v), np_bits(vp))
    out = dp.run_step()
    oracle_step_append(wl, kp, vp)
    assert np.array_equal(pool_bits(dp.k), np_bits(kp)) and np.array_equal(pool_bits(dp.v), np_bits(vp))
    lens = wl.context_lens + 1
    want = orc.decode(wl.q, kp, vp, wl.block_tables, lens.astype(np.int32),
                      num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
                      head_dim=wl.head_dim, num_blocks=wl.num_blocks, scale=wl.scale, dtype=orc.F32)
    assert_close(wl, as_f64(out), want, "gpt2 tiny fp32")
    assert int(dp.err.item()) == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("hq,hkv,d", [(12, 12, 64), (14, 2, 64), (32, 8, 128), (8, 1, 128),
                                      (4, 4, 128), (16, 2, 64)])
def test_ragged_lengths_against_oracle(dtype, hq, hkv, d):
    lens = [L for L in RAGGED if L > 0]
    wl = W.make_decode_workload("ragged", context_lens=np.array(lens) - 1, num_q_heads=hq,
                                num_kv_heads=hkv, head_dim=d, dtype=dtype, seed=hq * 31 + d,
                                device="cuda", pool_blocks=600)
    dp = DevicePools(wl)
    out = dp.run_step()
    pairs = _all_pairs(wl)
    want = oracle_contig(wl, pairs)
    assert_close(wl, as_f64(out).reshape(len(pairs), d), want, f"{dtype} {hq}/{hkv}x{d}")
    assert int(dp.err.item()) == 0


def test_zero_length_context_gives_zeros_and_no_nan():
    wl = W.make_decode_workload("zero", context_lens=[0, 40, 0, 600], num_q_heads=8,
                                num_kv_heads=2, head_dim=128, dtype="bf16", seed=5, device="cuda")
    dp = DevicePools(wl)
    lens = torch.tensor([0, 41, 0, 601], dtype=torch.int32, device="cuda")
    k_new, v_new, start, cu, _ = dp.step_inputs()
    pk.append_kv(dp.k, dp.v, k_new, v_new, dp.tables, start, cu, err_flag=dp.err)
    out = dp.decode(lens)
    o = as_f64(out)
    assert np.all(o[0] == 0) and np.all(o[2] == 0) and np.all(np.isfinite(o))
    want = oracle_contig(wl, [(1, h) for h in range(8)], lens_after=[0, 41, 0, 601])
    assert_close(wl, o[1], want)


def test_batched_equals_alone_bitwise():
    wl = W.make_decode_workload("batch", context_lens=[5, 700, 1300, 63, 2100, 512], num_q_heads=32,
                                num_kv_heads=8, head_dim=128, dtype="bf16", seed=8, device="cuda")
    dp = DevicePools(wl)
    batched = dp.run_step()
    _, _, start, _, lens = dp.step_inputs()
    for s in range(wl.num_seqs):
        alone = dp.decode(lens[s:s + 1], q=wl.q[s:s + 1], tables=dp.tables[s:s + 1].contiguous())
        assert torch.equal(alone[0], batched[s]), s


def test_paged_equals_contiguous_bitwise():
    # identical logical data through a shuffled table and through an identity table
    lens = [37, 513, 1100]
    wl = W.make_decode_workload("shuffled", context_lens=np.array(lens) - 1, num_q_heads=14,
                                num_kv_heads=2, head_dim=64, dtype="bf16", seed=13, device="cuda",
                                pool_blocks=400)
    dp = DevicePools(wl)
    shuffled = dp.run_step()
    ident = W.make_decode_workload("identity", context_lens=np.array(lens) - 1, num_q_heads=14,
                                   num_kv_heads=2, head_dim=64, dtype="bf16", seed=13, device="cuda",
                                   pool_blocks=400)
    need = [(L + 15) // 16 for L in lens]
    tbl = np.full_like(ident.block_tables, -1)
    k = 0
    for s, n in enumerate(need):
        tbl[s, :n] = np.arange(k, k + n)
        k += n
    ident.block_tables = tbl
    di = DevicePools(ident)
    contiguous = di.run_step()
    assert torch.equal(shuffled, contiguous)


def test_copy_on_write_child_matches_parent_and_leaves_parent_untouched():
    torch.manual_seed(0)
    Hq, Hkv, D = 32, 8, 128
    bm = pk.BlockManager(64)
    parent = bm.add_seq()
    bm.prepare_append(parent, 0, 20)         # blocks [a, b], b partial (4 tokens)
    child = bm.fork(parent)
    shape = pk.pool_shape(64, Hkv, D, torch.bfloat16)
    kp = torch.randn(shape, device="cuda").to(torch.bfloat16)
    vp = torch.randn(shape, device="cuda").to(torch.bfloat16)
    q = torch.randn(2, Hq, D, device="cuda").to(torch.bfloat16)
    q[1] = q[0]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def tables():
        return torch.tensor([bm.block_table(parent, 4), bm.block_table(child, 4)],
                            dtype=torch.int32, device="cuda")

    def decode(lens):
        out = torch.empty_like(q)
        pk.decode_attention(out, q, kp, vp, tables(), torch.tensor(lens, dtype=torch.int32,
                            device="cuda"), 0.088, err_flag=err)
        return out

    before = decode([20, 20])
    assert torch.equal(before[0], before[1])
    parent_bytes = (kp.clone(), vp.clone())
    # child appends one token at position 20: the shared partial block is copied first
    pairs = bm.prepare_append(child, 20, 1)
    assert len(pairs) == 1
    pk.copy_block(kp, vp, torch.tensor(pairs, dtype=torch.int32, device="cuda"), err_flag=err)
    src, dst = pairs[0]
    assert torch.equal(kp[dst], kp[src]) and torch.equal(vp[dst], vp[src])
    t = tables()
    k_new = torch.randn(1, Hkv, D, device="cuda").to(torch.bfloat16)
    v_new = torch.randn(1, Hkv, D, device="cuda").to(torch.bfloat16)
    pk.append_kv(kp, vp, k_new, v_new, t[1:2].contiguous(),
                 torch.tensor([20], dtype=torch.int32, device="cuda"),
                 torch.tensor([0, 1], dtype=torch.int32, device="cuda"), err_flag=err)
    # every block but the child's fresh copy is byte-identical to before
    changed = [b for b in range(64) if not (torch.equal(kp[b], parent_bytes[0][b]) and
                                            torch.equal(vp[b], parent_bytes[1][b]))]
    assert changed == [dst]
    after = decode([20, 21])
    assert torch.equal(after[0], before[0])
    assert int(err.item()) == 0


def test_gqa_equals_mha_with_replicated_kv_heads():
    G = 4
    wl = W.make_decode_workload("gqa", context_lens=[30, 600, 1200], num_q_heads=32, num_kv_heads=8,
                                head_dim=128, dtype="bf16", seed=21, device="cuda")
    dp = DevicePools(wl)
    gqa = dp.run_step()
    rep = W.make_decode_workload("mha", context_lens=[30, 600, 1200], num_q_heads=32,
                                 num_kv_heads=32, head_dim=128, dtype="bf16", seed=21,
                                 device="cuda")
    rep.q = wl.q
    rep.k_rows = wl.k_rows.repeat_interleave(G, dim=1).contiguous()
    rep.v_rows = wl.v_rows.repeat_interleave(G, dim=1).contiguous()
    dr = DevicePools(rep)
    mha = dr.run_step()
    assert_close(wl, as_f64(gqa), as_f64(mha))
    assert torch.equal(gqa, mha)


def test_twelve_layers_append_at_explicit_start_then_decode_sees_every_token():
    # spindle, "Two bugs worth recording": twelve layers each append the new token at the
    # same explicit start position and decode with the explicit length start + 1.
    layers = [W.make_decode_workload("layer", context_lens=[16, 47, 300], num_q_heads=12,
                                     num_kv_heads=12, head_dim=64, dtype="bf16", seed=100 + l,
                                     device="cuda") for l in range(12)]
    for wl in layers:
        dp = DevicePools(wl)
        out = dp.run_step()
        want = oracle_contig(wl, _all_pairs(wl))
        assert_close(wl, as_f64(out).reshape(-1, 64), want)
        # a length that misses the appended token gives a different answer
        short = dp.decode(torch.from_numpy(wl.context_lens.astype(np.int32)).cuda())
        assert not torch.equal(short, out)


def test_bf16_append_pools_bit_exact_llama_heads_chunked_and_ragged():
    """bf16 pools at the Llama-3-8B head shape (8 kv heads x 128): every sequence's context
    goes in as two chunks (two calls at explicit starts, chunks crossing block borders),
    then one step's token; after each call the device pools equal the oracle append's
    bytes, NaN canaries in every slot nothing wrote included."""
    ctx = [1, 15, 16, 17, 100, 513, 40]
    wl = W.make_decode_workload("append_bf16", context_lens=ctx, num_q_heads=32, num_kv_heads=8,
                                head_dim=128, dtype="bf16", seed=91, device="cuda", pool_blocks=80)
    shape = pk.pool_shape(wl.num_blocks, 8, 128, torch.bfloat16)
    kd = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    vd = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    kd.view(torch.int16).fill_(-1)          # 0xFFFF: a NaN no N(0, 1) draw gives
    vd.view(torch.int16).fill_(-1)
    tables = torch.from_numpy(wl.block_tables).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ko = np.full(orc.pool_shape(wl.num_blocks, 8, 128, orc.BF16), 0xFFFF, np.uint16)
    vo = ko.copy()
    kr, vr = wl.k_rows.cpu(), wl.v_rows.cpu()
    cut = [c // 2 + (c % 3) for c in ctx]     # first chunk: positions [0, cut)
    for lo_of, hi_of in ((lambda s: 0, lambda s: min(cut[s], ctx[s])),
                         (lambda s: min(cut[s], ctx[s]), lambda s: ctx[s])):
        rows, starts, ns = [], [], []
        for s in range(wl.num_seqs):
            logical = wl.logical_rows(s)
            a, b = lo_of(s), hi_of(s)
            rows.append(logical[a:b])
            starts.append(a)
            ns.append(b - a)
        idx = torch.from_numpy(np.concatenate(rows))
        cu = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
        pk.append_kv(kd, vd, wl.k_rows[idx.cuda()].contiguous(), wl.v_rows[idx.cuda()].contiguous(),
                     tables, torch.tensor(starts, dtype=torch.int32, device="cuda"),
                     torch.from_numpy(cu).cuda(), err_flag=err)
        assert orc.append_kv(ko, vo, kr[idx], vr[idx], wl.block_tables, np.array(starts, np.int32),
                             cu, num_kv_heads=8, head_dim=128, num_blocks=wl.num_blocks,
                             dtype=orc.BF16) == 0
        torch.cuda.synchronize()
        assert np.array_equal(pool_bits(kd), ko) and np.array_equal(pool_bits(vd), vo)
    k_new, v_new = wl.k_rows[torch.from_numpy(wl.new_rows).cuda()], wl.v_rows[torch.from_numpy(wl.new_rows).cuda()]
    start = torch.from_numpy(wl.context_lens.astype(np.int32)).cuda()
    pk.append_kv(kd, vd, k_new.contiguous(), v_new.contiguous(), tables, start,
                 torch.arange(wl.num_seqs + 1, dtype=torch.int32, device="cuda"), err_flag=err)
    oracle_step_append(wl, ko, vo)
    torch.cuda.synchronize()
    assert np.array_equal(pool_bits(kd), ko) and np.array_equal(pool_bits(vd), vo)
    assert int(err.item()) == 0
    # slots nothing wrote still hold the canary
    assert int((ko == 0xFFFF).sum()) > 0


def test_copy_block_bit_exact_against_oracle():
    Hkv, D, nb = 8, 128, 40
    shape = pk.pool_shape(nb, Hkv, D, torch.bfloat16)
    g = torch.Generator(device="cuda").manual_seed(3)
    kp = torch.randint(-32768, 32767, shape, dtype=torch.int16, device="cuda", generator=g).view(torch.bfloat16)
    vp = torch.randint(-32768, 32767, shape, dtype=torch.int16, device="cuda", generator=g).view(torch.bfloat16)
    ko, vo = kp.view(torch.int16).cpu().numpy().view(np.uint16).copy(), vp.view(torch.int16).cpu().numpy().view(np.uint16).copy()
    pairs = [(1, 7), (3, 3), (10, 30), (39, 0)]
    pk.copy_block(kp, vp, torch.tensor(pairs, dtype=torch.int32, device="cuda"))
    assert orc.copy_block(ko, vo, pairs, num_blocks=nb, num_kv_heads=Hkv, head_dim=D, dtype=orc.BF16) == 0
    assert np.array_equal(pool_bits(kp), ko) and np.array_equal(pool_bits(vp), vo)


def test_device_errors_are_flagged_and_skipped_without_faulting():
    Hkv, D, nb = 2, 64, 8
    shape = pk.pool_shape(nb, Hkv, D, torch.bfloat16)
    kp = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rows = torch.ones(2, Hkv, D, dtype=torch.bfloat16, device="cuda")
    # table entry 99 is outside the pool; position 40 is beyond a 2-block table
    tables = torch.tensor([[1, 99], [2, 3]], dtype=torch.int32, device="cuda")
    pk.append_kv(kp, vp, rows, rows, tables, torch.tensor([16, 40], dtype=torch.int32, device="cuda"),
                 torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda"), err_flag=err)
    assert int(err.item()) == pk.DEV_ERR_BAD_BLOCK | pk.DEV_ERR_BAD_POS
    assert int((kp != 0).sum().item()) == 0 and int((vp != 0).sum().item()) == 0
    # decode over a context whose second block is out of range: that block is skipped
    err.zero_()
    q = torch.zeros(2, 4, D, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    pk.decode_attention(out, q, kp, vp, tables, torch.tensor([20, 33], dtype=torch.int32, device="cuda"),
                        0.125, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == pk.DEV_ERR_BAD_BLOCK | pk.DEV_ERR_BAD_POS
    assert torch.isfinite(out.float()).all()
    # a context that needs more split-KV partitions than the host hint allows is flagged
    # (hint 300: one partition of 1024 tokens at head_dim 64; the context needs two)
    err.zero_()
    tables = torch.tensor([[0, 1, 2, 3, 4, 5, 6, 7] * 12], dtype=torch.int32, device="cuda")
    q1 = torch.zeros(1, 4, D, dtype=torch.bfloat16, device="cuda")
    out1 = torch.empty_like(q1)
    ws = pk.decode_workspace(1, 4, Hkv, D, 96)
    assert pk.partition_tokens(D) == 1024
    pk.decode_attention(out1, q1, kp, vp, tables, torch.tensor([1500], dtype=torch.int32, device="cuda"),
                        0.125, workspace=ws, max_context_len_hint=300, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pk.DEV_ERR_HINT


def test_output_guard_regions_untouched():
    wl = W.make_decode_workload("guard", context_lens=[100, 900], num_q_heads=8, num_kv_heads=2,
                                head_dim=128, dtype="bf16", seed=4, device="cuda")
    dp = DevicePools(wl)
    k_new, v_new, start, cu, lens = dp.step_inputs()
    pk.append_kv(dp.k, dp.v, k_new, v_new, dp.tables, start, cu)
    n = wl.q.numel()
    buf = torch.full((n + 2048,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[1024:1024 + n].view(wl.q.shape)
    ws_b = pk.decode_workspace_size(2, 8, 2, 128, wl.max_blocks)
    ws = torch.zeros(ws_b + 4096, dtype=torch.uint8, device="cuda")
    pk.decode_attention(out, wl.q.cuda(), dp.k, dp.v, dp.tables, lens, wl.scale, workspace=ws)
    torch.cuda.synchronize()
    assert torch.all(buf[:1024] == 7.0) and torch.all(buf[1024 + n:] == 7.0)


# ---- the named workloads at full size, sampled outputs -------------------------------

def _sample_pairs(wl, n, seed):
    rng = np.random.default_rng(seed)
    lens = wl.context_lens
    pick = {int(np.argmax(lens)), int(np.argmin(lens))}
    pick |= set(rng.choice(wl.num_seqs, size=min(n, wl.num_seqs), replace=False).tolist())
    return [(s, int(rng.integers(wl.num_q_heads))) for s in sorted(pick)] + \
           [(int(np.argmax(lens)), h) for h in range(wl.num_q_heads)]


@pytest.mark.parametrize("one_call", [False, True])
@pytest.mark.parametrize("name,nsample", [("qwen2.5-0.5b_gqa", 24), ("llama3-8b_batch256", 24),
                                          ("llama3-8b_long_context", 8),
                                          ("llama3-8b_shared_prefix", 16)])
def test_named_workload_full_size_sampled(name, nsample, one_call):
    # each workload at full size, as append + decode and as the bench's one call (with the
    # shared-prefix workload's 4096 shared tokens through the prefix-sharing kernels)
    wl = W.WORKLOADS[name](device="cuda")
    dp = DevicePools(wl, canary=False)
    hint = int(wl.context_lens.max()) + 1
    if one_call:
        out = dp.run_step_one_call(hint=hint, shared=4096 if name == "llama3-8b_shared_prefix" else 0)
    else:
        out = dp.run_step(hint=hint)
    torch.cuda.synchronize()
    assert int(dp.err.item()) == 0
    pairs = _sample_pairs(wl, nsample, 7)
    want = oracle_contig(wl, pairs)
    got = np.stack([as_f64(out[s, h]) for s, h in pairs])
    assert_close(wl, got, want, name)
    assert torch.isfinite(out.float()).all()


def test_group_boundaries_of_the_partition_merge():
    # 16 partitions fill one merge group; 17 and 33 need a second and third group
    P = pk.PARTITION_TOKENS
    lens = [16 * P, 16 * P + 1, 17 * P, 33 * P + 100, 5]
    wl = W.make_decode_workload("groups", context_lens=np.array(lens) - 1, num_q_heads=8,
                                num_kv_heads=2, head_dim=128, dtype="bf16", seed=77, device="cuda")
    dp = DevicePools(wl, canary=False)
    out = dp.run_step()
    pairs = _all_pairs(wl)
    want = oracle_contig(wl, pairs)
    assert_close(wl, as_f64(out).reshape(len(pairs), 128), want, "merge groups")
    assert int(dp.err.item()) == 0


def test_repeated_calls_on_one_workspace_give_the_same_bits():
    # whatever an earlier call left in the workspace does not leak into the next one
    wl = W.make_decode_workload("reuse", context_lens=[3000, 700, 9000], num_q_heads=32,
                                num_kv_heads=8, head_dim=128, dtype="bf16", seed=9, device="cuda")
    dp = DevicePools(wl, canary=False)
    k_new, v_new, start, cu, lens = dp.step_inputs()
    pk.append_kv(dp.k, dp.v, k_new, v_new, dp.tables, start, cu, err_flag=dp.err)
    ws = pk.decode_workspace(3, 32, 8, 128, wl.max_blocks)
    outs = []
    for _ in range(3):
        out = torch.empty_like(wl.q)
        pk.decode_attention(out, wl.q, dp.k, dp.v, dp.tables, lens, wl.scale, workspace=ws,
                            err_flag=dp.err)
        torch.cuda.synchronize()
        outs.append(out)
        ws.fill_(0x7F)     # garbage for the next call
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    assert int(dp.err.item()) == 0


def test_one_workspace_across_batch_sizes_and_head_dims():
    # a workspace sized for the largest call serves smaller calls of other shapes, in
    # between and after: no call depends on what another left in it
    big = W.make_decode_workload("ws_big", context_lens=[5000, 700, 2600, 3100], num_q_heads=32,
                                 num_kv_heads=8, head_dim=128, dtype="bf16", seed=12, device="cuda")
    small = W.make_decode_workload("ws_small", context_lens=[1500, 3000], num_q_heads=14,
                                   num_kv_heads=2, head_dim=64, dtype="bf16", seed=13, device="cuda")
    ws = pk.decode_workspace(4, 32, 8, 128, big.max_blocks)
    for wl in (big, small, big):
        dp = DevicePools(wl, canary=False)
        k_new, v_new, start, cu, lens = dp.step_inputs()
        pk.append_kv(dp.k, dp.v, k_new, v_new, dp.tables, start, cu, err_flag=dp.err)
        out = torch.empty_like(wl.q)
        assert ws.numel() >= pk.decode_workspace_size(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads,
                                                      wl.head_dim, wl.max_blocks)
        pk.decode_attention(out, wl.q, dp.k, dp.v, dp.tables, lens, wl.scale, workspace=ws,
                            err_flag=dp.err)
        torch.cuda.synchronize()
        pairs = _all_pairs(wl)
        assert_close(wl, as_f64(out).reshape(len(pairs), wl.head_dim), oracle_contig(wl, pairs),
                     f"shared workspace {wl.name}")
        assert int(dp.err.item()) == 0

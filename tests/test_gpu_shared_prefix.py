"""GPU parity of prefix-sharing decode (pa_decode_attention_shared_prefix).

Sequences that share their first positions in the same physical blocks (the
layout refcounted copy-on-write forks leave behind; spindle, "Paging") are
decoded with the prefix read once per kv head.  Results must match the oracle
computed on each sequence's logical rows, for prefixes of whole and partial
partitions, empty suffixes, several query-head groupings and row counts that
leave the last 64-row tile partly empty.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_207_gb300 as pk
from paged_kv_cache_207_gb300 import workloads as W
from _gpu_common import DevicePools, as_f64, assert_close, oracle_contig

pytestmark = pytest.mark.gpu


def _prefix_step(wl, dp, shared, hint=0):
    k_new, v_new, start, cu, lens = dp.step_inputs()
    pk.append_kv(dp.k, dp.v, k_new, v_new, dp.tables, start, cu, err_flag=dp.err)
    out = torch.empty_like(wl.q)
    ws = pk.decode_workspace(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                             wl.max_blocks)
    pk.decode_attention_shared_prefix(out, wl.q, dp.k, dp.v, dp.tables, lens, wl.scale, shared,
                                      workspace=ws, max_context_len_hint=hint, err_flag=dp.err)
    torch.cuda.synchronize()
    return out, lens


@pytest.mark.parametrize("shared,suffixes,hq,hkv,d", [
    (512, [1, 16, 17, 600, 1], 32, 8, 128),
    (1024, [1, 100, 513, 2, 77, 1000, 3], 14, 2, 64),
    (2048, [5, 40], 12, 12, 64),
    (528, [1, 30, 700], 8, 1, 128),
    (4096, [16, 512, 300, 1, 64, 128, 256, 400, 9, 33, 65], 32, 8, 128),
])
def test_shared_prefix_against_oracle(shared, suffixes, hq, hkv, d):
    lens = [shared + n - 1 for n in suffixes]       # context before the step's append
    wl = W.make_decode_workload("prefix", context_lens=lens, num_q_heads=hq, num_kv_heads=hkv,
                                head_dim=d, dtype="bf16", seed=shared + hq,
                                device="cuda", shared_prefix=shared)
    dp = DevicePools(wl)
    out, _ = _prefix_step(wl, dp, shared)
    pairs = [(s, h) for s in range(wl.num_seqs) for h in range(hq)]
    want = oracle_contig(wl, pairs)
    assert_close(wl, as_f64(out).reshape(len(pairs), d), want, f"prefix {shared}")
    assert int(dp.err.item()) == 0
    # and the ordinary path on the same cache agrees within the same tolerance
    ref = dp.decode(torch.from_numpy(np.array(lens, np.int32) + 1).cuda())
    assert_close(wl, as_f64(out), as_f64(ref), "prefix vs ordinary")


@pytest.mark.parametrize("rows_hq", [(8, 32), (64, 32)])
def test_shared_prefix_negative_scale(rows_hq):
    # The prefix partitions run on the tensor cores with |scale| on -q (the sign moved into
    # the query tile): 8 sequences give one 128-row Q tile per prefix CTA, 64 give two.
    S, hq = rows_hq
    suffixes = [1 + 37 * i % 400 for i in range(S)]
    lens = [1024 + n - 1 for n in suffixes]
    wl = W.make_decode_workload("prefix_neg", context_lens=lens, num_q_heads=hq, num_kv_heads=8,
                                head_dim=128, dtype="bf16", seed=77 + S, device="cuda",
                                shared_prefix=1024, scale=-1.0 / np.sqrt(128.0))
    dp = DevicePools(wl)
    out, _ = _prefix_step(wl, dp, 1024)
    pairs = [(s, h) for s in range(wl.num_seqs) for h in range(hq)]
    want = oracle_contig(wl, pairs)
    assert_close(wl, as_f64(out).reshape(len(pairs), 128), want, "prefix, negative scale")
    assert int(dp.err.item()) == 0


def test_short_prefix_falls_back_to_the_ordinary_path_bitwise():
    lens = [300 + n for n in (1, 50, 200)]
    wl = W.make_decode_workload("short", context_lens=lens, num_q_heads=32, num_kv_heads=8,
                                head_dim=128, dtype="bf16", seed=3, device="cuda",
                                shared_prefix=256)
    dp = DevicePools(wl)
    out, lens_t = _prefix_step(wl, dp, 256)
    ref = dp.decode(lens_t)
    assert torch.equal(out, ref)


def test_one_partition_table_falls_back_to_the_ordinary_path_bitwise():
    # a 512-token prefix in a table of 32 blocks: every context is the prefix and fits one
    # partition, no workspace is needed, and the call takes the ordinary path
    wl = W.make_decode_workload("one_part", context_lens=[511, 511, 511], num_q_heads=32,
                                num_kv_heads=8, head_dim=128, dtype="bf16", seed=4,
                                device="cuda", shared_prefix=512)
    assert wl.max_blocks == 32
    assert pk.decode_workspace_size(wl.num_seqs, 32, 8, 128, 32) == 0
    dp = DevicePools(wl)                  # the 512 prefix rows, written once
    lens_t = torch.full((3,), 512, dtype=torch.int32, device="cuda")
    out = torch.empty_like(wl.q)
    pk.decode_attention_shared_prefix(out, wl.q, dp.k, dp.v, dp.tables, lens_t, wl.scale, 512,
                                      err_flag=dp.err)
    ref = dp.decode(lens_t)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert int(dp.err.item()) == 0


def test_broken_prefix_promise_is_flagged():
    # sequence 1's table points one prefix block elsewhere (as after a copy-on-write split),
    # sequence 2's context is shorter than the prefix: both break the caller's promise
    shared = 1024
    lens = [shared + 40, shared + 300, shared + 5]
    wl = W.make_decode_workload("broken", context_lens=lens, num_q_heads=8, num_kv_heads=2,
                                head_dim=128, dtype="bf16", seed=6, device="cuda",
                                shared_prefix=shared, pool_blocks=400)
    dp = DevicePools(wl)
    out, _ = _prefix_step(wl, dp, shared)
    assert int(dp.err.item()) == 0                     # the promise holds: no flag
    tables = dp.tables.clone()
    tables[1, 10] = 399                                 # an unused block of the pool
    k_new, v_new, start, cu, lens_t = dp.step_inputs()
    ws = pk.decode_workspace(wl.num_seqs, 8, 2, 128, wl.max_blocks)
    pk.decode_attention_shared_prefix(out, wl.q, dp.k, dp.v, tables, lens_t, wl.scale, shared,
                                      workspace=ws, err_flag=dp.err)
    torch.cuda.synchronize()
    assert int(dp.err.item()) == pk.DEV_ERR_BAD_PREFIX
    dp.err.zero_()
    short = lens_t.clone()
    short[2] = shared - 3
    pk.decode_attention_shared_prefix(out, wl.q, dp.k, dp.v, dp.tables, short, wl.scale, shared,
                                      workspace=ws, err_flag=dp.err)
    torch.cuda.synchronize()
    assert int(dp.err.item()) == pk.DEV_ERR_BAD_PREFIX


def test_shared_prefix_workload_full_size_sampled():
    wl = W.llama8b_shared_prefix(device="cuda")
    dp = DevicePools(wl, canary=False)
    out, _ = _prefix_step(wl, dp, 4096, hint=int(wl.context_lens.max()) + 1)
    assert int(dp.err.item()) == 0
    rng = np.random.default_rng(5)
    pairs = [(int(s), int(rng.integers(32))) for s in rng.choice(wl.num_seqs, 16, replace=False)]
    pairs += [(0, h) for h in range(32)]
    want = oracle_contig(wl, pairs)
    got = np.stack([as_f64(out[s, h]) for s, h in pairs])
    assert_close(wl, got, want, "shared prefix full size")


def test_shared_prefix_two_q_tiles_per_cta():
    # 120 sequences x 4 query heads per kv head = 480 rows in two groups of 256 (the second
    # group's second Q tile partly empty); with 16 prefix partitions and 8 kv heads there are
    # enough CTAs to hold 256 rows each
    lens = [8192 + n - 1 for n in np.random.default_rng(11).integers(1, 300, 120)]
    wl = W.make_decode_workload("prefix2", context_lens=lens, num_q_heads=32, num_kv_heads=8,
                                head_dim=128, dtype="bf16", seed=12, device="cuda",
                                shared_prefix=8192)
    dp = DevicePools(wl, canary=False)
    out, lens_t = _prefix_step(wl, dp, 8192, hint=int(max(lens)) + 1)
    assert int(dp.err.item()) == 0
    rng = np.random.default_rng(13)
    seqs = sorted(set(rng.choice(120, 10, replace=False).tolist()) | {0, 31, 32, 63, 64, 95, 96, 119})
    pairs = [(s, int(rng.integers(32))) for s in seqs]
    want = oracle_contig(wl, pairs)
    got = np.stack([as_f64(out[s, h]) for s, h in pairs])
    assert_close(wl, got, want, "two Q tiles per CTA")
    ref = dp.decode(lens_t)
    assert_close(wl, as_f64(out), as_f64(ref), "prefix vs ordinary, two Q tiles per CTA")


def test_repeated_shared_prefix_calls_give_the_same_bits():
    lens = [2048 + n - 1 for n in (1, 100, 513, 7, 300, 64)]
    wl = W.make_decode_workload("prefix_rep", context_lens=lens, num_q_heads=32, num_kv_heads=8,
                                head_dim=128, dtype="bf16", seed=21, device="cuda",
                                shared_prefix=2048)
    dp = DevicePools(wl)
    out, lens_t = _prefix_step(wl, dp, 2048)
    ws = pk.decode_workspace(wl.num_seqs, 32, 8, 128, wl.max_blocks)
    for _ in range(20):
        again = torch.full_like(out, float("nan"))
        pk.decode_attention_shared_prefix(again, wl.q, dp.k, dp.v, dp.tables, lens_t, wl.scale, 2048,
                                          workspace=ws, err_flag=dp.err)
        torch.cuda.synchronize()
        assert torch.equal(again, out)
    assert int(dp.err.item()) == 0


def test_shared_prefix_two_q_tiles_per_cta_head_dim_64():
    # 300 sequences x 1 query head per kv head = 300 rows (the second group's tile b partly
    # empty), 12 kv heads, 8 prefix partitions: 192 CTAs of 256 rows at head_dim 64
    lens = [4096 + n - 1 for n in np.random.default_rng(17).integers(1, 200, 300)]
    wl = W.make_decode_workload("prefix64", context_lens=lens, num_q_heads=12, num_kv_heads=12,
                                head_dim=64, dtype="bf16", seed=18, device="cuda",
                                shared_prefix=4096)
    dp = DevicePools(wl, canary=False)
    out, lens_t = _prefix_step(wl, dp, 4096, hint=int(max(lens)) + 1)
    assert int(dp.err.item()) == 0
    rng = np.random.default_rng(19)
    seqs = sorted(set(rng.choice(300, 10, replace=False).tolist()) | {0, 127, 128, 255, 256, 299})
    pairs = [(s, int(rng.integers(12))) for s in seqs]
    want = oracle_contig(wl, pairs)
    got = np.stack([as_f64(out[s, h]) for s, h in pairs])
    assert_close(wl, got, want, "two Q tiles per CTA, head_dim 64")
    ref = dp.decode(lens_t)
    assert_close(wl, as_f64(out), as_f64(ref), "prefix vs ordinary, head_dim 64")


def test_shared_prefix_step_loop_full_size_stays_exact():
    # The step loop of a serving engine at full size: append then shared-prefix decode,
    # back to back with no synchronisation, cycling over four copies of the pools.  Rare
    # orderings between the tensor-core kernel's warps show up here as a wait that gives up
    # (the TIMEOUT bit) or as differing bits; every call must give the first call's bits.
    wl = W.llama8b_shared_prefix(device="cuda")
    dp = DevicePools(wl, canary=False)
    k_new, v_new, start, cu, lens = dp.step_inputs()
    pools = [(dp.k, dp.v)] + [(dp.k.clone(), dp.v.clone()) for _ in range(3)]
    ws = pk.decode_workspace(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                             wl.max_blocks)
    hint = int(lens.max().item())
    outs = [torch.empty_like(wl.q) for _ in range(4)]
    first = None
    for rep in range(6):
        for i in range(20):
            kp, vp = pools[i % 4]
            pk.append_kv(kp, vp, k_new, v_new, dp.tables, start, cu, err_flag=dp.err)
            pk.decode_attention_shared_prefix(outs[i % 4], wl.q, kp, vp, dp.tables, lens, wl.scale,
                                              4096, workspace=ws, max_context_len_hint=hint,
                                              err_flag=dp.err)
        torch.cuda.synchronize()
        assert int(dp.err.item()) == 0, (rep, int(dp.err.item()))
        if first is None:
            first = outs[0].clone()
        for o in outs:
            assert torch.equal(o, first), rep
    pairs = [(0, h) for h in range(32)] + [(wl.num_seqs - 1, 7)]
    want = oracle_contig(wl, pairs)
    got = np.stack([as_f64(first[s, h]) for s, h in pairs])
    assert_close(wl, got, want, "shared prefix step loop")

"""Decode with append in one call (pa_append_decode_attention) against the two calls it
replaces -- pa_append_kv of one row per sequence at position context_len - 1, then
pa_decode_attention -- bit for bit (pools and outputs), and against the oracle
(spindle, "Paging": a decode step appends the token, then attends over the cache;
"Two bugs worth recording": the position is explicit).

The lengths put the new token at the edges of the layout: the only token of a
sequence, the first and last slot of a block, the first token of a new split-KV
partition, the last token of a full partition.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_207_gb300 as pk
from paged_kv_cache_207_gb300 import workloads as W
from _gpu_common import DevicePools, as_f64, assert_close, oracle_contig

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_207_gb300 import build
    build.build()
    pk.lib()


def _edge_lengths(part_tokens):
    """Context lengths BEFORE the step (the new token goes to this position)."""
    P = part_tokens
    return [0, 15, 16, 17, 31, P - 1, P, P + 1, 2 * P - 1, 2 * P, 3 * P + 200, 4 * P + 16, 37]


def _pair(wl):
    """Two copies of the workload's pools (context filled) and the step's inputs."""
    a = DevicePools(wl)
    b_k, b_v = a.k.clone(), a.v.clone()
    return a, b_k, b_v, a.step_inputs()


def _bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


def _all_pairs(wl):
    return [(s, h) for s in range(wl.num_seqs) for h in range(wl.num_q_heads)]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (14, 2, 64), (8, 1, 128), (12, 12, 64)])
def test_append_decode_equals_append_then_decode(dtype, hq, hkv, d):
    lens = _edge_lengths(pk.partition_tokens(d))
    wl = W.make_decode_workload("append_decode", context_lens=lens, num_q_heads=hq,
                                num_kv_heads=hkv, head_dim=d, dtype=dtype, seed=hq * 7 + d,
                                device="cuda")
    a, b_k, b_v, (k_new, v_new, start, cu, lens_after) = _pair(wl)
    ws = pk.decode_workspace(wl.num_seqs, hq, hkv, d, wl.max_blocks)
    # the two calls
    pk.append_kv(a.k, a.v, k_new, v_new, a.tables, start, cu, err_flag=a.err)
    want = torch.empty_like(wl.q)
    pk.decode_attention(want, wl.q, a.k, a.v, a.tables, lens_after, wl.scale, workspace=ws,
                        err_flag=a.err)
    # the one call, on the other copy
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = torch.empty_like(wl.q)
    pk.append_decode_attention(got, wl.q, b_k, b_v, k_new, v_new, a.tables, lens_after, wl.scale,
                               workspace=ws, err_flag=err)
    torch.cuda.synchronize()
    assert int(a.err.item()) == 0 and int(err.item()) == 0
    assert torch.equal(_bits(a.k), _bits(b_k)) and torch.equal(_bits(a.v), _bits(b_v))
    assert torch.equal(_bits(want), _bits(got))
    pairs = _all_pairs(wl)
    assert_close(wl, as_f64(got).reshape(len(pairs), d),
                 oracle_contig(wl, pairs, lens_after=lens_after.cpu().numpy()),
                 f"append+decode {dtype} {hq}/{hkv}x{d}")


def test_append_decode_twenty_steps_in_a_row():
    # twenty steps in a row, each appending one token per sequence and attending over it
    # (positions start - 19 .. start, inside the blocks each table holds): the one-call
    # pools and outputs stay equal to the two-call ones at every step
    wl = W.make_decode_workload("append_decode_steps", context_lens=[500, 20, 1023, 2040, 60],
                                num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16",
                                seed=5, device="cuda")
    a, b_k, b_v, (k_new, v_new, start, cu, lens_after) = _pair(wl)
    ws = pk.decode_workspace(wl.num_seqs, 32, 8, 128, wl.max_blocks)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(5)
    for step in range(20):
        kn = torch.randn(k_new.shape, generator=gen, device="cuda").to(k_new.dtype)
        vn = torch.randn(v_new.shape, generator=gen, device="cuda").to(v_new.dtype)
        pos = start - 19 + step
        pk.append_kv(a.k, a.v, kn, vn, a.tables, pos, cu, err_flag=a.err)
        want = torch.empty_like(wl.q)
        pk.decode_attention(want, wl.q, a.k, a.v, a.tables, pos + 1, wl.scale, workspace=ws,
                            err_flag=a.err)
        got = torch.empty_like(wl.q)
        pk.append_decode_attention(got, wl.q, b_k, b_v, kn, vn, a.tables, pos + 1, wl.scale,
                                   workspace=ws, err_flag=err)
        torch.cuda.synchronize()
        assert torch.equal(_bits(want), _bits(got)), f"step {step}"
    assert int(a.err.item()) == 0 and int(err.item()) == 0
    assert torch.equal(_bits(a.k), _bits(b_k)) and torch.equal(_bits(a.v), _bits(b_v))


def test_append_decode_flags_like_the_two_calls():
    # a table entry out of range at the new position, a length past the table, and a grid
    # hint shorter than a context: the same flags, pools and outputs as the two calls
    wl = W.make_decode_workload("append_decode_err", context_lens=[40, 700, 100, 1500],
                                num_q_heads=8, num_kv_heads=2, head_dim=128, dtype="bf16",
                                seed=8, device="cuda")
    a, b_k, b_v, (k_new, v_new, start, cu, lens_after) = _pair(wl)
    tables = a.tables.clone()
    tables[0, 40 // 16] = wl.num_blocks + 3              # sequence 0's new position: bad block
    lens_bad = lens_after.clone()
    lens_bad[2] = wl.max_blocks * 16 + 5                 # sequence 2: past its table
    ws = pk.decode_workspace(wl.num_seqs, 8, 2, 128, wl.max_blocks)
    for hint in (0, 600):                                # 600: one partition; 1500 needs three
        a2_k, a2_v = a.k.clone(), a.v.clone()
        b2_k, b2_v = b_k.clone(), b_v.clone()
        e1 = torch.zeros(1, dtype=torch.int32, device="cuda")
        e2 = torch.zeros(1, dtype=torch.int32, device="cuda")
        pk.append_kv(a2_k, a2_v, k_new, v_new, tables, lens_bad - 1, cu, err_flag=e1)
        want = torch.empty_like(wl.q)
        pk.decode_attention(want, wl.q, a2_k, a2_v, tables, lens_bad, wl.scale, workspace=ws,
                            max_context_len_hint=hint, err_flag=e1)
        got = torch.empty_like(wl.q)
        pk.append_decode_attention(got, wl.q, b2_k, b2_v, k_new, v_new, tables, lens_bad, wl.scale,
                                   workspace=ws, max_context_len_hint=hint, err_flag=e2)
        torch.cuda.synchronize()
        f = int(e1.item())
        assert f & pk.DEV_ERR_BAD_BLOCK and f & pk.DEV_ERR_BAD_POS
        assert bool(f & pk.DEV_ERR_HINT) == (hint > 0)
        assert int(e2.item()) == f
        assert torch.equal(_bits(a2_k), _bits(b2_k)) and torch.equal(_bits(a2_v), _bits(b2_v))
        # every row, flagged or not, is the same bits (an unreadable block is skipped on
        # both sides)
        assert torch.equal(_bits(want), _bits(got))


def test_append_decode_writes_nothing_while_timeout_is_set():
    wl = W.make_decode_workload("append_decode_abort", context_lens=[30, 900, 2000],
                                num_q_heads=8, num_kv_heads=2, head_dim=128, dtype="bf16",
                                seed=9, device="cuda")
    a, _, _, (k_new, v_new, start, cu, lens_after) = _pair(wl)
    k0, v0 = a.k.clone(), a.v.clone()
    ws = pk.decode_workspace(wl.num_seqs, 8, 2, 128, wl.max_blocks)
    err = torch.full((1,), pk.DEV_ERR_TIMEOUT, dtype=torch.int32, device="cuda")
    out = torch.empty_like(wl.q)
    out.view(torch.int16).fill_(0x5A5A)
    pk.append_decode_attention(out, wl.q, a.k, a.v, k_new, v_new, a.tables, lens_after, wl.scale,
                               workspace=ws, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == pk.DEV_ERR_TIMEOUT
    assert bool((out.view(torch.int16) == 0x5A5A).all().item())
    assert torch.equal(_bits(a.k), _bits(k0)) and torch.equal(_bits(a.v), _bits(v0))


# ---- with a shared prefix (pa_append_decode_attention_shared_prefix) ---------------

@pytest.mark.parametrize("shared,suffixes,hq,hkv,d", [
    (512, [1, 16, 17, 600, 1], 32, 8, 128),           # one whole shared partition
    (1024, [1, 100, 513, 2, 77, 1000, 3], 14, 2, 64),  # head_dim 64, 1024-token partitions
    (528, [1, 30, 700], 8, 1, 128),                    # a prefix past a partition edge
    (4096, [16, 512, 300, 1, 64, 128, 256, 400, 9, 33, 65], 32, 8, 128),
    (256, [1, 40, 300], 8, 2, 128),                    # shorter than a partition: fallback
])
def test_append_decode_shared_prefix_equals_the_two_calls(shared, suffixes, hq, hkv, d):
    lens = [shared + n - 1 for n in suffixes]          # the new row goes past the prefix
    wl = W.make_decode_workload("append_decode_prefix", context_lens=lens, num_q_heads=hq,
                                num_kv_heads=hkv, head_dim=d, dtype="bf16", seed=shared + hq,
                                device="cuda", shared_prefix=shared)
    a, b_k, b_v, (k_new, v_new, start, cu, lens_after) = _pair(wl)
    ws = pk.decode_workspace(wl.num_seqs, hq, hkv, d, wl.max_blocks)
    pk.append_kv(a.k, a.v, k_new, v_new, a.tables, start, cu, err_flag=a.err)
    want = torch.empty_like(wl.q)
    pk.decode_attention_shared_prefix(want, wl.q, a.k, a.v, a.tables, lens_after, wl.scale, shared,
                                      workspace=ws, err_flag=a.err)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = torch.empty_like(wl.q)
    pk.append_decode_attention_shared_prefix(got, wl.q, b_k, b_v, k_new, v_new, a.tables,
                                             lens_after, wl.scale, shared, workspace=ws,
                                             err_flag=err)
    torch.cuda.synchronize()
    assert int(a.err.item()) == 0 and int(err.item()) == 0
    assert torch.equal(_bits(a.k), _bits(b_k)) and torch.equal(_bits(a.v), _bits(b_v))
    assert torch.equal(_bits(want), _bits(got))
    pairs = _all_pairs(wl)
    assert_close(wl, as_f64(got).reshape(len(pairs), d),
                 oracle_contig(wl, pairs, lens_after=lens_after.cpu().numpy()),
                 f"append+prefix {shared}")


@pytest.mark.parametrize("shared", [1024, 256])
def test_append_decode_shared_prefix_refuses_a_row_inside_the_prefix(shared):
    # sequence 1's context ends one short of the prefix, so its new row would land on the
    # prefix's last position, in a block every sequence reads: it is not written, and the
    # call says so (1024: the shared-prefix kernels; 256: the fallback to the plain path)
    lens = [shared + 40, shared - 1, shared + 600]     # before the step
    wl = W.make_decode_workload("append_decode_prefix_bad", context_lens=lens, num_q_heads=8,
                                num_kv_heads=2, head_dim=128, dtype="bf16", seed=shared,
                                device="cuda", shared_prefix=shared)
    a, _, _, (k_new, v_new, start, cu, lens_after) = _pair(wl)
    k0, v0 = a.k.clone(), a.v.clone()
    ws = pk.decode_workspace(wl.num_seqs, 8, 2, 128, wl.max_blocks)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(wl.q)
    pk.append_decode_attention_shared_prefix(out, wl.q, a.k, a.v, k_new, v_new, a.tables,
                                             lens_after, wl.scale, shared, workspace=ws,
                                             err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pk.DEV_ERR_BAD_PREFIX
    # the shared blocks (sequence 0's first shared / 16 table entries) are unchanged
    pre = a.tables[0, :shared // 16].long()
    assert torch.equal(_bits(a.k[pre]), _bits(k0[pre])) and torch.equal(_bits(a.v[pre]), _bits(v0[pre]))


# ---- FP8 cache (pa_append_decode_attention_fp8) ---------------------------------------

def _fp8_pools(wl):
    shape = pk.fp8_pool_shape(wl.num_blocks, wl.num_kv_heads, wl.head_dim)
    kp = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    vp = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    tables = torch.from_numpy(wl.block_tables).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if wl.fill:
        seqs = [f[0] for f in wl.fill]
        ns = [f[3] for f in wl.fill]
        first, end = wl.fill[0][2], wl.fill[-1][2] + wl.fill[-1][3]
        pk.append_kv_fp8(kp, vp, wl.k_rows[first:end].contiguous(), wl.v_rows[first:end].contiguous(),
                         tables[torch.tensor(seqs, device="cuda")].contiguous(),
                         torch.tensor([f[1] for f in wl.fill], dtype=torch.int32, device="cuda"),
                         torch.tensor(np.concatenate([[0], np.cumsum(ns)]), dtype=torch.int32,
                                      device="cuda"), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return kp, vp, tables


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (14, 2, 64), (8, 1, 128)])
def test_append_decode_fp8_equals_the_two_calls(hq, hkv, d):
    P = 1024                                            # FP8 partition tokens
    lens = [0, 15, 16, 17, P - 1, P, P + 1, 2 * P - 1, 2 * P, 3 * P - 50, 37]
    wl = W.make_decode_workload("append_decode_fp8", context_lens=lens, num_q_heads=hq,
                                num_kv_heads=hkv, head_dim=d, dtype="bf16", seed=hq + d,
                                device="cuda", big_key_frac=0.01)
    ka, va, tables = _fp8_pools(wl)
    kb, vb = ka.clone(), va.clone()
    rows = torch.from_numpy(wl.new_rows).cuda()
    k_new, v_new = wl.k_rows[rows].contiguous(), wl.v_rows[rows].contiguous()
    start = torch.from_numpy(wl.context_lens.astype(np.int32)).cuda()
    cu = torch.arange(wl.num_seqs + 1, dtype=torch.int32, device="cuda")
    ws = pk.decode_workspace(wl.num_seqs, hq, hkv, d, wl.max_blocks)
    e1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    e2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    pk.append_kv_fp8(ka, va, k_new, v_new, tables, start, cu, err_flag=e1)
    want = torch.empty_like(wl.q)
    pk.decode_attention_fp8(want, wl.q, ka, va, tables, start + 1, wl.scale, workspace=ws,
                            err_flag=e1)
    got = torch.empty_like(wl.q)
    pk.append_decode_attention_fp8(got, wl.q, kb, vb, k_new, v_new, tables, start + 1, wl.scale,
                                   workspace=ws, err_flag=e2)
    torch.cuda.synchronize()
    assert int(e1.item()) == 0 and int(e2.item()) == 0
    assert torch.equal(ka, kb) and torch.equal(va, vb)
    assert torch.equal(_bits(want), _bits(got))
    assert bool(torch.isfinite(got.float()).all())

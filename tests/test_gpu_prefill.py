"""GPU parity of chunked prefill attention (pa_prefill_attention).

A chunk of n tokens at explicit positions start .. start+n-1, appended to the
cache first, attends causally: the token at position p sees positions 0 .. p
of its own sequence.  Each output row must match the oracle computed on that
sequence's logical rows 0 .. p -- the same definition as decode with context
length p + 1 (spindle, "Two bugs worth recording": positions are explicit).
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_207_gb300 as pk
from paged_kv_cache_207_gb300 import workloads as W
from _gpu_common import BF16_ATOL, DevicePools
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def _prefill_case(chunks, hq, hkv, d, seed, max_chunk=None, scale=None):
    """chunks: list of (start, n).  Returns (workload, pools, q, out, starts, ns)."""
    totals = [s + n for s, n in chunks]
    wl = W.make_decode_workload("prefill", context_lens=np.array(totals) - 1, num_q_heads=hq,
                                num_kv_heads=hkv, head_dim=d, dtype="bf16", seed=seed,
                                device="cuda")
    dp = DevicePools(wl)                                   # positions 0 .. total-2
    k_new, v_new, start, cu, _ = dp.step_inputs()          # the last position
    pk.append_kv(dp.k, dp.v, k_new, v_new, dp.tables, start, cu, err_flag=dp.err)
    ns = [n for _, n in chunks]
    starts = [s for s, _ in chunks]
    g = torch.Generator(device="cuda").manual_seed(seed + 1)
    q = torch.randn(sum(ns), hq, d, generator=g, device="cuda").to(torch.bfloat16)
    out = torch.full_like(q, float("nan"))
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(ns)]), dtype=torch.int32, device="cuda")
    pk.prefill_attention(out, q, dp.k, dp.v, dp.tables,
                         torch.tensor(starts, dtype=torch.int32, device="cuda"), cu_q,
                         wl.scale if scale is None else scale,
                         max_chunk=max(ns) if max_chunk is None else max_chunk, err_flag=dp.err)
    torch.cuda.synchronize()
    return wl, dp, q, out, starts, ns


def _check(wl, q, out, starts, ns, rows_per_seq=None, only=None, scale=None):
    kr, vr = wl.k_rows.cpu(), wl.v_rows.cpu()
    qc, oc = q.cpu(), out.float().cpu().double().numpy()
    G = wl.num_q_heads // wl.num_kv_heads
    rng = np.random.default_rng(0)
    worst = 0.0
    base = 0
    for s, (st, n) in enumerate(zip(starts, ns)):
        if only is not None and s not in only:
            base += n
            continue
        logical = torch.from_numpy(wl.logical_rows(s))
        idx = range(n) if rows_per_seq is None else sorted(set(rng.integers(0, n, rows_per_seq).tolist()) | {0, n - 1})
        for i in idx:
            p = st + i
            K = kr[logical[:p + 1]].contiguous()
            V = vr[logical[:p + 1]].contiguous()
            for h in range(wl.num_q_heads):
                want = orc.decode_contig(qc[base + i, h], K, V, h // G, num_kv_heads=wl.num_kv_heads,
                                         head_dim=wl.head_dim, scale=wl.scale if scale is None else scale,
                                         dtype=orc.BF16)
                worst = max(worst, float(np.abs(oc[base + i, h] - want).max()))
        base += n
    assert worst <= BF16_ATOL, worst


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (14, 2, 64), (12, 12, 64), (8, 1, 128)])
def test_prefill_chunks_against_oracle(hq, hkv, d):
    chunks = [(0, 100), (300, 64), (513, 1), (0, 1), (1000, 77), (16, 16), (40, 130)]
    wl, dp, q, out, starts, ns = _prefill_case(chunks, hq, hkv, d, seed=hq + d)
    assert int(dp.err.item()) == 0
    assert torch.isfinite(out.float()).all()
    _check(wl, q, out, starts, ns)


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (14, 2, 64)])
def test_prefill_items_beyond_the_schedule_lists(hq, hkv, d):
    # A host bound on the chunk length far above the chunks (4096 against 1-9 tokens) gives
    # 256 sequences x 57-114 query tiles x the kv heads as work items, and as many (sequence,
    # query tile) groups: more than a CTA's shared-memory schedule holds, so every CTA walks
    # the items by a stride over their natural order instead of a sorted list.  Most items are
    # empty; every row must still match the oracle and nothing may be flagged.
    rng = np.random.default_rng(31)
    chunks = [(int(a), int(b)) for a, b in zip(rng.integers(0, 300, 256), rng.integers(1, 10, 256))]
    wl, dp, q, out, starts, ns = _prefill_case(chunks, hq, hkv, d, seed=31, max_chunk=4096)
    assert int(dp.err.item()) == 0
    assert torch.isfinite(out.float()).all()
    _check(wl, q, out, starts, ns, only=set(range(0, 256, 4)) | {255})


@pytest.mark.parametrize("hq,hkv,d,sign", [(32, 8, 128, -1.0), (14, 2, 64, -1.0), (32, 8, 128, 0.0)])
def test_prefill_negative_and_zero_scale(hq, hkv, d, sign):
    # A negative scale goes to the tensor cores as |scale| on -q (the sign flipped in the
    # query tile); a zero scale weighs every visible key alike (each row: the mean of V).
    chunks = [(0, 70), (300, 130), (17, 9)]
    scale = sign / float(np.sqrt(d))
    wl, dp, q, out, starts, ns = _prefill_case(chunks, hq, hkv, d, seed=5, scale=scale)
    assert int(dp.err.item()) == 0
    assert torch.isfinite(out.float()).all()
    _check(wl, q, out, starts, ns, scale=scale)


def test_prefill_last_row_equals_decode_at_that_position():
    chunks = [(200, 50), (0, 33), (777, 8)]
    wl, dp, q, out, starts, ns = _prefill_case(chunks, 32, 8, 128, seed=9)
    base = 0
    for s, (st, n) in enumerate(zip(starts, ns)):
        qd = q[base + n - 1:base + n].contiguous()
        dec = torch.empty_like(qd)
        ws = pk.decode_workspace(1, 32, 8, 128, wl.max_blocks)
        pk.decode_attention(dec, qd, dp.k, dp.v, dp.tables[s:s + 1].contiguous(),
                            torch.tensor([st + n], dtype=torch.int32, device="cuda"), wl.scale,
                            workspace=ws)
        torch.cuda.synchronize()
        diff = (dec.float() - out[base + n - 1:base + n].float()).abs().max().item()
        assert diff <= BF16_ATOL, diff
        base += n


def test_prefill_long_chunks_sampled():
    chunks = [(0, 2048), (3000, 512), (100, 1500)]
    wl, dp, q, out, starts, ns = _prefill_case(chunks, 32, 8, 128, seed=21)
    assert int(dp.err.item()) == 0
    _check(wl, q, out, starts, ns, rows_per_seq=12)


def test_twelve_layers_prefill_at_the_same_explicit_start():
    # spindle, "Two bugs worth recording": with positions inferred from a length advanced
    # once per step, prefill at layer 0 saw a context of zero.  Here every layer appends
    # its chunk at the same explicit start and attends with explicit positions.
    for layer in range(12):
        wl, dp, q, out, starts, ns = _prefill_case([(64, 32), (0, 20)], 12, 12, 64, seed=300 + layer)
        _check(wl, q, out, starts, ns)


def _prefill_with(chunks, hq, hkv, d, seed, edit):
    """Append as _prefill_case does, then run the prefill on inputs changed by `edit`."""
    totals = [s + n for s, n in chunks]
    wl = W.make_decode_workload("prefill_err", context_lens=np.array(totals) - 1, num_q_heads=hq,
                                num_kv_heads=hkv, head_dim=d, dtype="bf16", seed=seed,
                                device="cuda")
    dp = DevicePools(wl)
    k_new, v_new, start, cu, _ = dp.step_inputs()
    pk.append_kv(dp.k, dp.v, k_new, v_new, dp.tables, start, cu, err_flag=dp.err)
    torch.cuda.synchronize()
    assert int(dp.err.item()) == 0
    ns = [n for _, n in chunks]
    starts = [s for s, _ in chunks]
    g = torch.Generator(device="cuda").manual_seed(seed + 1)
    q = torch.randn(sum(ns), hq, d, generator=g, device="cuda").to(torch.bfloat16)
    out = torch.zeros_like(q)
    tables = dp.tables.clone()
    st = torch.tensor(starts, dtype=torch.int32, device="cuda")
    edit(wl, tables, st)
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(ns)]), dtype=torch.int32, device="cuda")
    pk.prefill_attention(out, q, dp.k, dp.v, tables, st, cu_q, wl.scale, max_chunk=max(ns),
                         err_flag=dp.err)
    torch.cuda.synchronize()
    return wl, dp, q, out, starts, ns


def test_prefill_block_outside_the_pool_is_flagged_and_others_are_exact():
    # sequence 1's first block points past the pool: its tiles are skipped and flagged, the
    # barrier accounting still completes (no timeout bit), other sequences are unaffected
    def edit(wl, tables, st):
        tables[1, 0] = wl.num_blocks
    wl, dp, q, out, starts, ns = _prefill_with([(100, 64), (300, 40), (0, 90)], 32, 8, 128, 41, edit)
    assert int(dp.err.item()) == pk.DEV_ERR_BAD_BLOCK
    _check(wl, q, out, starts, ns, only={0, 2})


def test_prefill_negative_start_is_flagged_and_others_are_exact():
    def edit(wl, tables, st):
        st[0] = -1
    wl, dp, q, out, starts, ns = _prefill_with([(50, 30), (200, 70)], 14, 2, 64, 43, edit)
    assert int(dp.err.item()) == pk.DEV_ERR_BAD_POS
    _check(wl, q, out, starts, ns, only={1})


def test_repeated_prefill_calls_give_the_same_bits():
    # the warp roles of the kernel hand tiles to each other through barriers; any ordering
    # slip would show as run-to-run differences, so repeat the call on unchanged inputs
    chunks = [(0, 300), (1000, 200), (37, 5), (2500, 513)]
    wl, dp, q, out, starts, ns = _prefill_case(chunks, 32, 8, 128, seed=77)
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(ns)]), dtype=torch.int32, device="cuda")
    st = torch.tensor(starts, dtype=torch.int32, device="cuda")
    for _ in range(20):
        again = torch.full_like(out, float("nan"))
        pk.prefill_attention(again, q, dp.k, dp.v, dp.tables, st, cu_q, wl.scale,
                             max_chunk=max(ns), err_flag=dp.err)
        torch.cuda.synchronize()
        assert torch.equal(again, out)
    assert int(dp.err.item()) == 0


def test_prefill_step_loop_full_size_stays_exact():
    # The prefill workload of the benchmark (16 sequences, 512-token chunks at starts up to
    # 3584), run as a step loop: append the chunk, then prefill, back to back with no
    # synchronisation, alternating two copies of the pools.  A wait that gives up (TIMEOUT)
    # or an ordering slip between the kernel's warp roles would show as a flag or as bits
    # that differ from the first step's.
    rng = np.random.default_rng(213)
    S, n = 16, 512
    starts = rng.integers(0, 3585, size=S)
    wl = W.make_decode_workload("prefill_loop", context_lens=starts + n - 1, num_q_heads=32,
                                num_kv_heads=8, head_dim=128, dtype="bf16", seed=213,
                                device="cuda")
    shape = pk.pool_shape(wl.num_blocks, 8, 128, torch.bfloat16)
    kp = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    tables = torch.from_numpy(wl.block_tables).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rows = [torch.from_numpy(wl.logical_rows(s)) for s in range(S)]
    ctx = torch.cat([r[:int(st)] for r, st in zip(rows, starts)]).cuda()
    chunk = torch.cat([r[int(st):int(st) + n] for r, st in zip(rows, starts)]).cuda()
    cu_ctx = torch.tensor(np.concatenate([[0], np.cumsum(starts)]), dtype=torch.int32, device="cuda")
    pk.append_kv(kp, vp, wl.k_rows[ctx].contiguous(), wl.v_rows[ctx].contiguous(), tables,
                 torch.zeros(S, dtype=torch.int32, device="cuda"), cu_ctx, err_flag=err)
    k_chunk, v_chunk = wl.k_rows[chunk].contiguous(), wl.v_rows[chunk].contiguous()
    pools = [(kp, vp), (kp.clone(), vp.clone())]
    g = torch.Generator(device="cuda").manual_seed(7)
    q = torch.randn(S * n, 32, 128, generator=g, device="cuda").to(torch.bfloat16)
    start_t = torch.from_numpy(starts.astype(np.int32)).cuda()
    cu_q = torch.arange(0, S * n + 1, n, dtype=torch.int32, device="cuda")
    outs = [torch.empty_like(q) for _ in range(2)]
    first = None
    for rep in range(4):
        for i in range(10):
            kpp, vpp = pools[i % 2]
            pk.append_kv(kpp, vpp, k_chunk, v_chunk, tables, start_t, cu_q, err_flag=err)
            pk.prefill_attention(outs[i % 2], q, kpp, vpp, tables, start_t, cu_q, wl.scale,
                                 max_chunk=n, err_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, (rep, int(err.item()))
        if first is None:
            first = outs[0].clone()
        assert torch.equal(outs[0], first) and torch.equal(outs[1], first), rep
    # one sampled row per sequence against the oracle (the full-size parity lives elsewhere)
    s = int(np.argmax(starts))
    base = s * n
    p = int(starts[s]) + n - 1
    K = wl.k_rows[rows[s][:p + 1].cuda()].cpu().contiguous()
    V = wl.v_rows[rows[s][:p + 1].cuda()].cpu().contiguous()
    qc = q.cpu()
    for h in (0, 13, 31):
        want = orc.decode_contig(qc[base + n - 1, h], K, V, h // 4, num_kv_heads=8, head_dim=128,
                                 scale=wl.scale, dtype=orc.BF16)
        got = first[base + n - 1, h].float().cpu().double().numpy()
        assert np.abs(got - want).max() <= BF16_ATOL

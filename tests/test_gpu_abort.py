"""A cache that gave up must fail visibly (spindle, "Two bugs worth recording": a wrong
cache produces fluent wrong output, so a failure has to be seen, not papered over).

When a bulk-copy wait runs past its 200 ms bound, the kernel ORs PA_DEV_ERR_TIMEOUT
into the caller's error flag.  While that bit is set, every later decode, prefill and
partition-merge kernel that shares the flag returns without writing its output, so a
broken pipeline cannot keep the GPU busy or overwrite results.  Clearing the bit
resumes normal work.

The failure is made on the host: the test writes the TIMEOUT bit into the flag before
the call (no wait is made to run out on the GPU).  It checks that the output's canary
fill is untouched, that the flag still reads TIMEOUT, and that after clearing the bit
the same call gives the same bits as a clean run.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_207_gb300 as pk
from paged_kv_cache_207_gb300 import workloads as W
from _gpu_common import DevicePools

pytestmark = pytest.mark.gpu

TIMEOUT = pk._native.DEV_ERR_TIMEOUT
CANARY = 0x5A5A          # a bf16 bit pattern (about 1.5e16) no output here can take


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_207_gb300 import build
    build.build()
    pk.lib()


def _canary_like(t):
    out = torch.empty_like(t)
    out.view(torch.int16).fill_(CANARY)
    return out


def _is_canary(t):
    return bool((t.view(torch.int16) == CANARY).all().item())


def _aborted_then_resumed(run, like, err):
    """run(out) enqueues the call writing `out`; returns (clean, resumed) outputs after
    checking the aborted call left its output and the flag as they were."""
    err.zero_()
    clean = _canary_like(like)
    run(clean)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert not _is_canary(clean)

    err.fill_(TIMEOUT)
    out = _canary_like(like)
    run(out)
    torch.cuda.synchronize()
    assert _is_canary(out), "an aborted call wrote its output"
    assert int(err.item()) == TIMEOUT

    err.zero_()
    out2 = _canary_like(like)
    run(out2)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return clean, out2


def _decode_case():
    # one-partition sequences (written by the main kernel) and multi-partition ones
    # (written by the partition merge)
    wl = W.make_decode_workload("abort", context_lens=[16, 600, 2000, 40, 1500], num_q_heads=8,
                                num_kv_heads=2, head_dim=128, dtype="bf16", seed=71,
                                device="cuda")
    dp = DevicePools(wl)
    k_new, v_new, start, cu, lens = dp.step_inputs()
    pk.append_kv(dp.k, dp.v, k_new, v_new, dp.tables, start, cu, err_flag=dp.err)
    torch.cuda.synchronize()
    assert int(dp.err.item()) == 0
    return wl, dp, lens


def test_decode_returns_without_writing_while_timeout_is_set():
    wl, dp, lens = _decode_case()
    ws = pk.decode_workspace(wl.num_seqs, 8, 2, 128, wl.max_blocks)

    def run(out):
        pk.decode_attention(out, wl.q, dp.k, dp.v, dp.tables, lens, wl.scale, workspace=ws,
                            err_flag=dp.err)
    clean, resumed = _aborted_then_resumed(run, wl.q, dp.err)
    assert torch.equal(clean.view(torch.int16), resumed.view(torch.int16))


def test_shared_prefix_decode_returns_without_writing_while_timeout_is_set():
    wl = W.make_decode_workload("abort_prefix", context_lens=np.array([1100, 1030, 1700]) - 1,
                                num_q_heads=8, num_kv_heads=2, head_dim=128, dtype="bf16",
                                seed=72, device="cuda", shared_prefix=1024)
    dp = DevicePools(wl)
    k_new, v_new, start, cu, lens = dp.step_inputs()
    pk.append_kv(dp.k, dp.v, k_new, v_new, dp.tables, start, cu, err_flag=dp.err)
    ws = pk.decode_workspace(wl.num_seqs, 8, 2, 128, wl.max_blocks)

    def run(out):
        pk.decode_attention_shared_prefix(out, wl.q, dp.k, dp.v, dp.tables, lens, wl.scale, 1024,
                                          workspace=ws, err_flag=dp.err)
    clean, resumed = _aborted_then_resumed(run, wl.q, dp.err)
    assert torch.equal(clean.view(torch.int16), resumed.view(torch.int16))


def test_fp8_decode_returns_without_writing_while_timeout_is_set():
    wl = W.make_decode_workload("abort_fp8", context_lens=[16, 1500, 3000], num_q_heads=8,
                                num_kv_heads=2, head_dim=128, dtype="bf16", seed=73, device="cuda")
    shape = pk.fp8_pool_shape(wl.num_blocks, 2, 128)
    kp = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    vp = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    tables = torch.from_numpy(wl.block_tables).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seqs = [f[0] for f in wl.fill]
    ns = [f[3] for f in wl.fill]
    pk.append_kv_fp8(kp, vp, wl.k_rows[:sum(ns)].contiguous(), wl.v_rows[:sum(ns)].contiguous(),
                     tables[torch.tensor(seqs, device="cuda")].contiguous(),
                     torch.tensor([f[1] for f in wl.fill], dtype=torch.int32, device="cuda"),
                     torch.tensor(np.concatenate([[0], np.cumsum(ns)]), dtype=torch.int32,
                                  device="cuda"), err_flag=err)
    lens = torch.from_numpy(wl.context_lens.astype(np.int32)).cuda()
    ws = pk.decode_workspace(wl.num_seqs, 8, 2, 128, wl.max_blocks)

    def run(out):
        pk.decode_attention_fp8(out, wl.q, kp, vp, tables, lens, wl.scale, workspace=ws,
                                err_flag=err)
    clean, resumed = _aborted_then_resumed(run, wl.q, err)
    assert torch.equal(clean.view(torch.int16), resumed.view(torch.int16))


def test_prefill_returns_without_writing_while_timeout_is_set():
    chunks = [(0, 100), (300, 300), (1000, 1)]
    totals = [s + n for s, n in chunks]
    wl = W.make_decode_workload("abort_prefill", context_lens=np.array(totals) - 1, num_q_heads=8,
                                num_kv_heads=2, head_dim=128, dtype="bf16", seed=74,
                                device="cuda")
    dp = DevicePools(wl)
    k_new, v_new, start, cu, _ = dp.step_inputs()
    pk.append_kv(dp.k, dp.v, k_new, v_new, dp.tables, start, cu, err_flag=dp.err)
    ns = [n for _, n in chunks]
    g = torch.Generator(device="cuda").manual_seed(75)
    q = torch.randn(sum(ns), 8, 128, generator=g, device="cuda").to(torch.bfloat16)
    starts = torch.tensor([s for s, _ in chunks], dtype=torch.int32, device="cuda")
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(ns)]), dtype=torch.int32, device="cuda")

    def run(out):
        pk.prefill_attention(out, q, dp.k, dp.v, dp.tables, starts, cu_q, wl.scale,
                             max_chunk=max(ns), err_flag=dp.err)
    clean, resumed = _aborted_then_resumed(run, q, dp.err)
    assert torch.equal(clean.view(torch.int16), resumed.view(torch.int16))

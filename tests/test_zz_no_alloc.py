"""The decode entry point that allocates nothing (pa_decode_attention_noalloc).

It exists for callers that cannot allocate device memory -- a plugin inside a
framework that owns all device memory and gives it no scratch buffer, or a
latency-critical loop that must not call cudaMalloc because an allocation can
synchronise the device.  It runs the same kernels as pa_decode_attention with
the library's built-in 16 MiB scratch array instead of a caller workspace.

The test calls it through the C ABI twice in a row, on two different batches
that both need scratch (so the second call starts from what the first left in
the shared array), and compares each result with pa_decode_attention given a
fresh workspace.  Both run the same kernels on the same inputs, so the results
must be identical bit for bit (a tolerance could hide a stale-scratch read).  It
also checks that the library's limit is the documented size: a call needing just
under 16 MiB runs, one needing just over is refused.  This file is collected last
so that a failure here cannot hide the other tests' results.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

PA_OK = 0


def _batch(W, pk, seed, lens, hq=32, hkv=8, d=128, dtype="bf16"):
    wl = W.make_decode_workload("noalloc", context_lens=lens, num_q_heads=hq, num_kv_heads=hkv,
                                head_dim=d, dtype=dtype, seed=seed, device="cuda")
    tdt = wl.torch_dtype()
    shape = pk.pool_shape(wl.num_blocks, hkv, d, tdt)
    kp = torch.zeros(shape, dtype=tdt, device="cuda")
    vp = torch.zeros(shape, dtype=tdt, device="cuda")
    tables = torch.from_numpy(wl.block_tables).cuda()
    seqs = [f[0] for f in wl.fill]
    ns = [f[3] for f in wl.fill]
    pk.append_kv(kp, vp, wl.k_rows[:sum(ns)].contiguous(), wl.v_rows[:sum(ns)].contiguous(),
                 tables[torch.tensor(seqs, device="cuda")].contiguous(),
                 torch.tensor([f[1] for f in wl.fill], dtype=torch.int32, device="cuda"),
                 torch.tensor(np.concatenate([[0], np.cumsum(ns)]), dtype=torch.int32,
                              device="cuda"))
    lens_t = torch.from_numpy(wl.context_lens.astype(np.int32)).cuda()
    return wl, kp, vp, tables, lens_t


def test_noalloc_decode_matches_workspace_decode_on_two_calls():
    from paged_kv_cache_207_gb300 import build
    build.build()
    import paged_kv_cache_207_gb300 as pk
    from paged_kv_cache_207_gb300 import workloads as W
    L = pk.lib()
    stream = torch.cuda.current_stream().cuda_stream
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    # (context lengths, query heads, kv heads, head_dim, element type); the second call
    # of each pair starts from the partials the first left in the shared array
    cases = [([3000, 17, 1200, 513, 4000, 640], 32, 8, 128, "bf16"),
             ([900, 2500, 5, 1536], 32, 8, 128, "bf16"),
             ([2100, 700, 33], 12, 12, 64, "f32"),
             ([1025, 3333], 14, 2, 64, "bf16")]
    for i, (lens_, hq, hkv, d, dt) in enumerate(cases):
        wl, kp, vp, tables, lens = _batch(W, pk, 31 + i, lens_, hq, hkv, d, dt)
        S = wl.num_seqs
        need = pk.decode_workspace_size(S, hq, hkv, d, wl.max_blocks)
        assert 0 < need <= pk._native.NOALLOC_SCRATCH_BYTES
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        ref = torch.empty_like(wl.q)
        pk.decode_attention(ref, wl.q, kp, vp, tables, lens, wl.scale, workspace=ws, err_flag=err)
        out = torch.full_like(wl.q, float("nan"))
        st = L.pa_decode_attention_noalloc(out.data_ptr(), wl.q.data_ptr(), kp.data_ptr(),
                                           vp.data_ptr(), tables.data_ptr(), lens.data_ptr(), S,
                                           hq, hkv, d, wl.max_blocks, 0, wl.num_blocks,
                                           ctypes.c_float(wl.scale), 1 if dt == "bf16" else 0,
                                           err.data_ptr(), stream)
        assert st == PA_OK, L.pa_status_string(st)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(out, ref), (out.float() - ref.float()).abs().max().item()

    # a call that would need more than the built-in scratch is refused, nothing launched
    big_blocks = 8192
    need = pk.decode_workspace_size(256, 32, 8, 128, big_blocks)
    assert need > pk._native.NOALLOC_SCRATCH_BYTES
    st = L.pa_decode_attention_noalloc(16, 16, kp.data_ptr(), vp.data_ptr(), 16, 16, 256, 32, 8,
                                       128, big_blocks, 0, wl.num_blocks, ctypes.c_float(0.1), 1,
                                       None, stream)
    assert st == pk._native.PA_ERR_SCRATCH_LIMIT
    assert b"scratch" in L.pa_status_string(st)


def test_noalloc_limit_is_the_documented_size():
    """One sequence, one head of 64 dims: each partition slot takes 64 * 4 + 8 = 264 bytes,
    so a table of 32 * 63550 blocks needs 16 777 200 bytes (just under 16 MiB) and one more
    partition needs 16 777 464 (just over).  The first call runs (its context is one token,
    so it touches one partition), the second is refused before launching anything."""
    from paged_kv_cache_207_gb300 import build
    build.build()
    import paged_kv_cache_207_gb300 as pk
    L = pk.lib()
    stream = torch.cuda.current_stream().cuda_stream
    limit = pk._native.NOALLOC_SCRATCH_BYTES
    under, over = 63550 * 32, 63551 * 32
    assert pk.decode_workspace_size(1, 1, 1, 64, under) <= limit < \
        pk.decode_workspace_size(1, 1, 1, 64, over)
    tables = torch.zeros(1, over, dtype=torch.int32, device="cuda")
    shape = pk.pool_shape(1, 1, 64, torch.bfloat16)
    kp = torch.ones(shape, dtype=torch.bfloat16, device="cuda")
    vp = torch.full(shape, 0.5, dtype=torch.bfloat16, device="cuda")
    q = torch.ones(1, 1, 64, dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(q)
    st = L.pa_decode_attention_noalloc(out.data_ptr(), q.data_ptr(), kp.data_ptr(), vp.data_ptr(),
                                       tables.data_ptr(), lens.data_ptr(), 1, 1, 1, 64, under, 0,
                                       1, ctypes.c_float(0.125), 1, err.data_ptr(), stream)
    assert st == PA_OK, L.pa_status_string(st)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.all(out == 0.5)                # one token: the output is its V row
    st = L.pa_decode_attention_noalloc(out.data_ptr(), q.data_ptr(), kp.data_ptr(), vp.data_ptr(),
                                       tables.data_ptr(), lens.data_ptr(), 1, 1, 1, 64, over, 0,
                                       1, ctypes.c_float(0.125), 1, err.data_ptr(), stream)
    assert st == pk._native.PA_ERR_SCRATCH_LIMIT

"""The decode entry point that allocates nothing (pa_decode_attention_noalloc).

It exists for callers that cannot allocate device memory -- a plugin inside a
framework that owns all device memory and gives it no scratch buffer, or a
latency-critical loop that must not call cudaMalloc because an allocation can
synchronise the device.  It runs the same kernels as pa_decode_attention with
the library's built-in 16 MiB scratch array instead of a caller workspace.

The test calls it through the C ABI twice in a row, on two different batches
that both need scratch (so the second call starts from what the first left in
the shared array), and compares each result with pa_decode_attention given a
fresh workspace, within the bf16 tolerance the parity tests use.  It also checks
that a call needing more than the built-in scratch is refused.  This file is
collected last so that a failure here cannot hide the other tests' results.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

BF16_ATOL = 2e-2   # the bf16 tolerance of the parity tests (tests/_gpu_common.py)


def _batch(W, pk, seed, lens):
    wl = W.make_decode_workload("noalloc", context_lens=lens, num_q_heads=32, num_kv_heads=8,
                                head_dim=128, dtype="bf16", seed=seed, device="cuda")
    shape = pk.pool_shape(wl.num_blocks, 8, 128, torch.bfloat16)
    kp = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
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

    batches = [_batch(W, pk, 31, [3000, 17, 1200, 513, 4000, 640]),
               _batch(W, pk, 32, [900, 2500, 5, 1536])]
    for wl, kp, vp, tables, lens in batches:
        S = wl.num_seqs
        need = pk.decode_workspace_size(S, 32, 8, 128, wl.max_blocks)
        assert 0 < need <= pk._native.NOALLOC_SCRATCH_BYTES
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        ref = torch.empty_like(wl.q)
        pk.decode_attention(ref, wl.q, kp, vp, tables, lens, wl.scale, workspace=ws, err_flag=err)
        out = torch.full_like(wl.q, float("nan"))
        st = L.pa_decode_attention_noalloc(out.data_ptr(), wl.q.data_ptr(), kp.data_ptr(),
                                           vp.data_ptr(), tables.data_ptr(), lens.data_ptr(), S,
                                           32, 8, 128, wl.max_blocks, 0, wl.num_blocks,
                                           ctypes.c_float(wl.scale), 1, err.data_ptr(), stream)
        assert st == 0, L.pa_status_string(st)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        diff = (out.float() - ref.float()).abs().max().item()
        assert diff <= BF16_ATOL, diff

    # a call that would need more than the built-in scratch is refused, nothing launched
    big_blocks = 8192
    need = pk.decode_workspace_size(256, 32, 8, 128, big_blocks)
    assert need > pk._native.NOALLOC_SCRATCH_BYTES
    wl, kp, vp, tables, lens = batches[1]
    st = L.pa_decode_attention_noalloc(16, 16, kp.data_ptr(), vp.data_ptr(), 16, 16, 256, 32, 8,
                                       128, big_blocks, 0, wl.num_blocks, ctypes.c_float(0.1), 1,
                                       None, stream)
    assert st == pk._native.PA_ERR_SCRATCH_LIMIT
    assert b"scratch" in L.pa_status_string(st)

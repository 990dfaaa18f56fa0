"""GPU parity of the spindle-shaped replay: continuous batching over the paged cache.

Every iteration appends one token per running sequence in all 12 layers and decodes;
the decode output of one layer per iteration (rotating) is checked against the oracle
computed on that sequence's logical rows, so the paging machinery -- admissions,
reused blocks that still hold old data, copy-on-write children, preemption and
recomputation -- must leave every sequence with exactly its own context.
"""
import numpy as np
import pytest

from _gpu_common import BF16_ATOL
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def _run_checked(rw, reruns=0, **kw):
    from paged_kv_cache_207_gb300 import build
    build.build()
    from paged_kv_cache_207_gb300.replay import Replay
    kc, vc, qc = rw.k.cpu(), rw.v.cpu(), rw.q.cpu()
    worst = [0.0]
    checked = [0]

    def observer(rp, run, ctx, outs):
        it = rp.stats.iterations
        l = it % rw.num_layers
        got = outs[l].float().cpu().double().numpy()
        for i, s in enumerate(run):
            L = int(ctx[i]) + 1
            K = kc[s, l, :L].contiguous()
            V = vc[s, l, :L].contiguous()
            for h in range(rw.num_heads):
                want = orc.decode_contig(qc[s, l, L - 1, h], K, V, h, num_kv_heads=rw.num_heads,
                                         head_dim=rw.head_dim, scale=rw.scale, dtype=orc.BF16)
                worst[0] = max(worst[0], float(np.abs(got[i, h] - want).max()))
                checked[0] += 1

    rp = Replay(rw, device="cuda", **kw)
    stats = rp.run(observer=observer)
    for _ in range(reruns):
        # the same workload again on the same pools and captured graphs: blocks now hold
        # the first run's values instead of NaN, and every read must still be this run's
        rp.reset()
        checked[0] = 0
        stats = rp.run(observer=observer)
    assert all(s == "done" for s in rp.state)
    assert worst[0] <= BF16_ATOL, worst[0]
    assert checked[0] > 0
    return stats


def test_spindle_replay_default_pool():
    from paged_kv_cache_207_gb300 import workloads as W
    rw = W.spindle_replay(device="cuda")
    stats = _run_checked(rw)
    assert stats.generated_tokens == int(rw.gen_lens.sum())


def test_spindle_replay_tight_pool_preempts_and_recomputes():
    from paged_kv_cache_207_gb300 import workloads as W
    rw = W.spindle_replay(device="cuda", num_blocks=150)
    stats = _run_checked(rw)
    assert stats.preemptions > 0


def test_spindle_replay_with_cuda_graphs():
    from paged_kv_cache_207_gb300 import workloads as W
    rw = W.spindle_replay(device="cuda", num_blocks=150)
    stats = _run_checked(rw, use_graphs=True)
    assert stats.preemptions > 0


def test_spindle_replay_reset_reuses_pools_and_graphs():
    from paged_kv_cache_207_gb300 import workloads as W
    rw = W.spindle_replay(device="cuda", num_blocks=150)
    stats = _run_checked(rw, reruns=1, use_graphs=True)
    assert stats.preemptions > 0
    assert stats.generated_tokens == int(rw.gen_lens.sum())


def test_spindle_replay_partial_parent_copies_on_write():
    from paged_kv_cache_207_gb300 import workloads as W
    rw = W.spindle_replay(device="cuda", parent_prompt=20, num_independent=8, num_blocks=64)
    stats = _run_checked(rw)
    assert stats.cow_copies >= 3

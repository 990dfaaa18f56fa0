"""The replay's host schedule (no GPU): continuous batching over the block manager.

spindle, "Paging": 64 requests, 8192 token slots, block size 16, four forks of a
16-token parent.  The schedule must drain every request, keep each sequence's
waste under one block, share the parent's block among the children, and drive
the product block manager and the oracle's plain model to identical tables,
copy pairs and counts, iteration by iteration.
"""
import pytest

from oracle.block_manager import OracleBlockManager, OutOfBlocks


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_207_gb300 import build
    build.build()
    import paged_kv_cache_207_gb300 as pk
    return pk


class OracleAdapter:
    """The oracle's block-manager model behind the product manager's interface."""

    def __init__(self, pk, nb):
        self.pk = pk
        self.m = OracleBlockManager(nb)

    def add_seq(self):
        return self.m.add_sequence()

    def fork(self, parent):
        return self.m.fork(parent)

    def free(self, s):
        self.m.free(s)

    def prepare_append(self, s, start, n):
        try:
            return self.m.prepare_append(s, start, n)
        except OutOfBlocks:
            raise self.pk.PagedKVError("prepare_append", 4, "out of free blocks")

    def block_table(self, s, mb):
        t = self.m.tables[s]
        return t + [-1] * (mb - len(t))

    def stats(self):
        return self.m.stats()


def _trace(pk, rw, bm=None):
    from paged_kv_cache_207_gb300.replay import Replay
    log = []

    def rec(rp, run, ctx, prefill, pairs):
        tables = [tuple(rp.bm.block_table(rp.bm_id[s], rp.max_blocks)) for s in run]
        log.append((tuple(run), tuple(int(c) for c in ctx), tuple(tables), tuple(pairs),
                    tuple((p[0], p[2]) for p in prefill), rp.bm.stats()["physical_blocks"]))
        # waste bound: every running sequence holds less than one spare block
        for s, c in zip(run, ctx):
            held = sum(1 for b in rp.bm.block_table(rp.bm_id[s], rp.max_blocks) if b >= 0)
            assert held * 16 - (int(c) + 1) < 16

    rp = Replay(rw, device=None, block_manager=bm, on_schedule=rec)
    stats = rp.run()
    return rp, stats, log


def test_replay_schedule_drains_and_matches_the_oracle_block_manager(pk):
    from paged_kv_cache_207_gb300 import workloads as W
    rw = W.spindle_replay(values=False)
    rp, stats, log = _trace(pk, rw)
    assert all(s == "done" for s in rp.state)
    assert stats.generated_tokens == int(rw.gen_lens.sum())   # each token once
    assert stats.iterations == len(log)
    assert rp.bm.stats()["physical_blocks"] == 0
    # the pool (8192 slots) is smaller than the demand, so the schedule preempts
    assert int((rw.prompt_lens + rw.gen_lens).sum()) > 8192
    # the four children were admitted together and shared the parent's block
    first = [e for e in log if 60 in e[0]][0]
    idx = [first[0].index(c) for c in range(60, 64)]
    assert len({first[2][i][0] for i in idx}) == 1
    _, stats_o, log_o = _trace(pk, rw, bm=OracleAdapter(pk, rw.num_blocks))
    assert log == log_o
    assert (stats.preemptions, stats.cow_copies, stats.peak_physical_slots) == \
        (stats_o.preemptions, stats_o.cow_copies, stats_o.peak_physical_slots)


def test_replay_with_a_partial_parent_block_makes_copy_on_write_pairs(pk):
    # a 20-token parent leaves its second block partial: each child's first write copies it
    from paged_kv_cache_207_gb300 import workloads as W
    rw = W.spindle_replay(values=False, parent_prompt=20, num_independent=8, num_blocks=64)
    rp, stats, log = _trace(pk, rw)
    assert all(s == "done" for s in rp.state)
    assert stats.cow_copies >= 3      # the last holder writes in place
    _, stats_o, log_o = _trace(pk, rw, bm=OracleAdapter(pk, rw.num_blocks))
    assert log == log_o


def test_replay_under_a_tight_pool_preempts_and_recomputes(pk):
    from paged_kv_cache_207_gb300 import workloads as W
    rw = W.spindle_replay(values=False, num_blocks=150)
    rp, stats, log = _trace(pk, rw)
    assert all(s == "done" for s in rp.state)
    assert stats.preemptions > 0
    assert stats.prefill_tokens > int(rw.prompt_lens[:60].sum()) + 16   # recomputed contexts
    assert stats.generated_tokens == int(rw.gen_lens.sum())
    _, stats_o, log_o = _trace(pk, rw, bm=OracleAdapter(pk, rw.num_blocks))
    assert log == log_o

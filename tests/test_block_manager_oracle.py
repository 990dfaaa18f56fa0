"""Pins of the plain-Python block-manager model (no GPU needed).

spindle, section "Paging": fixed 16-token blocks and per-sequence block tables
bound waste by the final partial block; refcounts give copy-on-write forking,
and four forks of a 16-token parent hold 64 logical tokens in 16 physical ones.
"""
import json
import os
import random

import pytest

from oracle.block_manager import OracleBlockManager, OutOfBlocks

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _check_invariants(bm: OracleBlockManager):
    # brute force: each refcount equals the number of table entries naming the block,
    # and no sequence holds more than one partial block's worth of unused slots
    counts = [0] * bm.num_blocks
    for sid, table in bm.tables.items():
        for b in table:
            counts[b] += 1
        L = bm.lengths[sid]
        assert len(table) * bm.block_size - L < bm.block_size or L == 0 and not table
    assert counts == bm.refcount


def test_four_forks_of_a_16_token_parent_hold_64_tokens_in_16_slots():
    g = json.load(open(os.path.join(GOLDEN, "spindle_cow_fork.json")))
    bm = OracleBlockManager(64, g["block_size"])
    parent = bm.add_sequence()
    assert bm.prepare_append(parent, 0, g["parent_tokens"]) == []
    kids = [bm.fork(parent) for _ in range(g["forks"])]
    bm.free(parent)
    st = bm.stats()
    assert st["logical_tokens"] == g["logical_tokens"]
    assert st["physical_slots"] == g["physical_slots"]
    assert all(bm.refcount[bm.tables[k][0]] == g["forks"] for k in kids)
    # the parent filled its block, so each child's next token opens a private block
    for k in kids:
        assert bm.prepare_append(k, g["parent_tokens"], 1) == []
    _check_invariants(bm)


def test_write_into_shared_partial_block_copies_it_once():
    bm = OracleBlockManager(16)
    parent = bm.add_sequence()
    bm.prepare_append(parent, 0, 20)                 # blocks [a, b], b holds 4 tokens
    a, b = bm.tables[parent]
    child = bm.fork(parent)
    pairs = bm.prepare_append(child, 20, 1)          # child writes into shared b
    assert len(pairs) == 1 and pairs[0][0] == b
    new = pairs[0][1]
    assert bm.tables[child] == [a, new] and bm.tables[parent] == [a, b]
    assert bm.refcount[a] == 2 and bm.refcount[b] == 1 and bm.refcount[new] == 1
    # the parent is now the last holder of b and writes in place, no copy
    assert bm.prepare_append(parent, 20, 1) == []
    _check_invariants(bm)


def test_out_of_blocks_leaves_state_unchanged():
    bm = OracleBlockManager(2)
    s = bm.add_sequence()
    bm.prepare_append(s, 0, 30)
    before = (list(bm.refcount), list(bm.tables[s]), bm.lengths[s])
    with pytest.raises(OutOfBlocks):
        bm.prepare_append(s, 30, 5)
    assert (list(bm.refcount), list(bm.tables[s]), bm.lengths[s]) == before


def test_random_operations_keep_refcounts_and_waste_bound():
    rnd = random.Random(5)
    bm = OracleBlockManager(200)
    live = []
    for _ in range(2000):
        op = rnd.random()
        if op < 0.1 or not live:
            live.append(bm.add_sequence())
        elif op < 0.2:
            live.append(bm.fork(rnd.choice(live)))
        elif op < 0.3:
            s = live.pop(rnd.randrange(len(live)))
            bm.free(s)
        else:
            s = rnd.choice(live)
            n = rnd.randint(1, 20)
            try:
                bm.prepare_append(s, bm.lengths[s], n)
            except OutOfBlocks:
                pass
        _check_invariants(bm)

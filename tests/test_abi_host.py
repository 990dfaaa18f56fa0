"""Host-side checks of the C ABI library (no GPU needed).

The library must load, export every function ``include/pa.h`` declares, reject
host-checkable bad arguments before touching the GPU, and its host block
manager must agree with the plain-Python block-manager model of the oracle.
"""
import ctypes
import os
import random
import re

import pytest

from oracle.block_manager import OracleBlockManager, OutOfBlocks

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def native():
    from paged_kv_cache_207_gb300 import build, _native
    build.build()
    return _native


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_function_is_exported(native):
    L = native.lib()
    names = _declared_functions()
    assert len(names) >= 17
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(native.EXPORTED)
    assert L.pa_abi_version() == 1


def test_status_strings(native):
    L = native.lib()
    assert L.pa_status_string(0) == b"ok"
    assert L.pa_status_string(4) == b"out of free blocks"


def test_workspace_size_formula(native):
    L = native.lib()
    # one partition (max 32 blocks = 512 tokens) needs no workspace
    assert L.pa_decode_workspace_size(4, 12, 12, 64, 7) == 0
    assert L.pa_decode_workspace_size(4, 12, 12, 64, 32) == 0
    # 33 blocks -> 2 partitions: S*Hq*2 rows of (D floats + (max, sum))
    assert L.pa_decode_workspace_size(4, 12, 12, 64, 33) == 4 * 12 * 2 * (64 * 4 + 8)
    assert L.pa_decode_workspace_size(8, 32, 8, 128, 8192) == 8 * 32 * 256 * (128 * 4 + 8)


def _decode(L, **kw):
    a = dict(out=16, q=16, k=16, v=16, tables=16, lens=16, S=1, Hq=4, Hkv=2, D=64, mb=4, hint=0,
             nb=8, scale=0.125, dtype=1, ws=None, wsb=0, err=None)
    a.update(kw)
    return L.pa_decode_attention(a["out"], a["q"], a["k"], a["v"], a["tables"], a["lens"], a["S"],
                                 a["Hq"], a["Hkv"], a["D"], a["mb"], a["hint"], a["nb"], a["scale"],
                                 a["dtype"], a["ws"], a["wsb"], a["err"], None)


def test_decode_rejects_bad_arguments_without_launching(native):
    L = native.lib()
    INVALID, UNSUPPORTED = 1, 2
    assert _decode(L, D=96) == UNSUPPORTED
    assert _decode(L, Hq=5) == INVALID
    assert _decode(L, Hq=18, Hkv=2) == UNSUPPORTED          # 9 query heads per kv head
    assert _decode(L, q=None) == INVALID
    assert _decode(L, k=8) == INVALID                          # not 16-byte aligned
    assert _decode(L, dtype=7) == INVALID
    assert _decode(L, scale=float("nan")) == INVALID
    assert _decode(L, mb=40) == INVALID                        # needs a workspace, none given
    assert _decode(L, mb=40, ws=16, wsb=10) == INVALID         # workspace too small
    assert _decode(L, S=0) == 0                                # nothing to do


def _append_decode(L, kn=16, vn=16, **kw):
    a = dict(out=16, q=16, k=16, v=16, tables=16, lens=16, S=1, Hq=4, Hkv=2, D=64, mb=4, hint=0,
             nb=8, scale=0.125, dtype=1, ws=None, wsb=0, err=None)
    a.update(kw)
    return L.pa_append_decode_attention(a["out"], a["q"], a["k"], a["v"], kn, vn, a["tables"],
                                        a["lens"], a["S"], a["Hq"], a["Hkv"], a["D"], a["mb"],
                                        a["hint"], a["nb"], a["scale"], a["dtype"], a["ws"],
                                        a["wsb"], a["err"], None)


def test_append_decode_rejects_bad_arguments_without_launching(native):
    L = native.lib()
    INVALID, UNSUPPORTED = 1, 2
    assert _append_decode(L, kn=None) == INVALID               # the new rows are required
    assert _append_decode(L, vn=None) == INVALID
    assert _append_decode(L, kn=8) == INVALID                  # not 16-byte aligned
    assert _append_decode(L, vn=24) == INVALID
    assert _append_decode(L, D=96) == UNSUPPORTED
    assert _append_decode(L, dtype=2) == INVALID               # the FP8 cache has its own append
    assert _append_decode(L, dtype=3) == INVALID               # and so has the FP4 one
    assert _append_decode(L, mb=40) == INVALID                 # needs a workspace, none given
    assert _append_decode(L, S=0, kn=None, vn=None) == 0       # nothing to do


def test_append_and_copy_reject_bad_arguments(native):
    L = native.lib()
    assert L.pa_append_kv(16, 16, 16, 16, 16, 4, 16, 16, 1, 1, 8, 2, 64, 5, None, None) == 1
    assert L.pa_append_kv(None, 16, 16, 16, 16, 4, 16, 16, 1, 1, 8, 2, 64, 1, None, None) == 1
    assert L.pa_append_kv(16, 16, 16, 16, 16, 4, 16, 16, 0, 0, 8, 2, 64, 1, None, None) == 0
    assert L.pa_append_kv(16, 16, 16, 16, 16, 4, 16, 16, 1, 1, 8, 2, 4, 1, None, None) == 2
    assert L.pa_copy_block(16, 16, 16, 0, 8, 2, 64, 1, None, None) == 0
    assert L.pa_copy_block(16, 16, None, 3, 8, 2, 64, 1, None, None) == 1
    assert L.pa_copy_block(24, 16, 16, 3, 8, 2, 64, 1, None, None) == 1


# ---- host block manager against the oracle's model ---------------------------------

def test_block_manager_matches_oracle_model_op_for_op(native):
    rnd = random.Random(11)
    nb = 120
    bm = native.BlockManager(nb)
    om = OracleBlockManager(nb)
    ids = {}          # oracle id -> product id
    for _ in range(3000):
        live = list(ids)
        op = rnd.random()
        if op < 0.08 or not live:
            ids[om.add_sequence()] = bm.add_seq()
        elif op < 0.16:
            par = rnd.choice(live)
            ids[om.fork(par)] = bm.fork(ids[par])
        elif op < 0.24:
            s = rnd.choice(live)
            om.free(s)
            bm.free(ids.pop(s))
        else:
            s = rnd.choice(live)
            L = om.lengths[s]
            start = L if rnd.random() < 0.8 else rnd.randint(max(0, L - 20), L)
            n = rnd.randint(1, 40)
            try:
                want = om.prepare_append(s, start, n)
            except OutOfBlocks:
                with pytest.raises(native.PagedKVError) as ei:
                    bm.prepare_append(ids[s], start, n)
                assert ei.value.status == 4
                continue
            got = bm.prepare_append(ids[s], start, n)
            assert got == want
        for s, p in ids.items():
            assert bm.block_table(p, 64)[:len(om.tables[s])] == om.tables[s]
            assert bm.seq_len(p) == om.lengths[s]
        if ids:
            # the batched tables equal the per-sequence ones, row for row (-1 padded)
            order = list(ids)
            rnd.shuffle(order)
            rows = bm.block_tables([ids[s] for s in order], 64)
            for r, s in zip(rows, order):
                want = om.tables[s] + [-1] * (64 - len(om.tables[s]))
                assert r.tolist() == want
        st = bm.stats()
        assert st["physical_blocks"] == om.physical_blocks()
        assert st["logical_tokens"] == om.logical_tokens()
    for b in range(nb):
        assert bm.refcount(b) == om.refcount[b]


def test_block_manager_fork_numbers_from_the_paging_section(native):
    import json
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "spindle_cow_fork.json")))
    bm = native.BlockManager(64)
    parent = bm.add_seq()
    assert bm.prepare_append(parent, 0, g["parent_tokens"]) == []
    kids = [bm.fork(parent) for _ in range(g["forks"])]
    bm.free(parent)
    st = bm.stats()
    assert st["logical_tokens"] == g["logical_tokens"]
    assert st["physical_slots"] == g["physical_slots"]
    blk = bm.block_table(kids[0], 1)[0]
    assert bm.refcount(blk) == g["forks"]


def test_block_manager_rejects_holes_and_unknown_sequences(native):
    bm = native.BlockManager(8)
    s = bm.add_seq()
    with pytest.raises(native.PagedKVError):
        bm.block_tables([s, 99], 4)           # an unknown sequence in the batch
    t = bm.add_seq()
    bm.prepare_append(t, 0, 40)
    with pytest.raises(native.PagedKVError):
        bm.block_tables([t], 2)               # three blocks do not fit in two entries
    assert bm.block_tables([], 4).shape == (0, 4)
    with pytest.raises(native.PagedKVError):
        bm.prepare_append(s, 17, 1)          # would skip block 0
    with pytest.raises(native.PagedKVError):
        bm.free(99)
    L = native.lib()
    h = ctypes.c_void_p()
    assert L.pa_bm_create(0, ctypes.byref(h)) == 1


def test_one_call_bindings_check_the_new_rows_on_the_host(native):
    # the bindings refuse new rows of the wrong shape, type or layout before any call
    import torch
    pool = torch.zeros(native.pool_shape(4, 2, 64, torch.bfloat16), dtype=torch.bfloat16)
    q = torch.zeros(3, 4, 64, dtype=torch.bfloat16)
    good = torch.zeros(3, 2, 64, dtype=torch.bfloat16)
    bad = [torch.zeros(3, 2, 32, dtype=torch.bfloat16),        # head_dim
           torch.zeros(2, 2, 64, dtype=torch.bfloat16),        # sequences
           torch.zeros(3, 2, 64, dtype=torch.float32),         # type
           torch.zeros(3, 64, 2, dtype=torch.bfloat16).transpose(1, 2)]   # layout
    tables = torch.zeros(3, 4, dtype=torch.int32)
    lens = torch.ones(3, dtype=torch.int32)
    for b in bad:
        with pytest.raises(ValueError):
            native.append_decode_attention(q.clone(), q, pool, pool, b, good, tables, lens, 0.125)
        with pytest.raises(ValueError):
            native.append_decode_attention_shared_prefix(q.clone(), q, pool, pool, good, b, tables,
                                                         lens, 0.125, 512)
    fp8 = torch.zeros(native.fp8_pool_shape(4, 2, 64), dtype=torch.uint8)
    for b in bad:
        with pytest.raises(ValueError):
            native.append_decode_attention_fp8(q.clone(), q, fp8, fp8, b, good, tables, lens, 0.125)

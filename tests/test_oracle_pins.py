"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Every test here checks the oracle against something it does not compute from
its own formula: hand-worked values, closed forms, special cases that reduce to
a library routine (torch's scaled_dot_product_attention, torch's bf16 rounding),
and invariants of paging stated on spindle's "Paging" and "Two bugs worth
recording" sections.  Each is chosen so that a plausible slip in the oracle (a
dropped max subtraction, a flipped sign, a wrong block / slot index, a wrong
query-to-kv head map, a transposed operand) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32, BF16 = 0, 1


def _x(dtype):
    return 8 if dtype == BF16 else 4


def _empty_pool(o, nb, hkv, d, dtype, fill=None):
    shape = o.pool_shape(nb, hkv, d, dtype)
    et = np.uint16 if dtype == BF16 else np.float32
    a = np.zeros(shape, et)
    if fill is not None:
        a.view(np.uint16 if dtype == BF16 else np.uint32)[...] = fill
    return a


def _to_elems(x: torch.Tensor, dtype):
    """fp32 tensor -> numpy array of the element type (bf16 as RNE bits via torch)."""
    if dtype == BF16:
        return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return x.to(torch.float32).numpy()


def _to_f64(a, dtype):
    if dtype == BF16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _fill(o, rows_k, rows_v, tables, lens, nb, hkv, d, dtype):
    """Put each sequence's rows (dict s -> [L][Hkv][D] elems) into fresh pools with the
    oracle's own append (start 0, explicit length)."""
    kp = _empty_pool(o, nb, hkv, d, dtype, fill=0xFFFF if dtype == BF16 else 0x7FC00000)
    vp = _empty_pool(o, nb, hkv, d, dtype, fill=0xFFFF if dtype == BF16 else 0x7FC00000)
    S = len(lens)
    for s in range(S):
        L = lens[s]
        if L == 0:
            continue
        one_t = np.array(tables[s:s + 1], np.int32)
        rc = o.append_kv(kp, vp, rows_k[s], rows_v[s], one_t, np.array([0], np.int32),
                         np.array([0, L], np.int32), num_kv_heads=hkv, head_dim=d,
                         num_blocks=nb, dtype=dtype)
        assert rc == 0
    return kp, vp


def _random_case(seed, S, hq, hkv, d, lens, dtype, nb=None):
    g = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    need = [(L + 15) // 16 for L in lens]
    nb = nb or sum(need) + 3
    mb = max(need + [1])
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.full((S, mb), -1, np.int32)
    k = 0
    for s in range(S):
        tables[s, :need[s]] = perm[k:k + need[s]]
        k += need[s]
    rk = {s: _to_elems(torch.randn(lens[s], hkv, d, generator=g), dtype) for s in range(S)}
    rv = {s: _to_elems(torch.randn(lens[s], hkv, d, generator=g), dtype) for s in range(S)}
    q = _to_elems(torch.randn(S, hq, d, generator=g), dtype)
    return q, rk, rv, tables, nb


# ---- element conversion -------------------------------------------------------

def test_bf16_rounding_hand_worked_cases(oracle_mod):
    cases = json.load(open(os.path.join(GOLDEN, "bf16_rounding.json")))["cases"]
    for c in cases:
        assert oracle_mod.double_to_bf16(c["x"]) == int(c["bits"], 16), c
        assert oracle_mod.double_to_bf16(-c["x"]) == int(c["bits"], 16) ^ 0x8000, c


def test_bf16_rounding_matches_torch_on_fp32_values(oracle_mod):
    # For inputs that are fp32 values, one-step double -> bf16 rounding must equal
    # torch's fp32 -> bf16 conversion (round to nearest even), a library routine.
    g = torch.Generator().manual_seed(1)
    x = torch.cat([torch.randn(20000, generator=g) * 10 ** torch.randint(-30, 30, (20000,), generator=g).float(),
                   torch.randn(2000, generator=g) * 1e-39])
    want = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle_mod.round_out(x.double().numpy(), BF16)
    assert np.array_equal(got, want)


def test_bf16_widening_is_exact(oracle_mod):
    for bits, val in [(0x3F80, 1.0), (0xC000, -2.0), (0x0001, 2.0 ** -133), (0x4049, 3.140625),
                      (0x7F7F, (2 - 2 ** -7) * 2.0 ** 127)]:
        assert oracle_mod.bf16_to_double(bits) == val
    assert math.isinf(oracle_mod.bf16_to_double(0x7F80))


# ---- attention closed forms ------------------------------------------------------

@pytest.mark.parametrize("dtype", [F32, BF16])
def test_single_token_context_returns_its_value_row(oracle_mod, dtype):
    q, rk, rv, tables, nb = _random_case(3, 2, 4, 2, 64, [1, 1], dtype)
    kp, vp = _fill(oracle_mod, rk, rv, tables, [1, 1], nb, 2, 64, dtype)
    out = oracle_mod.decode(q, kp, vp, tables, np.array([1, 1], np.int32), num_q_heads=4,
                            num_kv_heads=2, head_dim=64, num_blocks=nb, scale=0.125, dtype=dtype)
    for s in range(2):
        for h in range(4):
            assert np.array_equal(out[s, h], _to_f64(rv[s][0, h // 2], dtype))


@pytest.mark.parametrize("dtype", [F32, BF16])
def test_zero_query_gives_mean_of_values(oracle_mod, dtype):
    lens = [1, 17, 40, 100]
    q, rk, rv, tables, nb = _random_case(4, 4, 6, 3, 64, lens, dtype)
    q[...] = 0
    kp, vp = _fill(oracle_mod, rk, rv, tables, lens, nb, 3, 64, dtype)
    out = oracle_mod.decode(q, kp, vp, tables, np.array(lens, np.int32), num_q_heads=6,
                            num_kv_heads=3, head_dim=64, num_blocks=nb, scale=0.3, dtype=dtype)
    for s, L in enumerate(lens):
        for h in range(6):
            want = _to_f64(rv[s][:, h // 2], dtype).mean(axis=0)
            np.testing.assert_allclose(out[s, h], want, rtol=0, atol=1e-13)


def test_two_token_closed_form(oracle_mod):
    # x0 = 2, x1 = 0 at scale 1: p0 = 1 / (1 + e^-2), p1 = 1 - p0.
    D = 8
    k = np.zeros((2, 1, D), np.float32); k[0, 0, 0] = 2.0
    v = np.zeros((2, 1, D), np.float32); v[0, 0, 0] = 1.0; v[1, 0, 1] = 1.0
    q = np.zeros((1, 1, D), np.float32); q[0, 0, 0] = 1.0
    tables = np.array([[5]], np.int32)
    kp, vp = _fill(oracle_mod, {0: k}, {0: v}, tables, [2], 8, 1, D, F32)
    out = oracle_mod.decode(q, kp, vp, tables, np.array([2], np.int32), num_q_heads=1,
                            num_kv_heads=1, head_dim=D, num_blocks=8, scale=1.0, dtype=F32)
    p0 = 1.0 / (1.0 + math.exp(-2.0))
    want = np.zeros(D); want[0] = p0; want[1] = 1.0 - p0
    np.testing.assert_allclose(out[0, 0], want, rtol=0, atol=1e-15)


@pytest.mark.parametrize("hot", [0, 15, 16, 37, 99])
def test_dominant_key_selects_its_value(oracle_mod, hot):
    # One key aligned with q scores 100 above all others (others score 0): the output is
    # that token's value within e^-100.  A flipped score sign or a wrong slot/block
    # index picks a different row.
    L, D = 100, 64
    k = np.zeros((L, 1, D), np.float32); k[hot, 0, 3] = 100.0
    v = np.arange(L, dtype=np.float32)[:, None, None] * np.ones((1, 1, D), np.float32)
    q = np.zeros((1, 1, D), np.float32); q[0, 0, 3] = 1.0
    rng = np.random.default_rng(hot)
    tables = rng.permutation(20)[:7].astype(np.int32)[None, :]
    kp, vp = _fill(oracle_mod, {0: k}, {0: v}, tables, [L], 20, 1, D, F32)
    out = oracle_mod.decode(q, kp, vp, tables, np.array([L], np.int32), num_q_heads=1,
                            num_kv_heads=1, head_dim=D, num_blocks=20, scale=1.0, dtype=F32)
    np.testing.assert_allclose(out[0, 0], np.full(D, float(hot)), rtol=0, atol=1e-9)


def test_positions_reach_the_right_block_and_slot(oracle_mod):
    # Value rows encode their logical position; with q = 0 the output is the mean
    # position (L - 1) / 2 whatever block order the table uses.
    D = 64
    for L in (1, 15, 16, 17, 33, 100):
        v = np.arange(L, dtype=np.float32)[:, None, None] * np.ones((1, 2, D), np.float32)
        k = np.zeros((L, 2, D), np.float32)
        rng = np.random.default_rng(L)
        nblk = (L + 15) // 16
        tables = rng.permutation(3 * nblk + 2)[:nblk].astype(np.int32)[None, :]
        nb = 3 * nblk + 2
        kp, vp = _fill(oracle_mod, {0: k}, {0: v}, tables, [L], nb, 2, D, F32)
        out = oracle_mod.decode(np.zeros((1, 2, D), np.float32), kp, vp, tables,
                                np.array([L], np.int32), num_q_heads=2, num_kv_heads=2,
                                head_dim=D, num_blocks=nb, scale=1.0, dtype=F32)
        np.testing.assert_allclose(out[0], (L - 1) / 2.0, rtol=0, atol=1e-12)


def test_gqa_query_head_reads_kv_head_h_div_group(oracle_mod):
    # 8 query heads over 2 kv heads: heads 0-3 read kv head 0, 4-7 read kv head 1.
    # kv head g holds the constant value g + 1, so the output is h // 4 + 1 exactly.
    L, D = 20, 64
    v = np.zeros((L, 2, D), np.float32); v[:, 0] = 1.0; v[:, 1] = 2.0
    k = np.random.default_rng(0).standard_normal((L, 2, D)).astype(np.float32)
    q = np.random.default_rng(1).standard_normal((1, 8, D)).astype(np.float32)
    tables = np.array([[3, 1]], np.int32)
    kp, vp = _fill(oracle_mod, {0: k}, {0: v}, tables, [L], 4, 2, D, F32)
    out = oracle_mod.decode(q, kp, vp, tables, np.array([L], np.int32), num_q_heads=8,
                            num_kv_heads=2, head_dim=D, num_blocks=4, scale=0.125, dtype=F32)
    for h in range(8):
        np.testing.assert_allclose(out[0, h], h // 4 + 1.0, rtol=0, atol=1e-14)


def test_zero_length_context_is_zero(oracle_mod):
    q, rk, rv, tables, nb = _random_case(5, 2, 2, 2, 64, [0, 5], F32)
    kp, vp = _fill(oracle_mod, rk, rv, tables, [0, 5], nb, 2, 64, F32)
    out = oracle_mod.decode(q, kp, vp, tables, np.array([0, 5], np.int32), num_q_heads=2,
                            num_kv_heads=2, head_dim=64, num_blocks=nb, scale=0.125, dtype=F32)
    assert np.all(out[0] == 0.0) and np.all(np.isfinite(out[1]))


def test_large_scores_do_not_overflow(oracle_mod):
    # Scores near 1000 overflow exp() without the max subtraction.
    L, D = 40, 64
    k = np.full((L, 1, D), 1.0, np.float32); k[7] = 1.01
    v = np.random.default_rng(2).standard_normal((L, 1, D)).astype(np.float32)
    q = np.full((1, 1, D), 16.0, np.float32)
    tables = np.array([[0, 1, 2]], np.int32)
    kp, vp = _fill(oracle_mod, {0: k}, {0: v}, tables, [L], 3, 1, D, F32)
    out = oracle_mod.decode(q, kp, vp, tables, np.array([L], np.int32), num_q_heads=1,
                            num_kv_heads=1, head_dim=D, num_blocks=3, scale=1.0, dtype=F32)
    assert np.all(np.isfinite(out))
    # token 7 scores 16 * 64 * (1.01f - 1) (about 10.24) above the rest
    gap = 16.0 * 64.0 * (float(np.float32(1.01)) - 1.0)
    w7 = math.exp(gap) / (math.exp(gap) + (L - 1))
    want = w7 * v[7, 0].astype(np.float64) + (1 - w7) * np.delete(v[:, 0], 7, axis=0).astype(np.float64).mean(0)
    np.testing.assert_allclose(out[0, 0], want, rtol=0, atol=1e-5)


# ---- against a library routine ---------------------------------------------------

@pytest.mark.parametrize("dtype", [F32, BF16])
@pytest.mark.parametrize("hq,hkv,d", [(12, 12, 64), (14, 2, 64), (8, 2, 128)])
def test_matches_torch_sdpa_on_contiguous_rows(oracle_mod, dtype, hq, hkv, d):
    # The contiguous case of the method is ordinary scaled-dot-product attention:
    # compare the paged oracle with torch's float64 SDPA over the same rows, with each
    # kv head repeated for its group of query heads.
    lens = [1, 16, 17, 40, 64, 100]
    S = len(lens)
    scale = 1.0 / math.sqrt(d)
    q, rk, rv, tables, nb = _random_case(11 + hq, S, hq, hkv, d, lens, dtype, nb=60)
    kp, vp = _fill(oracle_mod, rk, rv, tables, lens, nb, hkv, d, dtype)
    out = oracle_mod.decode(q, kp, vp, tables, np.array(lens, np.int32), num_q_heads=hq,
                            num_kv_heads=hkv, head_dim=d, num_blocks=nb, scale=scale, dtype=dtype)
    G = hq // hkv
    for s, L in enumerate(lens):
        K = torch.from_numpy(_to_f64(rk[s], dtype)).permute(1, 0, 2).repeat_interleave(G, 0)
        V = torch.from_numpy(_to_f64(rv[s], dtype)).permute(1, 0, 2).repeat_interleave(G, 0)
        Q = torch.from_numpy(_to_f64(q[s], dtype)).unsqueeze(1)           # [Hq][1][D]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=scale)[:, 0]
        np.testing.assert_allclose(out[s], ref.numpy(), rtol=0, atol=1e-12)


# ---- paging invariants -------------------------------------------------------------

@pytest.mark.parametrize("dtype", [F32, BF16])
def test_paged_equals_contiguous_and_batched_equals_alone(oracle_mod, dtype):
    lens = [3, 16, 31, 64, 65]
    S, hq, hkv, d = len(lens), 4, 2, 64
    q, rk, rv, tables, nb = _random_case(21, S, hq, hkv, d, lens, dtype, nb=40)
    kp, vp = _fill(oracle_mod, rk, rv, tables, lens, nb, hkv, d, dtype)
    batched = oracle_mod.decode(q, kp, vp, tables, np.array(lens, np.int32), num_q_heads=hq,
                                num_kv_heads=hkv, head_dim=d, num_blocks=nb, scale=0.125,
                                dtype=dtype)
    for s, L in enumerate(lens):
        alone = oracle_mod.decode(q[s:s + 1], kp, vp, tables[s:s + 1], np.array([L], np.int32),
                                  num_q_heads=hq, num_kv_heads=hkv, head_dim=d, num_blocks=nb,
                                  scale=0.125, dtype=dtype)
        assert np.array_equal(alone[0], batched[s])
        for h in range(hq):
            contig = oracle_mod.decode_contig(q[s, h], rk[s], rv[s], h // (hq // hkv),
                                              num_kv_heads=hkv, head_dim=d, scale=0.125,
                                              dtype=dtype)
            assert np.array_equal(contig, batched[s, h])


def test_append_writes_only_its_slots_and_reads_back(oracle_mod):
    # A NaN canary fills both pools; an append of n tokens at an explicit start changes
    # exactly n * Hkv * D elements per pool, and attention over a 1-token window made of
    # the last written token with q = 0 returns that token's value row.
    hkv, d, nb = 2, 64, 6
    kp = _empty_pool(oracle_mod, nb, hkv, d, BF16, fill=0xFFFF)
    vp = _empty_pool(oracle_mod, nb, hkv, d, BF16, fill=0xFFFF)
    g = torch.Generator().manual_seed(9)
    n, start = 5, 13
    kn = _to_elems(torch.randn(n, hkv, d, generator=g), BF16)
    vn = _to_elems(torch.randn(n, hkv, d, generator=g), BF16)
    tables = np.array([[4, 2, -1]], np.int32)
    rc = oracle_mod.append_kv(kp, vp, kn, vn, tables, np.array([start], np.int32),
                              np.array([0, n], np.int32), num_kv_heads=hkv, head_dim=d,
                              num_blocks=nb, dtype=BF16)
    assert rc == 0
    assert int((kp != 0xFFFF).sum()) == n * hkv * d and int((vp != 0xFFFF).sum()) == n * hkv * d
    # whole blocks other than 4 and 2 are untouched
    for b in (0, 1, 3, 5):
        assert np.all(kp[b] == 0xFFFF) and np.all(vp[b] == 0xFFFF)
    # positions 13..17: 13, 14, 15 in block 4 and 16, 17 in block 2
    one = np.array([[2, -1, -1]], np.int32)
    # a table whose only entry is block 2 sees written positions 16 and 17 as its 0 and 1
    out = oracle_mod.decode(np.zeros((1, hkv, d), np.uint16), kp, vp, one, np.array([2], np.int32),
                            num_q_heads=hkv, num_kv_heads=hkv, head_dim=d, num_blocks=nb,
                            scale=1.0, dtype=BF16)
    want = (_to_f64(vn[3], BF16) + _to_f64(vn[4], BF16)) / 2.0
    np.testing.assert_allclose(out[0], want, rtol=0, atol=1e-12)


def test_append_rejects_bad_block_and_position(oracle_mod):
    hkv, d, nb = 1, 64, 4
    kp = _empty_pool(oracle_mod, nb, hkv, d, F32)
    vp = _empty_pool(oracle_mod, nb, hkv, d, F32)
    kn = np.ones((1, hkv, d), np.float32)
    bad = np.array([[7]], np.int32)
    assert oracle_mod.append_kv(kp, vp, kn, kn, bad, np.array([0], np.int32),
                                np.array([0, 1], np.int32), num_kv_heads=hkv, head_dim=d,
                                num_blocks=nb, dtype=F32) == 2
    ok = np.array([[1]], np.int32)
    assert oracle_mod.append_kv(kp, vp, kn, kn, ok, np.array([16], np.int32),
                                np.array([0, 1], np.int32), num_kv_heads=hkv, head_dim=d,
                                num_blocks=nb, dtype=F32) == 3
    assert np.all(kp == 0) and np.all(vp == 0)


def test_copy_block_copies_every_byte_of_both_pools(oracle_mod):
    hkv, d, nb = 3, 64, 5
    rng = np.random.default_rng(4)
    kp = rng.integers(0, 65535, size=oracle_mod.pool_shape(nb, hkv, d, BF16), dtype=np.uint16)
    vp = rng.integers(0, 65535, size=oracle_mod.pool_shape(nb, hkv, d, BF16), dtype=np.uint16)
    k0, v0 = kp.copy(), vp.copy()
    assert oracle_mod.copy_block(kp, vp, [[1, 3], [4, 0]], num_blocks=nb, num_kv_heads=hkv,
                                 head_dim=d, dtype=BF16) == 0
    assert np.array_equal(kp[3], k0[1]) and np.array_equal(vp[3], v0[1])
    assert np.array_equal(kp[0], k0[4]) and np.array_equal(vp[0], v0[4])
    for b in (1, 2, 4):
        assert np.array_equal(kp[b], k0[b]) and np.array_equal(vp[b], v0[b])
    assert oracle_mod.copy_block(kp, vp, [[1, 9]], num_blocks=nb, num_kv_heads=hkv,
                                 head_dim=d, dtype=BF16) == 2

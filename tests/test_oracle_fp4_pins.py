"""Pins of the oracle's block-scaled FP4 (MXFP4) cache (no GPU needed).

The format is the microscaling one that Slipstream's "Companion work" points to
(qgemm-mx, a block-scaled FP4 kernel for the same bandwidth-bound decode):
E2M1 values, one power-of-two E8M0 scale per 32 values along head_dim.

Pins, each independent of the oracle's own code:
  * E2M1 rounding against hand-worked cases (tests/golden/e2m1_rounding.json)
    and against a brute-force nearest-value search written here;
  * the 16-code value table and the code <-> value bijection;
  * the shared scale against hand-worked cases and torch's float8_e8m0fnu
    encoding of exact powers of two (a library routine);
  * the quantised append: scales, the error bound of each stored value, and
    stored values equal to a quantiser written here with numpy;
  * the record layout at hand-computed byte and nibble positions;
  * decode over the quantised cache against torch float64 SDPA on the values
    this test dequantises itself, and the zero-query / one-token closed forms.
"""
import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _golden():
    return json.load(open(os.path.join(GOLDEN, "e2m1_rounding.json")))


def _nearest_code(x: float) -> int:
    """Brute force: the E2M1 magnitude nearest |x|, a tie going to the code whose
    mantissa bit (its lowest bit) is 0; beyond 6, code 7."""
    m = abs(x)
    d = np.abs(E2M1 - m)
    best = np.flatnonzero(d == d.min())
    code = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
    return code | (8 if np.signbit(x) else 0)


def test_e2m1_value_table(oracle_mod):
    vals = [float(v) for v in _golden()["values"]]
    for code in range(16):
        got = oracle_mod.e2m1_to_double(code)
        assert got == vals[code] and np.signbit(got) == np.signbit(vals[code]), code


def test_e2m1_hand_worked_cases(oracle_mod):
    for c in _golden()["cases"]:
        assert oracle_mod.f32_to_e2m1(c["x"]) == int(c["code"], 16), c
        assert oracle_mod.f32_to_e2m1(-c["x"]) == int(c["code"], 16) | 8, c


def test_e2m1_matches_brute_force_nearest(oracle_mod):
    rng = np.random.default_rng(11)
    xs = np.concatenate([rng.normal(0, 2.5, 4000), rng.uniform(-8, 8, 4000),
                         np.arange(-7.0, 7.01, 0.25), np.arange(-2.0, 2.0, 0.125)])
    for x in xs.astype(np.float32):
        assert oracle_mod.f32_to_e2m1(float(x)) == _nearest_code(float(x)), float(x)


def test_e2m1_codes_and_values_are_a_bijection(oracle_mod):
    seen = {}
    for code in range(16):
        v = oracle_mod.e2m1_to_double(code)
        back = oracle_mod.f32_to_e2m1(v)
        assert back == code, (code, v, back)
        if code & 7:
            assert v not in seen
            seen[v] = code


def test_mx_scale_hand_worked_and_library(oracle_mod):
    for c in _golden()["scales"]:
        assert oracle_mod.mx_scale_code(c["amax"]) == c["code"], c
    # amax = 2^k: the scale is 2^(k - 2); torch encodes exact powers of two in E8M0
    for k in range(-100, 100, 7):
        want = torch.tensor([2.0 ** (k - 2)]).to(torch.float8_e8m0fnu).view(torch.uint8).item()
        assert oracle_mod.mx_scale_code(2.0 ** k) == want, k
        # every amax in [2^k, 2^(k+1)) shares the code, and amax / scale lands in [4, 8)
        for f in (1.0, 1.3, 1.99):
            code = oracle_mod.mx_scale_code(f * 2.0 ** k)
            assert code == want
            assert 4.0 <= f * 2.0 ** k / 2.0 ** (code - 127) < 8.0


def _bf16(x):
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _quantise_here(row):
    """This test's own MXFP4 quantiser of one row (float64 values of bf16 numbers):
    per 32-value block the scale 2^(floor(log2 amax) - 2), then nearest E2M1 value
    (brute force, ties to the even code), saturating at 6."""
    out = np.zeros_like(row)
    for b in range(0, row.size, 32):
        blk = row[b:b + 32]
        amax = np.abs(blk).max()
        if amax == 0:
            continue
        X = 2.0 ** (np.floor(np.log2(amax)) - 2)
        for i, v in enumerate(blk):
            c = _nearest_code(v / X)
            out[b + i] = (-1 if c & 8 else 1) * E2M1[c & 7] * X
    return out


def _append(o, k, v, table, D, Hkv, nb=8):
    kp = np.zeros(o.fp4_pool_shape(nb, Hkv, D), np.uint8)
    vp = np.zeros(o.fp4_pool_shape(nb, Hkv, D), np.uint8)
    n = k.shape[0]
    assert o.append_kv_fp4(kp, vp, k, v, np.array([table], np.int32), np.array([0], np.int32),
                           np.array([0, n], np.int32), num_kv_heads=Hkv, head_dim=D,
                           num_blocks=nb) == 0
    return kp, vp


def test_quantised_append_scales_values_and_error_bound(oracle_mod):
    D, Hkv = 64, 2
    g = torch.Generator().manual_seed(13)
    k = _bf16(torch.randn(20, Hkv, D, generator=g) * torch.tensor([1.0, 40.0]).view(1, 2, 1))
    v = _bf16(torch.randn(20, Hkv, D, generator=g) * 0.01)
    table = [5, 2]
    kp, vp = _append(oracle_mod, k, v, table, D, Hkv)
    recs = {}
    for t in range(20):
        blk, slot = table[t // 16], t % 16
        for h in range(Hkv):
            if (blk, h) not in recs:
                recs[(blk, h)] = oracle_mod.fp4_record_values(kp[blk, h], vp[blk, h], D)
            kv, vv = recs[(blk, h)]
            for rows, vals, pool in ((k, kv, kp), (v, vv, vp)):
                x = _f(rows[t, h])
                np.testing.assert_array_equal(vals[slot], _quantise_here(x))
                for b in range(D // 32):
                    amax = np.abs(x[32 * b:32 * b + 32]).max()
                    sc = pool[blk, h, 8 * D + slot * (D // 32) + b]
                    assert sc == oracle_mod.mx_scale_code(amax)
                    X = 2.0 ** (int(sc) - 127)
                    y = np.abs(x[32 * b:32 * b + 32]) / X
                    step = np.where(y < 2, 0.5, np.where(y < 4, 1.0, 2.0))
                    bound = np.maximum(step / 2, y - 6.0) * X
                    assert np.all(np.abs(vals[slot, 32 * b:32 * b + 32] - x[32 * b:32 * b + 32]) <= bound)


def test_record_layout_positions(oracle_mod):
    """D = 64, one token at slot 5 whose every value is 0 except dim 19 (value 6 after
    scaling: code 7).  Worked by hand from the documented layout:
      K: dim 19 -> ks = 1, half = 0, c = 1: byte 5 * 32 + 1 * 8 + 1 * 2 + 0 = 170, high
         nibble (odd dim); the scale byte of block 0 at 8 * 64 + 5 * 2 = 522.
      V: dim 19 -> mi = 1, dh = 0, r = 3; slot 5 -> half = 0, c = 2:
         byte ((3 * 4 + 2) * 4 + 1) * 4 + 0 * 2 + 0 = 228, high nibble (odd slot)."""
    D, Hkv = 64, 1
    row = np.zeros((6, Hkv, D), np.float32)
    row[5, 0, 19] = 6.0                     # amax 6: scale 2^0 = code 127, value code 7
    bits = _bf16(torch.from_numpy(row))
    kp, vp = _append(oracle_mod, bits, bits, [3], D, Hkv, nb=4)
    krec, vrec = kp[3, 0], vp[3, 0]
    assert krec[170] == 0x70 and vrec[228] == 0x70
    assert krec[8 * D + 5 * 2] == 127 and vrec[8 * D + 5 * 2] == 127
    assert krec[8 * D + 5 * 2 + 1] == 0      # block 1 of slot 5 is all zero: code 0
    nonzero_k = set(np.flatnonzero(krec[:8 * D]).tolist())
    nonzero_v = set(np.flatnonzero(vrec[:8 * D]).tolist())
    assert nonzero_k == {170} and nonzero_v == {228}


def test_fp4_decode_closed_forms_and_library_routine(oracle_mod):
    D, Hkv, Hq = 128, 2, 8
    g = torch.Generator().manual_seed(14)
    L = 37
    k = _bf16(torch.randn(L, Hkv, D, generator=g))
    v = _bf16(torch.randn(L, Hkv, D, generator=g) * 3)
    table = [6, 1, 3]
    kp, vp = _append(oracle_mod, k, v, table, D, Hkv)
    tables = np.array([table], np.int32)
    K = np.stack([[_quantise_here(_f(k[t, h])) for h in range(Hkv)] for t in range(L)])
    V = np.stack([[_quantise_here(_f(v[t, h])) for h in range(Hkv)] for t in range(L)])
    pairs = [(0, h) for h in range(Hq)]
    kw = dict(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, num_blocks=8, scale=0.125)
    q0 = np.zeros((1, Hq, D), np.uint16)
    out = oracle_mod.decode_fp4_pairs(pairs, q0, kp, vp, tables, np.array([L], np.int32), **kw)
    for h in range(Hq):                       # q = 0: the mean of the stored values
        np.testing.assert_allclose(out[h], V[:, h // 4].mean(0), rtol=0, atol=1e-13)
    one = oracle_mod.decode_fp4_pairs(pairs, _bf16(torch.randn(1, Hq, D, generator=g)), kp, vp,
                                      tables, np.array([1], np.int32), **kw)
    for h in range(Hq):                       # one token: its stored value row
        np.testing.assert_array_equal(one[h], V[0, h // 4])
    q = _bf16(torch.randn(1, Hq, D, generator=g))
    out = oracle_mod.decode_fp4_pairs(pairs, q, kp, vp, tables, np.array([L], np.int32), **kw)
    Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(4, 0)
    Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(4, 0)
    Q = torch.from_numpy(_f(q[0])).unsqueeze(1)
    ref = torch.nn.functional.scaled_dot_product_attention(Q, Kt, Vt, scale=0.125)[:, 0]
    np.testing.assert_allclose(out, ref.numpy(), rtol=0, atol=1e-12)

"""Pins of the oracle's FP8 (E4M3) cache (no GPU needed).

E4M3 rounding against hand-worked cases and torch's float8_e4m3fn conversion
(a library routine); the code <-> value map is a bijection on finite codes; the
quantised append stores per-slot scales amax / 448 and codes whose dequantised
values are within half a step of the input; decode over the quantised cache
reduces to the plain oracle on the dequantised rows and to the closed forms.
"""
import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e4m3_hand_worked_cases(oracle_mod):
    for c in json.load(open(os.path.join(GOLDEN, "e4m3_rounding.json")))["cases"]:
        assert oracle_mod.f32_to_e4m3(c["x"]) == int(c["code"], 16), c
        assert oracle_mod.f32_to_e4m3(-c["x"]) == int(c["code"], 16) ^ 0x80, c


def test_e4m3_matches_torch_in_range(oracle_mod):
    g = torch.Generator().manual_seed(2)
    x = torch.randn(20000, generator=g) * 10 ** torch.empty(20000).uniform_(-4, 2.3, generator=g)
    x = x[x.abs() < 440]
    want = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_mod.f32_to_e4m3(float(v)) for v in x.numpy()], np.uint8)
    assert np.array_equal(got, want)


def test_e4m3_codes_and_values_are_a_bijection(oracle_mod):
    for code in range(256):
        v = oracle_mod.e4m3_to_double(code)
        if code & 0x7F == 0x7F:
            assert math.isnan(v)
            continue
        back = oracle_mod.f32_to_e4m3(v)
        assert back == code or (v == 0.0 and back & 0x7F == 0), (hex(code), v, hex(back))
    assert oracle_mod.e4m3_to_double(0x7E) == 448.0
    assert oracle_mod.e4m3_to_double(0x01) == 2.0 ** -9


def _bf16(x):
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _append_one(o, rows_k, rows_v, table, D, nb=8, Hkv=2):
    kp = np.zeros(o.fp8_pool_shape(nb, Hkv, D), np.uint8)
    vp = np.zeros(o.fp8_pool_shape(nb, Hkv, D), np.uint8)
    n = rows_k.shape[0]
    assert o.append_kv_fp8(kp, vp, rows_k, rows_v, np.array([table], np.int32),
                           np.array([0], np.int32), np.array([0, n], np.int32),
                           num_kv_heads=Hkv, head_dim=D, num_blocks=nb) == 0
    return kp, vp


def test_quantised_append_scales_and_codes(oracle_mod):
    D, Hkv = 64, 2
    g = torch.Generator().manual_seed(3)
    k = _bf16(torch.randn(20, Hkv, D, generator=g) * 3)
    v = _bf16(torch.randn(20, Hkv, D, generator=g))
    kp, vp = _append_one(oracle_mod, k, v, [5, 2], D)
    for t in range(20):
        blk, slot = [5, 2][t // 16], t % 16
        for h in range(Hkv):
            rec = kp[blk, h]
            scale = rec[16 * D + 4 * slot:16 * D + 4 * slot + 4].view(np.float32)[0]
            row = _f(k[t, h])
            assert scale == np.float32(np.float32(np.abs(row).max()) / np.float32(448.0))
            codes = np.array([rec[((d // 16) * 16 + slot) * 16 + d % 16] for d in range(D)])
            deq = np.array([oracle_mod.e4m3_to_double(c) for c in codes]) * float(scale)
            # within half a step of E4M3 at each value's magnitude (relative 2^-4), or the
            # subnormal spacing near zero
            err = np.abs(deq - row)
            assert np.all(err <= np.maximum(np.abs(row) * 2.0 ** -4, float(scale) * 2.0 ** -10) + 1e-30)
            # V codes are stored one 16-byte row per dim
            vrec = vp[blk, h]
            vscale = vrec[16 * D + 4 * slot:16 * D + 4 * slot + 4].view(np.float32)[0]
            vdeq = np.array([oracle_mod.e4m3_to_double(vrec[d * 16 + slot]) for d in range(D)]) * float(vscale)
            assert np.abs(vdeq - _f(v[t, h])).max() <= np.abs(_f(v[t, h])).max() * 2.0 ** -4


def test_fp8_decode_closed_forms_and_library_routine(oracle_mod):
    D, Hkv, Hq = 64, 2, 8
    g = torch.Generator().manual_seed(4)
    L = 37
    k = _bf16(torch.randn(L, Hkv, D, generator=g))
    v = _bf16(torch.randn(L, Hkv, D, generator=g))
    table = [6, 1, 3]
    kp, vp = _append_one(oracle_mod, k, v, table, D)
    tables = np.array([table], np.int32)

    def deq_rows(pool, layout_v):
        rows = np.zeros((L, Hkv, D))
        for t in range(L):
            blk, slot = table[t // 16], t % 16
            for h in range(Hkv):
                rec = pool[blk, h]
                sc = float(rec[16 * D + 4 * slot:16 * D + 4 * slot + 4].view(np.float32)[0])
                for d in range(D):
                    c = rec[d * 16 + slot] if layout_v else rec[((d // 16) * 16 + slot) * 16 + d % 16]
                    rows[t, h, d] = oracle_mod.e4m3_to_double(c) * sc
        return rows

    K, V = deq_rows(kp, False), deq_rows(vp, True)
    q0 = np.zeros((1, Hq, D), np.uint16)
    pairs = [(0, h) for h in range(Hq)]
    out = oracle_mod.decode_fp8_pairs(pairs, q0, kp, vp, tables, np.array([L], np.int32),
                                      num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, num_blocks=8,
                                      scale=0.125)
    for h in range(Hq):                       # q = 0: mean of the dequantised values
        np.testing.assert_allclose(out[h], V[:, h // 4].mean(0), rtol=0, atol=1e-13)
    q = _bf16(torch.randn(1, Hq, D, generator=g))
    out = oracle_mod.decode_fp8_pairs(pairs, q, kp, vp, tables, np.array([L], np.int32),
                                      num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, num_blocks=8,
                                      scale=0.125)
    Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(4, 0)
    Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(4, 0)
    Q = torch.from_numpy(_f(q[0])).unsqueeze(1)
    ref = torch.nn.functional.scaled_dot_product_attention(Q, Kt, Vt, scale=0.125)[:, 0]
    np.testing.assert_allclose(out, ref.numpy(), rtol=0, atol=1e-12)

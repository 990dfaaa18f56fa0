"""Python face of the CPU oracle (``pa_oracle.c``).

TEST INFRASTRUCTURE, NOT PRODUCT CODE: only the test suite, the smoke check
and the benchmark's CPU-baseline leg may import this module.  It compiles the
plain C oracle with gcc on first use and marshals numpy arrays into it.

Element types follow the C file: 0 = fp32 (numpy float32), 1 = bf16 (raw
16-bit patterns as numpy uint16).  Pools use the layout documented at the top
of ``pa_oracle.c``: ``[num_blocks][Hkv][D / X][16][X]`` with ``X = 16 / elem_bytes``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "libpa_oracle.so")

F32, BF16 = 0, 1
BLOCK = 16

_lib = None


def build(force: bool = False) -> str:
    """Compile ``pa_oracle.c`` into ``libpa_oracle.so`` next to it.

    ``-ffp-contract=off`` keeps every multiply and add separately rounded so
    the oracle gives the same doubles on x86-64 and on aarch64."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        compile_source(_SRC, tmp)
        os.replace(tmp, _LIB)
    return _LIB


def _bind(L: ctypes.CDLL) -> ctypes.CDLL:
    p = ctypes.c_void_p
    i = ctypes.c_int
    L.oracle_decode.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, ctypes.c_double, i]
    L.oracle_decode_pairs.argtypes = [p, p, i, p, p, p, p, p, i, i, i, i, i, ctypes.c_double, i]
    L.oracle_decode_one.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, i, ctypes.c_double, i]
    L.oracle_decode_contig.argtypes = [p, p, p, p, i, i, i, i, ctypes.c_double, i]
    L.oracle_append_kv.argtypes = [p, p, p, p, p, i, p, p, i, i, i, i, i]
    L.oracle_copy_block.argtypes = [p, p, p, i, i, i, i, i]
    L.oracle_round_out.argtypes = [p, p, ctypes.c_int64, i]
    L.oracle_double_to_bf16.argtypes = [ctypes.c_double]
    L.oracle_double_to_bf16.restype = ctypes.c_uint16
    L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    L.oracle_bf16_to_double.restype = ctypes.c_double
    L.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
    L.oracle_f32_to_e4m3.restype = ctypes.c_uint8
    L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_to_double.restype = ctypes.c_double
    L.oracle_append_kv_fp8.argtypes = [p, p, p, p, p, i, p, p, i, i, i, i]
    L.oracle_decode_fp8_pairs.argtypes = [p, p, i, p, p, p, p, p, i, i, i, i, i, ctypes.c_double]
    L.oracle_e2m1_to_double.argtypes = [ctypes.c_uint8]
    L.oracle_e2m1_to_double.restype = ctypes.c_double
    L.oracle_f32_to_e2m1.argtypes = [ctypes.c_float]
    L.oracle_f32_to_e2m1.restype = ctypes.c_uint8
    L.oracle_mx_scale_code.argtypes = [ctypes.c_float]
    L.oracle_mx_scale_code.restype = ctypes.c_uint8
    L.oracle_append_kv_fp4.argtypes = [p, p, p, p, p, i, p, p, i, i, i, i]
    L.oracle_decode_fp4_pairs.argtypes = [p, p, i, p, p, p, p, p, i, i, i, i, i, ctypes.c_double]
    L.oracle_fp4_record_values.argtypes = [p, p, p, p, i]
    return L


def compile_source(src: str, out_path: str) -> str:
    """Compile a C source file with the oracle's flags into a shared library."""
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", out_path, src, "-lm"])
    return out_path


class use_library:
    """Context manager: route every call of this module to another build of the oracle
    (used by the tests that plant mistakes in a copy of the source)."""

    def __init__(self, path: str):
        self.L = _bind(ctypes.CDLL(path))

    def __enter__(self):
        global _lib
        self.prev = _lib
        _lib = self.L
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.prev
        return False


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _np(a, dtype=None):
    """Accept numpy arrays or CPU torch tensors (bf16 tensors become uint16 bits)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            t = a.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                a = t.view(torch.int16).numpy().view(np.uint16)
            else:
                a = t.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if dtype is not None and a.dtype != dtype:
        raise TypeError(f"oracle expects {dtype}, got {a.dtype}")
    return a


def _elem_dtype(dtype: int):
    return np.uint16 if dtype == BF16 else np.float32


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def decode(q, k_pool, v_pool, block_tables, context_lens, *, num_q_heads, num_kv_heads,
           head_dim, num_blocks, scale, dtype) -> np.ndarray:
    """Dense-softmax decode attention for every (sequence, query head): float64 [S][Hq][D]."""
    et = _elem_dtype(dtype)
    q, k_pool, v_pool = _np(q, et), _np(k_pool, et), _np(v_pool, et)
    tables = _np(block_tables, np.int32)
    lens = _np(context_lens, np.int32)
    S = lens.shape[0]
    out = np.zeros((S, num_q_heads, head_dim), np.float64)
    rc = lib().oracle_decode(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(tables),
                             _ptr(lens), S, num_q_heads, num_kv_heads, head_dim,
                             tables.shape[1] if tables.ndim == 2 else 0, num_blocks,
                             float(scale), dtype)
    if rc != 0:
        raise ValueError(f"oracle_decode failed with code {rc}")
    return out


def decode_pairs(pairs, q, k_pool, v_pool, block_tables, context_lens, *, num_q_heads,
                 num_kv_heads, head_dim, num_blocks, scale, dtype) -> np.ndarray:
    """Decode attention for chosen (sequence, query head) pairs: float64 [n][D]."""
    et = _elem_dtype(dtype)
    q, k_pool, v_pool = _np(q, et), _np(k_pool, et), _np(v_pool, et)
    tables = _np(block_tables, np.int32)
    lens = _np(context_lens, np.int32)
    pairs = np.ascontiguousarray(np.asarray(pairs, np.int32).reshape(-1, 2))
    out = np.zeros((pairs.shape[0], head_dim), np.float64)
    rc = lib().oracle_decode_pairs(_ptr(out), _ptr(pairs), pairs.shape[0], _ptr(q), _ptr(k_pool),
                                   _ptr(v_pool), _ptr(tables), _ptr(lens), num_q_heads,
                                   num_kv_heads, head_dim, tables.shape[1], num_blocks,
                                   float(scale), dtype)
    if rc != 0:
        raise ValueError(f"oracle_decode_pairs failed with code {rc}")
    return out


def decode_contig(q_row, k_rows, v_rows, kv_head, *, num_kv_heads, head_dim, scale,
                  dtype) -> np.ndarray:
    """One query row against contiguous context rows ``[L][Hkv][D]`` (no paging):
    float64 [D].  The "contiguous" side of paged == contiguous."""
    et = _elem_dtype(dtype)
    q_row, k_rows, v_rows = _np(q_row, et), _np(k_rows, et), _np(v_rows, et)
    L = k_rows.shape[0]
    out = np.zeros(head_dim, np.float64)
    rc = lib().oracle_decode_contig(_ptr(out), _ptr(q_row), _ptr(k_rows), _ptr(v_rows), L,
                                    kv_head, num_kv_heads, head_dim, float(scale), dtype)
    if rc != 0:
        raise ValueError(f"oracle_decode_contig failed with code {rc}")
    return out


def append_kv(k_pool, v_pool, k_new, v_new, block_tables, start_pos, cu_new_tokens, *,
              num_kv_heads, head_dim, num_blocks, dtype) -> int:
    """Write new tokens into numpy pools in place (byte copy).  Returns the C return code
    (0 = ok, 2 = a table entry out of range, 3 = a position beyond the table)."""
    et = _elem_dtype(dtype)
    for p in (k_pool, v_pool):
        if not (isinstance(p, np.ndarray) and p.dtype == et and p.flags.c_contiguous):
            raise TypeError("pools must be C-contiguous numpy arrays of the element type")
    k_new, v_new = _np(k_new, et), _np(v_new, et)
    tables = _np(block_tables, np.int32)
    start = _np(start_pos, np.int32)
    cu = _np(cu_new_tokens, np.int32)
    return lib().oracle_append_kv(_ptr(k_pool), _ptr(v_pool), _ptr(k_new), _ptr(v_new),
                                  _ptr(tables), tables.shape[1], _ptr(start), _ptr(cu),
                                  start.shape[0], num_blocks, num_kv_heads, head_dim, dtype)


def copy_block(k_pool, v_pool, pairs, *, num_blocks, num_kv_heads, head_dim, dtype) -> int:
    """Copy whole blocks src -> dst in numpy pools in place."""
    pairs = np.ascontiguousarray(np.asarray(pairs, np.int32).reshape(-1, 2))
    return lib().oracle_copy_block(_ptr(k_pool), _ptr(v_pool), _ptr(pairs), pairs.shape[0],
                                   num_blocks, num_kv_heads, head_dim, dtype)


def round_out(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round float64 results once to the output element type (RNE)."""
    x = np.ascontiguousarray(x, np.float64)
    out = np.empty(x.shape, _elem_dtype(dtype))
    lib().oracle_round_out(_ptr(x), _ptr(out), x.size, dtype)
    return out


def double_to_bf16(x: float) -> int:
    return int(lib().oracle_double_to_bf16(float(x)))


def bf16_to_double(b: int) -> float:
    return float(lib().oracle_bf16_to_double(int(b)))


# ---- FP8 (E4M3) cache with per-slot scales --------------------------------------

def f32_to_e4m3(x: float) -> int:
    return int(lib().oracle_f32_to_e4m3(float(x)))


def e4m3_to_double(code: int) -> float:
    return float(lib().oracle_e4m3_to_double(int(code)))


def fp8_pool_shape(num_blocks: int, num_kv_heads: int, head_dim: int):
    """One FP8 pool: per (block, kv head) a record of 16*D code bytes + 16 fp32 scales."""
    return (num_blocks, num_kv_heads, 16 * head_dim + 64)


def append_kv_fp8(k_pool, v_pool, k_new, v_new, block_tables, start_pos, cu_new_tokens, *,
                  num_kv_heads, head_dim, num_blocks) -> int:
    """Quantise bf16 rows (uint16 bits or torch bf16) into numpy uint8 FP8 pools in place."""
    for p in (k_pool, v_pool):
        if not (isinstance(p, np.ndarray) and p.dtype == np.uint8 and p.flags.c_contiguous):
            raise TypeError("FP8 pools must be C-contiguous numpy uint8 arrays")
    k_new, v_new = _np(k_new, np.uint16), _np(v_new, np.uint16)
    tables = _np(block_tables, np.int32)
    start = _np(start_pos, np.int32)
    cu = _np(cu_new_tokens, np.int32)
    return lib().oracle_append_kv_fp8(_ptr(k_pool), _ptr(v_pool), _ptr(k_new), _ptr(v_new),
                                      _ptr(tables), tables.shape[1], _ptr(start), _ptr(cu),
                                      start.shape[0], num_blocks, num_kv_heads, head_dim)


def decode_fp8_pairs(pairs, q, k_pool, v_pool, block_tables, context_lens, *, num_q_heads,
                     num_kv_heads, head_dim, num_blocks, scale) -> np.ndarray:
    """Decode attention over FP8 pools for chosen (sequence, query head) pairs: float64 [n][D]."""
    q = _np(q, np.uint16)
    k_pool, v_pool = _np(k_pool, np.uint8), _np(v_pool, np.uint8)
    tables = _np(block_tables, np.int32)
    lens = _np(context_lens, np.int32)
    pairs = np.ascontiguousarray(np.asarray(pairs, np.int32).reshape(-1, 2))
    out = np.zeros((pairs.shape[0], head_dim), np.float64)
    rc = lib().oracle_decode_fp8_pairs(_ptr(out), _ptr(pairs), pairs.shape[0], _ptr(q),
                                       _ptr(k_pool), _ptr(v_pool), _ptr(tables), _ptr(lens),
                                       num_q_heads, num_kv_heads, head_dim, tables.shape[1],
                                       num_blocks, float(scale))
    if rc != 0:
        raise ValueError(f"oracle_decode_fp8_pairs failed with code {rc}")
    return out


def pool_shape(num_blocks: int, num_kv_heads: int, head_dim: int, dtype: int):
    """Shape of one pool as a numpy array in the documented layout."""
    x = 8 if dtype == BF16 else 4
    return (num_blocks, num_kv_heads, head_dim // x, BLOCK, x)


# ---- block-scaled FP4 (MXFP4) cache ---------------------------------------------

def e2m1_to_double(code: int) -> float:
    return float(lib().oracle_e2m1_to_double(int(code)))


def f32_to_e2m1(x: float) -> int:
    return int(lib().oracle_f32_to_e2m1(float(x)))


def mx_scale_code(amax: float) -> int:
    """E8M0 code of the shared scale of a 32-value block whose largest magnitude is amax."""
    return int(lib().oracle_mx_scale_code(float(amax)))


def fp4_record_bytes(head_dim: int) -> int:
    return 8 * head_dim + head_dim // 2


def fp4_pool_shape(num_blocks: int, num_kv_heads: int, head_dim: int):
    """One MXFP4 pool: per (block, kv head) 8*D code bytes + D/2 scale bytes."""
    return (num_blocks, num_kv_heads, fp4_record_bytes(head_dim))


def append_kv_fp4(k_pool, v_pool, k_new, v_new, block_tables, start_pos, cu_new_tokens, *,
                  num_kv_heads, head_dim, num_blocks) -> int:
    """Quantise bf16 rows (uint16 bits or torch bf16) into numpy uint8 MXFP4 pools in place."""
    for p in (k_pool, v_pool):
        if not (isinstance(p, np.ndarray) and p.dtype == np.uint8 and p.flags.c_contiguous):
            raise TypeError("FP4 pools must be C-contiguous numpy uint8 arrays")
    k_new, v_new = _np(k_new, np.uint16), _np(v_new, np.uint16)
    tables = _np(block_tables, np.int32)
    start = _np(start_pos, np.int32)
    cu = _np(cu_new_tokens, np.int32)
    return lib().oracle_append_kv_fp4(_ptr(k_pool), _ptr(v_pool), _ptr(k_new), _ptr(v_new),
                                      _ptr(tables), tables.shape[1], _ptr(start), _ptr(cu),
                                      start.shape[0], num_blocks, num_kv_heads, head_dim)


def decode_fp4_pairs(pairs, q, k_pool, v_pool, block_tables, context_lens, *, num_q_heads,
                     num_kv_heads, head_dim, num_blocks, scale) -> np.ndarray:
    """Decode attention over MXFP4 pools for chosen (sequence, query head) pairs: float64 [n][D]."""
    q = _np(q, np.uint16)
    k_pool, v_pool = _np(k_pool, np.uint8), _np(v_pool, np.uint8)
    tables = _np(block_tables, np.int32)
    lens = _np(context_lens, np.int32)
    pairs = np.ascontiguousarray(np.asarray(pairs, np.int32).reshape(-1, 2))
    out = np.zeros((pairs.shape[0], head_dim), np.float64)
    rc = lib().oracle_decode_fp4_pairs(_ptr(out), _ptr(pairs), pairs.shape[0], _ptr(q),
                                       _ptr(k_pool), _ptr(v_pool), _ptr(tables), _ptr(lens),
                                       num_q_heads, num_kv_heads, head_dim, tables.shape[1],
                                       num_blocks, float(scale))
    if rc != 0:
        raise ValueError(f"oracle_decode_fp4_pairs failed with code {rc}")
    return out


def fp4_record_values(k_rec, v_rec, head_dim: int):
    """Dequantised K and V rows ([16][D] float64 each) of one (block, kv head) record."""
    k_rec, v_rec = _np(k_rec, np.uint8), _np(v_rec, np.uint8)
    ko = np.zeros((BLOCK, head_dim), np.float64)
    vo = np.zeros((BLOCK, head_dim), np.float64)
    rc = lib().oracle_fp4_record_values(_ptr(ko), _ptr(vo), _ptr(k_rec), _ptr(v_rec), head_dim)
    if rc != 0:
        raise ValueError(f"oracle_fp4_record_values failed with code {rc}")
    return ko, vo

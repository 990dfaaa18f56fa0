"""ctypes binding of ``libpaged_kv.so`` (the C ABI declared in ``include/pa.h``).

Argument marshalling only: tensors become device pointers and sizes, the current
torch stream becomes the ``void* stream`` argument, and a non-OK status becomes
an exception.  Every step of the computation runs in the library's kernels;
there is no fallback, and the import fails loudly if the library was not built.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpaged_kv.so")

PA_OK = 0
PA_F32, PA_BF16 = 0, 1
BLOCK_SIZE = 16
PARTITION_TOKENS = 512          # split-KV partition of pa_decode_attention at head_dim 128


def partition_tokens(head_dim: int) -> int:
    """Tokens per split-KV partition of pa_decode_attention (head_dim 64: twice as many)."""
    return 2 * PARTITION_TOKENS if head_dim == 64 else PARTITION_TOKENS

DEV_ERR_BAD_BLOCK = 1
DEV_ERR_BAD_POS = 2
DEV_ERR_HINT = 4
DEV_ERR_BAD_CU = 8
DEV_ERR_TIMEOUT = 16
DEV_ERR_BAD_PAIR = 32
DEV_ERR_BAD_PREFIX = 64

EXPORTED = [
    "pa_status_string", "pa_abi_version", "pa_append_kv", "pa_copy_block",
    "pa_decode_workspace_size", "pa_decode_attention", "pa_append_decode_attention",
    "pa_decode_attention_shared_prefix", "pa_append_decode_attention_shared_prefix",
    "pa_decode_attention_noalloc", "pa_append_kv_fp8", "pa_decode_attention_fp8",
    "pa_append_decode_attention_fp8",
    "pa_append_kv_fp4", "pa_decode_attention_fp4",
    "pa_prefill_attention", "pa_bm_create", "pa_bm_destroy",
    "pa_bm_add_seq", "pa_bm_fork", "pa_bm_free_seq", "pa_bm_blocks_needed",
    "pa_bm_prepare_append", "pa_bm_block_table", "pa_bm_block_tables", "pa_bm_seq_len",
    "pa_bm_refcount", "pa_bm_stats",
]


class PagedKVError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {status})")
        self.status = status


class BmStats(ctypes.Structure):
    _fields_ = [("physical_blocks", ctypes.c_int64), ("free_blocks", ctypes.c_int64),
                ("logical_tokens", ctypes.c_int64), ("num_seqs", ctypes.c_int64)]


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"{_LIB_PATH} is missing: build it with "
                          "`python -m paged_kv_cache_207_gb300.build` (nvcc, sm_103a)")
    L = ctypes.CDLL(_LIB_PATH)
    p, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    ip = ctypes.POINTER(ctypes.c_int32)
    L.pa_status_string.argtypes = [ctypes.c_int]
    L.pa_status_string.restype = ctypes.c_char_p
    L.pa_abi_version.restype = i32
    L.pa_append_kv.argtypes = [p, p, p, p, p, i32, p, p, i32, i32, i32, i32, i32, ctypes.c_int, p, p]
    L.pa_append_kv.restype = ctypes.c_int
    L.pa_copy_block.argtypes = [p, p, p, i32, i32, i32, i32, ctypes.c_int, p, p]
    L.pa_copy_block.restype = ctypes.c_int
    L.pa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    L.pa_decode_workspace_size.restype = sz
    L.pa_decode_attention.argtypes = [p, p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32,
                                      ctypes.c_float, ctypes.c_int, p, sz, p, p]
    L.pa_decode_attention.restype = ctypes.c_int
    L.pa_append_decode_attention.argtypes = [p, p, p, p, p, p, p, p, i32, i32, i32, i32, i32, i32,
                                             i32, ctypes.c_float, ctypes.c_int, p, sz, p, p]
    L.pa_append_decode_attention.restype = ctypes.c_int
    L.pa_decode_attention_shared_prefix.argtypes = [p, p, p, p, p, p, i32, i32, i32, i32, i32, i32,
                                                    i32, ctypes.c_float, ctypes.c_int, i32, p, sz,
                                                    p, p]
    L.pa_decode_attention_shared_prefix.restype = ctypes.c_int
    L.pa_append_decode_attention_shared_prefix.argtypes = [p, p, p, p, p, p, p, p, i32, i32, i32,
                                                           i32, i32, i32, i32, ctypes.c_float,
                                                           ctypes.c_int, i32, p, sz, p, p]
    L.pa_append_decode_attention_shared_prefix.restype = ctypes.c_int
    L.pa_append_kv_fp8.argtypes = [p, p, p, p, p, i32, p, p, i32, i32, i32, i32, i32, p, p]
    L.pa_append_kv_fp8.restype = ctypes.c_int
    L.pa_decode_attention_fp8.argtypes = [p, p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32,
                                          ctypes.c_float, p, sz, p, p]
    L.pa_decode_attention_fp8.restype = ctypes.c_int
    L.pa_append_decode_attention_fp8.argtypes = [p, p, p, p, p, p, p, p, i32, i32, i32, i32, i32,
                                                 i32, i32, ctypes.c_float, p, sz, p, p]
    L.pa_append_decode_attention_fp8.restype = ctypes.c_int
    L.pa_append_kv_fp4.argtypes = [p, p, p, p, p, i32, p, p, i32, i32, i32, i32, i32, p, p]
    L.pa_append_kv_fp4.restype = ctypes.c_int
    L.pa_decode_attention_fp4.argtypes = [p, p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32,
                                          ctypes.c_float, p, sz, p, p]
    L.pa_decode_attention_fp4.restype = ctypes.c_int
    L.pa_prefill_attention.argtypes = [p, p, p, p, p, i32, p, p, i32, i32, i32, i32, i32, i32, i32,
                                       ctypes.c_float, ctypes.c_int, p, p]
    L.pa_prefill_attention.restype = ctypes.c_int
    L.pa_decode_attention_noalloc.argtypes = [p, p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32,
                                              ctypes.c_float, ctypes.c_int, p, p]
    L.pa_decode_attention_noalloc.restype = ctypes.c_int
    L.pa_bm_create.argtypes = [i32, ctypes.POINTER(p)]
    L.pa_bm_destroy.argtypes = [p]
    L.pa_bm_destroy.restype = None
    L.pa_bm_add_seq.argtypes = [p, ip]
    L.pa_bm_fork.argtypes = [p, i32, ip]
    L.pa_bm_free_seq.argtypes = [p, i32]
    L.pa_bm_blocks_needed.argtypes = [p, i32, i32, i32, ip]
    L.pa_bm_prepare_append.argtypes = [p, i32, i32, i32, ip, i32, ip]
    L.pa_bm_block_table.argtypes = [p, i32, ip, i32, ip]
    L.pa_bm_block_tables.argtypes = [p, ip, i32, ip, i32]
    L.pa_bm_seq_len.argtypes = [p, i32, ip]
    L.pa_bm_refcount.argtypes = [p, i32, ip]
    L.pa_bm_stats.argtypes = [p, ctypes.POINTER(BmStats)]
    for n in ("pa_bm_create", "pa_bm_add_seq", "pa_bm_fork", "pa_bm_free_seq",
              "pa_bm_blocks_needed", "pa_bm_prepare_append", "pa_bm_block_table",
              "pa_bm_block_tables",
              "pa_bm_seq_len", "pa_bm_refcount", "pa_bm_stats"):
        getattr(L, n).restype = ctypes.c_int
    _lib = L
    return L


def check(fn: str, status: int) -> None:
    if status != PA_OK:
        raise PagedKVError(fn, status, lib().pa_status_string(status).decode())


def _ptr(t) -> int:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor (device pointer)")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _i32(t, name):
    if t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")
    return _ptr(t)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype == torch.float32:
        return PA_F32
    raise TypeError(f"unsupported element type {t.dtype}")


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def pool_shape(num_blocks: int, num_kv_heads: int, head_dim: int, dtype: torch.dtype):
    """Shape of one K or V pool in the library's layout."""
    x = 16 // torch.empty((), dtype=dtype).element_size()
    return (num_blocks, num_kv_heads, head_dim // x, BLOCK_SIZE, x)


def fp8_pool_shape(num_blocks: int, num_kv_heads: int, head_dim: int):
    """Shape of one FP8 (E4M3) pool: per (block, kv head) a record of 16*D codes + 16 scales."""
    return (num_blocks, num_kv_heads, 16 * head_dim + 64)


def _fp8_dims(k_pool: torch.Tensor):
    if k_pool.dim() != 3 or k_pool.dtype != torch.uint8 or (k_pool.shape[2] - 64) % 16:
        raise ValueError("FP8 pools must be uint8 [num_blocks][Hkv][16*D + 64]")
    return k_pool.shape[0], k_pool.shape[1], (k_pool.shape[2] - 64) // 16


def append_kv_fp8(k_pool, v_pool, k_new, v_new, block_tables, start_pos, cu_new_tokens,
                  err_flag=None, stream=None) -> None:
    """Quantise bf16 rows ([tokens][Hkv][D]) into FP8 pools at explicit positions."""
    nb, hkv, d = _fp8_dims(k_pool)
    if k_new.dtype != torch.bfloat16 or v_new.dtype != torch.bfloat16:
        raise TypeError("new rows must be bf16")
    check("pa_append_kv_fp8", lib().pa_append_kv_fp8(
        _ptr(k_pool), _ptr(v_pool), _ptr(k_new), _ptr(v_new), _i32(block_tables, "block_tables"),
        block_tables.shape[1], _i32(start_pos, "start_pos"), _i32(cu_new_tokens, "cu_new_tokens"),
        start_pos.shape[0], k_new.shape[0], nb, hkv, d,
        None if err_flag is None else _i32(err_flag, "err_flag"), _stream(stream)))


def decode_attention_fp8(out, q, k_pool, v_pool, block_tables, context_lens, scale, workspace=None,
                         max_context_len_hint: int = 0, err_flag=None, stream=None) -> None:
    """decode_attention over FP8 pools (bf16 q and out)."""
    nb, hkv, d = _fp8_dims(k_pool)
    if q.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
        raise TypeError("q and out must be bf16")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check("pa_decode_attention_fp8", lib().pa_decode_attention_fp8(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _i32(block_tables, "block_tables"),
        _i32(context_lens, "context_lens"), q.shape[0], q.shape[1], hkv, d, block_tables.shape[1],
        int(max_context_len_hint), nb, float(scale),
        None if workspace is None else _ptr(workspace), ws_bytes,
        None if err_flag is None else _i32(err_flag, "err_flag"), _stream(stream)))


def append_decode_attention_fp8(out, q, k_pool, v_pool, k_new, v_new, block_tables, context_lens,
                                scale, workspace=None, max_context_len_hint: int = 0,
                                err_flag=None, stream=None) -> None:
    """decode_attention_fp8 with the step's bf16 rows k_new / v_new ([S][Hkv][D]) quantised
    and written at position context_lens[s] - 1 by the decode kernel itself."""
    nb, hkv, d = _fp8_dims(k_pool)
    if q.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
        raise TypeError("q and out must be bf16")
    for t, name in ((k_new, "k_new"), (v_new, "v_new")):
        if tuple(t.shape) != (q.shape[0], hkv, d) or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 [num_seqs][num_kv_heads][head_dim] tensor")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check("pa_append_decode_attention_fp8", lib().pa_append_decode_attention_fp8(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_new), _ptr(v_new),
        _i32(block_tables, "block_tables"), _i32(context_lens, "context_lens"), q.shape[0],
        q.shape[1], hkv, d, block_tables.shape[1], int(max_context_len_hint), nb, float(scale),
        None if workspace is None else _ptr(workspace), ws_bytes,
        None if err_flag is None else _i32(err_flag, "err_flag"), _stream(stream)))


def copy_block_fp8(k_pool, v_pool, pairs, err_flag=None, stream=None) -> None:
    """copy_block for FP8 pools."""
    nb, hkv, d = _fp8_dims(k_pool)
    check("pa_copy_block", lib().pa_copy_block(
        _ptr(k_pool), _ptr(v_pool), _i32(pairs, "pairs"), pairs.shape[0], nb, hkv, d, 2,
        None if err_flag is None else _i32(err_flag, "err_flag"), _stream(stream)))


def fp4_pool_shape(num_blocks: int, num_kv_heads: int, head_dim: int):
    """Shape of one MXFP4 pool: per (block, kv head) 8*D code bytes + D/2 scale bytes."""
    return (num_blocks, num_kv_heads, 8 * head_dim + head_dim // 2)


def _fp4_dims(k_pool: torch.Tensor):
    if k_pool.dim() != 3 or k_pool.dtype != torch.uint8 or k_pool.shape[2] % 17:
        raise ValueError("FP4 pools must be uint8 [num_blocks][Hkv][8*D + D/2]")
    return k_pool.shape[0], k_pool.shape[1], k_pool.shape[2] * 2 // 17


def append_kv_fp4(k_pool, v_pool, k_new, v_new, block_tables, start_pos, cu_new_tokens,
                  err_flag=None, stream=None) -> None:
    """Quantise bf16 rows ([tokens][Hkv][D]) into MXFP4 pools at explicit positions."""
    nb, hkv, d = _fp4_dims(k_pool)
    if k_new.dtype != torch.bfloat16 or v_new.dtype != torch.bfloat16:
        raise TypeError("new rows must be bf16")
    check("pa_append_kv_fp4", lib().pa_append_kv_fp4(
        _ptr(k_pool), _ptr(v_pool), _ptr(k_new), _ptr(v_new), _i32(block_tables, "block_tables"),
        block_tables.shape[1], _i32(start_pos, "start_pos"), _i32(cu_new_tokens, "cu_new_tokens"),
        start_pos.shape[0], k_new.shape[0], nb, hkv, d,
        None if err_flag is None else _i32(err_flag, "err_flag"), _stream(stream)))


def decode_attention_fp4(out, q, k_pool, v_pool, block_tables, context_lens, scale, workspace=None,
                         max_context_len_hint: int = 0, err_flag=None, stream=None) -> None:
    """decode_attention over MXFP4 pools (bf16 q and out)."""
    nb, hkv, d = _fp4_dims(k_pool)
    if q.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
        raise TypeError("q and out must be bf16")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check("pa_decode_attention_fp4", lib().pa_decode_attention_fp4(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _i32(block_tables, "block_tables"),
        _i32(context_lens, "context_lens"), q.shape[0], q.shape[1], hkv, d, block_tables.shape[1],
        int(max_context_len_hint), nb, float(scale),
        None if workspace is None else _ptr(workspace), ws_bytes,
        None if err_flag is None else _i32(err_flag, "err_flag"), _stream(stream)))


def copy_block_fp4(k_pool, v_pool, pairs, err_flag=None, stream=None) -> None:
    """copy_block for MXFP4 pools."""
    nb, hkv, d = _fp4_dims(k_pool)
    check("pa_copy_block", lib().pa_copy_block(
        _ptr(k_pool), _ptr(v_pool), _i32(pairs, "pairs"), pairs.shape[0], nb, hkv, d, 3,
        None if err_flag is None else _i32(err_flag, "err_flag"), _stream(stream)))


def _pool_dims(k_pool: torch.Tensor):
    if k_pool.dim() != 5 or k_pool.shape[3] != BLOCK_SIZE:
        raise ValueError("pools must have shape [num_blocks][Hkv][D/X][16][X]")
    return k_pool.shape[0], k_pool.shape[1], k_pool.shape[2] * k_pool.shape[4]


def append_kv(k_pool, v_pool, k_new, v_new, block_tables, start_pos, cu_new_tokens,
              err_flag=None, stream=None) -> None:
    """Write rows of k_new / v_new ([tokens][Hkv][D]) at explicit positions."""
    nb, hkv, d = _pool_dims(k_pool)
    check("pa_append_kv", lib().pa_append_kv(
        _ptr(k_pool), _ptr(v_pool), _ptr(k_new), _ptr(v_new), _i32(block_tables, "block_tables"),
        block_tables.shape[1], _i32(start_pos, "start_pos"), _i32(cu_new_tokens, "cu_new_tokens"),
        start_pos.shape[0], k_new.shape[0], nb, hkv, d, _dtype_code(k_pool),
        None if err_flag is None else _i32(err_flag, "err_flag"), _stream(stream)))


def copy_block(k_pool, v_pool, pairs, err_flag=None, stream=None) -> None:
    """Copy whole blocks src -> dst (pairs: int32 [n][2] on the device)."""
    nb, hkv, d = _pool_dims(k_pool)
    check("pa_copy_block", lib().pa_copy_block(
        _ptr(k_pool), _ptr(v_pool), _i32(pairs, "pairs"), pairs.shape[0], nb, hkv, d,
        _dtype_code(k_pool), None if err_flag is None else _i32(err_flag, "err_flag"),
        _stream(stream)))


def decode_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                          max_blocks_per_seq: int) -> int:
    return int(lib().pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                              max_blocks_per_seq))


def decode_workspace(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                     max_blocks_per_seq: int, device="cuda"):
    """A zero-filled workspace for decode_attention (None when none is needed)."""
    n = decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq)
    return torch.zeros(n, dtype=torch.uint8, device=device) if n else None


def decode_attention(out, q, k_pool, v_pool, block_tables, context_lens, scale, workspace=None,
                     max_context_len_hint: int = 0, err_flag=None, stream=None) -> None:
    """Single-token attention of q ([S][Hq][D]) over the paged cache into out."""
    nb, hkv, d = _pool_dims(k_pool)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check("pa_decode_attention", lib().pa_decode_attention(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _i32(block_tables, "block_tables"),
        _i32(context_lens, "context_lens"), q.shape[0], q.shape[1], hkv, d, block_tables.shape[1],
        int(max_context_len_hint), nb, float(scale), _dtype_code(q),
        None if workspace is None else _ptr(workspace), ws_bytes,
        None if err_flag is None else _i32(err_flag, "err_flag"), _stream(stream)))


def append_decode_attention(out, q, k_pool, v_pool, k_new, v_new, block_tables, context_lens,
                            scale, workspace=None, max_context_len_hint: int = 0, err_flag=None,
                            stream=None) -> None:
    """One decode step in one call: k_new / v_new ([S][Hkv][D]) go to position
    context_lens[s] - 1 (context_lens counts the new token), then decode_attention."""
    nb, hkv, d = _pool_dims(k_pool)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    for t, name in ((k_new, "k_new"), (v_new, "v_new")):
        if tuple(t.shape) != (q.shape[0], hkv, d) or t.dtype != k_pool.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [num_seqs][num_kv_heads][head_dim] "
                             f"tensor of the pool's type")
    check("pa_append_decode_attention", lib().pa_append_decode_attention(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_new), _ptr(v_new),
        _i32(block_tables, "block_tables"), _i32(context_lens, "context_lens"), q.shape[0],
        q.shape[1], hkv, d, block_tables.shape[1], int(max_context_len_hint), nb, float(scale),
        _dtype_code(q), None if workspace is None else _ptr(workspace), ws_bytes,
        None if err_flag is None else _i32(err_flag, "err_flag"), _stream(stream)))


def append_decode_attention_shared_prefix(out, q, k_pool, v_pool, k_new, v_new, block_tables,
                                          context_lens, scale, shared_prefix_tokens: int,
                                          workspace=None, max_context_len_hint: int = 0,
                                          err_flag=None, stream=None) -> None:
    """decode_attention_shared_prefix with the step's new rows written by the decode kernel
    (k_new / v_new [S][Hkv][D] go to position context_lens[s] - 1, past the prefix)."""
    nb, hkv, d = _pool_dims(k_pool)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    for t, name in ((k_new, "k_new"), (v_new, "v_new")):
        if tuple(t.shape) != (q.shape[0], hkv, d) or t.dtype != k_pool.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [num_seqs][num_kv_heads][head_dim] "
                             f"tensor of the pool's type")
    check("pa_append_decode_attention_shared_prefix", lib().pa_append_decode_attention_shared_prefix(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_new), _ptr(v_new),
        _i32(block_tables, "block_tables"), _i32(context_lens, "context_lens"), q.shape[0],
        q.shape[1], hkv, d, block_tables.shape[1], int(max_context_len_hint), nb, float(scale),
        _dtype_code(q), int(shared_prefix_tokens), None if workspace is None else _ptr(workspace),
        ws_bytes, None if err_flag is None else _i32(err_flag, "err_flag"), _stream(stream)))


def decode_attention_shared_prefix(out, q, k_pool, v_pool, block_tables, context_lens, scale,
                                   shared_prefix_tokens: int, workspace=None,
                                   max_context_len_hint: int = 0, err_flag=None,
                                   stream=None) -> None:
    """decode_attention for a batch whose sequences share their first
    ``shared_prefix_tokens`` positions in the same physical blocks."""
    nb, hkv, d = _pool_dims(k_pool)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check("pa_decode_attention_shared_prefix", lib().pa_decode_attention_shared_prefix(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _i32(block_tables, "block_tables"),
        _i32(context_lens, "context_lens"), q.shape[0], q.shape[1], hkv, d, block_tables.shape[1],
        int(max_context_len_hint), nb, float(scale), _dtype_code(q), int(shared_prefix_tokens),
        None if workspace is None else _ptr(workspace), ws_bytes,
        None if err_flag is None else _i32(err_flag, "err_flag"), _stream(stream)))


def prefill_attention(out, q, k_pool, v_pool, block_tables, start_pos, cu_q, scale,
                      max_chunk: int, err_flag=None, stream=None) -> None:
    """Causal attention of chunk rows q ([total][Hq][D]) over the paged cache."""
    nb, hkv, d = _pool_dims(k_pool)
    check("pa_prefill_attention", lib().pa_prefill_attention(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _i32(block_tables, "block_tables"),
        block_tables.shape[1], _i32(start_pos, "start_pos"), _i32(cu_q, "cu_q"),
        start_pos.shape[0], q.shape[0], int(max_chunk), q.shape[1], hkv, d, nb, float(scale),
        _dtype_code(q), None if err_flag is None else _i32(err_flag, "err_flag"), _stream(stream)))


NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024
PA_ERR_SCRATCH_LIMIT = 5


def decode_attention_noalloc(out, q, k_pool, v_pool, block_tables, context_lens, scale,
                             max_context_len_hint: int = 0, err_flag=None, stream=None) -> None:
    """decode_attention without a caller workspace: the library's built-in 16 MiB device
    scratch is used instead (for callers that cannot allocate device memory)."""
    nb, hkv, d = _pool_dims(k_pool)
    check("pa_decode_attention_noalloc", lib().pa_decode_attention_noalloc(
        _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _i32(block_tables, "block_tables"),
        _i32(context_lens, "context_lens"), q.shape[0], q.shape[1], hkv, d, block_tables.shape[1],
        int(max_context_len_hint), nb, float(scale), _dtype_code(q),
        None if err_flag is None else _i32(err_flag, "err_flag"), _stream(stream)))


class BlockManager:
    """Host block manager (refcounts, block tables, copy-on-write pairs)."""

    def __init__(self, num_blocks: int):
        self._h = ctypes.c_void_p()
        check("pa_bm_create", lib().pa_bm_create(num_blocks, ctypes.byref(self._h)))
        self.num_blocks = num_blocks

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.pa_bm_destroy(h)
            self._h = None

    def add_seq(self) -> int:
        out = ctypes.c_int32()
        check("pa_bm_add_seq", lib().pa_bm_add_seq(self._h, ctypes.byref(out)))
        return out.value

    def fork(self, parent: int) -> int:
        out = ctypes.c_int32()
        check("pa_bm_fork", lib().pa_bm_fork(self._h, parent, ctypes.byref(out)))
        return out.value

    def free(self, seq: int) -> None:
        check("pa_bm_free_seq", lib().pa_bm_free_seq(self._h, seq))

    def blocks_needed(self, seq: int, start: int, n: int) -> int:
        out = ctypes.c_int32()
        check("pa_bm_blocks_needed", lib().pa_bm_blocks_needed(self._h, seq, start, n,
                                                                 ctypes.byref(out)))
        return out.value

    def prepare_append(self, seq: int, start: int, n: int) -> list:
        """Returns the copy-on-write pairs [(src, dst), ...]; raises on out-of-blocks."""
        cap = n // BLOCK_SIZE + 2
        buf = (ctypes.c_int32 * (2 * cap))()
        npairs = ctypes.c_int32()
        check("pa_bm_prepare_append", lib().pa_bm_prepare_append(
            self._h, seq, start, n, buf, cap, ctypes.byref(npairs)))
        return [(buf[2 * i], buf[2 * i + 1]) for i in range(npairs.value)]

    def block_table(self, seq: int, max_blocks: int) -> list:
        buf = (ctypes.c_int32 * max(max_blocks, 1))()
        check("pa_bm_block_table", lib().pa_bm_block_table(self._h, seq, buf, max_blocks, None))
        return list(buf[:max_blocks])

    def block_tables(self, seqs, max_blocks: int, out=None):
        """The tables of several sequences in one call: int32 array [len(seqs)][max_blocks]
        (written into `out`, a C-contiguous int32 numpy array of that shape, if given)."""
        ids = np.ascontiguousarray(np.asarray(seqs, np.int32))
        n = int(ids.size)
        if out is None:
            out = np.empty((n, max_blocks), np.int32)
        if out.dtype != np.int32 or not out.flags.c_contiguous or out.shape != (n, max_blocks):
            raise ValueError("out: a C-contiguous int32 array of shape (len(seqs), max_blocks)")
        ipp = ctypes.POINTER(ctypes.c_int32)
        check("pa_bm_block_tables", lib().pa_bm_block_tables(
            self._h, ids.ctypes.data_as(ipp), n, out.ctypes.data_as(ipp), max_blocks))
        return out

    def seq_len(self, seq: int) -> int:
        out = ctypes.c_int32()
        check("pa_bm_seq_len", lib().pa_bm_seq_len(self._h, seq, ctypes.byref(out)))
        return out.value

    def refcount(self, block: int) -> int:
        out = ctypes.c_int32()
        check("pa_bm_refcount", lib().pa_bm_refcount(self._h, block, ctypes.byref(out)))
        return out.value

    def stats(self) -> dict:
        st = BmStats()
        check("pa_bm_stats", lib().pa_bm_stats(self._h, ctypes.byref(st)))
        return {"physical_blocks": st.physical_blocks, "free_blocks": st.free_blocks,
                "logical_tokens": st.logical_tokens, "num_seqs": st.num_seqs,
                "physical_slots": st.physical_blocks * BLOCK_SIZE}

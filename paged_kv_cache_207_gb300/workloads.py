"""Seeded synthetic inputs for paged decode attention.

This module only draws inputs: sequence lengths, block tables (which physical
block holds which logical block) and the query / key / value numbers.  It holds
none of the attention arithmetic and no pool layout; the CUDA library and the
CPU oracle each place the generated token rows into their own pools through
their own append.

Shapes follow the workloads the pages describe: GPT-2 124M heads (12 x 64) from
spindle, Qwen2.5-0.5B heads (14 query / 2 kv x 64) from Slipstream's "Where it
actually stands", and a Llama-3-8B head shape (32 / 8 x 128) for large-batch and
long-context decode.  Values are i.i.d. N(0, 1) drawn in fp32 and rounded once
to bf16 (round to nearest even) where the workload is bf16.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK = 16


@dataclass
class DecodeWorkload:
    """One decode step over a batch of sequences.

    ``context_lens[s]`` is the length *before* this step; the step appends one
    token at position ``context_lens[s]`` and attends over ``context_lens[s] + 1``
    tokens.  Token rows (``k_rows`` / ``v_rows``: [rows][Hkv][D]) hold every
    token once; ``fill`` lists the appends ``(seq, start_pos, first_row, n)`` that
    put the context into a pool; ``logical_rows(s)`` gives, in order, the rows of
    sequence ``s``'s context including the new token."""

    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str                      # "f32" or "bf16"
    scale: float
    context_lens: np.ndarray        # int32 [S], before the step's append
    block_tables: np.ndarray        # int32 [S][max_blocks], -1 = unused
    num_blocks: int
    q: torch.Tensor                 # [S][Hq][D]
    k_rows: torch.Tensor            # [rows][Hkv][D]
    v_rows: torch.Tensor
    fill: list                      # (seq, start_pos, first_row, n)
    new_rows: np.ndarray            # int64 [S], row of each sequence's new token
    seq_rows: list = field(default_factory=list)   # per seq: list of (first_row, n) segments

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    def logical_rows(self, s: int) -> np.ndarray:
        idx = [np.arange(a, a + n, dtype=np.int64) for a, n in self.seq_rows[s]]
        return np.concatenate(idx + [np.array([self.new_rows[s]], np.int64)])

    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


def _values(gen: torch.Generator, shape, device, dtype, big_key_frac: float = 0.0,
            big_key_scale: float = 8.0, chunk_rows: int = 1 << 16) -> torch.Tensor:
    """N(0,1) numbers in fp32, optionally with a fraction of (row, head) vectors scaled,
    then rounded once to ``dtype``.  Drawn in row chunks to bound temporary memory."""
    out = torch.empty(shape, dtype=dtype, device=device)
    rows = shape[0]
    for a in range(0, rows, chunk_rows):
        b = min(rows, a + chunk_rows)
        x = torch.randn((b - a,) + tuple(shape[1:]), generator=gen, device=device,
                        dtype=torch.float32)
        if big_key_frac > 0.0:
            m = torch.rand((b - a,) + tuple(shape[1:-1]), generator=gen, device=device) < big_key_frac
            x = torch.where(m.unsqueeze(-1), x * big_key_scale, x)
        out[a:b] = x.to(dtype)
    return out


def _tables_from_perm(perm: np.ndarray, blocks_per_seq: np.ndarray, max_blocks: int) -> np.ndarray:
    """Hand out physical blocks to sequences in order from a shuffled list of block ids."""
    S = blocks_per_seq.shape[0]
    tables = np.full((S, max_blocks), -1, np.int32)
    k = 0
    for s in range(S):
        n = int(blocks_per_seq[s])
        tables[s, :n] = perm[k:k + n]
        k += n
    return tables


def make_decode_workload(name: str, *, context_lens, num_q_heads: int, num_kv_heads: int,
                         head_dim: int, dtype: str, seed: int, device="cpu",
                         pool_blocks: int | None = None, scale: float | None = None,
                         big_key_frac: float = 0.0, max_blocks: int | None = None,
                         shared_prefix: int = 0) -> DecodeWorkload:
    """Build a decode workload.  ``shared_prefix`` > 0 makes every sequence share its
    first ``shared_prefix`` tokens (whole blocks, one physical copy: the layout a
    refcounted copy-on-write fork leaves behind)."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(context_lens, np.int32)
    S = lens.shape[0]
    if shared_prefix % BLOCK:
        raise ValueError("a shared prefix must be whole blocks")
    total = lens + 1                                         # after the step's append
    need = (total + BLOCK - 1) // BLOCK
    pre_blocks = shared_prefix // BLOCK
    private = need - pre_blocks
    if np.any(private < 0):
        raise ValueError("context shorter than the shared prefix")
    uniq_blocks = int(private.sum()) + pre_blocks
    nb = pool_blocks if pool_blocks is not None else uniq_blocks
    if nb < uniq_blocks:
        raise ValueError("pool too small")
    mb = max_blocks if max_blocks is not None else int(need.max())
    perm = rng.permutation(nb).astype(np.int32)
    if pre_blocks:
        prefix_ids = perm[:pre_blocks]
        rest = _tables_from_perm(perm[pre_blocks:], private, mb - pre_blocks)
        tables = np.full((S, mb), -1, np.int32)
        tables[:, :pre_blocks] = prefix_ids
        tables[:, pre_blocks:] = rest
    else:
        tables = _tables_from_perm(perm, need, mb)

    # token rows: the shared prefix once, then each sequence's private context,
    # then one new token per sequence
    fill, seq_rows = [], [[] for _ in range(S)]
    row = 0
    if shared_prefix:
        fill.append((0, 0, 0, shared_prefix))
        for s in range(S):
            seq_rows[s].append((0, shared_prefix))
        row = shared_prefix
    for s in range(S):
        n = int(lens[s]) - shared_prefix
        if n > 0:
            fill.append((s, shared_prefix, row, n))
            seq_rows[s].append((row, n))
            row += n
    new_rows = np.arange(row, row + S, dtype=np.int64)
    rows = row + S

    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q = _values(gen, (S, num_q_heads, head_dim), device, tdt)
    k_rows = _values(gen, (rows, num_kv_heads, head_dim), device, tdt, big_key_frac=big_key_frac)
    v_rows = _values(gen, (rows, num_kv_heads, head_dim), device, tdt)
    return DecodeWorkload(name=name, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                          head_dim=head_dim, dtype=dtype,
                          scale=scale if scale is not None else 1.0 / float(np.sqrt(head_dim)),
                          context_lens=lens, block_tables=tables, num_blocks=nb, q=q,
                          k_rows=k_rows, v_rows=v_rows, fill=fill, new_rows=new_rows,
                          seq_rows=seq_rows)


# ---- named workloads -------------------------------------------------------

def gpt2_tiny_f32(device="cpu", seed=207) -> DecodeWorkload:
    """4 sequences, GPT-2 124M heads (12 x 64), fp32, contexts {17, 40, 64, 100},
    a 64-block pool handed out in a seeded random order, scale 1/8."""
    return make_decode_workload("gpt2_tiny_f32", context_lens=[17, 40, 64, 100], num_q_heads=12,
                                num_kv_heads=12, head_dim=64, dtype="f32", seed=seed,
                                device=device, pool_blocks=64, scale=1.0 / 8.0)


def qwen05b_gqa(device="cpu", seed=209, num_seqs=128, lo=512, hi=4096,
                pool_blocks=40000) -> DecodeWorkload:
    """Qwen2.5-0.5B heads: 14 query / 2 kv heads x 64, bf16, contexts U[512, 4096],
    block tables drawn from a seeded shuffle of a 40 000-block pool."""
    rng = np.random.default_rng(seed + 1000)
    lens = rng.integers(lo, hi + 1, size=num_seqs).astype(np.int32)
    return make_decode_workload("qwen2.5-0.5b_gqa", context_lens=lens, num_q_heads=14,
                                num_kv_heads=2, head_dim=64, dtype="bf16", seed=seed,
                                device=device, pool_blocks=pool_blocks)


def lognormal_lengths(rng, n, median, sigma, cap, floor=1) -> np.ndarray:
    z = rng.standard_normal(n)
    return np.clip(np.round(median * np.exp(sigma * z)), floor, cap).astype(np.int32)


def llama8b_batch(device="cpu", seed=210, num_seqs=256, median=1024, sigma=1.0,
                  cap=8192) -> DecodeWorkload:
    """Llama-3-8B heads (32 query / 8 kv x 128), bf16, 256 sequences with context
    lengths lognormal (median 1024, sigma 1) capped at 8192; 1 % of key vectors
    (per token and kv head) scaled by 8 before rounding to bf16."""
    rng = np.random.default_rng(seed + 1000)
    lens = lognormal_lengths(rng, num_seqs, median, sigma, cap - 1)
    return make_decode_workload("llama3-8b_batch256", context_lens=lens, num_q_heads=32,
                                num_kv_heads=8, head_dim=128, dtype="bf16", seed=seed,
                                device=device, big_key_frac=0.01)


def llama8b_long(device="cpu", seed=211, num_seqs=8, lo=32768, hi=131072) -> DecodeWorkload:
    """Llama-3-8B heads, bf16, 8 sequences with contexts U[32768, 131072]."""
    rng = np.random.default_rng(seed + 1000)
    lens = rng.integers(lo, hi + 1, size=num_seqs).astype(np.int32) - 1
    return make_decode_workload("llama3-8b_long_context", context_lens=lens, num_q_heads=32,
                                num_kv_heads=8, head_dim=128, dtype="bf16", seed=seed,
                                device=device)


def llama8b_shared_prefix(device="cpu", seed=212, num_seqs=64, prefix=4096, lo=16,
                          hi=512) -> DecodeWorkload:
    """Llama-3-8B heads, bf16, 64 sequences that share one 4096-token prefix (256
    blocks held 64 times) followed by a private suffix of U[16, 512] tokens."""
    rng = np.random.default_rng(seed + 1000)
    suffix = rng.integers(lo, hi + 1, size=num_seqs).astype(np.int32)
    lens = prefix + suffix - 1
    return make_decode_workload("llama3-8b_shared_prefix", context_lens=lens, num_q_heads=32,
                                num_kv_heads=8, head_dim=128, dtype="bf16", seed=seed,
                                device=device, shared_prefix=prefix)


WORKLOADS = {
    "gpt2_tiny_f32": gpt2_tiny_f32,
    "qwen2.5-0.5b_gqa": qwen05b_gqa,
    "llama3-8b_batch256": llama8b_batch,
    "llama3-8b_long_context": llama8b_long,
    "llama3-8b_shared_prefix": llama8b_shared_prefix,
}


# ---- the spindle-shaped replay ------------------------------------------------

@dataclass
class ReplayWorkload:
    """64 requests replayed through continuous batching (spindle, "Paging" and
    "Continuous batching, and the control"): 60 independent requests plus 4
    copy-on-write children forked from one 16-token parent prompt.  GPT-2 124M
    heads (12 x 64), 12 layers, bf16, a pool of 8192 token slots (512 blocks) per
    layer.  Prompt lengths U[16, 128]; generated lengths lognormal (median 40,
    sigma 1) capped at 192.  All requests arrive at time 0.

    Values are drawn once for every (sequence, layer, position): ``q/k/v`` are
    [seqs][layers][max_len][heads][head_dim]; the children's first 16 positions
    hold the parent's prompt rows, so a recomputed (preempted) sequence gets the
    same numbers again."""

    prompt_lens: np.ndarray       # int32 [64]; the children's entry is the parent prompt (16)
    gen_lens: np.ndarray          # int32 [64]
    num_children: int             # the last num_children sequences are the forks
    parent_prompt: int
    num_blocks: int
    num_layers: int
    num_heads: int
    head_dim: int
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor

    @property
    def num_seqs(self) -> int:
        return int(self.prompt_lens.shape[0])

    @property
    def max_len(self) -> int:
        return int(self.q.shape[2])

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.head_dim))


def spindle_replay(device="cpu", seed=208, num_independent=60, num_children=4, parent_prompt=16,
                   prompt_lo=16, prompt_hi=128, gen_median=40, gen_sigma=1.0, gen_cap=192,
                   num_blocks=512, num_layers=12, num_heads=12, head_dim=64,
                   values: bool = True) -> ReplayWorkload:
    """``values=False`` draws the lengths only (for host-side schedule checks)."""
    rng = np.random.default_rng(seed + 1000)
    prompts = rng.integers(prompt_lo, prompt_hi + 1, size=num_independent).astype(np.int32)
    prompts = np.concatenate([prompts, np.full(num_children, parent_prompt, np.int32)])
    n = num_independent + num_children
    gens = lognormal_lengths(rng, n, gen_median, gen_sigma, gen_cap)
    max_len = prompt_hi + gen_cap
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    shape = (n, num_layers, max_len, num_heads, head_dim)
    if not values:
        empty = torch.empty((n, num_layers, max_len, 0, 0))
        return ReplayWorkload(prompt_lens=prompts, gen_lens=gens, num_children=num_children,
                              parent_prompt=parent_prompt, num_blocks=num_blocks,
                              num_layers=num_layers, num_heads=num_heads, head_dim=head_dim,
                              q=empty, k=empty, v=empty)
    vals = []
    for _ in range(3):
        t = _values(gen, (n * num_layers * max_len, num_heads, head_dim), device, torch.bfloat16)
        vals.append(t.view(shape))
    q, k, v = vals
    first = num_independent
    for c in range(first + 1, n):           # every child starts from the same parent prompt
        k[c, :, :parent_prompt] = k[first, :, :parent_prompt]
        v[c, :, :parent_prompt] = v[first, :, :parent_prompt]
    return ReplayWorkload(prompt_lens=prompts, gen_lens=gens, num_children=num_children,
                          parent_prompt=parent_prompt, num_blocks=num_blocks,
                          num_layers=num_layers, num_heads=num_heads, head_dim=head_dim,
                          q=q, k=k, v=v)

/*
 * pa.h -- C ABI of the paged KV-cache decode-attention library (sm_103a).
 *
 * The operations follow the engines described on two pages:
 *   spindle ("A faster engine for running language models"):
 *     - section "Paging": K/V live in a pool of fixed-size blocks (block size
 *       16) shared by every sequence; each sequence reaches its blocks through
 *       a block table; reference counts give copy-on-write forks.
 *     - section "Two bugs worth recording": append takes an explicit start
 *       position and the attention read takes an explicit length; the runner,
 *       not the cache, advances lengths once per step.
 *     - section "Why write the forward pass": batched decoding must equal
 *       decoding each sequence alone (no attention across sequences).
 *   Slipstream, section "The thesis" and Fig. 01: decode is bandwidth-bound,
 *     so the kernels are built to stream K/V at HBM speed.
 *   mlsystems topic list, the Flash-Decoding entry: decode (q_len = 1)
 *     attention split over chunks of the KV sequence, then reduced.
 *
 * Conventions for every call
 *   - All array arguments are DEVICE pointers unless the name says "host";
 *     the caller owns and allocates every buffer.  Nothing is allocated,
 *     freed, synchronised or kept between calls by the GPU entry points.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls only enqueue work; they return before it runs.
 *   - Device arrays must be 16-byte aligned.
 *   - Host-checkable faults return a status and launch nothing.  Faults that
 *     depend on device data (a table entry outside [0, num_blocks), a
 *     position beyond the table) are OR-ed as PA_DEV_ERR_* bits into
 *     *dev_err_flag (an int32 in device memory, may be NULL) and the
 *     offending element is skipped; nothing traps.
 *
 * Pool layout (the pages fix none; this library's choice):
 *   k_pool, v_pool: [num_blocks][num_kv_heads][head_dim / X][16][X]
 *   with X = 16 / sizeof(element) (8 for bf16, 4 for fp32).  Element
 *   (block b, kv head h, slot t, dim d) is at
 *     ((((b * Hkv + h) * (D / X) + d / X) * 16 + t) * X + d % X).
 *   Each (block, kv head) tile is one contiguous 16 * D * sizeof(element)
 *   byte chunk, and the 16-byte pieces of the 16 slots for the same dims sit
 *   side by side, so a tile moves as one bulk copy and is read back from
 *   shared memory without bank conflicts.
 *   Logical position p of sequence s is slot p % 16 of block
 *   block_tables[s][p / 16].
 */
#ifndef PAGED_KV_PA_H
#define PAGED_KV_PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_BLOCK_SIZE 16
#define PA_ABI_VERSION 1

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misalignment, small workspace */
    PA_ERR_UNSUPPORTED = 2,   /* head_dim not 64/128, more than 8 query heads per kv head */
    PA_ERR_CUDA = 3,          /* a CUDA launch or runtime call failed */
    PA_ERR_OUT_OF_BLOCKS = 4, /* block manager: not enough free blocks (nothing changed) */
    PA_ERR_SCRATCH_LIMIT = 5  /* pa_decode_attention_noalloc: the call needs more scratch
                                 than the library's built-in PA_NOALLOC_SCRATCH_BYTES */
} pa_status;

typedef enum {
    PA_F32 = 0,
    PA_BF16 = 1,
    PA_FP8_E4M3 = 2,  /* pools only: E4M3 codes with per-slot fp32 scales (see pa_append_kv_fp8) */
    PA_FP4_E2M1 = 3   /* pools only: MXFP4 records (see pa_append_kv_fp4) */
} pa_dtype;

/* Bits OR-ed into *dev_err_flag by the kernels. */
#define PA_DEV_ERR_BAD_BLOCK 1   /* a table entry read for a live position is outside [0, num_blocks) */
#define PA_DEV_ERR_BAD_POS 2     /* a position < 0 or >= max_blocks_per_seq * 16 */
#define PA_DEV_ERR_HINT 4        /* a context is longer than max_context_len_hint */
#define PA_DEV_ERR_BAD_CU 8      /* cu_new_tokens is not a prefix sum ending at total_new_tokens */
#define PA_DEV_ERR_TIMEOUT 16    /* a bulk-copy or tensor-core wait gave up after 200 ms.  The
                                    outputs of the work that gave up are written as NaN.
                                    While this bit is set in the flag, every decode, prefill
                                    and partition-merge kernel given the flag returns without
                                    writing anything (so a broken pipeline cannot hold the GPU
                                    or overwrite results); clear the bit to resume.  Without a
                                    flag (NULL) the NaN outputs are the only sign. */
#define PA_DEV_ERR_BAD_PAIR 32   /* a copy pair names a block outside [0, num_blocks) */
#define PA_DEV_ERR_BAD_PREFIX 64 /* pa_decode_attention_shared_prefix: a sequence's table does
                                    not hold sequence 0's prefix blocks, or its context is
                                    shorter than the shared prefix (its output is wrong); with
                                    the step's new rows (pa_append_decode_attention_shared_prefix),
                                    also a new row that would fall inside the prefix (not
                                    written) */

/* Tokens per split-KV partition of pa_decode_attention at head_dim 128 (a multiple
 * of 16); head_dim 64 uses 2 * PA_PARTITION_TOKENS, the same bytes per partition. */
#define PA_PARTITION_TOKENS 512

const char* pa_status_string(pa_status s);
int32_t pa_abi_version(void);

/*
 * pa_append_kv -- write new K/V tokens at explicit positions (spindle,
 * "Two bugs worth recording": append takes an explicit start position).
 *
 *   k_new, v_new     [total_new_tokens][num_kv_heads][head_dim], plain row-major,
 *                    rows of sequence s are cu_new_tokens[s] .. cu_new_tokens[s+1]-1
 *   block_tables     int32 [num_seqs][max_blocks_per_seq]
 *   start_pos        int32 [num_seqs]: row cu_new_tokens[s] + i goes to position
 *                    start_pos[s] + i of sequence s
 *   cu_new_tokens    int32 [num_seqs + 1], cu_new_tokens[0] = 0,
 *                    cu_new_tokens[num_seqs] = total_new_tokens (host value)
 * The pools are written bit for bit.  Positions whose table entry is out of
 * range are skipped and flagged.  The caller guarantees that no two rows
 * target the same slot and that no target block is shared (refcount > 1);
 * the block manager below gives those guarantees.  Nothing is read back.
 */
pa_status pa_append_kv(void* k_pool, void* v_pool, const void* k_new, const void* v_new,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* start_pos, const int32_t* cu_new_tokens, int32_t num_seqs,
                       int32_t total_new_tokens, int32_t num_blocks, int32_t num_kv_heads,
                       int32_t head_dim, pa_dtype dtype, int32_t* dev_err_flag, void* stream);

/*
 * pa_copy_block -- materialise copy-on-write forks (spindle, "Paging":
 * reference counts give copy-on-write forking).
 *
 *   src_dst_pairs    int32 [num_pairs][2] (device): every byte of block src is
 *                    copied to block dst in both pools, all kv heads and slots.
 * Pairs naming a block outside [0, num_blocks) are skipped and flagged; a pair
 * with src == dst is a no-op.  Destinations must be distinct and no
 * destination may be another pair's source.
 */
pa_status pa_copy_block(void* k_pool, void* v_pool, const int32_t* src_dst_pairs,
                        int32_t num_pairs, int32_t num_blocks, int32_t num_kv_heads,
                        int32_t head_dim, pa_dtype dtype, int32_t* dev_err_flag, void* stream);

/*
 * pa_decode_workspace_size -- bytes of device workspace pa_decode_attention
 * needs for these sizes (0 when no sequence can span two partitions).  The
 * workspace holds the per-partition partial results of the split-KV merge.
 */
size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t max_blocks_per_seq);

/*
 * pa_decode_attention -- single-token (q_len = 1) attention over the paged
 * cache (spindle, "Paging" and "Why write the forward pass"; the split over
 * KV partitions follows the Flash-Decoding entry of the mlsystems list).
 *
 *   out, q           [num_seqs][num_q_heads][head_dim], element type `dtype`
 *   context_lens     int32 [num_seqs]: sequence s attends over positions
 *                    0 .. context_lens[s]-1 (an explicit length; never changed)
 *   block_tables     int32 [num_seqs][max_blocks_per_seq]
 * For each sequence s and query head h, with kv head g = h / (Hq / Hkv):
 *   out[s][h] = sum_t softmax_t(scale * <q[s][h], K[s][t][g]>) V[s][t][g]
 * computed in fp32 (bf16 inputs are exact in fp32) and rounded once to the
 * output type.  Contexts are cut into fixed partitions (PA_PARTITION_TOKENS
 * tokens at head_dim 128, twice that at head_dim 64) whose partial results are merged with their log-sum-exp
 * weights; the partition of a token depends only on its position, so a
 * sequence's result does not depend on the rest of the batch.  A zero-length
 * context gives zeros.
 *   max_context_len_hint  host bound on every context_lens[s] used to size
 *                    the grid; <= 0 means max_blocks_per_seq * 16.  A context
 *                    that needs more partitions than the hint's sets
 *                    PA_DEV_ERR_HINT and its output is incomplete.
 *   workspace        device scratch of at least pa_decode_workspace_size()
 *                    bytes (may be NULL when that size is 0); its contents on
 *                    entry do not matter.  Calls sharing a workspace must not
 *                    overlap on the GPU.
 * head_dim must be 64 or 128 and num_q_heads / num_kv_heads at most 8.
 */
pa_status pa_decode_attention(void* out, const void* q, const void* k_pool, const void* v_pool,
                              const int32_t* block_tables, const int32_t* context_lens,
                              int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t max_blocks_per_seq,
                              int32_t max_context_len_hint, int32_t num_blocks, float scale,
                              pa_dtype dtype, void* workspace, size_t workspace_bytes,
                              int32_t* dev_err_flag, void* stream);

/*
 * pa_append_decode_attention -- one decode step in one call: the step's new
 * token is written into the cache, then attended over with the rest (spindle,
 * "Paging" for the step, "Two bugs worth recording" for the explicit position).
 *
 *   k_new, v_new     [num_seqs][num_kv_heads][head_dim], element type `dtype`,
 *                    16-byte aligned: sequence s's new K and V rows
 *   context_lens     int32 [num_seqs]: the length AFTER the append; the new
 *                    rows go to position context_lens[s] - 1
 * Every other argument, the workspace and the result are those of
 * pa_decode_attention.  The pools after the call hold exactly the bytes of
 * pa_append_kv(k_new, v_new, start_pos = context_lens - 1, one row per
 * sequence), and `out` equals pa_decode_attention's after that append, bit for
 * bit: this call is the two in one kernel (the CTA of the partition holding
 * the last position stores the row into the pools and into its own copy of
 * that block).  A sequence of
 * length 0 appends nothing.  A table entry out of range for the new position
 * sets PA_DEV_ERR_BAD_BLOCK and nothing is written there; a length beyond the
 * table sets PA_DEV_ERR_BAD_POS, appends nothing (as pa_append_kv) and is
 * clamped for the attention (as in pa_decode_attention).
 * While PA_DEV_ERR_TIMEOUT is set the call writes neither `out` nor the pools.
 * bf16 and f32 caches (the FP8 and FP4 paths keep their own append).
 */
pa_status pa_append_decode_attention(void* out, const void* q, void* k_pool, void* v_pool,
                                     const void* k_new, const void* v_new,
                                     const int32_t* block_tables, const int32_t* context_lens,
                                     int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t max_blocks_per_seq,
                                     int32_t max_context_len_hint, int32_t num_blocks, float scale,
                                     pa_dtype dtype, void* workspace, size_t workspace_bytes,
                                     int32_t* dev_err_flag, void* stream);

/*
 * pa_prefill_attention -- causal attention of chunks of new tokens over the
 * paged cache (chunked prefill; Slipstream, "Horizon", lists chunked prefill
 * among the engine's parts; spindle, "Two bugs worth recording": positions are
 * explicit, never inferred).
 *
 *   q, out           [total_q][num_q_heads][head_dim] bf16; rows of sequence s
 *                    are cu_q[s] .. cu_q[s+1]-1
 *   start_pos        int32 [num_seqs]: row cu_q[s] + i is the token at position
 *                    start_pos[s] + i, whose K/V the caller has already appended
 *   max_chunk        host bound on cu_q[s+1] - cu_q[s] (sizes the grid)
 * Row (s, i, h) attends over positions 0 .. start_pos[s] + i of sequence s
 * (query head h reads kv head h / G), i.e. it equals pa_decode_attention of
 * that query with context length start_pos[s] + i + 1.  bf16 only; head_dim 64
 * or 128; at most 8 query heads per kv head.  Positions past the table set
 * PA_DEV_ERR_BAD_POS and the tile is skipped.
 */
pa_status pa_prefill_attention(void* out, const void* q, const void* k_pool, const void* v_pool,
                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                               const int32_t* start_pos, const int32_t* cu_q, int32_t num_seqs,
                               int32_t total_q, int32_t max_chunk, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                               float scale, pa_dtype dtype, int32_t* dev_err_flag, void* stream);

/*
 * FP8 (E4M3) KV cache -- half the bytes per token for the bandwidth-bound decode
 * (Slipstream, "Companion work": a block-scaled low-precision kernel plugs into
 * the same bandwidth-bound decode path; the per-slot scale is this library's
 * choice for an 8-bit cache).
 *
 * Pools: uint8 [num_blocks][num_kv_heads][PA_FP8_RECORD_BYTES(head_dim)].  A
 * record holds the 16 slots of one (block, kv head): 16 * head_dim E4M3 codes
 * -- K as [head_dim / 16][16 slots][16 dims], V as [head_dim][16 slots] -- then
 * 16 fp32 scales, one per slot; value = code * scale.  pa_copy_block takes
 * dtype PA_FP8_E4M3 for these pools.
 */
#define PA_FP8_RECORD_BYTES(head_dim) (16 * (head_dim) + 64)

/* pa_append_kv_fp8 -- like pa_append_kv, with bf16 rows k_new / v_new that are
 * quantised on the way in: each (row, kv head) gets scale = max|x| / 448 and
 * codes = E4M3(x / scale) (fp32 arithmetic, round to nearest even, saturating at
 * 448; an all-zero row gets scale 0 and zero codes).  head_dim 64 or 128. */
pa_status pa_append_kv_fp8(void* k_pool, void* v_pool, const void* k_new, const void* v_new,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* start_pos, const int32_t* cu_new_tokens,
                           int32_t num_seqs, int32_t total_new_tokens, int32_t num_blocks,
                           int32_t num_kv_heads, int32_t head_dim, int32_t* dev_err_flag,
                           void* stream);

/* pa_decode_attention_fp8 -- pa_decode_attention over FP8 pools; q and out are
 * bf16, scores and the softmax in fp32, the products on the tensor cores in f16
 * (every E4M3 code is exact in f16).  Same workspace, partitions, errors. */
pa_status pa_decode_attention_fp8(void* out, const void* q, const void* k_pool, const void* v_pool,
                                  const int32_t* block_tables, const int32_t* context_lens,
                                  int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_blocks_per_seq,
                                  int32_t max_context_len_hint, int32_t num_blocks, float scale,
                                  void* workspace, size_t workspace_bytes, int32_t* dev_err_flag,
                                  void* stream);

/*
 * pa_append_decode_attention_fp8 -- one FP8 decode step in one call, as
 * pa_append_decode_attention is for bf16: the new bf16 rows k_new, v_new
 * ([num_seqs][num_kv_heads][head_dim], 16-byte aligned) are quantised exactly as
 * pa_append_kv_fp8 quantises them and written at position context_lens[s] - 1,
 * then attended over.  Pools and `out` equal those of pa_append_kv_fp8 (one row
 * per sequence) followed by pa_decode_attention_fp8, bit for bit; flags,
 * workspace and partitions as pa_decode_attention_fp8.
 */
pa_status pa_append_decode_attention_fp8(void* out, const void* q, void* k_pool, void* v_pool,
                                         const void* k_new, const void* v_new,
                                         const int32_t* block_tables, const int32_t* context_lens,
                                         int32_t num_seqs, int32_t num_q_heads,
                                         int32_t num_kv_heads, int32_t head_dim,
                                         int32_t max_blocks_per_seq, int32_t max_context_len_hint,
                                         int32_t num_blocks, float scale, void* workspace,
                                         size_t workspace_bytes, int32_t* dev_err_flag,
                                         void* stream);

/*
 * Block-scaled FP4 (MXFP4) KV cache -- a quarter of the bf16 bytes per token
 * (Slipstream, "Companion work": qgemm-mx, a block-scaled FP4 kernel for the same
 * bandwidth-bound decode path).  The format is the microscaling one: E2M1 codes
 * (1 sign, 2 exponent bits with bias 1, 1 mantissa bit: magnitudes 0, 0.5, 1,
 * 1.5, 2, 3, 4, 6), and one E8M0 scale byte (value 2^(code - 127)) per 32 values
 * along head_dim of each (token, kv head); value = code * scale.
 *
 * Pools: uint8 [num_blocks][num_kv_heads][PA_FP4_RECORD_BYTES(head_dim)].  A record
 * holds the 16 slots of one (block, kv head): 8 * head_dim code bytes, then
 * 16 * head_dim / 32 scale bytes ([16 slots][head_dim / 32]).  Code bytes (D =
 * head_dim; the low nibble holds the first of the two codes):
 *   K: slot t's row of D / 2 bytes at t * D / 2; the byte at c * (D / 8) +
 *      2 ks + half (c < 4, ks < D / 16, half < 2) holds dims 16 ks + 8 half + 2 c
 *      and + 1.
 *   V: the byte at ((4 r + c) * (D / 16) + mi) * 4 + 2 dh + half (r < 8, c < 4,
 *      mi < D / 16, dh < 2, half < 2) holds dim 16 mi + 8 dh + r of slots
 *      2 c + 8 half and + 1.
 * (These byte orders put each tensor-core fragment of a decode thread in adjacent
 * bytes.)  pa_copy_block takes dtype PA_FP4_E2M1 for these pools.
 */
#define PA_FP4_RECORD_BYTES(head_dim) (8 * (head_dim) + (head_dim) / 2)

/* pa_append_kv_fp4 -- like pa_append_kv, with bf16 rows k_new / v_new quantised on
 * the way in: each block of 32 values of a (row, kv head) gets the scale code
 * 127 + floor(log2 amax) - 2 (at least 0; an all-zero block gets 0) and codes
 * E2M1(x / scale) (exact power-of-two scaling, round to nearest even, saturating
 * at 6).  Rows of one call may share slots' V bytes; the kernel updates them
 * atomically.  head_dim 64 or 128. */
pa_status pa_append_kv_fp4(void* k_pool, void* v_pool, const void* k_new, const void* v_new,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* start_pos, const int32_t* cu_new_tokens,
                           int32_t num_seqs, int32_t total_new_tokens, int32_t num_blocks,
                           int32_t num_kv_heads, int32_t head_dim, int32_t* dev_err_flag,
                           void* stream);

/* pa_decode_attention_fp4 -- pa_decode_attention over MXFP4 pools; q and out are
 * bf16, scores and the softmax in fp32, the products on the tensor cores in f16
 * (every E2M1 code is exact in f16; the scales are applied in fp32, and to the
 * probabilities as powers of two).  Same workspace and errors; 2048-token
 * partitions. */
pa_status pa_decode_attention_fp4(void* out, const void* q, const void* k_pool, const void* v_pool,
                                  const int32_t* block_tables, const int32_t* context_lens,
                                  int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_blocks_per_seq,
                                  int32_t max_context_len_hint, int32_t num_blocks, float scale,
                                  void* workspace, size_t workspace_bytes, int32_t* dev_err_flag,
                                  void* stream);

/*
 * pa_decode_attention_shared_prefix -- pa_decode_attention for a batch whose
 * sequences all share their first shared_prefix_tokens positions in the same
 * physical blocks (the layout refcounted copy-on-write forks leave behind;
 * spindle, "Paging").  The whole 512-token partitions of the prefix are read
 * once per kv head and group of 128 or 256 query rows (not once per sequence)
 * and applied to the queries of every sequence on the tensor cores; the rest
 * of each context goes through the ordinary kernel; the two are merged with
 * their log-sum-exp weights.
 *   Same arguments as pa_decode_attention plus shared_prefix_tokens (a multiple
 *   of 16).  The caller guarantees that block_tables[s][b] == block_tables[0][b]
 *   for every s and every b < shared_prefix_tokens / 16, and that every
 *   context_lens[s] >= shared_prefix_tokens; the kernels read the prefix through
 *   sequence 0's table row, and a sequence that breaks the promise within the
 *   shared partitions sets PA_DEV_ERR_BAD_PREFIX.  bf16 only (fp32 returns
 *   PA_ERR_UNSUPPORTED when a whole partition is shared).  A prefix shorter than
 *   one partition, or a table of at most one partition (max_blocks_per_seq <=
 *   32), falls back to pa_decode_attention.  The workspace is the one
 *   pa_decode_workspace_size gives.
 */
pa_status pa_decode_attention_shared_prefix(void* out, const void* q, const void* k_pool,
                                            const void* v_pool, const int32_t* block_tables,
                                            const int32_t* context_lens, int32_t num_seqs,
                                            int32_t num_q_heads, int32_t num_kv_heads,
                                            int32_t head_dim, int32_t max_blocks_per_seq,
                                            int32_t max_context_len_hint, int32_t num_blocks,
                                            float scale, pa_dtype dtype,
                                            int32_t shared_prefix_tokens, void* workspace,
                                            size_t workspace_bytes, int32_t* dev_err_flag,
                                            void* stream);

/*
 * pa_append_decode_attention_shared_prefix -- pa_decode_attention_shared_prefix
 * with the step's new rows written by the decode kernel, as
 * pa_append_decode_attention does for pa_decode_attention: k_new and v_new
 * ([num_seqs][num_kv_heads][head_dim] bf16, 16-byte aligned) go to position
 * context_lens[s] - 1, and pools and `out` equal those of pa_append_kv followed
 * by pa_decode_attention_shared_prefix, bit for bit.  A new row must lie past
 * the shared prefix (context_lens[s] > shared_prefix_tokens: it goes to the
 * sequence's own block); one that would not is not written and sets
 * PA_DEV_ERR_BAD_PREFIX.  The fallbacks of pa_decode_attention_shared_prefix
 * fall back to pa_append_decode_attention, with the same check.
 */
pa_status pa_append_decode_attention_shared_prefix(
    void* out, const void* q, void* k_pool, void* v_pool, const void* k_new, const void* v_new,
    const int32_t* block_tables, const int32_t* context_lens, int32_t num_seqs,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t max_blocks_per_seq,
    int32_t max_context_len_hint, int32_t num_blocks, float scale, pa_dtype dtype,
    int32_t shared_prefix_tokens, void* workspace, size_t workspace_bytes, int32_t* dev_err_flag,
    void* stream);

/*
 * pa_decode_attention_noalloc -- pa_decode_attention for callers that cannot
 * allocate device memory.  (The pages have no counterpart; this entry point is
 * this library's own addition.)
 *
 * pa_decode_attention wants a caller-provided scratch workspace.  Some callers
 * cannot provide one: a plugin inside a host framework that owns all device
 * memory and gives plugins no scratch buffer, or a latency-critical decode loop
 * that must never call cudaMalloc because an allocation can synchronise the
 * whole device.  This entry point takes the same arguments minus the
 * workspace and runs the same kernels with the library's own scratch: one
 * file-scope device array of PA_NOALLOC_SCRATCH_BYTES (16 MiB), which every GPU
 * that loads the library holds until the process exits.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 *   - Limit: a call may need at most PA_NOALLOC_SCRATCH_BYTES, i.e.
 *     pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
 *     max_blocks_per_seq) <= 16 MiB (for head_dim 128, about num_seqs *
 *     num_q_heads * ceil(max_blocks_per_seq / 32) <= 32 000); larger calls
 *     return PA_ERR_SCRATCH_LIMIT and launch nothing.
 *   - Set-up: the first call on a device that needs scratch looks up the
 *     array's device address (cudaGetSymbolAddress) with that device current;
 *     make that first call before any stream capture.
 *   - Sharing: every call on a device uses the same array and leaves its
 *     partial results in it; no call depends on what an earlier call left
 *     there.  Calls whose kernels overlap on the GPU (other streams, other host
 *     threads) race on the array: serialise them.
 */
#define PA_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
pa_status pa_decode_attention_noalloc(void* out, const void* q, const void* k_pool,
                                      const void* v_pool, const int32_t* block_tables,
                                      const int32_t* context_lens, int32_t num_seqs,
                                      int32_t num_q_heads, int32_t num_kv_heads,
                                      int32_t head_dim, int32_t max_blocks_per_seq,
                                      int32_t max_context_len_hint, int32_t num_blocks,
                                      float scale, pa_dtype dtype, int32_t* dev_err_flag,
                                      void* stream);

/* ---------------------------------------------------------------------------
 * Host block manager (no GPU; spindle, "Paging").
 *
 * Owns the refcounts of a pool of num_blocks blocks and one block table per
 * live sequence.  Readings where the page is silent:
 *   - writing into a block whose refcount is above one first copies it into a
 *     newly allocated block (one (src, dst) pair for pa_copy_block), drops one
 *     reference to the old block and points the writer's table at the copy; a
 *     block held once is written in place;
 *   - refcounts count live sequences only;
 *   - free blocks are handed out lowest id first.
 * Handles are not thread-safe; use one per thread or lock around calls.
 * ------------------------------------------------------------------------- */
typedef struct pa_block_manager pa_block_manager;

typedef struct {
    int64_t physical_blocks;   /* blocks with refcount > 0 */
    int64_t free_blocks;
    int64_t logical_tokens;    /* sum of live sequence lengths */
    int64_t num_seqs;
} pa_bm_stats_t;

pa_status pa_bm_create(int32_t num_blocks, pa_block_manager** out);
void pa_bm_destroy(pa_block_manager* bm);
/* A new empty sequence; its id is written to *seq_out. */
pa_status pa_bm_add_seq(pa_block_manager* bm, int32_t* seq_out);
/* A child sharing every block of `parent` (each refcount + 1), same length. */
pa_status pa_bm_fork(pa_block_manager* bm, int32_t parent, int32_t* child_out);
/* Drop the sequence and one reference to each of its blocks. */
pa_status pa_bm_free_seq(pa_block_manager* bm, int32_t seq);
/* Blocks an append of num_tokens tokens at start_pos would take (host). */
pa_status pa_bm_blocks_needed(const pa_block_manager* bm, int32_t seq, int32_t start_pos,
                              int32_t num_tokens, int32_t* blocks_out);
/* Make positions start_pos .. start_pos+num_tokens-1 writable: allocate missing
 * blocks and copy shared ones.  Host array pairs_out receives the (src, dst)
 * copy pairs (at most max_pairs).  start_pos may not leave a hole past the
 * table's end.  On PA_ERR_OUT_OF_BLOCKS or a too-small max_pairs nothing
 * changes.  The sequence length becomes max(length, start_pos + num_tokens). */
pa_status pa_bm_prepare_append(pa_block_manager* bm, int32_t seq, int32_t start_pos,
                               int32_t num_tokens, int32_t* pairs_out, int32_t max_pairs,
                               int32_t* num_pairs_out);
/* Host array row_out (max_blocks entries) receives the block table, -1 padded. */
pa_status pa_bm_block_table(const pa_block_manager* bm, int32_t seq, int32_t* row_out,
                            int32_t max_blocks, int32_t* num_blocks_out);
/* The block tables of num_seqs sequences in one call (an engine's per-iteration batch):
 * host array rows_out [num_seqs][max_blocks] receives row i = the table of seqs[i], -1
 * padded, as pa_bm_block_table would write it.  PA_ERR_INVALID_ARG for an unknown sequence
 * or a table longer than max_blocks (rows before it may have been written). */
pa_status pa_bm_block_tables(const pa_block_manager* bm, const int32_t* seqs, int32_t num_seqs,
                             int32_t* rows_out, int32_t max_blocks);
pa_status pa_bm_seq_len(const pa_block_manager* bm, int32_t seq, int32_t* len_out);
pa_status pa_bm_refcount(const pa_block_manager* bm, int32_t block, int32_t* refcount_out);
pa_status pa_bm_stats(const pa_block_manager* bm, pa_bm_stats_t* out);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_PA_H */

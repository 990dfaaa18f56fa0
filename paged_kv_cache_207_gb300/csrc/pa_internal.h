// pa_internal.h -- launch interfaces shared by the C ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "pa.h"

namespace pa {

constexpr int kBlockTokens = PA_BLOCK_SIZE;                     // tokens per block
constexpr int kPartTokens = PA_PARTITION_TOKENS;                // tokens per split-KV partition
constexpr int kPartBlocks = kPartTokens / kBlockTokens;         // blocks per partition
static_assert(kPartTokens % kBlockTokens == 0, "partition must be whole blocks");

inline int elem_bytes(pa_dtype t) { return t == PA_BF16 ? 2 : (t == PA_FP8_E4M3 ? 1 : 4); }

// Blocks per split-KV partition of the FP4 path (a multiple of kPartBlocks).
#ifndef PA_FP4_PARTITION_BLOCKS
#define PA_FP4_PARTITION_BLOCKS 128
#endif
constexpr int kFp4PartBlocks = PA_FP4_PARTITION_BLOCKS;
static_assert(PA_FP4_PARTITION_BLOCKS % 32 == 0, "FP4 partitions are whole 512-token units");

struct DecodeArgs {
    void* out;
    const void* q;
    const void* k_pool;
    const void* v_pool;
    const int32_t* block_tables;
    const int32_t* context_lens;
    int32_t* err;            // device error flag, may be null
    void* workspace;
    // decode with append (bf16 / f32 caches): the new K and V rows [num_seqs][Hkv][D],
    // written at position context_len - 1 by the decode kernel itself; null otherwise
    const void* k_new = nullptr;
    const void* v_new = nullptr;
    int new_min_pos = 0;     // a new row below this position (inside a shared prefix) is
                             // flagged PA_DEV_ERR_BAD_PREFIX and not written
    int num_seqs, num_q_heads, num_kv_heads, head_dim;
    int max_blocks, num_blocks;
    int grid_parts;          // partitions launched per (sequence, kv head)
    int part_stride;         // partitions reserved per (sequence, query head) in the workspace
    int part_blocks;         // blocks per split-KV partition of this path
    int first_part;          // leading partitions inside a prefix shared by every sequence
                             // (0: none); computed once per kv head by the prefix kernel
    float scale;
    pa_dtype dtype;
};

// Partitions a sequence of up to max_blocks blocks can span.
inline int decode_part_stride(int max_blocks) {
    return (max_blocks + kPartBlocks - 1) / kPartBlocks;
}

// Blocks per split-KV partition of pa_decode_attention for a head_dim (a multiple of
// kPartBlocks, so decode_part_stride bounds the partitions of every path).
#ifndef PA_D64_PARTITION_BLOCKS
#define PA_D64_PARTITION_BLOCKS 64
#endif
static_assert(PA_D64_PARTITION_BLOCKS % 32 == 0, "partitions are whole 512-token units");
inline int decode_part_blocks(int head_dim) {
    return head_dim == 64 ? PA_D64_PARTITION_BLOCKS : kPartBlocks;
}

// Shared-prefix decode: one prefix CTA covers this many decode partitions (its keys are
// that many times a partition's) when the prefix is a whole number of such groups, else
// one.  Its partial goes to the first workspace slot of the group; the merge reads only
// those slots of the prefix.
#ifndef PA_PREFIX_PART_MULT
#define PA_PREFIX_PART_MULT 2
#endif
inline int prefix_slot_mult(int first_part) {
    return first_part % PA_PREFIX_PART_MULT == 0 ? PA_PREFIX_PART_MULT : 1;
}

// Blocks per split-KV partition of the FP8 path: its tiles are half the bytes of
// bf16 ones, so a partition covers twice the tokens for the same bytes per CTA.
#ifndef PA_FP8_PARTITION_BLOCKS
#define PA_FP8_PARTITION_BLOCKS 64
#endif
constexpr int kFp8PartBlocks = PA_FP8_PARTITION_BLOCKS;
static_assert(kFp8PartBlocks % kPartBlocks == 0, "FP8 partitions are whole bf16 partitions");
size_t decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                              int max_blocks);

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

struct AppendArgs {
    void* k_pool;
    void* v_pool;
    const void* k_new;
    const void* v_new;
    const int32_t* block_tables;
    const int32_t* start_pos;
    const int32_t* cu_new;
    int32_t* err;
    int max_blocks, num_seqs, total_new, num_blocks, num_kv_heads, head_dim;
    pa_dtype dtype;
};
cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream);

struct CopyArgs {
    void* k_pool;
    void* v_pool;
    const int32_t* pairs;
    int32_t* err;
    int num_pairs, num_blocks, num_kv_heads, head_dim;
    pa_dtype dtype;
};
cudaError_t launch_copy(const CopyArgs& a, cudaStream_t stream);

}  // namespace pa

namespace pa {

// FP8 (E4M3) cache: per (block, kv head) a record of 16 * D code bytes
// (K: [D/16][16 slots][16]; V: [D][16 slots]) followed by 16 fp32 slot scales.
__host__ __device__ inline size_t fp8_record_bytes(int head_dim) { return (size_t)16 * head_dim + 64; }

cudaError_t launch_append_fp8(const AppendArgs& a, cudaStream_t stream);

struct PrefillArgs {
    void* out;
    const void* q;
    const void* k_pool;
    const void* v_pool;
    const int32_t* block_tables;
    const int32_t* start_pos;
    const int32_t* cu_q;
    int32_t* err;
    int num_seqs, max_chunk, num_q_heads, num_kv_heads, head_dim, max_blocks, num_blocks;
    float scale;
};
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);
// The prefix partitions [0, first_part) of a decode with a shared prefix, on tcgen05:
// writes their (o, max, sum) partials into the decode workspace for the merge.
// after_suffix: the suffix decode kernel was launched just before (see PParams).
cudaError_t launch_prefix_tc(const DecodeArgs& a, bool after_suffix, cudaStream_t stream);
cudaError_t launch_decode_fp8(const DecodeArgs& a, cudaStream_t stream);

// MXFP4 cache: per (block, kv head) a record of 8 * D code bytes then D / 2 E8M0 scale
// bytes (layout in pa.h).
__host__ __device__ inline size_t fp4_record_bytes(int head_dim) {
    return (size_t)8 * head_dim + (size_t)head_dim / 2;
}
cudaError_t launch_append_fp4(const AppendArgs& a, cudaStream_t stream);
cudaError_t launch_decode_fp4(const DecodeArgs& a, cudaStream_t stream);

}  // namespace pa

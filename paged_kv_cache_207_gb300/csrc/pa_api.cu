// pa_api.cu -- the C ABI entry points: argument checks, then kernel launches.
//
// Every check that needs only host values happens here and launches nothing
// on failure.  Checks that need device data happen in the kernels, which OR
// PA_DEV_ERR_* bits into the caller's flag and skip the offending element.
#include <cmath>
#include <cstdint>

#include "pa_internal.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

bool dtype_ok(pa_dtype t) { return t == PA_F32 || t == PA_BF16; }

}  // namespace

extern "C" {

const char* pa_status_string(pa_status s) {
    switch (s) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported configuration";
        case PA_ERR_CUDA: return "CUDA error";
        case PA_ERR_OUT_OF_BLOCKS: return "out of free blocks";
        case PA_ERR_SCRATCH_LIMIT: return "needs more than the built-in no-alloc scratch";
    }
    return "unknown status";
}

int32_t pa_abi_version(void) { return PA_ABI_VERSION; }

pa_status pa_append_kv(void* k_pool, void* v_pool, const void* k_new, const void* v_new,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* start_pos, const int32_t* cu_new_tokens, int32_t num_seqs,
                       int32_t total_new_tokens, int32_t num_blocks, int32_t num_kv_heads,
                       int32_t head_dim, pa_dtype dtype, int32_t* dev_err_flag, void* stream) {
    if (!dtype_ok(dtype)) return PA_ERR_INVALID_ARG;
    if (num_seqs < 0 || total_new_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 ||
        max_blocks_per_seq <= 0 || head_dim <= 0)
        return PA_ERR_INVALID_ARG;
    if ((head_dim * pa::elem_bytes(dtype)) % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0 && total_new_tokens != 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!k_pool || !v_pool || !block_tables || !start_pos || !cu_new_tokens) return PA_ERR_INVALID_ARG;
    if (total_new_tokens > 0 && (!k_new || !v_new)) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool) || (k_new && !aligned16(k_new)) ||
        (v_new && !aligned16(v_new)))
        return PA_ERR_INVALID_ARG;
    if ((long long)max_blocks_per_seq * pa::kBlockTokens > INT32_MAX) return PA_ERR_INVALID_ARG;
    pa::AppendArgs a;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.k_new = k_new;
    a.v_new = v_new;
    a.block_tables = block_tables;
    a.start_pos = start_pos;
    a.cu_new = cu_new_tokens;
    a.err = dev_err_flag;
    a.max_blocks = max_blocks_per_seq;
    a.num_seqs = num_seqs;
    a.total_new = total_new_tokens;
    a.num_blocks = num_blocks;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.dtype = dtype;
    return cuda_status(pa::launch_append(a, static_cast<cudaStream_t>(stream)));
}

pa_status pa_copy_block(void* k_pool, void* v_pool, const int32_t* src_dst_pairs,
                        int32_t num_pairs, int32_t num_blocks, int32_t num_kv_heads,
                        int32_t head_dim, pa_dtype dtype, int32_t* dev_err_flag, void* stream) {
    if (!dtype_ok(dtype) && dtype != PA_FP8_E4M3 && dtype != PA_FP4_E2M1) return PA_ERR_INVALID_ARG;
    if (num_pairs < 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return PA_ERR_INVALID_ARG;
    if (dtype == PA_FP4_E2M1 ? (head_dim % 32 != 0) : ((head_dim * pa::elem_bytes(dtype)) % 16 != 0))
        return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PA_OK;
    if (!k_pool || !v_pool || !src_dst_pairs) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool)) return PA_ERR_INVALID_ARG;
    pa::CopyArgs a;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.pairs = src_dst_pairs;
    a.err = dev_err_flag;
    a.num_pairs = num_pairs;
    a.num_blocks = num_blocks;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.dtype = dtype;
    return cuda_status(pa::launch_copy(a, static_cast<cudaStream_t>(stream)));
}

size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t max_blocks_per_seq) {
    if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        max_blocks_per_seq <= 0)
        return 0;
    return pa::decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                      max_blocks_per_seq);
}

// pa_decode_attention, and pa_append_decode_attention when k_new / v_new are given.
static pa_status decode_call(void* out, const void* q, const void* k_pool, const void* v_pool,
                             const void* k_new, const void* v_new, int32_t new_min_pos,
                             const int32_t* block_tables,
                             const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                             int32_t num_kv_heads, int32_t head_dim, int32_t max_blocks_per_seq,
                             int32_t max_context_len_hint, int32_t num_blocks, float scale,
                             pa_dtype dtype, void* workspace, size_t workspace_bytes,
                             int32_t* dev_err_flag, void* stream) {
    if (!dtype_ok(dtype)) return PA_ERR_INVALID_ARG;
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
        max_blocks_per_seq <= 0 || !std::isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (num_q_heads / num_kv_heads > 8) return PA_ERR_UNSUPPORTED;
    if ((long long)max_blocks_per_seq * pa::kBlockTokens > INT32_MAX) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return PA_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr)) return PA_ERR_INVALID_ARG;
    if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return PA_ERR_INVALID_ARG;
    const size_t need =
        pa::decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
        return PA_ERR_INVALID_ARG;

    const int cap = max_blocks_per_seq * pa::kBlockTokens;
    const int bound = (max_context_len_hint > 0 && max_context_len_hint < cap) ? max_context_len_hint : cap;
    pa::DecodeArgs a;
    a.out = out;
    a.q = q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.k_new = k_new;
    a.v_new = v_new;
    a.new_min_pos = new_min_pos;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.err = dev_err_flag;
    a.workspace = need > 0 ? workspace : nullptr;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.part_blocks = pa::decode_part_blocks(head_dim);
    a.grid_parts = (bound + a.part_blocks * pa::kBlockTokens - 1) / (a.part_blocks * pa::kBlockTokens);
    a.part_stride = pa::decode_part_stride(max_blocks_per_seq);
    a.first_part = 0;
    a.scale = scale;
    a.dtype = dtype;
    return cuda_status(pa::launch_decode(a, static_cast<cudaStream_t>(stream)));
}

pa_status pa_decode_attention(void* out, const void* q, const void* k_pool, const void* v_pool,
                              const int32_t* block_tables, const int32_t* context_lens,
                              int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t max_blocks_per_seq,
                              int32_t max_context_len_hint, int32_t num_blocks, float scale,
                              pa_dtype dtype, void* workspace, size_t workspace_bytes,
                              int32_t* dev_err_flag, void* stream) {
    return decode_call(out, q, k_pool, v_pool, nullptr, nullptr, 0, block_tables, context_lens,
                       num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                       max_context_len_hint, num_blocks, scale, dtype, workspace, workspace_bytes,
                       dev_err_flag, stream);
}

pa_status pa_append_decode_attention(void* out, const void* q, void* k_pool, void* v_pool,
                                     const void* k_new, const void* v_new,
                                     const int32_t* block_tables, const int32_t* context_lens,
                                     int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t max_blocks_per_seq,
                                     int32_t max_context_len_hint, int32_t num_blocks, float scale,
                                     pa_dtype dtype, void* workspace, size_t workspace_bytes,
                                     int32_t* dev_err_flag, void* stream) {
    if (num_seqs > 0 && (!k_new || !v_new)) return PA_ERR_INVALID_ARG;
    return decode_call(out, q, k_pool, v_pool, k_new, v_new, 0, block_tables, context_lens,
                       num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                       max_context_len_hint, num_blocks, scale, dtype, workspace, workspace_bytes,
                       dev_err_flag, stream);
}

// pa_decode_attention_shared_prefix, and its one-call form when k_new / v_new are given.
static pa_status shared_call(
    void* out, const void* q, const void* k_pool, const void* v_pool, const void* k_new,
    const void* v_new, const int32_t* block_tables, const int32_t* context_lens, int32_t num_seqs,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t max_blocks_per_seq,
    int32_t max_context_len_hint, int32_t num_blocks, float scale, pa_dtype dtype,
    int32_t shared_prefix_tokens, void* workspace, size_t workspace_bytes, int32_t* dev_err_flag,
    void* stream) {
    if (shared_prefix_tokens < 0 || shared_prefix_tokens % pa::kBlockTokens != 0)
        return PA_ERR_INVALID_ARG;
    if ((long long)shared_prefix_tokens > (long long)max_blocks_per_seq * pa::kBlockTokens)
        return PA_ERR_INVALID_ARG;
    const int first_part = shared_prefix_tokens / pa::kPartTokens;
    // nothing whole to share, or every context fits one partition: the ordinary path
    if (first_part == 0 || num_seqs <= 0 || max_blocks_per_seq <= pa::kPartBlocks)
        return decode_call(out, q, k_pool, v_pool, k_new, v_new, k_new ? shared_prefix_tokens : 0,
                           block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
                           head_dim, max_blocks_per_seq, max_context_len_hint, num_blocks, scale,
                           dtype, workspace, workspace_bytes, dev_err_flag, stream);
    if (dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 ||
        !std::isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (num_q_heads / num_kv_heads > 8) return PA_ERR_UNSUPPORTED;
    if ((long long)max_blocks_per_seq * pa::kBlockTokens > INT32_MAX) return PA_ERR_INVALID_ARG;
    if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return PA_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr)) return PA_ERR_INVALID_ARG;
    if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return PA_ERR_INVALID_ARG;
    const size_t need =
        pa::decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
    if (need == 0 || !workspace || workspace_bytes < need || !aligned16(workspace))
        return PA_ERR_INVALID_ARG;
    const int cap = max_blocks_per_seq * pa::kBlockTokens;
    int bound = (max_context_len_hint > 0 && max_context_len_hint < cap) ? max_context_len_hint : cap;
    if (bound < shared_prefix_tokens) bound = shared_prefix_tokens;
    pa::DecodeArgs a;
    a.out = out;
    a.q = q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.k_new = k_new;
    a.v_new = v_new;
    a.new_min_pos = k_new ? shared_prefix_tokens : 0;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.err = dev_err_flag;
    a.workspace = workspace;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.grid_parts = (bound + pa::kPartTokens - 1) / pa::kPartTokens;
    if (a.grid_parts < first_part) a.grid_parts = first_part;
    a.part_stride = pa::decode_part_stride(max_blocks_per_seq);
    a.part_blocks = pa::kPartBlocks;
    a.first_part = first_part;
    a.scale = scale;
    a.dtype = dtype;
    return cuda_status(pa::launch_decode(a, static_cast<cudaStream_t>(stream)));
}

pa_status pa_decode_attention_shared_prefix(
    void* out, const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
    const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t max_blocks_per_seq, int32_t max_context_len_hint, int32_t num_blocks,
    float scale, pa_dtype dtype, int32_t shared_prefix_tokens, void* workspace,
    size_t workspace_bytes, int32_t* dev_err_flag, void* stream) {
    return shared_call(out, q, k_pool, v_pool, nullptr, nullptr, block_tables, context_lens,
                       num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                       max_context_len_hint, num_blocks, scale, dtype, shared_prefix_tokens,
                       workspace, workspace_bytes, dev_err_flag, stream);
}

pa_status pa_append_decode_attention_shared_prefix(
    void* out, const void* q, void* k_pool, void* v_pool, const void* k_new, const void* v_new,
    const int32_t* block_tables, const int32_t* context_lens, int32_t num_seqs,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t max_blocks_per_seq,
    int32_t max_context_len_hint, int32_t num_blocks, float scale, pa_dtype dtype,
    int32_t shared_prefix_tokens, void* workspace, size_t workspace_bytes, int32_t* dev_err_flag,
    void* stream) {
    if (num_seqs > 0 && (!k_new || !v_new)) return PA_ERR_INVALID_ARG;
    return shared_call(out, q, k_pool, v_pool, k_new, v_new, block_tables, context_lens,
                       num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                       max_context_len_hint, num_blocks, scale, dtype, shared_prefix_tokens,
                       workspace, workspace_bytes, dev_err_flag, stream);
}

pa_status pa_append_kv_fp8(void* k_pool, void* v_pool, const void* k_new, const void* v_new,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* start_pos, const int32_t* cu_new_tokens,
                           int32_t num_seqs, int32_t total_new_tokens, int32_t num_blocks,
                           int32_t num_kv_heads, int32_t head_dim, int32_t* dev_err_flag,
                           void* stream) {
    if (num_seqs < 0 || total_new_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 ||
        max_blocks_per_seq <= 0)
        return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0 && total_new_tokens != 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!k_pool || !v_pool || !block_tables || !start_pos || !cu_new_tokens) return PA_ERR_INVALID_ARG;
    if (total_new_tokens > 0 && (!k_new || !v_new)) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool) || (k_new && !aligned16(k_new)) ||
        (v_new && !aligned16(v_new)))
        return PA_ERR_INVALID_ARG;
    if ((long long)max_blocks_per_seq * pa::kBlockTokens > INT32_MAX) return PA_ERR_INVALID_ARG;
    pa::AppendArgs a;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.k_new = k_new;
    a.v_new = v_new;
    a.block_tables = block_tables;
    a.start_pos = start_pos;
    a.cu_new = cu_new_tokens;
    a.err = dev_err_flag;
    a.max_blocks = max_blocks_per_seq;
    a.num_seqs = num_seqs;
    a.total_new = total_new_tokens;
    a.num_blocks = num_blocks;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.dtype = PA_FP8_E4M3;
    return cuda_status(pa::launch_append_fp8(a, static_cast<cudaStream_t>(stream)));
}

// pa_decode_attention_fp8, and its one-call form when k_new / v_new are given.
static pa_status fp8_call(void* out, const void* q, const void* k_pool, const void* v_pool,
                          const void* k_new, const void* v_new, const int32_t* block_tables,
                          const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t max_blocks_per_seq,
                          int32_t max_context_len_hint, int32_t num_blocks, float scale,
                          void* workspace, size_t workspace_bytes, int32_t* dev_err_flag,
                          void* stream) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
        max_blocks_per_seq <= 0 || !std::isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (num_q_heads / num_kv_heads > 8) return PA_ERR_UNSUPPORTED;
    if ((long long)max_blocks_per_seq * pa::kBlockTokens > INT32_MAX) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return PA_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr)) return PA_ERR_INVALID_ARG;
    if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return PA_ERR_INVALID_ARG;
    const size_t need =
        pa::decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
        return PA_ERR_INVALID_ARG;
    const int cap = max_blocks_per_seq * pa::kBlockTokens;
    const int bound = (max_context_len_hint > 0 && max_context_len_hint < cap) ? max_context_len_hint : cap;
    pa::DecodeArgs a;
    a.out = out;
    a.q = q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.k_new = k_new;
    a.v_new = v_new;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.err = dev_err_flag;
    a.workspace = need > 0 ? workspace : nullptr;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    const int fp8_part_tokens = pa::kFp8PartBlocks * pa::kBlockTokens;
    a.grid_parts = (bound + fp8_part_tokens - 1) / fp8_part_tokens;
    a.part_stride = pa::decode_part_stride(max_blocks_per_seq);   // >= the FP8 partitions used
    a.part_blocks = pa::kFp8PartBlocks;
    a.first_part = 0;
    a.scale = scale;
    a.dtype = PA_FP8_E4M3;
    return cuda_status(pa::launch_decode_fp8(a, static_cast<cudaStream_t>(stream)));
}

pa_status pa_decode_attention_fp8(void* out, const void* q, const void* k_pool, const void* v_pool,
                                  const int32_t* block_tables, const int32_t* context_lens,
                                  int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_blocks_per_seq,
                                  int32_t max_context_len_hint, int32_t num_blocks, float scale,
                                  void* workspace, size_t workspace_bytes, int32_t* dev_err_flag,
                                  void* stream) {
    return fp8_call(out, q, k_pool, v_pool, nullptr, nullptr, block_tables, context_lens, num_seqs,
                    num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, max_context_len_hint,
                    num_blocks, scale, workspace, workspace_bytes, dev_err_flag, stream);
}

pa_status pa_append_decode_attention_fp8(void* out, const void* q, void* k_pool, void* v_pool,
                                         const void* k_new, const void* v_new,
                                         const int32_t* block_tables, const int32_t* context_lens,
                                         int32_t num_seqs, int32_t num_q_heads,
                                         int32_t num_kv_heads, int32_t head_dim,
                                         int32_t max_blocks_per_seq, int32_t max_context_len_hint,
                                         int32_t num_blocks, float scale, void* workspace,
                                         size_t workspace_bytes, int32_t* dev_err_flag,
                                         void* stream) {
    if (num_seqs > 0 && (!k_new || !v_new)) return PA_ERR_INVALID_ARG;
    return fp8_call(out, q, k_pool, v_pool, k_new, v_new, block_tables, context_lens, num_seqs,
                    num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, max_context_len_hint,
                    num_blocks, scale, workspace, workspace_bytes, dev_err_flag, stream);
}

pa_status pa_append_kv_fp4(void* k_pool, void* v_pool, const void* k_new, const void* v_new,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* start_pos, const int32_t* cu_new_tokens,
                           int32_t num_seqs, int32_t total_new_tokens, int32_t num_blocks,
                           int32_t num_kv_heads, int32_t head_dim, int32_t* dev_err_flag,
                           void* stream) {
    if (num_seqs < 0 || total_new_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 ||
        max_blocks_per_seq <= 0)
        return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0 && total_new_tokens != 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!k_pool || !v_pool || !block_tables || !start_pos || !cu_new_tokens) return PA_ERR_INVALID_ARG;
    if (total_new_tokens > 0 && (!k_new || !v_new)) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool) || (k_new && !aligned16(k_new)) ||
        (v_new && !aligned16(v_new)))
        return PA_ERR_INVALID_ARG;
    if ((long long)max_blocks_per_seq * pa::kBlockTokens > INT32_MAX) return PA_ERR_INVALID_ARG;
    pa::AppendArgs a;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.k_new = k_new;
    a.v_new = v_new;
    a.block_tables = block_tables;
    a.start_pos = start_pos;
    a.cu_new = cu_new_tokens;
    a.err = dev_err_flag;
    a.max_blocks = max_blocks_per_seq;
    a.num_seqs = num_seqs;
    a.total_new = total_new_tokens;
    a.num_blocks = num_blocks;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.dtype = PA_FP4_E2M1;
    return cuda_status(pa::launch_append_fp4(a, static_cast<cudaStream_t>(stream)));
}

pa_status pa_decode_attention_fp4(void* out, const void* q, const void* k_pool, const void* v_pool,
                                  const int32_t* block_tables, const int32_t* context_lens,
                                  int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_blocks_per_seq,
                                  int32_t max_context_len_hint, int32_t num_blocks, float scale,
                                  void* workspace, size_t workspace_bytes, int32_t* dev_err_flag,
                                  void* stream) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
        max_blocks_per_seq <= 0 || !std::isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (num_q_heads / num_kv_heads > 8) return PA_ERR_UNSUPPORTED;
    if ((long long)max_blocks_per_seq * pa::kBlockTokens > INT32_MAX) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return PA_ERR_INVALID_ARG;
    const size_t need =
        pa::decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
        return PA_ERR_INVALID_ARG;
    const int cap = max_blocks_per_seq * pa::kBlockTokens;
    const int bound = (max_context_len_hint > 0 && max_context_len_hint < cap) ? max_context_len_hint : cap;
    pa::DecodeArgs a;
    a.out = out;
    a.q = q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.err = dev_err_flag;
    a.workspace = need > 0 ? workspace : nullptr;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    const int part_tokens = pa::kFp4PartBlocks * pa::kBlockTokens;
    a.grid_parts = (bound + part_tokens - 1) / part_tokens;
    a.part_stride = pa::decode_part_stride(max_blocks_per_seq);   // >= the FP4 partitions used
    a.part_blocks = pa::kFp4PartBlocks;
    a.first_part = 0;
    a.scale = scale;
    a.dtype = PA_FP4_E2M1;
    return cuda_status(pa::launch_decode_fp4(a, static_cast<cudaStream_t>(stream)));
}

pa_status pa_prefill_attention(void* out, const void* q, const void* k_pool, const void* v_pool,
                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                               const int32_t* start_pos, const int32_t* cu_q, int32_t num_seqs,
                               int32_t total_q, int32_t max_chunk, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                               float scale, pa_dtype dtype, int32_t* dev_err_flag, void* stream) {
    if (num_seqs < 0 || total_q < 0 || max_chunk < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_blocks <= 0 || max_blocks_per_seq <= 0 || !std::isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (dtype != PA_BF16) return dtype_ok(dtype) ? PA_ERR_UNSUPPORTED : PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (num_q_heads / num_kv_heads > 8) return PA_ERR_UNSUPPORTED;
    if ((long long)max_blocks_per_seq * pa::kBlockTokens > INT32_MAX) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0 || total_q == 0 || max_chunk == 0) return PA_OK;
    if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !start_pos || !cu_q)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return PA_ERR_INVALID_ARG;
    pa::PrefillArgs a;
    a.out = out;
    a.q = q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.block_tables = block_tables;
    a.start_pos = start_pos;
    a.cu_q = cu_q;
    a.err = dev_err_flag;
    a.num_seqs = num_seqs;
    a.max_chunk = max_chunk;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.scale = scale;
    return cuda_status(pa::launch_prefill(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

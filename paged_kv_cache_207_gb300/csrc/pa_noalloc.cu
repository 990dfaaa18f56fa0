// pa_noalloc.cu -- decode attention for callers that cannot allocate device memory.
//
// pa_decode_attention needs a scratch workspace for the split-KV partials and
// expects the caller to provide it.  Some callers cannot: a plugin running
// inside a host framework that owns all device memory and hands plugins no
// scratch buffer, or a latency-critical decode loop that must never call
// cudaMalloc because an allocation can synchronise the whole device.  For
// them this file keeps one fixed scratch array in the library itself (a
// file-scope __device__ array, created when the library's GPU code is loaded
// onto a device and held until the process exits) and runs the same decode
// kernels with it.  Nothing here allocates or frees memory.
#include <mutex>

#include "pa_internal.h"

namespace {

static_assert(PA_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size must be a multiple of 256");

// The shared scratch.  Every call uses as much of it as it needs and leaves its
// partial results behind; the next call overwrites them (the decode kernels never
// read partial results they did not write in the same call), so nothing in it
// needs clearing.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};   // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device.  In host code the
// symbol g_noalloc_scratch is only a host-side handle, so the address is taken
// once per device through the runtime, with that device current.
pa_status scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_attention_noalloc(
    void* out, const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
    const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t max_blocks_per_seq, int32_t max_context_len_hint, int32_t num_blocks,
    float scale, pa_dtype dtype, int32_t* dev_err_flag, void* stream) {
    const size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                 max_blocks_per_seq);
    if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    if (need > 0) {
        const pa_status st = scratch_for_current_device(&scratch);
        if (st != PA_OK) return st;
    }
    return pa_decode_attention(out, q, k_pool, v_pool, block_tables, context_lens, num_seqs,
                               num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                               max_context_len_hint, num_blocks, scale, dtype, scratch,
                               need > 0 ? (size_t)PA_NOALLOC_SCRATCH_BYTES : 0, dev_err_flag,
                               stream);
}

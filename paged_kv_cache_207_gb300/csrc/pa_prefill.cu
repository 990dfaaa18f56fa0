// pa_prefill.cu -- causal attention of a chunk of new tokens over the paged cache
// (chunked prefill).
//
// A chunk of n_s tokens of sequence s sits at positions start_pos[s] .. +n_s-1
// and has already been appended to the pools (pa_append_kv takes several rows
// per sequence).  Each chunk token at position p attends over positions 0 .. p
// of its own sequence (spindle, "Two bugs worth recording": prefill at layer 0
// must see the explicit positions, not an inferred length of zero; chunked
// prefill is one of the engine parts Slipstream lists in "Horizon").
//
// Work split: CTA = (query tile, kv head, sequence).  Rows are (chunk token,
// query head of the kv head) pairs, token-major, TQ = 64 / G tokens per tile;
// each of the 4 consumer warps owns 16 rows.  A producer warp streams the
// sequence's K/V tiles (blocks 0 .. the tile's last position / 16) through a
// ring shared by the CTA; scores Q K^T and P.V run on the tensor cores
// (mma.sync bf16, FlashAttention-2 register layout: P stays in registers as
// the A operand, V is read with ldmatrix.trans), with the causal mask applied
// per row.  Later tiles (which read more blocks) are scheduled first.
#include <cuda_bf16.h>

#include <cmath>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

namespace {

constexpr uint64_t kWaitLimitNs = 200000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kConsumers = 4;
constexpr int kRows = 16 * kConsumers;        // rows per CTA
#ifndef PA_PREFILL_STAGES
#define PA_PREFILL_STAGES 4
#endif
constexpr int kStages = PA_PREFILL_STAGES;

struct PParams {
    void* out;
    const void* q;
    const char* k_pool;
    const char* v_pool;
    const int32_t* tables;
    const int32_t* start_pos;
    const int32_t* cu_q;
    int32_t* err;
    int Hq, Hkv, G, TQ, max_blocks, num_blocks;
    float scale_log2;
};

__device__ __forceinline__ void raise_flag(int32_t* err, int bits) {
    if (err) atomicOr(err, bits);
}

template <int D>
constexpr int prefill_smem() { return kStages * 2 * kBlockTokens * D * 2 + 2 * kStages * 8; }

template <int D>
__global__ void __launch_bounds__((kConsumers + 1) * 32, 1)
prefill_bf16_kernel(const PParams p) {
    constexpr int TILE = kBlockTokens * D * 2;
    constexpr int KS = D / 16;
    constexpr int NT = D / 8;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, c = lane & 3;
    const int qt = gridDim.x - 1 - blockIdx.x;            // later (longer) tiles first
    const int kvh = blockIdx.y, s = blockIdx.z;
    const int q0 = __ldg(p.cu_q + s);
    const int n = __ldg(p.cu_q + s + 1) - q0;
    const int i0 = qt * p.TQ;
    if (i0 >= n) return;
    const int start = __ldg(p.start_pos + s);
    const int i_end = min(n, i0 + p.TQ);
    const int p_last = start + i_end - 1;                 // last position this tile attends to
    if (start < 0 || p_last >= p.max_blocks * kBlockTokens) {
        if (threadIdx.x == 0 && kvh == 0) raise_flag(p.err, PA_DEV_ERR_BAD_POS);
        return;
    }
    const int nblk = p_last / kBlockTokens + 1;
    const int32_t* trow = p.tables + (size_t)s * p.max_blocks;

    const uint32_t ring0 = smem_u32(smem);
    const uint32_t full0 = ring0 + kStages * 2 * TILE, empty0 = full0 + kStages * 8;
    if (threadIdx.x == 0) {
#pragma unroll
        for (int st = 0; st < kStages; ++st) {
            mbar_init(full0 + st * 8, 1);
            mbar_init(empty0 + st * 8, kConsumers);
        }
        fence_proxy_async_smem();
    }
    __syncthreads();

    if (warp == kConsumers) {       // ---- producer warp
        if (lane == 0) {
            grid_dependency_wait();   // the chunk's own K/V come from the append before
            grid_launch_dependents();
            const uint64_t pol = l2_policy_evict_first();
            for (int i = 0; i < nblk; ++i) {
                const int st = i % kStages;
                if (i >= kStages &&
                    !mbar_wait_bounded(empty0 + st * 8, ((i / kStages) - 1) & 1, kWaitLimitNs)) {
                    raise_flag(p.err, PA_DEV_ERR_TIMEOUT);
                    break;
                }
                int32_t blk = __ldg(trow + i);
                if (blk < 0 || blk >= p.num_blocks) {
                    raise_flag(p.err, PA_DEV_ERR_BAD_BLOCK);
                    blk = -1;
                }
                const uint32_t bar = full0 + st * 8;
                if (blk >= 0) {
                    const size_t off = ((size_t)blk * p.Hkv + kvh) * (size_t)TILE;
                    fence_proxy_async_smem();
                    mbar_arrive_expect_tx(bar, 2 * TILE);
                    bulk_g2s(ring0 + st * 2 * TILE, p.k_pool + off, TILE, bar, pol);
                    bulk_g2s(ring0 + st * 2 * TILE + TILE, p.v_pool + off, TILE, bar, pol);
                } else {
                    mbar_arrive_expect_tx(bar, 0);   // complete the phase; the flag is set
                }
            }
        }
        return;
    }

    // ---- consumer warps: rows rr0 = 16 w + r and rr1 = rr0 + 8 of the tile
    const int rr0 = warp * 16 + r, rr1 = rr0 + 8;
    const int tl0 = rr0 / p.G, g0 = rr0 - tl0 * p.G;
    const int tl1 = rr1 / p.G, g1 = rr1 - tl1 * p.G;
    const bool v0 = tl0 < p.TQ && i0 + tl0 < n, v1 = tl1 < p.TQ && i0 + tl1 < n;
    // positions; rows outside the tile see every token (finite, never written)
    const int pos0 = v0 ? start + i0 + tl0 : 0x7fffffff;
    const int pos1 = v1 ? start + i0 + tl1 : 0x7fffffff;
    uint32_t qa[KS][4];
    {
        const uint16_t* qrow0 = reinterpret_cast<const uint16_t*>(p.q) +
                                ((size_t)(q0 + i0 + (v0 ? tl0 : 0)) * p.Hq + (size_t)kvh * p.G + (v0 ? g0 : 0)) * D;
        const uint16_t* qrow1 = reinterpret_cast<const uint16_t*>(p.q) +
                                ((size_t)(q0 + i0 + (v1 ? tl1 : 0)) * p.Hq + (size_t)kvh * p.G + (v1 ? g1 : 0)) * D;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            qa[kk][0] = v0 ? __ldg(reinterpret_cast<const uint32_t*>(qrow0 + 16 * kk + 2 * c)) : 0u;
            qa[kk][1] = v1 ? __ldg(reinterpret_cast<const uint32_t*>(qrow1 + 16 * kk + 2 * c)) : 0u;
            qa[kk][2] = v0 ? __ldg(reinterpret_cast<const uint32_t*>(qrow0 + 16 * kk + 8 + 2 * c)) : 0u;
            qa[kk][3] = v1 ? __ldg(reinterpret_cast<const uint32_t*>(qrow1 + 16 * kk + 8 + 2 * c)) : 0u;
        }
    }
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    const int km = lane >> 3;
    const uint32_t k_lane = (uint32_t)((((km & 1) * 16) + (km >> 1) * 8 + (lane & 7)) * 16);
    const uint32_t v_lane = (uint32_t)((((km >> 1) * 16) + (km & 1) * 8 + (lane & 7)) * 16);
    bool failed = false;
    for (int i = 0; i < nblk; ++i) {
        const int st = i % kStages;
        if (!mbar_wait_bounded(full0 + st * 8, (i / kStages) & 1, kWaitLimitNs)) {
            failed = true;
            break;
        }
        const int tok0 = i * kBlockTokens;
        const uint32_t kt = ring0 + st * 2 * TILE, vt = kt + TILE;
        float sc[2][4], sx[2][4];
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[t][e] = sx[t][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(kt + kk * 512 + k_lane, b0, b1, b2, b3);
            float (&a)[2][4] = (kk & 1) ? sx : sc;
            mma_bf16_16816(a[0], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
            mma_bf16_16816(a[1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
        }
        // scale and the causal mask: element (row, token t) is kept when t <= row position
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int ta = tok0 + 8 * t + 2 * c;
            sc[t][0] = ta <= pos0 ? (sc[t][0] + sx[t][0]) * p.scale_log2 : -INFINITY;
            sc[t][1] = ta + 1 <= pos0 ? (sc[t][1] + sx[t][1]) * p.scale_log2 : -INFINITY;
            sc[t][2] = ta <= pos1 ? (sc[t][2] + sx[t][2]) * p.scale_log2 : -INFINITY;
            sc[t][3] = ta + 1 <= pos1 ? (sc[t][3] + sx[t][3]) * p.scale_log2 : -INFINITY;
        }
        float bm0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
        float bm1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 1));
        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 2));
        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 1));
        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 2));
        // every kept row sees token 0 in block 0, so its maximum is finite from then on
        const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
        const float al0 = mn0 == -INFINITY ? 1.f : fast_exp2(m0 - mn0);
        const float al1 = mn1 == -INFINITY ? 1.f : fast_exp2(m1 - mn1);
        const float e0 = mn0 == -INFINITY ? 0.f : mn0, e1 = mn1 == -INFINITY ? 0.f : mn1;
        m0 = mn0;
        m1 = mn1;
        const uint32_t a0 = pack_bf16x2(fast_exp2(sc[0][0] - e0), fast_exp2(sc[0][1] - e0));
        const uint32_t a1 = pack_bf16x2(fast_exp2(sc[0][2] - e1), fast_exp2(sc[0][3] - e1));
        const uint32_t a2 = pack_bf16x2(fast_exp2(sc[1][0] - e0), fast_exp2(sc[1][1] - e0));
        const uint32_t a3 = pack_bf16x2(fast_exp2(sc[1][2] - e1), fast_exp2(sc[1][3] - e1));
        l0 = l0 * al0 + (bf16_lo_to_f32(a0) + bf16_hi_to_f32(a0) + bf16_lo_to_f32(a2) + bf16_hi_to_f32(a2));
        l1 = l1 * al1 + (bf16_lo_to_f32(a1) + bf16_hi_to_f32(a1) + bf16_lo_to_f32(a3) + bf16_hi_to_f32(a3));
        if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
            for (int nd = 0; nd < NT; ++nd) {
                o[nd][0] *= al0; o[nd][1] *= al0; o[nd][2] *= al1; o[nd][3] *= al1;
            }
        }
        // V rows past the tile's last position may hold anything (even NaN): zero them
        uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
        if (tok0 + kBlockTokens - 1 > p_last) {
            mlo = (tok0 + 2 * c <= p_last ? 0x0000ffffu : 0u) | (tok0 + 2 * c + 1 <= p_last ? 0xffff0000u : 0u);
            mhi = (tok0 + 8 + 2 * c <= p_last ? 0x0000ffffu : 0u) |
                  (tok0 + 9 + 2 * c <= p_last ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int nd = 0; nd < NT; nd += 2) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4_trans(vt + nd * 256 + v_lane, b0, b1, b2, b3);
            mma_bf16_16816(o[nd], a0, a1, a2, a3, b0 & mlo, b1 & mhi);
            mma_bf16_16816(o[nd + 1], a0, a1, a2, a3, b2 & mlo, b3 & mhi);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + st * 8);
    }
    if (failed && lane == 0) raise_flag(p.err, PA_DEV_ERR_TIMEOUT);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    auto store_row = [&](bool valid, int tl, int g, float l, int half) {
        if (!valid) return;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) +
                              ((size_t)(q0 + i0 + tl) * p.Hq + (size_t)kvh * p.G + g) * D;
#pragma unroll
        for (int nd = 0; nd < NT; ++nd) {
            const uint32_t v = pack_bf16x2(o[nd][2 * half] * inv, o[nd][2 * half + 1] * inv);
            *reinterpret_cast<uint32_t*>(orow + 8 * nd + 2 * c) = v;
        }
    };
    store_row(v0, tl0, g0, l0, 0);
    store_row(v1, tl1, g1, l1, 1);
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int D>
cudaError_t launch_for_dim(const PParams& pp, int num_seqs, int max_chunk, cudaStream_t stream) {
    auto k = prefill_bf16_kernel<D>;
    constexpr int smem = prefill_smem<D>();
    cudaError_t e = set_smem(k, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((max_chunk + pp.TQ - 1) / pp.TQ, pp.Hkv, num_seqs);
    cfg.blockDim = dim3((kConsumers + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, pp);
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
    PParams pp;
    pp.out = a.out;
    pp.q = a.q;
    pp.k_pool = static_cast<const char*>(a.k_pool);
    pp.v_pool = static_cast<const char*>(a.v_pool);
    pp.tables = a.block_tables;
    pp.start_pos = a.start_pos;
    pp.cu_q = a.cu_q;
    pp.err = a.err;
    pp.Hq = a.num_q_heads;
    pp.Hkv = a.num_kv_heads;
    pp.G = a.num_q_heads / a.num_kv_heads;
    pp.TQ = kRows / pp.G;
    pp.max_blocks = a.max_blocks;
    pp.num_blocks = a.num_blocks;
    pp.scale_log2 = a.scale * kLog2e;
    if (a.head_dim == 64) return launch_for_dim<64>(pp, a.num_seqs, a.max_chunk, stream);
    return launch_for_dim<128>(pp, a.num_seqs, a.max_chunk, stream);
}

}  // namespace pa

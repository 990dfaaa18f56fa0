// pa_decode.cu -- single-token decode attention over the block-paged KV cache.
//
// What is computed (spindle, "Paging" and "Why write the forward pass"): for
// every sequence s and query head h, attention of q[s][h] over the keys and
// values of positions 0 .. context_lens[s]-1, found through the sequence's
// block table; query head h reads kv head h / G (G = Hq / Hkv).
//
// How (split-KV after the Flash-Decoding entry of the mlsystems list; the
// bandwidth bound after Slipstream, "The thesis" / Fig. 01):
//   grid = (partition j, kv head, sequence).  A CTA owns one partition of
//   PA_PARTITION_TOKENS tokens of one (sequence, kv head) and serves all G
//   query heads that read it, so each K/V byte leaves HBM once.
//   Each warp streams every NW-th block of the partition through a private
//   ring of NST shared-memory stages: lane 0 issues two 1-D bulk copies (the
//   TMA engine) per block -- the contiguous K tile and V tile of that
//   (block, kv head) -- completing on the stage's mbarrier.
//   bf16: scores S[16 tokens][8 heads] = K_tile (16 x D) * Q^T (D x 8) on the
//   tensor cores (mma.m16n8k16, tokens on M, the G query heads padded to 8 on
//   N), fp32 online softmax in registers, P transposed in-register with
//   movmatrix, then O^T[D][8] += V^T (D x 16) * P (16 x 8).
//   fp32: the same pipeline with CUDA-core FMAs (no tensor-core path reaches
//   fp32 accuracy).
//   At the end the warps of a CTA merge through shared memory; a sequence
//   with one partition writes `out` directly, otherwise the partition's
//   unnormalised output and its (max, sum) go to the workspace and a second
//   kernel merges partitions with log-sum-exp weights in fixed order.
#include <cuda_bf16.h>

#include <cmath>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

namespace {

constexpr uint64_t kWaitLimitNs = 200000000ull;   // 200 ms: a real tile copy takes microseconds
constexpr float kLog2e = 1.4426950408889634f;

struct KParams {
    void* out;
    const void* q;
    const char* k_pool;
    const char* v_pool;
    const int32_t* tables;
    const int32_t* lens;
    float* part_o;      // [S*Hq][part_stride][D]
    float2* part_ml;    // [S*Hq][part_stride] : (max in log2 units, sum)
    // decode with append: each sequence's new K and V rows ([S][Hkv][D]), written at
    // position L - 1 (into the pools above) before it is read; null for a plain decode
    const char* k_new;
    const char* v_new;
    int new_min_pos;    // with a shared prefix: the first position a new row may take
    int32_t* err;
    int Hq, Hkv, G, max_blocks, num_blocks;
    int grid_parts;     // partitions covered per (sequence, kv head): first_part + launched
    int part_stride;
    int first_part;     // partitions below this are a shared prefix done by the prefix kernel
    int prefix_stride;  // ... which wrote a partial into every prefix_stride-th of their slots
    int part_blocks;    // blocks per split-KV partition (a fixed constant of each path)
    float scale_log2;   // scale * log2(e): scores live in log2 units
    // shared-prefix suffix kernel launched after the prefix kernel, which starts it only
    // once every kernel before the prefix (the append) has finished: it needs no wait of
    // its own, and CTA 0 waits for the prefix grid before exiting so that this grid never
    // completes before it
    int after_prefix;
};

__device__ __forceinline__ bool first_cta() {
    return blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
}

// Rescale the output accumulators only in blocks where a running maximum moved
// (any lane of the warp); after the first blocks of a partition it rarely does.
#ifndef PA_LAZY_RESCALE
#define PA_LAZY_RESCALE 1
#endif
constexpr bool kLazyRescale = PA_LAZY_RESCALE != 0;

__device__ __forceinline__ void raise_flag(int32_t* err, int bits) {
    if (err) atomicOr(err, bits);
}

// Context length clamped to the table's capacity; flags bad values once per
// sequence (from the CTA of partition 0, kv head 0).
__device__ __forceinline__ int clamped_len(const KParams& p, int s) {
    int L = __ldg(p.lens + s);
    const int cap = p.max_blocks * kBlockTokens;
    const bool leader = blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0;
    if (L < 0 || L > cap) {
        if (leader) raise_flag(p.err, PA_DEV_ERR_BAD_POS);
        L = L < 0 ? 0 : cap;
    }
    return L;
}

// True when some CTA has already given up on a copy: later CTAs return at once
// so that a broken pipeline cannot keep the GPU busy for long.
__device__ __forceinline__ bool aborted(const int32_t* err) {
    if (!err) return false;
    return (*reinterpret_cast<const volatile int32_t*>(err) & PA_DEV_ERR_TIMEOUT) != 0;
}

__device__ __forceinline__ int num_parts(int L, int part_blocks) {
    const int pt = part_blocks * kBlockTokens;
    return L > 0 ? (L + pt - 1) / pt : 1;
}

// Per-warp ring of NST stages, each holding one K tile and one V tile.
template <int TILE, int NW, int NST>
struct Ring {
    uint32_t stage0;   // shared address of this warp's stage 0
    uint32_t bar0;     // shared address of this warp's first mbarrier
    __device__ __forceinline__ uint32_t k(int st) const { return stage0 + st * 2 * TILE; }
    __device__ __forceinline__ uint32_t v(int st) const { return stage0 + st * 2 * TILE + TILE; }
    __device__ __forceinline__ uint32_t bar(int st) const { return bar0 + st * 8; }
};

// Shared-memory bytes of the stage rings plus the barriers.
template <int TILE, int NW, int NST>
constexpr int ring_smem_bytes() { return NW * NST * 2 * TILE + NW * NST * 8; }

// Decode with append, f32 kernel: the new token's K and V rows go to position L - 1 of the
// sequence (the bytes pa_append_kv writes there), written by one warp of the CTA of the
// partition that holds it, before the CTA issues its copies.  Each lane stores 16-byte
// pieces and fences them to the async proxy; the caller's CTA barrier then orders the
// stores before the bulk copies that read the block.  An invalid table entry is left to
// the copy issue, which flags it; a length past the table (flagged, clamped) writes nothing.
template <int ROWB>   // bytes of one (token, kv head) row
__device__ __forceinline__ void write_new_token(const KParams& p, int s, int kvh, int L,
                                                const int32_t* trow, int lane) {
    constexpr int PIECES = ROWB / 16;
    if (__ldg(p.lens + s) != L) return;
    const int pos = L - 1;
    if (pos < p.new_min_pos) {            // inside a shared prefix: every sequence's block
        if (lane == 0) raise_flag(p.err, PA_DEV_ERR_BAD_PREFIX);
        return;
    }
    const int32_t blk = __ldg(trow + pos / kBlockTokens);
    if (blk < 0 || blk >= p.num_blocks) return;
    for (int t = lane; t < 2 * PIECES; t += 32) {
        const bool is_v = t >= PIECES;
        const int ch = is_v ? t - PIECES : t;
        const size_t src = (((size_t)s * p.Hkv + kvh) * PIECES + ch) * 16;
        const size_t dst =
            ((((size_t)blk * p.Hkv + kvh) * PIECES + ch) * kBlockTokens + pos % kBlockTokens) * 16;
        // (the new rows may come from the kernel before: a plain load after the grid wait)
        const uint4 v = *reinterpret_cast<const uint4*>((is_v ? p.v_new : p.k_new) + src);
        // the pools are writable when k_new is given (the caller's pointers are not const)
        *reinterpret_cast<uint4*>(const_cast<char*>(is_v ? p.v_pool : p.k_pool) + dst) = v;
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Decode with append, bf16 kernel: the warp whose copies read the new position's block
// loads its lane's 16-byte piece of the new K or V row (lanes 0 .. P-1: K, P .. 2P-1: V),
// stores it into the pool for later steps (no fence: this grid's copies never need it
// there), and keeps it to patch into its own copy of the block once that lands.  Returns
// the piece's byte offset within a (block, kv head) tile, or -1 (no piece for this lane,
// an invalid table entry -- flagged by the copy issue -- or a length past the table).
template <int D>
__device__ __forceinline__ int new_token_piece(const KParams& p, int s, int kvh, int L,
                                               const int32_t* trow, int lane, uint4& piece,
                                               bool& is_v) {
    constexpr int PIECES = D / 8;                 // 16-byte pieces of one bf16 row
    if (__ldg(p.lens + s) != L) return -1;
    const int pos = L - 1;
    if (pos < p.new_min_pos) {            // inside a shared prefix: every sequence's block
        if (lane == 0) raise_flag(p.err, PA_DEV_ERR_BAD_PREFIX);
        return -1;
    }
    if (lane >= 2 * PIECES) return -1;
    const int32_t blk = __ldg(trow + pos / kBlockTokens);
    if (blk < 0 || blk >= p.num_blocks) return -1;
    is_v = lane >= PIECES;
    const int ch = is_v ? lane - PIECES : lane;
    const size_t src = (((size_t)s * p.Hkv + kvh) * PIECES + ch) * 16;
    // (the new rows may come from the kernel before: a plain load after the grid wait)
    piece = *reinterpret_cast<const uint4*>((is_v ? p.v_new : p.k_new) + src);
    const int off = (ch * kBlockTokens + pos % kBlockTokens) * 16;
    // the pools are writable when k_new is given (the caller's pointers are not const)
    *reinterpret_cast<uint4*>(const_cast<char*>(is_v ? p.v_pool : p.k_pool) +
                              ((size_t)blk * p.Hkv + kvh) * (size_t)(kBlockTokens * D * 2) + off) = piece;
    return off;
}

// Decode with append, FP8 kernel: as new_token_piece, with the row quantised the way the FP8
// append does it (fp8_quantize_rows, by the whole warp) and written into the pool records
// (fp8_put_row).  Returns the new row's slot in its block, or -1 (invalid table entry --
// flagged by the copy issue --, a length past the table, or a row inside a shared prefix).
template <int D>
__device__ __forceinline__ int new_token_fp8(const KParams& p, int s, int kvh, int L,
                                             const int32_t* trow, int lane, uint32_t& kc,
                                             uint32_t& vc, float& ks, float& vs) {
    if (__ldg(p.lens + s) != L) return -1;
    const int pos = L - 1;
    if (pos < p.new_min_pos) {
        if (lane == 0) raise_flag(p.err, PA_DEV_ERR_BAD_PREFIX);
        return -1;
    }
    const int32_t blk = __ldg(trow + pos / kBlockTokens);
    if (blk < 0 || blk >= p.num_blocks) return -1;
    const size_t src = ((size_t)s * p.Hkv + kvh) * D * 2;
    fp8_quantize_rows<D>(p.k_new + src, p.v_new + src, lane, kc, vc, ks, vs);
    const size_t rec = ((size_t)blk * p.Hkv + kvh) * fp8_record_bytes(D);
    // the pools are writable when k_new is given (the caller's pointers are not const)
    fp8_put_row<D>(const_cast<char*>(p.k_pool) + rec, const_cast<char*>(p.v_pool) + rec, lane,
                   pos % kBlockTokens, kc, vc, ks, vs);
    return pos % kBlockTokens;
}

// Cross-warp merge of one partition (both element types).  Every warp holds,
// per padded head g < 8: running max m (log2 units), sum l and unnormalised
// output row o[g][:] already written to shared memory by the caller.
// A CTA in which a copy wait gave up (`failed`) writes NaN instead: the result is
// incomplete, and it must not pass for a correct one even when no error flag was given.
template <int D, int NW, typename OutT>
__device__ __forceinline__ void merge_and_store(const KParams& p, const float* sm_o,
                                                const float* sm_m, const float* sm_l, int s,
                                                int kvh, int j, int nparts, bool failed) {
    constexpr int OS = D + 4;
    for (int idx = threadIdx.x; idx < p.G * D; idx += NW * 32) {
        const int g = idx / D, d = idx - (idx / D) * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_m[w * 8 + g]);
        float acc = 0.f, lsum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float wt = fast_exp2(sm_m[w * 8 + g] - M);
                acc += wt * sm_o[(w * 8 + g) * OS + d];
                lsum += wt * sm_l[w * 8 + g];
            }
        }
        if (failed) M = acc = lsum = __int_as_float(0x7fc00000);
        const size_t row = (size_t)s * p.Hq + (size_t)kvh * p.G + g;
        if (nparts == 1 && p.first_part == 0) {
            const float v = failed ? acc : (lsum > 0.f ? acc / lsum : 0.f);
            if constexpr (sizeof(OutT) == 2)
                reinterpret_cast<__nv_bfloat16*>(p.out)[row * D + d] = __float2bfloat16_rn(v);
            else
                reinterpret_cast<float*>(p.out)[row * D + d] = v;
        } else {
            p.part_o[(row * p.part_stride + j) * D + d] = acc;
            if (d == 0) p.part_ml[row * p.part_stride + j] = make_float2(M, lsum);
        }
    }
}

// ---------------------------------------------------------------------------
// bf16 kernel: tensor-core scores and P.V
// ---------------------------------------------------------------------------
template <int D, int NW, int NST>
__global__ void __launch_bounds__(NW * 32)
decode_bf16_kernel(const KParams p) {
    constexpr int TILE = kBlockTokens * D * 2;   // bytes of one (block, kv head) tile
    constexpr int KS = D / 16;                   // k-steps of the score MMA = m-tiles of P.V
    extern __shared__ __align__(128) uint8_t smem[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, c = lane & 3;
    const int j = blockIdx.x + p.first_part, kvh = blockIdx.y, s = blockIdx.z;
    const int32_t* trow = p.tables + (size_t)s * p.max_blocks;

    // This warp's first NST table entries are read before the context length is known,
    // so both loads are in flight together (entries past the table row are not read).
    int32_t first_blk[NST];
#pragma unroll
    for (int i = 0; i < NST; ++i) {
        const int b = j * p.part_blocks + warp + i * NW;
        first_blk[i] = b < p.max_blocks ? __ldg(trow + b) : -1;
    }
    const int L = clamped_len(p, s);
    const int nparts = num_parts(L, p.part_blocks);
    if (blockIdx.x == 0 && kvh == 0 && threadIdx.x == 0 && nparts > p.grid_parts)
        raise_flag(p.err, PA_DEV_ERR_HINT);
    if (j >= nparts || aborted(p.err)) {
        // a dependent grid never completes before the one it follows
        if (!p.after_prefix || first_cta()) grid_dependency_wait();
        return;
    }

    const int blk0 = j * p.part_blocks;                            // first logical block
    const int tok_end = min(L, (j + 1) * p.part_blocks * kBlockTokens);           // one past the last token
    const int nblk = (tok_end - blk0 * kBlockTokens + kBlockTokens - 1) / kBlockTokens;
    const int nb_w = nblk > warp ? (nblk - warp + NW - 1) / NW : 0;

    Ring<TILE, NW, NST> ring;
    ring.stage0 = smem_u32(smem) + warp * NST * 2 * TILE;
    ring.bar0 = smem_u32(smem) + NW * NST * 2 * TILE + warp * NST * 8;
    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < NST; ++st) mbar_init(ring.bar(st), 1);
        fence_proxy_async_smem();
    }
    __syncwarp();

    // Everything above reads only the tables and the lengths, which no kernel of this
    // library writes.  The pools (an append) and the query (any earlier call's output)
    // may still be being written by the previous kernel: wait for it (after the prefix
    // kernel, that kernel's start already did).
    if (!p.after_prefix) grid_dependency_wait();
    grid_launch_dependents();

    const uint64_t pol = l2_policy_evict_first();
    auto issue_blk = [&](int32_t blk, int st) -> bool {
        const bool ok = blk >= 0 && blk < p.num_blocks;
        if (lane == 0) {
            if (ok) {
                const size_t off = ((size_t)blk * p.Hkv + kvh) * (size_t)TILE;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(ring.bar(st), 2 * TILE);
                bulk_g2s(ring.k(st), p.k_pool + off, TILE, ring.bar(st), pol);
                bulk_g2s(ring.v(st), p.v_pool + off, TILE, ring.bar(st), pol);
            } else {
                raise_flag(p.err, PA_DEV_ERR_BAD_BLOCK);
            }
        }
        return ok;
    };

    float m0 = -INFINITY, m1 = -INFINITY;   // running max of heads 2c, 2c+1 (log2 units)
    float l0 = 0.f, l1 = 0.f;               // this thread's share of the running sums
    float o[KS][4];
#pragma unroll
    for (int i = 0; i < KS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    uint32_t issued = 0, phase = 0;
    bool failed = false;
#pragma unroll
    for (int i = 0; i < NST; ++i)
        if (i < nb_w && issue_blk(first_blk[i], i)) issued |= 1u << i;

    // Decode with append: the new position is in this partition's last block (or, past the
    // grid's hint, in none of this CTA's blocks); the warp that reads that block writes the
    // new row to the pools while its first tiles are in flight, and patches it into its copy
    // of the block at iteration patch_it.
    uint4 piece = make_uint4(0u, 0u, 0u, 0u);
    bool piece_v = false;
    int piece_off = -1, patch_it = -1;
    if (p.k_new && L > 0 && j == min(nparts, p.grid_parts) - 1 && warp == (nblk - 1) % NW) {
        piece_off = new_token_piece<D>(p, s, kvh, L, trow, lane, piece, piece_v);
        if (j == nparts - 1) patch_it = (nblk - 1) / NW;
    }

    // Query fragments (B operand, k = dim, n = query head of the group), loaded while
    // the first tiles are in flight.
    uint32_t qb[KS][2];
    {
        const bool live = r < p.G;
        const uint16_t* qrow = reinterpret_cast<const uint16_t*>(p.q) +
                               ((size_t)s * p.Hq + (size_t)kvh * p.G + (live ? r : 0)) * D;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            qb[kk][0] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * c)) : 0u;
            qb[kk][1] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 8 + 2 * c)) : 0u;
        }
    }

    // ldmatrix row addresses: K tile k-step kk reads 512 contiguous bytes.
    const uint32_t k_lane = lane * 16;
    const int vm = lane >> 3;
    const uint32_t v_lane = (uint32_t)(((vm & 1) * 16 + (vm >> 1) * 8 + (lane & 7)) * 16);

    for (int i = 0; i < nb_w; ++i) {
        const int st = i % NST;
        if ((issued >> st) & 1u) {
            if (!mbar_wait_bounded(ring.bar(st), (phase >> st) & 1u, kWaitLimitNs)) {
                failed = true;
                break;
            }
            phase ^= 1u << st;
            issued &= ~(1u << st);
            if (i == patch_it) {
                // the new token's block: its row as written, whatever the copy read there; the
                // proxy fence orders the store before the stage's next bulk copy
                if (piece_off >= 0) {
                    st_shared_v4((piece_v ? ring.v(st) : ring.k(st)) + piece_off, piece);
                    fence_proxy_async_smem();
                }
                __syncwarp();
            }
            const int tok0 = (blk0 + warp + i * NW) * kBlockTokens;
            // scores: 16 tokens x 8 heads
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t kt = ring.k(st);
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                uint32_t a0, a1, a2, a3;
                ldmatrix_x4(kt + kk * 512 + k_lane, a0, a1, a2, a3);
                mma_bf16_16816(acc, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
            }
            const bool lo_ok = tok0 + r < tok_end, hi_ok = tok0 + r + 8 < tok_end;
            const float s0 = lo_ok ? acc[0] * p.scale_log2 : -INFINITY;
            const float s1 = lo_ok ? acc[1] * p.scale_log2 : -INFINITY;
            const float s2 = hi_ok ? acc[2] * p.scale_log2 : -INFINITY;
            const float s3 = hi_ok ? acc[3] * p.scale_log2 : -INFINITY;
            float bm0 = fmaxf(s0, s2), bm1 = fmaxf(s1, s3);
#pragma unroll
            for (int x = 4; x < 32; x <<= 1) {
                bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, x));
                bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, x));
            }
            const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
            const float al0 = fast_exp2(m0 - mn0), al1 = fast_exp2(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            const uint32_t x0 = pack_bf16x2(fast_exp2(s0 - mn0), fast_exp2(s1 - mn1));   // token r
            const uint32_t x1 = pack_bf16x2(fast_exp2(s2 - mn0), fast_exp2(s3 - mn1));   // token r+8
            l0 = l0 * al0 + (bf16_lo_to_f32(x0) + bf16_lo_to_f32(x1));
            l1 = l1 * al1 + (bf16_hi_to_f32(x0) + bf16_hi_to_f32(x1));
            const uint32_t pb0 = movmatrix_trans(x0), pb1 = movmatrix_trans(x1);
            const bool rescale = !kLazyRescale || __any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f);

            // V^T fragments hold tokens 2c, 2c+1 (regs 0,1) and 2c+8, 2c+9 (regs 2,3);
            // slots past the context may hold anything (even NaN), so zero them.
            uint32_t mask_a = 0xffffffffu, mask_b = 0xffffffffu;
            if (tok0 + kBlockTokens > tok_end) {
                mask_a = (tok0 + 2 * c < tok_end ? 0x0000ffffu : 0u) |
                         (tok0 + 2 * c + 1 < tok_end ? 0xffff0000u : 0u);
                mask_b = (tok0 + 2 * c + 8 < tok_end ? 0x0000ffffu : 0u) |
                         (tok0 + 2 * c + 9 < tok_end ? 0xffff0000u : 0u);
            }
            const uint32_t vt = ring.v(st);
#pragma unroll
            for (int mi = 0; mi < KS; ++mi) {
                uint32_t v0, v1, v2, v3;
                ldmatrix_x4_trans(vt + mi * 512 + v_lane, v0, v1, v2, v3);
                v0 &= mask_a; v1 &= mask_a; v2 &= mask_b; v3 &= mask_b;
                if (rescale) {
                    o[mi][0] *= al0; o[mi][1] *= al1; o[mi][2] *= al0; o[mi][3] *= al1;
                }
                mma_bf16_16816(o[mi], v0, v1, v2, v3, pb0, pb1);
            }
        }
        __syncwarp();
        if (i + NST < nb_w && issue_blk(__ldg(trow + blk0 + warp + (i + NST) * NW), st))
            issued |= 1u << st;
    }

    if (failed) {
        // Drain every copy still in flight into this warp's stages before the
        // shared memory is reused or the CTA exits.
        if (lane == 0) raise_flag(p.err, PA_DEV_ERR_TIMEOUT);
        for (int st = 0; st < NST; ++st)
            if ((issued >> st) & 1u) mbar_wait_bounded(ring.bar(st), (phase >> st) & 1u, kWaitLimitNs);
    }

#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, x);
        l1 += __shfl_xor_sync(0xffffffffu, l1, x);
    }

    if (p.after_prefix && first_cta()) grid_dependency_wait();
    const bool cta_failed = __syncthreads_or(failed);   // every warp is done with its stages
    constexpr int OS = D + 4;
    float* sm_o = reinterpret_cast<float*>(smem);       // [NW][8][OS]
    float* sm_m = sm_o + NW * 8 * OS;                    // [NW][8]
    float* sm_l = sm_m + NW * 8;                         // [NW][8]
    {
        float* ow = sm_o + warp * 8 * OS;
#pragma unroll
        for (int mi = 0; mi < KS; ++mi) {
            const int d0 = 16 * mi + r, d1 = d0 + 8;
            ow[(2 * c) * OS + d0] = o[mi][0];
            ow[(2 * c + 1) * OS + d0] = o[mi][1];
            ow[(2 * c) * OS + d1] = o[mi][2];
            ow[(2 * c + 1) * OS + d1] = o[mi][3];
        }
        if (r == 0) {
            sm_m[warp * 8 + 2 * c] = m0;
            sm_m[warp * 8 + 2 * c + 1] = m1;
            sm_l[warp * 8 + 2 * c] = l0;
            sm_l[warp * 8 + 2 * c + 1] = l1;
        }
    }
    __syncthreads();
    merge_and_store<D, NW, __nv_bfloat16>(p, sm_o, sm_m, sm_l, s, kvh, j, nparts, cta_failed);
}

// ---------------------------------------------------------------------------
// FP8 kernel: E4M3 K/V records (codes + per-slot fp32 scales), bf16 q and out.
// Same pipeline as the bf16 kernel; the codes are converted to f16 in registers
// (exact) and the tensor cores run f16 x f16 -> fp32.
//   K: ldmatrix of a tile's 16-byte rows gives each thread 4 consecutive dims of
//      one token; the dot product's index is permuted (logical k 2c+e <-> dim
//      4c+e, 2c+8+e <-> 4c+2+e) identically in the query fragment.  The A rows
//      are gathered in the token order pi(m) = 4(m/2) + m%2, pi(8+m) = pi(m) + 2,
//      which makes the transposed probabilities line up with V below.
//   V: each dim's 16 tokens form one 16-byte row, so ldmatrix of V^T rows gives
//      each thread 4 consecutive tokens of one dim: logical k 2c+e <-> token
//      4c+e, 2c+8+e <-> token 4c+2+e, which is what movmatrix of the score tile
//      in the pi order delivers.
//   Scales: scores are multiplied by the key's slot scale; probabilities by the
//   value's slot scale (and 2^8, to stay in f16's normal range; the sum gets the
//   same 2^8) before the P.V product.
// ---------------------------------------------------------------------------
template <int D, int NW, int NST>
__global__ void __launch_bounds__(NW * 32)
decode_fp8_kernel(const KParams p) {
    constexpr int REC = 16 * D + 64;            // bytes of one (block, kv head) record
    constexpr int KS = D / 16;                  // k-steps (one 16-dim piece each) = m-tiles of P.V
    constexpr float kPScale = 256.f;
    extern __shared__ __align__(128) uint8_t smem[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, c = lane & 3;
    const int j = blockIdx.x + p.first_part, kvh = blockIdx.y, s = blockIdx.z;
    const int32_t* trow = p.tables + (size_t)s * p.max_blocks;
    int32_t first_blk[NST];
#pragma unroll
    for (int i = 0; i < NST; ++i) {
        const int b = j * p.part_blocks + warp + i * NW;
        first_blk[i] = b < p.max_blocks ? __ldg(trow + b) : -1;
    }
    const int L = clamped_len(p, s);
    const int nparts = num_parts(L, p.part_blocks);
    if (blockIdx.x == 0 && kvh == 0 && threadIdx.x == 0 && nparts > p.grid_parts)
        raise_flag(p.err, PA_DEV_ERR_HINT);
    if (j >= nparts || aborted(p.err)) {
        grid_dependency_wait();   // a dependent grid never completes before the one it follows
        return;
    }

    const int blk0 = j * p.part_blocks;
    const int tok_end = min(L, (j + 1) * p.part_blocks * kBlockTokens);
    const int nblk = (tok_end - blk0 * kBlockTokens + kBlockTokens - 1) / kBlockTokens;
    const int nb_w = nblk > warp ? (nblk - warp + NW - 1) / NW : 0;

    const uint32_t stage0 = smem_u32(smem) + warp * NST * 2 * REC;
    const uint32_t bar0 = smem_u32(smem) + NW * NST * 2 * REC + warp * NST * 8;
    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < NST; ++st) mbar_init(bar0 + st * 8, 1);
        fence_proxy_async_smem();
    }
    __syncwarp();

    // the pools and the query may be written by the previous kernel: wait for it
    grid_dependency_wait();
    grid_launch_dependents();

    const uint64_t pol = l2_policy_evict_first();
    auto issue_blk = [&](int32_t blk, int st) -> bool {
        const bool ok = blk >= 0 && blk < p.num_blocks;
        if (lane == 0) {
            if (ok) {
                const size_t off = ((size_t)blk * p.Hkv + kvh) * (size_t)REC;
                const uint32_t bar = bar0 + st * 8;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, 2 * REC);
                bulk_g2s(stage0 + st * 2 * REC, p.k_pool + off, REC, bar, pol);
                bulk_g2s(stage0 + st * 2 * REC + REC, p.v_pool + off, REC, bar, pol);
            } else {
                raise_flag(p.err, PA_DEV_ERR_BAD_BLOCK);
            }
        }
        return ok;
    };

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[KS][4];
#pragma unroll
    for (int i = 0; i < KS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    uint32_t issued = 0, phase = 0;
    bool failed = false;
#pragma unroll
    for (int i = 0; i < NST; ++i)
        if (i < nb_w && issue_blk(first_blk[i], i)) issued |= 1u << i;

    // Decode with append (as in the bf16 kernel): the warp that reads the new row's block
    // quantises and writes the row while its first records are in flight, and patches it into
    // its copy of the block at iteration patch_it.
    uint32_t nkc = 0u, nvc = 0u;
    float nks = 0.f, nvs = 0.f;
    int nslot = -1, patch_it = -1;
    if (p.k_new && L > 0 && j == min(nparts, p.grid_parts) - 1 && warp == (nblk - 1) % NW) {
        nslot = new_token_fp8<D>(p, s, kvh, L, trow, lane, nkc, nvc, nks, nvs);
        if (nslot >= 0 && j == nparts - 1) patch_it = (nblk - 1) / NW;
    }

    // query fragments in f16 with the permuted dims: b0 <- dims 16kk+4c, +1; b1 <- +2, +3
    // (loaded while the first records are in flight)
    uint32_t qb[KS][2];
    {
        const bool live = r < p.G;
        const uint16_t* qrow = reinterpret_cast<const uint16_t*>(p.q) +
                               ((size_t)s * p.Hq + (size_t)kvh * p.G + (live ? r : 0)) * D;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            if (live) {
                const uint2 u = __ldg(reinterpret_cast<const uint2*>(qrow + 16 * kk + 4 * c));
                qb[kk][0] = pack_f16x2(bf16_lo_to_f32(u.x), bf16_hi_to_f32(u.x));
                qb[kk][1] = pack_f16x2(bf16_lo_to_f32(u.y), bf16_hi_to_f32(u.y));
            } else {
                qb[kk][0] = qb[kk][1] = 0u;
            }
        }
    }

    // K rows gathered in the pi order; lane l addresses row l%8 of matrix l/8:
    // matrices 0 / 1 = rows 0-7 / 8-15 of piece kk, 2 / 3 = the same of piece kk+1
    const int km = lane >> 3, kr = lane & 7;
    const int ktok = 4 * (kr >> 1) + (kr & 1) + ((km & 1) ? 2 : 0);
    const uint32_t k_lane = (uint32_t)(((km >> 1) * kBlockTokens + ktok) * 16);
    const int tr0 = 4 * (r >> 1) + (r & 1), tr1 = tr0 + 2;     // tokens of score rows r, r+8

    for (int i = 0; i < nb_w; ++i) {
        const int st = i % NST;
        if ((issued >> st) & 1u) {
            if (!mbar_wait_bounded(bar0 + st * 8, (phase >> st) & 1u, kWaitLimitNs)) {
                failed = true;
                break;
            }
            phase ^= 1u << st;
            issued &= ~(1u << st);
            const int tok0 = (blk0 + warp + i * NW) * kBlockTokens;
            const uint32_t kt = stage0 + st * 2 * REC, vt = kt + REC;
            if (i == patch_it) {
                // the new row's block: its codes and scales as written, whatever the copy read;
                // the proxy fence orders the stores before the stage's next bulk copy
                fp8_put_row<D>(reinterpret_cast<char*>(smem) + (kt - smem_u32(smem)),
                               reinterpret_cast<char*>(smem) + (vt - smem_u32(smem)), lane, nslot,
                               nkc, nvc, nks, nvs);
                fence_proxy_async_smem();
                __syncwarp();
            }
            const float* kscale = reinterpret_cast<const float*>(smem + (kt - smem_u32(smem)) + 16 * D);
            const float* vscale = reinterpret_cast<const float*>(smem + (vt - smem_u32(smem)) + 16 * D);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < KS; kk += 2) {
                uint32_t x0, x1, x2, x3;
                ldmatrix_x4(kt + kk * 256 + k_lane, x0, x1, x2, x3);
                mma_f16_16816(acc, e4m3x2_to_f16x2((uint16_t)(x0 & 0xffffu)),
                              e4m3x2_to_f16x2((uint16_t)(x1 & 0xffffu)),
                              e4m3x2_to_f16x2((uint16_t)(x0 >> 16)),
                              e4m3x2_to_f16x2((uint16_t)(x1 >> 16)), qb[kk][0], qb[kk][1]);
                if (kk + 1 < KS)
                    mma_f16_16816(acc, e4m3x2_to_f16x2((uint16_t)(x2 & 0xffffu)),
                                  e4m3x2_to_f16x2((uint16_t)(x3 & 0xffffu)),
                                  e4m3x2_to_f16x2((uint16_t)(x2 >> 16)),
                                  e4m3x2_to_f16x2((uint16_t)(x3 >> 16)), qb[kk + 1][0], qb[kk + 1][1]);
            }
            const bool ok0 = tok0 + tr0 < tok_end, ok1 = tok0 + tr1 < tok_end;
            const float sk0 = kscale[tr0] * p.scale_log2, sk1 = kscale[tr1] * p.scale_log2;
            const float s0 = ok0 ? acc[0] * sk0 : -INFINITY;
            const float s1 = ok0 ? acc[1] * sk0 : -INFINITY;
            const float s2 = ok1 ? acc[2] * sk1 : -INFINITY;
            const float s3 = ok1 ? acc[3] * sk1 : -INFINITY;
            float bm0 = fmaxf(s0, s2), bm1 = fmaxf(s1, s3);
#pragma unroll
            for (int x = 4; x < 32; x <<= 1) {
                bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, x));
                bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, x));
            }
            const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
            const float al0 = fast_exp2(m0 - mn0), al1 = fast_exp2(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            const float p0 = fast_exp2(s0 - mn0), p1 = fast_exp2(s1 - mn1);
            const float p2 = fast_exp2(s2 - mn0), p3 = fast_exp2(s3 - mn1);
            l0 = l0 * al0 + (p0 + p2);
            l1 = l1 * al1 + (p1 + p3);
            // slots past the context carry arbitrary scales (even inf after the 2^8): their
            // probabilities are zero and must stay zero, so select rather than multiply
            const float sv0 = vscale[tr0] * kPScale, sv1 = vscale[tr1] * kPScale;
            const uint32_t pb0 = movmatrix_trans(
                pack_f16x2(ok0 ? p0 * sv0 : 0.f, ok0 ? p1 * sv0 : 0.f));
            const uint32_t pb1 = movmatrix_trans(
                pack_f16x2(ok1 ? p2 * sv1 : 0.f, ok1 ? p3 * sv1 : 0.f));
            // V^T rows: thread holds tokens 4c..4c+3 of one dim; past the context the
            // codes may be anything, so zero them
            const bool rescale = !kLazyRescale || __any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f);
            uint32_t vmask = 0xffffffffu;
            if (tok0 + kBlockTokens > tok_end) {
                vmask = 0u;
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    if (tok0 + 4 * c + b < tok_end) vmask |= 0xffu << (8 * b);
            }
#pragma unroll
            for (int mi = 0; mi < KS; mi += 2) {
                uint32_t y0, y1, y2, y3;   // dims 16mi+0..7, 16mi+8..15, 16(mi+1)+0..7, +8..15
                ldmatrix_x4(vt + mi * 256 + lane * 16, y0, y1, y2, y3);
                y0 &= vmask; y1 &= vmask; y2 &= vmask; y3 &= vmask;
                if (rescale) {
                    o[mi][0] *= al0; o[mi][1] *= al1; o[mi][2] *= al0; o[mi][3] *= al1;
                }
                mma_f16_16816(o[mi], e4m3x2_to_f16x2((uint16_t)(y0 & 0xffffu)),
                              e4m3x2_to_f16x2((uint16_t)(y1 & 0xffffu)),
                              e4m3x2_to_f16x2((uint16_t)(y0 >> 16)),
                              e4m3x2_to_f16x2((uint16_t)(y1 >> 16)), pb0, pb1);
                if (mi + 1 < KS) {
                    if (rescale) {
                        o[mi + 1][0] *= al0; o[mi + 1][1] *= al1; o[mi + 1][2] *= al0;
                        o[mi + 1][3] *= al1;
                    }
                    mma_f16_16816(o[mi + 1], e4m3x2_to_f16x2((uint16_t)(y2 & 0xffffu)),
                                  e4m3x2_to_f16x2((uint16_t)(y3 & 0xffffu)),
                                  e4m3x2_to_f16x2((uint16_t)(y2 >> 16)),
                                  e4m3x2_to_f16x2((uint16_t)(y3 >> 16)), pb0, pb1);
                }
            }
        }
        __syncwarp();
        if (i + NST < nb_w && issue_blk(__ldg(trow + blk0 + warp + (i + NST) * NW), st))
            issued |= 1u << st;
    }
    if (failed) {
        if (lane == 0) raise_flag(p.err, PA_DEV_ERR_TIMEOUT);
        for (int st = 0; st < NST; ++st)
            if ((issued >> st) & 1u) mbar_wait_bounded(bar0 + st * 8, (phase >> st) & 1u, kWaitLimitNs);
    }
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, x);
        l1 += __shfl_xor_sync(0xffffffffu, l1, x);
    }
    l0 *= kPScale;   // the P.V products carry the same factor
    l1 *= kPScale;

    const bool cta_failed = __syncthreads_or(failed);
    constexpr int OS = D + 4;
    float* sm_o = reinterpret_cast<float*>(smem);
    float* sm_m = sm_o + NW * 8 * OS;
    float* sm_l = sm_m + NW * 8;
    {
        float* ow = sm_o + warp * 8 * OS;
#pragma unroll
        for (int mi = 0; mi < KS; ++mi) {
            const int d0 = 16 * mi + r, d1 = d0 + 8;
            ow[(2 * c) * OS + d0] = o[mi][0];
            ow[(2 * c + 1) * OS + d0] = o[mi][1];
            ow[(2 * c) * OS + d1] = o[mi][2];
            ow[(2 * c + 1) * OS + d1] = o[mi][3];
        }
        if (r == 0) {
            sm_m[warp * 8 + 2 * c] = m0;
            sm_m[warp * 8 + 2 * c + 1] = m1;
            sm_l[warp * 8 + 2 * c] = l0;
            sm_l[warp * 8 + 2 * c + 1] = l1;
        }
    }
    __syncthreads();
    merge_and_store<D, NW, __nv_bfloat16>(p, sm_o, sm_m, sm_l, s, kvh, j, nparts, cta_failed);
}

// ---------------------------------------------------------------------------
// FP4 kernel: MXFP4 records (E2M1 codes; one E8M0 scale per token and 32 dims),
// bf16 q and out.  The bf16 pipeline again, with the codes converted to f16 in
// registers (exact) and the tensor cores running f16 x f16 -> fp32.
//   K: a record row is one token; thread (r, c) reads D / 8 adjacent bytes of
//      tokens r and r + 8, whose byte 2 ks + half holds dims 16 ks + 8 half + 2c,
//      +1 -- the A fragment of k-step ks.  The scale varies along the dot product,
//      so each 32-dim block gets its own 2-MMA product, multiplied by the token's
//      scale and summed in fp32.
//   V: a record byte holds two tokens of one dim; thread (r, c) reads D / 4
//      adjacent bytes, byte 4 mi + 2 dh + half holding dim 16 mi + 8 dh + r of
//      tokens 2c + 8 half, +1 -- the A fragments of P.V for m-tile mi.  The scale
//      varies along the contraction (tokens), so it multiplies the probabilities:
//      block b's output dims take P_b = p 2^(e_b(t) - 127) c_b, with c_b =
//      2^(135 - R_b) and R_b the largest scale code of block b seen so far (raised,
//      and block b's accumulators rescaled, when a tile brings a larger one), so P_b
//      stays at most 2^8, within f16's range.  A scale code of 0 (a block below
//      2^-123) counts as 0.
//   Codes reach f16 through E4M3: the E2M1 code (s, e1 e0, m) is bit for bit the
//   E4M3 code (s, 0 0 e1 e0, m 0 0) of the value times 2^-6, and E4M3 -> f16 is the
//   exact conversion the FP8 kernel uses; the 2^-6 is undone with the scales.
// ---------------------------------------------------------------------------
// The NB (2 or 4) E8M0 scale bytes of one token, byte b in bits 8b .. 8b+7.
template <int NB>
__device__ __forceinline__ uint32_t scale_bytes(const uint8_t* sm) {
    if constexpr (NB == 4) return *reinterpret_cast<const uint32_t*>(sm);
    else return *reinterpret_cast<const uint16_t*>(sm);
}

// Scale byte b of w as the fp32 2^(code - 127) (its bits are code << 23; code 0 gives 0).
template <int B>
__device__ __forceinline__ float scale_value(uint32_t w) {
    constexpr int sh = 23 - 8 * B;
    return __uint_as_float((sh >= 0 ? (w << sh) : (w >> -sh)) & 0x7F800000u);
}

// E2M1 codes of a word as four f16x2 (byte i -> o[i]), times 2^kFp4CodeExp.
#ifndef PA_FP4_UNPACK_E4M3
#define PA_FP4_UNPACK_E4M3 0
#endif
constexpr int kFp4CodeExp = PA_FP4_UNPACK_E4M3 ? -6 : 0;
__device__ __forceinline__ void fp4_unpack(uint32_t w, uint32_t (&o)[4]) {
    if constexpr (PA_FP4_UNPACK_E4M3) e2m1x8_to_f16x2x4_scaled(w, o);
    else e2m1x8_to_f16x2x4(w, o);
}

#ifndef PA_FP4_MIN_CTAS
#define PA_FP4_MIN_CTAS 1
#endif
template <int D, int NW, int NST>
__global__ void __launch_bounds__(NW * 32, PA_FP4_MIN_CTAS)
decode_fp4_kernel(const KParams p) {
    constexpr int REC = 8 * D + D / 2;          // bytes of one (block, kv head) record
    constexpr int KS = D / 16;                  // k-steps of the scores = m-tiles of P.V
    constexpr int NB = D / 32;                  // scale blocks per token
    constexpr int KW = D / 32;                  // 32-bit words of a thread's K bytes per token
    constexpr int VW = D / 16;                  // 32-bit words of a thread's V bytes
    // the stage rings, reused by the cross-warp merge at the end; the barriers after both
    constexpr int RING = NW * NST * 2 * REC;
    constexpr int MERGE = NW * 8 * (D + 4) * 4 + 2 * NW * 8 * 4;
    constexpr int BAR_OFF = RING > MERGE ? RING : MERGE;
    extern __shared__ __align__(128) uint8_t smem[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, c = lane & 3;
    const int j = blockIdx.x + p.first_part, kvh = blockIdx.y, s = blockIdx.z;
    const int32_t* trow = p.tables + (size_t)s * p.max_blocks;
    int32_t first_blk[NST];
#pragma unroll
    for (int i = 0; i < NST; ++i) {
        const int b = j * p.part_blocks + warp + i * NW;
        first_blk[i] = b < p.max_blocks ? __ldg(trow + b) : -1;
    }
    const int L = clamped_len(p, s);
    const int nparts = num_parts(L, p.part_blocks);
    if (blockIdx.x == 0 && kvh == 0 && threadIdx.x == 0 && nparts > p.grid_parts)
        raise_flag(p.err, PA_DEV_ERR_HINT);
    if (j >= nparts || aborted(p.err)) {
        grid_dependency_wait();   // a dependent grid never completes before the one it follows
        return;
    }

    const int blk0 = j * p.part_blocks;
    const int tok_end = min(L, (j + 1) * p.part_blocks * kBlockTokens);
    const int nblk = (tok_end - blk0 * kBlockTokens + kBlockTokens - 1) / kBlockTokens;
    const int nb_w = nblk > warp ? (nblk - warp + NW - 1) / NW : 0;

    const uint32_t stage0 = smem_u32(smem) + warp * NST * 2 * REC;
    const uint32_t bar0 = smem_u32(smem) + BAR_OFF + warp * NST * 8;
    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < NST; ++st) mbar_init(bar0 + st * 8, 1);
        fence_proxy_async_smem();
    }
    __syncwarp();
    grid_dependency_wait();
    grid_launch_dependents();

    const uint64_t pol = l2_policy_evict_first();
    auto issue_blk = [&](int32_t blk, int st) -> bool {
        const bool ok = blk >= 0 && blk < p.num_blocks;
        if (lane == 0) {
            if (ok) {
                const size_t off = ((size_t)blk * p.Hkv + kvh) * (size_t)REC;
                const uint32_t bar = bar0 + st * 8;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, 2 * REC);
                bulk_g2s(stage0 + st * 2 * REC, p.k_pool + off, REC, bar, pol);
                bulk_g2s(stage0 + st * 2 * REC + REC, p.v_pool + off, REC, bar, pol);
            } else {
                raise_flag(p.err, PA_DEV_ERR_BAD_BLOCK);
            }
        }
        return ok;
    };

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[KS][4];
#pragma unroll
    for (int i = 0; i < KS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    int ref[NB];                                // R_b, warp-uniform
    uint32_t ref_packed = 0;                    // the R_b as bytes
    float cb[NB];                               // c_b = 2^(135 - R_b), at most 2^127
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        ref[b] = 0;
        cb[b] = exp2i(127);
    }
    // score factor: log2(e) scale, and the 2^-kFp4CodeExp the unpacked codes lack
    const float ksl = p.scale_log2 * exp2i(-kFp4CodeExp);
    uint32_t issued = 0, phase = 0;
    bool failed = false;
#pragma unroll
    for (int i = 0; i < NST; ++i)
        if (i < nb_w && issue_blk(first_blk[i], i)) issued |= 1u << i;

    // query fragments in f16: b0 <- dims 16kk + 2c, +1; b1 <- dims 16kk + 8 + 2c, +1
    uint32_t qb[KS][2];
    {
        const bool live = r < p.G;
        const uint16_t* qrow = reinterpret_cast<const uint16_t*>(p.q) +
                               ((size_t)s * p.Hq + (size_t)kvh * p.G + (live ? r : 0)) * D;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            const uint32_t u0 = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * c)) : 0u;
            const uint32_t u1 = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 8 + 2 * c)) : 0u;
            qb[kk][0] = pack_f16x2(bf16_lo_to_f32(u0), bf16_hi_to_f32(u0));
            qb[kk][1] = pack_f16x2(bf16_lo_to_f32(u1), bf16_hi_to_f32(u1));
        }
    }

    for (int i = 0; i < nb_w; ++i) {
        const int st = i % NST;
        // the table entry of the block this stage takes next, in flight during the tile
        const int32_t nxt = i + NST < nb_w ? __ldg(trow + blk0 + warp + (i + NST) * NW) : -1;
        if ((issued >> st) & 1u) {
            if (!mbar_wait_bounded(bar0 + st * 8, (phase >> st) & 1u, kWaitLimitNs)) {
                failed = true;
                break;
            }
            phase ^= 1u << st;
            issued &= ~(1u << st);
            const int tok0 = (blk0 + warp + i * NW) * kBlockTokens;
            const uint8_t* kt = smem + (size_t)(warp * NST + st) * 2 * REC;
            const uint8_t* vt = kt + REC;
            const bool ok0 = tok0 + r < tok_end, ok1 = tok0 + r + 8 < tok_end;

            // ---- scores: per 32-dim block, codes . q, times the token's block scale
            uint32_t kr[KW], kr8[KW];
#pragma unroll
            for (int w = 0; w < KW; ++w) {
                kr[w] = *reinterpret_cast<const uint32_t*>(kt + r * (D / 2) + c * (D / 8) + 4 * w);
                kr8[w] = *reinterpret_cast<const uint32_t*>(kt + (r + 8) * (D / 2) + c * (D / 8) + 4 * w);
            }
            const uint32_t ksr = scale_bytes<NB>(kt + 8 * D + r * NB);     // tokens r, r + 8
            const uint32_t ksr8 = scale_bytes<NB>(kt + 8 * D + (r + 8) * NB);
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                uint32_t a[4], a8[4];
                fp4_unpack(kr[b], a);                   // bytes 4b .. 4b+3: k-steps 2b, 2b+1
                fp4_unpack(kr8[b], a8);
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                mma_f16_16816(acc, a[0], a8[0], a[1], a8[1], qb[2 * b][0], qb[2 * b][1]);
                mma_f16_16816(acc, a[2], a8[2], a[3], a8[3], qb[2 * b + 1][0], qb[2 * b + 1][1]);
                float f0, f1;
                if (b == 0) { f0 = scale_value<0>(ksr); f1 = scale_value<0>(ksr8); }
                else if (b == 1) { f0 = scale_value<1>(ksr); f1 = scale_value<1>(ksr8); }
                else if (b == 2) { f0 = scale_value<2>(ksr); f1 = scale_value<2>(ksr8); }
                else { f0 = scale_value<3>(ksr); f1 = scale_value<3>(ksr8); }
                f0 *= ksl;
                f1 *= ksl;
                sc[0] = fmaf(acc[0], f0, sc[0]);
                sc[1] = fmaf(acc[1], f0, sc[1]);
                sc[2] = fmaf(acc[2], f1, sc[2]);
                sc[3] = fmaf(acc[3], f1, sc[3]);
            }
            // slots past the context may hold anything: select, never multiply
            const float s0 = ok0 ? sc[0] : -INFINITY;
            const float s1 = ok0 ? sc[1] : -INFINITY;
            const float s2 = ok1 ? sc[2] : -INFINITY;
            const float s3 = ok1 ? sc[3] : -INFINITY;
            float bm0 = fmaxf(s0, s2), bm1 = fmaxf(s1, s3);
#pragma unroll
            for (int x = 4; x < 32; x <<= 1) {
                bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, x));
                bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, x));
            }
            const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
            const float al0 = fast_exp2(m0 - mn0), al1 = fast_exp2(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            const float p0 = fast_exp2(s0 - mn0), p1 = fast_exp2(s1 - mn1);
            const float p2 = fast_exp2(s2 - mn0), p3 = fast_exp2(s3 - mn1);
            l0 = l0 * al0 + (p0 + p2);
            l1 = l1 * al1 + (p1 + p3);
            const bool rescale = !kLazyRescale || __any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f);

            // ---- value scales: the tile's largest per block (live tokens only) raises R_b
            const uint32_t vsr = ok0 ? scale_bytes<NB>(vt + 8 * D + r * NB) : 0u;
            const uint32_t vsr8 = ok1 ? scale_bytes<NB>(vt + 8 * D + (r + 8) * NB) : 0u;
            uint32_t tmax = __vmaxu4(vsr, vsr8);
#pragma unroll
            for (int x = 4; x < 32; x <<= 1) tmax = __vmaxu4(tmax, __shfl_xor_sync(0xffffffffu, tmax, x));
            // one warp-uniform test per tile (the packed references are compared bytewise);
            // after the first tile of a partition a raise is rare
            if (__vmaxu4(tmax, ref_packed) != ref_packed) {
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const int eb = (int)((tmax >> (8 * b)) & 0xffu);
                    if (eb > ref[b]) {
                        const float cn = exp2i(min(135 - eb, 127));
                        const float f = cn / cb[b];      // a power of two: exact
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            o[2 * b][x] *= f;
                            o[2 * b + 1][x] *= f;
                        }
                        ref[b] = eb;
                        cb[b] = cn;
                    }
                }
                ref_packed = __vmaxu4(tmax, ref_packed);
            }
            if (rescale) {
#pragma unroll
                for (int mi = 0; mi < KS; ++mi) {
                    o[mi][0] *= al0; o[mi][1] *= al1; o[mi][2] *= al0; o[mi][3] *= al1;
                }
            }

            // ---- P_b . V for each block of output dims
            uint32_t vw[VW];
#pragma unroll
            for (int w = 0; w < VW; ++w)
                vw[w] = *reinterpret_cast<const uint32_t*>(vt + (r * 4 + c) * (KS * 4) + 4 * w);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                // slots past the context have p = 0 and scale code 0 here (g = 0): no select
                float g0, g1;
                if (b == 0) { g0 = scale_value<0>(vsr); g1 = scale_value<0>(vsr8); }
                else if (b == 1) { g0 = scale_value<1>(vsr); g1 = scale_value<1>(vsr8); }
                else if (b == 2) { g0 = scale_value<2>(vsr); g1 = scale_value<2>(vsr8); }
                else { g0 = scale_value<3>(vsr); g1 = scale_value<3>(vsr8); }
                g0 *= cb[b];
                g1 *= cb[b];
                const uint32_t pb0 = movmatrix_trans(pack_f16x2(p0 * g0, p1 * g0));
                const uint32_t pb1 = movmatrix_trans(pack_f16x2(p2 * g1, p3 * g1));
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int mi = 2 * b + h2;
                    uint32_t a[4];                       // (dh 0, half 0), (0, 1), (1, 0), (1, 1)
                    fp4_unpack(vw[mi], a);
                    mma_f16_16816(o[mi], a[0], a[2], a[1], a[3], pb0, pb1);
                }
            }
        }
        __syncwarp();
        if (i + NST < nb_w && issue_blk(nxt, st)) issued |= 1u << st;
    }
    if (failed) {
        if (lane == 0) raise_flag(p.err, PA_DEV_ERR_TIMEOUT);
        for (int st = 0; st < NST; ++st)
            if ((issued >> st) & 1u) mbar_wait_bounded(bar0 + st * 8, (phase >> st) & 1u, kWaitLimitNs);
    }
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, x);
        l1 += __shfl_xor_sync(0xffffffffu, l1, x);
    }
    // back to true units: block b's outputs carry c_b and the codes' 2^kFp4CodeExp
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const float f = exp2i(-kFp4CodeExp) / cb[b];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            o[2 * b][x] *= f;
            o[2 * b + 1][x] *= f;
        }
    }

    const bool cta_failed = __syncthreads_or(failed);
    constexpr int OS = D + 4;
    float* sm_o = reinterpret_cast<float*>(smem);
    float* sm_m = sm_o + NW * 8 * OS;
    float* sm_l = sm_m + NW * 8;
    {
        float* ow = sm_o + warp * 8 * OS;
#pragma unroll
        for (int mi = 0; mi < KS; ++mi) {
            const int d0 = 16 * mi + r, d1 = d0 + 8;
            ow[(2 * c) * OS + d0] = o[mi][0];
            ow[(2 * c + 1) * OS + d0] = o[mi][1];
            ow[(2 * c) * OS + d1] = o[mi][2];
            ow[(2 * c + 1) * OS + d1] = o[mi][3];
        }
        if (r == 0) {
            sm_m[warp * 8 + 2 * c] = m0;
            sm_m[warp * 8 + 2 * c + 1] = m1;
            sm_l[warp * 8 + 2 * c] = l0;
            sm_l[warp * 8 + 2 * c + 1] = l1;
        }
    }
    __syncthreads();
    merge_and_store<D, NW, __nv_bfloat16>(p, sm_o, sm_m, sm_l, s, kvh, j, nparts, cta_failed);
}

// ---------------------------------------------------------------------------
// fp32 kernel: CUDA-core FMAs on the same pipeline
// ---------------------------------------------------------------------------
template <int D, int NW, int NST>
__global__ void __launch_bounds__(NW * 32)
decode_f32_kernel(const KParams p) {
    constexpr int TILE = kBlockTokens * D * 4;
    constexpr int NCH = D / 4;          // 16-byte chunks per token row
    constexpr int DPL = D / 32;         // output dims per lane
    extern __shared__ __align__(128) uint8_t smem[];

    grid_dependency_wait();
    grid_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = blockIdx.x + p.first_part, kvh = blockIdx.y, s = blockIdx.z;
    const int L = clamped_len(p, s);
    const int nparts = num_parts(L, p.part_blocks);
    if (blockIdx.x == 0 && kvh == 0 && threadIdx.x == 0 && nparts > p.grid_parts)
        raise_flag(p.err, PA_DEV_ERR_HINT);
    if (j >= nparts || aborted(p.err)) return;

    const int blk0 = j * p.part_blocks;
    const int tok_end = min(L, (j + 1) * p.part_blocks * kBlockTokens);
    const int nblk = (tok_end - blk0 * kBlockTokens + kBlockTokens - 1) / kBlockTokens;
    const int nb_w = nblk > warp ? (nblk - warp + NW - 1) / NW : 0;

    constexpr int RING = ring_smem_bytes<TILE, NW, NST>();
    float* sq = reinterpret_cast<float*>(smem + RING);                 // [8][D] query rows
    float* sp = sq + 8 * D + warp * 8 * kBlockTokens;                  // [8][16] this warp's P

    Ring<TILE, NW, NST> ring;
    ring.stage0 = smem_u32(smem) + warp * NST * 2 * TILE;
    ring.bar0 = smem_u32(smem) + NW * NST * 2 * TILE + warp * NST * 8;
    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < NST; ++st) mbar_init(ring.bar(st), 1);
        fence_proxy_async_smem();
    }
    const int32_t* trow = p.tables + (size_t)s * p.max_blocks;
    if (p.k_new && L > 0 && j == min(nparts, p.grid_parts) - 1 && warp == 0)
        write_new_token<D * 4>(p, s, kvh, L, trow, lane);    // ordered by the barrier below
    const float* qbase = reinterpret_cast<const float*>(p.q) + ((size_t)s * p.Hq + (size_t)kvh * p.G) * D;
    for (int idx = threadIdx.x; idx < 8 * D; idx += NW * 32)
        sq[idx] = idx < p.G * D ? __ldg(qbase + idx) : 0.f;
    __syncthreads();

    const uint64_t pol = l2_policy_evict_first();
    auto issue = [&](int i, int st) -> bool {
        const int b = blk0 + warp + i * NW;
        const int32_t blk = __ldg(trow + b);
        const bool ok = blk >= 0 && blk < p.num_blocks;
        if (lane == 0) {
            if (ok) {
                const size_t off = ((size_t)blk * p.Hkv + kvh) * (size_t)TILE;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(ring.bar(st), 2 * TILE);
                bulk_g2s(ring.k(st), p.k_pool + off, TILE, ring.bar(st), pol);
                bulk_g2s(ring.v(st), p.v_pool + off, TILE, ring.bar(st), pol);
            } else {
                raise_flag(p.err, PA_DEV_ERR_BAD_BLOCK);
            }
        }
        return ok;
    };

    float m[8], l[8], o[8][DPL];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int k = 0; k < DPL; ++k) o[g][k] = 0.f;
    }

    uint32_t issued = 0, phase = 0;
    bool failed = false;
    const int npro = nb_w < NST ? nb_w : NST;
    for (int i = 0; i < npro; ++i)
        if (issue(i, i)) issued |= 1u << i;

    const int t = lane & 15, half = lane >> 4;
    for (int i = 0; i < nb_w; ++i) {
        const int st = i % NST;
        if ((issued >> st) & 1u) {
            if (!mbar_wait_bounded(ring.bar(st), (phase >> st) & 1u, kWaitLimitNs)) {
                failed = true;
                break;
            }
            phase ^= 1u << st;
            issued &= ~(1u << st);
            const int tok0 = (blk0 + warp + i * NW) * kBlockTokens;
            const int nvalid = min(kBlockTokens, tok_end - tok0);
            const float* kt = reinterpret_cast<const float*>(smem + (warp * NST + st) * 2 * TILE);
            const float* vt = kt + TILE / 4;
            // lane (t, half): partial dots of token t over the half's chunks
            float acc[8];
#pragma unroll
            for (int g = 0; g < 8; ++g) acc[g] = 0.f;
#pragma unroll 4
            for (int ch = half * (NCH / 2); ch < (half + 1) * (NCH / 2); ++ch) {
                const float4 kv = *reinterpret_cast<const float4*>(kt + (ch * kBlockTokens + t) * 4);
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    if (g < p.G) {
                        const float4 qv = *reinterpret_cast<const float4*>(sq + g * D + ch * 4);
                        acc[g] = fmaf(qv.x, kv.x, acc[g]);
                        acc[g] = fmaf(qv.y, kv.y, acc[g]);
                        acc[g] = fmaf(qv.z, kv.z, acc[g]);
                        acc[g] = fmaf(qv.w, kv.w, acc[g]);
                    }
                }
            }
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                if (g < p.G) {
                    float sc = acc[g] + __shfl_xor_sync(0xffffffffu, acc[g], 16);
                    sc = t < nvalid ? sc * p.scale_log2 : -INFINITY;
                    float bm = sc;
#pragma unroll
                    for (int x = 1; x < 16; x <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, x));
                    const float mn = fmaxf(m[g], bm);
                    const float al = exp2f(m[g] - mn);
                    const float pr = exp2f(sc - mn);
                    float bs = pr;
#pragma unroll
                    for (int x = 1; x < 16; x <<= 1) bs += __shfl_xor_sync(0xffffffffu, bs, x);
                    m[g] = mn;
                    l[g] = l[g] * al + bs;
#pragma unroll
                    for (int k = 0; k < DPL; ++k) o[g][k] *= al;
                    if (half == 0) sp[g * kBlockTokens + t] = pr;
                }
            }
            __syncwarp();
            for (int tt = 0; tt < nvalid; ++tt) {
#pragma unroll
                for (int k = 0; k < DPL; ++k) {
                    const int d = lane + 32 * k;
                    const float v = vt[((d >> 2) * kBlockTokens + tt) * 4 + (d & 3)];
#pragma unroll
                    for (int g = 0; g < 8; ++g)
                        if (g < p.G) o[g][k] = fmaf(sp[g * kBlockTokens + tt], v, o[g][k]);
                }
            }
        }
        __syncwarp();
        if (i + NST < nb_w && issue(i + NST, st)) issued |= 1u << st;
    }

    if (failed) {
        if (lane == 0) raise_flag(p.err, PA_DEV_ERR_TIMEOUT);
        for (int st = 0; st < NST; ++st)
            if ((issued >> st) & 1u) mbar_wait_bounded(ring.bar(st), (phase >> st) & 1u, kWaitLimitNs);
    }

    const bool cta_failed = __syncthreads_or(failed);
    constexpr int OS = D + 4;
    float* sm_o = reinterpret_cast<float*>(smem);
    float* sm_m = sm_o + NW * 8 * OS;
    float* sm_l = sm_m + NW * 8;
    {
        float* ow = sm_o + warp * 8 * OS;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
#pragma unroll
            for (int k = 0; k < DPL; ++k) ow[g * OS + lane + 32 * k] = o[g][k];
        }
        if (lane < 8) {
            float mm = m[0], ll = l[0];
#pragma unroll
            for (int g = 1; g < 8; ++g)
                if (lane == g) { mm = m[g]; ll = l[g]; }
            sm_m[warp * 8 + lane] = mm;
            sm_l[warp * 8 + lane] = ll;
        }
    }
    __syncthreads();
    merge_and_store<D, NW, float>(p, sm_o, sm_m, sm_l, s, kvh, j, nparts, cta_failed);
}

// ---------------------------------------------------------------------------
// Partition merge: out = sum_j 2^(m_j - M) o_j / sum_j 2^(m_j - M) l_j.
// RPC rows (sequence, query head) per 256-thread CTA: RPC = 8 gives one warp per
// row (few partitions); RPC = 1 gives the whole CTA to one row, warp w summing
// partitions w, w + 8, ... and the warps combined in order through shared memory
// (many partitions).  Lane k owns D/32 dims.  The order of every sum is fixed.
// ---------------------------------------------------------------------------
template <int D, int RPC, typename OutT>
__global__ void __launch_bounds__(256)
decode_reduce_kernel(const KParams p, int num_rows) {
    constexpr int DPL = D / 32;
    constexpr int WPR = 8 / RPC;                    // warps per row
    __shared__ float sm_acc[8][D];
    __shared__ float sm_l[8];
    // the next kernel of the stream may start its set-up; every kernel of this library
    // waits for this grid before reading what it writes (`out`)
    grid_launch_dependents();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int row = blockIdx.x * RPC + warp / WPR;  // s * Hq + h
    const int wr = warp % WPR;                      // this warp's share of the row
    const bool live = row < num_rows;
    int n = 0;
    if (live) {
        const int s = row / p.Hq;
        int L = __ldg(p.lens + s);
        const int cap = p.max_blocks * kBlockTokens;
        L = L < 0 ? 0 : (L > cap ? cap : L);
        n = num_parts(L, p.part_blocks);
        if (n > p.grid_parts) n = p.grid_parts;     // flagged by the main kernel
    }
    // one partition and no shared prefix: written directly by the main kernel
    const int min_n = p.first_part > 0 ? 1 : 2;
    if (WPR == 1 && (!live || n < min_n)) {
        grid_dependency_wait();   // a dependent grid never completes before the one it follows
        return;
    }
    if (p.first_part > 0 && live && wr == 0 && row % p.Hq == 0) {
        // shared prefix: check the caller's promise once per sequence -- its table holds
        // sequence 0's blocks for the shared partitions and its context covers them.  Tables
        // and lengths are inputs, so this runs while the kernels before are finishing.
        const int s = row / p.Hq;
        const int nb = p.first_part * p.part_blocks;
        const int len = __ldg(p.lens + s);
        // (with the step's new rows, a row must also lie past the whole shared prefix)
        bool bad = len < nb * kBlockTokens || (p.k_new != nullptr && len - 1 < p.new_min_pos);
        for (int b = lane; b < nb; b += 32)
            bad |= __ldg(p.tables + (size_t)s * p.max_blocks + b) != __ldg(p.tables + b);
        if (__any_sync(0xffffffffu, bad) && lane == 0) raise_flag(p.err, PA_DEV_ERR_BAD_PREFIX);
    }
    grid_dependency_wait();     // the partials of the kernels before are complete and visible
    // after a copy wait gave up (this call or an earlier one) the partials are not all
    // written: leave `out` untouched, as the main kernel does
    const bool work = live && n >= min_n && !aborted(p.err);
    // the row's partials: with a shared prefix, one per prefix_stride prefix slots, then
    // one per suffix partition (slots first_part ..); without, slots 0 .. n - 1
    const int np = p.first_part / p.prefix_stride;
    const int nm = min(np, n) + max(n - p.first_part, 0);    // partials to merge
    auto slot = [&](int i) { return i < np ? i * p.prefix_stride : p.first_part + (i - np); };
    const size_t prow = (size_t)(work ? row : 0) * p.part_stride;
    const float2* ml = p.part_ml + prow;
    const float* po = p.part_o + prow * D + lane * DPL;
    float acc[DPL];
#pragma unroll
    for (int k = 0; k < DPL; ++k) acc[k] = 0.f;
    float lsum = 0.f;
    if constexpr (WPR == 1) {
        // a warp per row, at most 32 partitions: the maxima (one per lane) and the first
        // kChunk partial rows are loaded together, so the merge takes one round trip
        constexpr int kChunk = 8;
        float2 mlv = make_float2(-INFINITY, 0.f);
        if (work && lane < nm) mlv = ml[slot(lane)];
        float ov[kChunk][DPL];
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            const bool has = work && i < nm;
            const size_t off = (size_t)slot(i) * D;
            if constexpr (DPL == 4) {
                const float4 o = has ? *reinterpret_cast<const float4*>(po + off)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                ov[i][0] = o.x; ov[i][1] = o.y; ov[i][2] = o.z; ov[i][3] = o.w;
            } else {
                const float2 o = has ? *reinterpret_cast<const float2*>(po + off)
                                     : make_float2(0.f, 0.f);
                ov[i][0] = o.x; ov[i][1] = o.y;
            }
        }
        float M = mlv.x;
#pragma unroll
        for (int x = 16; x > 0; x >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x));
        if (work && M != -INFINITY) {
            // partials in order 0, 1, ...: the sum's order is fixed; one whose maximum is
            // -inf (no key) is skipped, whatever its row holds
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                const float mi = __shfl_sync(0xffffffffu, mlv.x, i);
                const float li = __shfl_sync(0xffffffffu, mlv.y, i);
                if (i < nm && mi != -INFINITY) {
                    const float wt = fast_exp2(mi - M);
                    lsum += wt * li;
#pragma unroll
                    for (int k = 0; k < DPL; ++k) acc[k] += wt * ov[i][k];
                }
            }
            for (int i = kChunk; i < nm; ++i) {
                const float mi = __shfl_sync(0xffffffffu, mlv.x, i);
                const float li = __shfl_sync(0xffffffffu, mlv.y, i);
                if (mi == -INFINITY) continue;
                const float wt = fast_exp2(mi - M);
                lsum += wt * li;
#pragma unroll
                for (int k = 0; k < DPL; ++k) acc[k] += wt * po[(size_t)slot(i) * D + k];
            }
        }
    } else {
    float M = -INFINITY;
    if (work)
        for (int i = lane; i < nm; i += 32) M = fmaxf(M, ml[slot(i)].x);
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x));
    if (work && M != -INFINITY) {
#pragma unroll 8
        for (int i = wr; i < nm; i += WPR) {
            const float2 v = ml[slot(i)];
            if (v.x == -INFINITY) continue;               // no key
            const float wt = fast_exp2(v.x - M);
            lsum += wt * v.y;
            if constexpr (DPL == 4) {
                const float4 o = *reinterpret_cast<const float4*>(po + (size_t)slot(i) * D);
                acc[0] += wt * o.x; acc[1] += wt * o.y; acc[2] += wt * o.z; acc[3] += wt * o.w;
            } else {
                const float2 o = *reinterpret_cast<const float2*>(po + (size_t)slot(i) * D);
                acc[0] += wt * o.x; acc[1] += wt * o.y;
            }
        }
    }
    }
    if constexpr (WPR > 1) {
#pragma unroll
        for (int k = 0; k < DPL; ++k) sm_acc[warp][lane * DPL + k] = acc[k];
        if (lane == 0) sm_l[warp] = lsum;
        __syncthreads();
        if (!work || wr != 0) return;
        lsum = 0.f;
#pragma unroll
        for (int k = 0; k < DPL; ++k) acc[k] = 0.f;
        for (int w = 0; w < WPR; ++w) {
            lsum += sm_l[w];
#pragma unroll
            for (int k = 0; k < DPL; ++k) acc[k] += sm_acc[w][lane * DPL + k];
        }
    }
    if (!work) return;
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
    for (int k = 0; k < DPL; ++k) {
        const size_t idx = (size_t)row * D + lane * DPL + k;
        if constexpr (sizeof(OutT) == 2)
            reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(acc[k] * inv);
        else
            reinterpret_cast<float*>(p.out)[idx] = acc[k] * inv;
    }
}

// Launch configuration of the main kernels.
// 4 warps x 2 ring stages (64 KB of shared memory for head_dim 128, 3 CTAs per SM)
// measured fastest on GB300 among 1-8 warps x 2-6 stages.
#ifndef PA_DECODE_WARPS
#define PA_DECODE_WARPS 4
#endif
#ifndef PA_DECODE_STAGES
#define PA_DECODE_STAGES 2
#endif
#ifndef PA_DECODE_STAGES_D64
#define PA_DECODE_STAGES_D64 PA_DECODE_STAGES
#endif
constexpr int kWarps = PA_DECODE_WARPS;        // warps per CTA
// ring stages per warp (bf16), per head_dim
template <int D>
constexpr int stages_bf16() { return D == 64 ? PA_DECODE_STAGES_D64 : PA_DECODE_STAGES; }
constexpr int kStagesF32 = 2;

template <int D>
constexpr int bf16_smem() { return ring_smem_bytes<kBlockTokens * D * 2, kWarps, stages_bf16<D>()>(); }
template <int D>
constexpr int f32_smem() {
    return ring_smem_bytes<kBlockTokens * D * 4, kWarps, kStagesF32>() +
           (8 * D + kWarps * 8 * kBlockTokens) * 4;
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    // all of the SM's unified memory as shared memory, so that CTAs of the decode and
    // prefix kernels can share an SM whatever the carve-out the other asked for
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// Launch with programmatic stream serialisation: the kernel may start while the
// previous kernel of the stream finishes, and waits (griddepcontrol.wait) before
// reading anything that kernel writes.
#ifndef PA_USE_PDL
#define PA_USE_PDL 1
#endif

template <typename K>
cudaError_t launch_dependent(K kernel, dim3 grid, dim3 block, int smem, cudaStream_t stream,
                             const KParams& kp) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = PA_USE_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, kp);
}

template <typename K>
cudaError_t launch_dependent_rows(K kernel, dim3 grid, dim3 block, cudaStream_t stream,
                                  const KParams& kp, int rows) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = PA_USE_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, kp, rows);
}

// FP8 launch shape: 4 warps x 2 stages of 4.2 KB records (34 KB, 6 CTAs per SM) and
// 1024-token partitions measured fastest on GB300 (of 2-6 stages, 512-2048 tokens).
#ifndef PA_FP8_STAGES
#define PA_FP8_STAGES 2
#endif
#ifndef PA_FP8_WARPS
#define PA_FP8_WARPS 4
#endif
constexpr int kStagesFp8 = PA_FP8_STAGES;
constexpr int kWarpsFp8 = PA_FP8_WARPS;

template <int D>
constexpr int fp8_smem() {
    return kWarpsFp8 * kStagesFp8 * 2 * (16 * D + 64) + kWarpsFp8 * kStagesFp8 * 8;
}

template <int D>
cudaError_t launch_fp8_for_dim(const KParams& kp, const DecodeArgs& a, cudaStream_t stream);

template <int D>
cudaError_t launch_for_dim(const KParams& kp_in, const DecodeArgs& a, cudaStream_t stream) {
    cudaError_t e = cudaSuccess;
    KParams kp = kp_in;
    const int launched = a.grid_parts - kp.first_part;   // partitions of the main kernel
    if (kp.first_part > 0) {
        // the shared prefix first: its CTAs take one SM each for a chain of tensor-core
        // steps; the suffix kernel after it fills the rest of the GPU and runs beside it
        e = launch_prefix_tc(a, false, stream);
        if (e != cudaSuccess) return e;
        kp.after_prefix = 1;
    }
    if (launched > 0) {
        const dim3 grid(launched, a.num_kv_heads, a.num_seqs);
        if (a.dtype == PA_BF16) {
            auto k = decode_bf16_kernel<D, kWarps, stages_bf16<D>()>;
            if ((e = set_smem(k, bf16_smem<D>())) != cudaSuccess) return e;
            e = launch_dependent(k, grid, dim3(kWarps * 32), bf16_smem<D>(), stream, kp);
        } else {
            auto k = decode_f32_kernel<D, kWarps, kStagesF32>;
            if ((e = set_smem(k, f32_smem<D>())) != cudaSuccess) return e;
            e = launch_dependent(k, grid, dim3(kWarps * 32), f32_smem<D>(), stream, kp);
        }
        if (e != cudaSuccess) return e;
    }

    if (a.grid_parts > 1 || kp.first_part > 0) {
        const int rows = a.num_seqs * a.num_q_heads;
        if (a.grid_parts <= 32) {          // few partitions: a warp per row
            const dim3 rgrid((rows + 7) / 8);
            e = a.dtype == PA_BF16
                    ? launch_dependent_rows(decode_reduce_kernel<D, 8, __nv_bfloat16>, rgrid, dim3(256), stream, kp, rows)
                    : launch_dependent_rows(decode_reduce_kernel<D, 8, float>, rgrid, dim3(256), stream, kp, rows);
        } else {                           // many partitions: a CTA per row
            e = a.dtype == PA_BF16
                    ? launch_dependent_rows(decode_reduce_kernel<D, 1, __nv_bfloat16>, dim3(rows), dim3(256), stream, kp, rows)
                    : launch_dependent_rows(decode_reduce_kernel<D, 1, float>, dim3(rows), dim3(256), stream, kp, rows);
        }
    }
    return e;
}

// FP4 launch shape (MXFP4 records of 8.5 D bytes).
#ifndef PA_FP4_STAGES
#define PA_FP4_STAGES 4
#endif
#ifndef PA_FP4_WARPS
#define PA_FP4_WARPS 4
#endif
constexpr int kStagesFp4 = PA_FP4_STAGES;
constexpr int kWarpsFp4 = PA_FP4_WARPS;

template <int D>
constexpr int fp4_smem() {
    // the stage rings (or the cross-warp merge that reuses them, if larger), then the barriers
    constexpr int ring = kWarpsFp4 * kStagesFp4 * 2 * (8 * D + D / 2);
    constexpr int merge = kWarpsFp4 * 8 * (D + 4) * 4 + 2 * kWarpsFp4 * 8 * 4;
    return (ring > merge ? ring : merge) + kWarpsFp4 * kStagesFp4 * 8;
}

template <int D>
cudaError_t launch_fp4_for_dim(const KParams& kp, const DecodeArgs& a, cudaStream_t stream) {
    cudaError_t e;
    const dim3 grid(a.grid_parts, a.num_kv_heads, a.num_seqs);
    auto k = decode_fp4_kernel<D, kWarpsFp4, kStagesFp4>;
    if ((e = set_smem(k, fp4_smem<D>())) != cudaSuccess) return e;
    if ((e = launch_dependent(k, grid, dim3(kWarpsFp4 * 32), fp4_smem<D>(), stream, kp)) != cudaSuccess)
        return e;
    if (a.grid_parts > 1) {
        const int rows = a.num_seqs * a.num_q_heads;
        if (a.grid_parts <= 32)
            e = launch_dependent_rows(decode_reduce_kernel<D, 8, __nv_bfloat16>, dim3((rows + 7) / 8),
                                      dim3(256), stream, kp, rows);
        else
            e = launch_dependent_rows(decode_reduce_kernel<D, 1, __nv_bfloat16>, dim3(rows), dim3(256),
                                      stream, kp, rows);
    }
    return e;
}

template <int D>
cudaError_t launch_fp8_for_dim(const KParams& kp, const DecodeArgs& a, cudaStream_t stream) {
    cudaError_t e;
    const dim3 grid(a.grid_parts, a.num_kv_heads, a.num_seqs);
    auto k = decode_fp8_kernel<D, kWarpsFp8, kStagesFp8>;
    if ((e = set_smem(k, fp8_smem<D>())) != cudaSuccess) return e;
    if ((e = launch_dependent(k, grid, dim3(kWarpsFp8 * 32), fp8_smem<D>(), stream, kp)) != cudaSuccess)
        return e;
    if (a.grid_parts > 1) {
        const int rows = a.num_seqs * a.num_q_heads;
        if (a.grid_parts <= 32)
            e = launch_dependent_rows(decode_reduce_kernel<D, 8, __nv_bfloat16>, dim3((rows + 7) / 8),
                                      dim3(256), stream, kp, rows);
        else
            e = launch_dependent_rows(decode_reduce_kernel<D, 1, __nv_bfloat16>, dim3(rows), dim3(256),
                                      stream, kp, rows);
    }
    return e;
}

}  // namespace

size_t decode_workspace_bytes(int num_seqs, int num_q_heads, int /*num_kv_heads*/, int head_dim,
                              int max_blocks) {
    const int stride = decode_part_stride(max_blocks);
    if (stride <= 1) return 0;
    const size_t rows = (size_t)num_seqs * (size_t)num_q_heads * (size_t)stride;
    return rows * (size_t)head_dim * sizeof(float) + rows * sizeof(float2);
}

namespace {
KParams make_params(const DecodeArgs& a);
}

cudaError_t launch_decode_fp8(const DecodeArgs& a, cudaStream_t stream) {
    const KParams kp = make_params(a);
    if (a.head_dim == 64) return launch_fp8_for_dim<64>(kp, a, stream);
    return launch_fp8_for_dim<128>(kp, a, stream);
}

cudaError_t launch_decode_fp4(const DecodeArgs& a, cudaStream_t stream) {
    const KParams kp = make_params(a);
    if (a.head_dim == 64) return launch_fp4_for_dim<64>(kp, a, stream);
    return launch_fp4_for_dim<128>(kp, a, stream);
}

namespace {
KParams make_params(const DecodeArgs& a) {
    KParams kp;
    kp.out = a.out;
    kp.q = a.q;
    kp.k_pool = static_cast<const char*>(a.k_pool);
    kp.v_pool = static_cast<const char*>(a.v_pool);
    kp.tables = a.block_tables;
    kp.lens = a.context_lens;
    const size_t rows = (size_t)a.num_seqs * a.num_q_heads * a.part_stride;
    kp.part_o = static_cast<float*>(a.workspace);
    kp.part_ml = a.workspace ? reinterpret_cast<float2*>(static_cast<char*>(a.workspace) +
                                                         rows * a.head_dim * sizeof(float))
                             : nullptr;
    kp.k_new = static_cast<const char*>(a.k_new);
    kp.v_new = static_cast<const char*>(a.v_new);
    kp.new_min_pos = a.new_min_pos;
    kp.err = a.err;
    kp.Hq = a.num_q_heads;
    kp.Hkv = a.num_kv_heads;
    kp.G = a.num_q_heads / a.num_kv_heads;
    kp.max_blocks = a.max_blocks;
    kp.num_blocks = a.num_blocks;
    kp.grid_parts = a.grid_parts;
    kp.part_stride = a.part_stride;
    kp.first_part = a.first_part;
    kp.prefix_stride = a.first_part > 0 ? prefix_slot_mult(a.first_part) : 1;
    kp.part_blocks = a.part_blocks;
    kp.scale_log2 = a.scale * kLog2e;
    kp.after_prefix = 0;
    return kp;
}
}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    const KParams kp = make_params(a);
    if (a.head_dim == 64) return launch_for_dim<64>(kp, a, stream);
    return launch_for_dim<128>(kp, a, stream);
}

}  // namespace pa

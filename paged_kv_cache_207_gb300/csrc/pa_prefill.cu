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
// query head of the kv head) pairs, token-major, 256 / G tokens per CTA, in two
// Q tiles of 128 rows that share every K/V tile.  The 5th-generation tensor cores
// (tcgen05) compute, per key tile of 128 tokens (8 blocks) and Q tile h,
//   S_h = Q_h K^T   into TMEM (one M128 N128 K16 MMA per 16 dims),
//   O_h += P_h V    into TMEM (one M128 N=D K16 MMA per block, P_h from TMEM),
// one thread issuing every MMA; the softmax runs one row per thread of eight
// warps (a warpgroup per Q tile), with the causal mask applied per row.
// Later query tiles (which read more blocks) are scheduled first.
#include <cuda_bf16.h>

#include <cmath>

#include "pa_internal.h"
#include "pa_ptx.cuh"
#include "pa_tc.cuh"

namespace pa {

namespace {

constexpr uint64_t kWaitLimitNs = 200000000ull;
constexpr float kLog2e = 1.4426950408889634f;

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
    // shared-prefix mode: partials of one partition per (sequence, query head) row
    float* part_o;
    float2* part_ml;
    int part_stride, part_blocks, num_seqs, rows_per_cta;
    // prefix mode: wait for the previous kernel of the stream (the append) before reading
    // the query or the pools (set by every launch of the decode path, which starts this
    // kernel first and the suffix kernel after it)
    int wait_first;
    // prefix mode: a CTA covers slot_mult split-KV partitions of the decode (part_blocks is
    // slot_mult times the decode's) and writes its partial into the first of their
    // workspace slots
    int slot_mult;
};

__device__ __forceinline__ void raise_flag(int32_t* err, int bits) {
    if (err) atomicOr(err, bits);
}

// ============================================================================
// The tcgen05 kernel.
//
// Warp roles (two Q tiles): 0-7 softmax (0-3 for Q tile a, 4-7 for tile b; a warp
// reaches the TMEM lanes 32 (warp % 4) ..), 8 streams V tiles with bulk copies, 9 owns
// the TMEM and issues the MMAs, 10-11 copy K tiles in with 16-byte copies.  setmaxnreg
// moves registers from the copy / MMA warps (104 each) to the softmax warps (200 each),
// which hold a 128-column row of S.  setmaxnreg is collective over a warpgroup: every
// warp of a warpgroup runs the same one, so the copy / MMA warps fill whole warpgroups
// (idle warps pad them) and lower their budget together, at the head of their branch.
// A K tile lands chunk-major, [D/8][8 blocks][16 slots][16 B]: every 8-token group
// of the tile is 128 B after the previous one, so Q K^T over the tile's 128 tokens is
// one MMA per 16 dims.  The pool holds a block as [D/8][16 slots][16 B], so each
// 16-byte piece has its own place in the stage.  K comes through the load/store path
// and V through the bulk-copy engine: an SM takes in more from DRAM through both than
// through either (measured on GB300 with 64 busy SMs: 4 KB bulk copies alone about
// 77 GB/s per SM, both about 97 GB/s), and small bulk copies are slow (1 KB ones: about
// 33 GB/s per SM), so the 256-byte pieces are not placed that way.
// Each softmax thread reads its row of S_h from TMEM, applies the causal mask,
// keeps a running maximum that is raised only when a tile exceeds it by more than
// 2^8 (O_h is then rescaled in TMEM), writes its bf16 probabilities over the
// first half of S_h's columns, and at the end reads its row of O_h, divides by
// the row sum and stores it (the prefix mode stores the unnormalised partial and
// its maximum and sum instead).  A CTA with a single Q tile uses tile b's S
// columns as a second S buffer for tile a.
// ============================================================================

namespace tc {

// Two Q tiles of 128 rows (a, b) per CTA share every K/V tile; each has its own softmax
// warpgroup, S and O in TMEM.  The MMA thread interleaves them so that one tile's
// softmax runs while the tensor cores work for the other:
//   S_a(0) S_b(0) | PV_a(0) S_a(1) PV_b(0) S_b(1) | PV_a(1) S_a(2) ...
constexpr int kHalfRows = 128;
constexpr int kRowsTC = 2 * kHalfRows;
constexpr int kKeyBlocks = 8;
constexpr int kKeyTok = kKeyBlocks * kBlockTokens;
// Warp roles for SW softmax warpgroups (2: Q tiles a and b; 1: tile a only, the
// 128-row prefix mode): warps 0 .. 4 SW - 1 softmax, then the V producer, the MMA
// warp and the K copy warps: two with two Q tiles (the register budget holds no more),
// four with one, whose CTAs stream their keys from DRAM (copies in flight are limited
// per scheduler, so the K copies are spread over all four).
template <int SW>
struct Roles {
    static constexpr int kSoftWarps = 4 * SW;
    static constexpr int kProducerWarp = kSoftWarps;       // V tiles
    static constexpr int kMmaWarp = kSoftWarps + 1;        // TMEM owner, MMA issue
    static constexpr int kKWarp = kSoftWarps + 2;          // K tiles
    static constexpr int kKWarps = SW == 1 ? 4 : 2;
    static constexpr int kOtherWarps = (2 + kKWarps + 3) / 4 * 4;   // whole warpgroups
    static constexpr int kThreads = (kSoftWarps + kOtherWarps) * 32;
};
constexpr int kThreadsTC = Roles<2>::kThreads;  // the register budget is set for this size
static_assert(Roles<1>::kThreads <= kThreadsTC, "launch bounds");
constexpr int kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;

// TMEM columns: S of tile h at 128 h (its bf16 P over the first 64 once S is read), O of
// tile h at 256 + 128 h.
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 2 * kKeyTok;

// NQ Q tiles (the softmax warpgroups of the launch) and rings of KST K and VST V tiles,
// as deep as 227 KB allow: three K stages keep the next copies in flight while a tile
// is used (a copy takes a few microseconds to land when the GPU is busy).
template <int D, int NQ = 2>
struct Smem {
    static constexpr int TILE = kBlockTokens * D * 2;          // one (block, kv head) tile
    static constexpr int KTILE = kKeyBlocks * TILE;            // one ring stage
    static constexpr int QTILE = kHalfRows * D * 2;            // [D/8][16][8 rows][16 B]
    static constexpr int KST = 3;
    static constexpr int VST = (NQ == 1 || D == 64) ? 3 : 2;
    static constexpr int Q = 0;                                // tiles a (, b)
    static constexpr int K = Q + NQ * QTILE;                   // K tiles, chunk-major
    static constexpr int V = K + KST * KTILE;                  // V tiles as copied
    static constexpr int BAR = V + VST * KTILE;
    static constexpr int NBAR = 24;
    static constexpr int SLOT = BAR + NBAR * 8;
    // at least 120 KB so that one CTA (and its 512 TMEM columns) owns an SM
    static constexpr int BYTES = SLOT + 16 < 122880 ? 122880 : SLOT + 16;
    static_assert(SLOT + 16 <= 232448, "shared memory of one CTA");
};

// barrier indices (rings of up to 4 stages)
constexpr int kKFull = 0, kKEmpty = 4, kVFull = 8, kVEmpty = 12, kSFull = 16, kPFull = 18,
              kODone = 20, kDone = 22, kPVDone = 23;

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// All lanes wait; the result is made uniform across the warp.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
    const bool ok = mbar_wait_bounded(bar, parity, kWaitLimitNs);
    return __all_sync(0xffffffffu, ok);
}

// Three-input maximum and packed two-lane fp32 arithmetic (one instruction for two
// values); a packed pair holds its first value in the low 32 bits.
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    return ((uint64_t)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float lo_f32(uint64_t x) { return __uint_as_float((uint32_t)x); }
__device__ __forceinline__ float hi_f32(uint64_t x) { return __uint_as_float((uint32_t)(x >> 32)); }
__device__ __forceinline__ uint64_t ffma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t fadd_f32x2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// The copy warps read the table in windows of 32 entries, four key tiles, one entry per
// lane (-1 past the CTA's last block), a window ahead of its use: read one tile ahead,
// every tile would wait for a dependent load (over a microsecond when HBM is busy).
constexpr int kWinTiles = 32 / kKeyBlocks;
__device__ __forceinline__ int32_t fetch_window(const int32_t* trow, int w, int lim, int lane) {
    const int b = 32 * w + lane;
    return b < lim ? __ldg(trow + b) : -1;
}
// Table entry of block `lane` of key tile j from the window holding it (-1 for lanes past
// the tile's blocks or the CTA's last block).
__device__ __forceinline__ int32_t window_block(int32_t win, int j, int lane, int nblk) {
    const int32_t b = __shfl_sync(0xffffffffu, win, (j % kWinTiles) * kKeyBlocks + (lane & (kKeyBlocks - 1)));
    return (lane < kKeyBlocks && j * kKeyBlocks + lane < nblk) ? b : -1;
}

// Flags a needed block whose entry is not a block of the pool (its tile is skipped) and
// returns the bytes of the tile's valid block tiles.
__device__ __forceinline__ uint32_t check_blocks(const PParams& p, int32_t& blk, int j, int nblk,
                                                 int lane, uint32_t tile) {
    const bool needed = lane < kKeyBlocks && j * kKeyBlocks + lane < nblk;
    if (needed && (blk < 0 || blk >= p.num_blocks)) {
        raise_flag(p.err, PA_DEV_ERR_BAD_BLOCK);
        blk = -1;
    }
    return (uint32_t)__popc(__ballot_sync(0xffffffffu, blk >= 0)) * tile;
}

// PREFIX = false: causal prefill of chunk rows (CTA = query tile, kv head, sequence).
// PREFIX = true: rows are (sequence, query head) pairs of the kv head (CTA = row group,
// kv head, partition j of a prefix shared by every sequence, read through table row 0);
// every key is visible and the CTA writes unnormalised partials (o, max, sum) of
// partition j for the split-KV merge instead of outputs.
// SW = 1 launches 256 threads under the same per-thread register budget (168), so a
// CTA takes 256 x 168 registers and leaves room for a decode CTA on its SM.
template <int D, bool PREFIX, int SW>
__global__ void __launch_bounds__(kThreadsTC, 1) prefill_tc_kernel(const PParams p) {
    using L = Smem<D, SW>;
    constexpr int kSoftWarps = Roles<SW>::kSoftWarps;
    constexpr int kProducerWarp = Roles<SW>::kProducerWarp;
    constexpr int kMmaWarp = Roles<SW>::kMmaWarp;
    constexpr int kKWarp = Roles<SW>::kKWarp, kKWarps = Roles<SW>::kKWarps;
    constexpr int TILE = L::TILE, KTILE = L::KTILE, KST = L::KST, VST = L::VST;
    constexpr int KSTEPS = D / 16;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kvh = blockIdx.y;
    if (PREFIX && p.wait_first) grid_dependency_wait();
    int q0 = 0, n = 0, i0 = 0, start = 0, p_last, nblk, row_base = 0, rows_total = 0;
    bool has_b;
    const int32_t* trow = PREFIX ? p.tables + (size_t)blockIdx.z * p.part_blocks
                                 : p.tables + (size_t)blockIdx.z * p.max_blocks;
    // The copy warps' first table windows load at once, bounded by the table row (the
    // CTA's own last block is known one round trip later; no kernel of this library writes
    // the tables).
    // The TIMEOUT bit of the flag: set when a copy wait gave up in this or an earlier call
    // (then nothing is written).  Thread 0 reads it for the softmax and MMA warps, which
    // act on it after their setup barrier; the copy warps read it themselves.
    int32_t win = -1, win_next = -1, flag_in = 0;
    if (warp == kProducerWarp || (warp >= kKWarp && warp < kKWarp + kKWarps)) {
        const int lim = PREFIX ? p.part_blocks : p.max_blocks;
        win = fetch_window(trow, 0, lim, lane);
        win_next = fetch_window(trow, 1, lim, lane);
        if (lane == 0 && p.err) flag_in = *reinterpret_cast<const volatile int32_t*>(p.err);
    }
    if (threadIdx.x == 0 && p.err) flag_in = *reinterpret_cast<const volatile int32_t*>(p.err);
    if constexpr (PREFIX) {
        rows_total = p.num_seqs * p.G;
        row_base = blockIdx.x * p.rows_per_cta;
        nblk = p.part_blocks;
        p_last = nblk * kBlockTokens - 1;                 // positions relative to the partition
        has_b = SW == 2 && p.rows_per_cta > kHalfRows && row_base + kHalfRows < rows_total;
    } else {
        const int qt = gridDim.x - 1 - blockIdx.x;        // later (longer) tiles first
        const int s = blockIdx.z;
        // the chunk's place: three loads in flight together
        q0 = __ldg(p.cu_q + s);
        n = __ldg(p.cu_q + s + 1);
        start = __ldg(p.start_pos + s);
        n -= q0;
        i0 = qt * p.TQ;
        // (a CTA that exits early still waits for the previous grid: a dependent grid never
        // completes before the one it follows)
        if (i0 >= n) {
            grid_dependency_wait();
            return;
        }
        const int i_end = min(n, i0 + p.TQ);
        p_last = start + i_end - 1;                       // last position this CTA attends to
        if (start < 0 || p_last >= p.max_blocks * kBlockTokens) {
            if (threadIdx.x == 0 && kvh == 0) raise_flag(p.err, PA_DEV_ERR_BAD_POS);
            grid_dependency_wait();
            return;
        }
        nblk = p_last / kBlockTokens + 1;
        // tile b holds rows 128 .. 255; it is skipped when none of them is a chunk row
        const int tl_b = kHalfRows / p.G;
        has_b = SW == 2 && tl_b < p.TQ && i0 + tl_b < n;
    }
    const int ntiles = (nblk + kKeyBlocks - 1) / kKeyBlocks;

    const uint32_t aborted_in = (uint32_t)(flag_in & PA_DEV_ERR_TIMEOUT);   // (thread 0)
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + L::Q, sK = sbase + L::K, sV = sbase + L::V;
    const uint32_t bar0 = sbase + L::BAR;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

    if (threadIdx.x == 0) {
#pragma unroll
        for (int i = 0; i < KST; ++i) {
            mbar_init(bar(kKFull + i), kKWarps);
            mbar_init(bar(kKEmpty + i), 1);
        }
#pragma unroll
        for (int i = 0; i < VST; ++i) {
            mbar_init(bar(kVFull + i), 1);
            mbar_init(bar(kVEmpty + i), 1);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kSFull + i), 1);
            mbar_init(bar(kPFull + i), 4);
            mbar_init(bar(kODone + i), 1);
        }
        mbar_init(bar(kDone), 1);
        mbar_init(bar(kPVDone), 1);
        fence_proxy_async_smem();
    }
    // The copy warps start at once, without the setup barrier of the others: warp 0
    // tells them that the mbarriers exist (and whether an earlier call gave up).
    constexpr int kCopyThreads = 32 * (2 + kKWarps);       // warp 0 and the copy warps
    if (warp == 0) {
        __syncwarp();
        named_bar_arrive(1, kCopyThreads);
        // for the softmax and MMA warps, after their setup barrier
        if (lane == 0) *reinterpret_cast<volatile uint32_t*>(smem + L::SLOT + 4) = aborted_in;
    }
    // ---- copy warps.  V: one bulk copy per (block, kv head) tile, lane b handles block b.
    // K: the threads of the K warps copy each block tile's 16-byte pieces (piece c * 16 +
    // slot), consecutive threads on consecutive pieces, each to its chunk-major place, one
    // commit group per tile; a tile is published (its barrier completes) once every
    // thread has seen its own copies land and made them visible to the tensor cores (a
    // proxy fence in the writing thread).  Blocks past the tile's last one and entries
    // that are not blocks of the pool (flagged) are not copied: their columns of S are
    // masked, or the call has failed.  The copy warps start while the others set up.
    const bool vwarp = warp == kProducerWarp, kwarp = warp >= kKWarp && warp < kKWarp + kKWarps;
    int wcur = 0, issued = 0;
    auto block_of = [&](int j) {
        while (j / kWinTiles > wcur) {
            win = win_next;
            ++wcur;
            win_next = fetch_window(trow, wcur + 1, nblk, lane);
        }
        return window_block(win, j, lane, nblk);
    };
    auto issue_v = [&](int j, uint64_t pol) {
        const int st = j % VST;
        int32_t blk = block_of(j);
        const uint32_t bytes = check_blocks(p, blk, j, nblk, lane, TILE);
        if (lane == 0) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar(kVFull + st), bytes);
        }
        __syncwarp();
        if (lane < kKeyBlocks && blk >= 0)
            bulk_g2s(sV + st * KTILE + lane * TILE, p.v_pool + ((size_t)blk * p.Hkv + kvh) * (size_t)TILE,
                     TILE, bar(kVFull + st), pol);
        issued = j + 1;
    };
    auto issue_k = [&](int j, uint64_t pol) {
        constexpr int kPer = kBlockTokens * (D / 8) / (32 * kKWarps);   // pieces per thread and block
        const int kt = (warp - kKWarp) * 32 + lane;
        const int st = j % KST;
        int32_t blk = block_of(j);
        check_blocks(p, blk, j, nblk, lane, TILE);
        const uint32_t dst = sK + st * KTILE;
#pragma unroll
        for (int b = 0; b < kKeyBlocks; ++b) {
            const int32_t bb = __shfl_sync(0xffffffffu, blk, b);
            if (bb >= 0) {
                const char* src = p.k_pool + ((size_t)bb * p.Hkv + kvh) * (size_t)TILE;
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const int piece = u * 32 * kKWarps + kt;
                    cp_async_16(dst + (piece >> 4) * (kKeyBlocks * 256) + b * 256 + (piece & 15) * 16,
                                src + piece * 16, pol);
                }
            }
        }
        cp_async_commit();
        issued = j + 1;
    };
    // before exit: every copy of the warp has landed (and every arrival it triggers)
    auto drain = [&]() {
        if (kwarp) {
            cp_async_wait<0>();
        } else if (vwarp && lane == 0) {
            for (int jj = max(0, issued - VST); jj < issued; ++jj)
                mbar_wait_bounded(bar(kVFull + jj % VST), (jj / VST) & 1, kWaitLimitNs);
        }
    };
    // Roles.  setmaxnreg is collective over a warpgroup, so each runs at the head of its
    // branch: the copy / MMA warpgroups hand registers to the softmax warpgroups, which
    // take them after their setup (8 x 32 x 200 + 4 x 32 x 104 <= 384 x 168, the launch's
    // allocation, with two Q tiles; 4 x 32 x 200 + 8 x 32 x 104 with one).
    if (warp >= kSoftWarps) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 104;" ::: "memory");
    if (vwarp || kwarp) {
        const bool gave_up = __shfl_sync(0xffffffffu, flag_in & PA_DEV_ERR_TIMEOUT, 0) != 0;
        named_bar_sync(1, kCopyThreads);
        if (!gave_up) {
            if (!PREFIX) grid_dependency_wait();  // the chunk's own K/V come from the append before
            __syncwarp();
            if (vwarp) {
                // ---------------------------------------------------------------- V tiles
                if (lane == 0) grid_launch_dependents();
                const uint64_t pol = l2_policy_evict_last();   // tiles are re-read by other query tiles
                bool ok = true;
                for (int j = 0; j < ntiles; ++j) {
                    if (j >= VST) {                          // PV of tile j - VST is done
                        ok = warp_wait(bar(kVEmpty + j % VST), (j / VST - 1) & 1);
                        if (!ok) break;
                    }
                    issue_v(j, pol);
                }
                if (!ok && lane == 0) raise_flag(p.err, PA_DEV_ERR_TIMEOUT);
                } else {
                // ---------------------------------------------------------------- K tiles
                // Tiles are published in order, each as soon as its copies have landed; a new
                // tile is issued whenever its stage is free (the S MMAs of the tile KST earlier
                // are done), tested without waiting while copies are in flight.
                static_assert(KST <= 3, "the landing waits below cover up to two newer tiles");
                const uint64_t pol = l2_policy_evict_last();   // tiles are re-read by other query tiles
                auto stage_free = [&](int j) {
                    return j < KST || __all_sync(0xffffffffu, mbar_test(bar(kKEmpty + j % KST), (j / KST - 1) & 1));
                };
                bool ok = true;
                for (int pub = 0; pub < ntiles; ++pub) {
                    // (two tiles ahead at most; the first alone, as the first scores wait for it)
                    while (issued < ntiles && issued - pub < (pub == 0 ? 1 : 2) && stage_free(issued))
                        issue_k(issued, pol);
                    if (issued == pub) {               // nothing in flight: wait for the stage
                        ok = warp_wait(bar(kKEmpty + issued % KST), (issued / KST - 1) & 1);
                        if (!ok) break;
                        issue_k(issued, pol);
                    }
                    const int newer = issued - pub - 1;   // this thread's tiles after `pub` in flight
                    if (newer >= 2) cp_async_wait<2>();
                    else if (newer == 1) cp_async_wait<1>();
                    else cp_async_wait<0>();
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(kKFull + pub % KST));
                }
                if (!ok && lane == 0) raise_flag(p.err, PA_DEV_ERR_TIMEOUT);
                }
        }
        drain();
    } else if (warp == kMmaWarp) {
    tmem_alloc<kTmemCols>(sbase + L::SLOT);
    tc_fence_before();
    named_bar_sync(2, 32 * (kSoftWarps + 1));          // Q is in place, the TMEM allocated
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::SLOT);
    if (*reinterpret_cast<volatile uint32_t*>(smem + L::SLOT + 4) == 0u) {   // (else write nothing)

        // ---------------------------------------------------------------- MMA issue
        // S_h(j) = Q_h K_j^T: A = Q_h (shared), B = the chunk-major K tile, N = 128 tokens.
        // O_h += P_h(j) V_j: A = P_h(j) in TMEM (over S_h's first columns), B = one V block
        // tile (MN-major), K = 16 tokens.  MMAs of this thread execute in issue order, so
        // S_h(j + 1) overwrites P_h(j) only after PV_h(j) has read it, and a commit after
        // S_h(j + 1) also covers PV_h(j).  Without a tile b its S columns are a second S
        // buffer for tile a: S(j) goes to buffer j % 2 and S(j + 2) is issued right after
        // PV(j), so the scores of the next tile are ready when the softmax finishes.
        constexpr uint32_t idS = umma_idesc_bf16(128, kKeyTok, 0);
        constexpr uint32_t idO = umma_idesc_bf16(128, D, 1);
        bool ok = true;
        auto issue_s = [&](int hh, int buf, int j) {
            tc_fence_after();
            if (lane == 0) {
                // columns of blocks past the tile's last one hold stale products (masked)
                const uint64_t qdesc = umma_desc(sQ + hh * L::QTILE, 2048, 128);
                const uint64_t kdesc = umma_desc(sK + (j % KST) * KTILE, kKeyBlocks * 256, 128);
                const uint32_t dcol = tmem + kColS + (uint32_t)(buf * kKeyTok);
#pragma unroll
                for (int ks = 0; ks < KSTEPS; ++ks)
                    umma_ss(dcol, qdesc + (uint64_t)(ks * 256),
                            kdesc + (uint64_t)((ks * 2 * kKeyBlocks * 256) >> 4), idS, ks > 0);
                umma_commit(bar(kSFull + buf));
            }
            __syncwarp();
        };
        auto issue_pv = [&](int hh, int j, int buf) {
            const int st = j % VST;
            // (one Q tile: P(j) comes on barrier j % 2, as S is double-buffered -- the softmax
            // may write P(j + 1) before this wait for P(j) begins, and a parity wait on one
            // barrier could not tell its phase j + 2 from phase j)
            ok = has_b ? warp_wait(bar(kPFull + hh), j & 1) : warp_wait(bar(kPFull + (j & 1)), (j >> 1) & 1);
            if (!ok) return;
            const int nb = min(kKeyBlocks, nblk - j * kKeyBlocks);
            if (hh == 0) {
                ok = warp_wait(bar(kVFull + st), (j / VST) & 1);
                if (!ok) return;
                if (j == ntiles - 1) {
                    // V rows past the last attended position may hold anything (even NaN)
                    const int first_stale = p_last - (nblk - 1) * kBlockTokens + 1;
                    if (first_stale < kBlockTokens) {
                        const int nst = kBlockTokens - first_stale;
                        uint8_t* vt = smem + L::V + st * KTILE + (nb - 1) * TILE;
                        for (int idx = lane; idx < (D / 8) * nst; idx += 32) {
                            const int c = idx / nst, sl = first_stale + (idx - c * nst);
                            *reinterpret_cast<uint4*>(vt + c * 256 + sl * 16) = make_uint4(0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();
                    }
                    __syncwarp();
                }
            }
            tc_fence_after();
            if (lane == 0) {
                const uint64_t vdesc = umma_desc(sV + st * KTILE, 128, 256);
                const uint32_t pcol = tmem + kColS + (uint32_t)(buf * kKeyTok);
                const uint32_t ocol = tmem + kColO + (uint32_t)(hh * kKeyTok);
                for (int b = 0; b < nb; ++b)
                    umma_ts(ocol, pcol + 8 * b, vdesc + (uint64_t)((b * TILE) >> 4), idO,
                            (j > 0 || b > 0) ? 1u : 0u);
                if (j == ntiles - 1) umma_commit(bar(kODone + hh));
                if (hh == 1 || !has_b) umma_commit(bar(kVEmpty + st));
                if (!has_b) umma_commit(bar(kPVDone));
            }
            __syncwarp();
        };
        auto k_ready = [&](int j) { return warp_wait(bar(kKFull + j % KST), (j / KST) & 1); };
        auto k_free = [&](int j) {                // after the tile's last S MMA
            if (lane == 0) umma_commit(bar(kKEmpty + j % KST));
            __syncwarp();
        };
        auto next_s = [&](int j, int buf) {       // S of tile j for tile a, then free the K tile
            ok = k_ready(j);
            if (!ok) return;
            issue_s(0, buf, j);
            k_free(j);
        };
        if (!has_b) {
            // one Q tile, S double-buffered: S(0) S(1) | PV(0) S(2) | PV(1) S(3) ...
            next_s(0, 0);
            if (ok && ntiles > 1) next_s(1, 1);
            for (int j = 0; ok && j < ntiles; ++j) {
                issue_pv(0, j, j & 1);
                if (ok && j + 2 < ntiles) next_s(j + 2, j & 1);
            }
        } else {
            // two Q tiles: S_a(0) S_b(0) | PV_a(0) S_a(1) PV_b(0) S_b(1) | ...
            ok = k_ready(0);
            if (ok) {
                issue_s(0, 0, 0);
                issue_s(1, 1, 0);
                k_free(0);
            }
            for (int j = 0; ok && j < ntiles; ++j) {
                const bool more = j + 1 < ntiles;
                issue_pv(0, j, 0);
                if (!ok) break;
                if (more) {
                    ok = k_ready(j + 1);
                    if (!ok) break;
                    issue_s(0, 0, j + 1);
                }
                issue_pv(1, j, 1);
                if (!ok) break;
                if (more) {
                    issue_s(1, 1, j + 1);
                    k_free(j + 1);
                }
            }
        }
        if (!ok && lane == 0) raise_flag(p.err, PA_DEV_ERR_TIMEOUT);
        // nothing may still be running on the tensor cores when TMEM is freed
        if (lane == 0) umma_commit(bar(kDone));
        __syncwarp();
        mbar_wait_bounded(bar(kDone), 0, kWaitLimitNs);
            }
    }
    } else {
    // rows: (chunk token, query head of this kv head), token-major; one per softmax thread
    const int row = threadIdx.x;                          // 0 .. 255 for the softmax warps
    const int h = warp >> 2;                              // Q tile of a softmax warp
    int pos = p_last;                                     // rows outside the chunk see all (finite)
    bool row_valid = false;
    size_t orow = 0;
    if (warp < kSoftWarps) {
        if constexpr (PREFIX) {
            const int r = row_base + row, sq = r / p.G, g = r - sq * p.G;
            row_valid = row < p.rows_per_cta && r < rows_total;
            if (row_valid) orow = (size_t)sq * p.Hq + (size_t)kvh * p.G + g;   // partial row
        } else {
            const int tl = row / p.G, g = row - tl * p.G;
            row_valid = tl < p.TQ && i0 + tl < n;
            if (row_valid) {
                pos = start + i0 + tl;
                orow = ((size_t)(q0 + i0 + tl) * p.Hq + (size_t)kvh * p.G + g) * D;
            }
            grid_dependency_wait();
        }
        const uint4* qsrc = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                           (PREFIX ? orow * D : orow));
        const int lr = row & (kHalfRows - 1);
        const uint32_t qdst = sQ + h * L::QTILE + (uint32_t)((lr >> 3) * 128 + (lr & 7) * 16);
        // a negative scale is applied as |scale| to -q (exact), so that the softmax can
        // take the row maximum of the unscaled scores
        const uint32_t flip = p.scale_log2 < 0.f ? 0x80008000u : 0u;
        // the whole row's loads in flight together, then the stores: one round trip on the
        // critical path of the CTA's first scores
        constexpr int QB = D / 8;
#pragma unroll
        for (int k0 = 0; k0 < D / 8; k0 += QB) {
            uint4 qv[QB];
#pragma unroll
            for (int u = 0; u < QB; ++u)
                qv[u] = row_valid ? __ldg(qsrc + k0 + u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int u = 0; u < QB; ++u) {
                uint4 v = qv[u];
                v.x ^= flip;
                v.y ^= flip;
                v.z ^= flip;
                v.w ^= flip;
                st_shared_v4(qdst + (k0 + u) * 2048, v);
            }
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    named_bar_sync(2, 32 * (kSoftWarps + 1));
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::SLOT);
    if (*reinterpret_cast<volatile uint32_t*>(smem + L::SLOT + 4) == 0u) {   // (else write nothing)
    // (every warp of both softmax warpgroups, at this one instruction)
    asm volatile("setmaxnreg.inc.sync.aligned.u32 200;" ::: "memory");
    if (h == 0 || has_b) {
        // ---------------------------------------------------------------- softmax rows
        // Warp w reaches TMEM lanes 32 (w % 4) ..; this thread's row of tile h is lane
        // row % 128.  With two tiles a commit after S_h(j) covers every earlier MMA, so when
        // S_h(j) is seen complete, PV_h(j - 1) is too: O_h may be rescaled and P_h(j)
        // written at once.
        const uint32_t tl_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        // without a tile b, tile a's S alternates between both S buffers (see the MMA warp)
        const uint32_t ocol = kColO + (uint32_t)(h * kKeyTok);
        const float cs = fabsf(p.scale_log2);          // a negative scale was moved into Q
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const int sb = has_b ? h : (j & 1);
            const uint32_t scol = kColS + (uint32_t)(sb * kKeyTok);
            ok = warp_wait(bar(kSFull + sb), has_b ? (j & 1) : ((j >> 1) & 1));
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tl_addr + scol + 32 * c, sr[c]);
            tmem_wait_ld();
            const int tok0 = j * kKeyTok;
            // every key of the tile is visible to every row of the warp: warp-uniform, so
            // that the warp-collective TMEM stores below run with all 32 lanes
            const bool full = __all_sync(0xffffffffu, tok0 + kKeyTok - 1 <= pos);
            float mx;
            if (full) {
                // the row maximum of the unscaled scores (c >= 0), four independent chains
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; i += 2)
                        m4[c] = max3f(m4[c], __uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1]));
                mx = max3f(m4[0], m4[1], fmaxf(m4[2], m4[3])) * cs;
            } else {
                // scale and causal mask (select: unread or stale columns may hold NaN)
                mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float x = tok0 + 32 * c + i <= pos ? __uint_as_float(sr[c][i]) * cs : -INFINITY;
                        sr[c][i] = __float_as_uint(x);
                        mx = fmaxf(mx, x);
                    }
            }
            float alpha = 1.f;
            bool resc = false;
            if (mx > m_used + kRescaleLog2) {              // first tile: m_used = -inf
                alpha = fast_exp2(m_used - mx);
                resc = j > 0;
                m_used = mx;
            }
            if (__any_sync(0xffffffffu, resc)) {
                // with S double-buffered, S(j) complete does not imply PV(j - 1) complete:
                // wait for it before O changes (the barrier is at most one phase ahead)
                if (!has_b) {
                    ok = warp_wait(bar(kPVDone), (j - 1) & 1);
                    if (!ok) break;
                    tc_fence_after();
                }
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tl_addr + ocol + 32 * c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(tl_addr + ocol + 32 * c, o);
                }
            }
            // probabilities, bf16 pairs, over the first 64 columns of S_h (already read);
            // a full tile takes s c - m for two keys in one packed FFMA and sums in pairs
            float sum;
            if (full) {
                const uint64_t c2 = pack_f32x2(cs, cs), nm2 = pack_f32x2(-m_used, -m_used);
                uint64_t sum2[2] = {pack_f32x2(0.f, 0.f), pack_f32x2(0.f, 0.f)};
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t pk[32];
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const int c = 2 * half + cc;
                            const uint64_t x2 = ffma_f32x2(pack_f32x2(__uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1])), c2, nm2);
                            const float e0 = fast_exp2(lo_f32(x2)), e1 = fast_exp2(hi_f32(x2));
                            sum2[(i >> 1) & 1] = fadd_f32x2(sum2[(i >> 1) & 1], pack_f32x2(e0, e1));
                            pk[16 * cc + (i >> 1)] = pack_bf16x2(e0, e1);
                        }
                    tmem_st32(tl_addr + scol + 32 * half, pk);
                }
                const uint64_t t = fadd_f32x2(sum2[0], sum2[1]);
                sum = lo_f32(t) + hi_f32(t);
            } else {
                sum = 0.f;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t pk[32];
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const int c = 2 * half + cc;
                            const float e0 = fast_exp2(__uint_as_float(sr[c][i]) - m_used);
                            const float e1 = fast_exp2(__uint_as_float(sr[c][i + 1]) - m_used);
                            sum += e0 + e1;
                            pk[16 * cc + (i >> 1)] = pack_bf16x2(e0, e1);
                        }
                    tmem_st32(tl_addr + scol + 32 * half, pk);
                }
            }
            l = l * alpha + sum;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kPFull + (has_b ? h : (j & 1))));
        }
        if (ok) ok = warp_wait(bar(kODone + h), 0);
        if (ok && PREFIX) {
            tc_fence_after();
            // Each 32-column piece of the warp's 32 rows passes through shared memory (the K
            // stages: every MMA has completed), 16-byte units of row r at unit u ^ (r % 8),
            // so that both the writes and the reads are free of bank conflicts and each
            // global store covers 128 contiguous bytes of four rows (a thread storing its
            // own row scatters 16-byte pieces over 32 rows per instruction).
            const size_t slot = orow * p.part_stride + (size_t)blockIdx.z * p.slot_mult;
            const uint32_t stg = sK + (uint32_t)warp * (32 * 128);
            const uint32_t valid = __ballot_sync(0xffffffffu, row_valid);
            const int sub = lane >> 3, unit = lane & 7;       // row 4 i + sub, unit `unit`
            float* dst[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const unsigned long long a = __shfl_sync(0xffffffffu, (unsigned long long)(p.part_o + slot * D), 4 * i + sub);
                dst[i] = reinterpret_cast<float*>(a) + unit * 4;
            }
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tl_addr + ocol + 32 * c, o);
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    st_shared_v4(stg + lane * 128 + ((u ^ (lane & 7)) * 16),
                                 make_uint4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]));
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = 4 * i + sub;
                    const uint4 v = ld_shared_v4(stg + r * 128 + ((unit ^ (r & 7)) * 16));
                    if ((valid >> r) & 1u)
                        *reinterpret_cast<uint4*>(dst[i] + 32 * c) = v;
                }
                __syncwarp();
            }
            if (row_valid) p.part_ml[slot] = make_float2(m_used, l);
        } else if (ok) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + orow);
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tl_addr + ocol + 32 * c, o);
                tmem_wait_ld();
                if (row_valid) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
                        dst[4 * c + v] = w;
                    }
                }
            }
        } else {
            // a wait gave up: the row's result is incomplete, so it is written as NaN (visible
            // even when no error flag was given)
            if (lane == 0) raise_flag(p.err, PA_DEV_ERR_TIMEOUT);
            if (row_valid) {
                if constexpr (PREFIX) {
                    p.part_ml[orow * p.part_stride + (size_t)blockIdx.z * p.slot_mult] =
                        make_float2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + orow);
                    for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
                }
            }
        }
    }
            }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc<kTmemCols>(*reinterpret_cast<volatile uint32_t*>(smem + L::SLOT));
    }
    // (prefix mode: every thread has waited for the previous grid; this is a no-op then)
    if (PREFIX) grid_dependency_wait();
}

}  // namespace tc

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    // all of the SM's unified memory as shared memory, so that CTAs of the decode and
    // prefix kernels can share an SM whatever the carve-out the other asked for
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int D, bool PREFIX, int SW>
cudaError_t launch_tc(const PParams& pp, dim3 grid, cudaStream_t stream) {
    auto k = tc::prefill_tc_kernel<D, PREFIX, SW>;
    constexpr int smem = tc::Smem<D, SW>::BYTES;
    cudaError_t e = set_smem(k, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(tc::Roles<SW>::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, pp);
}

PParams common_params(const void* q, const void* k_pool, const void* v_pool, const int32_t* tables,
                      int32_t* err, int Hq, int Hkv, int max_blocks, int num_blocks, float scale) {
    PParams pp = {};
    pp.q = q;
    pp.k_pool = static_cast<const char*>(k_pool);
    pp.v_pool = static_cast<const char*>(v_pool);
    pp.tables = tables;
    pp.err = err;
    pp.Hq = Hq;
    pp.Hkv = Hkv;
    pp.G = Hq / Hkv;
    pp.max_blocks = max_blocks;
    pp.num_blocks = num_blocks;
    pp.scale_log2 = scale * kLog2e;
    return pp;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 148;
    return n;
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
    PParams pp = common_params(a.q, a.k_pool, a.v_pool, a.block_tables, a.err, a.num_q_heads,
                               a.num_kv_heads, a.max_blocks, a.num_blocks, a.scale);
    pp.out = a.out;
    pp.start_pos = a.start_pos;
    pp.cu_q = a.cu_q;
    pp.TQ = tc::kRowsTC / pp.G;
    const dim3 grid((a.max_chunk + pp.TQ - 1) / pp.TQ, pp.Hkv, a.num_seqs);
    if (a.head_dim == 64) return launch_tc<64, false, 2>(pp, grid, stream);
    return launch_tc<128, false, 2>(pp, grid, stream);
}

cudaError_t launch_prefix_tc(const DecodeArgs& a, bool after_suffix, cudaStream_t stream) {
    // (after_suffix: an older launch order; the decode path now starts this kernel first)
    PParams pp = common_params(a.q, a.k_pool, a.v_pool, a.block_tables, a.err, a.num_q_heads,
                               a.num_kv_heads, a.max_blocks, a.num_blocks, a.scale);
    const size_t prow = (size_t)a.num_seqs * a.num_q_heads * a.part_stride;
    pp.part_o = static_cast<float*>(a.workspace);
    pp.part_ml = reinterpret_cast<float2*>(static_cast<char*>(a.workspace) + prow * a.head_dim * sizeof(float));
    pp.part_stride = a.part_stride;
    pp.num_seqs = a.num_seqs;
    pp.wait_first = after_suffix ? 0 : 1;
    // Prefix CTAs take an SM each; one covers several decode partitions: fewer CTAs, each
    // longer, which leaves SMs to the suffix decode running beside them and cuts the
    // partials the merge reads.
    pp.slot_mult = prefix_slot_mult(a.first_part);
    pp.part_blocks = a.part_blocks * pp.slot_mult;
    const int pre_parts = a.first_part / pp.slot_mult;
    // 256 rows (two Q tiles) per CTA when that still gives every SM a CTA, else 128
    const int rows = a.num_seqs * pp.G;
    const long long ctas256 = (long long)((rows + tc::kRowsTC - 1) / tc::kRowsTC) * a.num_kv_heads * pre_parts;
    pp.rows_per_cta = ctas256 >= sm_count() ? tc::kRowsTC : tc::kHalfRows;
#ifdef PA_PREFIX_TC_ROWS
    pp.rows_per_cta = PA_PREFIX_TC_ROWS;              // tuning builds: 128 or 256
#endif
    const dim3 grid((rows + pp.rows_per_cta - 1) / pp.rows_per_cta, a.num_kv_heads, pre_parts);
    const bool one = pp.rows_per_cta <= tc::kHalfRows;    // one Q tile: one softmax warpgroup
    if (a.head_dim == 64)
        return one ? launch_tc<64, true, 1>(pp, grid, stream) : launch_tc<64, true, 2>(pp, grid, stream);
    return one ? launch_tc<128, true, 1>(pp, grid, stream) : launch_tc<128, true, 2>(pp, grid, stream);
}

}  // namespace pa

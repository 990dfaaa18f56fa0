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
// Work split: an item = (query tile, kv head, sequence).  Rows are (chunk token,
// query head of the kv head) pairs, token-major, 256 / G tokens per item, in two
// Q tiles of 128 rows that share every K/V tile.  The grid is persistent, one CTA
// per SM; each CTA sorts the items by their key tiles (the same way in every CTA)
// and takes its share of them, dealt out largest first, and while one item ends
// it already loads the next one's query rows and K/V tiles.  The 5th-generation
// tensor cores (tcgen05) compute, per key tile of 128 tokens (8 blocks) and Q tile h,
//   S_h = Q_h K^T   into TMEM (one M128 N128 K16 MMA per 16 dims),
//   O_h += P_h V    into TMEM (one M128 N=D K16 MMA per block, P_h from TMEM),
// one thread issuing every MMA; the softmax runs one row per thread of eight
// warps (a warpgroup per Q tile), with the causal mask applied per row.
#include <cuda_bf16.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>

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
    // prefill: query tiles per chunk (of TQ tokens) and work items (nqt x Hkv x num_seqs)
    int nqt, num_items;
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
// columns as a second S buffer for tile a.  (Scores in 64-key halves, double-buffered
// per Q tile in the same TMEM columns, were measured slower: an M128 N64 MMA takes
// about as long as an M128 N128 one, 33-36 ns on GB300, so the halves double the cost
// of Q K^T.)
// ============================================================================

namespace tc {

// Two Q tiles of 128 rows (a, b) per item share every K/V tile; each has its own softmax
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
    static constexpr int NBAR = 28;
    // SLOT: TMEM address, aborted flag, length of the CTA's item list (-1: none)
    static constexpr int SLOT = BAR + NBAR * 8;
    static constexpr int LIST = SLOT + 16;                     // the CTA's items, in order
    static constexpr int LISTCAP = (232448 - LIST) / 16 < 1024 ? (232448 - LIST) / 16 : 1024;
    // at least 120 KB so that one CTA (and its 512 TMEM columns) owns an SM
    static constexpr int END = LIST + 16 * LISTCAP;
    static constexpr int BYTES = END < 122880 ? 122880 : END;
    static_assert(END <= 232448, "shared memory of one CTA");
    // the schedule's counters and group costs use the Q tiles before the queries are stored
    static constexpr int SCRATCH = NQ * QTILE / 4;
};

// barrier indices (rings of up to 4 stages)
constexpr int kKFull = 0, kKEmpty = 4, kVFull = 8, kVEmpty = 12, kSFull = 16, kPFull = 18,
              kODone = 20, kDone = 22, kPVDone = 23, kQFull = 24, kOFree = 26;

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

// One 32-byte store (the address a multiple of 32).
__device__ __forceinline__ void st_global_v8(void* addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                             uint32_t e, uint32_t f, uint32_t g, uint32_t h) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(addr), "r"(a), "r"(b),
                 "r"(c), "r"(d), "r"(e), "r"(f), "r"(g), "r"(h)
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

// One work item: the prefill's (query tile, kv head, sequence) triple, natural index
// (s Hkv + kvh) nqt + x with query tile nqt - 1 - x, or the prefix mode's one (row group,
// kv head, partition range) per CTA.
struct Item {
    int kvh, row_base;          // row_base: prefix mode
    int qrow0, p0, rows;        // prefill: the tile's first chunk row (a row of q), its position, its rows
    int p_last, nblk;           // last position attended to, blocks read
    const int32_t* trow;
    bool live;                  // rows and keys to process
    bool bad_pos;               // a position outside the table (flagged, skipped)
};
// The prefill's items as the CTA's list keeps them: the natural index and the geometry that
// would otherwise take three dependent loads per item.
struct ListEntry { int it, qrow0, p0, rows; };

__device__ __forceinline__ Item finish_item(const PParams& p, int it, int qrow0, int p0, int rows) {
    Item g{};
    const int s = it / (p.nqt * p.Hkv);
    g.kvh = it / p.nqt - s * p.Hkv;
    g.qrow0 = qrow0;
    g.p0 = p0;
    g.rows = rows;
    g.trow = p.tables + (size_t)s * p.max_blocks;
    if (rows <= 0) return g;
    g.p_last = p0 + rows - 1;
    if (p0 < 0 || g.p_last >= p.max_blocks * kBlockTokens) {
        g.bad_pos = true;
        return g;
    }
    g.nblk = g.p_last / kBlockTokens + 1;
    g.live = true;
    return g;
}
template <bool PREFIX>
__device__ __forceinline__ Item item_at(const PParams& p, int it) {
    if constexpr (PREFIX) {
        Item g{};
        g.kvh = blockIdx.y;
        g.row_base = blockIdx.x * p.rows_per_cta;
        g.nblk = p.part_blocks;
        g.p_last = g.nblk * kBlockTokens - 1;             // positions relative to the partition
        g.trow = p.tables + (size_t)blockIdx.z * p.part_blocks;
        g.live = true;
        return g;
    } else {
        const int x = it % p.nqt, s = it / (p.nqt * p.Hkv);
        const int i0 = (p.nqt - 1 - x) * p.TQ;
        // the chunk's place: three loads in flight together
        const int q0 = __ldg(p.cu_q + s), q1 = __ldg(p.cu_q + s + 1), start = __ldg(p.start_pos + s);
        // (a chunk's start is checked with its first tile's positions)
        return finish_item(p, it, q0 + i0, start < 0 ? -1 : start + i0, min(q1 - q0 - i0, p.TQ));
    }
}
// Cost of the items of query tile nqt - 1 - x of sequence s (every kv head alike): their
// key tiles, 0 without work, -1 for positions outside the table.
__device__ __forceinline__ int group_cost(const PParams& p, int grp) {
    const Item g = item_at<false>(p, grp / p.nqt * p.Hkv * p.nqt + grp % p.nqt);
    if (g.bad_pos) return -1;
    return g.live ? (g.nblk + kKeyBlocks - 1) / kKeyBlocks : 0;
}

// The prefill's schedule.  The grid is persistent (at most one CTA per SM); the items,
// sorted by decreasing cost (key tiles; ties by natural index), are dealt out in rounds of
// gridDim.x: in CTA order in even rounds and reverse order in odd ones, and the last round
// to the CTAs in order of their load so far (least loaded first, each item's estimated time
// being 1.79 us per key tile plus 3.7 us), so that every CTA ends up with about the same
// work (a static stride over the natural order leaves the CTAs that drew long chunks well
// behind, and the plain alternation leaves the CTAs that take a last item behind those that
// do not).  Every CTA sorts the (sequence, query tile) groups itself, the same way: the
// groups' costs and their histogram, a scan over the costs from the largest, and a
// placement of the groups in natural order by one warp (equal costs keep that order); it
// keeps the list of its own items with their geometry.  Where the costs or the list would
// not fit, the CTA takes items blockIdx.x, + gridDim.x, ... instead (list length -1).
constexpr int kTileCost = 179, kItemCost = 370;      // (units of 10 ns)
template <int D>
__device__ void build_schedule(const PParams& p, uint8_t* smem) {
    using L = Smem<D, 2>;
    int* cnt = reinterpret_cast<int*>(smem + L::Q);      // [ncost] counts, then offsets
    ListEntry* list = reinterpret_cast<ListEntry*>(smem + L::LIST);
    volatile int* nlist = reinterpret_cast<volatile int*>(smem + L::SLOT + 8);
    const int grid = gridDim.x, cta = blockIdx.x;
    const int ncost = (p.max_blocks + kKeyBlocks - 1) / kKeyBlocks + 1;     // costs 0 .. ncost - 1
    const int ngroups = p.num_seqs * p.nqt;
    // per group: cost, first row, its position, rows; the groups in sorted order; the CTAs' loads
    int* gcost = cnt + ncost;
    int* gq = gcost + ngroups;
    int* gp = gq + ngroups;
    int* gr = gp + ngroups;
    int* order = gr + ngroups;
    int* load = order + ngroups;
    const bool sorted = (long long)ncost + 5ll * ngroups + grid + 1 <= L::SCRATCH &&
                        (p.num_items + grid - 1) / grid <= L::LISTCAP;
    const int tid = threadIdx.x, nthr = blockDim.x;
    if (!sorted) {
        // positions outside the table, flagged once: each CTA checks its share of the groups
        for (int g = cta * nthr + tid; g < ngroups; g += grid * nthr)
            if (group_cost(p, g) < 0) raise_flag(p.err, PA_DEV_ERR_BAD_POS);
        if (tid == 0) *nlist = -1;
        __syncthreads();
        return;
    }
    for (int c = tid; c < ncost; c += nthr) cnt[c] = 0;
    __syncthreads();
    for (int g = tid; g < ngroups; g += nthr) {
        const Item it = item_at<false>(p, g / p.nqt * p.Hkv * p.nqt + g % p.nqt);
        const int c = it.bad_pos ? -1 : it.live ? (it.nblk + kKeyBlocks - 1) / kKeyBlocks : 0;
        gcost[g] = c;
        gq[g] = it.qrow0;
        gp[g] = it.p0;
        gr[g] = it.rows;
        if (c > 0) atomicAdd(&cnt[c], 1);
        else if (c < 0 && cta == 0) raise_flag(p.err, PA_DEV_ERR_BAD_POS);
    }
    __syncthreads();
    if (tid < 32) {
        const int lane = tid;
        // cnt[c] := groups of cost > c (an exclusive scan from the top)
        int run = 0;
        for (int c0 = ncost - 1; c0 >= 0; c0 -= 32) {
            const int c = c0 - lane;
            const int v = c >= 0 ? cnt[c] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            if (c >= 0) cnt[c] = run + incl - v;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        __syncwarp();
        // order[position] = group
        const uint32_t lt = (1u << lane) - 1u;
        for (int g0 = 0; g0 < ngroups; g0 += 32) {
            const int g = g0 + lane;
            const int c = g < ngroups ? gcost[g] : 0;
            const uint32_t same = __match_any_sync(0xffffffffu, c > 0 ? c : -1);
            int pos = 0;
            if (c > 0) pos = cnt[c] + __popc(same & lt);
            __syncwarp();
            if (c > 0 && (same & lt) == 0u) cnt[c] += __popc(same);
            __syncwarp();
            if (c > 0) order[pos] = g;
        }
        if (lane == 0) load[grid] = run;              // live groups
    }
    __syncthreads();
    const int total = load[grid] * p.Hkv;              // live items
    const int rounds = (total + grid - 1) / grid;
    // item of rank R (position R / Hkv of the sorted groups, kv head R % Hkv)
    auto entry = [&](int R) {
        const int g = order[R / p.Hkv], s = g / p.nqt, x = g - s * p.nqt;
        return ListEntry{(s * p.Hkv + R % p.Hkv) * p.nqt + x, gq[g], gp[g], gr[g]};
    };
    auto snake = [&](int rd, int c) { return rd * grid + ((rd & 1) ? grid - 1 - c : c); };
    // the rounds before the last, alternating: every CTA's load, and this CTA's items
    for (int c = tid; c < grid; c += nthr) {
        int l = 0;
        for (int rd = 0; rd + 1 < rounds; ++rd) l += gcost[order[snake(rd, c) / p.Hkv]] * kTileCost + kItemCost;
        load[c] = l;
    }
    for (int rd = tid; rd + 1 < rounds; rd += nthr) list[rd] = entry(snake(rd, cta));
    __syncthreads();
    if (tid == 0 && rounds > 0) {
        // the last round: its k-th largest item to the CTA with the k-th smallest load
        const int mine = load[cta];
        int k = 0;
        for (int c = 0; c < grid; ++c) {
            const int l = load[c];
            k += (l < mine || (l == mine && c < cta)) ? 1 : 0;
        }
        const int R = (rounds - 1) * grid + k;
        if (R < total) list[rounds - 1] = entry(R);
        *nlist = R < total ? rounds : rounds - 1;
    } else if (tid == 0) {
        *nlist = 0;
    }
    __syncthreads();
}

// PREFIX = false: causal prefill of chunk rows.  Persistent: each CTA walks its list of
// (query tile, kv head, sequence) items, the next item's query rows, table windows and first
// K/V tiles loading while the current one finishes.  A CTA always runs both Q tiles (an item
// whose second tile has no chunk rows computes it on zero rows and stores nothing), so that
// every item takes the same barrier phases.
// PREFIX = true: one item per CTA; rows are (sequence, query head) pairs of the kv head
// (CTA = row group, kv head, partition range of a prefix shared by every sequence, read
// through table row 0); every key is visible and the CTA writes each row's unnormalised
// partial (o, max, sum) into the decode workspace for the split-KV merge.
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
    static_assert(PREFIX || SW == 2, "the prefill runs two Q tiles per CTA");
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (PREFIX && p.wait_first) grid_dependency_wait();
    // two Q tiles: the prefill always, the prefix mode when its rows fill both
    const bool has_b = SW == 2 && (!PREFIX || (p.rows_per_cta > kHalfRows &&
                                               (int)blockIdx.x * p.rows_per_cta + kHalfRows < p.num_seqs * p.G));

    // The TIMEOUT bit of the flag: set when a copy wait gave up in this or an earlier call
    // (then nothing is written).  Thread 0 reads it for the softmax and MMA warps, which
    // act on it after their setup barrier; the copy warps read it themselves.
    int32_t flag_in = 0;
    const bool vwarp = warp == kProducerWarp, kwarp = warp >= kKWarp && warp < kKWarp + kKWarps;
    if ((vwarp || kwarp) ? lane == 0 : threadIdx.x == 0)
        if (p.err) flag_in = *reinterpret_cast<const volatile int32_t*>(p.err);
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
        mbar_init(bar(kQFull), 4);
        mbar_init(bar(kQFull + 1), 4);
        mbar_init(bar(kOFree), kSoftWarps);
        fence_proxy_async_smem();
    }
    // The CTA's items: the i-th is item_of(i, the (i-1)-th), -1 past the last.
    if constexpr (!PREFIX) build_schedule<D>(p, smem);
    const int nlist = PREFIX ? 1 : *reinterpret_cast<volatile int*>(smem + L::SLOT + 8);
    const ListEntry* list = reinterpret_cast<const ListEntry*>(smem + L::LIST);
    auto item_of = [&](int i, int prev) -> int {       // a list position, or a natural index
        if constexpr (PREFIX) {
            return i == 0 ? 0 : -1;
        } else {
            if (nlist >= 0) return i < nlist ? i : -1;
            for (int it = i == 0 ? (int)blockIdx.x : prev + (int)gridDim.x; it < p.num_items; it += gridDim.x)
                if (item_at<false>(p, it).live) return it;
            return -1;
        }
    };
    auto item_get = [&](int idx) -> Item {             // the item item_of gave
        if constexpr (PREFIX) {
            return item_at<true>(p, 0);
        } else {
            if (nlist < 0) return item_at<false>(p, idx);
            const ListEntry e = list[idx];
            return finish_item(p, e.it, e.qrow0, e.p0, e.rows);
        }
    };
    // The copy warps start at once, without the setup barrier of the others: warp 0
    // tells them that the mbarriers exist (and whether an earlier call gave up).
    constexpr int kCopyThreads = 32 * (2 + kKWarps);       // warp 0 and the copy warps
    if (warp == 0) {
        __syncwarp();
        named_bar_arrive(1, kCopyThreads);
        // for the softmax and MMA warps, after their setup barrier
        if (lane == 0) *reinterpret_cast<volatile uint32_t*>(smem + L::SLOT + 4) = aborted_in;
    }

    // Roles.  setmaxnreg is collective over a warpgroup, so each runs at the head of its
    // branch: the copy / MMA warpgroups hand registers to the softmax warpgroups, which
    // take them after their setup (8 x 32 x 200 + 4 x 32 x 104 <= 384 x 168, the launch's
    // allocation, with two Q tiles; 4 x 32 x 200 + 8 x 32 x 104 with one).  Tile and item
    // counts run on across the CTA's items, so barrier phases and ring stages do too.
    if (warp >= kSoftWarps) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 104;" ::: "memory");
    if (vwarp || kwarp) {
        // ---------------------------------------------------------------- copy warps
        // V: one bulk copy per (block, kv head) tile, lane b handles block b.  K: the threads
        // of the K warps copy each block tile's 16-byte pieces (piece c * 16 + slot),
        // consecutive threads on consecutive pieces, each to its chunk-major place, one commit
        // group per tile; a tile is published (its barrier completes) once every thread has
        // seen its own copies land and made them visible to the tensor cores (a proxy fence
        // in the writing thread).  Blocks past the tile's last one and entries that are not
        // blocks of the pool (flagged) are not copied: their columns of S are masked, or the
        // call has failed.  The table is read in windows of four tiles, one window ahead.
        const bool gave_up = __shfl_sync(0xffffffffu, flag_in & PA_DEV_ERR_TIMEOUT, 0) != 0;
        int issued = 0;                               // tiles of all items issued so far
        named_bar_sync(1, kCopyThreads);
        if (!gave_up) {
            if (!PREFIX) grid_dependency_wait();  // the chunks' K/V come from the append before
            __syncwarp();
            if (vwarp && lane == 0) grid_launch_dependents();
            const uint64_t pol = l2_policy_evict_last();   // tiles are re-read by other query tiles
            bool ok = true;
            int t0 = 0;                               // tiles of the earlier items
            for (int i = 0, it = item_of(0, -1); ok && it >= 0; it = item_of(++i, it)) {
                const Item g = item_get(it);
                const int ntiles = (g.nblk + kKeyBlocks - 1) / kKeyBlocks;
                int32_t win = fetch_window(g.trow, 0, g.nblk, lane), win_next = fetch_window(g.trow, 1, g.nblk, lane);
                int wcur = 0;
                auto block_of = [&](int j) {
                    while (j / kWinTiles > wcur) {
                        win = win_next;
                        ++wcur;
                        win_next = fetch_window(g.trow, wcur + 1, g.nblk, lane);
                    }
                    return window_block(win, j, lane, g.nblk);
                };
                if (vwarp) {
                    for (int j = 0; j < ntiles; ++j) {
                        const int t = t0 + j, st = t % VST;
                        if (t >= VST) {                      // PV of tile t - VST is done
                            ok = warp_wait(bar(kVEmpty + st), (t / VST - 1) & 1);
                            if (!ok) break;
                        }
                        int32_t blk = block_of(j);
                        const uint32_t bytes = check_blocks(p, blk, j, g.nblk, lane, TILE);
                        if (lane == 0) {
                            fence_proxy_async_smem();
                            mbar_arrive_expect_tx(bar(kVFull + st), bytes);
                        }
                        __syncwarp();
                        if (lane < kKeyBlocks && blk >= 0)
                            bulk_g2s(sV + st * KTILE + lane * TILE,
                                     p.v_pool + ((size_t)blk * p.Hkv + g.kvh) * (size_t)TILE, TILE,
                                     bar(kVFull + st), pol);
                        issued = t + 1;
                    }
                } else {
                    // Tiles are published in order, each as soon as its copies have landed; a
                    // new tile is issued whenever its stage is free (the S MMAs of the tile
                    // KST earlier are done), tested without waiting while copies are in flight.
                    static_assert(KST <= 3, "the landing waits below cover up to two newer tiles");
                    constexpr int kPer = kBlockTokens * (D / 8) / (32 * kKWarps);   // pieces per thread and block
                    const int kt = (warp - kKWarp) * 32 + lane;
                    int jn = 0;                              // this item's next tile to issue
                    auto issue_k = [&]() {
                        const int t = t0 + jn, st = t % KST;
                        int32_t blk = block_of(jn);
                        check_blocks(p, blk, jn, g.nblk, lane, TILE);
                        const uint32_t dst = sK + st * KTILE;
#pragma unroll
                        for (int b = 0; b < kKeyBlocks; ++b) {
                            const int32_t bb = __shfl_sync(0xffffffffu, blk, b);
                            if (bb >= 0) {
                                const char* src = p.k_pool + ((size_t)bb * p.Hkv + g.kvh) * (size_t)TILE;
#pragma unroll
                                for (int u = 0; u < kPer; ++u) {
                                    const int piece = u * 32 * kKWarps + kt;
                                    cp_async_16(dst + (piece >> 4) * (kKeyBlocks * 256) + b * 256 + (piece & 15) * 16,
                                                src + piece * 16, pol);
                                }
                            }
                        }
                        cp_async_commit();
                        ++jn;
                        issued = t + 1;
                    };
                    auto stage_free = [&](int t) {
                        return t < KST || __all_sync(0xffffffffu, mbar_test(bar(kKEmpty + t % KST), (t / KST - 1) & 1));
                    };
                    for (int pub = 0; pub < ntiles; ++pub) {
                        // (two tiles ahead at most; the CTA's first tile alone, as the first
                        // scores wait for it)
                        while (jn < ntiles && jn - pub < (t0 + pub == 0 ? 1 : 2) && stage_free(t0 + jn)) issue_k();
                        if (jn == pub) {                     // nothing in flight: wait for the stage
                            ok = warp_wait(bar(kKEmpty + (t0 + jn) % KST), ((t0 + jn) / KST - 1) & 1);
                            if (!ok) break;
                            issue_k();
                        }
                        const int newer = jn - pub - 1;      // this thread's tiles after `pub` in flight
                        if (newer >= 2) cp_async_wait<2>();
                        else if (newer == 1) cp_async_wait<1>();
                        else cp_async_wait<0>();
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(kKFull + (t0 + pub) % KST));
                    }
                }
                t0 += ntiles;
            }
            if (!ok && lane == 0) raise_flag(p.err, PA_DEV_ERR_TIMEOUT);
        }
        // before exit: every copy of the warp has landed
        if (kwarp) {
            cp_async_wait<0>();
        } else if (lane == 0) {
            for (int t = max(0, issued - VST); t < issued; ++t)
                mbar_wait_bounded(bar(kVFull + t % VST), (t / VST) & 1, kWaitLimitNs);
        }
    } else if (warp == kMmaWarp) {
    tmem_alloc<kTmemCols>(sbase + L::SLOT);
    tc_fence_before();
    named_bar_sync(2, 32 * (kSoftWarps + 1));          // the TMEM is allocated
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
        // PV(j), so the scores of the next tile are ready when the softmax finishes.  An
        // item's scores start once its query rows are in place; its first P V (which starts
        // O afresh) once the previous item's O has been read.
        constexpr uint32_t idS = umma_idesc_bf16(128, kKeyTok, 0);
        constexpr uint32_t idO = umma_idesc_bf16(128, D, 1);
        bool ok = true;
        int t0 = 0;                                   // tiles of the earlier items
        for (int ic = 0, it = item_of(0, -1); ok && it >= 0; it = item_of(++ic, it)) {
            const Item g = item_get(it);
            const int nblk = g.nblk, ntiles = (nblk + kKeyBlocks - 1) / kKeyBlocks;
            auto issue_s = [&](int hh, int buf, int j) {
                tc_fence_after();
                if (lane == 0) {
                    // columns of blocks past the tile's last one hold stale products (masked)
                    const uint64_t qdesc = umma_desc(sQ + hh * L::QTILE, 2048, 128);
                    const uint64_t kdesc = umma_desc(sK + ((t0 + j) % KST) * KTILE, kKeyBlocks * 256, 128);
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
                const int t = t0 + j, st = t % VST;
                // (one Q tile: P(j) comes on barrier j % 2, as S is double-buffered -- the softmax
                // may write P(j + 1) before this wait for P(j) begins, and a parity wait on one
                // barrier could not tell its phase j + 2 from phase j)
                ok = has_b ? warp_wait(bar(kPFull + hh), t & 1) : warp_wait(bar(kPFull + (j & 1)), (j >> 1) & 1);
                if (!ok) return;
                if (j == 0 && hh == 0 && ic > 0) {
                    ok = warp_wait(bar(kOFree), (ic - 1) & 1);     // the last item's O is read
                    if (!ok) return;
                }
                const int nb = min(kKeyBlocks, nblk - j * kKeyBlocks);
                if (hh == 0) {
                    ok = warp_wait(bar(kVFull + st), (t / VST) & 1);
                    if (!ok) return;
                    if (j == ntiles - 1) {
                        // V rows past the last attended position may hold anything (even NaN)
                        const int first_stale = g.p_last - (nblk - 1) * kBlockTokens + 1;
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
            auto k_ready = [&](int j) { return warp_wait(bar(kKFull + (t0 + j) % KST), ((t0 + j) / KST) & 1); };
            auto k_free = [&](int j) {                // after the tile's last S MMA
                if (lane == 0) umma_commit(bar(kKEmpty + (t0 + j) % KST));
                __syncwarp();
            };
            auto next_s = [&](int j, int buf) {       // S of tile j for tile a, then free the K tile
                ok = k_ready(j);
                if (!ok) return;
                issue_s(0, buf, j);
                k_free(j);
            };
            // (each Q tile's scores start once its query rows are in place)
            ok = warp_wait(bar(kQFull), ic & 1);
            if (!ok) break;
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
                if (ok) issue_s(0, 0, 0);
                if (ok) ok = warp_wait(bar(kQFull + 1), ic & 1);
                if (ok) {
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
            t0 += ntiles;
        }
        if (!ok && lane == 0) raise_flag(p.err, PA_DEV_ERR_TIMEOUT);
        // nothing may still be running on the tensor cores when TMEM is freed
        if (lane == 0) umma_commit(bar(kDone));
        __syncwarp();
        mbar_wait_bounded(bar(kDone), 0, kWaitLimitNs);
    }
    }
    } else {
    // ---------------------------------------------------------------- softmax warps
    // rows: (chunk token, query head of this kv head), token-major; one per softmax thread
    const int row = threadIdx.x;                          // 0 .. 255 for the softmax warps
    const int h = warp >> 2;                              // Q tile of a softmax warp
    const int lr = row & (kHalfRows - 1);
    const uint32_t qdst = sQ + h * L::QTILE + (uint32_t)((lr >> 3) * 128 + (lr & 7) * 16);
    // a negative scale is applied as |scale| to -q (exact), so that the softmax can take the
    // row maximum of the unscaled scores
    const uint32_t flip = p.scale_log2 < 0.f ? 0x80008000u : 0u;
    constexpr int QB = D / 8;                            // 16-byte pieces of a query row
    struct RowOf { int pos; bool valid; size_t orow; };
    auto row_of = [&](const Item& g) {
        RowOf r{g.p_last, false, 0};                      // rows outside the chunk see all (finite)
        if constexpr (PREFIX) {
            const int rr = g.row_base + row, sq = rr / p.G, gq = rr - sq * p.G;
            r.valid = row < p.rows_per_cta && rr < p.num_seqs * p.G;
            if (r.valid) r.orow = (size_t)sq * p.Hq + (size_t)g.kvh * p.G + gq;   // partial row
        } else {
            const int tl = row / p.G, gq = row - tl * p.G;
            r.valid = tl < g.rows;                        // (rows <= TQ)
            if (r.valid) {
                r.pos = g.p0 + tl;
                r.orow = ((size_t)(g.qrow0 + tl) * p.Hq + (size_t)g.kvh * p.G + gq) * D;
            }
        }
        return r;
    };
    // The row's query goes straight into its place in the Q tile by 16-byte async copies
    // (zeros for rows outside the chunk); publish_q waits for them, applies a negative
    // scale's sign and makes the tile visible to the tensor cores.
    auto load_q = [&](const RowOf& r) {
        if (r.valid) {
            const uint16_t* qsrc = static_cast<const uint16_t*>(p.q) + (PREFIX ? r.orow * D : r.orow);
#pragma unroll
            for (int u = 0; u < QB; ++u) cp_async_16(qdst + u * 2048, qsrc + 8 * u);
        } else {
#pragma unroll
            for (int u = 0; u < QB; ++u) st_shared_v4(qdst + u * 2048, make_uint4(0u, 0u, 0u, 0u));
        }
        cp_async_commit();
    };
    auto publish_q = [&]() {
        cp_async_wait<0>();
        __syncwarp();                                     // (the row came from the warp's lanes)
        if (flip) {
#pragma unroll 1
            for (int u = 0; u < QB; ++u) {
                uint4 v = ld_shared_v4(qdst + u * 2048);
                v.x ^= flip;
                v.y ^= flip;
                v.z ^= flip;
                v.w ^= flip;
                st_shared_v4(qdst + u * 2048, v);
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kQFull + h));
    };
    // Through an item's tiles a thread keeps only its row's position (its output row is
    // derived again for the epilogue: the registers go to the row of S).
    int it = item_of(0, -1);
    int ntiles = 0, pos = 0;
    if (!PREFIX) grid_dependency_wait();                 // the queries may come from a kernel before
    if (it >= 0) {
        const Item g = item_get(it);
        ntiles = (g.nblk + kKeyBlocks - 1) / kKeyBlocks;
        const RowOf r = row_of(g);
        pos = r.pos;
        load_q(r);
    }
    tc_fence_before();
    named_bar_sync(2, 32 * (kSoftWarps + 1));
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::SLOT);
    if (*reinterpret_cast<volatile uint32_t*>(smem + L::SLOT + 4) == 0u) {   // (else write nothing)
    // (every warp of both softmax warpgroups, at this one instruction)
    asm volatile("setmaxnreg.inc.sync.aligned.u32 200;" ::: "memory");
    // Warp w reaches TMEM lanes 32 (w % 4) ..; this thread's row of tile h is lane row % 128.
    // With two tiles a commit after S_h(j) covers every earlier MMA, so when S_h(j) is seen
    // complete, PV_h(j - 1) is too: O_h may be rescaled and P_h(j) written at once.
    const uint32_t tl_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    // without a tile b, tile a's S alternates between both S buffers (see the MMA warp)
    const uint32_t ocol = kColO + (uint32_t)(h * kKeyTok);
    const float cs = fabsf(p.scale_log2);              // a negative scale was moved into Q
    const bool active = h == 0 || has_b;
    bool ok = true;
    int t0 = 0, ic = 0;                                // tiles and items of the earlier items
    if (it >= 0) publish_q();
    while (ok && it >= 0) {
        float m_used = -INFINITY, l = 0.f;
        for (int j = 0; active && j < ntiles; ++j) {
            const int t = t0 + j;
            const int sb = has_b ? h : (j & 1);
            const uint32_t scol = kColS + (uint32_t)(sb * kKeyTok);
            ok = warp_wait(bar(kSFull + sb), has_b ? (t & 1) : ((j >> 1) & 1));
            if (!ok) break;
            if (!PREFIX && j == ntiles - 1 && nlist >= 0) {
                // S_h of the item's last tile is complete, so Q_h is free: the next item's query
                // rows start loading now, under this tile's softmax and the output's epilogue
                const int nx = item_of(ic + 1, it);
                if (nx >= 0) load_q(row_of(item_get(nx)));
            }
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
            // probabilities, bf16 pairs, over the first 64 columns of S_h (already read), 16
            // columns per store (32 scores: the fewest registers held beside the row); a full
            // tile takes s c - m for two keys in one packed FFMA and sums in pairs
            float sum;
            if (full) {
                const uint64_t c2 = pack_f32x2(cs, cs), nm2 = pack_f32x2(-m_used, -m_used);
                uint64_t sum2[2] = {pack_f32x2(0.f, 0.f), pack_f32x2(0.f, 0.f)};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const uint64_t x2 = ffma_f32x2(pack_f32x2(__uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1])), c2, nm2);
                        const float e0 = fast_exp2(lo_f32(x2)), e1 = fast_exp2(hi_f32(x2));
                        sum2[(i >> 1) & 1] = fadd_f32x2(sum2[(i >> 1) & 1], pack_f32x2(e0, e1));
                        pk[i >> 1] = pack_bf16x2(e0, e1);
                    }
                    tmem_st16(tl_addr + scol + 16 * c, pk);
                }
                const uint64_t tsum = fadd_f32x2(sum2[0], sum2[1]);
                sum = lo_f32(tsum) + hi_f32(tsum);
            } else {
                sum = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float e0 = fast_exp2(__uint_as_float(sr[c][i]) - m_used);
                        const float e1 = fast_exp2(__uint_as_float(sr[c][i + 1]) - m_used);
                        sum += e0 + e1;
                        pk[i >> 1] = pack_bf16x2(e0, e1);
                    }
                    tmem_st16(tl_addr + scol + 16 * c, pk);
                }
            }
            l = l * alpha + sum;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kPFull + (has_b ? h : (j & 1))));
        }
        if (!ok) break;
        // the next item's query rows (published once this item's output is read)
        const int it_next = item_of(ic + 1, it);
        int ntiles_next = 0, pos_next = 0;
        if (it_next >= 0) {
            const Item gn = item_get(it_next);
            ntiles_next = (gn.nblk + kKeyBlocks - 1) / kKeyBlocks;
            const RowOf rn = row_of(gn);
            pos_next = rn.pos;
            if (PREFIX || nlist < 0) load_q(rn);          // (else under way since the last tile)
        }
        const RowOf rw = row_of(item_get(it));
        if (active) {
            ok = warp_wait(bar(kODone + h), ic & 1);
            if (ok && PREFIX) {
                tc_fence_after();
                // Each 32-column piece of the warp's 32 rows passes through shared memory (the K
                // stages: every MMA has completed), 16-byte units of row r at unit u ^ (r % 8),
                // so that both the writes and the reads are free of bank conflicts and each
                // global store covers 128 contiguous bytes of four rows (a thread storing its
                // own row scatters 16-byte pieces over 32 rows per instruction).
                const size_t slot = rw.orow * p.part_stride + (size_t)blockIdx.z * p.slot_mult;
                const uint32_t stg = sK + (uint32_t)warp * (32 * 128);
                const uint32_t valid = __ballot_sync(0xffffffffu, rw.valid);
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
                if (rw.valid) p.part_ml[slot] = make_float2(m_used, l);
            } else if (ok) {
                tc_fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                uint16_t* dst = static_cast<uint16_t*>(p.out) + rw.orow;
                // 32-byte stores where the output allows them: the warp's 32 rows lie apart, so
                // a store instruction touches a sector per lane, and wider stores need half as many
                const bool wide = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0u;
                // 32 columns at a time (the next item's first scores may be in flight)
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tl_addr + ocol + 32 * c, o);
                    tmem_wait_ld();
                    if (rw.valid) {
                        uint32_t w[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
                        uint16_t* d = dst + 32 * c;
                        if (wide) {
                            st_global_v8(d, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
                            st_global_v8(d + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
                        } else {
#pragma unroll
                            for (int v = 0; v < 4; ++v)
                                reinterpret_cast<uint4*>(d)[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
                        }
                    }
                }
                // O is read: the next item's P V may start afresh
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kOFree));
            }
        } else if (lane == 0) {
            mbar_arrive(bar(kOFree));                     // (a tile b without rows)
        }
        if (ok && it_next >= 0) publish_q();
        if (!ok) break;
        if (PREFIX) break;                                // one item per CTA
        t0 += ntiles;
        ++ic;
        it = it_next;
        ntiles = ntiles_next;
        pos = pos_next;
    }
    if (!ok) {
        // a wait gave up: the rows of this item and of the CTA's later items are incomplete,
        // so they are written as NaN (visible even when no error flag was given)
        if (lane == 0) raise_flag(p.err, PA_DEV_ERR_TIMEOUT);
        for (; it >= 0; it = item_of(++ic, it)) {
            const RowOf rw = row_of(item_get(it));
            if (rw.valid && active) {
                if constexpr (PREFIX) {
                    p.part_ml[rw.orow * p.part_stride + (size_t)blockIdx.z * p.slot_mult] =
                        make_float2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + rw.orow);
                    for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
                }
            }
        }
    }
    }
    // (no query copy may still be landing when the CTA ends)
    cp_async_wait<0>();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc<kTmemCols>(*reinterpret_cast<volatile uint32_t*>(smem + L::SLOT));
    }
    // every thread waits for the previous grid before exiting: a dependent grid never
    // completes before the one it follows (a no-op where it already waited)
    grid_dependency_wait();
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
    pp.num_seqs = a.num_seqs;
    pp.nqt = (a.max_chunk + pp.TQ - 1) / pp.TQ;
    const long long items = (long long)pp.nqt * pp.Hkv * a.num_seqs;
    if (items <= 0) return cudaSuccess;
    if (items > INT32_MAX) return cudaErrorInvalidValue;
    pp.num_items = (int)items;
    // persistent: one CTA per SM at most (a CTA fills an SM's shared memory and TMEM)
    const dim3 grid((unsigned)std::min<long long>(items, sm_count()));
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

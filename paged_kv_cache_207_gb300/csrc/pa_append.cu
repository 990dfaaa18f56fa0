// pa_append.cu -- writing new tokens into the paged pools, and copy-on-write
// block copies.
//
// Append (spindle, "Two bugs worth recording": append takes an explicit start
// position): row i of sequence s goes to position start_pos[s] + i, i.e. slot
// (pos % 16) of block block_tables[s][pos / 16].  One thread moves one 16-byte
// piece of one (row, kv head) of K and of V.  A warp takes 16 consecutive rows and
// two adjacent pieces of one kv head (lane % 16 the row, lane / 16 the piece): it
// reads whole 32-byte sectors of the rows, and where the rows fill consecutive slots
// of a block (a chunk of a prefill) each store instruction writes two 256-byte runs
// of the tile (a piece's 16 slots are contiguous in the pool).
//
// Copy (spindle, "Paging": refcounted copy-on-write forking): every byte of
// block src goes to block dst in both pools; 16-byte vector loads and stores.
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

namespace {

__device__ __forceinline__ void raise_flag(int32_t* err, int bits) {
    if (err) atomicOr(err, bits);
}

struct AParams {
    char* k_pool;
    char* v_pool;
    const char* k_new;
    const char* v_new;
    const int32_t* tables;
    const int32_t* start_pos;
    const int32_t* cu;
    int32_t* err;
    int max_blocks, S, total, num_blocks, Hkv, chunks;   // chunks = 16-byte pieces per row and head
    long long items;                                      // (FP8 / FP4) total * Hkv warps; (plain)
                                                          // groups of 16 rows x Hkv x piece pairs x 32
};

// Sequence, position and physical block of new row `row` (reads only cu, start_pos
// and the tables, which no kernel of this library writes).  Flags and returns false
// when the row has no valid destination; `report` selects the thread that flags.
__device__ __forceinline__ bool locate_row(const AParams& p, int row, bool report, int& s_out,
                                           int& slot_out, int32_t& blk_out) {
    // sequence owning this row: cu[s] <= row < cu[s+1].  Guess by proportion (exact
    // when every sequence appends the same number of rows, e.g. one per decode step),
    // then fall back to a binary search.
    int s = (int)(((long long)row * p.S) / (p.total > 0 ? p.total : 1));
    if (s >= p.S) s = p.S - 1;
    int first = __ldg(p.cu + s);
    int next = __ldg(p.cu + s + 1);
    if (!(first <= row && row < next)) {
        int lo = 0, hi = p.S - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(p.cu + mid) <= row) lo = mid;
            else hi = mid - 1;
        }
        s = lo;
        first = __ldg(p.cu + s);
        next = __ldg(p.cu + s + 1);
        if (row < first || row >= next) {
            if (report) raise_flag(p.err, PA_DEV_ERR_BAD_CU);
            return false;
        }
    }
    const long long pos = (long long)__ldg(p.start_pos + s) + (row - first);
    if (pos < 0 || pos >= (long long)p.max_blocks * kBlockTokens) {
        if (report) raise_flag(p.err, PA_DEV_ERR_BAD_POS);
        return false;
    }
    const int32_t blk = __ldg(p.tables + (size_t)s * p.max_blocks + (int)(pos / kBlockTokens));
    if (blk < 0 || blk >= p.num_blocks) {
        if (report) raise_flag(p.err, PA_DEV_ERR_BAD_BLOCK);
        return false;
    }
    s_out = s;
    slot_out = (int)(pos % kBlockTokens);
    blk_out = blk;
    return true;
}

__global__ void __launch_bounds__(256) append_kernel(const AParams p) {
    // a decode launched after this kernel may start its set-up now; it waits for this
    // grid to finish before reading the pools
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long item = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (item == 0) {
        if (__ldg(p.cu) != 0 || __ldg(p.cu + p.S) != p.total) raise_flag(p.err, PA_DEV_ERR_BAD_CU);
    }
    const int pairs = (p.chunks + 1) >> 1;
    const long long wi = item >> 5;                       // the warp's (row group, head, pair)
    const int pr = (int)(wi % pairs);
    const long long gh = wi / pairs;
    const int h = (int)(gh % p.Hkv);
    const int row = (int)(gh / p.Hkv) * 16 + (int)(item & 15);
    const int ch = 2 * pr + (int)((item >> 4) & 1);
    int s, slot;
    int32_t blk;
    // (the two lanes of a row both look it up; the piece-0 lane reports a failure)
    const bool ok = item < p.items && row < p.total && ch < p.chunks &&
                    locate_row(p, row, ch == 0, s, slot, blk);

    // The address chain above read only inputs.  The pools (and, in principle, the new
    // rows) may still be in use by the previous kernel of the stream: wait for it.  Every
    // thread waits before it exits, so this grid never completes before that kernel.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!ok) return;
    const size_t src = (((size_t)row * p.Hkv + h) * p.chunks + ch) * 16;
    const uint4 kv = __ldg(reinterpret_cast<const uint4*>(p.k_new + src));
    const uint4 vv = __ldg(reinterpret_cast<const uint4*>(p.v_new + src));
    // pool byte offset: tile (blk, h), chunk ch, slot  -> 16 bytes
    const size_t dst = ((((size_t)blk * p.Hkv + h) * p.chunks + ch) * kBlockTokens + slot) * 16;
    *reinterpret_cast<uint4*>(p.k_pool + dst) = kv;
    *reinterpret_cast<uint4*>(p.v_pool + dst) = vv;
}

// FP8 append: one warp per (row, kv head).  The row's D bf16 values get one
// scale amax / 448 and E4M3 codes x / scale (fp32, each step correctly rounded,
// then round to nearest even with saturation); K codes go to the slot's 16-byte
// pieces of the record, V codes to byte `slot` of each dim's 16-byte row, and
// the two scales after the codes.
template <int D>
__global__ void __launch_bounds__(256) append_fp8_kernel(const AParams p) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (__ldg(p.cu) != 0 || __ldg(p.cu + p.S) != p.total) raise_flag(p.err, PA_DEV_ERR_BAD_CU);
    }
    const int h = (int)(wid % p.Hkv);
    const int row = (int)(wid / p.Hkv);
    int s, slot;
    int32_t blk;
    const bool ok = wid < (long long)p.total * p.Hkv && locate_row(p, row, lane == 0, s, slot, blk);
    asm volatile("griddepcontrol.wait;" ::: "memory");           // as in append_kernel
    if (!ok) return;                                              // warp-uniform
    const size_t src = ((size_t)row * p.Hkv + h) * D * 2;          // bytes of bf16 rows
    uint32_t kw, vw;
    float ks, vs;
    fp8_quantize_rows<D>(p.k_new + src, p.v_new + src, lane, kw, vw, ks, vs);
    const size_t rec = fp8_record_bytes(D);
    fp8_put_row<D>(p.k_pool + ((size_t)blk * p.Hkv + h) * rec, p.v_pool + ((size_t)blk * p.Hkv + h) * rec,
                   lane, slot, kw, vw, ks, vs);
}

// MXFP4 append: one warp per (row, kv head), D / 32 values per lane.  Each block of
// 32 values (8 or 16 lanes) gets the E8M0 scale 2^(floor(log2 amax) - 2) -- the
// biased exponent of amax minus 2, at least 0; an all-zero block gets code 0 --
// and E2M1 codes of x / scale (exact power-of-two scaling in fp32, then round to
// nearest even, saturating at 6).  K: the slot's row holds the codes in pairs of
// dims, the byte of dims (16 ks + 8 half + 2c, +1) at c (D / 8) + 2 ks + half.
// V: a byte holds two slots of one dim; the byte of (dim 16 mi + 8 dh + r, slots
// 2c + 8 half, +1) is at ((4 r + c) (D / 16) + mi) 4 + 2 dh + half, low nibble the
// even slot.  Rows appended by the same call may share these V bytes, so each
// nibble is cleared and set with atomics on its 32-bit word.  Scales: byte
// 8 D + slot (D / 32) + b of the record.
template <int D>
__global__ void __launch_bounds__(256) append_fp4_kernel(const AParams p) {
    constexpr int VPL = D / 32;          // values per lane: 4 (D = 128) or 2 (D = 64)
    constexpr int LPB = 32 / VPL;        // lanes per 32-value block
    constexpr int NB = D / 32;
    constexpr int REC = 8 * D + D / 2;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (__ldg(p.cu) != 0 || __ldg(p.cu + p.S) != p.total) raise_flag(p.err, PA_DEV_ERR_BAD_CU);
    }
    const int h = (int)(wid % p.Hkv);
    const int row = (int)(wid / p.Hkv);
    int s, slot;
    int32_t blk;
    const bool ok = wid < (long long)p.total * p.Hkv && locate_row(p, row, lane == 0, s, slot, blk);
    asm volatile("griddepcontrol.wait;" ::: "memory");           // as in append_kernel
    if (!ok) return;                                              // warp-uniform

    const size_t src = ((size_t)row * p.Hkv + h) * D + (size_t)lane * VPL;
    float kx[VPL], vx[VPL];
    if constexpr (VPL == 4) {
        const uint2 kr = __ldg(reinterpret_cast<const uint2*>(p.k_new) + src / 4);
        const uint2 vr = __ldg(reinterpret_cast<const uint2*>(p.v_new) + src / 4);
        kx[0] = __uint_as_float(kr.x << 16); kx[1] = __uint_as_float(kr.x & 0xffff0000u);
        kx[2] = __uint_as_float(kr.y << 16); kx[3] = __uint_as_float(kr.y & 0xffff0000u);
        vx[0] = __uint_as_float(vr.x << 16); vx[1] = __uint_as_float(vr.x & 0xffff0000u);
        vx[2] = __uint_as_float(vr.y << 16); vx[3] = __uint_as_float(vr.y & 0xffff0000u);
    } else {
        const uint32_t kr = __ldg(reinterpret_cast<const uint32_t*>(p.k_new) + src / 2);
        const uint32_t vr = __ldg(reinterpret_cast<const uint32_t*>(p.v_new) + src / 2);
        kx[0] = __uint_as_float(kr << 16); kx[1] = __uint_as_float(kr & 0xffff0000u);
        vx[0] = __uint_as_float(vr << 16); vx[1] = __uint_as_float(vr & 0xffff0000u);
    }
    float ka = 0.f, va = 0.f;
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
        ka = fmaxf(ka, fabsf(kx[k]));
        va = fmaxf(va, fabsf(vx[k]));
    }
#pragma unroll
    for (int x = 1; x < LPB; x <<= 1) {            // within the lane's 32-value block
        ka = fmaxf(ka, __shfl_xor_sync(0xffffffffu, ka, x));
        va = fmaxf(va, __shfl_xor_sync(0xffffffffu, va, x));
    }
    const int kcode = ka > 0.f ? max((int)(__float_as_uint(ka) >> 23) - 2, 0) : 0;
    const int vcode = va > 0.f ? max((int)(__float_as_uint(va) >> 23) - 2, 0) : 0;
    const float kinv = exp2i(127 - kcode), vinv = exp2i(127 - vcode);   // 1 / scale, exact

    char* krec = p.k_pool + ((size_t)blk * p.Hkv + h) * REC;
    char* vrec = p.v_pool + ((size_t)blk * p.Hkv + h) * REC;
    const int d0 = lane * VPL;
    // K: pairs of dims, one byte each
#pragma unroll
    for (int k = 0; k < VPL; k += 2) {
        const int d = d0 + k;
        const uint32_t byte = ka > 0.f ? pack_e2m1x2(kx[k] * kinv, kx[k + 1] * kinv) : 0u;
        const int ks = d / 16, half = (d % 16) / 8, c = (d % 8) / 2;
        krec[(size_t)slot * (D / 2) + c * (D / 8) + ks * 2 + half] = (char)byte;
    }
    // V: one nibble per dim, in words shared with other slots
    const int half = slot / 8, c = (slot % 8) / 2, nib = slot & 1;
#pragma unroll
    for (int k = 0; k < VPL; k += 2) {
        const uint32_t pair = va > 0.f ? pack_e2m1x2(vx[k] * vinv, vx[k + 1] * vinv) : 0u;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int d = d0 + k + e;
            const uint32_t code = (pair >> (4 * e)) & 0xfu;
            const int mi = d / 16, dh = (d % 16) / 8, rr = d % 8;
            const int idx = ((rr * 4 + c) * (D / 16) + mi) * 4 + dh * 2 + half;
            unsigned int* word = reinterpret_cast<unsigned int*>(vrec + (idx & ~3));
            const int shift = (idx & 3) * 8 + nib * 4;
            atomicAnd(word, ~(0xfu << shift));
            atomicOr(word, code << shift);
        }
    }
    // scales: the first lane of each 32-value block
    if (lane % LPB == 0) {
        const int b = lane / LPB;
        krec[8 * D + slot * NB + b] = (char)kcode;
        vrec[8 * D + slot * NB + b] = (char)vcode;
    }
}

struct CParams {
    char* k_pool;
    char* v_pool;
    const int32_t* pairs;
    int32_t* err;
    int num_blocks;
    size_t block_bytes;   // bytes of one block in one pool (all kv heads)
};

// grid = (pair, pool half: 0 = K, 1 = V, slice)
__global__ void __launch_bounds__(256) copy_kernel(const CParams p) {
    const int pair = blockIdx.x;
    const int32_t src = __ldg(p.pairs + 2 * pair), dst = __ldg(p.pairs + 2 * pair + 1);
    if (src < 0 || src >= p.num_blocks || dst < 0 || dst >= p.num_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) raise_flag(p.err, PA_DEV_ERR_BAD_PAIR);
        return;
    }
    if (src == dst) return;
    char* pool = blockIdx.y == 0 ? p.k_pool : p.v_pool;
    const uint4* from = reinterpret_cast<const uint4*>(pool + (size_t)src * p.block_bytes);
    uint4* to = reinterpret_cast<uint4*>(pool + (size_t)dst * p.block_bytes);
    const size_t n16 = p.block_bytes / 16;
    for (size_t i = (size_t)blockIdx.z * blockDim.x + threadIdx.x; i < n16;
         i += (size_t)gridDim.z * blockDim.x)
        to[i] = from[i];
}

// Launch as a programmatic dependent of the previous kernel of the stream: the append
// may start while that kernel finishes, computes its destinations, and waits for it
// (griddepcontrol.wait) before it reads the new rows or writes the pools.
template <typename K>
cudaError_t launch_dependent(K kernel, dim3 grid, cudaStream_t stream, const AParams& p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream) {
    AParams p;
    p.k_pool = static_cast<char*>(a.k_pool);
    p.v_pool = static_cast<char*>(a.v_pool);
    p.k_new = static_cast<const char*>(a.k_new);
    p.v_new = static_cast<const char*>(a.v_new);
    p.tables = a.block_tables;
    p.start_pos = a.start_pos;
    p.cu = a.cu_new;
    p.err = a.err;
    p.max_blocks = a.max_blocks;
    p.S = a.num_seqs;
    p.total = a.total_new;
    p.num_blocks = a.num_blocks;
    p.Hkv = a.num_kv_heads;
    p.chunks = a.head_dim * elem_bytes(a.dtype) / 16;
    p.items = (long long)((a.total_new + 15) / 16) * a.num_kv_heads * ((p.chunks + 1) / 2) * 32;
    if (a.total_new == 0 || p.chunks == 0) return cudaSuccess;
    const long long blocks = (p.items + 255) / 256;
    return launch_dependent(append_kernel, dim3((unsigned)blocks), stream, p);
}

cudaError_t launch_append_fp8(const AppendArgs& a, cudaStream_t stream) {
    AParams p;
    p.k_pool = static_cast<char*>(a.k_pool);
    p.v_pool = static_cast<char*>(a.v_pool);
    p.k_new = static_cast<const char*>(a.k_new);
    p.v_new = static_cast<const char*>(a.v_new);
    p.tables = a.block_tables;
    p.start_pos = a.start_pos;
    p.cu = a.cu_new;
    p.err = a.err;
    p.max_blocks = a.max_blocks;
    p.S = a.num_seqs;
    p.total = a.total_new;
    p.num_blocks = a.num_blocks;
    p.Hkv = a.num_kv_heads;
    p.chunks = 0;
    p.items = (long long)a.total_new * a.num_kv_heads;   // warps
    if (p.items == 0) return cudaSuccess;
    const long long blocks = (p.items * 32 + 255) / 256;
    return a.head_dim == 64 ? launch_dependent(append_fp8_kernel<64>, dim3((unsigned)blocks), stream, p)
                            : launch_dependent(append_fp8_kernel<128>, dim3((unsigned)blocks), stream, p);
}

cudaError_t launch_copy(const CopyArgs& a, cudaStream_t stream) {
    if (a.num_pairs == 0) return cudaSuccess;
    CParams p;
    p.k_pool = static_cast<char*>(a.k_pool);
    p.v_pool = static_cast<char*>(a.v_pool);
    p.pairs = a.pairs;
    p.err = a.err;
    p.num_blocks = a.num_blocks;
    p.block_bytes = a.dtype == PA_FP8_E4M3 ? (size_t)a.num_kv_heads * fp8_record_bytes(a.head_dim)
                  : a.dtype == PA_FP4_E2M1 ? (size_t)a.num_kv_heads * fp4_record_bytes(a.head_dim)
                  : (size_t)a.num_kv_heads * kBlockTokens * a.head_dim * elem_bytes(a.dtype);
    const size_t n16 = p.block_bytes / 16;
    const unsigned slices = (unsigned)((n16 + 256 * 4 - 1) / (256 * 4));   // ~4 vectors per thread
    const dim3 grid(a.num_pairs, 2, slices > 0 ? (slices < 64 ? slices : 64) : 1);
    copy_kernel<<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_append_fp4(const AppendArgs& a, cudaStream_t stream) {
    AParams p;
    p.k_pool = static_cast<char*>(a.k_pool);
    p.v_pool = static_cast<char*>(a.v_pool);
    p.k_new = static_cast<const char*>(a.k_new);
    p.v_new = static_cast<const char*>(a.v_new);
    p.tables = a.block_tables;
    p.start_pos = a.start_pos;
    p.cu = a.cu_new;
    p.err = a.err;
    p.max_blocks = a.max_blocks;
    p.S = a.num_seqs;
    p.total = a.total_new;
    p.num_blocks = a.num_blocks;
    p.Hkv = a.num_kv_heads;
    p.chunks = 0;
    p.items = (long long)a.total_new * a.num_kv_heads;   // warps
    if (p.items == 0) return cudaSuccess;
    const long long blocks = (p.items * 32 + 255) / 256;
    return a.head_dim == 64 ? launch_dependent(append_fp4_kernel<64>, dim3((unsigned)blocks), stream, p)
                            : launch_dependent(append_fp4_kernel<128>, dim3((unsigned)blocks), stream, p);
}

}  // namespace pa

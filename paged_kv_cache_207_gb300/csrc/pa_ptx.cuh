// pa_ptx.cuh -- thin inline-PTX wrappers used by the kernels (sm_103a).
//
// Bulk asynchronous copies (the TMA engine's 1-D mode) with mbarrier
// completion, shared-memory matrix loads, the legacy warp-level bf16 MMA and
// small conversions.  Every wait is bounded: a wait that runs past its time
// limit returns false and the caller records PA_DEV_ERR_TIMEOUT.
#pragma once

#include <cstdint>

#include "pa_internal.h"

namespace pa {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier --------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation (and earlier generic-proxy shared-memory
// accesses) visible to the async proxy before bulk copies use the memory.
// 16-byte store to shared memory (a generic-proxy write).
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                 :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Plain arrival (counts one of the barrier's expected arrivals).
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of the barrier, giving up after `limit_ns`
// nanoseconds of wall time.  Returns true when the phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0u && global_timer_ns() - t0 > limit_ns) return false;
    }
}

// ---- bulk copy global -> shared (TMA 1-D), completion on an mbarrier --------

// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst_smem),
        "l"(src_gmem), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// L2 policy: data read once (K/V tiles) is evicted first.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---- warp-level matrix ops ---------------------------------------------------

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

// 8x8 b16 transpose across the warp: thread i's pair (row i/4, cols 2(i%4)..+1)
// becomes the pair of the transposed matrix.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---- programmatic dependent launch ---------------------------------------------

// Wait until the grid this kernel depends on (the previous kernel in the stream)
// has completed and its memory is visible.  A no-op for ordinary launches.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Allow the next kernel in the stream, if launched as a dependent, to start its
// own set-up now (it still waits for this grid before touching its results).
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- conversions -------------------------------------------------------------

// Pack two fp32 into bf16x2 (round to nearest even): `lo` in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16_lo_to_f32(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi_to_f32(uint32_t x) {
    return __uint_as_float(x & 0xffff0000u);
}

// Two fp32 -> two E4M3 codes (round to nearest even, saturating): `lo` in bits 0..7.
__device__ __forceinline__ uint16_t pack_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// E4M3 quantisation of one (token, kv head) K row and V row (bf16, D values each) by one
// warp, as the FP8 cache stores them: lane l holds dims l*VPL .. l*VPL + VPL - 1 (VPL = D/32);
// each row's scale is amax / 448 and each code x / scale (fp32, each step correctly rounded,
// then E4M3 round to nearest even, saturating).  The lane's VPL K and V codes come back packed
// (dim l*VPL in bits 0..7).  The rows may come from the previous kernel: plain loads.
template <int D>
__device__ __forceinline__ void fp8_quantize_rows(const char* k_row, const char* v_row, int lane,
                                                  uint32_t& kc, uint32_t& vc, float& ks, float& vs) {
    constexpr int VPL = D / 32;
    float kx[VPL], vx[VPL];
    if constexpr (VPL == 4) {
        const uint2 kr = *reinterpret_cast<const uint2*>(k_row + (size_t)lane * 8);
        const uint2 vr = *reinterpret_cast<const uint2*>(v_row + (size_t)lane * 8);
        kx[0] = bf16_lo_to_f32(kr.x); kx[1] = bf16_hi_to_f32(kr.x);
        kx[2] = bf16_lo_to_f32(kr.y); kx[3] = bf16_hi_to_f32(kr.y);
        vx[0] = bf16_lo_to_f32(vr.x); vx[1] = bf16_hi_to_f32(vr.x);
        vx[2] = bf16_lo_to_f32(vr.y); vx[3] = bf16_hi_to_f32(vr.y);
    } else {
        const uint32_t kr = *reinterpret_cast<const uint32_t*>(k_row + (size_t)lane * 4);
        const uint32_t vr = *reinterpret_cast<const uint32_t*>(v_row + (size_t)lane * 4);
        kx[0] = bf16_lo_to_f32(kr); kx[1] = bf16_hi_to_f32(kr);
        vx[0] = bf16_lo_to_f32(vr); vx[1] = bf16_hi_to_f32(vr);
    }
    float ka = 0.f, va = 0.f;
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
        ka = fmaxf(ka, fabsf(kx[k]));
        va = fmaxf(va, fabsf(vx[k]));
    }
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) {
        ka = fmaxf(ka, __shfl_xor_sync(0xffffffffu, ka, x));
        va = fmaxf(va, __shfl_xor_sync(0xffffffffu, va, x));
    }
    ks = __fdiv_rn(ka, 448.f);
    vs = __fdiv_rn(va, 448.f);
    kc = 0u;
    vc = 0u;
#pragma unroll
    for (int k = 0; k < VPL; k += 2) {
        const uint32_t k2 = ks > 0.f ? pack_e4m3x2(__fdiv_rn(kx[k], ks), __fdiv_rn(kx[k + 1], ks)) : 0u;
        const uint32_t v2 = vs > 0.f ? pack_e4m3x2(__fdiv_rn(vx[k], vs), __fdiv_rn(vx[k + 1], vs)) : 0u;
        kc |= k2 << (8 * k);
        vc |= v2 << (8 * k);
    }
}

// One quantised row into an FP8 (block, kv head) record pair (krec, vrec: pool records in
// global memory, or a stage's copies of them in shared memory): K codes in the slot's
// 16-byte piece of each 16 dims, V codes at byte `slot` of each dim's 16-byte row, the two
// scales after the codes (lane 0).  kc, vc, ks, vs as fp8_quantize_rows gives them.
template <int D>
__device__ __forceinline__ void fp8_put_row(char* krec, char* vrec, int lane, int slot,
                                            uint32_t kc, uint32_t vc, float ks, float vs) {
    constexpr int VPL = D / 32;
    const int d0 = lane * VPL;                 // dims d0 .. d0 + VPL - 1 lie in one 16-dim piece
    char* kdst = krec + ((size_t)(d0 / 16) * kBlockTokens + slot) * 16 + (d0 % 16);
    if constexpr (VPL == 4)
        *reinterpret_cast<uint32_t*>(kdst) = kc;
    else
        *reinterpret_cast<uint16_t*>(kdst) = (uint16_t)kc;
#pragma unroll
    for (int k = 0; k < VPL; ++k) vrec[(size_t)(d0 + k) * kBlockTokens + slot] = (char)(vc >> (8 * k));
    if (lane == 0) {
        *reinterpret_cast<float*>(krec + (size_t)16 * D + 4 * slot) = ks;
        *reinterpret_cast<float*>(vrec + (size_t)16 * D + 4 * slot) = vs;
    }
}

// Two E4M3 codes (bits 0..7 and 8..15) -> f16x2 (exact: every E4M3 value is an f16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t x) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(x));
    return r;
}

// Pack two fp32 into f16x2 (round to nearest even): `lo` in bits 0..15.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col)
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The four bytes of a word, each a pair of E2M1 codes (low nibble first), as four
// f16x2 (exact: every E2M1 value is an f16 value); o[i] comes from byte i.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&o)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w));
}

// The same through E4M3: an E2M1 code (s, e1 e0, m) is, bit for bit, the E4M3 code
// (s, 0 0 e1 e0, m 0 0) of the value times 2^-6 (E2M1's subnormal 0.5 lands on an E4M3
// subnormal), and E4M3 -> f16 is exact.  o[i] from byte i as above, times 2^-6.
__device__ __forceinline__ void e2m1x8_to_f16x2x4_scaled(uint32_t w, uint32_t (&o)[4]) {
    const uint32_t lo = ((w << 2) & 0x1C1C1C1Cu) | ((w << 4) & 0x80808080u);   // low nibbles
    const uint32_t hi = ((w >> 2) & 0x1C1C1C1Cu) | (w & 0x80808080u);          // high nibbles
    const uint32_t p01 = __byte_perm(lo, hi, 0x5140), p23 = __byte_perm(lo, hi, 0x7362);
    o[0] = e4m3x2_to_f16x2((uint16_t)(p01 & 0xffffu));
    o[1] = e4m3x2_to_f16x2((uint16_t)(p01 >> 16));
    o[2] = e4m3x2_to_f16x2((uint16_t)(p23 & 0xffffu));
    o[3] = e4m3x2_to_f16x2((uint16_t)(p23 >> 16));
}

// Two fp32 -> two E2M1 codes in one byte (round to nearest even, saturating at 6):
// `lo` in bits 0..3, `hi` in bits 4..7.
__device__ __forceinline__ uint32_t pack_e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\tcvt.u32.u8 %0, b;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// 2^e as an fp32, exactly, for e <= 127 (subnormal results down to 2^-149, 0 below).
__device__ __forceinline__ float exp2i(int e) {
    if (e >= -126) return __uint_as_float((uint32_t)(e + 127) << 23);
    return e >= -149 ? __uint_as_float(1u << (e + 149)) : 0.f;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace pa

// e4m3 two-term forms of the FP8-cache MLA kernel (attn_mla_pair.cu): a
// value x is carried as hi + lo, hi = e4m3(x),
// lo = e4m3(x - hi), and every tensor-core product is issued once per term.
//   * split4: four probabilities -> hi and lo words (the residual is taken in
//     fp16, where p - hi is exact);
//   * qprep_row: one bf16 query row scaled by a power of two (its largest
//     magnitude in (224, 448]) and split into hi / lo, laid out as
//     hi[0:512] lo[0:512] hi[512:576] lo[512:576] (1152 bytes), the scale
//     2^e written to qscale.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "mla_common.cuh"

namespace dcp {
namespace mla_f8 {

constexpr int kQRowBytes = 2 * mla::kDk;  // 1152

// two fp32 -> packed e4m3 pair (first argument in the low byte), saturating
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
// packed f16 pair -> packed e4m3 pair (low half -> low byte), saturating
__device__ __forceinline__ uint32_t e4m3x2_h2(uint32_t h2) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h2));
    return r;
}
// packed e4m3 pair -> packed f16 pair (exact)
__device__ __forceinline__ uint32_t h2_of_e4m3x2(uint32_t e2) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)e2));
    return r;
}
// two fp32 -> packed f16 pair (first argument in the low half)
__device__ __forceinline__ uint32_t h2_of(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Four probabilities -> one 32-bit word of hi and one of lo (token order in
// byte order).  The residual is taken in fp16, where p - hi is exact.
__device__ __forceinline__ void split4(float p0, float p1, float p2, float p3, uint32_t& hi, uint32_t& lo) {
    const uint32_t h01 = e4m3x2(p0, p1), h23 = e4m3x2(p2, p3);
    const uint32_t r01 = hsub2(h2_of(p0, p1), h2_of_e4m3x2(h01));
    const uint32_t r23 = hsub2(h2_of(p2, p3), h2_of_e4m3x2(h23));
    hi = h01 | (h23 << 16);
    lo = e4m3x2_h2(r01) | (e4m3x2_h2(r23) << 16);
}

// ---------------------------------------------------------------------------
// Query preparation: one warp per query row (b, t, head).  The row is scaled
// by 2^-e (e chosen so that its largest magnitude lies in (224, 448]) and
// split into hi and lo; the row's scale 2^e goes to qscale.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void qprep_row(const uint16_t* __restrict__ q, int64_t row, uint8_t* __restrict__ qp,
                                          float* __restrict__ qscale) {
    using mla::kDk;
    const int lane = threadIdx.x & 31;
    const uint4* src = reinterpret_cast<const uint4*>(q + row * kDk);
    // 16-column groups g = lane and lane + 32 (36 groups)
    const bool two = lane + 32 < kDk / 16;
    uint4 v[4];
    v[0] = src[2 * lane];
    v[1] = src[2 * lane + 1];
    v[2] = two ? src[2 * (lane + 32)] : make_uint4(0, 0, 0, 0);
    v[3] = two ? src[2 * (lane + 32) + 1] : make_uint4(0, 0, 0, 0);
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t wv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(wv[k] << 16)), fabsf(__uint_as_float(wv[k] & 0xFFFF0000u))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int e = 0;  // scale 2^e with amax * 2^-e in (224, 448]
    if (amax > 0.f) {
        frexpf(amax / 448.f, &e);
        for (int it = 0; it < 4 && ldexpf(amax, -e) > 448.f; ++it) ++e;
        for (int it = 0; it < 4 && ldexpf(amax, 1 - e) <= 448.f; ++it) --e;
    }
    const float inv = ldexpf(1.f, -e);
    if (lane == 0) qscale[row] = ldexpf(1.f, e);
    uint8_t* dst = qp + row * kQRowBytes;
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
        const int g = lane + 32 * gi;
        if (g >= kDk / 16) break;
        const uint32_t wv[8] = {v[2 * gi].x, v[2 * gi].y, v[2 * gi].z, v[2 * gi].w,
                                v[2 * gi + 1].x, v[2 * gi + 1].y, v[2 * gi + 1].z, v[2 * gi + 1].w};
        uint32_t h[4], l[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t hw = 0, lw = 0;
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const uint32_t w = wv[2 * k + e2];
                const float a = __uint_as_float(w << 16) * inv, b = __uint_as_float(w & 0xFFFF0000u) * inv;
                const uint32_t h2 = e4m3x2(a, b);
                const uint32_t hb = h2_of_e4m3x2(h2);
                const float2 back = __half22float2(*reinterpret_cast<const __half2*>(&hb));
                hw |= h2 << (16 * e2);
                lw |= e4m3x2(a - back.x, b - back.y) << (16 * e2);
            }
            h[k] = hw;
            l[k] = lw;
        }
        const int hi_off = g < 32 ? 16 * g : 1024 + 16 * (g - 32);
        const int lo_off = g < 32 ? 512 + 16 * g : 1088 + 16 * (g - 32);
        *reinterpret_cast<uint4*>(dst + hi_off) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(dst + lo_off) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

}  // namespace mla_f8
}  // namespace dcp

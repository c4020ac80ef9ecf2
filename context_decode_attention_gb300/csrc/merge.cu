// Exact LSE merge of partial attention results.
//
// "vLLM DCP and PCP", Deep Dive 6: with l = max_i L_i and a_i = exp(L_i - l),
// O = sum_i a_i o_i / sum_i a_i and L = l + log sum_i a_i, independently for
// every (request, head) row.  Partials with L_i = -inf carry no weight.
#include "dcp_internal.cuh"

namespace dcp {
namespace {

// Merge n partials of one row held at o(i) / lse(i); lanes split the Dv
// columns.  Writes dst(d) for the lane's columns and returns the merged LSE.
template <typename OFn, typename LFn, typename DFn>
__device__ __forceinline__ float warp_merge_row(int n, int Dv, OFn o, LFn lse, DFn dst, int lane) {
    float mx = -INFINITY;
    for (int i = lane; i < n; i += 32) mx = fmaxf(mx, lse(i));
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
    if (mx == -INFINITY) {
        for (int d = lane; d < Dv; d += 32) dst(d, 0.f);
        return -INFINITY;
    }
    float sum = 0.f;
    for (int i = lane; i < n; i += 32) sum += expf(lse(i) - mx);
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, s);
    const float inv = 1.f / sum;
    for (int d = lane; d < Dv; d += 32) {
        float acc = 0.f;
        for (int i = 0; i < n; ++i) {
            const float li = lse(i);
            if (li == -INFINITY) continue;
            acc += expf(li - mx) * o(i, d);
        }
        dst(d, acc * inv);
    }
    return mx + logf(sum);
}

// The same merge for rows whose Dv is a multiple of 128, with fp32 partials
// at 16-byte aligned addresses: each lane owns four-column pieces
// (columns 4 lane + 128 k), the weights are computed once per partial, and
// the partials' loads are independent 16-byte vector loads.  dst4(k, v)
// stores the merged piece k.
template <typename O4Fn, typename LFn, typename DFn>
__device__ __forceinline__ float warp_merge_row_v4(int n, int Dv, O4Fn o4, LFn lse, DFn dst4, int lane) {
    float mx = -INFINITY;
    for (int i = lane; i < n; i += 32) mx = fmaxf(mx, lse(i));
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
    const int nk = Dv / 128;
    if (mx == -INFINITY) {
        for (int k = 0; k < nk; ++k) dst4(k, make_float4(0.f, 0.f, 0.f, 0.f));
        return -INFINITY;
    }
    float sum = 0.f;
    for (int i = lane; i < n; i += 32) sum += expf(lse(i) - mx);
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, s);
    const float inv = 1.f / sum;
    constexpr int kMaxK = 8;  // Dv up to 1024 in registers
    for (int k0 = 0; k0 < nk; k0 += kMaxK) {
        float4 acc[kMaxK];
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
        for (int i = 0; i < n; ++i) {
            const float li = lse(i);
            if (li == -INFINITY) continue;
            const float wgt = expf(li - mx) * inv;
#pragma unroll
            for (int k = 0; k < kMaxK; ++k) {
                if (k0 + k < nk) {
                    const float4 v = o4(i, k0 + k);
                    acc[k].x += wgt * v.x;
                    acc[k].y += wgt * v.y;
                    acc[k].z += wgt * v.z;
                    acc[k].w += wgt * v.w;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kMaxK; ++k)
            if (k0 + k < nk) dst4(k0 + k, acc[k]);
    }
    return mx + logf(sum);
}

__device__ __forceinline__ void store_out4(void* out, int64_t idx, float4 v, int dtype) {
    if (dtype == DCP_F32) {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + idx) = v;
    } else {
        __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&lo);
        u.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + idx) = u;
    }
}

// One warp per (group, row): merges the group's segment partials.
__global__ void segment_merge_kernel(AttnArgs a) {
    pdl_wait();  // the attention kernel's partials
    const int lane = threadIdx.x & 31;
    const int64_t g = blockIdx.x;
    const int row = blockIdx.y * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= a.rows) return;
    const int32_t* seg_base = reinterpret_cast<const int32_t*>(a.ws + a.lay.off_seg_base);
    const float* part_o = reinterpret_cast<const float*>(a.ws + a.lay.off_part_o);
    const float* part_lse = reinterpret_cast<const float*>(a.ws + a.lay.off_part_lse);
    const int base = seg_base[g];
    const int n = seg_base[g + 1] - base;
    // n == 0: a group that owns no chunk; the merge below gives zeros and -inf
    int b, kvh, r = 0;
    if (a.partial_mode) {
        r = (int)(g % a.N);
        b = (int)((g / a.N) / a.Hkv);
        kvh = (int)((g / a.N) % a.Hkv);
    } else {
        b = (int)(g / a.Hkv);
        kvh = (int)(g % a.Hkv);
    }
    const int t = row / a.G, gq = row % a.G;
    const int64_t orow = ((int64_t)b * a.Tq + t) * a.Hq + (int64_t)kvh * a.G + gq;
    const int rows = a.rows, Dv = a.Dv;
    auto o = [&](int i, int d) { return part_o[((int64_t)(base + i) * rows + row) * Dv + d]; };
    auto l = [&](int i) { return part_lse[(int64_t)(base + i) * rows + row]; };
    const uintptr_t dst_addr = reinterpret_cast<uintptr_t>(a.partial_mode ? (void*)a.out_partial : a.out);
    if (Dv % 128 == 0 && (dst_addr & 15u) == 0) {
        auto o4 = [&](int i, int k) {
            return *reinterpret_cast<const float4*>(part_o + ((int64_t)(base + i) * rows + row) * Dv + 128 * k +
                                                    4 * lane);
        };
        if (a.partial_mode) {
            const int64_t prow = (int64_t)r * a.B * a.Tq * a.Hq + orow;
            float* dst = a.out_partial + prow * Dv;
            const float L = warp_merge_row_v4(
                n, Dv, o4, l,
                [&](int k, float4 v) { *reinterpret_cast<float4*>(dst + 128 * k + 4 * lane) = v; }, lane);
            if (lane == 0) a.lse_partial[prow] = L;
        } else {
            const float L = warp_merge_row_v4(
                n, Dv, o4, l, [&](int k, float4 v) { store_out4(a.out, orow * Dv + 128 * k + 4 * lane, v, a.out_dtype); },
                lane);
            if (lane == 0 && a.lse) a.lse[orow] = L;
        }
        return;
    }
    if (a.partial_mode) {
        const int64_t prow = (int64_t)r * a.B * a.Tq * a.Hq + orow;
        float* dst = a.out_partial + prow * Dv;
        const float L = warp_merge_row(n, Dv, o, l, [&](int d, float v) { dst[d] = v; }, lane);
        if (lane == 0) a.lse_partial[prow] = L;
    } else {
        const float L = warp_merge_row(
            n, Dv, o, l, [&](int d, float v) { store_out(a.out, orow * Dv + d, v, a.out_dtype); }, lane);
        if (lane == 0 && a.lse) a.lse[orow] = L;
    }
}

__global__ void lse_merge_kernel(int N, int64_t rows, int Dv, const float* o_parts, const float* lse_parts,
                                 void* out, int out_dtype, float* lse) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    if (row >= rows) return;
    auto o = [&](int i, int d) { return o_parts[((int64_t)i * rows + row) * Dv + d]; };
    auto l = [&](int i) { return lse_parts[(int64_t)i * rows + row]; };
    // rows of a multiple of 128 columns at 16-byte aligned addresses: the vector
    // merge (weights once per part, independent 16-byte loads)
    const uintptr_t ends = reinterpret_cast<uintptr_t>(o_parts) | reinterpret_cast<uintptr_t>(out);
    if (Dv % 128 == 0 && (ends & 15u) == 0) {
        auto o4 = [&](int i, int k) {
            return *reinterpret_cast<const float4*>(o_parts + ((int64_t)i * rows + row) * Dv + 128 * k + 4 * lane);
        };
        const float L = warp_merge_row_v4(
            N, Dv, o4, l, [&](int k, float4 v) { store_out4(out, row * Dv + 128 * k + 4 * lane, v, out_dtype); },
            lane);
        if (lane == 0 && lse) lse[row] = L;
        return;
    }
    const float L = warp_merge_row(
        N, Dv, o, l, [&](int d, float v) { store_out(out, row * Dv + d, v, out_dtype); }, lane);
    if (lane == 0 && lse) lse[row] = L;
}

}  // namespace

cudaError_t launch_segment_merge(const AttnArgs& a, cudaStream_t s) {
    if (a.Gn == 0) return cudaSuccess;
    dim3 grid((unsigned)a.Gn, (unsigned)((a.rows + 3) / 4));
    return launch_pdl(segment_merge_kernel, grid, dim3(128), 0, s, a);
}

cudaError_t launch_lse_merge(int N, int64_t rows, int Dv, const float* o_parts, const float* lse_parts,
                             void* out, int out_dtype, float* lse, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const int64_t threads = rows * 32;
    lse_merge_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(N, rows, Dv, o_parts, lse_parts, out,
                                                                     out_dtype, lse);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace dcp

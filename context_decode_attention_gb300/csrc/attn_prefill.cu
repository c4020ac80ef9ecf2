// Causal prefill attention of a PCP-partitioned chunk against DCP-sharded KV.
//
// "Breaking the Long-Sequence Inference Bottleneck ...", section 5, AllGather Q
// path: once every rank's query rows are gathered, prefill is the DCP flow:
// the full query set against each rank's own KV shard gives one partial
// (o_r, lse_r) per rank, and the exact LSE merge of the partials is the
// output ("vLLM DCP and PCP", Deep Dive 6).  After the head-tail partition
// (section 4) the gathered rows are not in position order, so each row
// carries its global position p and sees the tokens 0..p: on rank r, its
// local positions below local_len(p + 1, r).
//
// GQA, bf16, D = 64 or 128.  A CTA takes 64 rows (16 / G query tokens x the
// G heads of one KV head, so every K/V byte it stages serves all of them) of
// one request and KV head against one rank's shard; 4 warps x 16 rows on
// mma.sync.m16n8k16 (bf16 in, fp32 accumulate), online softmax in base 2,
// K/V tiles of 64 local tokens double-buffered through cp.async into an
// XOR-swizzled shared ring.  Output: the rank's partial, normalised, fp32;
// rows whose position is -1 (partition padding) or that see no token of the
// shard get zeros and -inf.
#include "dcp_internal.cuh"
#include "mma_sync.cuh"
#include "sm100_prims.cuh"

namespace dcp {
namespace {

using namespace mma;

constexpr int kWarps = 4;
constexpr int kRows = 16 * kWarps;  // rows per CTA
constexpr int kKeys = 64;           // local tokens per K/V tile

// 16-byte copy that writes zeros when `valid` is false (src must still be a
// mapped address)
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, bool valid) {
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n) : "memory");
}

template <int D>
struct PCfg {
    static constexpr int kRowBytes = D * 2;
    static constexpr int kTileBytes = kKeys * kRowBytes;
    static constexpr int kStageBytes = 2 * kTileBytes;  // K + V
    static constexpr int kSmem = 2 * kStageBytes;
    static constexpr int kPieces = kTileBytes / 16;
    static constexpr int kKSteps = D / 16;
    static constexpr int kNT = D / 8;
};

template <int D>
__global__ void __launch_bounds__(kWarps * 32) prefill_partial_kernel(PrefillArgs a) {
    using C = PCfg<D>;
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    // CTA = (unit, row tile), row tiles of one unit adjacent so that they
    // share the unit's K/V tiles in L2; unit = (b * Hkv + kvh) * N + r
    const int64_t nrt = ((int64_t)a.Tq * a.G + kRows - 1) / kRows;
    const int64_t unit = blockIdx.x / nrt;
    const int row0 = (int)(blockIdx.x % nrt) * kRows;
    const int r = (int)(unit % a.N);
    const int64_t bk = unit / a.N;
    const int b = (int)(bk / a.Hkv), kvh = (int)(bk % a.Hkv);
    uint32_t* err = &reinterpret_cast<WsHeader*>(a.ws)->err;
    __shared__ int s_kv;  // local tokens the CTA's rows need

    // the shard: rank r's local length of request b (checked against the closed form)
    const int32_t L = a.seq_lens[b];
    int32_t len = 0;
    if (L > 0) {
        const uint32_t expect = local_len32((uint32_t)L, r, a.N, a.I);
        const int32_t given = a.local_lens[(int64_t)r * a.B + b];
        if (given != (int32_t)expect && tid == 0) raise_err(err, DCP_DEV_ERR_STALE);
        len = given < 0 ? 0 : ((uint32_t)given < expect ? given : (int32_t)expect);
        if (((int64_t)len + a.bs - 1) / a.bs > a.max_blocks) {
            if (tid == 0) raise_err(err, DCP_DEV_ERR_TABLE);
            len = a.max_blocks * a.bs;
        }
    }

    // rows of this warp: A = g8, B = g8 + 8 of the warp's 16
    const int g8 = lane >> 2, t4 = lane & 3;
    auto row_pos = [&](int row, int& t) -> int32_t {
        t = row / a.G;
        if (t >= a.Tq) return -1;
        const int32_t p = a.q_pos[(int64_t)b * a.Tq + t];
        if (p >= L) {
            raise_err(err, DCP_DEV_ERR_TOKEN);
            return -1;
        }
        return p;
    };
    const int rowA = row0 + warp * 16 + g8, rowB = rowA + 8;
    int tA, tB;
    const int32_t pA = row_pos(rowA, tA), pB = row_pos(rowB, tB);
    // causal bound of each row in rank r's local positions
    const int32_t boundA = pA < 0 ? 0 : min(len, (int32_t)local_len32((uint32_t)pA + 1u, r, a.N, a.I));
    const int32_t boundB = pB < 0 ? 0 : min(len, (int32_t)local_len32((uint32_t)pB + 1u, r, a.N, a.I));
    if (tid == 0) s_kv = 0;
    __syncthreads();
    int bmax = max(boundA, boundB);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bmax = max(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
    int bmin = min(boundA, boundB);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bmin = min(bmin, __shfl_xor_sync(0xffffffffu, bmin, o));
    if (lane == 0) atomicMax(&s_kv, bmax);
    __syncthreads();
    const int kv = s_kv;
    const int ntiles = (kv + kKeys - 1) / kKeys;

    // query fragments (rows past the request, or padding, are zero)
    const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(a.q);
    auto qrow = [&](int row, int t) -> const uint32_t* {
        if (t >= a.Tq) return nullptr;
        const int gq = row % a.G;
        return reinterpret_cast<const uint32_t*>(qb + (((int64_t)b * a.Tq + t) * a.Hq + (int64_t)kvh * a.G + gq) * D);
    };
    const uint32_t* qa = qrow(rowA, tA);
    const uint32_t* qbp = qrow(rowB, tB);
    uint32_t qf[C::kKSteps][4];
#pragma unroll
    for (int ks = 0; ks < C::kKSteps; ++ks) {
        const int e = ks * 8 + t4;
        qf[ks][0] = qa ? qa[e] : 0u;
        qf[ks][1] = qbp ? qbp[e] : 0u;
        qf[ks][2] = qa ? qa[e + 4] : 0u;
        qf[ks][3] = qbp ? qbp[e + 4] : 0u;
    }

    // K/V tile loads: piece i of a tile is row i / (D/8), 16-byte column i % (D/8)
    const int32_t* bt = a.block_tables + ((int64_t)r * a.B + b) * a.max_blocks;
    const uint8_t* kp = reinterpret_cast<const uint8_t*>(a.k_pool);
    const uint8_t* vp = reinterpret_cast<const uint8_t*>(a.v_pool);
    const uint32_t sbase = smem_u32(smem);
    auto issue = [&](int kt) {
        if (kt < ntiles) {
            const uint32_t st = sbase + (uint32_t)(kt & 1) * C::kStageBytes;
#pragma unroll
            for (int i = tid; i < C::kPieces; i += kWarps * 32) {
                const int row = i / (D / 8), pc = i % (D / 8);
                const int lp = kt * kKeys + row;
                bool valid = lp < kv;
                int64_t off = 0;
                if (valid) {
                    const int32_t blk = bt[lp / a.bs];
                    if (blk < 0 || blk >= a.num_blocks) {
                        raise_err(err, DCP_DEV_ERR_BLOCK_ID);
                        valid = false;
                    } else {
                        off = (((int64_t)blk * a.Hkv + kvh) * a.bs + lp % a.bs) * C::kRowBytes + pc * 16;
                    }
                }
                const uint32_t so = row * C::kRowBytes + ((pc ^ (row & 7)) << 4);
                cp_async16_zfill(st + so, kp + off, valid);
                cp_async16_zfill(st + C::kTileBytes + so, vp + off, valid);
            }
        }
        cp_async_commit();
    };

    float o[C::kNT][4];
#pragma unroll
    for (int j = 0; j < C::kNT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
    const float sl2 = a.softmax_scale * 1.4426950408889634f;

    issue(0);
    for (int kt = 0; kt < ntiles; ++kt) {
        issue(kt + 1);
        cp_async_wait<1>();
        __syncthreads();
        const uint32_t st = sbase + (uint32_t)(kt & 1) * C::kStageBytes;
        const int k0 = kt * kKeys;
        if (k0 < bmax) {  // some row of this warp sees a token of the tile
            // S = Q K^T: 8 n-tiles of 8 tokens
            float s[kKeys / 8][4];
#pragma unroll
            for (int nt = 0; nt < kKeys / 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
            {
                const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
                for (int ks = 0; ks < C::kKSteps; ++ks) {
#pragma unroll
                    for (int np = 0; np < kKeys / 16; ++np) {
                        const int tok = np * 16 + (mi >> 1) * 8 + rr;
                        const int pc = 2 * ks + (mi & 1);
                        uint32_t k0r, k1r, k2r, k3r;
                        ldsm_x4(st + tok * C::kRowBytes + ((pc ^ (tok & 7)) << 4), k0r, k1r, k2r, k3r);
                        mma_bf16(s[2 * np], qf[ks], k0r, k1r);
                        mma_bf16(s[2 * np + 1], qf[ks], k2r, k3r);
                    }
                }
            }
            // scale to base 2; mask tokens past a row's bound
            const bool all_visible = k0 + kKeys <= bmin;
            float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < kKeys / 8; ++nt) {
                if (all_visible) {
                    s[nt][0] *= sl2; s[nt][1] *= sl2; s[nt][2] *= sl2; s[nt][3] *= sl2;
                } else {
                    const int tok = k0 + nt * 8 + 2 * t4;
                    s[nt][0] = (tok < boundA) ? s[nt][0] * sl2 : -INFINITY;
                    s[nt][1] = (tok + 1 < boundA) ? s[nt][1] * sl2 : -INFINITY;
                    s[nt][2] = (tok < boundB) ? s[nt][2] * sl2 : -INFINITY;
                    s[nt][3] = (tok + 1 < boundB) ? s[nt][3] * sl2 : -INFINITY;
                }
                mxA = fmaxf(mxA, fmaxf(s[nt][0], s[nt][1]));
                mxB = fmaxf(mxB, fmaxf(s[nt][2], s[nt][3]));
            }
            mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
            mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
            mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
            mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
            const float mnA = fmaxf(mA, mxA), mnB = fmaxf(mB, mxB);
            const float useA = (mnA == -INFINITY) ? 0.f : mnA, useB = (mnB == -INFINITY) ? 0.f : mnB;
            if (__any_sync(0xffffffffu, (mnA != mA) || (mnB != mB))) {
                const float corrA = sm100::ex2_approx(mA - useA), corrB = sm100::ex2_approx(mB - useB);
                lA *= corrA;
                lB *= corrB;
#pragma unroll
                for (int j = 0; j < C::kNT; ++j) {
                    o[j][0] *= corrA; o[j][1] *= corrA;
                    o[j][2] *= corrB; o[j][3] *= corrB;
                }
            }
            mA = mnA;
            mB = mnB;
            // P as bf16 A fragments, 4 k-steps of 16 tokens
            uint32_t pf[kKeys / 16][4];
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk) {
                float p[2][4];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int nt = 2 * kk + h;
                    p[h][0] = sm100::ex2_approx(s[nt][0] - useA);
                    p[h][1] = sm100::ex2_approx(s[nt][1] - useA);
                    p[h][2] = sm100::ex2_approx(s[nt][2] - useB);
                    p[h][3] = sm100::ex2_approx(s[nt][3] - useB);
                    lA += p[h][0] + p[h][1];
                    lB += p[h][2] + p[h][3];
                }
                pf[kk][0] = pack_bf16(p[0][0], p[0][1]);
                pf[kk][1] = pack_bf16(p[0][2], p[0][3]);
                pf[kk][2] = pack_bf16(p[1][0], p[1][1]);
                pf[kk][3] = pack_bf16(p[1][2], p[1][3]);
            }
            // O += P V (V through ldmatrix.trans)
            {
                const uint32_t vt = st + C::kTileBytes;
                const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
                for (int kk = 0; kk < kKeys / 16; ++kk) {
                    const int tok = kk * 16 + (mi & 1) * 8 + rr;
#pragma unroll
                    for (int jp = 0; jp < C::kNT / 2; ++jp) {
                        const int pc = 2 * jp + (mi >> 1);
                        uint32_t v0, v1, v2, v3;
                        ldsm_x4_t(vt + tok * C::kRowBytes + ((pc ^ (tok & 7)) << 4), v0, v1, v2, v3);
                        mma_bf16(o[2 * jp], pf[kk], v0, v1);
                        mma_bf16(o[2 * jp + 1], pf[kk], v2, v3);
                    }
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    // the rank's partial: normalised output and natural-log LSE
    float la = lA + __shfl_xor_sync(0xffffffffu, lA, 1);
    la += __shfl_xor_sync(0xffffffffu, la, 2);
    float lb = lB + __shfl_xor_sync(0xffffffffu, lB, 1);
    lb += __shfl_xor_sync(0xffffffffu, lb, 2);
    const float ln2 = 0.6931471805599453f;
    const float invA = la > 0.f ? 1.f / la : 0.f, invB = lb > 0.f ? 1.f / lb : 0.f;
    auto prow = [&](int row, int t) -> int64_t {
        const int gq = row % a.G;
        return ((((int64_t)r * a.B + b) * a.Tq + t) * a.Hq + (int64_t)kvh * a.G + gq);
    };
    const bool okA = tA < a.Tq, okB = tB < a.Tq;
    const int64_t oA = okA ? prow(rowA, tA) : 0, oB = okB ? prow(rowB, tB) : 0;
#pragma unroll
    for (int j = 0; j < C::kNT; ++j) {
        const int d = j * 8 + 2 * t4;
        if (okA) *reinterpret_cast<float2*>(&a.out_partial[oA * D + d]) = make_float2(o[j][0] * invA, o[j][1] * invA);
        if (okB) *reinterpret_cast<float2*>(&a.out_partial[oB * D + d]) = make_float2(o[j][2] * invB, o[j][3] * invB);
    }
    if (t4 == 0) {
        if (okA) a.lse_partial[oA] = la > 0.f ? mA * ln2 + logf(la) : -INFINITY;
        if (okB) a.lse_partial[oB] = lb > 0.f ? mB * ln2 + logf(lb) : -INFINITY;
    }
}

template <int D>
cudaError_t launch_t(const PrefillArgs& a, cudaStream_t s) {
    using C = PCfg<D>;
    cudaError_t e = cudaFuncSetAttribute(prefill_partial_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    const int64_t ctas = ((int64_t)a.Tq * a.G + kRows - 1) / kRows * ((int64_t)a.B * a.Hkv * a.N);
    const dim3 grid((unsigned)ctas);
    return launch_pdl(prefill_partial_kernel<D>, grid, dim3(kWarps * 32), C::kSmem, s, a);
}

}  // namespace

bool prefill_supported(const dcp_params& p) {
    const int G = p.Hkv > 0 ? p.Hq / p.Hkv : 0;
    return p.layout == DCP_LAYOUT_GQA && p.q_dtype == DCP_BF16 && p.kv_dtype == DCP_BF16 && p.Dk == p.Dv &&
           (p.Dk == 64 || p.Dk == 128) && G >= 1 && G <= 16 && 16 % G == 0 && p.Hq % p.Hkv == 0;
}

cudaError_t launch_prefill_partial(const PrefillArgs& a, cudaStream_t s) {
    return a.D == 64 ? launch_t<64>(a, s) : launch_t<128>(a, s);
}

}  // namespace dcp

// MLA split-KV decode attention over an FP8 (e4m3) latent cache on tcgen05
// tensor cores, kind::f8f6f4 (sm_103a).
//
// "Breaking the Long-Sequence Inference Bottleneck ...", section 3 (MLA
// path): one compressed latent per token shared by every query head.  "vLLM
// DCP and PCP", Deep Dive 6: each virtual rank's partial (o_i, L_i) over its
// own shard, merged exactly by LSE weights.  Each CTA produces the partial of
// one segment (a contiguous run of one merge group's chunks); the segment
// merge kernel combines them.  Absorbed-MLA reading: keys are the 576-wide
// latent+RoPE rows, values their first 512 columns, 128 query heads.
//
// The cache is consumed as stored.  K sub-tiles [tile tokens x 128 fp8
// columns] go from HBM to shared memory by TMA and straight into the MMAs; the
// values are the same bytes (columns 0-511), read again as an MN-major
// operand.  The two other operands are brought to e4m3 as two-term sums
// x = hi + lo, hi = e4m3(x), lo = e4m3(x - hi), and every product is issued
// once per term:
//   * the query (bf16, prepared by mla_f8_qprep_kernel): each head row is
//     scaled by a power of two so that its largest magnitude lies in
//     (224, 448]; hi + lo then reproduces every element whose residual is an
//     e4m3 normal exactly (a bf16 value has 8 significant bits, hi keeps 4
//     and the residual the other 4), and the rest to within 2^-10 of a row
//     maximum of at least 224;
//   * the probabilities p' = 2^(s - m_ref + kPBias) <= 2^8: hi + lo keeps
//     about 8 significant bits (the residual goes through fp16) down to
//     2^-6; below that the absolute error is at most 2^-10 (values under
//     2^-10 vanish).  The reference follows the tiles both ways (a tile's
//     maximum stays above 2^(kPBias - kLowerLog2)), so a token is lost only
//     when it lies more than 15 - kLowerLog2 binades below the maximum of its
//     own 128-token tile, and a tile loses at most 127 such tokens.
// All products accumulate in fp32 in tensor memory.
//
// Work split as in the bf16 kernel: two CTAs share a token range, each owning
// half of the value columns (O half = 256 TMEM columns), both computing
// S = Q K^T.  A tile is up to two 64-token chunks.
//
// Warp roles (per CTA):
//   warps 0-2  TMA producers: TMA box b (two per ring item) is issued by
//              warp b % 3; warp 0 also loads each segment's hi/lo query
//   warp 3     TMEM owner and MMA issuer (one lane)
//   warps 4-7  softmax / O correction / segment epilogue, thread = head
// Ring items per tile: K sub-tiles 0-4 (columns 128 s .. 128 s + 127; the
// last holds columns 512-575 and zeros), then the previous tile's two value
// sub-tiles, placed in adjacent slots (a padding no-op first if needed) so
// P.V runs as N = 256 MMAs.
// TMEM: O half [0, 256), S double buffer [256, 384) and [384, 512).  The
// softmax walks S in 32-column chunks and writes chunk c's probabilities back
// over the chunk's own first 16 columns: hi in [32 c, 32 c + 8), lo in
// [32 c + 8, 32 c + 16) (4 per column), one 32-token k-step of P.V each.
// Every wait is bounded; a timeout sets DCP_DEV_ERR_TIMEOUT and the role stops.
#include <cuda_fp8.h>

#include "mla_common.cuh"
#include "sm100_prims.cuh"

namespace dcp {
namespace {

using namespace sm100;
using namespace mla;

constexpr int kSubCols = 128;                // fp8 columns per sub-tile (one 128-byte swizzle row)
constexpr int kKItems = (kDk + kSubCols - 1) / kSubCols;  // 5
constexpr int kVItems = kDvHalf / kSubCols;  // 2
constexpr int kSubBytes = 2 * kChunk * kSubCols;  // [128 rows x 128 B]: 16384
constexpr int kRing = 5;
constexpr int kProd = 3;
constexpr int kWarpMma = kProd;
constexpr int kWarpSoftmax = kWarpMma + 1;
constexpr int kSoftmaxWarps = 4;
constexpr int kThreads = 32 * (kWarpSoftmax + kSoftmaxWarps);
// Prepared query row (1152 bytes): hi of columns 0-511, lo of columns 0-511,
// hi of columns 512-575, lo of columns 512-575.  Its nine 128-byte column
// blocks land as nine SW128 [128 heads x 128 B] sub-tiles: hi (4), lo (4) and
// a tail whose bytes 0-63 / 64-127 are the hi / lo of columns 512-575.
constexpr int kQRowBytes = 2 * kDk;     // 1152
constexpr int kOffQHi = 0;
constexpr int kOffQLo = 4 * kSubBytes;
constexpr int kOffQTail = 8 * kSubBytes;
constexpr int kQBytes = 9 * kSubBytes;  // 147456
constexpr int kOffRing = kQBytes;
constexpr int kOffBar = kOffRing + kRing * kSubBytes;
constexpr int kNumBars = 2 * kRing + 8;
constexpr int kOffUnits = kOffBar + kNumBars * 8 + 16;
constexpr int kUnits = 64;      // cached unit-prefix entries (kUnitCache at most)
constexpr int kTileRing = 8;    // tile descriptors handed from the producers to the MMA issuer
constexpr int kOffTiles = kOffUnits + kUnits * 8;
constexpr int kSmem = kOffTiles + kTileRing * 16;  // the dynamic buffer is 1024-byte aligned (checked at entry)
static_assert(kUnits <= kUnitCache, "unit cache");
static_assert(kSmem <= 232448, "shared memory");
// Softmax reference (log2 units), kept lazily in both directions: it moves up
// when a tile's maximum passes it by more than kRescaleLog2 (p' would leave
// e4m3's range) and down to the tile's maximum when that lies more than
// kLowerLog2 below it (a tile far below the reference would otherwise fall
// under e4m3's smallest step and vanish from P.V), as long as the largest
// weight seen stays within 2^kMaxSpanLog2 of the new reference (fp32 O and l
// then cannot overflow).  kPBias keeps p' = 2^(s - m_ref + kPBias) <= 2^8.
constexpr float kRescaleLog2 = 3.f;
constexpr float kLowerLog2 = 4.f;
constexpr float kMaxSpanLog2 = 64.f;
constexpr float kPBias = 5.f;

// One tile as the producers saw it, for the MMA issuer (which then needs no
// cursor of its own): written before the arrive that publishes the tile's
// first K sub-tile, read after the wait on it.
struct TileMsg {
    int32_t n_ch, first, last, has_next;
};

struct Bars {
    uint64_t *full, *empty, *q_full, *q_empty, *s_full, *p_full, *o_done, *drain;
    uint32_t* tmem_slot;
};

__device__ __forceinline__ Bars carve(uint8_t* base) {
    uint64_t* b = reinterpret_cast<uint64_t*>(base + kOffBar);
    Bars s;
    s.full = b; b += kRing;
    s.empty = b; b += kRing;
    s.q_full = b++;
    s.q_empty = b++;
    s.s_full = b; b += 2;
    s.p_full = b; b += 2;
    s.o_done = b++;
    s.drain = b++;
    s.tmem_slot = reinterpret_cast<uint32_t*>(b);
    return s;
}

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

// Launched right after the planner and run beside it (the query is an input
// of the call, complete before the planner started); it waits for the
// planner before exiting, so the attention kernel that waits for it also
// sees the plan.
__global__ void __launch_bounds__(256) mla_f8_qprep_kernel(const uint16_t* __restrict__ q, int64_t nrows,
                                                           uint8_t* __restrict__ qp, float* __restrict__ qscale) {
    pdl_trigger();
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row < nrows) qprep_row(q, row, qp, qscale);
    pdl_wait();
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_f8_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_kv, const float* __restrict__ qscale) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* sRing = smem + kOffRing;
    int64_t* us_s = reinterpret_cast<int64_t*>(smem + kOffUnits);
    TileMsg* tmsg = reinterpret_cast<TileMsg*>(smem + kOffTiles);
    const Bars sh = carve(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = blockIdx.x & 1;    // value columns [256 half, 256 half + 256)
    const int64_t w = blockIdx.x >> 1;  // worker
    const int tq = blockIdx.y;          // query token
    pdl_wait();                         // the plan and the prepared query
    pdl_trigger();                      // the segment merge may launch
    uint32_t* err = &reinterpret_cast<WsHeader*>(a.ws)->err;
    const int64_t P = reinterpret_cast<const WsHeader*>(a.ws)->total_chunks;
    if (P == 0) return;
    const int64_t We = P < a.W ? P : a.W;
    if (w >= We) return;
    if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled layouts need 1024-byte alignment
        if (threadIdx.x == 0) raise_err(err, DCP_DEV_ERR_TIMEOUT);
        return;
    }
    const int64_t c0 = worker_begin(w, We, P), c1 = worker_begin(w + 1, We, P);
    const int64_t* us = reinterpret_cast<const int64_t*>(a.ws + a.lay.off_units);
    const int64_t u0 = unit_of_chunk(us, a.U, c0);
    const int64_t ncache = cache_units(us_s, us, a.U, u0, kUnits);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.empty[i], 1);
        }
        mbar_init(sh.q_full, 1);
        mbar_init(sh.q_empty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.s_full[i], 1);
            mbar_init(&sh.p_full[i], kSoftmaxWarps);
        }
        mbar_init(sh.o_done, 1);
        mbar_init(sh.drain, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_kv);
    }
    if (warp == kWarpMma) {
        tmem_alloc(sh.tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *sh.tmem_slot;
    const uint32_t tm_o = tm;
    const int per_group = a.partial_mode ? 1 : a.N;
    TileCursor cur;
    cur.init(us, us_s, ncache, c0, c1, u0, a.N, a.partial_mode);

    if (warp < kProd) {
        // ------------------------------------------------------------ TMA producers
        // Items are numbered in consumption order; item k goes to ring slot
        // k % kRing.  Block ids are read once per tile, one tile ahead of
        // their use.
        if (lane == 0) {
            const int me = warp;
            Ring ring;
            ring.n = kRing;
            uint32_t qe_phase = 0;
            bool alive = true, bad_block = false;
            struct Ahead {
                Tile t;
                int32_t blk[2];
                bool valid;
            };
            auto fetch = [&](Ahead& x) {
                x.valid = cur.next(x.t);
                if (!x.valid) return;
                const int r = (int)((uint32_t)x.t.u % (uint32_t)a.N), b = (int)((uint32_t)x.t.u / (uint32_t)a.N);
                const int32_t* bt = a.block_tables + ((int64_t)r * a.B + b) * a.max_blocks;
                for (int k = 0; k < 2; ++k)
                    x.blk[k] = (k < x.t.n_ch) ? bt[((x.t.chunk + k) * kChunk) / a.bs] : 0;
            };
            auto row_of = [&](const Ahead& x, int k) -> int {
                int32_t blk = x.blk[k];
                if (blk < 0 || blk >= a.num_blocks) { bad_block = true; blk = 0; }
                const int64_t p = (x.t.chunk + k) * kChunk;
                return (int)((int64_t)blk * a.bs + p % a.bs);
            };
            // TMA boxes are dealt to the producer warps in turn (box b to warp
            // b % kProd), so the two boxes of an item go out from two warps at
            // once; the warp with an item's first box posts its byte count.
            int64_t box = 0;
            auto pad_item = [&]() {
                if ((int)(box % kProd) == me) {
                    if (!mbar_wait_sleep(&sh.empty[ring.slot], ring.phase ^ 1u)) { alive = false; return; }
                    mbar_arrive(&sh.full[ring.slot]);
                }
                ++box;
                ring.advance();
            };
            auto load_sub = [&](const Ahead& x, int col) {
                constexpr int box_bytes = kChunk * kSubCols;  // 8192, zeros past column 575 included
                uint8_t* dst = sRing + ring.slot * kSubBytes;
                bool waited = false;
                for (int k = 0; k < x.t.n_ch; ++k, ++box) {
                    if ((int)(box % kProd) != me) continue;
                    if (!waited) {
                        if (!mbar_wait_sleep(&sh.empty[ring.slot], ring.phase ^ 1u)) { alive = false; return; }
                        waited = true;
                    }
                    if (k == 0) mbar_arrive_expect_tx(&sh.full[ring.slot], (uint32_t)(box_bytes * x.t.n_ch));
                    tma_load_2d(dst + k * box_bytes, &tmap_kv, col, row_of(x, k), &sh.full[ring.slot]);
                }
                ring.advance();
            };
            Ahead cur_t, nxt, prev;
            prev.valid = false;
            fetch(cur_t);
            int ti = 0;
            for (;;) {
                fetch(nxt);
                if (cur_t.valid && cur_t.t.first && me == 0) {
                    // the segment's prepared query, once the previous segment's QK has read the buffer
                    if (ti > 0) {
                        if (!mbar_wait_sleep(sh.q_empty, qe_phase)) { alive = false; break; }
                        qe_phase ^= 1u;
                    }
                    const int b = (int)((uint32_t)cur_t.t.u / (uint32_t)a.N);
                    const int row0 = (int)(((int64_t)b * a.Tq + tq) * kHeads);
                    mbar_arrive_expect_tx(sh.q_full, kQBytes);
                    for (int j = 0; j < 9; ++j) tma_load_2d(smem + j * kSubBytes, &tmap_q, 128 * j, row0, sh.q_full);
                }
                if (cur_t.valid) {
                    if ((int)(box % kProd) == me) {
                        TileMsg m;
                        m.n_ch = cur_t.t.n_ch;
                        m.first = cur_t.t.first;
                        m.last = cur_t.t.last;
                        m.has_next = nxt.valid;
                        tmsg[ti % kTileRing] = m;
                    }
                    for (int s = 0; s < kKItems && alive; ++s) load_sub(cur_t, kSubCols * s);
                }
                if (prev.valid) {
                    while (alive && ring.slot + kVItems > (uint32_t)kRing) pad_item();
                    for (int j = 0; j < kVItems && alive; ++j) load_sub(prev, kDvHalf * half + kSubCols * j);
                }
                if (!cur_t.valid || !alive) break;
                prev = cur_t;
                cur_t = nxt;
                ++ti;
            }
            if (bad_block) raise_err(err, DCP_DEV_ERR_BLOCK_ID);
            if (!alive) raise_err(err, DCP_DEV_ERR_TIMEOUT);
            // on a timeout, give this warp's TMA copies time to land before the
            // CTA exits (a copy completes within microseconds)
            if (!alive) tma_drain_pause();
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            Ring ring;
            ring.n = kRing;
            uint32_t qf_phase = 0, pf_phase[2] = {0u, 0u};
            bool alive = true;
            TileMsg prev{}, t{};
            int ti = 0;
            // descriptors (start address in 16-byte units in the low bits): a sub-tile at
            // byte offset x is dq + x / 16, ring slot i is dk + 1024 i, +2 per 32-byte k-step
            const uint64_t dq = smem_desc(smem_u32(smem), 16, 1024, kLayoutSW128);
            const uint64_t dk = smem_desc(smem_u32(sRing), 16, 1024, kLayoutSW128);
            // values: MN-major, the two 128-column halves one slot (16 KB) apart, +256 per 32 tokens
            const uint64_t dv = smem_desc(smem_u32(sRing), kSubBytes, 1024, kLayoutSW128);
            constexpr uint32_t kSubDesc = kSubBytes >> 4;
            const uint32_t idesc_pv = idesc_e4m3(128, 256, 0, 1);
            bool more = true;  // every worker owns at least one chunk
            for (;;) {
                if (more) {
                    if (!mbar_wait_sleep(&sh.full[ring.slot], ring.phase)) { alive = false; break; }
                    t = tmsg[ti % kTileRing];
                    if (t.first) {
                        if (!mbar_wait_sleep(sh.q_full, qf_phase)) { alive = false; break; }
                        qf_phase ^= 1u;
                    }
                    const int sb = ti & 1;
                    const uint32_t d = tm + 256 + 128 * sb;
                    const uint32_t idesc_qk = idesc_e4m3(128, 64 * t.n_ch, 0, 0);
                    // K sub-tile s against query hi and lo: sub-tiles 0-3 four 32-column
                    // k-steps each; the tail (columns 512-575) two, its hi in bytes 0-63
                    // and lo in bytes 64-127 of the tail query sub-tile
#pragma unroll 1
                    for (int s = 0; s < kKItems; ++s) {
                        if (s > 0 && !mbar_wait_sleep(&sh.full[ring.slot], ring.phase)) { alive = false; break; }
                        tc_fence_after();
                        const uint64_t kd = dk + ring.slot * kSubDesc;
                        const bool tail = s == kKItems - 1;
                        const uint64_t ah = dq + (tail ? (kOffQTail >> 4) : ((kOffQHi + s * kSubBytes) >> 4));
                        const uint64_t al = dq + (tail ? ((kOffQTail + 64) >> 4) : ((kOffQLo + s * kSubBytes) >> 4));
                        const int nk = tail ? 2 : 4;
#pragma unroll 1
                        for (int kk = 0; kk < nk; ++kk) {
                            mma_f8_ss(d, ah + 2 * kk, kd + 2 * kk, idesc_qk, (s | kk) != 0);
                            mma_f8_ss(d, al + 2 * kk, kd + 2 * kk, idesc_qk, 1u);
                        }
                        mma_commit(&sh.empty[ring.slot]);
                        ring.advance();
                    }
                    if (!alive) break;
                    mma_commit(&sh.s_full[sb]);
                    if (t.last) mma_commit(sh.q_empty);
                }
                if (ti > 0) {
                    // padding no-ops, then O[:, half] += (P hi + P lo) V over two adjacent slots
                    while (alive && ring.slot + kVItems > (uint32_t)kRing) {
                        if (!mbar_wait_sleep(&sh.full[ring.slot], ring.phase)) { alive = false; break; }
                        mbar_arrive(&sh.empty[ring.slot]);
                        ring.advance();
                    }
                    if (!alive) break;
                    const int sb = (ti - 1) & 1;
                    if (!mbar_wait_sleep(&sh.p_full[sb], pf_phase[sb])) { alive = false; break; }
                    pf_phase[sb] ^= 1u;
                    for (int j = 0; j < kVItems; ++j)
                        if (!mbar_wait_sleep(&sh.full[ring.slot + j], ring.phase)) { alive = false; break; }
                    if (!alive) break;
                    tc_fence_after();
                    const uint32_t pa = tm + 256 + 128 * sb;
                    const uint64_t vd = dv + ring.slot * kSubDesc;
                    for (int kk = 0; kk < 2 * prev.n_ch; ++kk) {
                        mma_f8_ts(tm_o, pa + 32 * kk, vd + 256 * kk, idesc_pv, !(prev.first && kk == 0));
                        mma_f8_ts(tm_o, pa + 32 * kk + 8, vd + 256 * kk, idesc_pv, 1u);
                    }
                    for (int j = 0; j < kVItems; ++j) {
                        mma_commit(&sh.empty[ring.slot]);
                        ring.advance();
                    }
                    mma_commit(sh.o_done);
                }
                if (!more) break;
                more = t.has_next;
                prev = t;
                ++ti;
            }
            if (!alive) raise_err(err, DCP_DEV_ERR_TIMEOUT);
            // every MMA this thread issued has completed before the CTA releases
            // tensor memory (also when a role stopped early on a timeout)
            mma_commit(sh.drain);
            mbar_wait_sleep(sh.drain, 0);
        }
    } else {
        // ------------------------------------------------------------ softmax warpgroup
        const int quarter = warp & 3;
        const int h = 32 * quarter + lane;  // head row = TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
        uint32_t sf_phase[2] = {0u, 0u}, od_phase = 0;
        bool alive = true;
        Tile prev{}, t{};
        int ti = 0;
        float m_ref = -INFINITY, m_top = -INFINITY, l = 0.f;
        const float sl2 = a.softmax_scale * a.kv_scale * 1.4426950408889634f;
        float sl2h = sl2;  // sl2 times this head's query scale
        float* part_o = reinterpret_cast<float*>(a.ws + a.lay.off_part_o);
        float* part_lse = reinterpret_cast<float*>(a.ws + a.lay.off_part_lse);
        const int32_t* seg_base = reinterpret_cast<const int32_t*>(a.ws + a.lay.off_seg_base);
        const int row = tq * kHeads + h;
        int64_t bound_u = -1, bound = 0;  // causal bound of the current unit

        auto epilogue = [&](const Tile& g) {
            if (!mbar_wait(sh.o_done, od_phase)) { alive = false; return; }
            od_phase ^= 1u;
            tc_fence_after();
            const int64_t first = us[g.group * per_group];
            const int64_t slot = seg_base[g.group] + (w - worker_of(first, We, P));
            const float inv = (l > 0.f) ? a.kv_scale / l : 0.f;
            float* dst = part_o + (slot * a.rows + row) * kDv + kDvHalf * half;
            uint32_t r[32];
#pragma unroll 1
            for (int i = 0; i < kDvHalf / 32; ++i) {
                tmem_ld32(tm_o + lane_off + 32 * i, r);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; k += 4)
                    *reinterpret_cast<float4*>(dst + 32 * i + k) =
                        make_float4(__uint_as_float(r[k]) * inv, __uint_as_float(r[k + 1]) * inv,
                                    __uint_as_float(r[k + 2]) * inv, __uint_as_float(r[k + 3]) * inv);
            }
            if (half == 0) {
                const float mu = (m_ref == -INFINITY) ? 0.f : m_ref - kPBias;
                part_lse[slot * a.rows + row] = (l > 0.f) ? (mu + log2f(l)) * 0.6931471805599453f : -INFINITY;
            }
        };

        for (;;) {
            if (!cur.next(t)) break;
            if (t.u != bound_u) {
                // causal bound of this query token in rank r's local positions
                const int r = (int)((uint32_t)t.u % (uint32_t)a.N), b = (int)((uint32_t)t.u / (uint32_t)a.N);
                bound = local_len((int64_t)a.seq_lens[b] - a.Tq + tq + 1, r, a.N, a.I);
                // given local lengths (sparse staging) end the rank's tokens themselves
                if (a.lens_given) bound = min(bound, (int64_t)a.local_lens[(int64_t)r * a.B + b]);
                bound_u = t.u;
            }
            bool o_waited = false;
            if (t.first) {
                if (ti > 0) {
                    epilogue(prev);
                    if (!alive) break;
                    o_waited = true;
                }
                const int b = (int)((uint32_t)t.u / (uint32_t)a.N);
                sl2h = sl2 * qscale[((int64_t)b * a.Tq + tq) * kHeads + h];
                m_ref = m_top = -INFINITY;
                l = 0.f;
            }
            const int sb = ti & 1;
            if (!mbar_wait(&sh.s_full[sb], sf_phase[sb])) { alive = false; break; }
            sf_phase[sb] ^= 1u;
            tc_fence_after();
            const uint32_t sbase = tm + 256 + 128 * sb + lane_off;
            const int nchunks = 2 * t.n_ch;  // 32-column chunks
            // columns [0, lim) are visible to this query token
            const int64_t lim64 = bound - t.chunk * kChunk;
            const int lim = lim64 <= 0 ? 0 : (lim64 >= 32 * nchunks ? 32 * nchunks : (int)lim64);
            // pass 1: the tile's row maximum, chunk by chunk (a small loop body:
            // the kernel's speed is bound by instruction fetch, not arithmetic)
            float mraw = -INFINITY;
            uint32_t rr[32];
#pragma unroll 1
            for (int c = 0; c < nchunks; ++c) {
                tmem_ld32(sbase + 32 * c, rr);
                tmem_wait_ld();
                const int lc = lim - 32 * c;
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                if (lc >= 32) {  // every column visible: no mask, three-input max
#pragma unroll
                    for (int k = 0; k < 32; k += 2)
                        m4[(k >> 1) & 3] = fmax3(m4[(k >> 1) & 3], __uint_as_float(rr[k]), __uint_as_float(rr[k + 1]));
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        m4[k & 3] = fmaxf(m4[k & 3], (k < lc) ? __uint_as_float(rr[k]) : -INFINITY);
                }
                mraw = fmax3(mraw, fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            }
            const float mx = (lim > 0) ? mraw * sl2h : -INFINITY;
            float corr = 1.f;
            bool rescale_o = false;
            if (mx > -INFINITY) {
                m_top = fmaxf(m_top, mx);
                if (m_ref == -INFINITY) {
                    m_ref = mx;  // first visible tokens of the segment: O not yet accumulated
                    corr = 0.f;
                } else if (mx > m_ref + kRescaleLog2 || (mx < m_ref - kLowerLog2 && m_top - mx <= kMaxSpanLog2)) {
                    corr = ex2_approx(m_ref - mx);  // < 1 up, > 1 down
                    m_ref = mx;
                    rescale_o = true;
                }
            }
            const float nb = (m_ref == -INFINITY) ? 0.f : kPBias - m_ref;
            // pass 2: 16 columns at a time, p' = 2^(s sl2h + nb) split into hi/lo;
            // chunk c's hi/lo go over its own first 16 columns (hi in [32 c,
            // 32 c + 8), lo in [32 c + 8, 32 c + 16)), after they are read.
            // Fully visible steps take no mask and scale, shift and sum two
            // columns per instruction (these warps are issue-bound)
            float lsum = 0.f;
            const uint64_t sc2 = pair_f32(sl2h, sl2h), nb2 = pair_f32(nb, nb);
#pragma unroll 1
            for (int qq = 0; qq < 2 * nchunks; ++qq) {
                uint32_t r16[16];
                tmem_ld16(sbase + 16 * qq, r16);
                tmem_wait_ld();
                const int lq = lim - 16 * qq;
                uint32_t hw[4], lw[4];
                float ls4[4] = {0.f, 0.f, 0.f, 0.f};
                if (lq >= 16) {
                    // every column visible: scale, shift and sum two columns per instruction
                    uint64_t a01 = pair_f32(0.f, 0.f), a23 = pair_f32(0.f, 0.f);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        float x[4];
                        unpair_f32(fma_f32x2(pair_f32(__uint_as_float(r16[4 * k]), __uint_as_float(r16[4 * k + 1])),
                                             sc2, nb2),
                                   x[0], x[1]);
                        unpair_f32(fma_f32x2(pair_f32(__uint_as_float(r16[4 * k + 2]),
                                                      __uint_as_float(r16[4 * k + 3])),
                                             sc2, nb2),
                                   x[2], x[3]);
                        float p[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) p[e] = ex2_approx(x[e]);
                        a01 = add_f32x2(a01, pair_f32(p[0], p[1]));
                        a23 = add_f32x2(a23, pair_f32(p[2], p[3]));
                        split4(p[0], p[1], p[2], p[3], hw[k], lw[k]);
                    }
                    unpair_f32(a01, ls4[0], ls4[1]);
                    unpair_f32(a23, ls4[2], ls4[3]);
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        float p[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float sc = (4 * k + e < lq) ? __uint_as_float(r16[4 * k + e]) : -INFINITY;
                            p[e] = ex2_approx(fmaf(sc, sl2h, nb));
                            ls4[e] += p[e];
                        }
                        split4(p[0], p[1], p[2], p[3], hw[k], lw[k]);
                    }
                }
                lsum += (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
                const uint32_t col = sbase + 32 * (qq >> 1) + 4 * (qq & 1);
                tmem_st4(col, hw);
                tmem_st4(col + 8, lw);
            }
            l = (corr == 0.f ? 0.f : l * corr) + lsum;
            // P.V of the previous tile must be complete before O is touched
            if (ti > 0 && !o_waited) {
                if (!mbar_wait(sh.o_done, od_phase)) { alive = false; break; }
                od_phase ^= 1u;
                tc_fence_after();
            }
            if (__any_sync(0xffffffffu, rescale_o)) {
                const float f = rescale_o ? corr : 1.f;
                uint32_t ov[32];
#pragma unroll 1
                for (int i = 0; i < kDvHalf / 32; ++i) {
                    tmem_ld32(tm_o + lane_off + 32 * i, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * f);
                    tmem_st32(tm_o + lane_off + 32 * i, ov);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.p_full[sb]);
            prev = t;
            ++ti;
        }
        if (alive && ti > 0) epilogue(prev);
        if (!alive && lane == 0) raise_err(err, DCP_DEV_ERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc(tm, 512);
}

}  // namespace

size_t mla_f8_qprep_bytes(int64_t B, int Tq) {
    const int64_t rows = B * Tq * kHeads;
    return (size_t)rows * kQRowBytes + 256 + (size_t)rows * sizeof(float);
}

cudaError_t launch_attn_mla_f8(const AttnArgs& a, cudaStream_t s) {
    const int64_t nrows = (int64_t)a.B * a.Tq * kHeads;
    uint8_t* qp = a.ws + a.lay.off_qprep;
    float* qscale = reinterpret_cast<float*>(qp + align256((size_t)nrows * kQRowBytes));
    const int rows_per_block = 8;
    cudaError_t e = launch_pdl(mla_f8_qprep_kernel, dim3((unsigned)((nrows + rows_per_block - 1) / rows_per_block)),
                               dim3(32 * rows_per_block), 0, s, reinterpret_cast<const uint16_t*>(a.q), nrows, qp,
                               qscale);
    if (e != cudaSuccess) return e;
    CUtensorMap tq, tkv;
    if (!make_map_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, qp, kQRowBytes, (uint64_t)nrows, kQRowBytes, kSubCols,
                     kHeads, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const uint64_t rows = (uint64_t)a.num_blocks * a.bs;
    if (!make_map_2d(&tkv, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.k_pool, kDk, rows, kDk, kSubCols, kChunk,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(mla_f8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(2 * a.W), (unsigned)a.Tq);
    return launch_pdl(mla_f8_kernel, grid, dim3(kThreads), kSmem, s, a, tq, tkv, qscale);
}

}  // namespace dcp

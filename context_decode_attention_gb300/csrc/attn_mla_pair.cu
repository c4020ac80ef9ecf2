// MLA split-KV decode attention on CTA pairs: tcgen05 pair MMAs
// (cta_group::2, one issue drives the tensor cores of two SMs), bf16 or FP8
// (e4m3) latent cache, sm_103a.
//
// "Breaking the Long-Sequence Inference Bottleneck ...", section 3 (MLA
// path): one compressed latent per token shared by every query head.  "vLLM
// DCP and PCP", Deep Dive 6: each virtual rank's partial (o_i, L_i) over its
// own shard, merged exactly by LSE weights.  Each CTA pair produces the
// partial of one segment (a contiguous run of one merge group's chunks); the
// segment merge kernel combines them.  Absorbed-MLA reading: keys are the
// 576-wide latent+RoPE rows, values their first 512 columns, 128 query heads.
//
// The products are taken transposed, so that the cached tokens are the MMA's
// M dimension and every product is one 256-row pair MMA:
//     S^T [256 tokens x 128 heads]  = K [256 x 576] . Q^T
//     O^T [512 values x 128 heads] += V^T [512 x 256] . P^T [256 x 128]
// A pair tile is up to four 64-token chunks of one unit.  CTA c (its rank in
// the cluster) holds chunks 2c and 2c + 1 as the rows of its K operand and of
// its half of S^T, and value rows [256 b + 128 c, +128) of O^T block b
// (b = 0, 1).  The B operands are split by N between the two CTAs.  P^T: CTA c
// keeps the columns of heads [64 c, 64 c + 64) for all 256 tokens, so each
// softmax thread sends half of its probabilities to the peer CTA (st.async,
// completing on the peer's barrier).  Query, bf16: CTA c keeps the rows of
// heads [64 c, 64 c + 64) (N = 128).  Query, FP8: N = 256, CTA 0 keeps the hi
// term of all 128 heads and CTA 1 the lo term, so one MMA yields S^T's hi and
// lo parts side by side (256 TMEM columns) and QK takes 18 instructions.  No
// product is computed twice, and each SM stages per tile its 128 tokens' keys
// plus its 256 value columns of all 256 tokens.
//
// Softmax, thread = token (a TMEM lane of S^T).  The thread loads its S^T row
// into registers and releases the TMEM buffer at once.  Per tile the head maxima are
// reduced across the warp (a transposing butterfly), across the four softmax
// warps (shared memory) and across the pair (st.async into the peer); thread
// 32 w + lane of each CTA owns head 32 w + lane: its reference and its share
// of the row sum.  Both CTAs take the same reference decisions from the same
// maxima.  bf16 cache: P in bf16 relative to a lazy reference that only rises
// (by more than 2^8 at a time; O^T's columns are then rescaled).  FP8 cache:
// kind::f8f6f4 on the cache as stored, the query and P as e4m3 hi + lo
// (mla_f8_split.cuh), P relative to a lazy reference that follows the tiles
// both ways: up when a tile's maximum passes it (p' would leave e4m3's range),
// down to a tile's maximum far below it (so that a long flat tail far under a
// strong key stays above e4m3's smallest step).
//
// Roles (per CTA, 16 warps):
//   warps 0-2   TMA producers (box b from warp b % 3; warp 0 also the query)
//   warp 3      TMEM owner; in CTA 0, lane 0 issues every MMA of the pair; in
//               CTA 1, lane 0 forwards the completion of its P^T to CTA 0
//   warps 4-7   softmax group A: head maxima, pair exchange and reference
//               decision of tile i + 1 (one warp per TMEM lane quarter) ...
//   warps 8-15  ... while group B computes tile i's probabilities, P^T, row
//               sums, O^T rescale and segment epilogue (thread = TMEM lane;
//               two warps per lane quarter, one per half of the heads)
// Shared memory: query half 72 KB | P^T 32 KB (FP8: two buffers) | ring of
// 16 KB slots (bf16 seven, FP8 five).
// TMEM (512 columns per CTA): S^T buffers [0, 128) and [128, 256), O^T blocks
// [256, 384) and [384, 512).
// Every wait is bounded; a timeout sets DCP_DEV_ERR_TIMEOUT and the role stops
// (the softmax warps leave together, through a flag read after each of their
// barriers).
#include <cuda_fp8.h>

#include "mla_common.cuh"
#include "mla_f8_split.cuh"
#include "sm100_prims.cuh"

namespace dcp {
namespace {

using namespace sm100;
using namespace mla;

constexpr int kTileCh = 4;             // chunks per pair tile (256 tokens)
constexpr int kBox = 8192;             // one TMA box: 64 rows x 128 bytes
constexpr int kSlot = 2 * kBox;        // ring slot: 128 rows x 128 bytes
constexpr int kRing = 7;               // ring slots, at most (bf16 7, FP8 5)
constexpr int kProd = 3;
constexpr int kWarpMma = kProd;
constexpr int kWarpSm = kWarpMma + 1;
constexpr int kAWarps = 4;              // softmax group A: one warp per lane quarter, all heads
constexpr int kSmWarps = 8;             // softmax group B: two per SM sub-partition (lane quarter x head half)
constexpr int kAThreads = 32 * kAWarps;
constexpr int kSmThreads = 32 * kSmWarps;
constexpr int kWarpB = kWarpSm + kAWarps;  // group B (probabilities); group A (maxima, references) before it
constexpr int kThreads = 32 * kWarpB + kSmThreads;
constexpr int kQBytes = 9 * kBox;      // this CTA's 64 query rows x 1152 bytes
constexpr int kOffP = kQBytes;
constexpr int kPBytes = 4 * kBox;      // P^T: 256 tokens x 64 heads (bf16, or e4m3 hi + lo)
constexpr uint32_t kPRemote = kPBytes / 2;  // the part of P^T the peer's 128 tokens write
constexpr int kOffMisc = kOffP + kPBytes + kRing * kSlot;  // the same for both layouts (Cfg)
constexpr int kUnits = 64;
constexpr int kTileRing = 8;
constexpr int kBarA = 1;               // named barriers of the two softmax groups
constexpr int kBarB = 2;
static_assert(kOffP % 1024 == 0, "swizzled operands need 1024-byte alignment");
static_assert(kUnits <= kUnitCache, "unit cache");

// Softmax references (log2 units).  bf16: p' = 2^(x - m_ref), the reference
// raised only when a tile's maximum passes it by more than kUpBf16.  FP8:
// p' = 2^(x - m_ref + kPBias) <= 2^8, the reference raised when a tile's
// maximum passes it by more than kRescaleLog2 and lowered to the tile's
// maximum when that lies more than kLowerLog2 below it, as long as the largest
// weight seen stays within 2^kMaxSpanLog2 of the new reference.
constexpr float kUpBf16 = 8.f;
constexpr float kRescaleLog2 = 3.f;
constexpr float kLowerLog2 = 4.f;
constexpr float kMaxSpanLog2 = 64.f;
constexpr float kPBias = 5.f;

// One tile as the producers saw it, for the MMA issuer.
struct TileMsg {
    int32_t n_ch, first, last, has_next;
};

// A tile's softmax reference decision, from group A to group B: per head the
// shift nb (p' = 2^(s sc + nb)), the log2 scale sc, the factor alpha that
// brings O^T and l to the new reference, and the reference itself.
struct Decision {
    alignas(16) float nb[kHeads];
    alignas(16) float sc[kHeads];
    alignas(16) float alpha[kHeads];
    alignas(16) float mref[kHeads];
    int32_t rescale;  // some head's reference moved
};

struct Misc {
    uint64_t full[kRing], empty[kRing];
    uint64_t q_full, q_empty, s_full[2], s_free[2], xmax[2], xl, drain;
    // per tile parity: a tile's P^T complete here (group B), the peer's part of it
    // landed here, CTA 1's complete (forwarded), its P.V done
    uint64_t p_full[2], p_in[2], p_peer[2], p_free[2];
    uint64_t dec_full[2], dec_free[2];
    uint32_t tmem_slot;
    int32_t abort;
    TileMsg tmsg[kTileRing];
    int64_t units[kUnits];
    alignas(16) float red_max[4][kHeads];
    alignas(16) float red_sum[4][kHeads];
    Decision dec[2];
    alignas(16) float linv[kHeads];
    alignas(16) float xbuf[2][kHeads];
    alignas(16) float lbuf[kHeads];
};
constexpr int kSmem = kOffMisc + (int)sizeof(Misc);
static_assert(kSmem <= 232448, "shared memory");
static_assert(kOffMisc % 16 == 0, "16-byte reads of the per-head arrays");

template <bool kF8>
struct Cfg;
template <>
struct Cfg<false> {                    // bf16 cache
    static constexpr int kPBufs = 1;   // P^T buffers
    static constexpr int kRingN = 7;   // ring slots
    static constexpr int kAhead = 1;   // QK(i + 1) is issued before P.V(i)
    static constexpr int kKItems = 9;  // K sub-tiles of 64 columns
    static constexpr int kVItems = 8;  // V^T items (block b, chunk k): 128 values x 64 tokens
    static constexpr int kCols = 64;   // elements per 128-byte box row
    static constexpr uint32_t kIdescQK = idesc_f16(1, 256, 128, 0, 0);
    static constexpr uint32_t kIdescPV = idesc_f16(1, 256, 128, 1, 1);
};
template <>
struct Cfg<true> {                     // e4m3 cache
    // two P^T buffers, so that group B never waits for the previous tile's P.V
    // before storing, and QK runs two tiles ahead of P.V (fewer items per tile:
    // five ring slots keep the cache stream going)
    static constexpr int kPBufs = 2;
    static constexpr int kRingN = 5;
    static constexpr int kAhead = 2;
    static constexpr int kKItems = 5;  // K sub-tiles of 128 columns (the last: 512-575, then zeros)
    static constexpr int kVItems = 4;  // V^T items (block b, token half h): 128 values x 128 tokens
    static constexpr int kCols = 128;
    static constexpr uint32_t kIdescQK = idesc_e4m3(256, 128, 0, 0);
    static constexpr uint32_t kIdescPV = idesc_e4m3(256, 128, 1, 1);
};

// v[k]: this lane's value of column k.  Returns, in lane j, the max / sum over
// the warp's 32 lanes of column j: a transposing butterfly in which every
// exchange halves the columns a lane still carries (31 shuffles in all).
template <bool kMax>
__device__ __forceinline__ float xpose_reduce(float (&v)[32]) {  // v is consumed
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const bool up = (lane & w) != 0;
#pragma unroll
        for (int k = 0; k < w; ++k) {
            const float send = up ? v[k] : v[k + w];
            const float keep = up ? v[k + w] : v[k];
            const float got = __shfl_xor_sync(0xffffffffu, send, w);
            v[k] = kMax ? fmaxf(keep, got) : keep + got;
        }
    }
    return v[0];
}

// The maximum form of the same butterfly over x[k] (or -inf where !keep),
// leaving x untouched: its first exchange reads x directly.
__device__ __forceinline__ float xpose_max(const float (&x)[32], bool keep) {
    const int lane = threadIdx.x & 31;
    const bool up = (lane & 16) != 0;
    float v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float lo = keep ? x[k] : -INFINITY, hi = keep ? x[k + 16] : -INFINITY;
        const float got = __shfl_xor_sync(0xffffffffu, up ? lo : hi, 16);
        v[k] = fmaxf(up ? hi : lo, got);
    }
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1) {
        const bool u = (lane & w) != 0;
#pragma unroll
        for (int k = 0; k < w; ++k) {
            const float send = u ? v[k] : v[k + w];
            const float kept = u ? v[k + w] : v[k];
            v[k] = fmaxf(kept, __shfl_xor_sync(0xffffffffu, send, w));
        }
    }
    return v[0];
}

__device__ __forceinline__ uint32_t bf16x2_of(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__global__ void __launch_bounds__(256) pair_qprep_kernel(const uint16_t* __restrict__ q, int64_t nrows,
                                                         uint8_t* __restrict__ qp, float* __restrict__ qscale) {
    pdl_trigger();
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row < nrows) mla_f8::qprep_row(q, row, qp, qscale);
    pdl_wait();
}

template <bool kF8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_pair_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap tmap_q,
                    const __grid_constant__ CUtensorMap tmap_kv, const float* __restrict__ qscale) {
    using C = Cfg<kF8>;
    extern __shared__ __align__(1024) uint8_t smem[];
    Misc& ms = *reinterpret_cast<Misc*>(smem + kOffMisc);
    uint8_t* const sQ = smem;
    uint8_t* const sP = smem + kOffP;
    uint8_t* const sRing = smem + kOffP + C::kPBufs * kPBytes;
    static_assert(kOffP + C::kPBufs * kPBytes + C::kRingN * kSlot <= kOffMisc, "ring");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t cta = cluster_rank();  // CTA 0 issues the pair's MMAs
    const int64_t w = blockIdx.x >> 1;    // worker = CTA pair
    const int tq = blockIdx.y;            // query token
    pdl_wait();                           // the plan (and the prepared query)
    pdl_trigger();                        // the segment merge may launch
    uint32_t* err = &reinterpret_cast<WsHeader*>(a.ws)->err;
    const int64_t P = reinterpret_cast<const WsHeader*>(a.ws)->total_chunks;
    if (reinterpret_cast<const WsHeader*>(a.ws)->plan_key != a.plan_key) {  // a plan for other arguments
        if (threadIdx.x == 0) raise_err(err, DCP_DEV_ERR_PLAN);
        return;                                                              // (every CTA: same header)
    }
    if (P == 0) return;
    const int64_t We = P < a.W ? P : a.W;
    if (w >= We) return;                  // both CTAs of the pair leave here together
    if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled layouts need 1024-byte alignment (same in every CTA)
        if (threadIdx.x == 0) raise_err(err, DCP_DEV_ERR_TIMEOUT);
        return;
    }
    const int64_t c0 = worker_begin(w, We, P), c1 = worker_begin(w + 1, We, P);
    const int64_t* us = reinterpret_cast<const int64_t*>(a.ws + a.lay.off_units);
    const int64_t u0 = a.worker_starts ? reinterpret_cast<const WorkerStart*>(a.ws + a.lay.off_wfirst)[w].u0
                                       : unit_of_chunk(us, a.U, c0);
    const int64_t ncache = cache_units(ms.units, us, a.U, u0, kUnits);

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kRingN; ++i) {
            mbar_init(&ms.full[i], 1);
            mbar_init(&ms.empty[i], 1);
        }
        mbar_init(&ms.q_full, 1);
        mbar_init(&ms.q_empty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ms.s_full[i], 1);
            mbar_init(&ms.s_free[i], 2 * kSmWarps);  // group B of both CTAs
            mbar_init(&ms.xmax[i], 1);
            mbar_init(&ms.dec_full[i], kAWarps);     // group A
            mbar_init(&ms.dec_free[i], kSmWarps);    // group B
            mbar_init(&ms.p_full[i], kSmWarps);      // this CTA's group B
            mbar_init(&ms.p_free[i], 1);
            mbar_init(&ms.p_in[i], 1);
            mbar_init(&ms.p_peer[i], 1);
        }
        mbar_init(&ms.xl, 1);
        mbar_init(&ms.drain, 1);
        ms.abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_kv);
    }
    if (warp == kWarpMma) {
        tmem_alloc_pair(&ms.tmem_slot, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers exist before any signal crosses the pair
    tc_fence_after();
    const uint32_t tm = ms.tmem_slot;
    const int per_group = a.partial_mode ? 1 : a.N;
    TileCursor cur;
    cur.init(us, ms.units, ncache, c0, c1, u0, a.N, a.partial_mode, kTileCh);

    if (warp < kProd) {
        // ------------------------------------------------------------ TMA producers (both CTAs)
        // Items in consumption order: the K sub-tiles of tile i, then the V^T
        // items of tile i - 1.  Each CTA loads its own part of an item into its
        // ring slot; both parts complete on CTA 0's full barrier of the slot.
        if (lane == 0) {
            const int me = warp;
            Ring ring;
            ring.n = C::kRingN;
            uint32_t qe_phase = 0;
            bool alive = true, bad_block = false;
            const int oob_row = (int)((int64_t)a.num_blocks * a.bs);  // a box from here reads zeros
            const uint32_t lead_full0 = mapa_shared(smem_u32(&ms.full[0]), 0);
            const uint32_t lead_qfull = mapa_shared(smem_u32(&ms.q_full), 0);
            struct Ahead {
                Tile t;
                int32_t blk[kTileCh];
                bool valid;
            };
            auto fetch = [&](Ahead& x) {
                x.valid = cur.next(x.t);
                if (!x.valid) return;
                const int r = (int)((uint32_t)x.t.u % (uint32_t)a.N), b = (int)((uint32_t)x.t.u / (uint32_t)a.N);
                const int32_t* bt = a.block_tables + ((int64_t)r * a.B + b) * a.max_blocks;
                for (int k = 0; k < kTileCh; ++k)
                    x.blk[k] = (k < x.t.n_ch) ? bt[((x.t.chunk + k) * kChunk) / a.bs] : 0;
            };
            // first cache row of chunk k of a tile; a chunk past the tile reads zeros
            auto row_of = [&](const Ahead& x, int k) -> int {
                if (k >= x.t.n_ch) return oob_row;
                const int32_t blk = x.blk[k];
                if (blk < 0 || blk >= a.num_blocks) {
                    bad_block = true;
                    return oob_row;
                }
                return (int)((int64_t)blk * a.bs + ((x.t.chunk + k) * kChunk) % a.bs);
            };
            // One ring item of two boxes, (x0, y0) and (x1, y1), into the two
            // halves of the slot.  Boxes are dealt to the producer warps in turn.
            int64_t box = 0;
            auto item = [&](int x0, int y0, int x1, int y1) {
                bool waited = false;
                for (int j = 0; j < 2; ++j, ++box) {
                    if ((int)(box % kProd) != me) continue;
                    if (!waited) {
                        if (!mbar_wait_sleep(&ms.empty[ring.slot], ring.phase ^ 1u)) {
                            alive = false;
                            return;
                        }
                        waited = true;
                    }
                    if (j == 0 && cta == 0) mbar_arrive_expect_tx(&ms.full[ring.slot], 2u * kSlot);
                    tma_load_2d_pair(sRing + ring.slot * kSlot + j * kBox, &tmap_kv, j ? x1 : x0, j ? y1 : y0,
                                     lead_full0 + 8u * ring.slot);
                }
                ring.advance();
            };
            // the V^T items of tile p: after the K items of tile p + kAhead (the order in
            // which the MMA issuer consumes them)
            auto load_v = [&](const Ahead& pt) {
                const int x = 128 * (int)cta;
                if constexpr (!kF8) {
                    for (int bb = 0; bb < 2 && alive; ++bb)
                        for (int k = 0; k < kTileCh && alive; ++k) {
                            const int y = row_of(pt, k);
                            item(256 * bb + x, y, 256 * bb + x + 64, y);
                        }
                } else {
                    for (int bb = 0; bb < 2 && alive; ++bb)
                        for (int hh = 0; hh < 2 && alive; ++hh)
                            item(256 * bb + x, row_of(pt, 2 * hh), 256 * bb + x, row_of(pt, 2 * hh + 1));
                }
            };
            Ahead cur_t, nxt, p1, p2;
            p1.valid = p2.valid = false;
            fetch(cur_t);
            int ti = 0;
            for (;;) {
                fetch(nxt);
                if (cur_t.valid && cur_t.t.first && me == 0) {
                    // this CTA's query rows for the segment, once the previous segment's QK has read them
                    if (ti > 0) {
                        if (!mbar_wait_sleep(&ms.q_empty, qe_phase)) {
                            alive = false;
                            break;
                        }
                        qe_phase ^= 1u;
                    }
                    const int b = (int)((uint32_t)cur_t.t.u / (uint32_t)a.N);
                    const int rowq = (int)(((int64_t)b * a.Tq + tq) * kHeads);
                    if (cta == 0) mbar_arrive_expect_tx(&ms.q_full, 2u * kQBytes);
                    // heads [64 cta, 64 cta + 64): nine [64 rows x 128 B] sub-tiles (bf16:
                    // 64 columns each; e4m3: the prepared row hi[0:512] lo[0:512] hi[512:576]
                    // lo[512:576], so sub-tiles 0-3 hi, 4-7 lo, 8 the tail's hi and lo)
                    for (int j = 0; j < 9; ++j)
                        tma_load_2d_pair(sQ + j * kBox, &tmap_q, C::kCols * j, rowq + 64 * (int)cta, lead_qfull);
                }
                if (cur_t.valid) {
                    if (cta == 0 && (int)(box % kProd) == me) {
                        TileMsg m;
                        m.n_ch = cur_t.t.n_ch;
                        m.first = cur_t.t.first;
                        m.last = cur_t.t.last;
                        m.has_next = nxt.valid;
                        ms.tmsg[ti % kTileRing] = m;
                    }
                    const int ya = row_of(cur_t, 2 * (int)cta), yb = row_of(cur_t, 2 * (int)cta + 1);
                    for (int s = 0; s < C::kKItems && alive; ++s) item(C::kCols * s, ya, C::kCols * s, yb);
                }
                const Ahead& pt = C::kAhead == 2 ? p2 : p1;
                if (pt.valid) load_v(pt);
                if (!cur_t.valid) {
                    if (C::kAhead == 2 && p1.valid) load_v(p1);  // the last tile's values
                    break;
                }
                if (!alive) break;
                p2 = p1;
                p1 = cur_t;
                cur_t = nxt;
                ++ti;
            }
            if (bad_block) raise_err(err, DCP_DEV_ERR_BLOCK_ID);
            if (!alive) {
                raise_err(err, DCP_DEV_ERR_TIMEOUT);
                tma_drain_pause();  // this warp's copies land before the CTA exits
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer (CTA 0, one thread)
        if (cta == 0 && lane == 0) {
            Ring ring;
            ring.n = C::kRingN;
            uint32_t qf_phase = 0, sfree_phase[2] = {0u, 0u};
            bool alive = true, more = true;
            // descriptors (start address in 16-byte units in the low bits)
            const uint64_t dq = smem_desc(smem_u32(sQ), 16, 1024, kLayoutSW128);
            const uint64_t dk = smem_desc(smem_u32(sRing), 16, 1024, kLayoutSW128);
            // V^T items, MN-major: bf16 two 64-value column blocks one box apart
            const uint64_t dv = smem_desc(smem_u32(sRing), kF8 ? 16 : kBox, 1024, kLayoutSW128);
            // P^T, MN-major: bf16 128-byte rows (SW128), e4m3 64-byte rows (SW64), lo 16 KB after hi
            const uint64_t dp = kF8 ? smem_desc(smem_u32(sP), 16, 512, kLayoutSW64)
                                    : smem_desc(smem_u32(sP), 16, 1024, kLayoutSW128);
            constexpr uint32_t kSlotD = kSlot >> 4, kBoxD = kBox >> 4;
            // QK of tile j is issued while j <= (oldest pending P.V) + kAhead: QK(j) needs only
            // that group B has loaded S^T(j - 2), which it does before its stores
            TileMsg hist[4];
            int qk = 0, pv = 0;
            for (;;) {
                while (alive && more && qk <= pv + C::kAhead) {
                    if (!mbar_wait_sleep(&ms.full[ring.slot], ring.phase)) { alive = false; break; }
                    const TileMsg t = ms.tmsg[qk % kTileRing];
                    hist[qk & 3] = t;
                    if (t.first) {
                        if (!mbar_wait_sleep(&ms.q_full, qf_phase)) { alive = false; break; }
                        qf_phase ^= 1u;
                    }
                    const int sb = qk & 1;  // S^T double buffer
                    if (qk >= 2) {  // both CTAs' group B has read the buffer's previous tile
                        if (!mbar_wait_sleep_cluster(&ms.s_free[sb], sfree_phase[sb])) { alive = false; break; }
                        sfree_phase[sb] ^= 1u;
                    }
                    const uint32_t d = tm + 128u * sb;
#pragma unroll 1
                    for (int s = 0; s < C::kKItems; ++s) {
                        if (s > 0 && !mbar_wait_sleep(&ms.full[ring.slot], ring.phase)) { alive = false; break; }
                        tc_fence_after();
                        const uint64_t ka = dk + ring.slot * kSlotD;
                        if constexpr (!kF8) {
                            const uint64_t qb = dq + s * kBoxD;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_pair_f16(d, ka + 2 * kk, qb + 2 * kk, C::kIdescQK, (s | kk) != 0);
                        } else {
                            // query sub-tiles: hi 0-3, lo 4-7; the tail (columns 512-575) holds hi in
                            // bytes 0-63 and lo in bytes 64-127; each K-step once per term
                            const bool tail = s == C::kKItems - 1;
                            const uint64_t qh = dq + (tail ? 8 * kBoxD : s * kBoxD);
                            const uint64_t ql = tail ? qh + 4 : dq + (4 + s) * kBoxD;
                            const int nk = tail ? 2 : 4;
#pragma unroll 1
                            for (int kk = 0; kk < nk; ++kk) {
                                mma_pair_f8(d, ka + 2 * kk, qh + 2 * kk, C::kIdescQK, (s | kk) != 0);
                                mma_pair_f8(d, ka + 2 * kk, ql + 2 * kk, C::kIdescQK, 1u);
                            }
                        }
                        mma_commit_pair(&ms.empty[ring.slot]);
                        ring.advance();
                    }
                    if (!alive) break;
                    mma_commit_pair(&ms.s_full[sb]);
                    if (t.last) mma_commit_pair(&ms.q_empty);
                    more = t.has_next != 0;
                    ++qk;
                }
                if (!alive || pv == qk) break;
                // O^T += V^T P^T of tile pv, once P^T is complete in both CTAs: this CTA's
                // group B (its stores here, its O^T rescale), the part CTA 1 sent here, and
                // CTA 1's own (forwarded by its warp 3)
                const TileMsg pt = hist[pv & 3];
                const int pq = pv & 1;
                const uint32_t pph = (uint32_t)((pv >> 1) & 1);
                if (!mbar_wait_sleep(&ms.p_full[pq], pph) || !mbar_wait_sleep_cluster(&ms.p_in[pq], pph) ||
                    !mbar_wait_sleep_cluster(&ms.p_peer[pq], pph)) { alive = false; break; }
                const uint64_t dpb = dp + (uint64_t)((C::kPBufs == 2 ? (pv & 1) : 0) * (kPBytes >> 4));
#pragma unroll 1
                for (int it = 0; it < C::kVItems; ++it) {
                    if (!mbar_wait_sleep(&ms.full[ring.slot], ring.phase)) { alive = false; break; }
                    tc_fence_after();
                    const uint64_t va = dv + ring.slot * kSlotD;
                    if constexpr (!kF8) {
                        const int bb = it >> 2, k = it & 3;
                        const uint32_t o = tm + 256u + 128u * bb;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_pair_f16(o, va + kk * (2048 >> 4), dpb + (64 * k + 16 * kk) * (128 >> 4), C::kIdescPV,
                                         !(pt.first && k == 0 && kk == 0));
                    } else {
                        const int bb = it >> 1, hh = it & 1;
                        const uint32_t o = tm + 256u + 128u * bb;
#pragma unroll 1
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t tok = 128 * hh + 32 * kk;
                            mma_pair_f8(o, va + kk * (4096 >> 4), dpb + tok * (64 >> 4), C::kIdescPV,
                                        !(pt.first && hh == 0 && kk == 0));
                            mma_pair_f8(o, va + kk * (4096 >> 4), dpb + (16384 >> 4) + tok * (64 >> 4), C::kIdescPV,
                                        1u);
                        }
                    }
                    mma_commit_pair(&ms.empty[ring.slot]);
                    ring.advance();
                }
                if (!alive) break;
                mma_commit_pair(&ms.p_free[pq]);
                ++pv;
            }
            if (!alive) raise_err(err, DCP_DEV_ERR_TIMEOUT);
            // every MMA of the pair completes before either CTA releases tensor memory
            mma_commit_pair(&ms.drain);
        }
        if (cta == 1 && lane == 0) {
            // CTA 1: once per tile, when this CTA's softmax warps are done (their P^T stores
            // here, their O^T rescale) and CTA 0's part of its P^T has landed here, one
            // release at cluster scope to the MMA issuer (the softmax threads then never
            // release at cluster scope behind their own outstanding remote stores)
            const uint32_t lead_ppeer0 = mapa_shared(smem_u32(&ms.p_peer[0]), 0);
            Tile tt;
            int i = 0;
            bool alive = true;
            while (alive && cur.next(tt)) {
                const uint32_t ph = (uint32_t)((i >> 1) & 1);
                if (!mbar_wait_sleep(&ms.p_full[i & 1], ph) || !mbar_wait_sleep_cluster(&ms.p_in[i & 1], ph)) {
                    alive = false;
                    break;
                }
                mbar_arrive_cluster(lead_ppeer0 + 8u * (i & 1));
                ++i;
            }
            if (!alive) raise_err(err, DCP_DEV_ERR_TIMEOUT);
        }
        if (lane == 0) mbar_wait_sleep(&ms.drain, 0);
    } else if (warp < kWarpB) {
        // ------------------------------------------------------------ softmax group A (both CTAs)
        // Per tile: the head maxima over the pair's visible tokens and the reference
        // decision, one tile ahead of group B.  Warp qw: TMEM lane quarter qw (tokens
        // 32 qw ..), all heads; thread 32 qw + lane owns that head's reference.
        const int qw = warp - kWarpSm;
        const uint32_t lane_off = (uint32_t)(32 * qw) << 16;
        const int hown = 32 * qw + lane;
        const int jrow = 128 * (int)cta + hown;  // this thread's token row of the pair tile
        uint32_t sf_phase[2] = {0u, 0u}, df_phase[2] = {0u, 0u};
        Tile t{};
        int ti = 0;
        float m_ref = -INFINITY, m_top = -INFINITY, sl2h = 0.f;
        const float sl2 = a.softmax_scale * (kF8 ? a.kv_scale : 1.f) * 1.4426950408889634f;
        int64_t bound_u = -1, bound = 0;
        const uint32_t peer = cta ^ 1u;
        const uint32_t peer_xbuf = mapa_shared(smem_u32(&ms.xbuf[0][0]), peer);
        const uint32_t peer_xmax0 = mapa_shared(smem_u32(&ms.xmax[0]), peer);
        volatile int32_t* abort_flag = &ms.abort;
        bool alive = true;
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
            if (t.first) {
                m_ref = m_top = -INFINITY;
                if constexpr (kF8) {
                    const int b = (int)((uint32_t)t.u / (uint32_t)a.N);
                    sl2h = sl2 * qscale[((int64_t)b * a.Tq + tq) * kHeads + hown];
                }
            }
            const int sb = ti & 1;
            bool ok = __all_sync(0xffffffffu, mbar_wait(&ms.s_full[sb], sf_phase[sb]));
            sf_phase[sb] ^= 1u;
            tc_fence_after();
            const bool vis = ok && jrow < kChunk * t.n_ch && t.chunk * kChunk + jrow < bound;
            const uint32_t sbase = tm + 128u * sb + lane_off;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                if (ok) {
                    tmem_ld32(sbase + 32u * c, r);
                    tmem_wait_ld();
                }
                ms.red_max[qw][32 * c + lane] = xpose_max(reinterpret_cast<const float(&)[32]>(r), vis);
            }
            if (!ok) *abort_flag = 1;
            named_sync(kBarA, kAThreads);
            if (*abort_flag) { alive = false; break; }
            // the decision buffer of this tile's parity: group B is done with tile ti - 2's
            const int db = ti & 1;
            if (ti >= 2) {
                if (!__all_sync(0xffffffffu, mbar_wait(&ms.dec_free[db], df_phase[db]))) *abort_flag = 1;
                df_phase[db] ^= 1u;
            }
            // the pair's maximum of head hown, then its reference
            const int xp = ti & 1;
            bool rescale = false;
            if (hown == 0) mbar_arrive_expect_tx(&ms.xmax[xp], 4u * kHeads);
            const float cmax = fmaxf(fmaxf(ms.red_max[0][hown], ms.red_max[1][hown]),
                                     fmaxf(ms.red_max[2][hown], ms.red_max[3][hown]));
            st_async_b32(peer_xbuf + 4u * (kHeads * xp + hown), __float_as_uint(cmax), peer_xmax0 + 8u * xp);
            ok = mbar_wait_cluster(&ms.xmax[xp], (uint32_t)((ti >> 1) & 1));
            const float hs = kF8 ? sl2h : sl2;
            const float mraw = fmaxf(cmax, ms.xbuf[xp][hown]);
            const float mx = (mraw > -INFINITY) ? mraw * hs : -INFINITY;
            float corr = 1.f;
            if (mx > -INFINITY) {
                if (m_ref == -INFINITY) {
                    m_ref = mx;  // first visible tokens of the segment: nothing accumulated yet
                } else if (kF8 ? (mx > m_ref + kRescaleLog2 ||
                                  (mx < m_ref - kLowerLog2 && fmaxf(m_top, mx) - mx <= kMaxSpanLog2))
                               : mx > m_ref + kUpBf16) {
                    corr = ex2_approx(m_ref - mx);  // < 1 up, > 1 down
                    m_ref = mx;
                    rescale = true;
                }
                m_top = fmaxf(m_top, mx);
            }
            Decision& d = ms.dec[db];
            d.nb[hown] = (m_ref == -INFINITY) ? 0.f : (kF8 ? kPBias : 0.f) - m_ref;
            d.sc[hown] = hs;
            d.alpha[hown] = corr;
            d.mref[hown] = m_ref;
            if (!ok) *abort_flag = 1;
            const bool any_rescale = named_sync_or(kBarA, kAThreads, rescale);
            if (*abort_flag) { alive = false; break; }
            if (hown == 0) d.rescale = any_rescale ? 1 : 0;
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.dec_full[db]);  // release: this warp's decision entries
            ++ti;
        }
        if (!alive && hown == 0) raise_err(err, DCP_DEV_ERR_TIMEOUT);
    } else {
        // ------------------------------------------------------------ softmax group B (both CTAs)
        // Per tile, with group A's decision: the probabilities, this CTA's P^T columns
        // (and the peer's, by st.async), the row sums, the O^T rescale and, at a
        // segment's end, the epilogue.  Warp (qw, hh) as in group A: its P^T columns
        // live in CTA hh, its O^T rows are block hh's of lane quarter qw.
        const int sw = warp - kWarpB;
        const int qw = sw & 3, hh = sw >> 2;
        const uint32_t lane_off = (uint32_t)(32 * qw) << 16;
        const int tau = 32 * qw + lane;          // S^T row (token) / O^T row (value) of this thread
        const int jrow = 128 * (int)cta + tau;   // token row of the pair tile (P^T row)
        const bool owner = qw < 2;
        const int hown = 64 * hh + 32 * qw + lane;  // the head whose row sum an owner keeps
        const int b_tid = threadIdx.x - 32 * kWarpB;
        uint32_t sf_phase[2] = {0u, 0u}, dc_phase[2] = {0u, 0u}, xl_phase = 0;
        int pv_done = -1;                        // last tile whose P.V this thread has seen complete
        Tile prev{}, t{};
        int ti = 0;
        float l = 0.f, m_fin = -INFINITY;
        float* part_o = reinterpret_cast<float*>(a.ws + a.lay.off_part_o);
        float* part_lse = reinterpret_cast<float*>(a.ws + a.lay.off_part_lse);
        const int32_t* seg_base = reinterpret_cast<const int32_t*>(a.ws + a.lay.off_seg_base);
        int64_t bound_u = -1, bound = 0;
        const uint32_t peer = cta ^ 1u;
        const uint32_t lead_sfree0 = mapa_shared(smem_u32(&ms.s_free[0]), 0);
        const uint32_t peer_lbuf = mapa_shared(smem_u32(&ms.lbuf[0]), peer);
        const uint32_t peer_xl = mapa_shared(smem_u32(&ms.xl), peer);
        const uint32_t peer_pin0 = mapa_shared(smem_u32(&ms.p_in[0]), peer);
        // this warp's P^T columns live in CTA hh; this token's row and its swizzle
        // (SW128 rows of 128 bytes, SW64 rows of 64 bytes)
        const bool p_local = hh == (int)cta;
        const uint32_t p_base0 = p_local ? smem_u32(sP) : mapa_shared(smem_u32(sP), peer);
        const uint32_t prow = kF8 ? (uint32_t)jrow * 64u : (uint32_t)jrow * 128u;
        const uint32_t pswz = kF8 ? (uint32_t)((jrow >> 1) & 3) : (uint32_t)(jrow & 7);
        volatile int32_t* abort_flag = &ms.abort;
        bool alive = true;

        // P.V of tile k has completed: P^T may be rewritten, O^T holds tile k
        auto wait_pv = [&](int k) -> bool {
            if (k < 0 || pv_done >= k) return true;
            // warp-uniform outcome: TMEM loads and stores follow under it
            if (!__all_sync(0xffffffffu, mbar_wait(&ms.p_free[k & 1], (uint32_t)((k >> 1) & 1)))) return false;
            pv_done = k;
            tc_fence_after();
            return true;
        };

        auto epilogue = [&](const Tile& g) -> bool {
            bool ok = wait_pv(ti - 1);
            // row sums of both CTAs' tokens
            if (b_tid == 0) mbar_arrive_expect_tx(&ms.xl, 4u * kHeads);
            if (owner) {
                st_async_b32(peer_lbuf + 4u * hown, __float_as_uint(l), peer_xl);
                ok = mbar_wait_cluster(&ms.xl, xl_phase) && ok;
            }
            xl_phase ^= 1u;
            const int64_t first_u = us[g.group * per_group];
            const int64_t slot = seg_base[g.group] + (w - worker_of(first_u, We, P));
            if (owner) {
                const float ltot = l + ms.lbuf[hown];
                ms.linv[hown] = (ltot > 0.f) ? (kF8 ? a.kv_scale : 1.f) / ltot : 0.f;
                if (cta == 0 && ok) {
                    const float mu = (m_fin == -INFINITY) ? 0.f : m_fin - (kF8 ? kPBias : 0.f);
                    part_lse[slot * a.rows + tq * kHeads + hown] =
                        (ltot > 0.f) ? (mu + log2f(ltot)) * 0.6931471805599453f : -INFINITY;
                }
            }
            if (!ok) *abort_flag = 1;
            named_sync(kBarB, kSmThreads);
            if (*abort_flag) return false;
            // O^T block hh, row tau of this CTA: value 256 hh + 128 cta + tau of every head
            float* dst = part_o + (slot * a.rows + tq * kHeads) * kDv + 256 * hh + 128 * (int)cta + tau;
            uint32_t r[32];
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                tmem_ld32(tm + 256u + 128u * hh + 32u * ch + lane_off, r);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    dst[(int64_t)(32 * ch + k) * kDv] = __uint_as_float(r[k]) * ms.linv[32 * ch + k];
            }
            return true;
        };

        for (;;) {
            if (!cur.next(t)) break;
            if (t.u != bound_u) {
                const int r = (int)((uint32_t)t.u % (uint32_t)a.N), b = (int)((uint32_t)t.u / (uint32_t)a.N);
                bound = local_len((int64_t)a.seq_lens[b] - a.Tq + tq + 1, r, a.N, a.I);
                if (a.lens_given) bound = min(bound, (int64_t)a.local_lens[(int64_t)r * a.B + b]);
                bound_u = t.u;
            }
            if (t.first) {
                if (ti > 0 && !epilogue(prev)) { alive = false; break; }
                l = 0.f;
            }
            // group A's decision for this tile (S^T is then in TMEM: A waited for it)
            const int sb = ti & 1;
            bool ok = __all_sync(0xffffffffu, mbar_wait(&ms.dec_full[sb], dc_phase[sb]));
            dc_phase[sb] ^= 1u;
            ok = __all_sync(0xffffffffu, mbar_wait(&ms.s_full[sb], sf_phase[sb])) && ok;
            sf_phase[sb] ^= 1u;
            tc_fence_after();
            const Decision& d = ms.dec[sb];
            const bool vis = ok && jrow < kChunk * t.n_ch && t.chunk * kChunk + jrow < bound;
            // P^T buffer of this tile: its previous user's P.V (tile ti - kPBufs) has read it,
            // here and in the peer
            const uint32_t p_base = p_base0 + (uint32_t)((C::kPBufs == 2 ? (ti & 1) : 0) * kPBytes);
            bool pv_ok = ok && wait_pv(ti - C::kPBufs);
            if (!pv_ok) *abort_flag = 1;
            if (b_tid == 0) mbar_arrive_expect_tx(&ms.p_in[ti & 1], kPRemote);  // the peer's half of this tile's P^T
            const uint32_t peer_pin = peer_pin0 + 8u * (ti & 1);
            const uint32_t sbase = tm + 128u * sb + 64u * hh + lane_off;
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                const int h0 = 64 * hh + 32 * c;
                uint32_t r[32];
                if (ok) {
                    tmem_ld32(sbase + 32u * c, r);
                    tmem_wait_ld();
                }
                float p[32];
                const float4* nb4 = reinterpret_cast<const float4*>(&d.nb[h0]);
                const float4* sc4 = reinterpret_cast<const float4*>(&d.sc[h0]);
#pragma unroll
                for (int k4 = 0; k4 < 8; ++k4) {
                    const float4 nb = nb4[k4];
                    const float4 sc = sc4[k4];
                    float x[4];
                    unpair_f32(fma_f32x2(pair_f32(__uint_as_float(r[4 * k4]), __uint_as_float(r[4 * k4 + 1])),
                                         pair_f32(sc.x, sc.y), pair_f32(nb.x, nb.y)),
                               x[0], x[1]);
                    unpair_f32(fma_f32x2(pair_f32(__uint_as_float(r[4 * k4 + 2]), __uint_as_float(r[4 * k4 + 3])),
                                         pair_f32(sc.z, sc.w), pair_f32(nb.z, nb.w)),
                               x[2], x[3]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) p[4 * k4 + e] = vis ? ex2_approx(x[e]) : 0.f;
                }
                if constexpr (!kF8) {
                    uint32_t wv[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) wv[i] = bf16x2_of(p[2 * i], p[2 * i + 1]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t off = prow + (((4u * c + i) ^ pswz) << 4);
                        if (p_local) st_shared_v4(p_base + off, wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
                        else st_async_v4(p_base + off, wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3], peer_pin);
                    }
                } else {
                    uint32_t hw[8], lw[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        mla_f8::split4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3], hw[i], lw[i]);
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const uint32_t off = prow + (((2u * c + i) ^ pswz) << 4);
                        if (p_local) {
                            st_shared_v4(p_base + off, hw[4 * i], hw[4 * i + 1], hw[4 * i + 2], hw[4 * i + 3]);
                            st_shared_v4(p_base + 16384u + off, lw[4 * i], lw[4 * i + 1], lw[4 * i + 2], lw[4 * i + 3]);
                        } else {
                            st_async_v4(p_base + off, hw[4 * i], hw[4 * i + 1], hw[4 * i + 2], hw[4 * i + 3], peer_pin);
                            st_async_v4(p_base + 16384u + off, lw[4 * i], lw[4 * i + 1], lw[4 * i + 2], lw[4 * i + 3],
                                        peer_pin);
                        }
                    }
                }
                ms.red_sum[qw][h0 + lane] = xpose_reduce<false>(p);
            }
            // S^T read by both groups: CTA 0 may compute the tile after next into it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(lead_sfree0 + 8u * sb);  // the loads were waited for
            if (p_local) fence_proxy_async_smem();  // this CTA's own P^T stores -> the MMA
            // O^T block hh, rows of lane quarter qw: columns of heads whose reference moved
            // (both CTAs apply the same factors to their rows), once O^T holds tile ti - 1
            if (d.rescale && pv_ok) {
                pv_ok = wait_pv(ti - 1);
                if (!pv_ok) *abort_flag = 1;
            }
            if (d.rescale && pv_ok) {
#pragma unroll 1
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t o[32];
                    const uint32_t ta = tm + 256u + 128u * hh + 32u * ch + lane_off;
                    tmem_ld32(ta, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * d.alpha[32 * ch + k]);
                    tmem_st32(ta, o);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            // warps that stored P^T here release those stores (CTA scope); the others (P^T
            // sent to the peer, tracked there by its receive barrier) only order their O^T
            // rescale, already waited for
            if (lane == 0) {
                if (p_local) mbar_arrive(&ms.p_full[ti & 1]);
                else mbar_arrive_relaxed(&ms.p_full[ti & 1]);
            }
            named_sync(kBarB, kSmThreads);
            if (*abort_flag) { alive = false; break; }
            if (owner) {
                l = l * d.alpha[hown] + (ms.red_sum[0][hown] + ms.red_sum[1][hown]) +
                    (ms.red_sum[2][hown] + ms.red_sum[3][hown]);
                m_fin = d.mref[hown];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.dec_free[sb]);  // group A may write this decision buffer again
            prev = t;
            ++ti;
        }
        if (alive && ti > 0) alive = epilogue(prev);
        if (!alive && b_tid == 0) raise_err(err, DCP_DEV_ERR_TIMEOUT);
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync();  // neither CTA leaves while the peer may still signal or store into it
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc_pair(tm, 512);
}

}  // namespace

bool mla_tc_supported(const dcp_params& p) {
    return p.layout == DCP_LAYOUT_MLA && p.Hq == kHeads && p.Hkv == 1 && p.Dk == kDk && p.Dv == kDv &&
           p.q_dtype == DCP_BF16 && (p.kv_dtype == DCP_BF16 || p.kv_dtype == DCP_FP8_E4M3) &&
           p.block_size % kChunk == 0 && p.Tq >= 1 && p.Tq <= 64;
}

// worker = a CTA pair; one CTA per SM
int64_t mla_tc_workers(int num_sms, int Tq) {
    const int64_t w = num_sms / (2 * (Tq > 0 ? Tq : 1));
    return w > 0 ? w : 1;
}

size_t mla_f8_qprep_bytes(int64_t B, int Tq) {
    const int64_t rows = B * Tq * kHeads;
    return (size_t)rows * mla_f8::kQRowBytes + 256 + (size_t)rows * sizeof(float);
}

namespace {

template <bool kF8>
cudaError_t launch_pair(const AttnArgs& a, cudaStream_t s) {
    const uint64_t qrows = (uint64_t)a.B * a.Tq * kHeads;
    const float* qscale = nullptr;
    CUtensorMap tq, tkv;
    if constexpr (kF8) {
        uint8_t* qp = a.ws + a.lay.off_qprep;
        float* qs = reinterpret_cast<float*>(qp + align256((size_t)qrows * mla_f8::kQRowBytes));
        const int rows_per_block = 8;
        cudaError_t e = launch_pdl(pair_qprep_kernel, dim3((unsigned)((qrows + rows_per_block - 1) / rows_per_block)),
                                   dim3(32 * rows_per_block), 0, s, reinterpret_cast<const uint16_t*>(a.q),
                                   (int64_t)qrows, qp, qs);
        if (e != cudaSuccess) return e;
        if (!make_map_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, qp, mla_f8::kQRowBytes, qrows, mla_f8::kQRowBytes, 128, 64,
                         CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        qscale = qs;
    } else {
        if (!make_map_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, kDk, qrows, kDk * 2, 64, 64,
                         CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    const uint64_t rows = (uint64_t)a.num_blocks * a.bs;
    if (rows + kChunk > 0x7FFFFFFFull) return cudaErrorInvalidValue;  // row coordinates are int32
    if (!make_map_2d(&tkv, kF8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.k_pool, kDk,
                     rows, kDk * (kF8 ? 1 : 2), kF8 ? 128 : 64, kChunk, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(mla_pair_kernel<kF8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(2 * a.W), (unsigned)a.Tq);
    return launch_pdl(mla_pair_kernel<kF8>, grid, dim3(kThreads), kSmem, s, a, tq, tkv, qscale);
}

}  // namespace

cudaError_t launch_attn_mla_tc(const AttnArgs& a, int kv_dtype, cudaStream_t s) {
    return kv_dtype == DCP_FP8_E4M3 ? launch_pair<true>(a, s) : launch_pair<false>(a, s);
}

}  // namespace dcp

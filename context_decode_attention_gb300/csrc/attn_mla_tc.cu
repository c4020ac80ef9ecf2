// MLA split-KV decode attention over a bf16 latent cache on tcgen05 tensor
// cores, kind::f16 (sm_103a).  The fp8 cache has its own kernel
// (attn_mla_f8.cu); launch_attn_mla_tc dispatches on the cache type.
//
// "Breaking the Long-Sequence Inference Bottleneck ...", section 3 (MLA
// path): the KV cache is one compressed latent per token shared by every
// query head ("KV head = 1").  "vLLM DCP and PCP", Deep Dive 6: every virtual
// rank's partial (o_i, L_i) over its own shard, merged exactly by LSE weights.
// Here each CTA produces the partial of one segment (a contiguous run of one
// merge group's chunks); the segment merge kernel combines them.
//
// Absorbed-MLA reading: keys are the 576-wide latent+RoPE rows, values their
// first 512 columns, 128 query heads per query token.
//
// Work split.  Q (128 heads x 576) stays in shared memory; O (128 x 512 fp32)
// would need all of TMEM, so two CTAs share a token range, each owning half of
// the value columns (O half = 256 TMEM columns) and computing S = Q K^T for
// the range itself.  A tile is up to two 64-token chunks (one TMA box each);
// K and V stream through a ring of [tile x 64-column] sub-tiles.
//
// Warp roles (per CTA):
//   warps 0-2     TMA producers: TMA box b (two per ring item) is issued by
//                 warp b % 3 (one TMA instruction occupies its issuing warp
//                 for ~440 cycles)
//   warp 3        TMEM owner and MMA issuer (one lane)
//   warps 4-7     softmax / O correction / segment epilogue; thread = head
// TMEM: O half [0, 256), S double buffer [256, 384) and [384, 512); P is
// written back as bf16 pairs over the first columns of its S buffer and read
// by the P.V MMA straight from TMEM.
// Online softmax in base 2 with a lazy reference: O is rescaled only when a
// row's max grows by more than 2^8.
// Every wait is bounded; a timeout sets DCP_DEV_ERR_TIMEOUT and the role stops.
#include "mla_common.cuh"
#include "sm100_prims.cuh"

namespace dcp {
namespace {

using namespace sm100;
using namespace mla;

constexpr int kKSub = kDk / 64;              // 9 K sub-tiles of 64 columns
constexpr int kVSub = kDvHalf / 64;          // 4 V sub-tiles per value half
constexpr int kQBytes = kHeads * kDk * 2;    // 147456
constexpr int kSubBytes = 2 * kChunk * 128;  // [128 rows x 64 cols] 16-bit, SW128: 16384
constexpr float kRescaleLog2 = 8.f;

// TMA issuing warps (one TMA instruction per ~440 cycles per warp).  Three keep
// the CTA at 8 warps: each of the four SM sub-partitions then hosts two warps
// and the softmax warps can hold 255 registers (the register file is split
// per sub-partition, 16K registers each).
constexpr int kProd = 3;
constexpr int kWarpMma = kProd;                // TMEM owner / MMA issuer
constexpr int kWarpSoftmax = kWarpMma + 1;     // 4 softmax warps
constexpr int kThreads = 32 * (kWarpSoftmax + 4);
// A 5-slot ring; every tile's items are K (9), padding no-ops, then the
// previous tile's 4 V sub-tiles, which therefore always sit in slots 1-4,
// contiguous, so P.V runs as N = 256 MMAs.
constexpr int kRing = 5;
constexpr int kOffQ = 0;
constexpr int kOffRing = kQBytes;
constexpr int kOffBar = kOffRing + kRing * kSubBytes;
constexpr int kNumBars = 2 * kRing + 8;
constexpr int kOffUnits = kOffBar + kNumBars * 8 + 16;
constexpr int kTileRing = 8;  // tile descriptors handed from the producers to the MMA issuer
constexpr int kOffTiles = kOffUnits + kUnitCache * 8;
constexpr int kSmem = kOffTiles + kTileRing * 16 + 1024;  // + alignment slack
static_assert(kSmem <= 232448, "shared memory");

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

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_tc_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_kv) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sQ = smem + kOffQ;
    uint8_t* sRing = smem + kOffRing;
    int64_t* us_s = reinterpret_cast<int64_t*>(smem + kOffUnits);
    TileMsg* tmsg = reinterpret_cast<TileMsg*>(smem + kOffTiles);
    const Bars sh = carve(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = blockIdx.x & 1;    // value columns [256 half, 256 half + 256)
    const int64_t w = blockIdx.x >> 1;  // worker
    const int tq = blockIdx.y;          // query token
    pdl_wait();                         // the plan
    pdl_trigger();                      // the segment merge may launch
    uint32_t* err = &reinterpret_cast<WsHeader*>(a.ws)->err;
    const int64_t P = reinterpret_cast<const WsHeader*>(a.ws)->total_chunks;
    if (P == 0) return;
    const int64_t We = P < a.W ? P : a.W;
    if (w >= We) return;
    const int64_t c0 = worker_begin(w, We, P), c1 = worker_begin(w + 1, We, P);
    const int64_t* us = reinterpret_cast<const int64_t*>(a.ws + a.lay.off_units);
    const int64_t u0 = unit_of_chunk(us, a.U, c0);
    const int64_t ncache = cache_units(us_s, us, a.U, u0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.empty[i], 1);
        }
        mbar_init(sh.q_full, 1);
        mbar_init(sh.q_empty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.s_full[i], 1);
            mbar_init(&sh.p_full[i], 4);
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
        // The ring items (K sub-tiles of tile t, then V sub-tiles of tile t-1)
        // are numbered in consumption order; item k goes to ring slot
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
            // a no-op item: keeps the ring aligned (the MMA warp just releases it)
            auto pad_item = [&]() {
                if ((int)(box % kProd) == me) {
                    if (!mbar_wait_sleep(&sh.empty[ring.slot], ring.phase ^ 1u)) { alive = false; return; }
                    mbar_arrive(&sh.full[ring.slot]);
                }
                ++box;
                ring.advance();
            };
            auto load_sub = [&](const Ahead& x, int col) {
                constexpr int box_bytes = kChunk * 128;
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
                fetch(nxt);  // next tile's block ids load while this tile's TMAs go out
                if (cur_t.valid) {
                    const Tile& t = cur_t.t;
                    if (t.first && me == 0) {
                        if (ti > 0) {
                            if (!mbar_wait_sleep(sh.q_empty, qe_phase)) { alive = false; break; }
                            qe_phase ^= 1u;
                        }
                        const int b = (int)((uint32_t)t.u / (uint32_t)a.N);
                        const int row0 = (int)(((int64_t)b * a.Tq + tq) * kHeads);
                        mbar_arrive_expect_tx(sh.q_full, kQBytes);
                        for (int j = 0; j < kKSub; ++j) tma_load_2d(sQ + j * 16384, &tmap_q, 64 * j, row0, sh.q_full);
                    }
                    if ((int)(box % kProd) == me) {
                        TileMsg m;
                        m.n_ch = t.n_ch;
                        m.first = t.first;
                        m.last = t.last;
                        m.has_next = nxt.valid;
                        tmsg[ti % kTileRing] = m;
                    }
                    for (int s2 = 0; s2 < kKSub && alive; ++s2) load_sub(cur_t, 64 * s2);
                }
                // V of the previous tile into slots 1..4; otherwise realign to slot 0
                const uint32_t target = prev.valid ? 1u : 0u;
                while (alive && ring.slot != target) pad_item();
                if (prev.valid)
                    for (int j = 0; j < kVSub && alive; ++j) load_sub(prev, kDvHalf * half + 64 * j);
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
            // descriptors (start address in 16-byte units in the low bits): Q
            // sub-tile s at dq + 1024 s, ring slot i at dk + 1024 i, +2 per
            // 32-byte k-step; V MN-major with its 64-column blocks one slot apart
            const uint64_t dq = smem_desc(smem_u32(sQ), 16, 1024, kLayoutSW128);
            const uint64_t dk = smem_desc(smem_u32(sRing), 16, 1024, kLayoutSW128);
            const uint64_t dv = smem_desc(smem_u32(sRing + 1 * kSubBytes), kSubBytes, 1024, kLayoutSW128);
            constexpr uint32_t kSubDesc = kSubBytes >> 4;
            const uint32_t idesc_pv = idesc_f16(1, 128, 256, 0, 1);
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
                    const uint32_t idesc_qk = idesc_f16(1, 128, 64 * t.n_ch, 0, 0);
#pragma unroll 1
                    for (int s = 0; s < kKSub; ++s) {
                        if (s > 0 && !mbar_wait_sleep(&sh.full[ring.slot], ring.phase)) { alive = false; break; }
                        tc_fence_after();
                        const uint64_t kd = dk + ring.slot * kSubDesc, qd = dq + s * kSubDesc;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) mma_ss(d, qd + 2 * kk, kd + 2 * kk, idesc_qk, (s | kk) != 0);
                        mma_commit(&sh.empty[ring.slot]);
                        ring.advance();
                    }
                    if (!alive) break;
                    mma_commit(&sh.s_full[sb]);
                    if (t.last) mma_commit(sh.q_empty);
                }
                // consume the padding items that realign the ring
                const uint32_t target = (ti > 0) ? 1u : 0u;
                while (ring.slot != target) {
                    if (!mbar_wait_sleep(&sh.full[ring.slot], ring.phase)) { alive = false; break; }
                    mbar_arrive(&sh.empty[ring.slot]);
                    ring.advance();
                }
                if (!alive) break;
                if (ti > 0) {
                    // O[:, half] += P V with V's four 64-column blocks in slots 1..4
                    const int sb = (ti - 1) & 1;
                    if (!mbar_wait_sleep(&sh.p_full[sb], pf_phase[sb])) { alive = false; break; }
                    pf_phase[sb] ^= 1u;
                    for (int j = 0; j < kVSub; ++j)
                        if (!mbar_wait_sleep(&sh.full[1 + j], ring.phase)) { alive = false; break; }
                    if (!alive) break;
                    tc_fence_after();
                    const uint32_t pa = tm + 256 + 128 * sb;
#pragma unroll 1
                    for (int kk = 0; kk < 4 * prev.n_ch; ++kk)
                        mma_ts(tm_o, pa + 8 * kk, dv + 128 * kk, idesc_pv, !(prev.first && kk == 0));
                    for (int j = 0; j < kVSub; ++j) {
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
        float m_ref = -INFINITY, l = 0.f;
        const float sl2 = a.softmax_scale * a.kv_scale * 1.4426950408889634f;
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
                const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
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
            if (t.first && ti > 0) {
                epilogue(prev);
                if (!alive) break;
                o_waited = true;
            }
            if (t.first) {
                m_ref = -INFINITY;
                l = 0.f;
            }
            const int sb = ti & 1;
            if (!mbar_wait(&sh.s_full[sb], sf_phase[sb])) { alive = false; break; }
            sf_phase[sb] ^= 1u;
            tc_fence_after();
            const uint32_t sbase = tm + 256 + 128 * sb + lane_off;
            const int ncols = 64 * t.n_ch;
            // columns [0, lim) are visible to this query token
            const int64_t lim64 = bound - t.chunk * kChunk;
            const int lim = lim64 <= 0 ? 0 : (lim64 >= ncols ? ncols : (int)lim64);
            // pass 1: the tile's row maximum, 32 columns at a time (small loop
            // bodies: these warps are bound by instruction fetch, not arithmetic)
            float mraw = -INFINITY;
            {
                uint32_t rr[32];
#pragma unroll 1
                for (int c = 0; c < ncols / 32; ++c) {
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
            }
            const float mx = (lim > 0) ? mraw * sl2 : -INFINITY;
            // lazy reference max
            float corr = 1.f;
            bool rescale_o = false;
            if (mx > -INFINITY) {
                if (m_ref == -INFINITY) {
                    m_ref = mx;  // first visible tokens of the segment: O not yet accumulated
                    corr = 0.f;
                } else if (mx > m_ref + kRescaleLog2) {
                    corr = ex2_approx(m_ref - mx);
                    m_ref = mx;
                    rescale_o = true;
                }
            }
            const float nmu = (m_ref == -INFINITY) ? 0.f : -m_ref;
            // pass 2: 16 columns at a time; their bf16 pairs go to columns
            // [8 q, 8 q + 8), which earlier steps have already read.  The
            // softmax warps are bound by instruction issue: fully visible steps
            // take no mask and scale, shift and sum two columns per instruction
            // (a second softmax warpgroup over half of the columns, with the
            // row maxima exchanged at a barrier, was slower)
            float lsum = 0.f;
            const uint64_t sc2 = pair_f32(sl2, sl2), mu2 = pair_f32(nmu, nmu);
#pragma unroll 1
            for (int q = 0; q < ncols / 16; ++q) {
                uint32_t r16[16], pk[8];
                tmem_ld16(sbase + 16 * q, r16);
                tmem_wait_ld();
                const int lq = lim - 16 * q;
                float ls2[2] = {0.f, 0.f};
                if (lq >= 16) {
                    // every column visible: scale, shift and sum two columns per instruction
                    uint64_t acc = pair_f32(0.f, 0.f);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        float x0, x1;
                        unpair_f32(fma_f32x2(pair_f32(__uint_as_float(r16[2 * k]), __uint_as_float(r16[2 * k + 1])),
                                             sc2, mu2),
                                   x0, x1);
                        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                        acc = add_f32x2(acc, pair_f32(p0, p1));
                        pk[k] = pack_bf16(p0, p1);
                    }
                    unpair_f32(acc, ls2[0], ls2[1]);
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float s0 = (2 * k < lq) ? __uint_as_float(r16[2 * k]) : -INFINITY;
                        const float s1 = (2 * k + 1 < lq) ? __uint_as_float(r16[2 * k + 1]) : -INFINITY;
                        const float p0 = ex2_approx(fmaf(s0, sl2, nmu)), p1 = ex2_approx(fmaf(s1, sl2, nmu));
                        ls2[0] += p0;
                        ls2[1] += p1;
                        pk[k] = pack_bf16(p0, p1);
                    }
                }
                lsum += ls2[0] + ls2[1];
                tmem_st8(sbase + 8 * q, pk);
            }
            l = (corr == 0.f ? 0.f : l * corr) + lsum;
            // PV of the previous tile must be complete before O is touched
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

bool mla_tc_supported(const dcp_params& p) {
    return p.layout == DCP_LAYOUT_MLA && p.Hq == kHeads && p.Hkv == 1 && p.Dk == kDk && p.Dv == kDv &&
           p.q_dtype == DCP_BF16 && (p.kv_dtype == DCP_BF16 || p.kv_dtype == DCP_FP8_E4M3) &&
           p.block_size % kChunk == 0 && p.Tq >= 1 && p.Tq <= 64;
}

// worker = a CTA pair (the two value halves); one CTA per SM
int64_t mla_tc_workers(int num_sms, int Tq) {
    const int64_t w = num_sms / (2 * (Tq > 0 ? Tq : 1));
    return w > 0 ? w : 1;
}

cudaError_t launch_attn_mla_tc(const AttnArgs& a, int kv_dtype, cudaStream_t s) {
    if (kv_dtype == DCP_FP8_E4M3) return launch_attn_mla_f8(a, s);
    CUtensorMap tq, tkv;
    if (!make_map_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, kDk, (uint64_t)a.B * a.Tq * kHeads, kDk * 2, 64,
                     128, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const uint64_t rows = (uint64_t)a.num_blocks * a.bs;
    if (!make_map_2d(&tkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.k_pool, kDk, rows, kDk * 2, 64, kChunk,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(2 * a.W), (unsigned)a.Tq);
    return launch_pdl(mla_tc_kernel, grid, dim3(kThreads), kSmem, s, a, tq, tkv);
}

}  // namespace dcp

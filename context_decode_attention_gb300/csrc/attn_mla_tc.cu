// MLA split-KV decode attention on tcgen05 tensor cores (sm_103a).
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
// Warp roles (per CTA), bf16 cache:
//   warps 0-2     TMA producers: ring item k is issued by warp k % 3 (one TMA
//                 instruction occupies its issuing warp for ~440 cycles)
//   warp 3        TMEM owner and MMA issuer (one lane)
//   warps 4-7     softmax / O correction / segment epilogue; thread = head
// fp8 cache: the same, with the producers filling an fp8 staging ring and
//   warps 8-11 converting it to fp16 into the MMA ring (12 warps, so the
//   register limit is 168).
// TMEM: O half [0, 256), S double buffer [256, 384) and [384, 512); P is
// written back as 16-bit pairs over the first columns of its S buffer and read
// by the P.V MMA straight from TMEM.
// Online softmax in base 2 with a lazy reference: O is rescaled only when a
// row's max grows by more than 2^8.
// Every wait is bounded; a timeout sets DCP_DEV_ERR_TIMEOUT and the role stops.
#include <cudaTypedefs.h>

#include "dcp_internal.cuh"
#include "sm100_prims.cuh"

namespace dcp {
namespace {

using namespace sm100;

constexpr int kHeads = 128;
constexpr int kDk = 576;
constexpr int kDv = 512;
constexpr int kDvHalf = 256;
constexpr int kChunk = 64;                   // tokens per chunk (one TMA box of rows)
constexpr int kKSub = kDk / 64;              // 9 K sub-tiles of 64 columns
constexpr int kVSub = kDvHalf / 64;          // 4 V sub-tiles per value half
constexpr int kQBytes = kHeads * kDk * 2;    // 147456
constexpr int kSubBytes = 2 * kChunk * 128;  // [128 rows x 64 cols] 16-bit, SW128: 16384
constexpr float kRescaleLog2 = 8.f;

// TMA issuing warps (one TMA instruction per ~440 cycles per warp).  Three keep
// the bf16 CTA at 8 warps: each of the four SM sub-partitions then hosts two
// warps and the softmax warps can hold 255 registers (the register file is
// split per sub-partition, 16K registers each).
constexpr int kProd = 3;

template <bool FP8>
struct MlaCfg {
    // bf16: a 5-slot ring; every tile's items are K (9), padding no-ops, then
    // the previous tile's 4 V sub-tiles, which therefore always sit in slots
    // 1-4, contiguous, so P.V runs as N = 256 MMAs.  fp8: 3-slot ring, N = 64.
    static constexpr bool kWideV = !FP8;
    static constexpr int kRing = FP8 ? 3 : 5;
    static constexpr int kStage = FP8 ? 4 : 0;          // fp8 staging slots
    static constexpr int kStageBytes = 2 * kChunk * 64;  // [128 rows x 64 fp8]
    static constexpr int kWarpMma = kProd;                 // TMEM owner / MMA issuer
    static constexpr int kWarpSoftmax = kWarpMma + 1;     // 4 softmax warps
    static constexpr int kWarpConv = kWarpSoftmax + 4;    // fp8: 4 converter warps
    static constexpr int kThreads = 32 * (FP8 ? kWarpConv + 4 : kWarpSoftmax + 4);
    static constexpr int kOffQ = 0;
    static constexpr int kOffRing = kQBytes;
    static constexpr int kOffStage = kOffRing + kRing * kSubBytes;
    static constexpr int kOffBar = kOffStage + kStage * kStageBytes;
    static constexpr int kNumBars = 2 * kRing + 2 * kStage + 10;
    static constexpr int kSmem = kOffBar + kNumBars * 8 + 16 + 1024;  // + TMEM slot + alignment slack
};

struct MlaTile {
    int64_t u, chunk, group;
    int n_ch;
    bool first, last;
};

// The same tile sequence in every role: walk the worker's chunk range; a tile
// is up to two consecutive chunks of one unit.
struct TileCursor {
    const int64_t* us;
    int64_t c, c1, u, prev_group;
    int N, partial;
    __device__ void init(const int64_t* us_, int64_t c0, int64_t c1_, int64_t u0, int N_, int pm) {
        us = us_; c = c0; c1 = c1_; u = u0; N = N_; partial = pm; prev_group = -1;
    }
    __device__ int64_t group_of(int64_t uu) const { return partial ? uu : uu / N; }
    __device__ bool next(MlaTile& t) {
        if (c >= c1) return false;
        while (us[u + 1] <= c) ++u;
        t.u = u;
        t.chunk = c - us[u];
        const int64_t end = us[u + 1] < c1 ? us[u + 1] : c1;
        t.n_ch = (end - c) >= 2 ? 2 : 1;
        t.group = group_of(u);
        c += t.n_ch;
        if (c >= c1) {
            t.last = true;
        } else {
            int64_t v = u;
            while (us[v + 1] <= c) ++v;
            t.last = group_of(v) != t.group;
        }
        t.first = t.group != prev_group;
        prev_group = t.group;
        return true;
    }
};

struct Ring {
    uint32_t slot = 0, phase = 0, n = 1;
    __device__ void advance() {
        if (++slot == n) { slot = 0; phase ^= 1u; }
    }
};

struct MlaBars {
    uint64_t *full, *empty, *sfull, *sempty, *q_full, *q_empty, *s_full, *p_full, *o_done, *q_conv;
    uint32_t* tmem_slot;
};

template <bool FP8>
__device__ __forceinline__ MlaBars carve(uint8_t* base) {
    using C = MlaCfg<FP8>;
    uint64_t* b = reinterpret_cast<uint64_t*>(base + C::kOffBar);
    MlaBars s;
    s.full = b; b += C::kRing;
    s.empty = b; b += C::kRing;
    s.sfull = b; b += C::kStage;
    s.sempty = b; b += C::kStage;
    s.q_full = b++;
    s.q_empty = b++;
    s.s_full = b; b += 2;
    s.p_full = b; b += 2;
    s.o_done = b++;
    s.q_conv = b++;
    b += 2;
    s.tmem_slot = reinterpret_cast<uint32_t*>(b);
    return s;
}

__device__ __forceinline__ uint32_t pack16(float lo, float hi, bool f16) {
    if (f16) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

template <bool FP8>
__global__ void __launch_bounds__(MlaCfg<FP8>::kThreads, 1)
    mla_tc_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_kv) {
    using C = MlaCfg<FP8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sQ = smem + C::kOffQ;
    uint8_t* sRing = smem + C::kOffRing;
    uint8_t* sStage = smem + C::kOffStage;
    const MlaBars sh = carve<FP8>(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = blockIdx.x & 1;    // value columns [256 half, 256 half + 256)
    const int64_t w = blockIdx.x >> 1;  // worker
    const int tq = blockIdx.y;          // query token
    uint32_t* err = &reinterpret_cast<WsHeader*>(a.ws)->err;
    const int64_t P = reinterpret_cast<const WsHeader*>(a.ws)->total_chunks;
    if (P == 0) return;
    const int64_t We = P < a.W ? P : a.W;
    if (w >= We) return;
    const int64_t c0 = worker_begin(w, We, P), c1 = worker_begin(w + 1, We, P);
    const int64_t* us = reinterpret_cast<const int64_t*>(a.ws + a.lay.off_units);
    int64_t lo = 0, hi = a.U - 1;
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) >> 1;
        if (us[mid] <= c0) lo = mid; else hi = mid - 1;
    }
    const int64_t u0 = lo;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kRing; ++i) {
            mbar_init(&sh.full[i], FP8 ? 4 : 1);
            mbar_init(&sh.empty[i], 1);
        }
        for (int i = 0; i < C::kStage; ++i) {
            mbar_init(&sh.sfull[i], 1);
            mbar_init(&sh.sempty[i], 4);
        }
        mbar_init(sh.q_full, 1);
        mbar_init(sh.q_empty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.s_full[i], 1);
            mbar_init(&sh.p_full[i], 4);
        }
        mbar_init(sh.o_done, 1);
        mbar_init(sh.q_conv, 4);
        fence_mbar_init();
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_kv);
    }
    if (warp == C::kWarpMma) {
        tmem_alloc(sh.tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *sh.tmem_slot;
    const uint32_t tm_o = tm;
    const int per_group = a.partial_mode ? 1 : a.N;

    if (warp < kProd) {
        // ------------------------------------------------------------ TMA producers
        // The ring items (K sub-tiles of tile t, then V sub-tiles of tile t-1)
        // are numbered in consumption order; item k goes to ring slot k % kRing
        // and is issued by producer warp k % nprod.  Block ids are read once per
        // tile, one tile ahead of their use.
        if (lane == 0) {
            const int nprod = kProd;
            const int me = warp;
            TileCursor cur;
            cur.init(us, c0, c1, u0, a.N, a.partial_mode);
            Ring ring;
            ring.n = FP8 ? C::kStage : C::kRing;
            uint32_t qe_phase = 0;
            bool alive = true, bad_block = false;
            struct Ahead {
                MlaTile t;
                int32_t blk[2];
                bool valid;
            };
            auto fetch = [&](Ahead& x) {
                x.valid = cur.next(x.t);
                if (!x.valid) return;
                const int r = (int)(x.t.u % a.N), b = (int)(x.t.u / a.N);
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
            int64_t item = 0;  // global item index in consumption order
            // a no-op item: keeps the ring aligned (the MMA warp just releases it)
            auto pad_item = [&]() {
                if ((int)(item % nprod) == me) {
                    uint64_t* fullb = FP8 ? &sh.sfull[ring.slot] : &sh.full[ring.slot];
                    uint64_t* emptyb = FP8 ? &sh.sempty[ring.slot] : &sh.empty[ring.slot];
                    if (!mbar_wait(emptyb, ring.phase ^ 1u)) { alive = false; return; }
                    mbar_arrive(fullb);
                }
                ++item;
                ring.advance();
            };
            auto load_sub = [&](const Ahead& x, int col) {
                if ((int)(item % nprod) == me) {
                    uint64_t* fullb = FP8 ? &sh.sfull[ring.slot] : &sh.full[ring.slot];
                    uint64_t* emptyb = FP8 ? &sh.sempty[ring.slot] : &sh.empty[ring.slot];
                    if (!mbar_wait(emptyb, ring.phase ^ 1u)) { alive = false; return; }
                    const int box_bytes = FP8 ? kChunk * 64 : kChunk * 128;
                    mbar_arrive_expect_tx(fullb, (uint32_t)(box_bytes * x.t.n_ch));
                    uint8_t* dst = FP8 ? sStage + ring.slot * C::kStageBytes : sRing + ring.slot * kSubBytes;
                    for (int k = 0; k < x.t.n_ch; ++k)
                        tma_load_2d(dst + k * box_bytes, &tmap_kv, col, row_of(x, k), fullb);
                }
                ++item;
                ring.advance();
            };
            Ahead cur_t, nxt, prev;
            prev.valid = false;
            fetch(cur_t);
            int ti = 0;
            for (;;) {
                fetch(nxt);  // next tile's block ids load while this tile's TMAs go out
                if (cur_t.valid) {
                    const MlaTile& t = cur_t.t;
                    if (t.first && me == 0) {
                        if (ti > 0) {
                            if (!mbar_wait(sh.q_empty, qe_phase)) { alive = false; break; }
                            qe_phase ^= 1u;
                        }
                        const int b = (int)(t.u / a.N);
                        const int row0 = (int)(((int64_t)b * a.Tq + tq) * kHeads);
                        mbar_arrive_expect_tx(sh.q_full, kQBytes);
                        for (int j = 0; j < kKSub; ++j) tma_load_2d(sQ + j * 16384, &tmap_q, 64 * j, row0, sh.q_full);
                    }
                    for (int s2 = 0; s2 < kKSub && alive; ++s2) load_sub(cur_t, 64 * s2);
                }
                if (C::kWideV) {
                    // V of the previous tile into slots 1..4; otherwise realign to slot 0
                    const uint32_t target = prev.valid ? 1u : 0u;
                    while (alive && ring.slot != target) pad_item();
                }
                if (prev.valid)
                    for (int j = 0; j < kVSub && alive; ++j) load_sub(prev, kDvHalf * half + 64 * j);
                if (!cur_t.valid || !alive) break;
                prev = cur_t;
                cur_t = nxt;
                ++ti;
            }
            if (bad_block) raise_err(err, DCP_DEV_ERR_BLOCK_ID);
            if (!alive) raise_err(err, DCP_DEV_ERR_TIMEOUT);
        }
    } else if (warp == C::kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            TileCursor cur;
            cur.init(us, c0, c1, u0, a.N, a.partial_mode);
            Ring ring;
            ring.n = C::kRing;
            uint32_t qf_phase = 0, pf_phase[2] = {0u, 0u};
            bool alive = true;
            MlaTile prev{}, t{};
            int ti = 0;
            const uint32_t ab = FP8 ? 0u : 1u;  // fp16 operands for the fp8 cache, bf16 otherwise
            uint64_t* qbar = FP8 ? sh.q_conv : sh.q_full;
            const uint32_t idesc_pv = idesc_f16(ab, 128, 64, 0, 1);
            for (;;) {
                const bool more = cur.next(t);
                if (more) {
                    if (t.first) {
                        if (!mbar_wait(qbar, qf_phase)) { alive = false; break; }
                        qf_phase ^= 1u;
                    }
                    const int sb = ti & 1;
                    const uint32_t d = tm + 256 + 128 * sb;
                    const uint32_t idesc_qk = idesc_f16(ab, 128, 64 * t.n_ch, 0, 0);
                    for (int s = 0; s < kKSub; ++s) {
                        if (!mbar_wait(&sh.full[ring.slot], ring.phase)) { alive = false; break; }
                        tc_fence_after();
                        const uint32_t kb = smem_u32(sRing + ring.slot * kSubBytes);
                        const uint32_t qb = smem_u32(sQ + s * 16384);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ss(d, smem_desc(qb + kk * 32, 16, 1024, kLayoutSW128),
                                   smem_desc(kb + kk * 32, 16, 1024, kLayoutSW128), idesc_qk, (s | kk) != 0);
                        mma_commit(&sh.empty[ring.slot]);
                        ring.advance();
                    }
                    if (!alive) break;
                    mma_commit(&sh.s_full[sb]);
                    if (t.last) mma_commit(sh.q_empty);
                }
                if (C::kWideV) {
                    // consume the padding items that realign the ring
                    const uint32_t target = (ti > 0) ? 1u : 0u;
                    while (ring.slot != target) {
                        if (!mbar_wait(&sh.full[ring.slot], ring.phase)) { alive = false; break; }
                        mbar_arrive(&sh.empty[ring.slot]);
                        ring.advance();
                    }
                    if (!alive) break;
                }
                if (ti > 0 && C::kWideV) {
                    // O[:, 0:256] += P V with V's four 64-column blocks in slots 1..4
                    const int sb = (ti - 1) & 1;
                    if (!mbar_wait(&sh.p_full[sb], pf_phase[sb])) { alive = false; break; }
                    pf_phase[sb] ^= 1u;
                    for (int j = 0; j < kVSub; ++j)
                        if (!mbar_wait(&sh.full[1 + j], ring.phase)) { alive = false; break; }
                    if (!alive) break;
                    tc_fence_after();
                    const uint32_t pa = tm + 256 + 128 * sb;
                    const uint32_t vb = smem_u32(sRing + 1 * kSubBytes);
                    const uint32_t idesc_pv256 = idesc_f16(ab, 128, 256, 0, 1);
                    for (int kk = 0; kk < 4 * prev.n_ch; ++kk)
                        mma_ts(tm_o, pa + 8 * kk, smem_desc(vb + kk * 2048, kSubBytes, 1024, kLayoutSW128), idesc_pv256,
                               !(prev.first && kk == 0));
                    for (int j = 0; j < kVSub; ++j) {
                        mma_commit(&sh.empty[ring.slot]);
                        ring.advance();
                    }
                    mma_commit(sh.o_done);
                } else if (ti > 0) {
                    const int sb = (ti - 1) & 1;
                    if (!mbar_wait(&sh.p_full[sb], pf_phase[sb])) { alive = false; break; }
                    pf_phase[sb] ^= 1u;
                    tc_fence_after();
                    const uint32_t pa = tm + 256 + 128 * sb;
                    const int ksteps = 4 * prev.n_ch;
                    for (int j = 0; j < kVSub; ++j) {
                        if (!mbar_wait(&sh.full[ring.slot], ring.phase)) { alive = false; break; }
                        tc_fence_after();
                        const uint32_t vb = smem_u32(sRing + ring.slot * kSubBytes);
                        for (int kk = 0; kk < ksteps; ++kk)
                            mma_ts(tm_o + 64 * j, pa + 8 * kk, smem_desc(vb + kk * 2048, 8192, 1024, kLayoutSW128),
                                   idesc_pv, !(prev.first && kk == 0));
                        mma_commit(&sh.empty[ring.slot]);
                        ring.advance();
                    }
                    if (!alive) break;
                    mma_commit(sh.o_done);
                }
                if (!more) break;
                prev = t;
                ++ti;
            }
            if (!alive) raise_err(err, DCP_DEV_ERR_TIMEOUT);
        }
    } else if (warp < C::kWarpSoftmax + 4) {
        // ------------------------------------------------------------ softmax warpgroup
        const int quarter = warp & 3;
        const int h = 32 * quarter + lane;  // head row = TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
        TileCursor cur;
        cur.init(us, c0, c1, u0, a.N, a.partial_mode);
        uint32_t sf_phase[2] = {0u, 0u}, od_phase = 0;
        bool alive = true;
        MlaTile prev{}, t{};
        int ti = 0;
        float m_ref = -INFINITY, l = 0.f;
        const float sl2 = a.softmax_scale * a.kv_scale * 1.4426950408889634f;
        float* part_o = reinterpret_cast<float*>(a.ws + a.lay.off_part_o);
        float* part_lse = reinterpret_cast<float*>(a.ws + a.lay.off_part_lse);
        const int32_t* seg_base = reinterpret_cast<const int32_t*>(a.ws + a.lay.off_seg_base);
        const int row = tq * kHeads + h;

        auto epilogue = [&](const MlaTile& g) {
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
            // causal bound of this query token in rank r's local positions
            const int r = (int)(t.u % a.N), b = (int)(t.u / a.N);
            const int64_t L = a.seq_lens[b];
            const int64_t bound = local_len(L - a.Tq + tq + 1, r, a.N, a.I);
            const int64_t p0 = t.chunk * kChunk;
            const uint32_t sbase = tm + 256 + 128 * sb + lane_off;
            const int ncols = 64 * t.n_ch;
            // columns [0, lim) are visible to this query token
            const int64_t lim64 = bound - p0;
            const int lim = lim64 <= 0 ? 0 : (lim64 >= ncols ? ncols : (int)lim64);
            float sv[128];
            uint32_t rr[32];
#pragma unroll
            for (int cch = 0; cch < 4; ++cch) {
                if (cch * 32 < ncols) {
                    tmem_ld32(sbase + 32 * cch, rr);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) sv[32 * cch + k] = __uint_as_float(rr[k]);
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) sv[32 * cch + k] = 0.f;
                }
            }
            float mraw = -INFINITY;
            if (lim == 128) {
#pragma unroll
                for (int j = 0; j < 128; ++j) mraw = fmaxf(mraw, sv[j]);
            } else {
#pragma unroll
                for (int j = 0; j < 128; ++j) mraw = (j < lim) ? fmaxf(mraw, sv[j]) : mraw;
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
            float lsum = 0.f;
            uint32_t pk[32];
#pragma unroll
            for (int cch = 0; cch < 2; ++cch) {
                if (cch * 64 < ncols) {
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const int j = 64 * cch + 2 * k;
                        float p_lo = ex2_approx(fmaf(sv[j], sl2, nmu));
                        float p_hi = ex2_approx(fmaf(sv[j + 1], sl2, nmu));
                        if (lim < 128) {
                            p_lo = (j < lim) ? p_lo : 0.f;
                            p_hi = (j + 1 < lim) ? p_hi : 0.f;
                        }
                        lsum += p_lo + p_hi;
                        pk[k] = pack16(p_lo, p_hi, FP8);
                    }
                    tmem_st32(tm + 256 + 128 * sb + lane_off + 32 * cch, pk);
                }
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
    } else if (FP8) {
        // ------------------------------------------------------------ fp8 -> fp16 converters
        const int ct = threadIdx.x - 32 * C::kWarpConv;  // 0..127
        TileCursor cur;
        cur.init(us, c0, c1, u0, a.N, a.partial_mode);
        Ring stg, ring;
        stg.n = C::kStage;
        ring.n = C::kRing;
        uint32_t qf_phase = 0;
        bool alive = true;
        MlaTile prev{}, t{};
        int ti = 0;
        auto convert_sub = [&](int n_ch) {
            if (!mbar_wait(&sh.sfull[stg.slot], stg.phase)) { alive = false; return; }
            if (!mbar_wait(&sh.empty[ring.slot], ring.phase ^ 1u)) { alive = false; return; }
            const int rows = 64 * n_ch;
            if (ct < rows) {
                const uint4* src = reinterpret_cast<const uint4*>(sStage + stg.slot * C::kStageBytes + ct * 64);
                uint8_t* dst = sRing + ring.slot * kSubBytes + ct * 128;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const uint4 v = src[q4];
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
                    uint32_t o[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t lo16 = wv[k] & 0xFFFFu, hi16 = wv[k] >> 16, h0, h1;
                        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h0) : "h"((unsigned short)lo16));
                        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h1) : "h"((unsigned short)hi16));
                        o[2 * k] = h0;
                        o[2 * k + 1] = h1;
                    }
                    // 16 fp16 = two 16-byte chunks: logical chunks 2 q4 and 2 q4 + 1
                    const int ch0 = 2 * q4, ch1 = 2 * q4 + 1;
                    *reinterpret_cast<uint4*>(dst + ((ch0 ^ (ct & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                    *reinterpret_cast<uint4*>(dst + ((ch1 ^ (ct & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sh.full[ring.slot]);
                mbar_arrive(&sh.sempty[stg.slot]);
            }
            stg.advance();
            ring.advance();
        };
        for (;;) {
            const bool more = cur.next(t);
            if (more) {
                if (t.first) {
                    if (!mbar_wait(sh.q_full, qf_phase)) { alive = false; break; }
                    qf_phase ^= 1u;
                    // Q bf16 -> fp16 in place (each thread a contiguous 1152-byte slice)
                    uint4* qs = reinterpret_cast<uint4*>(sQ + ct * (kQBytes / 128));
#pragma unroll 4
                    for (int i = 0; i < (kQBytes / 128) / 16; ++i) {
                        uint4 v = qs[i];
                        uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float f0 = __uint_as_float(wv[k] << 16), f1 = __uint_as_float(wv[k] & 0xFFFF0000u);
                            __half2 hh = __floats2half2_rn(f0, f1);
                            wv[k] = *reinterpret_cast<uint32_t*>(&hh);
                        }
                        qs[i] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sh.q_conv);
                }
                for (int s = 0; s < kKSub && alive; ++s) convert_sub(t.n_ch);
            }
            if (ti > 0)
                for (int j = 0; j < kVSub && alive; ++j) convert_sub(prev.n_ch);
            if (!more || !alive) break;
            prev = t;
            ++ti;
        }
        if (!alive && lane == 0) raise_err(err, DCP_DEV_ERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::kWarpMma) tmem_dealloc(tm, 512);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
                 uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool FP8>
cudaError_t launch_t(const AttnArgs& a, cudaStream_t s) {
    using C = MlaCfg<FP8>;
    CUtensorMap tq, tkv;
    if (!make_map_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, kDk, (uint64_t)a.B * a.Tq * kHeads, kDk * 2, 64,
                     128, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const uint64_t rows = (uint64_t)a.num_blocks * a.bs;
    if (FP8) {
        if (!make_map_2d(&tkv, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.k_pool, kDk, rows, kDk, 64, kChunk,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else {
        if (!make_map_2d(&tkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.k_pool, kDk, rows, kDk * 2, 64, kChunk,
                         CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(mla_tc_kernel<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(2 * a.W), (unsigned)a.Tq);
    mla_tc_kernel<FP8><<<grid, C::kThreads, C::kSmem, s>>>(a, tq, tkv);
    return cudaGetLastError();
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
    if (kv_dtype == DCP_FP8_E4M3) return launch_t<true>(a, s);
    return launch_t<false>(a, s);
}

}  // namespace dcp

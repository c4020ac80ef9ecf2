// Causal prefill of PCP-gathered query rows against one DCP rank's shard on
// tcgen05 tensor cores (kind::f16, bf16 in, fp32 accumulators in TMEM).
//
// What it computes is that of attn_prefill.cu ("Breaking the Long-Sequence
// Inference Bottleneck ...", section 5, AllGather Q path; "vLLM DCP and
// PCP", Deep Dive 6): every query row, at its own global position p, against
// rank r's local positions below local_len(p + 1, r), as a normalised
// partial with its LSE.  Here for D = 128 as a dense contraction:
//
//   CTA = 128 rows (128 / G query tokens x the G heads of one KV head) of one
//   (request, KV head, rank); M = 128.  Q stays in shared memory (SW128,
//   K-major).  K and V of 128 local tokens per tile go through a 3-stage
//   ring.  When block_size is a multiple of 64, every 64 tokens of a tile lie
//   in one page and come in as TMA boxes of [64 tokens x 64 columns] (SW128,
//   8 boxes per tile, dealt over the producer warps); otherwise producer
//   warps copy them with 16-byte cp.async into the same layout (zeros past
//   the rows' furthest position) and publish each stage after a proxy fence.
//   (Through TMA a tile's tokens past the shard's end come from the cache as
//   stored; their probabilities are exactly 0, so they must hold finite
//   values, as a zero-initialised pool does.)
//   S = Q K^T (N = 128) lands in one of two TMEM buffers; the softmax warps
//   (thread = row = TMEM lane) mask each row at its own bound, write P back
//   as bf16 pairs over the buffer's first columns, and the P.V MMA reads it
//   from TMEM (A operand) against V as an MN-major operand (N = 128 values).
//   O (128 x 128 fp32) stays in TMEM; the reference max is lazy (O is
//   rescaled only when a row's max grows by more than 2^8).
//
// Warps: 0-2 producers, 3 TMEM owner and MMA issuer (one lane), 4-7 and 8-11
// softmax (two warpgroups over the same 128 rows, 64 columns of each tile
// each: the exponentials of a tile are spread over twice the warps; the two
// half-row maxima meet in shared memory, and each group writes P over its own
// S columns and rescales / stores its own half of O).
// TMEM: O [0, 128), S buffers [128, 256) and [256, 384).  Every wait is
// bounded; a timeout raises DCP_DEV_ERR_TIMEOUT and the role stops.
#include "dcp_internal.cuh"
#include "mla_common.cuh"
#include "sm100_prims.cuh"

namespace dcp {
namespace {

using namespace sm100;

constexpr int kD = 128;
constexpr int kRows = 128;                   // M
constexpr int kKeys = 128;                   // local tokens per tile (N of QK)
constexpr int kSub = 128 * 64 * 2;           // [128 rows x 64 bf16] SW128 sub-tile: 16 KB
constexpr int kQBytes = 2 * kSub;            // 32 KB
constexpr int kStageBytes = 4 * kSub;        // K (2 sub-tiles) + V (2 sub-tiles): 64 KB
constexpr int kStages = 3;
constexpr int kProd = 3;                     // producer warps
constexpr int kProdThreads = 32 * kProd;
constexpr int kWarpMma = kProd;
constexpr int kWarpSoftmax = kWarpMma + 1;
constexpr int kSoftGroups = 2;  // softmax warpgroups, kKeys / kSoftGroups columns each (4: slower)
constexpr int kGroupCols = kKeys / kSoftGroups;
constexpr int kSoftThreads = 128 * kSoftGroups;
constexpr int kThreads = 32 * kWarpSoftmax + kSoftThreads;
constexpr float kRescaleLog2 = 8.f;
constexpr int kMaxPages = 32;                // pages a tile may touch: kKeys / bs + 2 <= 32 needs bs >= 8

constexpr int kOffQ = 0;
constexpr int kOffRing = kQBytes;
constexpr int kOffBar = kOffRing + kStages * kStageBytes;
constexpr int kNumBars = 2 * kStages + 1 + 2 + 2 + 1 + 1;
constexpr int kOffKv = kOffBar + kNumBars * 8 + 16;     // after the barriers and the TMEM address
constexpr int kOffBlk = kOffKv + 16;                    // [kProd][32] block ids of the producers' current tile
constexpr int kOffXch = kOffBlk + kProd * 32 * 4;       // [2][kSoftGroups][kRows] floats
constexpr int kSmem = kOffXch + 2 * kSoftGroups * kRows * 4;
static_assert(kSmem <= 232448, "shared memory");

struct Bars {
    uint64_t *full, *empty, *q_full, *s_full, *p_full, *o_done, *drain;
    uint32_t* tmem_slot;
};

__device__ __forceinline__ Bars carve(uint8_t* base) {
    uint64_t* b = reinterpret_cast<uint64_t*>(base + kOffBar);
    Bars s;
    s.full = b; b += kStages;
    s.empty = b; b += kStages;
    s.q_full = b++;
    s.s_full = b; b += 2;
    s.p_full = b; b += 2;
    s.o_done = b++;
    s.drain = b++;
    s.tmem_slot = reinterpret_cast<uint32_t*>(b);
    return s;
}

// byte offset of 16-byte chunk c16 (0..15) of row `row` in a [128 x 128 bf16]
// tile stored as two SW128 sub-tiles of 64 columns
__device__ __forceinline__ uint32_t sw128(int row, int c16) {
    const int c = c16 & 7;
    return (uint32_t)((c16 >> 3) * kSub + row * 128 + ((c ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, bool valid) {
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, int use_tma) {
    // all of the kernel's shared memory is dynamic, so it starts on the
    // 1024-byte boundary the swizzled layouts need (checked below)
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* sQ = smem + kOffQ;
    uint8_t* sRing = smem + kOffRing;
    const Bars sh = carve(smem);
    int& s_kv = *reinterpret_cast<int*>(smem + kOffKv);
    int32_t(*s_blk)[32] = reinterpret_cast<int32_t(*)[32]>(smem + kOffBlk);
    // the groups' row maxima (then row sums), double-buffered by tile parity:
    // a buffer is rewritten only after the next exchange barrier, which every
    // thread passes after reading it
    float(*s_xch2)[kSoftGroups][kRows] = reinterpret_cast<float(*)[kSoftGroups][kRows]>(smem + kOffXch);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    const int64_t nrt = ((int64_t)a.Tq * a.G + kRows - 1) / kRows;
    const int64_t unit = blockIdx.x / nrt;
    const int row0 = (int)(blockIdx.x % nrt) * kRows;
    const int r = (int)(unit % a.N);
    const int64_t bk = unit / a.N;
    const int b = (int)(bk / a.Hkv), kvh = (int)(bk % a.Hkv);
    uint32_t* err = &reinterpret_cast<WsHeader*>(a.ws)->err;
    if ((smem_u32(smem) & 1023u) != 0) {
        if (threadIdx.x == 0) raise_err(err, DCP_DEV_ERR_TIMEOUT);
        return;
    }

    // rank r's local length of request b
    const int32_t L = a.seq_lens[b];
    int32_t len = 0;
    if (L > 0) {
        const uint32_t expect = local_len32((uint32_t)L, r, a.N, a.I);
        const int32_t given = a.local_lens[(int64_t)r * a.B + b];
        if (given != (int32_t)expect && threadIdx.x == 0) raise_err(err, DCP_DEV_ERR_STALE);
        len = given < 0 ? 0 : ((uint32_t)given < expect ? given : (int32_t)expect);
        if (((int64_t)len + a.bs - 1) / a.bs > a.max_blocks) {
            if (threadIdx.x == 0) raise_err(err, DCP_DEV_ERR_TABLE);
            len = a.max_blocks * a.bs;
        }
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sh.full[i], use_tma ? 1 : kProdThreads);  // TMA: the expect-tx arrive; else every copier
            mbar_init(&sh.empty[i], 1);
        }
        mbar_init(sh.q_full, kSoftThreads);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.s_full[i], 1);
            mbar_init(&sh.p_full[i], 4 * kSoftGroups);
        }
        mbar_init(sh.o_done, 1);
        mbar_init(sh.drain, 1);
        fence_mbar_init();
        s_kv = 0;
    }
    if (warp == kWarpMma) {
        tmem_alloc(sh.tmem_slot, 512);
        tmem_relinquish();
    }
    __syncthreads();  // barriers initialised, s_kv zeroed

    // the softmax threads own the rows: position, causal bound, query row
    const int hs = threadIdx.x - 32 * kWarpSoftmax;  // softmax thread
    const int h = hs & (kRows - 1);                  // row = TMEM lane
    const int grp = hs >> 7;                         // softmax group: columns [64 grp, 64 grp + 64)
    int t_row = 0;
    int32_t bound = 0;
    if (warp >= kWarpSoftmax) {
        const int row = row0 + h;
        t_row = row / a.G;
        if (t_row < a.Tq) {
            const int32_t p = a.q_pos[(int64_t)b * a.Tq + t_row];
            if (p >= L) raise_err(err, DCP_DEV_ERR_TOKEN);
            else if (p >= 0) bound = min(len, (int32_t)local_len32((uint32_t)p + 1u, r, a.N, a.I));
        }
        atomicMax(&s_kv, bound);
        // the query row into Q (SW128, K-major); rows past the request are zero
        const uint4* src = nullptr;
        if (t_row < a.Tq) {
            const int gq = row % a.G;
            src = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.q) +
                                                 (((int64_t)b * a.Tq + t_row) * a.Hq + (int64_t)kvh * a.G + gq) * kD);
        }
#pragma unroll
        for (int c = 0; c < 16 / kSoftGroups; ++c) {
            const int c16 = (16 / kSoftGroups) * grp + c;  // each group stores its share of the row
            *reinterpret_cast<uint4*>(sQ + sw128(h, c16)) = src ? src[c16] : make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        mbar_arrive(sh.q_full);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *sh.tmem_slot;
    const int kv = s_kv;
    const int ntiles = (kv + kKeys - 1) / kKeys;

    if (warp < kProd && use_tma) {
        // ------------------------------------------------------------ TMA producers
        // Box j of a tile (j = 4 kv + 2 g + h: K or V, token group g of 64,
        // column half h) goes out from warp j % 3.  A group past the rows'
        // furthest position re-reads group 0 (finite values, probability 0).
        if (lane == 0) {
            const int32_t* bt = a.block_tables + ((int64_t)r * a.B + b) * a.max_blocks;
            bool alive = true, bad = false;
            auto group_row = [&](int t, int g) -> int {  // first pool row of token group g of tile t
                int lp0 = t * kKeys + 64 * g;
                if (lp0 >= kv) lp0 = t * kKeys;
                int32_t blk = bt[lp0 / a.bs];
                if (blk < 0 || blk >= a.num_blocks) {
                    bad = true;
                    blk = 0;
                }
                return (int)(((int64_t)blk * a.Hkv + kvh) * a.bs + lp0 % a.bs);
            };
            int nrow0 = 0, nrow1 = 0;
            if (ntiles > 0) { nrow0 = group_row(0, 0); nrow1 = group_row(0, 1); }
            for (int t = 0; t < ntiles && alive; ++t) {
                const int s = t % kStages;
                const int row_g0 = nrow0, row_g1 = nrow1;
                if (t + 1 < ntiles) { nrow0 = group_row(t + 1, 0); nrow1 = group_row(t + 1, 1); }
                bool waited = false;
                for (int j = warp; j < 8; j += kProd) {
                    if (!waited) {
                        if (!mbar_wait_sleep(&sh.empty[s], ((t / kStages) & 1) ^ 1u)) { alive = false; break; }
                        waited = true;
                    }
                    if (j == 0) mbar_arrive_expect_tx(&sh.full[s], (uint32_t)kStageBytes);
                    const int kvsel = j >> 2, g = (j >> 1) & 1, h = j & 1;
                    uint8_t* dst = sRing + (size_t)s * kStageBytes + kvsel * 2 * kSub + h * kSub + g * 8192;
                    if (kvsel)
                        tma_load_2d(dst, &tmap_v, 64 * h, g ? row_g1 : row_g0, &sh.full[s]);
                    else
                        tma_load_2d(dst, &tmap_k, 64 * h, g ? row_g1 : row_g0, &sh.full[s]);
                }
            }
            if (bad) raise_err(err, DCP_DEV_ERR_BLOCK_ID);
            if (!alive) raise_err(err, DCP_DEV_ERR_TIMEOUT);
            // on a timeout, give this warp's TMA copies time to land before the
            // CTA exits (a copy completes within microseconds)
            if (!alive) tma_drain_pause();
        }
    } else if (warp < kProd) {
        // ------------------------------------------------------------ cp.async producers
        // Thread pt copies the fixed 16-byte column c16 = pt % 16 of rows
        // pt / 16 + 6 i of K and V.  A tile's block ids (at most kKeys / bs + 2
        // pages) sit in a per-warp table, loaded one tile ahead so that no
        // copy waits on a block-table read.
        const int pt = threadIdx.x;  // 0 .. 95
        const int c16 = pt & 15, rbeg = pt >> 4;
        constexpr int kRowStep = kProdThreads / 16;
        const int32_t* bt = a.block_tables + ((int64_t)r * a.B + b) * a.max_blocks;
        const uint8_t* kp = reinterpret_cast<const uint8_t*>(a.k_pool) + c16 * 16;
        const uint8_t* vp = reinterpret_cast<const uint8_t*>(a.v_pool) + c16 * 16;
        const uint32_t ring = smem_u32(sRing);
        const bool pow2 = (a.bs & (a.bs - 1)) == 0;
        const int bsh = __ffs(a.bs) - 1;
        auto page_of = [&](int lp) -> int { return pow2 ? lp >> bsh : lp / a.bs; };
        auto page_id = [&](int t) -> int32_t {  // this lane's page of tile t
            const int pg = page_of(t * kKeys) + lane;
            return (lane < kMaxPages && pg * a.bs < kv) ? bt[pg] : -1;
        };
        bool alive = true, bad = false;
        int32_t nxt = ntiles > 0 ? page_id(0) : -1;
        for (int t = 0; t < ntiles && alive; ++t) {
            const int s = t % kStages;
            if (lane == 0 && !mbar_wait_sleep(&sh.empty[s], ((t / kStages) & 1) ^ 1u)) alive = false;
            alive = __shfl_sync(0xffffffffu, alive ? 1 : 0, 0) != 0;
            if (!alive) break;
            s_blk[warp][lane] = nxt;
            __syncwarp();
            if (t + 1 < ntiles) nxt = page_id(t + 1);
            const int pg0 = page_of(t * kKeys);
            const uint32_t st = ring + (uint32_t)s * kStageBytes;
            for (int row = rbeg; row < kKeys; row += kRowStep) {
                const int lp = t * kKeys + row;
                bool valid = lp < kv;
                int64_t off = 0;
                if (valid) {
                    const int32_t blk = s_blk[warp][page_of(lp) - pg0];
                    if (blk < 0 || blk >= a.num_blocks) {
                        bad = true;
                        valid = false;
                    } else {
                        const int in_pg = pow2 ? (lp & (a.bs - 1)) : lp % a.bs;
                        off = (((int64_t)blk * a.Hkv + kvh) * a.bs + in_pg) * (kD * 2);
                    }
                }
                const uint32_t so = sw128(row, c16);
                cp_async16_zfill(st + so, kp + off, valid);
                cp_async16_zfill(st + 2 * kSub + so, vp + off, valid);
            }
            cp_async_commit();
            __syncwarp();  // the table is rewritten for the next tile
            if (t > 0) {
                cp_async_wait<1>();
                fence_proxy_async_smem();
                mbar_arrive(&sh.full[(t - 1) % kStages]);
            }
        }
        cp_async_wait<0>();
        if (alive && ntiles > 0) {
            fence_proxy_async_smem();
            mbar_arrive(&sh.full[(ntiles - 1) % kStages]);
        }
        if (bad) raise_err(err, DCP_DEV_ERR_BLOCK_ID);
        if (!alive) raise_err(err, DCP_DEV_ERR_TIMEOUT);
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && ntiles > 0) {
            bool alive = true;
            const uint32_t idesc_qk = idesc_f16(1, kRows, kKeys, 0, 0);
            const uint32_t idesc_pv = idesc_f16(1, kRows, kD, 0, 1);
            const uint64_t dq = smem_desc(smem_u32(sQ), 16, 1024, kLayoutSW128);
            const uint64_t dring = smem_desc(smem_u32(sRing), 16, 1024, kLayoutSW128);
            // values: MN-major, the two 64-column halves one sub-tile apart
            const uint64_t dvr = smem_desc(smem_u32(sRing + 2 * kSub), kSub, 1024, kLayoutSW128);
            constexpr uint32_t kSubDesc = kSub >> 4, kStageDesc = kStageBytes >> 4;
            if (!mbar_wait_sleep(sh.q_full, 0)) alive = false;
            auto pv = [&](int t) -> bool {
                const int sb = t & 1;
                if (!mbar_wait_sleep(&sh.p_full[sb], (t >> 1) & 1)) return false;
                tc_fence_after();
                const uint32_t pa = tm + 128 + 128 * sb;
                const uint64_t vd = dvr + (uint64_t)(t % kStages) * kStageDesc;
#pragma unroll 1
                for (int kk = 0; kk < kKeys / 16; ++kk)  // group g's P: the first half of its S columns
                    mma_ts(tm, pa + kGroupCols * (kk / (kGroupCols / 16)) + 8 * (kk % (kGroupCols / 16)),
                           vd + 128 * kk, idesc_pv,
                           (t > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&sh.empty[t % kStages]);
                mma_commit(sh.o_done);
                return true;
            };
            for (int t = 0; t < ntiles && alive; ++t) {
                const int s = t % kStages;
                if (!mbar_wait_sleep(&sh.full[s], (t / kStages) & 1)) { alive = false; break; }
                tc_fence_after();
                const uint32_t d = tm + 128 + 128 * (t & 1);
                const uint64_t kd = dring + (uint64_t)s * kStageDesc;
#pragma unroll 1
                for (int kc = 0; kc < 2; ++kc)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_ss(d, dq + kc * kSubDesc + 2 * kk, kd + kc * kSubDesc + 2 * kk, idesc_qk,
                               (kc | kk) != 0 ? 1u : 0u);
                mma_commit(&sh.s_full[t & 1]);
                if (t > 0 && !pv(t - 1)) { alive = false; break; }
            }
            if (alive && !pv(ntiles - 1)) alive = false;
            if (!alive) raise_err(err, DCP_DEV_ERR_TIMEOUT);
            // every MMA this thread issued has completed before the CTA releases
            // tensor memory (also when a role stopped early on a timeout)
            mma_commit(sh.drain);
            mbar_wait_sleep(sh.drain, 0);
        }
    } else {
        // ------------------------------------------------------------ softmax warpgroups
        const int quarter = warp & 3;
        const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
        const float sl2 = a.softmax_scale * 1.4426950408889634f;
        const int c0 = kGroupCols * grp;  // this group's columns of a tile
        float m_ref = -INFINITY, l = 0.f;
        bool alive = true;
        // barrier over the two groups that also ANDs a flag: both groups leave
        // a loop together (a bar.sync cannot time out)
        auto both = [&](int id, bool ok) -> bool {
            uint32_t in = ok ? 1u : 0u, out;
            asm volatile("{\n.reg .pred pi, po;\nsetp.ne.u32 pi, %1, 0;\nbar.red.and.pred po, %2, %3, pi;\n"
                         "selp.u32 %0, 1, 0, po;\n}"
                         : "=r"(out)
                         : "r"(in), "r"(id), "r"(kSoftThreads)
                         : "memory");
            return out != 0;
        };
        bool ok_prev = true;
        for (int t = 0; t < ntiles; ++t) {
            const int sb = t & 1;
            const bool ok = __all_sync(0xffffffffu, mbar_wait(&sh.s_full[sb], (t >> 1) & 1));
            tc_fence_after();
            const uint32_t sbase = tm + 128 + 128 * sb + lane_off + c0;
            // columns [0, lim) of this group's 64 are visible to the row
            const int lim = max(0, min(kGroupCols, bound - t * kKeys - c0));
            // the group's 64 scores stay in registers for both passes; the
            // columns past the row's bound (diagonal tiles only) become -inf
            static_assert(kGroupCols == 64, "two 32-column loads per group");
            uint32_t sv0[32], sv1[32];
            tmem_ld32(sbase, sv0);
            tmem_ld32(sbase + 32, sv1);
            tmem_wait_ld();
#define SV(k) ((k) < 32 ? sv0[(k) & 31] : sv1[(k) & 31])
            if (lim < kGroupCols) {
#pragma unroll
                for (int k = 0; k < kGroupCols; ++k)
                    if (k >= lim) SV(k) = 0xff800000u;
            }
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int k = 0; k < kGroupCols; k += 2)
                m4[(k >> 1) & 3] = fmax3(m4[(k >> 1) & 3], __uint_as_float(SV(k)), __uint_as_float(SV(k + 1)));
            const float mraw = fmax3(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
            float(*s_xch)[kRows] = s_xch2[t & 1];
            s_xch[grp][h] = (lim > 0) ? mraw * sl2 : -INFINITY;
            // the exchange barrier also carries the previous tile's o_done outcome
            if (!both(1, ok && ok_prev)) { alive = false; break; }
            float mx = s_xch[0][h];  // the row's max over the tile (base 2)
#pragma unroll
            for (int g = 1; g < kSoftGroups; ++g) mx = fmaxf(mx, s_xch[g][h]);
            // lazy reference max (both groups take the same decision)
            float corr = 1.f;
            bool rescale_o = false;
            if (mx > -INFINITY) {
                if (m_ref == -INFINITY) {
                    m_ref = mx;  // first visible tokens of the row: O holds zeros
                    corr = 0.f;
                } else if (mx > m_ref + kRescaleLog2) {
                    corr = ex2_approx(m_ref - mx);
                    m_ref = mx;
                    rescale_o = true;
                }
            }
            const float nmu = (m_ref == -INFINITY) ? 0.f : -m_ref;
            // P as bf16 pairs over the group's first 32 columns.  The pass is
            // bound by instruction issue, not by the SFU (moving 1/8 or 1/4 of
            // the exponentials to an FMA-pipe polynomial made it slower): scale,
            // shift and sum go two columns per instruction (fp32x2), and the
            // scores come from registers
            uint64_t acc = pair_f32(0.f, 0.f);
            const uint64_t sc = pair_f32(sl2, sl2), mu = pair_f32(nmu, nmu);
#pragma unroll
            for (int q = 0; q < kGroupCols / 16; ++q) {
                uint32_t pk[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    float x0, x1;
                    unpair_f32(fma_f32x2(pair_f32(__uint_as_float(SV(16 * q + 2 * k)),
                                                  __uint_as_float(SV(16 * q + 2 * k + 1))),
                                         sc, mu),
                               x0, x1);
                    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                    acc = add_f32x2(acc, pair_f32(p0, p1));
                    pk[k] = pack_bf16(p0, p1);
                }
                tmem_st8(sbase + 8 * q, pk);
            }
#undef SV
            float ls0, ls1;
            unpair_f32(acc, ls0, ls1);
            const float lsum = ls0 + ls1;
            l = (corr == 0.f ? 0.f : l * corr) + lsum;
            // P.V of the previous tile must be complete before O is touched
            // (the outcome joins the next exchange barrier's flag)
            if (t > 0) ok_prev = __all_sync(0xffffffffu, mbar_wait(sh.o_done, (t - 1) & 1));
            tc_fence_after();
            if (__any_sync(0xffffffffu, rescale_o)) {
                const float f = rescale_o ? corr : 1.f;
                uint32_t ov[32];
#pragma unroll 1
                for (int i = 0; i < kGroupCols / 32; ++i) {
                    tmem_ld32(tm + lane_off + c0 + 32 * i, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * f);
                    tmem_st32(tm + lane_off + c0 + 32 * i, ov);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.p_full[sb]);
        }
        // epilogue: the last P.V, the row's total sum, then this group's half of
        // the row's normalised partial (and, group 0, the LSE)
        bool ok3 = alive;
        if (alive && ntiles > 0) ok3 = __all_sync(0xffffffffu, mbar_wait(sh.o_done, (ntiles - 1) & 1));
        float(*s_xch)[kRows] = s_xch2[ntiles & 1];
        s_xch[grp][h] = l;
        const bool read_o = both(1, ok3 && ok_prev) && ntiles > 0;  // uniform across both groups
        tc_fence_after();
        float lt = s_xch[0][h];
#pragma unroll
        for (int g = 1; g < kSoftGroups; ++g) lt += s_xch[g][h];
        // every lane reads its TMEM lane (rows past the request too: the load
        // is warp-aligned); only the request's rows are written
        const bool row_ok = t_row < a.Tq;
        const bool has = read_o && lt > 0.f;
        const float inv = has ? 1.f / lt : 0.f;
        int64_t prow = 0;
        if (row_ok) {
            const int gq = (row0 + h) % a.G;
            prow = (((int64_t)r * a.B + b) * a.Tq + t_row) * a.Hq + (int64_t)kvh * a.G + gq;
        }
        float* dst = a.out_partial + prow * kD + c0;
        uint32_t ov[32];
#pragma unroll 1
        for (int i = 0; i < kGroupCols / 32; ++i) {
            if (read_o) {
                tmem_ld32(tm + lane_off + c0 + 32 * i, ov);
                tmem_wait_ld();
            }
            if (row_ok) {
#pragma unroll
                for (int k = 0; k < 32; k += 4)
                    *reinterpret_cast<float4*>(dst + 32 * i + k) =
                        has ? make_float4(__uint_as_float(ov[k]) * inv, __uint_as_float(ov[k + 1]) * inv,
                                          __uint_as_float(ov[k + 2]) * inv, __uint_as_float(ov[k + 3]) * inv)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        if (row_ok && grp == 0) a.lse_partial[prow] = has ? (m_ref + log2f(lt)) * 0.6931471805599453f : -INFINITY;
        if (!read_o && ntiles > 0 && lane == 0) raise_err(err, DCP_DEV_ERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc(tm, 512);
}

}  // namespace

bool prefill_tc_supported(const PrefillArgs& a) {
    return a.D == kD && a.G >= 1 && kRows % a.G == 0 && a.bs >= 8;
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    CUtensorMap tk, tv;
    memset(&tk, 0, sizeof tk);
    memset(&tv, 0, sizeof tv);
    const int use_tma = a.bs % 64 == 0 ? 1 : 0;
    if (use_tma) {
        // the pools as [num_blocks * Hkv * block_size rows x 128 columns], boxes of 64 x 64
        const uint64_t rows = (uint64_t)a.num_blocks * a.Hkv * a.bs;
        if (!mla::make_map_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.k_pool, kD, rows, kD * 2, 64, 64,
                              CU_TENSOR_MAP_SWIZZLE_128B) ||
            !mla::make_map_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.v_pool, kD, rows, kD * 2, 64, 64,
                              CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    const int64_t ctas = ((int64_t)a.Tq * a.G + kRows - 1) / kRows * ((int64_t)a.B * a.Hkv * a.N);
    return launch_pdl(prefill_tc_kernel, dim3((unsigned)ctas), dim3(kThreads), kSmem, s, a, tk, tv, use_tma);
}

}  // namespace dcp

// GQA split-KV decode attention, bf16, with the exact LSE merge fused in.
//
// "vLLM DCP and PCP", Deep Dive 6: every virtual rank's partial
// (o_i, L_i) over its own KV shard, merged by LSE weights.  "Breaking the
// Long-Sequence Inference Bottleneck ...", section 3 (GQA path): many query
// heads share one KV head, so the query heads of a KV group (x the query
// tokens) are packed as the rows of one 16-row MMA tile and every KV byte read
// serves all of them.
//
// Decode at this shape is HBM-bound (~4 FLOP per KV byte), so the kernel is
// built around the page stream:
//  * worker = one warp; the chunks (16 local tokens of one rank / request /
//    KV head = 2 x 16 x D bf16, contiguous inside one physical block) of all
//    units are dealt to workers as equal contiguous ranges;
//  * each warp keeps NST chunks in flight with 16-byte cp.async.cg copies into
//    an XOR-swizzled smem ring (conflict-free ldmatrix), under an L2
//    evict-first policy: the pages are read once, and streaming them through
//    L2 at the default priority evicted the plan, block tables and partials
//    that the kernel reads again (6 us of a 32 x 8K-token step);
//  * S = Q K^T and O += P V on mma.sync.m16n8k16 (bf16 in, fp32 accumulate),
//    online softmax in base 2 on the accumulator fragments;
//  * a segment's result is either final (the group lies in one worker) or a
//    partial slot; the last arriving segment of a group merges the group's
//    partials (atomic counter, no waiting).
#include "dcp_internal.cuh"
#include "mma_sync.cuh"
#include "sm100_prims.cuh"

namespace dcp {
namespace {

using namespace mma;

constexpr int kWarps = 4;
constexpr int kChunk = 16;

template <int D, int NST>
struct Cfg {
    static constexpr int kRowBytes = D * 2;                 // one token row of K (or V)
    static constexpr int kTileBytes = kChunk * kRowBytes;   // 16 rows
    static constexpr int kStageBytes = 2 * kTileBytes;      // K + V
    static constexpr int kWarpBytes = NST * kStageBytes;
    static constexpr int kSmem = kWarps * kWarpBytes;
    static constexpr int kPieces = kTileBytes / 16;         // 16-byte pieces per tile
    static constexpr int kKSteps = D / 16;
    static constexpr int kNT = D / 8;                       // output n-tiles
};

template <int D, int NST>
__global__ void __launch_bounds__(kWarps * 32) gqa_mma_kernel(AttnArgs a) {
    using C = Cfg<D, NST>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t w = (int64_t)blockIdx.x * kWarps + warp;
    pdl_wait();  // the plan
    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(a.ws);
    // a plan made ahead holds where this worker starts: loaded beside the
    // header (it is used only once the header says the plan is this call's)
    WorkerStart ws0{0, 0, 0, 0};
    if (a.worker_starts && w < a.W) ws0 = reinterpret_cast<const WorkerStart*>(a.ws + a.lay.off_wfirst)[w];
    const int64_t P = hdr->total_chunks;
    if (hdr->plan_key != a.plan_key) {  // the workspace holds a plan for other arguments
        if (threadIdx.x == 0) raise_err(&reinterpret_cast<WsHeader*>(a.ws)->err, DCP_DEV_ERR_PLAN);
        return;
    }
    // groups that own no chunk: zeros and -inf, spread over the warps
    for (int64_t e = w; e < (int64_t)hdr->n_empty; e += (int64_t)gridDim.x * kWarps)
        write_empty_group(a, reinterpret_cast<const int32_t*>(a.ws + a.lay.off_empty)[e], lane);
    if (P == 0) return;
    const int64_t We = P < a.W ? P : a.W;  // workers in play: each owns >= 1 chunk
    if (w >= We) return;
    const int64_t c0 = worker_begin(w, We, P), c1 = worker_begin(w + 1, We, P);
    if (c0 >= c1) return;
    const int64_t* unit_start = reinterpret_cast<const int64_t*>(a.ws + a.lay.off_units);
    const int32_t* seg_base = reinterpret_cast<const int32_t*>(a.ws + a.lay.off_seg_base);
    uint32_t* counters = reinterpret_cast<uint32_t*>(a.ws + a.lay.off_counters);
    float* part_o = reinterpret_cast<float*>(a.ws + a.lay.off_part_o);
    float* part_lse = reinterpret_cast<float*>(a.ws + a.lay.off_part_lse);
    uint32_t* err = &reinterpret_cast<WsHeader*>(a.ws)->err;
    uint8_t* wsm = smem + warp * C::kWarpBytes;
    const uint32_t wsm_u32 = smem_u32(wsm);
    const int per_group = a.partial_mode ? 1 : a.N;
    const __nv_bfloat16* kp = reinterpret_cast<const __nv_bfloat16*>(a.k_pool);
    const __nv_bfloat16* vp = reinterpret_cast<const __nv_bfloat16*>(a.v_pool);

    // first unit: from a plan made ahead, else the last u with unit_start[u] <= c0
    int64_t lo = ws0.u0;
    if (!a.worker_starts) {
        int64_t hi = a.U - 1;
        while (lo < hi) {
            const int64_t mid = (lo + hi + 1) >> 1;
            if (unit_start[mid] <= c0) lo = mid; else hi = mid - 1;
        }
        ws0.ustart = unit_start[lo];
        ws0.uend = unit_start[lo + 1];
    }
    int64_t u_load = lo, u = lo;
    // producer-side cache of the current unit (divisions only when the unit changes)
    int64_t ld_start = ws0.ustart, ld_end = ws0.uend;
    const int32_t* ld_bt = nullptr;
    int ld_kvh = 0;
    auto ld_unit = [&]() {
        const int r = (int)(u_load % a.N);
        const int64_t bk = u_load / a.N;
        const int b = (int)(bk / a.Hkv);
        ld_kvh = (int)(bk % a.Hkv);
        ld_bt = a.block_tables + ((int64_t)r * a.B + b) * a.max_blocks;
    };
    ld_unit();

    uint64_t l2_first;  // the pages are read once: L2 evicts them first
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(l2_first));
    // ---- producer: issue the copies of chunk cc into its ring stage
    auto issue = [&](int64_t cc) {
        if (cc < c1) {
            if (cc >= ld_end) {
                while (unit_start[u_load + 1] <= cc) ++u_load;
                ld_start = unit_start[u_load];
                ld_end = unit_start[u_load + 1];
                ld_unit();
            }
            const int p0 = (int)(cc - ld_start) * kChunk;
            const int32_t blk = ld_bt[p0 / a.bs];
            if (blk >= 0 && blk < a.num_blocks) {
                const int64_t row0 = ((int64_t)blk * a.Hkv + ld_kvh) * a.bs + p0 % a.bs;
                const uint8_t* ks = reinterpret_cast<const uint8_t*>(kp + row0 * D);
                const uint8_t* vs = reinterpret_cast<const uint8_t*>(vp + row0 * D);
                const uint32_t st = wsm_u32 + (uint32_t)((cc - c0) % NST) * C::kStageBytes;
#pragma unroll
                for (int i = lane; i < C::kPieces; i += 32) {
                    const int row = i / (D / 8), pc = i % (D / 8);
                    const uint32_t so = row * C::kRowBytes + ((pc ^ (row & 7)) << 4);
                    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;\n" ::"r"(st + so),
                                 "l"(ks + i * 16), "l"(l2_first) : "memory");
                    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;\n" ::"r"(st + C::kTileBytes + so),
                                 "l"(vs + i * 16), "l"(l2_first) : "memory");
                }
            }
        }
        cp_async_commit();
    };

    // ---- per-thread fragment state
    const int g8 = lane >> 2, t4 = lane & 3;   // mma fragment coordinates
    const int rowA = g8, rowB = g8 + 8;
    uint32_t qf[C::kKSteps][4];
    float o[C::kNT][4];
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
    int64_t boundA = 0, boundB = 0;
    int64_t cur_group = -1, cur_bk = -1, cur_unit = -1;
    int cur_b = 0, cur_kvh = 0, cur_r = 0;
    int64_t cu_start = ws0.ustart, cu_end = ws0.uend, cu_bk = lo / a.N;
    int cu_r = (int)(lo % a.N);
    const int32_t* cu_bt = a.block_tables + ((int64_t)cu_r * a.B + (int)(cu_bk / a.Hkv)) * a.max_blocks;
    int fullvis = 0;  // chunks below this local position are visible to every row
    const float sl2 = a.softmax_scale * 1.4426950408889634f;  // log2(e)

    auto reset_state = [&]() {
        mA = mB = -INFINITY;
        lA = lB = 0.f;
#pragma unroll
        for (int j = 0; j < C::kNT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    };

    // One finished segment: the final output (a group inside one worker), or
    // a partial slot and an arrival on the group's counter, whose last arriver
    // merges the group.  (Spreading the fence and the arrival over the next
    // chunks, so that a segment ending mid-range would not stall the page
    // stream, measured 3 us slower on a 32-request, 8K-token, 8-KV-head decode.)
    struct Arrival {
        int64_t group;
        int nseg, b, kvh, r;
        uint32_t prev;  // the counter's value before this arrival (lane 0)
    };
    Arrival pend{0, 0, 0, 0, 0, 0u};
    auto out_row = [&](int b, int kvh, int r, int row) -> int64_t {
        const int t = row / a.G, gq = row % a.G;
        const int64_t orow = ((int64_t)b * a.Tq + t) * a.Hq + (int64_t)kvh * a.G + gq;
        return a.partial_mode ? (int64_t)r * a.B * a.Tq * a.Hq + orow : orow;
    };
    auto write_final = [&](int64_t orow, int d, float v) {
        if (a.partial_mode)
            a.out_partial[orow * a.Dv + d] = v;
        else
            store_out(a.out, orow * a.Dv + d, v, a.out_dtype);
    };
    auto write_lse = [&](int64_t orow, float v) {
        if (a.partial_mode) a.lse_partial[orow] = v;
        else if (a.lse) a.lse[orow] = v;
    };
    auto flush = [&](int64_t group) -> bool {  // true: a partial arrived on the counter
        float la = lA + __shfl_xor_sync(0xffffffffu, lA, 1);
        la += __shfl_xor_sync(0xffffffffu, la, 2);
        float lb = lB + __shfl_xor_sync(0xffffffffu, lB, 1);
        lb += __shfl_xor_sync(0xffffffffu, lb, 2);
        const float ln2 = 0.6931471805599453f;
        const float lseA = (la > 0.f) ? mA * ln2 + logf(la) : -INFINITY;
        const float lseB = (lb > 0.f) ? mB * ln2 + logf(lb) : -INFINITY;
        const float invA = (la > 0.f) ? 1.f / la : 0.f, invB = (lb > 0.f) ? 1.f / lb : 0.f;
        const int64_t first = unit_start[group * per_group];
        const int64_t last = unit_start[(group + 1) * per_group] - 1;
        const int64_t wf = worker_of(first, We, P);
        const int nseg = (int)(worker_of(last, We, P) - wf + 1);
        const int b = cur_b, kvh = cur_kvh, r = cur_r;
        if (nseg == 1) {
            const int64_t oA = out_row(b, kvh, r, rowA), oB = out_row(b, kvh, r, rowB);
#pragma unroll
            for (int j = 0; j < C::kNT; ++j) {
                const int d = j * 8 + 2 * t4;
                if (rowA < a.rows) { write_final(oA, d, o[j][0] * invA); write_final(oA, d + 1, o[j][1] * invA); }
                if (rowB < a.rows) { write_final(oB, d, o[j][2] * invB); write_final(oB, d + 1, o[j][3] * invB); }
            }
            if (t4 == 0) {
                if (rowA < a.rows) write_lse(oA, lseA);
                if (rowB < a.rows) write_lse(oB, lseB);
            }
            return false;
        }
        const int64_t slot = seg_base[group] + (w - wf);
#pragma unroll
        for (int j = 0; j < C::kNT; ++j) {
            const int d = j * 8 + 2 * t4;
            if (rowA < a.rows)
                *reinterpret_cast<float2*>(&part_o[(slot * a.rows + rowA) * a.Dv + d]) =
                    make_float2(o[j][0] * invA, o[j][1] * invA);
            if (rowB < a.rows)
                *reinterpret_cast<float2*>(&part_o[(slot * a.rows + rowB) * a.Dv + d]) =
                    make_float2(o[j][2] * invB, o[j][3] * invB);
        }
        if (t4 == 0) {
            if (rowA < a.rows) part_lse[slot * a.rows + rowA] = lseA;
            if (rowB < a.rows) part_lse[slot * a.rows + rowB] = lseB;
        }
        // the partial is visible before the counter moves
        pend = Arrival{group, nseg, b, kvh, r, 0u};
        __threadfence();
        __syncwarp();
        if (lane == 0) pend.prev = atomicAdd(&counters[pend.group], 1u);
        return true;
    };
    auto merge_if_last = [&]() {
        const uint32_t prev = __shfl_sync(0xffffffffu, pend.prev, 0);
        if (prev != (uint32_t)(pend.nseg - 1)) return;
        const int64_t group = pend.group;
        const int nseg = pend.nseg;
        // last arriver: merge the group's nseg partials.  It runs in the
        // kernel's tail (a group's last segment usually ends a worker's range),
        // so every load of it is made independent: 8 lanes per row, 4 rows per
        // pass, each lane D/8 output columns as float4 and, per batch of 8
        // segments, one segment's log-sum-exp; batches rescale online.
        __threadfence();
        const int64_t base = seg_base[group];
        constexpr int kLpr = 8, kCols = D / kLpr, kV4 = kCols / 4;
        constexpr float kLog2e = 1.4426950408889634f;
        const int q = lane & (kLpr - 1), lane0 = lane & ~(kLpr - 1);
        for (int r0 = 0; r0 < a.rows; r0 += 32 / kLpr) {
            const int row = r0 + lane / kLpr;
            const bool live = row < a.rows;
            float mx = -INFINITY, sum = 0.f;
            float4 acc[kV4];
#pragma unroll
            for (int v = 0; v < kV4; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int i0 = 0; i0 < nseg; i0 += kLpr) {
                const int i = i0 + q;
                const float li = (live && i < nseg) ? __ldcg(&part_lse[(base + i) * a.rows + row]) : -INFINITY;
                float bm = li;
#pragma unroll
                for (int o = 1; o < kLpr; o <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
                const float nm = fmaxf(mx, bm);
                const float sc = (nm == -INFINITY) ? 1.f : exp2f((mx - nm) * kLog2e);
                const float wi = (li == -INFINITY) ? 0.f : exp2f((li - nm) * kLog2e);
                float ws = wi;
#pragma unroll
                for (int o = 1; o < kLpr; o <<= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
                sum = sum * sc + ws;
#pragma unroll
                for (int v = 0; v < kV4; ++v) {
                    acc[v].x *= sc; acc[v].y *= sc; acc[v].z *= sc; acc[v].w *= sc;
                }
                const int nb = nseg - i0 < kLpr ? nseg - i0 : kLpr;
#pragma unroll
                for (int k = 0; k < kLpr; ++k) {
                    const float wk = __shfl_sync(0xffffffffu, wi, lane0 | k);
                    if (k < nb && live) {
                        const float4* src = reinterpret_cast<const float4*>(
                            &part_o[((base + i0 + k) * a.rows + row) * a.Dv + q * kCols]);
#pragma unroll
                        for (int v = 0; v < kV4; ++v) {
                            const float4 x = __ldcg(src + v);
                            acc[v].x += wk * x.x; acc[v].y += wk * x.y; acc[v].z += wk * x.z; acc[v].w += wk * x.w;
                        }
                    }
                }
                mx = nm;
            }
            if (live) {
                const float inv = (sum > 0.f) ? 1.f / sum : 0.f;
                const int64_t orow = out_row(pend.b, pend.kvh, pend.r, row);
#pragma unroll
                for (int v = 0; v < kV4; ++v) {
                    const int d = q * kCols + 4 * v;
                    write_final(orow, d, acc[v].x * inv);
                    write_final(orow, d + 1, acc[v].y * inv);
                    write_final(orow, d + 2, acc[v].z * inv);
                    write_final(orow, d + 3, acc[v].w * inv);
                }
                if (q == 0) write_lse(orow, (mx == -INFINITY) ? -INFINITY : mx + logf(sum));
            }
        }
        if (lane == 0) counters[group] = 0;
    };

#pragma unroll
    for (int k = 0; k < NST - 1; ++k) issue(c0 + k);

    for (int64_t c = c0; c < c1; ++c) {
        issue(c + NST - 1);
        cp_async_wait<NST - 1>();
        __syncwarp();

        if (c >= cu_end) {
            while (unit_start[u + 1] <= c) ++u;
            cu_start = unit_start[u];
            cu_end = unit_start[u + 1];
            cu_r = (int)(u % a.N);
            cu_bk = u / a.N;
            cu_bt = a.block_tables + ((int64_t)cu_r * a.B + (int)(cu_bk / a.Hkv)) * a.max_blocks;
        }
        const int r = cu_r;
        const int64_t bk = cu_bk;
        const int b = (int)(bk / a.Hkv), kvh = (int)(bk - (int64_t)b * a.Hkv);
        const int64_t group = a.partial_mode ? u : bk;
        if (group != cur_group) {
            if (cur_group >= 0) {
                if (flush(cur_group)) merge_if_last();
            }
            cur_group = group;
            reset_state();
        }
        cur_b = b; cur_kvh = kvh; cur_r = r;
        const int64_t L = a.seq_lens[b];
        if (bk != cur_bk) {
            cur_bk = bk;
            // Q rows (t, gq) -> A fragments; rows >= a.rows are zero
            const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(a.q);
            auto qrow_ptr = [&](int row) -> const uint32_t* {
                const int t = row / a.G, gq = row % a.G;
                return reinterpret_cast<const uint32_t*>(qb + (((int64_t)b * a.Tq + t) * a.Hq + (int64_t)kvh * a.G + gq) * D);
            };
            const uint32_t* qa = rowA < a.rows ? qrow_ptr(rowA) : nullptr;
            const uint32_t* qbp = rowB < a.rows ? qrow_ptr(rowB) : nullptr;
#pragma unroll
            for (int ks = 0; ks < C::kKSteps; ++ks) {
                const int e = ks * 8 + t4;  // 32-bit word index of columns 16ks + 2t4
                qf[ks][0] = qa ? qa[e] : 0u;
                qf[ks][1] = qbp ? qbp[e] : 0u;
                qf[ks][2] = qa ? qa[e + 4] : 0u;
                qf[ks][3] = qbp ? qbp[e + 4] : 0u;
            }
        }
        if (u != cur_unit) {
            cur_unit = u;
            boundA = rowA < a.rows ? local_len(L - a.Tq + rowA / a.G + 1, r, a.N, a.I) : 0;
            boundB = rowB < a.rows ? local_len(L - a.Tq + rowB / a.G + 1, r, a.N, a.I) : 0;
            // every row sees at least the first len(L - Tq + 1) local positions
            fullvis = (int)local_len(L - a.Tq + 1, r, a.N, a.I);
        }
        const int p0 = (int)(c - cu_start) * kChunk;
        const int32_t blk = cu_bt[p0 / a.bs];
        if (blk < 0 || blk >= a.num_blocks) {
            if (lane == 0) raise_err(err, DCP_DEV_ERR_BLOCK_ID);
            __syncwarp();
            continue;
        }
        const uint32_t st = wsm_u32 + (uint32_t)((c - c0) % NST) * C::kStageBytes;

        // S = Q K^T over the chunk's 16 tokens (two n-tiles of 8)
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
            const int mi = lane >> 3, rr = lane & 7;
            const int tok = (mi >> 1) * 8 + rr;
#pragma unroll
            for (int ks = 0; ks < C::kKSteps; ++ks) {
                const int pc = 2 * ks + (mi & 1);
                uint32_t k0, k1, k2, k3;
                ldsm_x4(st + tok * C::kRowBytes + ((pc ^ (tok & 7)) << 4), k0, k1, k2, k3);
                mma_bf16(s[0], qf[ks], k0, k1);
                mma_bf16(s[1], qf[ks], k2, k3);
            }
        }
        // scale to base 2, mask (only a chunk some row cannot fully see), online
        // softmax.  Rows past a.rows are padding: their values are never written.
        float mxA = -INFINITY, mxB = -INFINITY;
        const bool all_visible = (p0 + kChunk <= fullvis);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            if (all_visible) {
                s[nt][0] *= sl2; s[nt][1] *= sl2; s[nt][2] *= sl2; s[nt][3] *= sl2;
            } else {
                const int64_t tok = p0 + nt * 8 + 2 * t4;
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
        const bool changed = (mnA != mA) || (mnB != mB);
        if (__any_sync(0xffffffffu, changed)) {
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
        uint32_t pf[4];
        {
            float p[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                p[nt][0] = sm100::ex2_approx(s[nt][0] - useA);
                p[nt][1] = sm100::ex2_approx(s[nt][1] - useA);
                p[nt][2] = sm100::ex2_approx(s[nt][2] - useB);
                p[nt][3] = sm100::ex2_approx(s[nt][3] - useB);
                lA += p[nt][0] + p[nt][1];
                lB += p[nt][2] + p[nt][3];
            }
            pf[0] = pack_bf16(p[0][0], p[0][1]);
            pf[1] = pack_bf16(p[0][2], p[0][3]);
            pf[2] = pack_bf16(p[1][0], p[1][1]);
            pf[3] = pack_bf16(p[1][2], p[1][3]);
        }
        // O += P V (V tile through ldmatrix.trans)
        {
            const uint32_t vt = st + C::kTileBytes;
            const int mi = lane >> 3, rr = lane & 7;
            const int tok = (mi & 1) * 8 + rr;
#pragma unroll
            for (int jp = 0; jp < C::kNT / 2; ++jp) {
                const int pc = 2 * jp + (mi >> 1);
                uint32_t v0, v1, v2, v3;
                ldsm_x4_t(vt + tok * C::kRowBytes + ((pc ^ (tok & 7)) << 4), v0, v1, v2, v3);
                mma_bf16(o[2 * jp], pf, v0, v1);
                mma_bf16(o[2 * jp + 1], pf, v2, v3);
            }
        }
        __syncwarp();
    }
    cp_async_wait<0>();
    if (cur_group >= 0) {
        if (flush(cur_group)) merge_if_last();
    }
}

template <int D, int NST>
cudaError_t launch_t(const AttnArgs& a, cudaStream_t s) {
    using C = Cfg<D, NST>;
    cudaError_t e = cudaFuncSetAttribute(gqa_mma_kernel<D, NST>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    const unsigned blocks = (unsigned)((a.W + kWarps - 1) / kWarps);
    return launch_pdl(gqa_mma_kernel<D, NST>, dim3(blocks), dim3(kWarps * 32), C::kSmem, s, a);
}

}  // namespace

bool gqa_mma_supported(const dcp_params& p) {
    const int G = p.Hkv > 0 ? p.Hq / p.Hkv : 0;
    return p.layout == DCP_LAYOUT_GQA && p.q_dtype == DCP_BF16 && p.kv_dtype == DCP_BF16 && p.Dk == p.Dv &&
           (p.Dk == 64 || p.Dk == 128) && p.block_size % kChunk == 0 && G * p.Tq <= 16;
}

// 2 CTAs of 4 warps per SM (the smem ring sets the residency)
int64_t gqa_mma_workers(int num_sms) { return (int64_t)num_sms * 2 * kWarps; }

cudaError_t launch_attn_gqa_mma(const AttnArgs& a, cudaStream_t s) {
    if (a.Dk == 64) return launch_t<64, 4>(a, s);
    return launch_t<128, 3>(a, s);
}

}  // namespace dcp

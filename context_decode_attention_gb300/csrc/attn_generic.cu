// Split-KV partial decode attention on CUDA cores, for any storage dtype and
// widths up to 576 / 512 (fp32 everywhere inside).
//
// "vLLM DCP and PCP", Deep Dive 6: rank i computes s_j = q . k_j / sqrt(d)
// over its shard, L_i = log sum exp s_j and o_i = sum exp(s_j) v_j / exp(L_i).
// Here every chunk range of a worker yields such a partial (o, L) for its
// segment; segment_merge_kernel then merges them exactly.
//
// Grid: x = worker (one CTA of 4 warps), y = tile of 16 query rows; warp w
// owns rows w, w+4, w+8, w+12 of the tile; lanes split the Dk / Dv columns.
#include "dcp_internal.cuh"

namespace dcp {
namespace {

constexpr int kRowsPerWarp = 4;
constexpr int kTileRows = 16;
constexpr int kTok = 8;  // tokens scored together

template <int DKC, int DVC>
__global__ void __launch_bounds__(128) attn_generic_kernel(AttnArgs a, int q_dtype, int kv_dtype) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();     // the plan
    pdl_trigger();  // the segment merge may launch
    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(a.ws);
    const int64_t P = hdr->total_chunks;
    if (hdr->plan_key != a.plan_key) {  // the workspace holds a plan for other arguments
        if (threadIdx.x == 0) raise_err(&reinterpret_cast<WsHeader*>(a.ws)->err, DCP_DEV_ERR_PLAN);
        return;
    }
    if (P == 0) return;
    const int64_t w = blockIdx.x;
    const int64_t We = P < a.W ? P : a.W;  // workers in play: each owns >= 1 chunk
    if (w >= We) return;
    const int64_t c0 = worker_begin(w, We, P), c1 = worker_begin(w + 1, We, P);
    if (c0 >= c1) return;
    const int64_t* unit_start = reinterpret_cast<const int64_t*>(a.ws + a.lay.off_units);
    const int32_t* seg_base = reinterpret_cast<const int32_t*>(a.ws + a.lay.off_seg_base);
    float* part_o = reinterpret_cast<float*>(a.ws + a.lay.off_part_o);
    float* part_lse = reinterpret_cast<float*>(a.ws + a.lay.off_part_lse);
    uint32_t* err = &reinterpret_cast<WsHeader*>(a.ws)->err;

    // unit containing c0: the last u with unit_start[u] <= c0
    int64_t lo = 0, hi = a.U - 1;
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) >> 1;
        if (unit_start[mid] <= c0) lo = mid; else hi = mid - 1;
    }
    int64_t u = lo;

    const int per_group = a.partial_mode ? 1 : a.N;
    int my_rows[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) my_rows[i] = blockIdx.y * kTileRows + warp + 4 * i;

    float q[kRowsPerWarp][DKC], o[kRowsPerWarp][DVC], m[kRowsPerWarp], l[kRowsPerWarp];
    int64_t bound[kRowsPerWarp];
    int64_t cur_group = -1, cur_bk = -1, cur_unit = -1;
    const float s_scale = a.softmax_scale * a.kv_scale;

    auto flush = [&](int64_t group) {
        const int64_t first = unit_start[group * per_group];
        const int64_t slot = seg_base[group] + (w - worker_of(first, We, P));
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const int row = my_rows[i];
            if (row >= a.rows) continue;
            const bool empty = (l[i] == 0.f);
            const float inv = empty ? 0.f : a.kv_scale / l[i];
#pragma unroll
            for (int c = 0; c < DVC; ++c) {
                const int d = lane + 32 * c;
                if (d < a.Dv) part_o[(slot * a.rows + row) * a.Dv + d] = o[i][c] * inv;
            }
            if (lane == 0) part_lse[slot * a.rows + row] = empty ? -INFINITY : m[i] + logf(l[i]);
        }
    };

    for (int64_t c = c0; c < c1; ++c) {
        while (unit_start[u + 1] <= c) ++u;
        const int r = (int)(u % a.N);
        const int64_t bk = u / a.N;
        const int b = (int)(bk / a.Hkv), kvh = (int)(bk % a.Hkv);
        const int64_t group = a.partial_mode ? u : bk;
        if (group != cur_group) {
            if (cur_group >= 0) flush(cur_group);
            cur_group = group;
#pragma unroll
            for (int i = 0; i < kRowsPerWarp; ++i) {
                m[i] = -INFINITY;
                l[i] = 0.f;
#pragma unroll
                for (int cc = 0; cc < DVC; ++cc) o[i][cc] = 0.f;
            }
        }
        const int64_t L = a.seq_lens[b];
        if (bk != cur_bk) {
            cur_bk = bk;
#pragma unroll
            for (int i = 0; i < kRowsPerWarp; ++i) {
                const int row = my_rows[i] < a.rows ? my_rows[i] : 0;
                const int t = row / a.G, gq = row % a.G;
                const int64_t qrow = ((int64_t)b * a.Tq + t) * a.Hq + (int64_t)kvh * a.G + gq;
#pragma unroll
                for (int cc = 0; cc < DKC; ++cc) {
                    const int d = lane + 32 * cc;
                    q[i][cc] = (d < a.Dk) ? load_elem(a.q, qrow * a.Dk + d, q_dtype) : 0.f;
                }
            }
        }
        if (u != cur_unit) {
            cur_unit = u;
#pragma unroll
            for (int i = 0; i < kRowsPerWarp; ++i) {
                const int t = (my_rows[i] < a.rows ? my_rows[i] : 0) / a.G;
                bound[i] = my_rows[i] < a.rows ? local_len(L - a.Tq + t + 1, r, a.N, a.I) : 0;
            }
        }
        const int64_t len = local_len(L, r, a.N, a.I);
        const int64_t p0 = (c - unit_start[u]) * a.CH;
        const int64_t p1 = (p0 + a.CH < len) ? p0 + a.CH : len;
        const int64_t page = p0 / a.bs;
        const int32_t blk = a.block_tables[((int64_t)r * a.B + b) * a.max_blocks + page];
        if (blk < 0 || blk >= a.num_blocks) {
            if (lane == 0 && warp == 0 && blockIdx.y == 0) raise_err(err, DCP_DEV_ERR_BLOCK_ID);
            continue;
        }
        for (int64_t p = p0; p < p1; p += kTok) {
            float s[kRowsPerWarp][kTok];
#pragma unroll
            for (int k = 0; k < kTok; ++k) {
                const int64_t pk = p + k;
                float kv[DKC];
                if (pk < p1) {
                    const int64_t off = pk % a.bs;
                    const int64_t krow = (a.layout == DCP_LAYOUT_MLA)
                                             ? ((int64_t)blk * a.bs + off) * a.Dk
                                             : (((int64_t)blk * a.Hkv + kvh) * a.bs + off) * a.Dk;
#pragma unroll
                    for (int cc = 0; cc < DKC; ++cc) {
                        const int d = lane + 32 * cc;
                        kv[cc] = (d < a.Dk) ? load_elem(a.k_pool, krow + d, kv_dtype) : 0.f;
                    }
                }
#pragma unroll
                for (int i = 0; i < kRowsPerWarp; ++i) {
                    float acc = 0.f;
                    if (pk < p1) {
#pragma unroll
                        for (int cc = 0; cc < DKC; ++cc) acc = fmaf(q[i][cc], kv[cc], acc);
                    }
#pragma unroll
                    for (int sh = 16; sh > 0; sh >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sh);
                    s[i][k] = (pk < p1 && pk < bound[i]) ? acc * s_scale : -INFINITY;
                }
            }
            float pw[kRowsPerWarp][kTok];
#pragma unroll
            for (int i = 0; i < kRowsPerWarp; ++i) {
                float mx = m[i];
#pragma unroll
                for (int k = 0; k < kTok; ++k) mx = fmaxf(mx, s[i][k]);
                if (mx == -INFINITY) {
#pragma unroll
                    for (int k = 0; k < kTok; ++k) pw[i][k] = 0.f;
                    continue;
                }
                const float corr = expf(m[i] - mx);
                m[i] = mx;
                l[i] *= corr;
#pragma unroll
                for (int cc = 0; cc < DVC; ++cc) o[i][cc] *= corr;
#pragma unroll
                for (int k = 0; k < kTok; ++k) {
                    pw[i][k] = expf(s[i][k] - mx);
                    l[i] += pw[i][k];
                }
            }
#pragma unroll
            for (int k = 0; k < kTok; ++k) {
                const int64_t pk = p + k;
                if (pk >= p1) break;
                const int64_t off = pk % a.bs;
                const void* vbase;
                int64_t vrow;
                if (a.layout == DCP_LAYOUT_MLA) {
                    vbase = a.k_pool;
                    vrow = ((int64_t)blk * a.bs + off) * a.Dk;
                } else {
                    vbase = a.v_pool;
                    vrow = (((int64_t)blk * a.Hkv + kvh) * a.bs + off) * a.Dv;
                }
#pragma unroll
                for (int cc = 0; cc < DVC; ++cc) {
                    const int d = lane + 32 * cc;
                    const float vv = (d < a.Dv) ? load_elem(vbase, vrow + d, kv_dtype) : 0.f;
#pragma unroll
                    for (int i = 0; i < kRowsPerWarp; ++i) o[i][cc] = fmaf(pw[i][k], vv, o[i][cc]);
                }
            }
        }
    }
    if (cur_group >= 0) flush(cur_group);
}

template <int DKC, int DVC>
cudaError_t launch_t(const AttnArgs& a, int q_dtype, int kv_dtype, cudaStream_t s) {
    dim3 grid((unsigned)a.W, (unsigned)((a.rows + kTileRows - 1) / kTileRows));
    return launch_pdl(attn_generic_kernel<DKC, DVC>, grid, dim3(128), 0, s, a, q_dtype, kv_dtype);
}

}  // namespace

bool generic_supported(const dcp_params& p) {
    const int dkc = (p.Dk + 31) / 32, dvc = (p.Dv + 31) / 32;
    return (dkc <= 2 && dvc <= 2) || (dkc <= 4 && dvc <= 4) || (dkc <= 8 && dvc <= 8) ||
           (dkc <= 18 && dvc <= 16);
}

int64_t generic_workers(int num_sms) { return (int64_t)num_sms * 4; }

int generic_chunk(int bs) {
    int ch = 1;
    for (int c = 64; c >= 1; c >>= 1)
        if (bs % c == 0) { ch = c; break; }
    return ch;
}

cudaError_t launch_attn_generic(const AttnArgs& a, int q_dtype, int kv_dtype, cudaStream_t s) {
    const int dkc = (a.Dk + 31) / 32, dvc = (a.Dv + 31) / 32;
    if (dkc <= 2 && dvc <= 2) return launch_t<2, 2>(a, q_dtype, kv_dtype, s);
    if (dkc <= 4 && dvc <= 4) return launch_t<4, 4>(a, q_dtype, kv_dtype, s);
    if (dkc <= 8 && dvc <= 8) return launch_t<8, 8>(a, q_dtype, kv_dtype, s);
    return launch_t<18, 16>(a, q_dtype, kv_dtype, s);
}

}  // namespace dcp

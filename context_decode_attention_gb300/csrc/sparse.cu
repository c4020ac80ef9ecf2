// DCP-localised sparse (top-k) attention: candidate localisation and the
// staging of every rank's candidates for the dense decode kernels.
//
// "GLM-5.3 Optimizations, Part 2": sparse MLA attends to a selected set of
// 2,048 tokens per query, chosen by an indexer.  "vLLM DCP and PCP" (its
// source-and-test table): under DCP the candidates are localised, i.e. each
// rank keeps those it owns, at their local positions, and the exact result is
// the LSE merge of the ranks' partials over their own candidates.
//
// Localisation: each rank's candidates of a query row, compacted in list
// order.  Staging: rank r's candidates of query row i become rank r's local
// tokens of "request" i in a staging cache (64-token pages), so the dense
// decode kernels, given those counts as the local lengths, compute the ranks'
// partials and merge them exactly.
#include "dcp_internal.cuh"

namespace dcp {
namespace {

// One CTA per (query row i, rank rr): warp w scans a contiguous slice of the
// candidate list; the warps' counts give each slice its first output slot,
// and a second scan writes the rank's candidates in list order.
constexpr int kLocWarps = 8;

__global__ void __launch_bounds__(32 * kLocWarps) sparse_localize_kernel(int N, int I, int rows, int Tq, int k,
                                                                         const int32_t* __restrict__ cand,
                                                                         const int32_t* __restrict__ seq_lens,
                                                                         int32_t* __restrict__ local,
                                                                         int32_t* __restrict__ counts, uint32_t* err) {
    __shared__ int s_cnt[kLocWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t i = blockIdx.x / N;
    const int rr = (int)(blockIdx.x % N);
    const int b = (int)(i / Tq), t = (int)(i % Tq);
    const int64_t vis = (int64_t)seq_lens[b] - Tq + t + 1;  // positions this query token may see
    const int slice = (k + kLocWarps - 1) / kLocWarps;
    const int j_beg = min(k, warp * slice), j_end = min(k, j_beg + slice);
    const int32_t* row = cand + i * k;
    int32_t* out = local + ((int64_t)rr * rows + i) * k;
    auto owner = [&](int j, int32_t& lp) -> bool {  // candidate j is rank rr's; lp = its local position
        const int32_t tok = j < j_end ? row[j] : -1;
        if (tok < 0 || tok >= vis) {
            if (tok >= 0 && rr == 0) raise_err(err, DCP_DEV_ERR_TOKEN);  // reported once
            return false;
        }
        const uint32_t ut = (uint32_t)tok;
        if ((int)((ut / (uint32_t)I) % (uint32_t)N) != rr) return false;
        lp = (int32_t)((uint64_t)ut / ((uint64_t)N * I) * (uint64_t)I + ut % (uint32_t)I);
        return true;
    };
    int mine = 0;
    for (int j0 = j_beg; j0 < j_end; j0 += 32) {
        int32_t lp;
        mine += __popc(__ballot_sync(0xffffffffu, owner(j0 + lane, lp)));
    }
    if (lane == 0) s_cnt[warp] = mine;
    __syncthreads();
    int base = 0, total = 0;
    for (int w = 0; w < kLocWarps; ++w) {
        base += w < warp ? s_cnt[w] : 0;
        total += s_cnt[w];
    }
    for (int j0 = j_beg; j0 < j_end; j0 += 32) {
        int32_t lp = -1;
        const bool own = owner(j0 + lane, lp);
        const unsigned m = __ballot_sync(0xffffffffu, own);
        if (own) out[base + __popc(m & ((1u << lane) - 1u))] = lp;
        base += __popc(m);
    }
    for (int j = total + threadIdx.x; j < k; j += blockDim.x) out[j] = -1;
    if (threadIdx.x == 0) counts[(int64_t)rr * rows + i] = total;
}

// One CTA per staging request s = r R + i: its page table, and rank r's
// candidate rows of query row i copied contiguously (16-byte pieces).
__global__ void sparse_stage_kernel(SparseStageArgs a) {
    const int64_t s = blockIdx.x;
    const int r = (int)(s / a.R);
    const int64_t i = s % a.R;
    const int b = (int)(i / a.Tq);
    const int pages = a.kpad / 64;
    for (int p = threadIdx.x; p < pages; p += blockDim.x) a.st_tables[s * pages + p] = (int32_t)(s * pages + p);
    if (r == 0 && threadIdx.x == 0) a.st_lens[i] = a.N * a.kpad;
    const int cnt = a.counts[s];
    const int vec = a.row_bytes / 16;
    const int32_t* loc = a.local + s * a.k;
    const int32_t* bt = a.block_tables + ((int64_t)r * a.B + b) * a.max_blocks;
    const uint4* src = reinterpret_cast<const uint4*>(a.k_pool);
    uint4* dst = reinterpret_cast<uint4*>(a.st_pool) + s * a.kpad * vec;
    bool bad = false;
    for (int x = threadIdx.x; x < cnt * vec; x += blockDim.x) {
        const int j = x / vec, v = x - j * vec;
        const int32_t lp = loc[j];
        const int32_t blk = bt[lp / a.bs];
        if (blk < 0 || blk >= a.num_blocks) {
            bad = true;
            continue;
        }
        dst[(int64_t)j * vec + v] = src[((int64_t)blk * a.bs + lp % a.bs) * vec + v];
    }
    if (bad) raise_err(a.err, DCP_DEV_ERR_BLOCK_ID);
}

}  // namespace

cudaError_t launch_sparse_localize(int N, int I, int rows, int Tq, int k, const int32_t* cand, const int32_t* seq_lens,
                                   int32_t* local, int32_t* counts, uint32_t* err, cudaStream_t s) {
    sparse_localize_kernel<<<(unsigned)((int64_t)rows * N), 32 * kLocWarps, 0, s>>>(N, I, rows, Tq, k, cand, seq_lens,
                                                                                   local, counts, err);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_sparse_stage(const SparseStageArgs& a, cudaStream_t s) {
    sparse_stage_kernel<<<(unsigned)((int64_t)a.N * a.R), 256, 0, s>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace dcp

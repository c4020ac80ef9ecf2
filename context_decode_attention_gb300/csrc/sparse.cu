// DCP-localised sparse (top-k) attention: candidate localisation and the
// staging of every rank's candidates for the dense decode kernels.
//
// "GLM-5.3 Optimizations, Part 2": sparse MLA attends to a selected set of
// 2,048 tokens per query, chosen by an indexer.  "vLLM DCP and PCP" (its
// source-and-test table): under DCP the candidates are localised, i.e. each
// rank keeps those it owns, at their local positions, and the exact result is
// the LSE merge of the ranks' partials over their own candidates.
//
// Localisation: one warp per query row; candidates in list order, each
// rank's in a compacted list (warp ballots keep the list order).  Staging:
// rank r's candidates of query row i become the contiguous "request" r R + i
// of a staging cache (64-token pages, one query row per request), so the
// dense MLA kernels compute the rank partials as ordinary decode partials
// with one virtual rank.
#include "dcp_internal.cuh"

namespace dcp {
namespace {

__global__ void sparse_localize_kernel(int N, int I, int rows, int Tq, int k, const int32_t* __restrict__ cand,
                                       const int32_t* __restrict__ seq_lens, int32_t* __restrict__ local,
                                       int32_t* __restrict__ counts, uint32_t* err) {
    const int lane = threadIdx.x & 31;
    const int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (i >= rows) return;
    const int b = (int)(i / Tq), t = (int)(i % Tq);
    const int32_t L = seq_lens[b];
    const int64_t vis = (int64_t)L - Tq + t + 1;  // positions this query token may see
    const uint64_t NI = (uint64_t)N * (uint64_t)I;
    int my_cnt = 0;  // lane r < N holds rank r's count
    bool bad = false;
    for (int j0 = 0; j0 < k; j0 += 32) {
        const int j = j0 + lane;
        const int32_t tok = j < k ? cand[i * k + j] : -1;
        bool valid = tok >= 0;
        if (valid && tok >= vis) {
            bad = true;
            valid = false;
        }
        const uint32_t ut = (uint32_t)tok;
        const int r = valid ? (int)((ut / (uint32_t)I) % (uint32_t)N) : -1;
        const int32_t lp = valid ? (int32_t)((uint64_t)ut / NI * (uint64_t)I + ut % (uint32_t)I) : -1;
        for (int rr = 0; rr < N; ++rr) {
            const unsigned m = __ballot_sync(0xffffffffu, r == rr);
            if (m == 0) continue;
            const int base = __shfl_sync(0xffffffffu, my_cnt, rr);
            if (r == rr) local[((int64_t)rr * rows + i) * k + base + __popc(m & ((1u << lane) - 1u))] = lp;
            if (lane == rr) my_cnt += __popc(m);
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) raise_err(err, DCP_DEV_ERR_TOKEN);
    for (int rr = 0; rr < N; ++rr) {
        const int c = __shfl_sync(0xffffffffu, my_cnt, rr);
        if (lane == 0) counts[(int64_t)rr * rows + i] = c;
        for (int j = c + lane; j < k; j += 32) local[((int64_t)rr * rows + i) * k + j] = -1;
    }
}

// Staging request s = r R + i: seq_len = count, block table = its own Kpad /
// 64 pages, rows = copies of the candidates' cache rows, and the query row.
__global__ void sparse_stage_kernel(SparseStageArgs a) {
    const int64_t S = (int64_t)a.N * a.R;
    const int pages = a.kpad / 64;
    const int vec = a.row_bytes / 16;  // 16-byte pieces per cache row
    const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nt = (int64_t)gridDim.x * blockDim.x;
    // metadata
    for (int64_t x = gt; x < S * pages; x += nt) {
        const int64_t s = x / pages;
        const int p = (int)(x % pages);
        a.st_tables[x] = (int32_t)(s * pages + p);
        if (p == 0) {
            const int32_t c = a.counts[s];
            a.st_lens[s] = c;
        }
    }
    // candidate rows: piece v of row j of request s
    const int64_t pieces = S * a.kpad * vec;
    bool bad = false;
    for (int64_t x = gt; x < pieces; x += nt) {
        const int64_t row = x / vec;  // s * kpad + j
        const int v = (int)(x % vec);
        const int64_t s = row / a.kpad;
        const int j = (int)(row % a.kpad);
        if (j >= a.counts[s]) continue;
        const int r = (int)(s / a.R);
        const int64_t i = s % a.R;
        const int b = (int)(i / a.Tq);
        const int32_t lp = a.local[s * a.k + j];
        const int32_t blk = a.block_tables[((int64_t)r * a.B + b) * a.max_blocks + lp / a.bs];
        if (blk < 0 || blk >= a.num_blocks) {
            bad = true;
            continue;
        }
        const int64_t src_row = (int64_t)blk * a.bs + lp % a.bs;
        reinterpret_cast<uint4*>(a.st_pool)[row * vec + v] =
            reinterpret_cast<const uint4*>(a.k_pool)[src_row * vec + v];
    }
    if (bad) raise_err(a.err, DCP_DEV_ERR_BLOCK_ID);
    // query rows: request s = r R + i reads query row i
    const int qvec = a.q_row_bytes / 16;
    for (int64_t x = gt; x < S * qvec; x += nt) {
        const int64_t s = x / qvec;
        const int v = (int)(x % qvec);
        const int64_t i = s % a.R;
        reinterpret_cast<uint4*>(a.st_q)[s * qvec + v] = reinterpret_cast<const uint4*>(a.q)[i * qvec + v];
    }
}

}  // namespace

cudaError_t launch_sparse_localize(int N, int I, int rows, int Tq, int k, const int32_t* cand, const int32_t* seq_lens,
                                   int32_t* local, int32_t* counts, uint32_t* err, cudaStream_t s) {
    const int warps = 8;
    sparse_localize_kernel<<<(unsigned)((rows + warps - 1) / warps), 32 * warps, 0, s>>>(N, I, rows, Tq, k, cand,
                                                                                      seq_lens, local, counts, err);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_sparse_stage(const SparseStageArgs& a, cudaStream_t s) {
    sparse_stage_kernel<<<152 * 8, 256, 0, s>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace dcp

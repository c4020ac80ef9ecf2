// DCP-localised sparse (top-k) attention: candidate localisation and the
// staging of every rank's candidates for the dense decode kernels.
//
// The GLM-5.3 context-parallelism page (vLLM's second GLM-5.3 article),
// "What DP and TP leave unresolved": sparse MLA attends to a selected set of
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

// Rank rr's candidates of query row i, by one CTA of kLocWarps warps: warp w
// scans a contiguous slice of the candidate list; the warps' counts give each
// slice its first output slot, and a second scan writes the rank's
// candidates' local positions in list order.  Returns the count (every
// thread); fill_tail writes -1 past it.
constexpr int kLocWarps = 8;

__device__ int localize_cta(int N, int I, int Tq, int k, int64_t i, int rr, const int32_t* __restrict__ cand,
                            const int32_t* __restrict__ seq_lens, int32_t* __restrict__ out, bool fill_tail,
                            uint32_t* err) {
    __shared__ int s_cnt[kLocWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int b = (int)(i / Tq), t = (int)(i % Tq);
    const int64_t vis = (int64_t)seq_lens[b] - Tq + t + 1;  // positions this query token may see
    const int slice = (k + kLocWarps - 1) / kLocWarps;
    const int j_beg = min(k, warp * slice), j_end = min(k, j_beg + slice);
    const int32_t* row = cand + i * k;
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
    if (fill_tail)
        for (int j = total + threadIdx.x; j < k; j += blockDim.x) out[j] = -1;
    return total;
}

// One CTA per (query row i, rank rr).
__global__ void __launch_bounds__(32 * kLocWarps) sparse_localize_kernel(int N, int I, int rows, int Tq, int k,
                                                                         const int32_t* __restrict__ cand,
                                                                         const int32_t* __restrict__ seq_lens,
                                                                         int32_t* __restrict__ local,
                                                                         int32_t* __restrict__ counts, uint32_t* err) {
    const int64_t i = blockIdx.x / N;
    const int rr = (int)(blockIdx.x % N);
    const int total = localize_cta(N, I, Tq, k, i, rr, cand, seq_lens, local + ((int64_t)rr * rows + i) * k, true, err);
    if (threadIdx.x == 0) counts[(int64_t)rr * rows + i] = total;
}

// One CTA per staging request s = r R + i: rank r's candidates of query row i
// localised (as above; the positions go through the workspace, read back by
// the same CTA), the request's page table, and the candidate rows copied
// contiguously in 16-byte pieces.  The rows' pool offsets are resolved into
// shared memory a batch at a time, so the copy loop has no dependent loads
// and keeps kUnroll pieces per thread in flight.
constexpr int kStageThreads = 32 * kLocWarps;
constexpr int kStageBatch = 1024;  // candidate rows per batch
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kStageThreads) sparse_stage_kernel(SparseStageArgs a) {
    __shared__ int64_t s_row[kStageBatch];
    const int64_t s = blockIdx.x;
    const int r = (int)(s / a.R);
    const int64_t i = s % a.R;
    const int b = (int)(i / a.Tq);
    int32_t* loc = a.local + s * a.k;
    const int cnt = localize_cta(a.N, a.I, a.Tq, a.k, i, r, a.cand, a.seq_lens, loc, false, a.err);
    if (threadIdx.x == 0) a.counts[s] = cnt;
    const int pages = a.kpad / 64;
    for (int p = threadIdx.x; p < pages; p += kStageThreads) a.st_tables[s * pages + p] = (int32_t)(s * pages + p);
    if (r == 0 && threadIdx.x == 0) a.st_lens[i] = a.N * a.kpad;
    const int vec = a.row_bytes / 16;
    const int32_t* __restrict__ bt = a.block_tables + ((int64_t)r * a.B + b) * a.max_blocks;
    const uint4* __restrict__ src = reinterpret_cast<const uint4*>(a.k_pool);
    uint4* __restrict__ dst = reinterpret_cast<uint4*>(a.st_pool) + s * a.kpad * vec;
    bool bad = false;
    for (int j0 = 0; j0 < cnt; j0 += kStageBatch) {
        const int nb = min(kStageBatch, cnt - j0);
        __syncthreads();  // the localised positions are written; the previous batch's offsets are read
        for (int j = threadIdx.x; j < nb; j += kStageThreads) {
            const int32_t lp = loc[j0 + j];
            const int32_t blk = bt[lp / a.bs];
            const bool ok = blk >= 0 && blk < a.num_blocks;
            bad |= !ok;
            s_row[j] = ok ? ((int64_t)blk * a.bs + lp % a.bs) * vec : -1;
        }
        __syncthreads();
        const int tot = nb * vec;
        uint4* __restrict__ d0 = dst + (int64_t)j0 * vec;
        for (int x0 = threadIdx.x; x0 < tot; x0 += kUnroll * kStageThreads) {
            uint4 val[kUnroll];
            int at[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int x = x0 + u * kStageThreads;
                at[u] = -1;
                if (x < tot) {
                    const int j = x / vec, c = x - j * vec;
                    const int64_t o = s_row[j];
                    if (o >= 0) {
                        val[u] = src[o + c];
                        at[u] = x;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (at[u] >= 0) d0[at[u]] = val[u];
        }
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
    sparse_stage_kernel<<<(unsigned)((int64_t)a.N * a.R), kStageThreads, 0, s>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace dcp

// Blocks moved under prefill-decode disaggregation.
//
// "Breaking the Long-Sequence Inference Bottleneck ...", section 2
// ("Practical considerations for PD disaggregation"): KV moves between the
// prefill and decode nodes in whole blocks, and a block holding no token need
// not move; with interleave size 1 short requests leave every rank a barely
// filled block, with interleave size = block size the blocks fill first.
//
// A rank stores its tokens in local-position order, so the blocks holding
// tokens of request b on rank r are the first ceil(len / bs) entries of its
// block table (len = the rank's local length), all full but the last, which
// holds len - (count - 1) bs.  One thread per (rank, request, table entry).
#include "dcp_internal.cuh"

namespace dcp {
namespace {

struct TransferArgs {
    int N, I, bs, B, max_blocks;
    int64_t num_blocks;
    const int32_t* seq_lens;
    const int32_t* block_tables;
    int32_t* counts;
    int32_t* blocks;
    int32_t* fills;
    unsigned long long* totals;  // [2]: slots moved, tokens moved
    uint32_t* err;
};

__global__ void transfer_blocks_kernel(TransferArgs a) {
    const int64_t total = (int64_t)a.N * a.B * a.max_blocks;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int k = (int)(i % a.max_blocks);
        const int64_t rb = i / a.max_blocks;  // r * B + b
        const int b = (int)(rb % a.B), r = (int)(rb / a.B);
        const int64_t L = a.seq_lens[b];
        const int64_t len = L > 0 ? local_len(L, r, a.N, a.I) : 0;
        const int64_t need = ceil_div64(len, a.bs);
        const int64_t cnt = need < a.max_blocks ? need : a.max_blocks;
        if (k == 0) {
            if (need > a.max_blocks) raise_err(a.err, DCP_DEV_ERR_TABLE);
            a.counts[rb] = (int32_t)cnt;
            if (a.totals) {
                atomicAdd(&a.totals[0], (unsigned long long)(need * a.bs));
                atomicAdd(&a.totals[1], (unsigned long long)len);
            }
        }
        int32_t id = -1, fill = 0;
        if (k < cnt) {
            id = a.block_tables[i];
            if (id < 0 || id >= a.num_blocks) {
                raise_err(a.err, DCP_DEV_ERR_BLOCK_ID);
                id = -1;
            }
            const int64_t rest = len - (int64_t)k * a.bs;
            fill = (int32_t)(rest < a.bs ? rest : a.bs);
        }
        if (a.blocks) a.blocks[i] = id;
        if (a.fills) a.fills[i] = fill;
    }
}

}  // namespace

cudaError_t launch_transfer_blocks(int N, int I, int bs, int B, int max_blocks, int64_t num_blocks,
                                   const int32_t* seq_lens, const int32_t* block_tables, int32_t* counts,
                                   int32_t* blocks, int32_t* fills, int64_t* totals, uint32_t* err,
                                   cudaStream_t s) {
    if (totals) {
        cudaError_t e = cudaMemsetAsync(totals, 0, 2 * sizeof(int64_t), s);
        if (e != cudaSuccess) return e;
    }
    TransferArgs a;
    a.N = N; a.I = I; a.bs = bs; a.B = B; a.max_blocks = max_blocks; a.num_blocks = num_blocks;
    a.seq_lens = seq_lens; a.block_tables = block_tables; a.counts = counts; a.blocks = blocks; a.fills = fills;
    a.totals = reinterpret_cast<unsigned long long*>(totals);
    a.err = err;
    const int64_t total = (int64_t)N * B * max_blocks;
    const int threads = 256;
    int64_t grid = (total + threads - 1) / threads;
    if (grid > 4096) grid = 4096;
    if (grid < 1) grid = 1;
    transfer_blocks_kernel<<<(unsigned)grid, threads, 0, s>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace dcp

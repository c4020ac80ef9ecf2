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
// holds len - (count - 1) bs.
//
// One thread per (rank, request, table entry), 32-bit index arithmetic, every
// load of a thread issued at once (the launch is latency-bound: a few hundred
// KB).  The batch totals are reduced per block and then across blocks through
// two accumulators in the workspace header; the last block to finish
// publishes them and zeroes the accumulators for the next call, so no
// separate memset and no per-element atomics are needed.
#include "dcp_internal.cuh"

namespace dcp {
namespace {

constexpr int kThreads = 256, kWarps = kThreads / 32;

struct TransferArgs {
    int N, I, bs, B, max_blocks;
    int64_t num_blocks;
    const int32_t* seq_lens;
    const int32_t* block_tables;
    int32_t* counts;
    int32_t* blocks;
    int32_t* fills;
    int64_t* totals;  // [2]: slots moved, tokens moved (optional)
    WsHeader* hdr;
};

__global__ void __launch_bounds__(kThreads) transfer_blocks_kernel(TransferArgs a) {
    const uint32_t M = (uint32_t)a.max_blocks, B = (uint32_t)a.B;
    const uint32_t total = (uint32_t)a.N * B * M;
    unsigned long long slots = 0, toks = 0;  // this thread's share of the totals
    for (uint32_t i = blockIdx.x * kThreads + threadIdx.x; i < total; i += gridDim.x * kThreads) {
        const uint32_t p = i / M, k = i - p * M;  // p = r * B + b
        const uint32_t r = p / B, b = p - r * B;
        // both loads are in bounds for every i, so they issue together; the
        // table entry is used only when it is listed
        const int32_t L = a.seq_lens[b];
        const int32_t raw = a.block_tables[i];
        const uint32_t len = L > 0 ? local_len32((uint32_t)L, (int)r, a.N, a.I) : 0u;
        const uint32_t need = len / (uint32_t)a.bs + (len % (uint32_t)a.bs != 0);
        const uint32_t cnt = need < M ? need : M;
        if (k == 0) {
            if (need > M) raise_err(&a.hdr->err, DCP_DEV_ERR_TABLE);
            a.counts[p] = (int32_t)cnt;
            slots += (unsigned long long)need * (unsigned long long)a.bs;
            toks += len;
        }
        int32_t id = -1, fill = 0;
        if (k < cnt) {
            id = raw;
            if (id < 0 || id >= a.num_blocks) {
                raise_err(&a.hdr->err, DCP_DEV_ERR_BLOCK_ID);
                id = -1;
            }
            const uint32_t rest = len - k * (uint32_t)a.bs;  // k < cnt, so rest > 0
            fill = (int32_t)(rest < (uint32_t)a.bs ? rest : (uint32_t)a.bs);
        }
        if (a.blocks) a.blocks[i] = id;
        if (a.fills) a.fills[i] = fill;
    }
    if (a.totals == nullptr) return;

    for (int o = 16; o > 0; o >>= 1) {
        slots += __shfl_xor_sync(0xffffffffu, slots, o);
        toks += __shfl_xor_sync(0xffffffffu, toks, o);
    }
    __shared__ unsigned long long part[kWarps][2];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        part[warp][0] = slots;
        part[warp][1] = toks;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long s = 0, t = 0;
        for (int w = 0; w < kWarps; ++w) {
            s += part[w][0];
            t += part[w][1];
        }
        if (s) atomicAdd(&a.hdr->xfer_acc[0], s);
        if (t) atomicAdd(&a.hdr->xfer_acc[1], t);
        __threadfence();
        if (atomicAdd(&a.hdr->xfer_done, 1u) == gridDim.x - 1) {
            __threadfence();
            // atomic reads see every block's device-scope additions
            const unsigned long long S = atomicAdd(&a.hdr->xfer_acc[0], 0ull);
            const unsigned long long T = atomicAdd(&a.hdr->xfer_acc[1], 0ull);
            a.totals[0] = (int64_t)S;
            a.totals[1] = (int64_t)T;
            a.hdr->xfer_acc[0] = 0;
            a.hdr->xfer_acc[1] = 0;
            a.hdr->xfer_done = 0;
        }
    }
}

}  // namespace

cudaError_t launch_transfer_blocks(int N, int I, int bs, int B, int max_blocks, int64_t num_blocks,
                                   const int32_t* seq_lens, const int32_t* block_tables, int32_t* counts,
                                   int32_t* blocks, int32_t* fills, int64_t* totals, void* workspace,
                                   cudaStream_t s) {
    TransferArgs a;
    a.N = N; a.I = I; a.bs = bs; a.B = B; a.max_blocks = max_blocks; a.num_blocks = num_blocks;
    a.seq_lens = seq_lens; a.block_tables = block_tables; a.counts = counts; a.blocks = blocks; a.fills = fills;
    a.totals = totals;
    a.hdr = reinterpret_cast<WsHeader*>(workspace);
    const int64_t total = (int64_t)N * B * max_blocks;
    int64_t grid = (total + kThreads - 1) / kThreads;
    if (grid > 152 * 8) grid = 152 * 8;
    if (grid < 1) grid = 1;
    transfer_blocks_kernel<<<(unsigned)grid, kThreads, 0, s>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace dcp

// Head-tail (zigzag) partition of prefill tokens over K PCP ranks.
//
// "Breaking the Long-Sequence Inference Bottleneck ...", section 4 ("Head-tail
// concatenation strategy" and "Minimal state progression: PCP Size = 2"): a
// request's new tokens are padded to a multiple of 2K and cut into 2K equal
// chunks; rank k holds chunk k (head) followed by chunk 2K - 1 - k (tail), so
// every rank's causal work is the same.  Row j of request b in the gathered
// order (rank 0's rows, then rank 1's, ...) is rank j / 2c's row j % 2c, with
// c the chunk length: a closed form per row, one thread each.
#include "dcp_internal.cuh"

namespace dcp {
namespace {

__global__ void pcp_partition_kernel(int K, int B, const int32_t* ctx_lens, const int32_t* q_lens, int max_q,
                                     int32_t* pos, int32_t* padded_lens, uint32_t* err) {
    const int64_t total = (int64_t)B * max_q;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int b = (int)(i / max_q), j = (int)(i % max_q);
        const int64_t n = q_lens[b] > 0 ? q_lens[b] : 0;
        const int64_t aligned = (n + 2 * K - 1) / (2 * K) * (2 * K);
        if (j == 0) {
            padded_lens[b] = (int32_t)aligned;
            if (aligned > max_q) raise_err(err, DCP_DEV_ERR_ROWS);
        }
        int32_t p = -1;
        if (aligned <= max_q && j < aligned) {
            const int64_t c = aligned / (2 * K);
            const int64_t k = j / (2 * c), h = (j % (2 * c)) / c, jj = j % c;
            const int64_t chunk = h == 0 ? k : 2 * K - 1 - k;
            const int64_t rel = chunk * c + jj;
            if (rel < n) p = (int32_t)(ctx_lens[b] + rel);
        }
        pos[i] = p;
    }
}

}  // namespace

cudaError_t launch_pcp_partition(int K, int B, const int32_t* ctx_lens, const int32_t* q_lens, int max_q, int32_t* pos,
                                 int32_t* padded_lens, uint32_t* err, cudaStream_t s) {
    const int64_t total = (int64_t)B * max_q;
    int64_t grid = (total + 255) / 256;
    if (grid > 152 * 16) grid = 152 * 16;
    if (grid < 1) grid = 1;
    pcp_partition_kernel<<<(unsigned)grid, 256, 0, s>>>(K, B, ctx_lens, q_lens, max_q, pos, padded_lens, err);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace dcp

// Internal declarations shared by the libdcp translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include <utility>

#include "../../include/dcp.h"

namespace dcp {

// ---------------------------------------------------------------------------
// Interleaved ownership, closed forms.
// ("Breaking the Long-Sequence Inference Bottleneck ...", section 2: rank of
// token t is floor(t / I) mod N; "vLLM DCP and PCP", Deep Dive 5: the local
// lengths.)  A rank stores its tokens in token order, so token t sits at local
// position floor(t / (N I)) * I + t mod I, and the first L tokens leave
// floor(L / (N I)) * I + clamp(L mod (N I) - r I, 0, I) tokens on rank r.
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ int64_t owner_rank(int64_t t, int N, int I) {
    return (t / I) % N;
}
__host__ __device__ __forceinline__ int64_t local_pos(int64_t t, int N, int I) {
    const int64_t period = (int64_t)N * I;
    return (t / period) * I + t % I;
}
__host__ __device__ __forceinline__ int64_t local_len(int64_t L, int r, int N, int I) {
    const int64_t period = (int64_t)N * I;
    int64_t extra = L % period - (int64_t)r * I;
    extra = extra < 0 ? 0 : (extra > I ? I : extra);
    return (L / period) * I + extra;
}
__host__ __device__ __forceinline__ int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }
// local_len for L < 2^31 with 32-bit divisions only (the period N I may
// exceed 32 bits; then every token lies in the first period).
__host__ __device__ __forceinline__ uint32_t local_len32(uint32_t L, int r, int N, int I) {
    const uint64_t period = (uint64_t)N * (uint64_t)I;
    uint32_t full = 0, rem = L;
    if (period <= L) {
        full = L / (uint32_t)period;
        rem = L - full * (uint32_t)period;
    }
    int64_t extra = (int64_t)rem - (int64_t)r * I;
    extra = extra < 0 ? 0 : (extra > I ? I : extra);
    return full * (uint32_t)I + (uint32_t)extra;
}

// ---------------------------------------------------------------------------
// Workspace layout (all offsets 256-byte aligned):
//   header        256 B: error word, total chunk count
//   unit_start    int64[U + 1]   chunk prefix over units u = (b*Hkv + kvh)*N + r
//   seg_base      int32[G + 1]   partial-slot prefix over merge groups
//   counters      uint32[G]      arrivals per group (fused merge)
//   part_o        fp32[seg_max][rows][Dv]
//   part_lse      fp32[seg_max][rows]
//   qprep         kernel-specific staging of the query (fp8 MLA kernel), else empty
// ---------------------------------------------------------------------------
struct WsHeader {
    uint32_t err;
    uint32_t n_empty;      // merge groups that own no chunk (listed at off_empty)
    int64_t total_chunks;
    uint64_t plan_key;     // the arguments the plan was made for (plan_key_of)
    // block-transfer totals: per-block partials accumulate here, the last
    // block to finish publishes them and puts both words back to zero
    unsigned long long xfer_acc[2];
    uint32_t xfer_done;
};
static_assert(sizeof(WsHeader) <= 256, "the workspace header is 256 bytes");

struct WsLayout {
    size_t off_units, off_seg_base, off_counters, off_wfirst, off_empty, off_part_o, off_part_lse, off_qprep, total;
};

__host__ __forceinline__ size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// wfirst[w]: where worker w's chunk range starts (W workers), written by a
// plan made ahead of its attention call, so that a worker starts with one
// load instead of a search.  empty[i]: the merge groups that own no chunk.
struct WorkerStart {
    int64_t u0;              // the unit holding the worker's first chunk
    int64_t ustart, uend;    // that unit's chunk range [unit_start[u0], unit_start[u0 + 1])
    int64_t pad;
};
__host__ inline WsLayout ws_layout(int64_t U, int64_t G, int64_t seg_max, int64_t rows, int64_t Dv,
                                   size_t qprep_bytes, int64_t W) {
    WsLayout l;
    size_t o = 256;
    l.off_units = o; o = align256(o + sizeof(int64_t) * (size_t)(U + 1));
    l.off_seg_base = o; o = align256(o + sizeof(int32_t) * (size_t)(G + 1));
    l.off_counters = o; o = align256(o + sizeof(uint32_t) * (size_t)(G + 1));
    l.off_wfirst = o; o = align256(o + sizeof(WorkerStart) * (size_t)W);
    l.off_empty = o; o = align256(o + sizeof(int32_t) * (size_t)G);
    l.off_part_o = o; o = align256(o + sizeof(float) * (size_t)seg_max * rows * Dv);
    l.off_part_lse = o; o = align256(o + sizeof(float) * (size_t)seg_max * rows);
    l.off_qprep = o; o = align256(o + qprep_bytes);
    l.total = o;
    return l;
}

// Count kernel launches (dcp_launch_count).
void count_launches(int n);

// Programmatic dependent launch.  A kernel started by launch_pdl may begin
// while the kernel before it on the stream is still running: every thread
// calls pdl_wait() before it touches anything that kernel (or earlier work)
// wrote, and before it exits, so that its own completion implies its
// predecessor's.  pdl_trigger() lets the next launch_pdl kernel begin.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
__host__ inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                       Args&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Raise device error bits.
__device__ __forceinline__ void raise_err(uint32_t* err, uint32_t bit) { atomicOr(err, bit); }

// Chunks of unit u = ((b * Hkv + kvh) * N + r) with the plan's checks:
// seq_len < Tq -> DCP_DEV_ERR_TOKEN (no chunk); a local length that differs
// from the closed form -> DCP_DEV_ERR_STALE (the smaller one is used); more
// blocks than max_blocks -> DCP_DEV_ERR_TABLE (clamped).  Errors are raised
// only when `err` is non-null.  With lens_given the local lengths are the
// caller's (sparse staging: any length up to the closed form) and only the
// cap applies.  Lengths are int32, so 32-bit closed forms.
__device__ __forceinline__ int64_t unit_chunks(int64_t u, int N, int I, int Hkv, int B, int Tq, int bs, int CH,
                                               int max_blocks, const int32_t* seq_lens, const int32_t* local_lens,
                                               uint32_t* err, bool lens_given = false) {
    const int r = (int)(u % N);
    const int b = (int)((u / N) / Hkv);
    const int32_t L = seq_lens[b];
    const int32_t given = local_lens[(int64_t)r * B + b];
    if (L < Tq) {
        if (err) raise_err(err, DCP_DEV_ERR_TOKEN);
        return 0;
    }
    const uint32_t expect = local_len32((uint32_t)L, r, N, I);
    if (given != (int32_t)expect && err && !lens_given) raise_err(err, DCP_DEV_ERR_STALE);
    uint32_t n = given < 0 ? 0u : ((uint32_t)given < expect ? (uint32_t)given : expect);
    if (n / (uint32_t)bs + (n % (uint32_t)bs != 0) > (uint32_t)max_blocks) {
        if (err) raise_err(err, DCP_DEV_ERR_TABLE);
        n = (uint32_t)max_blocks * (uint32_t)bs;
    }
    return n / (uint32_t)CH + (n % (uint32_t)CH != 0);
}

// Which worker (of W over P chunks, worker w owning [w*P/W, (w+1)*P/W)) owns chunk x.
__host__ __device__ __forceinline__ int64_t worker_of(int64_t x, int64_t W, int64_t P) {
    return ((x + 1) * W - 1) / P;
}
__host__ __device__ __forceinline__ int64_t worker_begin(int64_t w, int64_t W, int64_t P) {
    return w * P / W;
}

// ---------------------------------------------------------------------------
// The work plan shared by the attention kernels.
//   unit u = ((b * Hkv + kvh) * N + r): rank r's tokens of request b, KV head kvh;
//   chunk: CH consecutive local positions of one unit (CH divides block_size
//   or is a multiple of it that stays inside one block);
//   merge group: decode mode = (b, kvh) (all ranks), partial mode = unit.
// ---------------------------------------------------------------------------
struct PlanArgs {
    int N, I, bs, Hkv, Tq, CH;
    int B;
    int partial_mode;  // 0: groups (b, kvh); 1: groups (b, kvh, r)
    int64_t W;         // workers of the attention kernel that follows
    int lens_given;    // local lengths are given, not derived (sparse staging)
    int max_blocks;
    int worker_starts;    // also write each worker's first unit (a plan made ahead)
    uint64_t plan_key;
    const int32_t* seq_lens;
    const int32_t* local_lens;
    uint8_t* ws;
    WsLayout lay;
    int64_t U, G;
};

void launch_plan(const PlanArgs& a, cudaStream_t s);

// Attention arguments common to the kernels.
struct AttnArgs {
    int N, I, bs, Hq, Hkv, Dk, Dv, Tq, G;  // G = Hq / Hkv (query heads per KV head)
    int B, max_blocks, layout, partial_mode, out_dtype, CH;
    int64_t num_blocks, U, Gn, W;           // Gn: merge groups
    float softmax_scale, kv_scale;
    const void* q;
    const void* k_pool;
    const void* v_pool;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const int32_t* local_lens;
    float* out_partial;
    float* lse_partial;
    void* out;
    float* lse;
    uint8_t* ws;
    WsLayout lay;
    int rows;        // rows per group = Tq * G
    int lens_given;  // local lengths are given (sparse staging): they also bound each rank's tokens
    int worker_starts;  // the plan holds each worker's first unit (wfirst)
    uint64_t plan_key;  // must equal the workspace header's (a plan for other arguments: DCP_DEV_ERR_PLAN)
};

// Causal prefill of a PCP-partitioned chunk: per-rank partials of query rows
// with explicit global positions (GQA, bf16).
struct PrefillArgs {
    int N, I, bs, Hq, Hkv, G, D, Tq, B, max_blocks;
    int64_t num_blocks;
    float softmax_scale;
    const void* q;           // [B][Tq][Hq][D]
    const int32_t* q_pos;    // [B][Tq], -1 = padding
    const void* k_pool;
    const void* v_pool;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const int32_t* local_lens;
    float* out_partial;      // [N][B][Tq][Hq][D]
    float* lse_partial;      // [N][B][Tq][Hq]
    uint8_t* ws;
};
bool prefill_supported(const dcp_params& p);
cudaError_t launch_prefill_partial(const PrefillArgs& a, cudaStream_t s);  // mma.sync, D 64 / 128
bool prefill_tc_supported(const PrefillArgs& a);                          // tcgen05, D 128
cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s);

// DCP-localised sparse attention: candidate localisation and the staging of
// every (rank, query row) candidate list as a contiguous request
struct SparseStageArgs {
    int N, I, R, Tq, B, k, kpad, bs, max_blocks;  // R = query rows (B * Tq); kpad = k rounded up to 64
    int row_bytes;                                 // cache row: Dk x element size
    int64_t num_blocks;
    const int32_t* cand;                           // [R][k] global positions, -1 unused
    const int32_t* seq_lens;                       // [B]
    int32_t* local;                                // [N][R][k] written (first counts entries)
    int32_t* counts;                               // [N][R] written
    const int32_t* block_tables;                   // [N][B][max_blocks]
    const void* k_pool;
    void* st_pool;                                 // [N][R][kpad] rows
    int32_t* st_tables;                            // [N][R][kpad / 64]
    int32_t* st_lens;                              // [R]: N kpad
    uint32_t* err;
};
cudaError_t launch_sparse_localize(int N, int I, int rows, int Tq, int k, const int32_t* cand, const int32_t* seq_lens,
                                   int32_t* local, int32_t* counts, uint32_t* err, cudaStream_t s);
// localisation and staging in one launch (one CTA per rank and row)
cudaError_t launch_sparse_stage(const SparseStageArgs& a, cudaStream_t s);

// head-tail prefill partition over K PCP ranks
cudaError_t launch_pcp_partition(int K, int B, const int32_t* ctx_lens, const int32_t* q_lens, int max_q, int32_t* pos,
                                 int32_t* padded_lens, uint32_t* err, cudaStream_t s);

// generic CUDA-core path (any dtype / width); writes all segment partials,
// then launch_segment_merge combines them.
bool generic_supported(const dcp_params& p);
int64_t generic_workers(int num_sms);
int generic_chunk(int bs);
cudaError_t launch_attn_generic(const AttnArgs& a, int q_dtype, int kv_dtype, cudaStream_t s);
cudaError_t launch_segment_merge(const AttnArgs& a, cudaStream_t s);

// bf16 GQA path on mma.sync with query-group packing and a fused merge.
bool gqa_mma_supported(const dcp_params& p);
int64_t gqa_mma_workers(int num_sms);
cudaError_t launch_attn_gqa_mma(const AttnArgs& a, cudaStream_t s);

// MLA (128 heads, 576/512 latent, bf16 or fp8 cache) on CTA pairs with
// tcgen05 pair MMAs (attn_mla_pair.cu); writes segment partials, then
// launch_segment_merge combines them.  The fp8-cache form (kind::f8f6f4,
// two-term query and probabilities) first runs a query preparation kernel; the
// prepared query lives in the workspace's qprep region (mla_f8_qprep_bytes).
bool mla_tc_supported(const dcp_params& p);
int64_t mla_tc_workers(int num_sms, int Tq);
cudaError_t launch_attn_mla_tc(const AttnArgs& a, int kv_dtype, cudaStream_t s);
size_t mla_f8_qprep_bytes(int64_t B, int Tq);

// blocks moved under prefill-decode disaggregation (dcp_transfer_blocks)
cudaError_t launch_transfer_blocks(int N, int I, int bs, int B, int max_blocks, int64_t num_blocks,
                                   const int32_t* seq_lens, const int32_t* block_tables, int32_t* counts,
                                   int32_t* blocks, int32_t* fills, int64_t* totals, void* workspace,
                                   cudaStream_t s);

// standalone merge for dcp_lse_merge
cudaError_t launch_lse_merge(int N, int64_t rows, int Dv, const float* o_parts, const float* lse_parts,
                             void* out, int out_dtype, float* lse, cudaStream_t s);

// slot mapping + cache write
struct SlotArgs {
    int N, I, bs, B, layout, Hkv, Dk, Dv, kv_esize, max_blocks;
    int64_t T, num_blocks;
    const int32_t* seq_lens;
    const int32_t* tok_req;
    const int64_t* tok_pos;
    const int32_t* block_tables;
    int8_t* owner;
    int64_t* slots;
    int32_t* local_lens;
    int32_t* virt_blocks;
    int32_t* rank_blocks;
    const void* new_k;
    const void* new_v;
    void* k_pool;
    void* v_pool;
    uint32_t* err;
};
cudaError_t launch_slot_mapping(const SlotArgs& a, cudaStream_t s);

// ---------------------------------------------------------------------------
// Small device helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(((uint32_t)b) << 16);
}

// fp8 e4m3fn -> fp32 through the hardware pair conversion (e4m3x2 -> f16x2).
__device__ __forceinline__ float2 fp8x2_to_float2(uint16_t two) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
    __half2 h = *reinterpret_cast<__half2*>(&h2);
    return __half22float2(h);
}

__device__ __forceinline__ float load_elem(const void* base, int64_t idx, int dtype) {
    if (dtype == DCP_F32) return reinterpret_cast<const float*>(base)[idx];
    if (dtype == DCP_BF16) return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(base)[idx]);
    // fp8: decode one byte (pair conversion with a zero partner)
    const uint8_t v = reinterpret_cast<const uint8_t*>(base)[idx];
    return fp8x2_to_float2((uint16_t)v).x;
}

__device__ __forceinline__ void store_out(void* out, int64_t idx, float v, int dtype) {
    if (dtype == DCP_F32)
        reinterpret_cast<float*>(out)[idx] = v;
    else
        reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
}

// The output of a merge group that owns no chunk (the plan lists them): out
// (or out_partial) zeros and lse -inf for its rows.  One warp.
__device__ __forceinline__ void write_empty_group(const AttnArgs& a, int64_t g, int lane) {
    int b, kvh, r = 0;
    if (a.partial_mode) {
        r = (int)(g % a.N);
        b = (int)((g / a.N) / a.Hkv);
        kvh = (int)((g / a.N) % a.Hkv);
    } else {
        b = (int)(g / a.Hkv);
        kvh = (int)(g % a.Hkv);
    }
    const int64_t total = (int64_t)a.rows * a.Dv;
    for (int64_t e = lane; e < total; e += 32) {
        const int row = (int)(e / a.Dv), d = (int)(e % a.Dv);
        const int t = row / a.G, gq = row % a.G;
        const int64_t orow = ((int64_t)b * a.Tq + t) * a.Hq + (int64_t)kvh * a.G + gq;
        if (a.partial_mode) {
            const int64_t prow = (int64_t)r * a.B * a.Tq * a.Hq + orow;
            a.out_partial[prow * a.Dv + d] = 0.f;
            if (d == 0) a.lse_partial[prow] = -INFINITY;
        } else {
            store_out(a.out, orow * a.Dv + d, 0.f, a.out_dtype);
            if (d == 0 && a.lse) a.lse[orow] = -INFINITY;
        }
    }
}

}  // namespace dcp

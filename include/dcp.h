/*
 * dcp.h -- C ABI of libdcp: decode-context-parallel (DCP) decode attention on
 * one GPU (sm_103a).
 *
 * The method (sources are the pages' titles and sections):
 *  - "Breaking the Long-Sequence Inference Bottleneck: A Deep Dive into vLLM's
 *    Distributed Context Parallelism Architecture", section 2 (interleaved
 *    storage and virtual blocks): token t of a request belongs to rank
 *    floor(t / I) mod N; a virtual block is block_size x N tokens; tokens a
 *    rank does not own get slot -1 and are skipped by the cache write.
 *  - "vLLM DCP and PCP: Decode and Prefill Context Parallelism", Deep Dive 5
 *    (per-rank local lengths: every rank's attention sees its local KV prefix)
 *    and Deep Dive 6 (each rank computes a partial output o_i and its
 *    log-sum-exp L_i over its own KV shard; the exact global output is
 *    O = sum_i a_i o_i / sum_i a_i with a_i = exp(L_i - max_j L_j) and
 *    L = max_j L_j + log sum_i a_i).
 *  - "vLLM Decode Context Parallelism for Long Context Workloads", "The DCP
 *    Execution Process" (every rank uses the full query against its local KV
 *    slice, then partial results are merged with their LSE values).
 *
 * Here all N ranks are virtual: their KV shards live in one physical block
 * pool on one GPU, and the merge runs through device memory, not collectives.
 *
 * Conventions for every call:
 *  - All pointers except `params`, `bytes` and `bits` are DEVICE pointers,
 *    owned and allocated by the caller.  The library allocates nothing; the
 *    only scratch is the caller's workspace (see dcp_workspace_size).
 *  - Work is enqueued on `stream` (asynchronous); nothing synchronizes except
 *    dcp_get_error.
 *  - Integers: seq/local lengths int32, token positions and slots int64.
 *  - Host-side validation returns DCP_ERR_INVALID_ARG / DCP_ERR_UNSUPPORTED
 *    before anything is enqueued.  Device-side checks never trap: a bad block
 *    id, token or stale length sets a bit in the workspace's error word and
 *    the offending access is skipped; read it with dcp_get_error.
 *
 * Data layouts (row-major, innermost last):
 *  - q           [B][Tq][Hq][Dk]          q_dtype (f32 or bf16)
 *  - GQA pools   k_pool [num_blocks][Hkv][block_size][Dk],
 *                v_pool [num_blocks][Hkv][block_size][Dv]      kv_dtype
 *  - MLA pool    k_pool [num_blocks][block_size][Dk] (latent + RoPE row);
 *                v_pool = NULL: values are the first Dv columns of that row
 *  - a slot s addresses block s / block_size, offset s % block_size
 *  - block_tables [N][B][max_blocks] int32: block ids of rank r's local
 *                blocks for request b, in local order (unused entries: any)
 *  - seq_lens    [B] global length of each request, including its Tq newest
 *                tokens (the queries); query t sees global positions
 *                0 .. seq_lens[b] - Tq + t
 *  - local_lens  [N][B] tokens of request b that rank r owns
 *  - out         [B][Tq][Hq][Dv] out_dtype;  lse [B][Tq][Hq] fp32 (natural log)
 *  - out_partial [N][B][Tq][Hq][Dv] fp32;  lse_partial [N][B][Tq][Hq] fp32;
 *                a rank with no visible token gives zeros and -inf.
 *  - GQA head mapping: query head h reads KV head h / (Hq / Hkv).
 *  - Slots of a rank's last block past its local length must hold finite
 *    values (a zero-initialised pool, or slots written earlier): the tensor-
 *    core kernels read whole 16/64-token tiles and weight those slots by 0.
 */
#ifndef DCP_H_
#define DCP_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime.h>

#ifdef __cplusplus
extern "C" {
#endif

/* return codes */
#define DCP_OK 0
#define DCP_ERR_INVALID_ARG 1   /* a shape, pointer or enum failed host validation */
#define DCP_ERR_UNSUPPORTED 2   /* valid, but no kernel here handles this combination */
#define DCP_ERR_CUDA 3          /* a CUDA runtime call failed (launch, copy, attribute) */
#define DCP_ERR_WORKSPACE 4     /* workspace NULL or smaller than dcp_workspace_size */

/* bits of the device error word (dcp_get_error) */
#define DCP_DEV_ERR_BLOCK_ID 0x1u   /* a block id outside [0, num_blocks) was read */
#define DCP_DEV_ERR_TOKEN 0x2u      /* a token's request or position lies outside its request */
#define DCP_DEV_ERR_TABLE 0x4u      /* a rank needs more blocks than max_blocks */
#define DCP_DEV_ERR_STALE 0x8u      /* local_lens disagree with seq_lens under (N, I) */
#define DCP_DEV_ERR_TIMEOUT 0x10u   /* a bounded wait inside a kernel gave up (or a tensor-core
                                       kernel found its shared memory off the 1024-byte boundary
                                       its swizzled layouts need, and did nothing) */
#define DCP_DEV_ERR_ROWS 0x20u      /* a request's padded prefill rows exceed the row capacity */
#define DCP_DEV_ERR_PLAN 0x40u      /* dcp_decode_attention_planned found no plan in the workspace made
                                       (by dcp_decode_plan) for its arguments, and did nothing */

typedef enum { DCP_F32 = 0, DCP_BF16 = 1, DCP_FP8_E4M3 = 2 } dcp_dtype;
typedef enum { DCP_LAYOUT_GQA = 0, DCP_LAYOUT_MLA = 1 } dcp_layout;

typedef struct dcp_params {
    int32_t N;             /* virtual DCP ranks, >= 1 */
    int32_t I;             /* interleave size: consecutive tokens per rank turn, >= 1 */
    int32_t block_size;    /* tokens per physical block of one rank, >= 1 */
    int32_t layout;        /* dcp_layout */
    int32_t Hq;            /* query heads */
    int32_t Hkv;           /* KV heads (MLA: 1, shared by every query head) */
    int32_t Dk;            /* key width (MLA: latent + RoPE, e.g. 512 + 64) */
    int32_t Dv;            /* value width (MLA: <= Dk, the leading columns) */
    int32_t Tq;            /* query tokens per request, >= 1 (1 = plain decode) */
    int32_t q_dtype;       /* DCP_F32 or DCP_BF16 */
    int32_t kv_dtype;      /* DCP_F32, DCP_BF16 or DCP_FP8_E4M3 */
    int32_t out_dtype;     /* DCP_F32 or DCP_BF16 */
    float kv_scale;        /* fp8 KV: stored value x kv_scale; otherwise must be 1 */
    float softmax_scale;   /* scores are softmax_scale * (q . k) */
} dcp_params;

/* Library ABI version (this header: 1). */
int dcp_version(void);

/* Static text for a return code. */
const char* dcp_error_string(int code);

/* Kernel launches this library has enqueued since it was loaded (all
 * devices, all calls): lets a caller count the GPU work of a region. */
uint64_t dcp_launch_count(void);

/* Name of the attention kernel that dcp_partial_attention and
 * dcp_decode_attention select for these params ("gqa_mma", "mla_tcgen05",
 * "generic"), or NULL if the params are invalid or no kernel supports them. */
const char* dcp_attention_kernel(const dcp_params* params);

/*
 * Bytes of scratch that dcp_partial_attention / dcp_decode_attention /
 * dcp_slot_mapping need for these params and batch size B on the CURRENT
 * device (the bound depends on its SM count).  max_seq_len bounds
 * seq_lens[b] (>= 1).  The workspace holds the device error word, the work
 * plan, the arrival counters of the fused merge and the split partials.
 */
int dcp_workspace_size(const dcp_params* params, int32_t B, int64_t max_seq_len, size_t* bytes);

/* Zero a freshly allocated workspace (error word and counters).  Call once
 * after allocation; later calls keep the workspace consistent themselves. */
int dcp_workspace_init(void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Synchronize `stream`, read the device error word of `workspace` into *bits
 * (0 = clean; DCP_DEV_ERR_* bits otherwise) and clear it.
 */
int dcp_get_error(void* workspace, cudaStream_t stream, uint32_t* bits);

/*
 * Token ownership, local lengths, virtual-block counts, slots and the cache
 * write ("Breaking the Long-Sequence Inference Bottleneck ...", section 2:
 * interleave rule, virtual block, slot mapping with -1 skip; "vLLM DCP and
 * PCP", Deep Dive 5: local lengths).
 *
 * For the B requests (global lengths seq_lens[B]) writes, each output
 * optional (NULL skips it):
 *   local_lens[N][B]   tokens of request b owned by rank r
 *   virt_blocks[B]     ceil(seq_lens[b] / (block_size * N))
 *   rank_blocks[N][B]  ceil(local_lens[r][b] / block_size): physical blocks
 *                      rank r needs for request b
 * For the T tokens (tok_req[T], tok_pos[T]) writes:
 *   owner[T]           owning rank floor(pos / I) mod N
 *   slots[N][T]        owner's slot block_tables[r][b][lp / bs] * bs + lp % bs
 *                      (lp = the token's local position: the number of earlier
 *                      tokens of the request that the same rank owns), and -1
 *                      in every other rank's row; needs block_tables
 * and, when new_k != NULL (needs block_tables and k_pool), copies each
 * token's row into its owner's slot: GQA new_k [T][Hkv][Dk] -> k_pool,
 * new_v [T][Hkv][Dv] -> v_pool; MLA new_k [T][Dk] -> k_pool (new_v NULL).
 * Rows are stored as given (kv_dtype; no requantisation).
 * Device checks: token outside its request -> DCP_DEV_ERR_TOKEN; local block
 * index >= max_blocks -> DCP_DEV_ERR_TABLE; block id outside
 * [0, num_blocks) -> DCP_DEV_ERR_BLOCK_ID; the token's slots stay -1 and its
 * row is not written.  The workspace needs at least dcp_workspace_size bytes
 * for (params, B).  owner holds ranks as int8: with owner != NULL, N must be
 * at most 127 (DCP_ERR_INVALID_ARG otherwise).
 */
int dcp_slot_mapping(const dcp_params* params, int32_t B, const int32_t* seq_lens,
                     int64_t T, const int32_t* tok_req, const int64_t* tok_pos,
                     const int32_t* block_tables, int32_t max_blocks, int64_t num_blocks,
                     int8_t* owner, int64_t* slots, int32_t* local_lens,
                     int32_t* virt_blocks, int32_t* rank_blocks,
                     const void* new_k, const void* new_v, void* k_pool, void* v_pool,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Blocks to move under prefill-decode disaggregation ("Breaking the
 * Long-Sequence Inference Bottleneck ...", section 2, "Practical
 * considerations for PD disaggregation"): KV moves between nodes in whole
 * blocks, and a block that holds no token need not move.  For every rank r
 * and request b (global lengths seq_lens[B], device int32), lists the physical
 * blocks that hold at least one of the request's tokens, in block-table order,
 * with their token counts.  A rank fills its blocks in local-position order,
 * so these are the first ceil(local_len / block_size) table entries, all full
 * but the last.
 *   counts[N][B]              (required) listed blocks per rank and request
 *   blocks[N][B][max_blocks]  (optional) their ids, -1 after the last
 *   fills[N][B][max_blocks]   (optional) tokens in each block, 0 after the last
 *   totals[2]                 (optional, 8-byte aligned, int64) the batch's
 *                             block slots moved (sum of counts * block_size)
 *                             and tokens moved; totals[1] / totals[0] is the
 *                             fill of the transfer
 * All outputs are device memory owned by the caller; block_tables as for
 * dcp_slot_mapping.  Device checks: a listed table entry outside
 * [0, num_blocks) -> DCP_DEV_ERR_BLOCK_ID (listed as -1); a rank needing more
 * than max_blocks blocks -> DCP_DEV_ERR_TABLE (the list stops at max_blocks;
 * totals still count every needed block).  N * B * max_blocks must fit in
 * int32 (else DCP_ERR_INVALID_ARG).
 * workspace: its 256-byte header only (error word and the totals'
 * accumulators, zeroed once by dcp_workspace_init and left zero by every
 * call); calls sharing a workspace must be ordered on one stream.
 * Asynchronous on `stream`.
 */
int dcp_transfer_blocks(const dcp_params* params, int32_t B, const int32_t* seq_lens,
                        const int32_t* block_tables, int32_t max_blocks, int64_t num_blocks,
                        int32_t* counts, int32_t* blocks, int32_t* fills, int64_t* totals,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Head-tail (zigzag) partition of prefill tokens over K PCP ranks ("Breaking
 * the Long-Sequence Inference Bottleneck ...", section 4, "Head-tail
 * concatenation strategy" and its PCP Size = 2 walk-through).  Request b's new
 * tokens are the global positions ctx_lens[b] .. ctx_lens[b] + q_lens[b] - 1;
 * their count is padded up to a multiple of 2K and cut into 2K equal chunks of
 * c tokens; PCP rank k holds chunk k followed by chunk 2K - 1 - k.
 *   pos[B][max_q]      (device int32) row j of request b in the gathered order
 *                      (rank 0's 2c rows, then rank 1's, ...: the order an
 *                      AllGather of the ranks' queries leaves them in): its
 *                      global position, or -1 for padding (an aligned slot
 *                      past the request's last token, or j >= the aligned
 *                      length)
 *   padded_lens[B]     (device int32) the aligned length of each request
 * K >= 1; a request whose aligned length exceeds max_q gets all -1 rows and
 * DCP_DEV_ERR_ROWS.  ctx_lens / q_lens: device int32 [B].  workspace: its
 * error word only (>= 256 bytes).  Asynchronous on `stream`.
 */
int dcp_pcp_partition(int32_t K, int32_t B, const int32_t* ctx_lens, const int32_t* q_lens, int32_t max_q,
                      int32_t* pos, int32_t* padded_lens, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream);

/*
 * Causal prefill attention of PCP-gathered query rows against the DCP-sharded
 * cache ("Breaking the Long-Sequence Inference Bottleneck ...", section 5,
 * AllGather Q path: with the full query set, prefill is the DCP flow; "vLLM
 * DCP and PCP", Deep Dive 6: per-rank partials and their exact LSE merge).
 * Query row t of request b is q[b][t] ([B][Tq][Hq][Dk], the gathered order
 * dcp_pcp_partition produces) at global position q_pos[b][t] (device int32,
 * -1 = padding); it attends to the request's tokens 0 .. q_pos, which must
 * already be in the cache (seq_lens[b] = cached tokens, including the chunk
 * itself; a position >= seq_lens[b] raises DCP_DEV_ERR_TOKEN and the row is
 * treated as padding).  For every virtual rank r:
 *   out_partial[r][b][t][h][:]  (required, fp32) the rank's normalised partial
 *   lse_partial[r][b][t][h]     (required, fp32) its natural-log LSE (-inf when
 *                                the rank holds none of the row's tokens)
 * and, when `out` is given, the merged output out[b][t][h][:] (params'
 * out dtype) and lse[b][t][h] (optional).  Padding rows get zeros and -inf.
 * Layouts, block tables, local lengths, device checks and workspace (error
 * word only, >= 256 bytes) as for dcp_partial_attention; params->Tq is
 * ignored (Tq is the row count here).  GQA, bf16 query and cache, Dk = Dv in
 * {64, 128}, Hq / Hkv dividing 16; other combinations return
 * DCP_ERR_UNSUPPORTED.  Asynchronous on `stream`.
 */
int dcp_prefill_attention(const dcp_params* params, int32_t B, int32_t Tq, const void* q, const int32_t* q_pos,
                          const void* k_pool, const void* v_pool, int64_t num_blocks, const int32_t* block_tables,
                          int32_t max_blocks, const int32_t* seq_lens, const int32_t* local_lens,
                          float* out_partial, float* lse_partial, void* out, float* lse, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream);

/*
 * DCP-localised sparse (top-k) attention, MLA layout (the GLM-5.3
 * context-parallelism page, "What DP and TP leave unresolved": sparse MLA attends to a selected set of 2,048 tokens per query,
 * chosen by an indexer; "vLLM DCP and PCP", its source-and-test table: under
 * DCP the candidates are localised to the ranks that own them, and the exact
 * result is the LSE merge of the ranks' partials).
 *
 * Query row i = b * Tq + t (params->Tq query tokens per request, at
 * positions seq_lens[b] - Tq + t) attends to the candidate positions
 * cand[i][0..k) (device int32, global positions of request b, -1 = unused;
 * a candidate past the row's own position raises DCP_DEV_ERR_TOKEN and is
 * dropped).  N <= 32.
 *
 * dcp_sparse_localize: for every rank r and row i, rank r's candidates in
 * list order at their local positions: local[r][i][0..counts[r][i]) (device
 * int32 [N][B Tq][k], -1 after the last) and counts[r][i] (device int32
 * [N][B Tq]).  workspace: its error word (>= 256 bytes).
 *
 * dcp_sparse_decode_attention: out[i][h][:] (params' out dtype) and lse[i][h]
 * (optional, fp32) = attention of row i's heads over its candidates only.
 * Localises the candidates, stages every (rank, row) candidate list as that
 * rank's local tokens of a contiguous 64-token-paged sequence in the
 * workspace, and runs the dense decode kernels over it with the candidate
 * counts as the ranks' local lengths: their exact merge over the ranks is the
 * result.  q [B][Tq][Hq][Dk] bf16; k_pool / block tables / seq_lens as for
 * dcp_decode_attention (MLA: one latent row per token, no v_pool).  A row
 * with no candidate gets zeros and -inf.  workspace: at least
 * dcp_sparse_workspace_size bytes, zeroed once by dcp_workspace_init
 * (includes a staging cache sized for every rank holding all k candidates of
 * every row).  Non-MLA layouts or non-bf16 queries: DCP_ERR_UNSUPPORTED.
 * Asynchronous on `stream`.
 */
int dcp_sparse_workspace_size(const dcp_params* params, int32_t B, int32_t k, size_t* bytes);
int dcp_sparse_localize(const dcp_params* params, int32_t B, int32_t k, const int32_t* cand, const int32_t* seq_lens,
                        int32_t* local, int32_t* counts, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream);
int dcp_sparse_decode_attention(const dcp_params* params, int32_t B, int32_t k, const void* q, const int32_t* cand,
                                const void* k_pool, int64_t num_blocks, const int32_t* block_tables,
                                int32_t max_blocks, const int32_t* seq_lens, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/*
 * Per-rank partial decode attention ("vLLM DCP and PCP", Deep Dive 6,
 * "Deriving the partial and global outputs"): for every virtual rank r,
 * request b, query token t and head h, with s_j = softmax_scale * q . k_j over
 * the tokens j of rank r that query t may see (local positions
 * < local_len_r(seq_lens[b] - Tq + t + 1)):
 *   lse_partial = log sum_j exp(s_j),  out_partial = sum_j exp(s_j - lse) v_j.
 * Inputs as in the layout notes above; local_lens must be the values
 * dcp_slot_mapping gives for seq_lens (checked on device: DCP_DEV_ERR_STALE).
 */
int dcp_partial_attention(const dcp_params* params, int32_t B, const void* q,
                          const void* k_pool, const void* v_pool, int64_t num_blocks,
                          const int32_t* block_tables, int32_t max_blocks,
                          const int32_t* seq_lens, const int32_t* local_lens,
                          float* out_partial, float* lse_partial,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Exact LSE merge of N partials per row ("vLLM DCP and PCP", Deep Dive 6):
 *   out_partial [N][rows][Dv] fp32, lse_partial [N][rows] fp32 (natural log)
 *   -> out [rows][Dv] (out_dtype: DCP_F32 or DCP_BF16), lse [rows] fp32.
 * Partials with lse = -inf carry no weight; a row whose partials are all
 * -inf gives zeros and -inf.  lse may be NULL.
 */
int dcp_lse_merge(int32_t N, int64_t rows, int32_t Dv, const float* out_partial,
                  const float* lse_partial, void* out, int32_t out_dtype, float* lse,
                  cudaStream_t stream);

/*
 * Fused decode attention: the partial attention of every virtual rank and the
 * exact LSE merge in one pass over the paged cache.  Same inputs as
 * dcp_partial_attention; writes out [B][Tq][Hq][Dv] (out_dtype) and
 * lse [B][Tq][Hq] fp32 (lse may be NULL).  Equal, up to fp32 rounding order,
 * to dcp_partial_attention followed by dcp_lse_merge.
 */
int dcp_decode_attention(const dcp_params* params, int32_t B, const void* q,
                         const void* k_pool, const void* v_pool, int64_t num_blocks,
                         const int32_t* block_tables, int32_t max_blocks,
                         const int32_t* seq_lens, const int32_t* local_lens,
                         void* out, float* lse,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Decode attention in two calls: the work plan made ahead, then the attention.
 *
 * The plan (how the units of every (rank, request, KV head) are cut into
 * chunks and dealt to the kernel's workers, and where each worker's segments
 * merge; "vLLM DCP and PCP", Deep Dive 6, the partials and their merge)
 * depends only on the lengths, not on the cache contents or the query.  A
 * serving step knows the lengths before it writes the step's new tokens into
 * the cache, so the plan can be made beside the cache write (another stream)
 * or once per step for every layer, instead of in front of each attention.
 *
 * dcp_decode_plan writes the plan for (params, B, seq_lens, local_lens,
 * max_blocks) into the workspace (dcp_workspace_size bytes); the device
 * checks of dcp_decode_attention on the lengths run here.
 * dcp_decode_attention_planned then computes exactly what
 * dcp_decode_attention computes, with the same arguments, without planning.
 * It must be ordered after the plan (same stream, or an event) and be made
 * with the same params, B, max_blocks, workspace and the same seq_lens /
 * local_lens pointers whose contents the plan saw.  One plan serves any number
 * of such calls (each call leaves the plan as it found it), until another
 * call on the same workspace writes a different plan (any dcp_decode_attention
 * or dcp_partial_attention call does).  A call whose arguments differ from the
 * plan's raises DCP_DEV_ERR_PLAN on the device and writes no output; a change
 * of the lengths' contents under the same pointers is not detected.
 */
int dcp_decode_plan(const dcp_params* params, int32_t B, const int32_t* seq_lens, const int32_t* local_lens,
                    int32_t max_blocks, void* workspace, size_t workspace_bytes, cudaStream_t stream);
int dcp_decode_attention_planned(const dcp_params* params, int32_t B, const void* q,
                                 const void* k_pool, const void* v_pool, int64_t num_blocks,
                                 const int32_t* block_tables, int32_t max_blocks,
                                 const int32_t* seq_lens, const int32_t* local_lens,
                                 void* out, float* lse,
                                 void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Decode attention for callers that cannot allocate device memory.
 *
 * No passage of the pages has a counterpart to this call: it exists for
 * callers that may not call cudaMalloc (or any allocator) when they run
 * attention -- for example a plugin inside an engine that owns all device
 * memory and hands none out, or code on a path where an allocation's latency
 * or possible failure is not acceptable.  It computes
 * exactly what dcp_decode_attention computes, with the same arguments minus
 * the workspace: the scratch is a buffer of DCP_STATIC_SCRATCH_BYTES that
 * this library declares as a static device array.  Every device that loads
 * the library holds one such buffer until the process exits.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *  - The first call on a device looks up the buffer's device address (with
 *    that device current); make that first call before any stream capture.
 *  - Returns DCP_ERR_WORKSPACE, without enqueuing work, when the problem
 *    needs more scratch than the buffer holds (dcp_workspace_size tells).
 *  - All calls share the one buffer and it keeps the last call's contents:
 *    calls that overlap on the GPU (other streams, other host threads) race
 *    and corrupt each other's results; serialize them.
 *  - Device-side checks still run; their error bits go to the shared
 *    buffer's error word, which each call clears when it starts.  Read them
 *    with dcp_noalloc_get_error.
 */
#define DCP_STATIC_SCRATCH_BYTES (64u << 20)
int dcp_decode_attention_noalloc(const dcp_params* params, int32_t B, const void* q,
                                 const void* k_pool, const void* v_pool, int64_t num_blocks,
                                 const int32_t* block_tables, int32_t max_blocks,
                                 const int32_t* seq_lens, const int32_t* local_lens,
                                 void* out, float* lse, cudaStream_t stream);

/*
 * The error word of dcp_decode_attention_noalloc's static buffer, for the
 * same callers (no passage of the pages has a counterpart either): waits for
 * `stream`, then reads the DCP_DEV_ERR_* bits the most recent call on this
 * device left (0 = clean) into *bits and clears them, like dcp_get_error does
 * for a caller's workspace.  Allocates nothing.
 */
int dcp_noalloc_get_error(cudaStream_t stream, uint32_t* bits);

#ifdef __cplusplus
}
#endif

#endif /* DCP_H_ */

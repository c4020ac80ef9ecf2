// extern "C" entry points of libdcp: host validation, kernel selection,
// workspace layout.  See include/dcp.h for the contract of every call.
#include <math.h>
#include <string.h>

#include <atomic>

#include "dcp_internal.cuh"

namespace dcp {

static std::atomic<uint64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

namespace {

// SM count of the current device, cached per device.  Host threads may call
// in concurrently; they all store the same value, through an atomic.
int device_sms() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= 64) return 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

bool valid_dtype(int d, bool allow_fp8) {
    return d == DCP_F32 || d == DCP_BF16 || (allow_fp8 && d == DCP_FP8_E4M3);
}

int esize(int d) { return d == DCP_F32 ? 4 : (d == DCP_BF16 ? 2 : 1); }

int validate_params(const dcp_params* p) {
    if (!p) return DCP_ERR_INVALID_ARG;
    if (p->N < 1 || p->I < 1 || p->block_size < 1) return DCP_ERR_INVALID_ARG;
    if (p->layout != DCP_LAYOUT_GQA && p->layout != DCP_LAYOUT_MLA) return DCP_ERR_INVALID_ARG;
    if (p->Hq < 1 || p->Hkv < 1 || p->Hq % p->Hkv != 0) return DCP_ERR_INVALID_ARG;
    if (p->Dk < 1 || p->Dv < 1 || p->Tq < 1) return DCP_ERR_INVALID_ARG;
    if (p->layout == DCP_LAYOUT_MLA && (p->Hkv != 1 || p->Dv > p->Dk)) return DCP_ERR_INVALID_ARG;
    if (!valid_dtype(p->q_dtype, false) || !valid_dtype(p->kv_dtype, true) || !valid_dtype(p->out_dtype, false))
        return DCP_ERR_INVALID_ARG;
    if (!(p->kv_scale > 0.f) || !isfinite(p->kv_scale)) return DCP_ERR_INVALID_ARG;
    if (p->kv_dtype != DCP_FP8_E4M3 && p->kv_scale != 1.f) return DCP_ERR_INVALID_ARG;
    if (!isfinite(p->softmax_scale)) return DCP_ERR_INVALID_ARG;
    return DCP_OK;
}

bool aligned16(const void* ptr) { return ((uintptr_t)ptr & 15) == 0; }
bool aligned8(const void* ptr) { return ((uintptr_t)ptr & 7) == 0; }

enum class Kernel { kNone, kGeneric, kGqaMma, kMlaTc };

const char* kernel_name(Kernel k) {
    switch (k) {
        case Kernel::kGqaMma: return "gqa_mma";
        case Kernel::kMlaTc: return "mla_tcgen05";
        case Kernel::kGeneric: return "generic";
        default: return nullptr;
    }
}

Kernel select_kernel(const dcp_params& p) {
    if (gqa_mma_supported(p)) return Kernel::kGqaMma;
    if (mla_tc_supported(p)) return Kernel::kMlaTc;
    if (generic_supported(p)) return Kernel::kGeneric;
    return Kernel::kNone;
}

int64_t kernel_workers(Kernel k, int sms, const dcp_params& p) {
    switch (k) {
        case Kernel::kGqaMma: return gqa_mma_workers(sms);
        case Kernel::kMlaTc: return mla_tc_workers(sms, p.Tq);
        case Kernel::kGeneric: return generic_workers(sms);
        default: return 0;
    }
}

int kernel_chunk(Kernel k, const dcp_params& p) {
    switch (k) {
        case Kernel::kGqaMma: return 16;
        case Kernel::kMlaTc: return 64;
        case Kernel::kGeneric: return generic_chunk(p.block_size);
        default: return 1;
    }
}

// Workspace layout for (params, B) with the kernel that would run.
bool layout_for(const dcp_params& p, int32_t B, WsLayout* out, Kernel* kout, int64_t* W) {
    const int sms = device_sms();
    if (sms <= 0) return false;
    const Kernel k = select_kernel(p);
    const int64_t U = (int64_t)B * p.Hkv * p.N;
    const int64_t w = k == Kernel::kNone ? 0 : kernel_workers(k, sms, p);
    const int64_t rows = (int64_t)p.Tq * (p.Hq / p.Hkv);
    const size_t qprep = (k == Kernel::kMlaTc && p.kv_dtype == DCP_FP8_E4M3) ? mla_f8_qprep_bytes(B, p.Tq) : 0;
    *out = ws_layout(U, U, w + U, rows, p.Dv, qprep, w);
    if (kout) *kout = k;
    if (W) *W = w;
    return true;
}

// Where the work plan of an attention call is made.
enum class PlanMode {
    kInline,   // the planner launches just before the kernels (PDL overlaps their launch)
    kOnly,     // a plan made ahead (dcp_decode_plan): the planner alone, with worker starts
    kPlanned,  // the kernels alone, on a plan made ahead with the same arguments
};

// The arguments a plan depends on, folded into 64 bits (FNV-1a).  Written by
// the planner into the workspace header; every attention kernel compares it
// with its own and refuses a plan made for other arguments.  Never 0 (a
// zeroed workspace holds no plan).
uint64_t plan_key_of(const dcp_params& p, int32_t B, int32_t max_blocks, const int32_t* seq_lens,
                     const int32_t* local_lens, bool partial_mode, bool lens_given, bool worker_starts, int64_t W,
                     int CH) {
    uint64_t h = 1469598103934665603ull;
    auto mix = [&](uint64_t v) {
        for (int i = 0; i < 8; ++i) {
            h ^= (v >> (8 * i)) & 0xffu;
            h *= 1099511628211ull;
        }
    };
    const int64_t f[] = {p.layout, p.N, p.I, p.block_size, p.Hq, p.Hkv, p.Dk, p.Dv, p.Tq, p.q_dtype, p.kv_dtype,
                         B, max_blocks, partial_mode, lens_given, worker_starts, W, CH};
    for (int64_t v : f) mix((uint64_t)v);
    mix((uint64_t)reinterpret_cast<uintptr_t>(seq_lens));
    mix((uint64_t)reinterpret_cast<uintptr_t>(local_lens));
    return h | 1u;
}

int run_attention(const dcp_params* params, int32_t B, const void* q, const void* k_pool,
                  const void* v_pool, int64_t num_blocks, const int32_t* block_tables, int32_t max_blocks,
                  const int32_t* seq_lens, const int32_t* local_lens, bool partial_mode, float* out_partial,
                  float* lse_partial, void* out, float* lse, void* workspace, size_t workspace_bytes,
                  cudaStream_t stream, bool lens_given = false, PlanMode mode = PlanMode::kInline) {
    int rc = validate_params(params);
    if (rc != DCP_OK) return rc;
    const dcp_params& p = *params;
    if (B < 0) return DCP_ERR_INVALID_ARG;
    if (B == 0) return DCP_OK;
    if (!seq_lens || !local_lens) return DCP_ERR_INVALID_ARG;
    if (max_blocks < 1) return DCP_ERR_INVALID_ARG;
    if (mode != PlanMode::kOnly) {
        if (!q || !k_pool || !block_tables) return DCP_ERR_INVALID_ARG;
        if (p.layout == DCP_LAYOUT_GQA && !v_pool) return DCP_ERR_INVALID_ARG;
        if (p.layout == DCP_LAYOUT_MLA && v_pool) return DCP_ERR_INVALID_ARG;
        if (partial_mode && (!out_partial || !lse_partial)) return DCP_ERR_INVALID_ARG;
        if (!partial_mode && !out) return DCP_ERR_INVALID_ARG;
        if (num_blocks < 1) return DCP_ERR_INVALID_ARG;
        if (!aligned16(q) || !aligned16(k_pool) || (v_pool && !aligned16(v_pool))) return DCP_ERR_INVALID_ARG;
    }
    if (!workspace) return DCP_ERR_WORKSPACE;
    WsLayout lay;
    Kernel kern;
    int64_t W;
    if (!layout_for(p, B, &lay, &kern, &W)) return DCP_ERR_CUDA;
    if (kern == Kernel::kNone) return DCP_ERR_UNSUPPORTED;
    if (workspace_bytes < lay.total) return DCP_ERR_WORKSPACE;
    const bool ahead = mode != PlanMode::kInline;  // the plan holds each worker's first unit

    AttnArgs a;
    memset(&a, 0, sizeof a);
    a.N = p.N; a.I = p.I; a.bs = p.block_size; a.Hq = p.Hq; a.Hkv = p.Hkv; a.Dk = p.Dk; a.Dv = p.Dv;
    a.Tq = p.Tq; a.G = p.Hq / p.Hkv; a.B = B; a.max_blocks = max_blocks; a.layout = p.layout;
    a.partial_mode = partial_mode ? 1 : 0; a.out_dtype = p.out_dtype; a.CH = kernel_chunk(kern, p);
    a.num_blocks = num_blocks; a.U = (int64_t)B * p.Hkv * p.N;
    if (a.U >= (int64_t)1 << 31) return DCP_ERR_INVALID_ARG;  // unit ids are 32-bit in the plan
    a.Gn = partial_mode ? a.U : (int64_t)B * p.Hkv; a.W = W;
    a.softmax_scale = p.softmax_scale; a.kv_scale = p.kv_scale;
    a.q = q; a.k_pool = k_pool; a.v_pool = v_pool; a.block_tables = block_tables; a.seq_lens = seq_lens;
    a.local_lens = local_lens; a.out_partial = out_partial; a.lse_partial = lse_partial; a.out = out;
    a.lse = lse; a.ws = reinterpret_cast<uint8_t*>(workspace); a.lay = lay; a.rows = p.Tq * a.G;
    a.lens_given = lens_given ? 1 : 0;
    a.worker_starts = ahead ? 1 : 0;
    a.plan_key = plan_key_of(p, B, max_blocks, seq_lens, local_lens, partial_mode, lens_given, ahead, W, a.CH);

    if (mode != PlanMode::kPlanned) {
        PlanArgs pa;
        memset(&pa, 0, sizeof pa);
        pa.N = p.N; pa.I = p.I; pa.bs = p.block_size; pa.Hkv = p.Hkv; pa.Tq = p.Tq; pa.CH = a.CH; pa.B = B;
        pa.partial_mode = a.partial_mode; pa.W = W; pa.lens_given = lens_given ? 1 : 0; pa.max_blocks = max_blocks;
        pa.worker_starts = a.worker_starts; pa.plan_key = a.plan_key; pa.seq_lens = seq_lens;
        pa.local_lens = local_lens; pa.ws = a.ws; pa.lay = lay; pa.U = a.U; pa.G = a.Gn;
        launch_plan(pa, stream);
        if (cudaGetLastError() != cudaSuccess) return DCP_ERR_CUDA;
        count_launches(1);
        if (mode == PlanMode::kOnly) return DCP_OK;
    }

    cudaError_t e = cudaSuccess;
    if (kern == Kernel::kGqaMma) {
        e = launch_attn_gqa_mma(a, stream);
        count_launches(1);
    } else if (kern == Kernel::kMlaTc) {
        e = launch_attn_mla_tc(a, p.kv_dtype, stream);
        count_launches(p.kv_dtype == DCP_FP8_E4M3 ? 2 : 1);  // fp8: query preparation + attention
        if (e == cudaSuccess && a.Gn > 0) {
            e = launch_segment_merge(a, stream);
            count_launches(1);
        }
    } else {
        e = launch_attn_generic(a, p.q_dtype, p.kv_dtype, stream);
        count_launches(1);
        if (e == cudaSuccess && a.Gn > 0) {
            e = launch_segment_merge(a, stream);
            count_launches(1);
        }
    }
    return e == cudaSuccess ? DCP_OK : DCP_ERR_CUDA;
}

// ---- DCP-localised sparse attention ------------------------------------------
// Workspace: the dense pass's own workspace first (its header is the caller's
// error word), then the localised lists, the staging cache and the partials.
// The dense pass sees query row i as request i with Tq 1 and rank r's
// candidates of it as rank r's local tokens: I = kpad and seq_len = N kpad
// make every rank's closed-form length kpad, a cap the given candidate counts
// never exceed, and every staged token visible; its fused merge over the
// ranks is then the exact sparse result.
struct SparseLayout {
    size_t inner, local, counts, st_pool, st_tables, st_lens, total;
    int64_t R, S;
    int kpad;
};

bool sparse_layout(const dcp_params& p, int32_t B, int32_t k, dcp_params* inner, SparseLayout* L) {
    L->R = (int64_t)B * p.Tq;
    L->S = L->R * p.N;
    L->kpad = (k + 63) / 64 * 64;
    *inner = p;
    inner->I = L->kpad;
    inner->block_size = 64;
    inner->Tq = 1;
    WsLayout lay;
    Kernel kern;
    int64_t W;
    if (!layout_for(*inner, (int32_t)L->R, &lay, &kern, &W)) return false;
    const size_t esz = p.kv_dtype == DCP_FP8_E4M3 ? 1 : (p.kv_dtype == DCP_BF16 ? 2 : 4);
    size_t o = align256(lay.total);
    L->inner = lay.total;
    L->local = o; o = align256(o + sizeof(int32_t) * (size_t)(p.N * L->R * k));
    L->counts = o; o = align256(o + sizeof(int32_t) * (size_t)(p.N * L->R));
    L->st_pool = o; o = align256(o + (size_t)L->S * L->kpad * p.Dk * esz);
    L->st_tables = o; o = align256(o + sizeof(int32_t) * (size_t)(L->S * (L->kpad / 64)));
    L->st_lens = o; o = align256(o + sizeof(int32_t) * (size_t)L->R);
    L->total = o;
    return true;
}

int sparse_check(const dcp_params* params, int32_t B, int32_t k) {
    int rc = validate_params(params);
    if (rc != DCP_OK) return rc;
    const dcp_params& p = *params;
    if (p.layout != DCP_LAYOUT_MLA || p.q_dtype != DCP_BF16 || p.N > 32) return DCP_ERR_UNSUPPORTED;
    if (B < 0 || k < 1) return DCP_ERR_INVALID_ARG;
    return DCP_OK;
}

}  // namespace
}  // namespace dcp

using namespace dcp;

extern "C" {

int dcp_version(void) { return 1; }

uint64_t dcp_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* dcp_attention_kernel(const dcp_params* params) {
    if (validate_params(params) != DCP_OK) return nullptr;
    return kernel_name(select_kernel(*params));
}

const char* dcp_error_string(int code) {
    switch (code) {
        case DCP_OK: return "ok";
        case DCP_ERR_INVALID_ARG: return "invalid argument";
        case DCP_ERR_UNSUPPORTED: return "unsupported combination";
        case DCP_ERR_CUDA: return "CUDA runtime error";
        case DCP_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown error code";
    }
}

int dcp_workspace_size(const dcp_params* params, int32_t B, int64_t max_seq_len, size_t* bytes) {
    int rc = validate_params(params);
    if (rc != DCP_OK) return rc;
    if (!bytes || B < 0 || max_seq_len < 1) return DCP_ERR_INVALID_ARG;
    WsLayout lay;
    Kernel k;
    if (!layout_for(*params, B, &lay, &k, nullptr)) return DCP_ERR_CUDA;
    *bytes = lay.total;
    return DCP_OK;
}

int dcp_workspace_init(void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!workspace || workspace_bytes < 256) return DCP_ERR_WORKSPACE;
    return cudaMemsetAsync(workspace, 0, workspace_bytes, stream) == cudaSuccess ? DCP_OK : DCP_ERR_CUDA;
}

int dcp_get_error(void* workspace, cudaStream_t stream, uint32_t* bits) {
    if (!workspace || !bits) return DCP_ERR_INVALID_ARG;
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return DCP_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return DCP_ERR_CUDA;
    *bits = v;
    if (v != 0) {
        if (cudaMemsetAsync(workspace, 0, sizeof v, stream) != cudaSuccess) return DCP_ERR_CUDA;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return DCP_ERR_CUDA;
    }
    return DCP_OK;
}

int dcp_slot_mapping(const dcp_params* params, int32_t B, const int32_t* seq_lens, int64_t T,
                     const int32_t* tok_req, const int64_t* tok_pos, const int32_t* block_tables,
                     int32_t max_blocks, int64_t num_blocks, int8_t* owner, int64_t* slots,
                     int32_t* local_lens, int32_t* virt_blocks, int32_t* rank_blocks, const void* new_k,
                     const void* new_v, void* k_pool, void* v_pool, void* workspace, size_t workspace_bytes,
                     cudaStream_t stream) {
    int rc = validate_params(params);
    if (rc != DCP_OK) return rc;
    const dcp_params& p = *params;
    if (B < 0 || T < 0) return DCP_ERR_INVALID_ARG;
    if (B > 0 && !seq_lens) return DCP_ERR_INVALID_ARG;
    if (T > 0 && (owner || slots || new_k) && (!tok_req || !tok_pos)) return DCP_ERR_INVALID_ARG;
    if (owner && p.N > 127) return DCP_ERR_INVALID_ARG;  // owner ranks are stored as int8
    if (T > 0 && B == 0 && (owner || slots || new_k)) return DCP_ERR_INVALID_ARG;
    if ((slots || new_k) && (!block_tables || max_blocks < 1 || num_blocks < 1)) return DCP_ERR_INVALID_ARG;
    if (new_k && !k_pool) return DCP_ERR_INVALID_ARG;
    if (p.layout == DCP_LAYOUT_GQA && new_k && (!new_v || !v_pool)) return DCP_ERR_INVALID_ARG;
    if (p.layout == DCP_LAYOUT_MLA && (new_v || v_pool)) return DCP_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < 256) return DCP_ERR_WORKSPACE;
    SlotArgs a;
    memset(&a, 0, sizeof a);
    a.N = p.N; a.I = p.I; a.bs = p.block_size; a.B = B; a.layout = p.layout; a.Hkv = p.Hkv; a.Dk = p.Dk;
    a.Dv = p.Dv; a.kv_esize = esize(p.kv_dtype); a.max_blocks = max_blocks; a.T = T; a.num_blocks = num_blocks;
    a.seq_lens = seq_lens; a.tok_req = tok_req; a.tok_pos = tok_pos; a.block_tables = block_tables;
    a.owner = owner; a.slots = slots; a.local_lens = local_lens; a.virt_blocks = virt_blocks;
    a.rank_blocks = rank_blocks; a.new_k = new_k; a.new_v = new_v; a.k_pool = k_pool; a.v_pool = v_pool;
    a.err = &reinterpret_cast<WsHeader*>(workspace)->err;
    return launch_slot_mapping(a, stream) == cudaSuccess ? DCP_OK : DCP_ERR_CUDA;
}

int dcp_transfer_blocks(const dcp_params* params, int32_t B, const int32_t* seq_lens,
                        const int32_t* block_tables, int32_t max_blocks, int64_t num_blocks, int32_t* counts,
                        int32_t* blocks, int32_t* fills, int64_t* totals, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
    int rc = validate_params(params);
    if (rc != DCP_OK) return rc;
    const dcp_params& p = *params;
    if (B < 0) return DCP_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < 256) return DCP_ERR_WORKSPACE;
    if (B == 0) {
        if (totals && cudaMemsetAsync(totals, 0, 2 * sizeof(int64_t), stream) != cudaSuccess) return DCP_ERR_CUDA;
        return DCP_OK;
    }
    if (!seq_lens || !block_tables || !counts || max_blocks < 1 || num_blocks < 1) return DCP_ERR_INVALID_ARG;
    if (!aligned8(totals) || (int64_t)p.N * B * max_blocks > INT32_MAX) return DCP_ERR_INVALID_ARG;
    return launch_transfer_blocks(p.N, p.I, p.block_size, B, max_blocks, num_blocks, seq_lens, block_tables,
                                  counts, blocks, fills, totals, workspace, stream) == cudaSuccess
               ? DCP_OK
               : DCP_ERR_CUDA;
}

int dcp_pcp_partition(int32_t K, int32_t B, const int32_t* ctx_lens, const int32_t* q_lens, int32_t max_q,
                      int32_t* pos, int32_t* padded_lens, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
    if (K < 1 || B < 0 || max_q < 0) return DCP_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < 256) return DCP_ERR_WORKSPACE;
    if (B == 0) return DCP_OK;
    if (!ctx_lens || !q_lens || !pos || !padded_lens) return DCP_ERR_INVALID_ARG;
    if (max_q == 0) return DCP_ERR_INVALID_ARG;
    return launch_pcp_partition(K, B, ctx_lens, q_lens, max_q, pos, padded_lens,
                                &reinterpret_cast<WsHeader*>(workspace)->err, stream) == cudaSuccess
               ? DCP_OK
               : DCP_ERR_CUDA;
}

int dcp_prefill_attention(const dcp_params* params, int32_t B, int32_t Tq, const void* q, const int32_t* q_pos,
                          const void* k_pool, const void* v_pool, int64_t num_blocks, const int32_t* block_tables,
                          int32_t max_blocks, const int32_t* seq_lens, const int32_t* local_lens,
                          float* out_partial, float* lse_partial, void* out, float* lse, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
    int rc = validate_params(params);
    if (rc != DCP_OK) return rc;
    const dcp_params& p = *params;
    if (B < 0 || Tq < 0) return DCP_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < 256) return DCP_ERR_WORKSPACE;
    if (!prefill_supported(p)) return DCP_ERR_UNSUPPORTED;
    if (B == 0 || Tq == 0) return DCP_OK;
    if (!q || !q_pos || !k_pool || !v_pool || !block_tables || !seq_lens || !local_lens || !out_partial ||
        !lse_partial)
        return DCP_ERR_INVALID_ARG;
    if (num_blocks < 1 || max_blocks < 1) return DCP_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out_partial))
        return DCP_ERR_INVALID_ARG;
    PrefillArgs a;
    memset(&a, 0, sizeof a);
    a.N = p.N; a.I = p.I; a.bs = p.block_size; a.Hq = p.Hq; a.Hkv = p.Hkv; a.G = p.Hq / p.Hkv; a.D = p.Dk;
    a.Tq = Tq; a.B = B; a.max_blocks = max_blocks; a.num_blocks = num_blocks; a.softmax_scale = p.softmax_scale;
    a.q = q; a.q_pos = q_pos; a.k_pool = k_pool; a.v_pool = v_pool; a.block_tables = block_tables;
    a.seq_lens = seq_lens; a.local_lens = local_lens; a.out_partial = out_partial; a.lse_partial = lse_partial;
    a.ws = reinterpret_cast<uint8_t*>(workspace);
    if ((prefill_tc_supported(a) ? launch_prefill_tc(a, stream) : launch_prefill_partial(a, stream)) != cudaSuccess)
        return DCP_ERR_CUDA;
    count_launches(1);
    if (out) {
        if (launch_lse_merge(p.N, (int64_t)B * Tq * p.Hq, p.Dv, out_partial, lse_partial, out, p.out_dtype, lse,
                             stream) != cudaSuccess)
            return DCP_ERR_CUDA;
    }
    return DCP_OK;
}


int dcp_sparse_workspace_size(const dcp_params* params, int32_t B, int32_t k, size_t* bytes) {
    int rc = sparse_check(params, B, k);
    if (rc != DCP_OK) return rc;
    if (!bytes) return DCP_ERR_INVALID_ARG;
    dcp_params inner;
    SparseLayout L;
    if (!sparse_layout(*params, B, k, &inner, &L)) return DCP_ERR_CUDA;
    *bytes = L.total;
    return DCP_OK;
}

int dcp_sparse_localize(const dcp_params* params, int32_t B, int32_t k, const int32_t* cand, const int32_t* seq_lens,
                        int32_t* local, int32_t* counts, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
    int rc = sparse_check(params, B, k);
    if (rc != DCP_OK) return rc;
    if (!workspace || workspace_bytes < 256) return DCP_ERR_WORKSPACE;
    if (B == 0) return DCP_OK;
    if (!cand || !seq_lens || !local || !counts) return DCP_ERR_INVALID_ARG;
    const dcp_params& p = *params;
    return launch_sparse_localize(p.N, p.I, B * p.Tq, p.Tq, k, cand, seq_lens, local, counts,
                                  &reinterpret_cast<WsHeader*>(workspace)->err, stream) == cudaSuccess
               ? DCP_OK
               : DCP_ERR_CUDA;
}

int dcp_sparse_decode_attention(const dcp_params* params, int32_t B, int32_t k, const void* q, const int32_t* cand,
                                const void* k_pool, int64_t num_blocks, const int32_t* block_tables,
                                int32_t max_blocks, const int32_t* seq_lens, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
    int rc = sparse_check(params, B, k);
    if (rc != DCP_OK) return rc;
    if (B == 0) return DCP_OK;
    if (!q || !cand || !k_pool || !block_tables || !seq_lens || !out) return DCP_ERR_INVALID_ARG;
    if (num_blocks < 1 || max_blocks < 1 || !aligned16(q) || !aligned16(k_pool)) return DCP_ERR_INVALID_ARG;
    if (!workspace) return DCP_ERR_WORKSPACE;
    const dcp_params& p = *params;
    dcp_params inner;
    SparseLayout L;
    if (!sparse_layout(p, B, k, &inner, &L)) return DCP_ERR_CUDA;
    if (workspace_bytes < L.total) return DCP_ERR_WORKSPACE;
    uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
    int32_t* local = reinterpret_cast<int32_t*>(ws + L.local);
    int32_t* counts = reinterpret_cast<int32_t*>(ws + L.counts);
    uint32_t* err = &reinterpret_cast<WsHeader*>(ws)->err;
    // 1. each rank's candidates at their local positions, and rank r's
    //    candidate rows of query row i copied contiguously (staging)
    SparseStageArgs sa;
    memset(&sa, 0, sizeof sa);
    sa.N = p.N; sa.I = p.I; sa.R = (int)L.R; sa.Tq = p.Tq; sa.B = B; sa.k = k; sa.kpad = L.kpad;
    sa.bs = p.block_size; sa.max_blocks = max_blocks; sa.num_blocks = num_blocks;
    sa.row_bytes = p.Dk * (p.kv_dtype == DCP_FP8_E4M3 ? 1 : (p.kv_dtype == DCP_BF16 ? 2 : 4));
    sa.cand = cand; sa.seq_lens = seq_lens;
    sa.local = local; sa.counts = counts; sa.block_tables = block_tables; sa.k_pool = k_pool;
    sa.st_pool = ws + L.st_pool;
    sa.st_tables = reinterpret_cast<int32_t*>(ws + L.st_tables);
    sa.st_lens = reinterpret_cast<int32_t*>(ws + L.st_lens);
    sa.err = err;
    if (launch_sparse_stage(sa, stream) != cudaSuccess) return DCP_ERR_CUDA;
    // 2. the dense decode pass over the staged candidates, ranks merged exactly
    return run_attention(&inner, (int32_t)L.R, q, sa.st_pool, nullptr, L.S * (L.kpad / 64), sa.st_tables,
                         L.kpad / 64, sa.st_lens, counts, false, nullptr, nullptr, out, lse, workspace, L.inner,
                         stream, /*lens_given=*/true);
}

int dcp_partial_attention(const dcp_params* params, int32_t B, const void* q, const void* k_pool,
                          const void* v_pool, int64_t num_blocks, const int32_t* block_tables,
                          int32_t max_blocks, const int32_t* seq_lens, const int32_t* local_lens,
                          float* out_partial, float* lse_partial, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
    return run_attention(params, B, q, k_pool, v_pool, num_blocks, block_tables, max_blocks, seq_lens,
                         local_lens, true, out_partial, lse_partial, nullptr, nullptr, workspace,
                         workspace_bytes, stream);
}

int dcp_decode_attention(const dcp_params* params, int32_t B, const void* q, const void* k_pool,
                         const void* v_pool, int64_t num_blocks, const int32_t* block_tables,
                         int32_t max_blocks, const int32_t* seq_lens, const int32_t* local_lens, void* out,
                         float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return run_attention(params, B, q, k_pool, v_pool, num_blocks, block_tables, max_blocks, seq_lens,
                         local_lens, false, nullptr, nullptr, out, lse, workspace, workspace_bytes, stream);
}

int dcp_decode_plan(const dcp_params* params, int32_t B, const int32_t* seq_lens, const int32_t* local_lens,
                    int32_t max_blocks, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return run_attention(params, B, nullptr, nullptr, nullptr, 0, nullptr, max_blocks, seq_lens, local_lens, false,
                         nullptr, nullptr, nullptr, nullptr, workspace, workspace_bytes, stream, false,
                         PlanMode::kOnly);
}

int dcp_decode_attention_planned(const dcp_params* params, int32_t B, const void* q, const void* k_pool,
                                 const void* v_pool, int64_t num_blocks, const int32_t* block_tables,
                                 int32_t max_blocks, const int32_t* seq_lens, const int32_t* local_lens, void* out,
                                 float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return run_attention(params, B, q, k_pool, v_pool, num_blocks, block_tables, max_blocks, seq_lens, local_lens,
                         false, nullptr, nullptr, out, lse, workspace, workspace_bytes, stream, false,
                         PlanMode::kPlanned);
}

int dcp_lse_merge(int32_t N, int64_t rows, int32_t Dv, const float* out_partial, const float* lse_partial,
                  void* out, int32_t out_dtype, float* lse, cudaStream_t stream) {
    if (N < 1 || rows < 0 || Dv < 1) return DCP_ERR_INVALID_ARG;
    if (out_dtype != DCP_F32 && out_dtype != DCP_BF16) return DCP_ERR_INVALID_ARG;
    if (rows == 0) return DCP_OK;
    if (!out_partial || !lse_partial || !out) return DCP_ERR_INVALID_ARG;
    return launch_lse_merge(N, rows, Dv, out_partial, lse_partial, out, out_dtype, lse, stream) == cudaSuccess
               ? DCP_OK
               : DCP_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode attention with library-owned scratch, for callers that cannot
// allocate device memory.
// ---------------------------------------------------------------------------
#include <mutex>

namespace dcp {
namespace {

constexpr size_t kStaticScratchBytes = DCP_STATIC_SCRATCH_BYTES;

// One copy per device that loads this library, held until the process exits.
// Host code must not use this name as a device address: it only stands in
// for the symbol; static_scratch() looks up the device address.
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
void* g_static_ptr[64] = {nullptr};

// Device address of g_static_scratch on the current device (looked up once
// per device, with that device current).  nullptr on failure.
void* static_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (g_static_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return nullptr;
        g_static_ptr[dev] = p;
    }
    return g_static_ptr[dev];
}

}  // namespace
}  // namespace dcp

extern "C" int dcp_noalloc_get_error(cudaStream_t stream, uint32_t* bits) {
    if (!bits) return DCP_ERR_INVALID_ARG;
    void* ws = static_scratch();
    if (ws == nullptr) return DCP_ERR_CUDA;
    // the same read-and-clear as dcp_get_error, on the library's own buffer
    return dcp_get_error(ws, stream, bits);
}

extern "C" int dcp_decode_attention_noalloc(const dcp_params* params, int32_t B, const void* q,
                                            const void* k_pool, const void* v_pool, int64_t num_blocks,
                                            const int32_t* block_tables, int32_t max_blocks,
                                            const int32_t* seq_lens, const int32_t* local_lens, void* out,
                                            float* lse, cudaStream_t stream) {
    int rc = validate_params(params);
    if (rc != DCP_OK) return rc;
    if (B < 0) return DCP_ERR_INVALID_ARG;
    if (B == 0) return DCP_OK;
    size_t need = 0;
    rc = dcp_workspace_size(params, B, 1, &need);
    if (rc != DCP_OK) return rc;
    if (need > kStaticScratchBytes) return DCP_ERR_WORKSPACE;  // problem too large for the static scratch
    void* ws = static_scratch();
    if (ws == nullptr) return DCP_ERR_CUDA;
    // the error word is the only scratch that must start at zero here: the
    // planner resets the arrival counters and rewrites the plan every call
    if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), stream) != cudaSuccess) return DCP_ERR_CUDA;
    return run_attention(params, B, q, k_pool, v_pool, num_blocks, block_tables, max_blocks, seq_lens, local_lens,
                         false, nullptr, nullptr, out, lse, ws, kStaticScratchBytes, stream);
}

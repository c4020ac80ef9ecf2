// Slot mapping and cache write for virtual DCP ranks on one GPU.
//
// "Breaking the Long-Sequence Inference Bottleneck ...", section 2: a token's
// owner is floor(t / I) mod N; the owner writes the token's KV row into its
// slot, every other rank sees slot -1 and skips it; the upper layer allocates
// virtual blocks of block_size x N by the total length and each rank derives
// its own physical block need.  "vLLM DCP and PCP", Deep Dive 5: per-rank
// local lengths.
#include "dcp_internal.cuh"

namespace dcp {
namespace {

__global__ void meta_kernel(SlotArgs a) {
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= (int64_t)a.N * a.B) return;
    const int r = (int)(i / a.B);
    const int b = (int)(i % a.B);
    const int64_t L = a.seq_lens[b];
    const int64_t n = L > 0 ? local_len(L, r, a.N, a.I) : 0;
    if (a.local_lens) a.local_lens[i] = (int32_t)n;
    if (a.rank_blocks) a.rank_blocks[i] = (int32_t)ceil_div64(n, a.bs);
    if (a.virt_blocks && r == 0) a.virt_blocks[b] = (int32_t)(L > 0 ? ceil_div64(L, (int64_t)a.bs * a.N) : 0);
}

// Copy `bytes` from src to dst with the 32 lanes of a warp (16-byte vectors
// when both ends and the size allow it).
__device__ __forceinline__ void warp_copy(uint8_t* dst, const uint8_t* src, int bytes, int lane) {
    if ((((uintptr_t)dst | (uintptr_t)src | (uintptr_t)bytes) & 15) == 0) {
        const uint4* s = reinterpret_cast<const uint4*>(src);
        uint4* d = reinterpret_cast<uint4*>(dst);
        for (int i = lane; i < bytes / 16; i += 32) d[i] = s[i];
    } else if ((((uintptr_t)dst | (uintptr_t)src | (uintptr_t)bytes) & 3) == 0) {
        const uint32_t* s = reinterpret_cast<const uint32_t*>(src);
        uint32_t* d = reinterpret_cast<uint32_t*>(dst);
        for (int i = lane; i < bytes / 4; i += 32) d[i] = s[i];
    } else {
        for (int i = lane; i < bytes; i += 32) dst[i] = src[i];
    }
}

// The token's rows of every KV head (K, then V) from their contiguous copy in
// new_k / new_v to their slots in the pools, 16-byte pieces only.  The pieces
// of one batch (32 lanes x kBatch) are loaded before the slot is known, so the
// row loads overlap the ownership / block-table lookups, and stored after.
constexpr int kBatch = 8;
struct TokenRows {
    int kq, vq, nk, n;  // 16-byte pieces per K row, per V row; K pieces; all pieces
    const uint4* ks;
    const uint4* vs;
};
__device__ __forceinline__ TokenRows token_rows(const SlotArgs& a, int64_t t) {
    TokenRows r;
    const int krow = a.Dk * a.kv_esize, vrow = a.Dv * a.kv_esize;
    r.kq = krow / 16;
    r.vq = vrow / 16;
    r.nk = a.Hkv * r.kq;
    r.n = r.nk + (a.new_v ? a.Hkv * r.vq : 0);
    r.ks = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(a.new_k) + t * a.Hkv * krow);
    r.vs = a.new_v ? reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(a.new_v) + t * a.Hkv * vrow)
                   : nullptr;
    return r;
}
__device__ __forceinline__ void load_batch(const TokenRows& r, int base, int lane, uint4 (&v)[kBatch]) {
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
        const int i = base + lane + 32 * j;
        if (i < r.n) v[j] = i < r.nk ? r.ks[i] : r.vs[i - r.nk];
    }
}
__device__ __forceinline__ void store_batch(const SlotArgs& a, const TokenRows& r, int64_t blk, int64_t off, int base,
                                            int lane, const uint4 (&v)[kBatch]) {
    const int krow = r.kq * 16, vrow = r.vq * 16;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
        int i = base + lane + 32 * j;
        if (i >= r.n) continue;
        uint4* dst;
        if (i < r.nk) {
            const int h = i / r.kq;
            dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(a.k_pool) + ((blk * a.Hkv + h) * a.bs + off) * krow) +
                  (i - h * r.kq);
        } else {
            i -= r.nk;
            const int h = i / r.vq;
            dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(a.v_pool) + ((blk * a.Hkv + h) * a.bs + off) * vrow) +
                  (i - h * r.vq);
        }
        *dst = v[j];
    }
}

// One warp per token: ownership, local position, slot, and the row copy.
__global__ void token_kernel(SlotArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t t = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    if (t >= a.T) return;
    // 16-byte pieces when every end allows them (MLA: one head, no V rows)
    const bool v16 = a.new_k != nullptr &&
                     ((reinterpret_cast<uintptr_t>(a.new_k) | reinterpret_cast<uintptr_t>(a.new_v) |
                       reinterpret_cast<uintptr_t>(a.k_pool) | reinterpret_cast<uintptr_t>(a.v_pool) |
                       (uintptr_t)(a.Dk * a.kv_esize) | (uintptr_t)(a.new_v ? a.Dv * a.kv_esize : 0)) & 15u) == 0;
    TokenRows rows{};
    uint4 first[kBatch];
    if (v16) {
        rows = token_rows(a, t);
        load_batch(rows, 0, lane, first);  // in flight during the lookups below
    }
    int owner = -1;
    int64_t slot = -1;
    int b = 0;
    if (lane == 0) {
        b = a.tok_req[t];
        const int64_t pos = a.tok_pos[t];
        if (b < 0 || b >= a.B || pos < 0) {
            raise_err(a.err, DCP_DEV_ERR_TOKEN);
        } else {
            // the block-table read goes out beside the length check
            const int own = (int)owner_rank(pos, a.N, a.I);
            const int64_t lp = local_pos(pos, a.N, a.I);
            const int64_t blk_idx = lp / a.bs;
            const bool in_table = a.block_tables && blk_idx < a.max_blocks;
            const int32_t id = in_table ? a.block_tables[((int64_t)own * a.B + b) * a.max_blocks + blk_idx] : -1;
            if (pos >= (int64_t)a.seq_lens[b]) {
                raise_err(a.err, DCP_DEV_ERR_TOKEN);
            } else {
                owner = own;
                if (a.block_tables) {
                    if (!in_table)
                        raise_err(a.err, DCP_DEV_ERR_TABLE);
                    else if (id < 0 || id >= a.num_blocks)
                        raise_err(a.err, DCP_DEV_ERR_BLOCK_ID);
                    else
                        slot = (int64_t)id * a.bs + lp % a.bs;
                }
            }
        }
    }
    owner = __shfl_sync(0xffffffffu, owner, 0);
    slot = __shfl_sync(0xffffffffu, slot, 0);
    if (a.owner && lane == 0) a.owner[t] = (int8_t)owner;
    if (a.slots)
        for (int r = lane; r < a.N; r += 32) a.slots[(int64_t)r * a.T + t] = (r == owner) ? slot : -1;
    if (slot < 0 || a.new_k == nullptr) return;
    const int64_t blk = slot / a.bs, off = slot % a.bs;
    if (v16) {
        store_batch(a, rows, blk, off, 0, lane, first);
        for (int base = 32 * kBatch; base < rows.n; base += 32 * kBatch) {
            uint4 v[kBatch];
            load_batch(rows, base, lane, v);
            store_batch(a, rows, blk, off, base, lane, v);
        }
        return;
    }
    if (a.layout == DCP_LAYOUT_MLA) {
        const int row = a.Dk * a.kv_esize;
        warp_copy(reinterpret_cast<uint8_t*>(a.k_pool) + (blk * a.bs + off) * row,
                  reinterpret_cast<const uint8_t*>(a.new_k) + t * row, row, lane);
    } else {
        const int krow = a.Dk * a.kv_esize, vrow = a.Dv * a.kv_esize;
        for (int h = 0; h < a.Hkv; ++h) {
            const int64_t dst = (blk * a.Hkv + h) * a.bs + off;
            warp_copy(reinterpret_cast<uint8_t*>(a.k_pool) + dst * krow,
                      reinterpret_cast<const uint8_t*>(a.new_k) + (t * a.Hkv + h) * krow, krow, lane);
            if (a.new_v)
                warp_copy(reinterpret_cast<uint8_t*>(a.v_pool) + dst * vrow,
                          reinterpret_cast<const uint8_t*>(a.new_v) + (t * a.Hkv + h) * vrow, vrow, lane);
        }
    }
}

}  // namespace

cudaError_t launch_slot_mapping(const SlotArgs& a, cudaStream_t s) {
    const int64_t nb = (int64_t)a.N * a.B;
    if (nb > 0 && (a.local_lens || a.rank_blocks || a.virt_blocks)) {
        meta_kernel<<<(unsigned)((nb + 255) / 256), 256, 0, s>>>(a);
        count_launches(1);
    }
    if (a.T > 0 && (a.owner || a.slots || a.new_k)) {
        token_kernel<<<(unsigned)((a.T * 32 + 255) / 256), 256, 0, s>>>(a);
        count_launches(1);
    }
    return cudaGetLastError();
}

}  // namespace dcp

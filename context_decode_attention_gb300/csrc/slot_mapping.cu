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
// new_k / new_v to their slots in the pools, 16-byte pieces only: every lane
// loads all of its pieces of a batch before it stores any, so a batch costs
// one memory round trip (a load-store pair per head costs one per head).
__device__ __forceinline__ void scatter_token16(const SlotArgs& a, int64_t t, int64_t blk, int64_t off, int lane) {
    const int krow = a.Dk * a.kv_esize, vrow = a.Dv * a.kv_esize;
    const int kq = krow / 16, vq = vrow / 16;  // 16-byte pieces per row
    const int nk = a.Hkv * kq, n = nk + (a.new_v ? a.Hkv * vq : 0);
    const uint4* ks = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(a.new_k) + t * a.Hkv * krow);
    const uint4* vs = a.new_v ? reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(a.new_v) + t * a.Hkv * vrow)
                              : nullptr;
    auto dst_of = [&](int i) -> uint4* {
        if (i < nk) {
            const int h = i / kq;
            return reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(a.k_pool) + ((blk * a.Hkv + h) * a.bs + off) * krow) +
                   (i - h * kq);
        }
        i -= nk;
        const int h = i / vq;
        return reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(a.v_pool) + ((blk * a.Hkv + h) * a.bs + off) * vrow) +
               (i - h * vq);
    };
    constexpr int kBatch = 8;
    for (int base = 0; base < n; base += 32 * kBatch) {
        uint4 v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int i = base + lane + 32 * j;
            if (i < n) v[j] = i < nk ? ks[i] : vs[i - nk];
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int i = base + lane + 32 * j;
            if (i < n) *dst_of(i) = v[j];
        }
    }
}

// One warp per token: ownership, local position, slot, and the row copy.
__global__ void token_kernel(SlotArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t t = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    if (t >= a.T) return;
    int owner = -1;
    int64_t slot = -1;
    int b = 0;
    if (lane == 0) {
        b = a.tok_req[t];
        const int64_t pos = a.tok_pos[t];
        if (b < 0 || b >= a.B || pos < 0 || pos >= (int64_t)a.seq_lens[b]) {
            raise_err(a.err, DCP_DEV_ERR_TOKEN);
        } else {
            owner = (int)owner_rank(pos, a.N, a.I);
            if (a.block_tables) {
                const int64_t lp = local_pos(pos, a.N, a.I);
                const int64_t blk_idx = lp / a.bs;
                if (blk_idx >= a.max_blocks) {
                    raise_err(a.err, DCP_DEV_ERR_TABLE);
                } else {
                    const int32_t id = a.block_tables[((int64_t)owner * a.B + b) * a.max_blocks + blk_idx];
                    if (id < 0 || id >= a.num_blocks)
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
    const int krow16 = a.Dk * a.kv_esize, vrow16 = a.Dv * a.kv_esize;
    if (((reinterpret_cast<uintptr_t>(a.new_k) | reinterpret_cast<uintptr_t>(a.new_v) |
          reinterpret_cast<uintptr_t>(a.k_pool) | reinterpret_cast<uintptr_t>(a.v_pool) | (uintptr_t)krow16 |
          (uintptr_t)(a.new_v ? vrow16 : 0)) & 15u) == 0) {
        scatter_token16(a, t, blk, off, lane);  // MLA: one head (Hkv 1), no V rows
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

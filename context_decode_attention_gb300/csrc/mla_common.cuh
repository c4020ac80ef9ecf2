// Pieces shared by the MLA tensor-core kernel (attn_mla_pair.cu) and its host
// check: the tile walk over a worker's chunk range, the ring-slot counter and
// the 2D tensor-map encoder.
#pragma once

#include <atomic>

#include <cudaTypedefs.h>

#include "dcp_internal.cuh"

namespace dcp {
namespace mla {

constexpr int kHeads = 128;
constexpr int kDk = 576;
constexpr int kDv = 512;
constexpr int kDvHalf = 256;
constexpr int kChunk = 64;  // tokens per chunk (one TMA box of rows)

struct Tile {
    int64_t u, chunk, group;
    int n_ch;
    bool first, last;
};

// Entries of the unit prefix kept in shared memory, from the worker's first
// unit on (a global read costs a full memory latency on the issuing thread's
// critical path, once or twice per tile).
constexpr int kUnitCache = 96;

// Copy us[u0 .. u0 + kUnitCache) (as far as it exists) into shared memory;
// every thread of the block takes part.  Returns the number of entries.
__device__ __forceinline__ int64_t cache_units(int64_t* us_s, const int64_t* us, int64_t U, int64_t u0,
                                               int64_t cap = kUnitCache) {
    const int64_t avail = U + 1 - u0;
    const int64_t n = avail < cap ? avail : cap;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) us_s[i] = us[u0 + i];
    return n;
}

// The same tile sequence in every role (host-callable too, for the CPU check
// of the walk): walk the worker's chunk range; a tile
// is up to `maxch` (default two) consecutive chunks of one unit.  `first` / `last` mark the
// tiles that open and close a merge group inside the range.
struct TileCursor {
    const int64_t* us;
    const int64_t* us_s;  // us[base .. base + ncache) in shared memory
    int64_t base, ncache;
    int64_t c, c1, u, ubeg, uend;  // current chunk, range end, unit and its chunk range
    int64_t prev_group;
    int N, partial, maxch;
    __host__ __device__ void init(const int64_t* us_, const int64_t* us_s_, int64_t ncache_, int64_t c0, int64_t c1_,
                         int64_t u0, int N_, int pm, int maxch_ = 2) {
        us = us_; us_s = us_s_; base = u0; ncache = ncache_;
        c = c0; c1 = c1_; u = u0; N = N_; partial = pm; prev_group = -1; maxch = maxch_;
        ubeg = at(u);
        uend = at(u + 1);
    }
    __host__ __device__ int64_t at(int64_t v) const { return (v - base < ncache) ? us_s[v - base] : us[v]; }
    // merge group of unit uu (units are (b * Hkv + kvh) * N + r, far below 2^31)
    __host__ __device__ int64_t group_of(int64_t uu) const { return partial ? uu : (int64_t)((uint32_t)uu / (uint32_t)N); }
    __host__ __device__ bool next(Tile& t) {
        if (c >= c1) return false;
        while (uend <= c) {
            ++u;
            ubeg = uend;
            uend = at(u + 1);
        }
        t.u = u;
        t.chunk = c - ubeg;
        const int64_t end = uend < c1 ? uend : c1;
        t.n_ch = (end - c) >= maxch ? maxch : (int)(end - c);
        t.group = group_of(u);
        c += t.n_ch;
        if (c >= c1) {
            t.last = true;
        } else if (c < uend) {
            t.last = false;  // the next tile stays in this unit
        } else {
            int64_t v = u + 1;
            while (at(v + 1) <= c) ++v;
            t.last = group_of(v) != t.group;
        }
        t.first = t.group != prev_group;
        prev_group = t.group;
        return true;
    }
};

// Position in a ring of n slots: slot index and the parity of the lap.
struct Ring {
    uint32_t slot = 0, phase = 0, n = 1;
    __device__ void advance() {
        if (++slot == n) { slot = 0; phase ^= 1u; }
    }
};

// First unit whose chunk range contains chunk c0 (binary search over the
// unit prefix us[0..U]).
__host__ __device__ __forceinline__ int64_t unit_of_chunk(const int64_t* us, int64_t U, int64_t c0) {
    int64_t lo = 0, hi = U - 1;
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) >> 1;
        if (us[mid] <= c0) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// The driver's tensor-map encoder, looked up on first use (through an atomic:
// host threads may call in concurrently; a failed lookup is retried).
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
    PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
    if (!f) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
            fn.store(f, std::memory_order_release);
        }
    }
    return f;
}

// Row-major [rows x cols] tensor with a row pitch of row_bytes; boxes of
// box_rows x box_cols.  Elements outside the tensor read as zero.
inline bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
                        uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace mla
}  // namespace dcp

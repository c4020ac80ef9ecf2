// Work plan for the split-KV attention kernels.
//
// Every virtual rank's local KV of every (request, KV head) is a "unit"; a
// unit is cut into chunks of CH local tokens; the chunks of all units, in
// unit order, are dealt to W workers as equal contiguous ranges (worker w
// owns chunks [w P / W, (w + 1) P / W)).  A worker's range can cross unit
// boundaries; each piece it owns of one merge group is a "segment" with its
// own partial (o, lse) slot.  The plan is computed on the device so the host
// never needs the lengths.
#include "dcp_internal.cuh"

namespace dcp {
namespace {

constexpr int kPlanThreads = 1024;

// Inclusive block-wide scan of one int64 per thread.
__device__ int64_t block_inclusive_scan(int64_t v, int64_t* warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int64_t t = (lane < (int)(blockDim.x >> 5)) ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t n = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += n;
        }
        warp_tot[lane] = t;
    }
    __syncthreads();
    const int64_t before = warp > 0 ? warp_tot[warp - 1] : 0;
    __syncthreads();
    return v + before;
}

// Unit prefix entries also kept in shared memory for the group pass (the
// rest are read back from the workspace).
constexpr int kUnitSmem = 4096;

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a) {
    __shared__ int64_t warp_tot[32];
    __shared__ int64_t carry;
    __shared__ int64_t us_s[kUnitSmem + 1];
    __shared__ int n_empty;
    WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
    int64_t* unit_start = reinterpret_cast<int64_t*>(a.ws + a.lay.off_units);
    int32_t* seg_base = reinterpret_cast<int32_t*>(a.ws + a.lay.off_seg_base);
    uint32_t* counters = reinterpret_cast<uint32_t*>(a.ws + a.lay.off_counters);
    const int tid = threadIdx.x;
    pdl_trigger();  // the attention kernel (or the query preparation) may launch now
    if (tid == 0) carry = 0;
    __syncthreads();

    // 1. chunks per unit, with the metadata checks
    for (int64_t base = 0; base < a.U; base += kPlanThreads) {
        const int64_t u = base + tid;
        const int64_t c = u < a.U ? unit_chunks(u, a.N, a.I, a.Hkv, a.B, a.Tq, a.bs, a.CH, a.max_blocks, a.seq_lens,
                                                a.local_lens, &hdr->err, a.lens_given != 0)
                                  : 0;
        const int64_t incl = block_inclusive_scan(c, warp_tot);
        if (u < a.U) {
            unit_start[u] = carry + incl - c;
            if (u <= kUnitSmem) us_s[u] = carry + incl - c;
        }
        __syncthreads();
        if (tid == kPlanThreads - 1) carry += incl;
        __syncthreads();
    }
    const int64_t P = carry;
    __syncthreads();  // every thread holds the total before carry is reused
    if (tid == 0) {
        unit_start[a.U] = P;
        if (a.U <= kUnitSmem) us_s[a.U] = P;
        hdr->total_chunks = P;
        carry = 0;
        n_empty = 0;
    }
    __syncthreads();
    auto us_at = [&](int64_t i) -> int64_t { return i <= kUnitSmem ? us_s[i] : unit_start[i]; };

    // 2. each worker's first unit (the last u with unit_start[u] <= its first
    // chunk) and that unit's chunk range.  Only a plan made ahead of its call
    // does this: behind the planner the kernel's own search costs less than
    // this pass does in the planner.
    const int64_t We = P < a.W ? P : a.W;
    if (a.worker_starts) {
        WorkerStart* wfirst = reinterpret_cast<WorkerStart*>(a.ws + a.lay.off_wfirst);
        for (int64_t w = tid; w < We; w += kPlanThreads) {
            const int64_t c0 = worker_begin(w, We, P);
            int64_t lo = 0, hi = a.U - 1;
            while (lo < hi) {
                const int64_t mid = (lo + hi + 1) >> 1;
                if (us_at(mid) <= c0) lo = mid; else hi = mid - 1;
            }
            wfirst[w] = WorkerStart{lo, us_at(lo), us_at(lo + 1), 0};
        }
    }

    // 3. segments per merge group.  With fewer chunks than workers only the
    // first P workers take part, so every worker in play owns >= 1 chunk.
    // Groups that own no chunk (rare) are listed; the attention kernels give
    // them zeros and -inf (the plan holds no output pointer, so one plan
    // serves every call made with its arguments).
    const int64_t per_group = a.partial_mode ? 1 : a.N;
    int32_t* empty = reinterpret_cast<int32_t*>(a.ws + a.lay.off_empty);
    for (int64_t base = 0; base < a.G; base += kPlanThreads) {
        const int64_t g = base + tid;
        int64_t cnt = 0;
        if (g < a.G) {
            const int64_t first = us_at(g * per_group);
            const int64_t end = us_at((g + 1) * per_group);
            if (end > first) cnt = worker_of(end - 1, We, P) - worker_of(first, We, P) + 1;
            else empty[atomicAdd(&n_empty, 1)] = (int32_t)g;
            counters[g] = 0;
        }
        const int64_t incl = block_inclusive_scan(cnt, warp_tot);
        if (g < a.G) seg_base[g] = (int32_t)(carry + incl - cnt);
        __syncthreads();
        if (tid == kPlanThreads - 1) carry += incl;
        __syncthreads();
    }
    if (tid == 0) {
        seg_base[a.G] = (int32_t)carry;
        hdr->n_empty = (uint32_t)n_empty;
        hdr->plan_key = a.plan_key;
    }
}

}  // namespace

void launch_plan(const PlanArgs& a, cudaStream_t s) { plan_kernel<<<1, kPlanThreads, 0, s>>>(a); }

}  // namespace dcp

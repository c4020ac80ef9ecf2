// Prints the CUDA path's closed forms (owner_rank, local_pos, local_len and
// the 32-bit local_len32 of dcp_internal.cuh, compiled as host code) for a
// fixed set of (N, I, t) and (N, I, L, r); tests/test_host_logic.py compares
// every line with the oracle.
//   "T N I t owner local_pos"
//   "L N I L r local_len local_len32"   (local_len32 = -1 where L >= 2^31)
#include <cstdint>
#include <cstdio>

#include "../../context_decode_attention_gb300/csrc/dcp_internal.cuh"

int main() {
    const int NI[][2] = {{1, 1}, {2, 1}, {3, 5}, {4, 4}, {8, 1}, {8, 64}, {5, 1000}, {7, 3}, {8, 1 << 28}, {3, 1 << 30}};
    for (auto& ni : NI) {
        const int N = ni[0], I = ni[1];
        const int64_t period = (int64_t)N * I;
        const int64_t ts[] = {0, 1, 2, I - 1, I, I + 1, period - 1, period, period + 1, 3 * period + 7,
                              (int64_t)2147483647, ((int64_t)1 << 40) + 12345};
        for (int64_t t : ts) {
            if (t < 0) continue;
            std::printf("T %d %d %lld %lld %lld\n", N, I, (long long)t, (long long)dcp::owner_rank(t, N, I),
                        (long long)dcp::local_pos(t, N, I));
        }
        if (period <= 64)
            for (int64_t t = 0; t < 3 * period + 5; ++t)
                std::printf("T %d %d %lld %lld %lld\n", N, I, (long long)t, (long long)dcp::owner_rank(t, N, I),
                            (long long)dcp::local_pos(t, N, I));
        const int64_t Ls[] = {0, 1, 2, I - 1, I, I + 1, period - 1, period, period + 1, 5 * period + 3,
                              (int64_t)2147483647, ((int64_t)1 << 33) + 77};
        for (int64_t L : Ls) {
            if (L < 0) continue;
            for (int r = 0; r < N; ++r) {
                const long long l32 = L < ((int64_t)1 << 31) ? (long long)dcp::local_len32((uint32_t)L, r, N, I) : -1;
                std::printf("L %d %d %lld %d %lld %lld\n", N, I, (long long)L, r,
                            (long long)dcp::local_len(L, r, N, I), l32);
            }
        }
    }
    return 0;
}

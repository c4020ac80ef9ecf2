// Host check of the work split the planner and the MLA kernels share, on the
// real header code (compiled by nvcc as host code, run on the CPU):
//   * worker_begin / worker_of: the P chunks dealt to We = min(W, P) workers
//     as equal contiguous ranges, every worker in play owning >= 1 chunk, and
//     worker_of inverting the ranges;
//   * unit_of_chunk: the unit whose chunk range holds a worker's first chunk;
//   * TileCursor: the tile walk of one worker over random unit layouts (empty
//     units, per-rank partials or merged groups, a short shared-memory copy of
//     the unit prefix): every chunk of the range exactly once, in order, each
//     tile one or two chunks of one unit, and `first` / `last` exactly at the
//     range's merge-group boundaries (tiles of up to two chunks, and of up
//     to four for the CTA-pair kernels).
// Prints "ok" and exits 0, or names the first violated property and exits 1.
#include <cstdio>
#include <random>
#include <vector>

#include "../../context_decode_attention_gb300/csrc/mla_common.cuh"

using dcp::worker_begin;
using dcp::worker_of;
using dcp::mla::Tile;
using dcp::mla::TileCursor;
using dcp::mla::unit_of_chunk;

static int fail(const char* what, int it) {
    std::printf("FAIL %s (trial %d)\n", what, it);
    return 1;
}

int main() {
    std::mt19937_64 rng(20261202);
    // worker ranges
    const int64_t PW[][2] = {{1, 1}, {1, 1216}, {7, 1216}, {300, 1216}, {1216, 1216}, {131072, 1216}, {5, 3},
                             {1000003, 608}, {2047, 152}};
    for (auto& pw : PW) {
        const int64_t P = pw[0], W = pw[1], We = P < W ? P : W;
        if (worker_begin(0, We, P) != 0 || worker_begin(We, We, P) != P) return fail("range ends", 0);
        for (int64_t w = 0; w < We; ++w) {
            const int64_t b = worker_begin(w, We, P), e = worker_begin(w + 1, We, P);
            if (e <= b) return fail("worker owns no chunk", (int)w);
            if (worker_of(b, We, P) != w || worker_of(e - 1, We, P) != w) return fail("worker_of", (int)w);
        }
    }
    // tile walk
    for (int it = 0; it < 40000; ++it) {
        const int maxch = (it & 1) ? 4 : 2;
        const int N = 1 + (int)(rng() % 8), B = 1 + (int)(rng() % 6), pm = (int)(rng() % 2);
        const int U = N * B;
        std::vector<int64_t> us(U + 1, 0);
        for (int u = 0; u < U; ++u) us[u + 1] = us[u] + (rng() % 4 == 0 ? 0 : (int64_t)(rng() % 7));
        const int64_t P = us[U];
        if (P == 0) continue;
        const int64_t W = 1 + (int64_t)(rng() % 12), We = P < W ? P : W;
        for (int64_t w = 0; w < We; ++w) {
            const int64_t c0 = worker_begin(w, We, P), c1 = worker_begin(w + 1, We, P);
            const int64_t u0 = unit_of_chunk(us.data(), U, c0);
            if (!(us[u0] <= c0 && c0 < us[u0 + 1])) return fail("unit_of_chunk", it);
            std::vector<int64_t> cache;
            const int ncache = (int)(rng() % 5);
            for (int i = 0; i < ncache && u0 + i <= U; ++i) cache.push_back(us[u0 + i]);
            TileCursor cur;
            cur.init(us.data(), cache.data(), (int64_t)cache.size(), c0, c1, u0, N, pm, maxch);
            Tile t;
            int64_t c = c0, prev_group = -1;
            bool prev_last = true;
            while (cur.next(t)) {
                if (t.n_ch < 1 || t.n_ch > maxch) return fail("tile size", it);
                if (!(us[t.u] <= c && c + t.n_ch <= us[t.u + 1]) || us[t.u] + t.chunk != c)
                    return fail("tile chunks", it);
                if (t.group != (pm ? t.u : t.u / N)) return fail("group", it);
                // a short tile only where the range or the unit ends
                if (t.n_ch < maxch && c + t.n_ch < c1 && c + t.n_ch < us[t.u + 1]) return fail("short tile", it);
                if (t.first != (t.group != prev_group)) return fail("first", it);
                if (t.first && !prev_last) return fail("group reopened", it);
                c += t.n_ch;
                bool last = true;
                if (c < c1) {
                    int64_t v = t.u;
                    while (us[v + 1] <= c) ++v;
                    last = (pm ? v : v / N) != t.group;
                }
                if (t.last != last) return fail("last", it);
                prev_group = t.group;
                prev_last = t.last;
            }
            if (c != c1) return fail("coverage", it);
        }
    }
    std::printf("ok\n");
    return 0;
}

/*
 * CPU oracle for decode-context-parallel (DCP) decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The CUDA path never
 * calls it, and it shares no code, header, table or constant with that path.
 *
 * Everything here is the plain definition, written for a reader to check by
 * eye against the pages, in double precision:
 *
 *  - token ownership: rank(t) = floor(t / I) mod N  ("Breaking the
 *    Long-Sequence Inference Bottleneck ... Distributed Context Parallelism",
 *    section 2, the interleave-size rank equation and its worked table);
 *  - a rank keeps its own tokens in token order, so the local position of
 *    token t is the number of earlier tokens the same rank owns, and the local
 *    length of a request of L tokens is the number of its tokens the rank owns
 *    (both counted by enumeration; "vLLM DCP and PCP", Deep Dive 5,
 *    get_dcp_local_seq_lens: each backend sees its valid local KV prefix);
 *  - virtual block = block_size x N tokens, allocated by the total length;
 *    each rank needs ceil(local_len / block_size) physical blocks (section 2,
 *    "Virtual Block");
 *  - slot = block_table[rank][req][lpos / bs] * bs + lpos % bs for the owner,
 *    -1 for every other rank (section 2, slot-mapping figure text: -1 = skip);
 *  - blocks moved under prefill-decode disaggregation: the blocks that hold
 *    at least one token, with their token counts (section 2, "Practical
 *    considerations for PD disaggregation");
 *  - the prefill head-tail (zigzag) partition over K PCP ranks: pad to a
 *    multiple of 2K, cut into 2K equal chunks, rank k takes chunks k and
 *    2K - 1 - k ("Breaking the Long-Sequence Inference Bottleneck ...",
 *    section 4, "Head-tail concatenation strategy" and the PCP Size = 2
 *    walk-through);
 *  - attention of one query row against a token set K:
 *      s_j = scale * q . k_j,  L = log sum_j exp(s_j),
 *      o = sum_j exp(s_j) v_j / exp(L)   ("vLLM DCP and PCP", Deep Dive 6,
 *    "Deriving the partial and global outputs"), evaluated with the usual
 *    max shift; an empty set gives o = 0, L = -inf;
 *  - merge of per-rank (o_i, L_i): l = max L_i, a_i = exp(L_i - l),
 *      O = sum a_i o_i / sum a_i,  L = l + log sum a_i  (same section).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - GQA head mapping: query head h reads KV head floor(h / (Hq / Hkv));
 *  - MLA (absorbed form): every query head reads the one latent row per token;
 *    keys are the whole Dk-wide row, values are its first Dv columns;
 *  - multi-token decode: the Tq newest tokens are the queries; query t
 *    (0-based) sees global positions 0 .. L - Tq + t;
 *  - fp8 KV is e4m3fn times one per-tensor scale; bf16 is the top half of an
 *    IEEE binary32.
 */

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_FP8_E4M3 = 2 };

/* ---- storage decoding --------------------------------------------------- */

/* bf16: the upper 16 bits of an IEEE binary32. */
static double orc_bf16_value(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* fp8 e4m3fn (OCP 8-bit floating point, E4M3): 1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent 0 is subnormal (2^-6 * m/8); the pattern
 * S.1111.111 is NaN; there is no infinity. */
static double orc_fp8_e4m3_value(uint8_t bits) {
    int sign = (bits >> 7) & 1;
    int e = (bits >> 3) & 0xF;
    int m = bits & 0x7;
    double mag;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

static double orc_load(const void* base, int64_t idx, int64_t dtype, double scale) {
    switch (dtype) {
        case ORC_F32: return (double)((const float*)base)[idx];
        case ORC_BF16: return orc_bf16_value(((const uint16_t*)base)[idx]);
        case ORC_FP8_E4M3: return orc_fp8_e4m3_value(((const uint8_t*)base)[idx]) * scale;
        default: return NAN;
    }
}

/* Decode n stored values to double (scale multiplies fp8 only). */
void orc_decode(const void* src, int64_t n, int64_t dtype, double scale, double* dst) {
    for (int64_t i = 0; i < n; ++i) dst[i] = orc_load(src, i, dtype, scale);
}

/* ---- token ownership and metadata -------------------------------------- */

/* The interleave rule: rank = floor(token_id / interleave_size) mod CP_size. */
int64_t orc_rank_of(int64_t t, int64_t N, int64_t I) { return (t / I) % N; }

/* For tokens 0..L-1: owning rank and local position (running count per rank). */
void orc_local_layout(int64_t L, int64_t N, int64_t I, int32_t* rank, int64_t* lpos) {
    int64_t* count = (int64_t*)calloc((size_t)N, sizeof(int64_t));
    for (int64_t t = 0; t < L; ++t) {
        int64_t r = orc_rank_of(t, N, I);
        rank[t] = (int32_t)r;
        lpos[t] = count[r]++;
    }
    free(count);
}

/* Number of the first L tokens that rank r owns (enumeration). */
int64_t orc_local_len(int64_t L, int64_t r, int64_t N, int64_t I) {
    int64_t n = 0;
    for (int64_t t = 0; t < L; ++t) n += (orc_rank_of(t, N, I) == r);
    return n;
}

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/*
 * Slot mapping for T tokens (tok_req[i], tok_pos[i]) of B requests whose
 * global lengths are seq_lens[b].  Writes:
 *   owner[T]            owning rank of each token
 *   local_lens[N][B]    tokens of request b that rank r owns
 *   virt_blocks[B]      ceil(L_b / (bs * N))
 *   rank_blocks[N][B]   ceil(local_lens / bs)
 *   slots[N][T]         slot in the pool for the owner, -1 for other ranks
 *                       (only when block_tables is not NULL)
 * Returns 0, or -1 if a token lies outside its request or a needed block id
 * is missing (< 0) in the table.
 */
int orc_slot_mapping(int64_t N, int64_t I, int64_t bs, int64_t B, const int32_t* seq_lens,
                     int64_t T, const int32_t* tok_req, const int64_t* tok_pos,
                     const int32_t* block_tables, int64_t max_blocks,
                     int8_t* owner, int64_t* slots, int32_t* local_lens,
                     int32_t* virt_blocks, int32_t* rank_blocks) {
    int status = 0;
    for (int64_t b = 0; b < B; ++b) {
        int64_t L = seq_lens[b];
        virt_blocks[b] = (int32_t)ceil_div(L, bs * N);
        for (int64_t r = 0; r < N; ++r) {
            int64_t n = orc_local_len(L, r, N, I);
            local_lens[r * B + b] = (int32_t)n;
            rank_blocks[r * B + b] = (int32_t)ceil_div(n, bs);
        }
    }
    /* bucket the tokens by request, then one running-count pass per request */
    int64_t* first = (int64_t*)calloc((size_t)B + 1, sizeof(int64_t));
    int64_t* order = (int64_t*)malloc((size_t)(T > 0 ? T : 1) * sizeof(int64_t));
    for (int64_t i = 0; i < T; ++i) {
        if (tok_req[i] < 0 || tok_req[i] >= B) {
            status = -1;
            owner[i] = -1;
            if (slots)
                for (int64_t r = 0; r < N; ++r) slots[r * T + i] = -1;
            continue;
        }
        first[tok_req[i] + 1]++;
    }
    for (int64_t b = 0; b < B; ++b) first[b + 1] += first[b];
    int64_t* fill = (int64_t*)calloc((size_t)B + 1, sizeof(int64_t));
    for (int64_t i = 0; i < T; ++i) {
        if (tok_req[i] < 0 || tok_req[i] >= B) continue;
        order[first[tok_req[i]] + fill[tok_req[i]]++] = i;
    }
    for (int64_t b = 0; b < B; ++b) {
        int64_t L = seq_lens[b];
        if (first[b + 1] == first[b]) continue;
        int32_t* rank = (int32_t*)malloc((size_t)(L > 0 ? L : 1) * sizeof(int32_t));
        int64_t* lpos = (int64_t*)malloc((size_t)(L > 0 ? L : 1) * sizeof(int64_t));
        orc_local_layout(L, N, I, rank, lpos);
        for (int64_t k = first[b]; k < first[b + 1]; ++k) {
            int64_t i = order[k];
            int64_t p = tok_pos[i];
            if (p < 0 || p >= L) {
                status = -1;
                owner[i] = -1;
                if (slots)
                    for (int64_t r = 0; r < N; ++r) slots[r * T + i] = -1;
                continue;
            }
            int64_t r_own = rank[p];
            owner[i] = (int8_t)r_own;
            if (!slots) continue;
            for (int64_t r = 0; r < N; ++r) slots[r * T + i] = -1;
            int64_t lp = lpos[p];
            int64_t blk = lp / bs;
            int32_t id = (blk < max_blocks) ? block_tables[(r_own * B + b) * max_blocks + blk] : -1;
            if (id < 0) { status = -1; continue; }
            slots[r_own * T + i] = (int64_t)id * bs + lp % bs;
        }
        free(rank);
        free(lpos);
    }
    free(first);
    free(order);
    free(fill);
    return status;
}

/*
 * Blocks moved under prefill-decode disaggregation ("Breaking the
 * Long-Sequence Inference Bottleneck ...", section 2, "Practical
 * considerations for PD disaggregation": KV moves between nodes in whole
 * blocks, and a block that holds no token need not move).  By enumeration:
 * walk every token of each request, put it in its owner's local block
 * lpos / bs, count the tokens per (rank, local block), and list each rank's
 * local blocks that hold at least one token, in block-table order.
 *   counts[N][B]              listed blocks
 *   blocks[N][B][max_blocks]  their ids, -1 after the last
 *   fills[N][B][max_blocks]   their token counts, 0 after the last
 *   totals[2]                 {sum of counts * bs (slots moved), sum of tokens}
 * Returns 0, or -1 if a listed block's table entry lies outside
 * [0, num_blocks) (listed as -1) or a rank needs more than max_blocks blocks
 * (the list stops at max_blocks).
 */
int orc_transfer_blocks(int64_t N, int64_t I, int64_t bs, int64_t B, const int32_t* seq_lens,
                        const int32_t* block_tables, int64_t max_blocks, int64_t num_blocks,
                        int32_t* counts, int32_t* blocks, int32_t* fills, int64_t* totals) {
    int status = 0;
    totals[0] = 0;
    totals[1] = 0;
    for (int64_t b = 0; b < B; ++b) {
        int64_t L = seq_lens[b] > 0 ? seq_lens[b] : 0;
        int64_t nblk = L / bs + 2;  /* local blocks any rank could touch */
        int64_t* tally = (int64_t*)calloc((size_t)(N * nblk), sizeof(int64_t));
        int32_t* rank = (int32_t*)malloc((size_t)(L > 0 ? L : 1) * sizeof(int32_t));
        int64_t* lpos = (int64_t*)malloc((size_t)(L > 0 ? L : 1) * sizeof(int64_t));
        orc_local_layout(L, N, I, rank, lpos);
        for (int64_t t = 0; t < L; ++t) tally[rank[t] * nblk + lpos[t] / bs]++;
        for (int64_t r = 0; r < N; ++r) {
            int32_t* ob = blocks + (r * B + b) * max_blocks;
            int32_t* of = fills + (r * B + b) * max_blocks;
            for (int64_t k = 0; k < max_blocks; ++k) { ob[k] = -1; of[k] = 0; }
            int64_t c = 0;
            for (int64_t k = 0; k < nblk; ++k) {
                int64_t n = tally[r * nblk + k];
                if (n == 0) continue;
                totals[1] += n;
                totals[0] += bs;
                if (c >= max_blocks || k >= max_blocks) { status = -1; continue; }
                int32_t id = block_tables[(r * B + b) * max_blocks + k];
                if (id < 0 || id >= num_blocks) { status = -1; id = -1; }
                ob[c] = id;
                of[c] = (int32_t)n;
                ++c;
            }
            counts[r * B + b] = (int32_t)c;
        }
        free(tally);
        free(rank);
        free(lpos);
    }
    return status;
}

/*
 * Prefill context parallelism, head-tail partition ("Breaking the
 * Long-Sequence Inference Bottleneck ...", section 4): request b's new tokens
 * are the positions ctx_lens[b] .. ctx_lens[b] + q_lens[b] - 1.  Following
 * the page's four steps: (1) align the count up to a multiple of 2K; (2) cut
 * the aligned run into 2K equal chunks; (3) PCP rank k takes chunk k (head)
 * and chunk 2K - 1 - k (tail); (4) rank k holds its head chunk followed by
 * its tail chunk.  pos[b][0 .. max_q) receives every rank's tokens in rank
 * order (rank 0's 2c positions, then rank 1's, ...: the order an AllGather of
 * the ranks' queries leaves them in); an aligned position past the request's
 * last token is padding, -1, as is every row past the aligned length.
 * padded_len[b] = the aligned length.  Returns 0, or -1 if a request's
 * aligned length exceeds max_q (its rows are then all -1).
 */
int orc_pcp_partition(int64_t K, int64_t B, const int32_t* ctx_lens, const int32_t* q_lens, int64_t max_q,
                      int32_t* pos, int32_t* padded_len) {
    int status = 0;
    for (int64_t b = 0; b < B; ++b) {
        int32_t* row = pos + b * max_q;
        for (int64_t j = 0; j < max_q; ++j) row[j] = -1;
        const int64_t n = q_lens[b] > 0 ? q_lens[b] : 0;
        const int64_t aligned = (n + 2 * K - 1) / (2 * K) * (2 * K); /* step 1 */
        padded_len[b] = (int32_t)aligned;
        if (aligned > max_q) {
            status = -1;
            continue;
        }
        const int64_t c = aligned / (2 * K); /* step 2: chunk i = [i c, (i + 1) c) */
        int64_t out = 0;
        for (int64_t k = 0; k < K; ++k) {
            const int64_t chunks[2] = {k, 2 * K - 1 - k}; /* step 3 */
            for (int h = 0; h < 2; ++h)                  /* step 4: head, then tail */
                for (int64_t j = 0; j < c; ++j) {
                    const int64_t rel = chunks[h] * c + j;
                    row[out++] = rel < n ? (int32_t)(ctx_lens[b] + rel) : -1;
                }
        }
    }
    return status;
}

/* ---- attention ---------------------------------------------------------- */

/*
 * Attention of query rows against the dense per-request keys/values.
 *   q      [B][Tq][Hq][Dk]        (q_dtype: f32 or bf16)
 *   k      [T_total][Hkv][Dk]     (kv_dtype; MLA: the latent rows, Hkv = 1)
 *   v      [T_total][Hkv][Dv]     (GQA only; NULL for MLA)
 *   request b owns rows req_start[b] .. req_start[b] + seq_lens[b] - 1
 * rank < 0: all tokens the query may see; rank >= 0: only those rank owns.
 * rows: flat ids ((b * Tq + t) * Hq + h), or NULL for all B*Tq*Hq rows.
 * out [nrows][Dv], lse [nrows] (natural log; -inf and zeros for an empty set).
 */
void orc_attention(int64_t layout, int64_t B, int64_t Tq, int64_t Hq, int64_t Hkv,
                   int64_t Dk, int64_t Dv, const int32_t* seq_lens, const int64_t* req_start,
                   const void* q, int64_t q_dtype, const void* k, const void* v,
                   int64_t kv_dtype, double kv_scale, double softmax_scale,
                   int64_t N, int64_t I, int64_t rank, int64_t nrows, const int64_t* rows,
                   double* out, double* lse, int64_t nthreads) {
    int64_t total_rows = rows ? nrows : B * Tq * Hq;
    int64_t max_len = 0;
    for (int64_t b = 0; b < B; ++b)
        if (seq_lens[b] > max_len) max_len = seq_lens[b];
    int64_t group = Hq / Hkv;
#pragma omp parallel num_threads((int)(nthreads > 0 ? nthreads : 1))
    {
        double* s = (double*)malloc((size_t)(max_len > 0 ? max_len : 1) * sizeof(double));
        int64_t* idx = (int64_t*)malloc((size_t)(max_len > 0 ? max_len : 1) * sizeof(int64_t));
        double* qv = (double*)malloc((size_t)Dk * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t n = 0; n < total_rows; ++n) {
            int64_t id = rows ? rows[n] : n;
            int64_t h = id % Hq;
            int64_t t = (id / Hq) % Tq;
            int64_t b = id / (Hq * Tq);
            int64_t L = seq_lens[b];
            int64_t g = L - Tq + t + 1; /* tokens 0..g-1 are visible */
            int64_t kvh = h / group;
            for (int64_t d = 0; d < Dk; ++d) qv[d] = orc_load(q, id * Dk + d, q_dtype, 1.0);
            int64_t cnt = 0;
            double m = -INFINITY;
            for (int64_t j = 0; j < g; ++j) {
                if (rank >= 0 && orc_rank_of(j, N, I) != rank) continue;
                int64_t row = (req_start[b] + j) * Hkv + kvh;
                double dot = 0.0;
                for (int64_t d = 0; d < Dk; ++d) dot += qv[d] * orc_load(k, row * Dk + d, kv_dtype, kv_scale);
                s[cnt] = softmax_scale * dot;
                idx[cnt] = row;
                if (s[cnt] > m) m = s[cnt];
                ++cnt;
            }
            double* o = out + n * Dv;
            for (int64_t d = 0; d < Dv; ++d) o[d] = 0.0;
            if (cnt == 0) {
                lse[n] = -INFINITY;
                continue;
            }
            double sum = 0.0;
            for (int64_t c = 0; c < cnt; ++c) sum += exp(s[c] - m);
            double L_row = m + log(sum);
            lse[n] = L_row;
            for (int64_t c = 0; c < cnt; ++c) {
                double w = exp(s[c] - L_row);
                if (layout == 1) {
                    for (int64_t d = 0; d < Dv; ++d) o[d] += w * orc_load(k, idx[c] * Dk + d, kv_dtype, kv_scale);
                } else {
                    for (int64_t d = 0; d < Dv; ++d) o[d] += w * orc_load(v, idx[c] * Dv + d, kv_dtype, kv_scale);
                }
            }
        }
        free(s);
        free(idx);
        free(qv);
    }
}

/*
 * Exact merge of N partial results per row.
 *   o_parts [N][rows][Dv], lse_parts [N][rows]  ->  out [rows][Dv], lse [rows]
 * Ranks whose LSE is -inf (no tokens) carry no weight.
 */
void orc_merge(int64_t N, int64_t rows, int64_t Dv, const double* o_parts, const double* lse_parts,
               double* out, double* lse) {
    for (int64_t n = 0; n < rows; ++n) {
        double l = -INFINITY;
        for (int64_t i = 0; i < N; ++i)
            if (lse_parts[i * rows + n] > l) l = lse_parts[i * rows + n];
        double* o = out + n * Dv;
        for (int64_t d = 0; d < Dv; ++d) o[d] = 0.0;
        if (l == -INFINITY) {
            lse[n] = -INFINITY;
            continue;
        }
        double asum = 0.0;
        for (int64_t i = 0; i < N; ++i) {
            double a = exp(lse_parts[i * rows + n] - l);
            asum += a;
            for (int64_t d = 0; d < Dv; ++d) o[d] += a * o_parts[(i * rows + n) * Dv + d];
        }
        for (int64_t d = 0; d < Dv; ++d) o[d] /= asum;
        lse[n] = l + log(asum);
    }
}

/*
 * Lightning Indexer — CPU oracle (TEST INFRASTRUCTURE ONLY).
 *
 * This file is the plain, slow, obviously-correct definition of what the
 * indexer computes. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it. The product path (the CUDA library under
 * sparse_attention_key_gb300/) never calls, links or includes it, and it
 * shares no code, header, table or helper with that path.
 *
 * Source of the method: the Hugging Face discussion "Notes from an NVFP4 port
 * of Kimi K3.1 Pro" (moonshotai/Kimi-K3.1-Pro, discussion 7): the paragraph
 * that describes the indexer, items (3) and (4) of the list "Details that
 * silently change the answer", and the closing paragraph on why the port's own
 * measurements leave selection unused. Readings of that text that
 * the page leaves open are stated at each function.
 *
 * Arithmetic: IEEE fp64 throughout, inputs converted exactly from bf16/fp32.
 * Build: plain C11, no intrinsics, no OpenMP, no -ffast-math:
 *     gcc -O2 -std=c11 -fPIC -shared indexer_oracle.c -o liboracle.so -lm
 *
 * Parity pins (tests/test_oracle.py, run without a GPU):
 *   - oracle_select: hand-derived tie-rule cases (tests/golden/), brute force
 *     over all subsets on tiny rows, keep-all for n <= K, all-equal rows,
 *     distinct-score rows against an independent sort, +0/-0 equality.
 *   - oracle_scores: a single nonzero head against a library GEMM (numpy
 *     float64 matmul + relu), linearity in the head weights, causal length.
 *   - oracle_key_layernorm: constant rows, +/-a rows (closed form), and the
 *     fp64 result against torch.nn.functional.layer_norm in float64; the
 *     bf16 rounding against the fp32 round-to-nearest-even bit rule.
 *   - oracle_sparse_mla: one selected row (o = its latent), identical rows,
 *     a zero query (o = the mean latent, lse = log n), a large scale (o tends
 *     to the top-logit row), order of the selected rows, and the result
 *     against scipy's softmax/logsumexp over a numpy matmul of the rows.
 *   - oracle_e4m3_to_double: hand-derived codes (zero, subnormals, 1.0, the
 *     largest finite 448, NaN) and every code against torch's float8_e4m3fn.
 *   - oracle_sparse_mla_fp8: equal to oracle_sparse_mla on rows whose
 *     dequantised values are exact bf16 values; one selected row.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define IDX_HEADS 32   /* indexer heads per query */
#define IDX_DIM 128    /* width of each head, of a key and of the LayerNorm */

/* ---------------------------------------------------------------------------
 * Number formats
 * ------------------------------------------------------------------------- */

/* bf16 bit pattern -> exact double (bf16 is the top half of an IEEE fp32). */
double oracle_bf16_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * double -> bf16, round to nearest, ties to even, in one rounding step.
 * bf16 has 8 significant bits for normal numbers (exponent >= -126) and a
 * fixed quantum of 2^-133 below that. The quantum q of x is a power of two,
 * x/q is exact in double, rint() rounds it to an integer in the current
 * (default: nearest-even) mode, and the product is the rounded value, which
 * is exactly representable in fp32 and therefore in bf16.
 */
uint16_t oracle_double_to_bf16(double x) {
    if (isnan(x)) return (uint16_t)0x7FC0;
    if (x == 0.0) return signbit(x) ? (uint16_t)0x8000 : (uint16_t)0x0000;
    if (isinf(x)) return signbit(x) ? (uint16_t)0xFF80 : (uint16_t)0x7F80;
    int e;
    (void)frexp(x, &e);        /* |x| = m * 2^e with m in [0.5, 1) */
    int exp_unbiased = e - 1;  /* |x| in [2^exp_unbiased, 2^(exp_unbiased+1)) */
    if (exp_unbiased < -126) exp_unbiased = -126;
    double q = ldexp(1.0, exp_unbiased - 7);
    double r = rint(x / q) * q;
    if (fabs(r) >= ldexp(1.0, 128)) return signbit(x) ? (uint16_t)0xFF80 : (uint16_t)0x7F80;
    float f = (float)r;        /* exact */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* ---------------------------------------------------------------------------
 * Step 1 — key LayerNorm.
 * The page: indexer keys are taken from the attention input and normalised by
 * a LayerNorm of width 128 that has a weight and a bias. Reading: the standard
 * LayerNorm over the 128 features of one key, biased variance, eps inside
 * the square root, y = (x - mean) / sqrt(var + eps) * gamma + beta; the
 * result is stored in the 16-bit key cache (the page keeps the indexer in
 * 16-bit), rounded to bf16 nearest-even.
 *
 * k_raw   [n_rows,128] bf16 bits (host)
 * gamma   [128] double, beta [128] double (exact copies of the parameters)
 * k_out   [n_rows,128] bf16 bits (host)
 * y_exact [n_rows,128] double, or NULL: the unrounded fp64 result
 * ------------------------------------------------------------------------- */
void oracle_key_layernorm(const uint16_t* k_raw, const double* gamma, const double* beta,
                          double eps, int64_t n_rows, uint16_t* k_out, double* y_exact) {
    for (int64_t r = 0; r < n_rows; ++r) {
        const uint16_t* x = k_raw + r * IDX_DIM;
        double mean = 0.0;
        for (int d = 0; d < IDX_DIM; ++d) mean += oracle_bf16_to_double(x[d]);
        mean /= IDX_DIM;
        double var = 0.0;
        for (int d = 0; d < IDX_DIM; ++d) {
            double c = oracle_bf16_to_double(x[d]) - mean;
            var += c * c;
        }
        var /= IDX_DIM;
        double inv = 1.0 / sqrt(var + eps);
        for (int d = 0; d < IDX_DIM; ++d) {
            double y = (oracle_bf16_to_double(x[d]) - mean) * inv * gamma[d] + beta[d];
            if (y_exact) y_exact[r * IDX_DIM + d] = y;
            k_out[r * IDX_DIM + d] = oracle_double_to_bf16(y);
        }
    }
}

/* ---------------------------------------------------------------------------
 * Steps 2-3 — head scores, relu, head-weighted sum, for one query.
 * The page: each of 32 heads (width 128) scores every key of the causal past
 * with relu of its dot product with the key, and a vector of per-head weights
 * combines the heads before selection. Reading: S[s] = sum_h w[h] * max(q_h . k_s, 0) for every key s of
 * the causal history 0..n-1 (n = query position + 1). There is no rotary
 * (index_rope_dim is 0, item (3) of the page's list). No scale factor is
 * printed; any scale is taken to be folded into w.
 *
 * q_t [32,128] bf16 bits, k_seq [n,128] bf16 bits (the sequence's post-LN
 * keys), w_t [32] fp32, S_out [n] double.
 * ------------------------------------------------------------------------- */
void oracle_scores(const uint16_t* q_t, const uint16_t* k_seq, const float* w_t, int64_t n,
                   double* S_out) {
    double q[IDX_HEADS][IDX_DIM];
    for (int h = 0; h < IDX_HEADS; ++h)
        for (int d = 0; d < IDX_DIM; ++d) q[h][d] = oracle_bf16_to_double(q_t[h * IDX_DIM + d]);
    double k[IDX_DIM];
    for (int64_t s = 0; s < n; ++s) {
        for (int d = 0; d < IDX_DIM; ++d) k[d] = oracle_bf16_to_double(k_seq[s * IDX_DIM + d]);
        double S = 0.0;
        for (int h = 0; h < IDX_HEADS; ++h) {
            double dot = 0.0;
            for (int d = 0; d < IDX_DIM; ++d) dot += q[h][d] * k[d];
            double relu = dot > 0.0 ? dot : 0.0;
            S += (double)w_t[h] * relu;
        }
        S_out[s] = S;
    }
}

/* ---------------------------------------------------------------------------
 * Steps 4-5 — exact top-K with the page's tie and order rule.
 * The page: the top 2048 positions are kept with no approximation (indexer
 * paragraph). Item (4): scores equal to the threshold at the K boundary are a
 * tie; the output first lists the kept positions that score above the
 * threshold, by increasing position, then the kept part of the tie group, by
 * increasing position starting from its lowest; it is not a list sorted by
 * score. Closing paragraph: a history of at most K keys loses nothing, so
 * every position is kept, in increasing order (sparse equals dense there).
 *
 * Reading of the threshold: sort all n positions by (score descending,
 * position ascending); tau is the score of the K-th entry. The first K
 * entries are kept: those with score > tau (fewer than K) and the lowest
 * positions of the group with score == tau. Scores compare numerically, so
 * -0 equals +0.
 *
 * S [n] double; idx_out [K] int32, filled with the selection and then -1.
 * Returns the number of positions emitted, min(n, K).
 * ------------------------------------------------------------------------- */
typedef struct {
    double score;
    int64_t pos;
} oracle_entry;

static int oracle_entry_order(const void* pa, const void* pb) {
    const oracle_entry* a = (const oracle_entry*)pa;
    const oracle_entry* b = (const oracle_entry*)pb;
    if (a->score > b->score) return -1;  /* higher score first */
    if (a->score < b->score) return 1;
    if (a->pos < b->pos) return -1;      /* then lower position first */
    if (a->pos > b->pos) return 1;
    return 0;
}

static int oracle_pos_ascending(const void* pa, const void* pb) {
    int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
    return (a > b) - (a < b);
}

int64_t oracle_select(const double* S, int64_t n, int32_t K, int32_t* idx_out) {
    for (int32_t i = 0; i < K; ++i) idx_out[i] = -1;
    if (n <= 0) return 0;
    if (n <= K) {  /* dormant selection: every position, ascending */
        for (int64_t s = 0; s < n; ++s) idx_out[s] = (int32_t)s;
        return n;
    }
    oracle_entry* e = (oracle_entry*)malloc((size_t)n * sizeof *e);
    if (!e) return -1;
    for (int64_t s = 0; s < n; ++s) {
        e[s].score = S[s];
        e[s].pos = s;
    }
    qsort(e, (size_t)n, sizeof *e, oracle_entry_order);
    double tau = e[K - 1].score;
    int32_t out = 0;
    for (int32_t i = 0; i < K; ++i)          /* strictly above the threshold */
        if (e[i].score > tau) idx_out[out++] = (int32_t)e[i].pos;
    int32_t n_above = out;
    qsort(idx_out, (size_t)n_above, sizeof *idx_out, oracle_pos_ascending);
    for (int32_t i = 0; i < K; ++i)          /* the boundary group's kept part */
        if (e[i].score == tau) idx_out[out++] = (int32_t)e[i].pos;
    qsort(idx_out + n_above, (size_t)(out - n_above), sizeof *idx_out, oracle_pos_ascending);
    free(e);
    return out;
}

/* ---------------------------------------------------------------------------
 * The whole indexer over a packed ragged batch, for query rows
 * [row_begin, row_end). Layout (the same one the CUDA library uses):
 *   q [T,32,128] bf16, k [cu_k[B],128] bf16 (post-LN cache), w [T,32] fp32,
 *   q_pos [T] int32 (position of the query within its sequence),
 *   cu_q [B+1], cu_k [B+1] int32 (sequence b owns query rows cu_q[b]..cu_q[b+1]
 *   and key rows cu_k[b]..cu_k[b+1]).
 * Output: idx [T,K] int32 sequence-local positions padded with -1;
 *   cnt [T] int32 (number emitted) or NULL; scores_out [T,ld] double or NULL
 *   (the row's n scores; the rest untouched).
 * Returns 0, or -1 on an argument error (position outside its sequence).
 * ------------------------------------------------------------------------- */
int oracle_score_topk(const uint16_t* q, const uint16_t* k, const float* w, const int32_t* q_pos,
                      const int32_t* cu_q, const int32_t* cu_k, int32_t B, int32_t K,
                      int32_t* idx, int32_t* cnt, double* scores_out, int64_t ld,
                      int64_t row_begin, int64_t row_end) {
    for (int32_t b = 0; b < B; ++b) {
        int64_t len_k = (int64_t)cu_k[b + 1] - cu_k[b];
        for (int64_t t = cu_q[b]; t < cu_q[b + 1]; ++t) {
            if (t < row_begin || t >= row_end) continue;
            int64_t n = (int64_t)q_pos[t] + 1;  /* causal: keys 0..q_pos inclusive */
            if (q_pos[t] < 0 || n > len_k) return -1;
            double* S = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof *S);
            if (!S) return -1;
            oracle_scores(q + t * IDX_HEADS * IDX_DIM, k + (int64_t)cu_k[b] * IDX_DIM,
                          w + t * IDX_HEADS, n, S);
            int64_t c = oracle_select(S, n, K, idx + t * K);
            if (cnt) cnt[t] = (int32_t)c;
            if (scores_out) memcpy(scores_out + t * ld, S, (size_t)n * sizeof *S);
            free(S);
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Sparse NoPE MLA attention over the selected positions (one query token)
 *
 * The port notes ("Notes from an NVFP4 port of Kimi K3.1 Pro", opening
 * paragraph and item (5)): the indexer keeps the best 2048 keys for each
 * full-attention layer, and those layers are NoPE multi-head latent attention
 * (the 64 "rope" dims are ordinary key dims). The TokenSpeed post on Kimi K3,
 * section 2 (MLA): per token the cache holds a shared 512-wide latent and a
 * 64-wide key component, there are 96 heads, and decode moves the query into
 * the compressed space. Neither page writes the attention out, so this is the
 * plain reading: head h of the absorbed query q_h (576 = 512 latent + 64 key
 * dims) attends to the selected cache rows c_j (576 wide),
 *     l_hj = scale * (q_h . c_j),   p_h = softmax over j of l_h,
 *     o_h  = sum_j p_hj * c_j[0..512),   lse_h = log sum_j exp(l_hj);
 * the value of a row is its 512-wide latent and the softmax scale is an
 * argument. With no selected row, o_h = 0 and lse_h = -infinity.
 * ------------------------------------------------------------------------- */
#define MLA_DIM 576    /* cache row: 512 latent + 64 key dims */
#define MLA_VDIM 512   /* latent (value) part */

void oracle_sparse_mla(const uint16_t* q_t, const uint16_t* cache, const int64_t* rows, int64_t n,
                       int32_t heads, double scale, double* o, double* lse) {
    double* logit = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    for (int32_t h = 0; h < heads; ++h) {
        const uint16_t* qh = q_t + (int64_t)h * MLA_DIM;
        double* oh = o + (int64_t)h * MLA_VDIM;
        for (int d = 0; d < MLA_VDIM; ++d) oh[d] = 0.0;
        if (n <= 0) {
            lse[h] = -INFINITY;
            continue;
        }
        double m = -INFINITY;
        for (int64_t j = 0; j < n; ++j) {
            const uint16_t* c = cache + rows[j] * MLA_DIM;
            double dot = 0.0;
            for (int d = 0; d < MLA_DIM; ++d) dot += oracle_bf16_to_double(qh[d]) * oracle_bf16_to_double(c[d]);
            logit[j] = scale * dot;
            if (logit[j] > m) m = logit[j];
        }
        double sum = 0.0;
        for (int64_t j = 0; j < n; ++j) sum += exp(logit[j] - m);
        for (int64_t j = 0; j < n; ++j) {
            const double p = exp(logit[j] - m) / sum;
            const uint16_t* c = cache + rows[j] * MLA_DIM;
            for (int d = 0; d < MLA_VDIM; ++d) oh[d] += p * oracle_bf16_to_double(c[d]);
        }
        lse[h] = m + log(sum);
    }
    free(logit);
}

/* ---------------------------------------------------------------------------
 * FP8 (E4M3) cache rows for the sparse MLA attention.
 * "Kimi K3 on AMD Instinct GPUs with TokenSpeed", section 2 (MLA), stores the
 * MLA cache in FP8. Reading: each cached row is 576 E4M3 codes and one scale
 * (a row's value is scale x the code's value); the pages give no scale
 * granularity, and per row is the plainest. E4M3 as commonly defined (OCP
 * 8-bit floating point): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 * bits; exponent 0 holds the subnormals m/8 x 2^-6; the pattern with all
 * exponent and mantissa bits set is NaN; there is no infinity.
 * ------------------------------------------------------------------------- */

double oracle_e4m3_to_double(uint8_t b) {
    const int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
    if (e == 15 && m == 7) return NAN;
    const double mag = e == 0 ? ldexp((double)m, -9)               /* m/8 x 2^(1-7) */
                              : ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/*
 * The attention of oracle_sparse_mla over FP8 rows: c_j[d] = scale_row[rows[j]]
 * x e4m3(cache8[rows[j] * 576 + d]), in fp64; the same softmax, output and
 * log-sum-exp.
 */
void oracle_sparse_mla_fp8(const uint16_t* q_t, const uint8_t* cache8, const double* row_scale,
                           const int64_t* rows, int64_t n, int32_t heads, double scale, double* o,
                           double* lse) {
    double* logit = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    for (int32_t h = 0; h < heads; ++h) {
        const uint16_t* qh = q_t + (int64_t)h * MLA_DIM;
        double* oh = o + (int64_t)h * MLA_VDIM;
        for (int d = 0; d < MLA_VDIM; ++d) oh[d] = 0.0;
        if (n <= 0) {
            lse[h] = -INFINITY;
            continue;
        }
        double m = -INFINITY;
        for (int64_t j = 0; j < n; ++j) {
            const uint8_t* c = cache8 + rows[j] * MLA_DIM;
            const double sr = row_scale[rows[j]];
            double dot = 0.0;
            for (int d = 0; d < MLA_DIM; ++d)
                dot += oracle_bf16_to_double(qh[d]) * (sr * oracle_e4m3_to_double(c[d]));
            logit[j] = scale * dot;
            if (logit[j] > m) m = logit[j];
        }
        double sum = 0.0;
        for (int64_t j = 0; j < n; ++j) sum += exp(logit[j] - m);
        for (int64_t j = 0; j < n; ++j) {
            const double p = exp(logit[j] - m) / sum;
            const uint8_t* c = cache8 + rows[j] * MLA_DIM;
            const double sr = row_scale[rows[j]];
            for (int d = 0; d < MLA_VDIM; ++d) oh[d] += p * (sr * oracle_e4m3_to_double(c[d]));
        }
        lse[h] = m + log(sum);
    }
    free(logit);
}

/*
 * Plain, slow CPU oracle for absorbed (MQA-mode) Multi-head Latent Attention decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU
 * baseline leg may load this code.  It shares nothing with the CUDA library: no
 * header, no helper, no table.  Every value is decoded from its stored bits and all
 * arithmetic is done in IEEE double.  The softmax is the textbook two-pass form
 * (maximum first, then the sum of exponentials); there is no blocking, no online
 * rescaling and no fusion.
 *
 * What it computes, for one request with query heads h and the token list N:
 *
 *   s_t       = scale * ( q~[h] . c[t]  +  q_R[h] . k_R[t] )             t in N
 *   m         = max_t s_t,       l = sum_t exp(s_t - m)
 *   out[h, :] = (1 / l) * sum_t exp(s_t - m) * c[t, :]
 *   lse[h]    = m + ln(l)
 *
 * Sources (page title, section):
 *  - "MLA 在极长上下文下的显存带宽突围：128K 场景下的算子访存深度解析", section
 *    "运行期矩阵吸收" (run-time matrix absorption): the absorbed query q~ = q^C W^UK and the
 *    score q~ (c^KV)^T + q^R (k^R)^T, read against a 576-wide cache entry (512 latent +
 *    64 decoupled-RoPE key).  The "+" between the two terms is lost in the extracted
 *    text; the guide below and the two-term form of the cache entry fix it.
 *  - "MLA & DSA 推理性能优化指南", §1.1 (absorbed path: W_UK folded into the query,
 *    attention computed in latent space, only c_t^KV and the 64-d RoPE key cached) and
 *    §4.1 (decode reads (d_c + d_rope) values per token).  The output stays in the
 *    512-d latent space; W^UV is applied afterwards (mla_oracle_project, at the end of
 *    this file, next to the query absorption mla_oracle_absorb).
 *  - Same guide, §4.2: the token-sparse (DSA) decode attends over the selected top-k
 *    tokens only.
 *  - Same guide, §5.3: the FP8 latent cache.  The pages do not fix the FP8 format; this
 *    oracle reads e4m3 "fn" (bias 7, no infinities, S.1111.111 is NaN) with one fp32
 *    scale per 128 latent channels.  The dequantized latent is what the guide defines:
 *    x = e4m3(code) * scale, exact in double (a 4-bit significand times a 24-bit one).
 *    A second mode, used only as a tighter check of one GPU operand choice, rounds that
 *    value the way a bf16 tensor-core operand would: x = bf16_rne(fp32(e4m3(code)) * scale),
 *    the product formed in fp32 and rounded once to bf16.  The pages fix no intermediate
 *    precision, so only the exact mode is the definition.
 *
 * Readings where the pages are silent: the scale multiplies the raw score before the
 * exponential; lse is the natural log of the normaliser of the scaled scores; an empty
 * token list gives out = 0 and lse = -inf; a sparse index of -1 is padding and is
 * skipped; a repeated index is attended once per occurrence.
 *
 * Paged cache addressing: logical token t of request b lives in physical page
 * block_table[b][t / 64] at row t % 64.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define D_LATENT 512
#define D_ROPE 64
#define D_ENTRY 576
#define PAGE_ROWS 64
#define FP8_RECORD_BYTES 656 /* 512 e4m3 codes, 4 fp32 scales, 64 bf16 RoPE values */

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* binary32 -> nearest bfloat16 (ties to even), returned as a double; NaN stays NaN. */
static double f32_to_bf16_double(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0) return NAN;
    u = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* e4m3 "fn": 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; no infinities;
 * exponent 1111 with mantissa 111 is NaN; exponent 0000 is subnormal. */
double mla_oracle_e4m3_to_double(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, 1 - 7);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* One dequantized latent value of an FP8 record: code times its block scale, exact in
 * double (the definition). */
double mla_oracle_fp8_latent_exact(uint8_t code, float scale) {
    return mla_oracle_e4m3_to_double(code) * (double)scale;
}

/* The same value formed in binary32 and rounded once to bfloat16 (the bf16-operand mode
 * described in the header). */
double mla_oracle_fp8_latent(uint8_t code, float scale) {
    return f32_to_bf16_double((float)mla_oracle_e4m3_to_double(code) * scale);
}

static double f32_bits_to_double(const uint8_t *p) {
    float f;
    memcpy(&f, p, sizeof f);
    return (double)f;
}

/* The definition above, for one request and all its heads, over N gathered tokens.
 * qn[H*512], qr[H*64], C[N*512], Kr[N*64] -> out[H*512], lse[H]. */
void mla_oracle_attend_f64(int H, int64_t N, const double *qn, const double *qr,
                           const double *C, const double *Kr, double scale, double *out,
                           double *lse) {
    double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    for (int h = 0; h < H; ++h) {
        double *o = out + (size_t)h * D_LATENT;
        for (int c = 0; c < D_LATENT; ++c) o[c] = 0.0;
        if (N == 0) {
            lse[h] = -INFINITY;
            continue;
        }
        /* pass 1: scores and their maximum */
        double m = -INFINITY;
        for (int64_t t = 0; t < N; ++t) {
            double dot = 0.0;
            for (int c = 0; c < D_LATENT; ++c)
                dot += qn[(size_t)h * D_LATENT + c] * C[(size_t)t * D_LATENT + c];
            for (int r = 0; r < D_ROPE; ++r)
                dot += qr[(size_t)h * D_ROPE + r] * Kr[(size_t)t * D_ROPE + r];
            s[t] = scale * dot;
            if (s[t] > m) m = s[t];
        }
        /* pass 2: normaliser and weighted sum of latents */
        double l = 0.0;
        for (int64_t t = 0; t < N; ++t) {
            double w = exp(s[t] - m);
            l += w;
            for (int c = 0; c < D_LATENT; ++c) o[c] += w * C[(size_t)t * D_LATENT + c];
        }
        for (int c = 0; c < D_LATENT; ++c) o[c] /= l;
        lse[h] = m + log(l);
    }
    free(s);
}

/* Merge of per-chunk results of one head: lse = ln sum_i exp(lse_i),
 * out = sum_i exp(lse_i - lse) out_i.  Chunks with lse_i = -inf hold no tokens. */
void mla_oracle_combine_f64(int S, int D, const double *outs, const double *lses,
                            double *out, double *lse) {
    double m = -INFINITY;
    for (int i = 0; i < S; ++i)
        if (lses[i] > m) m = lses[i];
    for (int c = 0; c < D; ++c) out[c] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double z = 0.0;
    for (int i = 0; i < S; ++i) z += exp(lses[i] - m);
    double L = m + log(z);
    for (int i = 0; i < S; ++i) {
        double w = exp(lses[i] - L);
        for (int c = 0; c < D; ++c) out[c] += w * outs[(size_t)i * D + c];
    }
    *lse = L;
}

/* ---------------------------------------------------------------------------------
 * Paged front ends.  They gather each request's token rows into double arrays and call
 * mla_oracle_attend_f64 on slices of its heads.  Work is spread with plain pthreads in
 * rounds: a round gathers up to `nthreads` requests (one thread per request), then every
 * thread takes (request, head slice) tasks of that round, so that a batch of a few long
 * requests still uses every core.  Parallelism only: each head's arithmetic is the
 * definition above, unchanged.
 * -------------------------------------------------------------------------------*/

enum { CACHE_BF16 = 0, CACHE_FP8 = 1, CACHE_FP8_EXACT = 2 };

typedef struct {
    int64_t N;          /* attended tokens */
    double *qn, *qr;    /* [H*512], [H*64] */
    double *C, *Kr;     /* [N*512], [N*64] */
    int rc;
} gathered_t;

typedef struct {
    int kind; /* CACHE_BF16, CACHE_FP8 (bf16-operand latent) or CACHE_FP8_EXACT */
    int B, H;
    const uint16_t *q_nope, *q_rope;
    const void *cache;
    int64_t num_pages;
    const int32_t *block_table;
    int max_pages;
    const int32_t *seq_lens;
    const int32_t *indices; /* NULL: dense (tokens 0..L-1) */
    int topk;
    double scale;
    double *out, *lse;
    /* the current round: requests b0 .. b0 + nb - 1, heads cut into `slices` slices */
    int b0, nb, slices;
    gathered_t *g;
    int next; /* shared task counter of the current phase */
    pthread_mutex_t mu;
    int error;
} job_t;

/* Decodes logical token t of request b into c[512], kr[64].  Returns 0 or -1. */
static int load_token(const job_t *J, int b, int64_t t, double *c, double *kr) {
    if (t < 0 || t >= J->seq_lens[b]) return -1;
    int64_t lp = t / PAGE_ROWS;
    if (lp >= J->max_pages) return -1;
    int64_t page = J->block_table[(size_t)b * J->max_pages + lp];
    if (page < 0 || page >= J->num_pages) return -1;
    int64_t row = page * PAGE_ROWS + t % PAGE_ROWS;
    if (J->kind == CACHE_BF16) {
        const uint16_t *e = (const uint16_t *)J->cache + (size_t)row * D_ENTRY;
        for (int i = 0; i < D_LATENT; ++i) c[i] = bf16_bits_to_double(e[i]);
        for (int i = 0; i < D_ROPE; ++i) kr[i] = bf16_bits_to_double(e[D_LATENT + i]);
    } else {
        const uint8_t *e = (const uint8_t *)J->cache + (size_t)row * FP8_RECORD_BYTES;
        float sc[4];
        for (int g = 0; g < 4; ++g) sc[g] = (float)f32_bits_to_double(e + 512 + 4 * g);
        for (int i = 0; i < D_LATENT; ++i)
            c[i] = J->kind == CACHE_FP8_EXACT ? mla_oracle_fp8_latent_exact(e[i], sc[i / 128])
                                              : mla_oracle_fp8_latent(e[i], sc[i / 128]);
        const uint8_t *rp = e + 528;
        for (int i = 0; i < D_ROPE; ++i) {
            uint16_t bits = (uint16_t)(rp[2 * i] | (rp[2 * i + 1] << 8));
            kr[i] = bf16_bits_to_double(bits);
        }
    }
    return 0;
}

/* Gathers request b's queries and attended token rows into *G. */
static void gather_request(const job_t *J, int b, gathered_t *G) {
    int H = J->H;
    int64_t N = 0;
    if (J->indices) {
        for (int j = 0; j < J->topk; ++j)
            if (J->indices[(size_t)b * J->topk + j] >= 0) ++N;
    } else {
        N = J->seq_lens[b];
    }
    G->N = N;
    G->qn = (double *)malloc(sizeof(double) * (size_t)H * D_LATENT);
    G->qr = (double *)malloc(sizeof(double) * (size_t)H * D_ROPE);
    G->C = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1) * D_LATENT);
    G->Kr = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1) * D_ROPE);
    int rc = 0;
    for (int i = 0; i < H * D_LATENT; ++i)
        G->qn[i] = bf16_bits_to_double(J->q_nope[(size_t)b * H * D_LATENT + i]);
    for (int i = 0; i < H * D_ROPE; ++i)
        G->qr[i] = bf16_bits_to_double(J->q_rope[(size_t)b * H * D_ROPE + i]);
    int64_t n = 0;
    if (J->indices) {
        for (int j = 0; j < J->topk && rc == 0; ++j) {
            int32_t t = J->indices[(size_t)b * J->topk + j];
            if (t == -1) continue;
            if (t < -1) { rc = -1; break; }
            rc = load_token(J, b, t, G->C + (size_t)n * D_LATENT, G->Kr + (size_t)n * D_ROPE);
            ++n;
        }
    } else {
        for (int64_t t = 0; t < N && rc == 0; ++t, ++n)
            rc = load_token(J, b, t, G->C + (size_t)t * D_LATENT, G->Kr + (size_t)t * D_ROPE);
    }
    G->rc = rc;
}

static void free_gathered(gathered_t *G) {
    free(G->qn); free(G->qr); free(G->C); free(G->Kr);
}

static int take_task(job_t *J) {
    pthread_mutex_lock(&J->mu);
    int k = J->next++;
    pthread_mutex_unlock(&J->mu);
    return k;
}

static void *gather_worker(void *arg) {
    job_t *J = (job_t *)arg;
    for (int k; (k = take_task(J)) < J->nb;) gather_request(J, J->b0 + k, &J->g[k]);
    return NULL;
}

/* Task k of the round: request b0 + k / slices, heads of slice k % slices. */
static void *attend_worker(void *arg) {
    job_t *J = (job_t *)arg;
    const int H = J->H;
    const int per = (H + J->slices - 1) / J->slices;
    for (int k; (k = take_task(J)) < J->nb * J->slices;) {
        const int r = k / J->slices, h0 = (k % J->slices) * per;
        const int h1 = h0 + per < H ? h0 + per : H;
        const gathered_t *G = &J->g[r];
        if (G->rc != 0 || h0 >= h1) continue;
        const int b = J->b0 + r;
        mla_oracle_attend_f64(h1 - h0, G->N, G->qn + (size_t)h0 * D_LATENT, G->qr + (size_t)h0 * D_ROPE,
                              G->C, G->Kr, J->scale, J->out + ((size_t)b * H + h0) * D_LATENT,
                              J->lse + (size_t)b * H + h0);
    }
    return NULL;
}

static void run_phase(job_t *J, int nthreads, void *(*fn)(void *)) {
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    J->next = 0;
    for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, fn, J);
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
}

static int run_jobs(job_t *J, int nthreads) {
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    pthread_mutex_init(&J->mu, NULL);
    J->error = 0;
    J->g = (gathered_t *)calloc((size_t)nthreads, sizeof(gathered_t));
    for (J->b0 = 0; J->b0 < J->B; J->b0 += nthreads) {
        J->nb = J->B - J->b0 < nthreads ? J->B - J->b0 : nthreads;
        /* enough head slices that every thread has work */
        J->slices = (nthreads + J->nb - 1) / J->nb;
        if (J->slices > J->H) J->slices = J->H;
        run_phase(J, J->nb, gather_worker);
        run_phase(J, nthreads, attend_worker);
        for (int r = 0; r < J->nb; ++r) {
            if (J->g[r].rc != 0) J->error = 1;
            free_gathered(&J->g[r]);
        }
    }
    free(J->g);
    pthread_mutex_destroy(&J->mu);
    return J->error ? -1 : 0;
}

/* Number of worker threads this library would use for nthreads <= 0. */
int mla_oracle_default_threads(void) { return (int)sysconf(_SC_NPROCESSORS_ONLN); }

/* Dense decode over a paged bf16 cache [num_pages][64][576].  Returns 0, or -1 if a
 * page or token reference falls outside the given arrays. */
int mla_oracle_decode_dense(int B, int H, const uint16_t *q_nope, const uint16_t *q_rope,
                            const uint16_t *cache, int64_t num_pages,
                            const int32_t *block_table, int max_pages,
                            const int32_t *seq_lens, double scale, double *out,
                            double *lse, int nthreads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.kind = CACHE_BF16; J.B = B; J.H = H; J.q_nope = q_nope; J.q_rope = q_rope;
    J.cache = cache; J.num_pages = num_pages; J.block_table = block_table;
    J.max_pages = max_pages; J.seq_lens = seq_lens; J.scale = scale; J.out = out; J.lse = lse;
    return run_jobs(&J, nthreads);
}

/* Dense decode over a paged FP8 cache: page = 64 records of 656 bytes
 * (512 e4m3 latent codes | 4 little-endian fp32 scales | 64 bf16 RoPE values).
 * exact != 0: latent = code * scale exactly (the definition); exact == 0: the bf16-operand
 * rounding of the header. */
int mla_oracle_decode_fp8(int B, int H, const uint16_t *q_nope, const uint16_t *q_rope,
                          const uint8_t *cache, int64_t num_pages,
                          const int32_t *block_table, int max_pages,
                          const int32_t *seq_lens, int exact, double scale, double *out,
                          double *lse, int nthreads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.kind = exact ? CACHE_FP8_EXACT : CACHE_FP8; J.B = B; J.H = H; J.q_nope = q_nope; J.q_rope = q_rope;
    J.cache = cache; J.num_pages = num_pages; J.block_table = block_table;
    J.max_pages = max_pages; J.seq_lens = seq_lens; J.scale = scale; J.out = out; J.lse = lse;
    return run_jobs(&J, nthreads);
}

/* Token-sparse decode: request b attends over the logical positions
 * indices[b][0..topk) that are >= 0 (each occurrence counts once); -1 is padding.
 * An index outside [-1, seq_lens[b]) makes the call return -1. */
int mla_oracle_decode_sparse(int B, int H, const uint16_t *q_nope, const uint16_t *q_rope,
                             const uint16_t *cache, int64_t num_pages,
                             const int32_t *block_table, int max_pages,
                             const int32_t *seq_lens, const int32_t *indices, int topk,
                             double scale, double *out, double *lse, int nthreads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.kind = CACHE_BF16; J.B = B; J.H = H; J.q_nope = q_nope; J.q_rope = q_rope;
    J.cache = cache; J.num_pages = num_pages; J.block_table = block_table;
    J.max_pages = max_pages; J.seq_lens = seq_lens; J.indices = indices; J.topk = topk;
    J.scale = scale; J.out = out; J.lse = lse;
    return run_jobs(&J, nthreads);
}

/* ------------------------------------------------------------------------------------
 * Cache append: the step after a decode step ("MLA & DSA 推理性能优化指南", §4, the decode
 * figure: each step's output token is appended to the cache).  Request b's new token
 * (latent c[512] and RoPE key k_R[64], bf16 bits) goes to logical position positions[b]:
 * page block_table[b][positions[b] / 64], row positions[b] % 64.  A bf16 cache stores the
 * 576 values.  An FP8 record (same guide, §5.3; the format is this library's reading) is
 * written per block of 128 latent channels: scale = max|x| / 448 in binary32 (1 for an
 * all-zero block), each code the e4m3 "fn" value nearest to x / scale (binary32 division,
 * clamped to [-448, 448] first), ties to the even code; then the four scales and the 64
 * RoPE values as they are.
 * ------------------------------------------------------------------------------------ */

/* The e4m3 "fn" code nearest to v (|v| <= 448), by exhaustive search over the 127 finite
 * non-negative codes; of two equally near codes the one with the even mantissa wins; the
 * sign bit follows v (so -0 gives 0x80). */
uint8_t mla_oracle_e4m3_encode(float v) {
    const double a = fabs((double)v);
    int best = 0;
    double bestd = a;
    for (int c = 1; c <= 0x7E; ++c) {
        const double d = fabs(mla_oracle_e4m3_to_double((uint8_t)c) - a);
        if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)(best | (signbit(v) ? 0x80 : 0));
}

/* Appends one token per request.  Returns the number of requests whose position or page
 * id is out of range (nothing is written for them); positions[b] < 0 skips request b. */
int mla_oracle_append(uint8_t *cache, int fp8, int64_t num_pages, const int32_t *block_table,
                      int max_pages, const int32_t *positions, const uint16_t *c_kv,
                      const uint16_t *k_rope, int B) {
    int errors = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t pos = positions[b];
        if (pos < 0) continue;
        const int32_t lp = pos / PAGE_ROWS;
        if (lp >= max_pages) {
            ++errors;
            continue;
        }
        const int32_t page = block_table[(int64_t)b * max_pages + lp];
        if (page < 0 || page >= num_pages) {
            ++errors;
            continue;
        }
        const int64_t row = (int64_t)page * PAGE_ROWS + pos % PAGE_ROWS;
        const uint16_t *c = c_kv + (int64_t)b * D_LATENT;
        const uint16_t *kr = k_rope + (int64_t)b * D_ROPE;
        if (!fp8) {
            uint8_t *dst = cache + row * D_ENTRY * 2;
            memcpy(dst, c, D_LATENT * 2);
            memcpy(dst + D_LATENT * 2, kr, D_ROPE * 2);
            continue;
        }
        uint8_t *dst = cache + row * FP8_RECORD_BYTES;
        for (int blk = 0; blk < 4; ++blk) {
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                const float x = (float)bf16_bits_to_double(c[blk * 128 + i]);
                if (fabsf(x) > amax) amax = fabsf(x);
            }
            const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
            for (int i = 0; i < 128; ++i) {
                float q = (float)bf16_bits_to_double(c[blk * 128 + i]) / s;
                if (q > 448.0f) q = 448.0f;
                if (q < -448.0f) q = -448.0f;
                dst[blk * 128 + i] = mla_oracle_e4m3_encode(q);
            }
            memcpy(dst + D_LATENT + 4 * blk, &s, 4);
        }
        memcpy(dst + D_LATENT + 16, kr, D_ROPE * 2);
    }
    return errors;
}

/* ------------------------------------------------------------------------------------
 * Absorption and output projection around the decode.
 *
 * "MLA 在极长上下文下的显存带宽突围", section "运行期矩阵吸收": the decode query of head h
 * is q~ = q^C W^UK, the per-head nope query (d_h wide) times that head's up-projection
 * (d_h x 512), so that the score is taken against the 512-d latent directly.  "MLA & DSA
 * 推理性能优化指南" §1.1: the absorbed path keeps the output in latent space; the value
 * up-projection W^UV (latent -> d_h per head) is applied to that output afterwards, which
 * equals attending over the decompressed values v_t = W^UV c_t (linearity).
 *
 * Layouts (row-major): q^C [B][H][dh], W^UK and W^UV [H][dh][512] (row j of head h is the
 * 512-d latent direction of output channel j), latent output [B][H][512], y [B][H][dh].
 * Plain double sums in index order.
 * ------------------------------------------------------------------------------------ */

/* q_abs[b][h][c] = sum_k qc[b][h][k] * w_uk[h][k][c] */
void mla_oracle_absorb(int B, int H, int dh, const double *qc, const double *w_uk, double *q_abs) {
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            const double *q = qc + ((int64_t)b * H + h) * dh;
            double *o = q_abs + ((int64_t)b * H + h) * D_LATENT;
            for (int c = 0; c < D_LATENT; ++c) {
                double s = 0.0;
                for (int k = 0; k < dh; ++k) s += q[k] * w_uk[((int64_t)h * dh + k) * D_LATENT + c];
                o[c] = s;
            }
        }
}

/* y[b][h][j] = sum_c w_uv[h][j][c] * out[b][h][c] */
void mla_oracle_project(int B, int H, int dh, const double *out, const double *w_uv, double *y) {
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            const double *o = out + ((int64_t)b * H + h) * D_LATENT;
            for (int j = 0; j < dh; ++j) {
                const double *w = w_uv + ((int64_t)h * dh + j) * D_LATENT;
                double s = 0.0;
                for (int c = 0; c < D_LATENT; ++c) s += w[c] * o[c];
                y[((int64_t)b * H + h) * dh + j] = s;
            }
        }
}

/* ------------------------------------------------------------------------------------
 * Non-absorbed (MHA-mode) prefill of one sequence.
 *
 * "MLA & DSA 推理性能优化指南" §3.1 and §1.1 (non-absorbed path): the cached latents are
 * first decompressed into per-head keys and values, K_h[t] = W^UK_h c_t and V_h[t] = W^UV_h
 * c_t (d_h = 128 each), then standard multi-head attention runs with the 192-wide key
 * [K_h[t] | k_R[t]] and query [q^C_h | q^R_h] ("MLA 最佳算子全景调研" §4: prefill is a
 * FlashAttention variant with these head widths).  Causal: query i sees keys t <= i.
 *
 * entries [L][576] (latent | RoPE key, the cache entry layout), q_nope [L][H][dh], q_rope
 * [L][H][64], w_uk and w_uv [H][dh][512]; out [L][H][dh], lse [L][H].  Plain double sums,
 * two-pass softmax per query row.  kv_bf16 != 0 rounds the decompressed keys and values to
 * bf16 (the tensors the attention reads); 0 keeps them exact.
 * ------------------------------------------------------------------------------------ */
void mla_oracle_prefill(int L, int H, int dh, const double *entries, const double *q_nope,
                        const double *q_rope, const double *w_uk, const double *w_uv,
                        double scale, int kv_bf16, double *out, double *lse) {
    double *K = (double *)malloc(sizeof(double) * (size_t)L * dh);
    double *V = (double *)malloc(sizeof(double) * (size_t)L * dh);
    double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    for (int h = 0; h < H; ++h) {
        for (int t = 0; t < L; ++t)
            for (int j = 0; j < dh; ++j) {
                const double *wk = w_uk + ((int64_t)h * dh + j) * D_LATENT;
                const double *wv = w_uv + ((int64_t)h * dh + j) * D_LATENT;
                const double *c = entries + (int64_t)t * D_ENTRY;
                double sk = 0.0, sv = 0.0;
                for (int x = 0; x < D_LATENT; ++x) {
                    sk += wk[x] * c[x];
                    sv += wv[x] * c[x];
                }
                /* kv_bf16: keys and values are materialised as bf16 tensors, as the
                 * attention that consumes them takes bf16 operands (sum rounded to binary32,
                 * then to bf16, nearest even) */
                K[(int64_t)t * dh + j] = kv_bf16 ? f32_to_bf16_double((float)sk) : sk;
                V[(int64_t)t * dh + j] = kv_bf16 ? f32_to_bf16_double((float)sv) : sv;
            }
        for (int i = 0; i < L; ++i) {
            const double *qn = q_nope + ((int64_t)i * H + h) * dh;
            const double *qr = q_rope + ((int64_t)i * H + h) * D_ROPE;
            double m = -INFINITY;
            for (int t = 0; t <= i; ++t) {
                double dot = 0.0;
                for (int j = 0; j < dh; ++j) dot += qn[j] * K[(int64_t)t * dh + j];
                for (int r = 0; r < D_ROPE; ++r) dot += qr[r] * entries[(int64_t)t * D_ENTRY + D_LATENT + r];
                s[t] = scale * dot;
                if (s[t] > m) m = s[t];
            }
            double l = 0.0;
            for (int t = 0; t <= i; ++t) l += exp(s[t] - m);
            double *o = out + ((int64_t)i * H + h) * dh;
            for (int j = 0; j < dh; ++j) o[j] = 0.0;
            for (int t = 0; t <= i; ++t) {
                const double w = exp(s[t] - m) / l;
                for (int j = 0; j < dh; ++j) o[j] += w * V[(int64_t)t * dh + j];
            }
            lse[(int64_t)i * H + h] = m + log(l);
        }
    }
    free(K);
    free(V);
    free(s);
}

/*
 * Plain CPU oracle for the MXFP4 speculative-verification hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library; it is written from the pages' definitions, in double
 * precision, with plain loops and no blocking, fusion or reordering.
 *
 * Sources (web pages the method is taken from):
 *   [M11]  "Module 11. Speculative Decoding and Quantization"
 *          (vladkulikov.com, modern-llms module 10 page)
 *          §4  "The exact propose-verify-correct cycle": acceptance
 *              a(x)=min(1,p(x)/q(x)) left to right, stop at the first
 *              rejection, replacement from r = norm((p-q)+), bonus token from
 *              the next position's law when every proposal survives.
 *          §5  "Worked example A" and block B18: strict "draw < acceptance",
 *              acceptance 0 where q = 0, residual normalised by its mass.
 *          §12 "Microscaled FP4, W4A4, and the role of hardware": E2M1 is
 *              1 sign, 2 exponent, 1 fraction bit with magnitudes
 *              0,0.5,1,1.5,2,3,4,6; E8M0 is a power of two with no fraction;
 *              MXFP4 shares one E8M0 across 32 E2M1 values.
 *          §13 teaching quantizer: one scale per group, an all-zero group
 *              gets scale 1, nearest grid value.
 *   [NW]   "Next-Gen Speculative Decoding and FP4 Quantization Shake Up LLM
 *          Inference Economics", section "Microscaling FP4 (MX-FP4)
 *          Integration": packed nibbles laid out [rows, K/2], scales
 *          [rows, K/32], fp32 accumulation.
 *
 * Readings where the pages are silent:
 *   - E8M0 value is 2^(e-127); code 255 is NaN.
 *   - element k of a row is in byte k/2, even k in the low nibble.
 *   - the acceptance test u*q(x) < p(x) is evaluated exactly (the product of
 *     two fp32 numbers is exact in double).
 *   - u[b,0..K-1] are the acceptance draws, u[b,K] drives the one
 *     inverse-CDF draw of the replacement or bonus token.
 *   - inverse CDF: smallest t with r_t > 0 and C_t > u*S (C inclusive
 *     prefix); if rounding leaves none, the last t with r_t > 0.
 *   - a zero residual mass falls back to sampling p_j itself.
 *   - pack: smallest exponent e with amax <= 6*2^e (no clipping), nearest
 *     E2M1 value with ties to the even fraction bit, sign bit kept.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Row flag bits reported by the acceptance oracle. */
#define ORC_ROW_BAD_DRAFT 1      /* a draft id outside [0, V) */
#define ORC_ROW_ZERO_Q 2         /* a proposal with q(x) = 0 was met */
#define ORC_ROW_ZERO_RESIDUAL 4  /* residual mass 0, fell back to p_j */
#define ORC_ROW_NONFINITE 8      /* no usable law (mass 0 or not finite) */

/* ------------------------------------------------------------------ */
/* Element formats ([M11] §12)                                          */
/* ------------------------------------------------------------------ */

/* Value of a 4-bit E2M1 code: sign bit 3, exponent bits 2..1 (bias 1),
 * fraction bit 0.  Exponent field 0 is the subnormal range (0 or 0.5). */
double mxs_oracle_e2m1_value(int code) {
    int sign = (code >> 3) & 1;
    int expo = (code >> 1) & 3;
    int frac = code & 1;
    double mag;
    if (expo == 0)
        mag = 0.5 * frac;
    else
        mag = ldexp(1.0 + 0.5 * frac, expo - 1);
    return sign ? -mag : mag;
}

/* Value of an E8M0 scale byte: a bare power of two, 2^(e-127). */
double mxs_oracle_e8m0_value(int e) {
    if (e == 255) return NAN;
    return ldexp(1.0, e - 127);
}

/* bf16 bit pattern -> double (bf16 is the top half of an fp32). */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Nibble of element k in a packed row: byte k/2, even k in bits 0..3. */
static int nibble_of(const uint8_t* row, int64_t k) {
    uint8_t byte = row[k / 2];
    return (k % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
}

/* Dequantise W [N, K]: w[n,k] = e2m1(nibble) * 2^(scale[n,k/32]-127). */
int mxs_oracle_dequant(const uint8_t* nibbles, const uint8_t* scales,
                       int64_t N, int64_t K, double* w) {
    if (N < 0 || K < 0 || K % 32 != 0) return 1;
    for (int64_t n = 0; n < N; ++n) {
        const uint8_t* row = nibbles + n * (K / 2);
        const uint8_t* srow = scales + n * (K / 32);
        for (int64_t k = 0; k < K; ++k)
            w[n * K + k] = mxs_oracle_e2m1_value(nibble_of(row, k)) *
                           mxs_oracle_e8m0_value(srow[k / 32]);
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Verification GEMM: Y[m,n] = sum_k x[m,k] * w[n,k]                    */
/* ------------------------------------------------------------------ */

typedef struct {
    const double* x;      /* [M, K] already decoded from bf16 */
    const uint8_t* nib;   /* [N, K/2] */
    const uint8_t* sc;    /* [N, K/32] */
    int64_t M, N, K;
    int64_t n_begin, n_end;
    double* y;            /* [M, N] */
} gemm_job;

static void* gemm_worker(void* arg) {
    gemm_job* j = (gemm_job*)arg;
    double* wrow = (double*)malloc(sizeof(double) * (size_t)(j->K > 0 ? j->K : 1));
    if (!wrow) return (void*)1;
    for (int64_t n = j->n_begin; n < j->n_end; ++n) {
        const uint8_t* row = j->nib + n * (j->K / 2);
        const uint8_t* srow = j->sc + n * (j->K / 32);
        for (int64_t k = 0; k < j->K; ++k)
            wrow[k] = mxs_oracle_e2m1_value(nibble_of(row, k)) *
                      mxs_oracle_e8m0_value(srow[k / 32]);
        for (int64_t m = 0; m < j->M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < j->K; ++k)  /* ascending k */
                acc += j->x[m * j->K + k] * wrow[k];
            j->y[m * j->N + n] = acc;
        }
    }
    free(wrow);
    return NULL;
}

/* x_bf16: [M, K] bf16 bit patterns; y: [M, N] doubles.  Rows n are split
 * over nthreads worker threads; each output is one ascending double sum. */
int mxs_oracle_gemm(const uint16_t* x_bf16, const uint8_t* nibbles,
                    const uint8_t* scales, int64_t M, int64_t N, int64_t K,
                    double* y, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || K % 32 != 0) return 1;
    if (M == 0 || N == 0) return 0;
    double* x = (double*)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    if (!x) return 2;
    for (int64_t i = 0; i < M * K; ++i) x[i] = bf16_to_double(x_bf16[i]);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > N) nthreads = (int)N;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    gemm_job* jobs = (gemm_job*)malloc(sizeof(gemm_job) * (size_t)nthreads);
    int rc = 0;
    if (!th || !jobs) rc = 2;
    for (int t = 0; rc == 0 && t < nthreads; ++t) {
        jobs[t].x = x; jobs[t].nib = nibbles; jobs[t].sc = scales;
        jobs[t].M = M; jobs[t].N = N; jobs[t].K = K; jobs[t].y = y;
        jobs[t].n_begin = N * t / nthreads;
        jobs[t].n_end = N * (t + 1) / nthreads;
    }
    int started = 0;
    for (int t = 0; rc == 0 && t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, gemm_worker, &jobs[t]) != 0) { rc = 3; break; }
        ++started;
    }
    for (int t = 0; t < started; ++t) {
        void* ret = NULL;
        pthread_join(th[t], &ret);
        if (ret) rc = 2;
    }
    free(jobs); free(th); free(x);
    return rc;
}

/* ------------------------------------------------------------------ */
/* Pack: real weights -> E2M1 nibbles + E8M0 scales                     */
/* ------------------------------------------------------------------ */

/* Nearest E2M1 magnitude code (0..7) to a (|a| <= 6), ties going to the
 * candidate whose fraction bit is 0. */
static int nearest_e2m1_magnitude(double a) {
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c < 8; ++c) {
        double d = fabs(a - mxs_oracle_e2m1_value(c));
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return best;
}

/* w: [N, K] doubles (exact images of fp32 or bf16 inputs).  Returns 0, or
 * 4 when a block held a non-finite value (that block gets scale byte 255
 * and zero nibbles). */
int mxs_oracle_pack(const double* w, int64_t N, int64_t K,
                    uint8_t* nibbles, uint8_t* scales) {
    if (N < 0 || K < 0 || K % 32 != 0) return 1;
    int rc = 0;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < K / 32; ++b) {
            const double* blk = w + n * K + b * 32;
            uint8_t* out = nibbles + n * (K / 2) + b * 16;
            double amax = 0.0;
            int finite = 1;
            for (int i = 0; i < 32; ++i) {
                if (!isfinite(blk[i])) finite = 0;
                else if (fabs(blk[i]) > amax) amax = fabs(blk[i]);
            }
            if (!finite) {
                scales[n * (K / 32) + b] = 255;
                memset(out, 0, 16);
                rc = 4;
                continue;
            }
            int e;
            if (amax == 0.0) {
                e = 0;  /* all-zero block: scale 1 */
            } else {
                /* smallest integer e with amax <= 6 * 2^e */
                int ex;
                frexp(amax, &ex);
                e = ex - 5;
                while (amax > ldexp(6.0, e)) ++e;
                if (e < -127) e = -127;
                if (e > 127) e = 127;
            }
            scales[n * (K / 32) + b] = (uint8_t)(e + 127);
            for (int i = 0; i < 32; i += 2) {
                int codes[2];
                for (int h = 0; h < 2; ++h) {
                    double v = ldexp(blk[i + h], -e);
                    int mag = nearest_e2m1_magnitude(fabs(v));
                    codes[h] = mag | (signbit(blk[i + h]) ? 8 : 0);
                }
                out[i / 2] = (uint8_t)(codes[0] | (codes[1] << 4));
            }
        }
    }
    return rc;
}

/* ------------------------------------------------------------------ */
/* Acceptance, residual / bonus sampling, emission ([M11] §4, §5)       */
/* ------------------------------------------------------------------ */

/* Inputs are reached through an element accessor so that the same row
 * routine serves fp32 inputs (the kernel's boundary type) and fp64 inputs
 * (used to pin the oracle on the pages' double-precision examples). */
typedef struct {
    const void* base;
    int is_f64;
} law_ref;

static double law_at(law_ref r, int64_t idx) {
    if (r.is_f64) return ((const double*)r.base)[idx];
    return (double)((const float*)r.base)[idx];
}

typedef struct {
    law_ref p, q, u;       /* p [B,K+1,V], q [B,K,V], u [B,K+1] */
    const int32_t* draft;  /* [B,K] */
    int64_t B, K, V;
    int32_t* tokens;       /* [B,K+1], -1 padded */
    int32_t* n_emitted;    /* [B] */
    int32_t* row_flags;    /* [B] */
    double* edge_dist;     /* [B] or NULL */
    int64_t b_begin, b_end;
} accept_job;

static void accept_row(const accept_job* J, int64_t b) {
    const int64_t K = J->K, V = J->V;
    int32_t* tok = J->tokens + b * (K + 1);
    int32_t flags = 0;
    for (int64_t i = 0; i <= K; ++i) tok[i] = -1;
    if (J->edge_dist) J->edge_dist[b] = INFINITY;

    /* every draft id must index the vocabulary */
    for (int64_t i = 0; i < K; ++i) {
        int32_t x = J->draft[b * K + i];
        if (x < 0 || x >= V) flags |= ORC_ROW_BAD_DRAFT;
    }
    if (flags & ORC_ROW_BAD_DRAFT) {
        J->n_emitted[b] = 0;
        J->row_flags[b] = flags;
        return;
    }

    /* left-to-right acceptance: keep x_i while u_i * q_i(x_i) < p_i(x_i);
     * q_i(x_i) = 0 gives acceptance 0, i.e. a rejection. */
    int64_t j = K;
    for (int64_t i = 0; i < K; ++i) {
        int32_t x = J->draft[b * K + i];
        double qx = law_at(J->q, (b * K + i) * V + x);
        double px = law_at(J->p, (b * (K + 1) + i) * V + x);
        double ui = law_at(J->u, b * (K + 1) + i);
        int accept;
        if (qx > 0.0) {
            accept = (ui * qx < px);
        } else {
            flags |= ORC_ROW_ZERO_Q;
            accept = 0;
        }
        if (!accept) { j = i; break; }
    }
    for (int64_t i = 0; i < j; ++i) tok[i] = J->draft[b * K + i];

    /* the law to sample: residual (p_j - q_j)+ after a rejection, p_K when
     * every proposal was accepted (bonus token) */
    const int64_t prow = (b * (K + 1) + j) * V;
    const int64_t qrow = (b * K + j) * V;
    int use_residual = (j < K);
    double* r = (double*)malloc(sizeof(double) * (size_t)V);
    if (!r) { J->n_emitted[b] = 0; J->row_flags[b] = flags | ORC_ROW_NONFINITE; return; }
    double S = 0.0;
    for (int64_t t = 0; t < V; ++t) {
        double pt = law_at(J->p, prow + t);
        double v;
        if (use_residual) {
            double d = pt - law_at(J->q, qrow + t);
            v = d > 0.0 ? d : 0.0;
        } else {
            v = pt;
        }
        r[t] = v;
        S += v;  /* ascending t */
    }
    if (!(S > 0.0)) {
        /* a positive residual exists whenever rejection is possible; only
         * rounding of the inputs can get here: sample p_j instead */
        flags |= ORC_ROW_ZERO_RESIDUAL;
        S = 0.0;
        for (int64_t t = 0; t < V; ++t) {
            r[t] = law_at(J->p, prow + t);
            S += r[t];
        }
    }
    if (!(S > 0.0) || !isfinite(S)) {
        free(r);
        for (int64_t i = 0; i <= K; ++i) tok[i] = -1;
        J->n_emitted[b] = 0;
        J->row_flags[b] = flags | ORC_ROW_NONFINITE;
        return;
    }

    /* inverse CDF with the one remaining uniform */
    double thr = law_at(J->u, b * (K + 1) + K) * S;
    double C = 0.0, C_before = 0.0;
    int64_t pick = -1, last_pos = -1;
    double pick_before = 0.0, pick_after = 0.0;
    for (int64_t t = 0; t < V; ++t) {
        C_before = C;
        C += r[t];
        if (r[t] > 0.0) {
            last_pos = t;
            if (pick < 0 && C > thr) {
                pick = t;
                pick_before = C_before;
                pick_after = C;
            }
        }
    }
    if (pick < 0) {
        /* rounding put u*S at or above the final sum */
        pick = last_pos;
        double c2 = 0.0;
        for (int64_t t = 0; t < last_pos; ++t) c2 += r[t];
        pick_before = c2;
        pick_after = c2 + r[last_pos];
    }
    free(r);
    tok[j] = (int32_t)pick;
    J->n_emitted[b] = (int32_t)(j + 1);
    J->row_flags[b] = flags;
    if (J->edge_dist) {
        double uu = law_at(J->u, b * (K + 1) + K);
        double d0 = fabs(uu - pick_before / S);
        double d1 = fabs(uu - pick_after / S);
        J->edge_dist[b] = d0 < d1 ? d0 : d1;
    }
}

static void* accept_worker(void* arg) {
    accept_job* J = (accept_job*)arg;
    for (int64_t b = J->b_begin; b < J->b_end; ++b) accept_row(J, b);
    return NULL;
}

static int run_accept(accept_job proto, int nthreads) {
    if (proto.B < 0 || proto.K < 0 || proto.V < 1) return 1;
    if (proto.B == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > proto.B) nthreads = (int)proto.B;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    accept_job* jobs = (accept_job*)malloc(sizeof(accept_job) * (size_t)nthreads);
    if (!th || !jobs) { free(th); free(jobs); return 2; }
    int rc = 0, started = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = proto;
        jobs[t].b_begin = proto.B * t / nthreads;
        jobs[t].b_end = proto.B * (t + 1) / nthreads;
    }
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, accept_worker, &jobs[t]) != 0) { rc = 3; break; }
        ++started;
    }
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    free(jobs); free(th);
    return rc;
}

/* fp32 laws, the kernel's boundary type. */
int mxs_oracle_spec_accept(const float* p, const float* q, const int32_t* draft,
                           const float* u, int64_t B, int64_t K, int64_t V,
                           int32_t* tokens, int32_t* n_emitted,
                           int32_t* row_flags, double* edge_dist, int nthreads) {
    accept_job J;
    memset(&J, 0, sizeof J);
    J.p.base = p; J.q.base = q; J.u.base = u;
    J.draft = draft; J.B = B; J.K = K; J.V = V;
    J.tokens = tokens; J.n_emitted = n_emitted; J.row_flags = row_flags;
    J.edge_dist = edge_dist;
    return run_accept(J, nthreads);
}

/* fp64 laws: the same row routine, used to pin the oracle on the pages'
 * double-precision examples. */
int mxs_oracle_spec_accept_f64(const double* p, const double* q,
                               const int32_t* draft, const double* u,
                               int64_t B, int64_t K, int64_t V,
                               int32_t* tokens, int32_t* n_emitted,
                               int32_t* row_flags, double* edge_dist,
                               int nthreads) {
    accept_job J;
    memset(&J, 0, sizeof J);
    J.p.base = p; J.p.is_f64 = 1;
    J.q.base = q; J.q.is_f64 = 1;
    J.u.base = u; J.u.is_f64 = 1;
    J.draft = draft; J.B = B; J.K = K; J.V = V;
    J.tokens = tokens; J.n_emitted = n_emitted; J.row_flags = row_flags;
    J.edge_dist = edge_dist;
    return run_accept(J, nthreads);
}

/* ------------------------------------------------------------------ */
/* The law tokens are actually sampled from ([M11] §4)                  */
/* ------------------------------------------------------------------ */
/*
 * [M11] §4 "The exact propose-verify-correct cycle": temperature changes the
 * sharpness of the logits, top-k keeps the k most probable tokens, top-p keeps
 * a smallest set of the most probable tokens whose cumulative mass reaches p,
 * and acceptance must use the transformed laws of both the target and the
 * draft.  Readings where the page is silent:
 *   - temperature divides the logits (T > 0);
 *   - top-k keeps every token whose logit is at least the k-th largest (ties
 *     at the boundary are kept); k = 0 or k >= V keeps every token;
 *   - top-p walks the kept tokens from the most probable down and stops at
 *     the first whose cumulative mass reaches p; every token at least as
 *     probable as that one is kept (ties kept); p >= 1 keeps every token;
 *   - the kept masses are renormalised; a logit of -inf (a masked token) has
 *     probability 0; a row with a NaN or +inf logit, or nothing of positive
 *     mass, has no law (every probability 0, kept count 0).
 * cut_margin[r] = distance of p from the cumulative mass at the positions
 * that decide the top-p cut -- the one where it stops and the one before it,
 * if any (infinity when top-p keeps every token): a kernel whose masses
 * differ by less than that makes the same cut.
 */
static const float* g_sort_row;  /* row being sorted (single-threaded use) */

static int by_logit_desc(const void* a, const void* b) {
    const int64_t i = *(const int64_t*)a, j = *(const int64_t*)b;
    const double li = g_sort_row[i], lj = g_sort_row[j];
    if (li > lj) return -1;
    if (li < lj) return 1;
    return (i > j) - (i < j);
}

int mxs_oracle_sampling_law(const float* logits, int64_t R, int64_t V, double temperature,
                            int64_t top_k, double top_p, double* probs, double* cut_margin,
                            int64_t* kept_count) {
    if (R < 0 || V < 1 || !(temperature > 0.0) || top_k < 0 || !(top_p > 0.0)) return 1;
    int64_t* order = (int64_t*)malloc((size_t)V * sizeof(int64_t));
    double* e = (double*)malloc((size_t)V * sizeof(double));
    if (!order || !e) { free(order); free(e); return 2; }
    for (int64_t r = 0; r < R; ++r) {
        const float* l = logits + r * V;
        double* pr = probs + r * V;
        cut_margin[r] = INFINITY;
        kept_count[r] = 0;
        int bad = 0;
        for (int64_t t = 0; t < V; ++t) {
            pr[t] = 0.0;
            if (isnan(l[t]) || (isinf(l[t]) && l[t] > 0)) bad = 1;
        }
        if (bad) continue;
        /* the tokens from the most probable down (equal logits in index order) */
        for (int64_t t = 0; t < V; ++t) order[t] = t;
        g_sort_row = l;
        qsort(order, (size_t)V, sizeof(int64_t), by_logit_desc);
        if (isinf(l[order[0]])) continue;  /* every token masked */
        /* top-k: at least the k-th largest logit */
        double lk = -INFINITY;
        if (top_k > 0 && top_k < V) lk = l[order[top_k - 1]];
        /* temperature, then the softmax over the kept tokens */
        const double zmax = (double)l[order[0]] / temperature;
        double S = 0.0;
        for (int64_t t = 0; t < V; ++t) {
            e[t] = 0.0;
            if ((double)l[t] >= lk && !isinf(l[t])) e[t] = exp((double)l[t] / temperature - zmax);
            S += e[t];
        }
        if (!(S > 0.0)) continue;
        /* top-p: the first position whose cumulative mass reaches p */
        double lp = lk;
        if (top_p < 1.0) {
            double c = 0.0, prev = -1.0;  /* prev < 0: no earlier position to stop at */
            for (int64_t i = 0; i < V; ++i) {
                const int64_t t = order[i];
                if (e[t] == 0.0) continue;
                c += e[t] / S;
                if (c >= top_p) {
                    lp = l[t];
                    cut_margin[r] = fabs(c - top_p);
                    if (prev >= 0.0) cut_margin[r] = fmin(cut_margin[r], fabs(top_p - prev));
                    break;
                }
                prev = c;
            }
        }
        /* renormalise over what is kept */
        double S2 = 0.0;
        for (int64_t t = 0; t < V; ++t) {
            if ((double)l[t] < lp) e[t] = 0.0;
            S2 += e[t];
        }
        for (int64_t t = 0; t < V; ++t) {
            pr[t] = e[t] / S2;
            if (e[t] > 0.0) ++kept_count[r];
        }
    }
    free(order);
    free(e);
    return 0;
}

/* ------------------------------------------------------------------ */
/* NVFP4 ([M11] §12)                                                    */
/* ------------------------------------------------------------------ */
/*
 * [M11] §12: NVFP4 holds E2M1 values in blocks of 16 that share an E4M3
 * scale, with one FP32 scale for the whole tensor (4.5 bits per value
 * counting the local scale).  E4M3: one sign bit, four exponent bits (bias
 * 7), three fraction bits, exponent field 0 subnormal.  Reading where the page
 * is silent: the two codes with every exponent and fraction bit set (0x7F,
 * 0xFF) are NaN and there is no infinity (the usual E4M3 convention); a scale
 * may carry a sign; the layout is nibbles [N, K/2] as for MXFP4 and scales
 * [N, K/16], one byte per 16 consecutive k of a row.
 */
double mxs_oracle_e4m3_value(int code) {
    code &= 0xFF;
    const int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    const double mag = e == 0 ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

int mxs_oracle_nvfp4_dequant(const uint8_t* nibbles, const uint8_t* scales, double global_scale,
                             int64_t N, int64_t K, double* w) {
    if (N < 0 || K < 0 || K % 16) return 1;
    for (int64_t n = 0; n < N; ++n) {
        const uint8_t* row = nibbles + n * (K / 2);
        for (int64_t k = 0; k < K; ++k) {
            const double s = mxs_oracle_e4m3_value(scales[n * (K / 16) + k / 16]);
            w[n * K + k] = mxs_oracle_e2m1_value(nibble_of(row, k)) * s * global_scale;
        }
    }
    return 0;
}

/* Y[m, n] = sum_k x[m, k] * w[n, k] with w the NVFP4 dequantisation, in
 * double, k in order (single-threaded: the shapes tested are small). */
int mxs_oracle_nvfp4_gemm(const uint16_t* x_bf16, const uint8_t* nibbles, const uint8_t* scales,
                          double global_scale, int64_t M, int64_t N, int64_t K, double* y) {
    if (M < 0 || N < 0 || K < 0 || K % 16) return 1;
    for (int64_t n = 0; n < N; ++n) {
        const uint8_t* row = nibbles + n * (K / 2);
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double s = mxs_oracle_e4m3_value(scales[n * (K / 16) + k / 16]);
                const double w = mxs_oracle_e2m1_value(nibble_of(row, k)) * s * global_scale;
                acc += bf16_to_double(x_bf16[m * K + k]) * w;
            }
            y[m * N + n] = acc;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* MX-FP4 KV cache of the verification block                           */
/* ------------------------------------------------------------------ */
/*
 * "Next-Gen Speculative Decoding and FP4 Quantization ...": keys and values
 * are stored as MX-FP4 (the "KV Cache Memory Pool (FP4)" of its pipeline
 * diagram; "Benchmarks and Real-World Impact", item 2).  [M11] §4: after
 * acceptance the unaccepted suffix and its cache entries are discarded and
 * decoding continues from the corrected prefix.
 *
 * Cache of one layer's keys (or values) for B sequences: nibbles
 * [B, L_max, W/2] and E8M0 scales [B, L_max, W/32], one row of W values
 * (all heads of one position) per position, blocks of 32 along the row.
 * lens[b] is the number of committed positions of sequence b.
 *
 * kv_append: the verification pass feeds T = K + 1 positions per sequence
 * (the last committed token and the K drafts); row t of kv [B, T, W] is
 * quantised by mxs_oracle_pack's rule into position lens[b] + t.  A position
 * at or beyond L_max is not written; *n_full counts them.
 */
int mxs_oracle_kv_append(const double* kv, int64_t B, int64_t T, int64_t W, uint8_t* nibbles,
                         uint8_t* scales, int64_t L_max, const int32_t* lens, int64_t* n_full) {
    if (B < 0 || T < 0 || W < 0 || W % 32 || L_max < 0) return 1;
    int64_t full = 0;
    int rc = 0;
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t t = 0; t < T; ++t) {
            const int64_t pos = (int64_t)lens[b] + t;
            if (pos < 0 || pos >= L_max) {
                ++full;
                continue;
            }
            const int r = mxs_oracle_pack(kv + (b * T + t) * W, 1, W, nibbles + (b * L_max + pos) * (W / 2),
                                          scales + (b * L_max + pos) * (W / 32));
            if (r == 4) rc = 4;
            else if (r) return r;
        }
    }
    if (n_full) *n_full = full;
    return rc;
}

/*
 * kv_commit: the verification block of sequence b emitted n_emitted[b]
 * tokens (the accepted drafts and one replacement or bonus token; 0 for a
 * row acceptance refused).  Its cache entries for the last committed token
 * and the accepted drafts stay, n_emitted[b] positions in all; the entries
 * of the rejected drafts are the discarded suffix.  So
 * lens[b] <- min(lens[b] + n_emitted[b], L_max), and the emitted
 * replacement or bonus token is fed, and cached, by the next pass.
 */
int mxs_oracle_kv_commit(int32_t* lens, const int32_t* n_emitted, int64_t B, int64_t L_max) {
    if (B < 0 || L_max < 0) return 1;
    for (int64_t b = 0; b < B; ++b) {
        int64_t n = n_emitted[b] > 0 ? n_emitted[b] : 0;
        int64_t l = (int64_t)lens[b] + n;
        lens[b] = (int32_t)(l < L_max ? l : L_max);
    }
    return 0;
}

/* kv_dequant: out[b, l, :] = the decoded row at position l for l < lens[b],
 * and 0 for the positions past the committed length. */
int mxs_oracle_kv_dequant(const uint8_t* nibbles, const uint8_t* scales, int64_t B, int64_t L_max,
                          int64_t W, const int32_t* lens, double* out) {
    if (B < 0 || L_max < 0 || W < 0 || W % 32) return 1;
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t l = 0; l < L_max; ++l) {
            double* o = out + (b * L_max + l) * W;
            if (l < lens[b]) {
                const int r = mxs_oracle_dequant(nibbles + (b * L_max + l) * (W / 2),
                                                 scales + (b * L_max + l) * (W / 32), 1, W, o);
                if (r) return r;
            } else {
                for (int64_t k = 0; k < W; ++k) o[k] = 0.0;
            }
        }
    }
    return 0;
}

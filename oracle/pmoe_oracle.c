/*
 * pmoe_oracle.c -- plain CPU reference ("oracle") for the paged fused-MoE layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or calls this file;
 * only the test-suite, the smoke check and the CPU-baseline leg of the benchmark load it.  It
 * shares no code, header, table or helper with the CUDA path.
 *
 * What it computes.  Rimuru (paper-daily.com/en, "Expert weights are scattered across pages.
 * How does the kernel read them?") keeps an MoE layer's arithmetic unchanged and only changes
 * where the kernel fetches expert rows from: the address rule addr_e(n,t) relocates rows of
 * W1 / W3 into pool pages or load-buffer slots, and buffered experts are the same bytes copied
 * from host memory.  The result the paged kernel must reach is therefore the ordinary MoE layer
 * over contiguous per-expert arrays, which is what this file writes out, with no pages at all:
 *
 *   route   ids[t] = the k largest logits of token t (ties: lower expert id first),
 *           p = softmax(logits[t,:]) over all E experts, w[t,j] = p[ids[t,j]],
 *           optionally w[t,:] /= sum_j w[t,j]                       (orc_route)
 *   align   stable counting sort of (token, slot) pairs by expert, each expert padded to a
 *           multiple of BM rows, plus the block->expert and pair->row maps  (orc_align)
 *   expert  g = W1 x, u = W3 x, h = silu(g) * u (h rounded to bf16), y = W2 h  (orc_expert_ffn)
 *           W1, W3 are the gate and up projections (one page each), W2 the down projection.
 *   shared  the same FFN with intermediate size S*f, weight 1, on every token
 *   combine out[t] = bf16( sum_j w[t,j] * y_{t,j} + y_shared_t )     (orc_forward)
 *
 * Arithmetic is IEEE fp64 throughout; bf16 inputs convert exactly.  The two bf16 roundings
 * (h before the down projection, and the output) are the readings this build takes where the
 * pages are silent; `round_h = 0` switches the first one off so that the closed-form pins can
 * compare in pure fp64.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -pthread pmoe_oracle.c -lm
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------------ */
/* bf16 <-> fp64                                                                                */
/* ------------------------------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32: widen by appending 16 zero bits. */
double orc_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round an fp64 value to the nearest bf16 (ties to even), in one rounding step.
 * bf16 keeps 8 significant bits and binary32's exponent range; below 2^-126 its spacing is
 * the fixed subnormal quantum 2^-133.  The value is scaled so that one bf16 ulp is 1, rounded
 * with rint() (round-half-even in the default mode), and scaled back; the result is exactly
 * representable in binary32, so the float conversion that follows is exact. */
uint16_t orc_f64_to_bf16(double x)
{
    if (isnan(x)) return (uint16_t)0x7FC0;
    if (isinf(x)) return x > 0 ? (uint16_t)0x7F80 : (uint16_t)0xFF80;
    if (x == 0.0) return signbit(x) ? (uint16_t)0x8000 : (uint16_t)0x0000;
    int e;
    frexp(x, &e);                       /* |x| = m * 2^e, 0.5 <= m < 1 */
    int qexp = e - 8;                   /* one ulp of an 8-bit significand */
    if (qexp < -133) qexp = -133;       /* subnormal range */
    double q = ldexp(1.0, qexp);
    double r = rint(x / q) * q;
    if (fabs(r) >= ldexp(1.0, 128)) return signbit(x) ? (uint16_t)0xFF80 : (uint16_t)0x7F80;
    float f = (float)r;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* Vector forms, for the Python side. */
void orc_bf16_to_f64_vec(const uint16_t* in, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f64(in[i]);
}
void orc_f64_to_bf16_vec(const double* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_bf16(in[i]);
}

/* ------------------------------------------------------------------------------------------ */
/* Routing                                                                                      */
/* ------------------------------------------------------------------------------------------ */

/* Top-k selection on one token's logits by k rounds of "largest remaining value, lowest id on
 * a tie", then softmax over all E logits (max-subtracted), then the optional renormalisation
 * over the k selected weights.  Returns 0, or -1 on bad sizes. */
int orc_route_one(int E, int k, int renormalize, const float* logits, int32_t* ids, double* w)
{
    if (E <= 0 || k <= 0 || k > E) return -1;
    unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
    if (!taken) return -1;
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (taken[e]) continue;
            if (best < 0 || logits[e] > logits[best]) best = e;   /* strict: earlier id keeps a tie */
        }
        taken[best] = 1;
        ids[j] = best;
    }
    free(taken);

    double mx = logits[0];
    for (int e = 1; e < E; ++e) if (logits[e] > mx) mx = logits[e];
    double denom = 0.0;
    for (int e = 0; e < E; ++e) denom += exp((double)logits[e] - mx);
    for (int j = 0; j < k; ++j) w[j] = exp((double)logits[ids[j]] - mx) / denom;

    if (renormalize) {
        double s = 0.0;
        for (int j = 0; j < k; ++j) s += w[j];
        for (int j = 0; j < k; ++j) w[j] /= s;
    }
    return 0;
}

int orc_route(int T, int E, int k, int renormalize, const float* logits, int32_t* ids, double* w)
{
    for (int t = 0; t < T; ++t) {
        int rc = orc_route_one(E, k, renormalize, logits + (int64_t)t * E, ids + (int64_t)t * k,
                               w + (int64_t)t * k);
        if (rc) return rc;
    }
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Sort + pad ("moe_align")                                                                     */
/* ------------------------------------------------------------------------------------------ */

/* The pairs of one layer call, and the expert each one goes to:
 *   routed pair i = t*k + j       (0 <= i < T*k)      -> expert ids[t*k + j]
 *   shared pair i = T*k + s*T + t (0 <= s < S)        -> expert E + s  (shared chunk s)
 * Pad entries of sorted_ids hold the sentinel NP = T*(k+S).
 *
 * Experts are visited in ascending id; within an expert the pairs keep ascending pair index;
 * an expert with c pairs owns ceil(c/BM) blocks of BM rows, one with none owns no block.
 * Outputs: sorted_ids[n_padded], block_expert[n_padded/BM], inv[NP] (row of each pair),
 * *n_padded.  `capacity` is the length of sorted_ids.  Returns 0, -1 on bad sizes, -2 when
 * capacity is too small. */
int orc_align(int T, int k, int E, int S, int BM, const int32_t* ids, int32_t capacity,
              int32_t* sorted_ids, int32_t* block_expert, int32_t* inv, int32_t* n_padded)
{
    if (T < 0 || k <= 0 || E <= 0 || S < 0 || BM <= 0) return -1;
    const int64_t NR = (int64_t)T * k;
    const int64_t NP = (int64_t)T * (k + S);
    for (int64_t i = 0; i < NR; ++i)
        if (ids[i] < 0 || ids[i] >= E) return -1;

    int64_t pos = 0;
    for (int e = 0; e < E + S; ++e) {
        int64_t start = pos;
        for (int64_t i = 0; i < NP; ++i) {
            int owner = (i < NR) ? ids[i] : E + (int)((i - NR) / T);
            if (owner != e) continue;
            if (pos >= capacity) return -2;
            sorted_ids[pos] = (int32_t)i;
            inv[i] = (int32_t)pos;
            ++pos;
        }
        int64_t c = pos - start;
        int64_t padded = ((c + BM - 1) / BM) * BM;
        for (int64_t r = c; r < padded; ++r) {
            if (pos >= capacity) return -2;
            sorted_ids[pos++] = (int32_t)NP;
        }
        for (int64_t b = start / BM; b < pos / BM; ++b) block_expert[b] = e;
    }
    *n_padded = (int32_t)pos;
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* One expert's SwiGLU FFN on one token                                                        */
/* ------------------------------------------------------------------------------------------ */

/* W1, W3: [f][d] row-major (row n = output column n of the gate / up projection).
 * W2: [d][f] row-major (row m = output element m, contiguous over the intermediate index).
 * x: [d].  y: [d] (fp64 out).  silu(z) = z / (1 + exp(-z)). */
void orc_expert_ffn(int d, int f, const uint16_t* W1, const uint16_t* W3, const uint16_t* W2,
                    const uint16_t* x, int round_h, double* y)
{
    double* xd = (double*)malloc(sizeof(double) * (size_t)d);
    double* h = (double*)malloc(sizeof(double) * (size_t)f);
    for (int c = 0; c < d; ++c) xd[c] = orc_bf16_to_f64(x[c]);
    for (int n = 0; n < f; ++n) {
        const uint16_t* w1 = W1 + (int64_t)n * d;
        const uint16_t* w3 = W3 + (int64_t)n * d;
        double g = 0.0, u = 0.0;
        for (int c = 0; c < d; ++c) {
            g += orc_bf16_to_f64(w1[c]) * xd[c];
            u += orc_bf16_to_f64(w3[c]) * xd[c];
        }
        double a = g / (1.0 + exp(-g)) * u;
        h[n] = round_h ? orc_bf16_to_f64(orc_f64_to_bf16(a)) : a;
    }
    for (int m = 0; m < d; ++m) {
        const uint16_t* w2 = W2 + (int64_t)m * f;
        double acc = 0.0;
        for (int n = 0; n < f; ++n) acc += orc_bf16_to_f64(w2[n]) * h[n];
        y[m] = acc;
    }
    free(xd);
    free(h);
}

/* ------------------------------------------------------------------------------------------ */
/* Whole layer, one token at a time                                                            */
/* ------------------------------------------------------------------------------------------ */

typedef struct {
    int32_t d, f, E, k, renormalize, S; /* S = shared chunks; shared intermediate size = S*f */
    const uint16_t* W1;   /* [E][f][d] */
    const uint16_t* W3;   /* [E][f][d] */
    const uint16_t* W2;   /* [E][d][f] */
    const uint16_t* W1s;  /* [S*f][d] or NULL when S == 0 */
    const uint16_t* W3s;  /* [S*f][d] */
    const uint16_t* W2s;  /* [d][S*f] */
} orc_layer;

typedef struct {
    const orc_layer* L;
    const uint16_t* hidden;
    const float* logits;
    int round_h;
    int t0, t1;
    double* out_f64;
    uint16_t* out_bf16;
    int32_t* ids;
    double* w;
    int rc;
} orc_job;

static void orc_token(const orc_layer* L, const uint16_t* x, const float* lg, int round_h,
                      double* acc, double* y, int32_t* ids, double* w, int* rc)
{
    const int d = L->d, f = L->f;
    if (orc_route_one(L->E, L->k, L->renormalize, lg, ids, w)) { *rc = -1; return; }
    for (int m = 0; m < d; ++m) acc[m] = 0.0;
    for (int j = 0; j < L->k; ++j) {
        const int64_t e = ids[j];
        orc_expert_ffn(d, f, L->W1 + e * f * d, L->W3 + e * f * d, L->W2 + e * d * f, x,
                       round_h, y);
        for (int m = 0; m < d; ++m) acc[m] += w[j] * y[m];
    }
    if (L->S > 0) {
        orc_expert_ffn(d, L->S * f, L->W1s, L->W3s, L->W2s, x, round_h, y);
        for (int m = 0; m < d; ++m) acc[m] += y[m];
    }
}

static void* orc_worker(void* arg)
{
    orc_job* J = (orc_job*)arg;
    const orc_layer* L = J->L;
    double* acc = (double*)malloc(sizeof(double) * (size_t)L->d);
    double* y = (double*)malloc(sizeof(double) * (size_t)L->d);
    J->rc = 0;
    for (int t = J->t0; t < J->t1 && J->rc == 0; ++t) {
        orc_token(L, J->hidden + (int64_t)t * L->d, J->logits + (int64_t)t * L->E, J->round_h, acc,
                  y, J->ids + (int64_t)t * L->k, J->w + (int64_t)t * L->k, &J->rc);
        for (int m = 0; m < L->d; ++m) {
            if (J->out_f64) J->out_f64[(int64_t)t * L->d + m] = acc[m];
            if (J->out_bf16) J->out_bf16[(int64_t)t * L->d + m] = orc_f64_to_bf16(acc[m]);
        }
    }
    free(acc);
    free(y);
    return NULL;
}

/* hidden [T][d] bf16, logits [T][E] fp32 -> ids [T][k], w [T][k], out_f64 [T][d] (pre-rounding
 * sum, may be NULL), out_bf16 [T][d] (may be NULL).  Tokens are independent; `nthreads` threads
 * take contiguous token ranges.  Returns 0 or -1. */
int orc_forward(const orc_layer* L, int T, const uint16_t* hidden, const float* logits,
                int round_h, int nthreads, double* out_f64, uint16_t* out_bf16, int32_t* ids,
                double* w)
{
    if (!L || T < 0 || L->k <= 0 || L->k > L->E || L->d <= 0 || L->f <= 0 || L->S < 0) return -1;
    if (T == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > T) nthreads = T;
    orc_job* jobs = (orc_job*)calloc((size_t)nthreads, sizeof(orc_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int i = 0; i < nthreads; ++i) {
        orc_job* J = &jobs[i];
        J->L = L; J->hidden = hidden; J->logits = logits; J->round_h = round_h;
        J->t0 = (int)((int64_t)T * i / nthreads);
        J->t1 = (int)((int64_t)T * (i + 1) / nthreads);
        J->out_f64 = out_f64; J->out_bf16 = out_bf16; J->ids = ids; J->w = w;
    }
    for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, orc_worker, &jobs[i]);
    orc_worker(&jobs[0]);
    int rc = jobs[0].rc;
    for (int i = 1; i < nthreads; ++i) {
        pthread_join(th[i], NULL);
        if (jobs[i].rc) rc = jobs[i].rc;
    }
    free(jobs);
    free(th);
    return rc;
}

/* ------------------------------------------------------------------------------------------ */
/* Whole layer, grouped by expert (the second formulation, for self-consistency)               */
/* ------------------------------------------------------------------------------------------ */

/* Same result as orc_forward reached the other way round: route every token, sort the pairs
 * by expert with orc_align, run each expert over its rows in sorted order, keep every pair's
 * y in its sorted row, then combine each token through the pair->row map.  The shared expert
 * is run chunk by chunk (S experts of width f), which equals the whole S*f-wide FFN because
 * SwiGLU is a sum over independent intermediate units.  Single-threaded; for small inputs. */
int orc_forward_grouped(const orc_layer* L, int T, int BM, const uint16_t* hidden,
                        const float* logits, int round_h, double* out_f64, uint16_t* out_bf16)
{
    const int d = L->d, f = L->f, E = L->E, k = L->k, S = L->S;
    if (T <= 0) return T == 0 ? 0 : -1;
    const int64_t NP = (int64_t)T * (k + S);
    const int64_t cap = NP + (int64_t)(E + S) * BM;
    int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * k);
    double* w = (double*)malloc(sizeof(double) * (size_t)T * k);
    int32_t* sorted = (int32_t*)malloc(sizeof(int32_t) * (size_t)cap);
    int32_t* bexp = (int32_t*)malloc(sizeof(int32_t) * (size_t)(cap / BM + 1));
    int32_t* inv = (int32_t*)malloc(sizeof(int32_t) * (size_t)NP);
    double* ybuf = (double*)malloc(sizeof(double) * (size_t)cap * d);
    uint16_t* w1c = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)f * d);
    uint16_t* w3c = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)f * d);
    uint16_t* w2c = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)f * d);
    int32_t npad = 0;
    int rc = orc_route(T, E, k, L->renormalize, logits, ids, w);
    if (!rc) rc = orc_align(T, k, E, S, BM, ids, (int32_t)cap, sorted, bexp, inv, &npad);
    for (int64_t r = 0; !rc && r < npad; ++r) {
        const int32_t pair = sorted[r];
        if (pair >= NP) continue;                      /* pad row */
        const int e = bexp[r / BM];
        const int64_t t = pair < (int64_t)T * k ? pair / k : (pair - (int64_t)T * k) % T;
        const uint16_t *W1, *W3, *W2;
        if (e < E) {
            W1 = L->W1 + (int64_t)e * f * d;
            W3 = L->W3 + (int64_t)e * f * d;
            W2 = L->W2 + (int64_t)e * d * f;
        } else {
            const int s = e - E;                        /* chunk s: rows / columns [s*f, s*f+f) */
            memcpy(w1c, L->W1s + (int64_t)s * f * d, sizeof(uint16_t) * (size_t)f * d);
            memcpy(w3c, L->W3s + (int64_t)s * f * d, sizeof(uint16_t) * (size_t)f * d);
            for (int m = 0; m < d; ++m)
                memcpy(w2c + (int64_t)m * f, L->W2s + (int64_t)m * S * f + (int64_t)s * f,
                       sizeof(uint16_t) * (size_t)f);
            W1 = w1c; W3 = w3c; W2 = w2c;
        }
        orc_expert_ffn(d, f, W1, W3, W2, hidden + t * d, round_h, ybuf + r * d);
    }
    for (int t = 0; !rc && t < T; ++t) {
        for (int m = 0; m < d; ++m) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) acc += w[(int64_t)t * k + j] * ybuf[(int64_t)inv[(int64_t)t * k + j] * d + m];
            for (int s = 0; s < S; ++s) acc += ybuf[(int64_t)inv[(int64_t)T * k + (int64_t)s * T + t] * d + m];
            if (out_f64) out_f64[(int64_t)t * d + m] = acc;
            if (out_bf16) out_bf16[(int64_t)t * d + m] = orc_f64_to_bf16(acc);
        }
    }
    free(ids); free(w); free(sorted); free(bexp); free(inv); free(ybuf);
    free(w1c); free(w3c); free(w2c);
    return rc;
}

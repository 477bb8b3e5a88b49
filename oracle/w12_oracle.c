/*
 * W12 CPU oracle — TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, scalar restatement of the W12 lossless 12-bit weight format and of the GEMM,
 * argmax and Q-view computations built on it, in fp64 where floating point is involved. It is
 * used by the test-suite, by the smoke check and by the benchmark's CPU baseline only; the
 * product path (the CUDA library) never calls it, and it shares no code with that path.
 *
 * Sources (cited by page title and section):
 *   [SP]    "SpecPilot: Autonomous Algorithm Discovery and Systems Optimization for Speculative
 *           Decoding" (arXiv 2611.02501).
 *   [SP-R]  the jaehun.me review of the same paper.
 *
 *   - format (planes A/E/B, per-channel 16-binade window, escapes, 12 KB 128x64 records with the
 *     8-bit view first): [SP] §4.1 "W12: A Lossless 12-bit Weight Format", Fig. 5a; [SP-R] §4.1.
 *   - load-time bit-for-bit check:  [SP] §4.1; Table A2 caption.
 *   - GEMM over exactly decoded weights: [SP] §4.1, Fig. 5b.
 *   - greedy argmax: [SP] §2.1 "Speculative Decoding".
 *   - Q view (A+E only, dropped mantissa bits at their midpoint): [SP] §4.3 "Zero-copy Q pass",
 *     Fig. 7.
 *   - certified LM head (INT8 copy, per-row Cauchy-Schwarz bound, exact rescoring of the
 *     survivors): [SP] §4.1 "Certified LM head".
 *   - INT6 Q-pass copy (per-row scale, 6-bit codes, its GEMM): [SP] §5.3 "Generality Through
 *     Memory"; App. C.
 *   - glue of the synthetic layer stream (residual add, row normalisation, gate-up product):
 *     no page gives a layer dataflow; these follow the library's written reading of one.
 *
 * Physical details the pages leave open (window tie rule, placeholders, byte and nibble order,
 * per-record escape index) follow the library's written W12 specification; every function states
 * the rule it implements. Parity status: every function here is pinned by a CPU test
 * (round trip over all 65,536 bf16 patterns, brute-force window search, exact rational GEMM,
 * brute-force argmax, hand-derived byte fixtures, the lossless case of the INT6 copy, rounding
 * ties and fp32 integer rounding for the bf16 conversion); none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define W12O_TILE_N 128
#define W12O_TILE_K 64
#define W12O_RECORD_BYTES 12288
#define W12O_VIEW_BYTES 8192

/* ---- bf16 field helpers ------------------------------------------------------------------ */

static int bf_sign(uint16_t u) { return u >> 15; }
static int bf_exp(uint16_t u) { return (u >> 7) & 0xFF; }
static int bf_mhi(uint16_t u) { return (u >> 4) & 0x7; }
static int bf_mlo(uint16_t u) { return u & 0xF; }
static int bf_is_normal(uint16_t u) { int e = bf_exp(u); return e >= 1 && e <= 254; }

/* exact value of a bf16 pattern as a double (a bf16 is the top half of an fp32) */
double w12o_bf16_to_double(uint16_t u) {
    uint32_t bits = (uint32_t)u << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ---- window choice: [SP] §4.1 (per channel n, the 16-binade window [E_n-15, E_n] holding
 *      the largest number of the channel's weights); ties -> smallest E_n ------------------ */

int w12o_window(const uint16_t *row, int K) {
    long hist[256];
    for (int e = 0; e < 256; ++e) hist[e] = 0;
    for (int k = 0; k < K; ++k)
        if (bf_is_normal(row[k])) hist[bf_exp(row[k])] += 1;
    int best_E = 16;
    long best_cover = -1;
    for (int E = 16; E <= 254; ++E) {
        long cover = 0;
        for (int e = E - 15; e <= E; ++e) cover += hist[e];
        if (cover > best_cover) { /* strict: the first (smallest) maximiser wins */
            best_cover = cover;
            best_E = E;
        }
    }
    return best_E;
}

/* Is weight u stored in-window for base E_n? ([SP] §4.1: outside-window weights, zeros and
 * denormals become escapes; Inf/NaN have e = 255 and are outside every window.) */
static int in_window(uint16_t u, int En) {
    int e = bf_exp(u);
    return bf_is_normal(u) && e >= En - 15 && e <= En;
}

/* Planes of one real weight: E offset, m_hi, low nibble, sign. Escapes get the placeholder. */
static void planes_of(uint16_t u, int En, int *E, int *mhi, int *b, int *s) {
    *s = bf_sign(u);
    if (in_window(u, En)) {
        *E = bf_exp(u) - (En - 15);
        *mhi = bf_mhi(u);
        *b = bf_mlo(u);
    } else if (bf_exp(u) == 255 || (bf_is_normal(u) && bf_exp(u) > En)) {
        *E = 15; *mhi = 7; *b = 15;          /* above the window: clamp to its top */
    } else {
        *E = 0; *mhi = 0; *b = 0;            /* zero, subnormal or below: clamp to its bottom */
    }
}

/* ---- record byte placement (the library's specification of the 12 KB record) --------------- */

static size_t view_offset(int nl, int kl) { return (size_t)2048 * (kl >> 4) + 16 * nl + (kl & 15); }
static size_t b_word_offset(int nl, int kl) {
    return W12O_VIEW_BYTES + (size_t)2048 * (kl >> 5) + 16 * nl + 4 * ((kl >> 3) & 3);
}
static int b_nibble_pos(int kl) { int i = kl & 7; return (i >> 1) + 4 * (i & 1); }

static uint32_t load_u32le(const uint8_t *p) {
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}
static void store_u32le(uint8_t *p, uint32_t v) {
    p[0] = v & 0xFF; p[1] = (v >> 8) & 0xFF; p[2] = (v >> 16) & 0xFF; p[3] = (v >> 24) & 0xFF;
}

/* ---- sizes ------------------------------------------------------------------------------- */

/* Counts of the canonical escape list and of the per-record index (words, headers included). */
void w12o_count(const uint16_t *w, int N, int K, int64_t *n_esc, int64_t *n_rec_esc) {
    int n_tiles = (N + W12O_TILE_N - 1) / W12O_TILE_N;
    int k_tiles = (K + W12O_TILE_K - 1) / W12O_TILE_K;
    int *En = (int *)malloc(sizeof(int) * (size_t)(N > 0 ? N : 1));
    for (int n = 0; n < N; ++n) En[n] = w12o_window(w + (size_t)n * K, K);
    int64_t total = 0, total_rec = 0;
    for (int nt = 0; nt < n_tiles; ++nt)
        for (int kt = 0; kt < k_tiles; ++kt) {
            int64_t c = 0;
            for (int nl = 0; nl < W12O_TILE_N; ++nl) {
                int n = nt * W12O_TILE_N + nl;
                if (n >= N) break;
                for (int kl = 0; kl < W12O_TILE_K; ++kl) {
                    int k = kt * W12O_TILE_K + kl;
                    if (k >= K) break;
                    if (!in_window(w[(size_t)n * K + k], En[n])) c += 1;
                }
            }
            total += c;
            total_rec += (c > 0) ? 4 + (c + 3) / 4 * 4 : 0;
        }
    free(En);
    *n_esc = total;
    *n_rec_esc = total_rec;
}

/* ---- encoder: [SP] §4.1 and Fig. 5a ------------------------------------------------------- */

void w12o_encode(const uint16_t *w, int N, int K,
                 uint8_t *records, uint8_t *base_exp,
                 uint32_t *esc_off, uint32_t *esc_k, uint16_t *esc_bits,
                 uint32_t *rec_esc_off, uint32_t *rec_esc) {
    int n_tiles = (N + W12O_TILE_N - 1) / W12O_TILE_N;
    int k_tiles = (K + W12O_TILE_K - 1) / W12O_TILE_K;

    /* step 1: window base per channel */
    for (int n = 0; n < n_tiles * W12O_TILE_N; ++n)
        base_exp[n] = (uint8_t)(n < N ? w12o_window(w + (size_t)n * K, K) : 16);

    /* step 2: canonical per-channel escape list, k ascending */
    uint32_t pos = 0;
    for (int n = 0; n < N; ++n) {
        esc_off[n] = pos;
        for (int k = 0; k < K; ++k) {
            uint16_t u = w[(size_t)n * K + k];
            if (!in_window(u, base_exp[n])) {
                esc_k[pos] = (uint32_t)k;
                esc_bits[pos] = u;
                pos += 1;
            }
        }
    }
    esc_off[N] = pos;

    /* step 3: records (planes) and the per-record escape index: per record with escapes, a
     * header of 4 cumulative quarter counts (rows < 32, < 64, < 96, < 128), its entries in
     * increasing pos, then padding to a multiple of 4 words */
    memset(records, 0, (size_t)n_tiles * k_tiles * W12O_RECORD_BYTES);
    uint32_t rpos = 0;
    for (int nt = 0; nt < n_tiles; ++nt)
        for (int kt = 0; kt < k_tiles; ++kt) {
            size_t r = (size_t)nt * k_tiles + kt;
            uint8_t *rec = records + r * W12O_RECORD_BYTES;
            rec_esc_off[r] = rpos;
            uint32_t quarter_end[4] = {0, 0, 0, 0};
            uint32_t count = 0;
            /* first pass: planes, and the escapes counted per quarter */
            for (int nl = 0; nl < W12O_TILE_N; ++nl)
                for (int kl = 0; kl < W12O_TILE_K; ++kl) {
                    int n = nt * W12O_TILE_N + nl, k = kt * W12O_TILE_K + kl;
                    if (n >= N || k >= K) continue; /* padding: byte 0, nibble 0 */
                    uint16_t u = w[(size_t)n * K + k];
                    int E, mhi, b, s;
                    planes_of(u, base_exp[n], &E, &mhi, &b, &s);
                    rec[view_offset(nl, kl)] = (uint8_t)((E << 4) | (mhi << 1) | s);
                    uint8_t *bw = rec + b_word_offset(nl, kl);
                    uint32_t word = load_u32le(bw);
                    word |= (uint32_t)b << (4 * b_nibble_pos(kl));
                    store_u32le(bw, word);
                    if (!in_window(u, base_exp[n])) {
                        count += 1;
                        for (int q = nl / 32; q < 4; ++q) quarter_end[q] += 1;
                    }
                }
            if (count == 0) continue; /* no escapes: an empty segment */
            for (int q = 0; q < 4; ++q) rec_esc[rpos++] = quarter_end[q];
            /* second pass: the entries, in increasing pos = 64 * n_l + k_l */
            for (int nl = 0; nl < W12O_TILE_N; ++nl)
                for (int kl = 0; kl < W12O_TILE_K; ++kl) {
                    int n = nt * W12O_TILE_N + nl, k = kt * W12O_TILE_K + kl;
                    if (n >= N || k >= K) continue;
                    uint16_t u = w[(size_t)n * K + k];
                    if (!in_window(u, base_exp[n]))
                        rec_esc[rpos++] = (uint32_t)(nl * W12O_TILE_K + kl) | ((uint32_t)u << 16);
                }
            while (rpos % 4 != 0) rec_esc[rpos++] = 0xFFFFFFFFu;
        }
    rec_esc_off[(size_t)n_tiles * k_tiles] = rpos;
}

/* ---- decoder (from records + the per-record index): [SP] §4.1 ----------------------------- */

void w12o_decode(const uint8_t *records, const uint8_t *base_exp,
                 const uint32_t *rec_esc_off, const uint32_t *rec_esc,
                 int N, int K, uint16_t *w_out) {
    int n_tiles = (N + W12O_TILE_N - 1) / W12O_TILE_N;
    int k_tiles = (K + W12O_TILE_K - 1) / W12O_TILE_K;
    for (int nt = 0; nt < n_tiles; ++nt)
        for (int kt = 0; kt < k_tiles; ++kt) {
            size_t r = (size_t)nt * k_tiles + kt;
            const uint8_t *rec = records + r * W12O_RECORD_BYTES;
            for (int nl = 0; nl < W12O_TILE_N; ++nl)
                for (int kl = 0; kl < W12O_TILE_K; ++kl) {
                    int n = nt * W12O_TILE_N + nl, k = kt * W12O_TILE_K + kl;
                    if (n >= N || k >= K) continue;
                    int V = rec[view_offset(nl, kl)];
                    int E = V >> 4, mhi = (V >> 1) & 7, s = V & 1;
                    int b = (load_u32le(rec + b_word_offset(nl, kl)) >> (4 * b_nibble_pos(kl))) & 0xF;
                    int e = E + base_exp[n] - 15;
                    w_out[(size_t)n * K + k] = (uint16_t)((s << 15) | (e << 7) | (mhi << 4) | b);
                }
            /* a non-empty segment starts with its 4-word quarter header */
            uint32_t first = rec_esc_off[r] + (rec_esc_off[r + 1] > rec_esc_off[r] ? 4u : 0u);
            for (uint32_t i = first; i < rec_esc_off[r + 1]; ++i) {
                uint32_t ent = rec_esc[i];
                uint32_t p = ent & 0xFFFF;
                if (p >= (uint32_t)(W12O_TILE_N * W12O_TILE_K)) continue; /* padding entry */
                int n = nt * W12O_TILE_N + (int)(p / W12O_TILE_K);
                int k = kt * W12O_TILE_K + (int)(p % W12O_TILE_K);
                w_out[(size_t)n * K + k] = (uint16_t)(ent >> 16);
            }
        }
}

/* decoder variant that restores escapes from the canonical per-channel list */
void w12o_decode_csr(const uint8_t *records, const uint8_t *base_exp,
                     const uint32_t *esc_off, const uint32_t *esc_k, const uint16_t *esc_bits,
                     int N, int K, uint16_t *w_out) {
    int k_tiles = (K + W12O_TILE_K - 1) / W12O_TILE_K;
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k) {
            int nt = n / W12O_TILE_N, nl = n % W12O_TILE_N, kt = k / W12O_TILE_K, kl = k % W12O_TILE_K;
            const uint8_t *rec = records + ((size_t)nt * k_tiles + kt) * W12O_RECORD_BYTES;
            int V = rec[view_offset(nl, kl)];
            int b = (load_u32le(rec + b_word_offset(nl, kl)) >> (4 * b_nibble_pos(kl))) & 0xF;
            int e = (V >> 4) + base_exp[n] - 15;
            w_out[(size_t)n * K + k] = (uint16_t)(((V & 1) << 15) | (e << 7) | (((V >> 1) & 7) << 4) | b);
        }
    for (int n = 0; n < N; ++n)
        for (uint32_t i = esc_off[n]; i < esc_off[n + 1]; ++i)
            w_out[(size_t)n * K + esc_k[i]] = esc_bits[i];
}

/* ---- Q view, by definition from W: [SP] §4.3 "Zero-copy Q pass" ----------------------------
 * sign, exponent offset and top three mantissa bits of the stored planes, low four mantissa
 * bits set to their midpoint 1000b; escapes keep their placeholder planes. */

void w12o_qview_weights(const uint16_t *w, int N, int K, uint16_t *wq) {
    for (int n = 0; n < N; ++n) {
        int En = w12o_window(w + (size_t)n * K, K);
        for (int k = 0; k < K; ++k) {
            int E, mhi, b, s;
            planes_of(w[(size_t)n * K + k], En, &E, &mhi, &b, &s);
            (void)b;
            wq[(size_t)n * K + k] = (uint16_t)((s << 15) | ((E + En - 15) << 7) | (mhi << 4) | 8);
        }
    }
}

/* ---- GEMM in fp64: y[m,n] = sum_k x[m,k] w[n,k]  ([SP] §4.1, Fig. 5b) ----------------------
 * Also returns sum_k |x[m,k] w[n,k]|, the scale of the stated error bound. */

void w12o_gemm(const uint16_t *x, int M, const uint16_t *w, int N, int K,
               double *y, double *absdot) {
    #pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        double *wd = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        for (int k = 0; k < K; ++k) wd[k] = w12o_bf16_to_double(w[(size_t)n * K + k]);
        for (int m = 0; m < M; ++m) {
            double acc = 0.0, aacc = 0.0;
            for (int k = 0; k < K; ++k) {
                double p = w12o_bf16_to_double(x[(size_t)m * K + k]) * wd[k];
                acc += p;
                aacc += fabs(p);
            }
            y[(size_t)m * N + n] = acc;
            if (absdot) absdot[(size_t)m * N + n] = aacc;
        }
        free(wd);
    }
}

/* the same sum for a list of sampled (m, n) output positions */
void w12o_gemm_sampled(const uint16_t *x, const uint16_t *w, int K,
                       const int32_t *ms, const int32_t *ns, int64_t count,
                       double *y, double *absdot) {
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i) {
        double acc = 0.0, aacc = 0.0;
        for (int k = 0; k < K; ++k) {
            double p = w12o_bf16_to_double(x[(size_t)ms[i] * K + k]) *
                       w12o_bf16_to_double(w[(size_t)ns[i] * K + k]);
            acc += p;
            aacc += fabs(p);
        }
        y[i] = acc;
        absdot[i] = aacc;
    }
}

/* ---- argmax per row: [SP] §2.1 (greedy acceptance takes the target's argmax) --------------
 * top1 = smallest index of the maximum; gap = max - (largest value at any other index);
 * scale = max |y| over the row. */

void w12o_argmax(const double *y, int M, int N, int32_t *idx, double *val, double *gap,
                 double *scale) {
    for (int m = 0; m < M; ++m) {
        const double *row = y + (size_t)m * N;
        int best = 0;
        for (int n = 1; n < N; ++n)
            if (row[n] > row[best]) best = n;
        double second = -INFINITY, sc = 0.0;
        for (int n = 0; n < N; ++n) {
            if (n != best && row[n] > second) second = row[n];
            if (fabs(row[n]) > sc) sc = fabs(row[n]);
        }
        idx[m] = best;
        val[m] = row[best];
        gap[m] = (N > 1) ? row[best] - second : INFINITY;
        scale[m] = sc;
    }
}

/* number of OpenMP threads the parallel loops above use */
#ifdef _OPENMP
#include <omp.h>
int w12o_threads(void) { return omp_get_max_threads(); }
/* threads the parallel loops use from now on (n >= 1): one core or all of them for the timings */
void w12o_set_threads(int n) { omp_set_num_threads(n > 0 ? n : 1); }
#else
int w12o_threads(void) { return 1; }
void w12o_set_threads(int n) { (void)n; }
#endif

/* ---- certified LM head: INT8 codes of the head and a bound per row ---------------------------
 * [SP] §4.1 "Certified LM head": INT8 codes of the head with a Cauchy-Schwarz bound per row;
 * a token whose upper bound lies below another's lower bound cannot win and is dropped, the
 * rest are scored again exactly, and a row keeping too many falls back to the whole head. The
 * pages give no formulas; this is
 * the plainest reading, in the library's written specification:
 *   scale   s_n = fp32(max_k |w[n,k]| / 127)   (0 for an all-zero row)
 *   code    q[n,k] = round-half-even(w[n,k] / s_n), clamped to [-127, 127]
 *   residual c_n = || w[n,:] - s_n q[n,:] ||_2          (+inf if the row holds Inf or NaN)
 *   approx  yh[m,n] = s_n sum_k x[m,k] q[n,k]
 *   bound   |y[m,n] - yh[m,n]| <= ||x[m,:]||_2 c_n       (Cauchy-Schwarz)
 *   L_m     = second largest of yh[m,n] - ||x_m|| c_n over n (the best lower bound's runner-up)
 *   survivors S_m = { n : yh[m,n] + ||x_m|| c_n >= L_m }: they hold the exact top-1 and top-2
 *   result  the exact argmax and top-1/top-2 gap of y over S_m (equal to those over all n).
 */

/* per row: scale, codes (row-major int8), residual norm c_n and code norm ||q_n|| */
void w12o_head_q8(const uint16_t *w, int N, int K, float *scale, int8_t *q, double *resid,
                  double *qnorm) {
    #pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        const uint16_t *row = w + (size_t)n * K;
        int finite = 1;
        double amax = 0.0;
        for (int k = 0; k < K; ++k) {
            if (bf_exp(row[k]) == 255) finite = 0;
            double a = fabs(w12o_bf16_to_double(row[k]));
            if (a > amax) amax = a;
        }
        int8_t *qr = q + (size_t)n * K;
        if (!finite || amax == 0.0) {
            scale[n] = 0.0f;
            for (int k = 0; k < K; ++k) qr[k] = 0;
            resid[n] = finite ? 0.0 : INFINITY;
            qnorm[n] = 0.0;
            continue;
        }
        const float s = (float)(amax / 127.0);
        const double sd = (double)s;
        double e2 = 0.0, q2 = 0.0;
        for (int k = 0; k < K; ++k) {
            double wk = w12o_bf16_to_double(row[k]);
            double t = nearbyint(wk / sd);  /* the default rounding mode: to nearest, ties to even */
            if (t > 127.0) t = 127.0;
            if (t < -127.0) t = -127.0;
            qr[k] = (int8_t)t;
            double e = wk - sd * t;         /* exact: both terms are exact in fp64 */
            e2 += e * e;
            q2 += t * t;
        }
        scale[n] = s;
        resid[n] = sqrt(e2);
        qnorm[n] = sqrt(q2);
    }
}

/* The certified argmax of each row, in fp64 from its definition above. x: bf16 [M,K]; w: bf16
 * [N,K] (the exact head, for rescoring); scale, q, resid: from w12o_head_q8. Returns the
 * survivor count per row; idx/val/gap are the argmax over the survivors (exact y). */
void w12o_certified_argmax(const uint16_t *x, int M, const uint16_t *w, int N, int K,
                           const float *scale, const int8_t *q, const double *resid,
                           int32_t *idx, double *val, double *gap, int64_t *n_surv) {
    double *yh = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    for (int m = 0; m < M; ++m) {
        const uint16_t *xm = x + (size_t)m * K;
        double xn2 = 0.0;
        for (int k = 0; k < K; ++k) {
            double a = w12o_bf16_to_double(xm[k]);
            xn2 += a * a;
        }
        const double xn = sqrt(xn2);
        #pragma omp parallel for schedule(static)
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k) acc += w12o_bf16_to_double(xm[k]) * (double)q[(size_t)n * K + k];
            yh[n] = (double)scale[n] * acc;
        }
        /* the two largest lower bounds */
        double l1 = -INFINITY, l2 = -INFINITY;
        for (int n = 0; n < N; ++n) {
            double lb = yh[n] - xn * resid[n];
            if (lb > l1) { l2 = l1; l1 = lb; }
            else if (lb > l2) l2 = lb;
        }
        int best = -1;
        double bv = -INFINITY, second = -INFINITY;
        int64_t cnt = 0;
        for (int n = 0; n < N; ++n) {
            if (!(yh[n] + xn * resid[n] >= l2)) continue;
            ++cnt;
            double y = 0.0;
            for (int k = 0; k < K; ++k)
                y += w12o_bf16_to_double(xm[k]) * w12o_bf16_to_double(w[(size_t)n * K + k]);
            if (isnan(y)) y = -INFINITY;  /* the GEMM argmax's rule: a NaN logit never wins */
            if (best < 0 || y > bv) {
                if (best >= 0) second = bv > second ? bv : second;
                best = n;
                bv = y;
            } else if (y > second) {
                second = y;
            }
        }
        idx[m] = best;
        val[m] = bv;
        gap[m] = bv - second;
        n_surv[m] = cnt;
    }
    free(yh);
}

/* ---- INT6 Q-pass copy -------------------------------------------------------------------
 * [SP] §5.3 (a later drafter brought an INT6 copy for the Q pass; INT6 and INT8 Q-pass copies
 * are both named) and App. C (the Q pass reads the nested 8-bit view or a separate low-precision copy). The pages
 * give no formulas; the plainest reading, fixed in the library's written specification, is the
 * INT8 copy's per-row symmetric quantisation with 6-bit codes:
 *   scale   s_n = fp32(max_k |w[n,k]| / 31)  (0 for an all-zero row and for a row holding Inf
 *                                             or NaN, whose codes are then all 0)
 *   code    c[n,k] = round-half-even(w[n,k] / s_n), clamped to [-31, 31]
 *   Q pass  yq[m,n] = s_n sum_k x[m,k] c[n,k]
 */
void w12o_copy_q6(const uint16_t *w, int N, int K, float *scale, int8_t *q) {
    #pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        const uint16_t *row = w + (size_t)n * K;
        int finite = 1;
        double amax = 0.0;
        for (int k = 0; k < K; ++k) {
            if (bf_exp(row[k]) == 255) finite = 0;
            double a = fabs(w12o_bf16_to_double(row[k]));
            if (a > amax) amax = a;
        }
        int8_t *qr = q + (size_t)n * K;
        if (!finite || amax == 0.0) {
            scale[n] = 0.0f;
            for (int k = 0; k < K; ++k) qr[k] = 0;
            continue;
        }
        const float s = (float)(amax / 31.0);
        for (int k = 0; k < K; ++k) {
            double t = nearbyint(w12o_bf16_to_double(row[k]) / (double)s);  /* ties to even */
            if (t > 31.0) t = 31.0;
            if (t < -31.0) t = -31.0;
            qr[k] = (int8_t)t;
        }
        scale[n] = s;
    }
}

/* The INT6 copy's records, from row-major codes c [N,K] (the library's specification). One record
 * per 128 x 64 tile, record r = n_tile * k_tiles + k_tile, 6144 bytes, holding u = c + 32
 * (1..63; padding rows and columns hold code 0, u = 32) as two planes of 32-bit little-endian
 * words. For local row n_l, k_l = 16 g + 2 j + h (group g 0..3, pair j 0..7, half h 0..1):
 *   plane L (bytes 0..4095), the low four bits of u:  word 2g + (j >> 2) of the row, where row
 *     words 0..3 sit at byte 16 n_l + 4 i and words 4..7 at 2048 + 16 n_l + 4 (i - 4);
 *     bits 4 (j & 3) + 16 h .. +3
 *   plane T (bytes 4096..6143), the top two bits of u: word g of the row at byte
 *     4096 + 16 n_l + 4 g; bits 2 j + 16 h .. +1 */
void w12o_q6_pack(const int8_t *q, int N, int K, uint8_t *records) {
    const int nt_n = (N + W12O_TILE_N - 1) / W12O_TILE_N, kt_n = (K + W12O_TILE_K - 1) / W12O_TILE_K;
    #pragma omp parallel for schedule(static)
    for (int nt = 0; nt < nt_n; ++nt) {
        for (int kt = 0; kt < kt_n; ++kt) {
            uint8_t *rec = records + ((size_t)nt * kt_n + kt) * 6144;
            uint32_t words[128][12];
            for (int nl = 0; nl < 128; ++nl)
                for (int i = 0; i < 12; ++i) words[nl][i] = 0;
            for (int nl = 0; nl < 128; ++nl) {
                for (int kl = 0; kl < 64; ++kl) {
                    const int n = nt * 128 + nl, k = kt * 64 + kl;
                    const int c = (n < N && k < K) ? q[(size_t)n * K + k] : 0;
                    const uint32_t u = (uint32_t)(c + 32);
                    const int g = kl >> 4, j = (kl & 15) >> 1, h = kl & 1;
                    words[nl][2 * g + (j >> 2)] |= (u & 15u) << (4 * (j & 3) + 16 * h);
                    words[nl][8 + g] |= (u >> 4) << (2 * j + 16 * h);
                }
            }
            for (int nl = 0; nl < 128; ++nl) {
                for (int i = 0; i < 12; ++i) {
                    size_t off;
                    if (i < 4) off = (size_t)16 * nl + 4 * i;
                    else if (i < 8) off = 2048 + (size_t)16 * nl + 4 * (i - 4);
                    else off = 4096 + (size_t)16 * nl + 4 * (i - 8);
                    for (int b = 0; b < 4; ++b) rec[off + b] = (uint8_t)(words[nl][i] >> (8 * b));
                }
            }
        }
    }
}

/* yq [M,N] = s_n sum_k x[m,k] c[n,k] and ad [M,N] = s_n sum_k |x[m,k] c[n,k]| (the scale of
 * the rounding error of any evaluation order), in fp64 (each product is exact). */
void w12o_gemm_q6(const uint16_t *x, int M, const int8_t *q, const float *scale, int N, int K, double *y,
                  double *ad) {
    #pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        for (int m = 0; m < M; ++m) {
            double acc = 0.0, aacc = 0.0;
            for (int k = 0; k < K; ++k) {
                const double p = w12o_bf16_to_double(x[(size_t)m * K + k]) * (double)q[(size_t)n * K + k];
                acc += p;
                aacc += fabs(p);
            }
            y[(size_t)m * N + n] = (double)scale[n] * acc;
            ad[(size_t)m * N + n] = (double)scale[n] * aacc;
        }
    }
}

/* ---- glue of the synthetic layer stream --------------------------------------------------
 * The pages give no layer dataflow; the synthetic 64-layer stream that carries M rows from layer
 * to layer (the reading taken here) needs three steps besides the GEMMs: the residual add (y += x W^T,
 * one fp32 addition per output), the row normalisation and the gate-up product below. */

/* bf16 bits of a double, rounded to nearest even (normal, subnormal, overflow to Inf, NaN). */
uint16_t w12o_double_to_bf16(double v) {
    if (isnan(v)) return 0x7FC0;
    const uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);               /* a = m 2^e, m in [0.5, 1) */
    int q_exp = e - 8;          /* quantum of an 8-significant-bit value in that binade */
    if (q_exp < -133) q_exp = -133;  /* bf16 subnormals: quantum 2^-133 */
    double q = nearbyint(ldexp(a, -q_exp));  /* exact scaling; ties to even */
    double r = ldexp(q, q_exp);
    if (r > 0x1.FEp127) return sign | 0x7F80;  /* rounded beyond the largest finite bf16: Inf */
    /* r is now exactly representable in bf16: take its fp32 bits */
    float f = (float)r;
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | ((bits >> 16) & 0x7FFF));
}

/* x[m,k] = bf16(h[m,k] * (1 / sqrt(mean_k h[m,k]^2))), computed in fp64: the squares of fp32
 * values are exact in fp64 and summed in increasing k, the reciprocal of the root is rounded
 * once, and each product once before the rounding to bf16; an all-zero row gives zeros. */
void w12o_rms_bf16(const float *h, int M, int K, uint16_t *x) {
    for (int m = 0; m < M; ++m) {
        const float *hr = h + (size_t)m * K;
        double ss = 0.0;
        for (int k = 0; k < K; ++k) ss += (double)hr[k] * (double)hr[k];
        const double r = sqrt(ss / (double)K);
        const double inv = (r > 0.0) ? 1.0 / r : 0.0;
        for (int k = 0; k < K; ++k)
            x[(size_t)m * K + k] = (r > 0.0) ? w12o_double_to_bf16((double)hr[k] * inv) : (uint16_t)0;
    }
}

/* p[m,n] = bf16(fp32(g[m,n] u[m,n])): the fp32 product (exact in fp64, rounded once to fp32),
 * then rounded to nearest even; g and u have row stride ld. */
void w12o_mul_bf16(const float *g, const float *u, int M, int N, int ld, uint16_t *p) {
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            const float prod = (float)((double)g[(size_t)m * ld + n] * (double)u[(size_t)m * ld + n]);
            p[(size_t)m * N + n] = w12o_double_to_bf16((double)prod);
        }
}

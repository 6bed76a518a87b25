/*
 * CPU oracle for the fused RoPE + causal attention forward (prefill).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library; the two meet only in the seeded bf16 input bits.
 *
 * What it computes, in float64, straight from the definitions on the source
 * pages, one query row at a time, with the whole score row materialised
 * (no online recurrence, no tiling, no reordering):
 *
 *   theta_r  = base^(-2r/D), r = 0..D/2-1                (RoFormer; the RoPE
 *              convention is the NeoX half split: "AttnFuse", sec. 4.1 Fused RoPE)
 *   rotation of x at position p, pair (r, r+D/2), angle a = p*theta_r:
 *              x'_r       = x_r cos a - x_{r+D/2} sin a
 *              x'_{r+D/2} = x_{r+D/2} cos a + x_r sin a
 *   window   : W_r = floor(k * 2*pi / theta_r); the pair-r terms of cell (i,j)
 *              are kept iff the distance i-j <= W_r ("ATFlash", The idea:
 *              w_r = k*lambda_r, lambda_r = 2*pi/theta_r, terms beyond w_r are zero)
 *   score    : s_ij = (1/sqrt(D)) * sum_r keep_r(i-j) * (q'_{i,r} k'_{j,r}
 *                                   + q'_{i,r+D/2} k'_{j,r+D/2})
 *   mask     : keys j > i are excluded before the softmax when causal
 *              ("Attention block decomposition", Things that break;
 *              "Flash Attention: Causal Prefill D=128", reverse traversal mask)
 *   softmax  : m_i = max_j s_ij, p_ij = exp(s_ij - m_i), l_i = sum_j p_ij
 *   output   : O_i = sum_j p_ij V_j / l_i,  LSE_i = m_i + ln l_i
 *              ("AttnFuse", sec. 4.4: the forward keeps L = m + log l per row)
 *   GQA      : query head h reads KV head floor(h / (Hq/Hkv))
 *              ("AttnFuse", sec. 6.5 Llama-3-8B: Hq=32, Hkv=8)
 *
 * Positions are p = index + pos_offset for both Q and K (pos_offset is 0
 * except in the relative-position shift test).
 *
 * Built with -ffp-contract=off so that x86 and Arm builds round alike.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static const double ORACLE_TWO_PI = 6.283185307179586476925286766559;

static double bf16_to_f64(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* theta_r = base^(-2r/D) */
static void rope_thetas(int D, double base, double* theta) {
    for (int r = 0; r < D / 2; ++r) theta[r] = pow(base, -2.0 * (double)r / (double)D);
}

/* W_r = floor(k * 2*pi / theta_r); +inf when the window is off (k <= 0 or k infinite). */
void oracle_window_widths(int D, double rope_base, double window_k, double* w_out) {
    double theta[512];
    rope_thetas(D, rope_base, theta);
    for (int r = 0; r < D / 2; ++r) {
        if (!(window_k > 0.0) || isinf(window_k))
            w_out[r] = INFINITY;
        else
            w_out[r] = floor(window_k * ORACLE_TWO_PI / theta[r]);
    }
}

/* Rotate one bf16 vector x (length D, stride 1) at position pos into out (float64). */
static void rope_rotate(const uint16_t* x, int D, const double* theta, double pos, int rope_on, double* out) {
    int h = D / 2;
    for (int r = 0; r < h; ++r) {
        double a = bf16_to_f64(x[r]);
        double b = bf16_to_f64(x[r + h]);
        if (rope_on) {
            double ang = pos * theta[r];
            double c = cos(ang), s = sin(ang);
            out[r] = a * c - b * s;
            out[r + h] = b * c + a * s;
        } else {
            out[r] = a;
            out[r + h] = b;
        }
    }
}

/* Every row (b, s, h) of a BSHD bf16 tensor rotated at its position s, in
   float64 ("AttnFuse", sec. 4.1: pair r with r + D/2, theta_r = base^(-2r/D)). */
void oracle_rope_rotate(const uint16_t* x, int B, int S, int H, int D, double rope_base, double* out) {
    double theta[512];
    rope_thetas(D, rope_base, theta);
    const long long rows = (long long)B * S * H;
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < rows; ++i) {
        const long long s = (i / H) % S;
        rope_rotate(x + i * D, D, theta, (double)s, 1, out + i * D);
    }
}

int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Attention output for a list of query rows.
 *   q: [B][S][Hq][D] bf16 bits, k, v: [B][S][Hkv][D] bf16 bits (BSHD).
 *   rows n = 0..n_rows-1 select (row_b[n], row_h[n], row_i[n]).
 *   o_out: [n_rows][D] float64, lse_out: [n_rows] float64 (natural log).
 *   rope_base <= 0: RoPE off.  window_k <= 0 or infinite: window off.
 * Returns 0, or -1 on bad arguments (window without RoPE and causal masking,
 * Hq not a multiple of Hkv, out-of-range rows).
 */
int oracle_attn_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     int B, int Hq, int Hkv, int S, int D,
                     int causal, double rope_base, double window_k, long long pos_offset,
                     int n_rows, const int* row_b, const int* row_h, const int* row_i,
                     double* o_out, double* lse_out) {
    if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 2 || D % 2 != 0 || D > 1024) return -1;
    int rope_on = rope_base > 0.0;
    int window_on = window_k > 0.0 && !isinf(window_k);
    if (window_on && !(rope_on && causal)) return -1;
    for (int n = 0; n < n_rows; ++n)
        if (row_b[n] < 0 || row_b[n] >= B || row_h[n] < 0 || row_h[n] >= Hq || row_i[n] < 0 || row_i[n] >= S)
            return -1;

    const int G = Hq / Hkv;
    const int half = D / 2;
    double theta[512], W[512];
    if (rope_on) rope_thetas(D, rope_base, theta);
    oracle_window_widths(D, rope_on ? rope_base : 10000.0, window_on ? window_k : 0.0, W);
    const double inv_sqrt_d = 1.0 / sqrt((double)D);

    /* Rows are handled one (batch, KV head) group at a time, so each group's
       keys are rotated once and shared by its rows. */
    char* done = (char*)calloc((size_t)n_rows, 1);
    int* idx = (int*)malloc(sizeof(int) * (size_t)(n_rows > 0 ? n_rows : 1));
    for (int first = 0; first < n_rows; ++first) {
        if (done[first]) continue;
        const int b = row_b[first];
        const int g = row_h[first] / G;
        int cnt = 0, max_key = 0;
        for (int n = first; n < n_rows; ++n) {
            if (!done[n] && row_b[n] == b && row_h[n] / G == g) {
                idx[cnt++] = n;
                done[n] = 1;
                int last = causal ? row_i[n] : S - 1;
                if (last > max_key) max_key = last;
            }
        }
        const int nkeys = max_key + 1;
        double* krot = (double*)malloc(sizeof(double) * (size_t)nkeys * (size_t)D);
#pragma omp parallel for schedule(static)
        for (int j = 0; j < nkeys; ++j) {
            const uint16_t* kj = k + (((size_t)b * S + j) * Hkv + g) * (size_t)D;
            rope_rotate(kj, D, theta, (double)(j + pos_offset), rope_on, krot + (size_t)j * D);
        }
#pragma omp parallel for schedule(dynamic, 1)
        for (int t = 0; t < cnt; ++t) {
            const int n = idx[t];
            const int h = row_h[n], i = row_i[n];
            const int last = causal ? i : S - 1;
            double qrot[1024];
            const uint16_t* qi = q + (((size_t)b * S + i) * Hq + h) * (size_t)D;
            rope_rotate(qi, D, theta, (double)(i + pos_offset), rope_on, qrot);

            /* 1. the full score row */
            double* s = (double*)malloc(sizeof(double) * (size_t)(last + 1));
            for (int j = 0; j <= last; ++j) {
                const double* kj = krot + (size_t)j * D;
                const double dist = (double)(i - j);
                double acc = 0.0;
                for (int r = 0; r < half; ++r) {
                    if (window_on && !(dist <= W[r])) continue; /* pair r pruned at this distance */
                    acc += qrot[r] * kj[r] + qrot[r + half] * kj[r + half];
                }
                s[j] = acc * inv_sqrt_d;
            }
            /* 2. row maximum */
            double m = s[0];
            for (int j = 1; j <= last; ++j)
                if (s[j] > m) m = s[j];
            /* 3. exponentials and their sum */
            double l = 0.0;
            for (int j = 0; j <= last; ++j) {
                s[j] = exp(s[j] - m);
                l += s[j];
            }
            /* 4. weighted sum of values, divided once by the sum */
            double* o = o_out + (size_t)n * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            for (int j = 0; j <= last; ++j) {
                const uint16_t* vj = v + (((size_t)b * S + j) * Hkv + g) * (size_t)D;
                for (int d = 0; d < D; ++d) o[d] += s[j] * bf16_to_f64(vj[d]);
            }
            for (int d = 0; d < D; ++d) o[d] /= l;
            lse_out[n] = m + log(l);
            free(s);
        }
        free(krot);
    }
    free(idx);
    free(done);
    return 0;
}

/*
 * Number of pruned (cell, pair) terms over the causal S x S triangle, counted
 * cell by cell with the same keep rule the attention above uses: pair r of
 * cell (i, j), j <= i, is pruned iff i - j > W_r.
 */
long long oracle_pruned_terms(int S, int D, double rope_base, double window_k) {
    double W[512];
    oracle_window_widths(D, rope_base, window_k, W);
    long long count = 0;
#pragma omp parallel for reduction(+ : count) schedule(dynamic, 16)
    for (int i = 0; i < S; ++i)
        for (int j = 0; j <= i; ++j) {
            const double dist = (double)(i - j);
            for (int r = 0; r < D / 2; ++r)
                if (!(dist <= W[r])) ++count;
        }
    return count;
}

/*
 * Gradients of the attention above (RoPE, causal or full, GQA; the pair
 * window off; optionally a block mask, a sliding window and ALiBi, below)
 * for a scalar loss whose gradient with respect to O is dO ("AttnFuse",
 * sec. 4.4 Backward Pass: the backward re-derives the softmax probabilities
 * from the forward's per-row L = m + log l).  Written from the chain rule on
 * the definitions, one (batch, KV head) group at a time, with every
 * probability row materialised:
 *
 *   p_ij   = exp(s_ij - LSE_i)                  (s as in the forward, with
 *            the local forward's -m_h |i - j| when ALiBi is on: a constant in
 *            q and k, so dS keeps its form)
 *   dV_j   = sum_i p_ij dO_i                    (summed over the group's heads)
 *   dP_ij  = dO_i . V_j
 *   Dlt_i  = sum_j p_ij dP_ij                   (= dO_i . O_i)
 *   dS_ij  = p_ij (dP_ij - Dlt_i)               (softmax Jacobian)
 *   dq'_i  = (1/sqrt(D)) sum_j dS_ij k'_j,  dk'_j = (1/sqrt(D)) sum_i dS_ij q'_i
 *   dq_i   = R(p_i)^T dq'_i,  dk_j = R(p_j)^T dk'_j   (the transpose of the
 *            rotation of pair r by angle a: (x, y) -> (x cos a + y sin a,
 *            -x sin a + y cos a))
 *
 * Inputs are float64 (the bf16 bits widened by the caller, or any values for
 * a finite-difference check): q, dO [B][S][Hq][D]; k, v [B][S][Hkv][D].
 * Outputs dq [B][S][Hq][D], dk, dv [B][S][Hkv][D], float64.
 * Returns 0, or -1 on bad arguments.
 */
static int attn_bwd_masked(const double* q, const double* k, const double* v, const double* dO,
                           int B, int Hq, int Hkv, int S, int D, int causal, double rope_base,
                           const char* active, int block, int nb, int window, int alibi,
                           double* dq, double* dk, double* dv) {
    if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 2 || D % 2 != 0 || D > 1024 || window < 0)
        return -1;
    const int rope_on = rope_base > 0.0;
    const int G = Hq / Hkv;
    const int half = D / 2;
    double theta[512];
    if (rope_on) rope_thetas(D, rope_base, theta);
    const double inv_sqrt_d = 1.0 / sqrt((double)D);

#pragma omp parallel for schedule(dynamic, 1)
    for (int bg = 0; bg < B * Hkv; ++bg) {
        const int b = bg / Hkv, g = bg % Hkv;
        double* kr = (double*)malloc(sizeof(double) * (size_t)S * D);   /* rotated keys */
        double* dkr = (double*)calloc((size_t)S * D, sizeof(double));   /* gradient wrt rotated keys */
        double* qr = (double*)malloc(sizeof(double) * (size_t)D);
        double* dqr = (double*)malloc(sizeof(double) * (size_t)D);
        double* p = (double*)malloc(sizeof(double) * (size_t)S);
        double* dp = (double*)malloc(sizeof(double) * (size_t)S);
        double* dvg = dv + ((size_t)b * S * Hkv + g) * D;  /* row j at dvg + j * Hkv * D */
        for (int j = 0; j < S; ++j)
            for (int d = 0; d < D; ++d) dvg[(size_t)j * Hkv * D + d] = 0.0;
        /* rotated keys */
        for (int j = 0; j < S; ++j) {
            const double* kj = k + (((size_t)b * S + j) * Hkv + g) * D;
            double* o = kr + (size_t)j * D;
            for (int r = 0; r < half; ++r) {
                const double x = kj[r], y = kj[r + half];
                if (rope_on) {
                    const double a = (double)j * theta[r], c = cos(a), s = sin(a);
                    o[r] = x * c - y * s;
                    o[r + half] = y * c + x * s;
                } else {
                    o[r] = x;
                    o[r + half] = y;
                }
            }
        }
        for (int h = g * G; h < (g + 1) * G; ++h) {
            const double slope = alibi ? pow(2.0, -8.0 * (double)(h + 1) / (double)Hq) : 0.0;
            for (int i = 0; i < S; ++i) {
                const int last = causal ? i : S - 1;
                /* key j is visible iff j <= last, (no mask, or block (i/block, j/block) listed) and
                 * (no window, or |i - j| < window) */
#define DIST(j) ((i) >= (j) ? (i) - (j) : (j) - (i))
#define VISIBLE(j) ((active == NULL || active[(size_t)(i / block) * nb + (j) / block]) && \
                    (window == 0 || DIST(j) < window))
                const double* qi = q + (((size_t)b * S + i) * Hq + h) * D;
                const double* doi = dO + (((size_t)b * S + i) * Hq + h) * D;
                for (int r = 0; r < half; ++r) {
                    const double x = qi[r], y = qi[r + half];
                    if (rope_on) {
                        const double a = (double)i * theta[r], c = cos(a), s = sin(a);
                        qr[r] = x * c - y * s;
                        qr[r + half] = y * c + x * s;
                    } else {
                        qr[r] = x;
                        qr[r + half] = y;
                    }
                }
                /* probabilities of row i */
                double m = -INFINITY;
                for (int j = 0; j <= last; ++j) {
                    if (!VISIBLE(j)) continue;
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d) acc += qr[d] * kr[(size_t)j * D + d];
                    p[j] = acc * inv_sqrt_d - slope * (double)DIST(j);
                    if (p[j] > m) m = p[j];
                }
                double l = 0.0;
                for (int j = 0; j <= last; ++j) {
                    p[j] = VISIBLE(j) ? exp(p[j] - m) : 0.0; /* a hidden key has probability 0 */
                    l += p[j];
                }
                if (l == 0.0) { /* a row that sees no key: no gradient flows through it */
                    double* dqi = dq + (((size_t)b * S + i) * Hq + h) * D;
                    for (int d = 0; d < D; ++d) dqi[d] = 0.0;
                    continue;
                }
                for (int j = 0; j <= last; ++j) p[j] /= l;
                /* dV, dP and the row's Dlt */
                double dlt = 0.0;
                for (int j = 0; j <= last; ++j) {
                    const double* vj = v + (((size_t)b * S + j) * Hkv + g) * D;
                    double* dvj = dvg + (size_t)j * Hkv * D;
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d) {
                        dvj[d] += p[j] * doi[d];
                        acc += doi[d] * vj[d];
                    }
                    dp[j] = acc;
                    dlt += p[j] * acc;
                }
                /* dS, then the gradients wrt the rotated q and k */
                for (int d = 0; d < D; ++d) dqr[d] = 0.0;
                for (int j = 0; j <= last; ++j) {
                    if (!VISIBLE(j)) continue;
                    const double ds = p[j] * (dp[j] - dlt) * inv_sqrt_d;
                    for (int d = 0; d < D; ++d) {
                        dqr[d] += ds * kr[(size_t)j * D + d];
                        dkr[(size_t)j * D + d] += ds * qr[d];
                    }
                }
                /* back through the rotation of q */
                double* dqi = dq + (((size_t)b * S + i) * Hq + h) * D;
                for (int r = 0; r < half; ++r) {
                    const double x = dqr[r], y = dqr[r + half];
                    if (rope_on) {
                        const double a = (double)i * theta[r], c = cos(a), s = sin(a);
                        dqi[r] = x * c + y * s;
                        dqi[r + half] = -x * s + y * c;
                    } else {
                        dqi[r] = x;
                        dqi[r + half] = y;
                    }
                }
            }
        }
        /* back through the rotation of k */
        for (int j = 0; j < S; ++j) {
            const double* x0 = dkr + (size_t)j * D;
            double* dkj = dk + (((size_t)b * S + j) * Hkv + g) * D;
            for (int r = 0; r < half; ++r) {
                const double x = x0[r], y = x0[r + half];
                if (rope_on) {
                    const double a = (double)j * theta[r], c = cos(a), s = sin(a);
                    dkj[r] = x * c + y * s;
                    dkj[r + half] = -x * s + y * c;
                } else {
                    dkj[r] = x;
                    dkj[r + half] = y;
                }
            }
        }
        free(kr);
        free(dkr);
        free(qr);
        free(dqr);
        free(p);
        free(dp);
    }
#undef VISIBLE
#undef DIST
    return 0;
}

int oracle_attn_bwd(const double* q, const double* k, const double* v, const double* dO,
                    int B, int Hq, int Hkv, int S, int D, int causal, double rope_base,
                    double* dq, double* dk, double* dv) {
    return attn_bwd_masked(q, k, v, dO, B, Hq, Hkv, S, D, causal, rope_base, NULL, 1, 1, 0, 0, dq, dk, dv);
}

/*
 * The same gradients with a sliding window and/or ALiBi ("AttnFuse", sec. 3:
 * the sliding_window and alibi combinators; sec. 4.4: the backward re-derives
 * P from the forward's statistics): key j is visible to query i iff j <= i
 * when causal and |i - j| < window when window > 0, and the score carries
 * -m_h |i - j| (m_h = 2^(-8 (h+1) / Hq)) when alibi is 1, as in
 * oracle_attn_rows_local.  Returns 0, or -1 on bad arguments.
 */
int oracle_attn_bwd_local(const double* q, const double* k, const double* v, const double* dO,
                          int B, int Hq, int Hkv, int S, int D, int causal, double rope_base,
                          int window, int alibi, double* dq, double* dk, double* dv) {
    if (alibi != 0 && alibi != 1) return -1;
    return attn_bwd_masked(q, k, v, dO, B, Hq, Hkv, S, D, causal, rope_base, NULL, 1, 1, window, alibi, dq, dk, dv);
}

/*
 * The same gradients under a block-sparse mask ("AttnFuse", sec. 4.3: the
 * backward also sees only the listed blocks): key j is visible to query i iff
 * block (i / block, j / block) is listed in the CSR mask (and j <= i when
 * causal); hidden keys have probability 0, and a row that sees no key passes
 * no gradient.  Returns 0, or -1 on bad arguments.
 */
int oracle_attn_bwd_bs(const double* q, const double* k, const double* v, const double* dO,
                       int B, int Hq, int Hkv, int S, int D, int causal, double rope_base,
                       int block, const int* row_ptr, const int* col_idx,
                       double* dq, double* dk, double* dv) {
    if (block < 1 || S < 1) return -1;
    const int nb = (S + block - 1) / block;
    for (int r = 0; r < nb; ++r) {
        if (row_ptr[r + 1] < row_ptr[r]) return -1;
        for (int e = row_ptr[r]; e < row_ptr[r + 1]; ++e)
            if (col_idx[e] < 0 || col_idx[e] >= nb) return -1;
    }
    char* active = (char*)calloc((size_t)nb * nb, 1);
    for (int r = 0; r < nb; ++r)
        for (int e = row_ptr[r]; e < row_ptr[r + 1]; ++e) active[(size_t)r * nb + col_idx[e]] = 1;
    const int rc = attn_bwd_masked(q, k, v, dO, B, Hq, Hkv, S, D, causal, rope_base, active, block, nb, 0, 0,
                                   dq, dk, dv);
    free(active);
    return rc;
}

/*
 * Block-sparse attention output ("AttnFuse", sec. 4.3 Block-Sparse Attention:
 * a CSR BlockMask lists, per row of blocks, the active key blocks; only those
 * blocks' scores enter the softmax).  Blocks are `block` x `block`; the mask
 * is shared by every batch element and head: key j is visible to query i iff
 * block (i / block, j / block) is listed (and j <= i when causal).  Each row's
 * score vector is materialised over the visible keys only, then handled as in
 * oracle_attn_rows (RoPE, scale, max, exponentials, weighted sum, LSE).
 * A row that sees no key gets O = 0 and LSE = -inf.
 *   row_ptr [ceil(S/block) + 1], col_idx [row_ptr[last]]: the CSR mask.
 * Returns 0, or -1 on bad arguments.
 */
int oracle_attn_rows_bs(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        int B, int Hq, int Hkv, int S, int D, int causal, double rope_base,
                        int block, const int* row_ptr, const int* col_idx,
                        int n_rows, const int* row_b, const int* row_h, const int* row_i,
                        double* o_out, double* lse_out) {
    if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 2 || D % 2 != 0 || D > 1024 || block < 1)
        return -1;
    const int nb = (S + block - 1) / block;
    for (int r = 0; r < nb; ++r) {
        if (row_ptr[r + 1] < row_ptr[r]) return -1;
        for (int e = row_ptr[r]; e < row_ptr[r + 1]; ++e)
            if (col_idx[e] < 0 || col_idx[e] >= nb) return -1;
    }
    for (int n = 0; n < n_rows; ++n)
        if (row_b[n] < 0 || row_b[n] >= B || row_h[n] < 0 || row_h[n] >= Hq || row_i[n] < 0 || row_i[n] >= S)
            return -1;
    /* the active table, one byte per (query block, key block) */
    char* active = (char*)calloc((size_t)nb * nb, 1);
    for (int r = 0; r < nb; ++r)
        for (int e = row_ptr[r]; e < row_ptr[r + 1]; ++e) active[(size_t)r * nb + col_idx[e]] = 1;
    const int rope_on = rope_base > 0.0;
    const int G = Hq / Hkv;
    double theta[512];
    if (rope_on) rope_thetas(D, rope_base, theta);
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
#pragma omp parallel for schedule(dynamic, 1)
    for (int n = 0; n < n_rows; ++n) {
        const int b = row_b[n], h = row_h[n], i = row_i[n], g = h / G;
        double qrot[1024], krot[1024];
        rope_rotate(q + (((size_t)b * S + i) * Hq + h) * D, D, theta, (double)i, rope_on, qrot);
        double* s = (double*)malloc(sizeof(double) * (size_t)S);
        int* key = (int*)malloc(sizeof(int) * (size_t)S);
        int cnt = 0;
        for (int j = 0; j < S; ++j) {
            if (!active[(size_t)(i / block) * nb + j / block]) continue;
            if (causal && j > i) continue;
            rope_rotate(k + (((size_t)b * S + j) * Hkv + g) * D, D, theta, (double)j, rope_on, krot);
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += qrot[d] * krot[d];
            s[cnt] = acc * inv_sqrt_d;
            key[cnt++] = j;
        }
        double* o = o_out + (size_t)n * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (cnt == 0) {
            lse_out[n] = -INFINITY;
        } else {
            double m = s[0];
            for (int c = 1; c < cnt; ++c)
                if (s[c] > m) m = s[c];
            double l = 0.0;
            for (int c = 0; c < cnt; ++c) {
                s[c] = exp(s[c] - m);
                l += s[c];
            }
            for (int c = 0; c < cnt; ++c) {
                const uint16_t* vj = v + (((size_t)b * S + key[c]) * Hkv + g) * D;
                for (int d = 0; d < D; ++d) o[d] += s[c] * bf16_to_f64(vj[d]);
            }
            for (int d = 0; d < D; ++d) o[d] /= l;
            lse_out[n] = m + log(l);
        }
        free(s);
        free(key);
    }
    free(active);
    return 0;
}

/*
 * Attention with a sliding window and/or ALiBi ("AttnFuse", sec. 3: the
 * sliding_window and alibi combinators; sliding windows and linear biases
 * after its refs. 6 and 7), for a list of query rows, from the definitions:
 *   visible(i, j) = (j <= i when causal) and (|i - j| < window when window > 0)
 *   s_ij = q'_i . k'_j / sqrt(D) - m_h |i - j|   (ALiBi on: m_h = 2^(-8 (h+1) / Hq))
 * then the row's maximum, exponentials, weighted sum and LSE as in
 * oracle_attn_rows, over the visible keys only.
 * Returns 0, or -1 on bad arguments.
 */
int oracle_attn_rows_local(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           int B, int Hq, int Hkv, int S, int D, int causal, double rope_base,
                           int window, int alibi,
                           int n_rows, const int* row_b, const int* row_h, const int* row_i,
                           double* o_out, double* lse_out) {
    if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 2 || D % 2 != 0 || D > 1024 || window < 0)
        return -1;
    for (int n = 0; n < n_rows; ++n)
        if (row_b[n] < 0 || row_b[n] >= B || row_h[n] < 0 || row_h[n] >= Hq || row_i[n] < 0 || row_i[n] >= S)
            return -1;
    const int rope_on = rope_base > 0.0;
    const int G = Hq / Hkv;
    double theta[512];
    if (rope_on) rope_thetas(D, rope_base, theta);
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
#pragma omp parallel for schedule(dynamic, 1)
    for (int n = 0; n < n_rows; ++n) {
        const int b = row_b[n], h = row_h[n], i = row_i[n], g = h / G;
        const double slope = alibi ? pow(2.0, -8.0 * (double)(h + 1) / (double)Hq) : 0.0;
        double qrot[1024], krot[1024];
        rope_rotate(q + (((size_t)b * S + i) * Hq + h) * D, D, theta, (double)i, rope_on, qrot);
        double* s = (double*)malloc(sizeof(double) * (size_t)S);
        int* key = (int*)malloc(sizeof(int) * (size_t)S);
        int cnt = 0;
        for (int j = 0; j < S; ++j) {
            const int dist = i >= j ? i - j : j - i;
            if (causal && j > i) continue;
            if (window > 0 && dist >= window) continue;
            rope_rotate(k + (((size_t)b * S + j) * Hkv + g) * D, D, theta, (double)j, rope_on, krot);
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += qrot[d] * krot[d];
            s[cnt] = acc * inv_sqrt_d - slope * (double)dist;
            key[cnt++] = j;
        }
        double* o = o_out + (size_t)n * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        double m = s[0];
        for (int c = 1; c < cnt; ++c)
            if (s[c] > m) m = s[c];
        double l = 0.0;
        for (int c = 0; c < cnt; ++c) {
            s[c] = exp(s[c] - m);
            l += s[c];
        }
        for (int c = 0; c < cnt; ++c) {
            const uint16_t* vj = v + (((size_t)b * S + key[c]) * Hkv + g) * D;
            for (int d = 0; d < D; ++d) o[d] += s[c] * bf16_to_f64(vj[d]);
        }
        for (int d = 0; d < D; ++d) o[d] /= l;
        lse_out[n] = m + log(l);
        free(s);
        free(key);
    }
    return 0;
}

/*
 * ssd_oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.
 *
 * A plain, slow, sequential float64 CPU implementation of the Mamba-2 SSD
 * (state-space duality) scan and its exact adjoint.  Only tests/, the smoke
 * check and bench.py's CPU-baseline leg may load this file's library.  It shares
 * no code, header or table with the CUDA library.
 *
 * What it computes (the recurrence stated for Mamba-2 SSD; the Mamba-3-Lite
 * "SSD Reference" page, section "Math: the recurrence both functions implement",
 * writes the same recurrence without the dt factor on the input, and its
 * "ssd_naive_complex -- the O(T) oracle" section gives the literal-loop design
 * followed here):
 *
 *   dt_t  = softplus(dt_raw_t + dt_bias_h)
 *   a_t   = exp(dt_t * A_h)
 *   h_t   = a_t * h_{t-1} + dt_t * x_t (outer) B_t          state h is [P][N]
 *   ypre_t= C_t . h_t  (contract N)  + D_h * x_t
 *   y_t   = ypre_t * silu(z_t)     if z is given, else ypre_t
 *
 * Head h reads B/C group g = h / (H/G).  h_{-1} = initial state (0 if absent);
 * the final state is h after the last token of the sequence.  State layout is
 * [P][N] (head dim before state dim), as in that page's "Shape contract".
 *
 * Sequences: the token axis is flat; sequence s covers tokens [cu[s], cu[s+1]).
 * A fixed-length batch of B rows of length L is cu = {0, L, 2L, ...}.
 *
 * The backward is the reverse-mode adjoint of exactly this loop, for the loss
 * L = sum(dy * y) + sum(dfinal * final).  States are checkpointed every `ckpt`
 * steps and recomputed inside each segment.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int64_t nseq, H, P, G, N;
    const int64_t *cu;      /* [nseq+1] token offsets */
    const double *x;        /* [T][H][P] */
    const double *dt_raw;   /* [T][H] */
    const double *A;        /* [H] */
    const double *Bm;       /* [T][G][N] */
    const double *Cm;       /* [T][G][N] */
    const double *D;        /* [H] or NULL */
    const double *z;        /* [T][H][P] or NULL */
    const double *dt_bias;  /* [H] or NULL */
    const double *init;     /* [nseq][H][P][N] or NULL */
    const int32_t *head_mask; /* [H] nonzero = compute this head; NULL = all */
} ssd_oracle_in;

static double softplus(double v) { return v > 0.0 ? v + log1p(exp(-v)) : log1p(exp(v)); }
static double sigmoid(double v) {
    if (v >= 0.0) return 1.0 / (1.0 + exp(-v));
    double e = exp(v);
    return e / (1.0 + e);
}

static int head_on(const ssd_oracle_in *in, int64_t h) {
    return in->head_mask == NULL || in->head_mask[h] != 0;
}

/* One forward step of the recurrence on state st[P][N]; returns nothing, fills
 * ypre[P] (before gating).  dt and a are returned through pointers. */
static void fwd_step(const ssd_oracle_in *in, int64_t t, int64_t h, int64_t g, double *st,
                     double *ypre, double *dt_out, double *a_out, double *v_out) {
    const int64_t H = in->H, P = in->P, G = in->G, N = in->N;
    double v = in->dt_raw[t * H + h] + (in->dt_bias ? in->dt_bias[h] : 0.0);
    double dt = softplus(v);
    double a = exp(dt * in->A[h]);
    const double *xr = in->x + (t * H + h) * P;
    const double *br = in->Bm + (t * G + g) * N;
    const double *cr = in->Cm + (t * G + g) * N;
    for (int64_t p = 0; p < P; ++p) {
        double *row = st + p * N;
        double dx = dt * xr[p];
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            row[n] = a * row[n] + dx * br[n];
            acc += cr[n] * row[n];
        }
        ypre[p] = acc + (in->D ? in->D[h] * xr[p] : 0.0);
    }
    if (dt_out) *dt_out = dt;
    if (a_out) *a_out = a;
    if (v_out) *v_out = v;
}

int ssd_oracle_fwd(const ssd_oracle_in *in, double *y, double *final_states, int nthreads) {
    const int64_t S = in->nseq, H = in->H, P = in->P, G = in->G, N = in->N;
    if (H % G != 0) return 1;
    const int64_t hpg = H / G;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t sh = 0; sh < S * H; ++sh) {
        const int64_t s = sh / H, h = sh % H, g = h / hpg;
        if (!head_on(in, h)) continue;
        double *st = (double *)malloc(sizeof(double) * (size_t)(P * N));
        double *ypre = (double *)malloc(sizeof(double) * (size_t)P);
        if (!st || !ypre) { free(st); free(ypre); err = 2; continue; }
        if (in->init) memcpy(st, in->init + (s * H + h) * P * N, sizeof(double) * (size_t)(P * N));
        else memset(st, 0, sizeof(double) * (size_t)(P * N));
        for (int64_t t = in->cu[s]; t < in->cu[s + 1]; ++t) {
            fwd_step(in, t, h, g, st, ypre, NULL, NULL, NULL);
            double *yr = y + (t * H + h) * P;
            if (in->z) {
                const double *zr = in->z + (t * H + h) * P;
                for (int64_t p = 0; p < P; ++p) yr[p] = ypre[p] * zr[p] * sigmoid(zr[p]);
            } else {
                for (int64_t p = 0; p < P; ++p) yr[p] = ypre[p];
            }
        }
        if (final_states) memcpy(final_states + (s * H + h) * P * N, st, sizeof(double) * (size_t)(P * N));
        free(st);
        free(ypre);
    }
    return err;
}

/*
 * Adjoint.  Work is split by (sequence, head).  Each task writes its head's dB/dC
 * contributions into a private buffer; afterwards the buffers of the heads of
 * each group are summed in ascending head order, and the per-head scalars
 * (dA, dD, ddt_bias) are summed over sequences in order -- so the result does
 * not depend on the thread count.
 */
int ssd_oracle_bwd(const ssd_oracle_in *in, const double *dy, const double *dfinal,
                   double *dx, double *ddt_raw, double *dA, double *dB, double *dC,
                   double *dD, double *dz, double *ddt_bias, double *dinit,
                   int64_t ckpt, int nthreads) {
    const int64_t S = in->nseq, H = in->H, P = in->P, G = in->G, N = in->N;
    if (H % G != 0) return 1;
    if (ckpt <= 0) ckpt = 128;
    const int64_t hpg = H / G;
    const int64_t T = in->cu[S];
    const size_t PN = (size_t)(P * N);
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    double *pA = (double *)calloc((size_t)(S * H), sizeof(double));
    double *pD = (double *)calloc((size_t)(S * H), sizeof(double));
    double *pBias = (double *)calloc((size_t)(S * H), sizeof(double));
    /* per-head dB/dC rows: [H][T][N], only touched for computed heads */
    double *hB = (double *)calloc((size_t)(H * T * N) + 1, sizeof(double));
    double *hC = (double *)calloc((size_t)(H * T * N) + 1, sizeof(double));
    if (!pA || !pD || !pBias || !hB || !hC) {
        free(pA); free(pD); free(pBias); free(hB); free(hC);
        return 2;
    }
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t sh = 0; sh < S * H; ++sh) {
        const int64_t s = sh / H, h = sh % H, g = h / hpg;
        if (!head_on(in, h)) continue;
        const int64_t t0 = in->cu[s], t1 = in->cu[s + 1], len = t1 - t0;
        const int64_t nck = len / ckpt + 1;
        double *ck = (double *)malloc(sizeof(double) * PN * (size_t)nck);
        double *seg = (double *)malloc(sizeof(double) * PN * (size_t)(ckpt + 1));
        double *Gs = (double *)malloc(sizeof(double) * PN);
        double *ypre = (double *)malloc(sizeof(double) * (size_t)P);
        double *dyp = (double *)malloc(sizeof(double) * (size_t)P);
        if (!ck || !seg || !Gs || !ypre || !dyp) {
            free(ck); free(seg); free(Gs); free(ypre); free(dyp);
            err = 2;
            continue;
        }
        const double Ah = in->A[h];
        const double Dh = in->D ? in->D[h] : 0.0;
        /* forward: checkpoints ck[k] = state before token t0 + k*ckpt */
        double *st = seg; /* scratch */
        if (in->init) memcpy(st, in->init + (s * H + h) * PN, sizeof(double) * PN);
        else memset(st, 0, sizeof(double) * PN);
        for (int64_t k = 0; k < len; ++k) {
            if (k % ckpt == 0) memcpy(ck + (size_t)(k / ckpt) * PN, st, sizeof(double) * PN);
            fwd_step(in, t0 + k, h, g, st, ypre, NULL, NULL, NULL);
        }
        /* reverse sweep */
        if (dfinal) memcpy(Gs, dfinal + (s * H + h) * PN, sizeof(double) * PN);
        else memset(Gs, 0, sizeof(double) * PN);
        double accA = 0.0, accD = 0.0, accBias = 0.0;
        for (int64_t sgi = (len > 0 ? (len - 1) / ckpt : -1); sgi >= 0; --sgi) {
            const int64_t k0 = sgi * ckpt;
            const int64_t k1 = (k0 + ckpt < len) ? k0 + ckpt : len;
            /* seg[j] = state before token k0+j, j = 0..k1-k0 */
            memcpy(seg, ck + (size_t)sgi * PN, sizeof(double) * PN);
            for (int64_t k = k0; k < k1; ++k) {
                double *nx = seg + (size_t)(k - k0 + 1) * PN;
                memcpy(nx, seg + (size_t)(k - k0) * PN, sizeof(double) * PN);
                fwd_step(in, t0 + k, h, g, nx, ypre, NULL, NULL, NULL);
            }
            for (int64_t k = k1 - 1; k >= k0; --k) {
                const int64_t t = t0 + k;
                const double *hprev = seg + (size_t)(k - k0) * PN;
                const double *hcur = seg + (size_t)(k - k0 + 1) * PN;
                double v = in->dt_raw[t * H + h] + (in->dt_bias ? in->dt_bias[h] : 0.0);
                double dt = softplus(v);
                double a = exp(dt * Ah);
                const double *xr = in->x + (t * H + h) * P;
                const double *br = in->Bm + (t * G + g) * N;
                const double *cr = in->Cm + (t * G + g) * N;
                const double *dyr = dy + (t * H + h) * P;
                /* ypre recomputed from h_t */
                for (int64_t p = 0; p < P; ++p) {
                    double acc = 0.0;
                    for (int64_t n = 0; n < N; ++n) acc += cr[n] * hcur[p * N + n];
                    ypre[p] = acc + Dh * xr[p];
                }
                if (in->z) {
                    const double *zr = in->z + (t * H + h) * P;
                    double *dzr = dz + (t * H + h) * P;
                    for (int64_t p = 0; p < P; ++p) {
                        double sg_ = sigmoid(zr[p]);
                        dyp[p] = dyr[p] * zr[p] * sg_;
                        dzr[p] = dyr[p] * ypre[p] * sg_ * (1.0 + zr[p] * (1.0 - sg_));
                    }
                } else {
                    for (int64_t p = 0; p < P; ++p) dyp[p] = dyr[p];
                }
                /* dL/dh_t += C_t (outer) dypre ; dC_t += dypre . h_t */
                double *dcr = hC + ((size_t)h * (size_t)T + (size_t)t) * (size_t)N;
                for (int64_t p = 0; p < P; ++p) {
                    double *grow = Gs + p * N;
                    const double *hrow = hcur + p * N;
                    for (int64_t n = 0; n < N; ++n) {
                        grow[n] += cr[n] * dyp[p];
                        dcr[n] += dyp[p] * hrow[n];
                    }
                    accD += dyp[p] * xr[p];
                }
                /* through h_t = a h_{t-1} + dt x (outer) B */
                double *dxr = dx + (t * H + h) * P;
                double *dbr = hB + ((size_t)h * (size_t)T + (size_t)t) * (size_t)N;
                double ddt = 0.0, dAa = 0.0;
                for (int64_t p = 0; p < P; ++p) {
                    const double *grow = Gs + p * N;
                    const double *hrow = hprev + p * N;
                    double gb = 0.0;
                    for (int64_t n = 0; n < N; ++n) {
                        gb += grow[n] * br[n];
                        dbr[n] += dt * grow[n] * xr[p];
                        dAa += grow[n] * hrow[n];
                    }
                    dxr[p] = Dh * dyp[p] + dt * gb;
                    ddt += xr[p] * gb;
                }
                /* dAa = <G, h_{t-1}>; d a_t contributes via a = exp(dt*A) */
                ddt += dAa * a * Ah;
                accA += dAa * a * dt;
                double dv = ddt * sigmoid(v);
                ddt_raw[t * H + h] = dv;
                accBias += dv;
                for (size_t i = 0; i < PN; ++i) Gs[i] *= a;
            }
        }
        if (dinit) memcpy(dinit + (s * H + h) * PN, Gs, sizeof(double) * PN);
        pA[s * H + h] = accA;
        pD[s * H + h] = accD;
        pBias[s * H + h] = accBias;
        free(ck); free(seg); free(Gs); free(ypre); free(dyp);
    }
    /* dB/dC: heads of each group summed in ascending order */
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t g = 0; g < G; ++g) {
            double *ob = dB + (t * G + g) * N;
            double *oc = dC + (t * G + g) * N;
            for (int64_t n = 0; n < N; ++n) { ob[n] = 0.0; oc[n] = 0.0; }
            for (int64_t h = g * hpg; h < (g + 1) * hpg; ++h) {
                if (!head_on(in, h)) continue;
                const double *sb = hB + ((size_t)h * (size_t)T + (size_t)t) * (size_t)N;
                const double *sc = hC + ((size_t)h * (size_t)T + (size_t)t) * (size_t)N;
                for (int64_t n = 0; n < N; ++n) { ob[n] += sb[n]; oc[n] += sc[n]; }
            }
        }
    }
    for (int64_t h = 0; h < H; ++h) {
        double a = 0.0, d = 0.0, b = 0.0;
        for (int64_t s = 0; s < S; ++s) {
            a += pA[s * H + h];
            d += pD[s * H + h];
            b += pBias[s * H + h];
        }
        dA[h] = a;
        if (dD) dD[h] = d;
        if (ddt_bias) ddt_bias[h] = b;
    }
    free(pA); free(pD); free(pBias); free(hB); free(hC);
    return err;
}

int ssd_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

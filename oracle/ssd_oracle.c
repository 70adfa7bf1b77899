/*
 * ssd_oracle.c -- plain fp64 CPU oracle of the Mamba-2 (SSD) mixer core.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path (the
 * CUDA library under ssd_scan_gb300/) shares no code, header, table or helper
 * with this file, and never calls it.
 *
 * Everything is computed in double precision, row-major, one element at a
 * time, in the order the method is written on the pages.  There is no
 * blocking or fusion beyond what each definition states.
 *
 * Sources (page title, section):
 *  [TS]  TensorSharp "docs/models/nemotron.md" (Nemotron-H), section 3
 *        "Forward graph" (Mamba2 branch) and section 4.1 "Mamba2 SSM layer"
 *        (the single-step formulas: dA, dB, state update, y = state.C,
 *        y += x*D), section 6 "Weight naming convention" (parameter shapes:
 *        ssm_conv1d.weight [xBCSize, convKernel], optional ssm_conv1d.bias,
 *        ssm_dt.bias [nHead], ssm_a [nHead], optional ssm_d [nHead]) and
 *        section 10 "Memory and KV cache strategy" (conv state holds
 *        convKernel-1 rows of the xBC stream; SSM state has
 *        dState x headDim x nHead floats).
 *  [TRT] TensorRT-Model-Connect PR #2207 "perf(nemotron_h): prefill
 *        single-GPU prompts in multi-token chunks", section "Implementation"
 *        (chunk form with a_t = dt_t A, gamma_t = sum_{i<=t} a_i, gamma_S read
 *        from the last cumulative-sum element, every exponent clamped at
 *        <= 0, causal depthwise conv over previous conv state plus chunk).
 *  [VLC] vllm.cpp PR #1362 "NemotronH decodes on the single-step recurrent
 *        kernels", summary (stream split z | xBC | dt then x | B | C, the
 *        head -> group mapping h / heads_per_group, in-place state update at
 *        the state slot).
 *
 * Readings where the pages are silent or garbled (each also listed in the
 * design notes of the repository):
 *  - A is stored negative; the per-row decay is exp(dt*A) <= 1.  (The
 *    TensorSharp page writes exp(-softplus(dt)*A) with A > 0; the chunk form
 *    on the TensorRT page writes a_t = dt_t*A.  Both are the same decay.)
 *  - dt = softplus(dt_raw + dt_bias), softplus(v) = max(v,0)+log1p(exp(-|v|))
 *    with no threshold.  With flag ORACLE_DT_SOFTPLUS clear, dt = dt_raw.
 *  - conv tap k = W-1 multiplies the newest row; conv state holds the W-1
 *    most recent raw rows, oldest first.
 *  - y uses the post-update state (state first, then y = state.C).
 *  - z gate is y * silu(z) (the group RMSNorm is a separate step, below).
 *  - group RMSNorm then gate: out = silu(z) * y / sqrt(mean_group(y^2) + eps)
 *    * w, in that order ([TS] 4.1: the norm acts on y, then the gate); eps is
 *    not on the pages and is an argument.
 *
 * Parity unpinned: none of the functions below (each has at least one pin in
 * the CPU test-suite that does not re-type its formula).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

/* ORACLE_MUTANT (default 0) plants one known mistake, for the mutation tests
 * that prove the pins can see it; a normal build never defines it.  In the
 * chunk form: 10 drops every clamp, 11 takes gamma_L from a separate
 * reduction (fp32, rows in reverse) with the state exponent unclamped, 12
 * clamps gamma_t and gamma_s one by one instead of their difference; 13
 * combines two segments' states without the second segment's decay. */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

#define ORACLE_DT_SOFTPLUS 1u
#define ORACLE_HAS_Z 2u

typedef struct {
    int batch, seqlen, nheads, headdim, dstate, ngroups;
} oracle_dims;

static double oracle_softplus(double v)
{
    /* log(1 + e^v) written so that neither branch overflows. */
    return (v > 0.0 ? v : 0.0) + log1p(exp(-fabs(v)));
}

static double oracle_silu(double v)
{
    return v / (1.0 + exp(-v));
}

/*
 * Causal depthwise conv1d with SiLU over [previous conv state ; rows].
 * [TS] section 3 (Conv1dStep then SiLU) and section 10; [TRT] Implementation
 * (add_short_conv_rows: conv over the previous conv state plus the chunk).
 *
 *   u = [state_in (W-1 rows) ; xbc (S rows)]          per sequence
 *   v[t,c] = bias[c] + sum_{k=0}^{W-1} w[c,k] * u[t+k, c]
 *   out[t,c] = silu(v[t,c])   (or v when apply_silu == 0)
 *   state_out = the last W-1 rows of u
 */
void oracle_conv1d(int B, int S, int Cdim, int W,
                   const double* xbc, const double* conv_w,
                   const double* conv_b, const double* state_in,
                   double* out, double* state_out, int apply_silu)
{
    const int nhist = W - 1;
    const int U = nhist + S;
    double* u = (double*)malloc(sizeof(double) * (size_t)(U > 0 ? U : 1) * (size_t)Cdim);
    for (int b = 0; b < B; ++b) {
        /* build u row by row */
        for (int r = 0; r < nhist; ++r)
            for (int c = 0; c < Cdim; ++c)
                u[(size_t)r * Cdim + c] =
                    state_in ? state_in[((size_t)b * nhist + r) * Cdim + c] : 0.0;
        for (int t = 0; t < S; ++t)
            for (int c = 0; c < Cdim; ++c)
                u[(size_t)(nhist + t) * Cdim + c] = xbc[((size_t)b * S + t) * Cdim + c];
        for (int t = 0; t < S; ++t) {
            for (int c = 0; c < Cdim; ++c) {
                double v = conv_b ? conv_b[c] : 0.0;
                for (int k = 0; k < W; ++k)
                    v += conv_w[(size_t)c * W + (ORACLE_MUTANT == 4 ? W - 1 - k : k)] *
                         u[(size_t)(t + k) * Cdim + c];
                out[((size_t)b * S + t) * Cdim + c] = apply_silu ? oracle_silu(v) : v;
            }
        }
        if (state_out) {
            for (int r = 0; r < nhist; ++r)
                for (int c = 0; c < Cdim; ++c)
                    state_out[((size_t)b * nhist + r) * Cdim + c] =
                        u[(size_t)(U - nhist + r) * Cdim + c];
        }
    }
    free(u);
}

/* ------------------------------------------------------------------------ */
/* Shared argument block for the two scan forms.                            */

typedef struct {
    const oracle_dims* d;
    unsigned flags;
    const double* xbc;      /* [B,S,Cdim] post-conv, Cdim = H*P + 2*G*N      */
    const double* dt_raw;   /* [B,S,H]                                       */
    const double* dt_bias;  /* [H] or NULL                                   */
    const double* A;        /* [H]                                           */
    const double* D;        /* [H] or NULL                                   */
    const double* z;        /* [B,S,H*P], used iff ORACLE_HAS_Z              */
    const double* h0;       /* [B,H,P,N] or NULL = zeros                     */
    double* y;              /* [B,S,H,P]                                     */
    double* hS;             /* [B,H,P,N]                                     */
    const int* chunk_lens;  /* chunked form only: partition of S             */
    int nchunks;
} oracle_scan_args;

/* Column of x / B / C in the post-conv stream: x | B | C ([VLC] summary;
 * [TS] section 4.1: xBC carries dInner + 2*nGroup*dState values). */
static size_t col_x(const oracle_dims* d, int h, int p) { return (size_t)h * d->headdim + p; }
static size_t col_B(const oracle_dims* d, int g, int n)
{
    return (size_t)d->nheads * d->headdim + (size_t)g * d->dstate + n;
}
static size_t col_C(const oracle_dims* d, int g, int n)
{
    return (size_t)d->nheads * d->headdim + (size_t)d->ngroups * d->dstate +
           (size_t)g * d->dstate + n;
}

static double dt_of(const oracle_scan_args* a, int b, int t, int h)
{
    const oracle_dims* d = a->d;
    double v = a->dt_raw[((size_t)b * d->seqlen + t) * d->nheads + h];
    if (a->flags & ORACLE_DT_SOFTPLUS) {
        if (a->dt_bias && ORACLE_MUTANT != 5) v += a->dt_bias[h];
        return oracle_softplus(v);
    }
    return v;
}

static void gate_and_store(const oracle_scan_args* a, int b, int t, int h, int p, double yv)
{
    const oracle_dims* d = a->d;
    if (a->flags & ORACLE_HAS_Z) {
        double zv = a->z[((size_t)b * d->seqlen + t) * ((size_t)d->nheads * d->headdim) +
                         (size_t)h * d->headdim + p];
        yv = yv * oracle_silu(zv);
    }
    a->y[(((size_t)b * d->seqlen + t) * d->nheads + h) * d->headdim + p] = yv;
}

/*
 * The recurrence, one row at a time ([TS] section 4.1):
 *   dA = exp(dt * A_h)
 *   state[p,n] = dA * state[p,n] + dt * x[p] * B[g,n]
 *   y[p] = sum_n state[p,n] * C[g,n]  +  D_h * x[p]
 * with g = h / (H/G) ([VLC] summary, group mapping).
 * This is the definition the GPU path is held to.
 */
static void seq_one(const oracle_scan_args* a, int b, int h, double* st)
{
    const oracle_dims* d = a->d;
    const int S = d->seqlen, H = d->nheads, P = d->headdim, N = d->dstate, G = d->ngroups;
    const size_t Cdim = (size_t)H * P + 2 * (size_t)G * N;
    const int g = ORACLE_MUTANT == 1 ? (h / (H / G) < 1 ? h / (H / G) : 1) : h / (H / G);
    const size_t PN = (size_t)P * N;
    const size_t sbase = ((size_t)b * H + h) * PN;
    for (size_t i = 0; i < PN; ++i) st[i] = a->h0 ? a->h0[sbase + i] : 0.0;
    for (int t = 0; t < S; ++t) {
        const double* row = a->xbc + ((size_t)b * S + t) * Cdim;
        const double dt = dt_of(a, b, t, h);
        const double dA = exp(dt * a->A[h]);
        for (int p = 0; p < P; ++p) {
            const double xp = row[col_x(d, h, p)];
            double yv = 0.0;
            for (int n = 0; n < N; ++n) {
                double s = dA * st[(size_t)p * N + n] + dt * xp * row[col_B(d, g, n)];
                if (ORACLE_MUTANT == 2) yv += st[(size_t)p * N + n] * row[col_C(d, g, n)];
                st[(size_t)p * N + n] = s;
                if (ORACLE_MUTANT != 2) yv += s * row[col_C(d, g, n)];
            }
            if (a->D) yv += a->D[h] * xp;
            gate_and_store(a, b, t, h, p, yv);
        }
    }
    for (size_t i = 0; i < PN; ++i) a->hS[sbase + i] = st[i];
}

/*
 * The chunk form ([TRT] Implementation), brute force, for a given partition
 * of the S rows.  Within a chunk of rows [r0, r0+L) with carried state h:
 *   a_t = dt_t * A_h,   gamma_t = sum_{i<=t} a_i        (i, t inside chunk)
 *   y_t = sum_{s<=t} (C_t . B_s) exp(min(gamma_t - gamma_s, 0)) dt_s x_s
 *         + exp(min(gamma_t, 0)) (C_t . h)  +  D x_t
 *   h  <- exp(min(gamma_L, 0)) h + sum_s exp(min(gamma_L - gamma_s, 0)) dt_s x_s B_s^T
 * gamma_L is the last element of the cumulative sum, not a separate sum.
 * No step of the recurrence above is used here.
 */
/* exp of the clamped exponent gamma_t - gamma_s of the chunk form ([TRT]
 * Implementation: every exponent is at most 0). */
static double decay_of(double gt, double gs)
{
    if (ORACLE_MUTANT == 12) return exp((gt < 0.0 ? gt : 0.0) - (gs < 0.0 ? gs : 0.0));
    double e = gt - gs;
    if (e > 0.0 && ORACLE_MUTANT != 10) e = 0.0;
    return exp(e);
}

static void chunked_one(const oracle_scan_args* a, int b, int h, double* st, double* gam,
                        double* dts, double* st_next)
{
    const oracle_dims* d = a->d;
    const int S = d->seqlen, H = d->nheads, P = d->headdim, N = d->dstate, G = d->ngroups;
    const size_t Cdim = (size_t)H * P + 2 * (size_t)G * N;
    const int g = h / (H / G);
    const size_t PN = (size_t)P * N;
    const size_t sbase = ((size_t)b * H + h) * PN;
    for (size_t i = 0; i < PN; ++i) st[i] = a->h0 ? a->h0[sbase + i] : 0.0;
    int r0 = 0;
    for (int c = 0; c < a->nchunks; ++c) {
        const int L = a->chunk_lens[c];
        double run = 0.0;
        for (int t = 0; t < L; ++t) {
            dts[t] = dt_of(a, b, r0 + t, h);
            run += dts[t] * (ORACLE_MUTANT == 6 ? -a->A[h] : a->A[h]);
            gam[t] = run;
        }
        for (int t = 0; t < L; ++t) {
            const double* rt = a->xbc + ((size_t)b * S + r0 + t) * Cdim;
            for (int p = 0; p < P; ++p) {
                double yv = 0.0;
                for (int s = 0; s <= t; ++s) {
                    const double* rs = a->xbc + ((size_t)b * S + r0 + s) * Cdim;
                    double cb = 0.0;
                    for (int n = 0; n < N; ++n) cb += rt[col_C(d, g, n)] * rs[col_B(d, g, n)];
                    yv += cb * decay_of(gam[t], gam[s]) * dts[s] * rs[col_x(d, h, p)];
                }
                double ch = 0.0;
                for (int n = 0; n < N; ++n) ch += rt[col_C(d, g, n)] * st[(size_t)p * N + n];
                yv += decay_of(gam[t], 0.0) * ch;
                if (a->D) yv += a->D[h] * rt[col_x(d, h, p)];
                gate_and_store(a, b, r0 + t, h, p, yv);
            }
        }
        double gL = gam[L - 1];
        if (ORACLE_MUTANT == 11) {
            float r = 0.0f;
            for (int s = L - 1; s >= 0; --s) r += (float)(dts[s] * a->A[h]);
            gL = (double)r;
        }
        const double eL = decay_of(gL, 0.0);
        for (int p = 0; p < P; ++p)
            for (int n = 0; n < N; ++n) {
                double acc = eL * st[(size_t)p * N + n];
                for (int s = 0; s < L; ++s) {
                    const double* rs = a->xbc + ((size_t)b * S + r0 + s) * Cdim;
                    const double w = ORACLE_MUTANT == 11 ? exp(gL - gam[s]) : decay_of(gL, gam[s]);
                    acc += w * dts[s] * rs[col_x(d, h, p)] * rs[col_B(d, g, n)];
                }
                st_next[(size_t)p * N + n] = acc;
            }
        if (ORACLE_MUTANT == 3) memset(st_next, 0, sizeof(double) * PN);
        memcpy(st, st_next, sizeof(double) * PN);
        r0 += L;
    }
    for (size_t i = 0; i < PN; ++i) a->hS[sbase + i] = st[i];
}

/* ------------------------------------------------------------------------ */
/* Work split over independent (sequence, head) pairs.  Only the order in   */
/* which independent pairs are visited changes; each pair runs as above.    */

typedef struct {
    const oracle_scan_args* a;
    int chunked;
    int first, step, total;
} oracle_worker;

static void* oracle_worker_main(void* arg)
{
    oracle_worker* w = (oracle_worker*)arg;
    const oracle_dims* d = w->a->d;
    const size_t PN = (size_t)d->headdim * d->dstate;
    double* st = (double*)malloc(sizeof(double) * PN);
    double* st2 = (double*)malloc(sizeof(double) * PN);
    double* gam = (double*)malloc(sizeof(double) * (size_t)(d->seqlen > 0 ? d->seqlen : 1));
    double* dts = (double*)malloc(sizeof(double) * (size_t)(d->seqlen > 0 ? d->seqlen : 1));
    for (int u = w->first; u < w->total; u += w->step) {
        int b = u / d->nheads, h = u % d->nheads;
        if (w->chunked) chunked_one(w->a, b, h, st, gam, dts, st2);
        else seq_one(w->a, b, h, st);
    }
    free(st); free(st2); free(gam); free(dts);
    return NULL;
}

static int run_pairs(const oracle_scan_args* a, int chunked, int nthreads)
{
    const oracle_dims* d = a->d;
    if (d->batch < 0 || d->seqlen < 0 || d->nheads <= 0 || d->headdim <= 0 ||
        d->dstate <= 0 || d->ngroups <= 0 || d->nheads % d->ngroups != 0)
        return -1;
    const int total = d->batch * d->nheads;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > total) nthreads = total > 0 ? total : 1;
    oracle_worker* ws = (oracle_worker*)calloc((size_t)nthreads, sizeof(oracle_worker));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int i = 0; i < nthreads; ++i) {
        ws[i].a = a; ws[i].chunked = chunked;
        ws[i].first = i; ws[i].step = nthreads; ws[i].total = total;
    }
    if (nthreads == 1) {
        oracle_worker_main(&ws[0]);
    } else {
        for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, oracle_worker_main, &ws[i]);
        for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    }
    free(ws); free(th);
    return 0;
}

/* Sequential recurrence over all rows (the definition). */
int oracle_ssd_sequential(const oracle_dims* d, unsigned flags, const double* xbc,
                          const double* dt_raw, const double* dt_bias, const double* A,
                          const double* D, const double* z, const double* h0,
                          double* y, double* hS, int nthreads)
{
    oracle_scan_args a = {d, flags, xbc, dt_raw, dt_bias, A, D, z, h0, y, hS, NULL, 0};
    return run_pairs(&a, 0, nthreads);
}

/* Brute-force chunk form over the partition chunk_lens[0..nchunks) of S. */
int oracle_ssd_chunked(const oracle_dims* d, unsigned flags, const double* xbc,
                       const double* dt_raw, const double* dt_bias, const double* A,
                       const double* D, const double* z, const double* h0,
                       double* y, double* hS, const int* chunk_lens, int nchunks,
                       int nthreads)
{
    long tot = 0;
    for (int c = 0; c < nchunks; ++c) {
        if (chunk_lens[c] <= 0) return -1;
        tot += chunk_lens[c];
    }
    if (tot != d->seqlen) return -1;
    oracle_scan_args a = {d, flags, xbc, dt_raw, dt_bias, A, D, z, h0, y, hS, chunk_lens, nchunks};
    return run_pairs(&a, 1, nthreads);
}

/*
 * Slot-indexed single-step decode ([VLC] summary: the state update runs at
 * the state slot, in place; [TS] section 11: per-slot SSM state pool).
 * Row i continues the sequence whose state lives in pool[slot_ids[i]]:
 *   gather -> one step of the recurrence above -> scatter back.
 * xbc is post-conv [R, Cdim].  Returns -1 (and writes nothing for that row)
 * when a slot id is out of range; rows are otherwise independent.
 */
int oracle_decode_step(int R, int H, int P, int N, int G, unsigned flags,
                       const double* xbc, const double* dt_raw, const double* dt_bias,
                       const double* A, const double* D, const double* z,
                       const int32_t* slot_ids, int num_slots, double* pool, double* y)
{
    oracle_dims d = {R, 1, H, P, N, G};
    const size_t PN = (size_t)P * N;
    double* h0 = (double*)malloc(sizeof(double) * (size_t)H * PN);
    double* h1 = (double*)malloc(sizeof(double) * (size_t)H * PN);
    const size_t Cdim = (size_t)H * P + 2 * (size_t)G * N;
    int rc = 0;
    for (int i = 0; i < R; ++i) {
        int s = slot_ids[i];
        if (s < 0 || s >= num_slots) { rc = -1; continue; }
        memcpy(h0, pool + (size_t)s * H * PN, sizeof(double) * (size_t)H * PN);
        oracle_dims d1 = d; d1.batch = 1;
        oracle_scan_args a = {&d1, flags, xbc + (size_t)i * Cdim, dt_raw + (size_t)i * H,
                              dt_bias, A, D, z ? z + (size_t)i * H * P : NULL, h0,
                              y + (size_t)i * H * P, h1, NULL, 0};
        for (int h = 0; h < H; ++h) {
            double* st = (double*)malloc(sizeof(double) * PN);
            seq_one(&a, 0, h, st);
            free(st);
        }
        memcpy(pool + (size_t)s * H * PN, h1, sizeof(double) * (size_t)H * PN);
    }
    free(h0); free(h1);
    return rc;
}

/*
 * Group RMSNorm of y, then the SiLU gate.  [TS] section 3 (Mamba2 branch:
 * out = SiLU(z) * GroupRMSNorm(y), ssm_norm.weight), section 4.1 (the group
 * norm normalises y per group before the gate SiLU(z) multiplies), section 6
 * (ssm_norm.weight, one weight per channel of dInner).  rows x C values;
 * group g holds the C / G contiguous channels g*C/G .. (g+1)*C/G - 1.
 *
 *   ms_g     = (1 / (C/G)) * sum_{c in g} y[r,c]^2
 *   out[r,c] = silu(z[r,c]) * (y[r,c] / sqrt(ms_g + eps)) * w[c]
 */
void oracle_gated_group_rmsnorm(long rows, int C, int G, double eps, const double* y,
                                const double* z, const double* w, double* out)
{
    const int gs = C / G;
    for (long r = 0; r < rows; ++r) {
        const double* yr = y + (size_t)r * C;
        const double* zr = z + (size_t)r * C;
        double* o = out + (size_t)r * C;
        for (int g = 0; g < G; ++g) {
            /* mutant 7: one norm over the whole row instead of per group */
            const int c0 = ORACLE_MUTANT == 7 ? 0 : g * gs;
            const int n = ORACLE_MUTANT == 7 ? C : gs;
            double ss = 0.0;
            for (int c = c0; c < c0 + n; ++c) {
                double v = yr[c];
                if (ORACLE_MUTANT == 9) v *= oracle_silu(zr[c]); /* gate before the norm */
                ss += v * v;
            }
            const double ms = ss / n;
            /* mutant 8: eps added outside the square root */
            const double inv = ORACLE_MUTANT == 8 ? 1.0 / (sqrt(ms) + eps) : 1.0 / sqrt(ms + eps);
            for (int c = g * gs; c < (g + 1) * gs; ++c)
                o[c] = oracle_silu(zr[c]) * (yr[c] * inv) * w[c];
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Sequence-parallel state passing: the rows of a sequence split into       */
/* consecutive segments, each scanned from a zero state, then chained.      */

/*
 * The total decay of a segment, per (sequence, head): the last element of
 * the cumulative sum gamma_t = sum_{i<=t} dt_i A_h over the segment's rows
 * ([TRT] Implementation, where gamma of a chunk is that cumulative sum and
 * its last element carries the state to the next chunk).
 *   gamma[b,h] = sum_{t=0}^{S-1} dt[b,t,h] * A[h]
 * with dt = softplus(dt_raw + dt_bias) under ORACLE_DT_SOFTPLUS, else dt_raw.
 */
void oracle_segment_decay(int B, int S, int H, unsigned flags, const double* dt_raw,
                          const double* dt_bias, const double* A, double* gamma)
{
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            double g = 0.0;
            for (int t = 0; t < S; ++t) {
                double v = dt_raw[((size_t)b * S + t) * H + h];
                if (flags & ORACLE_DT_SOFTPLUS) {
                    if (dt_bias && ORACLE_MUTANT != 5) v += dt_bias[h];
                    v = oracle_softplus(v);
                }
                g += v * A[h];
            }
            gamma[(size_t)b * H + h] = g;
        }
}

/*
 * The state after two consecutive segments: the first one's final state
 * h_prev decays through the second segment, whose own contribution h_seg is
 * its final state from a zero start ([TRT] Implementation: the chunk form's
 * carry h <- exp(min(gamma_L, 0)) h + (the chunk's terms), applied with the
 * second segment as the chunk).
 *   out[b,h,:,:] = exp(min(gamma[b,h], 0)) * h_prev[b,h,:,:] + h_seg[b,h,:,:]
 * h_prev NULL means zeros.
 */
void oracle_state_combine(int BH, long PN, const double* gamma, const double* h_prev,
                          const double* h_seg, double* out)
{
    for (int i = 0; i < BH; ++i) {
        const double e = ORACLE_MUTANT == 13 ? 1.0 : exp(gamma[i] < 0.0 ? gamma[i] : 0.0);
        for (long k = 0; k < PN; ++k) {
            const size_t j = (size_t)i * PN + k;
            out[j] = (h_prev ? e * h_prev[j] : 0.0) + h_seg[j];
        }
    }
}

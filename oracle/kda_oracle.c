/*
 * KDA recurrence oracle: plain, slow, sequential fp64 CPU code.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path includes, links or
 * calls this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no header, helper or constant with the
 * CUDA library.
 *
 * What it computes (the Kimi Delta Attention recurrence, the gated delta rule
 * with one decay per key channel).  The step list and its order follow
 * "Ascend day-0 support for Kimi K3" (hwcomputing.csdn.net/6a695b59...),
 * section "Fused-operator acceleration: KDA Prefill and Decode dual path",
 * paragraph on the decode kernel: Q/K L2Norm, gate and beta processing,
 * state decay, delta rule, outer-product update, output, in-place write-back
 * of the final state.  The state is the V x K matrix named there (rows are
 * value channels, the key channel is the fast index).  Per token:
 *
 *   q^ = q / sqrt(sum q^2 + eps),  k^ = k / sqrt(sum k^2 + eps)
 *   alpha_c = exp(g_c) (one per key channel),  beta = 1 / (1 + exp(-b))
 *   S'   = S diag(alpha)                      (column c scaled by alpha_c)
 *   u    = beta (v - S' k^)                   (delta rule)
 *   S    = S' + u k^T                         (outer-product update)
 *   o    = scale * S q^                       (output on the updated state)
 *
 * The record/replay pair follows "2.8x faster Kimi K3 inference on CANN"
 * (hwcomputing.csdn.net/6ac7907e...), section 04 "ReplaySSM": verification
 * keeps only the per-token update records, and the commit replays the
 * accepted records in order onto the committed state.  The prefill variant
 * is the same recurrence over every token of a sequence (the chunked form is
 * a re-association of this loop, checked separately).
 *
 * Slot convention shared with the library's documented semantics: a negative
 * slot id is padding (output zero, no state access); a slot id >= num_slots
 * is an error (output zero, no state access, counted in the return value).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- one token of the recurrence on one (sequence, head) state ---------- */

/* x_hat = x / sqrt(sum x^2 + eps) */
static void l2norm(int d, const double *x, double eps, double *out)
{
    double ss = 0.0;
    for (int c = 0; c < d; ++c) ss += x[c] * x[c];
    double den = sqrt(ss + eps);
    for (int c = 0; c < d; ++c) out[c] = x[c] / den;
}

static double sigmoid(double b) { return 1.0 / (1.0 + exp(-b)); }

/*
 * Applies one token to S ([dv][dk], row-major).  q may be NULL (no output is
 * produced then).  If khat_out/beta_out are non-NULL, the update record the
 * token used is stored there.
 */
static void kda_token(int dk, int dv, double *S, const double *q,
                      const double *k, const double *v, const double *g,
                      double b, double eps, double scale, double *o,
                      double *khat_out, double *beta_out)
{
    double *kh = (double *)malloc(sizeof(double) * (size_t)dk * 3);
    double *qh = kh + dk;
    double *alpha = kh + 2 * dk;

    /* Q/K L2Norm */
    l2norm(dk, k, eps, kh);
    if (q) l2norm(dk, q, eps, qh);
    /* gate and beta processing */
    for (int c = 0; c < dk; ++c) alpha[c] = exp(g[c]);
    double beta = sigmoid(b);
    /* state decay: S' = S diag(alpha) */
    for (int i = 0; i < dv; ++i)
        for (int c = 0; c < dk; ++c) S[(size_t)i * dk + c] *= alpha[c];
    /* delta rule and outer-product update, row by row */
    for (int i = 0; i < dv; ++i) {
        double *s = S + (size_t)i * dk;
        double r = 0.0;
        for (int c = 0; c < dk; ++c) r += s[c] * kh[c];
        double u = beta * (v[i] - r);
        for (int c = 0; c < dk; ++c) s[c] += u * kh[c];
    }
    /* output on the updated state */
    if (q && o) {
        for (int i = 0; i < dv; ++i) {
            const double *s = S + (size_t)i * dk;
            double acc = 0.0;
            for (int c = 0; c < dk; ++c) acc += s[c] * qh[c];
            o[i] = scale * acc;
        }
    }
    if (khat_out) memcpy(khat_out, kh, sizeof(double) * (size_t)dk);
    if (beta_out) *beta_out = beta;
    free(kh);
}

/* One record replayed: S = S diag(exp g); S = S + beta (v - S k^) k^T. */
static void kda_apply_record(int dk, int dv, double *S, const double *khat,
                             const double *v, const double *g, double beta)
{
    for (int i = 0; i < dv; ++i) {
        double *s = S + (size_t)i * dk;
        for (int c = 0; c < dk; ++c) s[c] *= exp(g[c]);
        double r = 0.0;
        for (int c = 0; c < dk; ++c) r += s[c] * khat[c];
        double u = beta * (v[i] - r);
        for (int c = 0; c < dk; ++c) s[c] += u * khat[c];
    }
}

static int slot_state(int32_t slot, int64_t num_slots)
{
    if (slot < 0) return 0;           /* padding */
    if ((int64_t)slot >= num_slots) return -1; /* error */
    return 1;
}

int kda_oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* ---- recurrence over a run of tokens for one (sequence, head) ----------- */

/*
 * n tokens; token t of this (sequence, head) lives at q + t*tok_stride_k etc.
 * S is [dv][dk] in/out.  o (may be NULL) receives [n] rows at o + t*tok_stride_v.
 */
void kda_oracle_recurrence(int dk, int dv, int64_t n,
                           const double *q, const double *k, const double *v,
                           const double *g, const double *b,
                           int64_t tok_stride_k, int64_t tok_stride_v,
                           int64_t tok_stride_b, double eps, double scale,
                           double *S, double *o)
{
    for (int64_t t = 0; t < n; ++t)
        kda_token(dk, dv, S, q ? q + t * tok_stride_k : NULL,
                  k + t * tok_stride_k, v + t * tok_stride_v,
                  g + t * tok_stride_k, b[t * tok_stride_b], eps, scale,
                  o ? o + t * tok_stride_v : NULL, NULL, NULL);
}

/* ---- decode: one token per sequence over the state pool ----------------- */
/*
 * q,k,g [B][H][dk]; v [B][H][dv]; b [B][H]; slot_ids [B];
 * pool [num_slots][H][dv][dk] (updated in place); out [B][H][dv].
 * Returns the number of (sequence, head) items with an out-of-range slot.
 */
int64_t kda_oracle_decode(int B, int H, int dk, int dv, const double *q,
                          const double *k, const double *v, const double *g,
                          const double *b, const int32_t *slot_ids,
                          double *pool, int64_t num_slots, double eps,
                          double scale, double *out)
{
    int64_t errors = 0;
    int64_t items = (int64_t)B * H;
#pragma omp parallel for schedule(dynamic) reduction(+ : errors)
    for (int64_t it = 0; it < items; ++it) {
        int n = (int)(it / H), h = (int)(it % H);
        double *o = out + it * dv;
        int st = slot_state(slot_ids[n], num_slots);
        if (st <= 0) {
            for (int i = 0; i < dv; ++i) o[i] = 0.0;
            if (st < 0) errors += 1;
            continue;
        }
        double *S = pool + ((int64_t)slot_ids[n] * H + h) * dv * dk;
        kda_token(dk, dv, S, q + it * dk, k + it * dk, v + it * dv,
                  g + it * dk, b[it], eps, scale, o, NULL, NULL);
    }
    return errors;
}

/* ---- speculative verify: D draft tokens, records kept, pool untouched ---- */
/*
 * q,k,g [B][D][H][dk]; v [B][D][H][dv]; b [B][D][H]; pool read only.
 * out [B][D][H][dv]; records: khat [B][D][H][dk], vrec [B][D][H][dv],
 * grec [B][D][H][dk], beta [B][D][H].
 */
int64_t kda_oracle_verify(int B, int D, int H, int dk, int dv,
                          const double *q, const double *k, const double *v,
                          const double *g, const double *b,
                          const int32_t *slot_ids, const double *pool,
                          int64_t num_slots, double eps, double scale,
                          double *out, double *khat, double *vrec,
                          double *grec, double *beta)
{
    int64_t errors = 0;
    int64_t items = (int64_t)B * H;
#pragma omp parallel for schedule(dynamic) reduction(+ : errors)
    for (int64_t it = 0; it < items; ++it) {
        int n = (int)(it / H), h = (int)(it % H);
        int st = slot_state(slot_ids[n], num_slots);
        double *S = (double *)malloc(sizeof(double) * (size_t)dv * dk);
        if (st > 0)
            memcpy(S, pool + ((int64_t)slot_ids[n] * H + h) * dv * dk,
                   sizeof(double) * (size_t)dv * dk);
        else if (st < 0)
            errors += 1;
        for (int j = 0; j < D; ++j) {
            int64_t tk = (((int64_t)n * D + j) * H + h);
            double *o = out + tk * dv;
            /* the record always holds the token's inputs, padding or not */
            l2norm(dk, k + tk * dk, eps, khat + tk * dk);
            memcpy(vrec + tk * dv, v + tk * dv, sizeof(double) * (size_t)dv);
            memcpy(grec + tk * dk, g + tk * dk, sizeof(double) * (size_t)dk);
            beta[tk] = sigmoid(b[tk]);
            if (st <= 0) {
                for (int i = 0; i < dv; ++i) o[i] = 0.0;
                continue;
            }
            kda_token(dk, dv, S, q + tk * dk, k + tk * dk, v + tk * dv,
                      g + tk * dk, b[tk], eps, scale, o, NULL, NULL);
        }
        free(S);
    }
    return errors;
}

/* ---- commit: replay the first a_n records onto the committed state ------ */
/*
 * Records as written by kda_oracle_verify; num_accepted [B] in 0..D.
 * Returns the number of (sequence, head) items rejected (slot out of range,
 * or a_n outside 0..D); those leave the pool untouched.
 */
int64_t kda_oracle_replay(int B, int D, int H, int dk, int dv,
                          const double *khat, const double *vrec,
                          const double *grec, const double *beta,
                          const int32_t *num_accepted,
                          const int32_t *slot_ids, double *pool,
                          int64_t num_slots)
{
    int64_t errors = 0;
    int64_t items = (int64_t)B * H;
#pragma omp parallel for schedule(dynamic) reduction(+ : errors)
    for (int64_t it = 0; it < items; ++it) {
        int n = (int)(it / H), h = (int)(it % H);
        int a = num_accepted[n];
        int st = slot_state(slot_ids[n], num_slots);
        if (a < 0 || a > D) { errors += 1; continue; }
        if (st < 0) { errors += 1; continue; }
        if (st == 0 || a == 0) continue;
        double *S = pool + ((int64_t)slot_ids[n] * H + h) * dv * dk;
        for (int j = 0; j < a; ++j) {
            int64_t tk = (((int64_t)n * D + j) * H + h);
            kda_apply_record(dk, dv, S, khat + tk * dk, vrec + tk * dv,
                             grec + tk * dk, beta[tk]);
        }
    }
    return errors;
}

/* ---- prefill: every token of each sequence, final state to its slot ----- */
/*
 * Variable-length batch: sequence s covers tokens cu_seqlens[s] ..
 * cu_seqlens[s+1]-1.  q,k,g [T][H][dk]; v [T][H][dv]; b [T][H];
 * out [T][H][dv].  The initial state is the slot's state when
 * init_from_pool != 0, else zero; the final state is written to the slot.
 * Padding sequences (slot < 0) produce zero outputs and touch no state.
 */
int64_t kda_oracle_prefill(int num_seqs, const int64_t *cu_seqlens, int H,
                           int dk, int dv, const double *q, const double *k,
                           const double *v, const double *g, const double *b,
                           const int32_t *slot_ids, double *pool,
                           int64_t num_slots, int init_from_pool, double eps,
                           double scale, double *out)
{
    int64_t errors = 0;
    int64_t items = (int64_t)num_seqs * H;
#pragma omp parallel for schedule(dynamic) reduction(+ : errors)
    for (int64_t it = 0; it < items; ++it) {
        int s = (int)(it / H), h = (int)(it % H);
        int64_t t0 = cu_seqlens[s], t1 = cu_seqlens[s + 1];
        int st = slot_state(slot_ids[s], num_slots);
        if (st <= 0) {
            for (int64_t t = t0; t < t1; ++t)
                for (int i = 0; i < dv; ++i) out[(t * H + h) * dv + i] = 0.0;
            if (st < 0) errors += 1;
            continue;
        }
        double *slot = pool + ((int64_t)slot_ids[s] * H + h) * dv * dk;
        double *S = (double *)calloc((size_t)dv * dk, sizeof(double));
        if (init_from_pool) memcpy(S, slot, sizeof(double) * (size_t)dv * dk);
        kda_oracle_recurrence(dk, dv, t1 - t0, q + (t0 * H + h) * dk,
                              k + (t0 * H + h) * dk, v + (t0 * H + h) * dv,
                              g + (t0 * H + h) * dk, b + (t0 * H + h),
                              (int64_t)H * dk, (int64_t)H * dv, H, eps, scale,
                              S, out + (t0 * H + h) * dv);
        memcpy(slot, S, sizeof(double) * (size_t)dv * dk);
        free(S);
    }
    return errors;
}

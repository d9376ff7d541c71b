/*
 * gdn_oracle.c -- float64 CPU oracle for the GatedDeltaNet record / replay
 * step and the tiled GQA repeat.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct
 * statement of what the GPU path computes.  Only the test-suite, the smoke
 * check and the benchmark's CPU-baseline leg may build or call it; the
 * product path never does.  It shares no code, header or table with the CUDA
 * library.
 *
 * Sources (page titles as printed):
 *   [P1] "metaltile-std 0.1.0 -- src/ffai/gated_delta_replay.rs":
 *        module doc (tape layout, replay rule), kernel
 *        gated_delta_step_record (record), kernel state_replay (replay).
 *   [P3] "mlx-native 0.6.5 -- ops/repeat_tiled.rs": module doc (mapping
 *        dst[t,h,k] = src[t,h%Hg,k]) and dispatch_repeat_tiled_f32.
 *
 * Every value is float64.  Inputs are the exact values the GPU sees (bf16 /
 * f16 / f32 storage widened without rounding by the caller); outputs are
 * unrounded float64.  Loops follow the page kernels: one independent state
 * row s[Dk] per (b, hv, dv), the timestep loop inside it.  The only
 * parallelism is an OpenMP loop over the independent (b, hv) pairs.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (no FMA
 * contraction, so results do not depend on the host ISA).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int gdn_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void gdn_oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Record [P1, kernel gated_delta_step_record].
 *
 * For every row (b, hv, dv) and for t = 0 .. T-1 whose mask is on
 * (mask == NULL means every step is on), with the key head
 *     hk = hv / (Hv / Hk)   block GQA mapping (the record kernel's own rule),
 *     hk = hv % Hk          tiled mapping when tiled_gqa != 0 ("mlx-native
 *                           repeat_tiled.rs", module doc "Mapping": the head
 *                           order of a tiled repeat, read in place):
 *     s      <- g[b,t,hv] * s
 *     kv      = sum_i s[i] * k[b,t,hk,i]
 *     delta   = (v[b,t,hv,dv] - kv) * beta[b,t,hv]
 *     delta_log[b,t,hv,dv] = delta
 *     s      <- s + k[b,t,hk,:] * delta
 *     y[b,t,hv,dv] = sum_i s[i] * q[b,t,hk,i]
 * A step whose mask is 0 writes nothing and leaves s unchanged.
 * state_out[b,hv,dv,:] = s after the last step.
 *
 * Tape capture (module doc: k_log [B,T,Hv,Dk] "GQA-expanded", g_log
 * [B,T,Hv]): when k_log / g_log are non-NULL they receive k[b,t,hk,:] (hk by
 * the same mapping) and
 * g[b,t,hv] at exactly the (b,t,hv) positions where delta_log is written.
 *
 * Layouts (row-major): q,k [B,T,Hk,Dk]; v,y,delta_log [B,T,Hv,Dv];
 * g,beta,g_log [B,T,Hv]; k_log [B,T,Hv,Dk]; state [B,Hv,Dv,Dk]; mask [B,T].
 */
void gdn_oracle_record(int64_t B, int64_t T, int64_t Hk, int64_t Hv,
                       int64_t Dk, int64_t Dv, int64_t tiled_gqa,
                       const double *q, const double *k, const double *v,
                       const double *g, const double *beta,
                       const double *state_in, const uint32_t *mask,
                       double *y, double *state_out, double *delta_log,
                       double *k_log, double *g_log)
{
    const int64_t group = Hv / Hk;
    int64_t n;
#pragma omp parallel for schedule(dynamic, 1)
    for (n = 0; n < B * Hv; ++n) {
        const int64_t b = n / Hv;
        const int64_t hv = n % Hv;
        const int64_t hk = tiled_gqa ? hv % Hk : hv / group;
        double *s = (double *)malloc((size_t)Dk * sizeof(double));
        for (int64_t dv = 0; dv < Dv; ++dv) {
            const double *row_in = state_in + (n * Dv + dv) * Dk;
            for (int64_t i = 0; i < Dk; ++i) s[i] = row_in[i];
            for (int64_t t = 0; t < T; ++t) {
                const uint32_t m = mask ? mask[b * T + t] : 1u;
                if (m == 0) continue;
                const double *kt = k + ((b * T + t) * Hk + hk) * Dk;
                const double *qt = q + ((b * T + t) * Hk + hk) * Dk;
                const int64_t gb = (b * T + t) * Hv + hv;
                const int64_t vi = ((b * T + t) * Hv + hv) * Dv + dv;
                const double gt = g[gb];
                const double bt = beta[gb];
                double kv = 0.0;
                for (int64_t i = 0; i < Dk; ++i) {
                    s[i] = s[i] * gt;
                    kv += s[i] * kt[i];
                }
                const double delta = (v[vi] - kv) * bt;
                delta_log[vi] = delta;
                double out = 0.0;
                for (int64_t i = 0; i < Dk; ++i) {
                    s[i] = s[i] + kt[i] * delta;
                    out += s[i] * qt[i];
                }
                y[vi] = out;
            }
            double *row_out = state_out + (n * Dv + dv) * Dk;
            for (int64_t i = 0; i < Dk; ++i) row_out[i] = s[i];
        }
        free(s);
        if (k_log || g_log) {
            for (int64_t t = 0; t < T; ++t) {
                const uint32_t m = mask ? mask[b * T + t] : 1u;
                if (m == 0) continue;
                const int64_t gb = (b * T + t) * Hv + hv;
                if (g_log) g_log[gb] = g[gb];
                if (k_log) {
                    const double *kt = k + ((b * T + t) * Hk + hk) * Dk;
                    double *kl = k_log + gb * Dk;
                    for (int64_t i = 0; i < Dk; ++i) kl[i] = kt[i];
                }
            }
        }
    }
}

/*
 * Replay [P1, module doc and kernel state_replay].
 *
 * Re-folds the accepted prefix of the tape onto a snapshot.  For every row
 * (b, hv, dv) and t = 0 .. T-1:
 *     do_step = (t < accepted) && mask[b,t] != 0      (mask NULL: always on)
 *     s <- do_step ? s * g_log[b,t,hv] + k_log[b,t,hv,:] * delta_log[b,t,hv,dv]
 *                  : s
 * The selected-away branch is never evaluated here, so whatever a masked or
 * unaccepted tape slot holds (NaN included) cannot reach the state, as with
 * the page's select.  accepted >= T folds every step whose mask is on.
 *
 * Per-sequence acceptance (the module doc's speculative-decode use: each
 * sequence of the batch keeps its own accepted prefix): when
 * accepted_per_seq is non-NULL, sequence b uses accepted_per_seq[b] in place
 * of the scalar; a negative entry accepts nothing.
 */
void gdn_oracle_replay(int64_t B, int64_t T, int64_t Hv, int64_t Dk, int64_t Dv,
                       int64_t accepted, const int64_t *accepted_per_seq,
                       const double *delta_log, const double *k_log,
                       const double *g_log, const double *state_in,
                       const uint32_t *mask, double *state_out)
{
    int64_t n;
#pragma omp parallel for schedule(dynamic, 1)
    for (n = 0; n < B * Hv; ++n) {
        const int64_t b = n / Hv;
        const int64_t hv = n % Hv;
        const int64_t acc = accepted_per_seq ? accepted_per_seq[b] : accepted;
        double *s = (double *)malloc((size_t)Dk * sizeof(double));
        for (int64_t dv = 0; dv < Dv; ++dv) {
            const double *row_in = state_in + (n * Dv + dv) * Dk;
            for (int64_t i = 0; i < Dk; ++i) s[i] = row_in[i];
            for (int64_t t = 0; t < T; ++t) {
                const uint32_t m = mask ? mask[b * T + t] : 1u;
                const int do_step = (t < acc) && (m != 0);
                if (!do_step) continue;
                const int64_t gi = (b * T + t) * Hv + hv;
                const double gt = g_log[gi];
                const double d = delta_log[gi * Dv + dv];
                const double *kt = k_log + gi * Dk;
                for (int64_t i = 0; i < Dk; ++i) s[i] = s[i] * gt + kt[i] * d;
            }
            double *row_out = state_out + (n * Dv + dv) * Dk;
            for (int64_t i = 0; i < Dk; ++i) row_out[i] = s[i];
        }
        free(s);
    }
}

/*
 * Tiled GQA repeat [P3, module doc "Mapping"]:
 *     dst[t, h, x] = src[t, h % hg, x],   src [seq,hg,kdim] -> dst [seq,h,kdim]
 * A pure copy of elem_bytes-sized elements, so it is bit-exact for any dtype.
 */
void gdn_oracle_repeat_tiled(int64_t seq, int64_t hg, int64_t h, int64_t kdim,
                             int64_t elem_bytes, const void *src, void *dst)
{
    const unsigned char *s = (const unsigned char *)src;
    unsigned char *d = (unsigned char *)dst;
    for (int64_t t = 0; t < seq; ++t)
        for (int64_t hh = 0; hh < h; ++hh)
            memcpy(d + ((t * h + hh) * kdim) * elem_bytes,
                   s + ((t * hg + hh % hg) * kdim) * elem_bytes,
                   (size_t)(kdim * elem_bytes));
}

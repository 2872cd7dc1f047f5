/*
 * CPU oracle for the Mamba-2 SSD varlen forward prefill scan.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code with the CUDA path.
 *
 * What it computes is the plain per-token recurrence printed in the
 * "Per-token recurrence" section of the Modular page "mamba2_ssd_scan"
 * (Mojo module, state_space kernels), evaluated in fp64:
 *
 *   dt_t      = softplus(dt[t,h] + dt_bias[h])          (per token and head)
 *   dA_t      = exp(A[h] * dt_t)
 *   state[n] <- state[n] * dA_t + dt_t * B[t,g,n] * x[t,h,p]
 *   y[t,h,p]  = sum_n C[t,g,n] * state[n] + D[h] * x[t,h,p]
 *
 * with g = h / (nheads / ngroups) (module description, "B/C are GROUPED").
 * The state is reset at every query_start_loc boundary, or loaded from
 * ssm_pool[cache_indices[b]] when has_initial_state[b] is set, and the final
 * state of each sequence is written back into that pool slot (page
 * "Mamba2SSDChunkScanVarlenFwdInplace", description and "Tensor shapes").
 *
 * Readings where the pages leave a step open (each is listed in the design
 * notes of the repository):
 *   - softplus is the exact log(1 + e^v), evaluated as max(v,0) + log1p(e^-|v|);
 *   - with dt_softplus = 0 the bias is still added, only softplus is skipped;
 *   - no clamp of dt;
 *   - the state is updated before y_t is formed, so y_t includes token t;
 *   - empty optionals (D, dt_bias, has_initial_state) read as zero / false;
 *   - a zero-length sequence still writes its slot (the initial state, or 0);
 *   - the slot is written whether or not has_initial_state[b] is set;
 *   - the final fp64 state is rounded to fp32 (round to nearest) in the pool.
 *
 * bf16 inputs arrive as uint16 bit patterns and are widened exactly.
 * Parallelism: OpenMP over (sequence, head) pairs; each pair owns a private
 * head_dim x dstate state, so with distinct cache_indices no two pairs touch
 * the same pool bytes.  Results do not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_f64(uint16_t v)
{
    uint32_t u = ((uint32_t)v) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* softplus(v) = log(1 + exp(v)), written so that neither branch overflows. */
static double softplus_f64(double v)
{
    return fmax(v, 0.0) + log1p(exp(-fabs(v)));
}

/* Returns 0 on success, 1 on an invalid size or pointer, 2 on a bad
 * query_start_loc / cache index (nothing is written in that case). */
int ssd_oracle_varlen_fwd(
    double *y,                    /* (T, H, P) out, fp64; rows of unselected work untouched */
    float *ssm_pool,              /* (max_slots, H, P, N) in/out */
    const uint16_t *x,            /* (T, H, P) bf16 bits */
    const uint16_t *dt,           /* (T, H) bf16 bits */
    const float *A,               /* (H) */
    const uint16_t *B,            /* (T, G, N) bf16 bits */
    const uint16_t *C,            /* (T, G, N) bf16 bits */
    const float *D,               /* (H) or NULL */
    const float *dt_bias,         /* (H) or NULL */
    const int32_t *query_start_loc, /* (batch + 1) */
    const uint8_t *has_initial_state, /* (batch) or NULL */
    const uint32_t *cache_indices, /* (batch) */
    int64_t total_len, int32_t batch, int32_t nheads, int32_t head_dim,
    int32_t ngroups, int32_t dstate, int64_t max_slots, int32_t dt_softplus,
    const uint8_t *seq_select,    /* (batch) or NULL: 0 skips a sequence entirely */
    int32_t head_begin, int32_t head_end, /* heads [head_begin, head_end) are computed */
    int32_t num_threads)          /* <= 0: OpenMP default */
{
    if (!y || !ssm_pool || !x || !dt || !A || !B || !C || !query_start_loc || !cache_indices)
        return 1;
    if (total_len < 0 || batch < 0 || nheads <= 0 || head_dim <= 0 || ngroups <= 0 ||
        dstate <= 0 || max_slots < 0 || nheads % ngroups != 0)
        return 1;
    if (head_begin < 0 || head_end > nheads || head_begin > head_end)
        return 1;
    if (query_start_loc[0] != 0 || (int64_t)query_start_loc[batch] != total_len)
        return 2;
    for (int32_t b = 0; b < batch; ++b) {
        if (query_start_loc[b + 1] < query_start_loc[b])
            return 2;
        if ((int64_t)cache_indices[b] >= max_slots)
            return 2;
    }

    const int64_t H = nheads, P = head_dim, N = dstate, G = ngroups;
    const int64_t heads_per_group = H / G;
    const int64_t nh = head_end - head_begin;
    const int64_t npairs = (int64_t)batch * nh;

#ifdef _OPENMP
    if (num_threads > 0)
        omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif

#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)(P * N));
        double *Bt = (double *)malloc(sizeof(double) * (size_t)N);
        double *Ct = (double *)malloc(sizeof(double) * (size_t)N);
        double *xt = (double *)malloc(sizeof(double) * (size_t)P);

#pragma omp for schedule(dynamic, 1)
        for (int64_t pair = 0; pair < npairs; ++pair) {
            const int64_t b = pair / nh;
            const int64_t h = head_begin + pair % nh;
            if (seq_select && !seq_select[b])
                continue;
            const int64_t g = h / heads_per_group;
            const int64_t t0 = query_start_loc[b], t1 = query_start_loc[b + 1];
            const int64_t slot = cache_indices[b];
            float *slot_h = ssm_pool + ((slot * H + h) * P) * N;
            const int init = has_initial_state ? (has_initial_state[b] != 0) : 0;

            for (int64_t i = 0; i < P * N; ++i)
                S[i] = init ? (double)slot_h[i] : 0.0;

            const double bias = dt_bias ? (double)dt_bias[h] : 0.0;
            const double Dh = D ? (double)D[h] : 0.0;
            const double Ah = (double)A[h];

            for (int64_t t = t0; t < t1; ++t) {
                const double v = bf16_to_f64(dt[t * H + h]) + bias;
                const double d = dt_softplus ? softplus_f64(v) : v;
                const double dA = exp(Ah * d);
                for (int64_t n = 0; n < N; ++n) {
                    Bt[n] = bf16_to_f64(B[(t * G + g) * N + n]);
                    Ct[n] = bf16_to_f64(C[(t * G + g) * N + n]);
                }
                for (int64_t p = 0; p < P; ++p)
                    xt[p] = bf16_to_f64(x[(t * H + h) * P + p]);
                for (int64_t p = 0; p < P; ++p) {
                    double *Sp = S + p * N;
                    const double dx = d * xt[p];
                    double acc = 0.0;
                    for (int64_t n = 0; n < N; ++n) {
                        Sp[n] = Sp[n] * dA + dx * Bt[n];
                        acc += Ct[n] * Sp[n];
                    }
                    y[(t * H + h) * P + p] = acc + Dh * xt[p];
                }
            }
            for (int64_t i = 0; i < P * N; ++i)
                slot_h[i] = (float)S[i];
        }
        free(S);
        free(Bt);
        free(Ct);
        free(xt);
    }
    return 0;
}

/* The number of threads an OpenMP parallel region of this library uses. */
int ssd_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

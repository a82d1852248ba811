/* gdn_cpu_recurrence.c - fp32 per-token CPU recurrence of the gated delta rule: the
 * measured CPU baseline that the GPU forward is reported beside.
 *
 * "Exp 2026-07-13 - Linear-Attention Scans on the NPU", §4: the CPU operator that won
 * on the RK3588 steps the state token by token (no chunking, no triangular solve).
 * This is that operator written for any host: one chain per (sequence, v head), the
 * chains spread over OpenMP threads, the fp32 state [dk][dv] of a chain in a private
 * buffer.  Per token t (h = S^T, the [dk][dv] state the GPU path keeps):
 *     h <- exp(g_t) h
 *     u  = beta_t (v_t - h^T k_t)
 *     h <- h + k_t u^T
 *     o_t = h^T (scale q_t)
 * Two passes over the state per token: decay fused with the read h^T k, then the
 * rank-1 update fused with the output read.  Plain C: the inner loops run over the
 * contiguous dv index and vectorise with the compiler's default target.
 *
 * Not the oracle (that is the fp64 code under oracle/); not on the GPU path.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* q, k [rows, T, Hqk, dk]; v, o [rows, T, Hv, dv]; g, beta [rows, T, Hv]; h0, hT
 * [N, Hv, dk, dv] (h0 may be NULL for zeros, hT NULL for not written).  Without
 * cu_seqlens rows = N and every sequence has T tokens; with it (int32 [N + 1]) rows = 1
 * and sequence n spans tokens [cu[n], cu[n + 1]).  Grouped GQA map: v head hv reads
 * q/k head hv / (Hv / Hqk).  Returns 0, or -1 when a state buffer cannot be had. */
int gdn_cpu_recurrence_f32(const float* q, const float* k, const float* v, const float* g,
                           const float* beta, const float* h0, float* o, float* hT, int N, int T,
                           int Hqk, int Hv, int dk, int dv, float scale,
                           const int32_t* cu_seqlens, int threads) {
  const long long chains = (long long)N * Hv;
  int failed = 0;
  if (threads < 1) threads = 1;
#pragma omp parallel num_threads(threads) reduction(| : failed)
  {
    float* h = (float*)malloc(sizeof(float) * (size_t)dk * dv);
    float* u = (float*)malloc(sizeof(float) * (size_t)dv);
    float* acc = (float*)malloc(sizeof(float) * (size_t)dv);
    const int ok = h && u && acc;
    {
      /* every thread takes part in the loop (a worksharing loop must be met by all) */
#pragma omp for schedule(dynamic, 1)
      for (long long c = 0; c < chains; ++c) {
        if (!ok) {
          failed = 1;
          continue;
        }
        const int n = (int)(c / Hv), hv = (int)(c % Hv);
        const int hq = hv / (Hv / Hqk);
        const long long t_begin = cu_seqlens ? cu_seqlens[n] : (long long)n * T;
        const long long t_end = cu_seqlens ? cu_seqlens[n + 1] : t_begin + T;
        if (h0) memcpy(h, h0 + (size_t)c * dk * dv, sizeof(float) * (size_t)dk * dv);
        else memset(h, 0, sizeof(float) * (size_t)dk * dv);
        for (long long t = t_begin; t < t_end; ++t) {
          const float* qt = q + ((size_t)t * Hqk + hq) * dk;
          const float* kt = k + ((size_t)t * Hqk + hq) * dk;
          const float* vt = v + ((size_t)t * Hv + hv) * dv;
          float* ot = o + ((size_t)t * Hv + hv) * dv;
          const float a = expf(g[(size_t)t * Hv + hv]);
          const float b = beta[(size_t)t * Hv + hv];
          /* decay, and the read h^T k */
          for (int j = 0; j < dv; ++j) acc[j] = 0.f;
          for (int i = 0; i < dk; ++i) {
            float* hi = h + (size_t)i * dv;
            const float ki = kt[i];
            for (int j = 0; j < dv; ++j) {
              hi[j] *= a;
              acc[j] += ki * hi[j];
            }
          }
          for (int j = 0; j < dv; ++j) {
            u[j] = b * (vt[j] - acc[j]);
            acc[j] = 0.f;
          }
          /* rank-1 update, and the output read h^T q */
          for (int i = 0; i < dk; ++i) {
            float* hi = h + (size_t)i * dv;
            const float ki = kt[i], qi = scale * qt[i];
            for (int j = 0; j < dv; ++j) {
              hi[j] += ki * u[j];
              acc[j] += qi * hi[j];
            }
          }
          for (int j = 0; j < dv; ++j) ot[j] = acc[j];
        }
        if (hT) memcpy(hT + (size_t)c * dk * dv, h, sizeof(float) * (size_t)dk * dv);
      }
    }
    free(h);
    free(u);
    free(acc);
  }
  return failed ? -1 : 0;
}

/* Threads an OpenMP region would use by default (0 without OpenMP). */
int gdn_cpu_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 0;
#endif
}

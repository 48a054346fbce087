/*
 * gdn_oracle.c -- plain, slow fp64 CPU reference for the gated delta rule (the per-token
 * recurrence of gated-delta linear attention).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library under
 * softmax_attention_gb300/) may link, load or call this file; only the test suite, the
 * package smoke check and the CPU-baseline leg of the benchmark do.  It shares no code,
 * header, table or constant with the CUDA path.
 *
 * The page "perf(kernels): speed up linear-attention prefill ~2.6x" (hip-ep PR, Summary and
 * Test plan) speeds up a gated-delta chunked linear-attention prefill kernel and checks it
 * against a per-token decode oracle, but does not write the recurrence down.  The reading
 * taken is the published gated delta rule (Gated Delta Networks, Yang, Kautz and
 * Hatamizadeh, 2024), with a state S of dv rows by dk columns per value head:
 *
 *   S_t = S_{t-1} ( alpha_t ( I - beta_t k_t k_t^T ) ) + beta_t v_t k_t^T
 *   o_t = S_t ( scale * q_t )
 *
 * with alpha_t = exp(g_t) (g_t <= 0 is the log decay) and beta_t the write strength.  This
 * file evaluates exactly that, one token after another, for each (batch, value head): the
 * per-token form the page calls its oracle.  Value head h reads query/key head
 * h / (Hv / Hk) (grouped value heads).  S starts from the given initial state, or zero.
 *
 * Inputs are read in their storage type and widened exactly to fp64; every sum is a plain
 * left-to-right fp64 sum; exp is the C library's fp64 function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { GD_BF16 = 0, GD_FP16 = 1, GD_FP32 = 2, GD_FP64 = 3 };

static double gd_bf16(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE binary16 -> double from the format's definition. */
static double gd_fp16(uint16_t h) {
  int sign = (h >> 15) & 1, e = (h >> 10) & 0x1f, f = h & 0x3ff;
  double v;
  if (e == 0) v = ldexp((double)f, -24);
  else if (e == 31) v = f ? NAN : INFINITY;
  else v = ldexp((double)(1024 + f), e - 25);
  return sign ? -v : v;
}

static double gd_load(const void* base, int64_t i, int dtype) {
  switch (dtype) {
    case GD_BF16: return gd_bf16(((const uint16_t*)base)[i]);
    case GD_FP16: return gd_fp16(((const uint16_t*)base)[i]);
    case GD_FP32: return (double)((const float*)base)[i];
    default: return ((const double*)base)[i];
  }
}

/*
 * q, k [B, Hk, T, dk], v [B, Hv, T, dv] in `dtype`; g, beta [B, Hv, T] in `gb_dtype`;
 * s0 [B, Hv, dv, dk] fp64 or NULL.  Writes out [B, Hv, T, dv] and, if s_final is not NULL,
 * the state after the last token [B, Hv, dv, dk], both fp64.  Returns 0, or -1 on bad sizes.
 */
int oracle_gated_delta(const void* q, const void* k, const void* v, int dtype, const void* g,
                       const void* beta, int gb_dtype, const double* s0, int64_t B, int64_t T,
                       int64_t Hk, int64_t Hv, int64_t dk, int64_t dv, double scale,
                       double* out, double* s_final) {
  if (B < 0 || T < 0 || Hk <= 0 || Hv <= 0 || Hv % Hk != 0 || dk <= 0 || dv <= 0) return -1;
  const int64_t r = Hv / Hk;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < B * Hv; ++bh) {
    const int64_t b = bh / Hv, h = bh % Hv, hk = h / r;
    double* S = (double*)malloc(sizeof(double) * dv * dk);
    double* w = (double*)malloc(sizeof(double) * dv);
    double* kt = (double*)malloc(sizeof(double) * dk);
    double* qt = (double*)malloc(sizeof(double) * dk);
    for (int64_t i = 0; i < dv * dk; ++i) S[i] = s0 ? s0[bh * dv * dk + i] : 0.0;
    for (int64_t t = 0; t < T; ++t) {
      const int64_t qk_row = ((b * Hk + hk) * T + t) * dk;
      const int64_t v_row = ((b * Hv + h) * T + t) * dv;
      const double alpha = exp(gd_load(g, bh * T + t, gb_dtype));
      const double bt = gd_load(beta, bh * T + t, gb_dtype);
      for (int64_t j = 0; j < dk; ++j) {
        kt[j] = gd_load(k, qk_row + j, dtype);
        qt[j] = scale * gd_load(q, qk_row + j, dtype);
      }
      /* S (I - beta k k^T) = S - beta (S k) k^T */
      for (int64_t i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int64_t j = 0; j < dk; ++j) acc += S[i * dk + j] * kt[j];
        w[i] = acc;
      }
      /* S_t = alpha (S - beta w k^T) + beta v k^T */
      for (int64_t i = 0; i < dv; ++i) {
        const double vi = gd_load(v, v_row + i, dtype);
        for (int64_t j = 0; j < dk; ++j)
          S[i * dk + j] = alpha * (S[i * dk + j] - bt * w[i] * kt[j]) + bt * vi * kt[j];
      }
      /* o_t = S_t (scale q_t) */
      for (int64_t i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int64_t j = 0; j < dk; ++j) acc += S[i * dk + j] * qt[j];
        out[v_row + i] = acc;
      }
    }
    if (s_final) memcpy(s_final + bh * dv * dk, S, sizeof(double) * dv * dk);
    free(S);
    free(w);
    free(kt);
    free(qt);
  }
  return 0;
}

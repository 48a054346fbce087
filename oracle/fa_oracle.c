/*
 * fa_oracle.c -- plain, slow fp64 CPU reference for scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library under
 * softmax_attention_gb300/) may link, load or call this file; only the test suite,
 * the package smoke check and the CPU-baseline leg of the benchmark do.  It shares
 * no code, header, table or constant with the CUDA path.
 *
 * What it computes (the textbook definition of softmax attention, which the
 * FlashAttention kernels discussed in "CUDA: fix FA occupancy, optimize tile kernel"
 * (llama.cpp, first two paragraphs) and "perf: FlashAttention-3 style MLA
 * PageAttention" (flashinfer, change list) compute blockwise):
 *
 *   s_j   = scale * <q, k_j> + mask_j            (mask_j = -inf removes key j)
 *   m     = max_j s_j
 *   l     = sum_j exp(s_j - m)
 *   out   = sum_j exp(s_j - m) * v_j / l
 *   lse   = m + ln(l)                            (natural log; of the scaled, masked scores)
 *
 * Readings taken where the pages are silent:
 *   - causal is bottom-right aligned: query i sits at absolute position Lkv - Lq + i and
 *     may see keys j <= Lkv - Lq + i;
 *   - grouped-query attention maps query head h to kv head h / (Hq / Hkv);
 *   - a row that sees no key (all masked, or seq_len == 0) gives out = 0, lse = -inf;
 *   - the paged cache is [num_pages, Hkv, page_size, D] and key t of sequence b lives on
 *     page page_table[b, t / page_size] at slot t % page_size;
 *   - the MLA latent cache has one head: ckv [num_pages, page_size, Dc] serves as both K
 *     and V (flashinfer PR above, item 4) and kpe [num_pages, page_size, Dr] adds the
 *     rope term q_pe . kpe_t to the score.
 *
 * Inputs are read in their storage type (bf16 / fp16 / fp32 / fp64) and widened exactly to
 * fp64; every sum is a plain left-to-right fp64 sum; exp/log are the C library's fp64
 * functions.  No blocking, no online rescaling, no reordering: a direct two-pass softmax.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_BF16 = 0, OR_FP16 = 1, OR_FP32 = 2, OR_FP64 = 3 };

/* bf16 is the top half of an IEEE binary32: widening is a 16-bit shift. */
static double bf16_bits_to_double(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE binary16 -> double, from the format's definition (sign, 5-bit exponent with bias 15,
 * 10-bit fraction; exponent 0 is subnormal, exponent 31 is inf/nan). */
static double fp16_bits_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24);
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + f), e - 25);
  }
  return sign ? -v : v;
}

static double load_elem(const void* base, int64_t idx, int dtype) {
  switch (dtype) {
    case OR_BF16: return bf16_bits_to_double(((const uint16_t*)base)[idx]);
    case OR_FP16: return fp16_bits_to_double(((const uint16_t*)base)[idx]);
    case OR_FP32: return (double)((const float*)base)[idx];
    default: return ((const double*)base)[idx];
  }
}

/* One attention row given its scores (already scaled and masked; -inf = masked) and a
 * callback-free description of where the value rows are.  v_index[j] is the flat element
 * offset of value row j; the row has Dv elements. */
static void softmax_row(const double* s, int64_t n, const void* v, const int64_t* v_index,
                        int vdtype, int64_t Dv, double* out, double* lse) {
  double m = -INFINITY;
  for (int64_t j = 0; j < n; ++j)
    if (s[j] > m) m = s[j];
  for (int64_t d = 0; d < Dv; ++d) out[d] = 0.0;
  if (m == -INFINITY) { /* no visible key */
    *lse = -INFINITY;
    return;
  }
  double l = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    if (s[j] == -INFINITY) continue;
    double p = exp(s[j] - m);
    l += p;
    for (int64_t d = 0; d < Dv; ++d) out[d] += p * load_elem(v, v_index[j] + d, vdtype);
  }
  for (int64_t d = 0; d < Dv; ++d) out[d] /= l;
  *lse = m + log(l);
}

/*
 * Dense attention (prefill).  q [B,Hq,Lq,Dk], k [B,Hkv,Lkv,Dk], v [B,Hkv,Lkv,Dv], all
 * contiguous in `dtype`.  mask (optional, NULL = none) is an additive [Bm,Lq,Lkv] tensor in
 * `mask_dtype`, Bm in {1,B} (Bm == 1 broadcasts over the batch), shared by every head.
 * rows (optional) lists flat row ids (b*Hq + h)*Lq + i to evaluate; NULL = all rows in
 * order.  out [n_rows, Dv] and lse [n_rows] are fp64, in the order of `rows`.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_attention(const void* q, const void* k, const void* v, int dtype,
                     const void* mask, int mask_dtype, int64_t mask_batches,
                     int64_t B, int64_t Hq, int64_t Hkv, int64_t Lq, int64_t Lkv,
                     int64_t Dk, int64_t Dv, int causal, double scale,
                     const int64_t* rows, int64_t n_rows, double* out, double* lse) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Lq < 0 || Lkv < 0 || Dk <= 0 || Dv <= 0)
    return -1;
  if (mask && mask_batches != 1 && mask_batches != B) return -1;
  const int64_t G = Hq / Hkv;
  const int64_t total = B * Hq * Lq;
  if (!rows) n_rows = total;
  int bad = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(Lkv > 0 ? Lkv : 1));
    int64_t* vi = (int64_t*)malloc(sizeof(int64_t) * (size_t)(Lkv > 0 ? Lkv : 1));
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < n_rows; ++r) {
      int64_t flat = rows ? rows[r] : r;
      if (flat < 0 || flat >= total) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      int64_t i = flat % Lq;
      int64_t h = (flat / Lq) % Hq;
      int64_t b = flat / (Lq * Hq);
      int64_t hk = h / G;
      int64_t qoff = ((b * Hq + h) * Lq + i) * Dk;
      int64_t kbase = (b * Hkv + hk) * Lkv;
      for (int64_t j = 0; j < Lkv; ++j) {
        vi[j] = (kbase + j) * Dv;
        if (causal && j > i + (Lkv - Lq)) {
          s[j] = -INFINITY;
          continue;
        }
        double dot = 0.0;
        for (int64_t d = 0; d < Dk; ++d)
          dot += load_elem(q, qoff + d, dtype) * load_elem(k, (kbase + j) * Dk + d, dtype);
        double sj = scale * dot;
        if (mask) {
          int64_t mb = (mask_batches == 1) ? 0 : b;
          sj += load_elem(mask, (mb * Lq + i) * Lkv + j, mask_dtype);
        }
        s[j] = sj;
      }
      softmax_row(s, Lkv, v, vi, dtype, Dv, out + r * Dv, lse + r);
    }
    free(s);
    free(vi);
  }
  return bad ? -1 : 0;
}

/*
 * Paged grouped-query decode (one query token per sequence).  q [B,Hq,D];
 * k_pages, v_pages [num_pages,Hkv,page_size,D]; page_table [B,max_pages] int32;
 * seq_lens [B] int32.  Key t of sequence b is row t % page_size of page
 * page_table[b, t / page_size].  rows lists flat ids b*Hq + h (NULL = all).
 * Returns 0, or -1 on a bad argument (including a page id outside [0,num_pages)).
 */
int oracle_decode_paged(const void* q, const void* k_pages, const void* v_pages, int dtype,
                        const int32_t* page_table, const int32_t* seq_lens,
                        int64_t B, int64_t Hq, int64_t Hkv, int64_t D, int64_t page_size,
                        int64_t max_pages, int64_t num_pages, double scale,
                        const int64_t* rows, int64_t n_rows, double* out, double* lse) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || page_size <= 0) return -1;
  const int64_t G = Hq / Hkv;
  const int64_t total = B * Hq;
  if (!rows) n_rows = total;
  int64_t max_len = max_pages * page_size;
  int bad = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    int64_t* vi = (int64_t*)malloc(sizeof(int64_t) * (size_t)(max_len > 0 ? max_len : 1));
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
      int64_t flat = rows ? rows[r] : r;
      if (flat < 0 || flat >= total) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      int64_t h = flat % Hq, b = flat / Hq, hk = h / G;
      int64_t n = seq_lens[b];
      if (n < 0 || n > max_len) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      int row_bad = 0;
      for (int64_t t = 0; t < n; ++t) {
        int64_t page = page_table[b * max_pages + t / page_size];
        if (page < 0 || page >= num_pages) {
          row_bad = 1;
          break;
        }
        int64_t row = (page * Hkv + hk) * page_size + (t % page_size);
        vi[t] = row * D;
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d)
          dot += load_elem(q, flat * D + d, dtype) * load_elem(k_pages, row * D + d, dtype);
        s[t] = scale * dot;
      }
      if (row_bad) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      softmax_row(s, n, v_pages, vi, dtype, D, out + r * D, lse + r);
    }
    free(s);
    free(vi);
  }
  return bad ? -1 : 0;
}

/*
 * MLA paged decode in the absorbed (latent) form.  q_nope [B,H,Dc], q_pe [B,H,Dr];
 * ckv [num_pages,page_size,Dc], kpe [num_pages,page_size,Dr] (one latent head shared by
 * all H query heads); page_table [B,max_pages] int32; seq_lens [B] int32.
 *   s_t = scale * (q_nope . ckv_t + q_pe . kpe_t),  out = softmax(s) . ckv  (V = ckv).
 * out [n_rows, Dc], lse [n_rows]; rows lists flat ids b*H + h (NULL = all).
 */
int oracle_mla_decode_paged(const void* q_nope, const void* q_pe, const void* ckv,
                            const void* kpe, int dtype, const int32_t* page_table,
                            const int32_t* seq_lens, int64_t B, int64_t H, int64_t Dc,
                            int64_t Dr, int64_t page_size, int64_t max_pages,
                            int64_t num_pages, double scale, const int64_t* rows,
                            int64_t n_rows, double* out, double* lse) {
  if (B < 0 || H <= 0 || Dc <= 0 || Dr < 0 || page_size <= 0) return -1;
  const int64_t total = B * H;
  if (!rows) n_rows = total;
  int64_t max_len = max_pages * page_size;
  int bad = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    int64_t* vi = (int64_t*)malloc(sizeof(int64_t) * (size_t)(max_len > 0 ? max_len : 1));
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
      int64_t flat = rows ? rows[r] : r;
      if (flat < 0 || flat >= total) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      int64_t b = flat / H;
      int64_t n = seq_lens[b];
      if (n < 0 || n > max_len) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      int row_bad = 0;
      for (int64_t t = 0; t < n; ++t) {
        int64_t page = page_table[b * max_pages + t / page_size];
        if (page < 0 || page >= num_pages) {
          row_bad = 1;
          break;
        }
        int64_t row = page * page_size + (t % page_size);
        vi[t] = row * Dc;
        double dot = 0.0;
        for (int64_t d = 0; d < Dc; ++d)
          dot += load_elem(q_nope, flat * Dc + d, dtype) * load_elem(ckv, row * Dc + d, dtype);
        for (int64_t d = 0; d < Dr; ++d)
          dot += load_elem(q_pe, flat * Dr + d, dtype) * load_elem(kpe, row * Dr + d, dtype);
        s[t] = scale * dot;
      }
      if (row_bad) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      softmax_row(s, n, ckv, vi, dtype, Dc, out + r * Dc, lse + r);
    }
    free(s);
    free(vi);
  }
  return bad ? -1 : 0;
}

/*
 * Merge of attention states computed over disjoint key sets (split-KV).  For each row,
 * o_parts [rows, S, D] holds each part's normalised output and lse_parts [rows, S] its
 * log-sum-exp (-inf for a part that saw no key).  The merged state is
 *   lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * o_s
 * which is the softmax over the union of the parts' keys.  A row whose parts are all
 * -inf gives out = 0, lse = -inf.  o_parts/lse_parts are fp64 or fp32 (parts_dtype).
 */
int oracle_merge(const void* o_parts, const void* lse_parts, int parts_dtype, int64_t rows,
                 int64_t S, int64_t D, double* out, double* lse) {
  if (rows < 0 || S <= 0 || D <= 0) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    double m = -INFINITY;
    for (int64_t s = 0; s < S; ++s) {
      double x = load_elem(lse_parts, r * S + s, parts_dtype);
      if (x > m) m = x;
    }
    for (int64_t d = 0; d < D; ++d) out[r * D + d] = 0.0;
    if (m == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    double sum = 0.0;
    for (int64_t s = 0; s < S; ++s) {
      double x = load_elem(lse_parts, r * S + s, parts_dtype);
      if (x != -INFINITY) sum += exp(x - m);
    }
    double total = m + log(sum);
    for (int64_t s = 0; s < S; ++s) {
      double x = load_elem(lse_parts, r * S + s, parts_dtype);
      if (x == -INFINITY) continue;
      double w = exp(x - total);
      for (int64_t d = 0; d < D; ++d)
        out[r * D + d] += w * load_elem(o_parts, (r * S + s) * D + d, parts_dtype);
    }
    lse[r] = total;
  }
  return 0;
}

/* Number of threads the parallel regions above use (for reporting the baseline's cores). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

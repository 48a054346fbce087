// prefill_common.cuh -- per-row pieces shared by the prefill kernels: the row's visibility
// limits, one KV tile of the online softmax, the lazy O rescale, and the epilogue.  Each
// softmax thread owns one packed (query head, query) row of a 128-row tile; TMEM lane =
// row, so a warp touches the 32 lanes of its sub-partition.
#pragma once

#include <math.h>

#include "internal.h"
#include "sm103.cuh"

namespace fa {
namespace prefill {

constexpr int kRows = 128;
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the running max grows by > 2^8
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

struct Row {
  bool valid;         // a real (head, query) row of the problem
  int key_lim;        // keys j < key_lim are visible before the additive mask
  const char* mask;   // this query's additive mask row, or nullptr
  size_t flat;        // (b * Hq + h) * Lq + i
};

// Row r (0..127) of the tile whose first query is q0, for a sequence of Lkv keys.  Rows are
// packed head-major: r = g * q_per_tile + (i - q0), query head h = hk * G + g.
__device__ __forceinline__ Row make_row(const PrefillParams& p, int b, int hk, int q0, int r,
                                        int Lkv) {
  Row row;
  const int g = r / p.q_per_tile, i = q0 + r % p.q_per_tile;
  row.valid = (g < p.G) && (i < p.Lq);
  row.key_lim = 0;
  if (row.valid) row.key_lim = p.causal ? min(Lkv, i + (Lkv - p.Lq) + 1) : Lkv;
  row.mask = nullptr;
  if (p.mask && row.valid) {
    const int mb = p.mask_batches == 1 ? 0 : b;
    const size_t off = (static_cast<size_t>(mb) * p.Lq + i) * static_cast<size_t>(p.Lkv);
    row.mask = static_cast<const char*>(p.mask) + off * (p.mask_is_bf16 ? 2 : 4);
  }
  row.flat = (static_cast<size_t>(b) * p.Hq + hk * p.G + g) * p.Lq + i;
  return row;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// One KV tile of the online softmax for one row: raw = the tile's S row (fp32 bits, keys
// key0..key0+BN-1).  Updates the running max m (log2 units) and sum l, writes P (16-bit
// pairs, even key in the low half) to pk, and returns whether O must be rescaled by alpha.
// Lazy rescale: m moves only when the tile's max exceeds it by more than 2^8, so P may be
// computed against a stale max; the final division by l makes that exact.
template <int BN, bool BF16, bool kMax3>
__device__ __forceinline__ bool softmax_tile(const PrefillParams& p, const Row& row, int key0,
                                             const uint32_t (&raw)[BN], float& m, float& l,
                                             float& alpha, uint32_t (&pk)[BN / 2]) {
  // x[c] is either the raw score (fast path: no mask tensor and scale > 0, so the max of the
  // raw scores times scale is the max of the scaled ones) or the finished log2-domain score.
  // Masked keys hold -inf either way.  Eight independent max accumulators keep the
  // reduction's dependency chain short.
  const bool fast = !row.mask && p.scale_log2 > 0.f;
  // kMax3: reduce the max after x is built, with three-input max instructions; otherwise a
  // two-input max is folded into the loops that build x.  Which is faster depends on the
  // instantiation (measured; the caller chooses).
  float x[BN];
  float mx[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
  if (fast) {
    if (key0 + BN <= row.key_lim) {
#pragma unroll
      for (int c = 0; c < BN; ++c) {
        x[c] = __uint_as_float(raw[c]);
        if constexpr (!kMax3) mx[c & 7] = fmaxf(mx[c & 7], x[c]);
      }
    } else {
#pragma unroll
      for (int c = 0; c < BN; ++c) {
        x[c] = (key0 + c < row.key_lim) ? __uint_as_float(raw[c]) : -INFINITY;
        if constexpr (!kMax3) mx[c & 7] = fmaxf(mx[c & 7], x[c]);
      }
    }
  } else if (row.mask) {
#pragma unroll
    for (int c = 0; c < BN; ++c) {
      const int key = key0 + c;
      float v = -INFINITY;
      if (key < row.key_lim) {
        const float mv = p.mask_is_bf16
                             ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(row.mask)[key])
                             : reinterpret_cast<const float*>(row.mask)[key];
        v = fmaf(__uint_as_float(raw[c]), p.scale_log2, mv * kLog2e);
      }
      x[c] = v;
      if constexpr (!kMax3) mx[c & 7] = fmaxf(mx[c & 7], v);
    }
  } else {
#pragma unroll
    for (int c = 0; c < BN; ++c) {
      x[c] = (key0 + c < row.key_lim) ? __uint_as_float(raw[c]) * p.scale_log2 : -INFINITY;
      if constexpr (!kMax3) mx[c & 7] = fmaxf(mx[c & 7], x[c]);
    }
  }
  float row_max;
  if constexpr (kMax3) {
#pragma unroll
    for (int e = 0; e < 8; ++e) mx[e] = fmax3(x[e], x[e + 8], -INFINITY);
#pragma unroll
    for (int c = 16; c < BN; c += 16) {
#pragma unroll
      for (int e = 0; e < 8; ++e) mx[e] = fmax3(mx[e], x[c + e], x[c + 8 + e]);
    }
    row_max = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
  } else {
    row_max = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                    fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
  }
  if (fast) row_max *= p.scale_log2;
  const float m_new = fmaxf(m, row_max);
  const bool need = m_new > m + kRescaleLog2;
  alpha = 1.f;
  if (need) {
    alpha = exp2_approx(m - m_new);  // 0 when m is -inf
    m = m_new;
    l *= alpha;
  }
  const float m_use = (m == -INFINITY) ? 0.f : m;
  // p = 2^(x * a - m): one packed fp32x2 FMA per pair, packed adds into four partial sums.
  const float a = fast ? p.scale_log2 : 1.f;
  const float2 a2 = make_float2(a, a), nm2 = make_float2(-m_use, -m_use);
  float2 sum2[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) sum2[e] = make_float2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < BN / 2; ++c) {
    const float2 t = __ffma2_rn(make_float2(x[2 * c], x[2 * c + 1]), a2, nm2);
    const float p0 = exp2_approx(t.x);
    const float p1 = exp2_approx(t.y);
    sum2[c & 3] = __fadd2_rn(sum2[c & 3], make_float2(p0, p1));
    pk[c] = BF16 ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
  }
  const float2 s01 = __fadd2_rn(sum2[0], sum2[1]), s23 = __fadd2_rn(sum2[2], sum2[3]);
  l += (s01.x + s01.y) + (s23.x + s23.y);
  return need;
}

// Reads the tile's S row from tensor memory (all 32 lanes of the warp must call it).
template <int BN>
__device__ __forceinline__ void load_s(uint32_t t_s, uint32_t (&raw)[BN]) {
#pragma unroll
  for (int c = 0; c < BN / 32; ++c)
    tmem_ld32(t_s + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&raw[c * 32]));
  tmem_ld_wait();
}

// O row *= alpha in tensor memory (warp-collective; lanes that need no rescale pass 1).
template <int D>
__device__ __forceinline__ void rescale_o(uint32_t t_o, float alpha) {
#pragma unroll 1
  for (int c = 0; c < D / 32; ++c) {
    uint32_t o[32];
    tmem_ld32(t_o + c * 32, o);
    tmem_ld_wait();
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
    tmem_st32(t_o + c * 32, o);
  }
}

// Writes P (packed pairs) over the first BN/2 columns of the S buffer (warp-collective).
template <int BN>
__device__ __forceinline__ void store_p(uint32_t t_s, const uint32_t (&pk)[BN / 2]) {
#pragma unroll
  for (int c = 0; c < BN / 2; c += 16)
    tmem_st16(t_s + c, *reinterpret_cast<const uint32_t(*)[16]>(&pk[c]));
}

// log-sum-exp (natural log) of a row from its running max (log2 units) and sum
__device__ __forceinline__ float row_lse(float m, float l) {
  return l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

// Epilogue of one row with per-thread stores: O / l to the output in out_dtype, lse to p.lse.
// Warp-collective: every lane reads its TMEM lane; rows that are not valid store nothing.
// have_o is false when no P V product was issued (no KV tile in this part): the row is then
// empty.
template <int D>
__device__ __forceinline__ void epilogue(const PrefillParams& p, const Row& row, uint32_t t_o,
                                         bool have_o, float m, float l) {
  const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
  for (int c = 0; c < D / 32; ++c) {
    uint32_t o[32];
    if (have_o) {
      tmem_ld32(t_o + c * 32, o);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = 0u;
    }
    if (!row.valid) continue;
    float v[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(o[e]) * inv_l;
    if (p.out_dtype == Dtype::FP32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + row.flat * D + c * 32);
#pragma unroll
      for (int e = 0; e < 8; ++e) dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
    } else {
      uint32_t w[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        w[e] = (p.out_dtype == Dtype::BF16) ? pack_bf16x2(v[2 * e], v[2 * e + 1])
                                            : pack_f16x2(v[2 * e], v[2 * e + 1]);
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + row.flat * D + c * 32);
#pragma unroll
      for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
    }
  }
  if (row.valid && p.lse) p.lse[row.flat] = row_lse(m, l);
}

// 4-D tiled TMA store from shared to global memory, completed through the bulk group
// (coordinates non-negative; the innermost one a multiple of 16 bytes).
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, uint32_t src, int32_t c0,
                                             int32_t c1, int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until the committed bulk stores have read their shared-memory sources.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// tcgen05.wait::ld tied to the 32 registers of one earlier tmem_ld32: the compiler cannot move
// a use of them above it (a plain wait orders memory only), so a second load may be in
// flight while these are used.
__device__ __forceinline__ void tmem_ld_wait_tied(uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
        "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
        "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
        "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
        "+r"(r[31])
      :
      : "memory");
}

// Staging of one row's output for TMA stores, 32 columns (one tcgen05.ld) at a time.  A slab
// of fp32 partial state holds columns 32c .. 32c+31 of the 128 rows as 128-byte rows; a
// 16-bit tile holds columns 64t .. 64t+63, two slabs' worth.  Both use the 128-byte swizzle:
// 16-byte chunk ch of row r sits at chunk ch ^ (r & 7), so the 32 rows of a warp write
// whole 128-byte bank lines.
__device__ __forceinline__ void stage_slab_f32(const uint32_t (&o)[32], float inv_l, uint8_t* slab,
                                               int r) {
  uint8_t* row = slab + r * 128;
#pragma unroll
  for (int ch = 0; ch < 8; ++ch)
    *reinterpret_cast<float4*>(row + ((ch ^ (r & 7)) * 16)) =
        make_float4(__uint_as_float(o[4 * ch]) * inv_l, __uint_as_float(o[4 * ch + 1]) * inv_l,
                    __uint_as_float(o[4 * ch + 2]) * inv_l, __uint_as_float(o[4 * ch + 3]) * inv_l);
}

// Columns 32c .. 32c+31 in 16 bits (BF16 selects bf16, else fp16): chunks 4(c % 2) .. +3 of
// the row in its 64-column tile.
template <bool BF16>
__device__ __forceinline__ void stage_slab16(const uint32_t (&o)[32], float inv_l, uint8_t* tile,
                                             int r, int c) {
  uint8_t* row = tile + r * 128;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = __uint_as_float(o[8 * q + 2 * e]) * inv_l;
      const float b = __uint_as_float(o[8 * q + 2 * e + 1]) * inv_l;
      w[e] = BF16 ? pack_bf16x2(a, b) : pack_f16x2(a, b);
    }
    const int ch = 4 * (c % 2) + q;
    *reinterpret_cast<uint4*>(row + ((ch ^ (r & 7)) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}


// KV tiles [t_begin, t_end) of one split for a tile set whose last query is q_last, in a
// sequence of Lkv keys.
__device__ __forceinline__ void kv_range(const PrefillParams& p, int q_last, int bn, int split,
                                         int Lkv, int& t_begin, int& t_end) {
  int kv_end = Lkv;
  if (p.causal) kv_end = min(Lkv, q_last + (Lkv - p.Lq) + 1);
  const int n_kv_tiles = kv_end > 0 ? (kv_end + bn - 1) / bn : 0;
  const int per_split = (n_kv_tiles + p.n_splits - 1) / p.n_splits;
  t_begin = min(n_kv_tiles, split * per_split);
  t_end = min(n_kv_tiles, t_begin + per_split);
}

}  // namespace prefill
}  // namespace fa

// gated_delta.cu -- chunked prefill of gated-delta linear attention on sm_103a.
//
// The hip-ep PR "perf(kernels): speed up linear-attention prefill ~2.6x" (Summary) speeds up
// a gated-delta chunked linear-attention prefill; the recurrence it computes is the gated
// delta rule, with a state S of dv rows by dk columns per value head:
//   S_t = S_{t-1} alpha_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t (scale q_t)
// with alpha_t = exp(g_t).  Over a chunk of C = 64 tokens with cumulative log decays
// gamma_i = g_1 + ... + g_i (Gamma_i = e^gamma_i) and the state S entering the chunk, the
// chunk's writes u_i = beta_i (v_i - alpha_i S_{i-1} k_i) satisfy
//   (I + A) U = beta (V - Gamma K S^T),   A_ij = beta_i (Gamma_i / Gamma_j) k_i.k_j (j < i)
// so, with X = (I + A)^-1 applied to beta Gamma K (= W) and to beta V (= U~):
//   U = U~ - W S^T
//   O = Gamma (scale Q) S^T + P U,        P_ij = scale (Gamma_i / Gamma_j) q_i.k_j (j <= i)
//   S <- Gamma_C S + U^T (Gamma_C / Gamma_j) K
// Two kernels:
//   1. chunk preparation (every chunk of every head in parallel): the Gram products Q K^T
//      and K K^T in one tensor-core MMA (the chunk's Q and K rows stacked as a 128-row A
//      operand against its K rows), T = (I + A)^-1 on the CUDA cores in fp32 (blocked: the
//      four 16x16 diagonal blocks by substitution, then the off-diagonal blocks one block
//      diagonal at a time), then W = T diag(beta Gamma) K and U~ = T diag(beta) V on the
//      tensor cores (T's scaled columns split into bf16 high and low parts, so the products
//      keep ~16 bits; K and V exact in bf16), P, and the per-token decay factors Gamma_i and
//      Gamma_C / Gamma_i; written to a workspace (W and P in bf16 as tensor-core operands,
//      U~ and the factors in fp32);
//   2. the recurrence across chunks (one CTA per (batch, value head), tensor cores): the state
//      lives in tensor memory in fp32 (dv lanes x dk columns), with a bf16 copy in shared
//      memory as the A operand; per chunk  U^T = U~^T - S W^T,  O^T = S Q^T (scaled per token)
//      + U^T P^T,  S <- Gamma_C S + (U^T scaled per token) K,  with the chunk's W, Q, K, P and
//      decay factors streamed by TMA through a two-stage ring.
// The output O and the final state are written per chunk; no chunk's state is kept.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "../../include/fa.h"
#include "internal.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kC = 64;     // tokens per chunk
constexpr int kDk = 128;
constexpr int kDv = 128;

struct GdnParams {
  const uint16_t* q;     // [B,Hk,T,dk] bf16
  const uint16_t* k;     // [B,Hk,T,dk] bf16
  const uint16_t* v;     // [B,Hv,T,dv] bf16
  const float* g;        // [B,Hv,T]
  const float* beta;     // [B,Hv,T]
  const float* s0;       // [B,Hv,dv,dk] or nullptr
  uint16_t* out;         // [B,Hv,T,dv] bf16
  float* s_final;        // [B,Hv,dv,dk] or nullptr
  int B, T, Hk, Hv, n_chunks, Tpad;
  float scale;
  uint16_t* w_ws;        // [B*Hv*Tpad, dk] bf16
  float* u_ws;           // [B*Hv*Tpad, dv] fp32
  uint16_t* p_ws;        // [B*Hv*Tpad, C] bf16 (rows of each chunk's P)
  float* f_ws;           // [B*Hv*n_chunks, 2C] fp32: Gamma_i, then Gamma_C / Gamma_i
  uint32_t* status;
};

// ------------------------------------------------------------------------------------------
// Kernel 1: chunk preparation.  One CTA per (chunk, value head, batch), 256 threads.  Thread
// 0 loads the chunk's Q, K and V rows with TMA (128-byte swizzled, rows past the sequence
// read as zero) and issues the MMAs; warps 0-3 read the Gram rows back; all threads form T.
// ------------------------------------------------------------------------------------------
constexpr int kPrepThreads = 256;
constexpr int kTriF = kC + 4;                  // padded fp32 row of A and T (float4-aligned)
constexpr int kPQK = 0;                        // [Q rows; K rows]: 2 column blocks of 128 x 128 B
constexpr int kPV = kPQK + 2 * 128 * 128;      // V rows: 2 column blocks of 64 x 128 B
constexpr int kPA = kPV + 2 * kC * 128;        // A, fp32 [C][kTriF]
constexpr int kPT = kPA + kC * kTriF * 4;      // T = (I + A)^-1, fp32 [C][kTriF]
constexpr int kPM = kPT + kC * kTriF * 4;      // off-diagonal block sums, 3 x 16 x 16 fp32
constexpr int kPSmall = kPM + 3 * 256 * 4;     // gamma, beta, raw g, Gamma: 4 x C fp32
constexpr int kPBar = kPSmall + 4 * kC * 4;    // three mbarriers + the tensor-memory slot
constexpr int kPrepSmem = kPBar + 32 + 1024;
// The MMA operands T diag(beta Gamma) and T diag(beta) (64 x 64 bf16, K-major, 128-byte
// swizzled, high and low parts) reuse dead space once T is formed: the Q rows of the [Q; K]
// tile (read only by the Gram MMA) and the A matrix.
constexpr int kOpWHi = kPQK, kOpWLo = kPQK + 128 * 128, kOpUHi = kPA, kOpULo = kPA + kC * 128;
static_assert(kPA % 1024 == 0 && kC * kTriF * 4 >= 2 * kC * 128, "operand tiles over A");
static_assert(2 * kPrepSmem <= 232448, "two CTAs per SM");

__global__ void __launch_bounds__(kPrepThreads, 2)
    gdn_prep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const GdnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_addr(smem);
  float* As = reinterpret_cast<float*>(smem + kPA);
  float* Ts = reinterpret_cast<float*>(smem + kPT);
  float* Ms = reinterpret_cast<float*>(smem + kPM);
  float* gam = reinterpret_cast<float*>(smem + kPSmall);
  float* bet = gam + kC;
  float* graw = bet + kC;  // raw g, then gamma_i in log2 units (after the scan)
  float* Gam = graw + kC;  // Gamma_i = e^gamma_i
  const uint32_t bar_ld = s_base + kPBar, bar_mma = s_base + kPBar + 8;
  const uint32_t bar_mma2 = s_base + kPBar + 24;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kPBar + 16);

  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  const int warp = tid / 32, lane = tid % 32;
  const int hk = h / (p.Hv / p.Hk);
  const int t0 = c * kC, n = min(kC, p.T - t0);
  const size_t bh = static_cast<size_t>(b) * p.Hv + h;

  if (tid == 0) {
    mbar_init(bar_ld, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_mma2, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    // Gram result (M = 128, 64 columns), later W and U~ (M = 64, 2 x 128 columns)
    tmem_alloc(smem_addr(tmem_slot), 256);
    tmem_relinquish();
  }
  if (tid < kC) {
    const bool ok = tid < n;
    graw[tid] = ok ? p.g[bh * p.T + t0 + tid] : 0.f;  // padding: no decay, no write
    bet[tid] = ok ? p.beta[bh * p.T + t0 + tid] : 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_ld, 6 * kC * 128);
    for (int cb = 0; cb < 2; ++cb) {
      tma_load_3d(s_base + kPQK + cb * 128 * 128, &tm_q, bar_ld, cb * 64, t0, b * p.Hk + hk);
      tma_load_3d(s_base + kPQK + cb * 128 * 128 + kC * 128, &tm_k, bar_ld, cb * 64, t0, b * p.Hk + hk);
      tma_load_3d(s_base + kPV + cb * kC * 128, &tm_v, bar_ld, cb * 64, t0, static_cast<int>(bh));
    }
    // [Q; K] K^T: M = 128 (query rows, then key rows), N = 64 key rows, K = 128
    bool ok = mbar_wait(bar_ld, 0, p.status);
    if (ok) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_f16(true, 128, kC, false, false);
#pragma unroll
      for (int kk = 0; kk < kDk / 16; ++kk) {
        const uint32_t off = (kk / 4) * (128 * 128) + (kk % 4) * 32;
        mma_ss(tmem, sdesc_sw128(s_base + kPQK + off, 16, 1024),
               sdesc_sw128(s_base + kPQK + off + kC * 128, 16, 1024), idesc, kk > 0 ? 1u : 0u);
      }
    }
    tc_commit(bar_mma);  // arrives once the MMAs (if any) are done
  }
  // cumulative log decay within the chunk (inclusive scan by warp 4, two tokens per lane)
  if (warp == 4) {
    const int l = tid - 128;
    const float a = graw[2 * l], a2 = graw[2 * l + 1];
    float sc = a + a2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, sc, o);
      if (l >= o) sc += y;
    }
    const float excl = sc - (a + a2);
    gam[2 * l] = excl + a;
    gam[2 * l + 1] = excl + a + a2;
    constexpr float kLog2e = 1.44269504088896340736f;
    graw[2 * l] = (excl + a) * kLog2e;
    graw[2 * l + 1] = (excl + a + a2) * kLog2e;
  }
  __syncthreads();
  bool ok = __syncthreads_and(mbar_wait(bar_mma, 0, p.status));
  {
    // lane r of the Gram result: r < 64 is row r of Q K^T (-> P), r >= 64 row r - 64 of K K^T;
    // warps q and q + 4 share the sub-partition's lanes and take columns 0-31 and 32-63
    tc_fence_after();
    const int quad = warp % 4, j0 = 32 * (warp / 4);
    uint32_t raw[32];
    tmem_ld32(tmem + (static_cast<uint32_t>(quad * 32) << 16) + j0, raw);
    tmem_ld_wait();
    // Gamma_i / Gamma_j = 2^(gl_i - gl_j) <= 1 for j <= i (gl = gamma in log2 units)
    const float* gl = graw;
    const int r = quad * 32 + lane;
    if (r < kC) {
      const int i = r;
      const float gi = gl[i];
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        const int j = j0 + e;
        const float p0 = (j <= i && i < n) ? p.scale * exp2_approx(gi - gl[j]) * __uint_as_float(raw[e]) : 0.f;
        const float p1 = (j + 1 <= i && i < n) ? p.scale * exp2_approx(gi - gl[j + 1]) * __uint_as_float(raw[e + 1]) : 0.f;
        pk[e / 2] = pack_bf16x2(p0, p1);
      }
      uint4* dst = reinterpret_cast<uint4*>(p.p_ws + (bh * p.Tpad + t0 + i) * kC + j0);
#pragma unroll
      for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
    } else {
      const int i = r - kC;
      const float gi = gl[i], bi = bet[i];
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const int j = j0 + e;
        float4 a;
        a.x = j < i ? bi * exp2_approx(gi - gl[j]) * __uint_as_float(raw[e]) : 0.f;
        a.y = j + 1 < i ? bi * exp2_approx(gi - gl[j + 1]) * __uint_as_float(raw[e + 1]) : 0.f;
        a.z = j + 2 < i ? bi * exp2_approx(gi - gl[j + 2]) * __uint_as_float(raw[e + 2]) : 0.f;
        a.w = j + 3 < i ? bi * exp2_approx(gi - gl[j + 3]) * __uint_as_float(raw[e + 3]) : 0.f;
        *reinterpret_cast<float4*>(As + i * kTriF + j) = a;
      }
    }
  }
  if (tid < 2 * kC) {
    // decay factors of the chunk: Gamma_i, then Gamma_C / Gamma_i
    const int e = tid;
    const float v = e < kC ? expf(gam[e]) : expf(gam[kC - 1] - gam[e - kC]);
    p.f_ws[(bh * p.n_chunks + c) * (2 * kC) + e] = v;
    if (e < kC) Gam[e] = v;
  }
  if (!ok) {
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
      tc_fence_after();
      tmem_dealloc(tmem, 256);
    }
    return;
  }
  // T = (I + A)^-1 (A strictly lower triangular, 16 x 16 blocks A_ik): T_ii = (I + A_ii)^-1
  // by substitution, then for i > j, one block diagonal at a time,
  //   T_ij = -T_ii M_ij,   M_ij = sum_{k=j}^{i-1} A_ik T_kj.
  for (int e = tid; e < kC * kC; e += kPrepThreads) Ts[(e / kC) * kTriF + e % kC] = 0.f;
  __syncthreads();
  if (tid < kC) {
    const int blk = tid / 16, cj = tid % 16, o = 16 * blk;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float acc = r == cj ? 1.f : 0.f;
#pragma unroll
      for (int q = 0; q < r; ++q) acc -= As[(o + r) * kTriF + o + q] * x[q];
      x[r] = acc;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) Ts[(o + r) * kTriF + o + cj] = x[r];
  }
  __syncthreads();
  // (the loops have constant trip counts so they unroll, with four partial sums each)
#pragma unroll
  for (int d = 1; d < 4; ++d) {
    // M for the 4 - d blocks (i = j + d): one entry (r, cc) of one block per thread and pass
#pragma unroll
    for (int pass = 0; pass < 4 - d; ++pass) {
      const int e = tid + pass * kPrepThreads;
      const int jb = e / 256, r = (e / 16) % 16, cc = e % 16, ib = jb + d;
      const float* arow = As + (16 * ib + r) * kTriF + 16 * jb;
      const float* tcol = Ts + 16 * jb * kTriF + 16 * jb + cc;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < 16 * d; ++k) acc[k & 3] += arow[k] * tcol[k * kTriF];
      Ms[e] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
    __syncthreads();
    // T_ij = -T_ii M_ij (T_ii is zero above its diagonal, so every row sums all 16 terms)
#pragma unroll
    for (int pass = 0; pass < 4 - d; ++pass) {
      const int e = tid + pass * kPrepThreads;
      const int jb = e / 256, r = (e / 16) % 16, cc = e % 16, ib = jb + d;
      const float* trow = Ts + (16 * ib + r) * kTriF + 16 * ib;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < 16; ++q) acc[q & 3] += trow[q] * Ms[jb * 256 + q * 16 + cc];
      Ts[(16 * ib + r) * kTriF + 16 * jb + cc] = -((acc[0] + acc[1]) + (acc[2] + acc[3]));
    }
    __syncthreads();
  }

  // The MMA operands: T diag(beta Gamma) for W and T diag(beta) for U~, each as a bf16 high
  // part and the bf16 rounding of the remainder, written K-major in the 128-byte swizzle
  // (row i, 16-byte chunk ch at chunk ch ^ (i & 7)).  A is no longer read.
  {
    const int i = tid / 4, g = tid % 4;
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int ch = 2 * g + h2;
      uint32_t whi[4], wlo[4], uhi[4], ulo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j0 = 8 * ch + 2 * e;
        float w2[2], u2[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const float tv = Ts[i * kTriF + j0 + t];
          u2[t] = tv * bet[j0 + t];
          w2[t] = u2[t] * Gam[j0 + t];
        }
        whi[e] = pack_bf16x2(w2[0], w2[1]);
        uhi[e] = pack_bf16x2(u2[0], u2[1]);
        const float wh0 = __uint_as_float(whi[e] << 16), wh1 = __uint_as_float(whi[e] & 0xFFFF0000u);
        const float uh0 = __uint_as_float(uhi[e] << 16), uh1 = __uint_as_float(uhi[e] & 0xFFFF0000u);
        wlo[e] = pack_bf16x2(w2[0] - wh0, w2[1] - wh1);
        ulo[e] = pack_bf16x2(u2[0] - uh0, u2[1] - uh1);
      }
      const int off = i * 128 + ((ch ^ (i & 7)) * 16);
      *reinterpret_cast<uint4*>(smem + kOpWHi + off) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
      *reinterpret_cast<uint4*>(smem + kOpWLo + off) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
      *reinterpret_cast<uint4*>(smem + kOpUHi + off) = make_uint4(uhi[0], uhi[1], uhi[2], uhi[3]);
      *reinterpret_cast<uint4*>(smem + kOpULo + off) = make_uint4(ulo[0], ulo[1], ulo[2], ulo[3]);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    tc_fence_after();
    // W (columns 0-127) and U~ (columns 128-255): M = 64 chunk rows, N = 128, K = 64 tokens;
    // A = the operand tiles (K-major), B = the chunk's K or V rows read MN-major.
    constexpr uint32_t idesc = idesc_f16(true, kC, 128, false, true);
    const uint32_t kb = s_base + kPQK + kC * 128, vb = s_base + kPV;
#pragma unroll
    for (int part = 0; part < 4; ++part) {
      const uint32_t a_tile = s_base + (part == 0 ? kOpWHi : part == 1 ? kOpWLo : part == 2 ? kOpUHi : kOpULo);
      const uint32_t d = tmem + (part < 2 ? 0u : 128u);
#pragma unroll
      for (int kk = 0; kk < kC / 16; ++kk) {
        const uint64_t ad = sdesc_sw128(a_tile + kk * 32, 16, 1024);
        const uint64_t bd = part < 2 ? sdesc_sw128(kb + kk * 2048, 128 * 128, 1024)
                                     : sdesc_sw128(vb + kk * 2048, kC * 128, 1024);
        mma_ss(d, ad, bd, idesc, ((part & 1) || kk > 0) ? 1u : 0u);
      }
    }
    tc_commit(bar_mma2);
  }
  ok = __syncthreads_and(mbar_wait(bar_mma2, 0, p.status));
  if (ok) {
    // M = 64 result: row 16 q + l (l < 16) sits in lane 32 q + l; warps q and q + 4 share the
    // sub-partition's lanes, the first writing W (columns 0-127), the second U~ (128-255)
    tc_fence_after();
    const int quad = warp % 4, half = warp / 4;
    const int i = 16 * quad + lane % 16;
    const size_t row = bh * p.Tpad + t0 + i;
#pragma unroll 1
    for (int cb = 4 * half; cb < 4 * half + 4; ++cb) {
      uint32_t r32[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(quad * 32) << 16) + cb * 32, r32);
      tmem_ld_wait();
      if (lane < 16) {
        if (cb < 4) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(r32[2 * e]), __uint_as_float(r32[2 * e + 1]));
          uint4* dst = reinterpret_cast<uint4*>(p.w_ws + row * kDk + cb * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        } else {
          float4* dst = reinterpret_cast<float4*>(p.u_ws + row * kDv + (cb - 4) * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(r32[4 * e]), __uint_as_float(r32[4 * e + 1]),
                                 __uint_as_float(r32[4 * e + 2]), __uint_as_float(r32[4 * e + 3]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ------------------------------------------------------------------------------------------
// Kernel 2: the recurrence across chunks.  One CTA per (value head, batch), 320 threads:
// warps 0-7 own the state rows (thread (d, half): tensor-memory lane d = value dim d, warps
// 0-3 and 4-7 taking the two halves of every row's columns), warp 8 loads the chunk operands
// with TMA, warp 9 issues the MMAs and owns the tensor memory.
// ------------------------------------------------------------------------------------------
constexpr int kStateWarps = 8;
constexpr int kStateThreads = (kStateWarps + 2) * 32;
constexpr int kProducerWarp = kStateWarps, kMmaWarp = kStateWarps + 1;
constexpr int kBlkTok = kC * 128;                // one 64-column block of a 64-row tile
constexpr int kStageW = 0;
constexpr int kStageQ = kStageW + 2 * kBlkTok;
constexpr int kStageK = kStageQ + 2 * kBlkTok;
constexpr int kStageP = kStageK + 2 * kBlkTok;
constexpr int kStageF = kStageP + kBlkTok;       // decay factors: Gamma_i, Gamma_C / Gamma_i
constexpr int kStageTx = kStageF + 2 * kC * 4;   // bytes landing per chunk
constexpr int kStageBytes = (kStageTx + 1023) / 1024 * 1024;
constexpr int kSbfOff = 2 * kStageBytes;         // S as bf16, [128 rows][2 blocks of 128 B]
constexpr int kSBlk = kDv * 128;                 // 16384: one 64-column block of S
constexpr int kUtOff = kSbfOff + 2 * kSBlk;      // U^T, [128 rows][128 B]
constexpr int kUptOff = kUtOff + kSBlk;          // U^T with each token's decay to the chunk end
constexpr int kUtlOff = kUptOff + kSBlk;         // U~ of the chunk, fp32 [64 tokens][128 dv]
constexpr int kUtlBytes = kC * kDv * 4;
constexpr int kBarOff = kUtlOff + kUtlBytes;
// full[2], empty[2], s_ready, u_ready, u_done, o_done, mma_done, s_done, utl_full, utl_empty
constexpr int kNumBars = 12;
constexpr int kStateSmem = kBarOff + kNumBars * 8 + 16 + 1024;
static_assert(kStateSmem <= 232448, "shared memory budget");
// tensor memory: the state (128 columns), D_U (64), and two sets of output accumulators D_O1,
// D_O2 (64 each), used by alternate chunks
constexpr uint32_t kTmS = 0, kTmU = 128, kTmO1 = 192, kTmO2 = 256, kTmOSet = 128;
constexpr uint32_t kStateArrivals = kStateWarps * 32;

__global__ void __launch_bounds__(kStateThreads, 1)
    gdn_state_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_p,
                     const GdnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_addr(smem);
  const uint32_t bars = s_base + kBarOff;
  auto bar_full = [&](int s) { return bars + 8u * s; };
  auto bar_empty = [&](int s) { return bars + 8u * (2 + s); };
  const uint32_t bar_sready = bars + 8u * 4, bar_uready = bars + 8u * 5;
  const uint32_t bar_udone = bars + 8u * 6, bar_odone = bars + 8u * 7, bar_done = bars + 8u * 8;
  const uint32_t bar_sdone = bars + 8u * 9;  // the state update of the chunk has finished
  const uint32_t bar_utl_full = bars + 8u * 10, bar_utl_empty = bars + 8u * 11;  // U~ tile
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + kNumBars * 8);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int h = blockIdx.x, b = blockIdx.y;
  const int hk = h / (p.Hv / p.Hk);
  const size_t bh = static_cast<size_t>(b) * p.Hv + h;
  const int nc = p.n_chunks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_full(s), 1);
      // a stage is free again once its MMAs are done (one commit) and every state thread
      // has read its decay factors
      mbar_init(bar_empty(s), 1 + kStateArrivals);
    }
    mbar_init(bar_sready, kStateArrivals);
    mbar_init(bar_uready, kStateArrivals);
    mbar_init(bar_udone, 1);
    mbar_init(bar_odone, 1);
    mbar_init(bar_done, 1);
    mbar_init(bar_sdone, 1);
    mbar_init(bar_utl_full, 1);
    mbar_init(bar_utl_empty, kStateArrivals);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    // ---------------------------------- TMA producer ------------------------------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_w);
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_p);
      int issued = 0, u_issued = 0;
      for (int c = 0; c < nc; ++c) {
        const int st = c & 1;
        if (c >= 2 && !mbar_wait(bar_empty(st), ((c >> 1) - 1) & 1, p.status)) break;
        const uint32_t base = s_base + st * kStageBytes;
        const int row = static_cast<int>(bh * p.Tpad) + c * kC;
        mbar_arrive_expect_tx(bar_full(st), kStageTx);
        for (int cb = 0; cb < 2; ++cb) {
          tma_load_2d(base + kStageW + cb * kBlkTok, &tm_w, bar_full(st), cb * 64, row);
          tma_load_3d(base + kStageQ + cb * kBlkTok, &tm_q, bar_full(st), cb * 64, c * kC, b * p.Hk + hk);
          tma_load_3d(base + kStageK + cb * kBlkTok, &tm_k, bar_full(st), cb * 64, c * kC, b * p.Hk + hk);
        }
        tma_load_2d(base + kStageP, &tm_p, bar_full(st), 0, row);
        bulk_load(base + kStageF, p.f_ws + (bh * nc + c) * (2 * kC), 2 * kC * 4, bar_full(st));
        issued = c + 1;
        // the chunk's U~ (64 contiguous rows), once the state warps have read the previous one
        if (c >= 1 && !mbar_wait(bar_utl_empty, (c - 1) & 1, p.status)) break;
        mbar_arrive_expect_tx(bar_utl_full, kUtlBytes);
        bulk_load(s_base + kUtlOff, p.u_ws + (bh * p.Tpad + c * kC) * kDv, kUtlBytes, bar_utl_full);
        u_issued = c + 1;
      }
      // a wait ran out: let the copies in flight land before the CTA exits
      for (int c = max(0, issued - 2); c < issued && issued < nc; ++c)
        mbar_wait(bar_full(c & 1), (c >> 1) & 1, nullptr);
      if (u_issued > 0 && u_issued < nc) mbar_wait(bar_utl_full, (u_issued - 1) & 1, nullptr);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------- MMA issuer --------------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc_n64 = idesc_f16(true, 128, 64, false, false);
      constexpr uint32_t idesc_s = idesc_f16(true, 128, 128, false, true);
      const uint32_t sbf = s_base + kSbfOff, ut = s_base + kUtOff, upt = s_base + kUptOff;
      bool ok = true;
      for (int c = 0; ok && c < nc; ++c) {
        const int st = c & 1;
        const uint32_t base = s_base + st * kStageBytes;
        if (!(ok = mbar_wait(bar_full(st), (c >> 1) & 1, p.status))) break;
        if (!(ok = mbar_wait(bar_sready, c & 1, p.status))) break;
        tc_fence_after();
        // S W^T -> D_U (M = 128 value dims, N = 64 tokens, K = 128 key dims)
#pragma unroll
        for (int kk = 0; kk < kDk / 16; ++kk) {
          const uint32_t off = (kk / 4) * kSBlk + (kk % 4) * 32;
          mma_ss(tmem + kTmU, sdesc_sw128(sbf + off, 16, 1024),
                 sdesc_sw128(base + kStageW + (kk / 4) * kBlkTok + (kk % 4) * 32, 16, 1024),
                 idesc_n64, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar_udone);
        // S Q^T -> D_O1 of this chunk's output set
        const uint32_t oset = (c & 1) * kTmOSet;
#pragma unroll
        for (int kk = 0; kk < kDk / 16; ++kk) {
          const uint32_t off = (kk / 4) * kSBlk + (kk % 4) * 32;
          mma_ss(tmem + kTmO1 + oset, sdesc_sw128(sbf + off, 16, 1024),
                 sdesc_sw128(base + kStageQ + (kk / 4) * kBlkTok + (kk % 4) * 32, 16, 1024),
                 idesc_n64, kk > 0 ? 1u : 0u);
        }
        if (!(ok = mbar_wait(bar_uready, c & 1, p.status))) break;
        tc_fence_after();
        // D_S (already Gamma_C S) += U'^T K (N = 128 key dims, K = 64 tokens; K read MN-major),
        // first: the next chunk's state copy waits only for this
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_ss(tmem + kTmS, sdesc_sw128(upt + kk * 32, 16, 1024),
                 sdesc_sw128(base + kStageK + kk * 2048, kBlkTok, 1024), idesc_s, 1u);
        tc_commit(bar_sdone);
        // U^T P^T -> D_O2 (N = 64 query tokens, K = 64 key tokens)
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_ss(tmem + kTmO2 + oset, sdesc_sw128(ut + kk * 32, 16, 1024),
                 sdesc_sw128(base + kStageP + kk * 32, 16, 1024), idesc_n64, kk > 0 ? 1u : 0u);
        tc_commit(bar_odone);
        tc_commit(bar_empty(st));
      }
      tc_commit(bar_done);
      mbar_wait(bar_done, 0, nullptr);
    }
  } else {
    // ------------------ state rows: thread (d, half), d = value dim d ------------------
    const int d = (warp & 3) * 32 + lane;
    const int half = warp >> 2;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint8_t* sbf = smem + kSbfOff;
    uint8_t* utp = smem + kUtOff;
    uint8_t* uptp = smem + kUptOff;
    // Row d of a K-major 128-byte-swizzled tile: 16-byte chunk ch sits at chunk ch ^ (d % 8).
    auto put_row32 = [&](uint8_t* blk, int ch0, const float (&v)[32]) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(blk + d * 128 + (((ch0 + q) ^ (d & 7)) * 16)) =
            make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                       pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
    };
    // This thread's columns: tokens 32 half .. +31 of D_U, D_O1, D_O2 and of U^T; key dims
    // 64 half .. +63 of the state (block `half` of its bf16 copy).
    // Per chunk c the state in tensor memory enters already scaled by Gamma_C of chunk c (the
    // chunk's MMA adds U'^T K to it), while the bf16 copy holds the unscaled state S.  Chunk
    // c's outputs are formed as soon as its products land but stored only after chunk c+1's
    // U has been published, so the stores overlap the next chunk's MMAs.
    auto fct_of = [&](int cc) {
      return reinterpret_cast<const float*>(smem + (cc & 1) * kStageBytes + kStageF);
    };
    bool ok = __all_sync(0xffffffffu, mbar_wait(bar_full(0), 0, p.status));
    {
      const float g0 = ok ? fct_of(0)[kC - 1] : 1.f;
#pragma unroll 1
      for (int pc = 0; pc < 2; ++pc) {
        float s[32];
#pragma unroll
        for (int e = 0; e < 32; ++e)
          s[e] = p.s0 ? p.s0[(bh * kDv + d) * kDk + half * 64 + pc * 32 + e] : 0.f;
        put_row32(sbf + half * kSBlk, pc * 4, s);
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(s[e] * g0);
        tmem_st32(tmem + kTmS + lane_off + half * 64 + pc * 32, w);
      }
    }
    tmem_st_wait();
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(bar_sready);
    const float* utl = reinterpret_cast<const float*>(smem + kUtlOff);  // U~ [token][dv]
    // outputs of the previous chunk, bf16 pairs, waiting to be stored
    uint32_t opk[16];
    int out_t0 = -1, out_n = 0;
    auto store_out = [&]() {
      if (out_t0 < 0 || !ok) return;
      uint16_t* orow = p.out + (bh * p.T + out_t0 + half * 32) * kDv + d;
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (half * 32 + e < out_n)
          orow[static_cast<size_t>(e) * kDv] = static_cast<uint16_t>((e & 1) ? (opk[e / 2] >> 16) : (opk[e / 2] & 0xFFFFu));
    };
#pragma unroll 1
    for (int c = 0; c < nc; ++c) {
      const int st = c & 1;
      const float* fct = fct_of(c);
      // ---- U^T = U~^T - S W^T, and U'^T = U^T with token i scaled by Gamma_C / Gamma_i ----
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_udone, c & 1, p.status));
      tc_fence_after();
      {
        uint32_t du[32];
        tmem_ld32(tmem + kTmU + lane_off + half * 32, du);
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_utl_full, c & 1, p.status));
        tmem_ld_wait();
        float u[32], up[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          u[e] = utl[(half * 32 + e) * kDv + d] - __uint_as_float(du[e]);
          up[e] = u[e] * fct[kC + half * 32 + e];
        }
        mbar_arrive(bar_utl_empty);  // this thread has read the chunk's U~
        put_row32(utp, half * 4, u);
        put_row32(uptp, half * 4, up);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_uready);
      store_out();  // the previous chunk's outputs, while this chunk's last MMAs run
      // ---- the state's bf16 copy (and the next chunk's scaled state) once D_S is final ----
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_sdone, c & 1, p.status));
      tc_fence_after();
      const bool last = c + 1 == nc;
      // the next chunk's Gamma_C (its stage was loaded ahead)
      float g_next = 1.f;
      if (!last) {
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_full((c + 1) & 1), ((c + 1) >> 1) & 1, p.status));
        g_next = ok ? fct_of(c + 1)[kC - 1] : 1.f;
      }
#pragma unroll 1
      for (int pc = 0; pc < 2; ++pc) {
        uint32_t w[32];
        tmem_ld32(tmem + kTmS + lane_off + half * 64 + pc * 32, w);
        tmem_ld_wait();
        float s[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) s[e] = __uint_as_float(w[e]);
        if (last) {
          if (ok && p.s_final) {
            float4* dst = reinterpret_cast<float4*>(p.s_final + (bh * kDv + d) * kDk + half * 64 + pc * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e) dst[e] = make_float4(s[4 * e], s[4 * e + 1], s[4 * e + 2], s[4 * e + 3]);
          }
        } else {
          put_row32(sbf + half * kSBlk, pc * 4, s);
#pragma unroll
          for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(s[e] * g_next);
          tmem_st32(tmem + kTmS + lane_off + half * 64 + pc * 32, w);
        }
      }
      if (!last) {
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar_sready);
      }
      // ---- O = Gamma_i scale S q_i + (P U)_i from this chunk's output set: the next chunk's
      // products go to the other set, so this read may follow the state's publication ----
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_odone, c & 1, p.status));
      tc_fence_after();
      {
        const uint32_t oset = (c & 1) * kTmOSet;
        uint32_t o1[32], o2[32];
        tmem_ld32(tmem + kTmO1 + oset + lane_off + half * 32, o1);
        tmem_ld32(tmem + kTmO2 + oset + lane_off + half * 32, o2);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float a0 = fct[half * 32 + 2 * e] * p.scale * __uint_as_float(o1[2 * e]) + __uint_as_float(o2[2 * e]);
          const float a1 = fct[half * 32 + 2 * e + 1] * p.scale * __uint_as_float(o1[2 * e + 1]) +
                           __uint_as_float(o2[2 * e + 1]);
          opk[e] = pack_bf16x2(a0, a1);
        }
        out_t0 = c * kC;
        out_n = min(kC, p.T - out_t0);
      }
      tc_fence_before();
      mbar_arrive(bar_empty(st));  // this thread is done with the stage's decay factors
    }
    store_out();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

struct GdnPlan {
  int n_chunks, Tpad;
  size_t off_w, off_u, off_p, off_f, total;
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

GdnPlan plan_gdn(const gated_delta_args* a) {
  GdnPlan pl{};
  pl.n_chunks = (a->T + kC - 1) / kC;
  pl.Tpad = pl.n_chunks * kC;
  const size_t rows = static_cast<size_t>(a->B) * a->Hv * pl.Tpad;
  pl.off_w = 0;
  pl.off_u = align256(pl.off_w + rows * kDk * 2);
  pl.off_p = align256(pl.off_u + rows * kDv * 4);
  pl.off_f = align256(pl.off_p + rows * kC * 2);
  pl.total = align256(pl.off_f + rows * 2 * 4);
  return pl;
}

int fail_gd(int code, const char* msg) { return set_error(code, msg); }

int validate_gdn(const gated_delta_args* a, bool pointers) {
  char msg[200];
  if (!a) return fail_gd(FA_ERR_INVALID_ARG, "gated_delta_prefill: null argument struct");
  if (a->B < 0 || a->T < 0 || a->Hk <= 0 || a->Hv <= 0 || a->Hv % a->Hk != 0) {
    snprintf(msg, sizeof msg, "gated_delta_prefill: need B, T >= 0, Hk, Hv > 0, Hv %% Hk == 0 "
             "(got %d, %d, %d, %d)", a->B, a->T, a->Hk, a->Hv);
    return fail_gd(FA_ERR_INVALID_ARG, msg);
  }
  if (a->dk != kDk || a->dv != kDv) {
    snprintf(msg, sizeof msg, "gated_delta_prefill: dk and dv must be 128 (got %d, %d)", a->dk, a->dv);
    return fail_gd(FA_ERR_UNSUPPORTED, msg);
  }
  if (a->dtype != FA_BF16)
    return fail_gd(FA_ERR_UNSUPPORTED, "gated_delta_prefill: dtype must be FA_BF16");
  if (a->B > 65535 || a->Hv > 65535 ||
      static_cast<long>(a->B) * a->Hv * (static_cast<long>(a->T) + kC) > 2147483647L)
    return fail_gd(FA_ERR_UNSUPPORTED, "gated_delta_prefill: B * Hv * T must fit in int32");
  if (!(a->scale == a->scale) || isinf(a->scale))
    return fail_gd(FA_ERR_INVALID_ARG, "gated_delta_prefill: scale must be finite");
  if (!pointers || a->B == 0 || a->T == 0) return FA_OK;
  if (!a->q || !a->k || !a->v || !a->g || !a->beta || !a->out)
    return fail_gd(FA_ERR_INVALID_ARG, "gated_delta_prefill: null q/k/v/g/beta/out pointer");
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!al16(a->q) || !al16(a->k) || !al16(a->v) || !al16(a->g) || !al16(a->beta) ||
      !al16(a->out) || !al16(a->initial_state) || !al16(a->final_state))
    return fail_gd(FA_ERR_INVALID_ARG, "gated_delta_prefill: tensors must be 16-byte aligned");
  return FA_OK;
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

size_t gated_delta_workspace_size(const gated_delta_args* a) {
  if (validate_gdn(a, false) != FA_OK || a->B == 0 || a->T == 0) return 0;
  return plan_gdn(a).total;
}

int gated_delta_prefill(const gated_delta_args* a, void* stream) {
  int rc = validate_gdn(a, true);
  if (rc != FA_OK || a->B == 0) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (a->T == 0) {
    // no token: the final state is the initial one (or zero)
    if (!a->final_state) return FA_OK;
    const size_t bytes = static_cast<size_t>(a->B) * a->Hv * kDv * kDk * 4;
    cudaError_t e = a->initial_state
                        ? cudaMemcpyAsync(a->final_state, a->initial_state, bytes, cudaMemcpyDeviceToDevice, st)
                        : cudaMemsetAsync(a->final_state, 0, bytes, st);
    if (e != cudaSuccess) return fail_gd(FA_ERR_CUDA, "gated_delta_prefill: state copy failed");
    return FA_OK;
  }
  const GdnPlan pl = plan_gdn(a);
  char msg[200];
  if (!a->workspace || a->workspace_bytes < pl.total) {
    snprintf(msg, sizeof msg, "gated_delta_prefill: workspace of %zu bytes needed (got %zu)",
             pl.total, a->workspace ? a->workspace_bytes : static_cast<size_t>(0));
    return fail_gd(FA_ERR_WORKSPACE, msg);
  }
  if ((reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0)
    return fail_gd(FA_ERR_INVALID_ARG, "gated_delta_prefill: workspace must be 256-byte aligned");
  uint32_t* status = device_status_ptr();
  if (!status) return fail_gd(FA_ERR_CUDA, "gated_delta_prefill: no usable CUDA device");
  uint8_t* ws = static_cast<uint8_t*>(a->workspace);
  GdnParams p{};
  p.q = static_cast<const uint16_t*>(a->q);
  p.k = static_cast<const uint16_t*>(a->k);
  p.v = static_cast<const uint16_t*>(a->v);
  p.g = a->g;
  p.beta = a->beta;
  p.s0 = a->initial_state;
  p.out = static_cast<uint16_t*>(a->out);
  p.s_final = a->final_state;
  p.B = a->B;
  p.T = a->T;
  p.Hk = a->Hk;
  p.Hv = a->Hv;
  p.n_chunks = pl.n_chunks;
  p.Tpad = pl.Tpad;
  p.scale = a->scale;
  p.w_ws = reinterpret_cast<uint16_t*>(ws + pl.off_w);
  p.u_ws = reinterpret_cast<float*>(ws + pl.off_u);
  p.p_ws = reinterpret_cast<uint16_t*>(ws + pl.off_p);
  p.f_ws = reinterpret_cast<float*>(ws + pl.off_f);
  p.status = status;

  CUtensorMap tw, tq, tk, tp, tv;
  const uint64_t rows = static_cast<uint64_t>(a->B) * a->Hv * pl.Tpad;
  {
    const uint64_t dims[2] = {kDk, rows}, str[1] = {kDk * 2};
    const uint32_t box[2] = {64, kC};
    if (!encode_tiled(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.w_ws, dims, str, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return fail_gd(FA_ERR_CUDA, "gated_delta_prefill: tensor map (W) rejected");
  }
  {
    const uint64_t dims[2] = {kC, rows}, str[1] = {kC * 2};
    const uint32_t box[2] = {64, kC};
    if (!encode_tiled(&tp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.p_ws, dims, str, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return fail_gd(FA_ERR_CUDA, "gated_delta_prefill: tensor map (P) rejected");
  }
  {
    const uint64_t dims[3] = {kDk, static_cast<uint64_t>(a->T), static_cast<uint64_t>(a->B) * a->Hk};
    const uint64_t str[2] = {kDk * 2, static_cast<uint64_t>(a->T) * kDk * 2};
    const uint32_t box[3] = {64, kC, 1};
    if (!encode_tiled(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a->q, dims, str, box,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a->k, dims, str, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return fail_gd(FA_ERR_CUDA, "gated_delta_prefill: tensor map (Q/K) rejected");
  }
  {
    const uint64_t dims[3] = {kDv, static_cast<uint64_t>(a->T), static_cast<uint64_t>(a->B) * a->Hv};
    const uint64_t str[2] = {kDv * 2, static_cast<uint64_t>(a->T) * kDv * 2};
    const uint32_t box[3] = {64, kC, 1};
    if (!encode_tiled(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a->v, dims, str, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return fail_gd(FA_ERR_CUDA, "gated_delta_prefill: tensor map (V) rejected");
  }
  cudaError_t e = ensure_smem_limit(gdn_prep_kernel, kPrepSmem);
  if (e == cudaSuccess) e = ensure_smem_limit(gdn_state_kernel, kStateSmem);
  if (e != cudaSuccess) return fail_gd(FA_ERR_CUDA, "gated_delta_prefill: shared memory limit");
  gdn_prep_kernel<<<dim3(pl.n_chunks, a->Hv, a->B), kPrepThreads, kPrepSmem, st>>>(tq, tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail_gd(FA_ERR_CUDA, "gated_delta_prefill: chunk kernel launch failed");
  gdn_state_kernel<<<dim3(a->Hv, a->B), kStateThreads, kStateSmem, st>>>(tw, tq, tk, tp, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail_gd(FA_ERR_CUDA, "gated_delta_prefill: state kernel launch failed");
  return FA_OK;
}

}  // extern "C"

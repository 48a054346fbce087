// decode.cu -- split-KV paged grouped-query decode (one query token per sequence).
//
// The work is HBM-bound (about 4 flops per byte of K/V for 4 query heads per kv head), so
// it runs on the CUDA cores and is shaped for the memory system rather than the tensor
// cores.  Grid = (KV chunk, kv head, sequence); a chunk is `chunk` consecutive tokens.  All
// G query heads that share the kv head are processed together, so each K/V byte is read
// once ("GQA optimization", llama.cpp PR "CUDA: fix FA occupancy, optimize tile kernel").
// Each of the 4 warps streams its own 16-token blocks through a private 2-slot ring: one
// lane issues cp.async.bulk copies of the contiguous page slabs (16 tokens x D x 2 bytes of
// the [num_pages, Hkv, page_size, D] cache) and the warp computes while the next block
// lands.  Scores use a per-lane slice of D with a reduce-scatter across lanes; the online
// softmax keeps a running max and sum per head.  Each CTA writes its chunk's normalised
// partial output and log-sum-exp; merge.cu combines the chunks.
#include <math.h>

#include "internal.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kBT = 16;     // tokens per block
constexpr int kStages = 2;  // ring slots per warp
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct DecLayout {
  static constexpr int kBlockBytes = kBT * D * 2;  // one K (or V) block
  static constexpr int kSlot = 2 * kBlockBytes;
  static constexpr int kRing = kWarps * kStages * kSlot;
};

// 16-bit pairs (bf16, or fp16 when F16) -> fp32
template <bool F16>
__device__ __forceinline__ void x2_to_f32(uint32_t w, float& lo, float& hi) {
  if constexpr (F16) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
    lo = f.x;
    hi = f.y;
  } else {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
  }
}

template <int DPL, bool F16>
__device__ __forceinline__ void load_row_slice(const uint8_t* row, int lane, float (&f)[DPL]) {
  if constexpr (DPL == 2) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(row + lane * 4);
    x2_to_f32<F16>(w, f[0], f[1]);
  } else if constexpr (DPL == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(row + lane * 8);
    x2_to_f32<F16>(w.x, f[0], f[1]);
    x2_to_f32<F16>(w.y, f[2], f[3]);
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(row + lane * 16);
    x2_to_f32<F16>(w.x, f[0], f[1]);
    x2_to_f32<F16>(w.y, f[2], f[3]);
    x2_to_f32<F16>(w.z, f[4], f[5]);
    x2_to_f32<F16>(w.w, f[6], f[7]);
  }
}

template <int D, int G, bool F16>
__global__ void __launch_bounds__(kThreads) decode_kernel(const DecodeParams p) {
  constexpr int DPL = D / 32;         // dims per lane
  constexpr int V = kBT * G;          // partial dot products per lane per block
  constexpr int R = V >= 32 ? V / 32 : 1;  // complete scores per lane after the reduce
  using L = DecLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kWarps][kStages];
  __shared__ float pbuf[kWarps][kBT][G];
  __shared__ float abuf[kWarps][G];

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int c = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int len = p.seq_lens[b];
  if (len < 0 || len > p.max_pages * p.page_size) {
    if (threadIdx.x == 0) record_error(p.status, kDevBounds);
    return;
  }
  const int t_start = c * p.chunk;
  if (t_start >= len) return;
  const int t_stop = min(len, t_start + p.chunk);
  const int n_blocks = (t_stop - t_start + kBT - 1) / kBT;
  const int my_blocks = warp < n_blocks ? (n_blocks - warp + kWarps - 1) / kWarps : 0;

  uint8_t* ring = smem + warp * (kStages * L::kSlot);
  const uint32_t ring_s = smem_addr(ring);
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_addr(&bars[warp][s]), 1);
    fence_barrier_init();
  }
  __syncwarp();

  // q pre-scaled into log2 units: scores come out ready for exp2.
  float q[G][DPL];
  {
    const uint8_t* qrow = static_cast<const uint8_t*>(p.q) +
                          (static_cast<size_t>(b) * p.Hq + hk * G) * D * 2;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      load_row_slice<DPL, F16>(qrow + g * D * 2, lane, q[g]);
#pragma unroll
      for (int d = 0; d < DPL; ++d) q[g][d] *= p.scale_log2;
    }
  }

  const int32_t* table = p.page_table + static_cast<size_t>(b) * p.max_pages;
  const uint8_t* kbase = static_cast<const uint8_t*>(p.k_pages);
  const uint8_t* vbase = static_cast<const uint8_t*>(p.v_pages);
  const size_t head_stride = static_cast<size_t>(p.page_size) * D * 2;  // one page of one head

  // Lane 0: start the copy of this warp's i-th block into slot i % kStages.  Pieces whose
  // page id is out of range are not read; they are zero-filled and the error is recorded.
  auto issue = [&](int i) {
    const int slot = i % kStages;
    const uint32_t bar = smem_addr(&bars[warp][slot]);
    const uint32_t dk = ring_s + slot * L::kSlot, dv = dk + L::kBlockBytes;
    const int tok0 = t_start + (warp + i * kWarps) * kBT;
    const int per = p.page_size >= kBT ? kBT : p.page_size;  // tokens per piece
    const int pieces = kBT / per;
    const uint32_t piece_bytes = per * D * 2;
    uint32_t bytes = 0;
    int page_ids[kBT];
#pragma unroll 1
    for (int k = 0; k < pieces; ++k) {
      const int tok = tok0 + k * per;
      int page = -1;
      if (tok < t_stop) {
        page = table[tok / p.page_size];
        if (page < 0 || page >= p.num_pages) {
          record_error(p.status, kDevBounds);
          page = -1;
        }
      }
      page_ids[k] = page;
      if (page >= 0) bytes += 2 * piece_bytes;
    }
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, bytes);
#pragma unroll 1
    for (int k = 0; k < pieces; ++k) {
      const int tok = tok0 + k * per;
      if (page_ids[k] >= 0) {
        const size_t off = (static_cast<size_t>(page_ids[k]) * p.Hkv + hk) * head_stride +
                           static_cast<size_t>(tok % p.page_size) * D * 2;
        bulk_load(dk + k * piece_bytes, kbase + off, piece_bytes, bar);
        bulk_load(dv + k * piece_bytes, vbase + off, piece_bytes, bar);
      } else {
        uint4* zk = reinterpret_cast<uint4*>(ring + slot * L::kSlot + k * piece_bytes);
        uint4* zv = reinterpret_cast<uint4*>(ring + slot * L::kSlot + L::kBlockBytes + k * piece_bytes);
        for (uint32_t e = 0; e < piece_bytes / 16; ++e) {
          zk[e] = make_uint4(0, 0, 0, 0);
          zv[e] = make_uint4(0, 0, 0, 0);
        }
      }
    }
  };

  if (lane == 0)
    for (int i = 0; i < min(kStages, my_blocks); ++i) issue(i);
  __syncwarp();  // zero-filled pieces are written by lane 0 with ordinary stores

  // Lane l holds, after the reduce, token (l >> 1) and heads (l & 1) * R + k, k < R
  // (for G == 1 lanes l and l ^ 1 hold the same value).
  float m_run[R], l_run[R];
#pragma unroll
  for (int k = 0; k < R; ++k) {
    m_run[k] = -INFINITY;
    l_run[k] = 0.f;
  }
  float o[G][DPL];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int d = 0; d < DPL; ++d) o[g][d] = 0.f;

  const int my_tok = lane >> 1;
  const int g_base = (G >= 2) ? (lane & 1) * R : 0;
  bool ok = true;
#pragma unroll 1
  for (int i = 0; i < my_blocks; ++i) {
    const int slot = i % kStages;
    ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&bars[warp][slot]), (i / kStages) & 1, p.status));
    if (!ok) break;
    const uint8_t* Ks = ring + slot * L::kSlot;
    const uint8_t* Vs = Ks + L::kBlockBytes;
    const int tok0 = t_start + (warp + i * kWarps) * kBT;
    const int n_valid = min(kBT, t_stop - tok0);

    // ---- scores: partial dot products over this lane's D slice ----
    float acc[V];
#pragma unroll
    for (int t = 0; t < kBT; ++t) {
      float kf[DPL];
      load_row_slice<DPL, F16>(Ks + t * D * 2, lane, kf);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float a = 0.f;
#pragma unroll
        for (int d = 0; d < DPL; ++d) a = fmaf(q[g][d], kf[d], a);
        acc[t * G + g] = a;
      }
    }
    // ---- reduce-scatter across the warp: each level halves the values a lane keeps ----
    int cnt = V;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
      if (cnt > 1) {
        const int half = cnt / 2;
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int k = 0; k < V / 2; ++k) {
          if (k < half) {
            const float send = upper ? acc[k] : acc[k + half];
            const float keep = upper ? acc[k + half] : acc[k];
            acc[k] = keep + __shfl_xor_sync(0xffffffffu, send, m);
          }
        }
        cnt = half;
      } else {
        acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], m);
      }
    }
    // ---- online softmax over this block ----
    const bool tok_ok = my_tok < n_valid;
    float x[R], alpha[R];
#pragma unroll
    for (int k = 0; k < R; ++k) {
      x[k] = tok_ok ? acc[k] : -INFINITY;
      float bm = x[k];
#pragma unroll
      for (int m = 2; m <= 16; m <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, m));
      const float m_new = fmaxf(m_run[k], bm);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      alpha[k] = exp2_approx(m_run[k] - m_use);
      m_run[k] = m_new;
      const float pe = exp2_approx(x[k] - m_use);
      l_run[k] = l_run[k] * alpha[k] + pe;
      pbuf[warp][my_tok][g_base + k] = pe;
      if (my_tok == 0) abuf[warp][g_base + k] = alpha[k];
    }
    __syncwarp();
    // ---- O = alpha * O + P V ----
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float a = abuf[warp][g];
#pragma unroll
      for (int d = 0; d < DPL; ++d) o[g][d] *= a;
    }
#pragma unroll
    for (int t = 0; t < kBT; ++t) {
      float vf[DPL];
      load_row_slice<DPL, F16>(Vs + t * D * 2, lane, vf);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float pg = pbuf[warp][t][g];
#pragma unroll
        for (int d = 0; d < DPL; ++d) o[g][d] = fmaf(pg, vf[d], o[g][d]);
      }
    }
    __syncwarp();
    if (lane == 0 && i + kStages < my_blocks) issue(i + kStages);
  }

  // ---- combine the warps' states, then write this chunk's partial state ----
  // per-head sums of the lane-partial l over the 16 token lanes (bits 1-4 of the lane id;
  // for G == 1 lanes l and l^1 hold the same token, so summing over bits 1-4 counts each
  // token once)
#pragma unroll
  for (int k = 0; k < R; ++k) {
#pragma unroll
    for (int m = 2; m <= 16; m <<= 1) l_run[k] += __shfl_xor_sync(0xffffffffu, l_run[k], m);
  }
  ok = __syncthreads_and(ok);
  if (!ok) return;
  float* mbuf = reinterpret_cast<float*>(smem);  // [kWarps][G]
  float* lbuf = mbuf + kWarps * G;               // [kWarps][G]
  float* obuf = lbuf + kWarps * G;               // [kWarps][G][D]
  if (lane < 2 && (G >= 2 || lane == 0)) {
#pragma unroll
    for (int k = 0; k < R; ++k) {
      mbuf[warp * G + g_base + k] = m_run[k];
      lbuf[warp * G + g_base + k] = l_run[k];
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int d = 0; d < DPL; ++d) obuf[(warp * G + g) * D + lane * DPL + d] = o[g][d];
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
    const int g = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mbuf[w * G + g]);
    float num = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float s = exp2_approx(mbuf[w * G + g] - M);
        num = fmaf(s, obuf[(w * G + g) * D + d], num);
        den = fmaf(s, lbuf[w * G + g], den);
      }
    }
    const size_t row = static_cast<size_t>(b) * p.Hq + hk * G + g;
    p.o_part[(row * p.n_chunks + c) * D + d] = den > 0.f ? num / den : 0.f;
    if (d == 0) p.lse_part[row * p.n_chunks + c] = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
  }
}

template <int D, int G>
cudaError_t launch_impl(const DecodeParams& p, cudaStream_t stream) {
  using L = DecLayout<D>;
  auto kern = p.f16 ? decode_kernel<D, G, true> : decode_kernel<D, G, false>;
  const int smem = L::kRing;
  cudaError_t e = ensure_smem_limit(kern, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.n_chunks, p.Hkv, p.B);
  kern<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
#define FA_DEC_CASE(DD, GG) \
  if (p.D == DD && p.G == GG) return launch_impl<DD, GG>(p, stream);
  FA_DEC_CASE(64, 1) FA_DEC_CASE(64, 2) FA_DEC_CASE(64, 4) FA_DEC_CASE(64, 8) FA_DEC_CASE(64, 16)
  FA_DEC_CASE(128, 1) FA_DEC_CASE(128, 2) FA_DEC_CASE(128, 4) FA_DEC_CASE(128, 8)
  FA_DEC_CASE(256, 1) FA_DEC_CASE(256, 2) FA_DEC_CASE(256, 4)
#undef FA_DEC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fa

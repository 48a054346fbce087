// prefill_f32.cu -- attention for fp32 inputs, in fp32 on the CUDA cores.
//
// fp32 inputs keep their range and precision: nothing is narrowed to a 16-bit type (an fp16
// operand overflows above 65504 and loses precision below 6e-5; tf32 keeps the range but
// only ten mantissa bits).  The operation is the same as the tensor-core path's: softmax
// attention with grouped-query heads, bottom-right causal masking and an additive mask
// (llama.cpp PR "CUDA: fix FA occupancy, optimize tile kernel", opening paragraphs: the
// attention the FA kernels compute), evaluated with an online softmax in fp32: one warp per
// query row, each lane holding D/32 of the row's dimensions, every score reduced across the
// warp, the running max, sum and output updated key by key.  The output is kept normalised
// (a weighted mean of the values seen so far), so it never exceeds the largest |v|: values
// near the fp32 limit do not overflow the accumulator.  It serves the small fp32
// problems such inputs come with; bulk throughput is the 16-bit paths' business.
#include <math.h>

#include "internal.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kWarps = 4;

template <int D>
__global__ void __launch_bounds__(kWarps * 32) attn_f32_kernel(const PrefillParams p) {
  constexpr int DPL = D / 32;  // dimensions per lane
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const long rows = static_cast<long>(p.B) * p.Hq * p.Lq;
  const long r = static_cast<long>(blockIdx.x) * kWarps + warp;
  if (r >= rows) return;
  const int i = static_cast<int>(r % p.Lq);
  const int h = static_cast<int>((r / p.Lq) % p.Hq);
  const int b = static_cast<int>(r / (static_cast<long>(p.Lq) * p.Hq));
  const int hk = h / p.G;
  const int key_lim = p.causal ? min(p.Lkv, i + (p.Lkv - p.Lq) + 1) : p.Lkv;
  const float scale = p.scale_log2 * 0.69314718055994530942f;  // natural-log units
  const char* mrow = nullptr;
  if (p.mask) {
    const int mb = p.mask_batches == 1 ? 0 : b;
    mrow = static_cast<const char*>(p.mask) +
           ((static_cast<size_t>(mb) * p.Lq + i) * static_cast<size_t>(p.Lkv)) * (p.mask_is_bf16 ? 2 : 4);
  }
  const float* qrow = static_cast<const float*>(p.q) + static_cast<size_t>(r) * D;
  const float* kbase = static_cast<const float*>(p.k) + (static_cast<size_t>(b) * p.Hkv + hk) * p.Lkv * D;
  const float* vbase = static_cast<const float*>(p.v) + (static_cast<size_t>(b) * p.Hkv + hk) * p.Lkv * D;
  float q[DPL], o[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) {
    q[e] = qrow[lane * DPL + e] * scale;
    o[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int j = 0; j < key_lim; ++j) {
    const float* kr = kbase + static_cast<size_t>(j) * D + lane * DPL;
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) s = fmaf(q[e], kr[e], s);
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) s += __shfl_xor_sync(0xffffffffu, s, w);
    if (mrow)
      s += p.mask_is_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(mrow)[j])
                          : reinterpret_cast<const float*>(mrow)[j];
    if (s == -INFINITY) continue;  // a masked key (every lane agrees)
    const float m_new = fmaxf(m, s);
    const float la = l * expf(m - m_new);  // 0 while m is -inf
    const float pj = expf(s - m_new);
    const float l_new = la + pj;
    const float w_old = la / l_new, w_new = pj / l_new;
    m = m_new;
    l = l_new;
    const float* vr = vbase + static_cast<size_t>(j) * D + lane * DPL;
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[e] = fmaf(w_new, vr[e], o[e] * w_old);
  }
  float* orow = static_cast<float*>(p.out) + static_cast<size_t>(r) * D;
#pragma unroll
  for (int e = 0; e < DPL; ++e) orow[lane * DPL + e] = l > 0.f ? o[e] : 0.f;
  if (lane == 0 && p.lse) p.lse[r] = l > 0.f ? m + logf(l) : -INFINITY;
}

}  // namespace

cudaError_t launch_prefill_f32(const PrefillParams& p, cudaStream_t stream) {
  const long rows = static_cast<long>(p.B) * p.Hq * p.Lq;
  if (rows <= 0) return cudaSuccess;
  const long ctas = (rows + kWarps - 1) / kWarps;
  if (ctas > 0x7fffffffL) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(ctas));
  switch (p.D) {
    case 64: attn_f32_kernel<64><<<grid, kWarps * 32, 0, stream>>>(p); break;
    case 128: attn_f32_kernel<128><<<grid, kWarps * 32, 0, stream>>>(p); break;
    case 256: attn_f32_kernel<256><<<grid, kWarps * 32, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace fa

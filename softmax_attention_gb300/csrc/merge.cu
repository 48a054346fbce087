// merge.cu -- combination of attention states computed over disjoint key ranges.
//
// For one output row with partial states (o_s, lse_s), s < n:
//   lse = ln sum_s exp(lse_s)        out = sum_s exp(lse_s - lse) * o_s
// which is the softmax over the union of the ranges.  Parts with lse_s = -inf (no key) get
// weight 0; a row with no part, or only such parts, gives out = 0 and lse = -inf.  This is
// the combine step of split-KV decoding and of a prefill whose KV loop is split across CTAs.
#include <math.h>

#include "internal.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.44269504088896340736f;

__device__ __forceinline__ void store4(void* out, Dtype t, size_t idx, float4 v) {
  if (t == Dtype::FP32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + idx) = v;
  } else if (t == Dtype::BF16) {
    uint2 w = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + idx) = w;
  } else {
    uint2 w = make_uint2(pack_f16x2(v.x, v.y), pack_f16x2(v.z, v.w));
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + idx) = w;
  }
}

// One CTA (4 warps) per (row, 128-column chunk).  Every warp reduces the row's log-sum-exps
// (cheap, L1-resident); warp w accumulates the parts s = w, w+4, ... of the chunk (lane l
// reads the 16-byte vector l, part loop unrolled so several loads are in flight), and the
// four partial sums are combined through shared memory.  Splitting the row across CTAs keeps
// few-row, many-part merges (a short query chunk split over the KV loop) parallel.
constexpr int kMergeWarps = 4;
constexpr int kChunkCols = 128;

__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const MergeParams p) {
  __shared__ float4 part[kMergeWarps][32];
  const int row = blockIdx.x;
  const int v = blockIdx.y * 32 + threadIdx.x % 32;  // float4 index in the row
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  int n = p.max_splits;
  if (p.n_splits) {
    n = p.n_splits[row];
  } else if (p.seq_lens) {
    const int len = p.seq_lens[row / p.rows_per_seq];
    n = len > 0 ? (len + p.chunk - 1) / p.chunk : 0;
  }
  n = max(0, min(n, p.max_splits));
  const float* lrow = p.lse_part + static_cast<size_t>(row) * p.max_splits;
  float m = -INFINITY;
  for (int s = lane; s < n; s += 32) m = fmaxf(m, lrow[s]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float sum = 0.f;
  if (m != -INFINITY)
    for (int s = lane; s < n; s += 32) sum += exp2_approx((lrow[s] - m) * kLog2e);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float lse = (m == -INFINITY) ? -INFINITY : m + logf(sum);
  const float* orow = p.o_part + static_cast<size_t>(row) * p.max_splits * p.D;
  const bool in_row = v < p.D / 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (in_row && m != -INFINITY) {
#pragma unroll 4
    for (int s = warp; s < n; s += kMergeWarps) {
      const float ls = lrow[s];
      const float w = (ls == -INFINITY) ? 0.f : exp2_approx((ls - lse) * kLog2e);
      const float4 x = reinterpret_cast<const float4*>(orow + static_cast<size_t>(s) * p.D)[v];
      acc.x = fmaf(w, x.x, acc.x);
      acc.y = fmaf(w, x.y, acc.y);
      acc.z = fmaf(w, x.z, acc.z);
      acc.w = fmaf(w, x.w, acc.w);
    }
  }
  part[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && in_row) {
    float4 t = part[0][lane];
#pragma unroll
    for (int w = 1; w < kMergeWarps; ++w) {
      t.x += part[w][lane].x;
      t.y += part[w][lane].y;
      t.z += part[w][lane].z;
      t.w += part[w][lane].w;
    }
    store4(p.out, p.out_dtype, static_cast<size_t>(row) * p.D + 4 * v, t);
  }
  if (threadIdx.x == 0 && blockIdx.y == 0 && p.lse) p.lse[row] = lse;
}

__global__ void f32_to_f16_kernel(const float* __restrict__ src, __half* __restrict__ dst, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = __float2half_rn(src[i]);
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  if (p.D > 512 || p.D % 4 != 0) return cudaErrorInvalidValue;
  dim3 grid(p.rows, (p.D + kChunkCols - 1) / kChunkCols);
  merge_kernel<<<grid, kMergeWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_f32_to_f16(const float* src, void* dst, size_t n, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  size_t blocks = (n + threads - 1) / threads;
  if (blocks > 4096) blocks = 4096;
  f32_to_f16_kernel<<<(unsigned)blocks, threads, 0, stream>>>(src, static_cast<__half*>(dst), n);
  return cudaGetLastError();
}

}  // namespace fa

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

// kMergeWarps warps per CTA; W of them (1, 2, 4 or 8, from the largest part count) share one
// row, so a CTA merges kMergeWarps / W rows.  Every warp of a row reduces the row's
// log-sum-exps (a few loads, L1-resident), then accumulates the parts s = k, k + W, ... of
// the row over all D columns: lane l holds the 16-byte vectors l, l + 32, ... (VPL of them).
// Parts are taken in batches of kBatch whose loads are all issued before their
// multiply-adds, and the first batch is issued before the log-sum-exp reduction, so that its
// latency overlaps it.  With W > 1 the warps' sums are combined through shared memory.  Few
// parts: one warp per row and eight rows per CTA; many parts: eight warps on one row.
constexpr int kMergeWarps = 8;

template <int VPL>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const MergeParams p, int W) {
  extern __shared__ float4 part[];  // [kMergeWarps][VPL * 32] when W > 1
  constexpr int kBatch = 8 / VPL;   // parts per batch: 8 float4 per lane in flight
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int rows_per_cta = kMergeWarps / W;
  const int row = blockIdx.x * rows_per_cta + warp / W;
  const int k = warp % W;  // this warp's share of the row's parts
  const bool live = row < p.rows;
  const int nv = p.D / 4;  // float4 per row
  float4 acc[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  float lse = -INFINITY;
  if (live) {
    int n = p.max_splits;
    if (p.n_splits) {
      n = p.n_splits[row];
    } else if (p.seq_lens) {
      const int len = p.seq_lens[row / p.rows_per_seq];
      n = len > 0 ? (len + p.chunk - 1) / p.chunk : 0;
    }
    n = max(0, min(n, p.max_splits));
    const float* lrow = p.lse_part + static_cast<size_t>(row) * p.max_splits;
    const float4* orow = reinterpret_cast<const float4*>(p.o_part + static_cast<size_t>(row) * p.max_splits * p.D);
    auto load_batch = [&](int s0, float4 (&xv)[kBatch][VPL]) {
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int s = s0 + u * W;
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          const int v = lane + 32 * j;
          xv[u][j] = (s < n && v < nv) ? orow[static_cast<size_t>(s) * nv + v] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    };
    float4 xv[kBatch][VPL];
    load_batch(k, xv);
    float m = -INFINITY;
    for (int s = lane; s < n; s += 32) m = fmaxf(m, lrow[s]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float sum = 0.f;
    if (m != -INFINITY)
      for (int s = lane; s < n; s += 32) sum += exp2_approx((lrow[s] - m) * kLog2e);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    lse = (m == -INFINITY) ? -INFINITY : m + logf(sum);
    if (m != -INFINITY) {
      for (int s0 = k;; ) {
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int s = s0 + u * W;
          const float ls = s < n ? lrow[s] : -INFINITY;
          const float w = (ls == -INFINITY) ? 0.f : exp2_approx((ls - lse) * kLog2e);
#pragma unroll
          for (int j = 0; j < VPL; ++j) {
            acc[j].x = fmaf(w, xv[u][j].x, acc[j].x);
            acc[j].y = fmaf(w, xv[u][j].y, acc[j].y);
            acc[j].z = fmaf(w, xv[u][j].z, acc[j].z);
            acc[j].w = fmaf(w, xv[u][j].w, acc[j].w);
          }
        }
        s0 += kBatch * W;
        if (s0 >= n) break;
        load_batch(s0, xv);
      }
    }
  }
  if (W > 1) {
#pragma unroll
    for (int j = 0; j < VPL; ++j) part[warp * (VPL * 32) + j * 32 + lane] = acc[j];
    __syncthreads();
    if (k != 0) return;
    for (int w2 = 1; w2 < W; ++w2) {
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const float4 t = part[(warp + w2) * (VPL * 32) + j * 32 + lane];
        acc[j].x += t.x;
        acc[j].y += t.y;
        acc[j].z += t.z;
        acc[j].w += t.w;
      }
    }
  }
  if (!live) return;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int v = lane + 32 * j;
    if (v < nv) store4(p.out, p.out_dtype, static_cast<size_t>(row) * p.D + 4 * v, acc[j]);
  }
  if (lane == 0 && p.lse) p.lse[row] = lse;
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  if (p.D > 512 || p.D % 4 != 0) return cudaErrorInvalidValue;
  const int W = p.max_splits <= 8 ? 1 : p.max_splits <= 16 ? 2 : p.max_splits <= 32 ? 4 : 8;
  const int rows_per_cta = kMergeWarps / W;
  const unsigned grid = static_cast<unsigned>((p.rows + rows_per_cta - 1) / rows_per_cta);
  const int vpl = (p.D / 4 + 31) / 32;
  const size_t smem = W > 1 ? static_cast<size_t>(kMergeWarps) * vpl * 32 * sizeof(float4) : 0;
  switch (vpl) {
    case 1: merge_kernel<1><<<grid, kMergeWarps * 32, smem, stream>>>(p, W); break;
    case 2: merge_kernel<2><<<grid, kMergeWarps * 32, smem, stream>>>(p, W); break;
    case 3: merge_kernel<3><<<grid, kMergeWarps * 32, smem, stream>>>(p, W); break;
    default: merge_kernel<4><<<grid, kMergeWarps * 32, smem, stream>>>(p, W); break;
  }
  return cudaGetLastError();
}

}  // namespace fa

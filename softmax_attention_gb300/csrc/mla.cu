// mla.cu -- MLA paged decode in the latent (absorbed) form on sm_103a.
//
// One compressed matrix ckv serves as both K and V and a separate rope part kpe adds
// q_pe . kpe_t to every score (flashinfer PR "perf: FlashAttention-3 style MLA
// PageAttention", change list item 4):
//   s_t = scale * (q_nope . ckv_t + q_pe . kpe_t),   out = softmax(s) . ckv
// with 64 query heads sharing one latent head (Dc = 512, Dr = 64).
//
// One CTA handles one chunk of one sequence's tokens, streamed through a ring of 32-token
// stages; each stage holds the 576-wide [ckv | kpe] rows of its tokens as nine
// 128-byte-swizzled 64-column blocks.  With page_size 1 (the flashinfer PR's results section)
// rows are gathered through the page table with 16-byte cp.async copies by a producer
// warpgroup, written at their swizzled addresses (LDGSTS-style gathers; measured on GB300
// they move these 1152-byte rows faster than TMA tile::gather4).  With pages of 8, 16 or a
// multiple of 32 tokens a full stage is whole page slices, copied by 2-D TMA boxes into the
// same layout.  Like the flashinfer design the ring is shared by the K and V roles (one
// pipeline, small tiles, several stages in flight), but the MMAs are Blackwell's:
//   S  = Q [64 heads x 576] . KV^T         tcgen05 M=64 (heads), N=64 tokens (the two
//                                           32-token stages of a tile), S in TMEM
//   O^T += ckv^T [512 x tokens] . P^T       tcgen05 M=128 (latent dims, four blocks),
//                                           N=64 heads, A = the same ckv stage read
//                                           MN-major, B = P^T staged in shared memory
// so O (64 x 512 fp32) lives in 256 tensor-memory columns as four 128-lane blocks and the
// PV product runs at full tensor rate.  Softmax: two threads per head row (the M=64 S layout
// puts heads 16q..16q+15 in lanes 32q..32q+15; lanes 32q+16.. take the second half of each
// tile's tokens), online max/sum with O rescaled only when a head's running max grows by
// more than 2^8.  A CTA that owns a whole sequence writes its final output and log-sum-exp;
// one that owns a chunk writes the chunk's normalised partial output and log-sum-exp, and
// merge.cu combines the chunks.
//
// Warp roles (288 threads): warps 0-3 softmax + epilogue, warps 4-7 producer (row ids and
// cp.async gathers), warp 8 MMA issuer and tensor-memory owner.
#include <math.h>

#include "internal.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kH = 64;
constexpr int kDc = 512;
constexpr int kDr = 64;
constexpr int kBlocks = (kDc + kDr) / 64;  // nine 64-column blocks per token row
constexpr int kHalf = 32;                  // tokens per ring stage
constexpr int kTile = 64;                  // tokens per softmax tile (two stages)
constexpr int kStages = 4;
constexpr int kThreads = 288;
constexpr int kProducerThreads = 128;
constexpr int kMmaWarp = 8;

constexpr int kMaxChunk = 2048;            // tokens per CTA: 512, 1024 or 2048
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;

constexpr int kQBytes = kH * (kDc + kDr) * 2;    // 73728
constexpr int kBlk = kHalf * 128;                // one 64-column block of one stage
constexpr int kStageBytes = kBlocks * kBlk;      // 36864
// The ring holds two tiles, each [9 blocks][64 rows][128 B]: the two 32-token stages of tile
// t (2t, 2t+1) are the first and second 32 rows of every block of ring tile t % 2, so one
// N=64 MMA covers a tile, and a tile's eight ckv blocks are one dense 64 KB region.
constexpr int kBlockStride = kTile * 128;        // 8192: block to block within a tile
constexpr int kTileBytes = kBlocks * kBlockStride;  // 73728: ring tile to ring tile
constexpr int kPBytes = kH * kTile * 2;          // 8192
constexpr int kQOff = 0;
constexpr int kKVOff = kQOff + kQBytes;
constexpr int kPOff = kKVOff + 2 * kTileBytes;
static_assert(2 * kTileBytes == kStages * kStageBytes, "two tiles of two stages");
constexpr int kBarOff = kPOff + kPBytes;
// q_full, kv_full[S], kv_empty[S], s_full[2], p_full, o_full, mma_done
constexpr int kNumBars = 1 + 2 * kStages + 2 + 3;
constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 64 * 4 * 2 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kTmemO = 0;      // O^T: 4 blocks x 64 columns
constexpr uint32_t kTmemS = 256;    // S buffers: 2 x 64 columns

__device__ __forceinline__ bool softmax_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Adds `bytes` to the barrier's expected transaction count without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    mla_kernel(const __grid_constant__ CUtensorMap tm_qn, const __grid_constant__ CUtensorMap tm_qp,
               const __grid_constant__ CUtensorMap tm_ckv, const __grid_constant__ CUtensorMap tm_kpe,
               const MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_addr(smem);
  const uint32_t sQ = s_base + kQOff, sKV = s_base + kKVOff, sP = s_base + kPOff;
  const uint32_t bars = s_base + kBarOff;
  const uint32_t bar_q = bars;
  auto bar_full = [&](int s) { return bars + 8u * (1 + s); };
  auto bar_empty = [&](int s) { return bars + 8u * (1 + kStages + s); };
  auto bar_s = [&](int b) { return bars + 8u * (1 + 2 * kStages + b); };
  const uint32_t bar_p = bars + 8u * (3 + 2 * kStages);
  const uint32_t bar_o = bars + 8u * (4 + 2 * kStages);
  const uint32_t bar_done = bars + 8u * (5 + 2 * kStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + kNumBars * 8);
  float* alpha_s = reinterpret_cast<float*>(smem + kBarOff + kNumBars * 8 + 16);
  float* stat_s = alpha_s + 64;  // [0..63]: l per head (epilogue)

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Each CTA takes one group of up to 64 heads (hb .. hb + hv - 1) of one work item; items
  // are whole sequences first, then the chunks of the split ones.  Head rows past H read as
  // zero and are not written.
  const int n_groups = (p.H + kH - 1) / kH;
  const int bx = blockIdx.x / n_groups;
  const int hb = (blockIdx.x % n_groups) * kH, hv = min(kH, p.H - hb);
  const bool direct = bx < p.n_whole;
  const int b = direct ? bx : p.n_whole + (bx - p.n_whole) / p.n_chunks;
  const int c = direct ? 0 : (bx - p.n_whole) % p.n_chunks;
  const int chunk = direct ? p.whole_chunk : p.chunk;
  const int len = p.seq_lens[b];
  if (len < 0 || len > p.max_pages * p.page_size) {
    if (threadIdx.x == 0) record_error(p.status, kDevBounds);
    return;
  }
  const int t_start = c * chunk;
  if (t_start >= len) {
    // an empty sequence still owns its final output when this launch writes it directly
    if (direct) {
      const size_t r0 = static_cast<size_t>(b) * p.H + hb;
      for (int i = threadIdx.x; i < hv * kDc / 8; i += kThreads)
        reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + r0 * kDc)[i] = make_uint4(0, 0, 0, 0);
      if (threadIdx.x < hv && p.lse) p.lse[r0 + threadIdx.x] = -INFINITY;
    }
    return;
  }
  const int t_stop = min(len, t_start + chunk);
  const int n_tiles = (t_stop - t_start + kTile - 1) / kTile;
  const int n_stages = 2 * n_tiles;  // every tile is two 32-token stages

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full(s), kProducerThreads);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_s(0), 1);
    mbar_init(bar_s(1), 1);
    mbar_init(bar_p, 128);
    mbar_init(bar_o, 1);
    mbar_init(bar_done, 1);
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

  if (warp >= 4 && warp < kMmaWarp) {
    // ----------------------------------- producer ----------------------------------------
    // Producer warp pw copies tokens 8pw..8pw+7 of every 32-token stage: per token two
    // 512-byte halves of the ckv row (lane l copies 16-byte chunk l of the half, so a warp
    // instruction reads 512 contiguous bytes) and its 128-byte kpe row.
    const int pw = warp - 4;
    const int32_t* table = p.page_table + static_cast<size_t>(b) * p.max_pages;
    const int n_rows = p.num_pages * p.page_size;
    if (threadIdx.x == 4 * 32) {
      tma_prefetch_desc(&tm_qn);
      tma_prefetch_desc(&tm_qp);
      if (p.tma_rows > 0) {
        tma_prefetch_desc(&tm_ckv);
        tma_prefetch_desc(&tm_kpe);
      }
      mbar_arrive_expect_tx(bar_q, kQBytes);
      for (int kb = 0; kb < kDc / 64; ++kb)
        tma_load_3d(sQ + kb * (kH * 128), &tm_qn, bar_q, kb * 64, hb, b);
      tma_load_3d(sQ + (kDc / 64) * (kH * 128), &tm_qp, bar_q, 0, hb, b);
    }
    // Row ids: a group is four 32-token stages; lane l holds the row of token
    // 32 * (4g + (l >> 3)) + 8pw + (l & 7) of the current group g, and the page id of the
    // same token of group g + 1 is loaded one group ahead.
    const int first_page = __ldg(table + t_start / p.page_size);
    int fill_row = (first_page >= 0 && first_page < p.num_pages)
                       ? first_page * p.page_size + t_start % p.page_size : 0;
    if (fill_row >= n_rows) fill_row = 0;
    auto group_token = [&](int g) { return t_start + 32 * (4 * g + (lane >> 3)) + 8 * pw + (lane & 7); };
    auto load_page = [&](int g) {
      const int tok = group_token(g);
      return tok < t_stop ? __ldg(table + tok / p.page_size) : -1;
    };
    auto page_to_row = [&](int page, int g) {
      const int tok = group_token(g);
      int row = fill_row;  // tokens past the end read a valid row; their scores are masked
      if (tok < t_stop) {
        if (page >= 0 && page < p.num_pages) {
          row = page * p.page_size + tok % p.page_size;
        } else {
          record_error(p.status, kDevBounds);
        }
      }
      return (row >= 0 && row < n_rows) ? row : fill_row;
    };
    int row_cur = page_to_row(load_page(0), 0);
    int page_next = load_page(1);
    int cur_group = 0;
    const uint8_t* ckv = static_cast<const uint8_t*>(p.ckv);
    const uint8_t* kpe = static_cast<const uint8_t*>(p.kpe);
    // Issue a stage whenever its ring slot is free; otherwise publish the oldest issued
    // stage once this thread's copies for it have landed (wait, then fence so the tensor
    // core's async-proxy reads see them, then arrive).  Publishing never waits on a slot.
    int issued = 0, published = 0;
    uint64_t t_last = global_timer_ns();
    while (published < n_stages) {
      bool can_issue = issued < n_stages;
      if (can_issue && issued >= kStages) {
        const bool free_slot = mbar_test_wait(bar_empty(issued % kStages),
                                              ((issued / kStages) - 1) & 1);
        can_issue = __shfl_sync(0xffffffffu, free_slot ? 1 : 0, 0) != 0;
        if (can_issue) mbar_wait(bar_empty(issued % kStages), ((issued / kStages) - 1) & 1, nullptr);
      }
      if (can_issue) {
        const int n = issued;
        const uint32_t dst = sKV + ((n >> 1) & 1) * kTileBytes + (n & 1) * kBlk;  // stage n
        if ((n >> 2) != cur_group) {
          cur_group = n >> 2;
          row_cur = page_to_row(page_next, cur_group);
          page_next = load_page(cur_group + 1);
        }
        // Pages of a multiple of 64 tokens: a full 64-token tile is a 64-row slice of one
        // page, and its eight ckv blocks arrive as one 3-D TMA box (64 columns x 64 rows x 8
        // blocks: whole 1 KB rows, landing block after block in the ring tile) plus one kpe
        // box, both 128-byte swizzled like the gathers.  Every producer thread reads the
        // tile's page id (the same address), so all agree on the path without talking.  At
        // the tile's first stage one thread waits for the second stage's slot as well, puts
        // the whole tile's bytes on the first stage's full barrier and issues the two boxes;
        // the second stage issues nothing.  Everyone still arrives on both stages when
        // publishing, as for gathered stages.  Partial tiles and bad page ids are gathered.
        bool by_tma = false;
        int tile_row = 0;
        if (p.tma_rows > 0) {
          const int t0 = t_start + kHalf * (n & ~1);
          if (t0 + kTile <= t_stop) {
            const int page = __ldg(table + t0 / p.page_size);
            by_tma = page >= 0 && page < p.num_pages;
            tile_row = page * p.page_size + t0 % p.page_size;
          }
        }
        if (by_tma) {
          if ((n & 1) == 0 && threadIdx.x == 4 * 32) {
            if (n + 1 >= kStages)
              mbar_wait(bar_empty((n + 1) % kStages), (((n + 1) / kStages) - 1) & 1, p.status);
            const uint32_t full = bar_full(n % kStages);
            mbar_expect_tx(full, 2 * kStageBytes);
            tma_load_3d(dst, &tm_ckv, full, 0, tile_row, 0);
            tma_load_2d(dst + (kDc / 64) * kBlockStride, &tm_kpe, full, 0, tile_row);
          }
        } else {
        const int rsel = row_cur;
#pragma unroll
        for (int t8 = 0; t8 < 8; ++t8) {
          const int tok = 8 * pw + t8;
          const int row = __shfl_sync(0xffffffffu, rsel, ((n & 3) << 3) + t8);
          const uint8_t* src = ckv + static_cast<size_t>(row) * (kDc * 2);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int q = hf * 32 + lane;  // 16-byte chunk of the ckv row
            cp_async_16(dst + (q >> 3) * kBlockStride + tok * 128 + (((q & 7) ^ (tok & 7)) * 16),
                        src + q * 16);
          }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int idx = k * 32 + lane, t8 = idx >> 3, cc = idx & 7, tok = 8 * pw + t8;
          const int row = __shfl_sync(0xffffffffu, rsel, ((n & 3) << 3) + t8);
          cp_async_16(dst + (kDc / 64) * kBlockStride + tok * 128 + ((cc ^ (tok & 7)) * 16),
                      kpe + static_cast<size_t>(row) * (kDr * 2) + cc * 16);
        }
        }
        cp_async_commit();  // an empty group for a TMA stage keeps the per-thread count
        ++issued;
        t_last = global_timer_ns();
      } else if (published < issued) {
        cp_async_wait_dyn(issued - published - 1);
        fence_proxy_async_smem();
        mbar_arrive(bar_full(published % kStages));
        ++published;
        t_last = global_timer_ns();
      } else if (global_timer_ns() - t_last > kWaitLimitNs) {
        // Nothing moved for the whole limit: this thread's gathers are waited for below, and
        // a TMA stage it issued (microseconds of copying) landed long before.
        record_error(p.status, kDevTimeout);
        break;
      }
    }
    cp_async_wait<0>();
  } else if (warp == kMmaWarp) {
    // ----------------------------------- MMA issuer --------------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16(BF16, 64, kTile, false, false);
      constexpr uint32_t idesc_o = idesc_f16(BF16, 128, kH, true, false);
      // S of tile j: one N=64 MMA per 16-column K step over its two stages (contiguous rows
      // of every block in the block-major ring), into S buffer j & 1
      const uint64_t q_desc = sdesc_sw128(sQ, 16, 1024);
      const uint64_t kv_desc = sdesc_sw128(sKV, 16, 1024);
      const uint64_t kv_desc_mn = sdesc_sw128(sKV, kBlockStride, 1024);
      const uint64_t p_desc = sdesc_sw128(sP, 16, 1024);
      auto issue_s = [&](int j) {
        const uint64_t b0 = sdesc_add(kv_desc, (j & 1) * kTileBytes);
        const uint32_t d0 = tmem + kTmemS + (j & 1) * kTile;
#pragma unroll
        for (int kk = 0; kk < kBlocks * 4; ++kk) {
          const uint32_t off = (kk % 4) * 32;
          mma_ss(d0, sdesc_add(q_desc, (kk / 4) * (kH * 128) + off),
                 sdesc_add(b0, (kk / 4) * kBlockStride + off), idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar_s(j & 1));
      };
      // O^T += ckv^T P^T for tile j, then release its two stages
      auto issue_pv = [&](int j) {
        const uint64_t kv = sdesc_add(kv_desc_mn, (j & 1) * kTileBytes);
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks) {
          const uint64_t bd = sdesc_add(p_desc, ks * 32);
#pragma unroll
          for (int db = 0; db < kDc / 128; ++db) {  // four independent accumulators
            const uint64_t ad = sdesc_add(kv, (2 * db) * kBlockStride + ks * (16 * 128));
            mma_ss(tmem + kTmemO + db * kH, ad, bd, idesc_o, (j > 0 || ks > 0) ? 1u : 0u);
          }
        }
        tc_commit(bar_o);
        tc_commit(bar_empty((2 * j) % kStages));
        tc_commit(bar_empty((2 * j + 1) % kStages));
      };
      auto stage_landed = [&](int n) {
        return mbar_test_wait(bar_full(n % kStages), (n / kStages) & 1);
      };
      // Issue whichever MMA is ready: S_j once tile j has landed (and S buffer j & 1 is
      // free, i.e. PV_{j-2} has been issued), PV_j once P_j is written.  PV never waits for
      // the next tile's data, so stages are released as soon as their tile is done.
      bool ok = mbar_wait(bar_q, 0, p.status);
      if (ok) tc_fence_after();
      int next_s = 0, next_pv = 0;
      uint64_t t_last = global_timer_ns();
      while (ok && next_pv < n_tiles) {
        bool progress = false;
        if (next_s < n_tiles && next_s <= next_pv && stage_landed(2 * next_s) &&
            stage_landed(2 * next_s + 1)) {
          tc_fence_after();
          issue_s(next_s++);
          progress = true;
        }
        if (next_pv < next_s && mbar_test_wait(bar_p, next_pv & 1)) {
          tc_fence_after();
          issue_pv(next_pv++);
          progress = true;
        }
        if (progress) {
          t_last = global_timer_ns();
        } else if (global_timer_ns() - t_last > kWaitLimitNs) {
          record_error(p.status, kDevTimeout);
          ok = false;
        }
      }
      tc_commit(bar_done);
      mbar_wait(bar_done, 0, nullptr);
    }
  } else {
    // ---------------------- softmax (two threads per head) + epilogue ---------------------
    // Lanes i and 16 + i of warp w both work on head h = 16w + i: the first on the tile's
    // tokens 0-31, the second on tokens 32-63.  The M=64 score layout puts the head's row in
    // tensor-memory lane 32w + i, so the second half is handed over with shuffles.  Both
    // lanes keep the same running max and sum.
    const int hl = lane & 15, half_t = lane >> 4;
    const bool lead = half_t == 0;
    const int h = warp * 16 + hl;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    // No early exit from this loop: the four softmax warps meet at named barriers, so after
    // a failed wait a warp keeps going without waiting (its results are discarded).
    for (int j = 0; j < n_tiles; ++j) {
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_s(j & 1), (j >> 1) & 1, p.status));
      tc_fence_after();
      uint32_t raw[kTile];
      const uint32_t ts = tmem + kTmemS + lane_off + (j & 1) * kTile;
      tmem_ld32(ts, *reinterpret_cast<uint32_t(*)[32]>(&raw[0]));
      tmem_ld32(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(&raw[32]));
      tmem_ld_wait();
      const int n_valid = t_stop - (t_start + j * kTile + half_t * (kTile / 2));
      float s[kTile / 2];
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int e = 0; e < kTile / 2; ++e) {
        const uint32_t hi = __shfl_sync(0xffffffffu, raw[kTile / 2 + e], hl);
        const float v = __uint_as_float(half_t ? hi : raw[e]);
        s[e] = (e < n_valid) ? v * p.scale_log2 : -INFINITY;
        mx[e & 3] = fmaxf(mx[e & 3], s[e]);
      }
      float mloc = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 16));
      const float m_new = fmaxf(m_run, mloc);
      if (j > 0 && ok) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar_o, (j - 1) & 1, p.status));
        tc_fence_after();
      }
      const bool need = m_new > m_run + kRescaleLog2;
      if (softmax_any(need)) {
        float alpha = 1.f;
        if (need) {
          alpha = exp2_approx(m_run - m_new);
          m_run = m_new;
          l_run *= alpha;
        }
        if (lead) alpha_s[h] = alpha;
        softmax_sync();
        if (j > 0) {
          // O^T column h belongs to head h; every lane holds one latent dim of every head
#pragma unroll 1
          for (int db = 0; db < kDc / 128; ++db) {
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
              uint32_t o[32];
              const uint32_t ta = tmem + kTmemO + lane_off + db * kH + half * 32;
              tmem_ld32(ta, o);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e)
                o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha_s[half * 32 + e]);
              tmem_st32(ta, o);
            }
          }
          tmem_st_wait();
        }
        softmax_sync();  // alpha_s may be rewritten on the next tile
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      float sum[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[kTile / 4];
#pragma unroll
      for (int e = 0; e < kTile / 4; ++e) {
        const float p0 = exp2_approx(s[2 * e] - m_use);
        const float p1 = exp2_approx(s[2 * e + 1] - m_use);
        sum[e & 3] += p0 + p1;
        pk[e] = BF16 ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
      }
      const float lsum = (sum[0] + sum[1]) + (sum[2] + sum[3]);
      l_run += lsum + __shfl_xor_sync(0xffffffffu, lsum, 16);  // the same total in both lanes
      // P^T row h: 64 tokens x bf16 = 128 bytes, 16-byte chunks swizzled by h % 8; this
      // lane's tokens are chunks 4 * half_t .. 4 * half_t + 3
      uint8_t* prow = smem + kPOff + h * 128;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        *reinterpret_cast<uint4*>(prow + (((4 * half_t + k) ^ (h & 7)) * 16)) =
            make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_p);
    }
    if (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_o, (n_tiles - 1) & 1, p.status));
      tc_fence_after();
    }
    // every softmax thread must reach these barriers, even after a failed wait
    if (lead) stat_s[h] = l_run > 0.f ? 1.f / l_run : 0.f;
    softmax_sync();
    // Normalise O into the (now idle) KV ring as [head][latent dim] fp32 rows, then write
    // each head's 2 KB row with 16-byte coalesced stores.
    float* ostage = reinterpret_cast<float*>(smem + kKVOff);
    if (ok) {
      // the 64 per-head scales go to registers first: read from shared memory between the
      // staging stores, each would wait for the stores before it (the compiler cannot tell
      // the two arrays apart)
      float inv[kH];
#pragma unroll
      for (int e = 0; e < kH; ++e) inv[e] = stat_s[e];
#pragma unroll 1
      for (int db = 0; db < kDc / 128; ++db) {
        const int d = db * 128 + warp * 32 + lane;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t o[32];
          tmem_ld32(tmem + kTmemO + lane_off + db * kH + half * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e)
            ostage[(half * 32 + e) * kDc + d] = __uint_as_float(o[e]) * inv[half * 32 + e];
        }
      }
    }
    softmax_sync();
    if (ok) {
      const size_t row0 = static_cast<size_t>(b) * p.H + hb;               // output rows
      const size_t prow0 = static_cast<size_t>(b - p.n_whole) * p.H + hb;  // partial-state rows
#pragma unroll 1
      for (int r = 0; r < 16; ++r) {
        const int hh = warp * 16 + r;
        if (hh >= hv) break;
        const float4* src = reinterpret_cast<const float4*>(ostage + hh * kDc);
        if (direct) {
          // the whole sequence was this CTA's chunk: write the final bf16 row
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + (row0 + hh) * kDc);
#pragma unroll
          for (int k = 0; k < kDc / 8 / 32; ++k) {
            const float4 a = src[2 * (lane + 32 * k)], b2 = src[2 * (lane + 32 * k) + 1];
            dst[lane + 32 * k] =
                BF16 ? make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w),
                                  pack_bf16x2(b2.x, b2.y), pack_bf16x2(b2.z, b2.w))
                     : make_uint4(pack_f16x2(a.x, a.y), pack_f16x2(a.z, a.w),
                                  pack_f16x2(b2.x, b2.y), pack_f16x2(b2.z, b2.w));
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(p.o_part + ((prow0 + hh) * p.n_chunks + c) * kDc);
#pragma unroll
          for (int k = 0; k < kDc / 4 / 32; ++k) dst[lane + 32 * k] = src[lane + 32 * k];
        }
      }
      if (lead && h < hv) {
        const float lse_v = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
        if (!direct) p.lse_part[(prow0 + h) * p.n_chunks + c] = lse_v;
        else if (p.lse) p.lse[row0 + h] = lse_v;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

// Tokens per CTA: each CTA pays a fixed cost (pipeline start, epilogue) worth a few hundred
// tokens of streaming, so prefer long chunks, but keep the waves of CTAs balanced.
int mla_chunk_tokens(int B, int H, int max_seq_len) {
  const int sms = num_sms() > 0 ? num_sms() : 148;
  B *= (H + kH - 1) / kH;  // CTAs per chunk of the batch: one per group of 64 heads
  const int len = ((max_seq_len + kTile - 1) / kTile) * kTile;
  int best = 512;
  long best_cost = -1;
  for (int c = 512; c <= kMaxChunk; c *= 2) {
    const long ctas = static_cast<long>(B) * ((max_seq_len + c - 1) / c);
    const long waves = (ctas + sms - 1) / sms;
    const long cost = waves * (static_cast<long>(c < len ? c : len) + 384);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = c;
    }
  }
  return best;
}

// The plan of a full MLA call.  With several chunks per sequence every sequence is split.
// With one, every sequence is one CTA writing its final output, unless the last wave of
// CTAs would be at most half full: then the sequences of that wave are cut into chunks that
// together fill it (whole sequences are dispatched first), so the call ends after a short
// wave instead of a full-length one, and only those sequences' rows are merged.
MlaPlan mla_plan(int B, int H, int max_seq_len) {
  MlaPlan pl{};
  const int chunk = mla_chunk_tokens(B, H, max_seq_len);
  const int n_chunks = max_seq_len > 0 ? (max_seq_len + chunk - 1) / chunk : 0;
  if (n_chunks != 1) {
    pl.n_whole = 0;
    pl.chunk = chunk;
    pl.n_chunks = n_chunks;
    return pl;
  }
  pl.n_whole = B;
  pl.whole_chunk = chunk;
  pl.chunk = chunk;
  pl.n_chunks = 1;
  if (H > kH) return pl;  // several head groups per sequence: no short-wave split
  const int sms = num_sms() > 0 ? num_sms() : 148;
  const int waves = (B + sms - 1) / sms;
  const int tail = B - (waves - 1) * sms;  // sequences in the last wave
  if (waves >= 2 && 2 * tail <= sms) {
    const int k = sms / tail;
    const int ct = ((max_seq_len + k - 1) / k + kTile - 1) / kTile * kTile;
    const int kc = (max_seq_len + ct - 1) / ct;
    if (kc >= 2) {
      pl.n_whole = B - tail;
      pl.chunk = ct;
      pl.n_chunks = kc;
    }
  }
  return pl;
}

cudaError_t launch_mla(const MlaParams& params, cudaStream_t stream) {
  MlaParams p = params;
  if (p.H < 1 || p.Dc != kDc || p.Dr != kDr || p.n_whole < 0 || p.n_whole > p.B)
    return cudaErrorInvalidValue;
  if (p.n_whole > 0 && (p.whole_chunk % kTile != 0 || p.whole_chunk > kMaxChunk))
    return cudaErrorInvalidValue;
  if (p.n_whole < p.B &&
      (p.n_chunks < 1 || p.chunk % kTile != 0 || p.chunk > kMaxChunk || !p.o_part || !p.lse_part))
    return cudaErrorInvalidValue;
  CUtensorMap tqn, tqp;
  const CUtensorMapDataType dt = p.f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  {
    // (latent column, head, sequence): a box of 64 columns x 64 heads, heads past H zero
    const uint64_t dims[3] = {kDc, static_cast<uint64_t>(p.H), static_cast<uint64_t>(p.B)};
    const uint64_t str[2] = {kDc * 2, static_cast<uint64_t>(p.H) * kDc * 2};
    const uint32_t box[3] = {64, kH, 1};
    if (!encode_tiled(&tqn, dt, 3, p.q_nope, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {kDr, static_cast<uint64_t>(p.H), static_cast<uint64_t>(p.B)};
    const uint64_t str[2] = {kDr * 2, static_cast<uint64_t>(p.H) * kDr * 2};
    const uint32_t box[3] = {64, kH, 1};
    if (!encode_tiled(&tqp, dt, 3, p.q_pe, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  // Tile-sized TMA copies (see the producer) when a page holds whole 64-token tiles.  The
  // ckv map walks (64 columns, row, 64-column block) so a box of 64 x 64 x 8 lands as the
  // tile's eight blocks one after another.
  CUtensorMap tckv = tqn, tkpe = tqp;  // placeholders when every stage is gathered
  const int ps = p.page_size;
  p.tma_rows = (ps > 0 && ps % kTile == 0) ? kTile : 0;
  if (p.tma_rows > 0) {
    const uint64_t rows = static_cast<uint64_t>(p.num_pages) * ps;
    const uint64_t dims_c[3] = {64, rows, kDc / 64}, str_c[2] = {kDc * 2, 128};
    const uint32_t box_c[3] = {64, kTile, kDc / 64};
    const uint64_t dims_r[2] = {kDr, rows}, str_r[1] = {kDr * 2};
    const uint32_t box_r[2] = {64, kTile};
    if (!encode_tiled(&tckv, dt, 3, p.ckv, dims_c, str_c, box_c, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&tkpe, dt, 2, p.kpe, dims_r, str_r, box_r, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  auto kern = p.f16 ? mla_kernel<false> : mla_kernel<true>;
  cudaError_t e = ensure_smem_limit(kern, kSmemBytes);
  if (e != cudaSuccess) return e;
  const long ctas = static_cast<long>((p.H + kH - 1) / kH) *
                    (p.n_whole + static_cast<long>(p.B - p.n_whole) * (p.n_whole < p.B ? p.n_chunks : 0));
  if (ctas <= 0) return cudaSuccess;
  if (ctas > 0x7fffffffL) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(ctas));
  kern<<<grid, kThreads, kSmemBytes, stream>>>(tqn, tqp, tckv, tkpe, p);
  return cudaGetLastError();
}

}  // namespace fa

// prefill.cu -- fused attention forward for dense (prefill) inputs on sm_103a.
//
// One CTA computes one 128-row tile of packed (query head, query) rows against one range of
// KV tiles of one kv head.  Grouped-query heads are packed into the tile ("GQA optimization",
// llama.cpp PR "CUDA: fix FA occupancy, optimize tile kernel", second paragraph), so K, V and
// the mask are read once per kv head.  The loop is FlashAttention's: S = Q K^T on the tensor
// cores, an online softmax on the CUDA cores, O += P V on the tensor cores, with the softmax
// overlapping the next tile's Q K^T (the FA3 software pipeline described in flashinfer PR
// "perf: FlashAttention-3 style MLA PageAttention", change list items 1-3), rebuilt for
// Blackwell: TMA loads into a multi-stage shared-memory ring, tcgen05.mma accumulating in
// tensor memory, three S/P buffers in tensor memory with P (16-bit) written over S, and O
// resident in tensor memory for the whole KV loop.  The paged instantiation reads K/V
// through a page table (chunked prefill against a paged cache): each page of a KV tile is
// one 5-D TMA box, and each sequence has its own length.
//
// Warp roles (224 threads): warps 0-3 softmax + epilogue (thread t owns row t), warp 4 TMA
// producer, warp 5 the P V issuer (one elected thread) and tensor-memory owner, warp 6 the
// S issuer (one elected thread).  Once a thread has committed MMAs, its next shared-memory
// access (an mbarrier wait included) is held until those MMAs finish, so a single issuer that
// waits for P_j drains the tensor pipe every tile.  With two issuers each wait holds only
// its own thread's MMAs: while the P V issuer waits for the softmax, the S issuer's next
// products keep the tensor pipe busy, and the other way round.  S/P has three buffers in
// tensor memory (S_j in buffer j % 3), so S can run up to two tiles ahead of the softmax;
// S_{j+3} is issued into P_j's buffer once P_j V_j has finished.
#include <math.h>

#include "internal.h"
#include "prefill_common.cuh"
#include "sm103.cuh"

namespace fa {
namespace {

using prefill::kRows;
constexpr int kThreads = 224;
constexpr int kLptMaxSeqs = kThreads;  // paged: order sequences by length (one ranking thread each)

// 5-D tiled TMA load (the paged K/V boxes below).
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2, int32_t c3,
                                            int32_t c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
      "r"(bar)
      : "memory");
}

constexpr int kNumS = 3;  // S/P buffers in tensor memory

// Named barrier `id` over `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <int D, int BN, int STAGES>
struct Layout {
  static constexpr int kQBytes = kRows * D * 2;
  static constexpr int kKVBytes = BN * D * 2;  // one K (or V) stage
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQBytes;
  static constexpr int kVOff = kKOff + STAGES * kKVBytes;
  static constexpr int kBarOff = kVOff + STAGES * kKVBytes;
  // Q, the A operand of S, also goes into tensor memory when it fits beside O and the S/P
  // buffers (D/2 columns): S then reads only K from shared memory.
  static constexpr bool kQInTmem = D + kNumS * BN + D / 2 <= 512;
  // q_full, k_full[S], v_full[S], k_empty[S], v_empty[S], s_full[3], p_full[3], pv_done[3],
  // pv_issuer_done, s_issuer_done, q_in_tmem
  static constexpr int kNumBars = 1 + 4 * STAGES + 3 * kNumS + 3;
  static constexpr int kBytes = kBarOff + kNumBars * 8 + 16;
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024 bytes
  static_assert(D + kNumS * BN <= 512, "tensor memory budget (O and the S/P buffers)");
  static_assert(kAlloc <= 232448, "shared memory budget");
};

// One CTA per (query tile, split) x kv head x batch.  PAGED: K/V through a page table.
// SPLIT: the KV loop is split across CTAs and each writes a partial state (a separate
// instantiation, so that the unsplit kernel carries none of its epilogue).
template <int D, int BN, int STAGES, bool BF16, bool PAGED, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_po,
                   const PrefillParams p) {
  using L = Layout<D, BN, STAGES>;
  constexpr bool kStagedOut = D <= 128;  // final 16-bit output through TMA stores
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_addr(smem);
  const uint32_t sQ = s_base + L::kQOff, sK = s_base + L::kKOff, sV = s_base + L::kVOff;
  const uint32_t bars = s_base + L::kBarOff;
  const uint32_t bar_q = bars;
  auto bar_k = [&](int s) { return bars + 8u * (1 + s); };
  auto bar_v = [&](int s) { return bars + 8u * (1 + STAGES + s); };
  auto bar_ke = [&](int s) { return bars + 8u * (1 + 2 * STAGES + s); };
  auto bar_ve = [&](int s) { return bars + 8u * (1 + 3 * STAGES + s); };
  // per S/P buffer b (tile j with j % 3 == b): S_j computed, P_j written, P_j V_j finished
  auto bar_s = [&](int b) { return bars + 8u * (1 + 4 * STAGES + b); };
  auto bar_p = [&](int b) { return bars + 8u * (1 + 4 * STAGES + kNumS + b); };
  auto bar_pv = [&](int b) { return bars + 8u * (1 + 4 * STAGES + 2 * kNumS + b); };
  const uint32_t bar_done = bars + 8u * (1 + 4 * STAGES + 3 * kNumS);
  const uint32_t bar_sdone = bar_done + 8u;
  const uint32_t bar_qt = bar_done + 16u;  // Q copied into tensor memory (kQInTmem)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBarOff + L::kNumBars * 8);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // A K or V stage holds BN rows x D columns as 1024-byte SW128 atoms (8 rows x 64 columns).
  // Dense: the atoms of one 64-column block follow each other down the rows, block after
  // block, so a column block of a tile is one TMA box.  Paged: the D/64 atoms of one 8-row
  // group sit side by side, group after group, so a page (whole 8-row groups) is one box.
  constexpr uint32_t kCB = PAGED ? 1024u : BN * 128u;             // column-block stride
  constexpr uint32_t kRG = PAGED ? (D / 64) * 1024u : 1024u;      // 8-row-group stride

  // ---- work item: (query tile, split) x kv head x batch; heavier (later) tiles first ----
  const int split = blockIdx.x % p.n_splits;
  const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x) / p.n_splits;
  const int hk = blockIdx.y;
  int b = blockIdx.z;
  if constexpr (PAGED) {
    // Sequences have different lengths: hand them out longest first (blockIdx.z is a rank
    // in decreasing length, ties by index), so the last CTAs to start are short ones.
    // Thread i ranks sequence i; the one whose rank is this CTA's publishes its index.
    __shared__ int lpt_seq;
    if (p.B <= kLptMaxSeqs) {
      if (threadIdx.x < p.B) {
        const int li = p.kv_lens[threadIdx.x];
        int rank = 0;
        for (int j = 0; j < p.B; ++j) {
          const int lj = p.kv_lens[j];
          rank += (lj > li || (lj == li && j < static_cast<int>(threadIdx.x))) ? 1 : 0;
        }
        if (rank == static_cast<int>(blockIdx.z)) lpt_seq = threadIdx.x;
      }
      __syncthreads();
      b = lpt_seq;
    }
  }
  const int q0 = qt * p.q_per_tile;
  const int q_last = min(p.Lq, q0 + p.q_per_tile) - 1;
  // keys of this sequence: dense Lkv, or the sequence's length in the paged cache
  int Lkv = p.Lkv;
  if constexpr (PAGED) {
    Lkv = p.kv_lens[b];
    if (Lkv < 0 || Lkv > p.max_pages * p.page_size) {
      if (threadIdx.x == 0) record_error(p.status, kDevBounds);
      Lkv = 0;
    }
  }
  int t_begin, t_end;
  prefill::kv_range(p, q_last, BN, split, Lkv, t_begin, t_end);
  const int n = t_end - t_begin;

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_k(s), 1);
      mbar_init(bar_v(s), 1);
      mbar_init(bar_ke(s), 1);
      mbar_init(bar_ve(s), 1);
    }
    for (int i = 0; i < kNumS; ++i) {
      mbar_init(bar_s(i), 1);
      mbar_init(bar_p(i), 4 * 32);
      mbar_init(bar_pv(i), 1);
    }
    mbar_init(bar_done, 1);
    mbar_init(bar_sdone, 1);
    mbar_init(bar_qt, 4 * 32);
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tm_o = tmem;           // O: columns [0, D)
  const uint32_t tm_s0 = tmem + D;      // S/P buffer b: columns [D + b*BN, D + (b+1)*BN)
  // Q (kQInTmem): row r in lane r, element pairs packed per column (D/2 columns)
  const uint32_t tq_tmem = tmem + D + kNumS * BN;

  if (warp == 4) {
    // ------------------------------- TMA producer ---------------------------------------
    if (n > 0) {
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        mbar_arrive_expect_tx(bar_q, static_cast<uint32_t>(D * 2 * p.q_per_tile * p.G));
        for (int kb = 0; kb < D / 64; ++kb)
          tma_load_4d(sQ + kb * (kRows * 128), &tm_q, bar_q, kb * 64, q0, hk * p.G, b);
      }
      int issued = 0, k_only = -1;  // k_only: a K load issued without its V
      // K and V slots are released separately: K_j once S_j is done, V_j once P_j V_j is.
      if constexpr (!PAGED) {
        if (lane == 0) {
          const int kv_row = b * p.Hkv + hk;
          for (int jj = 0; jj < n; ++jj) {
            const int stage = jj % STAGES;
            if (jj >= STAGES && !mbar_wait(bar_ke(stage), ((jj / STAGES) - 1) & 1, p.status)) break;
            const int key0 = (t_begin + jj) * BN;
            mbar_arrive_expect_tx(bar_k(stage), L::kKVBytes);
            for (int kb = 0; kb < D / 64; ++kb)
              tma_load_3d(sK + stage * L::kKVBytes + kb * (BN * 128), &tm_k, bar_k(stage), kb * 64,
                          key0, kv_row);
            if (jj >= STAGES && !mbar_wait(bar_ve(stage), ((jj / STAGES) - 1) & 1, p.status)) {
              k_only = jj;  // K_jj is in flight; let it land below
              break;
            }
            mbar_arrive_expect_tx(bar_v(stage), L::kKVBytes);
            for (int kb = 0; kb < D / 64; ++kb)
              tma_load_3d(sV + stage * L::kKVBytes + kb * (BN * 128), &tm_v, bar_v(stage), kb * 64,
                          key0, kv_row);
            issued = jj + 1;
          }
        }
      } else {
        // Paged: a KV tile is BN / page_size pages and each page is one TMA box of page_size
        // rows x D columns (page_size / 8 whole row groups).  The 5-D map walks a page as
        // (64 columns, 8 rows, D/64 column blocks, page_size/8 row groups) so the box lands
        // in the row-group-major atom order above; its last coordinate is page * Hkv + head.
        // Lane i holds the page id of page i of a tile, loaded one tile ahead, and issues that
        // page's box itself, so one warp instruction starts the copies of every page.
        const int ps = p.page_size, tp = BN / ps;
        const int32_t* table = p.page_table + static_cast<size_t>(b) * p.max_pages;
        auto tile_page = [&](int jj) {
          int id = 0;  // pages past the sequence's end read page 0; those keys are masked
          if (lane < tp) {
            const int lp = (t_begin + jj) * tp + lane;
            const int v = lp < p.max_pages ? __ldg(table + lp) : -1;
            if (v >= 0 && v < p.num_pages) {
              id = v;
            } else if (lp * ps < Lkv) {
              record_error(p.status, kDevBounds);
            }
          }
          return id;
        };
        auto load_pages = [&](uint32_t dst, const CUtensorMap* map, uint32_t bar, int id) {
          if (lane < tp)
            tma_load_5d(dst + lane * (ps / 8) * kRG, map, bar, 0, 0, 0, 0, id * p.Hkv + hk);
        };
        int ids_next = tile_page(0);
        for (int jj = 0; jj < n; ++jj) {
          const int ids = ids_next;
          if (jj + 1 < n) ids_next = tile_page(jj + 1);
          const int stage = jj % STAGES;
          bool okw = jj < STAGES || mbar_wait(bar_ke(stage), ((jj / STAGES) - 1) & 1, p.status);
          if (!__shfl_sync(0xffffffffu, okw ? 1 : 0, 0)) break;
          if (lane == 0) mbar_arrive_expect_tx(bar_k(stage), L::kKVBytes);
          __syncwarp();
          load_pages(sK + stage * L::kKVBytes, &tm_k, bar_k(stage), ids);
          okw = jj < STAGES || mbar_wait(bar_ve(stage), ((jj / STAGES) - 1) & 1, p.status);
          if (!__shfl_sync(0xffffffffu, okw ? 1 : 0, 0)) {
            k_only = jj;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(bar_v(stage), L::kKVBytes);
          __syncwarp();
          load_pages(sV + stage * L::kKVBytes, &tm_v, bar_v(stage), ids);
          issued = jj + 1;
        }
      }
      if (lane == 0 && issued < n) {
        // A wait ran out: let the copies already in flight land before the CTA exits.  A K
        // issued without its V (k_only) reused the stage of K_{k_only - STAGES} and was issued
        // only after S_{k_only - STAGES}, that older K's reader, had finished: the older K has
        // landed, and its barrier may be two phases on, where a parity wait would read "not
        // yet" and run out its limit.  It is not waited for.
        mbar_wait(bar_q, 0, nullptr);
        for (int jj = max(0, issued - STAGES); jj < issued; ++jj) {
          if (!(k_only >= 0 && jj == k_only - STAGES))
            mbar_wait(bar_k(jj % STAGES), (jj / STAGES) & 1, nullptr);
          mbar_wait(bar_v(jj % STAGES), (jj / STAGES) & 1, nullptr);
        }
        if (k_only >= 0) mbar_wait(bar_k(k_only % STAGES), (k_only / STAGES) & 1, nullptr);
      }
    }
  } else if (warp == 5) {
    // ------------------------------- P V issuer -----------------------------------------
    if (lane == 0 && n > 0) {
      constexpr uint32_t idesc_o = idesc_f16(BF16, kRows, D, false, true);
      // descriptors are built once; per tile and K step only their start address moves
      const uint64_t v_desc = sdesc_sw128(sV, kCB, kRG);
      bool ok = true;
      for (int jj = 0; ok && jj < n; ++jj) {
        const int stage = jj % STAGES, buf = jj % kNumS;
        // the first wait is held until P_{j-1} V_j-1 finishes; the second then finds V_j
        if (!(ok = mbar_wait(bar_p(buf), (jj / kNumS) & 1, p.status))) break;
        if (!(ok = mbar_wait(bar_v(stage), (jj / STAGES) & 1, p.status))) break;
        tc_fence_after();
        const uint64_t vd = sdesc_add(v_desc, stage * L::kKVBytes);
        const uint32_t a_p = tm_s0 + buf * BN;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(tm_o, a_p + kk * 8, sdesc_add(vd, kk * (2 * kRG)), idesc_o,
                 (jj > 0 || kk > 0) ? 1u : 0u);
        tc_commit(bar_pv(buf));
        tc_commit(bar_ve(stage));
      }
      // Every MMA this thread issued must finish before tensor memory is released.
      tc_commit(bar_done);
      mbar_wait(bar_done, 0, nullptr);
    }
  } else if (warp == 6) {
    // --------------------------------- S issuer -----------------------------------------
    // S_j = Q K_j^T into buffer j % 3 once K_j has landed and, from j = 3 on, P_{j-3} V_{j-3}
    // (the last reader of that buffer) has finished.  It runs at most two tiles ahead of the
    // softmax, and the K ring bounds it by STAGES.
    if (lane == 0 && n > 0) {
      constexpr uint32_t idesc_s = idesc_f16(BF16, kRows, BN, false, false);
      const uint64_t k_desc = sdesc_sw128(sK, 16, kRG);
      const uint64_t q_desc = sdesc_sw128(sQ, 16, 1024);
      bool ok = L::kQInTmem ? mbar_wait(bar_qt, 0, p.status) : mbar_wait(bar_q, 0, p.status);
      for (int jj = 0; ok && jj < n; ++jj) {
        const int stage = jj % STAGES, buf = jj % kNumS;
        if (!(ok = mbar_wait(bar_k(stage), (jj / STAGES) & 1, p.status))) break;
        if (jj >= kNumS && !(ok = mbar_wait(bar_pv(buf), ((jj - kNumS) / kNumS) & 1, p.status))) break;
        tc_fence_after();
        const uint64_t kd = sdesc_add(k_desc, stage * L::kKVBytes);
        const uint32_t d_s = tm_s0 + buf * BN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk % 4) * 32;
          const uint64_t bd = sdesc_add(kd, (kk / 4) * kCB + off);
          if constexpr (L::kQInTmem) {
            mma_ts(d_s, tq_tmem + kk * 8, bd, idesc_s, kk > 0 ? 1u : 0u);
          } else {
            mma_ss(d_s, sdesc_add(q_desc, (kk / 4) * (kRows * 128) + off), bd, idesc_s,
                   kk > 0 ? 1u : 0u);
          }
        }
        tc_commit(bar_s(buf));
        tc_commit(bar_ke(stage));
      }
      tc_commit(bar_sdone);
      mbar_wait(bar_sdone, 0, nullptr);
    }
  } else {
    // ------------------------- softmax + epilogue (row per thread) ----------------------
    const prefill::Row row = prefill::make_row(p, b, hk, q0, threadIdx.x, Lkv);
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    if (L::kQInTmem && n > 0) {
      // Copy this thread's Q row from the swizzled shared-memory tile into its tensor-memory
      // lane: 64-column block kb, 16-byte chunk ch of row r sits at chunk ch ^ (r & 7).
      ok = __all_sync(0xffffffffu, mbar_wait(bar_q, 0, p.status));
      if (ok) {
        const int r = threadIdx.x;
        const uint8_t* qrow = smem + L::kQOff + r * 128;
#pragma unroll 1
        for (int kb = 0; kb < D / 64; ++kb) {
          uint32_t w[32];
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint4 v = *reinterpret_cast<const uint4*>(qrow + kb * (kRows * 128) + ((ch ^ (r & 7)) * 16));
            w[4 * ch] = v.x;
            w[4 * ch + 1] = v.y;
            w[4 * ch + 2] = v.z;
            w[4 * ch + 3] = v.w;
          }
          tmem_st32(tq_tmem + lane_off + kb * 32, w);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar_qt);
      }
    }
    for (int jj = 0; ok && jj < n; ++jj) {
      const int buf = jj % kNumS;
      const uint32_t t_s = tm_s0 + lane_off + buf * BN;
      ok = __all_sync(0xffffffffu, mbar_wait(bar_s(buf), (jj / kNumS) & 1, p.status));
      if (!ok) break;
      tc_fence_after();
      uint32_t raw[BN];
      prefill::load_s<BN>(t_s, raw);
      float alpha;
      uint32_t pk[BN / 2];
      // the exponentials overlap the previous tile's P V on the tensor cores
      // three-input max: faster for 64-key tiles and the paged instantiations, slower for
      // the dense 128-key one (measured)
      const bool need = prefill::softmax_tile<BN, BF16, (BN <= 64 || PAGED)>(
          p, row, (t_begin + jj) * BN, raw, m_run, l_run, alpha, pk);
      // O is rescaled only once every earlier P V product is in it (the P V issuer runs its
      // products in order, so P_{j-1} V_{j-1} finishing means all have).  A tile with no
      // rescale does not wait: P_j V_j is issued after P_j anyway, and this warp cannot get
      // two phases ahead on a P V barrier, since S_j itself needed P_{j-3} V_{j-3} finished.
      const bool rescale = jj > 0 && __any_sync(0xffffffffu, need);
      if (rescale) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar_pv((jj - 1) % kNumS), ((jj - 1) / kNumS) & 1, p.status));
        if (!ok) break;
        tc_fence_after();
        prefill::rescale_o<D>(tm_o + lane_off, alpha);
      }
      prefill::store_p<BN>(t_s, pk);
      tmem_st_wait();
      const int key0 = (t_begin + jj) * BN;
      if (PAGED && key0 + BN > Lkv) {
        // Rows past the sequence's end hold whatever the pool has there; P is 0 for them,
        // but 0 times a non-finite V would still poison O, so clear them once V has landed.
        // The parity wait for V_j is exact only once the stage's previous tile V_{j-STAGES}
        // has landed: waiting first for P_{j-1} V_{j-1} (in order, so V_{j-STAGES} was read)
        // makes sure of it.
        const int stage = jj % STAGES;
        if (jj > 0 && !rescale) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar_pv((jj - 1) % kNumS), ((jj - 1) / kNumS) & 1, p.status));
          if (!ok) break;
        }
        ok = __all_sync(0xffffffffu, mbar_wait(bar_v(stage), (jj / STAGES) & 1, p.status));
        if (!ok) break;
        const int r0 = Lkv - key0;
        uint8_t* vst = smem + L::kVOff + stage * L::kKVBytes;
        for (int i = threadIdx.x; i < (BN - r0) * (D / 64) * 8; i += 128) {
          const int blk = i / ((BN - r0) * 8), rem = i % ((BN - r0) * 8);
          const int r = r0 + rem / 8;
          *reinterpret_cast<uint4*>(vst + (r / 8) * kRG + blk * kCB + (r % 8) * 128 + (rem % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive(bar_p(buf));
    }
    if (ok && n > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar_pv((n - 1) % kNumS), ((n - 1) / kNumS) & 1, p.status));
      tc_fence_after();
    }
    if constexpr (SPLIT || kStagedOut) {
      if (SPLIT || (p.Lq > 1 && p.out_dtype != Dtype::FP32)) {
        // The row's output is staged in the K ring (free once the loop is done) one
        // 32-column slab at a time and written by TMA stores: a split's fp32 partial state
        // through 32-column boxes over the [rows, n_splits, D] buffer (rows are 1 KB apart
        // there, so per-thread stores would not coalesce), the 16-bit output of D <= 128
        // through 64-column boxes of a Q-shaped map.  Thread 0 starts each box as soon as the
        // four softmax warps have staged it, so the copy-out overlaps the staging that
        // follows, and the next slab's tensor-memory load is in flight while one is staged.
        // Every softmax thread reaches every barrier; a warp whose waits ran out flags the
        // tile so that nothing half-written is stored.
        volatile uint32_t& stage_bad = tmem_slot[1];  // spare word beside the tensor-memory slot
        if (threadIdx.x == 0) stage_bad = 0;
        named_barrier_sync(1, 4 * 32);
        if (!ok && lane == 0) stage_bad = 1;
        const bool have_o = ok && n > 0;
        const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
        uint8_t* stage = smem + L::kKOff;
        uint32_t oa[32], ob[32];
        if (have_o) tmem_ld32(tm_o + lane_off, oa);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t(&cur)[32] = (c & 1) ? ob : oa;
          uint32_t(&nxt)[32] = (c & 1) ? oa : ob;
          if (have_o) {
            prefill::tmem_ld_wait_tied(cur);
            if (c + 1 < D / 32) tmem_ld32(tm_o + lane_off + (c + 1) * 32, nxt);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) cur[e] = 0u;
          }
          if constexpr (SPLIT) {
            if (ok) prefill::stage_slab_f32(cur, inv_l, stage + c * (kRows * 128), threadIdx.x);
            fence_proxy_async_smem();
            named_barrier_sync(1, 4 * 32);
            if (threadIdx.x == 0 && !stage_bad) {
              // box: 32 columns x 1 split x q_per_tile queries x G heads; rows past Lq clipped
              prefill::tma_store_4d(&tm_po, sK + c * (kRows * 128), c * 32, split, q0,
                                    b * p.Hq + hk * p.G);
              prefill::bulk_commit_group();
            }
          } else {
            if (ok) prefill::stage_slab16<BF16>(cur, inv_l, stage + (c / 2) * (kRows * 128), threadIdx.x, c);
            if (c & 1) {
              fence_proxy_async_smem();
              named_barrier_sync(1, 4 * 32);
              if (threadIdx.x == 0 && !stage_bad) {
                prefill::tma_store_4d(&tm_po, sK + (c / 2) * (kRows * 128), (c / 2) * 64, q0,
                                      hk * p.G, b);
                prefill::bulk_commit_group();
              }
            }
          }
        }
        if (ok && row.valid) {
          if constexpr (SPLIT) p.lse_part[row.flat * p.n_splits + split] = prefill::row_lse(m_run, l_run);
          else if (p.lse) p.lse[row.flat] = prefill::row_lse(m_run, l_run);
        }
        if (threadIdx.x == 0 && !stage_bad) prefill::bulk_wait_read_all();
      } else if (ok) {
        prefill::epilogue<D>(p, row, tm_o + lane_off, n > 0, m_run, l_run);
      }
    } else if (ok) {
      prefill::epilogue<D>(p, row, tm_o + lane_off, n > 0, m_run, l_run);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int BN, int STAGES, bool BF16, bool PAGED>
cudaError_t launch_impl(const PrefillParams& p, cudaStream_t stream) {
  using L = Layout<D, BN, STAGES>;
  const CUtensorMapDataType dt = BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap tq, tk, tv;
  const uint64_t lkv = p.Lkv > 0 ? p.Lkv : 1;
  {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)p.Lq, (uint64_t)p.Hq, (uint64_t)p.B};
    const uint64_t str[3] = {(uint64_t)D * 2, (uint64_t)p.Lq * D * 2, (uint64_t)p.Hq * p.Lq * D * 2};
    const uint32_t box[4] = {64, (uint32_t)p.q_per_tile, (uint32_t)p.G, 1};
    if (!encode_tiled(&tq, dt, 4, p.q, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  if constexpr (PAGED) {
    // pages [num_pages, Hkv, page_size, D] seen as (column, row in group, column block, row
    // group, page * Hkv + head); one box = one page of one kv head, every column
    if (p.page_size < 8 || BN % p.page_size != 0) return cudaErrorInvalidValue;
    const uint64_t ps = (uint64_t)p.page_size, row = (uint64_t)D * 2;
    const uint64_t dims[5] = {64, 8, (uint64_t)D / 64, ps / 8, (uint64_t)p.num_pages * p.Hkv};
    const uint64_t str[4] = {row, 128, 8 * row, ps * row};
    const uint32_t box[5] = {64, 8, (uint32_t)D / 64, (uint32_t)p.page_size / 8, 1};
    if (!encode_tiled(&tk, dt, 5, p.k, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&tv, dt, 5, p.v, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else {
    const uint64_t dims[3] = {(uint64_t)D, lkv, (uint64_t)p.Hkv * p.B};
    const uint64_t str[2] = {(uint64_t)D * 2, lkv * D * 2};
    const uint32_t box[3] = {64, (uint32_t)BN, 1};
    if (!encode_tiled(&tk, dt, 3, p.k, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&tv, dt, 3, p.v, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  // the partial states [B*Hq rows: (b, h, i)][n_splits][D] fp32, as (column, split, query,
  // b*Hq + h); one store box = 32 columns x 1 split x q_per_tile queries x G heads
  CUtensorMap tpo = tq;
  if (D <= 128 && p.Lq > 1 && p.n_splits <= 1 && p.out_dtype != Dtype::FP32) {
    // the 16-bit output [B, Hq, Lq, D], as Q: one store box = 64 columns x q_per_tile queries
    // x G heads
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)p.Lq, (uint64_t)p.Hq, (uint64_t)p.B};
    const uint64_t str[3] = {(uint64_t)D * 2, (uint64_t)p.Lq * D * 2, (uint64_t)p.Hq * p.Lq * D * 2};
    const uint32_t box[4] = {64, (uint32_t)p.q_per_tile, (uint32_t)p.G, 1};
    if (!encode_tiled(&tpo, dt, 4, p.out, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  if (p.n_splits > 1) {
    const uint64_t ns = (uint64_t)p.n_splits;
    const uint64_t dims[4] = {(uint64_t)D, ns, (uint64_t)p.Lq, (uint64_t)p.Hq * p.B};
    const uint64_t str[3] = {(uint64_t)D * 4, ns * D * 4, (uint64_t)p.Lq * ns * D * 4};
    const uint32_t box[4] = {32, 1, (uint32_t)p.q_per_tile, (uint32_t)p.G};
    if (!encode_tiled(&tpo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.o_part, dims, str, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  auto kern = p.n_splits > 1 ? prefill_kernel<D, BN, STAGES, BF16, PAGED, true>
                             : prefill_kernel<D, BN, STAGES, BF16, PAGED, false>;
  cudaError_t e = ensure_smem_limit(kern, L::kAlloc);
  if (e != cudaSuccess) return e;
  const dim3 grid(p.n_qtiles * p.n_splits, p.Hkv, p.B);
  kern<<<grid, kThreads, L::kAlloc, stream>>>(tq, tk, tv, tpo, p);
  return cudaGetLastError();
}

// The dense and paged kernels are separate instantiations, so the dense one carries none of
// the page-table reads, the per-sequence length or the V-tail clearing.
template <int D, int BN, int STAGES>
cudaError_t launch_d(const PrefillParams& p, bool bf16, cudaStream_t stream) {
  if (p.page_table)
    return bf16 ? launch_impl<D, BN, STAGES, true, true>(p, stream)
                : launch_impl<D, BN, STAGES, false, true>(p, stream);
  return bf16 ? launch_impl<D, BN, STAGES, true, false>(p, stream)
              : launch_impl<D, BN, STAGES, false, false>(p, stream);
}

}  // namespace

int prefill_block_n(int D) { return D == 256 ? 64 : 128; }

cudaError_t launch_prefill(const PrefillParams& p, Dtype operand, cudaStream_t stream) {
  const bool bf16 = operand == Dtype::BF16;
  switch (p.D) {
    case 64:
      return launch_d<64, 128, 5>(p, bf16, stream);
    case 128:
      return launch_d<128, 128, 3>(p, bf16, stream);
    case 256:
      return launch_d<256, 64, 2>(p, bf16, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace fa

// internal.h -- host-side interfaces between the C ABI (abi.cu) and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

struct fa_decode_args;

namespace fa {

// Element types of the public ABI (same numbering as fa_dtype in include/fa.h).
enum class Dtype : int { BF16 = 0, FP16 = 1, FP32 = 2 };

// ---------------------------------------------------------------------------------------
// Dense prefill
// ---------------------------------------------------------------------------------------
struct PrefillParams {
  // q [B,Hq,Lq,D] in bf16 or fp16 (the kernel's operand type); k/v either dense
  // [B,Hkv,Lkv,D] or, when page_table is set, pages [num_pages,Hkv,page_size,D].
  const void* q;
  const void* k;
  const void* v;
  void* out;            // [B,Hq,Lq,D] in out_dtype
  float* lse;           // [B,Hq,Lq] or nullptr
  const void* mask;     // additive [mask_batches,Lq,Lkv] or nullptr
  int mask_is_bf16;     // else fp32
  int mask_batches;     // 1 or B
  int B, Hq, Hkv, G, Lq, Lkv, D;
  int causal;
  float scale_log2;     // scale * log2(e)
  int q_per_tile;       // queries per 128-row tile (floor(128 / G))
  int n_qtiles;
  int n_splits;         // > 1: write partial states to o_part / lse_part
  float* o_part;        // [rows, n_splits, D] fp32
  float* lse_part;      // [rows, n_splits] fp32 (natural log)
  Dtype out_dtype;
  uint32_t* status;
  // Paged K/V (nullptr: dense).  Sequence b holds kv_lens[b] keys in pages
  // page_table[b * max_pages + i]; its Lq queries are its last Lq positions.
  const int32_t* page_table;
  const int32_t* kv_lens;
  int page_size, max_pages, num_pages;
};

// Launch on `stream`; returns a CUDA error code (cudaSuccess on launch success).
cudaError_t launch_prefill(const PrefillParams& p, Dtype operand, cudaStream_t stream);

// Tensor-core tile shape for a given head dimension (exposed for the planner).
int prefill_block_n(int D);

// ---------------------------------------------------------------------------------------
// Paged decode
// ---------------------------------------------------------------------------------------
struct DecodeParams {
  const void* q;          // [B,Hq,D] bf16
  const void* k_pages;    // [num_pages,Hkv,page_size,D]
  const void* v_pages;
  const int32_t* page_table;  // [B,max_pages]
  const int32_t* seq_lens;    // [B]
  int B, Hq, Hkv, G, D, page_size, max_pages, num_pages;
  int chunk;              // tokens per split (multiple of page_size)
  int n_chunks;           // ceil(max_seq_len / chunk)
  float scale_log2;
  float* o_part;          // [B*Hq, n_chunks, D]
  float* lse_part;        // [B*Hq, n_chunks]
  uint32_t* status;
  int f16;                // q and pages are fp16 (else bf16)
};
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream);

// ---------------------------------------------------------------------------------------
// MLA paged decode
// ---------------------------------------------------------------------------------------
struct MlaParams {
  const void* q_nope;     // [B,H,Dc]
  const void* q_pe;       // [B,H,Dr]
  const void* ckv;        // [num_pages,page_size,Dc]
  const void* kpe;        // [num_pages,page_size,Dr]
  const int32_t* page_table;
  const int32_t* seq_lens;
  int B, H, Dc, Dr, page_size, max_pages, num_pages;
  // Sequences [0, n_whole) take one CTA each (up to whole_chunk tokens) and write the final
  // out/lse directly.  Sequences [n_whole, B) are cut into n_chunks chunks of `chunk` tokens
  // whose partial states go to o_part/lse_part, rows counted from sequence n_whole.  The grid
  // is one-dimensional: n_whole + (B - n_whole) * n_chunks CTAs, the whole sequences first.
  int n_whole, whole_chunk;
  int chunk, n_chunks;
  float scale_log2;
  float* o_part;          // [(B - n_whole)*H, n_chunks, Dc]
  float* lse_part;        // [(B - n_whole)*H, n_chunks]
  void* out;              // [B,H,Dc] in the inputs' type (whole sequences)
  float* lse;             // [B,H] or nullptr (whole sequences)
  uint32_t* status;
  int f16;                // q, ckv and kpe are fp16 (else bf16)
  // 64 when page_size is a multiple of 64: a full 64-token tile is a slice of one page and is
  // copied with TMA boxes; 0: every stage is gathered row by row.  Set by launch_mla.
  int tma_rows;
};
cudaError_t launch_mla(const MlaParams& p, cudaStream_t stream);

// Self-test of the bounded-wait failure path (selftest.cu).
cudaError_t launch_selftest_wait(uint64_t limit_ns, uint32_t* status, cudaStream_t stream);
int mla_chunk_tokens(int B, int H, int max_seq_len);
// Plan of a full MLA call (see MlaParams): n_whole whole sequences of up to whole_chunk
// tokens, the rest in n_chunks chunks of `chunk` tokens.
struct MlaPlan {
  int n_whole, whole_chunk, chunk, n_chunks;
};
MlaPlan mla_plan(int B, int H, int max_seq_len);

// ---------------------------------------------------------------------------------------
// Merge of split states
// ---------------------------------------------------------------------------------------
struct MergeParams {
  const float* o_part;     // [rows, max_splits, D]
  const float* lse_part;   // [rows, max_splits]
  const int32_t* n_splits; // per-row split count or nullptr (= max_splits)
  // Alternative to n_splits for paged decode: the valid count of row r is
  // ceil(seq_lens[r / rows_per_seq] / chunk).
  const int32_t* seq_lens;
  int rows_per_seq, chunk;
  void* out;               // [rows, D] in out_dtype
  float* lse;              // [rows] or nullptr
  int rows, D, max_splits;
  Dtype out_dtype;
};
cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);

// Attention for fp32 inputs in fp32 on the CUDA cores (prefill_f32.cu): dense K/V, no split.
cudaError_t launch_prefill_f32(const PrefillParams& p, cudaStream_t stream);

// Checks a decode call's arguments (sizes, dtype, pointers, alignment of q, pages and out)
// as fa_decode_paged_ex does; sets the error text and returns the fa_status code.
int validate_decode_call(const fa_decode_args* a);

// ---------------------------------------------------------------------------------------
// Shared host helpers
// ---------------------------------------------------------------------------------------
uint32_t* device_status_ptr();  // the library's sticky device status word on this device
int set_error(int code, const char* msg);  // sets fa_last_error() text; returns code
int current_device_index();      // cudaGetDevice, or -1

// Sets a kernel's dynamic shared-memory limit once per (kernel, device): the first launch
// on each device does it; later launches, including ones captured into a CUDA graph, do not.
cudaError_t ensure_smem_limit_fn(const void* kernel, int bytes);
template <typename Kernel>
cudaError_t ensure_smem_limit(Kernel k, int bytes) {
  return ensure_smem_limit_fn(reinterpret_cast<const void*>(k), bytes);
}
int num_sms();                  // SM count of the current device (cached)
bool encode_tiled(CUtensorMap* map, CUtensorMapDataType t, int rank, const void* base,
                  const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                  CUtensorMapSwizzle swz);

}  // namespace fa

// abi.cu -- the C ABI declared in include/fa.h: argument validation, planning (split
// counts, KV chunking, grids sized from the SM count), tensor-map encoding, and launches.
// Argument errors are reported synchronously; nothing is enqueued for a rejected call.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <set>
#include <utility>

#include "../../include/fa.h"
#include "internal.h"
#include "sm103.cuh"

namespace fa {
namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(const char* where, cudaError_t e) {
  return fail(FA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Sticky device status word (one per device the library runs on).
__device__ uint32_t g_device_status;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t* g_status_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

uint32_t* device_status_ptr() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<uint32_t*>(p);
  }
  return g_status_ptr[dev];
}

int current_device_index() { return current_device(); }

int set_error(int code, const char* msg) { return fail(code, "%s", msg); }

cudaError_t ensure_smem_limit_fn(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({kernel, dev})) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({kernel, dev});
  return e;
}

int num_sms() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

bool encode_tiled(CUtensorMap* map, CUtensorMapDataType t, int rank, const void* base,
                  const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                  CUtensorMapSwizzle swz) {
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return false;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  }
  cuuint64_t d[5], s[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  return g_encode(map, t, rank, const_cast<void*>(base), d, s, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// ---------------------------------------------------------------------------------------
// Prefill planning
// ---------------------------------------------------------------------------------------
struct PrefillPlan {
  int G, q_per_tile, n_qtiles, n_splits;
  size_t part_bytes, total_bytes;
  size_t off_o, off_lse;
};

int validate_prefill(const fa_prefill_args* a, bool check_pointers = true) {
  if (!a) return fail(FA_ERR_INVALID_ARG, "fa_prefill: null argument struct");
  if (a->B < 0 || a->Lq < 0 || a->Lkv < 0)
    return fail(FA_ERR_INVALID_ARG, "fa_prefill: B, Lq, Lkv must be >= 0 (got %d, %d, %d)", a->B,
                a->Lq, a->Lkv);
  if (a->Hq <= 0 || a->Hkv <= 0 || a->Hq % a->Hkv != 0)
    return fail(FA_ERR_INVALID_ARG, "fa_prefill: need Hq, Hkv > 0 and Hq %% Hkv == 0 (got %d, %d)",
                a->Hq, a->Hkv);
  if (a->Hq / a->Hkv > 128)
    return fail(FA_ERR_UNSUPPORTED, "fa_prefill: query heads per kv head must be <= 128 (got %d)",
                a->Hq / a->Hkv);
  if (a->D != 64 && a->D != 128 && a->D != 256)
    return fail(FA_ERR_UNSUPPORTED, "fa_prefill: D must be 64, 128 or 256 (got %d)", a->D);
  if (a->dtype != FA_BF16 && a->dtype != FA_FP16 && a->dtype != FA_FP32)
    return fail(FA_ERR_INVALID_ARG, "fa_prefill: unknown dtype %d", (int)a->dtype);
  if (a->Hkv > 65535 || a->B > 65535)
    return fail(FA_ERR_UNSUPPORTED, "fa_prefill: B and Hkv must be <= 65535");
  if (!(a->scale == a->scale) || isinf(a->scale))
    return fail(FA_ERR_INVALID_ARG, "fa_prefill: scale must be finite");
  const bool work = a->B > 0 && a->Lq > 0;
  if (work && a->mask) {
    if (a->mask_batches != 1 && a->mask_batches != a->B)
      return fail(FA_ERR_INVALID_ARG, "fa_prefill: mask_batches must be 1 or B (got %d)",
                  a->mask_batches);
    if (a->mask_dtype != FA_FP32 && a->mask_dtype != FA_BF16)
      return fail(FA_ERR_UNSUPPORTED, "fa_prefill: mask dtype must be FA_FP32 or FA_BF16");
  }
  if (work && a->num_splits < 0)
    return fail(FA_ERR_INVALID_ARG, "fa_prefill: num_splits must be >= 0");
  if (a->page_size < 0) return fail(FA_ERR_INVALID_ARG, "fa_prefill: page_size must be >= 0");
  if (a->page_size > 0) {
    const int bn = prefill_block_n(a->D);
    if (a->page_size < 8 || a->page_size > bn || (a->page_size & (a->page_size - 1)) != 0)
      return fail(FA_ERR_UNSUPPORTED,
                  "fa_prefill: page_size must be a power of two in [8, %d] (got %d)", bn,
                  a->page_size);
    if (a->dtype == FA_FP32)
      return fail(FA_ERR_UNSUPPORTED, "fa_prefill: paged K/V must be bf16 or fp16");
    if (work && (a->max_pages <= 0 || a->num_pages <= 0))
      return fail(FA_ERR_INVALID_ARG, "fa_prefill: max_pages and num_pages must be > 0");
    if ((long)a->num_pages * a->Hkv > 2147483647L)
      return fail(FA_ERR_UNSUPPORTED, "fa_prefill: num_pages * Hkv must fit in int32");
    if ((long)a->Lkv > (long)a->max_pages * a->page_size)
      return fail(FA_ERR_INVALID_ARG, "fa_prefill: Lkv %d exceeds max_pages * page_size",
                  a->Lkv);
    if (work && check_pointers && (!a->page_table || !a->seq_lens))
      return fail(FA_ERR_INVALID_ARG, "fa_prefill: null page_table or seq_lens");
  }
  if (work && check_pointers) {
    if (!a->q || !a->out || ((a->Lkv > 0 || a->page_size > 0) && (!a->k || !a->v)))
      return fail(FA_ERR_INVALID_ARG, "fa_prefill: null q/k/v/out pointer");
    if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->out))
      return fail(FA_ERR_INVALID_ARG, "fa_prefill: q, k, v and out must be 16-byte aligned");
  }
  return FA_OK;
}

PrefillPlan plan_prefill(const fa_prefill_args* a) {
  PrefillPlan pl{};
  pl.G = a->Hq / a->Hkv;
  pl.q_per_tile = 128 / pl.G;
  pl.n_qtiles = a->Lq > 0 ? (a->Lq + pl.q_per_tile - 1) / pl.q_per_tile : 0;
  const int bn = prefill_block_n(a->D);
  const int kv_tiles = a->Lkv > 0 ? (a->Lkv + bn - 1) / bn : 0;
  int s = 1;
  if (a->dtype == FA_FP32) {
    // fp32 inputs run on the fp32 kernel, one warp per query row over all its keys
  } else if (a->num_splits > 0) {
    s = a->num_splits;
  } else if (kv_tiles > 0) {
    const long tiles = (long)pl.n_qtiles * a->Hkv * a->B;
    const int sms = num_sms() > 0 ? num_sms() : 148;
    // One CTA per SM fits.  Split the KV loop only when the tiles cover less than half the
    // SMs, into as many parts as still fit one wave, keeping at least four KV tiles per
    // part: each part pays a fixed cost (Q load, pipeline fill) and writes a partial state
    // as large as its output, so more parts than that cost more than they gain.
    if (tiles > 0 && tiles * 2 <= sms) {
      s = (int)(sms / tiles);
      const int cap = kv_tiles / 4 > 1 ? kv_tiles / 4 : 1;
      if (s > cap) s = cap;
    }
  }
  if (kv_tiles > 0 && s > kv_tiles) s = kv_tiles;
  if (s < 1 || a->dtype == FA_FP32) s = 1;
  pl.n_splits = s;
  const size_t rows = (size_t)a->B * a->Hq * a->Lq;
  size_t off = 0;
  if (s > 1) {
    pl.off_o = off;
    off = align_up(off + rows * s * a->D * sizeof(float), 256);
    pl.off_lse = off;
    off = align_up(off + rows * s * sizeof(float), 256);
  }
  pl.part_bytes = off;
  pl.total_bytes = off;
  return pl;
}

int run_prefill(const fa_prefill_args* a, cudaStream_t stream) {
  int rc = validate_prefill(a);
  if (rc != FA_OK) return rc;
  if (a->B == 0 || a->Lq == 0) return FA_OK;
  const PrefillPlan pl = plan_prefill(a);
  if (pl.total_bytes > 0) {
    if (!a->workspace || a->workspace_bytes < pl.total_bytes)
      return fail(FA_ERR_WORKSPACE, "fa_prefill: workspace of %zu bytes needed (got %zu)",
                  pl.total_bytes, a->workspace ? a->workspace_bytes : (size_t)0);
    if ((reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0)
      return fail(FA_ERR_INVALID_ARG, "fa_prefill: workspace must be 256-byte aligned");
  }
  uint32_t* status = device_status_ptr();
  if (!status) return fail(FA_ERR_CUDA, "fa_prefill: no usable CUDA device");
  uint8_t* ws = static_cast<uint8_t*>(a->workspace);
  PrefillParams p{};
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  const Dtype operand = static_cast<Dtype>(a->dtype);
  if (a->Lkv == 0 && a->page_size == 0) {  // keep the tensor maps valid; no key is read
    p.k = p.q;
    p.v = p.q;
  }
  if (a->page_size > 0) {
    p.page_table = a->page_table;
    p.kv_lens = a->seq_lens;
    p.page_size = a->page_size;
    p.max_pages = a->max_pages;
    p.num_pages = a->num_pages;
  }
  p.out = a->out;
  p.lse = a->lse;
  p.mask = a->mask;
  p.mask_is_bf16 = a->mask && a->mask_dtype == FA_BF16;
  p.mask_batches = a->mask_batches > 0 ? a->mask_batches : 1;
  p.B = a->B;
  p.Hq = a->Hq;
  p.Hkv = a->Hkv;
  p.G = pl.G;
  p.Lq = a->Lq;
  p.Lkv = a->Lkv;
  p.D = a->D;
  p.causal = a->causal ? 1 : 0;
  p.scale_log2 = a->scale * 1.44269504088896340736f;
  p.q_per_tile = pl.q_per_tile;
  p.n_qtiles = pl.n_qtiles;
  p.n_splits = pl.n_splits;
  p.o_part = pl.n_splits > 1 ? reinterpret_cast<float*>(ws + pl.off_o) : nullptr;
  p.lse_part = pl.n_splits > 1 ? reinterpret_cast<float*>(ws + pl.off_lse) : nullptr;
  p.out_dtype = static_cast<Dtype>(a->dtype);
  p.status = status;
  if (operand == Dtype::FP32) {
    cudaError_t e = launch_prefill_f32(p, stream);
    if (e != cudaSuccess) return cuda_fail("fa_prefill (fp32 kernel)", e);
    return FA_OK;
  }
  cudaError_t e = launch_prefill(p, operand, stream);
  if (e != cudaSuccess) return cuda_fail("fa_prefill (attention kernel)", e);
  if (pl.n_splits > 1) {
    MergeParams m{};
    m.o_part = p.o_part;
    m.lse_part = p.lse_part;
    m.out = a->out;
    m.lse = a->lse;
    m.rows = a->B * a->Hq * a->Lq;
    m.D = a->D;
    m.max_splits = pl.n_splits;
    m.out_dtype = static_cast<Dtype>(a->dtype);
    e = launch_merge(m, stream);
    if (e != cudaSuccess) return cuda_fail("fa_prefill (merge kernel)", e);
  }
  return FA_OK;
}

// ---------------------------------------------------------------------------------------
// Decode planning: fixed-size KV chunks, one partial state per (row, chunk)
// ---------------------------------------------------------------------------------------
int decode_chunk(int B, int Hq, int max_seq_len) {
  // 512-token chunks keep the partial-state traffic small next to the K/V stream; with
  // few sequences the chunk shrinks (to 128) so the grid still covers the SMs.
  const int sms = num_sms() > 0 ? num_sms() : 148;
  int chunk = 512;
  while (chunk > 128) {
    const long ctas = (long)B * (Hq >= 4 ? Hq / 4 : 1) * ((max_seq_len + chunk - 1) / chunk);
    if (ctas >= 4L * sms) break;
    chunk /= 2;
  }
  return chunk;
}

size_t split_ws_bytes(long rows, int n_chunks, int D) {
  return align_up((size_t)rows * n_chunks * D * sizeof(float), 256) +
         align_up((size_t)rows * n_chunks * sizeof(float), 256);
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

int fa_prefill(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
               int Hkv, int Lq, int Lkv, int D, int causal, float scale, void* stream) {
  fa_prefill_args a;
  memset(&a, 0, sizeof a);
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Lq = Lq;
  a.Lkv = Lkv;
  a.D = D;
  a.causal = causal;
  a.scale = scale;
  a.dtype = FA_BF16;
  a.num_splits = 1;
  return run_prefill(&a, static_cast<cudaStream_t>(stream));
}

int fa_prefill_ex(const fa_prefill_args* args, void* stream) {
  return run_prefill(args, static_cast<cudaStream_t>(stream));
}

size_t fa_prefill_workspace_size(const fa_prefill_args* args) {
  if (validate_prefill(args, false) != FA_OK) return 0;
  if (args->B == 0 || args->Lq == 0) return 0;
  return plan_prefill(args).total_bytes;
}

int fa_prefill_num_splits(const fa_prefill_args* args) {
  if (validate_prefill(args, false) != FA_OK) return 0;
  if (args->B == 0 || args->Lq == 0) return 1;
  return plan_prefill(args).n_splits;
}

int fa_prefill_paged(const void* q, const void* k_pages, const void* v_pages,
                     const int32_t* page_table, const int32_t* seq_lens, void* out, float* lse,
                     int B, int Hq, int Hkv, int Lq, int D, int page_size, int max_pages,
                     int num_pages, int max_seq_len, int causal, float scale, void* workspace,
                     size_t workspace_bytes, void* stream) {
  fa_prefill_args a;
  memset(&a, 0, sizeof a);
  a.q = q;
  a.k = k_pages;
  a.v = v_pages;
  a.out = out;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Lq = Lq;
  a.Lkv = max_seq_len;
  a.D = D;
  a.causal = causal;
  a.scale = scale;
  a.dtype = FA_BF16;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.page_size = page_size;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  return run_prefill(&a, static_cast<cudaStream_t>(stream));
}

size_t fa_prefill_paged_workspace_size(int B, int Hq, int Hkv, int Lq, int D, int max_seq_len) {
  fa_prefill_args a;
  memset(&a, 0, sizeof a);
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Lq = Lq;
  a.Lkv = max_seq_len;
  a.D = D;
  a.scale = 1.f;
  a.dtype = FA_BF16;  // the plan depends on neither the page geometry nor the pointers
  return fa_prefill_workspace_size(&a);
}

size_t fa_decode_workspace_size(int B, int Hq, int D, int max_seq_len) {
  if (B <= 0 || Hq <= 0 || D <= 0 || max_seq_len <= 0) return 0;
  // Enough for either decode path whatever Hkv and the page size are: the CUDA-core path's
  // chunk states, or the tensor-core path's split states, which are largest with one kv head
  // (the fewest (sequence, kv head) units, so the most splits).
  const int chunk = decode_chunk(B, Hq, max_seq_len);
  const size_t cc = split_ws_bytes((long)B * Hq, (max_seq_len + chunk - 1) / chunk, D);
  fa_prefill_args p;
  memset(&p, 0, sizeof p);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = 1;
  p.Lq = 1;
  p.Lkv = max_seq_len;
  p.D = D;
  p.dtype = FA_BF16;
  const size_t tc = plan_prefill(&p).total_bytes;
  return cc > tc ? cc : tc;
}

int fa_decode_chunk_tokens(int B, int Hq, int max_seq_len) {
  return decode_chunk(B > 0 ? B : 1, Hq > 0 ? Hq : 1, max_seq_len > 0 ? max_seq_len : 1);
}

}  // extern "C"

namespace fa {
namespace {

int check_decode(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                 const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int page_size,
                 int max_pages_per_seq, int num_pages, int max_seq_len, float scale) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0)
    return fail(FA_ERR_INVALID_ARG, "fa_decode_paged: need B >= 0, Hq, Hkv > 0, Hq %% Hkv == 0");
  if (D != 64 && D != 128 && D != 256)
    return fail(FA_ERR_UNSUPPORTED, "fa_decode_paged: D must be 64, 128 or 256 (got %d)", D);
  if (Hq / Hkv > 128)
    return fail(FA_ERR_UNSUPPORTED, "fa_decode_paged: query heads per kv head must be <= 128 (got %d)",
                Hq / Hkv);
  if (page_size <= 0 || (page_size & (page_size - 1)) != 0)
    return fail(FA_ERR_INVALID_ARG, "fa_decode_paged: page_size must be a power of two (got %d)",
                page_size);
  if (max_pages_per_seq < 0 || num_pages < 0 || max_seq_len < 0)
    return fail(FA_ERR_INVALID_ARG, "fa_decode_paged: negative size");
  if ((long)max_pages_per_seq * page_size < max_seq_len)
    return fail(FA_ERR_INVALID_ARG,
                "fa_decode_paged: max_seq_len %d exceeds max_pages_per_seq*page_size", max_seq_len);
  if (Hkv > 65535 || B > 65535) return fail(FA_ERR_UNSUPPORTED, "fa_decode_paged: B, Hkv <= 65535");
  if (!(scale == scale) || isinf(scale))
    return fail(FA_ERR_INVALID_ARG, "fa_decode_paged: scale must be finite");
  if (B == 0) return FA_OK;
  if (!q || !seq_lens || (max_seq_len > 0 && (!k_pages || !v_pages || !page_table)))
    return fail(FA_ERR_INVALID_ARG, "fa_decode_paged: null pointer");
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages))
    return fail(FA_ERR_INVALID_ARG, "fa_decode_paged: q, k_pages, v_pages must be 16-byte aligned");
  return FA_OK;
}

// The two decode kernels.  The CUDA-core split-KV kernel (decode.cu) takes power-of-two
// groups of at most 16 query heads per kv head with G*D <= 1024 and any power-of-two page
// size.  The paged attention kernel (prefill.cu with one query per sequence: the group's
// heads packed into its 128-row tile, S and P V on the tensor cores) takes any group of at
// most 128 heads and pages of 8 tokens up to its key tile.
bool cc_decode_supports(int G, int D) { return G <= 16 && (G & (G - 1)) == 0 && G * D <= 1024; }

bool tc_decode_supports(int G, int D, int page_size, int num_pages, int Hkv) {
  return G <= 128 && page_size >= 8 && page_size <= prefill_block_n(D) &&
         (page_size & (page_size - 1)) == 0 && (long)num_pages * Hkv <= 2147483647L;
}

// fa_prefill_ex arguments of a decode call on the tensor-core path: Lq = 1, the query being
// the sequence's last position, so it sees all of the sequence's keys.
fa_prefill_args decode_as_prefill(const fa_decode_args* a) {
  fa_prefill_args p;
  memset(&p, 0, sizeof p);
  p.q = a->q;
  p.k = a->k_pages;
  p.v = a->v_pages;
  p.out = a->out;
  p.lse = a->lse;
  p.B = a->B;
  p.Hq = a->Hq;
  p.Hkv = a->Hkv;
  p.Lq = 1;
  p.Lkv = a->max_seq_len;
  p.D = a->D;
  p.scale = a->scale;
  p.dtype = a->dtype;
  p.workspace = a->workspace;
  p.workspace_bytes = a->workspace_bytes;
  p.page_table = a->page_table;
  p.seq_lens = a->seq_lens;
  p.page_size = a->page_size;
  p.max_pages = a->max_pages_per_seq;
  p.num_pages = a->num_pages;
  return p;
}

struct DecodePlan {
  fa_decode_path path;
  int chunk, n_chunks;   // CUDA-core path: tokens per chunk, chunks of the longest sequence
  int n_splits;          // KV splits per (sequence, kv head)
  int launches;
  size_t ws_bytes;
};

// Chooses the kernel for a validated decode call.  Automatic choice: the tensor-core path
// when the (sequence, kv head) units alone fill the GPU (its planner then splits nothing) or
// when the CUDA-core kernel cannot take the group size; otherwise the CUDA-core kernel,
// whose fixed-size chunks spread few long sequences over every SM.  No key at all
// (max_seq_len == 0): only the merge runs, writing empty rows.
int plan_decode(const fa_decode_args* a, DecodePlan* pl) {
  const int G = a->Hq / a->Hkv;
  const bool cc = cc_decode_supports(G, a->D);
  const bool tc = tc_decode_supports(G, a->D, a->page_size, a->num_pages, a->Hkv);
  memset(pl, 0, sizeof *pl);
  if (a->path != FA_DECODE_AUTO && a->path != FA_DECODE_CUDA_CORES &&
      a->path != FA_DECODE_TENSOR_CORES)
    return fail(FA_ERR_INVALID_ARG, "fa_decode_paged: unknown path %d", (int)a->path);
  if (a->path == FA_DECODE_CUDA_CORES && !cc)
    return fail(FA_ERR_UNSUPPORTED,
                "fa_decode_paged: the CUDA-core path needs a power-of-two group of at most 16 "
                "heads with G*D <= 1024 (got G=%d, D=%d)", G, a->D);
  if (a->path == FA_DECODE_TENSOR_CORES && !tc)
    return fail(FA_ERR_UNSUPPORTED,
                "fa_decode_paged: the tensor-core path needs page_size a power of two in "
                "[8, %d] (got %d)", prefill_block_n(a->D), a->page_size);
  if (!cc && !tc)
    return fail(FA_ERR_UNSUPPORTED,
                "fa_decode_paged: G=%d needs the tensor-core path, which takes page sizes that "
                "are powers of two in [8, %d] (got %d)", G, prefill_block_n(a->D), a->page_size);
  const int sms = num_sms() > 0 ? num_sms() : 148;
  bool use_tc = a->path == FA_DECODE_TENSOR_CORES ||
                (a->path == FA_DECODE_AUTO && tc && (!cc || 2L * a->B * a->Hkv > sms));
  if (a->max_seq_len == 0) {
    pl->path = use_tc ? FA_DECODE_TENSOR_CORES : FA_DECODE_CUDA_CORES;
    pl->launches = a->B > 0 ? 1 : 0;
    return FA_OK;
  }
  if (use_tc) {
    const fa_prefill_args p = decode_as_prefill(a);
    const PrefillPlan pp = plan_prefill(&p);
    pl->path = FA_DECODE_TENSOR_CORES;
    pl->n_splits = pp.n_splits;
    pl->launches = a->B > 0 ? 1 + (pp.n_splits > 1) : 0;
    pl->ws_bytes = a->B > 0 ? pp.total_bytes : 0;
    return FA_OK;
  }
  pl->path = FA_DECODE_CUDA_CORES;
  pl->chunk = decode_chunk(a->B > 0 ? a->B : 1, a->Hq, a->max_seq_len);
  pl->n_chunks = (a->max_seq_len + pl->chunk - 1) / pl->chunk;
  pl->n_splits = pl->n_chunks;
  pl->launches = a->B > 0 ? 2 : 0;
  pl->ws_bytes = a->B > 0 ? split_ws_bytes((long)a->B * a->Hq, pl->n_chunks, a->D) : 0;
  return FA_OK;
}

int check_decode_struct(const fa_decode_args* a) {
  if (!a) return fail(FA_ERR_INVALID_ARG, "fa_decode_paged: null argument struct");
  if (a->dtype != FA_BF16 && a->dtype != FA_FP16)
    return fail(FA_ERR_UNSUPPORTED, "fa_decode_paged: dtype must be FA_BF16 or FA_FP16");
  return check_decode(a->q, a->k_pages, a->v_pages, a->page_table, a->seq_lens, a->B, a->Hq,
                      a->Hkv, a->D, a->page_size, a->max_pages_per_seq, a->num_pages,
                      a->max_seq_len, a->scale);
}

cudaError_t decode_states(const void* q, const void* k_pages, const void* v_pages,
                          const int32_t* page_table, const int32_t* seq_lens, float* o_part,
                          float* lse_part, int chunk, int n_chunks, int B, int Hq, int Hkv, int D,
                          int page_size, int max_pages_per_seq, int num_pages, float scale,
                          uint32_t* status, cudaStream_t st, bool f16 = false) {
  DecodeParams p{};
  p.f16 = f16 ? 1 : 0;
  p.q = q;
  p.k_pages = k_pages;
  p.v_pages = v_pages;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.D = D;
  p.page_size = page_size;
  p.max_pages = max_pages_per_seq;
  p.num_pages = num_pages;
  p.chunk = chunk;
  p.n_chunks = n_chunks;
  p.scale_log2 = scale * 1.44269504088896340736f;
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.status = status;
  return launch_decode(p, st);
}

int check_mla(const void* q_nope, const void* q_pe, const void* ckv_pages, const void* kpe_pages,
              const int32_t* page_table, const int32_t* seq_lens, int B, int H, int Dc, int Dr,
              int page_size, int max_pages_per_seq, int num_pages, int max_seq_len, float scale) {
  if (B < 0 || H <= 0 || Dc <= 0 || Dr < 0)
    return fail(FA_ERR_INVALID_ARG, "mla_decode_paged: need B >= 0, H, Dc > 0, Dr >= 0");
  if (Dc != 512 || Dr != 64)
    return fail(FA_ERR_UNSUPPORTED, "mla_decode_paged: supports Dc=512, Dr=64 (got %d, %d)", Dc, Dr);
  if (H > 1024)
    return fail(FA_ERR_UNSUPPORTED, "mla_decode_paged: H must be <= 1024 (got %d)", H);
  if (page_size <= 0) return fail(FA_ERR_INVALID_ARG, "mla_decode_paged: page_size must be > 0");
  if (max_pages_per_seq < 0 || num_pages < 0 || max_seq_len < 0)
    return fail(FA_ERR_INVALID_ARG, "mla_decode_paged: negative size");
  if ((long)max_pages_per_seq * page_size < max_seq_len)
    return fail(FA_ERR_INVALID_ARG, "mla_decode_paged: max_seq_len exceeds max_pages_per_seq*page_size");
  if (B > 65535) return fail(FA_ERR_UNSUPPORTED, "mla_decode_paged: B <= 65535");
  if (!(scale == scale) || isinf(scale))
    return fail(FA_ERR_INVALID_ARG, "mla_decode_paged: scale must be finite");
  if (B == 0) return FA_OK;
  if (!q_nope || !q_pe || !seq_lens || (max_seq_len > 0 && (!ckv_pages || !kpe_pages || !page_table)))
    return fail(FA_ERR_INVALID_ARG, "mla_decode_paged: null pointer");
  if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(ckv_pages) || !aligned16(kpe_pages))
    return fail(FA_ERR_INVALID_ARG, "mla_decode_paged: tensors must be 16-byte aligned");
  return FA_OK;
}

cudaError_t mla_states(const void* q_nope, const void* q_pe, const void* ckv_pages,
                       const void* kpe_pages, const int32_t* page_table, const int32_t* seq_lens,
                       float* o_part, float* lse_part, const MlaPlan& pl, int B, int H,
                       int Dc, int Dr, int page_size, int max_pages_per_seq, int num_pages,
                       float scale, uint32_t* status, cudaStream_t st, void* out = nullptr,
                       float* lse = nullptr, bool f16 = false) {
  MlaParams p{};
  p.f16 = f16 ? 1 : 0;
  p.n_whole = pl.n_whole;
  p.whole_chunk = pl.whole_chunk;
  p.out = out;
  p.lse = lse;
  p.q_nope = q_nope;
  p.q_pe = q_pe;
  p.ckv = ckv_pages;
  p.kpe = kpe_pages;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.B = B;
  p.H = H;
  p.Dc = Dc;
  p.Dr = Dr;
  p.page_size = page_size;
  p.max_pages = max_pages_per_seq;
  p.num_pages = num_pages;
  p.chunk = pl.chunk;
  p.n_chunks = pl.n_chunks;
  p.scale_log2 = scale * 1.44269504088896340736f;
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.status = status;
  return launch_mla(p, st);
}

// Splits a caller workspace into the partial-output and partial-lse arrays.
void carve(void* ws, long rows, int n_chunks, int D, float** o, float** l) {
  *o = static_cast<float*>(ws);
  *l = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                align_up((size_t)rows * n_chunks * D * sizeof(float), 256));
}

int merge_chunks(float* o_part, float* lse_part, const int32_t* seq_lens, int rows_per_seq,
                 int chunk, int n_chunks, void* out, float* lse, int rows, int D, cudaStream_t st,
                 const char* who, Dtype out_dtype = Dtype::BF16) {
  MergeParams m{};
  m.o_part = o_part;
  m.lse_part = lse_part;
  m.seq_lens = n_chunks > 0 ? seq_lens : nullptr;
  m.rows_per_seq = rows_per_seq;
  m.chunk = chunk;
  m.out = out;
  m.lse = lse;
  m.rows = rows;
  m.D = D;
  m.max_splits = n_chunks;
  m.out_dtype = out_dtype;
  cudaError_t e = launch_merge(m, st);
  if (e != cudaSuccess) return cuda_fail(who, e);
  return FA_OK;
}

}  // namespace

int validate_decode_call(const fa_decode_args* a) {
  int rc = check_decode_struct(a);
  if (rc != FA_OK || a->B == 0) return rc;
  if (!a->out || !aligned16(a->out))
    return fail(FA_ERR_INVALID_ARG, "fa_decode_paged: out must be a 16-byte aligned pointer");
  return FA_OK;
}

}  // namespace fa

extern "C" {

int fa_decode_paged_ex(const fa_decode_args* a, void* stream) {
  int rc = validate_decode_call(a);
  if (rc != FA_OK || a->B == 0) return rc;
  DecodePlan pl;
  rc = plan_decode(a, &pl);
  if (rc != FA_OK) return rc;
  const int B = a->B, Hq = a->Hq, D = a->D;
  if (pl.ws_bytes > 0 && (!a->workspace || a->workspace_bytes < pl.ws_bytes))
    return fail(FA_ERR_WORKSPACE, "fa_decode_paged: workspace of %zu bytes needed (got %zu)",
                pl.ws_bytes, a->workspace ? a->workspace_bytes : (size_t)0);
  if (pl.ws_bytes > 0 && (reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0)
    return fail(FA_ERR_INVALID_ARG, "fa_decode_paged: workspace must be 256-byte aligned");
  uint32_t* status = device_status_ptr();
  if (!status) return fail(FA_ERR_CUDA, "fa_decode_paged: no usable CUDA device");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool f16 = a->dtype == FA_FP16;
  if (pl.path == FA_DECODE_TENSOR_CORES && a->max_seq_len > 0) {
    const fa_prefill_args p = decode_as_prefill(a);
    return run_prefill(&p, st);
  }
  float *o_part = nullptr, *lse_part = nullptr;
  if (pl.n_chunks > 0) {
    carve(a->workspace, (long)B * Hq, pl.n_chunks, D, &o_part, &lse_part);
    cudaError_t e = decode_states(a->q, a->k_pages, a->v_pages, a->page_table, a->seq_lens,
                                  o_part, lse_part, pl.chunk, pl.n_chunks, B, Hq, a->Hkv, D,
                                  a->page_size, a->max_pages_per_seq, a->num_pages, a->scale,
                                  status, st, f16);
    if (e != cudaSuccess) return cuda_fail("fa_decode_paged (decode kernel)", e);
  }
  // with no key anywhere (n_chunks == 0) the merge alone writes the empty rows
  return merge_chunks(o_part, lse_part, a->seq_lens, Hq, pl.chunk, pl.n_chunks, a->out, a->lse,
                      B * Hq, D, st, "fa_decode_paged (merge kernel)", f16 ? Dtype::FP16 : Dtype::BF16);
}

int fa_decode_get_plan(const fa_decode_args* a, fa_decode_plan* plan) {
  if (!plan) return fail(FA_ERR_INVALID_ARG, "fa_decode_get_plan: null plan");
  if (!a) return fail(FA_ERR_INVALID_ARG, "fa_decode_get_plan: null argument struct");
  const fa_decode_args b = *a;
  // sizes only: the pointers are not read
  int rc = check_decode(reinterpret_cast<const void*>(4096), reinterpret_cast<const void*>(4096),
                        reinterpret_cast<const void*>(4096), reinterpret_cast<const int32_t*>(4096),
                        reinterpret_cast<const int32_t*>(4096), b.B, b.Hq, b.Hkv, b.D, b.page_size,
                        b.max_pages_per_seq, b.num_pages, b.max_seq_len, b.scale);
  if (rc == FA_OK && b.dtype != FA_BF16 && b.dtype != FA_FP16)
    rc = fail(FA_ERR_UNSUPPORTED, "fa_decode_paged: dtype must be FA_BF16 or FA_FP16");
  if (rc != FA_OK) return rc;
  DecodePlan pl;
  rc = plan_decode(&b, &pl);
  if (rc != FA_OK) return rc;
  plan->path = pl.path;
  plan->n_splits = pl.n_splits;
  plan->launches = pl.launches;
  plan->workspace_bytes = pl.ws_bytes;
  return FA_OK;
}

int fa_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                    const int32_t* page_table, const int32_t* seq_lens, void* out, float* lse,
                    int B, int Hq, int Hkv, int D, int page_size, int max_pages_per_seq,
                    int num_pages, int max_seq_len, float scale, void* workspace,
                    size_t workspace_bytes, void* stream) {
  const fa_decode_args a = {q, k_pages, v_pages, page_table, seq_lens, out, lse, B, Hq, Hkv, D,
                            page_size, max_pages_per_seq, num_pages, max_seq_len, scale, FA_BF16,
                            workspace, workspace_bytes, FA_DECODE_AUTO};
  return fa_decode_paged_ex(&a, stream);
}

int fa_decode_paged_states(const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* page_table, const int32_t* seq_lens, float* o_parts,
                           float* lse_parts, int n_chunks, int B, int Hq, int Hkv, int D,
                           int page_size, int max_pages_per_seq, int num_pages, int max_seq_len,
                           float scale, void* stream) {
  int rc = check_decode(q, k_pages, v_pages, page_table, seq_lens, B, Hq, Hkv, D, page_size,
                        max_pages_per_seq, num_pages, max_seq_len, scale);
  if (rc != FA_OK || B == 0 || max_seq_len == 0) return rc;
  if (!cc_decode_supports(Hq / Hkv, D))
    return fail(FA_ERR_UNSUPPORTED,
                "fa_decode_paged_states: the split states come from the CUDA-core kernel, which "
                "needs a power-of-two group of at most 16 heads with G*D <= 1024");
  const int chunk = decode_chunk(B, Hq, max_seq_len);
  const int want = (max_seq_len + chunk - 1) / chunk;
  if (n_chunks != want)
    return fail(FA_ERR_INVALID_ARG, "fa_decode_paged_states: n_chunks must be %d (got %d)", want,
                n_chunks);
  if (!o_parts || !lse_parts || !aligned16(o_parts))
    return fail(FA_ERR_INVALID_ARG, "fa_decode_paged_states: o_parts/lse_parts missing or misaligned");
  uint32_t* status = device_status_ptr();
  if (!status) return fail(FA_ERR_CUDA, "fa_decode_paged_states: no usable CUDA device");
  cudaError_t e = decode_states(q, k_pages, v_pages, page_table, seq_lens, o_parts, lse_parts,
                                chunk, n_chunks, B, Hq, Hkv, D, page_size, max_pages_per_seq,
                                num_pages, scale, status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("fa_decode_paged_states", e);
  return FA_OK;
}

size_t mla_decode_workspace_size(int B, int H, int Dc, int max_seq_len) {
  if (B <= 0 || H <= 0 || Dc <= 0 || max_seq_len <= 0) return 0;
  const MlaPlan pl = mla_plan(B, H, max_seq_len);
  if (pl.n_whole >= B) return 0;
  return split_ws_bytes((long)(B - pl.n_whole) * H, pl.n_chunks, Dc);
}

int mla_decode_chunk_tokens(int B, int H, int max_seq_len) {
  return mla_chunk_tokens(B > 0 ? B : 1, H > 0 ? H : 1, max_seq_len > 0 ? max_seq_len : 1);
}

int mla_decode_paged_ex(const mla_decode_args* a, void* stream) {
  if (!a) return fail(FA_ERR_INVALID_ARG, "mla_decode_paged: null argument struct");
  if (a->dtype != FA_BF16 && a->dtype != FA_FP16)
    return fail(FA_ERR_UNSUPPORTED, "mla_decode_paged: dtype must be FA_BF16 or FA_FP16");
  const int B = a->B, H = a->H, Dc = a->Dc, max_seq_len = a->max_seq_len;
  int rc = check_mla(a->q_nope, a->q_pe, a->ckv_pages, a->kpe_pages, a->page_table, a->seq_lens,
                     B, H, Dc, a->Dr, a->page_size, a->max_pages_per_seq, a->num_pages,
                     max_seq_len, a->scale);
  if (rc != FA_OK || B == 0) return rc;
  if (!a->out || !aligned16(a->out))
    return fail(FA_ERR_INVALID_ARG, "mla_decode_paged: out must be a 16-byte aligned pointer");
  if (max_seq_len == 0) {
    // no sequence holds a key: every row is empty (out 0, lse -inf)
    return merge_chunks(nullptr, nullptr, a->seq_lens, H, 1, 0, a->out, a->lse, B * H, Dc,
                        static_cast<cudaStream_t>(stream), "mla_decode_paged (merge kernel)",
                        a->dtype == FA_FP16 ? Dtype::FP16 : Dtype::BF16);
  }
  const MlaPlan pl = mla_plan(B, H, max_seq_len);
  const int n_split = B - pl.n_whole;  // sequences cut into chunks
  const size_t need = n_split > 0 ? split_ws_bytes((long)n_split * H, pl.n_chunks, Dc) : 0;
  if (need > 0 && (!a->workspace || a->workspace_bytes < need))
    return fail(FA_ERR_WORKSPACE, "mla_decode_paged: workspace of %zu bytes needed (got %zu)", need,
                a->workspace ? a->workspace_bytes : (size_t)0);
  if (need > 0 && (reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0)
    return fail(FA_ERR_INVALID_ARG, "mla_decode_paged: workspace must be 256-byte aligned");
  uint32_t* status = device_status_ptr();
  if (!status) return fail(FA_ERR_CUDA, "mla_decode_paged: no usable CUDA device");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool f16 = a->dtype == FA_FP16;
  float *o_part = nullptr, *lse_part = nullptr;
  if (n_split > 0) carve(a->workspace, (long)n_split * H, pl.n_chunks, Dc, &o_part, &lse_part);
  // one launch: whole sequences write their final rows, the others their chunks' states
  cudaError_t e = mla_states(a->q_nope, a->q_pe, a->ckv_pages, a->kpe_pages, a->page_table,
                             a->seq_lens, o_part, lse_part, pl, B, H, Dc, a->Dr, a->page_size,
                             a->max_pages_per_seq, a->num_pages, a->scale, status, st, a->out,
                             a->lse, f16);
  if (e != cudaSuccess) return cuda_fail("mla_decode_paged (MLA kernel)", e);
  if (n_split == 0) return FA_OK;
  // merge the split sequences' rows, which follow the whole ones in out, lse and seq_lens
  const size_t row0 = (size_t)pl.n_whole * H;
  void* out_split = static_cast<uint8_t*>(a->out) + row0 * Dc * 2;
  float* lse_split = a->lse ? a->lse + row0 : nullptr;
  return merge_chunks(o_part, lse_part, a->seq_lens + pl.n_whole, H, pl.chunk, pl.n_chunks,
                      out_split, lse_split, n_split * H, Dc, st, "mla_decode_paged (merge kernel)",
                      f16 ? Dtype::FP16 : Dtype::BF16);
}

int mla_decode_paged(const void* q_nope, const void* q_pe, const void* ckv_pages,
                     const void* kpe_pages, const int32_t* page_table, const int32_t* seq_lens,
                     void* out, float* lse, int B, int H, int Dc, int Dr, int page_size,
                     int max_pages_per_seq, int num_pages, int max_seq_len, float scale,
                     void* workspace, size_t workspace_bytes, void* stream) {
  const mla_decode_args a = {q_nope, q_pe, ckv_pages, kpe_pages, page_table, seq_lens, out, lse,
                             B, H, Dc, Dr, page_size, max_pages_per_seq, num_pages, max_seq_len,
                             scale, FA_BF16, workspace, workspace_bytes};
  return mla_decode_paged_ex(&a, stream);
}

int mla_decode_paged_states(const void* q_nope, const void* q_pe, const void* ckv_pages,
                            const void* kpe_pages, const int32_t* page_table,
                            const int32_t* seq_lens, float* o_parts, float* lse_parts,
                            int n_chunks, int B, int H, int Dc, int Dr, int page_size,
                            int max_pages_per_seq, int num_pages, int max_seq_len, float scale,
                            void* stream) {
  int rc = check_mla(q_nope, q_pe, ckv_pages, kpe_pages, page_table, seq_lens, B, H, Dc, Dr,
                     page_size, max_pages_per_seq, num_pages, max_seq_len, scale);
  if (rc != FA_OK || B == 0 || max_seq_len == 0) return rc;
  const int chunk = mla_chunk_tokens(B, H, max_seq_len);
  const int want = (max_seq_len + chunk - 1) / chunk;
  if (n_chunks != want)
    return fail(FA_ERR_INVALID_ARG, "mla_decode_paged_states: n_chunks must be %d (got %d)", want,
                n_chunks);
  if (!o_parts || !lse_parts || !aligned16(o_parts))
    return fail(FA_ERR_INVALID_ARG, "mla_decode_paged_states: o_parts/lse_parts missing or misaligned");
  uint32_t* status = device_status_ptr();
  if (!status) return fail(FA_ERR_CUDA, "mla_decode_paged_states: no usable CUDA device");
  MlaPlan pl{};
  pl.n_whole = 0;
  pl.chunk = chunk;
  pl.n_chunks = n_chunks;
  cudaError_t e = mla_states(q_nope, q_pe, ckv_pages, kpe_pages, page_table, seq_lens, o_parts,
                             lse_parts, pl, B, H, Dc, Dr, page_size, max_pages_per_seq, num_pages,
                             scale, status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("mla_decode_paged_states", e);
  return FA_OK;
}

int fa_merge_states(const float* o_parts, const float* lse_parts, const int32_t* n_splits,
                    void* out, float* lse, int rows, int D, int max_splits, fa_dtype out_dtype,
                    void* stream) {
  if (rows < 0 || D <= 0 || D % 4 != 0 || max_splits < 0)
    return fail(FA_ERR_INVALID_ARG, "fa_merge_states: need rows >= 0, D > 0 with D %% 4 == 0, max_splits >= 0");
  if (D > 512) return fail(FA_ERR_UNSUPPORTED, "fa_merge_states: D must be <= 512 (got %d)", D);
  if (out_dtype != FA_BF16 && out_dtype != FA_FP16 && out_dtype != FA_FP32)
    return fail(FA_ERR_INVALID_ARG, "fa_merge_states: unknown out dtype %d", (int)out_dtype);
  if (rows == 0) return FA_OK;
  if (!out || (max_splits > 0 && (!o_parts || !lse_parts)))
    return fail(FA_ERR_INVALID_ARG, "fa_merge_states: null pointer");
  if (!aligned16(o_parts) || !aligned16(out))
    return fail(FA_ERR_INVALID_ARG, "fa_merge_states: o_parts and out must be 16-byte aligned");
  if (!device_status_ptr()) return fail(FA_ERR_CUDA, "fa_merge_states: no usable CUDA device");
  MergeParams m{};
  m.o_part = o_parts;
  m.lse_part = lse_parts;
  m.n_splits = n_splits;
  m.out = out;
  m.lse = lse;
  m.rows = rows;
  m.D = D;
  m.max_splits = max_splits;
  m.out_dtype = static_cast<Dtype>(out_dtype);
  cudaError_t e = launch_merge(m, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("fa_merge_states", e);
  return FA_OK;
}

int fa_get_device_status(void* stream) {
  uint32_t* st = device_status_ptr();
  if (!st) return fail(FA_ERR_CUDA, "fa_get_device_status: no usable CUDA device");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("fa_get_device_status (synchronize)", e);
  uint32_t v = 0;
  e = cudaMemcpy(&v, st, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail("fa_get_device_status (read)", e);
  const uint32_t zero = 0;
  e = cudaMemcpy(st, &zero, sizeof zero, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail("fa_get_device_status (clear)", e);
  if (v == kDevTimeout) return fail(FA_ERR_TIMEOUT, "a bounded wait inside a kernel ran out");
  if (v == kDevBounds) return fail(FA_ERR_BOUNDS, "a page id or sequence length was out of range");
  return FA_OK;
}

int fa_selftest_wait_timeout(unsigned timeout_us, void* stream) {
  if (timeout_us == 0 || timeout_us > kWaitLimitNs / 1000)
    return fail(FA_ERR_INVALID_ARG, "fa_selftest_wait_timeout: timeout_us must be in [1, %llu]",
                static_cast<unsigned long long>(kWaitLimitNs / 1000));
  uint32_t* status = device_status_ptr();
  if (!status) return fail(FA_ERR_CUDA, "fa_selftest_wait_timeout: no usable CUDA device");
  cudaError_t e = launch_selftest_wait(static_cast<uint64_t>(timeout_us) * 1000, status,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("fa_selftest_wait_timeout", e);
  return FA_OK;
}

const char* fa_last_error(void) { return g_err; }

int fa_version(void) { return 400; }

}  // extern "C"

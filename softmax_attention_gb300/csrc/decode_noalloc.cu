// decode_noalloc.cu -- paged decode for callers that cannot allocate device memory.
//
// fa_decode_paged keeps its split-KV partial states in a workspace the caller allocates.
// Some callers have no way to allocate at the point where they decode: a runtime whose
// device memory is owned by its own arena allocator (and forbids cudaMalloc next to it), an
// embedding host that only hands the library pre-existing buffers, or a serving loop that
// must not allocate on its latency-critical path.  fa_decode_paged_noalloc serves them: it
// runs exactly the fa_decode_paged computation, with the scratch taken from one fixed
// device array that belongs to this library.
//
// The array is a file-scope __device__ variable, so every GPU that loads the library holds
// its kNoAllocScratchBytes until the process exits.  Its address is a device address that
// host code can only learn through cudaGetSymbolAddress (the array's name in host code is a
// host-side stand-in, not a device pointer); that lookup happens once per device, on the
// first call made with that device current, and the address is kept for the life of the
// process (a device reset inside the process is not supported; see include/fa.h).
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "../../include/fa.h"
#include "internal.h"

namespace fa {
namespace {

// Largest scratch the no-allocation entry point can use: 32 MiB holds the partial states
// of, e.g., 128 sequences x 32 query heads x 4096 tokens at D = 128 (16.9 MB).
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    char msg[160];
    snprintf(msg, sizeof msg, "fa_decode_paged_noalloc: no usable CUDA device (%s)",
             cudaGetErrorString(e));
    return set_error(FA_ERR_CUDA, msg);
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      char msg[160];
      snprintf(msg, sizeof msg, "fa_decode_paged_noalloc: cudaGetSymbolAddress failed (%s)",
               cudaGetErrorString(e));
      return set_error(FA_ERR_CUDA, msg);
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" int fa_decode_paged_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                       const int32_t* page_table, const int32_t* seq_lens,
                                       void* out, float* lse, int B, int Hq, int Hkv, int D,
                                       int page_size, int max_pages_per_seq, int num_pages,
                                       int max_seq_len, float scale, void* stream) {
  fa_decode_args a = {q, k_pages, v_pages, page_table, seq_lens, out, lse, B, Hq, Hkv, D,
                      page_size, max_pages_per_seq, num_pages, max_seq_len, scale, FA_BF16,
                      nullptr, 0, FA_DECODE_AUTO};
  // The arguments are checked first, exactly as fa_decode_paged checks them, so a malformed
  // call gets the error that names its bad argument.
  int rc = fa::validate_decode_call(&a);
  if (rc != FA_OK || B == 0) return rc;
  // The scratch this problem needs (the plan fa_decode_paged would follow) must fit the
  // fixed array; larger problems are refused before anything touches the device.
  fa_decode_plan plan;
  rc = fa_decode_get_plan(&a, &plan);
  if (rc != FA_OK) return rc;
  if (plan.workspace_bytes > fa::kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "fa_decode_paged_noalloc: this problem needs %zu bytes of scratch but the built-in "
             "array holds %zu; call fa_decode_paged with a caller workspace instead",
             plan.workspace_bytes, fa::kNoAllocScratchBytes);
    return fa::set_error(FA_ERR_WORKSPACE, msg);
  }
  void* scratch = nullptr;
  rc = fa::scratch_address(&scratch);
  if (rc != FA_OK) return rc;
  // Both decode kernels write every partial state the merge later reads, so no part of the
  // array has to start at zero and stale contents from an earlier call are never read.
  a.workspace = scratch;
  a.workspace_bytes = fa::kNoAllocScratchBytes;
  return fa_decode_paged_ex(&a, stream);
}

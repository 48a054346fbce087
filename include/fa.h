/*
 * fa.h -- C ABI of the GB300 (sm_103a) fused softmax-attention forward library (libfa.so).
 *
 * The operation everywhere is softmax attention computed exactly, blockwise, with an online
 * softmax (FlashAttention; llama.cpp PR "CUDA: fix FA occupancy, optimize tile kernel",
 * opening paragraphs; flashinfer PR "perf: FlashAttention-3 style MLA PageAttention",
 * change list):
 *
 *     s_j = scale * <q, k_j> + mask_j,   out = sum_j softmax(s)_j v_j,   lse = ln sum_j e^{s_j}
 *
 * Conventions (the pages leave them open; these are the readings this library takes):
 *   - every pointer argument is a DEVICE pointer unless stated otherwise, to a contiguous,
 *     row-major array whose last dimension is innermost, aligned to 16 bytes;
 *   - grouped-query attention: query head h reads kv head h / (Hq / Hkv);
 *   - causal masking is bottom-right aligned: query i (of Lq) sits at absolute position
 *     Lkv - Lq + i and sees keys j <= Lkv - Lq + i;
 *   - lse is the natural log-sum-exp of the scaled, masked scores, stored as fp32;
 *   - a row that sees no key (fully masked, or seq_len 0) gets out = 0 and lse = -inf;
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous: they enqueue kernels and return without synchronising;
 *   - the library never allocates device memory during a call.  Split-KV scratch is a
 *     caller-provided workspace sized by the matching *_workspace_size function;
 *   - argument errors are detected on the host before anything is enqueued: the call
 *     returns a nonzero fa_status and fa_last_error() describes it.  Errors found on the
 *     device (a page id out of range, a wait that ran out) are recorded in a sticky status
 *     word read by fa_get_device_status(); the kernel skips the offending access;
 *   - the library keeps per-device facts for the life of the process (the SM count, kernel
 *     attributes, the device addresses of its status word and scratch array), so a
 *     cudaDeviceReset inside the process is not supported.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, inconsistent sizes */
  FA_ERR_UNSUPPORTED = 2, /* valid but not implemented (head dim, group size, dtype) */
  FA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than *_workspace_size */
  FA_ERR_CUDA = 4,        /* a CUDA runtime call failed (no device, launch failure) */
  FA_ERR_TIMEOUT = 5,     /* device: a bounded wait inside a kernel ran out */
  FA_ERR_BOUNDS = 6       /* device: a page id or sequence length was out of range */
} fa_status;

typedef enum fa_dtype { FA_BF16 = 0, FA_FP16 = 1, FA_FP32 = 2 } fa_dtype;

/*
 * Dense attention (prefill of a query chunk against a KV cache), bf16.
 * Defined by the formula above over all keys of the batch entry; the query chunk attends
 * to a cache of Lkv keys (the pp16384 workloads of the llama.cpp PR above process query
 * micro-batches against a 16K-token context).
 *   q   [B, Hq,  Lq,  D] bf16        k, v [B, Hkv, Lkv, D] bf16
 *   out [B, Hq,  Lq,  D] bf16        lse  [B, Hq, Lq] fp32, or NULL
 *   Hq % Hkv == 0, Hq / Hkv <= 128, D in {64, 128, 256}; Lq, Lkv >= 0; causal 0/1.
 * No workspace: the KV loop is not split across CTAs (use fa_prefill_ex for that).
 * Returns FA_OK or an fa_status code.
 */
int fa_prefill(const void* q, const void* k, const void* v, void* out, float* lse, int B,
               int Hq, int Hkv, int Lq, int Lkv, int D, int causal, float scale, void* stream);

/* Extended prefill arguments (zero-initialise, then set the fields you need). */
typedef struct fa_prefill_args {
  const void* q;         /* [B, Hq, Lq, D] in dtype */
  const void* k;         /* [B, Hkv, Lkv, D] in dtype */
  const void* v;         /* [B, Hkv, Lkv, D] in dtype */
  void* out;             /* [B, Hq, Lq, D] in dtype */
  float* lse;            /* [B, Hq, Lq] fp32, or NULL */
  int B, Hq, Hkv, Lq, Lkv, D;
  int causal;
  float scale;
  fa_dtype dtype;        /* FA_BF16, FA_FP16 (tensor cores, fp32 accumulation), or FA_FP32:
                            fp32 inputs are computed in fp32 on the CUDA cores, keeping fp32
                            range and precision (no split, no workspace; for small problems) */
  const void* mask;      /* optional additive mask [mask_batches, Lq, Lkv]; -inf removes a
                            key; shared by all heads; NULL = none */
  fa_dtype mask_dtype;   /* FA_FP32 or FA_BF16 */
  int mask_batches;      /* 1 (broadcast over the batch) or B */
  int num_splits;        /* 0: the library picks; >= 1: split the KV loop this many ways
                            (16-bit inputs; fp32 inputs are never split) */
  void* workspace;       /* device scratch, >= fa_prefill_workspace_size(args) bytes */
  size_t workspace_bytes;
  /* Paged K/V (page_size = 0: dense k and v as above).  With page_size > 0, k and v are
     pages [num_pages, Hkv, page_size, D]; key t of sequence b is slot t % page_size of page
     page_table[b, t / page_size]; sequence b holds seq_lens[b] keys (device memory) and its
     Lq queries are its last Lq positions.  Lkv is then the largest seq_lens[b]: it sizes the
     KV split and is the last dimension of the mask.  dtype FA_BF16 or FA_FP16; page_size a
     power of two in [8, 128] (at most 64 when D = 256); Lkv <= max_pages * page_size;
     num_pages * Hkv < 2^31 (FA_ERR_UNSUPPORTED otherwise). */
  const int32_t* page_table; /* [B, max_pages] int32 */
  const int32_t* seq_lens;   /* [B] int32 */
  int page_size, max_pages, num_pages;
} fa_prefill_args;

int fa_prefill_ex(const fa_prefill_args* args, void* stream);

/* Workspace bytes fa_prefill_ex needs for these arguments on the current device (0 when
 * the plan needs none).  Depends only on sizes, dtype and num_splits; the pointer fields
 * are not read. */
size_t fa_prefill_workspace_size(const fa_prefill_args* args);

/* The split count fa_prefill_ex will use for these arguments on the current device. */
int fa_prefill_num_splits(const fa_prefill_args* args);

/*
 * Split-KV paged grouped-query decode: one query token per sequence attends to the
 * seq_lens[b] tokens of its paged cache (flashinfer PR above, results section: paged KV
 * cache with a page_size; page_table + seq_lens addressing).
 *   q        [B, Hq, D] bf16
 *   k_pages, v_pages [num_pages, Hkv, page_size, D] bf16 (each page holds page_size
 *            consecutive tokens of every kv head)
 *   page_table [B, max_pages_per_seq] int32: key t of sequence b is slot t % page_size of
 *            page page_table[b, t / page_size]; entries past the sequence are not read
 *   seq_lens [B] int32 (device), each in [0, max_seq_len]
 *   out [B, Hq, D] bf16;  lse [B, Hq] fp32 or NULL
 *   D in {64, 128, 256}; Hq / Hkv <= 128; page_size a power of two; max_seq_len <=
 *   max_pages*page_size is a host-side bound used to size the grid (no device-to-host read).
 *   workspace >= fa_decode_workspace_size(B, Hq, D, max_seq_len) bytes (an upper bound over
 *   both kernels below; fa_decode_get_plan gives the exact figure), 256-byte aligned.
 * Two kernels serve it (fa_decode_get_plan says which one a call takes):
 *   - CUDA cores: fixed chunks of fa_decode_chunk_tokens() tokens per CTA, each writing a
 *     partial state, then the merge (fa_merge_states).  Power-of-two groups G = Hq / Hkv of
 *     at most 16 with G * D <= 1024, any power-of-two page size;
 *   - tensor cores: the paged attention kernel of fa_prefill_paged with one query per
 *     sequence (the G heads of a kv head in one 128-row tile, tcgen05 MMAs), its KV loop split
 *     and merged only when the (sequence, kv head) units cover less than half the SMs.  Any
 *     G <= 128; page sizes that are powers of two from 8 to 128 (64 when D = 256).
 *   The automatic choice takes the tensor cores when the units fill the GPU unsplit or when
 *   the CUDA-core kernel cannot take G, the CUDA cores otherwise.
 */
int fa_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                    const int32_t* page_table, const int32_t* seq_lens, void* out, float* lse,
                    int B, int Hq, int Hkv, int D, int page_size, int max_pages_per_seq,
                    int num_pages, int max_seq_len, float scale, void* workspace,
                    size_t workspace_bytes, void* stream);

size_t fa_decode_workspace_size(int B, int Hq, int D, int max_seq_len);

typedef enum fa_decode_path {
  FA_DECODE_AUTO = 0,         /* the library chooses (see fa_decode_paged) */
  FA_DECODE_CUDA_CORES = 1,   /* chunked split-KV kernel on the CUDA cores, then the merge */
  FA_DECODE_TENSOR_CORES = 2  /* paged attention kernel on the tensor cores */
} fa_decode_path;

/* fa_decode_paged with the element type as an argument: the same fields, plus dtype
 * FA_BF16 or FA_FP16 for q, the pages and out (the split states and lse stay fp32), and the
 * kernel to use (FA_DECODE_AUTO unless a test or benchmark wants one of them). */
typedef struct fa_decode_args {
  const void* q;
  const void* k_pages;
  const void* v_pages;
  const int32_t* page_table;
  const int32_t* seq_lens;
  void* out;
  float* lse;
  int B, Hq, Hkv, D, page_size, max_pages_per_seq, num_pages, max_seq_len;
  float scale;
  fa_dtype dtype;
  void* workspace;
  size_t workspace_bytes;
  fa_decode_path path;
} fa_decode_args;

int fa_decode_paged_ex(const fa_decode_args* args, void* stream);

/* What a decode call with these arguments does on the current device: the kernel it runs
 * (never FA_DECODE_AUTO), the KV splits per (sequence, kv head), the kernels it enqueues
 * (a merge follows split work) and the workspace bytes it needs.  Only sizes, dtype and path
 * are read.  Returns FA_OK, or the error the call itself would return for these sizes. */
typedef struct fa_decode_plan {
  fa_decode_path path;
  int n_splits;
  int launches;
  size_t workspace_bytes;
} fa_decode_plan;

int fa_decode_get_plan(const fa_decode_args* args, fa_decode_plan* plan);

/*
 * fa_decode_paged for callers that cannot allocate device memory (the pages describe no
 * such entry point; it has no counterpart there).  Same arguments and results as
 * fa_decode_paged minus the workspace: the split-KV scratch comes from a fixed 32 MiB
 * device array inside the library, which every GPU that loads the library keeps reserved
 * until the process exits.  Use it where allocating is not possible, e.g. a runtime whose
 * arena allocator owns all device memory, or a serving loop that must not allocate.
 *   - The arguments are checked as fa_decode_paged checks them.  A problem whose scratch
 *     (fa_decode_get_plan's workspace_bytes for these sizes, automatic path) exceeds 32 MiB
 *     is then rejected with FA_ERR_WORKSPACE before anything is enqueued.
 *   - The first call on each device looks up the array's device address (a
 *     cudaGetSymbolAddress call) and keeps it for the life of the process; make that first
 *     call before any stream capture, and do not use this entry point across a
 *     cudaDeviceReset (the kept address may then no longer be the array's).
 *   - Calls make no allocation of any kind.
 *   - Every call uses the same array: two calls whose kernels overlap on the GPU (different
 *     streams, or different threads without ordering) race on it and give wrong results.
 *     Calls ordered on one stream are safe; the array needs no clearing between calls.
 */
int fa_decode_paged_noalloc(const void* q, const void* k_pages, const void* v_pages,
                            const int32_t* page_table, const int32_t* seq_lens, void* out,
                            float* lse, int B, int Hq, int Hkv, int D, int page_size,
                            int max_pages_per_seq, int num_pages, int max_seq_len, float scale,
                            void* stream);

/* Tokens per split-KV chunk of the CUDA-core decode kernel for these sizes on the current
 * device (a multiple of 64; depends only on B, Hq, max_seq_len and the SM count). */
int fa_decode_chunk_tokens(int B, int Hq, int max_seq_len);

/*
 * The CUDA-core decode kernel without the final merge: writes the split-KV state of every query row
 * r = b*Hq + h and chunk c (tokens [c*chunk, (c+1)*chunk) of the sequence, chunk =
 * fa_decode_chunk_tokens(B, Hq, max_seq_len)): the normalised partial output
 * o_parts[r, c, :] (fp32) and its log-sum-exp lse_parts[r, c] (natural log).  Chunks at or
 * past seq_lens[b] are not written.  fa_merge_states with n_splits[r] =
 * ceil(seq_lens[b] / chunk) combines them; these states are also what a merge across
 * devices holding different key ranges would exchange.
 *   o_parts [B*Hq, n_chunks, D] fp32, lse_parts [B*Hq, n_chunks] fp32 with
 *   n_chunks = ceil(max_seq_len / chunk), passed for checking.
 */
int fa_decode_paged_states(const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* page_table, const int32_t* seq_lens, float* o_parts,
                           float* lse_parts, int n_chunks, int B, int Hq, int Hkv, int D,
                           int page_size, int max_pages_per_seq, int num_pages, int max_seq_len,
                           float scale, void* stream);

/*
 * MLA paged decode in the latent (absorbed) form: the compressed ckv matrix serves as both
 * K and V and a separate rope part kpe adds q_pe . kpe_t to each score (flashinfer PR
 * above, change list item 4; results section: 64 heads, page_size 1):
 *   s_t = scale * (q_nope . ckv_t + q_pe . kpe_t),   out = softmax(s) . ckv
 *   q_nope [B, H, Dc] bf16, q_pe [B, H, Dr] bf16
 *   ckv_pages [num_pages, page_size, Dc] bf16, kpe_pages [num_pages, page_size, Dr] bf16
 *   page_table [B, max_pages_per_seq] int32, seq_lens [B] int32
 *   out [B, H, Dc] bf16 (latent space), lse [B, H] fp32 or NULL
 *   Dc == 512, Dr == 64, 1 <= H <= 1024: each CTA takes one group of up to 64 heads (one
 *   tensor-core tile of heads), so 128 heads read a sequence's cache twice (the second read
 *   mostly from L2) and fewer than 64 heads leave part of the tile idle.  Any page_size >= 1;
 *   pages of a multiple of 64 tokens are copied a 64-token tile at a time with TMA.
 *   workspace >= mla_decode_workspace_size(B, H, Dc, max_seq_len) bytes.
 */
int mla_decode_paged(const void* q_nope, const void* q_pe, const void* ckv_pages,
                     const void* kpe_pages, const int32_t* page_table, const int32_t* seq_lens,
                     void* out, float* lse, int B, int H, int Dc, int Dr, int page_size,
                     int max_pages_per_seq, int num_pages, int max_seq_len, float scale,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes mla_decode_paged needs on the current device: partial states for the
 * sequences it cuts into chunks.  0 when every sequence is one chunk written directly; when
 * there are more sequences than SMs and the last wave of CTAs would be at most half full,
 * only that wave's sequences are cut (and merged), the others written directly. */
size_t mla_decode_workspace_size(int B, int H, int Dc, int max_seq_len);

/* mla_decode_paged with the element type as an argument: the same fields, plus dtype
 * FA_BF16 or FA_FP16 for q_nope, q_pe, the pages and out. */
typedef struct mla_decode_args {
  const void* q_nope;
  const void* q_pe;
  const void* ckv_pages;
  const void* kpe_pages;
  const int32_t* page_table;
  const int32_t* seq_lens;
  void* out;
  float* lse;
  int B, H, Dc, Dr, page_size, max_pages_per_seq, num_pages, max_seq_len;
  float scale;
  fa_dtype dtype;
  void* workspace;
  size_t workspace_bytes;
} mla_decode_args;

int mla_decode_paged_ex(const mla_decode_args* args, void* stream);

/* Tokens per split-KV chunk of mla_decode_paged_states (a multiple of the kernel's tile);
 * mla_decode_paged uses it too, except for the sequences of a split last wave. */
int mla_decode_chunk_tokens(int B, int H, int max_seq_len);

/* mla_decode_paged without the final merge (same contract as fa_decode_paged_states):
 *   o_parts [B*H, n_chunks, Dc] fp32, lse_parts [B*H, n_chunks] fp32,
 *   n_chunks = ceil(max_seq_len / mla_decode_chunk_tokens(B, H, max_seq_len)). */
int mla_decode_paged_states(const void* q_nope, const void* q_pe, const void* ckv_pages,
                            const void* kpe_pages, const int32_t* page_table,
                            const int32_t* seq_lens, float* o_parts, float* lse_parts,
                            int n_chunks, int B, int H, int Dc, int Dr, int page_size,
                            int max_pages_per_seq, int num_pages, int max_seq_len, float scale,
                            void* stream);

/*
 * Paged prefill (chunked prefill against a paged KV cache), bf16 short form of
 * fa_prefill_ex with page_size > 0: each sequence's keys and values are read through a page
 * table, in the layout of the paged decode path.  Sequence b has kv_len_b = seq_lens[b]
 * cached tokens, the query chunk included; its Lq queries are its last Lq positions, so
 * with causal = 1 query i sees keys j <= kv_len_b - Lq + i (a query with no key gets
 * out = 0 and lse = -inf).
 *   q        [B, Hq, Lq, D] bf16              out [B, Hq, Lq, D] bf16, lse [B, Hq, Lq] fp32 or NULL
 *   k_pages, v_pages [num_pages, Hkv, page_size, D] bf16
 *   page_table [B, max_pages] int32, seq_lens [B] int32 (device memory)
 *   page_size a power of two in [8, 128] (at most 64 when D = 256); Hq % Hkv == 0,
 *   Hq / Hkv <= 128, D in {64, 128, 256}; max_seq_len >= every seq_lens[b] (it sizes the
 *   KV split) and <= max_pages * page_size.
 *   workspace: fa_prefill_paged_workspace_size(B, Hq, Hkv, Lq, D, max_seq_len) bytes,
 *   256-byte aligned (none when that size is 0).
 * A sequence length outside [0, max_pages * page_size] or a page id of a key inside the
 * sequence outside [0, num_pages) sets FA_ERR_BOUNDS in the device status word; the kernel
 * then reads page 0 instead.  Returns FA_OK or an fa_status code.
 */
int fa_prefill_paged(const void* q, const void* k_pages, const void* v_pages,
                     const int32_t* page_table, const int32_t* seq_lens, void* out, float* lse,
                     int B, int Hq, int Hkv, int Lq, int D, int page_size, int max_pages,
                     int num_pages, int max_seq_len, int causal, float scale, void* workspace,
                     size_t workspace_bytes, void* stream);
size_t fa_prefill_paged_workspace_size(int B, int Hq, int Hkv, int Lq, int D, int max_seq_len);

/*
 * Gated-delta linear attention, chunked prefill: the gated-delta chunked linear-attention
 * prefill of hip-ep PR "perf(kernels): speed up linear-attention prefill ~2.6x" (Summary;
 * checked there against a per-token oracle).  The page does not write the recurrence; the
 * one computed is the gated delta rule (Gated Delta Networks, 2024), per value head h with a
 * state S of dv rows by dk columns:
 *     S_t = S_{t-1} alpha_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   alpha_t = e^{g_t}
 *     o_t = S_t (scale q_t)
 * Value head h reads query/key head h / (Hv / Hk).  S starts from initial_state (or zero);
 * the state after the last token is written to final_state when given.  L2 normalisation of
 * q and k, which models apply before the recurrence, is the caller's.
 *   q, k [B, Hk, T, dk] bf16;  v [B, Hv, T, dv] bf16;  g, beta [B, Hv, T] fp32
 *   initial_state, final_state [B, Hv, dv, dk] fp32 or NULL;  out [B, Hv, T, dv] bf16
 *   dk == dv == 128; Hv % Hk == 0; B * Hv * (T + 64) < 2^31.
 *   workspace >= gated_delta_workspace_size(args) bytes, 256-byte aligned (chunk operands:
 *   about 0.9 KB per token and value head).
 * The prefill runs in 64-token chunks: a kernel prepares every chunk of every head in
 * parallel, then one CTA per (batch, value head) carries the state through its chunks on the
 * tensor cores (bf16 operands, fp32 accumulation and state).
 */
typedef struct gated_delta_args {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* initial_state;
  void* out;
  float* final_state;
  int B, T, Hk, Hv, dk, dv;
  float scale;           /* applied to q; 1/sqrt(dk) is the usual value */
  fa_dtype dtype;        /* FA_BF16 */
  void* workspace;
  size_t workspace_bytes;
} gated_delta_args;

int gated_delta_prefill(const gated_delta_args* args, void* stream);

/* Workspace bytes gated_delta_prefill needs for these sizes (pointers are not read). */
size_t gated_delta_workspace_size(const gated_delta_args* args);

/*
 * Merge of attention states over disjoint key sets (the split-KV combine):
 *   lse = ln sum_s e^{lse_s},   out = sum_s e^{lse_s - lse} o_s
 *   o_parts [rows, max_splits, D] fp32 (normalised partial outputs), lse_parts
 *   [rows, max_splits] fp32 (natural log; -inf = empty part); n_splits [rows] int32 or NULL
 *   (= max_splits for every row); out [rows, D] in out_dtype; lse [rows] fp32 or NULL.
 *   D a multiple of 4, at most 512.
 */
int fa_merge_states(const float* o_parts, const float* lse_parts, const int32_t* n_splits,
                    void* out, float* lse, int rows, int D, int max_splits, fa_dtype out_dtype,
                    void* stream);

/* Synchronises `stream`, returns the sticky device status of the current device (FA_OK,
 * FA_ERR_TIMEOUT or FA_ERR_BOUNDS; FA_ERR_CUDA if the synchronisation itself failed) and
 * clears it. */
int fa_get_device_status(void* stream);

/* Self-test of the device failure path shared by every kernel above: launches one CTA that
 * waits, with a limit of timeout_us microseconds (1 .. 2000000, the kernels' own limit being
 * 2 s), on a barrier that nothing arrives on.  The wait runs out, the kernel records
 * FA_ERR_TIMEOUT in the sticky status word and ends, so a following fa_get_device_status()
 * returns FA_ERR_TIMEOUT and the device stays usable.  Returns FA_OK once enqueued,
 * FA_ERR_INVALID_ARG for a timeout outside the range. */
int fa_selftest_wait_timeout(unsigned timeout_us, void* stream);

/* Message for the last error returned on the calling thread ("" if none). */
const char* fa_last_error(void);

/* ABI version: major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */

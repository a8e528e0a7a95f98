/*
 * paged_attn.h -- C ABI of the GB300 (sm_103a) paged grouped-query attention library.
 *
 * Two calls, one per phase, over one paged KV cache:
 *   paged_attn_decode   split-K flash-decoding of one query token per sequence
 *   paged_attn_prefill  causal (or full) attention of the new tokens of each sequence
 *
 * The operation (defined by the pages this library follows; each source is a page title
 * and the section on it):
 *  - "[None][feat] Run Gemma4 head_dim 512 attention on Triton" (TensorRT-LLM PR #17772),
 *    Approach: both phases read the combined HND cache
 *    [num_pages, 2, num_kv_heads, page_size, head_dim] through kv_indptr / kv_indices /
 *    kv_last_page_len (the same slicing as the FlashInfer decode plan); prefill is causal
 *    when no custom mask is given; FP8 KV is dequantised in the kernel ("cast on load").
 *    Test Coverage: head_dim up to 512, GQA ratios with non-power-of-two groups (12/4,
 *    24/4) padded inside the kernel, page sizes 1..64 with partial and exact last pages,
 *    split-K, sliding windows.  Not covered: unsupported inputs fail loudly instead of
 *    returning wrong results.
 *  - "feat(attention): asymmetric VO-split NVFP4 paged prefill (qk=512/vo=256) for
 *    Gemma-4 on SM120/121" (FlashInfer PR #3684), Summary: head_dim_qk = 512 with
 *    head_dim_vo = 256, independent K/V strides, NVFP4 KV with explicit scale strides in a
 *    contiguous [all-data | all-SF] layout; NVFP4 split-KV correctness: packed e2m1 with
 *    one FP8 scale per 16 consecutive head-dim elements of one token.
 *
 * Per sequence b and query head h (kv head h / (Hq/Hkv)), a query at position
 * pos = kv_len - qo_len + i (decode: pos = kv_len - 1) sees key j < kv_len when
 * (causal ? j <= pos : 1) and (window_left >= 0 ? j >= pos - window_left : 1):
 *   out = softmax_j(sm_scale * q . K[j]) V[j],   lse = m + ln(sum_j exp(s_j - m))
 * (natural log of the scaled scores).  A row with no visible key gets out = 0,
 * lse = -inf.
 *
 * ---------------------------------------------------------------------------------
 * Memory layout (all device memory, caller-owned; the library keeps no pointer after a
 * call returns):
 *  q          bf16, [batch, Hq, head_dim_qk] (decode) or [total_q, Hq, head_dim_qk]
 *             (prefill), rows contiguous.  16-byte aligned.
 *  kv_cache   page p (0 <= p < num_pages) is one contiguous block: the K block
 *             [Hkv][page_size][head_dim_qk] followed by the V block
 *             [Hkv][page_size][head_dim_vo], elements of kv_dtype.  With
 *             head_dim_qk == head_dim_vo this is exactly
 *             [num_pages, 2, Hkv, page_size, head_dim].  NVFP4 elements are packed two
 *             per byte, element 2i in the low nibble of byte i.  16-byte aligned.
 *  kv_indptr  int32 [batch+1]; sequence b owns logical pages
 *             kv_indices[kv_indptr[b] .. kv_indptr[b+1]).
 *  kv_indices int32 physical page ids, each in [0, num_pages).
 *  kv_last_page_len int32 [batch], in [1, page_size] for a sequence with pages;
 *             kv_len = (npages - 1) * page_size + kv_last_page_len.
 *  qo_indptr  int32 [batch+1] (prefill): the new tokens of sequence b are q rows
 *             qo_indptr[b] .. qo_indptr[b+1]; they are the last qo_len of its kv_len
 *             tokens (the cache already holds them).  Requires kv_len >= qo_len.
 *  out        bf16, [rows, Hq, head_dim_vo]; lse fp32 [rows, Hq] or NULL.
 *  scales     see pa_kv_scales.
 * Values inside the device arrays (page ids, lengths) are the caller's contract; they
 * are not read on the host (no host-device synchronisation happens in a call).
 *
 * Streams and workspace: work is enqueued on `stream` (a cudaStream_t, NULL = legacy
 * default stream) and the call returns without waiting.  The library owns a grow-only
 * device workspace per stream (work lists, split-K partials, the prefill's copy of FP8 /
 * NVFP4 pages, an error word); it grows with cudaMalloc (and the cudaFree of the smaller
 * one, which waits for the device) only when a call needs more than it has, so once
 * warmed up a call allocates nothing.  Calls on different streams use different
 * workspaces and may overlap on the GPU; calls on one stream are ordered by it.  A call
 * captured into a CUDA graph allocates nothing: it uses the capturing stream's workspace
 * if that is large enough, else the legacy default stream's, else it fails with
 * PA_ERR_CUDA; so make an eager call of the same shape on one of those streams before
 * capturing.  The graph keeps that workspace's address, and replays share it with the
 * eager calls on its stream.
 *
 * Errors: every entry point returns 0 (PA_OK) or a negative pa_status, and launches
 * nothing when it rejects its arguments.
 */
#ifndef PAGED_ATTN_H_
#define PAGED_ATTN_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = -1, /* a null required pointer, a bad size, Hq % Hkv != 0, ... */
  PA_ERR_UNSUPPORTED = -2, /* valid but not built (see the lists on each call) */
  PA_ERR_ALIGNMENT = -3,   /* a pointer that is not 16-byte aligned */
  PA_ERR_SMEM = -4,        /* the kernel's shared memory exceeds the device opt-in limit */
  PA_ERR_CUDA = -5,        /* a CUDA runtime / driver call failed */
  PA_ERR_DEVICE = -6,      /* a kernel gave up on a bounded wait (see the error query) */
  PA_ERR_SCRATCH = -7      /* the problem needs more scratch than paged_attn_decode_noalloc holds */
} pa_status;

typedef enum { PA_KV_BF16 = 0, PA_KV_FP8_E4M3 = 1, PA_KV_NVFP4 = 2 } pa_kv_dtype;

/* Dequantisation scales of the KV cache (all device pointers).
 *  PA_KV_BF16:      all fields ignored (may be NULL).
 *  PA_KV_FP8_E4M3:  k_scale, v_scale: one fp32 each, K^ = e4m3(code) * k_scale,
 *                   V^ = e4m3(code) * v_scale (e4m3 "fn": bias 7, max 448, no inf).
 *  PA_KV_NVFP4:     k_scale, v_scale: one fp32 global scale each; sf: the block-scale
 *                   pool, page p holding [Hkv][page_size][head_dim_qk/16] K scales
 *                   then [Hkv][page_size][head_dim_vo/16] V scales (e4m3 bytes), i.e.
 *                   the contiguous [all-data | all-SF] arrangement;
 *                   K^ = e2m1(nibble) * e4m3(sf) * k_scale (likewise V).
 *                   16-byte aligned. */
typedef struct {
  const float* k_scale;
  const float* v_scale;
  const uint8_t* sf;
} pa_kv_scales;

/*
 * paged_attn_decode -- one query token per sequence, split-K over the KV length.
 *
 * q [batch, num_qo_heads, head_dim_qk] bf16; out [batch, num_qo_heads, head_dim_vo]
 * bf16; lse [batch, num_qo_heads] fp32 or NULL.  Every query head of one kv head is
 * served by the same CTA (groups up to 16, padded inside the kernel).  The KV length of
 * each sequence is cut into page-aligned chunks on the device; chunks of one sequence
 * write partial (O, m, l) to the workspace that a merge kernel combines by their lse
 * weights.
 *
 * Supported: (head_dim_qk, head_dim_vo) in {(512,512), (512,256), (256,256)};
 * num_qo_heads / num_kv_heads in [1, 16]; page_size in {1,2,4,8,16,32,64};
 * kv_dtype any pa_kv_dtype.  window_left = -1 disables the sliding window.
 * Returns PA_OK, or PA_ERR_INVALID_ARG (a null required pointer, batch < 0,
 * num_pages < 1, num_qo_heads not a multiple of num_kv_heads, a non-finite sm_scale,
 * window_left < -1, an unknown kv_dtype, missing scales), PA_ERR_UNSUPPORTED (a group
 * num_qo_heads / num_kv_heads above 16, another head-dim pair, another page size),
 * PA_ERR_ALIGNMENT, PA_ERR_SMEM or PA_ERR_CUDA; nothing is launched on error.
 */
int paged_attn_decode(const void* q, const void* kv_cache, const int32_t* kv_indptr,
                      const int32_t* kv_indices, const int32_t* kv_last_page_len, int batch,
                      int num_pages, int num_qo_heads, int num_kv_heads, int head_dim_qk,
                      int head_dim_vo, int page_size, float sm_scale, int window_left,
                      int kv_dtype, const pa_kv_scales* kv_scales, void* out, float* lse,
                      void* stream);

/*
 * paged_attn_prefill -- attention of the new tokens (q rows qo_indptr[b]..[b+1]) of each
 * sequence over its paged KV, causal when `causal` != 0 (bottom-right aligned: the new
 * tokens are the last qo_len of kv_len).
 *
 * q [total_q, num_qo_heads, head_dim_qk] bf16; out [total_q, num_qo_heads, head_dim_vo]
 * bf16; lse [total_q, num_qo_heads] fp32 or NULL.  QK^T and PV run as tcgen05 MMAs with
 * TMEM accumulators; for head_dim_vo = 512 the VO dimension is processed in two halves
 * (the second reuses the first's softmax probabilities from a workspace scratch).
 * Shapes and dtypes as for decode; group size up to 16.  FP8 / NVFP4 KV: the pages
 * kv_indices references are first converted to a bf16 copy in the library workspace
 * (num_pages * num_kv_heads * page_size * (head_dim_qk + head_dim_vo) * 2 bytes) when
 * that fits the limit set by paged_attn_set_prefill_dequant_limit (default 4 GiB), else
 * converted inside the kernel on every read; both give the same values (the conversions
 * are exact).  Page sizes 1, 2 and 4 (any dtype): the pages are read from a bf16 copy
 * that pads each page to 8 rows per kv head (num_pages * num_kv_heads * 8 *
 * (head_dim_qk + head_dim_vo) * 2 bytes), under the same limit; beyond it the call
 * returns PA_ERR_UNSUPPORTED.  When the
 * (query tile, kv head) items are fewer than the SMs (a few new tokens over a long
 * prefix), the device planner may split long KV ranges into chunks whose fp32 partials a
 * merge kernel combines (paged_attn_set_prefill_split_kv); the workspace then also holds
 * 3 x SMs partial slots of 128 x head_dim_vo floats.  Everything runs on `stream` with no
 * host synchronisation.
 * Returns as paged_attn_decode.
 */
int paged_attn_prefill(const void* q, const int32_t* qo_indptr, int total_q,
                       const void* kv_cache, const int32_t* kv_indptr,
                       const int32_t* kv_indices, const int32_t* kv_last_page_len, int batch,
                       int num_pages, int num_qo_heads, int num_kv_heads, int head_dim_qk,
                       int head_dim_vo, int page_size, float sm_scale, int window_left,
                       int causal, int kv_dtype, const pa_kv_scales* kv_scales, void* out,
                       float* lse, void* stream);

/*
 * paged_attn_prefill_custom_mask -- paged_attn_prefill with a custom mask ("[None][feat]
 * Run Gemma4 head_dim 512 attention on Triton", Approach: prefill is causal when no custom
 * mask is given; the multimodal Gemma layers attend bidirectionally inside spans of the
 * new tokens).  New token i (0 <= i < qo_len) of sequence b may attend key j
 * (0 <= j < kv_len) only when bit mask_indptr[b] * 8 + i * kv_len + j of custom_mask is 1
 * (bit k of a byte is its 2^k bit): each sequence's qo_len x kv_len row-major bit grid
 * starts at byte offset mask_indptr[b] (int64, device, [batch] or more entries).  The mask
 * narrows the causal and window rules (pass causal = 0 for a mask that replaces the causal
 * rule); a row with no allowed key gives out = 0 and lse = -inf.  custom_mask is read only
 * where bits of allowed-by-causal/window keys lie; mask_indptr must be 8-byte aligned.
 * Everything else as paged_attn_prefill.
 */
int paged_attn_prefill_custom_mask(const void* q, const int32_t* qo_indptr, int total_q,
                                   const void* kv_cache, const int32_t* kv_indptr,
                                   const int32_t* kv_indices, const int32_t* kv_last_page_len,
                                   int batch, int num_pages, int num_qo_heads, int num_kv_heads,
                                   int head_dim_qk, int head_dim_vo, int page_size,
                                   float sm_scale, int window_left, int causal, int kv_dtype,
                                   const pa_kv_scales* kv_scales, void* out, float* lse,
                                   const uint8_t* custom_mask, const int64_t* mask_indptr,
                                   void* stream);

/*
 * paged_attn_append_kv -- write the K and V of new tokens (bf16) into the paged cache,
 * converted to the cache's element type (quantise-on-write): the step that produces the
 * FP8 / NVFP4 caches the attention calls read ("feat(attention): asymmetric VO-split NVFP4
 * paged prefill (qk=512/vo=256) for Gemma-4 on SM120/121", validation on caches written by
 * an in-tree NVFP4 KV quantisation kernel from bf16 sources).
 *
 * k_new [total_new, num_kv_heads, head_dim_qk] and v_new [total_new, num_kv_heads,
 * head_dim_vo] bf16, rows append_indptr[b]..append_indptr[b+1] belonging to sequence b
 * (append_indptr int32 [batch + 1], append_indptr[batch] = total_new).  The page table
 * (kv_indptr, kv_indices, kv_last_page_len) describes each sequence after the append: its
 * last n_b = append_indptr[b+1] - append_indptr[b] tokens are the new ones, so new row j
 * of sequence b goes to position t = kv_len_b - n_b + j, page kv_indices[kv_indptr[b] +
 * t / page_size], slot t % page_size, in the cache layout paged_attn_decode reads.
 * Nothing else in the cache or the scale pool is written.
 *
 * Conversion of a bf16 value x (as fp32), with correctly rounded fp32 operations in
 * this order; a code carries the sign of its operand, also when it rounds to zero:
 *   PA_KV_BF16      x copied;
 *   PA_KV_FP8_E4M3  e4m3 code of x / s, round to nearest even, saturating at +-448;
 *                   s = *k_scale for K, *v_scale for V (per-tensor fp32, on the device);
 *   PA_KV_NVFP4     per block of 16 consecutive head-dim elements of one token and head,
 *                   with the global scale G = *k_scale or *v_scale: amax = max |x|,
 *                   sf = e4m3 code of (amax / 6) / G (nearest even, saturating), d =
 *                   value(sf) * G; codes = e2m1 of x / d (nearest even, saturating at +-6),
 *                   or 0 when d = 0; sf goes to the block-scale pool `sf` (layout as in
 *                   pa_kv_scales.sf), the codes two per byte, element 2i in the low nibble.
 * k_scale / v_scale (device fp32 scalars) are required for FP8 and NVFP4 and ignored for
 * bf16; sf is required for NVFP4 and ignored otherwise.  The caller owns every buffer.
 * k_new, v_new and kv_cache must be 16-byte aligned.  A new row whose position falls
 * outside its sequence (n_b > kv_len_b) or whose page id is outside [0, num_pages) is
 * skipped and sets the device error word (paged_attn_check_device_error).
 * Returns PA_OK, or PA_ERR_INVALID_ARG / PA_ERR_UNSUPPORTED / PA_ERR_ALIGNMENT /
 * PA_ERR_CUDA; nothing is launched on error.  PA_ERR_UNSUPPORTED also when one page
 * (num_kv_heads * page_size rows of K and V) takes 2^31 bytes or more.
 */
int paged_attn_append_kv(const void* k_new, const void* v_new, const int32_t* append_indptr,
                         int total_new, void* kv_cache, const int32_t* kv_indptr,
                         const int32_t* kv_indices, const int32_t* kv_last_page_len, int batch,
                         int num_pages, int num_kv_heads, int head_dim_qk, int head_dim_vo,
                         int page_size, int kv_dtype, const float* k_scale,
                         const float* v_scale, uint8_t* sf, void* stream);

/* Human-readable text of a pa_status value (static storage, never NULL). */
const char* paged_attn_status_string(int status);

/* Frees the library-owned workspaces of the current device, one per stream that has made
 * a call (blocking).  Returns PA_OK or PA_ERR_CUDA.  The next call on a stream allocates
 * that stream's again. */
int paged_attn_release_workspace(void);

/* Synchronises the current device, then reports and clears the device error words that
 * kernels set when a bounded wait gives up (each stream's workspace's and, once
 * paged_attn_decode_noalloc has run on the device, the one in its fixed array):
 * *code = 0 (none) or the wait site id (a workspace's first when several are set).
 * Returns PA_OK, PA_ERR_DEVICE when a wait gave up, PA_ERR_CUDA on a CUDA error. */
int paged_attn_check_device_error(int* code);

/* Test hook: stores `code` in a device error word of the current device (blocking):
 * target 0 = the legacy default stream's workspace's (allocating that workspace if there
 * is none), 1 = the one in
 * paged_attn_decode_noalloc's fixed array.  Lets a test check that
 * paged_attn_check_device_error reports and clears each word without making a kernel
 * wait time out.  Returns PA_OK, PA_ERR_INVALID_ARG or PA_ERR_CUDA. */
int paged_attn_debug_set_error_word(int target, int code);

/* Test hook for split-K: force every decode chunk to `pages` pages (0 = automatic).
 * The device still widens chunks when the workspace bound requires it.  Process-wide. */
int paged_attn_set_decode_chunk_pages(int pages);

/* Single-launch decode.  A decode call whose (sequence, kv head) items number at most the
 * device's SMs and whose page pool holds at most 256 KiB of K and V per kv head runs as one
 * kernel: each item covers its sequence's whole visible range and writes its rows
 * directly, without the planner and merge launches (the split-K scheme of "[None][feat]
 * Run Gemma4 head_dim 512 attention on Triton", Approach, pays off only where there is
 * KV to split).  mode -1 = that rule (the default), 0 = never, 1 = whenever the items fit
 * one round (a test hook).  A forced chunk size (paged_attn_set_decode_chunk_pages) turns
 * it off.  Process-wide.  Returns PA_OK or PA_ERR_INVALID_ARG. */
int paged_attn_set_decode_direct(int mode);

/* Largest bf16 copy (bytes) of FP8 / NVFP4 pages that paged_attn_prefill may build in its
 * workspace; 0 = always convert inside the prefill kernel, negative = the default (4 GiB).
 * Process-wide.  Returns PA_OK. */
int paged_attn_set_prefill_dequant_limit(long long bytes);

/* Prefill with bf16 KV (or the bf16 copy of FP8 / NVFP4 pages) on CTA pairs: two CTAs of
 * a cluster on neighbouring SMs compute two query tiles of the same KV head with shared
 * MMAs (M = 256), each loading half of every K/V tile.  mode 1 uses pairs whenever
 * two-CTA clusters fit on the device; 0 and -1 (the default) use one CTA per query tile,
 * which was faster on every measured workload.  Both give the same results up to
 * summation order.  Process-wide.  Returns PA_OK, or PA_ERR_INVALID_ARG for another mode. */
int paged_attn_set_prefill_cta_pairs(int mode);

/* Split KV for prefills whose (query tile, kv head) items are fewer than the SMs (short
 * queries over long KV, "extend"): the device planner then cuts long KV ranges into
 * chunks, each chunk writes an fp32 partial (normalised output, lse) to the workspace and
 * a merge kernel combines them (lse-weighted, as split-K decode).  mode -1 (default)
 * allows it, 0 never splits; results agree up to summation order.  Process-wide.
 * Returns PA_OK, or PA_ERR_INVALID_ARG for another mode. */
int paged_attn_set_prefill_split_kv(int mode);

/* Name of the kernel variant the last successful call on this host thread launched
 * (for tests that must know which path ran).  Returns PA_OK; the text is truncated to
 * len-1 characters. */
int paged_attn_last_variant(char* buf, int len);

/*
 * paged_attn_decode_noalloc -- paged_attn_decode for callers that cannot allocate device
 * memory.  (No counterpart in the pages: it is a deployment variant of the decode call.)
 *
 * Who needs it: code that runs inside a host framework that owns every byte of device
 * memory (an inference-engine plugin handed a fixed pool, a service with a hard memory
 * budget), and code that must not trigger cudaMalloc's implicit device-wide
 * synchronisation in the middle of a step.  paged_attn_decode may grow its workspace
 * with cudaMalloc; this entry point never does.  It calls no cudaMalloc, cudaFree or
 * other allocating routine.
 *
 * Its scratch (work list, split-K partials, error word) is one statically sized device
 * array of PA_NOALLOC_SCRATCH_BYTES (32 MiB) inside the library; every GPU that loads the
 * library holds that array until the process exits.  The caller still passes every input
 * and output.  A problem whose scratch does not fit returns PA_ERR_SCRATCH before
 * anything is launched; the scratch needed grows with batch * num_qo_heads *
 * head_dim_vo (the split-K partials), and the call first uses fewer KV splits when that
 * keeps it inside the array.
 *
 * The first call on a device resolves the array's device address (with that device
 * current), caches it and zeroes the array's error word (a blocking cudaMemset); make
 * that first call before any stream capture.  Every call shares the one array and it
 * keeps the last call's contents (the planner kernel of each call rewrites the work
 * list, and every partial is written before it is read), so calls that overlap on the
 * GPU -- on different streams, or from different threads -- race; serialise them.  A bounded wait that gives up is recorded
 * in the array's error word, which paged_attn_check_device_error reports and clears.
 *
 * Arguments, layouts and the supported set are those of paged_attn_decode.
 */
#define PA_NOALLOC_SCRATCH_BYTES (32u << 20)
int paged_attn_decode_noalloc(const void* q, const void* kv_cache, const int32_t* kv_indptr,
                              const int32_t* kv_indices, const int32_t* kv_last_page_len,
                              int batch, int num_pages, int num_qo_heads, int num_kv_heads,
                              int head_dim_qk, int head_dim_vo, int page_size, float sm_scale,
                              int window_left, int kv_dtype, const pa_kv_scales* kv_scales,
                              void* out, float* lse, void* stream);

/* Measurement hook.  After paged_attn_profile_begin(n), the next n calls record a pair of
 * CUDA events on their stream around their main attention kernel (decode_kernel or
 * prefill_kernel; not the planning or merge kernels).  paged_attn_profile_end waits for
 * the last recorded event, returns the number of recorded launches and their summed
 * device time in milliseconds, and stops recording.  Process-wide, not thread-safe.
 * Returns PA_OK, PA_ERR_INVALID_ARG or PA_ERR_CUDA. */
int paged_attn_profile_begin(int max_launches);
int paged_attn_profile_end(int* launches, float* total_ms);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_ATTN_H_ */

// api.cu -- the C ABI (include/paged_attn.h): argument validation, the library-owned
// workspace, TMA tensor maps over the paged cache, and the kernel launches.
//
// Every rejection happens on the host before anything is launched ("Run Gemma4 head_dim
// 512 attention on Triton", Not covered: unsupported inputs fail loudly rather than
// returning incorrect results; "feat(attention): asymmetric VO-split NVFP4 paged prefill
// (qk=512/vo=256) for Gemma-4 on SM120/121", commit "support-or-reject-explicitly" and
// the shared-memory validation guards).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <vector>

#include "launch.h"
#include "paged_attn.h"

namespace pa {
namespace {

thread_local char g_variant[64] = "none";

// measurement hook state: event pairs recorded around the main kernel of each call
struct Profile {
  std::vector<cudaEvent_t> start, stop;
  int used = 0;
  bool on = false;
};
Profile g_prof;
std::mutex g_prof_mutex;

void prof_mark(cudaStream_t s, bool begin) {
  std::lock_guard<std::mutex> lock(g_prof_mutex);
  if (!g_prof.on || g_prof.used >= (int)g_prof.start.size()) return;
  if (begin) {
    cudaEventRecord(g_prof.start[g_prof.used], s);
  } else {
    cudaEventRecord(g_prof.stop[g_prof.used], s);
    ++g_prof.used;
  }
}
int g_forced_chunk_pages = 0;
int g_decode_direct = -1;  // -1: single-launch decode where it applies, 0: never, 1: whenever every item fits one round
std::mutex g_ws_mutex;

constexpr int kMaxDevices = 64;
struct Workspace {
  void* base = nullptr;
  size_t bytes = 0;
};
// one grow-only workspace per (device, stream): calls on different streams may overlap on
// the GPU, calls on one stream are ordered by it
std::map<cudaStream_t, Workspace> g_ws[kMaxDevices];
constexpr size_t kErrOffset = 0;      // int error word
constexpr size_t kFixedBytes = 256;   // error word region
constexpr int kReuseTiles = 64;       // prefill P reuse: items of up to 64 KV tiles (8192 keys)
constexpr uint64_t kDefaultDequantLimit = 4ull << 30;  // prefill: largest bf16 copy of FP8 / NVFP4 pages
std::atomic<uint64_t> g_prefill_dequant_limit{kDefaultDequantLimit};
// prefill with bf16 KV on CTA pairs: 1 = whenever two-CTA clusters fit, 0 = never (the
// default: on the measured workloads one CTA per query tile is faster)
std::atomic<int> g_prefill_pairs{0};
// split KV for prefills that leave SMs idle: -1 = when the planner finds it useful, 0 = never
std::atomic<int> g_prefill_split{-1};
// two-CTA clusters of the pair kernel per device and shape (512x512, 512x256, 256x256);
// -1 = not asked yet
std::atomic<int> g_pair_clusters[kMaxDevices][3];
std::once_flag g_pair_clusters_init;

int pair_clusters(int dqk, int dvo) {
  std::call_once(g_pair_clusters_init, [] {
    for (auto& d : g_pair_clusters)
      for (auto& v : d) v = -1;
  });
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  const int shape = dvo == 512 ? 0 : (dqk == 512 ? 1 : 2);
  int n = g_pair_clusters[dev][shape].load();
  if (n < 0) {
    n = prefill_pair_clusters(dqk, dvo);
    g_pair_clusters[dev][shape] = n;
  }
  return n;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Make sure the workspace of `stream` on the current device holds at least `need` bytes;
// returns its base or nullptr.  Growth frees the old buffer (cudaFree waits for the
// device, so no kernel still uses it).
void* workspace(size_t need, cudaStream_t stream, int* status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *status = PA_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (stream && cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    *status = PA_ERR_CUDA;
    return nullptr;
  }
  if (cs != cudaStreamCaptureStatusNone) {
    // a call being captured into a graph may not allocate: the capturing stream's own
    // workspace if it is large enough, else the legacy default stream's (which an eager
    // warm-up call on that stream has grown), else an error
    for (cudaStream_t key : {stream, static_cast<cudaStream_t>(nullptr)}) {
      const auto it = g_ws[dev].find(key);
      if (it != g_ws[dev].end() && it->second.bytes >= need) return it->second.base;
    }
    *status = PA_ERR_CUDA;
    return nullptr;
  }
  Workspace& w = g_ws[dev][stream];
  if (w.bytes >= need) return w.base;
  if (w.base) cudaFree(w.base);
  w.base = nullptr;
  w.bytes = 0;
  size_t bytes = align_up(need + need / 4, 1 << 20);
  if (cudaMalloc(&w.base, bytes) != cudaSuccess) {
    cudaGetLastError();
    *status = PA_ERR_CUDA;
    return nullptr;
  }
  if (cudaMemset(w.base, 0, kFixedBytes) != cudaSuccess) {
    *status = PA_ERR_CUDA;
    return nullptr;
  }
  w.bytes = bytes;
  return w.base;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D byte tensor [pages][rows][row_bytes] with the given page stride; boxes of
// [1][box_rows][box_inner] bytes.
bool make_map(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t pages,
              uint64_t page_stride, uint32_t box_inner, uint32_t box_rows, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {row_bytes, rows, pages};
  cuuint64_t strides[2] = {row_bytes, page_stride};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D byte tensor [pages][segments][rows][128 B] over rows of row_bytes = segments x 128 B
// (the segment dimension steps 128 bytes inside a row); boxes of [1][segments][box_rows]
// [128 B]: every segment of box_rows consecutive rows of one page in one load.
bool make_map_rows(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t pages,
                   uint64_t page_stride, uint32_t box_rows, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const uint64_t segs = row_bytes / 128;
  cuuint64_t dims[4] = {128, rows, segs, pages};
  cuuint64_t strides[3] = {row_bytes, 128, page_stride};
  cuuint32_t box[4] = {128, box_rows, (cuuint32_t)segs, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int x2_of(int kvt) { return kvt == KV_BF16 ? 4 : (kvt == KV_FP8 ? 2 : 1); }

// Decode chunks of at least about 4 MiB of K and V per kv head (NVFP4: with its scales).
int decode_min_chunk_pages(int kvt, int dqk, int dvo, int page_size) {
  const long row = (long)(dqk + dvo) * x2_of(kvt) / 2 + (kvt == KV_NVFP4 ? (dqk + dvo) / 16 : 0);
  const long page = row * page_size;
  return (int)std::max(1l, ((4l << 20) + page - 1) / page);
}

// A decode call small enough for one launch: every (sequence, kv head) item gets its own
// CTA in a single round, and even a single sequence holding the whole pool would cost its
// CTA little (about 6 us) against the planner and merge launches it saves (at most
// 256 KiB of K and V per kv head in the pool).
bool decode_direct(int kvt, int dqk, int dvo, int page_size, long long num_pages, int batch, int hkv, int sms) {
  if (g_decode_direct == 0 || g_forced_chunk_pages > 0) return false;
  if ((long long)batch * hkv > sms) return false;
  if (g_decode_direct == 1) return true;
  const double per_elem = kvt == PA_KV_BF16 ? 2.0 : (kvt == PA_KV_FP8_E4M3 ? 1.0 : 0.5 + 1.0 / 16.0);
  return (double)num_pages * page_size * (dqk + dvo) * per_elem <= 256.0 * 1024.0;
}

// Checks shared by both phases.  Returns PA_OK or an error status.
int check_common(const void* q, const void* kv_cache, const int32_t* kv_indptr, const int32_t* kv_indices,
                 const int32_t* kv_last_page_len, int batch, int num_pages, int Hq, int Hkv, int dqk, int dvo,
                 int page_size, float sm_scale, int window_left, int kv_dtype, const pa_kv_scales* sc,
                 const void* out, const float* lse) {
  if (batch < 0 || num_pages < 1 || Hq < 1 || Hkv < 1) return PA_ERR_INVALID_ARG;
  if (!q || !kv_cache || !kv_indptr || !kv_indices || !kv_last_page_len || !out) return PA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return PA_ERR_INVALID_ARG;
  if (Hq / Hkv > 16) return PA_ERR_UNSUPPORTED;
  if (!((dqk == 512 && dvo == 512) || (dqk == 512 && dvo == 256) || (dqk == 256 && dvo == 256)))
    return PA_ERR_UNSUPPORTED;
  if (page_size < 1 || page_size > 64 || (page_size & (page_size - 1))) return PA_ERR_UNSUPPORTED;
  if (!std::isfinite(sm_scale) || window_left < -1) return PA_ERR_INVALID_ARG;
  if (kv_dtype != PA_KV_BF16 && kv_dtype != PA_KV_FP8_E4M3 && kv_dtype != PA_KV_NVFP4) return PA_ERR_INVALID_ARG;
  if (kv_dtype != PA_KV_BF16) {
    if (!sc || !sc->k_scale || !sc->v_scale) return PA_ERR_INVALID_ARG;
    if (!aligned(sc->k_scale, 4) || !aligned(sc->v_scale, 4)) return PA_ERR_ALIGNMENT;
  }
  if (kv_dtype == PA_KV_NVFP4) {
    if (!sc->sf) return PA_ERR_INVALID_ARG;
    if (!aligned(sc->sf, 16)) return PA_ERR_ALIGNMENT;
  }
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16)) return PA_ERR_ALIGNMENT;
  if (!aligned(kv_indptr, 4) || !aligned(kv_indices, 4) || !aligned(kv_last_page_len, 4)) return PA_ERR_ALIGNMENT;
  if (lse && !aligned(lse, 4)) return PA_ERR_ALIGNMENT;
  const uint64_t page_bytes = (uint64_t)Hkv * page_size * (dqk + dvo) * x2_of(kv_dtype) / 2;
  if ((uint64_t)num_pages * page_bytes >= (1ull << 46)) return PA_ERR_INVALID_ARG;
  return PA_OK;
}

int device_sms(int* smem_optin) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  return sms;
}

// K, V (and NVFP4 scale) maps over the cache; boxes of box_rows rows of box_inner bytes
// (the scale boxes hold whole scale rows).
bool make_kv_maps(CUtensorMap* tk, CUtensorMap* tv, CUtensorMap* tsfk, CUtensorMap* tsfv, const void* kv_cache,
                  const uint8_t* sf, int num_pages, int Hkv, int dqk, int dvo, int ps, int kvt, int box_rows,
                  bool swz, uint32_t box_inner = 128) {
  const int x2 = x2_of(kvt);
  const uint64_t k_row = (uint64_t)dqk * x2 / 2, v_row = (uint64_t)dvo * x2 / 2;
  const uint64_t rows = (uint64_t)Hkv * ps;
  const uint64_t page_bytes = rows * (k_row + v_row);
  const uint8_t* base = static_cast<const uint8_t*>(kv_cache);
  if (!make_map(tk, base, k_row, rows, num_pages, page_bytes, box_inner, box_rows, swz)) return false;
  if (!make_map(tv, base + rows * k_row, v_row, rows, num_pages, page_bytes, box_inner, box_rows, swz)) return false;
  if (kvt == KV_NVFP4) {
    const uint64_t sk = dqk / 16, sv = dvo / 16, sf_page = rows * (sk + sv);
    if (!make_map(tsfk, sf, sk, rows, num_pages, sf_page, (uint32_t)sk, box_rows, false)) return false;
    if (!make_map(tsfv, sf + rows * sk, sv, rows, num_pages, sf_page, (uint32_t)sv, box_rows, false)) return false;
  } else {
    *tsfk = *tk;
    *tsfv = *tv;
  }
  return true;
}

// Decode: K and V maps whose boxes hold every 128-byte segment of box_rows rows of one
// page (one load per page piece), NVFP4 scale maps as for the prefill.
bool make_decode_maps(CUtensorMap* tk, CUtensorMap* tv, CUtensorMap* tsfk, CUtensorMap* tsfv, const void* kv_cache,
                      const uint8_t* sf, int num_pages, int Hkv, int dqk, int dvo, int ps, int kvt, int box_rows,
                      bool swz) {
  const int x2 = x2_of(kvt);
  const uint64_t k_row = (uint64_t)dqk * x2 / 2, v_row = (uint64_t)dvo * x2 / 2;
  const uint64_t rows = (uint64_t)Hkv * ps;
  const uint64_t page_bytes = rows * (k_row + v_row);
  const uint8_t* base = static_cast<const uint8_t*>(kv_cache);
  if (!make_map_rows(tk, base, k_row, rows, num_pages, page_bytes, box_rows, swz)) return false;
  if (!make_map_rows(tv, base + rows * k_row, v_row, rows, num_pages, page_bytes, box_rows, swz)) return false;
  if (kvt == KV_NVFP4) {
    const uint64_t sk = dqk / 16, sv = dvo / 16, sf_page = rows * (sk + sv);
    if (!make_map(tsfk, sf, sk, rows, num_pages, sf_page, (uint32_t)sk, box_rows, false)) return false;
    if (!make_map(tsfv, sf + rows * sk, sv, rows, num_pages, sf_page, (uint32_t)sv, box_rows, false)) return false;
  } else {
    *tsfk = *tk;
    *tsfv = *tv;
  }
  return true;
}

}  // namespace
}  // namespace pa

// ---------------------------------------------------------------------------------------
// paged_attn_decode_noalloc's scratch: the decode call for callers that cannot allocate
// device memory (an engine plugin handed a fixed pool, a memory-budgeted service, code
// that must not trigger cudaMalloc's implicit device synchronisation mid-step) uses this
// statically sized device array instead of the grow-only workspace; it calls no
// cudaMalloc, cudaFree or other allocating routine.
//
// In host code `g_pa_noalloc_scratch` names only a host-side stand-in of the device
// array: handing it to a kernel would fault or, where the GPU can reach host memory,
// silently use the wrong memory.  Its device address comes from cudaGetSymbolAddress,
// resolved once per device (with that device current) by the first call on that device,
// which also zeroes the array's error word; that first call should therefore come before
// any stream capture.
static __device__ __align__(256) uint8_t g_pa_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

namespace pa {
namespace {
void* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mutex;

void* noalloc_scratch(int* status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *status = PA_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_pa_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      *status = PA_ERR_CUDA;
      return nullptr;
    }
    // the error word starts at zero; afterwards only paged_attn_check_device_error clears it
    if (cudaMemset(static_cast<char*>(p) + kErrOffset, 0, sizeof(int)) != cudaSuccess) {
      cudaGetLastError();
      *status = PA_ERR_CUDA;
      return nullptr;
    }
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

// Reads and clears one device error word (blocking); returns its value, or -1 on a CUDA error.
int take_error_word(void* base) {
  int v = 0;
  char* e = static_cast<char*>(base) + kErrOffset;
  if (cudaMemcpy(&v, e, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
  if (v != 0 && cudaMemset(e, 0, sizeof v) != cudaSuccess) return -1;
  return v;
}
}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

const char* paged_attn_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration (shape, group size, page size or dtype not built)";
    case PA_ERR_ALIGNMENT: return "pointer not aligned (device arrays need 16-byte alignment, int32 arrays 4)";
    case PA_ERR_SMEM: return "kernel shared memory exceeds the device opt-in limit";
    case PA_ERR_CUDA: return "CUDA runtime or driver call failed";
    case PA_ERR_DEVICE: return "a kernel gave up on a bounded wait";
    case PA_ERR_SCRATCH: return "problem needs more scratch than paged_attn_decode_noalloc's fixed array holds";
    default: return "unknown status";
  }
}

int paged_attn_last_variant(char* buf, int len) {
  if (!buf || len <= 0) return PA_ERR_INVALID_ARG;
  std::snprintf(buf, (size_t)len, "%s", g_variant);
  return PA_OK;
}

int paged_attn_set_prefill_dequant_limit(long long bytes) {
  g_prefill_dequant_limit = bytes < 0 ? kDefaultDequantLimit : (uint64_t)bytes;
  return PA_OK;
}

int paged_attn_set_prefill_cta_pairs(int mode) {
  if (mode < -1 || mode > 1) return PA_ERR_INVALID_ARG;
  g_prefill_pairs = mode < 0 ? 0 : mode;
  return PA_OK;
}

int paged_attn_set_prefill_split_kv(int mode) {
  if (mode < -1 || mode > 0) return PA_ERR_INVALID_ARG;
  g_prefill_split = mode;
  return PA_OK;
}

int paged_attn_set_decode_direct(int mode) {
  if (mode < -1 || mode > 1) return PA_ERR_INVALID_ARG;
  g_decode_direct = mode;
  return PA_OK;
}

int paged_attn_set_decode_chunk_pages(int pages) {
  if (pages < 0) return PA_ERR_INVALID_ARG;
  g_forced_chunk_pages = pages;
  return PA_OK;
}

int paged_attn_release_workspace(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  for (auto& kv : g_ws[dev])
    if (kv.second.base && cudaFree(kv.second.base) != cudaSuccess) return PA_ERR_CUDA;
  g_ws[dev].clear();
  return PA_OK;
}

int paged_attn_profile_begin(int max_launches) {
  if (max_launches < 1 || max_launches > (1 << 20)) return PA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_prof_mutex);
  for (size_t i = 0; i < g_prof.start.size(); ++i) {
    cudaEventDestroy(g_prof.start[i]);
    cudaEventDestroy(g_prof.stop[i]);
  }
  g_prof.start.assign(max_launches, nullptr);
  g_prof.stop.assign(max_launches, nullptr);
  for (int i = 0; i < max_launches; ++i)
    if (cudaEventCreate(&g_prof.start[i]) != cudaSuccess || cudaEventCreate(&g_prof.stop[i]) != cudaSuccess)
      return PA_ERR_CUDA;
  g_prof.used = 0;
  g_prof.on = true;
  return PA_OK;
}

int paged_attn_profile_end(int* launches, float* total_ms) {
  std::lock_guard<std::mutex> lock(g_prof_mutex);
  g_prof.on = false;
  double sum = 0.0;
  for (int i = 0; i < g_prof.used; ++i) {
    if (cudaEventSynchronize(g_prof.stop[i]) != cudaSuccess) return PA_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_prof.start[i], g_prof.stop[i]) != cudaSuccess) return PA_ERR_CUDA;
    sum += ms;
  }
  if (launches) *launches = g_prof.used;
  if (total_ms) *total_ms = (float)sum;
  return PA_OK;
}

int paged_attn_check_device_error(int* code) {
  if (code) *code = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  // the error word of every stream's workspace and, once paged_attn_decode_noalloc has
  // run on this device, the one in its fixed array; all are cleared, the first nonzero
  // is reported
  int v = 0;
  {
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    for (auto& kv : g_ws[dev]) {
      if (!kv.second.base) continue;
      const int w = take_error_word(kv.second.base);
      if (w < 0) return PA_ERR_CUDA;
      if (v == 0) v = w;
    }
  }
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev]) {
      const int w = take_error_word(g_noalloc_ptr[dev]);
      if (w < 0) return PA_ERR_CUDA;
      if (v == 0) v = w;
    }
  }
  if (code) *code = v;
  return v ? PA_ERR_DEVICE : PA_OK;
}

int paged_attn_debug_set_error_word(int target, int code) {
  if (target != 0 && target != 1) return PA_ERR_INVALID_ARG;
  int st = PA_OK;
  void* base = target == 0 ? workspace(kFixedBytes, nullptr, &st) : noalloc_scratch(&st);
  if (!base) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
  if (cudaMemcpy(static_cast<char*>(base) + kErrOffset, &code, sizeof code, cudaMemcpyHostToDevice) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

int paged_attn_decode(const void* q, const void* kv_cache, const int32_t* kv_indptr, const int32_t* kv_indices,
                      const int32_t* kv_last_page_len, int batch, int num_pages, int num_qo_heads,
                      int num_kv_heads, int head_dim_qk, int head_dim_vo, int page_size, float sm_scale,
                      int window_left, int kv_dtype, const pa_kv_scales* kv_scales, void* out, float* lse,
                      void* stream) {
  int st = check_common(q, kv_cache, kv_indptr, kv_indices, kv_last_page_len, batch, num_pages, num_qo_heads,
                        num_kv_heads, head_dim_qk, head_dim_vo, page_size, sm_scale, window_left, kv_dtype,
                        kv_scales, out, lse);
  if (st != PA_OK) return st;
  if (batch == 0) return PA_OK;
  const int group = num_qo_heads / num_kv_heads;
  const int hp = group <= 8 ? 8 : 16;
  int smem_optin = 0;
  const int sms = device_sms(&smem_optin);
  if (sms <= 0) return PA_ERR_CUDA;
  const int smem = decode_smem_bytes(kv_dtype, head_dim_qk, head_dim_vo, hp);
  if (smem > smem_optin) return PA_ERR_SMEM;

  DecodeLaunch L;
  std::memset(&L, 0, sizeof L);
  const int T = decode_tile_tokens(kv_dtype, head_dim_qk);
  const int box_rows = page_size < T ? page_size : T;
  const bool swz = page_size >= 8;
  if (!make_decode_maps(&L.tk, &L.tv, &L.tsfk, &L.tsfv, kv_cache, kv_scales ? kv_scales->sf : nullptr, num_pages,
                        num_kv_heads, head_dim_qk, head_dim_vo, page_size, kv_dtype, box_rows, swz))
    return PA_ERR_CUDA;

  const bool direct = decode_direct(kv_dtype, head_dim_qk, head_dim_vo, page_size, num_pages, batch, num_kv_heads, sms);
  const int grid = direct ? std::min(sms, batch * num_kv_heads) : sms;
  const int forced = g_forced_chunk_pages;
  const int target = forced > 0 ? 2048 : (16 * grid + num_kv_heads - 1) / num_kv_heads;
  const int max_chunks = target + batch;
  size_t off = kFixedBytes;
  const size_t o_hdr = off; off = align_up(off + 64, 256);
  const size_t o_chunks = off; off = align_up(off + (size_t)max_chunks * sizeof(DecodeChunk), 256);
  const size_t o_seq = off; off = align_up(off + (size_t)batch * sizeof(int2), 256);
  const size_t o_ml = off; off = align_up(off + (size_t)max_chunks * num_qo_heads * sizeof(float2), 256);
  const size_t o_o = off; off = align_up(off + (size_t)max_chunks * num_qo_heads * head_dim_vo * sizeof(float), 256);
  char* ws = static_cast<char*>(workspace(off, static_cast<cudaStream_t>(stream), &st));
  if (!ws) return st;

  DecodeParams& p = L.p;
  p.q = static_cast<const uint16_t*>(q);
  p.kv_indptr = kv_indptr;
  p.kv_indices = kv_indices;
  p.kv_last_page_len = kv_last_page_len;
  p.k_scale = kv_dtype != PA_KV_BF16 ? kv_scales->k_scale : nullptr;
  p.v_scale = kv_dtype != PA_KV_BF16 ? kv_scales->v_scale : nullptr;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.err = reinterpret_cast<int*>(ws + kErrOffset);
  p.hdr = reinterpret_cast<int*>(ws + o_hdr);
  p.chunks = reinterpret_cast<DecodeChunk*>(ws + o_chunks);
  p.seq_info = reinterpret_cast<int2*>(ws + o_seq);
  p.ws_ml = reinterpret_cast<float2*>(ws + o_ml);
  p.ws_o = reinterpret_cast<float*>(ws + o_o);
  p.batch = batch;
  p.Hq = num_qo_heads;
  p.Hkv = num_kv_heads;
  p.group = group;
  p.page_size = page_size;
  p.window_left = window_left;
  p.max_chunks = max_chunks;
  p.target_chunks = target;
  p.forced_chunk_pages = forced;
  p.min_chunk_pages = decode_min_chunk_pages(kv_dtype, head_dim_qk, head_dim_vo, page_size);
  p.grid = grid;
  p.box_rows = box_rows;
  p.box_shift = __builtin_ctz((unsigned)box_rows);
  p.swz = swz ? 7 : 0;
  p.direct = direct ? 1 : 0;
  p.sm_scale = sm_scale;
  L.grid = grid;
  L.stream = static_cast<cudaStream_t>(stream);

  if (!direct && launch_decode_plan(p, L.stream) != cudaSuccess) return PA_ERR_CUDA;
  const char* name = "?";
  cudaError_t e;
  prof_mark(L.stream, true);
  if (kv_dtype == PA_KV_BF16) e = launch_decode_bf16(head_dim_qk, head_dim_vo, hp, L, &name);
  else if (kv_dtype == PA_KV_FP8_E4M3) e = launch_decode_fp8(head_dim_qk, head_dim_vo, hp, L, &name);
  else e = launch_decode_nvfp4(head_dim_qk, head_dim_vo, hp, L, &name);
  prof_mark(L.stream, false);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  if (!direct && launch_decode_merge(head_dim_vo, p, L.grid, L.stream) != cudaSuccess) return PA_ERR_CUDA;
  static const char* kv_names[3] = {"bf16", "fp8", "nvfp4"};
  std::snprintf(g_variant, sizeof g_variant, "%s_%s%s", name, kv_names[kv_dtype], direct ? "_direct" : "");
  return PA_OK;
}

}  // extern "C"

namespace {
// paged_attn_prefill and paged_attn_prefill_custom_mask (mask == nullptr: none)
int prefill_call(const void* q, const int32_t* qo_indptr, int total_q, const void* kv_cache,
                 const int32_t* kv_indptr, const int32_t* kv_indices, const int32_t* kv_last_page_len, int batch,
                 int num_pages, int num_qo_heads, int num_kv_heads, int head_dim_qk, int head_dim_vo,
                 int page_size, float sm_scale, int window_left, int causal, int kv_dtype,
                 const pa_kv_scales* kv_scales, void* out, float* lse, const uint8_t* mask,
                 const int64_t* mask_indptr, void* stream) {
  int st = check_common(q, kv_cache, kv_indptr, kv_indices, kv_last_page_len, batch, num_pages, num_qo_heads,
                        num_kv_heads, head_dim_qk, head_dim_vo, page_size, sm_scale, window_left, kv_dtype,
                        kv_scales, out, lse);
  if (st != PA_OK) return st;
  if (!qo_indptr || total_q < 0) return PA_ERR_INVALID_ARG;
  if (!aligned(qo_indptr, 4)) return PA_ERR_ALIGNMENT;
  if (batch == 0 || total_q == 0) return PA_OK;
  // K/V tiles are 128B-swizzled TMA boxes of page_size rows, which need whole 8-row atoms:
  // pages of 1, 2 or 4 tokens are read from a bf16 copy that pads each page to 8 rows
  const bool pad = page_size < 8;
  const int rows_copy = pad ? 8 : page_size;
  const int group = num_qo_heads / num_kv_heads;
  const int rows_per_tile = 128 / group;
  int smem_optin = 0;
  const int sms = device_sms(&smem_optin);
  if (sms <= 0) return PA_ERR_CUDA;
  // FP8 / NVFP4: convert the referenced pages once into a bf16 copy and run the bf16
  // kernel on it, when the copy fits the limit; else convert inside the kernel
  const bool quant = kv_dtype != PA_KV_BF16;
  const uint64_t bf16_page = (uint64_t)num_kv_heads * rows_copy * (head_dim_qk + head_dim_vo) * 2;
  const bool dequant = (quant || pad) && (uint64_t)num_pages * bf16_page <= g_prefill_dequant_limit.load();
  if (pad && !dequant) return PA_ERR_UNSUPPORTED;  // the padded copy would exceed the limit
  const int run_kvt = dequant ? (int)PA_KV_BF16 : kv_dtype;
  if (prefill_smem_bytes(run_kvt, head_dim_qk, head_dim_vo) > smem_optin) return PA_ERR_SMEM;
  // bf16 kernel (or the bf16 copy): CTA pairs share each MMA and each K/V tile
  int pair_grid = 0;
  if (run_kvt == PA_KV_BF16 && !pad && g_prefill_pairs.load() == 1)
    pair_grid = 2 * std::min(sms / 2, pair_clusters(head_dim_qk, head_dim_vo));

  // split KV (short queries over long KV): when even one item per (query tile, kv head)
  // cannot fill the SMs, the planner may split KV ranges; up to 3 x sms items and slots
  const long tiles_bound = ((long)total_q + rows_per_tile - 1) / rows_per_tile + batch;
  const bool split = g_prefill_split.load() != 0 && pair_grid == 0 && tiles_bound * num_kv_heads < sms;
  const int max_slots = split ? 3 * sms : 0;
  const long max_items = std::max(((long)total_q / rows_per_tile + batch) * num_kv_heads, (long)max_slots);
  if (max_items > (1l << 30)) return PA_ERR_INVALID_ARG;
  size_t off = kFixedBytes;
  const size_t o_hdr = off; off = align_up(off + 64, 256);
  const size_t o_items = off; off = align_up(off + (size_t)max_items * sizeof(PrefillItem), 256);
  const size_t o_toff = off; off = align_up(off + (size_t)(batch + 1) * sizeof(int), 256);
  // head_dim_vo 512: per-CTA P tiles of the first pass for items of up to kReuseTiles KV
  // tiles (longer ones recompute S in the second pass)
  const int reuse_tiles = head_dim_vo == 512 ? kReuseTiles : 0;
  const size_t o_pscr = off; off = align_up(off + (size_t)sms * reuse_tiles * 32768, 256);
  const size_t o_mscr = off; off = align_up(off + (size_t)sms * reuse_tiles * 128 * sizeof(float), 256);
  const size_t o_shadow = off; off = align_up(off + (dequant ? (size_t)num_pages * bf16_page : 0), 256);
  const size_t o_part = off; off = align_up(off + (size_t)max_slots * 128 * head_dim_vo * sizeof(float), 256);
  const size_t o_plse = off; off = align_up(off + (size_t)max_slots * 128 * sizeof(float), 256);
  const size_t o_merge = off; off = align_up(off + (size_t)max_slots * sizeof(PrefillMerge), 256);
  char* ws = static_cast<char*>(workspace(off, static_cast<cudaStream_t>(stream), &st));
  if (!ws) return st;

  PrefillLaunch L;
  std::memset(&L, 0, sizeof L);
  // bf16 K/V (or the bf16 copy): 128B-swizzled boxes of [page_size][64 elements], read by
  // the MMAs as they land.  FP8 / NVFP4 converted in the kernel: unswizzled boxes of the
  // packed bytes of 64 elements per key (64 / 32 B) and whole block-scale rows, staged for
  // the converter warps.
  const void* kv_read = dequant ? static_cast<const void*>(ws + o_shadow) : kv_cache;
  const bool packed = run_kvt != PA_KV_BF16;
  if (!make_kv_maps(&L.tk, &L.tv, &L.tsfk, &L.tsfv, kv_read, packed ? kv_scales->sf : nullptr, num_pages,
                    num_kv_heads, head_dim_qk, head_dim_vo, rows_copy, run_kvt, rows_copy, !packed,
                    packed ? (run_kvt == KV_FP8 ? 64u : 32u) : 128u))
    return PA_ERR_CUDA;
  // Q as [total_q][Hq][d_qk] bf16 bytes: boxes of [rows_per_tile][group][128 B]
  {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return PA_ERR_CUDA;
    cuuint64_t dims[3] = {(cuuint64_t)head_dim_qk * 2, (cuuint64_t)num_qo_heads, (cuuint64_t)total_q};
    cuuint64_t strides[2] = {(cuuint64_t)head_dim_qk * 2, (cuuint64_t)num_qo_heads * head_dim_qk * 2};
    cuuint32_t box[3] = {128, (cuuint32_t)group, (cuuint32_t)rows_per_tile};
    cuuint32_t estr[3] = {1, 1, 1};
    if (fn(&L.tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(q), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PA_ERR_CUDA;
  }
  // CTA pairs: the P scratch as rows of 128 bytes, one P tile (32 KB) per box
  L.tp = L.tq;
  if (pair_grid > 0 && reuse_tiles > 0) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return PA_ERR_CUDA;
    cuuint64_t dims[2] = {128, (cuuint64_t)sms * reuse_tiles * 256};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {128, 256};
    cuuint32_t estr[2] = {1, 1};
    if (fn(&L.tp, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, ws + o_pscr, dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PA_ERR_CUDA;
  }
  PrefillParams& p = L.p;
  p.q = static_cast<const uint16_t*>(q);
  p.qo_indptr = qo_indptr;
  p.kv_indptr = kv_indptr;
  p.kv_indices = kv_indices;
  p.kv_last_page_len = kv_last_page_len;
  p.k_scale = kv_dtype != PA_KV_BF16 ? kv_scales->k_scale : nullptr;
  p.v_scale = kv_dtype != PA_KV_BF16 ? kv_scales->v_scale : nullptr;
  p.kv_cache = static_cast<const uint8_t*>(kv_cache);
  p.sf = kv_scales ? kv_scales->sf : nullptr;
  p.out = static_cast<uint16_t*>(out);
  p.out_v8 = aligned(out, 32) ? 1 : 0;
  p.lse = lse;
  p.err = reinterpret_cast<int*>(ws + kErrOffset);
  p.hdr = reinterpret_cast<int*>(ws + o_hdr);
  p.items = reinterpret_cast<PrefillItem*>(ws + o_items);
  p.tile_off = reinterpret_cast<int*>(ws + o_toff);
  p.p_scratch = reinterpret_cast<uint8_t*>(ws + o_pscr);
  p.m_scratch = reinterpret_cast<float*>(ws + o_mscr);
  p.reuse_tiles = reuse_tiles;
  p.batch = batch;
  p.total_q = total_q;
  p.Hq = num_qo_heads;
  p.Hkv = num_kv_heads;
  p.group = group;
  p.page_size = page_size;
  p.window_left = window_left;
  p.causal = causal ? 1 : 0;
  p.num_pages = num_pages;
  p.rows_per_tile = rows_per_tile;
  p.pair = pair_grid > 0 ? 1 : 0;
  p.mask = mask;
  p.mask_indptr = mask_indptr;
  p.split_target = split ? sms : 0;
  p.part_o = reinterpret_cast<float*>(ws + o_part);
  p.part_lse = reinterpret_cast<float*>(ws + o_plse);
  p.merges = reinterpret_cast<PrefillMerge*>(ws + o_merge);
  p.max_slots = max_slots;
  p.max_items = (int)max_items;
  p.box_rows = rows_copy;
  p.tile_tok = 128 / rows_copy * page_size;
  p.swz = 7;
  p.sm_scale = sm_scale;
  L.grid = pair_grid > 0 ? pair_grid : sms;
  L.stream = static_cast<cudaStream_t>(stream);

  DequantParams d;
  std::memset(&d, 0, sizeof d);
  if (dequant) {
    d.cache = static_cast<const uint8_t*>(kv_cache);
    d.sf = kv_scales ? kv_scales->sf : nullptr;
    d.kv_indptr = kv_indptr;
    d.kv_indices = kv_indices;
    d.shadow = reinterpret_cast<uint16_t*>(ws + o_shadow);
    d.batch = batch;
    d.Hkv = num_kv_heads;
    d.page_size = page_size;
    d.out_rows = rows_copy;
  }
  if (launch_prefill_prep(kv_dtype, head_dim_qk, head_dim_vo, pad ? 2 : (dequant ? 1 : 0), p, d, sms, L.stream) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  const char* name = "?";
  prof_mark(L.stream, true);
  cudaError_t e = launch_prefill(run_kvt, head_dim_qk, head_dim_vo, L, &name);
  prof_mark(L.stream, false);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  if (split && launch_prefill_merge(head_dim_vo, p, sms, L.stream) != cudaSuccess) return PA_ERR_CUDA;
  static const char* kv_names[3] = {"bf16", "fp8", "nvfp4"};
  std::snprintf(g_variant, sizeof g_variant, "%s_%s%s%s%s", name, kv_names[kv_dtype],
                pad ? "_padded" : (dequant ? "_dequant" : ""), mask ? "_mask" : "", split ? "_splitkv" : "");
  return PA_OK;
}
}  // namespace

extern "C" {

int paged_attn_prefill(const void* q, const int32_t* qo_indptr, int total_q, const void* kv_cache,
                       const int32_t* kv_indptr, const int32_t* kv_indices, const int32_t* kv_last_page_len,
                       int batch, int num_pages, int num_qo_heads, int num_kv_heads, int head_dim_qk,
                       int head_dim_vo, int page_size, float sm_scale, int window_left, int causal, int kv_dtype,
                       const pa_kv_scales* kv_scales, void* out, float* lse, void* stream) {
  return prefill_call(q, qo_indptr, total_q, kv_cache, kv_indptr, kv_indices, kv_last_page_len, batch, num_pages,
                      num_qo_heads, num_kv_heads, head_dim_qk, head_dim_vo, page_size, sm_scale, window_left, causal,
                      kv_dtype, kv_scales, out, lse, nullptr, nullptr, stream);
}

int paged_attn_prefill_custom_mask(const void* q, const int32_t* qo_indptr, int total_q, const void* kv_cache,
                                   const int32_t* kv_indptr, const int32_t* kv_indices,
                                   const int32_t* kv_last_page_len, int batch, int num_pages, int num_qo_heads,
                                   int num_kv_heads, int head_dim_qk, int head_dim_vo, int page_size, float sm_scale,
                                   int window_left, int causal, int kv_dtype, const pa_kv_scales* kv_scales,
                                   void* out, float* lse, const uint8_t* custom_mask, const int64_t* mask_indptr,
                                   void* stream) {
  if (!custom_mask || !mask_indptr) return PA_ERR_INVALID_ARG;
  if (!aligned(mask_indptr, 8)) return PA_ERR_ALIGNMENT;
  return prefill_call(q, qo_indptr, total_q, kv_cache, kv_indptr, kv_indices, kv_last_page_len, batch, num_pages,
                      num_qo_heads, num_kv_heads, head_dim_qk, head_dim_vo, page_size, sm_scale, window_left, causal,
                      kv_dtype, kv_scales, out, lse, custom_mask, mask_indptr, stream);
}


int paged_attn_append_kv(const void* k_new, const void* v_new, const int32_t* append_indptr, int total_new,
                         void* kv_cache, const int32_t* kv_indptr, const int32_t* kv_indices,
                         const int32_t* kv_last_page_len, int batch, int num_pages, int num_kv_heads,
                         int head_dim_qk, int head_dim_vo, int page_size, int kv_dtype, const float* k_scale,
                         const float* v_scale, uint8_t* sf, void* stream) {
  if (batch < 0 || total_new < 0 || num_pages < 1 || num_kv_heads < 1) return PA_ERR_INVALID_ARG;
  if (kv_dtype != PA_KV_BF16 && kv_dtype != PA_KV_FP8_E4M3 && kv_dtype != PA_KV_NVFP4) return PA_ERR_INVALID_ARG;
  if (!((head_dim_qk == 512 && head_dim_vo == 512) || (head_dim_qk == 512 && head_dim_vo == 256) ||
        (head_dim_qk == 256 && head_dim_vo == 256)))
    return PA_ERR_UNSUPPORTED;
  if (page_size < 1 || page_size > 64 || (page_size & (page_size - 1))) return PA_ERR_UNSUPPORTED;
  if (batch == 0 || total_new == 0) return PA_OK;
  if (!k_new || !v_new || !append_indptr || !kv_cache || !kv_indptr || !kv_indices || !kv_last_page_len)
    return PA_ERR_INVALID_ARG;
  if (kv_dtype != PA_KV_BF16) {
    if (!k_scale || !v_scale) return PA_ERR_INVALID_ARG;
    if (!aligned(k_scale, 4) || !aligned(v_scale, 4)) return PA_ERR_ALIGNMENT;
  }
  if (kv_dtype == PA_KV_NVFP4 && !sf) return PA_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(kv_cache, 16)) return PA_ERR_ALIGNMENT;
  if (!aligned(append_indptr, 4) || !aligned(kv_indptr, 4) || !aligned(kv_indices, 4) ||
      !aligned(kv_last_page_len, 4))
    return PA_ERR_ALIGNMENT;
  const uint64_t page_bytes =
      (uint64_t)num_kv_heads * page_size * (head_dim_qk + head_dim_vo) * x2_of(kv_dtype) / 2;
  if ((uint64_t)num_pages * page_bytes >= (1ull << 46)) return PA_ERR_INVALID_ARG;
  if (page_bytes >= (1ull << 31)) return PA_ERR_UNSUPPORTED;  // the kernel's in-page offsets are 32-bit
  int st = PA_OK;
  char* ws = static_cast<char*>(workspace(kFixedBytes, static_cast<cudaStream_t>(stream), &st));
  if (!ws) return st;
  AppendParams p;
  std::memset(&p, 0, sizeof p);
  p.k_new = static_cast<const uint16_t*>(k_new);
  p.v_new = static_cast<const uint16_t*>(v_new);
  p.append_indptr = append_indptr;
  p.kv_indptr = kv_indptr;
  p.kv_indices = kv_indices;
  p.kv_last_page_len = kv_last_page_len;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.cache = static_cast<uint8_t*>(kv_cache);
  p.sf = sf;
  p.err = reinterpret_cast<int*>(ws + kErrOffset);
  p.batch = batch;
  p.total_new = total_new;
  p.num_pages = num_pages;
  p.Hkv = num_kv_heads;
  p.d_qk = head_dim_qk;
  p.d_vo = head_dim_vo;
  p.page_size = page_size;
  prof_mark(static_cast<cudaStream_t>(stream), true);
  int smem_optin = 0;
  const int sms = device_sms(&smem_optin);
  const cudaError_t e = launch_append_kv(kv_dtype, p, sms, static_cast<cudaStream_t>(stream));
  prof_mark(static_cast<cudaStream_t>(stream), false);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  static const char* kv_names[3] = {"bf16", "fp8", "nvfp4"};
  std::snprintf(g_variant, sizeof g_variant, "append_kv_%s", kv_names[kv_dtype]);
  return PA_OK;
}

}  // extern "C"

extern "C" int paged_attn_decode_noalloc(const void* q, const void* kv_cache, const int32_t* kv_indptr,
                                         const int32_t* kv_indices, const int32_t* kv_last_page_len, int batch,
                                         int num_pages, int num_qo_heads, int num_kv_heads, int head_dim_qk,
                                         int head_dim_vo, int page_size, float sm_scale, int window_left,
                                         int kv_dtype, const pa_kv_scales* kv_scales, void* out, float* lse,
                                         void* stream) {
  int st = check_common(q, kv_cache, kv_indptr, kv_indices, kv_last_page_len, batch, num_pages, num_qo_heads,
                        num_kv_heads, head_dim_qk, head_dim_vo, page_size, sm_scale, window_left, kv_dtype,
                        kv_scales, out, lse);
  if (st != PA_OK) return st;
  if (batch == 0) return PA_OK;
  const int group = num_qo_heads / num_kv_heads;
  const int hp = group <= 8 ? 8 : 16;
  int smem_optin = 0;
  const int sms = device_sms(&smem_optin);
  if (sms <= 0) return PA_ERR_CUDA;
  if (decode_smem_bytes(kv_dtype, head_dim_qk, head_dim_vo, hp) > smem_optin) return PA_ERR_SMEM;

  // Size the work list to the fixed array: fewer KV splits when the usual number does
  // not fit, PA_ERR_SCRATCH when not even one split per sequence fits.
  const size_t cap = PA_NOALLOC_SCRATCH_BYTES;
  const size_t per_chunk =
      sizeof(DecodeChunk) + (size_t)num_qo_heads * sizeof(float2) + (size_t)num_qo_heads * head_dim_vo * 4;
  const size_t fixed = kFixedBytes + 256 + align_up((size_t)batch * sizeof(int2), 256) + 4 * 256;
  if (fixed >= cap) return PA_ERR_SCRATCH;
  const long fit = (long)((cap - fixed) / per_chunk) - batch;
  const int forced = g_forced_chunk_pages;
  const bool direct = decode_direct(kv_dtype, head_dim_qk, head_dim_vo, page_size, num_pages, batch, num_kv_heads, sms);
  const int grid = direct ? std::min(sms, batch * num_kv_heads) : sms;
  const long usual = forced > 0 ? 2048 : (16 * grid + num_kv_heads - 1) / num_kv_heads;
  const long target = fit < usual ? fit : usual;
  if (target < 1) return PA_ERR_SCRATCH;
  const int max_chunks = (int)target + batch;
  size_t off = kFixedBytes;
  const size_t o_hdr = off; off = align_up(off + 64, 256);
  const size_t o_chunks = off; off = align_up(off + (size_t)max_chunks * sizeof(DecodeChunk), 256);
  const size_t o_seq = off; off = align_up(off + (size_t)batch * sizeof(int2), 256);
  const size_t o_ml = off; off = align_up(off + (size_t)max_chunks * num_qo_heads * sizeof(float2), 256);
  const size_t o_o = off; off = align_up(off + (size_t)max_chunks * num_qo_heads * head_dim_vo * sizeof(float), 256);
  if (off > cap) return PA_ERR_SCRATCH;
  char* ws = static_cast<char*>(noalloc_scratch(&st));
  if (!ws) return st;

  DecodeLaunch L;
  std::memset(&L, 0, sizeof L);
  const int T = decode_tile_tokens(kv_dtype, head_dim_qk);
  const int box_rows = page_size < T ? page_size : T;
  const bool swz = page_size >= 8;
  if (!make_decode_maps(&L.tk, &L.tv, &L.tsfk, &L.tsfv, kv_cache, kv_scales ? kv_scales->sf : nullptr, num_pages,
                        num_kv_heads, head_dim_qk, head_dim_vo, page_size, kv_dtype, box_rows, swz))
    return PA_ERR_CUDA;
  L.grid = grid;
  L.stream = static_cast<cudaStream_t>(stream);
  // nothing else must start at zero: the error word was zeroed at set-up and is cleared
  // only by paged_attn_check_device_error, the planner rewrites the work list, and every
  // partial is written before it is read

  DecodeParams& p = L.p;
  p.q = static_cast<const uint16_t*>(q);
  p.kv_indptr = kv_indptr;
  p.kv_indices = kv_indices;
  p.kv_last_page_len = kv_last_page_len;
  p.k_scale = kv_dtype != PA_KV_BF16 ? kv_scales->k_scale : nullptr;
  p.v_scale = kv_dtype != PA_KV_BF16 ? kv_scales->v_scale : nullptr;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.err = reinterpret_cast<int*>(ws + kErrOffset);
  p.hdr = reinterpret_cast<int*>(ws + o_hdr);
  p.chunks = reinterpret_cast<DecodeChunk*>(ws + o_chunks);
  p.seq_info = reinterpret_cast<int2*>(ws + o_seq);
  p.ws_ml = reinterpret_cast<float2*>(ws + o_ml);
  p.ws_o = reinterpret_cast<float*>(ws + o_o);
  p.batch = batch;
  p.Hq = num_qo_heads;
  p.Hkv = num_kv_heads;
  p.group = group;
  p.page_size = page_size;
  p.window_left = window_left;
  p.max_chunks = max_chunks;
  p.target_chunks = (int)target;
  p.forced_chunk_pages = forced;
  p.min_chunk_pages = decode_min_chunk_pages(kv_dtype, head_dim_qk, head_dim_vo, page_size);
  p.grid = grid;
  p.box_rows = box_rows;
  p.box_shift = __builtin_ctz((unsigned)box_rows);
  p.swz = swz ? 7 : 0;
  p.direct = direct ? 1 : 0;
  p.sm_scale = sm_scale;

  if (!direct && launch_decode_plan(p, L.stream) != cudaSuccess) return PA_ERR_CUDA;
  const char* name = "?";
  cudaError_t e;
  prof_mark(L.stream, true);
  if (kv_dtype == PA_KV_BF16) e = launch_decode_bf16(head_dim_qk, head_dim_vo, hp, L, &name);
  else if (kv_dtype == PA_KV_FP8_E4M3) e = launch_decode_fp8(head_dim_qk, head_dim_vo, hp, L, &name);
  else e = launch_decode_nvfp4(head_dim_qk, head_dim_vo, hp, L, &name);
  prof_mark(L.stream, false);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  if (!direct && launch_decode_merge(head_dim_vo, p, L.grid, L.stream) != cudaSuccess) return PA_ERR_CUDA;
  static const char* kv_names[3] = {"bf16", "fp8", "nvfp4"};
  std::snprintf(g_variant, sizeof g_variant, "%s_%s%s_noalloc", name, kv_names[kv_dtype], direct ? "_direct" : "");
  return PA_OK;
}

// launch.h -- host-side launch descriptors passed from api.cu to the per-dtype
// translation units that instantiate the kernels.
#pragma once

#include <atomic>

#include <cuda.h>
#include <cuda_runtime.h>

#include "kernel_params.h"

namespace pa {

struct DecodeLaunch {
  CUtensorMap tk, tv, tsfk, tsfv;
  DecodeParams p;
  int grid;
  cudaStream_t stream;
};

struct PrefillLaunch {
  CUtensorMap tq, tk, tv, tsfk, tsfv;
  CUtensorMap tp;  // CTA pairs: the P scratch (rows of 128 bytes, boxes of one P tile)
  PrefillParams p;
  int grid;
  cudaStream_t stream;
};

// Launch `kern` on `stream` with programmatic stream serialization: it may begin while
// the preceding kernel on the stream finishes (the kernel itself waits for that one
// before it touches global memory, see grid_dep_wait in common.cuh).
// Raise a kernel's dynamic shared-memory limit to `bytes` on the current device, once per
// device: `done` is the caller's per-kernel record of the devices already set (the
// attribute is per device, and setting it on every call costs host time on every call).
template <typename Kern>
inline cudaError_t set_smem_limit_once(Kern kern, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, int cluster_x,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Each returns cudaSuccess or the launch error; `variant` receives a static name.
// Returns cudaErrorInvalidValue for a shape that has no instantiation.
cudaError_t launch_decode_bf16(int dqk, int dvo, int hp, const DecodeLaunch& L, const char** variant);
cudaError_t launch_decode_fp8(int dqk, int dvo, int hp, const DecodeLaunch& L, const char** variant);
cudaError_t launch_decode_nvfp4(int dqk, int dvo, int hp, const DecodeLaunch& L, const char** variant);
cudaError_t launch_decode_plan(const DecodeParams& p, cudaStream_t s);
cudaError_t launch_decode_merge(int dvo, const DecodeParams& p, int sms, cudaStream_t s);
// Shared memory (bytes) the decode kernel of this shape needs.
int decode_smem_bytes(int kvt, int dqk, int dvo, int hp);
// Tokens per decode tile of this shape.
int decode_tile_tokens(int kvt, int dqk);

cudaError_t launch_prefill(int kvt, int dqk, int dvo, const PrefillLaunch& L, const char** variant);
// The prefill's planner (block 0) and, when the kernel reads a bf16 copy of the pages,
// the copy (the other blocks), in one launch.  copy: 0 none, 1 FP8 / NVFP4 pages
// converted, 2 pages of fewer than 8 tokens padded to 8 rows (any dtype, converted).
cudaError_t launch_prefill_prep(int kvt, int dqk, int dvo, int copy, const PrefillParams& p,
                                const DequantParams& d, int sms, cudaStream_t s);
// Split KV: merges the partial slots the plan listed (hdr[1] entries) into the output.
cudaError_t launch_prefill_merge(int dvo, const PrefillParams& p, int grid, cudaStream_t s);
int prefill_smem_bytes(int kvt, int dqk, int dvo);
// Two-CTA clusters of the bf16 prefill kernel that fit on the device at once.
int prefill_pair_clusters(int dqk, int dvo);
// New tokens' bf16 K / V -> the paged cache in its element type (quantise-on-write).
cudaError_t launch_append_kv(int kvt, const AppendParams& p, int sms, cudaStream_t s);

}  // namespace pa

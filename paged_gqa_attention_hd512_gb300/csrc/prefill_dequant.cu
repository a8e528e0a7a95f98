// prefill_dequant.cu -- FP8 / NVFP4 pages -> a bf16 copy, for the tensor-core prefill.
//
// In a prefill every KV tile is read by every query tile at or after it (36 times per
// tile on average for 8 x 1024-token sequences with 8 query heads per kv head), so
// converting the packed values once, into a bf16 copy of the pages the batch references,
// costs far less than converting them on each read.  The copy has the bf16 page layout
// (K block [Hkv][page_size][d_qk], then V block [Hkv][page_size][d_vo]) at the same page
// index, so the bf16 kernel reads it with the caller's kv_indices.  Values: e4m3(code) and
// e2m1(nibble) x e4m3(block scale), both exact in bf16; the per-tensor / global scales are
// left to the prefill kernel ("feat(attention): asymmetric VO-split NVFP4 paged prefill
// (qk=512/vo=256) for Gemma-4 on SM120/121", NVFP4 split-KV correctness: scales of 16
// elements along head_dim of one token).
#include "common.cuh"
#include "launch.h"
#include "tc_helpers.cuh"

namespace pa {

template <int KVT, int DQK, int DVO>
__global__ void __launch_bounds__(256) prefill_dequant_kernel(DequantParams d) {
  const int n_entries = d.kv_indptr[d.batch];
  const size_t elems = (size_t)d.Hkv * d.page_size * (DQK + DVO);  // per page
  const size_t units = elems / 16;                                 // 16 outputs = one NVFP4 scale block
  const size_t in_page = KVT == KV_FP8 ? elems : elems / 2;
  for (int e = blockIdx.x; e < n_entries; e += gridDim.x) {
    const size_t page = (size_t)__ldg(d.kv_indices + e);
    const uint8_t* src = d.cache + page * in_page;
    uint4* dst = reinterpret_cast<uint4*>(d.shadow + page * elems);  // elems bf16 values per page
    for (size_t u = threadIdx.x; u < units; u += blockDim.x) {
      uint32_t w[8];
      if constexpr (KVT == KV_FP8) {
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(src) + u);
        const uint32_t in[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          w[2 * k] = f16x2_to_bf16x2(e4m3x2_to_f16x2(in[k] & 0xFFFFu));
          w[2 * k + 1] = f16x2_to_bf16x2(e4m3x2_to_f16x2(in[k] >> 16));
        }
      } else {
        const uint2 a = __ldg(reinterpret_cast<const uint2*>(src) + u);
        const uint32_t sb = __ldg(d.sf + page * units + u);
        const uint32_t sf2 = e4m3x2_to_f16x2(sb | (sb << 8));
        e2m1x8_to_f16x2x4(a.x, w);
        e2m1x8_to_f16x2x4(a.y, w + 4);
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = f16x2_to_bf16x2(hmul2_u32(w[k], sf2));
      }
      dst[2 * u] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[2 * u + 1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
}

template <int KVT>
static cudaError_t run_dequant(int dqk, int dvo, const DequantParams& d, int grid, cudaStream_t s) {
  if (dqk == 512 && dvo == 512) prefill_dequant_kernel<KVT, 512, 512><<<grid, 256, 0, s>>>(d);
  else if (dqk == 512 && dvo == 256) prefill_dequant_kernel<KVT, 512, 256><<<grid, 256, 0, s>>>(d);
  else if (dqk == 256 && dvo == 256) prefill_dequant_kernel<KVT, 256, 256><<<grid, 256, 0, s>>>(d);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_prefill_dequant(int kvt, int dqk, int dvo, const DequantParams& d, int grid, cudaStream_t s) {
  if (kvt == KV_FP8) return run_dequant<KV_FP8>(dqk, dvo, d, grid, s);
  if (kvt == KV_NVFP4) return run_dequant<KV_NVFP4>(dqk, dvo, d, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace pa

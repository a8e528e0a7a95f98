// prefill_dequant.cuh -- FP8 / NVFP4 pages -> a bf16 copy, for the tensor-core prefill.
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
#pragma once

#include "common.cuh"
#include "tc_helpers.cuh"

namespace pa {

// The blocks blk of nblk (blockDim.x threads each) convert the units of 16 values of every
// page entry kv_indices[0 .. kv_indptr[batch]) as one flat range, four units per thread
// and pass with their loads issued first.  A page listed by several sequences is
// converted by each of them, to the same values.
template <int KVT, int DQK, int DVO>
__device__ __forceinline__ void prefill_dequant_body(const DequantParams& d, int blk, int nblk) {
  constexpr int U = 4;
  const int n_entries = d.kv_indptr[d.batch];
  const uint32_t units = (uint32_t)d.Hkv * d.page_size * ((DQK + DVO) / 16);  // per page
  const uint64_t total = (uint64_t)n_entries * units;
  const uint64_t stride = (uint64_t)nblk * blockDim.x;
  const size_t elems = (size_t)units * 16;                             // values per page
  const size_t in_page = KVT == KV_FP8 ? elems : elems / 2;            // packed bytes per page
  for (uint64_t g0 = (uint64_t)blk * blockDim.x + threadIdx.x; g0 < total; g0 += U * stride) {
    uint4 a8[U];
    uint2 a4[U];
    uint32_t sb[U];
    size_t page[U];
    uint32_t u[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const uint64_t g = g0 + k * stride;
      if (g >= total) break;
      const uint32_t e = (uint32_t)(g / units);
      u[k] = (uint32_t)(g - (uint64_t)e * units);
      page[k] = (size_t)__ldg(d.kv_indices + e);
      const uint8_t* src = d.cache + page[k] * in_page;
      if constexpr (KVT == KV_FP8) {
        a8[k] = __ldg(reinterpret_cast<const uint4*>(src) + u[k]);
      } else {
        a4[k] = __ldg(reinterpret_cast<const uint2*>(src) + u[k]);
        sb[k] = __ldg(d.sf + page[k] * units + u[k]);
      }
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      if (g0 + k * stride >= total) break;
      uint32_t w[8];
      if constexpr (KVT == KV_FP8) {
        const uint32_t in[4] = {a8[k].x, a8[k].y, a8[k].z, a8[k].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          w[2 * j] = f16x2_to_bf16x2(e4m3x2_to_f16x2(in[j] & 0xFFFFu));
          w[2 * j + 1] = f16x2_to_bf16x2(e4m3x2_to_f16x2(in[j] >> 16));
        }
      } else {
        const uint32_t sf2 = e4m3x2_to_f16x2(sb[k] | (sb[k] << 8));
        e2m1x8_to_f16x2x4(a4[k].x, w);
        e2m1x8_to_f16x2x4(a4[k].y, w + 4);
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = f16x2_to_bf16x2(hmul2_u32(w[j], sf2));
      }
      uint4* dst = reinterpret_cast<uint4*>(d.shadow + page[k] * elems) + 2 * (size_t)u[k];
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
}

}  // namespace pa

// prefill_dequant.cuh -- FP8 / NVFP4 pages -> a bf16 copy, for the tensor-core prefill;
// pages of 1, 2 or 4 tokens (any dtype) -> a bf16 copy padded to 8 rows per kv head.
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
//
// Pages of fewer than 8 tokens cannot be loaded as the 128B-swizzled boxes of whole 8-row
// atoms the MMAs read, so the copy gives each page 8 rows per kv head: its page_size
// tokens, then zero rows; the kernel reads such a page as 8 rows and masks the padding.
#pragma once

#include "common.cuh"
#include "tc_helpers.cuh"

namespace pa {

// Copy unit u of a page (16 consecutive head-dim values of one row; K rows first, then V
// rows, each [Hkv][rows][dim]) in a page of `rows` rows per kv head: its kv head h, row r
// and first element in a page of `rows_to` rows per kv head.
template <int DQK, int DVO>
__device__ __forceinline__ void unit_place(uint32_t u, int Hkv, int rows, int& r, size_t& elem_src, int rows_src,
                                           size_t& elem_dst, int rows_dst) {
  constexpr uint32_t KB = DQK / 16, VB = DVO / 16;
  const uint32_t k_units = (uint32_t)Hkv * rows * KB;
  if (u < k_units) {
    const uint32_t h = u / (rows * KB), rem = u % (rows * KB);
    r = (int)(rem / KB);
    const uint32_t blk = rem % KB;
    elem_src = ((size_t)h * rows_src + r) * DQK + blk * 16;
    elem_dst = ((size_t)h * rows_dst + r) * DQK + blk * 16;
  } else {
    const uint32_t v = u - k_units;
    const uint32_t h = v / (rows * VB), rem = v % (rows * VB);
    r = (int)(rem / VB);
    const uint32_t blk = rem % VB;
    elem_src = (size_t)Hkv * rows_src * DQK + ((size_t)h * rows_src + r) * DVO + blk * 16;
    elem_dst = (size_t)Hkv * rows_dst * DQK + ((size_t)h * rows_dst + r) * DVO + blk * 16;
  }
}

// The blocks blk of nblk (blockDim.x threads each) write the copy units of 16 values of
// every page entry kv_indices[0 .. kv_indptr[batch]) as one flat range, four units per
// thread and pass with their loads issued first.  PAD: copy pages have out_rows (8) rows
// per kv head, rows past the page's page_size tokens zero.  A page listed by several
// sequences is written by each of them, with the same values.
template <int KVT, int DQK, int DVO, bool PAD>
__device__ __forceinline__ void prefill_dequant_body(const DequantParams& d, int blk, int nblk) {
  constexpr int U = 4;
  const int n_entries = d.kv_indptr[d.batch];
  const int rows_out = PAD ? d.out_rows : d.page_size;
  const uint32_t units_in = (uint32_t)d.Hkv * d.page_size * ((DQK + DVO) / 16);  // per caller page
  const uint32_t units = (uint32_t)d.Hkv * rows_out * ((DQK + DVO) / 16);        // per copy page
  const uint64_t total = (uint64_t)n_entries * units;
  const uint64_t stride = (uint64_t)nblk * blockDim.x;
  const size_t elems_out = (size_t)units * 16;                                 // values per copy page
  // bytes per caller page: 16 values per unit of 2, 1 or 1/2 bytes
  const size_t in_page = (size_t)units_in * (KVT == KV_BF16 ? 32 : (KVT == KV_FP8 ? 16 : 8));
  const uint64_t pol_keep = l2_policy_evict_last();
  for (uint64_t g0 = (uint64_t)blk * blockDim.x + threadIdx.x; g0 < total; g0 += U * stride) {
    uint4 a8[U], b8[U];
    uint2 a4[U];
    uint32_t sb[U];
    size_t page[U], dst_elem[U];
    bool zero[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const uint64_t g = g0 + k * stride;
      if (g >= total) break;
      const uint32_t e = (uint32_t)(g / units);
      const uint32_t u = (uint32_t)(g - (uint64_t)e * units);
      page[k] = (size_t)__ldg(d.kv_indices + e);
      uint32_t us = u;
      zero[k] = false;
      dst_elem[k] = (size_t)u * 16;
      if constexpr (PAD) {
        int r;
        size_t es;
        unit_place<DQK, DVO>(u, d.Hkv, rows_out, r, es, d.page_size, dst_elem[k], rows_out);
        zero[k] = r >= d.page_size;
        us = (uint32_t)(es / 16);
      }
      if (zero[k]) continue;
      if constexpr (KVT == KV_BF16) {
        const uint4* src = reinterpret_cast<const uint4*>(d.cache + page[k] * in_page) + 2 * (size_t)us;
        a8[k] = __ldg(src);
        b8[k] = __ldg(src + 1);
      } else if constexpr (KVT == KV_FP8) {
        a8[k] = __ldg(reinterpret_cast<const uint4*>(d.cache + page[k] * in_page) + us);
      } else {
        a4[k] = __ldg(reinterpret_cast<const uint2*>(d.cache + page[k] * in_page) + us);
        sb[k] = __ldg(d.sf + page[k] * units_in + us);
      }
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      if (g0 + k * stride >= total) break;
      uint32_t w[8];
      if (zero[k]) {
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = 0u;
      } else if constexpr (KVT == KV_BF16) {
        w[0] = a8[k].x, w[1] = a8[k].y, w[2] = a8[k].z, w[3] = a8[k].w;
        w[4] = b8[k].x, w[5] = b8[k].y, w[6] = b8[k].z, w[7] = b8[k].w;
      } else if constexpr (KVT == KV_FP8) {
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
      // one 32-byte store per unit (the copy's pages and units are 32-byte aligned), kept in
      // L2 for the prefill kernel that reads the copy next
      st_global_v8_hint(d.shadow + page[k] * elems_out + dst_elem[k], w, w + 4, pol_keep);
    }
  }
}

}  // namespace pa

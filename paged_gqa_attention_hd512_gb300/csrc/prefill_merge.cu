// prefill_merge.cu -- split KV for prefills of short queries over long KV: the output rows
// of each split (query tile, kv head) from its chunks' partial slots.
//
// Each chunk wrote its normalised rows (fp32) and lse = m + ln l; the row is the split-K
// merge of "[None][feat] Run Gemma4 head_dim 512 attention on Triton" (Not covered /
// Test Coverage: split-K): weights exp(lse_s - lse) with lse = ln sum_s exp(lse_s); a row
// that no chunk saw gives 0 and lse -inf.
//
// Grid: (merge entries, 16 blocks of 8 rows); a warp per row, its lanes over 4-column
// groups; every part's values are loaded before any is summed, so the loads of a row are
// in flight together.
#include "launch.h"
#include "common.cuh"

namespace pa {

namespace {

template <int DVO>
__global__ void __launch_bounds__(256) prefill_merge_kernel(const PrefillParams p) {
  constexpr int G4 = DVO / 128;  // float4 groups per lane
  grid_dep_wait();  // the prefill kernel's partial slots are complete
  const int n = p.hdr[1];
  const int g = p.group;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y * 8 + warp;  // row of the tile (position * g + head)
  for (int u = blockIdx.x; u < n; u += gridDim.x) {
    const PrefillMerge m = p.merges[u];
    const int qo_len = p.qo_indptr[m.b + 1] - p.qo_indptr[m.b];
    const int n_pos = min(p.rows_per_tile, qo_len - m.q_begin);
    if (r >= n_pos * g) continue;
    const int q_row0 = p.qo_indptr[m.b] + m.q_begin;
    float M = -INFINITY;
    for (int s = 0; s < m.parts; ++s) M = fmaxf(M, p.part_lse[(size_t)(m.slot0 + s) * 128 + r]);
    float L = 0.f;
    if (M != -INFINITY)
      for (int s = 0; s < m.parts; ++s) L += expf(p.part_lse[(size_t)(m.slot0 + s) * 128 + r] - M);
    const float lse = M == -INFINITY ? -INFINITY : M + logf(L);
    float4 acc[G4];
#pragma unroll
    for (int k = 0; k < G4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll 2
      for (int s = 0; s < m.parts; ++s) {
        const size_t base = (size_t)(m.slot0 + s) * 128 + r;
        const float w = expf(p.part_lse[base] - lse);
        float4 v[G4];
#pragma unroll
        for (int k = 0; k < G4; ++k) v[k] = __ldg(reinterpret_cast<const float4*>(p.part_o + base * DVO) + lane + 32 * k);
#pragma unroll
        for (int k = 0; k < G4; ++k) {
          acc[k].x += w * v[k].x;
          acc[k].y += w * v[k].y;
          acc[k].z += w * v[k].z;
          acc[k].w += w * v[k].w;
        }
      }
    }
    const size_t orow = ((size_t)(q_row0 + r / g) * p.Hq + m.kvh * g + r % g) * DVO;
#pragma unroll
    for (int k = 0; k < G4; ++k)
      *reinterpret_cast<uint2*>(p.out + orow + 4 * (lane + 32 * k)) =
          make_uint2(pack_bf16x2(acc[k].x, acc[k].y), pack_bf16x2(acc[k].z, acc[k].w));
    if (lane == 0 && p.lse) p.lse[(size_t)(q_row0 + r / g) * p.Hq + m.kvh * g + r % g] = lse;
  }
}

}  // namespace

cudaError_t launch_prefill_merge(int dvo, const PrefillParams& p, int grid, cudaStream_t s) {
  const dim3 g(grid, 16);
  if (dvo == 512) return launch_pdl(prefill_merge_kernel<512>, g, dim3(256), 0, s, 1, p);
  if (dvo == 256) return launch_pdl(prefill_merge_kernel<256>, g, dim3(256), 0, s, 1, p);
  return cudaErrorInvalidValue;
}

}  // namespace pa

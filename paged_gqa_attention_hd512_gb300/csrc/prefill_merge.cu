// prefill_merge.cu -- split KV for prefills of short queries over long KV: the output rows
// of each split (query tile, kv head) from its chunks' partial slots.
//
// Each chunk wrote its normalised rows (fp32) and lse = m + ln l; the row is the split-K
// merge of "[None][feat] Run Gemma4 head_dim 512 attention on Triton" (Not covered /
// Test Coverage: split-K): weights exp(lse_s - lse) with lse = ln sum_s exp(lse_s); a row
// that no chunk saw gives 0 and lse -inf.
//
// Grid: (merge entries, 16 blocks of 8 rows); a warp per row.  Lane s takes the lse of
// part s (32 parts at a time): the row's max and sum are warp reductions, and each lane
// forms its part's weight once.  The lanes then own 4-column groups and load four parts'
// values before summing them with the weights broadcast from their lanes, so the warp
// waits on memory once per four parts.
#include "launch.h"
#include "common.cuh"

namespace pa {

namespace {

template <int DVO>
__global__ void __launch_bounds__(256) prefill_merge_kernel(const PrefillParams p) {
  constexpr int G4 = DVO / 128;  // float4 groups per lane
  constexpr int B = 4;           // parts loaded together
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
    const float* plse = p.part_lse + (size_t)m.slot0 * 128 + r;  // part s at plse[s * 128]
    float M = -INFINITY;
    for (int s = lane; s < m.parts; s += 32) M = fmaxf(M, plse[(size_t)s * 128]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    if (M != -INFINITY)
      for (int s = lane; s < m.parts; s += 32) L += expf(plse[(size_t)s * 128] - M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    const float lse = M == -INFINITY ? -INFINITY : M + logf(L);
    float4 acc[G4];
#pragma unroll
    for (int k = 0; k < G4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
      const float4* src = reinterpret_cast<const float4*>(p.part_o + ((size_t)m.slot0 * 128 + r) * DVO) + lane;
      const size_t step = (size_t)128 * DVO / 4;  // float4s between consecutive parts
      for (int s0 = 0; s0 < m.parts; s0 += 32) {
        const float w = s0 + lane < m.parts ? expf(plse[(size_t)(s0 + lane) * 128] - lse) : 0.f;
        const int cnt = min(32, m.parts - s0);
        for (int k0 = 0; k0 < cnt; k0 += B) {
          float4 v[B][G4];
#pragma unroll
          for (int b = 0; b < B; ++b)
#pragma unroll
            for (int k = 0; k < G4; ++k)
              v[b][k] = k0 + b < cnt ? __ldg(src + (size_t)(s0 + k0 + b) * step + 32 * k) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int b = 0; b < B; ++b) {
            const float wb = __shfl_sync(0xffffffffu, w, (k0 + b) & 31);
#pragma unroll
            for (int k = 0; k < G4; ++k) {
              acc[k].x += wb * v[b][k].x;
              acc[k].y += wb * v[b][k].y;
              acc[k].z += wb * v[b][k].z;
              acc[k].w += wb * v[b][k].w;
            }
          }
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

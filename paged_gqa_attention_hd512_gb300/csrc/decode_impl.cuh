// decode_impl.cuh -- split-K flash-decoding over the paged HND cache (sm_103a).
//
// One query token per sequence ("Run Gemma4 head_dim 512 attention on Triton",
// Approach: decode over [num_pages, 2, num_kv_heads, page_size, head_dim] addressed by
// kv_indptr / kv_indices / kv_last_page_len; Test Coverage: split-K, sliding windows,
// FP8 KV, GQA 12/4 and 24/4 with head padding).  Three kernels per call:
//   decode_plan_kernel   cuts every sequence's (windowed) page range into page-aligned
//                        chunks on the device; no host synchronisation
//   decode_kernel        persistent CTAs; each work item is (chunk, kv head).  A producer
//                        warp streams K/V pages into a shared-memory ring with TMA; eight
//                        consumer warps run QK^T and PV as m16n8k16 tensor-core MMAs with
//                        all query heads of the kv head packed into the MMA N dimension
//                        (padded to 8 or 16), an online softmax, and write either the
//                        final row (one chunk) or a partial (O, m, l)
//   decode_merge_kernel  one warp per (sequence, query head) combines the partials
#pragma once

#include "common.cuh"

namespace pa {

// ----------------------------------------------------------------------------- config
template <int KVT, int DQK, int DVO>
struct DecodeCfg {
  static constexpr int X2 = KVT == KV_BF16 ? 4 : (KVT == KV_FP8 ? 2 : 1);  // 2 * bytes/elem
  static constexpr int K_ROW = DQK * X2 / 2;  // bytes of one K row
  static constexpr int V_ROW = DVO * X2 / 2;
  static constexpr int T = (KVT == KV_BF16 && DQK == 512) ? 32 : 64;  // tokens per tile
  static constexpr int K_SEGS = K_ROW / 128;  // 128-byte swizzle segments per row
  static constexpr int V_SEGS = V_ROW / 128;
  static constexpr int K_TILE = K_SEGS * T * 128;
  static constexpr int V_TILE = V_SEGS * T * 128;
  static constexpr int SFK_ROW = KVT == KV_NVFP4 ? DQK / 16 : 0;
  static constexpr int SFV_ROW = KVT == KV_NVFP4 ? DVO / 16 : 0;
  static constexpr int SFK_TILE = SFK_ROW * T;
  static constexpr int SFV_TILE = SFV_ROW * T;
  static constexpr int STAGE = ((K_TILE + V_TILE + SFK_TILE + SFV_TILE) + 1023) / 1024 * 1024;
  static constexpr int NS_RAW = 196608 / STAGE;
  static constexpr int NS = NS_RAW > 6 ? 6 : NS_RAW;  // ring depth
  static constexpr int ROW_BYTES = K_ROW + V_ROW + SFK_ROW + SFV_ROW;  // per loaded token
  static constexpr int NM = T / 16;          // token m-tiles of QK^T
  static constexpr int NDQ = 8 / NM;         // head-dim slices of QK^T (one per warp group)
  static constexpr int DQW = DQK / NDQ;      // head-dim columns of QK^T per warp
  static constexpr int KSW = DQW / 16;       // k-steps of QK^T per warp
  static constexpr int DVW = DVO / 8;        // output columns per warp
  static constexpr int MTV = DVW / 16;       // m-tiles of (PV)^T per warp
  static_assert(K_ROW % 128 == 0 && V_ROW % 128 == 0, "rows must be whole 128-byte segments");
  static_assert(NS >= 2, "ring too shallow");
};

template <int KVT, int DQK, int DVO, int HP>
struct DecodeSmem {
  using C = DecodeCfg<KVT, DQK, DVO>;
  static constexpr int SRED = C::NDQ * HP * (C::T + 4) * 4;  // fp32 partial scores
  static constexpr int P_STRIDE = C::T + 8;                   // 16-bit elements per P row
  static constexpr int PS = HP * P_STRIDE * 2;
  static constexpr int OFF_SRED = C::NS * C::STAGE;
  static constexpr int OFF_P = OFF_SRED + SRED;
  static constexpr int OFF_ALPHA = OFF_P + PS;
  static constexpr int OFF_ML = OFF_ALPHA + HP * 4;
  static constexpr int OFF_QMAX = OFF_ML + HP * 8;
  static constexpr int OFF_BAR = (OFF_QMAX + 8 * 4 + 7) / 8 * 8;
  static constexpr int BYTES = OFF_BAR + 2 * C::NS * 8;
  static constexpr int ALLOC = BYTES + 1024;  // slack to align the base to 1024 bytes
};

// ----------------------------------------------------------------------------- plan
// Cut the visible page range of every sequence into page-aligned chunks.  With W the
// total visible pages, chunks hold C >= ceil(W / target_chunks) pages (raised towards
// min_chunk_pages, or set by the chunk-size test hook), so the number of chunks never
// exceeds target_chunks + batch (the workspace bound); each sequence's range is then
// split evenly into ceil(pages / C) chunks.
#ifdef PA_DECODE_AUX
__global__ void __launch_bounds__(1024) decode_plan_kernel(DecodeParams p) {
  __shared__ int s_red[32], s_max[32], s_min[32];
  __shared__ int s_carry;
  grid_dep_launch();  // the decode kernel may start its set-up (it waits for this grid)
  const int tid = threadIdx.x;
  const int ps = p.page_size;
  // pass 1: total visible pages, and their largest and smallest count over the sequences
  // that have any
  int mine = 0, pmax = 0, pmin = INT_MAX;
  for (int b = tid; b < p.batch; b += blockDim.x) {
    int np = p.kv_indptr[b + 1] - p.kv_indptr[b];
    if (np <= 0) continue;
    int kv_len = (np - 1) * ps + p.kv_last_page_len[b];
    int first = 0;
    if (p.window_left >= 0) first = max(0, kv_len - 1 - p.window_left) / ps;
    mine += np - first;
    pmax = max(pmax, np - first);
    pmin = min(pmin, np - first);
  }
  for (int o = 16; o > 0; o >>= 1) {
    mine += __shfl_xor_sync(0xffffffffu, mine, o);
    pmax = max(pmax, __shfl_xor_sync(0xffffffffu, pmax, o));
    pmin = min(pmin, __shfl_xor_sync(0xffffffffu, pmin, o));
  }
  if ((tid & 31) == 0) {
    s_red[tid >> 5] = mine;
    s_max[tid >> 5] = pmax;
    s_min[tid >> 5] = pmin;
  }
  __syncthreads();
  if (tid < 32) {
    const bool in = tid < (int)(blockDim.x >> 5);
    int v = in ? s_red[tid] : 0, vmax = in ? s_max[tid] : 0, vmin = in ? s_min[tid] : INT_MAX;
    for (int o = 16; o > 0; o >>= 1) {
      v += __shfl_xor_sync(0xffffffffu, v, o);
      vmax = max(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
      vmin = min(vmin, __shfl_xor_sync(0xffffffffu, vmin, o));
    }
    if (tid == 0) {
      s_red[0] = v;
      s_max[0] = vmax;
      s_min[0] = vmin;
    }
  }
  __syncthreads();
  const int total = s_red[0];
  const bool uniform = s_max[0] > 0 && s_max[0] == s_min[0];  // every sequence the same pages
  int cp = (total + p.target_chunks - 1) / max(1, p.target_chunks);
  if (p.forced_chunk_pages > 0) {
    cp = max(cp, p.forced_chunk_pages);
  } else {
    // a split costs a partial row written and merged: chunks of up to min_chunk_pages
    // (about 4 MiB of K and V per kv head), as long as a quarter of the target number of
    // chunks (about four items per CTA) remains for the balance of the persistent CTAs ...
    const int cap = (int)max(1ll, 4ll * total / max(1, p.target_chunks));
    const int cp_big = max(cp, min(p.min_chunk_pages, cap));
    const long long grid = max(1, p.grid);
    if (cp_big > cp && uniform) {
      // equal sequences give equal items, and the kernel's time is the rounds of items over
      // the CTAs times the item size: the fewest chunks per sequence, between those of
      // cp_big and those of cp, with the least of that product
      const int P = s_max[0];
      const int n_lo = (P + cp_big - 1) / cp_big, n_hi = (P + cp - 1) / cp;
      const long long seq_items = (long long)(total / P) * p.Hkv;  // items per chunk of every sequence
      long long best = LLONG_MAX;
      int best_n = n_hi;
      for (int n = n_lo; n <= n_hi; ++n) {
        const long long t = (seq_items * n + grid - 1) / grid * ((P + n - 1) / n);
        if (t < best) {
          best = t;
          best_n = n;
        }
      }
      cp = (P + best_n - 1) / best_n;
    } else if (cp_big > cp) {
      // ... then the smallest chunks that keep the same number of rounds of items over
      // the CTAs, so the last round is as full as the others
      int n = 0;
      for (int b = tid; b < p.batch; b += blockDim.x) {
        const int np = p.kv_indptr[b + 1] - p.kv_indptr[b];
        if (np <= 0) continue;
        const int kv_len = (np - 1) * ps + p.kv_last_page_len[b];
        const int first = p.window_left >= 0 ? max(0, kv_len - 1 - p.window_left) / ps : 0;
        n += (np - first + cp_big - 1) / cp_big;
      }
      for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
      __syncthreads();
      if ((tid & 31) == 0) s_red[tid >> 5] = n;
      __syncthreads();
      if (tid < 32) {
        int v = (tid < (int)(blockDim.x >> 5)) ? s_red[tid] : 0;
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (tid == 0) s_red[0] = v;
      }
      __syncthreads();
      // (aiming below the full last round by one item per sequence and kv head, since each
      // sequence's chunk count rounds up)
      const long long items = (long long)s_red[0] * p.Hkv;
      const long long rounds = (items + grid - 1) / grid;
      const long long room = max(1ll, rounds * grid - (long long)p.batch * p.Hkv);
      const int cp_fill = (int)min((long long)cp_big, (cp_big * items + room - 1) / room);
      cp = max(cp, cp_fill);
    }
  }
  __syncthreads();
  if (tid == 0) s_carry = 0;
  __syncthreads();
  // pass 2: chunk counts, block-wide exclusive scan in rounds of blockDim.x sequences
  for (int base = 0; base < p.batch; base += blockDim.x) {
    int b = base + tid;
    int np = 0, first = 0, nch = 0;
    if (b < p.batch) {
      np = p.kv_indptr[b + 1] - p.kv_indptr[b];
      if (np > 0) {
        int kv_len = (np - 1) * ps + p.kv_last_page_len[b];
        if (p.window_left >= 0) first = max(0, kv_len - 1 - p.window_left) / ps;
        nch = (np - first + cp - 1) / cp;
      }
    }
    // inclusive warp scan, then across warps
    int v = nch;
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, v, o);
      if ((tid & 31) >= o) v += t;
    }
    if ((tid & 31) == 31) s_red[tid >> 5] = v;
    __syncthreads();
    if (tid < 32) {
      int w = (tid < (int)(blockDim.x >> 5)) ? s_red[tid] : 0;
      for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, w, o);
        if (tid >= o) w += t;
      }
      s_red[tid] = w;  // inclusive prefix over warps
    }
    __syncthreads();
    int excl = s_carry + v - nch + ((tid >> 5) > 0 ? s_red[(tid >> 5) - 1] : 0);
    if (b < p.batch) {
      p.seq_info[b] = make_int2(excl, nch);
      int span = np - first;
      int per = nch > 0 ? (span + nch - 1) / nch : 0;  // even split of this sequence
      for (int k = 0; k < nch; ++k) {
        DecodeChunk c;
        c.b = b;
        c.page_begin = first + k * per;
        c.page_end = min(np, first + (k + 1) * per);
        c.split = k;
        p.chunks[excl + k] = c;
      }
    }
    __syncthreads();
    if (tid == blockDim.x - 1) s_carry = excl + nch;
    __syncthreads();
  }
  if (tid == 0) {
    p.hdr[0] = s_carry;
    p.hdr[1] = cp;
  }
}
#endif  // PA_DECODE_AUX

// The chunk of decode item it: from the planner's list, or (direct calls) the whole
// visible page range of sequence it / Hkv, as the planner would give it in one chunk.
__device__ __forceinline__ DecodeChunk decode_item_chunk(const DecodeParams& p, int it) {
  if (!p.direct) return p.chunks[it / p.Hkv];
  DecodeChunk c;
  c.b = it / p.Hkv;
  c.split = 0;
  const int np = p.kv_indptr[c.b + 1] - p.kv_indptr[c.b];
  int first = 0;
  if (np > 0 && p.window_left >= 0) {
    const int kv_len = (np - 1) * p.page_size + p.kv_last_page_len[c.b];
    first = max(0, kv_len - 1 - p.window_left) / p.page_size;
  }
  c.page_begin = first;
  c.page_end = max(np, 0);
  return c;
}

// ----------------------------------------------------------------------------- merge
// out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s,  lse = ln2 * (M + log2 L).
// One (row, 128-column quarter) unit of the merge, by one warp.
template <int DVO>
__device__ __forceinline__ void decode_merge_unit(const DecodeParams& p, int gw, int lane) {
  constexpr int NQ = DVO / 128;
  const int row = gw / NQ, qc = gw % NQ;
  const int b = row / p.Hq, hq = row % p.Hq;
  const int2 si = p.seq_info[b];
  if (si.y == 1) return;  // the decode kernel wrote this row directly
  uint2* orow = reinterpret_cast<uint2*>(p.out + (size_t)row * DVO + qc * 128) + lane;
  if (si.y == 0) {  // no visible key
    *orow = make_uint2(0, 0);
    if (p.lse && qc == 0 && lane == 0) p.lse[row] = -INFINITY;
    return;
  }
  const float2* ml = p.ws_ml + (size_t)si.x * p.Hq + hq;  // partial s at ml[s * Hq]
  float M = -INFINITY;
  for (int s = lane; s < si.y; s += 32) M = fmaxf(M, ml[(size_t)s * p.Hq].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  const float4* src = reinterpret_cast<const float4*>(p.ws_o + ((size_t)si.x * p.Hq + hq) * DVO + qc * 128) + lane;
  const size_t step = (size_t)p.Hq * DVO / 4;  // float4s between consecutive partials
  for (int s0 = 0; s0 < si.y; s0 += 32) {
    // this lane's partial s0 + lane: weight 2^(m - M) (0 for an empty partial)
    float w = 0.f;
    if (s0 + lane < si.y) {
      const float2 v = ml[(size_t)(s0 + lane) * p.Hq];
      w = v.x == -INFINITY ? 0.f : fast_exp2(v.x - M);
      L += w * v.y;
    }
    const int n = min(32, si.y - s0);
    for (int k0 = 0; k0 < n; k0 += 8) {
      float4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k0 + k < n) v[k] = src[(size_t)(s0 + k0 + k) * step];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float wk = __shfl_sync(0xffffffffu, w, (k0 + k) & 31);
        if (k0 + k < n) {
          acc.x += wk * v[k].x;
          acc.y += wk * v[k].y;
          acc.z += wk * v[k].z;
          acc.w += wk * v[k].w;
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  *orow = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  if (p.lse && qc == 0 && lane == 0) p.lse[row] = (L > 0.f) ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
}

// One warp per (sequence, query head, 128 output columns) unit, the units strided over a
// grid of at most two blocks per SM (most rows were written by the decode kernel itself,
// and a block per few units would cost more to schedule than to run): lane s of the warp
// reads the (m, l) of partial s (32 at a time) and forms its weight once; every lane then
// owns 4 columns and issues the loads of 8 partials before it sums them, so the warp
// waits on L2 once per 8 partials rather than once per partial.
template <int DVO>
__global__ void __launch_bounds__(256) decode_merge_kernel(DecodeParams p) {
  constexpr int NQ = DVO / 128;  // column quarters (warps) per row
  grid_dep_wait();  // the decode kernel's partials are complete
  const int lane = threadIdx.x & 31;
  const int units = p.batch * p.Hq * NQ;
  for (int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; gw < units; gw += (gridDim.x * blockDim.x) >> 5)
    decode_merge_unit<DVO>(p, gw, lane);
}

}  // namespace pa

namespace pa {

// Byte address inside a K or V tile: row t, byte offset bo within the row.  A tile is a
// run of pieces of box_rows = 2^lbr rows (one page, or part of one); each piece is one TMA
// box stored [128-byte segment][row][128 B], SEGS segments per row.  With swizzling the
// 16-byte chunks of a row are permuted by (row & 7), exactly as the 128B-swizzled TMA
// writes them (box_rows is then a multiple of 8, so the row's phase is t & 7).
template <int SEGS>
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int t, int bo, int swz, int lbr) {
  const int piece = t >> lbr, r = t & ((1 << lbr) - 1);
  return base + (uint32_t)(((piece * SEGS + (bo >> 7)) << (lbr + 7)) + r * 128 + ((((bo >> 4) & 7) ^ (t & swz)) << 4));
}

// First of the two consecutive head-dim indices held by B-fragment register `half` of
// k-step `ks` (local to the warp's slice starting at `base`), thread column group `tig`.
// The fp8 / fp4 K fragments come from ldmatrix rows of 16 / 32 head-dim elements, so the
// reduction index is permuted within each group; Q is permuted to match.
template <int KVT>
__device__ __forceinline__ int q_col(int base, int ks, int half, int tig) {
  if constexpr (KVT == KV_BF16) {
    return base + 16 * ks + 2 * tig + 8 * half;
  } else if constexpr (KVT == KV_FP8) {
    return base + 32 * (ks >> 1) + 16 * (ks & 1) + 4 * tig + 2 * half;
  } else {
    return base + 64 * (ks >> 2) + 32 * ((ks >> 1) & 1) + 8 * tig + 4 * (ks & 1) + 2 * half;
  }
}

// Output column of accumulator row-half `half` (0: rows gid, 1: rows gid+8) of (PV)^T
// m-tile `i` of a warp whose columns start at dv0.
template <int KVT>
__device__ __forceinline__ int o_col(int dv0, int i, int half, int gid) {
  if constexpr (KVT == KV_BF16) {
    return dv0 + 16 * i + gid + 8 * half;
  } else if constexpr (KVT == KV_FP8) {
    return dv0 + 32 * (i >> 1) + 16 * (i & 1) + 2 * gid + half;
  } else {
    return dv0 + 64 * (i >> 2) + 32 * ((i >> 1) & 1) + 4 * gid + 2 * (i & 1) + half;
  }
}

__device__ __forceinline__ uint32_t sf_pair_f16x2(uint32_t sf_lo, uint32_t sf_hi) {
  return e4m3x2_to_f16x2(sf_lo | (sf_hi << 8));
}

// (t_a, t_b) pairs of fp4 values at four consecutive head-dim columns, from one
// transposed ldmatrix register (low half: token t_a, 4 nibbles; high half: token t_b).
__device__ __forceinline__ void fp4_vt_pairs(uint32_t r, uint32_t* f) {
  const uint32_t lo = r & 0x0F0F0F0Fu;         // e0 t_a, e2 t_a, e0 t_b, e2 t_b
  const uint32_t hi = (r >> 4) & 0x0F0F0F0Fu;  // e1 t_a, e3 t_a, e1 t_b, e3 t_b
  const uint32_t ta = prmt(lo, hi, 0x5140);    // e0..e3 of t_a
  const uint32_t tb = prmt(lo, hi, 0x7362);    // e0..e3 of t_b
  e2m1x8_to_f16x2x4(ta | (tb << 4), f);        // byte e = (t_a, t_b) at column e
}

template <int KVT, int DQK, int DVO, int HP>
__global__ void __launch_bounds__(288, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_sfk,
                  const __grid_constant__ CUtensorMap tm_sfv, const DecodeParams p) {
  using C = DecodeCfg<KVT, DQK, DVO>;
  using L = DecodeSmem<KVT, DQK, DVO, HP>;
  constexpr int T = C::T, NS = C::NS, NT = HP / 8;
  constexpr bool BF = (KVT == KV_BF16);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* sred = reinterpret_cast<float*>(smem + L::OFF_SRED);
  uint16_t* Ps = reinterpret_cast<uint16_t*>(smem + L::OFF_P);
  float* alpha_s = reinterpret_cast<float*>(smem + L::OFF_ALPHA);
  float2* ml_s = reinterpret_cast<float2*>(smem + L::OFF_ML);
  float* qmax_s = reinterpret_cast<float*>(smem + L::OFF_QMAX);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* empty = full + NS;
  const uint32_t stage0 = smem_u32(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 8);
    }
    fence_mbar_init();
  }
  __syncthreads();
  grid_dep_wait();  // the planner of this call is complete
  const int n_items = p.direct ? p.batch * p.Hkv : p.hdr[0] * p.Hkv;
  const int ps = p.page_size;

  if (warp == 8) {
    // ------------------------------------------------------------------ producer
    if (lane != 0) return;
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    if constexpr (KVT == KV_NVFP4) {
      tma_prefetch_desc(&tm_sfk);
      tma_prefetch_desc(&tm_sfv);
    }
    const int br = p.box_rows;
    uint32_t g = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
      const DecodeChunk ch = decode_item_chunk(p, it);
      const int kvh = it % p.Hkv;
      const int ip0 = p.kv_indptr[ch.b];
      const int np = p.kv_indptr[ch.b + 1] - ip0;
      const int kv_len = (np - 1) * ps + p.kv_last_page_len[ch.b];
      const int tok_end = min(ch.page_end * ps, kv_len);
      const int load_cap = ch.page_end * ps;
      for (int tok0 = ch.page_begin * ps; tok0 < tok_end; tok0 += T, ++g) {
        const int s = g % NS;
        mbar_wait(&empty[s], ((g / NS) & 1) ^ 1, p.err, SITE_DEC_EMPTY);
        const int pieces = (min(tok0 + T, load_cap) - tok0 + br - 1) / br;
        mbar_arrive_expect_tx(&full[s], (uint32_t)(pieces * br * C::ROW_BYTES));
        const uint32_t kbase = stage0 + s * C::STAGE;
        const uint32_t vbase = kbase + C::K_TILE;
        const uint32_t sfkbase = vbase + C::V_TILE;
        const uint32_t sfvbase = sfkbase + C::SFK_TILE;
        for (int k = 0; k < pieces; ++k) {
          const int tok = tok0 + k * br;
          const int page = p.kv_indices[ip0 + tok / ps];
          const int row = kvh * ps + tok % ps;
          // the piece's rows of every 128-byte segment in one box ([segment][row][128 B])
          tma_load_4d(kbase + k * br * C::K_ROW, &tm_k, 0, row, 0, page, &full[s]);
          tma_load_4d(vbase + k * br * C::V_ROW, &tm_v, 0, row, 0, page, &full[s]);
          if constexpr (KVT == KV_NVFP4) {
            tma_load_3d(sfkbase + k * br * C::SFK_ROW, &tm_sfk, 0, row, page, &full[s]);
            tma_load_3d(sfvbase + k * br * C::SFV_ROW, &tm_sfv, 0, row, page, &full[s]);
          }
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------------- consumers
  const int cw = warp;  // 0..7
  const int gid = lane >> 2, tig = lane & 3;
  const int mat = lane >> 3, mr = lane & 7;  // ldmatrix: matrix and row this lane addresses
  const int mt = cw % C::NM, dq = cw / C::NM;
  const int dqk0 = dq * C::DQW;  // QK^T head-dim slice of this warp
  const int dv0 = cw * C::DVW;   // output columns of this warp
  const int swz = p.swz;
  const int lbr = p.box_shift;
  const int gsz = p.group;
  const float kscale = BF ? 1.f : __ldg(p.k_scale);
  const float vscale = BF ? 1.f : __ldg(p.v_scale);
  constexpr int PST = L::P_STRIDE;
  uint32_t g = 0;

  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const DecodeChunk ch = decode_item_chunk(p, it);
    const int kvh = it % p.Hkv;
    const int b = ch.b;
    const int ip0 = p.kv_indptr[b];
    const int np = p.kv_indptr[b + 1] - ip0;
    const int kv_len = (np - 1) * ps + p.kv_last_page_len[b];
    const int tok_begin = ch.page_begin * ps;
    const int tok_end = min(ch.page_end * ps, kv_len);
    const int win_lo = p.window_left >= 0 ? kv_len - 1 - p.window_left : 0;

    // ---- Q as MMA B fragments (bf16 pairs; the fp8 / fp4 paths convert them to f16)
    uint32_t qf[C::KSW][NT][2];
    const uint16_t* qbase = p.q + ((size_t)b * p.Hq + (size_t)kvh * gsz) * DQK;
#pragma unroll
    for (int ks = 0; ks < C::KSW; ++ks)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int h = nt * 8 + gid;
          uint32_t v = 0;
          if (h < gsz)
            v = __ldg(reinterpret_cast<const uint32_t*>(qbase + (size_t)h * DQK +
                                                        q_col<KVT>(dqk0, ks, hf, tig)));
          qf[ks][nt][hf] = v;
        }
    float sm_log2 = p.sm_scale * 1.4426950408889634f * kscale;
    if constexpr (!BF) {
      // f16 MMAs: scale q by a power of two so max|q| lands in [2^14, 2^15) (exact for
      // every bf16 value that stays in the f16 normal range), undo it in the score scale.
      float mx = 0.f;
#pragma unroll
      for (int ks = 0; ks < C::KSW; ++ks)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const uint32_t v = qf[ks][nt][hf];
            mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(v << 16)), fabsf(__uint_as_float(v & 0xFFFF0000u))));
          }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (lane == 0) qmax_s[cw] = mx;
      named_bar_sync(1, 256);
      float m8 = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) m8 = fmaxf(m8, qmax_s[w]);
      int ex = 0;
      if (m8 > 0.f) {
        int x;
        frexpf(m8, &x);
        ex = 15 - x;
      }
      const float qs = ldexpf(1.f, ex);
      sm_log2 *= ldexpf(1.f, -ex);
#pragma unroll
      for (int ks = 0; ks < C::KSW; ++ks)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const uint32_t v = qf[ks][nt][hf];
            qf[ks][nt][hf] = pack_f16x2(__uint_as_float(v << 16) * qs, __uint_as_float(v & 0xFFFF0000u) * qs);
          }
    }

    float o[C::MTV][NT][4];
#pragma unroll
    for (int i = 0; i < C::MTV; ++i)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[i][nt][e] = 0.f;
    float m_run[NT], l_run[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      m_run[j] = -INFINITY;
      l_run[j] = 0.f;
    }

    const int n_tiles = (tok_end - tok_begin + T - 1) / T;
    for (int ti = 0; ti < n_tiles; ++ti, ++g) {
      const int s = g % NS;
      const int tok0 = tok_begin + ti * T;
      const int n_valid = min(T, tok_end - tok0);
      uint8_t* kp = smem + s * C::STAGE;
      const uint32_t kbase = stage0 + s * C::STAGE;
      const uint32_t vbase = kbase + C::K_TILE;
      const uint8_t* sfk = kp + C::K_TILE + C::V_TILE;
      const uint8_t* sfv = sfk + C::SFK_TILE;
      mbar_wait(&full[s], (g / NS) & 1, p.err, SITE_DEC_FULL);
      __syncwarp();  // ldmatrix / mma.sync below are warp-collective
      if (n_valid < T) {
        // rows past the end of the chunk hold stale or unused-slot bytes: zero the V rows
        // (and their scales) so that P = 0 never meets a NaN
        uint8_t* vp = kp + C::K_TILE;
        const int nrow = T - n_valid;
        for (int idx = threadIdx.x; idx < nrow * C::V_SEGS * 8; idx += 256) {
          const int r = n_valid + idx / (C::V_SEGS * 8);
          const int rem = idx % (C::V_SEGS * 8);
          *reinterpret_cast<uint4*>(vp + ((((r >> lbr) * C::V_SEGS + (rem >> 3)) << (lbr + 7)) +
                                          (r & ((1 << lbr) - 1)) * 128 + (rem & 7) * 16)) = make_uint4(0, 0, 0, 0);
        }
        if constexpr (KVT == KV_NVFP4) {
          uint8_t* sv = kp + C::K_TILE + C::V_TILE + C::SFK_TILE;
          for (int idx = threadIdx.x; idx < nrow * (C::SFV_ROW / 16); idx += 256)
            *reinterpret_cast<uint4*>(sv + n_valid * C::SFV_ROW + idx * 16) = make_uint4(0, 0, 0, 0);
        }
      }

      // ---- S^T = K q^T over this warp's head-dim slice (rows: 16 tokens, cols: heads)
      float sacc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
      const int t0 = mt * 16;
      if constexpr (KVT == KV_BF16) {
#pragma unroll
        for (int ks = 0; ks < C::KSW; ++ks) {
          uint32_t a0, a1, a2, a3;
          const int t = t0 + mr + 8 * (mat & 1);
          const int d = dqk0 + 16 * ks + 8 * (mat >> 1);
          ldsm_x4(tile_addr<C::K_SEGS>(kbase, t, 2 * d, swz, lbr), a0, a1, a2, a3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma16816<true>(sacc[nt], a0, a1, a2, a3, qf[ks][nt][0], qf[ks][nt][1]);
        }
      } else if constexpr (KVT == KV_FP8) {
#pragma unroll
        for (int kg = 0; kg < C::KSW / 2; ++kg) {
          uint32_t R[4];
          const int t = t0 + mr + 8 * (mat & 1);
          const int d = dqk0 + 32 * kg + 16 * (mat >> 1);
          ldsm_x4(tile_addr<C::K_SEGS>(kbase, t, d, swz, lbr), R[0], R[1], R[2], R[3]);
#pragma unroll
          for (int sub = 0; sub < 2; ++sub) {
            const uint32_t ra = R[2 * sub], rb = R[2 * sub + 1];
            const uint32_t a0 = e4m3x2_to_f16x2(ra & 0xFFFFu), a2 = e4m3x2_to_f16x2(ra >> 16);
            const uint32_t a1 = e4m3x2_to_f16x2(rb & 0xFFFFu), a3 = e4m3x2_to_f16x2(rb >> 16);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma16816<false>(sacc[nt], a0, a1, a2, a3, qf[2 * kg + sub][nt][0], qf[2 * kg + sub][nt][1]);
          }
        }
      } else {
#pragma unroll
        for (int kg = 0; kg < C::KSW / 4; ++kg) {
          uint32_t R[4];
          const int t = t0 + mr + 8 * (mat & 1);
          const int d = dqk0 + 64 * kg + 32 * (mat >> 1);
          ldsm_x4(tile_addr<C::K_SEGS>(kbase, t, d >> 1, swz, lbr), R[0], R[1], R[2], R[3]);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {  // head-dim halves: +0 (R0, R1), +32 (R2, R3)
            const int blk = (dqk0 + 64 * kg + 32 * hh + 8 * tig) >> 4;
            const uint32_t sa = sfk[(t0 + gid) * C::SFK_ROW + blk];
            const uint32_t sb = sfk[(t0 + 8 + gid) * C::SFK_ROW + blk];
            const uint32_t sfa = sf_pair_f16x2(sa, sa), sfb = sf_pair_f16x2(sb, sb);
            uint32_t fa[4], fb[4];
            e2m1x8_to_f16x2x4(R[2 * hh], fa);
            e2m1x8_to_f16x2x4(R[2 * hh + 1], fb);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              fa[j] = hmul2_u32(fa[j], sfa);
              fb[j] = hmul2_u32(fb[j], sfb);
            }
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
              const int ks = 4 * kg + 2 * hh + sub;
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma16816<false>(sacc[nt], fa[2 * sub], fb[2 * sub], fa[2 * sub + 1], fb[2 * sub + 1],
                                qf[ks][nt][0], qf[ks][nt][1]);
            }
          }
        }
      }
      {
        float* sr = sred + dq * HP * (T + 4);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int h0 = nt * 8 + 2 * tig;
          sr[h0 * (T + 4) + t0 + gid] = sacc[nt][0];
          sr[(h0 + 1) * (T + 4) + t0 + gid] = sacc[nt][1];
          sr[h0 * (T + 4) + t0 + 8 + gid] = sacc[nt][2];
          sr[(h0 + 1) * (T + 4) + t0 + 8 + gid] = sacc[nt][3];
        }
      }
      named_bar_sync(1, 256);

      // ---- online softmax: warp cw owns heads cw + 8j, lanes own tokens
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int h = cw + 8 * j;
        float x[T / 32];
        float tmax = -INFINITY;
#pragma unroll
        for (int k = 0; k < T / 32; ++k) {
          const int t = lane + 32 * k;
          float sv = 0.f;
#pragma unroll
          for (int q = 0; q < C::NDQ; ++q) sv += sred[(q * HP + h) * (T + 4) + t];
          const bool ok = (t < n_valid) && (tok0 + t >= win_lo);
          x[k] = ok ? sv * sm_log2 : -INFINITY;
          tmax = fmaxf(tmax, x[k]);
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o2));
        const float m_new = fmaxf(m_run[j], tmax);
        const float base = (m_new == -INFINITY) ? 0.f : m_new;
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < T / 32; ++k) {
          const float pv = fast_exp2(x[k] - base);
          sum += pv;
          uint16_t bits;
          if constexpr (BF) bits = __bfloat16_as_ushort(__float2bfloat16_rn(pv));
          else bits = __half_as_ushort(__float2half_rn(pv));
          Ps[h * PST + lane + 32 * k] = bits;
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o2);
        const float alpha = fast_exp2(m_run[j] - base);
        l_run[j] = l_run[j] * alpha + sum;
        m_run[j] = m_new;
        if (lane == 0) {
          alpha_s[h] = alpha;
          ml_s[h] = make_float2(m_new, l_run[j]);
        }
      }
      named_bar_sync(1, 256);

      // ---- (O^T) = alpha * (O^T) + V^T P^T over this warp's output columns
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float al0 = alpha_s[nt * 8 + 2 * tig], al1 = alpha_s[nt * 8 + 2 * tig + 1];
#pragma unroll
        for (int i = 0; i < C::MTV; ++i) {
          o[i][nt][0] *= al0;
          o[i][nt][1] *= al1;
          o[i][nt][2] *= al0;
          o[i][nt][3] *= al1;
        }
      }
#pragma unroll
      for (int kk = 0; kk < T / 16; ++kk) {
        const int tb = kk * 16;
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint16_t* prow = Ps + (nt * 8 + gid) * PST + tb + 2 * tig;
          pb[nt][0] = *reinterpret_cast<const uint32_t*>(prow);
          pb[nt][1] = *reinterpret_cast<const uint32_t*>(prow + 8);
        }
        if constexpr (KVT == KV_BF16) {
#pragma unroll
          for (int i = 0; i < C::MTV; ++i) {
            uint32_t a0, a1, a2, a3;
            const int t = tb + mr + 8 * (mat >> 1);
            const int d = dv0 + 16 * i + 8 * (mat & 1);
            ldsm_x4_t(tile_addr<C::V_SEGS>(vbase, t, 2 * d, swz, lbr), a0, a1, a2, a3);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma16816<true>(o[i][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
          }
        } else if constexpr (KVT == KV_FP8) {
#pragma unroll
          for (int ip = 0; ip < C::MTV / 2; ++ip) {
            uint32_t R[4];
            const int t = tb + mr + 8 * (mat & 1);
            const int d = dv0 + 32 * ip + 16 * (mat >> 1);
            ldsm_x4_t(tile_addr<C::V_SEGS>(vbase, t, d, swz, lbr), R[0], R[1], R[2], R[3]);
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
              const uint32_t ra = R[2 * sub], rb = R[2 * sub + 1];
              const uint32_t a0 = e4m3x2_to_f16x2(prmt(ra, 0, 0x20)), a1 = e4m3x2_to_f16x2(prmt(ra, 0, 0x31));
              const uint32_t a2 = e4m3x2_to_f16x2(prmt(rb, 0, 0x20)), a3 = e4m3x2_to_f16x2(prmt(rb, 0, 0x31));
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma16816<false>(o[2 * ip + sub][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
            }
          }
        } else {
          uint32_t R[4];
          const int t = tb + mr + 8 * (mat & 1);
          const int d = dv0 + 32 * (mat >> 1);
          if constexpr (C::DVW == 64) {
            ldsm_x4_t(tile_addr<C::V_SEGS>(vbase, t, d >> 1, swz, lbr), R[0], R[1], R[2], R[3]);
          } else {
            ldsm_x2_t(tile_addr<C::V_SEGS>(vbase, t, (dv0 >> 1), swz, lbr), R[0], R[1]);
            R[2] = R[3] = 0;
          }
#pragma unroll
          for (int hh = 0; hh < C::DVW / 32; ++hh) {
            const int blk = (dv0 + 32 * hh + 4 * gid) >> 4;
            const int ta = tb + 2 * tig;
            const uint32_t s0 = sf_pair_f16x2(sfv[ta * C::SFV_ROW + blk], sfv[(ta + 1) * C::SFV_ROW + blk]);
            const uint32_t s1 = sf_pair_f16x2(sfv[(ta + 8) * C::SFV_ROW + blk], sfv[(ta + 9) * C::SFV_ROW + blk]);
            uint32_t f0[4], f1[4];
            fp4_vt_pairs(R[2 * hh], f0);
            fp4_vt_pairs(R[2 * hh + 1], f1);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              f0[j] = hmul2_u32(f0[j], s0);
              f1[j] = hmul2_u32(f1[j], s1);
            }
#pragma unroll
            for (int sub = 0; sub < 2; ++sub)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma16816<false>(o[2 * hh + sub][nt], f0[2 * sub], f0[2 * sub + 1], f1[2 * sub], f1[2 * sub + 1],
                                pb[nt][0], pb[nt][1]);
          }
        }
      }
      if (n_valid < T) fence_proxy_async_smem();  // zeroed rows -> next TMA write
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ---- epilogue: the final row (single chunk) or a partial (O, m, l)
    // (a direct item without a visible key wrote no (m, l): its row is 0, its lse -inf)
    const int2 si = p.direct ? make_int2(0, 1) : p.seq_info[b];
    const bool direct = (si.y == 1);
    const bool keys = n_tiles > 0;
    const size_t prow = (size_t)(si.x + ch.split);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int h = nt * 8 + 2 * tig + c;
        if (h >= gsz) continue;
        const int hq = kvh * gsz + h;
        const float2 ml = keys ? ml_s[h] : make_float2(-INFINITY, 0.f);
        if (direct) {
          const float inv = ml.y > 0.f ? vscale / ml.y : 0.f;
          uint16_t* orow = p.out + ((size_t)b * p.Hq + hq) * DVO;
#pragma unroll
          for (int i = 0; i < C::MTV; ++i)
#pragma unroll
            for (int r = 0; r < 2; ++r)
              orow[o_col<KVT>(dv0, i, r, gid)] = __bfloat16_as_ushort(__float2bfloat16_rn(o[i][nt][2 * r + c] * inv));
        } else {
          float* dst = p.ws_o + (prow * p.Hq + hq) * DVO;
#pragma unroll
          for (int i = 0; i < C::MTV; ++i)
#pragma unroll
            for (int r = 0; r < 2; ++r) dst[o_col<KVT>(dv0, i, r, gid)] = o[i][nt][2 * r + c] * vscale;
        }
      }
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int h = cw + 8 * j;
        if (h >= gsz) continue;
        const int hq = kvh * gsz + h;
        const float2 ml = keys ? ml_s[h] : make_float2(-INFINITY, 0.f);
        if (direct) {
          if (p.lse)
            p.lse[(size_t)b * p.Hq + hq] = ml.y > 0.f ? (ml.x + log2f(ml.y)) * 0.69314718055994531f : -INFINITY;
        } else {
          p.ws_ml[prow * p.Hq + hq] = ml;
        }
      }
    }
  }
}

}  // namespace pa

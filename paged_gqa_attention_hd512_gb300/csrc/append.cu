// append.cu -- write new tokens' K and V into the paged cache, converting them to the
// cache's element type on the way (quantise-on-write).
//
// The step before attention: the pages' NVFP4 prefill is validated on caches written by
// an in-tree NVFP4 KV quantisation kernel from bf16 sources ("feat(attention): asymmetric
// VO-split NVFP4 paged prefill (qk=512/vo=256) for Gemma-4 on SM120/121", commit
// "support-or-reject-explicitly" notes), and FP8 KV is a per-tensor-scaled e4m3 cache
// that the attention kernels cast on load ("[None][feat] Run Gemma4 head_dim 512
// attention on Triton", Approach).  Element formats and page layout are those the
// attention calls read:
//   bf16   copied;
//   FP8    code = e4m3(x / scale), round to nearest even, saturating at +-448;
//   NVFP4  per 16 consecutive head-dim elements of one token and head:
//          sf = e4m3((amax / 6) / global), d = value(sf) * global,
//          code = e2m1(x / d) (nearest even, saturating at +-6), or 0 when d is 0;
//          two codes per byte, element 2i in the low nibble.
// A code carries the sign of its operand, also when the magnitude rounds to zero.
// Every operation is a correctly rounded fp32 operation in this order, so the codes are
// a function of the inputs alone.
//
// A warp writes one to four consecutive new tokens, eight warps per CTA; each lane converts
// 16-element units (32 bytes of bf16), so a warp reads 1 KB of consecutive input at a time.
#include "launch.h"
#include "common.cuh"

namespace pa {

namespace {

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// two fp32 -> two e4m3 codes (low byte: a), RNE, saturating
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}
// two fp32 -> one byte of e2m1 codes (low nibble: a), RNE, saturating
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float a, float b) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(b), "f"(a));
  return r;
}
// one e4m3 code with the sign of v (also for a magnitude that rounds to zero), RNE and
// saturating
__device__ __forceinline__ uint32_t e4m3_code(float v) {
  return (f32x2_to_e4m3x2(fabsf(v), 0.f) & 0x7Fu) | ((__float_as_uint(v) >> 24) & 0x80u);
}
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  const uint32_t h2 = e4m3x2_to_f16x2(code & 0xFFu);
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// a / b rounded to nearest even, from y = RN(1/b): the estimate a*y (within two units in
// the last place of a/b) corrected twice by exact FMA residuals.  Markstein's theorem (P.
// Markstein, "Computation of elementary functions on the IBM RISC System/6000 processor",
// IBM J. Res. Develop. 34, 1990): with y the correctly rounded reciprocal of b and q within
// one unit in the last place of a/b, RN(q + (a - b q) y) is the correctly rounded a/b; the
// first correction brings the estimate within that unit.  It holds while a, b, y and the
// quotient stay in the normal range and finite; callers take the IEEE division otherwise.
// Below the normal range the result keeps the sign and stays below it, which is all a
// code of e4m3 or e2m1 (whose smallest step is far above it) depends on there.
// The corrections turn a zero quotient into +0 (the residual of -0 is +0), so the result
// takes the sign of the first estimate, which is the sign of a/b (also when it rounds to
// zero).
__device__ __forceinline__ float quot_recip(float a, float b, float y) {
  const float q0 = __fmul_rn(a, y);
  const float q1 = __fmaf_rn(__fmaf_rn(-q0, b, a), y, q0);
  return copysignf(__fmaf_rn(__fmaf_rn(-q1, b, a), y, q1), q0);
}
// |b| in the range where b, 1/b and quotients of bounded magnitude stay normal
__device__ __forceinline__ bool recip_ok(float b) { return fabsf(b) >= 0x1p-100f && fabsf(b) <= 0x1p100f; }

constexpr int kAppendWarps = 8;  // warps per CTA

// Each warp writes `tokens` consecutive new tokens (one after the other), so the search
// for the token's sequence, the scales and their reciprocals are found once for several.
template <int KVT>
__global__ void __launch_bounds__(32 * kAppendWarps) append_kv_kernel(const AppendParams p, const int tokens) {
  const int lane = threadIdx.x & 31;
  const int i_first = (blockIdx.x * kAppendWarps + (threadIdx.x >> 5)) * tokens;
  if (i_first >= p.total_new) return;
  const int i_end = min(i_first + tokens, p.total_new);
  const int ku = p.d_qk / 16, vu = p.d_vo / 16, kvu = ku + vu, units = p.Hkv * kvu;
  // element widths in bytes x2: bf16 4, fp8 2, nvfp4 1
  constexpr int X2 = KVT == KV_BF16 ? 4 : (KVT == KV_FP8 ? 2 : 1);
  // offsets inside one page in 32 bits (the host bounds a page below 2^31 bytes)
  const uint32_t rows = (uint32_t)p.Hkv * p.page_size;
  const uint32_t k_row = (uint32_t)p.d_qk * X2 / 2, v_row = (uint32_t)p.d_vo * X2 / 2;
  float ks = 1.f, vs = 1.f;
  if (KVT != KV_BF16) {
    ks = __ldg(p.k_scale);
    vs = __ldg(p.v_scale);
  }
  // FP8: the reciprocal of each per-tensor scale, and the largest |x| below which x / scale
  // stays under 2^100 (0: always the IEEE division)
  const float yk = __frcp_rn(ks), yv = __frcp_rn(vs);
  const float lim_k = recip_ok(ks) ? fminf(0x1p100f * fabsf(ks), 0x1p100f) : 0.f;
  const float lim_v = recip_ok(vs) ? fminf(0x1p100f * fabsf(vs), 0x1p100f) : 0.f;
  // unit u of a token is unit w of kv head h (h = u / kvu, w = u % kvu; a head's K units
  // first, then its V units); a lane's units are 32 apart, so (h, w) advances by adding 32
  // to w and carrying whole heads, without a division per unit
  auto carry = [&](int& h, int& w) {
    while (w >= kvu) {
      w -= kvu;
      ++h;
    }
  };
  int b = 0, a0 = 0, a_end = 0, ip0 = 0, kv_len = 0;  // the current token's sequence
  for (int i = i_first; i < i_end; ++i) {
    if (i == i_first || i >= a_end) {
      // the last sequence b with append_indptr[b] <= i, 32 candidates per round (a chain
      // of dependent loads is what a token's work waits on, so it is kept to a few
      // rounds), from the previous token's sequence on
      int lo = i == i_first ? 0 : min(b + 1, p.batch - 1);
      int hi = p.batch;  // append_indptr[lo] <= i, and i < append_indptr[hi] unless hi == batch
      while (hi - lo > 1) {
        const int step = (hi - lo + 31) / 32;
        const int c = lo + step * lane;
        const bool le = lane > 0 && c < hi && __ldg(p.append_indptr + c) <= i;
        const unsigned m = __ballot_sync(0xffffffffu, le);
        if (m) lo += step * (31 - __clz(m));
        hi = min(hi, lo + step);
      }
      b = lo;
      a0 = __ldg(p.append_indptr + b);
      a_end = __ldg(p.append_indptr + b + 1);
      ip0 = __ldg(p.kv_indptr + b);
      const int np = __ldg(p.kv_indptr + b + 1) - ip0;
      kv_len = np > 0 ? (np - 1) * p.page_size + __ldg(p.kv_last_page_len + b) : 0;
    }
    const int t = kv_len - (a_end - a0) + (i - a0);  // position in the sequence
    int page = -1;
    if (t >= 0 && t < kv_len) page = __ldg(p.kv_indices + ip0 + t / p.page_size);
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0) record_error(p.err, SITE_APPEND_POS);
      continue;
    }
    const int slot = t % p.page_size;
    uint8_t* page_base = p.cache + (size_t)page * rows * (k_row + v_row);
    uint8_t* sf_base = KVT == KV_NVFP4 ? p.sf + (size_t)page * rows * kvu : nullptr;
    const uint16_t* k_tok = p.k_new + (size_t)i * p.Hkv * p.d_qk;
    const uint16_t* v_tok = p.v_new + (size_t)i * p.Hkv * p.d_vo;
    // the 32 input bytes of unit w of kv head h
    auto src_of = [&](int h, int w) -> const uint4* {
      return reinterpret_cast<const uint4*>(w < ku ? k_tok + (h * p.d_qk + w * 16) : v_tok + (h * p.d_vo + (w - ku) * 16));
    };
    int h = 0, w = lane;
    carry(h, w);
    // each lane's next unit is loaded before the current one is converted, so two units'
    // loads of each warp are in flight (the kernel waits on memory latency otherwise)
    uint4 a_n = make_uint4(0, 0, 0, 0), c_n = a_n;
    if (lane < units) {
      a_n = __ldg(src_of(h, w));
      c_n = __ldg(src_of(h, w) + 1);
    }
    for (int u = lane; u < units; u += 32) {
      const bool is_k = w < ku;
      const int blk = is_k ? w : w - ku;
      int hn = h, wn = w + 32;
      carry(hn, wn);
      const uint4 a = a_n, c = c_n;
      if (u + 32 < units) {
        a_n = __ldg(src_of(hn, wn));
        c_n = __ldg(src_of(hn, wn) + 1);
      }
      const uint32_t row = (uint32_t)h * p.page_size + slot;
      uint8_t* dst = page_base + (is_k ? row * k_row : rows * k_row + row * v_row) + (uint32_t)blk * 16 * X2 / 2;
      if constexpr (KVT == KV_BF16) {
        reinterpret_cast<uint4*>(dst)[0] = a;
        reinterpret_cast<uint4*>(dst)[1] = c;
      } else {
        const uint32_t wv[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
        float x[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          x[2 * k] = bf16_to_f32(wv[k] & 0xFFFFu);
          x[2 * k + 1] = bf16_to_f32(wv[k] >> 16);
        }
        const float scale = is_k ? ks : vs;
        if constexpr (KVT == KV_FP8) {
          // two codes per conversion (the conversion keeps the operand's sign, also on a
          // magnitude that rounds to zero).  The unit's largest magnitude (bf16 bits, NaN
          // above infinity) decides between the reciprocal form and the IEEE division.
          uint32_t mb = 0u;
#pragma unroll
          for (int k = 0; k < 8; ++k) mb = __vmaxu2(mb, wv[k] & 0x7FFF7FFFu);
          const float amax = bf16_to_f32(max(mb & 0xFFFFu, mb >> 16));
          uint32_t o[4] = {0u, 0u, 0u, 0u};
          if (amax < (is_k ? lim_k : lim_v)) {
            const float y = is_k ? yk : yv;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              o[k >> 1] |= f32x2_to_e4m3x2(quot_recip(x[2 * k], scale, y), quot_recip(x[2 * k + 1], scale, y))
                           << (16 * (k & 1));
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              o[k >> 1] |= f32x2_to_e4m3x2(__fdiv_rn(x[2 * k], scale), __fdiv_rn(x[2 * k + 1], scale)) << (16 * (k & 1));
          }
          *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
          float amax = 0.f;
#pragma unroll
          for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(x[k]));
          const uint32_t sf_code = e4m3_code(__fdiv_rn(__fdiv_rn(amax, 6.f), scale));
          const float d = __fmul_rn(e4m3_to_f32(sf_code), scale);
          uint32_t o[2] = {0u, 0u};
          if (d != 0.f) {
            // |x / d| <= amax / d, about 6 unless the block scale saturated at the e4m3
            // maximum: the reciprocal form while d is in range and amax / d <= 2^100
            if (recip_ok(d) && amax <= fminf(0x1p100f, 0x1p100f * fabsf(d))) {
              const float y = __frcp_rn(d);
#pragma unroll
              for (int k = 0; k < 8; ++k)
                o[k >> 2] |= f32x2_to_e2m1x2(quot_recip(x[2 * k], d, y), quot_recip(x[2 * k + 1], d, y)) << (8 * (k & 3));
            } else {
#pragma unroll
              for (int k = 0; k < 8; ++k)
                o[k >> 2] |= f32x2_to_e2m1x2(__fdiv_rn(x[2 * k], d), __fdiv_rn(x[2 * k + 1], d)) << (8 * (k & 3));
            }
          }
          *reinterpret_cast<uint2*>(dst) = make_uint2(o[0], o[1]);
          sf_base[(is_k ? row * ku : rows * ku + row * vu) + blk] = (uint8_t)sf_code;
        }
      }
      h = hn;
      w = wn;
    }
  }
}

}  // namespace

cudaError_t launch_append_kv(int kvt, const AppendParams& p, int sms, cudaStream_t s) {
  if (p.total_new == 0) return cudaSuccess;
  // 4 (or 2) tokens a warp while that still leaves at least 32 warps for every SM (4
  // resident CTAs of 8), else one: a short append (a decode step's) keeps its parallelism
  int tokens = 1;
  while (tokens < 4 && (long long)p.total_new >= 2ll * tokens * 32 * sms) tokens *= 2;
  const long long warps = (p.total_new + tokens - 1) / tokens;
  const int grid = (int)((warps + kAppendWarps - 1) / kAppendWarps), threads = 32 * kAppendWarps;
  if (kvt == KV_BF16) append_kv_kernel<KV_BF16><<<grid, threads, 0, s>>>(p, tokens);
  else if (kvt == KV_FP8) append_kv_kernel<KV_FP8><<<grid, threads, 0, s>>>(p, tokens);
  else if (kvt == KV_NVFP4) append_kv_kernel<KV_NVFP4><<<grid, threads, 0, s>>>(p, tokens);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace pa

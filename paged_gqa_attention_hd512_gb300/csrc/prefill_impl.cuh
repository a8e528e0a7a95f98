// prefill_impl.cuh -- causal paged prefill at head_dim 512 with tcgen05 MMAs (sm_103a).
//
// Attention of the new tokens of each sequence over its paged KV ("Run Gemma4 head_dim 512
// attention on Triton", Approach: prefill over the HND paged layout, causal when no custom
// mask is given; "feat(attention): asymmetric VO-split NVFP4 paged prefill (qk=512/vo=256)
// for Gemma-4 on SM120/121", Summary: head_dim_qk 512 with head_dim_vo 256, VO split).
//
// One CTA per SM (persistent).  A work item is 128 query rows = P positions x g heads of
// one kv head (P = 128 / g), so every K/V tile loaded into shared memory serves all g
// query heads that read it.  Warp roles:
//   warp 0      producer: TMA loads of the Q tile (once per item) and, for bf16 KV, of K/V
//               chunks ([128 keys][128 head-dim], two 128B-swizzled 16 KB blocks) into a
//               ring of 32 KB slots (V rows past the end of the sequence are zeroed before
//               release); for FP8 / NVFP4 KV converted in the kernel, of the packed chunks
//               and block scales into staging rings
//   warp 1      MMA issuer (lane 0 issues): S = Q K^T into TMEM (M 128, N 128, K 16
//               steps), O += P V with P read from TMEM (M 128, N 128 per V chunk)
//   warp 2      gate: polls the mbarriers and meets the MMA warp at named barriers
//   warp 3      (head_dim_vo 512, bf16) the first pass's P tiles into the P slots
//   warps 4-11  softmax + epilogue (two warpgroups, half of the keys each; warps 4-7 alone
//               when 8-11 convert FP8 / NVFP4): thread r owns row r (TMEM lane r): causal,
//               window and custom masks, online softmax in base 2 with lazy rescaling, P
//               into TMEM, at the end O / l as bf16 rows and lse (or, for a chunk of a
//               split KV range, fp32 rows and lse into a partial slot)
//   warps 8-11  (FP8 / NVFP4 KV converted in the kernel) converters: staged chunks -> ring
// TMEM (512 columns): two S buffers [0, 128) and [128, 256), used by alternate KV steps,
// each holding its step's P once the softmax has read S, and O [256, 512).  With two S
// buffers the QK of the next step runs while the softmax works on this one.  A 128 x 512
// fp32 O tile would fill all of TMEM, so head_dim_vo 512 is computed in two passes of 256
// columns over the same KV range: the second reads the first pass's P tiles back from a
// per-CTA scratch (items of up to 64 KV tiles) or recomputes S (longer items).
// With PAIR, two CTAs of a cluster share every MMA (cta_group::2, M 256), each loading
// half of every K/V tile (see PrefillCfg).
#pragma once

#include "common.cuh"
#include "tc_helpers.cuh"

namespace pa {

template <int DQK, int DVO, int KVT, bool PAIR_ = false>
struct PrefillCfg {
  // PAIR: two CTAs (a cluster) share every MMA (tcgen05 cta_group::2, M = 256): each holds
  // its own 128 query rows and loads half of every K/V tile, so the pair reads each K/V
  // byte once instead of twice and each SM takes in half the K/V bytes per MMA cycle
  static constexpr bool PAIR = PAIR_;
  static constexpr int CL = PAIR ? 2 : 1;       // CTAs per MMA
  static constexpr int M = 128;                 // query rows per tile
  static constexpr int N = 128;                 // keys per KV tile
  static constexpr int HALF = N * 128;          // one [128 keys][64 dims] bf16 block (16 KB)
  static constexpr int CHUNK = 2 * HALF;        // one ring slot: [128 keys][128 dims], two blocks
  static constexpr int NQB = DQK / 64;          // Q blocks of 64 head-dim columns
  static constexpr int NQC = DQK / 128;         // K chunks per step (8 QK MMAs each)
  static constexpr int DVP = DVO > 256 ? 256 : DVO;  // output columns per pass
  static constexpr int NPASS = DVO / DVP;
  static constexpr int NVC = DVP / 128;         // V chunks per pass (one N=128 PV group each)
  // PAIR: a K chunk is this CTA's 64 keys x 256 dims (four [64 keys][64 dims] 128B-swizzled
  // blocks of 8 KB), a V chunk this CTA's 128 of the pass's 256 output columns
  static constexpr int KBLK = 64 * 128;
  static constexpr int NKC = PAIR ? DQK / 256 : NQC;  // K chunks per step
  static constexpr int NVS_P = PAIR ? 1 : NVC;         // V chunks per step
  static constexpr int Q_BYTES = NQB * HALF;
  static constexpr int SMEM_BUDGET = 232448 - 1024 - 512;
  static constexpr bool QUANT = KVT != KV_BF16;
  // bf16 KV, one CTA per tile: a V chunk is 64 keys of the tile by the pass's 256 output
  // columns (four [64 keys][64 dims] 128B-swizzled blocks of 8 KB), so that P.V runs as
  // N = 256 MMAs (one per 16 keys, four per chunk): on this GPU an N = 128 MMA takes about
  // 90 cycles and an N = 256 one about 130, against 64 and 128 of arithmetic
  static constexpr bool VKEYS = !PAIR && !QUANT && DVP == 256;
  // warps 8-11: converters for quantised KV (one key row per thread); for bf16 KV a second
  // softmax warpgroup, so each softmax thread handles half of its row's 128 keys
  static constexpr int THREADS = 384;
  static constexpr int SMW = QUANT ? 1 : 2;   // softmax warpgroups
  static constexpr int NCOL = 128 / SMW;      // S columns per softmax thread
  // Quantised KV: warp 0 streams the packed bytes of each 64-dim half chunk ([128 keys][CW
  // bytes]) and, for NVFP4, the block scales of each K or V tile ([128 keys][D / 16 bytes])
  // into staging rings with TMA; the converters turn two staged halves into one slot of the
  // bf16 / f16 ring the MMAs read.  The staging rings hide the L2 latency, so the converted
  // ring only covers the conversion.
  static constexpr int CW = KVT == KV_FP8 ? 64 : (KVT == KV_NVFP4 ? 32 : 0);  // packed bytes per key and half
  static constexpr int STG_BYTES = N * CW;
  static constexpr int NQS = 2 * NQC, NVS = 2 * NVC;                         // staged halves per step
  static constexpr int SFW_K = DQK / 16, SFW_V = DVO / 16;                  // scale bytes per key
  static constexpr int SF_BYTES = KVT == KV_NVFP4 ? N * SFW_K : 0;
  static constexpr int NSF = KVT == KV_NVFP4 ? 2 : 0;
  static constexpr int NSLOT_RAW = (SMEM_BUDGET - Q_BYTES) / CHUNK;
  static constexpr int NSLOT = QUANT ? (DQK > 256 ? 2 : 3) : (NSLOT_RAW > 4 ? 4 : NSLOT_RAW);
  static constexpr int NSTG_RAW = QUANT ? (SMEM_BUDGET - Q_BYTES - NSLOT * CHUNK - NSF * SF_BYTES) / (STG_BYTES + 8) : 0;
  static constexpr int NSTG = NSTG_RAW > 8 ? 8 : NSTG_RAW;
  static constexpr int OFF_RING = Q_BYTES;
  static constexpr int OFF_STG = Q_BYTES + NSLOT * CHUNK;
  static constexpr int OFF_SF = OFF_STG + NSTG * STG_BYTES;
  static constexpr int OFF_DESC = OFF_SF + NSF * SF_BYTES;  // int2 per staging slot: valid keys, flags
  static constexpr int OFF_XCH = OFF_DESC + NSTG * 8;  // [2][128] floats: partial row maxima / sums
  // head_dim_vo 512 with P reuse: per KV tile of an item, the item's local index + 1 when
  // the first pass rescaled O before that tile's PV (the second pass replays only those)
  static constexpr int MAX_RT = 64;
  static constexpr int OFF_RTAG = OFF_XCH + (SMW == 2 ? 1024 : 0);
  static constexpr int OFF_BAR = OFF_RTAG + (NPASS == 2 ? MAX_RT * 4 : 0);
  // head_dim_vo 512 with P reuse: the second pass reads the first pass's P tiles into
  // NPS slots of the Q region (Q is not needed by then)
  static constexpr int NPS = NPASS == 2 ? Q_BYTES / CHUNK : 0;
  // barriers: (unused), q_empty, s_full[2], p_full[2], pv_done[2], o_free, aux, sfree[2],
  // ps_done, o_done, o_ready, resc_done, tags_done, qreg_free, kv_full[], kv_empty[], stg_full[], stg_empty[],
  // sf_full[], sf_empty[], pslot_full[], pslot_empty[].  Every waiter of a barrier is at
  // most one phase behind or ahead of it (a parity wait cannot tell more apart): hence one
  // s_full / p_full / pv_done / sfree per S buffer.
  static constexpr int NB_FIXED = 18;
  // q_part[NKC]: the Q columns of K chunk c have landed (the first QK of an item starts on
  // the first part of Q instead of waiting for the whole 128 KB tile)
  static constexpr int NBAR = NB_FIXED + 2 * NSLOT + 2 * NSTG + 2 * NSF + 2 * NPS + NKC;
  static constexpr int QB_PER = NQB / NKC;  // 64-column Q blocks per K chunk
  static constexpr int BYTES = OFF_BAR + NBAR * 8 + 16;
  static constexpr int ALLOC = BYTES + 1024;
  // TMEM columns: two S buffers of 128 keys (step j uses buffer j & 1; its P, 128 keys of
  // bf16 / f16, is written over the first 64 columns of the same buffer), O from 256
  static constexpr uint32_t TM_S = 0, TM_O = 256;
  // Named (hardware) barriers between the gate warp and the MMA warp, 64 threads each:
  // one per ring slot, per S buffer for P and for PV completion, Q tile, O free.
  static constexpr int NB_SLOT = 1, NB_P = NB_SLOT + NSLOT, NB_SFREE = NB_P + 2, NB_Q = NB_SFREE + 2,
                       NB_OFREE = NB_Q + 1, NB_PSLOT = NB_OFREE + 1;
  static_assert(NSLOT >= 2, "KV ring too shallow");
  static_assert(!QUANT || NSTG >= 3, "staging ring too shallow");
  static_assert(ALLOC <= 232448, "shared memory");
  static constexpr int NB_SMX = 15;  // the two softmax warpgroups (256 threads)
  static_assert(NB_PSLOT + NPS <= NB_SMX, "named barriers");
  static_assert(NPASS == 1 || NPS >= 2, "P slots");
  static_assert(DVP % 128 == 0 && DQK % 128 == 0, "head dims");
  static_assert(!PAIR || (KVT == KV_BF16 && DVP == 256 && DQK % 256 == 0), "CTA pairs: bf16 KV");
};

// ----------------------------------------------------------------------------- plan
// Items (sequence, first new-token index, kv head) in descending order of the KV tiles
// they visit, so that a static round-robin over persistent CTAs balances.
constexpr int kPlanBuckets = 2048;

// KV tiles visited by the item starting at new-token q_begin (one query tile, or the two
// consecutive tiles of a CTA pair)
__device__ __forceinline__ int prefill_tile_cost(const PrefillParams& p, int kv_len, int qo_len, int q_begin) {
  const int n_pos = min(p.rows_per_tile * (p.pair ? 2 : 1), qo_len - q_begin);
  const int pos0 = kv_len - qo_len + q_begin;
  const int hi = p.causal ? min(kv_len - 1, pos0 + n_pos - 1) : kv_len - 1;
  const int lo = p.window_left >= 0 ? max(0, pos0 - p.window_left) : 0;
  if (hi < lo || hi < 0) return 0;
  return hi / p.tile_tok - lo / p.tile_tok + 1;
}

// First KV tile and number of KV tiles of the item starting at new-token q_begin (the
// range prefill_item_info computes); nt 0 when no key is visible.
__device__ __forceinline__ void prefill_tile_range(const PrefillParams& p, int kv_len, int qo_len, int q_begin,
                                                   int& jlo, int& nt) {
  const int n_pos = min(p.rows_per_tile * (p.pair ? 2 : 1), qo_len - q_begin);
  const int pos0 = kv_len - qo_len + q_begin;
  int hi = p.causal ? min(kv_len - 1, pos0 + n_pos - 1) : kv_len - 1;
  int lo = p.window_left >= 0 ? max(0, pos0 - p.window_left) : 0;
  hi = max(hi, 0);
  lo = min(lo, hi);
  jlo = lo / p.tile_tok;
  nt = hi / p.tile_tok - jlo + 1;
}

#ifdef PA_PREFILL_PLAN
// Per-sequence tile offsets (exclusive scan over ceil(qo_len / P)), then a cost histogram
// and a scatter over all tiles in parallel.  Run by one block of 1024 threads.
// Batches of up to kPlanCache sequences keep their tile offsets and lengths in shared
// memory, so the per-tile lookups below are shared-memory reads, not chains of dependent
// global loads.
constexpr int kPlanCache = 2048;

__device__ __forceinline__ void prefill_plan_body(const PrefillParams& p) {
  __shared__ int hist[kPlanBuckets];
  __shared__ int s_red[32];
  __shared__ int s_carry;
  __shared__ int c_off[kPlanCache + 1], c_qo[kPlanCache], c_kv[kPlanCache];
  const int tid = threadIdx.x;
  for (int i = tid; i < kPlanBuckets; i += blockDim.x) hist[i] = 0;
  if (tid == 0) s_carry = 0;
  __syncthreads();
  const int P = p.rows_per_tile * (p.pair ? 2 : 1), ps = p.page_size;  // positions per item
  const bool cached = p.batch <= kPlanCache;
  int* off = cached ? c_off : p.tile_off;  // [batch + 1]
  for (int base = 0; base < p.batch; base += blockDim.x) {
    const int b = base + tid;
    int qo_len = 0;
    if (b < p.batch) {
      qo_len = p.qo_indptr[b + 1] - p.qo_indptr[b];
      if (cached) {
        const int np = p.kv_indptr[b + 1] - p.kv_indptr[b];
        c_qo[b] = qo_len;
        c_kv[b] = np > 0 ? (np - 1) * ps + p.kv_last_page_len[b] : 0;
      }
    }
    const int n = (qo_len + P - 1) / P;
    int v = n;
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, v, o);
      if ((tid & 31) >= o) v += t;
    }
    if ((tid & 31) == 31) s_red[tid >> 5] = v;
    __syncthreads();
    if (tid < 32) {
      int w = (tid < (int)(blockDim.x >> 5)) ? s_red[tid] : 0;
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, w, o);
        if (tid >= o) w += t;
      }
      s_red[tid] = w;
    }
    __syncthreads();
    const int excl = s_carry + v - n + ((tid >> 5) > 0 ? s_red[(tid >> 5) - 1] : 0);
    if (b < p.batch) off[b] = excl;
    __syncthreads();
    if (tid == blockDim.x - 1) s_carry = excl + n;
    __syncthreads();
  }
  const int n_tiles = s_carry;
  if (tid == 0) off[p.batch] = n_tiles;
  __syncthreads();
  auto tile_of = [&](int t, int& b, int& q0, int& cost) {
    int lo = 0, hi = p.batch - 1;  // last b with off[b] <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (off[mid] <= t) lo = mid; else hi = mid - 1;
    }
    b = lo;
    q0 = (t - off[b]) * P;
    int qo_len, kv_len;
    if (cached) {
      qo_len = c_qo[b];
      kv_len = c_kv[b];
    } else {
      qo_len = p.qo_indptr[b + 1] - p.qo_indptr[b];
      const int np = p.kv_indptr[b + 1] - p.kv_indptr[b];
      kv_len = np > 0 ? (np - 1) * ps + p.kv_last_page_len[b] : 0;
    }
    cost = prefill_tile_cost(p, kv_len, qo_len, q0);
  };
  // split KV: fewer tiles x kv heads than split_target (short queries over long KV): every
  // (tile, kv head) whose range is long enough becomes several items over consecutive
  // parts of it, each with its own partial slot, plus one merge entry; the part counts
  // follow the ranges' lengths so that at most about 2 x split_target items exist.  A
  // thread per tile finds its
  // range and part count, one thread turns the counts into offsets (the tiles number
  // fewer than split_target), and every thread then writes items and merges in parallel.
  if (p.split_target > 0 && n_tiles * p.Hkv < p.split_target && n_tiles <= 256) {
    // per-tile records in the (here unused) histogram
    int* t_b = hist;
    int* t_q0 = hist + 256;
    int* t_jlo = hist + 512;
    int* t_nt = hist + 768;
    int* t_parts = hist + 1024;
    int* t_ioff = hist + 1280;  // first item
    int* t_soff = hist + 1536;  // first partial slot
    int* t_moff = hist + 1792;  // first merge entry
    int cost = 0;
    if (tid < n_tiles) {
      int b, q0;
      tile_of(tid, b, q0, cost);
      int qo_len, kv_len;
      if (cached) {
        qo_len = c_qo[b];
        kv_len = c_kv[b];
      } else {
        qo_len = p.qo_indptr[b + 1] - p.qo_indptr[b];
        const int np = p.kv_indptr[b + 1] - p.kv_indptr[b];
        kv_len = np > 0 ? (np - 1) * p.page_size + p.kv_last_page_len[b] : 0;
      }
      int jlo, nt;
      prefill_tile_range(p, kv_len, qo_len, q0, jlo, nt);
      t_b[tid] = b;
      t_q0[tid] = q0;
      t_jlo[tid] = jlo;
      t_nt[tid] = nt;
    }
    // the total cost of the tiles
    for (int o = 16; o > 0; o >>= 1) cost += __shfl_xor_sync(0xffffffffu, cost, o);
    __syncthreads();  // (s_red was last read before the tile offsets' scan finished)
    if ((tid & 31) == 0) s_red[tid >> 5] = cost;
    __syncthreads();
    long long total = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) total += s_red[w];
    // parts in proportion to each range, rounded down, so that the items number at most
    // 2 x split_target (two rounds over the CTAs) and come out of near-equal size; at
    // least 4 KV tiles a part.  (Chunks of one fixed size rounded each range's part
    // count up: 4 x 32 new tokens over 16384 keys gave 320 items of 13 tiles, a third
    // round for 16 CTAs.)
    if (tid < n_tiles) {
      const int nt = t_nt[tid];
      const long long want = (long long)nt * 2 * p.split_target / max(1ll, total * p.Hkv);
      const int parts = (int)max(1ll, min((long long)(nt + 3) / 4, want));
      // as many parts as parts of ceil(nt / parts) tiles need: none comes out empty
      // (25 tiles in 6 parts of 5 would leave the sixth empty)
      const int step = (nt + parts - 1) / parts;
      t_parts[tid] = (nt + step - 1) / step;
    }
    __syncthreads();
    if (tid == 0) {
      int ni = 0, ns = 0, nm = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const int parts = t_parts[t];
        t_ioff[t] = ni;
        t_soff[t] = ns;
        t_moff[t] = nm;
        ni += parts * p.Hkv;
        if (parts > 1) {
          ns += parts * p.Hkv;
          nm += p.Hkv;
        }
      }
      // stay inside the host's bounds (cannot trigger with chunk as chosen above): no split
      if (ni > p.max_items || ns > p.max_slots) {
        for (int t = 0; t < n_tiles; ++t) {
          t_parts[t] = 1;
          t_ioff[t] = t * p.Hkv;
          t_soff[t] = t_moff[t] = 0;
        }
        ni = n_tiles * p.Hkv;
        nm = 0;
      }
      s_carry = ni;
      s_red[0] = nm;
      p.hdr[0] = ni;
      p.hdr[1] = nm;
      p.hdr[2] = 0;  // full item records
    }
    __syncthreads();
    const int n_items = s_carry, n_merge = s_red[0];
    // the last tile whose first entry (in off[]) is at or before i
    auto tile_at = [&](const int* off, int i) {
      int lo = 0, hi = n_tiles - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= i) lo = mid; else hi = mid - 1;
      }
      return lo;
    };
    for (int i = tid; i < n_items; i += blockDim.x) {
      const int t = tile_at(t_ioff, i);
      const int parts = t_parts[t], local = i - t_ioff[t];
      const int k = local / parts, s2 = local % parts;
      const int jlo = t_jlo[t], nt = t_nt[t], step = (nt + parts - 1) / parts;
      PrefillItem it;
      it.b = t_b[t];
      it.q_begin = t_q0[t];
      it.kvh = k;
      it.kv_t0 = jlo + s2 * step;
      it.kv_t1 = min(jlo + nt, jlo + (s2 + 1) * step);
      it.cost = it.kv_t1 - it.kv_t0;
      it.slot = parts > 1 ? t_soff[t] + k * parts + s2 : -1;
      p.items[i] = it;
    }
    for (int i = tid; i < n_merge; i += blockDim.x) {
      // split tiles only own merge entries, and a split tile's entries precede every later
      // tile's offset, so the last tile at or before i is the split tile that owns i
      const int t = tile_at(t_moff, i);
      const int k = i - t_moff[t];
      PrefillMerge m;
      m.b = t_b[t];
      m.q_begin = t_q0[t];
      m.kvh = k;
      m.slot0 = t_soff[t] + k * t_parts[t];
      m.parts = t_parts[t];
      p.merges[i] = m;
    }
    return;
  }
  // bucket counts aggregated per warp: the lanes of a warp with the same cost add once
  // (tiles of equal cost are common: neighbouring tiles of a sequence differ by one KV
  // tile at most), so a warp makes one shared-memory atomic per distinct cost
  auto bucket_add = [&](int key, bool valid) -> int {
    const int lane = tid & 31;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? key : -1 - lane);
    const int first = __ffs(peers) - 1;
    int base = 0;
    if (valid && lane == first) base = atomicAdd(&hist[key], __popc(peers));
    base = __shfl_sync(0xffffffffu, base, first);
    return base + __popc(peers & ((1u << lane) - 1u));
  };
  for (int t0 = 0; t0 < n_tiles; t0 += blockDim.x) {  // blockDim.x is a multiple of 32
    const int t = t0 + tid;
    int b = 0, q0 = 0, cost = 0;
    if (t < n_tiles) tile_of(t, b, q0, cost);
    bucket_add(min(kPlanBuckets - 1, cost), t < n_tiles);
  }
  __syncthreads();
  // exclusive prefix in descending cost order: bucket c starts after all buckets > c
  {
    constexpr int PER = kPlanBuckets / 1024;
    int loc[PER], sum = 0;
    for (int i = 0; i < PER; ++i) {  // thread tid owns buckets kPlanBuckets-1-(tid*PER+i)
      loc[i] = hist[kPlanBuckets - 1 - (tid * PER + i)];
      sum += loc[i];
    }
    int v = sum;
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, v, o);
      if ((tid & 31) >= o) v += t;
    }
    if ((tid & 31) == 31) s_red[tid >> 5] = v;
    __syncthreads();
    if (tid < 32) {
      int w = s_red[tid];
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, w, o);
        if (tid >= o) w += t;
      }
      s_red[tid] = w;
    }
    __syncthreads();
    int run = v - sum + ((tid >> 5) > 0 ? s_red[(tid >> 5) - 1] : 0);
    for (int i = 0; i < PER; ++i) {
      hist[kPlanBuckets - 1 - (tid * PER + i)] = run;
      run += loc[i];
    }
  }
  __syncthreads();
  for (int t0 = 0; t0 < n_tiles; t0 += blockDim.x) {
    const int t = t0 + tid;
    int b = 0, q0 = 0, cost = 0;
    if (t < n_tiles) tile_of(t, b, q0, cost);
    const int slot = bucket_add(min(kPlanBuckets - 1, cost), t < n_tiles);
    // one 16-byte record per tile (sequence, first new token, cost); item it is the
    // tile's record it / Hkv with kv head it % Hkv
    if (t < n_tiles && (slot + 1) * p.Hkv <= p.max_items)  // always within the host bound
      reinterpret_cast<int4*>(p.items)[slot] = make_int4(b, q0, cost, 0);
  }
  if (tid == 0) {
    p.hdr[0] = min(n_tiles * p.Hkv, p.max_items);
    p.hdr[1] = 0;
    p.hdr[2] = 1;  // tile records
  }
}

#endif  // PA_PREFILL_PLAN

// Everything one role needs to know about a work item.
struct PrefillItemInfo {
  int b, kvh, q_begin, n_pos, qo_len, kv_len, q_row0, pos0, jlo, nt, ip0, np;
  int slot;  // split KV: partial slot of this item, -1 when it writes the output
};

// The plan record of item it: one 16-byte record per tile (sequence, first new token,
// cost), item it being record it / Hkv with kv head it % Hkv, when tile_list; otherwise
// full item records.
__device__ __forceinline__ PrefillItem prefill_item_record(const PrefillParams& p, int it, bool tile_list) {
  PrefillItem item;
  if (tile_list) {
    const int4 r = reinterpret_cast<const int4*>(p.items)[it / p.Hkv];
    item.b = r.x;
    item.q_begin = r.y;
    item.kvh = it % p.Hkv;
    item.cost = r.z;
    item.kv_t0 = item.kv_t1 = 0;
    item.slot = -1;
  } else {
    item = p.items[it];
  }
  return item;
}

// An item's record with the entries of its sequence's index arrays.
struct PrefillItemRaw {
  PrefillItem item;
  int qo0, qo1, kv0, kv1, last;
};

__device__ __forceinline__ PrefillItemRaw prefill_item_raw(const PrefillParams& p, const PrefillItem& item) {
  PrefillItemRaw w;
  w.item = item;
  w.qo0 = p.qo_indptr[item.b];
  w.qo1 = p.qo_indptr[item.b + 1];
  w.kv0 = p.kv_indptr[item.b];
  w.kv1 = p.kv_indptr[item.b + 1];
  w.last = p.kv_last_page_len[item.b];
  return w;
}

// `rank`: which tile of a CTA pair's item this CTA computes (0 without pairs).  Both CTAs
// of a pair walk the KV range of the whole item; the second tile may be empty (n_pos 0).
__device__ __forceinline__ PrefillItemInfo prefill_item_finish(const PrefillParams& p, const PrefillItemRaw& w,
                                                               int rank) {
  const PrefillItem& item = w.item;
  PrefillItemInfo f;
  f.b = item.b;
  f.kvh = item.kvh;
  f.q_begin = item.q_begin + rank * p.rows_per_tile;
  f.qo_len = w.qo1 - w.qo0;
  f.ip0 = w.kv0;
  f.np = w.kv1 - w.kv0;
  f.kv_len = f.np > 0 ? (f.np - 1) * p.page_size + w.last : 0;
  f.n_pos = max(0, min(p.rows_per_tile, f.qo_len - f.q_begin));
  f.q_row0 = w.qo0 + f.q_begin;
  f.pos0 = f.kv_len - f.qo_len + f.q_begin;
  const int ipos0 = f.kv_len - f.qo_len + item.q_begin;
  const int inpos = min(p.rows_per_tile * (p.pair ? 2 : 1), f.qo_len - item.q_begin);
  int hi = p.causal ? min(f.kv_len - 1, ipos0 + inpos - 1) : f.kv_len - 1;
  int lo = p.window_left >= 0 ? max(0, ipos0 - p.window_left) : 0;
  hi = max(hi, 0);  // at least one tile: rows without a visible key come out as 0 / -inf
  lo = min(lo, hi);
  f.jlo = lo / p.tile_tok;
  f.nt = hi / p.tile_tok - f.jlo + 1;
  f.slot = item.slot;
  if (item.kv_t1 > item.kv_t0) {  // split KV: one chunk of the range
    const int t0 = max(f.jlo, item.kv_t0), t1 = min(f.jlo + f.nt, item.kv_t1);
    f.jlo = t0;
    f.nt = max(1, t1 - t0);
  }
  return f;
}

__device__ __forceinline__ PrefillItemInfo prefill_item_info(const PrefillParams& p, int it, int rank,
                                                             bool tile_list) {
  return prefill_item_finish(p, prefill_item_raw(p, prefill_item_record(p, it, tile_list)), rank);
}

// Bits [s, s + n) of a little-endian bit array (bit k of the result = bit s + k; n <= 0
// gives 0, n is clamped to 64).  Only the bytes that hold those bits are read.
__device__ __forceinline__ uint64_t load_mask_bits(const uint8_t* m, int64_t s, int n) {
  if (n <= 0) return 0;
  n = min(n, 64);
  const int64_t b0 = s >> 3, b1 = (s + n - 1) >> 3;
  const int sh = (int)(s & 7);
  uint64_t lo = 0;
  uint32_t top = 0;
  for (int64_t b = b0; b <= b1; ++b) {
    const uint32_t v = __ldg(m + b);
    const int k = (int)(b - b0);
    if (k < 8) lo |= (uint64_t)v << (8 * k);
    else top = v;
  }
  uint64_t r = lo >> sh;
  if (sh) r |= (uint64_t)top << (64 - sh);
  return n < 64 ? r & ((1ull << n) - 1) : r;
}

// r-th item of this CTA (or CTA pair): rounds of one item per CTA (pair), alternating
// direction, over a list sorted by descending cost.
template <bool PAIR>
__device__ __forceinline__ int prefill_item_at(int r) {
  const int n = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const int u = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int off = (r & 1) ? n - 1 - u : u;
  return r * n + off;
}

// The items of this CTA (or CTA pair) in order.  The loads behind an item's info form a
// chain (plan record, then its sequence's index arrays), which a role that fetched them at
// the item boundary would wait out there, twice: so the record of item r + 2 and the index
// entries of item r + 1 are fetched while item r runs, and only the arithmetic is left for
// the boundary.
template <bool PAIR>
struct PrefillItemWalk {
  int r = 0;
  PrefillItemRaw next;  // item r + 1
  PrefillItem rec;      // the record of item r + 2
  __device__ __forceinline__ void start(const PrefillParams& p, int n_items, bool tile_list) {
    const int i0 = prefill_item_at<PAIR>(0), i1 = prefill_item_at<PAIR>(1);
    if (i0 < n_items) next = prefill_item_raw(p, prefill_item_record(p, i0, tile_list));
    if (i1 < n_items) rec = prefill_item_record(p, i1, tile_list);
  }
  // false when the CTA has no item left; else the current item's info in f
  __device__ __forceinline__ bool advance(const PrefillParams& p, int n_items, bool tile_list, int rank,
                                          PrefillItemInfo& f) {
    if (prefill_item_at<PAIR>(r) >= n_items) return false;
    f = prefill_item_finish(p, next, rank);
    if (prefill_item_at<PAIR>(r + 1) < n_items) next = prefill_item_raw(p, rec);
    const int i2 = prefill_item_at<PAIR>(r + 2);
    if (i2 < n_items) rec = prefill_item_record(p, i2, tile_list);
    ++r;
    return true;
  }
};

// tm_p (CTA pairs only): the P scratch as rows of 128 bytes, boxes of one 32 KB P tile
// GEN: custom masks and small padded pages may occur (false: neither, their code is not
// compiled in, which the plain causal / windowed calls run)
template <int KVT, int DQK, int DVO, bool PAIR, bool GEN = true>
__global__ void __launch_bounds__(PrefillCfg<DQK, DVO, KVT, PAIR>::THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_sfk,
                   const __grid_constant__ CUtensorMap tm_sfv, const __grid_constant__ CUtensorMap tm_p,
                   const PrefillParams p) {
  using C = PrefillCfg<DQK, DVO, KVT, PAIR>;
  constexpr int NSLOT = C::NSLOT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t q_s = smem_u32(smem);
  const uint32_t ring = q_s + C::OFF_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  // bars + 0: unused (the Q tile completes on q_part[] below)
  uint64_t* q_empty = bars + 1;
  uint64_t* s_full = bars + 2;  // [2]: S of step j complete in buffer j & 1
  uint64_t* p_full = bars + 4;  // [2]: P of step j written over buffer j & 1
  uint64_t* pv_done = bars + 6;  // [2]: PV of step j (which reads buffer j & 1) complete
  uint64_t* o_free = bars + 8;
  uint64_t* aux = bars + 9;
  uint64_t* sfree = bars + 10;    // [2]: the PV that read P from S buffer b is complete
  uint64_t* ps_done = bars + 12;  // the first pass's P tiles of an item are in global memory
  uint64_t* o_done = bars + 13;   // the last PV of a pass is complete (once per pass)
  uint64_t* o_ready = bars + 14;  // P reuse: the PVs before a replayed rescale are complete
  uint64_t* resc_done = bars + 15;  // P reuse: the softmax warps rescaled O
  uint64_t* tags_done = bars + 16;  // CTA pairs: both CTAs' rescale tags of an item are written
  uint64_t* qreg_free = bars + 17;  // P reuse: the item's last QK is done (P slots may fill)
  uint64_t* kv_full = bars + C::NB_FIXED;
  uint64_t* kv_empty = kv_full + NSLOT;
  uint64_t* stg_full = kv_full + 2 * NSLOT;
  uint64_t* stg_empty = stg_full + C::NSTG;
  uint64_t* sf_full = stg_empty + C::NSTG;
  uint64_t* sf_empty = sf_full + C::NSF;
  uint64_t* pslot_full = sf_empty + C::NSF;
  uint64_t* pslot_empty = pslot_full + C::NPS;
  uint64_t* q_part = pslot_empty + C::NPS;  // [NKC]
  int2* stg_desc = reinterpret_cast<int2*>(smem + C::OFF_DESC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA pairs: the barriers the MMA issuer waits on live in the pair's first CTA (rank 0)
  // and count the arrivals of both CTAs; the barriers MMA completion signals exist in both
  // CTAs (multicast commits).  `lead` gives a barrier's address in the first CTA.
  const uint32_t rank = C::PAIR ? cluster_ctarank() : 0;
  auto lead = [&](uint64_t* b) -> uint32_t { return C::PAIR ? mapa_shared(smem_u32(b), 0) : smem_u32(b); };
  if (threadIdx.x == 0) {
    for (int c = 0; c < C::NKC; ++c) mbar_init(&q_part[c], C::CL);
    mbar_init(q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 4 * C::SMW * C::CL);
      mbar_init(&pv_done[b], 1);
      mbar_init(&sfree[b], 1);
    }
    mbar_init(ps_done, 4 * C::SMW);
    mbar_init(o_done, 1);
    mbar_init(o_ready, 1);
    mbar_init(resc_done, 4 * C::SMW * C::CL);
    mbar_init(tags_done, 4 * C::SMW * C::CL);
    mbar_init(qreg_free, 1);
    for (int s = 0; s < C::NPS; ++s) {
      mbar_init(&pslot_full[s], C::CL);
      mbar_init(&pslot_empty[s], 1);
    }
    mbar_init(o_free, 4 * C::SMW * C::CL);
    mbar_init(aux, 1);
    for (int s = 0; s < NSLOT; ++s) {
      // quantised KV: the four converter warps arrive; pairs: both CTAs' producers
      mbar_init(&kv_full[s], KVT == KV_BF16 ? C::CL : 4);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < C::NSTG; ++s) {
      mbar_init(&stg_full[s], 1);
      mbar_init(&stg_empty[s], 4);
    }
    for (int s = 0; s < C::NSF; ++s) {
      mbar_init(&sf_full[s], 1);
      mbar_init(&sf_empty[s], 4);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (C::PAIR) tmem_alloc_pair(tmem_slot, 512);
    else tmem_alloc(tmem_slot, 512);
  }
  if (C::NPASS == 2)
    for (int i = threadIdx.x; i < C::MAX_RT; i += C::THREADS) reinterpret_cast<int*>(smem + C::OFF_RTAG)[i] = 0;
  tc_fence_before();
  if constexpr (C::PAIR) cluster_sync_all();  // the peer's barriers exist before any remote arrival
  else __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  grid_dep_wait();  // the planner (and the page conversion) of this call are complete
  const int n_items = min(p.hdr[0], p.max_items);
  const bool tile_list = p.hdr[2] != 0;
  const int ps = p.page_size, g = p.group;
  // head_dim_vo 512 (bf16 KV): the second pass reads P of the first from global scratch
  // instead of recomputing S, for items whose KV range fits the scratch
  auto item_reuse = [&](const PrefillItemInfo& f) {
    return C::NPASS == 2 && !C::QUANT && f.nt <= p.reuse_tiles && f.nt <= C::MAX_RT;
  };
  int* rtag = reinterpret_cast<int*>(smem + C::OFF_RTAG);

  if (warp == 0 && KVT == KV_BF16) {
    // ------------------------------------------------------------ producer (whole warp)
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    uint32_t rc = 0, aux_phase = 0, qe = 0;
    const uint64_t pol_kv = l2_policy_evict_last(), pol_q = l2_policy_evict_first();
    PrefillItemWalk<C::PAIR> walk;
    walk.start(p, n_items, tile_list);
    for (;;) {
      PrefillItemInfo f;
      if (!walk.advance(p, n_items, tile_list, rank, f)) break;
      const bool reuse = item_reuse(f);
      // Q part c (the columns of K chunk c), into its own barrier
      auto load_q_part = [&](int c) {
        if (lane != 0) return;
        const uint32_t qbytes = (uint32_t)(C::QB_PER * 128 * g * p.rows_per_tile);
        if constexpr (C::PAIR) {
          mbar_arrive_expect_tx_cluster(lead(&q_part[c]), qbytes);
          for (int b = c * C::QB_PER; b < (c + 1) * C::QB_PER; ++b)
            tma_load_3d_pair(q_s + b * C::HALF, &tm_q, b * 128, f.kvh * g, f.q_row0, lead(&q_part[c]), pol_q);
        } else {
          mbar_arrive_expect_tx(&q_part[c], qbytes);
          for (int b = c * C::QB_PER; b < (c + 1) * C::QB_PER; ++b)
            tma_load_3d_hint(q_s + b * C::HALF, &tm_q, b * 128, f.kvh * g, f.q_row0, &q_part[c], pol_q);
        }
      };
      // steps that compute S: both passes, or only the first when the second reuses P
      const int steps = reuse ? f.nt : C::NPASS * f.nt;
      // a KV tile is ppt pages of rpp rows each (rpp = page_size, or 8 for the padded copy
      // of smaller pages: then only the first page_size rows of a page are tokens)
      const int rpp = p.box_rows, ppt = 128 / rpp;
      // page ids of a step's KV tile, one per lane (lane < pieces); loaded a few steps
      // ahead so the producer never waits on them
      auto step_pages = [&](int st) -> int {
        if (st < 0 || st >= C::NPASS * f.nt) return 0;
        const int pg0 = (f.jlo + st % f.nt) * ppt;
        const int pieces = max(0, min(ppt, f.np - pg0));
        return (lane < pieces) ? __ldg(p.kv_indices + f.ip0 + pg0 + lane) : 0;
      };
      // the K or V chunks of step st into the ring (K: chunks [c_lo, c_hi), one CTA per tile)
      auto emit = [&](bool is_k, int st, int my_page, int c_lo = 0, int c_hi = C::NQC) {
        const int pass = st / f.nt, jt = st % f.nt;
        // tile rows before the first that holds no token of the sequence
        const int rem = max(0, f.kv_len - (f.jlo + jt) * p.tile_tok);
        const int valid = min(128, rem / ps * rpp + rem % ps);
        if constexpr (C::PAIR) {
          if (is_k) {
            // this CTA's 64 keys of the tile (B rows of its half of N), in chunks of 256
            // dims: four [64 keys][64 dims] blocks per page piece
            // (pairs read the caller's pages: a tile is 128 tokens)
            const int h0 = (f.jlo + jt) * 128 + 64 * (int)rank;
            const int pieces = max(0, min(64, f.np * ps - h0)) / ps;
            const int pg0 = 64 * (int)rank / ps;
            for (int c = 0; c < C::NKC; ++c, ++rc) {
              const int slot = rc % NSLOT;
              mbar_wait<C::PAIR>(&kv_empty[slot], ((rc / NSLOT) & 1) ^ 1, p.err, SITE_PRE_KV_EMPTY);
              const uint32_t dst = ring + slot * C::CHUNK;
              const uint32_t fb = lead(&kv_full[slot]);
              if (lane == 0) mbar_arrive_expect_tx_cluster(fb, (uint32_t)(4 * pieces * ps * 128));
              for (int pc = 0; pc < pieces; ++pc) {
                const int page = __shfl_sync(0xffffffffu, my_page, pg0 + pc);
                if (lane == 0)
                  for (int blk = 0; blk < 4; ++blk)
                    tma_load_3d_pair(dst + blk * C::KBLK + pc * ps * 128, &tm_k, c * 512 + blk * 128, f.kvh * ps,
                                     page, fb, pol_kv);
              }
            }
            return;
          }
        }
        const int pieces = max(0, min(ppt, f.np - (f.jlo + jt) * ppt));
        if (C::VKEYS && !is_k) {
          // V by keys: chunk c = tile rows [64 c, 64 c + 64), all of the pass's 256 columns
          for (int c = 0; c < 2; ++c, ++rc) {
            const int slot = rc % NSLOT;
            mbar_wait(&kv_empty[slot], ((rc / NSLOT) & 1) ^ 1, p.err, SITE_PRE_KV_EMPTY);
            const uint32_t dst = ring + slot * C::CHUNK;
            const int pc0 = 64 * c / rpp, pc1 = min(pieces, (64 * c + 64) / rpp);
            const int vrows = min(64, max(0, valid - 64 * c));  // rows that hold tokens
            const bool fix = vrows < 64;  // V rows past the sequence must be zeroed
            uint64_t* bar = fix ? aux : &kv_full[slot];
            if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(4 * max(0, pc1 - pc0) * rpp * 128));
            for (int pc = pc0; pc < pc1; ++pc) {
              const int page = __shfl_sync(0xffffffffu, my_page, pc);
              if (lane == 0)
                for (int b = 0; b < 4; ++b)
                  tma_load_3d_hint(dst + b * C::KBLK + (pc - pc0) * rpp * 128, &tm_v, (pass * C::DVP + b * 64) * 2,
                                   f.kvh * rpp, page, bar, pol_kv);
            }
            if (fix) {
              mbar_wait(aux, aux_phase, p.err, SITE_PRE_DEQ);
              aux_phase ^= 1;
              uint8_t* sp = smem + C::OFF_RING + slot * C::CHUNK;
              const int nz = (64 - vrows) * 8;  // 16-byte pieces per block
              for (int i = lane; i < 4 * nz; i += 32) {
                const int b = i / nz, k = i - b * nz;
                *reinterpret_cast<uint4*>(sp + b * C::KBLK + (vrows + (k >> 3)) * 128 + (k & 7) * 16) =
                    make_uint4(0, 0, 0, 0);
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) mbar_arrive(&kv_full[slot]);
            }
          }
          return;
        }
        const int c_end = is_k ? c_hi : C::NVS_P;
        for (int c = is_k ? c_lo : 0; c < c_end; ++c, ++rc) {
          const int slot = rc % NSLOT;
          mbar_wait<C::PAIR>(&kv_empty[slot], ((rc / NSLOT) & 1) ^ 1, p.err, SITE_PRE_KV_EMPTY);
          const uint32_t dst = ring + slot * C::CHUNK;
          const uint32_t bytes = (uint32_t)(2 * pieces * rpp * 128);
          const bool fix = !is_k && valid < 128;  // V rows past the sequence must be zeroed
          // pairs: the chunk completes on the first CTA's barrier (the zeroing path on this
          // CTA's aux first)
          const bool remote = C::PAIR && !fix;
          uint64_t* bar = fix ? aux : &kv_full[slot];
          const uint32_t fb = lead(&kv_full[slot]);
          if (lane == 0) {
            if (remote) mbar_arrive_expect_tx_cluster(fb, bytes);
            else mbar_arrive_expect_tx(bar, bytes);
          }
          // the chunk's two 64-dim blocks: bytes of dims [128 c, 128 c + 128) of the row
          // (pairs: of this CTA's 128 of the pass's output columns)
          const int col = is_k ? c * 256 : (pass * C::DVP + (C::PAIR ? (int)rank : c) * 128) * 2;
          for (int pc = 0; pc < pieces; ++pc) {
            const int page = __shfl_sync(0xffffffffu, my_page, pc);
            if (lane == 0)
              for (int h = 0; h < 2; ++h) {
                if (remote)
                  tma_load_3d_pair(dst + h * C::HALF + pc * rpp * 128, &tm_v, col + h * 128, f.kvh * rpp, page, fb,
                                   pol_kv);
                else
                  tma_load_3d_hint(dst + h * C::HALF + pc * rpp * 128, is_k ? &tm_k : &tm_v, col + h * 128,
                                   f.kvh * rpp, page, bar, pol_kv);
              }
          }
          if (fix) {
            mbar_wait(aux, aux_phase, p.err, SITE_PRE_DEQ);
            aux_phase ^= 1;
            uint8_t* sp = smem + C::OFF_RING + slot * C::CHUNK;
            const int nz = (128 - valid) * 8;  // 16-byte pieces per block
            for (int i = lane; i < 2 * nz; i += 32) {
              const int h = i >= nz, k = i - h * nz;
              *reinterpret_cast<uint4*>(sp + h * C::HALF + (valid + (k >> 3)) * 128 + (k & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if constexpr (C::PAIR) mbar_arrive_cluster(fb);
              else mbar_arrive(&kv_full[slot]);
            }
          }
        }
      };
      // chunks in the MMA thread's order: K of step 0, then per step k: K of k + 1, V of k.
      // One CTA per tile: warp 3 loads the Q tiles, so that the next item's Q is requested
      // as soon as the Q region is free, not after this warp has queued the V chunks of the
      // item's last steps (which wait for ring slots).  CTA pairs: Q here, before K.
      // (the first pages are fetched before the wait for the Q region, so their loads run
      // during it)
      int pg_a = step_pages(0), pg_b = step_pages(1);
      if constexpr (C::PAIR) {
        mbar_wait<C::PAIR>(q_empty, (qe++ & 1) ^ 1, p.err, SITE_PRE_Q);
        for (int c = 0; c < C::NKC; ++c) load_q_part(c);
      }
      emit(true, 0, pg_a);
      for (int k = 0; k < steps; ++k) {
        const int pg_c = step_pages(k + 2);
        if (k + 1 < steps) emit(true, k + 1, pg_b);
        emit(false, k, pg_a);
        pg_a = pg_b;
        pg_b = pg_c;
      }
      if (reuse) {
        // second pass: V of the upper output half (the P tiles come from warp 3)
        if constexpr (C::PAIR) mbar_wait<C::PAIR>(q_empty, (qe++ & 1) ^ 1, p.err, SITE_PRE_Q);
        int pg = step_pages(f.nt);
        for (int j = 0; j < f.nt; ++j) {
          const int pg_n = step_pages(f.nt + j + 1);
          emit(false, f.nt + j, pg);
          pg = pg_n;
        }
      }
    }
  } else if (warp == 3 && !C::QUANT && (C::NPASS == 2 || !C::PAIR)) {
    // ------------------------------- Q tiles (one CTA per tile) and P tiles of second passes
    // Q: each item's tile, in parts of the K chunks' dims on their own barriers, as soon as
    // the previous item has released the Q region (its last QK, or its second pass).
    // P: the first pass's P tiles of an item (usually back from HBM) go into the P slots of
    // the Q region once the item's last QK is done and the softmax has written them; up to
    // NPS tiles ahead of the PVs, independently of the V chunks in the ring.
    constexpr int NPS = C::NPS > 0 ? C::NPS : 1;
    const uint8_t* pscr = p.p_scratch + (size_t)blockIdx.x * p.reuse_tiles * C::CHUNK;
    const uint64_t pol_p = l2_policy_evict_first(), pol_q = l2_policy_evict_first();
    uint32_t np = 0, n_reuse = 0, qe = 0;
    PrefillItemWalk<C::PAIR> walk;
    walk.start(p, n_items, tile_list);
    for (;;) {
      PrefillItemInfo f;
      if (!walk.advance(p, n_items, tile_list, rank, f)) break;
      const bool reuse = item_reuse(f);
      if constexpr (!C::PAIR) {
        mbar_wait(q_empty, (qe++ & 1) ^ 1, p.err, SITE_PRE_Q);
        if (lane == 0) {
          const uint32_t qbytes = (uint32_t)(C::QB_PER * 128 * g * p.rows_per_tile);
          for (int c = 0; c < C::NKC; ++c) {
            mbar_arrive_expect_tx(&q_part[c], qbytes);
            for (int b = c * C::QB_PER; b < (c + 1) * C::QB_PER; ++b)
              tma_load_3d_hint(q_s + b * C::HALF, &tm_q, b * 128, f.kvh * g, f.q_row0, &q_part[c], pol_q);
          }
        }
        __syncwarp();
        // an item that reuses P releases the Q region twice: after its last QK (the P slots
        // may fill) and after its second pass (the next Q may load)
        if (reuse) mbar_wait(q_empty, (qe++ & 1) ^ 1, p.err, SITE_PRE_Q);
      }
      if (!reuse) continue;
      mbar_wait<C::PAIR>(qreg_free, n_reuse & 1, p.err, SITE_PRE_Q);
      mbar_wait(ps_done, n_reuse & 1, p.err, SITE_PRE_P_FULL);
      ++n_reuse;
      for (int j = 0; j < f.nt; ++j, ++np) {
        const int s = np % NPS;
        mbar_wait<C::PAIR>(&pslot_empty[s], ((np / NPS) & 1) ^ 1, p.err, SITE_PRE_KV_EMPTY);
        if (lane == 0) {
          if constexpr (C::PAIR) {
            mbar_arrive_expect_tx_cluster(lead(&pslot_full[s]), (uint32_t)C::CHUNK);
            tma_load_2d_pair(q_s + s * C::CHUNK, &tm_p, 0, ((int)blockIdx.x * p.reuse_tiles + j) * 256,
                             lead(&pslot_full[s]), pol_p);
          } else {
            mbar_arrive_expect_tx(&pslot_full[s], (uint32_t)C::CHUNK);
            bulk_load_g2s_hint(q_s + s * C::CHUNK, pscr + (size_t)j * C::CHUNK, (uint32_t)C::CHUNK, &pslot_full[s],
                               pol_p);
          }
        }
        __syncwarp();
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------ producer for quantised KV (whole warp)
    // Q tiles as in the bf16 producer; K / V as packed bytes into the staging ring, one
    // chunk per slot with a descriptor (valid keys, flags) the converters read after the
    // slot fills; NVFP4 block scales of each K or V tile into the scale ring.
    if constexpr (C::QUANT) {
      constexpr int FL_V = 1, FL_FIRST = 2, FL_LAST = 4, FL_END = 8;
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        if constexpr (KVT == KV_NVFP4) {
          tma_prefetch_desc(&tm_sfk);
          tma_prefetch_desc(&tm_sfv);
        }
      }
      const uint64_t pol_kv = l2_policy_evict_last(), pol_q = l2_policy_evict_first();
      const uint32_t stg = q_s + C::OFF_STG, sfb = q_s + C::OFF_SF;
      uint32_t n = 0, nsf = 0;
      int it_local = 0;
      PrefillItemWalk<C::PAIR> walk;
      walk.start(p, n_items, tile_list);
      for (;; ++it_local) {
        PrefillItemInfo f;
        if (!walk.advance(p, n_items, tile_list, rank, f)) break;
        mbar_wait(q_empty, (it_local & 1) ^ 1, p.err, SITE_PRE_Q);
        if (lane == 0)
          for (int c = 0; c < C::NKC; ++c) {
            mbar_arrive_expect_tx(&q_part[c], (uint32_t)(C::QB_PER * 128 * g * p.rows_per_tile));
            for (int b = c * C::QB_PER; b < (c + 1) * C::QB_PER; ++b)
              tma_load_3d_hint(q_s + b * C::HALF, &tm_q, b * 128, f.kvh * g, f.q_row0, &q_part[c], pol_q);
          }
        const int steps = C::NPASS * f.nt;
        const int page_tok_cap = f.np * ps;
        auto step_pages = [&](int st) -> int {
          if (st < 0 || st >= steps) return 0;
          const int key0 = (f.jlo + st % f.nt) * 128;
          const int pieces = max(0, min(128, page_tok_cap - key0)) / ps;
          return (lane < pieces) ? __ldg(p.kv_indices + f.ip0 + key0 / ps + lane) : 0;
        };
        // per iteration k: K of step k + 1 (pages pg_b), V of step k (pages pg_a)
        int pg_a = 0, pg_b = step_pages(0);
        for (int k = -1; k < steps; ++k) {
          const int pg_c = step_pages(k + 2);
          for (int part = 0; part < 2; ++part) {
            const bool is_k = part == 0;
            const int st = is_k ? k + 1 : k;
            if (st < 0 || st >= steps) continue;
            const int pass = st / f.nt, jt = st % f.nt;
            const int key0 = (f.jlo + jt) * 128;
            const int valid = max(0, min(128, f.kv_len - key0));
            const int pieces = max(0, min(128, page_tok_cap - key0)) / ps;
            const int my_page = is_k ? pg_b : pg_a;
            if constexpr (KVT == KV_NVFP4) {
              const int sw = is_k ? C::SFW_K : C::SFW_V;
              const int si = nsf % C::NSF;
              mbar_wait(&sf_empty[si], ((nsf / C::NSF) & 1) ^ 1, p.err, SITE_PRE_SF);
              if (lane == 0) mbar_arrive_expect_tx(&sf_full[si], (uint32_t)(pieces * ps * sw));
              for (int pc = 0; pc < pieces; ++pc) {
                const int page = __shfl_sync(0xffffffffu, my_page, pc);
                if (lane == 0)
                  tma_load_3d_hint(sfb + si * C::SF_BYTES + pc * ps * sw, is_k ? &tm_sfk : &tm_sfv, 0, f.kvh * ps,
                                   page, &sf_full[si], pol_kv);
              }
              ++nsf;
            }
            const int nch = is_k ? C::NQS : C::NVS;  // staged 64-dim halves
            for (int c = 0; c < nch; ++c, ++n) {
              const int stage = n % C::NSTG;
              mbar_wait(&stg_empty[stage], ((n / C::NSTG) & 1) ^ 1, p.err, SITE_PRE_STG);
              const int d0 = is_k ? c * 64 : pass * C::DVP + c * 64;  // first head-dim element
              const int col = d0 * C::CW / 64;                        // its byte in the packed row
              if (lane == 0) {
                const int flags = (is_k ? 0 : FL_V) | (c == 0 ? FL_FIRST : 0) | (c == nch - 1 ? FL_LAST : 0) |
                                  ((d0 / 16) << 8);
                stg_desc[stage] = make_int2(valid, flags);
                mbar_arrive_expect_tx(&stg_full[stage], (uint32_t)(pieces * ps * C::CW));
              }
              for (int pc = 0; pc < pieces; ++pc) {
                const int page = __shfl_sync(0xffffffffu, my_page, pc);
                if (lane == 0)
                  tma_load_3d_hint(stg + stage * C::STG_BYTES + pc * ps * C::CW, is_k ? &tm_k : &tm_v, col,
                                   f.kvh * ps, page, &stg_full[stage], pol_kv);
              }
            }
          }
          pg_a = pg_b;
          pg_b = pg_c;
        }
      }
      // end marker
      const int stage = n % C::NSTG;
      mbar_wait(&stg_empty[stage], ((n / C::NSTG) & 1) ^ 1, p.err, SITE_PRE_STG);
      if (lane == 0) {
        stg_desc[stage] = make_int2(0, FL_END);
        mbar_arrive(&stg_full[stage]);
      }
    }
  } else if (C::QUANT && warp >= 8) {
    if constexpr (C::QUANT) {
      // ---------------------------------------------------------- converters (warps 8-11)
      // Staged halves come in pairs, the two 64-dim blocks of one ring slot.  Thread t owns
      // key t of each staged half: it converts the half's packed values
      // exactly (e4m3 and e2m1 x e4m3 are exact in f16 and in bf16; the per-tensor / global
      // scales are applied to the scores and the output instead) and writes them in the
      // 128B-swizzled layout the MMAs read: K as bf16 (the type of q), V as f16 (P is written
      // in f16 for these kernels, and e4m3 / e2m1 convert to f16 in one instruction).  Keys
      // past the end of the sequence are written as 0, whatever the slot holds.
      constexpr int FL_V = 1, FL_FIRST = 2, FL_LAST = 4, FL_END = 8;
      constexpr int RAW16 = C::CW / 16;
      const int t = threadIdx.x - 256;
      const uint8_t* stg = smem + C::OFF_STG;
      const uint8_t* sfb = smem + C::OFF_SF;
      uint32_t nsf = 0;
      for (uint32_t j = 0;; ++j) {
        const int stage = j % C::NSTG;
        mbar_wait(&stg_full[stage], (j / C::NSTG) & 1, p.err, SITE_PRE_STG);
        const int2 d = stg_desc[stage];
        if (d.y & FL_END) break;
        const bool is_v = d.y & FL_V;
        const int si = C::NSF > 0 ? nsf % (C::NSF > 0 ? C::NSF : 1) : 0;
        if constexpr (KVT == KV_NVFP4)
          if (d.y & FL_FIRST) mbar_wait(&sf_full[si], (nsf / C::NSF) & 1, p.err, SITE_PRE_SF);
        const uint32_t rj = j >> 1, half = j & 1;  // ring chunk and block
        const int slot = rj % NSLOT;
        if (half == 0) mbar_wait(&kv_empty[slot], ((rj / NSLOT) & 1) ^ 1, p.err, SITE_PRE_KV_EMPTY);
        __syncwarp();
        uint8_t* sp = smem + C::OFF_RING + slot * C::CHUNK + half * C::HALF;
        const bool ok = t < d.x;
        uint4 raw[RAW16];
#pragma unroll
        for (int q = 0; q < RAW16; ++q)
          raw[q] = ok ? *reinterpret_cast<const uint4*>(stg + stage * C::STG_BYTES + t * C::CW + 16 * q)
                      : make_uint4(0, 0, 0, 0);
        uint32_t sfw = 0;
        if constexpr (KVT == KV_NVFP4)
          if (ok)
            sfw = *reinterpret_cast<const uint32_t*>(sfb + si * C::SF_BYTES + t * (is_v ? C::SFW_V : C::SFW_K) +
                                                     (d.y >> 8));
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {  // 16-byte output chunk jj = elements 8jj .. 8jj+7
          uint32_t w[4];
          if constexpr (KVT == KV_FP8) {
            const uint4 a = raw[jj >> 1];
            const uint32_t w0 = (jj & 1) ? a.z : a.x, w1 = (jj & 1) ? a.w : a.y;
            w[0] = e4m3x2_to_f16x2(w0 & 0xFFFFu);
            w[1] = e4m3x2_to_f16x2(w0 >> 16);
            w[2] = e4m3x2_to_f16x2(w1 & 0xFFFFu);
            w[3] = e4m3x2_to_f16x2(w1 >> 16);
          } else {
            const uint4 a = raw[jj >> 2];
            const uint32_t word = (jj & 3) == 0 ? a.x : (jj & 3) == 1 ? a.y : (jj & 3) == 2 ? a.z : a.w;
            const uint32_t sb = (sfw >> (8 * (jj >> 1))) & 0xFFu;
            const uint32_t sf2 = e4m3x2_to_f16x2(sb | (sb << 8));
            uint32_t f4[4];
            e2m1x8_to_f16x2x4(word, f4);
#pragma unroll
            for (int q = 0; q < 4; ++q) w[q] = hmul2_u32(f4[q], sf2);
          }
          if (!is_v) {
#pragma unroll
            for (int q = 0; q < 4; ++q) w[q] = f16x2_to_bf16x2(w[q]);
          }
          *reinterpret_cast<uint4*>(sp + t * 128 + ((jj ^ (t & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (half == 1) mbar_arrive(&kv_full[slot]);
          mbar_arrive(&stg_empty[stage]);
          if (KVT == KV_NVFP4 && (d.y & FL_LAST)) mbar_arrive(&sf_empty[si]);
        }
        if (KVT == KV_NVFP4 && (d.y & FL_LAST)) ++nsf;
      }
      (void)FL_FIRST;
    }
  } else if ((warp == 1 || warp == 2) && rank == 0) {
    // ------------------------------------------------------- MMA issuer (1) and gate (2)
    // Both warps walk the same schedule.  The gate polls the mbarriers; the MMA warp waits
    // on a named barrier the gate meets once its poll succeeded, and lane 0 issues the
    // MMAs and commits (a commit tracks the MMAs of the thread that issues it).  A shared
    // memory poll from the issuing warp stalls the tensor pipe for hundreds of cycles
    // while it reads its operands from shared memory; a named barrier does not touch it.
    // Both sides use bar.sync, so the gate never runs more than one barrier ahead.
    const bool gate = warp == 2;
    const bool leader = warp == 1 && lane == 0;
    constexpr uint32_t ID_QK = idesc_f16<true>(128 * C::CL, 128, false);
    // quantised KV: P and V in f16.  Pairs: one N = 256 MMA per 16 keys covers the pass's
    // output columns (128 from each CTA's V chunk)
    constexpr uint32_t ID_PV = idesc_f16<!C::QUANT>(128 * C::CL, 128 * C::CL, true);
    constexpr uint32_t ID_PV2 = idesc_f16<true>(128, 256, true);  // V by keys
    // MMA issue and commits: the pair forms (cta_group::2) in a CTA pair.  commit_both
    // signals the barrier in both CTAs, commit_here only in this (the first) CTA.
    auto mma_ss = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
      if constexpr (C::PAIR) tc_mma_ss_pair(d, a, b, id, acc);
      else tc_mma_ss(d, a, b, id, acc);
    };
    auto mma_ts = [&](uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
      if constexpr (C::PAIR) tc_mma_ts_pair(d, a, b, id, acc);
      else tc_mma_ts(d, a, b, id, acc);
    };
    auto commit_both = [&](uint64_t* b) {
      if constexpr (C::PAIR) tc_commit_pair_both(b);
      else tc_commit(b);
    };
    auto commit_here = [&](uint64_t* b) {
      if constexpr (C::PAIR) tc_commit_pair_local(b);
      else tc_commit(b);
    };
    // one synchronisation point of the schedule: the gate waits for the phase, then both
    // warps meet at named barrier `id`
    auto point = [&](int id, uint64_t* bar, uint32_t parity, int site) {
      if (gate) mbar_wait<C::PAIR>(bar, parity, p.err, site);
      named_bar_sync(id, 64);
    };
    // steps issued so far (QK into S buffer n_qk & 1; PV reads P of step n_spv from buffer
    // n_spv & 1) and passes finished.  QK of step j + 2 reuses the buffer of step j, where
    // PV of step j reads P: it waits for that PV to complete (an MMA that reads its A
    // operand from TMEM is not ordered against a later MMA writing the same columns).
    // Order: QK(0), then per step j: QK(j + 1), PV(j).  The S of step j + 1 is computed
    // while the softmax of step j runs, and PV(j) follows at once, so the pipe waits for
    // a softmax only when the softmax is slower than a QK (measured 1.7 % faster than
    // issuing QK QK PV PV in pairs).  One mbarrier per buffer: the next PV on a buffer
    // follows the QK that waits on it, so a barrier is never two phases ahead of its waiter.
    // n_spv counts the PVs that read P from an S buffer (their order is the QKs' order);
    // np counts P slots, n_rs the rescales replayed in second passes that reuse P.  The
    // last PV of every pass commits o_done, which the epilogue waits for.
    uint32_t rc = 0, n_qk = 0, n_spv = 0, n_pass = 0, np = 0, n_rs = 0;
    int it_local = 0;
    // TMEM halves of this item: S buffers at tm_s, O of the first pass at tm_o; a second
    // pass that reuses P accumulates at tm_s (the S buffers are free by then), so it need
    // not wait for the first pass's O to drain; after such an item the halves swap
    uint32_t flip = 0, tm_s = C::TM_S, tm_o = C::TM_O;
    // q_wait: the item's first QK, which waits for each Q part before its K chunk
    auto issue_qk = [&](bool q_wait) {
      const uint32_t s_col = tm_s + 128 * (n_qk & 1);
      if (n_qk >= 2) point(C::NB_SFREE + (n_qk & 1), &sfree[n_qk & 1], ((n_qk - 2) >> 1) & 1, SITE_PRE_O_DONE);
      for (int c = 0; c < C::NKC; ++c, ++rc) {
        if (q_wait) point(C::NB_Q, &q_part[c], it_local & 1, SITE_PRE_Q);
        const int slot = rc % NSLOT;
        point(C::NB_SLOT + slot, &kv_full[slot], (rc / NSLOT) & 1, SITE_PRE_KV_FULL);
        if (warp == 1) {
          tc_fence_after();
          if (leader) {
            const uint32_t bsm = ring + slot * C::CHUNK;
            if constexpr (C::PAIR) {
              // dims [256 c, 256 c + 256): Q blocks 4c..4c+3, this CTA's 64 keys in 8 KB blocks
#pragma unroll
              for (int h = 0; h < 4; ++h)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_ss(tbase + s_col, desc_kmajor_sw128(q_s + (4 * c + h) * C::HALF + kk * 32),
                         desc_kmajor_sw128(bsm + h * C::KBLK + kk * 32), ID_QK, (c | h | kk) != 0);
            } else {
#pragma unroll
              for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_ss(tbase + s_col, desc_kmajor_sw128(q_s + (2 * c + h) * C::HALF + kk * 32),
                         desc_kmajor_sw128(bsm + h * C::HALF + kk * 32), ID_QK, (c | h | kk) != 0);
            }
            commit_both(&kv_empty[slot]);
          }
        }
      }
      if (leader) commit_both(&s_full[n_qk & 1]);
      ++n_qk;
    };
    auto issue_pv = [&](bool first_of_pass, bool last_of_pass) {
      point(C::NB_P + (n_spv & 1), &p_full[n_spv & 1], (n_spv >> 1) & 1, SITE_PRE_P_FULL);
      const uint32_t p_col = tm_s + 128 * (n_spv & 1);
      if (first_of_pass && n_pass > 0) point(C::NB_OFREE, o_free, (n_pass - 1) & 1, SITE_PRE_O_DONE);
      // V by keys: one N = 256 MMA per 16 keys of the chunk covers the pass's 256 output
      // columns (four 64-column atoms 8 KB apart).  Otherwise one N = 128 MMA per 16 keys
      // covers the chunk's 128 output columns (pairs: N = 256 over both CTAs' chunks).
      for (int c = 0; c < C::NVS_P; ++c, ++rc) {
        const int slot = rc % NSLOT;
        point(C::NB_SLOT + slot, &kv_full[slot], (rc / NSLOT) & 1, SITE_PRE_KV_FULL);
        if (warp == 1) {
          tc_fence_after();
          if (leader) {
            const uint32_t bsm = ring + slot * C::CHUNK;
            if constexpr (C::VKEYS) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ts(tbase + tm_o, tbase + p_col + (4 * c + kk) * 8, desc_mnmajor_sw128(bsm + kk * 2048, C::KBLK),
                       ID_PV2, (!first_of_pass) || c > 0 || kk > 0);
            } else {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_ts(tbase + tm_o + c * 128, tbase + p_col + kk * 8,
                       desc_mnmajor_sw128(bsm + kk * 2048, C::HALF), ID_PV, (!first_of_pass) || kk > 0);
            }
            commit_both(&kv_empty[slot]);
          }
        }
      }
      if (leader) {
        commit_here(&sfree[n_spv & 1]);
        commit_both(&pv_done[n_spv & 1]);
        if (last_of_pass) commit_both(o_done);
      }
      ++n_spv;
      if (first_of_pass) ++n_pass;
    };
    // second pass with P reuse: P tile j from a P slot (shared memory) times V.  The PVs
    // follow one another without the softmax, except where the first pass rescaled O
    // before tile j: then the MMAs so far are committed to o_ready, and the PV waits until
    // the softmax warps have applied the same factor (resc_done).
    // p1: index of the item's first pass (its o_done / o_free phases)
    auto issue_pv_reuse = [&](int j, int last, uint64_t rmask, uint32_t p1) {
      // the first pass's MMAs are complete (its last PVs read P from the columns this pass
      // accumulates in); its O may still be draining from the other half
      if (j == 0) point(C::NB_OFREE, o_done, p1 & 1, SITE_PRE_O_DONE);
      if ((rmask >> j) & 1) {
        if (leader) commit_both(o_ready);
        point(C::NB_OFREE, resc_done, n_rs & 1, SITE_PRE_P_FULL);
        ++n_rs;
      }
      constexpr int NPS = C::NPS > 0 ? C::NPS : 1;
      const int s = np % NPS;
      point(C::NB_PSLOT + s, &pslot_full[s], (np / NPS) & 1, SITE_PRE_KV_FULL);
      for (int c = 0; c < C::NVS_P; ++c, ++rc) {
        const int slot = rc % NSLOT;
        point(C::NB_SLOT + slot, &kv_full[slot], (rc / NSLOT) & 1, SITE_PRE_KV_FULL);
        if (warp == 1) {
          tc_fence_after();
          if (leader) {
            const uint32_t bsm = ring + slot * C::CHUNK, psm = q_s + s * C::CHUNK;
            // P: K-major without swizzle, key group g8 (8 keys) of every row at g8 x 2048
            if constexpr (C::VKEYS) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ss(tbase + tm_s, desc_kmajor_plain(psm + (4 * c + kk) * 2 * 2048, 2048, 128),
                       desc_mnmajor_sw128(bsm + kk * 2048, C::KBLK), ID_PV2, (j > 0) || c > 0 || kk > 0);
            } else {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_ss(tbase + tm_s + c * 128, desc_kmajor_plain(psm + kk * 2 * 2048, 2048, 128),
                       desc_mnmajor_sw128(bsm + kk * 2048, C::HALF), ID_PV, (j > 0) || kk > 0);
            }
            commit_both(&kv_empty[slot]);
          }
        }
      }
      if (leader) commit_both(&pslot_empty[s]);
      if (j == last) {
        // the first pass's O has drained before the next item writes S over it (waited here,
        // before this pass's o_done exists, so o_free is never two phases ahead)
        point(C::NB_OFREE, o_free, p1 & 1, SITE_PRE_O_DONE);
        if (leader) commit_both(o_done);
      }
      ++np;
      if (j == 0) ++n_pass;
    };
    PrefillItemWalk<C::PAIR> walk;
    walk.start(p, n_items, tile_list);
    for (;; ++it_local) {
      PrefillItemInfo f;
      if (!walk.advance(p, n_items, tile_list, rank, f)) break;
      const bool reuse = item_reuse(f);
      const int steps = reuse ? f.nt : C::NPASS * f.nt;
      // QK(k + 1) runs while the softmax of step k works, then PV(k)
      for (int k = -1; k < steps; ++k) {
        if (k + 1 < steps) {
          issue_qk(k < 0);
          if (leader && k + 1 == steps - 1) {  // the item's last QK
            commit_both(q_empty);
            if (reuse) commit_both(qreg_free);
          }
        }
        if (k >= 0) issue_pv(k % f.nt == 0, (k + 1) % f.nt == 0);
      }
      if (reuse) {
        // the tiles the first pass tagged, read once per item into a mask (a shared-memory
        // read in the issuing warp waits behind the MMAs' operand reads); every first-pass
        // tag of the item is visible here, after the gate's p_full waits of the whole pass
        static_assert(C::MAX_RT <= 64, "rescale tags");
        const int tag = it_local + 1;
        const uint64_t rmask = (uint64_t)__ballot_sync(0xffffffffu, lane < C::MAX_RT && rtag[lane] == tag) |
                               ((uint64_t)__ballot_sync(0xffffffffu, lane + 32 < C::MAX_RT && rtag[lane + 32] == tag)
                                << 32);
        const uint32_t p1 = n_pass - 1;
        for (int j = 0; j < f.nt; ++j) issue_pv_reuse(j, f.nt - 1, rmask, p1);
        if (leader) commit_both(q_empty);  // the P slots (Q region) are free
        flip ^= 1;
        tm_s = flip ? C::TM_O : C::TM_S;
        tm_o = flip ? C::TM_S : C::TM_O;
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    // Thread r of a warpgroup owns row r (TMEM lane r); with two warpgroups (bf16 KV) the
    // first handles keys [0, 64) of each tile and the upper output columns' half of the
    // O rescales and of the epilogue is split the same way; the row maximum is combined
    // through shared memory once per tile, the row sums at the end of a pass.
    constexpr int NCOL = C::NCOL;
    const int wg = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = 32 * quarter + lane;  // TMEM lane == tile row
    const int col0 = wg * NCOL;           // first key of this thread's columns
    const uint32_t lane_base = tbase + ((uint32_t)(32 * quarter) << 16);
    float* xch = reinterpret_cast<float*>(smem + C::OFF_XCH);
    // combine a per-row value with the other warpgroup's (max or sum)
    auto combine = [&](float v, bool is_max) -> float {
      if constexpr (C::SMW == 1) {
        return v;
      } else {
        xch[wg * 128 + row] = v;
        named_bar_sync(C::NB_SMX, 256);
        const float o = xch[(wg ^ 1) * 128 + row];
        named_bar_sync(C::NB_SMX, 256);
        return is_max ? fmaxf(v, o) : v + o;
      }
    };
    // O columns this thread rescales and writes out
    constexpr int OCOL = C::DVP / C::SMW;
    const int ocol0 = wg * OCOL;
    // FP8 per-tensor / NVFP4 global K scale folds into the scores, the V scale into the output
    // (also given for bf16 KV when it is the bf16 copy of FP8 / NVFP4 pages)
    const float scale_log2 = p.sm_scale * 1.4426950408889634f * (p.k_scale ? __ldg(p.k_scale) : 1.f);
    // scores are scaled inside the exponent's FMA; a non-positive scale is applied up
    // front instead (the maximum of the raw scores is only the scaled maximum for scale > 0)
    const bool pos_scale = scale_log2 > 0.f;
    const float eff_scale = pos_scale ? scale_log2 : 1.f;
    const float v_scale = p.v_scale ? __ldg(p.v_scale) : 1.f;
    // TMEM halves as the MMA warp uses them: S at tm_s, the first pass's O at tm_o, a
    // second pass that reuses P at tm_s; swapped after every such item
    uint32_t flip = 0, tm_s = C::TM_S, tm_o = C::TM_O;
    auto rescale_o = [&](float a, uint32_t o_col) {
#pragma unroll 1
      for (int c = 0; c < OCOL / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(lane_base + o_col + ocol0 + 32 * c, ov);
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * a);
        tmem_st32(lane_base + o_col + ocol0 + 32 * c, ov);
      }
      tc_wait_st();
    };
    // sstep counts the steps that read an S buffer, n_epi the epilogues (passes), n_rs the
    // rescales replayed in second passes that reuse P
    uint32_t sstep = 0, n_epi = 0, n_rs = 0, n_tags = 0;
    // arrival on a barrier the MMA issuer waits for (pairs: the first CTA's)
    auto arrive_lead = [&](uint64_t* b) {
      if constexpr (C::PAIR) mbar_arrive_cluster(lead(b));
      else mbar_arrive(b);
    };
    int it_local = 0;
    uint8_t* pscr = p.p_scratch + (size_t)blockIdx.x * p.reuse_tiles * C::CHUNK;
    float* mscr = p.m_scratch + (size_t)blockIdx.x * p.reuse_tiles * 128;
    // the first pass's P tiles are read back by the second pass of the same item: keep
    // them in L2 ahead of streaming data; the second pass reads them with evict-first
    const uint64_t pol_keep = l2_policy_evict_last();
    // bf16 KV: the next item's info is fetched in the last epilogue of the current one,
    // while it waits for the last PV (holding it through the softmax loop would cost
    // registers).  Quantised KV (one softmax warpgroup, more registers a thread): at the
    // item's start.
    int it_next = prefill_item_at<C::PAIR>(0);
    PrefillItemInfo f_next;
    if (!C::QUANT && it_next < n_items) f_next = prefill_item_info(p, it_next, rank, tile_list);
    for (int r = 0;; ++r, ++it_local) {
      if (it_next >= n_items) break;
      if constexpr (C::QUANT) f_next = prefill_item_info(p, it_next, rank, tile_list);
      const PrefillItemInfo f = f_next;
      const bool reuse = item_reuse(f);
      const int tag = it_local + 1;
      const int p_local = row / g, h_local = row % g;
      const bool row_ok = (row < g * p.rows_per_tile) && (p_local < f.n_pos);
      const int pos = f.pos0 + p_local;
      const int khi = p.causal ? pos : f.kv_len - 1;
      const int klo = p.window_left >= 0 ? pos - p.window_left : 0;
      const int hq = f.kvh * g + h_local;
      // custom mask: bit index of (this row, key 0)
      const int64_t mbase = (GEN && p.mask != nullptr && row_ok)
                                ? p.mask_indptr[f.b] * 8 + (int64_t)(f.q_begin + p_local) * f.kv_len
                                : 0;
      float m_used = -INFINITY, l = 0.f;
      for (int pass = 0; pass < C::NPASS; ++pass) {
        if (reuse && pass == 1) {
          // second pass reusing P: no S; replay the first pass's O rescales at the tiles
          // tagged in the first pass (every softmax warp takes part in each, so that the
          // barrier phases stay in step).  The tags of all warps are visible here: the
          // first pass's epilogue met at the warpgroups' named barrier after them.  This
          // thread wrote its factors itself.
          for (int j = 0; j < f.nt; ++j) {
            if (rtag[j] != tag) continue;
            const float a = mscr[j * 128 + row];
            mbar_wait<C::PAIR>(o_ready, n_rs & 1, p.err, SITE_PRE_O_DONE);
            ++n_rs;
            __syncwarp();
            tc_fence_after();
            if (__any_sync(0xffffffffu, a != 1.f)) rescale_o(a, tm_s);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_lead(resc_done);
          }
        } else {
          m_used = -INFINITY;
          l = 0.f;
          for (int jt = 0; jt < f.nt; ++jt, ++sstep) {
            const uint32_t s_col = tm_s + 128 * (sstep & 1);
            mbar_wait<C::PAIR>(&s_full[sstep & 1], (sstep >> 1) & 1, p.err, SITE_PRE_S_FULL);
            __syncwarp();  // the tcgen05 loads below are warp-collective
            tc_fence_after();
            uint32_t sr[NCOL];
#pragma unroll
            for (int c = 0; c < NCOL / 32; ++c) tmem_ld32(lane_base + s_col + col0 + 32 * c, sr + 32 * c);
            tc_wait_ld();
            // visible keys of this row as indices [lo, hi] into this thread's columns.
            // Tiles every row of the warp sees in full skip the mask; otherwise it is a
            // select on two compares (short-circuit forms compiled to per-element
            // branches).  The maximum is taken over the raw scores (the scale is positive,
            // or applied first when it is not); max and sum run as four chains.
            const int key0 = (f.jlo + jt) * 128 + col0;
            const int lo = klo - key0, hi = min(khi, f.kv_len - 1) - key0;
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (!pos_scale) {
#pragma unroll
              for (int i = 0; i < NCOL; ++i) sr[i] = __float_as_uint(__uint_as_float(sr[i]) * scale_log2);
            }
            // pages of fewer than 8 tokens, read from their copy padded to 8 rows: column i
            // of this thread is token tok0 + (i / 8) * page_size + i % 8 when i % 8 <
            // page_size and padding otherwise (at most 8 * 4 tokens per thread)
            const bool padded = GEN && p.box_rows != ps;
            const int tok0 = padded ? (f.jlo + jt) * p.tile_tok + (col0 >> 3) * ps : 0;
            // the row maximum over the visible keys of this thread's columns, masked scores
            // set to -inf; a tile every row of the warp sees in full skips the mask
            auto mask_and_max = [&](const uint32_t* mw, bool use_mw) {
#pragma unroll
              for (int i = 0; i < NCOL; ++i) {
                const bool ok = (i >= lo) & (i <= hi) & (use_mw ? ((mw[i >> 5] >> (i & 31)) & 1u) != 0u : true);
                const float x = ok ? __uint_as_float(sr[i]) : -INFINITY;
                sr[i] = __float_as_uint(x);
                mx4[i & 3] = fmaxf(mx4[i & 3], x);
              }
            };
            auto plain_max = [&]() {
#pragma unroll
              for (int i = 0; i < NCOL; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], __uint_as_float(sr[i]));
            };
            if (padded) {
              const int thi = min(khi, f.kv_len - 1) - tok0, tlo = klo - tok0;
              uint64_t mb = ~0ull;  // custom-mask bits of tokens tok0 .. tok0 + 63 of this row
              if (p.mask != nullptr && row_ok) mb = load_mask_bits(p.mask, mbase + tok0, min(64, f.kv_len - tok0));
#pragma unroll
              for (int i = 0; i < NCOL; ++i) {
                const int r = i & 7, t = (i >> 3) * ps + r;
                const bool ok = (r < ps) & (t >= tlo) & (t <= thi) & (((mb >> (t & 63)) & 1ull) != 0ull);
                const float x = ok ? __uint_as_float(sr[i]) : -INFINITY;
                sr[i] = __float_as_uint(x);
                mx4[i & 3] = fmaxf(mx4[i & 3], x);
              }
            } else if (!GEN || p.mask == nullptr) {
              if (__all_sync(0xffffffffu, (lo <= 0) & (hi >= NCOL - 1))) plain_max();
              else mask_and_max(nullptr, false);
            } else {
              // custom-mask bits of this row's columns (1 = may attend; all ones for rows
              // that are not written)
              uint32_t mw[NCOL / 32];
#pragma unroll
              for (int c = 0; c < NCOL / 32; ++c) mw[c] = 0xffffffffu;
              if (row_ok) {
                const int nvalid = max(0, min(NCOL, f.kv_len - key0));
#pragma unroll
                for (int c = 0; c < NCOL / 64; ++c) {
                  const uint64_t w = load_mask_bits(p.mask, mbase + key0 + 64 * c, nvalid - 64 * c);
                  mw[2 * c] = (uint32_t)w;
                  mw[2 * c + 1] = (uint32_t)(w >> 32);
                }
              }
              bool all_ok = true;
#pragma unroll
              for (int c = 0; c < NCOL / 32; ++c) all_ok &= mw[c] == 0xffffffffu;
              if (__all_sync(0xffffffffu, (lo <= 0) & (hi >= NCOL - 1) & all_ok)) plain_max();
              else mask_and_max(mw, true);
            }
            const float mx =
                combine(fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])), true) * eff_scale;
            const float m_new = fmaxf(m_used, mx);
            bool resc = false;
            float alpha = 1.f;
            if (jt == 0) {
              m_used = m_new;
            } else if (m_new > m_used + 8.f) {  // lazy rescale: only when the max grows by > 2^8
              alpha = fast_exp2(m_used - m_new);
              m_used = m_new;
              resc = true;
            }
            const float base = (m_used == -INFINITY) ? 0.f : m_used;
            const float nbase = -base;
            float sum4[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t pk[NCOL / 2];
#pragma unroll
            for (int i = 0; i < NCOL / 2; ++i) {
              const float p0 = fast_exp2(fmaf(__uint_as_float(sr[2 * i]), eff_scale, nbase));
              const float p1 = fast_exp2(fmaf(__uint_as_float(sr[2 * i + 1]), eff_scale, nbase));
              sum4[i & 3] += p0 + p1;
              pk[i] = C::QUANT ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
            }
            const float sum = (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
            // tcgen05.ld / st are warp-collective (.sync.aligned): the whole warp rescales
            // when any of its rows needs it, the other rows with a factor of 1, once the PV
            // of the previous step has finished with O
            if (__any_sync(0xffffffffu, resc)) {
              mbar_wait<C::PAIR>(&pv_done[(sstep - 1) & 1], ((sstep - 1) >> 1) & 1, p.err, SITE_PRE_O_DONE);
              __syncwarp();
              tc_fence_after();
              rescale_o(resc ? alpha : 1.f, tm_o);
              if (reuse && lane == 0) {  // the second pass replays this rescale (pairs: in both CTAs)
                rtag[jt] = tag;
                if constexpr (C::PAIR) st_shared_cluster_u32(mapa_shared(smem_u32(&rtag[jt]), rank ^ 1), (uint32_t)tag);
              }
            }
            if (resc) l *= alpha;
            l += sum;
#pragma unroll
            for (int c = 0; c < NCOL / 64; ++c) tmem_st32(lane_base + s_col + col0 / 2 + 32 * c, pk + 32 * c);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_lead(&p_full[sstep & 1]);
            if (reuse) {
              // after the PV may start: this thread's keys of P tile jt and the rescale
              // factor applied before it.  The tile is the second pass's MMA operand image
              // without swizzle, [16 groups of 8 keys][128 rows][16 B] (8 x 16-byte core
              // matrices, rows 16 bytes apart), so each store instruction of a warp writes
              // one key group of 32 consecutive rows: 512 contiguous bytes.
              uint8_t* prow = pscr + (size_t)jt * C::CHUNK + row * 16;
#pragma unroll
              for (int k = 0; k < NCOL / 8; ++k)
                st_global_v4_hint(prow + (size_t)(col0 / 8 + k) * (128 * 16), pk + 4 * k, pol_keep);
              mscr[jt * 128 + row] = resc ? alpha : 1.f;
            }
          }
          if (reuse) {  // the P tiles of this pass are in global memory for the producer
            fence_proxy_async_global();
            __syncwarp();
            if (lane == 0) mbar_arrive(ps_done);
            if constexpr (C::PAIR) {
              // both CTAs' rescale tags of the item are in both copies before either CTA's
              // second pass reads them
              if (lane == 0) {
                mbar_arrive_cluster(mapa_shared(smem_u32(tags_done), 0));
                mbar_arrive_cluster(mapa_shared(smem_u32(tags_done), 1));
              }
              mbar_wait<true>(tags_done, n_tags & 1, p.err, SITE_PRE_P_FULL);
              ++n_tags;
            }
          }
        }
        // ---- epilogue of this pass: O / l -> bf16
        static_assert(C::NPASS == 1 || C::QUANT || C::SMW == 2, "P reuse orders the rescale tags through the warpgroups' barrier");
        const float lt = combine(l, false);
        if (pass == C::NPASS - 1) {
          it_next = prefill_item_at<C::PAIR>(r + 1);
          if (!C::QUANT && it_next < n_items) f_next = prefill_item_info(p, it_next, rank, tile_list);
        }
        mbar_wait<C::PAIR>(o_done, n_epi & 1, p.err, SITE_PRE_O_DONE);
        ++n_epi;
        __syncwarp();
        tc_fence_after();
        const float inv = lt > 0.f ? v_scale / lt : 0.f;
        const uint32_t o_col = (reuse && pass == 1) ? tm_s : tm_o;  // this pass's O
        uint16_t* orow = p.out + ((size_t)(f.q_row0 + p_local) * p.Hq + hq) * DVO + pass * C::DVP + ocol0;
        const float row_lse = lt > 0.f ? (m_used + log2f(lt)) * 0.69314718055994531f : -INFINITY;
        if (f.slot >= 0) {
          // split KV: this chunk's normalised rows (fp32) and lse into its partial slot
          float* prow = p.part_o + ((size_t)f.slot * 128 + row) * DVO + pass * C::DVP + ocol0;
#pragma unroll 1
          for (int c = 0; c < OCOL / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(lane_base + o_col + ocol0 + 32 * c, ov);
            tc_wait_ld();
            if (row_ok) {
              // 32-byte stores: each writes a whole sector of the thread's row
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * inv);
#pragma unroll
              for (int i = 0; i < 4; ++i) st_global_v8(prow + 32 * c + 8 * i, ov + 8 * i, ov + 8 * i + 4);
            }
          }
          if (pass == C::NPASS - 1 && row_ok && wg == 0) p.part_lse[(size_t)f.slot * 128 + row] = row_lse;
        } else {
#pragma unroll 1
          for (int c = 0; c < OCOL / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(lane_base + o_col + ocol0 + 32 * c, ov);
            tc_wait_ld();
            uint32_t pkd[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pkd[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv, __uint_as_float(ov[2 * i + 1]) * inv);
            if (row_ok) {
              // 32-byte stores where out allows them: a warp's instruction then writes 32
              // whole sectors (the rows of a warp are 2 * DVO bytes apart, so 16-byte stores
              // leave every sector half written and take twice the instructions)
              if (p.out_v8) {
                st_global_stream_v8(orow + 32 * c, pkd);
                st_global_stream_v8(orow + 32 * c + 16, pkd + 8);
              } else {
                uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  st_global_stream_v4(dst + i, make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]));
              }
            }
          }
          if (pass == C::NPASS - 1 && row_ok && p.lse && wg == 0)
            p.lse[(size_t)(f.q_row0 + p_local) * p.Hq + hq] = row_lse;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_lead(o_free);
      }
      if (reuse) {
        flip ^= 1;
        tm_s = flip ? C::TM_O : C::TM_S;
        tm_o = flip ? C::TM_S : C::TM_O;
      }
    }
  }
  tc_fence_before();
  // pairs: neither CTA leaves (or frees TMEM) while the other may still reach its shared
  // memory or barriers
  if constexpr (C::PAIR) cluster_sync_all();
  else __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (C::PAIR) tmem_dealloc_pair(tbase, 512);
    else tmem_dealloc(tbase, 512);
  }
  if constexpr (C::PAIR) cluster_sync_all();
}

}  // namespace pa

// prefill.cu -- instantiates the tcgen05 prefill kernel and its preparation kernel
// (planner, plus the bf16 copy of FP8 / NVFP4 pages).
#define PA_PREFILL_PLAN 1
#include "launch.h"
#include "prefill_dequant.cuh"
#include "prefill_impl.cuh"

namespace pa {

// Block 0 plans the work items; blocks 1.. (COPY: FP8 / NVFP4 pages converted to a bf16
// copy, or pages of fewer than 8 tokens padded in one) write the copy.  The prefill
// kernel that follows is launched as its programmatic dependent and waits for the whole
// grid before it reads either result.
template <int KVT, int DQK, int DVO, bool COPY, bool PAD>
__global__ void __launch_bounds__(1024) prefill_prep_kernel(const PrefillParams p, const DequantParams d) {
  grid_dep_launch();
  if (blockIdx.x == 0) {
    prefill_plan_body(p);
    return;
  }
  if constexpr (COPY) prefill_dequant_body<KVT, DQK, DVO, PAD>(d, blockIdx.x - 1, gridDim.x - 1);
}

template <int KVT, bool PAD>
static cudaError_t run_prep(int dqk, int dvo, int grid, const PrefillParams& p, const DequantParams& d,
                            cudaStream_t s) {
  if (dqk == 512 && dvo == 512) prefill_prep_kernel<KVT, 512, 512, true, PAD><<<grid, 1024, 0, s>>>(p, d);
  else if (dqk == 512 && dvo == 256) prefill_prep_kernel<KVT, 512, 256, true, PAD><<<grid, 1024, 0, s>>>(p, d);
  else if (dqk == 256 && dvo == 256) prefill_prep_kernel<KVT, 256, 256, true, PAD><<<grid, 1024, 0, s>>>(p, d);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_prefill_prep(int kvt, int dqk, int dvo, int copy, const PrefillParams& p,
                                const DequantParams& d, int sms, cudaStream_t s) {
  if (copy == 0) {
    prefill_prep_kernel<KV_BF16, 512, 512, false, false><<<1, 1024, 0, s>>>(p, d);
    return cudaGetLastError();
  }
  // two 1024-thread blocks per SM, the planner's among them, all resident at once (one
  // block more would wait for a slot and run as a second wave)
  const int grid = 2 * sms;
  const bool pad = copy == 2;
  if (kvt == KV_BF16) return pad ? run_prep<KV_BF16, true>(dqk, dvo, grid, p, d, s) : cudaErrorInvalidValue;
  if (kvt == KV_FP8) return pad ? run_prep<KV_FP8, true>(dqk, dvo, grid, p, d, s) : run_prep<KV_FP8, false>(dqk, dvo, grid, p, d, s);
  if (kvt == KV_NVFP4)
    return pad ? run_prep<KV_NVFP4, true>(dqk, dvo, grid, p, d, s) : run_prep<KV_NVFP4, false>(dqk, dvo, grid, p, d, s);
  return cudaErrorInvalidValue;
}

template <int KVT, int DQK, int DVO, bool PAIR>
static cudaError_t run_prefill(const PrefillLaunch& L) {
  using C = PrefillCfg<DQK, DVO, KVT, PAIR>;
  // the bf16 kernel on one CTA per tile without a custom mask or padded pages: the
  // instantiation without that code
  const bool plain = KVT == KV_BF16 && !PAIR && L.p.mask == nullptr && L.p.box_rows == L.p.page_size;
  auto kern = plain ? prefill_kernel<KVT, DQK, DVO, PAIR, !(KVT == KV_BF16 && !PAIR)>
                    : prefill_kernel<KVT, DQK, DVO, PAIR, true>;
  static std::atomic<uint64_t> smem_set[2];
  cudaError_t e = set_smem_limit_once(kern, C::ALLOC, smem_set[plain ? 1 : 0]);
  if (e != cudaSuccess) return e;
  // a programmatic dependent of the preparation kernel (pairs: clusters of two CTAs, one
  // per SM of a pair)
  return launch_pdl(kern, dim3(L.grid), dim3(C::THREADS), C::ALLOC, L.stream, PAIR ? 2 : 1, L.tq, L.tk, L.tv,
                    L.tsfk, L.tsfv, L.tp, L.p);
}

template <int KVT, bool PAIR>
static cudaError_t dispatch_prefill(int dqk, int dvo, const PrefillLaunch& L, const char** variant) {
  if (dqk == 512 && dvo == 512) {
    *variant = PAIR ? "prefill_512x512_pair" : "prefill_512x512";
    return run_prefill<KVT, 512, 512, PAIR>(L);
  }
  if (dqk == 512 && dvo == 256) {
    *variant = PAIR ? "prefill_512x256_pair" : "prefill_512x256";
    return run_prefill<KVT, 512, 256, PAIR>(L);
  }
  if (dqk == 256 && dvo == 256) {
    *variant = PAIR ? "prefill_256x256_pair" : "prefill_256x256";
    return run_prefill<KVT, 256, 256, PAIR>(L);
  }
  return cudaErrorInvalidValue;
}

// Largest number of two-CTA clusters of the bf16 kernel that fit on the device at once
// (0 when none can, or on error).
int prefill_pair_clusters(int dqk, int dvo) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  auto query = [&](auto kern, int threads, int smem) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return;
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  };
  if (dqk == 512 && dvo == 512) {
    using C = PrefillCfg<512, 512, KV_BF16, true>;
    query(prefill_kernel<KV_BF16, 512, 512, true>, C::THREADS, C::ALLOC);
  } else if (dqk == 512 && dvo == 256) {
    using C = PrefillCfg<512, 256, KV_BF16, true>;
    query(prefill_kernel<KV_BF16, 512, 256, true>, C::THREADS, C::ALLOC);
  } else if (dqk == 256 && dvo == 256) {
    using C = PrefillCfg<256, 256, KV_BF16, true>;
    query(prefill_kernel<KV_BF16, 256, 256, true>, C::THREADS, C::ALLOC);
  }
  cudaGetLastError();  // a failed query leaves no sticky error
  return n;
}

cudaError_t launch_prefill(int kvt, int dqk, int dvo, const PrefillLaunch& L, const char** variant) {
  if (kvt == KV_BF16)
    return L.p.pair ? dispatch_prefill<KV_BF16, true>(dqk, dvo, L, variant)
                    : dispatch_prefill<KV_BF16, false>(dqk, dvo, L, variant);
  if (kvt == KV_FP8) return dispatch_prefill<KV_FP8, false>(dqk, dvo, L, variant);
  if (kvt == KV_NVFP4) return dispatch_prefill<KV_NVFP4, false>(dqk, dvo, L, variant);
  return cudaErrorInvalidValue;
}

template <int KVT>
static int smem_bytes(int dqk, int dvo) {
  if (dqk == 512 && dvo == 512) return PrefillCfg<512, 512, KVT>::ALLOC;
  if (dqk == 512 && dvo == 256) return PrefillCfg<512, 256, KVT>::ALLOC;
  return PrefillCfg<256, 256, KVT>::ALLOC;
}

int prefill_smem_bytes(int kvt, int dqk, int dvo) {
  if (kvt == KV_FP8) return smem_bytes<KV_FP8>(dqk, dvo);
  if (kvt == KV_NVFP4) return smem_bytes<KV_NVFP4>(dqk, dvo);
  return smem_bytes<KV_BF16>(dqk, dvo);
}

}  // namespace pa

// prefill.cu -- instantiates the tcgen05 prefill kernel and its planner.
#define PA_PREFILL_PLAN 1
#include "launch.h"
#include "prefill_impl.cuh"

namespace pa {

template <int KVT, int DQK, int DVO>
static cudaError_t run_prefill(const PrefillLaunch& L) {
  using C = PrefillCfg<DQK, DVO, KVT>;
  auto kern = prefill_kernel<KVT, DQK, DVO>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::ALLOC);
  if (e != cudaSuccess) return e;
  kern<<<L.grid, C::THREADS, C::ALLOC, L.stream>>>(L.tq, L.tk, L.tv, L.tsfk, L.tsfv, L.p);
  return cudaGetLastError();
}

template <int KVT>
static cudaError_t dispatch_prefill(int dqk, int dvo, const PrefillLaunch& L, const char** variant) {
  if (dqk == 512 && dvo == 512) {
    *variant = "prefill_512x512";
    return run_prefill<KVT, 512, 512>(L);
  }
  if (dqk == 512 && dvo == 256) {
    *variant = "prefill_512x256";
    return run_prefill<KVT, 512, 256>(L);
  }
  if (dqk == 256 && dvo == 256) {
    *variant = "prefill_256x256";
    return run_prefill<KVT, 256, 256>(L);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill(int kvt, int dqk, int dvo, const PrefillLaunch& L, const char** variant) {
  if (kvt == KV_BF16) return dispatch_prefill<KV_BF16>(dqk, dvo, L, variant);
  if (kvt == KV_FP8) return dispatch_prefill<KV_FP8>(dqk, dvo, L, variant);
  if (kvt == KV_NVFP4) return dispatch_prefill<KV_NVFP4>(dqk, dvo, L, variant);
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_plan(const PrefillParams& p, cudaStream_t s) {
  prefill_plan_kernel<<<1, 1024, 0, s>>>(p);
  return cudaGetLastError();
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

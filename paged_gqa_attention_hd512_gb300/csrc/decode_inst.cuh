// decode_inst.cuh -- instantiates the decode kernel for one KV dtype.  Included by
// decode_bf16.cu / decode_fp8.cu / decode_nvfp4.cu with PA_KVT defined, so that the three
// dtypes compile as separate translation units in parallel.
#pragma once

#include "decode_impl.cuh"
#include "launch.h"

namespace pa {

template <int KVT, int DQK, int DVO, int HP>
static cudaError_t run_decode(const DecodeLaunch& L) {
  using Sm = DecodeSmem<KVT, DQK, DVO, HP>;
  auto kern = decode_kernel<KVT, DQK, DVO, HP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sm::ALLOC);
  if (e != cudaSuccess) return e;
  // a programmatic dependent of the planner
  return launch_pdl(kern, dim3(L.grid), dim3(288), Sm::ALLOC, L.stream, 1, L.tk, L.tv, L.tsfk, L.tsfv, L.p);
}

template <int KVT>
static cudaError_t dispatch_decode(int dqk, int dvo, int hp, const DecodeLaunch& L, const char** variant) {
  static const char* names[3][2] = {
      {"decode_512x512_hp8", "decode_512x512_hp16"},
      {"decode_512x256_hp8", "decode_512x256_hp16"},
      {"decode_256x256_hp8", "decode_256x256_hp16"}};
  int shape = (dqk == 512 && dvo == 512) ? 0 : (dqk == 512 && dvo == 256) ? 1 : (dqk == 256 && dvo == 256) ? 2 : -1;
  if (shape < 0 || (hp != 8 && hp != 16)) return cudaErrorInvalidValue;
  *variant = names[shape][hp == 16];
  if (shape == 0) return hp == 8 ? run_decode<KVT, 512, 512, 8>(L) : run_decode<KVT, 512, 512, 16>(L);
  if (shape == 1) return hp == 8 ? run_decode<KVT, 512, 256, 8>(L) : run_decode<KVT, 512, 256, 16>(L);
  return hp == 8 ? run_decode<KVT, 256, 256, 8>(L) : run_decode<KVT, 256, 256, 16>(L);
}

template <int KVT>
static int smem_of(int dqk, int dvo, int hp) {
  if (dqk == 512 && dvo == 512) return hp == 8 ? DecodeSmem<KVT, 512, 512, 8>::ALLOC : DecodeSmem<KVT, 512, 512, 16>::ALLOC;
  if (dqk == 512 && dvo == 256) return hp == 8 ? DecodeSmem<KVT, 512, 256, 8>::ALLOC : DecodeSmem<KVT, 512, 256, 16>::ALLOC;
  return hp == 8 ? DecodeSmem<KVT, 256, 256, 8>::ALLOC : DecodeSmem<KVT, 256, 256, 16>::ALLOC;
}

}  // namespace pa

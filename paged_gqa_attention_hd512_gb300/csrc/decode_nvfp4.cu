// decode_nvfp4.cu -- decode kernels for nvfp4 KV.
#include "decode_inst.cuh"

namespace pa {
cudaError_t launch_decode_nvfp4(int dqk, int dvo, int hp, const DecodeLaunch& L, const char** variant) {
  return dispatch_decode<KV_NVFP4>(dqk, dvo, hp, L, variant);
}
}  // namespace pa

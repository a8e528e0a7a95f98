// decode_fp8.cu -- decode kernels for fp8 KV.
#include "decode_inst.cuh"

namespace pa {
cudaError_t launch_decode_fp8(int dqk, int dvo, int hp, const DecodeLaunch& L, const char** variant) {
  return dispatch_decode<KV_FP8>(dqk, dvo, hp, L, variant);
}
}  // namespace pa

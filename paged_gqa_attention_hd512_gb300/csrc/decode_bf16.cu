// decode_bf16.cu -- decode kernels for bf16 KV.
#include "decode_inst.cuh"

namespace pa {
cudaError_t launch_decode_bf16(int dqk, int dvo, int hp, const DecodeLaunch& L, const char** variant) {
  return dispatch_decode<KV_BF16>(dqk, dvo, hp, L, variant);
}
}  // namespace pa

// decode_aux.cu -- the decode work planner, the split-K merge and shape queries.
#define PA_DECODE_AUX 1
#include <algorithm>
#include "decode_inst.cuh"

namespace pa {

cudaError_t launch_decode_plan(const DecodeParams& p, cudaStream_t s) {
  // one thread per sequence up to 1024 (at least 256: fewer warps meet faster at the
  // planner's block-wide scans; 256 took 1 us off the 256-sequence sliding-window step)
  const int threads = std::min(1024, std::max(256, (p.batch + 31) / 32 * 32));
  decode_plan_kernel<<<1, threads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode_merge(int dvo, const DecodeParams& p, int sms, cudaStream_t s) {
  const long warps = (long)p.batch * p.Hq * (dvo / 128);
  // one warp per unit up to eight 256-thread blocks per SM (every unit of the bf16 GQA
  // decode at once: 0.3883 -> 0.3873 ms per step against two blocks per SM); the warps
  // stride over the rest
  const int blocks = (int)std::min<long>((warps * 32 + 255) / 256, 8l * sms);
  if (blocks == 0) return cudaSuccess;
  // a programmatic dependent of the decode kernel
  if (dvo == 512) return launch_pdl(decode_merge_kernel<512>, dim3(blocks), dim3(256), 0, s, 1, p);
  return launch_pdl(decode_merge_kernel<256>, dim3(blocks), dim3(256), 0, s, 1, p);
}

int decode_smem_bytes(int kvt, int dqk, int dvo, int hp) {
  if (kvt == KV_BF16) return smem_of<KV_BF16>(dqk, dvo, hp);
  if (kvt == KV_FP8) return smem_of<KV_FP8>(dqk, dvo, hp);
  return smem_of<KV_NVFP4>(dqk, dvo, hp);
}

int decode_tile_tokens(int kvt, int dqk) {
  return (kvt == KV_BF16 && dqk == 512) ? 32 : 64;
}

}  // namespace pa

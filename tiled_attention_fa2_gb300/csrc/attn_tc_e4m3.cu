// FP8 E4M3 instances of the tcgen05 forward kernel (d = 128; causal or not).
#include "attn_tc_sm103.cuh"

namespace attn {

cudaError_t launch_tc_e4m3(const TcParams& p, int d, bool causal, int num_sms, cudaStream_t stream) {
  if (d == 128) return causal ? launch_tc<TcCfg<true, 128, true>>(p, num_sms, stream) : launch_tc<TcCfg<true, 128, false>>(p, num_sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn

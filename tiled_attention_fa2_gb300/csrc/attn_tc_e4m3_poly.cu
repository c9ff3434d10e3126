// FP8 E4M3 instances of the tcgen05 forward kernel with the split exponential
// (one exponential pair in four on the FMA pipe; attn_set_poly_exp2).
#include "attn_tc_sm103.cuh"

namespace attn {

cudaError_t launch_tc_e4m3_poly(const TcParams& p, int d, bool causal, int num_sms, cudaStream_t stream) {
  if (d == 128)
    return causal ? launch_tc<TcCfg<true, 128, true, true>>(p, num_sms, stream)
                  : launch_tc<TcCfg<true, 128, false, true>>(p, num_sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn

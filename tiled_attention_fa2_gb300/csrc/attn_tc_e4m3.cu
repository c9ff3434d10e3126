// FP8 E4M3 instances of the tcgen05 forward kernel (d = 128; causal or not).
#include "attn_tc_sm103.cuh"

namespace attn {

cudaError_t launch_tc_e4m3(const TcParams& p, int d, bool causal, int num_sms, cudaStream_t stream) {
  if (d == 128) return causal ? launch_tc<TcCfg<true, 128, true>>(p, num_sms, stream) : launch_tc<TcCfg<true, 128, false>>(p, num_sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn

#ifdef ATTN_TRACE
// Trace builds only: select the traced CTA (cta >= 0) and/or read the stamps of the last launch.
extern "C" int attn_trace_e4m3(unsigned long long* host, int cta) {
  if (cta >= 0) return static_cast<int>(cudaMemcpyToSymbol(attn::g_attn_trace_cta, &cta, sizeof(int)));
  return static_cast<int>(cudaMemcpyFromSymbol(host, attn::g_attn_trace, sizeof(attn::g_attn_trace)));
}
#endif

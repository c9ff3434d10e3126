// Split-KV merge ("Kernels and Memory in LLM Inference", Flash-Decoding: each
// chunk of the keys yields a partial result with its own running max and sum;
// the partials are rescaled by their log-sum-exp and added).  Split s of a row
// holds O_s (already divided by its own l_s) and L_s = m_s + ln l_s, so
//   L = ln sum_s exp(L_s),   O = sum_s exp(L_s - L) O_s.
// One warp per row; lane i owns features [i*d/32, (i+1)*d/32).
#include <cuda_bf16.h>

#include "attn_kernels.h"

namespace attn {
namespace {

template <int D>
__global__ void __launch_bounds__(128) split_combine_kernel(const CombineParams p) {
  constexpr int F = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long r = static_cast<long long>(blockIdx.x) * 4 + warp;
  if (r >= p.rows) return;
  float lmax = -INFINITY;
  for (int s = 0; s < p.n_splits; ++s) lmax = fmaxf(lmax, p.part_l[static_cast<size_t>(s) * p.rows + r]);
  float acc[F];
#pragma unroll
  for (int i = 0; i < F; ++i) acc[i] = 0.f;
  float den = 0.f;
  for (int s = 0; s < p.n_splits; ++s) {
    const size_t pr = static_cast<size_t>(s) * p.rows + r;
    const float wgt = __expf(p.part_l[pr] - lmax);
    den += wgt;
    const float* src = p.part_o + pr * D + lane * F;
    if constexpr (F == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      acc[0] = fmaf(wgt, v.x, acc[0]);
      acc[1] = fmaf(wgt, v.y, acc[1]);
      acc[2] = fmaf(wgt, v.z, acc[2]);
      acc[3] = fmaf(wgt, v.w, acc[3]);
    } else {
      const float2 v = *reinterpret_cast<const float2*>(src);
      acc[0] = fmaf(wgt, v.x, acc[0]);
      acc[1] = fmaf(wgt, v.y, acc[1]);
    }
  }
  const float inv = 1.f / den;
  __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.o) + static_cast<size_t>(r) * D + lane * F;
  if constexpr (F == 4) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
    uint2 u;
    u.x = *reinterpret_cast<const unsigned*>(&a);
    u.y = *reinterpret_cast<const unsigned*>(&b);
    *reinterpret_cast<uint2*>(dst) = u;
  } else {
    *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
  }
  if (lane == 0) p.lse[r] = lmax + logf(den);
}

}  // namespace

cudaError_t launch_split_combine(const CombineParams& p, int d, cudaStream_t stream) {
  const long long blocks = (static_cast<long long>(p.rows) + 3) / 4;
  if (d == 128) split_combine_kernel<128><<<dim3(static_cast<unsigned>(blocks)), dim3(128), 0, stream>>>(p);
  else if (d == 64) split_combine_kernel<64><<<dim3(static_cast<unsigned>(blocks)), dim3(128), 0, stream>>>(p);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace attn

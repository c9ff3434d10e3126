// FlashAttention-2 forward for fp32 inputs on the CUDA cores (exact FFMA).
//
// Same method as the tensor-core kernels ("FlashAttention-2 from PyTorch to
// Triton": per query row, stream key tiles, running max m and sum l, an
// unnormalised O rescaled by exp(m_old - m_new), one division by l at the end,
// L = m + log l), laid out for fp32: each query row is owned by TPR = d / 32
// neighbouring threads (one for d <= 32), each holding 32 features of q and O;
// a dot product is a per-thread partial sum reduced across the TPR lanes with
// shuffles -- the quad reduction of "1.8x Faster Attention on an RTX 5080"
// ("Online softmax, one strip at a time"), applied to features instead of keys.
// Key/value tiles of 32 rows are staged in shared memory and read as warp
// broadcasts.  Used for the fp32 interface; the bf16/e4m3 paths use tcgen05.
#include "attn_kernels.h"

namespace attn {
namespace {

constexpr int kThreads = 128;
constexpr int kKeyTile = 32;

template <int D, bool kCausal>
__global__ void __launch_bounds__(kThreads) attn_fwd_simt_f32_kernel(const SimtParams p) {
  constexpr int DPT = D < 32 ? D : 32;  // features per thread
  constexpr int TPR = D / DPT;          // threads per query row
  constexpr int ROWS = kThreads / TPR;  // query rows per CTA
  __shared__ float sk[kKeyTile][D];
  __shared__ float sv[kKeyTile][D];

  const int N = p.N;
  const int n_rb = (N + ROWS - 1) / ROWS;
  const int bh = blockIdx.x / n_rb;
  const int row0 = (blockIdx.x % n_rb) * ROWS;
  const int tid = threadIdx.x;
  const int row = row0 + tid / TPR;
  const int off = (tid % TPR) * DPT;
  const bool live = row < N;
  const size_t head = static_cast<size_t>(bh) * N * D;
  const size_t kv_head = static_cast<size_t>(kv_head_index(bh, p.H, p.kv_group)) * N * D;

  float q[DPT], o[DPT];
#pragma unroll
  for (int i = 0; i < DPT; ++i) {
    q[i] = live ? p.q[head + static_cast<size_t>(row) * D + off + i] : 0.f;
    o[i] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int n_keys = kCausal ? min(N, row0 + ROWS) : N;

  for (int k0 = 0; k0 < n_keys; k0 += kKeyTile) {
    __syncthreads();
    for (int e = tid; e < kKeyTile * D; e += kThreads) {
      const int r = e / D, c = e % D;
      const bool in = k0 + r < N;
      const size_t g = kv_head + static_cast<size_t>(k0 + r) * D + c;
      sk[r][c] = in ? p.k[g] : 0.f;
      sv[r][c] = in ? p.v[g] : 0.f;
    }
    __syncthreads();
    float s[kKeyTile];
#pragma unroll
    for (int c = 0; c < kKeyTile; ++c) {
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < DPT; ++i) part = fmaf(q[i], sk[c][off + i], part);
#pragma unroll
      for (int w = 1; w < TPR; w <<= 1) part += __shfl_xor_sync(0xffffffffu, part, w);
      const int key = k0 + c;
      const bool keep = key < N && (!kCausal || key <= row);
      s[c] = keep ? part * p.scale_log2 : -INFINITY;
    }
    float mx = s[0];
#pragma unroll
    for (int c = 1; c < kKeyTile; ++c) mx = fmaxf(mx, s[c]);
    const float m_new = fmaxf(m, mx);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = exp2f(m - m_use);
    float rs = 0.f;
#pragma unroll
    for (int c = 0; c < kKeyTile; ++c) {
      s[c] = exp2f(s[c] - m_use);
      rs += s[c];
    }
    l = l * alpha + rs;
#pragma unroll
    for (int i = 0; i < DPT; ++i) {
      float acc = o[i] * alpha;
#pragma unroll
      for (int c = 0; c < kKeyTile; ++c) acc = fmaf(s[c], sv[c][off + i], acc);
      o[i] = acc;
    }
    m = m_new;
  }

  if (live) {
    const float inv = 1.f / l;
    float* dst = p.o + head + static_cast<size_t>(row) * D + off;
#pragma unroll
    for (int i = 0; i < DPT; ++i) dst[i] = o[i] * inv;
    if (off == 0) p.lse[static_cast<size_t>(bh) * N + row] = (m + log2f(l)) * 0.69314718055994530942f;
  }
}

template <int D, bool kCausal>
cudaError_t launch_d(const SimtParams& p, cudaStream_t stream) {
  constexpr int DPT = D < 32 ? D : 32;
  constexpr int ROWS = kThreads / (D / DPT);
  const long long n_rb = (p.N + ROWS - 1) / ROWS;
  const long long grid = n_rb * p.BH;
  attn_fwd_simt_f32_kernel<D, kCausal><<<dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_c(const SimtParams& p, bool causal, cudaStream_t stream) {
  return causal ? launch_d<D, true>(p, stream) : launch_d<D, false>(p, stream);
}

}  // namespace

cudaError_t launch_simt_f32(const SimtParams& p, int d, bool causal, cudaStream_t stream) {
  switch (d) {
    case 16: return launch_c<16>(p, causal, stream);
    case 32: return launch_c<32>(p, causal, stream);
    case 64: return launch_c<64>(p, causal, stream);
    case 128: return launch_c<128>(p, causal, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn

// Internal interface between the C-ABI layer (attn_api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

// Sets a kernel's dynamic shared-memory limit on the current device, once per
// device: `done` (one per kernel instantiation) records the devices already
// set (ordinals >= 64 are set on every call).  A repeated set from another
// thread is harmless.
template <class Kernel>
cudaError_t smem_opt_in_once(Kernel kern, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Arguments of the tensor-core forward kernels (bf16 and e4m3 inputs).
// Q, K, V are [B, H, N, d] row-major and reached only through the TMA
// descriptors; O ([B, H, N, d] bf16) and L ([B, H, N] fp32) are written with
// plain stores.
struct TcParams {
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  void* o;              // bf16 [BH, N, d]
  float* lse;           // fp32 [BH, N], natural log
  int* status;          // device status word (timeouts)
  int BH;               // B * H (query heads)
  int H;                // query heads per batch entry
  int kv_group;         // query heads per K/V head (grouped-query attention; 1 = multi-head):
                        //   K/V are [B, H / kv_group, N, d] and query head h reads K/V head h / kv_group
  int N;                // sequence length (queries = keys)
  int n_pairs;          // ceil(N / 256): CTAs per head (two 128-row query tiles each)
  float scale_log2;     // softmax scale * log2(e) * q_descale * k_descale
  float o_scale;        // multiplies O after the division by l (v_descale for e4m3, 1 for bf16)
  unsigned long long timeout_ns;
  // Split-KV (non-causal only): the key tiles are cut into n_splits ranges of
  // kt_per_split tiles; each (query tile pair, range) is a separate work item
  // whose normalised O (fp32) and L go to part_o [n_splits, BH, N, d] and
  // part_l [n_splits, BH, N].  n_splits == 1 and part_o == nullptr: O and L are
  // written directly.
  int n_splits;
  int kt_per_split;
  float* part_o;
  float* part_l;
};

// Arguments of the split-KV combine kernel.
struct CombineParams {
  const float* part_o;  // [n_splits, rows, d]
  const float* part_l;  // [n_splits, rows]
  void* o;              // bf16 [rows, d]
  float* lse;           // fp32 [rows]
  int rows;             // B * H * N
  int n_splits;
};

// Arguments of the SIMT fp32 forward kernel.
struct SimtParams {
  const float* q;
  const float* k;
  const float* v;
  float* o;
  float* lse;
  int BH;
  int H;                // query heads per batch entry
  int kv_group;         // query heads per K/V head (K/V are [B, H / kv_group, N, d])
  int N;
  float scale_log2;     // softmax scale * log2(e)
};

// K/V head (over B * H_kv) read by query head bh (over B * H) under grouped-query
// attention: groups of kv_group consecutive query heads share one K/V head.
__host__ __device__ __forceinline__ int kv_head_index(int bh, int H, int kv_group) {
  return kv_group == 1 ? bh : (bh / H) * (H / kv_group) + (bh % H) / kv_group;
}

// Arguments of the backward kernels (bf16, d = 64 or 128).
struct BwdParams {
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_do;
  CUtensorMap tm_dqacc; // fp32 [BH, N, d] dQ accumulator (TMA reduce-add target)
  CUtensorMap tm_dv;    // bf16 [BH, N, d] dV, 32-row boxes (TMA store target)
  CUtensorMap tm_dk;    // bf16 [BH, N, d] dK, 32-row boxes
  const void* o;        // bf16 [BH, N, d] (forward output)
  const void* dout;     // bf16 [BH, N, d] (upstream gradient dO)
  const float* lse;     // fp32 [BH, N], natural log (forward's L)
  float* lse2;          // fp32 [BH, n_pad] workspace: -L * log2 e per row, -inf on padding rows
  float* drow;          // fp32 [BH, n_pad] workspace: -D, D = rowsum(dO * O), 0 on padding rows
                        //   (n_pad = N rounded up to a multiple of 128; negated so the pass adds them)
  float* dq_acc;        // fp32 [BH, N, d] workspace: dQ accumulator
  void* dq;             // bf16 [BH, N, d]
  void* dk;             // bf16 [BH, N, d]
  void* dv;             // bf16 [BH, N, d]
  int* status;          // device status word (timeouts)
  int BH;
  int N;
  float scale;          // softmax scale
  float scale_log2;     // scale * log2(e)
  unsigned long long timeout_ns;
};

// Launchers (defined next to their kernels).  Return the launch error.
// The tensor-core kernels are persistent: min(#work items, num_sms) CTAs.
cudaError_t launch_tc_bf16(const TcParams& p, int d, bool causal, int num_sms, cudaStream_t stream);
cudaError_t launch_tc_e4m3(const TcParams& p, int d, bool causal, int num_sms, cudaStream_t stream);
// e4m3 with the split exponential (one exponential pair in four by polynomial).
cudaError_t launch_tc_e4m3_poly(const TcParams& p, int d, bool causal, int num_sms, cudaStream_t stream);
cudaError_t launch_simt_f32(const SimtParams& p, int d, bool causal, cudaStream_t stream);
cudaError_t launch_split_combine(const CombineParams& p, int d, cudaStream_t stream);
// Backward: D and the zeroed dQ accumulator, the tensor-core pass, dQ to bf16.
cudaError_t launch_bwd(const BwdParams& p, int d, bool causal, cudaStream_t stream);

}  // namespace attn

// C-ABI layer of libattn_fa2.so: argument validation, TMA descriptor encoding,
// kernel selection and launch, device status word.  The entry points are
// declared (with their contracts) in include/attn_fa2.h.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "attn_fa2.h"
#include "attn_kernels.h"
#include "ptx_sm103.cuh"

namespace {

// Device status word: a kernel that gives up on a wait writes ATTN_ERR_TIMEOUT here.
__device__ int g_attn_status = 0;

thread_local char g_last_error[256] = "";
uint64_t g_wait_limit_ns = 2000000000ull;
std::atomic<int> g_poly_exp2{0};  // attn_set_poly_exp2

int fail(int status, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Address of the status word on the current device (looked up once per device).
int status_ptr(int** out) {
  constexpr int kMaxDev = 64;
  static int* cache[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDev) return fail(ATTN_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_status);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
    cache[dev] = static_cast<int*>(p);
  }
  *out = cache[dev];
  return ATTN_OK;
}

// Number of SMs of the current device (looked up once per device).
int num_sms(int* out) {
  constexpr int kMaxDev = 64;
  static int cache[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDev) return fail(ATTN_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(multiprocessor count)");
    cache[dev] = n;
  }
  *out = cache[dev];
  return ATTN_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Recently encoded tensor maps of this thread.  A map is a pure function of
// its arguments (address, element type, sizes), so an entry stays valid for
// as long as it is in the table, whatever happened to the memory meanwhile.
struct MapCacheEntry {
  const void* base;
  CUtensorMapDataType dt;
  int elem_bytes, BH, N, d, box_rows;
  CUtensorMap map;
};
constexpr int kMapCacheSize = 8;
thread_local MapCacheEntry g_map_cache[kMapCacheSize];
thread_local int g_map_cache_used = 0, g_map_cache_next = 0;

int encode_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, int BH, int N, int d,
               int box_rows);

// 3-D map over a [BH, N, d] tensor: dims (d, N, BH), boxes of `box_rows` rows
// (128 by default) of one 128-byte column block, 128-byte swizzle, zero fill
// outside [0, N) on loads (stores are clipped there).  Encoded once per
// distinct argument set (per thread), then reused.
int make_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, int BH, int N, int d,
             int box_rows = 128) {
  for (int i = 0; i < g_map_cache_used; ++i) {
    const MapCacheEntry& e = g_map_cache[i];
    if (e.base == base && e.dt == dt && e.elem_bytes == elem_bytes && e.BH == BH && e.N == N && e.d == d &&
        e.box_rows == box_rows) {
      *map = e.map;
      return ATTN_OK;
    }
  }
  const int st = encode_map(map, base, dt, elem_bytes, BH, N, d, box_rows);
  if (st != ATTN_OK) return st;
  MapCacheEntry& e = g_map_cache[g_map_cache_next];
  e = MapCacheEntry{base, dt, elem_bytes, BH, N, d, box_rows, *map};
  g_map_cache_next = (g_map_cache_next + 1) % kMapCacheSize;
  if (g_map_cache_used < kMapCacheSize) ++g_map_cache_used;
  return ATTN_OK;
}

int encode_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, int BH, int N, int d,
               int box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * elem_bytes,
                                 static_cast<cuuint64_t>(N) * d * elem_bytes};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elem_bytes), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", int(r));
  return ATTN_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_common(const void* q, const void* k, const void* v, const void* o, const float* lse, int B, int H,
                 int N, int d, float scale, int causal) {
  if (!q || !k || !v || !o || !lse) return fail(ATTN_ERR_INVALID_ARG, "null pointer argument");
  if (B < 1 || H < 1 || N < 1 || d < 1)
    return fail(ATTN_ERR_INVALID_ARG, "sizes must be >= 1 (B=%d H=%d N=%d d=%d)", B, H, N, d);
  if (static_cast<long long>(B) * H > 0x7fffffffLL) return fail(ATTN_ERR_INVALID_ARG, "B*H overflows int");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0 (got %g)", double(scale));
  if (causal != 0 && causal != 1) return fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1 (got %d)", causal);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return fail(ATTN_ERR_MISALIGNED, "q, k, v and o must be 16-byte aligned");
  if (!aligned(lse, 4)) return fail(ATTN_ERR_MISALIGNED, "lse must be 4-byte aligned");
  return ATTN_OK;
}

constexpr float kLog2e = 1.4426950408889634f;

// Split-KV plan: the number of key ranges (resolved from `req`, 0 = enough
// work items to fill every SM), the key tiles per range, and the workspace bytes.
struct SplitPlan {
  int splits, kt_per;
  size_t ws_bytes, part_l_offset;
};

int plan_split(int B, int H, int N, int d, int req, SplitPlan* out) {
  if (req < 0) return fail(ATTN_ERR_INVALID_ARG, "n_splits must be >= 0 (got %d)", req);
  const long long n_kt = (static_cast<long long>(N) + 127) / 128;
  const long long items = static_cast<long long>(B) * H * ((static_cast<long long>(N) + 255) / 256);
  long long s = req;
  if (s == 0) {
    int sms = 0;
    int st = num_sms(&sms);
    if (st != ATTN_OK) return st;
    s = items >= sms ? 1 : (sms + items - 1) / items;
  }
  if (s > n_kt) s = n_kt;
  if (s < 1) s = 1;
  const long long kt_per = (n_kt + s - 1) / s;
  s = (n_kt + kt_per - 1) / kt_per;  // no empty key range
  out->splits = static_cast<int>(s);
  out->kt_per = static_cast<int>(kt_per);
  const size_t rows = static_cast<size_t>(B) * H * N;
  const size_t o_bytes = (s * rows * static_cast<size_t>(d) * 4 + 255) / 256 * 256;
  out->part_l_offset = o_bytes;
  out->ws_bytes = s == 1 ? 0 : o_bytes + s * rows * 4;
  return ATTN_OK;
}

int run_tc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           float scale, float qds, float kds, float vds, int causal, bool fp8, cudaStream_t stream,
           int n_splits = 1, int kt_per = 0, float* part_o = nullptr, float* part_l = nullptr, int Hkv = 0) {
  if (Hkv == 0) Hkv = H;
  if (fp8 ? (d != 128) : (d != 64 && d != 128))
    return fail(ATTN_ERR_UNSUPPORTED, "%s tensor-core path supports d in %s (got %d)", fp8 ? "e4m3" : "bf16",
                fp8 ? "{128}" : "{64, 128}", d);
  if (!aligned(o, 32)) return fail(ATTN_ERR_MISALIGNED, "o must be 32-byte aligned for bf16/e4m3 inputs");
  const int BH = B * H;
  const long long n_pairs = (static_cast<long long>(N) + 255) / 256;
  if (n_pairs * BH > 0x7fffffffLL) return fail(ATTN_ERR_UNSUPPORTED, "grid too large (B*H*ceil(N/256))");
  attn::TcParams p;
  std::memset(&p, 0, sizeof(p));
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int eb = fp8 ? 1 : 2;
  int st;
  if ((st = make_map(&p.tm_q, q, dt, eb, BH, N, d)) != ATTN_OK) return st;
  if ((st = make_map(&p.tm_k, k, dt, eb, B * Hkv, N, d)) != ATTN_OK) return st;
  if ((st = make_map(&p.tm_v, v, dt, eb, B * Hkv, N, d)) != ATTN_OK) return st;
  if ((st = status_ptr(&p.status)) != ATTN_OK) return st;
  p.o = o;
  p.lse = lse;
  p.BH = BH;
  p.H = H;
  p.kv_group = H / Hkv;
  p.N = N;
  p.n_pairs = static_cast<int>(n_pairs);
  p.scale_log2 = scale * kLog2e * qds * kds;
  p.o_scale = vds;
  p.timeout_ns = g_wait_limit_ns;
  p.n_splits = n_splits;
  p.kt_per_split = n_splits == 1 ? (N + 127) / 128 : kt_per;
  p.part_o = part_o;
  p.part_l = part_l;
  if (n_pairs * BH * n_splits > 0x7fffffffLL) return fail(ATTN_ERR_UNSUPPORTED, "too many work items");
  int sms = 0;
  if ((st = num_sms(&sms)) != ATTN_OK) return st;
  cudaError_t e = !fp8 ? attn::launch_tc_bf16(p, d, causal != 0, sms, stream)
                 : g_poly_exp2.load(std::memory_order_relaxed) ? attn::launch_tc_e4m3_poly(p, d, causal != 0, sms, stream)
                                                               : attn::launch_tc_e4m3(p, d, causal != 0, sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return ATTN_OK;
}

int run_f32(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
            float scale, int causal, cudaStream_t stream, int Hkv = 0) {
  if (Hkv == 0) Hkv = H;
  if (d != 16 && d != 32 && d != 64 && d != 128)
    return fail(ATTN_ERR_UNSUPPORTED, "fp32 path supports d in {16, 32, 64, 128} (got %d)", d);
  attn::SimtParams p;
  p.q = static_cast<const float*>(q);
  p.k = static_cast<const float*>(k);
  p.v = static_cast<const float*>(v);
  p.o = static_cast<float*>(o);
  p.lse = lse;
  p.BH = B * H;
  p.H = H;
  p.kv_group = H / Hkv;
  p.N = N;
  p.scale_log2 = scale * kLog2e;
  cudaError_t e = attn::launch_simt_f32(p, d, causal != 0, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return ATTN_OK;
}

// The requirements of the kernel that serves `dtype` (head dimension, output
// alignment, grid size), checked without launching anything; run_tc and
// run_f32 check the same before their launches.
int check_kernel(const void* o, int B, int H, int N, int d, int dtype) {
  switch (dtype) {
    case ATTN_F32:
      if (d != 16 && d != 32 && d != 64 && d != 128)
        return fail(ATTN_ERR_UNSUPPORTED, "fp32 path supports d in {16, 32, 64, 128} (got %d)", d);
      return ATTN_OK;
    case ATTN_BF16:
    case ATTN_E4M3: {
      const bool fp8 = dtype == ATTN_E4M3;
      if (fp8 ? (d != 128) : (d != 64 && d != 128))
        return fail(ATTN_ERR_UNSUPPORTED, "%s tensor-core path supports d in %s (got %d)", fp8 ? "e4m3" : "bf16",
                    fp8 ? "{128}" : "{64, 128}", d);
      if (!aligned(o, 32)) return fail(ATTN_ERR_MISALIGNED, "o must be 32-byte aligned for bf16/e4m3 inputs");
      const long long n_pairs = (static_cast<long long>(N) + 255) / 256;
      if (n_pairs * B * H > 0x7fffffffLL) return fail(ATTN_ERR_UNSUPPORTED, "grid too large (B*H*ceil(N/256))");
      return ATTN_OK;
    }
    default: return fail(ATTN_ERR_INVALID_ARG, "unknown dtype %d", dtype);
  }
}

int dispatch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
             float scale, float qds, float kds, float vds, int causal, int dtype, cudaStream_t stream,
             int Hkv = 0) {
  int st = check_common(q, k, v, o, lse, B, H, N, d, scale, causal);
  if (st != ATTN_OK) return st;
  if ((st = check_kernel(o, B, H, N, d, dtype)) != ATTN_OK) return st;
  switch (dtype) {
    case ATTN_F32: return run_f32(q, k, v, o, lse, B, H, N, d, scale, causal, stream, Hkv);
    case ATTN_BF16:
      return run_tc(q, k, v, o, lse, B, H, N, d, scale, 1.f, 1.f, 1.f, causal, false, stream, 1, 0, nullptr,
                    nullptr, Hkv);
    case ATTN_E4M3:
      return run_tc(q, k, v, o, lse, B, H, N, d, scale, qds, kds, vds, causal, true, stream, 1, 0, nullptr,
                    nullptr, Hkv);
    default: return fail(ATTN_ERR_INVALID_ARG, "unknown dtype %d", dtype);
  }
}

bool good_descale(float x) { return x > 0.f && std::isfinite(x); }

// One thread waits on an mbarrier that is never signalled; the bounded wait
// gives up after limit_ns and writes the timeout status.
__global__ void selftest_wait_kernel(int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    attn::mbar_init(attn::smem_u32(&bar), 1);
    attn::fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)attn::mbar_wait(attn::smem_u32(&bar), 0, status, limit_ns);
}

}  // namespace

namespace attn {
// Records `msg` as this thread's last error and returns `status` (for other
// translation units of the library).
int set_last_error(int status, const char* msg) { return fail(status, "%s", msg); }
}  // namespace attn

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
             float scale, int causal, int dtype, void* stream) {
  g_last_error[0] = '\0';
  return dispatch(q, k, v, o, lse, B, H, N, d, scale, 1.f, 1.f, 1.f, causal, dtype,
                  static_cast<cudaStream_t>(stream));
}

int attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, float q_descale, float k_descale, float v_descale, int causal, void* stream) {
  g_last_error[0] = '\0';
  if (!good_descale(q_descale) || !good_descale(k_descale) || !good_descale(v_descale))
    return fail(ATTN_ERR_INVALID_ARG, "descales must be finite and > 0");
  return dispatch(q, k, v, o, lse, B, H, N, d, scale, q_descale, k_descale, v_descale, causal, ATTN_E4M3,
                  static_cast<cudaStream_t>(stream));
}

int attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N,
                 int d, float scale, float q_descale, float k_descale, float v_descale, int causal, int dtype,
                 void* stream) {
  g_last_error[0] = '\0';
  if (H_kv < 1 || H < 1 || H % H_kv != 0)
    return fail(ATTN_ERR_INVALID_ARG, "H (%d) must be a positive multiple of H_kv (%d)", H, H_kv);
  const bool fp8 = dtype == ATTN_E4M3;
  if (fp8 && (!good_descale(q_descale) || !good_descale(k_descale) || !good_descale(v_descale)))
    return fail(ATTN_ERR_INVALID_ARG, "descales must be finite and > 0");
  return dispatch(q, k, v, o, lse, B, H, N, d, scale, fp8 ? q_descale : 1.f, fp8 ? k_descale : 1.f,
                  fp8 ? v_descale : 1.f, causal, dtype, static_cast<cudaStream_t>(stream), H_kv);
}

int attn_fwd_host(const void* h_q, const void* h_k, const void* h_v, void* h_o, float* h_lse, void* d_q,
                  void* d_k, void* d_v, void* d_o, float* d_lse, int B, int H, int N, int d, float scale,
                  float q_descale, float k_descale, float v_descale, int causal, int dtype, void* stream) {
  g_last_error[0] = '\0';
  if (!h_q || !h_k || !h_v || !h_o || !h_lse) return fail(ATTN_ERR_INVALID_ARG, "null host pointer");
  int st = check_common(d_q, d_k, d_v, d_o, d_lse, B, H, N, d, scale, causal);
  if (st != ATTN_OK) return st;
  if (dtype != ATTN_F32 && dtype != ATTN_BF16 && dtype != ATTN_E4M3)
    return fail(ATTN_ERR_INVALID_ARG, "unknown dtype %d", dtype);
  if (dtype == ATTN_E4M3 && (!good_descale(q_descale) || !good_descale(k_descale) || !good_descale(v_descale)))
    return fail(ATTN_ERR_INVALID_ARG, "descales must be finite and > 0");
  // Everything the forward would reject is rejected before the first copy is enqueued.
  if ((st = check_kernel(d_o, B, H, N, d, dtype)) != ATTN_OK) return st;
  const size_t in_elem = dtype == ATTN_F32 ? 4 : (dtype == ATTN_BF16 ? 2 : 1);
  const size_t out_elem = dtype == ATTN_F32 ? 4 : 2;
  const size_t rows = static_cast<size_t>(B) * H * N;
  const size_t in_bytes = rows * d * in_elem;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if ((e = cudaMemcpyAsync(d_q, h_q, in_bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess) return cuda_fail(e, "copy q");
  if ((e = cudaMemcpyAsync(d_k, h_k, in_bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess) return cuda_fail(e, "copy k");
  if ((e = cudaMemcpyAsync(d_v, h_v, in_bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess) return cuda_fail(e, "copy v");
  const bool fp8 = dtype == ATTN_E4M3;
  st = dispatch(d_q, d_k, d_v, d_o, d_lse, B, H, N, d, scale, fp8 ? q_descale : 1.f, fp8 ? k_descale : 1.f,
                fp8 ? v_descale : 1.f, causal, dtype, s);
  if (st != ATTN_OK) return st;
  if ((e = cudaMemcpyAsync(h_o, d_o, rows * d * out_elem, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(e, "copy o");
  if ((e = cudaMemcpyAsync(h_lse, d_lse, rows * sizeof(float), cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(e, "copy lse");
  return ATTN_OK;
}

int attn_get_device_status(void* stream) {
  g_last_error[0] = '\0';
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int* dptr = nullptr;
  int st = status_ptr(&dptr);
  if (st != ATTN_OK) return st;
  int h = 0;
  if ((e = cudaMemcpy(&h, dptr, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "read status");
  if (h != 0) {
    const int zero = 0;
    if ((e = cudaMemcpy(dptr, &zero, sizeof(int), cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "clear status");
    return fail(ATTN_ERR_TIMEOUT, "a kernel gave up on a device-side wait");
  }
  return ATTN_OK;
}

int attn_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  g_last_error[0] = '\0';
  if (limit_ns < 1000000ull) return fail(ATTN_ERR_INVALID_ARG, "limit must be >= 1e6 ns");
  int* status = nullptr;
  int st = status_ptr(&status);
  if (st != ATTN_OK) return st;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, limit_ns);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return ATTN_OK;
}

int attn_fwd_split_plan(int B, int H, int N, int d, int n_splits, int* splits_out, size_t* workspace_bytes_out) {
  g_last_error[0] = '\0';
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128))
    return fail(ATTN_ERR_INVALID_ARG, "sizes must be >= 1 and d in {64, 128}");
  SplitPlan plan;
  int st = plan_split(B, H, N, d, n_splits, &plan);
  if (st != ATTN_OK) return st;
  if (splits_out) *splits_out = plan.splits;
  if (workspace_bytes_out) *workspace_bytes_out = plan.ws_bytes;
  return ATTN_OK;
}

int attn_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                   float scale, float q_descale, float k_descale, float v_descale, int causal, int dtype,
                   int n_splits, void* workspace, size_t workspace_bytes, void* stream) {
  g_last_error[0] = '\0';
  int st = check_common(q, k, v, o, lse, B, H, N, d, scale, causal);
  if (st != ATTN_OK) return st;
  if (dtype != ATTN_BF16 && dtype != ATTN_E4M3)
    return fail(ATTN_ERR_UNSUPPORTED, "split-KV runs on the tensor-core paths (bf16, e4m3) only");
  if (causal) return fail(ATTN_ERR_UNSUPPORTED, "split-KV is implemented for non-causal attention only");
  const bool fp8 = dtype == ATTN_E4M3;
  if (fp8 && (!good_descale(q_descale) || !good_descale(k_descale) || !good_descale(v_descale)))
    return fail(ATTN_ERR_INVALID_ARG, "descales must be finite and > 0");
  SplitPlan plan;
  if ((st = plan_split(B, H, N, d, n_splits, &plan)) != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float qds = fp8 ? q_descale : 1.f, kds = fp8 ? k_descale : 1.f, vds = fp8 ? v_descale : 1.f;
  if (plan.splits == 1) return run_tc(q, k, v, o, lse, B, H, N, d, scale, qds, kds, vds, 0, fp8, s);
  if (static_cast<long long>(B) * H * N > 0x7fffffffLL) return fail(ATTN_ERR_UNSUPPORTED, "B*H*N too large for split-KV");
  if (!workspace) return fail(ATTN_ERR_INVALID_ARG, "workspace is null (%zu bytes needed)", plan.ws_bytes);
  if (workspace_bytes < plan.ws_bytes)
    return fail(ATTN_ERR_INVALID_ARG, "workspace too small: %zu bytes given, %zu needed", workspace_bytes,
                plan.ws_bytes);
  if (!aligned(workspace, 256)) return fail(ATTN_ERR_MISALIGNED, "workspace must be 256-byte aligned");
  float* part_o = static_cast<float*>(workspace);
  float* part_l = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.part_l_offset);
  st = run_tc(q, k, v, o, lse, B, H, N, d, scale, qds, kds, vds, 0, fp8, s, plan.splits, plan.kt_per, part_o, part_l);
  if (st != ATTN_OK) return st;
  attn::CombineParams cp;
  cp.part_o = part_o;
  cp.part_l = part_l;
  cp.o = o;
  cp.lse = lse;
  cp.rows = B * H * N;
  cp.n_splits = plan.splits;
  cudaError_t e = attn::launch_split_combine(cp, d, s);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return ATTN_OK;
}

int attn_bwd_workspace_size(int B, int H, int N, int d, size_t* bytes_out) {
  g_last_error[0] = '\0';
  if (!bytes_out) return fail(ATTN_ERR_INVALID_ARG, "bytes_out is null");
  if (B < 1 || H < 1 || N < 1) return fail(ATTN_ERR_INVALID_ARG, "sizes must be >= 1 (B=%d H=%d N=%d)", B, H, N);
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "the backward supports d = 64 or 128 (got %d)", d);
  const size_t rows = static_cast<size_t>(B) * H * N;
  const size_t prows = static_cast<size_t>(B) * H * ((static_cast<size_t>(N) + 127) / 128 * 128);
  // dQ accumulator (fp32, rows x d), then L log2 e and D (fp32, one per row with
  // each head padded to whole 128-row tiles), each 256-byte aligned.
  const size_t acc = (rows * d * sizeof(float) + 255) / 256 * 256;
  *bytes_out = acc + 2 * ((prows * sizeof(float) + 255) / 256 * 256);
  return ATTN_OK;
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
             void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
             float scale, int causal, void* stream) {
  g_last_error[0] = '\0';
  int st = check_common(q, k, v, o, lse, B, H, N, d, scale, causal);
  if (st != ATTN_OK) return st;
  if (!dout || !dq || !dk || !dv || !workspace) return fail(ATTN_ERR_INVALID_ARG, "null pointer argument");
  size_t need = 0;
  if ((st = attn_bwd_workspace_size(B, H, N, d, &need)) != ATTN_OK) return st;
  if (workspace_bytes < need)
    return fail(ATTN_ERR_INVALID_ARG, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, need);
  if (!aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16))
    return fail(ATTN_ERR_MISALIGNED, "dout, dq, dk and dv must be 16-byte aligned");
  if (!aligned(workspace, 256)) return fail(ATTN_ERR_MISALIGNED, "workspace must be 256-byte aligned");
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 65535) return fail(ATTN_ERR_UNSUPPORTED, "B*H must be <= 65535 for the backward grid (got %lld)", BH);
  attn::BwdParams p;
  const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if ((st = make_map(&p.tm_q, q, dt, 2, static_cast<int>(BH), N, d)) != ATTN_OK) return st;
  if ((st = make_map(&p.tm_k, k, dt, 2, static_cast<int>(BH), N, d)) != ATTN_OK) return st;
  if ((st = make_map(&p.tm_v, v, dt, 2, static_cast<int>(BH), N, d)) != ATTN_OK) return st;
  if ((st = make_map(&p.tm_do, dout, dt, 2, static_cast<int>(BH), N, d)) != ATTN_OK) return st;
  if ((st = make_map(&p.tm_dqacc, workspace, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, static_cast<int>(BH), N, d)) !=
      ATTN_OK)
    return st;
  // dV and dK leave the kernel as TMA stores of 32-row boxes (one per pass warp).
  if ((st = make_map(&p.tm_dv, dv, dt, 2, static_cast<int>(BH), N, d, 32)) != ATTN_OK) return st;
  if ((st = make_map(&p.tm_dk, dk, dt, 2, static_cast<int>(BH), N, d, 32)) != ATTN_OK) return st;
  if ((st = status_ptr(&p.status)) != ATTN_OK) return st;
  const size_t rows = static_cast<size_t>(BH) * N;
  const size_t prows = static_cast<size_t>(BH) * ((static_cast<size_t>(N) + 127) / 128 * 128);
  const size_t acc_bytes = (rows * d * sizeof(float) + 255) / 256 * 256;
  const size_t vec_bytes = (prows * sizeof(float) + 255) / 256 * 256;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.dq_acc = static_cast<float*>(workspace);
  p.lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + acc_bytes);
  p.drow = reinterpret_cast<float*>(static_cast<char*>(workspace) + acc_bytes + vec_bytes);
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.BH = static_cast<int>(BH);
  p.N = N;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.timeout_ns = g_wait_limit_ns;
  cudaError_t e = attn::launch_bwd(p, d, causal != 0, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  return ATTN_OK;
}

int attn_set_poly_exp2(int on) {
  if (on != 0 && on != 1) return -1;
  return g_poly_exp2.exchange(on);
}

uint64_t attn_set_wait_limit_ns(uint64_t ns) {
  const uint64_t old = g_wait_limit_ns;
  g_wait_limit_ns = ns < 1000000ull ? 1000000ull : ns;
  return old;
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_MISALIGNED: return "misaligned pointer";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

const char* attn_last_error(void) { return g_last_error; }

}  // extern "C"

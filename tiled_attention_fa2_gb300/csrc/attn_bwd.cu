// Attention backward (bf16, d = 64 or 128): dQ, dK, dV from Q, K, V, O, dO and
// the forward's L.
//
// The structure follows the backward the pages outline ("FlashAttention-2 from
// PyTorch to Triton", item 5 of what its first kernel leaves out; "Kernels and
// Memory in LLM Inference", "Training detour (brief)"): a first pass computes
// D = rowsum(dO * O); then, per key tile, the query tiles that see it are
// visited one after the other, P = exp(S - L) is rebuilt on chip, dK and dV
// accumulate in TMEM, and dQ is accumulated in fp32 global memory by TMA
// reduce-adds; a last pass converts dQ to bf16.  With S = scale Q K^T and P its row
// softmax:  dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  dQ = scale dS K,
// dK = scale dS^T Q.
//
// Main kernel, one CTA of 128 threads per (key tile j, b*h): thread r owns key
// row r of dK and dV (TMEM lane r) and query row r of each visited query tile.
// Per query tile i:
//   TMA Q_i, dO_i -> MMA S = Q_i K_j^T and dP = dO_i V_j^T (TMEM) ->
//   threads: P = 2^(S * scale * log2 e - L * log2 e) (masked keys 0),
//   dS = P * (dP - D), both to shared memory as bf16 in the 128-byte swizzled
//   layout -> MMA dV += P^T dO_i, dK += dS^T Q_i (P^T and dS^T are the same bytes
//   read as MN-major A operands), dQ_i' = dS K_j -> threads stage scale dQ_i'
//   in shared memory -> TMA reduce-add into the fp32 dQ accumulator.
// After the last query tile: dK * scale and dV to bf16.
#include <cuda_bf16.h>

#include "attn_kernels.h"
#include "ptx_sm103.cuh"

namespace attn {
namespace {

constexpr int kBwdThreads = 128;
constexpr int kPSBytes = 128 * 128 * 2;  // one [128 query][128 key] bf16 tile (P or dS)

template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = 128 * D * 2;  // one 128-row bf16 tile of Q, K, V or dO
  static constexpr int kBlocks = D / 64;          // 128-byte column blocks per row
  static constexpr int kK = 0, kV = kTileBytes, kQ = 2 * kTileBytes, kDO = 3 * kTileBytes;
  static constexpr int kP = 4 * kTileBytes, kDS = kP + kPSBytes;
  static constexpr int kBar = kDS + kPSBytes;
  static constexpr int kSmemBytes = kBar + 1024 /*barriers*/ + 1024 /*alignment slack*/;
  // TMEM columns: dV | dK | S (then dS K) | dP
  static constexpr uint32_t kColDV = 0, kColDK = D, kColS = 2 * D, kColDP = 2 * D + 128;
  static constexpr uint32_t kIdescQK = make_idesc(1, 128, 128, 0, 0);  // S, dP: both operands K-major
  static constexpr uint32_t kIdescT = make_idesc(1, 128, D, 1, 1);     // dV, dK: A = P^T / dS^T, B = dO / Q
  static constexpr uint32_t kIdescDQ = make_idesc(1, 128, D, 0, 1);    // dS K: A K-major, B MN-major
};

// Bulk tensor reduce-add shared -> global (element type and box from the map),
// tracked by the issuing thread's bulk async-groups.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The source shared memory of every committed group has been read.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Every committed group has completed (its global writes are done).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Byte address of the 16-byte chunk holding columns [8c, 8c + 8) of row r of a
// [128 x 128] bf16 tile stored as two 128-byte-swizzled column blocks (the
// layout TMA writes for a 128 x 64 box with 128-byte swizzle).
__device__ __forceinline__ uint32_t sw128_chunk(uint32_t tile, int r, int c) {
  return tile + (c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// Two 32-lane x 64-column TMEM loads with a single wait (both in one statement,
// so no use of the registers can move above the wait).
__device__ __forceinline__ void tmem_ld64x2_sync(uint32_t ta, uint32_t (&a)[64], uint32_t tb, uint32_t (&b)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%128];\n"
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,"
      "%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,"
      "%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, "
      "[%129];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]), "=r"(a[8]),
        "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(a[16]),
        "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]), "=r"(a[24]),
        "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31]), "=r"(a[32]),
        "=r"(a[33]), "=r"(a[34]), "=r"(a[35]), "=r"(a[36]), "=r"(a[37]), "=r"(a[38]), "=r"(a[39]), "=r"(a[40]),
        "=r"(a[41]), "=r"(a[42]), "=r"(a[43]), "=r"(a[44]), "=r"(a[45]), "=r"(a[46]), "=r"(a[47]), "=r"(a[48]),
        "=r"(a[49]), "=r"(a[50]), "=r"(a[51]), "=r"(a[52]), "=r"(a[53]), "=r"(a[54]), "=r"(a[55]), "=r"(a[56]),
        "=r"(a[57]), "=r"(a[58]), "=r"(a[59]), "=r"(a[60]), "=r"(a[61]), "=r"(a[62]), "=r"(a[63]), "=r"(b[0]),
        "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]),
        "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]), "=r"(b[16]), "=r"(b[17]),
        "=r"(b[18]), "=r"(b[19]), "=r"(b[20]), "=r"(b[21]), "=r"(b[22]), "=r"(b[23]), "=r"(b[24]), "=r"(b[25]),
        "=r"(b[26]), "=r"(b[27]), "=r"(b[28]), "=r"(b[29]), "=r"(b[30]), "=r"(b[31]), "=r"(b[32]), "=r"(b[33]),
        "=r"(b[34]), "=r"(b[35]), "=r"(b[36]), "=r"(b[37]), "=r"(b[38]), "=r"(b[39]), "=r"(b[40]), "=r"(b[41]),
        "=r"(b[42]), "=r"(b[43]), "=r"(b[44]), "=r"(b[45]), "=r"(b[46]), "=r"(b[47]), "=r"(b[48]), "=r"(b[49]),
        "=r"(b[50]), "=r"(b[51]), "=r"(b[52]), "=r"(b[53]), "=r"(b[54]), "=r"(b[55]), "=r"(b[56]), "=r"(b[57]),
        "=r"(b[58]), "=r"(b[59]), "=r"(b[60]), "=r"(b[61]), "=r"(b[62]), "=r"(b[63])
      : "r"(ta), "r"(tb)
      : "memory");
}

// S (or dP) = A B^T for 128 x 128 tiles with d-long rows: both operands K-major.
template <int D>
__device__ __forceinline__ void mma_rows(uint32_t tmem_d, uint32_t a, uint32_t b) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t byte = kk * 32;
    const uint32_t off = (byte / 128) * 16384 + (byte % 128);
    mma_f16_ss_elect(tmem_d, sdesc_sw128(a + off, 16, 1024), sdesc_sw128(b + off, 16, 1024),
                     BwdCfg<D>::kIdescQK, kk > 0);
  }
}

// acc (+)= X^T Y for X = [128 query][128 key] (P or dS) and Y = [128 query][d]
// (dO or Q): contraction over the query rows; X read as an MN-major A operand,
// Y as an MN-major B operand.
template <int D>
__device__ __forceinline__ void mma_t(uint32_t tmem_d, uint32_t x, uint32_t y, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    mma_f16_ss_elect(tmem_d, sdesc_sw128(x + kk * 2048, 16384, 1024), sdesc_sw128(y + kk * 2048, 16384, 1024),
                     BwdCfg<D>::kIdescT, accumulate || kk > 0);
  }
}

// dQ' = dS K_j: contraction over the keys; dS K-major, K_j ([key][d]) MN-major.
template <int D>
__device__ __forceinline__ void mma_dq(uint32_t tmem_d, uint32_t ds, uint32_t k) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t byte = kk * 32;
    const uint32_t off = (byte / 128) * 16384 + (byte % 128);
    mma_f16_ss_elect(tmem_d, sdesc_sw128(ds + off, 16, 1024), sdesc_sw128(k + kk * 2048, 16384, 1024),
                     BwdCfg<D>::kIdescDQ, kk > 0);
  }
}

// D_i = sum_c dO_ic O_ic (fp32), and dQ accumulator rows zeroed.  One warp per row.
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const BwdParams p) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<long long>(p.BH) * p.N) return;
  constexpr int kPer = D / 32;  // elements per lane (2 or 4)
  const __nv_bfloat16* o = reinterpret_cast<const __nv_bfloat16*>(p.o) + row * D + lane * kPer;
  const __nv_bfloat16* g = reinterpret_cast<const __nv_bfloat16*>(p.dout) + row * D + lane * kPer;
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc = fmaf(__bfloat162float(o[e]), __bfloat162float(g[e]), acc);
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (lane == 0) p.drow[row] = acc;
  float* dq = p.dq_acc + row * D + lane * kPer;
#pragma unroll
  for (int e = 0; e < kPer; ++e) dq[e] = 0.f;
}

// dQ (bf16) = the fp32 accumulator, four elements per thread and step.
__global__ void __launch_bounds__(256) attn_bwd_dq_kernel(const BwdParams p, long long n4) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 v = reinterpret_cast<const float4*>(p.dq_acc)[i];
    uint2 out;
    out.x = pack_bf16x2(v.x, v.y);
    out.y = pack_bf16x2(v.z, v.w);
    reinterpret_cast<uint2*>(p.dq)[i] = out;
  }
}

template <int D, bool kCausal>
__global__ void __launch_bounds__(kBwdThreads, 1) attn_bwd_tc_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + C::kBar);
  const uint32_t kv_bar = smem_u32(bars), qd_bar = kv_bar + 8, mma1_bar = kv_bar + 16, mma2_bar = kv_bar + 24,
                 done_bar = kv_bar + 32;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 5);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int N = p.N, n_kt = (N + 127) >> 7;
  const int j = blockIdx.x, bh = blockIdx.y;
  const uint64_t lim = p.timeout_ns;

  if (tid == 0) {
    mbar_init(kv_bar, 1);
    mbar_init(qd_bar, 1);
    mbar_init(mma1_bar, 1);
    mbar_init(mma2_bar, 1);
    mbar_init(done_bar, 1);
    fence_mbarrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_holder);
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t sK = base + C::kK, sV = base + C::kV, sQ = base + C::kQ, sDO = base + C::kDO;
  const uint32_t sP = base + C::kP, sDS = base + C::kDS;

  if (warp == 0) {
    mbar_arrive_expect_tx_elect(kv_bar, 2 * C::kTileBytes);
    for (int b = 0; b < C::kBlocks; ++b) {
      tma_load_3d_elect(sK + b * 16384, &p.tm_k, kv_bar, b * 64, j * 128, bh);
      tma_load_3d_elect(sV + b * 16384, &p.tm_v, kv_bar, b * 64, j * 128, bh);
    }
  }
  bool ok = __syncthreads_and(mbar_wait(kv_bar, 0, p.status, lim));

  const float sl2 = p.scale_log2;
  const int key_r = j * 128 + tid;  // this thread's key row (dK, dV)
  const int i0 = kCausal ? j : 0;   // first query tile that sees key tile j
  // Q_i and dO_i of query tile i into shared memory (issued by warp 0).
  auto load_qdo = [&](int i) {
    mbar_arrive_expect_tx_elect(qd_bar, 2 * C::kTileBytes);
    for (int b = 0; b < C::kBlocks; ++b) {
      tma_load_3d_elect(sQ + b * 16384, &p.tm_q, qd_bar, b * 64, i * 128, bh);
      tma_load_3d_elect(sDO + b * 16384, &p.tm_do, qd_bar, b * 64, i * 128, bh);
    }
  };
  if (warp == 0) load_qdo(i0);
  int it = 0;
  for (int i = i0; ok && i < n_kt; ++i, ++it) {
    const int row = i * 128 + tid;  // this thread's query row
    // Rows past N: L = +inf makes every P of the row 0.
    const float l2 = row < N ? p.lse[static_cast<size_t>(bh) * N + row] * 1.4426950408889634f : INFINITY;
    const float drow = row < N ? p.drow[static_cast<size_t>(bh) * N + row] : 0.f;
    ok = __syncthreads_and(mbar_wait(qd_bar, it & 1, p.status, lim));
    if (!ok) break;
    if (warp == 0) {
      tc_fence_after();
      mma_rows<D>(tmem + C::kColS, sQ, sK);
      mma_rows<D>(tmem + C::kColDP, sDO, sV);
      mma_commit_elect(mma1_bar);
    }
    // The previous tile's dQ reduce has read its staging copy (P and dS buffers).
    if (tid == 0) bulk_wait_read_all();
    ok = __syncthreads_and(mbar_wait(mma1_bar, it & 1, p.status, lim));
    if (!ok) break;
    tc_fence_after();
    // P and dS of this thread's query row, 64 keys at a time (S and dP columns
    // loaded together, one wait).
#pragma unroll 1
    for (int c0 = 0; c0 < 128; c0 += 64) {
      uint32_t s[64], dp[64];
      tmem_ld64x2_sync(tmem + lane_base + C::kColS + c0, s, tmem + lane_base + C::kColDP + c0, dp);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pw[16], dw[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float pv[2], dv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int c = 32 * h + e + u;
            const int key = j * 128 + c0 + c;
            const bool keep = key < N && (!kCausal || key <= row);
            const float pe = keep ? ex2_approx(fmaf(__uint_as_float(s[c]), sl2, -l2)) : 0.f;
            pv[u] = pe;
            dv[u] = pe * (__uint_as_float(dp[c]) - drow);
          }
          pw[e / 2] = pack_bf16x2(pv[0], pv[1]);
          dw[e / 2] = pack_bf16x2(dv[0], dv[1]);
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int c = ((c0 + 32 * h) >> 3) + q4;  // 8-column chunk index 0..15
          st_shared_v4(sw128_chunk(sP, tid, c), pw[4 * q4], pw[4 * q4 + 1], pw[4 * q4 + 2], pw[4 * q4 + 3]);
          st_shared_v4(sw128_chunk(sDS, tid, c), dw[4 * q4], dw[4 * q4 + 1], dw[4 * q4 + 2], dw[4 * q4 + 3]);
        }
      }
    }
    // The tensor core reads P and dS through the async proxy; S's columns are
    // free for dS K once every thread has read them.
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
      tc_fence_after();
      mma_t<D>(tmem + C::kColDV, sP, sDO, it > 0);
      mma_t<D>(tmem + C::kColDK, sDS, sQ, it > 0);
      mma_dq<D>(tmem + C::kColS, sDS, sK);
      mma_commit_elect(mma2_bar);
    }
    ok = __syncthreads_and(mbar_wait(mma2_bar, it & 1, p.status, lim));
    if (!ok) break;
    // Q_i and dO_i are read: the next query tile's copies overlap the dQ adds below.
    if (warp == 0 && i + 1 < n_kt) load_qdo(i + 1);
    tc_fence_after();
    // dQ contribution scale * dS K_j: staged as fp32 in the P and dS buffers (no
    // MMA reads them any more) in the 128-byte-swizzled layout of a 128-row x
    // 32-float TMA box, then added to the fp32 accumulator by TMA reduce-adds,
    // which clip the rows past N.  tcgen05.ld is warp-collective: every lane loads.
#pragma unroll 1
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t g[32];
      tmem_ld32_sync(tmem + lane_base + C::kColS + c0, g);
      const uint32_t blk = sP + (c0 / 32) * 16384 + tid * 128;
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4)
        st_shared_v4(blk + ((q4 ^ (tid & 7)) << 4), __float_as_uint(__uint_as_float(g[4 * q4]) * p.scale),
                     __float_as_uint(__uint_as_float(g[4 * q4 + 1]) * p.scale),
                     __float_as_uint(__uint_as_float(g[4 * q4 + 2]) * p.scale),
                     __float_as_uint(__uint_as_float(g[4 * q4 + 3]) * p.scale));
    }
    fence_proxy_async_smem();
    // Next query tile: Q/dO and S/dP columns are reused.
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      for (int b = 0; b < D / 32; ++b) tma_reduce_add_3d(&p.tm_dqacc, sP + b * 16384, b * 32, i * 128, bh);
      bulk_commit_group();
    }
  }

  if (ok) {
    // Warp-collective TMEM loads by every lane; only key rows < N are stored.
    tc_fence_after();
    const size_t kr = static_cast<size_t>(bh) * N + (key_r < N ? key_r : 0);
    __nv_bfloat16* dvp = reinterpret_cast<__nv_bfloat16*>(p.dv) + kr * D;
    __nv_bfloat16* dkp = reinterpret_cast<__nv_bfloat16*>(p.dk) + kr * D;
#pragma unroll 1
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t a[32], b[32];
      tmem_ld32_sync(tmem + lane_base + C::kColDV + c0, a);
      tmem_ld32_sync(tmem + lane_base + C::kColDK + c0, b);
      if (key_r >= N) continue;
#pragma unroll
      for (int e = 0; e < 32; e += 8) {
        uint4 va, vb;
        va.x = pack_bf16x2(__uint_as_float(a[e]), __uint_as_float(a[e + 1]));
        va.y = pack_bf16x2(__uint_as_float(a[e + 2]), __uint_as_float(a[e + 3]));
        va.z = pack_bf16x2(__uint_as_float(a[e + 4]), __uint_as_float(a[e + 5]));
        va.w = pack_bf16x2(__uint_as_float(a[e + 6]), __uint_as_float(a[e + 7]));
        vb.x = pack_bf16x2(__uint_as_float(b[e]) * p.scale, __uint_as_float(b[e + 1]) * p.scale);
        vb.y = pack_bf16x2(__uint_as_float(b[e + 2]) * p.scale, __uint_as_float(b[e + 3]) * p.scale);
        vb.z = pack_bf16x2(__uint_as_float(b[e + 4]) * p.scale, __uint_as_float(b[e + 5]) * p.scale);
        vb.w = pack_bf16x2(__uint_as_float(b[e + 6]) * p.scale, __uint_as_float(b[e + 7]) * p.scale);
        *reinterpret_cast<uint4*>(dvp + c0 + e) = va;
        *reinterpret_cast<uint4*>(dkp + c0 + e) = vb;
      }
    }
  }

  // ---- teardown: the dQ reduce-adds have completed, every MMA of this CTA has
  // completed before TMEM is freed
  if (tid == 0) bulk_wait_all();
  if (warp == 0) {
    mma_commit_elect(done_bar);
    mbar_wait(done_bar, 0, p.status, lim);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool kCausal>
cudaError_t launch_main(const BwdParams& p, cudaStream_t stream) {
  auto kern = attn_bwd_tc_kernel<D, kCausal>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdCfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int n_kt = (p.N + 127) / 128;
  kern<<<dim3(static_cast<unsigned>(n_kt), static_cast<unsigned>(p.BH)), dim3(kBwdThreads), BwdCfg<D>::kSmemBytes,
         stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdParams& p, int d, bool causal, cudaStream_t stream) {
  if (d != 64 && d != 128) return cudaErrorInvalidValue;
  const long long rows = static_cast<long long>(p.BH) * p.N;
  const unsigned prep_blocks = static_cast<unsigned>((rows + 7) / 8);
  if (d == 128) attn_bwd_prep_kernel<128><<<prep_blocks, 256, 0, stream>>>(p);
  else attn_bwd_prep_kernel<64><<<prep_blocks, 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (d == 128) e = causal ? launch_main<128, true>(p, stream) : launch_main<128, false>(p, stream);
  else e = causal ? launch_main<64, true>(p, stream) : launch_main<64, false>(p, stream);
  if (e != cudaSuccess) return e;
  const long long n4 = rows * d / 4;
  const long long want = (n4 + 255) / 256;
  const unsigned blocks = static_cast<unsigned>(want < 152LL * 16 ? want : 152LL * 16);
  attn_bwd_dq_kernel<<<blocks, 256, 0, stream>>>(p, n4);
  return cudaGetLastError();
}

}  // namespace attn

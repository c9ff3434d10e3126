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
// Main kernel, persistent (one CTA per SM, each walking a snake-ordered list of
// work items (key tile j, b*h)), scores held transposed: TMEM lane
// r is key r of the tile, so S^T = K_j Q_i^T and dP^T = V_j dO_i^T put one key
// row of each per thread, and the P^T and dS^T that thread computes are already
// the A operands of dV += P^T dO_i and dK += dS^T Q_i, straight from TMEM.
// Warp roles (320 threads):
//   warps 0-7  elementwise pass: warp w owns TMEM lanes 32 (w % 4).. (keys) and
//              query columns 64 (w / 4)..; P^T = 2^(S^T scale log2 e - L log2 e),
//              dS^T = P^T (dP^T - D), written back to TMEM as bf16 over dP^T, and
//              dS^T also to shared memory for dQ; then they move dQ_i out of
//              TMEM and stage it for the reduce-adds;
//   warp 8     TMA producer: K_j, V_j once, then Q_i, dO_i and the tile's L and D
//              vectors into one of two slots, one query tile ahead; it also
//              issues the dQ reduce-adds from the slots (d = 128: the dO half
//              of a slot first, so that dO reloads while the Q half is read);
//   warp 9     MMA issuer, per query tile i:
//                dV += P^T dO_i, dK += dS^T Q_i   (A from TMEM; half of each once the
//                                                   first 32-query chunks are written;
//                                                   the last readers of the slot)
//                dQ_i = dS K_j          (into the S^T columns, drained by warps 0-7)
//                dP^T_{i+1} = V_j dO_{i+1}^T   (over P^T, dS^T: issued after their readers)
//                S^T_{i+1} = K_j Q_{i+1}^T    (once the dQ_i drain has read its columns)
// The pass warps move dQ_i from TMEM into registers, then (the slot's Q and dO
// being read by then) stage it, scaled, in that slot as fp32 TMA boxes; the
// producer warp issues the reduce-adds into the fp32 accumulator and waits for
// them to read the slot before loading the query tile after next into it, so
// neither the reduce nor its completion sits on the pass warps' path.  After an
// item's last query tile: dK * scale and dV to bf16 (d = 128: staged per warp in
// the then idle dS^T buffer and written by TMA stores).  Across items the next item
// starts under the current one's tail: its first Q, dO load into the slot the
// finished query tiles freed, its K, V as soon as the last MMA that reads the
// current ones completes, and its S^T, dP^T while the pass warps drain the last
// dQ and read dV, dK out; only its first dV/dK products wait for that read-out.
// The main and conversion kernels are launched with programmatic stream
// serialisation: each starts under its predecessor's tail and waits on the
// device for that predecessor's results before it reads them.
#include <cstdlib>
#include <cstring>
#include <utility>

#include <cuda_bf16.h>

#include "attn_kernels.h"
#include "ptx_sm103.cuh"

namespace attn {
namespace {

// Optional event trace (compile with -DATTN_TRACE): cycle stamps of the first
// 64 steps of CTA 0, for timeline analysis.
#ifdef ATTN_TRACE
__device__ unsigned long long g_bwd_trace[64 * 16];
#define BWD_TRACE(cond, step, ev)                                                        \
  do {                                                                                   \
    if ((cond) && blockIdx.x == 0 && (step) < 64) g_bwd_trace[(step) * 16 + (ev)] = clock64(); \
  } while (0)
#else
#define BWD_TRACE(cond, step, ev) \
  do {                            \
  } while (0)
#endif

constexpr int kBwdThreads = 320;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int kPSBytes = 128 * 128 * 2;  // one [128 key][128 query] bf16 tile (dS^T)
constexpr int kMaxSmem = 232448;         // opt-in dynamic shared memory per CTA

template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = 128 * D * 2;  // one 128-row bf16 tile of Q, K, V or dO
  static constexpr int kBlocks = D / 64;          // 128-byte column blocks per row
  // d = 64 leaves room for a third Q/dO slot in shared memory and a second S^T
  // buffer in TMEM: the next query tile's S^T is then computed during the current
  // pass, and the next pass does not wait for the dQ drain.
  static constexpr bool kDblS = (D == 64);
  static constexpr int kSlots = kDblS ? 3 : 2;
  // Shared memory (from a 1024-byte aligned base): K | V | slots (Q, dO) | dS^T |
  // L2 per slot | D per slot | barriers.  A slot, once its Q and dO are read,
  // stages that query tile's fp32 dQ (128 x d x 4 bytes = the slot's size) as
  // d/32 TMA boxes of 128 rows x 32 floats.
  static constexpr int kK = 0, kV = kTileBytes, kSlot = 2 * kTileBytes, kSlotBytes = 2 * kTileBytes;
  static constexpr int kDS = kSlot + kSlots * kSlotBytes;
  static constexpr int kBoxes = D / 32;  // dQ staging boxes per query tile
  static constexpr int kL2 = kDS + kPSBytes, kDrow = kL2 + kSlots * 512;
  static constexpr int kBar = kDrow + kSlots * 512;
  static constexpr int kUsed = kBar + 17 * 8 + 16;  // 17 mbarriers, then the TMEM address
  static constexpr int kSmemBytes = (kUsed + 1024 < kMaxSmem) ? kUsed + 1024 : kMaxSmem;
  static_assert(kUsed <= kMaxSmem, "shared memory layout too large");
  // TMEM columns: dV | dK | S^T (then dQ; two buffers when kDblS) | dP^T (then P^T
  // and dS^T, bf16)
  static constexpr uint32_t kColDV = 0, kColDK = D, kColS = 2 * D, kColDP = 2 * D + (kDblS ? 256 : 128);
  static_assert(kColDP + 128 <= 512, "TMEM columns");
  static constexpr uint32_t kIdescQK = make_idesc(1, 128, 128, 0, 0);  // S^T, dP^T: both operands K-major
  static constexpr uint32_t kIdescTS = make_idesc(1, 128, D, 0, 1);    // dV, dK: A in TMEM, B = dO / Q MN-major
  static constexpr uint32_t kIdescDQ = make_idesc(1, 128, D, 1, 1);    // dS K: A = dS^T tile MN-major, B = K MN-major
};

// TMEM column (relative to the S^T block) of the bf16 P^T values of queries
// [16 kk, 16 kk + 16); their dS^T follow at + 8.  The pass writes each 16-query
// group over the 16 S^T columns it has just read, so later groups' S^T (and all
// of dP^T) stay intact while their loads are in flight.
__device__ __forceinline__ uint32_t pds_col(int kk) { return 16u * static_cast<uint32_t>(kk); }

// Bulk tensor reduce-add shared -> global (element type and box from the map),
// tracked by the issuing thread's bulk async-groups.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}
// Bulk tensor store shared -> global (box from the map; rows outside the
// tensor are not written), tracked like the reduce-adds.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The source shared memory of every committed group has been read.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Adds `bytes` to the transactions the barrier's current phase waits for,
// without arriving (elected lane).
__device__ __forceinline__ void mbar_expect_tx_elect(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;\n}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}
// The source shared memory of every committed group but the most recent one has been read.
__device__ __forceinline__ void bulk_wait_read_all_but_last() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Every committed group has completed (its global writes are done).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Programmatic dependent launch.  The kernel launched after this one with
// programmatic stream serialisation may start once every CTA of this grid has
// executed launch_dependents or exited; all of this grid's CTAs are then
// resident or done, so the early start cannot take their SMs away.
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Returns once the grid this one was launched behind has completed and its
// memory writes are visible (at once when there is no such grid).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Contiguous global -> shared copy (16-byte aligned addresses, size a multiple
// of 16), completion counted in bytes on `bar`; elected lane.
__device__ __forceinline__ void bulk_load_elect(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}


// The same threads agree on a flag: true only if it is true in every one of
// them, so a failed (timed-out) wait makes all pass warps leave together and
// none is left waiting at a pass barrier.
__device__ __forceinline__ bool pass_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, 2, 256, q;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}



// Byte address of the 16-byte chunk holding columns [8c, 8c + 8) of row r of a
// [128 x 128] bf16 tile stored as two 128-byte-swizzled column blocks (the
// layout TMA writes for a 128 x 64 box with 128-byte swizzle).
__device__ __forceinline__ uint32_t sw128_chunk(uint32_t tile, int r, int c) {
  return tile + (c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// Two 32-lane x 32-column TMEM loads with a single wait (both in one statement,
// so no use of the registers can move above the wait).
__device__ __forceinline__ void tmem_ld32x2_sync(uint32_t ta, uint32_t (&a)[32], uint32_t tb, uint32_t (&b)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"
      "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]), "=r"(a[8]),
        "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(a[16]),
        "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]), "=r"(a[24]),
        "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31]), "=r"(b[0]),
        "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]),
        "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]), "=r"(b[16]), "=r"(b[17]),
        "=r"(b[18]), "=r"(b[19]), "=r"(b[20]), "=r"(b[21]), "=r"(b[22]), "=r"(b[23]), "=r"(b[24]), "=r"(b[25]),
        "=r"(b[26]), "=r"(b[27]), "=r"(b[28]), "=r"(b[29]), "=r"(b[30]), "=r"(b[31])
      : "r"(ta), "r"(tb)
      : "memory");
}

// acc = A B^T for 128 x 128 tiles with d-long rows (S^T = K Q^T, dP^T = V dO^T):
// both operands K-major.
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

// acc (+)= X Y over the queries of chunk q (k-steps kk with (kk >> 1) & 1 == q:
// queries [32q, 32q + 32) and [64 + 32q, 96 + 32q)), for X = [128 key][128 query]
// bf16 in TMEM (P^T or dS^T, at the columns pds_col gives, dS^T at + 8) and
// Y = [128 query][d] in shared memory (dO or Q) as an MN-major B operand.
template <int D>
__device__ __forceinline__ void mma_ts_half(uint32_t tmem_d, uint32_t x_tmem, uint32_t y, int q, bool accumulate) {
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const int kk = (h >> 1) * 4 + q * 2 + (h & 1);
    mma_f16_ts_elect(tmem_d, x_tmem + pds_col(kk), sdesc_sw128(y + kk * 2048, 16384, 1024), BwdCfg<D>::kIdescTS,
                     accumulate || h > 0);
  }
}

// dQ' = dS K_j: contraction over the keys; the dS^T tile ([key][query]) read as an
// MN-major A operand, K_j ([key][d]) as an MN-major B operand.
template <int D>
__device__ __forceinline__ void mma_dq(uint32_t tmem_d, uint32_t ds_t, uint32_t k) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    mma_f16_ss_elect(tmem_d, sdesc_sw128(ds_t + kk * 2048, 16384, 1024), sdesc_sw128(k + kk * 2048, 16384, 1024),
                     BwdCfg<D>::kIdescDQ, kk > 0);
  }
}

// Two bf16 (low half first) to floats.
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

// Per row of every head, padded to whole 128-row tiles: -L log2 e (-inf on
// padding rows, so their P is 0) and -D with D = sum_c dO_c O_c (0 on padding
// rows), negated so the pass adds them; real rows of the dQ accumulator zeroed.
// A row is read by d/8 lanes, 16 bytes of O and of dO each; a warp covers
// 256/d rows per access and kPrepIter accesses, all issued before the first
// product so that each lane keeps several loads in flight.
constexpr int kPrepIter = 4;
template <int D>
constexpr int prep_rows_per_block() {
  return 8 /*warps*/ * (32 / (D / 8)) * kPrepIter;
}
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const BwdParams p, int n_pad) {
  // The main kernel may launch under this grid's last wave: it waits for this
  // grid's results before it reads them.
  grid_launch_dependents();
  constexpr int kLanes = D / 8;         // lanes per row: 16 bytes of bf16 each
  constexpr int kRows = 32 / kLanes;    // rows per warp access
  const int lane = threadIdx.x & 31, sub = lane / kLanes, piece = lane % kLanes;
  const long long total = static_cast<long long>(p.BH) * n_pad;
  const long long row0 =
      (static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * (kRows * kPrepIter) + sub;
  uint4 ov[kPrepIter], gv[kPrepIter];
  long long row[kPrepIter];  // row of O, dO, L and the accumulator; -1: padding or past the end
#pragma unroll
  for (int k = 0; k < kPrepIter; ++k) {
    const long long prow = row0 + k * kRows;
    row[k] = -1;
    ov[k] = gv[k] = make_uint4(0u, 0u, 0u, 0u);
    if (prow < total) {
      const int bh = static_cast<int>(prow / n_pad), r = static_cast<int>(prow % n_pad);
      if (r < p.N) {
        row[k] = static_cast<long long>(bh) * p.N + r;
        ov[k] = reinterpret_cast<const uint4*>(p.o)[row[k] * kLanes + piece];
        gv[k] = reinterpret_cast<const uint4*>(p.dout)[row[k] * kLanes + piece];
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kPrepIter; ++k) {
    const long long prow = row0 + k * kRows;
    float acc = 0.f;
    if (row[k] >= 0) {
      const uint32_t o4[4] = {ov[k].x, ov[k].y, ov[k].z, ov[k].w}, g4[4] = {gv[k].x, gv[k].y, gv[k].z, gv[k].w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float2 o2 = bf16x2_to_f2(o4[c]), g2 = bf16x2_to_f2(g4[c]);
        acc = fmaf(o2.x, g2.x, fmaf(o2.y, g2.y, acc));
      }
      // d fp32 per accumulator row: two 16-byte pieces per lane.
      float4* dq = reinterpret_cast<float4*>(p.dq_acc) + row[k] * (D / 4) + 2 * piece;
      dq[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      dq[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // Sum over the row's lanes (every lane takes part; padding rows add zeros).
#pragma unroll
    for (int m = kLanes / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (piece == 0 && prow < total) {
      p.drow[prow] = row[k] >= 0 ? -acc : 0.f;
      p.lse2[prow] = row[k] >= 0 ? -p.lse[row[k]] * 1.4426950408889634f : -INFINITY;
    }
  }
}

// dQ (bf16) = the fp32 accumulator.  A block converts 4 x 256 consecutive
// groups of four elements per pass, each thread four groups 256 apart, all four
// loads issued before the first store.
constexpr int kDqPerThread = 4;
__global__ void __launch_bounds__(256) attn_bwd_dq_kernel(const BwdParams p, long long n4) {
  grid_dependency_wait();  // launched behind the main kernel: its reduce-adds are complete
  const float4* src = reinterpret_cast<const float4*>(p.dq_acc);
  uint2* dst = reinterpret_cast<uint2*>(p.dq);
  const long long per_pass = static_cast<long long>(gridDim.x) * 256 * kDqPerThread;
  for (long long base = static_cast<long long>(blockIdx.x) * 256 * kDqPerThread + threadIdx.x; base < n4;
       base += per_pass) {
    float4 v[kDqPerThread];
#pragma unroll
    for (int k = 0; k < kDqPerThread; ++k)
      if (base + 256 * k < n4) v[k] = src[base + 256 * k];
#pragma unroll
    for (int k = 0; k < kDqPerThread; ++k)
      if (base + 256 * k < n4) dst[base + 256 * k] = make_uint2(pack_bf16x2(v[k].x, v[k].y), pack_bf16x2(v[k].z, v[k].w));
  }
}

// P^T and dS^T of one 16-query group of this thread's key row, two queries per
// packed f32x2 instruction: P = 2^(S sl2 + (-L log2 e)), dS = P (dP + (-D)); 8
// packed P^T and 8 packed dS^T words out.  kMask: the group needs the key mask
// (keys past N, or causal keys after the query).
template <bool kMask>
__device__ __forceinline__ void pass_sub16(const uint32_t (&s)[16], const uint32_t (&dp)[16], uint32_t nl2_addr,
                                           uint32_t nd_addr, uint64_t sl2x2, int key_local, int q_local0, bool key_ok,
                                           bool diag, uint32_t (&pw)[8], uint32_t (&dw)[8]) {
#pragma unroll
  for (int c = 0; c < 16; c += 4) {
    const float4 nl = ld_shared_f4(nl2_addr + 4 * c);
    const float4 nd = ld_shared_f4(nd_addr + 4 * c);
    const uint64_t x01 = f2_fma(f2_pack(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sl2x2, f2_pack(nl.x, nl.y));
    const uint64_t x23 =
        f2_fma(f2_pack(__uint_as_float(s[c + 2]), __uint_as_float(s[c + 3])), sl2x2, f2_pack(nl.z, nl.w));
    float e[4] = {ex2_approx(f2_lo(x01)), ex2_approx(f2_hi(x01)), ex2_approx(f2_lo(x23)), ex2_approx(f2_hi(x23))};
    if (kMask) {
      // The group's query columns this key keeps start at `thr` (keys past N
      // keep none; on the causal diagonal a key keeps the queries at or after
      // it).  A compound per-element predicate for the same test ran about 3.5
      // times slower.
      const int thr = !key_ok ? 32 : (diag ? key_local - q_local0 : -32);
#pragma unroll
      for (int u = 0; u < 4; ++u) e[u] = (c + u >= thr) ? e[u] : 0.f;
    }
    const uint64_t g01 = f2_add(f2_pack(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])), f2_pack(nd.x, nd.y));
    const uint64_t g23 = f2_add(f2_pack(__uint_as_float(dp[c + 2]), __uint_as_float(dp[c + 3])), f2_pack(nd.z, nd.w));
    const uint64_t d01 = f2_mul(f2_pack(e[0], e[1]), g01);
    const uint64_t d23 = f2_mul(f2_pack(e[2], e[3]), g23);
    pw[c / 2] = pack_bf16x2(e[0], e[1]);
    pw[c / 2 + 1] = pack_bf16x2(e[2], e[3]);
    dw[c / 2] = pack_bf16x2(f2_lo(d01), f2_hi(d01));
    dw[c / 2 + 1] = pack_bf16x2(f2_lo(d23), f2_hi(d23));
  }
}

// Two 32-lane x 16-column TMEM loads issued without waiting; their registers
// become usable only through tmem_wait_ld16x2 below.
__device__ __forceinline__ void tmem_ld16x2_issue(uint32_t ta, uint32_t (&a)[16], uint32_t tb, uint32_t (&b)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]), "=r"(a[8]),
        "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(b[0]),
        "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]),
        "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15])
      : "r"(ta), "r"(tb)
      : "memory");
}
// Waits for every TMEM load of this thread; the registers pass through the
// statement, so no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld16x2(uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
                 "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]),
                 "+r"(a[15]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]),
                 "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]),
                 "+r"(b[14]), "+r"(b[15])
               :
               : "memory");
}
// Two 32-lane x 8-column TMEM stores, not waited for (tmem_wait_st does).
__device__ __forceinline__ void tmem_st8x2_issue(uint32_t ta, const uint32_t (&a)[8], uint32_t tb, const uint32_t (&b)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%2,%3,%4,%5,%6,%7,%8,%9};\n"
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%1], {%10,%11,%12,%13,%14,%15,%16,%17};" ::"r"(ta),
      "r"(tb), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]), "r"(b[0]),
      "r"(b[1]), "r"(b[2]), "r"(b[3]), "r"(b[4]), "r"(b[5]), "r"(b[6]), "r"(b[7])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

template <int D, bool kCausal>
__global__ void __launch_bounds__(kBwdThreads, 1) attn_bwd_tc_kernel(const __grid_constant__ BwdParams p,
                                                                      int head_major) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  // The layout does not fit this base: report, touch nothing.
  if (base + C::kUsed > raw + C::kSmemBytes) {
    if (threadIdx.x == 0) atomicExch(p.status, kStatusTimeout);
    return;
  }
  uint8_t* base_ptr = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + C::kBar);
  const uint32_t b0 = smem_u32(bars);
  const uint32_t kv_bar = b0, s_full = b0 + 8, dq_full = b0 + 16, drain_done = b0 + 24, fin_bar = b0 + 32;
  // dV and dK of the current item read out of TMEM by the epilogue (the next
  // item's first dV/dK products may overwrite them).
  const uint32_t acc_free = b0 + 128;
  // P^T / dS^T chunk q (queries [32q, 32q + 32) and [64 + 32q, 96 + 32q)) written
  auto p_full = [&](int q) { return b0 + 40 + 8 * q; };
  auto q_full = [&](int s) { return b0 + 56 + 8 * s; };       // slot loaded
  auto q_empty = [&](int s) { return b0 + 80 + 8 * s; };      // slot's Q, dO read by the MMAs
  auto stage_free = [&](int s) { return b0 + 104 + 8 * s; };  // slot's dQ staged
  // Steps (one query tile of one work item) are numbered T across the CTA's
  // items: step T uses slot T % kSlots for the (T / kSlots)-th time, per-step
  // barriers complete one phase per step, per-item ones (kv_bar, fin_bar,
  // acc_free) one phase per item.
  constexpr int kSl = C::kSlots;
  auto slot_of = [](int t) { return t % kSl; };
  auto use_par = [](int t) { return static_cast<uint32_t>((t / kSl) & 1); };
  // S^T (then dQ) columns of step t.
  auto col_s = [](int t) { return C::kColS + (C::kDblS ? 128u * static_cast<uint32_t>(t & 1) : 0u); };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 17);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = p.N, n_kt = (N + 127) >> 7, n_pad = n_kt * 128;
  // Persistent: work item x = (key tile j, b*h); round r of CTA c takes item
  // r G + c (even r) or r G + G - 1 - c (odd r), a snake over the item order.
  // Item order: key-tile-major (all heads' key tile 0, then key tile 1, ...: the
  // heaviest causal items first) or head-major (one head's key tiles after the
  // other, heaviest first within the head, so the CTAs running together reduce
  // into one head's dQ, which stays in L2).  Non-causal grids are always
  // head-major.
  const bool hm = !kCausal || head_major != 0;
  const int total = n_kt * p.BH;
  auto item_of = [&](int r) {
    const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    return r * G + ((r & 1) ? (G - 1 - c) : c);
  };
  auto key_tile_of = [&](int x) { return hm ? x % n_kt : x / p.BH; };
  auto head_of = [&](int x) { return hm ? x / n_kt : x % p.BH; };
  auto steps_of = [&](int j) { return kCausal ? n_kt - j : n_kt; };  // causal: query tiles j .. n_kt - 1
  // Query tile of the t-th step of an item with key tile j.
  auto qtile = [&](int j, int t) { return kCausal || j + t < n_kt ? j + t : j + t - n_kt; };
  const uint64_t lim = p.timeout_ns;

  if (tid == 0) {
    mbar_init(kv_bar, 1);
    mbar_init(s_full, 1);
    mbar_init(p_full(0), 8);
    mbar_init(p_full(1), 8);
    mbar_init(dq_full, 1);
    mbar_init(drain_done, 8);
    mbar_init(fin_bar, 1);
    mbar_init(acc_free, 8);
    for (int s = 0; s < kSl; ++s) {
      mbar_init(q_full(s), 1);
      mbar_init(q_empty(s), 1);
      mbar_init(stage_free(s), 8);
    }
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_holder);
  const uint32_t sK = base + C::kK, sV = base + C::kV, sDS = base + C::kDS;
  auto sSlot = [&](int s) { return base + C::kSlot + s * C::kSlotBytes; };
  auto sQ = [&](int s) { return sSlot(s); };
  auto sDO = [&](int s) { return sSlot(s) + C::kTileBytes; };
  auto sL2 = [&](int s) { return base + C::kL2 + s * 512; };
  auto sDr = [&](int s) { return base + C::kDrow + s * 512; };

  if (warp == kProducerWarp) {
    // ============================================================ TMA producer
    // The kernel may start under the preparation kernel (programmatic launch):
    // the row vectors and the zeroed dQ accumulator it writes are read and
    // reduce-added only by this warp, after this wait.
    grid_dependency_wait();
    // (b*h, query tile) of the last kSl steps, by slot: where their dQ goes.
    int ring_bh[kSl], ring_q[kSl];
    // dQ of step t, staged in its slot by the pass warps: reduce-add the boxes
    // into the accumulator and wait until they are read, so the slot can be
    // reloaded.
    auto finish_tile = [&](int t) {
      const int s = slot_of(t);
      if (!__all_sync(0xffffffffu, mbar_wait_sleep(stage_free(s), use_par(t), p.status, lim, 64))) return false;
      BWD_TRACE(lane == 0, t, 14);
      if (lane == 0) {
        for (int b = 0; b < C::kBoxes; ++b)
          tma_reduce_add_3d(&p.tm_dqacc, sSlot(s) + b * 16384, 32 * b, ring_q[s] * 128, ring_bh[s]);
        bulk_commit_group();
        bulk_wait_read_all();
      }
      BWD_TRACE(lane == 0, t, 15);
      __syncwarp();
      return true;
    };
    int T = 0, n_items = 0, issued = 0;  // steps done, items and steps whose loads were issued
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int x = item_of(r);
      if (x >= total) break;
      const int j = key_tile_of(x), bh = head_of(x), n_it = steps_of(j);
      for (int it = 0; ok && it < n_it; ++it, ++T) {
        const int s = slot_of(T), i = qtile(j, it);
        const size_t v0 = static_cast<size_t>(bh) * n_pad + static_cast<size_t>(i) * 128;
        if (!C::kDblS && T >= kSl) {
          // The slot holds step T - 2's staged dQ: reduce-add its dO half first
          // (own bulk group), and once that half is read load dO and the row
          // vectors there, their bytes added to the slot's phase without
          // arriving; the Q load and the phase's one arrival follow when the
          // rest is read.  Half of the reload overlaps the reduce's reads.
          const int t0 = T - kSl;
          ok = __all_sync(0xffffffffu, mbar_wait_sleep(stage_free(s), use_par(t0), p.status, lim, 64));
          if (!ok) break;
          BWD_TRACE(lane == 0, t0, 14);
          if (lane == 0) {
            for (int b = C::kBoxes / 2; b < C::kBoxes; ++b)  // boxes over the dO half of the slot
              tma_reduce_add_3d(&p.tm_dqacc, sSlot(s) + b * 16384, 32 * b, ring_q[s] * 128, ring_bh[s]);
            bulk_commit_group();
            for (int b = 0; b < C::kBoxes / 2; ++b)
              tma_reduce_add_3d(&p.tm_dqacc, sSlot(s) + b * 16384, 32 * b, ring_q[s] * 128, ring_bh[s]);
            bulk_commit_group();
            bulk_wait_read_all_but_last();
          }
          __syncwarp();
          BWD_TRACE(lane == 0, T, 6);
          mbar_expect_tx_elect(q_full(s), C::kTileBytes + 1024);
          for (int b = 0; b < C::kBlocks; ++b)
            tma_load_3d_elect(sDO(s) + b * 16384, &p.tm_do, q_full(s), b * 64, i * 128, bh);
          bulk_load_elect(sL2(s), p.lse2 + v0, 512, q_full(s));
          bulk_load_elect(sDr(s), p.drow + v0, 512, q_full(s));
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
          BWD_TRACE(lane == 0, t0, 15);
          mbar_arrive_expect_tx_elect(q_full(s), C::kTileBytes);
          for (int b = 0; b < C::kBlocks; ++b)
            tma_load_3d_elect(sQ(s) + b * 16384, &p.tm_q, q_full(s), b * 64, i * 128, bh);
        } else {
          if (T >= kSl) {  // the slot's previous step is read and its dQ reduced
            ok = finish_tile(T - kSl);
            if (!ok) break;
          }
          BWD_TRACE(lane == 0, T, 6);
          mbar_arrive_expect_tx_elect(q_full(s), 2 * C::kTileBytes + 1024);
          for (int b = 0; b < C::kBlocks; ++b) {
            tma_load_3d_elect(sQ(s) + b * 16384, &p.tm_q, q_full(s), b * 64, i * 128, bh);
            tma_load_3d_elect(sDO(s) + b * 16384, &p.tm_do, q_full(s), b * 64, i * 128, bh);
          }
          bulk_load_elect(sL2(s), p.lse2 + v0, 512, q_full(s));
          bulk_load_elect(sDr(s), p.drow + v0, 512, q_full(s));
        }
        ring_bh[s] = bh;
        ring_q[s] = i;
        issued = T + 1;
        if (it == 0) {
          // K_j, V_j over the previous item's, once its last MMAs (which read them) are done.
          if (r > 0) ok = __all_sync(0xffffffffu, mbar_wait(fin_bar, (r - 1) & 1, p.status, lim));
          if (!ok) break;
          mbar_arrive_expect_tx_elect(kv_bar, 2 * C::kTileBytes);
          for (int b = 0; b < C::kBlocks; ++b) {
            tma_load_3d_elect(sK + b * 16384, &p.tm_k, kv_bar, b * 64, j * 128, bh);
            tma_load_3d_elect(sV + b * 16384, &p.tm_v, kv_bar, b * 64, j * 128, bh);
          }
          ++n_items;
        }
      }
    }
    for (int t = T >= kSl ? T - kSl : 0; ok && t < T; ++t) ok = finish_tile(t);
    if (lane == 0) bulk_wait_all();  // the dQ reduce-adds have completed
    // Copies still in flight (only after a failed wait elsewhere) land before exit.
    if (n_items > 0) mbar_wait(kv_bar, (n_items - 1) & 1, p.status, lim);
    for (int t = issued > kSl ? issued - kSl : 0; t < issued; ++t)
      mbar_wait(q_full(slot_of(t)), use_par(t), p.status, lim);
  } else if (warp == kMmaWarp) {
    // ============================================================ MMA issuer
    int T = 0, n_fin = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int x = item_of(r);
      if (x >= total) break;
      const int n_it = steps_of(key_tile_of(x));
      // The item's K_j, V_j and first Q, dO; its first S^T goes over the
      // previous step's dQ columns, once they are drained.
      ok = mbar_wait(kv_bar, r & 1, p.status, lim) && mbar_wait(q_full(slot_of(T)), use_par(T), p.status, lim) &&
           (T == 0 || mbar_wait(drain_done, (T - 1) & 1, p.status, lim));
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      mma_rows<D>(tmem + col_s(T), sK, sQ(slot_of(T)));
      mma_rows<D>(tmem + C::kColDP, sV, sDO(slot_of(T)));
      mma_commit_elect(s_full);
      BWD_TRACE(lane == 0, T, 0);
      for (int it = 0; ok && it < n_it; ++it, ++T) {
        const int s = slot_of(T);
        if (C::kDblS && it + 1 < n_it) {
          // The next step's S^T into the other buffer, to run during this pass,
          // once that buffer's dQ (step T - 1) is out of TMEM.
          const int s1 = slot_of(T + 1);
          ok = __all_sync(0xffffffffu, mbar_wait(q_full(s1), use_par(T + 1), p.status, lim) &&
                                           (it == 0 || mbar_wait(drain_done, (T - 1) & 1, p.status, lim)));
          if (!ok) break;
          tc_fence_after();
          mma_rows<D>(tmem + col_s(T + 1), sK, sQ(s1));
        }
        if (it == 0 && r > 0) {
          // The first dV/dK products of the item overwrite the accumulators:
          // the previous item's epilogue must have read them.
          ok = __all_sync(0xffffffffu, mbar_wait(acc_free, (r - 1) & 1, p.status, lim));
          if (!ok) break;
          tc_fence_after();
        }
        // dV and dK over the queries of the first P^T / dS^T chunks while the pass
        // computes the second ones.
        ok = __all_sync(0xffffffffu, mbar_wait(p_full(0), T & 1, p.status, lim));
        if (!ok) break;
        BWD_TRACE(lane == 0, T, 1);
        tc_fence_after();
        mma_ts_half<D>(tmem + C::kColDV, tmem + col_s(T), sDO(s), 0, it > 0);
        mma_ts_half<D>(tmem + C::kColDK, tmem + col_s(T) + 8, sQ(s), 0, it > 0);
        ok = __all_sync(0xffffffffu, mbar_wait(p_full(1), T & 1, p.status, lim));
        if (!ok) break;
        BWD_TRACE(lane == 0, T, 2);
        tc_fence_after();
        mma_ts_half<D>(tmem + C::kColDV, tmem + col_s(T), sDO(s), 1, true);
        mma_ts_half<D>(tmem + C::kColDK, tmem + col_s(T) + 8, sQ(s), 1, true);
        mma_commit_elect(q_empty(s));
        mma_dq<D>(tmem + col_s(T), sDS, sK);
        mma_commit_elect(dq_full);
        BWD_TRACE(lane == 0, T, 3);
        if (it + 1 < n_it) {
          const int s1 = slot_of(T + 1);
          if (!C::kDblS) {
            ok = __all_sync(0xffffffffu, mbar_wait(q_full(s1), use_par(T + 1), p.status, lim));
            if (!ok) break;
            tc_fence_after();
          }
          mma_rows<D>(tmem + C::kColDP, sV, sDO(s1));  // the pass has read dP^T
          if (!C::kDblS) {
            ok = __all_sync(0xffffffffu, mbar_wait(drain_done, T & 1, p.status, lim));
            if (!ok) break;
            BWD_TRACE(lane == 0, T, 4);
            tc_fence_after();
            mma_rows<D>(tmem + col_s(T + 1), sK, sQ(s1));
          }
          mma_commit_elect(s_full);
          BWD_TRACE(lane == 0, T + 1, 0);
        }
      }
      if (!ok) break;
      // dV, dK of the item complete (the epilogue may read them) and K_j, V_j
      // are no longer read (the producer may load the next item's).
      mma_commit_elect(fin_bar);
      ++n_fin;
    }
    // Every MMA of this CTA completes before TMEM is freed.
    if (!ok) {
      mma_commit_elect(fin_bar);
      ++n_fin;
    }
    if (n_fin > 0) mbar_wait(fin_bar, (n_fin - 1) & 1, p.status, lim);
  } else {
    // ============================================================ pass / drain warps
    const int qd = warp & 3, g = warp >> 2;
    const int key_local = qd * 32 + lane;       // this thread's key row (TMEM lane)
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
    const uint64_t sl2x2 = f2_pack(p.scale_log2, p.scale_log2);
    bool ok = true;
    int T = 0;
    for (int r = 0; ok; ++r) {
      const int x = item_of(r);
      if (x >= total) break;
      const int j = key_tile_of(x), bh = head_of(x), n_it = steps_of(j);
      const int key = j * 128 + key_local;
      const bool key_ok = key < N;
      for (int it = 0; ok && it < n_it; ++it, ++T) {
        const int s = slot_of(T), i = qtile(j, it);
        ok = pass_all(mbar_wait(s_full, T & 1, p.status, lim) && mbar_wait(q_full(s), use_par(T), p.status, lim));
        if (!ok) break;
        BWD_TRACE(tid == 0, T, 8);
        tc_fence_after();
        const bool diag = kCausal && i == j;
        const bool mask = diag || !key_ok;
        // Four 16-query groups (queries 64g + 16u ..): group u + 1's S^T and dP^T
        // loads are in flight while group u is computed; P^T and dS^T go over the
        // group's own S^T columns.  After groups 1 and 3 (a 32-query chunk) the
        // stores are waited for and the chunk is handed to the MMA warp.
        uint32_t sv[2][16], dpv[2][16];
        tmem_ld16x2_issue(tmem + lane_base + col_s(T) + 64 * g, sv[0], tmem + lane_base + C::kColDP + 64 * g, dpv[0]);
        tmem_wait_ld16x2(sv[0], dpv[0]);
  #pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int b = u & 1;
          const int col0 = 64 * g + 16 * u;  // first query (tile-local) of this group
          if (u < 3)
            tmem_ld16x2_issue(tmem + lane_base + col_s(T) + col0 + 16, sv[b ^ 1],
                              tmem + lane_base + C::kColDP + col0 + 16, dpv[b ^ 1]);
          uint32_t pw[8], dw[8];
          if (mask)
            pass_sub16<true>(sv[b], dpv[b], sL2(s) + 4 * col0, sDr(s) + 4 * col0, sl2x2, key_local, col0, key_ok, diag,
                             pw, dw);
          else
            pass_sub16<false>(sv[b], dpv[b], sL2(s) + 4 * col0, sDr(s) + 4 * col0, sl2x2, key_local, col0, key_ok, diag,
                              pw, dw);
          tmem_st8x2_issue(tmem + lane_base + col_s(T) + col0, pw, tmem + lane_base + col_s(T) + col0 + 8, dw);
          st_shared_v4(sw128_chunk(sDS, key_local, col0 >> 3), dw[0], dw[1], dw[2], dw[3]);
          st_shared_v4(sw128_chunk(sDS, key_local, (col0 >> 3) + 1), dw[4], dw[5], dw[6], dw[7]);
          if (u & 1) {
            // P^T and dS^T of this chunk in TMEM are read by dV and dK; dS^T in
            // shared memory (async proxy) by dQ after the last chunk.
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(u >> 1));
            BWD_TRACE(tid == 0, T, 9 + (u >> 1));
          }
          if (u < 3) tmem_wait_ld16x2(sv[b ^ 1], dpv[b ^ 1]);
        }

        // ---- drain dQ_i = dS K_j (S^T columns).  Warp w holds query rows 32 (w % 4)..
        // and columns [g d/2, (g+1) d/2).  First out of TMEM (the next S^T may then
        // be issued over it), then staged in this query tile's slot once its Q and
        // dO are read; the producer warp reduce-adds the staged boxes.
        ok = pass_all(mbar_wait(dq_full, T & 1, p.status, lim));
        if (!ok) break;
        BWD_TRACE(tid == 0, T, 11);
        tc_fence_after();
        const int row_local = key_local;  // TMEM lane = query row of dQ_i
        uint32_t gq[D / 2];
  #pragma unroll
        for (int c = 0; c < D / 2; c += 32)
          tmem_ld32_sync(tmem + lane_base + col_s(T) + g * (D / 2) + c, *reinterpret_cast<uint32_t(*)[32]>(gq + c));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(drain_done);
        BWD_TRACE(tid == 0, T, 12);
        // Staging address of this thread's 16-byte chunk q4 of box b (row row_local).
        const uint32_t stg = sSlot(s);
        auto chunk_addr = [&](uint32_t slot_base, int b, int q4) {
          return slot_base + b * 16384 + row_local * 128 + ((q4 ^ (row_local & 7)) << 4);
        };
        // The slot's Q and dO have been read (dV and dK were issued before dQ_i).
        ok = pass_all(mbar_wait(q_empty(s), use_par(T), p.status, lim));
        if (!ok) break;
  #pragma unroll
        for (int c = 0; c < D / 2; c += 32)
  #pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            st_shared_v4(chunk_addr(stg, (g * (D / 2) + c) / 32, q4),
                         __float_as_uint(__uint_as_float(gq[c + 4 * q4]) * p.scale),
                         __float_as_uint(__uint_as_float(gq[c + 4 * q4 + 1]) * p.scale),
                         __float_as_uint(__uint_as_float(gq[c + 4 * q4 + 2]) * p.scale),
                         __float_as_uint(__uint_as_float(gq[c + 4 * q4 + 3]) * p.scale));
        fence_proxy_async_smem();  // read by the producer's TMA reduce-adds
        __syncwarp();
        if (lane == 0) mbar_arrive(stage_free(s));
        BWD_TRACE(tid == 0, T, 13);
      }

      // ---- epilogue of the item: dK * scale and dV to bf16.  Warp-collective
      // TMEM loads by every lane; only key rows < N are stored.  Once this warp's
      // loads are done, the next item's first dV/dK products may overwrite them.
      ok = pass_all(ok && mbar_wait(fin_bar, r & 1, p.status, lim));
      if (!ok) break;
      BWD_TRACE(tid == 0, T - 1, 5);
      tc_fence_after();
      if constexpr (D == 128) {
        // Staged through this warp's 4 KB of the dS^T buffer (the item's last
        // reader of it, the last dQ product, has completed; the same warp
        // writes that part again in its next pass): its 32 key rows x 64
        // columns of dV, then of dK * scale, as 128-byte rows in the 128-byte
        // swizzle, each written by one TMA store (rows >= N are clipped).
        const uint32_t stg = sDS + warp * 4096;
  #pragma unroll 1
        for (int m = 0; m < 2; ++m) {
          const float f = m ? p.scale : 1.f;
  #pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 32) {
            uint32_t a[32];
            tmem_ld32_sync(tmem + lane_base + (m ? C::kColDK : C::kColDV) + 64 * g + c0, a);
  #pragma unroll
            for (int e = 0; e < 32; e += 8) {
              const int c = (c0 + e) >> 3;  // 16-byte chunk of the 128-byte row
              st_shared_v4(stg + lane * 128 + ((c ^ (lane & 7)) << 4),
                           pack_bf16x2(__uint_as_float(a[e]) * f, __uint_as_float(a[e + 1]) * f),
                           pack_bf16x2(__uint_as_float(a[e + 2]) * f, __uint_as_float(a[e + 3]) * f),
                           pack_bf16x2(__uint_as_float(a[e + 4]) * f, __uint_as_float(a[e + 5]) * f),
                           pack_bf16x2(__uint_as_float(a[e + 6]) * f, __uint_as_float(a[e + 7]) * f));
            }
          }
          if (m == 1) {  // every TMEM read of this warp is done
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_free);
            BWD_TRACE(tid == 0, T - 1, 7);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(m ? &p.tm_dk : &p.tm_dv, stg, 64 * g, j * 128 + 32 * qd, bh);
            bulk_commit_group();
            bulk_wait_read_all();  // the staging is reused (dK, then the next pass's dS^T)
          }
          __syncwarp();
        }
      } else {
        const size_t kr = static_cast<size_t>(bh) * N + (key_ok ? key : 0);
        __nv_bfloat16* dvp = reinterpret_cast<__nv_bfloat16*>(p.dv) + kr * D;
        __nv_bfloat16* dkp = reinterpret_cast<__nv_bfloat16*>(p.dk) + kr * D;
  #pragma unroll 1
        for (int c0 = g * (D / 2); c0 < (g + 1) * (D / 2); c0 += 32) {
          uint32_t a[32], b[32];
          tmem_ld32x2_sync(tmem + lane_base + C::kColDV + c0, a, tmem + lane_base + C::kColDK + c0, b);
          if (!key_ok) continue;
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
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_free);
      }
    }
    if (lane == 0) bulk_wait_all();  // this warp's dV / dK stores have landed
  }

  // ---- teardown: every role has finished with TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Item order of a causal backward.  Key-tile-major puts the heaviest items
// (key tile 0 sees every query tile) first across all heads, and the snake that
// deals the items to the persistent CTAs then evens out their work.  Head-major
// keeps one head's dQ accumulator in L2, but with the static snake its uneven
// item weights balance badly (long causal shape: 1034 against 1202 TFLOP/s for
// key-tile-major), so key-tile-major is the default and
// ATTN_BWD_GRID_ORDER=head (or =key) in the environment chooses explicitly.
cudaError_t causal_head_major(int* out) {
  const char* env = std::getenv("ATTN_BWD_GRID_ORDER");
  *out = (env && std::strcmp(env, "head") == 0) ? 1 : 0;
  return cudaSuccess;
}

// Launches `kern` with programmatic stream serialisation: it may start before
// the previous kernel in the stream has finished, and waits for that kernel's
// results on the device (grid_dependency_wait) before it reads them.
template <class... Params, class... Args>
cudaError_t launch_behind(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <int D, bool kCausal>
cudaError_t launch_main(const BwdParams& p, cudaStream_t stream) {
  auto kern = attn_bwd_tc_kernel<D, kCausal>;
  static std::atomic<unsigned long long> opted_in{0};
  cudaError_t e = smem_opt_in_once(kern, BwdCfg<D>::kSmemBytes, opted_in);
  if (e != cudaSuccess) return e;
  int head_major = 1;
  if (kCausal && (e = causal_head_major(&head_major)) != cudaSuccess) return e;
  const long long n_kt = (p.N + 127) / 128;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long items = n_kt * p.BH;
  const long long grid = items < sms ? items : sms;  // persistent: at most one CTA per SM
  return launch_behind(kern, dim3(static_cast<unsigned>(grid)), dim3(kBwdThreads), BwdCfg<D>::kSmemBytes, stream, p,
                       head_major);
}

}  // namespace

#ifdef ATTN_TRACE
// Trace builds only: read the stamps of the last backward launch.
extern "C" int attn_trace_bwd(unsigned long long* host) {
  return static_cast<int>(cudaMemcpyFromSymbol(host, g_bwd_trace, sizeof(g_bwd_trace)));
}
#endif

cudaError_t launch_bwd(const BwdParams& p, int d, bool causal, cudaStream_t stream) {
  if (d != 64 && d != 128) return cudaErrorInvalidValue;
  const int n_pad = (p.N + 127) / 128 * 128;
  const long long prows = static_cast<long long>(p.BH) * n_pad;
  if (d == 128) {
    constexpr int rpb = prep_rows_per_block<128>();
    attn_bwd_prep_kernel<128><<<static_cast<unsigned>((prows + rpb - 1) / rpb), 256, 0, stream>>>(p, n_pad);
  } else {
    constexpr int rpb = prep_rows_per_block<64>();
    attn_bwd_prep_kernel<64><<<static_cast<unsigned>((prows + rpb - 1) / rpb), 256, 0, stream>>>(p, n_pad);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (d == 128) e = causal ? launch_main<128, true>(p, stream) : launch_main<128, false>(p, stream);
  else e = causal ? launch_main<64, true>(p, stream) : launch_main<64, false>(p, stream);
  if (e != cudaSuccess) return e;
  const long long n4 = static_cast<long long>(p.BH) * p.N * d / 4;
  const long long want = (n4 + 256 * kDqPerThread - 1) / (256 * kDqPerThread);
  const unsigned blocks = static_cast<unsigned>(want < 152LL * 16 ? want : 152LL * 16);
  return launch_behind(attn_bwd_dq_kernel, dim3(blocks), dim3(256), 0, stream, p, n4);
}

}  // namespace attn

// FlashAttention-2-style fused attention forward for sm_103a on the fifth-
// generation tensor cores (tcgen05 + TMEM), fed by TMA.
//
// What it computes follows "FlashAttention-2 from PyTorch to Triton" (the FA2
// forward pass: per query tile, stream key/value tiles, keep running m, l and
// an unnormalised O rescaled by exp(m_old - m_new), divide by l once at the
// end and write L = m + log l) and "1.8x Faster Attention on an RTX 5080: an
// FP8 Flash Attention Kernel in CuTe-DSL" (FP8 descales folded into the score
// scale, P scaled by 256 before the FP8 cast).  How it runs is GB300-first:
//
//   * one CTA = two 128-row query tiles of one (batch, head); the two tiles
//     ping-pong so the tensor core runs one tile's GEMM while the other tile's
//     softmax runs on the CUDA cores ("Kernels and Memory in LLM Inference",
//     FlashAttention-3/-4 sections: overlap the two jobs);
//   * warp specialisation: warps 0-3 and 4-7 are the softmax warpgroups of
//     tile 0 and tile 1 (thread r owns query row r: TMEM lane r), warp 8 is the
//     TMA producer, warp 9 allocates TMEM and issues every tcgen05.mma;
//   * S = Q K^T accumulates in TMEM (128 fp32 columns per tile); P (bf16 or
//     e4m3) is written back over the same columns and used as the A operand of
//     O += P V straight from TMEM; O (d fp32 columns per tile) stays in TMEM
//     for the whole key loop.  512 columns: S0 | S1 | O0 | O1;
//   * K and V stream through one ring of 128-key shared-memory slots
//     (K0, V0, K1, V1, ...) with full/empty mbarriers;
//   * exp2 with scale*log2(e) folded into one FFMA per score; the O rescale is
//     skipped for a warp whose 32 rows all kept their max;
//   * causal: only key tiles up to the diagonal are visited, the mask is
//     applied on the diagonal tile only, and heavy query tiles launch first;
//     a ragged last key tile is masked (keys >= N are not phantom zeros).
#pragma once

#include "attn_kernels.h"
#include "ptx_sm103.cuh"

namespace attn {

template <bool kFp8, int kD, bool kCausal, bool kPolyExp2 = false>
struct TcCfg {
  static constexpr bool kIsFp8 = kFp8;
  // Split exponential ("Kernels and Memory in LLM Inference", FlashAttention-4
  // section, item 1): when set, one exponential pair in four is evaluated by
  // the polynomial of exp2_poly.h on the FMA pipe instead of the exponential
  // unit.  An option (attn_set_poly_exp2), off by default.
  static constexpr bool kPoly = kPolyExp2;
  static constexpr int D = kD;
  static constexpr bool kCaus = kCausal;
  static constexpr int kElem = kFp8 ? 1 : 2;                 // bytes per element
  static constexpr int kRowBytes = kD * kElem;               // bytes per tile row
  static_assert(kRowBytes % 128 == 0, "rows must be whole 128-byte swizzle atoms");
  static constexpr int kBlocks = kRowBytes / 128;            // 128-byte column blocks per row
  static constexpr int kBoxCols = 128 / kElem;               // elements per 128-byte block
  static constexpr int kBlockBytes = 128 * 128;              // one column block of a 128-row tile
  static constexpr int kTileBytes = 128 * kRowBytes;         // one 128-row tile
  static constexpr int kMmaK = kFp8 ? 32 : 16;               // K of one tcgen05.mma
  static constexpr int kQkSteps = kD / kMmaK;
  static constexpr int kPvSteps = 128 / kMmaK;
  static constexpr int kStages = (kTileBytes == 32768) ? 5 : 8;
  static constexpr int kPCols = kFp8 ? 32 : 64;              // TMEM columns of one P tile
  // Conditional rescale ("Kernels and Memory in LLM Inference", FlashAttention-4
  // section, item 2): the reference max used in the exponentials moves only
  // when the row max grows by more than kTau (log2 units), so p <= 2^kTau:
  // 8 doublings for bf16 (the section's figure); e4m3 stores P as p * 2^kPExp
  // and keeps 2^(kTau + kPExp) = 256 <= 448 (its largest finite value) with a
  // bound of 4, so that small weights keep their e4m3 precision.  A stale reference leaves a row's dominant weight at 2^x, x in
  // (0, kTau], which the P format rounds while l sums the unrounded p; the
  // normaliser of O adds that rounding back (top_weight_rounding), so the drift
  // costs no accuracy.
  static constexpr float kTau = kFp8 ? 4.f : 8.f;
  static constexpr float kPExp = kFp8 ? 4.f : 0.f;
  static constexpr uint32_t kFmt = kFp8 ? 0u : 1u;
  static constexpr uint32_t kIdescQK = make_idesc(kFmt, 128, 128, 0, 0);
  static constexpr uint32_t kIdescPV = make_idesc(kFmt, 128, kD, 0, 1);
  static constexpr int kQBytes = 2 * kTileBytes;
  static constexpr int kBarOff = kQBytes + kStages * kTileBytes;  // 2*kStages + 15 barriers + TMEM holder
  static constexpr int kSmemBytes = kBarOff + 1024 /*barriers*/ + 1024 /*alignment slack*/;
  // Non-causal: 384 threads with a register split (setmaxnreg) that gives the
  // softmax warps 200 registers; causal: 320 threads at 168 (measured faster
  // there: short items, where the extra warpgroup only adds set-up).
  static constexpr bool kRegSplit = !kCausal;
  static constexpr int kThreads = kRegSplit ? 384 : 320;
  static constexpr uint32_t kRegsSoftmax = 200, kRegsOther = 104;
  // setmaxnreg draws on the registers the block was launched with (168 each).
  static_assert(!kRegSplit || 128 * kRegsOther + 256 * kRegsSoftmax <= 168 * kThreads, "register split too large");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOCol0 = 256;
};

template <int kCols>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[kCols]) {
  if constexpr (kCols == 128) tmem_ld128_sync(taddr, r);
  else if constexpr (kCols == 64) tmem_ld64_sync(taddr, r);
  else tmem_ld32_sync(taddr, r);
}

// A shared-memory descriptor advanced by `off` (bytes / 16) in its start
// address field.  Shared addresses stay below 2^18, so the 14-bit field never
// carries: a 32-bit add on the low word suffices.
__device__ __forceinline__ uint64_t desc_plus(uint64_t d, uint32_t off) {
  return (d & 0xFFFFFFFF00000000ull) | static_cast<uint32_t>(static_cast<uint32_t>(d) + off);
}

// A group of SS-form MMAs (kind::f16 or kind::f8f6f4) from one elected lane:
// slice kk uses descriptors a0 + da[kk], b0 + da[kk]; the first accumulates
// only if `acc0`, the others always.
template <bool kFp8, int kN>
__device__ __forceinline__ void mma_ss_group(uint32_t d, uint64_t a0, uint64_t b0, const uint32_t (&da)[kN],
                                             uint32_t idesc, uint32_t acc0) {
  uint64_t a[kN], b[kN];
#pragma unroll
  for (int i = 0; i < kN; ++i) {
    a[i] = desc_plus(a0, da[i]);
    b[i] = desc_plus(b0, da[i]);
  }
  if constexpr (kN == 4) {
    if constexpr (kFp8)
      asm volatile(
          "{\n .reg .pred p, e;\n setp.ne.b32 p, %10, 0;\n elect.sync _|e, 0xffffffff;\n"
          " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %9, p;\n"
          " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %3, %4, %9, 1;\n"
          " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %5, %6, %9, 1;\n"
          " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %7, %8, %9, 1;\n}" ::"r"(d),
          "l"(a[0]), "l"(b[0]), "l"(a[1]), "l"(b[1]), "l"(a[2]), "l"(b[2]), "l"(a[3]), "l"(b[3]), "r"(idesc),
          "r"(acc0)
          : "memory");
    else
      asm volatile(
          "{\n .reg .pred p, e;\n setp.ne.b32 p, %10, 0;\n elect.sync _|e, 0xffffffff;\n"
          " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %9, p;\n"
          " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %4, %9, 1;\n"
          " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %9, 1;\n"
          " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %9, 1;\n}" ::"r"(d),
          "l"(a[0]), "l"(b[0]), "l"(a[1]), "l"(b[1]), "l"(a[2]), "l"(b[2]), "l"(a[3]), "l"(b[3]), "r"(idesc),
          "r"(acc0)
          : "memory");
  } else {
    static_assert(kN % 4 == 0, "groups of four");
#pragma unroll
    for (int g = 0; g < kN; g += 4) {
      const uint32_t sub[4] = {da[g] - da[g], da[g + 1] - da[g], da[g + 2] - da[g], da[g + 3] - da[g]};
      mma_ss_group<kFp8, 4>(d, desc_plus(a0, da[g]), desc_plus(b0, da[g]), sub, idesc, g == 0 ? acc0 : 1u);
    }
  }
}

// Shared-memory descriptors of a Q or K tile (K-major, 128-byte swizzle) and
// of a V tile (the B operand of P V, MN-major: d contiguous, SBO = 8 key rows,
// LBO = the next 128-byte column block).
template <class C>
__device__ __forceinline__ uint64_t qk_desc(uint32_t tile) { return sdesc_sw128(tile, 16, 1024); }
template <class C>
__device__ __forceinline__ uint64_t v_desc(uint32_t tile) { return sdesc_sw128(tile, C::kBlockBytes, 1024); }

// S = Q K^T from the tiles' descriptors (qk_desc); slice kk of the
// contraction starts `off` bytes further on, which adds off / 16 to the
// start-address field.
template <class C>
__device__ __forceinline__ void issue_qk(uint32_t tmem_s, uint64_t qd, uint64_t kd) {
  uint32_t da[C::kQkSteps];
#pragma unroll
  for (int kk = 0; kk < C::kQkSteps; ++kk) {
    const uint32_t byte = kk * C::kMmaK * C::kElem;                 // offset inside a row
    da[kk] = ((byte / 128) * C::kBlockBytes + (byte % 128)) >> 4;
  }
  mma_ss_group<C::kIsFp8, C::kQkSteps>(tmem_s, qd, kd, da, C::kIdescQK, 0u);
}

// A group of TS-form MMAs (A from TMEM) from one elected lane, in one
// statement: MMA i reads A at TMEM address a[i] and B by descriptor b[i]; the
// first accumulates only if `acc0`, the others always.
#define ATTN_TS_MMA(kind, ia, ib, acc) " @e tcgen05.mma.cta_group::1.kind::" kind " [%0], [%" ia "], %" ib ", %1, " acc ";\n"
template <bool kFp8, int kN>
__device__ __forceinline__ void mma_ts_group(uint32_t d, const uint32_t (&a)[kN], const uint64_t (&b)[kN],
                                             uint32_t idesc, uint32_t acc0) {
  static_assert(kN == 2 || kN == 4, "groups of two or four");
  if constexpr (kN == 2) {
    if constexpr (kFp8)
      asm volatile("{\n .reg .pred p, e;\n setp.ne.b32 p, %2, 0;\n elect.sync _|e, 0xffffffff;\n" ATTN_TS_MMA(
                       "f8f6f4", "3", "5", "p") ATTN_TS_MMA("f8f6f4", "4", "6", "1") "}" ::"r"(d),
                   "r"(idesc), "r"(acc0), "r"(a[0]), "r"(a[1]), "l"(b[0]), "l"(b[1])
                   : "memory");
    else
      asm volatile("{\n .reg .pred p, e;\n setp.ne.b32 p, %2, 0;\n elect.sync _|e, 0xffffffff;\n" ATTN_TS_MMA(
                       "f16", "3", "5", "p") ATTN_TS_MMA("f16", "4", "6", "1") "}" ::"r"(d),
                   "r"(idesc), "r"(acc0), "r"(a[0]), "r"(a[1]), "l"(b[0]), "l"(b[1])
                   : "memory");
  } else {
    if constexpr (kFp8)
      asm volatile("{\n .reg .pred p, e;\n setp.ne.b32 p, %2, 0;\n elect.sync _|e, 0xffffffff;\n" ATTN_TS_MMA(
                       "f8f6f4", "3", "7", "p") ATTN_TS_MMA("f8f6f4", "4", "8", "1")
                       ATTN_TS_MMA("f8f6f4", "5", "9", "1") ATTN_TS_MMA("f8f6f4", "6", "10", "1") "}" ::"r"(d),
                   "r"(idesc), "r"(acc0), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "l"(b[0]), "l"(b[1]),
                   "l"(b[2]), "l"(b[3])
                   : "memory");
    else
      asm volatile("{\n .reg .pred p, e;\n setp.ne.b32 p, %2, 0;\n elect.sync _|e, 0xffffffff;\n" ATTN_TS_MMA(
                       "f16", "3", "7", "p") ATTN_TS_MMA("f16", "4", "8", "1") ATTN_TS_MMA("f16", "5", "9", "1")
                       ATTN_TS_MMA("f16", "6", "10", "1") "}" ::"r"(d),
                   "r"(idesc), "r"(acc0), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "l"(b[0]), "l"(b[1]),
                   "l"(b[2]), "l"(b[3])
                   : "memory");
  }
}
#undef ATTN_TS_MMA

// One half (keys [64h, 64h + 64)) of O += P V, V given by its descriptor
// (v_desc), issued as one group.
template <class C, int kHalf>
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint64_t vd, bool accumulate) {
  constexpr int kSteps = C::kPvSteps / 2;
  uint32_t a[kSteps];
  uint64_t b[kSteps];
#pragma unroll
  for (int i = 0; i < kSteps; ++i) {
    const int kk = kHalf * kSteps + i;
    b[i] = desc_plus(vd, (kk * C::kMmaK * 128) >> 4);
    a[i] = tmem_p + kk * 8;  // kMmaK elements of P = 8 TMEM columns
  }
  mma_ts_group<C::kIsFp8, kSteps>(tmem_o, a, b, C::kIdescPV, accumulate ? 1u : 0u);
}

// Exponentials of one packed pair of exponents (log2 units), in place into
// s[c], s[c + 1]: the exponential unit, or (pairs the split-exponential option
// selects) the polynomial on the FMA pipe.  Pair k of a 64-key half is
// polynomial when C::kPoly and k % 4 == 0.
template <class C>
__device__ __forceinline__ void exp2_pair(uint64_t x2, float& lo, float& hi, int pair) {
  if (C::kPoly && (pair & 3) == 0) {
    const uint64_t y = exp2_poly_x2(x2);
    lo = f2_lo(y);
    hi = f2_hi(y);
  } else {
    lo = ex2_approx(f2_lo(x2));
    hi = ex2_approx(f2_hi(x2));
  }
}

// Exponentials of keys [64h, 64h + 64) of this thread's score row, in place,
// and their packed row sums.
template <class C, int kHalf>
__device__ __forceinline__ void exp_half(float (&s)[128], uint64_t sl2x2, uint64_t negx2, uint64_t& rs0,
                                         uint64_t& rs1) {
#pragma unroll
  for (int c = 64 * kHalf; c < 64 * kHalf + 64; c += 4) {
    const uint64_t a = f2_fma(f2_pack(s[c], s[c + 1]), sl2x2, negx2);
    const uint64_t b = f2_fma(f2_pack(s[c + 2], s[c + 3]), sl2x2, negx2);
    exp2_pair<C>(a, s[c], s[c + 1], c / 2);
    exp2_pair<C>(b, s[c + 2], s[c + 3], c / 2 + 1);
    rs0 = f2_add(rs0, f2_pack(s[c], s[c + 1]));
    rs1 = f2_add(rs1, f2_pack(s[c + 2], s[c + 3]));
  }
}

// P for keys [64h, 64h + 64) written to TMEM over the S columns already
// consumed (bf16: 32 columns at 32h; e4m3: 16 columns at 16h).
template <class C, int kHalf>
__device__ __forceinline__ void store_half(const float (&s)[128], uint32_t t_s) {
  if constexpr (C::kIsFp8) {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = 64 * kHalf + 4 * i;
      pk[i] = pack_e4m3x4(s[c], s[c + 1], s[c + 2], s[c + 3]);
    }
    tmem_st16_sync(t_s + 16 * kHalf, pk);
  } else {
    uint32_t pk[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(s[64 * kHalf + 2 * i], s[64 * kHalf + 2 * i + 1]);
    tmem_st32_sync(t_s + 32 * kHalf, pk);
  }
}

template <class C, int kHalf>
__device__ __forceinline__ void softmax_half(float (&s)[128], uint64_t sl2x2, uint64_t negx2, uint64_t& rs0,
                                             uint64_t& rs1, uint32_t t_s) {
  exp_half<C, kHalf>(s, sl2x2, negx2, rs0, rs1);
  store_half<C, kHalf>(s, t_s);
}

// The rounding error that storing a row's largest weight of a key tile in P
// adds (e4m3 or bf16, as store_half rounds it), with p_max computed exactly as
// the exponential pass computes that key's weight (same FFMA, same ex2).
template <class C>
__device__ __forceinline__ float top_weight_rounding(float mx, float sl2, float neg_ref) {
  const float p_max = ex2_approx(fmaf(mx, sl2, neg_ref));
  if constexpr (C::kIsFp8) return e4m3_round(p_max) - p_max;
  else return __bfloat162float(__float2bfloat16_rn(p_max)) - p_max;
}

// Optional event trace (compile with -DATTN_TRACE): per-CTA cycle stamps of
// the pipeline hand-offs of one chosen CTA, for timeline analysis.
#ifdef ATTN_TRACE
static __device__ unsigned long long g_attn_trace[9 * 64 * 8];
static __device__ int g_attn_trace_cta = 0;
// per-CTA [start_ns, end_ns, smid, unused] for occupancy analysis (first 8192 CTAs)
static __device__ unsigned long long g_attn_cta_span[8192 * 4];
#define ATTN_TRACE_EV(on, role, j, ev)                                                      \
  do {                                                                                      \
    if ((on) && (j) < 64) g_attn_trace[((role) * 64 + (j)) * 8 + (ev)] = clock64();        \
  } while (0)
#else
#define ATTN_TRACE_EV(on, role, j, ev) \
  do {                                 \
  } while (0)
#endif

// Work item -> (b*h, pair of query tiles) and the key tiles each query tile visits.
struct Item {
  int bh, pair, split;
  int kv_bh;             // K/V head read by query head bh (differs from bh under grouped-query attention)
  int kv0;               // first key tile of the item's range
  int kv_end0, kv_end1;  // key tiles visited by query tile 0 / 1 (counted from kv0)
};

template <class C>
__device__ __forceinline__ Item decode_item(const TcParams& p, int item, int n_kt) {
  Item it;
  if constexpr (C::kCaus) {
    it.pair = p.n_pairs - 1 - item / p.BH;  // heaviest pairs first
    it.bh = item % p.BH;
    it.split = 0;
    it.kv0 = 0;
    it.kv_end0 = min(2 * it.pair + 1, n_kt);
    it.kv_end1 = min(2 * it.pair + 2, n_kt);
  } else {
    // (b*h, key range, query pair), fastest last: consecutive items share the
    // same head and key range, so concurrent CTAs reuse those K/V tiles in L2.
    const int per_bh = p.n_pairs * p.n_splits;
    it.bh = item / per_bh;
    const int rem = item % per_bh;
    it.split = rem / p.n_pairs;
    it.pair = rem % p.n_pairs;
    it.kv0 = it.split * p.kt_per_split;
    it.kv_end0 = min(n_kt - it.kv0, p.kt_per_split);
    it.kv_end1 = it.kv_end0;
  }
  it.kv_bh = kv_head_index(it.bh, p.H, p.kv_group);
  return it;
}

// Persistent schedule: round r of CTA c takes item r*G + c (even r) or
// r*G + G-1-c (odd r); with items ordered heaviest first this deals the work
// out in a snake, so every CTA ends with about the same total.
__device__ __forceinline__ int item_of_round(int r) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return r * G + ((r & 1) ? (G - 1 - c) : c);
}

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1) attn_fwd_tc_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);

  const uint32_t q_base = base;
  const uint32_t slot_base = base + C::kQBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + C::kBarOff);
  // q_full[2] | q_empty[2] | slot_full[S] | slot_empty[S] | s_full[2] | p_lo[2] | p_hi[2] | o_full[2] |
  // o_empty[2] | mma_done
  const uint32_t bar0 = smem_u32(bars);
  const int kS = C::kStages;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * i; };
  auto q_full = [&](int t) { return bar(t); };
  auto q_empty = [&](int t) { return bar(2 + t); };
  auto slot_full = [&](int s) { return bar(4 + s); };
  auto slot_empty = [&](int s) { return bar(4 + kS + s); };
  auto s_full = [&](int t) { return bar(4 + 2 * kS + t); };
  auto p_lo = [&](int t) { return bar(6 + 2 * kS + t); };
  auto p_hi = [&](int t) { return bar(8 + 2 * kS + t); };
  auto o_full = [&](int t) { return bar(10 + 2 * kS + t); };
  auto o_empty = [&](int t) { return bar(12 + 2 * kS + t); };
  const uint32_t mma_done = bar(14 + 2 * kS);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 15 + 2 * kS);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
#ifdef ATTN_TRACE
  const bool tr = static_cast<int>(blockIdx.x) == g_attn_trace_cta;
#else
  const bool tr = false;
#endif
  (void)tr;

  const int N = p.N;
  const int n_kt = (N + 127) >> 7;
  const int total = p.BH * p.n_pairs * p.n_splits;

  // ---- setup: barriers, TMEM
  if (tid == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(q_full(t), 1);
      mbar_init(q_empty(t), 1);
    }
    for (int s = 0; s < kS; ++s) {
      mbar_init(slot_full(s), 1);
      mbar_init(slot_empty(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(p_lo(t), 4);  // one arrival per softmax warp
      mbar_init(p_hi(t), 4);
      mbar_init(o_full(t), 1);
      mbar_init(o_empty(t), 4);
    }
    mbar_init(mma_done, 1);
    fence_mbarrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_holder);
  const uint64_t lim = p.timeout_ns;
#ifdef ATTN_TRACE
  if (tid == 0 && blockIdx.x < 8192) {
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    g_attn_cta_span[blockIdx.x * 4 + 0] = globaltimer_ns();
    g_attn_cta_span[blockIdx.x * 4 + 2] = smid;
  }
#endif

  // Register split (non-causal instantiations, 384 threads): launched at 168
  // registers per thread (384 x 168 = 64 512); warpgroup 2 (producer, MMA and two
  // idle warps) drops to 104 and the softmax warpgroups rise to 200:
  // 128 x 104 + 256 x 200 = 64 512.  Each warpgroup executes its setmaxnreg once,
  // ahead of its role code.
  if (warp >= 8) {
    if constexpr (C::kRegSplit) setmaxnreg_dec<C::kRegsOther>();
    if (warp == 8) {
      // ================================================================ TMA producer
      // The whole warp runs this loop; one elected lane issues each copy.  The
      // K/V ring position `it` runs on across work items.
      if (lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
      }
      __syncwarp();
      int it = 0, nq = 0;
      bool ok = true;
      auto load_kv = [&](int k, const Item& w) -> bool {  // ring position `it` <- K_{k/2} (even k) or V_{k/2}
        const int s = it % kS;
        if (!__all_sync(0xffffffffu, mbar_wait(slot_empty(s), ((it / kS) & 1) ^ 1u, p.status, lim))) return false;
        mbar_arrive_expect_tx_elect(slot_full(s), C::kTileBytes);
        const CUtensorMap* map = (k & 1) ? &p.tm_v : &p.tm_k;
        for (int b = 0; b < C::kBlocks; ++b)
          tma_load_3d_elect(slot_base + s * C::kTileBytes + b * C::kBlockBytes, map, slot_full(s), b * C::kBoxCols,
                            (w.kv0 + (k >> 1)) * 128, w.kv_bh);
        ++it;
        return true;
      };
      auto load_q = [&](int t, const Item& w) -> bool {
        // Q_t's buffer is free once the previous item's last S_t = Q_t K^T completed.
        if (nq > 0 && !__all_sync(0xffffffffu, mbar_wait(q_empty(t), (nq - 1) & 1, p.status, lim))) return false;
        // A query tile wholly past N (odd tile count) loads rows 0..127 instead;
        // its results are never stored.
        const int y = (2 * w.pair + t) * 128 < N ? (2 * w.pair + t) * 128 : 0;
        mbar_arrive_expect_tx_elect(q_full(t), C::kTileBytes);
        for (int b = 0; b < C::kBlocks; ++b)
          tma_load_3d_elect(q_base + t * C::kTileBytes + b * C::kBlockBytes, &p.tm_q, q_full(t), b * C::kBoxCols, y,
                            w.bh);
        return true;
      };
      for (int r = 0; ok; ++r) {
        const int item = item_of_round(r);
        if (item >= total) break;
        const Item w = decode_item<C>(p, item, n_kt);
        ATTN_TRACE_EV(tr && lane == 0, 8, r, 0);
        // Ring order: K_0, V_0, K_1, V_1, ...; Q_0 goes ahead of K_0 and Q_1 ahead of V_0,
        // so the item's first S_0 = Q_0 K_0^T can start before the previous item's tile 1 is done.
        ok = load_q(0, w) && load_kv(0, w) && load_q(1, w);
        ++nq;
        // Warm L2 with the next item's Q tiles and first K/V tiles.
        const int nitem = item_of_round(r + 1);
        if (ok && nitem < total) {
          const Item nw = decode_item<C>(p, nitem, n_kt);
          for (int t = 0; t < 2; ++t) {
            const int y = (2 * nw.pair + t) * 128 < N ? (2 * nw.pair + t) * 128 : 0;
            for (int b = 0; b < C::kBlocks; ++b) tma_prefetch_3d_elect(&p.tm_q, b * C::kBoxCols, y, nw.bh);
          }
          for (int b = 0; b < C::kBlocks; ++b) {
            tma_prefetch_3d_elect(&p.tm_k, b * C::kBoxCols, nw.kv0 * 128, nw.kv_bh);
            tma_prefetch_3d_elect(&p.tm_v, b * C::kBoxCols, nw.kv0 * 128, nw.kv_bh);
          }
        }
        for (int k = 1; ok && k < 2 * w.kv_end1; ++k) ok = load_kv(k, w);
      }
      // Drain: every copy this warp issued has landed before the CTA may exit.
      for (int t = 0; nq > 0 && t < 2; ++t) mbar_wait(q_full(t), (nq - 1) & 1, p.status, lim);
      for (int k = max(0, it - kS); k < it; ++k) mbar_wait(slot_full(k % kS), (k / kS) & 1, p.status, lim);
    } else if (warp == 9) {
      // ================================================================ MMA issuer
      // Order per key tile j: for each query tile t, O_t += P_t V_j in two halves
      // (each half as soon as the softmax has written it), then S_t = Q_t K_{j+1}^T
      // into the same TMEM columns (tcgen05.mma issued by one thread executes in
      // order, so the P_t reads precede the S_t overwrite).  The whole warp runs
      // the loop; one elected lane issues every tcgen05 instruction.
      auto wait_all = [&](uint32_t b, uint32_t par) {
        return __all_sync(0xffffffffu, mbar_wait(b, par, p.status, lim));
      };
      int it = 0, nq = 0;
      int np[2] = {0, 0};  // P tiles consumed per query tile (phase of p_lo / p_hi)
      const uint64_t qd0 = qk_desc<C>(q_base), qd1 = qk_desc<C>(q_base + C::kTileBytes);
      constexpr bool kShallowRing = C::kStages <= 5;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int item = item_of_round(r);
        if (item >= total) break;
        const Item w = decode_item<C>(p, item, n_kt);
        ok = wait_all(q_full(0), nq & 1);
        if (ok) ok = wait_all(slot_full(it % kS), (it / kS) & 1);
        if (!ok) break;
        tc_fence_after();
        {
          const uint64_t kd = qk_desc<C>(slot_base + (it % kS) * C::kTileBytes);
          issue_qk<C>(tmem + 0, qd0, kd);
          mma_commit_elect(s_full(0));
          if (w.kv_end0 == 1) mma_commit_elect(q_empty(0));  // the item's last use of Q_0
          ok = wait_all(q_full(1), nq & 1);
          if (!ok) break;
          tc_fence_after();
          issue_qk<C>(tmem + 128, qd1, kd);
          mma_commit_elect(s_full(1));
          if (w.kv_end1 == 1) mma_commit_elect(q_empty(1));
          mma_commit_elect(slot_empty(it % kS));
          ++it;
          ATTN_TRACE_EV(tr && lane == 0, 8, r, 1);
        }
        for (int j = 0; ok && j < w.kv_end1; ++j) {
          const int sv = it % kS;
          ok = wait_all(slot_full(sv), (it / kS) & 1);
          if (!ok) break;
          ATTN_TRACE_EV(tr && lane == 0 && nq == 0, 2, j, 4);
          const int itk = it + 1;
          const int sk = itk % kS;
          const bool next = (j + 1 < w.kv_end1);
          // Descriptors and K_{j+1} (loaded right after V_j) ahead of the P
          // waits, so that only the MMA issue itself stands between the
          // softmax's last P store and the next S.  A shallow ring (five 32 KB
          // slots) can still have K_{j+1} in flight here: it is only tested,
          // and waited for after P V if it has not landed.
          const uint64_t vd = v_desc<C>(slot_base + sv * C::kTileBytes);
          uint64_t kd = 0;
          bool k_ready = false;
          if (next) {
            if constexpr (kShallowRing) {
              k_ready = __all_sync(0xffffffffu, mbar_test(slot_full(sk), (itk / kS) & 1));
              if (k_ready) tc_fence_after();
            } else {
              ok = wait_all(slot_full(sk), (itk / kS) & 1);
              if (!ok) break;
              tc_fence_after();
            }
            kd = qk_desc<C>(slot_base + sk * C::kTileBytes);
          }
          (void)k_ready;
          for (int t = 0; t < 2 && ok; ++t) {
            const int kv_end = t ? w.kv_end1 : w.kv_end0;
            if (j < kv_end) {
              // The first O_t += P_t V of an item overwrites O_t: the previous
              // item's epilogue must have read it out.
              if (j == 0 && nq > 0) {
                ok = wait_all(o_empty(t), (nq - 1) & 1);
                if (!ok) break;
              }
              ok = wait_all(p_lo(t), np[t] & 1);
              if (!ok) break;
              ATTN_TRACE_EV(tr && lane == 0 && nq == 0, 2 + t, j, 0);
              tc_fence_after();
              issue_pv<C, 0>(tmem + C::kOCol0 + t * C::D, tmem + t * 128, vd, j > 0);
              ok = wait_all(p_hi(t), np[t] & 1);
              if (!ok) break;
              ATTN_TRACE_EV(tr && lane == 0 && nq == 0, 2 + t, j, 1);
              tc_fence_after();
              issue_pv<C, 1>(tmem + C::kOCol0 + t * C::D, tmem + t * 128, vd, true);
              ATTN_TRACE_EV(tr && lane == 0 && nq == 0, 2 + t, j, 2);
              // V_j's last reader: with a shallow ring its slot is released
              // before the next S is issued, otherwise after it.
              if constexpr (kShallowRing) {
                if (t == 1) mma_commit_elect(slot_empty(sv));
              }
              if (j + 1 < kv_end) {
                if constexpr (kShallowRing) {
                  if (!k_ready) {
                    ok = wait_all(slot_full(sk), (itk / kS) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    k_ready = true;
                  }
                }
                issue_qk<C>(tmem + t * 128, t ? qd1 : qd0, kd);
                mma_commit_elect(s_full(t));
                if (j + 2 == kv_end) mma_commit_elect(q_empty(t));  // the item's last S_t = Q_t K^T
                ATTN_TRACE_EV(tr && lane == 0 && nq == 0, 2 + t, j, 3);
              }
              ++np[t];
              // O_t is read only after its last P.V of the item; earlier rescales
              // rely on S_{j+1} completing after P_j V_j instead.
              if (j == kv_end - 1) mma_commit_elect(o_full(t));
            } else if constexpr (kShallowRing) {
              if (t == 1) mma_commit_elect(slot_empty(sv));
            }
            if constexpr (!kShallowRing) {
              if (t == 1) mma_commit_elect(slot_empty(sv));
            }
          }
          if (!ok) break;
          if (next) mma_commit_elect(slot_empty(sk));
          it += next ? 2 : 1;  // V_j, and K_{j+1} if this item has one (the producer loads 2 per key tile)
        }
        ++nq;
      }
      // Every MMA issued by this warp has completed before TMEM is freed.
      mma_commit_elect(mma_done);
      mbar_wait(mma_done, 0, p.status, lim);
    }
  } else {
    if constexpr (C::kRegSplit) setmaxnreg_inc<C::kRegsSoftmax>();
    // ================================================================ softmax warpgroups
    const int t = tid >> 7;                      // query tile of this warpgroup
    const int r = tid & 127;                     // row inside the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_base + t * 128;
    const uint32_t t_o = tmem + lane_base + C::kOCol0 + t * C::D;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    const bool trw = tr && r == 0;
    (void)trw;
    int ns = 0, nq = 0;  // S tiles consumed, items finished
    bool ok = true;

    for (int rr = 0; ok; ++rr) {
      const int item = item_of_round(rr);
      if (item >= total) break;
      const Item w = decode_item<C>(p, item, n_kt);
      const int qt = 2 * w.pair + t;
      const int row = qt * 128 + r;
      const int kv_end = t ? w.kv_end1 : w.kv_end0;
      float m2 = -INFINITY;  // reference max of s * sl2 (log2 domain)
      float l = 0.f;         // running sum of p * 2^kPExp (fp32 p: gives L)
      float lc = 0.f;        // running sum of the P rounding errors of each key tile's largest weight

      for (int j = 0; j < kv_end; ++j, ++ns) {
        ok = __all_sync(0xffffffffu, mbar_wait(s_full(t), ns & 1, p.status, lim));
        if (!ok) break;
        ATTN_TRACE_EV(trw && nq == 0, t, j, 0);
        ATTN_TRACE_EV(trw && j == 0, 8, rr, 2 + 3 * t);
        ATTN_TRACE_EV(tr && lane == 0 && nq == 0, 4, j, t * 4 + (warp & 3));
        tc_fence_after();
        float s[128];
        {
          uint32_t u[128];
          tmem_ld128_sync(t_s, u);
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(u[c]);
        }
        ATTN_TRACE_EV(tr && lane == 0 && nq == 0, 6, j, t * 4 + (warp & 3));
        const int jj = w.kv0 + j;  // absolute key tile
        const bool diag = C::kCaus && (jj == qt);
        const bool ragged = (jj == n_kt - 1) && ((N & 127) != 0);
        const int key0 = jj * 128;
        const int lim_key = C::kCaus ? min(N - 1, row) : (N - 1);
        if (diag || ragged) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (key0 + c > lim_key) s[c] = -INFINITY;
        }
        // Fast path (every key tile after the first): with the drift bound of
        // kTau doublings the reference max rarely moves, so the exponentials of
        // keys 0..63 are computed with the current reference while the same pass
        // finds the row max; only if some row of the warp grew past the bound is
        // the tile redone on the exact path below (S is still intact in TMEM: P
        // has not been written yet).
        uint64_t rs0 = 0, rs1 = 0;  // packed partial row sums (0 bits == 0.0f)
        bool fast = false;
        if (j > 0) {
          const uint64_t neg_ref = f2_pack(C::kPExp - m2, C::kPExp - m2);
          float ma = -INFINITY, mb = -INFINITY, mc = -INFINITY, md = -INFINITY;
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            ma = fmax3(ma, s[c], s[c + 1]);
            mb = fmax3(mb, s[c + 2], s[c + 3]);
            const uint64_t a = f2_fma(f2_pack(s[c], s[c + 1]), sl2x2, neg_ref);
            const uint64_t b = f2_fma(f2_pack(s[c + 2], s[c + 3]), sl2x2, neg_ref);
            exp2_pair<C>(a, s[c], s[c + 1], c / 2);
            exp2_pair<C>(b, s[c + 2], s[c + 3], c / 2 + 1);
            rs0 = f2_add(rs0, f2_pack(s[c], s[c + 1]));
            rs1 = f2_add(rs1, f2_pack(s[c + 2], s[c + 3]));
          }
#pragma unroll
          for (int c = 64; c < 128; c += 4) {
            mc = fmax3(mc, s[c], s[c + 1]);
            md = fmax3(md, s[c + 2], s[c + 3]);
          }
          const float mx = fmaxf(fmaxf(ma, mb), fmaxf(mc, md));
          fast = !__any_sync(0xffffffffu, mx * sl2 > m2 + C::kTau);
          if (fast) {
            ATTN_TRACE_EV(trw && nq == 0, t, j, 1);
            store_half<C, 0>(s, t_s);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_lo(t));
            ATTN_TRACE_EV(trw && nq == 0, t, j, 2);
            ATTN_TRACE_EV(tr && lane == 0 && nq == 0, 7, j, t * 4 + (warp & 3));
            softmax_half<C, 1>(s, sl2x2, neg_ref, rs0, rs1, t_s);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_hi(t));
            ATTN_TRACE_EV(trw && nq == 0, t, j, 3);
            const uint64_t rs = f2_add(rs0, rs1);
            l += f2_lo(rs) + f2_hi(rs);
            lc += top_weight_rounding<C>(mx, sl2, C::kPExp - m2);
            continue;
          }
          // Slow path: reload the raw scores of keys 0..63 and mask them again.
          uint32_t u2[64];
          tmem_ld64_sync(t_s, u2);
#pragma unroll
          for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(u2[c]);
          if (diag || ragged) {
            const int key0 = jj * 128;
            const int lim_key = C::kCaus ? min(N - 1, row) : (N - 1);
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (key0 + c > lim_key) s[c] = -INFINITY;
          }
          rs0 = rs1 = 0;
        }
        // Exact path: row max first (eight independent three-input max chains,
        // then a short tree), then the reference and the rescale of O and l.
        float mx8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(s[i], s[i + 8]);
#pragma unroll
        for (int c = 16; c < 128; c += 16) {
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            mx8[i] = fmax3(mx8[i], s[c + i], s[c + i + 1]);
            mx8[i + 1] = fmax3(mx8[i + 1], s[c + i + 8], s[c + i + 9]);
          }
        }
        const float mx =
            fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
        // Reference max: moves only when the row max grew by more than kTau (then
        // O and l are rescaled); otherwise p may exceed 1 by at most 2^kTau.
        const float m_cand = fmaxf(m2, mx * sl2);
        const float m_new = (m_cand > m2 + C::kTau) ? m_cand : m2;
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2_approx(m2 - m_use);
        ATTN_TRACE_EV(trw && nq == 0, t, j, 1);
        const uint64_t negx2 = f2_pack(C::kPExp - m_use, C::kPExp - m_use);
        softmax_half<C, 0>(s, sl2x2, negx2, rs0, rs1, t_s);
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // O holds the sum up to key tile j-1 at the old reference: rescale it
          // before the first P V half is released.  S_j being complete implies
          // O += P_{j-1} V_{j-1} is complete (the MMAs of one thread complete in
          // issue order and S_j was committed later).  Keys 0..63 are consumed by
          // now, which leaves registers for 64 columns of O at a time.
          const uint64_t ax2 = f2_pack(alpha, alpha);
#pragma unroll 1
          for (int c0 = 0; c0 < C::D; c0 += 64) {
            uint32_t o[64];
            tmem_ld64_sync(t_o + c0, o);
#pragma unroll
            for (int i = 0; i < 64; i += 2) {
              const uint64_t v = f2_mul(f2_pack(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), ax2);
              o[i] = static_cast<uint32_t>(v);
              o[i + 1] = static_cast<uint32_t>(v >> 32);
            }
            tmem_st64_sync(t_o + c0, o);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_lo(t));
        ATTN_TRACE_EV(trw && nq == 0, t, j, 2);
        ATTN_TRACE_EV(tr && lane == 0 && nq == 0, 7, j, t * 4 + (warp & 3));
        softmax_half<C, 1>(s, sl2x2, negx2, rs0, rs1, t_s);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_hi(t));
        ATTN_TRACE_EV(trw && nq == 0, t, j, 3);
        const uint64_t rs = f2_add(rs0, rs1);
        l = fmaf(l, alpha, f2_lo(rs) + f2_hi(rs));
        lc = fmaf(lc, alpha, top_weight_rounding<C>(mx, sl2, C::kPExp - m_use));
        m2 = m_new;
      }
      if (!ok) break;

      // ---- epilogue of this item: O / l -> bf16, L
      ok = __all_sync(0xffffffffu, mbar_wait(o_full(t), nq & 1, p.status, lim));
      if (!ok) break;
      ATTN_TRACE_EV(trw, 8, rr, 3 + 3 * t);
      tc_fence_after();
      uint32_t o[C::D];
      tmem_ld_cols<C::D>(t_o, o);
      // O is in registers: the next item's first P.V may overwrite it.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty(t));
      // P.V accumulated the rounded P (e4m3 or bf16) while l sums the fp32
      // weights.  On a peaked row one weight carries most of the sum, and its
      // rounding (relative error up to 2^-4 for e4m3, 2^-9 for bf16) would
      // scale O by as much; the normaliser of O therefore adds back each key
      // tile's largest-weight rounding error, so a row's dominant weight divides
      // out exactly.  L keeps the fp32 sum, which has none of that rounding.
      const float inv = p.o_scale / (l + lc);
      const float lse_v = (m2 + log2f(l) - C::kPExp) * 0.69314718055994530942f;
      if (row < N) {
        if (p.part_o != nullptr) {
          // Split-KV: this key range's normalised O (fp32) and L, merged later.
          const size_t prow = (static_cast<size_t>(w.split) * p.BH + w.bh) * N + row;
          float* dst = p.part_o + prow * C::D;
#pragma unroll
          for (int i = 0; i < C::D / 8; ++i) {
            const float* f = reinterpret_cast<const float*>(o) + 8 * i;
            st_global_v8(dst + 8 * i, __float_as_uint(f[0] * inv), __float_as_uint(f[1] * inv),
                         __float_as_uint(f[2] * inv), __float_as_uint(f[3] * inv), __float_as_uint(f[4] * inv),
                         __float_as_uint(f[5] * inv), __float_as_uint(f[6] * inv), __float_as_uint(f[7] * inv));
          }
          p.part_l[prow] = lse_v;
        } else {
          __nv_bfloat16* dst =
              reinterpret_cast<__nv_bfloat16*>(p.o) + (static_cast<size_t>(w.bh) * N + row) * C::D;
#pragma unroll
          for (int i = 0; i < C::D / 16; ++i) {
            const float* f = reinterpret_cast<const float*>(o) + 16 * i;
            st_global_v8(dst + 16 * i, pack_bf16x2(f[0] * inv, f[1] * inv), pack_bf16x2(f[2] * inv, f[3] * inv),
                         pack_bf16x2(f[4] * inv, f[5] * inv), pack_bf16x2(f[6] * inv, f[7] * inv),
                         pack_bf16x2(f[8] * inv, f[9] * inv), pack_bf16x2(f[10] * inv, f[11] * inv),
                         pack_bf16x2(f[12] * inv, f[13] * inv), pack_bf16x2(f[14] * inv, f[15] * inv));
          }
          p.lse[static_cast<size_t>(w.bh) * N + row] = lse_v;
        }
      }
      ATTN_TRACE_EV(trw, 8, rr, 4 + 3 * t);
      ++nq;
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
#ifdef ATTN_TRACE
  if (tid == 0 && blockIdx.x < 8192) g_attn_cta_span[blockIdx.x * 4 + 1] = globaltimer_ns();
#endif
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <class C>
cudaError_t launch_tc(const TcParams& p, int num_sms, cudaStream_t stream) {
  auto kern = attn_fwd_tc_kernel<C>;
  static std::atomic<unsigned long long> opted_in{0};
  cudaError_t e = smem_opt_in_once(kern, C::kSmemBytes, opted_in);
  if (e != cudaSuccess) return e;
  const long long items = static_cast<long long>(p.BH) * p.n_pairs * p.n_splits;
  const long long grid = items < num_sms ? items : num_sms;  // persistent: at most one CTA per SM
  kern<<<dim3(static_cast<unsigned>(grid)), dim3(C::kThreads), C::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace attn

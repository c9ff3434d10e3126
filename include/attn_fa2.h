/*
 * attn_fa2.h -- C ABI of the GB300 (sm_103a) FlashAttention-2-style fused
 * attention forward library (libattn_fa2.so).
 *
 * The operation (per batch b, head h, query row i):
 *     s_ij = scale * sum_c q[i,c] k[j,c]     for every key j (j <= i if causal)
 *     O[i,:] = sum_j exp(s_ij - m_i) v[j,:] / l_i,   m_i = max_j s_ij,
 *     l_i = sum_j exp(s_ij - m_i),   L[i] = m_i + ln l_i   (natural log)
 * Defined by "Kernels and Memory in LLM Inference" (section "Attention, said
 * plainly again": scores, row softmax with the max subtracted, weighted sum of
 * V) and "FlashAttention-2 from PyTorch to Triton" (the FA2 forward pass: the
 * N x N scores never leave the chip; L is the per-row logsumexp kept for the
 * backward pass; causal keeps key j iff j <= query i).  FP8 inputs carry one
 * descale per tensor, folded into the score scale and the output as in
 * "1.8x Faster Attention on an RTX 5080: an FP8 Flash Attention Kernel in
 * CuTe-DSL" (section "Who am I, what's mine?").
 *
 * Conventions for every entry point:
 *   - Alignment: q, k, v 16 bytes; o 16 bytes (fp32 inputs) or 32 bytes
 *     (bf16 / e4m3 inputs); lse 4 bytes.
 *   - Layout: q, k, v, o are [B, H, N, d] row-major and contiguous (d is the
 *     fastest axis; heads of one batch entry follow each other); lse is
 *     [B, H, N] fp32.  Queries and keys have the same length N.
 *   - Ownership: the caller allocates and owns every buffer; the library
 *     allocates no memory and keeps no pointer after the call returns.
 *   - Execution: device entry points only enqueue work on `stream` (a
 *     cudaStream_t passed as void*, NULL = the legacy default stream) and
 *     return without synchronising.  The device pointers must stay valid until
 *     the stream reaches the work.
 *   - Errors: arguments are validated before anything is enqueued; on an
 *     invalid argument nothing is launched and a non-zero attn_status_t is
 *     returned; attn_last_error() gives a one-line message (per thread).
 *     Device-side timeouts (a wait that exceeded the limit set by
 *     attn_set_wait_limit_ns) are reported by attn_get_device_status().
 */
#ifndef ATTN_FA2_H
#define ATTN_FA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of q, k, v.  O is fp32 for ATTN_F32 and bf16 otherwise. */
typedef enum {
  ATTN_F32 = 0,  /* IEEE binary32; d in {16, 32, 64, 128}; CUDA-core kernel           */
  ATTN_BF16 = 1, /* bfloat16; d in {64, 128}; tcgen05 tensor-core kernel             */
  ATTN_E4M3 = 2  /* FP8 E4M3 (finite, max 448) codes; d = 128; tcgen05 tensor cores  */
} attn_dtype_t;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null pointer, size < 1, non-finite or non-positive scale, bad flag */
  ATTN_ERR_UNSUPPORTED = 2, /* valid request the library has no kernel for (e.g. d = 96 for bf16) */
  ATTN_ERR_MISALIGNED = 3,  /* q/k/v/o not 16-byte aligned (o: 32 for bf16/e4m3), lse not 4-byte */
  ATTN_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed; see attn_last_error()            */
  ATTN_ERR_TIMEOUT = 5      /* a device-side wait exceeded its limit (attn_get_device_status)      */
} attn_status_t;

/*
 * Attention forward on device buffers.
 *   q, k, v : device, [B,H,N,d] of `dtype` (ATTN_E4M3: raw codes, descales 1).
 *   o       : device, [B,H,N,d]; fp32 if dtype == ATTN_F32, else bf16.
 *   lse     : device, [B,H,N] fp32, natural-log logsumexp of the scaled scores.
 *   scale   : softmax scale (finite, > 0; 1/sqrt(d) is the usual value).
 *   causal  : 0 = every key; 1 = key j kept iff j <= query i.
 * Returns ATTN_OK once the kernel is enqueued on `stream`.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
             float scale, int causal, int dtype, void* stream);

/*
 * FP8 E4M3 forward with per-tensor descales: the real value of a code c of q
 * is e4m3(c) * q_descale (likewise k, v).  O is bf16, lse fp32.  Descales must
 * be finite and > 0.  Other arguments as attn_fwd.
 */
int attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, float q_descale, float k_descale, float v_descale, int causal, void* stream);

/*
 * Grouped-query attention forward ("Kernels and Memory in LLM Inference",
 * "Store less: MQA, GQA, MLA", "Grouped-query attention (2023)": the query
 * heads are split into groups, and each group reads one K/V head of its own;
 * H_kv = 1 is multi-query attention, H_kv = H ordinary multi-head attention).
 *   q, o, lse : as attn_fwd, with H query heads.
 *   k, v      : device, [B, H_kv, N, d] of `dtype`.
 *   H_kv      : number of K/V heads, >= 1, dividing H.  Query head h reads K/V
 *               head h / (H / H_kv): a group is H / H_kv consecutive query
 *               heads (the pages do not say which heads form a group).
 *   descales  : used for ATTN_E4M3 only (as attn_fwd_fp8), ignored otherwise.
 * Same kernels, dtypes, head dimensions and causal modes as attn_fwd; the
 * shared K/V tiles are fetched once per group from L2.  Invalid H / H_kv:
 * ATTN_ERR_INVALID_ARG, nothing launched.
 */
int attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N,
                 int d, float scale, float q_descale, float k_descale, float v_descale, int causal, int dtype,
                 void* stream);

/*
 * End-to-end forward from host buffers, for callers whose data lives in host
 * memory: enqueues on `stream` the copies h_q/h_k/h_v -> d_q/d_k/d_v, the
 * forward (as attn_fwd_fp8 for ATTN_E4M3, attn_fwd otherwise; descales are
 * ignored unless dtype == ATTN_E4M3), then the copies d_o -> h_o and
 * d_lse -> h_lse.  The caller provides both the host buffers (page-locked for
 * the copies to be asynchronous) and the device buffers, and synchronises the
 * stream before reading h_o / h_lse.  One cudaMemcpyAsync per buffer.
 */
int attn_fwd_host(const void* h_q, const void* h_k, const void* h_v, void* h_o, float* h_lse, void* d_q,
                  void* d_k, void* d_v, void* d_o, float* d_lse, int B, int H, int N, int d, float scale,
                  float q_descale, float k_descale, float v_descale, int causal, int dtype, void* stream);

/*
 * Split-KV planning ("Kernels and Memory in LLM Inference", Flash-Decoding:
 * split the keys into chunks processed in parallel, then merge the partial
 * results by a log-sum-exp rescale).  For the given sizes and requested split
 * count (0 = enough work items to fill every SM of the current device; the
 * count never exceeds the number of 128-key tiles and no key range is left
 * empty) writes the resolved count to *splits_out and the workspace size
 * attn_fwd_split needs to *workspace_bytes_out (0 when it resolves to 1).
 * Either output pointer may be NULL.  d in {64, 128}.
 */
int attn_fwd_split_plan(int B, int H, int N, int d, int n_splits, int* splits_out, size_t* workspace_bytes_out);

/*
 * Non-causal forward with the keys split into ranges (see attn_fwd_split_plan):
 * each (query tile pair, key range) is a separate work item, which keeps every
 * SM busy when B*H*ceil(N/256) is small.  Each range writes its normalised O
 * (fp32) and its L into `workspace`, then a merge kernel writes o (bf16) and
 * lse (fp32) exactly as attn_fwd would.
 *   dtype     : ATTN_BF16 (descales ignored) or ATTN_E4M3 (per-tensor descales).
 *   causal    : must be 0 (ATTN_ERR_UNSUPPORTED otherwise).  Splitting keys is
 *               for grids smaller than the GPU, i.e. few long query rows such
 *               as decode, where a query sees every key; under a causal mask a
 *               query tile's keys end at its diagonal, so equal key ranges
 *               would leave most ranges of early tiles empty, and causal
 *               shapes large enough to need it already give the persistent
 *               kernel (heaviest tiles first) enough work items.
 *   workspace : device, 256-byte aligned, >= the planned bytes, owned by the
 *               caller; its contents are scratch (overwritten by every call).
 * With one resolved range it runs attn_fwd's kernel and touches no workspace.
 */
int attn_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                   float scale, float q_descale, float k_descale, float v_descale, int causal, int dtype,
                   int n_splits, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Allocation-free split-KV forward.  The pages have no counterpart to this
 * entry point: it exists for callers that cannot allocate device memory when
 * they call us -- a plugin inside a host application that owns all device
 * memory through its own pool and gives plugins no allocator, or a
 * latency-critical loop that cannot pay cudaMalloc's implicit synchronisation.
 * It computes exactly what attn_fwd_split computes, but the scratch for the
 * per-range partial results is a 64 MiB array the library itself declares in
 * device memory, so the caller passes only inputs and outputs and the call
 * allocates nothing.
 *   - Sizes whose planned workspace (attn_fwd_split_plan) exceeds 64 MiB are
 *     rejected with ATTN_ERR_UNSUPPORTED; other arguments as attn_fwd_split.
 *   - The array belongs to the library's device code, which CUDA loads onto a
 *     device lazily (by default): the first call on a device loads it there,
 *     which commits the 64 MiB, and looks up the array's device address (once
 *     per device, with that device current).  That first call can therefore
 *     fail with ATTN_ERR_CUDA (out of memory) where later calls cannot; make it
 *     at set-up time, before any stream capture.  From then on the device keeps
 *     the array until the process exits.
 *   - The looked-up address is cached per device ordinal: do not call
 *     cudaDeviceReset on a device while this library is in use there.
 *   - All calls share the array, which keeps the last call's contents; every
 *     byte a call reads it has written first, so nothing needs clearing.
 *     Calls whose work overlaps on the GPU (several streams or threads) race on
 *     the array: serialise them.
 */
int attn_fwd_split_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                           int d, float scale, float q_descale, float k_descale, float v_descale, int causal,
                           int dtype, int n_splits, void* stream);

/*
 * Attention backward ("FlashAttention-2 from PyTorch to Triton", item 5 of what
 * its first kernel leaves out; "Kernels and Memory in LLM Inference", "Training
 * detour (brief)"): the gradients of the forward above with respect to q, k, v
 * for the upstream gradient dout, rebuilding P = exp(S - L) tile by tile from the
 * forward's lse.  With S = scale q k^T and P its row softmax:
 *     dv = P^T dout,  dS = P * (dout v^T - rowsum(dout * o)),
 *     dq = scale dS k,  dk = scale dS^T q.
 *   q, k, v, o, dout : device, [B,H,N,d] bf16 (o and lse as attn_fwd returned them).
 *   lse              : device, [B,H,N] fp32, natural log.
 *   dq, dk, dv       : device, [B,H,N,d] bf16 outputs, 16-byte aligned.
 *   workspace        : device, 256-byte aligned, >= attn_bwd_workspace_size()
 *                      bytes, owned by the caller; scratch (fp32 dq accumulator
 *                      and two fp32 per row, each head's rows padded to a
 *                      multiple of 128), overwritten by every call.
 *   d in {64, 128}; B*H <= 65535.  Other arguments and errors as attn_fwd.
 *   The outputs and the workspace overlap neither each other nor the inputs:
 *   the main kernel may start while the preparation kernel still reads o and
 *   dout (programmatic dependent launch).
 * The launch order of a causal backward (key tile by key tile across heads, or
 * head by head) is chosen from the sizes; the environment variable
 * ATTN_BWD_GRID_ORDER=key or =head, read at each call, forces one.  dk and dv
 * do not depend on the order; dq only through the order of its fp32 additions.
 */
int attn_bwd_workspace_size(int B, int H, int N, int d, size_t* bytes_out);
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
             void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
             float scale, int causal, void* stream);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device: ATTN_OK, or ATTN_ERR_TIMEOUT if a kernel gave up on a wait
 * since the last call (its outputs are then undefined), or ATTN_ERR_CUDA if the
 * synchronisation itself failed.
 */
int attn_get_device_status(void* stream);

/*
 * Split exponential for the e4m3 forward ("Kernels and Memory in LLM
 * Inference", "FlashAttention-4: when the roof moves", item 1: a short
 * polynomial on the CUDA cores computes some exponentials while the
 * exponential unit computes the rest).  on = 1: later e4m3 launches from this
 * process evaluate one exponential pair in four with a degree-3 polynomial on
 * the FMA pipe (max relative error 7.5e-5; exp2_poly.h); on = 0 (the default):
 * every exponential on the exponential unit.  Returns the previous setting, or
 * -1 (nothing changed) for any other value of on.  A tuning knob: results stay
 * within the stated tolerances either way.
 */
int attn_set_poly_exp2(int on);

/* Upper bound (nanoseconds, >= 1e6) on any single device-side wait of later
 * launches from this process; default 2e9 (2 s).  Returns the previous value. */
uint64_t attn_set_wait_limit_ns(uint64_t ns);

/*
 * Self-test of the bounded device-side wait that every kernel of this library
 * uses: enqueues one thread that waits on an mbarrier nothing ever signals,
 * with the given limit (nanoseconds, >= 1e6).  The wait gives up, records
 * ATTN_ERR_TIMEOUT in the device status word and the kernel returns; a later
 * attn_get_device_status() reports (and clears) it.  No fault, no trap, and the
 * device stays usable.  Returns ATTN_OK once enqueued.
 */
int attn_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/* Static description of a status code. */
const char* attn_status_string(int status);

/* Message of the last failed call made by this thread ("" if none). */
const char* attn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_FA2_H */

// Internal declarations shared by the CUDA translation units of libgdn.
// Nothing here is part of the C ABI (include/gdn.h is).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr float kL2Eps = 1e-6f;  // inside the root of the L2 norm of q and k
constexpr int kMaxConvK = 4;

// Per-layer work area, library-owned, laid out as int32 words:
//   [0]            error word (uint32, OR of GDN_FLAG_*)
//   [1 .. 15]      counters, see Cnt
//   then           blk_count[num_blocks]   block-use counts (duplicate check)
//                  items[num_blocks]       active sequences (any length)
//                  dec[num_blocks]         active sequences of length 1
//                  pre_tmp[num_blocks]     active sequences of length > 1, unsorted
//                  pre[num_blocks]         the same, longest first
//                  pre_cp[num_blocks + 1]  chunk prefix: 64-token chunks of pre[0..k)
//                  redo[2 * num_blocks]    per entry k of pre[], a 64-bit mask of the
//                                          v-heads whose chunked prefill met an fp16
//                                          operand out of range (rerun token-serially)
enum Cnt : int {
  kErr = 0,
  kNItems = 1,
  kNDec = 2,
  kNPre = 3,
  kPreTokens = 4,  // total tokens of the length>1 sequences
  kWorkHead = 5,   // dynamic work counter of persistent kernels (reset by the scheduler)
  kPreChunks = 6,  // total 64-token chunks of the length>1 sequences
  kItemHeadC = 7,  // item counters of the persistent chunk-parallel kernels
  kItemHeadK = 8,  // (cintra_kernel, kintra_kernel; reset by the scheduler)
  kDecHead = 9,    // unit counter of the decode kernel (reset by the scheduler)
  kHeaderWords = 16,
};

struct WorkArea {
  int32_t* base;  // kHeaderWords + 5 * num_blocks words
  int num_blocks;
  __host__ __device__ int32_t* header() const { return base; }
  __host__ __device__ int32_t* blk_count() const { return base + kHeaderWords; }
  __host__ __device__ int32_t* items() const { return base + kHeaderWords + 1 * num_blocks; }
  __host__ __device__ int32_t* dec() const { return base + kHeaderWords + 2 * num_blocks; }
  __host__ __device__ int32_t* pre_tmp() const { return base + kHeaderWords + 3 * num_blocks; }
  __host__ __device__ int32_t* pre() const { return base + kHeaderWords + 4 * num_blocks; }
  __host__ __device__ int32_t* pre_cp() const { return base + kHeaderWords + 5 * num_blocks; }
  __host__ __device__ int32_t* redo() const { return base + kHeaderWords + 6 * num_blocks + 1; }
  static constexpr size_t words(int num_blocks) { return kHeaderWords + 8 * (size_t)num_blocks + 1; }
};

// Everything a forward kernel needs, passed by value.
struct FwdParams {
  const void* x;        // [T][C] act
  const void* a;        // [T][Hv] act
  const void* b;        // [T][Hv] act
  const int32_t* cu;    // [N+1]
  const int32_t* blk;   // [N]
  const uint8_t* has_past;  // [N]
  const void* conv_w;   // [C][K] act
  const float* A_log;   // [Hv]
  const float* dt_bias; // [Hv]
  void* out;            // [T][Hv][dv] act
  unsigned char* layer_base;  // first byte of this layer's page
  size_t stride;        // block stride (bytes)
  size_t rec_off;       // recurrent sub-state offset inside a block (bytes)
  int T, N, Hk, Hv, C, K, num_blocks;
  int max_seqlen_hint;  // 0 = unknown; else longer sequences are flagged and skipped
  int decode_late;      // (decode kernel) launched behind the prefill's recurrence
  WorkArea work;
  // prefill scratch, chunk-major over the scheduler's 64-token prefill chunks
  // (chunk index g); nullptr when the pool has not enough of it (the fused
  // chunked kernel is used).  Every tile is in the 128-byte-swizzled shared
  // memory layout of the MMA operand it becomes:
  //   scr_qk [g][Hk] 32 KiB  [q~ ; k~]: 2 K-blocks of (64 q~ rows, 64 k~ rows)
  //   scr_g  [g][Hk]  1 KiB  fp32 [64 tokens][(G, beta) of the two v-heads]
  //   scr_w  [g][Hv] 16 KiB  -w: 2 boxes of 64 channels x 64 tokens
  //   scr_u  [g][Hv] 16 KiB  u = T diag(beta) v, same layout
  //   scr_p  [g][Hv]  8 KiB  P [64 i][64 j]
  //   scr_c  [g]     int4    (first packed row, valid tokens, chunk index
  //                          inside its sequence, index of the sequence in
  //                          the prefill list) (scheduler)
  // (the tiles written by cintra_kernel, read by seq_kernel)
  void* scr_qk = nullptr;
  void* scr_g = nullptr;
  void* scr_w = nullptr;
  void* scr_u = nullptr;
  void* scr_p = nullptr;
  void* scr_c = nullptr;
  // the per-channel-decay rule's split prefill: its gate tile scr_g holds
  // e^{Gamma_C}, the chunk's decay of every key channel, fp32 [2 v-heads][128],
  // and it adds
  //   scr_v  [g][Hv] 16 KiB  v: 2 boxes of 64 channels x 64 tokens (conv output)
  //   scr_qh [g][Hv] 32 KiB  [q~ e^{Gamma_i} ; k~ e^{Gamma_C - Gamma_j}] in
  //                          the [q~ ; k~] layout, per v-head
  void* scr_v = nullptr;
  void* scr_qh = nullptr;
};

// The Mamba2 mixer's forward (conv over x | B | C, then the selective scan).
struct SsdParams {
  const void* xbc;         // [T][C] act, C = H*P + 2*G*N
  const void* dt;          // [T][H] act
  const int32_t* cu;       // [N+1]
  const int32_t* blk;      // [N]
  const uint8_t* has_past; // [N]
  const void* conv_w;      // [C][K] act
  const float* A_log;      // [H]
  const float* dt_bias;    // [H]
  const float* Dskip;      // [H]
  void* y;                 // [T][H][P] act
  unsigned char* layer_base;
  size_t stride;           // block stride (bytes)
  size_t ssm_off;          // SSM sub-state [H][P][N] fp32 offset inside a block
  int T, N, H, G, C, K;
  WorkArea work;
};

// Launch with programmatic stream serialization: the grid may be scheduled
// before the previous kernel on the stream completes; the kernel orders
// itself with pdl_wait_then_release() before touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
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
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Launchers (each returns a cudaError_t from the launch).
cudaError_t launch_schedule(const FwdParams& p, cudaStream_t stream);
// The token-serial kernel runs over all active sequences (long_only = false)
// or only over those longer than one token (long_only = true).
cudaError_t launch_recurrent(const FwdParams& p, int d, int act, int max_items, bool long_only,
                             cudaStream_t stream);
// The token-serial kernel in redo mode: for every prefill-list entry whose
// redo mask (WorkArea::redo) has bits set, recompute exactly those v-heads
// from the states still in the block, writing their outputs and recurrent
// states (not the conv state, which the conv-state update writes after it).
cudaError_t launch_redo(const FwdParams& p, int d, int act, int max_pre, cudaStream_t stream);
// Mark v-head h of prefill-list entry k for the redo.
__device__ __forceinline__ void mark_redo(const WorkArea& w, int k, int h) {
  atomicOr(reinterpret_cast<unsigned*>(w.redo()) + 2 * k + (h >> 5), 1u << (h & 31));
}
__device__ __forceinline__ bool redo_marked(const WorkArea& w, int k, int h) {
  return (reinterpret_cast<const unsigned*>(w.redo())[2 * k + (h >> 5)] >> (h & 31)) & 1u;
}
// The persistent decode kernel (length-1 sequences): d_k = d_v = 128, bf16
// activations, Hv = 2 Hk, K = 4.  late: launched right behind the prefill's
// recurrence, whose idle SMs it takes without waiting for it (it waits only
// before its CTAs end); otherwise right behind the scheduler.
bool decode_supported(int d, int act, int Hk, int Hv, int K);
cudaError_t launch_decode(const FwdParams& p, int max_dec, cudaStream_t stream, bool late = false);
// The tcgen05 chunked prefill kernel (length > 1 sequences) and the conv-state
// update that follows it: d_k = d_v = 128, bf16 activations, K = 4.  With
// max_dec > 0 the decode kernel runs late, between the recurrence and the
// redo.
bool chunk_supported(int d, int act, int K);
cudaError_t launch_chunk(const FwdParams& p, int max_pre, cudaStream_t stream, int max_dec = 0);
// Conv, gates and the state-independent products of every prefill (64-token
// chunk, k-head), on a persistent grid of up to 2 num_sms CTAs, writing the
// scratch the recurrence kernel reads (max_chunks: host bound on the number
// of 64-token chunks of the prefill sequences).  x_map: the CUtensorMap of x
// (boxes of 64 channels x 67 rows, 128-byte swizzle).
// With conv_only, only the conv: the [q~ ; k~] tiles to scr_qk and the v
// tiles to scr_v (the per-channel-decay rule's first pass).
cudaError_t launch_cintra(const FwdParams& p, const void* x_map, int max_chunks, bool conv_only,
                          int num_sms, cudaStream_t stream);
// The state recurrence over the prefill chains, reading the chunk-major tiles
// cintra_kernel (kda: kintra_kernel) leaves in the prefill scratch.
cudaError_t launch_seq(const FwdParams& p, int grid, bool kda, cudaStream_t stream);
// The per-channel-decay rule's state-independent chunk products of every (64-token chunk,
// v-head), from the conv-only pass's tiles: gates, the decayed q / k tiles, A
// and P, the solve, u and -w; a persistent grid of up to num_sms CTAs.
cudaError_t launch_kintra(const FwdParams& p, int max_chunks, int num_sms, cudaStream_t stream);
// The per-channel-decay (KDA) rule: p.a is [T][Hv][d_k] and p.dt_bias
// [Hv][d_k].  Decode kernel for the shapes decode_supported() accepts, and the
// token-serial kernel (as launch_recurrent) for everything else.
cudaError_t launch_kda_decode(const FwdParams& p, int max_dec, cudaStream_t stream,
                              bool late = false);
cudaError_t launch_kda_recurrent(const FwdParams& p, int d, int act, int max_items,
                                 bool long_only, cudaStream_t stream);
// The KDA token-serial kernel in redo mode (as launch_redo; d = 128, bf16).
cudaError_t launch_kda_redo(const FwdParams& p, int max_pre, cudaStream_t stream);
// The KDA split prefill (d = 128, bf16, Hv = 2 Hk, K = 4, scratch present):
// conv-only pass, kintra, the recurrence, the redo of out-of-range chains and
// the conv-state update; with max_dec > 0 the KDA decode kernel runs late,
// between the recurrence and the redo.
cudaError_t launch_kda_chunk(const FwdParams& p, int max_pre, cudaStream_t stream,
                             int max_dec = 0);
// The Mamba2 scan: token-serial kernel over every active sequence (or, with
// long_only, those longer than one token), then their conv-state update (head
// dim P in {32, 64}, state size in {32, 64, 128}); and the persistent decode
// kernel for length-1 sequences at P = 64, N = 128, K = 4, bf16, H/G a
// multiple of 8 up to 16.
bool ssd_supported(int P, int NS);
cudaError_t launch_ssd(const SsdParams& p, int P, int NS, int act, int max_items,
                       bool long_only, cudaStream_t stream);
bool ssd_decode_supported(int H, int P, int NS, int G, int K, int act);
cudaError_t launch_ssd_decode(const SsdParams& p, int max_dec, cudaStream_t stream);
// The chunked tensor-core scan of the prefill sequences (P = 64, N = 128, bf16,
// H even): conv into the fp16 scratch xs [T][C], the chunk kernel, the
// conv-state update.
bool ssd_chunk_supported(int H, int P, int NS, int K, int act);
cudaError_t launch_ssd_chunk(const SsdParams& p, void* xs, int max_pre, cudaStream_t stream);

// The scalar-gate split prefill's scratch (host side, gdn_api.cu): bytes per
// 64-token chunk, the chunks a call with T tokens and N sequences can need on
// a pool of num_blocks blocks, and the part pointers of a buffer of cap_units
// chunks laid out part-major.
size_t prefill_scratch_unit_bytes(int Hk, int Hv, int dk, int dv);
size_t prefill_scratch_units(long long T, long long N, int num_blocks);
void prefill_scratch_parts(unsigned char* base, size_t cap_units, int Hk, int Hv, int dk, int dv,
                           FwdParams* fp);

// The dense neighbours (gdn_proj.cu): C_g = A B_g^T for up to four groups
// sharing A (bf16, row-major, K contiguous; fp32 accumulation; bf16 out), and
// the gated RMS norm of the output (d_v = 128).
cudaError_t launch_gemm(const void* A, int M, int K, int lda, int n_groups, const void* const* B,
                        const int* N, const int* ldb, void* const* C, const int* ldc,
                        unsigned* flags, cudaStream_t stream);
cudaError_t launch_gated_norm(const void* o, const void* z, const float* w, void* on, int rows,
                              float eps, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Device helpers.

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// softplus(x) = log(1 + e^x) without overflow: x + log1p(e^-x) for x > 0.
__device__ __forceinline__ float softplus_f32(float x) {
  return x > 0.f ? x + log1pf(__expf(-x)) : log1pf(__expf(x));
}
// Fast reciprocal division (__fdividef): 2 ulp, and exactly 0 once the
// denominator overflows, which is the limit of both functions there.
__device__ __forceinline__ float sigmoid_f32(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }
__device__ __forceinline__ float silu_f32(float y) { return __fdividef(y, 1.f + __expf(-y)); }
// max(|a|, |b|, |c|) in one instruction (the three-input max of sm_100 and
// later, on absolute values); a NaN input is skipped, as fmaxf does.
__device__ __forceinline__ float max_abs3(float a, float b, float c) {
  float r;
  asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// The same, but a NaN input gives NaN.
__device__ __forceinline__ float max_abs3_nan(float a, float b, float c) {
  float r;
  asm("max.NaN.abs.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

}  // namespace gdn

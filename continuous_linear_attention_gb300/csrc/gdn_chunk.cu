// Fused chunked prefill kernel: the gated delta rule over sequences longer
// than one token, in chunks of C = 64 tokens with the WY / UT-transform form,
// conv prologue included, the dense intra-chunk and state products on the
// 5th-generation tensor cores (tcgen05.mma, fp16 operands from
// 128-byte-swizzled shared tiles, fp32 accumulators in tensor memory).  The
// recurrent state stays in tensor memory (fp32) for the whole sequence; only
// the final state is written back.  This single-kernel form runs when the pool
// has not enough prefill scratch (see gdn_state_pool_reserve); with scratch,
// the same computation runs split into cintra_kernel and seq_kernel.
//
// Persistent CTAs (8 warps, one per SM) pull (sequence, v-head) chains,
// longest sequences first.
// Per chunk, with G_i the inclusive cumulative gate inside the chunk, beta_i
// the write strength, q~/k~ the normalised rows and S0 the state at the chunk
// start (S is d_v x d_k, S[v][k]):
//   prep (CUDA cores): conv + SiLU + L2 norms + gates from the chunk's x rows,
//        which 2-D TMA copies staged in shared memory while the previous chunk
//        ran; fp16 tiles [q~ ; k~], (k~ e^{G_C - G})^T, beta v
//   state hand-over: S0 -> fp16 tile; TMEM S <- e^{G_C} S0
//   MMA  X  = [q~ ; k~] k~^T                     (QK^T and KK^T, 128 x 64)
//   MMA  [Oq | Yk] = S0 [q~ ; k~]^T              (S0 q~_i and S0 k~_i, 128 x 128)
//   CUDA A_ij = beta_i e^{G_i-G_j} (k~_i.k~_j) (j<i);  P_ij = (q~_i.k~_j) e^{G_i-G_j} (j<=i)
//        R^T[.,i] = beta_i v_i - beta_i e^{G_i} Yk[.,i];  T = (I + A)^{-1} (blocked
//        forward substitution: 16 x 16 diagonal blocks, then the off-diagonal
//        blocks level by level)
//   MMA  U^T = R^T T^T          (the per-token updates u_i, 128 x 64)
//   MMA  O2  = U^T P^T
//        o_i = e^{G_i} Oq[.,i] + O2[.,i] = e^{G_i} S0 q~_i + sum_{j<=i} e^{G_i-G_j}(q~_i.k~_j) u_j
//   MMA  S  += U^T (k~ e^{G_C-G})  (S_C = e^{G_C} S0 + sum_j e^{G_C-G_j} u_j k~_j^T)
// MMA operands are fp16 (same tensor-core rate as bf16, 3 more mantissa bits:
// the bf16 version of this kernel sat at ~4.5e-3 relative error on slowly
// decaying states).  A chain with an operand outside the fp16 range leaves its
// block's state untouched and is rerun by the token-serial kernel (redo mode)
// in the same call.
// Every exponent is of a non-positive number.  Tokens past the end of a
// partial chunk get zero q/k/v, beta = 0 and g = 0, which leaves everything
// unchanged.  This is the chunked form of the gated delta rule (Gated Delta
// Networks); "Continuous batching for linear attention layers" runs such a
// kernel over cu_seqlens with per-sequence initial and final states.
//
// The conv state is only read here; the new conv states of these sequences
// are written by tail_update_kernel, launched after this kernel, so no chain
// can see another chain's write.
#include <cuda.h>

#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

using E = __half;             // MMA operand type
constexpr int D = 128;
constexpr int CH = 64;        // chunk
constexpr int KC = 4;         // conv taps
constexpr int kThreads = 256;
constexpr int kLocalCh = 3 * D;  // q, k of the k-head and v of the v-head
constexpr float kF16Max = 65000.f;

// shared memory map (offsets from a 1024-byte aligned base).  Row pitches of
// the row-parallel buffers are padded (fp32 68, fp16 136, bf16 392 elements)
// so that rows spread over all shared-memory banks.
constexpr int AP = 68;                 // pitch of A and T rows (floats)
constexpr int BVP = 136;               // pitch of beta v rows (halves)
constexpr int XROWS = CH + KC - 1;     // 67 staged rows: 3 halo + 64 chunk rows
constexpr uint32_t XSUB = 9216;        // one staged box: 72 rows x 128 B (64 channels), swizzled
constexpr uint32_t XBOX_BYTES = 64 * XROWS * 2;
constexpr uint32_t OFF_QK = 0;         // [q~ ; k~]   2 x (128 rows x 128 B)
constexpr uint32_t OFF_S0 = 32768;     // S0 tile 2 x (128 x 128 B); during the solve: T fp32, Z
constexpr uint32_t OFF_TS = OFF_S0;    // T fp32 [64][AP]
constexpr uint32_t OFF_Z = OFF_S0 + 17408;  // blocked-solve scratch fp32 [6][16][16]
constexpr uint32_t OFF_KPT = 65536;    // k'^T        128 x 128 B
constexpr uint32_t OFF_P = 81920;      // P           64 x 128 B
constexpr uint32_t OFF_T = 90112;      // T           64 x 128 B
constexpr uint32_t OFF_RU = 98304;     // R^T, then U^T   128 x 128 B
constexpr uint32_t OFF_BV = 114688;    // beta v fp16 [64][BVP]
constexpr uint32_t OFF_AM = 132096;    // A fp32 [64][AP]; then the out tile bf16 [64][128]
constexpr uint32_t OFF_XT = 150528;    // 6 staged x boxes (q0 q1 k0 k1 v0 v1), 1024-aligned
constexpr uint32_t OFF_G = 205824;     // G fp32 [64]
constexpr uint32_t OFF_BETA = 206080;  // beta fp32 [64]
constexpr uint32_t OFF_EG = 206336;    // e^{G} fp32 [64]
constexpr uint32_t OFF_F = 206592;     // beta e^{G} fp32 [64]
constexpr uint32_t OFF_TOT = 206848;   // scan partials [2]
constexpr uint32_t OFF_DS = 206864;    // e^{G_C - G} fp32 [64]
constexpr uint32_t OFF_W = 207120;     // conv taps fp32 [4][384]
constexpr uint32_t SMEM_BYTES = 213264 + 1024;
constexpr uint32_t KB_STRIDE = 16384;  // bytes between K-blocks of a 128-row tile

// tensor memory columns
constexpr uint32_t TM_X = 0, TM_OQ = 64, TM_Y = 128, TM_UT = 192, TM_S = 256, TM_O2 = 384;
constexpr uint32_t TM_COLS = 512;

__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, int* flag) {
  if (threadIdx.x == 0) *flag = mbar_wait_bounded(bar, parity) ? 1 : 0;
  __syncthreads();
  return *flag != 0;
}

// Packed fp32 pairs: d = a * b + c on both lanes (one fma.rn.f32x2).
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long pack_f2(float lo, float hi) {
  return (unsigned long long)__float_as_uint(lo) | ((unsigned long long)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ float lo_f(unsigned long long v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_f(unsigned long long v) { return __uint_as_float((uint32_t)(v >> 32)); }

// 8 bf16 -> 4 packed fp32 pairs (bf16 is the high half of an fp32)
__device__ __forceinline__ void load8_bf16_f2(const __nv_bfloat16* p, unsigned long long* v) {
  const uint4 w = *reinterpret_cast<const uint4*>(p);
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j)
    v[j] = (unsigned long long)(u[j] << 16) | ((unsigned long long)(u[j] & 0xffff0000u) << 32);
}

// Running max of |v| (NaN propagates through the final comparison).
__device__ __forceinline__ void track_abs(float& m, const float* v, int n) {
#pragma unroll
  for (int e = 0; e < n; ++e) m = fmaxf(m, fabsf(v[e]));
}

// The conv prologue runs here from 2-D TMA boxes of x (tmx = x map).
__global__ void __launch_bounds__(kThreads, 1)
chunk_kernel(FwdParams p, const __grid_constant__ CUtensorMap tmx) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t bar;   // MMA completion
  __shared__ uint64_t xbar;  // staged x rows
  __shared__ uint32_t tmem_slot;
  __shared__ int flag;
  __shared__ int s_chain;

  pdl_wait_then_release();
  const int tid = threadIdx.x;
  const int Hk = p.Hk, Hv = p.Hv, C = p.C;
  const int R = Hv / Hk;
  int32_t* hdr = p.work.header();
  const int n_chains = hdr[kNPre] * Hv;
  if ((int)blockIdx.x >= n_chains) return;
  const __nv_bfloat16* __restrict__ wconv = reinterpret_cast<const __nv_bfloat16*>(p.conv_w);
  const __nv_bfloat16* __restrict__ av = reinterpret_cast<const __nv_bfloat16*>(p.a);
  const __nv_bfloat16* __restrict__ bv = reinterpret_cast<const __nv_bfloat16*>(p.b);
  __nv_bfloat16* __restrict__ out = reinterpret_cast<__nv_bfloat16*>(p.out);

  float* G = reinterpret_cast<float*>(sm + OFF_G);
  float* BETA = reinterpret_cast<float*>(sm + OFF_BETA);
  float* EG = reinterpret_cast<float*>(sm + OFF_EG);
  float* F = reinterpret_cast<float*>(sm + OFF_F);
  float* DSC = reinterpret_cast<float*>(sm + OFF_DS);
  float* WS = reinterpret_cast<float*>(sm + OFF_W);
  __half* BV = reinterpret_cast<__half*>(sm + OFF_BV);
  float* AM = reinterpret_cast<float*>(sm + OFF_AM);
  __nv_bfloat16* OT = reinterpret_cast<__nv_bfloat16*>(sm + OFF_AM);
  unsigned char* XT = sm + OFF_XT;
  float* TS = reinterpret_cast<float*>(sm + OFF_TS);
  float* Z = reinterpret_cast<float*>(sm + OFF_Z);
  float* TOT = reinterpret_cast<float*>(sm + OFF_TOT);
  const uint32_t sbase = smem_u32(sm);

  // ---- set-up: barriers, TMEM (kept for every chain this CTA runs)
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init(&xbar, 1);
    fence_mbar_init();
  }
  if (tid < 32) tc::tmem_alloc(&tmem_slot, TM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  // TMEM lane quarter of this warp (warps w and w + 4 share lanes 32 (w % 4) ..)
  const uint32_t lane = (uint32_t)(tid & 96) << 16;
  const int r128 = tid & 127;  // TMEM row (lane) of this thread
  const int chalf = tid >> 7;  // which half of the columns this thread handles
  uint32_t phase = 0, xphase = 0;
  const float inv_sqrt_d = rsqrtf((float)D);
  bool failed = false;
  float amax = 0.f;  // largest |value| converted to an fp16 operand in this chain

  // ---- chains, longest sequences first, pulled from the scheduler's counter
  for (;;) {
  if (tid == 0) s_chain = atomicAdd(&hdr[kWorkHead], 1);
  __syncthreads();
  const int chain = s_chain;
  if (chain >= n_chains) break;
  const int s = p.work.pre()[chain / Hv];
  const int h = chain % Hv;
  const int kh = h / R;
  const int seq0 = p.cu[s];
  const int L = p.cu[s + 1] - seq0;
  const int wblk = p.blk[s];
  const int rblk = p.has_past[s] ? wblk : 0;
  const unsigned char* rbase = p.layer_base + (size_t)rblk * p.stride;
  unsigned char* wbase = p.layer_base + (size_t)wblk * p.stride;
  const __nv_bfloat16* __restrict__ tail_r = reinterpret_cast<const __nv_bfloat16*>(rbase);

  // global channel of local channel lc (q | k of the k-head, v of the v-head)
  auto gch = [&](int lc) {
    return lc < D ? kh * D + lc
                  : (lc < 2 * D ? Hk * D + kh * D + (lc - D) : 2 * Hk * D + h * D + (lc - 2 * D));
  };
  // Stage chunk cc's inputs, thread 0: the x rows (packed rows
  // seq0 + cc*64 - 3 .. + 63) of this chain's q, k and v channels into XT, six
  // 64-channel x 67-row TMA boxes, 128-byte swizzled; rows outside the
  // sequence are loaded too but never used.
  auto stage = [&](int cc) {
    const int r0 = seq0 + cc * CH - (KC - 1);
    mbar_arrive_expect_tx(&xbar, 6u * XBOX_BYTES);
#pragma unroll
    for (int b6 = 0; b6 < 6; ++b6) tma_load_2d(XT + b6 * XSUB, &tmx, gch(b6 * 64), r0, &xbar);
  };
  // gate inputs of chunk cc, token tid (threads < 64)
  auto load_gates = [&](int cc, float& a_, float& b_) {
    const int cc0 = cc * CH;
    if (tid < CH && cc0 + tid < L) {
      const size_t row = (size_t)(seq0 + cc0 + tid);
      a_ = __bfloat162float(av[row * Hv + h]);
      b_ = __bfloat162float(bv[row * Hv + h]);
    }
  };
  if (tid == 0) stage(0);
  float a_nx = 0.f, b_nx = 0.f;
  load_gates(0, a_nx, b_nx);
  for (int lc = tid; lc < kLocalCh; lc += kThreads) {
    const int gc = gch(lc);
#pragma unroll
    for (int j = 0; j < KC; ++j) WS[j * kLocalCh + lc] = __bfloat162float(wconv[(size_t)gc * KC + j]);
  }
  const float A_neg = -__expf(p.A_log[h]);
  const float dtb = p.dt_bias[h];
  __syncthreads();

  const int n_chunks = (L + CH - 1) / CH;
  for (int c = 0; c < n_chunks; ++c) {
    const int c0 = c * CH;                 // chunk start inside the sequence
    const int n = min(CH, L - c0);         // valid tokens
    // ---------------- gates and their in-chunk cumulative sum
    if (tid < CH) {
      float g = 0.f, beta = 0.f;
      if (tid < n) {
        g = A_neg * softplus_f32(a_nx + dtb);
        beta = sigmoid_f32(b_nx);
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, g, o);
        if ((tid & 31) >= o) g += t;
      }
      if ((tid & 31) == 31) TOT[tid >> 5] = g;
      G[tid] = g;
      BETA[tid] = beta;
    }
    __syncthreads();
    if (tid < CH) {
      const float Gi = G[tid] + (tid >= 32 ? TOT[0] : 0.f);
      G[tid] = Gi;
      const float e = __expf(Gi);
      EG[tid] = e;
      F[tid] = BETA[tid] * e;
    }
    if (!cta_wait(&xbar, xphase, &flag)) { failed = true; break; }  // also publishes G
    xphase ^= 1;
    const float GC = G[CH - 1];
    if (tid < CH) DSC[tid] = __expf(GC - G[tid]);
    if (c == 0) {
      // the first chunk's three halo rows are the conv state, not packed rows
      // of another sequence: overwrite the staged ones (16 bytes per thread)
      if (tid < 3 * 48) {
        const int r = tid / 48, q8 = tid % 48;   // row, 8-channel group (6 boxes x 8)
        const int b6 = q8 >> 3, cc = (q8 & 7) * 8;
        *reinterpret_cast<uint4*>(XT + b6 * XSUB + tc::sw128_offset(r, cc)) =
            *reinterpret_cast<const uint4*>(tail_r + (size_t)r * C + gch(b6 * 64 + cc));
      }
      __syncthreads();
    }

    // ---------------- prep: conv + SiLU + norms -> fp16 tiles
    // Thread (tq, g) computes 8-channel group g of q, of k and of v for the four
    // tokens 4tq .. 4tq+3 with a sliding window over 7 staged rows; the 16
    // threads of a token quad reduce the norms with shuffles.
    {
      const int tq = tid >> 4, g = tid & 15;
      const int i0 = 4 * tq;
#pragma unroll
      for (int part = 0; part < 3; ++part) {   // 0: q, 1: k, 2: v
        const int lc0 = part * D + g * 8;
        const int sub = lc0 >> 6, cc = lc0 & 63;
        unsigned long long w2[KC][4];  // taps as packed channel pairs
#pragma unroll
        for (int j = 0; j < KC; ++j) {
          const float4 w0 = *reinterpret_cast<const float4*>(WS + j * kLocalCh + lc0);
          const float4 w1 = *reinterpret_cast<const float4*>(WS + j * kLocalCh + lc0 + 4);
          w2[j][0] = pack_f2(w0.x, w0.y); w2[j][1] = pack_f2(w0.z, w0.w);
          w2[j][2] = pack_f2(w1.x, w1.y); w2[j][3] = pack_f2(w1.z, w1.w);
        }
        unsigned long long acc2[4][4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc2[t][e] = 0ull;
#pragma unroll
        for (int rr = 0; rr < 4 + KC - 1; ++rr) {
          const int r = i0 + rr;    // staged row
          unsigned long long xv2[4];
          load8_bf16_f2(reinterpret_cast<const __nv_bfloat16*>(XT + sub * XSUB + tc::sw128_offset(r, cc)), xv2);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int j = rr - t;   // tap of this row for token i0 + t
            if (j >= 0 && j < KC) {
#pragma unroll
              for (int e = 0; e < 4; ++e) acc2[t][e] = fma2(w2[j][e], xv2[e], acc2[t][e]);
            }
          }
        }
        float acc[4][8];
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[t][2 * e] = lo_f(acc2[t][e]);
            acc[t][2 * e + 1] = hi_f(acc2[t][e]);
          }
        float y[4][8], ss[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const bool valid = i0 + t < n;
          ss[t] = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            y[t][e] = valid ? silu_f32(acc[t][e]) : 0.f;
            ss[t] += y[t][e] * y[t][e];
          }
        }
        if (part < 2) {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) ss[t] += __shfl_xor_sync(0xffffffffu, ss[t], o);
            const bool valid = i0 + t < n;
            const float sc = valid ? rsqrtf(ss[t] + kL2Eps) * (part == 0 ? inv_sqrt_d : 1.f) : 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) y[t][e] *= sc;
            const int i = i0 + t;
            tc::sw128_store8<E>(sm + OFF_QK + (g >> 3) * KB_STRIDE, part * CH + i, (g & 7) * 8, y[t]);
          }
        } else {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int i = i0 + t;
            const float bi = BETA[i];
            uint4 wv;
            wv.x = tc::pack2(bi * y[t][0], bi * y[t][1], (__half*)nullptr);
            wv.y = tc::pack2(bi * y[t][2], bi * y[t][3], (__half*)nullptr);
            wv.z = tc::pack2(bi * y[t][4], bi * y[t][5], (__half*)nullptr);
            wv.w = tc::pack2(bi * y[t][6], bi * y[t][7], (__half*)nullptr);
            track_abs(amax, y[t], 8);
            *reinterpret_cast<uint4*>(BV + i * BVP + g * 8) = wv;
          }
        }
      }
    }

    // ---------------- state hand-over: S0 -> fp16 tile, TMEM S <- e^{G_C} S0
    {
      const int v = r128;
      float srow[64];
      if (c == 0) {
        const float* S_r = reinterpret_cast<const float*>(rbase + p.rec_off) + (size_t)h * D * D;
#pragma unroll
        for (int k = 0; k < 64; ++k) srow[k] = S_r[(size_t)(chalf * 64 + k) * D + v];
      } else {
        tc::tmem_ld32(tmem + lane + TM_S + chalf * 64, srow);
        tc::tmem_ld32(tmem + lane + TM_S + chalf * 64 + 32, srow + 32);
        tc::tmem_wait_ld();
      }
      track_abs(amax, srow, 64);
#pragma unroll
      for (int g8 = 0; g8 < 8; ++g8)
        tc::sw128_store8<E>(sm + OFF_S0 + chalf * KB_STRIDE, v, g8 * 8, srow + g8 * 8);
      const float dc = __expf(GC);
#pragma unroll
      for (int k = 0; k < 64; ++k) srow[k] *= dc;
      tc::tmem_st32(tmem + lane + TM_S + chalf * 64, srow);
      tc::tmem_st32(tmem + lane + TM_S + chalf * 64 + 32, srow + 32);
      tc::tmem_wait_st();
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
      tc::mma_tile(tmem + TM_X, sbase + OFF_QK, KB_STRIDE, sbase + OFF_QK + CH * 128, KB_STRIDE, 2,
                   tc::idesc_f16_f32(128, 64), false);
      tc::mma_tile(tmem + TM_OQ, sbase + OFF_S0, KB_STRIDE, sbase + OFF_QK, KB_STRIDE, 2,
                   tc::idesc_f16_f32(128, 128), false);
      tc::commit(&bar);
    }
    // fused: the staged rows are consumed; bring in the next chunk's while
    // this one runs
    if (c + 1 < n_chunks) {
      if (tid == 0) stage(c + 1);
      load_gates(c + 1, a_nx, b_nx);
    }
    // while the tensor core runs: (k~ e^{G_C - G_i})^T, row k of the 128-row tile
    // read as a column of the k~ tile (thread k, half of the tokens each)
    {
      const int k = r128;
      const unsigned char* ksrc = sm + OFF_QK + (k >> 6) * KB_STRIDE;
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8) {
        const int i0 = chalf * 32 + g8 * 8;
        float v8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          v8[e] = i0 + e < n ? __half2float(*reinterpret_cast<const __half*>(
                                   ksrc + tc::sw128_offset(CH + i0 + e, k & 63))) * DSC[i0 + e]
                             : 0.f;
        tc::sw128_store8<E>(sm + OFF_KPT, k, i0, v8);
      }
    }
    if (!cta_wait(&bar, phase, &flag)) { failed = true; break; }
    phase ^= 1;
    tc::fence_after_sync();

    // ---------------- A, P from X; R^T from Yk (each thread: one row, 32 columns)
    {
      float xr[32];
      tc::tmem_ld32(tmem + lane + TM_X + chalf * 32, xr);
      tc::tmem_wait_ld();
      float Gj[32];
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        const float4 t4 = *reinterpret_cast<const float4*>(G + chalf * 32 + q4 * 4);
        Gj[q4 * 4] = t4.x; Gj[q4 * 4 + 1] = t4.y; Gj[q4 * 4 + 2] = t4.z; Gj[q4 * 4 + 3] = t4.w;
      }
      if (r128 < CH) {
        const int i = r128;
        const float Gi = G[i];
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8) {
          float v8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j = chalf * 32 + g8 * 8 + e;
            v8[e] = (j <= i && i < n) ? xr[g8 * 8 + e] * __expf(Gi - Gj[g8 * 8 + e]) : 0.f;
          }
          tc::sw128_store8<E>(sm + OFF_P, i, chalf * 32 + g8 * 8, v8);
        }
      } else {
        const int i = r128 - CH;
        const float Gi = G[i], bi = BETA[i];
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const int j = chalf * 32 + j4 * 4;
          float4 a4;
          const bool vi = i < n;
          a4.x = (vi && j + 0 < i) ? bi * __expf(Gi - Gj[j4 * 4 + 0]) * xr[j4 * 4 + 0] : 0.f;
          a4.y = (vi && j + 1 < i) ? bi * __expf(Gi - Gj[j4 * 4 + 1]) * xr[j4 * 4 + 1] : 0.f;
          a4.z = (vi && j + 2 < i) ? bi * __expf(Gi - Gj[j4 * 4 + 2]) * xr[j4 * 4 + 2] : 0.f;
          a4.w = (vi && j + 3 < i) ? bi * __expf(Gi - Gj[j4 * 4 + 3]) * xr[j4 * 4 + 3] : 0.f;
          *reinterpret_cast<float4*>(AM + i * AP + j) = a4;
        }
      }
      float yr[32];
      tc::tmem_ld32(tmem + lane + TM_Y + chalf * 32, yr);
      tc::tmem_wait_ld();
      const int v = r128;
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8) {
        const int ib = chalf * 32 + g8 * 8;
        const float4 f0 = *reinterpret_cast<const float4*>(F + ib);
        const float4 f1 = *reinterpret_cast<const float4*>(F + ib + 4);
        const float fv[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
        float v8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int i = ib + e;
          const float bvv = __half2float(BV[i * BVP + v]);
          v8[e] = i < n ? bvv - fv[e] * yr[g8 * 8 + e] : 0.f;
        }
        track_abs(amax, v8, 8);
        tc::sw128_store8<E>(sm + OFF_RU, v, chalf * 32 + g8 * 8, v8);
      }
    }
    __syncthreads();
    // ---------------- T = (I + A)^{-1}: diagonal 16 x 16 blocks, column per thread
    if (tid < CH) {
      const int b = tid >> 4, m = tid & 15;
      const float* Ab = AM + (16 * b) * AP + 16 * b;
      float col[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float acc = r == m ? 1.f : 0.f;
#pragma unroll
        for (int j = 0; j < r; ++j) acc -= Ab[r * AP + j] * col[j];
        col[r] = acc;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) TS[(16 * b + r) * AP + 16 * b + m] = col[r];
    }
    __syncthreads();
    // off-diagonal blocks: B_ij = T_ii A_ij for every i > j (independent), then
    // level by level T_ij = -sum_{k=j}^{i-1} B_ik T_kj; four adjacent columns
    // per thread.  B block (i, j) lives at Z + (i(i-1)/2 + j) * 256.
    for (int task = tid; task < 6 * 64; task += kThreads) {
      const int bi = task >> 6, rr = (task >> 2) & 15, c4 = (task & 3) * 4;
      const int i = bi < 1 ? 1 : (bi < 3 ? 2 : 3);
      const int j = bi - i * (i - 1) / 2;
      float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float t = TS[(16 * i + rr) * AP + 16 * i + q];
        const float4 a4 = *reinterpret_cast<const float4*>(AM + (16 * i + q) * AP + 16 * j + c4);
        z.x += t * a4.x; z.y += t * a4.y; z.z += t * a4.z; z.w += t * a4.w;
      }
      *reinterpret_cast<float4*>(Z + bi * 256 + rr * 16 + c4) = z;
    }
    __syncthreads();
    for (int Lv = 1; Lv < 4; ++Lv) {
      if (tid < (4 - Lv) * 64) {
        const int j = tid >> 6, i = j + Lv, rr = (tid >> 2) & 15, c4 = (tid & 3) * 4;
        float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = j; k < i; ++k) {
          const float* Bik = Z + (i * (i - 1) / 2 + k) * 256 + rr * 16;
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const float bq = Bik[q];
            const float4 t4 = *reinterpret_cast<const float4*>(TS + (16 * k + q) * AP + 16 * j + c4);
            t.x -= bq * t4.x; t.y -= bq * t4.y; t.z -= bq * t4.z; t.w -= bq * t4.w;
          }
        }
        *reinterpret_cast<float4*>(TS + (16 * i + rr) * AP + 16 * j + c4) = t;
      }
      __syncthreads();
    }
    // T -> fp16 tile (upper blocks are zero)
#pragma unroll
    for (int q2 = 0; q2 < 2; ++q2) {
      const int idx = tid + kThreads * q2;
      const int i = idx >> 3, c8 = idx & 7;
      float v8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int j = c8 * 8 + e;
        v8[e] = (j >> 4) <= (i >> 4) ? TS[i * AP + j] : 0.f;
      }
      track_abs(amax, v8, 8);
      tc::sw128_store8<E>(sm + OFF_T, i, c8 * 8, v8);
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
      tc::mma_tile(tmem + TM_UT, sbase + OFF_RU, 0, sbase + OFF_T, 0, 1, tc::idesc_f16_f32(128, 64),
                   false);
      tc::commit(&bar);
    }
    if (!cta_wait(&bar, phase, &flag)) { failed = true; break; }
    phase ^= 1;
    tc::fence_after_sync();
    // ---------------- U^T -> fp16 tile (over R^T, which MMA-D has consumed)
    {
      float ur[32];
      tc::tmem_ld32(tmem + lane + TM_UT + chalf * 32, ur);
      tc::tmem_wait_ld();
      track_abs(amax, ur, 32);
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8)
        tc::sw128_store8<E>(sm + OFF_RU, r128, chalf * 32 + g8 * 8, ur + g8 * 8);
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
      tc::mma_tile(tmem + TM_O2, sbase + OFF_RU, 0, sbase + OFF_P, 0, 1, tc::idesc_f16_f32(128, 64),
                   false);
      tc::mma_tile(tmem + TM_S, sbase + OFF_RU, 0, sbase + OFF_KPT, 0, 1,
                   tc::idesc_f16_f32(128, 128), true);
      tc::commit(&bar);
    }
    if (!cta_wait(&bar, phase, &flag)) { failed = true; break; }
    phase ^= 1;
    tc::fence_after_sync();
    // ---------------- outputs of the chunk, transposed through shared memory
    {
      float oq[32], o2[32];
      tc::tmem_ld32(tmem + lane + TM_OQ + chalf * 32, oq);
      tc::tmem_ld32(tmem + lane + TM_O2 + chalf * 32, o2);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int i = chalf * 32 + e;
        OT[i * D + r128] = __float2bfloat16_rn(EG[i] * oq[e] + o2[e]);
      }
    }
    __syncthreads();
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const int idx = tid + kThreads * q4;
      const int i = idx >> 4, c16 = idx & 15;
      if (i < n)
        *reinterpret_cast<uint4*>(out + ((size_t)(seq0 + c0 + i) * Hv + h) * D + c16 * 8) =
            *reinterpret_cast<const uint4*>(OT + i * D + c16 * 8);
    }
  }
  if (failed) break;
  // an fp16 operand of this chain out of range: the block keeps the old state
  // and the chain is rerun token-serially; else the final state -> the write
  // block, S[v][k] at (h*D + k)*D + v
  if (__syncthreads_or(!(amax <= kF16Max) ? 1 : 0)) {
    if (tid == 0) mark_redo(p.work, chain / Hv, h);
  } else {
    float srow[64];
    tc::tmem_ld32(tmem + lane + TM_S + chalf * 64, srow);
    tc::tmem_ld32(tmem + lane + TM_S + chalf * 64 + 32, srow + 32);
    tc::tmem_wait_ld();
    float* S_w = reinterpret_cast<float*>(wbase + p.rec_off) + (size_t)h * D * D;
#pragma unroll
    for (int k = 0; k < 64; ++k) S_w[(size_t)(chalf * 64 + k) * D + r128] = srow[k];
  }
  amax = 0.f;
  }  // chains
  if (failed && tid == 0) atomicOr((unsigned*)&hdr[kErr], GDN_FLAG_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (tid < 32) tc::tmem_dealloc(tmem, TM_COLS);
}

// New conv states of the length > 1 sequences: the last K-1 inputs of
// [old conv state ; x_seq], written after every chain has read the old one.
// Grid (sequence, channel slice); each thread moves 8 channels of the K-1 rows.
__global__ void __launch_bounds__(256) tail_update_kernel(FwdParams p) {
  pdl_wait_then_release();
  const int n_pre = p.work.header()[kNPre];
  if ((int)blockIdx.x >= n_pre) return;
  const int s = p.work.pre()[blockIdx.x];
  const int seq0 = p.cu[s];
  const int L = p.cu[s + 1] - seq0;
  const int wblk = p.blk[s];
  const int rblk = p.has_past[s] ? wblk : 0;
  const int C = p.C;
  const int ch = (blockIdx.y * blockDim.x + threadIdx.x) * 8;
  if (ch >= C) return;
  const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(p.x);
  const __nv_bfloat16* tail_r =
      reinterpret_cast<const __nv_bfloat16*>(p.layer_base + (size_t)rblk * p.stride);
  __nv_bfloat16* tail_w = reinterpret_cast<__nv_bfloat16*>(p.layer_base + (size_t)wblk * p.stride);
  uint4 nv[KC - 1];
#pragma unroll
  for (int j = 0; j < KC - 1; ++j) {
    const int pp = L - (KC - 1) + j;
    nv[j] = *reinterpret_cast<const uint4*>(pp >= 0 ? x + (size_t)(seq0 + pp) * C + ch
                                                    : tail_r + (size_t)(KC - 1 + pp) * C + ch);
  }
#pragma unroll
  for (int j = 0; j < KC - 1; ++j) *reinterpret_cast<uint4*>(tail_w + (size_t)j * C + ch) = nv[j];
}

}  // namespace

bool chunk_supported(int d, int act, int K) { return d == D && act == GDN_BF16 && K == KC; }

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return nullptr;
    encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return encode;
}

// Tensor map of a row-major 16-bit [rows][cols] array read in boxes of
// 64 columns x box_rows rows, 128-byte swizzled, zero fill outside.
cudaError_t make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int rows, int cols,
                     int box_rows) {
  EncodeTiledFn encode = encoder();
  if (!encode) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_chunk(const FwdParams& p, int max_pre, cudaStream_t stream, int max_dec) {
  if (max_pre <= 0) return cudaSuccess;
  const bool fused = p.scr_qk == nullptr;
  cudaError_t e = cudaSuccess;
  if (fused) {
    e = cudaFuncSetAttribute(chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  static int num_sms = 0;
  if (num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (num_sms <= 0) num_sms = 1;
  }
  const long long chains = (long long)max_pre * p.Hv;
  const int grid = (int)(chains < num_sms ? chains : num_sms);
  if (fused) {
    CUtensorMap tmx;
    e = make_map(&tmx, p.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.T, p.C, XROWS);
    if (e != cudaSuccess) return e;
    e = launch_pdl(chunk_kernel, dim3(grid), dim3(kThreads), SMEM_BYTES, stream, p, tmx);
    if (e != cudaSuccess) return e;
  } else {
    // split: conv, gates and the state-independent products of every chunk
    // (cintra_kernel), then the recurrence over the chains (seq_kernel); at
    // most T/64 + (number of prefill sequences) chunks
    const int max_chunks = p.T / CH + max_pre;
    CUtensorMap tmx;
    e = make_map(&tmx, p.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.T, p.C, XROWS);
    if (e != cudaSuccess) return e;
    e = launch_cintra(p, &tmx, max_chunks, false, num_sms, stream);
    if (e == cudaSuccess) e = launch_seq(p, grid, false, stream);
    if (e != cudaSuccess) return e;
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the batch's decodes, on the SMs the recurrence's last chains leave idle
  if (max_dec > 0 && (e = launch_decode(p, max_dec, stream, true)) != cudaSuccess) return e;
  // chains whose fp16 operands left their range, token-serially, before the
  // conv states change
  e = launch_redo(p, D, GDN_BF16, max_pre, stream);
  if (e != cudaSuccess) return e;
  return launch_pdl(tail_update_kernel, dim3(max_pre, (p.C / 8 + 255) / 256), dim3(256), 0, stream, p);
}

cudaError_t launch_kda_chunk(const FwdParams& p, int max_pre, cudaStream_t stream, int max_dec) {
  if (max_pre <= 0) return cudaSuccess;
  if (!p.scr_qk || !p.scr_v || !p.scr_qh) return cudaErrorInvalidValue;
  static int num_sms = 0;
  if (num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (num_sms <= 0) num_sms = 1;
  }
  const long long chains = (long long)max_pre * p.Hv;
  const int grid = (int)(chains < num_sms ? chains : num_sms);
  // at most T/64 + (number of prefill sequences) chunks: the conv pass, the
  // per-channel-decay chunk products, the recurrence
  const int max_chunks = p.T / CH + max_pre;
  CUtensorMap tmx;
  cudaError_t e = make_map(&tmx, p.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.T, p.C, XROWS);
  if (e != cudaSuccess) return e;
  e = launch_cintra(p, &tmx, max_chunks, true, num_sms, stream);
  if (e == cudaSuccess) e = launch_kintra(p, max_chunks, num_sms, stream);
  if (e == cudaSuccess) e = launch_seq(p, grid, true, stream);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the batch's decodes, on the SMs the recurrence's last chains leave idle
  if (max_dec > 0 && (e = launch_kda_decode(p, max_dec, stream, true)) != cudaSuccess) return e;
  // chains whose fp16 operands left their range, token-serially, before the
  // conv states change
  e = launch_kda_redo(p, max_pre, stream);
  if (e != cudaSuccess) return e;
  return launch_pdl(tail_update_kernel, dim3(max_pre, (p.C / 8 + 255) / 256), dim3(256), 0, stream, p);
}

}  // namespace gdn

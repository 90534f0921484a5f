// Conv prologue and state-independent chunk products of the prefill path in
// one kernel, fully parallel over the 64-token chunks of the prefill
// sequences: an item per (chunk, k-head), both v-heads of the k-head at once,
// on a persistent grid of two CTAs per SM.
//
// Per chunk (rows past the sequence end count as zero tokens), following
// "Continuous batching for linear attention layers" (a varlen causal
// convolution continues every sequence from its own conv state; the chunked
// kernels take the per-sequence states through cu_seqlens) and the chunk-64 WY
// form of the gated delta rule (Gated Delta Networks, chunkwise form):
//   conv + SiLU over the k-head's q | k channels and its two v-heads' v
//     channels, continued from the conv state on the first chunk; L2 norms of
//     q and k (q also scaled by 1/sqrt(d_k)): q~, k~, v
//   gates of both v-heads: g = -e^{A_log} softplus(a + dt_bias), beta =
//     sigmoid(b), G the inclusive cumulative sum of g inside the chunk
//   X = [q~ ; k~] k~^T                               (tcgen05, once for both heads)
//   per head:  A_ij = beta_i e^{G_i - G_j} (k~_i . k~_j)  (j < i)
//              P_ij = e^{G_i - G_j} (q~_i . k~_j)          (j <= i)
//              T = (I + A)^{-1}     (16 x 16 diagonal blocks by column
//                                    substitution, off-diagonal blocks as
//                                    product chains on mma.sync with a tf32
//                                    head/tail split)
//   [-w_0 ; -w_1] = [-T_0 diag(beta_0 e^{G_0}) ; -T_1 diag(beta_1 e^{G_1})] k~
//   u_h = T_h diag(beta_h) v_h                       (tcgen05)
// and writes to the pool's prefill scratch, chunk-major (by the scheduler's
// chunk index), the tiles the recurrence kernel loads: the [q~ ; k~] tile of
// the k-head, (G, beta) of its two v-heads, and -w, u and P of each v-head.
// Every tile is built in shared memory in the 128-byte-swizzled layout of the
// MMA operand it becomes and leaves with one bulk copy, so no thread stores
// scattered rows.  Rows past the sequence end are zero in every tile.  The
// chunk's first row, valid tokens and sequence come from the scheduler's chunk
// records.
//
// The x rows reach shared memory as 2-D TMA boxes of 64 channels x 67 rows
// (3 halo rows + 64), the conv taps of a box in its padding, in two passes
// through one 36 KiB staging area: q | k first (whose conv writes the
// [q~ ; k~] operand tile, so the X product starts while the v boxes load),
// then the two v-heads (whose conv writes the token-major v tiles the u
// products read as MN-major operands).  v never goes to HBM.
//
// The conv-only instance serves the per-channel-decay rule: it stops after
// the conv and writes the [q~ ; k~] tile and the two v tiles to the scratch
// for kintra_kernel (no gates, no products).
#include <cuda.h>

#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"
#include "gdn_solve.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

using E = __half;
constexpr int D = 128;
constexpr int CH = 64;
constexpr int KC = 4;
constexpr int kThreads = 256;
constexpr int R = 2;  // v-heads per k-head
// the thread that fetches the item counter: a global atomic holds its thread
// for the round trip, so a thread of the warps that sit out the gate
// computation takes it
constexpr int kCtr = 224;
constexpr int XROWS = CH + KC - 1;
constexpr uint32_t XSUB = 9216;  // one staged box: 72 rows x 128 B, 1024-aligned
constexpr uint32_t XBOX_BYTES = 64 * XROWS * 2;
constexpr uint32_t WS_OFF = XBOX_BYTES;  // the box's 64 channels' taps, bf16 [64][4]
constexpr uint32_t WS_BYTES = 64 * KC * 2;
static_assert(WS_OFF + WS_BYTES <= XSUB && WS_OFF % 16 == 0, "taps must fit the box padding");
constexpr int AP = solve::AP;  // pitch (floats) of the fp32 A / T rows
constexpr uint32_t BOX = 8192;         // 64 rows x 128 B
constexpr uint32_t KB_STRIDE = 16384;  // K-blocks of the 128-row [q~ ; k~] tile
constexpr float kF16Max = 65000.f;
constexpr float kLog2e = 1.4426950408889634f;

// Shared memory (offsets from a 1024-byte aligned base):
//   S   staging of 4 x boxes (pass 1: q, q, k, k; pass 2: v0, v0, v1, v1);
//       then A / T of both heads fp32 [2][64][AP]; then the MMA A tiles
//       A_w = [-T_0 diag(beta_0 e^G_0) ; -T_1 ...] and A_u = [T_0 diag(beta_0) ;
//       T_1 ...], fp16 128 rows x 64 K each
//   QK  [q~ ; k~] fp16, 2 K-blocks x 128 rows (K-major for X, the k~ rows read
//       MN-major by the w product); once X is done the q~ rows of K-block h
//       hold head h's B blocks of the solve
//   V   v0 | v1 fp16 token-major: 4 blocks of 64 channels x 64 tokens
//       (MN-major B operands of the u products)
//   gates: G log2 e, beta, -beta e^G of both heads [2][64]
//   WT  the conv taps of each pass, halved (see silu_half2) and converted to
//       fp32, as [box][tap][64 channels] with the 16-byte groups of 4 channels
//       ordered 0, 2, 4, ..., 14, 1, 3, ..., 15, so that a thread's 8
//       channels of one tap are two conflict-free 16-byte loads
//   GIN the next item's gate inputs, staged by cp.async
constexpr uint32_t OFF_S = 0;
constexpr uint32_t OFF_AW = OFF_S;
constexpr uint32_t OFF_AU = OFF_S + 16384;
constexpr uint32_t OFF_QK = 4 * XSUB;
constexpr uint32_t OFF_V = OFF_QK + 2 * KB_STRIDE;
constexpr uint32_t OFF_GH = OFF_V + 4 * BOX;
constexpr uint32_t OFF_GB = OFF_GH + 512;
constexpr uint32_t OFF_GBE = OFF_GB + 512;
constexpr uint32_t WT_TAP = 64 * 4;        // one tap of a box's 64 channels, fp32
constexpr uint32_t OFF_WT = OFF_GBE + 512;  // taps of each pass, fp32 [2 passes][4 boxes][4 taps][64 ch]
// gate inputs of the next item (cp.async): per token the aligned word of a
// and of b holding both v-heads' values, then A_log and dt_bias of both
constexpr uint32_t OFF_GIN = OFF_WT + 2 * 4 * KC * WT_TAP;
constexpr uint32_t GIN_BYTES = 2 * CH * 4 + 16;
constexpr uint32_t SMEM_BYTES = OFF_GIN + GIN_BYTES + 1024;
static_assert(2 * CH * AP * 4 <= 4 * XSUB, "A / T of both heads fit the staging area");
static_assert(solve::kZFloats * 4 <= BOX, "B blocks of one head fit the q~ rows of a K-block");
static_assert(OFF_QK % 1024 == 0 && OFF_V % 1024 == 0, "operand tiles on 1024-byte boundaries");
static_assert(2 * (SMEM_BYTES + 1024) <= 228 * 1024, "two CTAs per SM");
constexpr uint32_t TM_COLS = 256;  // X (64 columns), then [-w] (0..127) and u (128..255)

// hardware base-2 exponential and logarithm (MUFU; lg2(0) = -inf, ex2(-inf) = 0)
__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float r;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Packed fp32 pairs: d = a * b + c on both lanes (one fma.rn.f32x2).
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long mul2p(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float tanh_approx(float x) {
  float r;
  asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ unsigned long long pack2f(float lo, float hi) {
  return (unsigned long long)__float_as_uint(lo) | ((unsigned long long)__float_as_uint(hi) << 32);
}
// SiLU of a packed fp32 pair given h = y / 2 (the conv taps are halved, which
// is exact): y sigmoid(y) = y (1 + tanh(y/2)) / 2 = h + h tanh(h), one MUFU
// operation per value (tanh.approx: absolute error about 2^-11 on tanh, so
// about |y| 2^-12 on the result, the size of the fp16 rounding that follows)
__device__ __forceinline__ unsigned long long silu_half2(unsigned long long h2) {
  const unsigned long long t2 = pack2f(tanh_approx(__uint_as_float((uint32_t)h2)),
                                       tanh_approx(__uint_as_float((uint32_t)(h2 >> 32))));
  return fma2(h2, t2, h2);
}
// bf16 pair (low, high halves of a word) -> packed fp32 pair
__device__ __forceinline__ unsigned long long bf2_to_f2(uint32_t u) {
  return (unsigned long long)(u << 16) | ((unsigned long long)(u & 0xffff0000u) << 32);
}

__device__ __forceinline__ uint4 pack8(const float* v) {
  uint4 w;
  w.x = tc::pack2(v[0], v[1], (E*)nullptr);
  w.y = tc::pack2(v[2], v[3], (E*)nullptr);
  w.z = tc::pack2(v[4], v[5], (E*)nullptr);
  w.w = tc::pack2(v[6], v[7], (E*)nullptr);
  return w;
}

__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, int* flag) {
  if (threadIdx.x == 0) *flag = mbar_wait_bounded(bar, parity) ? 1 : 0;
  __syncthreads();
  return *flag != 0;
}

__device__ __forceinline__ void cp_async4(uint32_t saddr, const void* g) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(saddr), "l"(g) : "memory");
}
// The gate inputs of an item (record rec, k-head kh) into the GIN words, by
// cp.async on warps 4..7 (thread 0 drives the bulk copies and issues none):
// per token the aligned 4-byte word of a and of b that holds the values of
// v-heads 2kh and 2kh + 1 (low and high half; Hv is even), A_log and dt_bias
// of both heads.
__device__ __forceinline__ void stage_gates(const FwdParams& p, int4 rec, int kh, int tid,
                                            uint32_t gin) {
  const int u = tid - 2 * CH, row0 = rec.x, n = rec.y, Hv = p.Hv;
  if (u < 0) return;
  const int i = u & 63;
  if (i < n) {
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(u < CH ? p.a : p.b);
    cp_async4(gin + 4 * u, src + (size_t)(row0 + i) * Hv + kh * R);
  }
  if (u < R) {
    cp_async4(gin + 2 * CH * 4 + 4 * u, p.A_log + kh * R + u);
    cp_async4(gin + 2 * CH * 4 + 8 + 4 * u, p.dt_bias + kh * R + u);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Persistent: CTA blockIdx.x takes the items (chunk, k-head) blockIdx.x,
// + gridDim.x, ... (item = chunk * Hk + k-head; two CTAs per SM).  The next
// item's record and gate inputs are read during the current one, and its
// first x boxes load during the current one's last readout.
template <bool kConvOnly>
__global__ void __launch_bounds__(kThreads, 2)
cintra_kernel(FwdParams p, const __grid_constant__ CUtensorMap tmx) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t xbar1, xbar2, mbar, rbar;
  __shared__ uint32_t tmem_slot;
  // the outcome of a CTA-wide wait; the record wait has its own, as it comes
  // right after the X product's wait with no barrier in between
  __shared__ int flag, rflag;
  __shared__ int s_ni;  // the CTA's next item (a dynamic counter hands them out)
  __shared__ float gtot[R];
  __shared__ int4 s_nx[2];  // the record of the item of each parity (by bulk copy on rbar)
  pdl_wait_then_release();
  int32_t* hdr = p.work.header();
  const int Hk = p.Hk, Hv = p.Hv, C = p.C;
  // items: the scheduler's chunk records (first packed row, valid tokens,
  // chunk index inside its sequence, sequence) times the k-heads
  const int n_items = hdr[kPreChunks] * Hk;
  int item = blockIdx.x;
  if (item >= n_items) return;
  const int4* recs = reinterpret_cast<const int4*>(p.scr_c);
  const __nv_bfloat16* wconv = reinterpret_cast<const __nv_bfloat16*>(p.conv_w);
  const int tid = threadIdx.x;
  const uint32_t sbase = smem_u32(sm);
  float* GH = reinterpret_cast<float*>(sm + OFF_GH);
  float* GB = reinterpret_cast<float*>(sm + OFF_GB);
  float* GBE = reinterpret_cast<float*>(sm + OFF_GBE);

  // global channel of staged box b of pass ps for k-head kh_: q | q | k | k,
  // then v of head 2kh_ (two boxes) and of head 2kh_+1 (two boxes)
  auto gch = [&](int kh_, int ps, int b) {
    return ps == 0 ? (b < 2 ? kh_ * D + b * 64 : Hk * D + kh_ * D + (b - 2) * 64)
                   : 2 * Hk * D + kh_ * R * D + b * 64;
  };
  auto issue_x = [&](int row0_, int kh_, int ps, uint64_t* bar) {
    mbar_arrive_expect_tx(bar, 4u * (XBOX_BYTES + WS_BYTES));
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      tma_load_2d(sm + OFF_S + b * XSUB, &tmx, gch(kh_, ps, b), row0_ - (KC - 1), bar);
      bulk_g2s(sm + OFF_S + b * XSUB + WS_OFF, wconv + (size_t)gch(kh_, ps, b) * KC, WS_BYTES, bar);
    }
  };
  int4 rec = recs[item / Hk];
  // (thread 0) 1 + parity of an x-box or record phase in flight, or 0
  int xpend1 = 0, xpend2 = 0, rpend = 0;
  if (tid == 0) {
    mbar_init(&xbar1, 1);
    mbar_init(&xbar2, 1);
    mbar_init(&mbar, 1);
    mbar_init(&rbar, 1);
    fence_mbar_init();
    s_ni = (int)gridDim.x + atomicAdd(&hdr[kItemHeadC], 1);
    issue_x(rec.x, item % Hk, 0, &xbar1);
    xpend1 = 1;
  }
  if (tid < 32) tc::tmem_alloc(&tmem_slot, TM_COLS);
  if (!kConvOnly) {
    stage_gates(p, rec, item % Hk, tid, sbase + OFF_GIN);
    asm volatile("cp.async.wait_all;" ::: "memory");
  }
  __syncthreads();
  bool ok = true;
  uint32_t par = 0;  // parity of this item's x-box barriers and first product barrier

  for (;;) {
  const int gidx = item / Hk, kh = item % Hk;
  const int row0 = rec.x, n = rec.y, c = rec.z, kpre = rec.w;
  const int next = s_ni;
  int nn = 0;  // (thread kCtr) counter value of the item after next
  if (tid == 0 && next < n_items) {
    mbar_arrive_expect_tx(&rbar, 16);
    bulk_g2s(&s_nx[par ^ 1u], recs + next / Hk, 16, &rbar);
    rpend = 1 + (int)par;
  }
  if (tid == kCtr && next < n_items) nn = atomicAdd(&hdr[kItemHeadC], 1);
  int rblk = 0;  // the conv state is read on chunk 0 only
  if (c == 0) {
    const int s = p.work.pre()[kpre];
    rblk = p.has_past[s] ? p.blk[s] : 0;
  }
  const __nv_bfloat16* tail =
      reinterpret_cast<const __nv_bfloat16*>(p.layer_base + (size_t)rblk * p.stride);

  // ---- gates of the chunk's tokens for both v-heads (threads 0..127, token
  // tid % 64 of head 2kh + tid / 64, from the staged inputs): g, beta and the
  // inclusive cumulative sum G of g inside the chunk; tokens past the end
  // take g = 0 and beta = 0
  float gcum = 0.f, gbeta = 0.f;
  if (!kConvOnly && tid < R * CH) {
    const int hl = tid >> 6, i = tid & 63;
    if (i < n) {
      const uint32_t* gw = reinterpret_cast<const uint32_t*>(sm + OFF_GIN);
      const float* gs = reinterpret_cast<const float*>(sm + OFF_GIN + 2 * CH * 4);
      const uint32_t aw = gw[i] >> (16 * hl), bw = gw[CH + i] >> (16 * hl);
      gcum = -__expf(gs[hl]) * softplus_f32(__uint_as_float(aw << 16) + gs[2 + hl]);
      gbeta = sigmoid_f32(__uint_as_float(bw << 16));
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, gcum, o);
      if ((tid & 31) >= o) gcum += t;
    }
    if ((tid & 63) == 31) gtot[tid >> 6] = gcum;
  }
  // (kConvOnly) the previous item's [q~ ; k~] store has read its source
  // before the conv writes it again
  if (kConvOnly && tid == 0) bulk_wait_read_but_last();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  if (!kConvOnly && tid < R * CH) {
    const int hl = tid >> 6, i = tid & 63;
    if (i >= 32) gcum += gtot[hl];
    GH[hl * CH + i] = gcum * kLog2e;
    GB[hl * CH + i] = gbeta;
    GBE[hl * CH + i] = -gbeta * __expf(gcum);
    // the chunk's gate tile of the k-head: [64 tokens][(G, beta) of both heads]
    reinterpret_cast<float2*>(p.scr_g)[((size_t)gidx * Hk + kh) * (CH * R) + i * R + hl] =
        make_float2(gcum, gbeta);
  }

  const int tq = tid >> 4, g = tid & 15;
  const int i0 = 4 * tq;
  const float inv_sqrt_d = rsqrtf((float)D);
  float vmax = 0.f;   // largest |v| (NaN if any is NaN)
  float amax = 0.f;   // largest |value| entering an fp16 operand or the u / w scratch

  // conv + SiLU of part (0 q, 1 k, 2 v of head 2kh, 3 v of head 2kh+1) for
  // tokens i0 .. i0+3, channels g*8 .. g*8+7 of the part, from the staged
  // boxes of the current pass (the part's channels are boxes (part & 1) * 2
  // and (part & 1) * 2 + 1); q and k L2-normalised over the 16 threads of a
  // token.  Rows past the sequence end are written as zeros.  conv_load reads
  // the 7 staged rows and the taps, conv_finish does the arithmetic and the
  // stores, so that the staging area can be released in between.
  struct ConvIn {
    uint4 xw[4 + KC - 1];
    uint4 wt[KC][2];  // halved taps of channels c..c+3 and c+4..c+7, fp32
  };
  auto conv_load = [&](int part, ConvIn& in) {
    const int lc = (part & 1) * D + g * 8;  // pass-local channel: box lc / 64, column lc % 64
    const unsigned char* box = sm + OFF_S + (lc >> 6) * XSUB;
    // channel group m = (lc % 64) / 8 has its two 4-channel halves at 16-byte
    // positions m and 8 + m of each tap
    const unsigned char* wt = sm + OFF_WT + ((part >> 1) * 4 + (lc >> 6)) * (KC * WT_TAP) +
                              ((lc & 63) >> 3) * 16;
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      in.wt[j][0] = *reinterpret_cast<const uint4*>(wt + j * WT_TAP);
      in.wt[j][1] = *reinterpret_cast<const uint4*>(wt + j * WT_TAP + 128);
    }
#pragma unroll
    for (int rr = 0; rr < 4 + KC - 1; ++rr)
      in.xw[rr] = *reinterpret_cast<const uint4*>(box + tc::sw128_offset(i0 + rr, lc & 63));
  };
  auto conv_finish = [&](int part, const ConvIn& in) {
    unsigned long long acc2[4][4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc2[t][e] = 0ull;
#pragma unroll
    for (int rr = 0; rr < 4 + KC - 1; ++rr) {
      const uint4 xw = in.xw[rr];
      const unsigned long long xv2[4] = {bf2_to_f2(xw.x), bf2_to_f2(xw.y), bf2_to_f2(xw.z),
                                         bf2_to_f2(xw.w)};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int j = rr - t;
        if (j >= 0 && j < KC) {
          const unsigned long long wj[4] = {
              (unsigned long long)in.wt[j][0].x | ((unsigned long long)in.wt[j][0].y << 32),
              (unsigned long long)in.wt[j][0].z | ((unsigned long long)in.wt[j][0].w << 32),
              (unsigned long long)in.wt[j][1].x | ((unsigned long long)in.wt[j][1].y << 32),
              (unsigned long long)in.wt[j][1].z | ((unsigned long long)in.wt[j][1].w << 32)};
#pragma unroll
          for (int e = 0; e < 4; ++e) acc2[t][e] = fma2(wj[e], xv2[e], acc2[t][e]);
        }
      }
    }
    float y[4][8];
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const unsigned long long s2 = silu_half2(acc2[t][e]);
        y[t][2 * e] = __uint_as_float((uint32_t)s2);
        y[t][2 * e + 1] = __uint_as_float((uint32_t)(s2 >> 32));
      }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int i = i0 + t;
      if (part < 2) {
        unsigned long long ss2 = 0ull;
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const unsigned long long y2 = pack2f(y[t][e], y[t][e + 1]);
          ss2 = fma2(y2, y2, ss2);
        }
        float ss = __uint_as_float((uint32_t)ss2) + __uint_as_float((uint32_t)(ss2 >> 32));
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float sc = rsqrtf(ss + kL2Eps) * (part == 0 ? inv_sqrt_d : 1.f);
        const unsigned long long sc2 = pack2f(sc, sc);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const unsigned long long r2 = mul2p(pack2f(y[t][e], y[t][e + 1]), sc2);
          y[t][e] = __uint_as_float((uint32_t)r2);
          y[t][e + 1] = __uint_as_float((uint32_t)(r2 >> 32));
        }
      } else if (i < n) {
#pragma unroll
        for (int e = 0; e < 8; e += 2) vmax = max_abs3_nan(vmax, y[t][e], y[t][e + 1]);
      }
      const uint4 wv = i < n ? pack8(y[t]) : make_uint4(0, 0, 0, 0);
      if (part < 2) {
        // [q~ ; k~] tile: row i (q~) or 64 + i (k~), K-block g / 8
        *reinterpret_cast<uint4*>(sm + OFF_QK + (g >> 3) * KB_STRIDE +
                                  tc::sw128_offset(part * CH + i, (g & 7) * 8)) = wv;
      } else {
        // v tile of head part - 2: token row i, channel block g / 8
        *reinterpret_cast<uint4*>(sm + OFF_V + (2 * (part - 2) + (g >> 3)) * BOX +
                                  tc::sw128_offset(i, (g & 7) * 8)) = wv;
      }
    }
  };
  // after a pass's boxes land: the halo rows of a sequence's first chunk are
  // its conv state (rows 0..2 of the 4 boxes), and the taps (bf16 [64][4] in
  // each box's padding) are transposed to [tap][64 channels] (thread = one
  // channel of one box)
  auto pass_setup = [&](int ps) {
    if (c == 0) {
      for (int t = tid; t < (KC - 1) * 4 * 8; t += kThreads) {
        const int r = t >> 5, b = (t >> 3) & 3, cc = (t & 7) * 8;
        *reinterpret_cast<uint4*>(sm + OFF_S + b * XSUB + tc::sw128_offset(r, cc)) =
            *reinterpret_cast<const uint4*>(tail + (size_t)r * C + gch(kh, ps, b) + cc);
      }
    }
    {
      // thread = channel ch of box b: its 4 taps, halved, to the fp32 tap
      // rows; 4-channel group q = ch / 4 sits at 16-byte position
      // q / 2 + 8 (q % 2)
      const int b = tid >> 6, ch = tid & 63;
      const uint2 w4 = *reinterpret_cast<const uint2*>(sm + OFF_S + b * XSUB + WS_OFF + ch * KC * 2);
      const int q = ch >> 2;
      float* wt = reinterpret_cast<float*>(sm + OFF_WT + (ps * 4 + b) * (KC * WT_TAP) +
                                           ((q >> 1) + 8 * (q & 1)) * 16) + (ch & 3);
      const uint32_t u[2] = {w4.x, w4.y};
#pragma unroll
      for (int j = 0; j < KC; ++j) {
        const uint32_t bits = (j & 1) ? (u[j >> 1] & 0xffff0000u) : (u[j >> 1] << 16);
        wt[j * (WT_TAP / 4)] = 0.5f * __uint_as_float(bits);
      }
    }
    __syncthreads();
  };

  ok = cta_wait(&xbar1, par, &flag);
  if (ok && tid == 0) xpend1 = 0;
  if (ok) {
    pass_setup(0);
    {
      ConvIn in;
      conv_load(0, in);
      conv_finish(0, in);
      conv_load(1, in);
      // every read of the staged q | k boxes is done and the halo writes are
      // visible to the async proxy: the v boxes come in while k is finished
      tc::fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        issue_x(row0, kh, 1, &xbar2);
        xpend2 = 1 + (int)par;
      }
      conv_finish(1, in);
    }
    // the [q~ ; k~] operand tile is complete: X product
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      if constexpr (!kConvOnly) {
        tc::fence_after_sync();
        tc::mma_tile(tmem, sbase + OFF_QK, KB_STRIDE, sbase + OFF_QK + CH * 128, KB_STRIDE, 2,
                     tc::idesc_f16_f32(128, 64), false);
        tc::commit(&mbar);
      }
      // the [q~ ; k~] tile to the scratch, as the recurrence kernel loads it
      bulk_s2g(static_cast<unsigned char*>(p.scr_qk) + ((size_t)gidx * Hk + kh) * (2 * KB_STRIDE),
               sm + OFF_QK, 2 * KB_STRIDE);
      bulk_commit();
    }
    ok = cta_wait(&xbar2, par, &flag);
    if (ok && tid == 0) xpend2 = 0;
  }
  if (ok) {
    // the previous item's last tile store (its u_1 or v tiles) has read the
    // v area before the conv writes it
    if (tid == 0) bulk_wait_read_but_last();
    pass_setup(1);
    {
      ConvIn in;
      conv_load(2, in);
      conv_finish(2, in);
      conv_load(3, in);
      conv_finish(3, in);
    }
    tc::fence_proxy_async_smem();  // the v tiles, read by the u products (or stored)
    if constexpr (kConvOnly) {
      // the conv-only pass ends here: the two v-heads' v tiles to the scratch
      // (and the next item's record has landed)
      if (next < n_items) {
        ok = cta_wait(&rbar, par, &rflag);
        if (ok && tid == 0) rpend = 0;
      } else {
        __syncthreads();
      }
      if (ok && tid == 0) {
        bulk_s2g(static_cast<unsigned char*>(p.scr_v) + ((size_t)gidx * Hv + kh * R) * (2 * BOX),
                 sm + OFF_V, 4 * BOX);
        bulk_commit();
        // every read of the staged v boxes is done: the next item's q | k boxes
        if (next < n_items) {
          issue_x(s_nx[par ^ 1u].x, next % Hk, 0, &xbar1);
          xpend1 = 1 + (int)(par ^ 1u);
        }
      }
    } else {
      // the q~ rows take the P tiles next: the [q~ ; k~] store has read them
      if (tid == 0) bulk_wait_read_all();
      ok = cta_wait(&mbar, par, &flag);  // X done; every read of the staging area done
      // the next item's record has landed (its bulk copy on rbar, issued at
      // this item's start): stage its gate inputs (this item's were read
      // before the first barrier)
      if (ok && next < n_items) {
        ok = cta_wait(&rbar, par, &rflag);
        if (ok && tid == 0) rpend = 0;
        if (ok) stage_gates(p, s_nx[par ^ 1u], next % Hk, tid, sbase + OFF_GIN);
      }
    }
  }
  if constexpr (!kConvOnly) {
  float* AT = reinterpret_cast<float*>(sm + OFF_S);  // [2][64][AP]
  const uint32_t lane = (uint32_t)(tid & 96) << 16;  // TMEM lane quarter of this warp
  const int r128 = tid & 127;                        // TMEM row of this thread
  const int hf = tid >> 7;                           // column half of this thread
  if (ok) {
    tc::fence_after_sync();
    // this thread's row of X (q~_i . k~_j for rows < 64, k~_i . k~_j above),
    // 32 columns j = 32 hf .. 32 hf + 31; both heads' rows of P or A from it
    float xr[32];
    tc::tmem_ld32(tmem + lane + hf * 32, xr);
    tc::tmem_wait_ld();
    const bool prow = r128 < CH;
    const int i = r128 & 63, ib = i >> 4;
    const int lim = prow ? i : i - 1;  // last kept column
#pragma unroll
    for (int hl = 0; hl < R; ++hl) {
      // e^{G_i - G_j} beta_i = 2^{(G_i + lg beta_i) - G_j} in log2 units (beta = 0 gives 0)
      const float* gh = GH + hl * CH;
      const float Gi2 = gh[i] + (prow ? 0.f : lg2_approx(GB[hl * CH + i]));
      float val[32];
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const int jb = 2 * hf + blk;
        if (jb <= ib) {
          // val_j = X_ij 2^{Gi2 - G_j log2 e}, two columns per packed step
          const unsigned long long gi2 = pack2f(Gi2, Gi2);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 t = *reinterpret_cast<const float4*>(gh + 16 * jb + 4 * q);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const unsigned long long d2 =
                  fma2(pack2f(hh ? t.z : t.x, hh ? t.w : t.y), pack2f(-1.f, -1.f), gi2);
              const unsigned long long e2 = pack2f(ex2_approx(__uint_as_float((uint32_t)d2)),
                                                   ex2_approx(__uint_as_float((uint32_t)(d2 >> 32))));
              const int e = blk * 16 + 4 * q + 2 * hh;
              const unsigned long long v2 = mul2p(pack2f(xr[e], xr[e + 1]), e2);
              val[e] = __uint_as_float((uint32_t)v2);
              val[e + 1] = __uint_as_float((uint32_t)(v2 >> 32));
            }
          }
          if (jb == ib) {  // the diagonal block: columns past the row's last kept one
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (16 * jb + e > lim) val[blk * 16 + e] = 0.f;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) val[blk * 16 + e] = 0.f;
        }
      }
      if (prow) {
        // |P_ij| <= |q~_i| |k~_j| <= d^{-1/2}: no fp16 range check needed.
        // Head hl's P tile [64 i][64 j] (K-major B operand of the output
        // product) in the q~ rows of K-block hl
        unsigned char* pt = sm + OFF_QK + hl * KB_STRIDE;
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8)
          *reinterpret_cast<uint4*>(pt + tc::sw128_offset(i, (hf * 4 + g8) * 8)) =
              pack8(val + g8 * 8);
      } else {
        // (the solve and the operand tiles read only blocks at or left of the diagonal)
        float* Ar = AT + (hl * CH + i) * AP + hf * 32;
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4)
          if (2 * hf + (j4 >> 2) <= ib)
            *reinterpret_cast<float4*>(Ar + j4 * 4) =
                make_float4(val[j4 * 4], val[j4 * 4 + 1], val[j4 * 4 + 2], val[j4 * 4 + 3]);
      }
    }
    tc::fence_proxy_async_smem();  // the P tiles
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int hl = 0; hl < R; ++hl)
        bulk_s2g(static_cast<unsigned char*>(p.scr_p) + ((size_t)gidx * Hv + kh * R + hl) * BOX,
                 sm + OFF_QK + hl * KB_STRIDE, BOX);
      bulk_commit();
    }
    // ---- T_h = (I + A_h)^{-1}: diagonal 16 x 16 blocks, one column per
    // thread (threads 0..127: head, block, column), written over the A blocks
    {
      float col[16];
      const int hl = tid >> 6, b = (tid >> 4) & 3, m = tid & 15;
      float* Ab = AT + (hl * CH + 16 * b) * AP + 16 * b;
      if (tid < R * CH) solve::diag_col(Ab, m, col);
      __syncthreads();
      if (tid < R * CH) solve::diag_col_store(Ab, m, col);
    }
    // the q~ rows take the B blocks next: the P stores have read them
    if (tid == 0) bulk_wait_read_all();
    __syncthreads();
    // ---- off-diagonal blocks of both heads, a head's six product chains on
    // its four warps (the block barriers are the CTA's)
    {
      const int warp = tid >> 5;
      const int hl = warp >> 2, wl = warp & 3;
      float* ATh = AT + hl * CH * AP;
      float* Z = reinterpret_cast<float*>(sm + OFF_QK + hl * KB_STRIDE);
      solve::offdiag_chains<4>(ATh, Z, wl, [] { __syncthreads(); },
                               [](int, int, const float(&)[4], const float(&)[4]) {});
    }
    __syncthreads();
    // ---- the MMAs' A tiles over the A / T array once every T value is read:
    // row 64 hl + i of A_w = -T_hl[i][:] beta_j e^{G_j}, of A_u = T_hl[i][:] beta_j
    {
      uint4 wtb[R][2], wtbe[R][2];
#pragma unroll
      for (int hl = 0; hl < R; ++hl)
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          const int idx = tid + kThreads * q2;
          const int i = idx >> 3, c8 = idx & 7;
          const bool live = (c8 >> 1) <= (i >> 4);  // an 8-column group at or left of the diagonal
          const float4 b0 = *reinterpret_cast<const float4*>(GB + hl * CH + c8 * 8);
          const float4 b1 = *reinterpret_cast<const float4*>(GB + hl * CH + c8 * 8 + 4);
          const float4 e0 = *reinterpret_cast<const float4*>(GBE + hl * CH + c8 * 8);
          const float4 e1 = *reinterpret_cast<const float4*>(GBE + hl * CH + c8 * 8 + 4);
          const float bj[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
          const float ej[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
          float4 t0 = make_float4(0.f, 0.f, 0.f, 0.f), t1 = t0;
          if (live) {
            t0 = *reinterpret_cast<const float4*>(AT + (hl * CH + i) * AP + c8 * 8);
            t1 = *reinterpret_cast<const float4*>(AT + (hl * CH + i) * AP + c8 * 8 + 4);
          }
          const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
          float tb[8], tbe[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            tb[e] = tv[e] * bj[e];
            tbe[e] = tv[e] * ej[e];
          }
#pragma unroll
          for (int e = 0; e < 8; e += 2) amax = max_abs3(amax, tb[e], tb[e + 1]);
          wtb[hl][q2] = pack8(tb);
          wtbe[hl][q2] = pack8(tbe);
        }
      __syncthreads();
#pragma unroll
      for (int hl = 0; hl < R; ++hl)
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          const int idx = tid + kThreads * q2;
          const int i = idx >> 3, c8 = idx & 7;
          *reinterpret_cast<uint4*>(sm + OFF_AW + tc::sw128_offset(hl * CH + i, c8 * 8)) =
              wtbe[hl][q2];
          *reinterpret_cast<uint4*>(sm + OFF_AU + tc::sw128_offset(hl * CH + i, c8 * 8)) =
              wtb[hl][q2];
        }
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    // [-w_0 ; -w_1] = A_w k~ into columns 0..127 (k~ rows of the [q~ ; k~]
    // tile as an MN-major operand); A_u v_0 into columns 128..255 (rows
    // 0..63 are u_0)
    if (tid == 0) {
      tc::fence_after_sync();
      tc::mma_op(tmem, tc::Opnd{sbase + OFF_AW, 0u, false},
                 tc::Opnd{sbase + OFF_QK + CH * 128, KB_STRIDE, true}, CH / 16,
                 tc::idesc_f16_f32(128, 128, false, true), false);
      tc::mma_op(tmem + 128, tc::Opnd{sbase + OFF_AU, 0u, false},
                 tc::Opnd{sbase + OFF_V, BOX, true}, CH / 16,
                 tc::idesc_f16_f32(128, 128, false, true), false);
      tc::commit(&mbar);
    }
    ok = cta_wait(&mbar, par ^ 1u, &flag);
  }
  // read out 64 columns (col0 .. col0 + 63) of this thread's TMEM row (token
  // r128 % 64) into row r128 % 64 of box hf of a staged 2-box tile (boxes of
  // 64 channels x 64 tokens, the layout the recurrence kernel loads)
  auto readout = [&](uint32_t col0, unsigned char* tile) {
    const int i = r128 & 63;
    unsigned char* box = tile + hf * BOX;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float vv[32];
      tc::tmem_ld32(tmem + lane + col0 + hf * 64 + hh * 32, vv);
      tc::tmem_wait_ld();
      float m4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 32; e += 2)
        m4[(e >> 1) & 3] = max_abs3(m4[(e >> 1) & 3], vv[e], vv[e + 1]);
      amax = fmaxf(amax, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8)
        *reinterpret_cast<uint4*>(box + tc::sw128_offset(i, hh * 32 + g8 * 8)) = pack8(vv + g8 * 8);
    }
  };
  unsigned char* const Wg = static_cast<unsigned char*>(p.scr_w);
  unsigned char* const Ug = static_cast<unsigned char*>(p.scr_u);
  const size_t tile0 = ((size_t)gidx * Hv + kh * R) * (2 * BOX);  // head 2kh's tile
  if (ok) {
    tc::fence_after_sync();
    // -w of head r128 / 64 into the [q~ ; k~] area (free: the w product is
    // done); u_0 (lanes 0..63, warp-uniform) into the A_w tile (free too)
    readout(0, sm + OFF_QK + (r128 >> 6) * (2 * BOX));
    if (r128 < CH) readout(128, sm + OFF_AW);
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      // A_u v_1 into columns 0..127 (rows 64..127 are u_1), and the -w and
      // u_0 tiles to the scratch
      tc::fence_after_sync();
      tc::mma_op(tmem, tc::Opnd{sbase + OFF_AU, 0u, false},
                 tc::Opnd{sbase + OFF_V + 2 * BOX, BOX, true}, CH / 16,
                 tc::idesc_f16_f32(128, 128, false, true), false);
      tc::commit(&mbar);
      bulk_s2g(Wg + tile0, sm + OFF_QK, 4 * BOX);
      bulk_s2g(Ug + tile0, sm + OFF_AW, 2 * BOX);
      bulk_commit();
    }
    ok = cta_wait(&mbar, par, &flag);
    // the products are done and the -w / u_0 stores have read the staging
    // area: the next item's q | k boxes load during this readout
    if (ok && tid == 0 && next < n_items) {
      bulk_wait_read_all();
      issue_x(s_nx[par ^ 1u].x, next % Hk, 0, &xbar1);
      xpend1 = 1 + (int)(par ^ 1u);
    }
    if (ok) {
      // u_1 (lanes 64..127) into the v_0 tile (free: the u_0 product is done)
      tc::fence_after_sync();
      if (r128 >= CH) readout(0, sm + OFF_V);
      tc::fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        bulk_s2g(Ug + tile0 + 2 * BOX, sm + OFF_V, 2 * BOX);
        bulk_commit();
      }
    }
  }
  }  // !kConvOnly
  if (!ok) break;
  // v, w, u and the operand tiles enter tensor-core operands in fp16: a value
  // out of its range sends both v-heads of this sequence to the token-serial
  // redo.  (The next item's staged gate inputs are visible after this barrier.)
  tc::fence_before_sync();
  if (!kConvOnly) asm volatile("cp.async.wait_all;" ::: "memory");
  if (tid == kCtr && next < n_items) s_ni = (int)gridDim.x + nn;  // read after the barrier
  if (__syncthreads_or(!(amax <= kF16Max) || !(vmax <= kF16Max)) && tid == 0) {
    mark_redo(p.work, kpre, kh * R);
    mark_redo(p.work, kpre, kh * R + 1);
  }
  if (next >= n_items) break;
  item = next;
  rec = s_nx[par ^ 1u];
  par ^= 1u;
  }  // items

  if (!ok && tid == 0) {
    atomicOr((unsigned*)&hdr[kErr], GDN_FLAG_TIMEOUT);
    // copies still in flight land before the CTA ends (bounded waits)
    if (xpend1) (void)mbar_wait_bounded(&xbar1, (uint32_t)(xpend1 - 1));
    if (xpend2) (void)mbar_wait_bounded(&xbar2, (uint32_t)(xpend2 - 1));
    if (rpend) (void)mbar_wait_bounded(&rbar, (uint32_t)(rpend - 1));
  }
  tc::fence_before_sync();
  __syncthreads();
  if (tid < 32) tc::tmem_dealloc(tmem_slot, TM_COLS);
  // the shared-memory sources of the tile stores are read before the CTA ends;
  // the stores themselves complete with the grid (the recurrence kernel, launched
  // after it, waits for that)
  if (tid == 0) bulk_wait_read_all();
}

}  // namespace

cudaError_t launch_cintra(const FwdParams& p, const void* x_map, int max_chunks, bool conv_only,
                          int num_sms, cudaStream_t stream) {
  if (max_chunks <= 0) return cudaSuccess;
  auto kern = conv_only ? cintra_kernel<true> : cintra_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // a persistent grid of two CTAs per SM
  const long long items = (long long)max_chunks * p.Hk;
  const int grid = (int)(items < 2LL * num_sms ? items : 2LL * num_sms);
  return launch_pdl(kern, dim3(grid), dim3(kThreads), SMEM_BYTES, stream, p,
                    *static_cast<const CUtensorMap*>(x_map));
}

}  // namespace gdn

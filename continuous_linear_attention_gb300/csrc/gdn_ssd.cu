// Kernels of the Mamba2 mixer's varlen conv + selective scan under continuous
// batching (the groundwork the model support tracker asks for: a varlen scan
// with per-sequence states, next to the varlen causal convolution).  Per head
// h of group g = h / (H/G), per token, with the SSD recurrence of
// "Transformers are SSMs" (scalar A per head):
//   y[c]  = SiLU( sum_j w[c][j] xhat[t-K+1+j][c] )   over the channels x | B | C
//   dt    = softplus(dt_raw + dt_bias[h]),  a = exp(-exp(A_log[h]) dt)
//   h_t   = a h_{t-1} + dt x_t B_t^T   (P x N state, row p = head channel)
//   out_t = h_t C_t + D[h] x_t
//
//  - ssd_recurrent_kernel: token-serial, one CTA per (sequence, head), the
//    head's P x N fp32 state in registers for the whole sequence.  The B and
//    C channels of a group are shared by its H/G heads, so every CTA of the
//    group recomputes their conv (cheap) and none writes the conv state.
//  - ssd_tail_kernel: launched after it, writes each sequence's new conv state
//    (the last K-1 inputs of [old state ; x]) once every read of the old one
//    has completed.
//  - ssd_decode_kernel: one token per request at the production shape (head
//    dim 64, state 128, bf16), HBM bound: every head's 32 KiB state is read
//    once and written once.  Persistent and warp-specialised: a producer warp
//    bulk-copies each head's state several heads ahead (with a unit's first
//    head also the unit's conv inputs) and eight compute warps update it and
//    write it from registers to HBM.  A unit is (request, group): it owns the
//    x channels of the group's heads and the group's B and C channels, so it
//    writes its part of the conv state in place.  A CTA's first unit is its
//    index, the next ones come from a counter.  Longer sequences then run on
//    the token-serial kernel, or, at that shape and when the pool's scratch
//    holds the call's rows, on the chunked scan below.
//  - ssd_prep_kernel + ssd_chunk_kernel: the chunked scan of the prefill
//    sequences on the tensor cores (chunks of 128 tokens, one CTA per
//    (sequence, pair of heads of one group), the pair's two 64 x 128 states
//    stacked as one 128-lane fp32 accumulator in tensor memory).  The chunk
//    form of the SSD recurrence needs no triangular solve: with dt_h and the
//    in-chunk cumulative log decay cum_h,
//      CB  = C B^T,  M_h[t][s] = CB[t][s] e^{cum_h[t] - cum_h[s]} dt_h[s] (s <= t)
//      y_h = M_h X_h + e^{cum_h[t]} (C h_h^T)[t] + D_h x_h
//      h_h <- e^{cum_h[end]} h_h + (X_h e^{cum_h[end] - cum_h} dt_h)^T B
//    (state space duality, "Transformers are SSMs").
#include <cuda.h>

#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int kSsdThreads = 256;

template <int P, int NS, typename Act>
__global__ void __launch_bounds__(kSsdThreads) ssd_recurrent_kernel(SsdParams p, bool long_only) {
  constexpr int NC = kSsdThreads / P;  // threads per state row
  constexpr int NPT = NS / NC;         // state entries per thread
  constexpr int NCH = P + 2 * NS;      // conv channels of one head: x | B | C
  static_assert(NC * P == kSsdThreads && NPT * NC == NS && NPT % 4 == 0, "state split");
  static_assert(NC <= 32 && 32 % NC == 0, "a state row's threads sit in one warp");
  static_assert(NCH <= 2 * kSsdThreads, "at most two conv channels per thread");
  __shared__ float yv[NCH];
  __shared__ float gate[2];
  pdl_wait_then_release();
  const int n_items = p.work.header()[long_only ? kNPre : kNItems];
  if ((int)blockIdx.x >= n_items) return;
  const int s = (long_only ? p.work.pre() : p.work.items())[blockIdx.x];
  const int hd = blockIdx.y;
  const int H = p.H, G = p.G, C = p.C, K = p.K;
  const int g = hd / (H / G);
  const int t0 = p.cu[s];
  const int L = p.cu[s + 1] - t0;
  const int wblk = p.blk[s];
  const int rblk = p.has_past[s] ? wblk : 0;
  const unsigned char* rbase = p.layer_base + (size_t)rblk * p.stride;
  unsigned char* wbase = p.layer_base + (size_t)wblk * p.stride;
  const Act* tail_r = reinterpret_cast<const Act*>(rbase);
  const Act* __restrict__ x = reinterpret_cast<const Act*>(p.xbc);
  const Act* __restrict__ wconv = reinterpret_cast<const Act*>(p.conv_w);
  const Act* __restrict__ dtv = reinterpret_cast<const Act*>(p.dt);
  Act* __restrict__ out = reinterpret_cast<Act*>(p.y);
  const int tid = threadIdx.x;

  // ---- conv channels of this thread (at most 2): local -> global
  int gch[2];
  float win[2][kMaxConvK - 1];
  float wc[2][kMaxConvK];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int lc = tid + c * kSsdThreads;
    gch[c] = -1;
    if (lc < NCH) {
      gch[c] = lc < P ? hd * P + lc
                      : (lc < P + NS ? H * P + g * NS + (lc - P)
                                     : H * P + G * NS + g * NS + (lc - P - NS));
#pragma unroll
      for (int j = 0; j < kMaxConvK - 1; ++j)
        win[c][j] = j < K - 1 ? to_f32(tail_r[(size_t)j * C + gch[c]]) : 0.f;
#pragma unroll
      for (int j = 0; j < kMaxConvK; ++j)
        wc[c][j] = j < K ? to_f32(wconv[(size_t)gch[c] * K + j]) : 0.f;
    }
  }

  // ---- state: row pr (head channel), entries [cc*NPT, (cc+1)*NPT) of the N axis
  const int pr = tid / NC, cc = tid % NC;
  const size_t hoff = ((size_t)hd * P + pr) * NS + (size_t)cc * NPT;
  const float* h_r = reinterpret_cast<const float*>(rbase + p.ssm_off) + hoff;
  float* h_w = reinterpret_cast<float*>(wbase + p.ssm_off) + hoff;
  float hs[NPT];
#pragma unroll
  for (int j = 0; j < NPT; j += 4) {
    const float4 v = *reinterpret_cast<const float4*>(h_r + j);
    hs[j] = v.x; hs[j + 1] = v.y; hs[j + 2] = v.z; hs[j + 3] = v.w;
  }
  const float A = __expf(p.A_log[hd]);
  const float dtb = p.dt_bias[hd];
  const float Dh = p.Dskip[hd];

  for (int t = 0; t < L; ++t) {
    const size_t row = (size_t)(t0 + t);
    // 1. conv + SiLU of the owned channels; time step and decay of the head
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      if (gch[c] < 0) continue;
      const float xv = to_f32(x[row * C + gch[c]]);
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxConvK; ++j) {
        if (j < K - 1) acc += wc[c][j] * win[c][j];
        else if (j == K - 1) acc += wc[c][j] * xv;
      }
#pragma unroll
      for (int j = 0; j < kMaxConvK - 1; ++j) {
        if (j < K - 2) win[c][j] = win[c][j + 1];
        else if (j == K - 2) win[c][j] = xv;
      }
      yv[tid + c * kSsdThreads] = silu_f32(acc);
    }
    if (tid == 0) {
      const float d = softplus_f32(to_f32(dtv[row * H + hd]) + dtb);
      gate[0] = d;
      gate[1] = __expf(-A * d);
    }
    __syncthreads();
    // 2. h <- a h + dt x B^T on this thread's entries; out = h C + D x
    const float xp = yv[pr];
    const float dx = gate[0] * xp;
    const float a = gate[1];
    const float* Bv = yv + P + cc * NPT;
    const float* Cv = yv + P + NS + cc * NPT;
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
      hs[j] = a * hs[j] + dx * Bv[j];
      acc += hs[j] * Cv[j];
    }
#pragma unroll
    for (int o = NC / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (cc == 0) out[(row * H + hd) * P + pr] = from_f32<Act>(acc + Dh * xp);
    // the next token rewrites yv and gate
    __syncthreads();
  }

#pragma unroll
  for (int j = 0; j < NPT; j += 4)
    *reinterpret_cast<float4*>(h_w + j) = make_float4(hs[j], hs[j + 1], hs[j + 2], hs[j + 3]);
}

// New conv state of every active sequence: the last K-1 rows of
// [old state ; x_seq], one thread per channel (all K-1 reads before any write,
// so an in-place shift of a short sequence is safe).
template <typename Act>
__global__ void __launch_bounds__(256) ssd_tail_kernel(SsdParams p, bool long_only) {
  pdl_wait_then_release();
  const int n_items = p.work.header()[long_only ? kNPre : kNItems];
  if ((int)blockIdx.x >= n_items) return;
  const int s = (long_only ? p.work.pre() : p.work.items())[blockIdx.x];
  const int ch = blockIdx.y * blockDim.x + threadIdx.x;
  const int C = p.C, K = p.K;
  if (ch >= C) return;
  const int seq0 = p.cu[s];
  const int L = p.cu[s + 1] - seq0;
  const int wblk = p.blk[s];
  const int rblk = p.has_past[s] ? wblk : 0;
  const Act* x = reinterpret_cast<const Act*>(p.xbc);
  const Act* tail_r = reinterpret_cast<const Act*>(p.layer_base + (size_t)rblk * p.stride);
  Act* tail_w = reinterpret_cast<Act*>(p.layer_base + (size_t)wblk * p.stride);
  Act nv[kMaxConvK - 1];
#pragma unroll
  for (int j = 0; j < kMaxConvK - 1; ++j) {
    if (j >= K - 1) break;
    const int pp = L - (K - 1) + j;
    nv[j] = pp >= 0 ? x[(size_t)(seq0 + pp) * C + ch] : tail_r[(size_t)(K - 1 + pp) * C + ch];
  }
#pragma unroll
  for (int j = 0; j < kMaxConvK - 1; ++j) {
    if (j >= K - 1) break;
    tail_w[(size_t)j * C + ch] = nv[j];
  }
}

// ---------------------------------------------------------------------------
// Decode kernel.

constexpr int DP = 64;                 // head dim
constexpr int DN = 128;                // state size
constexpr int DKC = 4;                 // conv taps
constexpr int kDConsumers = 256;       // 8 compute warps
constexpr int kDThreads = kDConsumers + 32;
constexpr int kDStages = 5;
constexpr int kMaxHpg = 16;            // heads per group
constexpr int kXOff = 0;               // unit-local channel offsets: x | B | C
constexpr int kBOff = kMaxHpg * DP;    // 1024
constexpr int kCOff = kBOff + DN;      // 1152
constexpr int kDUnitCh = kCOff + DN;   // 1280
constexpr uint32_t kDHeadBytes = DP * DN * sizeof(float);
constexpr int kDRows = DP / (kDConsumers / 32);  // state rows per thread (8)

struct SsdConvIn {
  __nv_bfloat16 x[kDUnitCh];
  __nv_bfloat16 tail[DKC - 1][kDUnitCh];
  __nv_bfloat16 w[kDUnitCh][DKC];
  __nv_bfloat16 dt[kMaxHpg];
};

struct SsdDecodeSmem {
  float buf[kDStages][DP * DN];
  SsdConvIn cin[2];
  float y[kDUnitCh];
  float dtv[kMaxHpg];
  float av[kMaxHpg];
  int row[kDStages];
  int wblk[kDStages];
  int unit[kDStages];  // the stage's unit, or -1: no more units
  uint64_t full[kDStages];
  uint64_t empty[kDStages];
  uint64_t cempty[2];
  int ok;
  volatile int issued;  // stages the producer has issued (for the drain on a timeout)
};

static_assert(sizeof(SsdDecodeSmem) <= 227 * 1024, "shared memory of one CTA");
static_assert(sizeof(SsdConvIn) % 16 == 0 && offsetof(SsdConvIn, dt) % 16 == 0 &&
                  offsetof(SsdConvIn, w) % 16 == 0 && (kBOff * 2) % 16 == 0 &&
                  (kCOff * 2) % 16 == 0,
              "bulk-copy destinations on 16-byte boundaries");
static_assert(offsetof(SsdDecodeSmem, cin) % 16 == 0, "conv inputs on 16-byte boundaries");

__device__ __forceinline__ void ssd_consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDConsumers) : "memory");
}

__device__ __forceinline__ void ssd_mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__global__ void __launch_bounds__(kDThreads, 1) ssd_decode_kernel(SsdParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SsdDecodeSmem& sm = *reinterpret_cast<SsdDecodeSmem*>(smem_raw);
  pdl_wait_then_release();
  const int tid = threadIdx.x;
  const int H = p.H, G = p.G, C = p.C;
  const int hpg = H / G;
  int32_t* hdr = p.work.header();
  const int n_units = hdr[kNDec] * G;
  if ((int)blockIdx.x >= n_units) return;

  if (tid == 0) {
    for (int i = 0; i < kDStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], kDConsumers / 32);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&sm.cempty[i], kDConsumers / 32);
    fence_mbar_init();
  }
  __syncthreads();

  if (tid >= kDConsumers) {
    // ======================= producer warp =======================
    if (tid != kDConsumers) return;
    const int* dec = p.work.dec();
    const uint32_t unit_ch = (uint32_t)(hpg * DP + 2 * DN);
    // this CTA's units (request, group): its index, then from a counter the
    // scheduler resets, each claimed when its first stage is issued, so that
    // no CTA ends far behind
    int unit = blockIdx.x;
    sm.issued = 0;
    for (int n = 0;; ++n) {
      const int st = n % kDStages;
      if (n >= kDStages && !mbar_wait_bounded(&sm.empty[st], ((n / kDStages) - 1) & 1)) {
        atomicOr((unsigned*)&hdr[kErr], GDN_FLAG_TIMEOUT);
        return;
      }
      const int k = n / hpg, j = n % hpg;
      if (j == 0 && k > 0) unit = (int)gridDim.x + atomicAdd(&hdr[kDecHead], 1);
      if (unit >= n_units) {
        // no more units: an empty stage tells the compute warps
        sm.unit[st] = -1;
        ssd_mbar_arrive(&sm.full[st]);
        return;
      }
      const int s = dec[unit / G];
      const int g = unit % G;
      const int h = g * hpg + j;
      const int row = p.cu[s];
      const int wblk = p.blk[s];
      const int rblk = p.has_past[s] ? wblk : 0;
      sm.row[st] = row;
      sm.wblk[st] = wblk;
      sm.unit[st] = unit;
      const unsigned char* rbase = p.layer_base + (size_t)rblk * p.stride;
      const float* src = reinterpret_cast<const float*>(rbase + p.ssm_off) + (size_t)h * DP * DN;
      uint32_t bytes = kDHeadBytes;
      SsdConvIn* ci = nullptr;
      if (j == 0) {
        const int cb = k & 1;
        if (k >= 2 && !mbar_wait_bounded(&sm.cempty[cb], ((k >> 1) - 1) & 1)) {
          atomicOr((unsigned*)&p.work.header()[kErr], GDN_FLAG_TIMEOUT);
          return;
        }
        ci = &sm.cin[cb];
        bytes += DKC * unit_ch * 2 + unit_ch * DKC * 2 + (uint32_t)hpg * 2;
      }
      mbar_arrive_expect_tx(&sm.full[st], bytes);
      bulk_g2s(sm.buf[st], src, kDHeadBytes / 2, &sm.full[st]);
      bulk_g2s(sm.buf[st] + DP * DN / 2, src + DP * DN / 2, kDHeadBytes / 2, &sm.full[st]);
      if (ci) {
        const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(p.xbc) + (size_t)row * C;
        const __nv_bfloat16* tail = reinterpret_cast<const __nv_bfloat16*>(rbase);
        const __nv_bfloat16* w = reinterpret_cast<const __nv_bfloat16*>(p.conv_w);
        const int cx = g * hpg * DP, cB = H * DP + g * DN, cC = H * DP + G * DN + g * DN;
        bulk_g2s(ci->x + kXOff, x + cx, hpg * DP * 2, &sm.full[st]);
        bulk_g2s(ci->x + kBOff, x + cB, DN * 2, &sm.full[st]);
        bulk_g2s(ci->x + kCOff, x + cC, DN * 2, &sm.full[st]);
        for (int jj = 0; jj < DKC - 1; ++jj) {
          const __nv_bfloat16* tr = tail + (size_t)jj * C;
          bulk_g2s(ci->tail[jj] + kXOff, tr + cx, hpg * DP * 2, &sm.full[st]);
          bulk_g2s(ci->tail[jj] + kBOff, tr + cB, DN * 2, &sm.full[st]);
          bulk_g2s(ci->tail[jj] + kCOff, tr + cC, DN * 2, &sm.full[st]);
        }
        bulk_g2s(ci->w[kXOff], w + (size_t)cx * DKC, hpg * DP * DKC * 2, &sm.full[st]);
        bulk_g2s(ci->w[kBOff], w + (size_t)cB * DKC, DN * DKC * 2, &sm.full[st]);
        bulk_g2s(ci->w[kCOff], w + (size_t)cC * DKC, DN * DKC * 2, &sm.full[st]);
        bulk_g2s(ci->dt, reinterpret_cast<const __nv_bfloat16*>(p.dt) + (size_t)row * H + g * hpg,
                 hpg * 2, &sm.full[st]);
      }
      sm.issued = n + 1;
    }
  }

  // ======================= compute warps =======================
  __nv_bfloat16* __restrict__ out = reinterpret_cast<__nv_bfloat16*>(p.y);
  const int cv = tid & 31;   // float4 column of the state rows: n = 4 cv .. 4 cv + 3
  const int rg = tid >> 5;   // row group: rows rg + 8 i
  const int lane = tid & 31;

  for (int n = 0;; ++n) {
    const int st = n % kDStages;
    const int k = n / hpg, j = n % hpg;

    if (tid == 0) sm.ok = mbar_wait_bounded(&sm.full[st], (n / kDStages) & 1) ? 1 : 0;
    ssd_consumer_sync();
    if (!sm.ok) {
      if (tid == 0) {
        atomicOr((unsigned*)&hdr[kErr], GDN_FLAG_TIMEOUT);
        // the copies already issued land before the CTA ends
        for (int m = n + 1; m < sm.issued && m < n + kDStages; ++m)
          mbar_wait_bounded(&sm.full[m % kDStages], (m / kDStages) & 1);
      }
      return;
    }
    const int unit = sm.unit[st];
    if (unit < 0) break;
    const int g = unit % G;
    const int h = g * hpg + j;
    const int row = sm.row[st];
    unsigned char* wbase = p.layer_base + (size_t)sm.wblk[st] * p.stride;

    if (j == 0) {
      // ---- conv + SiLU of the unit's channels, their new conv state; time steps
      const SsdConvIn& ci = sm.cin[k & 1];
      __nv_bfloat16* tail_w = reinterpret_cast<__nv_bfloat16*>(wbase);
      for (int lc = tid; lc < kDUnitCh; lc += kDConsumers) {
        if (lc >= hpg * DP && lc < kBOff) continue;  // x slots of absent heads
        const float xv = __bfloat162float(ci.x[lc]);
        float acc = __bfloat162float(ci.w[lc][DKC - 1]) * xv;
#pragma unroll
        for (int jj = 0; jj < DKC - 1; ++jj)
          acc += __bfloat162float(ci.w[lc][jj]) * __bfloat162float(ci.tail[jj][lc]);
        sm.y[lc] = silu_f32(acc);
        const int ch = lc < kBOff ? g * hpg * DP + lc
                                  : (lc < kCOff ? H * DP + g * DN + (lc - kBOff)
                                                : H * DP + G * DN + g * DN + (lc - kCOff));
#pragma unroll
        for (int jj = 0; jj < DKC - 2; ++jj) tail_w[(size_t)jj * C + ch] = ci.tail[jj + 1][lc];
        tail_w[(size_t)(DKC - 2) * C + ch] = ci.x[lc];
      }
      if (tid < hpg) {
        const int hh = g * hpg + tid;
        const float d = softplus_f32(__bfloat162float(ci.dt[tid]) + p.dt_bias[hh]);
        sm.dtv[tid] = d;
        sm.av[tid] = __expf(-__expf(p.A_log[hh]) * d);
      }
      ssd_consumer_sync();
      if (lane == 0) ssd_mbar_arrive(&sm.cempty[k & 1]);
    }

    // ---- h <- a h + dt x B^T for this head, out = h C + D x
    const float* buf = sm.buf[st];
    float4 hv[kDRows];
#pragma unroll
    for (int i = 0; i < kDRows; ++i)
      hv[i] = *reinterpret_cast<const float4*>(buf + (rg + 8 * i) * DN + 4 * cv);
    __syncwarp();
    if (lane == 0) ssd_mbar_arrive(&sm.empty[st]);  // this warp is done with the buffer
    const float d = sm.dtv[j], a = sm.av[j];
    const float Dh = p.Dskip[h];
    const float4 B4 = *reinterpret_cast<const float4*>(&sm.y[kBOff + 4 * cv]);
    const float4 C4 = *reinterpret_cast<const float4*>(&sm.y[kCOff + 4 * cv]);
    float* S_w = reinterpret_cast<float*>(wbase + p.ssm_off) + (size_t)h * DP * DN;
#pragma unroll
    for (int i = 0; i < kDRows; ++i) {
      const int r = rg + 8 * i;
      const float xp = sm.y[j * DP + r];
      const float dx = d * xp;
      float4 s4 = hv[i];
      s4.x = a * s4.x + dx * B4.x;
      s4.y = a * s4.y + dx * B4.y;
      s4.z = a * s4.z + dx * B4.z;
      s4.w = a * s4.w + dx * B4.w;
      float part = s4.x * C4.x + s4.y * C4.y + s4.z * C4.z + s4.w * C4.w;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if (lane == 0) out[((size_t)row * H + h) * DP + r] = __float2bfloat16_rn(part + Dh * xp);
      *reinterpret_cast<float4*>(S_w + (size_t)r * DN + 4 * cv) = s4;
    }
  }
}

int g_ssd_num_sms = 0;

template <int P, int NS, typename Act>
cudaError_t launch_rec_t(const SsdParams& p, int max_items, bool long_only, cudaStream_t stream) {
  cudaError_t e = launch_pdl(ssd_recurrent_kernel<P, NS, Act>, dim3(max_items, p.H),
                             dim3(kSsdThreads), 0, stream, p, long_only);
  if (e != cudaSuccess) return e;
  e = launch_pdl(ssd_tail_kernel<Act>, dim3(max_items, (p.C + 255) / 256), dim3(256), 0, stream,
                 p, long_only);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int P, typename Act>
cudaError_t launch_by_state(const SsdParams& p, int NS, int max_items, bool long_only,
                            cudaStream_t stream) {
  if (NS == 32) return launch_rec_t<P, 32, Act>(p, max_items, long_only, stream);
  if (NS == 64) return launch_rec_t<P, 64, Act>(p, max_items, long_only, stream);
  return launch_rec_t<P, 128, Act>(p, max_items, long_only, stream);
}

// ---------------------------------------------------------------------------
// Chunked scan (prefill).  Per chunk (r0 = first row, n valid tokens), heads
// h0 = 2 hp and h0 + 1 of group g:
//   TMA   X = xs[r0.., h0*64 .. h0*64+127] (2 boxes), B and C of the group
//   CUDA  dt_h, cum_h (inclusive scan over the chunk); rows t >= n of X, B, C
//         zeroed (another sequence's rows or stale scratch)
//   CUDA  hand-over: h (TMEM, lane = (head, p), column = n) -> h16 (fp16
//         K-major B operand), h <- e^{cum_h[n-1]} h
//   CUDA  X'[s][(head,p)] = X dt_h[s] e^{cum_h[n-1] - cum_h[s]}
//   MMA   CB = C B^T, YI = C h16^T, h += X'^T B (X' and B MN-major)
//   CUDA  M_0 and M_1 from one read of CB; MMA Y[:, 64 head ..] = M_h X_h for both
//   CUDA  y = Y + e^{cum_h[t]} YI + D_h x  -> bf16
// fp16 operands, fp32 accumulators and state; |h| is range-checked against
// the fp16 limit (GDN_FLAG_RANGE).  16 warps, one chunk ahead: X and M_0
// swap regions every chunk, so the next chunk's X is loaded as soon as this
// chunk's M products are done (while its outputs are made), the next B and C
// once the state update has read these, and the next chunk's dt / cum are
// scanned while the tensor core runs.

using E = __half;
constexpr int SP = 64;     // head dim
constexpr int SN = 128;    // state size
constexpr int SQ = 128;    // chunk
constexpr int kCThreads = 512;
constexpr uint32_t CBOX = 16384;  // one [128 rows][64 cols] fp16 box, 128-byte swizzled
constexpr uint32_t OFF_X = 0;          // X pair: 2 boxes (head 0, head 1)
constexpr uint32_t OFF_B = 2 * CBOX;    // B: 2 boxes (n 0..63, 64..127)
constexpr uint32_t OFF_C = 4 * CBOX;    // C: 2 boxes
constexpr uint32_t OFF_XP = 6 * CBOX;   // X' (same layout as X)
constexpr uint32_t OFF_H16 = 8 * CBOX;  // h16: [128 rows (head,p)][128 n], 2 K-blocks
constexpr uint32_t OFF_M = 10 * CBOX;   // M_0: [128 t][128 s], 2 K-blocks (M_1 over X')
// X and M_0 alternate between the two regions OFF_X and OFF_M by chunk
// parity, so the next chunk's X can land while this chunk's outputs are made
constexpr uint32_t TILE_BYTES = 12 * CBOX;               // 196608
constexpr uint32_t CSMEM_BYTES = TILE_BYTES + 1024;      // + alignment slack
// (with the kernel's ~4 KiB of static shared memory)
static_assert(CSMEM_BYTES + 8192 <= 227 * 1024, "shared memory of one CTA");
constexpr uint32_t TM_CB = 0, TM_YI = 128, TM_Y = 256, TM_H = 384, TM_COLS = 512;
constexpr float kCF16Max = 65000.f;

// 2^x on the MFU (ex2.approx: relative error about 2^-22; 2^-inf = 0)
__device__ __forceinline__ float ssd_ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ bool ssd_cta_wait(uint64_t* bar, uint32_t parity, int* flag) {
  if (threadIdx.x == 0) *flag = mbar_wait_bounded(bar, parity) ? 1 : 0;
  __syncthreads();
  return *flag != 0;
}

__global__ void __launch_bounds__(kCThreads, 1)
ssd_chunk_kernel(SsdParams p, const __grid_constant__ CUtensorMap txs) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t full_x[2], full_bc, mma_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int okf;
  // [chunk parity][head][token]: dt and the in-chunk cumulative log decay, in
  // log2 units (so every decay factor is one ex2)
  __shared__ __align__(16) float cum[2][2][SQ];
  __shared__ __align__(16) float dts[2][2][SQ];
  __shared__ float wsum[2][SQ / 32];
  pdl_wait_then_release();
  const int tid = threadIdx.x;
  const int H = p.H, G = p.G;
  const int hpg = H / G;
  const int pairs = H / 2;
  const int n_pre = p.work.header()[kNPre];
  if ((int)blockIdx.x >= n_pre * pairs) return;
  const int s = p.work.pre()[blockIdx.x / pairs];
  const int hp = blockIdx.x % pairs;
  const int h0 = 2 * hp;
  const int g = h0 / hpg;
  const int seq0 = p.cu[s];
  const int L = p.cu[s + 1] - seq0;
  const int wblk = p.blk[s];
  const int rblk = p.has_past[s] ? wblk : 0;
  const uint32_t sbase = smem_u32(sm);
  const int nc = (L + SQ - 1) / SQ;

  // loads: X of chunk cc into region xb (OFF_X or OFF_M); B and C of chunk cc
  auto issue_x = [&](int cc, int xb) {
    unsigned char* xt = sm + (xb ? OFF_M : OFF_X);
    mbar_arrive_expect_tx(&full_x[xb], 2 * CBOX);
    tma_load_2d(xt, &txs, h0 * SP, seq0 + cc * SQ, &full_x[xb]);
    tma_load_2d(xt + CBOX, &txs, h0 * SP + SP, seq0 + cc * SQ, &full_x[xb]);
  };
  auto issue_bc = [&](int cc) {
    const int r = seq0 + cc * SQ;
    mbar_arrive_expect_tx(&full_bc, 4 * CBOX);
    tma_load_2d(sm + OFF_B, &txs, H * SP + g * SN, r, &full_bc);
    tma_load_2d(sm + OFF_B + CBOX, &txs, H * SP + g * SN + 64, r, &full_bc);
    tma_load_2d(sm + OFF_C, &txs, H * SP + G * SN + g * SN, r, &full_bc);
    tma_load_2d(sm + OFF_C + CBOX, &txs, H * SP + G * SN + g * SN + 64, r, &full_bc);
  };
  bool x_pending[2] = {false, false}, bc_pending = false;  // (thread 0's record)
  if (tid == 0) {
    mbar_init(&full_x[0], 1);
    mbar_init(&full_x[1], 1);
    mbar_init(&full_bc, 1);
    mbar_init(&mma_bar, 1);
    fence_mbar_init();
    issue_x(0, 0);
    issue_bc(0);
    x_pending[0] = bc_pending = true;
  }
  if (tid < 32) tc::tmem_alloc(&tmem_slot, TM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  // thread = (TMEM lane row = tid % 128 of this warp's lane quarter, column
  // quarter cg = tid / 128): 32 columns of every 128-column accumulator
  const uint32_t lane = (uint32_t)(tid & 96) << 16;
  const int row = tid & 127;                          // TMEM lane: token t or (head, p)
  const int cg = tid >> 7;                            // column quarter
  const int rhead = row >> 6, rp = row & 63;          // (head, p) of a state row
  uint32_t ph_x[2] = {0, 0}, ph_bc = 0, ph_mma = 0;
  bool dead = false;
  float amax = 0.f;
  const float* S_r = reinterpret_cast<const float*>(p.layer_base + (size_t)rblk * p.stride +
                                                    p.ssm_off);
  float* S_w = reinterpret_cast<float*>(p.layer_base + (size_t)wblk * p.stride + p.ssm_off);
  __nv_bfloat16* __restrict__ yout = reinterpret_cast<__nv_bfloat16*>(p.y);
  const __nv_bfloat16* __restrict__ dtr = reinterpret_cast<const __nv_bfloat16*>(p.dt);

  // time steps and in-chunk cumulative log decays of the two heads for chunk
  // cc into parity buffer cb (threads 0..255: head tid / 128, token tid %
  // 128; an inclusive scan by warp shuffles, then the warp prefix); every
  // thread calls it (one barrier inside)
  auto gates = [&](int cc, int cb) {
    const int n = min(SQ, L - cc * SQ);
    const int hh = tid >> 7, t = tid & 127, ln = tid & 31;
    float v = 0.f;
    if (tid < 2 * SQ) {
      const int h = h0 + hh;
      float d = 0.f;
      if (t < n)
        d = softplus_f32(__bfloat162float(dtr[(size_t)(seq0 + cc * SQ + t) * H + h]) + p.dt_bias[h]);
      dts[cb][hh][t] = d;
      v = -__expf(p.A_log[h]) * d * 1.4426950408889634f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, v, o);
        if (ln >= o) v += u;
      }
      if (ln == 31) wsum[hh][t >> 5] = v;
    }
    __syncthreads();
    if (tid < 2 * SQ) {
      float add = 0.f;
      for (int w = 0; w < (t >> 5); ++w) add += wsum[hh][w];
      cum[cb][hh][t] = v + add;
    }
  };

  // ---- initial state into TMEM (row = (head, p), columns n of this quarter;
  // 128 contiguous bytes of the state row, 16-byte loads)
  {
    float hv[32];
    const int n0 = cg * 32;
    const float4* src = reinterpret_cast<const float4*>(S_r + ((size_t)(h0 + rhead) * SP + rp) * SN + n0);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float4 v = rblk != 0 ? src[e] : make_float4(0.f, 0.f, 0.f, 0.f);
      hv[4 * e] = v.x; hv[4 * e + 1] = v.y; hv[4 * e + 2] = v.z; hv[4 * e + 3] = v.w;
    }
    tc::tmem_st32(tmem + lane + TM_H + n0, hv);
    tc::tmem_wait_st();
  }
  gates(0, 0);

  for (int c = 0; c < nc; ++c) {
    const int r0 = seq0 + c * SQ;
    const int n = min(SQ, L - c * SQ);
    const int xb = c & 1;
    const uint32_t OX = xb ? OFF_M : OFF_X;  // this chunk's X; its M_0 goes to the other
    const uint32_t OM = xb ? OFF_X : OFF_M;
    // ---- this chunk's tiles (issued one chunk ahead)
    if (tid == 0) {
      const bool bc_ok = mbar_wait_bounded(&full_bc, ph_bc);
      const bool x_ok = bc_ok && mbar_wait_bounded(&full_x[xb], ph_x[xb]);
      if (bc_ok) bc_pending = false;
      if (x_ok) x_pending[xb] = false;
      okf = x_ok ? 1 : 0;
    }
    __syncthreads();
    if (!okf) { dead = true; break; }
    ph_bc ^= 1;
    ph_x[xb] ^= 1;
    const float* CU = cum[xb][0];
    const float* DT = dts[xb][0];
    // ---- rows t >= n of X, B, C -> 0 (another sequence's rows or stale data)
    if (n < SQ) {
      for (int i = tid; i < (SQ - n) * 8 * 6; i += kCThreads) {
        const int box = i / ((SQ - n) * 8);
        const int rem = i % ((SQ - n) * 8);
        const int r = n + rem / 8, ch = rem % 8;
        const uint32_t base = box < 2 ? OX + box * CBOX : OFF_B + (box - 2) * CBOX;
        *reinterpret_cast<uint4*>(sm + base + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
      }
    }
    // ---- hand-over: h16 <- h (fp16, K-major rows (head,p)), h <- e^{cum[n-1]} h
    {
      const float dc = ssd_ex2(CU[rhead * SQ + n - 1]);
      const int n0 = cg * 32;
      float hv[32];
      tc::tmem_ld32(tmem + lane + TM_H + n0, hv);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; e += 8) {
        amax = fmaxf(amax, max_abs3(max_abs3(hv[e], hv[e + 1], hv[e + 2]),
                                    max_abs3(hv[e + 3], hv[e + 4], hv[e + 5]),
                                    max_abs3(hv[e + 6], hv[e + 7], 0.f)));
        tc::sw128_store8<E>(sm + OFF_H16 + (cg >> 1) * CBOX, row, (cg & 1) * 32 + e, hv + e);
      }
#pragma unroll
      for (int e = 0; e < 32; ++e) hv[e] *= dc;
      tc::tmem_st32(tmem + lane + TM_H + n0, hv);
      tc::tmem_wait_st();
    }
    // ---- X'[s][(head,p)] = X dt e^{cum[n-1] - cum[s]}: thread = token s, one
    // box, one half of its 64 columns
    {
      const int sidx = tid & 127, hh = (tid >> 7) & 1, half = tid >> 8;
      const float f = sidx < n ? DT[hh * SQ + sidx] * ssd_ex2(CU[hh * SQ + n - 1] - CU[hh * SQ + sidx]) : 0.f;
      const unsigned char* xr = sm + OX + hh * CBOX;
      unsigned char* xw = sm + OFF_XP + hh * CBOX;
#pragma unroll
      for (int k0 = 32 * half; k0 < 32 * half + 32; k0 += 8) {
        const uint4 w = *reinterpret_cast<const uint4*>(xr + tc::sw128_offset(sidx, k0));
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
        float v8[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 fl = __half22float2(*reinterpret_cast<const __half2*>(&u[e]));
          v8[2 * e] = fl.x * f;
          v8[2 * e + 1] = fl.y * f;
        }
        tc::sw128_store8<E>(xw, sidx, k0, v8);
      }
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    // ---- CB, YI, state update
    if (tid == 0) {
      tc::fence_after_sync();
      const uint32_t idesc = tc::idesc_f16_f32(128, 128);
      tc::mma_tile(tmem + TM_CB, sbase + OFF_C, CBOX, sbase + OFF_B, CBOX, 2, idesc, false);
      tc::mma_tile(tmem + TM_YI, sbase + OFF_C, CBOX, sbase + OFF_H16, CBOX, 2, idesc, false);
      tc::mma_op(tmem + TM_H, tc::Opnd{sbase + OFF_XP, CBOX, true}, tc::Opnd{sbase + OFF_B, CBOX, true},
                 SQ / 16, tc::idesc_f16_f32(128, 128, true, true), true);
      tc::commit(&mma_bar);
    }
    // while they run: the next chunk's gates into the other parity buffer
    if (c + 1 < nc) gates(c + 1, xb ^ 1);
    if (!ssd_cta_wait(&mma_bar, ph_mma, &okf)) { dead = true; break; }
    ph_mma ^= 1;
    tc::fence_after_sync();
    // B and C are read: the next chunk's come in now
    if (tid == 0 && c + 1 < nc) {
      issue_bc(c + 1);
      bc_pending = true;
    }
    // ---- M_h from CB for both heads (thread: token row t, columns s of this
    // quarter; M_0 to the region X does not use this chunk, M_1 over X', which
    // the state update has read), then Y[:, 64 head ..] = M_h X_h for both
    {
      // a warp's 32 rows t = 32 (warp % 4) + lane against its 32 columns s =
      // 32 cg ..: above the diagonal (cg > warp % 4) the block is zero, below
      // it (cg < warp % 4) every entry is kept (warp-uniform cases)
      const int t = row;
      const int s0 = cg * 32;
      const int rq = (tid >> 5) & 3;
      float cb[32];
      tc::tmem_ld32(tmem + lane + TM_CB + s0, cb);
      tc::tmem_wait_ld();
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float m[32];
        if (cg > rq || t >= n) {
#pragma unroll
          for (int e = 0; e < 32; ++e) m[e] = 0.f;
        } else {
          const float ct = CU[hh * SQ + t];
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 cu4 = *reinterpret_cast<const float4*>(CU + hh * SQ + s0 + e);
            const float4 dt4 = *reinterpret_cast<const float4*>(DT + hh * SQ + s0 + e);
            m[e] = cb[e] * ssd_ex2(ct - cu4.x) * dt4.x;
            m[e + 1] = cb[e + 1] * ssd_ex2(ct - cu4.y) * dt4.y;
            m[e + 2] = cb[e + 2] * ssd_ex2(ct - cu4.z) * dt4.z;
            m[e + 3] = cb[e + 3] * ssd_ex2(ct - cu4.w) * dt4.w;
          }
          if (cg == rq) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (s0 + e > t) m[e] = 0.f;
          }
        }
        unsigned char* mt = sm + (hh ? OFF_XP : OM) + (cg >> 1) * CBOX;
#pragma unroll
        for (int e = 0; e < 32; e += 8) tc::sw128_store8<E>(mt, t, (cg & 1) * 32 + e, m + e);
      }
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      tc::fence_after_sync();
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
        tc::mma_op(tmem + TM_Y + hh * 64, tc::Opnd{sbase + (hh ? OFF_XP : OM), CBOX, false},
                   tc::Opnd{sbase + OX + hh * CBOX, CBOX, true}, SQ / 16,
                   tc::idesc_f16_f32(128, 64, false, true), false);
      tc::commit(&mma_bar);
    }
    if (!ssd_cta_wait(&mma_bar, ph_mma, &okf)) { dead = true; break; }
    ph_mma ^= 1;
    tc::fence_after_sync();
    // M_0 is read: the next chunk's X comes into its region now
    if (tid == 0 && c + 1 < nc) {
      issue_x(c + 1, xb ^ 1);
      x_pending[xb ^ 1] = true;
    }
    // ---- outputs: thread = token t (lane), head cg / 2, columns 32 (cg % 2) ..
    // of y = Y + e^{cum[t]} YI + D x, staged as the chunk's bf16 output rows
    // (token t: the pair's 2 x 64 values, 256 bytes, its 16-byte chunks
    // XOR-rotated by t % 16) over X', which the Y products have read; then
    // written out a whole row per 16 threads
    {
      const int t = row, hh = cg >> 1, q = cg & 1;
      const int h = h0 + hh;
      float yv[32], yi[32];
      const float et = ssd_ex2(CU[hh * SQ + t]);
      const float Dh = p.Dskip[h];
      tc::tmem_ld32(tmem + lane + TM_Y + hh * 64 + q * 32, yv);
      tc::tmem_ld32(tmem + lane + TM_YI + hh * 64 + q * 32, yi);
      tc::tmem_wait_ld();
      uint32_t w[16];
#pragma unroll
      for (int e = 0; e < 32; e += 8) {
        // 8 x values of this row: one 16-byte load
        const uint4 xw = *reinterpret_cast<const uint4*>(
            sm + OX + hh * CBOX + tc::sw128_offset(t, q * 32 + e));
        const uint32_t xu[4] = {xw.x, xw.y, xw.z, xw.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 xf = __half22float2(*reinterpret_cast<const __half2*>(&xu[u]));
          const float o0 = yv[e + 2 * u] + et * yi[e + 2 * u] + Dh * xf.x;
          const float o1 = yv[e + 2 * u + 1] + et * yi[e + 2 * u + 1] + Dh * xf.y;
          w[(e >> 1) + u] = tc::pack2(o0, o1, (__nv_bfloat16*)nullptr);
        }
      }
      unsigned char* orow = sm + OFF_XP + t * 256;
      const int c0 = hh * 8 + q * 4;  // the row's first 16-byte chunk of these 32 values
#pragma unroll
      for (int v4 = 0; v4 < 4; ++v4)
        *reinterpret_cast<uint4*>(orow + (((c0 + v4) ^ (t & 15)) << 4)) =
            make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < SQ * 16 / kCThreads; ++k) {
      const int i = tid + k * kCThreads;
      const int t = i >> 4, ch = i & 15;
      if (t < n) {
        const uint4 v = *reinterpret_cast<const uint4*>(sm + OFF_XP + t * 256 + ((ch ^ (t & 15)) << 4));
        reinterpret_cast<uint4*>(yout + ((size_t)(r0 + t) * H + h0) * SP)[ch] = v;
      }
    }
    tc::fence_proxy_async_smem();  // generic accesses of the tiles before the next TMA writes
    tc::fence_before_sync();
    __syncthreads();  // every read of this chunk's X is done (its region takes M_0 next)
  }

  if (!dead) {
    // ---- final state (row = (head, p), this quarter's columns)
    float hv[32];
    const int n0 = cg * 32;
    tc::tmem_ld32(tmem + lane + TM_H + n0, hv);
    tc::tmem_wait_ld();
    float4* dst = reinterpret_cast<float4*>(S_w + ((size_t)(h0 + rhead) * SP + rp) * SN + n0);
#pragma unroll
    for (int e = 0; e < 8; ++e)
      dst[e] = make_float4(hv[4 * e], hv[4 * e + 1], hv[4 * e + 2], hv[4 * e + 3]);
  } else if (tid == 0) {
    atomicOr((unsigned*)&p.work.header()[kErr], GDN_FLAG_TIMEOUT);
    // the loads still in flight land before the CTA's shared memory goes
    if (bc_pending) mbar_wait_bounded(&full_bc, ph_bc);
    for (int b = 0; b < 2; ++b)
      if (x_pending[b]) mbar_wait_bounded(&full_x[b], ph_x[b]);
  }
  if (!(amax <= kCF16Max)) atomicOr((unsigned*)&p.work.header()[kErr], GDN_FLAG_RANGE);
  tc::fence_before_sync();
  __syncthreads();
  if (tid < 32) tc::tmem_dealloc(tmem, TM_COLS);
}

// Conv + SiLU of every prefill token into the fp16 scratch xs [T][C], token-
// parallel: one CTA per (64-token prefill chunk of the scheduler's chunk
// prefix, every kPrepSlices-th slice of 256 channels); thread (v, q) takes 8
// channels (one 16-byte vector) of the chunk's tokens 8q .. 8q+7, its K-1
// window read from the sequence's earlier rows or, before its first token,
// from the conv state (block 0, all zeros, for a sequence without a past).
// The chunk lookup (a chain of dependent loads) is paid once per CTA, not
// once per slice; two CTAs per SM, so that one loads while the other
// computes.
//
// SiLU as h + h tanh(h) with h = y/2 (the taps are halved, which is exact):
// y sigmoid(y) = y (1 + tanh(y/2)) / 2, one MUFU operation per value;
// tanh.approx has an absolute error of about 2^-11, so the result is off by
// about |y| 2^-12, the size of the fp16 rounding that follows.
constexpr int kPrepTok = 8;     // tokens per thread
constexpr int kPrepCh = 256;    // channels per slice
constexpr int kPrepCtaY = 5;    // CTAs per chunk (each takes every 5th slice)
__device__ __forceinline__ float tanh_approx_f32(float x) {
  float r;
  asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 t = __bfloat1622float2(h2[e]);
    f[2 * e] = t.x;
    f[2 * e + 1] = t.y;
  }
}

template <int KW>
__global__ void __launch_bounds__(256, 2) ssd_prep_kernel(SsdParams p, __half* __restrict__ xs) {
  static_assert(KW >= 2 && KW <= kMaxConvK, "conv width");
  pdl_wait_then_release();
  const int32_t* hdr = p.work.header();
  const int g = blockIdx.x;
  if (g >= hdr[kPreChunks]) return;
  const int n_pre = hdr[kNPre];
  const int32_t* pre_cp = p.work.pre_cp();
  int lo = 0, hi = n_pre - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre_cp[mid] <= g) lo = mid; else hi = mid - 1;
  }
  const int s = p.work.pre()[lo];
  const int c = g - pre_cp[lo];
  const int C = p.C;
  const int seq0 = p.cu[s];
  const int L = p.cu[s + 1] - seq0;
  const int t0 = 64 * c + kPrepTok * (threadIdx.x >> 5);  // first token, sequence-local
  const int t1 = min(t0 + kPrepTok, L);
  if (t0 >= t1) return;
  const int rblk = p.has_past[s] ? p.blk[s] : 0;
  const __nv_bfloat16* __restrict__ tail =
      reinterpret_cast<const __nv_bfloat16*>(p.layer_base + (size_t)rblk * p.stride);
  const __nv_bfloat16* __restrict__ x = reinterpret_cast<const __nv_bfloat16*>(p.xbc);
  const __nv_bfloat16* __restrict__ w = reinterpret_cast<const __nv_bfloat16*>(p.conv_w);
  constexpr int kW = KW - 1;  // window rows
  for (int ch0 = blockIdx.y * kPrepCh + (threadIdx.x & 31) * 8; ch0 < C;
       ch0 += kPrepCtaY * kPrepCh) {
    // rows: the window (oldest first), then the thread's tokens
    uint4 rows[kW + kPrepTok];
#pragma unroll
    for (int j = 0; j < kW; ++j) {
      const int pos = t0 - kW + j;  // sequence-local row
      rows[j] = pos >= 0 ? *reinterpret_cast<const uint4*>(x + (size_t)(seq0 + pos) * C + ch0)
                         : *reinterpret_cast<const uint4*>(tail + (size_t)(kW + pos) * C + ch0);
    }
#pragma unroll
    for (int i = 0; i < kPrepTok; ++i)
      rows[kW + i] = t0 + i < t1
                         ? *reinterpret_cast<const uint4*>(x + (size_t)(seq0 + t0 + i) * C + ch0)
                         : make_uint4(0, 0, 0, 0);
    // the 8 channels' taps, [channel][tap] contiguous: KW 16-byte vectors
    uint4 wraw[KW];
#pragma unroll
    for (int j = 0; j < KW; ++j) wraw[j] = reinterpret_cast<const uint4*>(w + (size_t)ch0 * KW)[j];
    const __nv_bfloat16* wv = reinterpret_cast<const __nv_bfloat16*>(wraw);
    // wh[m][e] = half the tap of channel e on the input m rows before the
    // current one (tap KW-1 is on the current token)
    float wh[KW][8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
#pragma unroll
      for (int m = 0; m < KW; ++m) wh[m][e] = 0.5f * __bfloat162float(wv[e * KW + (KW - 1 - m)]);
#pragma unroll
    for (int i = 0; i < kPrepTok; ++i) {
      float h[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) h[e] = 0.f;
#pragma unroll
      for (int m = 0; m < KW; ++m) {
        float f[8];
        bf16x8_to_f32(rows[kW + i - m], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) h[e] = fmaf(wh[m][e], f[e], h[e]);
      }
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const float a0 = fmaf(h[e], tanh_approx_f32(h[e]), h[e]);
        const float a1 = fmaf(h[e + 1], tanh_approx_f32(h[e + 1]), h[e + 1]);
        const __half2 hv = __floats2half2_rn(a0, a1);
        o[e / 2] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      if (t0 + i < t1)
        *reinterpret_cast<uint4*>(xs + (size_t)(seq0 + t0 + i) * C + ch0) =
            make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

typedef CUresult (*SsdEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Tensor map of the fp16 scratch [rows][cols] in boxes of 64 columns x 128
// rows, 128-byte swizzled, zero fill outside.
cudaError_t ssd_scratch_map(CUtensorMap* m, const void* base, int rows, int cols) {
  static SsdEncodeFn encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<SsdEncodeFn>(fn);
  }
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
}  // namespace

bool ssd_decode_supported(int H, int P, int NS, int G, int K, int act) {
  const int hpg = H / G;
  return P == DP && NS == DN && K == DKC && act == GDN_BF16 && hpg <= kMaxHpg && hpg % 8 == 0;
}

cudaError_t launch_ssd_decode(const SsdParams& p, int max_dec, cudaStream_t stream) {
  if (max_dec <= 0) return cudaSuccess;
  if (g_ssd_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_ssd_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_ssd_num_sms <= 0) g_ssd_num_sms = 1;
  }
  const long long max_units = (long long)max_dec * p.G;
  const int grid = (int)(max_units < g_ssd_num_sms ? max_units : g_ssd_num_sms);
  const size_t smem = sizeof(SsdDecodeSmem);
  cudaError_t e = cudaFuncSetAttribute(ssd_decode_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(ssd_decode_kernel, dim3(grid), dim3(kDThreads), smem, stream, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

bool ssd_supported(int P, int NS) {
  return (P == 32 || P == 64) && (NS == 32 || NS == 64 || NS == 128);
}

cudaError_t launch_ssd(const SsdParams& p, int P, int NS, int act, int max_items,
                       bool long_only, cudaStream_t stream) {
  if (max_items <= 0) return cudaSuccess;
  if (!ssd_supported(P, NS)) return cudaErrorInvalidValue;
  if (act == GDN_F32)
    return P == 32 ? launch_by_state<32, float>(p, NS, max_items, long_only, stream)
                   : launch_by_state<64, float>(p, NS, max_items, long_only, stream);
  return P == 32 ? launch_by_state<32, __nv_bfloat16>(p, NS, max_items, long_only, stream)
                 : launch_by_state<64, __nv_bfloat16>(p, NS, max_items, long_only, stream);
}

bool ssd_chunk_supported(int H, int P, int NS, int K, int act) {
  return P == SP && NS == SN && act == GDN_BF16 && H % 2 == 0 && K <= kMaxConvK;
}

cudaError_t launch_ssd_chunk(const SsdParams& p, void* xs, int max_pre, cudaStream_t stream) {
  if (max_pre <= 0) return cudaSuccess;
  CUtensorMap m;
  cudaError_t e = ssd_scratch_map(&m, xs, p.T, p.C);
  if (e != cudaSuccess) return e;
  // at most T/64 + (prefill sequences) 64-token chunks
  const dim3 pgrid(p.T / 64 + max_pre, kPrepCtaY);
  __half* xh = static_cast<__half*>(xs);
  switch (p.K) {
    case 2: e = launch_pdl(ssd_prep_kernel<2>, pgrid, dim3(256), 0, stream, p, xh); break;
    case 3: e = launch_pdl(ssd_prep_kernel<3>, pgrid, dim3(256), 0, stream, p, xh); break;
    case 4: e = launch_pdl(ssd_prep_kernel<4>, pgrid, dim3(256), 0, stream, p, xh); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(ssd_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)CSMEM_BYTES);
  if (e != cudaSuccess) return e;
  e = launch_pdl(ssd_chunk_kernel, dim3(max_pre * (p.H / 2)), dim3(kCThreads), CSMEM_BYTES,
                 stream, p, m);
  if (e != cudaSuccess) return e;
  e = launch_pdl(ssd_tail_kernel<__nv_bfloat16>, dim3(max_pre, (p.C + 255) / 256), dim3(256), 0,
                 stream, p, true);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace gdn

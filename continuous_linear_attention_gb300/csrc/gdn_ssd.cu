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
//    writes its part of the conv state in place.  Longer sequences then run on
//    the token-serial kernel.
#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"

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
  uint64_t full[kDStages];
  uint64_t empty[kDStages];
  uint64_t cempty[2];
  int ok;
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
  const int n_units = p.work.header()[kNDec] * G;
  const int my_units = n_units > (int)blockIdx.x
                           ? (n_units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int n_stages = my_units * hpg;
  if (n_stages == 0) return;

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
    for (int n = 0; n < n_stages; ++n) {
      const int st = n % kDStages;
      if (n >= kDStages && !mbar_wait_bounded(&sm.empty[st], ((n / kDStages) - 1) & 1)) {
        atomicOr((unsigned*)&p.work.header()[kErr], GDN_FLAG_TIMEOUT);
        return;
      }
      const int k = n / hpg, j = n % hpg;
      const int unit = blockIdx.x + k * gridDim.x;
      const int s = dec[unit / G];
      const int g = unit % G;
      const int h = g * hpg + j;
      const int row = p.cu[s];
      const int wblk = p.blk[s];
      const int rblk = p.has_past[s] ? wblk : 0;
      sm.row[st] = row;
      sm.wblk[st] = wblk;
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
    }
    return;
  }

  // ======================= compute warps =======================
  __nv_bfloat16* __restrict__ out = reinterpret_cast<__nv_bfloat16*>(p.y);
  const int cv = tid & 31;   // float4 column of the state rows: n = 4 cv .. 4 cv + 3
  const int rg = tid >> 5;   // row group: rows rg + 8 i
  const int lane = tid & 31;

  for (int n = 0; n < n_stages; ++n) {
    const int st = n % kDStages;
    const int k = n / hpg, j = n % hpg;
    const int unit = blockIdx.x + k * gridDim.x;
    const int g = unit % G;
    const int h = g * hpg + j;

    if (tid == 0) sm.ok = mbar_wait_bounded(&sm.full[st], (n / kDStages) & 1) ? 1 : 0;
    ssd_consumer_sync();
    if (!sm.ok) {
      if (tid == 0) {
        atomicOr((unsigned*)&p.work.header()[kErr], GDN_FLAG_TIMEOUT);
        for (int m = n + 1; m < n_stages && m < n + kDStages; ++m)
          mbar_wait_bounded(&sm.full[m % kDStages], (m / kDStages) & 1);
      }
      return;
    }
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

}  // namespace gdn

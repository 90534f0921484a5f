// Kernels of the per-channel-decay (KDA) variant of the layer forward: the
// gated delta rule with one decay per key channel (Kimi Linear, the KDA
// recurrence), which the model support tracker lists for the Kimi Linear and
// GLM5-next families.  Same pool, conv, states and scheduler as the scalar
// rule; per token (v-head h, k-head h / (Hv/Hk)) with alpha = e^{g}:
//   g[c]  = -exp(A_log[h]) softplus(a_t[h][c] + dt_bias[h][c]),  beta = sigmoid(b_t[h])
//   S'    = S Diag(alpha)            (key column c of S[v][k] decays by alpha[c])
//   p = S' k, r = S' q,  u = beta (v - p),  o = r + (k.q) u,  S <- S' + u k^T.
// With the state stored k-major (row c = key channel c, v contiguous) the
// decay scales whole rows, so both kernels below keep the data flow of their
// scalar-gate counterparts and fold alpha into the k and q used for the
// reductions and into the row update.
//
//  - kda_decode_kernel: one token per request, HBM bound (each 64 KiB state
//    read once and written once), persistent and warp-specialised exactly
//    like the scalar decode kernel; the unit's gate rows (2 v-heads x d_k)
//    arrive with its conv inputs.
//  - kda_recurrent_kernel: token-serial conv + rule for every other case
//    (longer sequences, other head sizes), state in registers.
#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"

namespace gdn {
namespace {

// ---------------------------------------------------------------------------
// Decode.

constexpr int D = 128;                 // d_k = d_v
constexpr int KC = 4;                  // conv taps
constexpr int kConsumers = 256;        // 8 compute warps
constexpr int kThreads = kConsumers + 32;
constexpr int kStages = 3;
constexpr int kCV = D / 4;             // float4 columns of a state row
constexpr int kG = kConsumers / kCV;   // row groups (8)
constexpr int kRows = D / kG;          // rows per thread (16)
constexpr uint32_t kHeadBytes = D * D * sizeof(float);
constexpr int R = 2;                   // v-heads per k-head
constexpr int kUnitCh = (2 + R) * D;   // conv channels of a unit (512)
constexpr int kMaxHv = 64;

struct KdaConvIn {
  __nv_bfloat16 x[kUnitCh];
  __nv_bfloat16 tail[KC - 1][kUnitCh];
  __nv_bfloat16 w[kUnitCh][KC];
  __nv_bfloat16 a[R][D];  // gate rows of the unit's v-heads
  __nv_bfloat16 b[kMaxHv];
};

struct KdaMeta {
  int row, wblk, pad0, pad1;
};

struct KdaDecodeSmem {
  float buf[kStages][D * D];
  KdaConvIn cin[2];
  float part[2][kG][D];
  float y[kUnitCh];
  float u[D];
  float alpha[R][D];
  float red[4];
  float beta[R];
  KdaMeta meta[kStages];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t cempty[2];
  int ok;
};

static_assert(R * D == kConsumers, "one key-channel decay per compute thread");
static_assert(sizeof(KdaDecodeSmem) <= 227 * 1024, "shared memory of one CTA");
static_assert(offsetof(KdaConvIn, a) % 16 == 0 && sizeof(KdaConvIn) % 16 == 0,
              "bulk-copy destinations on 16-byte boundaries");

__device__ __forceinline__ void kda_consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

__device__ __forceinline__ void kda_mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1) kda_decode_kernel(FwdParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  KdaDecodeSmem& sm = *reinterpret_cast<KdaDecodeSmem*>(smem_raw);
  pdl_wait_then_release();
  const int tid = threadIdx.x;
  const int Hk = p.Hk, Hv = p.Hv, C = p.C;
  const int n_units = p.work.header()[kNDec] * Hk;
  const int my_units = n_units > (int)blockIdx.x
                           ? (n_units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int n_stages = my_units * R;
  if (n_stages == 0) return;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], kConsumers / 32);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&sm.cempty[i], kConsumers / 32);
    fence_mbar_init();
  }
  __syncthreads();

  if (tid >= kConsumers) {
    // ======================= producer warp =======================
    if (tid != kConsumers) return;
    const int* dec = p.work.dec();
    for (int n = 0; n < n_stages; ++n) {
      const int st = n % kStages;
      if (n >= kStages && !mbar_wait_bounded(&sm.empty[st], ((n / kStages) - 1) & 1)) {
        atomicOr((unsigned*)&p.work.header()[kErr], GDN_FLAG_TIMEOUT);
        return;
      }
      const int k = n / R, jh = n % R;
      const int unit = blockIdx.x + k * gridDim.x;
      const int s = dec[unit / Hk];
      const int kh = unit % Hk;
      const int h = kh * R + jh;
      const int row = p.cu[s];
      const int wblk = p.blk[s];
      const int rblk = p.has_past[s] ? wblk : 0;
      sm.meta[st].row = row;
      sm.meta[st].wblk = wblk;
      const unsigned char* rbase = p.layer_base + (size_t)rblk * p.stride;
      const float* src = reinterpret_cast<const float*>(rbase + p.rec_off) + (size_t)h * D * D;
      uint32_t bytes = kHeadBytes;
      KdaConvIn* ci = nullptr;
      if (jh == 0) {
        const int cb = k & 1;
        if (k >= 2 && !mbar_wait_bounded(&sm.cempty[cb], ((k >> 1) - 1) & 1)) {
          atomicOr((unsigned*)&p.work.header()[kErr], GDN_FLAG_TIMEOUT);
          return;
        }
        ci = &sm.cin[cb];
        bytes += (uint32_t)(KC * kUnitCh * 2 + kUnitCh * KC * 2 + R * D * 2 + Hv * 2);
      }
      mbar_arrive_expect_tx(&sm.full[st], bytes);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        bulk_g2s(sm.buf[st] + c * (D * D / 4), src + c * (D * D / 4), kHeadBytes / 4,
                 &sm.full[st]);
      if (ci) {
        const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(p.x) + (size_t)row * C;
        const __nv_bfloat16* tail = reinterpret_cast<const __nv_bfloat16*>(rbase);
        const __nv_bfloat16* w = reinterpret_cast<const __nv_bfloat16*>(p.conv_w);
        const int cq = kh * D, ck = Hk * D + kh * D, cv = 2 * Hk * D + kh * R * D;
        bulk_g2s(ci->x, x + cq, D * 2, &sm.full[st]);
        bulk_g2s(ci->x + D, x + ck, D * 2, &sm.full[st]);
        bulk_g2s(ci->x + 2 * D, x + cv, R * D * 2, &sm.full[st]);
        for (int j = 0; j < KC - 1; ++j) {
          bulk_g2s(ci->tail[j], tail + (size_t)j * C + cq, D * 2, &sm.full[st]);
          bulk_g2s(ci->tail[j] + D, tail + (size_t)j * C + ck, D * 2, &sm.full[st]);
          bulk_g2s(ci->tail[j] + 2 * D, tail + (size_t)j * C + cv, R * D * 2, &sm.full[st]);
        }
        bulk_g2s(ci->w[0], w + (size_t)cq * KC, D * KC * 2, &sm.full[st]);
        bulk_g2s(ci->w[D], w + (size_t)ck * KC, D * KC * 2, &sm.full[st]);
        bulk_g2s(ci->w[2 * D], w + (size_t)cv * KC, R * D * KC * 2, &sm.full[st]);
        // a is [T][Hv][D]: the unit's two v-heads are adjacent rows
        bulk_g2s(ci->a[0],
                 reinterpret_cast<const __nv_bfloat16*>(p.a) + ((size_t)row * Hv + kh * R) * D,
                 R * D * 2, &sm.full[st]);
        bulk_g2s(ci->b, reinterpret_cast<const __nv_bfloat16*>(p.b) + (size_t)row * Hv, Hv * 2,
                 &sm.full[st]);
      }
    }
    return;
  }

  // ======================= compute warps =======================
  __nv_bfloat16* __restrict__ out = reinterpret_cast<__nv_bfloat16*>(p.out);
  const float inv_sqrt_d = rsqrtf((float)D);
  const int cv = tid % kCV;
  const int rg = tid / kCV;
  const int warp = tid >> 5, lane = tid & 31;

  for (int n = 0; n < n_stages; ++n) {
    const int st = n % kStages;
    const int k = n / R, jh = n % R;
    const int unit = blockIdx.x + k * gridDim.x;
    const int kh = unit % Hk;
    const int h = kh * R + jh;

    if (tid == 0) sm.ok = mbar_wait_bounded(&sm.full[st], (n / kStages) & 1) ? 1 : 0;
    kda_consumer_sync();
    if (!sm.ok) {
      if (tid == 0) {
        atomicOr((unsigned*)&p.work.header()[kErr], GDN_FLAG_TIMEOUT);
        for (int m = n + 1; m < n_stages && m < n + kStages; ++m)
          mbar_wait_bounded(&sm.full[m % kStages], (m / kStages) & 1);
      }
      return;
    }
    const int row = sm.meta[st].row;
    const int wblk = sm.meta[st].wblk;
    unsigned char* wbase = p.layer_base + (size_t)wblk * p.stride;

    if (jh == 0) {
      // ---- conv + SiLU of the unit's channels; new conv state; gates
      const KdaConvIn& ci = sm.cin[k & 1];
      __nv_bfloat16* tail_w = reinterpret_cast<__nv_bfloat16*>(wbase);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int lc = tid + c * kConsumers;
        const float xv = __bfloat162float(ci.x[lc]);
        float acc = __bfloat162float(ci.w[lc][KC - 1]) * xv;
#pragma unroll
        for (int j = 0; j < KC - 1; ++j)
          acc += __bfloat162float(ci.w[lc][j]) * __bfloat162float(ci.tail[j][lc]);
        sm.y[lc] = silu_f32(acc);
        const int ch = lc < D ? kh * D + lc
                              : (lc < 2 * D ? Hk * D + kh * D + (lc - D)
                                            : 2 * Hk * D + kh * R * D + (lc - 2 * D));
#pragma unroll
        for (int j = 0; j < KC - 2; ++j) tail_w[(size_t)j * C + ch] = ci.tail[j + 1][lc];
        tail_w[(size_t)(KC - 2) * C + ch] = ci.x[lc];
      }
      {
        // one key-channel decay per thread: R v-heads x D channels = kConsumers
        const int jg = tid / D, c = tid % D;
        const int hh = kh * R + jg;
        const float araw = __bfloat162float(ci.a[jg][c]) + p.dt_bias[(size_t)hh * D + c];
        sm.alpha[jg][c] = __expf(-__expf(p.A_log[hh]) * softplus_f32(araw));
      }
      if (tid < R) sm.beta[tid] = sigmoid_f32(__bfloat162float(ci.b[kh * R + tid]));
      kda_consumer_sync();
      if (lane == 0) kda_mbar_arrive(&sm.cempty[k & 1]);
      if (tid < 96) {
        float acc = 0.f;
        for (int i = lane; i < D; i += 32) {
          const float qv = sm.y[i], kv = sm.y[D + i];
          acc += warp == 0 ? qv * qv : (warp == 1 ? kv * kv : qv * kv);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) sm.red[warp] = acc;
      }
      kda_consumer_sync();
    }
    const float qs = rsqrtf(sm.red[0] + kL2Eps) * inv_sqrt_d;
    const float ks = rsqrtf(sm.red[1] + kL2Eps);
    const float beta = sm.beta[jh];
    const float* buf = sm.buf[st];
    const float* alpha = sm.alpha[jh];

    // ---- pass 1: state rows into registers, partial S' k and S' q
    float4 S[kRows];
    float kr[kRows];
    float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const int r = rg + kG * i;
      S[i] = *reinterpret_cast<const float4*>(buf + r * D + 4 * cv);
      kr[i] = sm.y[D + r] * ks;
      const float al = alpha[r];
      const float ka = al * kr[i];
      const float qa = al * sm.y[r] * qs;
      pk.x += S[i].x * ka; pk.y += S[i].y * ka; pk.z += S[i].z * ka; pk.w += S[i].w * ka;
      pq.x += S[i].x * qa; pq.y += S[i].y * qa; pq.z += S[i].z * qa; pq.w += S[i].w * qa;
    }
    __syncwarp();
    if (lane == 0) kda_mbar_arrive(&sm.empty[st]);
    *reinterpret_cast<float4*>(&sm.part[0][rg][4 * cv]) = pk;
    *reinterpret_cast<float4*>(&sm.part[1][rg][4 * cv]) = pq;
    kda_consumer_sync();
    if (tid < D) {
      float sk = 0.f, sq = 0.f;
#pragma unroll
      for (int g2 = 0; g2 < kG; ++g2) {
        sk += sm.part[0][g2][tid];
        sq += sm.part[1][g2][tid];
      }
      const float vv = sm.y[2 * D + jh * D + tid];
      const float u = beta * (vv - sk);
      sm.u[tid] = u;
      out[((size_t)row * Hv + h) * D + tid] = __float2bfloat16_rn(sq + sm.red[2] * qs * ks * u);
    }
    kda_consumer_sync();
    // ---- pass 2: S <- S Diag(alpha) + u k^T, straight to the write block
    float* S_w = reinterpret_cast<float*>(wbase + p.rec_off) + (size_t)h * D * D;
    const float4 u4 = *reinterpret_cast<const float4*>(&sm.u[4 * cv]);
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const int r = rg + kG * i;
      const float al = alpha[r];
      float4 s4 = S[i];
      s4.x = al * s4.x + u4.x * kr[i];
      s4.y = al * s4.y + u4.y * kr[i];
      s4.z = al * s4.z + u4.z * kr[i];
      s4.w = al * s4.w + u4.w * kr[i];
      *reinterpret_cast<float4*>(S_w + (size_t)r * D + 4 * cv) = s4;
    }
    // the next unit's gate pass rewrites alpha only after its own full-barrier
    // wait and a consumer barrier, which every thread reaches after this loop
  }
}

// ---------------------------------------------------------------------------
// Token-serial kernel.

constexpr int kHeadThreads = 256;  // threads per v-head

// mode: kAll every active sequence, kLong those longer than one token, kRedo
// the v-heads of the prefill list that the chunked prefill marked for a redo
// (outputs and recurrent states of those heads only; the conv state is left
// to the conv-state update)
enum Mode : int { kAll = 0, kLong = 1, kRedo = 2 };

template <int DD, typename Act>
__global__ void __launch_bounds__(2 * kHeadThreads)
kda_recurrent_kernel(FwdParams p, int mode) {
  constexpr int CV = DD / 4;
  constexpr int G = kHeadThreads / CV;
  constexpr int NJ = DD / G;
  static_assert(NJ * G == DD, "row split");
  pdl_wait_then_release();
  const int RR = p.Hv / p.Hk;
  const WorkArea& wk = p.work;
  const bool long_only = mode != kAll;
  const int n_items = wk.header()[long_only ? kNPre : kNItems];
  if ((int)blockIdx.x >= n_items) return;
  const int kh = blockIdx.y;
  // redo: the marked v-heads of this k-head group (bits kh*RR .. kh*RR+RR-1)
  uint32_t marks = (1u << RR) - 1u;
  if (mode == kRedo) {
    const int h0 = kh * RR;
    marks = (reinterpret_cast<const uint32_t*>(wk.redo())[2 * blockIdx.x + (h0 >> 5)] >>
             (h0 & 31)) & ((1u << RR) - 1u);
    if (!marks) return;
  }
  const int s = (long_only ? wk.pre() : wk.items())[blockIdx.x];
  const int t0 = p.cu[s];
  const int L = p.cu[s + 1] - t0;
  const int wblk = p.blk[s];
  const int rblk = p.has_past[s] ? wblk : 0;
  const int C = p.C, K = p.K, Hk = p.Hk, Hv = p.Hv;
  const unsigned char* rbase = p.layer_base + (size_t)rblk * p.stride;
  unsigned char* wbase = p.layer_base + (size_t)wblk * p.stride;
  const Act* tail_r = reinterpret_cast<const Act*>(rbase);
  Act* tail_w = reinterpret_cast<Act*>(wbase);
  const Act* __restrict__ x = reinterpret_cast<const Act*>(p.x);
  const Act* __restrict__ wconv = reinterpret_cast<const Act*>(p.conv_w);
  const Act* __restrict__ av = reinterpret_cast<const Act*>(p.a);
  const Act* __restrict__ bv = reinterpret_cast<const Act*>(p.b);
  Act* __restrict__ out = reinterpret_cast<Act*>(p.out);

  extern __shared__ float smem[];
  const int NCH = (2 + RR) * DD;
  float* y = smem;                      // [4 D] conv + SiLU output of the token
  float* part = y + 4 * DD;             // [2][2][G][D] partial S' k, S' q
  float* uo = part + 2 * 2 * G * DD;    // [2][D] u
  float* al = uo + 2 * DD;              // [2][D] key-channel decays
  float* red = al + 2 * DD;             // [4] sum q^2, sum k^2, q.k
  float* gb = red + 4;                  // [2] beta

  const int tid = threadIdx.x;
  const int nt = blockDim.x;

  int gch[2];
  float win[2][kMaxConvK - 1];
  float wc[2][kMaxConvK];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int lc = tid + c * nt;
    gch[c] = -1;
    if (lc < NCH) {
      if (lc < DD) gch[c] = kh * DD + lc;
      else if (lc < 2 * DD) gch[c] = Hk * DD + kh * DD + (lc - DD);
      else gch[c] = 2 * Hk * DD + kh * RR * DD + (lc - 2 * DD);
#pragma unroll
      for (int j = 0; j < kMaxConvK - 1; ++j)
        win[c][j] = j < K - 1 ? to_f32(tail_r[(size_t)j * C + gch[c]]) : 0.f;
#pragma unroll
      for (int j = 0; j < kMaxConvK; ++j)
        wc[c][j] = j < K ? to_f32(wconv[(size_t)gch[c] * K + j]) : 0.f;
    }
  }

  const int j_head = tid / kHeadThreads;
  const int li = tid % kHeadThreads;
  const int h = kh * RR + j_head;
  const bool mine = (marks >> j_head) & 1u;  // this thread's v-head is written
  const int cv = li % CV;
  const int rg = li / CV;
  const float* S_r = reinterpret_cast<const float*>(rbase + p.rec_off) + (size_t)h * DD * DD;
  float* S_w = reinterpret_cast<float*>(wbase + p.rec_off) + (size_t)h * DD * DD;
  float4 S[NJ];
#pragma unroll
  for (int i = 0; i < NJ; ++i)
    S[i] = *reinterpret_cast<const float4*>(S_r + (size_t)(rg + G * i) * DD + 4 * cv);

  const float inv_sqrt_d = rsqrtf((float)DD);
  for (int t = 0; t < L; ++t) {
    const size_t row = (size_t)(t0 + t);
    // 1. conv + SiLU of the owned channels; decays and beta of the group's v-heads
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
      y[tid + c * nt] = silu_f32(acc);
    }
    if (tid < RR * DD) {
      const int jg = tid / DD, c = tid % DD;
      const int hh = kh * RR + jg;
      const float araw = to_f32(av[(row * Hv + hh) * DD + c]) + p.dt_bias[(size_t)hh * DD + c];
      al[jg * DD + c] = __expf(-__expf(p.A_log[hh]) * softplus_f32(araw));
    }
    if (tid < RR) gb[tid] = sigmoid_f32(to_f32(bv[row * Hv + kh * RR + tid]));
    __syncthreads();
    // 2. sums of squares and q.k (warps 0..2)
    if (tid < 96) {
      const int w = tid >> 5, lane = tid & 31;
      float acc = 0.f;
      for (int i = lane; i < DD; i += 32) {
        const float qv = y[i], kv = y[DD + i];
        acc += w == 0 ? qv * qv : (w == 1 ? kv * kv : qv * kv);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) red[w] = acc;
    }
    __syncthreads();
    const float qs = rsqrtf(red[0] + kL2Eps) * inv_sqrt_d;
    const float ks = rsqrtf(red[1] + kL2Eps);
    const float beta = gb[j_head];
    const float* alh = al + j_head * DD;
    // 3. partial S' k and S' q over this thread's rows (S' = S Diag(alpha))
    float kr[NJ];
    float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
    for (int i = 0; i < NJ; ++i) {
      const int r = rg + G * i;
      kr[i] = y[DD + r] * ks;
      const float ka = alh[r] * kr[i];
      const float qa = alh[r] * y[r] * qs;
      pk.x += S[i].x * ka; pk.y += S[i].y * ka; pk.z += S[i].z * ka; pk.w += S[i].w * ka;
      pq.x += S[i].x * qa; pq.y += S[i].y * qa; pq.z += S[i].z * qa; pq.w += S[i].w * qa;
    }
    float* myp = part + (size_t)j_head * 2 * G * DD;
    *reinterpret_cast<float4*>(myp + (size_t)rg * DD + 4 * cv) = pk;
    *reinterpret_cast<float4*>(myp + (size_t)(G + rg) * DD + 4 * cv) = pq;
    __syncthreads();
    // 4. u and o for each v column
    if (li < DD) {
      float sk = 0.f, sq = 0.f;
      for (int g2 = 0; g2 < G; ++g2) {
        sk += myp[(size_t)g2 * DD + li];
        sq += myp[(size_t)(G + g2) * DD + li];
      }
      const float vv = y[2 * DD + j_head * DD + li];
      const float u = beta * (vv - sk);
      const float kq = red[2] * qs * ks;
      uo[j_head * DD + li] = u;
      if (mine) out[(row * Hv + h) * DD + li] = from_f32<Act>(sq + kq * u);
    }
    __syncthreads();
    // 5. S <- S Diag(alpha) + u k^T
    const float4 u4 = *reinterpret_cast<const float4*>(uo + j_head * DD + 4 * cv);
#pragma unroll
    for (int i = 0; i < NJ; ++i) {
      const float a_r = alh[rg + G * i];
      S[i].x = a_r * S[i].x + u4.x * kr[i];
      S[i].y = a_r * S[i].y + u4.y * kr[i];
      S[i].z = a_r * S[i].z + u4.z * kr[i];
      S[i].w = a_r * S[i].w + u4.w * kr[i];
    }
    // the next token's gate pass overwrites al[] and gb[]: every thread must
    // be done reading them
    __syncthreads();
  }

  if (mine) {
#pragma unroll
    for (int i = 0; i < NJ; ++i)
      *reinterpret_cast<float4*>(S_w + (size_t)(rg + G * i) * DD + 4 * cv) = S[i];
  }
  if (mode == kRedo) return;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    if (gch[c] < 0) continue;
#pragma unroll
    for (int j = 0; j < kMaxConvK - 1; ++j)
      if (j < K - 1) tail_w[(size_t)j * C + gch[c]] = from_f32<Act>(win[c][j]);
  }
}

template <int DD, typename Act>
cudaError_t launch_kda_rec(const FwdParams& p, int max_items, int mode, cudaStream_t stream) {
  const int RR = p.Hv / p.Hk;
  constexpr int G = kHeadThreads / (DD / 4);
  const size_t smem = sizeof(float) * (4 * DD + 2 * 2 * G * DD + 2 * DD + 2 * DD + 4 + 4);
  dim3 grid(max_items, p.Hk);
  const cudaError_t e = launch_pdl(kda_recurrent_kernel<DD, Act>, grid, dim3(RR * kHeadThreads),
                                   smem, stream, p, mode);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

int g_kda_num_sms = 0;

}  // namespace

cudaError_t launch_kda_recurrent(const FwdParams& p, int d, int act, int max_items,
                                 bool long_only, cudaStream_t stream) {
  if (max_items <= 0) return cudaSuccess;
  const int mode = long_only ? kLong : kAll;
  if (act == GDN_F32) {
    if (d == 32) return launch_kda_rec<32, float>(p, max_items, mode, stream);
    if (d == 64) return launch_kda_rec<64, float>(p, max_items, mode, stream);
    return launch_kda_rec<128, float>(p, max_items, mode, stream);
  }
  if (d == 32) return launch_kda_rec<32, __nv_bfloat16>(p, max_items, mode, stream);
  if (d == 64) return launch_kda_rec<64, __nv_bfloat16>(p, max_items, mode, stream);
  return launch_kda_rec<128, __nv_bfloat16>(p, max_items, mode, stream);
}

cudaError_t launch_kda_redo(const FwdParams& p, int max_pre, cudaStream_t stream) {
  if (max_pre <= 0) return cudaSuccess;
  return launch_kda_rec<128, __nv_bfloat16>(p, max_pre, kRedo, stream);
}

cudaError_t launch_kda_decode(const FwdParams& p, int max_dec, cudaStream_t stream) {
  if (max_dec <= 0) return cudaSuccess;
  if (g_kda_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_kda_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_kda_num_sms <= 0) g_kda_num_sms = 1;
  }
  const long long max_units = (long long)max_dec * p.Hk;
  const int grid = (int)(max_units < g_kda_num_sms ? max_units : g_kda_num_sms);
  const size_t smem = sizeof(KdaDecodeSmem);
  cudaError_t e = cudaFuncSetAttribute(kda_decode_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kda_decode_kernel, dim3(grid), dim3(kThreads), smem, stream, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace gdn

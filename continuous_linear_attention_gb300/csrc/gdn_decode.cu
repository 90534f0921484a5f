// Decode kernel: one new token per request (the engine's decode fast path,
// "Continuous batching for linear attention layers").  The step is bound by
// HBM: every v-head's d_k x d_v fp32 state (64 KiB at d = 128) is read once
// and written once, which is ~97% of the bytes of the call.
//
// Design (GB300): a persistent grid of one CTA per SM, warp-specialised.
//  - Work units are (request, k-head group).  A unit owns the q/k conv
//    channels of its k-head and the v channels and states of its v-heads, so
//    reading the old conv/recurrent state and overwriting it in place needs no
//    cross-CTA ordering.  A CTA's first unit is its index, the next ones come
//    from a counter the scheduler resets, so that CTAs which start late (see
//    below) take fewer.
//  - One producer warp streams, kStages heads ahead, each v-head's state
//    (64 KiB) into a ring of shared-memory buffers with bulk (TMA) copies, and
//    with the first head of a unit also that unit's conv inputs (its x row,
//    conv-state rows, conv taps, gate rows).  It resolves the request's block
//    indices itself, so the compute warps never wait on a global load.
//  - Eight compute warps read a state buffer once into registers (releasing
//    it to the producer at once), reduce S k and S q across warps, and write
//    the new state straight from registers to HBM with 16-byte stores.
//  - In a batch that also has prefills it is launched after the prefill's
//    recurrence (p.decode_late): its CTAs start on the SMs the recurrence's
//    last chains leave idle, without waiting for it (no data is shared: other
//    requests, other blocks), and wait for it only before they end, so that
//    the kernels after them still see everything before them complete.
//
// Per token (v-head h, k-head h / (Hv/Hk)), as in the gated delta rule:
//   y = SiLU(conv over [conv state ; x]),  q, k L2-normalised, q /= sqrt(d_k)
//   g = -exp(A_log) softplus(a + dt_bias),  beta = sigmoid(b)
//   p = S k, r = S q,  u = beta (v - e^g p),  o = e^g r + (k.q) u,
//   S <- e^g S + u k^T.
// The per-channel-decay (KDA) instance takes one decay per key channel,
// alpha[c] = e^{-exp(A_log) softplus(a[c] + dt_bias[c])}, and with S' = S
// Diag(alpha): p = S' k, r = S' q, u = beta (v - p), o = r + (k.q) u,
// S <- S' + u k^T; the state is stored k-major (row c = key channel c), so
// the decay scales whole rows, folded into the k and q of the reductions and
// into the row update.  Its unit's gate rows (2 v-heads x d_k bf16) arrive
// with the conv inputs.
#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"

namespace gdn {
namespace {

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

// Conv inputs of one unit, bf16, channel order q | k | v of the unit, and the
// gate pre-activations: the token's row of a (scalar gate) or the unit's two
// v-heads' rows of a (per-channel decay), and the token's row of b.
template <bool kKda> struct GateIn;
template <> struct GateIn<false> {
  __nv_bfloat16 a[kMaxHv];
};
template <> struct GateIn<true> {
  __nv_bfloat16 a[R][D];
};
template <bool kKda>
struct ConvIn {
  __nv_bfloat16 x[kUnitCh];
  __nv_bfloat16 tail[KC - 1][kUnitCh];
  __nv_bfloat16 w[kUnitCh][KC];
  GateIn<kKda> g;
  __nv_bfloat16 b[kMaxHv];
};

// Gates of the unit's two v-heads: (e^g, beta), or the key-channel decays
// and beta.
template <bool kKda> struct Gates;
template <> struct Gates<false> {
  float gate[R][2];
};
template <> struct Gates<true> {
  float alpha[R][D];
  float beta[R];
};

struct Meta {
  int row;   // packed row of the token
  int wblk;  // block written
  int unit;  // the unit, or -1: no more units
  int pad;
};

template <bool kKda>
struct DecodeSmem {
  float buf[kStages][D * D];  // state ring
  ConvIn<kKda> cin[2];        // conv inputs, double-buffered by unit
  float part[2][kG][D];       // partial S k and S q
  float y[kUnitCh];           // conv + SiLU outputs of the unit
  float u[D];
  float red[4];
  Gates<kKda> gt;
  Meta meta[kStages];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t cempty[2];
  int ok;
  volatile int issued;  // stages the producer has issued (for the drain on a timeout)
};

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

static_assert(R * D == kConsumers, "one key-channel decay per compute thread");
static_assert(sizeof(DecodeSmem<false>) <= 227 * 1024 && sizeof(DecodeSmem<true>) <= 227 * 1024,
              "shared memory of one CTA");
static_assert(sizeof(ConvIn<false>) % 16 == 0 && sizeof(ConvIn<true>) % 16 == 0 &&
                  offsetof(ConvIn<true>, g) % 16 == 0 && offsetof(ConvIn<false>, g) % 16 == 0 &&
                  offsetof(ConvIn<false>, b) % 16 == 0 && offsetof(ConvIn<true>, b) % 16 == 0,
              "bulk-copy destinations on 16-byte boundaries");

template <bool kKda>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(FwdParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  DecodeSmem<kKda>& sm = *reinterpret_cast<DecodeSmem<kKda>*>(smem_raw);
  const bool late = p.decode_late != 0;
  if (late)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  else
    pdl_wait_then_release();
  const int tid = threadIdx.x;
  const int Hk = p.Hk, Hv = p.Hv, C = p.C;
  int32_t* hdr = p.work.header();
  const int n_units = hdr[kNDec] * Hk;
  if ((int)blockIdx.x >= n_units) {
    if (late && tid == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
    return;
  }

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
    // this CTA's units: its index, then from the counter, each claimed when
    // its first stage is issued (the ring's lead covers the atomic's round
    // trip; a unit claimed a whole unit ahead left CTAs up to two units apart
    // at the end)
    int unit = blockIdx.x;
    sm.issued = 0;
    for (int n = 0;; ++n) {
      const int st = n % kStages;
      if (n >= kStages && !mbar_wait_bounded(&sm.empty[st], ((n / kStages) - 1) & 1)) {
        atomicOr((unsigned*)&hdr[kErr], GDN_FLAG_TIMEOUT);
        return;
      }
      const int k = n / R, jh = n % R;
      if (jh == 0 && k > 0) unit = (int)gridDim.x + atomicAdd(&hdr[kDecHead], 1);
      if (unit >= n_units) {
        // no more units: an empty stage tells the compute warps
        sm.meta[st].unit = -1;
        mbar_arrive(&sm.full[st]);
        return;
      }
      const int s = dec[unit / Hk];
      const int kh = unit % Hk;
      const int h = kh * R + jh;
      const int row = p.cu[s];
      const int wblk = p.blk[s];
      const int rblk = p.has_past[s] ? wblk : 0;
      sm.meta[st].row = row;
      sm.meta[st].wblk = wblk;
      sm.meta[st].unit = unit;
      const unsigned char* rbase = p.layer_base + (size_t)rblk * p.stride;
      const float* src = reinterpret_cast<const float*>(rbase + p.rec_off) + (size_t)h * D * D;
      uint32_t bytes = kHeadBytes;
      ConvIn<kKda>* ci = nullptr;
      if (jh == 0) {
        const int cb = k & 1;
        if (k >= 2 && !mbar_wait_bounded(&sm.cempty[cb], ((k >> 1) - 1) & 1)) {
          atomicOr((unsigned*)&p.work.header()[kErr], GDN_FLAG_TIMEOUT);
          return;
        }
        ci = &sm.cin[cb];
        bytes += (uint32_t)(KC * kUnitCh * 2 + kUnitCh * KC * 2 + (kKda ? R * D * 2 : Hv * 2) +
                            Hv * 2);
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
        if constexpr (kKda) {
          // a is [T][Hv][D]: the unit's two v-heads are adjacent rows
          bulk_g2s(ci->g.a[0],
                   reinterpret_cast<const __nv_bfloat16*>(p.a) + ((size_t)row * Hv + kh * R) * D,
                   R * D * 2, &sm.full[st]);
        } else {
          bulk_g2s(ci->g.a, reinterpret_cast<const __nv_bfloat16*>(p.a) + (size_t)row * Hv,
                   Hv * 2, &sm.full[st]);
        }
        bulk_g2s(ci->b, reinterpret_cast<const __nv_bfloat16*>(p.b) + (size_t)row * Hv, Hv * 2,
                 &sm.full[st]);
      }
      sm.issued = n + 1;
    }
  }

  // ======================= compute warps =======================
  __nv_bfloat16* __restrict__ out = reinterpret_cast<__nv_bfloat16*>(p.out);
  const float inv_sqrt_d = rsqrtf((float)D);
  const int cv = tid % kCV;
  const int rg = tid / kCV;
  const int warp = tid >> 5, lane = tid & 31;

  for (int n = 0;; ++n) {
    const int st = n % kStages;
    const int k = n / R, jh = n % R;

    if (tid == 0) sm.ok = mbar_wait_bounded(&sm.full[st], (n / kStages) & 1) ? 1 : 0;
    consumer_sync();
    if (!sm.ok) {
      if (tid == 0) {
        atomicOr((unsigned*)&hdr[kErr], GDN_FLAG_TIMEOUT);
        // the copies already issued land before the CTA ends
        for (int m = n + 1; m < sm.issued && m < n + kStages; ++m)
          mbar_wait_bounded(&sm.full[m % kStages], (m / kStages) & 1);
        if (late) asm volatile("griddepcontrol.wait;" ::: "memory");
      }
      return;
    }
    const int unit = sm.meta[st].unit;
    if (unit < 0) break;
    const int kh = unit % Hk;
    const int h = kh * R + jh;
    const int row = sm.meta[st].row;
    const int wblk = sm.meta[st].wblk;
    unsigned char* wbase = p.layer_base + (size_t)wblk * p.stride;

    if (jh == 0) {
      // ---- conv + SiLU of the unit's channels; new conv state; gates
      const ConvIn<kKda>& ci = sm.cin[k & 1];
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
        // new conv state: the last K-1 inputs of [old state ; x]
#pragma unroll
        for (int j = 0; j < KC - 2; ++j) tail_w[(size_t)j * C + ch] = ci.tail[j + 1][lc];
        tail_w[(size_t)(KC - 2) * C + ch] = ci.x[lc];
      }
      if constexpr (kKda) {
        // one key-channel decay per thread: R v-heads x D channels = kConsumers
        const int jg = tid / D, c = tid % D;
        const int hh = kh * R + jg;
        const float araw = __bfloat162float(ci.g.a[jg][c]) + p.dt_bias[(size_t)hh * D + c];
        sm.gt.alpha[jg][c] = __expf(-__expf(p.A_log[hh]) * softplus_f32(araw));
        if (tid < R) sm.gt.beta[tid] = sigmoid_f32(__bfloat162float(ci.b[kh * R + tid]));
      } else if (tid < R) {
        const int hh = kh * R + tid;
        const float araw = __bfloat162float(ci.g.a[hh]) + p.dt_bias[hh];
        const float g = -__expf(p.A_log[hh]) * softplus_f32(araw);
        sm.gt.gate[tid][0] = __expf(g);
        sm.gt.gate[tid][1] = sigmoid_f32(__bfloat162float(ci.b[hh]));
      }
      consumer_sync();
      if (lane == 0) mbar_arrive(&sm.cempty[k & 1]);
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
      consumer_sync();
    }
    const float qs = rsqrtf(sm.red[0] + kL2Eps) * inv_sqrt_d;
    const float ks = rsqrtf(sm.red[1] + kL2Eps);
    // scalar gate: e^g scales the whole state (decay); per-channel decay:
    // alpha[r] scales state row r (decay stays 1)
    float decay = 1.f, beta;
    const float* alpha = nullptr;
    if constexpr (kKda) {
      beta = sm.gt.beta[jh];
      alpha = sm.gt.alpha[jh];
    } else {
      decay = sm.gt.gate[jh][0];
      beta = sm.gt.gate[jh][1];
    }
    const float* buf = sm.buf[st];

    // ---- pass 1: state rows into registers, partial S k and S q (S' k and
    // S' q with the per-channel decay)
    float4 S[kRows];
    float kr[kRows];
    float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const int r = rg + kG * i;
      S[i] = *reinterpret_cast<const float4*>(buf + r * D + 4 * cv);
      kr[i] = sm.y[D + r] * ks;
      float ka = kr[i], qr = sm.y[r] * qs;
      if constexpr (kKda) {
        ka *= alpha[r];
        qr *= alpha[r];
      }
      pk.x += S[i].x * ka; pk.y += S[i].y * ka; pk.z += S[i].z * ka; pk.w += S[i].w * ka;
      pq.x += S[i].x * qr; pq.y += S[i].y * qr; pq.z += S[i].z * qr; pq.w += S[i].w * qr;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[st]);  // this warp is done with the buffer
    *reinterpret_cast<float4*>(&sm.part[0][rg][4 * cv]) = pk;
    *reinterpret_cast<float4*>(&sm.part[1][rg][4 * cv]) = pq;
    consumer_sync();
    if (tid < D) {
      float sk = 0.f, sq = 0.f;
#pragma unroll
      for (int g2 = 0; g2 < kG; ++g2) {
        sk += sm.part[0][g2][tid];
        sq += sm.part[1][g2][tid];
      }
      const float vv = sm.y[2 * D + jh * D + tid];
      const float u = beta * (vv - decay * sk);
      sm.u[tid] = u;
      out[((size_t)row * Hv + h) * D + tid] =
          __float2bfloat16_rn(decay * sq + sm.red[2] * qs * ks * u);
    }
    consumer_sync();
    // ---- pass 2: S <- e^g S + u k^T (S Diag(alpha) + u k^T) from registers,
    // straight to the write block
    float* S_w = reinterpret_cast<float*>(wbase + p.rec_off) + (size_t)h * D * D;
    const float4 u4 = *reinterpret_cast<const float4*>(&sm.u[4 * cv]);
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const int r = rg + kG * i;
      const float dr = kKda ? alpha[r] : decay;
      float4 s4 = S[i];
      s4.x = dr * s4.x + u4.x * kr[i];
      s4.y = dr * s4.y + u4.y * kr[i];
      s4.z = dr * s4.z + u4.z * kr[i];
      s4.w = dr * s4.w + u4.w * kr[i];
      *reinterpret_cast<float4*>(S_w + (size_t)r * D + 4 * cv) = s4;
    }
    // (per-channel decay: the next unit's gate pass rewrites alpha only after
    // its own full-barrier wait and a consumer barrier, which every thread
    // reaches after this loop)
  }
  // launched early behind the prefill's recurrence: it has completed before
  // this CTA ends
  if (late && tid == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

int g_num_sms = 0;

}  // namespace

bool decode_supported(int d, int act, int Hk, int Hv, int K) {
  return d == D && act == GDN_BF16 && Hv == R * Hk && K == KC && Hv % 8 == 0 && Hv <= kMaxHv;
}

namespace {

template <bool kKda>
cudaError_t launch_decode_t(const FwdParams& pin, int max_dec, bool late, cudaStream_t stream) {
  FwdParams p = pin;
  p.decode_late = late ? 1 : 0;
  if (max_dec <= 0) return cudaSuccess;
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 1;
  }
  const long long max_units = (long long)max_dec * p.Hk;
  const int grid = (int)(max_units < g_num_sms ? max_units : g_num_sms);
  const size_t smem = sizeof(DecodeSmem<kKda>);
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<kKda>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(decode_kernel<kKda>, dim3(grid), dim3(kThreads), smem, stream, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const FwdParams& p, int max_dec, cudaStream_t stream, bool late) {
  return launch_decode_t<false>(p, max_dec, late, stream);
}
cudaError_t launch_kda_decode(const FwdParams& p, int max_dec, cudaStream_t stream, bool late) {
  return launch_decode_t<true>(p, max_dec, late, stream);
}

}  // namespace gdn

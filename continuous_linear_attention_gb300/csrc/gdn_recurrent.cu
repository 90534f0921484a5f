// Token-serial kernel of the layer forward: the varlen causal conv1d + SiLU and
// the gated delta rule, one CTA per (sequence, k-head group), the recurrent
// state of every v-head of the group held in registers for the whole
// sequence.  It computes exactly the definition token by token, so it is the
// path for short sequences and for head sizes the chunked kernel does not
// cover.
//
// What it computes (per token t of a sequence, v-head h reading k-head
// h / (Hv/Hk)):
//   y[c]  = SiLU( sum_j w[c][j] * xhat[t-K+1+j][c] )    (conv continued from the
//           sequence's conv state; "Continuous batching for linear attention
//           layers": a varlen causal convolution continues every sequence from
//           its own conv state)
//   q,k   = L2-normalised q and k parts of y, q scaled by 1/sqrt(d_k)
//   g     = -exp(A_log[h]) softplus(a_t + dt_bias[h]),  beta = sigmoid(b_t)
//   p = S k, r = S q (old S),  u = beta (v - e^g p),
//   S    <- e^g S + u k^T,     o = S q = e^g r + (k.q) u    (gated delta rule)
// The conv window of each channel lives in registers, so after the last token
// it IS the new conv state (the last K-1 inputs of [old state ; x]).
//
// The per-channel-decay (KDA) instance takes one decay per key channel,
// alpha[c] = e^{-exp(A_log[h]) softplus(a_t[h][c] + dt_bias[h][c])}, and with
// S' = S Diag(alpha): p = S' k, r = S' q, u = beta (v - p), o = r + (k.q) u,
// S <- S' + u k^T (Kimi Linear's delta rule with per-channel decay); with
// the state stored k-major the decay scales whole rows, folded into the k and
// q of the reductions and into the row update.
//
// Ownership: this CTA is the only one touching the q/k channels of its k-head
// and the v channels of its v-heads, and the recurrent states of those
// v-heads, so reading the old state and overwriting it in place is race-free.
#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"

namespace gdn {
namespace {

constexpr int kHeadThreads = 256;  // threads per v-head

// mode: kAll every active sequence, kLong those longer than one token, kRedo
// the v-heads of the prefill list marked for a redo (outputs and recurrent
// states of those heads only; the conv state is left to the conv-state update)
enum Mode : int { kAll = 0, kLong = 1, kRedo = 2 };

template <int D, typename Act, bool kKda>
__global__ void __launch_bounds__(2 * kHeadThreads)
recurrent_kernel(FwdParams p, int mode) {
  constexpr int CV = D / 4;                 // float4 columns per state row
  constexpr int G = kHeadThreads / CV;      // row groups
  constexpr int NJ = D / G;                 // rows per thread
  static_assert(NJ * G == D, "row split");
  pdl_wait_then_release();
  const int R = p.Hv / p.Hk;                // v-heads per k-head (1 or 2)
  const WorkArea& wk = p.work;
  const bool long_only = mode != kAll;
  const int n_items = wk.header()[long_only ? kNPre : kNItems];
  if ((int)blockIdx.x >= n_items) return;
  const int kh = blockIdx.y;
  // redo: the marked v-heads of this k-head group (bits kh*R .. kh*R+R-1)
  uint32_t marks = (1u << R) - 1u;
  if (mode == kRedo) {
    const int h0 = kh * R;
    marks = (reinterpret_cast<const uint32_t*>(wk.redo())[2 * blockIdx.x + (h0 >> 5)] >> (h0 & 31)) &
            ((1u << R) - 1u);
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
  const int NCH = (2 + R) * D;
  float* y = smem;                      // [NCH] conv + SiLU output of the token
  float* part = y + 4 * D;              // [R][2][G][D] partial S k, S q
  float* uo = part + 2 * 2 * G * D;     // [R][D] u
  float* al = uo + 2 * D;               // [R][D] key-channel decays (per-channel decay only)
  float* red = kKda ? al + 2 * D : al;  // [4] sum q^2, sum k^2, q.k
  float* gb = red + 4;                  // [R][2] e^g (scalar gate only), beta

  const int tid = threadIdx.x;
  const int nt = blockDim.x;

  // ---- conv channels owned by this thread (at most 2): local -> global
  int gch[2];
  float win[2][kMaxConvK - 1];
  float wc[2][kMaxConvK];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int lc = tid + c * nt;
    gch[c] = -1;
    if (lc < NCH) {
      if (lc < D) gch[c] = kh * D + lc;
      else if (lc < 2 * D) gch[c] = Hk * D + kh * D + (lc - D);
      else gch[c] = 2 * Hk * D + kh * R * D + (lc - 2 * D);
#pragma unroll
      for (int j = 0; j < kMaxConvK - 1; ++j)
        win[c][j] = j < K - 1 ? to_f32(tail_r[(size_t)j * C + gch[c]]) : 0.f;
#pragma unroll
      for (int j = 0; j < kMaxConvK; ++j)
        wc[c][j] = j < K ? to_f32(wconv[(size_t)gch[c] * K + j]) : 0.f;
    }
  }

  // ---- recurrent state of this thread's v-head, rows r_i = rg + G*i, float4 column cv
  const int j_head = tid / kHeadThreads;
  const int li = tid % kHeadThreads;
  const int h = kh * R + j_head;
  const bool mine = (marks >> j_head) & 1u;  // this thread's v-head is written
  const int cv = li % CV;
  const int rg = li / CV;
  const float* S_r = reinterpret_cast<const float*>(rbase + p.rec_off) + (size_t)h * D * D;
  float* S_w = reinterpret_cast<float*>(wbase + p.rec_off) + (size_t)h * D * D;
  float4 S[NJ];
#pragma unroll
  for (int i = 0; i < NJ; ++i)
    S[i] = *reinterpret_cast<const float4*>(S_r + (size_t)(rg + G * i) * D + 4 * cv);

  const float inv_sqrt_d = rsqrtf((float)D);
  for (int t = 0; t < L; ++t) {
    const size_t row = (size_t)(t0 + t);
    // 1. conv + SiLU of the owned channels; gates of the group's v-heads
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      if (gch[c] < 0) continue;
      const float xv = to_f32(x[row * C + gch[c]]);
      // window slots 0..K-2 hold the previous K-1 inputs, oldest first; the
      // unrolled selects keep every index static (registers, no local memory)
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
    if constexpr (kKda) {
      if (tid < R * D) {
        const int jg = tid / D, c = tid % D;
        const int hh = kh * R + jg;
        const float araw = to_f32(av[(row * Hv + hh) * D + c]) + p.dt_bias[(size_t)hh * D + c];
        al[jg * D + c] = __expf(-__expf(p.A_log[hh]) * softplus_f32(araw));
      }
      if (tid < R) gb[2 * tid + 1] = sigmoid_f32(to_f32(bv[row * Hv + kh * R + tid]));
    } else if (tid < R) {
      const int hh = kh * R + tid;
      const float araw = to_f32(av[row * Hv + hh]) + p.dt_bias[hh];
      const float g = -__expf(p.A_log[hh]) * softplus_f32(araw);
      gb[2 * tid] = __expf(g);
      gb[2 * tid + 1] = sigmoid_f32(to_f32(bv[row * Hv + hh]));
    }
    __syncthreads();
    // 2. sums of squares and q.k (warps 0..2)
    if (tid < 96) {
      const int w = tid >> 5, lane = tid & 31;
      float acc = 0.f;
      for (int i = lane; i < D; i += 32) {
        const float qv = y[i], kv = y[D + i];
        acc += w == 0 ? qv * qv : (w == 1 ? kv * kv : qv * kv);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) red[w] = acc;
    }
    __syncthreads();
    const float qs = rsqrtf(red[0] + kL2Eps) * inv_sqrt_d;
    const float ks = rsqrtf(red[1] + kL2Eps);
    // scalar gate: e^g scales the whole state; per-channel decay: alpha[r]
    // scales state row r (decay stays 1)
    const float decay = kKda ? 1.f : gb[2 * j_head];
    const float beta = gb[2 * j_head + 1];
    const float* alh = al + j_head * D;
    // 3. partial S k and S q (S' k and S' q) over this thread's rows
    float kr[NJ];
    float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
    for (int i = 0; i < NJ; ++i) {
      const int r = rg + G * i;
      kr[i] = y[D + r] * ks;
      float ka = kr[i], qr = y[r] * qs;
      if constexpr (kKda) {
        ka *= alh[r];
        qr *= alh[r];
      }
      pk.x += S[i].x * ka; pk.y += S[i].y * ka; pk.z += S[i].z * ka; pk.w += S[i].w * ka;
      pq.x += S[i].x * qr; pq.y += S[i].y * qr; pq.z += S[i].z * qr; pq.w += S[i].w * qr;
    }
    float* myp = part + (size_t)j_head * 2 * G * D;
    *reinterpret_cast<float4*>(myp + (size_t)rg * D + 4 * cv) = pk;
    *reinterpret_cast<float4*>(myp + (size_t)(G + rg) * D + 4 * cv) = pq;
    __syncthreads();
    // 4. u and o for each v column
    if (li < D) {
      float sk = 0.f, sq = 0.f;
      for (int g2 = 0; g2 < G; ++g2) {
        sk += myp[(size_t)g2 * D + li];
        sq += myp[(size_t)(G + g2) * D + li];
      }
      const float vv = y[2 * D + j_head * D + li];
      const float u = beta * (vv - decay * sk);
      const float kq = red[2] * qs * ks;
      uo[j_head * D + li] = u;
      if (mine) out[(row * Hv + h) * D + li] = from_f32<Act>(decay * sq + kq * u);
    }
    __syncthreads();
    // 5. S <- e^g S + u k^T  (S Diag(alpha) + u k^T)
    const float4 u4 = *reinterpret_cast<const float4*>(uo + j_head * D + 4 * cv);
#pragma unroll
    for (int i = 0; i < NJ; ++i) {
      const float dr = kKda ? alh[rg + G * i] : decay;
      S[i].x = dr * S[i].x + u4.x * kr[i];
      S[i].y = dr * S[i].y + u4.y * kr[i];
      S[i].z = dr * S[i].z + u4.z * kr[i];
      S[i].w = dr * S[i].w + u4.w * kr[i];
    }
    // per-channel decay: the next token's gate pass overwrites al[], which
    // step 5 just read
    if constexpr (kKda) __syncthreads();
  }

  // ---- write back: recurrent state, then the conv window as the new conv state
  if (mine) {
#pragma unroll
    for (int i = 0; i < NJ; ++i)
      *reinterpret_cast<float4*>(S_w + (size_t)(rg + G * i) * D + 4 * cv) = S[i];
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

template <int D, typename Act, bool kKda = false>
cudaError_t launch_rec(const FwdParams& p, int max_items, int mode, cudaStream_t stream) {
  const int R = p.Hv / p.Hk;
  constexpr int G = kHeadThreads / (D / 4);
  const size_t smem = sizeof(float) * (4 * D + 2 * 2 * G * D + 2 * D + (kKda ? 2 * D : 0) + 4 + 4);
  dim3 grid(max_items, p.Hk);
  const cudaError_t e = launch_pdl(recurrent_kernel<D, Act, kKda>, grid, dim3(R * kHeadThreads),
                                   smem, stream, p, mode);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_recurrent(const FwdParams& p, int d, int act, int max_items, bool long_only,
                             cudaStream_t stream) {
  if (max_items <= 0) return cudaSuccess;
  const int mode = long_only ? kLong : kAll;
  if (act == GDN_F32) {
    if (d == 32) return launch_rec<32, float>(p, max_items, mode, stream);
    if (d == 64) return launch_rec<64, float>(p, max_items, mode, stream);
    return launch_rec<128, float>(p, max_items, mode, stream);
  }
  if (d == 32) return launch_rec<32, __nv_bfloat16>(p, max_items, mode, stream);
  if (d == 64) return launch_rec<64, __nv_bfloat16>(p, max_items, mode, stream);
  return launch_rec<128, __nv_bfloat16>(p, max_items, mode, stream);
}

cudaError_t launch_redo(const FwdParams& p, int d, int act, int max_pre, cudaStream_t stream) {
  if (max_pre <= 0) return cudaSuccess;
  if (d != 128 || act != GDN_BF16) return cudaErrorInvalidValue;  // the chunked kernels' shape
  return launch_rec<128, __nv_bfloat16>(p, max_pre, kRedo, stream);
}

cudaError_t launch_kda_recurrent(const FwdParams& p, int d, int act, int max_items,
                                 bool long_only, cudaStream_t stream) {
  if (max_items <= 0) return cudaSuccess;
  const int mode = long_only ? kLong : kAll;
  if (act == GDN_F32) {
    if (d == 32) return launch_rec<32, float, true>(p, max_items, mode, stream);
    if (d == 64) return launch_rec<64, float, true>(p, max_items, mode, stream);
    return launch_rec<128, float, true>(p, max_items, mode, stream);
  }
  if (d == 32) return launch_rec<32, __nv_bfloat16, true>(p, max_items, mode, stream);
  if (d == 64) return launch_rec<64, __nv_bfloat16, true>(p, max_items, mode, stream);
  return launch_rec<128, __nv_bfloat16, true>(p, max_items, mode, stream);
}

cudaError_t launch_kda_redo(const FwdParams& p, int max_pre, cudaStream_t stream) {
  if (max_pre <= 0) return cudaSuccess;
  return launch_rec<128, __nv_bfloat16, true>(p, max_pre, kRedo, stream);
}

}  // namespace gdn

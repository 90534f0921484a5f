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
#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"

namespace gdn {
namespace {

constexpr int kSsdThreads = 256;

template <int P, int NS, typename Act>
__global__ void __launch_bounds__(kSsdThreads) ssd_recurrent_kernel(SsdParams p) {
  constexpr int NC = kSsdThreads / P;  // threads per state row
  constexpr int NPT = NS / NC;         // state entries per thread
  constexpr int NCH = P + 2 * NS;      // conv channels of one head: x | B | C
  static_assert(NC * P == kSsdThreads && NPT * NC == NS && NPT % 4 == 0, "state split");
  static_assert(NC <= 32 && 32 % NC == 0, "a state row's threads sit in one warp");
  static_assert(NCH <= 2 * kSsdThreads, "at most two conv channels per thread");
  __shared__ float yv[NCH];
  __shared__ float gate[2];
  pdl_wait_then_release();
  const int n_items = p.work.header()[kNItems];
  if ((int)blockIdx.x >= n_items) return;
  const int s = p.work.items()[blockIdx.x];
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
__global__ void __launch_bounds__(256) ssd_tail_kernel(SsdParams p) {
  pdl_wait_then_release();
  const int n_items = p.work.header()[kNItems];
  if ((int)blockIdx.x >= n_items) return;
  const int s = p.work.items()[blockIdx.x];
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

template <int P, int NS, typename Act>
cudaError_t launch_rec_t(const SsdParams& p, int max_items, cudaStream_t stream) {
  cudaError_t e = launch_pdl(ssd_recurrent_kernel<P, NS, Act>, dim3(max_items, p.H),
                             dim3(kSsdThreads), 0, stream, p);
  if (e != cudaSuccess) return e;
  e = launch_pdl(ssd_tail_kernel<Act>, dim3(max_items, (p.C + 255) / 256), dim3(256), 0, stream,
                 p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int P, typename Act>
cudaError_t launch_by_state(const SsdParams& p, int NS, int max_items, cudaStream_t stream) {
  if (NS == 32) return launch_rec_t<P, 32, Act>(p, max_items, stream);
  if (NS == 64) return launch_rec_t<P, 64, Act>(p, max_items, stream);
  return launch_rec_t<P, 128, Act>(p, max_items, stream);
}

}  // namespace

bool ssd_supported(int P, int NS) {
  return (P == 32 || P == 64) && (NS == 32 || NS == 64 || NS == 128);
}

cudaError_t launch_ssd(const SsdParams& p, int P, int NS, int act, int max_items,
                       cudaStream_t stream) {
  if (max_items <= 0) return cudaSuccess;
  if (!ssd_supported(P, NS)) return cudaErrorInvalidValue;
  if (act == GDN_F32)
    return P == 32 ? launch_by_state<32, float>(p, NS, max_items, stream)
                   : launch_by_state<64, float>(p, NS, max_items, stream);
  return P == 32 ? launch_by_state<32, __nv_bfloat16>(p, NS, max_items, stream)
                 : launch_by_state<64, __nv_bfloat16>(p, NS, max_items, stream);
}

}  // namespace gdn

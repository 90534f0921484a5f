// Conv prologue of the prefill path as its own memory-bound kernel: for every
// token of the sequences longer than one token, the varlen causal depthwise
// conv1d + SiLU continued from the sequence's conv state ("Continuous
// batching for linear attention layers": a varlen causal convolution
// continues every sequence from its own conv state), then the L2 norms of q
// and k (q also scaled by 1/sqrt(d_k)).  Results go to a pool-owned scratch
// in fp16, which the chunked kernel loads tile by tile with TMA:
//   qk[row][kh][0..127]   = q~ of k-head kh,  qk[row][kh][128..255] = k~
//   vv[row][h][0..127]    = v of v-head h (SiLU output)
// Computing q~/k~ once per k-head here, instead of once per v-head inside the
// chunked kernel, halves the q/k conv work, and keeps the chunked kernel's
// instruction stream for the recurrence.
//
// The same CTA writes the gates of its chunk for both v-heads of the k-head:
//   g[row][h] = (G, beta), G the inclusive cumulative sum of the log decay
//   g = -e^{A_log} softplus(a + dt_bias) inside the 64-token chunk.
//
// One CTA per (64-token chunk of a prefill sequence, k-head); chunks are
// found from the scheduler's chunk prefix over the sorted prefill list.  The
// CTA's 67 x rows (3 halo + 64) of its 512 channels arrive as eight 2-D TMA
// boxes (128-byte swizzled, 72 KiB) so three CTAs per SM keep ~200 KiB of
// loads in flight; the first chunk's halo rows are then replaced by the
// sequence's conv state.  Thread (tq, g) computes channel group g (8
// channels) of q, k and the two v-heads for tokens 4tq .. 4tq+3 with a
// sliding window over 7 staged rows.
#include <cuda.h>

#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int D = 128;
constexpr int CH = 64;
constexpr int KC = 4;
constexpr int kThreads = 256;
constexpr int R = 2;  // v-heads per k-head
constexpr int XROWS = CH + KC - 1;
constexpr uint32_t XSUB = 9216;  // one box: 72 rows x 128 B, 1024-aligned
constexpr uint32_t XBOX_BYTES = 64 * XROWS * 2;
// the conv taps of a box's 64 channels (bf16 [64][4], 512 bytes) sit in the
// box's padding rows, right after its 67 staged rows
constexpr uint32_t WS_OFF = XBOX_BYTES;
constexpr uint32_t WS_BYTES = 64 * KC * 2;
static_assert(WS_OFF + WS_BYTES <= XSUB && WS_OFF % 16 == 0, "taps must fit the box padding");
constexpr uint32_t SMEM_BYTES = 8 * XSUB + 1024;

// Packed fp32 pairs: d = a * b + c on both lanes (one fma.rn.f32x2).
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// bf16 pair (low, high halves of a word) -> packed fp32 pair
__device__ __forceinline__ unsigned long long bf2_to_f2(uint32_t u) {
  return (unsigned long long)(u << 16) | ((unsigned long long)(u & 0xffff0000u) << 32);
}

__device__ __forceinline__ uint4 pack8_f16(const float* v) {
  uint4 w;
  __half2 h0 = __floats2half2_rn(v[0], v[1]), h1 = __floats2half2_rn(v[2], v[3]);
  __half2 h2 = __floats2half2_rn(v[4], v[5]), h3 = __floats2half2_rn(v[6], v[7]);
  w.x = *reinterpret_cast<uint32_t*>(&h0);
  w.y = *reinterpret_cast<uint32_t*>(&h1);
  w.z = *reinterpret_cast<uint32_t*>(&h2);
  w.w = *reinterpret_cast<uint32_t*>(&h3);
  return w;
}

__global__ void __launch_bounds__(kThreads, 3) prep_kernel(FwdParams p,
                                                       const __grid_constant__ CUtensorMap tmx) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* xt = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t xbar;
  __shared__ float gtot[2];
  __shared__ int ok;
  pdl_wait_then_release();
  int32_t* hdr = p.work.header();
  const int n_chunks = hdr[kPreChunks];
  const int gidx = blockIdx.x;
  if (gidx >= n_chunks) return;
  // which prefill sequence / chunk: binary search in the chunk prefix
  const int n_pre = hdr[kNPre];
  const int32_t* cp = p.work.pre_cp();
  int lo = 0, hi = n_pre - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cp[mid] <= gidx) lo = mid; else hi = mid - 1;
  }
  const int s = p.work.pre()[lo];
  const int c = gidx - cp[lo];
  const int kh = blockIdx.y;
  const int Hk = p.Hk, Hv = p.Hv, C = p.C;
  const int seq0 = p.cu[s];
  const int L = p.cu[s + 1] - seq0;
  const int c0 = c * CH;
  const int n = min(CH, L - c0);
  const int rblk = p.has_past[s] ? p.blk[s] : 0;
  const __nv_bfloat16* tail = reinterpret_cast<const __nv_bfloat16*>(p.layer_base + (size_t)rblk * p.stride);
  const __nv_bfloat16* w = reinterpret_cast<const __nv_bfloat16*>(p.conv_w);
  __half* qk = reinterpret_cast<__half*>(p.scr_qk);
  __half* vv = reinterpret_cast<__half*>(p.scr_v);

  const int tid = threadIdx.x;
  // local channel block b (64 channels): 0,1 q | 2,3 k | 4..7 v of heads 2kh, 2kh+1
  auto gch = [&](int b) {
    return b < 2 ? kh * D + b * 64
                 : (b < 4 ? Hk * D + kh * D + (b - 2) * 64 : 2 * Hk * D + kh * R * D + (b - 4) * 64);
  };
  if (tid == 0) {
    mbar_init(&xbar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&xbar, 8u * (XBOX_BYTES + WS_BYTES));
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      tma_load_2d(xt + b * XSUB, &tmx, gch(b), seq0 + c0 - (KC - 1), &xbar);
      bulk_g2s(xt + b * XSUB + WS_OFF, w + (size_t)gch(b) * KC, WS_BYTES, &xbar);
    }
  }
  // gates of the chunk's tokens for the k-head's two v-heads (threads 0..127,
  // token tid % 64 of head 2kh + tid / 64): g = -e^{A_log} softplus(a + dt_bias),
  // beta = sigmoid(b), and the inclusive cumulative sum G of g inside the chunk
  float gcum = 0.f, gbeta = 0.f;
  if (tid < R * CH) {
    const int h = kh * R + (tid >> 6), i = tid & 63;
    if (i < n) {
      const size_t row = (size_t)(seq0 + c0 + i);
      const __nv_bfloat16* av = reinterpret_cast<const __nv_bfloat16*>(p.a);
      const __nv_bfloat16* bv = reinterpret_cast<const __nv_bfloat16*>(p.b);
      gcum = -__expf(p.A_log[h]) * softplus_f32(__bfloat162float(av[row * Hv + h]) + p.dt_bias[h]);
      gbeta = sigmoid_f32(__bfloat162float(bv[row * Hv + h]));
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, gcum, o);
      if ((tid & 31) >= o) gcum += t;
    }
    if ((tid & 63) == 31) gtot[tid >> 6] = gcum;
  }
  if (tid == 0 && kh == 0)
    reinterpret_cast<int2*>(p.scr_c)[gidx] = make_int2(seq0 + c0, n);  // the chunk's record
  if (tid == 0) ok = mbar_wait_bounded(&xbar, 0) ? 1 : 0;
  __syncthreads();
  if (tid < R * CH) {
    const int h = kh * R + (tid >> 6), i = tid & 63;
    if (i >= 32) gcum += gtot[tid >> 6];
    if (i < n) {
      float2* dst = reinterpret_cast<float2*>(p.scr_g) + (size_t)(seq0 + c0 + i) * Hv + h;
      *dst = make_float2(gcum, gbeta);
    }
  }
  if (!ok) {
    if (tid == 0) atomicOr((unsigned*)&hdr[kErr], GDN_FLAG_TIMEOUT);
    return;
  }
  if (c == 0) {
    // the halo rows of the first chunk are the conv state
    for (int t = tid; t < (KC - 1) * 64; t += kThreads) {
      const int r = t >> 6, q8 = t & 63, b = q8 >> 3, cc = (q8 & 7) * 8;
      *reinterpret_cast<uint4*>(xt + b * XSUB + tc::sw128_offset(r, cc)) =
          *reinterpret_cast<const uint4*>(tail + (size_t)r * C + gch(b) + cc);
    }
    __syncthreads();
  }
  const int tq = tid >> 4, g = tid & 15;
  const int i0 = 4 * tq;
  const float inv_sqrt_d = rsqrtf((float)D);
  float vmax = 0.f;  // largest |v| written (NaN if any is NaN)
#pragma unroll 1
  for (int part = 0; part < 2 + R; ++part) {  // q, k, v of head 2kh, v of head 2kh+1
    const int lc = part * D + g * 8;  // local channel: box lc / 64, column lc % 64
    // taps as packed channel pairs: w2[j][p] = (w[c+2p][j], w[c+2p+1][j])
    unsigned long long w2[KC][4];
#pragma unroll
    for (int p2 = 0; p2 < 4; ++p2) {
      const unsigned char* wp = xt + (lc >> 6) * XSUB + WS_OFF + ((lc + 2 * p2) & 63) * KC * 2;
      const uint2 wa = *reinterpret_cast<const uint2*>(wp);            // channel c+2p, taps 0..3
      const uint2 wb = *reinterpret_cast<const uint2*>(wp + KC * 2);   // channel c+2p+1
      const uint32_t a4[4] = {wa.x << 16, wa.x & 0xffff0000u, wa.y << 16, wa.y & 0xffff0000u};
      const uint32_t b4[4] = {wb.x << 16, wb.x & 0xffff0000u, wb.y << 16, wb.y & 0xffff0000u};
#pragma unroll
      for (int j = 0; j < KC; ++j) w2[j][p2] = (unsigned long long)a4[j] | ((unsigned long long)b4[j] << 32);
    }
    unsigned long long acc2[4][4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc2[t][e] = 0ull;
#pragma unroll
    for (int rr = 0; rr < 4 + KC - 1; ++rr) {
      const uint4 xw = *reinterpret_cast<const uint4*>(xt + (lc >> 6) * XSUB +
                                                       tc::sw128_offset(i0 + rr, lc & 63));
      const unsigned long long xv2[4] = {bf2_to_f2(xw.x), bf2_to_f2(xw.y), bf2_to_f2(xw.z),
                                         bf2_to_f2(xw.w)};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int j = rr - t;
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
        acc[t][2 * e] = __uint_as_float((uint32_t)acc2[t][e]);
        acc[t][2 * e + 1] = __uint_as_float((uint32_t)(acc2[t][e] >> 32));
      }
    float y[4][8];
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int e = 0; e < 8; ++e) y[t][e] = silu_f32(acc[t][e]);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int i = i0 + t;
      if (part < 2) {  // q and k: L2 norm over the 16 threads of the token
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss += y[t][e] * y[t][e];
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float sc = rsqrtf(ss + kL2Eps) * (part == 0 ? inv_sqrt_d : 1.f);
#pragma unroll
        for (int e = 0; e < 8; ++e) y[t][e] *= sc;
      }
      if (i < n) {
        if (part >= 2) {
#pragma unroll
          for (int e = 0; e < 8; e += 2) vmax = max_abs3_nan(vmax, y[t][e], y[t][e + 1]);
        }
        const size_t row = (size_t)(seq0 + c0 + i);
        __half* dst = part < 2 ? qk + (row * Hk + kh) * (2 * D) + part * D + g * 8
                               : vv + (row * Hv + kh * R + part - 2) * D + g * 8;
        *reinterpret_cast<uint4*>(dst) = pack8_f16(y[t]);
      }
    }
  }
  // v enters the tensor-core operands in fp16: report values outside its range
  if (__syncthreads_or(!(vmax <= 65000.f) ? 1 : 0) && tid == 0)
    atomicOr((unsigned*)&p.work.header()[kErr], GDN_FLAG_RANGE);
}

}  // namespace

cudaError_t launch_prep(const FwdParams& p, const void* x_map, int max_chunks,
                        cudaStream_t stream) {
  if (max_chunks <= 0) return cudaSuccess;
  cudaError_t e =
      cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(max_chunks, p.Hk);
  return launch_pdl(prep_kernel, grid, dim3(kThreads), SMEM_BYTES, stream, p,
                    *static_cast<const CUtensorMap*>(x_map));
}

}  // namespace gdn

// State-independent half of the chunked prefill, fully parallel over the
// 64-token chunks of the prefill sequences: one CTA per (chunk, v-head),
// four CTAs per SM.
//
// With G_i the inclusive cumulative gate inside the chunk, beta_i the write
// strength and q~/k~ the normalised rows (all from prep_kernel), the chunk-64
// WY form of the gated delta rule (Gated Delta Networks, chunkwise form;
// "Continuous batching for linear attention layers" runs it over cu_seqlens)
// needs, per chunk and v-head, three products that do not involve the state:
//   A_ij = beta_i e^{G_i - G_j} (k~_i . k~_j)   (j < i)
//   T    = (I + A)^{-1}                         (unit lower triangular)
//   P_ij = e^{G_i - G_j} (q~_i . k~_j)           (j <= i)
// and with them the state path (seq_kernel) reduces to
//   U^T  = v^T (T diag beta)^T - S0 w^T,   w = T diag(beta e^G) k~
//   o_i  = e^{G_i} S0 q~_i + sum_{j<=i} P_ij u_j
//   S_C  = e^{G_C} S0 + sum_j e^{G_C - G_j} u_j k~_j^T.
// This kernel writes, per packed row i < n of the chunk and v-head h
// (token-major, fp16, next to q~/k~/v in the pool's prefill scratch):
//   U0[row][h][0..127] = u_i = (T diag(beta) V)_i   (the updates for a zero state)
//   Wn[row][h][0..127] = -w_i = -(T diag(beta e^G) K~)_i
//   P [row][h][0..63]  = P_ij
// Tensor cores: X = [q~ ; k~] k~^T (128 x 64 x 128), then
// [-T diag(beta e^G) ; T diag(beta)] times k~ and times v (128 x 128 x 64
// each, k~ and v as MN-major operands straight from their token-major tiles:
// rows 0..63 of the first product are -w, rows 64..127 of the second are u),
// and the 16 x 16 block products of the solve on the warp-level path
// (mma.sync, tf32 with a head/tail split).  CUDA cores: the masks, the
// diagonal 16 x 16 blocks of T by column substitution, and the conversions.
// Rows of the tiles past the end of the sequence are zeroed in shared memory
// first, so that no value of another sequence (or stale scratch) reaches a
// product.
#include <cuda.h>

#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

using E = __half;
constexpr int D = 128;
constexpr int CH = 64;
constexpr int kThreads = 256;
constexpr int R = 2;    // v-heads per k-head
constexpr int AP = 68;  // pitch (floats) of the fp32 A / T rows
constexpr float kF16Max = 65000.f;
constexpr float kLog2e = 1.4426950408889634f;

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

// shared memory map (offsets from a 1024-byte aligned base).  Once X is done
// the two q~ slots of the [q~ ; k~] tile are reused: slot 1 takes v columns
// 64..127 at once, slot 0 holds the B blocks of the solve and then v columns
// 0..63.  The A/T array becomes the MMAs' A tile when T is done.
constexpr uint32_t BOX = 8192;         // one 64 x 64 fp16 box
constexpr uint32_t KB_STRIDE = 16384;  // K-blocks of the 128-row [q~ ; k~] tile
constexpr uint32_t OFF_QK = 0;         // [q~ ; k~], 2 K-blocks x 128 rows
constexpr uint32_t OFF_Z = 0;          // B blocks of the solve fp32 [6][16][20] (q~ slot 0)
constexpr uint32_t OFF_AT = 32768;     // A, overwritten block by block by T: fp32 [64][AP]
constexpr uint32_t OFF_TT = OFF_AT;    // then [-T diag(beta e^G) ; T diag(beta)] fp16, 128 rows
constexpr uint32_t OFF_GT = 50176;     // gates [64][4] fp32: (G, beta) of the k-head's v-heads
constexpr uint32_t OFF_GH = 51200;     // this head's G [64] in log2 units (G log2 e)
constexpr uint32_t OFF_GB = 51456;     // this head's beta [64]
constexpr uint32_t OFF_GBE = 51712;    // this head's -beta e^G [64]
constexpr uint32_t SMEM_BYTES = 51968 + 1024;
constexpr uint32_t TM_COLS = 128;      // X (64 columns), then the 128-column products

__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, int* flag) {
  if (threadIdx.x == 0) *flag = mbar_wait_bounded(bar, parity) ? 1 : 0;
  __syncthreads();
  return *flag != 0;
}

__device__ __forceinline__ uint4 pack8(const float* v) {
  uint4 w;
  w.x = tc::pack2(v[0], v[1], (E*)nullptr);
  w.y = tc::pack2(v[2], v[3], (E*)nullptr);
  w.z = tc::pack2(v[4], v[5], (E*)nullptr);
  w.w = tc::pack2(v[6], v[7], (E*)nullptr);
  return w;
}

// ---- 16 x 16 block products of the solve on the warp-level tensor-core path
// (mma.sync m16n8k8, tf32 inputs, fp32 accumulation), each fp32 operand split
// into a tf32 head (rounded to nearest) and a tail (the exact remainder, which
// the tensor core reads truncated to tf32: within 2^-21 of the operand), with
// the three significant cross products kept (hh + ht + th), which keeps the
// products at fp32-level accuracy.
constexpr int ZP = 20;        // pitch (floats) of the B blocks of the solve
constexpr int ZB = 16 * ZP;   // floats per B block

__device__ __forceinline__ uint32_t tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// The A fragment of k-step k0 of X (16 x 16 at xp, pitch px floats; rows and
// xp 16-byte aligned): X[g][k0+t], X[g+8][k0+t], X[g][k0+t+4], X[g+8][k0+t+4]
// (g = lane / 4, t = lane % 4) in one ldmatrix.x4 — each 8 x 8 16-bit matrix
// of it is an 8 x 4 block of fp32, and lane L gives the row address of row
// L % 8 of block L / 8 — split into its tf32 head and tail.
__device__ __forceinline__ void a_frag(const float* xp, int px, int k0, uint32_t (&ah)[4],
                                       uint32_t (&al)[4]) {
  const int lane = threadIdx.x & 31, mi = lane >> 3;
  const float* rowp = xp + ((mi & 1) * 8 + (lane & 7)) * px + k0 + (mi >> 1) * 4;
  uint32_t r[4];
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(rowp)));
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float a = __uint_as_float(r[e]);
    ah[e] = tf32_rna(a);
    al[e] = __float_as_uint(a - __uint_as_float(ah[e]));
  }
}
// The B fragment Y[k0+t][n0+g], Y[k0+t+4][n0+g] (Y at yp, pitch py), split.
__device__ __forceinline__ void b_frag(const float* yp, int py, int k0, int n0, uint32_t (&bh)[2],
                                       uint32_t (&bl)[2]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const float bf[2] = {yp[(k0 + t) * py + n0 + g], yp[(k0 + t + 4) * py + n0 + g]};
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    bh[e] = tf32_rna(bf[e]);
    bl[e] = __float_as_uint(bf[e] - __uint_as_float(bh[e]));
  }
}
// A 16 x 16 block product on one warp: acc0 / acc1 (this warp's fragments of
// the two 16 x 8 halves: row g col 2t, 2t+1 and row g+8 col 2t, 2t+1) +=
// X (16 x 16 at xp, pitch px) * Y[:, 0..7] / Y[:, 8..15] (Y at yp, pitch py),
// the A fragments loaded and split once for both halves.
__device__ __forceinline__ void blk_mma3_pair(float (&acc0)[4], float (&acc1)[4], const float* xp,
                                              int px, const float* yp, int py) {
  float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    uint32_t ah[4], al[4], bh[2], bl[2], bh1[2], bl1[2];
    a_frag(xp, px, 8 * ks, ah, al);
    b_frag(yp, py, 8 * ks, 0, bh, bl);
    b_frag(yp, py, 8 * ks, 8, bh1, bl1);
    mma_tf32(c0, al, bh);
    mma_tf32(c1, al, bh1);
    mma_tf32(c0, ah, bl);
    mma_tf32(c1, ah, bl1);
    mma_tf32(acc0, ah, bh);
    mma_tf32(acc1, ah, bh1);
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    acc0[e] += c0[e];
    acc1[e] += c1[e];
  }
}
// store a fragment (scaled by s) into a 16 x 16 block at dp (pitch pd), columns n0 ..
__device__ __forceinline__ void blk_store(float* dp, int pd, int n0, const float (&acc)[4], float s) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  *reinterpret_cast<float2*>(dp + g * pd + n0 + 2 * t) = make_float2(s * acc[0], s * acc[1]);
  *reinterpret_cast<float2*>(dp + (g + 8) * pd + n0 + 2 * t) = make_float2(s * acc[2], s * acc[3]);
}

__global__ void __launch_bounds__(kThreads, 4)
intra_kernel(FwdParams p, const __grid_constant__ CUtensorMap tqk,
             const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t lbar, vbar0, vbar1, mbar;
  __shared__ uint32_t tmem_slot;
  __shared__ int flag;
  pdl_wait_then_release();
  int32_t* hdr = p.work.header();
  const int n_chunks = hdr[kPreChunks];
  const int h = (int)(blockIdx.x % (unsigned)p.Hv);   // heads of a chunk run next to each other
  const int gidx = (int)(blockIdx.x / (unsigned)p.Hv);
  if (gidx >= n_chunks) return;
  // the chunk's first packed row and valid tokens, as prep_kernel recorded them
  const int2 rec = reinterpret_cast<const int2*>(p.scr_c)[gidx];
  const int kh = h / R, r2 = h % R;
  const int Hv = p.Hv;
  const int n = rec.y;
  const int row0 = rec.x;
  const size_t orow = (size_t)row0 * Hv + h;  // (packed row, head) index of row 0
  const int tid = threadIdx.x;
  const uint32_t lane = (uint32_t)(tid & 96) << 16;  // TMEM lane quarter of this warp
  const int r128 = tid & 127;                        // TMEM row of this thread
  const int hf = tid >> 7;                           // column half of this thread
  const uint32_t sbase = smem_u32(sm);
  float* AT = reinterpret_cast<float*>(sm + OFF_AT);
  float* Z = reinterpret_cast<float*>(sm + OFF_Z);
  float* GT = reinterpret_cast<float*>(sm + OFF_GT);
  float* GH = reinterpret_cast<float*>(sm + OFF_GH);
  float* GB = reinterpret_cast<float*>(sm + OFF_GB);
  float* GBE = reinterpret_cast<float*>(sm + OFF_GBE);
  const int gc = 2 * r2;  // this head's G column in GT (beta at gc + 1)

  if (tid == 0) {
    mbar_init(&lbar, 1);
    mbar_init(&vbar0, 1);
    mbar_init(&vbar1, 1);
    mbar_init(&mbar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&lbar, 4u * BOX + 1024u);
    tma_load_2d(sm + OFF_QK, &tqk, kh * 2 * D, row0, &lbar);
    tma_load_2d(sm + OFF_QK + KB_STRIDE, &tqk, kh * 2 * D + 64, row0, &lbar);
    tma_load_2d(sm + OFF_QK + CH * 128, &tqk, kh * 2 * D + D, row0, &lbar);
    tma_load_2d(sm + OFF_QK + KB_STRIDE + CH * 128, &tqk, kh * 2 * D + D + 64, row0, &lbar);
    tma_load_2d(sm + OFF_GT, &tg, 4 * kh, row0, &lbar);
  }
  if (tid < 32) tc::tmem_alloc(&tmem_slot, TM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  bool ok = cta_wait(&lbar, 0, &flag);
  if (ok) {
    if (n < CH) {
      // rows past the sequence: zero q~/k~, gates frozen at the last token
      const int nz = CH - n;
      for (int t = tid; t < 2 * 2 * nz * 8; t += kThreads) {
        const int q = t & 7, rr = (t >> 3) % nz, part = (t >> 3) / nz;  // part: kb * 2 + (q|k)
        const int row = (part & 1) * CH + n + rr;
        *reinterpret_cast<uint4*>(sm + OFF_QK + (part >> 1) * KB_STRIDE +
                                  tc::sw128_offset(row, q * 8)) = make_uint4(0, 0, 0, 0);
      }
      for (int i = n + tid; i < CH; i += kThreads) {
        GT[i * 4 + gc] = GT[(n - 1) * 4 + gc];
        GT[i * 4 + gc + 1] = 0.f;
      }
      tc::fence_proxy_async_smem();
      __syncthreads();
    }
    if (tid == 0) {
      tc::fence_after_sync();
      tc::mma_tile(tmem, sbase + OFF_QK, KB_STRIDE, sbase + OFF_QK + CH * 128, KB_STRIDE, 2,
                   tc::idesc_f16_f32(128, 64), false);
      tc::commit(&mbar);
    }
    if (tid < CH) {
      const float g = GT[tid * 4 + gc], bt = GT[tid * 4 + gc + 1];
      GH[tid] = g * kLog2e;
      GB[tid] = bt;
      GBE[tid] = -bt * __expf(g);
    }
    ok = cta_wait(&mbar, 0, &flag);
  }
  float amax = 0.f;
  if (ok) {
    tc::fence_after_sync();
    // this thread's row of X (q~_i . k~_j for rows < 64, k~_i . k~_j above), 32 columns
    float xr[32];
    tc::tmem_ld32(tmem + lane + hf * 32, xr);
    tc::tmem_wait_ld();
    // the X product has read the q~ rows: v columns 64..127 come into q~ slot 1
    if (tid == 0) {
      mbar_arrive_expect_tx(&vbar1, BOX);
      tma_load_2d(sm + OFF_QK + KB_STRIDE, &tv, h * D + 64, row0, &vbar1);
    }
    {
      // row i of P (rows 0..63 of X) or of A (rows 64..127), this thread's 32
      // columns j as two 16-blocks; blocks right of row i's block are zero
      const bool prow = r128 < CH;
      const int i = r128 & 63, ib = i >> 4;
      // e^{G_i - G_j} beta_i = 2^{(G_i + ln beta_i) log2 e - G_j log2 e}: the
      // row's exponent offset once (beta_i for A, 1 for P; beta = 0 gives 0)
      const float Gi2 = GH[i] + (prow ? 0.f : lg2_approx(GT[i * 4 + gc + 1]));
      const int lim = prow ? i : i - 1;  // last kept column
      float val[32];
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const int jb = 2 * hf + blk;
        if (jb <= ib) {
          float g16[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 t = *reinterpret_cast<const float4*>(GH + 16 * jb + 4 * q);
            g16[4 * q] = t.x; g16[4 * q + 1] = t.y; g16[4 * q + 2] = t.z; g16[4 * q + 3] = t.w;
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j = 16 * jb + e;
            val[blk * 16 + e] = j <= lim ? xr[blk * 16 + e] * ex2_approx(Gi2 - g16[e]) : 0.f;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) val[blk * 16 + e] = 0.f;
        }
      }
      if (prow) {
        // |P_ij| <= |q~_i| |k~_j| <= d^{-1/2} (the decays are at most 1): P
        // needs no fp16 range check
        if (i < n) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__half*>(p.scr_p) +
                                                (orow + (size_t)i * Hv) * CH + hf * 32);
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) dst[g8] = pack8(val + g8 * 8);
        }
      } else {
        // (the solve and the operand tile read only blocks at or left of the diagonal)
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4)
          if (2 * hf + (j4 >> 2) <= ib)
            *reinterpret_cast<float4*>(AT + i * AP + hf * 32 + j4 * 4) =
                make_float4(val[j4 * 4], val[j4 * 4 + 1], val[j4 * 4 + 2], val[j4 * 4 + 3]);
      }
    }
    __syncthreads();
    // T = (I + A)^{-1}: diagonal 16 x 16 blocks, one column per thread, written
    // over the A blocks once every column is done
    {
      float col[16];
      const int b = tid >> 4, m = tid & 15;
      if (tid < CH) {
        const float* Ab = AT + (16 * b) * AP + 16 * b;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float a[16];
#pragma unroll
          for (int q = 0; q < (r + 3) / 4; ++q) {
            const float4 t = *reinterpret_cast<const float4*>(Ab + r * AP + 4 * q);
            a[4 * q] = t.x; a[4 * q + 1] = t.y; a[4 * q + 2] = t.z; a[4 * q + 3] = t.w;
          }
          float acc = r == m ? 1.f : 0.f;
#pragma unroll
          for (int j = 0; j < r; ++j) acc -= a[j] * col[j];
          col[r] = acc;
        }
      }
      __syncthreads();
      if (tid < CH) {
#pragma unroll
        for (int r = 0; r < 16; ++r) AT[(16 * b + r) * AP + 16 * b + m] = col[r];
      }
    }
    __syncthreads();
    // off-diagonal blocks: B_ij = T_ii A_ij for every i > j, then level by
    // level T_ij = -sum_{k=j}^{i-1} B_ik T_kj over A_ij (B block (i, j) at
    // Z + (i(i-1)/2 + j) * ZB); one warp per 16 x 16 block, the first level
    // by the warps that made its B blocks
    {
      const int warp = tid >> 5;
      if (warp < 6) {  // one warp per B block, both column halves
        const int bi = warp;
        const int i = bi < 1 ? 1 : (bi < 3 ? 2 : 3);
        const int j = bi - i * (i - 1) / 2;
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
        blk_mma3_pair(acc0, acc1, AT + (16 * i) * AP + 16 * i, AP, AT + (16 * i) * AP + 16 * j, AP);
        blk_store(Z + bi * ZB, ZP, 0, acc0, 1.f);
        blk_store(Z + bi * ZB, ZP, 8, acc1, 1.f);
        if (j == i - 1) {
          // the first level right away, from this warp's own B block:
          // T_{i,i-1} = -B_{i,i-1} T_{i-1,i-1} over A_{i,i-1} (read only by this warp)
          __syncwarp();
#pragma unroll
          for (int e = 0; e < 4; ++e) acc0[e] = acc1[e] = 0.f;
          blk_mma3_pair(acc0, acc1, Z + bi * ZB, ZP, AT + (16 * j) * AP + 16 * j, AP);
          blk_store(AT + (16 * i) * AP + 16 * j, AP, 0, acc0, -1.f);
          blk_store(AT + (16 * i) * AP + 16 * j, AP, 8, acc1, -1.f);
        }
      }
      __syncthreads();
      // the second level on warps 0 and 1; warp 0 goes on to the third, which
      // needs only its own second-level block and the first level
      auto level_block = [&](int i, int j) {
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
        for (int k = j; k < i; ++k)
          blk_mma3_pair(acc0, acc1, Z + (i * (i - 1) / 2 + k) * ZB, ZP, AT + (16 * k) * AP + 16 * j, AP);
        blk_store(AT + (16 * i) * AP + 16 * j, AP, 0, acc0, -1.f);
        blk_store(AT + (16 * i) * AP + 16 * j, AP, 8, acc1, -1.f);
      };
      if (warp < 2) level_block(warp + 2, warp);
      if (warp == 0) {
        __syncwarp();
        level_block(3, 0);
      }
      tc::fence_proxy_async_smem();  // the B blocks' slot goes back to TMA
      __syncthreads();
    }
    // the B blocks are consumed: v columns 0..63 come into q~ slot 0
    if (tid == 0) {
      mbar_arrive_expect_tx(&vbar0, BOX);
      tma_load_2d(sm + OFF_QK, &tv, h * D, row0, &vbar0);
    }
    // [-T diag(beta e^G) ; T diag(beta)] -> the MMAs' A tile, over the A/T
    // array once every T value is read (upper blocks of T are zero)
    {
      uint4 wtb[2], wtbe[2];
#pragma unroll
      for (int q2 = 0; q2 < 2; ++q2) {
        const int idx = tid + kThreads * q2;
        const int i = idx >> 3, c8 = idx & 7;
        float tb[8], tbe[8];
        const bool live = (c8 >> 1) <= (i >> 4);  // this 8-column group is in a block at or left of the diagonal
        const float4 b0 = *reinterpret_cast<const float4*>(GB + c8 * 8);
        const float4 b1 = *reinterpret_cast<const float4*>(GB + c8 * 8 + 4);
        const float4 e0 = *reinterpret_cast<const float4*>(GBE + c8 * 8);
        const float4 e1 = *reinterpret_cast<const float4*>(GBE + c8 * 8 + 4);
        const float bj[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        const float ej[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
        float4 t0 = make_float4(0.f, 0.f, 0.f, 0.f), t1 = t0;
        if (live) {
          t0 = *reinterpret_cast<const float4*>(AT + i * AP + c8 * 8);
          t1 = *reinterpret_cast<const float4*>(AT + i * AP + c8 * 8 + 4);
        }
        const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          tb[e] = tv[e] * bj[e];
          tbe[e] = tv[e] * ej[e];
        }
#pragma unroll
        for (int e = 0; e < 8; e += 2) amax = max_abs3(amax, tb[e], tb[e + 1]);
        wtb[q2] = pack8(tb);
        wtbe[q2] = pack8(tbe);
      }
      __syncthreads();
#pragma unroll
      for (int q2 = 0; q2 < 2; ++q2) {
        const int idx = tid + kThreads * q2;
        const int i = idx >> 3, c8 = idx & 7;
        *reinterpret_cast<uint4*>(sm + OFF_TT + tc::sw128_offset(i, c8 * 8)) = wtbe[q2];
        *reinterpret_cast<uint4*>(sm + OFF_TT + tc::sw128_offset(CH + i, c8 * 8)) = wtb[q2];
      }
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    // rows 0..63: -w = -T diag(beta e^G) k~ (k~ rows, MN-major), then wait for
    // it and for this head's v rows together
    if (tid == 0) {
      tc::fence_after_sync();
      tc::mma_op(tmem, tc::Opnd{sbase + OFF_TT, 0u, false},
                 tc::Opnd{sbase + OFF_QK + CH * 128, KB_STRIDE, true}, CH / 16,
                 tc::idesc_f16_f32(128, 128, false, true), false);
      tc::commit(&mbar);
      flag = (mbar_wait_bounded(&vbar1, 0) && mbar_wait_bounded(&vbar0, 0) &&
              mbar_wait_bounded(&mbar, 1)) ? 1 : 0;
    }
    __syncthreads();
    ok = flag != 0;
    if (ok && n < CH) {
      // v rows past the sequence -> 0 (made visible to the u product below)
      const int nz = CH - n;
      for (int t = tid; t < 2 * nz * 8; t += kThreads) {
        const int q = t & 7, rr = (t >> 3) % nz, bx = (t >> 3) / nz;
        *reinterpret_cast<uint4*>(sm + OFF_QK + bx * KB_STRIDE + tc::sw128_offset(n + rr, q * 8)) =
            make_uint4(0, 0, 0, 0);
      }
    }
  }
  // read out rows 0..63 (-w) or 64..127 (u) of the product in TMEM, 64 columns
  auto readout = [&](bool mine, void* base) {
    if (!mine) return;  // warp-uniform: TMEM lane quarters
    const int i = r128 & 63;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float vv[32];
      tc::tmem_ld32(tmem + lane + hf * 64 + hh * 32, vv);
      tc::tmem_wait_ld();
      float m4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 32; e += 2) m4[(e >> 1) & 3] = max_abs3(m4[(e >> 1) & 3], vv[e], vv[e + 1]);
      amax = fmaxf(amax, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
      if (i < n) {
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__half*>(base) +
                                              (orow + (size_t)i * Hv) * D + hf * 64 + hh * 32);
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8) dst[g8] = pack8(vv + g8 * 8);
      }
    }
  };
  if (ok) {
    tc::fence_after_sync();
    readout(r128 < CH, p.scr_w);
    tc::fence_proxy_async_smem();  // the zeroed v rows
    tc::fence_before_sync();
    __syncthreads();
    // rows 64..127: u = T diag(beta) v   (v rows in the q~ slots, MN-major)
    if (tid == 0) {
      tc::fence_after_sync();
      tc::mma_op(tmem, tc::Opnd{sbase + OFF_TT, 0u, false},
                 tc::Opnd{sbase + OFF_QK, KB_STRIDE, true}, CH / 16,
                 tc::idesc_f16_f32(128, 128, false, true), false);
      tc::commit(&mbar);
    }
    ok = cta_wait(&mbar, 0, &flag);
    if (ok) {
      tc::fence_after_sync();
      readout(r128 >= CH, p.scr_u);
    }
  }
  if (!ok && tid == 0) atomicOr((unsigned*)&hdr[kErr], GDN_FLAG_TIMEOUT);
  // w and u (and the operand tile) enter tensor-core operands in fp16
  if (!(amax <= kF16Max)) atomicOr((unsigned*)&hdr[kErr], GDN_FLAG_RANGE);
  tc::fence_before_sync();
  __syncthreads();
  if (tid < 32) tc::tmem_dealloc(tmem, TM_COLS);
}

}  // namespace

cudaError_t launch_intra(const FwdParams& p, const void* qk_map, const void* v_map,
                         const void* g_map, int max_chunks, cudaStream_t stream) {
  if (max_chunks <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(intra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_pdl(intra_kernel, dim3((unsigned)max_chunks * (unsigned)p.Hv), dim3(kThreads),
                    SMEM_BYTES, stream, p, *static_cast<const CUtensorMap*>(qk_map),
                    *static_cast<const CUtensorMap*>(v_map), *static_cast<const CUtensorMap*>(g_map));
}

}  // namespace gdn

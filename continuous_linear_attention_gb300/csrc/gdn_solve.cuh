// The unit lower-triangular solve of the chunked prefill, shared by the
// chunk-parallel kernels of both gate forms: T = (I + A)^{-1} for a strictly
// lower-triangular 64 x 64 fp32 matrix A (the chunk's A_ij = beta_i
// (decayed k_i . k_j), j < i), overwritten by T in place, in 16 x 16 blocks:
//   diagonal blocks T_ii = (I + A_ii)^{-1} by column substitution, one thread
//   per column (64 threads per matrix);
//   the six blocks below the diagonal as six chains of block products that
//   start from B_ij = T_ii A_ij, in four dependent product steps with two
//   barriers (offdiag_chains).
// The block products run on the warp-level tensor-core path (mma.sync
// m16n8k8, tf32 inputs, fp32 accumulation) with every fp32 operand split into
// a tf32 head (rounded to nearest) and a tail (the exact remainder, which the
// tensor core reads truncated to tf32: within 2^-21 of the operand), keeping
// the three significant cross products (hh + ht + th): fp32-level accuracy.
#pragma once

#include "gdn_ptx.cuh"

namespace gdn {
namespace solve {

constexpr int AP = 68;  // pitch (floats) of the fp32 A / T rows
constexpr int ZP = 20;  // pitch (floats) of the B blocks
constexpr int ZB = 16 * ZP;
constexpr int kZFloats = 6 * ZB;  // the six B blocks of one matrix

__device__ __forceinline__ uint32_t tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// A fragment of k-step k0 of a 16 x 16 block X (at xp, pitch px floats, rows
// 16-byte aligned) by one ldmatrix.x4 (each 8 x 8 16-bit matrix is an 8 x 4
// block of fp32), split into its tf32 head and tail.
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
// B fragment Y[k0+t][n0+g], Y[k0+t+4][n0+g] (Y at yp, pitch py), split.
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
// acc0 / acc1 (this warp's fragments of the two 16 x 8 halves of a 16 x 16
// block) += X (16 x 16 at xp) * Y[:, 0..7] / Y[:, 8..15] (Y at yp).
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
__device__ __forceinline__ void blk_store(float* dp, int pd, int n0, const float (&acc)[4],
                                          float s) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  *reinterpret_cast<float2*>(dp + g * pd + n0 + 2 * t) = make_float2(s * acc[0], s * acc[1]);
  *reinterpret_cast<float2*>(dp + (g + 8) * pd + n0 + 2 * t) =
      make_float2(s * acc[2], s * acc[3]);
}
// Column m of the inverse of the unit lower-triangular diagonal block at Ab
// (pitch AP; only the entries below its diagonal are read).
__device__ __forceinline__ void diag_col(const float* Ab, int m, float (&col)[16]) {
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
__device__ __forceinline__ void diag_col_store(float* Ab, int m, const float (&col)[16]) {
#pragma unroll
  for (int r = 0; r < 16; ++r) Ab[r * AP + m] = col[r];
}
// The off-diagonal blocks in four dependent product steps instead of eight:
// six chains c = (i, j), (1,0) (2,1) (3,2) (2,0) (3,1) (3,0), each first
// B_ij = T_ii A_ij (kept in Z block c for the other chains), then for the
// first three T_ij = -B_ij T_jj and for the others the partial sum
// P_ij = B_ij T_jj in registers; after a barrier T_20 = -(P_20 + B_21 T_10),
// T_31 = -(P_31 + B_32 T_21) and P_30 += B_31 T_10; after another
// T_30 = -(P_30 + B_32 T_20).  Chain c runs on warp c % NW of the NW warps
// (wl = this warp's index among them) and bar() is their barrier; A's
// diagonal blocks must already be inverted.  on_t(i, j, t0, t1) sees each
// block T_ij as this warp's fragments of its two 16 x 8 halves (blk_store's
// layout, signs applied).
template <int NW, typename Bar, typename OnT>
__device__ __forceinline__ void offdiag_chains(float* AT, float* Z, int wl, Bar bar, OnT on_t) {
  auto put = [&](int i, int j, float (&a0)[4], float (&a1)[4]) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      a0[e] = -a0[e];
      a1[e] = -a1[e];
    }
    blk_store(AT + (16 * i) * AP + 16 * j, AP, 0, a0, 1.f);
    blk_store(AT + (16 * i) * AP + 16 * j, AP, 8, a1, 1.f);
    on_t(i, j, a0, a1);
  };
  auto blk = [&](int i, int j) { return AT + (16 * i) * AP + 16 * j; };
  float p0[4] = {0.f, 0.f, 0.f, 0.f}, p1[4] = {0.f, 0.f, 0.f, 0.f};  // this warp's P (chains 3..5)
#pragma unroll 1
  for (int c = wl; c < 6; c += NW) {
    const int i = c == 0 ? 1 : (c == 1 || c == 3 ? 2 : 3);
    const int j = c == 0 || c == 3 || c == 5 ? 0 : (c == 1 || c == 4 ? 1 : 2);
    float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
    blk_mma3_pair(a0, a1, blk(i, i), AP, blk(i, j), AP);  // B_ij
    blk_store(Z + c * ZB, ZP, 0, a0, 1.f);
    blk_store(Z + c * ZB, ZP, 8, a1, 1.f);
    __syncwarp();
    float b0[4] = {0.f, 0.f, 0.f, 0.f}, b1[4] = {0.f, 0.f, 0.f, 0.f};
    blk_mma3_pair(b0, b1, Z + c * ZB, ZP, blk(j, j), AP);  // B_ij T_jj
    if (c < 3) {
      put(i, j, b0, b1);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        p0[e] = b0[e];
        p1[e] = b1[e];
      }
    }
  }
  bar();
  // chains 3, 4, 5: one more product each (Z blocks: 1 = B_21, 2 = B_32, 4 = B_31)
#pragma unroll 1
  for (int c = wl; c < 6; c += NW) {
    if (c < 3) continue;
    if (c == 3) {
      blk_mma3_pair(p0, p1, Z + 1 * ZB, ZP, blk(1, 0), AP);
      put(2, 0, p0, p1);
    } else if (c == 4) {
      blk_mma3_pair(p0, p1, Z + 2 * ZB, ZP, blk(2, 1), AP);
      put(3, 1, p0, p1);
    } else {
      blk_mma3_pair(p0, p1, Z + 4 * ZB, ZP, blk(1, 0), AP);
    }
  }
  bar();
  if (5 % NW == wl) {
    blk_mma3_pair(p0, p1, Z + 2 * ZB, ZP, blk(2, 0), AP);
    put(3, 0, p0, p1);
  }
}

}  // namespace solve
}  // namespace gdn

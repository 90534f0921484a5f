// tcgen05 (5th-generation tensor core) and TMEM helpers for sm_103a, written
// from the PTX ISA: shared-memory matrix descriptors, the kind::f16
// instruction descriptor, MMA issue/commit, TMEM allocation and loads/stores.
//
// Operand convention used throughout: every MMA operand is a 16-bit float
// matrix (fp16 or bf16, both operands of one MMA the same type) in shared
// memory, K-major, in the 128-byte swizzled canonical layout.  A tile
// of R rows x 64 K-elements (one "K-block", 128 bytes per row) is stored as
// R/8 groups of 8 rows x 128 bytes (1024 bytes per group, groups contiguous);
// inside a group, the 16-byte chunk j of row r sits at chunk position
// j ^ (r % 8).  Tiles start on 1024-byte boundaries.  A K extent of 128 is two
// such K-block tiles placed one after the other.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gdn_ptx.cuh"

namespace gdn {
namespace tc {

// Byte offset of element (row, k) (k < 64) inside a swizzled K-block tile.
__device__ __forceinline__ uint32_t sw128_offset(int row, int k) {
  const uint32_t chunk = (uint32_t)(k >> 3) ^ (uint32_t)(row & 7);
  return (uint32_t)(row >> 3) * 1024u + (uint32_t)(row & 7) * 128u + chunk * 16u +
         (uint32_t)(k & 7) * 2u;
}

__device__ __forceinline__ uint32_t pack2(float a, float b, __nv_bfloat16*) {
  __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&p);
}
__device__ __forceinline__ uint32_t pack2(float a, float b, __half*) {
  __half2 p = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&p);
}

// Writes 8 consecutive K-elements (k0 % 8 == 0) of one row as one 16-byte
// store, converted to the 16-bit type E (round to nearest even).
template <typename E = __nv_bfloat16>
__device__ __forceinline__ void sw128_store8(unsigned char* tile, int row, int k0,
                                             const float* v) {
  uint4 w;
  w.x = pack2(v[0], v[1], (E*)nullptr);
  w.y = pack2(v[2], v[3], (E*)nullptr);
  w.z = pack2(v[4], v[5], (E*)nullptr);
  w.w = pack2(v[6], v[7], (E*)nullptr);
  *reinterpret_cast<uint4*>(tile + sw128_offset(row, k0)) = w;
}

template <typename E = __nv_bfloat16>
__device__ __forceinline__ void sw128_store1(unsigned char* tile, int row, int k, float v);
template <>
__device__ __forceinline__ void sw128_store1<__nv_bfloat16>(unsigned char* tile, int row, int k,
                                                            float v) {
  *reinterpret_cast<__nv_bfloat16*>(tile + sw128_offset(row, k)) = __float2bfloat16_rn(v);
}
template <>
__device__ __forceinline__ void sw128_store1<__half>(unsigned char* tile, int row, int k, float v) {
  *reinterpret_cast<__half*>(tile + sw128_offset(row, k)) = __float2half_rn(v);
}

// Shared-memory matrix descriptor (sm_100 family): start address >> 4 in bits
// 0-13, leading byte offset >> 4 in 16-29 (unused for swizzled K-major), stride
// byte offset >> 4 in 32-45 (1024: distance between 8-row groups), version 1
// in bits 46-47, layout type in 61-63 (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16u >> 4) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Descriptor of an MN-major 128-byte swizzled tile: each 128-byte row holds
// 64 consecutive M (or N) elements of one K index, rows of 8 consecutive K
// indices form a 1024-byte swizzle group (stride byte offset 1024), and the
// next 64 M/N elements sit `mn_stride` bytes further (leading byte offset).
// A 2-D TMA box of [K rows][64 columns] with 128-byte swizzle lands in exactly
// this layout, so a token-major tile is an MN-major operand as loaded.
__device__ __forceinline__ uint64_t sw128_desc_mn(uint32_t smem_addr, uint32_t mn_stride) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((mn_stride & 0x3FFFFu) >> 4) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1),
// A and B bf16 (bits 7-9 = 1, 10-12 = 1) or fp16 (both 0), A / B MN-major
// when bit 15 / 16 is set (K-major otherwise), N >> 3 in bits 17-22, M >> 4 in
// bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn = false,
                                                      bool b_mn = false) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool a_mn = false,
                                                     bool b_mn = false) {
  return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// One MMA operand in shared memory.  K-major: `addr` is the first K-block
// tile, `stride` the byte distance between K-blocks of 64.  MN-major: `addr`
// is the first row (K index), `stride` the distance between 64-wide M/N
// blocks.
struct Opnd {
  uint32_t addr, stride;
  bool mn;
};

// Descriptor of K step s (elements 16s .. 16s+15) of an operand.
__device__ __forceinline__ uint64_t opnd_desc(const Opnd& o, int s) {
  return o.mn ? sw128_desc_mn(o.addr + (uint32_t)s * 2048u, o.stride)
              : sw128_desc(o.addr + (uint32_t)(s >> 2) * o.stride + (uint32_t)(s & 3) * 32u);
}

// D[tmem] (+)= A[smem] * B[smem]^T for one K=16 step (cta_group::1).
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (M=128 rows) (+)= A * B^T over K = 64 * kblocks, A and B K-major swizzled
// tiles with the given byte distance between their K-blocks.
__device__ __forceinline__ void mma_tile(uint32_t d_tmem, uint32_t a_smem, uint32_t a_kb_stride,
                                         uint32_t b_smem, uint32_t b_kb_stride, int kblocks,
                                         uint32_t idesc, bool accumulate) {
  for (int kb = 0; kb < kblocks; ++kb) {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const uint64_t ad = sw128_desc(a_smem + kb * a_kb_stride + ks * 32);
      const uint64_t bd = sw128_desc(b_smem + kb * b_kb_stride + ks * 32);
      mma_bf16(d_tmem, ad, bd, idesc, (accumulate || kb > 0 || ks > 0) ? 1u : 0u);
    }
  }
}

// D (M=128 rows) (+)= A * B^T over K = 16 * ksteps for operands of either
// major-ness; idesc must carry the matching MN-major bits.
__device__ __forceinline__ void mma_op(uint32_t d_tmem, const Opnd& a, const Opnd& b, int ksteps,
                                       uint32_t idesc, bool accumulate) {
#pragma unroll 4
  for (int s = 0; s < ksteps; ++s)
    mma_bf16(d_tmem, opnd_desc(a, s), opnd_desc(b, s), idesc, (accumulate || s > 0) ? 1u : 0u);
}

// D[tmem] (+)= A[tmem] * B[smem]^T for one K=16 step (cta_group::1).  A sits
// in tensor memory: row m in lane m, its 16 K-elements in 8 consecutive
// 32-bit columns, two per column (the lower K index in the low half).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (M=128 rows) (+)= A * B^T over K = 16 * ksteps with A in tensor memory
// from column a_tmem on (K-major by construction: the A bit of idesc is 0).
__device__ __forceinline__ void mma_op_ts(uint32_t d_tmem, uint32_t a_tmem, const Opnd& b,
                                          int ksteps, uint32_t idesc, bool accumulate) {
#pragma unroll 4
  for (int s = 0; s < ksteps; ++s)
    mma_ts(d_tmem, a_tmem + 8u * (uint32_t)s, opnd_desc(b, s), idesc,
           (accumulate || s > 0) ? 1u : 0u);
}

// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Generic-proxy shared-memory writes -> visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMEM allocation by one full warp; the base address lands in *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols)
               : "memory");
}

// 32 consecutive TMEM columns of this thread's lane (warp w reads lanes
// 32w..32w+31; taddr must carry that lane base in bits 16-31).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  uint32_t r[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 16 consecutive TMEM columns of this thread's lane, raw 32-bit words (e.g.
// two packed 16-bit operand elements each).
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace tc
}  // namespace gdn

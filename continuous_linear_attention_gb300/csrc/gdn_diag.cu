// Diagnostic tensor-core GEMM (see include/gdn_diag.h): exercises the shared
// tile layout, descriptors, MMA issue/commit (A from shared or from tensor
// memory) and TMEM load/store helpers of gdn_tc.cuh on plain matrices.
#include <type_traits>

#include "gdn.h"
#include "gdn_diag.h"
#include "gdn_internal.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int kM = 128;

// Shared tiles: A at byte 0, B at byte kBOff of the 1024-aligned region.
// K-major tiles are K/64 K-blocks of 128 (A) or N (B) rows; MN-major tiles
// (K = 64 only) are 64-wide M/N blocks of K rows, kMnStride bytes apart.
constexpr uint32_t kBOff = 80 * 1024;
constexpr uint32_t kMnStride = 64 * 128;
constexpr uint32_t kSmem = 160 * 1024 + 1024;
// tensor memory: D in columns 0..N-1, an A staged in tensor memory from 256 on
constexpr uint32_t kATmem = 256;

template <typename E>
__global__ void __launch_bounds__(128, 1)
diag_umma_kernel(const __nv_bfloat16* __restrict__ A, const __nv_bfloat16* __restrict__ B,
                 const float* __restrict__ Cin, float* __restrict__ D, int N, int K, int a_mn,
                 int b_mn, unsigned* err) {
  extern __shared__ unsigned char smem_raw[];
  // swizzled tiles need 1024-byte alignment: round the dynamic base up
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* a_tile = smem;
  unsigned char* b_tile = smem + kBOff;
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int ok;
  const int tid = threadIdx.x;
  const uint32_t a_kb = kM * 128, b_kb = (uint32_t)N * 128;
  // element (row r, k) of an operand with `rows` rows -> byte offset in its tile
  auto off = [&](bool mn, uint32_t kb_stride, int r, int k) -> uint32_t {
    return mn ? (uint32_t)(r >> 6) * kMnStride + tc::sw128_offset(k, r & 63)
              : (uint32_t)(k >> 6) * kb_stride + tc::sw128_offset(r, k & 63);
  };
  for (int idx = tid; a_mn != 2 && idx < kM * K; idx += 128) {
    const int r = idx / K, k = idx % K;
    const float v = __bfloat162float(A[idx]);
    unsigned char* dst = a_tile + off(a_mn != 0, a_kb, r, k);
    if (std::is_same<E, __half>::value) *reinterpret_cast<__half*>(dst) = __float2half_rn(v);
    else *reinterpret_cast<__nv_bfloat16*>(dst) = __float2bfloat16_rn(v);
  }
  for (int idx = tid; idx < N * K; idx += 128) {
    const int r = idx / K, k = idx % K;
    const float v = __bfloat162float(B[idx]);
    unsigned char* dst = b_tile + off(b_mn != 0, b_kb, r, k);
    if (std::is_same<E, __half>::value) *reinterpret_cast<__half*>(dst) = __float2half_rn(v);
    else *reinterpret_cast<__nv_bfloat16*>(dst) = __float2bfloat16_rn(v);
  }
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  if (tid < 32) tc::tmem_alloc(&tmem_slot, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  const uint32_t lane_base = (uint32_t)(tid & ~31) << 16;
  if (Cin) {
    for (int c0 = 0; c0 < N; c0 += 32) {
      float v[32];
      for (int j = 0; j < 32; ++j) v[j] = Cin[(size_t)tid * N + c0 + j];
      tc::tmem_st32(tmem + lane_base + c0, v);
    }
    tc::tmem_wait_st();
  }
  if (a_mn == 2) {
    // A row tid -> lane tid, columns kATmem.., K-elements 2c and 2c+1 in column c
    for (int c0 = 0; c0 < K / 2; c0 += 16) {
      uint32_t w[16];
      for (int j = 0; j < 16; ++j) {
        const float lo = __bfloat162float(A[(size_t)tid * K + 2 * (c0 + j)]);
        const float hi = __bfloat162float(A[(size_t)tid * K + 2 * (c0 + j) + 1]);
        w[j] = tc::pack2(lo, hi, (E*)nullptr);
      }
      tc::tmem_st16u(tmem + lane_base + kATmem + c0, w);
    }
    tc::tmem_wait_st();
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    tc::fence_after_sync();
    constexpr bool kF16 = std::is_same<E, __half>::value;
    const tc::Opnd a{smem_u32(a_tile), a_mn ? kMnStride : a_kb, a_mn == 1};
    const tc::Opnd b{smem_u32(b_tile), b_mn ? kMnStride : b_kb, b_mn != 0};
    const uint32_t idesc = kF16 ? tc::idesc_f16_f32(kM, N, a_mn == 1, b_mn != 0)
                                : tc::idesc_bf16_f32(kM, N, a_mn == 1, b_mn != 0);
    if (a_mn == 2) tc::mma_op_ts(tmem, tmem + kATmem, b, K / 16, idesc, Cin != nullptr);
    else tc::mma_op(tmem, a, b, K / 16, idesc, Cin != nullptr);
    tc::commit(&bar);
    ok = mbar_wait_bounded(&bar, 0) ? 1 : 0;
  }
  __syncthreads();
  tc::fence_after_sync();
  if (ok) {
    for (int c0 = 0; c0 < N; c0 += 32) {
      float v[32];
      tc::tmem_ld32(tmem + lane_base + c0, v);
      tc::tmem_wait_ld();
      for (int j = 0; j < 32; ++j) D[(size_t)tid * N + c0 + j] = v[j];
    }
  } else if (tid == 0) {
    atomicOr(err, GDN_FLAG_TIMEOUT);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (tid < 32) tc::tmem_dealloc(tmem, 512);
}

// Issue cost of tcgen05.mma: one thread issues `reps` MMAs (M = 128, K = 16,
// the given N; A from shared or tensor memory; all into one accumulator,
// operands zero) back to back with precomputed descriptors, then commits.
// out[0] = clock cycles spent issuing, out[1] = cycles until the commit is
// observed, out[2] = 1 if it was.
__global__ void __launch_bounds__(128, 1)
diag_mma_timing_kernel(unsigned long long* out, int N, int a_tmem, int reps) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x;
  // A: 128 x 64 K-major (16 KiB) at 0; B: up to 256 x 64 K-major at 16 KiB
  for (int i = tid; i < (48 * 1024) / 16; i += 128)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  if (tid < 32) tc::tmem_alloc(&tmem_slot, 512);
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  {
    // a tensor-memory A of zeros in columns kATmem .. kATmem + 15
    uint32_t z[16];
    for (int j = 0; j < 16; ++j) z[j] = 0u;
    tc::tmem_st16u(tmem + ((uint32_t)(tid & ~31) << 16) + kATmem, z);
    tc::tmem_wait_st();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid == 0) {
    const uint32_t sb = smem_u32(smem);
    const uint32_t idesc = tc::idesc_f16_f32(kM, N);
    uint64_t ad[4], bd[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      ad[s] = tc::opnd_desc(tc::Opnd{sb, 16384u, false}, s);
      bd[s] = tc::opnd_desc(tc::Opnd{sb + 16384u, 32768u, false}, s);
    }
    const unsigned long long t0 = clock64();
    for (int r = 0; r < reps; r += 8) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (a_tmem) tc::mma_ts(tmem, tmem + kATmem + 8 * (u & 1), bd[u & 3], idesc, 1u);
        else tc::mma_bf16(tmem, ad[u & 3], bd[u & 3], idesc, 1u);
      }
    }
    const unsigned long long t1 = clock64();
    tc::commit(&bar);
    const bool ok = mbar_wait_bounded(&bar, 0);
    const unsigned long long t2 = clock64();
    out[0] = t1 - t0;
    out[1] = t2 - t0;
    out[2] = ok ? 1ull : 0ull;
  }
  tc::fence_before_sync();
  __syncthreads();
  if (tid < 32) tc::tmem_dealloc(tmem, 512);
}

}  // namespace
}  // namespace gdn

extern "C" int gdn_diag_umma_issue_timing(int N, int a_tmem, int reps, unsigned long long* out,
                                          void* stream) {
  if (!out) return GDN_ERR_NULL;
  if ((N != 16 && N != 32 && N != 64 && N != 128 && N != 256) || (a_tmem != 0 && a_tmem != 1) ||
      reps < 8 || reps > 4096 || reps % 8 != 0)
    return GDN_ERR_DIMS;
  if ((uintptr_t)out & 7) return GDN_ERR_ALIGN;
  const int smem = 49 * 1024;
  if (cudaFuncSetAttribute(gdn::diag_mma_timing_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return GDN_ERR_CUDA;
  gdn::diag_mma_timing_kernel<<<1, 128, smem, (cudaStream_t)stream>>>(out, N, a_tmem, reps);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" int gdn_diag_umma_gemm_ex(const void* A, const void* B, const float* C, float* D,
                                     int N, int K, int operand_f16, int a_mn, int b_mn,
                                     void* stream) {
  if (!A || !B || !D) return GDN_ERR_NULL;
  if ((N != 64 && N != 128 && N != 192 && N != 256) || (K != 64 && K != 128))
    return GDN_ERR_DIMS;
  if (a_mn < 0 || a_mn > 2 || b_mn < 0 || b_mn > 1) return GDN_ERR_DIMS;
  if ((a_mn == 1 || b_mn) && K != 64) return GDN_ERR_DIMS;
  if (((uintptr_t)A & 15) || ((uintptr_t)B & 15) || ((uintptr_t)D & 15) || ((uintptr_t)C & 15))
    return GDN_ERR_ALIGN;
  static unsigned* err = nullptr;
  if (!err && cudaMalloc((void**)&err, sizeof(unsigned)) != cudaSuccess) return GDN_ERR_CUDA;
  const int smem = (int)gdn::kSmem;
  if (operand_f16) {
    if (cudaFuncSetAttribute(gdn::diag_umma_kernel<__half>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return GDN_ERR_CUDA;
    gdn::diag_umma_kernel<__half><<<1, 128, smem, (cudaStream_t)stream>>>(
        (const __nv_bfloat16*)A, (const __nv_bfloat16*)B, C, D, N, K, a_mn, b_mn, err);
  } else {
    if (cudaFuncSetAttribute(gdn::diag_umma_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return GDN_ERR_CUDA;
    gdn::diag_umma_kernel<__nv_bfloat16><<<1, 128, smem, (cudaStream_t)stream>>>(
        (const __nv_bfloat16*)A, (const __nv_bfloat16*)B, C, D, N, K, a_mn, b_mn, err);
  }
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" int gdn_diag_umma_gemm(const void* A, const void* B, const float* C, float* D, int N,
                                  int K, int operand_f16, void* stream) {
  return gdn_diag_umma_gemm_ex(A, B, C, D, N, K, operand_f16, 0, 0, stream);
}

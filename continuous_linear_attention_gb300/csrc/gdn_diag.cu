// Diagnostic tensor-core GEMM (see include/gdn_diag.h): exercises the shared
// tile layout, descriptors, MMA issue/commit and TMEM load/store helpers of
// gdn_tc.cuh on plain matrices.
#include <type_traits>

#include "gdn.h"
#include "gdn_diag.h"
#include "gdn_internal.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int kM = 128;

template <typename E>
__global__ void __launch_bounds__(128, 1)
diag_umma_kernel(const __nv_bfloat16* __restrict__ A, const __nv_bfloat16* __restrict__ B,
                 const float* __restrict__ Cin, float* __restrict__ D, int N, int K,
                 unsigned* err) {
  extern __shared__ unsigned char smem_raw[];
  // swizzled tiles need 1024-byte alignment: round the dynamic base up
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  // A tile: K/64 K-blocks of 128 rows (16 KiB each); B tile: K/64 K-blocks of N rows
  unsigned char* a_tile = smem;
  unsigned char* b_tile = smem + (size_t)(K / 64) * kM * 128;
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int ok;
  const int tid = threadIdx.x;
  const int kblocks = K / 64;
  const uint32_t a_kb = kM * 128, b_kb = (uint32_t)N * 128;
  for (int kb = 0; kb < kblocks; ++kb) {
    for (int k0 = 0; k0 < 64; k0 += 8) {
      float v[8];
      for (int j = 0; j < 8; ++j) v[j] = __bfloat162float(A[(size_t)tid * K + kb * 64 + k0 + j]);
      tc::sw128_store8<E>(a_tile + kb * a_kb, tid, k0, v);
      for (int r = tid; r < N; r += 128) {
        for (int j = 0; j < 8; ++j) v[j] = __bfloat162float(B[(size_t)r * K + kb * 64 + k0 + j]);
        tc::sw128_store8<E>(b_tile + kb * b_kb, r, k0, v);
      }
    }
  }
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  if (tid < 32) tc::tmem_alloc(&tmem_slot, 256);
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
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    tc::fence_after_sync();
    constexpr bool kF16 = std::is_same<E, __half>::value;
    tc::mma_tile(tmem, smem_u32(a_tile), a_kb, smem_u32(b_tile), b_kb, kblocks,
                 kF16 ? tc::idesc_f16_f32(kM, N) : tc::idesc_bf16_f32(kM, N), Cin != nullptr);
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
  if (tid < 32) tc::tmem_dealloc(tmem, 256);
}

}  // namespace
}  // namespace gdn

extern "C" int gdn_diag_umma_gemm(const void* A, const void* B, const float* C, float* D, int N,
                                  int K, int operand_f16, void* stream) {
  if (!A || !B || !D) return GDN_ERR_NULL;
  if ((N != 64 && N != 128 && N != 192 && N != 256) || (K != 64 && K != 128))
    return GDN_ERR_DIMS;
  if (((uintptr_t)A & 15) || ((uintptr_t)B & 15) || ((uintptr_t)D & 15) || ((uintptr_t)C & 15))
    return GDN_ERR_ALIGN;
  static unsigned* err = nullptr;
  if (!err && cudaMalloc((void**)&err, sizeof(unsigned)) != cudaSuccess) return GDN_ERR_CUDA;
  const size_t smem = (size_t)(K / 64) * (128 + N) * 128 + 1024;
  if (operand_f16) {
    if (cudaFuncSetAttribute(gdn::diag_umma_kernel<__half>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return GDN_ERR_CUDA;
    gdn::diag_umma_kernel<__half><<<1, 128, smem, (cudaStream_t)stream>>>(
        (const __nv_bfloat16*)A, (const __nv_bfloat16*)B, C, D, N, K, err);
  } else {
    if (cudaFuncSetAttribute(gdn::diag_umma_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return GDN_ERR_CUDA;
    gdn::diag_umma_kernel<__nv_bfloat16><<<1, 128, smem, (cudaStream_t)stream>>>(
        (const __nv_bfloat16*)A, (const __nv_bfloat16*)B, C, D, N, K, err);
  }
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

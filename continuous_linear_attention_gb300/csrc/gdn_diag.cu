// Diagnostic entry points (see include/gdn_diag.h): a tensor-core GEMM that
// exercises the shared tile layout, descriptors, MMA issue/commit (A from
// shared or from tensor memory) and TMEM load/store helpers of gdn_tc.cuh on
// plain matrices, and a wait that must run out, which checks the bounded-wait
// path that reports GDN_FLAG_TIMEOUT.
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

// The bounded wait every kernel of the library uses, run where it must give
// up: thread 0 waits on an mbarrier that nothing arrives on, with no bulk copy
// and no MMA in flight, and raises GDN_FLAG_TIMEOUT in *flags when the wait
// returns unfinished, exactly as the forward kernels report a timeout.
__global__ void __launch_bounds__(32, 1) diag_wait_timeout_kernel(unsigned* flags) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait_bounded(&bar, 0)) atomicOr(flags, GDN_FLAG_TIMEOUT);
  }
}

}  // namespace
}  // namespace gdn

extern "C" int gdn_diag_wait_timeout(uint32_t* flags, void* stream) {
  if (!flags) return GDN_ERR_NULL;
  if ((uintptr_t)flags & 3) return GDN_ERR_ALIGN;
  gdn::diag_wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(
      reinterpret_cast<unsigned*>(flags));
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

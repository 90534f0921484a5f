/*
 * gdn_diag.h -- diagnostic entry points of libgdn, outside the forward path.
 *
 * gdn_diag_umma_gemm runs the tensor-core building blocks of the chunked
 * prefill kernels on plain matrices, so a test can check them against a
 * library GEMM: one CTA stages A and B into 128-byte-swizzled K-major shared
 * tiles, optionally preloads C into tensor memory with tcgen05.st, issues
 * tcgen05.mma (kind::f16, bf16 inputs, fp32 accumulator in tensor memory) and
 * reads the result back with tcgen05.ld:
 *     D[128][N] = (C ? C : 0) + A[128][K] * B[N][K]^T
 * A, B: bf16 row-major device arrays; C, D: fp32 row-major device arrays
 * (C may be NULL).  operand_f16 != 0 converts A and B to fp16 tiles and runs
 * the fp16 form of the MMA (the prefill kernels' operand type), else bf16.
 * N in {64, 128, 192, 256}, K in {64, 128}.  Returns GDN_OK
 * or GDN_ERR_NULL / GDN_ERR_DIMS / GDN_ERR_ALIGN / GDN_ERR_CUDA (nothing
 * launched on error).  Stream-ordered, no synchronisation.
 *
 * gdn_diag_umma_gemm_ex is the same GEMM with a choice of operand layout:
 * a_mn / b_mn != 0 stage A / B MN-major (each 128-byte row holds 64
 * consecutive M / N elements of one K index, the layout a 2-D TMA box of a
 * token-major matrix lands in) and set the matching instruction-descriptor
 * bits.  MN-major operands need K == 64 (GDN_ERR_DIMS otherwise).
 * a_mn == 2 instead places A in tensor memory (row m in lane m, two 16-bit
 * K-elements per 32-bit column, the lower K index in the low half) and issues
 * the MMA form that reads A from there; any K of the list above.  a_mn outside
 * 0..2 or b_mn outside 0..1: GDN_ERR_DIMS.  (Reference for the chunked
 * kernels' design: tcgen05, kind::f16, cta_group::1, from the PTX ISA.)
 *
 * gdn_diag_wait_timeout checks the time-out path of the library's bounded
 * waits without faulting or hanging anything: one thread waits on an mbarrier
 * that nothing arrives on (no bulk copy, no MMA in flight) with the same
 * bounded wait the forward kernels use (about 2 s), and when that wait gives
 * up it ORs GDN_FLAG_TIMEOUT into the device word *flags, as the forward
 * kernels do into a layer's error word.  flags: device uint32, 4-byte
 * aligned.  Returns GDN_OK or GDN_ERR_NULL / GDN_ERR_ALIGN / GDN_ERR_CUDA.
 * Stream-ordered; the kernel ends by itself after the limit and leaves the
 * context usable.
 */
#ifndef GDN_DIAG_H_
#define GDN_DIAG_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int gdn_diag_umma_gemm(const void* A, const void* B, const float* C, float* D, int N, int K,
                       int operand_f16, void* stream);
int gdn_diag_umma_gemm_ex(const void* A, const void* B, const float* C, float* D, int N, int K,
                          int operand_f16, int a_mn, int b_mn, void* stream);
int gdn_diag_wait_timeout(uint32_t* flags, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_DIAG_H_ */

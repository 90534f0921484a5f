/*
 * gdn_diag.h -- diagnostic entry point of libgdn, outside the forward path.
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
 * 0..2 or b_mn outside 0..1: GDN_ERR_DIMS.
 *
 * gdn_diag_umma_issue_timing measures what one tcgen05.mma costs the thread
 * that issues it: one CTA, one thread issues `reps` MMAs (kind::f16, M = 128,
 * K = 16, the given N; A from shared memory, or from tensor memory when
 * a_tmem != 0; zero operands, one fp32 accumulator) with precomputed
 * descriptors, commits, and waits (bounded) for the commit.  It writes three
 * unsigned 64-bit values to the device array `out`: SM clock cycles spent
 * issuing, cycles until the commit was observed, and 1 if it was (0 on
 * timeout).  N in {16, 32, 64, 128, 256}, a_tmem in {0, 1}, reps a multiple
 * of 8 in [8, 4096]; `out` 8-byte aligned.  Returns GDN_OK or GDN_ERR_NULL /
 * GDN_ERR_DIMS / GDN_ERR_ALIGN / GDN_ERR_CUDA.  Stream-ordered, no
 * synchronisation.  (Reference for the chunked kernels' design: tcgen05,
 * kind::f16, cta_group::1, from the PTX ISA.)
 */
#ifndef GDN_DIAG_H_
#define GDN_DIAG_H_

#ifdef __cplusplus
extern "C" {
#endif

int gdn_diag_umma_gemm(const void* A, const void* B, const float* C, float* D, int N, int K,
                       int operand_f16, void* stream);
int gdn_diag_umma_gemm_ex(const void* A, const void* B, const float* C, float* D, int N, int K,
                          int operand_f16, int a_mn, int b_mn, void* stream);
int gdn_diag_umma_issue_timing(int N, int a_tmem, int reps, unsigned long long* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_DIAG_H_ */

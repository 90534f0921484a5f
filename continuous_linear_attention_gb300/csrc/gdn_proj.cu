// The dense neighbours of the layer forward: the input projection in front of
// it and the gated RMS norm + output projection behind it (a hybrid model's
// gated-delta-net layer: hidden -> [q | k | v | z | b | a] -> conv + gated
// delta rule -> RMSNorm(o) * silu(z) -> out_proj).
//
// gemm_kernel computes, for up to four groups g sharing one A operand,
//   C_g[M][N_g] = A[M][K] B_g[N_g][K]^T      (bf16 in, fp32 accumulate, bf16 out)
// with A and every B_g row-major (K contiguous: both K-major MMA operands), on
// the 5th-generation tensor cores: persistent CTAs (one per SM) walk the
// output tiles of 128 rows x 256 columns; warp 0 streams 64-wide K-blocks of A
// and B_g into a 4-stage shared-memory ring with 2-D TMA (128-byte swizzle),
// warp 1 issues tcgen05.mma (M = 128, N = 256, K = 16) into one of two fp32
// accumulators in tensor memory, and warps 2-5 read the other accumulator
// out (tcgen05.ld), convert to bf16 and store it through a per-warp
// shared-memory transpose so that every global store writes whole 64-byte row
// segments.  Rows or columns past M or N_g read as zero (TMA fill) and are not
// stored.
//
// gated_norm_kernel: per token and v-head, o' = o / sqrt(mean(o^2) + eps) *
// w * silu(z) (one warp per (token, head)), the A operand of the output
// projection.
#include <cuda.h>

#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStagesG = 4;
constexpr uint32_t A_BYTES = BM * BK * 2;  // 16 KiB
constexpr uint32_t B_BYTES = BN * BK * 2;  // 32 KiB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int kEpiWarps = 4;
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t EPI_BYTES = 32 * 64;  // per epilogue warp: 32 rows x 32 bf16
constexpr uint32_t OFF_EPI = kStagesG * STAGE_BYTES;
constexpr uint32_t GEMM_SMEM = OFF_EPI + kEpiWarps * EPI_BYTES + 1024;
constexpr uint32_t kAccCols = BN;  // one fp32 accumulator
static_assert(GEMM_SMEM <= 227 * 1024, "shared memory of one CTA");

struct GemmGroup {
  void* C;     // [M][N] bf16, row pitch ldc elements
  int N, ldc;
  int tiles_n;  // ceil(N / BN)
};
struct GemmParams {
  int M, K, n_groups, tiles_m, total_tiles;
  GemmGroup g[4];
  unsigned* flags;  // optional device word: GDN_FLAG_TIMEOUT
};

// tile t -> (group, m-tile, n-tile): groups in order, inside a group the
// n-tiles of one m-tile next to each other.  The CTAs working at one time
// then share a few 128-row bands of A, read from DRAM once, and walk all of
// B_g, which stays in L2 (the layer's weight matrices are 17-34 MB, its A
// operands 65-130 MB); the other order re-reads A once per n-tile.
__device__ __forceinline__ void tile_coords(const GemmParams& p, int t, int& g, int& mt, int& nt) {
  g = 0;
  while (g < p.n_groups - 1 && t >= p.tiles_m * p.g[g].tiles_n) {
    t -= p.tiles_m * p.g[g].tiles_n;
    ++g;
  }
  mt = t / p.g[g].tiles_n;
  nt = t % p.g[g].tiles_n;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_kernel(GemmParams p, const __grid_constant__ CUtensorMap ta,
            const __grid_constant__ CUtensorMap tb0, const __grid_constant__ CUtensorMap tb1,
            const __grid_constant__ CUtensorMap tb2, const __grid_constant__ CUtensorMap tb3) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t full[kStagesG], empty[kStagesG], acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < kStagesG; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiWarps);
    }
    fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc(&tmem_slot, 2 * kAccCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  const int kblocks = (p.K + BK - 1) / BK;  // a partial last K-block reads zeros
  bool dead = false;

  if (warp == 0) {
    // ================= TMA producer =================
    if (tid == 0) {
      const CUtensorMap* tbs[4] = {&tb0, &tb1, &tb2, &tb3};
      int it = 0;
      for (int t = blockIdx.x; t < p.total_tiles && !dead; t += gridDim.x) {
        int g, mt, nt;
        tile_coords(p, t, g, mt, nt);
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % kStagesG;
          if (it >= kStagesG && !mbar_wait_bounded(&empty[s], ((it / kStagesG) - 1) & 1)) {
            dead = true;
            break;
          }
          unsigned char* st = sm + s * STAGE_BYTES;
          mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
          tma_load_2d(st, &ta, kb * BK, mt * BM, &full[s]);
          tma_load_2d(st + A_BYTES, tbs[g], kb * BK, nt * BN, &full[s]);
        }
      }
    }
  } else if (warp == 1) {
    // ================= MMA issue =================
    if (tid == 32) {
      const uint32_t idesc = tc::idesc_bf16_f32(BM, BN);
      int it = 0, local = 0;
      for (int t = blockIdx.x; t < p.total_tiles && !dead; t += gridDim.x, ++local) {
        const int buf = local & 1;
        // the epilogue has read this accumulator out (its previous use)
        if (local >= 2 && !mbar_wait_bounded(&acc_empty[buf], ((local >> 1) - 1) & 1)) {
          dead = true;
          break;
        }
        tc::fence_after_sync();
        const uint32_t acc = tmem + buf * kAccCols;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % kStagesG;
          if (!mbar_wait_bounded(&full[s], (it / kStagesG) & 1)) {
            dead = true;
            break;
          }
          tc::fence_after_sync();
          const uint32_t sa = smem_u32(sm + s * STAGE_BYTES);
          tc::mma_tile(acc, sa, 0u, sa + A_BYTES, 0u, 1, idesc, kb > 0);
          tc::commit(&empty[s]);  // the stage is free once these MMAs are done
        }
        if (dead) break;
        tc::commit(&acc_full[buf]);
      }
    }
  } else {
    // ================= epilogue (warps 2..5) =================
    const int q = warp & 3;  // TMEM lane quarter of this warp
    const int l = tid & 31;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    unsigned char* epi = sm + OFF_EPI + (warp - 2) * EPI_BYTES;
    int local = 0;
    for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++local) {
      const int buf = local & 1;
      uint32_t okw = 1;
      if (l == 0) okw = mbar_wait_bounded(&acc_full[buf], (local >> 1) & 1) ? 1u : 0u;
      okw = __shfl_sync(0xffffffffu, okw, 0);
      if (!okw) {
        dead = true;
        break;
      }
      tc::fence_after_sync();
      int g, mt, nt;
      tile_coords(p, t, g, mt, nt);
      const GemmGroup& G = p.g[g];
      __nv_bfloat16* C = static_cast<__nv_bfloat16*>(G.C);
      const int row0 = mt * BM + q * 32;
      const int col0 = nt * BN;
      const uint32_t acc = tmem + buf * kAccCols;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        if (col0 + c * 32 >= G.N) break;  // warp-uniform
        float v[32];
        tc::tmem_ld32(acc + lane_base + c * 32, v);
        tc::tmem_wait_ld();
        // row l of this warp's 32 x 32 block: four 16-byte chunks at the
        // XOR-rotated positions chunk ^ (l & 3), conflict-free
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint4 w;
          w.x = tc::pack2(v[8 * ch + 0], v[8 * ch + 1], (__nv_bfloat16*)nullptr);
          w.y = tc::pack2(v[8 * ch + 2], v[8 * ch + 3], (__nv_bfloat16*)nullptr);
          w.z = tc::pack2(v[8 * ch + 4], v[8 * ch + 5], (__nv_bfloat16*)nullptr);
          w.w = tc::pack2(v[8 * ch + 6], v[8 * ch + 7], (__nv_bfloat16*)nullptr);
          *reinterpret_cast<uint4*>(epi + l * 64 + ((ch ^ (l & 3)) << 4)) = w;
        }
        __syncwarp();
        // each thread: rows (l / 4) + 8 i, chunk l % 4 -> 16 bytes of a
        // 64-byte row segment
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = (l >> 2) + 8 * i, ch = l & 3;
          const int row = row0 + r, col = col0 + c * 32 + ch * 8;
          const uint4 w = *reinterpret_cast<const uint4*>(epi + r * 64 + ((ch ^ (r & 3)) << 4));
          if (row < p.M && col < G.N)
            *reinterpret_cast<uint4*>(C + (size_t)row * G.ldc + col) = w;
        }
        __syncwarp();
      }
      tc::fence_before_sync();
      __syncwarp();
      if (l == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&acc_empty[buf])) : "memory");
    }
  }
  if (dead && p.flags) atomicOr(p.flags, GDN_FLAG_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 2 * kAccCols);
}

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                             const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                             const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                             CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Row-major bf16 [rows][cols] read in boxes of 64 columns x box_rows rows,
// 128-byte swizzled, zero fill outside.
cudaError_t bf16_map(CUtensorMap* m, const void* base, int rows, int cols, int ld, int box_rows) {
  static EncodeFn encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<EncodeFn>(fn);
  }
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int g_proj_num_sms = 0;

// Gated RMS norm per (token, v-head): one warp, 4 channels per lane.
__global__ void __launch_bounds__(256) gated_norm_kernel(const __nv_bfloat16* __restrict__ o,
                                                          const __nv_bfloat16* __restrict__ z,
                                                          const float* __restrict__ w,
                                                          __nv_bfloat16* __restrict__ on, int rows,
                                                          float eps) {
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int l = threadIdx.x & 31;
  if (r >= rows) return;
  const size_t base = (size_t)r * 128 + l * 4;
  const uint2 ov = *reinterpret_cast<const uint2*>(o + base);
  const uint2 zv = *reinterpret_cast<const uint2*>(z + base);
  const float4 wv = *reinterpret_cast<const float4*>(w + l * 4);
  const float2 o01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ov.x));
  const float2 o23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ov.y));
  const float2 z01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&zv.x));
  const float2 z23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&zv.y));
  float ss = o01.x * o01.x + o01.y * o01.y + o23.x * o23.x + o23.y * o23.y;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float rs = rsqrtf(ss * (1.f / 128.f) + eps);
  const float y0 = o01.x * rs * wv.x * silu_f32(z01.x);
  const float y1 = o01.y * rs * wv.y * silu_f32(z01.y);
  const float y2 = o23.x * rs * wv.z * silu_f32(z23.x);
  const float y3 = o23.y * rs * wv.w * silu_f32(z23.y);
  uint2 out;
  out.x = tc::pack2(y0, y1, (__nv_bfloat16*)nullptr);
  out.y = tc::pack2(y2, y3, (__nv_bfloat16*)nullptr);
  *reinterpret_cast<uint2*>(on + base) = out;
}

}  // namespace

// C_g = A B_g^T for the given groups (at most 4), one persistent launch.
cudaError_t launch_gemm(const void* A, int M, int K, int lda, int n_groups, const void* const* B,
                        const int* N, const int* ldb, void* const* C, const int* ldc,
                        unsigned* flags, cudaStream_t stream) {
  if (g_proj_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_proj_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_proj_num_sms <= 0) g_proj_num_sms = 1;
  }
  GemmParams p = {};
  p.M = M;
  p.K = K;
  p.n_groups = n_groups;
  p.tiles_m = (M + BM - 1) / BM;
  p.flags = flags;
  CUtensorMap ta, tb[4];
  cudaError_t e = bf16_map(&ta, A, M, K, lda, BM);
  if (e != cudaSuccess) return e;
  for (int g = 0; g < 4; ++g) {
    const int gg = g < n_groups ? g : n_groups - 1;  // unused maps repeat the last group
    e = bf16_map(&tb[g], B[gg], N[gg], K, ldb[gg], BN);
    if (e != cudaSuccess) return e;
    if (g < n_groups) {
      p.g[g].C = C[g];
      p.g[g].N = N[g];
      p.g[g].ldc = ldc[g];
      p.g[g].tiles_n = (N[g] + BN - 1) / BN;
      p.total_tiles += p.tiles_m * p.g[g].tiles_n;
    }
  }
  if (p.total_tiles == 0) return cudaSuccess;
  e = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)GEMM_SMEM);
  if (e != cudaSuccess) return e;
  const int grid = p.total_tiles < g_proj_num_sms ? p.total_tiles : g_proj_num_sms;
  gemm_kernel<<<grid, kGemmThreads, GEMM_SMEM, stream>>>(p, ta, tb[0], tb[1], tb[2], tb[3]);
  return cudaGetLastError();
}

cudaError_t launch_gated_norm(const void* o, const void* z, const float* w, void* on, int rows,
                              float eps, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  gated_norm_kernel<<<(rows + 7) / 8, 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(z), w,
      static_cast<__nv_bfloat16*>(on), rows, eps);
  return cudaGetLastError();
}

}  // namespace gdn

namespace {
bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
}  // namespace

extern "C" int gdn_in_proj(const void* hidden, int T, int d_model, const void* w_qkv,
                           const void* w_z, const void* w_b, const void* w_a, int C, int Hv,
                           int d_v, void* x_qkv, void* z, void* b, void* a, uint32_t* flags,
                           void* stream) {
  if (T < 0 || d_model <= 0 || C <= 0 || Hv <= 0 || d_v <= 0) return GDN_ERR_RANGE;
  if (T == 0) return GDN_OK;
  if (!hidden || !w_qkv || !w_z || !w_b || !w_a || !x_qkv || !z || !b || !a) return GDN_ERR_NULL;
  if (d_model % 8 || C % 8 || Hv % 8 || (Hv * d_v) % 8) return GDN_ERR_DIMS;
  const void* ptrs[] = {hidden, w_qkv, w_z, w_b, w_a, x_qkv, z, b, a};
  for (const void* q : ptrs)
    if (!al16(q)) return GDN_ERR_ALIGN;
  if (flags && ((uintptr_t)flags & 3u)) return GDN_ERR_ALIGN;
  const void* B[4] = {w_qkv, w_z, w_b, w_a};
  const int N[4] = {C, Hv * d_v, Hv, Hv};
  const int ldb[4] = {d_model, d_model, d_model, d_model};
  void* Cp[4] = {x_qkv, z, b, a};
  const int ldc[4] = {C, Hv * d_v, Hv, Hv};
  return gdn::launch_gemm(hidden, T, d_model, d_model, 4, B, N, ldb, Cp, ldc,
                          reinterpret_cast<unsigned*>(flags), (cudaStream_t)stream) == cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}

extern "C" int gdn_out_proj(const void* o, const void* z, const float* norm_w, float eps,
                            const void* w_out, int T, int Hv, int d_v, int d_model, void* o_norm,
                            void* y, uint32_t* flags, void* stream) {
  if (T < 0 || Hv <= 0 || d_model <= 0 || !(eps >= 0.f)) return GDN_ERR_RANGE;
  if (d_v != 128) return GDN_ERR_DIMS;
  if (T == 0) return GDN_OK;
  if (!o || !z || !norm_w || !w_out || !o_norm || !y) return GDN_ERR_NULL;
  if (d_model % 8 || Hv % 8) return GDN_ERR_DIMS;
  const void* ptrs[] = {o, z, norm_w, w_out, o_norm, y};
  for (const void* q : ptrs)
    if (!al16(q)) return GDN_ERR_ALIGN;
  if (flags && ((uintptr_t)flags & 3u)) return GDN_ERR_ALIGN;
  cudaStream_t s = (cudaStream_t)stream;
  if (gdn::launch_gated_norm(o, z, norm_w, o_norm, T * Hv, eps, s) != cudaSuccess)
    return GDN_ERR_CUDA;
  const void* B[1] = {w_out};
  const int N[1] = {d_model};
  const int K = Hv * d_v;
  const int ldb[1] = {K};
  void* Cp[1] = {y};
  const int ldc[1] = {d_model};
  return gdn::launch_gemm(o_norm, T, K, K, 1, B, N, ldb, Cp, ldc,
                          reinterpret_cast<unsigned*>(flags), s) == cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}

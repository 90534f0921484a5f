// State half of the chunked prefill: the recurrence across the 64-token
// chunks of each (sequence, v-head) chain, with every state-independent
// product precomputed (q~, k~, gates by prep_kernel; u, -w, P by
// intra_kernel).  Per chunk, with S0 the state at the chunk start (S[v][k],
// fp32 in tensor memory for the whole chain), G_C the cumulative gate of the
// chunk's last valid token and n its valid tokens, one 128 x 128 accumulator
// D (rows = tokens, columns = v) carries
//   rows 0..63  : U = u - w S0^T                 (the chunk's updates u_j)
//   rows 64..127: O = (e^G q~) S0^T + P U        (the chunk's outputs o_i)
// as
//   CUDA  S0 -> fp16 operand tile;  TMEM S <- e^{G_C} S0
//   MMA   D  = [-w ; q~] S0^T
//   CUDA  k~_j <- e^{G_C - G_j} k~_j in the staged tile (rows past n zeroed),
//         while the D product runs
//   CUDA  U  = u + D[0..63] -> fp16 token-major tile (rows past n zeroed);
//         D[64 + i] <- e^{G_i} D[64 + i] in TMEM
//   MMA   S += U^T (e^{G_C - G} k~)            (U and k~ as MN-major operands)
//   MMA   D += [0 ; P] U                       (rows 64..127: + P U)
//   CUDA  o_i = D[64 + i] -> bf16              (while the next chunk's MMAs run)
// This is the chunked gated delta rule (Gated Delta Networks, chunkwise WY
// form) run over cu_seqlens from per-sequence initial states, as a continuous
// batching engine does for a linear-attention layer.
//
// Persistent CTAs, one per SM: warp 8 is the producer (one TMA issue lane
// that pulls chains, longest sequences first, from the scheduler's counter
// and streams each chunk's tiles into a 2-stage ring), warp 9 issues the
// MMAs when the compute warps release it through named barriers, and warps
// 0-7 run the chain.  A compute thread owns TMEM lane (tid % 128) and one half
// of the columns; the warps on lanes 0..63 convert U, those on lanes 64..127
// scale the k~ tile and write outputs.
#include <cuda.h>

#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

using E = __half;
constexpr int D = 128;
constexpr int CH = 64;
constexpr int kCompute = 256;
constexpr int kProducer = kCompute;       // first thread of the TMA warp
constexpr int kIssuer = kCompute + 32;    // first thread of the MMA warp
constexpr int kThreads = kCompute + 64;
// named barriers: 1 the compute warps; 2 compute warps -> MMA warp (S0 tile
// written); 3 compute warps -> MMA warp (k~ tile scaled, U tile written);
// 4 output warps -> MMA warp (output rows rescaled)
constexpr int kBarC = 1, kBarD = 2, kBarS = 3, kBarO = 4;
constexpr int kGateD = kCompute + 32, kGateS = kCompute + 32, kGateO = kCompute / 2 + 32;
constexpr int R = 2;  // v-heads per k-head
constexpr float kF16Max = 65000.f;

// one stage (offsets inside the stage; every tile 1024-byte aligned)
constexpr uint32_t BOX = 8192;      // one 64 x 64 fp16 box
constexpr uint32_t KB_STRIDE = 16384;
constexpr uint32_t ST_QW = 0;       // [-w ; q~]: 2 K-blocks x 128 rows
constexpr uint32_t ST_K = 32768;    // k~ [64 tokens][128]: two 64-column boxes
constexpr uint32_t ST_U = 49152;    // u  [64 tokens][128]: two 64-column boxes
constexpr uint32_t ST_ZP = 65536;   // a zero 64 x 64 tile, then P [64][64]
constexpr uint32_t ST_G = 81920;    // gates [64][4] fp32
constexpr uint32_t ST_BYTES = 82944;
constexpr uint32_t ST_TX = ST_BYTES - BOX;  // what the TMA brings (all but the zero tile)
// CTA shared memory
constexpr uint32_t OFF_S0 = 2 * ST_BYTES;    // S0 fp16, 2 K-blocks x 128 rows
// U fp16 [64 tokens][128]: two 64-column boxes (apart from S0: D += P U may
// still read it while the next chunk's S0 is written)
constexpr uint32_t OFF_UT = OFF_S0 + 32768;
constexpr uint32_t SMEM_BYTES = OFF_UT + 16384 + 1024;
// tensor memory columns: the state, two accumulators D
constexpr uint32_t TM_S = 0, TM_D = 128, TM_COLS = 512;

struct ChunkDesc {
  int seq0, c0, n;    // sequence start row, chunk start, valid tokens
  int h, rblk, wblk;  // v-head, block read, block written
  int flags;          // 1 first chunk of the chain, 2 last, 4 end of work
};

__device__ __forceinline__ void cbar() {  // the compute warps only
  asm volatile("bar.sync %0, %1;" ::"n"(kBarC), "n"(kCompute) : "memory");
}

// compute warps release the MMA warp, which waits with mma_gate
template <int kId, int kCount>
__device__ __forceinline__ void mma_release() {
  asm volatile("bar.arrive %0, %1;" ::"n"(kId), "n"(kCount) : "memory");
}
template <int kId, int kCount>
__device__ __forceinline__ void mma_gate() {
  asm volatile("bar.sync %0, %1;" ::"n"(kId), "n"(kCount) : "memory");
}

// Packed fp32 pair sum (one add.rn.f32x2 on sm_100 and later): (a, b) += (x, y).
__device__ __forceinline__ void add2(float& a, float& b, float x, float y) {
  unsigned long long v = (unsigned long long)__float_as_uint(a) | ((unsigned long long)__float_as_uint(b) << 32);
  const unsigned long long w = (unsigned long long)__float_as_uint(x) | ((unsigned long long)__float_as_uint(y) << 32);
  asm("add.rn.f32x2 %0, %0, %1;" : "+l"(v) : "l"(w));
  a = __uint_as_float((uint32_t)v);
  b = __uint_as_float((uint32_t)(v >> 32));
}

// Packed fp32 pair product (one mul.rn.f32x2 on sm_100 and later).
__device__ __forceinline__ void mul2(float& a, float& b, float s) {
  unsigned long long v = (unsigned long long)__float_as_uint(a) | ((unsigned long long)__float_as_uint(b) << 32);
  const unsigned long long m = (unsigned long long)__float_as_uint(s) | ((unsigned long long)__float_as_uint(s) << 32);
  asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(v) : "l"(m));
  a = __uint_as_float((uint32_t)v);
  b = __uint_as_float((uint32_t)(v >> 32));
}

__device__ __forceinline__ uint4 pack8(const float* v) {
  uint4 w;
  w.x = tc::pack2(v[0], v[1], (E*)nullptr);
  w.y = tc::pack2(v[2], v[3], (E*)nullptr);
  w.z = tc::pack2(v[4], v[5], (E*)nullptr);
  w.w = tc::pack2(v[6], v[7], (E*)nullptr);
  return w;
}
__device__ __forceinline__ void unpack8(const uint4& w, float* v) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[e]));
    v[2 * e] = f.x;
    v[2 * e + 1] = f.y;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
seq_kernel(FwdParams p, const __grid_constant__ CUtensorMap tqk, const __grid_constant__ CUtensorMap tw,
           const __grid_constant__ CUtensorMap tu, const __grid_constant__ CUtensorMap tp,
           const __grid_constant__ CUtensorMap tg) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t full[2], empty[2], mma_y, mma_s;
  __shared__ ChunkDesc desc[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int ok_c;
  __shared__ volatile int mma_stop;

  const int tid = threadIdx.x;
  const int Hv = p.Hv;
  int32_t* hdr = p.work.header();
  const int n_chains = hdr[kNPre] * Hv;
  if ((int)blockIdx.x >= n_chains) return;
  const uint32_t sbase = smem_u32(sm);

  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&full[b], 1);
      mbar_init(&empty[b], 1);
    }
    mbar_init(&mma_y, 1);
    mbar_init(&mma_s, 1);
    fence_mbar_init();
    mma_stop = 0;
  }
  // the zero tiles in front of each stage's P
  for (int t = tid; t < 2 * (int)(BOX / 16); t += kThreads)
    *reinterpret_cast<uint4*>(sm + (t >> 9) * ST_BYTES + ST_ZP + (t & 511) * 16) = make_uint4(0, 0, 0, 0);
  tc::fence_proxy_async_smem();
  if (tid < 32) tc::tmem_alloc(&tmem_slot, TM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;

  if (tid >= kIssuer) {
    // ============================= MMA warp ==============================
    // Chunk k: gate kBarD (S0 tile ready)          -> D = [-w ; q~] S0^T;
    //          gate kBarS (k~ scaled, U tile ready) -> S += U^T (e^{G_C-G} k~);
    //          gate kBarO (output rows rescaled)    -> D += [0 ; P] U.
    // mma_s covers the state update only (the next hand-over waits for it),
    // except on a chain's last chunk, whose outputs are written right away.
    // The compute warps only ever leave while this warp waits at kBarD or
    // kBarS, so the stop flag is read there.
    for (int k = 0;; ++k) {
      const int b = k & 1;
      const uint32_t sb = sbase + b * ST_BYTES;
      const uint32_t dcol = TM_D + (k & 1) * 128;
      mma_gate<kBarD, kGateD>();
      if (mma_stop) break;
      if (tid == kIssuer) {
        tc::fence_after_sync();
        tc::mma_op(tmem + dcol, tc::Opnd{sb + ST_QW, KB_STRIDE, false},
                   tc::Opnd{sbase + OFF_S0, KB_STRIDE, false}, D / 16, tc::idesc_f16_f32(128, 128),
                   false);
        tc::commit(&mma_y);
      }
      __syncwarp();
      mma_gate<kBarS, kGateS>();
      if (mma_stop) break;
      const bool last = (desc[b].flags & 2) != 0;
      const tc::Opnd ut{sbase + OFF_UT, BOX, true};
      if (tid == kIssuer) {
        tc::fence_after_sync();
        tc::mma_op(tmem + TM_S, ut, tc::Opnd{sb + ST_K, BOX, true}, CH / 16,
                   tc::idesc_f16_f32(128, 128, true, true), true);
        if (!last) tc::commit(&mma_s);
      }
      __syncwarp();
      mma_gate<kBarO, kGateO>();
      if (tid == kIssuer) {
        tc::fence_after_sync();
        tc::mma_op(tmem + dcol, tc::Opnd{sb + ST_ZP, 0u, false}, ut, CH / 16,
                   tc::idesc_f16_f32(128, 128, false, true), true);
        if (last) tc::commit(&mma_s);
        tc::commit(&empty[b]);  // the stage is free once these MMAs are done
      }
      __syncwarp();
    }
  } else if (tid >= kProducer) {
    // =========================== producer warp ===========================
    if (tid == kProducer) {
      int k = 0;
      bool dead = false;
      for (;;) {
        const int chain = atomicAdd(&hdr[kWorkHead], 1);
        const bool end = chain >= n_chains;
        int s = 0, h = 0, seq0 = 0, L = 0, nc = 1;
        if (!end) {
          s = p.work.pre()[chain / Hv];
          h = chain % Hv;
          seq0 = p.cu[s];
          L = p.cu[s + 1] - seq0;
          nc = (L + CH - 1) / CH;
        }
        for (int c = 0; c < nc; ++c, ++k) {
          const int b = k & 1;
          if (k >= 2 && !mbar_wait_bounded(&empty[b], ((k >> 1) - 1) & 1)) { dead = true; break; }
          ChunkDesc d;
          d.seq0 = seq0; d.c0 = c * CH; d.n = end ? 0 : min(CH, L - c * CH);
          d.h = h;
          d.wblk = end ? 0 : p.blk[s];
          d.rblk = (!end && p.has_past[s]) ? d.wblk : 0;
          d.flags = end ? 4 : ((c == 0 ? 1 : 0) | (c == nc - 1 ? 2 : 0));
          desc[b] = d;
          if (end) {
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&full[b]))
                         : "memory");
            break;
          }
          const int kh = h / R, r0 = seq0 + c * CH;
          unsigned char* st = sm + b * ST_BYTES;
          mbar_arrive_expect_tx(&full[b], ST_TX);
          tma_load_2d(st + ST_QW, &tw, h * D, r0, &full[b]);
          tma_load_2d(st + ST_QW + KB_STRIDE, &tw, h * D + 64, r0, &full[b]);
          tma_load_2d(st + ST_QW + CH * 128, &tqk, kh * 2 * D, r0, &full[b]);
          tma_load_2d(st + ST_QW + KB_STRIDE + CH * 128, &tqk, kh * 2 * D + 64, r0, &full[b]);
          tma_load_2d(st + ST_K, &tqk, kh * 2 * D + D, r0, &full[b]);
          tma_load_2d(st + ST_K + BOX, &tqk, kh * 2 * D + D + 64, r0, &full[b]);
          tma_load_2d(st + ST_U, &tu, h * D, r0, &full[b]);
          tma_load_2d(st + ST_U + BOX, &tu, h * D + 64, r0, &full[b]);
          tma_load_2d(st + ST_ZP + BOX, &tp, h * CH, r0, &full[b]);
          tma_load_2d(st + ST_G, &tg, 4 * kh, r0, &full[b]);
        }
        if (dead || end) break;
      }
      if (dead) atomicOr((unsigned*)&hdr[kErr], GDN_FLAG_TIMEOUT);
    }
    __syncwarp();
  } else {
    // =========================== compute warps ===========================
    const uint32_t lane = (uint32_t)(tid & 96) << 16;  // TMEM lane quarter of this warp
    const int r128 = tid & 127;                        // TMEM lane = state row v / D row
    const int hf = tid >> 7;                           // column half
    const bool urow = r128 < CH;                       // D rows 0..63: U; 64..127: outputs
    const int j = r128 & 63;                           // token of this thread's D row
    __nv_bfloat16* __restrict__ out = reinterpret_cast<__nv_bfloat16*>(p.out);
    auto wait_c = [&](uint64_t* bar, uint32_t parity) -> bool {
      if (tid == 0) ok_c = mbar_wait_bounded(bar, parity) ? 1 : 0;
      cbar();
      return ok_c != 0;
    };
    uint32_t ph_y = 0, ph_s = 0;
    bool s_busy = false;   // an MMA-S commit not waited for yet
    bool pending = false;  // outputs of the previous chunk not written yet
    int p_row = 0, p_n = 0, p_h = 0, p_ob = 0;
    bool dead = false;
    int next_gate = kBarD;  // the gate the MMA warp waits at
    float amax = 0.f;
    // outputs of the pending chunk: row 64 + i of its D is o_i (this thread's 64 v)
    // (tcgen05.ld is warp-collective: the lane predicate guards the stores only)
    auto flush = [&]() {
      if (urow) return;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float o[32];
        tc::tmem_ld32(tmem + lane + TM_D + p_ob * 128 + hf * 64 + hh * 32, o);
        tc::tmem_wait_ld();
        if (j < p_n) {
          uint4* dst = reinterpret_cast<uint4*>(out + ((size_t)(p_row + j) * Hv + p_h) * D + hf * 64 +
                                                hh * 32);
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {
            uint4 w;
            w.x = tc::pack2(o[g8 * 8 + 0], o[g8 * 8 + 1], (__nv_bfloat16*)nullptr);
            w.y = tc::pack2(o[g8 * 8 + 2], o[g8 * 8 + 3], (__nv_bfloat16*)nullptr);
            w.z = tc::pack2(o[g8 * 8 + 4], o[g8 * 8 + 5], (__nv_bfloat16*)nullptr);
            w.w = tc::pack2(o[g8 * 8 + 6], o[g8 * 8 + 7], (__nv_bfloat16*)nullptr);
            dst[g8] = w;
          }
        }
      }
    };
    for (int k = 0;; ++k) {
      const int b = k & 1;
      if (!wait_c(&full[b], (k >> 1) & 1)) { dead = true; break; }
      const ChunkDesc d = desc[b];
      if (d.flags & 4) break;
      unsigned char* st = sm + b * ST_BYTES;
      const float* GT = reinterpret_cast<const float*>(st + ST_G);
      const int r2 = d.h % R;
      const int n = d.n;
      const float GC = GT[(n - 1) * 4 + 2 * r2];
      // ---- the previous chunk's MMAs are done: S and its D readable
      if (s_busy) {
        if (!wait_c(&mma_s, ph_s)) { dead = true; break; }
        ph_s ^= 1;
        s_busy = false;
        tc::fence_after_sync();
      }
      // ---- state hand-over: S0 -> fp16 tile, TMEM S <- e^{G_C} S0 (32 columns at a time)
      {
        const int v = r128;
        const float dc = __expf(GC);
        const float* S_r = reinterpret_cast<const float*>(p.layer_base + (size_t)d.rblk * p.stride +
                                                          p.rec_off) + (size_t)d.h * D * D;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int k0 = hf * 64 + hh * 32;
          float srow[32];
          if (d.flags & 1) {
#pragma unroll
            for (int kk = 0; kk < 32; ++kk) srow[kk] = S_r[(size_t)(k0 + kk) * D + v];
          } else {
            tc::tmem_ld32(tmem + lane + TM_S + k0, srow);
            tc::tmem_wait_ld();
          }
          float m4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < 32; ++kk) m4[kk & 3] = fmaxf(m4[kk & 3], fabsf(srow[kk]));
          amax = fmaxf(amax, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8)
            *reinterpret_cast<uint4*>(sm + OFF_S0 + hf * KB_STRIDE +
                                      tc::sw128_offset(v, hh * 32 + g8 * 8)) = pack8(srow + g8 * 8);
#pragma unroll
          for (int kk = 0; kk < 32; kk += 2) mul2(srow[kk], srow[kk + 1], dc);
          tc::tmem_st32(tmem + lane + TM_S + k0, srow);
        }
        tc::tmem_wait_st();
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      mma_release<kBarD, kGateD>();  // D = [-w ; e^G q~] S0^T
      next_gate = kBarS;
      const int ob = k & 1;
      const uint32_t dcol = TM_D + ob * 128;
      // ---- while the tensor core runs: this chunk's u row (U-row warps), or
      // k~_j <- e^{G_C - G_j} k~_j for the state update, rows past the
      // sequence -> 0 (output warps: row j of column half hf, its 16-byte
      // chunks in an order rotated by j, which keeps the accesses conflict-free)
      uint4 ur[8];
      if (urow) {
        const unsigned char* urow_p = st + ST_U + hf * BOX + j * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          ur[c] = *reinterpret_cast<const uint4*>(urow_p + ((c ^ (j & 7)) << 4));
      } else {
        unsigned char* krow = st + ST_K + hf * BOX + j * 128;
        if (j < n) {
          const float ds = __expf(GC - GT[j * 4 + 2 * r2]);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4* q = reinterpret_cast<uint4*>(krow + (((c + j) & 7) << 4));
            float k8[8];
            unpack8(*q, k8);
#pragma unroll
            for (int e = 0; e < 8; e += 2) mul2(k8[e], k8[e + 1], ds);
            *q = pack8(k8);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(krow + (c << 4)) = make_uint4(0, 0, 0, 0);
        }
        tc::fence_proxy_async_smem();
        mma_release<kBarS, kGateS>();
      }
      if (!wait_c(&mma_y, ph_y)) { dead = true; break; }
      ph_y ^= 1;
      tc::fence_after_sync();
      // ---- U = u + D[0..63] -> fp16 token-major tile (same swizzled places as
      // u) on the U-row warps, which then release the state update; the
      // output warps meanwhile write the previous chunk's outputs (its
      // D += P U finished before this chunk's D product)
      if (urow) {
        unsigned char* dst = sm + OFF_UT + hf * BOX + j * 128;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float dv[32];
          tc::tmem_ld32(tmem + lane + dcol + hf * 64 + hh * 32, dv);
          tc::tmem_wait_ld();
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int c = hh * 4 + c4;
            uint4 w = make_uint4(0, 0, 0, 0);
            if (j < n) {
              float u8[8];
              unpack8(ur[c], u8);
              float m2 = 0.f;
#pragma unroll
              for (int e = 0; e < 8; e += 2) {
                add2(u8[e], u8[e + 1], dv[c4 * 8 + e], dv[c4 * 8 + e + 1]);
                m2 = fmaxf(m2, fmaxf(fabsf(u8[e]), fabsf(u8[e + 1])));
              }
              amax = fmaxf(amax, m2);
              w = pack8(u8);
            }
            *reinterpret_cast<uint4*>(dst + ((c ^ (j & 7)) << 4)) = w;
          }
        }
        tc::fence_proxy_async_smem();
      } else {
        if (pending) flush();
        // o rows: D[64 + i] <- e^{G_i} D[64 + i] before P U accumulates onto them
        const float eg = j < n ? __expf(GT[j * 4 + 2 * r2]) : 0.f;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float o[32];
          tc::tmem_ld32(tmem + lane + dcol + hf * 64 + hh * 32, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e += 2) mul2(o[e], o[e + 1], eg);
          tc::tmem_st32(tmem + lane + dcol + hf * 64 + hh * 32, o);
        }
        tc::tmem_wait_st();
      }
      tc::fence_before_sync();
      if (urow) mma_release<kBarS, kGateS>();  // S += U^T (e^{G_C - G} k~)
      else mma_release<kBarO, kGateO>();       // D += [0 ; P] U
      next_gate = kBarD;
      s_busy = true;
      pending = true;
      p_row = d.seq0 + d.c0;
      p_n = n;
      p_h = d.h;
      p_ob = ob;
      if (d.flags & 2) {
        // ---- last chunk of the chain: its outputs and the final state now
        if (!wait_c(&mma_s, ph_s)) { dead = true; break; }
        ph_s ^= 1;
        s_busy = false;
        tc::fence_after_sync();
        flush();
        pending = false;
        float* S_w = reinterpret_cast<float*>(p.layer_base + (size_t)d.wblk * p.stride + p.rec_off) +
                     (size_t)d.h * D * D;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float srow[32];
          tc::tmem_ld32(tmem + lane + TM_S + hf * 64 + half * 32, srow);
          tc::tmem_wait_ld();
#pragma unroll
          for (int kk = 0; kk < 32; ++kk)
            S_w[(size_t)(hf * 64 + half * 32 + kk) * D + r128] = srow[kk];
        }
      }
    }
    // let the MMA warp out of the gate it waits at
    if (tid == 0) mma_stop = 1;
    cbar();
    if (next_gate == kBarD) mma_release<kBarD, kGateD>();
    else if (urow) mma_release<kBarS, kGateS>();  // the output warps arrived after scaling k~
    if (dead && tid == 0) atomicOr((unsigned*)&hdr[kErr], GDN_FLAG_TIMEOUT);
    // the state and U enter tensor-core operands in fp16
    if (!(amax <= kF16Max)) atomicOr((unsigned*)&hdr[kErr], GDN_FLAG_RANGE);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (tid < 32) tc::tmem_dealloc(tmem, TM_COLS);
}

}  // namespace

cudaError_t launch_seq(const FwdParams& p, const void* const* maps, int grid, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(seq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  auto m = [&](int i) { return *static_cast<const CUtensorMap*>(maps[i]); };
  seq_kernel<<<grid, kThreads, SMEM_BYTES, stream>>>(p, m(0), m(1), m(2), m(3), m(4));
  return cudaGetLastError();
}

}  // namespace gdn

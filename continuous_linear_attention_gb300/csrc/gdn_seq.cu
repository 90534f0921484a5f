// State half of the chunked prefill: the recurrence across the 64-token
// chunks of each (sequence, v-head) chain, with every state-independent
// product precomputed by cintra_kernel (q~, k~, gates, u, -w, P).  Per
// chunk, with S0 the state at the chunk start (S[v][k],
// fp32 in tensor memory for the whole chain), G_C the cumulative gate of the
// chunk's last valid token and n its valid tokens, everything runs in the
// transposed orientation: tensor-memory lane = v, columns = k or tokens.  One
// 128 x 128 accumulator D^T carries
//   columns 0..63  : U^T = u^T - S0 w^T            (the chunk's updates u_j),
//                    then U^T P^T
//   columns 64..127: S0 q~^T
// as
//   CUDA  S0 -> fp16 A operand in tensor memory, in two passes over k (0..63,
//         then 64..127), each released to the tensor core before
//         S <- e^{G_C} S0 is written back
//   MMA   D^T  = S0 [-w ; q~]^T (the first pass's K-steps start while the
//         second pass runs);  D^T[:, j] += u_j  (u^T times an identity)
//   CUDA  k~_j <- e^{G_C - G_j} k~_j in the staged tile, rows past n zeroed
//         (while the D product runs)
//   CUDA  U^T = D^T[:, 0..63] -> fp16 A operand in tensor memory (columns
//         past n zeroed)
//   MMA   S  += U^T (e^{G_C - G} k~)             (k~ as an MN-major operand)
//   MMA   D^T[:, 0..63] = U^T P^T               (over the U^T columns, read)
//   CUDA  o_i = e^{G_i} D^T[:, 64 + i] + D^T[:, i] -> bf16  (while the next
//         chunk's MMAs run)
// This is the chunked gated delta rule (Gated Delta Networks, chunkwise WY
// form) run over cu_seqlens from per-sequence initial states, as a continuous
// batching engine does for a linear-attention layer.  With the state as the
// tensor-memory A operand, no state or update tile passes through shared
// memory, and every compute warp owns one lane quarter and one column half of
// each step, so the CUDA-core work spreads over all four SM sub-partitions.
//
// The per-channel-decay (KDA) instance runs the same steps on that rule's
// tiles: q^_i = q~_i e^{Gamma_i} and k^_j = k~_j e^{Gamma_C - Gamma_j} (per
// key channel, from kintra_kernel, one tile per v-head) take the places of
// q~ and e^{G_C - G_j} k~_j with the output scales 1, -w = -T diag(beta)
// (k~ e^{Gamma}), and the hand-over scales state column k by its own
// e^{Gamma_C[k]}: S <- S0 Diag(e^{Gamma_C}).
//
// Persistent CTAs, one per SM: warp 8 is the producer (one lane that pulls
// chains, longest sequences first, from the scheduler's counter and
// bulk-copies each chunk's tiles, chunk-major in the prefill scratch, into a
// 3-stage ring), warp 9 issues the
// MMAs when the compute warps release it through named barriers, and warps
// 0-7 run the chain: thread t owns lane v = t % 128 and column half t / 128.
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
constexpr int kProducer = kCompute;       // first thread of the bulk-copy warp
constexpr int kIssuer = kCompute + 32;    // first thread of the MMA warp
constexpr int kThreads = kCompute + 64;
// named barriers: 1 the compute warps; compute warps -> MMA warp: 5 S0
// columns k < 64 written, 2 all of S0 written, 3 k~ tile scaled and U^T
// written
constexpr int kBarC = 1, kBarD = 2, kBarS = 3, kBarD1 = 5;
constexpr int kGate = kCompute + 32;
constexpr int R = 2;  // v-heads per k-head
constexpr float kF16Max = 65000.f;
constexpr int kStages = 3;

// one stage (offsets inside the stage; every tile 1024-byte aligned)
constexpr uint32_t BOX = 8192;      // one 64 x 64 fp16 box
constexpr uint32_t KB_STRIDE = 16384;
constexpr uint32_t ST_QW = 0;       // [-w ; q~]: 2 K-blocks x 128 token rows (K-major B)
constexpr uint32_t ST_K = 32768;    // k~ [64 tokens][128]: two 64-column boxes
constexpr uint32_t ST_U = 49152;    // u  [64 tokens][128]: two 64-column boxes
constexpr uint32_t ST_P = 65536;    // P  [64 i][64 j]
constexpr uint32_t ST_G = 73728;    // gates [64][4] fp32
constexpr uint32_t ST_BYTES = 74752;
// CTA shared memory: the ring, then a 16 x 16 identity (K-major B operand)
constexpr uint32_t OFF_I = kStages * ST_BYTES;
constexpr uint32_t SMEM_BYTES = OFF_I + 2048 + 1024;
// tensor memory columns: the state (fp32), two accumulators D^T, then the
// fp16 A operands S0 (K = 128: 64 columns) and U^T (K = 64: 32 columns)
constexpr uint32_t TM_S = 0, TM_D = 128, TM_S0 = 384, TM_UT = 448, TM_COLS = 512;

struct ChunkDesc {
  int seq0, c0, n;    // sequence start row, chunk start, valid tokens
  int h, rblk, wblk;  // v-head, block read, block written
  int flags;          // 1 first chunk of the chain, 2 last, 4 end of work
  int kpre;           // index of the sequence in the prefill list
};

__device__ __forceinline__ void cbar() {  // the compute warps only
  asm volatile("bar.sync %0, %1;" ::"n"(kBarC), "n"(kCompute) : "memory");
}
// the same barrier, returning whether any compute thread passed true
__device__ __forceinline__ bool cbar_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kBarC), "n"(kCompute)
      : "memory");
  return r != 0;
}

// compute warps release the MMA warp, which waits with mma_gate
template <int kId>
__device__ __forceinline__ void mma_release() {
  asm volatile("bar.arrive %0, %1;" ::"n"(kId), "n"(kGate) : "memory");
}
template <int kId>
__device__ __forceinline__ void mma_gate() {
  asm volatile("bar.sync %0, %1;" ::"n"(kId), "n"(kGate) : "memory");
}

// Packed fp32 pair product (one mul.rn.f32x2 on sm_100 and later): (a, b) *= (x, y).
__device__ __forceinline__ void mul2v(float& a, float& b, float x, float y) {
  unsigned long long v = (unsigned long long)__float_as_uint(a) | ((unsigned long long)__float_as_uint(b) << 32);
  const unsigned long long m = (unsigned long long)__float_as_uint(x) | ((unsigned long long)__float_as_uint(y) << 32);
  asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(v) : "l"(m));
  a = __uint_as_float((uint32_t)v);
  b = __uint_as_float((uint32_t)(v >> 32));
}
__device__ __forceinline__ void mul2(float& a, float& b, float s) { mul2v(a, b, s, s); }
// Packed fp32 pair fma (one fma.rn.f32x2): (a, b) = (a, b) * (x, y) + (c, d).
__device__ __forceinline__ void fma2v(float& a, float& b, float x, float y, float c, float d) {
  unsigned long long v = (unsigned long long)__float_as_uint(a) | ((unsigned long long)__float_as_uint(b) << 32);
  const unsigned long long m = (unsigned long long)__float_as_uint(x) | ((unsigned long long)__float_as_uint(y) << 32);
  const unsigned long long ad = (unsigned long long)__float_as_uint(c) | ((unsigned long long)__float_as_uint(d) << 32);
  asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(v) : "l"(m), "l"(ad));
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

template <bool kKda>
__global__ void __launch_bounds__(kThreads, 1)
seq_kernel(FwdParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t full[kStages], empty[kStages], mma_y, mma_s;
  __shared__ ChunkDesc desc[kStages];
  // e^{G_i} of the chunks with D^T accumulator 0 / 1 (1 for the per-channel
  // decay, whose tiles carry the scales; 0 past a chunk's end)
  __shared__ __align__(16) float EF[2][CH];
  __shared__ uint32_t tmem_slot;
  // outcomes of the compute warps' waits, in two slots used in turn: two waits
  // in a row have no other barrier between them, and a thread may read a
  // slot after thread 0 has moved on to the next wait
  __shared__ int ok_c[2];
  __shared__ volatile int mma_stop;

  pdl_wait_then_release();
  const int tid = threadIdx.x;
  const int Hv = p.Hv;
  int32_t* hdr = p.work.header();
  const int n_chains = hdr[kNPre] * Hv;
  if ((int)blockIdx.x >= n_chains) return;
  const uint32_t sbase = smem_u32(sm);

  if (tid == 0) {
    for (int b = 0; b < kStages; ++b) {
      mbar_init(&full[b], 1);
      mbar_init(&empty[b], 1);
    }
    mbar_init(&mma_y, 1);
    mbar_init(&mma_s, 1);
    fence_mbar_init();
    mma_stop = 0;
  }
  // the 16 x 16 identity: row e holds 1.0 at K-element e (rows of 128 bytes,
  // 128-byte swizzle; only the first 32 bytes of a row are read)
  for (int t = tid; t < 128; t += kThreads)
    *reinterpret_cast<uint4*>(sm + OFF_I + t * 16) = make_uint4(0, 0, 0, 0);
  __syncthreads();
  if (tid < 16)
    *reinterpret_cast<__half*>(sm + OFF_I + tc::sw128_offset(tid, tid)) = __float2half_rn(1.f);
  tc::fence_proxy_async_smem();
  if (tid < 32) tc::tmem_alloc(&tmem_slot, TM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;

  if (tid >= kIssuer) {
    // ============================= MMA warp ==============================
    // Chunk k: gate kBarD1 (S0, k < 64)      -> D^T  = S0[:, :64] [-w ; q~][:, :64]^T;
    //          gate kBarD (all of S0)        -> D^T += S0[:, 64:] [-w ; q~][:, 64:]^T, + u^T I;
    //          gate kBarS (k~ scaled, U^T)   -> S += U^T (e^{G_C-G} k~);
    //                                           D^T[:, ..64] = U^T P^T.
    // mma_s covers the state update only (the next hand-over waits for it;
    // the outputs are read after the next chunk's D product), except on a
    // chain's last chunk, whose outputs are written right away.  The compute
    // warps only ever leave while this warp waits at kBarD1 or kBarS, so the
    // stop flag is read there.
    for (int k = 0;; ++k) {
      const int b = k % kStages;
      const uint32_t sb = sbase + b * ST_BYTES;
      const uint32_t dcol = TM_D + (k & 1) * 128;
      const tc::Opnd qw{sb + ST_QW, KB_STRIDE, false};
      mma_gate<kBarD1>();
      if (mma_stop) break;
      if (tid == kIssuer) {
        tc::fence_after_sync();
#pragma unroll
        for (int s = 0; s < 4; ++s)
          tc::mma_ts(tmem + dcol, tmem + TM_S0 + 8 * s, tc::opnd_desc(qw, s), tc::idesc_f16_f32(128, 128),
                     s > 0 ? 1u : 0u);
      }
      __syncwarp();
      mma_gate<kBarD>();
      if (tid == kIssuer) {
        tc::fence_after_sync();
#pragma unroll
        for (int s = 4; s < 8; ++s)
          tc::mma_ts(tmem + dcol, tmem + TM_S0 + 8 * s, tc::opnd_desc(qw, s), tc::idesc_f16_f32(128, 128), 1u);
        // + u_j on column j: u^T (MN-major; K-step s = tokens 16s..16s+15)
        // times the identity, into columns 16s..16s+15
#pragma unroll
        for (int s = 0; s < CH / 16; ++s)
          tc::mma_bf16(tmem + dcol + 16 * s, tc::opnd_desc(tc::Opnd{sb + ST_U, BOX, true}, s),
                       tc::sw128_desc(sbase + OFF_I), tc::idesc_f16_f32(128, 16, true, false), 1u);
        tc::commit(&mma_y);
      }
      __syncwarp();
      mma_gate<kBarS>();
      if (mma_stop) break;
      const bool last = (desc[b].flags & 2) != 0;
      if (tid == kIssuer) {
        tc::fence_after_sync();
        tc::mma_op_ts(tmem + TM_S, tmem + TM_UT, tc::Opnd{sb + ST_K, BOX, true}, CH / 16,
                      tc::idesc_f16_f32(128, 128, false, true), true);
        if (!last) tc::commit(&mma_s);
        // the outputs' U^T P^T over the U^T columns, which the compute warps
        // have read
        tc::mma_op_ts(tmem + dcol, tmem + TM_UT, tc::Opnd{sb + ST_P, 0u, false}, CH / 16,
                      tc::idesc_f16_f32(128, 64), false);
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
          h = chain % Hv;
          // a chain whose chunk products left the fp16 range goes to the
          // token-serial redo instead
          if (redo_marked(p.work, chain / Hv, h)) continue;
          s = p.work.pre()[chain / Hv];
          seq0 = p.cu[s];
          L = p.cu[s + 1] - seq0;
          nc = (L + CH - 1) / CH;
        }
        for (int c = 0; c < nc; ++c, ++k) {
          const int b = k % kStages;
          if (k >= kStages && !mbar_wait_bounded(&empty[b], ((k / kStages) - 1) & 1)) {
            dead = true;
            break;
          }
          ChunkDesc d;
          d.seq0 = seq0; d.c0 = c * CH; d.n = end ? 0 : min(CH, L - c * CH);
          d.h = h;
          d.wblk = end ? 0 : p.blk[s];
          d.rblk = (!end && p.has_past[s]) ? d.wblk : 0;
          d.flags = end ? 4 : ((c == 0 ? 1 : 0) | (c == nc - 1 ? 2 : 0));
          d.kpre = chain / Hv;
          desc[b] = d;
          if (end) {
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&full[b]))
                         : "memory");
            break;
          }
          // the chunk's tiles, as the chunk-parallel kernel left them
          // (chunk-major, each in its operand layout): -w and q~ interleaved
          // by K-block into [-w ; q~], k~, u, P and the gate tile
          const int kh = h / R;
          const size_t gi = (size_t)(p.work.pre_cp()[chain / Hv] + c);
          // scalar gate: the k-head's [q~ ; k~]; per-channel decay: the
          // v-head's decayed [q^ ; k^]
          const unsigned char* qk =
              kKda ? static_cast<const unsigned char*>(p.scr_qh) + (gi * Hv + h) * (2 * KB_STRIDE)
                   : static_cast<const unsigned char*>(p.scr_qk) + (gi * p.Hk + kh) * (2 * KB_STRIDE);
          const unsigned char* wt = static_cast<const unsigned char*>(p.scr_w) + (gi * Hv + h) * (2 * BOX);
          const unsigned char* ut = static_cast<const unsigned char*>(p.scr_u) + (gi * Hv + h) * (2 * BOX);
          const unsigned char* pt = static_cast<const unsigned char*>(p.scr_p) + (gi * Hv + h) * BOX;
          const unsigned char* gt = static_cast<const unsigned char*>(p.scr_g) + (gi * p.Hk + kh) * 1024;
          unsigned char* st = sm + b * ST_BYTES;
          mbar_arrive_expect_tx(&full[b], ST_BYTES);
          bulk_g2s(st + ST_QW, wt, BOX, &full[b]);
          bulk_g2s(st + ST_QW + KB_STRIDE, wt + BOX, BOX, &full[b]);
          bulk_g2s(st + ST_QW + BOX, qk, BOX, &full[b]);
          bulk_g2s(st + ST_QW + KB_STRIDE + BOX, qk + KB_STRIDE, BOX, &full[b]);
          bulk_g2s(st + ST_K, qk + BOX, BOX, &full[b]);
          bulk_g2s(st + ST_K + BOX, qk + KB_STRIDE + BOX, BOX, &full[b]);
          bulk_g2s(st + ST_U, ut, 2 * BOX, &full[b]);
          bulk_g2s(st + ST_P, pt, BOX, &full[b]);
          bulk_g2s(st + ST_G, gt, 1024, &full[b]);
        }
        if (dead || end) break;
      }
      if (dead) atomicOr((unsigned*)&hdr[kErr], GDN_FLAG_TIMEOUT);
    }
    __syncwarp();
  } else {
    // =========================== compute warps ===========================
    const uint32_t lane = (uint32_t)(tid & 96) << 16;  // TMEM lane quarter of this warp
    const int v = tid & 127;                           // TMEM lane = state row v
    const int hf = tid >> 7;                           // column half
    __nv_bfloat16* __restrict__ out = reinterpret_cast<__nv_bfloat16*>(p.out);
    int okslot = 0;
    auto wait_c = [&](uint64_t* bar, uint32_t parity) -> bool {
      if (tid == 0) ok_c[okslot] = mbar_wait_bounded(bar, parity) ? 1 : 0;
      cbar();
      const bool r = ok_c[okslot] != 0;
      okslot ^= 1;
      return r;
    };
    uint32_t ph_y = 0, ph_s = 0;
    bool s_busy = false;   // an MMA-S commit not waited for yet
    bool pending = false;  // outputs of the previous chunk not written yet
    int p_row = 0, p_n = 0, p_h = 0, p_ob = 0;
    bool dead = false;
    int next_gate = kBarD1;  // the gate the MMA warp waits at
    float amax = 0.f;
    // outputs i = 32 hf .. 32 hf + 31 of the pending chunk at this thread's
    // v: e^{G_i} D^T[:, 64 + i] + D^T[:, i] (tcgen05.ld and the pair exchange
    // are warp-collective, the token predicate guards the stores only)
    auto flush = [&]() {
      float o[32], y[32];
      tc::tmem_ld32(tmem + lane + TM_D + p_ob * 128 + CH + hf * 32, o);
      tc::tmem_ld32(tmem + lane + TM_D + p_ob * 128 + hf * 32, y);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 f = *reinterpret_cast<const float4*>(&EF[p_ob][hf * 32 + e]);
        fma2v(o[e], o[e + 1], f.x, f.y, y[e], y[e + 1]);
        fma2v(o[e + 2], o[e + 3], f.z, f.w, y[e + 2], y[e + 3]);
      }
      // a lane pair (v, v ^ 1) writes the two v of one token with one 4-byte
      // store: the even lane the even tokens, the odd lane the odd ones
      const bool odd = (v & 1) != 0;
      uint32_t* dst = reinterpret_cast<uint32_t*>(
          out + ((size_t)(p_row + hf * 32 + (odd ? 1 : 0)) * Hv + p_h) * D + (v & ~1));
      const size_t step2 = (size_t)Hv * D;  // two rows, in 4-byte words
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float mine = odd ? o[2 * m + 1] : o[2 * m];
        const float give = odd ? o[2 * m] : o[2 * m + 1];
        const float got = __shfl_xor_sync(0xffffffffu, give, 1);
        const uint32_t w = odd ? tc::pack2(got, mine, (__nv_bfloat16*)nullptr)
                               : tc::pack2(mine, got, (__nv_bfloat16*)nullptr);
        if (hf * 32 + 2 * m + (odd ? 1 : 0) < p_n) dst[m * step2] = w;
      }
    };
    for (int k = 0;; ++k) {
      const int b = k % kStages;
      // ---- the chunk's tiles have landed and the previous chunk's state
      // update is done (S readable): one wait by thread 0, one barrier
      if (tid == 0) {
        bool okw = mbar_wait_bounded(&full[b], (k / kStages) & 1);
        if (okw && s_busy) okw = mbar_wait_bounded(&mma_s, ph_s);
        ok_c[okslot] = okw ? 1 : 0;
      }
      cbar();
      const bool okt = ok_c[okslot] != 0;
      okslot ^= 1;
      if (!okt) { dead = true; break; }
      if (s_busy) {
        ph_s ^= 1;
        s_busy = false;
        tc::fence_after_sync();
      }
      const ChunkDesc d = desc[b];
      if (d.flags & 4) break;
      unsigned char* st = sm + b * ST_BYTES;
      const float* GT = reinterpret_cast<const float*>(st + ST_G);
      const int r2 = d.h % R;
      const int n = d.n;
      // scalar gate: G_C of the chunk; per-channel decay: e^{Gamma_C[k]} of
      // every key channel k, fp32 [2 v-heads][128]
      const float GC = kKda ? 0.f : GT[(n - 1) * 4 + 2 * r2];
      const float* DK = GT + r2 * D;
      if (n < CH) {
        // u rows past the sequence -> 0: the identity product reads every row
        for (int t = tid; t < (CH - n) * 16; t += kCompute)
          *reinterpret_cast<uint4*>(st + ST_U + (t & 8 ? BOX : 0) + (n + (t >> 4)) * 128 + (t & 7) * 16) =
              make_uint4(0, 0, 0, 0);
      }
      // ---- state hand-over: S0 -> fp16 A operand, S <- e^{G_C} S0
      // (this thread: row v, k = 32 hf .. 32 hf + 31, then 64 + the same;
      // each pass releases its K-block of the D product as soon as its fp16
      // copy is in, and the scaled state goes back while the product runs:
      // the state update waits for it with the U^T store)
      tc::fence_proxy_async_smem();  // the zeroed u rows
      {
        const float dc = __expf(GC);
        const float* S_r = reinterpret_cast<const float*>(p.layer_base + (size_t)d.rblk * p.stride +
                                                          p.rec_off) + (size_t)d.h * D * D;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int k0 = hh * 64 + hf * 32;
          float srow[32];
          if (d.flags & 1) {
            // a chain's first chunk: its past state, or zero (the trash block,
            // which stays zero) without touching memory
#pragma unroll
            for (int kk = 0; kk < 32; ++kk) srow[kk] = d.rblk != 0 ? S_r[(size_t)(k0 + kk) * D + v] : 0.f;
          } else {
            tc::tmem_ld32(tmem + lane + TM_S + k0, srow);
            tc::tmem_wait_ld();
          }
          float m4[4] = {0.f, 0.f, 0.f, 0.f};
          uint32_t w16[16];
#pragma unroll
          for (int kk = 0; kk < 32; kk += 2) {
            m4[(kk >> 1) & 3] = max_abs3(m4[(kk >> 1) & 3], srow[kk], srow[kk + 1]);
            w16[kk >> 1] = tc::pack2(srow[kk], srow[kk + 1], (E*)nullptr);
          }
          amax = fmaxf(amax, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
          tc::tmem_st16u(tmem + lane + TM_S0 + k0 / 2, w16);
          tc::tmem_wait_st();
          tc::fence_before_sync();
          if (hh == 0) mma_release<kBarD1>();  // D^T = S0[:, :64] [-w ; q~][:, :64]^T
          else mma_release<kBarD>();           // D^T += S0[:, 64:] [-w ; q~][:, 64:]^T + u^T
          if constexpr (kKda) {
#pragma unroll
            for (int kk = 0; kk < 32; kk += 4) {
              const float4 f = *reinterpret_cast<const float4*>(DK + k0 + kk);
              mul2v(srow[kk], srow[kk + 1], f.x, f.y);
              mul2v(srow[kk + 2], srow[kk + 3], f.z, f.w);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < 32; kk += 2) mul2(srow[kk], srow[kk + 1], dc);
          }
          tc::tmem_st32(tmem + lane + TM_S + k0, srow);
        }
      }
      next_gate = kBarS;
      const int ob = k & 1;
      const uint32_t dcol = TM_D + ob * 128;
      // ---- while the tensor core runs: k~_j <- e^{G_C - G_j} k~_j, rows past
      // the sequence -> 0 (thread: row j = tid % 64 of box (tid / 64) % 2,
      // four of its 16-byte chunks in an order rotated by j, which keeps the
      // accesses conflict-free), and the output scales e^{G_i}
      {
        const int j = tid & 63;
        unsigned char* krow = st + ST_K + ((tid >> 6) & 1) * BOX + j * 128;
        const int c0 = 4 * (tid >> 7);
        if (kKda) {
          // the per-channel decays are in the tile already; rows past n are
          // zero there too, zeroed again like the scalar tile's
          if (j >= n) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *reinterpret_cast<uint4*>(krow + (((c0 + c + j) & 7) << 4)) = make_uint4(0, 0, 0, 0);
          }
        } else if (j < n) {
          const float ds = __expf(GC - GT[j * 4 + 2 * r2]);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint4* q = reinterpret_cast<uint4*>(krow + (((c0 + c + j) & 7) << 4));
            float k8[8];
            unpack8(*q, k8);
#pragma unroll
            for (int e = 0; e < 8; e += 2) mul2(k8[e], k8[e + 1], ds);
            *q = pack8(k8);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            *reinterpret_cast<uint4*>(krow + (((c0 + c + j) & 7) << 4)) = make_uint4(0, 0, 0, 0);
        }
        if (tid < CH) EF[ob][tid] = tid < n ? (kKda ? 1.f : __expf(GT[tid * 4 + 2 * r2])) : 0.f;
        tc::fence_proxy_async_smem();
      }
      if (!wait_c(&mma_y, ph_y)) { dead = true; break; }
      ph_y ^= 1;
      tc::fence_after_sync();
      // ---- U^T columns j = 32 hf .. 32 hf + 31 -> fp16 A operand (past n: 0)
      {
        float dv[32];
        tc::tmem_ld32(tmem + lane + dcol + hf * 32, dv);
        tc::tmem_wait_ld();
        float m4[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t w16[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float a0 = hf * 32 + e < n ? dv[e] : 0.f;
          const float a1 = hf * 32 + e + 1 < n ? dv[e + 1] : 0.f;
          m4[(e >> 1) & 3] = max_abs3(m4[(e >> 1) & 3], a0, a1);
          w16[e >> 1] = tc::pack2(a0, a1, (E*)nullptr);
        }
        amax = fmaxf(amax, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
        tc::tmem_st16u(tmem + lane + TM_UT + hf * 16, w16);
        tc::tmem_wait_st();
      }
      tc::fence_before_sync();
      mma_release<kBarS>();  // S += U^T (e^{G_C - G} k~); D^T[:, ..64] = U^T P^T
      next_gate = kBarD1;
      // ---- the previous chunk's outputs (its U^T P^T finished before this
      // chunk's D product)
      if (pending) flush();
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
        // the state and U entered tensor-core operands in fp16: if any value
        // of this chain left that range, its block keeps the old state and the
        // chain is rerun token-serially (outputs included); else the final
        // state goes to the block
        const bool bad = cbar_or(!(amax <= kF16Max));
        amax = 0.f;
        if (bad) {
          if (tid == 0) mark_redo(p.work, d.kpre, d.h);
        } else {
          float* S_w = reinterpret_cast<float*>(p.layer_base + (size_t)d.wblk * p.stride +
                                                p.rec_off) + (size_t)d.h * D * D;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float srow[32];
            tc::tmem_ld32(tmem + lane + TM_S + hf * 64 + half * 32, srow);
            tc::tmem_wait_ld();
#pragma unroll
            for (int kk = 0; kk < 32; ++kk) S_w[(size_t)(hf * 64 + half * 32 + kk) * D + v] = srow[kk];
          }
        }
      }
    }
    // let the MMA warp out of the gate it waits at
    if (tid == 0) mma_stop = 1;
    cbar();
    if (next_gate == kBarD1) mma_release<kBarD1>();
    else mma_release<kBarS>();
    if (dead && tid == 0) atomicOr((unsigned*)&hdr[kErr], GDN_FLAG_TIMEOUT);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (tid < 32) tc::tmem_dealloc(tmem, TM_COLS);
}

}  // namespace

cudaError_t launch_seq(const FwdParams& p, int grid, bool kda, cudaStream_t stream) {
  auto kern = kda ? seq_kernel<true> : seq_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), SMEM_BYTES, stream, p);
}

}  // namespace gdn

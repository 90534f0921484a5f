// State-independent chunk products of the per-channel-decay (KDA) rule's
// prefill, per (64-token chunk, v-head) on a persistent grid (one CTA per SM
// walking its items, the next item's inputs loaded during the current one),
// between the conv-only pass of cintra_kernel (which leaves the chunk's
// [q~ ; k~] tile and v tiles in the prefill scratch) and the recurrence
// kernel's KDA instance.
//
// The rule (Kimi Linear's delta rule with a decay per key channel, applied to
// the key columns of S[v][k]) in chunk form, with alpha_s[c] = e^{g_s[c]},
// Gamma_i[c] = sum_{s <= i} g_s[c] inside the chunk and Gamma_C that of the
// chunk's last token:
//   A_ij = beta_i sum_c k~_i[c] k~_j[c] e^{Gamma_i[c] - Gamma_j[c]}   (j < i)
//   P_ij =        sum_c q~_i[c] k~_j[c] e^{Gamma_i[c] - Gamma_j[c]}   (j <= i)
//   T = (I + A)^{-1},  u = T diag(beta) v,  w = T diag(beta) (k~ e^{Gamma})
//   q^_i = q~_i e^{Gamma_i},  k^_j = k~_j e^{Gamma_C - Gamma_j}
// and the recurrence kernel then forms U = u - w S0^T, O = q^ S0^T + P U and
// S = S0 Diag(e^{Gamma_C}) + U^T k^.  Every decay factor above is a product
// of alphas over a token range (all <= 1), so this kernel takes no pairwise
// exponentials and no ratios of products: each thread (channel pair, 8-token
// block) forms the running products inside its block, forward and backward,
// and every factor is one of them times the totals E8 of whole blocks:
//   q^ and -k~ e^{Gamma} from the chunk start, k^ to its end, e^{Gamma_C};
//   for the three 16-token sub-chunks I = 1..3, with r the last token before
//   I: L_I = [q~ ; k~]_I e^{Gamma_i - Gamma_r} and R_I = k~_{j <= r}
//   e^{Gamma_r - Gamma_j}, so that the off-diagonal 16 x 16 blocks of A and P
//   are plain products L_I R_I^T (mma.sync, fp16 operands <= 1, fp32
//   accumulation);
//   inside each diagonal 16 x 16 block, with m its eighth token, the
//   lower-left 8 x 8 quadrant the same way (L'_I = [q~ ; k~]_i e^{Gamma_i -
//   Gamma_m}, R'_I = k~_j e^{Gamma_m - Gamma_j}), and the two diagonal 8 x 8
//   blocks by running products per pair column j (fp32, CUDA cores).
// Then the shared blocked solve for T, T diag(beta) as an fp16 operand, and u
// and -w on tcgen05 (fp32 in tensor memory).  Every tile leaves in the layout
// the recurrence kernel loads: [q^ ; k^] (per v-head) by plain stores as its
// rows are formed, P, u and -w by bulk copy, and e^{Gamma_C} into the
// k-head's gate tile.  A value of T diag(beta), u or
// w outside the fp16 range sends the (sequence, v-head) chain to the
// token-serial redo.
#include <cuda.h>

#include <type_traits>

#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"
#include "gdn_solve.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int D = 128;
constexpr int CH = 64;
constexpr int R = 2;  // v-heads per k-head
constexpr int kThreads = 512;
constexpr int kCtr = 480;  // the thread that fetches the item counter (a helper warp's)
constexpr uint32_t BOX = 8192;         // 64 rows x 128 B
constexpr uint32_t KB_STRIDE = 16384;  // K-blocks of a 128-row [q ; k] tile
constexpr int AP = solve::AP;
constexpr int LRP = 136;  // pitch (halves) of the L / R rows: conflict-free ldmatrix
constexpr float kF16Max = 65000.f;

// Shared memory (offsets from a 1024-byte aligned base):
//   QK  [q~ ; k~] of the k-head (loaded; the next item's lands here once the
//       A / P blocks have read it)
//   V   v of the v-head: 2 boxes of 64 channels x 64 tokens (loaded)
//   LM  the mid-block operands of the four 16-token blocks I: 24 rows each,
//       L'_I (8 q rows, 8 k rows) and R'_I (8 k rows), fp16 [96][LRP]
//   NK  -k~ e^{Gamma}: 2 token-major boxes (MN-major B operand of -w)
//   AL  alpha fp32 [64 tokens][128 channels]
//   LR  L_1..L_3 (32 rows each: 16 q rows, 16 k rows), then R_1..R_3 (16,
//       32, 48 rows), fp16 [192][LRP]; after the products: the T diag(beta)
//       operand (128 rows x 64 tokens, rows 64.. zero), written by the solve,
//       and at 16 KiB the solve's B blocks, then the u and -w staging tiles
//   PT  P fp16 [64 i][64 j] (K-major B operand of the output product)
//   AT  A, then T, fp32 [64][AP]
//   GB  beta fp32 [64]
//   E8  alpha products over each 8-token block, fp32 [8 blocks][128 channels]
constexpr uint32_t OFF_QK = 0;
constexpr uint32_t OFF_V = 32768;
constexpr uint32_t OFF_LM = 49152;
constexpr uint32_t OFF_NK = 81920;
constexpr uint32_t OFF_AL = 98304;
constexpr uint32_t OFF_LR = 131072;
constexpr uint32_t OFF_UW = OFF_LR + 16384;  // u, then -w: 2 boxes each
constexpr uint32_t OFF_Z = OFF_UW;  // the solve's B blocks (the staging is free then)
constexpr uint32_t OFF_AU = OFF_LR;
constexpr uint32_t OFF_PT = 184320;
constexpr uint32_t OFF_AT = OFF_PT + BOX;
constexpr uint32_t OFF_GB = OFF_AT + CH * AP * 4;
constexpr uint32_t OFF_E8 = OFF_GB + CH * 4;
constexpr uint32_t SMEM_BYTES = OFF_E8 + 8 * D * 4 + 1024;
constexpr int kLRows = 96;  // rows of L_1..L_3
static_assert(OFF_LR + 192 * LRP * 2 <= OFF_PT, "L / R rows");
static_assert(OFF_Z + solve::kZFloats * 4 <= OFF_PT, "solve blocks");
static_assert(OFF_LM + 96 * LRP * 2 <= OFF_NK, "mid-block rows");
static_assert(OFF_UW + 4 * BOX <= OFF_PT && OFF_UW % 1024 == 0, "u / -w staging");
static_assert(OFF_PT % 1024 == 0 && OFF_AU % 1024 == 0, "operand tiles on 1024-byte boundaries");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory of one CTA");
constexpr uint32_t TM_COLS = 256;  // u (0..127), -w (128..255)

__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, int* flag) {
  if (threadIdx.x == 0) *flag = mbar_wait_bounded(bar, parity) ? 1 : 0;
  __syncthreads();
  return *flag != 0;
}

// channel pair (c, c + 1) of row r of a 128-row [q ; k] tile / of a
// token-major 2-box tile
__device__ __forceinline__ uint32_t qk_off(int r, int c) {
  return (uint32_t)(c >> 6) * KB_STRIDE + tc::sw128_offset(r, c & 63);
}
__device__ __forceinline__ uint32_t box_off(int r, int c) {
  return (uint32_t)(c >> 6) * BOX + tc::sw128_offset(r, c & 63);
}
__device__ __forceinline__ float2 ld_h2(const unsigned char* p) {
  return __half22float2(*reinterpret_cast<const __half2*>(p));
}
__device__ __forceinline__ void st_h2(unsigned char* p, float a, float b) {
  *reinterpret_cast<__half2*>(p) = __floats2half2_rn(a, b);
}
__device__ __forceinline__ uint4 pack8(const float* v) {
  uint4 w;
  w.x = tc::pack2(v[0], v[1], (__half*)nullptr);
  w.y = tc::pack2(v[2], v[3], (__half*)nullptr);
  w.z = tc::pack2(v[4], v[5], (__half*)nullptr);
  w.w = tc::pack2(v[6], v[7], (__half*)nullptr);
  return w;
}

// Warp-level fp16 products (mma.sync m16n8k16, fp32 accumulation) with
// ldmatrix fragment loads.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t (&r)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4],
                                        const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Packed fp32 pairs (one fma.rn.f32x2 / mul.rn.f32x2 on sm_100 and later).
__device__ __forceinline__ unsigned long long f2p(float lo, float hi) {
  return (unsigned long long)__float_as_uint(lo) | ((unsigned long long)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// 4 fp16 (8 bytes) -> 2 packed fp32 pairs
__device__ __forceinline__ void ld_h4p(const unsigned char* p, unsigned long long* v) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
  v[0] = f2p(a.x, a.y);
  v[1] = f2p(b.x, b.y);
}

// named barrier 1 over warps 0..5 (the solve)
__device__ __forceinline__ void solve_bar() { asm volatile("bar.sync 1, 192;" ::: "memory"); }

// log2(1 + t) on [0, 1] as a degree-8 polynomial, coefficients of t^0 ..
// t^8: the least-squares fit in the Chebyshev basis over 4000 Chebyshev nodes
// of [0, 1], converted to the monomial basis and rounded to fp32; evaluated
// by Horner's rule in fp32 its largest absolute error is 1.7e-7 (a CPU test
// checks it against the exact function).
__device__ constexpr float kLog2OnePlus[9] = {
    4.886357985e-08f, 1.442686796e+00f, -7.211146355e-01f,
    4.783235490e-01f, -3.459960222e-01f, 2.392316610e-01f,
    -1.345342547e-01f, 5.027750880e-02f, -8.874696679e-03f};

__device__ __forceinline__ float ex2_fast(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// softplus(x) / ln 2 = log2(1 + e^x) = max(x, 0) log2 e + log2(1 + 2^{-|x| log2 e})
// with one MUFU operation (the exponential) and the polynomial: an absolute
// error of a few 1e-7, which moves e^{-e^{A_log} softplus} by a relative
// e^{A_log} ln 2 times that (below 1e-5 at e^{A_log} = 16).  The gates take
// three transcendental operations per value on the MUFU pipe without it.
__device__ __forceinline__ float softplus_log2(float x) {
  constexpr float kLog2e = 1.4426950408889634f;
  const float t = ex2_fast(-fabsf(x) * kLog2e);
  float r = kLog2OnePlus[8];
#pragma unroll
  for (int i = 7; i >= 0; --i) r = fmaf(r, t, kLog2OnePlus[i]);
  return fmaxf(x, 0.f) * kLog2e + r;
}

// The gate inputs of one item, copied asynchronously (cp.async: nothing
// held in registers while in flight) into the mid-block rows' space, which is
// free from the solve until the next item's products: the a tile [64
// tokens][128 channels] bf16 (16-byte copies, rows past the chunk's end
// skipped), dt_bias [128] and A_log of the head, and per token the aligned
// word of b that holds the head's value (Hv is even).  The copies are waited
// for by every thread before a barrier.
constexpr uint32_t OFF_GS = OFF_LM;
constexpr uint32_t OFF_GSD = OFF_GS + CH * D * 2;
constexpr uint32_t OFF_GSL = OFF_GSD + D * 4;
constexpr uint32_t OFF_GSB = OFF_GSL + 16;
static_assert(OFF_GSB + CH * 4 <= OFF_LM + 96 * LRP * 2, "gate staging");
__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t saddr, const void* g) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void stage_gates(const FwdParams& p, int4 rec, int h, int tid,
                                            uint32_t sbase) {
  const int Hv = p.Hv, row0 = rec.x, n = rec.y;
  const unsigned char* av = static_cast<const unsigned char*>(p.a);
  // all on warps 4..15 (warps 0..3 run the solve and thread 0 drives the
  // bulk copies: they issue none and never wait for these): 16-byte pieces
  // q = tid - 128 + 384 e
  const int u0 = tid - 2 * CH;
  if (u0 < 0) return;
#pragma unroll
  for (int e = 0; e < 3; ++e) {
    const int q = u0 + e * (kThreads - 2 * CH), r = q >> 4, ch = q & 15;
    if (q < CH * 16 && r < n)
      cp_async16(sbase + OFF_GS + r * (D * 2) + ch * 16,
                 av + ((size_t)(row0 + r) * Hv + h) * (D * 2) + ch * 16);
  }
  if (u0 < D) cp_async4(sbase + OFF_GSD + 4 * u0, p.dt_bias + (size_t)h * D + u0);
  if (u0 == D) cp_async4(sbase + OFF_GSL, p.A_log + h);
  const int tb = tid - 3 * CH - 1;
  if (tb >= 0 && tb < n && tb < CH)
    cp_async4(sbase + OFF_GSB + 4 * tb,
              reinterpret_cast<const __nv_bfloat16*>(p.b) + (size_t)(row0 + tb) * Hv + (h & ~1));
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Persistent: CTA blockIdx.x takes the items (chunk, v-head) blockIdx.x,
// + gridDim.x, ... (item = chunk * Hv + v-head, so that the two v-heads of a
// k-head run side by side and share its [q~ ; k~] tile in L2).  The next
// item's record and gate inputs are read during the current one's solve and
// its tiles are loaded during the current one's last products, so an item
// starts with its inputs on chip.
__global__ void __launch_bounds__(kThreads, 1) kintra_kernel(FwdParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t ldbar, mbar, rbar;
  __shared__ uint32_t tmem_slot;
  __shared__ int flag;
  __shared__ int s_ni;  // the CTA's next item (a dynamic counter hands them out)
  __shared__ int4 s_next;  // the next item's record (by bulk copy on rbar)
  pdl_wait_then_release();
  int32_t* hdr = p.work.header();
  const int Hk = p.Hk, Hv = p.Hv;
  // items: every chunk of the scheduler's records (first packed row, valid
  // tokens, chunk index inside its sequence, sequence) times the v-heads.  A
  // chain the conv pass already sent to the redo still gets its tiles: the
  // recurrence skips it, so they are never read (and no load waits on the
  // redo masks here)
  const int n_items = hdr[kPreChunks] * Hv;
  int item = blockIdx.x;
  if (item >= n_items) return;
  const int4* recs = reinterpret_cast<const int4*>(p.scr_c);
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t sbase = smem_u32(sm);
  float* AL = reinterpret_cast<float*>(sm + OFF_AL);
  float* AT = reinterpret_cast<float*>(sm + OFF_AT);
  float* GB = reinterpret_cast<float*>(sm + OFF_GB);
  // the tiles of an item: [q~ ; k~] of its k-head (expecting the v tile too)
  // and v of its v-head, on the load barrier's next phase
  auto issue_qk = [&](int it) {
    const int g = it / Hv, hh = it % Hv;
    mbar_arrive_expect_tx(&ldbar, 2 * KB_STRIDE + 2 * BOX);
    bulk_g2s(sm + OFF_QK,
             static_cast<const unsigned char*>(p.scr_qk) + ((size_t)g * Hk + hh / R) * (2 * KB_STRIDE),
             2 * KB_STRIDE, &ldbar);
  };
  auto issue_v = [&](int it) {
    bulk_g2s(sm + OFF_V, static_cast<const unsigned char*>(p.scr_v) + (size_t)it * (2 * BOX), 2 * BOX,
             &ldbar);
  };

  if (tid == 0) {
    mbar_init(&ldbar, 1);
    mbar_init(&mbar, 1);
    mbar_init(&rbar, 1);
    fence_mbar_init();
    s_ni = (int)gridDim.x + atomicAdd(&hdr[kItemHeadK], 1);
    issue_qk(item);
    issue_v(item);
  }
  if (tid < 32) tc::tmem_alloc(&tmem_slot, TM_COLS);
  int4 rec = recs[item / Hv];
  stage_gates(p, rec, item % Hv, tid, sbase);
  if (tid >= 2 * CH) cp_async_wait_all();
  __syncthreads();
  bool ok = true;
  uint32_t it_par = 0;   // parity of this item's load and product barriers
  int pending = 1;       // 1 + parity of a load phase in flight (thread 0's view), or 0
  int rpend = 0;         // the same for the record barrier

  for (;;) {
  const int gidx = item / Hv, h = item % Hv, kh = h / R, hl = h % R;
  const int n = rec.y, kpre = rec.w;
  const int next = s_ni;
  int nn = 0;  // (thread kCtr) counter value of the item after next
  if (tid == 0 && next < n_items) {
    mbar_arrive_expect_tx(&rbar, 16);
    bulk_g2s(&s_next, recs + next / Hv, 16, &rbar);
    rpend = 1 + (int)it_par;
  }
  bool rok = true;

  // ---- gates: alpha_i[c] = e^{-e^{A_log} softplus(a_i[c] + dt_bias[c])}
  // (thread: channel pair 2 (tid % 64), tokens of the 8-token block tid / 64;
  // 1 past the end), beta_i = sigmoid(b_i) (0 past the end).  The thread
  // keeps the products inside its block (b8[t] = alpha_{8b} .. alpha_{8b+t},
  // s8[t] = alpha_{8b+t+1} .. alpha_{8b+7}) and publishes the block's total
  // b8[7] in the E8 table
  float2 b8[8], s8[8];
  {
    const int c = 2 * (tid & 63), i0 = 8 * (tid >> 6);
    const float ea = __expf(*reinterpret_cast<const float*>(sm + OFF_GSL));
    const float2 db = *reinterpret_cast<const float2*>(sm + OFF_GSD + c * 4);
    float2 al[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      al[t] = make_float2(1.f, 1.f);
      if (i0 + t < n) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(sm + OFF_GS + (i0 + t) * (D * 2) + c * 2);
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
        // alpha = e^{-ea softplus} = 2^{-ea log2(1 + e^x)}
        al[t].x = ex2_fast(-ea * softplus_log2(x.x + db.x));
        al[t].y = ex2_fast(-ea * softplus_log2(x.y + db.y));
      }
      *reinterpret_cast<float2*>(AL + (i0 + t) * D + c) = al[t];
    }
    b8[0] = al[0];
#pragma unroll
    for (int t = 1; t < 8; ++t) b8[t] = make_float2(b8[t - 1].x * al[t].x, b8[t - 1].y * al[t].y);
    s8[7] = make_float2(1.f, 1.f);
#pragma unroll
    for (int t = 6; t >= 0; --t)
      s8[t] = make_float2(s8[t + 1].x * al[t + 1].x, s8[t + 1].y * al[t + 1].y);
    reinterpret_cast<float2*>(sm + OFF_E8)[tid] = b8[7];  // E8[block][pair]
    if (tid < CH) {
      const __nv_bfloat16* bw = reinterpret_cast<const __nv_bfloat16*>(sm + OFF_GSB + 4 * tid);
      GB[tid] = tid < n ? sigmoid_f32(__bfloat162float(bw[h & 1])) : 0.f;
    }
  }
  // the previous item's tile stores have read their sources (the P tile, the
  // u / -w staging) before they are written again
  if (tid == 0) bulk_wait_read_all();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  float amax = 0.f;  // largest |value| entering an fp16 operand or the u / w scratch
  ok = cta_wait(&ldbar, it_par, &flag);
  if (!ok) break;
  pending = 0;

  {
    reinterpret_cast<uint4*>(sm + OFF_PT)[tid] = make_uint4(0, 0, 0, 0);  // P starts zero
    // ---- decay products of every operand row, thread group gr = tid / 64
    // (the 8-token block b = gr, rows i = 8 b + t) and channel pair c = 2 (tid
    // % 64).  Each factor is the thread's in-block product times totals E8 of
    // whole blocks, all multiplications (no ratio of products, which could
    // meet 0 / 0 where the decay underflows):
    //   L_J (16-block J = b / 2 >= 1, from its first token): b8[t], times E8
    //     of block b - 1 in the second half;
    //   L'_J (b odd, from token 16 J + 8): b8[t];   R'_J (b even, to token
    //     16 J + 7): s8[t];
    //   R_I (I = J + 1 .. 3, to token 16 I - 1): s8[t] E8_{b+1} .. E8_{2I-1};
    //   -k~ e^{Gamma} and q^ (from the chunk start): b8[t] E8_0 .. E8_{b-1};
    //   k^ (to the chunk end): s8[t] E8_{b+1} .. E8_7;
    //   e^{Gamma_C}: E8_0 .. E8_7.
    // [q^ ; k^] goes straight to its scratch tile (the [q ; k] tile's layout)
    // by plain stores, so that the [q~ ; k~] space is free once the A / P
    // blocks have read it.
    const int gr = tid >> 6, c = 2 * (tid & 63), J = gr >> 1;
    const unsigned char* QK = sm + OFF_QK;
    unsigned char* qh = static_cast<unsigned char*>(p.scr_qh) + ((size_t)gidx * Hv + h) * (2 * KB_STRIDE);
    const float2* E8 = reinterpret_cast<const float2*>(sm + OFF_E8) + (c >> 1);  // block b at E8[64 b]
    float2 pb = make_float2(1.f, 1.f);   // E8_0 .. E8_{b-1}
    float2 fl = make_float2(1.f, 1.f);   // E8_{b-1} in a second half, else 1
    float2 mr[4];                        // mr[I] = E8_{b+1} .. E8_{2I-1}
    float2 m = make_float2(1.f, 1.f);    // at the end E8_{b+1} .. E8_7
    {
#pragma unroll
      for (int bb = 0; bb < 8; ++bb) {
        const float2 e = E8[64 * bb];
        if (bb < gr) pb = make_float2(pb.x * e.x, pb.y * e.y);
        if (bb == gr - 1 && (gr & 1)) fl = e;
        if (bb > gr) m = make_float2(m.x * e.x, m.y * e.y);
        if (bb & 1) mr[(bb + 1) >> 1 & 3] = m;
      }
      if (gr == 7) {
        // e^{Gamma_C} of every key channel to the gate tile
        const float2 e = E8[64 * 7];
        reinterpret_cast<float2*>(p.scr_g)[(((size_t)gidx * Hk + kh) * R + hl) * (D / 2) + (c >> 1)] =
            make_float2(pb.x * e.x, pb.y * e.y);
      }
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int i = 8 * gr + t;
      const float2 q = ld_h2(QK + qk_off(i, c)), k = ld_h2(QK + qk_off(CH + i, c));
      if (J >= 1) {  // L_J rows (gr & 1) * 8 + t: q and k
        const float fx = b8[t].x * fl.x, fy = b8[t].y * fl.y;
        unsigned char* lr = sm + OFF_LR + (size_t)((J - 1) * 32 + (gr & 1) * 8 + t) * (LRP * 2) + c * 2;
        st_h2(lr, q.x * fx, q.y * fy);
        st_h2(lr + 16 * (LRP * 2), k.x * fx, k.y * fy);
      }
      if (gr & 1) {  // L'_J rows t (q) and 8 + t (k)
        unsigned char* lm = sm + OFF_LM + (size_t)(24 * J + t) * (LRP * 2) + c * 2;
        st_h2(lm, q.x * b8[t].x, q.y * b8[t].y);
        st_h2(lm + 8 * (LRP * 2), k.x * b8[t].x, k.y * b8[t].y);
      } else {  // R'_J row t
        st_h2(sm + OFF_LM + (size_t)(24 * J + 16 + t) * (LRP * 2) + c * 2, k.x * s8[t].x, k.y * s8[t].y);
      }
#pragma unroll
      for (int I = 1; I < 4; ++I)
        if (I > J) {  // R_I row i
          const float fx = s8[t].x * mr[I].x, fy = s8[t].y * mr[I].y;
          st_h2(sm + OFF_LR + (size_t)(kLRows + 8 * I * (I - 1) + i) * (LRP * 2) + c * 2, k.x * fx,
                k.y * fy);
        }
      const float fqx = b8[t].x * pb.x, fqy = b8[t].y * pb.y;
      st_h2(sm + OFF_NK + box_off(i, c), -k.x * fqx, -k.y * fqy);
      st_h2(qh + qk_off(i, c), q.x * fqx, q.y * fqy);
      st_h2(qh + qk_off(CH + i, c), k.x * (s8[t].x * m.x), k.y * (s8[t].y * m.y));
    }
    tc::fence_proxy_async_smem();  // -k~ e^{Gamma} (MMA operand)
    __syncthreads();

    // ---- off-diagonal blocks (I, J), I > J: [P ; A / beta] = [L_I^q ; L_I^k]
    // R_I[16 J ..]^T, one block on each odd warp 1..11 (the odd warps have the
    // shorter share of the diagonal pass below)
    if ((warp & 1) && warp < 12) {
      const int ob = warp >> 1;
      const int I = ob < 1 ? 1 : (ob < 3 ? 2 : 3);
      const int J = ob - I * (I - 1) / 2;
      const int lane = tid & 31;
      const uint32_t lbase = sbase + OFF_LR + (uint32_t)((I - 1) * 32) * (LRP * 2);
      const uint32_t rbase = sbase + OFF_LR + (uint32_t)(kLRows + 8 * I * (I - 1) + 16 * J) * (LRP * 2);
      float acc[2][2][4] = {};
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a[2][4], b[2][2];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
          ldsm_x4(lbase + (uint32_t)(mt * 16 + (lane & 15)) * (LRP * 2) + (ks * 16 + (lane >> 4) * 8) * 2,
                  a[mt]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
          ldsm_x2(rbase + (uint32_t)(nt * 8 + (lane & 7)) * (LRP * 2) + (ks * 16 + ((lane >> 3) & 1) * 8) * 2,
                  b[nt]);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) mma_f16(acc[mt][nt], a[mt], b[nt]);
      }
      const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int i = 16 * I + g + 8 * hh, j = 16 * J + nt * 8 + 2 * t4;
          st_h2(sm + OFF_PT + tc::sw128_offset(i, j), acc[0][nt][2 * hh], acc[0][nt][2 * hh + 1]);
          const float bi = GB[i];
          *reinterpret_cast<float2*>(AT + i * AP + j) =
              make_float2(bi * acc[1][nt][2 * hh], bi * acc[1][nt][2 * hh + 1]);
        }
    }
    // ---- lower-left 8 x 8 quadrants of the diagonal 16-token blocks:
    // [P ; A / beta] = [L'_I^q ; L'_I^k] R'_I^T, blocks I = 0, 1 on warp 13
    // and I = 2, 3 on warp 15
#pragma unroll 1
    for (int I = warp - 13; I < warp - 11 && warp >= 13 && (warp & 1); ++I) {
      const int lane = tid & 31;
      const uint32_t lbase = sbase + OFF_LM + (uint32_t)(24 * I) * (LRP * 2);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a[4], b[2];
        ldsm_x4(lbase + (uint32_t)(lane & 15) * (LRP * 2) + (ks * 16 + (lane >> 4) * 8) * 2, a);
        ldsm_x2(lbase + (uint32_t)(16 + (lane & 7)) * (LRP * 2) + (ks * 16 + ((lane >> 3) & 1) * 8) * 2,
                b);
        mma_f16(acc, a, b);
      }
      const int g = lane >> 2, t4 = lane & 3;
      const int i = 16 * I + 8 + g, j = 16 * I + 2 * t4;
      st_h2(sm + OFF_PT + tc::sw128_offset(i, j), acc[0], acc[1]);
      const float bi = GB[i];
      *reinterpret_cast<float2*>(AT + i * AP + j) = make_float2(bi * acc[2], bi * acc[3]);
    }
    // ---- diagonal 8 x 8 blocks: warp (block B, column quad cg) covers the
    // columns j = 8 B + 4 cg + jj (jj < 4) and the rows from its first
    // column's on; lane l holds the channels 4 l .. 4 l + 3 and, per column,
    // the running decay product f = e^{Gamma_i - Gamma_j} on them.  A row's
    // eight sums (P and A / beta of the four columns) meet over the 32 lanes
    // in a butterfly (three halving levels, two plain ones); every row's
    // results wait in registers and are stored at the end.
    {
      const int B = warp >> 1, cg = warp & 1, lane = tid & 31;
      const int cl = 4 * lane;
      auto walk = [&](auto rows) {
        constexpr int NR = decltype(rows)::value, T0 = 8 - NR;  // T0 = 4 cg
        unsigned long long kj[4][2], f[4][2];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          ld_h4p(QK + qk_off(CH + 8 * B + T0 + jj, cl), kj[jj]);
          f[jj][0] = f[jj][1] = f2p(1.f, 1.f);
        }
        float res[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          const int tt = T0 + r, i = 8 * B + tt;
          const float4 a = *reinterpret_cast<const float4*>(AL + i * D + cl);
          const unsigned long long a01 = f2p(a.x, a.y), a23 = f2p(a.z, a.w);
          unsigned long long q2[2], k2[2];
          ld_h4p(QK + qk_off(i, cl), q2);
          ld_h4p(QK + qk_off(CH + i, cl), k2);
          float w[8];  // P of columns 0..3, then A / beta
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            if (tt > T0 + jj) {
              f[jj][0] = mul2(f[jj][0], a01);
              f[jj][1] = mul2(f[jj][1], a23);
            }
            const unsigned long long kf0 = mul2(kj[jj][0], f[jj][0]), kf1 = mul2(kj[jj][1], f[jj][1]);
            const unsigned long long sp2 = fma2(q2[1], kf1, mul2(q2[0], kf0));
            const unsigned long long sa2 = fma2(k2[1], kf1, mul2(k2[0], kf0));
            w[jj] = __uint_as_float((uint32_t)sp2) + __uint_as_float((uint32_t)(sp2 >> 32));
            w[4 + jj] = __uint_as_float((uint32_t)sa2) + __uint_as_float((uint32_t)(sa2 >> 32));
          }
          // lanes xor 16, 8, 4 each keep half of the values (the upper half
          // where the bit is set); lane l ends with w[(l >> 2) & 7] summed
          // over the eight lanes that share l & 3, then xor 2, 1 finish it
          float w4[4], w2[2];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const bool hi = lane & 16;
            w4[k] = (hi ? w[4 + k] : w[k]) + __shfl_xor_sync(0xffffffffu, hi ? w[k] : w[4 + k], 16);
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const bool hi = lane & 8;
            w2[k] = (hi ? w4[2 + k] : w4[k]) + __shfl_xor_sync(0xffffffffu, hi ? w4[k] : w4[2 + k], 8);
          }
          const bool hi = lane & 4;
          float x = (hi ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, hi ? w2[0] : w2[1], 4);
          x += __shfl_xor_sync(0xffffffffu, x, 2);
          x += __shfl_xor_sync(0xffffffffu, x, 1);
          res[r] = x;
        }
        if ((lane & 3) == 0) {
          const int idx = (lane >> 2) & 7, jj = idx & 3;
          const int j = 8 * B + T0 + jj;
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            const int tt = T0 + r, i = 8 * B + tt;
            if (idx < 4) {
              if (tt >= T0 + jj) *reinterpret_cast<__half*>(sm + OFF_PT + tc::sw128_offset(i, j)) = __float2half_rn(res[r]);
            } else if (tt > T0 + jj) {
              AT[i * AP + j] = GB[i] * res[r];
            }
          }
        }
      };
      if (cg)
        walk(std::integral_constant<int, 4>{});
      else
        walk(std::integral_constant<int, 8>{});
    }
    tc::fence_proxy_async_smem();  // the P tile
    __syncthreads();
    if (tid == 0) {
      bulk_s2g(static_cast<unsigned char*>(p.scr_p) + ((size_t)gidx * Hv + h) * BOX, sm + OFF_PT, BOX);
      bulk_commit();
      // nothing reads the [q~ ; k~] tile any more: the next item's
      if (next < n_items) {
        issue_qk(next);
        pending = 1 + (int)(it_par ^ 1u);
      }
    }
    // the next item's record (thread 0 read it at this item's start) and gate
    // inputs (the mid-block rows are read), in flight during the rest of this
    // item
    if (next < n_items) {
      rok = cta_wait(&rbar, it_par, &flag);
      if (rok && tid == 0) rpend = 0;
      if (rok) {
        rec = s_next;
        stage_gates(p, rec, next % Hv, tid, sbase);
      }
    }
    // ---- T = (I + A)^{-1} on warps 0..5 (diagonal blocks by threads 0..63,
    // then the off-diagonal blocks in four product steps, one chain per warp;
    // named barrier 1 over those 192 threads)
    // Every block of T goes to AT (fp32, for the solve's later steps) and,
    // scaled by beta_j, to the fp16 A operand T diag(beta) of the u / -w
    // products; the helper warps 6..15 zero that operand's blocks above the
    // diagonal and its rows 64..127.
    unsigned char* AU = sm + OFF_AU;
    if (warp < 6) {
      float col[16];
      const int b = (tid >> 4) & 3, m = tid & 15;
      float* Ab = AT + (16 * b) * AP + 16 * b;
      if (tid < CH) solve::diag_col(Ab, m, col);
      solve_bar();
      if (tid < CH) {
        solve::diag_col_store(Ab, m, col);
        const float bm = GB[16 * b + m];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const float t = col[r] * bm;
          amax = fmaxf(amax, fabsf(t));
          *reinterpret_cast<__half*>(AU + tc::sw128_offset(16 * b + r, 16 * b + m)) = __float2half_rn(t);
        }
      }
      solve_bar();
      float* Z = reinterpret_cast<float*>(sm + OFF_Z);
      const int lane = tid & 31, g = lane >> 2, t4 = lane & 3;
      solve::offdiag_chains<6>(AT, Z, warp, solve_bar,
                               [&](int i, int j, const float(&t0)[4], const float(&t1)[4]) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const float(&t)[4] = hh ? t1 : t0;
          const int col = 16 * j + 8 * hh + 2 * t4;
          const float b0 = GB[col], b1 = GB[col + 1];
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const float v0 = t[2 * rr] * b0, v1 = t[2 * rr + 1] * b1;
            amax = max_abs3(amax, v0, v1);
            *reinterpret_cast<__half2*>(AU + tc::sw128_offset(16 * i + g + 8 * rr, col)) =
                __floats2half2_rn(v0, v1);
          }
        }
      });
    } else {
      // a global atomic holds its thread for the round trip: a helper warp,
      // idle for most of the solve, fetches the item counter
      if (tid == kCtr && next < n_items) nn = atomicAdd(&hdr[kItemHeadK], 1);
      // zero rows 64..127 (64 x 128 B) and the six blocks above the diagonal
      // (16 rows x 32 B each) of the operand
      for (int q = tid - 192; q < 512 + 6 * 32; q += 320) {
        if (q < 512) {
          *reinterpret_cast<uint4*>(AU + (CH + (q >> 3)) * 128 + (q & 7) * 16) = make_uint4(0, 0, 0, 0);
        } else {
          const int z = q - 512, blkz = z >> 5, r = (z >> 1) & 15, hh = z & 1;
          const int bi = blkz < 3 ? 0 : (blkz < 5 ? 1 : 2);
          const int bj = blkz < 3 ? blkz + 1 : (blkz < 5 ? blkz - 1 : 3);
          *reinterpret_cast<uint4*>(AU + tc::sw128_offset(16 * bi + r, 16 * bj + 8 * hh)) =
              make_uint4(0, 0, 0, 0);
        }
      }
    }
    tc::fence_proxy_async_smem();  // T diag(beta) (MMA operand)
    tc::fence_before_sync();
    __syncthreads();
    // u = T diag(beta) v into columns 0..127, -w = T diag(beta) (-k~ e^{Gamma})
    // into 128..255 (v and -k~ e^{Gamma} as MN-major operands; rows 0..63)
    if (tid == 0) {
      tc::fence_after_sync();
      tc::mma_op(tmem, tc::Opnd{sbase + OFF_AU, 0u, false}, tc::Opnd{sbase + OFF_V, BOX, true},
                 CH / 16, tc::idesc_f16_f32(128, 128, false, true), false);
      tc::mma_op(tmem + 128, tc::Opnd{sbase + OFF_AU, 0u, false}, tc::Opnd{sbase + OFF_NK, BOX, true},
                 CH / 16, tc::idesc_f16_f32(128, 128, false, true), false);
      tc::commit(&mbar);
    }
    ok = cta_wait(&mbar, it_par, &flag) && rok;
    // the products have read v: the next item's v tile
    if (ok && tid == 0 && next < n_items) issue_v(next);
  }
  if (ok) {
    tc::fence_after_sync();
    // rows 0..63: u and -w of token r128 into the staging tiles
    // (thread: TMEM lane r128, column quarter cq4 of each 128-column part)
    const uint32_t lane = (uint32_t)(tid & 96) << 16;
    const int r128 = tid & 127, cq4 = tid >> 7;
    if (r128 < CH) {
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        unsigned char* box = sm + OFF_UW + part * (2 * BOX) + (cq4 >> 1) * BOX;
        float vv[32];
        tc::tmem_ld32(tmem + lane + part * 128 + cq4 * 32, vv);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 2) amax = max_abs3(amax, vv[e], vv[e + 1]);
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8)
          *reinterpret_cast<uint4*>(box + tc::sw128_offset(r128, (cq4 & 1) * 32 + g8 * 8)) =
              pack8(vv + g8 * 8);
      }
    }
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      const size_t tile = ((size_t)gidx * Hv + h) * (2 * BOX);
      bulk_s2g(static_cast<unsigned char*>(p.scr_u) + tile, sm + OFF_UW, 2 * BOX);
      bulk_s2g(static_cast<unsigned char*>(p.scr_w) + tile, sm + OFF_UW + 2 * BOX, 2 * BOX);
      bulk_commit();
    }
  }
  if (!ok) break;
  // T diag(beta), u and w enter tensor-core operands or the scratch in fp16:
  // a value out of its range sends this chain to the token-serial redo
  tc::fence_before_sync();
  if (tid >= 2 * CH) cp_async_wait_all();  // the next item's gate inputs, visible after the barrier
  if (tid == kCtr && next < n_items) s_ni = (int)gridDim.x + nn;  // read after the barrier
  if (__syncthreads_or(!(amax <= kF16Max)) && tid == 0) mark_redo(p.work, kpre, h);
  if (next >= n_items) break;
  item = next;
  it_par ^= 1u;
  }  // items

  if (!ok && tid == 0) {
    atomicOr((unsigned*)&hdr[kErr], GDN_FLAG_TIMEOUT);
    // tiles still in flight for an item this CTA will not take land before
    // it ends (a bounded wait)
    if (pending) (void)mbar_wait_bounded(&ldbar, (uint32_t)(pending - 1));
    if (rpend) (void)mbar_wait_bounded(&rbar, (uint32_t)(rpend - 1));
  }
  tc::fence_before_sync();
  __syncthreads();
  if (tid < 32) tc::tmem_dealloc(tmem_slot, TM_COLS);
  // the shared-memory sources of the tile stores are read before the CTA ends;
  // the stores themselves complete with the grid (the recurrence kernel, launched
  // after it, waits for that)
  if (tid == 0) bulk_wait_read_all();
}

}  // namespace

cudaError_t launch_kintra(const FwdParams& p, int max_chunks, int num_sms, cudaStream_t stream) {
  if (max_chunks <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kintra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long items = (long long)max_chunks * p.Hv;
  const int grid = (int)(items < num_sms ? items : num_sms);
  return launch_pdl(kintra_kernel, dim3(grid), dim3(kThreads), SMEM_BYTES, stream, p);
}

}  // namespace gdn

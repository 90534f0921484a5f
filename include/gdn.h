/*
 * gdn.h -- C ABI of the GB300 (sm_103a) library for the continuous-batching
 * forward of a gated delta net layer: a varlen causal depthwise conv1d + SiLU
 * continued from each request's conv state, then the gated delta rule over
 * cu_seqlens continued from each request's recurrent state, both states held
 * in one block per request of a paged state pool.
 *
 * Sources of the operations (pages on continuous batching for linear attention
 * layers, and the gated delta rule):
 *  - "Continuous batching for linear attention layers" (PR description): a
 *    linear attention layer keeps a fixed-size state per request (the last
 *    inputs of its causal convolution and its recurrent state); an allocator
 *    keeps it in one block per request for the request's whole life, read from
 *    the zeroed trash block while the request has no past and overwritten in
 *    place by every forward; indices hold one entry per sequence; the packed
 *    batch runs as one row through a varlen convolution and kernels taking the
 *    per-sequence states through cu_seqlens.  The commit that makes layers
 *    declare their states: any number of declared states per block, each on a
 *    128-byte boundary.
 *  - transformers generation/continuous_batching/input_ouputs.py
 *    (prepare_batch_tensors, get_model_kwargs): cu_seqlens are int32
 *    cumulative query lengths [0, l0, l0+l1, ...]; graph padding repeats the
 *    last value, i.e. adds zero-length sequences.
 *  - Gated delta rule (Gated Delta Networks, Yang et al.):
 *      g_t = -exp(A_log) * softplus(a_t + dt_bias), beta_t = sigmoid(b_t),
 *      S_t = e^{g_t} S_{t-1} + beta_t (v_t - e^{g_t} S_{t-1} k_t) k_t^T,
 *      o_t = S_t q_t, q and k L2-normalised (eps 1e-6 inside the root), q
 *      scaled by 1/sqrt(d_k).
 *
 * Conventions common to every entry point:
 *  - Every tensor pointer is DEVICE memory owned by the caller, except where
 *    stated.  Nothing is retained after a call returns.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and is stream-ordered: the caller must not rewrite an input until
 *    the stream has reached the call (the engine's warmup race, where a
 *    forward read cu_seqlens that were being rewritten, is exactly this).
 *  - Return value: GDN_OK (0) or a negative GDN_ERR_* code; on error nothing
 *    was launched and nothing was written.
 *  - No entry point except gdn_get_error synchronises with the device, so
 *    gdn_varlen_forward can be captured in a CUDA graph.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define GDN_OK 0
#define GDN_ERR_NULL (-1)        /* a required pointer is NULL */
#define GDN_ERR_DIMS (-2)        /* dimensions inconsistent or unsupported */
#define GDN_ERR_RANGE (-3)       /* T, N, layer, block or size out of range */
#define GDN_ERR_ALIGN (-4)       /* a pointer or row pitch is not 16-byte aligned */
#define GDN_ERR_CUDA (-5)        /* a CUDA runtime call failed */
#define GDN_ERR_NOMEM (-6)       /* device allocation failed / buffer too small */
#define GDN_ERR_DEVICE (-7)      /* called with a different current device than the pool's */

/* Activation dtypes (x_qkv, a, b, conv weight, conv state, out). */
#define GDN_F32 0
#define GDN_BF16 1

/* Bits of the device error word (see gdn_get_error).  A flagged sequence is
 * skipped: nothing is read for it, its block and its out rows are untouched. */
#define GDN_FLAG_SEQLENS 0x1u     /* cu_seqlens[0] != 0, decreasing, or cu_seqlens[N] != T: whole batch skipped */
#define GDN_FLAG_BLOCK_RANGE 0x2u /* block index >= num_blocks */
#define GDN_FLAG_TRASH_WRITE 0x4u /* block index 0 (the trash block) given as a write target */
#define GDN_FLAG_DUPLICATE 0x8u   /* two active sequences name the same block: both skipped */
#define GDN_FLAG_TIMEOUT 0x10u    /* a kernel's bounded wait gave up (its results are incomplete) */
#define GDN_FLAG_HINT 0x20u       /* a sequence is longer than max_seqlen_hint: it was skipped */
#define GDN_FLAG_RANGE 0x40u      /* Mamba2 pools only: an SSM state entering the chunked scan's
                                     fp16 operand left the fp16 range (|value| > 65000); that
                                     sequence's results are invalid.  (The gated delta net
                                     forwards never raise it: a (sequence, v-head) whose chunked-
                                     prefill operands leave the fp16 range is recomputed by the
                                     token-serial kernel within the same call.) */

typedef struct gdn_pool gdn_pool_t;

/* Layer weights, all device pointers.
 *   conv_w  : [C][K] activation dtype, C = 2*Hk*d_k + Hv*d_v channels in the
 *             order q | k | v, head-major within each part; w[c][K-1]
 *             multiplies the current token (PyTorch depthwise conv1d taps);
 *   A_log   : [Hv] fp32;  dt_bias : [Hv] fp32. */
typedef struct {
  const void* conv_w;
  const float* A_log;
  const float* dt_bias;
} gdn_weights_t;

/* Byte layout of a pool with these dimensions, without allocating.
 * Block b of layer l starts at base + (l*num_blocks + b) * block_stride.
 * Inside a block: conv state [K-1][C] (activation dtype, oldest row first) at
 * conv_off = 0; recurrent state [Hv][d_k][d_v] fp32 at rec_off =
 * roundup(conv bytes, 128), element S_h[v][k] at ((h*d_k)+k)*d_v+v;
 * block_stride = roundup(rec_off + rec bytes, max(128, block_align)).
 * Any output pointer may be NULL.  Returns GDN_ERR_DIMS for unsupported
 * dimensions (see gdn_state_pool_create). */
int gdn_state_pool_layout_for(int num_blocks, int num_layers, int num_k_heads, int num_v_heads,
                              int d_k, int d_v, int conv_k, int act_dtype, size_t block_align,
                              size_t* block_stride, size_t* conv_off, size_t* rec_off,
                              size_t* total_bytes);

/* Create a state pool on the current CUDA device: num_layers pages of
 * num_blocks blocks, block 0 of each page is the trash block.
 * Supported: num_blocks >= 2, num_layers >= 1, d_k == d_v in {32, 64, 128},
 * num_v_heads equal to num_k_heads or twice it,
 * 2 <= conv_k <= 4, act_dtype GDN_F32 or GDN_BF16, block_align 0 (= 128) or
 * a power of two >= 128.
 * device_mem: NULL -> the library allocates (cudaMalloc) and frees at
 * destroy; otherwise caller-owned device memory of device_bytes >= the
 * layout's total_bytes, 256-byte aligned, which must outlive the pool.
 * The whole pool memory is zeroed at creation (synchronously), so every trash
 * block reads zeros; it is never written afterwards.  The pool also holds a
 * small library-allocated work area (scheduler lists and error words).
 * *out receives the handle. */
int gdn_state_pool_create(gdn_pool_t** out, int num_blocks, int num_layers, int num_k_heads,
                          int num_v_heads, int d_k, int d_v, int conv_k, int act_dtype,
                          size_t block_align, void* device_mem, size_t device_bytes);

/* Free the pool's library-owned memory (synchronises the device first).
 * NULL is accepted. */
int gdn_state_pool_destroy(gdn_pool_t* pool);

/* Layout of an existing pool and its base device address (any output may be
 * NULL; for a Mamba2 pool rec_off is the SSM state's offset).  For views and
 * byte-exact tests. */
int gdn_state_pool_layout(const gdn_pool_t* pool, size_t* block_stride, size_t* conv_off,
                          size_t* rec_off, void** base);

/* Copy block src to block dst of one layer (a fork: a block is copied on fork
 * and never shared).  dst must not be 0 (the trash block).  Stream-ordered. */
int gdn_state_pool_copy_block(gdn_pool_t* pool, int layer, int src, int dst, void* stream);

/* Prefill scratch of the pool.  Sequences longer than one token run as two
 * kernels when the pool has scratch for the call: a chunk-parallel kernel
 * (conv, norms, gates and the state-independent products of every 64-token
 * chunk) writes per-chunk tiles, and the recurrence kernel loads them.  The
 * scratch is chunk-major (its capacity is counted in 64-token chunks; a call
 * with T tokens and N sequences needs at most T/64 + min(N, T/2,
 * num_blocks - 1) + 1 of them) and shared by the layers; at the full shape
 * (d_k = d_v = 128, Hk = 16, Hv = 32) a chunk takes about 1.8 MB.  Without
 * enough scratch the same computation runs as one fused kernel (same results
 * within rounding; gdn_pool_last_prefill_path tells which one ran).  By
 * default a gdn_varlen_forward that needs more scratch than the pool holds
 * grows it first, stream-ordered on the call's stream (cudaMallocAsync /
 * cudaFreeAsync: no device synchronisation), except during stream capture,
 * where it never allocates and takes the fused kernel if the scratch is too
 * small.
 *   max_tokens > 0 : grow the scratch now to cover any call of up to
 *                    max_tokens tokens (synchronous; call it before capturing
 *                    a graph)
 *   max_tokens == 0: free the scratch and never grow it (fused kernel only)
 *   max_tokens < 0 : grow on demand again (the default)
 * Returns GDN_ERR_NOMEM if the allocation fails (the forward still works).
 * For a Mamba2 pool the scratch is the chunked scan's fp16 conv output
 * (C * 2 bytes per token), with the same three modes. */
int gdn_state_pool_reserve(gdn_pool_t* pool, int max_tokens);

/* Forward of one gated-delta-net layer over a packed batch.
 *   x_qkv           : [T][C] activation dtype, the packed pre-convolution q|k|v rows
 *   a, b            : [T][Hv] activation dtype, gate and beta pre-activations
 *   cu_seqlens      : [N+1] int32 device, cumulative starts, cu_seqlens[N] == T
 *   state_block_idx : [N] int32 device, the block of each sequence; < 0 marks a
 *                     padding entry (skipped: nothing read or written)
 *   has_past        : [N] uint8 device; 0 -> the sequence starts from the trash
 *                     block (zeros); nonzero -> from its own block
 *   weights         : host struct of device pointers (see gdn_weights_t)
 *   out             : [T][Hv][d_v] activation dtype; rows of skipped or
 *                     padding sequences are not written
 *   T, N            : host ints, T >= 0, N >= 0
 *   max_seqlen_hint : host bound on the sequence lengths (0 = unknown).  With 1
 *                     (a pure decode batch) only the decode path is launched.
 *                     Never trusted: an active sequence longer than a nonzero
 *                     hint is skipped and GDN_FLAG_HINT raised
 * Each active sequence reads its conv and recurrent state from block
 * (has_past ? idx : 0) and overwrites block idx with the new ones.
 * Zero-length sequences are no-ops.  Bad data in the device arrays (see
 * GDN_FLAG_*) is flagged in the layer's error word and the affected sequences
 * are skipped.  x_qkv, a, b, out and conv_w must be 16-byte aligned.
 * Never synchronises (the prefill scratch grows stream-ordered, see
 * gdn_state_pool_reserve); graph-capturable.  Calls on the same pool must be
 * ordered on one stream (they share the layer's scheduler work area and the
 * pool's prefill scratch).  A Mamba2 pool (gdn_ssd_pool_create) is refused
 * with GDN_ERR_DIMS. */
int gdn_varlen_forward(gdn_pool_t* pool, int layer, const void* x_qkv, const void* a,
                       const void* b, const int32_t* cu_seqlens, const int32_t* state_block_idx,
                       const uint8_t* has_past, const gdn_weights_t* weights, void* out, int T,
                       int N, int max_seqlen_hint, void* stream);

/* Forward of one layer with the per-channel-decay rule (KDA: Kimi Delta
 * Attention, the decay of the Kimi Linear and GLM5-next families that the
 * model support tracker lists): the gated delta rule with one decay per key
 * channel instead of one per head,
 *   g_t[c] = -exp(A_log[h]) * softplus(a_t[h][c] + dt_bias[h][c]),
 *   S_t = S_{t-1} Diag(e^{g_t}) + beta_t (v_t - S_{t-1} Diag(e^{g_t}) k_t) k_t^T,
 *   o_t = S_t q_t
 * (Kimi Team, "Kimi Linear", the KDA recurrence, in the S[v][k] orientation).
 * Same pool, conv, conv and recurrent states, skip rules, error flags and
 * stream contract as gdn_varlen_forward, except:
 *   a        : [T][Hv][d_k] activation dtype, one gate pre-activation per key
 *              channel of every v-head
 *   weights  : dt_bias is [Hv][d_k] fp32 (A_log stays [Hv])
 * Length-1 sequences run on an HBM-streaming decode kernel (d = 128, bf16,
 * Hv = 2 Hk, K = 4).  At that shape longer sequences run on a split chunked
 * prefill (conv pass, per-(chunk, v-head) decay products on the tensor
 * cores, the recurrence with the state in tensor memory; chains whose fp16
 * operands leave their range are recomputed token-serially in the same call)
 * when the pool's prefill scratch holds the call in this forward's layout,
 * which needs about 1.9 times the scalar rule's bytes per chunk: the forward
 * grows the scratch stream-ordered as gdn_varlen_forward does, never under
 * stream capture, and gdn_state_pool_reserve sizes it for the scalar rule
 * only.  Otherwise, and at every other shape, a token-serial kernel runs;
 * gdn_pool_last_prefill_path reports which.  Never synchronises;
 * graph-capturable. */
int gdn_kda_varlen_forward(gdn_pool_t* pool, int layer, const void* x_qkv, const void* a,
                           const void* b, const int32_t* cu_seqlens,
                           const int32_t* state_block_idx, const uint8_t* has_past,
                           const gdn_weights_t* weights, void* out, int T, int N,
                           int max_seqlen_hint, void* stream);

/* ---------------------------------------------------------------------------
 * Mamba2 mixers (the families the model support tracker lists with a conv
 * state and an SSM state per request; the groundwork it asks for is a varlen
 * scan with per-sequence states next to the varlen causal convolution).  Per
 * head h of group g = h / (H/G), per token, the SSD recurrence of
 * "Transformers are SSMs" with a scalar A per head:
 *   y     = SiLU(causal depthwise conv over the channels x | B | C)
 *   dt    = softplus(dt_raw + dt_bias[h]),  a = exp(-exp(A_log[h]) * dt)
 *   h_t   = a * h_{t-1} + dt * x_t B_t^T        (h: P x N, fp32)
 *   out_t = h_t C_t + D[h] * x_t
 * The pool is the same kind of paged pool (block 0 = trash, one block per
 * request, overwritten in place; the destroy, layout, copy_block, get_error
 * and timing entry points apply to it), with a block holding
 *   conv state [K-1][C] activation dtype at offset 0, C = H*P + 2*G*N
 *   SSM state  [H][P][N] fp32 at ssm_off = roundup(conv bytes, 128),
 *              element h_h[p][n] at ((h*P)+p)*N + n
 *   block_stride = roundup(ssm_off + SSM bytes, max(128, block_align)).
 * Supported: head_dim P in {32, 64}, d_state N in {32, 64, 128}, H % G == 0,
 * 2 <= conv_k <= 4, GDN_F32 or GDN_BF16. */
typedef struct {
  const void* conv_w;    /* [C][K] activation dtype, channels x | B | C */
  const float* A_log;    /* [H] */
  const float* dt_bias;  /* [H] */
  const float* D;        /* [H] skip weight */
} gdn_ssd_weights_t;

int gdn_ssd_pool_layout_for(int num_blocks, int num_layers, int num_heads, int head_dim,
                            int d_state, int n_groups, int conv_k, int act_dtype,
                            size_t block_align, size_t* block_stride, size_t* conv_off,
                            size_t* ssm_off, size_t* total_bytes);

/* As gdn_state_pool_create, for a Mamba2 pool. */
int gdn_ssd_pool_create(gdn_pool_t** out, int num_blocks, int num_layers, int num_heads,
                        int head_dim, int d_state, int n_groups, int conv_k, int act_dtype,
                        size_t block_align, void* device_mem, size_t device_bytes);

/* Forward of one Mamba2 mixer's conv + scan over a packed batch.
 *   xbc : [T][C] activation dtype, the packed pre-convolution x | B | C rows
 *   dt  : [T][H] activation dtype, time-step pre-activations
 *   y   : [T][H][P] activation dtype (the scan output, before the gate and
 *         norm that follow it in the mixer)
 * cu_seqlens, state_block_idx, has_past, T, N, max_seqlen_hint, the skip
 * rules, error flags and stream contract: as gdn_varlen_forward.  The pool
 * must come from gdn_ssd_pool_create (GDN_ERR_DIMS otherwise).  Length-1
 * sequences run on an HBM-streaming decode kernel when P = 64, N = 128,
 * K = 4, bf16 and H/G is 8 or 16; at that shape the longer ones run as a
 * chunked tensor-core scan (128-token chunks) when the pool's scratch holds
 * the call's T rows (grown on demand like the prefill scratch, see
 * gdn_state_pool_reserve); everything else on a token-serial kernel (one CTA
 * per sequence and head, state in registers).  The conv states of the longer
 * sequences are written by a last kernel.  Never synchronises (the scratch
 * grows stream-ordered); graph-capturable, and takes the chunked scan under
 * capture once the scratch is reserved. */
int gdn_ssd_varlen_forward(gdn_pool_t* pool, int layer, const void* xbc, const void* dt,
                           const int32_t* cu_seqlens, const int32_t* state_block_idx,
                           const uint8_t* has_past, const gdn_ssd_weights_t* weights, void* y,
                           int T, int N, int max_seqlen_hint, void* stream);

/* Bytes of prefill scratch the split prefill needs for calls of at most
 * max_tokens tokens (any number of sequences) on a pool of these dimensions
 * (for callers that provide it themselves, see gdn_varlen_forward_noalloc).
 * Returns GDN_ERR_NULL, GDN_ERR_RANGE or GDN_ERR_DIMS on bad arguments. */
int gdn_prefill_scratch_bytes(int num_blocks, int num_k_heads, int num_v_heads, int d_k, int d_v,
                              int max_tokens, size_t* bytes);

/* gdn_varlen_forward for callers that cannot allocate device memory.  The
 * pages have no counterpart to this entry point: it exists for engines that
 * plan every byte of device memory ahead and forbid runtime allocation, and
 * for code that runs under another allocator's budget, which cannot use
 * gdn_state_pool_create (it calls cudaMalloc for the pool's work area).
 * Same computation, data errors and output contract as gdn_varlen_forward,
 * without a pool handle:
 *   pool_mem, pool_bytes : caller-owned device memory of a pool with these
 *                          dimensions, laid out as gdn_state_pool_layout_for
 *                          describes (256-byte aligned, pool_bytes >= its
 *                          total_bytes); the caller keeps block 0 of every
 *                          layer zeroed (the trash block).  Bytes past
 *                          total_bytes, from the next 256-byte boundary, are
 *                          the call's prefill scratch when there are at least
 *                          gdn_prefill_scratch_bytes(..., T, ...) of them:
 *                          prefills then run on the split kernels as in
 *                          gdn_varlen_forward, else on the fused kernel
 *   num_blocks .. block_align : the pool's dimensions (as for
 *                          gdn_state_pool_create)
 *   layer, x_qkv .. max_seqlen_hint : as for gdn_varlen_forward
 *   flags_out            : optional device uint32 receiving the GDN_FLAG_*
 *                          bits raised by this call (NULL: not reported)
 * Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 * The scheduler's work area is a static device array sized for pools of at
 * most 4096 blocks (about 128 KiB, held on every GPU that loads the library
 * until the process exits); num_blocks > 4096 returns GDN_ERR_RANGE.  Every
 * call on a device shares that array, so calls whose work overlaps on the
 * GPU race: order them on one stream.  The first call on each device looks
 * up the array's device address, so make it before any stream capture on
 * that device.  Does not synchronise. */
int gdn_varlen_forward_noalloc(void* pool_mem, size_t pool_bytes, int num_blocks, int num_layers,
                               int num_k_heads, int num_v_heads, int d_k, int d_v, int conv_k,
                               int act_dtype, size_t block_align, int layer, const void* x_qkv,
                               const void* a, const void* b, const int32_t* cu_seqlens,
                               const int32_t* state_block_idx, const uint8_t* has_past,
                               const gdn_weights_t* weights, void* out, int T, int N,
                               int max_seqlen_hint, uint32_t* flags_out, void* stream);

/* ---------------------------------------------------------------------------
 * The dense neighbours of the forward in a hybrid model's gated-delta-net
 * layer (the pages name the layer; its projections are the plainest reading
 * of what surrounds the varlen forward): the input projection that produces
 * the forward's inputs and the output gate z, and the gated RMS norm and
 * output projection behind it.  Both run on the tensor cores (bf16 operands,
 * fp32 accumulation, bf16 results), allocate nothing and do not synchronise.
 * Weights are row-major [out features][in features] (the layout of a linear
 * layer's weight); every pointer 16-byte aligned; flags: optional device
 * uint32 that receives GDN_FLAG_TIMEOUT if a bounded wait gave up.
 *
 * gdn_in_proj: for every token t,
 *   x_qkv[t] = W_qkv hidden[t]   ([C][d_model], q | k | v channels)
 *   z[t]     = W_z hidden[t]     ([Hv*d_v][d_model], the output gate)
 *   b[t]     = W_b hidden[t],  a[t] = W_a hidden[t]   ([Hv][d_model] each)
 * hidden [T][d_model], outputs [T][C], [T][Hv*d_v], [T][Hv], [T][Hv].
 * d_model, C, Hv and Hv*d_v must be multiples of 8 (GDN_ERR_DIMS). */
int gdn_in_proj(const void* hidden, int T, int d_model, const void* w_qkv, const void* w_z,
                const void* w_b, const void* w_a, int C, int Hv, int d_v, void* x_qkv, void* z,
                void* b, void* a, uint32_t* flags, void* stream);

/* gdn_out_proj: per token t and v-head h, the gated RMS norm of the layer's
 * output
 *   o_norm[t][h] = o[t][h] / sqrt(mean_v(o[t][h][v]^2) + eps) * norm_w * silu(z[t][h])
 * (norm_w [d_v] fp32, shared by the heads), written to the caller's o_norm
 * [T][Hv][d_v] bf16, then y[t] = W_out o_norm[t] with W_out [d_model][Hv*d_v]
 * and y [T][d_model].  o, z as the forward's out and gdn_in_proj's z.  d_v
 * must be 128, Hv and d_model multiples of 8. */
int gdn_out_proj(const void* o, const void* z, const float* norm_w, float eps, const void* w_out,
                 int T, int Hv, int d_v, int d_model, void* o_norm, void* y, uint32_t* flags,
                 void* stream);

/* Read (and optionally clear) the OR of GDN_FLAG_* raised by earlier forwards
 * on one layer (layer < 0: OR over all layers).  Synchronises `stream`; not
 * for the hot path. */
int gdn_get_error(gdn_pool_t* pool, int layer, uint32_t* flags, int reset, void* stream);

/* Which path the sequences longer than one token took in the last
 * gdn_varlen_forward (or gdn_varlen_forward enqueued into a captured graph)
 * on this pool, decided on the host when the call was made:
 *   GDN_PREFILL_NONE   no such sequence could be in the call (T < 2 or a
 *                      max_seqlen_hint of 1)
 *   GDN_PREFILL_SPLIT  the chunk-parallel kernel and the recurrence kernel on
 *                      the pool's scratch
 *   GDN_PREFILL_FUSED  the single fused chunked kernel (not enough scratch)
 *   GDN_PREFILL_SERIAL the token-serial kernel (shapes the chunked kernels do
 *                      not cover)
 * Does not synchronise. */
#define GDN_PREFILL_NONE 0
#define GDN_PREFILL_SPLIT 1
#define GDN_PREFILL_FUSED 2
#define GDN_PREFILL_SERIAL 3
int gdn_pool_last_prefill_path(const gdn_pool_t* pool, int* path);

/* Profiling aid: while set, every later gdn_varlen_forward on this pool
 * records cudaEvent_t `before` on its stream right after the scheduler kernel
 * and `after` right after the last compute kernel, so the caller can time the
 * compute kernels alone (cudaEventElapsedTime).  NULL, NULL turns it off.
 * The events are caller-owned; recording them does not synchronise. */
int gdn_pool_set_timing_events(gdn_pool_t* pool, void* before, void* after);

/* Static string for a status code. */
const char* gdn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */

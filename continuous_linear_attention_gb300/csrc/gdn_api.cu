// C ABI of libgdn: the paged state pool, host-side validation and the launch
// sequence of one layer forward.  The operations follow the pages on
// continuous batching for linear attention layers (per-request state block,
// zeroed trash block, in-place overwrite, 128-byte sub-state alignment) and
// the gated delta rule; see include/gdn.h for the full contract.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "gdn.h"
#include "gdn_internal.cuh"

struct gdn_pool {
  int num_blocks, num_layers, Hk, Hv, dk, dv, K, act;
  size_t stride, conv_off, rec_off, total;
  unsigned char* base;
  bool owns;
  int device;
  int32_t* work;  // num_layers * WorkArea::words(num_blocks) words
  cudaEvent_t ev_before, ev_after;  // optional timing events (caller-owned)
  // prefill scratch: chunk-major tiles of the split prefill path (gated delta
  // net pools, capacity in 64-token chunks) or the fp16 conv output of the
  // chunked scan (Mamba2 pools, capacity in tokens); allocated stream-ordered
  unsigned char* scr;
  size_t scr_bytes;
  bool scr_grow;  // false: never allocated; the fused chunked kernel is used
  int last_path;  // GDN_PREFILL_* of the last forward
  // 0: gated delta net pool (conv + recurrent state); 1: Mamba2 pool (conv +
  // SSM state [H][P][N] at rec_off), with its dimensions
  int kind;
  int ssd_H, ssd_P, ssd_N, ssd_G;
};

namespace {

size_t roundup(size_t v, size_t m) { return (v + m - 1) / m * m; }

// Prefill scratch of a gated delta net pool, chunk-major: for every 64-token
// chunk of the call's prefill sequences (by the scheduler's chunk index) the
// tiles the recurrence kernel loads, each in the 128-byte-swizzled shared
// memory layout of its MMA operand, so both kernels move them with plain bulk
// copies:
//   QK [chunk][Hk]  the [q~ ; k~] tile: 2 K-blocks x (64 q~ rows, 64 k~ rows) fp16
//   G  [chunk][Hk]  (G, beta) of the k-head's two v-heads per token, fp32 [64][4]
//                   (per-channel decay: e^{Gamma_C} of both v-heads, fp32 [2][128])
//   W  [chunk][Hv]  -w: 2 boxes of 64 channels x 64 tokens fp16
//   U  [chunk][Hv]  u:  2 boxes of 64 channels x 64 tokens fp16
//   P  [chunk][Hv]  P:  64 x 64 fp16
//   C  [chunk]      record (first packed row, valid tokens, chunk index, sequence)
// and, for the per-channel-decay forward only,
//   V  [chunk][Hv]  v:  2 boxes of 64 channels x 64 tokens fp16 (conv output)
//   QH [chunk][Hv]  [q^ ; k^]: the decayed q~ and k~ of the v-head, QK's layout
// The buffer is laid out part-major for the capacity of the layout a call
// uses (the scalar forward's six parts, or all eight).
enum ScrPart { kScrQK = 0, kScrG, kScrW, kScrU, kScrP, kScrC, kScrV, kScrQH, kScrParts };
constexpr int kScrScalarParts = kScrV;
size_t scratch_part_bytes(const gdn_pool* p, int part) {
  switch (part) {
    case kScrQK: return (size_t)p->Hk * 64 * 2 * p->dk * 2;
    case kScrG: return (size_t)p->Hk * 64 * 4 * 4;
    case kScrW: return (size_t)p->Hv * 64 * p->dk * 2;
    case kScrU: return (size_t)p->Hv * 64 * p->dv * 2;
    case kScrC: return 16;
    case kScrV: return (size_t)p->Hv * 64 * p->dv * 2;
    case kScrQH: return (size_t)p->Hv * 64 * 2 * p->dk * 2;
    default: return (size_t)p->Hv * 64 * 64 * 2;
  }
}
// Part sizes of a gated delta net scratch unit from the head dimensions alone
// (for callers without a pool object).
size_t part_bytes_of(int Hk, int Hv, int dk, int dv, int part) {
  gdn_pool q{};
  q.Hk = Hk;
  q.Hv = Hv;
  q.dk = dk;
  q.dv = dv;
  return scratch_part_bytes(&q, part);
}

// Bytes of one scratch unit: a 64-token chunk of the first `parts` parts
// (gated delta net pools) or one token row of C fp16 channels (Mamba2 pools).
size_t scratch_unit_bytes(const gdn_pool* p, int parts = kScrScalarParts) {
  if (p->kind != 0) return ((size_t)p->ssd_H * p->ssd_P + 2 * (size_t)p->ssd_G * p->ssd_N) * 2;
  size_t b = 0;
  for (int i = 0; i < parts; ++i) b += scratch_part_bytes(p, i);
  return b;
}
// Units the current buffer holds in the layout of the first `parts` parts.
size_t scratch_cap(const gdn_pool* p, int parts = kScrScalarParts) {
  return p->scr ? p->scr_bytes / scratch_unit_bytes(p, parts) : 0;
}
// Units a call with T tokens and N sequences can need: at most T/64 + (number
// of prefill sequences) chunks, and at most one prefill sequence per
// non-trash block and per two tokens.
size_t chunk_units_for(long long T, long long N, int num_blocks) {
  long long seqs = N < T / 2 ? N : T / 2;
  if (seqs > num_blocks - 1) seqs = num_blocks - 1;
  return (size_t)(T / 64 + seqs + 1);
}
size_t scratch_units_for(const gdn_pool* p, long long T, long long N) {
  if (p->kind != 0) return (size_t)T;
  return chunk_units_for(T, N, p->num_blocks);
}
void* scratch_part(const gdn_pool* p, int part, int parts = kScrScalarParts) {
  size_t off = 0;
  for (int i = 0; i < part; ++i) off += scratch_part_bytes(p, i);
  return p->scr + off * scratch_cap(p, parts);
}

// Make the scratch hold `units` units of the first `parts` parts' layout,
// stream-ordered on `s` (the old buffer is freed on the stream after every
// earlier use of it; nothing waits for the device).  With `sync`, waits for
// `s` afterwards.
int scratch_grow(gdn_pool* p, size_t units, cudaStream_t s, bool sync,
                 int parts = kScrScalarParts) {
  if (scratch_cap(p, parts) >= units) return GDN_OK;
  const size_t bytes = roundup(units, p->kind == 0 ? 64 : 4096) * scratch_unit_bytes(p, parts);
  void* np = nullptr;
  if (cudaMallocAsync(&np, bytes, s) != cudaSuccess || !np) {
    cudaGetLastError();
    return GDN_ERR_NOMEM;
  }
  if (p->scr) cudaFreeAsync(p->scr, s);
  p->scr = (unsigned char*)np;
  p->scr_bytes = bytes;
  if (sync && cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
  return GDN_OK;
}
void scratch_release(gdn_pool* p) {
  if (p->scr) {
    cudaFreeAsync(p->scr, 0);
    cudaStreamSynchronize(0);
  }
  p->scr = nullptr;
  p->scr_bytes = 0;
}
bool capturing(cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
    cudaGetLastError();
    return true;  // unknown: do not allocate
  }
  return cs != cudaStreamCaptureStatusNone;
}

bool is_pow2(size_t v) { return v && !(v & (v - 1)); }

}  // namespace

namespace gdn {
size_t prefill_scratch_unit_bytes(int Hk, int Hv, int dk, int dv) {
  size_t b = 0;
  for (int i = 0; i < kScrScalarParts; ++i) b += part_bytes_of(Hk, Hv, dk, dv, i);
  return b;
}
size_t prefill_scratch_units(long long T, long long N, int num_blocks) {
  return chunk_units_for(T, N, num_blocks);
}
void prefill_scratch_parts(unsigned char* base, size_t cap_units, int Hk, int Hv, int dk, int dv,
                           FwdParams* fp) {
  void* part[kScrScalarParts];
  size_t off = 0;
  for (int i = 0; i < kScrScalarParts; ++i) {
    part[i] = base + off * cap_units;
    off += part_bytes_of(Hk, Hv, dk, dv, i);
  }
  fp->scr_qk = part[kScrQK];
  fp->scr_g = part[kScrG];
  fp->scr_w = part[kScrW];
  fp->scr_u = part[kScrU];
  fp->scr_p = part[kScrP];
  fp->scr_c = part[kScrC];
}
}  // namespace gdn

namespace {

int check_dims(int num_blocks, int num_layers, int Hk, int Hv, int dk, int dv, int K, int act,
               size_t block_align) {
  if (num_blocks < 2 || num_layers < 1) return GDN_ERR_RANGE;
  if (Hk < 1 || Hv < 1 || Hv % Hk != 0) return GDN_ERR_DIMS;
  const int ratio = Hv / Hk;
  if (ratio > 2) return GDN_ERR_DIMS;
  if (dk != dv || (dk != 32 && dk != 64 && dk != 128)) return GDN_ERR_DIMS;
  if (K < 2 || K > gdn::kMaxConvK) return GDN_ERR_DIMS;
  if (act != GDN_F32 && act != GDN_BF16) return GDN_ERR_DIMS;
  if (block_align != 0 && (block_align < 128 || !is_pow2(block_align))) return GDN_ERR_DIMS;
  // every block byte offset must fit comfortably in size_t and indices in int
  if ((long long)num_blocks * num_layers > (1ll << 30)) return GDN_ERR_RANGE;
  return GDN_OK;
}

struct Layout {
  size_t stride, conv_off, rec_off, total;
};

Layout layout_of(int num_blocks, int num_layers, int Hk, int Hv, int dk, int dv, int K, int act,
                 size_t block_align) {
  const size_t C = 2 * (size_t)Hk * dk + (size_t)Hv * dv;
  const size_t act_bytes = act == GDN_F32 ? 4 : 2;
  const size_t conv_bytes = (size_t)(K - 1) * C * act_bytes;
  const size_t rec_bytes = (size_t)Hv * dk * dv * sizeof(float);
  Layout l;
  l.conv_off = 0;
  l.rec_off = roundup(conv_bytes, 128);
  size_t align = block_align > 128 ? block_align : 128;
  l.stride = roundup(l.rec_off + rec_bytes, align);
  l.total = l.stride * (size_t)num_blocks * (size_t)num_layers;
  return l;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Mamba2 pools: conv state [K-1][C] (C = H*P + 2*G*N, activation dtype) at 0,
// SSM state [H][P][N] fp32 at the next 128-byte boundary.
int check_ssd_dims(int num_blocks, int num_layers, int H, int P, int NS, int G, int K, int act,
                   size_t block_align) {
  if (num_blocks < 2 || num_layers < 1) return GDN_ERR_RANGE;
  if (H < 1 || G < 1 || H % G != 0 || H > 4096) return GDN_ERR_DIMS;
  if (!gdn::ssd_supported(P, NS)) return GDN_ERR_DIMS;
  if (K < 2 || K > gdn::kMaxConvK) return GDN_ERR_DIMS;
  if (act != GDN_F32 && act != GDN_BF16) return GDN_ERR_DIMS;
  if (block_align != 0 && (block_align < 128 || !is_pow2(block_align))) return GDN_ERR_DIMS;
  if ((long long)num_blocks * num_layers > (1ll << 30)) return GDN_ERR_RANGE;
  return GDN_OK;
}

Layout ssd_layout_of(int num_blocks, int num_layers, int H, int P, int NS, int G, int K, int act,
                     size_t block_align) {
  const size_t C = (size_t)H * P + 2 * (size_t)G * NS;
  const size_t act_bytes = act == GDN_F32 ? 4 : 2;
  const size_t conv_bytes = (size_t)(K - 1) * C * act_bytes;
  const size_t ssm_bytes = (size_t)H * P * NS * sizeof(float);
  Layout l;
  l.conv_off = 0;
  l.rec_off = roundup(conv_bytes, 128);
  size_t align = block_align > 128 ? block_align : 128;
  l.stride = roundup(l.rec_off + ssm_bytes, align);
  l.total = l.stride * (size_t)num_blocks * (size_t)num_layers;
  return l;
}

// Host checks and kernel parameters shared by the gated-delta-net forwards
// (scalar gate, or one gate per key channel with `channel_gate`): returns
// GDN_OK with *fp filled, or the status of the first failed check (nothing
// launched).  *fp_empty is set when there is nothing to do (N == 0, T == 0).
int prepare_forward(gdn_pool* p, int layer, const void* x_qkv, const void* a, const void* b,
                    const int32_t* cu_seqlens, const int32_t* state_block_idx,
                    const uint8_t* has_past, const gdn_weights_t* w, void* out, int T, int N,
                    int max_seqlen_hint, bool channel_gate, gdn::FwdParams* fp, bool* fp_empty) {
  *fp_empty = false;
  if (!p || !w) return GDN_ERR_NULL;
  if (p->kind != 0) return GDN_ERR_DIMS;
  if (layer < 0 || layer >= p->num_layers || T < 0 || N < 0 || max_seqlen_hint < 0)
    return GDN_ERR_RANGE;
  if (N == 0) {
    *fp_empty = true;
    return T == 0 ? GDN_OK : GDN_ERR_RANGE;
  }
  if (!cu_seqlens || !state_block_idx || !has_past || !w->conv_w || !w->A_log || !w->dt_bias)
    return GDN_ERR_NULL;
  if (T > 0 && (!x_qkv || !a || !b || !out)) return GDN_ERR_NULL;
  const int C = 2 * p->Hk * p->dk + p->Hv * p->dv;
  const size_t act_bytes = p->act == GDN_F32 ? 4 : 2;
  if ((long long)T * C > (1ll << 40)) return GDN_ERR_RANGE;
  if (T > 0 && (!aligned16(x_qkv) || !aligned16(a) || !aligned16(b) || !aligned16(out)))
    return GDN_ERR_ALIGN;
  if (!aligned16(w->conv_w) || ((size_t)C * act_bytes) % 16 != 0 ||
      ((size_t)p->dv * act_bytes) % 16 != 0 ||
      (channel_gate && ((size_t)p->dk * act_bytes) % 16 != 0))
    return GDN_ERR_ALIGN;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  if (dev != p->device) return GDN_ERR_DEVICE;
  fp->x = x_qkv;
  fp->a = a;  // [T][Hv], or [T][Hv][d_k] with one gate per key channel
  fp->b = b;
  fp->cu = cu_seqlens;
  fp->blk = state_block_idx;
  fp->has_past = has_past;
  fp->conv_w = w->conv_w;
  fp->A_log = w->A_log;
  fp->dt_bias = w->dt_bias;  // [Hv], or [Hv][d_k] with one gate per key channel
  fp->out = out;
  fp->layer_base = p->base + (size_t)layer * p->num_blocks * p->stride;
  fp->stride = p->stride;
  fp->rec_off = p->rec_off;
  fp->T = T;
  fp->N = N;
  fp->Hk = p->Hk;
  fp->Hv = p->Hv;
  fp->C = C;
  fp->K = p->K;
  fp->num_blocks = p->num_blocks;
  fp->max_seqlen_hint = max_seqlen_hint;
  fp->work.base = p->work + (size_t)layer * gdn::WorkArea::words(p->num_blocks);
  fp->work.num_blocks = p->num_blocks;
  return GDN_OK;
}

}  // namespace

extern "C" {

const char* gdn_status_string(int status) {
  switch (status) {
    case GDN_OK: return "ok";
    case GDN_ERR_NULL: return "a required pointer is NULL";
    case GDN_ERR_DIMS: return "dimensions inconsistent or unsupported";
    case GDN_ERR_RANGE: return "argument out of range";
    case GDN_ERR_ALIGN: return "pointer or row pitch not 16-byte aligned";
    case GDN_ERR_CUDA: return "CUDA runtime error";
    case GDN_ERR_NOMEM: return "out of device memory or buffer too small";
    case GDN_ERR_DEVICE: return "current device differs from the pool's device";
    default: return "unknown status";
  }
}

int gdn_state_pool_layout_for(int num_blocks, int num_layers, int Hk, int Hv, int dk, int dv,
                              int K, int act, size_t block_align, size_t* block_stride,
                              size_t* conv_off, size_t* rec_off, size_t* total_bytes) {
  int st = check_dims(num_blocks, num_layers, Hk, Hv, dk, dv, K, act, block_align);
  if (st != GDN_OK) return st;
  Layout l = layout_of(num_blocks, num_layers, Hk, Hv, dk, dv, K, act, block_align);
  if (block_stride) *block_stride = l.stride;
  if (conv_off) *conv_off = l.conv_off;
  if (rec_off) *rec_off = l.rec_off;
  if (total_bytes) *total_bytes = l.total;
  return GDN_OK;
}

int gdn_state_pool_create(gdn_pool_t** out, int num_blocks, int num_layers, int Hk, int Hv,
                          int dk, int dv, int K, int act, size_t block_align, void* device_mem,
                          size_t device_bytes) {
  if (!out) return GDN_ERR_NULL;
  *out = nullptr;
  int st = check_dims(num_blocks, num_layers, Hk, Hv, dk, dv, K, act, block_align);
  if (st != GDN_OK) return st;
  Layout l = layout_of(num_blocks, num_layers, Hk, Hv, dk, dv, K, act, block_align);
  if (device_mem) {
    if (device_bytes < l.total) return GDN_ERR_NOMEM;
    if (((uintptr_t)device_mem & 255u) != 0) return GDN_ERR_ALIGN;
  }
  gdn_pool* p = new (std::nothrow) gdn_pool();
  if (!p) return GDN_ERR_NOMEM;
  p->num_blocks = num_blocks;
  p->num_layers = num_layers;
  p->Hk = Hk;
  p->Hv = Hv;
  p->dk = dk;
  p->dv = dv;
  p->K = K;
  p->act = act;
  p->scr = nullptr;
  p->scr_bytes = 0;
  p->scr_grow = true;
  p->last_path = GDN_PREFILL_NONE;
  p->stride = l.stride;
  p->conv_off = l.conv_off;
  p->rec_off = l.rec_off;
  p->total = l.total;
  if (cudaGetDevice(&p->device) != cudaSuccess) {
    delete p;
    return GDN_ERR_CUDA;
  }
  if (device_mem) {
    p->base = (unsigned char*)device_mem;
    p->owns = false;
  } else {
    if (cudaMalloc((void**)&p->base, l.total) != cudaSuccess) {
      cudaGetLastError();
      delete p;
      return GDN_ERR_NOMEM;
    }
    p->owns = true;
  }
  const size_t work_bytes = gdn::WorkArea::words(num_blocks) * num_layers * sizeof(int32_t);
  if (cudaMalloc((void**)&p->work, work_bytes) != cudaSuccess) {
    cudaGetLastError();
    if (p->owns) cudaFree(p->base);
    delete p;
    return GDN_ERR_NOMEM;
  }
  if (cudaMemset(p->base, 0, l.total) != cudaSuccess ||
      cudaMemset(p->work, 0, work_bytes) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    if (p->owns) cudaFree(p->base);
    cudaFree(p->work);
    delete p;
    return GDN_ERR_CUDA;
  }
  *out = p;
  return GDN_OK;
}

int gdn_state_pool_destroy(gdn_pool_t* p) {
  if (!p) return GDN_OK;
  int prev = -1;
  cudaGetDevice(&prev);
  cudaSetDevice(p->device);
  cudaDeviceSynchronize();
  if (p->owns) cudaFree(p->base);
  cudaFree(p->work);
  scratch_release(p);
  if (prev >= 0) cudaSetDevice(prev);
  delete p;
  return GDN_OK;
}

int gdn_state_pool_layout(const gdn_pool_t* p, size_t* block_stride, size_t* conv_off,
                          size_t* rec_off, void** base) {
  if (!p) return GDN_ERR_NULL;
  if (block_stride) *block_stride = p->stride;
  if (conv_off) *conv_off = p->conv_off;
  if (rec_off) *rec_off = p->rec_off;
  if (base) *base = p->base;
  return GDN_OK;
}

int gdn_state_pool_copy_block(gdn_pool_t* p, int layer, int src, int dst, void* stream) {
  if (!p) return GDN_ERR_NULL;
  if (layer < 0 || layer >= p->num_layers) return GDN_ERR_RANGE;
  if (src < 0 || src >= p->num_blocks || dst <= 0 || dst >= p->num_blocks) return GDN_ERR_RANGE;
  if (src == dst) return GDN_OK;
  unsigned char* page = p->base + (size_t)layer * p->num_blocks * p->stride;
  cudaError_t e = cudaMemcpyAsync(page + (size_t)dst * p->stride, page + (size_t)src * p->stride,
                                  p->stride, cudaMemcpyDeviceToDevice, (cudaStream_t)stream);
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_varlen_forward(gdn_pool_t* p, int layer, const void* x_qkv, const void* a, const void* b,
                       const int32_t* cu_seqlens, const int32_t* state_block_idx,
                       const uint8_t* has_past, const gdn_weights_t* w, void* out, int T, int N,
                       int max_seqlen_hint, void* stream) {
  gdn::FwdParams fp;
  bool empty = false;
  const int st = prepare_forward(p, layer, x_qkv, a, b, cu_seqlens, state_block_idx, has_past, w,
                                 out, T, N, max_seqlen_hint, false, &fp, &empty);
  if (st != GDN_OK || empty) return st;
  cudaStream_t s = (cudaStream_t)stream;
  // prefill scratch of the split path: grown on demand, stream-ordered,
  // outside stream capture; without enough of it the fused chunked kernel runs
  const bool chunked = gdn::decode_supported(p->dk, p->act, p->Hk, p->Hv, p->K) &&
                       gdn::chunk_supported(p->dk, p->act, p->K);
  const bool may_prefill = T > 1 && max_seqlen_hint != 1;
  const size_t need = scratch_units_for(p, T, N);
  if (chunked && may_prefill && p->scr_grow && need > scratch_cap(p) && !capturing(s))
    scratch_grow(p, need, s, false);
  if (chunked && may_prefill && scratch_cap(p) >= need) {
    fp.scr_qk = scratch_part(p, kScrQK);
    fp.scr_g = scratch_part(p, kScrG);
    fp.scr_w = scratch_part(p, kScrW);
    fp.scr_u = scratch_part(p, kScrU);
    fp.scr_p = scratch_part(p, kScrP);
    fp.scr_c = scratch_part(p, kScrC);
  }
  p->last_path = !may_prefill ? GDN_PREFILL_NONE
                 : !chunked   ? GDN_PREFILL_SERIAL
                 : fp.scr_qk  ? GDN_PREFILL_SPLIT
                              : GDN_PREFILL_FUSED;
  if (gdn::launch_schedule(fp, s) != cudaSuccess) return GDN_ERR_CUDA;
  if (p->ev_before && cudaEventRecord(p->ev_before, s) != cudaSuccess) return GDN_ERR_CUDA;
  if (T == 0) {
    if (p->ev_after && cudaEventRecord(p->ev_after, s) != cudaSuccess) return GDN_ERR_CUDA;
    return GDN_OK;
  }
  // at most one active sequence per non-trash block, and at most T non-empty ones
  int max_items = N;
  if (max_items > p->num_blocks - 1) max_items = p->num_blocks - 1;
  if (max_items > T) max_items = T;
  if (gdn::decode_supported(p->dk, p->act, p->Hk, p->Hv, p->K)) {
    // length-1 sequences: persistent HBM-streaming decode kernel, right
    // after the scheduler, or with prefills behind their recurrence (on the
    // SMs its last chains leave idle); longer ones (at most T/2 of them):
    // the chunked prefill, else the token-serial kernel
    int max_long = max_items < T / 2 ? max_items : T / 2;
    if (max_seqlen_hint == 1) max_long = 0;  // longer sequences are flagged, never listed
    const bool chunk = gdn::chunk_supported(p->dk, p->act, p->K);
    const bool dec_late = chunk && max_long > 0;
    if (!dec_late && gdn::launch_decode(fp, max_items, s) != cudaSuccess) return GDN_ERR_CUDA;
    if (chunk) {
      if (gdn::launch_chunk(fp, max_long, s, dec_late ? max_items : 0) != cudaSuccess)
        return GDN_ERR_CUDA;
    } else if (gdn::launch_recurrent(fp, p->dk, p->act, max_long, true, s) != cudaSuccess) {
      return GDN_ERR_CUDA;
    }
  } else {
    if (gdn::launch_recurrent(fp, p->dk, p->act, max_items, false, s) != cudaSuccess)
      return GDN_ERR_CUDA;
  }
  if (p->ev_after && cudaEventRecord(p->ev_after, s) != cudaSuccess) return GDN_ERR_CUDA;
  return GDN_OK;
}

int gdn_state_pool_reserve(gdn_pool_t* p, int max_tokens) {
  if (!p) return GDN_ERR_NULL;
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != p->device) return GDN_ERR_DEVICE;
  if (max_tokens > 0) {
    p->scr_grow = true;
    return scratch_grow(p, scratch_units_for(p, max_tokens, max_tokens), 0, true);
  }
  if (max_tokens == 0) {
    scratch_release(p);
    p->scr_grow = false;
    return GDN_OK;
  }
  p->scr_grow = true;
  return GDN_OK;
}

int gdn_prefill_scratch_bytes(int num_blocks, int num_k_heads, int num_v_heads, int d_k, int d_v,
                              int max_tokens, size_t* bytes) {
  if (!bytes) return GDN_ERR_NULL;
  if (num_blocks < 2 || max_tokens < 0) return GDN_ERR_RANGE;
  if (num_k_heads < 1 || num_v_heads < 1 || d_k < 1 || d_v < 1) return GDN_ERR_DIMS;
  // any N: at most one prefill sequence per two tokens
  *bytes = gdn::prefill_scratch_units(max_tokens, max_tokens, num_blocks) *
           gdn::prefill_scratch_unit_bytes(num_k_heads, num_v_heads, d_k, d_v);
  return GDN_OK;
}

int gdn_pool_last_prefill_path(const gdn_pool_t* p, int* path) {
  if (!p || !path) return GDN_ERR_NULL;
  *path = p->last_path;
  return GDN_OK;
}

int gdn_pool_set_timing_events(gdn_pool_t* p, void* before, void* after) {
  if (!p) return GDN_ERR_NULL;
  if ((before == nullptr) != (after == nullptr)) return GDN_ERR_NULL;
  p->ev_before = (cudaEvent_t)before;
  p->ev_after = (cudaEvent_t)after;
  return GDN_OK;
}

int gdn_get_error(gdn_pool_t* p, int layer, uint32_t* flags, int reset, void* stream) {
  if (!p || !flags) return GDN_ERR_NULL;
  if (layer >= p->num_layers) return GDN_ERR_RANGE;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t words = gdn::WorkArea::words(p->num_blocks);
  uint32_t acc = 0;
  for (int l = 0; l < p->num_layers; ++l) {
    if (layer >= 0 && l != layer) continue;
    uint32_t v = 0;
    int32_t* word = p->work + (size_t)l * words + gdn::kErr;
    if (cudaMemcpyAsync(&v, word, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return GDN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
    acc |= v;
    if (reset && cudaMemsetAsync(word, 0, sizeof(uint32_t), s) != cudaSuccess) return GDN_ERR_CUDA;
  }
  if (reset && cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
  *flags = acc;
  return GDN_OK;
}

int gdn_kda_varlen_forward(gdn_pool_t* p, int layer, const void* x_qkv, const void* a,
                           const void* b, const int32_t* cu_seqlens,
                           const int32_t* state_block_idx, const uint8_t* has_past,
                           const gdn_weights_t* w, void* out, int T, int N, int max_seqlen_hint,
                           void* stream) {
  gdn::FwdParams fp;
  bool empty = false;
  const int st = prepare_forward(p, layer, x_qkv, a, b, cu_seqlens, state_block_idx, has_past, w,
                                 out, T, N, max_seqlen_hint, true, &fp, &empty);
  if (st != GDN_OK || empty) return st;
  cudaStream_t s = (cudaStream_t)stream;
  // the split prefill (conv pass, chunk products, recurrence) needs the
  // scratch in its eight-part layout: grown on demand, stream-ordered,
  // outside stream capture; without it the token-serial kernel runs
  const bool chunked = gdn::decode_supported(p->dk, p->act, p->Hk, p->Hv, p->K) &&
                       gdn::chunk_supported(p->dk, p->act, p->K);
  const bool may_prefill = T > 1 && max_seqlen_hint != 1;
  const size_t need = scratch_units_for(p, T, N);
  if (chunked && may_prefill && p->scr_grow && need > scratch_cap(p, kScrParts) && !capturing(s))
    scratch_grow(p, need, s, false, kScrParts);
  if (chunked && may_prefill && scratch_cap(p, kScrParts) >= need) {
    fp.scr_qk = scratch_part(p, kScrQK, kScrParts);
    fp.scr_g = scratch_part(p, kScrG, kScrParts);
    fp.scr_w = scratch_part(p, kScrW, kScrParts);
    fp.scr_u = scratch_part(p, kScrU, kScrParts);
    fp.scr_p = scratch_part(p, kScrP, kScrParts);
    fp.scr_c = scratch_part(p, kScrC, kScrParts);
    fp.scr_v = scratch_part(p, kScrV, kScrParts);
    fp.scr_qh = scratch_part(p, kScrQH, kScrParts);
  }
  p->last_path = !may_prefill ? GDN_PREFILL_NONE
                 : fp.scr_qk  ? GDN_PREFILL_SPLIT
                              : GDN_PREFILL_SERIAL;
  if (gdn::launch_schedule(fp, s) != cudaSuccess) return GDN_ERR_CUDA;
  if (p->ev_before && cudaEventRecord(p->ev_before, s) != cudaSuccess) return GDN_ERR_CUDA;
  if (T > 0) {
    int max_items = N;
    if (max_items > p->num_blocks - 1) max_items = p->num_blocks - 1;
    if (max_items > T) max_items = T;
    if (gdn::decode_supported(p->dk, p->act, p->Hk, p->Hv, p->K)) {
      int max_long = max_items < T / 2 ? max_items : T / 2;
      if (max_seqlen_hint == 1) max_long = 0;
      // decodes behind the split prefill's recurrence when there is one
      const bool dec_late = fp.scr_qk && max_long > 0;
      if (!dec_late && gdn::launch_kda_decode(fp, max_items, s) != cudaSuccess) return GDN_ERR_CUDA;
      if (fp.scr_qk) {
        if (gdn::launch_kda_chunk(fp, max_long, s, dec_late ? max_items : 0) != cudaSuccess)
          return GDN_ERR_CUDA;
      } else if (gdn::launch_kda_recurrent(fp, p->dk, p->act, max_long, true, s) != cudaSuccess) {
        return GDN_ERR_CUDA;
      }
    } else if (gdn::launch_kda_recurrent(fp, p->dk, p->act, max_items, false, s) !=
               cudaSuccess) {
      return GDN_ERR_CUDA;
    }
  }
  if (p->ev_after && cudaEventRecord(p->ev_after, s) != cudaSuccess) return GDN_ERR_CUDA;
  return GDN_OK;
}

int gdn_ssd_pool_layout_for(int num_blocks, int num_layers, int H, int P, int NS, int G, int K,
                            int act, size_t block_align, size_t* block_stride, size_t* conv_off,
                            size_t* ssm_off, size_t* total_bytes) {
  int st = check_ssd_dims(num_blocks, num_layers, H, P, NS, G, K, act, block_align);
  if (st != GDN_OK) return st;
  Layout l = ssd_layout_of(num_blocks, num_layers, H, P, NS, G, K, act, block_align);
  if (block_stride) *block_stride = l.stride;
  if (conv_off) *conv_off = l.conv_off;
  if (ssm_off) *ssm_off = l.rec_off;
  if (total_bytes) *total_bytes = l.total;
  return GDN_OK;
}

int gdn_ssd_pool_create(gdn_pool_t** out, int num_blocks, int num_layers, int H, int P, int NS,
                        int G, int K, int act, size_t block_align, void* device_mem,
                        size_t device_bytes) {
  if (!out) return GDN_ERR_NULL;
  *out = nullptr;
  int st = check_ssd_dims(num_blocks, num_layers, H, P, NS, G, K, act, block_align);
  if (st != GDN_OK) return st;
  Layout l = ssd_layout_of(num_blocks, num_layers, H, P, NS, G, K, act, block_align);
  if (device_mem) {
    if (device_bytes < l.total) return GDN_ERR_NOMEM;
    if (((uintptr_t)device_mem & 255u) != 0) return GDN_ERR_ALIGN;
  }
  gdn_pool* p = new (std::nothrow) gdn_pool();
  if (!p) return GDN_ERR_NOMEM;
  p->kind = 1;
  p->num_blocks = num_blocks;
  p->num_layers = num_layers;
  p->ssd_H = H;
  p->ssd_P = P;
  p->ssd_N = NS;
  p->ssd_G = G;
  p->K = K;
  p->act = act;
  p->scr = nullptr;
  p->scr_bytes = 0;
  p->scr_grow = true;  // the chunked scan's fp16 conv scratch, grown on demand
  p->last_path = GDN_PREFILL_NONE;
  p->stride = l.stride;
  p->conv_off = l.conv_off;
  p->rec_off = l.rec_off;
  p->total = l.total;
  if (cudaGetDevice(&p->device) != cudaSuccess) {
    delete p;
    return GDN_ERR_CUDA;
  }
  if (device_mem) {
    p->base = (unsigned char*)device_mem;
    p->owns = false;
  } else {
    if (cudaMalloc((void**)&p->base, l.total) != cudaSuccess) {
      cudaGetLastError();
      delete p;
      return GDN_ERR_NOMEM;
    }
    p->owns = true;
  }
  const size_t work_bytes = gdn::WorkArea::words(num_blocks) * num_layers * sizeof(int32_t);
  if (cudaMalloc((void**)&p->work, work_bytes) != cudaSuccess) {
    cudaGetLastError();
    if (p->owns) cudaFree(p->base);
    delete p;
    return GDN_ERR_NOMEM;
  }
  if (cudaMemset(p->base, 0, l.total) != cudaSuccess ||
      cudaMemset(p->work, 0, work_bytes) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    if (p->owns) cudaFree(p->base);
    cudaFree(p->work);
    delete p;
    return GDN_ERR_CUDA;
  }
  *out = p;
  return GDN_OK;
}

int gdn_ssd_varlen_forward(gdn_pool_t* p, int layer, const void* xbc, const void* dt,
                           const int32_t* cu_seqlens, const int32_t* state_block_idx,
                           const uint8_t* has_past, const gdn_ssd_weights_t* w, void* y, int T,
                           int N, int max_seqlen_hint, void* stream) {
  if (!p || !w) return GDN_ERR_NULL;
  if (p->kind != 1) return GDN_ERR_DIMS;
  if (layer < 0 || layer >= p->num_layers || T < 0 || N < 0 || max_seqlen_hint < 0)
    return GDN_ERR_RANGE;
  if (N == 0) return T == 0 ? GDN_OK : GDN_ERR_RANGE;
  if (!cu_seqlens || !state_block_idx || !has_past || !w->conv_w || !w->A_log || !w->dt_bias ||
      !w->D)
    return GDN_ERR_NULL;
  if (T > 0 && (!xbc || !dt || !y)) return GDN_ERR_NULL;
  const int C = p->ssd_H * p->ssd_P + 2 * p->ssd_G * p->ssd_N;
  if ((long long)T * C > (1ll << 40)) return GDN_ERR_RANGE;
  if (T > 0 && (!aligned16(xbc) || !aligned16(dt) || !aligned16(y))) return GDN_ERR_ALIGN;
  if (!aligned16(w->conv_w)) return GDN_ERR_ALIGN;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  if (dev != p->device) return GDN_ERR_DEVICE;

  gdn::SsdParams sp;
  sp.xbc = xbc;
  sp.dt = dt;
  sp.cu = cu_seqlens;
  sp.blk = state_block_idx;
  sp.has_past = has_past;
  sp.conv_w = w->conv_w;
  sp.A_log = w->A_log;
  sp.dt_bias = w->dt_bias;
  sp.Dskip = w->D;
  sp.y = y;
  sp.layer_base = p->base + (size_t)layer * p->num_blocks * p->stride;
  sp.stride = p->stride;
  sp.ssm_off = p->rec_off;
  sp.T = T;
  sp.N = N;
  sp.H = p->ssd_H;
  sp.G = p->ssd_G;
  sp.C = C;
  sp.K = p->K;
  sp.work.base = p->work + (size_t)layer * gdn::WorkArea::words(p->num_blocks);
  sp.work.num_blocks = p->num_blocks;

  // the scheduler reads only the batch description and the work area
  gdn::FwdParams fp;
  fp.cu = cu_seqlens;
  fp.blk = state_block_idx;
  fp.has_past = has_past;
  fp.T = T;
  fp.N = N;
  fp.num_blocks = p->num_blocks;
  fp.max_seqlen_hint = max_seqlen_hint;
  fp.work = sp.work;

  cudaStream_t s = (cudaStream_t)stream;
  // fp16 conv scratch of the chunked scan: grown on demand, stream-ordered,
  // outside stream capture
  if (p->scr_grow && (size_t)T > scratch_cap(p) && T > 1 && max_seqlen_hint != 1 &&
      gdn::ssd_chunk_supported(p->ssd_H, p->ssd_P, p->ssd_N, p->K, p->act) && !capturing(s))
    scratch_grow(p, (size_t)T, s, false);
  if (gdn::launch_schedule(fp, s) != cudaSuccess) return GDN_ERR_CUDA;
  if (p->ev_before && cudaEventRecord(p->ev_before, s) != cudaSuccess) return GDN_ERR_CUDA;
  if (T > 0) {
    int max_items = N;
    if (max_items > p->num_blocks - 1) max_items = p->num_blocks - 1;
    if (max_items > T) max_items = T;
    if (gdn::ssd_decode_supported(p->ssd_H, p->ssd_P, p->ssd_N, p->ssd_G, p->K, p->act)) {
      // length-1 sequences: HBM-streaming decode kernel; longer ones (at most
      // T/2 of them): the chunked scan when the scratch holds T rows, else the
      // token-serial kernel, then their conv-state update
      if (gdn::launch_ssd_decode(sp, max_items, s) != cudaSuccess) return GDN_ERR_CUDA;
      int max_long = max_items < T / 2 ? max_items : T / 2;
      if (max_seqlen_hint == 1) max_long = 0;
      const bool chunked = max_long > 0 && scratch_cap(p) >= (size_t)T &&
                           gdn::ssd_chunk_supported(p->ssd_H, p->ssd_P, p->ssd_N, p->K, p->act);
      if (chunked) {
        if (gdn::launch_ssd_chunk(sp, p->scr, max_long, s) != cudaSuccess) return GDN_ERR_CUDA;
      } else if (gdn::launch_ssd(sp, p->ssd_P, p->ssd_N, p->act, max_long, true, s) !=
                 cudaSuccess) {
        return GDN_ERR_CUDA;
      }
    } else if (gdn::launch_ssd(sp, p->ssd_P, p->ssd_N, p->act, max_items, false, s) !=
               cudaSuccess) {
      return GDN_ERR_CUDA;
    }
  }
  if (p->ev_after && cudaEventRecord(p->ev_after, s) != cudaSuccess) return GDN_ERR_CUDA;
  return GDN_OK;
}

}  // extern "C"

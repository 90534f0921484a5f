// gdn_varlen_forward_noalloc: the layer forward for callers that must not
// allocate device memory.  Some callers cannot call cudaMalloc at all: an
// engine that plans every byte of device memory up front and forbids runtime
// allocation, code that runs under a memory budget owned by another
// allocator, or a host thread that must not take the driver's allocation
// locks on its latency path.  gdn_state_pool_create allocates the scheduler's
// work area (and, by default, the pool), so those callers could not use the
// library; this entry point takes the pool memory from the caller and keeps
// the scheduler's work area in a statically sized device array instead.
//
// The work area is one file-scope __device__ array with room for pools of up
// to kNoAllocMaxBlocks blocks.  Every GPU that loads the library holds it
// until the process exits.  It is shared by every call of this entry point on
// a device, so calls whose work overlaps on the GPU (different streams, no
// ordering between them) race and must not be made; calls ordered on one
// stream are fine.
#include <cuda_runtime.h>

#include <mutex>

#include "gdn.h"
#include "gdn_internal.cuh"

namespace {

constexpr int kNoAllocMaxBlocks = 4096;
constexpr size_t kNoAllocWords = gdn::WorkArea::words(kNoAllocMaxBlocks);

// The scheduler's work area for this entry point (error word, counters,
// block-use counts, work lists, the prefill chunk prefix and the redo masks), ~128 KiB per
// device.
static __device__ __align__(256) int32_t g_noalloc_work[kNoAllocWords];

constexpr int kMaxDevices = 64;
int32_t* g_work_addr[kMaxDevices] = {};  // device address of g_noalloc_work, per device
std::mutex g_work_mu;

// Device address of the work area on the current device.  In host code the
// array's name only stands for the device symbol, so the address is looked up
// once per device, with that device current, and cached.
int work_area_of_current_device(int32_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_work_mu);
  if (!g_work_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_work) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return GDN_ERR_CUDA;
    }
    g_work_addr[dev] = static_cast<int32_t*>(ptr);
  }
  *out = g_work_addr[dev];
  return GDN_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" int gdn_varlen_forward_noalloc(void* pool_mem, size_t pool_bytes, int num_blocks,
                                          int num_layers, int num_k_heads, int num_v_heads,
                                          int d_k, int d_v, int conv_k, int act_dtype,
                                          size_t block_align, int layer, const void* x_qkv,
                                          const void* a, const void* b,
                                          const int32_t* cu_seqlens,
                                          const int32_t* state_block_idx,
                                          const uint8_t* has_past, const gdn_weights_t* w,
                                          void* out, int T, int N, int max_seqlen_hint,
                                          uint32_t* flags_out, void* stream) {
  size_t stride = 0, conv_off = 0, rec_off = 0, total = 0;
  int st = gdn_state_pool_layout_for(num_blocks, num_layers, num_k_heads, num_v_heads, d_k, d_v,
                                     conv_k, act_dtype, block_align, &stride, &conv_off, &rec_off,
                                     &total);
  if (st != GDN_OK) return st;
  if (num_blocks > kNoAllocMaxBlocks) return GDN_ERR_RANGE;
  if (!pool_mem || !w) return GDN_ERR_NULL;
  if (pool_bytes < total) return GDN_ERR_NOMEM;
  if (((uintptr_t)pool_mem & 255u) != 0) return GDN_ERR_ALIGN;
  if (layer < 0 || layer >= num_layers || T < 0 || N < 0 || max_seqlen_hint < 0)
    return GDN_ERR_RANGE;
  if (N == 0 && T != 0) return GDN_ERR_RANGE;
  if (N > 0 && (!cu_seqlens || !state_block_idx || !has_past)) return GDN_ERR_NULL;
  if (!w->conv_w || !w->A_log || !w->dt_bias) return GDN_ERR_NULL;
  if (T > 0 && (!x_qkv || !a || !b || !out)) return GDN_ERR_NULL;
  const int C = 2 * num_k_heads * d_k + num_v_heads * d_v;
  const size_t act_bytes = act_dtype == GDN_F32 ? 4 : 2;
  if ((long long)T * C > (1ll << 40)) return GDN_ERR_RANGE;
  if (T > 0 && (!aligned16(x_qkv) || !aligned16(a) || !aligned16(b) || !aligned16(out)))
    return GDN_ERR_ALIGN;
  if (!aligned16(w->conv_w) || ((size_t)C * act_bytes) % 16 != 0 ||
      ((size_t)d_v * act_bytes) % 16 != 0)
    return GDN_ERR_ALIGN;
  int32_t* work = nullptr;
  st = work_area_of_current_device(&work);
  if (st != GDN_OK) return st;

  cudaStream_t s = (cudaStream_t)stream;
  // the array keeps the previous call's contents: the error word must start
  // at zero; the scheduler rewrites every other word it reads
  if (cudaMemsetAsync(work + gdn::kErr, 0, sizeof(int32_t), s) != cudaSuccess) return GDN_ERR_CUDA;
  if (N > 0) {
    gdn::FwdParams fp;
    fp.x = x_qkv;
    fp.a = a;
    fp.b = b;
    fp.cu = cu_seqlens;
    fp.blk = state_block_idx;
    fp.has_past = has_past;
    fp.conv_w = w->conv_w;
    fp.A_log = w->A_log;
    fp.dt_bias = w->dt_bias;
    fp.out = out;
    fp.layer_base = (unsigned char*)pool_mem + (size_t)layer * num_blocks * stride;
    fp.stride = stride;
    fp.rec_off = rec_off;
    fp.T = T;
    fp.N = N;
    fp.Hk = num_k_heads;
    fp.Hv = num_v_heads;
    fp.C = C;
    fp.K = conv_k;
    fp.num_blocks = num_blocks;
    fp.max_seqlen_hint = max_seqlen_hint;
    fp.work.base = work;
    fp.work.num_blocks = num_blocks;
    // memory past the pool's layout (from the next 256-byte boundary) serves
    // as the split prefill's scratch when it holds this call's chunks;
    // otherwise prefills run on the fused kernel
    if (T > 1 && max_seqlen_hint != 1 && gdn::chunk_supported(d_k, act_dtype, conv_k)) {
      const size_t units = gdn::prefill_scratch_units(T, N, num_blocks);
      const size_t need = units * gdn::prefill_scratch_unit_bytes(num_k_heads, num_v_heads, d_k, d_v);
      const size_t start = (total + 255) / 256 * 256;
      if (pool_bytes >= start && pool_bytes - start >= need)
        gdn::prefill_scratch_parts(static_cast<unsigned char*>(pool_mem) + start, units,
                                   num_k_heads, num_v_heads, d_k, d_v, &fp);
    }
    if (gdn::launch_schedule(fp, s) != cudaSuccess) return GDN_ERR_CUDA;
    if (T > 0) {
      int max_items = N;
      if (max_items > num_blocks - 1) max_items = num_blocks - 1;
      if (max_items > T) max_items = T;
      if (gdn::decode_supported(d_k, act_dtype, num_k_heads, num_v_heads, conv_k)) {
        int max_long = max_items < T / 2 ? max_items : T / 2;
        if (max_seqlen_hint == 1) max_long = 0;
        // decodes behind the prefill's recurrence when there is one
        const bool chunk = gdn::chunk_supported(d_k, act_dtype, conv_k);
        const bool dec_late = chunk && max_long > 0;
        if (!dec_late && gdn::launch_decode(fp, max_items, s) != cudaSuccess) return GDN_ERR_CUDA;
        if (chunk) {
          if (gdn::launch_chunk(fp, max_long, s, dec_late ? max_items : 0) != cudaSuccess)
            return GDN_ERR_CUDA;
        } else if (gdn::launch_recurrent(fp, d_k, act_dtype, max_long, true, s) != cudaSuccess) {
          return GDN_ERR_CUDA;
        }
      } else if (gdn::launch_recurrent(fp, d_k, act_dtype, max_items, false, s) != cudaSuccess) {
        return GDN_ERR_CUDA;
      }
    }
  }
  if (flags_out && cudaMemcpyAsync(flags_out, work + gdn::kErr, sizeof(uint32_t),
                                   cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return GDN_ERR_CUDA;
  return GDN_OK;
}

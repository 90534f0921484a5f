// Device-side scheduler: turns cu_seqlens / block indices into work lists
// without a host round trip, so the whole forward stays capturable in a CUDA
// graph (the pages note that a chunked kernel which syncs with the host keeps
// accelerator graphs off on the varlen path; this removes that sync).
//
// One CTA.  It validates the batch the way the pool's contract demands (one
// block per request, never shared, the trash block never written, cu_seqlens
// monotonic and ending at T), raises GDN_FLAG_* bits in the layer's error word
// and writes:
//   items[] all active sequences, dec[] the length-1 ones, pre[] the longer
//   ones sorted longest first (ties by sequence id), their counts and the
//   total prefill tokens, the 64-token chunk prefix over the sorted prefill
//   list and (with prefill scratch) one record per chunk, and resets the
//   persistent kernels' work and item counters.
#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"

namespace gdn {
namespace {

constexpr int kSchedThreads = 1024;
// pools of up to this many blocks keep their block-use counts in shared
// memory (fast atomics, no global round trips); larger ones in the work area
constexpr int kSmemCounts = 8192;

__global__ void __launch_bounds__(kSchedThreads)
schedule_kernel(const int32_t* __restrict__ cu, const int32_t* __restrict__ blk, int N, int T,
                int num_blocks, int hint, WorkArea work, int4* __restrict__ chunk_rec) {
  __shared__ int s_bad;
  __shared__ int s_n_items, s_n_dec, s_n_pre, s_pre_tokens;
  __shared__ unsigned s_flags;
  __shared__ int32_t s_counts[kSmemCounts];
  // A programmatic dependent of the stream's previous kernel: the reads of
  // this call's inputs and the block counts (which only this kernel uses) run
  // before griddepcontrol.wait, overlapping that kernel's tail; every write
  // the previous forward's kernels could still read (the header, the lists,
  // the records) comes after it.  The next kernel may launch at once.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x;
  int32_t* hdr = work.header();
  int32_t* blk_count = num_blocks <= kSmemCounts ? s_counts : work.blk_count();
  if (tid == 0) {
    s_bad = (cu[0] != 0 || cu[N] != T) ? 1 : 0;
    s_n_items = s_n_dec = s_n_pre = s_pre_tokens = 0;
    s_flags = 0u;
  }
  for (int i = tid; i < num_blocks; i += kSchedThreads) blk_count[i] = 0;
  __syncthreads();
  for (int s = tid; s < N; s += kSchedThreads)
    if (cu[s + 1] < cu[s]) s_bad = 1;
  __syncthreads();
  if (s_bad) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0) {
      atomicOr((unsigned*)&hdr[kErr], GDN_FLAG_SEQLENS);
      hdr[kNItems] = hdr[kNDec] = hdr[kNPre] = hdr[kPreTokens] = hdr[kPreChunks] = 0;
      hdr[kWorkHead] = hdr[kItemHeadC] = hdr[kItemHeadK] = hdr[kDecHead] = 0;
    }
    return;
  }
  // Count how many active sequences name each block.
  for (int s = tid; s < N; s += kSchedThreads) {
    const int len = cu[s + 1] - cu[s];
    const int b = blk[s];
    if (b < 0 || len <= 0) continue;  // padding entry or empty sequence: no-op
    if (b >= num_blocks) {
      atomicOr(&s_flags, GDN_FLAG_BLOCK_RANGE);
    } else if (b == 0) {
      atomicOr(&s_flags, GDN_FLAG_TRASH_WRITE);
    } else {
      atomicAdd(&blk_count[b], 1);
    }
  }
  __syncthreads();
  // A batch of up to kEarly sequences per thread is classified before the
  // wait (list positions from the shared counters, kept in registers; the
  // inputs and the block counts are this call's own): after it the lists are
  // only written, with no global read on the way.
  constexpr int kEarly = 4;
  const bool early = N <= kEarly * kSchedThreads;
  int kind[kEarly], at[kEarly], lat[kEarly];  // 0 none, 1 decode, 2 prefill; item and list positions
#pragma unroll
  for (int k = 0; k < kEarly; ++k) kind[k] = 0;
  if (early) {
#pragma unroll
    for (int k = 0; k < kEarly; ++k) {
      const int s = tid + k * kSchedThreads;
      if (s >= N) continue;
      const int len = cu[s + 1] - cu[s];
      const int b = blk[s];
      if (b <= 0 || b >= num_blocks || len <= 0) continue;
      if (atomicAdd(&blk_count[b], 0) > 1) {
        atomicOr(&s_flags, GDN_FLAG_DUPLICATE);
        continue;
      }
      if (hint > 0 && len > hint) {
        atomicOr(&s_flags, GDN_FLAG_HINT);
        continue;
      }
      at[k] = atomicAdd(&s_n_items, 1);
      if (len == 1) {
        kind[k] = 1;
        lat[k] = atomicAdd(&s_n_dec, 1);
      } else {
        kind[k] = 2;
        lat[k] = atomicAdd(&s_n_pre, 1);
        atomicAdd(&s_pre_tokens, len);
      }
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int32_t* items = work.items();
  int32_t* dec = work.dec();
  int32_t* pre_tmp = work.pre_tmp();
  if (early) {
#pragma unroll
    for (int k = 0; k < kEarly; ++k) {
      if (!kind[k]) continue;
      const int s = tid + k * kSchedThreads;
      items[at[k]] = s;
      (kind[k] == 1 ? dec : pre_tmp)[lat[k]] = s;
    }
  }
  for (int s = early ? N : tid; s < N; s += kSchedThreads) {
    const int len = cu[s + 1] - cu[s];
    const int b = blk[s];
    if (b <= 0 || b >= num_blocks || len <= 0) continue;
    if (atomicAdd(&blk_count[b], 0) > 1) {
      atomicOr(&s_flags, GDN_FLAG_DUPLICATE);
      continue;
    }
    if (hint > 0 && len > hint) {
      atomicOr(&s_flags, GDN_FLAG_HINT);
      continue;
    }
    items[atomicAdd(&s_n_items, 1)] = s;
    if (len == 1) {
      dec[atomicAdd(&s_n_dec, 1)] = s;
    } else {
      pre_tmp[atomicAdd(&s_n_pre, 1)] = s;
      atomicAdd(&s_pre_tokens, len);
    }
  }
  __syncthreads();
  const int n_pre = s_n_pre;
  if (n_pre == 0) {
    // no prefill sequence: no sort, no chunk prefix beyond its zero, no records
    if (tid == 0) {
      work.pre_cp()[0] = 0;
      if (s_flags) atomicOr((unsigned*)&hdr[kErr], s_flags);
      hdr[kPreChunks] = 0;
      hdr[kNItems] = s_n_items;
      hdr[kNDec] = s_n_dec;
      hdr[kNPre] = 0;
      hdr[kPreTokens] = 0;
      hdr[kWorkHead] = hdr[kItemHeadC] = hdr[kItemHeadK] = hdr[kDecHead] = 0;
    }
    return;
  }
  // Rank sort of the prefill sequences: longest first, ties by sequence id.
  int32_t* pre = work.pre();
  for (int i = tid; i < n_pre; i += kSchedThreads) {
    const int si = pre_tmp[i];
    const int li = cu[si + 1] - cu[si];
    int rank = 0;
    for (int j = 0; j < n_pre; ++j) {
      const int sj = pre_tmp[j];
      const int lj = cu[sj + 1] - cu[sj];
      rank += (lj > li) || (lj == li && sj < si);
    }
    pre[rank] = si;
  }
  __syncthreads();
  // 64-token chunk prefix over the sorted prefill list (for kernels that
  // work per chunk): pre_cp[k] = chunks of pre[0..k)
  int32_t* pre_cp = work.pre_cp();
  for (int k = tid; k <= n_pre; k += kSchedThreads) {
    int acc = 0;
    for (int j = 0; j < k; ++j) {
      const int sj = pre[j];
      acc += (cu[sj + 1] - cu[sj] + 63) >> 6;
    }
    pre_cp[k] = acc;
  }
  __syncthreads();
  // clear the redo masks of the prefill list
  int32_t* redo = work.redo();
  for (int i = tid; i < 2 * n_pre; i += kSchedThreads) redo[i] = 0;
  // one record per 64-token prefill chunk, by chunk index (when the caller
  // has room for them): (first packed row, valid tokens, chunk index inside
  // its sequence, index of the sequence in the prefill list)
  if (chunk_rec) {
    const int total = pre_cp[n_pre];
    for (int g = tid; g < total; g += kSchedThreads) {
      int lo = 0, hi = n_pre - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre_cp[mid] <= g) lo = mid; else hi = mid - 1;
      }
      const int s = pre[lo];
      const int c = g - pre_cp[lo];
      const int seq0 = cu[s];
      const int L = cu[s + 1] - seq0;
      chunk_rec[g] = make_int4(seq0 + 64 * c, min(64, L - 64 * c), c, lo);
    }
  }
  if (tid == 0) {
    if (s_flags) atomicOr((unsigned*)&hdr[kErr], s_flags);
    hdr[kPreChunks] = pre_cp[n_pre];
    hdr[kNItems] = s_n_items;
    hdr[kNDec] = s_n_dec;
    hdr[kNPre] = n_pre;
    hdr[kPreTokens] = s_pre_tokens;
    hdr[kWorkHead] = hdr[kItemHeadC] = hdr[kItemHeadK] = hdr[kDecHead] = 0;
  }
}

}  // namespace

cudaError_t launch_schedule(const FwdParams& p, cudaStream_t stream) {
  return launch_pdl(schedule_kernel, dim3(1), dim3(kSchedThreads), 0, stream, p.cu, p.blk, p.N,
                    p.T, p.num_blocks, p.max_seqlen_hint, p.work, static_cast<int4*>(p.scr_c));
}

}  // namespace gdn

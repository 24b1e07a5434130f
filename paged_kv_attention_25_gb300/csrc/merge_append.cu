// Log-sum-exp merge of split-KV partials, and the paged KV append.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "append.cuh"
#include "internal.h"
#include "merge.cuh"
#include "ptx.cuh"

namespace pkv {
namespace {

// ---------------------------------------------------------------------------
// Merge: one warp per query row of a merge item (merge_row).
template <int D>
__global__ void __launch_bounds__(128) merge_kernel(const AttnArgs a, const MergeItem* __restrict__ items) {
  const MergeItem mi = items[blockIdx.x];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < mi.row_count) merge_row<D>(a, mi, mi.row_begin + warp, lane);
}

// ---------------------------------------------------------------------------
// Append: one warp per slice of a new token's row.  Token t's rows (all KV
// heads, K and V) go to
//   pool[block_tables[r][p / 16]][g][p % 16][:]
// for its request r and position p (fixed-size blocks in non-contiguous
// memory, "LLM上下文缓存与状态复用机制的分析和探索", section 3.1).  A slice is
// up to 32 * kAppendBatch 16-byte chunks of the row (every head, K and V
// alike); the warp issues their loads before it looks the slot up, so that
// the lookup's dependent loads (position, then block id after the request's
// binary search) overlap the data in flight, and each slice is one round of
// loads and stores.  Consecutive lanes copy consecutive chunks, so reads and
// writes are coalesced.  cu_q_lens is staged in shared memory when it has at
// most kAppendCuSmem entries (the search then costs no global round trips).
constexpr int kAppendBatch = 4;
constexpr int kAppendSlice = 32 * kAppendBatch;
constexpr int kAppendCuSmem = 2048;

template <bool F8>
__global__ void __launch_bounds__(256) append_kernel(void* __restrict__ kp, void* __restrict__ vp, int num_blocks,
                                                     int hkv, int cpr_log2, const int32_t* __restrict__ bt,
                                                     int max_blocks, int num_reqs, const int32_t* __restrict__ cu,
                                                     const int32_t* __restrict__ pos, const uint4* __restrict__ k_new,
                                                     const uint4* __restrict__ v_new, int num_tokens, unsigned* err,
                                                     float k_scale, float v_scale) {
  extern __shared__ int32_t s_cu[];
  const bool cu_in_smem = num_reqs + 1 <= kAppendCuSmem;
  if (cu_in_smem) {
    for (int i = threadIdx.x; i <= num_reqs; i += blockDim.x) s_cu[i] = __ldg(cu + i);
    __syncthreads();
  }
  const int lane = threadIdx.x & 31;
  const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int cpr = 1 << cpr_log2;              // 16-byte chunks of one head's row
  const int row_chunks = hkv << cpr_log2;     // chunks of a token's K (or V) row, all heads
  const int slices = (row_chunks + kAppendSlice - 1) / kAppendSlice;
  const int64_t units = static_cast<int64_t>(num_tokens) * slices;
  for (int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < units; w += warps) {
    const int ti = static_cast<int>(w / slices);
    const int c0 = static_cast<int>(w % slices) * kAppendSlice;
    const uint4* ks = k_new + static_cast<int64_t>(ti) * row_chunks;
    const uint4* vs = v_new + static_cast<int64_t>(ti) * row_chunks;
    uint4 kx[kAppendBatch], vx[kAppendBatch];
#pragma unroll
    for (int u = 0; u < kAppendBatch; ++u) {
      const int c = c0 + lane + 32 * u;
      if (c < row_chunks) {
        kx[u] = __ldg(ks + c);
        vx[u] = __ldg(vs + c);
      }
    }
    // The token's slot: request r = the last with cu[r] <= t, its position,
    // and the block id (an out-of-range position or id is flagged and the
    // slice skipped).
    const int p = __ldg(pos + ti);
    int lo = 0, hi = num_reqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((cu_in_smem ? s_cu[mid] : __ldg(cu + mid)) <= ti) lo = mid; else hi = mid - 1;
    }
    if (p < 0 || p >= max_blocks * kBlockSize) {
      if (lane == 0) atomicOr(err, PKV_DEVERR_POSITION);
      continue;
    }
    const int pb = __ldg(bt + static_cast<int64_t>(lo) * max_blocks + p / kBlockSize);
    if (pb < 0 || pb >= num_blocks) {
      if (lane == 0) atomicOr(err, PKV_DEVERR_BLOCK_ID);
      continue;
    }
    // Chunk c of the row (head c / cpr, chunk c % cpr) goes to this slot's chunk index.
    const int64_t slot = static_cast<int64_t>(pb) * hkv * kBlockSize + (p % kBlockSize);
#pragma unroll
    for (int u = 0; u < kAppendBatch; ++u) {
      const int c = c0 + lane + 32 * u;
      if (c < row_chunks) {
        const int64_t dst = ((slot + static_cast<int64_t>(c >> cpr_log2) * kBlockSize) << cpr_log2) + (c & (cpr - 1));
        append_store<F8>(kp, vp, dst, kx[u], vx[u], k_scale, v_scale);
      }
    }
  }
}

}  // namespace

int launch_merge(const AttnArgs& a, const MergeItem* items, int n_items, void* stream) {
  if (n_items <= 0) return cudaSuccess;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a.pool.head_dim == 128) merge_kernel<128><<<n_items, 32 * kMergeRowsPerCta, 0, s>>>(a, items);
  else merge_kernel<64><<<n_items, 32 * kMergeRowsPerCta, 0, s>>>(a, items);
  return cudaGetLastError();
}

int launch_append(const PoolView& pool, void* kp, void* vp, const int32_t* bt, int max_blocks, int num_reqs,
                  const int32_t* cu_q_lens, const int32_t* positions, const void* k_new, const void* v_new,
                  int num_tokens, void* stream) {
  if (num_tokens <= 0) return cudaSuccess;
  const int cpr = pool.head_dim / 8;
  const int cpr_log2 = cpr == 16 ? 4 : 3;   // head_dim 128 or 64
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // One warp per slice of a token's row, 8 warps a CTA, at most 8 CTAs an SM.
  const int64_t slices = (static_cast<int64_t>(pool.num_kv_heads) * cpr + kAppendSlice - 1) / kAppendSlice;
  const int64_t want = (static_cast<int64_t>(num_tokens) * slices + 7) / 8;
  const int grid = static_cast<int>(want < int64_t(sms) * 8 ? want : int64_t(sms) * 8);
  const size_t smem = num_reqs + 1 <= kAppendCuSmem ? static_cast<size_t>(num_reqs + 1) * sizeof(int32_t) : 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const auto kn = static_cast<const uint4*>(k_new);
  const auto vn = static_cast<const uint4*>(v_new);
  if (pool.elem_bytes == 1)
    append_kernel<true><<<grid, 256, smem, s>>>(kp, vp, pool.num_blocks, pool.num_kv_heads, cpr_log2, bt, max_blocks,
                                                num_reqs, cu_q_lens, positions, kn, vn, num_tokens, pool.err,
                                                pool.k_scale, pool.v_scale);
  else
    append_kernel<false><<<grid, 256, smem, s>>>(kp, vp, pool.num_blocks, pool.num_kv_heads, cpr_log2, bt, max_blocks,
                                                 num_reqs, cu_q_lens, positions, kn, vn, num_tokens, pool.err, 1.f,
                                                 1.f);
  return cudaGetLastError();
}

}  // namespace pkv

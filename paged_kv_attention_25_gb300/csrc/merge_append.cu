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
// Append: one thread per 16-byte chunk of a new K/V row (append_chunk);
// consecutive threads copy consecutive chunks of one row, so both the read of
// the new rows and the write into the block are coalesced.  Idx: the chunk
// index type, 32-bit whenever the batch's chunks fit (integer division is far
// cheaper there); chunks_per_row (D / 8) is a power of two.
template <typename Idx, bool F8>
__global__ void __launch_bounds__(256) append_kernel(void* __restrict__ kp, void* __restrict__ vp, int num_blocks,
                                                     int hkv, int cpr_log2, const int32_t* __restrict__ bt,
                                                     int max_blocks, int num_reqs, const int32_t* __restrict__ cu,
                                                     const int32_t* __restrict__ pos, const uint4* __restrict__ k_new,
                                                     const uint4* __restrict__ v_new, int num_tokens, unsigned* err,
                                                     float k_scale, float v_scale) {
  const Idx total = static_cast<Idx>(num_tokens) * static_cast<Idx>(hkv) * (static_cast<Idx>(1) << cpr_log2);
  for (Idx i = static_cast<Idx>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<Idx>(gridDim.x) * blockDim.x)
    append_chunk<Idx, F8>(i, kp, vp, num_blocks, hkv, cpr_log2, bt, max_blocks, num_reqs, cu, pos, k_new, v_new, err,
                          k_scale, v_scale);
}

template <typename Idx>
void append_launch(bool f8, int grid, cudaStream_t s, void* kp, void* vp, const PoolView& pool, int cpr_log2,
                   const int32_t* bt, int max_blocks, int num_reqs, const int32_t* cu, const int32_t* pos,
                   const uint4* kn, const uint4* vn, int num_tokens) {
  if (f8)
    append_kernel<Idx, true><<<grid, 256, 0, s>>>(kp, vp, pool.num_blocks, pool.num_kv_heads, cpr_log2, bt, max_blocks,
                                                   num_reqs, cu, pos, kn, vn, num_tokens, pool.err, pool.k_scale,
                                                   pool.v_scale);
  else
    append_kernel<Idx, false><<<grid, 256, 0, s>>>(kp, vp, pool.num_blocks, pool.num_kv_heads, cpr_log2, bt,
                                                    max_blocks, num_reqs, cu, pos, kn, vn, num_tokens, pool.err,
                                                    1.f, 1.f);
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
  const int64_t total = static_cast<int64_t>(num_tokens) * pool.num_kv_heads * cpr;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (total + 255) / 256;
  const int grid = static_cast<int>(want < int64_t(sms) * 8 ? want : int64_t(sms) * 8);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const auto kn = static_cast<const uint4*>(k_new);
  const auto vn = static_cast<const uint4*>(v_new);
  const bool f8 = pool.elem_bytes == 1;
  if (total + int64_t(grid) * 256 < (int64_t(1) << 31))   // the loop index stays below 2^31 too
    append_launch<uint32_t>(f8, grid, s, kp, vp, pool, cpr_log2, bt, max_blocks, num_reqs, cu_q_lens, positions, kn, vn,
                            num_tokens);
  else
    append_launch<uint64_t>(f8, grid, s, kp, vp, pool, cpr_log2, bt, max_blocks, num_reqs, cu_q_lens, positions, kn, vn,
                            num_tokens);
  return cudaGetLastError();
}

}  // namespace pkv

// Log-sum-exp merge of split-KV partials, and the paged KV append.
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math_constants.h>

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
// Append: every 16-byte chunk of a new K/V row goes to its slot
//   pool[block_tables[r][p / 16]][g][p % 16][:]
// (fixed-size blocks in non-contiguous memory, "LLM上下文缓存与状态复用机制的分析和探索",
// section 3.1).  Consecutive threads copy consecutive chunks of one row, so both
// the read of the new rows and the write into the block are coalesced.
// Idx: the chunk index type, 32-bit whenever the batch's chunks fit (integer
// division is far cheaper there); chunks_per_row (D / 8) is a power of two.
// F8: the pool holds e4m3 codes; each element is quantised on the way in to
// the code nearest (ties to even) to the fp32 quotient x / scale, finite
// values beyond 448 saturating (the conversion's satfinite mode), so an
// 8-element chunk of the new row becomes 8 bytes of the block.

// Four bf16 (two packed words, lowest element in the low half) -> four e4m3
// codes, lowest element in the lowest byte.
__device__ __forceinline__ uint32_t quant_e4m3x4(uint32_t w0, uint32_t w1, float scale) {
  const float x0 = __uint_as_float(w0 << 16), x1 = __uint_as_float(w0 & 0xffff0000u);
  const float x2 = __uint_as_float(w1 << 16), x3 = __uint_as_float(w1 & 0xffff0000u);
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(x0, scale), __fdiv_rn(x1, scale)), __NV_SATFINITE,
                                               __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(x2, scale), __fdiv_rn(x3, scale)), __NV_SATFINITE,
                                               __NV_E4M3);
  return lo | (hi << 16);
}

template <typename Idx, bool F8>
__global__ void __launch_bounds__(256) append_kernel(void* __restrict__ kp, void* __restrict__ vp, int num_blocks,
                                                     int hkv, int cpr_log2, const int32_t* __restrict__ bt,
                                                     int max_blocks, int num_reqs, const int32_t* __restrict__ cu,
                                                     const int32_t* __restrict__ pos, const uint4* __restrict__ k_new,
                                                     const uint4* __restrict__ v_new, int num_tokens, unsigned* err,
                                                     float k_scale, float v_scale) {
  const int chunks_per_row = 1 << cpr_log2;
  const Idx total = static_cast<Idx>(num_tokens) * static_cast<Idx>(hkv) * static_cast<Idx>(chunks_per_row);
  for (Idx i = static_cast<Idx>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<Idx>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i & static_cast<Idx>(chunks_per_row - 1));
    const Idx row = i >> cpr_log2;   // t * hkv + g
    const int g = static_cast<int>(row % static_cast<Idx>(hkv));
    const int t = static_cast<int>(row / static_cast<Idx>(hkv));
    int lo = 0, hi = num_reqs - 1;             // last r with cu[r] <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
    }
    const int p = __ldg(pos + t);
    if (p < 0 || p >= max_blocks * kBlockSize) {
      if (c == 0) atomicOr(err, PKV_DEVERR_POSITION);
      continue;
    }
    const int pb = __ldg(bt + static_cast<int64_t>(lo) * max_blocks + p / kBlockSize);
    if (pb < 0 || pb >= num_blocks) {
      if (c == 0) atomicOr(err, PKV_DEVERR_BLOCK_ID);
      continue;
    }
    const int64_t dst = ((static_cast<int64_t>(pb) * hkv + g) * kBlockSize + (p % kBlockSize)) * chunks_per_row + c;
    if constexpr (F8) {
      const uint4 kx = __ldg(k_new + i), vx = __ldg(v_new + i);
      static_cast<uint2*>(kp)[dst] = make_uint2(quant_e4m3x4(kx.x, kx.y, k_scale), quant_e4m3x4(kx.z, kx.w, k_scale));
      static_cast<uint2*>(vp)[dst] = make_uint2(quant_e4m3x4(vx.x, vx.y, v_scale), quant_e4m3x4(vx.z, vx.w, v_scale));
    } else {
      static_cast<uint4*>(kp)[dst] = __ldg(k_new + i);
      static_cast<uint4*>(vp)[dst] = __ldg(v_new + i);
    }
  }
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

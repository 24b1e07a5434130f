// The paged KV append of one 16-byte chunk of a new K/V row, and the FP8
// quantisation it uses (device code shared by the append kernel and the
// split-KV kernel's append CTAs of the fused call).
#pragma once
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace pkv {

// Four bf16 (two packed words, lowest element in the low half) -> four e4m3
// codes, lowest element in the lowest byte: the code nearest (ties to even)
// to the fp32 quotient x / scale, finite values beyond 448 saturating (the
// conversion's satfinite mode).
__device__ __forceinline__ uint32_t quant_e4m3x4(uint32_t w0, uint32_t w1, float scale) {
  const float x0 = __uint_as_float(w0 << 16), x1 = __uint_as_float(w0 & 0xffff0000u);
  const float x2 = __uint_as_float(w1 << 16), x3 = __uint_as_float(w1 & 0xffff0000u);
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(x0, scale), __fdiv_rn(x1, scale)), __NV_SATFINITE,
                                               __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(x2, scale), __fdiv_rn(x3, scale)), __NV_SATFINITE,
                                               __NV_E4M3);
  return lo | (hi << 16);
}

// Two bf16 (one packed word) -> two e4m3 codes (lowest element in the low byte).
__device__ __forceinline__ uint32_t quant_e4m3x2(uint32_t w, float scale) {
  const float x0 = __uint_as_float(w << 16), x1 = __uint_as_float(w & 0xffff0000u);
  return __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(x0, scale), __fdiv_rn(x1, scale)), __NV_SATFINITE, __NV_E4M3);
}

// Chunk i of the new rows, flattened as [token][KV head][chunk] with
// 2^cpr_log2 chunks (of 8 elements) per row, goes to its slot
//   pool[block_tables[r][p / 16]][g][p % 16][chunk]
// for the token's request r (binary search of cu_q_lens) and position p
// (fixed-size blocks in non-contiguous memory, "LLM上下文缓存与状态复用机制的
// 分析和探索", section 3.1).  append_dst returns that slot's chunk index, or
// -1 for an out-of-range position or block id (flagged in the error word).
template <typename Idx>
__device__ __forceinline__ int64_t append_dst(Idx i, int num_blocks, int hkv, int cpr_log2,
                                              const int32_t* __restrict__ bt, int max_blocks, int num_reqs,
                                              const int32_t* __restrict__ cu, const int32_t* __restrict__ pos,
                                              unsigned* err) {
  const int chunks_per_row = 1 << cpr_log2;
  const int c = static_cast<int>(i & static_cast<Idx>(chunks_per_row - 1));
  const Idx row = i >> cpr_log2;   // t * hkv + g
  const int g = static_cast<int>(row % static_cast<Idx>(hkv));
  const int t = static_cast<int>(row / static_cast<Idx>(hkv));
  int lo = 0, hi = num_reqs - 1;   // last r with cu[r] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
  }
  const int p = __ldg(pos + t);
  if (p < 0 || p >= max_blocks * kBlockSize) {
    if (c == 0) atomicOr(err, PKV_DEVERR_POSITION);
    return -1;
  }
  const int pb = __ldg(bt + static_cast<int64_t>(lo) * max_blocks + p / kBlockSize);
  if (pb < 0 || pb >= num_blocks) {
    if (c == 0) atomicOr(err, PKV_DEVERR_BLOCK_ID);
    return -1;
  }
  return ((static_cast<int64_t>(pb) * hkv + g) * kBlockSize + (p % kBlockSize)) * chunks_per_row + c;
}

// Stores one chunk (8 bf16 of K and of V) at chunk index dst of the pool.
// F8: quantised to 8 codes each.
template <bool F8>
__device__ __forceinline__ void append_store(void* __restrict__ kp, void* __restrict__ vp, int64_t dst, uint4 kx,
                                             uint4 vx, float k_scale, float v_scale) {
  if constexpr (F8) {
    static_cast<uint2*>(kp)[dst] = make_uint2(quant_e4m3x4(kx.x, kx.y, k_scale), quant_e4m3x4(kx.z, kx.w, k_scale));
    static_cast<uint2*>(vp)[dst] = make_uint2(quant_e4m3x4(vx.x, vx.y, v_scale), quant_e4m3x4(vx.z, vx.w, v_scale));
  } else {
    static_cast<uint4*>(kp)[dst] = kx;
    static_cast<uint4*>(vp)[dst] = vx;
  }
}

template <typename Idx, bool F8>
__device__ __forceinline__ void append_chunk(Idx i, void* __restrict__ kp, void* __restrict__ vp, int num_blocks,
                                             int hkv, int cpr_log2, const int32_t* __restrict__ bt, int max_blocks,
                                             int num_reqs, const int32_t* __restrict__ cu,
                                             const int32_t* __restrict__ pos, const uint4* __restrict__ k_new,
                                             const uint4* __restrict__ v_new, unsigned* err, float k_scale,
                                             float v_scale) {
  const int64_t dst = append_dst<Idx>(i, num_blocks, hkv, cpr_log2, bt, max_blocks, num_reqs, cu, pos, err);
  if (dst >= 0) append_store<F8>(kp, vp, dst, __ldg(k_new + i), __ldg(v_new + i), k_scale, v_scale);
}

}  // namespace pkv

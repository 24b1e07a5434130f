// Log-sum-exp merge of one query row's split partials (device code shared by
// the merge kernel and the split-KV kernel's last split of a group).
#pragma once
#include <cuda_runtime.h>
#include <math_constants.h>

#include "internal.h"
#include "ptx.cuh"

namespace pkv {

// One warp merges row r of merge item mi.  Split s of the row holds O_s
// (normalised, fp32) and LSE_s; the combined row is
//   LSE = M + ln sum_s exp(LSE_s - M),  O = sum_s exp(LSE_s - LSE) O_s,
// which equals attention over the union of the splits' key ranges (the
// split-and-merge of "PersistentKV: Page-Aware Decode Scheduling for
// Long-Context LLM Serving on Commodity GPUs", section 2).  Partials are read
// through L2 (other SMs wrote them in this launch or the previous one).
template <int D>
__device__ __forceinline__ void merge_row(const AttnArgs& a, const MergeItem& mi, int r, int lane) {
  constexpr int kDPL = D / 32;
  constexpr float kLog2e = 1.4426950408889634f;
  constexpr float kLn2 = 0.69314718055994530942f;
  const int G = a.group;
  const int rows = mi.q_count * G;
  float mx = -CUDART_INF_F;
  for (int s = lane; s < mi.nsplit; s += 32) mx = fmaxf(mx, __ldcg(a.part_lse + mi.part_base + s * rows + r));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float acc[kDPL];
#pragma unroll
  for (int d = 0; d < kDPL; ++d) acc[d] = 0.f;
  float wsum = 0.f;
  if (mx != -CUDART_INF_F) {
#pragma unroll 4
    for (int s = 0; s < mi.nsplit; ++s) {
      const int pr = mi.part_base + s * rows + r;
      const float w = fast_exp2((__ldcg(a.part_lse + pr) - mx) * kLog2e);
      wsum += w;
      const float* src = a.part_o + static_cast<int64_t>(pr) * D + lane * kDPL;
      if constexpr (kDPL == 4) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(src));
        acc[0] = fmaf(w, v.x, acc[0]); acc[1] = fmaf(w, v.y, acc[1]);
        acc[2] = fmaf(w, v.z, acc[2]); acc[3] = fmaf(w, v.w, acc[3]);
      } else {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(src));
        acc[0] = fmaf(w, v.x, acc[0]); acc[1] = fmaf(w, v.y, acc[1]);
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const int t = mi.q_start + r / G;
  const int h = mi.kv_head * G + r % G;
  uint16_t* dst = static_cast<uint16_t*>(a.o) + (static_cast<int64_t>(t) * a.num_q_heads + h) * D + lane * kDPL;
  if constexpr (kDPL == 4) {
    uint2 w;
    w.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    w.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = w;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
  if (lane == 0 && a.lse)
    a.lse[static_cast<int64_t>(t) * a.num_q_heads + h] = wsum > 0.f ? mx + fast_log2(wsum) * kLn2 : -CUDART_INF_F;
}

}  // namespace pkv

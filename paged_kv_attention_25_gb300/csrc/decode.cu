// Split-KV paged attention for the decode regime (few query rows per KV head).
//
// One CTA runs one work item: a request, one KV head, up to kDecodeMaxRows
// query rows (tokens x grouped query heads) and a range of key positions.
// The item's KV blocks are streamed from HBM exactly once: each (block, KV
// head) is one contiguous 16 x D bf16 chunk of the pool, fetched with a 1-D
// bulk copy (cp.async.bulk) into a per-warp ring of shared-memory stages
// tracked by mbarriers.  The four warps take blocks round-robin and keep their
// own online-softmax state (running max m, sum l, fp32 accumulator); the CTA
// merges the four states at the end and writes either the final O / LSE or a
// split partial; the last split of a group to finish combines the group's
// partials by log-sum-exp (split-KV as in
// "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving on
// Commodity GPUs", section 2; attention as in "Stateful Large Language Model
// Serving with Pensieve", abstract).
//
// Arithmetic: scores in fp32 with scale*log2(e) folded into q, exp2 on the
// SFU, fp32 accumulation; O rounded to bf16 once at the end.
//
// FP8 pools (F8): the chunks are e4m3 codes, half the bytes, so each warp
// keeps twice the stages in flight.  The codes are widened to f16 by the
// conversion instruction (exact) and multiplied with mixed-precision FMAs
// (f16 operands, fp32 accumulation; see load_row_f16); q and p are f16,
// k_scale goes into each score's scale and v_scale into the final 1/l.
// One-row FP8 items with D = 128 (plain decode) take their dot products on
// the warp-level MMA instead (see stream_item).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <type_traits>

#include "append.cuh"
#include "internal.h"
#include "merge.cuh"
#include "ptx.cuh"

namespace pkv {
namespace {

constexpr int kWarps = 4;

template <int D, bool F8>
struct DecodeSmem {
  static constexpr int kStages = F8 ? 4 : 2;                   // per-warp ring depth
  static constexpr int kChunk = kBlockSize * D * (F8 ? 1 : 2);  // bytes of one (block, head) of K or V
  static constexpr int kStage = 2 * kChunk;                    // K then V
  static constexpr int kRing = kWarps * kStages * kStage;
  static constexpr int kMergeFloats = kWarps * kDecodeMaxRows * (D + 2);
  static constexpr int kPBuf = kWarps * kDecodeMaxRows * kBlockSize * 4;
  static constexpr int kBars = kWarps * kStages * 8;
  // + 1024: the ring is placed at the first 1024-byte boundary (the tensor
  // map's 128-byte swizzle repeats every 1024 bytes).
  static constexpr int kTotal = kRing + kMergeFloats * 4 + kPBuf + kBars + 16 + 1024;
};

// Head dims [lane*kDPL, lane*kDPL + kDPL) of one bf16 row as floats (exact).
template <int kDPL>
__device__ __forceinline__ void load_row(const uint8_t* p, float* f) {
  if constexpr (kDPL == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    f[0] = bf16lo_to_f32(v.x); f[1] = bf16hi_to_f32(v.x);
    f[2] = bf16lo_to_f32(v.y); f[3] = bf16hi_to_f32(v.y);
  } else {
    const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
    f[0] = bf16lo_to_f32(v); f[1] = bf16hi_to_f32(v);
  }
}
// The same dims of one row of e4m3 codes as f16 values, two per 32-bit word
// (lowest element in the low half): the conversion instruction widens each
// pair of codes exactly (every e4m3 value is an f16 value).
template <int kDPL>
__device__ __forceinline__ void load_row_f16(const uint8_t* p, uint32_t* w) {
  if constexpr (kDPL == 4) e4m3x4_to_f16x4(*reinterpret_cast<const uint32_t*>(p), w[0], w[1]);
  else w[0] = e4m3x2_lo_to_f16x2(*reinterpret_cast<const uint16_t*>(p));
}
// c0 += lo(a) * lo(b), c1 += hi(a) * hi(b): f16 operands, exact products,
// fp32 accumulation.
__device__ __forceinline__ void fma_f16x2(float& c0, float& c1, uint32_t a, uint32_t b) {
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\tfma.rn.f32.f16 %1, ah, bh, %1;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "r"(a), "r"(b));
}
// c0 += p * lo(b), c1 += p * hi(b), p an f16.
__device__ __forceinline__ void fma_f16_bcast(float& c0, float& c1, uint16_t p, uint32_t b) {
  asm("{\n\t.reg .b16 bl, bh;\n\tmov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.f16 %0, %2, bl, %0;\n\tfma.rn.f32.f16 %1, %2, bh, %1;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "h"(p), "r"(b));
}
// d += A B for one 16 x 8 x 16 tile of the warp-level MMA: f16 operands, two
// per register (lower index in the low half), fp32 accumulators.  Thread
// t = 4g + c holds A elements (row, col) (g, 2c..2c+1), (g+8, 2c..2c+1),
// (g, 2c+8..2c+9), (g+8, 2c+8..2c+9); B elements (2c..2c+1, g) and
// (2c+8..2c+9, g); D elements (g, 2c), (g, 2c+1), (g+8, 2c), (g+8, 2c+1).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Byte offset of 16-byte chunk x of row r of a 128-byte-row tile landed with
// the tensor map's 128-byte swizzle.
__device__ __forceinline__ int swz128(int r, int x) { return r * 128 + ((x ^ (r & 7)) << 4); }

// The streaming part of one item for items of at most R query rows (R = 1, 2
// or 4: the row loops are unrolled for R, so a one-row decode item issues no
// instructions for absent rows).  Each warp streams its share of the blocks
// and leaves its online-softmax state (m, l, acc) for rows [0, rows) in
// `merge`.
//
// Lane layout.  Lane l holds head dims [l*D/32, (l+1)*D/32) of q, of every
// key and of the accumulator; a block's 16 partial dot products are then
// summed over the 32 lanes by a transpose-reduce (15 shuffles per row).
//
// One-row FP8 items with D = 128 (kMma: plain decode over an FP8 pool) are
// limited in that layout by the integer pipe, not by HBM: the CUDA cores have
// no FMA with f16 operands and fp32 accumulation, so the widening of every
// operand is issued besides each fp32 FMA.  The warp-level MMA (16 x 8 x 16,
// f16 operands, fp32 accumulation) has exactly that arithmetic, so these
// items take each 16-key block's dot products on it, all eight MMA columns
// copies of q (or of p): it serves as a dot-product instruction, not for its
// throughput.  Thread t = 4g + c (g = t / 4, c = t % 4):
//  * S = K q: k-step s (of 8) takes dims 32c + 4s .. 32c + 4s + 3 of keys g
//    and g+8 (A) and of q (B); the thread ends with the scores of keys g and
//    g+8 (D columns are copies).
//  * O^T += V^T p: the k index is the key (keys 2c, 2c+1, 2c+8 and 2c+9 in
//    the thread's A fragments); m-tile j (of 8) covers dims 16g + 2j (row g)
//    and 16g + 2j + 1 (row g+8).  A byte permute pairs the codes of keys 2c
//    and 2c+1 (2c+8 and 2c+9) of one dim before the conversion, so that each
//    converted pair is one A register.
//  * The blocks land through a 2-D tensor map with 128-byte swizzle (chunk x
//    of row r at chunk x ^ (r % 8)).  The four threads of a row group read
//    the same dims of four keys; the swizzle puts them on different banks.
//  * The accumulator is rescaled only in blocks that raise the running max.
// q and p are f16 and the codes are widened to f16 (exact) as in the
// general layout.
template <int D, bool F8, int R>
__device__ __forceinline__ void stream_item(const AttnArgs& a, const WorkItem& it, int rows, uint8_t* ring,
                                            float* merge, float* pbuf, uint64_t* bars, volatile int* s_abort,
                                            const CUtensorMap* dmk, const CUtensorMap* dmv) {
  using S = DecodeSmem<D, F8>;
  constexpr int kStages = S::kStages;
  constexpr int kDPL = D / 32;   // head dims per lane
  constexpr bool kMma = F8 && R == 1 && D == 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.group;
  const int Hkv = a.pool.num_kv_heads;
  const int g = it.kv_head;
  const int mg = lane >> 2, mc = lane & 3;   // kMma: row group and column pair of the MMA fragments

  // Per-row query (pre-scaled by scale*log2 e) and position; rows >= `rows`
  // are inert.  F8: q is held as f16 pairs (qw; exact for |q| within f16's
  // range) and the whole scale, k_scale included, goes onto each score.
  const float qs = a.scale_log2;
  const float s_scale = a.scale_log2 * a.pool.k_scale;
  float q[R][kDPL];
  uint32_t qw[R][kDPL / 2];
  uint32_t qb[8][2];   // kMma: q's B fragments (f16 pairs), dims 32c + 4s + {0,1} and {2,3}
  int qpos[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    qpos[r] = -1;
#pragma unroll
    for (int d = 0; d < kDPL; ++d) q[r][d] = 0.f;
#pragma unroll
    for (int j = 0; j < kDPL / 2; ++j) qw[r][j] = 0u;
    if constexpr (kMma) {
#pragma unroll
      for (int k = 0; k < 8; ++k) qb[k][0] = qb[k][1] = 0u;
    }
    if (r < rows) {
      const int t = it.q_start + r / G;
      const int h = g * G + r % G;
      qpos[r] = __ldg(a.q_positions + t);
      const uint16_t* qrow = static_cast<const uint16_t*>(a.q) + (static_cast<int64_t>(t) * a.num_q_heads + h) * D;
      const uint16_t* src = qrow + lane * kDPL;
      if constexpr (kMma) {
        // Dims 32c + 8u .. 32c + 8u + 7: k-steps 2u and 2u + 1.
        const uint4* qc = reinterpret_cast<const uint4*>(qrow + 32 * mc);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 w = __ldg(qc + u);
          qb[2 * u][0] = pack_f16x2(bf16lo_to_f32(w.x), bf16hi_to_f32(w.x));
          qb[2 * u][1] = pack_f16x2(bf16lo_to_f32(w.y), bf16hi_to_f32(w.y));
          qb[2 * u + 1][0] = pack_f16x2(bf16lo_to_f32(w.z), bf16hi_to_f32(w.z));
          qb[2 * u + 1][1] = pack_f16x2(bf16lo_to_f32(w.w), bf16hi_to_f32(w.w));
        }
      } else if constexpr (F8) {
#pragma unroll
        for (int j = 0; j < kDPL / 2; ++j) {
          const uint32_t w = reinterpret_cast<const uint32_t*>(src)[j];
          qw[r][j] = pack_f16x2(bf16lo_to_f32(w), bf16hi_to_f32(w));
        }
      } else {
        float qf[kDPL];
        load_row<kDPL>(reinterpret_cast<const uint8_t*>(src), qf);
#pragma unroll
        for (int d = 0; d < kDPL; ++d) q[r][d] = qf[d] * qs;
      }
    }
  }
  // Key range from the planner's position bound (the device positions only
  // mask), so that the block-table reads need not wait for them.
  const int kv_end = min(it.kv_end, it.pos_max[0] + 1);
  const int blk0 = it.kv_start / kBlockSize;
  const int nblk = kv_end > it.kv_start ? (kv_end - it.kv_start + kBlockSize - 1) / kBlockSize : 0;
  const int nb_w = nblk > warp ? (nblk - warp + kWarps - 1) / kWarps : 0;   // blocks of this warp

  uint8_t* my_ring = ring + warp * kStages * S::kStage;
  uint64_t* my_full = bars + warp * kStages;
  float* my_p = pbuf + warp * kDecodeMaxRows * kBlockSize;
  const int32_t* bt_row = a.block_tables + static_cast<int64_t>(it.req) * a.max_blocks;

  // Physical block ids of this warp's iterations, 32 at a time (lane l holds iteration base+l).
  auto load_ids = [&](int base) -> int {
    const int i = base + lane;
    int pb = -1;
    if (i < nb_w) {
      const int col = blk0 + warp + kWarps * i;
      pb = col < a.max_blocks ? __ldg(bt_row + col) : -1;
      if (pb < 0 || pb >= a.pool.num_blocks) {
        atomicOr(a.pool.err, PKV_DEVERR_BLOCK_ID);
        pb = -1;
      }
    }
    return pb;
  };
  int ids_cur = load_ids(0), ids_next = load_ids(32), win = 0;
  // Fused call: positions of the item's tokens (the request's new tokens),
  // whose keys and values come from the new rows rather than the pool.
  // [pmin, pmax]: this warp's iterations whose block holds one of them (an
  // empty range when none does), so that other blocks pay one test.
  const bool fused = a.k_new != nullptr;
  int tpos[kDecodeMaxRows];
  int pmin = 0x7fffffff, pmax = -1;
#pragma unroll
  for (int k = 0; k < kDecodeMaxRows; ++k) {
    tpos[k] = fused && k < it.q_count ? __ldg(a.q_positions + it.q_start + k) : -1;
    const int col = tpos[k] >= 0 ? tpos[k] / kBlockSize - blk0 : -1;   // block of the item's range
    if (col >= 0 && col % kWarps == warp) {
      pmin = min(pmin, col / kWarps);
      pmax = max(pmax, col / kWarps);
    }
  }
  __syncthreads();   // barrier initialisation visible (the id loads above are already in flight)

  auto issue = [&](int j) {
    // Only lane 0 issues; every lane evaluates the shuffle.
    const int src_lane = j & 31;
    const int pb = (j >> 5) == win ? __shfl_sync(0xffffffffu, ids_cur, src_lane)
                                   : __shfl_sync(0xffffffffu, ids_next, src_lane);
    // Test hook: CTA 0's warp 0 never issues its first copy, so that its
    // bounded wait for that stage runs out.
    const bool withheld = a.withhold == 1 && j == 0 && blockIdx.x == 0 && warp == 0;
    if (lane == 0 && !withheld) {
      const int st = j % kStages;
      uint8_t* dst = my_ring + st * S::kStage;
      if (pb >= 0) {
        const int64_t off = (static_cast<int64_t>(pb) * Hkv + g) * S::kChunk;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&my_full[st], 2 * S::kChunk);
        if constexpr (kMma) {   // the chunk's 16 rows of the [chunks * 16][D] code view, swizzled
          const int row = static_cast<int>((static_cast<int64_t>(pb) * Hkv + g) * kBlockSize);
          tma_load_2d(dst, dmk, 0, row, &my_full[st]);
          tma_load_2d(dst + S::kChunk, dmv, 0, row, &my_full[st]);
        } else {
          bulk_g2s(dst, static_cast<const uint8_t*>(a.pool.k) + off, S::kChunk, &my_full[st]);
          bulk_g2s(dst + S::kChunk, static_cast<const uint8_t*>(a.pool.v) + off, S::kChunk, &my_full[st]);
        }
      } else {
        mbar_arrive(&my_full[st]);   // invalid block: stage keeps stale data, error already flagged
      }
    }
  };

#pragma unroll
  for (int s = 0; s < kStages; ++s)
    if (s < nb_w) issue(s);

  float m[R], l[R], acc[R][kDPL];
  float acm[8][4];   // kMma: O^T fragments, m-tile j: dims 16g + 2j (elements 0, 1) and 16g + 2j + 1 (2, 3)
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m[r] = -CUDART_INF_F;
    l[r] = 0.f;
#pragma unroll
    for (int d = 0; d < kDPL; ++d) acc[r][d] = 0.f;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) acm[j][0] = acm[j][1] = acm[j][2] = acm[j][3] = 0.f;

  int consumed = 0;
  bool aborted = false;
  for (int i = 0; i < nb_w; ++i) {
    if ((i & 31) == 0 && i > 0) {   // slide the block-id window
      ids_cur = ids_next;
      win = i >> 5;
      ids_next = load_ids(i + 32);
    }
    const int st = i % kStages;
    if (!mbar_wait_warp(&my_full[st], (i / kStages) & 1, s_abort, a.wait_ns)) {
      aborted = true;
      break;
    }
    uint8_t* kb = my_ring + st * S::kStage;
    uint8_t* vb = kb + S::kChunk;
    const int key0 = (blk0 + warp + kWarps * i) * kBlockSize;
    constexpr int kRowBytes = D * (F8 ? 1 : 2);
    constexpr int kLaneBytes = kDPL * (F8 ? 1 : 2);
    if (i >= pmin && i <= pmax) {   // fused call only
      // The block's slots of this step's tokens may not be written yet (the
      // launch's append CTAs write them): take those rows from the new K/V,
      // quantised as the append stores them.  Each lane rewrites its own
      // slice of the row, the slice it reads below.
#pragma unroll
      for (int k = 0; k < kDecodeMaxRows; ++k) {
        const int rr = tpos[k] - key0;
        if (rr >= 0 && rr < kBlockSize) {
          const int64_t src = (static_cast<int64_t>(it.q_start + k) * Hkv + g) * D + lane * kDPL;   // elements
          const uint16_t* kn = static_cast<const uint16_t*>(a.k_new) + src;
          const uint16_t* vn = static_cast<const uint16_t*>(a.v_new) + src;
          const int dof = kMma ? swz128(rr, lane >> 2) + (lane & 3) * 4 : rr * kRowBytes + lane * kLaneBytes;
          uint8_t* kd = kb + dof;
          uint8_t* vd = vb + dof;
          if constexpr (F8) {
            if constexpr (kDPL == 4) {
              const uint2 kx = *reinterpret_cast<const uint2*>(kn), vx = *reinterpret_cast<const uint2*>(vn);
              *reinterpret_cast<uint32_t*>(kd) = quant_e4m3x4(kx.x, kx.y, a.pool.k_scale);
              *reinterpret_cast<uint32_t*>(vd) = quant_e4m3x4(vx.x, vx.y, a.pool.v_scale);
            } else {
              *reinterpret_cast<uint16_t*>(kd) =
                  static_cast<uint16_t>(quant_e4m3x2(*reinterpret_cast<const uint32_t*>(kn), a.pool.k_scale));
              *reinterpret_cast<uint16_t*>(vd) =
                  static_cast<uint16_t>(quant_e4m3x2(*reinterpret_cast<const uint32_t*>(vn), a.pool.v_scale));
            }
          } else {
            if constexpr (kDPL == 4) {
              *reinterpret_cast<uint2*>(kd) = *reinterpret_cast<const uint2*>(kn);
              *reinterpret_cast<uint2*>(vd) = *reinterpret_cast<const uint2*>(vn);
            } else {
              *reinterpret_cast<uint32_t*>(kd) = *reinterpret_cast<const uint32_t*>(kn);
              *reinterpret_cast<uint32_t*>(vd) = *reinterpret_cast<const uint32_t*>(vn);
            }
          }
          // These generic writes precede the next bulk copy into the stage.
          fence_proxy_async_smem();
        }
      }
      __syncwarp();   // the rows below are read by other lanes than their writers
    }

    if constexpr (kMma) {
      // S = K q over 8 k-steps; w0 / w1 hold dims 32c .. 32c + 31 of keys g and g + 8.
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
      {
        uint32_t w0[8], w1[8];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint4 x0 = *reinterpret_cast<const uint4*>(kb + swz128(mg, 2 * mc + u));
          const uint4 x1 = *reinterpret_cast<const uint4*>(kb + swz128(mg + 8, 2 * mc + u));
          w0[4 * u] = x0.x; w0[4 * u + 1] = x0.y; w0[4 * u + 2] = x0.z; w0[4 * u + 3] = x0.w;
          w1[4 * u] = x1.x; w1[4 * u + 1] = x1.y; w1[4 * u + 2] = x1.z; w1[4 * u + 3] = x1.w;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          uint32_t a0, a2, a1, a3;
          e4m3x4_to_f16x4(w0[k], a0, a2);
          e4m3x4_to_f16x4(w1[k], a1, a3);
          mma_16816(sc, a0, a1, a2, a3, qb[k][0], qb[k][1]);
        }
      }
      float s0 = sc[0] * s_scale, s1 = sc[2] * s_scale;   // keys g and g + 8
      if (key0 + mg > qpos[0] || key0 + mg >= kv_end) s0 = -CUDART_INF_F;
      if (key0 + mg + 8 > qpos[0] || key0 + mg + 8 >= kv_end) s1 = -CUDART_INF_F;
      // Max and sum over the block's 16 keys (the four threads of a row group hold copies).
      float mx = fmaxf(s0, s1);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_new = fmaxf(m[0], mx);
      const float m_use = m_new == -CUDART_INF_F ? 0.f : m_new;
      const float p0 = fast_exp2(s0 - m_use), p1 = fast_exp2(s1 - m_use);
      float ps = p0 + p1;
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      if (m_new != m[0]) {   // warp-uniform: m and mx are the same in every lane
        const float alpha = fast_exp2(m[0] - m_use);
        l[0] *= alpha;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          acm[j][0] *= alpha; acm[j][1] *= alpha; acm[j][2] *= alpha; acm[j][3] *= alpha;
        }
        m[0] = m_new;
      }
      l[0] += ps;
      // p's B fragments: (p(2c), p(2c+1)) and (p(2c+8), p(2c+9)), from the
      // row groups 2c and 2c + 1, which hold (p(g), p(g+8)).
      const uint32_t pk = pack_f16x2(p0, p1);
      const uint32_t px = __shfl_sync(0xffffffffu, pk, 8 * mc), py = __shfl_sync(0xffffffffu, pk, 8 * mc + 4);
      const uint32_t pb0 = __byte_perm(px, py, 0x5410), pb1 = __byte_perm(px, py, 0x7632);
      // O^T += V^T p.  v[k]: dims 16g .. 16g + 15 of keys 2c, 2c+1, 2c+8, 2c+9.
      // In the item's last block, keys at or past kv_end read as zero (stale
      // codes may be NaN).
      auto pv = [&](auto masked) {
        uint32_t v[4][4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int key = 2 * mc + (k & 1) + 8 * (k >> 1);
          const uint4 x = *reinterpret_cast<const uint4*>(vb + swz128(key, mg));
          v[k][0] = x.x; v[k][1] = x.y; v[k][2] = x.z; v[k][3] = x.w;
          if constexpr (decltype(masked)::value) {
            if (key0 + key >= kv_end) v[k][0] = v[k][1] = v[k][2] = v[k][3] = 0u;
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {   // word i: dims 16g + 4i .. 16g + 4i + 3 (m-tiles 2i and 2i + 1)
          const uint32_t lo01 = __byte_perm(v[0][i], v[1][i], 0x5140), hi01 = __byte_perm(v[0][i], v[1][i], 0x7362);
          const uint32_t lo89 = __byte_perm(v[2][i], v[3][i], 0x5140), hi89 = __byte_perm(v[2][i], v[3][i], 0x7362);
          uint32_t a[8];
          e4m3x4_to_f16x4(lo01, a[0], a[1]);
          e4m3x4_to_f16x4(lo89, a[2], a[3]);
          e4m3x4_to_f16x4(hi01, a[4], a[5]);
          e4m3x4_to_f16x4(hi89, a[6], a[7]);
          mma_16816(acm[2 * i], a[0], a[1], a[2], a[3], pb0, pb1);
          mma_16816(acm[2 * i + 1], a[4], a[5], a[6], a[7], pb0, pb1);
        }
      };
      if (key0 + kBlockSize > kv_end) pv(std::true_type{});   // warp-uniform
      else pv(std::false_type{});
    } else {
      // q . k for 16 keys, this lane's dims.
      float part[R][kBlockSize];
#pragma unroll
      for (int k = 0; k < kBlockSize; ++k) {
        if constexpr (F8) {
          uint32_t kw[kDPL / 2];
          load_row_f16<kDPL>(kb + k * kRowBytes + lane * kLaneBytes, kw);
#pragma unroll
          for (int r = 0; r < R; ++r) {
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int j = 0; j < kDPL / 2; ++j) fma_f16x2(s0, s1, qw[r][j], kw[j]);
            part[r][k] = s0 + s1;
          }
        } else {
          float kf[kDPL];
          load_row<kDPL>(kb + k * kRowBytes + lane * kLaneBytes, kf);
#pragma unroll
          for (int r = 0; r < R; ++r) {
            float s = 0.f;
#pragma unroll
            for (int d = 0; d < kDPL; ++d) s = fmaf(q[r][d], kf[d], s);
            part[r][k] = s;
          }
        }
      }

#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (r >= rows) break;
        // Transpose-reduce the 16 partial dot products over the 32 lanes:
        // afterwards lane holds the full score of key (lane >> 1).
        float v8[8], v4[4], v2[2], v1;
        const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float send = b4 ? part[r][j] : part[r][j + 8];
          const float keep = b4 ? part[r][j + 8] : part[r][j];
          v8[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float send = b3 ? v8[j] : v8[j + 4];
          const float keep = b3 ? v8[j + 4] : v8[j];
          v4[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float send = b2 ? v4[j] : v4[j + 2];
          const float keep = b2 ? v4[j + 2] : v4[j];
          v2[j] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
        {
          const float send = b1 ? v2[0] : v2[1];
          const float keep = b1 ? v2[1] : v2[0];
          v1 = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
        float s = v1 + __shfl_xor_sync(0xffffffffu, v1, 1);
        if constexpr (F8) s = s * s_scale;
        const int key = key0 + (lane >> 1);
        if (key > qpos[r] || key >= kv_end) s = -CUDART_INF_F;
        float mx = s;
#pragma unroll
        for (int o = 2; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_new = fmaxf(m[r], mx);
        const float m_use = m_new == -CUDART_INF_F ? 0.f : m_new;
        const float alpha = fast_exp2(m[r] - m_use);
        const float p = fast_exp2(s - m_use);
        float ps = p;
#pragma unroll
        for (int o = 2; o < 32; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        l[r] = l[r] * alpha + ps;
        m[r] = m_new;
#pragma unroll
        for (int d = 0; d < kDPL; ++d) acc[r][d] *= alpha;
        if ((lane & 1) == 0) {
          if constexpr (F8)   // f16 p for the mixed-precision PV FMAs
            reinterpret_cast<uint16_t*>(my_p)[r * kBlockSize + (lane >> 1)] =
                static_cast<uint16_t>(pack_f16x2(p, 0.f) & 0xffffu);
          else
            my_p[r * kBlockSize + (lane >> 1)] = p;
        }
      }
      __syncwarp();

      // acc += p . V for this lane's dims.  In the item's last block, keys at
      // or past kv_end read as zero, so that no stale value (NaN included) meets
      // their zero p; every other block is whole and skips the test.
      auto pv = [&](auto masked) {
#pragma unroll
        for (int k = 0; k < kBlockSize; ++k) {
          if constexpr (F8) {
            uint32_t vw[kDPL / 2];
            load_row_f16<kDPL>(vb + k * kRowBytes + lane * kLaneBytes, vw);
            if constexpr (decltype(masked)::value) {
              const bool live = key0 + k < kv_end;
#pragma unroll
              for (int j = 0; j < kDPL / 2; ++j) vw[j] = live ? vw[j] : 0u;
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
              if (r >= rows) break;
              const uint16_t p = reinterpret_cast<const uint16_t*>(my_p)[r * kBlockSize + k];
#pragma unroll
              for (int j = 0; j < kDPL / 2; ++j) fma_f16_bcast(acc[r][2 * j], acc[r][2 * j + 1], p, vw[j]);
            }
          } else {
            float vf[kDPL];
            load_row<kDPL>(vb + k * kRowBytes + lane * kLaneBytes, vf);
            if constexpr (decltype(masked)::value) {
              const bool live = key0 + k < kv_end;
#pragma unroll
              for (int d = 0; d < kDPL; ++d) vf[d] = live ? vf[d] : 0.f;
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
              if (r >= rows) break;
              const float p = my_p[r * kBlockSize + k];
#pragma unroll
              for (int d = 0; d < kDPL; ++d) acc[r][d] = fmaf(p, vf[d], acc[r][d]);
            }
          }
        }
      };
      if (key0 + kBlockSize > kv_end) pv(std::true_type{});   // warp-uniform
      else pv(std::false_type{});
    }
    __syncwarp();
    consumed = i + 1;
    if (i + kStages < nb_w) issue(i + kStages);
  }

  if (aborted) {
    if (lane == 0) atomicOr(a.pool.err, PKV_DEVERR_TIMEOUT);
    *s_abort = 1;
    // Let this warp's copies in flight land before the CTA's shared memory is released.
    for (int j = consumed; j < min(nb_w, consumed + kStages); ++j)
      (void)mbar_wait_warp(&my_full[j % kStages], (j / kStages) & 1, nullptr, a.wait_ns);
  }

  // This warp's (m, l, acc) states for the CTA-wide merge.
  float* wm = merge + (warp * kDecodeMaxRows) * (D + 2);
  if constexpr (kMma) {
    if (rows > 0) {
      if (mc == 0) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          wm[16 * mg + 2 * j] = acm[j][0];
          wm[16 * mg + 2 * j + 1] = acm[j][2];
        }
      }
      if (lane == 0) {
        wm[D] = m[0];
        wm[D + 1] = l[0];
      }
    }
  } else {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (r >= rows) break;
      float* dst = wm + r * (D + 2);
#pragma unroll
      for (int d = 0; d < kDPL; ++d) dst[lane * kDPL + d] = acc[r][d];
      if (lane == 0) {
        dst[D] = m[r];
        dst[D + 1] = l[r];
      }
    }
  }
}

// The fused call's append CTAs, the last n CTAs of the grid.  (Placed first,
// their wave, with the attention CTAs' shared-memory footprint, kept other
// work such as a concurrent swap off the SMs.)  The attention items of the
// launch never read the slots these CTAs write (they take the rows from the
// new K/V), so nothing orders the two inside the launch.
//
// The slot of chunk i is that of append_dst (the same arithmetic, checks and
// error flags), found in phases.  These CTAs inherit the attention's shared
// memory, so only 12 warps share an SM, and a chunk's lookup is a chain of
// dependent loads (request, position, block id); each thread therefore takes
// U chunks at once and runs each phase over all of them before the next:
// the new rows, then the tokens' positions, then their requests (one binary
// search of cu_q_lens per thread; the later chunks' tokens are not smaller,
// so a short forward walk finds theirs), then the block ids, then the stores.
template <bool F8>
__device__ __forceinline__ void append_role(const AttnArgs& a, int c, int n) {
  constexpr int U = 8;
  const int cpr_log2 = a.pool.head_dim == 128 ? 4 : 3;
  const int cpr = 1 << cpr_log2;
  const int hkv = a.pool.num_kv_heads;
  const uint32_t total = static_cast<uint32_t>(a.num_tokens) * hkv << cpr_log2;
  const uint32_t span = U * blockDim.x;
  const uint4* kn = static_cast<const uint4*>(a.k_new);
  const uint4* vn = static_cast<const uint4*>(a.v_new);
  for (uint32_t base = static_cast<uint32_t>(c) * span + threadIdx.x; base < total;
       base += static_cast<uint32_t>(n) * span) {
    uint4 kx[U], vx[U];
    int t[U], p[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t i = base + u * blockDim.x;
      t[u] = -1;
      if (i < total) {
        kx[u] = __ldg(kn + i);
        vx[u] = __ldg(vn + i);
        t[u] = static_cast<int>((i >> cpr_log2) / static_cast<uint32_t>(hkv));
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) p[u] = t[u] >= 0 ? __ldg(a.q_positions + t[u]) : -1;
    int r[U];
    {
      int lo = 0, hi = a.num_reqs - 1;   // last r with cu[r] <= t[0] (t[0] >= 0: base < total)
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(a.cu_q_lens + mid) <= t[0]) lo = mid; else hi = mid - 1;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (t[u] >= 0)
          while (lo + 1 < a.num_reqs && __ldg(a.cu_q_lens + lo + 1) <= t[u]) ++lo;
        r[u] = lo;
      }
    }
    int64_t dst[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      dst[u] = -1;
      if (t[u] < 0) continue;
      const uint32_t i = base + u * blockDim.x;
      const int ch = static_cast<int>(i & static_cast<uint32_t>(cpr - 1));
      if (p[u] < 0 || p[u] >= a.max_blocks * kBlockSize) {
        if (ch == 0) atomicOr(a.pool.err, PKV_DEVERR_POSITION);
        continue;
      }
      const int pb = __ldg(a.block_tables + static_cast<int64_t>(r[u]) * a.max_blocks + p[u] / kBlockSize);
      if (pb < 0 || pb >= a.pool.num_blocks) {
        if (ch == 0) atomicOr(a.pool.err, PKV_DEVERR_BLOCK_ID);
        continue;
      }
      const int g = static_cast<int>((i >> cpr_log2) % static_cast<uint32_t>(hkv));
      dst[u] = ((static_cast<int64_t>(pb) * hkv + g) * kBlockSize + (p[u] % kBlockSize)) * cpr + ch;
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (dst[u] >= 0)
        append_store<F8>(const_cast<void*>(a.pool.k), const_cast<void*>(a.pool.v), dst[u], kx[u], vx[u],
                         a.pool.k_scale, a.pool.v_scale);
  }
}

template <int D, bool F8>
__global__ void __launch_bounds__(kWarps * 32, 3)
decode_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap dmk, const __grid_constant__ CUtensorMap dmv,
              const WorkItem* __restrict__ items, int n_items) {
  if (static_cast<int>(blockIdx.x) >= n_items) {
    append_role<F8>(a, blockIdx.x - n_items, a.n_append_ctas);
    return;
  }
  using S = DecodeSmem<D, F8>;
  constexpr int kStages = S::kStages;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* ring = smem;
  float* merge = reinterpret_cast<float*>(smem + S::kRing);
  float* pbuf = merge + S::kMergeFloats;
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(pbuf) + S::kPBuf);
  volatile int* s_abort = reinterpret_cast<volatile int*>(bars + kWarps * kStages);

  // The work item and the launch's error word are read together: every global
  // round trip before the first copy is paid by every CTA.  Once any wait in
  // this launch has given up, the remaining CTAs do nothing (__syncthreads_or
  // makes the decision the same for every thread).
  const WorkItem it = items[blockIdx.x];
  const unsigned err0 = *reinterpret_cast<volatile unsigned*>(a.pool.err);
  if (__syncthreads_or((err0 & PKV_DEVERR_TIMEOUT) != 0)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.group;
  const int rows = it.q_count * G;
  const int g = it.kv_head;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kWarps * kStages; ++i) mbar_init(&bars[i], 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  // `rows` is the same for the whole CTA, so every thread takes the same branch.
  if (rows <= 1) stream_item<D, F8, 1>(a, it, rows, ring, merge, pbuf, bars, s_abort, &dmk, &dmv);
  else if (rows <= 2) stream_item<D, F8, 2>(a, it, rows, ring, merge, pbuf, bars, s_abort, &dmk, &dmv);
  else stream_item<D, F8, 4>(a, it, rows, ring, merge, pbuf, bars, s_abort, &dmk, &dmv);
  __syncthreads();

  constexpr float kLn2 = 0.69314718055994530942f;
  for (int idx = threadIdx.x; idx < rows * (D / 2); idx += blockDim.x) {
    const int r = idx / (D / 2);
    const int d = (idx % (D / 2)) * 2;
    float mw[kWarps], mstar = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      mw[w] = merge[(w * kDecodeMaxRows + r) * (D + 2) + D];
      mstar = fmaxf(mstar, mw[w]);
    }
    float lsum = 0.f, o0 = 0.f, o1 = 0.f;
    if (mstar != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float* src = merge + (w * kDecodeMaxRows + r) * (D + 2);
        const float f = fast_exp2(mw[w] - mstar);
        lsum += src[D + 1] * f;
        o0 += src[d] * f;
        o1 += src[d + 1] * f;
      }
    }
    const float inv = lsum > 0.f ? (F8 ? a.pool.v_scale : 1.f) / lsum : 0.f;
    o0 *= inv;
    o1 *= inv;
    const float lse = lsum > 0.f ? (mstar + fast_log2(lsum)) * kLn2 : -CUDART_INF_F;
    const int t = it.q_start + r / G;
    const int h = g * G + r % G;
    if (it.part < 0) {
      uint32_t* o = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.o) + (static_cast<int64_t>(t) * a.num_q_heads + h) * D + d);
      *o = pack_bf16x2(o0, o1);
      if (d == 0 && a.lse) a.lse[static_cast<int64_t>(t) * a.num_q_heads + h] = lse;
    } else {
      float2* o = reinterpret_cast<float2*>(a.part_o + static_cast<int64_t>(it.part + r) * D + d);
      *o = make_float2(o0, o1);
      if (d == 0) a.part_lse[it.part + r] = lse;
    }
  }

  // Split group: count this split as done; the split that completes the count
  // merges the group.  The barrier orders the CTA's partial writes before
  // thread 0's device-scope fence and count (release); the merging CTA's
  // thread 0 fences after the count (acquire) before the barrier that lets
  // the other warps read the partials.
  if (it.part >= 0 && it.merge_id >= 0) {
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const int last = atomicAdd(a.merge_cnt + it.merge_id, 1) == a.merge_dec[it.merge_id].nsplit - 1;
      if (last) __threadfence();
      s_last = last;
    }
    __syncthreads();
    if (s_last) {
      const MergeItem mi = a.merge_dec[it.merge_id];
      if (warp < mi.row_count) merge_row<D>(a, mi, mi.row_begin + warp, lane);
    }
  }
}

}  // namespace

template <int D, bool F8>
static int launch_decode_d(const AttnArgs& a, const void* dmap_k, const void* dmap_v, const WorkItem* items,
                           int n_items, void* stream) {
  const int smem = DecodeSmem<D, F8>::kTotal;
  cudaError_t e = smem_attr_once<decode_kernel<D, F8>>(smem);
  if (e != cudaSuccess) return e;
  decode_kernel<D, F8><<<n_items + a.n_append_ctas, kWarps * 32, smem, static_cast<cudaStream_t>(stream)>>>(
      a, *static_cast<const CUtensorMap*>(dmap_k), *static_cast<const CUtensorMap*>(dmap_v), items, n_items);
  return cudaGetLastError();
}

int launch_decode(const AttnArgs& a, const void* dmap_k, const void* dmap_v, const WorkItem* items, int n_items,
                  void* stream) {
  if (n_items + a.n_append_ctas <= 0) return cudaSuccess;
  const bool f8 = a.pool.elem_bytes == 1;
  if (a.pool.head_dim == 128)
    return f8 ? launch_decode_d<128, true>(a, dmap_k, dmap_v, items, n_items, stream)
              : launch_decode_d<128, false>(a, dmap_k, dmap_v, items, n_items, stream);
  return f8 ? launch_decode_d<64, true>(a, dmap_k, dmap_v, items, n_items, stream)
            : launch_decode_d<64, false>(a, dmap_k, dmap_v, items, n_items, stream);
}

}  // namespace pkv

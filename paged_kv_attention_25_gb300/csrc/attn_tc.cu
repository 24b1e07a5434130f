// Tensor-core paged attention for tiles of many query rows (new-turn
// prefills, recomputed evicted history, grouped-query decode): the
// "attention between multiple input tokens with a GPU cache spread over
// non-contiguous memory" of "Stateful Large Language Model Serving with
// Pensieve" (abstract), written for sm_103a.
//
// One CTA runs one work item: up to 128 query rows (tokens x grouped heads of
// one KV head, one row per TMEM lane) against a range of key positions in
// tiles of 64 keys (4 KV blocks).
//
//   warp 4  producer: reads the block table and gathers each block's K and V
//           (16 keys x 64 dims per TMA box, 128-byte swizzle) into a 2-stage
//           shared-memory ring with cp.async.bulk.tensor;
//   warp 5  MMA issuer: S = Q K^T (tcgen05.mma kind::f16, bf16 in, fp32 in
//           TMEM, double-buffered) and O += P V (P from shared memory);
//   warps 0-3 softmax: one query row per thread; read S from TMEM, apply the
//           causal mask on absolute positions, online softmax in fp32 (exp2
//           with scale*log2 e folded in), rescale O in TMEM when the running
//           max grows, write P as bf16 into shared memory; epilogue O / l.
//
// Two CTAs fit on one SM (112 KB shared memory, 256 TMEM columns each), so
// one CTA's softmax overlaps the other's tensor-core work.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "internal.h"
#include "ptx.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 192;
constexpr int kStagesTc = 2;
constexpr int kNK = kTcKeys;          // keys per tile (64)
constexpr uint32_t kTmemCols = 256;   // S0 [0,64), S1 [64,128), O [128, 128+D)
constexpr uint32_t kColO = 128;
constexpr float kRescaleLog2 = 8.f;   // lazy O rescale threshold (log2 units)

template <int D>
struct TcSmem {
  static constexpr int kHalves = D / 64;                 // 128-byte-wide column slabs
  static constexpr int kQ = kTcRows * D * 2;             // [halves][128 rows][64]
  static constexpr int kKV = kNK * D * 2;                // one stage of K (or V): [halves][64 keys][64]
  static constexpr int kP = kTcRows * kNK * 2;           // [128 rows][64 keys]
  static constexpr int kOffK = kQ;
  static constexpr int kOffV = kOffK + kStagesTc * kKV;
  static constexpr int kOffP = kOffV + kStagesTc * kKV;
  static constexpr int kOffBar = kOffP + kP;
  // barriers: k_full[2] k_empty[2] v_full[2] v_empty[2] q_full s_full[2] p_full pv_done drain
  static constexpr int kNumBars = 14;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kTotal = kOffMisc + 32;
};

enum Bar { kKFull = 0, kKEmpty = 2, kVFull = 4, kVEmpty = 6, kQFull = 8, kSFull = 9, kPFull = 11, kPvDone = 12, kDrain = 13 };

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
tc_attn_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
               const WorkItem* __restrict__ items) {
  using S = TcSmem<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {   // swizzle atoms need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(a.pool.err, PKV_DEVERR_INTERNAL);
    return;
  }
  // Once any wait in this launch has given up, the remaining CTAs do nothing.
  // (__syncthreads_or makes the decision the same for every thread of the CTA.)
  if (__syncthreads_or((*reinterpret_cast<volatile unsigned*>(a.pool.err) & PKV_DEVERR_TIMEOUT) != 0)) return;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + S::kOffMisc);
  int* s_info = reinterpret_cast<int*>(smem + S::kOffMisc + 4);   // [0] max pos, [1] min pos
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + S::kOffMisc + 12);

  const WorkItem it = items[blockIdx.x];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.group;
  const int rows = it.q_count * G;
  const int g = it.kv_head;
  const int Hkv = a.pool.num_kv_heads;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&bars[kKFull + i], 1);    // k_full, k_empty
    for (int i = 0; i < 4; ++i) mbar_init(&bars[kVFull + i], 1);    // v_full, v_empty
    mbar_init(&bars[kQFull], 128);
    mbar_init(&bars[kSFull], 1);
    mbar_init(&bars[kSFull + 1], 1);
    mbar_init(&bars[kPFull], 128);
    mbar_init(&bars[kPvDone], 1);
    mbar_init(&bars[kDrain], 1);
    s_info[0] = -1;
    s_info[1] = 0x7fffffff;
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }
  if (warp == 5) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  const int row = threadIdx.x;   // meaningful for warps 0-3
  int qpos = -1;
  if (row < 128 && row < rows) qpos = __ldg(a.q_positions + it.q_start + row / G);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (row < 128 && row < rows) {
    atomicMax(&s_info[0], qpos);
    atomicMin(&s_info[1], qpos);
  }
  __syncthreads();
  const uint32_t tmem = *s_tmem;
  const int max_pos = s_info[0];
  const int min_pos = s_info[1];
  const int kv_end = min(it.kv_end, max_pos + 1);
  const int ntiles = kv_end > it.kv_start ? (kv_end - it.kv_start + kNK - 1) / kNK : 0;

  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK = smem_u32(smem + S::kOffK);
  const uint32_t sV = smem_u32(smem + S::kOffV);
  const uint32_t sP = smem_u32(smem + S::kOffP);

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    const int32_t* bt_row = a.block_tables + static_cast<int64_t>(it.req) * a.max_blocks;
    int j = 0;
    for (; j < ntiles; ++j) {
      const int st = j % kStagesTc;
      const uint32_t ph = (j / kStagesTc) & 1;
      const int key0 = it.kv_start + j * kNK;
      const int nkeys = min(kNK, kv_end - key0);
      const int nblk = (nkeys + kBlockSize - 1) / kBlockSize;
      int pb = -1;
      if (lane < nblk) {
        const int col = key0 / kBlockSize + lane;
        pb = col < a.max_blocks ? __ldg(bt_row + col) : -1;
        if (pb < 0 || pb >= a.pool.num_blocks) {
          atomicOr(a.pool.err, PKV_DEVERR_BLOCK_ID);
          pb = -1;
        }
      }
      const int nvalid = __popc(__ballot_sync(0xffffffffu, pb >= 0));
      const uint32_t bytes = static_cast<uint32_t>(nvalid) * S::kHalves * (kBlockSize * 128);
      const int y = (pb * Hkv + g) * kBlockSize;   // row of the 2-D pool view
      if (!mbar_wait_warp(&bars[kKEmpty + st], ph ^ 1, s_abort)) break;
      if (lane == 0) mbar_arrive_expect_tx(&bars[kKFull + st], bytes);
      __syncwarp();
      if (pb >= 0) {
#pragma unroll
        for (int hf = 0; hf < S::kHalves; ++hf)
          tma_load_2d(smem + S::kOffK + st * S::kKV + hf * (kNK * 128) + lane * (kBlockSize * 128), &tmap_k,
                      hf * 64, y, &bars[kKFull + st]);
      }
      if (!mbar_wait_warp(&bars[kVEmpty + st], ph ^ 1, s_abort)) break;
      if (lane == 0) mbar_arrive_expect_tx(&bars[kVFull + st], bytes);
      __syncwarp();
      if (pb >= 0) {
#pragma unroll
        for (int hf = 0; hf < S::kHalves; ++hf)
          tma_load_2d(smem + S::kOffV + st * S::kKV + hf * (kNK * 128) + lane * (kBlockSize * 128), &tmap_v,
                      hf * 64, y, &bars[kVFull + st]);
      }
    }
    if (j < ntiles) {   // gave up: flag it and let copies already issued land
      if (lane == 0) atomicOr(a.pool.err, PKV_DEVERR_TIMEOUT);
      *s_abort = 1;
      for (int i = max(0, j - kStagesTc); i < j; ++i) {
        (void)mbar_wait(&bars[kKFull + i % kStagesTc], (i / kStagesTc) & 1, nullptr);
        (void)mbar_wait(&bars[kVFull + i % kStagesTc], (i / kStagesTc) & 1, nullptr);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_s = make_idesc_bf16(128, kNK, false);
    constexpr uint32_t idesc_o = make_idesc_bf16(128, D, true);
    bool ok = mbar_wait_warp(&bars[kQFull], 0, s_abort);
    auto issue_s = [&](int j) -> bool {
      const int st = j % kStagesTc;
      if (!mbar_wait_warp(&bars[kKFull + st], (j / kStagesTc) & 1, s_abort)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t d_tmem = tmem + (j & 1) * kNK;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int hf = ks / 4, kk = ks % 4;
          const uint64_t ad = make_sdesc_sw128(sQ + hf * (kTcRows * 128) + kk * 32, 16, 1024);
          const uint64_t bd = make_sdesc_sw128(sK + st * S::kKV + hf * (kNK * 128) + kk * 32, 16, 1024);
          tc_mma(d_tmem, ad, bd, idesc_s, ks > 0 ? 1u : 0u);
        }
        tc_commit(&bars[kSFull + (j & 1)]);
        tc_commit(&bars[kKEmpty + st]);
      }
      __syncwarp();
      return true;
    };
    if (ok && ntiles > 0) ok = issue_s(0);
    for (int j = 0; ok && j < ntiles; ++j) {
      const int st = j % kStagesTc;
      if (j + 1 < ntiles && !issue_s(j + 1)) { ok = false; break; }
      if (!mbar_wait_warp(&bars[kPFull], j & 1, s_abort)) { ok = false; break; }
      if (!mbar_wait_warp(&bars[kVFull + st], (j / kStagesTc) & 1, s_abort)) { ok = false; break; }
      tc_fence_after();
      const int key0 = it.kv_start + j * kNK;
      const int nkeys = min(kNK, kv_end - key0);
      if (nkeys < kNK) {
        // Keys past the item's end: zero their V rows so that 0 * garbage cannot
        // produce NaN in the tensor core (the pool's tail slots are not ours).
        uint8_t* vst = smem + S::kOffV + st * S::kKV;
        for (int idx = lane; idx < (kNK - nkeys) * S::kHalves * 8; idx += 32) {
          const int hf = idx / ((kNK - nkeys) * 8);
          const int rem = idx % ((kNK - nkeys) * 8);
          const int key = nkeys + rem / 8, chunk = rem % 8;
          *reinterpret_cast<uint4*>(vst + hf * (kNK * 128) + key * 128 + chunk * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
#pragma unroll
        for (int ks = 0; ks < kNK / 16; ++ks) {
          const uint64_t ad = make_sdesc_sw128(sP + ks * 32, 16, 1024);
          const uint64_t bd = make_sdesc_sw128(sV + st * S::kKV + ks * (16 * 128), kNK * 128, 1024);
          tc_mma(tmem + kColO, ad, bd, idesc_o, (j > 0 || ks > 0) ? 1u : 0u);
        }
        tc_commit(&bars[kPvDone]);
        tc_commit(&bars[kVEmpty + st]);
      }
      __syncwarp();
    }
    if (!ok) {
      if (lane == 0) atomicOr(a.pool.err, PKV_DEVERR_TIMEOUT);
      *s_abort = 1;
    }
    // Drain: every MMA this thread issued has completed before TMEM is released.
    if (lane == 0) tc_commit(&bars[kDrain]);
    __syncwarp();
    (void)mbar_wait_warp(&bars[kDrain], 0, nullptr);
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    // Q tile: row `row` = (token q_start + row / G, head g*G + row % G), swizzled K-major.
    {
      const uint4* src = nullptr;
      if (row < rows) {
        const int t = it.q_start + row / G;
        const int h = g * G + row % G;
        src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) +
                                             (static_cast<int64_t>(t) * a.num_q_heads + h) * D);
      }
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 v = src ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        const int hf = c / 8, cc = c % 8;
        *reinterpret_cast<uint4*>(smem + hf * (kTcRows * 128) + row * 128 + ((cc ^ (row & 7)) * 16)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars[kQFull]);
    }
    const float sl2 = a.scale_log2;
    float m = -CUDART_INF_F, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int key0 = it.kv_start + j * kNK;
      if (!mbar_wait_warp(&bars[kSFull + (j & 1)], (j >> 1) & 1, s_abort)) { ok = false; break; }
      tc_fence_after();
      float s[kNK];
#pragma unroll
      for (int c = 0; c < kNK; c += 16) tmem_ld16(tmem + lane_base + (j & 1) * kNK + c, s + c);
      tmem_wait_ld();
      if (key0 + kNK - 1 > min_pos || key0 + kNK > kv_end) {
#pragma unroll
        for (int c = 0; c < kNK; ++c) {
          const int key = key0 + c;
          if (key > qpos || key >= kv_end) s[c] = -CUDART_INF_F;
        }
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < kNK; ++c) mx = fmaxf(mx, s[c]);
      // Lazy rescaling: rows keep their reference max m while the tile max stays
      // within 2^kRescaleLog2 of it (P then stays <= 2^kRescaleLog2, fine for bf16
      // and fp32 sums); O and l always share the same reference, so the result
      // is exact.  The decision is per warp because TMEM loads and stores are
      // warp-collective.
      const float m_tile = mx * sl2;
      const bool grow = __any_sync(0xffffffffu, m_tile > m + kRescaleLog2);
      const float m_new = grow ? fmaxf(m, m_tile) : m;
      const float m_use = m_new == -CUDART_INF_F ? 0.f : m_new;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < kNK; ++c) {
        s[c] = fast_exp2(fmaf(s[c], sl2, -m_use));
        rs += s[c];
      }
      const float alpha = grow ? fast_exp2(m - m_use) : 1.f;
      if (j > 0) {
        // PV of the previous tile must be done before P is overwritten and O rescaled.
        if (!mbar_wait_warp(&bars[kPvDone], (j - 1) & 1, s_abort)) { ok = false; break; }
        tc_fence_after();
        if (grow) {
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            float o[32];
            tmem_ld16(tmem + lane_base + kColO + c, o);
            tmem_ld16(tmem + lane_base + kColO + c + 16, o + 16);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tmem_st16(tmem + lane_base + kColO + c, o);
            tmem_st16(tmem + lane_base + kColO + c + 16, o + 16);
          }
          tmem_wait_st();
        }
      }
      l = l * alpha + rs;
      m = m_new;
      // P row (bf16, K-major, 128-byte swizzle).
#pragma unroll
      for (int cc = 0; cc < kNK / 8; ++cc) {
        uint4 v;
        v.x = pack_bf16x2(s[cc * 8 + 0], s[cc * 8 + 1]);
        v.y = pack_bf16x2(s[cc * 8 + 2], s[cc * 8 + 3]);
        v.z = pack_bf16x2(s[cc * 8 + 4], s[cc * 8 + 5]);
        v.w = pack_bf16x2(s[cc * 8 + 6], s[cc * 8 + 7]);
        *reinterpret_cast<uint4*>(smem + S::kOffP + row * 128 + ((cc ^ (row & 7)) * 16)) = v;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars[kPFull]);
    }
    if (ok && ntiles > 0) {
      if (!mbar_wait_warp(&bars[kPvDone], (ntiles - 1) & 1, s_abort)) ok = false;
      tc_fence_after();
    }
    if (!ok) {
      if (lane == 0) atomicOr(a.pool.err, PKV_DEVERR_TIMEOUT);
      *s_abort = 1;
    }
    // Epilogue.  `ok` is uniform across the four warps; the TMEM loads are
    // executed by every thread, only the stores depend on the row being valid.
    if (ok) {
      constexpr float kLn2 = 0.69314718055994530942f;
      const bool valid = row < rows;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse = l > 0.f ? (m + fast_log2(l)) * kLn2 : -CUDART_INF_F;
      const int t = it.q_start + (valid ? row / G : 0);
      const int h = g * G + row % G;
      uint4* dst_o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.o) + (static_cast<int64_t>(t) * a.num_q_heads + h) * D);
      float4* dst_p = it.part >= 0 ? reinterpret_cast<float4*>(a.part_o + static_cast<int64_t>(it.part + row) * D) : nullptr;
#pragma unroll
      for (int c = 0; c < D; c += 16) {
        float o[16];
        if (ntiles > 0) {
          tmem_ld16(tmem + lane_base + kColO + c, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = 0.f;
        }
        if (valid) {
          if (it.part < 0) {
            uint4 w0, w1;
            w0.x = pack_bf16x2(o[0] * inv, o[1] * inv);   w0.y = pack_bf16x2(o[2] * inv, o[3] * inv);
            w0.z = pack_bf16x2(o[4] * inv, o[5] * inv);   w0.w = pack_bf16x2(o[6] * inv, o[7] * inv);
            w1.x = pack_bf16x2(o[8] * inv, o[9] * inv);   w1.y = pack_bf16x2(o[10] * inv, o[11] * inv);
            w1.z = pack_bf16x2(o[12] * inv, o[13] * inv); w1.w = pack_bf16x2(o[14] * inv, o[15] * inv);
            dst_o[c / 8] = w0;
            dst_o[c / 8 + 1] = w1;
          } else {
#pragma unroll
            for (int e = 0; e < 16; e += 4)
              dst_p[(c + e) / 4] = make_float4(o[e] * inv, o[e + 1] * inv, o[e + 2] * inv, o[e + 3] * inv);
          }
        }
      }
      if (valid) {
        if (it.part < 0) {
          if (a.lse) a.lse[static_cast<int64_t>(t) * a.num_q_heads + h] = lse;
        } else {
          a.part_lse[it.part + row] = lse;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

template <int D>
static int launch_tc_d(const AttnArgs& a, const CUtensorMap* tk, const CUtensorMap* tv, const WorkItem* items,
                       int n_items, void* stream) {
  const int smem = TcSmem<D>::kTotal;
  cudaError_t e = cudaFuncSetAttribute(tc_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  tc_attn_kernel<D><<<n_items, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(a, *tk, *tv, items);
  return cudaGetLastError();
}

int launch_tc(const AttnArgs& a, const void* tmap_k, const void* tmap_v, const WorkItem* items, int n_items,
              void* stream) {
  if (n_items <= 0) return cudaSuccess;
  const CUtensorMap* tk = static_cast<const CUtensorMap*>(tmap_k);
  const CUtensorMap* tv = static_cast<const CUtensorMap*>(tmap_v);
  if (a.pool.head_dim == 128) return launch_tc_d<128>(a, tk, tv, items, n_items, stream);
  return launch_tc_d<64>(a, tk, tv, items, n_items, stream);
}

}  // namespace pkv

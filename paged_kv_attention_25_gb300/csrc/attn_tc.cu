// Tensor-core paged attention for tiles of many query rows (new-turn
// prefills, recomputed evicted history, grouped-query decode): the
// "attention between multiple input tokens with a GPU cache spread over
// non-contiguous memory" of "Stateful Large Language Model Serving with
// Pensieve" (abstract), written for sm_103a.
//
// One CTA (one per SM) runs one work item: a query tile of up to 128 rows
// (tokens x grouped heads of one KV head; one row per TMEM lane) against a
// range of key positions in tiles of 128 keys (8 KV blocks).
//
//   warp 8     producer: reads the block table and gathers each block's K and
//              V (16 keys x 64 dims per TMA box, 128-byte swizzle) into a
//              shared-memory ring (cp.async.bulk.tensor, mbarrier tracked);
//   warp 9     MMA issuer (one thread): S(j) = Q K(j)^T (tcgen05.mma kind::f16,
//              M=128, N=128, bf16 in, fp32 accumulate in TMEM, two S buffers)
//              and O += P(j) V(j) with P(j) read from TMEM (two P buffers);
//   warps 0-7  softmax: warps w and w+4 share the 32 rows of TMEM lanes
//              32(w%4)..; the first takes key columns 0-63 of every tile and
//              the first half of O, the second columns 64-127 and the second
//              half.  Row max and sum are combined through shared memory.
//              Causal mask on absolute positions, online softmax in fp32 with
//              exp2 (scale * log2 e folded in; a quarter of the exponentials on
//              the FMA pipe by a polynomial, the rest on the SFU), lazy
//              rescaling of O, P written to TMEM as bf16.
//
// With S and P double-buffered in their own TMEM columns, S(j+1) is computed
// while the softmax works on S(j), and PV(j) runs while it works on S(j+1).
//
// TMEM columns: S0 [0,128)  S1 [128,256)  O [256,256+D)  P0 [384,448)  P1 [448,512).
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "internal.h"
#include "ptx.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 320;
constexpr int kNK = kTcKeys;            // keys per tile (128)
constexpr int kHalfK = kNK / 2;         // key columns per softmax warp
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;
constexpr float kRescaleLog2 = 8.f;     // lazy O rescale threshold (log2 units)

template <int D>
struct TcSmem {
  static constexpr int kHalves = D / 64;                 // 128-byte-wide column slabs
  static constexpr int kStages = D == 128 ? 3 : 4;
  static constexpr int kQ = kTcRows * D * 2;             // query tile: [halves][128 rows][64]
  static constexpr int kKV = kNK * D * 2;                // one stage of K (or V): [halves][128 keys][64]
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kQ;
  static constexpr int kOffV = kOffK + kStages * kKV;
  static constexpr int kOffX = kOffV + kStages * kKV;    // row max / row sum exchange [parity][half][row]
  static constexpr int kOffBar = kOffX + 4 * kTcRows * 4;
  static constexpr int kNumBars = 4 * kStages + 11;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kTotal = kOffMisc + 32;
};

template <int S>
struct Bars {
  static constexpr int kKFull = 0, kKEmpty = S, kVFull = 2 * S, kVEmpty = 3 * S;
  static constexpr int kQ = 4 * S;          // Q tile in shared memory (256 arrivals)
  static constexpr int kS = 4 * S + 1;      // + buffer: S ready in TMEM
  static constexpr int kP = 4 * S + 3;      // + buffer: P written (256 arrivals)
  static constexpr int kPv = 4 * S + 5;     // + buffer: the PV that read P buffer b is done
  static constexpr int kX = 4 * S + 7;      // + tile parity: row maxima exchanged (256 arrivals)
  static constexpr int kSum = 4 * S + 9;    // row sums exchanged (256 arrivals)
  static constexpr int kDrain = 4 * S + 10; // every MMA issued has completed
};

// 2^x on the FMA pipe, for x <= 2^kRescaleLog2: x = n + f with n = floor(x) and
// f in [0,1); 2^f from a cubic fitted to minimise the relative error on [0,1)
// (at most 7.5e-5, far below bf16's 2^-9), then n added to the exponent field.
// Inputs below -126 give 0.
__device__ __forceinline__ float exp2_poly(float x) {
  const float n = floorf(x);
  const float f = x - n;
  float p = fmaf(f, 0.0780244991f, 0.2260672152f);
  p = fmaf(p, f, 0.6958335042f);
  p = fmaf(p, f, 0.9999251962f);
  const int bits = __float_as_int(p) + (static_cast<int>(n) << 23);
  return x < -126.f ? 0.f : __int_as_float(bits);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
tc_attn_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
               const WorkItem* __restrict__ items) {
  using S = TcSmem<D>;
  using B = Bars<S::kStages>;
  constexpr int kSt = S::kStages;
  constexpr int kOHalf = D / 2;             // O columns per softmax warp
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {   // swizzle atoms need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(a.pool.err, PKV_DEVERR_INTERNAL);
    return;
  }
  // Once any wait in this launch has given up, the remaining CTAs do nothing.
  // (__syncthreads_or makes the decision the same for every thread of the CTA.)
  if (__syncthreads_or((*reinterpret_cast<volatile unsigned*>(a.pool.err) & PKV_DEVERR_TIMEOUT) != 0)) return;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  float* xmax = reinterpret_cast<float*>(smem + S::kOffX);          // [tile parity][half][row]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + S::kOffMisc);
  int* s_pos = reinterpret_cast<int*>(smem + S::kOffMisc + 8);      // max, min
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + S::kOffMisc + 16);

  const WorkItem it = items[blockIdx.x];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.group;
  const int g = it.kv_head;
  const int Hkv = a.pool.num_kv_heads;
  const int rows = it.q_count * G;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 4 * kSt; ++i) mbar_init(&bars[i], 1);
    mbar_init(&bars[B::kQ], 256);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[B::kS + b], 1);
      mbar_init(&bars[B::kP + b], 256);
      mbar_init(&bars[B::kPv + b], 1);
      mbar_init(&bars[B::kX + b], 256);
    }
    mbar_init(&bars[B::kSum], 256);
    mbar_init(&bars[B::kDrain], 1);
    s_pos[0] = -1;
    s_pos[1] = 0x7fffffff;
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }
  if (warp == 9) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  const int row = threadIdx.x & 127;        // softmax warps: row of the tile (TMEM lane)
  const int hw = (warp >> 2) & 1;           // softmax warps: which half of the columns
  int qpos = -1;
  if (warp < 8 && row < rows) qpos = __ldg(a.q_positions + it.q_start + row / G);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp < 4 && row < rows) {
    atomicMax(&s_pos[0], qpos);
    atomicMin(&s_pos[1], qpos);
  }
  __syncthreads();
  const uint32_t tmem = *s_tmem;
  const int kv_end = min(it.kv_end, s_pos[0] + 1);
  const int min_pos = s_pos[1];
  const int nt = kv_end > it.kv_start ? (kv_end - it.kv_start + kNK - 1) / kNK : 0;

  const uint32_t sQ = smem_u32(smem + S::kOffQ);
  const uint32_t sK = smem_u32(smem + S::kOffK);
  const uint32_t sV = smem_u32(smem + S::kOffV);

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    const int32_t* bt_row = a.block_tables + static_cast<int64_t>(it.req) * a.max_blocks;
    // Block ids are read a window ahead: lane l holds the id of block
    // (first block of the item) + 32 w + l, i.e. windows of four key tiles, and
    // the next window is already in flight while the current one is used.
    const int blk_first = it.kv_start / kBlockSize;
    const int blk_end = (kv_end + kBlockSize - 1) / kBlockSize;
    auto load_window = [&](int w) -> int {
      const int col = blk_first + w * 32 + lane;
      int pb = -1;
      if (col < blk_end) {
        pb = col < a.max_blocks ? __ldg(bt_row + col) : -1;
        if (pb < 0 || pb >= a.pool.num_blocks) {
          atomicOr(a.pool.err, PKV_DEVERR_BLOCK_ID);
          pb = -1;
        }
      }
      return pb;
    };
    int ids_cur = load_window(0), ids_next = load_window(1), win = 0;
    int j = 0;
    for (; j < nt; ++j) {
      const int st = j % kSt;
      const uint32_t ph = (j / kSt) & 1;
      if ((j >> 2) != win) {
        win = j >> 2;
        ids_cur = ids_next;
        ids_next = load_window(win + 1);
      }
      const int key0 = it.kv_start + j * kNK;
      const int nkeys = min(kNK, kv_end - key0);
      const int nblk = (nkeys + kBlockSize - 1) / kBlockSize;
      int pb = __shfl_sync(0xffffffffu, ids_cur, (j & 3) * 8 + (lane & 7));
      if (lane >= nblk) pb = -1;
      const int nvalid = __popc(__ballot_sync(0xffffffffu, pb >= 0));
      const uint32_t bytes = static_cast<uint32_t>(nvalid) * S::kHalves * (kBlockSize * 128);
      const int y = (pb * Hkv + g) * kBlockSize;   // row of the 2-D pool view
      if (!mbar_wait_warp(&bars[B::kKEmpty + st], ph ^ 1, s_abort)) break;
      if (lane == 0) mbar_arrive_expect_tx(&bars[B::kKFull + st], bytes);
      __syncwarp();
      if (pb >= 0) {
#pragma unroll
        for (int hf = 0; hf < S::kHalves; ++hf)
          tma_load_2d(smem + S::kOffK + st * S::kKV + hf * (kNK * 128) + lane * (kBlockSize * 128), &tmap_k,
                      hf * 64, y, &bars[B::kKFull + st]);
      }
      if (!mbar_wait_warp(&bars[B::kVEmpty + st], ph ^ 1, s_abort)) break;
      if (lane == 0) mbar_arrive_expect_tx(&bars[B::kVFull + st], bytes);
      __syncwarp();
      if (pb >= 0) {
#pragma unroll
        for (int hf = 0; hf < S::kHalves; ++hf)
          tma_load_2d(smem + S::kOffV + st * S::kKV + hf * (kNK * 128) + lane * (kBlockSize * 128), &tmap_v,
                      hf * 64, y, &bars[B::kVFull + st]);
      }
    }
    if (j < nt) {   // gave up: flag it and let copies already issued land
      if (lane == 0) atomicOr(a.pool.err, PKV_DEVERR_TIMEOUT);
      *s_abort = 1;
      for (int i = max(0, j - kSt); i < j; ++i) {
        (void)mbar_wait(&bars[B::kKFull + i % kSt], (i / kSt) & 1, nullptr);
        (void)mbar_wait(&bars[B::kVFull + i % kSt], (i / kSt) & 1, nullptr);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_s = make_idesc_bf16(128, kNK, false);
    constexpr uint32_t idesc_o = make_idesc_bf16(128, D, true);
    bool ok = mbar_wait_warp(&bars[B::kQ], 0, s_abort);
    // S(j) into S buffer j%2.  The softmax finished reading S(j-2) from that
    // buffer before it signalled P(j-2), which the issuer has waited for.
    auto issue_s = [&](int j) -> bool {
      const int st = j % kSt;
      if (!mbar_wait_warp(&bars[B::kKFull + st], (j / kSt) & 1, s_abort)) return false;
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int hf = ks / 4, kk = ks % 4;
          const uint64_t ad = make_sdesc_sw128(sQ + hf * (kTcRows * 128) + kk * 32, 16, 1024);
          const uint64_t bd = make_sdesc_sw128(sK + st * S::kKV + hf * (kNK * 128) + kk * 32, 16, 1024);
          tc_mma(tmem + kColS + (j & 1) * kNK, ad, bd, idesc_s, ks > 0 ? 1u : 0u);
        }
        tc_commit(&bars[B::kS + (j & 1)]);
        tc_commit(&bars[B::kKEmpty + st]);
      }
      __syncwarp();
      return true;
    };
    if (ok && nt > 0) ok = issue_s(0);
    if (ok && nt > 1) ok = issue_s(1);
    for (int j = 0; ok && j < nt; ++j) {
      const int st = j % kSt;
      if (!(ok = mbar_wait_warp(&bars[B::kP + (j & 1)], (j >> 1) & 1, s_abort))) break;
      if (!(ok = mbar_wait_warp(&bars[B::kVFull + st], (j / kSt) & 1, s_abort))) break;
      tc_fence_after();
      const int nkeys = min(kNK, kv_end - (it.kv_start + j * kNK));
      if (nkeys < kNK) {
        // Keys past the item's end: zero their V rows so that 0 * garbage
        // cannot produce NaN in the tensor core.
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
          const uint64_t bd = make_sdesc_sw128(sV + st * S::kKV + ks * (16 * 128), kNK * 128, 1024);
          tc_mma_ts(tmem + kColO, tmem + kColP + (j & 1) * (kNK / 2) + ks * 8, bd, idesc_o,
                    (j > 0 || ks > 0) ? 1u : 0u);
        }
        tc_commit(&bars[B::kPv + (j & 1)]);
        tc_commit(&bars[B::kVEmpty + st]);
      }
      __syncwarp();
      if (j + 2 < nt && !(ok = issue_s(j + 2))) break;
    }
    if (!ok) {
      if (lane == 0) atomicOr(a.pool.err, PKV_DEVERR_TIMEOUT);
      *s_abort = 1;
    }
    // Drain: every MMA this thread issued has completed before TMEM is released.
    if (lane == 0) tc_commit(&bars[B::kDrain]);
    __syncwarp();
    (void)mbar_wait_warp(&bars[B::kDrain], 0, nullptr);
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax / epilogue
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    // Q tile: this thread stores half of row `row`.
    {
      const uint4* src = nullptr;
      if (row < rows) {
        const int t = it.q_start + row / G;
        const int h = g * G + row % G;
        src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) +
                                             (static_cast<int64_t>(t) * a.num_q_heads + h) * D);
      }
#pragma unroll
      for (int cc = 0; cc < D / 16; ++cc) {
        const int c = hw * (D / 16) + cc;     // 16-byte chunk of the row
        const uint4 v = src ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        const int hf = c / 8, ch = c % 8;
        *reinterpret_cast<uint4*>(smem + S::kOffQ + hf * (kTcRows * 128) + row * 128 + ((ch ^ (row & 7)) * 16)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars[B::kQ]);
    }
    const float sl2 = a.scale_log2;
    float m = -CUDART_INF_F, l = 0.f;       // l: this thread's half of the row sum
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int key0 = it.kv_start + j * kNK + hw * kHalfK;
      if (!mbar_wait_warp(&bars[B::kS + (j & 1)], (j >> 1) & 1, s_abort)) { ok = false; break; }
      tc_fence_after();
      float s[kHalfK];
#pragma unroll
      for (int c = 0; c < kHalfK; c += 16)
        tmem_ld16(tmem + lane_base + kColS + (j & 1) * kNK + hw * kHalfK + c, s + c);
      tmem_wait_ld();
      if (key0 + kHalfK - 1 > min_pos || key0 + kHalfK > kv_end) {
#pragma unroll
        for (int c = 0; c < kHalfK; ++c) {
          const int key = key0 + c;
          if (key > qpos || key >= kv_end) s[c] = -CUDART_INF_F;
        }
      }
      // Row max: 8 independent partials, then combined with the other half.
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = s[k];
#pragma unroll
      for (int c = 8; c < kHalfK; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], s[c]);
      float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      float* xm = xmax + (j & 1) * 2 * kTcRows;
      xm[hw * kTcRows + row] = mx;
      mbar_arrive(&bars[B::kX + (j & 1)]);
      if (!mbar_wait_warp(&bars[B::kX + (j & 1)], (j >> 1) & 1, s_abort)) { ok = false; break; }
      mx = fmaxf(mx, xm[(hw ^ 1) * kTcRows + row]);
      // Lazy rescaling: rows keep their reference max m while the tile max stays
      // within 2^kRescaleLog2 of it (P then stays <= 2^kRescaleLog2, fine for bf16
      // and fp32 sums); O and l always share the same reference, so the result
      // is exact.  Both warps of a row see the same values, so they take the
      // same (warp-uniform) decision.
      const float m_tile = mx * sl2;
      const bool grow = __any_sync(0xffffffffu, m_tile > m + kRescaleLog2);
      const float m_new = grow ? fmaxf(m, m_tile) : m;
      const float m_use = m_new == -CUDART_INF_F ? 0.f : m_new;
      float rs8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      uint32_t pk[kHalfK / 2];
#pragma unroll
      for (int c = 0; c < kHalfK; c += 2) {
        const float x0 = fmaf(s[c], sl2, -m_use);
        const float x1 = fmaf(s[c + 1], sl2, -m_use);
        // A quarter of the exponentials on the FMA pipe, the rest on the SFU.
        const float p0 = fast_exp2(x0);
        const float p1 = (c & 2) ? exp2_poly(x1) : fast_exp2(x1);
        rs8[(c >> 1) & 7] += p0 + p1;
        pk[c / 2] = pack_bf16x2(p0, p1);
      }
      const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
      const float alpha = grow ? fast_exp2(m - m_use) : 1.f;
      // P buffer j%2 was last read by PV(j-2).
      if (j >= 2 && !mbar_wait_warp(&bars[B::kPv + (j & 1)], ((j >> 1) - 1) & 1, s_abort)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < kHalfK / 2; c += 16)
        tmem_st16(tmem + lane_base + kColP + (j & 1) * (kNK / 2) + hw * (kHalfK / 2) + c,
                  reinterpret_cast<const float*>(pk + c));
      if (grow && j > 0) {
        // O is accumulated by PV(j-1); rescale this half once it has completed.
        if (!mbar_wait_warp(&bars[B::kPv + ((j - 1) & 1)], ((j - 1) >> 1) & 1, s_abort)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kOHalf; c += 32) {
          float o[32];
          tmem_ld16(tmem + lane_base + kColO + hw * kOHalf + c, o);
          tmem_ld16(tmem + lane_base + kColO + hw * kOHalf + c + 16, o + 16);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_st16(tmem + lane_base + kColO + hw * kOHalf + c, o);
          tmem_st16(tmem + lane_base + kColO + hw * kOHalf + c + 16, o + 16);
        }
      }
      l = l * alpha + rs;
      m = m_new;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars[B::kP + (j & 1)]);
    }
    if (ok && nt > 0) {
      if (!mbar_wait_warp(&bars[B::kPv + ((nt - 1) & 1)], ((nt - 1) >> 1) & 1, s_abort)) ok = false;
      tc_fence_after();
    }
    // Row sum of the two halves, exchanged in the max slots of the tile parity
    // that no thread reads any more (the last tile used parity (nt-1)&1).
    float* xsum = xmax + (nt & 1) * 2 * kTcRows;
    xsum[hw * kTcRows + row] = l;
    mbar_arrive(&bars[B::kSum]);
    if (!mbar_wait_warp(&bars[B::kSum], 0, s_abort)) ok = false;
    l += xsum[(hw ^ 1) * kTcRows + row];
    // A wait that ran out anywhere sets the abort flag, so the two warps of a
    // row agree on skipping the epilogue.
    ok = __all_sync(0xffffffffu, ok && !*s_abort);
    if (!ok) {
      if (lane == 0) atomicOr(a.pool.err, PKV_DEVERR_TIMEOUT);
      *s_abort = 1;
    }
    // Epilogue: this thread writes dims [hw*D/2, hw*D/2 + D/2) of its row.  The
    // TMEM loads are executed by every thread of the warp; only the stores
    // depend on the row being valid.
    if (ok) {
      constexpr float kLn2 = 0.69314718055994530942f;
      const bool valid = row < rows;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse = l > 0.f ? (m + fast_log2(l)) * kLn2 : -CUDART_INF_F;
      const int t = it.q_start + (valid ? row / G : 0);
      const int h = g * G + row % G;
      uint4* dst_o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.o) +
                                              (static_cast<int64_t>(t) * a.num_q_heads + h) * D + hw * kOHalf);
      float4* dst_p = it.part >= 0
                          ? reinterpret_cast<float4*>(a.part_o + static_cast<int64_t>(it.part + row) * D + hw * kOHalf)
                          : nullptr;
#pragma unroll
      for (int c = 0; c < kOHalf; c += 16) {
        float o[16];
        if (nt > 0) {
          tmem_ld16(tmem + lane_base + kColO + hw * kOHalf + c, o);
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
      if (valid && hw == 0) {
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
  if (warp == 9) {
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

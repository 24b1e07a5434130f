// Tensor-core paged attention for tiles of many query rows (new-turn
// prefills, recomputed evicted history, grouped-query decode): the
// "attention between multiple input tokens with a GPU cache spread over
// non-contiguous memory" of "Stateful Large Language Model Serving with
// Pensieve" (abstract), written for sm_103a.
//
// One CTA (one per SM) runs one work item: two query tiles A and B of up to
// 128 rows each (tokens x grouped heads of one KV head; one row per TMEM
// lane) of the same request, against a range of key positions in tiles of 64
// keys (4 KV blocks).  Each K/V tile is brought into shared memory once and
// used by both query tiles: an SM can take in only a few tens of bytes per
// clock from the memory system, so query rows per byte loaded is what bounds
// this kernel.
//
//   warp 8     producer: reads the block table a window ahead and gathers each
//              block's K and V (16 keys x 64 dims per TMA box, 128-byte
//              swizzle) into a shared-memory ring (cp.async.bulk.tensor);
//   warps 9,10 MMA issuers, one per query tile (a tcgen05.mma costs its
//              issuing thread about a hundred cycles, and two issuing threads
//              overlap): S_t = Q_t K^T (kind::f16, M=128, N=64, bf16 in, fp32
//              accumulate in TMEM) and O_t += P_t V with P_t read from TMEM;
//   warps 0-3  softmax of tile A, warps 4-7 softmax of tile B: one query row
//              per thread.  Each thread loads its S row into registers and at
//              once releases the S columns (so the next S MMA overlaps the rest
//              of the softmax), applies the causal mask on absolute positions,
//              runs the online softmax in fp32 (exp2 with scale*log2 e folded
//              in; a quarter of the exponentials on the FMA pipe by a cubic,
//              the rest on the SFU; lazy rescaling of O) and writes P as bf16
//              into its own TMEM columns; epilogue O / l.
//
// TMEM columns: S_A [0,64)  S_B [64,128)  P_A [128,160)  P_B [160,192)
//               O_A [256, 256+D)  O_B [384, 384+D).
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "internal.h"
#include "ptx.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 352;
constexpr int kNK = kTcKeys;            // keys per tile (64)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColP = 128, kColO = 256;
constexpr float kRescaleLog2 = 8.f;     // lazy O rescale threshold (log2 units)

template <int D>
struct TcSmem {
  static constexpr int kHalves = D / 64;                 // 128-byte-wide column slabs
  static constexpr int kStages = D == 128 ? 4 : 6;
  static constexpr int kQ = kTcRows * D * 2;             // one query tile: [halves][128 rows][64]
  static constexpr int kKV = kNK * D * 2;                // one stage of K (or V): [halves][64 keys][64]
  static constexpr int kOffQ = 0;                        // tile A, then tile B
  static constexpr int kOffK = 2 * kQ;
  static constexpr int kOffV = kOffK + kStages * kKV;
  static constexpr int kOffBar = kOffV + kStages * kKV;
  static constexpr int kNumBars = 4 * kStages + 13;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kTotal = kOffMisc + 64;
};

template <int S>
struct Bars {
  static constexpr int kKFull = 0, kKEmpty = S, kVFull = 2 * S, kVEmpty = 3 * S;
  static constexpr int kQ = 4 * S;          // + tile: Q in shared memory (128 arrivals)
  static constexpr int kS = 4 * S + 2;      // + tile: S ready in TMEM
  static constexpr int kSFree = 4 * S + 4;  // + tile: S read into registers (128 arrivals)
  static constexpr int kP = 4 * S + 6;      // + tile: P written (128 arrivals)
  static constexpr int kPv = 4 * S + 8;     // + tile: PV done
  static constexpr int kDrain = 4 * S + 10; // + issuer: every MMA it issued has completed
  static constexpr int kTail = 4 * S + 12;  // V rows past the item's end zeroed (issuer A -> B)
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
  int* s_pos = reinterpret_cast<int*>(smem + S::kOffMisc + 16);   // max A, min A, max B, min B
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + S::kOffMisc + 32);

  const WorkItem it = items[blockIdx.x];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.group;
  const int g = it.kv_head;
  const int Hkv = a.pool.num_kv_heads;
  const int rows[2] = {it.q_count * G, it.q_count2 * G};
  const int tok0[2] = {it.q_start, it.q_start + it.q_count};

  if (threadIdx.x == 0) {
    for (int i = 0; i < 4 * kSt; ++i) mbar_init(&bars[i], (i >= kSt && i < 2 * kSt) || i >= 3 * kSt ? 2 : 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars[B::kQ + t], 128);
      mbar_init(&bars[B::kS + t], 1);
      mbar_init(&bars[B::kSFree + t], 128);
      mbar_init(&bars[B::kP + t], 128);
      mbar_init(&bars[B::kPv + t], 1);
    }
    mbar_init(&bars[B::kDrain], 1);
    mbar_init(&bars[B::kDrain + 1], 1);
    mbar_init(&bars[B::kTail], 1);
    s_pos[0] = -1;
    s_pos[1] = 0x7fffffff;
    s_pos[2] = -1;
    s_pos[3] = 0x7fffffff;
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
  const int X = (warp >> 2) & 1;            // query tile of a softmax warp (0 = A, 1 = B)
  const int row = threadIdx.x & 127;        // its row within the tile (TMEM lane)
  int qpos = -1;
  if (warp < 8 && row < rows[X]) qpos = __ldg(a.q_positions + tok0[X] + row / G);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp < 8 && row < rows[X]) {
    atomicMax(&s_pos[2 * X], qpos);
    atomicMin(&s_pos[2 * X + 1], qpos);
  }
  __syncthreads();
  const uint32_t tmem = *s_tmem;
  int ntile[2], min_pos[2];
  int kv_end = it.kv_start;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int e = min(it.kv_end, s_pos[2 * t] + 1);          // keys tile t can see
    ntile[t] = e > it.kv_start ? (e - it.kv_start + kNK - 1) / kNK : 0;
    min_pos[t] = s_pos[2 * t + 1];
    kv_end = max(kv_end, e);
  }
  const int ntiles = max(ntile[0], ntile[1]);

  const uint32_t sQ = smem_u32(smem + S::kOffQ);
  const uint32_t sK = smem_u32(smem + S::kOffK);
  const uint32_t sV = smem_u32(smem + S::kOffV);

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    const int32_t* bt_row = a.block_tables + static_cast<int64_t>(it.req) * a.max_blocks;
    constexpr int kBlk = kNK / kBlockSize;   // blocks per key tile (4)
    constexpr int kWin = 32 / kBlk;          // key tiles per window of 32 block ids
    // Block ids are read a window ahead: lane l holds the id of block
    // (first block of the item) + 32 w + l, and the next window is in flight
    // while the current one is used.
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
    for (; j < ntiles; ++j) {
      const int st = j % kSt;
      const uint32_t ph = (j / kSt) & 1;
      if (j / kWin != win) {
        win = j / kWin;
        ids_cur = ids_next;
        ids_next = load_window(win + 1);
      }
      const int key0 = it.kv_start + j * kNK;
      const int nkeys = min(kNK, kv_end - key0);
      const int nblk = (nkeys + kBlockSize - 1) / kBlockSize;
      int pb = __shfl_sync(0xffffffffu, ids_cur, (j % kWin) * kBlk + (lane % kBlk));
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
    if (j < ntiles) {   // gave up: flag it and let copies already issued land
      if (lane == 0) atomicOr(a.pool.err, PKV_DEVERR_TIMEOUT);
      *s_abort = 1;
      for (int i = max(0, j - kSt); i < j; ++i) {
        (void)mbar_wait(&bars[B::kKFull + i % kSt], (i / kSt) & 1, nullptr);
        (void)mbar_wait(&bars[B::kVFull + i % kSt], (i / kSt) & 1, nullptr);
      }
    }
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------ MMA issuer of query tile t
    const int t = warp - 9;
    const int nt_t = ntile[t];
    constexpr uint32_t idesc_s = make_idesc_bf16(128, kNK, false);
    constexpr uint32_t idesc_o = make_idesc_bf16(128, D, true);
    // Descriptors are built once; each MMA only advances the start-address
    // field (bits 0-13, in 16-byte units) by a constant offset.
    const uint64_t dq = make_sdesc_sw128(sQ + t * S::kQ, 16, 1024);
    const uint64_t dk = make_sdesc_sw128(sK, 16, 1024);
    const uint64_t dv = make_sdesc_sw128(sV, kNK * 128, 1024);
    const uint32_t d_s = tmem + kColS + t * kNK, d_o = tmem + kColO + t * 128, a_p = tmem + kColP + t * (kNK / 2);
    bool ok = mbar_wait_warp(&bars[B::kQ + t], 0, s_abort);
    // S_t(j) = Q_t K(j)^T into this tile's S columns; the softmax has read
    // S_t(j-1) into registers once it released them.
    auto issue_s = [&](int j) -> bool {
      const int st = j % kSt;
      if (!mbar_wait_warp(&bars[B::kKFull + st], (j / kSt) & 1, s_abort)) return false;
      if (j > 0 && !mbar_wait_warp(&bars[B::kSFree + t], (j - 1) & 1, s_abort)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint64_t kst = dk + static_cast<uint64_t>((st * S::kKV) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int hf = ks / 4, kk = ks % 4;
          tc_mma(d_s, dq + static_cast<uint64_t>((hf * (kTcRows * 128) + kk * 32) >> 4),
                 kst + static_cast<uint64_t>((hf * (kNK * 128) + kk * 32) >> 4), idesc_s, ks > 0 ? 1u : 0u);
        }
        tc_commit(&bars[B::kS + t]);
      }
      __syncwarp();
      return true;
    };
    // O_t += P_t(j) V(j).
    auto issue_pv = [&](int j, bool wait_tail) -> bool {
      const int st = j % kSt;
      if (!mbar_wait_warp(&bars[B::kP + t], j & 1, s_abort)) return false;
      if (!mbar_wait_warp(&bars[B::kVFull + st], (j / kSt) & 1, s_abort)) return false;
      if (wait_tail && !mbar_wait_warp(&bars[B::kTail], 0, s_abort)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint64_t vst = dv + static_cast<uint64_t>((st * S::kKV) >> 4);
#pragma unroll
        for (int ks = 0; ks < kNK / 16; ++ks)
          tc_mma_ts(d_o, a_p + ks * 8, vst + static_cast<uint64_t>((ks * (16 * 128)) >> 4), idesc_o,
                    (j > 0 || ks > 0) ? 1u : 0u);
        tc_commit(&bars[B::kPv + t]);
      }
      __syncwarp();
      return true;
    };
    // Keys past the item's end in its last tile: issuer A zeroes their V rows
    // (so that 0 * garbage cannot produce NaN in the tensor core) before either
    // tile's PV of that tile; issuer B waits for it.
    const int last_nkeys = ntiles > 0 ? min(kNK, kv_end - (it.kv_start + (ntiles - 1) * kNK)) : kNK;
    auto zero_v_tail = [&](int j) -> bool {
      const int st = j % kSt;
      if (!mbar_wait_warp(&bars[B::kVFull + st], (j / kSt) & 1, s_abort)) return false;
      uint8_t* vst = smem + S::kOffV + st * S::kKV;
      const int nkeys = last_nkeys;
      for (int idx = lane; idx < (kNK - nkeys) * S::kHalves * 8; idx += 32) {
        const int hf = idx / ((kNK - nkeys) * 8);
        const int rem = idx % ((kNK - nkeys) * 8);
        const int key = nkeys + rem / 8, chunk = rem % 8;
        *reinterpret_cast<uint4*>(vst + hf * (kNK * 128) + key * 128 + chunk * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B::kTail]);
      return true;
    };
    // Every issuer releases every K/V stage once per tile (the empty barriers
    // count two), and only after it has seen that tile land in the stage: an
    // mbarrier does not keep phases apart, so a release for a later use of a
    // stage must never arrive before the current use is complete.  An issuer
    // with no work for a tile therefore still waits for the tile's full phase.
    auto release_k = [&](int j, bool issued) -> bool {
      if (!issued && !mbar_wait_warp(&bars[B::kKFull + j % kSt], (j / kSt) & 1, s_abort)) return false;
      if (lane == 0) tc_commit(&bars[B::kKEmpty + j % kSt]);
      __syncwarp();
      return true;
    };
    auto release_v = [&](int j, bool issued) -> bool {
      if (!issued && !mbar_wait_warp(&bars[B::kVFull + j % kSt], (j / kSt) & 1, s_abort)) return false;
      if (lane == 0) tc_commit(&bars[B::kVEmpty + j % kSt]);
      __syncwarp();
      return true;
    };
    if (ok && nt_t > 0) ok = issue_s(0);
    if (ok && ntiles > 0) ok = release_k(0, nt_t > 0);
    for (int j = 0; ok && j < ntiles; ++j) {
      if (j + 1 < nt_t && !(ok = issue_s(j + 1))) break;
      if (j + 1 < ntiles && !(ok = release_k(j + 1, j + 1 < nt_t))) break;
      const bool last_partial = j == ntiles - 1 && last_nkeys < kNK;
      if (t == 0 && last_partial && !(ok = zero_v_tail(j))) break;
      if (j < nt_t && !(ok = issue_pv(j, t == 1 && last_partial))) break;
      if (!(ok = release_v(j, j < nt_t || (t == 0 && last_partial)))) break;
    }
    if (!ok) {
      if (lane == 0) atomicOr(a.pool.err, PKV_DEVERR_TIMEOUT);
      *s_abort = 1;
    }
    // Drain: every MMA this thread issued has completed before TMEM is released.
    if (lane == 0) tc_commit(&bars[B::kDrain + t]);
    __syncwarp();
    (void)mbar_wait_warp(&bars[B::kDrain + t], 0, nullptr);
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax / epilogue of tile X
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t colS = kColS + X * kNK, colP = kColP + X * (kNK / 2), colO = kColO + X * 128;
    const int nrows = rows[X];
    const int nt = ntile[X];
    // Q tile: row `row` = (token tok0[X] + row / G, head g*G + row % G), swizzled K-major.
    {
      const uint4* src = nullptr;
      if (row < nrows) {
        const int t = tok0[X] + row / G;
        const int h = g * G + row % G;
        src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) +
                                             (static_cast<int64_t>(t) * a.num_q_heads + h) * D);
      }
      uint8_t* qt = smem + S::kOffQ + X * S::kQ;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 v = src ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        const int hf = c / 8, cc = c % 8;
        *reinterpret_cast<uint4*>(qt + hf * (kTcRows * 128) + row * 128 + ((cc ^ (row & 7)) * 16)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars[B::kQ + X]);
    }
    const float sl2 = a.scale_log2;
    float m = -CUDART_INF_F, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int key0 = it.kv_start + j * kNK;
      if (!mbar_wait_warp(&bars[B::kS + X], j & 1, s_abort)) { ok = false; break; }
      tc_fence_after();
      float s[kNK];
#pragma unroll
      for (int c = 0; c < kNK; c += 16) tmem_ld16(tmem + lane_base + colS + c, s + c);
      tmem_wait_ld();
      // S is in registers: its TMEM columns may take the next S right away.
      tc_fence_before();
      mbar_arrive(&bars[B::kSFree + X]);
      if (key0 + kNK - 1 > min_pos[X] || key0 + kNK > kv_end) {
#pragma unroll
        for (int c = 0; c < kNK; ++c) {
          const int key = key0 + c;
          if (key > qpos || key >= kv_end) s[c] = -CUDART_INF_F;
        }
      }
      // Row max and sum as 8 independent partials (one long dependency chain
      // would leave the softmax warps latency-bound).
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = s[k];
#pragma unroll
      for (int c = 8; c < kNK; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], s[c]);
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      // Lazy rescaling: rows keep their reference max m while the tile max stays
      // within 2^kRescaleLog2 of it (P then stays <= 2^kRescaleLog2, fine for bf16
      // and fp32 sums); O and l always share the same reference, so the result
      // is exact.  The decision is per warp because TMEM loads and stores are
      // warp-collective.
      const float m_tile = mx * sl2;
      const bool grow = __any_sync(0xffffffffu, m_tile > m + kRescaleLog2);
      const float m_new = grow ? fmaxf(m, m_tile) : m;
      const float m_use = m_new == -CUDART_INF_F ? 0.f : m_new;
      float rs8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      uint32_t pk[kNK / 2];
#pragma unroll
      for (int c = 0; c < kNK; c += 2) {
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
      // PV(j-1) read the P columns and accumulated O: wait for it before
      // writing P(j) and rescaling O.
      if (j > 0) {
        if (!mbar_wait_warp(&bars[B::kPv + X], (j - 1) & 1, s_abort)) { ok = false; break; }
        tc_fence_after();
      }
#pragma unroll
      for (int c = 0; c < kNK / 2; c += 16) tmem_st16(tmem + lane_base + colP + c, reinterpret_cast<const float*>(pk + c));
      if (grow && j > 0) {
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          float o[32];
          tmem_ld16(tmem + lane_base + colO + c, o);
          tmem_ld16(tmem + lane_base + colO + c + 16, o + 16);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_st16(tmem + lane_base + colO + c, o);
          tmem_st16(tmem + lane_base + colO + c + 16, o + 16);
        }
      }
      l = l * alpha + rs;
      m = m_new;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars[B::kP + X]);
    }
    if (ok && nt > 0) {
      if (!mbar_wait_warp(&bars[B::kPv + X], (nt - 1) & 1, s_abort)) ok = false;
      tc_fence_after();
    }
    if (!ok) {
      if (lane == 0) atomicOr(a.pool.err, PKV_DEVERR_TIMEOUT);
      *s_abort = 1;
    }
    // Epilogue.  `ok` is uniform within a warp; the TMEM loads are executed by
    // every thread of the warp, only the stores depend on the row being valid.
    if (ok) {
      constexpr float kLn2 = 0.69314718055994530942f;
      const bool valid = row < nrows;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse = l > 0.f ? (m + fast_log2(l)) * kLn2 : -CUDART_INF_F;
      const int t = tok0[X] + (valid ? row / G : 0);
      const int h = g * G + row % G;
      const int prow = it.part + (X == 0 ? row : rows[0] + row);
      uint4* dst_o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.o) + (static_cast<int64_t>(t) * a.num_q_heads + h) * D);
      float4* dst_p = it.part >= 0 ? reinterpret_cast<float4*>(a.part_o + static_cast<int64_t>(prow) * D) : nullptr;
#pragma unroll
      for (int c = 0; c < D; c += 16) {
        float o[16];
        if (nt > 0) {
          tmem_ld16(tmem + lane_base + colO + c, o);
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
          a.part_lse[prow] = lse;
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

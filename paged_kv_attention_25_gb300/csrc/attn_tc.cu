// Tensor-core paged attention for tiles of many query rows (new-turn
// prefills, recomputed evicted history, grouped-query decode): the
// "attention between multiple input tokens with a GPU cache spread over
// non-contiguous memory" of "Stateful Large Language Model Serving with
// Pensieve" (abstract), written for sm_103a.
//
// One CTA (one per SM) runs one work item: two query tiles A and B of up to
// 128 rows each (tokens x grouped heads of one KV head; one row per TMEM
// lane) of the same request, against a range of key positions in tiles of
// 128 keys (8 KV blocks).  Each K/V tile is brought into shared memory once
// and used by both query tiles: an SM takes in only a few tens of bytes per
// clock from the memory system, so query rows per byte loaded bound this
// kernel next to the tensor cores.
//
//   warps 8,10 producers of K and of V: read the block table a window ahead
//              and gather each block's K (warp 8) or V (warp 10) into
//              shared-memory rings (cp.async.bulk.tensor, one 16 x D box per
//              block, 128-byte swizzle), 2 K and 3 V stages; separate warps
//              so that neither stream waits behind the other's free stages;
//   warp 9     MMA issuer: S_t = Q_t K^T (kind::f16, M=128, N=128 keys, bf16
//              in, fp32 in TMEM) and O_t += P_t V with P_t read from TMEM, in
//              the order PV_A(j) S_A(j+1) PV_B(j) S_B(j+1): tile B's softmax
//              runs while the tensor pipe works on tile A and the other way
//              round.  P_t(j) is written over S_t(j); S_t(j+1) may follow
//              PV_t(j) at once because MMAs issued by one thread run in order;
//   warps 0-3  softmax of tile A, warps 4-7 softmax of tile B: one query row
//              per thread.  Each thread loads its 128 S values, applies the
//              causal mask on absolute positions, runs the online softmax in
//              fp32 (exp2 with scale*log2 e folded in, on the SFU; paired fp32
//              FMA/add; lazy rescaling of O) and writes P as bf16 over S;
//              epilogue O / l.
//
// TMEM columns: S_A/P_A [0,128)  S_B/P_B [128,256)  O_A [256,384)  O_B [384,512).
#include <cuda.h>
#include <climits>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <cuda_fp8.h>

#include "append.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 352;
constexpr int kNK = kTcKeys;            // keys per tile (128)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr float kRescaleLog2 = 8.f;     // lazy O rescale threshold (log2 units)

template <int D>
struct TcSmem {
  static constexpr int kHalves = D / 64;                 // 128-byte-wide column slabs
  static constexpr int kKSt = D == 128 ? 2 : 4;          // K stages
  static constexpr int kVSt = D == 128 ? 3 : 4;          // V stages (the PV copies bound the pair period)
  static constexpr int kQ = kTcRows * D * 2;             // one query tile: [halves][128 rows][64]
  // One stage of K (or V), 128 keys: [8-key group][half][8 keys][64 columns],
  // each [8][64] piece a 1024-byte swizzle atom; one TMA box fills the two
  // groups of a block.  kGS: bytes between 8-key groups; kHS: between halves.
  static constexpr int kKV = kNK * D * 2;
  static constexpr int kGS = kHalves * 1024;
  static constexpr int kHS = 1024;
  static constexpr int kBlkBytes = 2 * kGS;              // one block (16 keys) of a stage
  static constexpr int kOffQ = 0;                        // tile A, then tile B
  static constexpr int kOffK = 2 * kQ;
  static constexpr int kOffV = kOffK + kKSt * kKV;
  static constexpr int kOffBar = kOffV + kVSt * kKV;
  static constexpr int kNumBars = 3 * kKSt + 3 * kVSt + 17;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kTotal = kOffMisc + 64;
};
static_assert(TcSmem<128>::kTotal <= 232448, "shared memory of the D=128 kernel");

template <int KS, int VS>
struct Bars {
  // The kernel is persistent: one CTA per SM takes work items one after
  // another, so every barrier below is reused across items and its phases are
  // counted by running counters, never by an item's own tile index.
  static constexpr int kKFull = 0, kKEmpty = KS, kKLanded = 2 * KS;
  static constexpr int kVFull = 3 * KS, kVEmpty = 3 * KS + VS, kVLanded = 3 * KS + 2 * VS;
  static constexpr int kT = 3 * KS + 3 * VS;
  static constexpr int kS = kT;            // + tile: S_t of the tile's current key tile in TMEM
  static constexpr int kP = kT + 2;        // + tile: P written, O rescaled (128 arrivals)
  static constexpr int kPv = kT + 4;       // + tile: the tile's last PV of the item done
  static constexpr int kQFull = kT + 6;    // + tile: the item's query tile in shared memory (TMA)
  static constexpr int kQEmpty = kT + 8;   // + tile: the item's last S MMA of the tile done (Q reusable)
  static constexpr int kQc = kT + 10;      // + tile: FP8 pools: the tile's Q rows converted to f16 (128 arrivals)
  static constexpr int kItemFull = kT + 12;    // + slot: next item index written
  static constexpr int kItemEmpty = kT + 14;   // + slot: every role has read it
  static constexpr int kDrain = kT + 16;       // every MMA issued has completed
  static constexpr int kCount = kT + 17;
  // Roles that read each item index from the ring: the V producer, the MMA
  // issuer and the eight softmax warps (one arrival per warp).
  static constexpr int kItemReaders = 10;
};

// Per-item values every role derives from the work item (scalars, not arrays
// indexed by tile: those would live in local memory).
struct TcItem {
  WorkItem it;
  int rows0, rows1;       // query rows of tile A / B (tokens x grouped heads)
  int tok00, tok01;       // first token of tile A / B
  int ntile0, ntile1;     // key tiles each query tile sees
  int ntiles, kv_end;     // key tiles of the item and its key range end
};

__device__ __forceinline__ TcItem tc_item(const WorkItem* items, int w, int G) {
  TcItem v;
  v.it = items[w];
  const WorkItem& it = v.it;
  v.rows0 = it.q_count * G;
  v.rows1 = it.q_count2 * G;
  v.tok00 = it.q_start;
  v.tok01 = it.q_start + it.q_count;
  // Key range of each tile from the planner's position bounds, so that the
  // block-table reads need not wait for the device positions.
  const int e0 = min(it.kv_end, it.pos_max[0] + 1), e1 = min(it.kv_end, it.pos_max[1] + 1);
  v.ntile0 = e0 > it.kv_start ? (e0 - it.kv_start + kNK - 1) / kNK : 0;
  v.ntile1 = e1 > it.kv_start ? (e1 - it.kv_start + kNK - 1) / kNK : 0;
  v.kv_end = max(it.kv_start, max(e0, e1));
  v.ntiles = max(v.ntile0, v.ntile1);
  return v;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (x0, x1) * s + (c, c) with one paired fp32 FMA.
__device__ __forceinline__ void fma2(float& x0, float& x1, float s, float c) {
  asm("{\n\t.reg .b64 p, q, r;\n\tmov.b64 p, {%0, %1};\n\tmov.b64 q, {%2, %2};\n\tmov.b64 r, {%3, %3};\n\t"
      "fma.rn.f32x2 p, p, q, r;\n\tmov.b64 {%0, %1}, p;\n\t}"
      : "+f"(x0), "+f"(x1) : "f"(s), "f"(c));
}

// (a0, a1) += (b0, b1) with one paired fp32 add.
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  asm("{\n\t.reg .b64 p, q;\n\tmov.b64 p, {%0, %1};\n\tmov.b64 q, {%2, %3};\n\t"
      "add.rn.f32x2 p, p, q;\n\tmov.b64 {%0, %1}, p;\n\t}"
      : "+f"(a0), "+f"(a1) : "f"(b0), "f"(b1));
}

// FP8 pools: a stage holds the tile's e4m3 codes, [128 keys][D] bytes, in its
// upper half (as the TMA landed them); widen them in place to the f16 operand
// layout of the whole stage: [8-key group][64-column half][8 keys][128 bytes],
// 16-byte chunk c of a key's 128-byte line at c ^ (key % 8).  One warp.
//
// Each lane converts 8 codes into one 16-byte chunk per step, so the 8 lanes
// of a store phase fill the 8 chunks of one line (distinct banks after the
// swizzle) and read one key's contiguous codes.  Keys go in increasing order,
// 16 steps' codes loaded before any of their stores (the loads would
// otherwise wait behind the previous step's store).  The f16 line of key r
// (for r >= 64, in the upper half) covers the codes of a key no later than r:
// a batch overwrites only codes it or an earlier batch has already read.
template <int D>
__device__ __forceinline__ void widen_stage(uint8_t* stage, int lane) {
  using S = TcSmem<D>;
  constexpr int kGroups = D / 8;              // 8-code groups per key
  constexpr int kKeysPerStep = 32 / kGroups;  // keys converted per warp step
  constexpr int kBatch = 16;                  // steps whose codes are loaded together
  const uint8_t* codes = stage + S::kKV / 2;
  const int kk = lane / kGroups, g8 = lane % kGroups;
  const int hf = (g8 * 8) / 64, cw = g8 % 8;
#pragma unroll 1
  for (int b = 0; b < kNK / kKeysPerStep; b += kBatch) {
    uint2 v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      v[u] = *reinterpret_cast<const uint2*>(codes + ((b + u) * kKeysPerStep + kk) * D + g8 * 8);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int r = (b + u) * kKeysPerStep + kk, r8 = r % 8;
      uint4 h;
      e4m3x4_to_f16x4(v[u].x, h.x, h.y);
      e4m3x4_to_f16x4(v[u].y, h.z, h.w);
      *reinterpret_cast<uint4*>(stage + (r / 8) * S::kGS + hf * S::kHS + r8 * 128 + ((cw ^ r8) * 16)) = h;
    }
  }
}

template <int D, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
tc_attn_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
               const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_kn,
               const __grid_constant__ CUtensorMap tmap_vn, const WorkItem* __restrict__ items, int n_items) {
  using S = TcSmem<D>;
  constexpr int kKSt = S::kKSt, kVSt = S::kVSt;
  using B = Bars<kKSt, kVSt>;
  static_assert(B::kCount == S::kNumBars, "barrier count");
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {   // swizzle atoms need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(a.pool.err, PKV_DEVERR_INTERNAL);
    return;
  }
  // Once any wait in this launch has given up, later CTAs do nothing
  // (__syncthreads_or makes the decision the same for every thread).
  const unsigned err0 = *reinterpret_cast<volatile unsigned*>(a.pool.err);
  if (__syncthreads_or((err0 & PKV_DEVERR_TIMEOUT) != 0)) return;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + S::kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + S::kOffMisc + 32);
  volatile int* s_item = reinterpret_cast<volatile int*>(smem + S::kOffMisc + 40);   // two slots

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.group;
  const int Hkv = a.pool.num_kv_heads;
  const bool fused = a.k_new != nullptr;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kKSt; ++i) {
      mbar_init(&bars[B::kKFull + i], 1);
      mbar_init(&bars[B::kKEmpty + i], 1);
      mbar_init(&bars[B::kKLanded + i], 1);
    }
    for (int i = 0; i < kVSt; ++i) {
      mbar_init(&bars[B::kVFull + i], 1);
      mbar_init(&bars[B::kVEmpty + i], 1);
      mbar_init(&bars[B::kVLanded + i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars[B::kS + t], 1);
      mbar_init(&bars[B::kP + t], 128);
      mbar_init(&bars[B::kPv + t], 1);
      mbar_init(&bars[B::kQFull + t], 1);
      mbar_init(&bars[B::kQEmpty + t], 1);
      mbar_init(&bars[B::kQc + t], 128);
      mbar_init(&bars[B::kItemFull + t], 1);
      mbar_init(&bars[B::kItemEmpty + t], B::kItemReaders);
    }
    mbar_init(&bars[B::kDrain], 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
    if (fused) {
      prefetch_tmap(&tmap_kn);
      prefetch_tmap(&tmap_vn);
    }
  }
  if (warp == 9) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t sQ = smem_u32(smem + S::kOffQ);
  const uint32_t sK = smem_u32(smem + S::kOffK);
  const uint32_t sV = smem_u32(smem + S::kOffV);

  // Item r of this CTA is in ring slot r % 2.  take_item: every reading role
  // waits for it, reads it and releases the slot (one arrival per warp);
  // the index n_items means no more items.
  auto take_item = [&](int r, int& w) -> bool {
    const int slot = r & 1;
    if (!mbar_wait_warp(&bars[B::kItemFull + slot], (r >> 1) & 1, s_abort, a.wait_ns)) return false;
    w = s_item[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[B::kItemEmpty + slot]);
    return true;
  };

  if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ producers: warp 8 K, warp 10 V
    // Warp 8 also claims the CTA's items (a launch-wide counter: a CTA that
    // starts late, beside the split-KV kernel, just takes fewer) and loads
    // each item's query tiles.  K and V stream from two warps, so that
    // neither waits behind the other's free stages: a K stage frees when its
    // key tile's S MMAs finish, a V stage when both tiles' PVs on it finish.
    const bool is_k = warp == 8;
    const int nst = is_k ? kKSt : kVSt;
    constexpr int kBlk = kNK / kBlockSize;   // blocks per key tile (8)
    constexpr int kWin = 32 / kBlk;          // key tiles per window of 32 block ids
    constexpr int kNoBlock = INT_MIN;        // past the item's blocks
    uint32_t landed_par = 0;   // bit st: parity of this warp's next wait on landed barrier st
    int cnt = 0;               // K (or V) tiles this warp has issued in the launch
    int fin = 0;               // FP8: tiles widened and handed to the issuer
    int nq = 0;                // warp 8: items whose query tiles it has issued
    bool ok = true;
    for (int r = 0; ok; ++r) {
      int w = n_items;
      if (is_k) {
        const int slot = r & 1;
        if (!(ok = mbar_wait_warp(&bars[B::kItemEmpty + slot], ((r >> 1) & 1) ^ 1, s_abort, a.wait_ns))) break;
        int v = 0;
        if (lane == 0) v = atomicAdd(a.tc_next, 1);
        w = min(__shfl_sync(0xffffffffu, v, 0), n_items);
        if (lane == 0) {
          s_item[slot] = w;
          mbar_arrive(&bars[B::kItemFull + slot]);
        }
        __syncwarp();
      } else if (!(ok = take_item(r, w))) {
        break;
      }
      if (w >= n_items) break;
      const TcItem iv = tc_item(items, w, G);
      const WorkItem& it = iv.it;
      const int g = it.kv_head;
      const int kv_end = iv.kv_end;
      if (is_k) {
        // Query tiles, each once the previous item's last S MMA on it has
        // completed.  Rows (token, head) of a tile land as [half][row][64
        // columns]; rows past the tile are other tokens' rows or zeros,
        // computed and never stored.
        for (int t = 0; t < 2 && ok; ++t) {
          if (!(ok = mbar_wait_warp(&bars[B::kQEmpty + t], (r & 1) ^ 1, s_abort, a.wait_ns))) break;
          if (lane == 0) {
            if ((t ? iv.rows1 : iv.rows0) > 0) {
              mbar_arrive_expect_tx(&bars[B::kQFull + t], static_cast<uint32_t>(D * 2 * G * a.q_box_tokens));
              uint8_t* qt = smem + S::kOffQ + t * S::kQ;
#pragma unroll
              for (int hf = 0; hf < S::kHalves; ++hf)
                tma_load_3d(qt + hf * (kTcRows * 128), &tmap_q, hf * 64, g * G, t ? iv.tok01 : iv.tok00,
                            &bars[B::kQFull + t]);
            } else {
              mbar_arrive(&bars[B::kQFull + t]);
            }
          }
          __syncwarp();
        }
        if (!ok) break;
        nq = r + 1;
      }
      // Block ids are read a window ahead: lane l holds the id of block
      // (first block of the item) + 32 w + l, and the next window is in
      // flight while the current one is used.  A window's ids are checked
      // (bad ids flagged) when it becomes current.
      const int32_t* bt_row = a.block_tables + static_cast<int64_t>(it.req) * a.max_blocks;
      const int blk_first = it.kv_start / kBlockSize;
      const int blk_end = (kv_end + kBlockSize - 1) / kBlockSize;
      auto load_window = [&](int wi) -> int {   // lane l: raw id of block blk_first + 32 wi + l
        const int col = blk_first + wi * 32 + lane;
        if (col >= blk_end) return kNoBlock;
        return col < a.max_blocks ? __ldg(bt_row + col) : -1;
      };
      auto check_window = [&](int pb) -> int {   // the id, or -1 for none (an invalid id is flagged)
        if (pb == kNoBlock) return -1;
        if (pb < 0 || pb >= a.pool.num_blocks) {
          atomicOr(a.pool.err, PKV_DEVERR_BLOCK_ID);
          return -1;
        }
        return pb;
      };
      int win = 0;
      int ids_cur = load_window(0), ids_next = load_window(1);
      int run_b = 0, run_e = 0;   // fused call: the request's runs of new positions
      if (fused) {
        run_b = __ldg(a.run_off + it.req);
        run_e = __ldg(a.run_off + it.req + 1);
      }
      ids_cur = check_window(ids_cur);
      // (block, head) chunk index of this lane's block in key tile j (-1: none).
      auto block_chunk = [&](int j) -> int {
        if (j / kWin != win) {
          win = j / kWin;
          ids_cur = check_window(ids_next);
          ids_next = load_window(win + 1);
        }
        const int key0 = it.kv_start + j * kNK;
        const int nblk = (min(kNK, kv_end - key0) + kBlockSize - 1) / kBlockSize;
        int pb = __shfl_sync(0xffffffffu, ids_cur, (j % kWin) * kBlk + (lane % kBlk));
        if (lane >= nblk) pb = -1;
        return pb < 0 ? -1 : pb * Hkv + g;
      };
      // Fused call: the tokens of this step are not in the pool yet (the
      // launch beside this one writes them), so their keys and values come from
      // the new rows.  Run r says positions [p0, p0 + n) are tokens [t0, t0 + n).
      auto run_at = [&](int r) {
        const int4 v = __ldg(reinterpret_cast<const int4*>(a.runs) + r);
        return RunDesc{v.x, v.y, v.z, v.w};
      };
      // Overwrites, in a landed stage, every slot of block `blk` (first key bp)
      // that holds a new key below kv_end with that token's row (swizzled as
      // the TMA lands it: 16-byte chunk c of row r at chunk c ^ (r % 8) of its
      // 128-byte line).
      auto patch_block = [&](uint8_t* blk, int bp, bool is_k) {
        int tok = -1;
        const int p = bp + (lane & 15);
        if (p < kv_end) {
          for (int r = run_b; r < run_e; ++r) {
            const RunDesc rd = run_at(r);
            if (rd.p0 > p) break;
            if (p < rd.p0 + rd.n) {
              tok = rd.t0 + (p - rd.p0);
              break;
            }
          }
        }
        const uint8_t* src = static_cast<const uint8_t*>(is_k ? a.k_new : a.v_new);
        constexpr int kCpr = D / 8;   // 16-byte chunks per row
#pragma unroll
        for (int idx = lane; idx < kBlockSize * kCpr; idx += 32) {
          const int rr = idx / kCpr, c = idx % kCpr;
          const int t = __shfl_sync(0xffffffffu, tok, rr);
          if (t >= 0) {
            const uint4 v = *reinterpret_cast<const uint4*>(src + ((static_cast<int64_t>(t) * Hkv + g) * D) * 2 + c * 16);
            *reinterpret_cast<uint4*>(blk + (rr / 8) * S::kGS + (c / 8) * S::kHS + (rr % 8) * 128 +
                                      (((c % 8) ^ (rr % 8)) * 16)) = v;
          }
        }
      };
      auto load = [&](int j, int gk, int y) -> bool {
        const int st = gk % nst;
        const uint32_t ph = (gk / nst) & 1;
        uint64_t* full = &bars[(is_k ? B::kKFull : B::kVFull) + st];
        // Where lane l's block (keys bp .. bp + 15) comes from: 1 the pool; 2
        // the new rows, tokens src .. src + 15 (every key below kv_end belongs
        // to one run); 3 the pool, then its new keys patched in; 0 nothing.
        int cls = y >= 0 ? 1 : 0, src = -1;
        if (fused) {
          const int bp = it.kv_start + j * kNK + lane * kBlockSize;
          if (lane < kBlk && bp < kv_end) {
            const int live = min(bp + kBlockSize, kv_end);
            int nnew = 0, nrun = 0;
            for (int r = run_b; r < run_e; ++r) {
              const RunDesc rd = run_at(r);
              if (rd.p0 >= live) break;
              const int lo = max(bp, rd.p0), hi = min(live, rd.p0 + rd.n);
              if (lo < hi) {
                nnew += hi - lo;
                if (nrun++ == 0) src = rd.t0 + (bp - rd.p0);
              }
            }
            if (nnew == live - bp && nrun == 1) cls = 2;
            else if (nnew > 0 && y >= 0) cls = 3;
          }
        }
        const bool patch = __any_sync(0xffffffffu, cls == 3);
        // A pool box is a whole block; a box of new rows holds kn_box_tokens
        // tokens (8, fewer only when the batch has fewer tokens).
        const uint32_t my_bytes = cls == 2   ? 2u * a.kn_box_tokens * S::kHalves * 128u
                                  : cls != 0 ? static_cast<uint32_t>(S::kHalves * kBlockSize * 128)
                                             : 0u;
        const uint32_t bytes = __reduce_add_sync(0xffffffffu, my_bytes);
        // Free stage: released by the issuer after the last MMA that reads it.
        // Before a stage's first use, parity 1 of a fresh barrier passes at once.
        const int empty = (is_k ? B::kKEmpty : B::kVEmpty) + st;
        if (!mbar_wait_warp(&bars[empty], ph ^ 1, s_abort, a.wait_ns)) return false;
        // Test hook: CTA 0 never issues its first K tile, so that the issuer's
        // bounded wait for it runs out.
        if (a.withhold == 2 && is_k && gk == 0 && blockIdx.x == 0) return true;
        uint64_t* landed = &bars[(is_k ? B::kKLanded : B::kVLanded) + st];
        uint64_t* bar = patch ? landed : full;
        if (lane == 0) mbar_arrive_expect_tx(bar, bytes);
        __syncwarp();
        uint8_t* dst = smem + (is_k ? S::kOffK : S::kOffV) + st * S::kKV + lane * S::kBlkBytes;
        if (cls == 2) {
          // Two 8-token boxes of the new rows, one per 8-key group of the block.
          const CUtensorMap* m = is_k ? &tmap_kn : &tmap_vn;
          if constexpr (D == 128) {
            tma_load_4d(dst, m, 0, g, src, 0, bar);
            tma_load_4d(dst + S::kGS, m, 0, g, src + 8, 0, bar);
          } else {
            tma_load_3d(dst, m, 0, g, src, bar);
            tma_load_3d(dst + S::kGS, m, 0, g, src + 8, bar);
          }
        } else if (cls != 0) {
          if constexpr (D == 128)
            tma_load_4d(dst, is_k ? &tmap_k : &tmap_v, 0, 0, 0, 2 * y, bar);
          else
            tma_load_2d(dst, is_k ? &tmap_k : &tmap_v, 0, y * kBlockSize, bar);
        }
        if (patch) {
          const uint32_t par = (landed_par >> st) & 1u;
          landed_par ^= 1u << st;
          if (!mbar_wait_warp(landed, par, s_abort, a.wait_ns)) {
            (void)mbar_wait(landed, par, nullptr, a.wait_ns);   // let this tile's copies land
            return false;
          }
          uint8_t* stage = smem + (is_k ? S::kOffK : S::kOffV) + st * S::kKV;
          uint32_t mm = __ballot_sync(0xffffffffu, cls == 3);
          while (mm) {
            const int b = __ffs(mm) - 1;
            mm &= mm - 1;
            patch_block(stage + b * S::kBlkBytes, it.kv_start + j * kNK + b * kBlockSize, is_k);
          }
          fence_proxy_async_smem();   // the patched slots are read by the tensor cores
          __syncwarp();
          if (lane == 0) mbar_arrive(full);
        }
        return true;
      };
      // FP8 pools: the codes of the warp's tile gk (of the launch) land, on
      // landed barrier gk % nst, in the upper half of its stage; the warp widens the stage in place to f16,
      // patches the fused call's new rows in (quantised as the append stores
      // them) and arrives on full.  Copies run one tile ahead of the widening.
      // Issues the copy of the warp's tile gk into its stage, which is free.
      auto issue_f8 = [&](int gk, int y) {
        const int st = gk % nst;
        const uint32_t bytes = static_cast<uint32_t>(__popc(__ballot_sync(0xffffffffu, y >= 0))) * (kBlockSize * D);
        if (a.withhold == 2 && is_k && gk == 0 && blockIdx.x == 0) return;   // test hook (above)
        uint64_t* landed = &bars[(is_k ? B::kKLanded : B::kVLanded) + st];
        if (lane == 0) mbar_arrive_expect_tx(landed, bytes);
        __syncwarp();
        if (y >= 0)
          tma_load_2d(smem + (is_k ? S::kOffK : S::kOffV) + st * S::kKV + S::kKV / 2 + lane * (kBlockSize * D),
                      is_k ? &tmap_k : &tmap_v, 0, y * kBlockSize, landed);
      };
      // The fused call's new rows of block b of a widened stage: each new key's
      // row, quantised to codes (as the append stores it) and widened to f16.
      auto patch_block_f8 = [&](uint8_t* stage, int b, int bp, bool is_k) {
        int tok = -1;
        const int p = bp + (lane & 15);
        if (p < kv_end) {
          for (int r = run_b; r < run_e; ++r) {
            const RunDesc rd = run_at(r);
            if (rd.p0 > p) break;
            if (p < rd.p0 + rd.n) {
              tok = rd.t0 + (p - rd.p0);
              break;
            }
          }
        }
        const uint8_t* src = static_cast<const uint8_t*>(is_k ? a.k_new : a.v_new);
        const float sc = is_k ? a.pool.k_scale : a.pool.v_scale;
        constexpr int kC8 = D / 8;   // 8-element chunks per row
#pragma unroll
        for (int idx = lane; idx < kBlockSize * kC8; idx += 32) {
          const int rr = idx / kC8, c = idx % kC8;
          const int t = __shfl_sync(0xffffffffu, tok, rr);
          if (t >= 0) {
            const uint4 x = *reinterpret_cast<const uint4*>(src + ((static_cast<int64_t>(t) * Hkv + g) * D) * 2 + c * 16);
            const uint32_t c0 = quant_e4m3x4(x.x, x.y, sc), c1 = quant_e4m3x4(x.z, x.w, sc);
            uint4 h;
            e4m3x4_to_f16x4(c0, h.x, h.y);
            e4m3x4_to_f16x4(c1, h.z, h.w);
            const int r = b * kBlockSize + rr, hf = c / 8, cw = c % 8, r8 = r % 8;
            *reinterpret_cast<uint4*>(stage + (r / 8) * S::kGS + hf * S::kHS + r8 * 128 + ((cw ^ r8) * 16)) = h;
          }
        }
      };
      // Widens the warp's landed tile gk (key tile j of the item) and hands it to the issuer.
      auto finish_f8 = [&](int j, int gk) {
        const int st = gk % nst;
        uint8_t* stage = smem + (is_k ? S::kOffK : S::kOffV) + st * S::kKV;
        widen_stage<D>(stage, lane);
        if (fused) {
          __syncwarp();
          const int key0 = it.kv_start + j * kNK;
          const int bp = key0 + lane * kBlockSize;
          bool has_new = false;
          if (lane < kBlk && bp < kv_end) {
            const int live = min(bp + kBlockSize, kv_end);
            for (int r = run_b; r < run_e; ++r) {
              const RunDesc rd = run_at(r);
              if (rd.p0 >= live) break;
              if (max(bp, rd.p0) < min(live, rd.p0 + rd.n)) has_new = true;
            }
          }
          uint32_t mm = __ballot_sync(0xffffffffu, has_new);
          while (mm) {
            const int b = __ffs(mm) - 1;
            mm &= mm - 1;
            patch_block_f8(stage, b, key0 + b * kBlockSize, is_k);
          }
        }
        fence_proxy_async_smem();   // the widened rows are read by the tensor cores
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[(is_k ? B::kKFull : B::kVFull) + st]);
      };
      if constexpr (F8) {
        // A tile's codes are copied as soon as a stage is free, and widened as
        // soon as they have landed.  The warp tests both (without suspending)
        // and does whichever is ready: waiting for the next free stage before
        // widening a landed tile would serialise the widening with the MMAs
        // that free the stage.
        int jl = 0, jw = 0;      // key tiles of the item copied / widened
        uint64_t idle0 = 0;      // start of the current stretch without progress
        while (jw < iv.ntiles) {
          bool moved = false;
          if (jl < iv.ntiles && cnt - fin < nst &&
              mbar_test_warp(&bars[(is_k ? B::kKEmpty : B::kVEmpty) + cnt % nst], ((cnt / nst) & 1) ^ 1)) {
            issue_f8(cnt, block_chunk(jl));
            ++cnt;
            ++jl;
            moved = true;
          }
          if (fin < cnt && mbar_test_warp(&bars[(is_k ? B::kKLanded : B::kVLanded) + fin % nst], (fin / nst) & 1)) {
            finish_f8(jw, fin);
            ++fin;
            ++jw;
            moved = true;
          }
          if (moved) {
            idle0 = 0;
          } else {
            const uint64_t now = globaltimer_ns();
            if (idle0 == 0) idle0 = now;
            // One decision for the warp (each lane reads its own clock).
            if (__any_sync(0xffffffffu, *s_abort != 0 || now - idle0 > a.wait_ns)) {
              ok = false;
              break;
            }
          }
        }
      } else {
        for (int j = 0; j < iv.ntiles; ++j) {
          if (!(ok = load(j, cnt, block_chunk(j)))) break;
          ++cnt;
        }
      }
    }
    if (!ok) {   // gave up: flag it and let copies already issued land
      if (lane == 0) atomicOr(a.pool.err, PKV_DEVERR_TIMEOUT);
      *s_abort = 1;
      if constexpr (F8) {
        for (int i = fin; i < cnt; ++i)
          (void)mbar_wait(&bars[(is_k ? B::kKLanded : B::kVLanded) + i % nst], (i / nst) & 1, nullptr, a.wait_ns);
      } else {
        for (int i = max(0, cnt - nst); i < cnt; ++i)
          (void)mbar_wait(&bars[(is_k ? B::kKFull : B::kVFull) + i % nst], (i / nst) & 1, nullptr, a.wait_ns);
      }
      if (is_k && nq > 0) {
        for (int t = 0; t < 2; ++t) (void)mbar_wait(&bars[B::kQFull + t], (nq - 1) & 1, nullptr, a.wait_ns);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // FP8 pools: Q, the widened K / V and P are all f16.
    constexpr uint32_t idesc_s = F8 ? make_idesc_f16(128, kNK, false) : make_idesc_bf16(128, kNK, false);
    constexpr uint32_t idesc_o = F8 ? make_idesc_f16(128, D, true) : make_idesc_bf16(128, D, true);
    // Descriptors are built once; each MMA only advances the start-address
    // field (bits 0-13, in 16-byte units) by a constant offset.
    // K: K-major, 8-key groups kGS apart; V: MN-major, 64-dim halves kHS
    // apart (leading offset) and 8-key groups kGS apart (stride offset).
    const uint64_t dk = make_sdesc_sw128(sK, 16, S::kGS);
    const uint64_t dv = make_sdesc_sw128(sV, S::kHS, S::kGS);
    const uint64_t dqA = make_sdesc_sw128(sQ, 16, 1024), dqB = make_sdesc_sw128(sQ + S::kQ, 16, 1024);
    auto k_desc = [&](int gk) { return dk + static_cast<uint64_t>(((gk % kKSt) * S::kKV) >> 4); };
    auto v_desc = [&](int gv) { return dv + static_cast<uint64_t>(((gv % kVSt) * S::kKV) >> 4); };
    // The warp stays converged through the MMA issue: every lane computes the
    // same descriptors and executes the issue instructions, predicated so
    // that only the elected lane issues (one thread's MMAs, in order).  A
    // lane-0 branch around the issue measured a 129-cycle MMA cadence in the
    // steady state, against 64 cycles of tensor work per MMA.
    const uint32_t lead = elect_one();
    auto release = [&](int bar) { tc_commit_lead(lead, &bars[bar]); };
    // S_t = Q_t K^T into tile t's S columns (the key tile is in its stage, kd).
    auto issue_s = [&](int t, uint64_t kd) {
      const uint64_t dq = t ? dqB : dqA;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int hf = ks / 4, kk = ks % 4;
        tc_mma_lead(lead, tmem + t * kNK, dq + static_cast<uint64_t>((hf * (kTcRows * 128) + kk * 32) >> 4),
                    kd + static_cast<uint64_t>((hf * S::kHS + kk * 32) >> 4), idesc_s, ks > 0 ? 1u : 0u);
      }
      release(B::kS + t);
    };
    // O_t (+)= P_t V, P_t from TMEM (over S_t); the key tile's V in its stage, vd.
    auto issue_pv = [&](int t, bool acc, uint64_t vd) {
#pragma unroll
      for (int ks = 0; ks < kNK / 16; ++ks)
        tc_mma_ts_lead(lead, tmem + kColO + t * 128, tmem + t * kNK + ks * 8,
                       vd + static_cast<uint64_t>((ks * 2 * S::kGS) >> 4), idesc_o, (acc || ks > 0) ? 1u : 0u);
    };
    // FP8 pools: wait for the softmax warps' f16 conversion of the tiles instead.
    constexpr int kQReady = F8 ? B::kQc : B::kQFull;
    int kc = 0, vc = 0;        // K / V tiles of the launch consumed so far
    uint32_t pc0 = 0, pc1 = 0; // P phases of tile A / B waited so far
    bool ok = true;
    for (int r = 0; ok; ++r) {
      int w = n_items;
      if (!(ok = take_item(r, w))) break;
      if (w >= n_items) break;
      const TcItem iv = tc_item(items, w, G);
      const int ntile0 = iv.ntile0, ntile1 = iv.ntile1, ntiles = iv.ntiles;
      auto ntile_of = [&](int t) { return t ? ntile1 : ntile0; };
      const int last_nkeys = ntiles > 0 ? min(kNK, iv.kv_end - (iv.it.kv_start + (ntiles - 1) * kNK)) : kNK;
      if (!(ok = mbar_wait_warp(&bars[kQReady], r & 1, s_abort, a.wait_ns) &&
                 mbar_wait_warp(&bars[kQReady + 1], r & 1, s_abort, a.wait_ns)))
        break;
      // Every tile releases its query buffer after its last S MMA, a tile
      // without key tiles at once.  Its last PV is reported (kPv) only for a
      // tile with key tiles: an immediate report would complete together with
      // the previous item's (both wait for the same MMAs), two phases before
      // the softmax warps look, and their parity wait would miss it.
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (ntile_of(t) == 0) release(B::kQEmpty + t);
      if (ntiles > 0) {
        if (!(ok = mbar_wait_warp(&bars[B::kKFull + kc % kKSt], (kc / kKSt) & 1, s_abort, a.wait_ns))) break;
        tc_fence_after();
        const uint64_t kd = k_desc(kc);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (ntile_of(t) > 0) {
            issue_s(t, kd);
            if (ntile_of(t) == 1) release(B::kQEmpty + t);
          }
        }
        release(B::kKEmpty + kc % kKSt);
        ++kc;
      }
      // Per key tile j: PV_A(j), S_A(j+1), PV_B(j), S_B(j+1), so that tile B's
      // softmax runs while the tensor pipe works on tile A and the other way
      // round.
      for (int j = 0; ok && j < ntiles; ++j) {
        bool k_next = false;   // key tile j+1 seen in its stage
        const uint64_t vd = v_desc(vc), kd_next = k_desc(kc);
        if (!(ok = mbar_wait_warp(&bars[B::kVFull + vc % kVSt], (vc / kVSt) & 1, s_abort, a.wait_ns))) break;
        if (j == ntiles - 1 && last_nkeys < kNK) {
          // Keys past the item's end in its last tile: zero their V rows (the
          // unused tail of the last block holds any bits, stages past it stale
          // or never written data) so that 0 * that data cannot produce NaN in
          // the tensor core.  Lane l clears 16-byte chunk l % kCh of a row.
          uint8_t* vst = smem + S::kOffV + (vc % kVSt) * S::kKV;
          constexpr int kCh = S::kHalves * 8;   // 16-byte chunks of a key's row
          const int ch = lane % kCh;
          uint8_t* col = vst + (ch / 8) * S::kHS + (ch % 8) * 16;
          for (int key = last_nkeys + lane / kCh; key < kNK; key += 32 / kCh)
            *reinterpret_cast<uint4*>(col + (key / 8) * S::kGS + (key % 8) * 128) = make_uint4(0, 0, 0, 0);
          fence_proxy_async_smem();
          __syncwarp();
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (j < ntile_of(t)) {
            if (!(ok = mbar_wait_warp(&bars[B::kP + t], (t ? pc1 : pc0) & 1, s_abort, a.wait_ns))) break;
            if (t) ++pc1; else ++pc0;
            tc_fence_after();
            issue_pv(t, j > 0, vd);
            // Only the epilogue waits for PV: earlier PVs are covered by the
            // next S commit of the tile (the tensor pipe completes one thread's
            // MMAs in order).
            if (j == ntile_of(t) - 1) release(B::kPv + t);
            if (j + 1 < ntile_of(t)) {
              if (!k_next &&
                  !(ok = mbar_wait_warp(&bars[B::kKFull + kc % kKSt], (kc / kKSt) & 1, s_abort, a.wait_ns)))
                break;
              k_next = true;
              // No tcgen05 fence: TMA data is ordered by the K barrier, and the P
              // wait above already ordered the softmax's TMEM writes before this
              // thread's MMAs, which the tensor pipe runs in issue order.
              issue_s(t, kd_next);
              if (j + 1 == ntile_of(t) - 1) release(B::kQEmpty + t);
            }
          }
        }
        if (!ok) break;
        if (k_next) {
          release(B::kKEmpty + kc % kKSt);
          ++kc;
        }
        release(B::kVEmpty + vc % kVSt);
        ++vc;
      }
    }
    if (!ok) {
      if (lane == 0) atomicOr(a.pool.err, PKV_DEVERR_TIMEOUT);
      *s_abort = 1;
    }
    // Drain: every MMA issued has completed before TMEM is released.
    release(B::kDrain);
    (void)mbar_wait_warp(&bars[B::kDrain], 0, nullptr, a.wait_ns);
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax / epilogue of tile X
    const int X = (warp >> 2) & 1;            // query tile of the warp (0 = A, 1 = B)
    const int row = threadIdx.x & 127;        // its row within the tile (TMEM lane)
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t colS = X * kNK, colO = kColO + X * 128;
    // FP8 pools: S holds q . code, so k_scale joins the score scale (and
    // v_scale the final 1/l).
    const float sl2 = F8 ? a.scale_log2 * a.pool.k_scale : a.scale_log2;
    uint32_t sc = 0;   // S phases of the tile waited so far
    uint32_t pvc = 0;  // its items with key tiles so far (kPv phases)
    // The next item (its index, descriptor and this row's query position) is
    // read before the current item's epilogue: its global loads then overlap
    // the epilogue instead of delaying the next item's first softmax step.
    // The K producer claims it once it has issued the current item's last K
    // tile, which the S MMAs of the steps already softmaxed have consumed.
    TcItem nv{};
    int nqpos = -1;
    auto fetch = [&](int wi) {
      if (wi >= n_items) return;
      nv = tc_item(items, wi, G);
      const int nr = X ? nv.rows1 : nv.rows0;
      nqpos = row < nr ? __ldg(a.q_positions + (X ? nv.tok01 : nv.tok00) + row / G) : -1;
    };
    int w = n_items;
    bool ok = take_item(0, w);
    if (ok) fetch(w);
    for (int r = 0; ok && w < n_items; ++r) {
      const TcItem iv = nv;
      const int qpos = nqpos;
      const WorkItem& it = iv.it;
      const int g = it.kv_head;
      const int nrows = X ? iv.rows1 : iv.rows0;
      const int nt = X ? iv.ntile1 : iv.ntile0;
      const int min_pos = X ? it.pos_min[1] : it.pos_min[0];
      const int kv_end = iv.kv_end;
      const int rows0 = iv.rows0;
      auto tok0_of = [&](int t) { return t ? iv.tok01 : iv.tok00; };
      float m = -CUDART_INF_F, l = 0.f;
      if constexpr (F8) {
        // The widened K and V are f16, and both operands of an MMA share one
        // type: convert this thread's Q row of its tile to f16 in place once the
        // tile has landed (exact within f16's range).
        ok = mbar_wait_warp(&bars[B::kQFull + X], r & 1, s_abort, a.wait_ns);
        if (ok) {
          uint8_t* qrow = smem + S::kOffQ + X * S::kQ + row * 128;
#pragma unroll
          for (int hf = 0; hf < S::kHalves; ++hf) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              uint4* q16 = reinterpret_cast<uint4*>(qrow + hf * (kTcRows * 128) + c * 16);
              uint4 v = *q16;
              v.x = pack_f16x2(bf16lo_to_f32(v.x), bf16hi_to_f32(v.x));
              v.y = pack_f16x2(bf16lo_to_f32(v.y), bf16hi_to_f32(v.y));
              v.z = pack_f16x2(bf16lo_to_f32(v.z), bf16hi_to_f32(v.z));
              v.w = pack_f16x2(bf16lo_to_f32(v.w), bf16hi_to_f32(v.w));
              *q16 = v;
            }
          }
          fence_proxy_async_smem();   // read by the tensor cores
        }
        mbar_arrive(&bars[B::kQc + X]);
      }
      for (int j = 0; ok && j < nt; ++j) {
        const int key0 = it.kv_start + j * kNK;
        if (!(ok = mbar_wait_warp(&bars[B::kS + X], sc & 1, s_abort, a.wait_ns))) break;
        ++sc;
          tc_fence_after();
          float s[kNK];
#pragma unroll
          for (int c = 0; c < kNK; c += 16) tmem_ld16(tmem + lane_base + colS + c, s + c);
          tmem_wait_ld();
          if (key0 + kNK - 1 > min_pos || key0 + kNK > kv_end) {
            // The row sees keys [0, min(qpos + 1, kv_end)): a prefix of the tile.
            const int lim = min(qpos + 1, kv_end) - key0;
#pragma unroll
            for (int c = 0; c < kNK; ++c) s[c] = c < lim ? s[c] : -CUDART_INF_F;
          }
          // Row max as 8 independent partials of 3-input maxima (one long
          // dependency chain would leave the softmax warps latency-bound).
          float mx8[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(s[2 * k], s[2 * k + 1]);
#pragma unroll
          for (int c = 16; c < kNK; c += 2) mx8[(c >> 1) & 7] = max3f(mx8[(c >> 1) & 7], s[c], s[c + 1]);
          const float mx = max3f(max3f(mx8[0], mx8[1], mx8[2]), max3f(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
          // Lazy rescaling: rows keep their reference max m while the tile max stays
          // within 2^kRescaleLog2 of it (P then stays <= 2^kRescaleLog2, fine for bf16
          // and fp32 sums); O and l always share the same reference, so the result
          // is exact.  The decision is per warp because TMEM loads and stores are
          // warp-collective.
          const float m_tile = mx * sl2;
          const bool grow = __any_sync(0xffffffffu, m_tile > m + kRescaleLog2);
          const float m_new = grow ? fmaxf(m, m_tile) : m;
          const float neg_m = m_new == -CUDART_INF_F ? 0.f : -m_new;
          float rs0[4] = {0.f, 0.f, 0.f, 0.f}, rs1[4] = {0.f, 0.f, 0.f, 0.f};
          // P = 2^(s * scale * log2 e - m) as bf16, written over S 32 keys at a
          // time (16 columns); S columns are all in registers already.
#pragma unroll
          for (int cc = 0; cc < kNK; cc += 32) {
            uint32_t pk[16];
#pragma unroll
            for (int c = cc; c < cc + 32; c += 2) {
              float x0 = s[c], x1 = s[c + 1];
              fma2(x0, x1, sl2, neg_m);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              add2(rs0[(c >> 1) & 3], rs1[(c >> 1) & 3], p0, p1);
              pk[(c - cc) / 2] = F8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
            }
            tmem_st16(tmem + lane_base + colS + cc / 2, reinterpret_cast<const float*>(pk));
          }
          const float rsum = ((rs0[0] + rs1[0]) + (rs0[1] + rs1[1])) + ((rs0[2] + rs1[2]) + (rs0[3] + rs1[3]));
          const float alpha = grow ? fast_exp2(m + neg_m) : 1.f;
          // O(j-1) is complete (S(j) was issued after PV(j-1) finished).
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
          l = l * alpha + rsum;
          m = m_new;
          tmem_wait_st();
          tc_fence_before();
        mbar_arrive(&bars[B::kP + X]);
      }
      int wn = n_items;
      if (ok && (ok = take_item(r + 1, wn))) fetch(wn);
      if (ok && nt > 0) {
        if (!(ok = mbar_wait_warp(&bars[B::kPv + X], pvc & 1, s_abort, a.wait_ns))) break;
        ++pvc;
      }
      tc_fence_after();
      // Epilogue.  `ok` is uniform within a warp; the TMEM loads are executed by
      // every thread of the warp, only the stores depend on the row being valid.
      if (ok) {
        constexpr float kLn2 = 0.69314718055994530942f;
        const bool valid = row < nrows;
        const float inv = l > 0.f ? (F8 ? a.pool.v_scale : 1.f) / l : 0.f;
        const float lse = l > 0.f ? (m + fast_log2(l)) * kLn2 : -CUDART_INF_F;
        const int t = tok0_of(X) + (valid ? row / G : 0);
        const int h = g * G + row % G;
        const int prow = it.part + (X == 0 ? row : rows0 + row);
        uint4* dst_o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.o) + (static_cast<int64_t>(t) * a.num_q_heads + h) * D);
        float4* dst_p = it.part >= 0 ? reinterpret_cast<float4*>(a.part_o + static_cast<int64_t>(prow) * D) : nullptr;
        // O in 64-column batches: four TMEM loads in flight per wait.
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 64) {
          float ob[64];
          if (nt > 0) {
#pragma unroll
            for (int c = 0; c < 64; c += 16) tmem_ld16(tmem + lane_base + colO + c0 + c, ob + c);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 64; ++e) ob[e] = 0.f;
          }
          if (valid) {
#pragma unroll
            for (int c = 0; c < 64; c += 16) {
              const float* o = ob + c;
              if (it.part < 0) {
                uint4 w0, w1;
                w0.x = pack_bf16x2(o[0] * inv, o[1] * inv);   w0.y = pack_bf16x2(o[2] * inv, o[3] * inv);
                w0.z = pack_bf16x2(o[4] * inv, o[5] * inv);   w0.w = pack_bf16x2(o[6] * inv, o[7] * inv);
                w1.x = pack_bf16x2(o[8] * inv, o[9] * inv);   w1.y = pack_bf16x2(o[10] * inv, o[11] * inv);
                w1.z = pack_bf16x2(o[12] * inv, o[13] * inv); w1.w = pack_bf16x2(o[14] * inv, o[15] * inv);
                // A thread writes its own row: one 32-byte store a sector
                // (half the requests of two 16-byte stores) where o allows it.
                if (a.o_align32) {
                  st_global_v8(dst_o + (c0 + c) / 8, w0, w1);
                } else {
                  dst_o[(c0 + c) / 8] = w0;
                  dst_o[(c0 + c) / 8 + 1] = w1;
                }
              } else {
#pragma unroll
                for (int e = 0; e < 16; e += 4)
                  dst_p[(c0 + c + e) / 4] = make_float4(o[e] * inv, o[e + 1] * inv, o[e + 2] * inv, o[e + 3] * inv);
              }
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
      w = wn;
    }

    if (!ok) {
      if (lane == 0) atomicOr(a.pool.err, PKV_DEVERR_TIMEOUT);
      *s_abort = 1;
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

template <int D, bool F8>
static int launch_tc_d(const AttnArgs& a, const CUtensorMap* tk, const CUtensorMap* tv, const CUtensorMap* tq,
                       const CUtensorMap* tkn, const CUtensorMap* tvn, const WorkItem* items, int n_items,
                       void* stream) {
  const int smem = TcSmem<D>::kTotal;
  cudaError_t e = smem_attr_once<tc_attn_kernel<D, F8>>(smem);
  if (e != cudaSuccess) return e;
  tc_attn_kernel<D, F8><<<a.tc_ctas, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(a, *tk, *tv, *tq, *tkn,
                                                                                          *tvn, items, n_items);
  return cudaGetLastError();
}

int launch_tc(const AttnArgs& a, const void* tmap_k, const void* tmap_v, const void* tmap_q, const void* tmap_kn,
              const void* tmap_vn, const WorkItem* items, int n_items, void* stream) {
  if (n_items <= 0) return cudaSuccess;
  const CUtensorMap* tk = static_cast<const CUtensorMap*>(tmap_k);
  const CUtensorMap* tv = static_cast<const CUtensorMap*>(tmap_v);
  const CUtensorMap* tq = static_cast<const CUtensorMap*>(tmap_q);
  const CUtensorMap* tkn = static_cast<const CUtensorMap*>(tmap_kn);
  const CUtensorMap* tvn = static_cast<const CUtensorMap*>(tmap_vn);
  const bool f8 = a.pool.elem_bytes == 1;
  if (a.pool.head_dim == 128)
    return f8 ? launch_tc_d<128, true>(a, tk, tv, tq, tkn, tvn, items, n_items, stream)
              : launch_tc_d<128, false>(a, tk, tv, tq, tkn, tvn, items, n_items, stream);
  return f8 ? launch_tc_d<64, true>(a, tk, tv, tq, tkn, tvn, items, n_items, stream)
            : launch_tc_d<64, false>(a, tk, tv, tq, tkn, tvn, items, n_items, stream);
}

}  // namespace pkv

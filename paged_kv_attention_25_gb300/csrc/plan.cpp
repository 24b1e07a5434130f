// Host worklist planner.
//
// Packs the ragged requests of one unified batch into CTA work items: one
// compact list holding only real work, with no padding to a common length and
// no launch per length bucket (the compact work queue of "PersistentKV:
// Page-Aware Decode Scheduling for Long-Context LLM Serving on Commodity
// GPUs", section 2), and long key ranges cut into partitions that run on
// different SMs and are merged by log-sum-exp (the same page's split of one
// long context into chapters).  Unlike that page, the split count is not a
// constant: it is chosen from the batch's total work so that every kernel has
// several items per CTA slot.
//
// Routing: a request whose query rows per KV head (q_len * G) fit in
// kDecodeMaxRows goes to the CUDA-core split-KV kernel (HBM streaming, one
// item per KV head); every other request goes to the tensor-core kernel in
// tiles of at most 128 query rows.
#include <algorithm>
#include <cstring>

#include "internal.h"

namespace pkv {

namespace {

constexpr int kDecodeCtasPerSm = 3;
constexpr int kTcCtasPerSm = 1;
// Split-KV items are cut to 1/s of the average per-slot load, with s the
// smallest of 1..kDecodeSplitsPerSlot that still yields kDecodeMinWaves waves
// of items (so that longest-first scheduling can balance the slots); every
// extra split costs a CTA's fixed latency and a partial merge, and occupies
// SMs the tensor-core kernel is waiting for.  A tensor-core partial is a
// 128-row fp32 tile, so those items are cut only when they exceed the average
// per-slot load (longest-first scheduling then keeps the tail within about
// one item of the mean).
constexpr int kDecodeSplitsPerSlot = 4;
constexpr int kDecodeMinWaves = 2;
constexpr int kTcSplitsPerSlot = 1;
constexpr int kMinDecodeChunk = 16;     // blocks (256 keys) per split at least
constexpr int kMinTcChunk = 4;          // 128-key tiles (512 keys) per split at least

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct QGroup {
  int req;
  int q_start;
  int q_count;   // tokens (of the first tile, for a tensor-core pair)
  int kv_len;    // keys the group can see: min(ctx, max position + 1)
  int q_count2;  // tokens of the second tensor-core tile (0: none)
  int pos_max[2], pos_min[2];   // position bounds of the tile(s)
};

}  // namespace

bool plan_matches(const Plan& plan, const PlanParams& pp, const pkv_host_meta& meta) {
  if (!plan.valid || !meta.cu_q_lens || !meta.ctx_lens) return false;
  const PlanParams& k = plan.key_pp;
  if (k.num_q_heads != pp.num_q_heads || k.num_kv_heads != pp.num_kv_heads || k.head_dim != pp.head_dim ||
      k.num_sms != pp.num_sms || k.num_reqs != pp.num_reqs || k.num_tokens != pp.num_tokens ||
      k.kv_elem_bytes != pp.kv_elem_bytes || plan.key_has_pos != (meta.q_positions != nullptr))
    return false;
  auto same = [](const std::vector<int32_t>& a, const int32_t* b, size_t n) {
    return a.size() == n && (n == 0 || std::memcmp(a.data(), b, n * sizeof(int32_t)) == 0);
  };
  return same(plan.key_cu, meta.cu_q_lens, static_cast<size_t>(pp.num_reqs) + 1) &&
         same(plan.key_ctx, meta.ctx_lens, static_cast<size_t>(pp.num_reqs)) &&
         (!plan.key_has_pos || same(plan.key_pos, meta.q_positions, static_cast<size_t>(pp.num_tokens)));
}

namespace {

// The cache key of a plan: exact copies of everything it was built from.
void remember_key(Plan* plan, const PlanParams& pp, const pkv_host_meta& meta) {
  plan->key_pp = pp;
  plan->key_cu.assign(meta.cu_q_lens, meta.cu_q_lens + pp.num_reqs + 1);
  plan->key_ctx.assign(meta.ctx_lens, meta.ctx_lens + pp.num_reqs);
  plan->key_has_pos = meta.q_positions != nullptr;
  if (plan->key_has_pos) plan->key_pos.assign(meta.q_positions, meta.q_positions + pp.num_tokens);
  else plan->key_pos.clear();
}

}  // namespace

int check_ctx_fits(const pkv_host_meta& meta, int num_reqs, int max_blocks, const char** err) {
  const int64_t cap = static_cast<int64_t>(max_blocks) * kBlockSize;
  for (int r = 0; r < num_reqs; ++r)
    if (meta.ctx_lens[r] > cap) {
      *err = "plan: ctx_len exceeds max_blocks * block_size";
      return PKV_EINVAL;
    }
  return PKV_OK;
}

int build_plan(const PlanParams& pp, const pkv_host_meta& meta, Plan* plan, const char** err) {
  // Reset, keeping every vector's capacity.
  plan->decode.clear();
  plan->tc.clear();
  plan->merge.clear();
  plan->merge_dec.clear();
  plan->runs.clear();
  plan->run_off.clear();
  plan->num_partial_rows = 0;
  plan->stats = pkv_plan_stats{};
  plan->off_decode = plan->off_tc = plan->off_merge = plan->off_merge_dec = plan->off_merge_cnt = 0;
  plan->off_runs = plan->off_run_off = plan->off_tc_next = 0;
  plan->off_part_o = plan->off_part_lse = plan->total = 0;
  plan->valid = false;
  const int R = pp.num_reqs, T = pp.num_tokens, Hq = pp.num_q_heads, Hkv = pp.num_kv_heads, D = pp.head_dim;
  if (R < 0 || T < 0 || Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0) {
    *err = "plan: bad head counts or sizes";
    return PKV_EINVAL;
  }
  const int G = Hq / Hkv;
  if (G > kTcRows) {
    *err = "plan: group size num_q_heads/num_kv_heads above 128";
    return PKV_EINVAL;
  }
  if (!meta.cu_q_lens || !meta.ctx_lens) {
    *err = "plan: host cu_q_lens and ctx_lens are required";
    return PKV_EINVAL;
  }
  const int32_t* cu = meta.cu_q_lens;
  const int32_t* ctx = meta.ctx_lens;
  const int32_t* pos = meta.q_positions;
  if (cu[0] != 0 || cu[R] != T) {
    *err = "plan: cu_q_lens must start at 0 and end at num_tokens";
    return PKV_EINVAL;
  }
  for (int r = 0; r < R; ++r) {
    if (cu[r + 1] < cu[r]) {
      *err = "plan: cu_q_lens must be nondecreasing";
      return PKV_EINVAL;
    }
    if (ctx[r] < 0 || (cu[r + 1] > cu[r] && ctx[r] < 1)) {
      *err = "plan: a request with query tokens needs ctx_len >= 1";
      return PKV_EINVAL;
    }
    if (pos) {
      for (int t = cu[r]; t < cu[r + 1]; ++t)
        if (pos[t] < 0 || pos[t] >= ctx[r]) {
          *err = "plan: query position outside [0, ctx_len)";
          return PKV_EINVAL;
        }
    }
  }

  // 1. Query groups: all tokens (split-KV route) or tiles of <= 128 rows.
  std::vector<QGroup> dec_groups, tc_groups;
  const int tq = kTcRows / G;  // tokens per tensor-core tile
  for (int r = 0; r < R; ++r) {
    const int n = cu[r + 1] - cu[r];
    if (n == 0) continue;
    auto kv_len_of = [&](int t0, int c) {
      if (!pos) return static_cast<int>(ctx[r]);
      int mx = 0;
      for (int t = t0; t < t0 + c; ++t) mx = std::max(mx, static_cast<int>(pos[t]));
      return std::min(static_cast<int>(ctx[r]), mx + 1);
    };
    // Position bounds of tokens [t0, t0 + c): exact with host positions, else
    // the whole context (masking then uses the device positions).
    auto bounds = [&](int t0, int c, int* mx, int* mn) {
      if (c == 0) {
        *mx = -1;
        *mn = 0;
      } else if (!pos) {
        *mx = static_cast<int>(ctx[r]) - 1;
        *mn = 0;
      } else {
        *mx = -1;
        *mn = 0x7fffffff;
        for (int t = t0; t < t0 + c; ++t) {
          *mx = std::max(*mx, static_cast<int>(pos[t]));
          *mn = std::min(*mn, static_cast<int>(pos[t]));
        }
      }
    };
    if (n * G <= kDecodeMaxRows) {
      QGroup q{r, cu[r], n, kv_len_of(cu[r], n), 0, {-1, -1}, {0, 0}};
      bounds(cu[r], n, &q.pos_max[0], &q.pos_min[0]);
      dec_groups.push_back(q);
      continue;
    }
    int t = cu[r];
    const int end = cu[r + 1];
    std::vector<std::pair<int, int>> tiles;   // (first token, tokens)
    while (t < end) {
      int c = 1;
      // A tile holds consecutive tokens; with known positions it also stops at
      // a jump in position (e.g. recomputed prefix [0,e) vs new tokens [c,..)),
      // so that each tile's key range ends near its own positions.
      while (c < tq && t + c < end) {
        if (pos && pos[t + c] != pos[t + c - 1] + 1) break;
        ++c;
      }
      tiles.push_back({t, c});
      t += c;
    }
    // Two consecutive tiles of a request share one CTA and every K/V tile it loads.
    for (size_t i = 0; i < tiles.size(); i += 2) {
      const int c0 = tiles[i].second;
      const int c1 = i + 1 < tiles.size() ? tiles[i + 1].second : 0;
      QGroup q{r, tiles[i].first, c0, kv_len_of(tiles[i].first, c0 + c1), c1, {-1, -1}, {0, 0}};
      bounds(tiles[i].first, c0, &q.pos_max[0], &q.pos_min[0]);
      bounds(tiles[i].first + c0, c1, &q.pos_max[1], &q.pos_min[1]);
      tc_groups.push_back(q);
    }
  }

  // 2. Split sizes from the total work of each kernel.
  int64_t dec_blocks = 0, tc_tiles = 0;
  for (const auto& g : dec_groups) dec_blocks += ceil_div(g.kv_len, kBlockSize) * Hkv;
  for (const auto& g : tc_groups) tc_tiles += ceil_div(g.kv_len, kTcKeys) * Hkv;   // per tile pair
  const int sms = std::max(1, pp.num_sms);
  const int64_t dec_slots = int64_t(sms) * kDecodeCtasPerSm;
  auto dec_chunk_for = [&](int s) { return std::max<int64_t>(kMinDecodeChunk, ceil_div(dec_blocks, dec_slots * s)); };
  auto dec_items_for = [&](int64_t chunk) {   // the split-KV item count emit() will produce
    int64_t n = 0;
    for (const auto& g : dec_groups) {
      const int64_t units = std::max<int64_t>(1, ceil_div(g.kv_len, kBlockSize));
      const int64_t per = ceil_div(units, std::max<int64_t>(1, ceil_div(units, chunk)));
      n += std::max<int64_t>(1, ceil_div(units, per)) * Hkv;
    }
    return n;
  };
  int64_t dec_chunk = dec_chunk_for(kDecodeSplitsPerSlot);
  for (int s = 1; s < kDecodeSplitsPerSlot; ++s) {
    const int64_t c = dec_chunk_for(s);
    if (dec_items_for(c) >= kDecodeMinWaves * dec_slots) {
      dec_chunk = c;
      break;
    }
  }
  const int64_t tc_chunk =
      std::max<int64_t>(kMinTcChunk, ceil_div(tc_tiles, int64_t(sms) * kTcCtasPerSm * kTcSplitsPerSlot));
  int merge_groups = 0;

  int part_rows = 0;
  // fused: the group's last split merges it inside the split-KV kernel (rows
  // fit one merge item); else the merge kernel does.
  auto emit = [&](const QGroup& g, int unit_keys, int64_t chunk_units, std::vector<WorkItem>& out, bool fused) {
    const int rows = (g.q_count + g.q_count2) * G;
    const int64_t units = ceil_div(g.kv_len, unit_keys);
    int nsplit = static_cast<int>(std::max<int64_t>(1, ceil_div(units, chunk_units)));
    // Even split in whole units; no split is left empty.
    const int64_t per = ceil_div(units, nsplit);
    nsplit = static_cast<int>(ceil_div(units, per));
    for (int kvh = 0; kvh < Hkv; ++kvh) {
      int base = -1, merge_id = -1;
      if (nsplit > 1) {
        base = part_rows;
        part_rows += nsplit * rows;
        ++merge_groups;
        std::vector<MergeItem>& ml = fused ? plan->merge_dec : plan->merge;
        if (fused) merge_id = static_cast<int>(ml.size());
        for (int r0 = 0; r0 < rows; r0 += kMergeRowsPerCta)
          ml.push_back({g.q_start, g.q_count + g.q_count2, kvh, nsplit, base, r0, std::min(kMergeRowsPerCta, rows - r0), 0});
      }
      for (int s = 0; s < nsplit; ++s) {
        const int64_t u0 = s * per;
        const int64_t u1 = std::min(units, u0 + per);
        WorkItem w;
        w.req = g.req;
        w.kv_head = kvh;
        w.q_start = g.q_start;
        w.q_count = static_cast<int16_t>(g.q_count);
        w.kv_start = static_cast<int32_t>(u0 * unit_keys);
        w.kv_end = static_cast<int32_t>(std::min<int64_t>(g.kv_len, u1 * unit_keys));
        w.part = nsplit > 1 ? base + s * rows : -1;
        w.q_count2 = static_cast<int16_t>(g.q_count2);
        w.merge_id = merge_id;
        for (int t = 0; t < 2; ++t) {
          w.pos_max[t] = g.pos_max[t];
          w.pos_min[t] = g.pos_min[t];
        }
        if (w.kv_end <= w.kv_start) {   // cannot happen with an even split; keep a valid empty item
          w.kv_end = w.kv_start;
        }
        out.push_back(w);
      }
    }
  };
  static_assert(kDecodeMaxRows <= kMergeRowsPerCta, "a split-KV group is one merge item");
  for (const auto& g : dec_groups) emit(g, kBlockSize, dec_chunk, plan->decode, true);
  for (const auto& g : tc_groups) emit(g, kTcKeys, tc_chunk, plan->tc, false);

  // 3. Longest items first, so that the tail of each launch is short; equal
  // lengths keep their emission order.  A stable LSD radix sort of the item
  // indices on (longest length - length), 8 bits a pass and only as many
  // passes as the longest length has bytes; the items are then moved once.
  auto longest_first = [plan](std::vector<WorkItem>& v) {
    const size_t n = v.size();
    if (n < 2) return;
    std::vector<uint32_t>& key = plan->order_key;
    std::vector<uint32_t>& idx = plan->order_idx;
    std::vector<uint32_t>& idx2 = plan->order_idx2;
    key.resize(n);
    idx.resize(n);
    idx2.resize(n);
    uint32_t longest = 0;
    for (size_t i = 0; i < n; ++i) {
      key[i] = static_cast<uint32_t>(v[i].kv_end - v[i].kv_start);
      longest = std::max(longest, key[i]);
    }
    for (size_t i = 0; i < n; ++i) {
      key[i] = longest - key[i];
      idx[i] = static_cast<uint32_t>(i);
    }
    for (int shift = 0; shift < 32 && (longest >> shift) != 0; shift += 8) {
      uint32_t start[257] = {};
      for (size_t i = 0; i < n; ++i) ++start[((key[idx[i]] >> shift) & 255u) + 1];
      for (int b = 0; b < 256; ++b) start[b + 1] += start[b];
      for (size_t i = 0; i < n; ++i) idx2[start[(key[idx[i]] >> shift) & 255u]++] = idx[i];
      idx.swap(idx2);
    }
    std::vector<WorkItem>& tmp = plan->order_tmp;
    tmp.resize(n);
    for (size_t i = 0; i < n; ++i) tmp[i] = v[idx[i]];
    v.swap(tmp);
  };
  longest_first(plan->decode);
  longest_first(plan->tc);
  // Tensor-core items of one request then go out together.  The request's
  // tile pairs read the same K/V (each pair a prefix of the request's keys),
  // so with them in flight at once a K/V tile comes from DRAM about once and
  // the other pairs find it in L2; ordered by their own lengths alone, the
  // pairs of a request end up hundreds of claims apart.  A request's rank is
  // the position of its first (longest) item, and a stable counting sort on
  // it keeps the longest-first order inside each request.
  if (plan->tc.size() > 1) {
    std::vector<WorkItem>& v = plan->tc;
    const size_t n = v.size();
    std::vector<uint32_t> rank(R, UINT32_MAX), start(R + 1, 0);
    uint32_t ranks = 0;
    for (size_t i = 0; i < n; ++i)
      if (rank[v[i].req] == UINT32_MAX) rank[v[i].req] = ranks++;
    for (size_t i = 0; i < n; ++i) ++start[rank[v[i].req] + 1];
    for (uint32_t b = 0; b < ranks; ++b) start[b + 1] += start[b];
    std::vector<WorkItem>& tmp = plan->order_tmp;
    tmp.resize(n);
    for (size_t i = 0; i < n; ++i) tmp[start[rank[v[i].req]]++] = v[i];
    v.swap(tmp);
  }
  plan->num_partial_rows = part_rows;

  // 4. Statistics (algorithmic work; each (request, KV head) KV read once).
  pkv_plan_stats& st = plan->stats;
  st.num_decode_items = static_cast<int>(plan->decode.size());
  st.num_tc_items = static_cast<int>(plan->tc.size());
  st.num_merge_items = merge_groups;
  st.num_partial_rows = part_rows;
  std::vector<int> req_kv_dec(R, 0), req_kv_tc(R, 0);
  for (const auto& g : dec_groups) req_kv_dec[g.req] = std::max(req_kv_dec[g.req], g.kv_len);
  for (const auto& g : tc_groups) req_kv_tc[g.req] = std::max(req_kv_tc[g.req], g.kv_len);
  const int64_t per_key = int64_t(2) * Hkv * D * pp.kv_elem_bytes;   // K and V, all KV heads
  for (int r = 0; r < R; ++r) {
    st.decode_kv_bytes += req_kv_dec[r] * per_key;
    st.tc_kv_bytes += req_kv_tc[r] * per_key;
  }
  auto row_flops = [&](const std::vector<QGroup>& gs) {
    int64_t f = 0;
    for (const auto& g : gs)
      for (int t = g.q_start; t < g.q_start + g.q_count + g.q_count2; ++t) {
        const int64_t vis = pos ? pos[t] + 1 : g.kv_len;
        f += int64_t(4) * D * vis * Hq;
      }
    return f;
  };
  st.decode_flops = row_flops(dec_groups);
  st.tc_flops = row_flops(tc_groups);
  auto io_bytes = [&](const std::vector<QGroup>& gs) {
    int64_t toks = 0;
    for (const auto& g : gs) toks += g.q_count + g.q_count2;
    return toks * Hq * (int64_t(D) * 2 * 2 + 4);   // Q in, O out (bf16), LSE out (fp32)
  };
  st.decode_io_bytes = io_bytes(dec_groups);
  st.tc_io_bytes = io_bytes(tc_groups);


  // 5. Runs of consecutive positions per request, sorted by first position
  // (the fused call's kernels look up which keys are new tokens).
  if (pos) {
    plan->run_off.resize(static_cast<size_t>(R) + 1);
    for (int r = 0; r < R; ++r) {
      plan->run_off[r] = static_cast<int32_t>(plan->runs.size());
      const size_t first = plan->runs.size();
      for (int t = cu[r]; t < cu[r + 1]; ++t) {
        if (t > cu[r] && pos[t] == pos[t - 1] + 1) {
          ++plan->runs.back().n;
        } else {
          plan->runs.push_back(RunDesc{pos[t], t, 1, 0});
        }
      }
      std::sort(plan->runs.begin() + first, plan->runs.end(),
                [](const RunDesc& x, const RunDesc& y) { return x.p0 < y.p0; });
    }
    plan->run_off[R] = static_cast<int32_t>(plan->runs.size());
  }

  // 6. Workspace layout.
  size_t off = 0;
  plan->off_decode = off;
  off = align256(off + plan->decode.size() * sizeof(WorkItem));
  plan->off_tc = off;
  off = align256(off + plan->tc.size() * sizeof(WorkItem));
  plan->off_merge = off;
  off = align256(off + plan->merge.size() * sizeof(MergeItem));
  plan->off_merge_dec = off;
  off = align256(off + plan->merge_dec.size() * sizeof(MergeItem));
  plan->off_merge_cnt = off;   // counters, uploaded as zeros with the work lists
  off = align256(off + plan->merge_dec.size() * sizeof(int32_t));
  plan->off_tc_next = off;     // the tensor-core kernel's next-item counter, uploaded as zero
  off = align256(off + sizeof(int32_t));
  plan->off_runs = off;
  off = align256(off + plan->runs.size() * sizeof(RunDesc));
  plan->off_run_off = off;
  off = align256(off + plan->run_off.size() * sizeof(int32_t));
  plan->off_part_o = off;
  off = align256(off + size_t(part_rows) * D * sizeof(float));
  plan->off_part_lse = off;
  off = align256(off + size_t(part_rows) * sizeof(float));
  plan->total = std::max<size_t>(off, 256);
  st.workspace_bytes = plan->total;
  remember_key(plan, pp, meta);
  ++plan->builds;
  plan->valid = true;
  return PKV_OK;
}

}  // namespace pkv

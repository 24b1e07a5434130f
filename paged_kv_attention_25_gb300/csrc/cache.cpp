// Two-tier KV block manager for multi-turn conversations: which blocks of
// which conversation sit in the GPU pool, in CPU host slots, or nowhere (to be
// recomputed), and the swaps and recomputation each step needs.
//
// "Stateful Large Language Model Serving with Pensieve" (abstract) keeps
// conversation history in a GPU/CPU cache and evicts it by conversation
// activity and recomputation cost, at block granularity, recomputing what was
// lost.  The pages give no formula; this file takes the plainest reading:
//   * A block's recompute cost is the prefill work of its tokens: for a token
//     at position p, a fixed `token_cost` (projections and MLP, in units of
//     one key's attention work) plus attention over its p + 1 keys.  Leading
//     blocks are therefore the cheapest to recompute.
//   * A conversation's blocks are ordered by position as [dropped][CPU][GPU].
//     Eviction moves the leading GPU block of an idle conversation to the CPU
//     tier, and the CPU tier drops its leading block when it is full, so that
//     what must be recomputed is always a prefix of positions (the
//     recompute-at-[0, e) shape the attention kernels take).
//   * Among the conversations not in the step, the victim is the one whose
//     leading block has the highest (steps since its last request) / (recompute
//     cost of that block); ties go to the lower conversation id.
// A returning conversation has its CPU blocks swapped in, its dropped prefix
// recomputed (positions [0, recompute)), and blocks added for its new tokens.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <map>
#include <set>
#include <string>
#include <vector>

#include "internal.h"

namespace {

struct Conv {
  int64_t len = 0;          // tokens whose K/V the cache holds or can recompute
  int dropped = 0;          // leading blocks not held anywhere
  std::vector<int> cpu;     // host slots of the next blocks, in position order
  std::vector<int> gpu;     // pool blocks of the remaining blocks, in position order
  int64_t last = 0;         // step of the conversation's last request
};

int64_t blocks_for(int64_t tokens) { return (tokens + pkv::kBlockSize - 1) / pkv::kBlockSize; }

}  // namespace

struct pkv_cache {
  int gpu_blocks = 0;
  int cpu_blocks = 0;
  double token_cost = 0;
  std::vector<int> gpu_free;   // stacks of free ids (lowest id on top)
  std::vector<int> cpu_free;
  std::map<int, Conv> convs;   // ordered by id: deterministic choices
  int64_t step = 0;

  // Prefill work of block b of c (its tokens only; a partial last block counts fewer).
  double cost(const Conv& c, int64_t b) const {
    const int64_t p0 = b * pkv::kBlockSize;
    const int64_t n = std::min<int64_t>(pkv::kBlockSize, c.len - p0);
    if (n <= 0) return 1.0;
    return n * token_cost + static_cast<double>(n) * p0 + n * (n + 1) / 2.0;
  }
  // The victim among conversations not in `skip` whose tier `cpu_tier` is not
  // empty: highest idle / cost of its leading block of that tier; -1 if none.
  int pick(bool cpu_tier, const std::set<int>& skip) const {
    int best = -1;
    double best_score = -1;
    for (const auto& [id, c] : convs) {
      if (skip.count(id) || (cpu_tier ? c.cpu.empty() : c.gpu.empty())) continue;
      const int64_t b = cpu_tier ? c.dropped : c.dropped + static_cast<int64_t>(c.cpu.size());
      const double score = static_cast<double>(step - c.last) / cost(c, b);
      if (score > best_score) {
        best_score = score;
        best = id;
      }
    }
    return best;
  }
};

extern "C" {

int pkv_cache_create(int gpu_blocks, int cpu_blocks, float token_cost, pkv_cache** out) {
  if (!out) return pkv::set_last_error(PKV_EINVAL, "out is NULL");
  *out = nullptr;
  if (gpu_blocks < 1 || cpu_blocks < 0 || !(token_cost >= 0.f))
    return pkv::set_last_error(PKV_EINVAL, "need gpu_blocks >= 1, cpu_blocks >= 0, token_cost >= 0");
  pkv_cache* c = new pkv_cache;
  c->gpu_blocks = gpu_blocks;
  c->cpu_blocks = cpu_blocks;
  c->token_cost = token_cost;
  for (int i = gpu_blocks - 1; i >= 0; --i) c->gpu_free.push_back(i);
  for (int i = cpu_blocks - 1; i >= 0; --i) c->cpu_free.push_back(i);
  *out = c;
  return PKV_OK;
}

int pkv_cache_destroy(pkv_cache* cache) {
  delete cache;
  return PKV_OK;
}

int pkv_cache_release(pkv_cache* cache, int conv) {
  if (!cache) return pkv::set_last_error(PKV_EINVAL, "cache is NULL");
  auto it = cache->convs.find(conv);
  if (it == cache->convs.end()) return PKV_OK;
  for (int b : it->second.gpu) cache->gpu_free.push_back(b);
  for (int s : it->second.cpu) cache->cpu_free.push_back(s);
  cache->convs.erase(it);
  return PKV_OK;
}

int pkv_cache_free_blocks(const pkv_cache* cache, int* gpu_free, int* cpu_free) {
  if (!cache) return pkv::set_last_error(PKV_EINVAL, "cache is NULL");
  if (gpu_free) *gpu_free = static_cast<int>(cache->gpu_free.size());
  if (cpu_free) *cpu_free = static_cast<int>(cache->cpu_free.size());
  return PKV_OK;
}

int pkv_cache_step(pkv_cache* cache, const int32_t* conv_ids, const int32_t* new_tokens, int n,
                   int32_t* block_tables, int max_blocks, int32_t* ctx_lens, int32_t* recompute, int32_t* swap_out,
                   int* num_swap_out, int32_t* swap_in, int* num_swap_in, int swap_cap) {
  if (!cache || n < 0 || (n > 0 && (!conv_ids || !new_tokens || !block_tables || !ctx_lens || !recompute)) ||
      !num_swap_out || !num_swap_in || swap_cap < 0 || max_blocks < 1)
    return pkv::set_last_error(PKV_EINVAL, "bad arguments");
  std::set<int> req;
  for (int r = 0; r < n; ++r) {
    if (conv_ids[r] < 0 || new_tokens[r] < 0) return pkv::set_last_error(PKV_EINVAL, "negative id or token count");
    if (!req.insert(conv_ids[r]).second) return pkv::set_last_error(PKV_EINVAL, "a conversation appears twice");
  }
  // Work on a copy: the cache changes only if the whole step fits.
  pkv_cache s = *cache;
  s.step += 1;
  int64_t demand = 0;
  for (int r = 0; r < n; ++r) {
    Conv& c = s.convs[conv_ids[r]];   // a new conversation starts empty
    const int64_t need = blocks_for(c.len + new_tokens[r]);
    if (need > max_blocks) return pkv::set_last_error(PKV_EINVAL, "a conversation needs more than max_blocks blocks");
    demand += need - static_cast<int64_t>(c.gpu.size());
  }
  int64_t evictable = 0;
  for (const auto& [id, c] : s.convs)
    if (!req.count(id)) evictable += static_cast<int64_t>(c.gpu.size());
  if (demand > static_cast<int64_t>(s.gpu_free.size()) + evictable)
    return pkv::set_last_error(PKV_ENOMEM, "the step's conversations do not fit in the GPU pool");

  std::vector<int32_t> outs, ins;   // pairs (gpu, cpu) and (cpu, gpu)
  // 1. Eviction until the step's blocks fit.
  while (static_cast<int64_t>(s.gpu_free.size()) < demand) {
    const int v = s.pick(false, req);
    Conv& cv = s.convs[v];
    const int blk = cv.gpu.front();
    if (s.cpu_free.empty() && s.cpu_blocks > 0) {
      const int w = s.pick(true, req);   // drop a CPU tier's leading block to make room
      if (w >= 0) {
        Conv& cw = s.convs[w];
        s.cpu_free.push_back(cw.cpu.front());
        cw.cpu.erase(cw.cpu.begin());
        cw.dropped += 1;
      }
    }
    if (!s.cpu_free.empty()) {
      const int slot = s.cpu_free.back();
      s.cpu_free.pop_back();
      outs.push_back(blk);
      outs.push_back(slot);
      cv.cpu.push_back(slot);
    } else {   // no CPU tier to move to: the block is dropped (its conversation has no CPU blocks)
      cv.dropped += 1;
    }
    cv.gpu.erase(cv.gpu.begin());
    s.gpu_free.push_back(blk);
  }
  // 2. Residency of each requested conversation, in request order.
  auto take_gpu = [&s]() {
    const int b = s.gpu_free.back();
    s.gpu_free.pop_back();
    return b;
  };
  std::vector<int> rec(n), len(n);
  for (int r = 0; r < n; ++r) {
    Conv& c = s.convs[conv_ids[r]];
    std::vector<int> table;
    for (int i = 0; i < c.dropped; ++i) table.push_back(take_gpu());   // recomputed by this step
    for (int slot : c.cpu) {
      const int b = take_gpu();
      ins.push_back(slot);
      ins.push_back(b);
      s.cpu_free.push_back(slot);
      table.push_back(b);
    }
    table.insert(table.end(), c.gpu.begin(), c.gpu.end());
    const int64_t total = blocks_for(c.len + new_tokens[r]);
    while (static_cast<int64_t>(table.size()) < total) table.push_back(take_gpu());
    rec[r] = static_cast<int>(std::min<int64_t>(static_cast<int64_t>(c.dropped) * pkv::kBlockSize, c.len));
    c.len += new_tokens[r];
    len[r] = static_cast<int>(c.len);
    c.dropped = 0;
    c.cpu.clear();
    c.gpu = table;
    c.last = s.step;
  }
  if (static_cast<int>(outs.size() / 2) > swap_cap || static_cast<int>(ins.size() / 2) > swap_cap)
    return pkv::set_last_error(PKV_EINVAL, "more swaps than swap_cap");
  if ((!outs.empty() && !swap_out) || (!ins.empty() && !swap_in))
    return pkv::set_last_error(PKV_EINVAL, "swap arrays are NULL");
  // 3. Results, then commit.
  for (int r = 0; r < n; ++r) {
    const Conv& c = s.convs[conv_ids[r]];
    int32_t* row = block_tables + static_cast<int64_t>(r) * max_blocks;
    for (int i = 0; i < max_blocks; ++i) row[i] = i < static_cast<int>(c.gpu.size()) ? c.gpu[i] : -1;
    ctx_lens[r] = len[r];
    recompute[r] = rec[r];
  }
  if (!outs.empty()) std::memcpy(swap_out, outs.data(), outs.size() * sizeof(int32_t));
  if (!ins.empty()) std::memcpy(swap_in, ins.data(), ins.size() * sizeof(int32_t));
  *num_swap_out = static_cast<int>(outs.size() / 2);
  *num_swap_in = static_cast<int>(ins.size() / 2);
  *cache = std::move(s);
  return PKV_OK;
}

}  // extern "C"

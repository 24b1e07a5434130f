// Host-only check of the plan cache key (compiled by tests/test_plan_cache_cpu.py
// against the library's planner source): a plan is reused only for exactly the
// metadata and parameters it was built from.  Prints one line per check and
// exits non-zero on the first failure.
#include <cstdio>
#include <vector>

#include "internal.h"

using namespace pkv;

static int fails = 0;
static void expect(bool ok, const char* what) {
  std::printf("%s %s\n", ok ? "ok  " : "FAIL", what);
  if (!ok) ++fails;
}

int main() {
  // Three requests: a decode, a new turn, a recompute.
  std::vector<int32_t> cu = {0, 1, 9, 14};
  std::vector<int32_t> ctx = {300, 108, 400};
  std::vector<int32_t> pos = {299, 100, 101, 102, 103, 104, 105, 106, 107, 0, 1, 2, 398, 399};
  PlanParams pp{8, 2, 128, 148, 3, 14, 2};
  pkv_host_meta meta{cu.data(), ctx.data(), pos.data()};
  Plan plan;
  const char* err = "";
  expect(!plan_matches(plan, pp, meta), "an empty cache matches nothing");
  expect(build_plan(pp, meta, &plan, &err) == PKV_OK, "the batch plans");
  expect(plan.builds == 1, "one plan built");
  expect(plan_matches(plan, pp, meta), "the same metadata hits the cache");

  // Equal contents at other addresses still hit: the key is the values.
  std::vector<int32_t> cu2 = cu, ctx2 = ctx, pos2 = pos;
  pkv_host_meta copy{cu2.data(), ctx2.data(), pos2.data()};
  expect(plan_matches(plan, pp, copy), "a copy of the metadata hits the cache");

  // Any single changed element misses.
  for (size_t i = 0; i < pos2.size(); ++i) {
    pos2[i] ^= 1;
    if (plan_matches(plan, pp, copy)) expect(false, "a changed query position misses");
    pos2[i] ^= 1;
  }
  expect(true, "every changed query position misses");
  for (size_t i = 0; i < ctx2.size(); ++i) {
    ctx2[i] += 1;
    if (plan_matches(plan, pp, copy)) expect(false, "a changed context length misses");
    ctx2[i] -= 1;
  }
  expect(true, "every changed context length misses");
  cu2[1] = 2;
  cu2[2] = 9;
  expect(!plan_matches(plan, pp, copy), "a moved request boundary misses");
  cu2 = cu;
  pkv_host_meta nopos{cu.data(), ctx.data(), nullptr};
  expect(!plan_matches(plan, pp, nopos), "metadata without host positions misses");
  PlanParams other = pp;
  other.num_sms = 152;
  expect(!plan_matches(plan, other, meta), "another SM count misses");
  other = pp;
  other.kv_elem_bytes = 1;
  expect(!plan_matches(plan, other, meta), "another KV element size misses");
  other = pp;
  other.num_q_heads = 4;
  expect(!plan_matches(plan, other, meta), "another head count misses");

  // Two batches with the same request and token counts get different plans.
  std::vector<int32_t> ctx_b = {5000, 108, 400};
  std::vector<int32_t> pos_b = {4999, 100, 101, 102, 103, 104, 105, 106, 107, 0, 1, 2, 398, 399};
  pkv_host_meta meta_b{cu.data(), ctx_b.data(), pos_b.data()};
  expect(!plan_matches(plan, pp, meta_b), "a second batch misses");
  const size_t items_a = plan.decode.size();
  expect(build_plan(pp, meta_b, &plan, &err) == PKV_OK, "the second batch plans");
  expect(plan.builds == 2, "two plans built");
  expect(plan.decode.size() > items_a, "the longer decode is split into more items");
  expect(plan_matches(plan, pp, meta_b) && !plan_matches(plan, pp, meta), "the cache now holds the second batch");

  // The block-table row length is checked per call, outside the plan.
  expect(check_ctx_fits(meta_b, 3, 313, &err) == PKV_OK, "ctx 5000 fits 313 blocks");
  expect(check_ctx_fits(meta_b, 3, 312, &err) == PKV_EINVAL, "ctx 5000 does not fit 312 blocks");
  return fails ? 1 : 0;
}

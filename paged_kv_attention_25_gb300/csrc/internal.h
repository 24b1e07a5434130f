// Internal types shared by the host API, the planner and the kernels.
#pragma once
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "../../include/pkv.h"

namespace pkv {

constexpr int kBlockSize = 16;        // tokens per KV block
constexpr int kDecodeMaxRows = 4;     // query rows (tokens x group) per split-KV item
constexpr int kTcRows = 128;          // query rows per tensor-core tile (TMEM lanes)
constexpr int kTcKeys = 128;          // keys per tensor-core KV tile (8 blocks)

// One CTA of work.  Rows of an item are (token q_start + i, query head
// kv_head*G + j) for i < q_count + q_count2, j < G, numbered i*G + j.  A
// tensor-core item holds two query tiles: tokens [q_start, q_start+q_count)
// and the q_count2 tokens after them (0 when there is one tile); a split-KV
// item has q_count2 = 0.
struct alignas(16) WorkItem {
  int32_t req;
  int32_t kv_head;
  int32_t q_start;   // first token (index into [0, num_tokens))
  int16_t q_count;   // tokens in the (first) tile (<= 128)
  int16_t q_count2;  // tokens in the second tensor-core tile (<= 128)
  int32_t kv_start;  // first key position (multiple of the kernel's key tile)
  int32_t kv_end;    // one past the last key position this item may read
  int32_t part;      // -1: write O / LSE directly; else first fp32 partial row
  // Split-KV item of a split group: index of the group's merge item in the
  // fused list (the group's last split to finish merges it); else -1.
  int32_t merge_id;
  // Query-position bounds of tile 0 (the whole item for split-KV) and tile 1:
  // exact when the host knows the positions, else [0, ctx_len - 1].  The
  // kernels size their key range with them before the device positions land.
  int32_t pos_max[2];
  int32_t pos_min[2];
};
static_assert(sizeof(WorkItem) == 48, "WorkItem layout: three 16-byte loads");
static_assert(kTcRows <= 32767, "token counts of a tile fit 16 bits");

// Log-sum-exp merge of `nsplit` partial results of one (token tile, KV head),
// for rows [row_begin, row_begin + row_count) of that tile (one CTA each).
// Partial row of split s and tile row i: part_base + s * (q_count * G) + i.
constexpr int kMergeRowsPerCta = 4;
struct MergeItem {
  int32_t q_start;
  int32_t q_count;
  int32_t kv_head;
  int32_t nsplit;
  int32_t part_base;
  int32_t row_begin;
  int32_t row_count;
  int32_t pad;
};
static_assert(sizeof(MergeItem) == 32, "MergeItem layout");

// A run of a request's query tokens with consecutive positions: positions
// [p0, p0 + n) are tokens [t0, t0 + n).  The fused call's attention kernels
// take these keys and values from the new rows instead of the pool.
struct alignas(16) RunDesc {
  int32_t p0;
  int32_t t0;
  int32_t n;
  int32_t pad;
};

struct PlanParams {
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int num_sms;
  int num_reqs;
  int num_tokens;
  int kv_elem_bytes = 2;   // bytes per pool element (2 bf16, 1 fp8)
};

struct Plan {
  std::vector<WorkItem> decode;   // split-KV CUDA-core kernel
  std::vector<WorkItem> tc;       // tensor-core kernel
  std::vector<MergeItem> merge;        // merged by the merge kernel (tensor-core groups)
  std::vector<MergeItem> merge_dec;    // merged inside the split-KV kernel
  // Runs of new positions per request (host positions only), sorted by p0:
  // request r's are runs[run_off[r] .. run_off[r + 1]).
  std::vector<RunDesc> runs;
  std::vector<int32_t> run_off;
  int num_partial_rows = 0;
  pkv_plan_stats stats{};
  // Workspace layout (byte offsets, 256-aligned sections).
  size_t off_decode = 0, off_tc = 0, off_merge = 0, off_merge_dec = 0, off_merge_cnt = 0, off_runs = 0, off_run_off = 0,
         off_tc_next = 0;
  size_t off_part_o = 0, off_part_lse = 0, total = 0;
  bool valid = false;
  int64_t builds = 0;   // plans built into this object so far
  // Cache key: exact copies of the parameters and host metadata the plan was
  // built from.  (The block-table row length is not part of a plan: it only
  // bounds ctx_lens, which check_ctx_fits tests on every call.)
  PlanParams key_pp{};
  std::vector<int32_t> key_cu, key_ctx, key_pos;
  bool key_has_pos = false;
  // Scratch of the longest-first ordering.  A pool re-plans into the same Plan
  // whenever the batch changes, so every vector keeps its capacity from one
  // plan to the next: no reallocation, and no fresh pages to fault in.
  std::vector<uint32_t> order_key, order_idx, order_idx2;
  std::vector<WorkItem> order_tmp;
};

// Record `msg` as this thread's pkv_last_error() and return `code`.
int set_last_error(int code, const std::string& msg);

// Host planner.  Returns PKV_OK or PKV_EINVAL (message in *err).
int build_plan(const PlanParams& pp, const pkv_host_meta& meta, Plan* plan, const char** err);
// True if `plan` was built from exactly these parameters and metadata (the
// plan cache: an element-wise comparison, so distinct batches never share a plan).
bool plan_matches(const Plan& plan, const PlanParams& pp, const pkv_host_meta& meta);
// PKV_EINVAL unless every ctx_lens[r] <= max_blocks * block_size.
int check_ctx_fits(const pkv_host_meta& meta, int num_reqs, int max_blocks, const char** err);

// Kernel launchers (defined in the .cu files); return cudaError_t as int.
struct PoolView {
  const void* k;
  const void* v;
  int num_blocks, num_kv_heads, head_dim;
  unsigned* err;     // device error word
  int elem_bytes;    // 2: bf16 pool; 1: fp8 e4m3 codes
  float k_scale, v_scale;   // fp8 dequantisation scales (1 for bf16)
};

// Block ids of one swap launch, passed by value as a kernel parameter.
constexpr int kSwapIdsPerLaunch = 2048;
struct SwapIds {
  int32_t id[kSwapIdsPerLaunch];
};

// Moves n pool blocks to / from `buf`, laid out [n][2][Hkv][B][D]: host memory
// through its device mapping, or a device buffer.  max_ctas = 0 takes the
// CTA count that saturates the CPU-GPU link in that direction.
int launch_swap(const PoolView& pool, void* kp, void* vp, void* buf, const int32_t* ids, int n, bool to_host,
                int max_ctas, void* stream);

int launch_append(const PoolView& pool, void* kp, void* vp, const int32_t* bt, int max_blocks, int num_reqs,
                  const int32_t* cu_q_lens, const int32_t* positions, const void* k_new, const void* v_new,
                  int num_tokens, void* stream);

struct AttnArgs {
  PoolView pool;
  const void* q;
  int num_q_heads;
  int group;             // num_q_heads / num_kv_heads
  const int32_t* q_positions;
  const int32_t* block_tables;
  int max_blocks;
  const int32_t* ctx_lens;
  float scale_log2;      // scale * log2(e)
  void* o;
  int o_align32;         // o is 32-byte aligned: output rows take 32-byte stores
  float* lse;
  float* part_o;         // [num_partial_rows][head_dim]
  float* part_lse;       // [num_partial_rows]
  const MergeItem* merge_dec;   // merge items of split-KV groups (merged by their last split)
  int* merge_cnt;               // splits finished per such item (zeroed by the work-list upload)
  int q_box_tokens;             // tokens per query-tile copy of the tensor-core kernel's Q tensor map
  int* tc_next;                 // the tensor-core kernel's next unclaimed item (zeroed by the work-list upload)
  int tc_ctas;                  // CTAs of the tensor-core launch: one per SM, at most one per item
  // Fused append (pkv_append_paged_attn); k_new is nullptr in a plain call.
  // The attention kernels read the new tokens' keys and values from k_new /
  // v_new ([T][Hkv][D] bf16), never from the pool, and n_append_ctas extra
  // CTAs of the split-KV launch write them into the pool.
  const void* k_new;
  const void* v_new;
  const int32_t* cu_q_lens;     // device
  int num_reqs, num_tokens;
  int n_append_ctas;
  int kn_box_tokens;            // tokens per box of the new-row tensor maps (min(8, T))
  const RunDesc* runs;          // the plan's runs of new positions (device copy)
  const int32_t* run_off;
  uint64_t wait_ns;             // wall-clock limit of every bounded wait in the kernels
  int withhold;                 // test hook: 1 / 2 = CTA 0 of the split-KV / tensor-core kernel
                                // skips its first K copy, so that a bounded wait runs out
};

// One paged-attention call as the C ABI receives it (pkv_paged_attn and its
// variants), handled by paged_attn_call in api.cu.
struct AttnCall {
  const void* q = nullptr;
  int num_q_heads = 0;
  const int32_t* q_positions = nullptr;
  const int32_t* block_tables = nullptr;
  int max_blocks = 0;
  const int32_t* ctx_lens = nullptr;
  const int32_t* cu_q_lens = nullptr;
  int num_reqs = 0, num_tokens = 0;
  const pkv_host_meta* host_meta = nullptr;
  float scale = 0.f;
  void* o = nullptr;
  float* lse = nullptr;
  void* workspace = nullptr;
  size_t workspace_bytes = 0;
  void* stream = nullptr;
  // Scratch shared by every pool (the static entry point): workspace is that
  // scratch, an over-size plan is reported against its fixed limit, and the
  // work-list upload waits on scratch_free, which the call records again on
  // `stream` after its kernels (so calls on any pools follow one another).
  bool static_scratch = false;
  void* scratch_free = nullptr;   // cudaEvent_t
  // Fused append (pkv_append_paged_attn): the new rows [T][Hkv][D] bf16.
  const void* k_new = nullptr;
  const void* v_new = nullptr;
};
int paged_attn_call(pkv_pool* pool, const AttnCall& c);

// Raises Kernel's dynamic shared-memory limit to `bytes` once per device
// (devices 0-63; the attribute call costs host time on every launch
// otherwise, time that lands inside a step whenever the GPU waits on the
// host).
#ifdef __CUDACC__
template <auto Kernel>
cudaError_t smem_attr_once(int bytes) {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}
#endif

// dmap_k / dmap_v: the pool's decode maps (FP8 pools with D = 128: codes
// viewed as [chunks * 16][D], (D, 16) box, 128-byte swizzle; any valid map
// otherwise), built with the pool.
int launch_decode(const AttnArgs& a, const void* dmap_k, const void* dmap_v, const WorkItem* items, int n_items,
                  void* stream);
// tmap_q: Q viewed as [T][Hq][D] with a (64, G, q_box_tokens) box (128-byte
// swizzle), built per call by make_q_tmap.
// tmap_kn / tmap_vn: the fused call's new K / V rows viewed as [T][Hkv][D] with
// an 8-token box (make_new_tmap); any valid map when a.k_new is nullptr.
int launch_tc(const AttnArgs& a, const void* tmap_k, const void* tmap_v, const void* tmap_q, const void* tmap_kn,
              const void* tmap_vn, const WorkItem* items, int n_items, void* stream);
int launch_merge(const AttnArgs& a, const MergeItem* items, int n_items, void* stream);

}  // namespace pkv

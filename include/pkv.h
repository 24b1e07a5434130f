/*
 * pkv.h - C ABI of a GB300 (sm_103a) library for paged multi-token attention.
 *
 * The operation is the generalised PagedAttention of "Stateful Large Language
 * Model Serving with Pensieve" (abstract): in one unified batch every request
 * brings one or more new input tokens (a new-turn prefill, a single decode
 * token, or recomputed evicted history) that attend over that conversation's
 * cached keys and values, which sit in fixed-size blocks scattered over
 * non-contiguous GPU memory.  The block pool and the per-request block table
 * follow the PagedAttention description in the blog "LLM上下文缓存与状态复用机制的
 * 分析和探索" (section 3.1: fixed-size blocks allocated on demand, stored in
 * non-contiguous physical memory).  The CPU tier of Pensieve's multi-tier
 * cache (abstract; "ahead-of-time swapping" in the method summary) is served
 * by the swap calls.
 *
 * Conventions for every call
 *   - Return value: PKV_OK (0) or one of the PKV_E* codes below.  On error,
 *     pkv_last_error() returns a message (thread-local, valid until the next
 *     call on the same thread).  Arguments are validated on the host before
 *     anything is launched; an invalid argument launches nothing.
 *   - "device" pointers are CUDA device memory of the current device;
 *     "host" pointers are CPU memory.  The caller owns every buffer it passes
 *     (queries, new K/V, outputs, metadata, workspace, host swap buffers); the
 *     library owns only what pkv_pool_create allocated.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous with respect to the host unless stated.
 *   - Data that violates a precondition which can only be seen on the device
 *     (a block id outside the pool, a position outside the block table) is
 *     skipped by the kernels and recorded in the pool's device error word;
 *     pkv_check_device_errors() reads it.  Kernels never trap.  Every wait
 *     inside a kernel is bounded; a wait that runs out records
 *     PKV_DEVERR_TIMEOUT and the kernel returns.
 *
 * Layouts (row-major, bf16 = IEEE bfloat16 bit patterns)
 *   Kpool, Vpool : [num_blocks][num_kv_heads][block_size][head_dim] bf16
 *   block_tables : [num_reqs][max_blocks] int32; entry i of request r is the
 *                  physical block holding positions [i*B, (i+1)*B).  Entries at
 *                  or beyond ceil(ctx_len/B) are never read (-1 is customary).
 *   cu_q_lens    : [num_reqs+1] int32, cu_q_lens[0] = 0, nondecreasing; the
 *                  query tokens of request r are rows [cu_q_lens[r], cu_q_lens[r+1]).
 *   positions / q_positions : [num_tokens] int32 absolute positions.
 *   Q            : [num_tokens][num_q_heads][head_dim] bf16
 *   K, V (new)   : [num_tokens][num_kv_heads][head_dim] bf16
 *   O            : [num_tokens][num_q_heads][head_dim] bf16
 *   LSE          : [num_tokens][num_q_heads] fp32, natural log
 *   swap buffer  : [n][2][num_kv_heads][block_size][head_dim] of the pool's
 *                  element type (K then V)
 *   FP8 pools hold e4m3 codes (one byte) in the pool layout above.
 *
 * Supported shapes: block_size 16; head_dim 64 or 128; num_q_heads a
 * multiple of num_kv_heads with group size G = num_q_heads/num_kv_heads <= 128.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_OK 0
#define PKV_EINVAL 1       /* invalid argument, shape or size */
#define PKV_ENOMEM 2       /* device allocation failed (pkv_pool_create only) */
#define PKV_ECUDA 3        /* a CUDA runtime or driver call failed */
#define PKV_ETIMEOUT 4     /* a bounded device-side wait ran out */
#define PKV_EDEVICE 5      /* kernels skipped invalid data; see the error word */
#define PKV_EUNSUPPORTED 6 /* valid but not supported (e.g. head_dim 96) */

#define PKV_DTYPE_BF16 0
/* FP8 KV cache: K and V stored as OCP FP8 E4M3 codes (1 sign, 4 exponent bits
 * with bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN; largest
 * finite 448), one scale per pool for K and one for V: the value of a code c
 * is e4m3(c) * k_scale (or v_scale).  pkv_append quantises each new bf16
 * element x to the code nearest (ties to even) to the fp32 quotient x / scale,
 * finite values beyond 448 saturating to +-448.  Attention reads the codes
 * (half the bytes of bf16) and widens them to f16 (exact): the split-KV
 * kernel takes the dot products with q converted to f16 and fp32
 * accumulation (for one-row items on the warp-level MMA); the tensor-core
 * kernel widens each K/V tile in shared memory and runs its MMAs with f16
 * operands, P rounded to f16.  Q is converted from bf16 to f16 (exact for
 * |q| within f16's range, below 65504).  Q, O and the new K/V given to
 * pkv_append stay bf16. */
#define PKV_DTYPE_FP8_E4M3 1

/* Bits of the device error word (pkv_check_device_errors). */
#define PKV_DEVERR_BLOCK_ID 1u   /* a block-table entry outside [0, num_blocks) */
#define PKV_DEVERR_POSITION 2u   /* a position outside [0, max_blocks*block_size) */
#define PKV_DEVERR_TIMEOUT 4u    /* a bounded wait inside a kernel gave up */
#define PKV_DEVERR_INTERNAL 8u   /* a kernel found its launch configuration unusable */

typedef struct pkv_pool pkv_pool; /* opaque */

typedef struct {
  int num_blocks;   /* physical blocks in the pool, >= 1 */
  int block_size;   /* tokens per block; must be 16 */
  int num_kv_heads; /* >= 1 */
  int head_dim;     /* 64 or 128 */
  int dtype;        /* PKV_DTYPE_BF16 or PKV_DTYPE_FP8_E4M3 */
  /* Optional caller-owned device storage for the two pools (each
   * num_blocks*num_kv_heads*block_size*head_dim*E bytes, E = 2 for bf16 and 1
   * for fp8, 16-byte aligned).  NULL: the library allocates (and zero-fills)
   * the storage itself. */
  void* k_storage;
  void* v_storage;
  /* PKV_DTYPE_FP8_E4M3 only: dequantisation scales (finite, > 0). */
  float k_scale;
  float v_scale;
} pkv_pool_desc;

/* Host copies of the batch metadata, used to plan the work split.
 * cu_q_lens [num_reqs+1] and ctx_lens [num_reqs] are required;
 * q_positions [num_tokens] is optional (NULL: every query tile is assumed to
 * see the whole context, and kernels clip their key ranges on the device). */
typedef struct {
  const int32_t* cu_q_lens;
  const int32_t* ctx_lens;
  const int32_t* q_positions;
} pkv_host_meta;

/* What one planned batch contains (for reporting and the roofline). */
typedef struct {
  int num_decode_items;     /* CTAs of the CUDA-core split-KV kernel */
  int num_tc_items;         /* CTAs of the tensor-core kernel */
  int num_merge_items;      /* (token tile, KV head) groups merged by log-sum-exp */
  int num_partial_rows;     /* fp32 partial rows held in the workspace */
  int64_t decode_kv_bytes;  /* algorithmic K+V bytes read by the split-KV kernel */
  int64_t tc_kv_bytes;      /* algorithmic K+V bytes read by the tensor-core kernel */
  int64_t decode_flops;     /* 4*D per visible (query row, key) pair */
  int64_t tc_flops;
  int64_t decode_io_bytes;  /* Q read + O/LSE written for the split-KV kernel's rows */
  int64_t tc_io_bytes;      /* Q read + O/LSE written for the tensor-core kernel's rows */
  size_t workspace_bytes;   /* what pkv_paged_attn needs for this batch */
  int64_t plans_built;      /* pkv_last_plan_stats: plans this pool has built so far
                               (a call whose metadata equals the cached plan's builds none) */
} pkv_plan_stats;

/* Accumulated device time per kernel family while profiling is on. */
typedef struct {
  int launches[5];          /* 0 append, 1 split-KV, 2 tensor-core, 3 merge, 4 swap */
  double total_ms[5];
} pkv_profile;

/* Create a KV block pool.  Allocates the pools (unless caller storage is
 * given), a device error word, a 4 MiB device buffer for the attention
 * calls' work lists with two pinned 4 MiB host staging buffers, and builds
 * the TMA descriptors the tensor-core kernel uses.  Synchronous.  Errors: PKV_EINVAL (bad desc),
 * PKV_EUNSUPPORTED (block_size != 16, head_dim not 64/128), PKV_ENOMEM,
 * PKV_ECUDA (no device, driver too old). */
int pkv_pool_create(const pkv_pool_desc* desc, pkv_pool** out);

/* Destroy a pool: synchronises the device, frees what the library allocated.
 * NULL is accepted.  Caller storage is not freed. */
int pkv_pool_destroy(pkv_pool* pool);

/* Device addresses of the K and V pools (for tests and host gathers). */
int pkv_pool_kv_ptrs(const pkv_pool* pool, void** k, void** v);

/*
 * Paged KV append ("LLM上下文缓存与状态复用机制的分析和探索" section 3.1; the new
 * tokens of Pensieve's unified batch): for every token t of request r at
 * position p = positions[t] and every KV head g,
 *   Kpool[block_tables[r][p / B]][g][p % B][:] = k_new[t][g][:]   (bit copy)
 * and the same for V.  Device inputs: block_tables, cu_q_lens, positions,
 * k_new, v_new.  Positions of one request must be distinct (two tokens writing
 * one slot leave either value).  Out-of-range slots are skipped and flagged in
 * the device error word.  num_tokens == 0 is a no-op.
 */
int pkv_append(pkv_pool* pool, const int32_t* block_tables, int max_blocks, int num_reqs,
               const int32_t* cu_q_lens, const int32_t* positions, const void* k_new,
               const void* v_new, int num_tokens, void* stream);

/*
 * Workspace bytes pkv_paged_attn needs for this batch (plans the batch on the
 * host; the plan is cached and reused by a following pkv_paged_attn with the
 * same metadata).  Synchronous, host only.
 * Plan cache: a pool keeps its last plan together with exact copies of the
 * parameters and host metadata (cu_q_lens, ctx_lens, q_positions) it was
 * built from, and reuses it only when a call's are equal element by element;
 * any other batch is planned afresh.
 */
int pkv_paged_attn_workspace_size(pkv_pool* pool, int num_q_heads, int num_reqs, int num_tokens,
                                  const pkv_host_meta* host_meta, size_t* bytes);

/*
 * Generalised paged attention (Pensieve abstract: attention between multiple
 * input tokens over a GPU cache spread across non-contiguous memory).
 * For query token t of request r at position p_t = q_positions[t] and query
 * head h, with KV head g = h / (num_q_heads / num_kv_heads):
 *   s_j = scale * q[t][h] . K_r[j][g]   for keys j = 0 .. p_t   (causal on
 *         absolute position; K_r[j] is slot j % B of block block_tables[r][j / B])
 *   O[t][h]   = sum_j exp(s_j - m) V_r[j][g] / sum_j exp(s_j - m),  m = max_j s_j
 *   LSE[t][h] = m + ln(sum_j exp(s_j - m))
 * Preconditions: 0 <= p_t < ctx_lens[r] <= max_blocks * 16; every key
 * position < ctx_lens[r] has been written (append before attention);
 * block-table entries for positions < ctx_lens[r] are valid pool blocks.
 * The host checks the first two against host_meta (PKV_EINVAL); the kernels
 * check block ids and never read past a block-table row.
 *
 * Device inputs: q, q_positions, block_tables, ctx_lens, cu_q_lens.
 * Device outputs: o (bf16), lse (fp32; may be NULL).  host_meta holds host
 * copies of cu_q_lens / ctx_lens (and optionally q_positions) for planning.
 * workspace: device memory of at least pkv_paged_attn_workspace_size() bytes,
 * 256-byte aligned, owned by the caller and not used by other work in flight.
 * The split-KV partials live there (and the work lists, for a batch whose
 * lists exceed the pool's 4 MiB work-list buffer).  The work lists are
 * uploaded into a device buffer the pool owns, on a copy stream of the pool,
 * ordered after this pool's previous attention call (whatever its stream),
 * so the upload overlaps the caller's earlier work; lists larger than that
 * buffer go into the workspace on `stream`, after the work already queued
 * there.  Other work on other streams must not use the workspace while the
 * call runs.
 * Streams: the kernels run after the upload and after the work already on
 * `stream`.  When the batch has both split-KV and tensor-core work, the
 * split-KV kernel runs on `stream` and the tensor-core kernel on a second
 * stream owned by the pool, forked from `stream` (event) and joined back into
 * it before the merge; every effect of the call is complete once `stream`
 * passes the point after it.  A pending ahead-of-time swap-in on the pool
 * (pkv_swap_in_ahead) lands on `stream` before the kernels.
 * num_tokens == 0 is a no-op.  Errors: PKV_EINVAL for bad shapes, a workspace
 * that is too small, or host metadata that is inconsistent.
 */
int pkv_paged_attn(pkv_pool* pool, const void* q, int num_q_heads, const int32_t* q_positions,
                   const int32_t* block_tables, int max_blocks, const int32_t* ctx_lens,
                   const int32_t* cu_q_lens, int num_reqs, int num_tokens,
                   const pkv_host_meta* host_meta, float scale, void* o, float* lse,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * Fused paged KV append and attention (Pensieve abstract: one generalised
 * kernel over a unified batch whose new input tokens join the conversation's
 * cache and attend to it).  The result is that of
 *   pkv_append(pool, block_tables, max_blocks, num_reqs, cu_q_lens,
 *              q_positions, k_new, v_new, num_tokens, stream);
 *   pkv_paged_attn(pool, q, ...same arguments..., stream);
 * bit for bit in the pool, and O / LSE within the same rounding, but the
 * attention kernels take the step's own keys and values from k_new / v_new
 * ([num_tokens][num_kv_heads][head_dim] bf16, device, 16-byte aligned)
 * instead of reading them back from the pool, so nothing waits for the pool
 * write: CTAs of the split-KV launch write the new rows into the pool beside
 * the attention work (one launch fewer than the two calls).
 *   - FP8 pools whose batch has tensor-core work: the call appends first (its
 *     own launch on `stream`), then attends to the pool.  Every tensor-core
 *     CTA that reads a new row would otherwise quantise it again; the result
 *     is the same.
 *   - host_meta->q_positions is required (the plan records, per request, the
 *     runs of consecutive new positions); PKV_EINVAL without it.
 *   - Workspace: pkv_paged_attn_workspace_size for the same batch.
 *   - The pool's slots of the new tokens are written during the call; no
 *     other work may read them until the call is complete on `stream`.
 * Errors: those of pkv_append and pkv_paged_attn.
 */
int pkv_append_paged_attn(pkv_pool* pool, const void* q, int num_q_heads, const int32_t* q_positions,
                          const int32_t* block_tables, int max_blocks, const int32_t* ctx_lens,
                          const int32_t* cu_q_lens, int num_reqs, int num_tokens, const pkv_host_meta* host_meta,
                          const void* k_new, const void* v_new, float scale, void* o, float* lse, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * Paged attention for callers that cannot allocate device memory (a process
 * whose device memory belongs to another framework's caching allocator, code
 * inside an allocator or stream callback where allocating CUDA calls are not
 * allowed, or a latency-critical loop that must not take cudaMalloc's
 * implicit device-wide synchronisation).  The paper has no counterpart to this
 * entry point.
 *
 * Same operation, arguments, results and errors as pkv_paged_attn, without
 * the workspace: the work lists and split-KV partials live in one static
 * device array of PKV_STATIC_SCRATCH_BYTES that every GPU loading this
 * library holds until the process exits.  The call makes no cudaMalloc,
 * cudaFree or other allocating call.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and creates the one
 *     CUDA event that orders calls (below).  Make that first call before any
 *     stream capture.
 *   - A batch whose plan needs more scratch than PKV_STATIC_SCRATCH_BYTES is
 *     rejected with PKV_EINVAL before anything is launched; use
 *     pkv_paged_attn with a caller workspace for it.
 *   - Every call uses the same array, which keeps the last call's contents.
 *     Nothing in it is read before the same call writes it (the merge
 *     counters are cleared by the call's own upload), so no clearing is
 *     needed.  Calls on one device are ordered on the GPU in the order they
 *     were made, whatever their pools and streams: each call's upload into the
 *     array waits for the previous call's kernels (an event the library
 *     records after them), and the host side holds a lock for the call's
 *     duration.  Work that other code runs on the array is not ordered: the
 *     array is this entry point's alone.
 */
#define PKV_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)
int pkv_paged_attn_static(pkv_pool* pool, const void* q, int num_q_heads, const int32_t* q_positions,
                          const int32_t* block_tables, int max_blocks, const int32_t* ctx_lens,
                          const int32_t* cu_q_lens, int num_reqs, int num_tokens,
                          const pkv_host_meta* host_meta, float scale, void* o, float* lse,
                          void* stream);

/* Statistics of the last plan built on this pool. */
int pkv_last_plan_stats(const pkv_pool* pool, pkv_plan_stats* out);

/*
 * CPU cache tier (Pensieve abstract: multi-tier GPU/CPU caching).  Copy n whole
 * physical blocks (all KV heads, K then V) from the pool to host memory laid
 * out [n][2][Hkv][B][D] (swap out), or back into the pool (swap in).
 * block_ids is a HOST array (copied into the launch; no upload).  With pinned
 * host_buf (cudaHostAlloc / registered, 16-byte aligned) one kernel moves all
 * blocks directly between HBM and host memory, asynchronously on `stream`,
 * on a few SMs only (8 CTAs out, 24 in: enough to saturate the CPU-GPU link,
 * so that it can run beside attention kernels);
 * with pageable memory the library falls back to DMA copies (one 2-D copy
 * per run of consecutive ids and pool), which the driver may serialise with
 * the host.  Issue on a side stream and record an event to overlap with
 * attention.
 * Errors: PKV_EINVAL for an id outside [0, num_blocks) (nothing is copied).
 */
int pkv_swap_out(pkv_pool* pool, const int32_t* block_ids, int n, void* host_buf, void* stream);
int pkv_swap_in(pkv_pool* pool, const int32_t* block_ids, int n, const void* host_buf, void* stream);

/*
 * Ahead-of-time swap-in (Pensieve method summary: ahead-of-time swapping and
 * pipelined data transfer that overlap data movement with computation).
 * pkv_swap_in_ahead starts a copy-engine transfer of host_buf
 * ([n][2][Hkv][B][D], the pkv_swap_in layout; pinned for the transfer to be
 * asynchronous) into a device staging buffer that the pool owns, on
 * `copy_stream`, and returns.  The transfer starts after the work queued on
 * `stream` before this call (for instance the swap-out that filled
 * host_buf), so it takes no SMs and overlaps whatever the caller queues next.
 * The blocks land in the pool at the start of the pool's next call that reads
 * or writes it (pkv_append, pkv_paged_attn, pkv_swap_out, pkv_swap_in,
 * another pkv_swap_in_ahead) or at pkv_swap_in_finish: that call's stream
 * waits for the transfer, and a kernel scatters the staged blocks into
 * block_ids.  Until then the pool's blocks keep their old contents, so calls
 * take effect in call order; read the storage from pkv_pool_kv_ptrs only
 * after pkv_swap_in_finish.
 * Layer pipelining: with one pool per model layer, issue every layer's
 * pkv_swap_in_ahead on one copy stream at the start of a step, then the
 * layers' attention in order on the compute stream; layer l then waits only
 * for its own blocks, and the transfers of later layers overlap the
 * attention of earlier ones.
 * The staging buffer grows (cudaMalloc, synchronising the device) when a call
 * moves more blocks than any earlier one on the pool; n * 2 * Hkv * B * D * 2
 * bytes.  host_buf must stay valid until the transfer has completed (a
 * stream or event synchronisation on copy_stream, or the landing call's
 * completion).  block_ids is a HOST array, copied by the call.
 * Errors: PKV_EINVAL (NULL pool, ids or buffer with n > 0; an id outside the
 * pool; nothing is started), PKV_ENOMEM (staging allocation), PKV_ECUDA.
 */
int pkv_swap_in_ahead(pkv_pool* pool, const int32_t* block_ids, int n, const void* host_buf, void* copy_stream,
                      void* stream);
int pkv_swap_in_finish(pkv_pool* pool, void* stream);

/*
 * Copy `bytes` bytes between device memory and host memory, asynchronously on
 * `stream`, by the copy engines (cudaMemcpyAsync): how a serving loop moves a
 * step's inputs in and its outputs out next to the library's calls.  Pinned
 * host memory (cudaHostAlloc / registered) makes the copy asynchronous; with
 * pageable memory the driver may serialise it with the host.  Any sizes and
 * alignments.  Errors: PKV_EINVAL for NULL pointers with bytes > 0, PKV_ECUDA
 * for a failed copy.
 */
int pkv_copy_to_device(void* dst, const void* host_src, size_t bytes, void* stream);
int pkv_copy_to_host(void* host_dst, const void* src, size_t bytes, void* stream);

/*
 * Two-tier block manager (host only, no GPU calls): which KV blocks of which
 * conversation live in the GPU pool (`gpu_blocks` physical blocks), in CPU
 * host slots (`cpu_blocks` slots of one [cpu_blocks][2][Hkv][16][D] pinned
 * buffer), or nowhere, and what each step must swap and recompute.  Pensieve
 * (abstract) evicts cached history by conversation activity and recompute
 * cost, at block granularity, and recomputes what was lost; the reading taken
 * here:
 *   - recompute cost of a token at position p = token_cost + p + 1 (fixed
 *     per-token work in units of one key's attention, plus attention over its
 *     p + 1 keys), so leading blocks are the cheapest to recompute;
 *   - a conversation's blocks are, by position, [dropped][CPU][GPU]: eviction
 *     moves an idle conversation's leading GPU block to the CPU tier (or drops
 *     it when there is no CPU tier), and a full CPU tier drops its leading
 *     block, so what must be recomputed is always a prefix [0, e);
 *   - the victim is the conversation not in the step whose leading block has
 *     the highest (steps since its last request) / (recompute cost); ties go
 *     to the lower id.
 * pkv_cache_step plans one step for n distinct conversations (conv_ids >= 0;
 * an unknown id starts a new, empty conversation) that each add new_tokens[r]
 * tokens, and fills:
 *   - block_tables [n][max_blocks]: the conversation's pool blocks in position
 *     order, -1 past ceil(ctx_lens[r] / 16);
 *   - ctx_lens [n]: tokens after the step;
 *   - recompute [n]: leading tokens [0, recompute[r]) to recompute this step
 *     (query positions [0, recompute) U [old length, ctx_lens)), whose blocks
 *     are fresh;
 *   - swap_out [num_swap_out][2] = (pool block, host slot) and
 *     swap_in [num_swap_in][2] = (host slot, pool block), each at most
 *     swap_cap pairs.
 * The caller runs every swap-out, then every swap-in, then appends the step's
 * tokens (recomputed and new): a block freed by a swap-out may be reused in
 * the same step.  Errors: PKV_EINVAL for bad arguments (a repeated id, a
 * conversation longer than max_blocks blocks, more swaps than swap_cap),
 * PKV_ENOMEM if the step's conversations cannot fit in the pool even after
 * evicting every other conversation; on an error the manager is unchanged.
 * pkv_cache_release forgets a conversation and frees its blocks and slots.
 */
typedef struct pkv_cache pkv_cache;
int pkv_cache_create(int gpu_blocks, int cpu_blocks, float token_cost, pkv_cache** out);
int pkv_cache_destroy(pkv_cache* cache);
int pkv_cache_step(pkv_cache* cache, const int32_t* conv_ids, const int32_t* new_tokens, int n,
                   int32_t* block_tables, int max_blocks, int32_t* ctx_lens, int32_t* recompute,
                   int32_t* swap_out, int* num_swap_out, int32_t* swap_in, int* num_swap_in, int swap_cap);
int pkv_cache_release(pkv_cache* cache, int conv);
int pkv_cache_free_blocks(const pkv_cache* cache, int* gpu_free, int* cpu_free);

/* Synchronise `stream`, read the device error word into *flags (may be NULL)
 * and clear it.  Returns PKV_EDEVICE if any bit was set (PKV_ETIMEOUT if the
 * timeout bit was), else PKV_OK. */
int pkv_check_device_errors(pkv_pool* pool, void* stream, unsigned* flags);

/* Test and diagnostic settings of a pool, for checking the failure path
 * without a GPU fault:
 *   PKV_DEBUG_WAIT_LIMIT_NS: wall-clock limit of every bounded wait in this
 *     pool's attention kernels (default 1 s; 1 us .. 60 s);
 *   PKV_DEBUG_WITHHOLD_COPY: 1 (2) = the first CTA of the split-KV
 *     (tensor-core) kernel never issues its first K copy, so that the wait for
 *     it runs out: the kernel records PKV_DEVERR_TIMEOUT, drains its copies,
 *     frees what it holds and returns, and that call's outputs are undefined;
 *     0 = off (default);
 *   PKV_DEBUG_FUSED_FORM: how pkv_append_paged_attn appends: 0 = chosen per
 *     batch (default), 1 = inside the attention launches whenever the pool
 *     allows it, 2 = the append kernel first.  Every form gives the same pool
 *     and the same O and LSE bits.
 * Errors: PKV_EINVAL for an unknown setting or a value out of range. */
#define PKV_DEBUG_WAIT_LIMIT_NS 1
#define PKV_DEBUG_WITHHOLD_COPY 2
#define PKV_DEBUG_FUSED_FORM 3
int pkv_debug_set(pkv_pool* pool, int what, int64_t value);

/* Kernel timing with CUDA events recorded around every launch on the launch
 * stream.  on: 0 off, 1 on, 2 on with the two attention kernels of a call run
 * one after the other on the caller's stream (instead of side by side), so
 * that each kernel's events bracket its own execution alone.  Enabling adds
 * one event pair per launch.  pkv_profile_read synchronises the recorded
 * events, adds their durations into *out and, if reset != 0, clears the
 * totals. */
int pkv_profile_enable(pkv_pool* pool, int on);
int pkv_profile_read(pkv_pool* pool, pkv_profile* out, int reset);

/* One planned work item, as reported by pkv_plan_inspect.  Rows of an item
 * are (token q_start + i, query head kv_head*G + j), i < q_count + q_count2,
 * j < G.  A tensor-core item holds two query tiles of at most 128 rows each:
 * q_count tokens, then q_count2 tokens (0 if there is one tile). */
typedef struct {
  int32_t kernel;    /* 1: split-KV (CUDA cores), 2: tensor-core tile pair */
  int32_t req;
  int32_t kv_head;
  int32_t q_start;
  int32_t q_count;
  int32_t kv_start;  /* key positions [kv_start, kv_end) */
  int32_t kv_end;
  int32_t part;      /* -1: writes O/LSE directly; else first partial row */
  int32_t q_count2;
  int32_t pos_max0;  /* query-position bounds of the first tile (the whole */
  int32_t pos_min0;  /* split-KV item) and of the second tile: exact with  */
  int32_t pos_max1;  /* host positions, else [0, ctx_len - 1]; an empty    */
  int32_t pos_min1;  /* tile has pos_max -1                                 */
} pkv_work_desc;

/* Plan a batch on the host only (no device needed) and copy out its work
 * items: the split-KV items first, then the tensor-core items.  At most
 * max_items are written; *num_items receives the total.  stats may be NULL;
 * its byte figures are those of a bf16 pool (pkv_last_plan_stats reports a
 * pool's own, FP8 included).  Used to test the planner; pkv_paged_attn plans
 * internally. */
int pkv_plan_inspect(int num_q_heads, int num_kv_heads, int head_dim, int num_sms, int num_reqs,
                     int num_tokens, const pkv_host_meta* host_meta, pkv_work_desc* items,
                     int max_items, int* num_items, pkv_plan_stats* stats);

/* Number of SMs the planner sizes the work split for (current device). */
int pkv_device_sm_count(int* sms);

/* Message of the last failed call on this thread ("" if none). */
const char* pkv_last_error(void);

/* Library version string. */
const char* pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */

// Host side of the C ABI declared in include/pkv.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

using namespace pkv;

namespace pkv {
int set_last_error(int code, const std::string& msg);
}

namespace {

thread_local std::string g_err;

int fail(int code, const std::string& msg) {
  g_err = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define PKV_CUDA(call, what)                 \
  do {                                       \
    cudaError_t e_ = (call);                 \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

struct ProfRec {
  int kernel;
  cudaEvent_t a, b;
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int pkv::set_last_error(int code, const std::string& msg) { return fail(code, msg); }

struct pkv_pool {
  int num_blocks = 0, block_size = 0, num_kv_heads = 0, head_dim = 0;
  int elem_bytes = 2;                 // 2: bf16; 1: fp8 e4m3 codes
  float k_scale = 1.f, v_scale = 1.f;
  void* k = nullptr;
  void* v = nullptr;
  bool owns = false;
  unsigned* d_err = nullptr;
  int device = 0, num_sms = 0;
  CUtensorMap tmap_k;  // 64-byte aligned by its type
  CUtensorMap tmap_v;
  CUtensorMap dmap_k;  // split-KV kernel's maps (FP8, D = 128); copies of tmap_* otherwise
  CUtensorMap dmap_v;
  std::mutex mu;
  Plan plan;
  // Pinned, double-buffered staging for work-list uploads (allocated at
  // creation; a work list larger than one slot goes through pageable memory).
  static constexpr size_t kStagingBytes = size_t(4) << 20;
  uint8_t* pinned[2] = {nullptr, nullptr};
  cudaEvent_t pinned_done[2] = {nullptr, nullptr};
  int pinned_slot = 0;
  std::vector<uint8_t> staging;
  // The tensor-core kernel runs on `side`, concurrently with the split-KV
  // kernel on the caller's stream (fork / join through the two events).
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  // Recorded after each attention call's kernels: the next call's work-list
  // upload waits for it before rewriting the work lists.
  cudaEvent_t ws_free = nullptr;
  // Device copy of the work lists, owned by the pool (kStagingBytes): the
  // upload into it runs on the pool's copy stream, ordered after the previous
  // call's kernels only, so it overlaps the caller's earlier work (the
  // append, the next step's input copies) and never queues behind it.  The
  // caller's workspace, whose memory may still be in use by work queued on
  // the caller's stream, is written only by kernels on that stream.
  // Two buffers, used by alternate calls (with the pinned staging slots): an
  // upload then waits only for the call before the previous one, long done,
  // so it is ready to run when it is submitted and does not queue on the
  // copy engine behind transfers submitted after it (a serving loop's next
  // inputs).
  uint8_t* d_wl[2] = {nullptr, nullptr};
  cudaEvent_t wl_free[2] = {nullptr, nullptr};
  cudaStream_t copy = nullptr;
  cudaEvent_t up_done = nullptr;
  // Ahead-of-time swap-in: the copy engines bring the blocks into a device
  // staging buffer on the caller's copy stream (swap_ready), and the pool's
  // next call scatters them into place on its own stream (staged_free).
  std::mutex swap_mu;
  void* swap_staging = nullptr;
  size_t swap_staging_bytes = 0;
  cudaEvent_t swap_ready = nullptr, swap_staged_free = nullptr, swap_after = nullptr;
  bool swap_pending = false;
  std::vector<int32_t> swap_ids;

  // Test and diagnostic settings (pkv_debug_set).
  uint64_t wait_ns = 1000000000ull;   // limit of every bounded wait in the kernels
  int withhold = 0;                   // see AttnArgs::withhold
  int fused_form = 0;                 // PKV_DEBUG_FUSED_FORM

  // profiling (prof_mode 2: the two attention kernels run one after the other)
  bool prof_on = false;
  int prof_mode = 0;
  std::vector<cudaEvent_t> ev_free;
  std::vector<ProfRec> pending;
  pkv_profile totals{};

  PoolView view() const {
    return PoolView{k, v, num_blocks, num_kv_heads, head_dim, d_err, elem_bytes, k_scale, v_scale};
  }
  // Bytes of one physical block of K (or V): all KV heads.
  size_t block_bytes() const { return static_cast<size_t>(num_kv_heads) * kBlockSize * head_dim * elem_bytes; }

  cudaEvent_t take_event() {
    if (ev_free.empty()) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
      return e;
    }
    cudaEvent_t e = ev_free.back();
    ev_free.pop_back();
    return e;
  }
};

namespace {

// Launch `fn` on `stream`, bracketed by profiling events when profiling is on.
template <class F>
int timed_launch(pkv_pool* pool, int kernel, void* stream, F&& fn) {
  cudaEvent_t a = nullptr, b = nullptr;
  if (pool->prof_on) {
    a = pool->take_event();
    b = pool->take_event();
    if (a && b) cudaEventRecord(a, static_cast<cudaStream_t>(stream));
  }
  const int rc = fn();
  if (a && b) {
    cudaEventRecord(b, static_cast<cudaStream_t>(stream));
    pool->pending.push_back({kernel, a, b});
  }
  return rc;
}

// swizzle: only for FP8 pools with D = 128 (the split-KV kernel's map, whose
// 128-byte rows land with 128-byte swizzle); the tensor-core kernel's FP8
// map lands unswizzled.
int make_tmap(CUtensorMap* map, void* base, int num_blocks, int hkv, int head_dim, bool fp8, bool swizzle = false) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return fail(PKV_ECUDA, "cuTensorMapEncodeTiled unavailable (driver too old?)");
  const cuuint64_t chunks = static_cast<cuuint64_t>(num_blocks) * hkv;   // (block, head) chunks of 16 x D
  if (chunks * kBlockSize >= (1ull << 31)) return fail(PKV_EUNSUPPORTED, "pool too large for 32-bit TMA coordinates");
  CUresult r;
  if (fp8 && swizzle) {
    // FP8 codes, D = 128: the chunk's 16 rows of 128 bytes land with
    // 128-byte swizzle (16-byte chunk x of row r at chunk x ^ (r % 8)).
    cuuint64_t dims[2] = {128, chunks * kBlockSize};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {128, static_cast<cuuint32_t>(kBlockSize)};
    cuuint32_t estr[2] = {1, 1};
    r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else if (fp8) {
    // FP8 codes: one (block, head) chunk per copy, 16 rows x D bytes, landing
    // unswizzled ([16 keys][D] bytes); the kernel widens them to f16.
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), chunks * kBlockSize};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(head_dim), static_cast<cuuint32_t>(kBlockSize)};
    cuuint32_t estr[2] = {1, 1};
    r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else if (head_dim == 128) {
    // One (block, head) chunk per copy, 16 rows x 256 bytes, landing as
    // [8-row group][64-column half][8 rows][128 bytes]: the 4-D view
    // (column within a half, row within a group, half, group) with strides
    // (2, 256, 128, 2048) bytes.  Each 1024-byte [8 rows][128 bytes] piece is
    // one 128-byte-swizzle atom of the MMA operand.
    cuuint64_t dims[4] = {64, 8, 2, chunks * 2};
    cuuint64_t strides[3] = {256, 128, 2048};
    cuuint32_t box[4] = {64, 8, 2, 2};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    // D = 64: a chunk is 16 rows of 128 bytes, already one column slab.
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), chunks * kBlockSize};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kBlockSize)};
    cuuint32_t estr[2] = {1, 1};
    r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) return fail(PKV_ECUDA, "cuTensorMapEncodeTiled failed: " + std::to_string(static_cast<int>(r)));
  return PKV_OK;
}

// Q viewed as [T][Hq][D] (bf16) for the tensor-core kernel's query tiles: a
// box of 64 columns x G heads (one KV head's group) x the tile's tokens lands
// as a [row][128 bytes] slab with 128-byte swizzle; tokens past T read zeros.
int make_q_tmap(CUtensorMap* map, const void* q, int num_tokens, int num_q_heads, int head_dim, int group,
                int* box_tokens) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return fail(PKV_ECUDA, "cuTensorMapEncodeTiled unavailable (driver too old?)");
  const int bt = std::min(kTcRows / group, num_tokens);
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(num_q_heads),
                        static_cast<cuuint64_t>(num_tokens)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2, static_cast<cuuint64_t>(num_q_heads) * head_dim * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(bt)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ECUDA, "cuTensorMapEncodeTiled (q) failed: " + std::to_string(static_cast<int>(r)));
  *box_tokens = bt;
  return PKV_OK;
}

// The fused call's new K (or V) rows [T][Hkv][D] (bf16) for the tensor-core
// kernel: a box of up to 8 tokens of one head lands as one 8-key group of a
// K/V stage ([half][8 rows][128 bytes], 128-byte swizzle, the pool boxes'
// layout); tokens past T read zeros.
int make_new_tmap(CUtensorMap* map, const void* base, int num_tokens, int hkv, int head_dim, int* box_tokens) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return fail(PKV_ECUDA, "cuTensorMapEncodeTiled unavailable (driver too old?)");
  const cuuint32_t bt = static_cast<cuuint32_t>(std::min(8, num_tokens));
  const cuuint64_t row = static_cast<cuuint64_t>(hkv) * head_dim * 2;   // bytes per token
  CUresult r;
  if (head_dim == 128) {
    // (column within a 64-column half, head, token, half)
    cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(hkv), static_cast<cuuint64_t>(num_tokens), 2};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(head_dim) * 2, row, 128};
    cuuint32_t box[4] = {64, 1, bt, 2};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(hkv), static_cast<cuuint64_t>(num_tokens)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2, row};
    cuuint32_t box[3] = {64, 1, bt};
    cuuint32_t estr[3] = {1, 1, 1};
    r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS)
    return fail(PKV_ECUDA, "cuTensorMapEncodeTiled (new rows) failed: " + std::to_string(static_cast<int>(r)));
  *box_tokens = static_cast<int>(bt);
  return PKV_OK;
}

}  // namespace

extern "C" {

const char* pkv_last_error(void) { return g_err.c_str(); }

const char* pkv_version(void) { return "pkv 0.1 (sm_103a)"; }

int pkv_device_sm_count(int* sms) {
  if (!sms) return fail(PKV_EINVAL, "sms is NULL");
  int dev = 0;
  PKV_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  PKV_CUDA(cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute");
  return PKV_OK;
}

int pkv_pool_create(const pkv_pool_desc* desc, pkv_pool** out) {
  if (!desc || !out) return fail(PKV_EINVAL, "desc/out is NULL");
  *out = nullptr;
  if (desc->num_blocks < 1 || desc->num_kv_heads < 1) return fail(PKV_EINVAL, "num_blocks and num_kv_heads must be >= 1");
  if (desc->block_size != kBlockSize) return fail(PKV_EUNSUPPORTED, "block_size must be 16");
  if (desc->head_dim != 64 && desc->head_dim != 128) return fail(PKV_EUNSUPPORTED, "head_dim must be 64 or 128");
  if (desc->dtype != PKV_DTYPE_BF16 && desc->dtype != PKV_DTYPE_FP8_E4M3)
    return fail(PKV_EUNSUPPORTED, "dtype must be PKV_DTYPE_BF16 or PKV_DTYPE_FP8_E4M3");
  const bool fp8 = desc->dtype == PKV_DTYPE_FP8_E4M3;
  if (fp8 && !(desc->k_scale > 0.f && desc->k_scale <= 3.4e38f && desc->v_scale > 0.f && desc->v_scale <= 3.4e38f))
    return fail(PKV_EINVAL, "fp8 pools need finite k_scale and v_scale > 0");
  if ((desc->k_storage == nullptr) != (desc->v_storage == nullptr))
    return fail(PKV_EINVAL, "give both k_storage and v_storage or neither");
  if (desc->k_storage && (!aligned16(desc->k_storage) || !aligned16(desc->v_storage)))
    return fail(PKV_EINVAL, "pool storage must be 16-byte aligned");
  auto* p = new pkv_pool();
  p->num_blocks = desc->num_blocks;
  p->block_size = desc->block_size;
  p->num_kv_heads = desc->num_kv_heads;
  p->head_dim = desc->head_dim;
  if (fp8) {
    p->elem_bytes = 1;
    p->k_scale = desc->k_scale;
    p->v_scale = desc->v_scale;
  }
  auto cleanup = [p](int rc) {
    if (p->owns) {
      cudaFree(p->k);
      cudaFree(p->v);
    }
    if (p->d_err) cudaFree(p->d_err);
    for (int i = 0; i < 2; ++i) {
      if (p->pinned[i]) cudaFreeHost(p->pinned[i]);
      if (p->pinned_done[i]) cudaEventDestroy(p->pinned_done[i]);
    }
    if (p->side) cudaStreamDestroy(p->side);
    if (p->fork) cudaEventDestroy(p->fork);
    if (p->join) cudaEventDestroy(p->join);
    if (p->ws_free) cudaEventDestroy(p->ws_free);
    for (int i = 0; i < 2; ++i) {
      if (p->d_wl[i]) cudaFree(p->d_wl[i]);
      if (p->wl_free[i]) cudaEventDestroy(p->wl_free[i]);
    }
    if (p->copy) cudaStreamDestroy(p->copy);
    if (p->up_done) cudaEventDestroy(p->up_done);
    delete p;
    return rc;
  };
  cudaError_t e = cudaGetDevice(&p->device);
  if (e != cudaSuccess) return cleanup(cuda_fail(e, "cudaGetDevice"));
  e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
  if (e != cudaSuccess) return cleanup(cuda_fail(e, "cudaDeviceGetAttribute"));
  const size_t bytes = static_cast<size_t>(desc->num_blocks) * p->block_bytes();
  if (desc->k_storage) {
    p->k = desc->k_storage;
    p->v = desc->v_storage;
  } else {
    p->owns = true;
    if (cudaMalloc(&p->k, bytes) != cudaSuccess) { p->k = nullptr; return cleanup(fail(PKV_ENOMEM, "cudaMalloc K pool")); }
    if (cudaMalloc(&p->v, bytes) != cudaSuccess) { p->v = nullptr; return cleanup(fail(PKV_ENOMEM, "cudaMalloc V pool")); }
    if (cudaMemset(p->k, 0, bytes) != cudaSuccess || cudaMemset(p->v, 0, bytes) != cudaSuccess)
      return cleanup(fail(PKV_ECUDA, "cudaMemset pool"));
  }
  if (cudaMalloc(&p->d_err, sizeof(unsigned)) != cudaSuccess) { p->d_err = nullptr; return cleanup(fail(PKV_ENOMEM, "cudaMalloc error word")); }
  if (cudaMemset(p->d_err, 0, sizeof(unsigned)) != cudaSuccess) return cleanup(fail(PKV_ECUDA, "cudaMemset error word"));
  for (int i = 0; i < 2; ++i) {
    if (cudaHostAlloc(reinterpret_cast<void**>(&p->pinned[i]), pkv_pool::kStagingBytes, cudaHostAllocDefault) !=
        cudaSuccess) {
      p->pinned[i] = nullptr;
      return cleanup(fail(PKV_ENOMEM, "cudaHostAlloc staging"));
    }
    if (cudaEventCreateWithFlags(&p->pinned_done[i], cudaEventDisableTiming) != cudaSuccess) {
      p->pinned_done[i] = nullptr;
      return cleanup(fail(PKV_ECUDA, "cudaEventCreate staging"));
    }
  }
  if (cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking) != cudaSuccess) {
    p->side = nullptr;
    return cleanup(fail(PKV_ECUDA, "cudaStreamCreate"));
  }
  if (cudaEventCreateWithFlags(&p->fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&p->join, cudaEventDisableTiming) != cudaSuccess)
    return cleanup(fail(PKV_ECUDA, "cudaEventCreate fork/join"));
  if (cudaEventCreateWithFlags(&p->ws_free, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&p->up_done, cudaEventDisableTiming) != cudaSuccess)
    return cleanup(fail(PKV_ECUDA, "cudaEventCreate upload"));
  if (cudaStreamCreateWithFlags(&p->copy, cudaStreamNonBlocking) != cudaSuccess) {
    p->copy = nullptr;
    return cleanup(fail(PKV_ECUDA, "cudaStreamCreate copy"));
  }
  for (int i = 0; i < 2; ++i) {
    if (cudaMalloc(&p->d_wl[i], pkv_pool::kStagingBytes) != cudaSuccess) {
      p->d_wl[i] = nullptr;
      return cleanup(fail(PKV_ENOMEM, "cudaMalloc work lists"));
    }
    if (cudaEventCreateWithFlags(&p->wl_free[i], cudaEventDisableTiming) != cudaSuccess) {
      p->wl_free[i] = nullptr;
      return cleanup(fail(PKV_ECUDA, "cudaEventCreate work lists"));
    }
  }

  // The attention kernels' block maps.
  {
    int rc = make_tmap(&p->tmap_k, p->k, p->num_blocks, p->num_kv_heads, p->head_dim, fp8);
    if (rc) return cleanup(rc);
    rc = make_tmap(&p->tmap_v, p->v, p->num_blocks, p->num_kv_heads, p->head_dim, fp8);
    if (rc) return cleanup(rc);
    p->dmap_k = p->tmap_k;
    p->dmap_v = p->tmap_v;
    if (fp8 && p->head_dim == 128) {
      rc = make_tmap(&p->dmap_k, p->k, p->num_blocks, p->num_kv_heads, 128, true, true);
      if (rc) return cleanup(rc);
      rc = make_tmap(&p->dmap_v, p->v, p->num_blocks, p->num_kv_heads, 128, true, true);
      if (rc) return cleanup(rc);
    }
  }
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cleanup(cuda_fail(e, "cudaDeviceSynchronize"));
  *out = p;
  return PKV_OK;
}

int pkv_pool_destroy(pkv_pool* pool) {
  if (!pool) return PKV_OK;
  cudaDeviceSynchronize();
  if (pool->owns) {
    cudaFree(pool->k);
    cudaFree(pool->v);
  }
  cudaFree(pool->d_err);
  for (int i = 0; i < 2; ++i) {
    if (pool->pinned[i]) cudaFreeHost(pool->pinned[i]);
    if (pool->pinned_done[i]) cudaEventDestroy(pool->pinned_done[i]);
  }
  cudaStreamDestroy(pool->side);
  cudaEventDestroy(pool->fork);
  cudaEventDestroy(pool->join);
  cudaEventDestroy(pool->ws_free);
  for (int i = 0; i < 2; ++i) {
    cudaFree(pool->d_wl[i]);
    cudaEventDestroy(pool->wl_free[i]);
  }
  cudaStreamDestroy(pool->copy);
  cudaEventDestroy(pool->up_done);
  if (pool->swap_staging) cudaFree(pool->swap_staging);
  for (cudaEvent_t e : {pool->swap_ready, pool->swap_staged_free, pool->swap_after})
    if (e) cudaEventDestroy(e);

  for (auto& r : pool->pending) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : pool->ev_free) cudaEventDestroy(e);
  delete pool;
  return PKV_OK;
}

int pkv_pool_kv_ptrs(const pkv_pool* pool, void** k, void** v) {
  if (!pool) return fail(PKV_EINVAL, "pool is NULL");
  if (k) *k = pool->k;
  if (v) *v = pool->v;
  return PKV_OK;
}

// Lands a pending ahead-of-time swap-in on `stream`: waits for its transfer,
// then scatters the staged blocks into the pool (every block at full HBM
// rate, on up to one CTA per SM).  Every call that reads or writes the pool
// starts with this, so the blocks are in place before the call's kernels.
static int finish_swap_in(pkv_pool* pool, void* stream) {
  std::lock_guard<std::mutex> lk(pool->swap_mu);
  if (!pool->swap_pending) return PKV_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PKV_CUDA(cudaStreamWaitEvent(s, pool->swap_ready, 0), "swap-in wait");
  const int rc = timed_launch(pool, 4, stream, [&] {
    return launch_swap(pool->view(), pool->k, pool->v, pool->swap_staging, pool->swap_ids.data(),
                       static_cast<int>(pool->swap_ids.size()), false, pool->num_sms, stream);
  });
  if (rc != cudaSuccess) return cuda_fail(static_cast<cudaError_t>(rc), "swap-in scatter launch");
  PKV_CUDA(cudaEventRecord(pool->swap_staged_free, s), "swap-in release");
  pool->swap_pending = false;
  return PKV_OK;
}

int pkv_append(pkv_pool* pool, const int32_t* block_tables, int max_blocks, int num_reqs, const int32_t* cu_q_lens,
               const int32_t* positions, const void* k_new, const void* v_new, int num_tokens, void* stream) {
  if (!pool) return fail(PKV_EINVAL, "pool is NULL");
  if (num_tokens < 0 || num_reqs < 0) return fail(PKV_EINVAL, "negative size");
  if (num_tokens == 0) return PKV_OK;
  if (num_reqs < 1 || max_blocks < 1) return fail(PKV_EINVAL, "num_reqs and max_blocks must be >= 1");
  if (!block_tables || !cu_q_lens || !positions || !k_new || !v_new) return fail(PKV_EINVAL, "NULL device pointer");
  if (!aligned16(k_new) || !aligned16(v_new)) return fail(PKV_EINVAL, "k_new / v_new must be 16-byte aligned");
  if (static_cast<int64_t>(max_blocks) * kBlockSize > (1ll << 31)) return fail(PKV_EINVAL, "max_blocks too large");
  int rc = finish_swap_in(pool, stream);
  if (rc) return rc;
  PoolView pv = pool->view();
  rc = timed_launch(pool, 0, stream, [&] {
    return launch_append(pv, pool->k, pool->v, block_tables, max_blocks, num_reqs, cu_q_lens, positions, k_new,
                         v_new, num_tokens, stream);
  });
  if (rc != cudaSuccess) return cuda_fail(static_cast<cudaError_t>(rc), "append launch");
  return PKV_OK;
}

// Plans the batch into pool->plan unless the cached plan was built from
// exactly the same parameters and host metadata (element-wise comparison).
static int plan_for(pkv_pool* pool, int num_q_heads, int num_reqs, int num_tokens, const pkv_host_meta* meta) {
  if (!meta) return fail(PKV_EINVAL, "host_meta is NULL");
  PlanParams pp{num_q_heads, pool->num_kv_heads, pool->head_dim, pool->num_sms, num_reqs, num_tokens,
                pool->elem_bytes};
  if (plan_matches(pool->plan, pp, *meta)) return PKV_OK;
  const char* err = "plan failed";
  int rc = build_plan(pp, *meta, &pool->plan, &err);
  if (rc) return fail(rc, err);
  return PKV_OK;
}

int pkv_paged_attn_workspace_size(pkv_pool* pool, int num_q_heads, int num_reqs, int num_tokens,
                                  const pkv_host_meta* host_meta, size_t* bytes) {
  if (!pool || !bytes) return fail(PKV_EINVAL, "pool/bytes is NULL");
  if (num_q_heads < 1 || num_q_heads % pool->num_kv_heads) return fail(PKV_EINVAL, "num_q_heads must be a multiple of num_kv_heads");
  if (num_reqs < 0 || num_tokens < 0) return fail(PKV_EINVAL, "negative size");
  std::lock_guard<std::mutex> lk(pool->mu);
  int rc = plan_for(pool, num_q_heads, num_reqs, num_tokens, host_meta);
  if (rc) return rc;
  *bytes = pool->plan.total;
  return PKV_OK;
}

}  // extern "C"

int pkv::paged_attn_call(pkv_pool* pool, const AttnCall& c) {
  if (!pool) return fail(PKV_EINVAL, "pool is NULL");
  if (c.num_tokens < 0 || c.num_reqs < 0) return fail(PKV_EINVAL, "negative size");
  if (c.num_tokens == 0) return PKV_OK;
  if (c.num_q_heads < 1 || c.num_q_heads % pool->num_kv_heads)
    return fail(PKV_EINVAL, "num_q_heads must be a multiple of num_kv_heads");
  if (c.num_q_heads / pool->num_kv_heads > kTcRows) return fail(PKV_EUNSUPPORTED, "group size above 128");
  if (c.num_reqs < 1 || c.max_blocks < 1) return fail(PKV_EINVAL, "num_reqs and max_blocks must be >= 1");
  if (!c.q || !c.q_positions || !c.block_tables || !c.ctx_lens || !c.cu_q_lens || !c.o)
    return fail(PKV_EINVAL, "NULL device pointer");
  if (!aligned16(c.q) || !aligned16(c.o)) return fail(PKV_EINVAL, "q and o must be 16-byte aligned");
  if (!(c.scale > 0.f)) return fail(PKV_EINVAL, "scale must be positive");
  const bool fused = c.k_new != nullptr || c.v_new != nullptr;
  if (fused) {
    if (!c.k_new || !c.v_new) return fail(PKV_EINVAL, "k_new and v_new are both required");
    if (!aligned16(c.k_new) || !aligned16(c.v_new)) return fail(PKV_EINVAL, "k_new / v_new must be 16-byte aligned");
    if (!c.host_meta || !c.host_meta->q_positions)
      return fail(PKV_EINVAL, "the fused call needs host copies of q_positions in host_meta");
    if (static_cast<int64_t>(c.num_tokens) * pool->num_kv_heads * (pool->head_dim / 8) >= (1ll << 31))
      return fail(PKV_EUNSUPPORTED, "too many new rows for one fused call");
  }
  int rc = finish_swap_in(pool, c.stream);
  if (rc) return rc;
  std::lock_guard<std::mutex> lk(pool->mu);
  rc = plan_for(pool, c.num_q_heads, c.num_reqs, c.num_tokens, c.host_meta);
  if (rc) return rc;
  const char* err = "";
  if ((rc = check_ctx_fits(*c.host_meta, c.num_reqs, c.max_blocks, &err))) return fail(rc, err);
  const Plan& pl = pool->plan;
  if (c.static_scratch) {
    if (pl.total > c.workspace_bytes)
      return fail(PKV_EINVAL, "pkv_paged_attn_static: this batch needs " + std::to_string(pl.total) +
                                  " bytes of scratch, above the static limit of " + std::to_string(c.workspace_bytes) +
                                  " bytes; use pkv_paged_attn with a caller workspace");
  } else if (!c.workspace || c.workspace_bytes < pl.total) {
    return fail(PKV_EINVAL, "workspace missing or smaller than pkv_paged_attn_workspace_size()");
  }
  if (reinterpret_cast<uintptr_t>(c.workspace) & 255u) return fail(PKV_EINVAL, "workspace must be 256-byte aligned");

  // Upload the work lists: through a pinned staging slot (asynchronous; the
  // slot is reused only after its previous upload has completed), or for an
  // unusually large list through pageable memory (free again on return).
  // Into the pool's own device buffer on the pool's copy stream (after the
  // pool's previous call, whatever its stream), or, for the static scratch
  // and for lists larger than that buffer, into the workspace on `stream`,
  // after the work the caller queued there (which may still use the
  // workspace's memory: a caching allocator hands out memory whose last
  // reader is queued on the same stream).
  const size_t meta_bytes = pl.off_part_o;
  cudaStream_t s = static_cast<cudaStream_t>(c.stream);
  uint8_t* ws = static_cast<uint8_t*>(c.workspace);
  const bool own = !c.static_scratch && meta_bytes <= pkv_pool::kStagingBytes;
  const int slot = pool->pinned_slot ^ 1;   // this call's staging slot and device buffer
  uint8_t* wl = own ? pool->d_wl[slot] : ws;   // where the work lists live on the device
  cudaStream_t up = own ? pool->copy : s;
  if (meta_bytes) {
    // The buffer's last reader: the call two back (own buffers), or the
    // previous call (the workspace).
    PKV_CUDA(cudaStreamWaitEvent(up, own ? pool->wl_free[slot] : pool->ws_free, 0), "upload wait");
    // Scratch shared with other pools: also wait for the last call that used it.
    if (c.scratch_free) PKV_CUDA(cudaStreamWaitEvent(up, static_cast<cudaEvent_t>(c.scratch_free), 0), "scratch wait");
    uint8_t* host = nullptr;
    const bool use_pinned = meta_bytes <= pkv_pool::kStagingBytes;
    if (use_pinned) {
      pool->pinned_slot ^= 1;
      PKV_CUDA(cudaEventSynchronize(pool->pinned_done[pool->pinned_slot]), "staging slot wait");
      host = pool->pinned[pool->pinned_slot];
    } else {
      pool->staging.assign(meta_bytes, 0);
      host = pool->staging.data();
    }
    if (!pl.decode.empty()) std::memcpy(host + pl.off_decode, pl.decode.data(), pl.decode.size() * sizeof(WorkItem));
    if (!pl.tc.empty()) {
      std::memcpy(host + pl.off_tc, pl.tc.data(), pl.tc.size() * sizeof(WorkItem));
      std::memset(host + pl.off_tc_next, 0, sizeof(int32_t));
    }
    if (!pl.merge.empty()) std::memcpy(host + pl.off_merge, pl.merge.data(), pl.merge.size() * sizeof(MergeItem));
    if (!pl.merge_dec.empty()) {
      std::memcpy(host + pl.off_merge_dec, pl.merge_dec.data(), pl.merge_dec.size() * sizeof(MergeItem));
      std::memset(host + pl.off_merge_cnt, 0, pl.merge_dec.size() * sizeof(int32_t));
    }
    if (!pl.runs.empty()) std::memcpy(host + pl.off_runs, pl.runs.data(), pl.runs.size() * sizeof(RunDesc));
    if (!pl.run_off.empty())
      std::memcpy(host + pl.off_run_off, pl.run_off.data(), pl.run_off.size() * sizeof(int32_t));
    PKV_CUDA(cudaMemcpyAsync(wl, host, meta_bytes, cudaMemcpyHostToDevice, up), "upload work list");
    if (use_pinned) PKV_CUDA(cudaEventRecord(pool->pinned_done[pool->pinned_slot], up), "staging slot record");
    if (own) {
      PKV_CUDA(cudaEventRecord(pool->up_done, up), "upload record");
      PKV_CUDA(cudaStreamWaitEvent(s, pool->up_done, 0), "upload join");
    }
  }

  AttnArgs a;
  a.pool = pool->view();
  a.q = c.q;
  a.num_q_heads = c.num_q_heads;
  a.group = c.num_q_heads / pool->num_kv_heads;
  a.q_positions = c.q_positions;
  a.block_tables = c.block_tables;
  a.max_blocks = c.max_blocks;
  a.ctx_lens = c.ctx_lens;
  a.scale_log2 = c.scale * 1.4426950408889634f;
  a.o = c.o;
  a.o_align32 = (reinterpret_cast<uintptr_t>(c.o) & 31u) == 0;
  a.lse = c.lse;
  a.part_o = reinterpret_cast<float*>(ws + pl.off_part_o);
  a.part_lse = reinterpret_cast<float*>(ws + pl.off_part_lse);
  a.merge_dec = reinterpret_cast<const MergeItem*>(wl + pl.off_merge_dec);
  a.merge_cnt = reinterpret_cast<int*>(wl + pl.off_merge_cnt);
  a.tc_next = reinterpret_cast<int*>(wl + pl.off_tc_next);
  a.tc_ctas = static_cast<int>(std::min<size_t>(pl.tc.size(), static_cast<size_t>(std::max(1, pool->num_sms))));
  a.q_box_tokens = 0;
  a.wait_ns = pool->wait_ns;
  a.withhold = pool->withhold;
  // A fused call over an FP8 pool with tensor-core items appends first, on
  // the caller's stream, and attends to the pool as a plain call does.  In
  // the fused form every tensor-core CTA that reads a new row would quantise
  // it again (correctly rounded divisions by the scale, as the append does,
  // so that the codes match the pool's) on its producer warp: measured about
  // seven times the attention's time on recompute-heavy batches.  The result
  // is the same either way.
  //
  // Any other fused call appends inside the split-KV launch (CTAs after its
  // work items) only when split-KV work dominates the batch.  Those CTAs take
  // about twice the stand-alone append kernel's time, which the split-KV
  // launch's own tail hides when its KV bytes are at least three times the
  // tensor-core kernel's; otherwise they hold SMs the tensor-core CTAs wait
  // for (measured: 13B mix 0.203 fused against 0.199 ms appending first, 70B
  // mix 0.564 against 0.561; decode 1.253 against 1.278 and long context
  // 0.338 against 0.344 the other way).  Either way the pool and the outputs
  // are the same bits.
  const bool in_kernel_ok = !(pool->elem_bytes == 1 && !pl.tc.empty());
  const bool in_kernel_pays =
      pl.tc.empty() || pl.stats.decode_kv_bytes >= 3 * pl.stats.tc_kv_bytes;
  const bool append_first =
      fused && (!in_kernel_ok || pool->fused_form == 2 || (pool->fused_form == 0 && !in_kernel_pays));
  const bool in_kernel = fused && !append_first;
  if (append_first) {
    PoolView pv = pool->view();
    rc = timed_launch(pool, 0, c.stream, [&] {
      return launch_append(pv, pool->k, pool->v, c.block_tables, c.max_blocks, c.num_reqs, c.cu_q_lens, c.q_positions,
                           c.k_new, c.v_new, c.num_tokens, c.stream);
    });
    if (rc != cudaSuccess) return cuda_fail(static_cast<cudaError_t>(rc), "append launch");
  }
  a.k_new = in_kernel ? c.k_new : nullptr;
  a.v_new = in_kernel ? c.v_new : nullptr;
  a.cu_q_lens = c.cu_q_lens;
  a.num_reqs = c.num_reqs;
  a.num_tokens = c.num_tokens;
  a.n_append_ctas = 0;
  a.kn_box_tokens = 0;
  a.runs = reinterpret_cast<const RunDesc*>(wl + pl.off_runs);
  a.run_off = reinterpret_cast<const int32_t*>(wl + pl.off_run_off);
  if (in_kernel) {
    // Append CTAs of the split-KV launch: about 8 chunks a thread.
    const int64_t chunks = static_cast<int64_t>(c.num_tokens) * pool->num_kv_heads * (pool->head_dim / 8);
    a.n_append_ctas = static_cast<int>(std::min<int64_t>(std::max<int64_t>(1, (chunks + 1023) / 1024),
                                                         static_cast<int64_t>(pool->num_sms) * 8));
  }
  CUtensorMap tmap_q, tmap_kn, tmap_vn;
  if (!pl.tc.empty()) {
    rc = make_q_tmap(&tmap_q, c.q, c.num_tokens, c.num_q_heads, pool->head_dim, a.group, &a.q_box_tokens);
    if (rc) return rc;
    if (in_kernel) {
      rc = make_new_tmap(&tmap_kn, c.k_new, c.num_tokens, pool->num_kv_heads, pool->head_dim, &a.kn_box_tokens);
      if (!rc) rc = make_new_tmap(&tmap_vn, c.v_new, c.num_tokens, pool->num_kv_heads, pool->head_dim, &a.kn_box_tokens);
      if (rc) return rc;
    } else {
      tmap_kn = pool->tmap_k;   // unused by a plain call; any valid map
      tmap_vn = pool->tmap_v;
    }
  }

  const WorkItem* d_dec = reinterpret_cast<const WorkItem*>(wl + pl.off_decode);
  const WorkItem* d_tc = reinterpret_cast<const WorkItem*>(wl + pl.off_tc);
  const MergeItem* d_merge = reinterpret_cast<const MergeItem*>(wl + pl.off_merge);
  // The two attention kernels are independent (disjoint outputs and workspace
  // regions): with both present, the split-KV kernel runs on the caller's
  // stream and the tensor-core kernel on the pool's side stream.  The caller's
  // stream is dispatched first (the side stream waits on the fork event), so
  // the split-KV CTAs (three per SM) take the SMs and tensor-core CTAs (one SM
  // each) fill them as the split-KV work drains; that order measured as fast
  // as or faster than the reverse on every mixed workload.  In the serialised
  // profiling mode both run on the caller's stream, one after the other, so
  // that each kernel's timing events bracket its own execution only.
  // A fused call always launches the split-KV kernel: its append CTAs write
  // the new rows into the pool.
  const bool dec_launch = !pl.decode.empty() || a.n_append_ctas > 0;
  const bool fork = !pl.tc.empty() && dec_launch && pool->prof_mode != 2;
  void* dec_stream = c.stream;
  void* tc_stream = c.stream;
  if (fork) {
    PKV_CUDA(cudaEventRecord(pool->fork, s), "fork record");
    PKV_CUDA(cudaStreamWaitEvent(pool->side, pool->fork, 0), "fork wait");
    tc_stream = pool->side;
  }
  if (dec_launch) {
    rc = timed_launch(pool, 1, dec_stream,
                      [&] { return launch_decode(a, &pool->dmap_k, &pool->dmap_v, d_dec, static_cast<int>(pl.decode.size()),
                                           dec_stream); });
    if (rc != cudaSuccess) return cuda_fail(static_cast<cudaError_t>(rc), "split-KV attention launch");
  }
  if (!pl.tc.empty()) {
    rc = timed_launch(pool, 2, tc_stream, [&] {
      return launch_tc(a, &pool->tmap_k, &pool->tmap_v, &tmap_q, &tmap_kn, &tmap_vn, d_tc,
                       static_cast<int>(pl.tc.size()), tc_stream);
    });
    if (rc != cudaSuccess) return cuda_fail(static_cast<cudaError_t>(rc), "tensor-core attention launch");
  }
  if (fork) {
    PKV_CUDA(cudaEventRecord(pool->join, pool->side), "join record");
    PKV_CUDA(cudaStreamWaitEvent(s, pool->join, 0), "join wait");
  }
  if (!pl.merge.empty()) {
    rc = timed_launch(pool, 3, c.stream,
                      [&] { return launch_merge(a, d_merge, static_cast<int>(pl.merge.size()), c.stream); });
    if (rc != cudaSuccess) return cuda_fail(static_cast<cudaError_t>(rc), "merge launch");
  }
  // The next calls' uploads may overwrite the work lists once these kernels are done.
  PKV_CUDA(cudaEventRecord(pool->ws_free, s), "workspace release");
  if (own) PKV_CUDA(cudaEventRecord(pool->wl_free[slot], s), "work-list release");
  if (c.scratch_free) PKV_CUDA(cudaEventRecord(static_cast<cudaEvent_t>(c.scratch_free), s), "scratch release");
  return PKV_OK;
}

extern "C" {

int pkv_paged_attn(pkv_pool* pool, const void* q, int num_q_heads, const int32_t* q_positions,
                   const int32_t* block_tables, int max_blocks, const int32_t* ctx_lens, const int32_t* cu_q_lens,
                   int num_reqs, int num_tokens, const pkv_host_meta* host_meta, float scale, void* o, float* lse,
                   void* workspace, size_t workspace_bytes, void* stream) {
  AttnCall c;
  c.q = q;
  c.num_q_heads = num_q_heads;
  c.q_positions = q_positions;
  c.block_tables = block_tables;
  c.max_blocks = max_blocks;
  c.ctx_lens = ctx_lens;
  c.cu_q_lens = cu_q_lens;
  c.num_reqs = num_reqs;
  c.num_tokens = num_tokens;
  c.host_meta = host_meta;
  c.scale = scale;
  c.o = o;
  c.lse = lse;
  c.workspace = workspace;
  c.workspace_bytes = workspace_bytes;
  c.stream = stream;
  return paged_attn_call(pool, c);
}

int pkv_append_paged_attn(pkv_pool* pool, const void* q, int num_q_heads, const int32_t* q_positions,
                          const int32_t* block_tables, int max_blocks, const int32_t* ctx_lens,
                          const int32_t* cu_q_lens, int num_reqs, int num_tokens, const pkv_host_meta* host_meta,
                          const void* k_new, const void* v_new, float scale, void* o, float* lse, void* workspace,
                          size_t workspace_bytes, void* stream) {
  AttnCall c;
  c.q = q;
  c.num_q_heads = num_q_heads;
  c.q_positions = q_positions;
  c.block_tables = block_tables;
  c.max_blocks = max_blocks;
  c.ctx_lens = ctx_lens;
  c.cu_q_lens = cu_q_lens;
  c.num_reqs = num_reqs;
  c.num_tokens = num_tokens;
  c.host_meta = host_meta;
  c.scale = scale;
  c.o = o;
  c.lse = lse;
  c.workspace = workspace;
  c.workspace_bytes = workspace_bytes;
  c.stream = stream;
  c.k_new = k_new;
  c.v_new = v_new;
  if (!k_new || !v_new) return fail(PKV_EINVAL, "k_new and v_new are both required");
  return paged_attn_call(pool, c);
}

int pkv_plan_inspect(int num_q_heads, int num_kv_heads, int head_dim, int num_sms, int num_reqs, int num_tokens,
                     const pkv_host_meta* host_meta, pkv_work_desc* items, int max_items, int* num_items,
                     pkv_plan_stats* stats) {
  if (!host_meta || !num_items) return fail(PKV_EINVAL, "host_meta/num_items is NULL");
  if (head_dim != 64 && head_dim != 128) return fail(PKV_EUNSUPPORTED, "head_dim must be 64 or 128");
  Plan plan;
  const char* err = "plan failed";
  PlanParams pp{num_q_heads, num_kv_heads, head_dim, num_sms, num_reqs, num_tokens};
  const int rc = build_plan(pp, *host_meta, &plan, &err);
  if (rc) return fail(rc, err);
  const int total = static_cast<int>(plan.decode.size() + plan.tc.size());
  *num_items = total;
  int k = 0;
  for (int which = 0; which < 2; ++which)
    for (const WorkItem& w : which == 0 ? plan.decode : plan.tc) {
      if (items && k < max_items)
        items[k] = pkv_work_desc{which + 1,     w.req,          w.kv_head,      w.q_start,
                                 w.q_count,     w.kv_start,     w.kv_end,       w.part,
                                 w.q_count2,    w.pos_max[0],   w.pos_min[0],   w.pos_max[1],
                                 w.pos_min[1]};
      ++k;
    }
  if (stats) *stats = plan.stats;
  return PKV_OK;
}

int pkv_last_plan_stats(const pkv_pool* pool, pkv_plan_stats* out) {
  if (!pool || !out) return fail(PKV_EINVAL, "pool/out is NULL");
  if (!pool->plan.valid) return fail(PKV_EINVAL, "no plan built yet");
  *out = pool->plan.stats;
  out->plans_built = pool->plan.builds;
  return PKV_OK;
}

static int swap_impl(pkv_pool* pool, const int32_t* ids, int n, void* host, bool out, void* stream) {
  if (!pool) return fail(PKV_EINVAL, "pool is NULL");
  if (n < 0) return fail(PKV_EINVAL, "negative count");
  if (n == 0) return PKV_OK;
  if (!ids || !host) return fail(PKV_EINVAL, "NULL block_ids or host buffer");
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= pool->num_blocks) return fail(PKV_EINVAL, "block id outside the pool");
  const int frc = finish_swap_in(pool, stream);
  if (frc) return frc;
  const size_t blk = pool->block_bytes();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Pinned (page-locked, device-mapped) host memory: one kernel moves every block.
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, host) == cudaSuccess && attr.type == cudaMemoryTypeHost &&
      attr.devicePointer != nullptr && (reinterpret_cast<uintptr_t>(attr.devicePointer) & 15u) == 0) {
    const int rc = timed_launch(pool, 4, stream, [&] {
      return launch_swap(pool->view(), pool->k, pool->v, attr.devicePointer, ids, n, out, 0, stream);
    });
    if (rc != cudaSuccess) return cuda_fail(static_cast<cudaError_t>(rc), "swap kernel launch");
    return PKV_OK;
  }
  cudaGetLastError();   // clear a failed attribute query on pageable memory
  // Pageable memory: DMA copies, one 2-D copy per run of consecutive block ids and pool.
  uint8_t* h = static_cast<uint8_t*>(host);
  int i = 0;
  while (i < n) {
    int j = i + 1;
    while (j < n && ids[j] == ids[j - 1] + 1) ++j;   // run of consecutive physical blocks
    const size_t run = static_cast<size_t>(j - i);
    for (int kv = 0; kv < 2; ++kv) {
      uint8_t* dev = static_cast<uint8_t*>(kv == 0 ? pool->k : pool->v) + static_cast<size_t>(ids[i]) * blk;
      uint8_t* hp = h + (static_cast<size_t>(i) * 2 + kv) * blk;
      cudaError_t e = out ? cudaMemcpy2DAsync(hp, 2 * blk, dev, blk, blk, run, cudaMemcpyDeviceToHost, s)
                          : cudaMemcpy2DAsync(dev, blk, hp, 2 * blk, blk, run, cudaMemcpyHostToDevice, s);
      if (e != cudaSuccess) return cuda_fail(e, out ? "swap out copy" : "swap in copy");
    }
    i = j;
  }
  return PKV_OK;
}

int pkv_swap_out(pkv_pool* pool, const int32_t* block_ids, int n, void* host_buf, void* stream) {
  return swap_impl(pool, block_ids, n, host_buf, true, stream);
}

int pkv_swap_in(pkv_pool* pool, const int32_t* block_ids, int n, const void* host_buf, void* stream) {
  return swap_impl(pool, block_ids, n, const_cast<void*>(host_buf), false, stream);
}

int pkv_swap_in_ahead(pkv_pool* pool, const int32_t* block_ids, int n, const void* host_buf, void* copy_stream,
                      void* stream) {
  if (!pool) return fail(PKV_EINVAL, "pool is NULL");
  if (n < 0) return fail(PKV_EINVAL, "negative count");
  if (n == 0) return PKV_OK;
  if (!block_ids || !host_buf) return fail(PKV_EINVAL, "NULL block_ids or host buffer");
  for (int i = 0; i < n; ++i)
    if (block_ids[i] < 0 || block_ids[i] >= pool->num_blocks) return fail(PKV_EINVAL, "block id outside the pool");
  // An earlier swap-in that has not landed yet lands first, on `stream`.
  int rc = finish_swap_in(pool, stream);
  if (rc) return rc;
  std::lock_guard<std::mutex> lk(pool->swap_mu);
  if (!pool->swap_ready) {
    for (cudaEvent_t* e : {&pool->swap_ready, &pool->swap_staged_free, &pool->swap_after})
      if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) {
        *e = nullptr;
        return fail(PKV_ECUDA, "cudaEventCreate swap-in");
      }
  }
  const size_t bytes = static_cast<size_t>(n) * 2 * pool->block_bytes();
  if (bytes > pool->swap_staging_bytes) {
    if (pool->swap_staging) {
      // the last scatter may still be reading the old buffer
      PKV_CUDA(cudaEventSynchronize(pool->swap_staged_free), "swap-in staging release");
      PKV_CUDA(cudaFree(pool->swap_staging), "cudaFree swap-in staging");
      pool->swap_staging = nullptr;
      pool->swap_staging_bytes = 0;
    }
    if (cudaMalloc(&pool->swap_staging, bytes) != cudaSuccess) {
      pool->swap_staging = nullptr;
      cudaGetLastError();
      return fail(PKV_ENOMEM, "cudaMalloc swap-in staging");
    }
    pool->swap_staging_bytes = bytes;
  }
  cudaStream_t cs = static_cast<cudaStream_t>(copy_stream);
  // The transfer follows the work queued on `stream` (a swap-out that fills
  // host_buf, the last reads of the blocks) and the previous scatter.
  PKV_CUDA(cudaEventRecord(pool->swap_after, static_cast<cudaStream_t>(stream)), "swap-in order");
  PKV_CUDA(cudaStreamWaitEvent(cs, pool->swap_after, 0), "swap-in order");
  PKV_CUDA(cudaStreamWaitEvent(cs, pool->swap_staged_free, 0), "swap-in staging wait");
  PKV_CUDA(cudaMemcpyAsync(pool->swap_staging, host_buf, bytes, cudaMemcpyHostToDevice, cs), "swap-in transfer");
  PKV_CUDA(cudaEventRecord(pool->swap_ready, cs), "swap-in record");
  pool->swap_ids.assign(block_ids, block_ids + n);
  pool->swap_pending = true;
  return PKV_OK;
}

int pkv_swap_in_finish(pkv_pool* pool, void* stream) {
  if (!pool) return fail(PKV_EINVAL, "pool is NULL");
  return finish_swap_in(pool, stream);
}

static int host_copy(void* dst, const void* src, size_t bytes, bool to_host, void* stream) {
  if (bytes == 0) return PKV_OK;
  if (!dst || !src) return fail(PKV_EINVAL, "NULL pointer");
  PKV_CUDA(cudaMemcpyAsync(dst, src, bytes, to_host ? cudaMemcpyDeviceToHost : cudaMemcpyHostToDevice,
                           static_cast<cudaStream_t>(stream)),
           to_host ? "copy to host" : "copy to device");
  return PKV_OK;
}

int pkv_copy_to_device(void* dst, const void* host_src, size_t bytes, void* stream) {
  return host_copy(dst, host_src, bytes, false, stream);
}

int pkv_copy_to_host(void* host_dst, const void* src, size_t bytes, void* stream) {
  return host_copy(host_dst, src, bytes, true, stream);
}

int pkv_check_device_errors(pkv_pool* pool, void* stream, unsigned* flags) {
  if (!pool) return fail(PKV_EINVAL, "pool is NULL");
  PKV_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "cudaStreamSynchronize");
  unsigned v = 0;
  PKV_CUDA(cudaMemcpy(&v, pool->d_err, sizeof v, cudaMemcpyDeviceToHost), "read error word");
  PKV_CUDA(cudaMemset(pool->d_err, 0, sizeof v), "clear error word");
  if (flags) *flags = v;
  if (v & PKV_DEVERR_TIMEOUT) return fail(PKV_ETIMEOUT, "a bounded wait inside a kernel ran out");
  if (v) return fail(PKV_EDEVICE, "kernels skipped invalid block ids or positions");
  return PKV_OK;
}

int pkv_profile_enable(pkv_pool* pool, int on) {
  if (!pool) return fail(PKV_EINVAL, "pool is NULL");
  if (on < 0 || on > 2) return fail(PKV_EINVAL, "profile mode must be 0, 1 or 2");
  pool->prof_on = on != 0;
  pool->prof_mode = on;
  return PKV_OK;
}

int pkv_debug_set(pkv_pool* pool, int what, int64_t value) {
  if (!pool) return fail(PKV_EINVAL, "pool is NULL");
  std::lock_guard<std::mutex> lk(pool->mu);
  switch (what) {
    case PKV_DEBUG_WAIT_LIMIT_NS:
      if (value < 1000 || value > 60ll * 1000000000ll) return fail(PKV_EINVAL, "wait limit must be 1 us .. 60 s");
      pool->wait_ns = static_cast<uint64_t>(value);
      return PKV_OK;
    case PKV_DEBUG_WITHHOLD_COPY:
      if (value < 0 || value > 2) return fail(PKV_EINVAL, "withhold must be 0, 1 or 2");
      pool->withhold = static_cast<int>(value);
      return PKV_OK;
    case PKV_DEBUG_FUSED_FORM:
      if (value < 0 || value > 2) return fail(PKV_EINVAL, "fused form must be 0, 1 or 2");
      pool->fused_form = static_cast<int>(value);
      return PKV_OK;
    default:
      return fail(PKV_EINVAL, "unknown debug setting");
  }
}

int pkv_profile_read(pkv_pool* pool, pkv_profile* out, int reset) {
  if (!pool) return fail(PKV_EINVAL, "pool is NULL");
  for (auto& r : pool->pending) {
    PKV_CUDA(cudaEventSynchronize(r.b), "cudaEventSynchronize");
    float ms = 0.f;
    PKV_CUDA(cudaEventElapsedTime(&ms, r.a, r.b), "cudaEventElapsedTime");
    pool->totals.launches[r.kernel] += 1;
    pool->totals.total_ms[r.kernel] += ms;
    pool->ev_free.push_back(r.a);
    pool->ev_free.push_back(r.b);
  }
  pool->pending.clear();
  if (out) *out = pool->totals;
  if (reset) pool->totals = pkv_profile{};
  return PKV_OK;
}

}  // extern "C"

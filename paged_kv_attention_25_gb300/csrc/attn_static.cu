// Paged attention without any device allocation.
//
// Some callers cannot call cudaMalloc: a serving process whose device memory
// is entirely carved up by another framework's caching allocator, code that
// runs inside an allocator or stream callback where allocating CUDA calls are
// not allowed, or a latency-critical loop where cudaMalloc's implicit
// device-wide synchronisation would stall every other stream.  They cannot
// provide pkv_paged_attn's workspace either, so this entry point keeps the
// work lists and split-KV partials in one static device array instead.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "internal.h"

namespace {

// The scratch of pkv_paged_attn_static.  Every GPU that loads this library
// holds these PKV_STATIC_SCRATCH_BYTES until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[PKV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_dev_addr[kMaxDevices] = {};
// Recorded after each call's kernels; the next call's upload into the array
// waits for it, so calls on any pools and streams follow one another.
cudaEvent_t g_scratch_free[kMaxDevices] = {};

}  // namespace

extern "C" int pkv_paged_attn_static(pkv_pool* pool, const void* q, int num_q_heads, const int32_t* q_positions,
                                     const int32_t* block_tables, int max_blocks, const int32_t* ctx_lens,
                                     const int32_t* cu_q_lens, int num_reqs, int num_tokens,
                                     const pkv_host_meta* host_meta, float scale, void* o, float* lse,
                                     void* stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pkv::set_last_error(PKV_ECUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return pkv::set_last_error(PKV_EUNSUPPORTED, "device index above 63");
  // Held for the whole call: the array's upload, kernels and release event of
  // one call are enqueued before the next call's.
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_dev_addr[dev] == nullptr) {
    // Host code cannot use g_static_scratch as an address: it names a
    // host-side stand-in.  Look up the array's address on this device once,
    // with the device current.
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr)
      return pkv::set_last_error(PKV_ECUDA, std::string("cudaGetSymbolAddress(static scratch): ") +
                                                cudaGetErrorString(e));
    cudaEvent_t ev = nullptr;
    e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess)
      return pkv::set_last_error(PKV_ECUDA, std::string("cudaEventCreate(static scratch): ") + cudaGetErrorString(e));
    g_scratch_free[dev] = ev;
    g_scratch_dev_addr[dev] = p;
  }
  // One plan serves the size check and the call: the work lists are rewritten
  // and every partial row is written by this call before it is read, so
  // nothing left by an earlier call needs clearing.
  pkv::AttnCall c;
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
  c.workspace = g_scratch_dev_addr[dev];
  c.workspace_bytes = PKV_STATIC_SCRATCH_BYTES;
  c.stream = stream;
  c.static_scratch = true;
  c.scratch_free = g_scratch_free[dev];
  return pkv::paged_attn_call(pool, c);
}

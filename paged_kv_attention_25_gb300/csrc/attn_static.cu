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
  void* scratch = nullptr;
  {
    // Host code cannot use g_static_scratch as an address: it names a host-side
    // stand-in.  Look up the array's address on this device once, with the
    // device current.
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_dev_addr[dev] == nullptr) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_static_scratch);
      if (e != cudaSuccess || p == nullptr)
        return pkv::set_last_error(PKV_ECUDA, std::string("cudaGetSymbolAddress(static scratch): ") +
                                                  cudaGetErrorString(e));
      g_scratch_dev_addr[dev] = p;
    }
    scratch = g_scratch_dev_addr[dev];
  }
  if (num_tokens > 0) {
    size_t need = 0;
    const int rc = pkv_paged_attn_workspace_size(pool, num_q_heads, num_reqs, num_tokens, host_meta, &need);
    if (rc != PKV_OK) return rc;
    if (need > PKV_STATIC_SCRATCH_BYTES)
      return pkv::set_last_error(
          PKV_EINVAL, "pkv_paged_attn_static: this batch needs " + std::to_string(need) +
                          " bytes of scratch, above the static limit of " +
                          std::to_string(static_cast<size_t>(PKV_STATIC_SCRATCH_BYTES)) +
                          " bytes; use pkv_paged_attn with a caller workspace");
  }
  // The work lists are rewritten and every partial row is written by this
  // call before it is read, so nothing left by an earlier call needs clearing.
  return pkv_paged_attn(pool, q, num_q_heads, q_positions, block_tables, max_blocks, ctx_lens, cu_q_lens, num_reqs,
                        num_tokens, host_meta, scale, o, lse, scratch, PKV_STATIC_SCRATCH_BYTES, stream);
}

// Block swap between the GPU pool and the CPU cache tier (Pensieve abstract:
// multi-tier caching that keeps conversation state in GPU and CPU memory).
//
// A pinned host buffer is mapped into the device address space, so one kernel
// moves every block of the request directly between HBM and host memory over
// the CPU-GPU link: reads and writes are 16-byte, coalesced, and there is no
// per-block copy set-up.  The block ids travel as a kernel parameter, so the
// call uploads and allocates nothing.
#include <cuda_runtime.h>

#include "internal.h"

namespace pkv {
namespace {

__global__ void __launch_bounds__(256) swap_kernel(uint4* __restrict__ kpool, uint4* __restrict__ vpool,
                                                   uint4* __restrict__ host, const SwapIds ids, int n,
                                                   int64_t blk_chunks, int to_host) {
  const int64_t per = 2 * blk_chunks;              // K then V of one block
  const int64_t total = static_cast<int64_t>(n) * per;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int b = static_cast<int>(i / per);
    const int64_t rem = i % per;
    const int kv = rem >= blk_chunks;
    const int64_t c = kv ? rem - blk_chunks : rem;
    uint4* pool = kv ? vpool : kpool;
    const int64_t p = static_cast<int64_t>(ids.id[b]) * blk_chunks + c;
    if (to_host) host[i] = pool[p];
    else pool[p] = host[i];
  }
}

}  // namespace

int launch_swap(const PoolView& pool, void* kp, void* vp, void* host_dev, const int32_t* ids, int n, bool to_host,
                int num_sms, void* stream) {
  const int64_t blk_chunks = static_cast<int64_t>(pool.num_kv_heads) * kBlockSize * pool.head_dim / 8;
  for (int i = 0; i < n; i += kSwapIdsPerLaunch) {
    const int m = n - i < kSwapIdsPerLaunch ? n - i : kSwapIdsPerLaunch;
    SwapIds s;
    for (int j = 0; j < m; ++j) s.id[j] = ids[i + j];
    const int64_t total = static_cast<int64_t>(m) * 2 * blk_chunks;
    const int64_t want = (total + 255) / 256;
    const int grid = static_cast<int>(want < int64_t(num_sms) * 8 ? want : int64_t(num_sms) * 8);
    uint4* h = static_cast<uint4*>(host_dev) + static_cast<int64_t>(i) * 2 * blk_chunks;
    swap_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4*>(kp), static_cast<uint4*>(vp), h, s, m, blk_chunks, to_host ? 1 : 0);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace pkv

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

// Each thread moves kUnroll 16-byte chunks per round (all loads, then all
// stores) so that enough requests are in flight to cover the link's latency.
constexpr int kSwapThreads = 512;
constexpr int kUnroll = 4;
// The CPU-GPU link saturates (about 190 GB/s each way on GB300) with 16 CTAs
// of 512 threads; more CTAs only take SMs away from attention kernels that
// run next to the swap.
constexpr int kSwapCtas = 16;

__global__ void __launch_bounds__(kSwapThreads) swap_kernel(uint4* __restrict__ kpool, uint4* __restrict__ vpool,
                                                            uint4* __restrict__ host, const SwapIds ids, int n,
                                                            int64_t blk_chunks, int to_host) {
  const int64_t per = 2 * blk_chunks;              // K then V of one block
  const int64_t total = static_cast<int64_t>(n) * per;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  // Host-side chunk i <-> pool chunk of (block i / per, K or V, offset).
  auto pool_ptr = [&](int64_t i) -> uint4* {
    const int b = static_cast<int>(i / per);
    const int64_t rem = i % per;
    const int kv = rem >= blk_chunks;
    const int64_t c = kv ? rem - blk_chunks : rem;
    return (kv ? vpool : kpool) + static_cast<int64_t>(ids.id[b]) * blk_chunks + c;
  };
  int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  for (; i + (kUnroll - 1) * stride < total; i += kUnroll * stride) {
    uint4 v[kUnroll];
    if (to_host) {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) v[u] = *pool_ptr(i + u * stride);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) host[i + u * stride] = v[u];
    } else {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) v[u] = host[i + u * stride];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) *pool_ptr(i + u * stride) = v[u];
    }
  }
  for (; i < total; i += stride) {
    if (to_host) host[i] = *pool_ptr(i);
    else *pool_ptr(i) = host[i];
  }
}

}  // namespace

int launch_swap(const PoolView& pool, void* kp, void* vp, void* host_dev, const int32_t* ids, int n, bool to_host,
                int num_sms, void* stream) {
  (void)num_sms;
  const int64_t blk_chunks = static_cast<int64_t>(pool.num_kv_heads) * kBlockSize * pool.head_dim / 8;
  for (int i = 0; i < n; i += kSwapIdsPerLaunch) {
    const int m = n - i < kSwapIdsPerLaunch ? n - i : kSwapIdsPerLaunch;
    SwapIds s;
    for (int j = 0; j < m; ++j) s.id[j] = ids[i + j];
    const int64_t total = static_cast<int64_t>(m) * 2 * blk_chunks;
    const int64_t want = (total + kSwapThreads * kUnroll - 1) / (kSwapThreads * kUnroll);
    const int grid = static_cast<int>(want < kSwapCtas ? want : kSwapCtas);
    uint4* h = static_cast<uint4*>(host_dev) + static_cast<int64_t>(i) * 2 * blk_chunks;
    swap_kernel<<<grid, kSwapThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4*>(kp), static_cast<uint4*>(vp), h, s, m, blk_chunks, to_host ? 1 : 0);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace pkv

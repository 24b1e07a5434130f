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
// stores): 64 KB a CTA in flight, which covers HBM latency while the
// attention kernels load HBM beside a swap (4 chunks a thread measured about
// half the link rate there).  A round past a block's end is predicated rather
// than finished one dependent chunk at a time.
constexpr int kSwapThreads = 256;
constexpr int kUnroll = 16;
// CTAs of 256 threads that saturate the CPU-GPU link on GB300 (measured):
// writes to host memory reach about 187 GB/s with 8, reads from it about
// 199 GB/s with 24.  More CTAs only take SMs from the attention kernels that
// run next to a swap.
constexpr int kSwapCtasOut = 8;
constexpr int kSwapCtasIn = 24;

__global__ void __launch_bounds__(kSwapThreads) swap_kernel(uint4* __restrict__ kpool, uint4* __restrict__ vpool,
                                                            uint4* __restrict__ host, const SwapIds ids, int n,
                                                            int blk_chunks, int to_host) {
  // CTA c takes blocks c, c + gridDim.x, ...; a block is two contiguous runs
  // (its K, then its V) of blk_chunks 16-byte chunks on both sides.
  for (int b = blockIdx.x; b < n; b += gridDim.x) {
    const int64_t pool_off = static_cast<int64_t>(ids.id[b]) * blk_chunks;
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
      uint4* p = (kv ? vpool : kpool) + pool_off;
      uint4* h = host + (2 * static_cast<int64_t>(b) + kv) * blk_chunks;
      const uint4* src = to_host ? p : h;
      uint4* dst = to_host ? h : p;
      for (int c0 = threadIdx.x; c0 < blk_chunks; c0 += kUnroll * kSwapThreads) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (c0 + u * kSwapThreads < blk_chunks) v[u] = src[c0 + u * kSwapThreads];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (c0 + u * kSwapThreads < blk_chunks) dst[c0 + u * kSwapThreads] = v[u];
      }
    }
  }
}

}  // namespace

int launch_swap(const PoolView& pool, void* kp, void* vp, void* host_dev, const int32_t* ids, int n, bool to_host,
                int max_ctas, void* stream) {
  const int blk_chunks = pool.num_kv_heads * kBlockSize * pool.head_dim * pool.elem_bytes / 16;
  for (int i = 0; i < n; i += kSwapIdsPerLaunch) {
    const int m = n - i < kSwapIdsPerLaunch ? n - i : kSwapIdsPerLaunch;
    SwapIds s;
    for (int j = 0; j < m; ++j) s.id[j] = ids[i + j];
    const int cap = max_ctas > 0 ? max_ctas : (to_host ? kSwapCtasOut : kSwapCtasIn);
    const int grid = m < cap ? m : cap;
    uint4* h = static_cast<uint4*>(host_dev) + static_cast<int64_t>(i) * 2 * blk_chunks;
    swap_kernel<<<grid, kSwapThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4*>(kp), static_cast<uint4*>(vp), h, s, m, blk_chunks, to_host ? 1 : 0);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace pkv

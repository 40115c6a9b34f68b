// Streaming HBM read probe: every thread reads four independent 16-byte words per step
// (grid-stride), folds them into a checksum, and one atomic per warp publishes it.
#include <cuda_runtime.h>
#include <stdint.h>

#include "sv_internal.h"
#include "sv_ptx.cuh"

namespace sv {
namespace {

__global__ void __launch_bounds__(256) probe_kernel(const uint4* __restrict__ p, size_t n,
                                                    unsigned long long* out) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  uint32_t acc = 0;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const uint4 a = __ldg(p + i), b = __ldg(p + i + stride);
    const uint4 c = __ldg(p + i + 2 * stride), d = __ldg(p + i + 3 * stride);
    acc += (a.x ^ b.y ^ c.z ^ d.w) + (a.y ^ b.z ^ c.w ^ d.x) + (a.z ^ b.w ^ c.x ^ d.y) +
           (a.w ^ b.x ^ c.y ^ d.z);
  }
  for (; i < n; i += stride) {
    const uint4 a = __ldg(p + i);
    acc += a.x ^ a.y ^ a.z ^ a.w;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) atomicAdd(out, static_cast<unsigned long long>(acc));
}

// One thread waits on an mbarrier that nothing arrives at, with the same bounded wait the
// kernels use, for `budget` clock cycles; when the wait gives up it raises bit 0 of the error
// word, as a kernel whose copy or peer never came would, and returns.
__global__ void wait_probe_kernel(long long budget, unsigned int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  if (!mbar_wait_bounded(&bar, 0, budget)) atomicOr(err, 1u);
}

}  // namespace

cudaError_t launch_wait_probe(long long budget_cycles, unsigned int* err, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(budget_cycles, err);
  return cudaGetLastError();
}

cudaError_t launch_probe(const void* buf, size_t bytes, unsigned long long* out,
                         cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  probe_kernel<<<sms * 8, 256, 0, stream>>>(static_cast<const uint4*>(buf), bytes / 16, out);
  return cudaGetLastError();
}

}  // namespace sv

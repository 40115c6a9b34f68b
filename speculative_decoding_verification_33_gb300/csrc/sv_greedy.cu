// Greedy verification of small batches with every target row in flight at once (LayerSkip
// guide, "Verification Phase": accept draft i while it equals the target's argmax, then emit the
// target's argmax at the first mismatch).
//
// In greedy mode the rows of a sequence do not depend on each other: the argmax of each target
// row can be taken independently, and only the scan over positions is sequential. For a batch
// whose rows are few (the chained cluster walk is then bound by the latency of its position
// after position), two launches do it:
//  1. greedy_rows: one CTA per (target row, slice of the vocabulary) for rows 0..L_b of every
//     sequence, reducing its slice to one sort key (the value's order bits, then the inverted id,
//     so the largest key is the largest value at the lowest id) or to a "bad" sentinel when the
//     slice holds a NaN or +inf;
//  2. greedy_decide: one warp per sequence combines a row's slice keys, walks the positions in
//     order (a row that is NaN / +inf / all -inf makes the sequence invalid, but only up to the
//     decided position) and writes the outcome.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "sv_greedy.h"
#include "sv_math.cuh"
#include "sv_ptx.cuh"

namespace sv {
namespace {

constexpr int kThreads = 256;
constexpr unsigned long long kBad = ~0ull;  // a slice with a NaN or +inf
constexpr int kMaxGreedyK = 8;              // positions per sequence (K <= 8)

// Programmatic dependent launch: let the next launch on the stream start its CTAs, and wait
// until the previous launch has finished and its writes are visible.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename T>
__global__ void __launch_bounds__(kThreads) greedy_rows(const GreedyParams P) {
  pdl_trigger();
  __shared__ unsigned long long wk[kThreads / 32];
  const int sl = blockIdx.x, r = blockIdx.y;
  const int b = r / (P.K + 1), i = r - b * (P.K + 1);
  const int L = P.lens ? P.lens[b] : P.K;
  if (L < 1 || L > P.K || i > L) return;  // rows the walk never reads
  const int e0 = sl * P.slice, e1 = min(P.V, e0 + P.slice);
  const T* row = static_cast<const T*>(P.tgt) + static_cast<long long>(r) * P.stride;
  unsigned long long best = 0;
  bool bad = false;
  auto take = [&](float z, int id) {
    bad |= isnan(z) || z == INFINITY;
    const unsigned long long k = make_key(z, static_cast<uint32_t>(id));
    best = k > best ? k : best;
  };
  if (P.aligned) {  // 8 elements per 16-byte load, whole vectors only
    const int v0 = (e0 + 7) >> 3, v1 = e1 >> 3;
    for (int e = e0 + threadIdx.x; e < min(e1, v0 * 8); e += kThreads) take(Elt<T>::val(row[e]), e);
    for (int g = v0 + threadIdx.x; g < v1; g += kThreads) {
      float z[8];
      Elt<T>::ldg8(row + 8 * g, z);
#pragma unroll
      for (int k = 0; k < 8; ++k) take(z[k], 8 * g + k);
    }
    for (int e = max(v1 * 8, v0 * 8) + threadIdx.x; e < e1; e += kThreads)
      take(Elt<T>::val(row[e]), e);
  } else {
    for (int e = e0 + threadIdx.x; e < e1; e += kThreads) take(Elt<T>::val(row[e]), e);
  }
  if (__any_sync(FULL, bad)) best = kBad;
  best = warp_max_u64(best);
  if ((threadIdx.x & 31) == 0) wk[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long m = wk[0];
    for (int w = 1; w < kThreads / 32; ++w) m = wk[w] > m ? wk[w] : m;
    P.keys[static_cast<long long>(r) * P.nslice + sl] = m;
  }
}

__global__ void greedy_decide(const GreedyParams P) {
  __shared__ unsigned long long pm[4][kMaxGreedyK + 1];
  const int wib = threadIdx.x >> 5;
  const int b = blockIdx.x * (blockDim.x >> 5) + wib;
  const int lane = threadIdx.x & 31;
  if (b >= P.B) return;  // whole warps
  const int K = P.K;
  const int L = P.lens ? P.lens[b] : K;
  const int32_t* x = P.tokens + static_cast<long long>(b) * K;
  bool ok = L >= 1 && L <= K;
  const int xi = (ok && lane < L) ? x[lane] : 0;
  ok = ok && __all_sync(FULL, lane >= L || (xi >= 0 && xi < P.V));
  int a = -1, last = -1;
  pdl_wait();  // the slice keys come from the row launch (the ids and lengths are inputs)
  if (ok) {
    // every slice key of rows 0..L in one round of loads, folded per row in shared memory
    if (lane <= L) pm[wib][lane] = 0ull;
    __syncwarp();
    const unsigned long long* k = P.keys + static_cast<long long>(b) * (K + 1) * P.nslice;
    for (int j = lane; j < (L + 1) * P.nslice; j += 32) atomicMax(&pm[wib][j / P.nslice], k[j]);
    __syncwarp();
    for (int i = 0; i <= L; ++i) {  // the oracle's order: a bad row counts only up to the stop
      const unsigned long long m = pm[wib][i];
      if (m == kBad || key_value(m) == -INFINITY) {  // NaN / +inf, or nothing but -inf
        ok = false;
        break;
      }
      const int g = key_id(m);
      if (i < L && __shfl_sync(FULL, xi, i) == g) continue;
      a = i;
      last = g;
      break;
    }
  }
  int32_t* tok = P.out_tok + static_cast<long long>(b) * (K + 1);
  for (int j = lane; j <= K; j += 32) tok[j] = (ok && j < a) ? x[j] : ((ok && j == a) ? last : -1);
  if (lane == 0) P.out_acc[b] = ok ? a : -1;
}

}  // namespace

void greedy_plan(int B, int K, int V, int sms, int* nslice, int* slice) {
  const long long rows = static_cast<long long>(B) * (K + 1);
  long long ns = (4LL * sms + rows - 1) / rows;  // about four CTAs per SM over all rows
  ns = std::max<long long>(1, std::min<long long>(ns, (V + 1023) / 1024));
  int sl = static_cast<int>((V + ns - 1) / ns);
  sl = (sl + 7) / 8 * 8;
  *slice = sl;
  *nslice = (V + sl - 1) / sl;
}

cudaError_t launch_greedy(const GreedyParams& P, int dtype, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(P.nslice), static_cast<unsigned>(P.B * (P.K + 1)));
  if (dtype == 1)
    greedy_rows<uint16_t><<<grid, kThreads, 0, stream>>>(P);
  else
    greedy_rows<float><<<grid, kThreads, 0, stream>>>(P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((P.B + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, greedy_decide, P);
}

}  // namespace sv

// The LM head fused with the softmax statistics of the verify step: logits = h W^T on the
// fifth-generation tensor cores, reduced to per-row statistics in the epilogue so that no logit
// reaches HBM (Kangaroo guide, "Exit 1": the head is Softmax(W h); LayerSkip guide: the early
// exit and the full model share that head).
//
// One CTA owns a 128-row tile of hidden states and a range of the vocabulary, walked in tiles
// of 256 columns:
//  - warp 0 (one thread) loads 128 x 64 tiles of h and 256 x 64 tiles of W with TMA (128-byte
//    swizzle) into a 4-stage shared-memory ring;
//  - warp 1 allocates 512 columns of tensor memory (two 128 x 256 fp32 accumulators) and one of
//    its threads issues tcgen05.mma (M 128, N 256, K 16, bf16 in, fp32 accumulate), committing
//    each stage back to the producer and each finished tile to the epilogue;
//  - warps 2..5 (one thread per row) read a finished accumulator 32 columns at a time and fold
//    it into the row's running maximum m and sum 2^(z c - fl(m c)), while the tensor cores
//    fill the other accumulator.
// A second small kernel combines the vocabulary ranges of a row into the maximum logit, the
// log-sum-exp of z / T and the logit of a requested id.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "sv_lmhead.h"
#include "sv_math.cuh"
#include "sv_ptx.cuh"
#include "sv_tc.cuh"

namespace sv {
namespace {

constexpr int BM = kHeadBM, BN = kHeadBN, BK = kHeadBK;
constexpr int kStages = 4;
constexpr int kABytes = BM * BK * 2;                // 16 KB
constexpr int kBBytes = BN * BK * 2;                // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;      // 48 KB
constexpr int kHeadThreads = 192;                   // 6 warps
constexpr uint32_t kTmemCols = 2 * BN;              // two accumulators
constexpr long long kWaitBudget = 4000000000LL;     // clock cycles (about 2 s) per wait
constexpr float kLn2 = 0.69314718055994531f;

// v[i] for a run-time i in 0..31, by halving on the bits of i (register selects only).
__device__ __forceinline__ float pick32(const float (&v)[32], int i) {
  float a[16], b[8], c[4], d[2];
#pragma unroll
  for (int j = 0; j < 16; ++j) a[j] = (i & 16) ? v[j + 16] : v[j];
#pragma unroll
  for (int j = 0; j < 8; ++j) b[j] = (i & 8) ? a[j + 8] : a[j];
#pragma unroll
  for (int j = 0; j < 4; ++j) c[j] = (i & 4) ? b[j + 4] : b[j];
#pragma unroll
  for (int j = 0; j < 2; ++j) d[j] = (i & 2) ? c[j + 2] : c[j];
  return (i & 1) ? d[1] : d[0];
}

__global__ void __launch_bounds__(kHeadThreads, 1)
    lmhead_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const HeadParams P) {
  extern __shared__ unsigned char dsm[];
  __shared__ uint64_t full[kStages], empty[kStages], accf[2], acce[2], drain;
  __shared__ uint32_t tmem_slot;
  unsigned char* base = dsm + ((1024u - (smem_u32(dsm) & 1023u)) & 1023u);  // 1024-aligned
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mtile = blockIdx.x / P.nsplit, split = blockIdx.x % P.nsplit;
  const int m0 = mtile * BM;
  const int t0 = split * P.tiles_per_split;
  const int nt = max(0, min(P.ntiles, t0 + P.tiles_per_split) - t0);
  const int KB = P.d / BK;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], 4);
    }
    mbar_init(&drain, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(&tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer ----
      int it = 0;
      bool ok = true;
      for (int t = 0; t < nt && ok; ++t) {
        const int n0 = (t0 + t) * BN;
        for (int kb = 0; kb < KB; ++kb) {
          const int s = it % kStages;
          if (it >= kStages &&
              !mbar_wait_bounded(&empty[s], static_cast<uint32_t>((it / kStages) - 1) & 1u,
                                 kWaitBudget)) {
            ok = false;
            break;
          }
          unsigned char* sa = base + static_cast<size_t>(s) * kStageBytes;
          mbar_arrive_expect_tx(&full[s], kStageBytes);
          tma_load_2d(sa, &tmA, kb * BK, m0, &full[s]);
          tma_load_2d(sa + kABytes, &tmB, kb * BK, n0, &full[s]);
          ++it;
        }
      }
      // no copy may still be writing shared memory when the CTA ends (matters only after a
      // wait above gave up): wait, bounded, for the last load of every stage
      for (int u = max(0, it - kStages); u < it; ++u)
        if (!mbar_wait_bounded(&full[u % kStages], static_cast<uint32_t>(u / kStages) & 1u,
                               kWaitBudget))
          ok = false;
      if (!ok) atomicOr(P.err, 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issuer ----
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
      int it = 0;
      bool ok = true;
      for (int t = 0; t < nt && ok; ++t) {
        const int b = t & 1;
        if (t >= 2 &&
            !mbar_wait_bounded(&acce[b], static_cast<uint32_t>((t >> 1) - 1) & 1u, kWaitBudget)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(b * BN);
        for (int kb = 0; kb < KB; ++kb) {
          const int s = it % kStages;
          if (!mbar_wait_bounded(&full[s], static_cast<uint32_t>(it / kStages) & 1u,
                                 kWaitBudget)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(base + static_cast<size_t>(s) * kStageBytes);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)  // K = 16 per instruction: 32 bytes along a row
            tc_mma_bf16(d_tmem, smem_desc_sw128(sa + 32 * kk), smem_desc_sw128(sb + 32 * kk),
                        idesc, (kb | kk) != 0 ? 1u : 0u);
          tc_commit(&empty[s]);
          ++it;
        }
        if (ok) tc_commit(&accf[b]);
      }
      // every MMA issued has completed before the tensor memory is released
      tc_commit(&drain);
      if (!mbar_wait_bounded(&drain, 0, kWaitBudget)) ok = false;
      if (!ok) atomicOr(P.err, 1u);
    }
  } else {  // ---- epilogue: warps 2..5, one thread per row of the tile ----
    const int q = warp & 3;  // tensor-memory lanes 32 q .. 32 q + 31
    const int row = m0 + 32 * q + lane;
    const int x = (P.ids && row < P.R) ? P.ids[row] : -1;
    const float c = P.c;
    float m = -INFINITY, mc = -INFINITY, s = 0.f, zx = NAN;
    for (int t = 0; t < nt; ++t) {
      const int b = t & 1;
      // the warp leaves together: tcgen05.ld below is a warp-wide (aligned) instruction
      const bool got = mbar_wait_bounded(&accf[b], static_cast<uint32_t>(t >> 1) & 1u, kWaitBudget);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) atomicOr(P.err, 1u);
        break;
      }
      tc_fence_after();
      const int n0 = (t0 + t) * BN;
      for (int ch = 0; ch < BN / 32; ++ch) {
        float v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(b * BN + ch * 32),
                  v);
        const int col0 = n0 + ch * 32;
        const int nvalid = min(32, P.V - col0);
        float cm = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < nvalid) cm = max_nan(cm, v[j]);
        if (x >= col0 && x < col0 + 32) zx = pick32(v, x - col0);
        if (P.out_logits && row < P.R) {
          float* o = P.out_logits + static_cast<long long>(row) * P.V + col0;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nvalid) o[j] = v[j];
        }
        const float mn = max_nan(m, cm);
        if (mn != m) {  // the running maximum rises: rescale the sum
          const float mcn = __fmul_rn(mn, c);
          s = m > -INFINITY ? s * exp2f(mc - mcn) : 0.f;
          m = mn;
          mc = mcn;
        }
        if (m > -INFINITY) {
          float2 acc = make_float2(0.f, 0.f);
          const float2 c2 = make_float2(c, c), n2 = make_float2(-mc, -mc);
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float2 a = __ffma2_rn(make_float2(v[j], v[j + 1]), c2, n2);
            acc = __fadd2_rn(acc, make_float2(j < nvalid ? ex2_fast(a.x) : 0.f,
                                              j + 1 < nvalid ? ex2_fast(a.y) : 0.f));
          }
          s += acc.x + acc.y;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[b]);
    }
    if (row < P.R) {
      float* pr = P.part + (static_cast<long long>(split) * P.R + row) * 3;
      pr[0] = m;
      pr[1] = s;
      pr[2] = zx;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// The vocabulary ranges of a row into its maximum logit, log-sum-exp of z / T (rounding of
// fl(m c) folded back) and the logit at its id.
__global__ void lmhead_combine(const HeadParams P, float* out_max, float* out_lse,
                               float* out_zx) {
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= P.R) return;
  const float c = P.c;
  float M = -INFINITY;
  for (int sp = 0; sp < P.nsplit; ++sp) M = max_nan(M, P.part[(static_cast<long long>(sp) * P.R + row) * 3]);
  float lse = M;
  if (!row_bad(M)) {
    const float Mc = __fmul_rn(M, c);
    float S = 0.f;
    for (int sp = 0; sp < P.nsplit; ++sp) {
      const float* pr = P.part + (static_cast<long long>(sp) * P.R + row) * 3;
      if (pr[0] > -INFINITY) S += pr[1] * exp2f(__fmul_rn(pr[0], c) - Mc);
    }
    lse = fmaf(M, P.inv_t, logf(S)) - fmaf(M, c, -Mc) * kLn2;
  }
  out_max[row] = M;
  out_lse[row] = lse;
  if (out_zx) {
    float zx = NAN;
    const int x = P.ids ? P.ids[row] : -1;
    if (x >= 0 && x < P.V) {
      const int sp = (x / BN) / P.tiles_per_split;
      zx = P.part[(static_cast<long long>(sp) * P.R + row) * 3 + 2];
    }
    out_zx[row] = zx;
  }
}

// ------------------------------------------------------------------------------------------
// tensor maps (the driver's encoder, looked up once through the runtime)
// ------------------------------------------------------------------------------------------
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
  static std::once_flag once;
  static EncodeFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// A 2-D bf16 tensor of `rows` rows of `cols` elements (row stride `stride` elements), read in
// boxes of `box_rows` x 64 with the 128-byte swizzle; rows or columns past the end read as 0.
bool make_map(CUtensorMap* m, const void* ptr, long long rows, long long cols, long long stride,
              int box_rows) {
  EncodeFn fn = encoder();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

void head_split(int R, int V, int sms, int* nsplit, int* tiles_per_split, int* ntiles) {
  const int mt = (R + BM - 1) / BM;
  const int nt = (V + BN - 1) / BN;
  int ns = std::max(1, std::min(nt, sms / std::max(1, mt)));
  const int per = (nt + ns - 1) / ns;
  ns = (nt + per - 1) / per;
  *nsplit = ns;
  *tiles_per_split = per;
  *ntiles = nt;
}

cudaError_t launch_lmhead(const void* hidden, long long hs, const void* weight, long long ws,
                          const HeadParams& P, float* out_max, float* out_lse, float* out_zx,
                          cudaStream_t stream) {
  CUtensorMap ta, tb;
  if (!encoder()) return cudaErrorNotSupported;
  if (!make_map(&ta, hidden, P.R, P.d, hs, BM) || !make_map(&tb, weight, P.V, P.d, ws, BN))
    return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(kStages) * kStageBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(lmhead_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int mt = (P.R + BM - 1) / BM;
  lmhead_kernel<<<mt * P.nsplit, kHeadThreads, smem, stream>>>(ta, tb, P);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  lmhead_combine<<<(P.R + 127) / 128, 128, 0, stream>>>(P, out_max, out_lse, out_zx);
  return cudaGetLastError();
}

}  // namespace sv

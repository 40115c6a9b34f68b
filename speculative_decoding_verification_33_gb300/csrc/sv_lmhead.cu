// The LM head fused with what the verify step needs from its softmax: logits = h W^T on the
// fifth-generation tensor cores, reduced in the epilogue so that no logit reaches HBM (Kangaroo
// guide, "Exit 1": the head is Softmax(W h); LayerSkip guide: the early exit and the full model
// share that head).
//
// A persistent grid (one CTA per SM) walks work items (a 128-row tile of A, a range of 256-column
// vocabulary tiles), range-major so that the CTAs running at the same time share head tiles in
// L2. Per CTA:
//  - warp 0 (one thread) loads 128 x 64 tiles of A and 256 x 64 tiles of W with TMA (128-byte
//    swizzle) into a 4-stage shared-memory ring, running ahead across tiles and items;
//  - warp 1 allocates 512 columns of tensor memory (two 128 x 256 fp32 accumulators) and one of
//    its threads issues tcgen05.mma (M 128, N 256, K 16, bf16 in, fp32 accumulate), committing
//    each stage back to the producer and each finished tile to the epilogue;
//  - warps 2..5 (one thread per row) read a finished accumulator 32 columns at a time while the
//    tensor cores fill the other one:
//      HEAD_STATS: the row's running maximum m (and the lowest id holding it), the sum
//        2^(z c - fl(m c)) rescaled when m rises, and the logit at a requested id; one partial
//        per (range, row), combined by a second kernel; HEAD_STATS_TOP8 keeps besides the row's
//        8 largest logits in the range (as keys: larger value first, then lower id), offered
//        only the chunks whose maximum reaches the 8th so far;
//      HEAD_RESID: rows come in (target, draft) pairs 16 lanes apart; each thread takes 16 of a
//        chunk's 32 ids, gets the other row's logits by a lane exchange, and writes the mass of
//        max(2^(z_t c - mc_t) - rho 2^(z_d c - mc_d), 0) over those 16 ids in 2^-44 units (rho
//        times beta on the ids of a Saguaro bias set).
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

// The work item w of a grid over `mt` row tiles: range-major.
struct Item {
  int m0, t0, nt, split;
};
__device__ __forceinline__ Item item_of(int w, int mt, const HeadParams& P) {
  Item it;
  it.split = w / mt;
  it.m0 = (w - it.split * mt) * BM;
  it.t0 = it.split * P.tiles_per_split;
  it.nt = max(0, min(P.ntiles, it.t0 + P.tiles_per_split) - it.t0);
  return it;
}

// ------------------------------------------------------------------------------------------
// epilogue of one 32-column chunk
// ------------------------------------------------------------------------------------------
struct StatsState {
  float m, mc, s, zx;
  int arg;
};

// Returns the chunk's maximum.
__device__ __forceinline__ float stats_chunk(StatsState& st, const float (&v)[32], int col0,
                                             int nvalid, int x, float c, float* logits_row) {
  float cm = -INFINITY;
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (j < nvalid) cm = max_nan(cm, v[j]);
  if (x >= col0 && x < col0 + 32) st.zx = pick32(v, x - col0);
  if (logits_row) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < nvalid) logits_row[col0 + j] = v[j];
  }
  if (cm > st.m) {  // a new maximum: the lowest id holding it in this chunk
    int j0 = 31;
#pragma unroll
    for (int j = 31; j >= 0; --j)
      if (j < nvalid && v[j] == cm) j0 = j;
    st.arg = col0 + j0;
  }
  const float mn = max_nan(st.m, cm);
  if (mn != st.m) {  // the running maximum rises (or turns NaN): rescale the sum
    const float mcn = __fmul_rn(mn, c);
    st.s = st.m > -INFINITY ? st.s * exp2f(st.mc - mcn) : 0.f;
    st.m = mn;
    st.mc = mcn;
  }
  if (st.m > -INFINITY) {
    float2 acc = make_float2(0.f, 0.f);
    const float2 c2 = make_float2(c, c), n2 = make_float2(-st.mc, -st.mc);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const float2 a = __ffma2_rn(make_float2(v[j], v[j + 1]), c2, n2);
      acc = __fadd2_rn(acc, make_float2(j < nvalid ? ex2_fast(a.x) : 0.f,
                                        j + 1 < nvalid ? ex2_fast(a.y) : 0.f));
    }
    st.s += acc.x + acc.y;
  }
  return cm;
}

// The chunk's logits that reach the row's 8th largest so far, into its 8 largest (keys, ids
// col0 + j); cm is the chunk's maximum.
__device__ __forceinline__ void top8_chunk(unsigned long long (&keys)[8], float& thr,
                                           const float (&v)[32], float cm, int col0, int nvalid) {
  if (!(cm >= thr)) return;
  unsigned mask = 0u;
#pragma unroll
  for (int j = 0; j < 32; ++j) mask |= (j < nvalid && v[j] >= thr) ? (1u << j) : 0u;
  while (mask) {
    const int j = __ffs(mask) - 1;
    mask &= mask - 1;
    top8_insert(keys, thr, pick32(v, j), static_cast<uint32_t>(col0 + j));
  }
}

// Residual mass (and target mass) of this thread's 16 ids of a chunk. Lane l < 16 holds the
// target row of its pair and takes ids col0 .. col0 + 15; lane l + 16 holds the draft row and
// takes the other 16. Both sums run in id order, one addition per id.
__device__ __forceinline__ float2 resid_chunk(const float (&v)[32], bool is_d, int col0,
                                              int nvalid, float c, const HeadPair& pp) {
  float acc = 0.f, accp = 0.f;
  const int base = is_d ? 16 : 0;
  // an id of the bias set among this thread's 16 (then each id is checked)
  bool hb = false;
#pragma unroll
  for (int k = 0; k < 8; ++k)
    hb |= k < pp.nS && static_cast<unsigned>(pp.ids[k] - (col0 + base)) < 16u;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float send = is_d ? v[j] : v[16 + j];
    const float got = __shfl_xor_sync(0xffffffffu, send, 16);
    const float zt = is_d ? got : v[j];
    const float zd = is_d ? v[16 + j] : got;
    const float et = ex2_fast(fmaf(zt, c, -pp.mc_t));
    const float ed = ex2_fast(fmaf(zd, c, -pp.mc_d));
    float rk = pp.rho;
    if (hb) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        rk = (k < pp.nS && pp.ids[k] == col0 + base + j) ? pp.rho_s : rk;
    }
    const float w = fmaxf(fmaf(-rk, ed, et), 0.f);
    acc += (base + j < nvalid) ? w : 0.f;
    accp += (base + j < nvalid) ? et : 0.f;
  }
  return make_float2(acc, accp);
}

// ------------------------------------------------------------------------------------------
// the persistent GEMM
// ------------------------------------------------------------------------------------------
template <int MODE>
__global__ void __launch_bounds__(kHeadThreads, 1)
    lmhead_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const HeadParams P) {
  extern __shared__ unsigned char dsm[];
  __shared__ uint64_t full[kStages], empty[kStages], accf[2], acce[2], drain;
  __shared__ uint32_t tmem_slot;
  unsigned char* base = dsm + ((1024u - (smem_u32(dsm) & 1023u)) & 1023u);  // 1024-aligned
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = P.R_dev ? max(0, min(*P.R_dev, P.R)) : P.R;
  const int mt = (R + BM - 1) / BM;
  const int nitems = mt * P.nsplit;
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
      for (int w = blockIdx.x; w < nitems && ok; w += gridDim.x) {
        const Item I = item_of(w, mt, P);
        for (int t = 0; t < I.nt && ok; ++t) {
          const int n0 = (I.t0 + t) * BN;
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
            tma_load_2d(sa, &tmA, kb * BK, I.m0, &full[s]);
            tma_load_2d(sa + kABytes, &tmB, kb * BK, n0, &full[s]);
            ++it;
          }
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
      int it = 0, T = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < nitems && ok; w += gridDim.x) {
        const Item I = item_of(w, mt, P);
        for (int t = 0; t < I.nt && ok; ++t, ++T) {
          const int b = T & 1;
          if (T >= 2 &&
              !mbar_wait_bounded(&acce[b], static_cast<uint32_t>((T >> 1) - 1) & 1u,
                                 kWaitBudget)) {
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
      }
      // every MMA issued has completed before the tensor memory is released
      tc_commit(&drain);
      if (!mbar_wait_bounded(&drain, 0, kWaitBudget)) ok = false;
      if (!ok) atomicOr(P.err, 1u);
    }
  } else {  // ---- epilogue: warps 2..5, one thread per row of the tile ----
    const int q = warp & 3;  // tensor-memory lanes 32 q .. 32 q + 31
    const float c = P.c;
    int T = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < nitems && ok; w += gridDim.x) {
      const Item I = item_of(w, mt, P);
      const int row = I.m0 + 32 * q + lane;
      StatsState st;
      st.m = -INFINITY;
      st.mc = -INFINITY;
      st.s = 0.f;
      st.zx = NAN;
      st.arg = -1;
      int x = -1;
      float* lrow = nullptr;
      HeadPair pp;
      pp.mc_t = pp.mc_d = pp.rho = pp.rho_s = 0.f;
      pp.skip = 1;
      pp.nS = 0;
      unsigned long long keys[8];
      float kthr = -INFINITY;
#pragma unroll
      for (int k = 0; k < 8; ++k) keys[k] = 0ull;
      const bool is_d = lane >= 16;
      const int pr = (I.m0 >> 1) + 16 * q + (lane & 15);
      if (MODE != HEAD_RESID) {
        x = (P.ids && row < R) ? P.ids[row] : -1;
        lrow = (P.out_logits && row < R) ? P.out_logits + static_cast<long long>(row) * P.V
                                         : nullptr;
      } else if (row < R) {
        pp = P.pair[pr];
      }
      for (int t = 0; t < I.nt; ++t, ++T) {
        const int b = T & 1;
        // the warp leaves together: tcgen05.ld below is a warp-wide (aligned) instruction
        const bool got =
            mbar_wait_bounded(&accf[b], static_cast<uint32_t>(T >> 1) & 1u, kWaitBudget);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) atomicOr(P.err, 1u);
          ok = false;
          break;
        }
        tc_fence_after();
        const int n0 = (I.t0 + t) * BN;
        for (int ch = 0; ch < BN / 32; ++ch) {
          float v[32];
          tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) +
                        static_cast<uint32_t>(b * BN + ch * 32),
                    v);
          const int col0 = n0 + ch * 32;
          const int nvalid = min(32, P.V - col0);
          if (MODE != HEAD_RESID) {
            const float cm = stats_chunk(st, v, col0, nvalid, x, c, lrow);
            if (MODE == HEAD_STATS_TOP8) top8_chunk(keys, kthr, v, cm, col0, nvalid);
          } else {
            const float2 s = resid_chunk(v, is_d, col0, nvalid, c, pp);
            if (row < R) {
              const long long at = static_cast<long long>(pr) * P.nh + col0 / 16 + (is_d ? 1 : 0);
              P.mass[at] = pp.skip ? 0ull : qfix(s.x);
              P.mass_p[at] = pp.skip ? 0ull : qfix(s.y);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce[b]);
      }
      if (MODE != HEAD_RESID && ok && row < R)
        P.part[static_cast<long long>(I.split) * P.R + row] =
            make_float4(st.m, st.s, st.zx, __int_as_float(st.arg));
      if (MODE == HEAD_STATS_TOP8 && ok && row < R) {
        ulonglong2* kp = reinterpret_cast<ulonglong2*>(
            P.keys + (static_cast<long long>(I.split) * P.R + row) * 8);
#pragma unroll
        for (int k = 0; k < 4; ++k) kp[k] = make_ulonglong2(keys[2 * k], keys[2 * k + 1]);
      }
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

// The vocabulary ranges of a row into its maximum logit (lowest id on ties: a larger range index
// only wins with a strictly larger maximum), the log-sum-exp of z / T (rounding of fl(m c) folded
// back), the logit at its id and the lowest id holding the maximum. One warp per row, the lanes
// striding over the ranges.
__global__ void lmhead_combine(const HeadParams P, float* out_max, float* out_lse, float* out_zx,
                               int32_t* out_arg, HeadRow* out_rows) {
  const int lane = threadIdx.x & 31;
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int R = P.R_dev ? max(0, min(*P.R_dev, P.R)) : P.R;
  if (row >= R) return;  // whole warps leave together
  const float c = P.c;
  float M = -INFINITY;
  int msp = 0x7fffffff;
  bool nan = false;
  for (int sp = lane; sp < P.nsplit; sp += 32) {
    const float m = P.part[static_cast<long long>(sp) * P.R + row].x;
    if (isnan(m)) nan = true;
    if (m > M) {
      M = m;
      msp = sp;
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, M, o);
    const int osp = __shfl_xor_sync(0xffffffffu, msp, o);
    if (om > M || (om == M && osp < msp)) {
      M = om;
      msp = osp;
    }
  }
  if (__any_sync(0xffffffffu, nan)) M = NAN;
  float lse = M, Mc = M, S = NAN;
  if (!row_bad(M)) {
    Mc = __fmul_rn(M, c);
    float part = 0.f;
    for (int sp = lane; sp < P.nsplit; sp += 32) {
      const float4 pr = P.part[static_cast<long long>(sp) * P.R + row];
      if (pr.x > -INFINITY) part += pr.y * exp2f(__fmul_rn(pr.x, c) - Mc);
    }
    S = warp_sum(part);
    lse = fmaf(M, P.inv_t, logf(S)) - fmaf(M, c, -Mc) * kLn2;
  }
  if (lane != 0) return;
  const int arg = row_bad(M) ? -1 : __float_as_int(P.part[static_cast<long long>(msp) * P.R + row].w);
  float zx = NAN;
  const int x = P.ids ? P.ids[row] : -1;
  if (x >= 0 && x < P.V) {
    const int sp = (x / BN) / P.tiles_per_split;
    zx = P.part[static_cast<long long>(sp) * P.R + row].z;
  }
  if (out_max) out_max[row] = M;
  if (out_lse) out_lse[row] = lse;
  if (out_zx) out_zx[row] = zx;
  if (out_arg) out_arg[row] = arg;
  if (out_rows) {
    HeadRow h;
    h.max = M;
    h.lse = lse;
    h.zx = zx;
    h.arg = arg;
    h.mc = Mc;
    h.sum = S;
    out_rows[row] = h;
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

int head_ctas(int sms) { return std::max(1, sms); }

void head_split(int R, int V, int sms, int* nsplit, int* tiles_per_split, int* ntiles,
                int max_ranges) {
  const int mt = std::max(1, (R + BM - 1) / BM);
  const int nt = (V + BN - 1) / BN;
  const int ctas = head_ctas(sms);
  if (max_ranges > 0) {  // any range length that keeps the ranges at most max_ranges
    long long best = -1;
    int best_tps = nt;
    for (int tps = (nt + max_ranges - 1) / max_ranges; tps <= nt; ++tps) {
      const int ns = (nt + tps - 1) / tps;
      const long long items = static_cast<long long>(mt) * ns;
      const long long cost = (items + ctas - 1) / ctas * tps;
      if (best < 0 || cost <= best) {
        best = cost;
        best_tps = tps;
      }
    }
    *tiles_per_split = best_tps;
    *nsplit = (nt + best_tps - 1) / best_tps;
    *ntiles = nt;
    return;
  }
  // the range length (in tiles) with the fewest tile-times on the busiest CTA; longer ranges
  // win ties (fewer partial statistics)
  long long best = -1;
  int best_tps = 1;
  for (int tps = 1; tps <= 16; tps <<= 1) {
    const int ns = (nt + tps - 1) / tps;
    const long long items = static_cast<long long>(mt) * ns;
    const long long waves = (items + ctas - 1) / ctas;
    const long long cost = waves * std::min(tps, nt);
    if (best < 0 || cost <= best) {
      best = cost;
      best_tps = tps;
    }
    if (tps >= nt) break;
  }
  *tiles_per_split = best_tps;
  *nsplit = (nt + best_tps - 1) / best_tps;
  *ntiles = nt;
}

cudaError_t launch_head_gemm(int mode, const void* A, long long as, const void* weight,
                             long long ws, const HeadParams& P, int ctas, cudaStream_t stream) {
  CUtensorMap ta, tb;
  if (!encoder()) return cudaErrorNotSupported;
  if (!make_map(&ta, A, std::max(1, P.R), P.d, as, BM) ||
      !make_map(&tb, weight, P.V, P.d, ws, BN))
    return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(kStages) * kStageBytes + 1024;
  auto kern = mode == HEAD_STATS        ? lmhead_kernel<HEAD_STATS>
              : mode == HEAD_STATS_TOP8 ? lmhead_kernel<HEAD_STATS_TOP8>
                                        : lmhead_kernel<HEAD_RESID>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<std::max(1, ctas), kHeadThreads, smem, stream>>>(ta, tb, P);
  return cudaGetLastError();
}

cudaError_t launch_head_combine(const HeadParams& P, float* out_max, float* out_lse,
                                float* out_zx, int32_t* out_arg, HeadRow* out_rows,
                                cudaStream_t stream) {
  if (P.R <= 0) return cudaSuccess;
  const long long threads = static_cast<long long>(P.R) * 32;
  lmhead_combine<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, stream>>>(
      P, out_max, out_lse, out_zx, out_arg, out_rows);
  return cudaGetLastError();
}

}  // namespace sv

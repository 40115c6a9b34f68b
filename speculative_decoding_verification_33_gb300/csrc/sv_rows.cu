// Row kernels beside the verify step, built from the same per-element arithmetic:
//
//  - Draft sampling, the draft generator's step: token x ~ q' (the beta-biased softmax of the draft
//    head's logits; Saguaro summary, "Method": drafts are drawn from the biased q'), drawn by the
//    same fixed-point inverse CDF as the verify step's draws, and the exit confidence
//    c = max_v q(v) of the unbiased softmax (Kangaroo guide, section 2, "Exit 2": drafting halts
//    once c falls below a threshold tau).
//  - Exact-residual top-F: for every draft position, the F most likely ids of the residual
//    max(p - q', 0) the verify step samples from after a rejection there, next to the top-F draft
//    ids a speculation cache prepares (Saguaro summary, "Key claims" and "Method"), and whether
//    the realised token at the decided position was among the cache's guesses.
//
// Persistent CTAs with three kinds of warps, one row (sampling) or one (sequence, position) pair
// (residual) -- a unit -- at a time, taken from a device queue:
//  - a producer warp streams the units' rows through a ring of shared-memory stages with bulk
//    asynchronous copies;
//  - eight chunk warps reduce every 64-element group of a row to its maximum g and (sampling)
//    its mass, the sum of 2^(z c - fl(g c)), or (residual) the target and draft maxima and the
//    largest log-ratio max (z_t - z_d), written to one of two group buffers, and each row to its
//    maximum and softmax sum;
//  - a team of four epilogue warps finishes a unit from its group buffer while the chunk warps
//    fill the other buffer with the next unit, so the stream never waits for an epilogue.
//
// The epilogue works from the group values, with a handful of groups read again:
//  - the row maximum and sum come with the buffer (softmax normaliser, exit confidence 1 / sum);
//  - the bias set (the bias_k largest draft logits): its elements lie in the 8 groups with the
//    largest maxima, and those in the threads' runs of groups whose maximum reaches a lower
//    bound of the 8th largest run maximum; one warp keeps the 8 largest such groups and reads
//    their elements;
//  - the draw: group masses scaled to the row maximum (the biased ids corrected) give the
//    fixed-point masses of the inverse CDF; the chosen group's 64 weights are recomputed to find
//    the element;
//  - the residual top F: each group's residual is bounded from its target maximum and its
//    log-ratio maximum once the normalisers are known, and groups are read in rounds of
//    decreasing bound until no bound left reaches the F-th best residual found.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "sv_internal.h"
#include "sv_math.cuh"
#include "sv_ptx.cuh"
#include "sv_rows.h"

namespace sv {
namespace {

constexpr int NCW = kRowChunkWarps;     // chunk warps
constexpr int NEW = kRowEpilogueWarps;  // epilogue warps
constexpr int CT = NCW * 32;            // chunk threads: 0 .. CT-1
constexpr int ET = NEW * 32;            // epilogue threads: CT .. CT+ET-1
constexpr int RT = kRowThreads;         // then the producer warp
constexpr uint32_t kBarC = 1;           // named barrier of the chunk threads
constexpr uint32_t kBarE = 2;           // named barrier of the epilogue threads
constexpr int kStage = kRowStageBytes;  // bytes per ring stage
constexpr int kGroup = 64;              // elements per group (8 vectors of 8)
constexpr float kLn2r = 0.69314718055994531f;
constexpr long long kWaitBudget = 4000000000LL;  // clock cycles (about 2 s) per barrier wait
constexpr int MODE_SAMPLE = 0, MODE_RESID = 1, MODE_TOP8 = 2;
constexpr int kEnd = -1;  // unit tag after the last unit
constexpr int kBatch = 8;  // residual: groups an epilogue warp reads per round trip
constexpr int kCandCap = 64;  // candidate groups of the bias set listed in shared memory
constexpr int kRoundCap = 256;  // residual: groups of one round listed in shared memory at once

static_assert(RT == CT + ET + 32, "chunk warps, epilogue warps, one producer warp");
static_assert(kStage % (8 * kGroup) == 0, "whole groups per stage");

struct RowShared {
  uint64_t full[kRowMaxStages], empty[kRowMaxStages];  // the ring
  uint64_t gfull[2], gfree[2];                         // the two group buffers
  int tag[kRowMaxStages];  // unit of the stage's chunk, or kEnd
  int gunit[2];            // unit of the group buffer, or kEnd
  float hdr[2][4];         // per buffer: row maximum and sum (target, then draft for a residual)
  float cm[NCW], cs[NCW];  // chunk-warp scratch
  // epilogue scratch
  float rmax[NEW], rb[NEW];
  unsigned long long ru[NEW];
  unsigned long long wtop[NEW][8];
  unsigned long long top[8];  // the last team top 8
  float N;
  int nS, gstar;
  int S_ids[8];
  float S_z[8];
  int sgrp[8];  // the groups of S_ids
  unsigned long long t_loc;
  // a bias set: the candidate groups of the 8 largest; sampling: the corrections of the groups
  // that hold ids of the set
  unsigned long long cand[kCandCap];
  int ncand;
  int dg[8];
  long long dq[8];
  // residual: the groups of the current round
  int tl[kRoundCap];
  int ntl;
};

// The epilogue team: thread t of ET, warp t / 32.
__device__ __forceinline__ int et() { return static_cast<int>(threadIdx.x) - CT; }
__device__ __forceinline__ void esync() { named_sync(kBarE, ET); }

// ------------------------------------------------------------------------------------------
// epilogue team reductions
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long warp_inclusive_u64(unsigned long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(FULL, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

__device__ unsigned long long team_exclusive_u64(unsigned long long v, RowShared& S,
                                                 unsigned long long* total = nullptr) {
  const int lane = threadIdx.x & 31, warp = et() >> 5;
  const unsigned long long inc = warp_inclusive_u64(v);
  if (lane == 31) S.ru[warp] = inc;
  esync();
  unsigned long long base = 0, all = 0;
  for (int w = 0; w < NEW; ++w) {
    if (w < warp) base += S.ru[w];
    all += S.ru[w];
  }
  esync();
  if (total) *total = all;
  return base + inc - v;
}

// ------------------------------------------------------------------------------------------
// top-8 selection: one running list per warp
// ------------------------------------------------------------------------------------------
struct Top8State {
  unsigned long long L;
  float thr;
  int kth;  // the threshold follows the key of this rank (0 .. 7) once it is held
};

// The insertion behind WarpTop8::offer, out of line (its loop is long and rarely taken); state in
// and out by value so that it stays in registers.
__device__ __noinline__ Top8State warp_top8_insert(unsigned pend, float z, uint32_t id,
                                                   Top8State st) {
  const int lane = threadIdx.x & 31;
  while (pend) {
    const int src = __ffs(pend) - 1;
    pend &= pend - 1;
    const float zs = __shfl_sync(FULL, z, src);
    const uint32_t is = __shfl_sync(FULL, id, src);
    if (!(zs >= st.thr)) continue;  // the threshold has risen past it
    const unsigned long long K = make_key(zs, is);
    const int pos = __popc(__ballot_sync(FULL, st.L > K));  // keys above it: lanes 0..pos-1
    if (pos < 8) {
      const unsigned long long up = __shfl_up_sync(FULL, st.L, 1);
      if (lane == pos) st.L = K;
      else if (lane > pos && lane < 8) st.L = up;
      const unsigned long long lk = __shfl_sync(FULL, st.L, st.kth);
      if (lk) st.thr = key_value(lk);
    }
  }
  return st;
}

// A warp's running top 8: the keys, descending, in lanes 0..7 (0 = empty; the other lanes hold
// 0), and a threshold every lane shares: nothing below it can enter. It is the value of the key
// of rank kth once that many are held (the 8th, or the F-th when only the first F of the list
// are wanted), or a known lower bound of that final key.
struct WarpTop8 {
  unsigned long long L;
  float thr;
  int kth;
  __device__ __forceinline__ void init(float lower, int rank = 7) {
    L = 0ull;
    thr = lower;
    kth = rank;
  }
  // Every lane of the warp calls this; a lane offers (z, id) when ok.
  __device__ __forceinline__ void offer(bool ok, float z, uint32_t id) {
    const unsigned pend = __ballot_sync(FULL, ok && z >= thr);
    if (!pend) return;
    const Top8State st = warp_top8_insert(pend, z, id, Top8State{L, thr, kth});
    L = st.L;
    thr = st.thr;
  }
};

// The warps' lists into the team's top 8, S.top (every epilogue thread may read it on return).
__device__ void team_top8(const WarpTop8& W, RowShared& S) {
  const int lane = threadIdx.x & 31, warp = et() >> 5;
  if (lane < 8) S.wtop[warp][lane] = W.L;
  esync();
  if (warp == 0) {
    static_assert(NEW * 8 == 32, "one candidate per lane");
    unsigned long long k8[8];
    k8[0] = S.wtop[lane >> 3][lane & 7];
#pragma unroll
    for (int j = 1; j < 8; ++j) k8[j] = 0ull;
    unsigned long long merged[8];
    warp_top8(k8, merged);
    if (lane < 8) {
      unsigned long long mine = merged[0];
#pragma unroll
      for (int r = 1; r < 8; ++r) mine = lane == r ? merged[r] : mine;
      S.top[lane] = mine;
    }
  }
  esync();
}

// The (r + 1)-th largest of the warp's 32 values (on every lane; r < 32): bitonic sort,
// descending by lane.
__device__ __forceinline__ float warp_rank_value(float v, int r) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float o = __shfl_xor_sync(FULL, v, j);
      const bool desc = (lane & k) == 0;
      const bool low = (lane & j) == 0;
      v = (low == desc) ? fmaxf(v, o) : fminf(v, o);
    }
  }
  return __shfl_sync(FULL, v, r);
}
__device__ __forceinline__ float warp_8th_largest(float v) { return warp_rank_value(v, 7); }

// A lower bound of the 8th largest of the elements whose per-thread maxima are m (distinct
// elements): some warp has 8 lanes whose maxima reach the largest of the warps' 8th-largest.
__device__ float team_bound(float m, RowShared& S) {
  const float w8 = warp_8th_largest(m);
  if ((threadIdx.x & 31) == 0) S.rb[et() >> 5] = w8;
  esync();
  float b = S.rb[0];
#pragma unroll
  for (int w = 1; w < NEW; ++w) b = fmaxf(b, S.rb[w]);
  esync();
  return b;
}

// ------------------------------------------------------------------------------------------
// element access and per-group values
// ------------------------------------------------------------------------------------------
// Two consecutive elements e, e+1 of a global row (e even; -inf past V); one load of both when
// the row is 16-byte aligned.
template <typename T>
__device__ __forceinline__ void ld2(const T* row, int e, int V, bool vec, float& a, float& b) {
  if (vec && e + 1 < V) {
    if constexpr (sizeof(T) == 2) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(row + e);
      a = __uint_as_float(w << 16);
      b = __uint_as_float(w & 0xFFFF0000u);
    } else {
      const float2 w = *reinterpret_cast<const float2*>(row + e);
      a = w.x;
      b = w.y;
    }
  } else {
    a = e < V ? Elt<T>::val(row[e]) : -INFINITY;
    b = e + 1 < V ? Elt<T>::val(row[e + 1]) : -INFINITY;
  }
}

// Elements of a row per ring stage.
template <typename T>
__host__ __device__ constexpr int chunk_elems() {
  return kStage / static_cast<int>(sizeof(T));
}

// Per-group values in shared memory: floats, or for the residual of bf16 rows 16-bit floats (the
// upper half of a float). A bf16 row's group maxima are bf16 values and stay exact; the log-ratio
// maxima and the bounds that replace them are upper bounds and are rounded up.
template <typename T, int MODE>
struct GroupVal {
  using type = float;
};
template <>
struct GroupVal<uint16_t, MODE_RESID> {
  using type = uint16_t;
};
__device__ __forceinline__ float gv_get(const float* a, int g) { return a[g]; }
__device__ __forceinline__ float gv_get(const uint16_t* a, int g) {
  return __uint_as_float(static_cast<uint32_t>(a[g]) << 16);
}
// v exactly (a 16-bit array takes only bf16 values here)
__device__ __forceinline__ void gv_put(float* a, int g, float v) { a[g] = v; }
__device__ __forceinline__ void gv_put(uint16_t* a, int g, float v) {
  a[g] = static_cast<uint16_t>(__float_as_uint(v) >> 16);
}
// v rounded toward +inf: a positive value with bits below the kept half goes up one unit (the
// largest finite ones to +inf); negative values lose them, which is up too; NaN stays NaN
__device__ __forceinline__ void gv_put_up(float* a, int g, float v) { a[g] = v; }
__device__ __forceinline__ void gv_put_up(uint16_t* a, int g, float v) {
  uint32_t u = __float_as_uint(v);
  if (!(u & 0x80000000u) && (u & 0xFFFFu) && !(v != v)) u += 0x10000u;
  a[g] = static_cast<uint16_t>(u >> 16);
}

// A thread's running maximum m and sum 2^(z c - fl(m c)) over the groups it has reduced.
struct RowRun {
  float m, mc, s;
  __device__ __forceinline__ void init() {
    m = -INFINITY;
    mc = -INFINITY;
    s = 0.f;
  }
  // a group with maximum g (gc = fl(g c)) and mass sm relative to gc
  __device__ __forceinline__ void add(float g, float gc, float sm) {
    const float mn = max_nan(m, g);
    if (mn != m) {
      s = (m > -INFINITY ? s * exp2f(mc - gc) : 0.f) + sm;
      m = mn;
      mc = gc;
    } else if (g > -INFINITY) {
      s += sm * exp2f(gc - mc);
    }
  }
};

// Chunk geometry per lane: EPL contiguous elements, PPL 16-byte pieces of EPP elements; a group
// of 64 elements spans LPG lanes.
template <typename T>
struct Lanes {
  static constexpr int EPL = chunk_elems<T>() / CT;
  static constexpr int EPP = 16 / static_cast<int>(sizeof(T));
  static constexpr int PPL = EPL / EPP;
  static constexpr int LPG = kGroup / EPL;
  static_assert((PPL == 2 || PPL == 4) && LPG >= 2 && LPG <= 8, "lane geometry");
  // The piece a lane reads in its j-th load: lanes take their pieces in rotated orders so that
  // the eight lanes of each shared-memory phase hit eight distinct 16-byte bank groups.
  static __device__ __forceinline__ int piece(int j, int lane) {
    return (j + (lane >> (PPL == 4 ? 1 : 2))) & (PPL - 1);
  }
};

// The lane's pieces of a staged chunk (n valid elements; elements at or past n read as -inf).
// Max and sum do not care in which order the pieces sit.
template <typename T>
__device__ __forceinline__ void load_pieces(const T* stage, int n, uint4 (&q)[Lanes<T>::PPL]) {
  using G = Lanes<T>;
  const int tid = threadIdx.x, lane = tid & 31;
  const int e_lane = G::EPL * tid;
  const uint4* src = reinterpret_cast<const uint4*>(stage) + G::PPL * tid;
#pragma unroll
  for (int j = 0; j < G::PPL; ++j) q[j] = src[G::piece(j, lane)];
  if (e_lane + G::EPL > n) {  // the row's last chunk
#pragma unroll
    for (int j = 0; j < G::PPL; ++j) {
      const int e = e_lane + G::EPP * G::piece(j, lane);
      uint32_t w[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        if constexpr (sizeof(T) == 2) {
          const uint32_t lo = e + 2 * h < n ? (w[h] & 0xFFFFu) : 0xFF80u;
          const uint32_t hi = e + 2 * h + 1 < n ? (w[h] & 0xFFFF0000u) : 0xFF800000u;
          w[h] = lo | hi;
        } else {
          w[h] = e + h < n ? w[h] : __float_as_uint(-INFINITY);
        }
      }
      q[j] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

template <typename T>
__device__ __forceinline__ void unpack_piece(const uint4& q, float (&z)[16 / sizeof(T)]) {
  if constexpr (sizeof(T) == 2) {
    Elt<uint16_t>::unpack(q, z);
  } else {
    z[0] = __uint_as_float(q.x);
    z[1] = __uint_as_float(q.y);
    z[2] = __uint_as_float(q.z);
    z[3] = __uint_as_float(q.w);
  }
}

// Maximum over the lane's pieces.
template <typename T>
__device__ __forceinline__ float pieces_max(const uint4 (&q)[Lanes<T>::PPL]) {
  if constexpr (sizeof(T) == 2) {
    uint32_t mx = 0xFF80FF80u;
#pragma unroll
    for (int j = 0; j < Lanes<T>::PPL; ++j)
      mx = max_nan_bf16x2(mx, max_nan_bf16x2(max_nan_bf16x2(q[j].x, q[j].y),
                                             max_nan_bf16x2(q[j].z, q[j].w)));
    return max_nan(__uint_as_float(mx << 16), __uint_as_float(mx & 0xFFFF0000u));
  } else {
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < Lanes<T>::PPL; ++j)
      m = max_nan(max_nan(m, max_nan(__uint_as_float(q[j].x), __uint_as_float(q[j].y))),
                  max_nan(__uint_as_float(q[j].z), __uint_as_float(q[j].w)));
    return m;
  }
}

// Sum of 2^(z c - gc) over the lane's pieces, two elements per packed instruction.
template <typename T>
__device__ __forceinline__ float pieces_mass(const uint4 (&q)[Lanes<T>::PPL], float c, float gc) {
  const float2 c2 = make_float2(c, c), n2 = make_float2(-gc, -gc);
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < Lanes<T>::PPL; ++j) {
    float z[Lanes<T>::EPP];
    unpack_piece<T>(q[j], z);
#pragma unroll
    for (int k = 0; k < Lanes<T>::EPP; k += 2) {
      const float2 a = __ffma2_rn(make_float2(z[k], z[k + 1]), c2, n2);
      acc = __fadd2_rn(acc, make_float2(ex2_fast(a.x), ex2_fast(a.y)));
    }
  }
  return acc.x + acc.y;
}

template <int LPG>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = 1; o < LPG; o <<= 1) v = max_nan(v, __shfl_xor_sync(FULL, v, o));
  return v;
}
template <int LPG>
__device__ __forceinline__ float group_fmax(float v) {
#pragma unroll
  for (int o = 1; o < LPG; o <<= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
  return v;
}
template <int LPG>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = 1; o < LPG; o <<= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

// Group maxima and masses of one staged chunk (n valid elements) into gmax / gmass at the
// chunk's first group; the groups also go into the thread's running row stats. Returns the
// lane's group maximum (every lane of the group holds it).
template <typename T>
__device__ __forceinline__ float chunk_groups(const T* stage, int n, float c, float* gmax,
                                              float* gmass, RowRun& run) {
  using G = Lanes<T>;
  const int tid = threadIdx.x, lane = tid & 31;
  uint4 q[G::PPL];
  load_pieces<T>(stage, n, q);
  const float g = group_max<G::LPG>(pieces_max<T>(q));
  const float gc = __fmul_rn(g, c);
  const float sm = group_sum<G::LPG>(g > -INFINITY ? pieces_mass<T>(q, c, gc) : 0.f);
  if ((lane & (G::LPG - 1)) == 0 && G::EPL * tid < n) {
    gmax[tid / G::LPG] = g;
    gmass[tid / G::LPG] = sm;
    run.add(g, gc, sm);
  }
  return g;
}

// Group maxima only (the top-8 prepass), and the row maximum in the thread's running stats.
template <typename T>
__device__ __forceinline__ void chunk_maxima(const T* stage, int n, float c, float* gmax,
                                             RowRun& run) {
  using G = Lanes<T>;
  const int tid = threadIdx.x, lane = tid & 31;
  uint4 q[G::PPL];
  load_pieces<T>(stage, n, q);
  const float g = group_max<G::LPG>(pieces_max<T>(q));
  if ((lane & (G::LPG - 1)) == 0 && G::EPL * tid < n) {
    gmax[tid / G::LPG] = g;
    run.add(g, __fmul_rn(g, c), 0.f);
  }
}

// Residual chunks: the same for a target and a draft chunk at once (n valid elements each), plus
// each group's largest log-ratio max (z_t - z_d), which bounds the group's residual from above
// once the normalisers are known.
template <typename T, typename GV>
__device__ __forceinline__ void chunk_pair(const T* st_t, const T* st_d, int n, float c,
                                           GV* gmax_t, GV* gmax_d, GV* gdel, RowRun& run_t,
                                           RowRun& run_d) {
  using G = Lanes<T>;
  const int tid = threadIdx.x, lane = tid & 31;
  uint4 qt[G::PPL], qd[G::PPL];
  load_pieces<T>(st_t, n, qt);
  load_pieces<T>(st_d, n, qd);
  float dl = -INFINITY;
  if constexpr (sizeof(T) == 2) {
    // the largest difference of packed bf16 pairs (-inf - -inf is NaN, which the plain max
    // ignores), rounded to bf16 and corrected upward: a bf16 difference is within half a unit
    // in the last place (2^-8 relative) of the exact one
    uint32_t xl = 0xFF80FF80u;
#pragma unroll
    for (int j = 0; j < G::PPL; ++j) {
      xl = max_bf16x2(xl, sub_bf16x2(qt[j].x, qd[j].x));
      xl = max_bf16x2(xl, sub_bf16x2(qt[j].y, qd[j].y));
      xl = max_bf16x2(xl, sub_bf16x2(qt[j].z, qd[j].z));
      xl = max_bf16x2(xl, sub_bf16x2(qt[j].w, qd[j].w));
    }
    dl = fmaxf(__uint_as_float(xl << 16), __uint_as_float(xl & 0xFFFF0000u));
    dl = dl + fabsf(dl) * 0.0078125f;
  } else {
#pragma unroll
    for (int j = 0; j < G::PPL; ++j) {
      // (-inf - -inf is NaN, which fmaxf ignores; a finite target over a -inf draft is +inf)
      dl = fmaxf(dl, __uint_as_float(qt[j].x) - __uint_as_float(qd[j].x));
      dl = fmaxf(dl, __uint_as_float(qt[j].y) - __uint_as_float(qd[j].y));
      dl = fmaxf(dl, __uint_as_float(qt[j].z) - __uint_as_float(qd[j].z));
      dl = fmaxf(dl, __uint_as_float(qt[j].w) - __uint_as_float(qd[j].w));
    }
  }
  const float gt = group_max<G::LPG>(pieces_max<T>(qt));
  const float gd = group_max<G::LPG>(pieces_max<T>(qd));
  const float gl = group_fmax<G::LPG>(dl);
  const float gtc = __fmul_rn(gt, c), gdc = __fmul_rn(gd, c);
  const float smt = group_sum<G::LPG>(gt > -INFINITY ? pieces_mass<T>(qt, c, gtc) : 0.f);
  const float smd = group_sum<G::LPG>(gd > -INFINITY ? pieces_mass<T>(qd, c, gdc) : 0.f);
  if ((lane & (G::LPG - 1)) == 0 && G::EPL * tid < n) {
    gv_put(gmax_t, tid / G::LPG, gt);
    gv_put(gmax_d, tid / G::LPG, gd);
    gv_put_up(gdel, tid / G::LPG, gl);
    run_t.add(gt, gtc, smt);
    run_d.add(gd, gdc, smd);
  }
}

// The chunk threads' running stats into a row maximum and sum 2^(z c - M c) (rounding of
// fl(M c) folded in), written to *hdr by chunk thread 0. Every chunk thread calls it.
__device__ void chunk_row_stats(const RowRun& run, float c, RowShared& S, float* hdr) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float M = warp_max_nan(run.m);
  const float Mc = __fmul_rn(M, c);
  const float part = (run.m > -INFINITY && !row_bad(M)) ? run.s * exp2f(run.mc - Mc) : 0.f;
  const float sw = warp_sum(part);
  if (lane == 0) {
    S.cm[warp] = M;
    S.cs[warp] = sw;
  }
  named_sync(kBarC, CT);
  if (threadIdx.x == 0) {
    float Mt = S.cm[0];
    for (int w = 1; w < NCW; ++w) Mt = max_nan(Mt, S.cm[w]);
    float St = 0.f;
    if (!row_bad(Mt)) {
      const float Mtc = __fmul_rn(Mt, c);
      for (int w = 0; w < NCW; ++w)
        if (S.cm[w] > -INFINITY) St += S.cs[w] * exp2f(__fmul_rn(S.cm[w], c) - Mtc);
      St *= fmaf(-fmaf(Mt, c, -Mtc), kLn2r, 1.f);
    }
    hdr[0] = Mt;
    hdr[1] = St;
  }
  named_sync(kBarC, CT);  // the scratch is free again
}

// The row's top-8 elements (the bias set's candidates) into S.top, in two steps so that the
// group reads can overlap other work. They lie in the 8 groups with the largest maxima (ties to
// the lower group): an element outside them is beaten by those 8 maxima.
//  - top8_groups: the 8 groups from the group maxima alone (only those at or above a lower bound
//    of the 8th are offered); each epilogue warp then starts reading its two of them (G8);
//  - top8_elements: their elements offered, from the 8th group maximum up (nothing below it can
//    be among the 8 largest: the 8 groups' maxima reach it).
struct G8 {
  int g0, g1;
  float a0, b0, a1, b1;
  float thr;
};

template <typename T, typename GV>
__device__ G8 top8_groups(const T* row, int V, bool vec, const GV* gmax, int ng, RowShared& S) {
  const int t = et(), lane = t & 31, warp = t >> 5;
  float m = -INFINITY;
  for (int g = t; g < ng; g += ET) m = fmaxf(m, gv_get(gmax, g));
  const float B = team_bound(m, S);
  WarpTop8 gtop;
  gtop.init(B);
  const int per = (ng + ET - 1) / ET;
  for (int k = 0; k < per; ++k) {
    const int g = t + k * ET;
    const float v = g < ng ? gv_get(gmax, g) : -INFINITY;
    gtop.offer(g < ng && v >= B, v, static_cast<uint32_t>(g));
  }
  team_top8(gtop, S);
  static_assert(NEW * 2 == 8, "two groups per epilogue warp");
  const unsigned long long k0 = S.top[2 * warp], k1 = S.top[2 * warp + 1], k7 = S.top[7];
  esync();  // S.top is read by every warp before it is rewritten
  G8 r;
  r.g0 = k0 ? key_id(k0) : -1;
  r.g1 = k1 ? key_id(k1) : -1;
  r.thr = k7 ? key_value(k7) : -INFINITY;
  r.a0 = r.b0 = r.a1 = r.b1 = -INFINITY;
  if (r.g0 >= 0) ld2<T>(row, kGroup * r.g0 + 2 * lane, V, vec, r.a0, r.b0);
  if (r.g1 >= 0) ld2<T>(row, kGroup * r.g1 + 2 * lane, V, vec, r.a1, r.b1);
  return r;
}

__device__ void top8_elements(const G8& r, int V, RowShared& S) {
  const int lane = threadIdx.x & 31;
  WarpTop8 top;
  top.init(r.thr);
  const int e0 = kGroup * r.g0 + 2 * lane, e1 = kGroup * r.g1 + 2 * lane;
  top.offer(r.g0 >= 0 && e0 < V, r.a0, static_cast<uint32_t>(e0));
  top.offer(r.g0 >= 0 && e0 + 1 < V, r.b0, static_cast<uint32_t>(e0 + 1));
  top.offer(r.g1 >= 0 && e1 < V, r.a1, static_cast<uint32_t>(e1));
  top.offer(r.g1 >= 0 && e1 + 1 < V, r.b1, static_cast<uint32_t>(e1 + 1));
  team_top8(top, S);
}

template <typename T, typename GV>
__device__ void row_top8(const T* row, int V, bool vec, const GV* gmax, int ng, RowShared& S) {
  top8_elements(top8_groups<T>(row, V, vec, gmax, ng, S), V, S);
}

// The Saguaro bias set (the bias_k largest draft logits, from S.top) and the renormalisation
// N = 1 - (1 - beta) sum_S q, the terms summed in key order. Epilogue warp 0.
__device__ void bias_set(const RowParams& P, RowShared& S, float Md, float Sd) {
  if (et() >= 32) return;
  const int lane = et();
  const unsigned long long k = lane < 8 ? S.top[lane] : 0ull;
  const bool in = lane < P.bias_k && k != 0ull;
  const float z = in ? key_value(k) : 0.f;
  const float term = in ? exp2f((z - Md) * P.c) / Sd : 0.f;
  const int nS = __popc(__ballot_sync(FULL, in));
  float sq = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float tj = __shfl_sync(FULL, term, j);
    if (j < nS) sq += tj;
  }
  if (in) {
    S.S_z[lane] = z;
    S.S_ids[lane] = key_id(k);
    S.sgrp[lane] = key_id(k) / kGroup;
  }
  if (lane == 0) {
    S.nS = nS;
    S.N = fmaf(-(1.f - P.beta), sq, 1.f);
  }
}

// ------------------------------------------------------------------------------------------
// the producer: units from the queue, their rows through the ring
// ------------------------------------------------------------------------------------------
template <typename T, int MODE>
__device__ void producer(const RowParams& P, RowShared& S, unsigned char* ring) {
  const int lane = threadIdx.x & 31;
  const int nst = P.nstages;
  constexpr int CE = chunk_elems<T>();
  const int nch = (P.V + CE - 1) / CE;
  const int nunits = MODE == MODE_SAMPLE ? P.B : P.B * P.K;
  const bool vec = P.use_vec != 0;
  int it = 0;  // stage fills so far
  bool ok = true;
  while (ok) {
    int u = 0;
    if (lane == 0) u = static_cast<int>(atomicAdd(&P.ws->next, 1u));
    u = __shfl_sync(FULL, u, 0);
    if (u >= nunits) break;
    // residual units are taken position by position across the sequences: the first positions,
    // which want the most ids (F_i falls with i) and whose epilogues read the most groups, go
    // while the stream still hides their epilogues; the last units taken want few
    if (MODE == MODE_RESID) u = (u % P.B) * P.K + u / P.B;
    const T* rows[2] = {nullptr, nullptr};
    int nrows = 1;
    if (MODE == MODE_SAMPLE) {
      rows[0] = static_cast<const T*>(P.dft) + static_cast<long long>(u) * P.d_stride;
    } else if (MODE == MODE_TOP8) {
      const int b = u / P.K, i = u % P.K;
      const int L = P.lens ? P.lens[b] : P.K;
      if (L < 1 || L > P.K || i >= L) continue;  // a row the verify step never asks about
      rows[0] = static_cast<const T*>(P.dft) + (static_cast<long long>(b) * P.K + i) * P.d_stride;
    } else {
      const int b = u / P.K, i = u % P.K;
      const int L = P.lens ? P.lens[b] : P.K;
      if (L < 1 || L > P.K || i >= L) {  // no residual here: its ids are -1
        if (lane < P.fmax) P.out_r2[static_cast<long long>(u) * P.fmax + lane] = -1;
        // a sequence of invalid length has no cache-hit flag (its first unit writes it)
        if (i == 0 && P.out_hit && lane == 0) P.out_hit[b] = -1;
        continue;
      }
      rows[0] = static_cast<const T*>(P.tgt) +
                (static_cast<long long>(b) * (P.K + 1) + i) * P.t_stride;
      rows[1] = static_cast<const T*>(P.dft) + (static_cast<long long>(b) * P.K + i) * P.d_stride;
      nrows = 2;
    }
    for (int ch = 0; ch < nch && ok; ++ch) {
      const int e0 = ch * CE;
      const int n = min(CE, P.V - e0);
      const int npad = (n + 7) & ~7;
      for (int r = 0; r < nrows && ok; ++r) {
        const int s = it % nst;
        // the chunk warps must have released the stage's previous fill
        if (it >= nst && !mbar_wait_bounded(&S.empty[s], ((it / nst) - 1) & 1, kWaitBudget)) {
          ok = false;
          if (lane == 0) atomicOr(&P.ws->error, 1u);
          break;
        }
        T* st = reinterpret_cast<T*>(ring + static_cast<size_t>(s) * kStage);
        const T* src = rows[r] + e0;
        if (vec) {
          // whole 16-byte units by one bulk copy; the last few elements and the padding by hand
          const int nb = static_cast<int>((static_cast<size_t>(n) * sizeof(T)) &
                                          ~static_cast<size_t>(15)) /
                         static_cast<int>(sizeof(T));
          for (int e = nb + lane; e < npad; e += 32) st[e] = e < n ? src[e] : Elt<T>::neg_inf();
          __syncwarp();
          if (lane == 0) {
            S.tag[s] = u;
            const uint32_t bytes = static_cast<uint32_t>(nb * sizeof(T));
            mbar_arrive_expect_tx(&S.full[s], bytes);
            if (bytes) bulk_g2s(st, src, bytes, &S.full[s]);
          }
        } else {
          for (int e = lane; e < npad; e += 32) st[e] = e < n ? src[e] : Elt<T>::neg_inf();
          __syncwarp();
          if (lane == 0) {
            S.tag[s] = u;
            mbar_arrive(&S.full[s]);
          }
        }
        ++it;
      }
    }
  }
  if (ok) {  // the end marker
    const int s = it % nst;
    if (it >= nst && !mbar_wait_bounded(&S.empty[s], ((it / nst) - 1) & 1, kWaitBudget)) {
      ok = false;
      if (lane == 0) atomicOr(&P.ws->error, 1u);
    } else {
      if (lane == 0) {
        S.tag[s] = kEnd;
        mbar_arrive(&S.full[s]);
      }
      ++it;
    }
  }
  if (!ok) {
    // a wait gave up: let the copies already issued land before leaving (bounded)
    for (int j = max(0, it - nst); j < it; ++j)
      mbar_wait_bounded(&S.full[j % nst], (j / nst) & 1, kWaitBudget);
  }
  // the queue is reset by the last CTA to stop taking units
  if (lane == 0) {
    __threadfence();
    const unsigned old = atomicAdd(&P.ws->done, 1u);
    if (old == gridDim.x - 1u) {
      atomicExch(&P.ws->next, 0u);
      atomicExch(&P.ws->done, 0u);
    }
  }
}

// ------------------------------------------------------------------------------------------
// the chunk warps: group values of every unit into the two group buffers in turn
// ------------------------------------------------------------------------------------------
template <typename T, int MODE>
__device__ void chunk_warps(const RowParams& P, RowShared& S, unsigned char* ring,
                            unsigned char* gbuf0, unsigned char* gbuf1, int ngmax) {
  using GV = typename GroupVal<T, MODE>::type;
  const int tid = threadIdx.x, lane = tid & 31;
  const int nst = P.nstages;
  constexpr int CE = chunk_elems<T>();
  const int nch = (P.V + CE - 1) / CE;
  int it = 0;        // ring stages taken
  int k = 0;         // units finished
  bool ab = false;   // a wait gave up: stop waiting (what is read from here on is meaningless)
  // wait for stage use number j (it, it + 1, ...) to be filled; returns its stage
  auto wait_full = [&](int j) {
    const int s = j % nst;
    if (!ab && !mbar_wait_bounded(&S.full[s], (j / nst) & 1, kWaitBudget)) {
      ab = true;
      atomicOr(&P.ws->error, 1u);
    }
    return s;
  };
  auto release = [&](int s) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);
    ++it;
  };
  // the group buffer of unit k, once the epilogue is done with unit k - 2
  auto take_buffer = [&]() {
    const int b = k & 1;
    if (k >= 2 && !ab && !mbar_wait_bounded(&S.gfree[b], ((k >> 1) - 1) & 1, kWaitBudget)) {
      ab = true;
      atomicOr(&P.ws->error, 1u);
    }
    return b;
  };
  auto hand_over = [&](int b, int u) {
    if (tid == 0) S.gunit[b] = u;
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.gfull[b]);
  };
  for (;;) {
    const int s0 = wait_full(it);
    const int u = S.tag[s0];
    if (named_sync_or(kBarC, CT, ab || u == kEnd)) break;
    const int b = take_buffer();
    float* gb = reinterpret_cast<float*>(b ? gbuf1 : gbuf0);
    GV* gv = reinterpret_cast<GV*>(b ? gbuf1 : gbuf0);
    RowRun run[2];
    run[0].init();
    run[1].init();
    const int go = CE / kGroup;  // groups per chunk
    for (int ch = 0; ch < nch; ++ch) {
      const int n = min(CE, P.V - ch * CE);
      const int s = ch == 0 ? s0 : wait_full(it);
      const T* st = reinterpret_cast<const T*>(ring + static_cast<size_t>(s) * kStage);
      if (MODE == MODE_SAMPLE) {  // maxima, then masses
        chunk_groups<T>(st, n, P.c, gb + ch * go, gb + ngmax + ch * go, run[0]);
        release(s);
      } else if (MODE == MODE_TOP8) {  // maxima
        chunk_maxima<T>(st, n, P.c, gb + ch * go, run[0]);
        release(s);
      } else {  // target maxima, draft maxima, log-ratio maxima
        const int s2 = wait_full(it + 1);
        chunk_pair<T>(st, reinterpret_cast<const T*>(ring + static_cast<size_t>(s2) * kStage), n,
                      P.c, gv + ch * go, gv + ngmax + ch * go, gv + 2 * ngmax + ch * go, run[0],
                      run[1]);
        release(s);
        release(s2);
      }
    }
    chunk_row_stats(run[0], P.c, S, &S.hdr[b][0]);
    if (MODE == MODE_RESID) chunk_row_stats(run[1], P.c, S, &S.hdr[b][2]);
    hand_over(b, u);
    ++k;
  }
  hand_over(take_buffer(), kEnd);  // no more units
}

// ------------------------------------------------------------------------------------------
// reads of whole groups of a global row
// ------------------------------------------------------------------------------------------
// The 16-byte piece of a global row at element e (a multiple of 16 / sizeof(T)): one vector load
// when the row is 16-byte aligned and the piece lies below V, else element by element; elements
// at or past V, and every element when e < 0, read as -inf.
template <typename T>
__device__ __forceinline__ uint4 row_piece(const T* row, int e, int V, bool vec) {
  constexpr int EPP = 16 / static_cast<int>(sizeof(T));
  if (e >= 0 && vec && e + EPP <= V) return ldg_nc_v4(row + e);
  uint32_t w[4];
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    if constexpr (sizeof(T) == 2) {
      const uint32_t lo = (e >= 0 && e + 2 * h < V) ? static_cast<uint32_t>(row[e + 2 * h]) : 0xFF80u;
      const uint32_t hi =
          (e >= 0 && e + 2 * h + 1 < V) ? static_cast<uint32_t>(row[e + 2 * h + 1]) : 0xFF80u;
      w[h] = lo | (hi << 16);
    } else {
      w[h] = (e >= 0 && e + h < V) ? __float_as_uint(row[e + h]) : __float_as_uint(-INFINITY);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// How a warp reads groups of a global row: 16-byte pieces of EPP elements, PPG pieces per group,
// GPL groups per warp-wide load; lane l takes piece l mod PPG of group slot l / PPG.
template <typename T>
struct GroupReads {
  static constexpr int EPP = 16 / static_cast<int>(sizeof(T));
  static constexpr int PPG = kGroup / EPP;
  static constexpr int GPL = 32 / PPG;
  static constexpr int NL = kBatch / GPL;  // loads per row and lane for kBatch groups
  static_assert(GPL * PPG == 32 && NL * GPL == kBatch, "group reads");
};

// Warp 0: the 8 largest elements of the n (<= kCandCap) candidate groups in S.cand (keys of group
// maxima), as keys on lanes 0..7, descending (0 where fewer; 0 on the other lanes). The 8 largest
// groups are read at once.
template <typename T>
__device__ unsigned long long warp_top8_of_candidates(RowShared& S, int n, const T* row, int V,
                                                     bool vec) {
  const int lane = threadIdx.x & 31;
  static_assert(kCandCap == 64, "two candidates per lane");
  unsigned long long a = lane < n ? S.cand[lane] : 0ull;
  unsigned long long b = lane + 32 < n ? S.cand[lane + 32] : 0ull;
  if (b > a) {
    const unsigned long long x = a;
    a = b;
    b = x;
  }
  unsigned long long gk = 0ull;  // lane r: the r-th largest group key
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const unsigned long long m = warp_max_key(a);
    if (lane == r) gk = m;
    if (m != 0ull && a == m) {
      a = b;
      b = 0ull;
    }
  }
  const unsigned long long k7 = __shfl_sync(FULL, gk, 7);
  using R = GroupReads<T>;
  constexpr int NP = 8 * R::PPG / 32;  // pieces per lane
  uint4 q[NP];
  int e[NP];
#pragma unroll
  for (int j = 0; j < NP; ++j) {
    const int p = lane + 32 * j;
    const unsigned long long kg = __shfl_sync(FULL, gk, p / R::PPG);
    e[j] = kg ? kGroup * key_id(kg) + R::EPP * (p % R::PPG) : -1;
    q[j] = row_piece<T>(row, e[j], V, vec);
  }
  // Each of the 8 groups holds an element at or above the 8th group maximum t8 (its own
  // maximum). When they are the only 8 such elements, the r-th largest element is the maximum
  // of the group of rank r (groups of equal maxima rank by index, as their ids do); otherwise
  // the elements from t8 up go through a list.
  const float t8 = k7 ? key_value(k7) : -INFINITY;
  float ze[NP][R::EPP];
  int cnt = 0;
#pragma unroll
  for (int j = 0; j < NP; ++j) {
    unpack_piece<T>(q[j], ze[j]);
#pragma unroll
    for (int kk = 0; kk < R::EPP; ++kk)
      cnt += (e[j] >= 0 && e[j] + kk < V && ze[j][kk] >= t8) ? 1 : 0;
  }
  unsigned long long k = 0ull;  // lanes 0..7: the 8 largest, descending; 0 elsewhere
  if (k7 != 0ull && __reduce_add_sync(FULL, cnt) == 8) {
#pragma unroll
    for (int j = 0; j < NP; ++j)
#pragma unroll
      for (int kk = 0; kk < R::EPP; ++kk)
        if (e[j] >= 0 && e[j] + kk < V && ze[j][kk] >= t8)
          S.wtop[0][(lane + 32 * j) / R::PPG] =
              make_key(ze[j][kk], static_cast<uint32_t>(e[j] + kk));
    __syncwarp();
    k = lane < 8 ? S.wtop[0][lane] : 0ull;
  } else {
    WarpTop8 top;
    top.init(t8);
#pragma unroll
    for (int j = 0; j < NP; ++j)
#pragma unroll
      for (int kk = 0; kk < R::EPP; ++kk)
        top.offer(e[j] >= 0 && e[j] + kk < V, ze[j][kk], static_cast<uint32_t>(e[j] + kk));
    k = top.L;
  }
  return k;
}

// ------------------------------------------------------------------------------------------
// epilogue: sampling
// ------------------------------------------------------------------------------------------
// Warp 0 of the sampling epilogue: the bias set (the bias_k largest of the row's 8 largest, keys k
// on lanes 0..7) into S (nS, S_ids, S_z, sgrp), and beta applied to the masses of the groups that
// hold its ids: the lane of the first id of each such group (in set order) rescales the group's
// mass by its ids from there on and records the change of its fixed-point value (S.dg, S.dq).
__device__ void sample_set(const RowParams& P, RowShared& S, unsigned long long k, float* gmass,
                           float Mdc) {
  const int lane = threadIdx.x & 31;
  const bool in = lane < P.bias_k && lane < 8 && k != 0ull;
  const int nS = __popc(__ballot_sync(FULL, in));
  const int id = in ? key_id(k) : -1;
  const float z = in ? key_value(k) : 0.f;
  const int g = in ? id / kGroup : -1;
  if (in) {
    S.S_ids[lane] = id;
    S.S_z[lane] = z;
    S.sgrp[lane] = g;
  }
  if (lane == 0) S.nS = nS;
  bool first = in;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int gi = __shfl_sync(FULL, g, i);
    if (i < lane && gi == g) first = false;
  }
  float w = first ? gmass[g] : 0.f;
  const unsigned long long before = qfix(w);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int gi = __shfl_sync(FULL, g, i);
    const float zi = __shfl_sync(FULL, z, i);
    if (first && i >= lane && i < nS && gi == g)
      w = fmaxf(fmaf(P.beta - 1.f, ex2_fast(fmaf(zi, P.c, -Mdc)), w), 0.f);
  }
  if (first) gmass[g] = w;
  if (lane < 8) {
    S.dg[lane] = first ? g : -1;
    S.dq[lane] = first ? static_cast<long long>(qfix(w) - before) : 0ll;
  }
}

template <typename T, bool BIAS>
__device__ void sample_epilogue(const RowParams& P, RowShared& S, int u, float* gmax,
                                float* gmass, const float* hdr) {
  const int t = et(), lane = t & 31;
  const float c = P.c;
  const int V = P.V;
  const int ng = (V + kGroup - 1) / kGroup;
  const T* row = static_cast<const T*>(P.dft) + static_cast<long long>(u) * P.d_stride;
  const bool vec = P.use_vec != 0;

  const float M = hdr[0], Sd = hdr[1];
  if (row_bad(M)) {
    if (t == 0) {
      P.out_tok[u] = -1;
      P.out_conf[u] = NAN;
      if (P.out_exit) P.out_exit[u] = -1;
    }
    return;
  }
  int nS = 0;
  // group masses relative to the row maximum, over contiguous runs of groups per thread (so that
  // the prefix of the inverse CDF follows the ids): fixed-point run totals, the run's largest
  // group maximum and its group
  const float Mdc = __fmul_rn(M, c);
  const int lo = static_cast<int>((static_cast<long long>(t) * ng) / ET);
  const int hi = static_cast<int>((static_cast<long long>(t + 1) * ng) / ET);
  unsigned long long csum = 0;
  float tmax = -INFINITY;
  int gtop = -1;
#pragma unroll 4
  for (int g = lo; g < hi; ++g) {
    const float gm = gmax[g];
    if (gm > tmax) {
      tmax = gm;
      gtop = g;
    }
    const float w = gm > -INFINITY ? gmass[g] * exp2f(__fmul_rn(gm, c) - Mdc) : 0.f;
    gmass[g] = w;
    csum += qfix(w);
  }
  unsigned long long W = 0, pre = 0;
  if (BIAS) {
    // The bias set: its 8 elements lie in the 8 groups with the largest maxima, those in the runs
    // whose maximum reaches a lower bound of the 8th largest run maximum, and there at or above
    // it (the candidates, listed while the prefix runs). Each run's largest group is fetched into
    // L2 meanwhile; most of the 8 are among them. Warp 0 then finds the set and its corrections.
    if (gtop >= 0)
      for (int o = 0; o < kGroup && kGroup * gtop + o < V; o += 128 / static_cast<int>(sizeof(T)))
        prefetch_l2(row + kGroup * gtop + o);
    if (t == 0) S.ncand = 0;
    const float th = team_bound(tmax, S);  // (its barriers order the reset before the adds)
    if (tmax >= th)
      for (int g = lo; g < hi; ++g) {
        const float v = gmax[g];
        if (v >= th) {
          const int k = atomicAdd(&S.ncand, 1);
          if (k < kCandCap) S.cand[k] = make_key(v, static_cast<uint32_t>(g));
        }
      }
    pre = team_exclusive_u64(csum, S, &W);  // (its barriers publish gmass and the candidates)
    const int n = S.ncand;
    if (n > kCandCap) {  // (ties beyond the list) every group offered
      top8_elements(top8_groups<T>(row, V, vec, gmax, ng, S), V, S);
      if (t < 32) sample_set(P, S, t < 8 ? S.top[t] : 0ull, gmass, Mdc);
    } else if (t < 32) {
      sample_set(P, S, warp_top8_of_candidates<T>(S, n, row, V, vec), gmass, Mdc);
    }
    esync();
    nS = S.nS;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int g = S.dg[j];
      if (g < 0) continue;
      const unsigned long long d = static_cast<unsigned long long>(S.dq[j]);
      W += d;
      if (g < lo) pre += d;
      else if (g < hi) csum += d;
    }
  } else {
    pre = team_exclusive_u64(csum, S, &W);  // (its barriers publish gmass)
  }
  const float uu = P.uni[u];
  const bool uok = uu >= 0.f && uu < 1.f;
  const unsigned long long tt = scale_floor(uu, W);
  if (t == 0) S.gstar = -1;
  esync();
  if (uok && pre <= tt && tt < pre + csum) {
    for (int g = lo; g < hi; ++g) {
      const unsigned long long q = qfix(gmass[g]);
      if (pre + q > tt) {
        S.gstar = g;
        S.t_loc = tt - pre;
        break;
      }
      pre += q;
    }
  }
  esync();
  // warp 0 of the team: the element within the group, by a warp prefix over its 64 weights
  if (t < 32) {
    const int gs = S.gstar;
    int token = -1;
    if (gs >= 0) {
      const unsigned long long tl = S.t_loc;
      const int e = kGroup * gs + 2 * lane;
      float a, b;
      ld2<T>(row, e, V, vec, a, b);
      float fa = 1.f, fb = 1.f;
      for (int j = 0; j < nS; ++j) {
        fa = S.S_ids[j] == e ? P.beta : fa;
        fb = S.S_ids[j] == e + 1 ? P.beta : fb;
      }
      const float wa = e < V ? fa * ex2_fast(fmaf(a, c, -Mdc)) : 0.f;
      const float wb = e + 1 < V ? fb * ex2_fast(fmaf(b, c, -Mdc)) : 0.f;
      const float pair = wa + wb;
      float inc = pair;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(FULL, inc, o);
        if (lane >= o) inc += y;
      }
      const float pa = inc - pair + wa;
      const unsigned hit_b = __ballot_sync(FULL, qfix(inc) > tl);
      const unsigned hit_a = __ballot_sync(FULL, qfix(pa) > tl);
      const unsigned pos_b = __ballot_sync(FULL, wb > 0.f), pos_a = __ballot_sync(FULL, wa > 0.f);
      if (hit_b) {
        const int l = __ffs(hit_b) - 1;
        token = kGroup * gs + 2 * l + (((hit_a >> l) & 1u) ? 0 : 1);
      } else {  // rounding left t past the recomputed total: the last element with weight
        const int lb = pos_b ? 31 - __clz(pos_b) : -1, la = pos_a ? 31 - __clz(pos_a) : -1;
        token = (lb >= 0 && lb >= la) ? kGroup * gs + 2 * lb + 1
                                      : (la >= 0 ? kGroup * gs + 2 * la : -1);
      }
    }
    if (lane == 0) {
      P.out_tok[u] = token;
      const float conf = 1.f / Sd;  // the unbiased softmax's largest probability
      P.out_conf[u] = conf;
      if (P.out_exit) P.out_exit[u] = conf < P.tau ? 1 : 0;
    }
  }
}

// ------------------------------------------------------------------------------------------
// epilogue: exact-residual top-F
// ------------------------------------------------------------------------------------------
// The bias set of a residual unit (the draft row's bias_k largest logits) and N, into S (nS, N,
// S_ids and sgrp, the groups of those ids) for every epilogue thread. The 8 largest logits lie in
// the 8 groups with the largest maxima (ties to the lower group), those groups in the runs (the
// threads' contiguous stretches of groups) whose maximum reaches a lower bound of the 8th largest
// run maximum, and there at or above that bound: the candidates. Warp 0 keeps the 8 largest
// candidates, reads their 512 elements at once, keeps the 8 largest of them (from the 8th group
// maximum up) and forms the set, its terms summed in key order.
template <typename T, typename GV>
__device__ void resid_bias_set(const RowParams& P, RowShared& S, const GV* gmax, int ng,
                               const T* row, int V, bool vec, float Md, float Sd) {
  const int t = et(), lane = t & 31, warp = t >> 5;
  const int lo = static_cast<int>((static_cast<long long>(t) * ng) / ET);
  const int hi = static_cast<int>((static_cast<long long>(t + 1) * ng) / ET);
  float tmax = -INFINITY;
  int gm = -1;
  for (int g = lo; g < hi; ++g) {
    const float v = gv_get(gmax, g);
    if (v > tmax) {
      tmax = v;
      gm = g;
    }
  }
  // the groups warp 0 reads below are mostly the maxima of some runs: into L2 meanwhile
  if (gm >= 0)
    for (int o = 0; o < kGroup && kGroup * gm + o < V; o += 128 / static_cast<int>(sizeof(T)))
      prefetch_l2(row + kGroup * gm + o);
  if (t == 0) S.ncand = 0;
  const float th = team_bound(tmax, S);  // (its barriers order the reset before the adds)
  if (tmax >= th)
    for (int g = lo; g < hi; ++g) {
      const float v = gv_get(gmax, g);
      if (v >= th) {
        const int k = atomicAdd(&S.ncand, 1);
        if (k < kCandCap) S.cand[k] = make_key(v, static_cast<uint32_t>(g));
      }
    }
  esync();
  const int n = S.ncand;
  if (n > kCandCap) {  // (ties beyond the list) every group offered
    top8_elements(top8_groups<T>(row, V, vec, gmax, ng, S), V, S);
    bias_set(P, S, Md, Sd);
    esync();
    return;
  }
  if (warp == 0) {
    const unsigned long long k = warp_top8_of_candidates<T>(S, n, row, V, vec);
    const bool in = lane < P.bias_k && k != 0ull;
    const float z = in ? key_value(k) : 0.f;
    const float term = in ? exp2f((z - Md) * P.c) / Sd : 0.f;
    const int nS = __popc(__ballot_sync(FULL, in));
    float sq = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float tj = __shfl_sync(FULL, term, j);
      if (j < nS) sq += tj;
    }
    if (in) {
      S.S_z[lane] = z;
      S.S_ids[lane] = key_id(k);
      S.sgrp[lane] = key_id(k) / kGroup;
    }
    if (lane == 0) {
      S.nS = nS;
      S.N = fmaf(-(1.f - P.beta), sq, 1.f);
    }
  }
  esync();
}

// Residual weights of up to kBatch groups, list[j0 .. min(j0 + kBatch, n)), offered to the warp's
// list; every load is issued before the first use, so the batch costs one round trip.
template <typename T, bool BIAS>
__device__ __forceinline__ void offer_groups(WarpTop8& top, const T* zt, const T* zd,
                                             const int* list, int j0, int n, int V, bool vec,
                                             float c, float Mtc, float Mdc, float rho, float rhoS,
                                             const RowShared& S, int nS) {
  using R = GroupReads<T>;
  const int lane = threadIdx.x & 31;
  const int slot = lane / R::PPG, piece = lane % R::PPG;
  uint4 qt[R::NL], qd[R::NL];
  int e[R::NL];
#pragma unroll
  for (int j = 0; j < R::NL; ++j) {
    const int at = j0 + j * R::GPL + slot;
    e[j] = at < n ? kGroup * list[at] + R::EPP * piece : -1;
    qt[j] = row_piece<T>(zt, e[j], V, vec);
    qd[j] = row_piece<T>(zd, e[j], V, vec);
  }
  uint32_t smask[R::NL];  // bit k: element e[j] + k is in the bias set
#pragma unroll
  for (int j = 0; j < R::NL; ++j) smask[j] = 0u;
  if (BIAS)
    for (int m = 0; m < nS; ++m) {
      const int id = S.S_ids[m];
#pragma unroll
      for (int j = 0; j < R::NL; ++j) {
        const uint32_t o = static_cast<uint32_t>(id - e[j]);
        if (e[j] >= 0 && o < static_cast<uint32_t>(R::EPP)) smask[j] |= 1u << o;
      }
    }
  float w[R::NL][R::EPP];
  float lm = -INFINITY;  // the lane's largest residual of the batch
#pragma unroll
  for (int j = 0; j < R::NL; ++j) {
    float ft[R::EPP], fd[R::EPP];
    unpack_piece<T>(qt[j], ft);
    unpack_piece<T>(qd[j], fd);
#pragma unroll
    for (int k = 0; k < R::EPP; ++k) {
      const float r = (BIAS && ((smask[j] >> k) & 1u)) ? rhoS : rho;
      w[j][k] = fmaxf(fmaf(-r, ex2_fast(fmaf(fd[k], c, -Mdc)), ex2_fast(fmaf(ft[k], c, -Mtc))),
                      0.f);
      if (e[j] >= 0 && e[j] + k < V && w[j][k] > 0.f) lm = fmaxf(lm, w[j][k]);
    }
  }
  // kth + 1 lanes hold a residual at least the (kth + 1)-th largest lane maximum: nothing below
  // it can be among the first kth + 1
  top.thr = fmaxf(top.thr, warp_rank_value(lm, top.kth));
#pragma unroll
  for (int j = 0; j < R::NL; ++j)
#pragma unroll
    for (int k = 0; k < R::EPP; ++k)
      top.offer(e[j] >= 0 && e[j] + k < V && w[j][k] > 0.f, w[j][k],
                static_cast<uint32_t>(e[j] + k));
}

template <typename T, bool BIAS, typename GV>
__device__ void resid_epilogue(const RowParams& P, RowShared& S, int u, const GV* gmax_t,
                               const GV* gmax_d, GV* gdel, const float* hdr) {
  const int t = et();
  const float c = P.c;
  const int V = P.V;
  const int ng = (V + kGroup - 1) / kGroup;
  const int b = u / P.K, i = u % P.K;
  const T* zt =
      static_cast<const T*>(P.tgt) + (static_cast<long long>(b) * (P.K + 1) + i) * P.t_stride;
  const T* zd = static_cast<const T*>(P.dft) + (static_cast<long long>(b) * P.K + i) * P.d_stride;
  int32_t* out = P.out_r2 + static_cast<long long>(u) * P.fmax;
  const bool vec = P.use_vec != 0;
  const int F = min(P.fan[i], 8);  // only the first F of the order are written
  // The sequence's cache-hit flag, by one lane for its first unit: 1 if the token the verify step
  // drew at a rejected position a is among the top-F draft ids it prepared for that position, 0
  // if not, -1 when every draft was accepted or the sequence is invalid.
  if (P.out_hit && i == 0 && t == ET - 32) {
    const int L = P.lens ? P.lens[b] : P.K;
    const int a = P.acc[b];
    int hit = -1;
    if (a >= 0 && a < L) {
      const int x = P.tok[static_cast<long long>(b) * (P.K + 1) + a];
      const int Fa = min(P.fan[a], P.fmax);
      const int32_t* r1 = P.r1 + (static_cast<long long>(b) * P.K + a) * P.fmax;
      hit = 0;
      for (int f = 0; f < Fa; ++f) hit |= r1[f] == x ? 1 : 0;
    }
    P.out_hit[b] = hit;
  }

  const float2 T2 = make_float2(hdr[0], hdr[1]);
  const float2 D2 = make_float2(hdr[2], hdr[3]);
  if (F <= 0 || row_bad(T2.x) || row_bad(D2.x)) {
    if (t < P.fmax) out[t] = -1;
    return;
  }
  // The rows streamed a while ago are leaving L2: the group of each thread whose target maximum
  // is largest (the bounds below are close to e_t,max for most groups, so these are the groups
  // the first round reads) is fetched into L2 at once, both rows, while the bias set and the
  // bounds are worked out.
  {
    float gm = -INFINITY;
    int gb = -1;
    for (int g = t; g < ng; g += ET) {
      const float v = gv_get(gmax_t, g);
      if (v > gm) {
        gm = v;
        gb = g;
      }
    }
    if (gb >= 0)
      for (int o = 0; o < kGroup && kGroup * gb + o < V; o += 128 / static_cast<int>(sizeof(T))) {
        prefetch_l2(zt + kGroup * gb + o);
        prefetch_l2(zd + kGroup * gb + o);
      }
  }
  int nS = 0;
  float N = 1.f;
  if (BIAS) {
    resid_bias_set<T>(P, S, gmax_d, ng, zd, V, vec, D2.x, D2.y);
    nS = S.nS;
    N = S.N;
  }
  // residual weights relative to p's scale: max(e_t - rho_v e_d, 0)
  const float Mtc = __fmul_rn(T2.x, c), Mdc = __fmul_rn(D2.x, c);
  const float ft = fmaf(-fmaf(T2.x, c, -Mtc), kLn2r, 1.f);
  const float fd = fmaf(-fmaf(D2.x, c, -Mdc), kLn2r, 1.f);
  const float rho = (fd * T2.y) / (ft * (D2.y * N));
  const float rhoS = rho * P.beta;

  // An upper bound of each group's residual: with delta = max (z_t - z_d) c over the group,
  // w = e_t (1 - rho_v 2^((z_d - z_t) c + Mtc - Mdc)) <= e_t,max (1 - 2^-(delta - kappa)),
  // kappa = log2(min rho_v) + Mtc - Mdc; 1 - 2^-x <= min(1, x ln 2). A small margin covers the
  // rounding of both sides; the bound is stored (rounded up) over the log-ratio maximum. A group
  // with x <= 0 gets 0: each of its residuals is below zero by a relative 7e-5 or more, far past
  // the rounding of the weights, so none is offered (and one whose e_t,max is below the smallest
  // normal float offers nothing either: the weights flush it to zero). min rho_v is rho except in
  // the groups that hold ids of the bias set (rho beta there): those few bounds are taken first
  // and put in place after the others.
  auto bound = [&](int g, float kap) {
    const float x = fmaf(gv_get(gdel, g), c, -kap) + 1e-4f;
    const float gt = gv_get(gmax_t, g);
    const float et = ex2_fast(fmaf(gt, c, -Mtc));
    const float f = x <= 0.f ? 0.f : (x < 0.25f ? x * 0.69314718f : 1.f - ex2_fast(-x) + 1e-6f);
    return gt > -INFINITY ? et * fminf(f, 1.f) * 1.001f : 0.f;
  };
  const float kappa = __log2f(rho) + Mtc - Mdc;
  int gS = -1;
  float bS = 0.f;
  if (BIAS && t < nS) {
    gS = S.sgrp[t];
    bS = bound(gS, __log2f(rhoS) + Mtc - Mdc);
  }
  if (BIAS) esync();  // the set's groups read their log-ratio maxima before they are replaced
  float bm = -INFINITY;
  for (int g = t; g < ng; g += ET) {
    const float bnd = bound(g, kappa);
    gv_put_up(gdel, g, bnd);
    bm = fmaxf(bm, bnd);
  }
  if (BIAS) {
    esync();
    if (gS >= 0) gv_put_up(gdel, gS, bS);  // (two ids of one group write the same bound)
  }
  // Rounds of groups in decreasing bound, a visited group's bound set to -1. Each round takes the
  // groups left whose bound reaches both the F-th best residual found so far and a lower bound
  // of the 8th largest bound left (some warp has 8 threads whose largest bound left reaches its
  // 8th largest), so a round reads the next few groups in bound order (up to kRoundCap; the rest
  // stay for the next round), each warp kBatch groups per round trip. The listing pass also
  // finds each thread's largest bound left: the rounds end when none reaches the F-th best (or
  // none is positive while fewer than F residuals are known).
  const int warp = t >> 5, lane = t & 31;
  WarpTop8 top;
  top.init(-INFINITY, F - 1);
  if (t == 0) S.ntl = 0;
  float lo = team_bound(bm, S);  // (its barriers publish the set's bounds and the reset)
  float thr = 0.f;  // the team's F-th best residual so far (0 until F are known)
  bool merged = false;  // S.top holds the team's list as it stands
  for (int round = 0;; ++round) {
    if (round > 0) {
      if (t == 0) S.ntl = 0;
      esync();
    }
    const float lr = fmaxf(lo, thr);
    float rest = -INFINITY;
    for (int g = t; g < ng; g += ET) {
      const float bg = gv_get(gdel, g);
      bool listed = false;
      if (bg > 0.f && bg >= lr) {
        const int at = atomicAdd(&S.ntl, 1);
        if (at < kRoundCap) {
          S.tl[at] = g;
          gv_put(gdel, g, -1.f);
          listed = true;
        }
      }
      if (!listed) rest = fmaxf(rest, bg);
    }
    const float r8 = warp_8th_largest(rest);
    const float rm = ord_to_float(__reduce_max_sync(FULL, float_to_ord(rest)));
    if (lane == 0) {
      S.rb[warp] = r8;
      S.rmax[warp] = rm;
    }
    esync();
    const int n = min(S.ntl, kRoundCap);
    if (n > 0)
      for (int j0 = kBatch * warp; j0 < n; j0 += kBatch * NEW)
        offer_groups<T, BIAS>(top, zt, zd, S.tl, j0, n, V, vec, c, Mtc, Mdc, rho, rhoS, S, nS);
    if (n > 0 || !merged) {
      team_top8(top, S);
      merged = true;
    }
    const unsigned long long kf = S.top[F - 1];
    thr = kf ? key_value(kf) : 0.f;
    if (thr > top.thr) top.thr = thr;
    float r8t = S.rb[0], rmt = S.rmax[0];
#pragma unroll
    for (int w = 1; w < NEW; ++w) {
      r8t = fmaxf(r8t, S.rb[w]);
      rmt = fmaxf(rmt, S.rmax[w]);
    }
    if (rmt <= 0.f || (kf && rmt < thr)) break;  // nothing left reaches the F-th best
    lo = r8t;
  }
  if (t < P.fmax) {
    const unsigned long long k = t < 8 ? S.top[t] : 0ull;
    out[t] = (t < F && k != 0ull) ? key_id(k) : -1;
  }
}

// ------------------------------------------------------------------------------------------
// epilogue: the top-8 prepass of the verify step's draft rows
// ------------------------------------------------------------------------------------------
// Keys of the 8 largest logits of draft row (b, i) = u (ties to the lower id), for the verify
// step's bias set and its top-F ids; a row that holds no distribution gets the key ~0 first. With
// top-F output requested, also the first F_i ids of the row.
template <typename T>
__device__ void top8_epilogue(const RowParams& P, RowShared& S, int u, const float* gmax,
                              const float* hdr) {
  const int t = et();
  const int V = P.V;
  const int ng = (V + kGroup - 1) / kGroup;
  const int i = u % P.K;
  const T* row = static_cast<const T*>(P.dft) +
                 (static_cast<long long>(u / P.K) * P.K + i) * P.d_stride;
  unsigned long long* keys = P.out_keys + static_cast<long long>(u) * 8;
  if (row_bad(hdr[0])) {
    if (t < 8) keys[t] = t == 0 ? ~0ull : 0ull;
    return;
  }
  row_top8<T>(row, V, P.use_vec != 0, gmax, ng, S);
  if (t < 8) keys[t] = S.top[t];
  if (P.out_topf && t < P.fmax) {
    const unsigned long long k = t < 8 ? S.top[t] : 0ull;
    P.out_topf[static_cast<long long>(u) * P.fmax + t] = (t < P.fan[i] && k != 0ull) ? key_id(k) : -1;
  }
}

template <typename T, int MODE, bool BIAS>
__device__ void epilogue_warps(const RowParams& P, RowShared& S, unsigned char* gbuf0,
                               unsigned char* gbuf1, int ngmax) {
  using GV = typename GroupVal<T, MODE>::type;
  int k = 0;
  for (;;) {
    const int b = k & 1;
    const bool ok = mbar_wait_bounded(&S.gfull[b], (k >> 1) & 1, kWaitBudget);
    if (!ok && et() == 0) atomicOr(&P.ws->error, 1u);
    const int u = S.gunit[b];
    if (named_sync_or(kBarE, ET, !ok || u == kEnd)) break;
    float* gb = reinterpret_cast<float*>(b ? gbuf1 : gbuf0);
    GV* gv = reinterpret_cast<GV*>(b ? gbuf1 : gbuf0);
    if (MODE == MODE_SAMPLE)
      sample_epilogue<T, BIAS>(P, S, u, gb, gb + ngmax, S.hdr[b]);
    else if (MODE == MODE_TOP8)
      top8_epilogue<T>(P, S, u, gb, S.hdr[b]);
    else
      resid_epilogue<T, BIAS>(P, S, u, gv, gv + ngmax, gv + 2 * ngmax, S.hdr[b]);
    esync();  // every epilogue thread is done with the buffer and the scratch
    if (et() == 0) mbar_arrive(&S.gfree[b]);
    ++k;
  }
}

// ------------------------------------------------------------------------------------------
// the kernel
// ------------------------------------------------------------------------------------------
template <typename T, int MODE, bool BIAS>
__global__ void __launch_bounds__(RT, 2) row_kernel(const RowParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ RowShared S;
  const int nst = P.nstages;
  unsigned char* ring = smem;
  const int ngmax = (P.V + kGroup - 1) / kGroup;
  const int narr = MODE == MODE_SAMPLE ? 2 : (MODE == MODE_TOP8 ? 1 : 3);  // arrays per buffer
  using GV = typename GroupVal<T, MODE>::type;
  unsigned char* gbuf0 = smem + static_cast<size_t>(nst) * kStage;
  unsigned char* gbuf1 = gbuf0 + static_cast<size_t>(narr) * ngmax * sizeof(GV);
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], NCW);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.gfull[b], NCW);
      mbar_init(&S.gfree[b], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (tid >= CT + ET)
    producer<T, MODE>(P, S, ring);
  else if (tid >= CT)
    epilogue_warps<T, MODE, BIAS>(P, S, gbuf0, gbuf1, ngmax);
  else
    chunk_warps<T, MODE>(P, S, ring, gbuf0, gbuf1, ngmax);
}

template <int MODE>
const void* pick_fn(int dtype, bool bias) {
  if (dtype == 1)
    return bias ? reinterpret_cast<const void*>(&row_kernel<uint16_t, MODE, true>)
                : reinterpret_cast<const void*>(&row_kernel<uint16_t, MODE, false>);
  return bias ? reinterpret_cast<const void*>(&row_kernel<float, MODE, true>)
              : reinterpret_cast<const void*>(&row_kernel<float, MODE, false>);
}

}  // namespace

size_t row_smem_bytes(int mode, int dtype, int V, int nstages) {
  const size_t ng = static_cast<size_t>((V + kGroup - 1) / kGroup);
  const size_t esz = (mode == MODE_RESID && dtype == 1) ? sizeof(GroupVal<uint16_t, MODE_RESID>::type)
                                                        : sizeof(float);
  return static_cast<size_t>(nstages) * kStage +
         2 * ng * esz * (mode == MODE_SAMPLE ? 2 : (mode == MODE_TOP8 ? 1 : 3));
}

int row_ctas_per_sm(int mode, int dtype, bool bias, int V, int nstages) {
  const void* fn = mode == MODE_SAMPLE ? pick_fn<MODE_SAMPLE>(dtype, bias)
                   : mode == MODE_TOP8  ? pick_fn<MODE_TOP8>(dtype, false)
                                        : pick_fn<MODE_RESID>(dtype, bias);
  const size_t smem = row_smem_bytes(mode, dtype, V, nstages);
  if (smem > kRowMaxSmem) return 0;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, RT, smem) != cudaSuccess) return 0;
  return n;
}

cudaError_t launch_rows(const RowParams& P, int mode, int dtype, int ctas, cudaStream_t stream) {
  const bool bias = P.bias_k > 0 && P.beta < 1.f;
  const void* fn = mode == MODE_SAMPLE ? pick_fn<MODE_SAMPLE>(dtype, bias)
                   : mode == MODE_TOP8  ? pick_fn<MODE_TOP8>(dtype, false)
                                        : pick_fn<MODE_RESID>(dtype, bias);
  if (P.nstages < 2 || P.nstages > kRowMaxStages) return cudaErrorInvalidValue;
  const size_t smem = row_smem_bytes(mode, dtype, P.V, P.nstages);
  if (smem > kRowMaxSmem) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (ctas > 0) {
    void* args[] = {const_cast<RowParams*>(&P)};
    e = cudaLaunchKernel(fn, dim3(static_cast<unsigned>(ctas)), dim3(RT), args, smem, stream);
  }
  return e;
}

}  // namespace sv

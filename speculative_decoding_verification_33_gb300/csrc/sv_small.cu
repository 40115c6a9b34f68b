// Stochastic verification of small batches with every row in flight at once (Kangaroo guide,
// section 3: accept x_i while u_i < p_i(x_i) / q_i(x_i), then draw from max(p_a - q_a, 0), or from
// p_L when every draft is accepted; SSD summary, "Method").
//
// The chained cluster walk takes a position's decision before it streams the next one, so a
// batch of few sequences spends its time on the latency of position after position, and it
// reads only the rows the outcome needs. When the rows a sequence has are few enough that
// reading all of them at full bandwidth costs less than that latency, three launches do it,
// each started early (programmatic dependent launch) and waiting for its predecessor's writes:
//  1. small_rows: one CTA per (row, slice of the vocabulary) for every row a sequence has
//     (target 0..L_b, draft 0..L_b-1) reduces its slice to (max, sum of 2^(z c - fl(max c)));
//  2. small_mass: one CTA per (sequence, slice of the vocabulary) combines the sequence's
//     partials, takes the accept tests in order (every CTA of the sequence reaches the same
//     decision) and sums its slice of the draw's weights: per 8-element vector the sequential
//     float sum of max(e_t - rho e_d, 0), truncated to an integer of 2^-44, both for the
//     residual and for p (the draw falls back to p when the residual has no mass left);
//  3. small_pick: one CTA per sequence finds the slice that holds floor(u W) from the slices'
//     masses, then the vector inside it by a block prefix of the vectors' integers, walks that
//     vector and writes the outcome.
// The integer masses make the prefix exact and independent of the order of the sums.
//
// A Saguaro bias set (the bias_k most likely draft ids reweighted by beta; Saguaro summary,
// "Method") and the top-F ids need the 8 largest logits of each draft row: small_rows keeps them
// per slice while it streams (a warp's 8 largest keys, offered only what can still enter), and
// small_mass merges the slices' lists of each row before the accept tests.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "sv_math.cuh"
#include "sv_ptx.cuh"
#include "sv_small.h"

namespace sv {
namespace {

constexpr int kRowThreads = 128;
constexpr int kMassThreads = 128;
constexpr int kPickThreads = 256;
constexpr int kPickVecs = 4;  // vectors of a slice per pick thread: slice_d <= 8192 ids
constexpr float kLn2 = 0.69314718055994531f;

// Programmatic dependent launch: let the next launch on the stream start its CTAs, and wait
// until the previous launch has finished and its writes are visible.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// row slot r of sequence b: target 0..K, then draft 0..K-1
__device__ __forceinline__ const void* small_row(const SmallParams& P, int b, int slot,
                                                 size_t elt) {
  const bool draft = slot > P.K;
  const int i = draft ? slot - P.K - 1 : slot;
  const char* base = static_cast<const char*>(draft ? P.dft : P.tgt);
  const long long rows = draft ? P.K : P.K + 1;
  const long long stride = draft ? P.d_stride : P.t_stride;
  return base + ((static_cast<long long>(b) * rows + i) * stride) * static_cast<long long>(elt);
}

// An L2 cache policy under which the lines a load brings in are the first to be evicted.
__device__ __forceinline__ unsigned long long l2_policy_evict_first() {
  unsigned long long pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// A 16-byte read-only global load that does not allocate in L1, under an L2 cache policy.
__device__ __forceinline__ uint4 ldg_nc_v4_hint(const void* p, unsigned long long pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

// 8 elements as they sit in memory: one 16-byte word for bf16, two for float
template <typename T>
struct Raw8 {
  uint4 w[sizeof(T) / 2];
};

template <typename T>
__device__ __forceinline__ void raw_load(const T* p, Raw8<T>& r) {
#pragma unroll
  for (int k = 0; k < static_cast<int>(sizeof(T) / 2); ++k)
    r.w[k] = ldg_nc_v4(reinterpret_cast<const char*>(p) + 16 * k);
}
template <typename T>
__device__ __forceinline__ void raw_load(const T* p, Raw8<T>& r, unsigned long long pol) {
#pragma unroll
  for (int k = 0; k < static_cast<int>(sizeof(T) / 2); ++k)
    r.w[k] = ldg_nc_v4_hint(reinterpret_cast<const char*>(p) + 16 * k, pol);
}

__device__ __forceinline__ void raw_unpack(const Raw8<uint16_t>& r, float (&z)[8]) {
  Elt<uint16_t>::unpack(r.w[0], z);
}
__device__ __forceinline__ void raw_unpack(const Raw8<float>& r, float (&z)[8]) {
  z[0] = __uint_as_float(r.w[0].x); z[1] = __uint_as_float(r.w[0].y);
  z[2] = __uint_as_float(r.w[0].z); z[3] = __uint_as_float(r.w[0].w);
  z[4] = __uint_as_float(r.w[1].x); z[5] = __uint_as_float(r.w[1].y);
  z[6] = __uint_as_float(r.w[1].z); z[7] = __uint_as_float(r.w[1].w);
}

// elements e..e+7 of a row of V ids, -inf past the end (one by one when not a whole vector)
template <typename T>
__device__ __forceinline__ void load8_at(const T* row, int e, int V, bool aligned, float (&z)[8]) {
  if (aligned && e + 8 <= V) {
    Raw8<T> r;
    raw_load(row + e, r);
    raw_unpack(r, z);
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) z[k] = (e + k < V) ? Elt<T>::val(row[e + k]) : -INFINITY;
  }
}

// One thread's vectors of a staged chunk of n ids (vectors tid, tid + kRowThreads, ...), -inf
// past n: their maximum (NaN sticks) and the values.
template <typename T, int VPT>
struct Staged;

template <int VPT>
struct Staged<uint16_t, VPT> {
  static constexpr int kVecs = VPT;
  uint4 v[VPT];
  __device__ __forceinline__ void load(const uint16_t* s, int n) {  // n: a multiple of 8
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int g = threadIdx.x + j * kRowThreads;
      v[j] = 8 * g + 8 <= n ? reinterpret_cast<const uint4*>(s)[g]
                            : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
    }
  }
  __device__ __forceinline__ float vmax() const {
    uint32_t m = max_nan_bf16x2(max_nan_bf16x2(v[0].x, v[0].y), max_nan_bf16x2(v[0].z, v[0].w));
#pragma unroll
    for (int j = 1; j < VPT; ++j)
      m = max_nan_bf16x2(m, max_nan_bf16x2(max_nan_bf16x2(v[j].x, v[j].y),
                                           max_nan_bf16x2(v[j].z, v[j].w)));
    return max_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
  }
  __device__ __forceinline__ void get(int j, float (&z)[8]) const {
    Elt<uint16_t>::unpack(v[j], z);
  }
};

template <int VPT>
struct Staged<float, VPT> {
  static constexpr int kVecs = VPT;
  float z[VPT][8];
  __device__ __forceinline__ void load(const float* s, int n) {  // n: a multiple of 4
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int g = threadIdx.x + j * kRowThreads;
      const float4 a = 8 * g + 4 <= n ? reinterpret_cast<const float4*>(s)[2 * g]
                                      : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      const float4 b = 8 * g + 8 <= n ? reinterpret_cast<const float4*>(s)[2 * g + 1]
                                      : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      z[j][0] = a.x; z[j][1] = a.y; z[j][2] = a.z; z[j][3] = a.w;
      z[j][4] = b.x; z[j][5] = b.y; z[j][6] = b.z; z[j][7] = b.w;
    }
  }
  __device__ __forceinline__ float vmax() const {
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < VPT; ++j)
#pragma unroll
      for (int k = 0; k < 8; ++k) m = max_nan(m, z[j][k]);
    return m;
  }
  __device__ __forceinline__ void get(int j, float (&out)[8]) const {
#pragma unroll
    for (int k = 0; k < 8; ++k) out[k] = z[j][k];
  }
};

// ------------------------------------------------------------------------------------------
// The 8 largest logits of a draft row slice (keys: larger value first, then lower id)
// ------------------------------------------------------------------------------------------
// Order-preserving 32 bits of a float, 0 for NaN (absent).
__device__ __forceinline__ uint32_t float_ord(float v) {
  const uint32_t b = __float_as_uint(v);
  return isnan(v) ? 0u : ((b & 0x80000000u) ? ~b : (b | 0x80000000u));
}
__device__ __forceinline__ float ord_value(uint32_t m) {
  return m == 0u ? -INFINITY : __uint_as_float((m & 0x80000000u) ? (m & 0x7FFFFFFFu) : ~m);
}

// The 8 largest of the lanes' order-preserving integers, with repeats (0 = absent): lane q < 8
// returns the q-th, 0 past those there are. Warp-wide.
__device__ __forceinline__ uint32_t warp_top8_u32(uint32_t o) {
  const int lane = threadIdx.x & 31;
  uint32_t mine = 0u;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const uint32_t m = __reduce_max_sync(FULL, o);
    if (lane == r) mine = m;
    const unsigned who = __ballot_sync(FULL, o == m && m != 0u);
    if (who && lane == __ffs(who) - 1) o = 0u;
  }
  return mine;
}

constexpr int kStages = 2;                      // bulk-copy ring of the row kernel
constexpr int kChunk = 8192;                    // bytes per stage
constexpr long long kWaitBudget = 4000000000LL;  // clock cycles (about 2 s) per barrier wait

// Fold 8 logits into the running (max, sum).
__device__ __forceinline__ void fold8(RowAcc& acc, const float (&z)[8], float c) {
  float vm = -INFINITY;
#pragma unroll
  for (int j = 0; j < 8; ++j) vm = max_nan(vm, z[j]);
  acc.rescale(vm, c);
  if (acc.m > -INFINITY) acc.sum8(z, c);
}

// A 16-byte aligned row slice [e0, e1) streamed through a ring of bulk copies into shared
// memory (up to kStages * kChunk bytes in flight per CTA, whatever the register budget); the
// ids past the last whole 16 bytes are read directly, by thread 0. Thread t folds the slice's
// vectors t, t + kRowThreads, ... (8 ids each, counted from e0). False when a copy did not land
// within the wait budget (the CTA then waits, bounded again, for the copies it issued and
// returns).
template <typename T>
__device__ bool rows_bulk(const T* row, int e0, int e1, float c, RowAcc& acc) {
  __shared__ __align__(128) unsigned char ring[kStages][kChunk];
  __shared__ uint64_t bar[kStages];
  constexpr int per = kChunk / static_cast<int>(sizeof(T));  // ids per stage
  constexpr int q16 = 16 / static_cast<int>(sizeof(T));      // ids per 16 bytes
  const int tid = threadIdx.x;
  const int eb = e0 + (e1 - e0) / q16 * q16;
  const int nch = (eb - e0 + per - 1) / per;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto issue = [&](int j) {
    const int s = j % kStages;
    const int ids = min(per, eb - (e0 + j * per));
    const uint32_t bytes = static_cast<uint32_t>(ids) * sizeof(T);
    mbar_arrive_expect_tx(&bar[s], bytes);
    bulk_g2s(ring[s], row + e0 + j * per, bytes, &bar[s]);
  };
  if (tid == 0)
    for (int j = 0; j < min(kStages, nch); ++j) issue(j);
  int j = 0;
  bool ok = true;
  for (; j < nch; ++j) {
    const int s = j % kStages;
    const bool landed = mbar_wait_bounded(&bar[s], (j / kStages) & 1, kWaitBudget);
    if (__syncthreads_or(!landed)) {
      ok = false;
      break;
    }
    // the thread's vectors of the chunk: their maximum first, one rescale, then the sums
    Staged<T, kChunk / static_cast<int>(sizeof(T)) / 8 / kRowThreads> st;
    st.load(reinterpret_cast<const T*>(ring[s]), min(per, eb - (e0 + j * per)));
    acc.rescale(st.vmax(), c);
    if (acc.m > -INFINITY) {
#pragma unroll
      for (int v = 0; v < st.kVecs; ++v) {
        float z[8];
        st.get(v, z);
        acc.sum8(z, c);
      }
    }
    __syncthreads();  // every thread is done with stage s before it is refilled
    if (tid == 0 && j + kStages < nch) issue(j + kStages);
  }
  if (!ok) {
    if (tid == 0)
      for (int k = j; k < min(nch, j + kStages); ++k)
        mbar_wait_bounded(&bar[k % kStages], (k / kStages) & 1, kWaitBudget);
    __syncthreads();
    return false;
  }
  if (tid == 0 && eb < e1) {  // fewer than 16 bytes left
    float z[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) z[k] = eb + k < e1 ? Elt<T>::val(row[eb + k]) : -INFINITY;
    fold8(acc, z, c);
  }
  return true;
}

// A row slice [e0, e1) that is not 16-byte aligned, element by element, a batch of loads in
// flight per thread; thread t folds vectors t, t + kRowThreads, ... as in rows_bulk.
template <typename T>
__device__ void rows_plain(const T* row, int e0, int e1, float c, RowAcc& acc) {
  const int nv = (e1 - e0 + 7) >> 3;
  constexpr int U = 4;
  for (int g0 = threadIdx.x; g0 < nv; g0 += U * kRowThreads) {
    float z[U][8];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int e = e0 + 8 * (g0 + k * kRowThreads);
#pragma unroll
      for (int q = 0; q < 8; ++q) z[k][q] = e + q < e1 ? Elt<T>::val(row[e + q]) : -INFINITY;
    }
#pragma unroll
    for (int k = 0; k < U; ++k)
      if (g0 + k * kRowThreads < nv) fold8(acc, z[k], c);
  }
}

// The 8 largest keys of a draft row slice [e0, e1) without NaN or +inf, after the stream
// (block-wide; lane q < 8 of warp 0 returns the q-th, 0 where the slice has fewer ids).
// Thread t has folded vectors t (mod kRowThreads) of the slice (and thread 0 the ids past the
// last whole 16 bytes, which lie in the slice's last vector); tmax is its running maximum. The
// 8th largest tmax, theta, is a value that 8 of the slice's elements reach: an element below
// theta is not among the 8 largest, and neither is any element of a thread whose tmax is below
// theta. The vectors of the other threads (and the last vector) are read again, from L2, and
// their elements at or above theta collected as keys in shared memory (up to kCand), of which
// the 8 largest are taken. Should more than kCand elements tie at or above theta, the 8 are
// found by 8 passes over those vectors instead, each taking the largest key below the one
// before.
constexpr int kCand = 256;
constexpr int kItemsInFlight = 2;  // vectors a thread reads again at once
template <typename T>
__device__ unsigned long long slice_top8(const T* row, int e0, int e1, bool aligned, float tmax,
                                         unsigned long long* cand, uint32_t* s_top, int* s_list,
                                         int* s_n) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = kRowThreads / 32;
  static_assert(kRowThreads == 128, "four warps' 8 largest fill one warp");
  const uint32_t wt = warp_top8_u32(float_ord(tmax));  // each warp's 8 largest, then the block's
  if (lane < 8) s_top[warp * 8 + lane] = wt;
  if (tid == 0) s_n[0] = s_n[1] = 0;
  __syncthreads();
  if (warp == 0) {
    const uint32_t t8 = __shfl_sync(FULL, warp_top8_u32(s_top[lane]), 7);
    if (lane == 0) s_top[32] = t8;
  }
  __syncthreads();
  const float th = ord_value(s_top[32]);
  const int nvec = (e1 - e0 + 7) >> 3;
  const int glast = nvec - 1;
  if (tmax >= th) s_list[atomicAdd(&s_n[1], 1)] = tid;  // this thread's vectors may hold one
  __syncthreads();
  const int ncand = s_n[1];
  // work items: (candidate thread c, its k-th vector), then the last vector unless its owner
  // is a candidate
  bool owner_in = false;
  for (int q = 0; q < ncand; ++q) owner_in |= s_list[q] == glast % kRowThreads;
  const int per_c = (nvec + kRowThreads - 1) / kRowThreads;
  const int items = ncand * per_c + (owner_in ? 0 : 1);
  auto each = [&](auto&& f) {  // f(z, id) for every element at or above theta
    for (int i0 = tid; i0 < items; i0 += kItemsInFlight * kRowThreads) {
      float z[kItemsInFlight][8];
      int g[kItemsInFlight];
#pragma unroll
      for (int u = 0; u < kItemsInFlight; ++u) {
        const int it = i0 + u * kRowThreads;
        g[u] = -1;
        if (it < items) {
          g[u] = it == ncand * per_c ? glast : s_list[it / per_c] + kRowThreads * (it % per_c);
          if (g[u] >= nvec) g[u] = -1;
        }
        if (g[u] >= 0) load8_at(row, e0 + 8 * g[u], e1, aligned, z[u]);
      }
#pragma unroll
      for (int u = 0; u < kItemsInFlight; ++u) {
        if (g[u] < 0) continue;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (e0 + 8 * g[u] + k < e1 && z[u][k] >= th) f(z[u][k], e0 + 8 * g[u] + k);
      }
    }
  };
  each([&](float z, int id) {
    const int at = atomicAdd(&s_n[0], 1);
    if (at < kCand) cand[at] = make_key(z, static_cast<uint32_t>(id));
  });
  __syncthreads();
  const int n = s_n[0];
  unsigned long long mine_key = 0ull;
  if (n <= kCand) {
    if (warp == 0) {
      unsigned long long a[kCand / 32];
#pragma unroll
      for (int q = 0; q < kCand / 32; ++q) a[q] = lane + 32 * q < n ? cand[lane + 32 * q] : 0ull;
#pragma unroll 1
      for (int r = 0; r < 8; ++r) {
        unsigned long long best = 0ull;
#pragma unroll
        for (int q = 0; q < kCand / 32; ++q) best = a[q] > best ? a[q] : best;
        const unsigned long long m = warp_max_key(best);
        if (lane == r) mine_key = m;
#pragma unroll
        for (int q = 0; q < kCand / 32; ++q)
          if (a[q] == m) a[q] = 0ull;
      }
    }
  } else {
    unsigned long long prev = ~0ull;
#pragma unroll 1
    for (int r = 0; r < 8; ++r) {
      unsigned long long best = 0ull;
      each([&](float z, int id) {
        const unsigned long long k = make_key(z, static_cast<uint32_t>(id));
        if (k < prev && k > best) best = k;
      });
      best = warp_max_key(best);
      __syncthreads();  // the previous pass's reads of cand are done
      if (lane == 0) cand[warp] = best;
      __syncthreads();
      unsigned long long m = cand[0];
#pragma unroll
      for (int w = 1; w < NW; ++w) m = cand[w] > m ? cand[w] : m;
      if (lane == r) mine_key = m;
      prev = m;
      if (m == 0ull) break;  // fewer than 8 keys below the last one: the rest stay 0
    }
  }
  return mine_key;
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads) small_rows(const SmallParams P) {
  pdl_trigger();
  __shared__ float sm[kRowThreads / 32], ss[kRowThreads / 32];
  const int sl = blockIdx.x, r = blockIdx.y;
  const int b = r / (2 * P.K + 1), slot = r - b * (2 * P.K + 1);
  const int L = P.lens ? P.lens[b] : P.K;
  if (L < 1 || L > P.K) return;
  if (slot <= P.K ? slot > L : slot - P.K - 1 >= L) return;  // rows the decision never reads
  const T* row = static_cast<const T*>(small_row(P, b, slot, sizeof(T)));
  const float c = P.c;
  const int e0 = sl * P.slice, e1 = min(P.V, e0 + P.slice);
  RowAcc acc;
  acc.init();
  bool ok = true;
  if (P.aligned)
    ok = rows_bulk(row, e0, e1, c, acc);
  else
    rows_plain(row, e0, e1, c, acc);
  if (!ok) {  // a copy that never landed: the row reads as NaN and the error word is raised
    if (threadIdx.x == 0) {
      atomicOr(P.err, 1u);
      P.part[static_cast<long long>(r) * P.nslice + sl] = make_float2(__int_as_float(0x7fffffff), 0.f);
    }
    return;
  }
  // the CTA's (max, sum relative to fl(max c)), with the rounding of max c folded back
  const float m = warp_max_nan(acc.m);
  if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = m;
  __syncthreads();
  float M = sm[0];
  for (int w = 1; w < kRowThreads / 32; ++w) M = max_nan(M, sm[w]);
  const float Mc = __fmul_rn(M, c);
  const float t = (!row_bad(M) && acc.m > -INFINITY) ? acc.total() * exp2f(acc.mc - Mc) : 0.f;
  const float s = warp_sum(t);
  if ((threadIdx.x & 31) == 0) ss[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float S = 0.f;
    for (int w = 0; w < kRowThreads / 32; ++w) S += ss[w];
    if (!row_bad(M)) S *= fmaf(-fmaf(M, c, -Mc), kLn2, 1.f);
    P.part[static_cast<long long>(r) * P.nslice + sl] = make_float2(M, S);
  }
  if (P.top8 && slot > P.K) {
    // a draft row's slice: its 8 largest keys (none for a row with NaN or +inf; a slice of -inf
    // only still has keys, of its lowest ids)
    __shared__ unsigned long long s_cand[kCand];
    __shared__ uint32_t s_top[33];
    __shared__ int s_list[kRowThreads], s_n[2];
    const unsigned long long k =
        (isnan(M) || M == INFINITY)
            ? 0ull
            : slice_top8(row, e0, e1, P.aligned != 0, acc.m, s_cand, s_top, s_list, s_n);
    if (threadIdx.x < 8)
      P.keys[((static_cast<long long>(b) * P.K + (slot - P.K - 1)) * P.nslice + sl) * 8 +
             threadIdx.x] = k;
  }
}

constexpr int kMaxSmallK = 8;   // positions per sequence
constexpr int kMaxSlices = 32;  // vocabulary slices per row, and per draw

// (M, S) of a row from its slices: the largest maximum, and the sum rescaled to it. Warp-wide.
__device__ __forceinline__ float2 combine_row(const float2* part, int nslice, float c) {
  const int lane = threadIdx.x & 31;
  const float2 p = lane < nslice ? part[lane] : make_float2(-INFINITY, 0.f);
  const float M = warp_max_nan(p.x);
  const float t = (!row_bad(M) && p.x > -INFINITY) ? p.y * exp2f((p.x - M) * c) : 0.f;
  return make_float2(M, warp_sum(t));
}

// The 8 largest keys of a draft row from its slices' lists (each descending; one slice per
// lane, nslice <= 32): lane q < 8 returns the q-th. Warp-wide.
__device__ __forceinline__ unsigned long long merge_slices(const unsigned long long* lists,
                                                          int nslice) {
  const int lane = threadIdx.x & 31;
  unsigned long long a[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) a[q] = 0ull;
  if (lane < nslice) {
    const ulonglong2* p = reinterpret_cast<const ulonglong2*>(lists + lane * 8);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const ulonglong2 v = p[q];
      a[2 * q] = v.x;
      a[2 * q + 1] = v.y;
    }
  }
  unsigned long long mine = 0ull;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const unsigned long long m = warp_max_key(a[0]);
    if (lane == q) mine = m;
    if (m != 0ull && a[0] == m) {
#pragma unroll
      for (int j = 0; j < 7; ++j) a[j] = a[j + 1];
      a[7] = 0ull;
    }
  }
  return mine;
}

// The decision of sequence b from the row partials, block-wide (every thread returns it): the
// accept tests in order; at a rejection the residual draw's constants (fl(M_t c), fl(M_d c) and
// rho = the ratio of the draft's scale to the target's), after every acceptance the bonus draw
// from p_L (rho = 0). A sequence is invalid (ok = 0) for a length outside 1..K, an id outside the
// vocabulary, a uniform outside [0, 1), or a row read before the stop that is NaN, +inf or all
// -inf; with top-F ids, also a draft row below L that is NaN, +inf or all -inf. The first CTA
// of the sequence writes its top-F ids: for i < L the first F_i ids of draft row i (-1 past
// them), -1 for i >= L and for an invalid sequence.
template <typename T, bool BIAS>
__device__ SmallDecision decide(const SmallParams& P, int b) {
  __shared__ float2 s_ms[2 * kMaxSmallK + 1];
  __shared__ float s_zx[2][kMaxSmallK];
  __shared__ int s_x[kMaxSmallK];
  __shared__ float s_u[kMaxSmallK + 1];
  __shared__ unsigned long long s_key[kMaxSmallK][8];
  __shared__ float s_N[kMaxSmallK], s_f[kMaxSmallK];
  __shared__ int s_nS[kMaxSmallK];
  __shared__ SmallDecision s_dec;
  const int tid = threadIdx.x, warp = tid >> 5, K = P.K;
  const int L = P.lens ? P.lens[b] : K;
  const int32_t* x = P.tokens + static_cast<long long>(b) * K;
  const float* u = P.uni + static_cast<long long>(b) * (K + 1);
  const float c = P.c;
  const bool lok = L >= 1 && L <= K;
  // the inputs first (no earlier launch writes them): ids, uniforms, the logits at the ids
  if (tid < K) s_x[tid] = x[tid];
  if (tid <= K) s_u[tid] = u[tid];
  if (lok && tid < 2 * L) {
    const int i = tid < L ? tid : tid - L, d = tid < L ? 0 : 1;
    const int xi = x[i];
    s_zx[d][i] = (xi >= 0 && xi < P.V)
                     ? Elt<T>::val(static_cast<const T*>(
                           small_row(P, b, d ? K + 1 + i : i, sizeof(T)))[xi])
                     : 0.f;
  }
  const bool bias = BIAS && P.bias_k > 0 && P.top8;
  pdl_wait();  // the row partials and the slices' keys come from the statistics launch
  if (lok) {
    const int nw = blockDim.x >> 5;
    for (int r = warp; r < 2 * L + 1; r += nw) {  // one warp per row
      const int slot = r <= L ? r : K + 1 + (r - L - 1);
      const float2 ms =
          combine_row(P.part + (static_cast<long long>(b) * (2 * K + 1) + slot) * P.nslice,
                      P.nslice, c);
      if ((tid & 31) == 0) s_ms[slot] = ms;
    }
    if (P.top8)  // the draft rows' top 8: one warp per row merges its slices
      for (int i = (warp + 2 * L + 1) % nw; i < L; i += nw) {
        const unsigned long long k =
            merge_slices(P.keys + (static_cast<long long>(b) * K + i) * P.nslice * 8, P.nslice);
        if ((tid & 31) < 8) s_key[i][tid & 31] = k;
      }
  }
  __syncthreads();
  if (bias && lok) {
    // per draft row i < L, one warp: the bias set (its first bias_k keys), q(set) summed in key
    // order, N = 1 - (1 - beta) q(set), and whether the draft id is in the set
    const int lane = tid & 31, nw = blockDim.x >> 5;
    for (int i = warp; i < L; i += nw) {
      const float2 q = s_ms[K + 1 + i];
      const unsigned long long kj = lane < 8 ? s_key[i][lane] : 0ull;
      const bool in = lane < P.bias_k && kj != 0ull;
      const float term = in ? exp2f((key_value(kj) - q.x) * c) / q.y : 0.f;
      const unsigned hit = __ballot_sync(FULL, in && key_id(kj) == s_x[i]);
      const unsigned n = __popc(__ballot_sync(FULL, in));
      float sq = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float tj = __shfl_sync(FULL, term, j);
        if (j < static_cast<int>(n)) sq += tj;
      }
      if (lane == 0) {
        s_N[i] = fmaf(-(1.f - P.beta), sq, 1.f);
        s_f[i] = hit ? P.beta : 1.f;
        s_nS[i] = static_cast<int>(n);
      }
    }
    __syncthreads();
  }
  if (tid == 0) {
    bool ok = lok;
    for (int i = 0; ok && i < L; ++i)
      ok = s_x[i] >= 0 && s_x[i] < P.V && s_u[i] >= 0.f && s_u[i] < 1.f;
    ok = ok && s_u[K] >= 0.f && s_u[K] < 1.f;
    for (int i = 0; ok && P.fmax > 0 && i < L; ++i) ok = !row_bad(s_ms[K + 1 + i].x);
    SmallDecision d;
    d.a = L;
    d.mct = d.mcd = d.rho = d.rho_s = 0.f;
    d.nS = 0;
    for (int i = 0; ok && i <= L; ++i) {
      const float2 t = s_ms[i];
      if (row_bad(t.x)) {
        ok = false;
        break;
      }
      if (i == L) {  // every draft accepted: the bonus draw from p_L
        d.mct = __fmul_rn(t.x, c);
        break;
      }
      const float2 q = s_ms[K + 1 + i];
      if (row_bad(q.x)) {
        ok = false;
        break;
      }
      // Saguaro bias set: the bias_k most likely draft ids get weight beta, and q' is q
      // reweighted and renormalised by N = 1 - (1 - beta) * q(set)
      float N = 1.f, f = 1.f;
      int nS = 0;
      if (bias) {
        N = s_N[i];
        f = s_f[i];
        nS = s_nS[i];
#pragma unroll
        for (int j = 0; j < 8; ++j) d.ids[j] = j < nS ? key_id(s_key[i][j]) : -1;
      }
      const float zt = s_zx[0][i], zd = s_zx[1][i];
      float ratio;
      if (zt == -INFINITY) ratio = 0.f;
      else if (zd == -INFINITY) ratio = INFINITY;
      else ratio = exp2f(((zt - zd) - (t.x - q.x)) * c) * (q.y / t.y) * (N / f);
      if (s_u[i] < ratio) continue;
      d.a = i;  // the residual draw: rho = q' scale / p scale
      d.mct = __fmul_rn(t.x, c);
      d.mcd = __fmul_rn(q.x, c);
      const float ft = fmaf(-fmaf(t.x, c, -d.mct), kLn2, 1.f);
      const float fd = fmaf(-fmaf(q.x, c, -d.mcd), kLn2, 1.f);
      d.rho = (fd * t.y) / (ft * (q.y * N));
      d.rho_s = d.rho * P.beta;
      d.nS = nS;
      break;
    }
    d.ok = ok ? 1 : 0;
    if (!ok) d.a = -1;
    s_dec = d;
  }
  __syncthreads();
  if (P.fmax > 0 && blockIdx.x == 0) {
    int32_t* tf = P.out_topf + static_cast<long long>(b) * K * P.fmax;
    const bool ok = s_dec.ok != 0;
    for (int e = tid; e < K * P.fmax; e += blockDim.x) {
      const int i = e / P.fmax, f = e - i * P.fmax;
      const unsigned long long k = (ok && i < L && f < P.fan[i] && f < 8) ? s_key[i][f] : 0ull;
      tf[e] = k ? key_id(k) : -1;
    }
  }
  return s_dec;
}

// The draw's weights of 8 elements: w = max(e_t - rho e_d, 0) with e = 2^(z c - fl(M c)), and the
// sequential float sums of w (residual) and of e_t (p). With rho = 0 both are e_t.
__device__ __forceinline__ void weights8(const float (&zt)[8], const float (&zd)[8], float c,
                                         float mc_t, float mc_d, const float (&rk)[8], bool two,
                                         float (&w)[8], float& s_res, float& s_p) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float et = ex2_fast(fmaf(zt[k], c, -mc_t));
    const float ed = two ? ex2_fast(fmaf(zd[k], c, -mc_d)) : 0.f;
    w[k] = fmaxf(fmaf(-rk[k], ed, et), 0.f);
    s_res = k ? __fadd_rn(s_res, w[k]) : w[0];
    s_p = k ? __fadd_rn(s_p, et) : et;
  }
}

// The draft weight's factor for ids e..e+7: rho, or rho * beta on the bias set of the decided
// draft row (rho = 0: a draw from p).
template <bool BIAS>
__device__ __forceinline__ void rho8(const SmallDecision& d, float rho, int e, float (&rk)[8],
                                     bool maybe = true) {
#pragma unroll
  for (int k = 0; k < 8; ++k) rk[k] = rho;
  if (!BIAS || !maybe || rho == 0.f || d.nS == 0) return;
  bool any = false;
#pragma unroll
  for (int j = 0; j < 8; ++j) any |= j < d.nS && static_cast<unsigned>(d.ids[j] - e) < 8u;
  if (!any) return;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int off = j < d.nS ? d.ids[j] - e : -1;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (k == off) rk[k] = d.rho_s;
  }
}

// Vectors (of each of the two rows) a mass thread keeps in flight: 64 bytes of each row.
template <typename T>
constexpr int kMassUnroll = 8 / static_cast<int>(sizeof(T));

// The draw's weights summed over slice `sl` of sequence b's decided rows (decision d): per
// 8-element vector the sequential float sums of the residual and of p, truncated to integers of
// 2^-44, summed per slice into P.mass. Block-wide.
template <typename T, bool BIAS, bool EF = false>
__device__ void slice_masses(const SmallParams& P, int b, const SmallDecision& d, int sl) {
  __shared__ unsigned long long s_r[kMassThreads / 32], s_p[kMassThreads / 32];
  const int tid = threadIdx.x;
  const int K = P.K;
  const int L = P.lens ? P.lens[b] : K;
  const T* gt = static_cast<const T*>(small_row(P, b, d.a, sizeof(T)));
  const T* gd = d.a < L ? static_cast<const T*>(small_row(P, b, K + 1 + d.a, sizeof(T))) : gt;
  const bool al = P.aligned != 0;
  const bool two = d.rho != 0.f;
  const float c = P.c;
  const int e0 = sl * P.slice_d, e1 = min(P.V, e0 + P.slice_d);
  const int nv = (e1 - e0 + 7) >> 3;
  constexpr int U = kMassUnroll<T>;
  // a bias-set id in one of this thread's vectors (g = tid mod kMassThreads)?
  bool maybe = false;
  if (BIAS && two)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int o = d.ids[j] - e0;
      maybe |= j < d.nS && o >= 0 && d.ids[j] < e1 && ((o >> 3) % kMassThreads) == tid;
    }
  unsigned long long own_r = 0, own_p = 0;
  const unsigned long long pol = EF ? l2_policy_evict_first() : 0ull;
  for (int g0 = tid; g0 < nv; g0 += U * kMassThreads) {
    Raw8<T> vt[U], vd[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int e = e0 + 8 * (g0 + k * kMassThreads);
      if (al && e + 8 <= e1) {
        if (EF) {
          raw_load(gt + e, vt[k], pol);
          if (two) raw_load(gd + e, vd[k], pol);
        } else {
          raw_load(gt + e, vt[k]);
          if (two) raw_load(gd + e, vd[k]);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int g = g0 + k * kMassThreads;
      if (g >= nv) break;
      const int e = e0 + 8 * g;
      float zt[8], zd[8], w[8], sr, sp;
      if (al && e + 8 <= e1) {
        raw_unpack(vt[k], zt);
        if (two) raw_unpack(vd[k], zd);
      } else {
        load8_at(gt, e, e1, al, zt);
        if (two) load8_at(gd, e, e1, al, zd);
      }
      float rk[8];
      rho8<BIAS>(d, d.rho, e, rk, maybe);
      weights8(zt, zd, c, d.mct, d.mcd, rk, two, w, sr, sp);
      own_r += qfix(sr);
      own_p += qfix(sp);
    }
  }
  own_r = warp_sum_u64(own_r);
  own_p = warp_sum_u64(own_p);
  if ((tid & 31) == 0) {
    s_r[tid >> 5] = own_r;
    s_p[tid >> 5] = own_p;
  }
  __syncthreads();
  if (tid == 0) {
    unsigned long long R = 0, Q = 0;
    for (int w = 0; w < kMassThreads / 32; ++w) {
      R += s_r[w];
      Q += s_p[w];
    }
    P.mass[(static_cast<long long>(b) * P.nslice_d + sl) * 2] = R;
    P.mass[(static_cast<long long>(b) * P.nslice_d + sl) * 2 + 1] = Q;
  }
}

template <typename T, bool BIAS>
__global__ void __launch_bounds__(kMassThreads, 8) small_mass(const SmallParams P) {
  pdl_trigger();
  const int sl = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const SmallDecision d = decide<T, BIAS>(P, b);
  if (sl == 0 && tid == 0) P.dec[b] = d;
  if (!d.ok) return;
  slice_masses<T, BIAS>(P, b, d, sl);
}

// The deferred draws of the walk: CTA (sl, k) sums slice sl of the k-th sequence the walk
// decided, once the walk has published it (seq + 1 in P.dlist[k], written after its decision;
// a bounded wait: the walk's clusters are all running before this launch can start, and none of
// them waits on it). CTAs start in the order the walk decides, so the sums of the sequences
// decided first run while the walk finishes the last ones.
template <typename T, bool BIAS>
__global__ void __launch_bounds__(kMassThreads, 8) walk_mass(const SmallParams P) {
  pdl_trigger();
  __shared__ int s_b;
  const int sl = blockIdx.x, k = blockIdx.y;
  if (threadIdx.x == 0) {
    int b = -1;
    const long long t0 = clock64();
    for (;;) {
      const int v = ld_acquire_gpu_s32(P.dlist + k);
      if (v > 0) {
        b = v - 1;
        break;
      }
      if (clock64() - t0 > kWaitBudget) {
        atomicOr(P.err, 1u);
        break;
      }
      __nanosleep(256);
    }
    s_b = b;
  }
  __syncthreads();
  const int b = s_b;
  if (b < 0 || b >= P.B) return;
  const SmallDecision d = P.dec[b];
  if (!d.ok || d.a < 0 || d.a > P.K) return;
  slice_masses<T, BIAS, true>(P, b, d, sl);
}

template <typename T, bool BIAS>
__global__ void __launch_bounds__(kPickThreads) small_pick(const SmallParams P) {
  __shared__ unsigned long long s_w[kPickThreads / 32];
  __shared__ int s_slice, s_tok;
  __shared__ unsigned long long s_tt;
  __shared__ float s_rho;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  const int K = P.K;
  int32_t* tok = P.out_tok + static_cast<long long>(b) * (K + 1);
  const int32_t* x = P.tokens + static_cast<long long>(b) * K;
  // inputs before the wait: the ids this thread may write out, the draw's uniform
  const int xj = tid < K ? x[tid] : -1;
  const float uK = P.uni[static_cast<long long>(b) * (K + 1) + K];
  pdl_wait();  // decisions and slice masses come from the mass launch
  const SmallDecision d = P.dec[b];
  unsigned long long mr = 0, mp = 0;  // slice masses, one slice per lane of warp 0
  if (tid < 32 && lane < P.nslice_d) {
    const unsigned long long* m = P.mass + (static_cast<long long>(b) * P.nslice_d + lane) * 2;
    mr = m[0];
    mp = m[1];
  }
  if (P.dlist && tid == 0 && d.q >= 0 && d.q < P.B)
    P.dlist[d.q] = 0;  // the walk's order list, empty for the next call
  if (!d.ok || d.a < 0 || d.a > K) {
    for (int j = tid; j <= K; j += kPickThreads) tok[j] = -1;
    // -1 invalid, -2 a bounded wait gave up (the walk's record; or a record out of range)
    if (tid == 0) P.out_acc[b] = (!d.ok && d.a == -1) ? -1 : -2;
    return;
  }
  const int a = d.a;
  if (tid < 32) {
    // the slice that holds floor(u W): the residual's masses, or p's when the residual has none
    const bool use_p = d.rho != 0.f && warp_sum_u64(mr) == 0ull;
    const unsigned long long own = use_p ? mp : mr;
    unsigned long long inc = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(FULL, inc, o);
      if (lane >= o) inc += y;
    }
    const unsigned long long W = __shfl_sync(FULL, inc, 31);
    const unsigned long long tt = scale_floor(uK, W);
    const bool here = W > 0 && tt >= inc - own && tt < inc;
    const unsigned hit = __ballot_sync(FULL, here);
    if (lane == 0) {
      s_slice = hit ? __ffs(hit) - 1 : -1;
      s_rho = use_p ? 0.f : d.rho;
      s_tok = -1;
    }
    if (here) s_tt = tt - (inc - own);
  }
  __syncthreads();
  const int sl = s_slice;
  if (sl >= 0) {
    // inside the slice: each thread's run of up to kPickVecs vectors, in id order
    const int L = P.lens ? P.lens[b] : K;
    const T* gt = static_cast<const T*>(small_row(P, b, a, sizeof(T)));
    const T* gd = a < L ? static_cast<const T*>(small_row(P, b, K + 1 + a, sizeof(T))) : gt;
    const float rho = s_rho, c = P.c;
    const bool al = P.aligned != 0;
    const int e0 = sl * P.slice_d, e1 = min(P.V, e0 + P.slice_d);
    const int nv = (e1 - e0 + 7) >> 3;
    const int per = (nv + kPickThreads - 1) / kPickThreads;  // <= kPickVecs
    const int v0 = tid * per;
    float w[kPickVecs][8];
    unsigned long long q[kPickVecs];
    unsigned long long own = 0;
#pragma unroll
    for (int j = 0; j < kPickVecs; ++j) {
      q[j] = 0;
      if (j < per && v0 + j < nv) {
        float zt[8], zd[8], sr, sp;
        load8_at(gt, e0 + 8 * (v0 + j), e1, al, zt);
        if (rho != 0.f) load8_at(gd, e0 + 8 * (v0 + j), e1, al, zd);
        float rk[8];
        rho8<BIAS>(d, rho, e0 + 8 * (v0 + j), rk);
        weights8(zt, zd, c, d.mct, d.mcd, rk, rho != 0.f, w[j], sr, sp);
        q[j] = qfix(sr);
        own += q[j];
      }
    }
    // block exclusive prefix of the threads' totals (ascending ids)
    unsigned long long inc = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(FULL, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 31) s_w[tid >> 5] = inc;
    __syncthreads();
    unsigned long long pre = inc - own;
    for (int k = 0; k < (tid >> 5); ++k) pre += s_w[k];
    const unsigned long long tt = s_tt;
    if (tt >= pre && tt < pre + own) {
      // the first of the thread's vectors whose end passes tt, then the id inside it
      int js = 0;
      unsigned long long ps = pre;
      bool found = false;
#pragma unroll
      for (int j = 0; j < kPickVecs; ++j) {
        if (!found && pre + q[j] > tt) {
          js = j;
          ps = pre;
          found = true;
        }
        pre += q[j];
      }
      float ws[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        ws[k] = w[0][k];
#pragma unroll
        for (int j = 1; j < kPickVecs; ++j) ws[k] = js == j ? w[j][k] : ws[k];
      }
      float s = 0.f;
      int pick = 7;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        s = k ? __fadd_rn(s, ws[k]) : ws[0];
        if (pick == 7 && ps + qfix(s) > tt) pick = k;
      }
      s_tok = e0 + 8 * (v0 + js) + pick;
    }
  }
  __syncthreads();
  if (tid <= K) tok[tid] = tid < a ? xj : (tid == a ? s_tok : -1);
  if (tid == 0) P.out_acc[b] = a;
}

template <typename Kern>
cudaError_t launch_pdl(Kern kernel, dim3 grid, int threads, cudaStream_t stream,
                       const SmallParams& P) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, P);
}

template <typename T>
cudaError_t launch_small_t(const SmallParams& P, cudaStream_t stream) {
  small_rows<T><<<dim3(static_cast<unsigned>(P.nslice), static_cast<unsigned>(P.B * (2 * P.K + 1))),
                  kRowThreads, 0, stream>>>(P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the bias set's per-id factor only in the variants that have one
  const bool bias = P.bias_k > 0 && P.top8;
  const dim3 gm(static_cast<unsigned>(P.nslice_d), static_cast<unsigned>(P.B));
  e = bias ? launch_pdl(small_mass<T, true>, gm, kMassThreads, stream, P)
           : launch_pdl(small_mass<T, false>, gm, kMassThreads, stream, P);
  if (e != cudaSuccess) return e;
  const dim3 gp(static_cast<unsigned>(P.B));
  return bias ? launch_pdl(small_pick<T, true>, gp, kPickThreads, stream, P)
              : launch_pdl(small_pick<T, false>, gp, kPickThreads, stream, P);
}

}  // namespace

int small_rows_per_sm(int dtype) {
  int n = 0;
  const cudaError_t e =
      dtype == 1
          ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, small_rows<uint16_t>, kRowThreads, 0)
          : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, small_rows<float>, kRowThreads, 0);
  return e == cudaSuccess ? n : 0;
}

bool small_plan(int B, int K, int V, int sms, int rows_per_sm, SmallParams* P) {
  if (B <= 0 || K < 1 || K > kMaxSmallK || V < 1 || sms <= 0 || rows_per_sm <= 0) return false;
  const long long rows = static_cast<long long>(B) * (2 * K + 1);
  // statistics: about one resident CTA per (row, slice), slices of >= 1024 ids
  long long ns = (static_cast<long long>(rows_per_sm) * sms) / rows;
  ns = std::max<long long>(1, std::min<long long>({ns, (V + 1023) / 1024, kMaxSlices}));
  const long long sl = ((V + ns - 1) / ns + 7) / 8 * 8;
  // the draw: about 4 CTAs per multiprocessor, slices of <= kPickThreads * kPickVecs * 8 ids
  const long long cap = static_cast<long long>(kPickThreads) * kPickVecs * 8;
  long long nd = (4LL * sms + B - 1) / B;
  nd = std::max<long long>({1, (V + cap - 1) / cap,
                            std::min<long long>({nd, (V + 1023) / 1024, kMaxSlices})});
  if (nd > kMaxSlices) return false;
  const long long sd = ((V + nd - 1) / nd + 7) / 8 * 8;
  if (sd > cap) return false;
  P->B = B;
  P->K = K;
  P->slice = static_cast<int>(sl);
  P->nslice = static_cast<int>((V + sl - 1) / sl);
  P->slice_d = static_cast<int>(sd);
  P->nslice_d = static_cast<int>((V + sd - 1) / sd);
  return true;
}

cudaError_t launch_small(const SmallParams& P, int dtype, cudaStream_t stream) {
  return dtype == 1 ? launch_small_t<uint16_t>(P, stream) : launch_small_t<float>(P, stream);
}

namespace {
template <typename T>
cudaError_t launch_walk_draws_t(const SmallParams& P, cudaStream_t stream) {
  const dim3 gm(static_cast<unsigned>(P.nslice_d), static_cast<unsigned>(P.B));
  cudaError_t e = launch_pdl(walk_mass<T, false>, gm, kMassThreads, stream, P);
  if (e != cudaSuccess) return e;
  return launch_pdl(small_pick<T, false>, dim3(static_cast<unsigned>(P.B)), kPickThreads, stream,
                    P);
}
}  // namespace

cudaError_t launch_walk_draws(const SmallParams& P, int dtype, cudaStream_t stream) {
  return dtype == 1 ? launch_walk_draws_t<uint16_t>(P, stream)
                    : launch_walk_draws_t<float>(P, stream);
}

}  // namespace sv

// Fused batched speculative-sampling verify kernel for sm_103a.
//
// One thread-block cluster of C CTAs owns one sequence at a time and walks its draft
// positions in order (Kangaroo guide, section "3. Lossless Speculative Verification":
// verification terminates at the first rejection). Each CTA owns a contiguous slice of the
// vocabulary; per position it stages its slice of the target row (and draft row) into its
// own shared memory with one bulk async copy per row, reduces it (max, sum of exponentials,
// argmax, top-8), and the CTAs exchange their partials through distributed shared memory.
// Every CTA then combines the C partials in the same order and reaches the same accept /
// reject decision. After a rejection (or when every draft is accepted) the residual or bonus
// draw runs on the rows that are still resident in the cluster's shared memory, so no row is
// read from HBM twice and rows after the outcome are never read at all.
//
// The residual / bonus mass is summed as 64-bit integers of 2^-44 so the cross-CTA prefix
// used by the inverse-CDF draw is exact and order independent.
//
// Bounded waits: each wait for a bulk copy gives up after ~2 s, raises the workspace error
// word, and the cluster marks the sequence -2 and leaves. There is no other spin-wait; all
// cross-CTA ordering uses the hardware cluster barrier.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "sv_internal.h"
#include "sv_ptx.cuh"

namespace sv {
namespace {

constexpr int NT = kThreads;
constexpr int NW = NT / 32;
constexpr unsigned FULL = 0xffffffffu;
constexpr float kLn2 = 0.69314718055994531f;
constexpr long long kWaitBudget = 4000000000LL;  // clock cycles (about 2 s)
constexpr unsigned XF_ABORT = 1u;

// Partial results one CTA publishes to every CTA of its cluster (7 chunks of 16 bytes).
struct __align__(16) Xchg {
  float m_t, s_t, m_d, s_d;     // chunk 0: slice maxima (raw logits) and sum 2^((z-m)c)
  int arg;                      // chunk 1: greedy, lowest index of the slice maximum
  int next_seq;                 //          rank 0, first exchange of a sequence
  unsigned flags;
  int pad0;
  unsigned long long top8[8];   // chunks 2..5: draft keys, descending
  unsigned long long w;         // chunk 6: residual / bonus mass, fixed point
  unsigned long long pad1;
};
static_assert(sizeof(Xchg) == 112, "exchange record layout");

struct CtaState {
  // sequence header
  int L, hdr_ok, next;
  int x[kMaxK];
  float u[kMaxK + 1];
  float zx_t, zx_d;
  // reduction scratch (one slot per kind, so consecutive reductions need one barrier each)
  float rmax[2][NW];
  float rsum[2][NW];
  int rarg[NW];
  unsigned long long ru[NW];
  unsigned long long wtop[NW][8];
  // record being published
  Xchg rec;
  // cluster-combined values of the current position (written by warp 0)
  float M_t, M_d, S_t, S_d, N;
  int bad_t, bad_d, arg, accept;
  int nS;
  int S_ids[8];
  // sampling
  unsigned long long t_loc;
  int cstar, token;
  // per-sequence outputs kept for the epilogue
  int topf[kMaxK][8];
  float lse_t[kMaxK + 1], lse_d[kMaxK], px[kMaxK], qx[kMaxK];
};

// ------------------------------------------------------------------------------------------
// element access: float rows, or bf16 rows kept as raw 16-bit patterns
// ------------------------------------------------------------------------------------------
template <typename T>
struct Elt;

template <>
struct Elt<float> {
  static __device__ __forceinline__ float val(float v) { return v; }
  static __device__ __forceinline__ float neg_inf() { return -INFINITY; }
  static __device__ __forceinline__ void load8(const float* s, int g, float (&z)[8]) {
    const float4* p = reinterpret_cast<const float4*>(s) + 2 * g;
    const float4 a = p[0], b = p[1];
    z[0] = a.x; z[1] = a.y; z[2] = a.z; z[3] = a.w;
    z[4] = b.x; z[5] = b.y; z[6] = b.z; z[7] = b.w;
  }
};

template <>
struct Elt<uint16_t> {
  static __device__ __forceinline__ float val(uint16_t v) {
    return __uint_as_float(static_cast<uint32_t>(v) << 16);
  }
  static __device__ __forceinline__ uint16_t neg_inf() { return 0xFF80u; }
  static __device__ __forceinline__ void load8(const uint16_t* s, int g, float (&z)[8]) {
    const uint4 v = reinterpret_cast<const uint4*>(s)[g];
    z[0] = __uint_as_float(v.x << 16); z[1] = __uint_as_float(v.x & 0xFFFF0000u);
    z[2] = __uint_as_float(v.y << 16); z[3] = __uint_as_float(v.y & 0xFFFF0000u);
    z[4] = __uint_as_float(v.z << 16); z[5] = __uint_as_float(v.z & 0xFFFF0000u);
    z[6] = __uint_as_float(v.w << 16); z[7] = __uint_as_float(v.w & 0xFFFF0000u);
  }
};

// ------------------------------------------------------------------------------------------
// small helpers
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = max_nan(v, __shfl_xor_sync(FULL, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}
__device__ __forceinline__ int warp_min_int(int v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(FULL, v, o));
  return v;
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(FULL, v, o);
    v = y > v ? y : v;
  }
  return v;
}
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

__device__ __forceinline__ bool row_bad(float m) {
  return isnan(m) || m == INFINITY || m == -INFINITY;
}

// Sort key of a logit: larger value first, then lower id. 0 means "empty".
__device__ __forceinline__ unsigned long long make_key(float z, uint32_t id) {
  const uint32_t b = __float_as_uint(z);
  const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<unsigned long long>(ord) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - id);
}
__device__ __forceinline__ float key_value(unsigned long long k) {
  const uint32_t ord = static_cast<uint32_t>(k >> 32);
  return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}
__device__ __forceinline__ int key_id(unsigned long long k) {
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k));
}

// Integer of 2^-44 units below s (s >= 0, s <= 8).
__device__ __forceinline__ unsigned long long qfix(float s) {
  return __float2ull_rz(__fmul_rn(s, 17592186044416.0f));
}

// floor(u * W) for u in [0, 1) given as a float and W < 2^63, exactly.
__device__ __forceinline__ unsigned long long scale_floor(float u, unsigned long long W) {
  const uint32_t b = __float_as_uint(u);
  const uint32_t e = (b >> 23) & 0xFFu;
  const unsigned long long m = (b & 0x7FFFFFu) | (e ? 0x800000u : 0u);
  if (m == 0) return 0;
  const int shift = (e ? 150 - static_cast<int>(e) : 149);  // u = m * 2^-shift
  const unsigned long long lo = m * W;
  const unsigned long long hi = __umul64hi(m, W);
  if (shift >= 128) return 0;
  if (shift >= 64) return hi >> (shift - 64);
  if (shift == 0) return lo;
  return (lo >> shift) | (hi << (64 - shift));
}

// ------------------------------------------------------------------------------------------
// block reductions (result returned to every thread)
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ float2 block_max2(float a, float b, CtaState& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = warp_max_nan(a);
  b = warp_max_nan(b);
  if (lane == 0) { S.rmax[0][warp] = a; S.rmax[1][warp] = b; }
  __syncthreads();
  float ra = S.rmax[0][0], rb = S.rmax[1][0];
#pragma unroll
  for (int w = 1; w < NW; ++w) { ra = max_nan(ra, S.rmax[0][w]); rb = max_nan(rb, S.rmax[1][w]); }
  return make_float2(ra, rb);
}

__device__ __forceinline__ float2 block_sum2(float a, float b, CtaState& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = warp_sum(a);
  b = warp_sum(b);
  if (lane == 0) { S.rsum[0][warp] = a; S.rsum[1][warp] = b; }
  __syncthreads();
  // pairwise over the warps keeps the rounding error at log2(NW) steps
  float va[NW], vb[NW];
#pragma unroll
  for (int w = 0; w < NW; ++w) { va[w] = S.rsum[0][w]; vb[w] = S.rsum[1][w]; }
#pragma unroll
  for (int s = NW / 2; s; s >>= 1)
#pragma unroll
    for (int w = 0; w < s; ++w) { va[w] += va[w + s]; vb[w] += vb[w + s]; }
  return make_float2(va[0], vb[0]);
}

__device__ __forceinline__ int block_min_int(int v, CtaState& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_min_int(v);
  if (lane == 0) S.rarg[warp] = v;
  __syncthreads();
  int r = S.rarg[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) r = min(r, S.rarg[w]);
  return r;
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, CtaState& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_u64(v);
  if (lane == 0) S.ru[warp] = v;
  __syncthreads();
  unsigned long long r = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) r += S.ru[w];
  __syncthreads();
  return r;
}

// Exclusive prefix over the threads in id order.
__device__ __forceinline__ unsigned long long block_exclusive_u64(unsigned long long v,
                                                                  CtaState& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(FULL, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) S.ru[warp] = inc;
  __syncthreads();
  unsigned long long base = 0;
  for (int w = 0; w < warp; ++w) base += S.ru[w];
  __syncthreads();
  return base + inc - v;
}

// ------------------------------------------------------------------------------------------
// row passes over the staged slice (vectors of 8 elements, vector g covers elements 8g..8g+7)
// ------------------------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ float slice_max(const T* row, int nvec) {
  if constexpr (sizeof(T) == 2) {
    uint32_t acc = 0xFF80FF80u;  // (-inf, -inf)
    for (int g = threadIdx.x; g < nvec; g += NT) {
      const uint4 v = reinterpret_cast<const uint4*>(row)[g];
      acc = max_nan_bf16x2(acc, max_nan_bf16x2(max_nan_bf16x2(v.x, v.y), max_nan_bf16x2(v.z, v.w)));
    }
    return max_nan(__uint_as_float(acc << 16), __uint_as_float(acc & 0xFFFF0000u));
  } else {
    float acc = -INFINITY;
    for (int g = threadIdx.x; g < nvec; g += NT) {
      float z[8];
      Elt<T>::load8(row, g, z);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc = max_nan(acc, z[k]);
    }
    return acc;
  }
}

// Sum of 2^(z c - mc) over the slice; mc is m*c rounded to float.
template <typename T>
__device__ __forceinline__ float slice_sum(const T* row, int nvec, float c, float mc) {
  float s0 = 0.f, s1 = 0.f;
  for (int g = threadIdx.x; g < nvec; g += NT) {
    float z[8];
    Elt<T>::load8(row, g, z);
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
      s0 += ex2_fast(fmaf(z[k], c, -mc));
      s1 += ex2_fast(fmaf(z[k + 1], c, -mc));
    }
  }
  return s0 + s1;
}

// Lowest slice-local index whose value equals m (INT_MAX if none).
template <typename T>
__device__ __forceinline__ int slice_first_index(const T* row, int nvec, float m) {
  for (int g = threadIdx.x; g < nvec; g += NT) {
    float z[8];
    Elt<T>::load8(row, g, z);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (z[k] == m) return 8 * g + k;
  }
  return 0x7FFFFFFF;
}

template <typename T>
__device__ __forceinline__ void slice_top8(const T* row, int nv, int nvec, int v0,
                                           unsigned long long (&keys)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) keys[j] = 0ull;
  float thr = -INFINITY;
  for (int g = threadIdx.x; g < nvec; g += NT) {
    float z[8];
    Elt<T>::load8(row, g, z);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int e = 8 * g + k;
      if (e < nv && z[k] >= thr) {
        unsigned long long key = make_key(z[k], static_cast<uint32_t>(v0 + e));
        if (key > keys[7]) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const unsigned long long hi = key > keys[j] ? key : keys[j];
            const unsigned long long lo = key > keys[j] ? keys[j] : key;
            keys[j] = hi;
            key = lo;
          }
          if (keys[7]) thr = key_value(keys[7]);
        }
      }
    }
  }
}

// Merge every thread's descending top-8 into the CTA's top-8 (written to S.rec.top8).
__device__ __forceinline__ void block_top8(unsigned long long (&keys)[8], CtaState& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const unsigned long long m = warp_max_u64(keys[0]);
    if (m != 0ull && keys[0] == m) {
#pragma unroll
      for (int j = 0; j < 7; ++j) keys[j] = keys[j + 1];
      keys[7] = 0ull;
    }
    if (lane == 0) S.wtop[warp][r] = m;
  }
  __syncthreads();
  if (warp == 0) {
    static_assert(NW * 8 == 64, "two candidates per lane");
    unsigned long long a0 = S.wtop[lane >> 3][lane & 7];
    unsigned long long a1 = S.wtop[(lane >> 3) + 4][lane & 7];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const unsigned long long b = a0 > a1 ? a0 : a1;
      const unsigned long long m = warp_max_u64(b);
      if (m != 0ull) {
        if (a0 == m) a0 = 0ull;
        else if (a1 == m) a1 = 0ull;
      }
      if (lane == 0) S.rec.top8[r] = m;
    }
  }
}

// Publish chunks [c0, c0 + nc) of S.rec into slot `rank` of buffer `par` of every CTA of the
// cluster, then wait for every CTA to have done the same.
__device__ __forceinline__ void exchange(CtaState& S, Xchg (*X)[kMaxCluster], uint32_t par,
                                         uint32_t rank, uint32_t C, int c0, int nc) {
  const int tid = threadIdx.x;
  if (tid < static_cast<int>(C) * nc) {
    const uint32_t peer = tid / nc;
    const int ch = c0 + tid % nc;
    const uint32_t dst = map_to_rank(smem_u32(&X[par][rank]) + 16u * ch, peer);
    st_cluster_v4(dst, reinterpret_cast<const uint4*>(&S.rec)[ch]);
  }
  cluster_sync();
}

// Stage this CTA's slice of the requested rows into shared memory. Returns true if the bulk
// copy did not complete within the wait budget (same answer in every thread of the CTA).
template <typename T>
__device__ __forceinline__ bool stage_rows(T* rt, T* rd, const T* gt, const T* gd, bool ld_t,
                                           bool ld_d, int nv, int nb, int nvec, uint64_t* bar,
                                           uint32_t& tpar) {
  const int tid = threadIdx.x;
  if (nb > 0 && tid == 0) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const uint32_t bytes = static_cast<uint32_t>(nb * sizeof(T));
    mbar_arrive_expect_tx(bar, bytes * ((ld_t ? 1u : 0u) + (ld_d ? 1u : 0u)));
    if (ld_t) bulk_g2s(rt, gt, bytes, bar);
    if (ld_d) bulk_g2s(rd, gd, bytes, bar);
  }
  // elements the bulk copy does not cover, then -inf padding to a whole vector of 8
  for (int e = nb + tid; e < 8 * nvec; e += NT) {
    if (ld_t) rt[e] = e < nv ? gt[e] : Elt<T>::neg_inf();
    if (ld_d) rd[e] = e < nv ? gd[e] : Elt<T>::neg_inf();
  }
  bool late = false;
  if (nb > 0) {
    late = !mbar_wait_bounded(bar, tpar, kWaitBudget);
    tpar ^= 1u;
  }
  return __syncthreads_or(late) != 0;
}

// ------------------------------------------------------------------------------------------
// residual / bonus draw
// ------------------------------------------------------------------------------------------
struct WeightConsts {
  float c, mc_t, mc_d, r_t, r_d, r_dS;
  int nloc;          // S ids that fall in this CTA's slice
  int loc[8];        // their slice-local indices
};

// Weights of vector g: bonus -> 2^(z_t c - mc_t); residual -> max(p - q', 0) with p and q'
// rebuilt from the staged rows. Returns the sequential sum of the 8 weights.
template <typename T, bool BONUS>
__device__ __forceinline__ float weights8(const T* rt, const T* rd, int g,
                                          const WeightConsts& K, float (&w)[8]) {
  float zt[8];
  Elt<T>::load8(rt, g, zt);
  if constexpr (BONUS) {
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = ex2_fast(fmaf(zt[k], K.c, -K.mc_t));
  } else {
    float zd[8];
    Elt<T>::load8(rd, g, zd);
    float rdk[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) rdk[k] = K.r_d;
    for (int j = 0; j < K.nloc; ++j) {
      const int e = K.loc[j] - 8 * g;
      if (e >= 0 && e < 8) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (k == e) rdk[k] = K.r_dS;
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float et = ex2_fast(fmaf(zt[k], K.c, -K.mc_t));
      const float ed = ex2_fast(fmaf(zd[k], K.c, -K.mc_d));
      w[k] = fmaxf(fmaf(et, K.r_t, -__fmul_rn(ed, rdk[k])), 0.f);
    }
  }
  float s = w[0];
#pragma unroll
  for (int k = 1; k < 8; ++k) s = __fadd_rn(s, w[k]);
  return s;
}

// The cluster draws the token at position `a` of sequence `seq` and the CTA that owns it
// writes out_tok. All threads of all CTAs of the cluster call this together.
template <typename T, bool BONUS>
__device__ void draw_token(const Params& P, CtaState& S, Xchg (*X)[kMaxCluster],
                           uint32_t& xpar, uint32_t rank, uint32_t C, const T* rt,
                           const T* rd, int nvec, int v0, int nv, int seq, int a) {
  const int tid = threadIdx.x;
  WeightConsts W;
  W.c = P.c;
  W.mc_t = __fmul_rn(S.M_t, P.c);
  const float err_t = fmaf(S.M_t, P.c, -W.mc_t);
  // p(v) = 2^(z c - mc_t) * 2^(-err_t) / S_t
  W.r_t = BONUS ? 1.f : fmaf(-err_t, kLn2, 1.f) / S.S_t;
  W.mc_d = __fmul_rn(S.M_d, P.c);
  const float err_d = fmaf(S.M_d, P.c, -W.mc_d);
  W.r_d = BONUS ? 0.f : fmaf(-err_d, kLn2, 1.f) / (S.S_d * S.N);
  W.r_dS = W.r_d * P.beta;
  W.nloc = 0;
  for (int j = 0; j < S.nS; ++j) {
    const int e = S.S_ids[j] - v0;
    if (e >= 0 && e < nv) W.loc[W.nloc++] = e;
  }
  unsigned long long Wc = 0, Wtot = 0;
  for (int attempt = 0; attempt < 2; ++attempt) {
    unsigned long long acc = 0;
    float w[8];
    for (int g = tid; g < nvec; g += NT) acc += qfix(weights8<T, BONUS>(rt, rd, g, W, w));
    Wc = block_sum_u64(acc, S);
    if (tid == 0) S.rec.w = Wc;
    __syncthreads();
    exchange(S, X, xpar, rank, C, 6, 1);
    const Xchg* XX = X[xpar];
    xpar ^= 1u;
    // every thread forms the same prefix over the CTAs
    Wtot = 0;
    for (uint32_t c = 0; c < C; ++c) Wtot += XX[c].w;
    if (tid == 0) {
      const unsigned long long t = scale_floor(S.u[P.K], Wtot);
      unsigned long long pre = 0;
      int cs = -1;
      for (uint32_t c = 0; c < C; ++c) {
        if (cs < 0 && t < pre + XX[c].w) { cs = static_cast<int>(c); S.t_loc = t - pre; }
        pre += XX[c].w;
      }
      S.cstar = cs;
      S.token = -1;
    }
    __syncthreads();
    if (Wtot > 0 || BONUS) break;
    // zero residual mass: draw from p at this position instead
    W.r_d = 0.f;
    W.r_dS = 0.f;
  }
  if (S.cstar == static_cast<int>(rank)) {
    // contiguous chunks of vectors per thread, so the CDF follows ascending ids
    const int lo = static_cast<int>((static_cast<long long>(tid) * nvec) / NT);
    const int hi = static_cast<int>((static_cast<long long>(tid + 1) * nvec) / NT);
    float w[8];
    unsigned long long csum = 0;
    for (int g = lo; g < hi; ++g) csum += qfix(weights8<T, BONUS>(rt, rd, g, W, w));
    unsigned long long pre = block_exclusive_u64(csum, S);
    const unsigned long long tl = S.t_loc;
    if (pre <= tl && tl < pre + csum) {
      for (int g = lo; g < hi; ++g) {
        const unsigned long long q = qfix(weights8<T, BONUS>(rt, rd, g, W, w));
        if (pre + q > tl) {
          float s = 0.f;
          int pick = 7;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            s = k ? __fadd_rn(s, w[k]) : w[0];
            if (pre + qfix(s) > tl) { pick = k; break; }
          }
          S.token = v0 + 8 * g + pick;
          break;
        }
        pre += q;
      }
    }
    __syncthreads();
    if (tid == 0) P.out_tok[static_cast<long long>(seq) * (P.K + 1) + a] = S.token;
  }
  __syncthreads();
}

// ------------------------------------------------------------------------------------------
// combine the C partials of a position (warp 0); results land in S
// ------------------------------------------------------------------------------------------
template <bool GREEDY>
__device__ void combine(const Params& P, CtaState& S, const Xchg* XX, uint32_t C, int i,
                        bool st_t, bool st_d, bool tk, bool ld_d) {
  const int lane = threadIdx.x & 31;
  const bool have = lane < static_cast<int>(C);
  const float mt = have ? XX[lane].m_t : -INFINITY;
  const float md = have ? XX[lane].m_d : -INFINITY;
  const float Mt = warp_max_nan(mt);
  const float Md = warp_max_nan(md);
  if constexpr (GREEDY) {
    const int arg = (have && mt == Mt) ? XX[lane].arg : 0x7FFFFFFF;
    const int best = warp_min_int(arg);
    if (lane == 0) { S.M_t = Mt; S.bad_t = row_bad(Mt); S.arg = best; }
    return;
  } else {
    const float c = P.c;
    float tt = 0.f, td = 0.f;
    if (have && st_t && !row_bad(Mt) && mt > -INFINITY) tt = XX[lane].s_t * exp2f((mt - Mt) * c);
    if (have && st_d && !row_bad(Md) && md > -INFINITY) td = XX[lane].s_d * exp2f((md - Md) * c);
    const float St = warp_sum(tt);
    const float Sd = warp_sum(td);
    unsigned long long mtop[8];
    if (tk) {
      int ptr = 0;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const unsigned long long h = (have && ptr < 8) ? XX[lane].top8[ptr] : 0ull;
        const unsigned long long m = warp_max_u64(h);
        if (m != 0ull && h == m) ++ptr;
        mtop[r] = m;
      }
    }
    if (lane != 0) return;
    S.M_t = Mt; S.M_d = Md; S.S_t = St; S.S_d = Sd;
    S.bad_t = row_bad(Mt);
    S.bad_d = ld_d ? row_bad(Md) : 0;
    // Saguaro bias set: the bias_k most likely draft ids
    float N = 1.f;
    int nS = 0;
    if (P.bias_k > 0 && tk && !S.bad_d) {
      float sq = 0.f;
      for (int j = 0; j < P.bias_k; ++j) {
        if (mtop[j] == 0ull) break;
        const float z = key_value(mtop[j]);
        sq += exp2f((z - Md) * c) / Sd;
        S.S_ids[nS++] = key_id(mtop[j]);
      }
      N = fmaf(-(1.f - P.beta), sq, 1.f);
    }
    S.nS = nS;
    S.N = N;
    if (tk && P.fmax > 0 && i < S.L) {
      for (int f = 0; f < 8; ++f)
        S.topf[i][f] = (f < P.fan[i] && mtop[f] != 0ull) ? key_id(mtop[f]) : -1;
    }
    if (st_t && !S.bad_t) S.lse_t[i] = Mt / P.temperature + logf(St);
    if (st_d && !S.bad_d) S.lse_d[i] = Md / P.temperature + logf(Sd);
    S.accept = 0;
    if (st_t && st_d && i < S.L && !S.bad_t && !S.bad_d) {
      const int x = S.x[i];
      const float zt = S.zx_t, zd = S.zx_d;
      bool inS = false;
      for (int j = 0; j < nS; ++j) inS |= (S.S_ids[j] == x);
      const float f = inS ? P.beta : 1.f;
      float ratio;
      if (zt == -INFINITY) ratio = 0.f;
      else if (zd == -INFINITY) ratio = INFINITY;
      else ratio = exp2f(((zt - zd) - (Mt - Md)) * c) * (Sd / St) * (N / f);
      const float px = zt == -INFINITY ? 0.f : exp2f((zt - Mt) * c) / St;
      const float qx = zd == -INFINITY ? 0.f : exp2f((zd - Md) * c) * f / (Sd * N);
      S.px[i] = px;
      S.qx[i] = qx;
      S.accept = S.u[i] < ratio;
    }
  }
}

// ------------------------------------------------------------------------------------------
// the kernel
// ------------------------------------------------------------------------------------------
template <typename T, bool GREEDY>
__global__ void __launch_bounds__(NT, 2) verify_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ CtaState S;
  __shared__ Xchg X[2][kMaxCluster];
  __shared__ uint64_t mbar;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const uint32_t C = cluster_nctarank();
  const int cid = static_cast<int>(cluster_id_x());
  T* rt = reinterpret_cast<T*>(dyn);
  T* rd = rt + P.slice;
  const int v0 = static_cast<int>(rank) * P.slice;
  const int nv = max(0, min(P.V - v0, P.slice));
  const int nvec = (nv + 7) >> 3;
  constexpr int kPer16 = 16 / static_cast<int>(sizeof(T));
  const int nb = P.use_bulk ? (nv / kPer16) * kPer16 : 0;
  const T* gtb = reinterpret_cast<const T*>(P.tgt);
  const T* gdb = reinterpret_cast<const T*>(P.dft);
  const int K = P.K;

  if (tid == 0) {
    mbar_init(&mbar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync();  // every CTA of the cluster is running before any shared-memory exchange

  uint32_t xpar = 0, tpar = 0;
  bool aborted = false;
  int seq = cid;
  while (seq < P.B) {
    // ---- sequence header: every CTA reads the same few words ----
    if (tid == 0) {
      const int L = P.lens ? P.lens[seq] : K;
      int ok = (L >= 1 && L <= K);
      for (int i = 0; i < K; ++i) {
        const int x = P.tokens[static_cast<long long>(seq) * K + i];
        S.x[i] = x;
        if (i < L && (x < 0 || x >= P.V)) ok = 0;
      }
      if (!GREEDY) {
        for (int i = 0; i <= K; ++i) {
          const float u = P.uni[static_cast<long long>(seq) * (K + 1) + i];
          S.u[i] = u;
          if ((i < L || i == K) && !(u >= 0.f && u < 1.f)) ok = 0;
        }
      }
      S.L = L;
      S.hdr_ok = ok;
      S.next = rank == 0 ? static_cast<int>(atomicAdd(&P.ws->next, 1u)) + P.n_clusters : 0;
      for (int i = 0; i < kMaxK; ++i) {
        for (int f = 0; f < 8; ++f) S.topf[i][f] = -1;
        S.lse_d[i] = S.px[i] = S.qx[i] = NAN;
      }
      for (int i = 0; i <= kMaxK; ++i) S.lse_t[i] = NAN;
    }
    __syncthreads();
    const int L = S.L;
    bool invalid = !S.hdr_ok;
    bool decided = invalid;
    bool first = true;
    int a = -1;
    int next = P.B;
    for (int i = 0;; ++i) {
      const bool st_t = !invalid && i <= L && (!decided || P.debug_all);
      const bool st_d = !GREEDY && !invalid && i < L && (!decided || P.debug_all);
      const bool tk = !GREEDY && !invalid && i < L && P.top8 &&
                      (!decided || P.fmax > 0 || P.debug_all);
      const bool ld_t = st_t, ld_d = st_d || tk;
      if (!ld_t && !ld_d && !first) break;
      bool late = false;
      if (ld_t || ld_d) {
        const T* gt = gtb + (static_cast<long long>(seq) * (K + 1) + i) * P.t_stride + v0;
        const T* gd = GREEDY ? nullptr
                             : gdb + (static_cast<long long>(seq) * K + i) * P.d_stride + v0;
        if (!GREEDY && tid == 0 && st_t && st_d && i < L) {
          const long long x = S.x[i] - v0;  // gathered logits of the draft token
          S.zx_t = Elt<T>::val(gt[x]);
          S.zx_d = Elt<T>::val(gd[x]);
        }
        late = stage_rows<T>(rt, rd, gt, gd, ld_t, ld_d, nv, nb, nvec, &mbar, tpar);
      }
      // ---- this CTA's partials ----
      const float2 mm = block_max2(ld_t && !late ? slice_max<T>(rt, nvec) : -INFINITY,
                                   ld_d && !late ? slice_max<T>(rd, nvec) : -INFINITY, S);
      float2 ss = make_float2(0.f, 0.f);
      int arg = 0x7FFFFFFF;
      if constexpr (GREEDY) {
        if (ld_t && !late && !row_bad(mm.x)) {
          const int e = slice_first_index<T>(rt, nvec, mm.x);
          arg = block_min_int(e, S);
          if (arg != 0x7FFFFFFF) arg += v0;
        }
      } else {
        const float c = P.c;
        const bool sum_t = st_t && !late && !row_bad(mm.x);
        const bool sum_d = st_d && !late && !row_bad(mm.y);
        const float mct = __fmul_rn(mm.x, c), mcd = __fmul_rn(mm.y, c);
        ss = block_sum2(sum_t ? slice_sum<T>(rt, nvec, c, mct) : 0.f,
                        sum_d ? slice_sum<T>(rd, nvec, c, mcd) : 0.f, S);
        // fold the rounding of m*c back in: the sums are relative to exactly m
        if (sum_t) ss.x *= fmaf(-fmaf(mm.x, c, -mct), kLn2, 1.f);
        if (sum_d) ss.y *= fmaf(-fmaf(mm.y, c, -mcd), kLn2, 1.f);
        if (tk && !late) {
          unsigned long long keys[8];
          slice_top8<T>(rd, nv, nvec, v0, keys);
          block_top8(keys, S);
        } else if (tk && tid == 0) {
          for (int r = 0; r < 8; ++r) S.rec.top8[r] = 0ull;
        }
      }
      if (tid == 0) {
        S.rec.m_t = mm.x; S.rec.s_t = ss.x;
        S.rec.m_d = mm.y; S.rec.s_d = ss.y;
        S.rec.arg = arg;
        S.rec.next_seq = first ? S.next : 0;
        S.rec.flags = late ? XF_ABORT : 0u;
        if (late) atomicOr(&P.ws->error, 1u);
      }
      __syncthreads();
      exchange(S, X, xpar, rank, C, 0, tk ? 6 : 2);
      const Xchg* XX = X[xpar];
      xpar ^= 1u;
      if (first) { next = XX[0].next_seq; first = false; }
      bool ab = false;
      for (uint32_t c = 0; c < C; ++c) ab |= (XX[c].flags & XF_ABORT) != 0u;
      if (ab) { aborted = true; break; }
      if (!ld_t && !ld_d) break;  // header was invalid: the exchange only carried `next`
      if (warp == 0) combine<GREEDY>(P, S, XX, C, i, st_t, st_d, tk, ld_d);
      __syncthreads();
      if (!decided) {
        if (S.bad_t || (i < L && !GREEDY && S.bad_d)) { invalid = true; break; }
        if constexpr (GREEDY) {
          if (!(i < L && S.x[i] == S.arg)) { a = i; decided = true; }
        } else {
          if (i < L) {
            if (!S.accept) {
              a = i;
              decided = true;
              draw_token<T, false>(P, S, X, xpar, rank, C, rt, rd, nvec, v0, nv, seq, a);
            }
          } else {
            a = L;
            decided = true;
            draw_token<T, true>(P, S, X, xpar, rank, C, rt, rd, nvec, v0, nv, seq, a);
          }
        }
      } else if (tk && P.fmax > 0 && S.bad_d) {
        invalid = true;  // a draft row the top-F output needs holds no distribution
        break;
      }
    }
    // ---- epilogue: rank 0 writes the outputs of this sequence ----
    if (rank == 0) {
      int32_t* tok = P.out_tok + static_cast<long long>(seq) * (K + 1);
      const bool bad = aborted || invalid;
      if (tid == 0) P.out_acc[seq] = aborted ? -2 : (invalid ? -1 : a);
      for (int j = tid; j <= K; j += NT) {
        if (bad || j > a) tok[j] = -1;
        else if (j < a) tok[j] = S.x[j];
        else if (GREEDY) tok[j] = S.arg;
      }
      if (P.fmax > 0) {
        int32_t* tf = P.out_topf + static_cast<long long>(seq) * K * P.fmax;
        for (int e = tid; e < K * P.fmax; e += NT) {
          const int i = e / P.fmax, f = e % P.fmax;
          tf[e] = (!bad && i < L && f < 8) ? S.topf[i][f] : -1;
        }
      }
      if (P.dbg_lse_t && tid <= K) P.dbg_lse_t[static_cast<long long>(seq) * (K + 1) + tid] = S.lse_t[tid];
      if (tid < K) {
        const long long o = static_cast<long long>(seq) * K + tid;
        if (P.dbg_lse_d) P.dbg_lse_d[o] = S.lse_d[tid];
        if (P.dbg_px) P.dbg_px[o] = S.px[tid];
        if (P.dbg_qx) P.dbg_qx[o] = S.qx[tid];
      }
    }
    __syncthreads();
    if (aborted) break;
    seq = next;
  }
  cluster_sync();
  if (rank == 0 && tid == 0) {
    __threadfence();
    const unsigned old = atomicAdd(&P.ws->done, 1u);
    if (old == static_cast<unsigned>(P.n_clusters) - 1u) {
      atomicExch(&P.ws->next, 0u);
      atomicExch(&P.ws->done, 0u);
    }
  }
}

template <typename T, bool GREEDY>
const void* kernel_ptr() {
  return reinterpret_cast<const void*>(&verify_kernel<T, GREEDY>);
}

const void* pick(int dtype, int greedy) {
  if (dtype == 1) return greedy ? kernel_ptr<uint16_t, true>() : kernel_ptr<uint16_t, false>();
  return greedy ? kernel_ptr<float, true>() : kernel_ptr<float, false>();
}

cudaError_t prepare(const void* fn, int cluster, size_t smem) {
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (cluster > 8) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

size_t smem_bytes(int dtype, int greedy, int slice) {
  const size_t elt = dtype == 1 ? 2 : 4;
  const size_t rows = greedy ? 1 : 2;
  return (rows * elt * static_cast<size_t>(slice) + 127) / 128 * 128;
}

int max_active_clusters(int dtype, int greedy, int cluster, size_t smem) {
  const void* fn = pick(dtype, greedy);
  if (prepare(fn, cluster, smem) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cluster) * 64u);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) return 0;
  return n;
}

cudaError_t launch(const Launch& L, cudaStream_t stream) {
  const void* fn = pick(L.dtype, L.greedy);
  cudaError_t e = prepare(fn, L.cluster, L.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(L.p.n_clusters * L.cluster));
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = L.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(L.cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<Params*>(&L.p)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace sv

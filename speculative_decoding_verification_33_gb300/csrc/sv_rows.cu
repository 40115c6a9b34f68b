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
// One thread-block cluster of C CTAs per row (sampling) or per (sequence, position) pair
// (residual); each CTA owns a contiguous slice of the vocabulary, read with 128-bit loads issued
// a batch at a time so that every thread keeps several in flight.
//
// Sampling reads its row once. Each 8-element vector's mass, the sum of 2^(z c - m c), is kept in
// shared memory relative to the thread's running maximum m (rescaled when m rises); once the
// cluster has combined the row maximum and sum, every mass is brought to the row maximum with
// one factor per thread and the (at most 8) biased ids are corrected. That gives the fixed-point
// masses of the inverse CDF without a second pass over the row: only the 8 elements of the
// chosen vector are read again.
//
// The residual needs the normalisers of both rows before any weight is known, so it reads the
// pair twice (the second pass mostly from L2). In that pass an element whose target weight
// 2^(z_t c - M_t c) is already below the warp's 8th best residual cannot enter the top 8 (the
// residual never exceeds it): the test is a compare in the log domain, and only the elements
// that pass it pay for exponentials.
//
// Top-8 selections (the bias set, the residual ids) keep one running list per warp, spread over
// lanes 0..7, with a threshold every lane shares: after the first few offers almost every
// element fails one compare and the warp moves on after a single vote.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "sv_internal.h"
#include "sv_math.cuh"
#include "sv_ptx.cuh"
#include "sv_rows.h"

namespace sv {
namespace {

constexpr int RT = kRowThreads;
constexpr int RW = RT / 32;
constexpr float kLn2r = 0.69314718055994531f;
constexpr int MODE_SAMPLE = 0, MODE_RESID = 1;

// ------------------------------------------------------------------------------------------
// raw 8-element vectors (loaded first, converted when used)
// ------------------------------------------------------------------------------------------
template <typename T>
struct Raw8;

template <>
struct Raw8<uint16_t> {
  uint4 a;
  static constexpr int kBatch = 4;  // vectors per thread per batch of loads
  __device__ __forceinline__ void load(const uint16_t* row, int e, int nv, bool vec) {
    if (vec && e + 8 <= nv) {
      a = ldg_nc_v4(row + e);
      return;
    }
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t lo = (e + 2 * k < nv) ? row[e + 2 * k] : 0xFF80u;
      const uint32_t hi = (e + 2 * k + 1 < nv) ? row[e + 2 * k + 1] : 0xFF80u;
      w[k] = lo | (hi << 16);
    }
    a = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __device__ __forceinline__ void get(float (&z)[8]) const { Elt<uint16_t>::unpack(a, z); }
};

template <>
struct Raw8<float> {
  uint4 a, b;
  static constexpr int kBatch = 2;
  __device__ __forceinline__ void load(const float* row, int e, int nv, bool vec) {
    if (vec && e + 8 <= nv) {
      a = ldg_nc_v4(row + e);
      b = ldg_nc_v4(row + e + 4);
      return;
    }
    float t[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) t[k] = (e + k < nv) ? row[e + k] : -INFINITY;
    a = make_uint4(__float_as_uint(t[0]), __float_as_uint(t[1]), __float_as_uint(t[2]),
                   __float_as_uint(t[3]));
    b = make_uint4(__float_as_uint(t[4]), __float_as_uint(t[5]), __float_as_uint(t[6]),
                   __float_as_uint(t[7]));
  }
  __device__ __forceinline__ void get(float (&z)[8]) const {
    z[0] = __uint_as_float(a.x); z[1] = __uint_as_float(a.y);
    z[2] = __uint_as_float(a.z); z[3] = __uint_as_float(a.w);
    z[4] = __uint_as_float(b.x); z[5] = __uint_as_float(b.y);
    z[6] = __uint_as_float(b.z); z[7] = __uint_as_float(b.w);
  }
};

__device__ __forceinline__ float max8(const float (&z)[8]) {
  return max_nan(max_nan(max_nan(z[0], z[1]), max_nan(z[2], z[3])),
                 max_nan(max_nan(z[4], z[5]), max_nan(z[6], z[7])));
}

// ------------------------------------------------------------------------------------------
// shared state and block / cluster reductions
// ------------------------------------------------------------------------------------------
// A CTA's pass-1 partial, read by every CTA of the cluster.
struct __align__(16) StatPart {
  float m_t, s_t, m_d, s_d;   // slice maxima and sums 2^(z c - M c) (rounding of M c folded in)
  unsigned long long top[8];  // the draft slice's top-8 keys (bias set), descending
};

struct RowShared {
  float rmax[2][RW], rsum[2][RW];
  unsigned long long ru[RW];
  unsigned long long wtop[RW][8];
  StatPart part;
  alignas(16) unsigned long long part_w[2];  // sampling: the slice's fixed-point mass
  alignas(16) unsigned long long part_r[8];  // residual: the slice's top-8 residual keys
  // cluster-combined values (identical in every CTA)
  float Mt, St, Md, Sd, N;
  int bad, nS;
  int S_ids[8];
  float S_z[8];
  unsigned long long t_loc;
  int cstar, token;
};

__device__ __forceinline__ void bsync() { __syncthreads(); }

// The two halves of cluster_sync(), for work that may run between them.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

__device__ float2 row_block_max2(float a, float b, RowShared& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = warp_max_nan(a);
  b = warp_max_nan(b);
  if (lane == 0) {
    S.rmax[0][warp] = a;
    S.rmax[1][warp] = b;
  }
  bsync();
  float ra = S.rmax[0][0], rb = S.rmax[1][0];
#pragma unroll
  for (int w = 1; w < RW; ++w) {
    ra = max_nan(ra, S.rmax[0][w]);
    rb = max_nan(rb, S.rmax[1][w]);
  }
  bsync();
  return make_float2(ra, rb);
}

__device__ float2 row_block_sum2(float a, float b, RowShared& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = warp_sum(a);
  b = warp_sum(b);
  if (lane == 0) {
    S.rsum[0][warp] = a;
    S.rsum[1][warp] = b;
  }
  bsync();
  float va = 0.f, vb = 0.f;
#pragma unroll
  for (int w = 0; w < RW; ++w) {
    va += S.rsum[0][w];
    vb += S.rsum[1][w];
  }
  bsync();
  return make_float2(va, vb);
}

__device__ unsigned long long row_block_sum_u64(unsigned long long v, RowShared& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_u64(v);
  if (lane == 0) S.ru[warp] = v;
  bsync();
  unsigned long long r = 0;
#pragma unroll
  for (int w = 0; w < RW; ++w) r += S.ru[w];
  bsync();
  return r;
}

__device__ __forceinline__ unsigned long long warp_inclusive_u64(unsigned long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(FULL, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

__device__ unsigned long long row_block_exclusive_u64(unsigned long long v, RowShared& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned long long inc = warp_inclusive_u64(v);
  if (lane == 31) S.ru[warp] = inc;
  bsync();
  unsigned long long base = 0;
  for (int w = 0; w < warp; ++w) base += S.ru[w];
  bsync();
  return base + inc - v;
}

// The insertion behind WarpTop8::offer, out of line (its loop is long and rarely taken); state in
// and out by value so that it stays in registers.
struct Top8State {
  unsigned long long L;
  float thr;
};

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
      const unsigned long long l7 = __shfl_sync(FULL, st.L, 7);
      if (l7) st.thr = key_value(l7);
    }
  }
  return st;
}

// A warp's running top 8: the keys, descending, in lanes 0..7 (0 = empty; the other lanes hold
// 0), and the value of the 8th (-inf until 8 are held). An offer below it cannot enter, so after
// the first few the common case is one compare and one vote per element.
struct WarpTop8 {
  unsigned long long L;
  float thr;
  __device__ __forceinline__ void init() {
    L = 0ull;
    thr = -INFINITY;
  }
  // Every lane of the warp calls this; lane offers (z, id) when ok. True if the threshold rose.
  __device__ __forceinline__ bool offer(bool ok, float z, uint32_t id) {
    const unsigned pend = __ballot_sync(FULL, ok && z >= thr);
    if (!pend) return false;
    const float before = thr;
    const Top8State st = warp_top8_insert(pend, z, id, Top8State{L, thr});
    L = st.L;
    thr = st.thr;
    return thr != before;
  }
};

// The warps' lists into the CTA's top 8 at dst (written by warp 0).
__device__ void row_block_top8w(const WarpTop8& W, RowShared& S, unsigned long long* dst) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane < 8) S.wtop[warp][lane] = W.L;
  bsync();
  if (warp == 0) {
    static_assert(RW * 8 == 64, "two candidates per lane");
    const unsigned long long c0 = S.wtop[lane >> 3][lane & 7];
    const unsigned long long c1 = S.wtop[(lane >> 3) + 4][lane & 7];
    unsigned long long k8[8];
    k8[0] = c0 > c1 ? c0 : c1;
    k8[1] = c0 > c1 ? c1 : c0;
#pragma unroll
    for (int j = 2; j < 8; ++j) k8[j] = 0ull;
    unsigned long long merged[8];
    warp_top8(k8, merged);
    if (lane == 0)
#pragma unroll
      for (int r = 0; r < 8; ++r) dst[r] = merged[r];
  }
  bsync();
}

// 16 bytes of a peer CTA's shared memory.
__device__ __forceinline__ uint4 ld_peer_v4(const void* local_addr, uint32_t rank) {
  const uint32_t a = map_to_rank(smem_u32(local_addr), rank);
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a)
               : "memory");
  return v;
}

// The top 8 of the C lists of 8 keys held at `list` in the CTAs of the cluster (one warp; the
// result on every lane).
__device__ void cluster_top8(const unsigned long long* list, uint32_t C,
                             unsigned long long (&out)[8]) {
  const int lane = threadIdx.x & 31;
  const bool have = lane < static_cast<int>(C);
  unsigned long long l[8];
#pragma unroll
  for (int r = 0; r < 8; r += 2) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (have) v = ld_peer_v4(list + r, static_cast<uint32_t>(lane));
    l[r] = (static_cast<unsigned long long>(v.y) << 32) | v.x;
    l[r + 1] = (static_cast<unsigned long long>(v.w) << 32) | v.z;
  }
  warp_top8(l, out);
}

// Warp 0 merges the C partials of the cluster (read from every CTA's shared memory, in rank
// order, so every CTA reaches the same values) into S.Mt .. S.S_z; with a bias set, also the
// draft row's top 8 and the Saguaro renormalisation N.
__device__ void row_combine(const RowParams& P, RowShared& S, uint32_t C, bool two, bool bias) {
  const int lane = threadIdx.x & 31;
  const float c = P.c;
  const bool have = lane < static_cast<int>(C);
  float mt = -INFINITY, st = 0.f, md = -INFINITY, sd = 0.f;
  if (have) {
    const uint4 a = ld_peer_v4(&S.part.m_t, static_cast<uint32_t>(lane));
    mt = __uint_as_float(a.x);
    st = __uint_as_float(a.y);
    md = __uint_as_float(a.z);
    sd = __uint_as_float(a.w);
  }
  const float Mt = warp_max_nan(mt), Md = warp_max_nan(md);
  const float tt = (two && have && mt > -INFINITY && !row_bad(Mt)) ? st * exp2f((mt - Mt) * c) : 0.f;
  const float td = (have && md > -INFINITY && !row_bad(Md)) ? sd * exp2f((md - Md) * c) : 0.f;
  const float St = warp_sum(tt), Sd = warp_sum(td);
  unsigned long long mtop[8];
  if (bias) cluster_top8(S.part.top, C, mtop);
  if (lane == 0) {
    S.Mt = Mt;
    S.St = St;
    S.Md = Md;
    S.Sd = Sd;
    S.bad = (two && row_bad(Mt)) || row_bad(Md);
    float N = 1.f;
    int nS = 0;
    if (bias && !S.bad) {  // Saguaro bias set: the bias_k most likely draft ids
      float sq = 0.f;
      for (int j = 0; j < P.bias_k; ++j) {
        if (mtop[j] == 0ull) break;
        const float z = key_value(mtop[j]);
        sq += exp2f((z - Md) * c) / Sd;
        S.S_z[nS] = z;
        S.S_ids[nS++] = key_id(mtop[j]);
      }
      N = fmaf(-(1.f - P.beta), sq, 1.f);
    }
    S.N = N;
    S.nS = nS;
  }
  __syncwarp();
}

// ------------------------------------------------------------------------------------------
// sampling: one cluster per row
// ------------------------------------------------------------------------------------------
template <typename T, bool BIAS>
__global__ void __launch_bounds__(RT, 4) sample_kernel(const RowParams P) {
  extern __shared__ __align__(16) float vmass[];  // one mass per 8-element vector of the slice
  __shared__ RowShared S;
  constexpr int NB = Raw8<T>::kBatch;
  const int tid = threadIdx.x;
  const uint32_t rank = cluster_ctarank();
  const uint32_t C = cluster_nctarank();
  const int cid = static_cast<int>(cluster_id_x());
  const float c = P.c;
  const int v0 = static_cast<int>(rank) * P.slice;
  const int nv = max(0, min(P.V - v0, P.slice));
  const int nvec = (nv + 7) >> 3;
  const bool vec = P.use_vec != 0;
  const T* row = static_cast<const T*>(P.dft) + static_cast<long long>(cid) * P.d_stride + v0;

  // ---- the one pass: running max, per-vector masses, the bias set's candidates ----
  float m = -INFINITY, mc = -INFINITY, s = 0.f;
  WarpTop8 top;
  top.init();
  int cnt = 0;  // vectors this thread has stored (at tid + i * RT)
  // (the loop runs to the warp's last vector so that every lane takes part in the votes)
  const int nvec_w = nvec + ((RT - (nvec % RT)) % RT);
  for (int g0 = tid; g0 < nvec_w; g0 += RT * NB) {
    Raw8<T> r[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j)
      if (g0 + j * RT < nvec) r[j].load(row, 8 * (g0 + j * RT), nv, vec);
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const int g = g0 + j * RT;
      if (__all_sync(FULL, g >= nvec)) break;
      float z[8];
      if (g < nvec) r[j].get(z);
      else
#pragma unroll
        for (int k = 0; k < 8; ++k) z[k] = -INFINITY;
      if (BIAS)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          top.offer(8 * g + k < nv, z[k], static_cast<uint32_t>(v0 + 8 * g + k));
      if (g >= nvec) continue;
      const float mn = max_nan(m, max8(z));
      if (mn != m) {  // the running max rises: rescale what is stored
        const float mcn = __fmul_rn(mn, c);
        const float f = exp2f(mc - mcn);
        s *= f;
        for (int i = 0; i < cnt; ++i) vmass[tid + i * RT] *= f;
        m = mn;
        mc = mcn;
      }
      float vs = 0.f;
      if (m > -INFINITY) {
#pragma unroll
        for (int k = 0; k < 8; ++k) vs += ex2_fast(fmaf(z[k], c, -mc));
      }
      vmass[g] = vs;
      s += vs;
      ++cnt;
    }
  }

  // ---- the CTA's partial; cluster combine ----
  const float M = row_block_max2(-INFINITY, m, S).y;
  const float Mc = __fmul_rn(M, c);
  const float pd = (m > -INFINITY && !row_bad(M)) ? s * exp2f(mc - Mc) : 0.f;
  float sd = row_block_sum2(0.f, pd, S).y;
  if (!row_bad(M)) sd *= fmaf(-fmaf(M, c, -Mc), kLn2r, 1.f);
  if (BIAS) row_block_top8w(top, S, S.part.top);
  if (tid == 0) {
    S.part.m_t = 0.f;
    S.part.s_t = 0.f;
    S.part.m_d = M;
    S.part.s_d = sd;
    S.token = -1;
  }
  cluster_sync();
  if (tid < 32) row_combine(P, S, C, false, BIAS);
  bsync();
  if (S.bad) {
    if (rank == 0 && tid == 0) {
      P.out_tok[cid] = -1;
      P.out_conf[cid] = NAN;
      if (P.out_exit) P.out_exit[cid] = -1;
    }
    cluster_sync();  // peers may still be reading this CTA's partial
    return;
  }

  // ---- masses relative to the row maximum, bias corrections, fixed-point slice mass ----
  const float Mdc = __fmul_rn(S.Md, c);
  const float F = m > -INFINITY ? exp2f(mc - Mdc) : 0.f;
  const float bm1 = P.beta - 1.f;
  const int nS = BIAS ? S.nS : 0;
  unsigned long long acc = 0;
  for (int g = tid; g < nvec; g += RT) {
    float v = vmass[g] * F;
    for (int j = 0; j < nS; ++j)
      if (((S.S_ids[j] - v0) >> 3) == g)
        v = fmaxf(fmaf(bm1, ex2_fast(fmaf(S.S_z[j], c, -Mdc)), v), 0.f);
    vmass[g] = v;
    acc += qfix(v);
  }
  const unsigned long long Wc = row_block_sum_u64(acc, S);
  if (tid == 0) S.part_w[0] = Wc;
  cluster_sync();

  // ---- which CTA holds the draw (every CTA reaches the same answer) ----
  if (tid < 32) {
    const int lane = tid;
    unsigned long long w = 0ull;
    if (lane < static_cast<int>(C)) {
      const uint4 v = ld_peer_v4(S.part_w, static_cast<uint32_t>(lane));
      w = (static_cast<unsigned long long>(v.y) << 32) | v.x;
    }
    const unsigned long long inc = warp_inclusive_u64(w);
    const unsigned long long Wt = __shfl_sync(FULL, inc, 31);
    const float u = P.uni[cid];
    const unsigned long long t = scale_floor(u, Wt);
    const unsigned hit = __ballot_sync(FULL, lane < static_cast<int>(C) && t < inc);
    const int cs = (u >= 0.f && u < 1.f && hit) ? __ffs(hit) - 1 : -1;
    if (lane == 0) S.cstar = cs;
    if (cs >= 0 && lane == cs) S.t_loc = t - (inc - w);
  }
  bsync();
  cluster_arrive();  // no more reads of the peers' shared memory from here on

  if (S.cstar == static_cast<int>(rank)) {
    // contiguous runs of vectors per thread, so the prefix follows ascending ids
    const int lo = static_cast<int>((static_cast<long long>(tid) * nvec) / RT);
    const int hi = static_cast<int>((static_cast<long long>(tid + 1) * nvec) / RT);
    unsigned long long csum = 0;
    for (int g = lo; g < hi; ++g) csum += qfix(vmass[g]);
    unsigned long long pre = row_block_exclusive_u64(csum, S);
    const unsigned long long tl = S.t_loc;
    if (pre <= tl && tl < pre + csum) {
      for (int g = lo; g < hi; ++g) {
        const unsigned long long q = qfix(vmass[g]);
        if (pre + q > tl) {
          Raw8<T> rv;
          rv.load(row, 8 * g, nv, vec);
          float z[8];
          rv.get(z);
          const int e0 = v0 + 8 * g;
          float sacc = 0.f;
          int pick = 7;
          for (int k = 0; k < 8; ++k) {
            float f = 1.f;
            for (int j = 0; j < nS; ++j) f = (S.S_ids[j] == e0 + k) ? P.beta : f;
            const float wk = (8 * g + k < nv) ? f * ex2_fast(fmaf(z[k], c, -Mdc)) : 0.f;
            sacc = k ? __fadd_rn(sacc, wk) : wk;
            if (pre + qfix(sacc) > tl) {
              pick = k;
              break;
            }
          }
          S.token = e0 + pick;
          break;
        }
        pre += q;
      }
    }
    bsync();
    if (tid == 0) P.out_tok[cid] = S.token;
  }
  if (rank == 0 && tid == 0) {
    if (S.cstar < 0) P.out_tok[cid] = -1;  // uniform outside [0, 1)
    const float conf = 1.f / S.Sd;        // the unbiased softmax's largest probability
    P.out_conf[cid] = conf;
    if (P.out_exit) P.out_exit[cid] = conf < P.tau ? 1 : 0;
  }
  cluster_wait();  // no CTA leaves while a peer may still read its shared memory
}

// ------------------------------------------------------------------------------------------
// exact-residual top-F: one cluster per (sequence, position) pair
// ------------------------------------------------------------------------------------------
template <typename T, bool BIAS>
__global__ void __launch_bounds__(RT, 3) resid_kernel(const RowParams P) {
  __shared__ RowShared S;
  constexpr int NB = (Raw8<T>::kBatch + 1) / 2;  // two rows per vector index
  const int tid = threadIdx.x;
  const uint32_t rank = cluster_ctarank();
  const uint32_t C = cluster_nctarank();
  const int cid = static_cast<int>(cluster_id_x());
  const float c = P.c;
  const int b = cid / P.K, i = cid % P.K;
  const int L = P.lens ? P.lens[b] : P.K;
  int32_t* out = P.out_r2 + static_cast<long long>(cid) * P.fmax;
  if (L < 1 || L > P.K || i >= L) {  // no residual at this position (uniform over the cluster)
    if (rank == 0 && tid < P.fmax) out[tid] = -1;
    return;
  }
  const int v0 = static_cast<int>(rank) * P.slice;
  const int nv = max(0, min(P.V - v0, P.slice));
  const int nvec = (nv + 7) >> 3;
  const bool vec = P.use_vec != 0;
  const T* zt = static_cast<const T*>(P.tgt) +
                (static_cast<long long>(b) * (P.K + 1) + i) * P.t_stride + v0;
  const T* zd = static_cast<const T*>(P.dft) +
                (static_cast<long long>(b) * P.K + i) * P.d_stride + v0;

  // ---- pass 1: maxima and sums of both rows; the draft row's top 8 for the bias set ----
  RowAcc at, ad;
  at.init();
  ad.init();
  WarpTop8 top;
  top.init();
  // (the loops run to the warp's last vector so that every lane takes part in the votes)
  const int nvec_w = nvec + ((RT - (nvec % RT)) % RT);
  for (int g0 = tid; g0 < nvec_w; g0 += RT * NB) {
    Raw8<T> rt[NB], rd[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j)
      if (g0 + j * RT < nvec) {
        rd[j].load(zd, 8 * (g0 + j * RT), nv, vec);
        rt[j].load(zt, 8 * (g0 + j * RT), nv, vec);
      }
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const int g = g0 + j * RT;
      if (__all_sync(FULL, g >= nvec)) break;
      float z[8];
      if (g < nvec) rd[j].get(z);
      else
#pragma unroll
        for (int k = 0; k < 8; ++k) z[k] = -INFINITY;
      if (BIAS)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          top.offer(8 * g + k < nv, z[k], static_cast<uint32_t>(v0 + 8 * g + k));
      if (g >= nvec) continue;
      ad.rescale(max8(z), c);
      if (ad.m > -INFINITY) ad.sum8(z, c);
      rt[j].get(z);
      at.rescale(max8(z), c);
      if (at.m > -INFINITY) at.sum8(z, c);
    }
  }
  const float2 mm = row_block_max2(at.m, ad.m, S);
  const float mct = __fmul_rn(mm.x, c), mcd = __fmul_rn(mm.y, c);
  const float pt = (at.m > -INFINITY && !row_bad(mm.x)) ? at.total() * exp2f(at.mc - mct) : 0.f;
  const float pd = (ad.m > -INFINITY && !row_bad(mm.y)) ? ad.total() * exp2f(ad.mc - mcd) : 0.f;
  float2 ss = row_block_sum2(pt, pd, S);
  if (!row_bad(mm.x)) ss.x *= fmaf(-fmaf(mm.x, c, -mct), kLn2r, 1.f);
  if (!row_bad(mm.y)) ss.y *= fmaf(-fmaf(mm.y, c, -mcd), kLn2r, 1.f);
  if (BIAS) row_block_top8w(top, S, S.part.top);
  if (tid == 0) {
    S.part.m_t = mm.x;
    S.part.s_t = ss.x;
    S.part.m_d = mm.y;
    S.part.s_d = ss.y;
  }
  cluster_sync();
  if (tid < 32) row_combine(P, S, C, true, BIAS);
  bsync();
  if (S.bad) {
    if (rank == 0 && tid < P.fmax) out[tid] = -1;
    cluster_sync();  // peers may still be reading this CTA's partial
    return;
  }

  // ---- pass 2: residual weights relative to p's scale, max(e_t - rho_v e_d, 0) ----
  const float Mtc = __fmul_rn(S.Mt, c), Mdc = __fmul_rn(S.Md, c);
  const float ft = fmaf(-fmaf(S.Mt, c, -Mtc), kLn2r, 1.f);
  const float fd = fmaf(-fmaf(S.Md, c, -Mdc), kLn2r, 1.f);
  const float rho = (fd * S.St) / (ft * (S.Sd * S.N));
  const float rhoS = rho * P.beta;
  const int nS = BIAS ? S.nS : 0;
  WarpTop8 rtop;
  rtop.init();
  float thrl = -INFINITY;  // log2 of the warp's 8th best residual, less a margin for rounding
  for (int g0 = tid; g0 < nvec_w; g0 += RT * NB) {
    Raw8<T> rt[NB], rd[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j)
      if (g0 + j * RT < nvec) {
        rt[j].load(zt, 8 * (g0 + j * RT), nv, vec);
        rd[j].load(zd, 8 * (g0 + j * RT), nv, vec);
      }
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const int g = g0 + j * RT;
      if (__all_sync(FULL, g >= nvec)) break;
      float a[8], d[8];
      if (g < nvec) {
        rt[j].get(a);
        rd[j].get(d);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) a[k] = d[k] = -INFINITY;
      }
      const int e0 = v0 + 8 * g;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        // e_t, hence the residual, below the warp's 8th best: no exponentials needed
        const float lt = fmaf(a[k], c, -Mtc);
        const bool pass = lt >= thrl && 8 * g + k < nv;
        if (!__any_sync(FULL, pass)) continue;
        float w = 0.f;
        if (pass) {
          float r = rho;
          for (int j2 = 0; j2 < nS; ++j2) r = (S.S_ids[j2] == e0 + k) ? rhoS : r;
          w = fmaxf(fmaf(-r, ex2_fast(fmaf(d[k], c, -Mdc)), ex2_fast(lt)), 0.f);
        }
        if (rtop.offer(pass && w > 0.f, w, static_cast<uint32_t>(e0 + k)))
          thrl = __log2f(rtop.thr) - 1e-3f;
      }
    }
  }
  row_block_top8w(rtop, S, S.part_r);
  cluster_sync();
  if (rank == 0 && tid < 32) {
    unsigned long long top[8];
    cluster_top8(S.part_r, C, top);
    if (tid < P.fmax) {
      const int F = P.fan[i];
      out[tid] = (tid < F && tid < 8 && top[tid] != 0ull) ? key_id(top[tid]) : -1;
    }
  }
  cluster_sync();  // no CTA leaves while rank 0 may still read its shared memory
}

// Cache-hit flags: 1 if the token the verify step drew at a rejected position is among the
// top-F draft ids prepared for that outcome, 0 if not, -1 when every draft was accepted or the
// sequence is invalid.
__global__ void hit_kernel(const RowParams P, const int32_t* acc, const int32_t* tok,
                           const int32_t* r1) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= P.B) return;
  const int a = acc[b];
  const int L = P.lens ? P.lens[b] : P.K;
  int hit = -1;
  if (a >= 0 && L >= 1 && L <= P.K && a < L) {
    const int x = tok[static_cast<long long>(b) * (P.K + 1) + a];
    const int F = min(P.fan[a], P.fmax);
    hit = 0;
    for (int f = 0; f < F; ++f)
      if (r1[(static_cast<long long>(b) * P.K + a) * P.fmax + f] == x) hit = 1;
  }
  P.out_hit[b] = hit;
}

template <int MODE, typename T, bool BIAS>
const void* row_fn() {
  if constexpr (MODE == MODE_SAMPLE)
    return reinterpret_cast<const void*>(&sample_kernel<T, BIAS>);
  else
    return reinterpret_cast<const void*>(&resid_kernel<T, BIAS>);
}

template <int MODE>
const void* pick_fn(int dtype, bool bias) {
  if (dtype == 1) return bias ? row_fn<MODE, uint16_t, true>() : row_fn<MODE, uint16_t, false>();
  return bias ? row_fn<MODE, float, true>() : row_fn<MODE, float, false>();
}

}  // namespace

cudaError_t launch_rows(const RowParams& P, int mode, int dtype, int nclusters, int C,
                        const int32_t* acc, const int32_t* tok, const int32_t* r1,
                        cudaStream_t stream) {
  const bool bias = P.bias_k > 0 && P.beta < 1.f;
  const void* fn = mode == MODE_SAMPLE ? pick_fn<MODE_SAMPLE>(dtype, bias)
                                       : pick_fn<MODE_RESID>(dtype, bias);
  const size_t smem = mode == MODE_SAMPLE ? static_cast<size_t>((P.slice + 7) / 8) * 4 : 0;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (C > 8) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  if (nclusters > 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nclusters) * static_cast<unsigned>(C));
    cfg.blockDim = dim3(RT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {const_cast<RowParams*>(&P)};
    e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) return e;
  }
  if (mode == MODE_RESID && P.out_hit && P.B > 0) {
    hit_kernel<<<(P.B + 127) / 128, 128, 0, stream>>>(P, acc, tok, r1);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace sv

// The verify step taken from hidden states: the LM head's GEMM reduces every row to the numbers
// the accept test needs, and the rows of the decided position are recomputed on the tensor cores
// only for the draw, so no logit row is written to HBM (Kangaroo guide, "Exit 1" and section 3;
// LayerSkip guide, "Verification Phase"; SSD summary, "Method").
//
// One call, in stream order:
//  1. hv_scan / hv_gather: the rows each sequence has (target 0..L_b, draft 0..L_b-1) packed
//     into one bf16 matrix, with the draft id each row is scored at;
//  2. the head GEMM with its statistics epilogue and the combine: per row the maximum, the sum
//     of 2^(z c - fl(m c)), the logit at the draft id and the lowest id of the maximum (with a
//     Saguaro bias set or top-F ids, also each row's 8 largest logits per vocabulary range);
//  3. hv_decide: per sequence the accept tests u_i < p_i(x_i) / q'_i(x_i) in order (greedy:
//     x_i == argmax), the first rejection a_b, the accepted ids, the top-F ids; it copies the
//     hidden states of position a_b (target, and draft unless every draft was accepted) into
//     pair slots;
//  4. the head GEMM again over those pairs with the residual epilogue: per sequence and per 16
//     ids the masses of max(p - q, 0) (or of p for the bonus draw) in 2^-44 units;
//  5. hv_pick: per sequence the inverse CDF over ascending ids: the 16-id block that holds
//     floor(u W) from the masses, then the id inside it from the 16 logits recomputed with the
//     same arithmetic.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "sv_hverify.h"
#include "sv_lmhead.h"
#include "sv_math.cuh"
#include "sv_ptx.cuh"

namespace sv {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kPickThreads = 256;

constexpr int kMaxRanges = 64;  // vocabulary ranges of the statistics GEMM when the top 8 are kept

struct HvLayout {
  int Rmax, npairs, nsplit, tps, ntiles, nh, rsplit, rtps;
  size_t off, count, ids, rows, part, keys, A, Ad, pairs, seqa, mass, massp, total;
};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

HvLayout layout(const HvProblem& p, int sms) {
  HvLayout L;
  L.Rmax = p.B * ((p.K + 1) + (p.greedy ? 0 : p.K));
  L.npairs = p.greedy ? 0 : (p.B + 63) / 64 * 64;
  head_split(L.Rmax, p.V, sms, &L.nsplit, &L.tps, &L.ntiles, hv_top8(p) ? kMaxRanges : 0);
  L.nh = L.ntiles * kHeadHalves;
  int nt2 = 0;
  head_split(std::max(1, 2 * L.npairs), p.V, sms, &L.rsplit, &L.rtps, &nt2);
  size_t o = 0;
  L.off = o;   o += up256(sizeof(int) * (p.B + 1));
  L.count = o; o += 256;
  L.ids = o;   o += up256(sizeof(int32_t) * L.Rmax);
  L.rows = o;  o += up256(sizeof(HeadRow) * L.Rmax);
  L.part = o;  o += up256(head_part_bytes(L.Rmax, L.nsplit));
  L.keys = o;  o += hv_top8(p) ? up256(static_cast<size_t>(L.Rmax) * L.nsplit * 64) : 0;
  L.A = o;     o += up256(static_cast<size_t>(L.Rmax) * p.d * 2);
  L.Ad = o;    o += up256(static_cast<size_t>(2 * L.npairs) * p.d * 2);
  L.pairs = o; o += up256(sizeof(HeadPair) * L.npairs);
  L.seqa = o;  o += up256(sizeof(int) * p.B);
  L.mass = o;  o += up256(sizeof(unsigned long long) * L.npairs * L.nh);
  L.massp = o; o += up256(sizeof(unsigned long long) * L.npairs * L.nh);
  L.total = o;
  return L;
}

__device__ __forceinline__ int rows_of(int L, int K, int greedy) {
  return (L >= 1 && L <= K) ? (L + 1) + (greedy ? 0 : L) : 0;
}

// Exclusive offsets of the packed rows of every sequence (one CTA, chunks of 1024 sequences).
__global__ void __launch_bounds__(kScanThreads) hv_scan(int B, int K, int greedy,
                                                        const int32_t* lens, int* off, int* count) {
  __shared__ int wsum[kScanThreads / 32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < B; base += kScanThreads) {
    const int b = base + tid;
    const int n = b < B ? rows_of(lens[b], K, greedy) : 0;
    int v = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int t = wsum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += y;
      }
      wsum[lane] = t;  // inclusive over warps
    }
    __syncthreads();
    const int before = carry + (warp ? wsum[warp - 1] : 0) + (v - n);
    if (b < B) off[b] = before;
    __syncthreads();
    if (tid == 0) carry += wsum[kScanThreads / 32 - 1];
    __syncthreads();
  }
  if (tid == 0) {
    off[B] = carry;
    *count = carry;
  }
}

// Pack row blockIdx.y of sequence blockIdx.x (target 0..L, then, stochastic, draft 0..L-1) with
// the id it is scored at (x_i; -1 for target row L). Row slots past the sequence's rows idle.
__global__ void __launch_bounds__(128) hv_gather(const HvProblem p, const int* off, uint16_t* A,
                                                 int32_t* ids) {
  const int b = blockIdx.x, r = blockIdx.y;
  const int L = p.lens[b];
  if (r >= rows_of(L, p.K, p.greedy)) return;
  const int o = off[b];
  const uint16_t* src = r <= L ? p.ht + (static_cast<long long>(b) * (p.K + 1) + r) * p.hts
                               : p.hd + (static_cast<long long>(b) * p.K + (r - L - 1)) * p.hds;
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(A + static_cast<long long>(o + r) * p.d);
  for (int v = threadIdx.x; v < p.d / 8; v += blockDim.x) d4[v] = s4[v];
  if (threadIdx.x == 0) {
    const int i = r <= L ? r : r - L - 1;
    ids[o + r] = (r <= L && i == L) ? -1 : p.x[static_cast<long long>(b) * p.K + i];
  }
}

// The 8 largest keys of a row from its vocabulary ranges' lists (each descending; list r at
// keys + (r * Rmax + row) * 8, nsplit <= 64): lane q < 8 returns the q-th. Warp-wide.
__device__ __forceinline__ unsigned long long merge_ranges(const unsigned long long* keys,
                                                          int nsplit, int Rmax, int row) {
  const int lane = threadIdx.x & 31;
  unsigned long long a[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) a[q] = 0ull;
  float thr = -INFINITY;
  for (int r = lane; r < nsplit; r += 32) {  // the lane's lists into one
    const unsigned long long* kr = keys + (static_cast<long long>(r) * Rmax + row) * 8;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const unsigned long long k = kr[q];
      if (k != 0ull) top8_insert(a, thr, key_value(k), static_cast<uint32_t>(key_id(k)));
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

// Decisions of sequence blockIdx.x, then the copy of the decided position's hidden states into
// its pair slot. Blocks past B only mark their pair slot as unused. With a bias set or top-F ids
// the draft rows' 8 largest logits are merged from the ranges' lists first (one warp per row);
// the bias set is the first bias_k of them, q' = q f / N with f = beta on the set and
// N = 1 - (1 - beta) q(set), so the accept ratio gains N / f and the residual's draft weight is
// rho = S_t / (S_d N) off the set and rho beta on it (Saguaro summary, "Method"). With top-F ids
// every draft row below L is needed.
__global__ void __launch_bounds__(128) hv_decide(const HvProblem p, float c, const int* off,
                                                 const uint16_t* A, const HeadRow* rows,
                                                 const unsigned long long* keys, int nsplit,
                                                 int Rmax, uint16_t* Ad, HeadPair* pairs,
                                                 int* seq_a) {
  __shared__ int s_src_t, s_src_d;  // packed rows to copy (-1: none / zeros)
  __shared__ unsigned long long s_key[8][8];
  __shared__ float s_N[8], s_f[8];
  __shared__ int s_nS[8], s_ok;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.K;
  const bool top8 = hv_top8(p);
  const bool bias = top8 && p.bias_k > 0 && p.beta < 1.f;
  const int L = b < p.B ? p.lens[b] : 0;
  const bool lok = b < p.B && L >= 1 && L <= K;
  const int o = lok ? off[b] : 0;
  if (top8 && lok) {
    for (int i = warp; i < L; i += blockDim.x >> 5) {
      const unsigned long long k = merge_ranges(keys, nsplit, Rmax, o + L + 1 + i);
      if (lane < 8) s_key[i][lane] = k;
    }
    __syncthreads();
    if (bias) {  // per draft row: q(set) summed in key order, N, and whether x_i is in the set
      for (int i = warp; i < L; i += blockDim.x >> 5) {
        const HeadRow rd = rows[o + L + 1 + i];
        const unsigned long long kj = lane < 8 ? s_key[i][lane] : 0ull;
        const bool in = lane < p.bias_k && kj != 0ull;
        const float term = in ? exp2f(fmaf(key_value(kj), c, -rd.mc)) / rd.sum : 0.f;
        const unsigned hit =
            __ballot_sync(0xffffffffu, in && key_id(kj) == p.x[static_cast<long long>(b) * K + i]);
        const int n = __popc(__ballot_sync(0xffffffffu, in));
        float sq = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float tj = __shfl_sync(0xffffffffu, term, j);
          if (j < n) sq += tj;
        }
        if (lane == 0) {
          s_N[i] = fmaf(-(1.f - p.beta), sq, 1.f);
          s_f[i] = hit ? p.beta : 1.f;
          s_nS[i] = n;
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    s_src_t = -1;
    s_src_d = -1;
    s_ok = 0;
    HeadPair pp;
    pp.mc_t = pp.mc_d = pp.rho = pp.rho_s = 0.f;
    pp.skip = 1;
    pp.nS = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) pp.ids[j] = -1;
    if (b < p.B) {
      const int32_t* x = p.x + static_cast<long long>(b) * K;
      const float* u = p.uni ? p.uni + static_cast<long long>(b) * (K + 1) : nullptr;
      int32_t* tok = p.out_tok + static_cast<long long>(b) * (K + 1);
      bool ok = lok;
      for (int i = 0; ok && i < L; ++i) ok = x[i] >= 0 && x[i] < p.V;
      if (ok && !p.greedy) {
        for (int i = 0; ok && i < L; ++i) ok = u[i] >= 0.f && u[i] < 1.f;
        ok = ok && u[K] >= 0.f && u[K] < 1.f;
      }
      for (int i = 0; ok && p.fmax > 0 && i < L; ++i) ok = !row_bad(rows[o + L + 1 + i].max);
      int a = -1, last = -1, draw = 0;
      if (ok) {
        if (p.greedy) {
          for (int i = 0; i <= L; ++i) {
            const HeadRow rt = rows[o + i];
            if (row_bad(rt.max)) {
              ok = false;
              break;
            }
            if (i < L && x[i] == rt.arg) continue;
            a = i;
            last = rt.arg;
            break;
          }
        } else {
          a = L;
          for (int i = 0; i < L; ++i) {
            const HeadRow rt = rows[o + i], rd = rows[o + L + 1 + i];
            if (row_bad(rt.max) || row_bad(rd.max)) {
              ok = false;
              break;
            }
            const float N = bias ? s_N[i] : 1.f, f = bias ? s_f[i] : 1.f;
            // p(x) / q'(x) = 2^(z_t c - mc_t) S_d N / (2^(z_d c - mc_d) S_t f)
            const float lr = fmaf(rt.zx, c, -rt.mc) - fmaf(rd.zx, c, -rd.mc);
            const float ratio = exp2f(lr) * (rd.sum / rt.sum) * (N / f);
            if (u[i] < ratio) continue;
            a = i;
            pp.mc_t = rt.mc;
            pp.mc_d = rd.mc;
            pp.rho = rt.sum / (rd.sum * N);
            pp.rho_s = pp.rho * p.beta;
            if (bias) {
              pp.nS = s_nS[i];
#pragma unroll
              for (int j = 0; j < 8; ++j) pp.ids[j] = j < pp.nS ? key_id(s_key[i][j]) : -1;
            }
            break;
          }
          if (ok && a == L) {
            const HeadRow rt = rows[o + L];
            if (row_bad(rt.max)) ok = false;
            pp.mc_t = rt.mc;
            pp.mc_d = 0.f;
            pp.rho = 0.f;
          }
          if (ok) {
            pp.skip = 0;
            draw = 1;
            s_src_t = o + a;
            s_src_d = a < L ? o + L + 1 + a : -1;
          }
        }
      }
      if (!ok) {
        a = -1;
        draw = 0;
        pp.skip = 1;
        pp.nS = 0;
        s_src_t = -1;
      }
      s_ok = ok ? 1 : 0;
      p.out_acc[b] = a;
      for (int i = 0; i <= K; ++i)
        tok[i] = (ok && i < a) ? x[i] : ((ok && i == a && p.greedy) ? last : -1);
      seq_a[b] = draw ? a : -1;
    }
    if (!p.greedy) pairs[b] = pp;
  }
  __syncthreads();
  if (p.fmax > 0 && b < p.B) {  // the first F_i draft ids of rows below L; -1 elsewhere
    int32_t* tf = p.out_topf + static_cast<long long>(b) * K * p.fmax;
    const bool ok = s_ok != 0;
    for (int e = tid; e < K * p.fmax; e += blockDim.x) {
      const int i = e / p.fmax, f = e - i * p.fmax;
      const unsigned long long k = (ok && i < L && f < p.fan[i] && f < 8) ? s_key[i][f] : 0ull;
      tf[e] = k ? key_id(k) : -1;
    }
  }
  if (p.greedy || s_src_t < 0) return;
  const int nvec = p.d / 8;
  uint4* dt = reinterpret_cast<uint4*>(Ad + static_cast<long long>(head_pair_row(b, 0)) * p.d);
  uint4* dd = reinterpret_cast<uint4*>(Ad + static_cast<long long>(head_pair_row(b, 1)) * p.d);
  const uint4* st = reinterpret_cast<const uint4*>(A + static_cast<long long>(s_src_t) * p.d);
  const uint4* sd = s_src_d >= 0
                        ? reinterpret_cast<const uint4*>(A + static_cast<long long>(s_src_d) * p.d)
                        : nullptr;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    dt[v] = st[v];
    dd[v] = sd ? sd[v] : make_uint4(0u, 0u, 0u, 0u);
  }
}

// Block-wide sum and exclusive prefix of one u64 per thread (kPickThreads threads).
__device__ __forceinline__ unsigned long long block_scan_u64(unsigned long long v,
                                                             unsigned long long* total,
                                                             unsigned long long* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  unsigned long long before = 0, all = 0;
  for (int w = 0; w < kPickThreads / 32; ++w) {
    if (w < warp) before += sh[w];
    all += sh[w];
  }
  __syncthreads();
  *total = all;
  return before + inc - v;
}

// One logit recomputed on the CUDA cores: a warp's dot product of a hidden row and a head row.
__device__ __forceinline__ float warp_dot(const uint16_t* h, const uint16_t* w, int d) {
  float acc = 0.f;
  const int nvec = d / 8;
  for (int v = threadIdx.x & 31; v < nvec; v += 32) {
    const uint4 a = reinterpret_cast<const uint4*>(h)[v];
    const uint4 b = reinterpret_cast<const uint4*>(w)[v];
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc = fmaf(__uint_as_float(av[k] << 16), __uint_as_float(bv[k] << 16), acc);
      acc = fmaf(__uint_as_float(av[k] & 0xFFFF0000u), __uint_as_float(bv[k] & 0xFFFF0000u), acc);
    }
  }
  return warp_sum(acc);
}

// The draw of sequence blockIdx.x: the 16-id block holding t = floor(u W) from the masses, then
// the id inside it.
__global__ void __launch_bounds__(kPickThreads) hv_pick(const HvProblem p, float c, int nh,
                                                        const HeadPair* pairs, const int* seq_a,
                                                        const uint16_t* Ad,
                                                        const unsigned long long* mass_r,
                                                        const unsigned long long* mass_p) {
  __shared__ unsigned long long sh[kPickThreads / 32];
  __shared__ int s_h;
  __shared__ unsigned long long s_t;
  __shared__ float zt[16], zd[16];
  const int b = blockIdx.x;
  const int a = seq_a[b];
  if (a < 0) return;
  const HeadPair pp = pairs[b];
  const int tid = threadIdx.x;
  const int run = (nh + kPickThreads - 1) / kPickThreads;
  const int h0 = min(nh, tid * run), h1 = min(nh, h0 + run);
  const unsigned long long* mr = mass_r + static_cast<long long>(b) * nh;
  unsigned long long loc = 0, W = 0;
  for (int h = h0; h < h1; ++h) loc += mr[h];
  unsigned long long before = block_scan_u64(loc, &W, sh);
  const bool use_p = W == 0;  // no residual mass left (rounding): draw from p
  if (use_p) {
    mr = mass_p + static_cast<long long>(b) * nh;
    loc = 0;
    for (int h = h0; h < h1; ++h) loc += mr[h];
    before = block_scan_u64(loc, &W, sh);
  }
  if (tid == 0) {
    s_h = -1;
    s_t = 0;
  }
  __syncthreads();
  const unsigned long long t = scale_floor(p.uni[static_cast<long long>(b) * (p.K + 1) + p.K], W);
  if (W > 0 && t >= before && t < before + loc) {
    unsigned long long cum = before;
    for (int h = h0; h < h1; ++h) {
      if (t < cum + mr[h]) {
        s_h = h;
        s_t = t - cum;
        break;
      }
      cum += mr[h];
    }
  }
  __syncthreads();
  const int h = s_h;
  int32_t* out = p.out_tok + static_cast<long long>(b) * (p.K + 1) + a;
  if (h < 0) {  // W == 0 for p as well: cannot happen for a finite row
    if (tid == 0) *out = -1;
    return;
  }
  const int v0 = h * 16;
  const int warp = tid >> 5;
  const uint16_t* rt = Ad + static_cast<long long>(head_pair_row(b, 0)) * p.d;
  const uint16_t* rd = Ad + static_cast<long long>(head_pair_row(b, 1)) * p.d;
  for (int j = warp; j < 16; j += kPickThreads / 32) {
    const int v = min(v0 + j, p.V - 1);
    const uint16_t* wr = p.W + static_cast<long long>(v) * p.ws;
    const float a1 = warp_dot(rt, wr, p.d);
    const float a2 = use_p ? 0.f : warp_dot(rd, wr, p.d);
    if ((tid & 31) == 0) {
      zt[j] = a1;
      zd[j] = a2;
    }
  }
  __syncthreads();
  if (tid != 0) return;
  // the same arithmetic, in the same order, as the residual epilogue of the head GEMM
  float cs = 0.f;
  int pick = -1, lastpos = -1;
  for (int j = 0; j < 16; ++j) {
    if (v0 + j >= p.V) break;
    const float et = ex2_fast(fmaf(zt[j], c, -pp.mc_t));
    const float ed = ex2_fast(fmaf(zd[j], c, -pp.mc_d));
    float rk = pp.rho;
    for (int k = 0; k < pp.nS; ++k) rk = pp.ids[k] == v0 + j ? pp.rho_s : rk;
    const float w = use_p ? et : fmaxf(fmaf(-rk, ed, et), 0.f);
    cs += w;
    if (w > 0.f) lastpos = j;
    if (qfix(cs) > s_t) {
      pick = j;
      break;
    }
  }
  // the recomputed logits can differ from the tensor cores' in their last bits: then the offset
  // may run past the block, and the last id with weight stands for it
  if (pick < 0) pick = lastpos >= 0 ? lastpos : 0;
  *out = v0 + pick;
}

}  // namespace

size_t hv_workspace_bytes(const HvProblem& p, int sms) { return layout(p, sms).total; }

cudaError_t hv_run(const HvProblem& p, int sms, void* ws, unsigned int* err, cudaStream_t stream) {
  const HvLayout L = layout(p, sms);
  char* w = static_cast<char*>(ws);
  int* off = reinterpret_cast<int*>(w + L.off);
  int* count = reinterpret_cast<int*>(w + L.count);
  int32_t* ids = reinterpret_cast<int32_t*>(w + L.ids);
  HeadRow* rows = reinterpret_cast<HeadRow*>(w + L.rows);
  uint16_t* A = reinterpret_cast<uint16_t*>(w + L.A);
  uint16_t* Ad = reinterpret_cast<uint16_t*>(w + L.Ad);
  HeadPair* pairs = reinterpret_cast<HeadPair*>(w + L.pairs);
  int* seqa = reinterpret_cast<int*>(w + L.seqa);
  unsigned long long* mr = reinterpret_cast<unsigned long long*>(w + L.mass);
  unsigned long long* mp = reinterpret_cast<unsigned long long*>(w + L.massp);
  const float c = static_cast<float>(1.4426950408889634 / static_cast<double>(p.temperature));

  hv_scan<<<1, kScanThreads, 0, stream>>>(p.B, p.K, p.greedy, p.lens, off, count);
  hv_gather<<<dim3(p.B, 2 * p.K + 1), 128, 0, stream>>>(p, off, A, ids);
  HeadParams P;
  memset(&P, 0, sizeof(P));
  P.R = L.Rmax;
  P.d = p.d;
  P.V = p.V;
  P.R_dev = count;
  P.c = c;
  P.inv_t = static_cast<float>(1.0 / static_cast<double>(p.temperature));
  P.ids = ids;
  P.part = reinterpret_cast<float4*>(w + L.part);
  P.nsplit = L.nsplit;
  P.tiles_per_split = L.tps;
  P.ntiles = L.ntiles;
  P.err = err;
  const bool top8 = hv_top8(p);
  unsigned long long* keys = top8 ? reinterpret_cast<unsigned long long*>(w + L.keys) : nullptr;
  P.keys = keys;
  cudaError_t e = launch_head_gemm(top8 ? HEAD_STATS_TOP8 : HEAD_STATS, A, p.d, p.W, p.ws, P,
                                   head_ctas(sms), stream);
  if (e != cudaSuccess) return e;
  e = launch_head_combine(P, nullptr, nullptr, nullptr, nullptr, rows, stream);
  if (e != cudaSuccess) return e;
  hv_decide<<<p.greedy ? p.B : L.npairs, 128, 0, stream>>>(p, c, off, A, rows, keys, L.nsplit,
                                                            L.Rmax, Ad, pairs, seqa);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.greedy) return e;
  HeadParams Q = P;
  Q.R = 2 * L.npairs;
  Q.R_dev = nullptr;
  Q.ids = nullptr;
  Q.part = nullptr;
  Q.keys = nullptr;
  Q.pair = pairs;
  Q.mass = mr;
  Q.mass_p = mp;
  Q.nh = L.nh;
  Q.nsplit = L.rsplit;
  Q.tiles_per_split = L.rtps;
  e = launch_head_gemm(HEAD_RESID, Ad, p.d, p.W, p.ws, Q, head_ctas(sms), stream);
  if (e != cudaSuccess) return e;
  hv_pick<<<p.B, kPickThreads, 0, stream>>>(p, c, L.nh, pairs, seqa, Ad, mr, mp);
  return cudaGetLastError();
}

}  // namespace sv

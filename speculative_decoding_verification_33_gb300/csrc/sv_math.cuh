// Per-element and per-warp arithmetic shared by the verify kernel and the row kernels: element
// access for fp32 / bf16 rows, warp reductions, sort keys for top-8 selection, the running
// (max, sum of exponentials) accumulator, and the fixed-point conversion of the inverse CDF.
#pragma once

#include <math.h>
#include <stdint.h>

#include "sv_ptx.cuh"

namespace sv {

constexpr unsigned FULL = 0xffffffffu;

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
  static __device__ __forceinline__ void ldg8(const float* g, float (&z)[8]) {
    const uint4 a = ldg_nc_v4(g), b = ldg_nc_v4(g + 4);
    z[0] = __uint_as_float(a.x); z[1] = __uint_as_float(a.y);
    z[2] = __uint_as_float(a.z); z[3] = __uint_as_float(a.w);
    z[4] = __uint_as_float(b.x); z[5] = __uint_as_float(b.y);
    z[6] = __uint_as_float(b.z); z[7] = __uint_as_float(b.w);
  }
  static __device__ __forceinline__ float vmax8(const float* s, int g, float (&z)[8]) {
    load8(s, g, z);
    return max_nan(max_nan(max_nan(z[0], z[1]), max_nan(z[2], z[3])),
                   max_nan(max_nan(z[4], z[5]), max_nan(z[6], z[7])));
  }
};

template <>
struct Elt<uint16_t> {
  static __device__ __forceinline__ float val(uint16_t v) {
    return __uint_as_float(static_cast<uint32_t>(v) << 16);
  }
  static __device__ __forceinline__ uint16_t neg_inf() { return 0xFF80u; }
  static __device__ __forceinline__ void unpack(const uint4 v, float (&z)[8]) {
    z[0] = __uint_as_float(v.x << 16); z[1] = __uint_as_float(v.x & 0xFFFF0000u);
    z[2] = __uint_as_float(v.y << 16); z[3] = __uint_as_float(v.y & 0xFFFF0000u);
    z[4] = __uint_as_float(v.z << 16); z[5] = __uint_as_float(v.z & 0xFFFF0000u);
    z[6] = __uint_as_float(v.w << 16); z[7] = __uint_as_float(v.w & 0xFFFF0000u);
  }
  static __device__ __forceinline__ void load8(const uint16_t* s, int g, float (&z)[8]) {
    unpack(reinterpret_cast<const uint4*>(s)[g], z);
  }
  static __device__ __forceinline__ void ldg8(const uint16_t* g, float (&z)[8]) {
    unpack(ldg_nc_v4(g), z);
  }
  static __device__ __forceinline__ float vmax8(const uint16_t* s, int g, float (&z)[8]) {
    const uint4 v = reinterpret_cast<const uint4*>(s)[g];
    const uint32_t m = max_nan_bf16x2(max_nan_bf16x2(v.x, v.y), max_nan_bf16x2(v.z, v.w));
    unpack(v, z);
    return max_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
  }
};

// Eight elements of a global row slice starting at slice offset e0 (elements at or past nv
// read as -inf); vector loads when the row is 16-byte aligned and the vector is whole.
template <typename T>
__device__ __forceinline__ void row8(const T* g, int e0, int nv, bool aligned, float (&z)[8]) {
  if (aligned && e0 + 8 <= nv) {
    Elt<T>::ldg8(g + e0, z);
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) z[k] = (e0 + k < nv) ? Elt<T>::val(g[e0 + k]) : -INFINITY;
  }
}

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

// Order-preserving 32 bits of a float (a larger float gives a larger integer), and back.
__device__ __forceinline__ uint32_t float_to_ord(float v) {
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float ord_to_float(uint32_t m) {
  return __uint_as_float((m & 0x80000000u) ? (m & 0x7FFFFFFFu) : ~m);
}

// Sort key of a logit: larger value first, then lower id (-0 and +0 are one value). 0 means
// "empty".
__device__ __forceinline__ unsigned long long make_key(float z, uint32_t id) {
  const uint32_t b = __float_as_uint(z == 0.f ? 0.f : z);
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

// Integer of 2^-44 units below s (0 <= s < 16): s * 2^44 is exact in float (a power-of-two
// scale, below 2^48), and the conversion truncates it.
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
// per-thread running statistics of one row
// ------------------------------------------------------------------------------------------
// Running max and sum of 2^(z c - m c) of one row, for one thread. The sum is kept in two packed
// fp32 pairs and built with the packed fp32 instructions (one fma for the exponent arguments of
// two elements, one add to accumulate two exponentials).
struct RowAcc {
  float m, mc;      // running max and its product with c (rounded)
  float2 s0, s1;    // four partial sums of 2^(z c - mc)
  __device__ __forceinline__ void init() {
    m = -INFINITY;
    mc = -INFINITY;
    s0 = s1 = make_float2(0.f, 0.f);
  }
  // Raise the running max to include vm (NaN sticks), rescaling what was summed so far.
  __device__ __forceinline__ void rescale(float vm, float c) {
    const float mn = max_nan(m, vm);
    if (mn != m) {
      const float mcn = __fmul_rn(mn, c);
      const float f = exp2f(mc - mcn);
      s0 = __fmul2_rn(s0, make_float2(f, f));
      s1 = __fmul2_rn(s1, make_float2(f, f));
      m = mn;
      mc = mcn;
    }
  }
  __device__ __forceinline__ void sum8(const float (&z)[8], float c) {
    const float2 c2 = make_float2(c, c), n2 = make_float2(-mc, -mc);
#pragma unroll
    for (int k = 0; k < 8; k += 4) {
      const float2 a = __ffma2_rn(make_float2(z[k], z[k + 1]), c2, n2);
      const float2 b = __ffma2_rn(make_float2(z[k + 2], z[k + 3]), c2, n2);
      s0 = __fadd2_rn(s0, make_float2(ex2_fast(a.x), ex2_fast(a.y)));
      s1 = __fadd2_rn(s1, make_float2(ex2_fast(b.x), ex2_fast(b.y)));
    }
  }
  __device__ __forceinline__ float total() const { return (s0.x + s0.y) + (s1.x + s1.y); }
};

__device__ __forceinline__ void top8_insert(unsigned long long (&keys)[8], float& thr, float z,
                                            uint32_t id) {
  if (!(z >= thr)) return;
  unsigned long long key = make_key(z, id);
  if (key <= keys[7]) return;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const unsigned long long hi = key > keys[j] ? key : keys[j];
    const unsigned long long lo = key > keys[j] ? keys[j] : key;
    keys[j] = hi;
    key = lo;
  }
  if (keys[7]) thr = key_value(keys[7]);
}


// The largest key over the warp (keys are distinct unless 0): the upper halves first, then the
// lower halves of the lanes that hold the largest upper half.
__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long k) {
  const uint32_t hi = static_cast<uint32_t>(k >> 32);
  const uint32_t mh = __reduce_max_sync(FULL, hi);
  const uint32_t ml = __reduce_max_sync(FULL, hi == mh ? static_cast<uint32_t>(k) : 0u);
  return (static_cast<unsigned long long>(mh) << 32) | ml;
}

// Merge every lane's descending list of 8 keys into the warp's top 8 (the result on every
// lane); the lanes' lists are consumed.
__device__ __forceinline__ void warp_top8(unsigned long long (&keys)[8],
                                          unsigned long long (&out)[8]) {
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const unsigned long long m = warp_max_u64(keys[0]);
    if (m != 0ull && keys[0] == m) {
#pragma unroll
      for (int j = 0; j < 7; ++j) keys[j] = keys[j + 1];
      keys[7] = 0ull;
    }
    out[r] = m;
  }
}

}  // namespace sv

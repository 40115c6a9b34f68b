// Fused batched speculative-sampling verify kernel for sm_103a.
//
// One thread-block cluster of C CTAs owns one sequence at a time and walks its draft
// positions in order (Kangaroo guide, section "3. Lossless Speculative Verification":
// verification terminates at the first rejection), so the rows after the outcome is fixed are
// not needed. Each CTA owns a contiguous slice of the vocabulary.
//
// Row path. Per CTA, a ring of NS shared-memory stages is filled with bulk async copies
// (cp.async.bulk, completion on an mbarrier) by one producer thread that runs ahead of the
// consumers: through the rest of the current position, speculatively into the next position
// of the sequence, and into the next sequence of the queue. Every thread folds its elements
// into a running maximum and a running sum of 2^(z c - m c) (single pass), so at the end of
// a position each CTA holds its slice's (max, sum) for the target and draft rows.
//
// Decision. The CTAs exchange their partials through distributed shared memory; every CTA
// combines the C partials in the same order and reaches the same accept / reject decision.
// The producer learns the decision and stops fetching rows the outcome no longer needs.
//
// Draw. After a rejection (or when every draft is accepted) each CTA re-reads its slice of the
// two rows at the decided position (they were streamed microseconds earlier and sit in L2)
// with 128-bit loads, turns them into residual (or bonus) weights, keeps one partial mass per
// 8-element vector in shared memory, and sums them as 64-bit integers of 2^-44, so the
// cross-CTA and block prefix sums of the inverse CDF are exact and order independent. The CTA
// whose range holds the draw scans its vector masses and walks the one vector that holds it.
//
// Bounded waits: each mbarrier wait gives up after ~2 s, raises the workspace error word, and
// the cluster marks the sequence -2 and leaves. There is no other spin-wait; cross-CTA ordering
// uses the hardware cluster barrier.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "sv_internal.h"
#include "sv_small.h"
#include "sv_math.cuh"
#include "sv_ptx.cuh"

namespace sv {
namespace {

constexpr int NT = kThreads;
constexpr int NW = NT / 32;
constexpr float kLn2 = 0.69314718055994531f;
constexpr long long kWaitBudget = 4000000000LL;  // clock cycles (about 2 s)
constexpr unsigned XF_ABORT = 1u;
constexpr int ROW_T = 1, ROW_D = 2;
constexpr int NC = NT;            // consumer threads (warps 0..7)
constexpr int NTOT = NT + 32;     // plus one producer warp
constexpr uint32_t kConsumerBar = 1;

// Barrier among the consumer warps only (the producer warp never joins it).
__device__ __forceinline__ void cbar() { named_sync(kConsumerBar, NC); }
__device__ __forceinline__ bool cbar_or(bool p) { return named_sync_or(kConsumerBar, NC, p); }

// Partial results one CTA publishes to every CTA of its cluster (7 chunks of 16 bytes).
struct __align__(16) Xchg {
  float m_t, s_t, m_d, s_d;     // chunk 0: slice maxima (raw logits) and sums 2^((z-m)c)
  int arg;                      // chunk 1: greedy, lowest index of the slice maximum
  int next_seq;                 //          rank 0, first exchange of a sequence
  unsigned flags;
  int pad0;
  unsigned long long top8[8];   // chunks 2..5: draft keys, descending
  unsigned long long w;         // chunk 6: residual / bonus mass, fixed point
  unsigned long long pad1;
};
static_assert(sizeof(Xchg) == 112, "exchange record layout");

struct __align__(16) Hdr {
  unsigned long long key[kMaxK][8];  // the prepass's top-8 keys of each draft row (if any)
  int L, ok;
  int x[kMaxK];
  float u[kMaxK + 1];
};

// What a stage holds, packed in one 64-bit word: sequence (bits 0..23), its epoch in the
// cluster's order mod 256 (bits 24..31), position + 64 (bits 32..39; positions below 0 mark
// chunks of the draw pass), chunk (bits 40..55), rows (ROW_T | ROW_D, bits 56..57).
__device__ __forceinline__ unsigned long long stage_tag(int seq, int ep, int pos, int k) {
  return static_cast<unsigned long long>((static_cast<uint32_t>(seq) & 0xFFFFFFu) |
                                         ((static_cast<uint32_t>(ep) & 0xFFu) << 24)) |
         (static_cast<unsigned long long>((pos + 64) & 0xFF) << 32) |
         (static_cast<unsigned long long>(k & 0xFFFF) << 40);
}
__device__ __forceinline__ int tag_ep(unsigned long long t) { return static_cast<int>((t >> 24) & 0xFF); }
__device__ __forceinline__ int tag_pos(unsigned long long t) { return static_cast<int>((t >> 32) & 0xFF) - 64; }
__device__ __forceinline__ int tag_k(unsigned long long t) { return static_cast<int>((t >> 40) & 0xFFFF); }
constexpr unsigned long long kTagMask = (1ull << 56) - 1ull;
__device__ __forceinline__ int tag_rows(unsigned long long t) { return static_cast<int>(t >> 56); }

// Position in the ring: running count, stage index and phase parity, advanced together; for the
// consumers also the epoch of the sequence they are on.
struct Cursor {
  int n = 0, s = 0;
  uint32_t ph = 0;
  int ep = 0;
  __device__ __forceinline__ void advance() {
    ++n;
    if (++s == NS) {
      s = 0;
      ph ^= 1u;
    }
  }
};

// What the consumers tell the producer warp: two 64-bit shared-memory words, each written and
// read with one 8-byte access (consumer thread 0 writes, the producer lane reads).
//   cur:  current sequence (bits 0..31), epoch = its place in the cluster's sequence order
//         (bits 32..47, mod 2^16), decided position + 2 (bits 48..55; 1 = undecided, 0 = nothing
//         more needed), consumers done (bit 56).
//   next: next sequence of the queue (bits 0..31), the epoch it follows (bits 32..47), known
//         (bit 48).
struct Pub {
  int seq, ep, stop, done;
};
__device__ __forceinline__ unsigned long long pack_cur(int seq, int ep, int stop, int done) {
  return static_cast<unsigned long long>(static_cast<uint32_t>(seq)) |
         (static_cast<unsigned long long>(ep & 0xFFFF) << 32) |
         (static_cast<unsigned long long>((stop + 2) & 0xFF) << 48) |
         (static_cast<unsigned long long>(done ? 1 : 0) << 56);
}
__device__ __forceinline__ Pub unpack_cur(unsigned long long w) {
  Pub v;
  v.seq = static_cast<int>(static_cast<uint32_t>(w));
  v.ep = static_cast<int>((w >> 32) & 0xFFFF);
  v.stop = static_cast<int>((w >> 48) & 0xFF) - 2;
  v.done = static_cast<int>((w >> 56) & 1);
  return v;
}
__device__ __forceinline__ unsigned long long pack_next(int seq, int ep) {
  return static_cast<unsigned long long>(static_cast<uint32_t>(seq)) |
         (static_cast<unsigned long long>(ep & 0xFFFF) << 32) | (1ull << 48);
}

struct CtaState {
  Hdr hdr[2];        // current and next sequence header (cp.async targets)
  int cur;           // hdr[cur] is the current sequence
  int n_hdr_wait;    // consumer thread 0 has a header copy in flight
  unsigned long long pub_cur, pub_next;  // consumer -> producer words (see Pub)
  int cons_final;    // stages the consumers took, published before `done`
  int seq0;          // this cluster's first sequence
  int dec;           // decision of the last combined position: -1 accept, a >= 0 stop at a,
                     // -2 unusable row, -3 a wait gave up (written by consumer warp 0)
  int next;          // the sequence this cluster takes next (from the first exchange)
  unsigned long long nxt_word;  // (epoch + 1) << 32 | next sequence, stored by rank 0 once the
                                // current sequence of a decision-ahead walk is decided
  // reduction scratch (one slot per kind)
  float rmax[2][NW];
  float rsum[2][NW];
  int rarg[NW];
  unsigned long long ru[NW];
  unsigned long long wtop[NW][8];
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
// block reductions (result returned to every thread)
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ float2 block_max2(float a, float b, CtaState& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = warp_max_nan(a);
  b = warp_max_nan(b);
  if (lane == 0) { S.rmax[0][warp] = a; S.rmax[1][warp] = b; }
  cbar();
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
  cbar();
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
  cbar();
  int r = S.rarg[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) r = min(r, S.rarg[w]);
  return r;
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, CtaState& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_u64(v);
  if (lane == 0) S.ru[warp] = v;
  cbar();
  unsigned long long r = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) r += S.ru[w];
  cbar();
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
  cbar();
  unsigned long long base = 0;
  for (int w = 0; w < warp; ++w) base += S.ru[w];
  cbar();
  return base + inc - v;
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
  cbar();
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

// Publish chunks [c0, c0 + nc) of S.rec into slot `rank` of buffer `round & 1` of every CTA
// of the cluster with st.async, and wait until every CTA's chunks have landed here (counted as
// transaction bytes on this CTA's exchange barrier). A buffer is rewritten two rounds later,
// which a CTA can only reach after every peer has pushed the round in between, i.e. after
// every peer has read this round. Returns false if the wait gave up.
__device__ __forceinline__ void exchange_post(CtaState& S, Xchg (*X)[kMaxCluster],
                                              uint64_t* xbar, uint32_t& round, uint32_t rank,
                                              uint32_t C, int c0, int nc) {
  const int tid = threadIdx.x;
  const uint32_t p = round & 1u;
  ++round;
  if (tid == 0) mbar_arrive_expect_tx(&xbar[p], C * static_cast<uint32_t>(nc) * 16u);
  if (tid < static_cast<int>(C) * nc) {
    const uint32_t peer = tid / nc;
    const int ch = c0 + tid % nc;
    const uint32_t dst = map_to_rank(smem_u32(&X[p][rank]) + 16u * ch, peer);
    const uint32_t bar = map_to_rank(smem_u32(&xbar[p]), peer);
    st_async_v4(dst, reinterpret_cast<const uint4*>(&S.rec)[ch], bar);
  }
}
__device__ __forceinline__ bool exchange(CtaState& S, Xchg (*X)[kMaxCluster], uint64_t* xbar,
                                         uint32_t& round, uint32_t rank, uint32_t C, int c0,
                                         int nc) {
  const uint32_t r = round;
  exchange_post(S, X, xbar, round, rank, C, c0, nc);
  return mbar_wait_cluster_bounded(&xbar[r & 1u], (r >> 1) & 1u, kWaitBudget);
}

// ------------------------------------------------------------------------------------------
// consumer -> producer publication
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void pub_store(unsigned long long* w, unsigned long long v) {
  *reinterpret_cast<volatile unsigned long long*>(w) = v;
}
__device__ __forceinline__ unsigned long long pub_load(const unsigned long long* w) {
  return *reinterpret_cast<const volatile unsigned long long*>(w);
}

// ------------------------------------------------------------------------------------------
// the stage ring: the producer warp fills stages with bulk async copies, consumers drain them
// ------------------------------------------------------------------------------------------
template <typename T, bool GREEDY>
struct Ring {
  static constexpr int kRows = GREEDY ? 1 : 2;
  static constexpr int CH = kStageRowBytes / static_cast<int>(sizeof(T));  // elements / chunk
  unsigned char* base;
  uint64_t* full;
  uint64_t* empty;
  unsigned long long* desc;  // stage_tag | rows << 56 of what each stage holds
  int nchunk;  // chunks per row of this CTA's slice
  int nv;      // elements of this CTA's slice
  int v0;      // first element of the slice
  T* scr;      // rows read in place from host memory: this CTA's copy of the slices of the
               // position last streamed (2 rows of `slice` elements), which the draw reads back

  __device__ __forceinline__ T* row(int s, int r) const {
    return reinterpret_cast<T*>(base + (static_cast<size_t>(s) * kRows + r) * kStageRowBytes);
  }
  __device__ __forceinline__ int chunk_len(int k) const { return min(CH, nv - k * CH); }
};

__device__ __forceinline__ const void* row_ptr(const Params& P, bool draft, int seq, int pos,
                                               size_t elt) {
  const char* base = static_cast<const char*>(draft ? P.dft : P.tgt);
  const long long rows = draft ? P.K : P.K + 1;
  const long long stride = draft ? P.d_stride : P.t_stride;
  return base + ((static_cast<long long>(seq) * rows + pos) * stride) * static_cast<long long>(elt);
}

__device__ __forceinline__ int load_len(const Params& P, int seq) {
  if (seq < 0 || seq >= P.B) return -1;
  const int L = P.lens ? P.lens[seq] : P.K;
  return (L >= 1 && L <= P.K) ? L : -1;
}

// One chunk into stage s: `src_t` / `src_d` point at this CTA's slice of the two rows (bytes),
// `tag` is the stage tag recorded for the consumers.
template <typename T, bool GREEDY>
__device__ __forceinline__ void issue_chunk(const Params& P, const Ring<T, GREEDY>& R, int s,
                                            const char* src_t, const char* src_d,
                                            unsigned long long tag, int k, int rows) {
  R.desc[s] = tag | (static_cast<unsigned long long>(rows) << 56);
  if (!P.use_bulk) {
    mbar_arrive(&R.full[s]);  // the consumers copy this chunk themselves
    return;
  }
  const int n = R.chunk_len(k);
  const size_t off = static_cast<size_t>(k) * kStageRowBytes;
  if (n == R.CH) {  // a whole chunk: one copy per row, nothing else to fill
    const uint32_t nrows = (rows & ROW_T ? 1u : 0u) + (rows & ROW_D ? 1u : 0u);
    mbar_arrive_expect_tx(&R.full[s], nrows * kStageRowBytes);
    if (rows & ROW_T) bulk_g2s(R.row(s, 0), src_t + off, kStageRowBytes, &R.full[s]);
    if (!GREEDY && (rows & ROW_D)) bulk_g2s(R.row(s, 1), src_d + off, kStageRowBytes, &R.full[s]);
    return;
  }
  constexpr int kPer16 = 16 / static_cast<int>(sizeof(T));
  const int nb = (n / kPer16) * kPer16;
  const int npad = (n + 7) & ~7;
  uint32_t bytes = 0;
  for (int r = 0; r < Ring<T, GREEDY>::kRows; ++r) {
    if (!(rows & (1 << r))) continue;
    const T* src = reinterpret_cast<const T*>((r ? src_d : src_t) + off);
    T* dst = R.row(s, r);
    for (int e = nb; e < npad; ++e) dst[e] = e < n ? src[e] : Elt<T>::neg_inf();
    bytes += static_cast<uint32_t>(nb * sizeof(T));
  }
  mbar_arrive_expect_tx(&R.full[s], bytes);
  if (nb > 0) {
    for (int r = 0; r < Ring<T, GREEDY>::kRows; ++r) {
      if (!(rows & (1 << r))) continue;
      bulk_g2s(R.row(s, r), (r ? src_d : src_t) + off, static_cast<uint32_t>(nb * sizeof(T)),
               &R.full[s]);
    }
  }
}

// The producer warp's lane 0. It walks the cluster's sequence order: the positions of the
// current sequence speculatively (all rows up to the bonus row), and once the consumers publish
// the decision, the draw pass over the decided position, then the rows the diagnostics or the
// top-F output still need, then the next sequence. It never runs past an undecided stochastic
// sequence, so the ring always holds chunks in the order the consumers take them.
template <typename T, bool GREEDY>
__device__ void producer(const Params& P, CtaState& S, const Ring<T, GREEDY>& R) {
  enum { STATS = 0, DRAW = 1, POST = 2 };
  int q_ep = 0, q_seq = S.seq0, q_L = load_len(P, S.seq0);
  int q_ph = STATS, q_pos = 0, q_k = 0;
  int q_mark = -1;  // greedy: the stop whose marker stage is still to be issued
  Cursor cur;
  int base_seq = -1, base_pos = -1;
  const char* src_t = nullptr;
  const char* src_d = nullptr;
  long long idle0 = clock64();
  while (true) {
    const Pub pub = unpack_cur(pub_load(&S.pub_cur));
    if (pub.done) break;
    if (clock64() - idle0 > kWaitBudget) {
      atomicOr(&P.ws->error, 1u);
      break;
    }
    if (R.nchunk == 0) {
      sleep_ns(256);
      idle0 = clock64();
      continue;
    }
    const int lag = static_cast<int16_t>(static_cast<uint16_t>(pub.ep - q_ep));
    if (lag > 0) {  // the consumers are past this sequence (it needed no chunks)
      q_ep += lag;
      q_seq = pub.seq;
      q_L = load_len(P, q_seq);
      q_ph = STATS;
      q_pos = 0;
      q_k = 0;
      q_mark = -1;  // nobody waits on the earlier sequence any more
    }
    int rows = 0;
    bool exhausted = q_seq >= P.B;
    if (!exhausted && lag >= 0) {  // the consumers' current sequence
      const int stop = pub.stop;
      if (stop != -1 && q_ph == STATS) {
        if (stop == -2) {  // an invalid sequence: nothing more to stream
          q_ph = POST;
          q_pos = P.K + 1;
          q_mark = 0;
        } else {  // the decision has landed
          // (a deferred draw, like a greedy stop, streams nothing more of this sequence)
          const bool nodraw = GREEDY || P.defer;
          q_ph = nodraw ? POST : DRAW;
          q_pos = nodraw ? stop + 1 : stop;
          if (nodraw) q_mark = stop;
        }
        q_k = 0;
      }
      if (q_mark >= 0) {
        // Without a draw pass (a greedy stop, an invalid sequence) no chunk would tell the
        // consumers still waiting on a chunk of the position being streamed that the producer
        // has moved on: one stage without data, tagged like a draw chunk, does (consumers that
        // are not waiting hand it back).
        if (cur.n >= NS && !mbar_try_wait_hint(&R.empty[cur.s], cur.ph ^ 1u, 1000)) continue;
        R.desc[cur.s] = stage_tag(q_seq, q_ep, -1 - q_mark, 0);
        mbar_arrive(&R.full[cur.s]);
        cur.advance();
        q_mark = -1;
        idle0 = clock64();
        continue;
      }
      if (stop == -2) {
        exhausted = true;
      } else {
        if (q_ph == STATS) {
          if (q_pos <= q_L) rows = (!GREEDY && q_pos < q_L) ? (ROW_T | ROW_D) : ROW_T;
        } else if (q_ph == DRAW) {
          rows = (q_pos < q_L) ? (ROW_T | ROW_D) : ROW_T;
        } else {
          if (q_pos <= q_L) {
            rows = P.debug_all ? ROW_T : 0;
            if (!GREEDY && q_pos < q_L && (P.fmax > 0 || P.debug_all)) rows |= ROW_D;
          }
          exhausted = rows == 0;
        }
      }
      if (exhausted && q_seq < P.B) {  // move on once the next sequence is known
        const unsigned long long nw = pub_load(&S.pub_next);
        const unsigned long long xw = *reinterpret_cast<volatile unsigned long long*>(&S.nxt_word);
        int nq = -1;
        if ((nw >> 48) & 1ull && static_cast<int>((nw >> 32) & 0xFFFF) == (q_ep & 0xFFFF))
          nq = static_cast<int>(static_cast<uint32_t>(nw));
        else if ((xw >> 32) == static_cast<unsigned long long>(static_cast<uint32_t>(q_ep + 1)))
          nq = static_cast<int>(static_cast<uint32_t>(xw));
        if (nq >= 0) {
          ++q_ep;
          q_seq = nq;
          q_L = load_len(P, q_seq);
          q_ph = STATS;
          q_pos = 0;
          q_k = 0;
          continue;
        }
      }
    } else if (!exhausted && q_ph == STATS && q_pos <= q_L) {  // the next sequence, early
      rows = (!GREEDY && q_pos < q_L) ? (ROW_T | ROW_D) : ROW_T;
    }
    if (exhausted || rows == 0) {
      sleep_ns(128);
      continue;
    }
    if (q_k == 0 || base_seq != q_seq || base_pos != q_pos) {  // row bases of this position
      base_seq = q_seq;
      base_pos = q_pos;
      src_t = static_cast<const char*>(row_ptr(P, false, q_seq, q_pos, sizeof(T))) +
              static_cast<size_t>(R.v0) * sizeof(T);
      src_d = GREEDY || q_pos >= P.K ? src_t
                                     : static_cast<const char*>(row_ptr(P, true, q_seq, q_pos, sizeof(T))) +
                                           static_cast<size_t>(R.v0) * sizeof(T);
    }
    if (cur.n >= NS && !mbar_try_wait_hint(&R.empty[cur.s], cur.ph ^ 1u, 1000)) {
      continue;  // the oldest stage is still being read (the wait above slept on it)
    }
    issue_chunk<T, GREEDY>(P, R, cur.s, src_t, src_d,
                           stage_tag(q_seq, q_ep, q_ph == DRAW ? -1 - q_pos : q_pos, q_k), q_k, rows);
    cur.advance();
    idle0 = clock64();
    if (++q_k >= R.nchunk) {
      q_k = 0;
      if (q_ph == DRAW) q_ph = POST;
      ++q_pos;
    }
  }
  // wait out the copies still in flight into stages nobody will read
  __threadfence_block();
  const int cons = *reinterpret_cast<volatile int*>(&S.cons_final);
  const bool done = unpack_cur(pub_load(&S.pub_cur)).done != 0;
  for (int j = done ? cons : cur.n; j < cur.n; ++j)
    mbar_wait_bounded(&R.full[j % NS], static_cast<uint32_t>(j / NS) & 1u, kWaitBudget);
}

__device__ __forceinline__ void release_stage(uint64_t* empty, Cursor& cons) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&empty[cons.s]);
  cons.advance();
}

// Wait for the stage holding chunk k of (seq, pos), handing back stale speculative chunks on
// the way. Returns the stage, or -1 once a wait has given up (`late`).
template <typename T, bool GREEDY>
__device__ __forceinline__ int acquire(const Ring<T, GREEDY>& R, int seq, int pos, int k,
                                       Cursor& cons, bool& late) {
  const unsigned long long want = stage_tag(seq, cons.ep, pos, k);
  while (!late) {
    if (!mbar_wait_bounded(&R.full[cons.s], cons.ph, kWaitBudget)) {
      late = true;
      break;
    }
    if ((R.desc[cons.s] & kTagMask) == want) return cons.s;
    release_stage(R.empty, cons);
  }
  return -1;
}

// Stats chunk k of position pos of the current sequence, while the decision of the previous
// position may still be open: stale chunks (an earlier sequence, or what this sequence's
// consumers have already moved past) are handed back; a chunk of the draw pass or of a later
// sequence means the producer has acted on a stop, and returns -2 without taking the stage.
// -1 once a wait has given up.
template <typename T, bool GREEDY>
__device__ __forceinline__ int acquire_open(const Ring<T, GREEDY>& R, int seq, int pos, int k,
                                           Cursor& cons, bool& late) {
  const unsigned long long want = stage_tag(seq, cons.ep, pos, k);
  while (!late) {
    if (!mbar_wait_bounded(&R.full[cons.s], cons.ph, kWaitBudget)) {
      late = true;
      break;
    }
    const unsigned long long t = R.desc[cons.s];
    if ((t & kTagMask) == want) return cons.s;
    const int d = static_cast<int8_t>(static_cast<uint8_t>(tag_ep(t) - cons.ep));
    const int tp = tag_pos(t), tk = tag_k(t);
    if (d == 0 && tp == pos && tk == k) return cons.s;
    if (d > 0 || (d == 0 && (tp < 0 || tp > pos || (tp == pos && tk > k)))) return -2;
    release_stage(R.empty, cons);
  }
  return -1;
}

// Rows that are not 16-byte aligned are not fetched by the producer: every consumer copies its
// share of the chunk, then the consumers synchronise. All consumers call this, `late` or not.
template <typename T, bool GREEDY>
__device__ int fill_unaligned(const Params& P, const Ring<T, GREEDY>& R, int s, int seq,
                              int pos, int k, bool& late, bool draw = false) {
  if (s >= 0) {
    const int rows = tag_rows(R.desc[s]);
    const int n = R.chunk_len(k), npad = (n + 7) & ~7;
    for (int r = 0; r < Ring<T, GREEDY>::kRows; ++r) {
      if (!(rows & (1 << r))) continue;
      // the draw reads the decided position back from this CTA's copy when it has one
      T* keep = R.scr ? R.scr + static_cast<size_t>(r) * P.slice + static_cast<size_t>(k) * R.CH
                      : nullptr;
      const T* src = (draw && keep) ? keep
                                    : static_cast<const T*>(row_ptr(P, r == 1, seq, pos, sizeof(T))) +
                                          R.v0 + k * R.CH;
      if (draw) keep = nullptr;
      T* dst = R.row(s, r);
      int e0 = 0;
      if (P.vec_fill) {  // whole 16-byte pieces, four loads in flight per thread
        constexpr int kPer16 = 16 / static_cast<int>(sizeof(T));
        const int n16 = n / kPer16;
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
        uint4* d4 = reinterpret_cast<uint4*>(dst);
        uint4* k4 = reinterpret_cast<uint4*>(keep);
        int e = threadIdx.x;
        for (; e + 3 * NC < n16; e += 4 * NC) {
          const uint4 a0 = s4[e], a1 = s4[e + NC], a2 = s4[e + 2 * NC], a3 = s4[e + 3 * NC];
          d4[e] = a0;
          d4[e + NC] = a1;
          d4[e + 2 * NC] = a2;
          d4[e + 3 * NC] = a3;
          if (k4) {
            k4[e] = a0;
            k4[e + NC] = a1;
            k4[e + 2 * NC] = a2;
            k4[e + 3 * NC] = a3;
          }
        }
        for (; e < n16; e += NC) {
          const uint4 a0 = s4[e];
          d4[e] = a0;
          if (k4) k4[e] = a0;
        }
        e0 = n16 * kPer16;
      }
      for (int e = e0 + threadIdx.x; e < npad; e += NC) {
        const T v = e < n ? src[e] : Elt<T>::neg_inf();
        dst[e] = v;
        if (keep && e < n) keep[e] = v;
      }
    }
  }
  late = cbar_or(late || s < 0);
  return late ? -1 : s;
}

// This thread's vectors of one staged chunk row (vector g = threadIdx.x + j * NC), loaded into
// registers before any arithmetic; vectors past nvec read as -inf.
template <typename T, int VPT>
struct ChunkRow;

template <int VPT>
struct ChunkRow<uint16_t, VPT> {
  uint4 v[VPT];
  __device__ __forceinline__ void load(const uint16_t* row, int nvec) {
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int g = threadIdx.x + j * NC;
      v[j] = g < nvec ? reinterpret_cast<const uint4*>(row)[g]
                      : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
    }
  }
  __device__ __forceinline__ void load_full(const uint16_t* row) {
#pragma unroll
    for (int j = 0; j < VPT; ++j) v[j] = reinterpret_cast<const uint4*>(row)[threadIdx.x + j * NC];
  }
  __device__ __forceinline__ float vmax() const {  // NaN-propagating
    uint32_t m = max_nan_bf16x2(max_nan_bf16x2(v[0].x, v[0].y), max_nan_bf16x2(v[0].z, v[0].w));
#pragma unroll
    for (int j = 1; j < VPT; ++j)
      m = max_nan_bf16x2(m, max_nan_bf16x2(max_nan_bf16x2(v[j].x, v[j].y),
                                           max_nan_bf16x2(v[j].z, v[j].w)));
    return max_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
  }
  __device__ __forceinline__ void get(int j, float (&z)[8]) const { Elt<uint16_t>::unpack(v[j], z); }
};

template <int VPT>
struct ChunkRow<float, VPT> {
  float4 v[VPT][2];
  __device__ __forceinline__ void load(const float* row, int nvec) {
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int g = threadIdx.x + j * NC;
      if (g < nvec) {
        v[j][0] = reinterpret_cast<const float4*>(row)[2 * g];
        v[j][1] = reinterpret_cast<const float4*>(row)[2 * g + 1];
      } else {
        v[j][0] = v[j][1] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
    }
  }
  __device__ __forceinline__ void load_full(const float* row) {
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
      const int g = threadIdx.x + j * NC;
      v[j][0] = reinterpret_cast<const float4*>(row)[2 * g];
      v[j][1] = reinterpret_cast<const float4*>(row)[2 * g + 1];
    }
  }
  __device__ __forceinline__ float vmax() const {
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < VPT; ++j)
      m = max_nan(m, max_nan(max_nan(max_nan(v[j][0].x, v[j][0].y), max_nan(v[j][0].z, v[j][0].w)),
                             max_nan(max_nan(v[j][1].x, v[j][1].y), max_nan(v[j][1].z, v[j][1].w))));
    return m;
  }
  __device__ __forceinline__ void get(int j, float (&z)[8]) const {
    z[0] = v[j][0].x; z[1] = v[j][0].y; z[2] = v[j][0].z; z[3] = v[j][0].w;
    z[4] = v[j][1].x; z[5] = v[j][1].y; z[6] = v[j][1].z; z[7] = v[j][1].w;
  }
};

// The stochastic stats pass over the whole chunks [0, kf) of a position: running max and sum of
// the target row and, when TWO, of the draft row. Same arithmetic, in the same order, as the
// general chunk loop; no per-vector bounds, no per-chunk mode tests. Returns the chunks done
// (fewer than kf only when a wait gave up).
template <typename T, bool TWO>
__device__ __forceinline__ int stream_whole(const Ring<T, false>& R, int seq, int i, int kf,
                                            Cursor& cons, bool& late, RowAcc& at, RowAcc& ad,
                                            float c) {
  constexpr int VPT = Ring<T, false>::CH / 8 / NC;
  for (int k = 0; k < kf; ++k) {
    const int s = acquire<T, false>(R, seq, i, k, cons, late);
    if (s < 0) return k;
    ChunkRow<T, VPT> ct, cd;
    ct.load_full(R.row(s, 0));
    if (TWO) cd.load_full(R.row(s, 1));
    at.rescale(ct.vmax(), c);
    if (TWO) ad.rescale(cd.vmax(), c);
    if (at.m > -INFINITY) {
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
        float z[8];
        ct.get(j, z);
        at.sum8(z, c);
      }
    }
    if (TWO && ad.m > -INFINITY) {
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
        float z[8];
        cd.get(j, z);
        ad.sum8(z, c);
      }
    }
    release_stage(R.empty, cons);
  }
  return kf;
}

// ------------------------------------------------------------------------------------------
// residual / bonus draw
// ------------------------------------------------------------------------------------------
struct WeightConsts {
  float c, mc_t, mc_d, rho, rho_S;
  int nloc;     // ids of the bias set that fall in this CTA's slice
  int loc[8];   // their slice-local indices
};

// Weights of the 8 elements at slice offset e0, up to one positive factor per draw (the inverse
// CDF does not depend on it): bonus -> e_t = 2^(z_t c - mc_t); residual ->
// max(e_t - rho e_d, 0) with e_d = 2^(z_d c - mc_d) and rho = q' scale / p scale, which is
// max(p - q', 0) / (p scale). Returns their sequential sum.
template <bool BONUS>
__device__ __forceinline__ float weights8(const float (&zt)[8], const float (&zd)[8], int e0,
                                          const WeightConsts& W, float (&w)[8]) {
  if constexpr (BONUS) {
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = ex2_fast(fmaf(zt[k], W.c, -W.mc_t));
  } else {
    float rk[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) rk[k] = W.rho;
    for (int j = 0; j < W.nloc; ++j) {
      const int e = W.loc[j] - e0;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k == e) rk[k] = W.rho_S;
    }
    const float2 c2 = make_float2(W.c, W.c), n2 = make_float2(-W.mc_t, -W.mc_d);
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
      // exponent arguments of the target and draft element together, then two weights together
      const float2 a0 = __ffma2_rn(make_float2(zt[k], zd[k]), c2, n2);
      const float2 a1 = __ffma2_rn(make_float2(zt[k + 1], zd[k + 1]), c2, n2);
      const float2 wv = __ffma2_rn(make_float2(-ex2_fast(a0.y), -ex2_fast(a1.y)),
                                   make_float2(rk[k], rk[k + 1]),
                                   make_float2(ex2_fast(a0.x), ex2_fast(a1.x)));
      w[k] = fmaxf(wv.x, 0.f);
      w[k + 1] = fmaxf(wv.y, 0.f);
    }
  }
  float s = w[0];
#pragma unroll
  for (int k = 1; k < 8; ++k) s = __fadd_rn(s, w[k]);
  return s;
}

// Sum of a u64 over the 8 lanes of an aligned group of 8 (every lane gets the sum).
__device__ __forceinline__ unsigned long long group8_sum_u64(unsigned long long v) {
  v += __shfl_xor_sync(FULL, v, 1);
  v += __shfl_xor_sync(FULL, v, 2);
  v += __shfl_xor_sync(FULL, v, 4);
  return v;
}

// The cluster draws the token at position `a` of sequence `seq`. The rows come back through
// the ring (the producer fetches them again right after the decision; they are still in L2);
// every 8-element vector's mass is truncated to 2^-44 units, and `gmass` keeps the sum of those
// units per group of 8 vectors (64 elements), so shared memory holds 8 bytes per 64 elements.
// The CTA whose range holds the draw finds the group by a prefix over `gmass`, recomputes the
// group's 8 vector masses and walks them, then the vector's elements, and writes out_tok. All
// consumers of all CTAs of the cluster call this together.
template <typename T, bool GREEDY, bool BONUS>
__device__ void draw_token(const Params& P, CtaState& S, Xchg (*X)[kMaxCluster],
                           uint64_t* xbar, uint32_t& xround, uint32_t rank, uint32_t C,
                           const Ring<T, GREEDY>& R, int seq, int a,
                           unsigned long long* gmass, Cursor& cons, bool& late) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int v0 = R.v0, nv = R.nv;
  const int nvec_all = (nv + 7) >> 3;
  const bool aligned = P.use_bulk != 0;
  const T* gt = static_cast<const T*>(row_ptr(P, false, seq, a, sizeof(T))) + v0;
  const T* gd = BONUS ? gt : static_cast<const T*>(row_ptr(P, true, seq, a, sizeof(T))) + v0;
  WeightConsts W;
  W.c = P.c;
  // p(v) = 2^(z_t c - mc_t) * (1 - err_t ln 2) / S_t and q'(v) = f(v) 2^(z_d c - mc_d) *
  // (1 - err_d ln 2) / (S_d N), with err the rounding of M c; weights are taken relative to p's
  // scale, so rho = q' scale / p scale.
  W.mc_t = __fmul_rn(S.M_t, P.c);
  W.mc_d = __fmul_rn(S.M_d, P.c);
  if (BONUS) {
    W.rho = W.rho_S = 0.f;
  } else {
    const float ft = fmaf(-fmaf(S.M_t, P.c, -W.mc_t), kLn2, 1.f);
    const float fd = fmaf(-fmaf(S.M_d, P.c, -W.mc_d), kLn2, 1.f);
    W.rho = (fd * S.S_t) / (ft * (S.S_d * S.N));
    W.rho_S = W.rho * P.beta;
  }
  W.nloc = 0;
  for (int j = 0; j < S.nS; ++j) {
    const int e = S.S_ids[j] - v0;
    if (e >= 0 && e < nv) W.loc[W.nloc++] = e;
  }
  unsigned long long acc = 0;
  for (int k = 0; k < R.nchunk; ++k) {
    int s = acquire<T, GREEDY>(R, seq, -1 - a, k, cons, late);
    if (!P.use_bulk) s = fill_unaligned<T, GREEDY>(P, R, s, seq, a, k, late, true);
    if (s < 0) break;
    const int n = R.chunk_len(k), nvec = (n + 7) >> 3;
    const T* rt = R.row(s, 0);
    const T* rd = R.row(s, GREEDY ? 0 : 1);
    // vector g of the chunk (lanes 8j .. 8j + 7 hold the 8 vectors of one group, since NC and
    // the chunk are multiples of 64 elements); every lane of the warp takes part
    auto vec = [&](int g, bool have) {
      unsigned long long q = 0;
      if (have) {
        float zt[8], zd[8], w[8];
        Elt<T>::load8(rt, g, zt);
        if (!BONUS) Elt<T>::load8(rd, g, zd);
        q = qfix(weights8<BONUS>(zt, BONUS ? zt : zd, k * R.CH + 8 * g, W, w));
      }
      acc += q;
      const unsigned long long gq = group8_sum_u64(q);
      if ((lane & 7) == 0 && have) gmass[(k * (R.CH / 8) + g) >> 3] = gq;
    };
    constexpr int VPT = Ring<T, GREEDY>::CH / 8 / NC;
    if (n == R.CH) {  // a whole chunk: exactly VPT vectors per thread
#pragma unroll
      for (int j = 0; j < VPT; ++j) vec(tid + j * NC, true);
    } else {
      for (int j = 0; j * NC < nvec; ++j) vec(tid + j * NC, tid + j * NC < nvec);
    }
    release_stage(R.empty, cons);
  }
  late = cbar_or(late);
  unsigned long long Wtot = 0;
  for (int attempt = 0; attempt < 2; ++attempt) {
    if (attempt == 1) {  // zero residual mass: draw from p at this position instead
      W.rho = 0.f;
      W.rho_S = 0.f;
      W.mc_d = INFINITY;  // the draft term becomes 2^-inf = 0 exactly
      acc = 0;
      for (int j = 0; j * NC < nvec_all; ++j) {
        const int g = tid + j * NC;
        const bool have = g < nvec_all;
        unsigned long long q = 0;
        if (have) {
          float zt[8], w[8];
          row8<T>(gt, 8 * g, nv, aligned, zt);
          q = qfix(weights8<BONUS>(zt, zt, 8 * g, W, w));
        }
        acc += q;
        const unsigned long long gq = group8_sum_u64(q);
        if ((lane & 7) == 0 && have) gmass[g >> 3] = gq;
      }
    }
    const unsigned long long Wc = block_sum_u64(acc, S);
    if (tid == 0) {
      S.rec.w = Wc;
      S.rec.flags = late ? XF_ABORT : 0u;
    }
    cbar();
    if (!exchange(S, X, xbar, xround, rank, C, 6, 1)) late = true;
    const Xchg* XX = X[(xround - 1) & 1u];
    Wtot = 0;
    for (uint32_t c = 0; c < C; ++c) Wtot += XX[c].w;
    if (tid == 0) {
      const unsigned long long t = scale_floor(S.hdr[S.cur].u[P.K], Wtot);
      unsigned long long pre = 0;
      int cs = -1;
      for (uint32_t c = 0; c < C; ++c) {
        if (cs < 0 && t < pre + XX[c].w) {
          cs = static_cast<int>(c);
          S.t_loc = t - pre;
        }
        pre += XX[c].w;
      }
      S.cstar = cs;
      S.token = -1;
    }
    late = cbar_or(late);
    if (late || Wtot > 0 || BONUS) break;
  }
  if (!late && S.cstar == static_cast<int>(rank)) {
    // contiguous runs of groups per thread, so the prefix follows ascending ids
    const int ngroup = (nvec_all + 7) >> 3;
    const int lo = static_cast<int>((static_cast<long long>(tid) * ngroup) / NC);
    const int hi = static_cast<int>((static_cast<long long>(tid + 1) * ngroup) / NC);
    unsigned long long csum = 0;
    for (int gr = lo; gr < hi; ++gr) csum += gmass[gr];
    unsigned long long pre = block_exclusive_u64(csum, S);
    const unsigned long long tl = S.t_loc;
    if (pre <= tl && tl < pre + csum) {
      int gr = lo;
      while (gr < hi - 1 && pre + gmass[gr] <= tl) pre += gmass[gr++];
      // the group's vectors again, with the arithmetic and truncation of the stream above
      int g = gr * 8;
      const int gend = min(g + 8, nvec_all);
      for (; g < gend; ++g) {
        float zt[8], zd[8], w[8];
        row8<T>(gt, 8 * g, nv, aligned, zt);
        if (!BONUS && W.rho != 0.f) row8<T>(gd, 8 * g, nv, aligned, zd);
        else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) zd[kk] = zt[kk];
        }
        const unsigned long long q = qfix(weights8<BONUS>(zt, zd, 8 * g, W, w));
        if (pre + q > tl || g == gend - 1) {
          float s = 0.f;
          int pick = 7;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            s = kk ? __fadd_rn(s, w[kk]) : w[0];
            if (pre + qfix(s) > tl) {
              pick = kk;
              break;
            }
          }
          S.token = v0 + 8 * g + pick;
          break;
        }
        pre += q;
      }
    }
    cbar();
    if (tid == 0) P.out_tok[static_cast<long long>(seq) * (P.K + 1) + a] = S.token;
  }
  cbar();
}

// ------------------------------------------------------------------------------------------
// combine the C partials of a position (consumer warp 0); results land in S
// ------------------------------------------------------------------------------------------
template <bool GREEDY>
__device__ void combine(const Params& P, CtaState& S, const Xchg* XX, uint32_t C, int i,
                        bool st_t, bool st_d, bool tk, bool ld_d, float zx_t, float zx_d) {
  const int lane = threadIdx.x & 31;
  const bool have = lane < static_cast<int>(C);
  const float mt = have ? XX[lane].m_t : -INFINITY;
  const float md = have ? XX[lane].m_d : -INFINITY;
  const float Mt = warp_max_nan(mt);
  const float Md = warp_max_nan(md);
  if constexpr (GREEDY) {
    const int arg = (have && mt == Mt) ? XX[lane].arg : 0x7FFFFFFF;
    const int best = warp_min_int(arg);
    if (lane == 0) {
      S.M_t = Mt;
      S.bad_t = row_bad(Mt);
      S.arg = best;
    }
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
    const int L = S.hdr[S.cur].L;
    // the prepass's keys of this draft row stand in for the in-stream top 8
    const bool kk = P.keys != nullptr && st_d && i < L;
    if (kk)
#pragma unroll
      for (int j = 0; j < 8; ++j) mtop[j] = S.hdr[S.cur].key[i][j];
    S.M_t = Mt;
    S.M_d = Md;
    S.S_t = St;
    S.S_d = Sd;
    S.bad_t = row_bad(Mt);
    S.bad_d = ld_d ? row_bad(Md) : 0;
    float N = 1.f;  // Saguaro bias set: the bias_k most likely draft ids
    int nS = 0;
    if (P.bias_k > 0 && (tk || kk) && !S.bad_d) {
      float sq = 0.f;
      for (int j = 0; j < P.bias_k; ++j) {
        if (mtop[j] == 0ull) break;
        sq += exp2f((key_value(mtop[j]) - Md) * c) / Sd;
        S.S_ids[nS++] = key_id(mtop[j]);
      }
      N = fmaf(-(1.f - P.beta), sq, 1.f);
    }
    S.nS = nS;
    S.N = N;
    if (tk && P.fmax > 0 && i < L) {
      for (int f = 0; f < 8; ++f)
        S.topf[i][f] = (f < P.fan[i] && mtop[f] != 0ull) ? key_id(mtop[f]) : -1;
    }
    if (P.debug_all) {
      if (st_t && !S.bad_t) S.lse_t[i] = Mt / P.temperature + logf(St);
      if (st_d && !S.bad_d) S.lse_d[i] = Md / P.temperature + logf(Sd);
    }
    S.accept = 0;
    if (st_t && st_d && i < L && !S.bad_t && !S.bad_d) {
      const int x = S.hdr[S.cur].x[i];
      bool inS = false;
      for (int j = 0; j < nS; ++j) inS |= (S.S_ids[j] == x);
      const float f = inS ? P.beta : 1.f;
      float ratio;
      if (zx_t == -INFINITY) ratio = 0.f;
      else if (zx_d == -INFINITY) ratio = INFINITY;
      else ratio = exp2f(((zx_t - zx_d) - (Mt - Md)) * c) * (Sd / St) * (N / f);
      if (P.debug_all) {
        S.px[i] = zx_t == -INFINITY ? 0.f : exp2f((zx_t - Mt) * c) / St;
        S.qx[i] = zx_d == -INFINITY ? 0.f : exp2f((zx_d - Md) * c) * f / (Sd * N);
      }
      S.accept = S.hdr[S.cur].u[i] < ratio;
    }
  }
}

// Header of sequence `seq` into hdr[slot] with 4-byte async copies (consumer thread 0).
__device__ __forceinline__ void fetch_header(const Params& P, CtaState& S, int slot, int seq,
                                             bool greedy) {
  Hdr& h = S.hdr[slot];
  if (P.lens) cp_async4(&h.L, P.lens + seq);
  else h.L = P.K;
  for (int i = 0; i < P.K; ++i) cp_async4(&h.x[i], P.tokens + static_cast<long long>(seq) * P.K + i);
  if (P.keys)
    for (int i = 0; i < P.K; ++i)
      for (int j = 0; j < 8; j += 2)
        cp_async16(&h.key[i][j], P.keys + (static_cast<long long>(seq) * P.K + i) * 8 + j);
  if (!greedy)
    for (int i = 0; i <= P.K; ++i)
      cp_async4(&h.u[i], P.uni + static_cast<long long>(seq) * (P.K + 1) + i);
  cp_async_commit();
}

__device__ __forceinline__ int header_ok(const Params& P, const Hdr& h, bool greedy) {
  const int L = h.L;
  if (L < 1 || L > P.K) return 0;
  for (int i = 0; i < L; ++i)
    if (h.x[i] < 0 || h.x[i] >= P.V) return 0;
  if (!greedy)
    for (int i = 0; i <= P.K; ++i)
      if ((i < L || i == P.K) && !(h.u[i] >= 0.f && h.u[i] < 1.f)) return 0;
  // with top-F ids, every draft row below L must hold a distribution (the prepass marks one that
  // does not with the key ~0)
  if (P.keys && P.fmax > 0)
    for (int i = 0; i < L; ++i)
      if (h.key[i][0] == ~0ull) return 0;
  return 1;
}

// ------------------------------------------------------------------------------------------
// decisions taken while the next position streams
// ------------------------------------------------------------------------------------------
// One staged chunk of a stats position: the target row (and, when `two`, the draft row) into
// this thread's running statistics; whole chunks without per-vector bounds.
template <typename T, bool GREEDY>
__device__ __forceinline__ void stats_chunk(const Ring<T, GREEDY>& R, int s, int k, bool two,
                                            RowAcc& at, RowAcc& ad, int& garg, float c) {
  using RingT = Ring<T, GREEDY>;
  constexpr int VPT = RingT::CH / 8 / NC;
  const int n = R.chunk_len(k);
  const bool whole = n == RingT::CH;
  const int nvec = (n + 7) >> 3;
  ChunkRow<T, VPT> ct;
  if (whole) ct.load_full(R.row(s, 0));
  else ct.load(R.row(s, 0), nvec);
  const float vm = ct.vmax();
  if constexpr (GREEDY) {
    if (isnan(vm)) {
      at.m = NAN;
    } else if (vm > at.m) {  // first index of the new maximum in this thread's elements
      at.m = vm;
      int e = 0x7FFFFFFF;
#pragma unroll
      for (int j = VPT - 1; j >= 0; --j) {
        float z[8];
        ct.get(j, z);
#pragma unroll
        for (int kk = 7; kk >= 0; --kk)
          if (z[kk] == vm) e = 8 * (static_cast<int>(threadIdx.x) + j * NC) + kk;
      }
      garg = R.v0 + k * RingT::CH + e;
    }
  } else {
    at.rescale(vm, c);
    if (at.m > -INFINITY) {
#pragma unroll
      for (int j = 0; j < VPT; ++j) {
        float z[8];
        ct.get(j, z);
        at.sum8(z, c);
      }
    }
    if (two) {
      ChunkRow<T, VPT> cd;
      if (whole) cd.load_full(R.row(s, 1));
      else cd.load(R.row(s, 1), nvec);
      ad.rescale(cd.vmax(), c);
      if (ad.m > -INFINITY) {
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
          float z[8];
          cd.get(j, z);
          ad.sum8(z, c);
        }
      }
    }
  }
}

// Consumer warp 0: wait for exchange round r (posted for position `pos`), combine it and take
// the decision into S.dec; on a stop or an unusable row tell the producer, which then stops
// streaming the positions after it. The round of position 0 also names the next sequence.
__device__ int lpt_seq(const Params& P, const int* cnt, int r);

// A 64-bit store into the shared memory of a CTA of the cluster (a mapped address).
__device__ __forceinline__ void st_cluster_u64(uint32_t addr, unsigned long long v) {
  asm volatile("st.relaxed.cluster.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

template <bool GREEDY>
__device__ void resolve_open(const Params& P, CtaState& S, Xchg (*X)[kMaxCluster],
                             uint64_t* xbar, uint32_t r, uint32_t C, uint32_t rank,
                             const int* lcnt, int seq, int ep, int pos, int L, float zx_t,
                             float zx_d) {
  const int lane = threadIdx.x & 31;
  const bool ok = mbar_wait_cluster_bounded(&xbar[r & 1u], (r >> 1) & 1u, kWaitBudget);
  const Xchg* XX = X[r & 1u];
  bool ab = !ok;
  if (ok)
    for (uint32_t cc = 0; cc < C; ++cc) ab |= (XX[cc].flags & XF_ABORT) != 0u;
  ab = __any_sync(FULL, ab);
  int stop = -3;
  if (!ab) {
    const bool st_d = !GREEDY && pos < L;
    combine<GREEDY>(P, S, XX, C, pos, true, st_d, false, st_d, zx_t, zx_d);
    __syncwarp();
    if (S.bad_t || (st_d && S.bad_d)) stop = -2;
    else if (GREEDY) stop = (pos < L && S.hdr[S.cur].x[pos] == S.arg) ? -1 : pos;
    else stop = (pos == L || !S.accept) ? pos : -1;
  }
  if (lane == 0) {
    S.dec = stop;
    if (stop != -1 && stop != -3) {
      __threadfence_block();  // S before the word the producer acts on
      pub_store(&S.pub_cur, pack_cur(seq, ep, stop, 0));
    }
  }
  // the sequence is decided: rank 0 takes the cluster's next sequence from the queue now (not
  // when this one started), so a cluster that drew a long outcome does not hold a second
  // sequence back, and tells every CTA of the cluster
  if (rank == 0 && stop != -1 && stop != -3) {
    int q = 0;
    if (lane == 0) q = static_cast<int>(atomicAdd(&P.ws->next, 1u));
    q = __shfl_sync(FULL, q, 0);
    const int nxt = lpt_seq(P, lcnt, q + P.n_clusters);
    if (lane < static_cast<int>(C)) {
      const unsigned long long w =
          (static_cast<unsigned long long>(static_cast<uint32_t>(ep + 1)) << 32) |
          static_cast<uint32_t>(nxt);
      st_cluster_u64(map_to_rank(smem_u32(&S.nxt_word), static_cast<uint32_t>(lane)), w);
    }
  }
  __syncwarp();
}

// The next sequence stored by rank 0 for epoch `ep` (bounded wait; P.B after a timeout, with the
// error word raised).
__device__ __forceinline__ int wait_next_word(const Params& P, CtaState& S, int ep) {
  const unsigned long long want = static_cast<unsigned long long>(static_cast<uint32_t>(ep + 1));
  const long long t0 = clock64();
  while (true) {
    const unsigned long long w = *reinterpret_cast<volatile unsigned long long*>(&S.nxt_word);
    if ((w >> 32) == want) return static_cast<int>(static_cast<uint32_t>(w));
    if (clock64() - t0 > kWaitBudget) {
      atomicOr(&P.ws->error, 1u);
      return P.B;
    }
    sleep_ns(64);
  }
}

// ------------------------------------------------------------------------------------------
// longest-draft-first order of the sequences (built once per launch by one CTA)
// ------------------------------------------------------------------------------------------
// Longest draft first: place r of the order is the sequence with the r-th largest draft length,
// ties in index order, unusable lengths last. Every CTA counts the lengths per bucket once
// (bucket K - L for L in 1..K, bucket K for the rest); a place is then found by one warp.
__device__ __forceinline__ int lpt_bucket(const Params& P, int b) {
  const int L = P.lens ? P.lens[b] : P.K;
  return (L >= 1 && L <= P.K) ? P.K - L : P.K;
}

// Sequence at place r (P.B when r >= P.B); all 32 lanes of one warp call it.
__device__ int lpt_seq(const Params& P, const int* cnt, int r) {
  const int lane = threadIdx.x & 31;
  if (r >= P.B) return P.B;
  if (!P.lpt) return r;
  int bk = 0, start = 0;
  while (bk < P.K && start + cnt[bk] <= r) {
    start += cnt[bk];
    ++bk;
  }
  const int want = r - start;  // rank inside bucket bk
  const int per = (P.B + 31) / 32;
  const int lo = min(P.B, lane * per), hi = min(P.B, lo + per);
  int n = 0;
  for (int b = lo; b < hi; ++b) n += lpt_bucket(P, b) == bk;
  int incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += y;
  }
  int found = 0x7FFFFFFF;
  if (want >= incl - n && want < incl) {
    int q = want - (incl - n);
    for (int b = lo; b < hi; ++b)
      if (lpt_bucket(P, b) == bk) {
        if (q == 0) {
          found = b;
          break;
        }
        --q;
      }
  }
  found = warp_min_int(found);
  return found == 0x7FFFFFFF ? P.B : found;
}

// ------------------------------------------------------------------------------------------
// the kernel: consumer warps 0..7 verify, warp 8 produces
// ------------------------------------------------------------------------------------------
template <typename T, bool GREEDY, bool TOP8>
__global__ void __launch_bounds__(NTOT, 3) verify_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ CtaState S;
  __shared__ Xchg X[2][kMaxCluster];
  __shared__ uint64_t full_bar[NS], empty_bar[NS], xbar[2];
  __shared__ unsigned long long sdesc[NS];
  __shared__ int lcnt[kMaxK + 1];

  // with deferred draws, let the draw launches start (their CTAs wait per sequence)
  if (P.defer) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  using RingT = Ring<T, GREEDY>;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const uint32_t C = cluster_nctarank();
  const int cid = static_cast<int>(cluster_id_x());
  const int K = P.K;
  RingT R;
  R.base = dyn;
  R.full = full_bar;
  R.empty = empty_bar;
  R.desc = sdesc;
  R.v0 = static_cast<int>(rank) * P.slice;
  R.nv = max(0, min(P.V - R.v0, P.slice));
  R.nchunk = (R.nv + RingT::CH - 1) / RingT::CH;
  R.scr = P.scratch ? static_cast<T*>(P.scratch) +
                          static_cast<size_t>(cid * static_cast<int>(C) + static_cast<int>(rank)) * 2 *
                              P.slice
                    : nullptr;
  unsigned long long* gmass = reinterpret_cast<unsigned long long*>(
      dyn + static_cast<size_t>(NS) * RingT::kRows * kStageRowBytes);
  const float c = P.c;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], NW);
    }
    mbar_init(&xbar[0], 1);
    mbar_init(&xbar[1], 1);
    fence_mbar_init();
    S.cur = 0;
    S.n_hdr_wait = 0;
    S.cons_final = 0;
    S.nxt_word = 0ull;
  }
  // the draft-length counts of the longest-first order (every CTA its own copy)
  if (P.lpt) {
    if (tid <= kMaxK) lcnt[tid] = 0;
    __syncthreads();
    for (int b = tid; b < P.B; b += NTOT) atomicAdd(&lcnt[lpt_bucket(P, b)], 1);
    __syncthreads();
  }
  int seq0 = 0;
  if (warp == 0) seq0 = lpt_seq(P, lcnt, cid);
  if (tid == 0) {
    S.seq0 = seq0;
    fetch_header(P, S, 0, seq0, GREEDY);
    cp_async_wait_all();
    S.hdr[0].ok = header_ok(P, S.hdr[0], GREEDY);
    pub_store(&S.pub_cur, pack_cur(seq0, 0, S.hdr[0].ok ? -1 : -2, 0));
    pub_store(&S.pub_next, 0ull);
  }
  __syncthreads();
  cluster_sync();  // every CTA of the cluster is running before any shared-memory exchange

  if (warp == NW) {
    if ((tid & 31) == 0) producer<T, GREEDY>(P, S, R);
    __syncwarp();
  } else {
    uint32_t xround = 0;
    Cursor cons;
    bool late = false;
    bool aborted = false;
    int seq = S.seq0;
    int ep = 0;
    while (seq < P.B) {
      cons.ep = ep;
      int next_local = 0;
      const bool ahead = !TOP8 && !P.debug_all && S.hdr[S.cur].ok && P.use_bulk;
      if (!ahead && rank == 0 && warp == 0) {  // the next sequence, named in the first exchange
        int q = 0;
        if (tid == 0) q = static_cast<int>(atomicAdd(&P.ws->next, 1u));
        q = __shfl_sync(FULL, q, 0);
        next_local = lpt_seq(P, lcnt, q + P.n_clusters);
      }
      if (tid == 0 && P.fmax + P.debug_all > 0) {
        for (int i = 0; i < kMaxK; ++i) {
          for (int f = 0; f < 8; ++f) S.topf[i][f] = -1;
          S.lse_d[i] = S.px[i] = S.qx[i] = NAN;
        }
        for (int i = 0; i <= kMaxK; ++i) S.lse_t[i] = NAN;
      }
      const int L = S.hdr[S.cur].L;
      bool invalid = !S.hdr[S.cur].ok;
      bool decided = invalid;
      bool first = true;
      int a = -1;
      int next = P.B;
      if (ahead) {
        // ---- decisions taken while the next position streams: position i is read while
        // consumer warp 0 combines the round of position i - 1 (polled between chunks, else
        // waited for at the end of position i); a stop makes the producer switch to the draw,
        // which cuts position i short in every consumer at the same stage ----
        int pend = -1;             // position whose round is posted but not yet combined
        uint32_t pend_round = 0;
        bool resolved = true;      // warp 0's view
        float pzx_t = 0.f, pzx_d = 0.f;
        int outcome = -3;
        for (int i = 0;; ++i) {
          const bool two = !GREEDY && i < L;
          float zx_t = 0.f, zx_d = 0.f;
          if (!GREEDY && tid == 0 && i < L) {
            const int x = S.hdr[S.cur].x[i];
            zx_t = Elt<T>::val(static_cast<const T*>(row_ptr(P, false, seq, i, sizeof(T)))[x]);
            zx_d = Elt<T>::val(static_cast<const T*>(row_ptr(P, true, seq, i, sizeof(T)))[x]);
          }
          RowAcc at, ad;
          at.init();
          ad.init();
          int garg = 0x7FFFFFFF;
          bool cut = false;
          for (int k = 0; k < R.nchunk; ++k) {
            if (warp == 0 && !resolved) {
              const int ready = __shfl_sync(
                  FULL, tid == 0 ? static_cast<int>(mbar_test_cluster(&xbar[pend_round & 1u], (pend_round >> 1) & 1u)) : 0, 0);
              if (ready) {
                resolve_open<GREEDY>(P, S, X, xbar, pend_round, C, rank, lcnt, seq, ep, pend, L, pzx_t, pzx_d);
                resolved = true;
              }
            }
            const int s = acquire_open<T, GREEDY>(R, seq, i, k, cons, late);
            if (s == -2) {
              cut = true;
              break;
            }
            if (s < 0) break;
            stats_chunk<T, GREEDY>(R, s, k, two, at, ad, garg, c);
            release_stage(R.empty, cons);
          }
          late = cbar_or(late);
          if (late) break;
          if (cut) {  // the producer acted on a stop of `pend`; warp 0 holds the decision
            outcome = *reinterpret_cast<volatile int*>(&S.dec);
            break;
          }
          // this CTA's partials of position i
          const float2 mm = block_max2(at.m, ad.m, S);
          float2 ss = make_float2(0.f, 0.f);
          int arg = 0x7FFFFFFF;
          if constexpr (GREEDY) {
            if (!row_bad(mm.x)) arg = block_min_int(at.m == mm.x ? garg : 0x7FFFFFFF, S);
          } else {
            const bool sum_t = !row_bad(mm.x);
            const bool sum_d = two && !row_bad(mm.y);
            const float mct = __fmul_rn(mm.x, c), mcd = __fmul_rn(mm.y, c);
            const float pt = (sum_t && at.m > -INFINITY) ? at.total() * exp2f(at.mc - mct) : 0.f;
            const float pd = (sum_d && ad.m > -INFINITY) ? ad.total() * exp2f(ad.mc - mcd) : 0.f;
            ss = block_sum2(pt, pd, S);
            if (sum_t) ss.x *= fmaf(-fmaf(mm.x, c, -mct), kLn2, 1.f);
            if (sum_d) ss.y *= fmaf(-fmaf(mm.y, c, -mcd), kLn2, 1.f);
          }
          // the previous position's decision, at the latest now
          if (warp == 0 && !resolved) {
            resolve_open<GREEDY>(P, S, X, xbar, pend_round, C, rank, lcnt, seq, ep, pend, L, pzx_t, pzx_d);
            resolved = true;
          }
          cbar();
          if (pend >= 0 && S.dec != -1) {  // position i is not needed
            outcome = S.dec;
            break;
          }
          if (tid == 0) {
            S.rec.m_t = mm.x;
            S.rec.s_t = ss.x;
            S.rec.m_d = mm.y;
            S.rec.s_d = ss.y;
            S.rec.arg = arg;
            S.rec.next_seq = i == 0 ? next_local : 0;
            S.rec.flags = 0u;
          }
          cbar();
          pend_round = xround;
          exchange_post(S, X, xbar, xround, rank, C, 0, 2);
          pend = i;
          resolved = false;
          pzx_t = zx_t;
          pzx_d = zx_d;
          if (i == L) {  // nothing after this position: its decision now
            if (warp == 0) {
              resolve_open<GREEDY>(P, S, X, xbar, pend_round, C, rank, lcnt, seq, ep, pend, L, pzx_t, pzx_d);
              resolved = true;
            }
            cbar();
            outcome = S.dec;
            break;
          }
        }
        cbar();
        next = P.B;
        if (late || outcome == -3 || outcome == -1) {
          aborted = true;
        } else if (outcome == -2) {
          invalid = true;
          decided = true;
        } else {
          decided = true;
          a = outcome;
          if (!GREEDY && !P.defer) {
            if (a < L)
              draw_token<T, GREEDY, false>(P, S, X, xbar, xround, rank, C, R, seq, a, gmass, cons, late);
            else
              draw_token<T, GREEDY, true>(P, S, X, xbar, xround, rank, C, R, seq, a, gmass, cons, late);
            if (late) aborted = true;
          }
        }
      } else
      for (int i = 0;; ++i) {
        const bool st_t = !invalid && i <= L && (!decided || P.debug_all);
        const bool st_d = !GREEDY && !invalid && i < L && (!decided || P.debug_all);
        const bool tk = TOP8 && !invalid && i < L && (!decided || P.fmax > 0 || P.debug_all);
        const bool ld_t = st_t, ld_d = st_d || tk;
        if (!ld_t && !ld_d && !first) break;
        // the draft token's logits for the accept test (thread 0; used after the exchange)
        float zx_t = 0.f, zx_d = 0.f;
        if (!GREEDY && tid == 0 && st_t && st_d && i < L) {
          const int x = S.hdr[S.cur].x[i];
          zx_t = Elt<T>::val(static_cast<const T*>(row_ptr(P, false, seq, i, sizeof(T)))[x]);
          zx_d = Elt<T>::val(static_cast<const T*>(row_ptr(P, true, seq, i, sizeof(T)))[x]);
        }
        // ---- stream this CTA's slice of the position's rows ----
        RowAcc at, ad;
        at.init();
        ad.init();
        int garg = 0x7FFFFFFF;
        unsigned long long keys[8];
        float thr = -INFINITY;
        if (TOP8) {
#pragma unroll
          for (int j = 0; j < 8; ++j) keys[j] = 0ull;
        }
        if (ld_t || ld_d) {
          int k = 0;
          if constexpr (!GREEDY) {
            if (P.use_bulk && st_t && !tk && st_d == ld_d) {  // the common case: whole chunks first
              const int kf = R.nv / RingT::CH;
              k = st_d ? stream_whole<T, true>(R, seq, i, kf, cons, late, at, ad, c)
                       : stream_whole<T, false>(R, seq, i, kf, cons, late, at, ad, c);
            }
          }
          for (; k < R.nchunk; ++k) {
            int s = acquire<T, GREEDY>(R, seq, i, k, cons, late);
            if (!P.use_bulk) s = fill_unaligned<T, GREEDY>(P, R, s, seq, i, k, late);
            if (s < 0) break;
            const int n = R.chunk_len(k);
            const int nvec = (n + 7) >> 3;
            constexpr int VPT = RingT::CH / 8 / NC;
            static_assert(VPT >= 1 && RingT::CH == VPT * 8 * NC, "whole vectors per thread");
            if (ld_t) {
              ChunkRow<T, VPT> cr;
              cr.load(R.row(s, 0), nvec);
              const float vm = cr.vmax();
              if constexpr (GREEDY) {
                if (isnan(vm)) {
                  at.m = NAN;
                } else if (vm > at.m) {  // first index of the new maximum in this thread's elements
                  at.m = vm;
                  int e = 0x7FFFFFFF;
#pragma unroll
                  for (int j = VPT - 1; j >= 0; --j) {
                    float z[8];
                    cr.get(j, z);
#pragma unroll
                    for (int kk = 7; kk >= 0; --kk)
                      if (z[kk] == vm) e = 8 * (tid + j * NC) + kk;
                  }
                  garg = R.v0 + k * RingT::CH + e;
                }
              } else {
                at.rescale(vm, c);
                if (at.m > -INFINITY) {
#pragma unroll
                  for (int j = 0; j < VPT; ++j) {
                    float z[8];
                    cr.get(j, z);
                    at.sum8(z, c);
                  }
                }
              }
            }
            if (!GREEDY && ld_d) {
              ChunkRow<T, VPT> cr;
              cr.load(R.row(s, 1), nvec);
              const float vm = cr.vmax();
              if (st_d) {
                ad.rescale(vm, c);
                if (ad.m > -INFINITY) {
#pragma unroll
                  for (int j = 0; j < VPT; ++j) {
                    float z[8];
                    cr.get(j, z);
                    ad.sum8(z, c);
                  }
                }
              } else {
                ad.m = max_nan(ad.m, vm);
              }
              if (TOP8 && tk) {
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                  float z[8];
                  cr.get(j, z);
                  const int eb = 8 * (tid + j * NC);
#pragma unroll
                  for (int kk = 0; kk < 8; ++kk)
                    if (eb + kk < n)
                      top8_insert(keys, thr, z[kk],
                                  static_cast<uint32_t>(R.v0 + k * RingT::CH + eb + kk));
                }
              }
            }
            release_stage(R.empty, cons);
          }
        }
        // ---- this CTA's partials ----
        late = cbar_or(late);
        const float2 mm = block_max2(at.m, ad.m, S);
        float2 ss = make_float2(0.f, 0.f);
        int arg = 0x7FFFFFFF;
        if constexpr (GREEDY) {
          if (ld_t && !row_bad(mm.x)) arg = block_min_int(at.m == mm.x ? garg : 0x7FFFFFFF, S);
        } else {
          const bool sum_t = st_t && !row_bad(mm.x);
          const bool sum_d = st_d && !row_bad(mm.y);
          const float mct = __fmul_rn(mm.x, c), mcd = __fmul_rn(mm.y, c);
          const float pt = (sum_t && at.m > -INFINITY) ? at.total() * exp2f(at.mc - mct) : 0.f;
          const float pd = (sum_d && ad.m > -INFINITY) ? ad.total() * exp2f(ad.mc - mcd) : 0.f;
          ss = block_sum2(pt, pd, S);
          // the sums are relative to m*c rounded; fold the rounding back in
          if (sum_t) ss.x *= fmaf(-fmaf(mm.x, c, -mct), kLn2, 1.f);
          if (sum_d) ss.y *= fmaf(-fmaf(mm.y, c, -mcd), kLn2, 1.f);
          if (TOP8 && tk) block_top8(keys, S);
        }
        if (tid == 0) {
          S.rec.m_t = mm.x;
          S.rec.s_t = ss.x;
          S.rec.m_d = mm.y;
          S.rec.s_d = ss.y;
          S.rec.arg = arg;
          S.rec.next_seq = first ? next_local : 0;
          S.rec.flags = late ? XF_ABORT : 0u;
          if (TOP8 && tk && !(ld_t || ld_d))
            for (int r = 0; r < 8; ++r) S.rec.top8[r] = 0ull;
        }
        cbar();
        if (!exchange(S, X, xbar, xround, rank, C, 0, (TOP8 && tk) ? 6 : 2)) late = true;
        const Xchg* XX = X[(xround - 1) & 1u];
        bool ab = late;
        for (uint32_t cc = 0; cc < C; ++cc) ab |= (XX[cc].flags & XF_ABORT) != 0u;
        ab = cbar_or(ab);  // the same answer in every consumer thread
        if (ab) {
          aborted = true;
          break;
        }
        if (first) {
          next = XX[0].next_seq;
          first = false;
          if (tid == 0) {  // start fetching the next sequence's header; tell the producer
            if (next < P.B) {
              fetch_header(P, S, S.cur ^ 1, next, GREEDY);
              S.n_hdr_wait = 1;
            }
            pub_store(&S.pub_next, pack_next(next, ep));
          }
        }
        if (!ld_t && !ld_d) break;  // header was invalid: the exchange only carried `next`
        if (warp == 0) combine<GREEDY>(P, S, XX, C, i, st_t, st_d, tk, ld_d, zx_t, zx_d);
        cbar();
        if (!decided) {
          int stop = -1;
          if (S.bad_t || (i < L && !GREEDY && S.bad_d)) {
            invalid = true;
            stop = -2;
          } else if constexpr (GREEDY) {
            if (!(i < L && S.hdr[S.cur].x[i] == S.arg)) stop = i;
          } else {
            if (i == L || !S.accept) stop = i;
          }
          if (stop != -1) {
            decided = true;
            a = stop;
            if (tid == 0) pub_store(&S.pub_cur, pack_cur(seq, ep, stop, 0));
          }
          if (invalid) break;
          if (!GREEDY && stop >= 0) {
            if (stop < L)
              draw_token<T, GREEDY, false>(P, S, X, xbar, xround, rank, C, R, seq, a, gmass, cons, late);
            else
              draw_token<T, GREEDY, true>(P, S, X, xbar, xround, rank, C, R, seq, a, gmass, cons, late);
            if (late) {
              aborted = true;
              break;
            }
          }
        } else if (tk && P.fmax > 0 && S.bad_d) {
          invalid = true;  // a draft row the top-F output needs holds no distribution
          if (tid == 0) pub_store(&S.pub_cur, pack_cur(seq, ep, -2, 0));
          break;
        }
      }
      // ---- epilogue: rank 0 writes the outputs of this sequence ----
      if (rank == 0) {
        int32_t* tok = P.out_tok + static_cast<long long>(seq) * (K + 1);
        const bool bad = aborted || invalid;
        if (tid == 0) P.out_acc[seq] = aborted ? -2 : (invalid ? -1 : a);
        for (int j = tid; j <= K; j += NC) {
          if (bad || j > a) tok[j] = -1;
          else if (j < a) tok[j] = S.hdr[S.cur].x[j];
          else if (GREEDY) tok[j] = S.arg;
        }
        if (P.fmax > 0) {
          int32_t* tf = P.out_topf + static_cast<long long>(seq) * K * P.fmax;
          for (int e = tid; e < K * P.fmax; e += NC) {
            const int i = e / P.fmax, f = e % P.fmax;
            if (P.keys) {  // the prepass wrote the ids of the rows below L
              if (bad || i >= L) tf[e] = -1;
            } else {
              tf[e] = (!bad && i < L && f < 8) ? S.topf[i][f] : -1;
            }
          }
        }
        if (!GREEDY && P.defer && tid == 0) {
          // the draw's constants for the deferred draw launches (the same as draw_token's),
          // then the sequence's place in the order they read
          SmallDecision d;
          d.ok = bad ? 0 : 1;
          d.a = aborted ? -2 : (invalid ? -1 : a);
          d.mct = __fmul_rn(S.M_t, P.c);
          d.mcd = 0.f;
          d.rho = d.rho_s = 0.f;
          d.nS = 0;
#pragma unroll
          for (int j = 0; j < 8; ++j) d.ids[j] = -1;
          if (!bad && a < L) {  // a residual draw; at a == L the bonus draw from p_L
            d.mcd = __fmul_rn(S.M_d, P.c);
            const float ft = fmaf(-fmaf(S.M_t, P.c, -d.mct), kLn2, 1.f);
            const float fd = fmaf(-fmaf(S.M_d, P.c, -d.mcd), kLn2, 1.f);
            d.rho = (fd * S.S_t) / (ft * (S.S_d * S.N));
            d.rho_s = d.rho * P.beta;
          }
          const int q = static_cast<int>(atomicAdd(&P.ws->dcount, 1u));
          d.q = q;
          static_cast<SmallDecision*>(P.ddec)[seq] = d;
          __threadfence();
          st_release_gpu_s32(P.dlist + q, seq + 1);
        }
        if (P.dbg_lse_t && tid <= K)
          P.dbg_lse_t[static_cast<long long>(seq) * (K + 1) + tid] = S.lse_t[tid];
        if (tid < K) {
          const long long o = static_cast<long long>(seq) * K + tid;
          if (P.dbg_lse_d) P.dbg_lse_d[o] = S.lse_d[tid];
          if (P.dbg_px) P.dbg_px[o] = S.px[tid];
          if (P.dbg_qx) P.dbg_qx[o] = S.qx[tid];
        }
      }
      cbar();
      if (aborted) {
        if (tid == 0) atomicOr(&P.ws->error, 1u);
        break;
      }
      // ---- move on to the next sequence of the queue ----
      if (tid == 0) {
        int nxs = next;
        if (ahead) {  // rank 0 stored it when this sequence was decided
          nxs = wait_next_word(P, S, ep);
          if (nxs < P.B) {
            fetch_header(P, S, S.cur ^ 1, nxs, GREEDY);
            S.n_hdr_wait = 1;
          }
        }
        S.next = nxs;
        if (S.n_hdr_wait) {
          cp_async_wait_all();
          S.n_hdr_wait = 0;
        }
        const int nx = S.cur ^ 1;
        if (nxs < P.B) S.hdr[nx].ok = header_ok(P, S.hdr[nx], GREEDY);
        S.cur = nx;
        pub_store(&S.pub_cur, pack_cur(nxs, ep + 1, (nxs < P.B && S.hdr[nx].ok) ? -1 : -2, 0));
      }
      cbar();
      seq = S.next;
      ++ep;
    }
    if (tid == 0) {
      cp_async_wait_all();
      *reinterpret_cast<volatile int*>(&S.cons_final) = cons.n;
      __threadfence_block();
      const Pub v = unpack_cur(pub_load(&S.pub_cur));
      pub_store(&S.pub_cur, pack_cur(v.seq, v.ep, v.stop, 1));
    }
  }
  __syncthreads();
  cluster_sync();
  if (rank == 0 && tid == 0) {
    __threadfence();
    const unsigned old = atomicAdd(&P.ws->done, 1u);
    if (old == static_cast<unsigned>(P.n_clusters) - 1u) {
      atomicExch(&P.ws->next, 0u);
      atomicExch(&P.ws->done, 0u);
      atomicExch(&P.ws->dcount, 0u);
    }
  }
}

template <typename T, bool GREEDY, bool TOP8>
const void* kernel_ptr() {
  return reinterpret_cast<const void*>(&verify_kernel<T, GREEDY, TOP8>);
}

const void* pick(int dtype, int greedy, int top8) {
  if (dtype == 1) {
    if (greedy) return kernel_ptr<uint16_t, true, false>();
    return top8 ? kernel_ptr<uint16_t, false, true>() : kernel_ptr<uint16_t, false, false>();
  }
  if (greedy) return kernel_ptr<float, true, false>();
  return top8 ? kernel_ptr<float, false, true>() : kernel_ptr<float, false, false>();
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
  (void)dtype;
  const size_t ring = static_cast<size_t>(NS) * (greedy ? 1 : 2) * kStageRowBytes;
  const size_t gmass = greedy ? 0 : (static_cast<size_t>(slice + 63) / 64 * 8 + 127) / 128 * 128;
  return ring + gmass;
}

int max_active_clusters(int dtype, int greedy, int top8, int cluster, size_t smem) {
  const void* fn = pick(dtype, greedy, top8);
  if (prepare(fn, cluster, smem) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cluster) * 64u);
  cfg.blockDim = dim3(NTOT);
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
  const void* fn = pick(L.dtype, L.greedy, L.p.top8);
  cudaError_t e = prepare(fn, L.cluster, L.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(L.p.n_clusters * L.cluster));
  cfg.blockDim = dim3(NTOT);
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

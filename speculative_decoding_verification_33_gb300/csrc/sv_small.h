// Interface between the host API (sv_api.cu) and the small-batch stochastic kernels
// (sv_small.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

// A sequence's decision, written by the draw's mass launch for its pick launch.
struct SmallDecision {
  int a;        // decided position, -1 for an invalid sequence
  int ok;       // 1 = valid
  float mct;    // fl(M_t c) of the target row at a
  float mcd;    // fl(M_d c) of the draft row at a (residual draws)
  float rho;    // q' scale / p scale off the bias set; 0 = draw from p
  float rho_s;  // the same on the bias set (rho * beta)
  int nS;       // ids in the bias set of the draft row at a
  int ids[8];   // those ids
  int q;        // deferred draws: the place of the sequence in the order list
};

struct SmallParams {
  const void* tgt;           // target logits [B][K+1][t_stride]
  const void* dft;           // draft logits [B][K][d_stride]
  long long t_stride, d_stride;
  const int32_t* lens;       // [B] draft lengths, or NULL (all K)
  const int32_t* tokens;     // [B][K] draft ids
  const float* uni;          // [B][K+1] uniforms
  int B, K, V;
  float c;                   // log2(e) / T
  int slice, nslice;         // row statistics: ids per CTA (multiple of 8), slices per row
  int slice_d, nslice_d;     // the draw: ids per CTA (multiple of 8), slices per row
  int aligned;               // rows 16-byte aligned: bulk copies and vector loads
  int top8;                  // 1: the draft rows' top 8 are kept (bias set or top-F ids)
  int bias_k;                // size of the bias set (0: none)
  float beta;                // its weight
  int fmax;                  // top-F ids per position, 0: none
  int fan[8];                // F_i of position i (at most 8)
  int32_t* out_topf;         // [B][K][fmax]: -1 where the sequence is invalid or i >= L
  float2* part;              // [B][2K+1][nslice] per slice (max, sum)
  unsigned long long* keys;  // [B][K][nslice][8] per slice of a draft row: its 8 largest keys
  SmallDecision* dec;        // [B]
  unsigned long long* mass;  // [B][nslice_d][2] the draw's residual and p masses per slice
  int* dlist;                // deferred draws: seq + 1 of the k-th sequence the walk decided
  unsigned int* err;         // error word: bit 0 = a bounded wait gave up
  int32_t* out_acc;          // [B]
  int32_t* out_tok;          // [B][K+1]
};

// Row-statistics CTAs resident per multiprocessor (occupancy of the kernel); dtype 1 = bf16.
int small_rows_per_sm(int dtype);

// Fills B, K and the slice fields of P for a batch of B sequences on `sms` multiprocessors;
// false when the problem does not fit this path (K > 8, or V above 32 draw slices of 8192 ids).
bool small_plan(int B, int K, int V, int sms, int rows_per_sm, SmallParams* P);

// Workspace bytes after the fixed header: partials, decisions, masses and, with top8 set, the
// slices' keys (each 256-byte aligned), and the pointers into it.
inline size_t small_align(size_t n) { return (n + 255) / 256 * 256; }
inline size_t small_keys_bytes(const SmallParams& P) {
  return P.top8 ? static_cast<size_t>(P.B) * P.K * P.nslice * 8 * 8 : 0;
}
// Device state of the deferred draws for batches of up to `cap` sequences: the order list first
// (it must read zero at the start of every call, so it stays where it is whatever the batch:
// the pick clears what the walk wrote), then the decisions and the masses of up to 32 draw
// slices per sequence (written before they are read in every call). Each part 256-byte aligned.
inline size_t walk_draw_ws_bytes(int cap) {
  return small_align(static_cast<size_t>(cap) * sizeof(int)) +
         small_align(static_cast<size_t>(cap) * sizeof(SmallDecision)) +
         small_align(static_cast<size_t>(cap) * 32 * 16);
}
inline void walk_draw_carve(SmallParams& P, char* base, int cap) {
  P.dlist = reinterpret_cast<int*>(base);
  base += small_align(static_cast<size_t>(cap) * sizeof(int));
  P.dec = reinterpret_cast<SmallDecision*>(base);
  base += small_align(static_cast<size_t>(cap) * sizeof(SmallDecision));
  P.mass = reinterpret_cast<unsigned long long*>(base);
}
inline size_t small_ws_bytes(const SmallParams& P) {
  return small_align(static_cast<size_t>(P.B) * (2 * P.K + 1) * P.nslice * 8) +
         small_align(static_cast<size_t>(P.B) * sizeof(SmallDecision)) +
         small_align(static_cast<size_t>(P.B) * P.nslice_d * 16) +
         small_align(small_keys_bytes(P));
}
inline void small_carve(SmallParams& P, char* base) {
  P.part = reinterpret_cast<float2*>(base);
  base += small_align(static_cast<size_t>(P.B) * (2 * P.K + 1) * P.nslice * 8);
  P.dec = reinterpret_cast<SmallDecision*>(base);
  base += small_align(static_cast<size_t>(P.B) * sizeof(SmallDecision));
  P.mass = reinterpret_cast<unsigned long long*>(base);
  base += small_align(static_cast<size_t>(P.B) * P.nslice_d * 16);
  P.keys = P.top8 ? reinterpret_cast<unsigned long long*>(base) : nullptr;
}

// The three launches (row slices; the draw's slice masses; one pick CTA per sequence) on
// `stream`, the last two chained by programmatic dependent launch; dtype 1 = bf16.
cudaError_t launch_small(const SmallParams& P, int dtype, cudaStream_t stream);

// The draws the walk deferred (P.dec and P.dlist written by the walk, P.mass and the slice
// fields as for launch_small): the slice masses of each sequence, its CTAs waiting (bounded)
// until the walk has decided it, then the pick; both chained by programmatic dependent launch
// after the walk on `stream`.
cudaError_t launch_walk_draws(const SmallParams& P, int dtype, cudaStream_t stream);

}  // namespace sv

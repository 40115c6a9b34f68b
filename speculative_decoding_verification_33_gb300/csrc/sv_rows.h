// Interface between the host API (sv_api.cu) and the row kernels (sv_rows.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sv_internal.h"

namespace sv {

constexpr int kRowChunkWarps = 8;      // warps reducing the streamed chunks
constexpr int kRowEpilogueWarps = 4;   // warps finishing units from their group values
constexpr int kRowThreads = (kRowChunkWarps + kRowEpilogueWarps + 1) * 32;  // + the producer
constexpr int kRowMaxStages = 8;       // ring stages per CTA (the launch picks 2 .. 8)
constexpr int kRowStageBytes = 16384;  // bytes per stage
constexpr size_t kRowMaxSmem = 227 * 1024;

struct RowParams {
  const void* tgt;
  const void* dft;
  long long t_stride, d_stride;  // elements between rows
  int V, K, B;                   // residual: B sequences of K positions; sampling: B rows
  const int32_t* lens;           // residual: draft lengths (NULL = K)
  const float* uni;              // sampling: one uniform per row
  float c;                       // log2(e) / T
  float beta;
  int bias_k;                    // 0 = no bias set
  int fmax;                      // residual: columns of out_r2
  int fan[kMaxK];
  int use_vec;                   // rows and strides 16-byte aligned: bulk copies
  int nstages;                   // ring stages (2 .. kRowMaxStages)
  float tau;                     // sampling: exit threshold for out_exit
  int32_t* out_tok;              // sampling
  float* out_conf;
  int32_t* out_exit;             // may be NULL
  int32_t* out_r2;               // residual
  int32_t* out_hit;              // may be NULL; else the verify outputs below give the flags
  const int32_t* acc;            // residual with out_hit: the verify step's [B] accept lengths,
  const int32_t* tok;            //   [B][K+1] tokens
  const int32_t* r1;             //   and [B][K][fmax] top-F ids
  unsigned long long* out_keys;  // top-8 prepass: 8 keys per (sequence, position)
  int32_t* out_topf;             // top-8 prepass: [B][K][fmax] top-F ids (may be NULL)
  Workspace* ws;                 // unit queue and error word (bit 0: a bounded wait gave up)
};

// Dynamic shared memory of one CTA: the ring and two buffers of per-group values (dtype 1 =
// bf16 rows, whose residual keeps 16-bit group values).
size_t row_smem_bytes(int mode, int dtype, int V, int nstages);
// Co-resident CTAs per SM of the kernel for this configuration (0: does not fit).
int row_ctas_per_sm(int mode, int dtype, bool bias, int V, int nstages);

// mode 0: sampling (B rows), 1: residual top-F, 2: top-8 prepass of the verify step's draft rows
// (both over B * K (sequence, position) pairs); `ctas` persistent CTAs. With out_hit set, the
// residual launch also writes the cache-hit flags.
cudaError_t launch_rows(const RowParams& P, int mode, int dtype, int ctas, cudaStream_t stream);

}  // namespace sv

// Interface between the host API (sv_api.cu) and the row kernels (sv_rows.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sv_internal.h"

namespace sv {

constexpr int kRowThreads = 256;  // threads per CTA of the row kernels

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
  int slice;                     // vocabulary entries per CTA (multiple of 8)
  int use_vec;                   // rows and strides 16-byte aligned: vector loads
  float tau;                     // sampling: exit threshold for out_exit
  int32_t* out_tok;              // sampling
  float* out_conf;
  int32_t* out_exit;             // may be NULL
  int32_t* out_r2;               // residual
  int32_t* out_hit;              // may be NULL
};

// mode 0: sampling (one cluster per row), 1: residual top-F (one cluster per (b, i) pair)
cudaError_t launch_rows(const RowParams& P, int mode, int dtype, int nclusters, int C,
                        const int32_t* acc, const int32_t* tok, const int32_t* r1,
                        cudaStream_t stream);

}  // namespace sv

// Interface between the host API (sv_api.cu) and the verify step taken from hidden states
// (sv_hverify.cu): the head GEMM's statistics, the decisions and the draw, with no logit row in
// HBM.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sv_lmhead.h"

namespace sv {

struct HvProblem {
  int B, K, V, d;
  int greedy;
  const uint16_t* ht;     // hidden states of the target rows, [B][K+1] rows of d (bf16)
  long long hts;          // elements between consecutive target rows
  const uint16_t* hd;     // hidden states of the early-exit draft rows, [B][K] rows (stochastic)
  long long hds;
  const uint16_t* W;      // head [V][d] (bf16)
  long long ws;           // elements between head rows
  const int32_t* x;       // [B][K] draft ids
  const int32_t* lens;    // [B] draft lengths
  const float* uni;       // [B][K+1] uniforms (stochastic)
  float temperature;
  float beta;             // weight of the Saguaro bias set (stochastic; 1 = none)
  int bias_k;             // its size, 0..8 (0 = none)
  int fmax;               // top-F ids per position (0 = none)
  int fan[8];             // F_i of position i
  int32_t* out_acc;       // [B]
  int32_t* out_tok;       // [B][K+1]
  int32_t* out_topf;      // [B][K][fmax] (fmax > 0)
};

// The draft rows' 8 largest logits are needed (a bias set or top-F ids).
__host__ __device__ inline bool hv_top8(const HvProblem& p) {
  return !p.greedy && ((p.bias_k > 0 && p.beta < 1.f) || p.fmax > 0);
}

// Bytes of device workspace the call needs beyond the 256-byte header.
size_t hv_workspace_bytes(const HvProblem& p, int sms);

// All launches of one call on `stream`, with `ws` (hv_workspace_bytes, 256-byte aligned) and the
// error word of the stream's workspace.
cudaError_t hv_run(const HvProblem& p, int sms, void* ws, unsigned int* err, cudaStream_t stream);

}  // namespace sv

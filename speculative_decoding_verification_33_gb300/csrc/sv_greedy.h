// Interface between the host API (sv_api.cu) and the parallel greedy kernels (sv_greedy.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

struct GreedyParams {
  const void* tgt;          // target logits [B][K+1][stride]
  long long stride;         // elements between rows
  const int32_t* lens;      // [B] draft lengths, or NULL (all K)
  const int32_t* tokens;    // [B][K] draft ids
  int B, K, V;
  int slice;                // vocabulary ids per CTA (multiple of 8)
  int nslice;               // slices per row
  int aligned;              // rows 16-byte aligned: vector loads
  unsigned long long* keys; // [B][K+1][nslice] workspace: the slice maxima as sort keys
  int32_t* out_acc;         // [B]
  int32_t* out_tok;         // [B][K+1]
};

// Slices per row for a batch of B sequences on `sms` multiprocessors.
void greedy_plan(int B, int K, int V, int sms, int* nslice, int* slice);

// Workspace bytes of the slice keys.
inline size_t greedy_keys_bytes(int B, int K, int nslice) {
  return static_cast<size_t>(B) * (K + 1) * nslice * sizeof(unsigned long long);
}

// The two launches (row slices, then one warp per sequence) on `stream`; dtype 1 = bf16.
cudaError_t launch_greedy(const GreedyParams& P, int dtype, cudaStream_t stream);

}  // namespace sv

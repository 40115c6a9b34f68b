// Interface between the host API (sv_api.cu) and the LM-head kernels (sv_lmhead.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

constexpr int kHeadBM = 128;  // rows (hidden states) per tile
constexpr int kHeadBN = 256;  // vocabulary columns per tile
constexpr int kHeadBK = 64;   // hidden units per pipeline stage (128 bytes of bf16)

struct HeadParams {
  int R, d, V;
  float c;               // log2(e) / T
  float inv_t;           // 1 / T
  const int32_t* ids;    // [R] token whose logit is reported, or NULL
  float* part;           // [nsplit][R][3]: maximum, sum 2^(z c - fl(max c)), logit at the id
  float* out_logits;     // [R][V] fp32 logits (tests only), or NULL
  int nsplit;            // vocabulary ranges (CTAs per 128-row tile)
  int tiles_per_split;   // 256-column tiles per range
  int ntiles;            // 256-column tiles of the vocabulary
  unsigned int* err;     // bit 0 raised when a bounded wait gives up
};

// Bytes of the partial statistics for R rows in `nsplit` ranges.
inline size_t head_part_bytes(int R, int nsplit) {
  return static_cast<size_t>(R) * static_cast<size_t>(nsplit) * 3 * sizeof(float);
}

// The split of the vocabulary for R rows on a device with `sms` multiprocessors.
void head_split(int R, int V, int sms, int* nsplit, int* tiles_per_split, int* ntiles);

// Row statistics of logits = hidden (R x d, bf16, row stride hs elements) * weight^T (V x d,
// bf16, row stride ws elements): per row the maximum logit, the natural log-sum-exp of z / T and
// the logit at ids[r]. Two launches (the GEMM with its epilogue, then the combine of the
// vocabulary ranges) on `stream`. Returns cudaErrorNotSupported when the tensor-map encoder of
// the driver cannot be had.
cudaError_t launch_lmhead(const void* hidden, long long hs, const void* weight, long long ws,
                          const HeadParams& P, float* out_max, float* out_lse, float* out_zx,
                          cudaStream_t stream);

}  // namespace sv

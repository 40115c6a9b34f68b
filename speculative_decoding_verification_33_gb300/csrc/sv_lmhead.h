// Interface between the host API (sv_api.cu, sv_hverify.cu) and the LM-head kernels
// (sv_lmhead.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

constexpr int kHeadBM = 128;  // rows (hidden states) per tile
constexpr int kHeadBN = 256;  // vocabulary columns per tile
constexpr int kHeadBK = 64;   // hidden units per pipeline stage (128 bytes of bf16)
constexpr int kHeadHalves = kHeadBN / 16;  // residual masses per tile and pair (16 columns each)

// Epilogues of the head GEMM.
enum HeadMode : int {
  HEAD_STATS = 0,  // per row: maximum, sum of 2^(z c - fl(m c)), logit at an id, first argmax
  HEAD_RESID = 1,  // per pair of rows (target, draft): masses of max(e_t - rho e_d, 0) and of e_t
                   // per 16 ids
  HEAD_STATS_TOP8 = 2,  // HEAD_STATS, and per row and range the 8 largest logits as keys
};

// Per-row statistics after the combine (HEAD_STATS).
struct HeadRow {
  float max;   // largest logit
  float lse;   // ln sum_v exp(z_v / T)
  float zx;    // logit at the requested id (NaN when none)
  int arg;     // lowest id holding the largest logit
  float mc;    // fl(max * c)
  float sum;   // sum_v 2^(z_v c - fl(max c))
};

// Per-pair inputs of HEAD_RESID: the residual weight of id v is
// max(2^(z_t c - mc_t) - rho_v 2^(z_d c - mc_d), 0) with rho_v = rho_s for the nS ids of the
// bias set and rho for the others; rho = 0 gives the bonus weights of p alone. A pair with
// skip != 0 produces zero masses.
struct HeadPair {
  float mc_t, mc_d, rho;
  int skip;
  float rho_s;
  int nS;
  int ids[8];
};

struct HeadParams {
  int R, d, V;               // R: rows of the A operand (an upper bound when R_dev is set)
  const int* R_dev;          // rows actually present, read on the device (NULL: R)
  float c;                   // log2(e) / T
  float inv_t;               // 1 / T
  const int32_t* ids;        // stats: id per row whose logit is reported, or NULL
  float4* part;              // stats: [nsplit][R] (max, sum, logit at the id, argmax bits)
  float* out_logits;         // stats: [R][V] fp32 logits (tests only), or NULL
  const HeadPair* pair;      // resid: [R / 2] pair inputs
  unsigned long long* mass;  // resid: [R / 2][nh] residual masses in 2^-44 units
  unsigned long long* mass_p;  // resid: [R / 2][nh] masses of 2^(z_t c - mc_t) alone
  unsigned long long* keys;  // stats with top 8: [nsplit][R][8] each row's 8 largest keys per
                             // range (larger value first, then lower id; 0 = none)
  int nh;                    // resid: masses per pair (ntiles * kHeadHalves)
  int nsplit;                // vocabulary ranges
  int tiles_per_split;       // 256-column tiles per range
  int ntiles;                // 256-column tiles of the vocabulary
  unsigned int* err;         // bit 0 raised when a bounded wait gives up
};

// Rows of A (R), pairs of rows in HEAD_RESID: tile m holds pairs 64 m .. 64 m + 63, row
// 128 m + 32 q + l holding the target row of pair 64 m + 16 q + l (l < 16) and the draft row of
// pair 64 m + 16 q + (l - 16) (l >= 16).
__host__ __device__ inline int head_pair_row(int pair, int draft) {
  return (pair >> 6) * kHeadBM + ((pair >> 4) & 3) * 32 + (pair & 15) + (draft ? 16 : 0);
}

// Bytes of the partial statistics for R rows in `nsplit` ranges.
inline size_t head_part_bytes(int R, int nsplit) {
  return static_cast<size_t>(R) * static_cast<size_t>(nsplit) * sizeof(float4);
}

// The split of the vocabulary into ranges for up to R rows: ranges of whole 256-column tiles,
// small enough that row tiles x ranges give every SM several work items; with max_ranges > 0,
// no more than that many ranges (each row's per-range top 8 are merged over the ranges).
void head_split(int R, int V, int sms, int* nsplit, int* tiles_per_split, int* ntiles,
                int max_ranges = 0);

// Persistent CTAs for the head GEMM on a device with `sms` multiprocessors.
int head_ctas(int sms);

// The head GEMM logits = A (R x d, bf16, row stride as elements) * W^T (V x d, bf16, row stride
// ws elements) with the epilogue `mode`, on `ctas` persistent CTAs. Returns
// cudaErrorNotSupported when the tensor-map encoder of the driver cannot be had.
cudaError_t launch_head_gemm(int mode, const void* A, long long as, const void* weight,
                             long long ws, const HeadParams& P, int ctas, cudaStream_t stream);

// The vocabulary ranges of every row (HEAD_STATS partials) into its statistics: any output may
// be NULL. Rows at or past *R_dev (when set) are left alone.
cudaError_t launch_head_combine(const HeadParams& P, float* out_max, float* out_lse,
                                float* out_zx, int32_t* out_arg, HeadRow* out_rows,
                                cudaStream_t stream);

}  // namespace sv

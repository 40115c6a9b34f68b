// Internal interface between the host API (sv_api.cu) and the verify kernels (sv_kernel.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

constexpr int kThreads = 256;     // threads per CTA
constexpr int kMaxCluster = 16;   // CTAs that share one sequence's rows
constexpr int kMaxK = 8;          // maximum draft length
constexpr int kMaxV = 262144;     // maximum vocabulary
constexpr int kQScale = 44;       // residual weights are summed as integers of 2^-44
constexpr int NS = 2;             // stages of the per-CTA row ring
constexpr int kStageRowBytes = 16384;  // bytes of one row in one stage
constexpr int kMaxSlice = 65536;  // elements of a row one CTA owns (bounds the draw's buffer)

// Device workspace shared by the clusters of one launch. The kernel returns the counters to
// zero when the last cluster leaves, so stream-ordered launches (and replays of a captured
// launch) can reuse it.
struct Workspace {
  unsigned int next;    // dynamic sequence queue
  unsigned int done;    // clusters that have finished
  unsigned int error;   // bit 0: a bounded wait gave up
  unsigned int dcount;  // deferred draws: sequences decided so far
  unsigned int pad[60];
};
static_assert(sizeof(Workspace) == 256, "workspace layout");

struct Params {
  const void* tgt;
  const void* dft;
  const int32_t* tokens;
  const int32_t* lens;
  const float* uni;
  int32_t* out_acc;
  int32_t* out_tok;
  int32_t* out_topf;
  float* dbg_lse_t;
  float* dbg_lse_d;
  float* dbg_px;
  float* dbg_qx;
  long long t_stride;
  long long d_stride;
  int B, K, V;
  float temperature;
  float c;        // log2(e) / T, rounded to float
  float beta;
  int bias_k;     // 0 when beta == 1
  int fmax;       // columns of out_topf (0 = no top-F output)
  int fan[kMaxK];
  int top8;       // draft rows need their top-8 ids
  int debug_all;  // read every row a sequence has and fill the diagnostics
  int slice;      // elements of a row owned by one CTA (multiple of 8)
  int use_bulk;   // rows and strides are 16-byte aligned: stage rows with bulk async copies
  int vec_fill;   // without bulk copies, rows 16-byte aligned: consumers fill chunks with 16-byte
                  // loads (rows read in place from pinned host memory)
  void* scratch;  // rows read in place from host memory: per CTA, a device copy of its slices of
                  // the position last streamed, for the draw ([clusters][C][2][slice]), or NULL
  int n_clusters;
  int lpt;         // take sequences longest draft first
  const unsigned long long* keys;  // top-8 keys of every draft row from the prepass, or NULL
  Workspace* ws;
  // Deferred draws (stochastic decision-ahead walk): instead of drawing, a decided sequence's
  // draw constants go to ddec[seq] (a SmallDecision, sv_small.h) and seq + 1 to dlist[k] for the
  // k-th sequence decided; the draw launches that follow the walk take them from there.
  int defer;
  void* ddec;
  int* dlist;
};

constexpr int kLptMaxB = 4096;  // larger batches keep the natural order

// The workspace does not grow with the batch.
constexpr size_t workspace_bytes_for(int /*B*/) { return sizeof(Workspace); }

struct Launch {
  Params p;
  int dtype;       // 0 f32, 1 bf16
  int greedy;
  int cluster;     // CTAs per cluster
  size_t smem;     // dynamic shared memory per CTA
};

// Dynamic shared memory per CTA: the stage ring plus the draw's per-vector masses.
size_t smem_bytes(int dtype, int greedy, int slice);
// Largest number of co-resident clusters for this configuration (0 on error).
int max_active_clusters(int dtype, int greedy, int top8, int cluster, size_t smem);
cudaError_t launch(const Launch& L, cudaStream_t stream);

cudaError_t launch_probe(const void* buf, size_t bytes, unsigned long long* out,
                         cudaStream_t stream);
// A bounded wait that runs out after `budget_cycles` clock cycles and raises *err bit 0.
cudaError_t launch_wait_probe(long long budget_cycles, unsigned int* err, cudaStream_t stream);

}  // namespace sv

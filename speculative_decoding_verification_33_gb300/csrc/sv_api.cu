// C ABI of the verify library: argument checks, per-(device, stream) workspace, the choice of
// cluster size, and the launch. Everything here is host code; every step of the verify path
// runs in the kernels of sv_kernel.cu.
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>
#include <vector>

#include "spec_verify.h"
#include "sv_internal.h"
#include "sv_rows.h"
#include "sv_lmhead.h"
#include "sv_hverify.h"
#include "sv_greedy.h"
#include "sv_small.h"
#include "sv_probe.h"

namespace {

using sv::Workspace;

constexpr size_t kMaxDynSmem = 200 * 1024;

struct StreamRes {
  Workspace* ws = nullptr;
  size_t ws_bytes = 0;
  void* stage = nullptr;  // device staging for spec_verify_host
  size_t stage_bytes = 0;
  void* scr = nullptr;    // rows read in place from host memory: the draw's device copies
  size_t scr_bytes = 0;
  void* dd = nullptr;     // deferred draws of the walk (sv::walk_draw_carve) for batches of up
  int dd_cap = 0;         // to dd_cap sequences: order list (all zero between calls), decisions,
};                        // masses

// Workspace of spec_verify_noalloc: the queue counters and error word the kernel needs (256
// bytes), for batches of up to kNoAllocMaxB sequences, in device memory that belongs to this
// module rather than to any allocation. Every GPU that loads the library holds it until the
// process exits. Host code must not use the symbol as a pointer: its device
// address comes from cudaGetSymbolAddress, once per device.
constexpr int kNoAllocMaxB = 65536;
static __device__ __align__(256) unsigned char g_noalloc_ws[sv::workspace_bytes_for(kNoAllocMaxB)];
std::map<int, void*> g_noalloc_ptr;  // device ordinal -> address of g_noalloc_ws there

// Device address of g_noalloc_ws on device `dev` (the current device). The first request with
// `create` looks the array up with cudaGetSymbolAddress and keeps the address; without
// `create`, *ws stays NULL until then. Caller holds g_mu.
sv_status noalloc_array(int dev, bool create, void** ws) {
  *ws = nullptr;
  auto it = g_noalloc_ptr.find(dev);
  if (it != g_noalloc_ptr.end()) {
    *ws = it->second;
    return SV_OK;
  }
  if (!create) return SV_OK;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess || !p) return SV_ERR_CUDA;
  g_noalloc_ptr[dev] = p;
  *ws = p;
  return SV_OK;
}

// Reads the error word of a workspace (after the caller synchronised its stream) and clears it.
// Returns SV_ERR_DEVICE_TIMEOUT if it was raised.
sv_status take_error(Workspace* ws) {
  unsigned int err = 0;
  if (cudaMemcpy(&err, &ws->error, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SV_ERR_CUDA;
  if (!err) return SV_OK;
  if (cudaMemset(&ws->error, 0, sizeof(err)) != cudaSuccess) return SV_ERR_CUDA;
  return SV_ERR_DEVICE_TIMEOUT;
}

std::mutex g_mu;
std::map<std::pair<int, cudaStream_t>, StreamRes> g_res;
std::map<std::tuple<int, int, int, int, int, size_t>, int> g_occ;  // dev,dtype,greedy,top8,C,smem
std::map<int, int> g_sms;

struct Checked {
  int greedy = 0;
  int beta_lt1 = 0;
  int fmax = 0;
  int fan[sv::kMaxK] = {0};
  size_t elt = 4;
};

bool finite_in(float v, float lo, float hi) { return std::isfinite(v) && v >= lo && v <= hi; }

sv_status check_args(const sv_problem* p, const void* tgt, const void* dft,
                     const int32_t* tok, const float* uni, float T, float beta, int mode,
                     const int32_t* out_acc, const int32_t* out_tok, const int32_t* out_topf,
                     Checked* c) {
  if (!p) return SV_ERR_INVALID_ARG;
  if (p->B < 0 || p->K < 1 || p->K > sv::kMaxK || p->V < 1 || p->V > sv::kMaxV)
    return SV_ERR_INVALID_ARG;
  if (p->dtype != SV_DTYPE_F32 && p->dtype != SV_DTYPE_BF16) return SV_ERR_INVALID_ARG;
  if (mode != SV_MODE_GREEDY && mode != SV_MODE_STOCHASTIC) return SV_ERR_INVALID_ARG;
  if (p->target_row_stride < p->V) return SV_ERR_INVALID_ARG;
  const int h = p->cluster_hint;
  if (!(h == 0 || h == 1 || h == 2 || h == 4 || h == 8 || h == 16)) return SV_ERR_INVALID_ARG;
  c->greedy = mode == SV_MODE_GREEDY;
  c->elt = p->dtype == SV_DTYPE_BF16 ? 2 : 4;
  if (!c->greedy) {
    if (p->draft_row_stride < p->V) return SV_ERR_INVALID_ARG;
    if (!finite_in(T, 1e-4f, 1e4f)) return SV_ERR_INVALID_ARG;
    if (!(std::isfinite(beta) && beta > 0.f && beta <= 1.f)) return SV_ERR_INVALID_ARG;
    if (p->bias_k < 0 || p->bias_k > 8) return SV_ERR_INVALID_ARG;
    c->beta_lt1 = beta < 1.f;
  }
  c->fmax = 0;
  if (p->fanout) {
    if (c->greedy) return SV_ERR_INVALID_ARG;
    for (int i = 0; i < p->K; ++i) {
      const int f = p->fanout[i];
      if (f < 0 || f > 8) return SV_ERR_INVALID_ARG;
      c->fan[i] = f;
      c->fmax = std::max(c->fmax, f);
    }
  }
  if (p->B == 0) return SV_OK;
  if (!tgt || !tok || !out_acc || !out_tok) return SV_ERR_INVALID_ARG;
  if (!c->greedy && (!dft || !uni)) return SV_ERR_INVALID_ARG;
  if (c->fmax > 0 && !out_topf) return SV_ERR_INVALID_ARG;
  if (!p->fanout && out_topf) return SV_ERR_INVALID_ARG;
  return SV_OK;
}

int sm_count(int dev) {
  auto it = g_sms.find(dev);
  if (it != g_sms.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 0;
  g_sms[dev] = n;
  return n;
}

StreamRes* resources(int dev, cudaStream_t s, size_t need, sv_status* st) {
  StreamRes& r = g_res[{dev, s}];
  if (!r.ws || r.ws_bytes < need) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) == cudaSuccess && cap != cudaStreamCaptureStatusNone) {
      *st = SV_ERR_UNSUPPORTED;  // the workspace must exist (and be large enough) before capture
      return nullptr;
    }
    if (r.ws) {
      if (cudaStreamSynchronize(s) != cudaSuccess) {
        *st = SV_ERR_CUDA;
        return nullptr;
      }
      cudaFree(r.ws);
      r.ws = nullptr;
      r.ws_bytes = 0;
    }
    void* w = nullptr;
    if (cudaMalloc(&w, need) != cudaSuccess || cudaMemset(w, 0, need) != cudaSuccess) {
      if (w) cudaFree(w);
      *st = SV_ERR_CUDA;
      return nullptr;
    }
    r.ws = static_cast<Workspace*>(w);
    r.ws_bytes = need;
  }
  *st = SV_OK;
  return &r;
}

// Resident clusters of C CTAs for this problem (cached per device and kernel variant); fills the
// slice and shared-memory size of that C. 0 when C cannot be launched.
int resident_clusters(const sv_problem* p, int dev, int dtype, int greedy, int top8, int C,
                      int* slice_out, size_t* smem_out) {
  const long long slice = ((static_cast<long long>(p->V) + C - 1) / C + 7) / 8 * 8;
  *slice_out = static_cast<int>(slice);
  *smem_out = sv::smem_bytes(dtype, greedy, static_cast<int>(slice));
  if (slice > sv::kMaxSlice || *smem_out > kMaxDynSmem) return 0;
  auto key = std::make_tuple(dev, dtype, greedy, top8, C, *smem_out);
  auto it = g_occ.find(key);
  if (it != g_occ.end()) return it->second;
  const int occ = sv::max_active_clusters(dtype, greedy, top8, C, *smem_out);
  g_occ[key] = occ;
  return occ;
}

// The draft rows' top 8 are needed (bias set or top-F ids).
bool needs_top8(const sv_problem* p, const Checked& c) {
  return !c.greedy && ((p->bias_k > 0 && c.beta_lt1) || c.fmax > 0);
}

// Bytes of the top-8 prepass keys in a workspace (after the counters): 8 keys per position.
size_t keys_bytes(const sv_problem* p) {
  return static_cast<size_t>(p->B) * static_cast<size_t>(p->K) * 8 * sizeof(unsigned long long);
}

// Ring stages and co-resident CTAs per SM of a row kernel (g_mu held): the most stages that
// still let two CTAs share an SM (at least 3); failing that, one CTA per SM with up to
// kRowMaxStages.
// dev, mode, dtype, bias, V -> (ring stages, CTAs per SM)
std::map<std::tuple<int, int, int, int, int>, std::pair<int, int>> g_row_occ;

std::pair<int, int> row_config(int dev, int mode, int dtype, bool bias, int V) {
  const auto key = std::make_tuple(dev, mode, dtype, bias ? 1 : 0, V);
  auto it = g_row_occ.find(key);
  if (it == g_row_occ.end()) {
    int nst = 0, per_sm = 0;
    for (int st = sv::kRowMaxStages; st >= 3 && !nst; --st)
      if (sv::row_smem_bytes(mode, dtype, V, st) <= 112 * 1024) nst = st;
    if (nst) per_sm = sv::row_ctas_per_sm(mode, dtype, bias, V, nst);
    if (per_sm < 2) {
      nst = 0;
      for (int st = sv::kRowMaxStages; st >= 2 && !nst; --st)
        if (sv::row_smem_bytes(mode, dtype, V, st) <= sv::kRowMaxSmem) nst = st;
      per_sm = nst ? sv::row_ctas_per_sm(mode, dtype, bias, V, nst) : 0;
    }
    it = g_row_occ.emplace(key, std::make_pair(nst, per_sm)).first;
  }
  return it->second;
}

// Cluster size, slice, shared memory and the number of clusters to launch (g_mu held).
//
// One sequence is verified by one cluster, position after position, so a sequence's latency
// falls as C grows while the work per byte (exchanges, barriers) rises. The choice: the largest C
// whose co-resident clusters still hold the whole batch at once, each CTA keeping at least 512
// vocabulary entries; when no C holds the batch, the smallest C whose slice fits shared memory
// (throughput). A cluster_hint overrides the choice.
// With `prepass`, the draft rows' top 8 come from the top-8 prepass and the verify kernel needs
// no in-stream top-8.
sv_status plan(const sv_problem* p, const Checked& c, int dev, sv::Launch* L,
               bool prepass = false) {
  if (sm_count(dev) <= 0) return SV_ERR_CUDA;
  const int dtype = p->dtype == SV_DTYPE_BF16 ? 1 : 0;
  const int top8 = !prepass && needs_top8(p, c);
  int C = p->cluster_hint, slice = 0, occ = 0;
  size_t smem = 0;
  if (C) {
    occ = resident_clusters(p, dev, dtype, c.greedy, top8, C, &slice, &smem);
  } else {
    int c_max = 1;
    while (c_max * 2 <= sv::kMaxCluster && static_cast<long long>(c_max) * 2 * 512 <= p->V)
      c_max <<= 1;
    int fallback = 0;  // smallest launchable C
    for (int cand = c_max; cand >= 1 && !C; cand >>= 1) {
      int s = 0;
      size_t m = 0;
      const int n = resident_clusters(p, dev, dtype, c.greedy, top8, cand, &s, &m);
      if (n <= 0) continue;
      fallback = cand;
      if (n >= p->B) C = cand;
    }
    if (!C) C = fallback;
    if (!C) return SV_ERR_UNSUPPORTED;
    occ = resident_clusters(p, dev, dtype, c.greedy, top8, C, &slice, &smem);
  }
  if (occ <= 0) return SV_ERR_UNSUPPORTED;
  L->p.slice = slice;
  L->dtype = dtype;
  L->greedy = c.greedy;
  L->cluster = C;
  L->smem = smem;
  L->p.top8 = top8;
  L->p.n_clusters = std::max(1, std::min(p->B, occ));
  return SV_OK;
}

// The kernels a call takes. The chained cluster walk serves every problem; two paths read every
// row a sequence has at once when that costs less than the walk's latency of position after
// position: greedy batches whose padded target rows fit in 64 MiB (argmax per row slice, then one
// warp per sequence), and stochastic batches whose rows fit in 256 MiB (row statistics, the
// draw's slice masses, one pick per sequence; the statistics launch keeps the draft rows' top 8
// for a bias set or top-F ids). A nonzero cluster_hint, the diagnostics entry point and rows read in place from host
// memory always take the walk.
enum Route { ROUTE_WALK = 0, ROUTE_GREEDY_ROWS = 1, ROUTE_SMALL = 2 };

// Row-statistics CTAs of the small-batch route resident per multiprocessor (cached per device
// and dtype; call under g_mu).
int small_rows_per_sm(int dev, int dtype) {
  static std::map<std::pair<int, int>, int> cache;
  auto it = cache.find({dev, dtype});
  if (it != cache.end()) return it->second;
  const int n = sv::small_rows_per_sm(dtype);
  cache[{dev, dtype}] = n;
  return n;
}

Route route_of(const sv_problem* p, const Checked& c, int dev, int sms, bool debug_all,
               bool zero_copy, sv::SmallParams* sp) {
  if (debug_all || p->cluster_hint != 0 || sms <= 0) return ROUTE_WALK;
  const long long B = p->B, K = p->K;
  if (c.greedy)
    return (B * (K + 1) <= 65535 && B * (K + 1) * p->target_row_stride * c.elt <= (64LL << 20))
               ? ROUTE_GREEDY_ROWS
               : ROUTE_WALK;
  if (zero_copy || B * (2 * K + 1) > 65535 ||
      B * (2 * K + 1) * std::max(p->target_row_stride, p->draft_row_stride) * c.elt >
          (256LL << 20))
    return ROUTE_WALK;
  const int dtype = p->dtype == SV_DTYPE_BF16 ? 1 : 0;
  return sv::small_plan(p->B, p->K, p->V, sms, small_rows_per_sm(dev, dtype), sp) ? ROUTE_SMALL
                                                                                : ROUTE_WALK;
}

// The top-8 prepass over the draft rows (bias set, top-F ids): 8 keys per draft row into `keys`,
// and the top-F ids of the rows below L into out_topf.
sv_status launch_prepass(const sv_problem* p, const Checked& c, int dev, int dtype,
                         const void* dft, const int32_t* lens, float cc,
                         unsigned long long* keys, int32_t* out_topf, Workspace* ws,
                         cudaStream_t stream) {
  sv::RowParams R;
  memset(&R, 0, sizeof(R));
  R.dft = dft;
  R.d_stride = p->draft_row_stride;
  R.V = p->V;
  R.K = p->K;
  R.B = p->B;
  R.lens = lens;
  R.c = cc;
  R.fmax = c.fmax;
  for (int i = 0; i < sv::kMaxK; ++i) R.fan[i] = c.fan[i];
  R.use_vec = (reinterpret_cast<uintptr_t>(dft) % 16 == 0 &&
               (p->draft_row_stride * static_cast<long long>(c.elt)) % 16 == 0)
                  ? 1
                  : 0;
  R.out_keys = keys;
  R.out_topf = c.fmax > 0 ? out_topf : nullptr;
  R.ws = ws;
  const std::pair<int, int> rc = row_config(dev, 2, dtype, false, p->V);
  if (rc.first < 2 || rc.second < 1) return SV_ERR_UNSUPPORTED;
  R.nstages = rc.first;
  const int units = p->B * p->K;
  const int ctas = std::min(units, rc.second * sm_count(dev));
  return sv::launch_rows(R, 2, dtype, ctas, stream) == cudaSuccess
             ? SV_OK
             : SV_ERR_CUDA;
}

sv_status run(const sv_problem* p, const void* tgt, const void* dft, const int32_t* tok,
              const int32_t* lens, const float* uni, float T, float beta, int mode,
              int32_t* out_acc, int32_t* out_tok, int32_t* out_topf, float* lse_t,
              float* lse_d, float* px, float* qx, int debug_all, Workspace* ws_user,
              size_t ws_user_bytes, cudaStream_t stream, bool zero_copy = false) {
  Checked c;
  sv_status st = check_args(p, tgt, dft, tok, uni, T, beta, mode, out_acc, out_tok, out_topf, &c);
  if (st != SV_OK || p->B == 0) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;

  sv::Launch L;
  memset(&L, 0, sizeof(L));
  sv::Params& P = L.p;
  P.tgt = tgt;
  P.dft = c.greedy ? nullptr : dft;
  P.tokens = tok;
  P.lens = lens;
  P.uni = c.greedy ? nullptr : uni;
  P.out_acc = out_acc;
  P.out_tok = out_tok;
  P.out_topf = c.fmax > 0 ? out_topf : nullptr;
  P.dbg_lse_t = lse_t;
  P.dbg_lse_d = lse_d;
  P.dbg_px = px;
  P.dbg_qx = qx;
  P.t_stride = p->target_row_stride;
  P.d_stride = c.greedy ? 0 : p->draft_row_stride;
  P.B = p->B;
  P.K = p->K;
  P.V = p->V;
  P.temperature = c.greedy ? 1.f : T;
  P.c = c.greedy ? 1.f : static_cast<float>(1.4426950408889634 / static_cast<double>(T));
  P.beta = c.greedy ? 1.f : beta;
  P.bias_k = (c.greedy || beta >= 1.f) ? 0 : p->bias_k;
  P.fmax = c.fmax;
  for (int i = 0; i < sv::kMaxK; ++i) P.fan[i] = c.fan[i];
  P.debug_all = debug_all;

  const uintptr_t a_t = reinterpret_cast<uintptr_t>(tgt);
  const uintptr_t a_d = reinterpret_cast<uintptr_t>(dft);
  bool aligned = (a_t % 16 == 0) && ((p->target_row_stride * c.elt) % 16 == 0);
  if (!c.greedy) aligned = aligned && (a_d % 16 == 0) && ((p->draft_row_stride * c.elt) % 16 == 0);
  // rows read in place from pinned host memory go through the consumers' own loads
  P.use_bulk = (aligned && !zero_copy) ? 1 : 0;
  P.vec_fill = aligned ? 1 : 0;

  sv::SmallParams G2;
  memset(&G2, 0, sizeof(G2));
  Route route;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    route = route_of(p, c, dev, sm_count(dev), debug_all != 0, zero_copy, &G2);
  }
  // Greedy verification of a small batch: every target row in flight at once, argmax per row
  // slice, then one warp per sequence walks the positions.
  if (route == ROUTE_GREEDY_ROWS) {
    std::lock_guard<std::mutex> lock(g_mu);
    sv::GreedyParams G;
    G.tgt = tgt;
    G.stride = p->target_row_stride;
    G.lens = lens;
    G.tokens = tok;
    G.B = p->B;
    G.K = p->K;
    G.V = p->V;
    G.aligned = aligned ? 1 : 0;
    G.out_acc = out_acc;
    G.out_tok = out_tok;
    const int sms = sm_count(dev);
    if (sms <= 0) return SV_ERR_CUDA;
    sv::greedy_plan(p->B, p->K, p->V, sms, &G.nslice, &G.slice);
    const size_t kb2 = sv::greedy_keys_bytes(p->B, p->K, G.nslice);
    Workspace* w = nullptr;
    if (ws_user) {
      if (ws_user_bytes >= sizeof(Workspace) + kb2) w = ws_user;
    } else {
      StreamRes* r = resources(dev, stream, sizeof(Workspace) + kb2, &st);
      if (!r) return st;
      w = r->ws;
    }
    if (w) {  // (a caller's workspace too small for the keys takes the cluster walk)
      G.keys = reinterpret_cast<unsigned long long*>(w + 1);
      return sv::launch_greedy(G, p->dtype == SV_DTYPE_BF16 ? 1 : 0, stream) == cudaSuccess
                 ? SV_OK
                 : SV_ERR_CUDA;
    }
  }

  // Stochastic verification of a small batch: every row's statistics at once, then the draw's
  // slice masses of the decided rows, then one CTA per sequence picks the token.
  if (route == ROUTE_SMALL) {
    std::lock_guard<std::mutex> lock(g_mu);
    sv::SmallParams& G = G2;  // layout filled by the route's plan
    G.tgt = tgt;
    G.dft = dft;
    G.t_stride = p->target_row_stride;
    G.d_stride = p->draft_row_stride;
    G.lens = lens;
    G.tokens = tok;
    G.uni = uni;
    G.B = p->B;
    G.K = p->K;
    G.V = p->V;
    G.c = P.c;
    G.aligned = aligned ? 1 : 0;
    G.out_acc = out_acc;
    G.out_tok = out_tok;
    // a bias set or top-F ids: the statistics launch keeps the draft rows' top 8 per slice
    G.top8 = needs_top8(p, c) ? 1 : 0;
    const size_t need = sv::small_ws_bytes(G);
    Workspace* w = nullptr;
    if (ws_user) {
      if (ws_user_bytes >= sizeof(Workspace) + need) w = ws_user;
    } else {
      StreamRes* r = resources(dev, stream, sizeof(Workspace) + need, &st);
      if (!r) return st;
      w = r->ws;
    }
    if (w) {  // (a caller's workspace too small for the partials takes the cluster walk)
      const int dtype = p->dtype == SV_DTYPE_BF16 ? 1 : 0;
      sv::small_carve(G, reinterpret_cast<char*>(w + 1));
      G.err = &w->error;
      G.bias_k = P.bias_k;
      G.beta = P.beta;
      G.fmax = c.fmax;
      for (int i = 0; i < sv::kMaxK; ++i) G.fan[i] = c.fan[i];
      G.out_topf = c.fmax > 0 ? out_topf : nullptr;
      return sv::launch_small(G, dtype, stream) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
    }
  }

  // The draft rows' top 8 (bias set, top-F ids) come from a prepass over the draft rows when the
  // workspace has room for its keys; otherwise (the fixed workspace of spec_verify_noalloc, or
  // the diagnostics entry point) from the verify kernel's own stream.
  const size_t kb = keys_bytes(p);
  const bool prepass = needs_top8(p, c) && !debug_all && (!ws_user || ws_user_bytes >= sizeof(Workspace) + kb);
  std::lock_guard<std::mutex> lock(g_mu);
  st = plan(p, c, dev, &L, prepass);
  if (st != SV_OK) return st;
  if (zero_copy) {  // the draw reads the decided position back from device copies
    const size_t need = static_cast<size_t>(P.n_clusters) * static_cast<size_t>(L.cluster) * 2 *
                        static_cast<size_t>(P.slice) * c.elt;
    StreamRes& r = g_res[{dev, stream}];
    if (r.scr_bytes < need) {
      cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
      if (cudaStreamIsCapturing(stream, &cap) == cudaSuccess && cap != cudaStreamCaptureStatusNone)
        return SV_ERR_UNSUPPORTED;
      if (r.scr) {
        if (cudaStreamSynchronize(stream) != cudaSuccess) return SV_ERR_CUDA;
        cudaFree(r.scr);
        r.scr = nullptr;
        r.scr_bytes = 0;
      }
      if (cudaMalloc(&r.scr, need) != cudaSuccess) {
        r.scr = nullptr;
        return SV_ERR_CUDA;
      }
      r.scr_bytes = need;
    }
    P.scratch = r.scr;
  }

  if (ws_user) {
    P.ws = ws_user;
  } else {
    StreamRes* r = resources(dev, stream, sv::workspace_bytes_for(p->B) + (prepass ? kb : 0), &st);
    if (!r) return st;
    P.ws = r->ws;
  }
  P.lpt = p->B <= sv::kLptMaxB ? 1 : 0;
  if (prepass) {
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(P.ws + 1);
    P.keys = keys;
    st = launch_prepass(p, c, dev, L.dtype, dft, lens, P.c, keys, out_topf, P.ws, stream);
    if (st != SV_OK) return st;
  }
  // Deferred draws: a stochastic decision-ahead walk (no top-8, no diagnostics, rows in device
  // memory and 16-byte aligned, the library's own workspace) publishes each decided sequence's
  // draw constants instead of drawing; two launches chained after it take the draws, the slice
  // masses of a sequence starting as soon as the walk has decided it.
  sv::SmallParams D;
  memset(&D, 0, sizeof(D));
  bool defer = !c.greedy && !L.p.top8 && !prepass && !debug_all && P.use_bulk && !zero_copy &&
               !ws_user && p->B <= 65535 &&
               sv::small_plan(p->B, p->K, p->V, sm_count(dev), small_rows_per_sm(dev, L.dtype),
                              &D);
  if (defer) {
    StreamRes& r = g_res[{dev, stream}];
    if (r.dd_cap < p->B) {
      const size_t need = sv::walk_draw_ws_bytes(p->B);
      cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
      if (cudaStreamIsCapturing(stream, &cap) == cudaSuccess && cap != cudaStreamCaptureStatusNone)
        return SV_ERR_UNSUPPORTED;  // the state must exist (and be large enough) before capture
      if (r.dd) {
        if (cudaStreamSynchronize(stream) != cudaSuccess) return SV_ERR_CUDA;
        cudaFree(r.dd);
        r.dd = nullptr;
        r.dd_cap = 0;
      }
      if (cudaMalloc(&r.dd, need) != cudaSuccess || cudaMemset(r.dd, 0, need) != cudaSuccess) {
        if (r.dd) cudaFree(r.dd);
        r.dd = nullptr;
        return SV_ERR_CUDA;
      }
      r.dd_cap = p->B;
    }
    D.tgt = tgt;
    D.dft = dft;
    D.t_stride = p->target_row_stride;
    D.d_stride = p->draft_row_stride;
    D.lens = lens;
    D.tokens = tok;
    D.uni = uni;
    D.V = p->V;
    D.c = P.c;
    D.aligned = 1;
    D.beta = 1.f;
    D.err = &P.ws->error;
    D.out_acc = out_acc;
    D.out_tok = out_tok;
    sv::walk_draw_carve(D, static_cast<char*>(r.dd), r.dd_cap);
    P.defer = 1;
    P.ddec = D.dec;
    P.dlist = D.dlist;
  }
  if (sv::launch(L, stream) != cudaSuccess) return SV_ERR_CUDA;
  if (defer && sv::launch_walk_draws(D, L.dtype, stream) != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}

}  // namespace

extern "C" {

sv_status spec_verify(const sv_problem* prob, const void* target_logits,
                      const void* draft_logits, const int32_t* draft_tokens,
                      const int32_t* draft_lens, const float* uniforms, float temperature,
                      float beta, int mode, int32_t* out_accept_len, int32_t* out_tokens,
                      int32_t* out_residual_topF, void* stream) {
  return run(prob, target_logits, draft_logits, draft_tokens, draft_lens, uniforms,
             temperature, beta, mode, out_accept_len, out_tokens, out_residual_topF, nullptr,
             nullptr, nullptr, nullptr, 0, nullptr, 0, static_cast<cudaStream_t>(stream));
}

sv_status spec_verify_plan(const sv_problem* prob, int mode, int* cluster, int* clusters,
                           size_t* smem_bytes) {
  Checked c;
  const int one = 1;
  const float u = 0.5f;
  const float beta = prob && prob->bias_k > 0 ? 0.5f : 1.f;  // a bias set implies beta < 1
  sv_status st = check_args(prob, &one, &one, &one, &u, 1.f, beta, mode, &one, &one,
                            prob && prob->fanout ? &one : nullptr, &c);
  if (st != SV_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  sv::Launch L;
  memset(&L, 0, sizeof(L));
  {
    std::lock_guard<std::mutex> lock(g_mu);
    st = plan(prob, c, dev, &L);
  }
  if (st != SV_OK) return st;
  if (cluster) *cluster = L.cluster;
  if (clusters) *clusters = L.p.n_clusters;
  if (smem_bytes) *smem_bytes = L.smem;
  return SV_OK;
}

sv_status spec_verify_route(const sv_problem* prob, int mode, int* route, int* launches) {
  Checked c;
  const int one = 1;
  const float u = 0.5f;
  const float beta = prob && prob->bias_k > 0 ? 0.5f : 1.f;  // a bias set implies beta < 1
  sv_status st = check_args(prob, &one, &one, &one, &u, 1.f, beta, mode, &one, &one,
                            prob && prob->fanout ? &one : nullptr, &c);
  if (st != SV_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  sv::SmallParams sp;
  memset(&sp, 0, sizeof(sp));
  Route r;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    const int sms = sm_count(dev);
    if (sms <= 0) return SV_ERR_CUDA;
    r = route_of(prob, c, dev, sms, false, false, &sp);
  }
  if (route) *route = static_cast<int>(r);
  if (launches)
    // (the stochastic walk without a top-8 prepass defers its draws to two launches)
    *launches = r == ROUTE_SMALL ? 3
                : (r == ROUTE_GREEDY_ROWS || needs_top8(prob, c)) ? 2
                : c.greedy ? 1 : 3;
  return SV_OK;
}

size_t spec_verify_workspace_bytes(const sv_problem* prob) {
  if (!prob) return sv::workspace_bytes_for(0);
  // a bias set or top-F ids: room for the top-8 prepass keys as well
  const bool top8 = prob->bias_k > 0 || prob->fanout != nullptr;
  return sv::workspace_bytes_for(prob->B) +
         (top8 && prob->B > 0 && prob->K > 0 ? keys_bytes(prob) : 0);
}

sv_status spec_verify_ws(const sv_problem* prob, const void* target_logits,
                         const void* draft_logits, const int32_t* draft_tokens,
                         const int32_t* draft_lens, const float* uniforms, float temperature,
                         float beta, int mode, int32_t* out_accept_len, int32_t* out_tokens,
                         int32_t* out_residual_topF, void* workspace, size_t workspace_bytes,
                         void* stream) {
  if (!workspace || !prob || workspace_bytes < sv::workspace_bytes_for(prob->B) ||
      reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
    return SV_ERR_INVALID_ARG;
  return run(prob, target_logits, draft_logits, draft_tokens, draft_lens, uniforms,
             temperature, beta, mode, out_accept_len, out_tokens, out_residual_topF, nullptr,
             nullptr, nullptr, nullptr, 0, static_cast<Workspace*>(workspace), workspace_bytes,
             static_cast<cudaStream_t>(stream));
}

sv_status spec_verify_noalloc(const sv_problem* prob, const void* target_logits,
                              const void* draft_logits, const int32_t* draft_tokens,
                              const int32_t* draft_lens, const float* uniforms,
                              float temperature, float beta, int mode, int32_t* out_accept_len,
                              int32_t* out_tokens, int32_t* out_residual_topF, void* stream) {
  Checked c;
  sv_status st = check_args(prob, target_logits, draft_logits, draft_tokens, uniforms,
                            temperature, beta, mode, out_accept_len, out_tokens,
                            out_residual_topF, &c);
  if (st != SV_OK || prob->B == 0) return st;
  if (prob->B > kNoAllocMaxB) return SV_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    st = noalloc_array(dev, true, &ws);
    if (st != SV_OK) return st;
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the queue counters must start at zero for every call (a call cut short by a bounded wait
  // leaves them set); the error word is left alone, for spec_verify_device_error to report
  if (cudaMemsetAsync(ws, 0, offsetof(Workspace, error), s) != cudaSuccess) return SV_ERR_CUDA;
  return run(prob, target_logits, draft_logits, draft_tokens, draft_lens, uniforms, temperature,
             beta, mode, out_accept_len, out_tokens, out_residual_topF, nullptr, nullptr, nullptr,
             nullptr, 0, static_cast<Workspace*>(ws), sizeof(Workspace), s);
}

sv_status spec_verify_debug(const sv_problem* prob, const void* target_logits,
                            const void* draft_logits, const int32_t* draft_tokens,
                            const int32_t* draft_lens, const float* uniforms,
                            float temperature, float beta, int mode, int32_t* out_accept_len,
                            int32_t* out_tokens, int32_t* out_residual_topF, float* out_lse_t,
                            float* out_lse_d, float* out_p_x, float* out_q_x, void* stream) {
  return run(prob, target_logits, draft_logits, draft_tokens, draft_lens, uniforms,
             temperature, beta, mode, out_accept_len, out_tokens, out_residual_topF, out_lse_t,
             out_lse_d, out_p_x, out_q_x, 1, nullptr, 0, static_cast<cudaStream_t>(stream));
}

sv_status spec_verify_host(const sv_problem* prob, const void* target_logits,
                           const void* draft_logits, const int32_t* draft_tokens,
                           const int32_t* draft_lens, const float* uniforms, float temperature,
                           float beta, int mode, int32_t* out_accept_len, int32_t* out_tokens,
                           int32_t* out_residual_topF, void* stream) {
  Checked c;
  sv_status st = check_args(prob, target_logits, draft_logits, draft_tokens, uniforms,
                            temperature, beta, mode, out_accept_len, out_tokens,
                            out_residual_topF, &c);
  if (st != SV_OK || prob->B == 0) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int B = prob->B, K = prob->K;
  const size_t elt = c.elt;
  const size_t t_row = static_cast<size_t>(prob->target_row_stride) * elt;
  const size_t d_row = c.greedy ? 0 : static_cast<size_t>(prob->draft_row_stride) * elt;
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  const size_t b_t = up(static_cast<size_t>(B) * (K + 1) * t_row);
  const size_t b_d = up(static_cast<size_t>(B) * K * d_row);
  const size_t b_tok = up(static_cast<size_t>(B) * K * 4);
  const size_t b_len = draft_lens ? up(static_cast<size_t>(B) * 4) : 0;
  const size_t b_uni = c.greedy ? 0 : up(static_cast<size_t>(B) * (K + 1) * 4);
  const size_t b_acc = up(static_cast<size_t>(B) * 4);
  const size_t b_otok = up(static_cast<size_t>(B) * (K + 1) * 4);
  const size_t b_topf = up(static_cast<size_t>(B) * K * c.fmax * 4);
  const size_t total = b_t + b_d + b_tok + b_len + b_uni + b_acc + b_otok + b_topf;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  char* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    StreamRes* r = resources(dev, s, sv::workspace_bytes_for(prob->B), &st);
    if (!r) return st;
    if (r->stage_bytes < total) {
      if (cudaStreamSynchronize(s) != cudaSuccess) return SV_ERR_CUDA;
      if (r->stage) cudaFree(r->stage);
      r->stage = nullptr;
      r->stage_bytes = 0;
      if (cudaMalloc(&r->stage, total) != cudaSuccess) return SV_ERR_CUDA;
      r->stage_bytes = total;
    }
    base = static_cast<char*>(r->stage);
  }
  char* d_t = base;
  char* d_d = d_t + b_t;
  int32_t* d_tok = reinterpret_cast<int32_t*>(d_d + b_d);
  int32_t* d_len = draft_lens ? reinterpret_cast<int32_t*>(reinterpret_cast<char*>(d_tok) + b_tok) : nullptr;
  float* d_uni = c.greedy ? nullptr
                          : reinterpret_cast<float*>(reinterpret_cast<char*>(d_tok) + b_tok + b_len);
  int32_t* d_acc = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(d_tok) + b_tok + b_len + b_uni);
  int32_t* d_otok = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(d_acc) + b_acc);
  int32_t* d_topf = c.fmax > 0 ? reinterpret_cast<int32_t*>(reinterpret_cast<char*>(d_otok) + b_otok) : nullptr;

  // Rows in pinned (page-locked, mapped) host memory are read in place by the verify kernel:
  // only the rows a sequence's outcome needs cross the host link, once. Not with a top-8 prepass
  // (its bulk copies stage device rows).
  auto mapped = [](const void* ptr) -> const void* {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return (a.type == cudaMemoryTypeHost && a.devicePointer) ? a.devicePointer : nullptr;
  };
  const void* zt = needs_top8(prob, c) ? nullptr : mapped(target_logits);
  const void* zd = (zt && !c.greedy) ? mapped(draft_logits) : nullptr;
  const bool zero_copy = zt && (c.greedy || zd);
  // rows each sequence has: target 0..L_b, draft 0..L_b-1 (one contiguous block each)
  long long need = 0;
  for (int b = 0; b < B; ++b) need += draft_lens ? std::clamp(draft_lens[b], 0, K) : K;
  const bool per_seq = draft_lens && (2 * need + B) * 4 < 3LL * B * (2 * K + 1);
  auto cp = [&](void* dst, const void* src, size_t n) {
    return n == 0 || cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, s) == cudaSuccess;
  };
  bool ok = true;
  if (zero_copy) {
    // nothing to stage: the kernel reads the rows where they are
  } else if (per_seq) {
    for (int b = 0; b < B && ok; ++b) {
      const int Lb = std::clamp(draft_lens[b], 0, K);
      const size_t ot = static_cast<size_t>(b) * (K + 1) * t_row;
      ok = cp(d_t + ot, static_cast<const char*>(target_logits) + ot, (Lb + 1) * t_row);
      if (ok && !c.greedy) {
        const size_t od = static_cast<size_t>(b) * K * d_row;
        ok = cp(d_d + od, static_cast<const char*>(draft_logits) + od, Lb * d_row);
      }
    }
  } else {
    ok = cp(d_t, target_logits, static_cast<size_t>(B) * (K + 1) * t_row);
    if (ok && !c.greedy) ok = cp(d_d, draft_logits, static_cast<size_t>(B) * K * d_row);
  }
  ok = ok && cp(d_tok, draft_tokens, static_cast<size_t>(B) * K * 4);
  if (draft_lens) ok = ok && cp(d_len, draft_lens, static_cast<size_t>(B) * 4);
  if (!c.greedy) ok = ok && cp(d_uni, uniforms, static_cast<size_t>(B) * (K + 1) * 4);
  if (!ok) return SV_ERR_CUDA;
  // (the stream's own workspace, sized by run for this problem)
  st = run(prob, zero_copy ? zt : d_t, c.greedy ? nullptr : (zero_copy ? zd : d_d), d_tok, d_len,
           d_uni, temperature, beta, mode, d_acc, d_otok, d_topf, nullptr, nullptr, nullptr,
           nullptr, 0, nullptr, 0, s, zero_copy);
  if (st != SV_OK) return st;
  Workspace* ws = nullptr;  // the workspace run used (it may have grown it)
  {
    std::lock_guard<std::mutex> lock(g_mu);
    ws = g_res[{dev, s}].ws;
  }
  if (cudaMemcpyAsync(out_accept_len, d_acc, static_cast<size_t>(B) * 4,
                      cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemcpyAsync(out_tokens, d_otok, static_cast<size_t>(B) * (K + 1) * 4,
                      cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SV_ERR_CUDA;
  if (c.fmax > 0 && cudaMemcpyAsync(out_residual_topF, d_topf,
                                    static_cast<size_t>(B) * K * c.fmax * 4,
                                    cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SV_ERR_CUDA;
  unsigned int err = 0;
  if (cudaMemcpyAsync(&err, &ws->error, sizeof(err), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SV_ERR_CUDA;
  if (err) {
    cudaMemsetAsync(&ws->error, 0, sizeof(err), s);
    cudaStreamSynchronize(s);
    return SV_ERR_DEVICE_TIMEOUT;
  }
  return SV_OK;
}

sv_status spec_verify_device_error(void* stream) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  Workspace* ws = nullptr;
  void* fixed = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_res.find({dev, s});
    if (it != g_res.end()) ws = it->second.ws;
    const sv_status st = noalloc_array(dev, false, &fixed);
    if (st != SV_OK) return st;
  }
  if (cudaStreamSynchronize(s) != cudaSuccess) return SV_ERR_CUDA;
  // both words are read and cleared, so one report covers both
  const sv_status a = ws ? take_error(ws) : SV_OK;
  const sv_status b = fixed ? take_error(static_cast<Workspace*>(fixed)) : SV_OK;
  if (a == SV_ERR_CUDA || b == SV_ERR_CUDA) return SV_ERR_CUDA;
  return (a == SV_ERR_DEVICE_TIMEOUT || b == SV_ERR_DEVICE_TIMEOUT) ? SV_ERR_DEVICE_TIMEOUT
                                                                    : SV_OK;
}

sv_status spec_verify_workspace_error(void* workspace, void* stream) {
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return SV_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SV_ERR_CUDA;
  return take_error(static_cast<Workspace*>(workspace));
}

// ---------------------------------------------------------------------------------------------
// row kernels: draft sampling and the exact-residual top-F
// ---------------------------------------------------------------------------------------------
}  // extern "C"

namespace {

bool aligned16(const void* p, long long stride, size_t elt) {
  return reinterpret_cast<uintptr_t>(p) % 16 == 0 && (stride * static_cast<long long>(elt)) % 16 == 0;
}

// Launch one row kernel over `units` rows / pairs with persistent CTAs (as many as fit on the
// device, at most one per unit), on the stream's workspace (queue counters and error word). The
// ring gets the most stages that still let two CTAs share an SM (at least 3); failing that, one
// CTA per SM with up to kRowMaxStages.
sv_status run_rows(sv::RowParams& P, int mode, int dtype, int units, cudaStream_t stream) {
  const bool bias = P.bias_k > 0 && P.beta < 1.f;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  const std::pair<int, int> rc = row_config(dev, mode, dtype, bias, P.V);
  const int nst = rc.first, per_sm = rc.second;
  if (nst < 2 || per_sm < 1) return SV_ERR_UNSUPPORTED;
  P.nstages = nst;
  sv_status st = SV_OK;
  StreamRes* r = resources(dev, stream, sv::workspace_bytes_for(0), &st);
  if (!r) return st;
  P.ws = r->ws;
  const int ctas = std::min(units, per_sm * sm_count(dev));
  return sv::launch_rows(P, mode, dtype, ctas, stream) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace

extern "C" {

sv_status spec_draft_sample(int rows, int V, sv_dtype dtype, long long row_stride,
                            const void* draft_logits, const float* uniforms, float temperature,
                            float beta, int bias_k, float tau, int32_t* out_tokens,
                            float* out_conf, int32_t* out_exit, void* stream) {
  if (rows < 0 || V < 1 || V > sv::kMaxV || row_stride < V) return SV_ERR_INVALID_ARG;
  if (dtype != SV_DTYPE_F32 && dtype != SV_DTYPE_BF16) return SV_ERR_INVALID_ARG;
  if (!finite_in(temperature, 1e-4f, 1e4f)) return SV_ERR_INVALID_ARG;
  if (!(std::isfinite(beta) && beta > 0.f && beta <= 1.f)) return SV_ERR_INVALID_ARG;
  if (bias_k < 0 || bias_k > 8 || !std::isfinite(tau)) return SV_ERR_INVALID_ARG;
  if (rows == 0) return SV_OK;
  if (!draft_logits || !uniforms || !out_tokens || !out_conf) return SV_ERR_INVALID_ARG;
  const size_t elt = dtype == SV_DTYPE_BF16 ? 2 : 4;
  sv::RowParams P;
  memset(&P, 0, sizeof(P));
  P.dft = draft_logits;
  P.d_stride = row_stride;
  P.V = V;
  P.K = 1;
  P.B = rows;
  P.uni = uniforms;
  P.c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  P.beta = beta;
  P.bias_k = beta < 1.f ? bias_k : 0;
  P.tau = tau;
  P.out_tok = out_tokens;
  P.out_conf = out_conf;
  P.out_exit = out_exit;
  P.use_vec = aligned16(draft_logits, row_stride, elt) ? 1 : 0;
  return run_rows(P, 0, dtype == SV_DTYPE_BF16 ? 1 : 0, rows, static_cast<cudaStream_t>(stream));
}

sv_status spec_residual_topf(const sv_problem* prob, const void* target_logits,
                             const void* draft_logits, const int32_t* draft_lens,
                             float temperature, float beta, const int32_t* accept_len,
                             const int32_t* out_tokens, const int32_t* r1_topF, int32_t* out_r2,
                             int32_t* out_hit, void* stream) {
  Checked c;
  const int one = 1;
  const float u = 0.5f;
  sv_status st = check_args(prob, target_logits, draft_logits, &one, &u, temperature, beta,
                            SV_MODE_STOCHASTIC, &one, &one, prob && prob->fanout ? &one : nullptr,
                            &c);
  if (st != SV_OK) return st;
  if (c.fmax < 1) return SV_ERR_INVALID_ARG;  // the top-F widths come from prob->fanout
  const bool want_hit = out_hit != nullptr;
  if (want_hit != (accept_len != nullptr) || want_hit != (out_tokens != nullptr) ||
      want_hit != (r1_topF != nullptr))
    return SV_ERR_INVALID_ARG;
  if (prob->B == 0) return SV_OK;
  if (!out_r2) return SV_ERR_INVALID_ARG;
  if (static_cast<long long>(prob->B) * prob->K > (1LL << 30)) return SV_ERR_UNSUPPORTED;
  sv::RowParams P;
  memset(&P, 0, sizeof(P));
  P.tgt = target_logits;
  P.dft = draft_logits;
  P.t_stride = prob->target_row_stride;
  P.d_stride = prob->draft_row_stride;
  P.V = prob->V;
  P.K = prob->K;
  P.B = prob->B;
  P.lens = draft_lens;
  P.c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  P.beta = beta;
  P.bias_k = beta < 1.f ? prob->bias_k : 0;
  P.fmax = c.fmax;
  for (int i = 0; i < sv::kMaxK; ++i) P.fan[i] = c.fan[i];
  P.out_r2 = out_r2;
  P.out_hit = out_hit;
  P.acc = accept_len;
  P.tok = out_tokens;
  P.r1 = r1_topF;
  P.use_vec = (aligned16(target_logits, prob->target_row_stride, c.elt) &&
               aligned16(draft_logits, prob->draft_row_stride, c.elt))
                  ? 1
                  : 0;
  return run_rows(P, 1, prob->dtype == SV_DTYPE_BF16 ? 1 : 0, prob->B * prob->K,
                  static_cast<cudaStream_t>(stream));
}

sv_status spec_lmhead_stats(int rows, int d, int V, const void* hidden, long long hidden_stride,
                            const void* weight, long long weight_stride, float temperature,
                            const int32_t* ids, float* out_max, float* out_lse, float* out_zx,
                            int32_t* out_argmax, float* out_logits, void* stream) {
  if (rows < 0 || d < 64 || d % 64 != 0 || V < 1 || V > (1 << 24)) return SV_ERR_INVALID_ARG;
  if (hidden_stride < d || weight_stride < d || (hidden_stride * 2) % 16 != 0 ||
      (weight_stride * 2) % 16 != 0)
    return SV_ERR_INVALID_ARG;
  if (!finite_in(temperature, 1e-4f, 1e4f)) return SV_ERR_INVALID_ARG;
  if (rows == 0) return SV_OK;
  if (!hidden || !weight || !out_max || !out_lse) return SV_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(hidden) % 16 != 0 || reinterpret_cast<uintptr_t>(weight) % 16 != 0)
    return SV_ERR_INVALID_ARG;
  if (out_zx && !ids) return SV_ERR_INVALID_ARG;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  const int sms = sm_count(dev);
  if (sms <= 0) return SV_ERR_CUDA;
  sv::HeadParams P;
  memset(&P, 0, sizeof(P));
  P.R = rows;
  P.d = d;
  P.V = V;
  P.c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  P.inv_t = static_cast<float>(1.0 / static_cast<double>(temperature));
  P.ids = ids;
  P.out_logits = out_logits;
  sv::head_split(rows, V, sms, &P.nsplit, &P.tiles_per_split, &P.ntiles);
  sv_status st = SV_OK;
  StreamRes* r = resources(dev, s, sizeof(Workspace) + sv::head_part_bytes(rows, P.nsplit), &st);
  if (!r) return st;
  P.part = reinterpret_cast<float4*>(r->ws + 1);
  P.err = &r->ws->error;
  cudaError_t e = sv::launch_head_gemm(sv::HEAD_STATS, hidden, hidden_stride, weight,
                                       weight_stride, P, sv::head_ctas(sms), s);
  if (e == cudaSuccess)
    e = sv::launch_head_combine(P, out_max, out_lse, out_zx, out_argmax, nullptr, s);
  if (e == cudaErrorNotSupported) return SV_ERR_UNSUPPORTED;
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status spec_verify_hidden(int B, int K, int V, int d, const void* hidden_target,
                             long long target_row_stride, const void* hidden_draft,
                             long long draft_row_stride, const void* weight,
                             long long weight_stride, const int32_t* draft_tokens,
                             const int32_t* draft_lens, const float* uniforms, float temperature,
                             float beta, int bias_k, const int* fanout, int mode,
                             int32_t* out_accept_len, int32_t* out_tokens,
                             int32_t* out_residual_topF, void* stream) {
  // V <= 2^18 as for spec_verify: the draw's masses (each at most 1 in 2^-44 units per id) then
  // sum below 2^63 even for a flat row
  if (B < 0 || K < 1 || K > 8 || V < 1 || V > (1 << 18) || d < 64 || d % 64 != 0)
    return SV_ERR_INVALID_ARG;
  if (mode != SV_MODE_GREEDY && mode != SV_MODE_STOCHASTIC) return SV_ERR_INVALID_ARG;
  const bool greedy = mode == SV_MODE_GREEDY;
  if (!greedy && !finite_in(temperature, 1e-4f, 1e4f)) return SV_ERR_INVALID_ARG;
  if (!greedy && (!(std::isfinite(beta) && beta > 0.f && beta <= 1.f) || bias_k < 0 || bias_k > 8))
    return SV_ERR_INVALID_ARG;
  int fan[sv::kMaxK] = {0};
  int fmax = 0;
  if (fanout) {
    if (greedy) return SV_ERR_INVALID_ARG;
    for (int i = 0; i < K; ++i) {
      if (fanout[i] < 0 || fanout[i] > 8) return SV_ERR_INVALID_ARG;
      fan[i] = fanout[i];
      fmax = std::max(fmax, fan[i]);
    }
  }
  if ((fmax > 0 && !out_residual_topF) || (!fanout && out_residual_topF))
    return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!hidden_target || !weight || !draft_tokens || !draft_lens || !out_accept_len ||
      !out_tokens)
    return SV_ERR_INVALID_ARG;
  if (!greedy && (!hidden_draft || !uniforms)) return SV_ERR_INVALID_ARG;
  if (target_row_stride < d || weight_stride < d || (!greedy && draft_row_stride < d))
    return SV_ERR_INVALID_ARG;
  if (!aligned16(hidden_target, target_row_stride, 2) || !aligned16(weight, weight_stride, 2) ||
      (!greedy && !aligned16(hidden_draft, draft_row_stride, 2)))
    return SV_ERR_INVALID_ARG;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  const int sms = sm_count(dev);
  if (sms <= 0) return SV_ERR_CUDA;
  sv::HvProblem p;
  p.B = B;
  p.K = K;
  p.V = V;
  p.d = d;
  p.greedy = greedy ? 1 : 0;
  p.ht = static_cast<const uint16_t*>(hidden_target);
  p.hts = target_row_stride;
  p.hd = greedy ? nullptr : static_cast<const uint16_t*>(hidden_draft);
  p.hds = greedy ? d : draft_row_stride;
  p.W = static_cast<const uint16_t*>(weight);
  p.ws = weight_stride;
  p.x = draft_tokens;
  p.lens = draft_lens;
  p.uni = greedy ? nullptr : uniforms;
  p.temperature = greedy ? 1.f : temperature;
  p.beta = greedy ? 1.f : beta;
  p.bias_k = (greedy || beta >= 1.f) ? 0 : bias_k;
  p.fmax = fmax;
  for (int i = 0; i < 8; ++i) p.fan[i] = i < sv::kMaxK ? fan[i] : 0;
  p.out_acc = out_accept_len;
  p.out_tok = out_tokens;
  p.out_topf = fmax > 0 ? out_residual_topF : nullptr;
  sv_status st = SV_OK;
  StreamRes* r = resources(dev, s, sizeof(Workspace) + sv::hv_workspace_bytes(p, sms), &st);
  if (!r) return st;
  const cudaError_t e = sv::hv_run(p, sms, r->ws + 1, &r->ws->error, s);
  if (e == cudaErrorNotSupported) return SV_ERR_UNSUPPORTED;
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

const char* spec_verify_status_string(sv_status status) {
  switch (status) {
    case SV_OK: return "ok";
    case SV_ERR_INVALID_ARG: return "invalid argument";
    case SV_ERR_UNSUPPORTED: return "unsupported shape or configuration";
    case SV_ERR_CUDA: return "CUDA runtime error";
    case SV_ERR_DEVICE_TIMEOUT: return "a device-side bounded wait gave up";
  }
  return "unknown status";
}

sv_status sv_wait_probe(unsigned int budget_us, void* stream) {
  if (budget_us == 0 || budget_us > 1000000u) return SV_ERR_INVALID_ARG;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0, khz = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  if (cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev) != cudaSuccess || khz <= 0)
    khz = 2000000;
  std::lock_guard<std::mutex> lock(g_mu);
  sv_status st = SV_OK;
  StreamRes* r = resources(dev, s, sizeof(Workspace), &st);
  if (!r) return st;
  const long long cycles = static_cast<long long>(budget_us) * (khz / 1000);
  return sv::launch_wait_probe(cycles, &r->ws->error, s) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status sv_wait_probe_at(unsigned int budget_us, int target, void* workspace, void* stream) {
  if (budget_us == 0 || budget_us > 1000000u) return SV_ERR_INVALID_ARG;
  if (target != SV_PROBE_NOALLOC && target != SV_PROBE_WORKSPACE) return SV_ERR_INVALID_ARG;
  if (target == SV_PROBE_WORKSPACE &&
      (!workspace || reinterpret_cast<uintptr_t>(workspace) % 16 != 0))
    return SV_ERR_INVALID_ARG;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0, khz = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  if (cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev) != cudaSuccess || khz <= 0)
    khz = 2000000;
  Workspace* ws = static_cast<Workspace*>(workspace);
  if (target == SV_PROBE_NOALLOC) {
    std::lock_guard<std::mutex> lock(g_mu);
    void* p = nullptr;
    const sv_status st = noalloc_array(dev, true, &p);
    if (st != SV_OK) return st;
    ws = static_cast<Workspace*>(p);
  }
  const long long cycles = static_cast<long long>(budget_us) * (khz / 1000);
  return sv::launch_wait_probe(cycles, &ws->error, s) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status sv_hbm_read_probe(const void* buf, size_t bytes, unsigned long long* out_checksum,
                            void* stream) {
  if (!buf || !out_checksum || bytes == 0 || bytes % 16 != 0 ||
      reinterpret_cast<uintptr_t>(buf) % 16 != 0)
    return SV_ERR_INVALID_ARG;
  return sv::launch_probe(buf, bytes, out_checksum, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? SV_OK
             : SV_ERR_CUDA;
}

}  // extern "C"

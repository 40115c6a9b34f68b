/*
 * spec_verify.h -- batched speculative-sampling verify step on one GPU (sm_103a).
 *
 * One call verifies B sequences. Sequence b carries L_b = draft_lens[b] draft tokens
 * x[b][0..L_b-1] (1 <= L_b <= K), the target logits of positions 0..L_b (one parallel target
 * pass scores every draft position plus the position after the last draft) and, in stochastic
 * mode, the draft logits of positions 0..L_b-1.
 *
 * What it computes (per sequence, positions in order):
 *   p_i = softmax(z_t[b][i] / T), q_i = softmax(z_d[b][i] / T) over the whole vocabulary
 *     (Kangaroo self-speculative decoding guide, "Exit 1", the softmax draft head).
 *   q'_i = q_i with the probabilities of its bias_k most likely ids (largest draft logit, ties
 *     to the lower id) scaled by beta and renormalised; q' = q when beta == 1 or bias_k == 0
 *     ("Speculative Speculative Decoding" summary, "Key claims" and "Method": Saguaro
 *     sampling down-weights the most likely draft tokens; drafts must be drawn from q').
 *   Draft i is accepted iff u[b][i] < p_i(x_i) / q'_i(x_i) (Kangaroo guide, section
 *     "3. Lossless Speculative Verification"; glossary "speculative decoding llm", "Why It
 *     Produces Identical Outputs"). q'(x) == 0 counts as an infinite ratio when p(x) > 0.
 *   Verification stops at the first rejection a_b (Kangaroo guide, section 3). The token at
 *     position a_b is drawn from max(p_a - q'_a, 0) normalised (same passages) or, when every
 *     draft was accepted (a_b = L_b), from p_{L_b} (bonus token; SSD summary, "Method": the
 *     outcome is the accepted-prefix length plus the bonus id). A zero residual mass falls
 *     back to p_a.
 *   The draw is the inverse CDF over ascending ids: the smallest v with C(v) > u[b][K] * W.
 *   Greedy mode (LayerSkip guide, "Systems Mechanics", Verification Phase and Prefix
 *     Acceptance): accept while x_i equals argmax z_t[b][i] (ties to the lower id), then emit
 *     the target argmax at a_b (including the bonus position when all drafts match).
 *   Optional top-F ids (SSD summary, "Key claims", capped geometric fan-out across positions):
 *     for i < L_b, the first fanout[i] ids of draft row i ordered by logit (descending, ties to
 *     the lower id), the bonus-token guesses a speculation cache would prepare.
 *
 * Outputs: out_accept_len[b] = a_b; out_tokens[b] = x[b][0..a_b-1], the sampled token, then -1.
 * A sequence whose inputs are unusable (L_b outside [1, K], a draft id outside [0, V), a used
 * uniform outside [0, 1), or a needed logit row holding NaN / +inf or only -inf) gets
 * out_accept_len[b] = -1 and all tokens -1. A sequence that a device-side bounded wait gave up
 * on gets -2 (see spec_verify_device_error). The needed rows are target rows 0..a_b and draft
 * rows 0..min(a_b, L_b - 1), plus every draft row below L_b when top-F ids are requested;
 * rows after the outcome is fixed are never read, so padding rows may hold anything.
 *
 * Memory: every pointer argument of spec_verify / spec_verify_debug / spec_verify_ws is DEVICE
 * memory owned by the caller; the library keeps no reference after the call returns. Logit
 * rows are contiguous; row r of sequence b starts at element (b * rows + r) * row_stride with
 * rows = K + 1 (target) or K (draft). All calls are asynchronous on `stream` (a cudaStream_t,
 * NULL for the legacy default stream) and do not synchronise, except spec_verify_host and
 * spec_verify_device_error.
 *
 * Errors: arguments are checked on the host before anything is launched; a bad argument
 * returns SV_ERR_INVALID_ARG and launches nothing. Shapes the kernels do not handle return
 * SV_ERR_UNSUPPORTED. A failing CUDA runtime call returns SV_ERR_CUDA. Nothing aborts, throws
 * or traps.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SV_OK = 0,
  SV_ERR_INVALID_ARG = 1,
  SV_ERR_UNSUPPORTED = 2,
  SV_ERR_CUDA = 3,
  SV_ERR_DEVICE_TIMEOUT = 4
} sv_status;

typedef enum { SV_DTYPE_F32 = 0, SV_DTYPE_BF16 = 1 } sv_dtype;
typedef enum { SV_MODE_GREEDY = 0, SV_MODE_STOCHASTIC = 1 } sv_mode;

/* Shapes and options, in host memory. */
typedef struct {
  int B;                        /* sequences, >= 0 (0 launches nothing)                       */
  int K;                        /* maximum draft length, 1..8                                 */
  int V;                        /* vocabulary size, 1..262144                                 */
  sv_dtype dtype;               /* element type of both logit tensors                         */
  long long target_row_stride;  /* elements between consecutive target rows, >= V            */
  long long draft_row_stride;   /* elements between consecutive draft rows, >= V             */
  int bias_k;                   /* size of the beta-down-weighted set, 0..8 (0 = none)        */
  const int* fanout;            /* host array of K entries F_i in 0..8, or NULL = no top-F    */
  int cluster_hint;             /* CTAs that share one sequence's rows: 0 = chosen by the
                                   library, else 1, 2, 4, 8 or 16. With 0 the library may also
                                   take a small batch without clusters (every row in flight
                                   at once; see spec_verify_route); a nonzero hint always
                                   walks the positions with clusters of that size             */
} sv_problem;

/*
 * The verify step (see the top of this file for what it computes).
 *   target_logits  [B][K+1][target_row_stride] of dtype.
 *   draft_logits   [B][K][draft_row_stride] of dtype; may be NULL in greedy mode.
 *   draft_tokens   [B][K] int32; entries at i >= L_b are ignored.
 *   draft_lens     [B] int32 in 1..K, or NULL (every sequence has K drafts).
 *   uniforms       [B][K+1] float32 in [0, 1): u[b][i] drives accept test i, u[b][K] the final
 *                  draw. Ignored (may be NULL) in greedy mode.
 *   temperature    stochastic mode: finite, in [1e-4, 1e4]. Ignored in greedy mode.
 *   beta           stochastic mode: in (0, 1]. Ignored in greedy mode.
 *   mode           SV_MODE_GREEDY or SV_MODE_STOCHASTIC.
 *   out_accept_len [B] int32; out_tokens [B][K+1] int32.
 *   out_residual_topF [B][K][max_i F_i] int32, -1 padded; required iff prob->fanout != NULL
 *                  (stochastic mode only), otherwise must be NULL.
 *   stream         cudaStream_t.
 * The library keeps a zero-initialised workspace per (device, stream) of
 * spec_verify_workspace_bytes(prob) bytes, created (or enlarged for a larger B) by the first
 * such call; make that call outside stream capture. Calls that may run at the same time must use
 * different streams.
 */
sv_status spec_verify(const sv_problem* prob, const void* target_logits,
                      const void* draft_logits, const int32_t* draft_tokens,
                      const int32_t* draft_lens, const float* uniforms, float temperature,
                      float beta, int mode, int32_t* out_accept_len, int32_t* out_tokens,
                      int32_t* out_residual_topF, void* stream);

/*
 * The launch spec_verify would make for this problem on the current device: CTAs that share
 * one sequence (*cluster), clusters launched (*clusters) and dynamic shared memory per CTA
 * (*smem_bytes). Host-side query; any output pointer may be NULL. Returns the same argument
 * and shape errors as spec_verify (temperature and beta are not checked here).
 */
sv_status spec_verify_plan(const sv_problem* prob, int mode, int* cluster, int* clusters,
                           size_t* smem_bytes);

/*
 * Which kernels spec_verify takes for this problem on the current device (*route) and how many
 * launches one call makes (*launches). Routes: SV_ROUTE_WALK, the chained cluster walk (one
 * launch for a greedy batch; three for a stochastic one, whose draws two launches chained after
 * the walk take as the walk decides each sequence; two with the top-8 prepass over the draft
 * rows for a bias set or top-F ids, the walk then drawing itself);
 * SV_ROUTE_GREEDY_ROWS, greedy batches whose padded target rows fit in 64 MiB (an argmax per row
 * slice of every target row, then one warp per sequence: two launches); SV_ROUTE_SMALL,
 * stochastic batches whose padded rows fit in 256 MiB (every row's statistics, the draw's slice
 * masses, one pick per sequence: three launches, four with the top-8 prepass). A nonzero
 * cluster_hint always walks. spec_verify_ws takes the walk as well when its workspace has no
 * room for the other routes' partials. Host-side query; either output may be NULL; the same
 * errors as spec_verify_plan.
 */
#define SV_ROUTE_WALK 0
#define SV_ROUTE_GREEDY_ROWS 1
#define SV_ROUTE_SMALL 2
sv_status spec_verify_route(const sv_problem* prob, int mode, int* route, int* launches);

/* Bytes of device workspace spec_verify_ws needs for this problem (256: the sequence queue and
 * the error word; the size does not depend on the problem). */
size_t spec_verify_workspace_bytes(const sv_problem* prob);

/*
 * spec_verify with a caller-owned workspace of spec_verify_workspace_bytes() bytes of device
 * memory, 16-byte aligned and zero-filled before its first use; the kernel leaves it ready for
 * the next call. Calls that may overlap on the GPU must use different workspaces. Same
 * arguments and errors as spec_verify otherwise. A device-side bounded wait that gives up
 * raises the error word inside this workspace; spec_verify_workspace_error reads it.
 */
sv_status spec_verify_ws(const sv_problem* prob, const void* target_logits,
                         const void* draft_logits, const int32_t* draft_tokens,
                         const int32_t* draft_lens, const float* uniforms, float temperature,
                         float beta, int mode, int32_t* out_accept_len, int32_t* out_tokens,
                         int32_t* out_residual_topF, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * spec_verify for callers that cannot allocate device memory. This entry point has no
 * counterpart in the method; it exists for the integration. Code running under an allocator
 * that forbids cudaMalloc (a serving loop that reserved all device memory up front, or a
 * runtime whose allocations must go through its own pool), or on a path where a cudaMalloc
 * would synchronise the device, cannot let the library create its workspace. This variant
 * allocates nothing: its workspace is a fixed array inside the library's device code (256
 * bytes on every GPU that loads the library, held until the process exits); it accepts at
 * most 65536 sequences, a larger B returns SV_ERR_UNSUPPORTED. Inputs and outputs are the
 * caller's device buffers, exactly as for spec_verify, and the results are identical. With
 * only that fixed array it always takes the cluster walk (route 0 of spec_verify_route): the
 * small-batch routes and the top-8 prepass need a larger workspace, so small batches run
 * slower than through spec_verify (greedy B=8, V=32000: about 15 us instead of 11 us).
 * The first call on a device (with that device current) looks the array up with
 * cudaGetSymbolAddress; make that first call before any stream capture. Each call clears the
 * array's queue counters with an asynchronous memset on `stream`, then launches; the array's
 * error word is kept until spec_verify_device_error reads and clears it. Every call shares
 * the one array, so calls that may overlap on the GPU (different streams, or different host
 * threads) race and must not be issued.
 */
sv_status spec_verify_noalloc(const sv_problem* prob, const void* target_logits,
                              const void* draft_logits, const int32_t* draft_tokens,
                              const int32_t* draft_lens, const float* uniforms,
                              float temperature, float beta, int mode, int32_t* out_accept_len,
                              int32_t* out_tokens, int32_t* out_residual_topF, void* stream);

/*
 * spec_verify plus per-position diagnostics, for parity checks. It reads every row a sequence
 * has (target rows 0..L_b, draft rows 0..L_b-1), not only the needed ones, and fills
 *   out_lse_t [B][K+1]  log-normaliser of z_t/T (natural log),
 *   out_lse_d [B][K]    log-normaliser of z_d/T,
 *   out_p_x   [B][K]    p_i(x_i),
 *   out_q_x   [B][K]    q'_i(x_i),
 * float32, NaN where a row was not read or holds no distribution (stochastic mode only; the
 * four pointers are device memory and may individually be NULL). Accept lengths and tokens
 * are those spec_verify returns.
 */
sv_status spec_verify_debug(const sv_problem* prob, const void* target_logits,
                            const void* draft_logits, const int32_t* draft_tokens,
                            const int32_t* draft_lens, const float* uniforms,
                            float temperature, float beta, int mode, int32_t* out_accept_len,
                            int32_t* out_tokens, int32_t* out_residual_topF, float* out_lse_t,
                            float* out_lse_d, float* out_p_x, float* out_q_x, void* stream);

/*
 * End-to-end form: every array argument is HOST memory (pinned memory makes the copies
 * asynchronous; pageable memory works too). The call copies the rows each sequence has to the
 * device (target rows 0..L_b, draft rows 0..L_b-1; draft_lens must then be a host array or
 * NULL), runs spec_verify on `stream`, copies the outputs back and synchronises the stream.
 * The device staging buffers are owned by the library (per device and stream) and grow on
 * demand. Returns SV_ERR_DEVICE_TIMEOUT if a bounded wait gave up during the call.
 */
sv_status spec_verify_host(const sv_problem* prob, const void* target_logits,
                           const void* draft_logits, const int32_t* draft_tokens,
                           const int32_t* draft_lens, const float* uniforms, float temperature,
                           float beta, int mode, int32_t* out_accept_len, int32_t* out_tokens,
                           int32_t* out_residual_topF, void* stream);

/*
 * Synchronises `stream` and reports whether a device-side bounded wait gave up since the last
 * check (SV_ERR_DEVICE_TIMEOUT; the sequences it gave up on read -2) in a call that used the
 * library's own workspaces on the current device: spec_verify, spec_verify_debug and
 * spec_verify_host on `stream` (their per-stream workspace), and spec_verify_noalloc on any
 * stream (its fixed array, shared by every stream of the device). Clears both error words.
 * SV_OK otherwise. A call with a caller-owned workspace (spec_verify_ws) reports through
 * spec_verify_workspace_error instead.
 */
sv_status spec_verify_device_error(void* stream);

/*
 * The same report for a caller-owned workspace of spec_verify_ws: synchronises `stream`, reads
 * the workspace's error word (device memory, 16-byte aligned), clears it, and returns
 * SV_ERR_DEVICE_TIMEOUT if a bounded wait of a call that used it gave up, SV_OK if not,
 * SV_ERR_INVALID_ARG for a null or misaligned pointer.
 */
sv_status spec_verify_workspace_error(void* workspace, void* stream);

/*
 * The draft generator's step, for `rows` independent rows of draft-head logits (row r at element
 * r * row_stride of draft_logits, device memory of dtype; uniforms [rows] fp32 in [0, 1)):
 *   out_tokens[r] = a token drawn from q'_r, the beta-biased softmax(z_r / T) (bias set: the
 *     bias_k ids with the largest logit, ties to the lower id, probabilities scaled by beta and
 *     renormalised; Saguaro summary, "Method": drafts are drawn from q'), by the same inverse CDF
 *     the verify step uses: the smallest v with C(v) > uniforms[r] * W over ascending ids;
 *   out_conf[r] = max_v q_r(v), the unbiased softmax's largest probability (Kangaroo guide,
 *     "Exit 2": c_i = max_v P-hat(v), drafting halts when c_i < tau);
 *   out_exit[r] (may be NULL) = 1 if out_conf[r] < tau, else 0.
 * A row holding NaN / +inf or only -inf gives token -1, conf NaN, exit -1. Same temperature and
 * beta checks as spec_verify; bias_k in 0..8. Asynchronous on `stream`, on the stream's workspace
 * (allocated on first use, like spec_verify's); a device-side wait that gave up is reported by
 * spec_verify_device_error on the same stream.
 */
sv_status spec_draft_sample(int rows, int V, sv_dtype dtype, long long row_stride,
                            const void* draft_logits, const float* uniforms, float temperature,
                            float beta, int bias_k, float tau, int32_t* out_tokens,
                            float* out_conf, int32_t* out_exit, void* stream);

/*
 * Exact-residual top-F ids: for every sequence b and position i < L_b, out_r2[b][i][f] for
 * f < F_i (prob->fanout, required) = the f-th id of the residual r_i = max(p_i - q'_i, 0) ordered by
 * value (descending, ties to the lower id), restricted to r > 0; -1 elsewhere and for invalid
 * sequences or rows. These are the ids the verify step's residual draw is most likely to emit
 * after a rejection at i, to be compared with the top-F draft ids a speculation cache prepares
 * (Saguaro summary, "Key claims"). With the outputs of a spec_verify call on the same inputs
 * (accept_len, out_tokens, and its out_residual_topF as r1_topF, all device memory), out_hit[b] =
 * 1 if the drawn token at the decided position a_b < L_b is among r1_topF[b][a_b][0..F_{a_b}), 0
 * if not, -1 when every draft was accepted or the sequence is invalid; pass all four as NULL to
 * skip. out_r2 is [B][K][max_i F_i] int32. Same shape and scalar checks as spec_verify
 * (prob->cluster_hint is not used). Asynchronous on `stream`, on the stream's workspace.
 */
sv_status spec_residual_topf(const sv_problem* prob, const void* target_logits,
                             const void* draft_logits, const int32_t* draft_lens,
                             float temperature, float beta, const int32_t* accept_len,
                             const int32_t* out_tokens, const int32_t* r1_topF, int32_t* out_r2,
                             int32_t* out_hit, void* stream);

/*
 * The LM head fused with the softmax statistics (Kangaroo guide, "Exit 1": the head is
 * Softmax(W h)): logits z = h W^T for `rows` hidden states h (bf16, rows of d elements at row
 * stride hidden_stride) and a head W (bf16, V rows of d at row stride weight_stride), reduced on
 * the GPU to, per row r:
 *   out_max[r] = max_v z[r][v],
 *   out_lse[r] = log sum_v exp(z[r][v] / T)   (natural log),
 *   out_zx[r]  = z[r][ids[r]] (NaN when ids[r] is outside [0, V)); out_zx may be NULL,
 *   out_argmax[r] = the lowest v with z[r][v] = out_max[r] (-1 for a row with a NaN); may be NULL.
 * No logit is written to memory unless out_logits ([rows][V] fp32, for tests) is given. The
 * logits are accumulated in fp32 from bf16 products on the tensor cores. d must be a multiple
 * of 64, strides multiples of 8 elements, both pointers 16-byte aligned; V <= 2^24.
 * Asynchronous on `stream`, on the stream's workspace; SV_ERR_UNSUPPORTED when the driver's
 * tensor-map encoder cannot be had.
 */
sv_status spec_lmhead_stats(int rows, int d, int V, const void* hidden, long long hidden_stride,
                            const void* weight, long long weight_stride, float temperature,
                            const int32_t* ids, float* out_max, float* out_lse, float* out_zx,
                            int32_t* out_argmax, float* out_logits, void* stream);

/*
 * The verify step taken from hidden states instead of logits (Kangaroo guide, "Exit 1" and
 * section 3; LayerSkip guide, "Verification Phase": the early-exit draft and the full model share
 * one LM head). The logits of every row are z = h W^T with the head W [V][d] (bf16, row stride
 * weight_stride), for the target hidden states [B][K+1] rows (bf16, target_row_stride elements
 * apart) and the draft hidden states [B][K] rows (draft_row_stride apart; unused and may be NULL
 * in greedy mode). The outcome is the one spec_verify gives for those logits with the same
 * beta, bias set size (bias_k, 0..8) and top-F widths (fanout: a host array of K entries in
 * 0..8, or NULL; stochastic mode only): out_accept_len [B], out_tokens [B][K+1] and, iff fanout
 * is given, out_residual_topF [B][K][max_i F_i], in the same layout, with the same validity
 * rules and uniforms (with top-F ids every draft row below L_b is needed). Only the rows each
 * sequence has are scored (target 0..L_b, draft 0..L_b-1); each row is reduced on the tensor
 * cores to its maximum, softmax sum, logit at the draft id and argmax (with a bias set or top-F
 * ids also to its 8 largest logits per vocabulary range, merged per draft row before the
 * decision), and the two rows of the decided position are scored again for the draw, so no row
 * of logits is written to memory. Logits are accumulated in fp32 from bf16 products.
 * d must be a multiple of 64, K <= 8, V <= 2^18; hidden states and head 16-byte aligned, with
 * row strides that are multiples of 8 elements. Asynchronous on `stream`, on the stream's
 * workspace (grown on demand: about B (2K+1) d 2 bytes for the packed rows plus 16 bytes per
 * sequence and 16 ids for the residual masses); device-side failures are read with
 * spec_verify_device_error.
 */
sv_status spec_verify_hidden(int B, int K, int V, int d, const void* hidden_target,
                             long long target_row_stride, const void* hidden_draft,
                             long long draft_row_stride, const void* weight,
                             long long weight_stride, const int32_t* draft_tokens,
                             const int32_t* draft_lens, const float* uniforms, float temperature,
                             float beta, int bias_k, const int* fanout, int mode,
                             int32_t* out_accept_len, int32_t* out_tokens,
                             int32_t* out_residual_topF, void* stream);

/* A static, human-readable name for a status code. */
const char* spec_verify_status_string(sv_status status);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */

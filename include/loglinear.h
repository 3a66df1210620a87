/*
 * loglinear.h — C ABI of the log-linear attention library (sm_103a).
 *
 * The operation (page "论文阅读：Log-Linear Attention — 基于 Fenwick 树与层次矩阵的对数线性
 * 复杂度注意力机制", sections 并行形式 and 与已有模型的组合; page "算力终结者来了！…", section
 * 结构矩阵):
 *
 *     O = (Q K^T ⊙ M^S ⊙ M^H) V,
 *     M^S[t,s] = prod_{r=s+1..t} a_r        (Mamba-2 scalar decay; all ones without it)
 *     M^H[t,s] = lambda[t, l(t,s)]           (Fenwick level l(t,s) of source s from query t)
 *
 * and its recurrent decode step with the lssb rule (first page, section 解码：基于 lssb 的
 * 状态更新).  l(t,t) = 0; for s < t, l(t,s) is the level of the Fenwick bucket of t holding s
 * (first page, section 层级判定算法), equal to the bit length of (t XOR s).
 *
 * Conventions shared by every entry point:
 *   - All tensor arguments are DEVICE pointers to dense row-major arrays, owned by the
 *     caller (loglinear_fwd_strided takes strided q, k, v and out).  The library never allocates, frees or synchronises; all work
 *     is enqueued on `stream` (NULL = the legacy default stream) and is asynchronous.
 *   - Sizes are element counts.  Positions t are 0-based and must fit in int32.
 *   - Every call validates its arguments on the host before launching anything and
 *     returns an ll_status code; on a non-zero status nothing has been enqueued, except
 *     LL_ERR_CUDA, which reports a failed launch (the message is in
 *     loglinear_last_cuda_error()).
 *   - `out` must not alias any input.  Calls are thread-safe.
 */
#ifndef LOGLINEAR_H
#define LOGLINEAR_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LL_API __attribute__((visibility("default")))
#else
#define LL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* ll_stream_t;

typedef enum {
  LL_OK = 0,
  LL_ERR_INVALID = 1,      /* a required pointer is NULL, a size is negative, unknown enum */
  LL_ERR_SHAPE = 2,        /* sizes violate the method: chunk not a power of two, too few levels */
  LL_ERR_DTYPE = 3,        /* unknown dtype code */
  LL_ERR_UNSUPPORTED = 4,  /* valid problem outside this build's kernels (e.g. head dim > 128) */
  LL_ERR_CUDA = 5,         /* a CUDA call or kernel launch failed */
  LL_ERR_WORKSPACE = 6,    /* workspace NULL or smaller than loglinear_fwd_workspace_size() */
  LL_ERR_ALIGN = 7         /* a pointer is not aligned as the chosen kernel path requires */
} ll_status;

typedef enum { LL_F32 = 0, LL_BF16 = 1 } ll_dtype;

/* Kernel path of the forward.  AUTO takes the tensor-core path when it applies (bf16
 * inputs, dk = 128, dv = 64 or 128) and the fp32 CUDA-core path otherwise. */
typedef enum { LL_PATH_AUTO = 0, LL_PATH_SIMT = 1, LL_PATH_TC = 2 } ll_path;

/* Library version, (major << 16) | minor. */
LL_API int loglinear_version(void);

/* Human-readable name of a status code (static string). */
LL_API const char* loglinear_status_string(int status);

/* Text of the last CUDA error seen by this thread (static per-thread buffer). */
LL_API const char* loglinear_last_cuda_error(void);

/* Path the forward would take for these arguments (LL_PATH_SIMT or LL_PATH_TC), or a
 * negative ll_status if the request is invalid. */
LL_API int loglinear_fwd_resolve_path(int64_t dk, int64_t dv, int chunk, int in_dtype, int path);

/*
 * Workspace bytes loglinear_fwd needs (written to *bytes).  The workspace holds the
 * per-chunk states U_i (chunk-local decayed sums of k v^T), the Fenwick block states the
 * inter-chunk readout uses, and the per-chunk log decays.  It is scratch: its content on
 * entry does not matter and is not meaningful on exit.
 */
LL_API int loglinear_fwd_workspace_size(int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                                 int chunk, int in_dtype, int path, size_t* bytes);

/*
 * Chunked-parallel forward (first page, sections 矩阵分解 and 两阶段计算; second page,
 * section 高效训练算法): intra-chunk masked attention for the levels inside a chunk, per-
 * chunk states, a level scan over Fenwick block pairs of chunks, and a lambda-weighted
 * readout of the block states fused into the output epilogue.
 *
 *   q, k    [B, T, Hqk, dk] in_dtype (LL_F32 or LL_BF16).  Hqk q/k heads shared by the
 *                           H value heads in contiguous groups of H / Hqk: head h reads
 *                           q/k head h / (H / Hqk).  Hqk = H is one q/k per head; Hqk = 1
 *                           shares one q/k across all heads (Mamba-2's multi-value form).
 *                           1 <= Hqk <= H and H % Hqk == 0, else LL_ERR_SHAPE.
 *   v       [B, T, H, dv]   in_dtype
 *   log_a   [B, T, H]       fp32, log of the decay a_t (<= 0 expected); NULL = no decay
 *   lambda  [B, T, H, L]    fp32 level weights lambda[t, l]; L >= bit_length(T-1) + 1;
 *                           levels above bit_length(T-1) are not read
 *   out     [B, T, H, dv]   out_dtype (LL_F32 or LL_BF16), fully overwritten
 *   chunk   C, a power of two.  The result does not depend on C: the decomposition into
 *           an intra-chunk block D plus inter-chunk levels is exact for any C.  The fp32
 *           path works on chunks of min(C, 64) tokens; the tensor-core path on 128-token
 *           tiles (levels <= 7 in the dense intra-tile product, the rest through block
 *           states).
 *   T need not be a multiple of C (the last chunk is partial).  B, T or H = 0 is a no-op.
 *   workspace: device scratch of at least loglinear_fwd_workspace_size() bytes, 256-byte
 *           aligned.  Two calls that run concurrently need two workspaces.
 * Errors: LL_ERR_INVALID, LL_ERR_SHAPE, LL_ERR_DTYPE, LL_ERR_UNSUPPORTED (dk or dv > 128;
 * LL_PATH_TC forced on a shape other than bf16 with dk = 128, dv in {64, 128}), LL_ERR_WORKSPACE, LL_ERR_ALIGN (tensor-core
 * path: q, k, v, out not 16-byte aligned), LL_ERR_CUDA.
 */
LL_API int loglinear_fwd(const void* q, const void* k, const void* v, const float* log_a,
                  const float* lambda, void* out, int64_t B, int64_t T, int64_t H,
                  int64_t Hqk, int64_t dk, int64_t dv, int64_t L, int chunk, int in_dtype,
                  int out_dtype, int path, void* workspace, size_t workspace_bytes,
                  ll_stream_t stream);

/*
 * Element strides of a [B, T, Hx, width] tensor whose feature dimension (width) is
 * contiguous: the distance between consecutive batch entries, positions and heads.  A
 * dense tensor has {T*Hx*width, Hx*width, width}.  A q, k or v slice of a fused
 * [B, T, H, 3*d] projection has {T*H*3d, H*3d, 3d}.
 */
typedef struct {
  int64_t b, t, h;
} ll_strides;

/*
 * loglinear_fwd on strided q, k, v and out (each pointer addresses element [0, 0, 0, 0];
 * a NULL stride descriptor means dense).  log_a and lambda stay dense.  Same operation,
 * workspace and errors as loglinear_fwd, and in addition:
 *   LL_ERR_INVALID      a negative stride, or out strides under which two output
 *                       elements would share an address;
 *   LL_ERR_ALIGN        tensor-core path: a stride of a dimension longer than 1 that is not
 *                       a multiple of 16 bytes (8 bf16 or 4 fp32 elements), as TMA requires;
 *   LL_ERR_UNSUPPORTED  tensor-core path: a zero stride on a dimension longer than 1.
 * Strides of dimensions of size 1 are ignored.
 */
LL_API int loglinear_fwd_strided(const void* q, const ll_strides* q_strides, const void* k,
                                 const ll_strides* k_strides, const void* v,
                                 const ll_strides* v_strides, const float* log_a,
                                 const float* lambda, void* out, const ll_strides* out_strides,
                                 int64_t B, int64_t T, int64_t H, int64_t Hqk, int64_t dk,
                                 int64_t dv, int64_t L, int chunk, int in_dtype, int out_dtype,
                                 int path, void* workspace, size_t workspace_bytes,
                                 ll_stream_t stream);

/*
 * loglinear_fwd with per-kernel timing: identical work and results, plus cudaEventRecord
 * of stage_events[0] before the first kernel and of stage_events[i+1] after kernel i, on
 * `stream`.  stage_events is a host array of n_events cudaEvent_t handles created by the
 * caller; events past the number of kernels launched are recorded after the last one.
 * *n_kernels (if not NULL) receives the number of kernels launched.
 */
LL_API int loglinear_fwd_with_events(const void* q, const void* k, const void* v,
                                     const float* log_a, const float* lambda, void* out,
                                     int64_t B, int64_t T, int64_t H, int64_t Hqk, int64_t dk,
                                     int64_t dv,
                                     int64_t L, int chunk, int in_dtype, int out_dtype, int path,
                                     void* workspace, size_t workspace_bytes, ll_stream_t stream,
                                     void* const* stage_events, int n_events, int* n_kernels);

/*
 * Prefill for decoding: loglinear_fwd over positions 0..T-1, plus the per-level decode
 * state at position T-1, so that loglinear_decode_step can continue at t = T (first page,
 * sections 循环形式与输出计算 (one state per Fenwick bucket) and 两阶段计算 (block states
 * of chunks)).  Level l of the state is the sum over the level-l Fenwick bucket of T-1 of
 * exp(cum_{T-1} - cum_s) k_s v_s^T.  Levels above the last chunk are the forward's block
 * states of chunks, decayed to T-1; the levels inside the last chunk (and level 0) are
 * summed from k and v; the other levels are zero.
 *   state_out [B, H, L, dk, dv] fp32, fully overwritten (all zero when T = 0).  On the
 *           tensor-core path the levels taken from block states carry their bf16
 *           rounding.
 * The other arguments, the workspace and the errors are those of loglinear_fwd; state_out
 * NULL or not 4-byte aligned is LL_ERR_INVALID / LL_ERR_ALIGN.
 */
LL_API int loglinear_prefill(const void* q, const void* k, const void* v, const float* log_a,
                             const float* lambda, void* out, float* state_out, int64_t B,
                             int64_t T, int64_t H, int64_t Hqk, int64_t dk, int64_t dv,
                             int64_t L, int chunk,
                             int in_dtype, int out_dtype, int path, void* workspace,
                             size_t workspace_bytes, ll_stream_t stream);

/*
 * loglinear_prefill with per-kernel timing, as loglinear_fwd_with_events: stage_events[0]
 * is recorded before the first kernel and stage_events[i+1] after kernel i, the last of
 * which is the kernel that forms the decode state.  T = 0 launches no kernel and records
 * no event (*n_kernels = 0).
 */
LL_API int loglinear_prefill_with_events(const void* q, const void* k, const void* v,
                                         const float* log_a, const float* lambda, void* out,
                                         float* state_out, int64_t B, int64_t T, int64_t H,
                                         int64_t Hqk, int64_t dk, int64_t dv, int64_t L,
                                         int chunk, int in_dtype, int out_dtype, int path,
                                         void* workspace, size_t workspace_bytes,
                                         ll_stream_t stream, void* const* stage_events,
                                         int n_events, int* n_kernels);

/*
 * One decode step at position t for every (b, h) (first page, section 解码：基于 lssb 的
 * 状态更新; slide deck "論文紹介：Log Linear Attention", slide 21).  With l = lssb(t) (index of
 * the lowest set bit of t > 0):
 *   S^(l+1) <- a_t * sum_{j<=l} S^(j);  S^(1..l) <- 0;  S^(j) <- a_t * S^(j) for j > l+1;
 *   S^(0) <- k_t v_t^T;  out = sum_j lambda[j] * S^(j)^T q_t   (non-empty levels only).
 * At t = 0 the state is (re)initialised: S^(0) <- k_0 v_0^T, every other level <- 0.
 * For t > 0 the state must hold the Fenwick states after position t-1: the levels that
 * are empty after t-1 (bit j-1 of t-1 clear, j >= 1) are neither read nor written.
 *
 *   state   [B, H, L, dk, dv] fp32, updated in place, 16-byte aligned
 *   q, k    [B, Hqk, dk] in_dtype (q/k heads shared as in loglinear_fwd);
 *   v       [B, H, dv]   in_dtype
 *   log_a   [B, H] fp32 or NULL (no decay);   lambda [B, H, L] fp32
 *   out     [B, H, dv]   out_dtype, overwritten
 *   t       >= 0, same for every (b, h); L >= bit_length(t) + 1
 * Supported: 1 <= dk <= 128; dv a power of two in [4, 128].
 * Errors: LL_ERR_INVALID, LL_ERR_SHAPE, LL_ERR_DTYPE, LL_ERR_UNSUPPORTED, LL_ERR_ALIGN,
 * LL_ERR_CUDA.
 */
LL_API int loglinear_decode_step(float* state, const void* q, const void* k, const void* v,
                          const float* log_a, const float* lambda, int64_t t, void* out,
                          int64_t B, int64_t H, int64_t Hqk, int64_t dk, int64_t dv,
                          int64_t L, int in_dtype, int out_dtype, ll_stream_t stream);

/*
 * One decode step of Log-Linear Gated DeltaNet at position t for every (b, h).  The pages
 * build the log-linear form of a model by keeping its transition and composing its mask
 * with the Fenwick mask (page "算力终结者来了！…", section 对Mamba-2和门控DeltaNet的对数线性
 * 推广; first page, section 与已有模型的组合); the transition is the published gated delta
 * rule (Yang, Kautz and Hatamizadeh, "Gated Delta Networks", 2024).  With the state
 * stored [d_k][d_v] and A_t = alpha_t (I - beta_t k_t k_t^T), alpha_t = exp(log_a_t):
 *   every level that holds data after t-1:  S^(j) <- A_t S^(j);  then, with l = lssb(t),
 *   S^(l+1) <- sum_{j<=l} S^(j);  S^(1..l) <- 0;  S^(0) <- beta_t k_t v_t^T;
 *   out = sum_j lambda[j] * S^(j)^T q_t   (non-empty levels only).
 * At t = 0 the state is (re)initialised: S^(0) <- beta_0 k_0 v_0^T, every other level <- 0.
 * Lambda constant across levels gives plain Gated DeltaNet; without the k k^T term it is
 * loglinear_decode_step with v scaled by beta.
 *   state   [B, H, L, dk, dv] fp32, updated in place, 16-byte aligned (levels that are
 *           empty after t-1, other than lssb(t)+1, are neither read nor written)
 *   q, k    [B, Hqk, dk] in_dtype (q/k heads shared as in loglinear_fwd); k is expected
 *           to have unit length, as the gated delta rule assumes (not checked)
 *   v       [B, H, dv]   in_dtype
 *   log_a   [B, H] fp32 or NULL (alpha = 1);   beta [B, H] fp32;   lambda [B, H, L] fp32
 *   out     [B, H, dv]   out_dtype, overwritten
 *   t       >= 0, same for every (b, h); L >= bit_length(t) + 1
 * Supported: 1 <= dk <= 128; dv a power of two in [4, 128].
 * Errors: LL_ERR_INVALID (a NULL required pointer, beta included), LL_ERR_SHAPE,
 * LL_ERR_DTYPE, LL_ERR_UNSUPPORTED, LL_ERR_ALIGN, LL_ERR_CUDA.
 */
LL_API int loglinear_gdn_decode_step(float* state, const void* q, const void* k, const void* v,
                                     const float* log_a, const float* beta, const float* lambda,
                                     int64_t t, void* out, int64_t B, int64_t H, int64_t Hqk,
                                     int64_t dk, int64_t dv, int64_t L, int in_dtype,
                                     int out_dtype, ll_stream_t stream);

/*
 * Forward of Log-Linear Gated DeltaNet over a whole sequence, in the recurrent form: the
 * lssb step of loglinear_gdn_decode_step applied at t = 0..T-1 for every (b, h), with every
 * level's state kept on chip (same sources as loglinear_gdn_decode_step).  Equivalently
 *   o_t = sum_{s<=t} lambda[t, level(t, s)] beta_s (q_t^T A_t ... A_{s+1} k_s) v_s,
 * the model's own attention matrix composed with the Fenwick mask.
 *   q, k       [B, T, Hqk, dk] in_dtype, 4-byte aligned (heads shared as in loglinear_fwd);
 *              k is expected to have unit length (not checked)
 *   v          [B, T, H, dv] in_dtype
 *   log_a      [B, T, H] fp32 or NULL (alpha = 1);  beta [B, T, H] fp32
 *   lambda     [B, T, H, L] fp32, L >= bit_length(T-1) + 1
 *   out        [B, T, H, dv] out_dtype, overwritten
 *   state_out  NULL, or [B, H, L, dk, dv] fp32, overwritten with the per-level state after
 *              position T-1 (all zero for T = 0): the state loglinear_gdn_decode_step
 *              continues from at t = T
 * Supported: 1 <= dk, dv <= 128 (dk even for bf16), L <= 64.  The recurrence is sequential
 * in t (one CTA per (b, h, 8 columns of d_v)); the chunked form is not provided.
 * Errors: LL_ERR_INVALID, LL_ERR_SHAPE, LL_ERR_DTYPE, LL_ERR_UNSUPPORTED, LL_ERR_ALIGN,
 * LL_ERR_CUDA.
 */
LL_API int loglinear_gdn_fwd(const void* q, const void* k, const void* v, const float* log_a,
                             const float* beta, const float* lambda, void* out, float* state_out,
                             int64_t B, int64_t T, int64_t H, int64_t Hqk, int64_t dk, int64_t dv,
                             int64_t L, int in_dtype, int out_dtype, ll_stream_t stream);

/*
 * The same forward of Log-Linear Gated DeltaNet in chunks of 64 tokens, fp32 on CUDA cores:
 * per chunk the UT-transform form of the delta rule (Yang et al., "Parallelizing Linear
 * Transformers with the Delta Rule over Sequence Length", 2024) gives the chunk's own
 * attention matrix (masked by the Fenwick levels inside the chunk), its queries carried
 * back to the chunk start, its d_k x d_k transition and its own state; a sequential scan over
 * the chunks then carries every chunk-level block state by the chunk transitions, merges
 * them by the lssb rule on chunk indices and adds their lambda-weighted readout (first
 * page, sections 矩阵分解 and 两阶段计算, with the transition in place of the scalar decay).
 * Arguments as loglinear_gdn_fwd, plus a workspace of
 * loglinear_gdn_fwd_chunked_workspace_size() bytes (256-byte aligned; the chunks' partial
 * outputs, carried queries, transitions and states in fp32).  state_out (optional) receives
 * the decode state after T-1: the chunk-level states from the scan, the levels inside the
 * last chunk from the lssb steps over its tokens alone (then q and k must be 4-byte aligned
 * and, for bf16, dk even).  Otherwise no alignment is needed of q, k, v.  Supported:
 * 1 <= dk, dv <= 128, L <= 64, T <= 2^25.
 * Errors: LL_ERR_INVALID, LL_ERR_SHAPE, LL_ERR_DTYPE, LL_ERR_UNSUPPORTED, LL_ERR_WORKSPACE,
 * LL_ERR_ALIGN, LL_ERR_CUDA.
 */
LL_API int loglinear_gdn_fwd_chunked_workspace_size(int64_t B, int64_t T, int64_t H, int64_t dk,
                                                    int64_t dv, size_t* bytes);
LL_API int loglinear_gdn_fwd_chunked(const void* q, const void* k, const void* v,
                                     const float* log_a, const float* beta, const float* lambda,
                                     void* out, float* state_out, int64_t B, int64_t T,
                                     int64_t H, int64_t Hqk,
                                     int64_t dk, int64_t dv, int64_t L, int in_dtype,
                                     int out_dtype, void* workspace, size_t workspace_bytes,
                                     ll_stream_t stream);

/*
 * Backward of loglinear_fwd (page "算力终结者来了！…", sections 结构矩阵 and 讨论与局限性:
 * training takes the gradients of the attention terms and of the level weights lambda):
 * given dout = dL/dO, the gradients of L with respect to every input, for
 * O = (Q K^T ⊙ M^S ⊙ M^H) V exactly as loglinear_fwd defines it:
 *   dq, dk  [B, T, Hqk, dk]  grad_dtype (summed over the heads that share a q/k head)
 *   dv      [B, T, H, dv]    grad_dtype
 *   dlog_a  [B, T, H] fp32   (required when log_a is given; ignored when log_a is NULL)
 *   dlambda [B, T, H, L] fp32 (levels above bit_length(T-1) receive 0)
 *   dout    [B, T, H, dv]    grad_dtype
 * q, k, v, log_a, lambda, B, T, H, Hqk, dk, dv and L as in loglinear_fwd; no chunk
 * argument: the gradients do not depend on it.  1 <= dk, dv <= 128, L <= 64.  All
 * outputs are fully overwritten.
 * path: LL_PATH_TC computes dq, dk, dv and dlambda on the tensor cores (bf16 inputs and
 *   gradients, dk = 128, dv in {64, 128}; q, k, v, dout, dq, dk, dv 16-byte aligned): the
 *   tensor-core forward, in a form that writes no output, publishes its block states into
 *   the workspace; 128-token tiles take dQ and dlambda from them with tcgen05; the
 *   mirrored states of later tiles that dk and dv read are summed per Fenwick slot with
 *   tcgen05 (fp32 accumulation, the scaled q split into a bf16 high part and residual),
 *   then dK and dV are formed per 128-token tile with tcgen05.  These carry the bf16
 *   roundings of P, P' and of the states.  LL_PATH_SIMT computes everything on CUDA cores
 *   in fp32.
 *   LL_PATH_AUTO takes the tensor cores when they apply.  The workspace size depends on
 *   the path.
 * fwd_workspace: NULL, or, on the tensor-core path, the workspace of a loglinear_fwd call
 *   that ran on the tensor-core path (LL_PATH_TC or AUTO with bf16, dk = 128) over these
 *   same q, k, v, log_a, lambda and sizes, with nothing written to it since.  Its block
 *   states are then read instead of being recomputed by a forward inside this call (the
 *   usual training step: forward, then backward).  The library cannot check that the
 *   contents match the inputs; that is the caller's contract.  It does check, on the GPU,
 *   the layout tag the tensor-core forward leaves in its workspace (sizes and path): a
 *   mismatch raises bit 2 of loglinear_device_error.  fwd_workspace_bytes must
 *   be at least loglinear_fwd_workspace_size() for the forward's arguments
 *   (LL_ERR_WORKSPACE); a non-NULL fwd_workspace on the CUDA-core path is
 *   LL_ERR_UNSUPPORTED.  An empty call (B, T or H zero) returns LL_OK before any of
 *   these checks of pointers and workspaces.
 * workspace: device scratch of at least loglinear_bwd_workspace_size() bytes, 256-byte
 * aligned (recomputed forward states, per-head q and k gradients).
 * Errors: LL_ERR_INVALID (null pointer, negative size, dlog_a NULL with log_a given),
 * LL_ERR_SHAPE (L too small, Hqk not dividing H), LL_ERR_DTYPE, LL_ERR_UNSUPPORTED,
 * LL_ERR_WORKSPACE, LL_ERR_ALIGN (workspace), LL_ERR_CUDA.
 */
LL_API int loglinear_bwd_workspace_size(int64_t B, int64_t T, int64_t H, int64_t Hqk,
                                        int64_t dk, int64_t dv, int64_t L, int in_dtype,
                                        int grad_dtype, int path, size_t* bytes);
LL_API int loglinear_bwd(const void* q, const void* k, const void* v, const float* log_a,
                         const float* lambda, const void* dout, void* dq, void* dk, void* dv,
                         float* dlog_a, float* dlambda, int64_t B, int64_t T, int64_t H,
                         int64_t Hqk, int64_t dk_dim, int64_t dv_dim, int64_t L, int in_dtype,
                         int grad_dtype, int path, const void* fwd_workspace,
                         size_t fwd_workspace_bytes, void* workspace, size_t workspace_bytes,
                         ll_stream_t stream);

/*
 * Reads and clears the device error word of the tensor-core path (synchronises `stream`).
 * *flags = 0 when every wait of the kernels run so far completed.  Bit 0: an mbarrier
 * wait ran out of time (the CTA then skipped its remaining work and its output tile is
 * not valid).  Bit 1: a wait for another tile's published state ran out of time (the
 * output of that tile is not valid).  Bit 2: loglinear_bwd was given a fwd_workspace
 * that a tensor-core loglinear_fwd with the same B, T, H, Hqk and dv did not write (its
 * layout tag does not match; the gradients are not valid).  The launch itself still
 * reported success.
 */
LL_API int loglinear_device_error(ll_stream_t stream, unsigned* flags);

/*
 * loglinear_fwd for callers that cannot allocate device memory.  The paper has no
 * counterpart to this entry point: it exists for callers such as a plugin inside a host
 * application that owns all device memory and hands extensions no allocator, or a
 * real-time loop where cudaMalloc (which may synchronise the device) is not allowed.
 *
 * Same arguments and result as loglinear_fwd, minus the workspace.  The scratch lives in
 * one fixed device array of LL_FWD_NOALLOC_SCRATCH_BYTES that the library declares; every
 * GPU that loads the library's device code holds it until the process exits.  This call
 * allocates nothing (no cudaMalloc, no allocating library routine).
 *   - The first call on a device (with that device current) looks up the array's device
 *     address and caches it with the ID of the current CUDA context; make that first call
 *     before any stream capture.  A call under a different context (after
 *     cudaDeviceReset, or when the application replaced the primary context) looks the
 *     address up again; make it, too, outside any stream capture.
 *   - The ready flags and the tile counter in the array are zeroed by every call, on
 *     `stream`, before the kernel that reads them; everything else in it is written
 *     before it is read.
 *   - All calls share the array and it keeps the last call's contents.  Nothing in it
 *     needs clearing between calls, but calls whose work overlaps on the GPU (another
 *     stream, another host thread) race on it: serialise them.
 *   - A problem whose scratch (loglinear_fwd_workspace_size) exceeds the array is
 *     rejected with LL_ERR_WORKSPACE before any launch.
 * Errors: those of loglinear_fwd; LL_ERR_WORKSPACE for problems too large; LL_ERR_CUDA if
 * the array's address cannot be obtained.
 */
#define LL_FWD_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
LL_API int loglinear_fwd_noalloc(const void* q, const void* k, const void* v,
                                 const float* log_a, const float* lambda, void* out,
                                 int64_t B, int64_t T, int64_t H, int64_t Hqk, int64_t dk,
                                 int64_t dv, int64_t L, int chunk, int in_dtype, int out_dtype,
                                 int path, ll_stream_t stream);

/*
 * Debug view of the forward's level indexing (first page, sections 层级判定算法 and 矩阵
 * 分解): writes levels[t * T + s] (int8, device) for 0 <= s, t < T: the Fenwick level the
 * given path assigns to the pair (query t, source s) through its intra-chunk formula or
 * its inter-chunk block pairing, and -1 for s > t.  chunk and path as in loglinear_fwd
 * (path AUTO resolves as for bf16, dk = dv = 128; the level map does not depend on dv).  T <= 16384.
 */
LL_API int loglinear_debug_level_map(int64_t T, int chunk, int path, int8_t* levels,
                              ll_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LOGLINEAR_H */

// C ABI of the library: argument validation, workspace carving and kernel dispatch.
// Nothing here allocates device memory or synchronises; every check happens on the host
// before the first launch.
#include <cstdio>
#include <cstring>

#include "ll_internal.cuh"

namespace ll {

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

FwdWorkspace fwd_workspace_layout(int64_t B, int64_t H, int64_t N, int64_t dk, int64_t dv,
                                  size_t state_elem_bytes) {
  FwdWorkspace w;
  const size_t states = (size_t)(B * H * N) * (size_t)(dk * dv);
  w.off_U = 0;
  w.off_nodes = align_up(w.off_U + states * state_elem_bytes, 256);
  w.off_lg = align_up(w.off_nodes + states * state_elem_bytes, 256);
  const size_t tiles = (size_t)(B * H * N);
  w.off_nlg = align_up(w.off_lg + tiles * sizeof(float), 256);
  w.off_rdy_u = align_up(w.off_nlg + tiles * sizeof(float), 256);
  w.off_rdy_n = w.off_rdy_u + tiles * sizeof(uint32_t);  // contiguous: zeroed by one memset
  w.off_tick = w.off_rdy_n + tiles * sizeof(uint32_t);
  w.off_tag = w.off_tick + sizeof(uint32_t);  // not zeroed: the forward writes it
  w.total = align_up(w.off_tag + sizeof(uint32_t), 256);
  return w;
}

// Fills levels[t*T + s] with the level the forward's decomposition gives the pair: the
// intra-tile formula when s and t share a tile, else the chunk level of the block pairing
// that contains s's tile, offset by lc; -1 above the diagonal; 127 if no block matched.
__global__ void level_map_kernel(int T, int tile, int lc, int8_t* levels) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)T * T) return;
  const int t = (int)(idx / T), s = (int)(idx - (int64_t)t * T);
  int8_t out = -1;
  if (s <= t) {
    const int j = t / tile, i = s / tile;
    if (i == j) {
      out = (int8_t)fenwick_level((uint32_t)t, (uint32_t)s);
    } else {
      out = 127;
      for (int m = 1; (int64_t(1) << (m - 1)) <= j; ++m) {
        int64_t c;
        if (inter_block(j, m, &c) && i >= c - (int64_t(1) << (m - 1)) && i < c)
          out = (int8_t)(lc + m);
      }
    }
  }
  levels[idx] = out;
}

cudaError_t launch_level_map(int T, int tile, int lc, int8_t* levels, cudaStream_t s) {
  const int64_t n = (int64_t)T * T;
  if (n == 0) return cudaSuccess;
  level_map_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(T, tile, lc, levels);
  return cudaGetLastError();
}

}  // namespace ll

using namespace ll;

namespace {

thread_local char g_cuda_err[256] = "no error";

int cuda_fail(cudaError_t e) {
  snprintf(g_cuda_err, sizeof(g_cuda_err), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return LL_ERR_CUDA;
}

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }
int log2_exact(int64_t x) {
  int n = 0;
  while ((int64_t(1) << n) < x) ++n;
  return n;
}
int bit_length(int64_t x) {
  int n = 0;
  while (x > 0) { ++n; x >>= 1; }
  return n;
}
bool dtype_ok(int d) { return d == LL_F32 || d == LL_BF16; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kSimtMaxChunk = 64;
constexpr int64_t kMaxHeadDim = 128;

// Shared validation of the forward's sizes; fills the resolved path and tile geometry.
int check_fwd_sizes(int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv, int chunk,
                    int in_dtype, int path, int* path_out, int* tile, int64_t* N) {
  if (B < 0 || T < 0 || H < 0 || dk < 1 || dv < 1) return LL_ERR_INVALID;
  if (!dtype_ok(in_dtype)) return LL_ERR_DTYPE;
  if (path != LL_PATH_AUTO && path != LL_PATH_SIMT && path != LL_PATH_TC) return LL_ERR_INVALID;
  if (!is_pow2(chunk)) return LL_ERR_SHAPE;
  if (T > INT32_MAX || B * H > INT32_MAX / 2) return LL_ERR_UNSUPPORTED;
  if (dk > kMaxHeadDim || dv > kMaxHeadDim) return LL_ERR_UNSUPPORTED;
  int p = path;
  if (p == LL_PATH_AUTO)
    p = tc_forward_supported(dk, dv, in_dtype, chunk) ? LL_PATH_TC : LL_PATH_SIMT;
  if (p == LL_PATH_TC && !tc_forward_supported(dk, dv, in_dtype, chunk)) return LL_ERR_UNSUPPORTED;
  *path_out = p;
  // The result does not depend on the chunk length: each path evaluates the same sum on
  // its own tile (CUDA cores: min(C, 64); tensor cores: 128).
  *tile = p == LL_PATH_TC ? kTcTile : (chunk < kSimtMaxChunk ? chunk : kSimtMaxChunk);
  *N = (T + *tile - 1) / *tile;
  return LL_OK;
}

size_t node_bytes(int path) { return path == LL_PATH_TC ? 2 : 4; }

// q/k heads: H = Hqk * (value heads per q/k head); with H = 0 any Hqk >= 0 passes (no-op).
int check_qk_heads(int64_t H, int64_t Hqk) {
  if (Hqk < 0) return LL_ERR_INVALID;
  if (H > 0 && (Hqk < 1 || Hqk > H || H % Hqk != 0)) return LL_ERR_SHAPE;
  return LL_OK;
}

// Strides of a [B, T, Hx, width] tensor with a contiguous feature dimension: the given
// ones (NULL: dense).  A dimension of size 1 takes its dense stride (it is never stepped).
void resolve_strides(const ll_strides* st, int64_t B, int64_t T, int64_t Hx, int64_t width,
                     int64_t* s) {
  dense_strides(s, T, Hx, width);
  if (!st) return;
  if (B > 1) s[0] = st->b;
  if (T > 1) s[1] = st->t;
  if (Hx > 1) s[2] = st->h;
}

// out: no two elements may share an address.  Sorting the dimensions by stride, each must
// step past the whole extent of the ones inside it.
bool non_overlapping(const int64_t* s, int64_t B, int64_t T, int64_t H, int64_t width) {
  int64_t d[4][2] = {{1, width}, {s[2], H}, {s[1], T}, {s[0], B}};  // {stride, size}
  for (int i = 1; i < 4; ++i)
    for (int j = i; j > 0 && d[j][0] < d[j - 1][0]; --j)
      for (int c = 0; c < 2; ++c) {
        const int64_t x = d[j][c];
        d[j][c] = d[j - 1][c];
        d[j - 1][c] = x;
      }
  int64_t reach = 1;  // largest offset covered by the dimensions so far, plus one
  for (int i = 0; i < 4; ++i) {
    if (d[i][1] <= 1) continue;
    if (d[i][0] < reach) return false;
    reach += d[i][0] * (d[i][1] - 1);
  }
  return true;
}

// The strides a path can take: none negative; out non-overlapping; on the tensor-core
// path every stride of a dimension longer than 1 a positive multiple of 16 bytes (TMA).
int check_strides(const int64_t* sq, const int64_t* sk, const int64_t* sv, const int64_t* so,
                  int64_t B, int64_t T, int64_t H, int64_t Hqk, int64_t dk, int64_t dv, int path,
                  int in_dtype, int out_dtype) {
  const int64_t* all[4] = {sq, sk, sv, so};
  for (const int64_t* x : all)
    for (int i = 0; i < 3; ++i)
      if (x[i] < 0) return LL_ERR_INVALID;
  if (!non_overlapping(so, B, T, H, dv)) return LL_ERR_INVALID;
  if (path == LL_PATH_TC) {
    const int64_t sizes[4][3] = {{B, T, Hqk}, {B, T, Hqk}, {B, T, H}, {B, T, H}};
    for (int x = 0; x < 4; ++x) {
      const int64_t unit = x == 3 && out_dtype == LL_F32 ? 4 : 8;  // elements per 16 bytes
      const int64_t u = x < 3 && in_dtype == LL_F32 ? 4 : unit;
      for (int i = 0; i < 3; ++i) {
        if (sizes[x][i] <= 1) continue;
        if (all[x][i] == 0) return LL_ERR_UNSUPPORTED;
        if (all[x][i] % u != 0) return LL_ERR_ALIGN;
      }
    }
  }
  return LL_OK;
}

}  // namespace

int ll::report_cuda_error(cudaError_t e) { return cuda_fail(e); }

extern "C" {

int loglinear_version(void) { return (0 << 16) | 1; }

const char* loglinear_status_string(int status) {
  switch (status) {
    case LL_OK: return "LL_OK";
    case LL_ERR_INVALID: return "LL_ERR_INVALID: null pointer, negative size or unknown enum";
    case LL_ERR_SHAPE: return "LL_ERR_SHAPE: sizes violate the method (chunk, levels)";
    case LL_ERR_DTYPE: return "LL_ERR_DTYPE: unknown dtype code";
    case LL_ERR_UNSUPPORTED: return "LL_ERR_UNSUPPORTED: no kernel for this shape or path";
    case LL_ERR_CUDA: return "LL_ERR_CUDA: CUDA call or launch failed";
    case LL_ERR_WORKSPACE: return "LL_ERR_WORKSPACE: workspace missing or too small";
    case LL_ERR_ALIGN: return "LL_ERR_ALIGN: pointer alignment";
    default: return "unknown status";
  }
}

const char* loglinear_last_cuda_error(void) { return g_cuda_err; }

int loglinear_fwd_resolve_path(int64_t dk, int64_t dv, int chunk, int in_dtype, int path) {
  int p, tile;
  int64_t N;
  const int st = check_fwd_sizes(1, 1, 1, dk, dv, chunk, in_dtype, path, &p, &tile, &N);
  return st == LL_OK ? p : -st;
}

int loglinear_fwd_workspace_size(int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                                 int chunk, int in_dtype, int path, size_t* bytes) {
  if (!bytes) return LL_ERR_INVALID;
  int p, tile;
  int64_t N;
  const int st = check_fwd_sizes(B, T, H, dk, dv, chunk, in_dtype, path, &p, &tile, &N);
  if (st != LL_OK) return st;
  *bytes = fwd_workspace_layout(B, H, N, dk, dv, node_bytes(p)).total;
  return LL_OK;
}

static int fwd_impl(const void* q, const void* k, const void* v, const float* log_a,
                    const float* lambda, void* out, int64_t B, int64_t T, int64_t H,
                    int64_t Hqk, int64_t dk, int64_t dv, int64_t L, int chunk, int in_dtype,
                    int out_dtype, int path, void* workspace, size_t workspace_bytes,
                    ll_stream_t stream, StageEvents* ev, float* state_out = nullptr,
                    const ll_strides* const* strides = nullptr) {
  int p, tile;
  int64_t N;
  int st = check_fwd_sizes(B, T, H, dk, dv, chunk, in_dtype, path, &p, &tile, &N);
  if (st != LL_OK) return st;
  if ((st = check_qk_heads(H, Hqk)) != LL_OK) return st;
  if (!dtype_ok(out_dtype)) return LL_ERR_DTYPE;
  if (L < 1) return LL_ERR_INVALID;
  if (B == 0 || T == 0 || H == 0) return LL_OK;
  if (!q || !k || !v || !lambda || !out) return LL_ERR_INVALID;
  if (L < bit_length(T - 1) + 1) return LL_ERR_SHAPE;
  if (L > 64) return LL_ERR_UNSUPPORTED;
  const FwdWorkspace w = fwd_workspace_layout(B, H, N, dk, dv, node_bytes(p));
  if (!workspace || workspace_bytes < w.total) return LL_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LL_ERR_ALIGN;
  if (p == LL_PATH_TC && !(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(out)))
    return LL_ERR_ALIGN;
  FwdArgs a;
  a.q = q; a.k = k; a.v = v; a.log_a = log_a; a.lam = lambda; a.out = out;
  a.B = (int)B; a.T = (int)T; a.H = (int)H; a.dk = (int)dk; a.dv = (int)dv; a.L = (int)L;
  a.Hqk = (int)Hqk; a.hg = (int)(H / Hqk);
  a.C = tile; a.lc = log2_exact(tile); a.N = (int)N;
  resolve_strides(strides ? strides[0] : nullptr, B, T, Hqk, dk, a.sq);
  resolve_strides(strides ? strides[1] : nullptr, B, T, Hqk, dk, a.sk);
  resolve_strides(strides ? strides[2] : nullptr, B, T, H, dv, a.sv);
  resolve_strides(strides ? strides[3] : nullptr, B, T, H, dv, a.so);
  if ((st = check_strides(a.sq, a.sk, a.sv, a.so, B, T, H, Hqk, dk, dv, p, in_dtype,
                          out_dtype)) != LL_OK)
    return st;
  char* ws = static_cast<char*>(workspace);
  a.U = ws + w.off_U;
  a.nodes = ws + w.off_nodes;
  a.lg = reinterpret_cast<float*>(ws + w.off_lg);
  a.nlg = reinterpret_cast<float*>(ws + w.off_nlg);
  a.rdy_u = reinterpret_cast<uint32_t*>(ws + w.off_rdy_u);
  a.rdy_n = reinterpret_cast<uint32_t*>(ws + w.off_rdy_n);
  a.tick = reinterpret_cast<uint32_t*>(ws + w.off_tick);
  a.tag = reinterpret_cast<uint32_t*>(ws + w.off_tag);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (ev && state_out) ev->hold = true;  // the state kernel follows the forward's kernels
  cudaError_t e = p == LL_PATH_TC ? launch_tc_forward(a, out_dtype, s, ev)
                                  : launch_simt_forward(a, in_dtype, out_dtype, s, ev);
  if (e == cudaSuccess && state_out) {
    e = launch_prefill_state(a, p == LL_PATH_TC, in_dtype, state_out, s);
    if (e == cudaSuccess && ev) {
      ev->hold = false;
      if ((e = ev->record(s)) == cudaSuccess) e = ev->finish(s);
    }
  }
  return e == cudaSuccess ? LL_OK : cuda_fail(e);
}

int loglinear_fwd(const void* q, const void* k, const void* v, const float* log_a,
                  const float* lambda, void* out, int64_t B, int64_t T, int64_t H, int64_t Hqk,
                  int64_t dk, int64_t dv, int64_t L, int chunk, int in_dtype, int out_dtype,
                  int path, void* workspace, size_t workspace_bytes, ll_stream_t stream) {
  return fwd_impl(q, k, v, log_a, lambda, out, B, T, H, Hqk, dk, dv, L, chunk, in_dtype,
                  out_dtype, path, workspace, workspace_bytes, stream, nullptr);
}

int loglinear_fwd_strided(const void* q, const ll_strides* q_strides, const void* k,
                          const ll_strides* k_strides, const void* v, const ll_strides* v_strides,
                          const float* log_a, const float* lambda, void* out,
                          const ll_strides* out_strides, int64_t B, int64_t T, int64_t H,
                          int64_t Hqk, int64_t dk, int64_t dv, int64_t L, int chunk, int in_dtype,
                          int out_dtype, int path, void* workspace, size_t workspace_bytes,
                          ll_stream_t stream) {
  const ll_strides* strides[4] = {q_strides, k_strides, v_strides, out_strides};
  return fwd_impl(q, k, v, log_a, lambda, out, B, T, H, Hqk, dk, dv, L, chunk, in_dtype,
                  out_dtype, path, workspace, workspace_bytes, stream, nullptr, nullptr, strides);
}

int loglinear_prefill(const void* q, const void* k, const void* v, const float* log_a,
                      const float* lambda, void* out, float* state_out, int64_t B, int64_t T,
                      int64_t H, int64_t Hqk, int64_t dk, int64_t dv, int64_t L, int chunk,
                      int in_dtype, int out_dtype, int path, void* workspace,
                      size_t workspace_bytes, ll_stream_t stream) {
  if (!state_out) return LL_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(state_out) & 3u) != 0) return LL_ERR_ALIGN;
  const int sh = check_qk_heads(H, Hqk);
  if (sh != LL_OK) return sh;
  if (B > 0 && H > 0 && T == 0 && L >= 1 && dk >= 1 && dv >= 1) {  // no prefix: empty state
    const cudaError_t e = cudaMemsetAsync(state_out, 0, sizeof(float) * (size_t)(B * H * L * dk * dv),
                                          reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LL_OK : cuda_fail(e);
  }
  return fwd_impl(q, k, v, log_a, lambda, out, B, T, H, Hqk, dk, dv, L, chunk, in_dtype,
                  out_dtype, path, workspace, workspace_bytes, stream, nullptr, state_out);
}

int loglinear_prefill_with_events(const void* q, const void* k, const void* v,
                                  const float* log_a, const float* lambda, void* out,
                                  float* state_out, int64_t B, int64_t T, int64_t H, int64_t Hqk,
                                  int64_t dk, int64_t dv, int64_t L, int chunk, int in_dtype,
                                  int out_dtype, int path, void* workspace,
                                  size_t workspace_bytes, ll_stream_t stream,
                                  void* const* stage_events, int n_events, int* n_kernels) {
  if (n_events < 0 || (n_events > 0 && !stage_events)) return LL_ERR_INVALID;
  if (n_kernels) *n_kernels = 0;
  if (!state_out) return LL_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(state_out) & 3u) != 0) return LL_ERR_ALIGN;
  if (T == 0)  // no kernels to time: the plain call zeroes the state
    return loglinear_prefill(q, k, v, log_a, lambda, out, state_out, B, T, H, Hqk, dk, dv, L,
                             chunk, in_dtype, out_dtype, path, workspace, workspace_bytes, stream);
  StageEvents ev;
  ev.ev = reinterpret_cast<cudaEvent_t*>(const_cast<void**>(stage_events));
  ev.n = n_events;
  const int st = fwd_impl(q, k, v, log_a, lambda, out, B, T, H, Hqk, dk, dv, L, chunk, in_dtype,
                          out_dtype, path, workspace, workspace_bytes, stream, &ev, state_out);
  if (n_kernels) *n_kernels = ev.launched;
  return st;
}

int loglinear_fwd_with_events(const void* q, const void* k, const void* v, const float* log_a,
                              const float* lambda, void* out, int64_t B, int64_t T, int64_t H,
                              int64_t Hqk, int64_t dk, int64_t dv, int64_t L, int chunk,
                              int in_dtype,
                              int out_dtype, int path, void* workspace, size_t workspace_bytes,
                              ll_stream_t stream, void* const* stage_events, int n_events,
                              int* n_kernels) {
  if (n_events < 0 || (n_events > 0 && !stage_events)) return LL_ERR_INVALID;
  StageEvents ev;
  ev.ev = reinterpret_cast<cudaEvent_t*>(const_cast<void**>(stage_events));
  ev.n = n_events;
  if (n_kernels) *n_kernels = 0;
  const int st = fwd_impl(q, k, v, log_a, lambda, out, B, T, H, Hqk, dk, dv, L, chunk,
                          in_dtype, out_dtype, path, workspace, workspace_bytes, stream, &ev);
  if (n_kernels) *n_kernels = ev.launched;
  return st;
}

}  // extern "C"

namespace {

// Checks shared by the decode steps and the levels a step at position t touches: 0..l
// (merged into l+1) and the levels above l+1 that hold data after t-1.
int check_decode(int64_t B, int64_t H, int64_t Hqk, int64_t dk, int64_t dv, int64_t L, int64_t t,
                 int in_dtype, int out_dtype) {
  if (B < 0 || H < 0 || dk < 1 || dv < 1 || t < 0 || L < 1) return LL_ERR_INVALID;
  const int sh = check_qk_heads(H, Hqk);
  if (sh != LL_OK) return sh;
  if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return LL_ERR_DTYPE;
  if (t > INT32_MAX) return LL_ERR_UNSUPPORTED;
  if (L < bit_length(t) + 1) return LL_ERR_SHAPE;
  if (dk > kMaxHeadDim || !is_pow2(dv) || dv < 4 || dv > kMaxHeadDim || L > 64)
    return LL_ERR_UNSUPPORTED;
  if (B * H > INT32_MAX / 32) return LL_ERR_UNSUPPORTED;
  return LL_OK;
}

DecodePlan decode_plan(int64_t t, int64_t L) {
  DecodePlan plan;
  memset(&plan, 0, sizeof(plan));
  if (t == 0) {
    plan.t_zero = 1;
  } else {
    int l = 0;
    while (!((t >> l) & 1)) ++l;
    plan.l = l;
    int n = 0;
    for (int i = 0; i <= l; ++i) plan.lv[n++] = i;
    for (int lv = l + 2; lv < L; ++lv)
      if (((t - 1) >> (lv - 1)) & 1) plan.lv[n++] = lv;
    plan.n_hi = n - (l + 1);
  }
  return plan;
}

}  // namespace

extern "C" {

int loglinear_decode_step(float* state, const void* q, const void* k, const void* v,
                          const float* log_a, const float* lambda, int64_t t, void* out,
                          int64_t B, int64_t H, int64_t Hqk, int64_t dk, int64_t dv, int64_t L,
                          int in_dtype, int out_dtype, ll_stream_t stream) {
  const int st = check_decode(B, H, Hqk, dk, dv, L, t, in_dtype, out_dtype);
  if (st != LL_OK) return st;
  if (B == 0 || H == 0) return LL_OK;
  if (!state || !q || !k || !v || !lambda || !out) return LL_ERR_INVALID;
  if (!aligned16(state)) return LL_ERR_ALIGN;
  const DecodePlan plan = decode_plan(t, L);
  const cudaError_t e = launch_decode(state, q, k, v, log_a, lambda, out, (int)B, (int)H,
                                      (int)Hqk, (int)dk, (int)dv, (int)L, plan, in_dtype, out_dtype,
                                      reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LL_OK : cuda_fail(e);
}

int loglinear_gdn_decode_step(float* state, const void* q, const void* k, const void* v,
                              const float* log_a, const float* beta, const float* lambda,
                              int64_t t, void* out, int64_t B, int64_t H, int64_t Hqk, int64_t dk,
                              int64_t dv, int64_t L, int in_dtype, int out_dtype,
                              ll_stream_t stream) {
  const int st = check_decode(B, H, Hqk, dk, dv, L, t, in_dtype, out_dtype);
  if (st != LL_OK) return st;
  if (B == 0 || H == 0) return LL_OK;
  if (!state || !q || !k || !v || !beta || !lambda || !out) return LL_ERR_INVALID;
  if (!aligned16(state)) return LL_ERR_ALIGN;
  const DecodePlan plan = decode_plan(t, L);
  const cudaError_t e = launch_gdn_decode(state, q, k, v, log_a, beta, lambda, out, (int)B,
                                          (int)H, (int)Hqk, (int)dk, (int)dv, (int)L, plan,
                                          in_dtype, out_dtype,
                                          reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LL_OK : cuda_fail(e);
}

int loglinear_gdn_fwd(const void* q, const void* k, const void* v, const float* log_a,
                      const float* beta, const float* lambda, void* out, float* state_out,
                      int64_t B, int64_t T, int64_t H, int64_t Hqk, int64_t dk, int64_t dv,
                      int64_t L, int in_dtype, int out_dtype, ll_stream_t stream) {
  if (B < 0 || T < 0 || H < 0 || dk < 1 || dv < 1 || L < 1) return LL_ERR_INVALID;
  const int sh = check_qk_heads(H, Hqk);
  if (sh != LL_OK) return sh;
  if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return LL_ERR_DTYPE;
  if (T > INT32_MAX || dk > kMaxHeadDim || dv > kMaxHeadDim || L > 64) return LL_ERR_UNSUPPORTED;
  if (in_dtype == LL_BF16 && (dk & 1)) return LL_ERR_UNSUPPORTED;
  if (B * H > INT32_MAX / 16) return LL_ERR_UNSUPPORTED;
  const int levels = T > 0 ? bit_length(T - 1) + 1 : 1;
  if (L < levels) return LL_ERR_SHAPE;
  if (B == 0 || H == 0) return LL_OK;
  if (T > 0 && (!q || !k || !v || !beta || !lambda || !out)) return LL_ERR_INVALID;
  if (T > 0 && (reinterpret_cast<uintptr_t>(q) % 4 || reinterpret_cast<uintptr_t>(k) % 4))
    return LL_ERR_ALIGN;
  if (state_out && reinterpret_cast<uintptr_t>(state_out) % 4) return LL_ERR_ALIGN;
  const cudaError_t e = launch_gdn_fwd(q, k, v, log_a, beta, lambda, out, state_out, (int)B,
                                       (int)T, (int)H, (int)Hqk, (int)dk, (int)dv, (int)L, levels,
                                       in_dtype, out_dtype, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LL_OK : cuda_fail(e);
}

int loglinear_gdn_fwd_chunked_workspace_size(int64_t B, int64_t T, int64_t H, int64_t dk,
                                              int64_t dv, size_t* bytes) {
  if (!bytes || B < 0 || T < 0 || H < 0 || dk < 1 || dv < 1) return LL_ERR_INVALID;
  if (dk > kMaxHeadDim || dv > kMaxHeadDim || T > INT32_MAX) return LL_ERR_UNSUPPORTED;
  *bytes = gdn_chunk_workspace_bytes(B, T, H, dk, dv);
  return LL_OK;
}

int loglinear_gdn_fwd_chunked(const void* q, const void* k, const void* v, const float* log_a,
                              const float* beta, const float* lambda, void* out,
                              float* state_out, int64_t B,
                              int64_t T, int64_t H, int64_t Hqk, int64_t dk, int64_t dv,
                              int64_t L, int in_dtype, int out_dtype, void* workspace,
                              size_t workspace_bytes, ll_stream_t stream) {
  if (B < 0 || T < 0 || H < 0 || dk < 1 || dv < 1 || L < 1) return LL_ERR_INVALID;
  const int sh = check_qk_heads(H, Hqk);
  if (sh != LL_OK) return sh;
  if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return LL_ERR_DTYPE;
  if (T > INT32_MAX || dk > kMaxHeadDim || dv > kMaxHeadDim || L > 64) return LL_ERR_UNSUPPORTED;
  if (B * H * ((T + 63) / 64) > INT32_MAX) return LL_ERR_UNSUPPORTED;
  // the scan keeps every chunk level of its columns in shared memory: up to 2^19 chunks
  if (T > ((int64_t)64 << 19)) return LL_ERR_UNSUPPORTED;
  if (T > 0 && L < bit_length(T - 1) + 1) return LL_ERR_SHAPE;
  if (in_dtype == LL_BF16 && (dk & 1) && state_out) return LL_ERR_UNSUPPORTED;
  if (B == 0 || H == 0) return LL_OK;
  if (state_out && reinterpret_cast<uintptr_t>(state_out) % 4) return LL_ERR_ALIGN;
  if (T == 0) {  // an empty prompt: an empty state
    const cudaError_t e = launch_gdn_chunked(q, k, v, log_a, beta, lambda, out, state_out,
                                             (int)B, 0, (int)H, (int)Hqk, (int)dk, (int)dv,
                                             (int)L, in_dtype, out_dtype, workspace,
                                             reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LL_OK : cuda_fail(e);
  }
  if (!q || !k || !v || !beta || !lambda || !out) return LL_ERR_INVALID;
  if (!workspace || workspace_bytes < gdn_chunk_workspace_bytes(B, T, H, dk, dv))
    return LL_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LL_ERR_ALIGN;
  if (state_out && (reinterpret_cast<uintptr_t>(q) % 4 || reinterpret_cast<uintptr_t>(k) % 4))
    return LL_ERR_ALIGN;  // the last chunk's run stages q and k with 4-byte copies
  const cudaError_t e = launch_gdn_chunked(q, k, v, log_a, beta, lambda, out, state_out, (int)B,
                                           (int)T, (int)H, (int)Hqk, (int)dk, (int)dv, (int)L,
                                           in_dtype, out_dtype, workspace,
                                           reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LL_OK : cuda_fail(e);
}

// ---------------------------------------------------------------- backward

// N: 32-token tiles of the CUDA-core part; *n_tc: 128-token tiles of the tensor-core dQ
// when that path is taken, else 0.
static int check_bwd(int64_t B, int64_t T, int64_t H, int64_t Hqk, int64_t dk, int64_t dv,
                     int64_t L, int in_dtype, int grad_dtype, int path, int64_t* N,
                     int64_t* n_tc) {
  if (B < 0 || T < 0 || H < 0 || dk < 1 || dv < 1 || L < 1) return LL_ERR_INVALID;
  if (!dtype_ok(in_dtype) || !dtype_ok(grad_dtype)) return LL_ERR_DTYPE;
  if (path != LL_PATH_AUTO && path != LL_PATH_SIMT && path != LL_PATH_TC) return LL_ERR_INVALID;
  const bool tc_ok = tc_bwd_dq_supported(dk, dv, in_dtype, grad_dtype);
  if (path == LL_PATH_TC && !tc_ok) return LL_ERR_UNSUPPORTED;
  const bool tc = path == LL_PATH_TC || (path == LL_PATH_AUTO && tc_ok);
  *n_tc = tc ? (T + kTcTile - 1) / kTcTile : 0;
  const int sh = check_qk_heads(H, Hqk);
  if (sh != LL_OK) return sh;
  if (T > INT32_MAX || B * H > INT32_MAX / 2) return LL_ERR_UNSUPPORTED;
  if (dk > kMaxHeadDim || dv > kMaxHeadDim || L > 64) return LL_ERR_UNSUPPORTED;
  if (T > 0 && L < bit_length(T - 1) + 1) return LL_ERR_SHAPE;
  *N = (T + kBwdTile - 1) / kBwdTile;
  return LL_OK;
}

int loglinear_bwd_workspace_size(int64_t B, int64_t T, int64_t H, int64_t Hqk, int64_t dk,
                                 int64_t dv, int64_t L, int in_dtype, int grad_dtype, int path,
                                 size_t* bytes) {
  if (!bytes) return LL_ERR_INVALID;
  int64_t N, n_tc;
  const int st = check_bwd(B, T, H, Hqk, dk, dv, L, in_dtype, grad_dtype, path, &N, &n_tc);
  if (st != LL_OK) return st;
  *bytes = bwd_workspace_layout(B, T, H, Hqk, N, dk, dv, n_tc).total;
  return LL_OK;
}

int loglinear_bwd(const void* q, const void* k, const void* v, const float* log_a,
                  const float* lambda, const void* dout, void* dq, void* dk_out, void* dv_out,
                  float* dlog_a, float* dlambda, int64_t B, int64_t T, int64_t H, int64_t Hqk,
                  int64_t dk, int64_t dv, int64_t L, int in_dtype, int grad_dtype, int path,
                  const void* fwd_workspace, size_t fwd_workspace_bytes, void* workspace,
                  size_t workspace_bytes, ll_stream_t stream) {
  int64_t N, n_tc;
  const int st = check_bwd(B, T, H, Hqk, dk, dv, L, in_dtype, grad_dtype, path, &N, &n_tc);
  if (st != LL_OK) return st;
  if (B == 0 || T == 0 || H == 0) return LL_OK;
  if (fwd_workspace && n_tc == 0) return LL_ERR_UNSUPPORTED;  // only the tensor-core path
                                                              // reads a forward's states
  if (!q || !k || !v || !lambda || !dout || !dq || !dk_out || !dv_out || !dlambda)
    return LL_ERR_INVALID;
  if (log_a && !dlog_a) return LL_ERR_INVALID;
  const BwdWorkspace w = bwd_workspace_layout(B, T, H, Hqk, N, dk, dv, n_tc);
  if (!workspace || workspace_bytes < w.total) return LL_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return LL_ERR_ALIGN;
  if (n_tc > 0 && !(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(dout) &&
                    aligned16(dq) && aligned16(dk_out) && aligned16(dv_out)))
    return LL_ERR_ALIGN;
  if (fwd_workspace) {
    if (fwd_workspace_bytes < w.fwd.total) return LL_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(fwd_workspace) & 255u) != 0) return LL_ERR_ALIGN;
  }
  BwdArgs A;
  FwdArgs& a = A.f;
  a.q = q; a.k = k; a.v = v; a.log_a = log_a; a.lam = lambda; a.out = nullptr;
  a.B = (int)B; a.T = (int)T; a.H = (int)H; a.dk = (int)dk; a.dv = (int)dv; a.L = (int)L;
  a.Hqk = (int)Hqk; a.hg = (int)(H / Hqk);
  a.C = kBwdTile; a.lc = log2_exact(kBwdTile); a.N = (int)N;
  set_dense_strides(a);
  char* ws = static_cast<char*>(workspace);
  a.U = ws + w.off_U;
  a.nodes = ws + w.off_nodes;
  a.lg = reinterpret_cast<float*>(ws + w.off_lg);
  a.nlg = nullptr; a.rdy_u = nullptr; a.rdy_n = nullptr; a.tick = nullptr; a.tag = nullptr;
  A.dout = dout; A.dq = dq; A.dk = dk_out; A.dv = dv_out;
  A.dlog_a = log_a ? dlog_a : nullptr;
  A.dlam = dlambda;
  A.dqh = reinterpret_cast<float*>(ws + w.off_dqh);
  A.dkh = reinterpret_cast<float*>(ws + w.off_dkh);
  A.dcq = log_a ? reinterpret_cast<float*>(ws + w.off_dcq) : nullptr;
  A.dck = log_a ? reinterpret_cast<float*>(ws + w.off_dck) : nullptr;
  A.scan = reinterpret_cast<float*>(ws + w.off_scan);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (n_tc > 0) {
    // dQ and dlambda on the tensor cores: a tensor-core forward in its states-only form
    // publishes the block states (no output), then the dQ kernel reads them
    FwdArgs f = a;
    f.C = kTcTile;
    f.lc = log2_exact(kTcTile);
    f.N = (int)n_tc;
    // the states: those a forward call left in its own workspace, else a forward here
    char* fw = fwd_workspace ? static_cast<char*>(const_cast<void*>(fwd_workspace))
                             : ws + w.off_fwd;
    f.out = nullptr;  // the states-only forward writes no output
    f.U = fw + w.fwd.off_U;
    f.nodes = fw + w.fwd.off_nodes;
    f.lg = reinterpret_cast<float*>(fw + w.fwd.off_lg);
    f.nlg = reinterpret_cast<float*>(fw + w.fwd.off_nlg);
    f.rdy_u = reinterpret_cast<uint32_t*>(fw + w.fwd.off_rdy_u);
    f.rdy_n = reinterpret_cast<uint32_t*>(fw + w.fwd.off_rdy_n);
    f.tick = reinterpret_cast<uint32_t*>(fw + w.fwd.off_tick);
    f.tag = reinterpret_cast<uint32_t*>(fw + w.fwd.off_tag);
    // the mirrored states on the same 128-token tiles go into U's buffer (fp32)
    float* R = reinterpret_cast<float*>(a.U);
    // with one q/k per head the kernels write dq and dk in bf16 themselves; with shared
    // q/k heads each head adds its fp32 dq and dk into its group's sum (atomics into
    // zeroed [B, T, Hqk, d_k] buffers), which the last pass casts
    const bool own_qk = a.hg == 1;
    if (!own_qk) {
      const size_t qk_bytes = sizeof(float) * (size_t)B * T * Hqk * dk;
      if ((e = cudaMemsetAsync(A.dqh, 0, qk_bytes, s)) == cudaSuccess)
        e = cudaMemsetAsync(A.dkh, 0, qk_bytes, s);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    if (!fwd_workspace) e = launch_tc_forward(f, LL_BF16, s, nullptr, /*states_only=*/true);
    if (e == cudaSuccess)
      e = launch_tc_bwd_dq(f, dout, A.dqh, own_qk ? dq : nullptr, A.dcq, dlambda, s);
    if (e == cudaSuccess && f.N > 1) e = launch_tc_bwd_rstate(f, dout, R, s);
    if (e == cudaSuccess)
      e = launch_tc_bwd_dkv(f, dout, R, A.dkh, own_qk ? dk_out : nullptr, A.dck, dv_out, s);
    if (e == cudaSuccess) e = launch_bwd_finish(A, grad_dtype, s, !own_qk, true);
    return e == cudaSuccess ? LL_OK : cuda_fail(e);
  }
  e = launch_simt_backward(A, in_dtype, grad_dtype, s);
  return e == cudaSuccess ? LL_OK : cuda_fail(e);
}

int loglinear_device_error(ll_stream_t stream, unsigned* flags) {
  if (!flags) return LL_ERR_INVALID;
  unsigned f1 = 0, f2 = 0;
  cudaError_t e = tc_take_error(reinterpret_cast<cudaStream_t>(stream), &f1);
  if (e == cudaSuccess) e = tcb_take_error(reinterpret_cast<cudaStream_t>(stream), &f2);
  *flags = f1 | f2;
  return e == cudaSuccess ? LL_OK : cuda_fail(e);
}

int loglinear_debug_level_map(int64_t T, int chunk, int path, int8_t* levels,
                              ll_stream_t stream) {
  if (T < 0 || T > 16384) return LL_ERR_INVALID;
  if (T > 0 && !levels) return LL_ERR_INVALID;
  int p, tile;
  int64_t N;
  const int st = check_fwd_sizes(1, T, 1, 128, 128, chunk, LL_BF16, path, &p, &tile, &N);
  if (st != LL_OK) return st;
  const cudaError_t e = launch_level_map((int)T, tile, log2_exact(tile), levels,
                                         reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LL_OK : cuda_fail(e);
}

}  // extern "C"

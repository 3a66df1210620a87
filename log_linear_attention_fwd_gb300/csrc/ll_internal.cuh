// Internal declarations shared by the translation units of the library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "loglinear.h"

namespace ll {

// ---------------------------------------------------------------- element access

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// ---------------------------------------------------------------- Fenwick indexing
//
// Level of source s seen from query t (s <= t): the Fenwick bucket of t that holds s is
// the one cut at the highest bit where s and t differ, so the level is the bit length of
// t XOR s; s == t gives 0, the sentinel bucket (page "论文阅读：Log-Linear Attention",
// sections 前缀的层次化分解 and 层级判定算法).
__host__ __device__ __forceinline__ int fenwick_level(uint32_t t, uint32_t s) {
#ifdef __CUDA_ARCH__
  return 32 - __clz(t ^ s);
#else
  uint32_t x = t ^ s;
  int n = 0;
  while (x) { ++n; x >>= 1; }
  return n;
#endif
}

// Inter-chunk block pairing.  Chunk j reads, at chunk level m (token level lc + m), the
// aligned block of 2^(m-1) chunks just below c = j with its low m-1 bits cleared; that
// block exists iff bit m-1 of j is set.  The block state is stored under index c, which
// is unique per (m, block) since ctz(c) = m-1.
__host__ __device__ __forceinline__ bool inter_block(int64_t j, int m, int64_t* c_out) {
  if (!((j >> (m - 1)) & 1)) return false;
  *c_out = (j >> (m - 1)) << (m - 1);
  return true;
}

// ---------------------------------------------------------------- forward arguments

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* log_a;  // may be null
  const float* lam;
  void* out;
  int B, T, H, dk, dv, L;
  int Hqk, hg;  // q/k heads and value heads per q/k head (H = Hqk * hg): head h reads
                // q/k head h / hg
  int C, lc;  // tile length and log2(tile)
  int N;      // tiles per (b, h)
  // element strides of the batch, position and head dimensions of q, k, v and out (the
  // feature dimension is contiguous); dense: {T*Hx*w, Hx*w, w}
  int64_t sq[3], sk[3], sv[3], so[3];
  // workspace
  void* U;        // [B*H][N][dk][dv] chunk states (fp32 on CUDA cores; bf16 on tensor cores,
                  // written for even tiles only: no reader takes an odd one)
  void* nodes;    // [B*H][N][dk*dv] Fenwick block states, slot c = first reader chunk
  float* lg;      // [B*H][N] log decay of each whole chunk
  // tensor cores only (block states published between CTAs of one launch):
  float* nlg;     // [B*H][N] log decay of the block in each even block-state slot
  uint32_t* rdy_u;  // [B*H][N] ready flags of U; followed in memory by
  uint32_t* rdy_n;  // [B*H][N] ready flags of the block states, and by
  uint32_t* tick;   // one tile ticket counter (the three are zeroed together)
  uint32_t* tag;    // tensor-core path: the workspace's layout tag (fwd_layout_tag), which
                    // the forward writes and a backward given this workspace checks
};

// Dense strides of [B, T, Hx, width]: {T*Hx*width, Hx*width, width}.
inline void dense_strides(int64_t* s, int64_t T, int64_t Hx, int64_t width) {
  s[2] = width;
  s[1] = Hx * width;
  s[0] = T * Hx * width;
}
inline void set_dense_strides(FwdArgs& a) {
  dense_strides(a.sq, a.T, a.Hqk, a.dk);
  dense_strides(a.sk, a.T, a.Hqk, a.dk);
  dense_strides(a.sv, a.T, a.H, a.dv);
  dense_strides(a.so, a.T, a.H, a.dv);
}

// Workspace carving (identical on host for size queries and for launches).
struct FwdWorkspace {
  size_t off_U, off_nodes, off_lg, off_nlg, off_rdy_u, off_rdy_n, off_tick, off_tag, total;
};
FwdWorkspace fwd_workspace_layout(int64_t B, int64_t H, int64_t N, int64_t dk, int64_t dv,
                                  size_t state_elem_bytes);
// The tag a tensor-core forward leaves in its workspace: a non-zero mix of the sizes that
// fix its layout, so that a backward reading that workspace can tell whether it matches.
inline uint32_t fwd_layout_tag(int64_t B, int64_t T, int64_t H, int64_t Hqk, int64_t dv) {
  uint64_t x = 0x4C4C5443ull;  // any fixed start
  const int64_t f[5] = {B, T, H, Hqk, dv};
  for (int64_t v : f) x = (x ^ (uint64_t)v) * 0x100000001B3ull;
  const uint32_t t = (uint32_t)(x ^ (x >> 32));
  return t ? t : 1u;
}

// Optional per-kernel event recording by the launchers (instrumentation only).
struct StageEvents {
  cudaEvent_t* ev = nullptr;
  int n = 0;
  int recorded = 0;
  cudaError_t record(cudaStream_t s) {
    if (recorded < n) return cudaEventRecord(ev[recorded++], s);
    return cudaSuccess;
  }
  bool hold = false;  // a later kernel of the same call still follows: finish() counts only
  cudaError_t finish(cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    const int kernels = recorded > 0 ? recorded - 1 : 0;
    launched = kernels;
    if (hold) return e;
    while (recorded < n && e == cudaSuccess) e = cudaEventRecord(ev[recorded++], s);
    return e;
  }
  int launched = 0;
};

// Launchers (return cudaError_t of the launches).
cudaError_t launch_simt_forward(const FwdArgs& a, int in_dtype, int out_dtype, cudaStream_t s,
                                StageEvents* ev);
// states_only: the tile states, block states and log decays (all a backward reads), no
// output; Q is not read.
cudaError_t launch_tc_forward(const FwdArgs& a, int out_dtype, cudaStream_t s, StageEvents* ev,
                              bool states_only = false);
cudaError_t launch_level_scan(const FwdArgs& a, cudaStream_t s);
// The CUDA-core path's chunk states U and fp32 block states of every slot (K1 and K2 of
// the forward, without the readout).
cudaError_t launch_simt_states(const FwdArgs& a, int in_dtype, cudaStream_t s);

// Backward (fp32 on CUDA cores): the forward's states are recomputed on tiles of
// kBwdTile tokens; U is then reused for the mirrored block states.
constexpr int kBwdTile = 32;
struct BwdArgs {
  FwdArgs f;            // inputs, tile geometry, recomputed states (U, nodes, lg)
  const void* dout;     // [B, T, H, dv] grad dtype
  void* dq;             // [B, T, Hqk, dk] grad dtype
  void* dk;             // [B, T, Hqk, dk] grad dtype
  void* dv;             // [B, T, H, dv] grad dtype
  float* dlog_a;        // [B, T, H] or null (no decay)
  float* dlam;          // [B, T, H, L]
  float* dqh;           // [B, T, H, dk] per-head dq (workspace)
  float* dkh;           // [B, T, H, dk] per-head dk (workspace)
  float* dcq;           // [B, T, H] q_t . dq_t per head (workspace)
  float* dck;           // [B, T, H] k_t . dk_t per head (workspace)
  float* scan;          // [B*H][ceil(T/1024)] chunk sums of the d log a scan (workspace)
};
struct BwdWorkspace {
  size_t off_U, off_nodes, off_lg, off_dqh, off_dkh, off_dcq, off_dck, off_scan;
  size_t off_fwd;  // tensor cores only: the workspace of the states-only forward
  FwdWorkspace fwd;         // that forward workspace's own layout (offsets from off_fwd)
  size_t total;
};
// N: 32-token tiles; n_tc: 128-token tiles of the tensor-core dQ, or 0 without it.
BwdWorkspace bwd_workspace_layout(int64_t B, int64_t T, int64_t H, int64_t Hqk, int64_t N,
                                  int64_t dk, int64_t dv, int64_t n_tc);
// The whole backward on CUDA cores (fp32, 32-token tiles).
cudaError_t launch_simt_backward(const BwdArgs& a, int in_dtype, int grad_dtype, cudaStream_t s);
// Tensor-core backward (bf16, d_k = 128, d_v in {64, 128}) on the 128-token tiles of a
// completed tensor-core forward over the same inputs (f: that forward's arguments and
// workspace).  dQ and dlambda from its block states: dQ (bf16 into dq_bf16 when every
// head has its own q/k, else fp32 per head into dqh), q . dQ (dcq may be null), dlambda.
bool tc_bwd_dq_supported(int64_t dk, int64_t dv, int in_dtype, int grad_dtype);
cudaError_t launch_tc_bwd_dq(const FwdArgs& f, const void* dout, float* dqh, void* dq_bf16,
                             float* dcq, float* dlam, cudaStream_t s);
// Tensor-core mirrored states on the forward's 128-token tiles into R ([B*H][N][d_k][d_v]
// fp32, zeroed here), then dK, dV and k . dK from them (f as above).  dv in bf16.
cudaError_t launch_tc_bwd_rstate(const FwdArgs& f, const void* dout, float* R, cudaStream_t s);
cudaError_t launch_tc_bwd_dkv(const FwdArgs& f, const void* dout, const float* R, float* dkh,
                              void* dk_bf16, float* dck, void* dv, cudaStream_t s);
// The group sums of dq and dk with their cast (skipped when with_qk is false: the
// kernels wrote them), and d log a (the last kernels of every backward path).
// qk_summed: dqh and dkh hold the q/k heads' sums [B, T, Hqk, d_k] (tensor-core path with
// shared q/k) rather than per value head [B, T, H, d_k].
cudaError_t launch_bwd_finish(const BwdArgs& a, int grad_dtype, cudaStream_t s, bool with_qk,
                              bool qk_summed);
cudaError_t tcb_take_error(cudaStream_t s, unsigned* flags);
size_t bwd_smem_max(int dk, int dv, int L);  // largest dynamic shared memory of a kernel
// The decode state at position T-1 from a completed forward's workspace (tc_layout: the
// tensor-core path's bf16 block states; both paths store them [d_k][d_v]).
cudaError_t launch_prefill_state(const FwdArgs& a, bool tc_layout, int in_dtype, float* state,
                                 cudaStream_t s);
// Reads and clears the tensor-core path's device error word (synchronises the stream).
cudaError_t tc_take_error(cudaStream_t s, unsigned* flags);
bool tc_forward_supported(int64_t dk, int64_t dv, int in_dtype, int chunk);
constexpr int kTcTile = 128;

struct DecodePlan {
  int t_zero;      // 1 if t == 0 (initialise)
  int l;           // lssb(t) for t > 0
  int n_hi;        // number of levels > l+1 holding data after t-1
  int lv[64];      // touched levels: 0..l, then the n_hi levels above l+1
};
cudaError_t launch_decode(float* state, const void* q, const void* k, const void* v,
                          const float* log_a, const float* lam, void* out, int B, int H,
                          int Hqk, int dk, int dv, int L, const DecodePlan& plan, int in_dtype,
                          int out_dtype, cudaStream_t s);

// Log-Linear Gated DeltaNet decode step (gated delta rule transition on every level).
cudaError_t launch_gdn_decode(float* state, const void* q, const void* k, const void* v,
                              const float* log_a, const float* beta, const float* lam, void* out,
                              int B, int H, int Hqk, int dk, int dv, int L, const DecodePlan& plan,
                              int in_dtype, int out_dtype, cudaStream_t s);
// Log-Linear Gated DeltaNet forward in chunks of 64 tokens (UT transform per chunk, then a
// sequential scan of the chunk-level states); workspace of gdn_chunk_workspace_bytes().
size_t gdn_chunk_workspace_bytes(int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv);
cudaError_t launch_gdn_chunked(const void* q, const void* k, const void* v, const float* log_a,
                               const float* beta, const float* lam, void* out, float* state,
                               int B, int T, int H, int Hqk, int dk, int dv, int L, int in_dtype,
                               int out_dtype, void* workspace, cudaStream_t s);
// The recurrent form over tokens [t0, Tfull) only, from an empty state: fp32 outputs into
// out_f32 ([B, Tfull, H, dv] indexing) and the first state_levels levels of the state.
cudaError_t launch_gdn_fwd_tail(const void* q, const void* k, const void* v, const float* log_a,
                                const float* beta, const float* lam, float* out_f32,
                                float* state, int B, int Tfull, int t0, int H, int Hqk, int dk,
                                int dv, int L, int state_levels, int in_dtype, cudaStream_t s);
// Log-Linear Gated DeltaNet forward in the recurrent form (levels = bit_length(T-1) + 1
// Fenwick levels in use); state, when non-null, receives the per-level state after T-1.
cudaError_t launch_gdn_fwd(const void* q, const void* k, const void* v, const float* log_a,
                           const float* beta, const float* lam, void* out, float* state, int B,
                           int T, int H, int Hqk, int dk, int dv, int L, int levels, int in_dtype,
                           int out_dtype, cudaStream_t s);

cudaError_t launch_level_map(int T, int tile, int lc, int8_t* levels, cudaStream_t s);

// Records a CUDA error for loglinear_last_cuda_error() and returns LL_ERR_CUDA.
int report_cuda_error(cudaError_t e);

}  // namespace ll

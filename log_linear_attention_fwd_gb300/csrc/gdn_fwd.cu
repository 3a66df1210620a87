// Forward of Log-Linear Gated DeltaNet in its recurrent form: the lssb decode step of
// gdn_decode.cu run over t = 0..T-1 with every level's state held on chip.
//
// The log-linear form keeps the model's transition and composes its mask with the Fenwick
// mask (page "算力终结者来了！…", section 对Mamba-2和门控DeltaNet的对数线性推广; page
// "论文阅读：Log-Linear Attention", sections 与已有模型的组合 and 解码：基于 lssb 的状态更新).
// The transition is the gated delta rule (Yang, Kautz and Hatamizadeh, "Gated Delta
// Networks", 2024): with the state stored [d_k][d_v] (o = S^T q),
//     A_t = alpha_t (I - beta_t k_t k_t^T),   every state held after t-1:  S <- A_t S,
// then levels 0..lssb(t) merge into level lssb(t)+1, levels 1..lssb(t) are cleared, and
// level 0 <- beta_t k_t v_t^T;  o_t = sum_l lambda_t[l] S_l^T q_t.
//
// Column e of A_t S needs only column e of S and u_e = (S^T k)_e, so a CTA takes 8 columns
// of one (b, h) and keeps, for each column, one thread per level (kLv consecutive lanes)
// holding that level's column of 128 rows in registers.  Per token a live level forms
// u = S^T k and w = S^T q by itself (no cross-thread sum), carries its state and reads out
// alpha (w - beta (k.q) u) (the carried state's readout); the merge sums the carried
// columns of levels 0..lssb(t) into lane lssb(t)+1 with a shuffle scan; the output sums
// lambda-weighted readouts over the column's lanes.  Sixteen tokens of q and k are staged in
// shared memory at a time (cp.async, one stage ahead) and converted to fp32 once.
//
// The recurrence is sequential in t: one token costs a few hundred instructions per
// thread, so this path is for correctness and moderate lengths; the chunked (WY) form is
// not built.
#include "ll_internal.cuh"

namespace ll {
namespace {

constexpr int kCols = 8;      // d_v columns per CTA
constexpr int kDk = 128;      // state rows per thread (d_k <= 128, zero-padded)
constexpr int kStage = 16;    // tokens staged at a time

__device__ __forceinline__ void cp_async_4(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

struct GdnFwdArgs {
  const void* q;        // [B, T, Hqk, dk]
  const void* k;        // [B, T, Hqk, dk]
  const void* v;        // [B, T, H, dv]
  const float* log_a;   // [B, T, H] or null
  const float* beta;    // [B, T, H]
  const float* lam;     // [B, T, H, L]
  void* out;            // [B, T, H, dv]
  float* state;         // [B, H, L, dk, dv] or null (zeroed by the host when given)
  int B, T, H, hg, dk, dv, L;
  int Tfull, t0;        // the run covers tokens [t0, t0 + T) of sequences of Tfull tokens
  int state_levels;     // levels of the final state written (the rest left as they are)
};

template <typename InT, typename OutT, int kLv>
__global__ void __launch_bounds__(kLv * kCols, 1) gdn_fwd_kernel(GdnFwdArgs a) {
  constexpr int kThreads = kLv * kCols;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // raw q and k of two stages (cp.async), then fp32 copies of the current stage
  const int dk = a.dk, dv = a.dv;
  const int row_words = dk * (int)sizeof(InT) / 4;  // 4-byte words of one q or k row
  unsigned char* raw = smem_raw;                     // [2][2][kStage][row_words] words
  const size_t raw_stage = (size_t)2 * kStage * row_words * 4;
  float* qf = reinterpret_cast<float*>(smem_raw + 2 * raw_stage);  // [kStage][kDk]
  float* kf = qf + kStage * kDk;                                    // [kStage][kDk]
  float* kq = kf + kStage * kDk;                                    // [kStage]
  float* vs = kq + kStage;                                          // [kStage][kCols]
  float* ls = vs + kStage * kCols;                                  // [kStage][kLv]
  float* al = ls + kStage * kLv;                                    // [kStage] alpha
  float* bt = al + kStage;                                          // [kStage] beta
  float* os = bt + kStage;                                          // [kStage][kCols]

  const int slices = (dv + kCols - 1) / kCols;
  const int64_t bh = blockIdx.x / slices;
  const int c0 = (int)(blockIdx.x - bh * slices) * kCols;
  const int b = (int)(bh / a.H), h = (int)(bh - (int64_t)b * a.H), hq = h / a.hg;
  const int Hqk = a.H / a.hg;
  const int tid = threadIdx.x;
  const int lv = tid % kLv;        // this thread's level
  const int cl = tid / kLv;        // this thread's column within the CTA
  const int col = c0 + cl;
  const bool col_ok = col < dv;
  const int T = a.T;
  const int nstage = (T + kStage - 1) / kStage;

  auto issue_stage = [&](int s) {  // cp.async of stage s's q and k rows into raw[s & 1]
    uint32_t* dst = reinterpret_cast<uint32_t*>(raw + (s & 1) * raw_stage);
    const int n = min(kStage, T - s * kStage);
    for (int i = tid; i < 2 * n * row_words; i += kThreads) {
      const int which = i / (n * row_words);  // 0: q, 1: k
      const int rem = i - which * n * row_words;
      const int tt = rem / row_words, wd = rem - tt * row_words;
      const int64_t tok = ((int64_t)b * a.Tfull + a.t0 + s * kStage + tt) * Hqk + hq;
      const uint32_t* src =
          reinterpret_cast<const uint32_t*>(static_cast<const InT*>(which ? a.k : a.q) + tok * dk);
      cp_async_4(dst + (which * kStage + tt) * row_words + wd, src + wd);
    }
  };

  float S[kDk];
#pragma unroll
  for (int d = 0; d < kDk; ++d) S[d] = 0.f;

  issue_stage(0);
  cp_async_commit();
  for (int s = 0; s < nstage; ++s) {
    if (s + 1 < nstage) issue_stage(s + 1);
    cp_async_commit();  // (an empty group on the last stage keeps the count uniform)
    cp_async_wait_1();  // stage s has landed
    __syncthreads();
    const int n = min(kStage, T - s * kStage);
    // ---- convert the stage: q, k to fp32 (zero-padded to 128), k . q, v, lambda, gates
    {
      const InT* rq = reinterpret_cast<const InT*>(raw + (s & 1) * raw_stage);
      const InT* rk = rq + kStage * dk;
      for (int i = tid; i < kStage * kDk; i += kThreads) {
        const int tt = i / kDk, d = i - tt * kDk;
        const bool in = tt < n && d < dk;
        qf[i] = in ? to_f32(rq[tt * dk + d]) : 0.f;
        kf[i] = in ? to_f32(rk[tt * dk + d]) : 0.f;
      }
      for (int i = tid; i < kStage * kCols; i += kThreads) {
        const int tt = i / kCols, c = i - tt * kCols;
        const int64_t tok = ((int64_t)b * a.Tfull + a.t0 + s * kStage + tt) * a.H + h;
        vs[i] = (tt < n && c0 + c < dv) ? to_f32(static_cast<const InT*>(a.v)[tok * dv + c0 + c])
                                        : 0.f;
      }
      for (int i = tid; i < kStage * kLv; i += kThreads) {
        const int tt = i / kLv, l = i - tt * kLv;
        const int64_t tok = ((int64_t)b * a.Tfull + a.t0 + s * kStage + tt) * a.H + h;
        ls[i] = (tt < n && l < a.L) ? a.lam[tok * a.L + l] : 0.f;
      }
      if (tid < kStage) {
        const int64_t tok = ((int64_t)b * a.Tfull + a.t0 + s * kStage + tid) * a.H + h;
        al[tid] = (tid < n && a.log_a) ? __expf(a.log_a[tok]) : 1.f;
        bt[tid] = tid < n ? a.beta[tok] : 0.f;
      }
    }
    __syncthreads();
    // k . q of the stage's tokens: warp w takes tokens w, w + warps, ...
    for (int tt = tid >> 5; tt < kStage; tt += kThreads / 32) {
      float x = 0.f;
      for (int d = tid & 31; d < kDk; d += 32) x = fmaf(kf[tt * kDk + d], qf[tt * kDk + d], x);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      if ((tid & 31) == 0) kq[tt] = x;
    }
    __syncthreads();

    // ---- the stage's tokens, one lssb step each
    for (int tt = 0; tt < n; ++tt) {
      const int t = s * kStage + tt;
      const float* kr = kf + tt * kDk;
      const float* qr = qf + tt * kDk;
      const float alpha = al[tt], beta = bt[tt], kqt = kq[tt];
      const float vc = vs[tt * kCols + cl];
      float contrib = 0.f;
      if (t > 0) {
        const int lsb = __ffs(t) - 1;  // lssb(t): levels 0..lsb merge into lsb + 1
        const bool live = lv == 0 || (((t - 1) >> (lv - 1)) & 1);
        if (live) {
          float u4[4] = {0.f, 0.f, 0.f, 0.f}, w4[4] = {0.f, 0.f, 0.f, 0.f};  // 4 short chains
#pragma unroll
          for (int d = 0; d < kDk; d += 4) {
            const float4 k4 = *reinterpret_cast<const float4*>(kr + d);
            const float4 q4 = *reinterpret_cast<const float4*>(qr + d);
            u4[0] = fmaf(S[d], k4.x, u4[0]); u4[1] = fmaf(S[d + 1], k4.y, u4[1]);
            u4[2] = fmaf(S[d + 2], k4.z, u4[2]); u4[3] = fmaf(S[d + 3], k4.w, u4[3]);
            w4[0] = fmaf(S[d], q4.x, w4[0]); w4[1] = fmaf(S[d + 1], q4.y, w4[1]);
            w4[2] = fmaf(S[d + 2], q4.z, w4[2]); w4[3] = fmaf(S[d + 3], q4.w, w4[3]);
          }
          const float u = (u4[0] + u4[1]) + (u4[2] + u4[3]);
          const float w = (w4[0] + w4[1]) + (w4[2] + w4[3]);
          // the carried state alpha (S - beta k u^T) and its readout alpha (w - beta (k.q) u)
          const float cu = alpha * beta * u;
#pragma unroll
          for (int d = 0; d < kDk; d += 4) {
            const float4 k4 = *reinterpret_cast<const float4*>(kr + d);
            S[d] = fmaf(-cu, k4.x, alpha * S[d]);
            S[d + 1] = fmaf(-cu, k4.y, alpha * S[d + 1]);
            S[d + 2] = fmaf(-cu, k4.z, alpha * S[d + 2]);
            S[d + 3] = fmaf(-cu, k4.w, alpha * S[d + 3]);
          }
          const float y = alpha * (w - beta * kqt * u);
          // a merged level reads out with the lambda of the level it lands in
          contrib = (lv <= lsb ? ls[tt * kLv + lsb + 1] : ls[tt * kLv + lv]) * y;
        }
        // merge: lane lsb+1 of the column takes the sum of the carried states of lanes
        // 0..lsb (its own state is empty after t-1), by an inclusive shuffle scan over
        // lanes 0..lsb+1 in place (lanes above keep their states; lanes 1..lsb are cleared
        // and lane 0 rewritten below)
        for (int off = 1; off <= lsb + 1; off <<= 1) {
#pragma unroll
          for (int d = 0; d < kDk; ++d) {
            const float y = __shfl_up_sync(0xffffffffu, S[d], off, kLv);
            if (lv >= off && lv <= lsb + 1) S[d] += y;
          }
        }
        if (lv >= 1 && lv <= lsb) {
#pragma unroll
          for (int d = 0; d < kDk; ++d) S[d] = 0.f;
        }
      }
      // level 0 <- beta k v^T (column vc); its readout is beta (k.q) v
      if (lv == 0) {
#pragma unroll
        for (int d = 0; d < kDk; d += 4) {
          const float4 k4 = *reinterpret_cast<const float4*>(kr + d);
          const float bv = beta * vc;
          S[d] = bv * k4.x;
          S[d + 1] = bv * k4.y;
          S[d + 2] = bv * k4.z;
          S[d + 3] = bv * k4.w;
        }
        contrib += ls[tt * kLv] * beta * kqt * vc;
      }
#pragma unroll
      for (int o = kLv / 2; o > 0; o >>= 1) contrib += __shfl_xor_sync(0xffffffffu, contrib, o, kLv);
      if (lv == 0) os[tt * kCols + cl] = contrib;
    }
    __syncthreads();
    // ---- the stage's outputs, coalesced over the CTA's columns
    for (int i = tid; i < n * kCols; i += kThreads) {
      const int tt = i / kCols, c = i - tt * kCols;
      if (c0 + c < dv) {
        const int64_t tok = ((int64_t)b * a.Tfull + a.t0 + s * kStage + tt) * a.H + h;
        static_cast<OutT*>(a.out)[tok * dv + c0 + c] = from_f32<OutT>(os[i]);
      }
    }
    // (the next stage's conversion overwrites qf, kf, vs, ls, al, bt only after the
    // barrier at its top; os is rewritten only after the next conversion's barriers)
  }
  // ---- the final per-level state (the decode state after position T-1)
  if (a.state && col_ok && lv < a.state_levels) {
    float* dst = a.state + ((bh * a.L + lv) * (int64_t)dk) * dv + col;
#pragma unroll
    for (int d = 0; d < kDk; ++d)
      if (d < dk) dst[(int64_t)d * dv] = S[d];
  }
}

template <typename InT, typename OutT, int kLv>
cudaError_t launch_lv(const GdnFwdArgs& a, cudaStream_t s) {
  const int row_words = a.dk * (int)sizeof(InT) / 4;
  const size_t smem = (size_t)2 * 2 * kStage * row_words * 4 +
                      sizeof(float) * ((size_t)2 * kStage * kDk + kStage + kStage * kCols +
                                       kStage * kLv + 2 * kStage + kStage * kCols);
  cudaError_t e = cudaFuncSetAttribute(gdn_fwd_kernel<InT, OutT, kLv>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int slices = (a.dv + kCols - 1) / kCols;
  const int64_t grid = (int64_t)a.B * a.H * slices;
  gdn_fwd_kernel<InT, OutT, kLv><<<(unsigned)grid, kLv * kCols, smem, s>>>(a);
  return cudaGetLastError();
}

template <typename InT, typename OutT>
cudaError_t launch_io(const GdnFwdArgs& a, int levels, cudaStream_t s) {
  return levels <= 16 ? launch_lv<InT, OutT, 16>(a, s) : launch_lv<InT, OutT, 32>(a, s);
}

}  // namespace

cudaError_t launch_gdn_fwd(const void* q, const void* k, const void* v, const float* log_a,
                           const float* beta, const float* lam, void* out, float* state, int B,
                           int T, int H, int Hqk, int dk, int dv, int L, int levels, int in_dtype,
                           int out_dtype, cudaStream_t s) {
  GdnFwdArgs a;
  a.q = q; a.k = k; a.v = v; a.log_a = log_a; a.beta = beta; a.lam = lam; a.out = out;
  a.state = state;
  a.B = B; a.T = T; a.H = H; a.hg = H / Hqk; a.dk = dk; a.dv = dv; a.L = L;
  a.Tfull = T; a.t0 = 0; a.state_levels = L;
  if (state) {
    const cudaError_t e =
        cudaMemsetAsync(state, 0, sizeof(float) * (size_t)B * H * L * dk * dv, s);
    if (e != cudaSuccess) return e;
  }
  if (T == 0) return cudaSuccess;
  if (in_dtype == LL_BF16)
    return out_dtype == LL_BF16 ? launch_io<__nv_bfloat16, __nv_bfloat16>(a, levels, s)
                                : launch_io<__nv_bfloat16, float>(a, levels, s);
  return out_dtype == LL_BF16 ? launch_io<float, __nv_bfloat16>(a, levels, s)
                              : launch_io<float, float>(a, levels, s);
}

cudaError_t launch_gdn_fwd_tail(const void* q, const void* k, const void* v, const float* log_a,
                                const float* beta, const float* lam, float* out_f32,
                                float* state, int B, int Tfull, int t0, int H, int Hqk, int dk,
                                int dv, int L, int state_levels, int in_dtype, cudaStream_t s) {
  GdnFwdArgs a;
  a.q = q; a.k = k; a.v = v; a.log_a = log_a; a.beta = beta; a.lam = lam; a.out = out_f32;
  a.state = state;
  a.B = B; a.T = Tfull - t0; a.H = H; a.hg = H / Hqk; a.dk = dk; a.dv = dv; a.L = L;
  a.Tfull = Tfull; a.t0 = t0; a.state_levels = state_levels;
  if (a.T <= 0) return cudaSuccess;
  const int levels = a.T > 1 ? 32 - __builtin_clz((unsigned)(a.T - 1)) + 1 : 1;
  return in_dtype == LL_BF16 ? launch_io<__nv_bfloat16, float>(a, levels, s)
                             : launch_io<float, float>(a, levels, s);
}

}  // namespace ll

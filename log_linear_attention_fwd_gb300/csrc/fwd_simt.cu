// Forward on CUDA cores in fp32 (any head dim <= 128, chunk <= 64, fp32 or bf16 inputs).
//
// Three kernels, following the chunked two-stage algorithm (page "论文阅读：Log-Linear
// Attention", sections 矩阵分解 and 两阶段计算; page "算力终结者来了！…", section 高效训练算法):
//
//   K1 simt_chunk_state   per chunk i: U_i = sum_{s in i} exp(cs_end - cs_s) k_s v_s^T and
//                         lg_i = sum of log a over the chunk (cs = chunk-local prefix sums)
//   K2 level_scan         (level_scan.cu) the Fenwick block states of chunks
//   K3 simt_intra_readout per chunk j: the dense causal C x C product masked by
//                         exp(cs_t - cs_s) * lambda[t, l(t,s)], plus, for every set bit
//                         m-1 of j, lambda[t, lc+m] exp(cs_t + D) q_t^T Tot, with D the log
//                         decay from the block's end to the start of chunk j.
//
// This path is the full-precision one (fp32 storage of every intermediate) and the
// fallback for shapes the tensor-core path does not take.
#include <algorithm>

#include "ll_internal.cuh"

namespace ll {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxOut = 32;     // outputs per thread in K3: C * dv / 256 <= 64 * 128 / 256
constexpr int kRowsPerStage = 32;

template <typename T>
__device__ __forceinline__ float ld(const void* p, int64_t i) {
  return to_f32(reinterpret_cast<const T*>(p)[i]);
}

// Inclusive chunk-local prefix sums of log a, computed by one thread (C <= 64).
__device__ __forceinline__ void chunk_cumsum(const FwdArgs& a, int b, int h, int t0, int n,
                                             float* cs) {
  if (threadIdx.x == 0) {
    float run = 0.f;
    for (int r = 0; r < n; ++r) {
      if (a.log_a) run += a.log_a[((int64_t)b * a.T + t0 + r) * a.H + h];
      cs[r] = run;
    }
  }
}

constexpr int kPad = 128;  // staged rows of K1 are zero-padded to the largest head dim

// K1: thread (td, te) owns U rows [8 td, +8) and columns [8 te, +8) (register-blocked
// outer products over the chunk's rows, k scaled by its decay when staged).
template <typename InT>
__global__ void __launch_bounds__(kThreads) simt_chunk_state(FwdArgs a) {
  extern __shared__ float sm[];
  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int C = a.C, dk = a.dk, dv = a.dv;
  const int t0 = i * C;
  const int n = min(C, a.T - t0);
  float* Ks = sm;               // [C][kPad] w_r k_r
  float* Vs = Ks + C * kPad;    // [C][kPad] v_r
  float* cs = Vs + C * kPad;    // [C]
  float* w = cs + C;            // [C]
  chunk_cumsum(a, b, h, t0, n, cs);
  __syncthreads();
  const float lgi = cs[n - 1];
  for (int r = threadIdx.x; r < n; r += kThreads) w[r] = expf(lgi - cs[r]);
  __syncthreads();
  for (int idx = threadIdx.x; idx < n * kPad; idx += kThreads) {
    const int r = idx / kPad, c = idx - r * kPad;
    const int64_t t = t0 + r;
    const int64_t rk = (int64_t)b * a.sk[0] + t * a.sk[1] + (int64_t)(h / a.hg) * a.sk[2];
    const int64_t rv = (int64_t)b * a.sv[0] + t * a.sv[1] + (int64_t)h * a.sv[2];
    Ks[idx] = c < dk ? w[r] * ld<InT>(a.k, rk + c) : 0.f;
    Vs[idx] = c < dv ? ld<InT>(a.v, rv + c) : 0.f;
  }
  __syncthreads();
  const int td = threadIdx.x >> 4, te = threadIdx.x & 15;
  float acc[8][8];
#pragma unroll
  for (int x = 0; x < 8; ++x)
#pragma unroll
    for (int y = 0; y < 8; ++y) acc[x][y] = 0.f;
  for (int r = 0; r < n; ++r) {
    const float4* kr = reinterpret_cast<const float4*>(Ks + r * kPad + 8 * td);
    const float4* vr = reinterpret_cast<const float4*>(Vs + r * kPad + 8 * te);
    const float4 k0 = kr[0], k1 = kr[1], v0 = vr[0], v1 = vr[1];
    const float kk[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
    const float vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int x = 0; x < 8; ++x)
#pragma unroll
      for (int y = 0; y < 8; ++y) acc[x][y] = fmaf(kk[x], vv[y], acc[x][y]);
  }
  const int64_t bh = (int64_t)b * a.H + h;
  float* U = reinterpret_cast<float*>(a.U) + (bh * a.N + i) * (int64_t)dk * dv;
#pragma unroll
  for (int x = 0; x < 8; ++x) {
    const int d = 8 * td + x;
    if (d >= dk) break;
#pragma unroll
    for (int y = 0; y < 8; ++y)
      if (8 * te + y < dv) U[(int64_t)d * dv + 8 * te + y] = acc[x][y];
  }
  if (threadIdx.x == 0) a.lg[bh * a.N + i] = lgi;
}

template <typename InT, typename OutT>
__global__ void __launch_bounds__(kThreads) simt_intra_readout(FwdArgs a) {
  extern __shared__ float sm[];
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int C = a.C, dk = a.dk, dv = a.dv, L = a.L;
  const int t0 = j * C;
  const int n = min(C, a.T - t0);
  const int64_t bh = (int64_t)b * a.H + h;
  float* Qs = sm;                         // [C][dk]
  float* Ks = Qs + C * dk;                // [C][dk]
  float* Vs = Ks + C * dk;                // [C][dv]
  float* P = Vs + C * dv;                 // [C][C]
  float* Sb = P + C * C;                  // [kRowsPerStage][dv]
  float* cs = Sb + kRowsPerStage * dv;    // [C]
  float* lamS = cs + C;                   // [C][L]
  chunk_cumsum(a, b, h, t0, n, cs);
  for (int idx = threadIdx.x; idx < C * dk; idx += kThreads) {
    const int r = idx / dk, c = idx - r * dk;
    const int64_t t = t0 + r, hq = h / a.hg;
    Qs[idx] = r < n ? ld<InT>(a.q, (int64_t)b * a.sq[0] + t * a.sq[1] + hq * a.sq[2] + c) : 0.f;
    Ks[idx] = r < n ? ld<InT>(a.k, (int64_t)b * a.sk[0] + t * a.sk[1] + hq * a.sk[2] + c) : 0.f;
  }
  for (int idx = threadIdx.x; idx < C * dv; idx += kThreads) {
    const int r = idx / dv, c = idx - r * dv;
    Vs[idx] = r < n ? ld<InT>(a.v, (int64_t)b * a.sv[0] + (int64_t)(t0 + r) * a.sv[1] +
                                       (int64_t)h * a.sv[2] + c)
                    : 0.f;
  }
  for (int idx = threadIdx.x; idx < C * L; idx += kThreads) {
    const int r = idx / L;
    lamS[idx] = r < n ? a.lam[((int64_t)b * a.T + t0) * a.H * L + ((int64_t)r * a.H + h) * L +
                              (idx - r * L)]
                      : 0.f;
  }
  __syncthreads();
  // masked scores of the intra-chunk block D
  for (int idx = threadIdx.x; idx < C * C; idx += kThreads) {
    const int t = idx / C, s = idx - t * C;
    float p = 0.f;
    if (s <= t && t < n) {
      float dot = 0.f;
      for (int d = 0; d < dk; ++d) dot = fmaf(Qs[t * dk + d], Ks[s * dk + d], dot);
      const int lvl = fenwick_level((uint32_t)(t0 + t), (uint32_t)(t0 + s));
      p = expf(cs[t] - cs[s]) * lamS[t * L + lvl] * dot;
    }
    P[idx] = p;
  }
  __syncthreads();
  const int n_out = (C * dv + kThreads - 1) / kThreads;
  float acc[kMaxOut];
#pragma unroll
  for (int o = 0; o < kMaxOut; ++o) {
    acc[o] = 0.f;
    const int idx = threadIdx.x + o * kThreads;
    if (o < n_out && idx < C * dv) {
      const int t = idx / dv, e = idx - t * dv;
      float x = 0.f;
      for (int s = 0; s <= t; ++s) x = fmaf(P[t * C + s], Vs[s * dv + e], x);
      acc[o] = x;
    }
  }
  // inter-chunk levels: one Fenwick block state per set bit of j
  const int elems = dk * dv;
  const float* nodes = reinterpret_cast<const float*>(a.nodes) + bh * a.N * (int64_t)elems;
  const float* lg = a.lg + bh * a.N;
  for (int m = 1; (int64_t(1) << (m - 1)) <= j; ++m) {
    int64_t c;
    if (!inter_block(j, m, &c)) continue;
    float D = 0.f;  // log decay from the end of the block to the start of chunk j
    for (int64_t i = c; i < j; ++i) D += lg[i];
    const float* S = nodes + c * elems;
    float part[kMaxOut];
#pragma unroll
    for (int o = 0; o < kMaxOut; ++o) part[o] = 0.f;
    for (int d0 = 0; d0 < dk; d0 += kRowsPerStage) {
      const int rows = min(kRowsPerStage, dk - d0);
      __syncthreads();
      for (int idx = threadIdx.x; idx < rows * dv; idx += kThreads) Sb[idx] = S[d0 * dv + idx];
      __syncthreads();
#pragma unroll
      for (int o = 0; o < kMaxOut; ++o) {
        const int idx = threadIdx.x + o * kThreads;
        if (o < n_out && idx < C * dv) {
          const int t = idx / dv, e = idx - t * dv;
          float x = part[o];
          for (int r = 0; r < rows; ++r) x = fmaf(Qs[t * dk + d0 + r], Sb[r * dv + e], x);
          part[o] = x;
        }
      }
    }
    const int lvl = a.lc + m;
#pragma unroll
    for (int o = 0; o < kMaxOut; ++o) {
      const int idx = threadIdx.x + o * kThreads;
      if (o < n_out && idx < C * dv) {
        const int t = idx / dv;
        acc[o] = fmaf(lamS[t * L + lvl] * expf(cs[t < n ? t : 0] + D), part[o], acc[o]);
      }
    }
  }
  OutT* out = reinterpret_cast<OutT*>(a.out);
#pragma unroll
  for (int o = 0; o < kMaxOut; ++o) {
    const int idx = threadIdx.x + o * kThreads;
    if (o < n_out && idx < C * dv) {
      const int t = idx / dv, e = idx - t * dv;
      if (t < n)
        out[(int64_t)b * a.so[0] + (int64_t)(t0 + t) * a.so[1] + (int64_t)h * a.so[2] + e] =
            from_f32<OutT>(acc[o]);
    }
  }
}

template <typename InT, typename OutT>
cudaError_t launch_typed(const FwdArgs& a, cudaStream_t s, StageEvents* ev) {
  const dim3 grid_c(a.N, a.H, a.B);
  const size_t sm1 = sizeof(float) * ((size_t)a.C * 2 * kPad + 2 * a.C);
  const size_t sm3 = sizeof(float) * ((size_t)a.C * (2 * a.dk + a.dv) + (size_t)a.C * a.C +
                                      (size_t)kRowsPerStage * a.dv + a.C + (size_t)a.C * a.L);
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(simt_chunk_state<InT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sm1)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(simt_intra_readout<InT, OutT>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3)) !=
      cudaSuccess)
    return e;
  if (ev && (e = ev->record(s)) != cudaSuccess) return e;
  simt_chunk_state<InT><<<grid_c, kThreads, sm1, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (ev && (e = ev->record(s)) != cudaSuccess) return e;
  if (a.N > 1) {
    if ((e = launch_level_scan(a, s)) != cudaSuccess) return e;
    if (ev && (e = ev->record(s)) != cudaSuccess) return e;
  }
  simt_intra_readout<InT, OutT><<<grid_c, kThreads, sm3, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (ev && (e = ev->record(s)) != cudaSuccess) return e;
  return ev ? ev->finish(s) : cudaSuccess;
}

template <typename InT>
cudaError_t launch_states_typed(const FwdArgs& a, cudaStream_t s) {
  const size_t sm1 = sizeof(float) * ((size_t)a.C * 2 * kPad + 2 * a.C);
  cudaError_t e = cudaFuncSetAttribute(simt_chunk_state<InT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1);
  if (e != cudaSuccess) return e;
  simt_chunk_state<InT><<<dim3(a.N, a.H, a.B), kThreads, sm1, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return a.N > 1 ? launch_level_scan(a, s) : cudaSuccess;
}

}  // namespace

cudaError_t launch_simt_states(const FwdArgs& a, int in_dtype, cudaStream_t s) {
  return in_dtype == LL_F32 ? launch_states_typed<float>(a, s)
                            : launch_states_typed<__nv_bfloat16>(a, s);
}

cudaError_t launch_simt_forward(const FwdArgs& a, int in_dtype, int out_dtype, cudaStream_t s,
                                StageEvents* ev) {
  if (in_dtype == LL_F32 && out_dtype == LL_F32) return launch_typed<float, float>(a, s, ev);
  if (in_dtype == LL_F32 && out_dtype == LL_BF16)
    return launch_typed<float, __nv_bfloat16>(a, s, ev);
  if (in_dtype == LL_BF16 && out_dtype == LL_F32)
    return launch_typed<__nv_bfloat16, float>(a, s, ev);
  return launch_typed<__nv_bfloat16, __nv_bfloat16>(a, s, ev);
}

}  // namespace ll

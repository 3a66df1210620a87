// Batched decode step with the lssb rule (page "论文阅读：Log-Linear Attention", section
// 解码：基于 lssb 的状态更新; slide deck "論文紹介：Log Linear Attention", slide 21).
//
// One CTA per (b, h).  Each thread owns one 4-column group of the d_k x d_v state and a
// strided set of rows; for every element it loads the levels that hold data, applies
// merge / promote / clear / decay, stores the levels that change and accumulates its
// share of the readout sum_l lambda_l q^T S_l.  The levels are streamed once with 16-byte
// loads and stores marked evict-first: the state (2 GB at B=128, H=16, L=15, d=128) is
// far larger than L2 and has no reuse inside a step.
#include "ll_internal.cuh"

namespace ll {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxLv = 64;   // levels whose lambda is staged

template <typename T>
__device__ __forceinline__ float ldx(const void* p, int64_t i) {
  return to_f32(reinterpret_cast<const T*>(p)[i]);
}

__device__ __forceinline__ float4 f4_fma(float s, float4 x, float4 y) {
  return make_float4(fmaf(s, x.x, y.x), fmaf(s, x.y, y.y), fmaf(s, x.z, y.z), fmaf(s, x.w, y.w));
}
__device__ __forceinline__ float4 f4_add(float4 x, float4 y) {
  return make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w);
}
__device__ __forceinline__ float4 f4_scale(float s, float4 x) {
  return make_float4(s * x.x, s * x.y, s * x.z, s * x.w);
}

// kFew > 0: up to kFew touched levels are loaded into registers before any is used (all
// loads of an element in flight at once); kFew == 0: any count, one level at a time.
template <typename InT, typename OutT, int kFew>
__global__ void __launch_bounds__(kThreads, kFew == 16 ? 1 : 2) decode_step_kernel(
    float* __restrict__ state, const void* __restrict__ q, const void* __restrict__ k,
    const void* __restrict__ v, const float* __restrict__ log_a, const float* __restrict__ lam,
    void* __restrict__ out, int H, int hg, int dk, int dv, int L, DecodePlan plan) {
  __shared__ float qs[128];
  __shared__ float ks[128];
  __shared__ float lam_s[kMaxLv];
  __shared__ float4 red[kThreads];
  const int64_t bh = blockIdx.x;
  const int64_t bq = bh / hg;  // (b, q/k head): H = Hqk * hg, head h reads q/k head h / hg
  const int tid = threadIdx.x;
  for (int i = tid; i < dk; i += kThreads) {
    qs[i] = ldx<InT>(q, bq * dk + i);
    ks[i] = ldx<InT>(k, bq * dk + i);
  }
  for (int i = tid; i < L && i < kMaxLv; i += kThreads) lam_s[i] = lam[bh * L + i];
  __syncthreads();
  const float a = log_a ? expf(log_a[bh]) : 1.f;
  const bool decay = log_a != nullptr;
  const int groups = dv >> 2;          // float4 column groups per row (divides kThreads)
  const int cg = tid % groups;
  const int row0 = tid / groups;
  const int row_step = kThreads / groups;
  const float4 vv = make_float4(ldx<InT>(v, bh * dv + 4 * cg), ldx<InT>(v, bh * dv + 4 * cg + 1),
                                ldx<InT>(v, bh * dv + 4 * cg + 2), ldx<InT>(v, bh * dv + 4 * cg + 3));
  const int64_t lstride = (int64_t)dk * dv;  // floats per level
  float4* S = reinterpret_cast<float4*>(state + bh * L * lstride);
  const int64_t l4 = lstride >> 2;           // float4 per level
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);

  if (plan.t_zero) {
    for (int r = row0; r < dk; r += row_step) {
      const int64_t off = (int64_t)r * groups + cg;
      const float4 kv = f4_scale(ks[r], vv);
      __stcs(S + off, kv);
      for (int lv = 1; lv < L; ++lv) __stcs(S + lv * l4 + off, zero);
      acc = f4_fma(qs[r] * lam_s[0], kv, acc);
    }
  } else if (kFew > 0) {
    // touched levels: plan.lv[0..n_low) = 0..l (merged), then the kept levels above l+1
    const int l = plan.l;
    const int n_low = l + 1;
    const int cnt = n_low + plan.n_hi;
    const float lam_m = lam_s[l + 1];
    // Two rows per pass, every load of both in flight before either is used: with 2
    // CTAs of 256 threads per SM that keeps ~100 KB of state reads outstanding per SM.
    for (int r2 = row0; r2 < dk; r2 += 2 * row_step) {
      float4 x2[2][kFew > 0 ? kFew : 1];
#pragma unroll
      for (int p2 = 0; p2 < 2; ++p2) {
        const int r = r2 + p2 * row_step;
        if (r < dk) {
          const int64_t off = (int64_t)r * groups + cg;
#pragma unroll
          for (int i = 0; i < kFew; ++i)
            if (i < cnt) x2[p2][i] = __ldcs(S + plan.lv[i] * l4 + off);
        }
      }
#pragma unroll
      for (int p2 = 0; p2 < 2; ++p2) {
        const int r = r2 + p2 * row_step;
        if (r >= dk) break;
        const int64_t off = (int64_t)r * groups + cg;
        const float4* x = x2[p2];
        float4 merged = zero;
#pragma unroll
        for (int i = 0; i < kFew; ++i)
          if (i < n_low) merged = f4_add(merged, x[i]);
        merged = f4_scale(a, merged);
        const float4 kv = f4_scale(ks[r], vv);
        __stcs(S + off, kv);
        __stcs(S + (l + 1) * l4 + off, merged);
        float4 ro = f4_fma(lam_s[0], kv, f4_scale(lam_m, merged));
#pragma unroll
        for (int i = 1; i < kFew; ++i) {
          if (i < n_low) {
            __stcs(S + i * l4 + off, zero);
          } else if (i < cnt) {
            float4 y = x[i];
            if (decay) {
              y = f4_scale(a, y);
              __stcs(S + plan.lv[i] * l4 + off, y);
            }
            ro = f4_fma(lam_s[plan.lv[i]], y, ro);
          }
        }
        acc = f4_fma(qs[r], ro, acc);
      }
    }
  } else {
    // any number of levels: same update, one level at a time
    const int l = plan.l;
    const int n_low = l + 1;
    const int cnt = n_low + plan.n_hi;
    const float lam_m = lam_s[l + 1];
    for (int r = row0; r < dk; r += row_step) {
      const int64_t off = (int64_t)r * groups + cg;
      float4 merged = zero;
      for (int i = 0; i < n_low; ++i) merged = f4_add(merged, __ldcs(S + i * l4 + off));
      merged = f4_scale(a, merged);
      float4 ro = f4_scale(lam_m, merged);
      for (int i = n_low; i < cnt; ++i) {
        float4 y = __ldcs(S + plan.lv[i] * l4 + off);
        if (decay) {
          y = f4_scale(a, y);
          __stcs(S + plan.lv[i] * l4 + off, y);
        }
        ro = f4_fma(lam_s[plan.lv[i]], y, ro);
      }
      const float4 kv = f4_scale(ks[r], vv);
      for (int i = 1; i < n_low; ++i) __stcs(S + i * l4 + off, zero);
      __stcs(S + (l + 1) * l4 + off, merged);
      __stcs(S + off, kv);
      acc = f4_fma(qs[r], f4_fma(lam_s[0], kv, ro), acc);
    }
  }
  // reduce the readout over the threads that share a column group
  red[tid] = acc;
  __syncthreads();
  if (tid < groups) {
    float4 s = red[tid];
    for (int i = tid + groups; i < kThreads; i += groups) s = f4_add(s, red[i]);
    OutT* o = reinterpret_cast<OutT*>(out) + bh * dv + 4 * tid;
    o[0] = from_f32<OutT>(s.x);
    o[1] = from_f32<OutT>(s.y);
    o[2] = from_f32<OutT>(s.z);
    o[3] = from_f32<OutT>(s.w);
  }
}

template <typename InT, typename OutT>
cudaError_t launch_typed(float* state, const void* q, const void* k, const void* v,
                         const float* log_a, const float* lam, void* out, int B, int H, int hg,
                         int dk, int dv, int L, const DecodePlan& plan, cudaStream_t s) {
  const unsigned grid = (unsigned)((int64_t)B * H);
  const int touched = plan.t_zero ? 0 : plan.l + 1 + plan.n_hi;
  if (touched <= 8)
    decode_step_kernel<InT, OutT, 8><<<grid, kThreads, 0, s>>>(state, q, k, v, log_a, lam, out, H,
                                                                hg, dk, dv, L, plan);
  else if (touched <= 16)
    decode_step_kernel<InT, OutT, 16><<<grid, kThreads, 0, s>>>(state, q, k, v, log_a, lam, out, H,
                                                                 hg, dk, dv, L, plan);
  else
    decode_step_kernel<InT, OutT, 0><<<grid, kThreads, 0, s>>>(state, q, k, v, log_a, lam, out, H,
                                                                hg, dk, dv, L, plan);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(float* state, const void* q, const void* k, const void* v,
                          const float* log_a, const float* lam, void* out, int B, int H, int Hqk,
                          int dk, int dv, int L, const DecodePlan& plan, int in_dtype,
                          int out_dtype, cudaStream_t s) {
  const int hg = H / Hqk;
  if (in_dtype == LL_F32 && out_dtype == LL_F32)
    return launch_typed<float, float>(state, q, k, v, log_a, lam, out, B, H, hg, dk, dv, L, plan, s);
  if (in_dtype == LL_F32)
    return launch_typed<float, __nv_bfloat16>(state, q, k, v, log_a, lam, out, B, H, hg, dk, dv, L,
                                              plan, s);
  if (out_dtype == LL_F32)
    return launch_typed<__nv_bfloat16, float>(state, q, k, v, log_a, lam, out, B, H, hg, dk, dv, L,
                                              plan, s);
  return launch_typed<__nv_bfloat16, __nv_bfloat16>(state, q, k, v, log_a, lam, out, B, H, hg, dk,
                                                    dv, L, plan, s);
}

}  // namespace ll

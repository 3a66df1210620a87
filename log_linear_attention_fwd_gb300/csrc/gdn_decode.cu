// Batched decode step of Log-Linear Gated DeltaNet with the lssb rule.
//
// The log-linear form keeps the model's own transition and composes its mask with the
// Fenwick mask (page "算力终结者来了！…", section 对Mamba-2和门控DeltaNet的对数线性推广; page
// "论文阅读：Log-Linear Attention", section 与已有模型的组合).  The transition is the gated
// delta rule (Yang, Kautz and Hatamizadeh, "Gated Delta Networks", 2024): with the state
// stored [d_k][d_v] (o = S^T q),
//     A_t = alpha_t (I - beta_t k_t k_t^T),  every state held after t-1:  S <- A_t S,
// then the lssb merge / promote / clear of the first page's section 解码：基于 lssb 的状态
// 更新, and level 0 <- beta_t k_t v_t^T; out = sum_l lambda_l S_l^T q.
//
// Column e of A_t S needs only column e of S and u_e = (S^T k)_e, so the d_v columns split
// across CTAs: one CTA per (b, h, 32-column slice), which covers one 128-byte line of every
// state row.  With u = S^T k and w = S^T q of an old level, its carried state is
// alpha (S - beta k u^T) and that state's readout is alpha (w - beta (k.q) u); a merged
// level reads out with lambda of the level it lands in.
//
// Two passes per CTA keep the registers few, so that four CTAs share an SM and keep many
// loads in flight: pass 1 streams the touched levels from HBM and forms u and w (each
// thread its rows, then the lanes and warps that share a column group), its first loads
// issued before the CTA reads q, k and lambda; pass 2 reads the same rows again, from L2
// where pass 1 just left them, and writes the carried states.  The second reads and
// every write are marked evict-first.  Measured at B128 H16 d128 L15 t = 12345 (six levels
// read, seven written): one pass holding every level in registers (two CTAs per SM) took
// 569 us; two passes at two, three and four CTAs per SM 422, 352 and 330 us; with the
// early first loads 320 us.
#include "ll_internal.cuh"

namespace ll {
namespace {

constexpr int kThreads = 256;
constexpr int kCols = 32;      // d_v columns per CTA (one 128-byte line of an fp32 row)
constexpr int kRows = 4;       // rows per thread: d_k <= 128 rows over >= 32 row slots
constexpr int kBatch1 = 2;     // levels whose loads are issued together: pass 1 (HBM)
constexpr int kBatch2 = 1;     // and pass 2 (L2), which also holds the merged rows
constexpr int kMaxLv = 64;

template <typename T>
__device__ __forceinline__ float ldx(const void* p, int64_t i) {
  return to_f32(reinterpret_cast<const T*>(p)[i]);
}

__device__ __forceinline__ float4 f4(float a) { return make_float4(a, a, a, a); }
__device__ __forceinline__ float4 f4_fma(float s, float4 x, float4 y) {
  return make_float4(fmaf(s, x.x, y.x), fmaf(s, x.y, y.y), fmaf(s, x.z, y.z), fmaf(s, x.w, y.w));
}
__device__ __forceinline__ float4 f4_add(float4 x, float4 y) {
  return make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w);
}
__device__ __forceinline__ float4 f4_scale(float s, float4 x) {
  return make_float4(s * x.x, s * x.y, s * x.z, s * x.w);
}
__device__ __forceinline__ float4 f4_shfl_xor(float4 x, int o) {
  return make_float4(__shfl_xor_sync(0xffffffffu, x.x, o), __shfl_xor_sync(0xffffffffu, x.y, o),
                     __shfl_xor_sync(0xffffffffu, x.z, o), __shfl_xor_sync(0xffffffffu, x.w, o));
}

template <typename InT, typename OutT>
__global__ void __launch_bounds__(kThreads, 4) gdn_decode_kernel(
    float* __restrict__ state, const void* __restrict__ q, const void* __restrict__ k,
    const void* __restrict__ v, const float* __restrict__ log_a, const float* __restrict__ beta,
    const float* __restrict__ lam, void* __restrict__ out, int hg, int dk, int dv, int L,
    DecodePlan plan) {
  __shared__ float qs[128];
  __shared__ float ks[128];
  __shared__ float lam_s[kMaxLv];
  __shared__ float4 part[kMaxLv][2][kCols / 4];  // u and w of every touched level
  const int cpc = dv < kCols ? dv : kCols;       // columns of this CTA
  const int slices = dv / cpc;
  const int64_t bh = blockIdx.x / slices;
  const int slice = blockIdx.x - (int)(bh * slices);
  const int64_t bq = bh / hg;  // (b, q/k head): head h reads q/k head h / hg
  const int tid = threadIdx.x, lane = tid & 31;
  const int groups = cpc >> 2;                 // float4 column groups of the slice: 1, 2, 4 or 8
  const int cg = tid % groups;
  const int row0 = tid / groups;
  const int row_step = kThreads / groups;      // 256, 128, 64 or 32
  const int col = slice * cpc + 4 * cg;        // first column of this thread's group
  const int64_t l4 = ((int64_t)dk * dv) >> 2;  // float4 per level
  float4* S = reinterpret_cast<float4*>(state + bh * L * (int64_t)dk * dv);
  const int g_all = dv >> 2;                   // float4 per row
  const float4 zero = f4(0.f);
  const int cnt = plan.t_zero ? 0 : plan.l + 1 + plan.n_hi;
  // the first batch of pass 1 goes out before anything else: it needs no q, k or lambda
  float4 x1[kBatch1][kRows];
#pragma unroll
  for (int i = 0; i < kBatch1; ++i)
#pragma unroll
    for (int rr = 0; rr < kRows; ++rr) {
      const int r = row0 + rr * row_step;
      x1[i][rr] = (i < cnt && r < dk) ? S[plan.lv[i] * l4 + (int64_t)r * g_all + (col >> 2)]
                                      : zero;
    }
  for (int i = tid; i < cnt * 2 * (kCols / 4); i += kThreads)
    (&part[0][0][0])[i] = zero;
  for (int i = tid; i < dk; i += kThreads) {
    qs[i] = ldx<InT>(q, bq * dk + i);
    ks[i] = ldx<InT>(k, bq * dk + i);
  }
  for (int i = tid; i < L && i < kMaxLv; i += kThreads) lam_s[i] = lam[bh * L + i];
  __syncthreads();
  const float a = log_a ? expf(log_a[bh]) : 1.f;
  const float bt = beta[bh];
  float kq = 0.f;  // k . q: every warp forms the same sum, lanes over features
  for (int i = lane; i < dk; i += 32) kq = fmaf(ks[i], qs[i], kq);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
  const float4 vv = make_float4(ldx<InT>(v, bh * dv + col), ldx<InT>(v, bh * dv + col + 1),
                                ldx<InT>(v, bh * dv + col + 2), ldx<InT>(v, bh * dv + col + 3));
  float4 o = f4_scale(lam_s[0] * bt * kq, vv);  // level 0 (beta k v^T) reads out
                                                // lambda_0 beta (k.q) v

  if (plan.t_zero) {
#pragma unroll
    for (int rr = 0; rr < kRows; ++rr) {
      const int r = row0 + rr * row_step;
      if (r < dk) {
        const int64_t off = (int64_t)r * g_all + (col >> 2);
        __stcs(S + off, f4_scale(bt * ks[r], vv));
        for (int lv = 1; lv < L; ++lv) __stcs(S + lv * l4 + off, zero);
      }
    }
  } else {
    const int l = plan.l;
    const int n_low = l + 1;                   // levels 0..l merge into level l+1
    // ---- pass 1: u = S^T k and w = S^T q of every touched level
    auto reduce_batch = [&](const float4 (&x)[kBatch1][kRows], int i0) {
#pragma unroll
      for (int i = 0; i < kBatch1; ++i) {
        if (i0 + i >= cnt) break;
        float4 pu = zero, pw = zero;
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
          const int r = row0 + rr * row_step;
          if (r < dk) {
            pu = f4_fma(ks[r], x[i][rr], pu);
            pw = f4_fma(qs[r], x[i][rr], pw);
          }
        }
        for (int off = groups; off < 32; off <<= 1) {  // lanes of the same column group
          pu = f4_add(pu, f4_shfl_xor(pu, off));
          pw = f4_add(pw, f4_shfl_xor(pw, off));
        }
        if (lane < groups) {  // then the warps, by shared-memory atomics
          float* du = reinterpret_cast<float*>(&part[i0 + i][0][lane]);
          float* dw = reinterpret_cast<float*>(&part[i0 + i][1][lane]);
          atomicAdd(du, pu.x); atomicAdd(du + 1, pu.y); atomicAdd(du + 2, pu.z); atomicAdd(du + 3, pu.w);
          atomicAdd(dw, pw.x); atomicAdd(dw + 1, pw.y); atomicAdd(dw + 2, pw.z); atomicAdd(dw + 3, pw.w);
        }
      }
    };
    reduce_batch(x1, 0);
    for (int i0 = kBatch1; i0 < cnt; i0 += kBatch1) {
      float4 x[kBatch1][kRows];
#pragma unroll
      for (int i = 0; i < kBatch1; ++i)
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
          const int r = row0 + rr * row_step;
          x[i][rr] = (i0 + i < cnt && r < dk)
                         ? S[plan.lv[i0 + i] * l4 + (int64_t)r * g_all + (col >> 2)]
                         : zero;
        }
      reduce_batch(x, i0);
    }
    __syncthreads();
    // ---- pass 2: the carried states (from L2), merged into level l+1 or stored in place
    float4 merged[kRows];
#pragma unroll
    for (int rr = 0; rr < kRows; ++rr) merged[rr] = zero;
    for (int i0 = 0; i0 < cnt; i0 += kBatch2) {
      float4 x[kBatch2][kRows];
#pragma unroll
      for (int i = 0; i < kBatch2; ++i)
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
          const int r = row0 + rr * row_step;
          x[i][rr] = (i0 + i < cnt && r < dk)
                         ? __ldcs(S + plan.lv[i0 + i] * l4 + (int64_t)r * g_all + (col >> 2))
                         : zero;
        }
#pragma unroll
      for (int i = 0; i < kBatch2; ++i) {
        if (i0 + i >= cnt) break;
        const float4 u = part[i0 + i][0][cg], w = part[i0 + i][1][cg];
        const int lv = plan.lv[i0 + i];
        const bool low = i0 + i < n_low;
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
          const int r = row0 + rr * row_step;
          if (r >= dk) break;
          const float4 y = f4_scale(a, f4_fma(-bt * ks[r], u, x[i][rr]));  // alpha (S - beta k u^T)
          if (low)
            merged[rr] = f4_add(merged[rr], y);
          else
            __stcs(S + lv * l4 + (int64_t)r * g_all + (col >> 2), y);
        }
        o = f4_fma(lam_s[low ? l + 1 : lv] * a, f4_fma(-bt * kq, u, w), o);
      }
    }
#pragma unroll
    for (int rr = 0; rr < kRows; ++rr) {
      const int r = row0 + rr * row_step;
      if (r >= dk) break;
      const int64_t off = (int64_t)r * g_all + (col >> 2);
      __stcs(S + (l + 1) * l4 + off, merged[rr]);
      for (int lv = 1; lv <= l; ++lv) __stcs(S + lv * l4 + off, zero);
      __stcs(S + off, f4_scale(bt * ks[r], vv));
    }
  }
  if (row0 == 0) {
    OutT* dst = reinterpret_cast<OutT*>(out) + bh * dv + col;
    dst[0] = from_f32<OutT>(o.x);
    dst[1] = from_f32<OutT>(o.y);
    dst[2] = from_f32<OutT>(o.z);
    dst[3] = from_f32<OutT>(o.w);
  }
}

template <typename InT, typename OutT>
cudaError_t launch_typed(float* state, const void* q, const void* k, const void* v,
                         const float* log_a, const float* beta, const float* lam, void* out, int B,
                         int H, int hg, int dk, int dv, int L, const DecodePlan& plan,
                         cudaStream_t s) {
  const int slices = dv / (dv < kCols ? dv : kCols);
  const unsigned grid = (unsigned)((int64_t)B * H * slices);
  gdn_decode_kernel<InT, OutT><<<grid, kThreads, 0, s>>>(state, q, k, v, log_a, beta, lam, out,
                                                          hg, dk, dv, L, plan);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gdn_decode(float* state, const void* q, const void* k, const void* v,
                              const float* log_a, const float* beta, const float* lam, void* out,
                              int B, int H, int Hqk, int dk, int dv, int L, const DecodePlan& plan,
                              int in_dtype, int out_dtype, cudaStream_t s) {
  const int hg = H / Hqk;
  if (in_dtype == LL_F32 && out_dtype == LL_F32)
    return launch_typed<float, float>(state, q, k, v, log_a, beta, lam, out, B, H, hg, dk, dv, L,
                                      plan, s);
  if (in_dtype == LL_F32)
    return launch_typed<float, __nv_bfloat16>(state, q, k, v, log_a, beta, lam, out, B, H, hg, dk,
                                              dv, L, plan, s);
  if (out_dtype == LL_F32)
    return launch_typed<__nv_bfloat16, float>(state, q, k, v, log_a, beta, lam, out, B, H, hg, dk,
                                              dv, L, plan, s);
  return launch_typed<__nv_bfloat16, __nv_bfloat16>(state, q, k, v, log_a, beta, lam, out, B, H,
                                                    hg, dk, dv, L, plan, s);
}

}  // namespace ll

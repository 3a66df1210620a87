// Prefill -> decode handoff: the per-level decode state at position T-1, built from what
// the forward leaves in its workspace (page "论文阅读：Log-Linear Attention", sections
// 循环形式与输出计算 (one state per Fenwick bucket) and 两阶段计算 (the block states of
// chunks); the Dynamic Linear Attention page restates the buckets).
//
// The state at position t holds, per level l, S^(l) = sum over the level-l Fenwick
// bucket of t of exp(cum_t - cum_s) k_s v_s^T.  With t = T-1 in tile j (tiles of
// 2^lc tokens):
//   * level 0 is {t}; levels 1..lc whose bit is set in t are token ranges inside tile j:
//     summed here from k and v with their decays to t;
//   * level lc + m whose bit m-1 is set in j is the aligned block of 2^(m-1) tiles
//     ending at tile c = (j >> (m-1)) << (m-1): the forward's block state of slot c,
//     decayed from the block's end to t by exp(D_m + cs_t) (D_m = sum of the tile log
//     decays over [c, j), cs_t = log decay from tile j's start to t);
//   * every other level is zero.
// One CTA per (level, b, h, slice of 32 state rows), so that a few CTAs per SM keep
// enough loads and stores in flight.
#include "ll_internal.cuh"

namespace ll {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxTile = 128;   // largest tile of either forward path
constexpr int kMaxDim = 128;    // d_k, d_v <= 128
constexpr int kSliceRows = 32;  // state rows per CTA (4 x 64 threads of 8 rows x 2 columns)

template <typename InT>
__device__ __forceinline__ float ld(const void* p, int64_t i) {
  return to_f32(reinterpret_cast<const InT*>(p)[i]);
}

// Inclusive prefix sum of x over the CTA (x may be zero past the valid range).
__device__ float block_prefix(float x, float* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  float pre = 0.f;
  for (int w = 0; w < warp; ++w) pre += sh[w];
  __syncthreads();
  return x + pre;
}

// Sum of x over the CTA.
__device__ float block_sum(float x, float* sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = x;
  __syncthreads();
  float s = 0.f;
  for (int w = 0; w < kThreads / 32; ++w) s += sh[w];
  __syncthreads();
  return s;
}

// tc_layout: block states are bf16 (tensor-core path; odd slots are U_{c-1}); otherwise
// fp32 for every slot.  Both are row-major [d_k][d_v], the layout of the state.
// One CTA per (level, b*h, slice of kSliceRows state rows).
template <typename InT, bool kTcLayout>
__global__ void __launch_bounds__(kThreads) prefill_state_kernel(FwdArgs a, float* state,
                                                                 bool vec_in) {
  extern __shared__ float sm[];
  const int lvl = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int r0 = blockIdx.z * kSliceRows;  // this CTA's state rows [r0, r0 + rows)
  const int b = (int)(bh / a.H), h = (int)(bh - (int64_t)b * a.H);
  const int dk = a.dk, dv = a.dv, lc = a.lc;
  if (r0 >= dk) return;
  const int rows = min(kSliceRows, dk - r0);
  const int64_t elems = (int64_t)rows * dv;  // of this slice, contiguous in the state
  float* S = state + (bh * a.L + lvl) * (int64_t)dk * dv + (int64_t)r0 * dv;
  const int t = a.T - 1, j = t >> lc, t0 = j << lc;
  const bool vec = (dv & 7) == 0;  // 8 columns per step: 16-byte loads and stores

  // this level's bucket [lo, hi) of positions
  int lo, hi;
  bool has;
  if (lvl == 0) {
    has = true;
    lo = t;
    hi = t + 1;
  } else {
    has = lvl <= 31 && ((t >> (lvl - 1)) & 1);
    hi = has ? (t >> (lvl - 1)) << (lvl - 1) : 0;
    lo = hi - (has ? 1 << (lvl - 1) : 0);
  }
  if (!has) {
    if (vec) {
      for (int64_t i = threadIdx.x; i < elems / 4; i += kThreads)
        reinterpret_cast<float4*>(S)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      for (int64_t i = threadIdx.x; i < elems; i += kThreads) S[i] = 0.f;
    }
    return;
  }

  // cs[i] = log decay over tile j from its start to position t0 + i (inclusive)
  float* red = sm;                  // [32]
  float* cs = sm + 32;              // [kMaxTile]
  float* w = cs + kMaxTile;         // [kMaxTile] weights of the bucket's positions
  float* ks = w + kMaxTile;         // [bucket][kSliceRows], then v [bucket][128]
  const int n = t - t0 + 1;         // positions of tile j up to t
  {
    const float la = (a.log_a && (int)threadIdx.x < n)
                         ? a.log_a[((int64_t)b * a.T + t0 + threadIdx.x) * a.H + h]
                         : 0.f;
    const float c = block_prefix(la, red);
    if ((int)threadIdx.x < n) cs[threadIdx.x] = c;
    __syncthreads();
  }
  const float cs_t = cs[n - 1];

  if (lvl <= lc) {
    // a range of positions inside tile j: sum_s exp(cs_t - cs_s) k_s v_s^T over the
    // slice's rows, as outer products accumulated in registers: thread (td, te) owns rows
    // [8 td, 8 td + 8) of the slice and columns 2 te, 2 te + 1; the slice's columns of k
    // (scaled by the decay) and the rows of v are staged zero-padded.
    const int nb = hi - lo;
    float* vs = ks + nb * kSliceRows;
    for (int i = threadIdx.x; i < nb; i += kThreads) w[i] = __expf(cs_t - cs[lo - t0 + i]);
    __syncthreads();
    if (sizeof(InT) == 2 && vec_in && rows == kSliceRows) {
      // bf16 rows with 16-byte alignment: 8 values per load, all of them in flight at once
      for (int i = threadIdx.x; i < nb * (kSliceRows / 8); i += kThreads) {
        const int r = i / (kSliceRows / 8), q = i - r * (kSliceRows / 8);
        const int64_t tok_k = ((int64_t)b * a.T + lo + r) * a.Hqk + h / a.hg;
        const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const InT*>(a.k) +
                                                        tok_k * dk + r0 + 8 * q);
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
          ks[r * kSliceRows + 8 * q + 2 * e] = w[r] * f.x;
          ks[r * kSliceRows + 8 * q + 2 * e + 1] = w[r] * f.y;
        }
      }
      const int vq = dv / 8;
      for (int i = threadIdx.x; i < nb * vq; i += kThreads) {
        const int r = i / vq, q = i - r * vq;
        const int64_t tok = ((int64_t)b * a.T + lo + r) * a.H + h;
        const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const InT*>(a.v) + tok * dv +
                                                        8 * q);
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
          vs[r * kMaxDim + 8 * q + 2 * e] = f.x;
          vs[r * kMaxDim + 8 * q + 2 * e + 1] = f.y;
        }
      }
      for (int i = threadIdx.x; i < nb * (kMaxDim - dv); i += kThreads) {
        const int r = i / (kMaxDim - dv), d = dv + i - r * (kMaxDim - dv);
        vs[r * kMaxDim + d] = 0.f;
      }
    } else {
      // (unrolled, so that each thread has several loads in flight)
#pragma unroll 8
      for (int i = threadIdx.x; i < nb * kSliceRows; i += kThreads) {
        const int r = i / kSliceRows, d = i - r * kSliceRows;
        const int64_t tok_k = ((int64_t)b * a.T + lo + r) * a.Hqk + h / a.hg;
        ks[i] = d < rows ? w[r] * ld<InT>(a.k, tok_k * dk + r0 + d) : 0.f;
      }
#pragma unroll 8
      for (int i = threadIdx.x; i < nb * kMaxDim; i += kThreads) {
        const int r = i / kMaxDim, d = i - r * kMaxDim;
        const int64_t tok = ((int64_t)b * a.T + lo + r) * a.H + h;
        vs[i] = d < dv ? ld<InT>(a.v, tok * dv + d) : 0.f;
      }
    }
    __syncthreads();
    const int td = threadIdx.x >> 6, te = threadIdx.x & 63;
    float acc[8][2];
#pragma unroll
    for (int x = 0; x < 8; ++x) acc[x][0] = acc[x][1] = 0.f;
    for (int r = 0; r < nb; ++r) {
      const float4* kr = reinterpret_cast<const float4*>(ks + r * kSliceRows + 8 * td);
      const float2 vv = reinterpret_cast<const float2*>(vs + r * kMaxDim)[te];
      const float4 k0 = kr[0], k1 = kr[1];
      const float kk[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        acc[x][0] = fmaf(kk[x], vv.x, acc[x][0]);
        acc[x][1] = fmaf(kk[x], vv.y, acc[x][1]);
      }
    }
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      const int d = 8 * td + x;
      if (d >= rows) break;
      float* row = S + (int64_t)d * dv;
      if ((dv & 1) == 0 && 2 * te < dv) {
        reinterpret_cast<float2*>(row)[te] = make_float2(acc[x][0], acc[x][1]);
      } else {
        if (2 * te < dv) row[2 * te] = acc[x][0];
        if (2 * te + 1 < dv) row[2 * te + 1] = acc[x][1];
      }
    }
    return;
  }

  // a block of 2^(lvl - lc - 1) tiles ending at tile c: the block state of slot c,
  // decayed to t
  const int c = hi >> lc;
  float D = 0.f;  // sum of the tile log decays over [c, j)
  for (int i = c + (int)threadIdx.x; i < j; i += kThreads) D += a.lg[bh * a.N + i];
  D = block_sum(D, red);
  const float g = __expf(D + cs_t);
  const int64_t src0 = (bh * a.N + ((kTcLayout && (c & 1)) ? c - 1 : c)) * (int64_t)dk * dv +
                       (int64_t)r0 * dv;
  if (kTcLayout) {
    const __nv_bfloat16* src =
        reinterpret_cast<const __nv_bfloat16*>((c & 1) ? a.U : a.nodes) + src0;
    if (vec) {  // 8 bf16 in, 8 fp32 out
      for (int64_t i = threadIdx.x; i < elems / 8; i += kThreads) {
        const uint4 u = __ldcs(reinterpret_cast<const uint4*>(src) + i);
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
        float f[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
          f[2 * e] = g * x.x;
          f[2 * e + 1] = g * x.y;
        }
        reinterpret_cast<float4*>(S)[2 * i] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4*>(S)[2 * i + 1] = make_float4(f[4], f[5], f[6], f[7]);
      }
    } else {
      for (int64_t i = threadIdx.x; i < elems; i += kThreads) S[i] = g * __bfloat162float(src[i]);
    }
  } else {
    const float* src = reinterpret_cast<const float*>(a.nodes) + src0;
    if (vec) {
      for (int64_t i = threadIdx.x; i < elems / 4; i += kThreads) {
        const float4 x = __ldcs(reinterpret_cast<const float4*>(src) + i);
        reinterpret_cast<float4*>(S)[i] = make_float4(g * x.x, g * x.y, g * x.z, g * x.w);
      }
    } else {
      for (int64_t i = threadIdx.x; i < elems; i += kThreads) S[i] = g * src[i];
    }
  }
}

}  // namespace

cudaError_t launch_prefill_state(const FwdArgs& a, bool tc_layout, int in_dtype, float* state,
                                 cudaStream_t s) {
  if (a.C > kMaxTile) return cudaErrorInvalidValue;
  if (a.dk > kMaxDim || a.dv > kMaxDim) return cudaErrorInvalidValue;
  const int nb_max = a.C / 2 > 1 ? a.C / 2 : 1;  // largest bucket inside a tile
  const size_t smem =
      sizeof(float) * (32 + 2 * kMaxTile + (size_t)nb_max * (kSliceRows + kMaxDim));
  const dim3 grid((unsigned)a.L, (unsigned)(a.B * a.H),
                  (unsigned)((a.dk + kSliceRows - 1) / kSliceRows));
  // 16-byte loads of bf16 k and v rows: dense rows of a multiple of 8 values, aligned bases
  const bool vec_in = in_dtype == LL_BF16 && a.dk % 8 == 0 && a.dv % 8 == 0 &&
                      (reinterpret_cast<uintptr_t>(a.k) & 15u) == 0 &&
                      (reinterpret_cast<uintptr_t>(a.v) & 15u) == 0 && a.sk[2] == a.dk &&
                      a.sv[2] == a.dv;
  cudaError_t e = cudaSuccess;
  if (in_dtype == LL_BF16) {
    if (tc_layout) {
      if ((e = cudaFuncSetAttribute(prefill_state_kernel<__nv_bfloat16, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) ==
          cudaSuccess)
        prefill_state_kernel<__nv_bfloat16, true><<<grid, kThreads, smem, s>>>(a, state, vec_in);
    } else if ((e = cudaFuncSetAttribute(prefill_state_kernel<__nv_bfloat16, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem)) == cudaSuccess) {
      prefill_state_kernel<__nv_bfloat16, false><<<grid, kThreads, smem, s>>>(a, state, vec_in);
    }
  } else if ((e = cudaFuncSetAttribute(prefill_state_kernel<float, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) ==
             cudaSuccess) {
    prefill_state_kernel<float, false><<<grid, kThreads, smem, s>>>(a, state, vec_in);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace ll

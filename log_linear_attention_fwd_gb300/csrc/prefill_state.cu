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
// One CTA per (level, b, h); a level is written whole.
#include "ll_internal.cuh"

namespace ll {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxTile = 128;   // largest tile of either forward path

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

// tc_layout: block states are bf16 [d_v][d_k] (tensor-core path; odd slots are U_{c-1});
// otherwise fp32 [d_k][d_v] for every slot.
template <typename InT, bool kTcLayout>
__global__ void __launch_bounds__(kThreads) prefill_state_kernel(FwdArgs a, float* state) {
  extern __shared__ float sm[];
  const int lvl = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int b = (int)(bh / a.H), h = (int)(bh - (int64_t)b * a.H);
  const int dk = a.dk, dv = a.dv, tile = a.C, lc = a.lc;
  const int64_t elems = (int64_t)dk * dv;
  float* S = state + (bh * a.L + lvl) * elems;
  const int t = a.T - 1, j = t >> lc, t0 = j << lc;

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
    for (int64_t i = threadIdx.x; i < elems; i += kThreads) S[i] = 0.f;
    return;
  }

  // cs[i] = log decay over tile j from its start to position t0 + i (inclusive)
  float* red = sm;                  // [32]
  float* cs = sm + 32;              // [kMaxTile]
  float* w = cs + kMaxTile;         // [kMaxTile] weights of the bucket's positions
  float* ks = w + kMaxTile;         // [bucket][dk]
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
    // a range of positions inside tile j: sum_s exp(cs_t - cs_s) k_s v_s^T
    const int nb = hi - lo;
    float* vs = ks + nb * dk;
    for (int i = threadIdx.x; i < nb; i += kThreads) w[i] = __expf(cs_t - cs[lo - t0 + i]);
    for (int i = threadIdx.x; i < nb * dk; i += kThreads) {
      const int r = i / dk, d = i - r * dk;
      ks[i] = ld<InT>(a.k, (((int64_t)b * a.T + lo + r) * a.H + h) * dk + d);
    }
    for (int i = threadIdx.x; i < nb * dv; i += kThreads) {
      const int r = i / dv, e = i - r * dv;
      vs[i] = ld<InT>(a.v, (((int64_t)b * a.T + lo + r) * a.H + h) * dv + e);
    }
    __syncthreads();
    for (int64_t i = threadIdx.x; i < elems; i += kThreads) {
      const int d = (int)(i / dv), e = (int)(i - (int64_t)d * dv);
      float acc = 0.f;
      for (int r = 0; r < nb; ++r) acc = fmaf(w[r] * ks[r * dk + d], vs[r * dv + e], acc);
      S[i] = acc;
    }
    return;
  }

  // a block of tiles [c - 2^(m-1), c): the block state of slot c, decayed to t
  const int m = lvl - lc;
  const int c = hi >> lc;
  float D = 0.f;  // sum of the tile log decays over [c, j)
  for (int i = c + (int)threadIdx.x; i < j; i += kThreads) D += a.lg[bh * a.N + i];
  D = block_sum(D, red);
  const float g = __expf(D + cs_t);
  (void)m;
  if (kTcLayout) {
    const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(
        (c & 1) ? a.U : a.nodes) + (bh * a.N + ((c & 1) ? c - 1 : c)) * elems;
    // [d_v][d_k] -> [d_k][d_v] through 32 x 32 shared tiles
    float* tt = ks;  // [32][33]
    for (int e0 = 0; e0 < dv; e0 += 32)
      for (int d0 = 0; d0 < dk; d0 += 32) {
        for (int i = threadIdx.x; i < 32 * 32; i += kThreads) {
          const int er = i >> 5, dc = i & 31;
          if (e0 + er < dv && d0 + dc < dk)
            tt[er * 33 + dc] = __bfloat162float(src[(int64_t)(e0 + er) * dk + d0 + dc]);
        }
        __syncthreads();
        for (int i = threadIdx.x; i < 32 * 32; i += kThreads) {
          const int dr = i >> 5, ec = i & 31;
          if (d0 + dr < dk && e0 + ec < dv)
            S[(int64_t)(d0 + dr) * dv + e0 + ec] = g * tt[ec * 33 + dr];
        }
        __syncthreads();
      }
  } else {
    const float* src = reinterpret_cast<const float*>(a.nodes) + (bh * a.N + c) * elems;
    for (int64_t i = threadIdx.x; i < elems; i += kThreads) S[i] = g * src[i];
  }
}

}  // namespace

cudaError_t launch_prefill_state(const FwdArgs& a, bool tc_layout, int in_dtype, float* state,
                                 cudaStream_t s) {
  if (a.C > kMaxTile) return cudaErrorInvalidValue;
  const int nb_max = a.C / 2 > 1 ? a.C / 2 : 1;  // largest bucket inside a tile
  const size_t smem =
      sizeof(float) * (32 + 2 * kMaxTile + (size_t)nb_max * (a.dk + a.dv) +
                       (tc_layout ? 32 * 33 : 0));
  const dim3 grid((unsigned)a.L, (unsigned)(a.B * a.H));
  cudaError_t e = cudaSuccess;
  if (in_dtype == LL_BF16) {
    if (tc_layout) {
      if ((e = cudaFuncSetAttribute(prefill_state_kernel<__nv_bfloat16, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) ==
          cudaSuccess)
        prefill_state_kernel<__nv_bfloat16, true><<<grid, kThreads, smem, s>>>(a, state);
    } else if ((e = cudaFuncSetAttribute(prefill_state_kernel<__nv_bfloat16, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem)) == cudaSuccess) {
      prefill_state_kernel<__nv_bfloat16, false><<<grid, kThreads, smem, s>>>(a, state);
    }
  } else if ((e = cudaFuncSetAttribute(prefill_state_kernel<float, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) ==
             cudaSuccess) {
    prefill_state_kernel<float, false><<<grid, kThreads, smem, s>>>(a, state);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace ll

// Level scan over the Fenwick block pairing of chunks (page "论文阅读：Log-Linear
// Attention", section 两阶段计算, the worked four-chunk example; page "算力终结者来了！…",
// section 高效训练算法).
//
// Input: per-chunk states U_i (decayed to the chunk's end) and per-chunk log decays lg_i.
// States are read and written in one storage type (fp32 on the CUDA-core path, bf16 on
// the tensor-core path); the block totals are always accumulated in fp32.
// At chunk level m the chunks form aligned blocks of 2^(m-1); each odd block reads the
// total of its even sibling,
//     Tot(m, p) = sum_{i in block p} exp(sum_{i' in block p, i' > i} lg_i') U_i,
// built bottom-up with Tot(m+1, q) = exp(LG(m, 2q+1)) Tot(m, 2q) + Tot(m, 2q+1).
// Every thread owns 4 (or, if d_k*d_v is not a multiple of 4, 1) consecutive state elements of one (b, h) and walks the chunks in
// order with a binary counter (one pending even block per level), so each block total is
// formed once, in fp32, and every even block is stored under the index c of its first
// reader chunk, c = (p+1) 2^(m-1).  The state layout inside a chunk is opaque here.
#include "ll_internal.cuh"

namespace ll {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxLevels = 40;  // chunk levels of the counter (N < 2^39)
constexpr int kPrefetch = 4;

template <int VW>
struct Vec {
  float x[VW];
};

template <int VW>
__device__ __forceinline__ Vec<VW> load_v(const float* p) {
  Vec<VW> r;
  if constexpr (VW == 4) {
    const float4 t = __ldcs(reinterpret_cast<const float4*>(p));
    r.x[0] = t.x; r.x[1] = t.y; r.x[2] = t.z; r.x[3] = t.w;
  } else {
#pragma unroll
    for (int k = 0; k < VW; ++k) r.x[k] = __ldcs(p + k);
  }
  return r;
}

template <int VW>
__device__ __forceinline__ Vec<VW> load_v(const __nv_bfloat16* p) {
  Vec<VW> r;
  if constexpr (VW == 4) {
    const uint2 t = __ldcs(reinterpret_cast<const uint2*>(p));
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&t.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&t.y));
    r.x[0] = lo.x; r.x[1] = lo.y; r.x[2] = hi.x; r.x[3] = hi.y;
  } else {
#pragma unroll
    for (int k = 0; k < VW; ++k) r.x[k] = __bfloat162float(p[k]);
  }
  return r;
}

template <int VW>
__device__ __forceinline__ void store_v(float* p, const Vec<VW>& v) {
  if constexpr (VW == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(v.x[0], v.x[1], v.x[2], v.x[3]);
  } else {
#pragma unroll
    for (int k = 0; k < VW; ++k) p[k] = v.x[k];
  }
}

template <int VW>
__device__ __forceinline__ void store_v(__nv_bfloat16* p, const Vec<VW>& v) {
  if constexpr (VW == 4) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x[0], v.x[1]);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.x[2], v.x[3]);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p) = u;
  } else {
#pragma unroll
    for (int k = 0; k < VW; ++k) p[k] = __float2bfloat16_rn(v.x[k]);
  }
}

template <typename StateT, int VW>
__global__ void __launch_bounds__(kThreads) level_scan_kernel(FwdArgs a) {
  using NodeT = StateT;
  const int64_t elems = (int64_t)a.dk * a.dv;
  const int64_t e = VW * ((int64_t)blockIdx.x * kThreads + threadIdx.x);
  if (e >= elems) return;
  const int64_t bh = (int64_t)blockIdx.z * a.H + blockIdx.y;
  const StateT* U = reinterpret_cast<const StateT*>(a.U) + bh * a.N * elems + e;
  NodeT* nodes = reinterpret_cast<NodeT*>(a.nodes) + bh * a.N * elems + e;
  const float* lg = a.lg + bh * a.N;
  Vec<VW> stk[kMaxLevels];
  float stk_lg[kMaxLevels];
  Vec<VW> pre[kPrefetch];
#pragma unroll
  for (int u = 0; u < kPrefetch; ++u)
    if (u < a.N) pre[u] = load_v<VW>(U + (int64_t)u * elems);
  for (int64_t i0 = 0; i0 < a.N; i0 += kPrefetch) {
#pragma unroll
    for (int u = 0; u < kPrefetch; ++u) {
      const int64_t i = i0 + u;
      if (i >= a.N) break;
      Vec<VW> cur = pre[u];
      if (i + kPrefetch < a.N) pre[u] = load_v<VW>(U + (i + kPrefetch) * elems);
      float cur_lg = lg[i];
      int64_t p = i;
      int m = 1;
      while (p & 1) {  // odd block: merge with the pending even sibling one level up
        const float g = expf(cur_lg);
#pragma unroll
        for (int k = 0; k < VW; ++k) cur.x[k] = fmaf(g, stk[m - 1].x[k], cur.x[k]);
        cur_lg += stk_lg[m - 1];
        p >>= 1;
        ++m;
      }
      const int64_t c = (p + 1) << (m - 1);
      if (c < a.N) store_v<VW>(nodes + c * elems, cur);
      stk[m - 1] = cur;
      stk_lg[m - 1] = cur_lg;
    }
  }
}

}  // namespace

cudaError_t launch_level_scan(const FwdArgs& a, bool bf16_states, cudaStream_t s) {
  const int64_t elems = (int64_t)a.dk * a.dv;
  if (elems % 4 == 0) {
    const dim3 grid((unsigned)((elems / 4 + kThreads - 1) / kThreads), a.H, a.B);
    if (bf16_states)
      level_scan_kernel<__nv_bfloat16, 4><<<grid, kThreads, 0, s>>>(a);
    else
      level_scan_kernel<float, 4><<<grid, kThreads, 0, s>>>(a);
  } else {
    const dim3 grid((unsigned)((elems + kThreads - 1) / kThreads), a.H, a.B);
    if (bf16_states)
      level_scan_kernel<__nv_bfloat16, 1><<<grid, kThreads, 0, s>>>(a);
    else
      level_scan_kernel<float, 1><<<grid, kThreads, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace ll

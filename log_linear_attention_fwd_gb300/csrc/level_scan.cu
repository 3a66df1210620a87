// Level scan over the Fenwick block pairing of chunks (page "论文阅读：Log-Linear
// Attention", section 两阶段计算, the worked four-chunk example; page "算力终结者来了！…",
// section 高效训练算法).
//
// Input: per-chunk fp32 states U_i (decayed to the chunk's end) and per-chunk log decays
// lg_i.  (The tensor-core path forms its block states inside its chunk-state kernel.)
// At chunk level m the chunks form aligned blocks of 2^(m-1); each odd block reads the
// total of its even sibling,
//     Tot(m, p) = sum_{i in block p} exp(sum_{i' in block p, i' > i} lg_i') U_i,
// built bottom-up with Tot(m+1, q) = exp(LG(m, 2q+1)) Tot(m, 2q) + Tot(m, 2q+1).
// A thread owns 4 consecutive state elements of one (b, h) (1 if d_k*d_v is not a
// multiple of 4) and walks chunks in order with a binary counter (one
// pending even block per level), so each block total is formed once, in fp32, and every
// even block is stored under the index c of its first reader chunk, c = (p+1) 2^(m-1).
// Loads run kPrefetch chunks ahead.  The state layout inside a chunk is opaque here.
#include "ll_internal.cuh"

namespace ll {
namespace {

constexpr int kSegs = 16;                 // segments per (b, h), one thread each
constexpr int kGroups = 8;                // element groups per CTA
constexpr int kThreads = kSegs * kGroups;
constexpr int kMaxSegLevels = 32;         // levels inside a segment (seg_len < 2^31)
constexpr int kPrefetch = 8;

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
__device__ __forceinline__ void store_v(float* p, const Vec<VW>& v) {
  if constexpr (VW == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(v.x[0], v.x[1], v.x[2], v.x[3]);
  } else {
#pragma unroll
    for (int k = 0; k < VW; ++k) p[k] = v.x[k];
  }
}

// One CTA covers kGroups element groups (VW elements each) of one (b, h) with kSegs
// threads per group: thread (s, g) first walks segment s, an aligned run of seg_len
// chunks, and stores every block inside it; the complete segments' totals then meet in
// shared memory, where one thread per group walks them to form the blocks of a segment
// or longer.  The sequential depth is seg_len + N/seg_len instead of N.
template <int VW>
__global__ void __launch_bounds__(kThreads) level_scan_kernel(FwdArgs a, int seg_lc) {
  __shared__ Vec<VW> seg_tot[kSegs][kGroups];
  __shared__ float seg_lg[kSegs];
  const int g = threadIdx.x % kGroups, sg = threadIdx.x / kGroups;
  const int64_t elems = (int64_t)a.dk * a.dv;
  const int64_t e = VW * ((int64_t)blockIdx.x * kGroups + g);
  const bool live = e < elems;
  const int64_t bh = (int64_t)blockIdx.z * a.H + blockIdx.y;
  const float* U = reinterpret_cast<const float*>(a.U) + bh * a.N * elems + e;
  float* nodes = reinterpret_cast<float*>(a.nodes) + bh * a.N * elems + e;
  const float* lg = a.lg + bh * a.N;
  const int64_t seg_len = int64_t(1) << seg_lc;
  const int64_t i_lo = sg * seg_len;
  const int64_t i_hi = i_lo + seg_len < (int64_t)a.N ? i_lo + seg_len : (int64_t)a.N;

  // phase 1: blocks of fewer than seg_len chunks, inside segment sg
  if (live && i_lo < a.N) {
    Vec<VW> stk[kMaxSegLevels];
    float stk_lg[kMaxSegLevels];
    Vec<VW> pre[kPrefetch];
#pragma unroll
    for (int u = 0; u < kPrefetch; ++u)
      if (i_lo + u < i_hi) pre[u] = load_v<VW>(U + (i_lo + u) * elems);
    for (int64_t i0 = i_lo; i0 < i_hi; i0 += kPrefetch) {
#pragma unroll
      for (int u = 0; u < kPrefetch; ++u) {
        const int64_t i = i0 + u;
        if (i >= i_hi) break;
        Vec<VW> cur = pre[u];
        if (i + kPrefetch < i_hi) pre[u] = load_v<VW>(U + (i + kPrefetch) * elems);
        float cur_lg = lg[i];
        int64_t p = i;
        int m = 1;
        while ((p & 1) && m <= seg_lc) {  // odd block: merge with its pending even sibling
          const float gl = expf(cur_lg);
#pragma unroll
          for (int k = 0; k < VW; ++k) cur.x[k] = fmaf(gl, stk[m - 1].x[k], cur.x[k]);
          cur_lg += stk_lg[m - 1];
          p >>= 1;
          ++m;
        }
        if (m <= seg_lc) {  // an even block shorter than a segment
          const int64_t c = (p + 1) << (m - 1);
          if (c < a.N) store_v<VW>(nodes + c * elems, cur);
          stk[m - 1] = cur;
          stk_lg[m - 1] = cur_lg;
        } else {            // the whole segment: hand it to phase 2
          seg_tot[sg][g] = cur;
          if (g == 0) seg_lg[sg] = cur_lg;
        }
      }
    }
  }
  __syncthreads();
  // phase 2: blocks of one segment or more, over the complete segments
  if (live && sg == 0) {
    const int64_t nfull = a.N >> seg_lc;
    Vec<VW> stk[kSegs];
    float stk_lg[kSegs];
    for (int64_t q = 0; q < nfull; ++q) {
      Vec<VW> cur = seg_tot[q][g];
      float cur_lg = seg_lg[q];
      int64_t p = q;
      int m = 1;  // level above the segment level
      while (p & 1) {
        const float gl = expf(cur_lg);
#pragma unroll
        for (int k = 0; k < VW; ++k) cur.x[k] = fmaf(gl, stk[m - 1].x[k], cur.x[k]);
        cur_lg += stk_lg[m - 1];
        p >>= 1;
        ++m;
      }
      const int64_t c = (p + 1) << (seg_lc + m - 1);
      if (c < a.N) store_v<VW>(nodes + c * elems, cur);
      stk[m - 1] = cur;
      stk_lg[m - 1] = cur_lg;
    }
  }
}

}  // namespace

cudaError_t launch_level_scan(const FwdArgs& a, cudaStream_t s) {
  const int64_t elems = (int64_t)a.dk * a.dv;
  int seg_lc = 0;  // segments of 2^seg_lc chunks, at most kSegs of them
  while (((int64_t)kSegs << seg_lc) < a.N) ++seg_lc;
  auto grid = [&](int vw) {
    return dim3((unsigned)((elems / vw + kGroups - 1) / kGroups), a.H, a.B);
  };
  if (elems % 4 == 0)  // 16-byte loads of 4 fp32
    level_scan_kernel<4><<<grid(4), kThreads, 0, s>>>(a, seg_lc);
  else
    level_scan_kernel<1><<<grid(1), kThreads, 0, s>>>(a, seg_lc);
  return cudaGetLastError();
}

}  // namespace ll

// Backward on CUDA cores in fp32 (any d_k, d_v <= 128; fp32 or bf16 inputs and gradients).
//
// The gradients of sum(dO ⊙ O) for O = (Q K^T ⊙ M) V, M[t, s] = exp(cum_t - cum_s)
// lambda[t, l(t, s)] (page "算力终结者来了！…", sections 结构矩阵 and 讨论与局限性: training
// needs the lambda gradients besides the attention ones), taken through the same chunked
// decomposition as the forward (page "论文阅读：Log-Linear Attention", sections 矩阵分解 and
// 两阶段计算) on tiles of 32 tokens:
//
//   dQ_t  = sum_s M[t, s] (dO_t . v_s) k_s
//         = intra-tile pairs + sum over the set bits m-1 of the tile index of
//           lambda[t, 5+m] exp(cs_t + D_m) Tot_m dO_t, Tot_m the forward's block state
//           (d_k x d_v, decayed to its end);
//   dlambda[t, l] = sum over the level-l bucket of exp(...) (dO_t . v_s)(q_t . k_s); on an
//           inter-tile level exp(cs_t + D_m) q_t^T Tot_m dO_t;
//   dK_s  = sum_t M[t, s] (dO_t . v_s) q_t,   dV_s = sum_t M[t, s] (q_t . k_s) dO_t:
//           the same pairs seen from the source.  Source s in tile i meets, at tile level
//           m (bit m-1 of i clear), the queries of the aligned block of 2^(m-1) tiles
//           starting at c' = ((i >> (m-1)) | 1) << (m-1); lambda[t, 5+m] depends on t, so
//           it is folded into that block's mirrored state
//           R_c' = sum_t exp(cum_t - cum_start(c')) lambda[t, 5+m] q_t dO_t^T, and
//           dK_s += exp(cum_start(c') - cum_s) R_c' v_s,  dV_s += (same) R_c'^T k_s (the
//           levels of a tile share the row factor and are summed into one state first);
//   dcum_t = q_t . dQ_t - k_t . dK_t  (the row and column sums of dA ⊙ A ⊙ M), and
//   dlog_a_i = sum over t >= i of dcum_t.
//
// Kernels: the forward's K1/K2 recompute U, the block states and the tile log decays;
// bwd_dq (dQ, dlambda, q.dQ); bwd_rstate (R, accumulated over the block's tiles, two
// tiles per CTA, with float4 atomics into the U buffer, which the level scan no longer
// needs); bwd_dkv (dK,
// dV, k.dK); bwd_reduce_qk (per-head dQ, dK summed over the heads sharing a q/k head,
// cast to the gradient type); bwd_dlog_a (reverse prefix sums over t).
#include <algorithm>

#include "ll_internal.cuh"

namespace ll {
namespace {

constexpr int kThreads = 256;
constexpr int kC = kBwdTile;          // tokens per tile
constexpr int kLc = 5;                // log2(kC)
constexpr int kSub = kThreads / kC;   // threads per tile row (8, lanes of one warp)
constexpr int kPer = 128 / kSub;      // features per thread and operand (d <= 128)
constexpr int kStage = 32;            // rows of a d_k x d_v state staged at a time
static_assert(kC == 1 << kLc, "tile");

template <typename T>
__device__ __forceinline__ float ld(const void* p, int64_t i) {
  return to_f32(reinterpret_cast<const T*>(p)[i]);
}

// Sum over the kSub lanes of one tile row (all 32 lanes of the warp must call it).
__device__ __forceinline__ float row_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  x += __shfl_xor_sync(0xffffffffu, x, 4);
  return x;
}

// Sum of lg[lo, hi) by the 32 lanes of warp 0, written to *dst by lane 0 (the caller
// reads it after a block barrier).
__device__ __forceinline__ void range_sum_warp0(const float* lg, int64_t lo, int64_t hi,
                                                float* dst) {
  if (threadIdx.x < 32) {
    float x = 0.f;
    for (int64_t i = lo + threadIdx.x; i < hi; i += 32) x += lg[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (threadIdx.x == 0) *dst = x;
  }
}

constexpr int kStageEl = kStage * 128 / kThreads;  // staged elements per thread (16)

// Shared-memory views of one tile's rows (row strides padded by one float) and its
// tile-local inclusive prefix sums of log a.
struct TileRows {
  float *q, *k, *v, *g, *cs, *lam;
  int lq, lv;
};

template <typename InT, typename GT>
__device__ void load_tile(const BwdArgs& A, int b, int h, int t0, int n, const TileRows& s) {
  const FwdArgs& a = A.f;
  const int dk = a.dk, dv = a.dv, L = a.L, hq = h / a.hg;
  if (threadIdx.x == 0) {
    float run = 0.f;
    for (int r = 0; r < kC; ++r) {
      if (r < n && a.log_a) run += a.log_a[((int64_t)b * a.T + t0 + r) * a.H + h];
      s.cs[r] = run;
    }
  }
  for (int idx = threadIdx.x; idx < kC * dk; idx += kThreads) {
    const int r = idx / dk, c = idx - r * dk;
    const int64_t row = ((int64_t)b * a.T + t0 + r) * a.Hqk + hq;
    s.q[r * s.lq + c] = r < n ? ld<InT>(a.q, row * dk + c) : 0.f;
    s.k[r * s.lq + c] = r < n ? ld<InT>(a.k, row * dk + c) : 0.f;
  }
  for (int idx = threadIdx.x; idx < kC * dv; idx += kThreads) {
    const int r = idx / dv, c = idx - r * dv;
    const int64_t row = ((int64_t)b * a.T + t0 + r) * a.H + h;
    s.v[r * s.lv + c] = r < n ? ld<InT>(a.v, row * dv + c) : 0.f;
    s.g[r * s.lv + c] = r < n ? ld<GT>(A.dout, row * dv + c) : 0.f;
  }
  for (int idx = threadIdx.x; idx < kC * L; idx += kThreads) {
    const int r = idx / L;
    s.lam[idx] =
        r < n ? a.lam[(((int64_t)b * a.T + t0 + r) * a.H + h) * L + (idx - r * L)] : 0.f;
  }
}

__host__ __device__ inline size_t tile_rows_floats(int dk, int dv, int L) {
  return (size_t)2 * kC * (dk + 1) + (size_t)2 * kC * (dv + 1) + kC + (size_t)kC * L;
}

__device__ TileRows carve_rows(float* sm, int dk, int dv) {
  TileRows s;
  s.lq = dk + 1;
  s.lv = dv + 1;
  s.q = sm;
  s.k = s.q + kC * s.lq;
  s.v = s.k + kC * s.lq;
  s.g = s.v + kC * s.lv;
  s.cs = s.g + kC * s.lv;
  s.lam = s.cs + kC;
  return s;
}

// ---------------------------------------------------------------- dQ, dlambda, q . dQ

template <typename InT, typename GT>
__global__ void __launch_bounds__(kThreads, 2) bwd_dq_kernel(BwdArgs A) {
  extern __shared__ float sm[];
  const FwdArgs& a = A.f;
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int dk = a.dk, dv = a.dv, L = a.L;
  const int t0 = j * kC, n = min(kC, a.T - t0);
  const int64_t bh = (int64_t)b * a.H + h;
  const TileRows s = carve_rows(sm, dk, dv);
  float* Ap = s.lam + kC * L;       // [kC][kC+1] exp(cs_t - cs_s) lambda (dO_t . v_s)
  float* Wm = Ap + kC * (kC + 1);   // [kC][kC+1] exp(cs_t - cs_s) (dO_t . v_s)(q_t . k_s)
  float* St = Wm + kC * (kC + 1);   // [kStage][128] staged block-state columns (swizzled)
  float* dl = St + kStage * 128;    // [kC][L] dlambda of the tile's rows
  float* Gt = s.v;                  // [dv][kC] dO transposed, in V's place (after the pairs)
  float* Xs = s.k;                  // [kC][dk+1] Tot dO_t, in K's place (after intra dQ)
  load_tile<InT, GT>(A, b, h, t0, n, s);
  for (int idx = threadIdx.x; idx < kC * L; idx += kThreads) dl[idx] = 0.f;
  __syncthreads();
  for (int idx = threadIdx.x; idx < kC * kC; idx += kThreads) {
    const int t = idx >> kLc, u = idx & (kC - 1);
    float ap = 0.f, w = 0.f;
    if (u <= t && t < n) {
      float dov = 0.f, qk = 0.f;
      for (int e = 0; e < dv; ++e) dov = fmaf(s.g[t * s.lv + e], s.v[u * s.lv + e], dov);
      for (int d = 0; d < dk; ++d) qk = fmaf(s.q[t * s.lq + d], s.k[u * s.lq + d], qk);
      const float ex = expf(s.cs[t] - s.cs[u]);
      // t0 is a multiple of the tile, so the level depends on the tile-local indices only
      ap = ex * s.lam[t * L + fenwick_level((uint32_t)t, (uint32_t)u)] * dov;
      w = ex * dov * qk;
    }
    Ap[t * (kC + 1) + u] = ap;
    Wm[t * (kC + 1) + u] = w;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < kC * dv; idx += kThreads) {  // V is no longer read
    const int r = idx / dv, e = idx - r * dv;
    Gt[e * kC + r] = s.g[r * s.lv + e];
  }
  // intra-tile dlambda: level 0 is the pair (t, t); level l >= 1 (bit l-1 of t set) the
  // sources [hi - 2^(l-1), hi), hi = t with its low l-1 bits cleared
  if (threadIdx.x < kC * (kLc + 1)) {
    const int t = threadIdx.x / (kLc + 1), l = threadIdx.x - t * (kLc + 1);
    if (t < n && l < L) {
      float x = 0.f;
      if (l == 0) {
        x = Wm[t * (kC + 1) + t];
      } else if ((t >> (l - 1)) & 1) {
        const int hi = (t >> (l - 1)) << (l - 1);
        for (int u = hi - (1 << (l - 1)); u < hi; ++u) x += Wm[t * (kC + 1) + u];
      }
      dl[t * L + l] = x;
    }
  }
  // dQ: this thread's row t, features d = sub + kSub i
  const int t = threadIdx.x / kSub, sub = threadIdx.x % kSub;
  float acc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
  for (int u = 0; u <= t; ++u) {
    const float p = Ap[t * (kC + 1) + u];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int d = sub + kSub * i;
      if (d < dk) acc[i] = fmaf(p, s.k[u * s.lq + d], acc[i]);
    }
  }
  // inter-tile levels: X = dO Tot_m^T ([kC] x [d_k]) for the block state of slot c, as a
  // register-blocked product: warp w owns rows 4w..4w+3, lane g columns 4g..4g+3; per
  // step one float4 of dO^T (broadcast) and one of the staged Tot^T columns (stored with
  // the 16-byte groups XOR-swizzled by the row, so the transposing stores and the float4
  // reads do not collide).  X then goes through shared memory to the row layout above.
  const int64_t elems = (int64_t)dk * dv;
  const float* nodes = reinterpret_cast<const float*>(a.nodes) + bh * a.N * elems;
  const float* lg = a.lg + bh * a.N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ float D_s[2];  // log decay from the block's end to the start of tile j
  __syncthreads();  // dO^T is in place; K is no longer read
  for (int m = 1; (int64_t(1) << (m - 1)) <= j; ++m) {
    int64_t c;
    if (!inter_block(j, m, &c)) continue;
    range_sum_warp0(lg, c, j, &D_s[m & 1]);
    const float* S = nodes + c * elems;
    float x[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int q = 0; q < 4; ++q) x[r][q] = 0.f;
    for (int e0 = 0; e0 < dv; e0 += kStage) {
      __syncthreads();
      for (int idx = threadIdx.x; idx < kStage * 128; idx += kThreads) {
        const int e = idx & (kStage - 1), f = idx >> 5;
        const float val = (f < dk && e0 + e < dv) ? S[(int64_t)f * dv + e0 + e] : 0.f;
        St[e * 128 + ((((f >> 2) ^ e) << 2) | (f & 3))] = val;
      }
      __syncthreads();
      const int ne = min(kStage, dv - e0);
      for (int e = 0; e < ne; ++e) {
        const float4 av = *reinterpret_cast<const float4*>(Gt + (e0 + e) * kC + 4 * warp);
        const float4 bv = *reinterpret_cast<const float4*>(St + e * 128 + ((lane ^ e) << 2));
        const float aa[4] = {av.x, av.y, av.z, av.w};
        const float bb[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int q = 0; q < 4; ++q) x[r][q] = fmaf(aa[r], bb[q], x[r][q]);
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (4 * lane + q < dk) Xs[(4 * warp + r) * s.lq + 4 * lane + q] = x[r][q];
    __syncthreads();
    const int lvl = kLc + m;
    const float D = D_s[m & 1];
    const float wq = t < n ? expf(s.cs[t] + D) : 0.f;
    const float wl = wq * s.lam[t * L + lvl];
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int d = sub + kSub * i;
      if (d < dk) {
        const float part = Xs[t * s.lq + d];
        acc[i] = fmaf(wl, part, acc[i]);
        dot = fmaf(s.q[t * s.lq + d], part, dot);
      }
    }
    dot = row_sum(dot);
    if (sub == 0 && t < n) dl[t * L + lvl] = wq * dot;
  }
  // outputs: per-head dQ, q . dQ, the tile rows' dlambda
  float qd = 0.f;
  const int64_t row = ((int64_t)b * a.T + t0 + t) * a.H + h;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int d = sub + kSub * i;
    if (d < dk) {
      if (t < n) A.dqh[row * dk + d] = acc[i];
      qd = fmaf(s.q[t * s.lq + d], acc[i], qd);
    }
  }
  qd = row_sum(qd);
  if (sub == 0 && t < n && A.dcq) A.dcq[row] = qd;
  __syncthreads();
  for (int idx = threadIdx.x; idx < n * L; idx += kThreads) {
    const int r = idx / L;
    A.dlam[(((int64_t)b * a.T + t0 + r) * a.H + h) * L + (idx - r * L)] = dl[idx];
  }
}

// ---------------------------------------------------------------- mirrored block states

// Tiles j0 = 2p and j1 = 2p + 1 (one CTA) add, for every set bit m-1 of their indices,
// their parts of the mirrored state of the block starting at c' = j with its low m-1
// bits cleared:
//   sum_{t in j} exp(cs_t + D_j) lambda[t, 5+m] q_t dO_t^T,  D_j = log decay over [c', j).
// At every level above the first both tiles lie in the same block, so their parts are
// summed before the atomics; level 1 is tile j1's alone.  Thread (td, te) owns rows
// [8 td, +8) and columns [8 te, +8) of the d_k x d_v state.
template <typename InT, typename GT>
__global__ void __launch_bounds__(kThreads, 2) bwd_rstate_kernel(BwdArgs A) {
  extern __shared__ float sm[];
  const FwdArgs& a = A.f;
  const int j0 = 2 * blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int j1 = j0 + 1;
  if (j1 >= a.N && j0 == 0) return;  // a single tile has no mirrored state
  const int dk = a.dk, dv = a.dv, L = a.L, hq = h / a.hg;
  const int n0 = min(kC, a.T - j0 * kC);
  const int n1 = j1 < a.N ? min(kC, a.T - j1 * kC) : 0;
  const int64_t bh = (int64_t)b * a.H + h;
  constexpr int kR = 2 * kC;   // rows of the pair
  float* Qr = sm;              // [kR][128] q, zero-padded
  float* Qw = Qr + kR * 128;   // [kR][128] weighted q
  float* Gd = Qw + kR * 128;   // [kR][128] dO, zero-padded
  float* cs = Gd + kR * 128;   // [kR] tile-local prefix sums of log a
  float* wt = cs + kR;         // [kR] row weights
  float* Ds = wt + kR;         // [2] D of the two tiles
  if (threadIdx.x == 0 || threadIdx.x == 32) {
    const int tile = threadIdx.x >> 5, n = tile ? n1 : n0;
    const int64_t tok0 = (int64_t)b * a.T + (int64_t)(j0 + tile) * kC;
    float run = 0.f;
    for (int r = 0; r < n; ++r) {
      if (a.log_a) run += a.log_a[(tok0 + r) * a.H + h];
      cs[tile * kC + r] = run;
    }
  }
  for (int idx = threadIdx.x; idx < kR * 128; idx += kThreads) {
    const int r = idx >> 7, c = idx & 127;
    const bool live = r < kC ? r < n0 : r - kC < n1;
    const int64_t tok = (int64_t)b * a.T + (int64_t)j0 * kC + r;
    Qr[idx] = (live && c < dk) ? ld<InT>(a.q, (tok * a.Hqk + hq) * dk + c) : 0.f;
    Gd[idx] = (live && c < dv) ? ld<GT>(A.dout, (tok * a.H + h) * dv + c) : 0.f;
  }
  const int64_t elems = (int64_t)dk * dv;
  float* R = reinterpret_cast<float*>(a.U) + bh * a.N * elems;
  const float* lg = a.lg + bh * a.N;
  const int td = threadIdx.x >> 4, te = threadIdx.x & 15;
  const int jtop = n1 > 0 ? j1 : j0;  // its set bits are the levels of the pair
  for (int m = 1; (int64_t(1) << (m - 1)) <= jtop; ++m) {
    if (!((jtop >> (m - 1)) & 1)) continue;
    const int64_t c0 = ((int64_t)jtop >> (m - 1)) << (m - 1);
    const bool in0 = (j0 >> (m - 1)) & 1, in1 = n1 > 0 && ((j1 >> (m - 1)) & 1);
    __syncthreads();  // cs ready (first level); Qw and Ds no longer read (later levels)
    if (threadIdx.x < 64) {  // warp w: D of tile j0 + w
      const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
      float x = 0.f;
      for (int64_t i = c0 + lane; i < j0 + w; i += 32) x += lg[i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      if (lane == 0) Ds[w] = x;
    }
    __syncthreads();
    if (threadIdx.x < kR) {
      const int r = threadIdx.x, tile = r >= kC, rr = r - tile * kC;
      const bool live = tile ? (in1 && rr < n1) : (in0 && rr < n0);
      const int64_t tok = (int64_t)b * a.T + (int64_t)j0 * kC + r;
      wt[r] = live ? expf(cs[r] + Ds[tile]) * a.lam[(tok * a.H + h) * L + kLc + m] : 0.f;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < kR * 128; idx += kThreads) Qw[idx] = wt[idx >> 7] * Qr[idx];
    __syncthreads();
    const int r0 = in0 ? 0 : kC, r1 = in1 ? kC + n1 : n0;  // rows that contribute
    float acc[8][8];
#pragma unroll
    for (int x = 0; x < 8; ++x)
#pragma unroll
      for (int y = 0; y < 8; ++y) acc[x][y] = 0.f;
    for (int r = r0; r < r1; ++r) {
      const float4* qr = reinterpret_cast<const float4*>(Qw + r * 128 + 8 * td);
      const float4* gr = reinterpret_cast<const float4*>(Gd + r * 128 + 8 * te);
      const float4 q0 = qr[0], q1 = qr[1], g0 = gr[0], g1 = gr[1];
      const float qq[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
      const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
      for (int x = 0; x < 8; ++x)
#pragma unroll
        for (int y = 0; y < 8; ++y) acc[x][y] = fmaf(qq[x], gg[y], acc[x][y]);
    }
    float* Rc = R + c0 * elems;
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      const int d = 8 * td + x;
      if (d >= dk) break;
      float* rr = Rc + (int64_t)d * dv;
      if ((dv & 3) == 0 && 8 * te + 8 <= dv) {  // 16-byte aligned: two vector atomics
        atomicAdd(reinterpret_cast<float4*>(rr + 8 * te),
                  make_float4(acc[x][0], acc[x][1], acc[x][2], acc[x][3]));
        atomicAdd(reinterpret_cast<float4*>(rr + 8 * te + 4),
                  make_float4(acc[x][4], acc[x][5], acc[x][6], acc[x][7]));
      } else {
#pragma unroll
        for (int y = 0; y < 8; ++y)
          if (8 * te + y < dv) atomicAdd(rr + 8 * te + y, acc[x][y]);
      }
    }
  }
}

// ---------------------------------------------------------------- dK, dV, k . dK

template <typename InT, typename GT>
__global__ void __launch_bounds__(kThreads) bwd_dkv_kernel(BwdArgs A) {
  extern __shared__ float sm[];
  const FwdArgs& a = A.f;
  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int dk = a.dk, dv = a.dv, L = a.L;
  const int t0 = i * kC, n = min(kC, a.T - t0);
  const int64_t bh = (int64_t)b * a.H + h;
  const TileRows s = carve_rows(sm, dk, dv);
  float* X1 = s.lam + kC * L;       // [kC][kC+1] M[t, s] (dO_t . v_s)
  float* X2 = X1 + kC * (kC + 1);   // [kC][kC+1] M[t, s] (q_t . k_s)
  float* St = X2 + kC * (kC + 1);   // [kStage][128] staged rows or columns of R_tot
  // after the intra-tile part: k and v transposed in the places of q and dO, and the
  // level products in the places of k and v
  float* Kt = s.q;                  // [dk][kC]
  float* Vt = s.g;                  // [dv][kC]
  float* Xd = s.k;                  // [kC][dk+1]  R_tot v_u
  float* Yd = s.v;                  // [kC][dv+1]  R_tot^T k_u
  load_tile<InT, GT>(A, b, h, t0, n, s);
  __syncthreads();
  for (int idx = threadIdx.x; idx < kC * kC; idx += kThreads) {
    const int t = idx >> kLc, u = idx & (kC - 1);
    float x1 = 0.f, x2 = 0.f;
    if (u <= t && t < n) {
      float dov = 0.f, qk = 0.f;
      for (int e = 0; e < dv; ++e) dov = fmaf(s.g[t * s.lv + e], s.v[u * s.lv + e], dov);
      for (int d = 0; d < dk; ++d) qk = fmaf(s.q[t * s.lq + d], s.k[u * s.lq + d], qk);
      const float mts =
          expf(s.cs[t] - s.cs[u]) * s.lam[t * L + fenwick_level((uint32_t)t, (uint32_t)u)];
      x1 = mts * dov;
      x2 = mts * qk;
    }
    X1[t * (kC + 1) + u] = x1;
    X2[t * (kC + 1) + u] = x2;
  }
  __syncthreads();
  // this thread: source row u, features sub + kSub i of dK (d) and of dV (e)
  const int u = threadIdx.x / kSub, sub = threadIdx.x % kSub;
  float ak[kPer], av[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q) ak[q] = av[q] = 0.f;
  for (int t = u; t < kC; ++t) {
    const float x1 = X1[t * (kC + 1) + u], x2 = X2[t * (kC + 1) + u];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int f = sub + kSub * q;
      if (f < dk) ak[q] = fmaf(x1, s.q[t * s.lq + f], ak[q]);
      if (f < dv) av[q] = fmaf(x2, s.g[t * s.lv + f], av[q]);
    }
  }
  // inter-tile levels: the mirrored states of the blocks of later tiles.  The weight
  // exp(cum_start(c1) - cum_u) of level m is exp(lg_i - cs_u) (a row factor, the same at
  // every level) times exp(E_m) (E_m: log decay of the tiles strictly between i and c1),
  // so the levels merge into R_tot = sum_m exp(E_m) R_{c1(m)} and one pair of products:
  //   dK_u += exp(lg_i - cs_u) R_tot v_u,   dV_u += exp(lg_i - cs_u) R_tot^T k_u.
  __shared__ long long lv_c[64];
  __shared__ float lv_w[64];
  __shared__ int lv_n;
  const int64_t elems = (int64_t)dk * dv;
  const float* R = reinterpret_cast<const float*>(a.U) + bh * a.N * elems;
  const float* lg = a.lg + bh * a.N;
  if (threadIdx.x < 32) {  // warp 0: the level list, E_m summed across the lanes
    const int lane0 = threadIdx.x;
    int nl = 0;
    for (int m = 1; (int64_t(1) << (m - 1)) < a.N; ++m) {
      if ((i >> (m - 1)) & 1) continue;
      const int64_t c1 = (((int64_t)i >> (m - 1)) | 1) << (m - 1);
      if (c1 >= a.N) continue;
      float E = 0.f;
      for (int64_t x = i + 1 + lane0; x < c1; x += 32) E += lg[x];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) E += __shfl_xor_sync(0xffffffffu, E, o);
      if (lane0 == 0) {
        lv_c[nl] = c1;
        lv_w[nl] = expf(E);
      }
      ++nl;
    }
    if (lane0 == 0) lv_n = nl;
  }
  __syncthreads();
  const int nl = lv_n;  // (the barrier above also ends the intra-tile reads of q and dO)
  for (int idx = threadIdx.x; idx < kC * dk; idx += kThreads) {
    const int r = idx / dk, c = idx - r * dk;
    Kt[c * kC + r] = s.k[r * s.lq + c];
  }
  for (int idx = threadIdx.x; idx < kC * dv; idx += kThreads) {
    const int r = idx / dv, c = idx - r * dv;
    Vt[c * kC + r] = s.v[r * s.lv + c];
  }
  if (nl > 0) {
    // register-blocked products: warp w owns source rows 4w..4w+3, lane g the features
    // 4g..4g+3; R_tot is formed while it is staged (levels summed with their weights)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float x[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int q = 0; q < 4; ++q) x[r][q] = 0.f;
    // X = V R_tot^T: columns e0..e0+31 of R_tot, transposed, 16-byte groups swizzled
    for (int e0 = 0; e0 < dv; e0 += kStage) {
      float val[kStageEl];  // summed over the levels before the barrier that frees the stage
#pragma unroll
      for (int it = 0; it < kStageEl; ++it) val[it] = 0.f;
      for (int l = 0; l < nl; ++l) {
        const float wl = lv_w[l];
        const float* Rl = R + lv_c[l] * elems;
#pragma unroll
        for (int it = 0; it < kStageEl; ++it) {
          const int idx = threadIdx.x + it * kThreads;
          const int e = idx & (kStage - 1), f = idx >> 5;
          if (f < dk && e0 + e < dv) val[it] = fmaf(wl, Rl[(int64_t)f * dv + e0 + e], val[it]);
        }
      }
      __syncthreads();
#pragma unroll
      for (int it = 0; it < kStageEl; ++it) {
        const int idx = threadIdx.x + it * kThreads;
        const int e = idx & (kStage - 1), f = idx >> 5;
        St[e * 128 + ((((f >> 2) ^ e) << 2) | (f & 3))] = val[it];
      }
      __syncthreads();
      const int ne = min(kStage, dv - e0);
      for (int e = 0; e < ne; ++e) {
        const float4 av4 = *reinterpret_cast<const float4*>(Vt + (e0 + e) * kC + 4 * warp);
        const float4 bv4 = *reinterpret_cast<const float4*>(St + e * 128 + ((lane ^ e) << 2));
        const float aa[4] = {av4.x, av4.y, av4.z, av4.w};
        const float bb[4] = {bv4.x, bv4.y, bv4.z, bv4.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int q = 0; q < 4; ++q) x[r][q] = fmaf(aa[r], bb[q], x[r][q]);
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)  // (k and v were transposed before the first barrier above)
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (4 * lane + q < dk) Xd[(4 * warp + r) * s.lq + 4 * lane + q] = x[r][q];
    float y[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int q = 0; q < 4; ++q) y[r][q] = 0.f;
    // Y = K R_tot: rows d0..d0+31 of R_tot, row-major
    for (int d0 = 0; d0 < dk; d0 += kStage) {
      float val[kStageEl];
#pragma unroll
      for (int it = 0; it < kStageEl; ++it) val[it] = 0.f;
      for (int l = 0; l < nl; ++l) {
        const float wl = lv_w[l];
        const float* Rl = R + lv_c[l] * elems;
#pragma unroll
        for (int it = 0; it < kStageEl; ++it) {
          const int idx = threadIdx.x + it * kThreads;
          const int f = idx >> 7, e = idx & 127;
          if (d0 + f < dk && e < dv) val[it] = fmaf(wl, Rl[(int64_t)(d0 + f) * dv + e], val[it]);
        }
      }
      __syncthreads();
#pragma unroll
      for (int it = 0; it < kStageEl; ++it) St[threadIdx.x + it * kThreads] = val[it];
      __syncthreads();
      const int nf = min(kStage, dk - d0);
      for (int f = 0; f < nf; ++f) {
        const float4 av4 = *reinterpret_cast<const float4*>(Kt + (d0 + f) * kC + 4 * warp);
        const float4 bv4 = *reinterpret_cast<const float4*>(St + f * 128 + 4 * lane);
        const float aa[4] = {av4.x, av4.y, av4.z, av4.w};
        const float bb[4] = {bv4.x, bv4.y, bv4.z, bv4.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int q = 0; q < 4; ++q) y[r][q] = fmaf(aa[r], bb[q], y[r][q]);
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (4 * lane + q < dv) Yd[(4 * warp + r) * s.lv + 4 * lane + q] = y[r][q];
    __syncthreads();
    const float lg_i = s.cs[kC - 1];  // this tile's log decay (tiles before the last are full)
    const float gs = u < n ? expf(lg_i - s.cs[u]) : 0.f;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int f = sub + kSub * q;
      if (f < dk) ak[q] = fmaf(gs, Xd[u * s.lq + f], ak[q]);
      if (f < dv) av[q] = fmaf(gs, Yd[u * s.lv + f], av[q]);
    }
  } else {
    __syncthreads();  // the transposed k is complete
  }
  float kd = 0.f;
  const int64_t row = ((int64_t)b * a.T + t0 + u) * a.H + h;
  GT* dvo = reinterpret_cast<GT*>(A.dv);
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int f = sub + kSub * q;
    if (f < dk) {
      if (u < n) A.dkh[row * dk + f] = ak[q];
      kd = fmaf(Kt[f * kC + u], ak[q], kd);
    }
    if (f < dv && u < n) dvo[row * dv + f] = from_f32<GT>(av[q]);
  }
  kd = row_sum(kd);
  if (sub == 0 && u < n && A.dck) A.dck[row] = kd;
}

// ---------------------------------------------------------------- group sums, d log a

// dq[b, t, g, :] = sum over the heads of group g of dq_h (same for dk), cast to the gradient
// type.  Block (x: position b*T+t, y: a slice of kThreads*4 of the row's Hqk*d_k values);
// 4 consecutive values per thread when d_k is a multiple of 4.
template <typename GT, bool kVec4>
__global__ void __launch_bounds__(kThreads) bwd_reduce_qk_kernel(BwdArgs A) {
  const FwdArgs& a = A.f;
  const int dk = a.dk, hg = a.hg, rowlen = a.Hqk * dk;
  const int64_t bt = blockIdx.x;
  const int i0 = (blockIdx.y * kThreads + threadIdx.x) * 4;
  if (i0 >= rowlen) return;
  GT* dq = reinterpret_cast<GT*>(A.dq) + bt * rowlen;
  GT* dko = reinterpret_cast<GT*>(A.dk) + bt * rowlen;
  const float* sq = A.dqh + bt * a.H * dk;
  const float* sk = A.dkh + bt * a.H * dk;
  if (kVec4) {  // the 4 values share their head group (d_k % 4 == 0)
    const int g = i0 / dk, d = i0 - g * dk;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
    for (int r = 0; r < hg; ++r) {
      const int off = (g * hg + r) * dk + d;
      const float4 u = *reinterpret_cast<const float4*>(sq + off);
      const float4 v = *reinterpret_cast<const float4*>(sk + off);
      x.x += u.x; x.y += u.y; x.z += u.z; x.w += u.w;
      y.x += v.x; y.y += v.y; y.z += v.z; y.w += v.w;
    }
    dq[i0] = from_f32<GT>(x.x); dq[i0 + 1] = from_f32<GT>(x.y);
    dq[i0 + 2] = from_f32<GT>(x.z); dq[i0 + 3] = from_f32<GT>(x.w);
    dko[i0] = from_f32<GT>(y.x); dko[i0 + 1] = from_f32<GT>(y.y);
    dko[i0 + 2] = from_f32<GT>(y.z); dko[i0 + 3] = from_f32<GT>(y.w);
  } else {
    for (int i = i0; i < i0 + 4 && i < rowlen; ++i) {
      const int g = i / dk, d = i - g * dk;
      float x = 0.f, y = 0.f;
      for (int r = 0; r < hg; ++r) {
        x += sq[(g * hg + r) * dk + d];
        y += sk[(g * hg + r) * dk + d];
      }
      dq[i] = from_f32<GT>(x);
      dko[i] = from_f32<GT>(y);
    }
  }
}

// The same sum when a position's Hqk * d_k values are few (Hqk * d_k / 4 columns of 4
// dividing the block): the block's threads split the hg heads of each group into slices,
// each slice summing its heads for 4 values (several loads in flight per thread), and the
// slices are added in shared memory.  Block x: position b*T+t.
template <typename GT>
__global__ void __launch_bounds__(kThreads) bwd_reduce_qk_sliced_kernel(BwdArgs A, int ncol4) {
  const FwdArgs& a = A.f;
  const int dk = a.dk, hg = a.hg, rowlen = a.Hqk * dk;
  const int nsl = kThreads / ncol4;
  const int col = threadIdx.x % ncol4, sl = threadIdx.x / ncol4;
  const int64_t bt = blockIdx.x;
  const int i0 = col * 4;
  const int g = i0 / dk, d = i0 - g * dk;
  const float* sq = A.dqh + (bt * a.H + (int64_t)g * hg) * dk + d;
  const float* sk = A.dkh + (bt * a.H + (int64_t)g * hg) * dk + d;
  float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
#pragma unroll 4
  for (int r = sl; r < hg; r += nsl) {
    const float4 u = *reinterpret_cast<const float4*>(sq + (int64_t)r * dk);
    const float4 v = *reinterpret_cast<const float4*>(sk + (int64_t)r * dk);
    x.x += u.x; x.y += u.y; x.z += u.z; x.w += u.w;
    y.x += v.x; y.y += v.y; y.z += v.z; y.w += v.w;
  }
  __shared__ float4 red[2][kThreads];
  red[0][threadIdx.x] = x;
  red[1][threadIdx.x] = y;
  __syncthreads();
  if (sl != 0) return;
  for (int o = 1; o < nsl; ++o) {
    const float4 u = red[0][o * ncol4 + col], v = red[1][o * ncol4 + col];
    x.x += u.x; x.y += u.y; x.z += u.z; x.w += u.w;
    y.x += v.x; y.y += v.y; y.z += v.z; y.w += v.w;
  }
  GT* dq = reinterpret_cast<GT*>(A.dq) + bt * rowlen + i0;
  GT* dko = reinterpret_cast<GT*>(A.dk) + bt * rowlen + i0;
  dq[0] = from_f32<GT>(x.x); dq[1] = from_f32<GT>(x.y);
  dq[2] = from_f32<GT>(x.z); dq[3] = from_f32<GT>(x.w);
  dko[0] = from_f32<GT>(y.x); dko[1] = from_f32<GT>(y.y);
  dko[2] = from_f32<GT>(y.z); dko[3] = from_f32<GT>(y.w);
}

// dlog_a_i = sum over t >= i of (q_t . dQ_t - k_t . dK_t), in two passes over chunks of
// kScanChunk positions of each (b, h): the chunks' sums, then each chunk's suffix scan
// plus the sum of the chunks after it.
constexpr int kScanChunk = 1024;
constexpr int kScanPer = kScanChunk / kThreads;  // positions per thread (4)

__device__ __forceinline__ float block_sum_all(float x, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < kThreads / 32; ++w) t += red[w];
  return t;
}

__global__ void __launch_bounds__(kThreads) bwd_dlog_a_sums_kernel(BwdArgs A, float* sums, int nch) {
  __shared__ float red[kThreads / 32];
  const FwdArgs& a = A.f;
  const int64_t bh = blockIdx.y;
  const int64_t b = bh / a.H, h = bh - b * a.H;
  const int c = blockIdx.x;
  float x = 0.f;
#pragma unroll
  for (int k = 0; k < kScanPer; ++k) {
    const int i = c * kScanChunk + k * kThreads + threadIdx.x;
    if (i < a.T) {
      const int64_t at = (b * a.T + i) * a.H + h;
      x += A.dcq[at] - A.dck[at];
    }
  }
  x = block_sum_all(x, red);
  if (threadIdx.x == 0) sums[bh * nch + c] = x;
}

__global__ void __launch_bounds__(kThreads) bwd_dlog_a_scan_kernel(BwdArgs A, const float* sums,
                                                                   int nch) {
  __shared__ float red[kThreads / 32];
  __shared__ float after_s;
  const FwdArgs& a = A.f;
  const int64_t bh = blockIdx.y;
  const int64_t b = bh / a.H, h = bh - b * a.H;
  const int c = blockIdx.x;
  if (threadIdx.x < 32) {  // the sum of the chunks after c
    float x = 0.f;
    for (int k = c + 1 + (int)threadIdx.x; k < nch; k += 32) x += sums[bh * nch + k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (threadIdx.x == 0) after_s = x;
  }
  // thread tid owns positions i = base + tid*kScanPer + k, base the chunk's first position;
  // the suffix sum inside the chunk = (own suffix) + (sum of the later threads' values)
  const int base = c * kScanChunk + threadIdx.x * kScanPer;
  float v[kScanPer];
  float own = 0.f;
#pragma unroll
  for (int k = 0; k < kScanPer; ++k) {
    const int i = base + k;
    float x = 0.f;
    if (i < a.T) {
      const int64_t at = (b * a.T + i) * a.H + h;
      x = A.dcq[at] - A.dck[at];
    }
    v[k] = x;
    own += x;
  }
  // exclusive suffix over threads: inclusive prefix over the reversed thread order
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float incl = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += y;
  }
  if (lane == 0) red[warp] = incl;  // the warp's total
  __syncthreads();
  float later_warps = 0.f;
  for (int w = warp + 1; w < kThreads / 32; ++w) later_warps += red[w];
  float run = (incl - own) + later_warps + after_s;  // everything after this thread's values
#pragma unroll
  for (int k = kScanPer - 1; k >= 0; --k) {
    run += v[k];
    const int i = base + k;
    if (i < a.T) A.dlog_a[(b * a.T + i) * a.H + h] = run;
  }
}

template <typename InT, typename GT>
cudaError_t launch_typed(const BwdArgs& A, cudaStream_t s) {
  const FwdArgs& a = A.f;
  const dim3 grid(a.N, a.H, a.B);
  const size_t rows = tile_rows_floats(a.dk, a.dv, a.L);
  const size_t sm_dq =
      sizeof(float) * (rows + 2 * kC * (kC + 1) + (size_t)kStage * 128 + (size_t)kC * a.L);
  const size_t sm_dkv = sizeof(float) * (rows + 2 * kC * (kC + 1) + (size_t)kStage * 128);
  const size_t sm_r = sizeof(float) * (3 * 2 * kC * 128 + 2 * 2 * kC + 2);
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(bwd_dq_kernel<InT, GT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sm_dq)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(bwd_dkv_kernel<InT, GT>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_dkv)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(bwd_rstate_kernel<InT, GT>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_r)) !=
          cudaSuccess)
    return e;
  bwd_dq_kernel<InT, GT><<<grid, kThreads, sm_dq, s>>>(A);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.N > 1) {
    const size_t rbytes = sizeof(float) * (size_t)a.B * a.H * a.N * a.dk * a.dv;
    if ((e = cudaMemsetAsync(a.U, 0, rbytes, s)) != cudaSuccess) return e;
    bwd_rstate_kernel<InT, GT><<<dim3((a.N + 1) / 2, a.H, a.B), kThreads, sm_r, s>>>(A);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  bwd_dkv_kernel<InT, GT><<<grid, kThreads, sm_dkv, s>>>(A);
  return cudaGetLastError();
}

}  // namespace

BwdWorkspace bwd_workspace_layout(int64_t B, int64_t T, int64_t H, int64_t Hqk, int64_t N,
                                  int64_t dk, int64_t dv, int64_t n_tc) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  BwdWorkspace w;
  const size_t rows = (size_t)(B * T * H);
  // CUDA cores: chunk states, fp32 block states of every slot, tile log decays, and
  // per-head fp32 dq and dk.  Tensor cores: the mirrored states on the 128-token tiles in
  // U's place (the block states come from the forward's workspace below), and fp32 dq and
  // dk per q/k head only when heads share them.
  const size_t states = (size_t)(B * H * (n_tc > 0 ? n_tc : N)) * (size_t)(dk * dv) * sizeof(float);
  const size_t nodes = n_tc > 0 ? 0 : states;
  const size_t lg = n_tc > 0 ? 0 : (size_t)(B * H * N) * sizeof(float);
  const size_t qk_rows = n_tc > 0 ? (Hqk < H ? (size_t)(B * T * Hqk) : 0) : rows;
  w.off_U = 0;
  w.off_nodes = up(w.off_U + states);
  w.off_lg = up(w.off_nodes + nodes);
  w.off_dqh = up(w.off_lg + lg);
  w.off_dkh = up(w.off_dqh + qk_rows * dk * sizeof(float));
  w.off_dcq = up(w.off_dkh + qk_rows * dk * sizeof(float));
  w.off_dck = up(w.off_dcq + rows * sizeof(float));
  w.off_scan = up(w.off_dck + rows * sizeof(float));
  w.off_fwd = 0;
  w.fwd = FwdWorkspace{};
  w.total = up(w.off_scan + (size_t)(B * H) * (size_t)((T + 1023) / 1024 + 1) * sizeof(float));
  if (n_tc > 0) {  // the states-only forward's workspace (it writes no output)
    w.fwd = fwd_workspace_layout(B, H, n_tc, dk, dv, 2);
    w.off_fwd = w.total;
    w.total = up(w.off_fwd + w.fwd.total);
  }
  return w;
}

size_t bwd_smem_max(int dk, int dv, int L) {
  return sizeof(float) * (tile_rows_floats(dk, dv, L) + 2 * kC * (kC + 1) + (size_t)kStage * 128 +
                          (size_t)kC * L);
}

cudaError_t launch_bwd_finish(const BwdArgs& A0, int grad_dtype, cudaStream_t s, bool with_qk,
                              bool qk_summed) {
  // qk_summed: dqh and dkh already hold each q/k head's sum ([B, T, Hqk, d_k]); the pass
  // below is then a cast (one head per group)
  BwdArgs As = A0;
  if (qk_summed) {
    As.f.H = A0.f.Hqk;
    As.f.hg = 1;
  }
  const BwdArgs& A = with_qk ? As : A0;
  const FwdArgs& a = A.f;
  cudaError_t e = cudaSuccess;
  if (with_qk) {
    const int rowlen = a.Hqk * a.dk;
    const dim3 grid_r((unsigned)((int64_t)a.B * a.T),
                      (unsigned)((rowlen + 4 * kThreads - 1) / (4 * kThreads)));
    const bool vec = a.dk % 4 == 0;
    const int ncol4 = rowlen / 4;
    if (vec && a.hg > 1 && ncol4 <= kThreads / 2 && kThreads % ncol4 == 0) {
      const unsigned grid_p = (unsigned)((int64_t)a.B * a.T);
      if (grad_dtype == LL_F32)
        bwd_reduce_qk_sliced_kernel<float><<<grid_p, kThreads, 0, s>>>(A, ncol4);
      else
        bwd_reduce_qk_sliced_kernel<__nv_bfloat16><<<grid_p, kThreads, 0, s>>>(A, ncol4);
    } else if (grad_dtype == LL_F32) {
      if (vec) bwd_reduce_qk_kernel<float, true><<<grid_r, kThreads, 0, s>>>(A);
      else bwd_reduce_qk_kernel<float, false><<<grid_r, kThreads, 0, s>>>(A);
    } else {
      if (vec) bwd_reduce_qk_kernel<__nv_bfloat16, true><<<grid_r, kThreads, 0, s>>>(A);
      else bwd_reduce_qk_kernel<__nv_bfloat16, false><<<grid_r, kThreads, 0, s>>>(A);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (A0.f.log_a && A0.dlog_a) {  // per value head: the original sizes
    const FwdArgs& f = A0.f;
    const int nch = (f.T + kScanChunk - 1) / kScanChunk;
    const dim3 grid_s((unsigned)nch, (unsigned)((int64_t)f.B * f.H));
    bwd_dlog_a_sums_kernel<<<grid_s, kThreads, 0, s>>>(A0, A0.scan, nch);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bwd_dlog_a_scan_kernel<<<grid_s, kThreads, 0, s>>>(A0, A0.scan, nch);
    e = cudaGetLastError();
  }
  return e;
}

cudaError_t launch_simt_backward(const BwdArgs& A, int in_dtype, int grad_dtype, cudaStream_t s) {
  cudaError_t e = launch_simt_states(A.f, in_dtype, s);
  if (e != cudaSuccess) return e;
  if (in_dtype == LL_F32 && grad_dtype == LL_F32) e = launch_typed<float, float>(A, s);
  else if (in_dtype == LL_F32) e = launch_typed<float, __nv_bfloat16>(A, s);
  else if (grad_dtype == LL_F32) e = launch_typed<__nv_bfloat16, float>(A, s);
  else e = launch_typed<__nv_bfloat16, __nv_bfloat16>(A, s);
  return e == cudaSuccess ? launch_bwd_finish(A, grad_dtype, s, true, false) : e;
}

}  // namespace ll

// Forward of Log-Linear Gated DeltaNet in chunks of 64 tokens (fp32 on CUDA cores).
//
// The log-linear form keeps the model's transition and composes its mask with the Fenwick
// mask (page "算力终结者来了！…", section 对Mamba-2和门控DeltaNet的对数线性推广; page
// "论文阅读：Log-Linear Attention", sections 与已有模型的组合 and 两阶段计算).  The
// transition is the gated delta rule (Yang, Kautz and Hatamizadeh, "Gated Delta Networks",
// 2024), A_t = alpha_t (I - beta_t k_t k_t^T), state S [d_k][d_v], o = S^T q.  Inside a
// chunk its products are taken in the UT-transform form of the delta rule (Yang et al.,
// "Parallelizing Linear Transformers with the Delta Rule over Sequence Length", 2024):
// with g_t the chunk-local cumulative log gate, Gam[t, s] = exp(g_t - g_s) (s <= t),
// gamma_t = exp(g_t),
//   A  = strictly_lower(diag(beta) (K K^T ⊙ Gam)),   T = (I + A)^-1,
//   Aqk = (Q K^T ⊙ Gam) on s <= t,
//   W  = Aqk T diag(beta)                     the chunk's own attention matrix,
//   X  = T diag(beta gamma) K,
//   Qt = diag(gamma) Q - Aqk X                 the queries carried back to the chunk start,
//   P  = gamma_end I - K^T diag(Gam[end, :]) X  the chunk's transition (d_k x d_k),
//   U  = K^T diag(Gam[end, :]) T diag(beta) V  the chunk's own writes at its end.
// Then, exactly as for Mamba-2 but with P in place of a scalar decay:
//   O[t] = (W ⊙ M^H) V [t] + sum over chunk levels m (bit m-1 of j) lambda[t, 6+m] Qt[t] Z^m,
// where Z^m, the block state of chunk level m, is carried through every later chunk by P
// and merged at chunk starts by the lssb rule on chunk indices (Z^{lssb(j)+1} <- U_{j-1} +
// sum_{m <= lssb(j)} Z^m).
//
// gdn_chunk_kernel: one CTA per (b, h, chunk), all chunks in parallel; it writes W ⊙ M^H V
// (fp32), Qt, P and U to the workspace.  gdn_chunk_scan_kernel: one CTA per (b, h, 16
// columns of d_v), sequential over the chunks, holds the Z^m of its columns in shared
// memory, adds the inter-chunk readout and writes the output.
#include "ll_internal.cuh"

namespace ll {
namespace {

constexpr int kC = 64;          // tokens per chunk
constexpr int kLc = 6;          // log2(kC)
constexpr int kD = 128;         // d_k, d_v <= 128 (zero-padded in shared memory)
constexpr int kThreads = 256;
constexpr int kLd = kD + 4;     // row stride of [64][128] fp32 tiles (16-byte rows, fewer conflicts)
constexpr int kLdc = kC + 4;    // row stride of [64][64] fp32 tiles
constexpr int kCols = 16;       // d_v columns per scan CTA

struct ChunkSmem {
  static constexpr int kQ = 0;                          // Q, then Y = T diag(beta) V
  static constexpr int kK = kQ + kC * kLd;
  static constexpr int kV = kK + kC * kLd;
  static constexpr int kX = kV + kC * kLd;              // X = T diag(beta gamma) K
  static constexpr int kAqk = kX + kC * kLd;            // [64][64]
  static constexpr int kT = kAqk + kC * kLdc;           // [64][64]
  static constexpr int kW = kT + kC * kLdc;             // [64][64]: A, then W ⊙ M^H
  static constexpr int kG = kW + kC * kLdc;             // g [64]
  static constexpr int kGam = kG + kC;                  // gamma [64]
  static constexpr int kBeta = kGam + kC;               // beta [64]
  static constexpr int kLam = kBeta + kC;               // [64][8] intra lambdas (levels 0..6)
  static constexpr int kEnd = kLam + kC * 8;            // floats
};

// acc[i][j] += sum_k A(m0 + i, k) B(k, n0 + j) over k in [k0, k1), A(m, k) = A[m lda + k]
// (or A[k lda + m] when AT), B(k, n) = B[k ldb + n] (or B[n ldb + k] when BT).
template <int TM, int TN, bool AT, bool BT>
__device__ __forceinline__ void mma_tile(float (&acc)[TM][TN], const float* A, int lda,
                                         const float* B, int ldb, int k0, int k1, int m0,
                                         int n0) {
  for (int k = k0; k < k1; ++k) {
    float a[TM], bv[TN];
#pragma unroll
    for (int i = 0; i < TM; ++i) a[i] = AT ? A[k * lda + m0 + i] : A[(m0 + i) * lda + k];
#pragma unroll
    for (int j = 0; j < TN; ++j) bv[j] = BT ? B[(n0 + j) * ldb + k] : B[k * ldb + n0 + j];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], bv[j], acc[i][j]);
  }
}

template <int TM, int TN>
__device__ __forceinline__ void zero(float (&acc)[TM][TN]) {
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
}

struct GdnChunkArgs {
  const void* q;      // [B, T, Hqk, dk]
  const void* k;
  const void* v;      // [B, T, H, dv]
  const float* log_a; // [B, T, H] or null
  const float* beta;  // [B, T, H]
  const float* lam;   // [B, T, H, L]
  void* out;          // [B, T, H, dv]
  float* o_intra;     // [B, T, H, dv]      workspace
  float* qt;          // [B*H][N][64][dk]   workspace
  float* P;           // [B*H][N][dk][dk]   workspace
  float* U;           // [B*H][N][dk][dv]   workspace
  int B, T, H, hg, dk, dv, L, N;
};

template <typename InT>
__global__ void __launch_bounds__(kThreads, 1) gdn_chunk_kernel(GdnChunkArgs a) {
  extern __shared__ __align__(16) float sm[];
  float* Qs = sm + ChunkSmem::kQ;
  float* Ks = sm + ChunkSmem::kK;
  float* Vs = sm + ChunkSmem::kV;
  float* Xs = sm + ChunkSmem::kX;
  float* Aqk = sm + ChunkSmem::kAqk;
  float* Ts = sm + ChunkSmem::kT;
  float* Ws = sm + ChunkSmem::kW;
  float* gs = sm + ChunkSmem::kG;
  float* gam = sm + ChunkSmem::kGam;
  float* bet = sm + ChunkSmem::kBeta;
  float* lms = sm + ChunkSmem::kLam;

  const int tid = threadIdx.x;
  const int j = blockIdx.x % a.N;
  const int64_t bh = blockIdx.x / a.N;
  const int b = (int)(bh / a.H), h = (int)(bh - (int64_t)b * a.H), hq = h / a.hg;
  const int Hqk = a.H / a.hg;
  const int t0 = j * kC, n = min(kC, a.T - t0);
  const int dk = a.dk, dv = a.dv;

  // ---- the chunk's q, k, v (fp32, zero past n rows and past dk / dv columns), gates
  for (int i = tid; i < kC * kD; i += kThreads) {
    const int t = i / kD, d = i - t * kD;
    const bool live = t < n;
    const int64_t tq = ((int64_t)b * a.T + t0 + t) * Hqk + hq;
    const int64_t tv = ((int64_t)b * a.T + t0 + t) * a.H + h;
    Qs[t * kLd + d] = live && d < dk ? to_f32(static_cast<const InT*>(a.q)[tq * dk + d]) : 0.f;
    Ks[t * kLd + d] = live && d < dk ? to_f32(static_cast<const InT*>(a.k)[tq * dk + d]) : 0.f;
    Vs[t * kLd + d] = live && d < dv ? to_f32(static_cast<const InT*>(a.v)[tv * dv + d]) : 0.f;
  }
  if (tid < kC) {
    const int64_t tv = ((int64_t)b * a.T + t0 + tid) * a.H + h;
    const bool live = tid < n;
    float la = live && a.log_a ? a.log_a[tv] : 0.f;
    // inclusive prefix sum over the chunk (two warps)
    const int lane = tid & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, la, o);
      if (lane >= o) la += y;
    }
    gs[tid] = la;
    bet[tid] = live ? a.beta[tv] : 0.f;
#pragma unroll
    for (int l = 0; l <= kLc; ++l) lms[tid * 8 + l] = live && l < a.L ? a.lam[tv * a.L + l] : 0.f;
  }
  __syncthreads();
  if (tid >= 32 && tid < kC) gs[tid] += gs[31];
  __syncthreads();
  if (tid < kC) gam[tid] = __expf(gs[tid]);

  const int tm = tid >> 4, tn = tid & 15;  // 16 x 16 thread grid
  // ---- Aqk = (Q K^T ⊙ Gam) on s <= t, and A = strictly_lower(diag(beta)(K K^T ⊙ Gam)) into W
  {
    float aq[4][4], ak[4][4];
    zero(aq);
    zero(ak);
    mma_tile<4, 4, false, true>(aq, Qs, kLd, Ks, kLd, 0, kD, 4 * tm, 4 * tn);
    mma_tile<4, 4, false, true>(ak, Ks, kLd, Ks, kLd, 0, kD, 4 * tm, 4 * tn);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int t = 4 * tm + i, s = 4 * tn + jj;
        const float G = s <= t ? __expf(gs[t] - gs[s]) : 0.f;
        Aqk[t * kLdc + s] = aq[i][jj] * G;
        Ws[t * kLdc + s] = s < t ? bet[t] * ak[i][jj] * G : 0.f;
      }
  }
  __syncthreads();
  // ---- T = (I + A)^-1 (unit lower triangular) by forward substitution, one row at a time:
  // T[i][c] = [i == c] - sum_{k = c}^{i-1} A[i][k] T[k][c]; thread (c, part) sums a quarter
  // of k for column c.
  {
    const int c = tid >> 2, part = tid & 3;
    for (int i = 0; i < kC; ++i) {
      float x = 0.f;
      if (c < i)
        for (int kk = c + part; kk < i; kk += 4) x = fmaf(Ws[i * kLdc + kk], Ts[kk * kLdc + c], x);
      x += __shfl_xor_sync(0xffffffffu, x, 1);
      x += __shfl_xor_sync(0xffffffffu, x, 2);
      if (part == 0) Ts[i * kLdc + c] = c < i ? -x : (c == i ? 1.f : 0.f);
      __syncthreads();
    }
  }
  // ---- W = Aqk T diag(beta), masked by lambda[t, level(t, s)] (s <= t) into W
  {
    float w[4][4];
    zero(w);
    mma_tile<4, 4, false, false>(w, Aqk, kLdc, Ts, kLdc, 0, kC, 4 * tm, 4 * tn);
    __syncthreads();  // every thread has read A (in W) and T... W is rewritten below
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int t = 4 * tm + i, s = 4 * tn + jj;
        const int lvl = s <= t ? fenwick_level((uint32_t)t, (uint32_t)s) : 0;
        Ws[t * kLdc + s] = s <= t ? w[i][jj] * bet[s] * lms[t * 8 + lvl] : 0.f;
      }
  }
  __syncthreads();
  // ---- O_intra = (W ⊙ M^H) V: thread (tm, tn) rows 4 tm.., columns 8 tn..
  {
    float o[4][8];
    zero(o);
    mma_tile<4, 8, false, false>(o, Ws, kLdc, Vs, kLd, 0, kC, 4 * tm, 8 * tn);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 4 * tm + i;
      if (t >= n) continue;
      float* dst = a.o_intra + (((int64_t)b * a.T + t0 + t) * a.H + h) * dv;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
        if (8 * tn + jj < dv) dst[8 * tn + jj] = o[i][jj];
    }
  }
  // ---- X = T diag(beta gamma) K: rows 4 tm.., columns 8 tn..
  {
    float x[4][8];
    zero(x);
    for (int k = 0; k < kC; ++k) {
      const float sc = bet[k] * gam[k];
      float tv[4], kv[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) tv[i] = Ts[(4 * tm + i) * kLdc + k];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) kv[jj] = sc * Ks[k * kLd + 8 * tn + jj];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) x[i][jj] = fmaf(tv[i], kv[jj], x[i][jj]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) Xs[(4 * tm + i) * kLd + 8 * tn + jj] = x[i][jj];
  }
  __syncthreads();
  const int64_t chunk = bh * a.N + j;
  // ---- Qt = diag(gamma) Q - Aqk X  (64 x dk) to the workspace
  {
    float qv[4][8];
    zero(qv);
    mma_tile<4, 8, false, false>(qv, Aqk, kLdc, Xs, kLd, 0, kC, 4 * tm, 8 * tn);
    float* dst = a.qt + chunk * kC * dk;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 4 * tm + i;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int d = 8 * tn + jj;
        if (d < dk) dst[t * dk + d] = gam[t] * Qs[t * kLd + d] - qv[i][jj];
      }
    }
  }
  // ---- P = gamma_end I - K^T diag(Gam[end, :]) X  (dk x dk): thread rows 8 tm.., cols 8 tn..
  {
    const float g_end = gs[n - 1];
    float pv[8][8];
    zero(pv);
    for (int s = 0; s < n; ++s) {
      const float ge = __expf(g_end - gs[s]);
      float kv[8], xv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) kv[i] = ge * Ks[s * kLd + 8 * tm + i];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) xv[jj] = Xs[s * kLd + 8 * tn + jj];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) pv[i][jj] = fmaf(kv[i], xv[jj], pv[i][jj]);
    }
    const float gend = gam[n - 1];
    float* dst = a.P + chunk * (int64_t)dk * dk;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = 8 * tm + i;
      if (r >= dk) continue;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int c = 8 * tn + jj;
        if (c < dk) dst[r * dk + c] = (r == c ? gend : 0.f) - pv[i][jj];
      }
    }
  }
  __syncthreads();  // Q is read for the last time above: Y goes in its place
  // ---- Y = T diag(beta) V  (64 x dv) into Q's buffer
  {
    float y[4][8];
    zero(y);
    for (int k = 0; k < kC; ++k) {
      float tv[4], vv[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) tv[i] = Ts[(4 * tm + i) * kLdc + k];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) vv[jj] = bet[k] * Vs[k * kLd + 8 * tn + jj];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) y[i][jj] = fmaf(tv[i], vv[jj], y[i][jj]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) Qs[(4 * tm + i) * kLd + 8 * tn + jj] = y[i][jj];
  }
  __syncthreads();
  // ---- U = K^T diag(Gam[end, :]) Y  (dk x dv)
  {
    const float g_end = gs[n - 1];
    float u[8][8];
    zero(u);
    for (int s = 0; s < n; ++s) {
      const float ge = __expf(g_end - gs[s]);
      float kv[8], yv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) kv[i] = ge * Ks[s * kLd + 8 * tm + i];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) yv[jj] = Qs[s * kLd + 8 * tn + jj];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) u[i][jj] = fmaf(kv[i], yv[jj], u[i][jj]);
    }
    float* dst = a.U + chunk * (int64_t)dk * dv;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = 8 * tm + i;
      if (r >= dk) continue;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int c = 8 * tn + jj;
        if (c < dv) dst[r * dv + c] = u[i][jj];
      }
    }
  }
}

// ---------------------------------------------------------------- the scan over chunks
//
// Thread layout: 256 threads = 16 columns x 16 row groups of 8 rows (d_k <= 128).  Z^m of
// the CTA's columns, [level][128][16] fp32, in shared memory.
template <typename OutT>
__global__ void __launch_bounds__(kThreads, 1) gdn_chunk_scan_kernel(GdnChunkArgs a, int levels) {
  extern __shared__ __align__(16) float zs[];   // [levels][kD][kCols], then P [kD][kD + 1]
  float* Ps = zs + (size_t)levels * kD * kCols;  // the chunk's transition (rows < dk)
  const int tid = threadIdx.x;
  const int slices = (a.dv + kCols - 1) / kCols;
  const int64_t bh = blockIdx.x / slices;
  const int c0 = (int)(blockIdx.x - bh * slices) * kCols;
  const int b = (int)(bh / a.H), h = (int)(bh - (int64_t)b * a.H);
  const int dk = a.dk, dv = a.dv;
  const int col = tid & (kCols - 1), rg = tid >> 4;  // column, row group (rows 8 rg..)
  for (int i = tid; i < levels * kD * kCols; i += kThreads) zs[i] = 0.f;
  __syncthreads();
  uint32_t live = 0;  // bit m: Z^m holds data
  for (int j = 0; j < a.N; ++j) {
    const int64_t chunk = bh * a.N + j;
    const int t0 = j * kC, n = min(kC, a.T - t0);
    // ---- merge at the chunk start: Z^{l+1} <- U_{j-1} + sum_{m <= l} Z^m, l = lssb(j)
    if (j > 0) {
      const int l = __ffs(j) - 1;
      const float* Up = a.U + (chunk - 1) * (int64_t)dk * dv;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = 8 * rg + i;
        float x = (r < dk && c0 + col < dv) ? Up[r * dv + c0 + col] : 0.f;
        for (int m = 1; m <= l; ++m) {
          float* z = zs + ((size_t)m * kD + r) * kCols + col;
          x += *z;
          *z = 0.f;
        }
        zs[((size_t)(l + 1) * kD + r) * kCols + col] = x;
      }
      live = (live & ~((2u << l) - 2u)) | (1u << (l + 1));
    }
    // the chunk's transition into shared memory
    const float* Pg = a.P + chunk * (int64_t)dk * dk;
    for (int i = tid; i < dk * dk; i += kThreads) {
      const int r = i / dk, c = i - r * dk;
      Ps[r * (kD + 1) + c] = Pg[i];
    }
    __syncthreads();
    // ---- readout: O[t][col] = O_intra + sum_m lambda[t, 6+m] sum_d Qt[t][d] Z^m[d][col];
    // thread (rg, col) takes tokens rg, rg + 16, ... (4 of them)
    const float* qt = a.qt + chunk * kC * dk;
    for (int t = rg; t < n; t += 16) {
      const int64_t tv = ((int64_t)b * a.T + t0 + t) * a.H + h;
      float o = (c0 + col < dv) ? a.o_intra[tv * dv + c0 + col] : 0.f;
      for (int m = 1; m < levels; ++m) {
        if (!((live >> m) & 1)) continue;
        const float* z = zs + (size_t)m * kD * kCols + col;
        float x = 0.f;
        for (int d = 0; d < dk; ++d) x = fmaf(qt[t * dk + d], z[d * kCols], x);
        o = fmaf(a.lam[tv * a.L + kLc + m], x, o);
      }
      if (c0 + col < dv) static_cast<OutT*>(a.out)[tv * dv + c0 + col] = from_f32<OutT>(o);
    }
    __syncthreads();
    // ---- carry every live level through the chunk: Z^m <- P Z^m
    for (int m = 1; m < levels; ++m) {
      if (!((live >> m) & 1)) continue;
      float* z = zs + (size_t)m * kD * kCols;
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      for (int d = 0; d < dk; ++d) {
        const float zv = z[d * kCols + col];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(Ps[(8 * rg + i) * (kD + 1) + d], zv, acc[i]);
      }
      __syncthreads();  // every thread has read the old Z^m
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (8 * rg + i < dk) z[(8 * rg + i) * kCols + col] = acc[i];
      __syncthreads();
    }
  }
}

}  // namespace

size_t gdn_chunk_workspace_bytes(int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv) {
  const int64_t N = (T + kC - 1) / kC;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  return up(sizeof(float) * (size_t)(B * T * H * dv)) +          // O_intra
         up(sizeof(float) * (size_t)(B * H * N * kC * dk)) +     // Qt
         up(sizeof(float) * (size_t)(B * H * N * dk * dk)) +     // P
         up(sizeof(float) * (size_t)(B * H * N * dk * dv));      // U
}

cudaError_t launch_gdn_chunked(const void* q, const void* k, const void* v, const float* log_a,
                               const float* beta, const float* lam, void* out, int B, int T, int H,
                               int Hqk, int dk, int dv, int L, int in_dtype, int out_dtype,
                               void* workspace, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  GdnChunkArgs a;
  a.q = q; a.k = k; a.v = v; a.log_a = log_a; a.beta = beta; a.lam = lam; a.out = out;
  a.B = B; a.T = T; a.H = H; a.hg = H / Hqk; a.dk = dk; a.dv = dv; a.L = L;
  a.N = (T + kC - 1) / kC;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  char* ws = static_cast<char*>(workspace);
  a.o_intra = reinterpret_cast<float*>(ws);
  ws += up(sizeof(float) * (size_t)B * T * H * dv);
  a.qt = reinterpret_cast<float*>(ws);
  ws += up(sizeof(float) * (size_t)B * H * a.N * kC * dk);
  a.P = reinterpret_cast<float*>(ws);
  ws += up(sizeof(float) * (size_t)B * H * a.N * dk * dk);
  a.U = reinterpret_cast<float*>(ws);
  const size_t smem1 = sizeof(float) * ChunkSmem::kEnd;
  cudaError_t e;
  const unsigned grid1 = (unsigned)((int64_t)B * H * a.N);
  if (in_dtype == LL_BF16) {
    if ((e = cudaFuncSetAttribute(gdn_chunk_kernel<__nv_bfloat16>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1)) !=
        cudaSuccess)
      return e;
    gdn_chunk_kernel<__nv_bfloat16><<<grid1, kThreads, smem1, s>>>(a);
  } else {
    if ((e = cudaFuncSetAttribute(gdn_chunk_kernel<float>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1)) !=
        cudaSuccess)
      return e;
    gdn_chunk_kernel<float><<<grid1, kThreads, smem1, s>>>(a);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  int levels = 1;  // chunk levels 1..bit_length(N-1), plus the unused slot 0
  while ((1 << (levels - 1)) < a.N) ++levels;
  const size_t smem2 = sizeof(float) * ((size_t)levels * kD * kCols + kD * (kD + 1));
  const unsigned grid2 = (unsigned)((int64_t)B * H * ((dv + kCols - 1) / kCols));
  if (out_dtype == LL_BF16) {
    if ((e = cudaFuncSetAttribute(gdn_chunk_scan_kernel<__nv_bfloat16>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2)) !=
        cudaSuccess)
      return e;
    gdn_chunk_scan_kernel<__nv_bfloat16><<<grid2, kThreads, smem2, s>>>(a, levels);
  } else {
    if ((e = cudaFuncSetAttribute(gdn_chunk_scan_kernel<float>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2)) !=
        cudaSuccess)
      return e;
    gdn_chunk_scan_kernel<float><<<grid2, kThreads, smem2, s>>>(a, levels);
  }
  return cudaGetLastError();
}

}  // namespace ll

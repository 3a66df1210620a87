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
constexpr int kLd = kD + 1;     // row stride of [64][128] fp32 tiles (odd: rows on all banks)
constexpr int kLdc = kC + 1;    // row stride of [64][64] fp32 tiles
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

// acc[i][j] += sum_k A(m0 + i, k) B(k, n0 + CS j) over k in [k0, k1), A(m, k) = A[m lda + k]
// (or A[k lda + m] when AT), B(k, n) = B[k ldb + n] (or B[n ldb + k] when BT).  CS = 16
// interleaves the 16 threads of a row of the thread grid over consecutive columns (no bank
// conflicts in B).
template <int TM, int TN, bool AT, bool BT, int CS = 1>
__device__ __forceinline__ void mma_tile(float (&acc)[TM][TN], const float* A, int lda,
                                         const float* B, int ldb, int k0, int k1, int m0,
                                         int n0) {
  for (int k = k0; k < k1; ++k) {
    float a[TM], bv[TN];
#pragma unroll
    for (int i = 0; i < TM; ++i) a[i] = AT ? A[k * lda + m0 + i] : A[(m0 + i) * lda + k];
#pragma unroll
    for (int j = 0; j < TN; ++j) bv[j] = BT ? B[(n0 + CS * j) * ldb + k] : B[k * ldb + n0 + CS * j];
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
  float* state;       // [B, H, L, dk, dv] or null: the chunk levels of the state after T-1
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
  if (sizeof(InT) == 2 && dk == kD && dv == kD &&
      ((reinterpret_cast<uintptr_t>(a.q) | reinterpret_cast<uintptr_t>(a.k) |
        reinterpret_cast<uintptr_t>(a.v)) & 15u) == 0) {  // aligned bf16 rows of 128: 8 values per load
#pragma unroll 4
    for (int i = tid; i < kC * (kD / 8); i += kThreads) {
      const int t = i / (kD / 8), d8 = 8 * (i - t * (kD / 8));
      const bool live = t < n;
      const int64_t tq = ((int64_t)b * a.T + t0 + t) * Hqk + hq;
      const int64_t tv = ((int64_t)b * a.T + t0 + t) * a.H + h;
      const uint4 z4 = make_uint4(0, 0, 0, 0);
      const uint4 uq = live ? *reinterpret_cast<const uint4*>(static_cast<const InT*>(a.q) + tq * dk + d8) : z4;
      const uint4 uk = live ? *reinterpret_cast<const uint4*>(static_cast<const InT*>(a.k) + tq * dk + d8) : z4;
      const uint4 uv = live ? *reinterpret_cast<const uint4*>(static_cast<const InT*>(a.v) + tv * dv + d8) : z4;
      const uint32_t wq[4] = {uq.x, uq.y, uq.z, uq.w}, wk[4] = {uk.x, uk.y, uk.z, uk.w},
                     wv[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fq = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wq[e]));
        const float2 fk = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wk[e]));
        const float2 fv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[e]));
        Qs[t * kLd + d8 + 2 * e] = fq.x; Qs[t * kLd + d8 + 2 * e + 1] = fq.y;
        Ks[t * kLd + d8 + 2 * e] = fk.x; Ks[t * kLd + d8 + 2 * e + 1] = fk.y;
        Vs[t * kLd + d8 + 2 * e] = fv.x; Vs[t * kLd + d8 + 2 * e + 1] = fv.y;
      }
    }
  } else
#pragma unroll 8
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
  // of k for column c.  A column depends only on its own earlier rows, and its four
  // threads are in one warp: a warp barrier orders each row before the next.
  {
    const int c = tid >> 2, part = tid & 3;
    for (int i = 0; i < kC; ++i) {
      float x = 0.f;
      if (c < i)
        for (int kk = c + part; kk < i; kk += 4) x = fmaf(Ws[i * kLdc + kk], Ts[kk * kLdc + c], x);
      x += __shfl_xor_sync(0xffffffffu, x, 1);
      x += __shfl_xor_sync(0xffffffffu, x, 2);
      if (part == 0) Ts[i * kLdc + c] = c < i ? -x : (c == i ? 1.f : 0.f);
      __syncwarp();
    }
  }
  __syncthreads();
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
    mma_tile<4, 8, false, false, 16>(o, Ws, kLdc, Vs, kLd, 0, kC, 4 * tm, tn);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 4 * tm + i;
      if (t >= n) continue;
      float* dst = a.o_intra + (((int64_t)b * a.T + t0 + t) * a.H + h) * dv;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
        if (tn + 16 * jj < dv) dst[tn + 16 * jj] = o[i][jj];
    }
  }
  // ---- X = T diag(beta gamma) K: rows 4 tm.., columns tn + 16 jj
  {
    float x[4][8];
    zero(x);
    for (int k = 0; k < kC; ++k) {
      const float sc = bet[k] * gam[k];
      float tv[4], kv[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) tv[i] = Ts[(4 * tm + i) * kLdc + k];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) kv[jj] = sc * Ks[k * kLd + tn + 16 * jj];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) x[i][jj] = fmaf(tv[i], kv[jj], x[i][jj]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) Xs[(4 * tm + i) * kLd + tn + 16 * jj] = x[i][jj];
  }
  __syncthreads();
  const int64_t chunk = bh * a.N + j;
  // ---- Qt = diag(gamma) Q - Aqk X  (64 x dk) to the workspace
  {
    float qv[4][8];
    zero(qv);
    mma_tile<4, 8, false, false, 16>(qv, Aqk, kLdc, Xs, kLd, 0, kC, 4 * tm, tn);
    float* dst = a.qt + chunk * kC * dk;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 4 * tm + i;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int d = tn + 16 * jj;
        if (d < dk) dst[t * dk + d] = gam[t] * Qs[t * kLd + d] - qv[i][jj];
      }
    }
  }
  // ---- P = gamma_end I - K^T diag(Gam[end, :]) X  (dk x dk): thread rows 8 tm.., columns
  // tn + 16 jj
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
      for (int jj = 0; jj < 8; ++jj) xv[jj] = Xs[s * kLd + tn + 16 * jj];
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
        const int c = tn + 16 * jj;
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
      for (int jj = 0; jj < 8; ++jj) vv[jj] = bet[k] * Vs[k * kLd + tn + 16 * jj];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) y[i][jj] = fmaf(tv[i], vv[jj], y[i][jj]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) Qs[(4 * tm + i) * kLd + tn + 16 * jj] = y[i][jj];
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
      for (int jj = 0; jj < 8; ++jj) yv[jj] = Qs[s * kLd + tn + 16 * jj];
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
        const int c = tn + 16 * jj;
        if (c < dv) dst[r * dv + c] = u[i][jj];
      }
    }
  }
}

// ---------------------------------------------------------------- the scan over chunks
//
// Thread layout: 256 threads = 16 columns x 16 row groups; thread (rg, col) holds rows
// [8 rg, 8 rg + 8) of column col of every chunk level in registers (Z^m, m < kLv: 12 slots
// up to 2^11 chunks, 20 up to 2^19).  Per
// chunk and live level the level's column block is staged in shared memory, then each
// thread adds its four tokens' readout (Qt Z^m) and carries its rows (P Z^m).  The chunk's
// P and Qt are in shared memory, the next chunk's loading meanwhile (cp.async, two buffers).
constexpr int kMaxLv = 20;     // chunk levels 1..19: up to 2^19 chunks
constexpr int kLdp = kD + 4;   // row stride of P and Qt in shared memory (16-byte rows)

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async4g(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

template <typename OutT, int kLv>
__global__ void __launch_bounds__(kThreads, 1) gdn_chunk_scan_kernel(GdnChunkArgs a, int levels) {
  extern __shared__ __align__(16) float sm2[];
  float* Pb = sm2;                          // [2][kD][kLdp]
  float* Qb = Pb + 2 * kD * kLdp;           // [2][kC][kLdp]
  float* Zs = Qb + 2 * kC * kLdp;           // [kD][kCols]: one level's column block
  float* Lb = Zs + kD * kCols;              // [2][kC][kMaxLv]: lambda of the chunk levels
  float* Zs2 = Lb + 2 * kC * kMaxLv;        // [kD][kCols]: a second level's column block
  const int tid = threadIdx.x;
  const int slices = (a.dv + kCols - 1) / kCols;
  const int64_t bh = blockIdx.x / slices;
  const int c0 = (int)(blockIdx.x - bh * slices) * kCols;
  const int b = (int)(bh / a.H), h = (int)(bh - (int64_t)b * a.H);
  const int dk = a.dk, dv = a.dv;
  const int col = tid & (kCols - 1), rg = tid >> 4;  // column, row group (rows 8 rg..)
  const bool col_ok = c0 + col < dv;
  const bool vec = (dk & 3) == 0;  // 16-byte copies of P and Qt rows

  // the chunk's transition P [dk][dk], carried queries Qt [64][dk] and the lambdas of its
  // tokens at the chunk levels into buffer j & 1
  auto issue = [&](int j) {
    const int64_t chunk = bh * a.N + j;
    const float* Pg = a.P + chunk * (int64_t)dk * dk;
    const float* Qg = a.qt + chunk * kC * dk;
    float* Pd = Pb + (j & 1) * kD * kLdp;
    float* Qd = Qb + (j & 1) * kC * kLdp;
    float* Ld = Lb + (j & 1) * kC * kMaxLv;
    const int nt = min(kC, a.T - j * kC);
    for (int i = tid; i < nt * (levels - 1); i += kThreads) {
      const int t = i / (levels - 1), m = 1 + i - t * (levels - 1);
      const int64_t tv = ((int64_t)b * a.T + j * kC + t) * a.H + h;
      cp_async4g(Ld + t * kMaxLv + m, a.lam + tv * a.L + kLc + m);
    }
    if (vec) {
      const int q4 = dk / 4;
      for (int i = tid; i < dk * q4; i += kThreads) {
        const int r = i / q4, c = i - r * q4;
        cp_async16(Pd + r * kLdp + 4 * c, Pg + r * dk + 4 * c);
      }
      for (int i = tid; i < kC * q4; i += kThreads) {
        const int r = i / q4, c = i - r * q4;
        cp_async16(Qd + r * kLdp + 4 * c, Qg + r * dk + 4 * c);
      }
    } else {
      for (int i = tid; i < dk * dk; i += kThreads) {
        const int r = i / dk, c = i - r * dk;
        cp_async4g(Pd + r * kLdp + c, Pg + i);
      }
      for (int i = tid; i < kC * dk; i += kThreads) {
        const int r = i / dk, c = i - r * dk;
        cp_async4g(Qd + r * kLdp + c, Qg + i);
      }
    }
  };

  float z[kLv][8];  // Z^m rows 8 rg.., column col (index m; slot 0 unused)
#pragma unroll
  for (int m = 0; m < kLv; ++m)
#pragma unroll
    for (int i = 0; i < 8; ++i) z[m][i] = 0.f;
  uint32_t live = 0;  // bit m: Z^m holds data
  float u_next[8];    // U_{j} rows 8 rg.., column col: merged at the start of chunk j+1
  // the copies fill columns [0, dk) of each row; the padding up to a multiple of 4, read
  // by the float4 loop (times zero rows of Z), stays zero
  for (int i = tid; i < 2 * kD * kLdp + 2 * kC * kLdp + 2 * kD * kCols + 2 * kC * kMaxLv; i += kThreads)
    Pb[i] = 0.f;
  __syncthreads();
  issue(0);
  cp_commit();
  for (int j = 0; j < a.N; ++j) {
    const int64_t chunk = bh * a.N + j;
    const int t0 = j * kC, n = min(kC, a.T - t0);
    if (j + 1 < a.N) issue(j + 1);
    cp_commit();
    // ---- merge at the chunk start: Z^{l+1} <- U_{j-1} + sum_{m <= l} Z^m, l = lssb(j)
    if (j > 0) {
      const int l = __ffs(j) - 1;
      float x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = u_next[i];
#pragma unroll
      for (int m = 1; m < kLv; ++m) {
        if (m > l) break;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          x[i] += z[m][i];
          z[m][i] = 0.f;
        }
      }
#pragma unroll
      for (int m = 1; m < kLv; ++m)
        if (m == l + 1) {
#pragma unroll
          for (int i = 0; i < 8; ++i) z[m][i] = x[i];
        }
      live = (live & ~((2u << l) - 2u)) | (1u << (l + 1));
    }
    // this chunk's own state (merged at the next chunk) and partial outputs: loads issued
    // now, used after the level work
    {
      const float* Uc = a.U + chunk * (int64_t)dk * dv;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = 8 * rg + i;
        u_next[i] = (r < dk && col_ok) ? Uc[r * dv + c0 + col] : 0.f;
      }
    }
    float oi[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = rg + 16 * i;
      const int64_t tv = ((int64_t)b * a.T + t0 + t) * a.H + h;
      oi[i] = (t < n && col_ok) ? a.o_intra[tv * dv + c0 + col] : 0.f;
    }
    cp_wait1();  // this chunk's P, Qt and lambdas have landed (the next chunk's may not)
    __syncthreads();
    const float* Ps = Pb + (j & 1) * kD * kLdp;
    const float* Qs = Qb + (j & 1) * kC * kLdp;
    const float* Ls = Lb + (j & 1) * kC * kMaxLv;
    // ---- the live levels two at a time: readout of four tokens (t = rg + 16 i) and the
    // carry of 8 rows for each, every row of P and Qt read once for both
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t todo = live & ~1u & (levels < 32 ? (1u << levels) - 1u : ~0u);
    while (todo) {
      const int m1 = __ffs(todo) - 1;
      todo &= todo - 1;
      const int m2 = todo ? __ffs(todo) - 1 : 0;  // 0: m1 is the last one
      todo &= todo - 1;
#pragma unroll
      for (int m = 1; m < kLv; ++m) {
        if (m == m1) {
#pragma unroll
          for (int i = 0; i < 8; ++i) Zs[(8 * rg + i) * kCols + col] = z[m][i];
        }
        if (m == m2) {
#pragma unroll
          for (int i = 0; i < 8; ++i) Zs2[(8 * rg + i) * kCols + col] = z[m][i];
        }
      }
      __syncthreads();
      float rd0[4] = {0.f, 0.f, 0.f, 0.f}, rd1[4] = {0.f, 0.f, 0.f, 0.f};
      float cr0[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      float cr1[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      // four d at a time: rows of P and Qt as float4 (padded to a multiple of 4 with the
      // zero rows of Z beyond d_k)
      if (m2) {
        for (int d = 0; d < dk; d += 4) {
          float zd[4], ze[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            zd[e] = Zs[(d + e) * kCols + col];
            ze[e] = Zs2[(d + e) * kCols + col];
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 q4 = *reinterpret_cast<const float4*>(Qs + (rg + 16 * i) * kLdp + d);
            rd0[i] = fmaf(q4.x, zd[0], fmaf(q4.y, zd[1], fmaf(q4.z, zd[2], fmaf(q4.w, zd[3], rd0[i]))));
            rd1[i] = fmaf(q4.x, ze[0], fmaf(q4.y, ze[1], fmaf(q4.z, ze[2], fmaf(q4.w, ze[3], rd1[i]))));
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 p4 = *reinterpret_cast<const float4*>(Ps + (8 * rg + i) * kLdp + d);
            cr0[i] = fmaf(p4.x, zd[0], fmaf(p4.y, zd[1], fmaf(p4.z, zd[2], fmaf(p4.w, zd[3], cr0[i]))));
            cr1[i] = fmaf(p4.x, ze[0], fmaf(p4.y, ze[1], fmaf(p4.z, ze[2], fmaf(p4.w, ze[3], cr1[i]))));
          }
        }
      } else {
        for (int d = 0; d < dk; d += 4) {
          float zd[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) zd[e] = Zs[(d + e) * kCols + col];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 q4 = *reinterpret_cast<const float4*>(Qs + (rg + 16 * i) * kLdp + d);
            rd0[i] = fmaf(q4.x, zd[0], fmaf(q4.y, zd[1], fmaf(q4.z, zd[2], fmaf(q4.w, zd[3], rd0[i]))));
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 p4 = *reinterpret_cast<const float4*>(Ps + (8 * rg + i) * kLdp + d);
            cr0[i] = fmaf(p4.x, zd[0], fmaf(p4.y, zd[1], fmaf(p4.z, zd[2], fmaf(p4.w, zd[3], cr0[i]))));
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        o[i] = fmaf(Ls[(rg + 16 * i) * kMaxLv + m1], rd0[i], o[i]);
        if (m2) o[i] = fmaf(Ls[(rg + 16 * i) * kMaxLv + m2], rd1[i], o[i]);
      }
#pragma unroll
      for (int m = 1; m < kLv; ++m) {
        if (m == m1) {
#pragma unroll
          for (int i = 0; i < 8; ++i) z[m][i] = 8 * rg + i < dk ? cr0[i] : 0.f;
        }
        if (m == m2) {
#pragma unroll
          for (int i = 0; i < 8; ++i) z[m][i] = 8 * rg + i < dk ? cr1[i] : 0.f;
        }
      }
      __syncthreads();  // Zs and Zs2 are rewritten by the next pair
    }
    // ---- the chunk's output rows: O_intra + readout
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = rg + 16 * i;
      if (t < n && col_ok) {
        const int64_t tv = ((int64_t)b * a.T + t0 + t) * a.H + h;
        static_cast<OutT*>(a.out)[tv * dv + c0 + col] = from_f32<OutT>(oi[i] + o[i]);
      }
    }
    __syncthreads();  // buffer j & 1 is refilled by the issue of chunk j + 2
  }
  // ---- the chunk-level states after the last chunk: levels 6 + m of the decode state
  if (a.state && col_ok) {
#pragma unroll
    for (int m = 1; m < kLv; ++m) {
      if (m >= levels || !((live >> m) & 1)) continue;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = 8 * rg + i;
        if (r < dk) a.state[((bh * a.L + kLc + m) * dk + r) * (int64_t)dv + c0 + col] = z[m][i];
      }
    }
  }
}

template <typename OutT, int kLv>
cudaError_t launch_scan(const GdnChunkArgs& a, int levels, unsigned grid, size_t smem,
                        cudaStream_t s) {
  const cudaError_t e = cudaFuncSetAttribute(gdn_chunk_scan_kernel<OutT, kLv>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
  if (e != cudaSuccess) return e;
  gdn_chunk_scan_kernel<OutT, kLv><<<grid, kThreads, smem, s>>>(a, levels);
  return cudaSuccess;
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
                               const float* beta, const float* lam, void* out, float* state,
                               int B, int T, int H, int Hqk, int dk, int dv, int L, int in_dtype,
                               int out_dtype, void* workspace, cudaStream_t s) {
  if (state) {  // levels the state does not reach stay zero
    const cudaError_t e =
        cudaMemsetAsync(state, 0, sizeof(float) * (size_t)B * H * L * dk * dv, s);
    if (e != cudaSuccess) return e;
  }
  if (T == 0) return cudaSuccess;
  GdnChunkArgs a;
  a.q = q; a.k = k; a.v = v; a.log_a = log_a; a.beta = beta; a.lam = lam; a.out = out;
  a.state = state;
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
  if (levels > kMaxLv) return cudaErrorInvalidValue;
  const size_t smem2 =
      sizeof(float) * ((size_t)2 * kD * kLdp + 2 * kC * kLdp + 2 * kD * kCols + 2 * kC * kMaxLv);
  const unsigned grid2 = (unsigned)((int64_t)B * H * ((dv + kCols - 1) / kCols));
  // the chunk-level states live in registers: the smallest instance that holds them
  if (out_dtype == LL_BF16)
    e = levels <= 10   ? launch_scan<__nv_bfloat16, 10>(a, levels, grid2, smem2, s)
        : levels <= 12 ? launch_scan<__nv_bfloat16, 12>(a, levels, grid2, smem2, s)
                       : launch_scan<__nv_bfloat16, kMaxLv>(a, levels, grid2, smem2, s);
  else
    e = levels <= 10   ? launch_scan<float, 10>(a, levels, grid2, smem2, s)
        : levels <= 12 ? launch_scan<float, 12>(a, levels, grid2, smem2, s)
                       : launch_scan<float, kMaxLv>(a, levels, grid2, smem2, s);
  if (e != cudaSuccess) return e;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (!state) return cudaSuccess;
  // the levels inside the last chunk (0..6): its own tokens run through the lssb steps from
  // an empty state (the chunk starts at a multiple of 64, so the low bits of the positions
  // are the same); the outputs of that run land in the partial-output scratch, which the
  // scan has consumed
  const int t_last = (a.N - 1) * kC;
  return launch_gdn_fwd_tail(q, k, v, log_a, beta, lam, a.o_intra, state, B, T, t_last, H, Hqk,
                             dk, dv, L, L < kLc + 1 ? L : kLc + 1, in_dtype, s);
}

}  // namespace ll

// Forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), bf16 inputs with
// fp32 accumulation, d_k = d_v = 128, 128-token tiles (the M = 128 datapath of one SM).
//
// The chunked two-stage algorithm (page "论文阅读：Log-Linear Attention", sections 矩阵分解
// and 两阶段计算; page "算力终结者来了！…", section 高效训练算法) with the tile as the chunk:
//
//   tc_chunk_state    per tile i: U_i^T = (w ⊙ V)^T K on tcgen05 (w_s = exp(cs_end - cs_s),
//                     cs = tile-local prefix sums of log a) into TMEM, and the tile's log
//                     decay lg_i.  The Fenwick block totals of tiles are merged in the same
//                     kernel as the tiles finish (fp32 in TMEM; the CTA that completes a
//                     sibling pair forms the parent) and stored bf16 [d_v][d_k] under the
//                     index of their first reader tile.
//   tc_intra_readout  per tile j: S = Q K^T (tcgen05, TMEM); P = S ⊙ exp(cs_t - cs_s) ⊙
//                     lambda[t, l(t,s)] on the causal half (CUDA cores, bf16 into shared
//                     memory); O = P V (tcgen05), moved to registers.  Then, for every set
//                     bit m-1 of j, one MMA Q Tot_m into one of two TMEM buffers while the
//                     previous level's product is added to O with the row weights
//                     r_t = lambda[t, 7+m] exp(cs_t + D_m) (D_m = log decay from the
//                     block's end to the tile's start).  The lambda-weighted per-level
//                     readout is thus fused into the output epilogue; no per-level output
//                     reaches memory.  bf16 output leaves through a TMA store.
//
// With 128-token tiles the chunk-pair level log2(C)+1 of a requested C = 64 lies inside a
// tile and is taken in the dense masked product; the sum is the same.
//
// Shared-memory tiles are 128 rows x 128 bf16 stored as two 64-column panels with the
// 128-byte swizzle TMA produces; K-major operands (Q, K, P, block states) and MN-major
// ones (V as the B of P V; V and K in the state GEMM) are described to tcgen05 with the
// matching descriptors.  Every mbarrier wait is bounded (see tc_ptx.cuh); a CTA whose
// wait times out raises g_tc_error, skips its remaining MMAs and stores, frees its TMEM
// and exits.
//
// Single-lane issue blocks (TMA, MMA) are followed by __syncwarp(): otherwise the other
// lanes of warp 0 reach the next mbarrier spin first and keep the issuing lane from
// being scheduled for microseconds.
#include <cudaTypedefs.h>

#include <mutex>

#include "ll_internal.cuh"
#include "tc_ptx.cuh"

namespace ll {

__device__ unsigned int g_tc_error = 0;

namespace {

using namespace tc;

constexpr int kTile = 128;                  // tokens per tile (= MMA M)
constexpr int kD = 128;                     // d_k = d_v
constexpr int kPanel = kTile * 64 * 2;      // one [128][64] bf16 panel: 16 KiB
constexpr int kOperand = 2 * kPanel;        // a 128 x 128 bf16 tile: 32 KiB
constexpr int kThreads = 128;               // one thread per tile row / TMEM lane
constexpr int kLamStride = 9;               // intra lambdas per row in smem (levels 0..7)
constexpr int kIntraLevels = 8;             // levels inside a 128-token tile: 0..7
constexpr int kTileLc = 7;                  // log2(kTile)
constexpr int kMaxChunkLevels = 32;         // chunk levels m = 1..31 (positions < 2^31)

struct TcParams {
  int B, T, H, L, N;
  const float* log_a;
  const float* lam;
  void* out;
  float* lg;         // [B*H][N] log decay of each tile
  uint8_t* nodes;    // [B*H][N] block states, bf16 [d_v][d_k], slot = first reader tile
  uint8_t* odd;      // [B*H][N] totals of odd blocks left for their sibling, slot = first tile
  float* blg;        // [B*H][N] log decays of the blocks left behind, slot = first tile
  uint32_t* cnt;     // [B*H][N] arrival counters of the sibling pairs, slot = midpoint tile
  int out_f32;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

// Inclusive prefix sum over the 128 threads of the CTA; red holds 4 floats and must not
// be reused before the next __syncthreads.
__device__ __forceinline__ float block_scan128(float x, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) red[warp] = x;
  __syncthreads();
  float pre = 0.f;
  for (int w = 0; w < warp; ++w) pre += red[w];
  return x + pre;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Multiplies row r of a 128 x 128 swizzled bf16 tile by s in place.  The swizzle only
// permutes the 16-byte chunks inside a row; walking them from chunk (r mod 8) makes the
// eight rows of a 1 KiB swizzle atom touch eight different bank groups at each step.
__device__ __forceinline__ void scale_row_inplace(uint8_t* buf, int r, float s) {
#pragma unroll
  for (int pnl = 0; pnl < 2; ++pnl) {
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
      const int c = (cc + r) & 7;
      uint4* ptr = reinterpret_cast<uint4*>(buf + pnl * kPanel + r * 128 + c * 16);
      uint4 u = *ptr;
      uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w[k]));
        w[k] = pack_bf16(f.x * s, f.y * s);
      }
      *ptr = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// Writes 32 fp32 values as bf16 into columns [32c, 32c+32) of row r of a swizzled tile.
__device__ __forceinline__ void put_row32_bf16(uint8_t* buf, int r, int c, const float* v) {
  uint8_t* panel = buf + (c >> 1) * kPanel;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4*>(panel + sw128_offset(r, (c & 1) * 4 + q)) =
        make_uint4(pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                   pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
}

__device__ __forceinline__ void put_row32_zero(uint8_t* buf, int r, int c) {
  uint8_t* panel = buf + (c >> 1) * kPanel;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4*>(panel + sw128_offset(r, (c & 1) * 4 + q)) = make_uint4(0, 0, 0, 0);
}

// A held block total: the 16-byte pieces q = it * 128 + tid (it = 0..15) of a row-major
// [128][128] bf16 matrix, 8 bf16 each, so that every warp moves 512 contiguous bytes per
// step.  Generic-proxy global accesses, so that another CTA can read the data after a
// release/acquire on a counter; the loads bypass L1 (the data was written by another SM
// during this launch).
constexpr int kPieces = kOperand / 16 / kThreads;  // 16 per thread

__device__ __forceinline__ void store_pieces(const uint4 (&x)[kPieces], uint8_t* dst, int tid) {
#pragma unroll
  for (int it = 0; it < kPieces; ++it) reinterpret_cast<uint4*>(dst)[it * kThreads + tid] = x[it];
}

// x <- bf16(g * left + right) elementwise, left/right = (x, the sibling's pieces) in the
// order `x_is_left` gives.  Both CTAs of a pair would compute the same bits.
__device__ __forceinline__ void merge_pieces(uint4 (&x)[kPieces], const uint8_t* sib, float g,
                                             bool x_is_left, int tid) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {  // 8 loads in flight per thread, bounded registers
    uint4 y[kPieces / 2];
#pragma unroll
    for (int u = 0; u < kPieces / 2; ++u)
      y[u] = __ldcg(reinterpret_cast<const uint4*>(sib) + (half * kPieces / 2 + u) * kThreads + tid);
#pragma unroll
    for (int u = 0; u < kPieces / 2; ++u) {
      const int it = half * kPieces / 2 + u;
      uint32_t a[4] = {x[it].x, x[it].y, x[it].z, x[it].w};
      const uint32_t c[4] = {y[u].x, y[u].y, y[u].z, y[u].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a[k]));
        const float2 fc = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&c[k]));
        const float2 l = x_is_left ? fa : fc, r = x_is_left ? fc : fa;
        a[k] = pack_bf16(fmaf(g, l.x, r.x), fmaf(g, l.y, r.y));
      }
      x[it] = make_uint4(a[0], a[1], a[2], a[3]);
    }
  }
}

// Whether the total of block pb at chunk level m (tiles [pb 2^(m-1), (pb+1) 2^(m-1))) is
// needed: an even block is the block state of its first reader tile (pb+1) 2^(m-1), if
// that tile exists; an odd block only feeds its parent.
__device__ __forceinline__ bool block_needed(int m, int64_t pb, int64_t N) {
  for (; m <= kMaxChunkLevels; ++m, pb >>= 1)
    if (!(pb & 1)) return ((pb + 1) << (m - 1)) < N;
  return false;
}

// ------------------------------------------------------------------ K1: chunk states
//
// Per tile i: U_i^T = (w ⊙ V)^T K into TMEM (fp32), then the Fenwick block states.  The
// block totals Tot(m+1, q) = exp(LG(2q+1)) Tot(m, 2q) + Tot(m, 2q+1) are merged as the
// tiles finish, without a separate scan and without waiting: each CTA holds the total of
// one block (first its own tile), stores it as a block state if the block is even (slot
// = its first reader tile), and counts itself in at the arrival counter of the block's
// sibling pair (keyed by the pair's midpoint tile, unique per pair).  The first of the two
// CTAs leaves its total for the other one (the block state of an even block; a scratch
// slot keyed by its first tile for an odd one, with the block's log decay) and exits; the
// second reads it, forms the parent and carries on one level up.  Only blocks some block
// state depends on are formed.  Totals cross CTAs in bf16, the format of the block states
// themselves, and both CTAs of a pair would compute the same bits.

__global__ void __launch_bounds__(kThreads, 3)
    tc_chunk_state_kernel(const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* Kb = smem;                // K, then U_i^T in bf16
  uint8_t* Vb = smem + kOperand;     // V
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * kOperand);  // [0] load, [1] mma
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
  float* red = reinterpret_cast<float*>(tslot + 4);
  float* lg_s = red + 4;
  uint32_t* flag_s = reinterpret_cast<uint32_t*>(lg_s + 1);  // 2 per chunk level

  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int t0 = i * kTile;
  const int n = min(kTile, p.T - t0);
  const int64_t bh = (int64_t)b * p.H + h;

  if (warp == 0) {
    tmem_alloc(tslot, 128);
    tmem_relinquish();
  }
  if (tid == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t lane = (uint32_t)(warp * 32) << 16;
  if (tid == 0) {
    mbar_arrive_expect_tx(&bars[0], 2 * kOperand);
    tma_load_4d(&tmK, &bars[0], Kb, 0, h, t0, b);
    tma_load_4d(&tmK, &bars[0], Kb + kPanel, 64, h, t0, b);
    tma_load_4d(&tmV, &bars[0], Vb, 0, h, t0, b);
    tma_load_4d(&tmV, &bars[0], Vb + kPanel, 64, h, t0, b);
  }
  __syncwarp();
  const float la = (p.log_a && tid < n) ? p.log_a[((int64_t)b * p.T + t0 + tid) * p.H + h] : 0.f;
  const float cs = block_scan128(la, red);
  if (tid == kThreads - 1) lg_s[0] = cs;  // padding rows add 0: the last prefix is the total
  __syncthreads();
  const float lg = lg_s[0];
  const float w = tid < n ? expf(lg - cs) : 0.f;

  bool ok = mbar_wait(&bars[0], 0);
  if (ok) scale_row_inplace(Vb, tid, w);
  fence_proxy_async_smem();
  const bool all_ok = __syncthreads_and(ok);
  if (all_ok && tid == 0) {
    tc_fence_after();
    constexpr uint32_t idesc = idesc_bf16(128, 128, /*A MN-major*/ 1, /*B MN-major*/ 1);
    const uint32_t a0 = smem_u32(Vb), b0 = smem_u32(Kb);
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk) {
      const uint64_t ad = smem_desc_sw128(a0 + kk * 2048, kPanel, 1024);
      const uint64_t bd = smem_desc_sw128(b0 + kk * 2048, kPanel, 1024);
      mma_bf16(tmem, ad, bd, idesc, kk > 0);
    }
    mma_commit(&bars[1]);
  }
  __syncwarp();  // lane 0 must finish issuing before its warp spins on the barrier
  const bool ok2 = all_ok && mbar_wait(&bars[1], 0);
  tc_fence_after();
  if (__syncthreads_and(ok2)) {
    if (tid == 0) p.lg[bh * p.N + i] = lg;
    // row tid of U^T (d_v index) -> bf16 into Kb (free since the MMA completed), then
    // re-read in the piece layout
#pragma unroll 1
    for (int c = 0; c < kD / 32; ++c) {
      float v[32];
      tmem_ld32(tmem + lane + c * 32, v);
      put_row32_bf16(Kb, tid, c, v);
    }
    __syncthreads();
    uint4 x[kPieces];
#pragma unroll
    for (int it = 0; it < kPieces; ++it) {
      const int q = it * kThreads + tid, row = q >> 4, c16 = q & 15;
      x[it] = *reinterpret_cast<const uint4*>(Kb + (c16 >> 3) * kPanel + sw128_offset(row, c16 & 7));
    }
    const int64_t N = p.N;
    uint8_t* nodes = p.nodes + bh * N * kOperand;
    uint8_t* odd = p.odd + bh * N * kOperand;
    float* blg = p.blg + bh * N;
    uint32_t* cnt = p.cnt + bh * N;
    float LGb = lg;  // log decay of the held block
    int64_t pb = i;  // the held block: index pb at chunk level m
    for (int m = 1; m <= kMaxChunkLevels; ++m, pb >>= 1) {
      const bool even = !(pb & 1);
      const int64_t start = pb << (m - 1), end = (pb + 1) << (m - 1);
      if (even) {
        if (end >= N) break;  // no reader tile and no sibling
        store_pieces(x, nodes + end * kOperand, tid);
      }
      if (!block_needed(m + 1, pb >> 1, N)) break;
      // Arrival at the pair (midpoint tile as key).  Publication protocol: every thread's
      // stores, then a block barrier, then thread 0 fences and counts in (the fence is
      // cumulative over the barrier); the CTA that finds the count at 1 fences again and
      // the barrier hands the acquire to every thread before the sibling is read.
      uint32_t* pair = cnt + (even ? end : start);
      uint32_t* fl = flag_s + 2 * m;
      bool second = false;
      if (!even) {  // a right half often finds its left sibling in already
        if (tid == 0) fl[0] = ld_acquire_gpu(pair);
        __syncthreads();
        second = fl[0] != 0;
      }
      if (!second) {
        if (!even) store_pieces(x, odd + start * kOperand, tid);
        if (tid == 0) blg[start] = LGb;
        __syncthreads();
        if (tid == 0) {
          __threadfence();
          fl[1] = atomicAdd(pair, 1u);
          __threadfence();
        }
        __syncthreads();
        second = fl[1] != 0;
        if (!second) break;  // the sibling's CTA forms the parent
      }
      const int64_t len = int64_t(1) << (m - 1);
      const float sib_lg = __ldcg(blg + (even ? end : start - len));
      const float g = expf(even ? sib_lg : LGb);  // decay across the right half
      merge_pieces(x, even ? odd + end * kOperand : nodes + start * kOperand, g, even, tid);
      LGb = even ? LGb + sib_lg : sib_lg + LGb;
    }
  } else if (tid == 0) {
    atomicOr(&g_tc_error, 1u);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

// ------------------------------------------------------------------ K3: intra + readout

// 8 warps: warps w and w+4 share TMEM lane quarter w mod 4 (tile rows 32(w mod 4)..+31).
// They split that quarter's causal chunks of P between them, and the output columns
// (64 each) of O and of every level epilogue.
constexpr int kThreads3 = 256;

struct K3Smem {
  // byte offsets from the 1024-aligned base
  static constexpr int kQ = 0, kK = kOperand, kV = 2 * kOperand;
  static constexpr int kBars = 3 * kOperand;                   // 7 mbarriers
  static constexpr int kTslot = kBars + 7 * 8;
  static constexpr int kRed = kTslot + 16;                     // 8 floats
  static constexpr int kCarry = kRed + 32;                     // 4 floats
  static constexpr int kCs = kCarry + 16;                      // 128 floats
  static constexpr int kLam = kCs + 4 * kTile;                 // 128 x kLamStride floats
  static constexpr int kDm = kLam + 4 * kTile * kLamStride;    // kMaxChunkLevels floats
  static constexpr int kRs = kDm + 4 * kMaxChunkLevels;        // [levels][128] floats
};

// Inclusive prefix sum over the 256 threads of the CTA; red holds 8 floats and must not
// be reused before the next __syncthreads.
__device__ __forceinline__ float block_scan256(float x, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) red[warp] = x;
  __syncthreads();
  float pre = 0.f;
  for (int w = 0; w < warp; ++w) pre += red[w];
  return x + pre;
}

__global__ void __launch_bounds__(kThreads3, 2)
    tc_intra_readout_kernel(const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV,
                            const __grid_constant__ CUtensorMap tmNode,
                            const __grid_constant__ CUtensorMap tmOut, TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* Qb = smem + K3Smem::kQ;
  uint8_t* Kb = smem + K3Smem::kK;   // K, then P, then the block states of odd levels
  uint8_t* Vb = smem + K3Smem::kV;   // V, then the block states of even levels
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + K3Smem::kBars);
  uint64_t* bar_load = &bars[0];
  uint64_t* bar_s = &bars[1];
  uint64_t* bar_o = &bars[2];
  uint64_t* bar_node = &bars[3];     // [2]
  uint64_t* bar_lvl = &bars[5];      // [2]
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + K3Smem::kTslot);
  float* red = reinterpret_cast<float*>(smem + K3Smem::kRed);
  float* carry_s = reinterpret_cast<float*>(smem + K3Smem::kCarry);
  float* cs_s = reinterpret_cast<float*>(smem + K3Smem::kCs);
  float* lam_s = reinterpret_cast<float*>(smem + K3Smem::kLam);
  float* Dm = reinterpret_cast<float*>(smem + K3Smem::kDm);
  float* rs = reinterpret_cast<float*>(smem + K3Smem::kRs);

  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int qt = warp & 3;           // row quarter (TMEM lane quarter) of this warp
  const int hh = warp >> 2;          // which of the quarter's two warps
  const int r = tid & (kTile - 1);   // tile row of this thread
  const int t0 = j * kTile;
  const int n = min(kTile, p.T - t0);
  const int64_t bh = (int64_t)b * p.H + h;
  const int64_t row = ((int64_t)b * p.T + t0 + r) * p.H + h;  // (b, t, h) of row r
  const int nlev = __popc((unsigned)j);                        // inter-chunk levels read

  // ---- per-row data.  Every global load of the prologue is issued first, before the
  // TMEM allocation and the tile loads (log a, the intra- and inter-level lambdas, the
  // tile log decays D_m sums over), so that their latencies overlap; the scans and
  // exponentials follow.  The two threads of a row split the loads.
  const float* lgp = p.lg + bh * p.N;
  const int top = nlev > 0 ? 31 - __clz((unsigned)j) : 0;
  const int span = nlev > 0 ? j - (1 << top) : 0;  // the longest range j - c_m
  const bool row_live = r < n;
  const float la = (hh == 0 && p.log_a && row_live) ? p.log_a[row] : 0.f;
  float lam_in[kIntraLevels / 2];
#pragma unroll
  for (int i = 0; i < kIntraLevels / 2; ++i) {
    const int l = hh * (kIntraLevels / 2) + i;
    lam_in[i] = (row_live && l < p.L) ? p.lam[row * p.L + l] : 0.f;
  }
  const float lg_first = tid < span ? lgp[j - 1 - tid] : 0.f;
  {  // raw inter-level lambdas, level-major in smem (weighted below); levels alternate
    int k = 0;  // between the two threads of a row
#pragma unroll 4
    for (int m = 1; m < kMaxChunkLevels; ++m) {
      if (!((j >> (m - 1)) & 1)) continue;
      if ((k & 1) == hh) rs[k * kTile + r] = row_live ? p.lam[row * p.L + kTileLc + m] : 0.f;
      ++k;
    }
  }
  if (warp == 0) {
    tmem_alloc(tslot, 256);
    tmem_relinquish();
  }
  if (tid == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    prefetch_tensormap(&tmNode);
    prefetch_tensormap(&tmOut);
    for (int q = 0; q < 7; ++q) mbar_init(&bars[q], 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t lane_base = (uint32_t)(qt * 32) << 16;
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_load, 3 * kOperand);
    tma_load_4d(&tmQ, bar_load, Qb, 0, h, t0, b);
    tma_load_4d(&tmQ, bar_load, Qb + kPanel, 64, h, t0, b);
    tma_load_4d(&tmK, bar_load, Kb, 0, h, t0, b);
    tma_load_4d(&tmK, bar_load, Kb + kPanel, 64, h, t0, b);
    tma_load_4d(&tmV, bar_load, Vb, 0, h, t0, b);
    tma_load_4d(&tmV, bar_load, Vb + kPanel, 64, h, t0, b);
  }
  if (tid == 32) {  // another warp warms L2 with every block state this tile will read
    for (int m = 1; m < kMaxChunkLevels; ++m) {
      int64_t c;
      if (!inter_block(j, m, &c)) continue;
      const int r0 = (int)((bh * p.N + c) * kD);
      tma_prefetch_2d(&tmNode, 0, r0);
      tma_prefetch_2d(&tmNode, 64, r0);
    }
  }
  __syncwarp();
  const float cs_scan = block_scan256(la, red);  // threads 0..127 hold row prefixes
  if (hh == 0) cs_s[r] = cs_scan;
#pragma unroll
  for (int i = 0; i < kIntraLevels / 2; ++i)
    lam_s[r * kLamStride + hh * (kIntraLevels / 2) + i] = lam_in[i];
  // D_m = sum of lg over tiles [c_m, j), from inclusive prefix sums of lg[j-1], lg[j-2], ..
  if (nlev > 0) {
    if (tid == 0) {
      carry_s[0] = 0.f;
      for (int m = 1; m <= top + 1; ++m)
        if (((j >> (m - 1)) & 1) && ((j >> (m - 1)) << (m - 1)) == j) Dm[m] = 0.f;
    }
    for (int base = 0; base < span; base += kThreads3) {
      __syncthreads();
      const int idx = base + tid;
      const float x = base == 0 ? lg_first : (idx < span ? lgp[j - 1 - idx] : 0.f);
      const float incl = block_scan256(x, red) + carry_s[0];
      for (int m = 1; m <= top + 1; ++m) {
        if (!((j >> (m - 1)) & 1)) continue;
        const int c = (j >> (m - 1)) << (m - 1);
        if (j - c - 1 == idx) Dm[m] = incl;
      }
      __syncthreads();
      if (tid == kThreads3 - 1) carry_s[0] = incl;
    }
  }
  __syncthreads();
  const float cs = cs_s[r];
  {  // per-level row weights r_t = lambda[t, 7+m] exp(cs_t + D_m)
    int k = 0;
    for (int m = 1; m < kMaxChunkLevels; ++m) {
      if (!((j >> (m - 1)) & 1)) continue;
      if ((k & 1) == hh) rs[k * kTile + r] *= __expf(cs + Dm[m]);
      ++k;
    }
  }

  // ---- S = Q K^T
  bool ok = mbar_wait(bar_load, 0);
  bool all_ok = __syncthreads_and(ok);
  if (all_ok && tid == 0) {
    tc_fence_after();
    constexpr uint32_t idesc = idesc_bf16(128, 128, 0, 0);
    const uint32_t qa = smem_u32(Qb), ka = smem_u32(Kb);
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
      mma_bf16(tmem, smem_desc_sw128(qa + off, 16, 1024), smem_desc_sw128(ka + off, 16, 1024),
               idesc, kk > 0);
    }
    mma_commit(bar_s);
  }
  __syncwarp();  // lane 0 must finish issuing before its warp spins on the barrier
  ok = all_ok && mbar_wait(bar_s, 0);
  tc_fence_after();
  all_ok = __syncthreads_and(ok);
  // ---- P = S ⊙ exp(cs_t - cs_s) ⊙ lambda[t, l(t, s)] on s <= t, bf16 into Kb (K-major).
  // The two warps of quarter qt take the 32-column chunks of their parity.  Chunks
  // c > qt lie above the diagonal (zero); chunks c < qt lie below it, where every pair
  // has the same level 5 + bit_length(qt XOR c); chunk qt holds the diagonal.
  if (all_ok) {
    const float* lam_r = lam_s + r * kLamStride;
    for (int c = hh; c < kTile / 32; c += 2) {
      if (c > qt) {
        put_row32_zero(Kb, r, c);
        continue;
      }
      float sv[32];
      tmem_ld32(tmem + lane_base + c * 32, sv);
      if (c < qt) {
        const float wl = lam_r[5 + (32 - __clz((unsigned)(qt ^ c)))];
#pragma unroll
        for (int k = 0; k < 32; ++k) sv[k] *= wl * __expf(cs - cs_s[c * 32 + k]);
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int s = c * 32 + k;
          float v = 0.f;
          if (s <= r && row_live)
            v = sv[k] * lam_r[fenwick_level((uint32_t)r, (uint32_t)s)] * __expf(cs - cs_s[s]);
          sv[k] = v;
        }
      }
      put_row32_bf16(Kb, r, c, sv);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  // ---- O = P V  (V MN-major as B)
  if (all_ok && tid == 0) {
    tc_fence_after();
    constexpr uint32_t idesc = idesc_bf16(128, 128, 0, 1);
    const uint32_t pa = smem_u32(Kb), va = smem_u32(Vb);
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk) {
      const uint32_t aoff = (kk >> 2) * kPanel + (kk & 3) * 32;
      mma_bf16(tmem + 128, smem_desc_sw128(pa + aoff, 16, 1024),
               smem_desc_sw128(va + kk * 2048, kPanel, 1024), idesc, kk > 0);
    }
    mma_commit(bar_o);
  }
  __syncwarp();
  ok = all_ok && mbar_wait(bar_o, 0);
  tc_fence_after();
  all_ok = __syncthreads_and(ok);
  // this thread's half of the output row: columns [64 hh, 64 hh + 64)
  float o[kD / 2];
#pragma unroll
  for (int q = 0; q < kD / 2; ++q) o[q] = 0.f;
  const uint32_t col0 = 64u * hh;
  if (all_ok) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float v[32];
      tmem_ld32(tmem + lane_base + 128 + col0 + c * 32, v);
#pragma unroll
      for (int q = 0; q < 32; ++q) o[c * 32 + q] = v[q];
    }
  }
  tc_fence_before();
  __syncthreads();  // Kb, Vb and all 256 TMEM columns are free from here on

  // ---- inter-chunk levels: MMA into alternating TMEM buffers, weighted adds into o.
  // Level k uses shared buffer (k odd ? Kb : Vb), TMEM columns [128 (k&1), +128),
  // mbarriers bar_node[k&1] (its block state arrived) and bar_lvl[k&1] (its MMA finished).
  if (all_ok && tid == 0) {
    int k = 0;
    for (int m = 1; m < kMaxChunkLevels && k < 2; ++m) {
      int64_t c;
      if (!inter_block(j, m, &c)) continue;
      const int r0 = (int)((bh * p.N + c) * kD);
      uint8_t* dst = (k & 1) ? Kb : Vb;
      mbar_arrive_expect_tx(&bar_node[k], kOperand);
      tma_load_2d(&tmNode, &bar_node[k], dst, 0, r0);
      tma_load_2d(&tmNode, &bar_node[k], dst + kPanel, 64, r0);
      ++k;
    }
  }
  uint32_t node_ph[2] = {0, 0}, lvl_ph[2] = {0, 0};
  int m_next = 1;  // scan position of the next block state to load (after the first two)
  if (tid == 0) {
    int seen = 0;
    for (; m_next < kMaxChunkLevels; ++m_next) {
      if (!((j >> (m_next - 1)) & 1)) continue;
      if (++seen > 2) break;
    }
  }
  __syncwarp();
  for (int k = 0; k <= nlev && all_ok; ++k) {
    if (k < nlev) {  // issue level k
      const int bf = k & 1;
      ok = mbar_wait(&bar_node[bf], node_ph[bf]);
      node_ph[bf] ^= 1;
      all_ok = __syncthreads_and(ok);
      if (!all_ok) break;
      if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t idesc = idesc_bf16(128, 128, 0, 0);
        const uint32_t qa = smem_u32(Qb), sa = smem_u32(bf ? Kb : Vb);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          mma_bf16(tmem + bf * 128, smem_desc_sw128(qa + off, 16, 1024),
                   smem_desc_sw128(sa + off, 16, 1024), idesc, kk > 0);
        }
        mma_commit(&bar_lvl[bf]);
      }
      __syncwarp();
    }
    if (k >= 1) {  // finish level k-1 while level k runs
      const int bf = (k - 1) & 1;
      ok = mbar_wait(&bar_lvl[bf], lvl_ph[bf]);
      lvl_ph[bf] ^= 1;
      tc_fence_after();
      all_ok = __syncthreads_and(ok);
      if (!all_ok) break;
      const float wr = rs[(k - 1) * kTile + r];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float v[32];
        tmem_ld32(tmem + lane_base + bf * 128 + col0 + c * 32, v);
#pragma unroll
        for (int q = 0; q < 32; ++q) o[c * 32 + q] = fmaf(wr, v[q], o[c * 32 + q]);
      }
      tc_fence_before();
      __syncthreads();  // buffer bf (TMEM and shared) is free again
      if (tid == 0 && k + 1 < nlev) {  // block state of level k+1 into buffer bf
        int64_t c = 0;
        while (m_next < kMaxChunkLevels && !inter_block(j, m_next, &c)) ++m_next;
        const int r0 = (int)((bh * p.N + c) * kD);
        ++m_next;
        uint8_t* dst = bf ? Kb : Vb;
        mbar_arrive_expect_tx(&bar_node[bf], kOperand);
        tma_load_2d(&tmNode, &bar_node[bf], dst, 0, r0);
        tma_load_2d(&tmNode, &bar_node[bf], dst + kPanel, 64, r0);
      }
      __syncwarp();
    }
  }

  // ---- epilogue
  if (all_ok) {
    if (p.out_f32) {
      if (row_live) {
        float4* dst =
            reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + row * kD + col0);
#pragma unroll
        for (int q = 0; q < kD / 8; ++q)
          dst[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
      }
    } else {
      // no MMA reads Q any more: stage the bf16 tile there and store it with TMA
#pragma unroll
      for (int c = 0; c < 2; ++c) put_row32_bf16(Qb, r, 2 * hh + c, o + c * 32);
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        tma_store_4d(&tmOut, Qb, 0, h, t0, b);
        tma_store_4d(&tmOut, Qb + kPanel, 64, h, t0, b);
        tma_store_commit();
        tma_store_wait_read();
      }
      __syncwarp();
    }
  } else if (tid == 0) {
    atomicOr(&g_tc_error, 1u);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// [B, T, H, 128] bf16, boxes of 128 tokens x 64 features of one (b, h); rows past T read
// as 0 and are not written.
bool make_tokens_map(CUtensorMap* m, const void* base, int B, int T, int H) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2,
                           (cuuint64_t)T * H * kD * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)kTile, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows][128] bf16 matrices (chunk states, block states), boxes of 128 rows x 64 columns.
bool make_rows_map(CUtensorMap* m, const void* base, int64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kTile};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr size_t kSmemK1 = 2 * kOperand + 1024 + 512;
size_t smem_k3(int levels) { return (size_t)K3Smem::kRs + 4 * kTile * levels + 1024; }

}  // namespace

bool tc_forward_supported(int64_t dk, int64_t dv, int in_dtype, int /*chunk*/) {
  return in_dtype == LL_BF16 && dk == kD && dv == kD;
}

cudaError_t launch_tc_forward(const FwdArgs& a, int out_dtype, cudaStream_t s, StageEvents* ev) {
  const int64_t rows = (int64_t)a.B * a.H * a.N * kD;
  CUtensorMap tmQ, tmK, tmV, tmOut, tmNode;
  if (!make_tokens_map(&tmQ, a.q, a.B, a.T, a.H) || !make_tokens_map(&tmK, a.k, a.B, a.T, a.H) ||
      !make_tokens_map(&tmV, a.v, a.B, a.T, a.H) ||
      !make_tokens_map(&tmOut, a.out, a.B, a.T, a.H) || !make_rows_map(&tmNode, a.nodes, rows))
    return cudaErrorInvalidValue;
  TcParams p;
  p.B = a.B; p.T = a.T; p.H = a.H; p.L = a.L; p.N = a.N;
  p.log_a = a.log_a; p.lam = a.lam; p.out = a.out; p.lg = a.lg;
  p.nodes = static_cast<uint8_t*>(a.nodes);
  p.odd = static_cast<uint8_t*>(a.U);
  p.blg = a.blg;
  p.cnt = a.cnt;
  p.out_f32 = out_dtype == LL_F32;
  int levels = 0;  // inter-chunk levels a tile can have: bit length of N-1
  while ((int64_t(1) << levels) < a.N) ++levels;
  cudaError_t e;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(tc_chunk_state_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemK1);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(tc_intra_readout_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem_k3(kMaxChunkLevels - 1));
  });
  if (attr_err != cudaSuccess) return attr_err;
  const dim3 grid(a.N, a.H, a.B);
  if (ev && (e = ev->record(s)) != cudaSuccess) return e;
  // the pair arrival counters start at zero in every call
  if ((e = cudaMemsetAsync(a.cnt, 0, sizeof(uint32_t) * (size_t)a.B * a.H * a.N, s)) !=
      cudaSuccess)
    return e;
  tc_chunk_state_kernel<<<grid, kThreads, kSmemK1, s>>>(tmK, tmV, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (ev && (e = ev->record(s)) != cudaSuccess) return e;
  tc_intra_readout_kernel<<<grid, kThreads3, smem_k3(levels), s>>>(tmQ, tmK, tmV, tmNode,
                                                                     tmOut, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (ev && (e = ev->record(s)) != cudaSuccess) return e;
  return ev ? ev->finish(s) : cudaSuccess;
}

cudaError_t tc_take_error(cudaStream_t s, unsigned* flags) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_tc_error, sizeof(v), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && v) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbolAsync(g_tc_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  *flags = v;
  return e;
}

}  // namespace ll

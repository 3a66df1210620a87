// Backward, dQ and dlambda, on the 5th-generation tensor cores (tcgen05 + TMEM + TMA):
// bf16 q, k, v and dO with fp32 accumulation, d_k = 128, d_v = 64 or 128, 128-token tiles.
//
// With A = Q K^T, M[t, s] = exp(cum_t - cum_s) lambda[t, l(t, s)] (s <= t) and dA = dO V^T
// (page "算力终结者来了！…", sections 结构矩阵 and 讨论与局限性: the backward needs the
// lambda gradients besides the attention ones):
//   dQ = (dA ⊙ M) K,
//   dlambda[t, l] = sum over the level-l bucket of t of exp(cum_t - cum_s) dA[t, s] A[t, s].
// Through the chunked decomposition with the 128-token tile as the chunk (page "论文阅读：
// Log-Linear Attention", sections 矩阵分解 and 两阶段计算):
//   * inside the tile both products are dense: S = Q K^T and S' = dO V^T go to TMEM;
//     P' = S' ⊙ M is written to shared memory in bf16 while the dlambda bucket sums of
//     exp(...) S' S are formed; dQ = P' K;
//   * for every set bit m-1 of the tile index j, the block state Tot of slot
//     c_m = (j >> (m-1)) << (m-1) (d_k x d_v) gives X = dO Tot^T, and
//       dQ_t += lambda[t, 7+m] exp(cs_t + D_m) X_t,
//       dlambda[t, 7+m] = exp(cs_t + D_m) q_t . X_t,
//     D_m being the log decay from the block's end to the tile's start.
// The block states are the ones a completed tensor-core forward over the same inputs left
// in its workspace (tile states, the even slots' block states, their log decays), so no
// CTA waits on another.  One CTA per tile, 8 warps (warps w and w+4 share TMEM lane
// quarter w mod 4 and split the columns), 512 TMEM columns, one CTA per SM.  Every
// mbarrier wait is bounded; a CTA whose wait times out sets g_tcb_error, skips what
// depends on it, frees TMEM and exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "ll_internal.cuh"
#include "tc_ptx.cuh"

namespace ll {

__device__ unsigned int g_tcb_error = 0;

namespace {

using namespace tc;

constexpr int kTile = 128;                  // tokens per tile (= MMA M)
constexpr int kD = 128;                     // d_k
constexpr int kPanel = kTile * 64 * 2;      // one [128][64] bf16 panel: 16 KiB
constexpr int kOperand = 2 * kPanel;        // a 128 x 128 bf16 tile: 32 KiB
constexpr int kThreadsB = 256;
constexpr int kIntra = 8;                   // levels inside a 128-token tile: 0..7
constexpr int kLamStride = 9;
constexpr int kTileLc = 7;
constexpr int kMaxChunkLevels = 32;

// The tile a CTA on this SM most likely takes next: one CTA per SM and tiles started in
// index order make it this tile + the number of SMs (`ahead`).  Its coordinates, or false
// when there is none.
struct TileAt {
  int b, h, hq, t0;
};

__device__ __forceinline__ bool next_tile(int ahead, int B, int T, int H, int hg, TileAt* t) {
  const int64_t nt = (int64_t)blockIdx.x + ahead;
  if (ahead <= 0 || nt >= (int64_t)gridDim.x) return false;
  const int BH = B * H;
  const int j = (int)(nt / BH), bhi = (int)(nt - (int64_t)j * BH);
  t->b = bhi / H;
  t->h = bhi - t->b * H;
  t->hq = t->h / hg;
  t->t0 = j * 128;
  return t->t0 < T;
}

struct BqParams {
  int B, T, H, hg, L, N;
  const float* log_a;
  const float* lam;
  const float* lgu;    // [B*H][N] the tiles' log decays (forward workspace)
  const float* nlg;    // [B*H][N] the even slots' block log decays (forward workspace)
  float* dqh;          // [B, T, Hqk, 128] fp32 dQ of each q/k head, added to with atomics
                       // by the hg heads that share it (zeroed before), or null
  const void* dq;      // non-null: dQ in bf16 through the dQ map (one q/k per head)
  float* dcq;          // [B, T, H] q . dQ, or null
  float* dlam;         // [B, T, H, L]
  int ahead;  // tiles between this one and the next on the same SM
  const uint32_t* tag;  // the forward workspace's layout tag, and the value it must have
  uint32_t tag_value;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Warms L2 with the box of a 4-d tensor map at (c0, c1, c2, c3), as tma_load_4d would read
// it; no shared memory, no completion signal.
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap* map, int c0, int c1, int c2,
                                                int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

// 32 fp32 values as bf16 into columns [32c, 32c+32) of row r of a tile of 128-byte
// swizzled [128][64] panels (the layout of a tokens map's TMA loads and stores).
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

// Columns [32c, 32c+32) of row r of a swizzled bf16 tile, as fp32.
__device__ __forceinline__ void get_row32(const uint8_t* buf, int r, int c, float* v) {
  const uint8_t* panel = buf + (c >> 1) * kPanel;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 w = *reinterpret_cast<const uint4*>(panel + sw128_offset(r, (c & 1) * 4 + q));
    const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
      v[8 * q + 2 * e] = f.x;
      v[8 * q + 2 * e + 1] = f.y;
    }
  }
}

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

struct BSmem {
  // byte offsets from the 1024-aligned base
  static constexpr int kQ = 0, kK = kOperand, kV = 2 * kOperand, kG = 3 * kOperand;
  static constexpr int kBars = 4 * kOperand;                   // 9 mbarriers
  static constexpr int kTslot = kBars + 12 * 8;
  static constexpr int kRed = kTslot + 16;                     // 8 floats
  static constexpr int kLg = kRed + 32;                        // 4 floats
  static constexpr int kNl = kLg + 16;                         // kMaxChunkLevels floats
  static constexpr int kCs = kNl + 4 * kMaxChunkLevels;        // 128 floats
  static constexpr int kFcol = kCs + 4 * kTile;                // 128 floats
  static constexpr int kLam = kFcol + 4 * kTile;               // [128][kLamStride] floats
  static constexpr int kDlb = kLam + 4 * kTile * kLamStride;   // [2][128][8] floats
  static constexpr int kLamX = kDlb + 4 * 2 * kTile * kIntra;  // [levels][128] floats
};

// ... then [levels][128] floats of inter-level dlambda sums after LamX
size_t smem_bwd_dq(int levels) {
  return (size_t)BSmem::kLamX + 2 * 4 * (size_t)kTile * levels + 1024;
}

template <int DV>
__global__ void __launch_bounds__(kThreadsB, 1)
    tc_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                     const __grid_constant__ CUtensorMap tmU,
                     const __grid_constant__ CUtensorMap tmNode,
                     const __grid_constant__ CUtensorMap tmDQ, BqParams p, int levels) {
  constexpr int kPanels = DV / 64;
  constexpr int kVBytes = kTile * DV * 2;
  constexpr int kStateBytes = kD * DV * 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* Qb = smem + BSmem::kQ;    // Q (S, then the q . X dots)
  uint8_t* Kb = smem + BSmem::kK;    // K (S, then dQ = P' K), then block states
  uint8_t* Vb = smem + BSmem::kV;    // V (S'), then P', then block states
  uint8_t* Gb = smem + BSmem::kG;    // dO (S' and the level MMAs)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BSmem::kBars);
  uint64_t* bar_load = &bars[0];
  uint64_t* bar_s = &bars[1];
  uint64_t* bar_dq = &bars[2];
  uint64_t* bar_lvl = &bars[3];      // [2]
  uint64_t* bar_node = &bars[5];     // [2]
  uint64_t* bar_free = &bars[7];     // [2]
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + BSmem::kTslot);
  float* red = reinterpret_cast<float*>(smem + BSmem::kRed);
  float* lg_s = reinterpret_cast<float*>(smem + BSmem::kLg);
  float* nl_s = reinterpret_cast<float*>(smem + BSmem::kNl);
  float* cs_s = reinterpret_cast<float*>(smem + BSmem::kCs);
  float* fcol = reinterpret_cast<float*>(smem + BSmem::kFcol);
  float* lam_s = reinterpret_cast<float*>(smem + BSmem::kLam);
  float* dlb = reinterpret_cast<float*>(smem + BSmem::kDlb);
  // the block states come from a tensor-core forward of exactly these sizes, or the
  // results are not valid: bit 2 of the error word says so
  if (blockIdx.x == 0 && threadIdx.x == 0 && (!p.tag || *p.tag != p.tag_value))
    atomicOr(&g_tcb_error, 4u);
  float* lamx = reinterpret_cast<float*>(smem + BSmem::kLamX);
  float* dli = lamx + levels * kTile;  // [levels][128] q . X sums of the inter levels

  const int tid = threadIdx.x, warp = tid >> 5;
  const int qt = warp & 3, hh = warp >> 2;
  const int r = tid & (kTile - 1);
  const int BH = p.B * p.H;
  const int j = blockIdx.x / BH, bhi = blockIdx.x - j * BH;  // tile j of every (b, h) in turn
  const int b = bhi / p.H, h = bhi - b * p.H, hq = h / p.hg;
  const int64_t N = p.N, bh = bhi;
  const int t0 = j * kTile;
  const int n = min(kTile, p.T - t0);
  const int64_t row = ((int64_t)b * p.T + t0 + r) * p.H + h;
  const int nlev = __popc((unsigned)j);
  const bool row_live = r < n;

  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  if (tid == 64) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    prefetch_tensormap(&tmG);
    prefetch_tensormap(&tmU);
    prefetch_tensormap(&tmNode);
    for (int q = 0; q < 7; ++q) mbar_init(&bars[q], 1);
    mbar_init(&bar_free[0], kThreadsB / 32);
    mbar_init(&bar_free[1], kThreadsB / 32);
    tslot[1] = tslot[2] = 0;  // block-state loads issued into Vb and Kb
    fence_mbar_init();
  }
  for (int i = tid; i < 2 * kTile * kIntra; i += kThreadsB) dlb[i] = 0.f;
  for (int i = tid; i < levels * kTile; i += kThreadsB) dli[i] = 0.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t lane_base = (uint32_t)(qt * 32) << 16;
  bool landed = true;
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_load, 2 * kOperand + 2 * kVBytes);
    tma_load_4d(&tmQ, bar_load, Qb, 0, hq, t0, b);
    tma_load_4d(&tmQ, bar_load, Qb + kPanel, 64, hq, t0, b);
    tma_load_4d(&tmK, bar_load, Kb, 0, hq, t0, b);
    tma_load_4d(&tmK, bar_load, Kb + kPanel, 64, hq, t0, b);
#pragma unroll
    for (int pv = 0; pv < kPanels; ++pv) {
      tma_load_4d(&tmV, bar_load, Vb + pv * kPanel, 64 * pv, h, t0, b);
      tma_load_4d(&tmG, bar_load, Gb + pv * kPanel, 64 * pv, h, t0, b);
    }
    TileAt nx;  // warm L2 with the next tile's operands
    if (next_tile(p.ahead, p.B, p.T, p.H, p.hg, &nx)) {
      tma_prefetch_4d(&tmQ, 0, nx.hq, nx.t0, nx.b);
      tma_prefetch_4d(&tmQ, 64, nx.hq, nx.t0, nx.b);
      tma_prefetch_4d(&tmK, 0, nx.hq, nx.t0, nx.b);
      tma_prefetch_4d(&tmK, 64, nx.hq, nx.t0, nx.b);
#pragma unroll
      for (int pv = 0; pv < kPanels; ++pv) {
        tma_prefetch_4d(&tmV, 64 * pv, nx.h, nx.t0, nx.b);
        tma_prefetch_4d(&tmG, 64 * pv, nx.h, nx.t0, nx.b);
      }
    }
  }
  __syncwarp();

  // per-row data: log a, the intra-tile lambdas (levels 0..7, split between the row's two
  // threads), the inter-level lambdas
  const float la = (hh == 0 && p.log_a && row_live) ? p.log_a[row] : 0.f;
  float lam_in[kIntra / 2];
#pragma unroll
  for (int i = 0; i < kIntra / 2; ++i) {
    const int l = hh * (kIntra / 2) + i;
    lam_in[i] = (row_live && l < p.L) ? p.lam[row * p.L + l] : 0.f;
  }
  {
    int k = 0;
    for (int m = 1; m < kMaxChunkLevels; ++m) {
      if (!((j >> (m - 1)) & 1)) continue;
      if ((k & 1) == hh)  // copied in the background: read only after the dQ MMA
        cp_async4(&lamx[k * kTile + r], row_live ? p.lam + row * p.L + kTileLc + m : p.lam,
                  row_live ? 4u : 0u);
      ++k;
    }
  }
  if (tid == 0) {  // S = Q K^T and S' = dO V^T as soon as the tiles land
    landed = mbar_wait(bar_load, 0);
    if (landed) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16(128, 128, 0, 0);
      const uint32_t qa = smem_u32(Qb), ka = smem_u32(Kb), ga = smem_u32(Gb), va = smem_u32(Vb);
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
        mma_bf16(tmem, smem_desc_sw128(qa + off, 16, 1024), smem_desc_sw128(ka + off, 16, 1024),
                 idesc, kk > 0);
      }
#pragma unroll
      for (int kk = 0; kk < DV / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
        mma_bf16(tmem + 128, smem_desc_sw128(ga + off, 16, 1024),
                 smem_desc_sw128(va + off, 16, 1024), idesc, kk > 0);
      }
      mma_commit(bar_s);
    }
  }
  const float cs_scan = block_scan256(la, red);
  if (hh == 0) cs_s[r] = cs_scan;
  if (tid == kTile - 1) lg_s[0] = cs_scan;
#pragma unroll
  for (int i = 0; i < kIntra / 2; ++i)
    lam_s[r * kLamStride + hh * (kIntra / 2) + i] = lam_in[i];
  __syncthreads();
  const float cs = cs_s[r];
  if (hh == 1) fcol[r] = __expf(cs_s[r | 31] - cs);

  bool all_ok = __syncthreads_and(landed);
  bool ok = all_ok && mbar_wait(bar_s, 0);
  tc_fence_after();
  all_ok = __syncthreads_and(ok);

  // the levels' block states: slot c_m holds U_{c-1} for odd c, the even block state else
  int my_c = 0;
  {
    const int k = tid - 32;
    if (k >= 0 && k < nlev) {
      int m = 0;
      for (int seen = -1; seen < k;) {
        ++m;
        if ((j >> (m - 1)) & 1) ++seen;
      }
      my_c = (j >> (m - 1)) << (m - 1);
      nl_s[k] = (my_c & 1) ? p.lgu[bh * N + my_c - 1] : p.nlg[bh * N + my_c];
    }
  }
  auto fetch = [&](int k) {  // thread 32+k: TMA of level k's block state into (k odd ? Kb : Vb)
    if (tid == 32 + k) {
      uint8_t* dst = (k & 1) ? Kb : Vb;
      const bool is_u = (my_c & 1) != 0;
      const int row0 = (int)((bh * N + (is_u ? my_c - 1 : my_c)) * kD);
      atomicAdd(&tslot[1 + (k & 1)], 1u);
      mbar_arrive_expect_tx(&bar_node[k & 1], kStateBytes);
#pragma unroll
      for (int pv = 0; pv < kPanels; ++pv)
        tma_load_2d(is_u ? &tmU : &tmNode, &bar_node[k & 1], dst + pv * kPanel, 64 * pv, row0);
    }
  };
  // V's tile is free (S' is done): the lowest level's block state loads now
  if (all_ok && nlev > 0) fetch(0);
  __syncwarp();

  // ---- P' = S' ⊙ M (bf16, two per column, into TMEM columns 384..447: chunk c of row r at
  // [384 + 16c, +16)) and the intra-tile dlambda bins sum_s exp(cs_t - cs_s) S'[t, s]
  // S[t, s] per level; chunk c of row r as in the forward
  float* bins = dlb + (hh * kTile + r) * kIntra;  // this thread's bins (private)
  if (all_ok) {
    const float* lam_r = lam_s + r * kLamStride;
    for (int c = hh; c < kTile / 32; c += 2) {
      if (c > qt) {
        uint32_t pz[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pz[e] = 0u;
        tmem_st16(tmem + lane_base + 384 + 16 * c, pz);
        continue;
      }
      float sp[32], sa[32];
      tmem_ld32(tmem + lane_base + 128 + c * 32, sp);
      tmem_ld32(tmem + lane_base + c * 32, sa);
      if (c < qt) {  // one level for the whole chunk: 5 + bit_length(qt XOR c)
        const int lvl = 5 + (32 - __clz((unsigned)(qt ^ c)));
        const float ge = __expf(cs - cs_s[c * 32 + 31]);
        const float wl = lam_r[lvl] * ge;
        float wsum = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float x = sp[k] * fcol[c * 32 + k];
          wsum = fmaf(x, sa[k], wsum);
          sp[k] = x * wl;
        }
        bins[lvl] += ge * wsum;
      } else if (cs_s[c * 32] - cs_s[c * 32 + 31] < 80.f) {
        // the diagonal chunk with a decay range that keeps exp(cs_t - cs_e) <= e^80: the
        // pair (r, s) has level bit_length(lane XOR k) <= 5 for column k <= lane, so the six
        // lambdas and dlambda bins of the levels inside a 32-token chunk stay in registers
        const int lane = tid & 31;
        const float gt = row_live ? __expf(cs - cs_s[c * 32 + 31]) : 0.f;
        const float l0 = lam_r[0], l1 = lam_r[1], l2 = lam_r[2], l3 = lam_r[3], l4 = lam_r[4],
                    l5 = lam_r[5];
        float b0 = 0.f, b1 = 0.f, b2 = 0.f, b3 = 0.f, b4 = 0.f, b5 = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int x = lane ^ k;
          const float xv = k <= lane ? sp[k] * (gt * fcol[c * 32 + k]) : 0.f;
          const float g = xv * sa[k];
          b5 += x >= 16 ? g : 0.f;
          b4 += (x >= 8 && x < 16) ? g : 0.f;
          b3 += (x >= 4 && x < 8) ? g : 0.f;
          b2 += (x >= 2 && x < 4) ? g : 0.f;
          b1 += x == 1 ? g : 0.f;
          b0 += x == 0 ? g : 0.f;
          sp[k] = xv * (x >= 16 ? l5 : x >= 8 ? l4 : x >= 4 ? l3 : x >= 2 ? l2 : x >= 1 ? l1 : l0);
        }
        bins[0] += b0;
        bins[1] += b1;
        bins[2] += b2;
        bins[3] += b3;
        bins[4] += b4;
        bins[5] += b5;
      } else {  // the diagonal chunk, any decay
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int s = c * 32 + k;
          float pv = 0.f;
          if (s <= r && row_live) {
            const int lvl = fenwick_level((uint32_t)r, (uint32_t)s);
            const float x = sp[k] * __expf(cs - cs_s[s]);
            bins[lvl] += x * sa[k];
            pv = x * lam_r[lvl];
          }
          sp[k] = pv;
        }
      }
      uint32_t pw[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) pw[e] = pack_bf16(sp[2 * e], sp[2 * e + 1]);
      tmem_st16(tmem + lane_base + 384 + 16 * c, pw);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  all_ok = __syncthreads_and(all_ok);
  // ---- dQ = P' K into TMEM columns 256..383 (P' from TMEM, K MN-major as B)
  if (all_ok && tid == 0) {
    tc_fence_after();
    constexpr uint32_t idesc = idesc_bf16(128, 128, 0, 1);
    const uint32_t ka = smem_u32(Kb);
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk)
      mma_bf16_ts(tmem + 256, tmem + 384 + 8 * kk, smem_desc_sw128(ka + kk * 2048, kPanel, 1024),
                  idesc, kk > 0);
    mma_commit(bar_dq);
  }
  __syncwarp();
  // the row's intra-tile dlambda (levels 0..7) and zeros for the levels above, which the
  // inter levels overwrite below (the same thread writes both)
  if (all_ok && hh == 0 && row_live) {
    for (int l = 0; l < p.L; ++l)
      p.dlam[row * p.L + l] = l < kIntra ? bins[l] + dlb[(kTile + r) * kIntra + l] : 0.f;
  }
  cp_async_wait_all();  // the inter-level lambdas (read after the barrier below)
  ok = all_ok && mbar_wait(bar_dq, 0);
  tc_fence_after();
  all_ok = __syncthreads_and(ok);
  if (all_ok && nlev > 1) fetch(1);  // K's tile is free (dQ's MMA is done)
  __syncwarp();

  // ---- dQ into registers: this thread's half row, d in [64 hh, 64 hh + 64)
  float dq[64];
#pragma unroll
  for (int q = 0; q < 64; ++q) dq[q] = 0.f;
  if (all_ok) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float v[32];
      tmem_ld32(tmem + lane_base + 256 + 64 * hh + c * 32, v);
#pragma unroll
      for (int q = 0; q < 32; ++q) dq[c * 32 + q] = v[q];
    }
  }
  tc_fence_before();
  __syncthreads();

  // ---- inter-tile levels (the forward's barrier-free loop): MMA k = dO Tot_k^T into TMEM
  // columns [128 (k & 1), +128); each warp adds level k-1 to dQ and its q . X to the
  // level's dlambda sum, then releases that TMEM buffer
  const int lane = tid & 31;
  uint32_t lvl_ph[2] = {0, 0}, node_ph[2] = {0, 0}, free_ph[2] = {0, 0};
  uint32_t used[2] = {0, 0};  // thread 0: block-state loads waited for, per buffer
  float D = 0.f;
  bool lv_ok = all_ok;
  for (int k = 0; k <= nlev && all_ok; ++k) {
    if (tid == 0 && k < nlev) {
      bool go = lv_ok && mbar_wait(&bar_node[k & 1], node_ph[k & 1]);
      if (go) ++used[k & 1];
      node_ph[k & 1] ^= 1;
      if (k >= 2) {
        go = go && mbar_wait(&bar_free[k & 1], free_ph[k & 1]);
        free_ph[k & 1] ^= 1;
      }
      if (go) {
        tc_fence_after();
        // A = dO (K-major over d_v), B = the block state [d_k][d_v] (K-major: N = d_k)
        constexpr uint32_t idesc = idesc_bf16(128, 128, 0, 0);
        const uint32_t ga = smem_u32(Gb), sa = smem_u32((k & 1) ? Kb : Vb);
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          mma_bf16(tmem + (k & 1) * 128, smem_desc_sw128(ga + off, 16, 1024),
                   smem_desc_sw128(sa + off, 16, 1024), idesc, kk > 0);
        }
        mma_commit(&bar_lvl[k & 1]);
      }
      lv_ok = go;
    }
    __syncwarp();
    if (k >= 1) {
      const int bf = (k - 1) & 1;
      const bool got = __all_sync(0xffffffffu, mbar_wait(&bar_lvl[bf], lvl_ph[bf]));
      lvl_ph[bf] ^= 1;
      if (!got) {
        lv_ok = false;
        break;
      }
      tc_fence_after();
      if (k + 1 < nlev) fetch(k + 1);  // into the buffer MMA k-1 has finished reading
      const float e = __expf(cs + D);
      const float wl = lamx[(k - 1) * kTile + r] * e;
      D += nl_s[k - 1];
      float dot = 0.f;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float v[32], qv[32];
        tmem_ld32(tmem + lane_base + bf * 128 + 64 * hh + c * 32, v);
        get_row32(Qb, r, 2 * hh + c, qv);
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          dq[c * 32 + q] = fmaf(wl, v[q], dq[c * 32 + q]);
          dot = fmaf(qv[q], v[q], dot);
        }
      }
      atomicAdd(&dli[(k - 1) * kTile + r], e * dot);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_free[bf]);
    }
  }
  all_ok = __syncthreads_and(all_ok && lv_ok);

  // ---- epilogue: the inter-level dlambda, dQ (fp32), and q . dQ = sum_l lambda[t, l]
  // dlambda[t, l] (O is linear in each row's lambdas), which takes q . dQ from the fp32
  // products S and S' rather than from dQ, whose P' was rounded to bf16
  if (all_ok) {
    if (hh == 0 && row_live) {
      const float* lam_r = lam_s + r * kLamStride;
      float qd = 0.f;
#pragma unroll
      for (int l = 0; l < kIntra; ++l)
        qd = fmaf(lam_r[l], dlb[r * kIntra + l] + dlb[(kTile + r) * kIntra + l], qd);
      int k = 0;
      for (int m = 1; m < kMaxChunkLevels && k < nlev; ++m) {
        if (!((j >> (m - 1)) & 1)) continue;
        const float v = dli[k * kTile + r];
        p.dlam[row * p.L + kTileLc + m] = v;
        qd = fmaf(lamx[k * kTile + r], v, qd);
        ++k;
      }
      if (p.dcq) p.dcq[row] = qd;
    }
    if (p.dq) {  // no MMA reads Q any more: stage dQ there and store it with TMA
      put_row32_bf16(Qb, r, 2 * hh, dq);
      put_row32_bf16(Qb, r, 2 * hh + 1, dq + 32);
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {  // rows past T are clipped by the map
        tma_store_4d(&tmDQ, Qb, 0, h, t0, b);
        tma_store_4d(&tmDQ, Qb + kPanel, 64, h, t0, b);
        tma_store_commit();
        tma_store_wait_read();
      }
    } else if (row_live) {  // shared q/k: this head's part of its group's dQ
      float4* dst = reinterpret_cast<float4*>(
          p.dqh + (((int64_t)b * p.T + t0 + r) * (p.H / p.hg) + hq) * kD + 64 * hh);
#pragma unroll
      for (int q = 0; q < 16; ++q)
        atomicAdd(dst + q, make_float4(dq[4 * q], dq[4 * q + 1], dq[4 * q + 2], dq[4 * q + 3]));
    }
  } else if (tid == 0) {
    atomicOr(&g_tcb_error, 1u);
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && !all_ok) {
    // after an error: wait (bounded) for the block-state loads still in flight into this
    // CTA's shared memory before it is handed to another CTA
    for (int bf = 0; bf < 2; ++bf)
      for (uint32_t c = used[bf]; c < tslot[1 + bf]; ++c) mbar_wait(&bar_node[bf], c & 1);
  }
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ dK and dV
//
// Source s of tile i receives, from the queries t of its own tile,
//   dK_s = sum_t P'[t, s] q_t,  dV_s = sum_t P[t, s] dO_t   (P = M ⊙ S, P' = M ⊙ S'),
// i.e. dK = P'^T Q and dV = P^T dO with P and P' read MN-major as the A operand; and from
// the later tiles, through the mirrored states (fp32, accumulated by the kernel above),
// summed over the tile's levels into R_tot = sum_m exp(E_m) R_{c_m} (E_m: log decay of the tiles strictly
// between i and c_m):
//   dK_s += g_s R_tot v_s,  dV_s += g_s R_tot^T k_s,  g_s = exp(lg_i - cs_s),
// taken as MMAs V R_tot^T and K R_tot whose row s the epilogue scales by g_s (in fp32).
// k_s . dK_s, which d log a needs, is the column sum of G = M ⊙ S ⊙ S' (from the fp32 S
// and S') plus v_s . dV_inter.

struct BkvParams {
  int B, T, H, hg, L, N;
  const float* log_a;
  const float* lam;
  const float* lgu;          // [B*H][N] the tiles' log decays (forward workspace)
  const float* R;            // [B*H][N][d_k][d_v] mirrored states, fp32
  const __nv_bfloat16* v;    // [B, T, H, d_v] (for v . dV)
  float* dkh;                // [B, T, Hqk, 128] fp32 dK of each q/k head, added to with
                             // atomics by the hg heads that share it (zeroed before), or null
  const void* dk;            // non-null: dK in bf16 through the dK map (one q/k per head)
  float* dck;                // [B, T, H] k . dK, or null
};

struct KvSmem {
  static constexpr int kQ = 0, kK = kOperand, kV = 2 * kOperand, kG = 3 * kOperand;
  static constexpr int kP1 = 4 * kOperand;   // P' (dK), then R_tot
  static constexpr int kP0 = 5 * kOperand;   // P (dV)
  static constexpr int kBars = 6 * kOperand; // load, s, kv, inter
  static constexpr int kTslot = kBars + 8 * 8;
  static constexpr int kRed = kTslot + 16;
  static constexpr int kLg = kRed + 32;
  static constexpr int kCs = kLg + 16;                         // 128 floats
  static constexpr int kFcol = kCs + 4 * kTile;                // 128 floats
  static constexpr int kCol = kFcol + 4 * kTile;               // 128 floats: column sums of G
  static constexpr int kVd = kCol + 4 * kTile;                 // [2][128] floats
  static constexpr int kLvC = kVd + 4 * 2 * kTile;             // 32 ints: block starts
  static constexpr int kLvW = kLvC + 4 * kMaxChunkLevels;      // 32 floats: exp(E_m)
  static constexpr int kLvN = kLvW + 4 * kMaxChunkLevels;      // 1 int
  static constexpr int kLam = kLvN + 16;                       // [128][kLamStride] floats
  static constexpr int kEnd = kLam + 4 * kTile * kLamStride;
};

size_t smem_bwd_dkv() { return (size_t)KvSmem::kEnd + 1024; }

// Column sums of a 32 x 32 block held one row per lane: a transpose-reduce butterfly
// (31 shuffles); on return a[0] of lane k is the sum of column k over the warp's rows.
__device__ __forceinline__ void warp_column_sums(float (&a)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = up ? a[i] : a[i + o];
      const float keep = up ? a[i + o] : a[i];
      a[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
}

template <int DV>
__global__ void __launch_bounds__(kThreadsB, 1)
    tc_bwd_dkv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                      const __grid_constant__ CUtensorMap tmDK,
                      const __grid_constant__ CUtensorMap tmDV, BkvParams p) {
  constexpr int kPanels = DV / 64;
  constexpr int kVBytes = kTile * DV * 2;
  constexpr int kHalf = DV / 2;      // d_v columns per thread
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* Qb = smem + KvSmem::kQ;
  uint8_t* Kb = smem + KvSmem::kK;
  uint8_t* Vb = smem + KvSmem::kV;
  uint8_t* Gb = smem + KvSmem::kG;
  uint8_t* P1 = smem + KvSmem::kP1;  // P', then R_tot, then the bf16 dK tile
  uint8_t* P0 = smem + KvSmem::kP0;  // P, then the bf16 dV tile
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + KvSmem::kBars);
  uint64_t* bar_qg = &bars[0];       // Q and dO of a tile landed
  uint64_t* bar_kv_in = &bars[1];    // K and V of a tile landed
  uint64_t* bar_s = &bars[2];
  uint64_t* bar_kv = &bars[3];
  uint64_t* bar_inter = &bars[4];
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + KvSmem::kTslot);
  float* red = reinterpret_cast<float*>(smem + KvSmem::kRed);
  float* lg_s = reinterpret_cast<float*>(smem + KvSmem::kLg);
  float* cs_s = reinterpret_cast<float*>(smem + KvSmem::kCs);
  float* fcol = reinterpret_cast<float*>(smem + KvSmem::kFcol);
  float* colsum = reinterpret_cast<float*>(smem + KvSmem::kCol);
  float* vd_s = reinterpret_cast<float*>(smem + KvSmem::kVd);
  int* lv_c = reinterpret_cast<int*>(smem + KvSmem::kLvC);
  float* lv_w = reinterpret_cast<float*>(smem + KvSmem::kLvW);
  int* lv_n = reinterpret_cast<int*>(smem + KvSmem::kLvN);
  float* lam_s = reinterpret_cast<float*>(smem + KvSmem::kLam);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = warp & 3, hh = warp >> 2;
  const int r = tid & (kTile - 1);
  const int BH = p.B * p.H;
  const int64_t tiles = (int64_t)BH * p.N;
  const int64_t elems = (int64_t)kD * DV;

  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  if (tid == 64) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    prefetch_tensormap(&tmG);
    prefetch_tensormap(&tmDK);
    prefetch_tensormap(&tmDV);
    for (int q = 0; q < 5; ++q) mbar_init(&bars[q], 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t lane_base = (uint32_t)(qt * 32) << 16;

  // Thread 0 loads a tile's operands in two halves: Q and dO once dK's and dV's MMAs of the
  // tile before are done with them, K and V once its inter MMAs are (both ahead of the
  // epilogue, so the loads overlap it).
  auto coords = [&](int64_t t, int* b, int* h, int* hq, int* t0) {
    const int i = (int)(t / BH), bhi = (int)(t - (int64_t)i * BH);
    *b = bhi / p.H;
    *h = bhi - *b * p.H;
    *hq = *h / p.hg;
    *t0 = i * kTile;
  };
  auto load_qg = [&](int64_t t) {
    int b, h, hq, t0;
    coords(t, &b, &h, &hq, &t0);
    mbar_arrive_expect_tx(bar_qg, kOperand + kVBytes);
    tma_load_4d(&tmQ, bar_qg, Qb, 0, hq, t0, b);
    tma_load_4d(&tmQ, bar_qg, Qb + kPanel, 64, hq, t0, b);
#pragma unroll
    for (int pv = 0; pv < kPanels; ++pv) tma_load_4d(&tmG, bar_qg, Gb + pv * kPanel, 64 * pv, h, t0, b);
  };
  auto load_kv = [&](int64_t t) {
    int b, h, hq, t0;
    coords(t, &b, &h, &hq, &t0);
    mbar_arrive_expect_tx(bar_kv_in, kOperand + kVBytes);
    tma_load_4d(&tmK, bar_kv_in, Kb, 0, hq, t0, b);
    tma_load_4d(&tmK, bar_kv_in, Kb + kPanel, 64, hq, t0, b);
#pragma unroll
    for (int pv = 0; pv < kPanels; ++pv) tma_load_4d(&tmV, bar_kv_in, Vb + pv * kPanel, 64 * pv, h, t0, b);
  };
  int64_t tile = blockIdx.x;
  // thread 0: loads issued and not yet waited for (bit 0: Q and dO, bit 1: K and V), and
  // whether a TMA store may still be reading P0 / P1
  uint32_t in_flight = 0, flight_ph = 0;  // flight_ph: the phase those loads complete
  bool store_pending = false;
  if (tid == 0 && tile < tiles) {
    load_qg(tile);
    load_kv(tile);
    in_flight = 3;
  }
  uint32_t ph = 0;        // phase of every per-tile barrier: one completion per tile
  uint32_t ph_inter = 0;  // bar_inter completes only for tiles with levels
  bool all_ok = true;
  for (; tile < tiles && all_ok; tile += gridDim.x, ph ^= 1) {
    const int64_t next = tile + gridDim.x;
    const int i = (int)(tile / BH), bhi = (int)(tile - (int64_t)i * BH);
    const int b = bhi / p.H, h = bhi - b * p.H, hq = h / p.hg;
    const int64_t bh = bhi;
    const int t0 = i * kTile;
    const int n = min(kTile, p.T - t0);
    const int64_t row = ((int64_t)b * p.T + t0 + r) * p.H + h;
    const bool row_live = r < n;

    // ---- the tile's levels and their weights (while its operands land)
    if (tid < kTile) colsum[tid] = 0.f;
    if (warp == 2) {  // the tile's levels: blocks of later tiles, with exp(E_m)
      int nl = 0;
      int64_t cmax = i + 1;
      for (int m = 1; (int64_t(1) << (m - 1)) < p.N; ++m) {
        if ((i >> (m - 1)) & 1) continue;
        const int64_t c1 = (((int64_t)i >> (m - 1)) | 1) << (m - 1);
        if (c1 >= p.N) continue;
        if (lane == 0) lv_c[nl] = (int)c1;
        cmax = c1;  // c1 grows with m
        ++nl;
      }
      __syncwarp();
      // E_m = the log decays of tiles [i+1, c1_m): running prefix sums over 32 tiles a step,
      // read off at c1_m - 1 (one pass for all levels)
      int k = 0;
      for (; k < nl && lv_c[k] == i + 1; ++k)
        if (lane == 0) lv_w[k] = 1.f;
      float run = 0.f;
      for (int64_t base = i + 1; base < cmax; base += 32) {
        float x = base + lane < cmax ? p.lgu[bh * p.N + base + lane] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        for (; k < nl && lv_c[k] - 1 < base + 32; ++k) {
          const float E = run + __shfl_sync(0xffffffffu, x, (int)(lv_c[k] - 1 - base));
          if (lane == 0) lv_w[k] = __expf(E);
        }
        run += __shfl_sync(0xffffffffu, x, 31);
      }
      if (lane == 0) *lv_n = nl;
    }
    __syncthreads();
    const int nl = *lv_n;
    if (tid >= 32 && tid < 32 + nl)  // warm L2 with the mirrored states summed below
      prefetch_l2_bulk(p.R + (bh * p.N + lv_c[tid - 32]) * elems, (uint32_t)(elems * 4));
    const float la = (hh == 0 && p.log_a && row_live) ? p.log_a[row] : 0.f;
    float lam_in[kIntra / 2];
#pragma unroll
    for (int q = 0; q < kIntra / 2; ++q) {
      const int l = hh * (kIntra / 2) + q;
      lam_in[q] = (row_live && l < p.L) ? p.lam[row * p.L + l] : 0.f;
    }
    bool landed = true;
    if (tid == 0) {  // S = Q K^T, S' = dO V^T
      landed = mbar_wait(bar_qg, ph);
      if (landed) in_flight &= ~1u;
      landed = landed && mbar_wait(bar_kv_in, ph);
      if (landed) in_flight &= ~2u;
      if (landed) {
        tc_fence_after();
        constexpr uint32_t idesc = idesc_bf16(128, 128, 0, 0);
        const uint32_t qa = smem_u32(Qb), ka = smem_u32(Kb), ga = smem_u32(Gb), va = smem_u32(Vb);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          mma_bf16(tmem, smem_desc_sw128(qa + off, 16, 1024), smem_desc_sw128(ka + off, 16, 1024),
                   idesc, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          mma_bf16(tmem + 128, smem_desc_sw128(ga + off, 16, 1024),
                   smem_desc_sw128(va + off, 16, 1024), idesc, kk > 0);
        }
        mma_commit(bar_s);
      }
      // the previous tile's dK and dV stores read P0 and P1, which P and P' overwrite below
      if (store_pending) tma_store_wait_read();
      store_pending = false;
    }
    const float cs_scan = block_scan256(la, red);
    if (hh == 0) cs_s[r] = cs_scan;
    if (tid == kTile - 1) lg_s[0] = cs_scan;
#pragma unroll
    for (int q = 0; q < kIntra / 2; ++q) lam_s[r * kLamStride + hh * (kIntra / 2) + q] = lam_in[q];
    __syncthreads();
    const float cs = cs_s[r];
    const float lg = lg_s[0];
    if (hh == 1) fcol[r] = __expf(cs_s[r | 31] - cs);

    all_ok = __syncthreads_and(landed);
    bool ok = all_ok && mbar_wait(bar_s, ph);
    tc_fence_after();
    all_ok = __syncthreads_and(ok);

    // ---- P (into P0) and P' (into P1) for row r's chunks, the column sums of G; and the
    // rows of K and V scaled by g_r = exp(lg - cs_r) for the inter-tile MMAs (S and S' are
    // done with K and V)
    if (all_ok) {
      const float* lam_r = lam_s + r * kLamStride;
      for (int c = hh; c < kTile / 32; c += 2) {
        if (c > qt) {
          put_row32_zero(P0, r, c);
          put_row32_zero(P1, r, c);
          continue;
        }
        float sa[32], sp[32];
        tmem_ld32(tmem + lane_base + c * 32, sa);
        tmem_ld32(tmem + lane_base + 128 + c * 32, sp);
        if (c < qt) {
          const int lvl = 5 + (32 - __clz((unsigned)(qt ^ c)));
          const float wl = lam_r[lvl] * __expf(cs - cs_s[c * 32 + 31]);
          float g[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const float m = wl * fcol[c * 32 + k];
            g[k] = m * sa[k] * sp[k];
            sa[k] *= m;
            sp[k] *= m;
          }
          warp_column_sums(g);
          atomicAdd(&colsum[c * 32 + lane], g[0]);
        } else {
          float g[32];
          if (cs_s[c * 32] - cs_s[c * 32 + 31] < 80.f) {
            // the diagonal chunk with a decay range that keeps exp(cs_t - cs_e) <= e^80; the
            // pair (r, s) has level bit_length(lane XOR k) <= 5 for column k <= lane: the six
            // lambdas of the levels inside a 32-token chunk are picked from registers
            const float gt = row_live ? __expf(cs - cs_s[c * 32 + 31]) : 0.f;
            const float l0 = lam_r[0], l1 = lam_r[1], l2 = lam_r[2], l3 = lam_r[3],
                        l4 = lam_r[4], l5 = lam_r[5];
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const int x = lane ^ k;
              const float lv = x >= 16 ? l5 : x >= 8 ? l4 : x >= 4 ? l3 : x >= 2 ? l2 : x >= 1 ? l1 : l0;
              const float m = k <= lane ? lv * (gt * fcol[c * 32 + k]) : 0.f;
              g[k] = m * sa[k] * sp[k];
              sa[k] *= m;
              sp[k] *= m;
            }
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const int s = c * 32 + k;
              float m = 0.f;
              if (s <= r && row_live)
                m = lam_r[fenwick_level((uint32_t)r, (uint32_t)s)] * __expf(cs - cs_s[s]);
              g[k] = m * sa[k] * sp[k];
              sa[k] *= m;
              sp[k] *= m;
            }
          }
          warp_column_sums(g);
          atomicAdd(&colsum[c * 32 + lane], g[0]);
        }
        put_row32_bf16(P0, r, c, sa);
        put_row32_bf16(P1, r, c, sp);
      }
    }
    tc_fence_after();
    fence_proxy_async_smem();
    tc_fence_before();
    all_ok = __syncthreads_and(all_ok);
    // ---- dK = P'^T Q into TMEM 256..383, dV = P^T dO into 384..384+DV (A MN-major)
    if (all_ok && tid == 0) {
      tc_fence_after();
      constexpr uint32_t idk = idesc_bf16(128, 128, 1, 1);
      constexpr uint32_t idv = idesc_bf16(128, DV, 1, 1);
      const uint32_t p1 = smem_u32(P1), p0 = smem_u32(P0), qa = smem_u32(Qb), ga = smem_u32(Gb);
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) {
        mma_bf16(tmem + 256, smem_desc_sw128(p1 + kk * 2048, kPanel, 1024),
                 smem_desc_sw128(qa + kk * 2048, kPanel, 1024), idk, kk > 0);
        mma_bf16(tmem + 384, smem_desc_sw128(p0 + kk * 2048, kPanel, 1024),
                 smem_desc_sw128(ga + kk * 2048, kPanel, 1024), idv, kk > 0);
      }
      mma_commit(bar_kv);
    }
    __syncwarp();
    // ---- R_tot summed over the levels while the MMAs run (fp32 loads, a warp reads whole
    // rows: lane owns 4 consecutive columns, warp w rows w, w+8, ...), then written in bf16
    // over P' once dK's MMA is done with it
    constexpr int kLanesPerRow = DV / 4;             // 32 or 16
    constexpr int kRowsPerIter = 32 / kLanesPerRow;  // 1 or 2
    constexpr int kIters = kTile / 8 / kRowsPerIter; // 16 or 8
    const int lrow = lane / kLanesPerRow, col = 4 * (lane % kLanesPerRow);
    float4 rt[kIters];
#pragma unroll
    for (int it = 0; it < kIters; ++it) rt[it] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (all_ok) {
#pragma unroll 2
      for (int l = 0; l < nl; ++l) {
        const float w = lv_w[l];
        const float* src = p.R + (bh * p.N + (int64_t)lv_c[l]) * elems + col;
#pragma unroll
        for (int it = 0; it < kIters; ++it) {
          const int d = (it * kRowsPerIter + lrow) * 8 + warp;
          const float4 x = __ldcg(reinterpret_cast<const float4*>(src + (int64_t)d * DV));
          rt[it].x = fmaf(w, x.x, rt[it].x);
          rt[it].y = fmaf(w, x.y, rt[it].y);
          rt[it].z = fmaf(w, x.z, rt[it].z);
          rt[it].w = fmaf(w, x.w, rt[it].w);
        }
      }
    }
    ok = all_ok && mbar_wait(bar_kv, ph);
    tc_fence_after();
    all_ok = __syncthreads_and(ok);
    // Q and dO are free (the MMAs above were their last readers): the next tile's load now
    if (all_ok && tid == 0 && next < tiles) {
      load_qg(next);
      in_flight |= 1u;
      flight_ph = ph ^ 1;
    }
    if (all_ok && nl > 0) {
#pragma unroll
      for (int it = 0; it < kIters; ++it) {
        const int d = (it * kRowsPerIter + lrow) * 8 + warp;
        uint8_t* dst = P1 + (col >> 6) * kPanel + sw128_offset(d, (col & 63) >> 3) + (col & 7) * 2;
        *reinterpret_cast<uint2*>(dst) =
            make_uint2(pack_bf16(rt[it].x, rt[it].y), pack_bf16(rt[it].z, rt[it].w));
      }
    }
    tc_fence_after();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- dK_inter = V R_tot^T into TMEM 128..255 (B K-major: N = d_k) and dV_inter = K R_tot
    // into 0..DV (B MN-major: N = d_v), both freed by the P build; the epilogue scales row s
    // of both by g_s
    if (all_ok && nl > 0 && tid == 0) {
      tc_fence_after();
      constexpr uint32_t idk = idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idv = idesc_bf16(128, DV, 0, 1);
      const uint32_t ra = smem_u32(P1), va = smem_u32(Vb), ka = smem_u32(Kb);
#pragma unroll
      for (int kk = 0; kk < DV / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
        mma_bf16(tmem + 128, smem_desc_sw128(va + off, 16, 1024), smem_desc_sw128(ra + off, 16, 1024),
                 idk, kk > 0);
      }
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
        mma_bf16(tmem, smem_desc_sw128(ka + off, 16, 1024),
                 smem_desc_sw128(ra + kk * 2048, kPanel, 1024), idv, kk > 0);
      }
      mma_commit(bar_inter);
    }
    __syncwarp();
    if (nl > 0) {
      ok = all_ok && mbar_wait(bar_inter, ph_inter);
      ph_inter ^= 1;
      tc_fence_after();
      all_ok = __syncthreads_and(ok);
    }
    // K and V are free (and P1 holds no operand any more): the next tile's K and V now
    if (all_ok && tid == 0 && next < tiles) {
      load_kv(next);
      in_flight |= 2u;
      flight_ph = ph ^ 1;
    }
    // ---- epilogue: dK (bf16, or fp32 per head), dV = intra + inter (bf16), k . dK.  The
    // bf16 dK and dV tiles are staged in P1 and P0, which no MMA reads any more, and stored
    // by TMA; the next tile's Q, dO, K and V load meanwhile.
    if (all_ok) {
      uint4 vrow[kHalf / 8];  // this row's half of v, loaded first so its latency overlaps
      if (row_live) {
        const uint4* vsrc = reinterpret_cast<const uint4*>(p.v + row * DV + kHalf * hh);
#pragma unroll
        for (int q = 0; q < kHalf / 8; ++q) vrow[q] = vsrc[q];
      }
      float vd = 0.f;
      const float g = row_live && nl > 0 ? __expf(lg - cs) : 0.f;  // decay from row r to the end
      {
        float v0[32];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          tmem_ld32(tmem + lane_base + 256 + 64 * hh + 32 * c, v0);
          if (nl > 0) {
            float v1[32];
            tmem_ld32(tmem + lane_base + 128 + 64 * hh + 32 * c, v1);
#pragma unroll
            for (int q = 0; q < 32; ++q) v0[q] = fmaf(g, v1[q], v0[q]);
          }
          if (p.dk) {
            put_row32_bf16(P1, r, 2 * hh + c, v0);
          } else if (row_live) {  // shared q/k: this head's part of its group's dK
            float4* dst = reinterpret_cast<float4*>(
                p.dkh + (((int64_t)b * p.T + t0 + r) * (p.H / p.hg) + hq) * kD + 64 * hh + 32 * c);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              atomicAdd(dst + q, make_float4(v0[4 * q], v0[4 * q + 1], v0[4 * q + 2], v0[4 * q + 3]));
          }
        }
      }
#pragma unroll
      for (int c = 0; c < kPanels; ++c) {
        float a[32], x[32];
        tmem_ld32(tmem + lane_base + 384 + kHalf * hh + 32 * c, a);
        if (nl > 0) {
          tmem_ld32(tmem + lane_base + kHalf * hh + 32 * c, x);
#pragma unroll
          for (int q = 0; q < 32; ++q) x[q] *= g;
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q) x[q] = 0.f;
        }
        if (row_live) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 w = vrow[4 * c + q];
            const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
              vd = fmaf(f.x, x[8 * q + 2 * e], vd);
              vd = fmaf(f.y, x[8 * q + 2 * e + 1], vd);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < 32; ++q) a[q] += x[q];
        put_row32_bf16(P0, r, kPanels * hh + c, a);
      }
      vd_s[hh * kTile + r] = vd;
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {  // rows past T are clipped by the maps
        if (p.dk) {
          tma_store_4d(&tmDK, P1, 0, h, t0, b);
          tma_store_4d(&tmDK, P1 + kPanel, 64, h, t0, b);
        }
#pragma unroll
        for (int pv = 0; pv < kPanels; ++pv) tma_store_4d(&tmDV, P0 + pv * kPanel, 64 * pv, h, t0, b);
        tma_store_commit();
        store_pending = true;
      }
      if (hh == 0 && row_live && p.dck)
        p.dck[row] = colsum[r] + vd_s[r] + vd_s[kTile + r];
    } else if (tid == 0) {
      atomicOr(&g_tcb_error, 1u);
    }
    tc_fence_before();
    __syncthreads();  // TMEM, colsum and vd_s are read: the next tile may overwrite them
  }
  if (tid == 0) {
    // the stores must finish reading shared memory, and after an error the loads still in
    // flight into it must land (bounded waits), before it is handed to another CTA
    if (store_pending) tma_store_wait_read();
    if (in_flight & 1u) mbar_wait(bar_qg, flight_ph);
    if (in_flight & 2u) mbar_wait(bar_kv_in, flight_ph);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ mirrored states
//
// The sources of tiles [c - 2^z, c) (z = ctz(c)) meet the queries of tiles [c, c + 2^z)
// at chunk level m = z + 1 (Fenwick level 7 + m).  Their mirrored state is
//   R_c = sum_{j in [c, c + 2^z)} sum_{t in j} w_t q_t dO_t^T,
//   w_t = exp(cs_t + D_j) lambda[t, 7+m],  D_j = log decay of the tiles [c, j).
// One CTA takes one slot c and a run of at most 2^kRunLog of its reader tiles and sums
// the run's products in one TMEM accumulator: per reader tile, Q and dO by TMA, the rows
// of Q scaled by w in place and split into a bf16 high part and a bf16 residual (w q to
// about 16 bits; dO is exact in bf16), and (w Q)^T dO = hi^T dO + lo^T dO (A and B
// MN-major).  The states feed k . dK, and with it d log a, a sum whose terms cancel,
// which is why w q is not rounded to bf16 alone.  The accumulator is staged in shared
// memory and goes to R_c with coalesced stores when the run is the slot's only one
// (z <= kRunLog), else with float4 atomics into the slot, zeroed before.  Two CTAs fit
// per SM, so one run's loads overlap the other's products.
//
// Runs: those of level z cover the reader tiles j with bit z set, in aligned runs of
// g = 2^min(z, kRunLog) tiles.  Their starts are s = q g for the q in [0, ceil(N / g))
// whose bit z - log2(g) is set.  The grid takes the runs level by level from the highest
// (the longest runs first), the (b, h) innermost.

constexpr int kRunLog = 5;

// How many q in [0, M) have bit b set.
__host__ __device__ inline int64_t count_with_bit(int64_t M, int b) {
  const int64_t full = (M >> (b + 1)) << b;
  const int64_t rem = (M & ((int64_t(2) << b) - 1)) - (int64_t(1) << b);
  return full + (rem > 0 ? rem : 0);
}

// Runs of level z for N tiles.
__host__ __device__ inline int64_t runs_at_level(int64_t N, int z) {
  const int lg = z < kRunLog ? z : kRunLog;
  return count_with_bit((N + (int64_t(1) << lg) - 1) >> lg, z - lg);
}

struct BrParams {
  int B, T, H, hg, L, N;
  int levels;          // chunk levels holding slots: the bit length of N - 1
  const float* log_a;
  const float* lam;
  const float* lgu;    // [B*H][N] the tiles' log decays (forward workspace)
  float* R;            // [B*H][N][d_k][d_v] mirrored states (slots with z > kRunLog zeroed before)
};

struct RsSmem {
  // Q (then its scaled high part), the residual, dO; the accumulator is staged over Q and
  // the residual at the end
  static constexpr int kQ = 0, kLo = kOperand, kG = 2 * kOperand;
  static constexpr int kBars = 3 * kOperand;  // load, mma
  static constexpr int kTslot = kBars + 2 * 8;
  static constexpr int kRed = kTslot + 16;    // 8 floats
  static constexpr int kD0 = kRed + 32;       // 4 floats
  static constexpr int kCs = kD0 + 16;        // 128 floats
  static constexpr int kEnd = kCs + 4 * kTile;
};

size_t smem_bwd_rstate() { return (size_t)RsSmem::kEnd + 1024; }

template <int DV>
__global__ void __launch_bounds__(kThreadsB, 2)
    tc_bwd_rstate_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmG, BrParams p) {
  constexpr int kPanels = DV / 64;
  constexpr int kVBytes = kTile * DV * 2;
  constexpr int kHalf = DV / 2;
  const int BH = p.B * p.H;

  // ---- the run
  int64_t e = (int64_t)blockIdx.x / BH;
  const int bhi = (int)((int64_t)blockIdx.x - e * BH);
  int z = p.levels - 1;
  for (; z > 0; --z) {
    const int64_t cnt = runs_at_level(p.N, z);
    if (e < cnt) break;
    e -= cnt;
  }
  const int lgr = z < kRunLog ? z : kRunLog;
  const int bq = z - lgr;
  const int64_t q = ((e >> bq) << (bq + 1)) | (int64_t(1) << bq) | (e & ((int64_t(1) << bq) - 1));
  const int s0 = (int)(q << lgr);               // the run's first reader tile
  const int c = (s0 >> z) << z;                 // its slot
  const int s1 = min(s0 + (1 << lgr), p.N);     // one past its last reader tile
  const bool whole = z <= kRunLog;              // the run is the slot's only one
  const int lam_l = kTileLc + z + 1;            // the Fenwick level of the run's pairs

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* Qb = smem + RsSmem::kQ;
  uint8_t* Lb = smem + RsSmem::kLo;
  uint8_t* Gb = smem + RsSmem::kG;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + RsSmem::kBars);
  uint64_t* bar_load = &bars[0];
  uint64_t* bar_mma = &bars[1];
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + RsSmem::kTslot);
  float* red = reinterpret_cast<float*>(smem + RsSmem::kRed);
  float* d0_s = reinterpret_cast<float*>(smem + RsSmem::kD0);
  float* cs_s = reinterpret_cast<float*>(smem + RsSmem::kCs);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = warp & 3, hh = warp >> 2;
  const int r = tid & (kTile - 1);
  const int b = bhi / p.H, h = bhi - b * p.H, hq = h / p.hg;
  const int64_t bh = bhi;

  if (warp == 1) {
    tmem_alloc(tslot, 128);
    tmem_relinquish();
  }
  if (tid == 64) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmG);
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t lane_base = (uint32_t)(qt * 32) << 16;

  // thread 0: Q and dO of reader tile j by TMA, and the next reader's boxes into L2
  auto issue_loads = [&](int j) {
    const int t0 = j * kTile;
    mbar_arrive_expect_tx(bar_load, kOperand + kVBytes);
    tma_load_4d(&tmQ, bar_load, Qb, 0, hq, t0, b);
    tma_load_4d(&tmQ, bar_load, Qb + kPanel, 64, hq, t0, b);
#pragma unroll
    for (int pv = 0; pv < kPanels; ++pv)
      tma_load_4d(&tmG, bar_load, Gb + pv * kPanel, 64 * pv, h, t0, b);
    if (j + 1 < s1) {
      tma_prefetch_4d(&tmQ, 0, hq, t0 + kTile, b);
      tma_prefetch_4d(&tmQ, 64, hq, t0 + kTile, b);
#pragma unroll
      for (int pv = 0; pv < kPanels; ++pv) tma_prefetch_4d(&tmG, 64 * pv, h, t0 + kTile, b);
    }
  };
  bool pending = false;  // thread 0: a load was issued and not yet waited for
  if (tid == 0) {
    issue_loads(s0);
    pending = true;
  }
  __syncwarp();
  if (warp == 2) {  // D of the first reader: the log decays of the tiles [c, s0)
    float x = 0.f;
    for (int i = c + lane; i < s0; i += 32) x += p.lgu[bh * p.N + i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) d0_s[0] = x;
  }

  bool ok = true;
  float D = 0.f;
  uint32_t ph = 0;
  // row r's log a and lambda of a reader tile (loaded one reader ahead)
  auto row_in = [&](int jj, float& la_o, float& lam_o, float& lg_o) {
    const int tt0 = jj * kTile;
    const bool live = r < min(kTile, p.T - tt0);
    const int64_t rw = ((int64_t)b * p.T + tt0 + r) * p.H + h;
    la_o = (hh == 0 && p.log_a && live) ? p.log_a[rw] : 0.f;
    lam_o = live ? p.lam[rw * p.L + lam_l] : 0.f;
    lg_o = p.lgu[bh * p.N + jj];
  };
  float la_n, lam_n, lg_n;
  row_in(s0, la_n, lam_n, lg_n);
  for (int j = s0; j < s1; ++j, ph ^= 1) {
    const float la = la_n, lam = lam_n, lgj = lg_n;
    const float cs_scan = block_scan256(la, red);  // threads 0..127 hold row prefixes
    if (hh == 0) cs_s[r] = cs_scan;
    bool landed = true;
    if (tid == 0) {
      landed = ok && mbar_wait(bar_load, ph);
      if (landed) pending = false;
    }
    ok = __syncthreads_and(ok && landed);
    if (!ok) break;
    if (j == s0) D = d0_s[0];
    const float w = __expf(cs_s[r] + D) * lam;  // lam = 0 on rows past T
    if (j + 1 < s1) row_in(j + 1, la_n, lam_n, lg_n);
    // rows of Q scaled by w: the high part in place, the residual into Lb
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const int off = hh * kPanel + sw128_offset(r, g);
      const uint4 u = *reinterpret_cast<const uint4*>(Qb + off);
      uint32_t x4[4] = {u.x, u.y, u.z, u.w}, y4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x4[k]));
        const float a0 = f.x * w, a1 = f.y * w;
        const __nv_bfloat162 hi = __floats2bfloat162_rn(a0, a1);
        const float2 hf = __bfloat1622float2(hi);
        x4[k] = *reinterpret_cast<const uint32_t*>(&hi);
        y4[k] = pack_bf16(a0 - hf.x, a1 - hf.y);
      }
      *reinterpret_cast<uint4*>(Qb + off) = make_uint4(x4[0], x4[1], x4[2], x4[3]);
      *reinterpret_cast<uint4*>(Lb + off) = make_uint4(y4[0], y4[1], y4[2], y4[3]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16(128, DV, 1, 1);
      const uint32_t wh = smem_u32(Qb), wl = smem_u32(Lb), ga = smem_u32(Gb);
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk)
        mma_bf16(tmem, smem_desc_sw128(wh + kk * 2048, kPanel, 1024),
                 smem_desc_sw128(ga + kk * 2048, kPanel, 1024), idesc, (j > s0 || kk > 0) ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk)
        mma_bf16(tmem, smem_desc_sw128(wl + kk * 2048, kPanel, 1024),
                 smem_desc_sw128(ga + kk * 2048, kPanel, 1024), idesc, 1u);
      mma_commit(bar_mma);
      // the buffers are free once the products are done: then the next reader's loads
      ok = mbar_wait(bar_mma, ph);
      if (ok && j + 1 < s1) {
        issue_loads(j + 1);
        pending = true;
      }
    }
    __syncwarp();
    D += lgj;
  }
  ok = __syncthreads_and(ok);
  tc_fence_after();

  if (ok) {
    // Row d = r, this thread's half of d_v, staged over Q and the residual as 16-byte
    // chunks, chunk x of row d at x ^ (d & 7): the stores of 8 consecutive rows and the
    // reads of one row are free of bank conflicts.
    float4* stage = reinterpret_cast<float4*>(smem + RsSmem::kQ);
    constexpr int kRowChunks = DV / 4;
#pragma unroll
    for (int cc = 0; cc < kPanels; ++cc) {
      float v[32];
      tmem_ld32(tmem + lane_base + kHalf * hh + 32 * cc, v);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int x = (kHalf * hh + 32 * cc) / 4 + u;
        stage[r * kRowChunks + (x ^ (r & 7))] = make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
      }
    }
    __syncthreads();
    // the slot is contiguous in R: one warp's accesses cover 512 bytes
    float4* dst = reinterpret_cast<float4*>(p.R + (bh * p.N + c) * kD * DV);
    if (whole) {
#pragma unroll 4
      for (int i = tid; i < kD * kRowChunks; i += kThreadsB) {
        const int d = i / kRowChunks, x = i - d * kRowChunks;
        dst[i] = stage[d * kRowChunks + (x ^ (d & 7))];
      }
    } else {
#pragma unroll 4
      for (int i = tid; i < kD * kRowChunks; i += kThreadsB) {
        const int d = i / kRowChunks, x = i - d * kRowChunks;
        atomicAdd(dst + i, stage[d * kRowChunks + (x ^ (d & 7))]);
      }
    }
  } else if (tid == 0) {
    atomicOr(&g_tcb_error, 1u);
    // wait (bounded) for a load still in flight into this CTA's shared memory before it
    // is handed to another CTA
    if (pending) mbar_wait(bar_load, ph);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 128);
}

}  // namespace

// SMs of the current device (queried per call: the library may run on several devices).
static int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    n = 0;
  return n;
}

bool tc_bwd_dq_supported(int64_t dk, int64_t dv, int in_dtype, int grad_dtype) {
  return in_dtype == LL_BF16 && grad_dtype == LL_BF16 && dk == kD && (dv == 64 || dv == 128);
}

cudaError_t launch_tc_bwd_dq(const FwdArgs& f, const void* dout, float* dqh, void* dq_bf16,
                             float* dcq, float* dlam, cudaStream_t s) {
  if (f.dk != kD || (f.dv != 64 && f.dv != 128) || f.C != kTile) return cudaErrorInvalidValue;
  const int64_t rows = (int64_t)f.B * f.H * f.N * kD;  // TMA row coordinates are int32
  if (rows > INT32_MAX) return cudaErrorInvalidValue;
  const int dv = f.dv;
  CUtensorMap tmQ, tmK, tmV, tmG, tmU, tmNode, tmDQ;
  if (!make_tokens_map(&tmQ, f.q, f.B, f.T, f.Hqk, kD) ||
      !make_tokens_map(&tmK, f.k, f.B, f.T, f.Hqk, kD) ||
      !make_tokens_map(&tmV, f.v, f.B, f.T, f.H, dv) ||
      !make_tokens_map(&tmG, dout, f.B, f.T, f.H, dv) || !make_rows_map(&tmU, f.U, rows, dv) ||
      !make_rows_map(&tmNode, f.nodes, rows, dv))
    return cudaErrorInvalidValue;
  if (dq_bf16) {  // one q/k per head: dQ is [B, T, H, 128]
    if (f.Hqk != f.H || !make_tokens_map(&tmDQ, dq_bf16, f.B, f.T, f.H, kD))
      return cudaErrorInvalidValue;
  } else {
    tmDQ = tmQ;  // not used
  }
  BqParams p;
  p.B = f.B; p.T = f.T; p.H = f.H; p.hg = f.hg; p.L = f.L; p.N = f.N;
  p.log_a = f.log_a; p.lam = f.lam; p.lgu = f.lg; p.nlg = f.nlg;
  p.dqh = dqh; p.dq = dq_bf16; p.dcq = dcq; p.dlam = dlam;
  p.ahead = sm_count();
  p.tag = f.tag;
  p.tag_value = fwd_layout_tag(f.B, f.T, f.H, f.Hqk, f.dv);
  int levels = 0;  // inter-chunk levels a tile can have: bit length of N-1
  while ((int64_t(1) << levels) < f.N) ++levels;
  // The shared-memory limit is an attribute of the function on each device: set it
  // on every launch (a host-side call), so that every device the library runs on has it.
  const cudaError_t attr_err =
      dv == 128 ? cudaFuncSetAttribute(tc_bwd_dq_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_bwd_dq(kMaxChunkLevels - 1))
                : cudaFuncSetAttribute(tc_bwd_dq_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_bwd_dq(kMaxChunkLevels - 1));
  if (attr_err != cudaSuccess) return attr_err;
  const unsigned tiles = (unsigned)((int64_t)f.B * f.H * f.N);
  if (dv == 128)
    tc_bwd_dq_kernel<128><<<tiles, kThreadsB, smem_bwd_dq(levels), s>>>(tmQ, tmK, tmV, tmG, tmU,
                                                                         tmNode, tmDQ, p, levels);
  else
    tc_bwd_dq_kernel<64><<<tiles, kThreadsB, smem_bwd_dq(levels), s>>>(tmQ, tmK, tmV, tmG, tmU,
                                                                        tmNode, tmDQ, p, levels);
  return cudaGetLastError();
}

cudaError_t launch_tc_bwd_dkv(const FwdArgs& f, const void* dout, const float* R, float* dkh,
                              void* dk_bf16, float* dck, void* dv, cudaStream_t s) {
  if (f.dk != kD || (f.dv != 64 && f.dv != 128) || f.C != kTile) return cudaErrorInvalidValue;
  const int dvw = f.dv;
  CUtensorMap tmQ, tmK, tmV, tmG, tmDK, tmDV;
  if (!make_tokens_map(&tmQ, f.q, f.B, f.T, f.Hqk, kD) ||
      !make_tokens_map(&tmK, f.k, f.B, f.T, f.Hqk, kD) ||
      !make_tokens_map(&tmV, f.v, f.B, f.T, f.H, dvw) ||
      !make_tokens_map(&tmG, dout, f.B, f.T, f.H, dvw) ||
      !make_tokens_map(&tmDV, dv, f.B, f.T, f.H, dvw))
    return cudaErrorInvalidValue;
  if (dk_bf16) {  // one q/k per head: dK is [B, T, H, 128]
    if (f.Hqk != f.H || !make_tokens_map(&tmDK, dk_bf16, f.B, f.T, f.H, kD))
      return cudaErrorInvalidValue;
  } else {
    tmDK = tmK;  // not used
  }
  BkvParams p;
  p.B = f.B; p.T = f.T; p.H = f.H; p.hg = f.hg; p.L = f.L; p.N = f.N;
  p.log_a = f.log_a; p.lam = f.lam; p.lgu = f.lg; p.R = R;
  p.v = static_cast<const __nv_bfloat16*>(f.v);
  p.dkh = dkh; p.dk = dk_bf16; p.dck = dck;
  // The shared-memory limit is an attribute of the function on each device: set it
  // on every launch (a host-side call), so that every device the library runs on has it.
  const cudaError_t attr_err =
      dvw == 128 ? cudaFuncSetAttribute(tc_bwd_dkv_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_bwd_dkv())
                : cudaFuncSetAttribute(tc_bwd_dkv_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_bwd_dkv());
  if (attr_err != cudaSuccess) return attr_err;
  // one persistent CTA per SM, taking tiles SM-count apart
  const int64_t tiles = (int64_t)f.B * f.H * f.N;
  const int sms = sm_count();
  const unsigned grid = (unsigned)(sms > 0 && sms < tiles ? sms : tiles);
  if (dvw == 128)
    tc_bwd_dkv_kernel<128><<<grid, kThreadsB, smem_bwd_dkv(), s>>>(tmQ, tmK, tmV, tmG, tmDK,
                                                                   tmDV, p);
  else
    tc_bwd_dkv_kernel<64><<<grid, kThreadsB, smem_bwd_dkv(), s>>>(tmQ, tmK, tmV, tmG, tmDK,
                                                                  tmDV, p);
  return cudaGetLastError();
}

cudaError_t launch_tc_bwd_rstate(const FwdArgs& f, const void* dout, float* R, cudaStream_t s) {
  if (f.dk != kD || (f.dv != 64 && f.dv != 128) || f.C != kTile) return cudaErrorInvalidValue;
  CUtensorMap tmQ, tmG;
  if (!make_tokens_map(&tmQ, f.q, f.B, f.T, f.Hqk, kD) ||
      !make_tokens_map(&tmG, dout, f.B, f.T, f.H, f.dv))
    return cudaErrorInvalidValue;
  BrParams p;
  p.B = f.B; p.T = f.T; p.H = f.H; p.hg = f.hg; p.L = f.L; p.N = f.N;
  p.log_a = f.log_a; p.lam = f.lam; p.lgu = f.lg; p.R = R;
  int levels = 0;  // slots c < N: levels z = ctz(c) < bit length of N - 1
  while ((int64_t(1) << levels) < f.N) ++levels;
  p.levels = levels;
  int64_t runs = 0;
  for (int z = 0; z < levels; ++z) runs += runs_at_level(f.N, z);
  const int64_t grid = runs * f.B * f.H;
  if (grid == 0) return cudaSuccess;
  if (grid > INT32_MAX) return cudaErrorInvalidValue;
  // The shared-memory limit is an attribute of the function on each device: set it
  // on every launch (a host-side call), so that every device the library runs on has it.
  const cudaError_t attr_err =
      f.dv == 128 ? cudaFuncSetAttribute(tc_bwd_rstate_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bwd_rstate())
                  : cudaFuncSetAttribute(tc_bwd_rstate_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bwd_rstate());
  if (attr_err != cudaSuccess) return attr_err;
  // Slots with more readers than one run (z > kRunLog: c a multiple of 2^(kRunLog+1)) are
  // sums of several runs' atomics: zeroed first.  With N a multiple of that period they are
  // every period-th slot of the flat [B*H][N] array.
  const int64_t period = int64_t(2) << kRunLog;
  if (levels > kRunLog + 1) {
    const size_t slot = sizeof(float) * (size_t)kD * f.dv;
    const size_t slots = (size_t)f.B * f.H * f.N;
    cudaError_t e = (f.N % period == 0)
                        ? cudaMemset2DAsync(R, period * slot, 0, slot, slots / period, s)
                        : cudaMemsetAsync(R, 0, slot * slots, s);
    if (e != cudaSuccess) return e;
  }
  if (f.dv == 128)
    tc_bwd_rstate_kernel<128><<<(unsigned)grid, kThreadsB, smem_bwd_rstate(), s>>>(tmQ, tmG, p);
  else
    tc_bwd_rstate_kernel<64><<<(unsigned)grid, kThreadsB, smem_bwd_rstate(), s>>>(tmQ, tmG, p);
  return cudaGetLastError();
}

cudaError_t tcb_take_error(cudaStream_t s, unsigned* flags) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_tcb_error, sizeof(v), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && v) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbolAsync(g_tcb_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  *flags = v;
  return e;
}

}  // namespace ll

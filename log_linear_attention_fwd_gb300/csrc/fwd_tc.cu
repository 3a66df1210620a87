// Forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), bf16 inputs with
// fp32 accumulation, d_k = 128, d_v = 64 or 128, 128-token tiles (the M = 128 datapath of
// one SM).
//
// The chunked two-stage algorithm (page "论文阅读：Log-Linear Attention", sections 矩阵分解
// and 两阶段计算; page "算力终结者来了！…", section 高效训练算法) with the tile as the chunk, in
// one kernel, tc_forward_kernel: per tile, the intra-tile product, the tile's chunk state,
// its part of the Fenwick block-state tree, and the lambda-weighted readout of the block
// states of the earlier tiles fused into the output epilogue (no per-level output reaches
// memory).  q, k and v are read once.
//
// With 128-token tiles the chunk-pair level log2(C)+1 of a requested C = 64 lies inside a
// tile and is taken in the dense masked product; the sum is the same.
//
// Shared-memory tiles are 128 rows x 64 or 128 bf16 stored as 64-column panels with the
// 128-byte swizzle TMA produces; K-major operands (Q, K, block states) and MN-major ones
// (V as the B of P V; V and K in the state GEMM) are described to tcgen05 with the
// matching descriptors.  P, the A of P V, is written to TMEM (two bf16 per column).  Every wait (mbarriers, block-state flags) is bounded (see
// tc_ptx.cuh); a CTA whose wait times out raises g_tc_error, skips the MMAs and stores
// that depend on it, frees its TMEM and exits.
//
// Single-lane issue blocks (TMA, MMA) are followed by __syncwarp(): otherwise the other
// lanes of the warp reach the next mbarrier spin first and keep the issuing lane from
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
constexpr int kD = 128;                     // d_k; d_v is the kernel's template argument
constexpr int kPanel = kTile * 64 * 2;      // one [128][64] bf16 panel: 16 KiB
constexpr int kOperand = 2 * kPanel;        // a 128 x 128 bf16 tile: 32 KiB
constexpr int kLamStride = 9;               // intra lambdas per row in smem (levels 0..7)
constexpr int kIntraLevels = 8;             // levels inside a 128-token tile: 0..7
constexpr int kTileLc = 7;                  // log2(kTile)
constexpr int kMaxChunkLevels = 32;         // chunk levels m = 1..31 (positions < 2^31)

struct TcParams {
  int B, T, H, L, N;
  int hg;            // value heads per q/k head: head h reads q/k head h / hg
  const float* log_a;
  const float* lam;
  void* out;
  int64_t so_b, so_t, so_h;  // element strides of out's b, t and h dimensions
  uint8_t* U;        // [B*H][N] tile states U_i, bf16 [d_k][d_v] (written for even i only)
  uint8_t* nodes;    // [B*H][N] block states of the even slots, bf16 [d_k][d_v]
  float* lgu;        // [B*H][N] log decay of each tile
  float* nlg;        // [B*H][N] log decay of the block in each even slot
  uint32_t* rdy_u;   // [B*H][N] ready flags of U, carrying the tile's log decay
  uint32_t* rdy_n;   // [B*H][N] ready flags of the even slots' block states, carrying the
                     // block's log decay (decay_flag: bit-inverted, never 0)
  uint32_t* tick;    // tile ticket counter
  uint32_t* tag;     // the workspace's layout tag, written by the CTA of ticket 0
  uint32_t tag_value;
  int out_f32;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
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

// ------------------------------------------------------------------ the forward kernel
//
// One CTA per 128-token tile; 8 warps: warps w and w+4 share TMEM lane quarter w mod 4
// (tile rows 32(w mod 4)..+31) and split its d_v columns (half each) and its P chunks.
//
// Tiles are taken in ticket order (an atomic counter; tile j of every (b,h) before tile
// j+1), so a CTA only waits for tiles with smaller tickets: those CTAs are resident or
// done, and they publish what others wait for before they wait on anything themselves.
//
//   1. Q, K, V by TMA; per-row log a and lambda; cs = tile-local prefix sums of log a.
//   2. S = Q K^T (tcgen05) into TMEM columns 0..127, issued as soon as Q and K land.
//   3. K rows scaled in place by w_s = exp(lg - cs_s); U = (w ⊙ K)^T V into columns
//      128..128+d_v (the tile's chunk state, d_k x d_v).
//   4. (after 5) P = S ⊙ exp(cs_t - cs_s) ⊙ lambda[t, l(t,s)] on the causal half, bf16
//      into TMEM columns 128..191 (the state's, read out by then); O = P V into columns
//      0..d_v.
//   5. Right after the state MMA (before P): U_j is staged bf16 in the K buffer; for even
//      j it is published (stored coalesced), for odd j the CTA forms the block state of
//      slot j+1 from it (below) and publishes that.  Q stays in shared memory for step 6.
//   6. For every set bit m-1 of j, in increasing m: the block state of slot c_m by TMA
//      into shared memory (K's tile holds one state of d_v = 128 or two of d_v = 64 and
//      is free before P is built: the lowest levels load then if their flags are up;
//      V's tile after P V), MMA Q Tot into one of two TMEM buffers (columns 0.. and
//      128..), and the previous level's product added to O with the row weights
//      lambda[t, 7+m] exp(cs_t + D_m).  D_m, the log decay from the block's end to the
//      tile's start, is the sum of the log decays of the lower levels' blocks, which
//      their producers store next to them.
//   7. O to bf16 through a TMA store, or fp32 stores.
//
// Block states.  Slot c holds the decayed total of the 2^z tiles before c, z = ctz(c):
// for odd c that is U_{c-1} itself; for even c it is formed by tile c-1 from
//     [c - 2^z, c) = [c - 2^z, c - 2^(z-1)) + ... + [c - 4, c - 2) + [c - 2, c - 1) + [c - 1, c)
// whose parts are the block states of slots c - 2^(k-1) (k = z..2), U_{c-2} (slot c-1)
// and U_{c-1}, tile c-1's own state: Tot = sum_k exp(LG of the parts to its right)
// part_k, in fp32, rounded once to bf16.  All the parts come from tiles that started
// earlier and publish them early, so there is no chain of merges, and a tile publishes
// what it forms before it waits for the block states it reads.
//
// Publication: every thread's generic stores, a block barrier, then thread 0 raises the
// ready flag with a release store; the flag's value is the published state's log decay
// (bit-inverted so that it is never 0), which readers need next and so get in the same
// load as the flag.  Readers: one thread acquires the flag; generic loads
// by the others follow a block barrier; a TMA load is issued by the acquiring thread
// itself after a global proxy fence.

constexpr int kThreadsF = 256;
// Stores an even tile's state and raises its flag: lane 0 of warp 4, whose rows (0..31)
// have no P chunk above the diagonal to compute, so its wait costs the P build nothing.
constexpr int kPubThread = 128;

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

// kOut: the whole forward; else only the tile states and block states (the backward's
// recompute, which needs no output): no Q, and K and V move to the front.
template <bool kOut>
struct FSmem {
  // byte offsets from the 1024-aligned base
  static constexpr int kQ = 0, kK = kOut ? kOperand : 0, kV = kK + kOperand;
  static constexpr int kBars = kV + kOperand;                  // 11 mbarriers (12 slots)
  static constexpr int kTslot = kBars + 12 * 8;
  static constexpr int kInt = kTslot + 16;                     // ticket, loads per buffer
  static constexpr int kRed = kInt + 16;                       // 8 floats
  static constexpr int kLg = kRed + 32;                        // 4 floats
  static constexpr int kNl = kLg + 16;                         // kMaxChunkLevels floats
  static constexpr int kCs = kNl + 4 * kMaxChunkLevels;        // 128 floats
  static constexpr int kFcol = kCs + 4 * kTile;                // 128 floats
  static constexpr int kLam = kFcol + 4 * kTile;               // 128 x kLamStride floats
  static constexpr int kLamX = kLam + 4 * kTile * kLamStride;  // [levels][128] floats
};

template <bool kOut>
size_t smem_fused(int levels) {
  return kOut ? (size_t)FSmem<true>::kLamX + 4 * kTile * levels + 1024
              : (size_t)FSmem<false>::kLam + 1024;  // no lambdas
}

// Multiplies columns [64 half, 64 half + 64) of row r of a swizzled bf16 tile by s.
__device__ __forceinline__ void scale_half_row_inplace(uint8_t* buf, int r, int half, float s) {
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) {
    const int c = (cc + r) & 7;
    uint4* ptr = reinterpret_cast<uint4*>(buf + half * kPanel + r * 128 + c * 16);
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

// Pieces of a 128 x DV bf16 state: piece q (16 bytes) is row q / (DV/8), columns
// 8 (q mod DV/8) .. +7 of the row-major matrix; each thread of the CTA moves the pieces
// it * 256 + tid.  piece_offset is where a piece sits in a swizzled smem tile of 64-column
// panels.
template <int DV>
struct Dv {
  static constexpr int kStateBytes = kD * DV * 2;             // one published state
  static constexpr int kVBytes = kTile * DV * 2;              // one V (or output) tile
  static constexpr int kPanels = DV / 64;                     // 64-column panels of d_v
  static constexpr int kStatePieces = kStateBytes / 16 / 256; // per thread: 8 or 4
  static constexpr int kHalf = DV / 2;                        // d_v columns per thread
  // shared buffers for the levels' block states: K's tile (one state of d_v = 128, two of
  // d_v = 64) and V's
  static constexpr int kNodeBufs = DV == 64 ? 3 : 2;
};

template <int DV>
__device__ __forceinline__ uint32_t piece_offset(uint32_t q) {
  const uint32_t row = q / (DV / 8), c16 = q % (DV / 8);
  return (c16 >> 3) * kPanel + sw128_offset(row, c16 & 7);
}

template <int DV, bool kOut>
__global__ void __launch_bounds__(kThreadsF, 2)
    tc_forward_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmOut,
                      const __grid_constant__ CUtensorMap tmU,
                      const __grid_constant__ CUtensorMap tmNode, TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  using FS = FSmem<kOut>;
  constexpr uint32_t kTmemCols = kOut ? 256 : 128;  // states only: U in columns 0..d_v
  constexpr uint32_t kUcol = kOut ? 128 : 0;
  uint8_t* Qb = smem + FS::kQ;    // Q (kept for the level MMAs), then the output
  uint8_t* Kb = smem + FS::kK;    // K, then w ⊙ K, then U in bf16, then P, then block states
  uint8_t* Vb = smem + FS::kV;    // V, then block states
  using G = Dv<DV>;
  constexpr int kStatePieces = G::kStatePieces;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + FS::kBars);
  uint64_t* bar_load = &bars[0];
  uint64_t* bar_s = &bars[1];
  uint64_t* bar_u = &bars[2];
  uint64_t* bar_o = &bars[3];
  uint64_t* bar_lvl = &bars[4];      // [2]: level MMAs
  uint64_t* bar_node = &bars[6];     // [3]: block-state loads, one per shared buffer
  uint64_t* bar_free = &bars[9];     // [2]: every warp has read a level's TMEM buffer
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + FS::kTslot);
  uint32_t* ints = reinterpret_cast<uint32_t*>(smem + FS::kInt);  // ticket, loads[3]
  float* red = reinterpret_cast<float*>(smem + FS::kRed);
  float* lg_s = reinterpret_cast<float*>(smem + FS::kLg);
  float* nl_s = reinterpret_cast<float*>(smem + FS::kNl);
  float* cs_s = reinterpret_cast<float*>(smem + FS::kCs);
  float* fcol = reinterpret_cast<float*>(smem + FS::kFcol);  // exp(cs_e - cs_s), e = s | 31
  float* lam_s = reinterpret_cast<float*>(smem + FS::kLam);
  float* lamx = reinterpret_cast<float*>(smem + FS::kLamX);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int qt = warp & 3;           // row quarter (TMEM lane quarter) of this warp
  const int hh = warp >> 2;          // which of the quarter's two warps
  const int r = tid & (kTile - 1);   // tile row of this thread

  // ---- the tile: by ticket
  if (tid == 0) ints[0] = atomicAdd(p.tick, 1u);
  if (warp == 1) {
    tmem_alloc(tslot, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 64) {
    if (kOut) prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    prefetch_tensormap(&tmOut);
    prefetch_tensormap(&tmU);
    prefetch_tensormap(&tmNode);
    for (int q = 0; q < 9; ++q) mbar_init(&bars[q], 1);
    for (int q = 1; q < 4; ++q) ints[q] = 0;
    mbar_init(&bar_free[0], kThreadsF / 32);
    mbar_init(&bar_free[1], kThreadsF / 32);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t lane_base = (uint32_t)(qt * 32) << 16;
  const int BH = p.B * p.H;
  const int tk = (int)ints[0];
  if (tk == 0 && tid == 0) *p.tag = p.tag_value;  // the layout a backward may read
  const int j = tk / BH, bhi = tk - j * BH;
  const int b = bhi / p.H, h = bhi - b * p.H;
  const int hq = h / p.hg;  // q/k head
  const int64_t N = p.N;
  const int64_t bh = bhi;
  const int t0 = j * kTile;
  const int n = min(kTile, p.T - t0);
  const int64_t row = ((int64_t)b * p.T + t0 + r) * p.H + h;  // (b, t, h) of row r
  const int nlev = __popc((unsigned)j);                        // inter-chunk levels read
  const bool row_live = r < n;
  bool landed = true;  // thread 0: Q, K and V arrived
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_load, (kOut ? 2 : 1) * kOperand + G::kVBytes);
    if (kOut) {
      tma_load_4d(&tmQ, bar_load, Qb, 0, hq, t0, b);
      tma_load_4d(&tmQ, bar_load, Qb + kPanel, 64, hq, t0, b);
    }
    tma_load_4d(&tmK, bar_load, Kb, 0, hq, t0, b);
    tma_load_4d(&tmK, bar_load, Kb + kPanel, 64, hq, t0, b);
#pragma unroll
    for (int pv = 0; pv < G::kPanels; ++pv)
      tma_load_4d(&tmV, bar_load, Vb + pv * kPanel, 64 * pv, h, t0, b);
  }
  if (kOut && tid == 64 && h == 0 && j + 2 < N) {  // warm L2 with tile j+2's log a and lambda (all heads)
    const int64_t tok0 = (int64_t)b * p.T + (int64_t)(j + 2) * kTile;
    const int64_t ntok = min(kTile, p.T - (j + 2) * kTile);
    prefetch_l2_range(p.lam + tok0 * p.H * p.L, ntok * p.H * p.L * 4);
    if (p.log_a) prefetch_l2_range(p.log_a + tok0 * p.H, ntok * p.H * 4);
  }
  __syncwarp();

  // ---- per-row data: log a, the intra-tile lambdas, the raw inter-level lambdas (the
  // two threads of a row split the loads; the last ones go straight to shared memory)
  const float la = (hh == 0 && p.log_a && row_live) ? p.log_a[row] : 0.f;
  float lam_in[kIntraLevels / 2];
#pragma unroll
  for (int i = 0; i < kIntraLevels / 2; ++i) {
    const int l = hh * (kIntraLevels / 2) + i;
    lam_in[i] = (kOut && row_live && l < p.L) ? p.lam[row * p.L + l] : 0.f;
  }
  if (kOut) {
    int k = 0;
#pragma unroll 4
    for (int m = 1; m < kMaxChunkLevels; ++m) {
      if (!((j >> (m - 1)) & 1)) continue;
      if ((k & 1) == hh)  // copied in the background: read only by the level loop
        cp_async4(&lamx[k * kTile + r], row_live ? p.lam + row * p.L + kTileLc + m : p.lam,
                  row_live ? 4u : 0u);
      ++k;
    }
  }
  if (tid == 0) {  // S = Q K^T as soon as the tiles land, before the scan needs log a
    landed = mbar_wait(bar_load, 0);
    if (kOut && landed) {
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
  }
  const float cs_scan = block_scan256(la, red);  // threads 0..127 hold row prefixes
  if (hh == 0) cs_s[r] = cs_scan;
  if (tid == kTile - 1) lg_s[0] = cs_scan;       // padding rows add 0: the tile's log decay
  if (kOut) {
#pragma unroll
    for (int i = 0; i < kIntraLevels / 2; ++i)
      lam_s[r * kLamStride + hh * (kIntraLevels / 2) + i] = lam_in[i];
  }
  __syncthreads();
  const float cs = cs_s[r];
  const float lg = lg_s[0];
  if (kOut && hh == 1) fcol[r] = __expf(cs_s[r | 31] - cs);  // <= 1: cs does not increase

  // ---- S = Q K^T (issued by thread 0 above)
  bool all_ok = __syncthreads_and(landed);
  bool ok = all_ok && (!kOut || mbar_wait(bar_s, 0));
  tc_fence_after();
  all_ok = __syncthreads_and(ok);

  // ---- U = (w ⊙ K)^T V, d_k x d_v: K rows scaled in place (S no longer reads K)
  if (all_ok) scale_half_row_inplace(Kb, r, hh, row_live ? expf(lg - cs) : 0.f);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (all_ok && tid == 0) {
    tc_fence_after();
    constexpr uint32_t idesc = idesc_bf16(128, DV, /*A MN-major*/ 1, /*B MN-major*/ 1);
    const uint32_t va = smem_u32(Vb), ka = smem_u32(Kb);
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk)
      mma_bf16(tmem + kUcol, smem_desc_sw128(ka + kk * 2048, kPanel, 1024),
               smem_desc_sw128(va + kk * 2048, kPanel, 1024), idesc, kk > 0);
    mma_commit(bar_u);
  }
  __syncwarp();

  ok = all_ok && mbar_wait(bar_u, 0);
  tc_fence_after();
  all_ok = __syncthreads_and(ok);

  // ---- stage U_j (bf16 in Kb, which the state MMA no longer reads); publish it (stored
  // coalesced) for even j; for odd j form the block state of slot j+1 and publish it.  Q stays
  // in Qb for the level MMAs.  Published states are row-major [d_k][d_v] bf16; thread tid
  // moves the 16-byte pieces q = it * 256 + tid.  This runs even after an error, so that
  // no reader waits for a flag that is never raised.
  const uint8_t* Ug = p.U + bh * N * G::kStateBytes;
  uint8_t* nodes = p.nodes + bh * N * G::kStateBytes;
  float* nlg = p.nlg + bh * N;
  uint32_t* rdy_u = p.rdy_u + bh * N;
  uint32_t* rdy_n = p.rdy_n + bh * N;
#pragma unroll
  for (int c = 0; c < G::kPanels; ++c) {  // U row r (d_k), this thread's half of d_v -> Kb
    float v[32];
    tmem_ld32(tmem + lane_base + kUcol + G::kHalf * hh + 32 * c, v);
    put_row32_bf16(Kb, r, G::kPanels * hh + c, v);
  }
  // Only U of even tiles is read by other tiles (slot j+1, odd, is U_j; an even slot's
  // parts are U_{c-2} and U_{c-1}, and U_{c-1} is summed by its own CTA), by the backward
  // and by the prefill: odd tiles keep theirs on chip.  Even tiles store the staged tile
  // with TMA (thread kPubThread), which raises the ready flag once the store is complete:
  // only that thread's warp waits for the store.
  const bool pub_u = !(j & 1);
  fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0) p.lgu[bh * N + j] = lg;
  if (pub_u && tid == kPubThread) {
    const int row0 = (int)((bh * N + j) * kD);
#pragma unroll
    for (int pv = 0; pv < G::kPanels; ++pv) tma_store_2d(&tmU, Kb + pv * kPanel, 64 * pv, row0);
    tma_store_commit();
    tma_store_wait_read();  // Kb is refilled below
  }
  const bool forms = (j & 1) && j + 1 < N;  // odd j forms the block state of slot j+1
  if (forms) {
    float acc[8 * kStatePieces];  // the block state of slot j+1, fp32, in this thread's pieces
#pragma unroll
    for (int it = 0; it < kStatePieces; ++it) {
      const uint4 w = *reinterpret_cast<const uint4*>(Kb + piece_offset<DV>(it * kThreadsF + tid));
      const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
        acc[8 * it + 2 * e] = f.x;
        acc[8 * it + 2 * e + 1] = f.y;
      }
    }
    // Slot c = j+1 holds [c - 2^z, c), z = ctz(c): the block states of slots c - 2^(k-1)
    // (k = z..2), then U_{j-1}, then U_j; summed right to left, each weighted by the
    // decay across what lies to its right, in fp32, rounded once to bf16.
    const int c = j + 1, zc = __ffs(c) - 1;
    bool fl = true;
    if (tid < zc) {  // thread 0: U_{j-1}; thread t >= 1: slot c - 2^t; each flag carries
                     // its part's log decay
      uint32_t fv;
      fl = wait_flag_acquire_value(tid == 0 ? &rdy_u[j - 1] : &rdy_n[c - (1 << tid)], &fv);
      nl_s[tid] = fl ? flag_decay(fv) : 0.f;
    }
    if (!__syncthreads_and(fl) && tid == 0) atomicOr(&g_tc_error, 2u);
    float G = lg;  // log decay of what has been summed so far
    for (int k = 1; k <= zc; ++k) {  // k = 1: U_{j-1}; k >= 2: slot c - 2^(k-1)
      const int cs_k = c - (1 << (k - 1));
      const uint4* src = reinterpret_cast<const uint4*>(
          k == 1 ? Ug + (int64_t)(j - 1) * G::kStateBytes : nodes + (int64_t)cs_k * G::kStateBytes);
      const float L = nl_s[k - 1];
      const float g = __expf(G);
      uint4 y[kStatePieces];
#pragma unroll
      for (int it = 0; it < kStatePieces; ++it) y[it] = __ldcg(src + it * kThreadsF + tid);
#pragma unroll
      for (int it = 0; it < kStatePieces; ++it) {
        const uint32_t w4[4] = {y[it].x, y[it].y, y[it].z, y[it].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
          acc[8 * it + 2 * e] = fmaf(g, f.x, acc[8 * it + 2 * e]);
          acc[8 * it + 2 * e + 1] = fmaf(g, f.y, acc[8 * it + 2 * e + 1]);
        }
      }
      G += L;
    }
#pragma unroll
    for (int it = 0; it < kStatePieces; ++it)
      reinterpret_cast<uint4*>(nodes + (int64_t)c * G::kStateBytes)[it * kThreadsF + tid] =
          make_uint4(pack_bf16(acc[8 * it], acc[8 * it + 1]), pack_bf16(acc[8 * it + 2], acc[8 * it + 3]),
                     pack_bf16(acc[8 * it + 4], acc[8 * it + 5]),
                     pack_bf16(acc[8 * it + 6], acc[8 * it + 7]));
    if (tid == 0) nlg[c] = G;
    __syncthreads();
    if (tid == 0) st_release_gpu(&rdy_n[c], decay_flag(G));
  }

  __syncthreads();  // the staged U in Kb is no longer read
  if (pub_u && tid == kPubThread) {  // once U_j is in memory, raise its flag
    tma_store_wait_all();
    fence_proxy_async_global();
    st_release_gpu(&rdy_u[j], decay_flag(lg));
  }

  uint32_t consumed = 0;  // thread 0: block-state loads waited for, 8 bits per buffer
  if constexpr (kOut) {
    // ---- the levels' block states.  Level k (the k-th set bit of j, from the lowest) is
    // owned by thread 32+k: it finds its slot c, acquires the slot's ready flag (which
    // carries the block's log decay) and issues the TMA load itself, after a proxy fence,
    // so the acquire and the async-proxy read are ordered in one thread.  Level k goes to
    // shared buffer k mod kNodeBufs: K's tile (free now; one buffer for d_v = 128, two for
    // d_v = 64), then V's (free once P V is done).  The block state of slot c is U_{c-1}
    // for odd c.
    int my_c = 0;         // thread 32+k, k < nlev: the slot of level k
    bool acquired = false;
    {
      const int k = tid - 32;
      if (k >= 0 && k < nlev) {
        int m = 0;
        for (int seen = -1; seen < k;) {
          ++m;
          if ((j >> (m - 1)) & 1) ++seen;
        }
        my_c = (j >> (m - 1)) << (m - 1);
      }
    }
    auto node_buf = [&](int b) -> uint8_t* {
      return b == G::kNodeBufs - 1 ? Vb : Kb + b * G::kStateBytes;
    };
    auto fetch = [&](int k) {  // thread 32+k: TMA of level k's block state
      if (tid == 32 + k) {
        const int b = k % G::kNodeBufs;
        uint8_t* dst = node_buf(b);
        const bool is_u = (my_c & 1) != 0;
        const int row0 = (int)((bh * N + (is_u ? my_c - 1 : my_c)) * kD);
        atomicAdd(&ints[1 + b], 1u);
        mbar_arrive_expect_tx(&bar_node[b], G::kStateBytes);
#pragma unroll
        for (int pv = 0; pv < G::kPanels; ++pv)
          tma_load_2d(is_u ? &tmU : &tmNode, &bar_node[b], dst + pv * kPanel, 64 * pv, row0);
      }
    };
    // levels whose buffer lies in K's tile: load now if the flag is already up (one poll)
    if (all_ok && tid >= 32 && tid - 32 < nlev && tid - 32 < G::kNodeBufs - 1) {
      const uint32_t fv = ld_acquire_gpu(my_c & 1 ? &rdy_u[my_c - 1] : &rdy_n[my_c]);
      if (fv != 0) {
        acquired = true;
        nl_s[tid - 32] = flag_decay(fv);
        fence_proxy_async_global();
        fetch(tid - 32);
      }
    }
    __syncwarp();

    // ---- P, bf16 (two per column) into TMEM columns 128..191: the state's columns, read
    // out above.  The two warps of quarter qt take the 32-column chunks of their parity;
    // chunk c of row r goes to columns [128 + 16c, +16).  Chunks c > qt lie above the
    // diagonal (zero), chunks c < qt below it (level 5 + bit_length(qt XOR c) for every
    // pair), chunk qt holds the diagonal.
    if (all_ok) {
      const float* lam_r = lam_s + r * kLamStride;
      for (int c = hh; c < kTile / 32; c += 2) {
        float sv[32];
        if (c <= qt) {
          tmem_ld32(tmem + lane_base + c * 32, sv);
          if (c < qt) {  // exp(cs_t - cs_s) = exp(cs_t - cs_e) exp(cs_e - cs_s), both <= 1
            const float wl = lam_r[5 + (32 - __clz((unsigned)(qt ^ c)))] *
                             __expf(cs - cs_s[c * 32 + 31]);
#pragma unroll
            for (int k = 0; k < 32; ++k) sv[k] *= wl * fcol[c * 32 + k];
          } else if (cs_s[c * 32] - cs_s[c * 32 + 31] < 80.f) {
            // the diagonal chunk with a decay range that keeps exp(cs_t - cs_e) <= e^80:
            // exp(cs_t - cs_s) = exp(cs_t - cs_e) exp(cs_e - cs_s).  The pair (r, s) has level
            // bit_length(lane XOR k) <= 5 for column k <= lane: the six lambdas of the levels
            // inside a 32-token chunk are held in registers and picked by select.
            const float gt = row_live ? __expf(cs - cs_s[c * 32 + 31]) : 0.f;
            const int lane = tid & 31;
            const float l0 = lam_r[0], l1 = lam_r[1], l2 = lam_r[2], l3 = lam_r[3],
                        l4 = lam_r[4], l5 = lam_r[5];
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const int x = lane ^ k;
              const float lv = x >= 16 ? l5 : x >= 8 ? l4 : x >= 4 ? l3 : x >= 2 ? l2 : x >= 1 ? l1 : l0;
              const float v = sv[k] * lv * (gt * fcol[c * 32 + k]);
              sv[k] = k <= lane ? v : 0.f;
            }
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
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) sv[k] = 0.f;
        }
        uint32_t pw[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pw[e] = pack_bf16(sv[2 * e], sv[2 * e + 1]);
        tmem_st16(tmem + lane_base + 128 + 16 * c, pw);
      }
      tmem_wait_st();
    }
    tc_fence_before();
    all_ok = __syncthreads_and(ok);
    // ---- O = P V into columns 0..DV (P from TMEM, V MN-major as B)
    if (all_ok && tid == 0) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16(128, DV, 0, 1);
      const uint32_t va = smem_u32(Vb);
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk)
        mma_bf16_ts(tmem, tmem + 128 + 8 * kk, smem_desc_sw128(va + kk * 2048, kPanel, 1024), idesc,
                    kk > 0);
      mma_commit(bar_o);
    }
    __syncwarp();

    // ---- while P V runs, the remaining levels' flags (waited for, bounded)
    {
      bool fl = true;
      const int k = tid - 32;
      if (k >= 0 && k < nlev && !acquired) {
        uint32_t fv;
        fl = wait_flag_acquire_value(my_c & 1 ? &rdy_u[my_c - 1] : &rdy_n[my_c], &fv);
        nl_s[k] = fl ? flag_decay(fv) : 0.f;
        fence_proxy_async_global();
      }
      if (!__syncthreads_and(fl) && tid == 0) atomicOr(&g_tc_error, 2u);
    }
    // ---- O = P V is done: V's tile is free
    ok = all_ok && mbar_wait(bar_o, 0);
    tc_fence_after();
    all_ok = __syncthreads_and(ok);
    if (all_ok && tid >= 32 && tid - 32 < nlev && tid - 32 < G::kNodeBufs && !acquired)
      fetch(tid - 32);
    __syncwarp();

    // ---- O from TMEM into registers: this thread's half row, columns [DV/2 hh, +DV/2)
    float o[G::kHalf];
#pragma unroll
    for (int q = 0; q < G::kHalf; ++q) o[q] = 0.f;
    const uint32_t col0 = (uint32_t)G::kHalf * hh;
    if (all_ok) {
#pragma unroll
      for (int c = 0; c < G::kPanels; ++c) {
        float v[32];
        tmem_ld32(tmem + lane_base + col0 + c * 32, v);
#pragma unroll
        for (int q = 0; q < 32; ++q) o[c * 32 + q] = v[q];
      }
    }
    cp_async_wait_all();  // the inter-level lambdas
    tc_fence_before();
    __syncthreads();  // TMEM is free

    // ---- inter-chunk levels, without block barriers.  Level k uses shared buffer
    // k mod kNodeBufs and TMEM columns [128 (k&1), +DV).  Thread 0 issues MMA k once its
    // block state has landed and every warp has added level k-2 to O (bar_free[k&1]); each
    // warp adds level k-1 to O once MMA k-1 is done (bar_lvl), then releases that TMEM
    // buffer.  The load of level k-1+kNodeBufs starts as soon as MMA k-1 is done with its
    // shared buffer.
    const int lane = tid & 31;
    uint32_t lvl_ph = 0, node_ph = 0, free_ph = 0;  // phase bits per buffer
    float D = 0.f;  // log decay from block k's end to the tile's start
    bool lv_ok = all_ok;
    int nb = 0;  // k mod kNodeBufs
    for (int k = 0; k <= nlev && all_ok; ++k) {
      if (tid == 0 && k < nlev) {  // issue level k
        bool go = lv_ok && mbar_wait(&bar_node[nb], (node_ph >> nb) & 1);
        node_ph ^= 1u << nb;
        if (go) consumed += 1u << (8 * nb);
        if (k >= 2) {
          go = go && mbar_wait(&bar_free[k & 1], (free_ph >> (k & 1)) & 1);
          free_ph ^= 1u << (k & 1);
        }
        if (go) {
          tc_fence_after();
          // A = Q (K-major), B = the block state [d_k][d_v] (MN-major, like V in P V)
          constexpr uint32_t idesc = idesc_bf16(128, DV, 0, 1);
          const uint32_t qa = smem_u32(Qb), sa = smem_u32(node_buf(nb));
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
            mma_bf16(tmem + (k & 1) * 128, smem_desc_sw128(qa + off, 16, 1024),
                     smem_desc_sw128(sa + kk * 2048, kPanel, 1024), idesc, kk > 0);
          }
          mma_commit(&bar_lvl[k & 1]);
        }
        lv_ok = go;
      }
      nb = nb + 1 == G::kNodeBufs ? 0 : nb + 1;
      __syncwarp();
      if (k >= 1) {  // level k-1 into O
        const int bf = (k - 1) & 1;
        const bool got = __all_sync(0xffffffffu, mbar_wait(&bar_lvl[bf], (lvl_ph >> bf) & 1));
        lvl_ph ^= 1u << bf;
        if (!got) {
          lv_ok = false;
          break;
        }
        tc_fence_after();
        if (k - 1 + G::kNodeBufs < nlev) fetch(k - 1 + G::kNodeBufs);  // into MMA k-1's buffer
        const float wr = lamx[(k - 1) * kTile + r] * __expf(cs + D);
        D += nl_s[k - 1];
#pragma unroll
        for (int c = 0; c < G::kPanels; ++c) {
          float v[32];
          tmem_ld32(tmem + lane_base + bf * 128 + col0 + c * 32, v);
#pragma unroll
          for (int q = 0; q < 32; ++q) o[c * 32 + q] = fmaf(wr, v[q], o[c * 32 + q]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_free[bf]);
      }
    }
    all_ok = __syncthreads_and(all_ok && lv_ok);

    // ---- epilogue
    if (all_ok) {
      if (p.out_f32) {
        if (row_live) {
          float4* dst = reinterpret_cast<float4*>(
              reinterpret_cast<float*>(p.out) + (int64_t)b * p.so_b + (int64_t)(t0 + r) * p.so_t +
              (int64_t)h * p.so_h + col0);
#pragma unroll
          for (int q = 0; q < G::kHalf / 4; ++q)
            dst[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        }
      } else {
        // no MMA reads Q any more: stage the bf16 tile there and store it with TMA
#pragma unroll
        for (int c = 0; c < G::kPanels; ++c) put_row32_bf16(Qb, r, G::kPanels * hh + c, o + c * 32);
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
          for (int pv = 0; pv < G::kPanels; ++pv)
            tma_store_4d(&tmOut, Qb + pv * kPanel, 64 * pv, h, t0, b);
          tma_store_commit();
          tma_store_wait_read();
        }
        __syncwarp();
      }
    } else if (tid == 0) {
      atomicOr(&g_tc_error, 1u);
    }
  } else if (!all_ok && tid == 0) {  // states only
    atomicOr(&g_tc_error, 1u);
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && !all_ok) {
    // after an error: wait (bounded) for the loads still in flight into this CTA's
    // shared memory before it is handed to another CTA
    if (!landed) mbar_wait(bar_load, 0);
    for (int b = 0; b < G::kNodeBufs; ++b)
      for (uint32_t c = (consumed >> (8 * b)) & 255u; c < ints[1 + b]; ++c)
        mbar_wait(&bar_node[b], c & 1);
  }
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

// ------------------------------------------------------------------ host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// [B, T, H, width] bf16 (width 64 or 128), boxes of 128 tokens x 64 features of one
// (b, h); rows past T read as 0 and are not written.
bool make_tokens_map(CUtensorMap* m, const void* base, int B, int T, int H, int width) {
  int64_t s[3];
  dense_strides(s, T, H, width);
  return make_tokens_map_strided(m, base, B, T, H, width, s);
}

bool make_tokens_map_strided(CUtensorMap* m, const void* base, int B, int T, int H, int width,
                             const int64_t* es) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)width, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)es[2] * 2, (cuuint64_t)es[1] * 2, (cuuint64_t)es[0] * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)kTile, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows][width] bf16 matrices (published tile and block states, width = d_v), boxes of
// 128 rows x 64 columns with the 128-byte swizzle.
bool make_rows_map(CUtensorMap* m, const void* base, int64_t rows, int width) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)width * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kTile};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_forward_supported(int64_t dk, int64_t dv, int in_dtype, int /*chunk*/) {
  return in_dtype == LL_BF16 && dk == kD && (dv == 64 || dv == 128);
}

cudaError_t launch_tc_forward(const FwdArgs& a, int out_dtype, cudaStream_t s, StageEvents* ev,
                              bool states_only) {
  const int64_t rows = (int64_t)a.B * a.H * a.N * kD;  // TMA row coordinates are int32
  if (rows > INT32_MAX) return cudaErrorInvalidValue;
  if (a.dk != kD || (a.dv != 64 && a.dv != 128)) return cudaErrorInvalidValue;
  const int dv = (int)a.dv;
  CUtensorMap tmQ, tmK, tmV, tmOut, tmU, tmNode;
  if (!make_tokens_map_strided(&tmQ, a.q, a.B, a.T, a.Hqk, kD, a.sq) ||
      !make_tokens_map_strided(&tmK, a.k, a.B, a.T, a.Hqk, kD, a.sk) ||
      !make_tokens_map_strided(&tmV, a.v, a.B, a.T, a.H, dv, a.sv) ||
      !make_rows_map(&tmU, a.U, rows, dv) ||
      !make_rows_map(&tmNode, a.nodes, rows, dv))
    return cudaErrorInvalidValue;
  if (states_only)
    tmOut = tmV;  // not used: the states-only form writes no output (a.out may be null)
  else if (!make_tokens_map_strided(&tmOut, a.out, a.B, a.T, a.H, dv, a.so))
    return cudaErrorInvalidValue;
  TcParams p;
  p.B = a.B; p.T = a.T; p.H = a.H; p.L = a.L; p.N = a.N; p.hg = a.hg;
  p.log_a = a.log_a; p.lam = a.lam; p.out = a.out;
  p.so_b = a.so[0]; p.so_t = a.so[1]; p.so_h = a.so[2];
  p.U = static_cast<uint8_t*>(a.U);
  p.nodes = static_cast<uint8_t*>(a.nodes);
  p.lgu = a.lg;
  p.nlg = a.nlg;
  p.rdy_u = a.rdy_u;
  p.rdy_n = a.rdy_n;
  p.tick = a.tick;
  p.tag = a.tag;
  p.tag_value = fwd_layout_tag(a.B, a.T, a.H, a.Hqk, a.dv);
  p.out_f32 = out_dtype == LL_F32;
  int levels = 0;  // inter-chunk levels a tile can have: bit length of N-1
  while ((int64_t(1) << levels) < a.N) ++levels;
  // The shared-memory limit is an attribute of the function on each device: set it
  // on every launch (a host-side call), so that every device the library runs on has it.
  auto kernel = dv == 128 ? (states_only ? tc_forward_kernel<128, false> : tc_forward_kernel<128, true>)
                          : (states_only ? tc_forward_kernel<64, false> : tc_forward_kernel<64, true>);
  const size_t smem = states_only ? smem_fused<false>(levels) : smem_fused<true>(levels);
  const cudaError_t attr_err = cudaFuncSetAttribute(
      kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)(states_only ? smem_fused<false>(0) : smem_fused<true>(kMaxChunkLevels - 1)));
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t tiles = (int64_t)a.B * a.H * a.N;
  cudaError_t e;
  if (ev && (e = ev->record(s)) != cudaSuccess) return e;
  // the ready flags and the ticket counter start at zero in every call
  if ((e = cudaMemsetAsync(a.rdy_u, 0, sizeof(uint32_t) * (size_t)(2 * tiles + 1), s)) !=
      cudaSuccess)
    return e;
  kernel<<<dim3((unsigned)tiles), kThreadsF, smem, s>>>(tmQ, tmK, tmV, tmOut, tmU, tmNode, p);
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

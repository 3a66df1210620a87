// Forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), bf16 inputs with
// fp32 accumulation, d_k = d_v = 128, 128-token tiles (the M = 128 datapath of one SM).
//
// The chunked two-stage algorithm (page "论文阅读：Log-Linear Attention", sections 矩阵分解
// and 两阶段计算; page "算力终结者来了！…", section 高效训练算法) with the tile as the chunk:
//
//   tc_chunk_state    per tile i: U_i^T = (w ⊙ V)^T K on tcgen05 (w_s = exp(cs_end - cs_s),
//                     cs = tile-local prefix sums of log a), written fp32 [d_v][d_k], plus the
//                     tile's log decay lg_i.
//   level_scan        (level_scan.cu) Fenwick block totals of tiles, stored bf16 [d_v][d_k]
//                     under the index of their first reader tile.
//   tc_intra_readout  per tile j: S = Q K^T (tcgen05, TMEM), P = S ⊙ exp(cs_t - cs_s) ⊙
//                     lambda[t, l(t,s)] on the causal half (CUDA cores, written back to shared
//                     memory as bf16), O = P V (tcgen05); then for every set bit m-1 of j one
//                     more MMA accumulates (r ⊙ Q) Tot into the same TMEM accumulator, with
//                     r_t = lambda[t, 7+m] exp(cs_t + D), D the log decay from the block's end
//                     to the tile's start.  The lambda-weighted per-level readout is thus
//                     fused into the output accumulator: no per-level output reaches memory.
//
// With 128-token tiles the chunk-pair level log2(C)+1 of a requested C = 64 lies inside a
// tile and is taken in the dense masked product; the sum is the same.
//
// Shared-memory tiles are 128 rows x 128 bf16 stored as two 64-column panels with the
// 128-byte swizzle TMA produces; K-major operands (Q, K, P, scaled Q, block states) and
// MN-major ones (V as the B of P V, V and K in the state GEMM) are described to tcgen05
// with the matching descriptors.  Every mbarrier wait is bounded (see tc_ptx.cuh); a CTA
// whose wait times out raises g_tc_error, skips its remaining MMAs and stores, frees its
// TMEM and exits.
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
constexpr int kMaxChunkLevels = 32;

struct TcParams {
  int B, T, H, L, N;
  const float* log_a;
  const float* lam;
  void* out;
  float* U;
  float* lg;
  int out_f32;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Inclusive prefix sum over the 128 threads of the CTA; red holds 4 floats.
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

// Multiplies row r of a 128 x 128 swizzled bf16 tile by s, from src into dst (same
// physical positions: the swizzle only permutes 16-byte chunks inside a row).
__device__ __forceinline__ void scale_row(const uint8_t* src, uint8_t* dst, int r, float s) {
#pragma unroll
  for (int pnl = 0; pnl < 2; ++pnl) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t off = pnl * kPanel + r * 128 + c * 16;
      uint4 u = *reinterpret_cast<const uint4*>(src + off);
      uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w[k]));
        w[k] = pack_bf16(f.x * s, f.y * s);
      }
      *reinterpret_cast<uint4*>(dst + off) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// ------------------------------------------------------------------ K1: chunk states

__global__ void __launch_bounds__(kThreads, 1)
    tc_chunk_state_kernel(const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* Kb = smem;
  uint8_t* Vb = smem + kOperand;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * kOperand);  // [0] load, [1] mma
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
  float* red = reinterpret_cast<float*>(tslot + 4);
  float* lg_s = red + 4;

  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int t0 = i * kTile;
  const int n = min(kTile, p.T - t0);

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
  if (tid == 0) {
    mbar_arrive_expect_tx(&bars[0], 2 * kOperand);
    tma_load_4d(&tmK, &bars[0], Kb, 0, h, t0, b);
    tma_load_4d(&tmK, &bars[0], Kb + kPanel, 64, h, t0, b);
    tma_load_4d(&tmV, &bars[0], Vb, 0, h, t0, b);
    tma_load_4d(&tmV, &bars[0], Vb + kPanel, 64, h, t0, b);
  }
  const float la = (p.log_a && tid < n) ? p.log_a[((int64_t)b * p.T + t0 + tid) * p.H + h] : 0.f;
  const float cs = block_scan128(la, red);
  if (tid == kThreads - 1) lg_s[0] = cs;  // padding rows add 0: the last prefix is the total
  __syncthreads();
  const float lg = lg_s[0];
  const float w = tid < n ? expf(lg - cs) : 0.f;

  bool ok = mbar_wait(&bars[0], 0);
  if (ok) scale_row(Vb, Vb, tid, w);
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
  bool ok2 = all_ok && mbar_wait(&bars[1], 0);
  tc_fence_after();
  if (__syncthreads_and(ok2)) {
    float* U = p.U + (((int64_t)b * p.H + h) * p.N + i) * (int64_t)(kD * kD) + (int64_t)tid * kD;
#pragma unroll
    for (int c = 0; c < kD / 32; ++c) {
      float v[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c * 32, v);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        reinterpret_cast<float4*>(U + c * 32)[q] =
            make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
    if (tid == 0) p.lg[((int64_t)b * p.H + h) * p.N + i] = lg;
  } else if (tid == 0) {
    atomicOr(&g_tc_error, 1u);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

// ------------------------------------------------------------------ K3: intra + readout

__global__ void __launch_bounds__(kThreads, 2)
    tc_intra_readout_kernel(const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV,
                            const __grid_constant__ CUtensorMap tmNode, TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* Qb = smem;
  uint8_t* Kb = smem + kOperand;      // K, then P, then the scaled Q of each level
  uint8_t* Vb = smem + 2 * kOperand;  // V, then the block state of each level
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 3 * kOperand);  // load, mma, node
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3);
  float* red = reinterpret_cast<float*>(tslot + 4);
  float* cs_s = red + 4;                       // [128]
  float* lam_s = cs_s + kTile;                 // [128][kLamStride]
  float* Dm = lam_s + kTile * kLamStride;      // [kMaxChunkLevels]

  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = j * kTile;
  const int n = min(kTile, p.T - t0);
  const int64_t bh = (int64_t)b * p.H + h;
  const int64_t row = ((int64_t)b * p.T + t0 + tid) * p.H + h;  // (b, t, h) of this thread

  if (warp == 0) {
    tmem_alloc(tslot, 256);
    tmem_relinquish();
  }
  if (tid == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    prefetch_tensormap(&tmNode);
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_init(&bars[2], 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  if (tid == 0) {
    mbar_arrive_expect_tx(&bars[0], 3 * kOperand);
    tma_load_4d(&tmQ, &bars[0], Qb, 0, h, t0, b);
    tma_load_4d(&tmQ, &bars[0], Qb + kPanel, 64, h, t0, b);
    tma_load_4d(&tmK, &bars[0], Kb, 0, h, t0, b);
    tma_load_4d(&tmK, &bars[0], Kb + kPanel, 64, h, t0, b);
    tma_load_4d(&tmV, &bars[0], Vb, 0, h, t0, b);
    tma_load_4d(&tmV, &bars[0], Vb + kPanel, 64, h, t0, b);
  }
  // per-row decay prefix and intra-tile lambdas, while the tiles are in flight
  const float la = (p.log_a && tid < n) ? p.log_a[row] : 0.f;
  const float cs = block_scan128(la, red);
  cs_s[tid] = cs;
#pragma unroll
  for (int l = 0; l < kIntraLevels; ++l)
    lam_s[tid * kLamStride + l] = (tid < n && l < p.L) ? p.lam[row * p.L + l] : 0.f;
  // log decay from the end of each inter-chunk block to the start of this tile
  if (warp == 0) {
    const float* lgp = p.lg + bh * p.N;
    for (int m = 1; m < kMaxChunkLevels && (1 << (m - 1)) <= j; ++m) {
      if (!((j >> (m - 1)) & 1)) continue;
      const int c = (j >> (m - 1)) << (m - 1);
      float s = 0.f;
      for (int i = c + lane; i < j; i += 32) s += lgp[i];
      s = warp_sum(s);
      if (lane == 0) Dm[m] = s;
    }
  }
  __syncthreads();

  bool ok = mbar_wait(&bars[0], 0);
  bool all_ok = __syncthreads_and(ok);
  // S = Q K^T
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
    mma_commit(&bars[1]);
  }
  uint32_t mma_phase = 0;
  ok = all_ok && mbar_wait(&bars[1], mma_phase);
  mma_phase ^= 1;
  tc_fence_after();
  all_ok = __syncthreads_and(ok);
  // P = S ⊙ exp(cs_t - cs_s) ⊙ lambda[t, l(t, s)] on s <= t, as bf16 into Kb (K-major)
  if (all_ok) {
    const uint32_t tq = (uint32_t)(t0 + tid);
    const float* lam_r = lam_s + tid * kLamStride;
#pragma unroll 1
    for (int c = 0; c < kTile / 32; ++c) {
      float sv[32];
      tmem_ld32(tmem + lane_base + c * 32, sv);
      uint32_t pk[16];
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        float pr[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int s = c * 32 + k + u;
          float v = 0.f;
          if (s <= tid && tid < n) {
            const int lvl = fenwick_level(tq, (uint32_t)(t0 + s));
            v = sv[k + u] * lam_r[lvl] * __expf(cs - cs_s[s]);
          }
          pr[u] = v;
        }
        pk[k >> 1] = pack_bf16(pr[0], pr[1]);
      }
      uint8_t* panel = Kb + (c >> 1) * kPanel;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(panel + sw128_offset(tid, (c & 1) * 4 + q)) =
            make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  // O = P V  (V MN-major as B)
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
    mma_commit(&bars[1]);
  }
  // inter-chunk levels: O += (r ⊙ Q) Tot for every set bit m-1 of j
  uint32_t node_phase = 0;
  for (int m = 1; m < kMaxChunkLevels && (1 << (m - 1)) <= j; ++m) {
    if (!((j >> (m - 1)) & 1)) continue;
    ok = all_ok && mbar_wait(&bars[1], mma_phase);  // previous MMA released Kb and Vb
    mma_phase ^= 1;
    all_ok = __syncthreads_and(ok);
    if (!all_ok) break;
    const int c = (j >> (m - 1)) << (m - 1);
    if (tid == 0) {
      const int r0 = (int)((bh * p.N + c) * kD);
      mbar_arrive_expect_tx(&bars[2], kOperand);
      tma_load_2d(&tmNode, &bars[2], Vb, 0, r0);
      tma_load_2d(&tmNode, &bars[2], Vb + kPanel, 64, r0);
    }
    const float r = tid < n ? p.lam[row * p.L + kTileLc + m] * __expf(cs + Dm[m]) : 0.f;
    scale_row(Qb, Kb, tid, r);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    ok = mbar_wait(&bars[2], node_phase);
    node_phase ^= 1;
    all_ok = __syncthreads_and(ok);
    if (!all_ok) break;
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16(128, 128, 0, 0);
      const uint32_t aa = smem_u32(Kb), sa = smem_u32(Vb);
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
        mma_bf16(tmem + 128, smem_desc_sw128(aa + off, 16, 1024),
                 smem_desc_sw128(sa + off, 16, 1024), idesc, 1);
      }
      mma_commit(&bars[1]);
    }
  }
  ok = all_ok && mbar_wait(&bars[1], mma_phase);
  tc_fence_after();
  all_ok = __syncthreads_and(ok);
  if (all_ok) {
    // every lane executes the warp-wide TMEM loads; padding rows skip only the stores
    const int64_t obase = row * kD;
#pragma unroll 1
    for (int c = 0; c < kD / 32; ++c) {
      float v[32];
      tmem_ld32(tmem + lane_base + 128 + c * 32, v);
      if (tid >= n) continue;
      if (p.out_f32) {
        float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + obase + c * 32);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      } else {
        uint4* o =
            reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + obase + c * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          o[q] = make_uint4(pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                            pack_bf16(v[8 * q + 4], v[8 * q + 5]),
                            pack_bf16(v[8 * q + 6], v[8 * q + 7]));
      }
    }
  }
  if (!all_ok && tid == 0) atomicOr(&g_tc_error, 1u);
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

// [B, T, H, 128] bf16, boxes of 128 tokens x 64 features of one (b, h); rows past T read 0.
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

// Block states [rows = B*H*N*128][128] bf16, boxes of 128 rows x 64 columns.
bool make_nodes_map(CUtensorMap* m, const void* base, int64_t rows) {
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

constexpr size_t kSmemK1 = 2 * kOperand + 1024 + 256;
constexpr size_t kSmemK3 =
    3 * kOperand + 1024 + 64 + 4 * (4 + kTile + kTile * kLamStride + kMaxChunkLevels);

}  // namespace

bool tc_forward_supported(int64_t dk, int64_t dv, int in_dtype, int /*chunk*/) {
  return in_dtype == LL_BF16 && dk == kD && dv == kD;
}

cudaError_t launch_tc_forward(const FwdArgs& a, int out_dtype, cudaStream_t s, StageEvents* ev) {
  CUtensorMap tmQ, tmK, tmV, tmNode;
  if (!make_tokens_map(&tmQ, a.q, a.B, a.T, a.H) || !make_tokens_map(&tmK, a.k, a.B, a.T, a.H) ||
      !make_tokens_map(&tmV, a.v, a.B, a.T, a.H) ||
      !make_nodes_map(&tmNode, a.nodes, (int64_t)a.B * a.H * a.N * kD))
    return cudaErrorInvalidValue;
  TcParams p;
  p.B = a.B; p.T = a.T; p.H = a.H; p.L = a.L; p.N = a.N;
  p.log_a = a.log_a; p.lam = a.lam; p.out = a.out; p.U = a.U; p.lg = a.lg;
  p.out_f32 = out_dtype == LL_F32;
  cudaError_t e;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(tc_chunk_state_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemK1);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(tc_intra_readout_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemK3);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const dim3 grid(a.N, a.H, a.B);
  if (ev && (e = ev->record(s)) != cudaSuccess) return e;
  tc_chunk_state_kernel<<<grid, kThreads, kSmemK1, s>>>(tmK, tmV, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (ev && (e = ev->record(s)) != cudaSuccess) return e;
  if (a.N > 1) {
    if ((e = launch_level_scan(a, /*bf16_nodes=*/true, s)) != cudaSuccess) return e;
    if (ev && (e = ev->record(s)) != cudaSuccess) return e;
  }
  tc_intra_readout_kernel<<<grid, kThreads, kSmemK3, s>>>(tmQ, tmK, tmV, tmNode, p);
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

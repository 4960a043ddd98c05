// Dense projections of the drafter: out = X . W^T, split along K.
//
// bf16: a tcgen05 tensor-core kernel.  The weight matrix streams through the
// MMA's M side (128 rows per tile) and the few activation rows ride on N
// (16..256), so an M = 16 draft block still fills the 128-row MMA (swap-AB).
// One thread issues TMA tile loads into a STAGES-deep shared-memory ring,
// one thread issues tcgen05.mma into a TMEM accumulator, and all four warps
// read the accumulator back with tcgen05.ld in the epilogue.  Weights are
// loaded with an L2 evict-first hint: each byte is used once per launch.
//
// Activations may come as an exact pair of bf16 terms (x = hi + lo, the
// residual of rounding x to bf16 rounded again): the kernel then issues two
// MMAs per k-slice into the same accumulator, W.hi + W.lo, so the product
// keeps about 16 significant bits of x while both MMA operands stay bf16.
// The weight-streaming GEMMs are HBM-bound, so the second MMA is hidden.
//
// fp32: a plain SIMT kernel (the fp32 workloads need fp32 products; TF32
// would not meet their tolerance).
#include <algorithm>
#include <cstdio>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "internal.h"

namespace dflash {

// --------------------------------------------------------------- tcgen05 kernel

template <int BN, bool SPLIT>
struct TcCfg {
  static constexpr int W_BYTES = kTileN * kTileK * 2;  // 16 KB
  static constexpr int X_BYTES = BN * kTileK * 2;
  static constexpr int STAGE_BYTES = W_BYTES + (SPLIT ? 2 : 1) * X_BYTES;
  // BN <= 64: two CTAs per SM; wider tiles: one CTA with a deeper ring
  static constexpr int BUDGET = BN <= 64 ? 110 * 1024 : 200 * 1024;
  static constexpr int STAGES = (BUDGET / STAGE_BYTES) < 8 ? (BUDGET / STAGE_BYTES) : 8;
  static constexpr int TMEM_COLS = BN < 32 ? 32 : BN;
  static constexpr int SMEM = 1024 /*align slack*/ + STAGES * STAGE_BYTES + 256 /*barriers*/ +
                              3 * 4 * BN * 4 /*LM-head reduction*/;
  static_assert(STAGES >= 2, "pipeline too shallow");
  // the own tile plus the reduced slice (at most half the rows, splits >= 2) fit in the stage ring
  static_assert(BN * 128 * 4 * 3 / 2 <= STAGES * STAGE_BYTES, "epilogue tiles must fit in the stage ring");
};

struct TcParams {
  int M, N;
  int n_kb, kb_per_split, splits;
  float* out;  // split-K partial planes [splits][M][ldo]
  long long split_stride;
  int ldo;
  const int* m_valid;
  int* status;
  EpiArgs epi;
  LmPartials lm;
  float* logits;
  long long ld_logits;
  const int* skip_rows;
};

template <int BN, bool LMHEAD, bool SPLIT>
__global__ void __launch_bounds__(128) k_gemm_tc(const __grid_constant__ CUtensorMap tmW,
                                                 const __grid_constant__ CUtensorMap tmX,
                                                 const __grid_constant__ CUtensorMap tmXlo, const TcParams p) {
  using C = TcCfg<BN, SPLIT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW = smem;                                   // [STAGES][W tile]
  uint8_t* sX = smem + C::STAGES * C::W_BYTES;          // [STAGES][X tile (+ X lo tile)]
  constexpr int XS = (SPLIT ? 2 : 1) * C::X_BYTES;      // X bytes per stage
  uint64_t* full = reinterpret_cast<uint64_t*>(sX + C::STAGES * XS);
  uint64_t* empty = full + C::STAGES;
  uint64_t* accb = empty + C::STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accb + 1);
  int* s_prog = reinterpret_cast<int*>(tmem_slot + 1);  // [0] stages issued, [1] stages consumed
  float* red = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE_BYTES + 256);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kTileN, m0 = blockIdx.y * BN, split = blockIdx.z;
  if (p.m_valid != nullptr && m0 >= __ldg(p.m_valid)) return;  // uniform: nothing allocated yet
  const int kb0 = split * p.kb_per_split;
  const int kb1 = min(p.n_kb, kb0 + p.kb_per_split);
  const int nkb = kb1 - kb0;

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    if (SPLIT) tma_prefetch_desc(&tmXlo);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accb, 1);
    s_prog[0] = 0;
    s_prog[1] = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      for (int it = 0; it < nkb; ++it) {
        const int s = it % C::STAGES;
        const uint32_t ph = (it / C::STAGES) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, p.status)) break;
        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
        const int kx = (kb0 + it) * kTileK;
        tma_load_2d_hint(sW + s * C::W_BYTES, &tmW, &full[s], kx, n0, pol);
        tma_load_2d(sX + s * XS, &tmX, &full[s], kx, m0);
        if (SPLIT) tma_load_2d(sX + s * XS + C::X_BYTES, &tmXlo, &full[s], kx, m0);
        s_prog[0] = it + 1;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = mma_idesc_bf16_f32(kTileN, BN);
      for (int it = 0; it < nkb; ++it) {
        const int s = it % C::STAGES;
        const uint32_t ph = (it / C::STAGES) & 1;
        if (!mbar_wait(&full[s], ph, p.status)) break;
        tc_fence_after();
        const uint32_t aW = smem_u32(sW + s * C::W_BYTES);
        const uint32_t aX = smem_u32(sX + s * XS);
#pragma unroll
        for (int k = 0; k < kTileK / 16; ++k) {
          const uint64_t dW = sw128_kmajor_desc(aW + 32 * k);
          tc_mma_bf16(tmem, dW, sw128_kmajor_desc(aX + 32 * k), idesc, (it | k) != 0 ? 1u : 0u);
          if (SPLIT) tc_mma_bf16(tmem, dW, sw128_kmajor_desc(aX + C::X_BYTES + 32 * k), idesc, 1u);
        }
        tc_commit(&empty[s]);
        s_prog[1] = it + 1;
      }
      tc_commit(accb);
    }
    __syncwarp();
  }

  // ---- epilogue: TMEM lane (32*warp + lane) holds weight row n, columns = activation rows
  mbar_wait(accb, 0, p.status);
  __syncwarp();  // lanes may leave the poll loop at different times; tcgen05.ld is warp-aligned
  tc_fence_after();
  __syncthreads();
  if (threadIdx.x == 0 && s_prog[1] < s_prog[0]) {
    // a wait gave up: let every copy still in flight land before the ring is reused
    for (int it = s_prog[1]; it < s_prog[0]; ++it) mbar_wait(&full[it % C::STAGES], (it / C::STAGES) & 1, p.status);
  }
  const int n = n0 + warp * 32 + lane;
  const bool nv = n < p.N;
  const uint32_t tbase = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  if constexpr (!LMHEAD) {
    // the accumulator goes to a [BN][128] fp32 tile in the (now idle) stage ring
    float* tile = reinterpret_cast<float*>(smem);
    __syncthreads();
#pragma unroll 1
    for (int c = 0; c < BN; c += 16) {
      float v[16];
      tc_ld_32x32b_x16(tbase + c, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) tile[(c + j) * 128 + warp * 32 + lane] = v[j];
    }
    tc_fence_before();
    __syncthreads();
    const int t = threadIdx.x;
    if (p.epi.kind == EPI_NONE) {
      float* o = p.out + split * p.split_stride;
      for (int j = 0; j < BN && m0 + j < p.M; ++j)
        if (nv) o[static_cast<long long>(m0 + j) * p.ldo + n] = tile[j * 128 + t];
    }
    if (p.epi.kind != EPI_NONE) {
      if (p.splits == 1) {
        apply_epilogue<__nv_bfloat16, __half>(p.epi, tile, m0, BN, n0);
      } else {
        // split-K reduction inside the cluster of this tile's `splits` CTAs:
        // each CTA sums a contiguous slice of the rows over every CTA's tile
        // (distributed shared memory, split order) and finishes those rows
        cluster_sync_all();
        const int S = p.splits, cr = static_cast<int>(cluster_ctarank());
        const int rpr = (BN + S - 1) / S;
        const int r_begin = min(BN, cr * rpr), r_end = min(BN, r_begin + rpr);
        float* sub = tile + BN * 128;
        const uint32_t tile_s = smem_u32(tile);
        for (int e = t; e < (r_end - r_begin) * 32; e += 128) {
          const int j = r_begin + e / 32, c4 = (e % 32) * 4;
          const uint32_t off = static_cast<uint32_t>((j * 128 + c4) * 4);
          float4 acc = ld_dsmem_f4(dsmem_map(tile_s + off, 0));
          for (int r = 1; r < S; ++r) {
            const float4 v = ld_dsmem_f4(dsmem_map(tile_s + off, r));
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
          }
          *reinterpret_cast<float4*>(sub + (j - r_begin) * 128 + c4) = acc;
        }
        cluster_sync_all();  // no CTA's tile is read after this point
        if (r_end > r_begin) apply_epilogue<__nv_bfloat16, __half>(p.epi, sub, m0 + r_begin, r_end - r_begin, n0);
      }
    }
  } else {
#pragma unroll 1
    for (int c = 0; c < BN; c += 16) {
      float v[16];
      tc_ld_32x32b_x16(tbase + c, v);
#pragma unroll 1
      for (int j = 0; j < 16; ++j) {
        const int m = m0 + c + j;
        const float val = nv ? v[j] : -INFINITY;
        if (p.logits != nullptr && nv && m < p.M && (p.skip_rows == nullptr || p.skip_rows[m] == 0))
          p.logits[m * p.ld_logits + n] = val;
        float mx = val;
        int ix = n;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float om = __shfl_xor_sync(0xffffffffu, mx, o);
          const int oi = __shfl_xor_sync(0xffffffffu, ix, o);
          if (om > mx || (om == mx && oi < ix)) {
            mx = om;
            ix = oi;
          }
        }
        const float e = nv ? expf(val - mx) : 0.f;
        const float se = warp_sum(e);
        if (lane == 0) {
          red[(0 * 4 + warp) * BN + c + j] = mx;
          red[(1 * 4 + warp) * BN + c + j] = se;
          red[(2 * 4 + warp) * BN + c + j] = __int_as_float(ix);
        }
      }
    }
    __syncthreads();
    for (int j = threadIdx.x; j < BN; j += blockDim.x) {
      const int m = m0 + j;
      if (m >= p.M) continue;
      float mx = red[0 * BN + j];
      int ix = __float_as_int(red[2 * 4 * BN + j]);
      for (int w = 1; w < 4; ++w) {  // warps cover increasing columns: strict > keeps the lowest id
        const float wm = red[(0 * 4 + w) * BN + j];
        if (wm > mx) {
          mx = wm;
          ix = __float_as_int(red[(2 * 4 + w) * BN + j]);
        }
      }
      float se = 0.f;
      for (int w = 0; w < 4; ++w) {
        const float wm = red[(0 * 4 + w) * BN + j];
        if (wm > -INFINITY) se += red[(1 * 4 + w) * BN + j] * expf(wm - mx);
      }
      const long long o = static_cast<long long>(m) * p.lm.n_tiles + blockIdx.x;
      p.lm.mx[o] = mx;
      p.lm.se[o] = se;
      p.lm.idx[o] = ix;
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Finishes an fp32 projection written by the SIMT kernel: one CTA per
// (128-column, 16-row) tile runs the same epilogue as the tensor-core path.
__global__ void __launch_bounds__(128) k_epilogue_apply_f32(const float* __restrict__ y, int M, int N, EpiArgs e) {
  __shared__ float tile[16 * 128];
  const int n0 = blockIdx.x * 128, m0 = blockIdx.y * 16, t = threadIdx.x;
  for (int j = 0; j < 16; ++j) {
    const int m = m0 + j, n = n0 + t;
    tile[j * 128 + t] = (m < M && n < N) ? y[static_cast<long long>(m) * N + n] : 0.f;
  }
  __syncthreads();
  apply_epilogue<float, float>(e, tile, m0, 16, n0);
}

// --------------------------------------------------------------- fp32 SIMT kernel

__global__ void __launch_bounds__(256) k_gemm_f32(const float* __restrict__ W, const float* __restrict__ X,
                                                  float* __restrict__ out, int M, int N, int K, int ldo,
                                                  const int* m_valid) {
  __shared__ float sW[16][65];
  __shared__ float sX[16][65];
  const int n0 = blockIdx.x * 64, m0 = blockIdx.y * 64;
  if (m_valid != nullptr && m0 >= *m_valid) return;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int i = threadIdx.x; i < 1024; i += 256) {
      const int r = i >> 4, kk = i & 15;
      sW[kk][r] = (n0 + r < N && k0 + kk < K) ? W[static_cast<long long>(n0 + r) * K + k0 + kk] : 0.f;
      sX[kk][r] = (m0 + r < M && k0 + kk < K) ? X[static_cast<long long>(m0 + r) * K + k0 + kk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = sX[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = sW[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
      if (m < M && n < N) out[static_cast<long long>(m) * ldo + n] = acc[i][j];
    }
}

// --------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// A bf16 [rows][cols] row-major matrix as a TMA map with boxes of box_rows x 64
// and 128-byte swizzling; out-of-range rows and columns read as zero.
static bool get_tmap(dflash_ctx* c, const void* ptr, int rows, int cols, int box_rows, CUtensorMap* out) {
  for (auto& e : c->tmaps)
    if (e.ptr == ptr && e.rows == rows && e.cols == cols && e.box_rows == box_rows) {
      *out = e.map;
      return true;
    }
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  TmapEntry e;
  e.ptr = ptr;
  e.rows = rows;
  e.cols = cols;
  e.box_rows = box_rows;
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = fn(&e.map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), gdim, gstride, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  c->tmaps.push_back(e);
  *out = e.map;
  return true;
}

int gemm_kb(int K) { return (K + kTileK - 1) / kTileK; }

template <int BN, bool LM, bool SPLIT>
static cudaError_t launch_tc(dflash_ctx* c, const GemmLaunch& g, const CUtensorMap& tw, const CUtensorMap& tx,
                             const CUtensorMap& txlo, cudaStream_t s) {
  using C = TcCfg<BN, SPLIT>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(k_gemm_tc<BN, LM, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  TcParams p;
  const int n_kb = gemm_kb(g.K);
  p.M = g.M;
  p.N = g.N;
  p.n_kb = n_kb;
  p.kb_per_split = (n_kb + g.splits - 1) / g.splits;
  p.splits = g.splits;
  p.epi = g.epi;
  p.out = g.out;
  p.split_stride = g.split_stride;
  p.ldo = g.ldo;
  p.m_valid = g.m_valid;
  p.status = c->status;
  p.lm = g.lm;
  p.logits = g.logits;
  p.ld_logits = g.ld_logits;
  p.skip_rows = g.skip_rows;
  // splits come from gemm_splits: every split owns at least one k-block
  dim3 grid((g.N + kTileN - 1) / kTileN, (g.M + BN - 1) / BN, g.splits);
  if (LM || g.epi.kind == EPI_NONE || g.splits == 1) {
    k_gemm_tc<BN, LM, SPLIT><<<grid, 128, C::SMEM, s>>>(tw, tx, txlo, p);
    return cudaGetLastError();
  }
  // the splits of one output tile form a thread-block cluster (reduced over DSMEM)
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = dim3(128);
  lc.dynamicSmemBytes = C::SMEM;
  lc.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 1;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = g.splits;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, k_gemm_tc<BN, LM, SPLIT>, tw, tx, txlo, p);
}

template <bool SPLIT>
static cudaError_t launch_tc_bn(dflash_ctx* c, const GemmLaunch& g, int bn, const CUtensorMap& tw,
                                const CUtensorMap& tx, const CUtensorMap& txlo, cudaStream_t s) {
  const bool lm = g.lm.mx != nullptr;
  switch (bn) {
    case 16:
      return lm ? launch_tc<16, true, SPLIT>(c, g, tw, tx, txlo, s) : launch_tc<16, false, SPLIT>(c, g, tw, tx, txlo, s);
    case 32:
      return lm ? launch_tc<32, true, SPLIT>(c, g, tw, tx, txlo, s) : launch_tc<32, false, SPLIT>(c, g, tw, tx, txlo, s);
    case 64:
      return lm ? launch_tc<64, true, SPLIT>(c, g, tw, tx, txlo, s) : launch_tc<64, false, SPLIT>(c, g, tw, tx, txlo, s);
    case 128:
      return lm ? launch_tc<128, true, SPLIT>(c, g, tw, tx, txlo, s)
                : launch_tc<128, false, SPLIT>(c, g, tw, tx, txlo, s);
    default:
      if constexpr (SPLIT) return cudaErrorInvalidValue;
      else
        return lm ? launch_tc<256, true, false>(c, g, tw, tx, txlo, s)
                  : launch_tc<256, false, false>(c, g, tw, tx, txlo, s);
  }
}

// How many clusters of `cluster` CTAs of the projection kernel (tile width
// bn, hi+lo operands or not) can be resident at once on this device.  GPCs
// have uneven SM counts, so this is not simply SMs x CTAs-per-SM / cluster.
template <int BN, bool SPLIT>
static int max_clusters_t(int cluster) {
  using C = TcCfg<BN, SPLIT>;
  if (cudaFuncSetAttribute(k_gemm_tc<BN, false, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
      cudaSuccess)
    return 0;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(1, 1, cluster);
  lc.blockDim = dim3(128);
  lc.dynamicSmemBytes = C::SMEM;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 1;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = cluster;
  lc.attrs = at;
  lc.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_gemm_tc<BN, false, SPLIT>, &lc) != cudaSuccess) return 0;
  return n;
}

int gemm_max_clusters(int bn, bool split, int cluster) {
  static int cache[2][5][9] = {};  // [split][log2(bn/16)][cluster]
  int bi = 0;
  while ((16 << bi) < bn && bi < 4) ++bi;
  if (cluster < 1 || cluster > 8) return 0;
  int& c = cache[split ? 1 : 0][bi][cluster];
  if (c == 0) {
    switch (bi) {
      case 0: c = split ? max_clusters_t<16, true>(cluster) : max_clusters_t<16, false>(cluster); break;
      case 1: c = split ? max_clusters_t<32, true>(cluster) : max_clusters_t<32, false>(cluster); break;
      case 2: c = split ? max_clusters_t<64, true>(cluster) : max_clusters_t<64, false>(cluster); break;
      case 3: c = split ? max_clusters_t<128, true>(cluster) : max_clusters_t<128, false>(cluster); break;
      default: c = split ? 0 : max_clusters_t<256, false>(cluster); break;
    }
    if (c <= 0) c = -1;
  }
  return c;
}

// Split-K count for `n_tiles` output tiles of width bn: the largest split
// count S <= 8 (a portable cluster) such that all n_tiles clusters of S CTAs
// are resident at once, with at least 4 k-blocks per split; normalised so that
// every split owns at least one k-block.
int gemm_splits(int n_tiles, int n_kb, int bn, bool split) {
  int s = std::min(8, std::max(1, n_kb / 4));
  for (; s > 1; --s)
    if (n_tiles <= gemm_max_clusters(bn, split, s)) break;
  const int per = (n_kb + s - 1) / s;
  return (n_kb + per - 1) / per;
}

int gemm_bn(int M, bool split) {
  const int cap = split ? 128 : 256;
  int bn = 16;
  while (bn < M && bn < cap) bn *= 2;
  return bn;
}

cudaError_t gemm_launch(dflash_ctx* c, const GemmLaunch& g, cudaStream_t s) {
  if (c->cfg.dtype == DFLASH_F32) {
    dim3 grid((g.N + 63) / 64, (g.M + 63) / 64);
    k_gemm_f32<<<grid, 256, 0, s>>>(static_cast<const float*>(g.W), static_cast<const float*>(g.X), g.out, g.M,
                                    g.N, g.K, g.ldo, g.m_valid);
    if (g.epi.kind != EPI_NONE) {
      dim3 eg((g.N + 127) / 128, (g.M + 15) / 16);
      k_epilogue_apply_f32<<<eg, 128, 0, s>>>(g.out, g.M, g.N, g.epi);
    }
    return cudaGetLastError();
  }
  const bool split = g.X_lo != nullptr;
  const int bn = gemm_bn(g.M, split);
  CUtensorMap tw, tx, txlo;
  if (!get_tmap(c, g.W, g.N, g.K, kTileN, &tw) || !get_tmap(c, g.X, g.M_alloc, g.K, bn, &tx))
    return cudaErrorInvalidValue;
  if (split) {
    if (!get_tmap(c, g.X_lo, g.M_alloc, g.K, bn, &txlo)) return cudaErrorInvalidValue;
    return launch_tc_bn<true>(c, g, bn, tw, tx, txlo, s);
  }
  return launch_tc_bn<false>(c, g, bn, tw, tx, tx, s);
}

// ---------------------------------------------------------------- launch without a map cache

// The same projection launch with both tensor maps encoded on the stack: no
// map cache and no host heap, for the entry point that must not allocate.
static bool encode_tmap_bf16(const void* ptr, int rows, int cols, int box_rows, CUtensorMap* out) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estride[2] = {1, 1};
  return fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), gdim, gstride, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t gemm_launch_uncached(int* status, const GemmLaunch& g, cudaStream_t s) {
  dflash_ctx tmp;  // holds only the status pointer; its containers stay empty
  tmp.cfg = dflash_config{};
  tmp.cfg.dtype = DFLASH_BF16;
  tmp.status = status;
  const bool split = g.X_lo != nullptr;
  const int bn = gemm_bn(g.M, split);
  CUtensorMap tw, tx, txlo;
  if (!encode_tmap_bf16(g.W, g.N, g.K, kTileN, &tw) || !encode_tmap_bf16(g.X, g.M_alloc, g.K, bn, &tx))
    return cudaErrorInvalidValue;
  if (split) {
    if (!encode_tmap_bf16(g.X_lo, g.M_alloc, g.K, bn, &txlo)) return cudaErrorInvalidValue;
    return launch_tc_bn<true>(&tmp, g, bn, tw, tx, txlo, s);
  }
  return launch_tc_bn<false>(&tmp, g, bn, tw, tx, tx, s);
}

}  // namespace dflash

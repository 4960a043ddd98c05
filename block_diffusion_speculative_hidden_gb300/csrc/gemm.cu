// Dense projections of the drafter: out = X . W^T, split along K.
//
// bf16 and E4M3 weights: the tcgen05 kernel of gemm_kernel.cuh (the E4M3
// variants are instantiated in gemm_w8.cu).  fp32: a plain SIMT kernel (the
// fp32 workloads need fp32 products; TF32 would not meet their tolerance).
// Host side: tensor maps, split-K sizing, the launch dispatch.
#include <algorithm>
#include <cstdio>
#include <cudaTypedefs.h>

#include "gemm_persist.cuh"

namespace dflash {

// --------------------------------------------------------------- tcgen05 kernel

// Finishes an fp32 projection written by the SIMT kernel: one CTA per
// (128-column, 16-row) tile runs the same epilogue as the tensor-core path.
__global__ void __launch_bounds__(128) k_epilogue_apply_f32(const float* __restrict__ y, int M, int N, EpiArgs e) {
  __shared__ float tile[16 * 128];
  __shared__ float rs[16], scratch[4 * 16];
  const int n0 = blockIdx.x * 128, m0 = blockIdx.y * 16, t = threadIdx.x;
  for (int j = 0; j < 16; ++j) {
    const int m = m0 + j, n = n0 + t;
    tile[j * 128 + t] = (m < M && n < N) ? y[static_cast<long long>(m) * N + n] : 0.f;
  }
  if (e.ss_in != nullptr && t < 16) rs[t] = m0 + t < M ? norm_row_scale(e, m0 + t) : 0.f;
  __syncthreads();
  apply_epilogue<float, float>(e, tile, m0, 16, n0, e.ss_in != nullptr ? rs : nullptr, nullptr, scratch);
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

// A [rows][cols] row-major matrix as a TMA map with boxes of box_rows rows of
// 128 bytes (bf16, kind 0: 64 columns; E4M3 codes, kind 1: 128 columns) and
// 128-byte swizzling; out-of-range rows and columns read as zero.
static bool encode_tmap(const void* ptr, int rows, int cols, int box_rows, int kind, CUtensorMap* out) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const int esize = kind == 1 ? 1 : 2;
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(cols) * esize};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kind == 1 ? 2 * kTileK : kTileK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estride[2] = {1, 1};
  return fn(out, kind == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(ptr), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// encode_tmap through the context's cache (maps are keyed by pointer, shape,
// box and kind).
static bool get_tmap(dflash_ctx* c, const void* ptr, int rows, int cols, int box_rows, CUtensorMap* out,
                     int kind = 0) {
  for (auto& e : c->tmaps)
    if (e.ptr == ptr && e.rows == rows && e.cols == cols && e.box_rows == box_rows && e.kind == kind) {
      *out = e.map;
      return true;
    }
  TmapEntry e;
  e.ptr = ptr;
  e.rows = rows;
  e.cols = cols;
  e.box_rows = box_rows;
  e.kind = kind;
  if (!encode_tmap(ptr, rows, cols, box_rows, kind, &e.map)) return false;
  c->tmaps.push_back(e);
  *out = e.map;
  return true;
}

int gemm_kb(int K) { return (K + kTileK - 1) / kTileK; }

// k-blocks per split for a requested split count: every split but the last
// owns the same whole number of pipeline stages (two k-blocks for E4M3
// weights), the last at least one k-block.
int gemm_kb_per_split(int n_kb, int splits, bool w8) {
  int per = (n_kb + splits - 1) / splits;
  if (w8) per += per & 1;
  return per;
}

int gemm_normalize_splits(int n_kb, int splits, bool w8) {
  const int per = gemm_kb_per_split(n_kb, std::max(1, splits), w8);
  return (n_kb + per - 1) / per;
}

// How many CTAs of the projection kernel (tile width bn, hi+lo operands or
// not, E4M3 weights or not) one SM holds at once.  Shared memory and TMEM are
// the limits that bind (128-192 threads, few registers).
template <int BN, bool SPLIT, bool W8>
static int blocks_per_sm_t() {
  using C = TcCfg<BN, SPLIT, W8>;
  int dev = 0, per_sm = 0, reserved = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  const int by_smem = per_sm / (C::SMEM + reserved);
  const int by_tmem = 512 / C::TMEM_COLS;
  return std::max(1, std::min(by_smem, by_tmem));
}

template <bool W8>
static int blocks_per_sm_w(int bi, bool split) {
  switch (bi) {
    case 0: return split ? blocks_per_sm_t<16, true, W8>() : blocks_per_sm_t<16, false, W8>();
    case 1: return split ? blocks_per_sm_t<32, true, W8>() : blocks_per_sm_t<32, false, W8>();
    case 2: return split ? blocks_per_sm_t<64, true, W8>() : blocks_per_sm_t<64, false, W8>();
    case 3: return split ? blocks_per_sm_t<128, true, W8>() : blocks_per_sm_t<128, false, W8>();
    default:
      if constexpr (W8) return blocks_per_sm_t<128, false, true>();  // E4M3 tiles stop at 128 rows
      else return split ? 1 : blocks_per_sm_t<256, false, false>();
  }
}

int gemm_blocks_per_sm(int bn, bool split, bool w8) {
  static int cache[2][2][5] = {};  // [w8][split][log2(bn/16)]
  int bi = 0;
  while ((16 << bi) < bn && bi < 4) ++bi;
  int& c = cache[w8 ? 1 : 0][split ? 1 : 0][bi];
  if (c == 0) c = w8 ? blocks_per_sm_w<true>(bi, split) : blocks_per_sm_w<false>(bi, split);
  return c;
}

// Split-K count for `n_tiles` output tiles of width bn.  A CTA streams its
// weights at a fraction of the HBM bandwidth an SM can draw, so the grid
// must keep every SM streaming: aim for about 1.5 CTAs per SM (all resident
// at once, at most max_ctas when positive; measured on the c2 round against
// 1.0, 1.25, 1.75 and 2.0), with at most 8 splits (a portable cluster) and at
// least 4 k-blocks per split; normalised so that every split owns a k-block.
int gemm_splits(int n_tiles, int n_kb, int bn, bool split, int num_sms, int max_ctas, bool w8) {
  int cap = gemm_blocks_per_sm(bn, split, w8) * num_sms;
  if (max_ctas > 0) cap = std::min(cap, max_ctas);
  const int want = std::min(cap, (3 * num_sms + 1) / 2);
  int s = (want + n_tiles - 1) / n_tiles;
  while (s > 1 && n_tiles * s > cap) --s;
  s = std::max(1, std::min({s, 8, n_kb / 4}));
  return gemm_normalize_splits(n_kb, s, w8);
}

template <bool W8>
static int ring_stages_w(int bn, bool split) {
  switch (bn) {
    case 16: return split ? TcCfg<16, true, W8>::STAGES : TcCfg<16, false, W8>::STAGES;
    case 32: return split ? TcCfg<32, true, W8>::STAGES : TcCfg<32, false, W8>::STAGES;
    case 64: return split ? TcCfg<64, true, W8>::STAGES : TcCfg<64, false, W8>::STAGES;
    case 128: return split ? TcCfg<128, true, W8>::STAGES : TcCfg<128, false, W8>::STAGES;
    default:
      if constexpr (W8) return TcCfg<128, false, true>::STAGES;  // E4M3 tiles stop at 128 rows
      else return TcCfg<256, false, false>::STAGES;
  }
}

int gemm_ring_stages(int bn, bool split, bool w8) {
  return w8 ? ring_stages_w<true>(bn, split) : ring_stages_w<false>(bn, split);
}

bool gemm_l2_plan(dflash_ctx* c, const NextGemm& nx, L2Plan* pl, CUtensorMap* map) {
  *pl = L2Plan{};
  // (E4M3 weights: no plan; their stages are two k-blocks wide)
  if (nx.W == nullptr || c->cfg.dtype != DFLASH_BF16 || nx.splits < 1) return true;
  const bool w8 = c->cfg.dtype == DFLASH_BF16_W8;
  const int bn = gemm_bn(nx.M, nx.split);
  const int n_tiles = (nx.N + kTileN - 1) / kTileN, n_kb = gemm_kb(nx.K);
  const int kbps = (n_kb + nx.splits - 1) / nx.splits;
  const int first = std::min(kbps, gemm_ring_stages(bn, nx.split, w8));
  const long long per_kb = static_cast<long long>(n_tiles) * nx.splits * kTileN * kTileK * (w8 ? 1 : 2);
  const int count = static_cast<int>(std::min<long long>(kbps - first, nx.budget_bytes / per_kb));
  if (count <= 0) return true;
  if (!get_tmap(c, nx.W, nx.N, nx.K, kTileN, map, w8 ? 1 : 0)) return false;
  pl->ctas = n_tiles * nx.splits;
  pl->n_tiles = n_tiles;
  pl->kb_per_split = kbps;
  pl->n_kb = n_kb;
  pl->first = first;
  pl->count = count;
  return true;
}

int pers_plan(int M, int N, int K, int num_sms, int split_slots, bool split_tail) {
  // the persistent kernel serves the tensor-bound sizes (at least 256
  // activation rows) with 128 x 128 tiles, one CTA a tile or a cluster pair
  // splitting K (each half a tile's time, a small price for the exchange);
  // it applies where its waves are at least 75 % full on average (measured:
  // 64-row activation tiles, and fewer tiles, ran slower than the split-K
  // kernel)
  if (M < 256 || num_sms < 1) return 0;
  const long long tiles = static_cast<long long>((N + kTileN - 1) / kTileN) * ((M + 127) / 128);
  const double ideal = static_cast<double>(tiles) / num_sms;  // in full-K tile times
  double t1 = static_cast<double>((tiles + num_sms - 1) / num_sms);
  // the split tail: the last, partial round's tiles split in K among up to
  // kPersMaxSeg CTAs each (plus the partial tiles' write-out and sum)
  const long long rem = tiles % num_sms;
  const int n_kb = gemm_kb(K);
  if (split_tail && tiles > num_sms && rem > 0) {
    const int seg = static_cast<int>(std::min<long long>(std::min<long long>(kPersMaxSeg, num_sms / rem), n_kb));
    if (seg >= 2) t1 = static_cast<double>(tiles / num_sms) + static_cast<double>((n_kb + seg - 1) / seg) / n_kb + 0.05;
  }
  double best_eff = tiles >= num_sms ? ideal / t1 : 0.0;
  int best = 1;
  double ok_eff = best_eff;
  if (split_slots > 0 && gemm_kb(K) >= 2) {
    const double t2 = 0.5 * static_cast<double>((tiles + split_slots - 1) / split_slots) * 1.05;
    const double eff2 = ideal / t2;
    // a split pair streams through three ring stages, a single CTA through
    // four (measured: the fourth stage is worth about 10 %)
    if (0.9 * eff2 > best_eff) {
      best_eff = 0.9 * eff2;
      best = 2;
    }
    ok_eff = std::max(ok_eff, eff2);
  }
  return ok_eff >= 0.75 ? best : 0;
}

int gemm_bn(int M, bool split, bool w8) {
  const int cap = split || w8 ? 128 : 256;  // E4M3: the 256-row tile's stages would not hold its epilogue
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
  const bool split = g.X_lo != nullptr, w8 = c->cfg.dtype == DFLASH_BF16_W8;
  const bool lm = g.lm.mx != nullptr;
  int plan = 0;
  if (!w8 && split && (g.splits == 1 || g.epi.kind != EPI_NONE) && g.M >= 256 && c->num_sms > 0) {
    if (!lm && c->pers_split_clusters < 0) c->pers_split_clusters = pers_split_clusters(PersCfg<128, false, 2>::SMEM);
    plan = pers_plan(g.M, g.N, g.K, c->num_sms, lm ? 0 : std::max(0, c->pers_split_clusters), !lm && c->pers_ws != nullptr);
  }
  if (plan > 0) {
    // many activation rows: the persistent kernel (a tile's reduction stays
    // within its CTA or CTA pair, so the caller's split count does not apply)
    CUtensorMap tw, tx, txlo;
    if (!get_tmap(c, g.W, g.N, g.K, kTileN, &tw) || !get_tmap(c, g.X, g.M_alloc, g.K, 128, &tx) ||
        !get_tmap(c, g.X_lo, g.M_alloc, g.K, 128, &txlo))
      return cudaErrorInvalidValue;
    if (lm) return launch_pers<128, true, 1>(c, g, tw, tx, txlo, s);
    return plan == 2 ? launch_pers<128, false, 2>(c, g, tw, tx, txlo, s)
                     : launch_pers<128, false, 1>(c, g, tw, tx, txlo, s);
  }
  const int bn = gemm_bn(g.M, split, w8);
  CUtensorMap tw, tx, txlo;
  if (!get_tmap(c, g.W, g.N, g.K, kTileN, &tw, w8 ? 1 : 0) || !get_tmap(c, g.X, g.M_alloc, g.K, bn, &tx))
    return cudaErrorInvalidValue;
  if (split && !get_tmap(c, g.X_lo, g.M_alloc, g.K, bn, &txlo)) return cudaErrorInvalidValue;
  if (w8) return launch_tc_w8(c, g, bn, tw, tx, split ? txlo : tx, s);
  return split ? launch_tc_bn<true, false>(c, g, bn, tw, tx, txlo, s)
               : launch_tc_bn<false, false>(c, g, bn, tw, tx, tx, s);
}

// ---------------------------------------------------------------- launch without a map cache

// The same projection launch with both tensor maps encoded on the stack: no
// map cache and no host heap, for the entry point that must not allocate.
cudaError_t gemm_launch_uncached(int* status, const GemmLaunch& g, cudaStream_t s) {
  dflash_ctx tmp;  // holds only the status pointer; its containers stay empty
  tmp.cfg = dflash_config{};
  tmp.cfg.dtype = DFLASH_BF16;
  tmp.status = status;
  const bool split = g.X_lo != nullptr;
  const int bn = gemm_bn(g.M, split);
  CUtensorMap tw, tx, txlo;
  if (!encode_tmap(g.W, g.N, g.K, kTileN, 0, &tw) || !encode_tmap(g.X, g.M_alloc, g.K, bn, 0, &tx))
    return cudaErrorInvalidValue;
  if (split) {
    if (!encode_tmap(g.X_lo, g.M_alloc, g.K, bn, 0, &txlo)) return cudaErrorInvalidValue;
    return launch_tc_bn<true, false>(&tmp, g, bn, tw, tx, txlo, s);
  }
  return launch_tc_bn<false, false>(&tmp, g, bn, tw, tx, tx, s);
}

}  // namespace dflash

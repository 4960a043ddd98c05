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

// Row stride (floats) of the LM head's logits tile in shared memory: 128
// columns + 8 keeps the per-row segment reads free of bank conflicts.
constexpr int kLmLd = 136;

template <int BN, bool SPLIT>
struct TcCfg {
  static constexpr int W_BYTES = kTileN * kTileK * 2;  // 16 KB
  static constexpr int X_BYTES = BN * kTileK * 2;
  static constexpr int STAGE_BYTES = W_BYTES + (SPLIT ? 2 : 1) * X_BYTES;
  // BN = 16 (single-sequence drafting): a 4-stage ring, so that a CTA fits
  // beside another one or beside an attention CTA; BN 32-64: two CTAs per SM;
  // wider tiles: one CTA with a deeper ring
  static constexpr int BUDGET = BN <= 16 ? 90 * 1024 : BN <= 64 ? 110 * 1024 : 200 * 1024;
  static constexpr int STAGES = (BUDGET / STAGE_BYTES) < 8 ? (BUDGET / STAGE_BYTES) : 8;
  static constexpr int TMEM_COLS = BN < 32 ? 32 : BN;
  static constexpr int SMEM = 1024 /*align slack*/ + STAGES * STAGE_BYTES + 256 /*barriers*/ +
                              4 * BN * 4 /*epilogue scratch*/ + BN * 4 /*row scales*/ + BN * 16 /*row info*/;
  static_assert(STAGES >= 2, "pipeline too shallow");
  // split-K with bulk-copy reduction when the tile, the receive slots (at most BN + 8 rows) and the
  // reduced slice fit in the stage ring; otherwise the slices are read over distributed shared memory
  static constexpr bool PUSH_REDUCE = (2 * BN + 8 + BN / 2 + 8) * 128 * 4 <= STAGES * STAGE_BYTES;
  // the own tile plus the reduced slice (at most half the rows, splits >= 2) fit in the stage ring, and
  // so does the LM head's padded tile
  static_assert(BN * 128 * 4 * 3 / 2 <= STAGES * STAGE_BYTES, "epilogue tiles must fit in the stage ring");
  static_assert(BN * kLmLd * 4 <= STAGES * STAGE_BYTES, "LM-head tile must fit in the stage ring");
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
  L2Plan l2;  // the next projection's weights, prefetched into L2 after this CTA's last load
};

// Warp 0 lane 0 issues TMA, warp 1 lane 0 the MMAs (warp 1 owns the TMEM
// allocation), the other warps gather the epilogue's row facts while the
// main loop runs; all warps read the accumulator and run the epilogue (the
// code also runs with 256 threads: warps w and w + 4 then share a TMEM lane
// quadrant and split its columns; measured no faster at 16 rows).
constexpr int kGemmThreads = kEpiThreads;

template <int BN, bool LMHEAD, bool SPLIT>
__global__ void __launch_bounds__(kGemmThreads) k_gemm_tc(const __grid_constant__ CUtensorMap tmW,
                                                 const __grid_constant__ CUtensorMap tmX,
                                                 const __grid_constant__ CUtensorMap tmXlo,
                                                 const __grid_constant__ CUtensorMap tmNext,
                                                 const __grid_constant__ TcParams p) {
  using C = TcCfg<BN, SPLIT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW = smem;                                   // [STAGES][W tile]
  uint8_t* sX = smem + C::STAGES * C::W_BYTES;          // [STAGES][X tile (+ X lo tile)]
  constexpr int XS = (SPLIT ? 2 : 1) * C::X_BYTES;      // X bytes per stage
  uint64_t* full = reinterpret_cast<uint64_t*>(sX + C::STAGES * XS);
  uint64_t* empty = full + C::STAGES;
  uint64_t* accb = empty + C::STAGES;
  uint64_t* recvb = accb + 1;  // split-K: this CTA's rows from every split have landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(recvb + 1);
  int* s_prog = reinterpret_cast<int*>(tmem_slot + 1);  // [0] stages issued, [1] stages consumed
  float* red = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE_BYTES + 256);  // [BN][4] epilogue scratch
  float* s_rs = red + 4 * BN;                             // folded-RMSNorm row scales of rows m0 .. m0 + BN - 1
  int4* s_ri = reinterpret_cast<int4*>(s_rs + BN);        // per-row epilogue facts (epi_row_info; LM head: skip)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kTileN, m0 = blockIdx.y * BN, split = blockIdx.z;
  // m_valid is written two kernels upstream (page allocation), never by the
  // predecessor, so it may be read before pdl_wait
  if (p.m_valid != nullptr && m0 >= __ldg(p.m_valid)) {  // uniform: nothing allocated yet
    pdl_wait();
    return;
  }
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
    mbar_init(recvb, 1);
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
      // the weights do not depend on the predecessor: fill the ring with them
      // while it finishes, then add the activations once it has completed
      const int pre = min(nkb, C::STAGES);
      for (int it = 0; it < pre; ++it) {
        mbar_arrive_expect_tx(&full[it], C::STAGE_BYTES);
        tma_load_2d_hint(sW + it * C::W_BYTES, &tmW, &full[it], (kb0 + it) * kTileK, n0, pol);
      }
      pdl_wait();
      pdl_trigger();
      for (int it = 0; it < pre; ++it) {
        const int kx = (kb0 + it) * kTileK;
        tma_load_2d(sX + it * XS, &tmX, &full[it], kx, m0);
        if (SPLIT) tma_load_2d(sX + it * XS + C::X_BYTES, &tmXlo, &full[it], kx, m0);
      }
      s_prog[0] = pre;
      for (int it = pre; it < nkb; ++it) {
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
      // this CTA's weights are all requested: start the next projection's
      if (p.l2.ctas > 0) l2_prefetch_plan(&tmNext, p.l2);
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
  } else {
    // idle during the main loop: gather what the epilogue reads from global
    // memory (folded-RMSNorm row scales, row positions and pages)
    pdl_wait();
    const int mv = p.m_valid != nullptr ? min(p.M, *p.m_valid) : p.M;
    for (int j = threadIdx.x - 64; j < BN; j += kGemmThreads - 64) {
      const int m = m0 + j;
      const bool ok = m < mv;
      if (p.epi.ss_in != nullptr) s_rs[j] = ok ? norm_row_scale(p.epi, m) : 0.f;
      if (LMHEAD)
        s_ri[j] = make_int4(0, 0, 0, ok && (p.skip_rows == nullptr || p.skip_rows[m] == 0) ? 1 : 0);
      else
        s_ri[j] = ok ? epi_row_info(p.epi, m) : make_int4(0, 0, 0, 0);
    }
  }
  pdl_wait();  // everything below may read the predecessor's output

  // ---- epilogue: TMEM lane (32*warp + lane) holds weight row n, columns = activation rows
  mbar_wait(accb, 0, p.status);
  __syncwarp();  // lanes may leave the poll loop at different times; tcgen05.ld is warp-aligned
  tc_fence_after();
  __syncthreads();
  if (threadIdx.x == 0 && s_prog[1] < s_prog[0]) {
    // a wait gave up: let every copy still in flight land before the ring is reused
    for (int it = s_prog[1]; it < s_prog[0]; ++it) mbar_wait(&full[it % C::STAGES], (it / C::STAGES) & 1, p.status);
  }
  // TMEM lane quadrant of this warp (warps w and w + 4 share one and split
  // the accumulator's columns in chunks of 16)
  const int quad = warp & 3, wg = warp >> 2;
  const int n = n0 + quad * 32 + lane;
  const bool nv = n < p.N;
  const uint32_t tbase = tmem + (static_cast<uint32_t>(quad * 32) << 16);
  if constexpr (!LMHEAD) {
    // the accumulator goes to a [BN][128] fp32 tile in the (now idle) stage ring
    float* tile = reinterpret_cast<float*>(smem);
    __syncthreads();
#pragma unroll 1
    for (int c = 16 * wg; c < BN; c += 16 * (kGemmThreads / 128)) {
      float v[16];
      tc_ld_32x32b_x16(tbase + c, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) tile[(c + j) * 128 + quad * 32 + lane] = v[j];
    }
    tc_fence_before();
    __syncthreads();
    // the epilogue's global inputs of the rows this CTA finishes, loaded now
    // (after the TMEM reads, whose waits would otherwise also wait for
    // them) so that their latency overlaps the split-K reduction
    EpiPre pre;
    if (p.epi.kind != EPI_NONE) {
      int r0 = 0, nr = BN;
      if (p.splits > 1) {
        const int rpr = (BN + p.splits - 1) / p.splits;
        r0 = min(BN, static_cast<int>(cluster_ctarank()) * rpr);
        nr = min(BN, r0 + rpr) - r0;
      }
      epilogue_preload<__nv_bfloat16>(p.epi, m0 + r0, nr, n0, s_ri + r0, pre);
    }
    const int t = threadIdx.x;
    if (p.epi.kind == EPI_NONE) {
      float* o = p.out + split * p.split_stride;
      const int col = t & 127, nc = n0 + col;
      for (int j = t >> 7; j < BN && m0 + j < p.M; j += kGemmThreads >> 7)
        if (nc < p.N) o[static_cast<long long>(m0 + j) * p.ldo + nc] = tile[j * 128 + col];
    }
    if (p.epi.kind != EPI_NONE) {
      const float* rs = p.epi.ss_in != nullptr ? s_rs : nullptr;
      if (p.splits == 1) {
        apply_epilogue<__nv_bfloat16, __half>(p.epi, tile, m0, BN, n0, rs, s_ri, red, &pre);
      } else {
        // split-K reduction inside the cluster of this tile's `splits` CTAs:
        // each CTA sums a contiguous slice of the rows over every CTA's tile
        // (split order) and finishes those rows
        const int S = p.splits, cr = static_cast<int>(cluster_ctarank());
        const int rpr = (BN + S - 1) / S;
        const int r_begin = min(BN, cr * rpr), r_end = min(BN, r_begin + rpr);
        if constexpr (C::PUSH_REDUCE) {
          // every split copies the rows owned by cluster rank k into slot
          // [split] of k's receive area with a bulk shared-memory copy that
          // completes on k's mbarrier; the owner then adds the slots from
          // local memory.  The cluster barrier is split around the epilogue
          // so that no CTA leaves while a copy it sources may still read.
          float* recv = tile + BN * 128;          // [S][rpr][128]
          float* sub = recv + S * rpr * 128;      // [rpr][128]
          if (t == 0) mbar_arrive_expect_tx(recvb, static_cast<uint32_t>(S * (r_end - r_begin) * 128 * 4));
          fence_proxy_async_smem();
          __syncthreads();  // this CTA's tile is complete and visible to the copy engine
          // every CTA of the cluster is past its main loop: every receive area
          // is idle (relaxed: the preloaded epilogue inputs may still be in
          // flight; a receive count may follow the bytes it counts)
          cluster_arrive_relaxed();
          cluster_wait();
          if (t == 0)
            for (int k = 0; k < S; ++k) {
              const int k0 = min(BN, k * rpr), k1 = min(BN, k0 + rpr);
              if (k1 > k0)
                bulk_copy_smem_to_rank(smem_u32(recv + cr * rpr * 128), smem_u32(tile + k0 * 128),
                                       static_cast<uint32_t>((k1 - k0) * 128 * 4), recvb, static_cast<uint32_t>(k));
            }
          mbar_wait(recvb, 0, p.status);
          cluster_arrive_relaxed();  // my incoming copies have landed
          for (int e = t; e < (r_end - r_begin) * 32; e += kGemmThreads) {
            const int j = e / 32, c4 = (e % 32) * 4;
            float4 acc = *reinterpret_cast<const float4*>(recv + j * 128 + c4);
            for (int r = 1; r < S; ++r) {
              const float4 v = *reinterpret_cast<const float4*>(recv + (r * rpr + j) * 128 + c4);
              acc.x += v.x;
              acc.y += v.y;
              acc.z += v.z;
              acc.w += v.w;
            }
            *reinterpret_cast<float4*>(sub + j * 128 + c4) = acc;
          }
          __syncthreads();
          if (r_end > r_begin)
            apply_epilogue<__nv_bfloat16, __half>(p.epi, sub, m0 + r_begin, r_end - r_begin, n0,
                                                  rs != nullptr ? rs + r_begin : nullptr, s_ri + r_begin, red, &pre);
          cluster_wait();
        } else {
        cluster_sync_all();
        float* sub = tile + BN * 128;
        const uint32_t tile_s = smem_u32(tile);
        for (int e = t; e < (r_end - r_begin) * 32; e += kGemmThreads) {
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
        if (r_end > r_begin)
          apply_epilogue<__nv_bfloat16, __half>(p.epi, sub, m0 + r_begin, r_end - r_begin, n0,
                                                rs != nullptr ? rs + r_begin : nullptr, s_ri + r_begin, red, &pre);
        }
      }
    }
  } else {
    // LM head: the scaled logits go to a padded [BN][kLmLd] tile (and, when
    // asked for, to global memory); then 8 threads per row reduce it to the
    // tile's (max, lowest argmax, sum of exp(z - max)), 16 rows at a time.
    float* tile = reinterpret_cast<float*>(smem);
    __syncthreads();
#pragma unroll 1
    for (int c = 16 * wg; c < BN; c += 16 * (kGemmThreads / 128)) {
      float v[16];
      tc_ld_32x32b_x16(tbase + c, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int m = m0 + c + j;
        const float val = nv ? (p.epi.ss_in != nullptr ? v[j] * s_rs[c + j] : v[j]) : -INFINITY;
        tile[(c + j) * kLmLd + quad * 32 + lane] = val;
        if (p.logits != nullptr && nv && s_ri[c + j].w != 0) p.logits[m * p.ld_logits + n] = val;
      }
    }
    tc_fence_before();
    __syncthreads();
    const int seg = threadIdx.x & 7;
#pragma unroll 1
    for (int rb = 0; rb < BN; rb += kGemmThreads >> 3) {
      const int j = rb + (threadIdx.x >> 3);
      if (j >= BN) continue;  // uniform per warp (4 rows a warp, BN a multiple of 16)
      const float* row = tile + j * kLmLd;
      float z[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) z[k] = row[seg + 8 * k];
      // columns seg, seg + 8, ... are scanned in increasing order: strict >
      // keeps the lowest column among equal maxima
      float mx = z[0];
      int ix = seg;
#pragma unroll
      for (int k = 1; k < 16; ++k)
        if (z[k] > mx) {
          mx = z[k];
          ix = seg + 8 * k;
        }
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, mx, o);
        const int oi = __shfl_xor_sync(0xffffffffu, ix, o);
        if (om > mx || (om == mx && oi < ix)) {
          mx = om;
          ix = oi;
        }
      }
      float se = 0.f;
      if (mx > -INFINITY)
#pragma unroll
        for (int k = 0; k < 16; ++k) se += expf(z[k] - mx);
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) se += __shfl_xor_sync(0xffffffffu, se, o);
      const int m = m0 + j;
      if (seg == 0 && m < p.M) {
        const long long o = static_cast<long long>(m) * p.lm.n_tiles + blockIdx.x;
        p.lm.mx[o] = mx;
        p.lm.se[o] = se;
        p.lm.idx[o] = n0 + ix;
      }
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
  CUtensorMap tn = tw;  // the next projection's weights (a placeholder when there is no plan)
  if (!gemm_l2_plan(c, g.next, &p.l2, &tn)) p.l2 = L2Plan{};
  // splits come from gemm_splits: every split owns at least one k-block
  dim3 grid((g.N + kTileN - 1) / kTileN, (g.M + BN - 1) / BN, g.splits);
  // the splits of one output tile form a thread-block cluster (reduced over DSMEM)
  const bool clustered = !(LM || g.epi.kind == EPI_NONE || g.splits == 1);
  return launch_k(k_gemm_tc<BN, LM, SPLIT>, grid, dim3(kGemmThreads), C::SMEM, s, dim3(1, 1, clustered ? g.splits : 1),
                  c->pdl, tw, tx, txlo, tn, p);
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

// How many CTAs of the projection kernel (tile width bn, hi+lo operands or
// not) one SM holds at once.
// Shared memory is the only limit that binds (128 threads, few registers,
// at most 512 TMEM columns per SM across resident CTAs).
template <int BN, bool SPLIT>
static int blocks_per_sm_t() {
  using C = TcCfg<BN, SPLIT>;
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

int gemm_blocks_per_sm(int bn, bool split) {
  static int cache[2][5] = {};  // [split][log2(bn/16)]
  int bi = 0;
  while ((16 << bi) < bn && bi < 4) ++bi;
  int& c = cache[split ? 1 : 0][bi];
  if (c == 0) {
    switch (bi) {
      case 0: c = split ? blocks_per_sm_t<16, true>() : blocks_per_sm_t<16, false>(); break;
      case 1: c = split ? blocks_per_sm_t<32, true>() : blocks_per_sm_t<32, false>(); break;
      case 2: c = split ? blocks_per_sm_t<64, true>() : blocks_per_sm_t<64, false>(); break;
      case 3: c = split ? blocks_per_sm_t<128, true>() : blocks_per_sm_t<128, false>(); break;
      default: c = split ? 1 : blocks_per_sm_t<256, false>(); break;
    }
  }
  return c;
}

// Split-K count for `n_tiles` output tiles of width bn.  A CTA streams its
// weights at a fraction of the HBM bandwidth an SM can draw, so the grid
// must keep every SM streaming: aim for about 1.25 CTAs per SM (all
// resident at once, at most max_ctas when positive), with at most 8 splits
// (a portable cluster) and at least 4 k-blocks per split; normalised so that
// every split owns a k-block.
int gemm_splits(int n_tiles, int n_kb, int bn, bool split, int num_sms, int max_ctas) {
  int cap = gemm_blocks_per_sm(bn, split) * num_sms;
  if (max_ctas > 0) cap = std::min(cap, max_ctas);
  const int want = std::min(cap, (5 * num_sms + 3) / 4);
  int s = (want + n_tiles - 1) / n_tiles;
  while (s > 1 && n_tiles * s > cap) --s;
  s = std::max(1, std::min({s, 8, n_kb / 4}));
  const int per = (n_kb + s - 1) / s;
  return (n_kb + per - 1) / per;
}

int gemm_ring_stages(int bn, bool split) {
  switch (bn) {
    case 16: return split ? TcCfg<16, true>::STAGES : TcCfg<16, false>::STAGES;
    case 32: return split ? TcCfg<32, true>::STAGES : TcCfg<32, false>::STAGES;
    case 64: return split ? TcCfg<64, true>::STAGES : TcCfg<64, false>::STAGES;
    case 128: return split ? TcCfg<128, true>::STAGES : TcCfg<128, false>::STAGES;
    default: return TcCfg<256, false>::STAGES;
  }
}

bool gemm_l2_plan(dflash_ctx* c, const NextGemm& nx, L2Plan* pl, CUtensorMap* map) {
  *pl = L2Plan{};
  if (nx.W == nullptr || c->cfg.dtype != DFLASH_BF16 || nx.splits < 1) return true;
  const int bn = gemm_bn(nx.M, nx.split);
  const int n_tiles = (nx.N + kTileN - 1) / kTileN, n_kb = gemm_kb(nx.K);
  const int kbps = (n_kb + nx.splits - 1) / nx.splits;
  const int first = std::min(kbps, gemm_ring_stages(bn, nx.split));
  const long long per_kb = static_cast<long long>(n_tiles) * nx.splits * kTileN * kTileK * 2;
  const int count = static_cast<int>(std::min<long long>(kbps - first, nx.budget_bytes / per_kb));
  if (count <= 0) return true;
  if (!get_tmap(c, nx.W, nx.N, nx.K, kTileN, map)) return false;
  pl->ctas = n_tiles * nx.splits;
  pl->n_tiles = n_tiles;
  pl->kb_per_split = kbps;
  pl->n_kb = n_kb;
  pl->first = first;
  pl->count = count;
  return true;
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

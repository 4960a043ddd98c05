// The tcgen05 projection kernel, shared by gemm.cu (bf16 weights) and
// gemm_w8.cu (E4M3 weights with per-row scales); each translation unit
// instantiates its own variants.
//
// The weight matrix streams through the MMA's M side (128 rows per tile)
// and the few activation rows ride on N (16..256), so an M = 16 draft block
// still fills the 128-row MMA (swap-AB).  One thread issues TMA tile loads
// into a STAGES-deep shared-memory ring, one thread issues tcgen05.mma into
// a TMEM accumulator, and four warps read the accumulator back with
// tcgen05.ld in the epilogue.  Weights are loaded with an L2 evict-first
// hint: each byte is used once per launch.
//
// Activations may come as an exact pair of bf16 terms (x = hi + lo, the
// residual of rounding x to bf16 rounded again): the two tiles form one
// K-major operand of 2 BN rows, so one MMA per k-slice yields W.hi and W.lo
// side by side in the accumulator and the epilogue adds them; the product
// keeps about 16 significant bits of x while both MMA operands stay bf16.
//
// E4M3 weights (W8): TMA brings the 8-bit codes (half the bytes of bf16)
// into a ring of their own; eight converter warps (two per TMEM lane
// quadrant) turn each weight row into exact bf16 values in registers and
// store them into TMEM (tcgen05.st); the MMA takes its A operand from TMEM
// and the activations from a second ring.  The per-row scale multiplies the
// accumulator row in the epilogue.  The projections are HBM-bound at decode
// sizes, so halving the weight bytes is the point; the conversion runs
// beside the stream.
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "internal.h"

namespace dflash {

// Row stride (floats) of the LM head's logits tile in shared memory: 128
// columns + 8 keeps the per-row segment reads free of bank conflicts.
constexpr int kLmLd = 136;

// Threads of the bf16 kernel: warp 0 lane 0 issues TMA, warp 1 lane 0 the
// MMAs (warp 1 owns the TMEM allocation), warps 2-3 gather the epilogue's
// row facts while the main loop runs; all four read the accumulator and run
// the epilogue.  The W8 kernel has ten warps: warps 0-7 convert the weights
// (two per TMEM lane quadrant, each half of every k-block), warps 0-3 then
// run the epilogue, warp 8 issues TMA and warp 9 the MMAs.
constexpr int kGemmThreads = kEpiThreads;

constexpr int tmem_cols_pow2(int n) {
  int c = 32;
  while (c < n) c *= 2;
  return c;
}

template <int BN, bool SPLIT, bool W8>
struct TcCfg {
  // k-blocks (kTileK wide) per pipeline stage: a stage moves 128-byte weight
  // rows, 64 bf16 or 128 E4M3 codes (TMA moves 128-byte rows at twice the
  // rate of 64-byte ones)
  static constexpr int KB_PER_STAGE = W8 ? 2 : 1;
  static constexpr int KS = KB_PER_STAGE * kTileK;                 // k per stage
  static constexpr int W_BYTES = kTileN * KS * (W8 ? 1 : 2);       // 16 KB
  static constexpr int X_BOX = BN * kTileK * 2;                    // one activation box (64 k)
  static constexpr int XPAIR = (SPLIT ? 2 : 1) * X_BOX;            // the hi (and lo) box of one 64-k block
  static constexpr int XS = KB_PER_STAGE * XPAIR;                  // activation bytes per stage
  static constexpr int STAGE_BYTES = W_BYTES + XS;
  // Shared memory for the rings.  BN <= 64: about 100-110 KB, two CTAs per
  // SM (BN = 16, single-sequence drafting: five bf16 stages; measured faster
  // than four on the c2 round); wider tiles: one CTA with deeper rings
  static constexpr int BUDGET = BN <= 16 ? (W8 ? 104 : 108) * 1024 : BN <= 64 ? 110 * 1024 : 200 * 1024;
  // One MMA covers both activation terms: their tiles lie back to back in
  // shared memory (hi rows, then lo rows), so they form one K-major operand
  // of 2 BN rows and the accumulator holds W.hi in columns 0 .. BN - 1 and
  // W.lo in BN .. 2 BN - 1, added in the epilogue.  At decode sizes the
  // chain of MMAs into one accumulator, not the tensor core's throughput,
  // bounds the main loop, so half as many MMAs is half the chain.
  static constexpr int NMMA = (SPLIT ? 2 : 1) * BN;
  static constexpr int ACC_COLS = NMMA < 32 ? 32 : NMMA;
  // bf16: one ring of STAGES (weights + activations), freed by the MMAs.
  // W8: a weight ring of WST stages, freed as soon as the converters hold a
  // stage's codes in registers, and NA stages of converted weights in TMEM,
  // each with its activations in shared memory, freed by the MMAs (128 lanes
  // x 128 bf16 = 64 TMEM columns a stage); the converters run ahead of the
  // MMAs by up to NA stages, the weight stream ahead of the converters by up
  // to WST
  static constexpr int A_COLS = KS / 2;
  static constexpr int TMEM_SHARE = BN <= 64 ? 256 : 512;  // this CTA's share: two CTAs an SM up to 64 rows
  static constexpr int NA_TMEM = (TMEM_SHARE - ACC_COLS) / A_COLS;
  static constexpr int NA_X = (BUDGET / 3) / XS > 2 ? (BUDGET / 3) / XS : 2;
  static constexpr int NA = !W8 ? 0 : NA_TMEM < NA_X ? (NA_TMEM < 8 ? NA_TMEM : 8) : (NA_X < 8 ? NA_X : 8);
  static constexpr int STAGES_RAW = W8 ? (BUDGET - NA * XS) / W_BYTES : BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW < 8 ? STAGES_RAW : 8;   // bf16: ring stages; W8: weight ring
  static constexpr int XST = W8 ? NA : STAGES;                     // stages of activations
  static constexpr int RING_BYTES = STAGES * W_BYTES + XST * XS;
  static constexpr int TMEM_COLS = W8 ? tmem_cols_pow2(ACC_COLS + NA * A_COLS) : ACC_COLS;
  static constexpr int CONV_WARPS = W8 ? 8 : 0;
  static constexpr int THREADS = W8 ? 32 * (CONV_WARPS + 2) : kGemmThreads;
  static constexpr int MIN_BLOCKS = W8 ? 2 : 1;  // W8: two CTAs an SM must fit in the register file
  static constexpr int BAR_BYTES = W8 ? 512 : 256;  // mbarriers, the TMEM address, progress counters
  static constexpr int SMEM = 1024 /*align slack*/ + RING_BYTES + BAR_BYTES +
                              4 * BN * 4 /*epilogue scratch*/ + BN * 4 /*row scales*/ + BN * 16 /*row info*/;
  static_assert(STAGES >= 2 && (!W8 || NA >= 2), "pipeline too shallow");
  static_assert(TMEM_COLS <= 512, "TMEM holds 512 columns");
  // split-K with bulk-copy reduction when the tile, the receive slots (at most BN + 8 rows) and the
  // reduced slice fit in the rings; otherwise the slices are read over distributed shared memory
  static constexpr bool PUSH_REDUCE = (2 * BN + 8 + BN / 2 + 8) * 128 * 4 <= RING_BYTES;
  // the own tile plus the reduced slice (at most half the rows, splits >= 2) fit in the rings, and
  // so does the LM head's padded tile
  static_assert(BN * 128 * 4 * 3 / 2 <= RING_BYTES, "epilogue tiles must fit in the rings");
  static_assert(BN * kLmLd * 4 <= RING_BYTES, "LM-head tile must fit in the rings");
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
  const int* logits_rows;  // nullable: row m's logits are stored at row logits_rows[m]
  int logits_bulk;         // logits rows 16-byte aligned: whole tiles leave by bulk copies
  const float* w_scale;  // W8: fp32 scale of every weight row [N]
  L2Plan l2;  // the next projection's weights, prefetched into L2 after this CTA's last load
};

// The converter side of the W8 kernel: lane l of warp w (w < 8) owns weight
// row r = 32 (w % 4) + l of the tile, i.e. TMEM lane r, and half h = w / 4
// of every stage (64 of its 128 codes).  Per stage it loads those codes from
// the 128-byte-swizzled weight tile (16-byte chunk c of row r sits at chunk
// c ^ (r & 7)) and frees the weight slot, converts them to 32 bf16x2 words,
// waits until the MMAs are done with TMEM stage `a` and stores the words in
// its columns 32 h .. 32 h + 31.  Returns false if a wait gave up.
template <int STAGES, int NA, int W_BYTES>
__device__ __forceinline__ bool convert_weights(const uint8_t* sW, uint64_t* full, uint64_t* empty, uint64_t* conv,
                                                uint64_t* aempty, uint32_t a_row, int n_st, int* status) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = (w & 3) * 32 + lane, h = w >> 2;
  const uint32_t swz = static_cast<uint32_t>(r & 7);
  for (int it = 0; it < n_st; ++it) {
    const int s = it % STAGES, a = it % NA;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (it / STAGES) & 1, status))) return false;
    const uint8_t* row = sW + s * W_BYTES + r * 128;
    uint4 q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      q[i] = *reinterpret_cast<const uint4*>(row + ((static_cast<uint32_t>(4 * h + i) ^ swz) << 4));
    __syncwarp();
    if (lane == 0) mbarrier_arrive_one(&empty[s]);  // the codes are in registers: the slot may refill
    uint32_t v[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      e4m3x4_to_bf16x4(q[i].x, v[8 * i + 0], v[8 * i + 1]);
      e4m3x4_to_bf16x4(q[i].y, v[8 * i + 2], v[8 * i + 3]);
      e4m3x4_to_bf16x4(q[i].z, v[8 * i + 4], v[8 * i + 5]);
      e4m3x4_to_bf16x4(q[i].w, v[8 * i + 6], v[8 * i + 7]);
    }
    if (!__all_sync(0xffffffffu, mbar_wait(&aempty[a], ((it / NA) & 1) ^ 1, status))) return false;
    tc_fence_after();
    tc_st_32x32b_x32(a_row + a * 64 + h * 32, v);
    tc_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbarrier_arrive_one(&conv[a]);  // TMEM stage a holds this warp's half of its 32 rows
  }
  return true;
}

template <int BN, bool LMHEAD, bool SPLIT, bool W8>
__global__ void __launch_bounds__(TcCfg<BN, SPLIT, W8>::THREADS, TcCfg<BN, SPLIT, W8>::MIN_BLOCKS)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
              const __grid_constant__ CUtensorMap tmXlo, const __grid_constant__ CUtensorMap tmNext,
              const __grid_constant__ TcParams p) {
  using C = TcCfg<BN, SPLIT, W8>;
  constexpr int PRODUCER = W8 ? C::CONV_WARPS : 0, MMA_WARP = W8 ? C::CONV_WARPS + 1 : 1, ALLOC_WARP = W8 ? 0 : 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW = smem;                                   // [STAGES][weight tile]
  uint8_t* sX = smem + C::STAGES * C::W_BYTES;          // [XST][activation tile (+ lo tile)]
  constexpr int XS = C::XS;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::RING_BYTES);  // [STAGES] stage (W8: weights) landed
  uint64_t* empty = full + C::STAGES;  // [STAGES] slot free (bf16: MMAs done; W8: codes taken by the converters)
  uint64_t* accb = empty + C::STAGES;
  uint64_t* recvb = accb + 1;          // split-K: this CTA's rows from every split have landed
  uint64_t* xfull = recvb + 1;         // W8 [NA]: a stage's activations landed
  uint64_t* conv = xfull + C::NA;      // W8 [NA]: TMEM stage converted (one arrival per converter warp)
  uint64_t* aempty = conv + C::NA;     // W8 [NA]: the MMAs are done with a TMEM stage and its activations
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aempty + C::NA);
  int* s_prog = reinterpret_cast<int*>(tmem_slot + 1);  // bf16: [0] stages issued, [1] stages consumed
  static_assert((2 * C::STAGES + 2 + 3 * C::NA) * 8 + 12 <= C::BAR_BYTES, "barrier area too small");
  float* red = reinterpret_cast<float*>(smem + C::RING_BYTES + C::BAR_BYTES);  // [BN][4] epilogue scratch
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
  const int n_st = (nkb + C::KB_PER_STAGE - 1) / C::KB_PER_STAGE;  // pipeline stages of this split
  // W8: the scale of the weight row this thread finishes in the epilogue (a
  // weight, not written by the predecessor)
  float wsc = 1.f;
  if constexpr (W8) {
    if (threadIdx.x < kEpiThreads) wsc = n0 + static_cast<int>(threadIdx.x) < p.N ? __ldg(p.w_scale + n0 + threadIdx.x) : 0.f;
  }

  if (warp == PRODUCER && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    if (SPLIT) tma_prefetch_desc(&tmXlo);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], W8 ? C::CONV_WARPS : 1);  // W8: every converter warp has its codes
    }
    for (int a = 0; a < C::NA; ++a) {
      mbar_init(&xfull[a], 1);
      mbar_init(&conv[a], C::CONV_WARPS);
      mbar_init(&aempty[a], 1);
    }
    mbar_init(accb, 1);
    mbar_init(recvb, 1);
    s_prog[0] = 0;
    s_prog[1] = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == ALLOC_WARP) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == PRODUCER) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      // stage it covers k-blocks kb0 + KB_PER_STAGE * it ...; a stage past
      // the end of K reads zeros (TMA fills out-of-range boxes)
      // activations of a stage: per 64-k block its hi box, then its lo box
      auto load_x = [&](uint8_t* dst, uint64_t* bar, int it) {
        const int kx = (kb0 + C::KB_PER_STAGE * it) * kTileK;
#pragma unroll
        for (int j = 0; j < C::KB_PER_STAGE; ++j) {
          tma_load_2d(dst + j * C::XPAIR, &tmX, bar, kx + j * kTileK, m0);
          if (SPLIT) tma_load_2d(dst + j * C::XPAIR + C::X_BOX, &tmXlo, bar, kx + j * kTileK, m0);
        }
      };
      auto load_w = [&](int s, int it, uint32_t bytes) {
        mbar_arrive_expect_tx(&full[s], bytes);
        tma_load_2d_hint(sW + s * C::W_BYTES, &tmW, &full[s], (kb0 + C::KB_PER_STAGE * it) * kTileK, n0, pol);
      };
      // the weights do not depend on the predecessor: fill the ring with them
      // while it finishes, then add the activations once it has completed
      const int pre = min(n_st, C::STAGES);
      for (int it = 0; it < pre; ++it) load_w(it, it, W8 ? C::W_BYTES : C::STAGE_BYTES);
      pdl_wait();
      pdl_trigger();
      if constexpr (W8) {
        // two rings, refilled as their slots free up: weight stages as the
        // converters take the codes, activation stages as the MMAs finish
        int iw = pre, ix = 0;
        unsigned long long t0 = globaltimer_ns();
        for (uint32_t spin = 1; iw < n_st || ix < n_st; ++spin) {
          if (ix < n_st && (ix < C::NA || mbar_try_wait(&aempty[ix % C::NA], ((ix / C::NA) & 1) ^ 1))) {
            mbar_arrive_expect_tx(&xfull[ix % C::NA], XS);
            load_x(sX + (ix % C::NA) * XS, &xfull[ix % C::NA], ix);
            ++ix;
            t0 = globaltimer_ns();
          } else if (iw < n_st && mbar_try_wait(&empty[iw % C::STAGES], ((iw / C::STAGES) & 1) ^ 1)) {
            load_w(iw % C::STAGES, iw, C::W_BYTES);
            ++iw;
            t0 = globaltimer_ns();
          } else if ((spin & 255u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(p.status, ST_WAIT_TIMEOUT);
            break;
          }
        }
        // leave only once every copy this thread issued has landed: the last
        // STAGES weight and NA activation stages may still be in flight
        for (int it = max(0, iw - C::STAGES); it < iw; ++it)
          mbar_wait(&full[it % C::STAGES], (it / C::STAGES) & 1, p.status);
        for (int it = max(0, ix - C::NA); it < ix; ++it) mbar_wait(&xfull[it % C::NA], (it / C::NA) & 1, p.status);
      } else {
        for (int it = 0; it < pre; ++it) load_x(sX + it * XS, &full[it], it);
        s_prog[0] = pre;
        for (int it = pre; it < n_st; ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, p.status)) break;
          load_w(s, it, C::STAGE_BYTES);
          load_x(sX + s * XS, &full[s], it);
          s_prog[0] = it + 1;
        }
        // this CTA's weights are all requested: start the next projection's
        if (p.l2.ctas > 0) l2_prefetch_plan(&tmNext, p.l2);
      }
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      constexpr uint32_t idesc = mma_idesc_bf16_f32(kTileN, C::NMMA);
      for (int it = 0; it < n_st; ++it) {
        if constexpr (W8) {
          const int a = it % C::NA;
          const uint32_t pa = (it / C::NA) & 1;
          if (!mbar_wait(&xfull[a], pa, p.status) || !mbar_wait(&conv[a], pa, p.status)) break;
          tc_fence_after();
          const uint32_t aX = smem_u32(sX + a * XS);
#pragma unroll
          for (int k = 0; k < C::KS / 16; ++k) {
            const uint32_t aA = tmem + C::ACC_COLS + a * C::A_COLS + k * 8;  // 16 k of bf16 = 8 columns
            const uint32_t bX = aX + (k >> 2) * C::XPAIR + 32 * (k & 3);      // 64-k box pair, 16-k slice
            tc_mma_bf16_ts(tmem, aA, sw128_kmajor_desc(bX), idesc, (it | k) != 0 ? 1u : 0u);
          }
          tc_commit(&aempty[a]);
        } else {
          const int s = it % C::STAGES;
          if (!mbar_wait(&full[s], (it / C::STAGES) & 1, p.status)) break;
          tc_fence_after();
          const uint32_t aW = smem_u32(sW + s * C::W_BYTES);
          const uint32_t aX = smem_u32(sX + s * XS);
#pragma unroll
          for (int k = 0; k < kTileK / 16; ++k) {
            tc_mma_bf16(tmem, sw128_kmajor_desc(aW + 32 * k), sw128_kmajor_desc(aX + 32 * k), idesc,
                        (it | k) != 0 ? 1u : 0u);
          }
          tc_commit(&empty[s]);
          s_prog[1] = it + 1;
        }
      }
      tc_commit(accb);
    }
    __syncwarp();
  } else {
    int j0 = threadIdx.x - 64, jstep = kGemmThreads - 64;  // bf16: warps 2-3 while the main loop runs
    if constexpr (W8) {
      // TMEM lane quadrant of this warp: warps w and w + 4 share quadrant w % 4
      convert_weights<C::STAGES, C::NA, C::W_BYTES>(
          sW, full, empty, conv, aempty, tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + C::ACC_COLS, n_st,
          p.status);
      j0 = warp < 4 ? static_cast<int>(threadIdx.x) : BN;  // W8: warps 0-3, after their last k-block
      jstep = kEpiThreads;
    }
    // gather what the epilogue reads from global memory (folded-RMSNorm row
    // scales, row positions and pages)
    pdl_wait();
    const int mv = p.m_valid != nullptr ? min(p.M, *p.m_valid) : p.M;
    for (int j = j0; j < BN; j += jstep) {
      const int m = m0 + j;
      const bool ok = m < mv;
      if (p.epi.ss_in != nullptr) s_rs[j] = ok ? norm_row_scale(p.epi, m) : 0.f;
      if (LMHEAD) {
        // x: the logits row this row is stored at; w: whether it is stored
        const int orow = ok ? (p.logits_rows != nullptr ? p.logits_rows[m] : m) : -1;
        s_ri[j] = make_int4(orow, 0, 0, orow >= 0 && (p.skip_rows == nullptr || p.skip_rows[m] == 0) ? 1 : 0);
      }
      else
        s_ri[j] = ok ? epi_row_info(p.epi, m) : make_int4(0, 0, 0, 0);
    }
  }
  if constexpr (W8) {
    if (warp >= 4) return;  // the other converters, TMA and MMA warps are done; the epilogue runs on warps 0-3
  }
  pdl_wait();  // everything below may read the predecessor's output

  // ---- epilogue: TMEM lane (32*warp + lane) holds weight row n, columns = activation rows
  mbar_wait(accb, 0, p.status);
  __syncwarp();  // lanes may leave the poll loop at different times; tcgen05.ld is warp-aligned
  tc_fence_after();
  epi_sync();
  if (!W8 && threadIdx.x == 0 && s_prog[1] < s_prog[0]) {
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
    epi_sync();
#pragma unroll 1
    for (int c = 16 * wg; c < BN; c += 16 * (kGemmThreads / 128)) {
      float v[16];
      tc_ld_32x32b_x16(tbase + c, v);
      if constexpr (SPLIT) {
        float v2[16];
        tc_ld_32x32b_x16(tbase + BN + c, v2);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] += v2[j];
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) tile[(c + j) * 128 + quad * 32 + lane] = W8 ? v[j] * wsc : v[j];
    }
    tc_fence_before();
    epi_sync();
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
          epi_sync();  // this CTA's tile is complete and visible to the copy engine
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
          epi_sync();
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
    // LM head: the scaled logits go to a padded [BN][kLmLd] tile; then 8
    // threads per row reduce it to the tile's (max, lowest argmax, sum of
    // exp(z - max)), 16 rows at a time.  When the logits are asked for, a
    // whole 128-column tile leaves by bulk copies, one 512-byte row each
    // (issued by warp 0 once the tile is complete, evict-first in L2, read
    // from shared memory while the reduction runs); a ragged tile, or rows
    // that are not 16-byte aligned, by streaming stores.
    float* tile = reinterpret_cast<float*>(smem);
    const bool bulk_out = p.logits != nullptr && p.logits_bulk && n0 + kTileN <= p.N;
    epi_sync();
#pragma unroll 1
    for (int c = 16 * wg; c < BN; c += 16 * (kGemmThreads / 128)) {
      float v[16];
      tc_ld_32x32b_x16(tbase + c, v);
      if constexpr (SPLIT) {
        float v2[16];
        tc_ld_32x32b_x16(tbase + BN + c, v2);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) v[jj] += v2[jj];
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float z = W8 ? v[j] * wsc : v[j];
        const float val = nv ? (p.epi.ss_in != nullptr ? z * s_rs[c + j] : z) : -INFINITY;
        tile[(c + j) * kLmLd + quad * 32 + lane] = val;
        if (!bulk_out && p.logits != nullptr && nv && s_ri[c + j].w != 0)
          __stcs(p.logits + s_ri[c + j].x * p.ld_logits + n, val);
      }
    }
    tc_fence_before();
    if (bulk_out) fence_proxy_async_smem();  // the tile, as the copy engine will read it
    epi_sync();
    if (bulk_out && warp == 0) {
      const uint64_t pol = l2_policy_evict_first();
      for (int j = lane; j < BN; j += 32)
        if (s_ri[j].w != 0)
          bulk_store_global(p.logits + s_ri[j].x * p.ld_logits + n0, smem_u32(tile + j * kLmLd), kTileN * 4, pol);
      bulk_commit();
    }
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
    if (bulk_out && warp == 0) bulk_wait_read_all();  // the tile stays put until the copies have read it
  }
  epi_sync();
  if (warp == ALLOC_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}


// --------------------------------------------------------------- launch

template <int BN, bool LM, bool SPLIT, bool W8>
cudaError_t launch_tc(dflash_ctx* c, const GemmLaunch& g, const CUtensorMap& tw, const CUtensorMap& tx,
                             const CUtensorMap& txlo, cudaStream_t s) {
  using C = TcCfg<BN, SPLIT, W8>;
  static FuncAttr smem_attr;
  cudaError_t ae = smem_attr.ensure(C::SMEM, [](int v) {
    return cudaFuncSetAttribute(k_gemm_tc<BN, LM, SPLIT, W8>, cudaFuncAttributeMaxDynamicSharedMemorySize, v);
  });
  if (ae != cudaSuccess) return ae;
  TcParams p;
  const int n_kb = gemm_kb(g.K);
  p.M = g.M;
  p.N = g.N;
  p.n_kb = n_kb;
  p.kb_per_split = gemm_kb_per_split(n_kb, g.splits, W8);
  if ((g.splits - 1) * p.kb_per_split >= n_kb) return cudaErrorInvalidValue;  // a split without k-blocks
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
  p.logits_rows = g.logits_rows;
  p.logits_bulk = g.logits != nullptr && (reinterpret_cast<uintptr_t>(g.logits) & 15) == 0 && g.ld_logits % 4 == 0;
  p.w_scale = g.w_scale;
  CUtensorMap tn = tw;  // the next projection's weights (a placeholder when there is no plan)
  if (!gemm_l2_plan(c, g.next, &p.l2, &tn)) p.l2 = L2Plan{};
  // splits come from gemm_splits: every split owns at least one k-block
  dim3 grid((g.N + kTileN - 1) / kTileN, (g.M + BN - 1) / BN, g.splits);
  // the splits of one output tile form a thread-block cluster (reduced over DSMEM)
  const bool clustered = !(LM || g.epi.kind == EPI_NONE || g.splits == 1);
  return launch_k(k_gemm_tc<BN, LM, SPLIT, W8>, grid, dim3(C::THREADS), C::SMEM, s, dim3(1, 1, clustered ? g.splits : 1),
                  c->pdl, tw, tx, txlo, tn, p);
}

template <bool SPLIT, bool W8>
cudaError_t launch_tc_bn(dflash_ctx* c, const GemmLaunch& g, int bn, const CUtensorMap& tw,
                                const CUtensorMap& tx, const CUtensorMap& txlo, cudaStream_t s) {
  const bool lm = g.lm.mx != nullptr;
  switch (bn) {
    case 16:
      return lm ? launch_tc<16, true, SPLIT, W8>(c, g, tw, tx, txlo, s) : launch_tc<16, false, SPLIT, W8>(c, g, tw, tx, txlo, s);
    case 32:
      return lm ? launch_tc<32, true, SPLIT, W8>(c, g, tw, tx, txlo, s) : launch_tc<32, false, SPLIT, W8>(c, g, tw, tx, txlo, s);
    case 64:
      return lm ? launch_tc<64, true, SPLIT, W8>(c, g, tw, tx, txlo, s) : launch_tc<64, false, SPLIT, W8>(c, g, tw, tx, txlo, s);
    case 128:
      return lm ? launch_tc<128, true, SPLIT, W8>(c, g, tw, tx, txlo, s)
                : launch_tc<128, false, SPLIT, W8>(c, g, tw, tx, txlo, s);
    default:
      if constexpr (SPLIT || W8) return cudaErrorInvalidValue;  // 256-row tiles: one bf16 term, bf16 weights
      else
        return lm ? launch_tc<256, true, false, W8>(c, g, tw, tx, txlo, s)
                  : launch_tc<256, false, false, W8>(c, g, tw, tx, txlo, s);
  }
}


}  // namespace dflash

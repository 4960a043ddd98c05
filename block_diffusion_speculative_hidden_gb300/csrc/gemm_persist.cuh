// The persistent tcgen05 projection kernel for many activation rows (the
// serving batches: 512 and more block rows), bf16 weights with the hi + lo
// activation pair.
//
// At these sizes the projections are tensor-bound, and a kernel that gives
// each CTA one output tile leaves the tensor pipe idle while the CTA starts
// (barriers, TMEM, the first loads) and while it finishes (accumulator
// readout, fused epilogue).  Here one CTA per SM walks a list of output
// tiles (128 weight rows x BN activation rows, activation tile fastest so
// that CTAs running at the same time share weight tiles in L2):
//
//   - warp 4, one thread: TMA loads of the weight tile and both activation
//     terms, 64 k a stage, into an STAGES-deep ring that runs across tile
//     boundaries;
//   - warp 5, one thread: one MMA of N = 2 BN per 16-k slice (the hi and lo
//     activation tiles lie back to back, so one MMA yields W.hi and W.lo
//     side by side) into one of two TMEM accumulators, alternating by tile;
//     warp 5 owns the TMEM allocation;
//   - warps 0-3 (TMEM lane quadrants 0-3): read an accumulator out, 32
//     activation rows at a time, into a shared-memory tile of their own and
//     run the fused epilogue on each chunk; the accumulator is released
//     after its last chunk is read (so the MMAs of the tile after next may
//     start), all while the MMAs of the next tile proceed;
//   - the tiles of the last, partial round may be split in K among several
//     CTAs (the split tail, below).
//
// Every wait is bounded; after a wait gives up the CTA marks the status
// word, the roles stop waiting on one another (a shared abort flag) and the
// epilogue warps still meet at every named barrier.
#pragma once

#include "gemm_kernel.cuh"

namespace dflash {

// A CTA that owns its tile's whole reduction (KSPLIT 1) reads the
// accumulator out 32 activation rows at a time, so its staging tile is a
// quarter of the tile and the ring has room for a fourth stage (the loads
// are latency-bound with three); a split pair exchanges whole tiles.
template <int BN, bool LMHEAD, int KSPLIT = 1>
struct PersCfg {
  static constexpr int W_BYTES = kTileN * kTileK * 2;          // 16 KB
  static constexpr int X_BOX = BN * kTileK * 2;                 // one activation term, 64 k
  static constexpr int STAGE_BYTES = W_BYTES + 2 * X_BOX;       // weights, hi, lo
  static constexpr int NMMA = 2 * BN;                           // MMA N: hi and lo rows
  static constexpr int ACC_COLS = NMMA;
  static constexpr int TMEM_COLS = 2 * ACC_COLS;                // two accumulators
  static constexpr int LD = LMHEAD ? kLmLd : 128;               // epilogue tile row stride (floats)
  static constexpr int CH = KSPLIT == 1 ? 32 : BN;              // activation rows a readout chunk
  static constexpr int EPI_BYTES = CH * LD * 4;
  static constexpr int AUX_BYTES = 256 /*barriers*/ + BN * 4 * 4 /*red*/ + BN * 4 /*row scales*/ + BN * 16;
  static constexpr int SMEM_MAX = 232448;                       // 227 KB a CTA
  static constexpr int STAGES_RAW = (SMEM_MAX - 1024 - EPI_BYTES - AUX_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW < 6 ? STAGES_RAW : 6;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int SMEM = 1024 + RING_BYTES + EPI_BYTES + AUX_BYTES;
  static constexpr int THREADS = 192;
  static constexpr int PRODUCER = 4, MMA_WARP = 5;
  static_assert(STAGES >= 3, "ring too shallow");
  static_assert(TMEM_COLS <= 512, "TMEM holds 512 columns");
  static_assert(SMEM <= SMEM_MAX, "shared memory");
};

struct PersParams {
  int M, N, n_kb;
  int n_tiles, m_tiles;  // weight tiles (128 rows) and activation tiles (BN rows), host bounds
  float* out;            // EPI_NONE: the result [M][ldo]
  int ldo;
  const int* m_valid;
  int* status;
  EpiArgs epi;
  LmPartials lm;
  float* logits;
  long long ld_logits;
  const int* skip_rows;
  const int* logits_rows;
  int logits_bulk;
  // split tail (single-CTA projections): fp32 partial tiles [grid][BN][128]
  // and one arrival counter per tail tile (zero between launches), or null
  float* ws;
  int* ws_cnt;
};

// The most CTAs that share one tile of the last, partial round.
constexpr int kPersMaxSeg = 8;

// STORE / RESIDUAL epilogue of one tile, row-major: warp w finishes rows
// w, w + 4, ... and lane l the columns n0 + 4l .. n0 + 4l + 3 (128-bit loads
// and stores), eight rows a batch with their loads in flight together; the
// sum of z^2 of a row over the tile's columns is one warp reduction.  The
// same function as apply_epilogue's STORE / RESIDUAL branch (e.N a multiple
// of 4, bf16 next input).
__device__ __forceinline__ void epilogue_rows_vec(const EpiArgs& e, const float* tile, int m0, int rows, int n0,
                                                  const float* rs) {
  constexpr int B = 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = n0 + 4 * lane;
  const bool nv = n < e.N;  // N % 4 == 0: the four columns are valid together
  float4 gn = make_float4(0.f, 0.f, 0.f, 0.f);
  if (e.nx_hi != nullptr && nv) {
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(static_cast<const __nv_bfloat16*>(e.nx_gain) + n);
    const float2 a = __bfloat1622float2(g2[0]), b = __bfloat1622float2(g2[1]);
    gn = make_float4(a.x, a.y, b.x, b.y);
  }
  for (int j0 = warp; j0 < rows; j0 += 4 * B) {
    float4 z[B];
#pragma unroll
    for (int u = 0; u < B; ++u) {
      const int j = j0 + 4 * u;
      z[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (nv && j < rows && e.kind == EPI_RESIDUAL)
        z[u] = *reinterpret_cast<const float4*>(e.out + static_cast<long long>(m0 + j) * e.N + n);
    }
#pragma unroll
    for (int u = 0; u < B; ++u) {
      const int j = j0 + 4 * u;
      float sq = 0.f;
      if (nv && j < rows) {
        const float sc = rs != nullptr ? rs[j] : 1.f;
        const float4 t = *reinterpret_cast<const float4*>(tile + j * 128 + 4 * lane);
        float4 v = z[u];
        v.x += t.x * sc;
        v.y += t.y * sc;
        v.z += t.z * sc;
        v.w += t.w * sc;
        const long long o = static_cast<long long>(m0 + j) * e.N + n;
        if (e.out != nullptr) *reinterpret_cast<float4*>(e.out + o) = v;
        if (e.nx_hi != nullptr) {
          const float a0 = gn.x * v.x, a1 = gn.y * v.y, a2 = gn.z * v.z, a3 = gn.w * v.w;
          const __nv_bfloat162 h01 = __floats2bfloat162_rn(a0, a1), h23 = __floats2bfloat162_rn(a2, a3);
          const __nv_bfloat162 l01 = __floats2bfloat162_rn(a0 - __low2float(h01), a1 - __high2float(h01));
          const __nv_bfloat162 l23 = __floats2bfloat162_rn(a2 - __low2float(h23), a3 - __high2float(h23));
          uint2 hv, lv;
          hv.x = *reinterpret_cast<const uint32_t*>(&h01);
          hv.y = *reinterpret_cast<const uint32_t*>(&h23);
          lv.x = *reinterpret_cast<const uint32_t*>(&l01);
          lv.y = *reinterpret_cast<const uint32_t*>(&l23);
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(e.nx_hi) + o) = hv;
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(e.nx_lo) + o) = lv;
        }
        sq = (v.x * v.x + v.y * v.y) + (v.z * v.z + v.w * v.w);
      }
      if (e.ss_out != nullptr && j < rows) {  // uniform per warp
        sq = warp_sum(sq);
        if (lane == 0) e.ss_out[static_cast<long long>(n0 >> 7) * e.ss_ld + m0 + j] = sq;
      }
    }
  }
}

// QKV epilogue of one tile, row-major like epilogue_rows_vec: lane l takes
// columns n0 + 4l .. n0 + 4l + 3, which lie in one head (4 divides dh) and
// are all q, all k or all v.  q and k are rotated (rotate-half RoPE at the
// row's position: the partner columns i +- dh/2 and the cos / sin of the
// four frequencies come as 128-bit loads), then q goes to the query buffer
// and k, v to the sequence's block page, four fp16 values a store.  The same
// function as apply_epilogue's QKV branch (e.N and dh multiples of 4).
__device__ __forceinline__ void epilogue_qkv_vec(const EpiArgs& e, const float* tile, int m0, int rows, int n0,
                                                 const float* rs, const int4* ri) {
  constexpr int B = 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = 4 * lane, n = n0 + t;
  if (n >= e.N) return;  // per lane; no collective operations below
  const int qd = e.Hq * e.dh, kvd = e.Hkv * e.dh, half = e.dh / 2;
  const int kind = n < qd ? 0 : n < qd + kvd ? 1 : 2;
  const int w = kind == 0 ? n : kind == 1 ? n - qd : n - qd - kvd;
  const int head = w / e.dh, i = w % e.dh;
  const int jr = i < half ? i : i - half;  // first of the four RoPE frequencies
  const int base = t - i;                  // tile column of the head's element 0
  __half* q = static_cast<__half*>(e.q);
  __half* pk = static_cast<__half*>(e.pool_k);
  __half* pv = static_cast<__half*>(e.pool_v);
  for (int j0 = warp; j0 < rows; j0 += 4 * B) {
    float4 cs[B], sn[B];
#pragma unroll
    for (int u = 0; u < B; ++u) {
      const int j = j0 + 4 * u;
      cs[u] = sn[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (kind != 2 && j < rows) {
        const long long o = static_cast<long long>(ri[j].x) * half + jr;
        cs[u] = *reinterpret_cast<const float4*>(e.rope_cos + o);
        sn[u] = *reinterpret_cast<const float4*>(e.rope_sin + o);
      }
    }
#pragma unroll
    for (int u = 0; u < B; ++u) {
      const int j = j0 + 4 * u;
      if (j >= rows) break;
      const float* row = tile + j * 128;
      const float sc = rs != nullptr ? rs[j] : 1.f;
      float4 v;
      if (kind == 2) {
        v = *reinterpret_cast<const float4*>(row + t);
        v.x *= sc;
        v.y *= sc;
        v.z *= sc;
        v.w *= sc;
      } else {
        const float4 x1 = *reinterpret_cast<const float4*>(row + base + jr);
        const float4 x2 = *reinterpret_cast<const float4*>(row + base + jr + half);
        const float a1[4] = {x1.x * sc, x1.y * sc, x1.z * sc, x1.w * sc};
        const float a2[4] = {x2.x * sc, x2.y * sc, x2.z * sc, x2.w * sc};
        const float c[4] = {cs[u].x, cs[u].y, cs[u].z, cs[u].w};
        const float s[4] = {sn[u].x, sn[u].y, sn[u].z, sn[u].w};
        float r[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) r[k] = i < half ? a1[k] * c[k] - a2[k] * s[k] : a2[k] * c[k] + a1[k] * s[k];
        v = make_float4(r[0], r[1], r[2], r[3]);
      }
      const __half2 h01 = __floats2half2_rn(v.x, v.y), h23 = __floats2half2_rn(v.z, v.w);
      uint2 pkd;
      pkd.x = *reinterpret_cast<const uint32_t*>(&h01);
      pkd.y = *reinterpret_cast<const uint32_t*>(&h23);
      if (kind == 0) {
        *reinterpret_cast<uint2*>(q + static_cast<long long>(m0 + j) * qd + n) = pkd;
      } else {
        const long long idx = pool_index(ri[j].y, head, ri[j].z, i, e.Hkv, e.dh);
        *reinterpret_cast<uint2*>((kind == 1 ? pk : pv) + idx) = pkd;
      }
    }
  }
}

// KV_INJECT epilogue of one tile, row-major like epilogue_qkv_vec: lane l
// takes columns n0 + 4l .. n0 + 4l + 3, which lie in one head of one layer's
// K or V (4 divides dh).  K gets the optional key offset and RoPE at the
// row's position (cos / sin of its four frequencies as 128-bit loads), then
// the four values go to the row's page slot as one 8-byte fp16 store.  The
// same function as apply_epilogue's KV_INJECT branch (e.N and dh multiples
// of 4).
__device__ __forceinline__ void epilogue_kvinj_vec(const EpiArgs& e, const float* tile, int m0, int rows, int n0,
                                                   const float* rs, const int4* ri) {
  constexpr int B = 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = 4 * lane, n = n0 + t;
  if (n >= e.N) return;  // per lane; no collective operations below
  const int kvd = e.Hkv * e.dh, half = e.dh / 2;
  const int l = n / (2 * kvd), w = n % (2 * kvd);
  const bool is_k = w < kvd;
  const int head = (is_k ? w : w - kvd) / e.dh, i = w % e.dh;
  const int jr = i < half ? i : i - half;  // first of the four RoPE frequencies
  const int base = t - i;                  // tile column of the head's element 0
  float olo[4] = {0.f, 0.f, 0.f, 0.f}, ohi[4] = {0.f, 0.f, 0.f, 0.f};
  if (is_k && e.key_offset != nullptr) {
    const float* ko = e.key_offset + (static_cast<long long>(l) * e.Hkv + head) * e.dh;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      olo[k] = ko[jr + k];
      ohi[k] = ko[jr + k + half];
    }
  }
  __half* dst = static_cast<__half*>(is_k ? e.pool_k : e.pool_v) + static_cast<long long>(l) * e.layer_stride;
  for (int j0 = warp; j0 < rows; j0 += 4 * B) {
    float4 cs[B], sn[B];
#pragma unroll
    for (int u = 0; u < B; ++u) {
      const int j = j0 + 4 * u;
      cs[u] = sn[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (is_k && j < rows) {
        const long long o = static_cast<long long>(ri[j].x) * half + jr;
        cs[u] = *reinterpret_cast<const float4*>(e.rope_cos + o);
        sn[u] = *reinterpret_cast<const float4*>(e.rope_sin + o);
      }
    }
#pragma unroll
    for (int u = 0; u < B; ++u) {
      const int j = j0 + 4 * u;
      if (j >= rows) break;
      const float* row = tile + j * 128;
      const float sc = rs != nullptr ? rs[j] : 1.f;
      float r[4];
      if (!is_k) {
        const float4 v = *reinterpret_cast<const float4*>(row + t);
        r[0] = v.x * sc;
        r[1] = v.y * sc;
        r[2] = v.z * sc;
        r[3] = v.w * sc;
      } else {
        const float4 x1 = *reinterpret_cast<const float4*>(row + base + jr);
        const float4 x2 = *reinterpret_cast<const float4*>(row + base + jr + half);
        const float a1[4] = {x1.x * sc + olo[0], x1.y * sc + olo[1], x1.z * sc + olo[2], x1.w * sc + olo[3]};
        const float a2[4] = {x2.x * sc + ohi[0], x2.y * sc + ohi[1], x2.z * sc + ohi[2], x2.w * sc + ohi[3]};
        const float c[4] = {cs[u].x, cs[u].y, cs[u].z, cs[u].w};
        const float s[4] = {sn[u].x, sn[u].y, sn[u].z, sn[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) r[k] = i < half ? a1[k] * c[k] - a2[k] * s[k] : a2[k] * c[k] + a1[k] * s[k];
      }
      const __half2 h01 = __floats2half2_rn(r[0], r[1]), h23 = __floats2half2_rn(r[2], r[3]);
      uint2 pkd;
      pkd.x = *reinterpret_cast<const uint32_t*>(&h01);
      pkd.y = *reinterpret_cast<const uint32_t*>(&h23);
      *reinterpret_cast<uint2*>(dst + pool_index(ri[j].y, head, ri[j].z, i, e.Hkv, e.dh)) = pkd;
    }
  }
}

// Split tail (KSPLIT = 1 projections, given a workspace): the tiles are
// dealt round-robin in whole rounds of one tile a CTA, and the R < grid
// tiles of the last, partial round are each split in K among s =
// min(kPersMaxSeg, grid / R) CTAs (when that is at least 2), CTA u taking
// k-segment u % s of tail tile u / s; it writes its partial tile to its own
// workspace slot and counts itself in; the last of the s to arrive sums the
// s slots in segment order (the same order whoever is last) and runs the
// fused epilogue, then resets the count.  Nobody waits for another CTA.
//
// KSPLIT = 2: the two CTAs of a cluster share each tile, CTA r multiplying
// the k-blocks of half r (rank 0 takes the larger half).  Both read their
// accumulator out into their own tile, then CTA r sums rows 64 r .. 64 r + 63
// of its tile and of its peer's (distributed shared memory, rank 0's term
// first) and finishes those 64 rows.  The pair meets through mbarriers
// rather than cluster barriers, so the TMA and MMA threads never stop:
// `ready` (the peer's tile is complete), `cons` (the peer has read this
// CTA's tile, which may then take the next one).
template <int BN, bool LMHEAD, int KSPLIT>
__global__ void __launch_bounds__(PersCfg<BN, LMHEAD, KSPLIT>::THREADS, 1)
    k_gemm_pers(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                const __grid_constant__ CUtensorMap tmXlo, const __grid_constant__ PersParams p) {
  using C = PersCfg<BN, LMHEAD, KSPLIT>;
  static_assert(KSPLIT == 1 || (KSPLIT == 2 && !LMHEAD && BN == 128), "split tiles: 128-row projections");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;                                         // [STAGES][W | X hi | X lo]
  float* tile = reinterpret_cast<float*>(smem + C::RING_BYTES);  // [CH][LD] epilogue tile (a readout chunk)
  uint8_t* aux = smem + C::RING_BYTES + C::EPI_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(aux);            // [STAGES] stage landed
  uint64_t* empty = full + C::STAGES;                           // [STAGES] stage consumed by the MMAs
  uint64_t* accf = empty + C::STAGES;                           // [2] accumulator complete
  uint64_t* acce = accf + 2;                                    // [2] accumulator read out
  uint64_t* ready = acce + 2;                                   // KSPLIT 2: the peer's tile is complete
  uint64_t* cons = ready + 1;                                   // KSPLIT 2: the peer has read this tile
  uint64_t* fixb = cons + 1;                                    // split tail: the partial tiles' chunk landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fixb + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_last = s_abort + 1;  // split tail: this CTA finishes its tail tile
  static_assert((2 * C::STAGES + 7) * 8 + 12 <= 256, "barrier area");
  static_assert(KSPLIT != 1 || LMHEAD || kPersMaxSeg * C::CH * 128 * 4 <= C::RING_BYTES, "a chunk of every partial fits the ring");
  float* red = reinterpret_cast<float*>(aux + 256);             // [BN][4]
  float* s_rs = red + 4 * BN;                                   // folded-RMSNorm row scales
  int4* s_ri = reinterpret_cast<int4*>(s_rs + BN);              // per-row epilogue facts

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = KSPLIT == 2 ? static_cast<int>(cluster_ctarank()) : 0;
  const int unit = static_cast<int>(blockIdx.x) / KSPLIT, n_units = static_cast<int>(gridDim.x) / KSPLIT;
  // this CTA's k-blocks of every tile
  const int kb_half = (p.n_kb + 1) / 2;
  const int kb0 = KSPLIT == 2 && rank == 1 ? kb_half : 0;
  const int kb1 = KSPLIT == 2 && rank == 0 ? kb_half : p.n_kb;
  const int nkb = kb1 - kb0;
  // the rows this CTA finishes: all of a tile, or its half
  constexpr int ROWS = BN / KSPLIT;
  const int r0 = rank * ROWS;
  // m_valid is written two kernels upstream (page allocation), never by the
  // predecessor, so every role may size the work list before pdl_wait
  const int mv = p.m_valid != nullptr ? min(p.M, __ldg(p.m_valid)) : p.M;
  const int m_tiles = min(p.m_tiles, (mv + BN - 1) / BN);
  const int n_work = p.n_tiles * m_tiles;
  // the split tail: n_full whole rounds, then rem tiles in n_seg segments each
  const int n_full = n_work / n_units, rem = n_work - n_full * n_units;
  // (at least one k-block a segment)
  const int n_seg = KSPLIT == 1 && !LMHEAD && p.ws != nullptr && rem > 0 ? min(min(kPersMaxSeg, n_units / rem), nkb) : 1;
  const bool split_tail = n_seg >= 2;
  const int my_tiles = split_tail ? n_full + (unit < rem * n_seg ? 1 : 0)
                       : unit < n_work ? (n_work - unit + n_units - 1) / n_units
                                       : 0;
  const int tail_idx = unit / n_seg;  // (split tail) this CTA's tail tile, after the n_full rounds
  // tile tl of this CTA: its corner and its k-blocks [ka, kz)
  auto tile_of = [&](int tl, int& n0, int& m0, int& ka, int& kz) {
    int t = unit + tl * n_units;
    ka = kb0;
    kz = kb1;
    if (split_tail && tl == n_full) {
      const int sg = unit % n_seg;
      t = n_full * n_units + tail_idx;
      ka = kb0 + sg * nkb / n_seg;
      kz = kb0 + (sg + 1) * nkb / n_seg;
    }
    n0 = (t / m_tiles) * kTileN;
    m0 = (t % m_tiles) * BN;
  };

  if (warp == C::PRODUCER && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmXlo);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accf[a], 1);
      mbar_init(&acce[a], 4);  // one arrival per epilogue warp
    }
    mbar_init(ready, 1);
    mbar_init(cons, 1);
    mbar_init(fixb, 1);
    *s_abort = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (KSPLIT == 2) {
    // the peer's barriers are initialised before anything arrives on them
    cluster_arrive();
    cluster_wait();
  }
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == C::PRODUCER) {
    if (lane == 0) {
      // a cursor over (tile, k-block) in issue order
      int total = 0;
      for (int tl = 0; tl < my_tiles; ++tl) {
        int n0, m0, ka, kz;
        tile_of(tl, n0, m0, ka, kz);
        total += kz - ka;
      }
      int c_tl = 0, c_kb = 0, c_kz = 0, c_n0 = 0, c_m0 = 0;
      if (my_tiles > 0) tile_of(0, c_n0, c_m0, c_kb, c_kz);
      auto coords = [&](int& n0, int& m0, int& kx) {  // the cursor's stage, then advance
        n0 = c_n0;
        m0 = c_m0;
        kx = c_kb * kTileK;
        if (++c_kb == c_kz && ++c_tl < my_tiles) tile_of(c_tl, c_n0, c_m0, c_kb, c_kz);
      };
      // the weights do not depend on the predecessor: the first stages'
      // weight tiles go out before its completion, their activations after
      const int pre = min(total, C::STAGES);
      int pm0[C::STAGES], pkx[C::STAGES];
      for (int it = 0; it < pre; ++it) {
        int n0;
        coords(n0, pm0[it], pkx[it]);
        mbar_arrive_expect_tx(&full[it], C::STAGE_BYTES);
        tma_load_2d(ring + it * C::STAGE_BYTES, &tmW, &full[it], pkx[it], n0);
      }
      pdl_wait();
      pdl_trigger();
      for (int it = 0; it < pre; ++it) {
        uint8_t* st = ring + it * C::STAGE_BYTES;
        tma_load_2d(st + C::W_BYTES, &tmX, &full[it], pkx[it], pm0[it]);
        tma_load_2d(st + C::W_BYTES + C::X_BOX, &tmXlo, &full[it], pkx[it], pm0[it]);
      }
      int issued = pre;
      for (int it = pre; it < total; ++it) {
        const int s = it % C::STAGES;
        if (*s_abort || !mbar_wait_spin(&empty[s], ((it / C::STAGES) & 1) ^ 1, p.status)) {
          *s_abort = 1;
          break;
        }
        int n0, m0, kx;
        coords(n0, m0, kx);
        uint8_t* st = ring + s * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
        tma_load_2d(st, &tmW, &full[s], kx, n0);
        tma_load_2d(st + C::W_BYTES, &tmX, &full[s], kx, m0);
        tma_load_2d(st + C::W_BYTES + C::X_BOX, &tmXlo, &full[s], kx, m0);
        issued = it + 1;
      }
      // leave only once every copy this thread issued has landed
      for (int it = max(0, issued - C::STAGES); it < issued; ++it)
        mbar_wait(&full[it % C::STAGES], (it / C::STAGES) & 1, p.status);
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    if (lane == 0) {
      constexpr uint32_t idesc = mma_idesc_bf16_f32(kTileN, C::NMMA);
      int it = 0;
      bool ok = true;
      for (int tl = 0; ok && tl < my_tiles; ++tl) {
        const int a = tl & 1;
        // the epilogue has read accumulator a out (its use two tiles ago)
        if (tl >= 2 && (*s_abort || !mbar_wait(&acce[a], ((tl >> 1) & 1) ^ 1, p.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + static_cast<uint32_t>(a * C::ACC_COLS);
        int n0, m0, ka, kz;
        tile_of(tl, n0, m0, ka, kz);
        for (int kb = 0; kb < kz - ka; ++kb, ++it) {
          const int s = it % C::STAGES;
          if (*s_abort || !mbar_wait_spin(&full[s], (it / C::STAGES) & 1, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t aW = smem_u32(ring + s * C::STAGE_BYTES);
          const uint32_t aX = aW + C::W_BYTES;
#pragma unroll
          for (int k = 0; k < kTileK / 16; ++k)
            tc_mma_bf16(acc, sw128_kmajor_desc(aW + 32 * k), sw128_kmajor_desc(aX + 32 * k), idesc,
                        (kb | k) != 0 ? 1u : 0u);
          tc_commit(&empty[s]);
        }
        if (ok) tc_commit(&accf[a]);
      }
      if (!ok) *s_abort = 1;
    }
    __syncwarp();
  } else {
    // ---- epilogue warps 0-3: TMEM lane quadrant = warp
    pdl_wait();  // the row facts below read the predecessor's output
    bool live = true;
    const uint32_t tquad = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    for (int tl = 0; tl < my_tiles; ++tl) {
      int n0, m0, ka, kz;
      tile_of(tl, n0, m0, ka, kz);
      const bool seg_tile = split_tail && tl == n_full;  // a k-segment of a tail tile
      const int n = n0 + warp * 32 + lane;
      const bool nv = n < p.N;
      // the fused epilogue of activation rows c0 .. of the tile, staged in
      // `mine` (fr: the first one's index in the row facts)
      auto finish = [&](int c0, float* mine, int fr) {
        const int mr0 = KSPLIT == 2 ? m0 + r0 : m0 + c0;  // first output row of `mine`
        constexpr int NR = KSPLIT == 2 ? ROWS : C::CH;
        const int rows = min(NR, mv - mr0);
        if constexpr (LMHEAD) {
          const bool bulk_out = p.logits != nullptr && p.logits_bulk && n0 + kTileN <= p.N;
          if (!bulk_out && p.logits != nullptr && nv)
            for (int j = 0; j < C::CH; ++j)
              if (s_ri[c0 + j].w != 0)
                __stcs(p.logits + s_ri[c0 + j].x * p.ld_logits + n, tile[j * C::LD + warp * 32 + lane]);
          if (bulk_out) fence_proxy_async_smem();
          epi_sync();
          if (bulk_out && warp == 0) {
            const uint64_t pol = l2_policy_evict_first();
            for (int j = lane; j < C::CH; j += 32)
              if (s_ri[c0 + j].w != 0)
                bulk_store_global(p.logits + s_ri[c0 + j].x * p.ld_logits + n0, smem_u32(tile + j * C::LD), kTileN * 4,
                                  pol);
            bulk_commit();
          }
          // (max, lowest argmax, sum of exp(z - max)) of each row over the
          // tile's 128 columns: 8 threads a row, 16 rows at a time
          const int seg = threadIdx.x & 7;
          const int ntile = n0 / kTileN;
#pragma unroll 1
          for (int rb = 0; rb < C::CH; rb += kEpiThreads >> 3) {
            const int j = rb + (threadIdx.x >> 3);
            const float* row = tile + j * C::LD;
            float z[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) z[k] = row[seg + 8 * k];
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
            const int m = mr0 + j;
            if (seg == 0 && m < mv) {
              const long long o = static_cast<long long>(m) * p.lm.n_tiles + ntile;
              p.lm.mx[o] = mx;
              p.lm.se[o] = se;
              p.lm.idx[o] = n0 + ix;
            }
          }
          if (bulk_out && warp == 0) bulk_wait_read_all();  // the copies have read the chunk
        } else {
          epi_sync();  // the rows are complete
          const float* rs = p.epi.ss_in != nullptr ? s_rs + fr : nullptr;
          if (rows > 0) {
            if (p.epi.kind == EPI_NONE) {
              const int t = threadIdx.x;
              for (int j = 0; j < rows; ++j)
                if (n0 + t < p.N) p.out[static_cast<long long>(mr0 + j) * p.ldo + n0 + t] = mine[j * 128 + t];
            } else if ((p.epi.kind == EPI_STORE || p.epi.kind == EPI_RESIDUAL) && p.N % 4 == 0) {
              epilogue_rows_vec(p.epi, mine, mr0, rows, n0, rs);
            } else if (p.epi.kind == EPI_QKV && p.N % 4 == 0 && p.epi.dh % 8 == 0) {
              epilogue_qkv_vec(p.epi, mine, mr0, rows, n0, rs, s_ri + fr);
            } else if (p.epi.kind == EPI_KV_INJECT && p.N % 4 == 0 && p.epi.dh % 8 == 0) {
              epilogue_kvinj_vec(p.epi, mine, mr0, rows, n0, rs, s_ri + fr);
            } else {
              EpiPre pre;
              epilogue_preload<__nv_bfloat16>(p.epi, mr0, NR, n0, s_ri + fr, pre);
              apply_epilogue<__nv_bfloat16, __half>(p.epi, mine, mr0, NR, n0, rs, s_ri + fr, red, &pre);
            }
          }
        }
      };
      // row facts of the rows this CTA finishes (s_rs / s_ri index j of row r0 + j)
      for (int j = threadIdx.x; j < ROWS; j += kEpiThreads) {
        const int m = m0 + r0 + j;
        const bool ok = m < mv;
        if (p.epi.ss_in != nullptr) s_rs[j] = ok ? norm_row_scale(p.epi, m) : 0.f;
        if constexpr (LMHEAD) {
          const int orow = ok ? (p.logits_rows != nullptr ? p.logits_rows[m] : m) : -1;
          s_ri[j] = make_int4(orow, 0, 0, orow >= 0 && (p.skip_rows == nullptr || p.skip_rows[m] == 0) ? 1 : 0);
        } else {
          s_ri[j] = ok ? epi_row_info(p.epi, m) : make_int4(0, 0, 0, 0);
        }
      }
      const int a = tl & 1;
      live = live && !*s_abort && mbar_wait(&accf[a], (tl >> 1) & 1, p.status);
      if constexpr (KSPLIT == 2) {
        // the peer has read this CTA's previous tile
        if (tl >= 1) live = live && !*s_abort && mbar_wait_cluster(cons, (tl - 1) & 1, p.status);
      }
      if (!live) *s_abort = 1;
      __syncwarp();
      tc_fence_after();
      epi_sync();  // the row facts are complete
      const uint32_t tacc = tquad + static_cast<uint32_t>(a * C::ACC_COLS);
      constexpr int CH = C::CH;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += CH) {
        // activation rows c0 .. c0 + CH - 1 of the tile into the staging tile
#pragma unroll 1
        for (int c = c0; c < c0 + CH; c += 16) {
          float v[16], v2[16];
          if (live) {
            tc_ld_32x32b_x16(tacc + c, v);
            tc_ld_32x32b_x16(tacc + BN + c, v2);
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float z = live ? v[j] + v2[j] : 0.f;
            if constexpr (LMHEAD) z = nv ? (p.epi.ss_in != nullptr ? z * s_rs[c + j] : z) : -INFINITY;
            tile[(c - c0 + j) * C::LD + warp * 32 + lane] = z;
          }
        }
        if (c0 + CH == BN) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbarrier_arrive_one(&acce[a]);  // accumulator a may take the tile after next
        }
        if (seg_tile) {
          // a k-segment's partial: the chunk into this CTA's workspace slot
          epi_sync();
          float* slot = p.ws + static_cast<long long>(unit) * BN * 128;
          for (int e = threadIdx.x; e < CH * 32; e += kEpiThreads) {
            const int j = e >> 5, c4 = (e & 31) * 4;
            __stcg(reinterpret_cast<float4*>(slot + (c0 + j) * 128 + c4),
                   *reinterpret_cast<const float4*>(tile + j * C::LD + c4));
          }
          epi_sync();  // the staging tile is free again
          continue;
        }
        // the rows this CTA finishes from this chunk: a chunk of its own
        // tile (KSPLIT 1), or its half of the pair's sum (KSPLIT 2); fr: the
        // first one's index in the row facts
        float* mine = tile;
        int fr = c0;
        if constexpr (KSPLIT == 2) {
          // both halves of the sum: the peer's tile complete, add its rows
          // r0 .. r0 + 63 to ours (rank 0's term first), then let it reuse
          // its tile
          mine = tile + r0 * C::LD;
          fr = 0;
          epi_sync();
          if (threadIdx.x == 0) {
            fence_acq_rel_cluster();
            mbar_remote_arrive(ready, static_cast<uint32_t>(rank ^ 1));
          }
          live = live && !*s_abort && mbar_wait_cluster(ready, tl & 1, p.status);
          if (!live) *s_abort = 1;
          const uint32_t peer = dsmem_map(smem_u32(mine), static_cast<uint32_t>(rank ^ 1));
          for (int e = threadIdx.x; e < ROWS * 32; e += kEpiThreads) {
            const int j = e >> 5, c4 = (e & 31) * 4;
            float4 own = *reinterpret_cast<const float4*>(mine + j * 128 + c4);
            const float4 oth =
                live ? ld_dsmem_f4(peer + static_cast<uint32_t>((j * 128 + c4) * 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
            float4 sum = rank == 0 ? make_float4(own.x + oth.x, own.y + oth.y, own.z + oth.z, own.w + oth.w)
                                   : make_float4(oth.x + own.x, oth.y + own.y, oth.z + own.z, oth.w + own.w);
            *reinterpret_cast<float4*>(mine + j * 128 + c4) = sum;
          }
          epi_sync();
          if (threadIdx.x == 0) {
            fence_acq_rel_cluster();
            mbar_remote_arrive(cons, static_cast<uint32_t>(rank ^ 1));
          }
        }
        finish(c0, mine, fr);
        epi_sync();  // the staging tile is free again
      }
      if (seg_tile) {
        // count this segment in; the last of the tile's n_seg sums their
        // slots in segment order and finishes the tile
        __threadfence();
        epi_sync();
        if (threadIdx.x == 0) *s_last = atomicAdd(&p.ws_cnt[tail_idx], 1) == n_seg - 1 ? 1 : 0;
        epi_sync();
        if (*s_last) {
          // chunk by chunk, the n_seg partials' rows come into the ring (idle:
          // this is the CTA's last tile) by bulk copies, are summed in segment
          // order into the staging tile and finished
          __threadfence();
          if (threadIdx.x == 0) fence_proxy_async_global();
          const float* base = p.ws + static_cast<long long>(tail_idx) * n_seg * BN * 128;
          const float* part = reinterpret_cast<const float*>(ring);  // [n_seg][CH][128]
          constexpr uint32_t CHUNK = CH * 128 * 4;
#pragma unroll 1
          for (int c0 = 0; c0 < BN; c0 += CH) {
            if (threadIdx.x == 0) {
              mbar_arrive_expect_tx(fixb, static_cast<uint32_t>(n_seg) * CHUNK);
              for (int sg = 0; sg < n_seg; ++sg)
                bulk_load_global(smem_u32(ring) + sg * CHUNK, base + (static_cast<long long>(sg) * BN + c0) * 128, CHUNK,
                                 fixb);
            }
            live = live && mbar_wait(fixb, (c0 / CH) & 1, p.status);
            for (int e = threadIdx.x; e < CH * 32; e += kEpiThreads) {
              const int j = e >> 5, c4 = (e & 31) * 4;
              float4 acc = *reinterpret_cast<const float4*>(part + j * 128 + c4);
              for (int sg = 1; sg < n_seg; ++sg) {
                const float4 v = *reinterpret_cast<const float4*>(part + (sg * CH + j) * 128 + c4);
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
              }
              *reinterpret_cast<float4*>(tile + j * C::LD + c4) = acc;
            }
            finish(c0, tile, c0);  // (its first step is a barrier: the chunk is complete, the ring read)
            epi_sync();            // the staging tile is free again
          }
          if (threadIdx.x == 0) p.ws_cnt[tail_idx] = 0;  // for the next launch
        }
      }
    }
    if constexpr (KSPLIT == 2) {
      // the peer has read the last tile before this CTA's shared memory goes
      if (my_tiles > 0 && live && !*s_abort) mbar_wait_cluster(cons, (my_tiles - 1) & 1, p.status);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Cluster pairs of k_gemm_pers<128, false, 2> that fit at once (0 if the
// query fails).
inline int pers_split_clusters(int smem) {
  static FuncAttr smem_attr;
  if (smem_attr.ensure(smem, [](int v) {
        return cudaFuncSetAttribute(k_gemm_pers<128, false, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, v);
      }) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(2, 1, 1);
  lc.blockDim = dim3(PersCfg<128, false, 2>::THREADS);
  lc.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_gemm_pers<128, false, 2>, &lc) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int BN, bool LM, int KSPLIT>
cudaError_t launch_pers(dflash_ctx* c, const GemmLaunch& g, const CUtensorMap& tw, const CUtensorMap& tx,
                        const CUtensorMap& txlo, cudaStream_t s) {
  using C = PersCfg<BN, LM, KSPLIT>;
  static FuncAttr smem_attr;
  cudaError_t ae = smem_attr.ensure(C::SMEM, [](int v) {
    return cudaFuncSetAttribute(k_gemm_pers<BN, LM, KSPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, v);
  });
  if (ae != cudaSuccess) return ae;
  PersParams p{};
  p.M = g.M;
  p.N = g.N;
  p.n_kb = gemm_kb(g.K);
  p.n_tiles = (g.N + kTileN - 1) / kTileN;
  p.m_tiles = (g.M + BN - 1) / BN;
  p.out = g.out;
  p.ldo = g.ldo;
  p.m_valid = g.m_valid;
  p.status = c->status;
  p.epi = g.epi;
  p.lm = g.lm;
  p.logits = g.logits;
  p.ld_logits = g.ld_logits;
  p.skip_rows = g.skip_rows;
  p.logits_rows = g.logits_rows;
  p.logits_bulk = g.logits != nullptr && (reinterpret_cast<uintptr_t>(g.logits) & 15) == 0 && g.ld_logits % 4 == 0;
  if (KSPLIT == 1 && !LM && c->pers_ws != nullptr && BN == 128) {
    p.ws = c->pers_ws;  // one slot per CTA: the grid is at most num_sms
    p.ws_cnt = c->pers_cnt;
  }
  const int work = p.n_tiles * p.m_tiles;
  int grid;
  if (KSPLIT == 2) {
    const int clusters = std::max(1, std::min(work, c->pers_split_clusters));
    grid = 2 * clusters;
  } else {
    grid = std::max(1, std::min(work, c->num_sms));
  }
  return launch_k(k_gemm_pers<BN, LM, KSPLIT>, dim3(grid), dim3(C::THREADS), C::SMEM, s, dim3(KSPLIT), c->pdl, tw, tx,
                  txlo, p);
}

}  // namespace dflash

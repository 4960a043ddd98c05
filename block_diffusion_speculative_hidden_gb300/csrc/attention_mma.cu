// Block attention on the fifth-generation tensor cores (tcgen05) for the fp16
// KV pool of bf16 workloads.
//
// The contraction is the one attention.cu computes in fp32: the K block
// queries of one sequence attend, unmasked, to every injected context key
// and to all K keys of the block itself (DFlash Guide, "1. Single-Pass
// Block-Diffusion Drafting": bidirectional attention inside the masked
// block; "3. Cross-Layer KV Injection": the context keys come from the
// target's fused features).  Layout and schedule:
//
//   - one CTA per (sequence, kv head, key split), 10 warps: warps 0-7 run
//     the softmax (two per TMEM lane quadrant, splitting the pages of a
//     block), warp 8 drives TMA, one thread of warp 9 issues the MMAs;
//   - the split's pages are taken KBP pages (16*KBP keys) at a time through
//     an NST-deep ring of K / V tiles (4-D TMA, 128-byte swizzle);
//   - S = Q K^T is one MMA chain per key block (query rows on M = 64 or
//     128, keys on N, accumulated in TMEM); the softmax threads read S, form
//     the block's row max, P = 2^(S*scale - max) in fp16 and the running
//     sums, and O_blk = P V follows (V enters as an MN-major operand).  Three
//     schedules:
//       * one key block (ONE): O over the columns of S, read out at the end;
//       * serial blocks (SEPO): S and O in TMEM columns of their own, P over
//         the block's K tile, O accumulated in TMEM over the blocks and
//         rescaled there only when a row's max passes the one P is taken
//         against by more than 2^8, so S of the next block waits for
//         neither P V nor a fold;
//       * pipelined 4-page blocks (PIPE, dh 64): two S and two O buffers, S
//         of the next block and P V of this one under the softmax, O folded
//         into registers a block late; the 128-row case (row-wise softmax,
//         one query row a thread) keeps P in TMEM over its S columns as the
//         P V product's A operand, three S buffers and one O accumulated in
//         TMEM with the same lazy rescale;
//   - only the real query rows of Q and P are stored: the MMA's padding rows
//     (G*16 .. 127) read whatever follows in shared memory, and the results
//     in those rows are never used;
//   - everything that does not depend on the QKV projection (barriers, TMEM,
//     page ids, the context pages) is set up before the programmatic-launch
//     wait; q and the block page come after it;
//   - with several splits, the splits of one (sequence, kv head) form a
//     cluster and merge (o, m, l) with bulk copies between the CTAs' shared
//     memories;
//   - grid slot z serves sequence order[z] when an order is given (longest
//     context first, so that in a grid of several waves the long streams
//     start early).
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"

namespace dflash {

namespace {

constexpr int kMergeMax = 16;  // splits merged in one cluster (16 needs the non-portable size)
constexpr int kAttnThreads = 320;  // 8 softmax warps, the TMA warp, the MMA warp
constexpr int kProducerWarp = 8, kMmaWarp = 9;

// TMEM layout of the accumulators (rows = query rows, columns = keys or head
// dims): with M = 64, row r sits in lane 32*(r/16) + r%16; with M = 128, row
// r in lane r.  The softmax reads 16-lane blocks with the 16x256b shape:
// thread t of the warp gets rows t/4 and t/4 + 8 of the block, columns
// 2*(t%4) and 2*(t%4) + 1 of every 8-column group.
//
// Columns (256 a CTA, two CTAs an SM): one key block — S at column 0 and O
// = P V over it; serial blocks — S at column 0, O after it; pipelined
// 4-page blocks (two S and two O buffers fit: dh 64) — S of the next key
// block is computed while the softmax turns this block's S into P, and O of
// a block is folded one block late (after the next block's P is written),
// so the P V product runs under the softmax too; with 128 rows, three S
// buffers and one O (see P_TMEM below).
template <int DH, int G, int KBP, int NST>
struct MmaAttnLayout {
  static constexpr int R = G * 16;                 // real query rows
  static constexpr int M = R <= 64 ? 64 : 128;     // MMA rows
  static constexpr int SUB = M / 64;               // 16-lane row blocks per TMEM quadrant
  static constexpr int QUADS = R <= 64 ? R / 16 : 4;  // quadrants holding real rows
  static constexpr int RPT = 2 * SUB;              // rows per softmax thread
  static constexpr int NCH = DH / 64;              // 128-byte column chunks of a head
  static constexpr bool ONE = NST == 1;            // the split is one key block
  static constexpr int SW = 16 * KBP;              // S columns of a key block
  static constexpr int TMEM_COLS = 256;
  static constexpr bool PIPE = !ONE && KBP <= 4 && 2 * SW + 2 * DH <= TMEM_COLS;
  // the pipelined 128-row variant (row-wise softmax) keeps P in TMEM: each
  // page's 16 fp16 values a row over the first 8 of that page's own S
  // columns, the P V product's A operand; O accumulates in one TMEM buffer,
  // so three S buffers fit (S of the next block never waits for the P V
  // product of the previous one)
  static constexpr bool P_TMEM = M == 128 && PIPE && DH == 64 && 3 * SW + DH <= TMEM_COLS;
  static constexpr int NSB = P_TMEM ? 3 : PIPE ? 2 : 1;  // S buffers
  static constexpr int NO = PIPE ? 2 : 1;          // O buffers (P in TMEM: one, two commit barriers)
  // the serial multi-block variants keep S and O in columns of their own: O
  // accumulates over the blocks in TMEM (rescaled there only when a row's
  // max moves, as in the row-wise variant), so S of the next block waits
  // neither for the P V product nor for a fold
  static constexpr bool SEPO = !ONE && !PIPE;
  __host__ __device__ static constexpr int s_col(int j) { return PIPE ? j * SW : 0; }
  __host__ __device__ static constexpr int o_col(int j) { return PIPE ? NSB * SW + j * DH : SEPO ? SW : 0; }
  static constexpr int Q_CH = R * 128;             // stride of the Q chunks (real rows only)
  static constexpr int Q_BYTES = NCH * Q_CH;
  static constexpr int P_CHUNKS = (KBP * 16 + 63) / 64;
  static constexpr int P_CH = R * 128;
  static constexpr int P_BYTES = P_CHUNKS * P_CH;
  static constexpr int KV_CH = KBP * 16 * 128;     // one 64-column chunk of the K (or V) tile
  static constexpr int KV_BYTES = NCH * KV_CH;
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;  // K then V
  // P overwrites the block's K tile (dead once S is computed) when it fits;
  // otherwise it has a buffer per O buffer (P of the next block is written
  // while the P V product of this one may still read its buffer)
  static constexpr bool P_IN_K = P_BYTES <= KV_BYTES;
  static constexpr int NPB = P_IN_K || P_TMEM ? 0 : NO;
  __host__ __device__ static constexpr int p_off(int blk) { return NPB > 1 ? (blk % (NPB > 1 ? NPB : 1)) * P_BYTES : 0; }
  static constexpr int OFF_P = Q_BYTES;
  static constexpr int OFF_KV = OFF_P + NPB * P_BYTES;
  static constexpr int OFF_BAR = OFF_KV + NST * STAGE_BYTES;
  static constexpr int BAR_AREA = 256;             // mbarriers and the TMEM address
  static constexpr int BAR_BYTES = BAR_AREA + 8 * 32 * RPT * 4;  // then the pair-exchange slots
  static constexpr int SMEM_FIXED = 1024 + OFF_BAR + BAR_BYTES;  // + 4 bytes per page id
  // the padding rows (R .. M-1) of the last Q / P chunk read into the
  // following buffers, never past the allocation
  static constexpr bool q_padding_inside = (NCH - 1) * Q_CH + M * 128 <= OFF_BAR + BAR_BYTES;
  static constexpr bool p_padding_inside =
      P_TMEM || (P_IN_K ? OFF_KV + (NST - 1) * STAGE_BYTES : OFF_P + (NPB - 1) * P_BYTES) + (P_CHUNKS - 1) * P_CH +
                        M * 128 <=
                    OFF_BAR + BAR_BYTES;
  // a split merge stages its rows [R][DH + 4] and receives the partials
  // [splits][rows per split][DH + 4] in Q, P and the ring: the largest split
  // count (at most kMergeMax) whose merge fits (one split needs no merge)
  static constexpr int merge_rows(int S) { return R + S * ((R + S - 1) / S); }
  static constexpr int max_merge() {
    int m = 1;
    for (int S = 2; S <= kMergeMax; ++S)
      if (merge_rows(S) * (DH + 4) * 4 <= OFF_BAR) m = S;
    return m;
  }
  static constexpr int MAX_MERGE = max_merge();
};

template <int DH, int G, int KBP, int NST>
struct MmaAttnCfg : MmaAttnLayout<DH, G, KBP, NST> {
  using L = MmaAttnLayout<DH, G, KBP, NST>;
  static_assert(KBP * 16 <= 256 && DH <= 256, "one MMA's N");
  static_assert(L::P_TMEM   ? 3 * L::SW + DH <= L::TMEM_COLS
                : L::PIPE ? 2 * L::SW + 2 * DH <= L::TMEM_COLS
                : L::SEPO ? L::SW + DH <= L::TMEM_COLS
                          : KBP * 16 <= L::TMEM_COLS && DH <= L::TMEM_COLS,
                "S and O buffers fit the allocation");
  static_assert((2 * NST + 13) * 8 <= L::BAR_AREA, "barriers fit their area");
  static_assert(L::q_padding_inside, "Q padding rows stay inside");
  static_assert(L::p_padding_inside, "P padding rows stay inside");
  // the 8-page variants merge any split count
  static_assert(KBP < 8 || L::MAX_MERGE == kMergeMax, "split partials must fit");
};

struct MmaAttnParams {
  const int32_t* page_table;
  const int32_t* seq_len;  // context length of block b
  const int32_t* row_of;   // page-table row of block b (null: row b)
  const int32_t* order;    // block served by grid slot z (null: z)
  int max_pages, block_page0, pool_pages, layer;
  int Hkv, splits;
  int page_slots;     // capacity of the shared-memory page-id list
  float scale_log2;   // log2(e) / sqrt(dh)
  void* o_hi;         // ActOut<bf16> of the attention output [B*16][Hq*DH]
  void* o_lo;
  int* status;
  L2Plan l2;          // the O projection's weights, prefetched into L2 once QKV completed
};

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                            int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

// 16 TMEM lanes x 16 (x2) or 32 (x4) columns in the 16x256b fragment layout.
__device__ __forceinline__ void tc_ld_16x256b_x2(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tc_ld_16x256b_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tc_st_16x256b_x4(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// 2^x for the softmax: one ex2.approx (results below 2^-126 flush to zero;
// P is stored in fp16, where they are zero anyway)
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// how far (log2 units) a row's max may pass the one its P is taken against
// before O is rescaled (row-wise variant): P stays at most 2^8 in fp16
constexpr float kLazyRescale = 8.f;
// the three-input maximum of sm_100 and later (one instruction)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

template <int DH, int G, int KBP, int NST>
__global__ void __launch_bounds__(kAttnThreads, KBP <= 4 ? 2 : 1) k_attn_mma(const __grid_constant__ CUtensorMap tmQ,
                                                              const __grid_constant__ CUtensorMap tmK,
                                                              const __grid_constant__ CUtensorMap tmV,
                                                              const __grid_constant__ CUtensorMap tmNext,
                                                              const __grid_constant__ MmaAttnParams p) {
  using C = MmaAttnCfg<DH, G, KBP, NST>;
  constexpr int R = C::R;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sP = smem + C::OFF_P;
  uint8_t* sKV = smem + C::OFF_KV;
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_empty = kv_full + NST;
  uint64_t* q_full = kv_empty + NST;
  uint64_t* s_full = q_full + 1;  // [3]: per S buffer
  uint64_t* p_full = q_full + 4;  // [3]: per S buffer (P of the block in it is written)
  uint64_t* o_full = q_full + 7;  // [2]: per O buffer (P in TMEM: by the block's parity)
  uint64_t* o_free = q_full + 9;  // [2]: per O buffer (folded into registers)
  uint64_t* recv_bar = q_full + 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_full + 12);
  float* s_red = reinterpret_cast<float*>(smem + C::OFF_BAR + C::BAR_AREA);  // [8 warps][32 lanes][RPT] pair exchange
  int* s_pages = reinterpret_cast<int*>(smem + C::OFF_BAR + C::BAR_BYTES);

  const int sp = blockIdx.x, kvh = blockIdx.y, b = p.order != nullptr ? p.order[blockIdx.z] : blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.seq_len[b];
  const int prow = p.row_of != nullptr ? p.row_of[b] : b;
  const int n_ctx_pages = (T + kPage - 1) / kPage;
  const int n_pages = n_ctx_pages + 1;  // + the block page
  const int per_split = (n_pages + p.splits - 1) / p.splits;
  const int vp_begin = min(n_pages, sp * per_split), vp_end = min(n_pages, vp_begin + per_split);
  const int np = min(vp_end - vp_begin, p.page_slots);
  const int nblk = (np + KBP - 1) / KBP;
  constexpr int SOFT = 2 * C::QUADS * 32;  // softmax threads: two warps per TMEM quadrant holding real rows

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(q_full, 1);
    for (int j = 0; j < 3; ++j) {
      mbar_init(&s_full[j], 1);
      mbar_init(&p_full[j], SOFT);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(&o_full[j], 1);
      mbar_init(&o_free[j], SOFT);
    }
    mbar_init(recv_bar, 1);
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == kProducerWarp) {
    // page ids of this split (context pages, then the block page), so that
    // issuing a block never waits on a global load
    for (int j = lane; j < np; j += 32) {
      const int vp = vp_begin + j;
      s_pages[j] = vp < n_ctx_pages ? p.page_table[prow * p.max_pages + vp] : p.block_page0 + b;
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Softmax warps: warp w serves TMEM quadrant qd = w % 4 (rows of that
  // quadrant) and half hf = w / 4 of each block's pages (and of the head
  // dims of O).  Thread state: RPT rows x (2 of every 8 of its head dims).
  // With a single stage the split is one key block (np <= page_slots <= KBP)
  // and O stays in TMEM until the output; otherwise it is folded into
  // registers with the online-softmax rescale (one block late where there
  // are two O buffers).
  constexpr int RPT = C::RPT, OG = DH / 16;  // 8-column groups per half of the head dims
  constexpr bool ONE = NST == 1;
  // Row-wise softmax (the pipelined 128-row variant): thread `lane` of warp
  // w owns query row 32 (w % 4) + lane (its TMEM lane) for half w / 4 of each
  // block's pages and of O's head dims; S comes in with 32x32b loads, so
  // the row's max and sum stay in the thread, P goes back into TMEM and O
  // accumulates there.  o_acc then holds the row's 32 head dims (index j:
  // o_acc[j / 8][j % 8]); m_run[0] and l_run[0] its max and sum.
  constexpr bool ROWT = C::M == 128 && C::PIPE && DH == 64;
  static_assert(!ROWT || (!ONE && RPT * 2 * OG == 32 && RPT >= 3), "a row-wise thread keeps 32 head dims");
  const int qd = warp & 3, hf = warp >> 2;
  const bool soft = warp < 8 && qd < C::QUADS;
  float o_acc[ONE ? 1 : RPT][ONE ? 1 : 2 * OG];
  float m_run[RPT], l_run[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    m_run[i] = -INFINITY;
    l_run[i] = 0.f;
#pragma unroll
    for (int d = 0; d < (ONE ? 1 : 2 * OG); ++d) o_acc[ONE ? 0 : i][d] = 0.f;
  }
  const int c4 = lane & 3, rq = lane >> 2;
  // query row of state row i (i = 2*sb + h: 16-lane block sb, half h) and its TMEM lane block
  auto row_of = [&](int i) { return (C::M == 64 ? 16 * qd : 32 * qd + 16 * (i >> 1)) + rq + 8 * (i & 1); };
  auto lanes_of = [&](int sb) { return static_cast<uint32_t>(C::M == 64 ? 32 * qd : 32 * qd + 16 * sb) << 16; };
  // pair exchange of per-row values between the two warps of a quadrant
  auto pair_combine = [&](float (&v)[RPT], bool is_max) {
#pragma unroll
    for (int i = 0; i < RPT; ++i) s_red[(warp * 32 + lane) * RPT + i] = v[i];
    named_sync(1 + qd, 64);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float o = s_red[(((warp + 4) & 7) * 32 + lane) * RPT + i];
      v[i] = is_max ? fmaxf(v[i], o) : v[i] + o;
    }
    named_sync(1 + qd, 64);  // the slots may be reused
  };

  if (warp == kProducerWarp) {
    // ---------------- TMA producer
    if (lane == 0) {
      const int l_off = p.layer * p.pool_pages;
      bool waited = false;
      auto issue = [&](int blk, bool may_wait) {
        const int s = blk % NST;
        const int pg0 = blk * KBP, npb = min(KBP, np - pg0);
        mbar_arrive_expect_tx(&kv_full[s], 2 * npb * C::NCH * 2048);
        uint8_t* kd = sKV + s * C::STAGE_BYTES;
        uint8_t* vd = kd + C::KV_BYTES;
        for (int j = 0; j < npb; ++j) {
          if (vp_begin + pg0 + j == n_ctx_pages && !waited) {
            // the block page is written by the QKV projection
            if (!may_wait) return false;
            pdl_wait();
            waited = true;
          }
          const int page = s_pages[pg0 + j];
          for (int c = 0; c < C::NCH; ++c) {
            tma_load_4d(kd + c * C::KV_CH + j * 2048, &tmK, &kv_full[s], c * 64, 0, kvh, l_off + page);
            tma_load_4d(vd + c * C::KV_CH + j * 2048, &tmV, &kv_full[s], c * 64, 0, kvh, l_off + page);
          }
        }
        return true;
      };
      int blk = 0;
      // context-only blocks stream while the QKV projection is still running
      for (; blk < nblk && blk < NST; ++blk) {
        const int last_vp = vp_begin + min(np, (blk + 1) * KBP) - 1;
        if (last_vp >= n_ctx_pages) break;
        issue(blk, false);
      }
      pdl_wait();
      waited = true;
      mbar_arrive_expect_tx(q_full, G * C::NCH * 2048);
      for (int g = 0; g < G; ++g)
        for (int c = 0; c < C::NCH; ++c)
          tma_load_2d(sQ + c * C::Q_CH + g * 2048, &tmQ, q_full, (kvh * G + g) * DH + c * 64, b * kBlockK);
      pdl_trigger();
      // HBM is mostly idle from here on: stream the O projection's weights into L2
      if (p.l2.ctas > 0) l2_prefetch_plan(&tmNext, p.l2);
      int issued = blk;
      for (; blk < nblk; ++blk) {
        if (blk >= NST && !mbar_wait(&kv_empty[blk % NST], ((blk / NST) & 1) ^ 1, p.status)) break;
        issue(blk, true);
        issued = blk + 1;
      }
      // every copy this CTA issued must have landed before it exits (bounded)
      for (int i = max(0, issued - NST); i < issued; ++i) mbar_wait(&kv_full[i % NST], (i / NST) & 1, p.status);
      mbar_wait(q_full, 0, p.status);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer.  Serial variants: S(j) (over the columns
    // of O(j - 1), once the softmax has folded it), PV(j) once P(j) is
    // written.  Pipelined: tensor-pipe order S(0), S(1), PV(0), S(2), PV(1),
    // ...; S(j) reuses the buffer of S(j - 2), whose P was waited for before
    // PV(j - 2), and PV(j) the O buffer of PV(j - 2), once the softmax has
    // folded that.  P in TMEM: S(j) reuses the buffer of S(j - 3) once PV(j - 3)
    // is done, and every PV adds into the one O in TMEM, which the softmax
    // rescales there (when it must) before it signals P.
    if (lane == 0) {
      const uint32_t aq = smem_u32(sQ);
      auto issue_s = [&](int j) {
        const int s = j % NST, npb = min(KBP, np - j * KBP);
        if (!mbar_wait(&kv_full[s], (j / NST) & 1, p.status)) return false;
        if (!C::PIPE && !C::SEPO && j > 0 && !mbar_wait(&o_free[0], (j - 1) & 1, p.status)) return false;
        // with P in TMEM, S(j) overwrites P(j - 3): MMAs into different
        // accumulators are not ordered, so wait for the P V product of j - 3
        // (its commit to o_full; only this thread advances that barrier, and
        // PV(j - 1), the next commit there, is issued after this)
        if (C::P_TMEM && j >= C::NSB &&
            !mbar_wait(&o_full[(j - C::NSB) % C::NO], ((j - C::NSB) / C::NO) & 1, p.status))
          return false;
        tc_fence_after();
        const uint32_t ak = smem_u32(sKV + s * C::STAGE_BYTES);
        const uint32_t id_s = mma_idesc_f16_f32(C::M, 16 * npb, false);
#pragma unroll
        for (int ks = 0; ks < DH / 16; ++ks) {
          const uint32_t off = (ks & 3) * 32;
          tc_mma_bf16(tmem + C::s_col(j % C::NSB), sw128_desc(aq + (ks >> 2) * C::Q_CH + off, 16, 1024),
                      sw128_desc(ak + (ks >> 2) * C::KV_CH + off, 16, 1024), id_s, ks > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[j % C::NSB]);
        return true;
      };
      bool ok = nblk == 0 || (mbar_wait(q_full, 0, p.status) && issue_s(0));
      for (int blk = 0; ok && blk < nblk; ++blk) {
        if (C::PIPE && blk + 1 < nblk && !issue_s(blk + 1)) break;
        const int s = blk % NST, npb = min(KBP, np - blk * KBP), ob = blk % C::NO;
        if (!mbar_wait(&p_full[blk % C::NSB], (blk / C::NSB) & 1, p.status)) break;
        if (C::PIPE && !C::P_TMEM && blk >= 2 && !mbar_wait(&o_free[ob], ((blk - 2) / 2) & 1, p.status)) break;
        tc_fence_after();
        const uint32_t ak = smem_u32(sKV + s * C::STAGE_BYTES);
        const uint32_t av = ak + C::KV_BYTES;
        const uint32_t ap = C::P_IN_K ? ak : smem_u32(sP + C::p_off(blk));
        const uint32_t id_o = mma_idesc_f16_f32(C::M, DH, true);
        if constexpr (C::P_TMEM) {
          // A = P from TMEM: page k16's 16 keys in the first 8 columns of its
          // S columns; O accumulates over the blocks in one TMEM buffer
          for (int k16 = 0; k16 < npb; ++k16)
            tc_mma_bf16_ts(tmem + C::o_col(0), tmem + C::s_col(blk % C::NSB) + 16 * k16,
                           sw128_desc(av + k16 * 2048, C::KV_CH, 1024), id_o, (blk | k16) > 0 ? 1u : 0u);
        } else {
          for (int k16 = 0; k16 < npb; ++k16)
            tc_mma_bf16(tmem + C::o_col(ob), sw128_desc(ap + (k16 >> 2) * C::P_CH + (k16 & 3) * 32, 16, 1024),
                        sw128_desc(av + k16 * 2048, C::KV_CH, 1024), id_o, (C::SEPO ? (blk | k16) : k16) > 0 ? 1u : 0u);
        }
        tc_commit(&o_full[ob]);
        tc_commit(&kv_empty[s]);
        if (!C::PIPE && blk + 1 < nblk && !issue_s(blk + 1)) break;
      }
    }
    __syncwarp();
  } else if (soft && ROWT) {
    // ---------------- row-wise softmax (see ROWT).  The two warps of a
    // quadrant meet at named barriers, so both always run every block.
    bool live = true;
    const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
    const uint32_t o_half = tmem + lane_base + C::o_col(0) + 32 * hf;  // this warp's 32 head dims of O
    float m_r = -INFINITY, l_r = 0.f;
    // O accumulates in TMEM (the P V products add up); m_r is the max P is
    // taken against, and it moves only when the row's max passes it by more
    // than kLazyRescale (log2 units), so P stays at most 2^kLazyRescale and
    // O is rescaled, in TMEM, only then (once P V of the previous block is done)
    auto rescale_o = [&](int blk, float al) {
      live = live && mbar_wait(&o_full[(blk - 1) % C::NO], ((blk - 1) / C::NO) & 1, p.status);
      __syncwarp();
      tc_fence_after();
      uint32_t v0[16], v1[16];
      tc_ld_32x32b_x16_nw(o_half, v0);
      tc_ld_32x32b_x16_nw(o_half + 16, v1);
      tc_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        v0[j] = __float_as_uint(__uint_as_float(v0[j]) * al);
        v1[j] = __float_as_uint(__uint_as_float(v1[j]) * al);
      }
      tc_st_32x32b_x16(o_half, v0);
      tc_st_32x32b_x16(o_half + 16, v1);
    };
    for (int blk = 0; blk < nblk; ++blk) {
      const int npb = min(KBP, np - blk * KBP);
      const int vp0 = vp_begin + blk * KBP;
      const int pg_split = (npb + 1) >> 1;
      const int pg_lo = hf == 0 ? 0 : pg_split, pg_hi = hf == 0 ? pg_split : npb;
      constexpr int HP = (KBP + 1) / 2;
      live = live && mbar_wait(&s_full[blk % C::NSB], (blk / C::NSB) & 1, p.status);
      __syncwarp();
      tc_fence_after();
      uint32_t sv[HP][16];
#pragma unroll
      for (int j = 0; j < HP; ++j)
        if (pg_lo + j < pg_hi) tc_ld_32x32b_x16_nw(tmem + lane_base + C::s_col(blk % C::NSB) + (pg_lo + j) * 16, sv[j]);
      tc_wait_ld();
      // P = 2^(S scale - m_r) in fp16 into TMEM, a page's 16 keys as 8
      // packed columns over the start of that page's own S columns (this
      // thread read them above; S of this buffer is recomputed only after
      // the P V product that reads P), the row sum as packed fp32 pairs;
      // with_max: the valid keys' max as well (only the last context page is
      // partial)
      float2 ls2;
      auto make_p = [&](bool with_max, float& mx) {
        ls2 = make_float2(0.f, 0.f);
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), mneg2 = make_float2(-m_r, -m_r);
#pragma unroll
        for (int j = 0; j < HP; ++j) {
          const int pg = pg_lo + j;
          if (pg >= pg_hi) break;
          const int vp = vp0 + pg;
          const int nvalid = vp < n_ctx_pages ? min(kPage, T - vp * kPage) : kPage;
          uint32_t pk[8];
          if (nvalid == kPage) {  // (no key mask)
            if (with_max) {
              float a = fmax3(__uint_as_float(sv[j][0]), __uint_as_float(sv[j][1]), __uint_as_float(sv[j][2]));
              float c = fmax3(__uint_as_float(sv[j][3]), __uint_as_float(sv[j][4]), __uint_as_float(sv[j][5]));
#pragma unroll
              for (int k = 6; k < 14; k += 4) {
                a = fmax3(a, __uint_as_float(sv[j][k]), __uint_as_float(sv[j][k + 1]));
                c = fmax3(c, __uint_as_float(sv[j][k + 2]), __uint_as_float(sv[j][k + 3]));
              }
              a = fmax3(a, __uint_as_float(sv[j][14]), __uint_as_float(sv[j][15]));
              mx = fmax3(mx, a, c);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float2 t = __ffma2_rn(
                  make_float2(__uint_as_float(sv[j][2 * k]), __uint_as_float(sv[j][2 * k + 1])), sc2, mneg2);
              const float e0 = ex2_ftz(t.x), e1 = ex2_ftz(t.y);
              ls2 = __fadd2_rn(ls2, make_float2(e0, e1));
              pk[k] = pack_half2(e0, e1);
            }
          } else {
            if (with_max) {
#pragma unroll
              for (int k = 0; k < 16; ++k)
                if (k < nvalid) mx = fmaxf(mx, __uint_as_float(sv[j][k]));
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float2 t = __ffma2_rn(
                  make_float2(__uint_as_float(sv[j][2 * k]), __uint_as_float(sv[j][2 * k + 1])), sc2, mneg2);
              const float e0 = 2 * k < nvalid ? ex2_ftz(t.x) : 0.f, e1 = 2 * k + 1 < nvalid ? ex2_ftz(t.y) : 0.f;
              ls2 = __fadd2_rn(ls2, make_float2(e0, e1));
              pk[k] = pack_half2(e0, e1);
            }
          }
          tc_st_32x32b_x8(tmem + lane_base + C::s_col(blk % C::NSB) + 16 * pg, pk);
        }
      };
      // the row's max over this half's keys, then over both halves (the
      // partner warp holds the row's other pages).  One barrier: the slot
      // alternates by block, and a slot is written again only after the
      // next block's barrier, which the partner passes after its read.
      auto pair_max = [&](float mx) {
        s_red[(warp * 32 + lane) * RPT + (blk & 1)] = mx;
        named_sync(1 + qd, 64);
        return fmaxf(mx, s_red[(((warp + 4) & 7) * 32 + lane) * RPT + (blk & 1)]);
      };
      float mx = -INFINITY, alpha;
      bool move;
      if (m_r == -INFINITY) {
        // the first block (every row at once): the max first, then P
#pragma unroll
        for (int j = 0; j < HP; ++j) {
          const int pg = pg_lo + j;
          if (pg >= pg_hi) break;
          const int vp = vp0 + pg;
          const int nvalid = vp < n_ctx_pages ? min(kPage, T - vp * kPage) : kPage;
#pragma unroll
          for (int k = 0; k < 16; ++k)
            if (k < nvalid) mx = fmaxf(mx, __uint_as_float(sv[j][k]));
        }
        m_r = pair_max(mx) * p.scale_log2;
        alpha = 0.f;
        move = true;
        make_p(false, mx);
      } else {
        // P against the current m_r while the block's max is taken; only if
        // a row's max passes m_r by more than kLazyRescale is m_r moved and
        // P taken again (the S values are still in registers)
        make_p(true, mx);
        const float m_cand = pair_max(mx) * p.scale_log2;
        move = m_cand > m_r + kLazyRescale;
        alpha = move ? ex2_ftz(m_r - m_cand) : 1.f;
        if (__any_sync(0xffffffffu, move)) {
          if (move) m_r = m_cand;
          float unused = -INFINITY;
          tc_wait_st();  // the first P stores have landed before they are overwritten
          make_p(false, unused);
          rescale_o(blk, alpha);
        }
      }
      l_r = l_r * alpha + (ls2.x + ls2.y);
      tc_wait_st();  // P (and a rescaled O) is in TMEM before the MMA thread hears of it
      tc_fence_before();
      mbarrier_arrive_one(&p_full[blk % C::NSB]);
    }
    if (nblk > 0) {
      // O of every block, once the last P V product is done
      live = live && mbar_wait(&o_full[(nblk - 1) % C::NO], ((nblk - 1) / C::NO) & 1, p.status);
      __syncwarp();
      tc_fence_after();
      uint32_t v0[16], v1[16];
      tc_ld_32x32b_x16_nw(o_half, v0);
      tc_ld_32x32b_x16_nw(o_half + 16, v1);
      tc_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) o_acc[j >> 3][j & 7] = __uint_as_float(j < 16 ? v0[j] : v1[j - 16]);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) o_acc[j >> 3][j & 7] = 0.f;
    }
    // the row's full sum: this half's plus the partner's (slot 2: the
    // block slots may still be read)
    s_red[(warp * 32 + lane) * RPT + 2] = l_r;
    named_sync(1 + qd, 64);
    l_r += s_red[(((warp + 4) & 7) * 32 + lane) * RPT + 2];
    m_run[0] = m_r;
    l_run[0] = l_r;
  } else if (soft) {
    // ---------------- softmax.  The two warps of a quadrant meet at named
    // barriers, so both always run every block: a wait that gives up only
    // marks the work as failed (status word) and later waits are skipped.
    bool live = true;
    // O of block f into the registers.  One O buffer: o = o al + O_f with
    // the rescale al of block f.  Two: O_f is folded one block late, after
    // the next block's rescale al is known, as o = (o + O_f) al (o then
    // refers to that block's running max); the last block adds O_f alone.
    auto fold = [&](int f, const float (&al)[RPT], bool last) {
      const int ob = f % C::NO;
      live = live && mbar_wait(&o_full[ob], (f / C::NO) & 1, p.status);
      __syncwarp();
      tc_fence_after();
      // this warp's half of the head dims
#pragma unroll
      for (int sb = 0; sb < C::SUB; ++sb) {
#pragma unroll
        for (int d0 = 0; d0 < DH / 2; d0 += 32) {
          uint32_t v[16];
          tc_ld_16x256b_x4(tmem + lanes_of(sb) + C::o_col(ob) + hf * (DH / 2) + d0, v);
          tc_wait_ld();
#pragma unroll
          for (int gq = 0; gq < 4; ++gq)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int i = 2 * sb + h, d = 2 * (d0 / 8 + gq) + e;
                float& o = o_acc[ONE ? 0 : i][ONE ? 0 : d];
                const float x = __uint_as_float(v[4 * gq + 2 * h + e]);
                o = last ? o + x : C::NO == 1 ? o * al[i] + x : (o + x) * al[i];
              }
        }
      }
      tc_fence_before();
      mbarrier_arrive_one(&o_free[ob]);
    };
    for (int blk = 0; blk < nblk; ++blk) {
      const int npb = min(KBP, np - blk * KBP);
      const int vp0 = vp_begin + blk * KBP;
      // this warp's pages of the block: [pg_lo, pg_hi)
      const int pg_split = (npb + 1) >> 1;
      const int pg_lo = hf == 0 ? 0 : pg_split, pg_hi = hf == 0 ? pg_split : npb;
      live = live && mbar_wait(&s_full[blk % C::NSB], (blk / C::NSB) & 1, p.status);
      __syncwarp();
      tc_fence_after();
      constexpr int HP = (KBP + 1) / 2;  // pages per warp at most
      float alpha[RPT], lsum[RPT], mx[RPT];
#pragma unroll
      for (int i = 0; i < RPT; ++i) mx[i] = -INFINITY;
      uint32_t sv[C::SUB][HP][8];
      // S columns of this warp's pages in registers (one wait)
#pragma unroll
      for (int sb = 0; sb < C::SUB; ++sb)
#pragma unroll
        for (int j = 0; j < HP; ++j)
          if (pg_lo + j < pg_hi)
            tc_ld_16x256b_x2(tmem + lanes_of(sb) + C::s_col(blk % C::NSB) + (pg_lo + j) * 16, sv[sb][j]);
      tc_wait_ld();
      // pass 1: row max over the valid keys (a full page needs no mask:
      // only the sequence's last context page is partial)
#pragma unroll
      for (int j = 0; j < HP; ++j) {
        const int pg = pg_lo + j;
        if (pg >= pg_hi) break;
        const int vp = vp0 + pg;
        const int nvalid = vp < n_ctx_pages ? min(kPage, T - vp * kPage) : kPage;
        if (nvalid == kPage) {
#pragma unroll
          for (int sb = 0; sb < C::SUB; ++sb) {
            const uint32_t* w = sv[sb][j];
            mx[2 * sb] = fmaxf(mx[2 * sb], fmaxf(fmaxf(__uint_as_float(w[0]), __uint_as_float(w[1])),
                                                 fmaxf(__uint_as_float(w[4]), __uint_as_float(w[5]))));
            mx[2 * sb + 1] = fmaxf(mx[2 * sb + 1], fmaxf(fmaxf(__uint_as_float(w[2]), __uint_as_float(w[3])),
                                                         fmaxf(__uint_as_float(w[6]), __uint_as_float(w[7]))));
          }
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) {  // keys 2c4, 2c4+1, 8+2c4, 9+2c4
            const int key = (q >> 1) * 8 + 2 * c4 + (q & 1);
            if (key < nvalid)
#pragma unroll
              for (int sb = 0; sb < C::SUB; ++sb) {
                mx[2 * sb] = fmaxf(mx[2 * sb], __uint_as_float(sv[sb][j][(q >> 1) * 4 + (q & 1)]));
                mx[2 * sb + 1] = fmaxf(mx[2 * sb + 1], __uint_as_float(sv[sb][j][(q >> 1) * 4 + 2 + (q & 1)]));
              }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
        mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
      }
      pair_combine(mx, true);
      float m_new[RPT];
      bool moved = false;
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        if constexpr (C::SEPO) {
          // O accumulates in TMEM: m_run moves only when passed by more than
          // kLazyRescale, and O is rescaled in TMEM then (below)
          const float mc = mx[i] * p.scale_log2;
          const bool mv = mc > m_run[i] + kLazyRescale;
          alpha[i] = !mv ? 1.f : m_run[i] == -INFINITY ? 0.f : ex2_ftz(m_run[i] - mc);
          if (mv) m_run[i] = mc;
          moved = moved || mv;
          m_new[i] = m_run[i];
        } else {
          m_new[i] = fmaxf(m_run[i], mx[i] * p.scale_log2);
          alpha[i] = m_run[i] == -INFINITY ? 0.f : ex2_ftz(m_run[i] - m_new[i]);
          m_run[i] = m_new[i];
        }
        lsum[i] = 0.f;
      }
      // pass 2: P = 2^(S scale - m) in fp16 into the swizzled A operand
      uint8_t* pbase = C::P_IN_K ? sKV + (blk % NST) * C::STAGE_BYTES : sP + C::p_off(blk);
#pragma unroll
      for (int j = 0; j < HP; ++j) {
        const int pg = pg_lo + j;
        if (pg >= pg_hi) break;
        const int vp = vp0 + pg;
        const int nvalid = vp < n_ctx_pages ? min(kPage, T - vp * kPage) : kPage;
        uint8_t* pch = pbase + (pg >> 2) * C::P_CH;
        const int u0 = 2 * (pg & 3);
        const bool full = nvalid == kPage;
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
          const int sb = i >> 1, h = i & 1;
          const float mneg = -m_new[i];
          float e[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int key = (q >> 1) * 8 + 2 * c4 + (q & 1);
            const float x = ex2_ftz(fmaf(__uint_as_float(sv[sb][j][(q >> 1) * 4 + 2 * h + (q & 1)]), p.scale_log2, mneg));
            e[q] = full || key < nvalid ? x : 0.f;
          }
          lsum[i] += (e[0] + e[1]) + (e[2] + e[3]);
          const int r = row_of(i);
          if (r < R) {
            // keys 2*c4, 2*c4+1 of the page's first / second 8-key unit
            // (16-byte units u0 and u0 + 1 of the 128-byte row, swizzled)
            uint8_t* prow = pch + r * 128 + 4 * c4;
            const int sw = (u0 ^ (r & 7)) << 4;
            *reinterpret_cast<uint32_t*>(prow + sw) = pack_half2(e[0], e[1]);
            *reinterpret_cast<uint32_t*>(prow + (sw ^ 16)) = pack_half2(e[2], e[3]);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < RPT; ++i) l_run[i] = l_run[i] * alpha[i] + lsum[i];
      if constexpr (C::SEPO) {
        // a row's max moved: O (this warp's half of the head dims) times
        // alpha, in TMEM.  P V of the previous block is done (S of this
        // block, whose completion this thread waited for, was issued after
        // it) and P V of this block waits for p_full.
        if (blk > 0 && __any_sync(0xffffffffu, moved)) {
#pragma unroll
          for (int sb = 0; sb < C::SUB; ++sb)
#pragma unroll
            for (int d0 = 0; d0 < DH / 2; d0 += 32) {
              const uint32_t ta = tmem + lanes_of(sb) + C::o_col(0) + hf * (DH / 2) + d0;
              uint32_t v[16];
              tc_ld_16x256b_x4(ta, v);
              tc_wait_ld();
#pragma unroll
              for (int gq = 0; gq < 4; ++gq)
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                  for (int e = 0; e < 2; ++e)
                    v[4 * gq + 2 * h + e] = __float_as_uint(__uint_as_float(v[4 * gq + 2 * h + e]) * alpha[2 * sb + h]);
              tc_st_16x256b_x4(ta, v);
            }
          tc_wait_st();
        }
      }
      fence_proxy_async_smem();  // P is read by the tensor cores
      tc_fence_before();
      mbarrier_arrive_one(&p_full[blk % C::NSB]);
      if constexpr (ONE) {
        // O stays in TMEM (a single block: both warps leave here)
        live = live && mbar_wait(&o_full[0], 0, p.status);
        __syncwarp();
        tc_fence_after();
        break;
      } else if constexpr (C::SEPO) {
        // (O stays in TMEM until the last block)
      } else if constexpr (C::NO == 1) {
        fold(blk, alpha, false);
      } else if (blk > 0) {
        // O of the previous block: its P V product ran while this block's P was formed
        fold(blk - 1, alpha, false);
      }
    }
    if constexpr (!ONE && (C::NO == 2 || C::SEPO)) {
      // the last O into the registers (SEPO: all blocks' O, accumulated in
      // TMEM; the wait is for P V of the last block)
      if (nblk > 0) fold(nblk - 1, l_run, true);  // (no rescale: al unused)
    }
    // full row sums: over the 4 threads of each row, then the warp pair
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 1);
      l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 2);
    }
    pair_combine(l_run, false);
  }

  // ---------------- output
  const int Hq = p.Hkv * G, q_dim = Hq * DH;
  ActOut<__nv_bfloat16> out{static_cast<__nv_bfloat16*>(p.o_hi), static_cast<__nv_bfloat16*>(p.o_lo)};
  // visits this thread's unnormalised O values: f(state row i, head dim d, o[d], o[d + 1])
  auto for_each_o = [&](auto&& f) {
    if constexpr (ONE) {
      const bool have = nblk > 0;  // with no keys O was never written (its l is 0)
#pragma unroll
      for (int sb = 0; sb < C::SUB; ++sb)
#pragma unroll
        for (int d0 = 0; d0 < DH / 2; d0 += 32) {
          uint32_t v[16];
          tc_ld_16x256b_x4(tmem + lanes_of(sb) + hf * (DH / 2) + d0, v);
          tc_wait_ld();
#pragma unroll
          for (int gq = 0; gq < 4; ++gq)
#pragma unroll
            for (int h = 0; h < 2; ++h)
              f(2 * sb + h, hf * (DH / 2) + d0 + 8 * gq + 2 * c4, have ? __uint_as_float(v[4 * gq + 2 * h]) : 0.f,
                have ? __uint_as_float(v[4 * gq + 2 * h + 1]) : 0.f);
        }
    } else {
#pragma unroll
      for (int i = 0; i < RPT; ++i)
#pragma unroll
        for (int j = 0; j < OG; ++j) f(i, hf * (DH / 2) + 8 * j + 2 * c4, o_acc[i][2 * j], o_acc[i][2 * j + 1]);
    }
  };
  if (p.splits == 1) {
    if (soft && ROWT) {
      // the row's 32 head dims of this half, 16-byte stores of both terms
      const int r = 32 * qd + lane;
      const float inv = l_run[0] > 0.f ? 1.f / l_run[0] : 0.f;
      const long long at = static_cast<long long>(b * kBlockK + (r & 15)) * q_dim + (kvh * G + (r >> 4)) * DH + 32 * hf;
#pragma unroll
      for (int j0 = 0; j0 < 32; j0 += 8) {
        uint32_t hv[4], lv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int j = j0 + 2 * k;
          const float v0 = o_acc[j >> 3][j & 7] * inv, v1 = o_acc[(j + 1) >> 3][(j + 1) & 7] * inv;
          const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
          const __nv_bfloat162 l = __floats2bfloat162_rn(v0 - __low2float(h), v1 - __high2float(h));
          hv[k] = *reinterpret_cast<const uint32_t*>(&h);
          lv[k] = *reinterpret_cast<const uint32_t*>(&l);
        }
        *reinterpret_cast<uint4*>(out.hi + at + j0) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        *reinterpret_cast<uint4*>(out.lo + at + j0) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
      }
    } else if (soft) {
      for_each_o([&](int i, int d, float o0, float o1) {
        const int r = row_of(i);
        if (r >= R) return;
        const float inv = l_run[i] > 0.f ? 1.f / l_run[i] : 0.f;
        const long long at = static_cast<long long>(b * kBlockK + (r & 15)) * q_dim + (kvh * G + (r >> 4)) * DH + d;
        const float v0 = o0 * inv, v1 = o1 * inv;
        const __nv_bfloat162 hv = __floats2bfloat162_rn(v0, v1);
        const __nv_bfloat162 lv = __floats2bfloat162_rn(v0 - __low2float(hv), v1 - __high2float(hv));
        *reinterpret_cast<__nv_bfloat162*>(out.hi + at) = hv;
        *reinterpret_cast<__nv_bfloat162*>(out.lo + at) = lv;
      });
    }
  } else {
    // Split merge inside the cluster.  Each split stages its unnormalised
    // rows (o, m, l) in row order; once every CTA is past its main loop
    // (cluster barrier), one thread copies the rows owned by cluster rank k
    // (rows k*rpr ..) into slot [split] of k's receive area with a bulk
    // shared-memory copy that completes on k's mbarrier; each CTA then
    // merges its rows from local memory in split order.  A final cluster
    // barrier keeps every CTA (and so every copy source) alive until all
    // copies have landed.
    const int S = p.splits, cr = static_cast<int>(cluster_ctarank());
    const int rpr = (R + S - 1) / S;
    constexpr int LD = DH + 4;  // floats per row: o, m, l, pad (16-byte multiple)
    float* stage = reinterpret_cast<float*>(smem);          // [R][LD] (Q, P and the ring are idle now)
    float* recv = stage + R * LD;                           // [S][rpr][LD]
    const int r0 = min(R, cr * rpr), r1 = min(R, r0 + rpr);
    __syncthreads();
    if (soft && ROWT) {
      const int r = 32 * qd + lane;
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4*>(stage + r * LD + 32 * hf + j) =
            make_float4(o_acc[j >> 3][j & 7], o_acc[(j + 1) >> 3][(j + 1) & 7], o_acc[(j + 2) >> 3][(j + 2) & 7],
                        o_acc[(j + 3) >> 3][(j + 3) & 7]);
      if (hf == 0) *reinterpret_cast<float2*>(stage + r * LD + DH) = make_float2(m_run[0], l_run[0]);
    } else if (soft) {
      for_each_o([&](int i, int d, float o0, float o1) {
        const int r = row_of(i);
        if (r < R) *reinterpret_cast<float2*>(stage + r * LD + d) = make_float2(o0, o1);
      });
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const int r = row_of(i);
        if (r < R && c4 == 0 && hf == 0) *reinterpret_cast<float2*>(stage + r * LD + DH) = make_float2(m_run[i], l_run[i]);
      }
    }
    if (threadIdx.x == 0) mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>(S * (r1 - r0) * LD * 4));
    fence_proxy_async_smem();
    __syncthreads();
    // every receive area is idle (a receive count may follow the bytes it counts)
    cluster_arrive_relaxed();
    cluster_wait();
    if (threadIdx.x == 0) {
      for (int k = 0; k < S; ++k) {
        const int k0 = min(R, k * rpr), k1 = min(R, k0 + rpr);
        if (k1 > k0)
          bulk_copy_smem_to_rank(smem_u32(recv + cr * rpr * LD), smem_u32(stage + k0 * LD),
                            static_cast<uint32_t>((k1 - k0) * LD * 4), recv_bar, static_cast<uint32_t>(k));
      }
    }
    mbar_wait(recv_bar, 0, p.status);
    cluster_arrive_relaxed();  // my incoming copies have landed
    for (int e = threadIdx.x; e < (r1 - r0) * (DH / 4); e += blockDim.x) {
      const int j = e / (DH / 4), d4 = (e % (DH / 4)) * 4, r = r0 + j;
      float M = -INFINITY;
      for (int s2 = 0; s2 < S; ++s2) M = fmaxf(M, recv[(s2 * rpr + j) * LD + DH]);
      float den = 0.f;
      float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s2 = 0; s2 < S; ++s2) {
        const float* row = recv + (s2 * rpr + j) * LD;
        const float ms = row[DH];
        if (ms == -INFINITY) continue;
        const float w = exp2f(ms - M);
        const float4 o4 = *reinterpret_cast<const float4*>(row + d4);
        den += w * row[DH + 1];
        num.x += w * o4.x;
        num.y += w * o4.y;
        num.z += w * o4.z;
        num.w += w * o4.w;
      }
      const float inv = den > 0.f ? 1.f / den : 0.f;
      const long long base = static_cast<long long>(b * kBlockK + (r & 15)) * q_dim + (kvh * G + (r >> 4)) * DH + d4;
      out.put(base + 0, num.x * inv);
      out.put(base + 1, num.y * inv);
      out.put(base + 2, num.z * inv);
      out.put(base + 3, num.w * inv);
    }
    cluster_wait();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_mma() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// The fp16 pool [L*pool_pages][Hkv][16][dh] as a 4-D map with 16 x 64 boxes.
bool pool_map4(const void* base, int dh, int Hkv, long long pages_total, CUtensorMap* out) {
  auto fn = encode_fn_mma();
  if (fn == nullptr) return false;
  cuuint64_t gdim[4] = {static_cast<cuuint64_t>(dh), 16, static_cast<cuuint64_t>(Hkv),
                        static_cast<cuuint64_t>(pages_total)};
  cuuint64_t gstride[3] = {static_cast<cuuint64_t>(dh) * 2, static_cast<cuuint64_t>(dh) * 2 * 16,
                           static_cast<cuuint64_t>(dh) * 2 * 16 * Hkv};
  cuuint32_t box[4] = {64, 16, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(out, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(base), gdim, gstride, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The block queries q [rows][Hq*dh] (fp16) as a 2-D map with 16-row x 64-column boxes.
bool q_map(const void* base, int rows, int cols, CUtensorMap* out) {
  auto fn = encode_fn_mma();
  if (fn == nullptr) return false;
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, 16};
  cuuint32_t es[2] = {1, 1};
  return fn(out, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), gdim, gstride, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Shared memory of a launch: the layout plus the page ids, raised where
// needed so that the CTAs one SM can hold never ask for more than its 512
// TMEM columns.  (An allocation that does not fit waits for another CTA on
// the SM to free its columns; if that CTA belonged to the same cluster and
// waited at the split merge, neither would finish.)
template <int DH, int G, int KBP, int NST>
int smem_bytes(int page_slots) {
  using C = MmaAttnCfg<DH, G, KBP, NST>;
  static int sm_smem = -1, reserved = 0;
  if (sm_smem < 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) {
      cudaGetLastError();
      sm_smem = 233472;  // 228 KB, the sm_100 family's figure
      reserved = 1024;
    }
  }
  constexpr int per_sm = 512 / C::TMEM_COLS;  // CTAs whose allocations fit at once
  const int floor = sm_smem / (per_sm + 1) - reserved + 128;  // (per_sm + 1) CTAs exceed the SM
  return std::max(C::SMEM_FIXED + 4 * page_slots, (floor + 127) & ~127);
}

template <int DH, int G, int KBP, int NST>
cudaError_t set_attrs(int smem) {
  static FuncAttr cluster_attr, smem_attr;
  cudaError_t e = cluster_attr.ensure(1, [](int v) {
    return cudaFuncSetAttribute(k_attn_mma<DH, G, KBP, NST>, cudaFuncAttributeNonPortableClusterSizeAllowed, v);
  });
  if (e != cudaSuccess) return e;
  return smem_attr.ensure(smem, [](int v) {
    return cudaFuncSetAttribute(k_attn_mma<DH, G, KBP, NST>, cudaFuncAttributeMaxDynamicSharedMemorySize, v);
  });
}

// Pages one split can hold at most (the split's share of the longest
// sequence plus its block page).
int split_pages_bound(const dflash_ctx* c, int splits) {
  return (c->cfg.max_pages_per_seq + 1 + splits - 1) / splits;
}

template <int DH, int G, int KBP, int NST>
cudaError_t launch_t(dflash_ctx* c, int layer, int B, int splits, cudaStream_t s, const NextGemm& next,
                     const AttnSrc& src) {
  const auto& g = c->cfg;
  const int page_slots = split_pages_bound(c, splits);
  const int smem = smem_bytes<DH, G, KBP, NST>(page_slots);
  cudaError_t e = set_attrs<DH, G, KBP, NST>(smem);
  if (e != cudaSuccess) return e;
  if (!c->attn_maps_ready) {
    const long long pages_total = static_cast<long long>(g.n_layers) * c->pool_pages;
    if (!pool_map4(c->pool_k, DH, g.n_kv_heads, pages_total, &c->attn_map_k) ||
        !pool_map4(c->pool_v, DH, g.n_kv_heads, pages_total, &c->attn_map_v) ||
        !q_map(c->q, g.max_batch * kBlockK, g.n_q_heads * DH, &c->attn_map_q))
      return cudaErrorInvalidValue;
    c->attn_maps_ready = true;
  }
  MmaAttnParams p;
  p.page_table = c->page_table;
  p.seq_len = src.seq_len != nullptr ? src.seq_len : c->seq_len;
  p.row_of = src.row_of;
  p.order = src.order;
  p.max_pages = g.max_pages_per_seq;
  p.block_page0 = g.n_pages;
  p.pool_pages = c->pool_pages;
  p.layer = layer;
  p.Hkv = g.n_kv_heads;
  p.splits = splits;
  p.page_slots = page_slots;
  p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(DH));
  p.o_hi = c->o;
  p.o_lo = c->o_lo;
  p.status = c->status;
  CUtensorMap tn = c->attn_map_k;  // placeholder when there is no plan
  if (!gemm_l2_plan(c, next, &p.l2, &tn)) p.l2 = L2Plan{};
  return launch_k(k_attn_mma<DH, G, KBP, NST>, dim3(splits, g.n_kv_heads, B), dim3(kAttnThreads), smem, s,
                  dim3(splits, 1, 1), c->pdl && src.pdl, c->attn_map_q, c->attn_map_k, c->attn_map_v, tn, p);
}

// How many clusters of `splits` CTAs of this kernel instance can be
// resident at once (0 if unknown).
template <int DH, int G, int KBP, int NST>
int max_clusters_t(dflash_ctx* c, int splits) {
  const int smem = smem_bytes<DH, G, KBP, NST>(split_pages_bound(c, splits));
  if (set_attrs<DH, G, KBP, NST>(smem) != cudaSuccess ||
      !prefer_max_smem(reinterpret_cast<const void*>(k_attn_mma<DH, G, KBP, NST>))) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(splits, 1, 1);
  lc.blockDim = dim3(kAttnThreads);
  lc.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = splits;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_attn_mma<DH, G, KBP, NST>, &lc) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// Short splits (at most 13 pages): all keys in one block, no ring, and (for
// up to 64 query rows of dh 128) a CTA of at most 124 KB, small enough to
// share an SM with a 102 KB projection CTA (so the context streams in while
// the QKV projection runs); longer splits stream 8-page blocks through a
// 2-deep ring.
constexpr int kShortPages = 13;

// The streaming variant with 4-page key blocks: half the shared memory and
// at most 102 registers a thread, so two CTAs share an SM.  It serves grids
// with more (sequence, kv head) problems than SMs (the serving batches, the
// training-time block attention), where each CTA streams a long prefix and
// twice the CTAs an SM hide its latency chain; with few problems and long
// contexts (c4) the 8-page ring streams faster.  It exists where its layout
// fits, and serves the split counts whose merge fits its smaller ring.
template <int DH, int G>
constexpr bool narrow_fits() {
  // (128 query rows of 128 dims do not fit 102 registers a thread)
  using L = MmaAttnLayout<DH, G, 4, 2>;
  return DH * G <= 512 && L::q_padding_inside && L::p_padding_inside;
}

// Ring depth of the 4-page variant: three stages where it is pipelined and
// two CTAs still share an SM with room for the page ids (on 128 sequences of
// 1-8k keys, dh 64, it measured the same as two stages: the loads are not
// what the softmax waits for), two otherwise.
template <int DH, int G>
constexpr int narrow_stages() {
  using L3 = MmaAttnLayout<DH, G, 4, 3>;
  using L5 = MmaAttnLayout<DH, G, 4, 5>;
  // with P in TMEM the shared memory of the P buffers holds two more stages
  if constexpr (L5::P_TMEM && L5::q_padding_inside && L5::SMEM_FIXED <= 104 * 1024) return 5;
  return L3::PIPE && L3::q_padding_inside && L3::p_padding_inside && L3::SMEM_FIXED <= 104 * 1024 ? 3 : 2;
}

template <int DH, int G>
int narrow_max_merge() {
  if constexpr (narrow_fits<DH, G>()) return MmaAttnCfg<DH, G, 4, narrow_stages<DH, G>()>::MAX_MERGE;
  else return 0;
}

// Runs F<DH, G, KBP, NST>(args) for the kernel instance serving `splits`.
template <template <int, int, int, int> class F, typename... A>
auto dispatch(dflash_ctx* c, int splits, bool narrow, A... args) {
  const bool short_split = split_pages_bound(c, splits) <= kShortPages;
  const int G = c->cfg.n_q_heads / c->cfg.n_kv_heads;
#define DFLASH_ATTN_CASE(DH_, G_)                                                              \
  if (c->cfg.head_dim == DH_ && G == G_)                                                       \
    return short_split ? F<DH_, G_, kShortPages, 1>::run(c, splits, args...)                   \
           : narrow && splits <= narrow_max_merge<DH_, G_>()                                   \
               ? F<DH_, G_, narrow_fits<DH_, G_>() ? 4 : 8,                                    \
                   narrow_fits<DH_, G_>() ? narrow_stages<DH_, G_>() : 2>::run(c, splits, args...)  \
               : F<DH_, G_, 8, 2>::run(c, splits, args...);
  DFLASH_ATTN_CASE(64, 1) DFLASH_ATTN_CASE(64, 2) DFLASH_ATTN_CASE(64, 4) DFLASH_ATTN_CASE(64, 8)
  DFLASH_ATTN_CASE(128, 1) DFLASH_ATTN_CASE(128, 2) DFLASH_ATTN_CASE(128, 4) DFLASH_ATTN_CASE(128, 8)
#undef DFLASH_ATTN_CASE
  return F<64, 1, 8, 2>::invalid();
}

template <int DH, int G, int KBP, int NST>
struct LaunchF {
  static cudaError_t run(dflash_ctx* c, int splits, int layer, int B, cudaStream_t s, const NextGemm* next,
                         const AttnSrc* src) {
    return launch_t<DH, G, KBP, NST>(c, layer, B, splits, s, *next, *src);
  }
  static cudaError_t invalid() { return cudaErrorInvalidValue; }
};

template <int DH, int G, int KBP, int NST>
struct ClustersF {
  static int run(dflash_ctx* c, int splits) { return max_clusters_t<DH, G, KBP, NST>(c, splits); }
  static int invalid() { return 0; }
};

}  // namespace

// Key splits per (sequence, kv head): the largest count up to 16 (and about
// two CTAs per SM overall) whose clusters all fit on the device at once;
// when none does, the plain share of the SMs.  GPCs bound how many clusters
// of a given size can be resident (on a GB300, 7 of 16 CTAs but 8 of 12), so
// the largest split is not always the fastest.
int attention_mma_splits(dflash_ctx* c, int B) {
  const int heads = B * c->cfg.n_kv_heads;
  const int s0 = std::max(1, std::min({kMergeMax, (2 * c->num_sms + heads - 1) / heads, c->attn_max_splits}));
  for (int S = s0; S > 1; --S) {
    int& n = c->attn_fit[S];
    if (n == 0) n = std::max(-1, dispatch<ClustersF>(c, S, heads > c->num_sms));
    if (n >= heads) return S;
  }
  return s0;
}

cudaError_t launch_attention_mma(dflash_ctx* c, int layer, int B, int splits, cudaStream_t s, const NextGemm& next,
                                 const AttnSrc& src) {
  return dispatch<LaunchF>(c, splits, B * c->cfg.n_kv_heads > c->num_sms, layer, B, s, &next, &src);
}

}  // namespace dflash

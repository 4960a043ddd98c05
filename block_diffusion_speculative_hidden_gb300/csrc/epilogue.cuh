// Fused epilogues of the drafter's projections.
//
// A projection's output tile (16..256 activation rows x 128 weight rows,
// fp32) is finished here, straight from shared memory, by the CTA that owns
// the complete sum (the only CTA, or one CTA per row slice of a split-K
// cluster):
//
//   EPI_STORE     z = v                             (feature-fusion FC)
//   EPI_RESIDUAL  z = x + v, x = z                  (O-proj, down-proj)
//   EPI_SWIGLU    act[m][f] = silu(g) * u           (gate/up interleaved per 64 features)
//   EPI_QKV       q (RoPE) ; block k (RoPE) and v into the sequence's block page
//   EPI_KV_INJECT K (offset + RoPE) and V of every layer into the row's page slot
//
// RMSNorm is folded into the projections instead of running as a kernel of
// its own.  RMSNorm(z) * g feeds the next projection W; since
// W (RMSNorm(z) * g) = r * W (g . z) with r = 1 / sqrt(mean(z^2) + eps) a
// per-row scalar, the producer of z (STORE or RESIDUAL) writes g . z as the
// next GEMM input together with per-(128-column tile, row) partial sums of
// z^2, and the consumer multiplies each output row by r, computed from those
// partials in a fixed order.  The result is the same function; only the
// point where the rounding to the GEMM input happens moves (g . z instead of
// r g . z, both carried as an exact two-term bf16 split).
//
// KT is the element type of q and of the KV pool: fp16 for the bf16
// workloads, fp32 for the fp32 ones.  The tile layout in shared memory is
// tile[j * 128 + t] = value of activation row m0 + j and output column
// n0 + t.  RoPE partners (i, i + dh/2) always sit in the same tile because
// tiles start on head boundaries (128 is a multiple of every head dim).
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace dflash {

// EPI_NONE: no epilogue; every split writes its raw fp32 partial plane.
enum EpiKind : int { EPI_NONE = 0, EPI_STORE = 1, EPI_RESIDUAL = 2, EPI_SWIGLU = 3, EPI_QKV = 4, EPI_KV_INJECT = 5 };

struct EpiArgs {
  int kind;
  int M, N;               // rows and columns of the projection
  const int* m_valid;     // nullable device row count (rows at or past it are left alone)
  float* out;             // STORE: nullable fp32 copy of z [M][N]; RESIDUAL: x [M][N]
  void* act_hi;           // SWIGLU: activation (ActOut of the config type) [M][F]
  void* act_lo;
  int F;
  // QKV and KV_INJECT
  void* q;                // QKV: [M][Hq*dh] (KT)
  void* pool_k;           // K pool (KT) base of the layer (QKV) or of layer 0 (KV_INJECT)
  void* pool_v;
  long long layer_stride; // elements per layer in the pool (KV_INJECT)
  int block_page0;        // QKV: page id of sequence 0's block page
  const int32_t* seq_len; // QKV: block position = seq_len[b] + i
  const int32_t* row_seq; // KV_INJECT: compact row -> sequence, absolute position
  const int32_t* row_pos;
  const int32_t* page_table;
  int max_pages;
  const float* rope_cos;
  const float* rope_sin;
  const float* key_offset;  // KV_INJECT: optional [L][Hkv][dh]
  int Hq, Hkv, dh;
  // folded RMSNorm, consumer side: nullable partial sums of squares of the
  // normalised rows, ss_in[t * ss_ld + m] for t < ss_tiles; row m of the
  // output is scaled by 1 / sqrt(sum_t ss_in / norm_dim + eps)
  const float* ss_in;
  int ss_tiles;
  float norm_dim_inv;
  float eps;
  int ss_ld;              // row stride of ss_in / ss_out
  // folded RMSNorm, producer side (STORE, RESIDUAL): nullable next input
  // (ActOut of the config type) nx[m][n] = nx_gain[n] * z[m][n], and
  // ss_out[(n0 / 128) * ss_ld + m] = sum over the tile's columns of z^2
  void* nx_hi;
  void* nx_lo;
  const void* nx_gain;
  float* ss_out;
};

__device__ __forceinline__ long long pool_index(int page, int head, int slot, int i, int Hkv, int dh) {
  return ((static_cast<long long>(page) * Hkv + head) * kPage + slot) * dh + i;
}

// 1 / RMS of row m from the partial sums of squares (fixed summation order).
__device__ __forceinline__ float norm_row_scale(const EpiArgs& e, int m) {
  float s = 0.f;
  for (int t = 0; t < e.ss_tiles; ++t) s += e.ss_in[static_cast<long long>(t) * e.ss_ld + m];
  return rsqrtf(s * e.norm_dim_inv + e.eps);
}

template <typename KT>
__device__ __forceinline__ KT kv_store(float v);
template <>
__device__ __forceinline__ float kv_store<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half kv_store<__half>(float v) { return __float2half_rn(v); }

// Per-row facts an epilogue needs from global memory, gathered ahead of it
// (by otherwise idle warps while the main loop runs): x = position, y = page
// of the row's K/V slot, z = slot in the page (QKV: the block page).
__device__ __forceinline__ int4 epi_row_info(const EpiArgs& e, int m) {
  if (e.kind == EPI_QKV) {
    const int b = m / kBlockK, slot = m % kBlockK;
    return make_int4(e.seq_len[b] + slot, e.block_page0 + b, slot, 0);
  }
  if (e.kind == EPI_KV_INJECT) {
    const int b = e.row_seq[m], pos = e.row_pos[m];
    return make_int4(pos, e.page_table[b * e.max_pages + pos / kPage], pos % kPage, 0);
  }
  return make_int4(0, 0, 0, 0);
}

constexpr int kEpiBatch = 8;  // rows finished together (their loads in flight at once); the
                              // sum-of-squares butterfly below assumes 8

// The epilogue runs on kEpiThreads threads: thread t finishes output column
// n0 + t % 128 of the rows j with j % NH == t / 128 (NH = kEpiThreads / 128),
// kEpiBatch of its rows at a time.
constexpr int kEpiThreads = 128;
__device__ __forceinline__ constexpr int epi_phases() { return kEpiThreads / 128; }
// The epilogue's threads (the first kEpiThreads of the block) meet at named
// barrier 1, so a kernel may have other warps that take no part in it.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory"); }

// Global inputs of the first kEpiBatch rows a thread finishes, loaded ahead
// of the epilogue so that their latency overlaps the accumulator readout and
// the split-K reduction.
struct EpiPre {
  float a[kEpiBatch];  // RESIDUAL: x; QKV / KV_INJECT: RoPE cos
  float b[kEpiBatch];  // QKV / KV_INJECT: RoPE sin
  float gn;            // STORE / RESIDUAL: gain of the next norm at this column
};

template <typename T>
__device__ __forceinline__ void epilogue_preload(const EpiArgs& e, int m0, int rows, int n0, const int4* ri,
                                                 EpiPre& pre) {
  const int NH = epi_phases(), h = threadIdx.x >> 7, n = n0 + (threadIdx.x & 127);
  if (e.m_valid != nullptr) rows = min(rows, *e.m_valid - m0);
  rows = min(rows, e.M - m0);
  pre.gn = 0.f;
#pragma unroll
  for (int u = 0; u < kEpiBatch; ++u) pre.a[u] = pre.b[u] = 0.f;
  if (rows <= 0 || n >= e.N) return;
  switch (e.kind) {
    case EPI_STORE:
    case EPI_RESIDUAL:
      if (e.nx_hi != nullptr) pre.gn = to_f32(static_cast<const T*>(e.nx_gain)[n]);
      if (e.kind == EPI_RESIDUAL)
#pragma unroll
        for (int u = 0; u < kEpiBatch; ++u) {
          const int j = u * NH + h;
          if (j < rows) pre.a[u] = e.out[static_cast<long long>(m0 + j) * e.N + n];
        }
      break;
    case EPI_QKV:
    case EPI_KV_INJECT: {
      bool is_v;
      int i;
      if (e.kind == EPI_QKV) {
        const int qd = e.Hq * e.dh, kvd = e.Hkv * e.dh;
        is_v = n >= qd + kvd;
        i = n % e.dh;
      } else {
        const int kvd = e.Hkv * e.dh, w = n % (2 * kvd);
        is_v = w >= kvd;
        i = w % e.dh;
      }
      if (is_v) break;
      const int half = e.dh / 2, jr = i < half ? i : i - half;
#pragma unroll
      for (int u = 0; u < kEpiBatch; ++u) {
        const int j = u * NH + h;
        if (j < rows) {
          pre.a[u] = e.rope_cos[ri[j].x * half + jr];
          pre.b[u] = e.rope_sin[ri[j].x * half + jr];
        }
      }
      break;
    }
    default:
      break;
  }
}

// Finishes one tile.  The first kEpiThreads threads of the block call it
// (see above).  `rs` (nullable) holds the row scales of rows
// m0 .. m0 + rows - 1 and `ri` (nullable) their epi_row_info; `scratch`
// holds 4 * rows floats and is used when e.ss_out is set; `pre` (nullable)
// holds each thread's first batch of global inputs (epilogue_preload).
// Every global load of a batch is issued before any of its results is used.
template <typename T, typename KT>
__device__ void apply_epilogue(const EpiArgs& e, const float* tile, int m0, int rows, int n0, const float* rs,
                               const int4* ri, float* scratch, const EpiPre* pre = nullptr) {
  const int NH = epi_phases(), h = threadIdx.x >> 7, t = threadIdx.x & 127;
  const int n = n0 + t;
  if (e.m_valid != nullptr) rows = min(rows, *e.m_valid - m0);
  rows = min(rows, e.M - m0);
  if (rows <= 0) return;
  KT* q = static_cast<KT*>(e.q);
  KT* pk = static_cast<KT*>(e.pool_k);
  KT* pv = static_cast<KT*>(e.pool_v);
  const int step = kEpiBatch * NH;  // rows covered by one batch of all phases
  switch (e.kind) {
    case EPI_STORE:
    case EPI_RESIDUAL: {
      const bool nv = n < e.N;
      const ActOut<T> nx{static_cast<T*>(e.nx_hi), static_cast<T*>(e.nx_lo)};
      const float gn = pre != nullptr ? pre->gn
                                      : (e.nx_hi != nullptr && nv) ? to_f32(static_cast<const T*>(e.nx_gain)[n]) : 0.f;
      const int warp = t >> 5, lane = t & 31;  // warp within this phase
      for (int j0 = 0; j0 < rows; j0 += step) {
        float z[kEpiBatch];
#pragma unroll
        for (int u = 0; u < kEpiBatch; ++u) {
          const int j = j0 + u * NH + h;
          z[u] = 0.f;
          if (nv && j < rows) {
            z[u] = tile[j * 128 + t] * (rs != nullptr ? rs[j] : 1.f);
            if (e.kind == EPI_RESIDUAL)
              z[u] += (pre != nullptr && j0 == 0) ? pre->a[u] : e.out[static_cast<long long>(m0 + j) * e.N + n];
          }
        }
#pragma unroll
        for (int u = 0; u < kEpiBatch; ++u) {
          const int j = j0 + u * NH + h;
          if (nv && j < rows) {
            const long long o = static_cast<long long>(m0 + j) * e.N + n;
            if (e.out != nullptr) e.out[o] = z[u];
            if (e.nx_hi != nullptr) nx.put(o, gn * z[u]);
          }
        }
        if (e.ss_out != nullptr) {
          // the warp's sums of z^2 for its 8 rows of the batch at once: a
          // transposing butterfly halves the rows a lane holds at each of the
          // first three steps (lane bits 4, 3, 2 pick the half), then two
          // steps finish the sums; lane 4u + (0..3) ends with row u
          float sq[kEpiBatch];
#pragma unroll
          for (int u = 0; u < kEpiBatch; ++u) sq[u] = z[u] * z[u];
#pragma unroll
          for (int o = 16, c = kEpiBatch; o >= 4; o >>= 1, c >>= 1) {
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < c / 2; ++i) {
              const float keep = up ? sq[i + c / 2] : sq[i], send = up ? sq[i] : sq[i + c / 2];
              sq[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
          }
          sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], 1);
          sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], 2);
          const int j = j0 + ((lane >> 2) & 7) * NH + h;
          if ((lane & 3) == 0 && j < rows) scratch[j * 4 + warp] = sq[0];
        }
      }
      if (e.ss_out != nullptr) {
        epi_sync();
        for (int j = threadIdx.x; j < rows; j += kEpiThreads)
          e.ss_out[static_cast<long long>(n0 >> 7) * e.ss_ld + m0 + j] =
              (scratch[j * 4 + 0] + scratch[j * 4 + 1]) + (scratch[j * 4 + 2] + scratch[j * 4 + 3]);
      }
      break;
    }
    case EPI_SWIGLU: {
      // tile = 64 gate rows then the 64 matching up rows; thread t takes
      // feature t % 64 of the rows j with j % P == t / 64 (P = kEpiThreads / 64)
      constexpr int P = kEpiThreads / 64;
      const int c = threadIdx.x & 63, ph = threadIdx.x >> 6;
      const int f = (n0 >> 7) * 64 + c;
      if (f < e.F) {
        ActOut<T> a{static_cast<T*>(e.act_hi), static_cast<T*>(e.act_lo)};
        for (int j0 = ph; j0 < rows; j0 += P * kEpiBatch) {
#pragma unroll
          for (int u = 0; u < kEpiBatch; ++u) {
            const int j = j0 + P * u;
            if (j < rows) {
              const float sc = rs != nullptr ? rs[j] : 1.f;
              const float g = tile[j * 128 + c] * sc, up = tile[j * 128 + c + 64] * sc;
              a.put(static_cast<long long>(m0 + j) * e.F + f, g / (1.f + expf(-g)) * up);
            }
          }
        }
      }
      break;
    }
    case EPI_QKV:
    case EPI_KV_INJECT: {
      if (n >= e.N) break;
      const int half = e.dh / 2;
      int kind;    // 0: q, 1: k, 2: v
      int head;    // q head (kind 0) or kv head
      int i;       // element within the head
      int l = 0;   // layer (KV_INJECT)
      float off_lo = 0.f, off_hi = 0.f;
      if (e.kind == EPI_QKV) {
        const int qd = e.Hq * e.dh, kvd = e.Hkv * e.dh;
        kind = n < qd ? 0 : n < qd + kvd ? 1 : 2;
        const int w = kind == 0 ? n : kind == 1 ? n - qd : n - qd - kvd;
        head = w / e.dh;
        i = w % e.dh;
      } else {
        const int kvd = e.Hkv * e.dh;
        l = n / (2 * kvd);
        const int w = n % (2 * kvd);
        kind = w < kvd ? 1 : 2;
        head = (kind == 1 ? w : w - kvd) / e.dh;
        i = w % e.dh;
        if (kind == 1 && e.key_offset != nullptr) {
          const float* ko = e.key_offset + (static_cast<long long>(l) * e.Hkv + head) * e.dh;
          const int jj = i < half ? i : i - half;
          off_lo = ko[jj];
          off_hi = ko[jj + half];
        }
      }
      const int jr = i < half ? i : i - half;  // RoPE frequency index
      const int base = t - i;                   // tile column of the head's element 0
      const long long lbase = static_cast<long long>(l) * e.layer_stride;
      for (int j0 = 0; j0 < rows; j0 += step) {
        int4 info[kEpiBatch];
        float cs[kEpiBatch], sn[kEpiBatch];
#pragma unroll
        for (int u = 0; u < kEpiBatch; ++u) {
          const int j = min(j0 + u * NH + h, rows - 1);
          info[u] = ri != nullptr ? ri[j] : epi_row_info(e, m0 + j);
          cs[u] = sn[u] = 0.f;
          if (kind != 2) {
            if (pre != nullptr && j0 == 0) {
              cs[u] = pre->a[u];
              sn[u] = pre->b[u];
            } else {
              cs[u] = e.rope_cos[info[u].x * half + jr];
              sn[u] = e.rope_sin[info[u].x * half + jr];
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kEpiBatch; ++u) {
          const int j = j0 + u * NH + h;
          if (j >= rows) continue;
          const float* row = tile + j * 128;
          const float sc = rs != nullptr ? rs[j] : 1.f;
          float v;
          if (kind == 2) {
            v = row[t] * sc;
          } else {
            const float x1 = row[base + jr] * sc + off_lo, x2 = row[base + jr + half] * sc + off_hi;
            v = i < half ? x1 * cs[u] - x2 * sn[u] : x2 * cs[u] + x1 * sn[u];
          }
          if (kind == 0) {
            q[static_cast<long long>(m0 + j) * (e.Hq * e.dh) + n] = kv_store<KT>(v);
          } else {
            const long long idx = lbase + pool_index(info[u].y, head, info[u].z, i, e.Hkv, e.dh);
            (kind == 1 ? pk : pv)[idx] = kv_store<KT>(v);
          }
        }
      }
      break;
    }
    default:
      break;
  }
}

}  // namespace dflash

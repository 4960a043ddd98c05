// Fused epilogues of the drafter's projections.
//
// A projection's output tile (16..256 activation rows x 128 weight rows,
// fp32) is finished here, straight from shared memory, by the CTA that owns
// the complete sum (the only CTA, or the last split-K CTA of the tile):
//
//   EPI_STORE     out[m][n] = v                     (feature-fusion FC)
//   EPI_RESIDUAL  x[m][n] += v                      (O-proj, down-proj)
//   EPI_SWIGLU    act[m][f] = silu(g) * u           (gate/up interleaved per 64 features)
//   EPI_QKV       q (RoPE) ; block k (RoPE) and v into the sequence's block page
//   EPI_KV_INJECT K (offset + RoPE) and V of every layer into the row's page slot
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
  float* out;             // STORE: [M][N]; RESIDUAL: x [M][N]
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
};

__device__ __forceinline__ long long pool_index(int page, int head, int slot, int i, int Hkv, int dh) {
  return ((static_cast<long long>(page) * Hkv + head) * kPage + slot) * dh + i;
}

// RoPE (rotate-half) of element i of the head whose element 0 sits at tile
// column t - i, at position pos; add_lo/add_hi are added to the pair first.
__device__ __forceinline__ float rope_col(const float* row, int t, int i, int dh, int pos, const float* rc,
                                          const float* rs, float add_lo = 0.f, float add_hi = 0.f) {
  const int half = dh / 2;
  const int base = t - i;
  const int j = i < half ? i : i - half;
  const float x1 = row[base + j] + add_lo, x2 = row[base + j + half] + add_hi;
  const float cs = rc[pos * half + j], sn = rs[pos * half + j];
  return i < half ? x1 * cs - x2 * sn : x2 * cs + x1 * sn;
}

template <typename KT>
__device__ __forceinline__ KT kv_store(float v);
template <>
__device__ __forceinline__ float kv_store<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half kv_store<__half>(float v) { return __float2half_rn(v); }

// Finishes one tile.  All threads of the block call it; thread t handles
// output column n0 + t (blockDim.x == 128).
template <typename T, typename KT>
__device__ void apply_epilogue(const EpiArgs& e, const float* tile, int m0, int rows, int n0) {
  const int t = threadIdx.x;
  const int n = n0 + t;
  if (e.m_valid != nullptr) rows = min(rows, *e.m_valid - m0);
  KT* q = static_cast<KT*>(e.q);
  KT* pk = static_cast<KT*>(e.pool_k);
  KT* pv = static_cast<KT*>(e.pool_v);
  switch (e.kind) {
    case EPI_STORE:
      if (n < e.N)
        for (int j = 0; j < rows && m0 + j < e.M; ++j)
          e.out[static_cast<long long>(m0 + j) * e.N + n] = tile[j * 128 + t];
      break;
    case EPI_RESIDUAL:
      if (n < e.N)
        for (int j = 0; j < rows && m0 + j < e.M; ++j)
          e.out[static_cast<long long>(m0 + j) * e.N + n] += tile[j * 128 + t];
      break;
    case EPI_SWIGLU: {
      const int f = (n0 >> 7) * 64 + t;  // tile = 64 gate rows then the 64 matching up rows
      if (t < 64 && f < e.F) {
        ActOut<T> a{static_cast<T*>(e.act_hi), static_cast<T*>(e.act_lo)};
        for (int j = 0; j < rows && m0 + j < e.M; ++j) {
          const float g = tile[j * 128 + t], u = tile[j * 128 + t + 64];
          a.put(static_cast<long long>(m0 + j) * e.F + f, g / (1.f + expf(-g)) * u);
        }
      }
      break;
    }
    case EPI_QKV: {
      if (n >= e.N) break;
      const int qd = e.Hq * e.dh, kvd = e.Hkv * e.dh;
      const int i = n % e.dh;
      for (int j = 0; j < rows && m0 + j < e.M; ++j) {
        const int m = m0 + j, b = m / kBlockK, slot = m % kBlockK;
        const float* row = tile + j * 128;
        if (n < qd) {
          const int pos = e.seq_len[b] + slot;
          q[static_cast<long long>(m) * qd + n] = kv_store<KT>(rope_col(row, t, i, e.dh, pos, e.rope_cos, e.rope_sin));
        } else if (n < qd + kvd) {
          const int pos = e.seq_len[b] + slot, g = (n - qd) / e.dh;
          pk[pool_index(e.block_page0 + b, g, slot, i, e.Hkv, e.dh)] =
              kv_store<KT>(rope_col(row, t, i, e.dh, pos, e.rope_cos, e.rope_sin));
        } else {
          const int g = (n - qd - kvd) / e.dh;
          pv[pool_index(e.block_page0 + b, g, slot, i, e.Hkv, e.dh)] = kv_store<KT>(row[t]);
        }
      }
      break;
    }
    case EPI_KV_INJECT: {
      if (n >= e.N) break;
      const int kvd = e.Hkv * e.dh;
      const int l = n / (2 * kvd), w = n % (2 * kvd);
      const bool is_k = w < kvd;
      const int g = (is_k ? w : w - kvd) / e.dh, i = w % e.dh, half = e.dh / 2;
      float off_lo = 0.f, off_hi = 0.f;
      if (is_k && e.key_offset != nullptr) {
        const float* ko = e.key_offset + (static_cast<long long>(l) * e.Hkv + g) * e.dh;
        const int jj = i < half ? i : i - half;
        off_lo = ko[jj];
        off_hi = ko[jj + half];
      }
      for (int j = 0; j < rows && m0 + j < e.M; ++j) {
        const int r = m0 + j;
        const int b = e.row_seq[r], pos = e.row_pos[r];
        const int page = e.page_table[b * e.max_pages + pos / kPage], slot = pos % kPage;
        const float* row = tile + j * 128;
        const long long idx = l * e.layer_stride + pool_index(page, g, slot, i, e.Hkv, e.dh);
        if (is_k)
          pk[idx] = kv_store<KT>(rope_col(row, t, i, e.dh, pos, e.rope_cos, e.rope_sin, off_lo, off_hi));
        else
          pv[idx] = kv_store<KT>(row[t]);
      }
      break;
    }
    default:
      break;
  }
}

}  // namespace dflash

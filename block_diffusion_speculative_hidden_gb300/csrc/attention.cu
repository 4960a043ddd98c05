// Block attention: the K block queries of one sequence attend, with no mask,
// to every injected context key in the paged cache and to all K block keys
// (the DFlash Guide: bidirectional self-attention across the masked block;
// the stable-lab chapter: a block position sees its neighbours' [MASK]
// placeholders, and the injected target context).
//
// One CTA per (sequence, kv head, key split).  The G query heads that share
// a kv head are stacked with the K block positions into R = 16 G query rows,
// so each K/V element read from HBM serves R rows.  Keys are walked in
// chunks of 32 with an online softmax; each split writes an unnormalised
// (o, m, l) partial and a second kernel merges the splits.  No CTA waits on
// another.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "kernels.cuh"

namespace dflash {

constexpr int kAttnThreads = 256;
constexpr int kChunk = 32;

template <int DH, int G>
struct AttnCfg {
  static constexpr int R = G * kBlockK;
  static constexpr int TPR = kAttnThreads / R;  // threads per row in the P.V phase
  static constexpr int DPT = DH / TPR;          // output dims per thread
  static constexpr int RPW = R / 8;             // score rows per warp
  static constexpr int SMEM = sizeof(float) * (R * (DH + 1) + 2 * kChunk * (DH + 1) + R * (kChunk + 1) + R);
};

// KT: element type of q and of the KV pool.  The block's own keys sit in
// page block_page0 + b of the pool, after the T_b context keys.
template <typename KT, int DH, int G>
__global__ void __launch_bounds__(kAttnThreads) k_attn_split(
    const KT* __restrict__ q, const KT* __restrict__ pool_k, const KT* __restrict__ pool_v,
    const int32_t* __restrict__ page_table, int max_pages, int block_page0, const int32_t* __restrict__ seq_len,
    float* __restrict__ part_o, float* __restrict__ part_ml, int Hkv, int splits, float scale) {
  using C = AttnCfg<DH, G>;
  constexpr int R = C::R;
  extern __shared__ float sm[];
  float* sQ = sm;                          // [R][DH+1]
  float* sK = sQ + R * (DH + 1);           // [32][DH+1]
  float* sV = sK + kChunk * (DH + 1);      // [32][DH+1]
  float* sP = sV + kChunk * (DH + 1);      // [R][33]
  float* sAlpha = sP + R * (kChunk + 1);   // [R]

  const int sp = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hq = Hkv * G, qd = Hq * DH;
  const int T_ctx = seq_len[b];
  const int n_keys = T_ctx + kBlockK;
  const int n_chunks = (n_keys + kChunk - 1) / kChunk;
  const int cps = (n_chunks + splits - 1) / splits;
  const int c_begin = sp * cps, c_end = min(n_chunks, c_begin + cps);

  // q rows: r = gi * 16 + i  <->  q head kvh*G + gi, block position i; pre-scaled by 1/sqrt(dh)
  for (int e = tid; e < R * DH; e += kAttnThreads) {
    const int r = e / DH, dd = e % DH, gi = r / kBlockK, i = r % kBlockK;
    sQ[r * (DH + 1) + dd] =
        to_f32(q[static_cast<long long>(b * kBlockK + i) * qd + (kvh * G + gi) * DH + dd]) * scale;
  }
  float m_run[C::RPW], l_run[C::RPW];
#pragma unroll
  for (int k = 0; k < C::RPW; ++k) {
    m_run[k] = -INFINITY;
    l_run[k] = 0.f;
  }
  float acc[C::DPT];
#pragma unroll
  for (int k = 0; k < C::DPT; ++k) acc[k] = 0.f;
  const int pr = tid / C::TPR, pd = tid % C::TPR;

  for (int ch = c_begin; ch < c_end; ++ch) {
    const int key0 = ch * kChunk;
    __syncthreads();
    for (int e = tid; e < kChunk * DH; e += kAttnThreads) {
      const int j = e / DH, dd = e % DH, key = key0 + j;
      float kv = 0.f, vv = 0.f;
      if (key < n_keys) {
        const int page = key < T_ctx ? page_table[b * max_pages + key / kPage] : block_page0 + b;
        const int slot = key < T_ctx ? key % kPage : key - T_ctx;
        const long long off = (static_cast<long long>(page) * Hkv + kvh) * (kPage * DH) + slot * DH + dd;
        kv = to_f32(pool_k[off]);
        vv = to_f32(pool_v[off]);
      }
      sK[j * (DH + 1) + dd] = kv;
      sV[j * (DH + 1) + dd] = vv;
    }
    __syncthreads();
    const bool kvalid = key0 + lane < n_keys;
#pragma unroll
    for (int k = 0; k < C::RPW; ++k) {
      const int r = warp + 8 * k;
      float s = 0.f;
#pragma unroll 8
      for (int dd = 0; dd < DH; ++dd) s = fmaf(sQ[r * (DH + 1) + dd], sK[lane * (DH + 1) + dd], s);
      s = kvalid ? s : -INFINITY;
      const float cmax = warp_max(s);
      const float m_new = fmaxf(m_run[k], cmax);
      const float alpha = (m_run[k] == -INFINITY) ? 0.f : expf(m_run[k] - m_new);
      const float p = kvalid ? expf(s - m_new) : 0.f;
      l_run[k] = l_run[k] * alpha + warp_sum(p);
      m_run[k] = m_new;
      sP[r * (kChunk + 1) + lane] = p;
      if (lane == 0) sAlpha[r] = alpha;
    }
    __syncthreads();
    const float al = sAlpha[pr];
#pragma unroll
    for (int k = 0; k < C::DPT; ++k) acc[k] *= al;
    for (int j = 0; j < kChunk; ++j) {
      const float p = sP[pr * (kChunk + 1) + j];
#pragma unroll
      for (int k = 0; k < C::DPT; ++k) acc[k] = fmaf(p, sV[j * (DH + 1) + pd + C::TPR * k], acc[k]);
    }
  }
  const long long base = (static_cast<long long>(b) * Hkv + kvh) * splits + sp;
#pragma unroll
  for (int k = 0; k < C::DPT; ++k) part_o[(base * R + pr) * DH + pd + C::TPR * k] = acc[k];
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < C::RPW; ++k) {
      const int r = warp + 8 * k;
      part_ml[(base * R + r) * 2 + 0] = m_run[k];
      part_ml[(base * R + r) * 2 + 1] = l_run[k];
    }
  }
}

// o[m][h*DH + d] = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s
template <typename T>
__global__ void k_attn_combine(const float* __restrict__ part_o, const float* __restrict__ part_ml, ActOut<T> o,
                               int Hkv, int G, int DH, int splits) {
  const int m = blockIdx.x;
  const int b = m / kBlockK, i = m % kBlockK;
  const int R = G * kBlockK, Hq = Hkv * G;
  for (int e = threadIdx.x; e < Hq * DH; e += blockDim.x) {
    const int h = e / DH, dd = e % DH, kvh = h / G, gi = h % G, r = gi * kBlockK + i;
    const long long base = (static_cast<long long>(b) * Hkv + kvh) * splits;
    float M = -INFINITY;
    for (int s = 0; s < splits; ++s) M = fmaxf(M, part_ml[((base + s) * R + r) * 2]);
    float num = 0.f, den = 0.f;
    for (int s = 0; s < splits; ++s) {
      const float ms = part_ml[((base + s) * R + r) * 2];
      if (ms == -INFINITY) continue;
      const float w = expf(ms - M);
      den += w * part_ml[((base + s) * R + r) * 2 + 1];
      num += w * part_o[((base + s) * R + r) * DH + dd];
    }
    o.put(static_cast<long long>(m) * Hq * DH + e, num / den);
  }
}

// Key splits per (sequence, kv head): enough CTAs for about two per SM; the
// tensor-core kernel merges its splits inside one cluster (at most 16).
int attn_splits(dflash_ctx* c, int B) {
  if (c->cfg.dtype != DFLASH_F32) return attention_mma_splits(c, B);
  const int heads = B * c->cfg.n_kv_heads;
  const int s = (2 * c->num_sms + heads - 1) / heads;
  return std::max(1, std::min(s, c->attn_max_splits));
}

template <typename T, int DH, int G>
static cudaError_t launch_attn_t(dflash_ctx* c, int layer, int B, int splits, cudaStream_t s) {
  using C = AttnCfg<DH, G>;
  using KT = typename std::conditional<std::is_same<T, float>::value, float, __half>::type;
  static FuncAttr smem_attr;
  cudaError_t ae = smem_attr.ensure(C::SMEM, [](int v) {
    return cudaFuncSetAttribute(k_attn_split<KT, DH, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, v);
  });
  if (ae != cudaSuccess) return ae;
  const auto& g = c->cfg;
  const long long layer_off = static_cast<long long>(layer) * c->pool_pages * g.n_kv_heads * kPage * DH;
  dim3 grid(splits, g.n_kv_heads, B);
  k_attn_split<KT, DH, G><<<grid, kAttnThreads, C::SMEM, s>>>(
      static_cast<const KT*>(c->q), static_cast<const KT*>(c->pool_k) + layer_off,
      static_cast<const KT*>(c->pool_v) + layer_off, c->page_table, g.max_pages_per_seq, g.n_pages, c->seq_len,
      c->attn_o, c->attn_ml, g.n_kv_heads, splits, 1.0f / sqrtf(static_cast<float>(DH)));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_attn_combine<T><<<B * kBlockK, 256, 0, s>>>(c->attn_o, c->attn_ml,
                                                ActOut<T>{static_cast<T*>(c->o), static_cast<T*>(c->o_lo)},
                                                g.n_kv_heads, G, DH, splits);
  return cudaGetLastError();
}

template <typename T, int DH>
static cudaError_t launch_attn_dh(dflash_ctx* c, int layer, int B, int splits, cudaStream_t s) {
  switch (c->cfg.n_q_heads / c->cfg.n_kv_heads) {
    case 1: return launch_attn_t<T, DH, 1>(c, layer, B, splits, s);
    case 2: return launch_attn_t<T, DH, 2>(c, layer, B, splits, s);
    case 4: return launch_attn_t<T, DH, 4>(c, layer, B, splits, s);
    case 8: return launch_attn_t<T, DH, 8>(c, layer, B, splits, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
static cudaError_t launch_attn_ty(dflash_ctx* c, int layer, int B, int splits, cudaStream_t s) {
  switch (c->cfg.head_dim) {
    case 32: return launch_attn_dh<T, 32>(c, layer, B, splits, s);
    case 64: return launch_attn_dh<T, 64>(c, layer, B, splits, s);
    case 128: return launch_attn_dh<T, 128>(c, layer, B, splits, s);
    default: return cudaErrorInvalidValue;
  }
}

// fp32 workloads: the fp32 SIMT kernel above; bf16 workloads (fp16 pool):
// the tcgen05 kernel of attention_mma.cu.
cudaError_t launch_attention(dflash_ctx* c, int layer, int B, int splits, cudaStream_t s, const NextGemm& next,
                             const AttnSrc& src) {
  if (c->cfg.dtype != DFLASH_F32) return launch_attention_mma(c, layer, B, splits, s, next, src);
  if (src.row_of != nullptr || src.seq_len != nullptr || src.order != nullptr)
    return cudaErrorInvalidValue;  // bf16 family only
  return launch_attn_ty<float>(c, layer, B, splits, s);
}

}  // namespace dflash

// Training-time block attention (the DFlash paper's Figure 4: a block sees
// the target context before its start and its own K positions, bidirectional;
// no other block).  Per block that is exactly the inference block attention
// over a context prefix, so the tcgen05 attention kernel runs all blocks of a
// batch at once: block v reads its sequence's context pages up to its
// prefix length and its own keys and values from block page n_pages + v.
// These kernels stage the blocks into that form and return the output.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "kernels.cuh"

namespace dflash {

// The sequence and prefix length of block v, checked against the sequence
// (an out-of-range sequence or a prefix longer than it is clamped; *bad set).
__device__ __forceinline__ int2 block_src(int v, int max_batch, const int32_t* seq, const int32_t* ctx_len,
                                          const int32_t* seq_len, bool* bad) {
  int s = seq[v], c = ctx_len[v];
  *bad = s < 0 || s >= max_batch;
  if (*bad) s = 0;
  const int L = seq_len[s];
  if (c < 0 || c > L) {
    *bad = true;
    c = c < 0 ? 0 : L;
  }
  return make_int2(s, c);
}

// One CTA per block v: the page-table row and prefix length (checked, see
// block_src; a bad block sets ST_BAD_BLOCK), the block's place in the
// attention's launch order (longest prefix first, ties by index: the rank of
// v among all blocks), the block's queries into the query buffer
// ([v*16 + i][Hq*dh], fp16, the layout they arrive in), and its keys and
// values from [16][Hkv][dh] (token-major) into the pool's block page
// [Hkv][16][dh] of the layer.
__global__ void k_blockattn_stage(int NB, int max_batch, const int32_t* __restrict__ seq,
                                  const int32_t* __restrict__ ctx_len, const int32_t* __restrict__ seq_len,
                                  int32_t* blk_row, int32_t* blk_len, int32_t* order, const __half* __restrict__ q,
                                  const __half* __restrict__ kb, const __half* __restrict__ vb, __half* q_buf,
                                  __half* pool_k_layer, __half* pool_v_layer, int block_page0, int qd, int Hkv,
                                  int dh, int* status) {
  const int v = blockIdx.x;
  if (v >= NB) return;
  bool bad;
  const int2 src = block_src(v, max_batch, seq, ctx_len, seq_len, &bad);
  int rank = 0;
  for (int u0 = 0; u0 < NB; u0 += blockDim.x) {
    const int u = u0 + threadIdx.x;
    bool before = false;
    if (u < NB) {
      bool bad_u;
      const int lu = block_src(u, max_batch, seq, ctx_len, seq_len, &bad_u).y;
      before = lu > src.y || (lu == src.y && u < v);
    }
    rank += __syncthreads_count(before);
  }
  if (threadIdx.x == 0) {
    if (bad) atomicOr(status, ST_BAD_BLOCK);
    blk_row[v] = src.x;
    blk_len[v] = src.y;
    order[rank] = v;
  }
  // queries: 16 rows of qd halves, copied 8 halves (16 bytes) at a time
  const long long q0 = static_cast<long long>(v) * kBlockK * qd;
  for (int e = threadIdx.x; e < kBlockK * qd / 8; e += blockDim.x)
    reinterpret_cast<uint4*>(q_buf + q0)[e] = reinterpret_cast<const uint4*>(q + q0)[e];
  // keys and values: element (i, h, d) of the block -> page (h, i, d)
  const int kvd = Hkv * dh;
  const long long b0 = static_cast<long long>(v) * kBlockK * kvd;
  const long long page = static_cast<long long>(block_page0 + v) * kvd * kPage;
  for (int e = threadIdx.x; e < kBlockK * kvd / 8; e += blockDim.x) {
    const int i = (e * 8) / kvd, r = (e * 8) % kvd, h = r / dh, d = r % dh;
    const long long dst = page + (static_cast<long long>(h) * kPage + i) * dh + d;
    *reinterpret_cast<uint4*>(pool_k_layer + dst) = reinterpret_cast<const uint4*>(kb + b0)[e];
    *reinterpret_cast<uint4*>(pool_v_layer + dst) = reinterpret_cast<const uint4*>(vb + b0)[e];
  }
}

// out[r][c] = o_hi[r][c] + o_lo[r][c] (the attention output's exact pair of
// bf16 terms) for the NB * 16 block rows.
__global__ void k_blockattn_out(long long n, const __nv_bfloat16* __restrict__ hi,
                                const __nv_bfloat16* __restrict__ lo, float* __restrict__ out) {
  for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < n;
       e += static_cast<long long>(gridDim.x) * blockDim.x)
    out[e] = __bfloat162float(hi[e]) + __bfloat162float(lo[e]);
}

cudaError_t launch_block_attention(dflash_ctx* c, int layer, int NB, const int32_t* seq, const int32_t* ctx_len,
                                   const void* q, const void* k_blk, const void* v_blk, float* out, cudaStream_t s) {
  const auto& g = c->cfg;
  const int qd = g.n_q_heads * g.head_dim;
  const long long per_layer = static_cast<long long>(c->pool_pages) * g.n_kv_heads * kPage * g.head_dim;
  __half* pk = static_cast<__half*>(c->pool_k) + per_layer * layer;
  __half* pv = static_cast<__half*>(c->pool_v) + per_layer * layer;
  k_blockattn_stage<<<NB, 256, 0, s>>>(NB, g.max_batch, seq, ctx_len, c->seq_len, c->blk_row, c->blk_len,
                                       c->attn_order, static_cast<const __half*>(q), static_cast<const __half*>(k_blk),
                                       static_cast<const __half*>(v_blk), static_cast<__half*>(c->q), pk, pv,
                                       g.n_pages, qd, g.n_kv_heads, g.head_dim, c->status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  AttnSrc src;
  src.row_of = c->blk_row;
  src.seq_len = c->blk_len;
  src.order = c->attn_order;
  src.pdl = false;  // the staging kernel just wrote the rows, lengths and order
  e = launch_attention(c, layer, NB, attn_splits(c, NB), s, NextGemm{}, src);
  if (e != cudaSuccess) return e;
  const long long n = static_cast<long long>(NB) * kBlockK * qd;
  k_blockattn_out<<<static_cast<int>(std::min<long long>((n + 255) / 256, 4L * c->num_sms)), 256, 0, s>>>(
      n, static_cast<const __nv_bfloat16*>(c->o), static_cast<const __nv_bfloat16*>(c->o_lo), out);
  return cudaGetLastError();
}

}  // namespace dflash

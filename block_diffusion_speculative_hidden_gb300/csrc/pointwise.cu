// Row-wise kernels around the projections: the gather of the injected
// feature rows, the block input embedding, the LM-head argmax merge and the
// S = 2 commit.  (Residual adds, the RMSNorms, SwiGLU, RoPE and the paged
// K/V stores run inside the projection epilogues, epilogue.cuh.)
//
// Passages: the DFlash Guide, "2. Target Hidden-State Conditioning" (fused
// features) and "3. Cross-Layer KV Injection" (K, V of every draft layer
// from the fused features); "1. Single-Pass Block-Diffusion Drafting" (a
// [MASK]-filled block, argmax over the vocabulary); the stable-lab chapter,
// "The Model at a Glance" (S refinement passes committing positions in
// confidence order).
#include "common.cuh"
#include "kernels.cuh"

namespace dflash {

// ------------------------------------------------------------ inject side

// Copy the valid feature rows into a compact [rows][F] buffer (rows ordered
// by sequence, then position).
template <typename T>
__global__ void k_gather_rows(const T* __restrict__ feats, T* __restrict__ out, const int* scal,
                              const int32_t* row_src, int F) {
  pdl_wait();  // the row map comes from the page allocation just before
  pdl_trigger();
  const int r = blockIdx.x;
  if (r >= scal[0]) return;
  const long long src = row_src[r];
  const int4* s = reinterpret_cast<const int4*>(feats + src * F);
  int4* d = reinterpret_cast<int4*>(out + static_cast<long long>(r) * F);
  const int n16 = F * static_cast<int>(sizeof(T)) / 16;
  for (int i = threadIdx.x; i < n16; i += blockDim.x) d[i] = s[i];
}

// ------------------------------------------------------------ draft side

// Block input: x[m] = E[token] (token = [MASK], or in pass 2 the committed
// pass-1 token).  Also the first layer's pre-norm in folded form (see
// epilogue.cuh): a[m] = g_in . x[m] and the per-128-column sums of x^2.
// CTAs of 128 threads per row, a warp per 128-column tile (four columns a
// lane); a row's tiles in one CTA when there are many rows, four a CTA when
// there are few.
template <typename T>
__device__ __forceinline__ void load4(const T* p, float (&v)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&v)[4]) {
  const float4 t = *reinterpret_cast<const float4*>(p);
  v[0] = t.x;
  v[1] = t.y;
  v[2] = t.z;
  v[3] = t.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 t = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&t.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&t.y));
  v[0] = a.x;
  v[1] = a.y;
  v[2] = b.x;
  v[3] = b.y;
}

template <typename T>
__global__ void __launch_bounds__(128) k_embed(const T* __restrict__ embed, const T* __restrict__ gain,
                                               float* __restrict__ x, ActOut<T> a, float* __restrict__ ss, int ss_ld,
                                               int d, int mask_id, int vocab, const int32_t* commit,
                                               const int32_t* tok1, int* status, const int32_t* seq_len,
                                               int32_t* order, int B, int tiles_per_cta) {
  pdl_wait();
  pdl_trigger();
  const int m = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (order != nullptr && m == 0 && blockIdx.x == 0) {
    // the attention's launch order: sequences by context length, longest
    // first (ties by index), so that the long ones do not start last
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
      const int lb = __ldg(seq_len + b);
      int rank = 0;
      for (int u = 0; u < B; ++u) {
        const int lu = __ldg(seq_len + u);
        rank += lu > lb || (lu == lb && u < b);
      }
      order[rank] = b;
    }
  }
  int tok = mask_id;
  if (commit != nullptr && commit[m] != 0) tok = tok1[m];
  if (tok < 0 || tok >= vocab) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(status, ST_BAD_TOKEN);
    tok = mask_id;
  }
  const T* row = embed + static_cast<long long>(tok) * d;
  // this CTA's 128-column tiles t0 .. t1 - 1; warp w takes t0 + w, t0 + w + 4,
  // ...; lane l their columns 4l .. 4l + 3
  const int t0 = blockIdx.x * tiles_per_cta, t1 = min(t0 + tiles_per_cta, (d + 127) / 128);
  for (int tile = t0 + warp; tile < t1; tile += 4) {
    const int n = tile * 128 + 4 * lane;
    float q = 0.f;
    if (n < d) {  // d % 4 == 0: the four columns are valid together
      float v[4], g[4];
      load4(row + n, v);
      load4(gain + n, g);
      const long long e = static_cast<long long>(m) * d + n;
      *reinterpret_cast<float4*>(x + e) = make_float4(v[0], v[1], v[2], v[3]);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        a.put(e + k, v[k] * g[k]);
        q += v[k] * v[k];
      }
    }
    q = warp_sum(q);
    if (lane == 0) ss[static_cast<long long>(tile) * ss_ld + m] = q;
  }
}

// fp32 path: per (row, 128-column tile) max / argmax / sum-exp of the logits,
// same format as the tensor-core LM-head epilogue; optional copy-out.
// The final RMSNorm arrives folded: z holds W (g . x) and row m is scaled
// by the row's 1 / RMS here.
__global__ void k_logits_tiles(const float* __restrict__ z, int V, LmPartials lm, float* user, const int32_t* skip,
                               EpiArgs norm) {
  __shared__ float smx[4];
  __shared__ int sidx[4];
  __shared__ float sse[4];
  __shared__ float s_r;
  const int m = blockIdx.y, tile = blockIdx.x;
  const int n = tile * kTileN + threadIdx.x;  // blockDim = 128
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) s_r = norm_row_scale(norm, m);
  __syncthreads();
  const bool nv = n < V;
  const float val = nv ? z[static_cast<long long>(m) * V + n] * s_r : -INFINITY;
  if (user != nullptr && nv && (skip == nullptr || skip[m] == 0)) user[static_cast<long long>(m) * V + n] = val;
  float mx = val;
  int ix = n;
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, mx, o);
    const int oi = __shfl_xor_sync(0xffffffffu, ix, o);
    if (om > mx || (om == mx && oi < ix)) {
      mx = om;
      ix = oi;
    }
  }
  const float se = warp_sum(nv ? expf(val - mx) : 0.f);
  if (lane == 0) {
    smx[warp] = mx;
    sidx[warp] = ix;
    sse[warp] = se;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = smx[0];
    int I = sidx[0];
    for (int w = 1; w < 4; ++w)
      if (smx[w] > M) {
        M = smx[w];
        I = sidx[w];
      }
    float S = 0.f;
    for (int w = 0; w < 4; ++w)
      if (smx[w] > -INFINITY) S += sse[w] * expf(smx[w] - M);
    const long long o = static_cast<long long>(m) * lm.n_tiles + tile;
    lm.mx[o] = M;
    lm.se[o] = S;
    lm.idx[o] = I;
  }
}

// One CTA per row: merge the tile partials into (argmax, confidence).
// Confidence = max softmax probability = exp(max - LSE) = 1 / sum exp(z - max).
// With `commit`, committed rows keep tok1/conf1 and only the others are merged.
// Each thread folds a strided set of tiles (increasing column order), then the
// CTA combines the per-thread states in a fixed tree, ties to the lower id.
__device__ __forceinline__ void lm_fold(float& mx, float& se, int& ix, float om, float os, int oi) {
  const float nm = fmaxf(mx, om);
  const float ns = (mx > -INFINITY ? se * expf(mx - nm) : 0.f) + (om > -INFINITY ? os * expf(om - nm) : 0.f);
  if (om > mx || (om == mx && oi < ix)) ix = oi;
  mx = nm;
  se = ns;
}

// compact (S = 2, second pass): the LM head ran on the uncommitted rows
// only, sequence b's in position order at rows b * K/2 ...; row m takes its
// partials from there.
__global__ void __launch_bounds__(256) k_lm_merge(LmPartials lm, int M, const int32_t* commit, const int32_t* tok1,
                                                  const float* conf1, int32_t* tok_out, float* conf_out,
                                                  int compact) {
  __shared__ float s_mx[8], s_se[8];
  __shared__ int s_ix[8];
  pdl_wait();
  pdl_trigger();
  const int m = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (commit != nullptr && commit[m] != 0) {
    if (threadIdx.x == 0) {
      tok_out[m] = tok1[m];
      if (conf_out != nullptr) conf_out[m] = conf1[m];
    }
    return;
  }
  int prow = m;
  if (compact) {
    const int b = m / kBlockK, i = m % kBlockK;
    int rank = 0;
    for (int j = 0; j < i; ++j) rank += commit[b * kBlockK + j] == 0 ? 1 : 0;
    prow = b * (kBlockK / 2) + rank;
  }
  const long long base = static_cast<long long>(prow) * lm.n_tiles;
  float mx = -INFINITY, se = 0.f;
  int ix = 0x7fffffff;
  for (int t = threadIdx.x; t < lm.n_tiles; t += blockDim.x) lm_fold(mx, se, ix, lm.mx[base + t], lm.se[base + t], lm.idx[base + t]);
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, mx, o), os = __shfl_xor_sync(0xffffffffu, se, o);
    const int oi = __shfl_xor_sync(0xffffffffu, ix, o);
    lm_fold(mx, se, ix, om, os, oi);
  }
  if (lane == 0) {
    s_mx[warp] = mx;
    s_se[warp] = se;
    s_ix[warp] = ix;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) lm_fold(mx, se, ix, s_mx[w], s_se[w], s_ix[w]);
    tok_out[m] = ix;
    if (conf_out != nullptr) conf_out[m] = 1.f / se;
  }
}

// S = 2, second pass: the K/2 uncommitted rows of each sequence, in position
// order, into compact rows b * K/2 + r (the two bf16 terms of the LM head's
// input and their folded-norm partial sums), so that the LM head runs on
// them alone; crow[j] records the block row of compact row j (where a logits
// store puts it back).  One CTA per compact row.
__global__ void k_compact_rows(const int32_t* __restrict__ commit, const __nv_bfloat16* __restrict__ a,
                               const __nv_bfloat16* __restrict__ a_lo, const float* __restrict__ ss, int ss_ld,
                               int d_tiles, int d, __nv_bfloat16* ac, __nv_bfloat16* ac_lo, float* ssc, int ssc_ld,
                               int32_t* crow) {
  __shared__ int s_m;
  pdl_wait();
  pdl_trigger();
  const int j = blockIdx.x, b = j / (kBlockK / 2), r = j % (kBlockK / 2);
  if (threadIdx.x == 0) {
    int m = -1;
    for (int i = 0, cnt = 0; i < kBlockK; ++i)
      if (commit[b * kBlockK + i] == 0) {
        if (cnt == r) m = b * kBlockK + i;
        ++cnt;
      }
    s_m = m;
    crow[j] = m;
  }
  __syncthreads();
  const int m = s_m;  // exactly K/2 rows of every sequence are uncommitted
  const long long src = static_cast<long long>(m) * d, dst = static_cast<long long>(j) * d;
  for (int e = threadIdx.x; e < d / 8; e += blockDim.x) {
    const uint4 zero = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(ac + dst)[e] = m >= 0 ? reinterpret_cast<const uint4*>(a + src)[e] : zero;
    reinterpret_cast<uint4*>(ac_lo + dst)[e] = m >= 0 ? reinterpret_cast<const uint4*>(a_lo + src)[e] : zero;
  }
  for (int t = threadIdx.x; t < d_tiles; t += blockDim.x)
    ssc[static_cast<long long>(t) * ssc_ld + j] = m >= 0 ? ss[static_cast<long long>(t) * ss_ld + m] : 0.f;
}

// S = 2: commit the K/2 most confident positions of each block (ties to the
// lower position).  One warp per sequence.
__global__ void k_commit(const float* __restrict__ conf1, int32_t* commit, int B) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  const float c = lane < kBlockK ? conf1[b * kBlockK + lane] : -INFINITY;
  int rank = 0;
  for (int j = 0; j < kBlockK; ++j) {
    const float cj = __shfl_sync(0xffffffffu, c, j);
    if (cj > c || (cj == c && j < lane)) ++rank;
  }
  if (lane < kBlockK) commit[b * kBlockK + lane] = rank < kBlockK / 2 ? 1 : 0;
}

// ------------------------------------------------------------ launchers

#define DFLASH_DISPATCH(c, ...)                       \
  do {                                                \
    if ((c)->cfg.dtype != DFLASH_F32) {               \
      using T = __nv_bfloat16;                        \
      __VA_ARGS__;                                    \
    } else {                                          \
      using T = float;                                \
      __VA_ARGS__;                                    \
    }                                                 \
  } while (0)

template <typename T>
static ActOut<T> act_out(void* hi, void* lo) {
  return ActOut<T>{static_cast<T*>(hi), static_cast<T*>(lo)};
}

cudaError_t launch_gather_rows(dflash_ctx* c, const void* feats, int rows, cudaStream_t s) {
  const int F = c->cfg.n_taps * c->cfg.tap_width;
  DFLASH_DISPATCH(c, return launch_k(k_gather_rows<T>, dim3(rows), dim3(128), 0, s, dim3(1), c->pdl,
                                     static_cast<const T*>(feats), static_cast<T*>(c->fc_in), c->scal, c->row_src,
                                     F));
}

cudaError_t launch_embed(dflash_ctx* c, int M, bool second_pass, int32_t* order, cudaStream_t s) {
  const auto& g = c->cfg;
  const int n_tiles = (g.hidden + 127) / 128, per = M >= 512 ? n_tiles : 4;
  const dim3 grid((n_tiles + per - 1) / per, M);
  DFLASH_DISPATCH(c, return launch_k(k_embed<T>, grid, dim3(128), 0, s, dim3(1), c->pdl,
                                     static_cast<const T*>(c->embed), static_cast<const T*>(c->g_in[0]), c->x,
                                     act_out<T>(c->a, c->a_lo), c->ss_x, g.max_batch * kBlockK, g.hidden,
                                     g.mask_id, g.vocab, second_pass ? c->commit : nullptr, c->tok1, c->status,
                                     c->seq_len, order, M / kBlockK, per));
}

cudaError_t launch_logits_tiles(dflash_ctx* c, int M, float* user_logits, const int32_t* skip, const EpiArgs& norm,
                                cudaStream_t s) {
  dim3 grid(c->lm.n_tiles, M);
  k_logits_tiles<<<grid, kTileN, 0, s>>>(c->logits_ws, c->cfg.vocab, c->lm, user_logits, skip, norm);
  return cudaGetLastError();
}

cudaError_t launch_lm_merge(dflash_ctx* c, int M, const int32_t* commit, int32_t* tok_out, float* conf_out,
                            cudaStream_t s, bool compact) {
  return launch_k(k_lm_merge, dim3(M), dim3(256), 0, s, dim3(1), c->pdl, c->lm, M, commit, c->tok1, c->conf1,
                  tok_out, conf_out, compact ? 1 : 0);
}

cudaError_t launch_compact_rows(dflash_ctx* c, int B, int Mmax, cudaStream_t s) {
  const int d = c->cfg.hidden, d_tiles = (d + kTileN - 1) / kTileN;
  return launch_k(k_compact_rows, dim3(B * kBlockK / 2), dim3(128), 0, s, dim3(1), c->pdl, c->commit,
                  static_cast<const __nv_bfloat16*>(c->a), static_cast<const __nv_bfloat16*>(c->a_lo), c->ss_x, Mmax,
                  d_tiles, d, static_cast<__nv_bfloat16*>(c->ac), static_cast<__nv_bfloat16*>(c->ac_lo), c->ss_c,
                  c->cfg.max_batch * kBlockK / 2, c->crow);
}

cudaError_t launch_commit(dflash_ctx* c, int B, cudaStream_t s) {
  return launch_k(k_commit, dim3((B + 3) / 4), dim3(128), 0, s, dim3(1), c->pdl, c->conf1, c->commit, B);
}

}  // namespace dflash

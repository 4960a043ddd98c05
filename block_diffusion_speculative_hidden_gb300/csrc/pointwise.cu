// Row-wise kernels around the GEMMs: split-K reduction fused with the
// operation that follows each projection (RMSNorm, RoPE + paged KV write,
// residual add, SwiGLU), the block input embedding, and the LM-head argmax
// merge and S = 2 commit.
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

// Sum of `splits` fp32 partial planes at element e.
__device__ __forceinline__ float sum_splits(const float* __restrict__ part, long long plane, int splits, long long e) {
  float v = part[e];
  for (int s = 1; s < splits; ++s) v += part[s * plane + e];
  return v;
}

// ------------------------------------------------------------ inject side

// Copy the valid feature rows into a compact [rows][F] buffer (rows ordered
// by sequence, then position).
template <typename T>
__global__ void k_gather_rows(const T* __restrict__ feats, T* __restrict__ out, const int* scal,
                              const int32_t* row_src, int F) {
  const int r = blockIdx.x;
  if (r >= scal[0]) return;
  const long long src = row_src[r];
  const int4* s = reinterpret_cast<const int4*>(feats + src * F);
  int4* d = reinterpret_cast<int4*>(out + static_cast<long long>(r) * F);
  const int n16 = F * static_cast<int>(sizeof(T)) / 16;
  for (int i = threadIdx.x; i < n16; i += blockDim.x) d[i] = s[i];
}

// h[r] = RMSNorm(sum of FC partials)[r] * g_fc
template <typename T>
__global__ void k_fc_norm(const float* __restrict__ part, long long plane, int splits, const T* __restrict__ gain,
                          ActOut<T> h, const int* scal, int d, float eps) {
  extern __shared__ float sbuf[];  // [d] + 32
  const int r = blockIdx.x;
  if (r >= scal[0]) return;
  float ss = 0.f;
  for (int n = threadIdx.x; n < d; n += blockDim.x) {
    const float u = sum_splits(part, plane, splits, static_cast<long long>(r) * d + n);
    sbuf[n] = u;
    ss += u * u;
  }
  ss = block_sum(ss, sbuf + d);
  const float inv = rsqrtf(ss / d + eps);
  for (int n = threadIdx.x; n < d; n += blockDim.x)
    h.put(static_cast<long long>(r) * d + n, sbuf[n] * inv * to_f32(gain[n]));
}

// Injected K (RoPE at the row's absolute position, optional pre-RoPE offset)
// and V of every layer, written into the row's page slot (fp32 pool).
// GEMM output columns: layer l -> [l*2*kvd, +kvd) keys, [+kvd, +2kvd) values.
__global__ void k_inject_kv(const float* __restrict__ part, long long plane, int splits, const int* scal,
                            const int32_t* __restrict__ row_seq, const int32_t* __restrict__ row_pos,
                            const int32_t* __restrict__ page_table, int max_pages, const float* __restrict__ rcos,
                            const float* __restrict__ rsin, const float* __restrict__ key_offset, float* pool_k,
                            float* pool_v, int L, int P, int Hkv, int dh) {
  const int r = blockIdx.x;
  if (r >= scal[0]) return;
  const int b = row_seq[r], pos = row_pos[r];
  const int page = page_table[b * max_pages + pos / kPage], slot = pos % kPage;
  const int kvd = Hkv * dh, half = dh / 2, ncol = 2 * L * kvd;
  const long long rowbase = static_cast<long long>(r) * ncol;
  // keys: one thread per rotated pair (l, head, i)
  for (int t = threadIdx.x; t < L * Hkv * half; t += blockDim.x) {
    const int i = t % half, hl = t / half, hh = hl % Hkv, l = hl / Hkv;
    const int c0 = l * 2 * kvd + hh * dh + i;
    float x1 = sum_splits(part, plane, splits, rowbase + c0);
    float x2 = sum_splits(part, plane, splits, rowbase + c0 + half);
    if (key_offset != nullptr) {
      x1 += key_offset[(l * Hkv + hh) * dh + i];
      x2 += key_offset[(l * Hkv + hh) * dh + i + half];
    }
    const float cs = rcos[pos * half + i], sn = rsin[pos * half + i];
    const long long o = ((static_cast<long long>(l) * P + page) * Hkv + hh) * (kPage * dh) + slot * dh + i;
    pool_k[o] = x1 * cs - x2 * sn;
    pool_k[o + half] = x2 * cs + x1 * sn;
  }
  // values
  for (int t = threadIdx.x; t < L * kvd; t += blockDim.x) {
    const int dd = t % dh, hl = t / dh, hh = hl % Hkv, l = hl / Hkv;
    const float v = sum_splits(part, plane, splits, rowbase + l * 2 * kvd + kvd + hh * dh + dd);
    const long long o = ((static_cast<long long>(l) * P + page) * Hkv + hh) * (kPage * dh) + slot * dh + dd;
    pool_v[o] = v;
  }
}

// ------------------------------------------------------------ draft side

// Block input: x[m] = E[token] (token = [MASK], or in pass 2 the committed
// pass-1 token), a[m] = RMSNorm(x[m]) * g_in of layer 0.
template <typename T>
__global__ void k_embed_norm(const T* __restrict__ embed, const T* __restrict__ gain, float* __restrict__ x,
                             ActOut<T> a, int d, int mask_id, int vocab, const int32_t* commit,
                             const int32_t* tok1, int* status, float eps) {
  __shared__ float red[32];
  const int m = blockIdx.x;
  int tok = mask_id;
  if (commit != nullptr && commit[m] != 0) tok = tok1[m];
  if (tok < 0 || tok >= vocab) {
    if (threadIdx.x == 0) atomicOr(status, ST_BAD_TOKEN);
    tok = mask_id;
  }
  float ss = 0.f;
  for (int n = threadIdx.x; n < d; n += blockDim.x) {
    const float v = to_f32(embed[static_cast<long long>(tok) * d + n]);
    x[static_cast<long long>(m) * d + n] = v;
    ss += v * v;
  }
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / d + eps);
  for (int n = threadIdx.x; n < d; n += blockDim.x) {
    const long long e = static_cast<long long>(m) * d + n;
    a.put(e, x[e] * inv * to_f32(gain[n]));
  }
}

// Reduce the QKV partials, rotate q and k at the block position
// seq_len[b] + i, and store q, k_blk, v_blk (fp32).
__global__ void k_qkv_rope(const float* __restrict__ part, long long plane, int splits, const int32_t* seq_len,
                           const float* __restrict__ rcos, const float* __restrict__ rsin, float* q, float* kb,
                           float* vb, int Hq, int Hkv, int dh) {
  const int m = blockIdx.x;
  const int b = m / kBlockK, i = m % kBlockK;
  const int pos = seq_len[b] + i;
  const int half = dh / 2, qd = Hq * dh, kvd = Hkv * dh, ncol = qd + 2 * kvd;
  const long long rowbase = static_cast<long long>(m) * ncol;
  for (int t = threadIdx.x; t < (Hq + Hkv) * half; t += blockDim.x) {
    const int j = t % half, h = t / half;
    const int c0 = h * dh + j;  // q heads, then k heads, contiguous
    const float x1 = sum_splits(part, plane, splits, rowbase + c0);
    const float x2 = sum_splits(part, plane, splits, rowbase + c0 + half);
    const float cs = rcos[pos * half + j], sn = rsin[pos * half + j];
    const float y1 = x1 * cs - x2 * sn, y2 = x2 * cs + x1 * sn;
    if (h < Hq) {
      q[static_cast<long long>(m) * qd + c0] = y1;
      q[static_cast<long long>(m) * qd + c0 + half] = y2;
    } else {
      const int kc = c0 - qd;
      kb[static_cast<long long>(m) * kvd + kc] = y1;
      kb[static_cast<long long>(m) * kvd + kc + half] = y2;
    }
  }
  for (int t = threadIdx.x; t < kvd; t += blockDim.x)
    vb[static_cast<long long>(m) * kvd + t] = sum_splits(part, plane, splits, rowbase + qd + kvd + t);
}

// x[m] += sum of partials; a[m] = RMSNorm(x[m]) * gain
template <typename T>
__global__ void k_residual_norm(const float* __restrict__ part, long long plane, int splits, float* __restrict__ x,
                                ActOut<T> a, const T* __restrict__ gain, int d, float eps) {
  __shared__ float red[32];
  const int m = blockIdx.x;
  float ss = 0.f;
  for (int n = threadIdx.x; n < d; n += blockDim.x) {
    const long long e = static_cast<long long>(m) * d + n;
    const float v = x[e] + sum_splits(part, plane, splits, e);
    x[e] = v;
    ss += v * v;
  }
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / d + eps);
  for (int n = threadIdx.x; n < d; n += blockDim.x) {
    const long long e = static_cast<long long>(m) * d + n;
    a.put(e, x[e] * inv * to_f32(gain[n]));
  }
}

// act[m][f] = silu(gate) * up, gate = columns [0, F), up = [F, 2F)
template <typename T>
__global__ void k_swiglu(const float* __restrict__ part, long long plane, int splits, ActOut<T> act, int F,
                         int M) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= static_cast<long long>(M) * F) return;
  const long long m = t / F, f = t % F;
  const float g = sum_splits(part, plane, splits, m * 2 * F + f);
  const float u = sum_splits(part, plane, splits, m * 2 * F + F + f);
  act.put(t, g / (1.f + expf(-g)) * u);
}

// fp32 path: per (row, 128-column tile) max / argmax / sum-exp of the logits,
// same format as the tensor-core LM-head epilogue; optional copy-out.
__global__ void k_logits_tiles(const float* __restrict__ z, int V, LmPartials lm, float* user, const int32_t* skip) {
  __shared__ float smx[4];
  __shared__ int sidx[4];
  __shared__ float sse[4];
  const int m = blockIdx.y, tile = blockIdx.x;
  const int n = tile * kTileN + threadIdx.x;  // blockDim = 128
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool nv = n < V;
  const float val = nv ? z[static_cast<long long>(m) * V + n] : -INFINITY;
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

// One warp per row: merge the tile partials into (argmax, confidence).
// Confidence = max softmax probability = exp(max - LSE) = 1 / sum exp(z - max).
// With `commit`, committed rows keep tok1/conf1 and only the others are merged.
__global__ void k_lm_merge(LmPartials lm, int M, const int32_t* commit, const int32_t* tok1, const float* conf1,
                           int32_t* tok_out, float* conf_out) {
  const int m = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (m >= M) return;
  if (commit != nullptr && commit[m] != 0) {
    if (lane == 0) {
      tok_out[m] = tok1[m];
      if (conf_out != nullptr) conf_out[m] = conf1[m];
    }
    return;
  }
  const long long base = static_cast<long long>(m) * lm.n_tiles;
  float mx = -INFINITY, se = 0.f;
  int ix = 0x7fffffff;
  for (int t = lane; t < lm.n_tiles; t += 32) {  // tiles in increasing column order
    const float tm = lm.mx[base + t], ts = lm.se[base + t];
    const int ti = lm.idx[base + t];
    if (tm > mx) {
      se = se * expf(mx - tm) + ts;
      mx = tm;
      ix = ti;
    } else {
      se += ts * expf(tm - mx);
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, mx, o);
    const float os = __shfl_xor_sync(0xffffffffu, se, o);
    const int oi = __shfl_xor_sync(0xffffffffu, ix, o);
    const float nm = fmaxf(mx, om);
    const float ns = (mx > -INFINITY ? se * expf(mx - nm) : 0.f) + (om > -INFINITY ? os * expf(om - nm) : 0.f);
    if (om > mx || (om == mx && oi < ix)) ix = oi;
    mx = nm;
    se = ns;
  }
  if (lane == 0) {
    tok_out[m] = ix;
    if (conf_out != nullptr) conf_out[m] = 1.f / se;
  }
}

// S = 2: commit the K/2 most confident positions of each block (ties to the
// lower position).  One warp per sequence.
__global__ void k_commit(const float* __restrict__ conf1, int32_t* commit, int B) {
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

#define DFLASH_DISPATCH(c, KERNEL_CALL)               \
  do {                                                \
    if ((c)->cfg.dtype == DFLASH_BF16) {              \
      using T = __nv_bfloat16;                        \
      KERNEL_CALL;                                    \
    } else {                                          \
      using T = float;                                \
      KERNEL_CALL;                                    \
    }                                                 \
  } while (0)

static long long part_plane(int rows, int cols) { return static_cast<long long>(rows) * cols; }

template <typename T>
static ActOut<T> act_out(void* hi, void* lo) {
  return ActOut<T>{static_cast<T*>(hi), static_cast<T*>(lo)};
}

cudaError_t launch_gather_rows(dflash_ctx* c, const void* feats, int rows, int max_rows, int first_seq,
                               cudaStream_t s) {
  (void)max_rows;
  (void)first_seq;
  const int F = c->cfg.n_taps * c->cfg.tap_width;
  DFLASH_DISPATCH(c, (k_gather_rows<T><<<rows, 128, 0, s>>>(static_cast<const T*>(feats), static_cast<T*>(c->fc_in),
                                                            c->scal, c->row_src, F)));
  return cudaGetLastError();
}

cudaError_t launch_fc_norm(dflash_ctx* c, int rows, int splits, cudaStream_t s) {
  const int d = c->cfg.hidden;
  const size_t smem = sizeof(float) * (d + 32);
  DFLASH_DISPATCH(c, (k_fc_norm<T><<<rows, 256, smem, s>>>(c->part, part_plane(rows, d), splits,
                                                           static_cast<const T*>(c->g_fc),
                                                           act_out<T>(c->h_fused, c->h_lo), c->scal, d,
                                                           c->cfg.rms_eps)));
  return cudaGetLastError();
}

cudaError_t launch_inject_kv(dflash_ctx* c, int rows, int splits, cudaStream_t s) {
  const auto& g = c->cfg;
  const int ncol = 2 * g.n_layers * g.n_kv_heads * g.head_dim;
  k_inject_kv<<<rows, 256, 0, s>>>(c->part, part_plane(rows, ncol), splits, c->scal, c->row_seq, c->row_pos,
                                   c->page_table, g.max_pages_per_seq, c->rope_cos, c->rope_sin, c->key_offset,
                                   static_cast<float*>(c->pool_k), static_cast<float*>(c->pool_v), g.n_layers,
                                   g.n_pages, g.n_kv_heads, g.head_dim);
  return cudaGetLastError();
}

cudaError_t launch_embed_norm(dflash_ctx* c, int M, bool second_pass, cudaStream_t s) {
  const auto& g = c->cfg;
  DFLASH_DISPATCH(c, (k_embed_norm<T><<<M, 256, 0, s>>>(static_cast<const T*>(c->embed),
                                                        static_cast<const T*>(c->g_in[0]), c->x,
                                                        act_out<T>(c->a, c->a_lo), g.hidden, g.mask_id, g.vocab,
                                                        second_pass ? c->commit : nullptr, c->tok1, c->status,
                                                        g.rms_eps)));
  return cudaGetLastError();
}

cudaError_t launch_qkv_rope(dflash_ctx* c, int M, int splits, cudaStream_t s) {
  const auto& g = c->cfg;
  const int ncol = (g.n_q_heads + 2 * g.n_kv_heads) * g.head_dim;
  k_qkv_rope<<<M, 256, 0, s>>>(c->part, part_plane(M, ncol), splits, c->seq_len, c->rope_cos, c->rope_sin, c->q,
                               c->kblk, c->vblk, g.n_q_heads, g.n_kv_heads, g.head_dim);
  return cudaGetLastError();
}

cudaError_t launch_residual_norm(dflash_ctx* c, int M, int splits, const void* gain, cudaStream_t s) {
  const int d = c->cfg.hidden;
  DFLASH_DISPATCH(c, (k_residual_norm<T><<<M, 256, 0, s>>>(c->part, part_plane(M, d), splits, c->x,
                                                           act_out<T>(c->a, c->a_lo), static_cast<const T*>(gain),
                                                           d, c->cfg.rms_eps)));
  return cudaGetLastError();
}

cudaError_t launch_swiglu(dflash_ctx* c, int M, int splits, cudaStream_t s) {
  const int F = c->cfg.ffn;
  const long long n = static_cast<long long>(M) * F;
  const int blocks = static_cast<int>((n + 255) / 256);
  DFLASH_DISPATCH(c, (k_swiglu<T><<<blocks, 256, 0, s>>>(c->part, part_plane(M, 2 * F), splits,
                                                         act_out<T>(c->act, c->act_lo), F, M)));
  return cudaGetLastError();
}

cudaError_t launch_logits_tiles(dflash_ctx* c, int M, float* user_logits, const int32_t* skip, cudaStream_t s) {
  dim3 grid(c->lm.n_tiles, M);
  k_logits_tiles<<<grid, kTileN, 0, s>>>(c->logits_ws, c->cfg.vocab, c->lm, user_logits, skip);
  return cudaGetLastError();
}

cudaError_t launch_lm_merge(dflash_ctx* c, int M, const int32_t* commit, int32_t* tok_out, float* conf_out,
                            cudaStream_t s) {
  k_lm_merge<<<(M + 3) / 4, 128, 0, s>>>(c->lm, M, commit, c->tok1, c->conf1, tok_out, conf_out);
  return cudaGetLastError();
}

cudaError_t launch_commit(dflash_ctx* c, int B, cudaStream_t s) {
  k_commit<<<(B + 3) / 4, 128, 0, s>>>(c->conf1, c->commit, B);
  return cudaGetLastError();
}

}  // namespace dflash

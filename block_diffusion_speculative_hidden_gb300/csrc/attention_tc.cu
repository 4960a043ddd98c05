// Block attention on tensor cores for the fp16 KV pool (bf16 workloads).
//
// Same contraction as attention.cu (the K block queries of one sequence
// attend, unmasked, to every injected context key and to all K block keys;
// DFlash Guide: bidirectional attention across the masked block; stable-lab
// chapter: positions see their neighbours' [MASK] placeholders), laid out
// for HBM speed:
//   - one CTA per (sequence, kv head, key split); one warp per query head of
//     the group (16 block rows each) plus one producer warp;
//   - the producer streams the sequence's pages (16 keys x head dim, fp16)
//     with 4-D TMA tiled loads (128-byte swizzle) into a STAGES-deep ring
//     guarded by mbarriers, the block's own keys coming last from the
//     sequence's block page;
//   - S = Q K^T and O += P V run as m16n8k16 fp16 MMAs with fp32
//     accumulation; the online softmax stays in registers (P is re-packed
//     from the S accumulators, V is read transposed by ldmatrix);
//   - with several splits, the splits of one (sequence, kv head) form a
//     thread-block cluster: each keeps its unnormalised (o, m, l) in shared
//     memory and, after a cluster barrier, merges a slice of the rows over
//     every split through distributed shared memory (split order).
// The kernel is HBM-bound (about 64-128 flop per K/V byte); the legacy MMA
// rate is ample for that intensity.
#include <algorithm>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.cuh"

namespace dflash {

namespace {

constexpr int kPPS = 2;        // pages per pipeline stage (32 keys)
constexpr int kStages = 4;
constexpr int kMaxSplits = 16;  // splits merged in one cluster (16 needs the non-portable size)

template <int DH, int G>
struct TcAttnCfg {
  static constexpr int NBOX = DH / 64;                          // 64-wide (128 B) boxes per row
  static constexpr int PAGE_BYTES = kPage * DH * 2;             // one (page, head) slab
  static constexpr int STAGE_BYTES = 2 * kPPS * PAGE_BYTES;     // K then V
  static constexpr int QROW = DH + 8;                           // padded q row (halves)
  static constexpr int Q_BYTES = G * 16 * QROW * 2;
  static constexpr int THREADS = (G + 1) * 32;
  static constexpr int ML_BYTES = G * 16 * 2 * 4;                // per-row (m, l) for the split merge
  static constexpr int SMEM_FIXED = 1024 + kStages * STAGE_BYTES + Q_BYTES + ML_BYTES + 256;  // + page ids
  static_assert(G * 16 * DH * 4 <= kStages * STAGE_BYTES, "the split partial must fit in the ring");
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                            int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

// Byte offset, inside one (page, head) slab as TMA lays it out (boxes of 16
// rows x 128 bytes, 128-byte swizzle), of key row r and the 8 halves that
// start at column d (d a multiple of 8).
__device__ __forceinline__ uint32_t slab_off(int r, int d) {
  const int box = d >> 6, chunk = (d & 63) >> 3;
  return static_cast<uint32_t>(((box * 16 + r) << 7) + ((chunk ^ (r & 7)) << 4));
}

struct TcAttnParams {
  const __half* q;            // [B*16][Hq*DH]
  const int32_t* page_table;
  const int32_t* seq_len;
  int max_pages, block_page0, pool_pages, layer;
  int Hkv, splits;
  int page_slots;             // capacity of the shared-memory page-id list
  float scale_log2;           // log2(e) / sqrt(dh)
  void* o_hi;                 // ActOut<bf16> of the attention output [B*16][Hq*DH]
  void* o_lo;
  int* status;
};

template <int DH, int G>
__global__ void __launch_bounds__((G + 1) * 32) k_attn_tc(const __grid_constant__ CUtensorMap tmK,
                                                          const __grid_constant__ CUtensorMap tmV,
                                                          const TcAttnParams p) {
  using C = TcAttnCfg<DH, G>;
  constexpr int R = G * 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;                                   // [kStages][K pages | V pages]
  __half* sQ = reinterpret_cast<__half*>(smem + kStages * C::STAGE_BYTES);
  float* sML = reinterpret_cast<float*>(smem + kStages * C::STAGE_BYTES + C::Q_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * C::STAGE_BYTES + C::Q_BYTES + C::ML_BYTES);
  uint64_t* empty = full + kStages;
  int* s_pages = reinterpret_cast<int*>(empty + kStages);  // this split's page ids, staged once

  const int sp = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.seq_len[b];
  const int n_ctx_pages = (T + kPage - 1) / kPage;
  const int n_pages = n_ctx_pages + 1;                    // + the block page
  const int per_split = (n_pages + p.splits - 1) / p.splits;
  const int vp_begin = min(n_pages, sp * per_split), vp_end = min(n_pages, vp_begin + per_split);
  const int n_st = (vp_end - vp_begin + kPPS - 1) / kPPS;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], G);
    }
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  __syncthreads();  // barriers initialised; from here each warp stages only what it uses itself
  if (warp == G) {
    // page id of every virtual page of this split (context pages, then the block
    // page; 0 past the end), so that issuing a stage never waits on a global load
    for (int j = lane; j < n_st * kPPS && j < p.page_slots; j += 32) {
      const int vp = vp_begin + j;
      s_pages[j] = vp >= vp_end ? 0 : vp < n_ctx_pages ? p.page_table[b * p.max_pages + vp] : p.block_page0 + b;
    }
  } else {
    // this warp's 16 block queries: query head kvh*G + warp, block positions 0..15
    const int qd = p.Hkv * G * DH;
    for (int e = lane; e < 16 * (DH / 8); e += 32) {
      const int i = e / (DH / 8), c8 = e % (DH / 8);
      const int4 v = *reinterpret_cast<const int4*>(p.q + static_cast<long long>(b * kBlockK + i) * qd +
                                                    (kvh * G + warp) * DH + c8 * 8);
      *reinterpret_cast<int4*>(sQ + (warp * 16 + i) * C::QROW + c8 * 8) = v;
    }
  }
  __syncwarp();

  float o[DH / 8][4];
#pragma unroll
  for (int i = 0; i < DH / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
  const int g = lane >> 2, t4 = lane & 3;

  if (warp == G) {
    // ---------------- producer
    if (lane == 0) {
      int issued = 0;
      const int l_off = p.layer * p.pool_pages;
      for (int st = 0; st < n_st; ++st) {
        const int s = st % kStages;
        if (!mbar_wait(&empty[s], ((st / kStages) & 1) ^ 1, p.status)) break;
        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
        uint8_t* kdst = ring + s * C::STAGE_BYTES;
        uint8_t* vdst = kdst + kPPS * C::PAGE_BYTES;
        for (int j = 0; j < kPPS; ++j) {
          // past this split's end: page 0 (finite data, fully masked)
          const int page = s_pages[st * kPPS + j];
          for (int bx = 0; bx < C::NBOX; ++bx) {
            tma_load_4d(kdst + j * C::PAGE_BYTES + bx * 2048, &tmK, &full[s], bx * 64, 0, kvh, l_off + page);
            tma_load_4d(vdst + j * C::PAGE_BYTES + bx * 2048, &tmV, &full[s], bx * 64, 0, kvh, l_off + page);
          }
        }
        issued = st + 1;
      }
      // every copy this CTA issued must have landed before it exits (bounded)
      for (int st = max(0, issued - kStages); st < issued; ++st)
        mbar_wait(&full[st % kStages], (st / kStages) & 1, p.status);
    }
    __syncwarp();
  } else {
    // ---------------- consumers: warp gi = query head kvh*G + gi, rows = block positions
    const int gi = warp;
    uint32_t qf[DH / 16][4];
    {
      const __half* qw = sQ + gi * 16 * C::QROW;
      const int mat = lane >> 3, r8 = lane & 7;
#pragma unroll
      for (int ks = 0; ks < DH / 16; ++ks) {
        const int row = r8 + ((mat & 1) << 3), col = ks * 16 + ((mat >> 1) << 3);
        ldsm_x4(smem_u32(qw + row * C::QROW + col), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
      }
    }
    for (int st = 0; st < n_st; ++st) {
      const int s = st % kStages;
      if (!mbar_wait(&full[s], (st / kStages) & 1, p.status)) break;
      const uint32_t kbase = smem_u32(ring + s * C::STAGE_BYTES);
      const uint32_t vbase = kbase + kPPS * C::PAGE_BYTES;
      // S = Q K^T over 32 keys: n8 tiles 0..3 (two per page)
      float sacc[2 * kPPS][4];
#pragma unroll
      for (int i = 0; i < 2 * kPPS; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < DH / 16; ++ks) {
#pragma unroll
        for (int j = 0; j < kPPS; ++j) {
          // matrices: keys 0-7 / d 0-7, keys 0-7 / d 8-15, keys 8-15 / d 0-7, keys 8-15 / d 8-15
          const int mat = lane >> 3, r = (lane & 7) + ((mat >> 1) << 3), d = ks * 16 + ((mat & 1) << 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kbase + j * C::PAGE_BYTES + slab_off(r, d), b0, b1, b2, b3);
          mma_f16(sacc[2 * j], qf[ks], b0, b1);
          mma_f16(sacc[2 * j + 1], qf[ks], b2, b3);
        }
      }
      // mask (this split's keys only), scale, online softmax on rows g and g + 8
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 2 * kPPS; ++nt) {
        const int vp = vp_begin + st * kPPS + (nt >> 1);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int slot = ((nt & 1) << 3) + 2 * t4 + (e & 1);
          const bool valid =
              vp < vp_end && ((vp < n_ctx_pages && vp * kPage + slot < T) || vp == n_ctx_pages);
          const float v = valid ? sacc[nt][e] * p.scale_log2 : -INFINITY;
          sacc[nt][e] = v;
          mx[e >> 1] = fmaxf(mx[e >> 1], v);
        }
      }
      float alpha[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
        const float m_new = fmaxf(m_r[h], mx[h]);
        alpha[h] = m_r[h] == -INFINITY ? 0.f : exp2f(m_r[h] - m_new);
        m_r[h] = m_new;
      }
      float rs[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < 2 * kPPS; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = e >> 1;
          const float pe = m_r[h] == -INFINITY ? 0.f : exp2f(sacc[nt][e] - m_r[h]);
          sacc[nt][e] = pe;
          rs[h] += pe;
        }
      l_r[0] = l_r[0] * alpha[0] + rs[0];
      l_r[1] = l_r[1] * alpha[1] + rs[1];
#pragma unroll
      for (int i = 0; i < DH / 8; ++i) {
        o[i][0] *= alpha[0];
        o[i][1] *= alpha[0];
        o[i][2] *= alpha[1];
        o[i][3] *= alpha[1];
      }
      // O += P V: one k16 step per page
#pragma unroll
      for (int j = 0; j < kPPS; ++j) {
        uint32_t a[4];
        a[0] = pack_half2(sacc[2 * j][0], sacc[2 * j][1]);
        a[1] = pack_half2(sacc[2 * j][2], sacc[2 * j][3]);
        a[2] = pack_half2(sacc[2 * j + 1][0], sacc[2 * j + 1][1]);
        a[3] = pack_half2(sacc[2 * j + 1][2], sacc[2 * j + 1][3]);
#pragma unroll
        for (int dn = 0; dn < DH / 16; ++dn) {
          // matrices (transposed): keys 0-7 / d 0-7, keys 8-15 / d 0-7, keys 0-7 / d 8-15, keys 8-15 / d 8-15
          const int mat = lane >> 3, r = (lane & 7) + ((mat & 1) << 3), d = dn * 16 + ((mat >> 1) << 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vbase + j * C::PAGE_BYTES + slab_off(r, d), b0, b1, b2, b3);
          mma_f16(o[2 * dn], a, b0, b1);
          mma_f16(o[2 * dn + 1], a, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbarrier_arrive_one(&empty[s]);
    }
    // row sums over the quad
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_r[h] += __shfl_xor_sync(0xffffffffu, l_r[h], 1);
      l_r[h] += __shfl_xor_sync(0xffffffffu, l_r[h], 2);
    }
  }
  __syncthreads();  // the producer has drained; the ring is free
  const int Hq = p.Hkv * G, qd = Hq * DH;
  ActOut<__nv_bfloat16> out{static_cast<__nv_bfloat16*>(p.o_hi), static_cast<__nv_bfloat16*>(p.o_lo)};
  if (p.splits == 1) {
    if (warp < G) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = g + 8 * h;
        const float inv = l_r[h] > 0.f ? 1.f / l_r[h] : 0.f;
        const long long base = static_cast<long long>(b * kBlockK + i) * qd + (kvh * G + warp) * DH;
#pragma unroll
        for (int nt = 0; nt < DH / 8; ++nt) {
          out.put(base + nt * 8 + 2 * t4, o[nt][2 * h] * inv);
          out.put(base + nt * 8 + 2 * t4 + 1, o[nt][2 * h + 1] * inv);
        }
      }
    }
    return;
  }
  // ---------------- split merge inside the cluster (distributed shared memory)
  float* sO = reinterpret_cast<float*>(ring);  // [R][DH] unnormalised partial
  if (warp < G) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = warp * 16 + g + 8 * h;
#pragma unroll
      for (int nt = 0; nt < DH / 8; ++nt)
        *reinterpret_cast<float2*>(sO + r * DH + nt * 8 + 2 * t4) = make_float2(o[nt][2 * h], o[nt][2 * h + 1]);
      if (t4 == 0) {
        sML[2 * r] = m_r[h];
        sML[2 * r + 1] = l_r[h];
      }
    }
  }
  cluster_sync_all();
  {
    const int S = p.splits, cr = static_cast<int>(cluster_ctarank());
    const int rpr = (R + S - 1) / S, r0 = min(R, cr * rpr), r1 = min(R, r0 + rpr);
    const uint32_t sO_s = smem_u32(sO), sML_s = smem_u32(sML);
    for (int e = threadIdx.x; e < (r1 - r0) * (DH / 4); e += blockDim.x) {
      const int r = r0 + e / (DH / 4), d4 = (e % (DH / 4)) * 4;
      // every split's (m, l, o) of this row and 4 columns, loads issued back to back
      float ms[kMaxSplits], ls[kMaxSplits];
      float4 os[kMaxSplits];
#pragma unroll
      for (int s2 = 0; s2 < kMaxSplits; ++s2)
        if (s2 < S) {
          ms[s2] = ld_dsmem_f32(dsmem_map(sML_s + 8 * r, s2));
          ls[s2] = ld_dsmem_f32(dsmem_map(sML_s + 8 * r + 4, s2));
          os[s2] = ld_dsmem_f4(dsmem_map(sO_s + 4 * (r * DH + d4), s2));
        }
      float M = -INFINITY;
#pragma unroll
      for (int s2 = 0; s2 < kMaxSplits; ++s2)
        if (s2 < S) M = fmaxf(M, ms[s2]);
      float den = 0.f;
      float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int s2 = 0; s2 < kMaxSplits; ++s2)
        if (s2 < S && ms[s2] > -INFINITY) {
          const float w = exp2f(ms[s2] - M);
          den += w * ls[s2];
          num.x += w * os[s2].x;
          num.y += w * os[s2].y;
          num.z += w * os[s2].z;
          num.w += w * os[s2].w;
        }
      const float inv = den > 0.f ? 1.f / den : 0.f;
      const int gi = r >> 4, i = r & 15;
      const long long base = static_cast<long long>(b * kBlockK + i) * qd + (kvh * G + gi) * DH + d4;
      out.put(base + 0, num.x * inv);
      out.put(base + 1, num.y * inv);
      out.put(base + 2, num.z * inv);
      out.put(base + 3, num.w * inv);
    }
  }
  cluster_sync_all();  // every CTA's partial stays alive until all merges are done
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_attn() {
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
bool pool_map(const void* base, int dh, int Hkv, long long pages_total, CUtensorMap* out) {
  auto fn = encode_fn_attn();
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

template <int DH, int G>
cudaError_t launch_tc_t(dflash_ctx* c, int layer, int B, int splits, cudaStream_t s) {
  using C = TcAttnCfg<DH, G>;
  static int attr_smem = 0;
  static bool attr_np = false;
  if (!attr_np) {
    cudaError_t e = cudaFuncSetAttribute(k_attn_tc<DH, G>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    attr_np = true;
  }
  const auto& g = c->cfg;
  const int page_slots = g.max_pages_per_seq + 1 + kPPS;  // a split holds at most every page + the block page
  const int smem = C::SMEM_FIXED + 4 * page_slots;
  if (smem > attr_smem) {
    cudaError_t e = cudaFuncSetAttribute(k_attn_tc<DH, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_smem = smem;
  }
  const long long pages_total = static_cast<long long>(g.n_layers) * c->pool_pages;
  if (!c->attn_maps_ready) {
    if (!pool_map(c->pool_k, DH, g.n_kv_heads, pages_total, &c->attn_map_k) ||
        !pool_map(c->pool_v, DH, g.n_kv_heads, pages_total, &c->attn_map_v))
      return cudaErrorInvalidValue;
    c->attn_maps_ready = true;
  }
  TcAttnParams p;
  p.q = static_cast<const __half*>(c->q);
  p.page_table = c->page_table;
  p.seq_len = c->seq_len;
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
  dim3 grid(splits, g.n_kv_heads, B);
  if (splits == 1) {
    k_attn_tc<DH, G><<<grid, C::THREADS, smem, s>>>(c->attn_map_k, c->attn_map_v, p);
    return cudaGetLastError();
  }
  // the splits of one (sequence, kv head) form a cluster (at most 8: portable)
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = dim3(C::THREADS);
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = splits;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, k_attn_tc<DH, G>, c->attn_map_k, c->attn_map_v, p);
}

template <int DH>
cudaError_t launch_tc_dh(dflash_ctx* c, int layer, int B, int splits, cudaStream_t s) {
  switch (c->cfg.n_q_heads / c->cfg.n_kv_heads) {
    case 1: return launch_tc_t<DH, 1>(c, layer, B, splits, s);
    case 2: return launch_tc_t<DH, 2>(c, layer, B, splits, s);
    case 4: return launch_tc_t<DH, 4>(c, layer, B, splits, s);
    case 8: return launch_tc_t<DH, 8>(c, layer, B, splits, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// Largest cluster (= split count) the tensor-core attention may use here:
// 16 when the device can hold such clusters of this kernel, else the
// portable 8.  Queried once per context.
template <int DH, int G>
static int max_splits_t(dflash_ctx* c) {
  using C = TcAttnCfg<DH, G>;
  const int smem = C::SMEM_FIXED + 4 * (c->cfg.max_pages_per_seq + 1 + kPPS);
  if (cudaFuncSetAttribute(k_attn_tc<DH, G>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
      cudaFuncSetAttribute(k_attn_tc<DH, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return 8;
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(16, 1, 1);
  lc.blockDim = dim3(C::THREADS);
  lc.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 16;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_attn_tc<DH, G>, &lc) != cudaSuccess) {
    cudaGetLastError();
    return 8;
  }
  return n > 0 ? 16 : 8;
}

template <int DH>
static int max_splits_dh(dflash_ctx* c) {
  switch (c->cfg.n_q_heads / c->cfg.n_kv_heads) {
    case 1: return max_splits_t<DH, 1>(c);
    case 2: return max_splits_t<DH, 2>(c);
    case 4: return max_splits_t<DH, 4>(c);
    default: return max_splits_t<DH, 8>(c);
  }
}

int attention_tc_max_splits(dflash_ctx* c) {
  if (c->attn_tc_max_splits == 0)
    c->attn_tc_max_splits = c->cfg.head_dim == 128 ? max_splits_dh<128>(c) : max_splits_dh<64>(c);
  return c->attn_tc_max_splits;
}

cudaError_t launch_attention_tc(dflash_ctx* c, int layer, int B, int splits, cudaStream_t s) {
  switch (c->cfg.head_dim) {
    case 64: return launch_tc_dh<64>(c, layer, B, splits, s);
    case 128: return launch_tc_dh<128>(c, layer, B, splits, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dflash

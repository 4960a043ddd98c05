// Internal declarations shared by the libdflash translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "../../include/dflash.h"
#include "epilogue.cuh"

namespace dflash {

// A kernel attribute (the dynamic shared-memory limit, a cluster flag) is
// a property of the kernel on one device: it must be set on every device a
// kernel runs on, and calls may come from several host threads.  FuncAttr
// remembers, per device, the largest value set so far; ensure() sets it
// (through set(value)) only when a launch needs more.
struct FuncAttr {
  static constexpr int kMaxDevices = 64;
  std::mutex mu;
  int value[kMaxDevices] = {};
  template <class Set>
  cudaError_t ensure(int need, Set&& set) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (value[dev] >= need) return cudaSuccess;
    e = set(need);
    if (e == cudaSuccess) value[dev] = need;
    return e;
  }
};

constexpr int kTileN = 128;   // weight rows per GEMM tile (MMA M)
constexpr int kTileK = 64;    // reduction depth per pipeline stage (one 128-byte swizzle row)

// Per-row, per-128-column-tile reduction of logits: running max, its
// (lowest) column, and sum of exp(logit - max).
struct LmPartials {
  float* mx;
  float* se;
  int32_t* idx;
  int n_tiles;  // row stride of the three arrays
};

// The projection that follows a launch in the chain, for its L2 prefetch
// (W == nullptr: none).  budget_bytes bounds the bytes prefetched.
struct NextGemm {
  const void* W = nullptr;
  int N = 0, K = 0, M = 0;
  bool split = true;  // hi+lo activations
  int splits = 1;
  long long budget_bytes = 0;
};

struct GemmLaunch {
  // out[split][m][n] = sum_{k in split} X[m][k] * W[n][k]
  const void* W;  // [N][K]
  const void* X;  // [M_alloc][K]
  const void* X_lo;  // nullable: second bf16 term of X (x = hi + lo), same layout
  int N, K;
  int M;          // rows computed (host bound)
  int M_alloc;    // rows the X buffer holds
  int splits;
  float* out;
  long long split_stride;
  int ldo;
  const int* m_valid;  // nullable device row count; tiles at or past it exit
  EpiArgs epi;         // fused epilogue; EPI_NONE writes raw partial planes (no cluster)
  // LM-head epilogue (bf16 only): when lm.mx != nullptr the kernel reduces
  // each tile to LmPartials instead of writing `out`.
  LmPartials lm;
  float* logits;       // nullable: raw logits [M][ld_logits]
  long long ld_logits;
  const int* skip_rows;  // nullable: rows whose logits are not stored
  const int* logits_rows;  // nullable: row m's logits go to row logits_rows[m] (compacted rows)
  NextGemm next;         // the projection after this one (L2 prefetch of its weights)
  const float* w_scale;  // E4M3 weights (DFLASH_BF16_W8): fp32 scale of every weight row [N]
};

// Where block attention takes its sequences from: by default the context's
// page table and lengths, block b being sequence b; the training-time block
// attention passes a page-table row and a context length per block.
struct AttnSrc {
  const int32_t* row_of = nullptr;   // page-table row of block b (null: row b)
  const int32_t* seq_len = nullptr;  // context length of block b (null: the context's seq_len)
  bool pdl = true;                   // false: the immediate predecessor wrote row_of / seq_len
  // launch order: grid slot z serves block order[z] (null: block z); written
  // at least two kernels earlier, or by the immediate predecessor with pdl off
  const int32_t* order = nullptr;
};

struct TmapEntry {
  const void* ptr;
  int rows, cols, box_rows;
  int kind;  // 0 bf16, 1 E4M3 codes
  CUtensorMap map;
};

}  // namespace dflash

struct dflash_graph {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

struct dflash_ctx {
  dflash_config cfg;
  int elem;  // bytes per element of the config dtype
  int num_sms = 0;  // 0: unknown (the persistent projection kernel is not used)
  int pers_split_clusters = -1;  // cluster pairs of the split persistent kernel that fit at once (-1: not asked yet)
  // weights
  const void *w_fc, *g_fc, *embed, *g_final, *w_lm, *w_kv_inj;
  const float* key_offset;
  std::vector<const void*> w_qkv, w_o, w_gu, w_down, g_in, g_post;
  // DFLASH_BF16_W8: row scales of the E4M3 projection weights (else null)
  const float *s_fc = nullptr, *s_lm = nullptr, *s_kv_inj = nullptr;
  std::vector<const float*> s_qkv, s_o, s_gu, s_down;
  // cache
  void *pool_k, *pool_v;
  int32_t *page_table, *seq_len;
  // workspace carve-outs
  int* status;
  int* scal;  // [0] rows of the current inject, [1] free-list head, [2] free count
  int32_t *free_ring, *row_seq, *row_pos, *row_src;
  int32_t *blk_row, *blk_len;  // training-time block attention: page-table row and context length per block
  int32_t* attn_order;          // [max_batch] attention launch order, longest context first
  float *rope_cos, *rope_sin;
  int rope_rows;
  int pool_pages;  // pages per layer in the pool: n_pages context pages + max_batch block pages
  int kv_elem;     // bytes per KV-pool / q element: 2 (fp16) for bf16 workloads, 4 for fp32
  void *fc_in, *h_fused, *h_lo;
  float* y;        // fp32 projection output (FC output u; fp32-path staging)
  float* x;        // residual stream [M][d]
  void *a, *a_lo, *o, *o_lo, *act, *act_lo;  // GEMM inputs (lo: second bf16 term, bf16 only)
  void* q;         // block queries [M][Hq*dh] (KV element type)
  float *attn_o, *attn_ml;
  int attn_max_splits;
  bool attn_maps_ready = false;
  CUtensorMap attn_map_k, attn_map_v;  // 4-D maps over the fp16 pool
  CUtensorMap attn_map_q;              // 2-D map over the fp16 block queries
  int attn_fit[17] = {};               // resident clusters per split count (0: not queried, -1: none)
  dflash::LmPartials lm;
  float* logits_ws;  // fp32 mode: full logits [M][V]
  int32_t* tok1;
  float* conf1;
  int32_t* commit;
  std::vector<dflash::TmapEntry> tmaps;
  // launch the inject / draft / accept chain with programmatic dependent
  // launch (each kernel may start while its predecessor finishes)
  bool pdl = false;
  // folded RMSNorm: partial sums of squares, [ceil(hidden/128)][rows]
  float* ss_x;   // draft rows (row stride max_batch * 16)
  float* ss_h;   // inject rows (row stride max_inject_rows)
  // S = 2, second pass: the uncommitted rows compacted for the LM head
  // (bf16 family): [max_batch * K/2][hidden] twice, partial sums [ceil(hidden/128)][max_batch * K/2]
  void *ac = nullptr, *ac_lo = nullptr;
  float* ss_c = nullptr;
  int32_t* crow = nullptr;  // compact row -> block row ([max_batch * K/2])
  // persistent projections, split tail: a partial tile per CTA
  // [num_sms][128][128] fp32 and an arrival count per tail tile [num_sms]
  // (zero between launches); null where the persistent kernel never runs
  float* pers_ws = nullptr;
  int* pers_cnt = nullptr;
  // stream being recorded into a graph (dflash_graph_begin), else null
  cudaStream_t capture = nullptr;
  bool capturing = false;
  // launch timing (dflash_profile_enable)
  bool prof_on = false;
  struct ProfRec {
    cudaEvent_t a, b;
    int cls, launches;
  };
  std::vector<ProfRec> prof_live;
  std::vector<cudaEvent_t> prof_pool;
};

namespace dflash {

// Every kernel of the library runs with the largest shared-memory carveout:
// CTAs of different kernels share an SM only under the same carveout, and
// the chain relies on a kernel's CTAs starting beside its predecessor's.
// Returns false if the attribute could not be set.
bool prefer_max_smem(const void* kernel);

// Launches kernel k on stream s, as a grid of thread-block clusters when
// cluster has more than one CTA, and with programmatic stream serialisation
// (the kernel may start before its predecessor completes; it must follow
// the pdl_wait / pdl_trigger rule of common.cuh) when pdl is set.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, dim3 cluster,
                     bool pdl, Args&&... args) {
  if (!prefer_max_smem(reinterpret_cast<const void*>(k))) return cudaErrorInvalidValue;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  cudaLaunchAttribute at[2];
  int n = 0;
  if (cluster.x * cluster.y * cluster.z > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = cluster.x;
    at[n].val.clusterDim.y = cluster.y;
    at[n].val.clusterDim.z = cluster.z;
    ++n;
  }
  if (pdl) {
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  lc.attrs = at;
  lc.numAttrs = n;
  return cudaLaunchKernelEx(&lc, k, static_cast<Args&&>(args)...);
}

// gemm.cu
cudaError_t gemm_launch(dflash_ctx* c, const GemmLaunch& g, cudaStream_t s);
int gemm_kb(int K);
int gemm_bn(int M, bool split, bool w8 = false);
// The persistent projection kernel's plan for an M x N x K projection with
// hi + lo activations: CTAs per tile (1, or 2 splitting K), 0 where the
// kernel does not apply.  split_slots: cluster pairs that fit at once.
int pers_plan(int M, int N, int K, int num_sms, int split_slots, bool split_tail);
int gemm_kb_per_split(int n_kb, int splits, bool w8);
int gemm_normalize_splits(int n_kb, int splits, bool w8);
int gemm_blocks_per_sm(int bn, bool split, bool w8);
int gemm_ring_stages(int bn, bool split, bool w8);
// The L2 prefetch plan (and the weight tensor map) of projection `nx`.
bool gemm_l2_plan(dflash_ctx* c, const NextGemm& nx, L2Plan* plan, CUtensorMap* map);
int gemm_splits(int n_tiles, int n_kb, int bn, bool split, int num_sms, int max_ctas = 0, bool w8 = false);
// gemm_w8.cu: the E4M3-weight variants of the projection kernel
cudaError_t launch_tc_w8(dflash_ctx* c, const GemmLaunch& g, int bn, const CUtensorMap& tw, const CUtensorMap& tx,
                         const CUtensorMap& txlo, cudaStream_t s);
cudaError_t gemm_launch_uncached(int* status, const GemmLaunch& g, cudaStream_t s);

}  // namespace dflash

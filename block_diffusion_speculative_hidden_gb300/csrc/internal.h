// Internal declarations shared by the libdflash translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "../../include/dflash.h"
#include "epilogue.cuh"

namespace dflash {

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
};

struct TmapEntry {
  const void* ptr;
  int rows, cols, box_rows;
  CUtensorMap map;
};

}  // namespace dflash

struct dflash_ctx {
  dflash_config cfg;
  int elem;  // bytes per element of the config dtype
  int num_sms;
  // weights
  const void *w_fc, *g_fc, *embed, *g_final, *w_lm, *w_kv_inj;
  const float* key_offset;
  std::vector<const void*> w_qkv, w_o, w_gu, w_down, g_in, g_post;
  // cache
  void *pool_k, *pool_v;
  int32_t *page_table, *seq_len;
  // workspace carve-outs
  int* status;
  int* scal;  // [0] rows of the current inject, [1] free-list head, [2] free count
  int32_t *free_ring, *row_seq, *row_pos, *row_src;
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
  int attn_tc_max_splits = 0;  // 8 or 16, queried on first use
  CUtensorMap attn_map_k, attn_map_v;  // 4-D maps over the fp16 pool
  dflash::LmPartials lm;
  float* logits_ws;  // fp32 mode: full logits [M][V]
  int32_t* tok1;
  float* conf1;
  int32_t* commit;
  std::vector<dflash::TmapEntry> tmaps;
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

// gemm.cu
cudaError_t gemm_launch(dflash_ctx* c, const GemmLaunch& g, cudaStream_t s);
int gemm_kb(int K);
int gemm_bn(int M, bool split);
int gemm_max_clusters(int bn, bool split, int cluster);
int gemm_splits(int n_tiles, int n_kb, int bn, bool split);
cudaError_t gemm_launch_uncached(int* status, const GemmLaunch& g, cudaStream_t s);

}  // namespace dflash

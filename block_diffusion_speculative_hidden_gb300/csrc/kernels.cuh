// Launch interfaces of the non-GEMM kernels (defined in paging.cu,
// pointwise.cu, attention.cu and accept.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace dflash {

// paging.cu
cudaError_t launch_reset(dflash_ctx* c, cudaStream_t s);
cudaError_t launch_release(dflash_ctx* c, int b, cudaStream_t s);
cudaError_t launch_truncate(dflash_ctx* c, int b, int new_len, cudaStream_t s);
cudaError_t launch_alloc(dflash_ctx* c, const int32_t* n_rows, int first_seq, int B, int max_rows, cudaStream_t s);
cudaError_t launch_rope_table(dflash_ctx* c, cudaStream_t s);

// pointwise.cu (T = the config element type, chosen by c->cfg.dtype)
cudaError_t launch_gather_rows(dflash_ctx* c, const void* feats, int rows, cudaStream_t s);
// order (null: none): also writes the attention launch order of the M / 16 sequences
cudaError_t launch_embed(dflash_ctx* c, int M, bool second_pass, int32_t* order, cudaStream_t s);
cudaError_t launch_logits_tiles(dflash_ctx* c, int M, float* user_logits, const int32_t* skip, const EpiArgs& norm,
                                cudaStream_t s);
cudaError_t launch_lm_merge(dflash_ctx* c, int M, const int32_t* commit, int32_t* tok_out, float* conf_out,
                            cudaStream_t s, bool compact = false);
// S = 2, second pass: the uncommitted rows' LM-head inputs into c->ac / ac_lo / ss_c
cudaError_t launch_compact_rows(dflash_ctx* c, int B, int Mmax, cudaStream_t s);
cudaError_t launch_commit(dflash_ctx* c, int B, cudaStream_t s);

// attention.cu
int attn_splits(dflash_ctx* c, int B);
cudaError_t launch_attention(dflash_ctx* c, int layer, int B, int splits, cudaStream_t s, const NextGemm& next,
                             const AttnSrc& src = AttnSrc{});
// attention_mma.cu (fp16 pool, tcgen05)
// train_attn.cu
cudaError_t launch_block_attention(dflash_ctx* c, int layer, int NB, const int32_t* seq, const int32_t* ctx_len,
                                   const void* q, const void* k_blk, const void* v_blk, float* out, cudaStream_t s);
cudaError_t launch_attention_mma(dflash_ctx* c, int layer, int B, int splits, cudaStream_t s, const NextGemm& next,
                                 const AttnSrc& src = AttnSrc{});
int attention_mma_splits(dflash_ctx* c, int B);

// accept.cu
cudaError_t launch_accept_greedy(int B, int K, const int32_t* d, const int32_t* y, int32_t* tau, int32_t* emitted,
                                 int32_t* n_emit, bool pdl, cudaStream_t s);
cudaError_t launch_accept_stochastic(int B, int K, int V, const int32_t* d, const float* z, const float* q,
                                     float temperature, uint64_t seed, uint64_t round, int* round_ctr,
                                     int32_t* tau, int32_t* emitted, int32_t* n_emit, int num_sms, bool pdl,
                                     cudaStream_t s);

}  // namespace dflash

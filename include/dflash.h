/*
 * libdflash — GB300 (sm_103a) hot path of DFlash block-diffusion speculative
 * drafting: target-feature fusion and KV injection into a paged draft KV
 * cache, one parallel draft pass over a K = 16 masked block (S = 1 or 2), and
 * the lossless acceptance step.
 *
 * Sources of the operations (the method's pages):
 *   [Guide]  "DFlash Guide: Block Diffusion for Speculative Decoding"
 *            (aifetchly blog): "1. Single-Pass Block-Diffusion Drafting",
 *            "2. Target Hidden-State Conditioning", "3. Cross-Layer KV
 *            Injection", "The Cost Breakdown of Speculative Rounds".
 *   [Paper]  "DFlash: Block Diffusion for Flash Speculative Decoding"
 *            (arXiv 2602.06036 abstract page): Figure 2 (context features
 *            fused and injected into each draft layer's KV cache).
 *   [Chapter] "DFlash: Diffusion Drafts the Block" (stable-lab): "KV
 *            Injection", "The Model at a Glance", "The systems side: Spec V2",
 *            the [MASK]-neighbour paragraph after "Common misconception".
 *
 * Conventions for every call:
 *   - Pointers marked "device" are CUDA device memory owned by the caller
 *     (e.g. allocated with PyTorch); the library only borrows them.  The
 *     library allocates no device memory at all: scratch lives in the
 *     caller's workspace (dflash_workspace_size) and the KV pool in the
 *     caller's pool buffer (dflash_kv_pool_size).
 *   - Every call validates its host-side arguments first; on a host-side
 *     error it returns that error and enqueues nothing.
 *   - Work is enqueued on the given stream and returns without waiting.
 *     Errors found on the device (pool exhausted, bad token id, a bounded
 *     wait that gave up) set bits in a sticky device status word, and the
 *     affected call writes nothing further; read it with dflash_get_status.
 *   - A context is not thread-safe; use one context per stream.
 *   - Row-major everywhere; matrices are [out_features, in_features].
 *   - dtype DFLASH_BF16: weights and features are bf16 and every projection
 *     is a bf16 x bf16 tensor-core product with fp32 accumulation.  An
 *     activation that enters a projection is carried as an exact pair of
 *     bf16 terms (hi + lo, two MMAs), so it keeps about 16 significant bits;
 *     block queries and the KV pool are fp16; the residual stream, logits
 *     and confidences are fp32.  dtype DFLASH_F32: everything fp32 (SIMT
 *     kernels).
 */
#ifndef DFLASH_H_
#define DFLASH_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dflash_stream; /* same type as cudaStream_t; NULL = legacy default stream */
typedef struct dflash_ctx dflash_ctx;      /* opaque, owned by the library */

typedef enum {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARG = 1,       /* null pointer, bad count or size */
  DFLASH_ERR_UNSUPPORTED_SHAPE = 2, /* a shape the kernels do not handle */
  DFLASH_ERR_POOL_EXHAUSTED = 3,    /* (status word bit 1) */
  DFLASH_ERR_CUDA = 4,              /* a CUDA runtime call failed */
  DFLASH_ERR_STATE = 5,             /* the device status word is non-zero */
  DFLASH_ERR_WORKSPACE = 6,         /* workspace or pool buffer too small */
  DFLASH_ERR_TOO_LARGE = 7,         /* request exceeds the fixed scratch of dflash_gemm_bf16_noalloc */
  DFLASH_ERR_CAPTURE = 8            /* not allowed in the context's capture state (dflash_graph_begin) */
} dflash_status;

/* Bits of the device status word (dflash_get_status). */
#define DFLASH_DEV_POOL_EXHAUSTED 1 /* an inject needed more pages than were free */
#define DFLASH_DEV_SEQ_TOO_LONG 2   /* a sequence would exceed max_pages_per_seq */
#define DFLASH_DEV_WAIT_TIMEOUT 4   /* a bounded device wait gave up (2 s) */
#define DFLASH_DEV_BAD_TOKEN 8      /* a token id outside [0, vocab) */
#define DFLASH_DEV_BAD_ROWS 16      /* an n_rows entry outside [0, max_rows] */
#define DFLASH_DEV_BAD_BLOCK 32     /* dflash_block_attention: a block's sequence or prefix out of range */

/* DFLASH_BF16_W8: DFLASH_BF16 with FP8 projection weights.  Every projection
 * weight (w_fc, w_kv_inject, w_qkv, w_o, w_gu, w_down, w_lm) is one E4M3 code
 * per entry (OCP 8-bit floating point: 4 exponent bits, bias 7, 3 mantissa
 * bits; code S.1111.111 must not occur) and the matrix is
 * W = diag(s) . decode(codes) with one fp32 scale per row (the s_* arrays of
 * dflash_weights).  The codes are widened exactly to bf16 inside the
 * projection kernel, so the arithmetic is that of DFLASH_BF16 on W; only the
 * weight bytes read from HBM halve.  Features, the embedding, norm gains and
 * key_offset stay bf16 / fp32 as for DFLASH_BF16.  Row lengths of the
 * projections (hidden, ffn, n_q_heads*head_dim, n_taps*tap_width) must be
 * multiples of 16.  [Guide] "Production Benchmarks on NVIDIA Blackwell B200"
 * (FP4/FP8 mixed execution). */
typedef enum { DFLASH_F32 = 0, DFLASH_BF16 = 1, DFLASH_BF16_W8 = 2 } dflash_dtype;

typedef struct {
  int n_layers;          /* draft layers L */
  int hidden;            /* draft hidden size d */
  int n_q_heads;         /* Hq */
  int n_kv_heads;        /* Hkv; Hq % Hkv == 0, G = Hq / Hkv in {1, 2, 4, 8} */
  int head_dim;          /* dh in {64, 128} (DFLASH_BF16) or {32, 64, 128} (DFLASH_F32) */
  int ffn;               /* SwiGLU width F */
  int vocab;             /* V */
  int mask_id;           /* the [MASK] token id */
  int n_taps;            /* tapped target layers */
  int tap_width;         /* width of one tapped hidden state */
  int block_k;           /* K, must be 16 */
  int page_size;         /* tokens per KV page, must be 16 */
  int max_batch;         /* largest B of any call */
  int max_pages_per_seq; /* page-table row length */
  int n_pages;           /* pages in the pool */
  int max_rows;          /* largest per-sequence row count of one inject call */
  int max_inject_rows;   /* largest B * max_rows of one inject call */
  float rope_theta;      /* RoPE base */
  float rms_eps;         /* RMSNorm epsilon */
  int dtype;             /* dflash_dtype */
} dflash_config;

/* Device pointers to the drafter's weights, in the config dtype (key_offset
 * is fp32).  Pointer arrays (w_qkv ... g_post) are HOST arrays of n_layers
 * device pointers; the library copies them during dflash_create. */
typedef struct {
  const void* w_fc;    /* [hidden, n_taps*tap_width]  feature-fusion FC */
  const void* g_fc;    /* [hidden]  RMSNorm gain after the FC */
  const void* embed;   /* [vocab, hidden]  token embedding */
  const void* g_final; /* [hidden]  final RMSNorm gain */
  const void* w_lm;    /* [vocab, hidden]  LM head (untied) */
  const void* w_kv_inject; /* [n_layers*2*n_kv_heads*head_dim, hidden]: for layer l,
                              rows l*2*kvd .. +kvd are W_k^l, the next kvd rows W_v^l
                              (kvd = n_kv_heads*head_dim; same values as w_qkv's k/v rows) */
  const float* key_offset; /* optional [n_layers, n_kv_heads, head_dim] fp32 added to the
                              injected keys before RoPE (a workload knob; NULL = none) */
  const void* const* w_qkv;  /* per layer [Hq*dh + 2*kvd, hidden]: q rows, then k, then v */
  const void* const* w_o;    /* per layer [hidden, Hq*dh] */
  const void* const* w_gu;   /* per layer [128*ceil(ffn/64), hidden]: for each group of 64
                                features, its 64 gate rows then its 64 up rows; rows of
                                features past ffn are zero */
  const void* const* w_down; /* per layer [hidden, ffn] */
  const void* const* g_in;   /* per layer [hidden]  pre-attention RMSNorm gain */
  const void* const* g_post; /* per layer [hidden]  pre-MLP RMSNorm gain */
  /* DFLASH_BF16_W8 only (ignored otherwise): fp32 row scales of the E4M3
     projection weights above, one per row in the same row order (packed
     matrices: packed the same way; zero-padded rows may have any scale). */
  const float* s_fc;                /* [hidden] */
  const float* s_lm;                /* [vocab] */
  const float* s_kv_inject;         /* [n_layers*2*n_kv_heads*head_dim] */
  const float* const* s_qkv;        /* per layer [Hq*dh + 2*kvd] */
  const float* const* s_o;          /* per layer [hidden] */
  const float* const* s_gu;         /* per layer [128*ceil(ffn/64)] */
  const float* const* s_down;       /* per layer [hidden] */
} dflash_weights;

/* Bytes of caller-provided scratch the context needs; 0 on a bad config. */
size_t dflash_workspace_size(const dflash_config* cfg);

/* Bytes of the paged KV pool: K then V, each [n_layers][n_pages + max_batch]
 * [n_kv_heads][page_size][head_dim], fp16 (DFLASH_BF16) or fp32 (DFLASH_F32).
 * Pages n_pages + b hold sequence b's draft-block keys and values of the
 * current pass; pages 0..n_pages-1 the injected context.  [Guide] "3. Cross-Layer KV
 * Injection" ("Zero Redundant KV Caching"): the draft cache holds only the
 * injected target context, never the block's own keys. */
size_t dflash_kv_pool_size(const dflash_config* cfg);

/* Create a context.  kv_pool (device, >= dflash_kv_pool_size bytes),
 * page_table (device int32 [max_batch, max_pages_per_seq]), seq_len (device
 * int32 [max_batch]) and workspace (device, >= dflash_workspace_size bytes,
 * 256-byte aligned) stay owned by the caller and must outlive the context.
 * Synchronous: fills the RoPE table in the workspace and resets the cache
 * (every sequence empty, free list 0..n_pages-1, status 0).  Errors:
 * INVALID_ARG, UNSUPPORTED_SHAPE, WORKSPACE, CUDA. */
dflash_status dflash_create(const dflash_config* cfg, const dflash_weights* w, void* kv_pool,
                            size_t kv_pool_bytes, int32_t* page_table, int32_t* seq_len,
                            void* workspace, size_t workspace_bytes, dflash_ctx** out);

/* Free the host-side context.  Does not touch the caller's buffers. */
dflash_status dflash_destroy(dflash_ctx* ctx);

/* Empty every sequence, refill the free list 0..n_pages-1 and clear the
 * device status word (asynchronous on `stream`). */
dflash_status dflash_reset(dflash_ctx* ctx, dflash_stream stream);

/* Return sequence b's pages to the tail of the free list (in page-table
 * order) and set its length to 0 (asynchronous). */
dflash_status dflash_release(dflash_ctx* ctx, int b, dflash_stream stream);

/* Shorten sequence b to new_len tokens (asynchronous; no-op when the
 * sequence is not longer): its pages past ceil(new_len/16) return to the
 * tail of the free list in page-table order.  Used to drop context that a
 * caller no longer wants attended; accepted drafts never need it because
 * rejected drafts are never cached. */
dflash_status dflash_truncate(dflash_ctx* ctx, int b, int new_len, dflash_stream stream);

/* KV injection.  [Guide] "2. Target Hidden-State Conditioning" (H_cond =
 * W_proj H_T) and "3. Cross-Layer KV Injection" (K^(l) = W_K^(l) H_cond,
 * V^(l) = W_V^(l) H_cond); [Paper] Fig. 2; [Chapter] "KV Injection".
 *
 * For sequences b = first_seq .. first_seq+B-1 appends n_rows[b-first_seq]
 * (device int32, each in [0, max_rows]) rows of tapped target hidden states
 * at positions seq_len[b] ...: h = RMSNorm(feats . W_fc^T); for every layer
 * l the keys RoPE(h W_k^lT (+ key_offset)) at their absolute positions and
 * the values h W_v^lT are written into newly allocated pages.  Pages come
 * from a FIFO free list, sequences served in index order, each taking
 * ceil((len+n)/16) - ceil(len/16) pages; if the pool cannot hold all of
 * them the call sets DFLASH_DEV_POOL_EXHAUSTED and changes nothing.
 * feats: device [B, max_rows, n_taps*tap_width] in the config dtype, taps
 * concatenated in ascending layer order; rows past n_rows are ignored.
 * Requires max_rows <= cfg.max_rows and B*max_rows <= cfg.max_inject_rows.
 * No host synchronisation: after dflash_accept pass its n_emit as n_rows. */
dflash_status dflash_inject_kv(dflash_ctx* ctx, const void* feats, const int32_t* n_rows,
                               int first_seq, int B, int max_rows, dflash_stream stream);

/* One parallel draft of a K-token block for sequences 0..B-1 (B <=
 * max_batch).  [Guide] "1. Single-Pass Block-Diffusion Drafting" (x_hat =
 * argmax D_theta(m_{1:gamma} | x_{<t}, H_T), one forward pass); [Chapter]
 * "The Model at a Glance" (a fully masked block, S refinement passes
 * committing positions in confidence order) and the [MASK]-neighbour
 * paragraph (block positions see each other's [MASK] placeholders).
 *
 * The block holds K [MASK] embeddings at positions seq_len[b] .. +K-1 and
 * runs the pre-norm drafter (RMSNorm, QKV, RoPE, unmasked attention over the
 * injected context and the whole block, O-proj, SwiGLU MLP) then the final
 * RMSNorm and LM head.  S = 1: tokens = per-row argmax (ties to the lowest
 * id).  S = 2: the K/2 most confident rows (max softmax probability, ties to
 * the lower position) keep their pass-1 tokens; the block is re-run with
 * those tokens embedded and the other rows take the pass-2 argmax.
 * Outputs (device, caller-owned): draft_tokens int32 [B, K]; conf fp32
 * [B, K] (max softmax probability) or NULL; logits fp32 [B, K, vocab] or
 * NULL (for S = 2: pass-1 rows on committed positions, pass-2 rows
 * elsewhere); committed int32 [B, K] (1 = committed in pass 1; all 0 for
 * S = 1) or NULL. */
dflash_status dflash_draft_block(dflash_ctx* ctx, int B, int S, int32_t* draft_tokens, float* conf,
                                 float* logits, int32_t* committed, dflash_stream stream);

/* Lossless acceptance.  [Guide] "The Cost Breakdown of Speculative Rounds"
 * (the longest valid prefix tau <= gamma is accepted); [Chapter] "Common
 * misconception" (the output distribution is exactly the target's).
 *
 * mode 0, greedy: target_tokens device int32 [B, K+1] (the target's greedy
 *   token at each block position and the bonus position); tau = first i
 *   with draft_tokens[i] != target_tokens[i], else K; emits
 *   target_tokens[0..tau].
 * mode 1, stochastic: target_logits device fp32 [B, K+1, vocab];
 *   p_i = softmax(z_i / temperature); draft_probs device fp32 [B, K, vocab]
 *   or NULL for the point mass at the draft token (argmax drafts).  Accept
 *   d_i iff u_i < min(1, p_i(d_i)/q_i(d_i)); on the first reject emit a draw
 *   from max(0, p_i - q_i) (p_i if that is all zero) and stop; if all K are
 *   accepted emit a draw from p_K.  Uniforms: Philox4x32-10 with key =
 *   seed and counter (v, i | stream << 16, b, round); stream 0 is the accept
 *   test (v = 0), stream 1 the exponential race argmax_v r(v) / -ln U_v.
 *   round = DFLASH_ROUND_DEVICE takes the round from a counter on the
 *   device instead: the call uses its current value and advances it by one
 *   (dflash_create and dflash_reset set it to 0), so a captured round
 *   (dflash_graph_begin) draws fresh uniforms at every replay.
 * Outputs (device): accept_len int32 [B] (tau), emitted int32 [B, K+1]
 * (-1 padded), n_emit int32 [B] = tau + 1.  The KV cache is not touched:
 * the next dflash_inject_kv appends n_emit rows. */
#define DFLASH_ROUND_DEVICE UINT64_MAX

dflash_status dflash_accept(dflash_ctx* ctx, int mode, int B, const int32_t* draft_tokens,
                            const int32_t* target_tokens, const float* target_logits,
                            const float* draft_probs, float temperature, uint64_t seed,
                            uint64_t round, int32_t* accept_len, int32_t* emitted, int32_t* n_emit,
                            dflash_stream stream);

/* Training-time block attention.  [Paper] Figure 4 (the training mask: the
 * positions of a masked block see each other and the target context before
 * the block, and nothing of any other block).
 *
 * For NB blocks of K = 16 positions (NB <= max_batch): block j belongs to
 * sequence seq[j] (device int32 [NB]) and sees that sequence's injected
 * context at positions 0 .. ctx_len[j] - 1 (device int32 [NB], at most the
 * sequence's length) and all 16 positions of its own block, nothing of any
 * other block.  q: device fp16 [NB, 16, n_q_heads, head_dim]; k_blk, v_blk:
 * device fp16 [NB, 16, n_kv_heads, head_dim], the blocks' own keys (their
 * positions already encoded) and values; out: device fp32 [NB, 16,
 * n_q_heads, head_dim], softmax(q k^T / sqrt(head_dim)) v with query head h
 * reading kv head h / (n_q_heads / n_kv_heads).  layer selects the context
 * K/V of that draft layer.  The blocks' keys and values are staged in the
 * pool's block pages and the queries in the workspace, so the call must not
 * overlap a dflash_draft_block on the same context.  A sequence index
 * outside [0, max_batch) or a prefix outside [0, seq_len] sets
 * DFLASH_DEV_BAD_BLOCK and is clamped.  DFLASH_BF16 and DFLASH_BF16_W8
 * contexts (fp16 pool) only: DFLASH_F32 returns UNSUPPORTED_SHAPE.
 * Asynchronous. */
dflash_status dflash_block_attention(dflash_ctx* ctx, int layer, int NB, const int32_t* seq,
                                     const int32_t* ctx_len, const void* q, const void* k_blk,
                                     const void* v_blk, float* out, dflash_stream stream);

/* Host-free rounds.  [Chapter] "The systems side: Spec V2" (the host's
 * bookkeeping of a round is overlapped with the GPU's work) and the
 * [Guide]'s "Production Benchmarks on NVIDIA Blackwell B200" (the
 * deployment runs on CUDA graphs).
 *
 * Every call of inject, draft and accept is asynchronous and keeps tau,
 * lengths and pages on the device, so a whole round (dflash_inject_kv with
 * the previous round's n_emit as n_rows, dflash_draft_block, the caller's
 * own verification work, dflash_accept) can be recorded once and replayed
 * as one CUDA graph launch.  dflash_graph_begin starts recording `stream`
 * (a created stream, not the legacy default one) in thread-local capture
 * mode: every call on that stream up to dflash_graph_end, of this library or
 * of the caller (kernels, async copies), is recorded instead of run, with
 * the arguments it had (pointers, B, S, mode, seed; use DFLASH_ROUND_DEVICE
 * for stochastic rounds).  Make each recorded call once outside the capture
 * first, with the same shapes: the first call of a shape sets up host-side
 * state (tensor maps, occupancy figures) that capture does not allow.
 * While recording, dflash_get_status, dflash_profile_enable and
 * dflash_profile_read return DFLASH_ERR_CAPTURE, and so does a second
 * dflash_graph_begin.  The graph borrows every buffer the recorded calls
 * name; they must outlive it and stay where they are. */
typedef struct dflash_graph dflash_graph; /* opaque, owned by the caller after dflash_graph_end */

/* Start recording `stream`.  Errors: INVALID_ARG (NULL stream), CAPTURE
 * (already recording, or per-launch profiling is on), CUDA. */
dflash_status dflash_graph_begin(dflash_ctx* ctx, dflash_stream stream);

/* Stop recording and instantiate the graph into *out.  If a call failed
 * while recording (the capture was invalidated) returns CUDA and *out is
 * NULL; the stream is no longer recording either way.  Errors: INVALID_ARG,
 * CAPTURE (not recording, or another stream), CUDA. */
dflash_status dflash_graph_end(dflash_ctx* ctx, dflash_stream stream, dflash_graph** out);

/* Enqueue one replay of the recorded round on `stream` (any stream). */
dflash_status dflash_graph_launch(dflash_graph* graph, dflash_stream stream);

/* Free the graph (after its replays have completed). */
dflash_status dflash_graph_destroy(dflash_graph* graph);

/* The drafter's dense projection kernel on its own, for testing it in
 * isolation: out[s][m][n] = sum over the k-blocks of split s of
 * (X[m][k] + X_lo[m][k]) * W[n][k], with W device bf16 [N, K], X and the
 * optional second term X_lo (NULL = none) device bf16 [M, K] (row-major,
 * K a multiple of 8, 16-byte aligned) and out device fp32 [splits, M, N].  splits is normalised so that every split owns at least
 * one 64-wide k-block; the count used is returned in *splits_used (host).
 * status: device int32, caller-owned; a wait timeout sets its
 * DFLASH_DEV_WAIT_TIMEOUT bit.  Asynchronous on `stream`.  No counterpart
 * on the pages: it is the tensor-core GEMM behind every projection of the
 * three calls above, exposed so it can be checked on its own. */
dflash_status dflash_gemm_bf16(const void* W, int N, int K, const void* X, const void* X_lo, int M, float* out,
                               int splits, int* splits_used, int* status, dflash_stream stream);

/* dflash_gemm_bf16 with E4M3 weights (the DFLASH_BF16_W8 projection kernel
 * on its own, for testing it in isolation): out[s][m][n] = w_scale[n] *
 * sum over the k-blocks of split s of (X[m][k] + X_lo[m][k]) * decode(W[n][k]),
 * with W device uint8 E4M3 codes [N, K] (K a multiple of 16, 16-byte
 * aligned) and w_scale device fp32 [N]; everything else as for
 * dflash_gemm_bf16.  No counterpart on the pages beyond the FP8 storage
 * format itself. */
dflash_status dflash_gemm_w8(const void* W, const float* w_scale, int N, int K, const void* X, const void* X_lo,
                             int M, float* out, int splits, int* splits_used, int* status, dflash_stream stream);

/* dflash_gemm_bf16 for callers that cannot allocate device memory.  Some
 * callers must not call cudaMalloc or have it called on their behalf: a
 * process whose HBM is handed in full to another allocator up front (a
 * framework's caching allocator, a serving engine's KV reserve), where an
 * extra allocation fails or fragments that memory, or code that cannot take
 * cudaMalloc's implicit device synchronisation.  No counterpart on the
 * pages: it is a packaging of the projection kernel, not a step of the
 * method.
 *
 * out (device fp32 [M, N], caller-owned) = (X + X_lo) . W^T summed over all
 * k-blocks; W, X, X_lo and splits as for dflash_gemm_bf16 (splits_used:
 * host, nullable).  The split-K partials live in a fixed 8 MiB array inside
 * the library (a __device__ object that every GPU loading the library holds
 * until exit): splits_used * M * N must not exceed 2^21 - 64 floats, else
 * DFLASH_ERR_TOO_LARGE and nothing is enqueued.  status: device int32
 * (caller-owned), where a bounded device wait that gives up sets
 * DFLASH_DEV_WAIT_TIMEOUT (out then holds partial sums); the word is only
 * ever OR-ed into, so clear it before the call.  With status NULL the call
 * uses a slot of the library's array, cleared by each call, that no entry
 * point reads back: a device-side failure is then not reported, so callers
 * that need to know of one pass a status word.
 * The call allocates nothing (no cudaMalloc, no cudaFree, no allocating
 * library routine).  Its first call on a device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture.  All calls share the one array and it
 * keeps the last call's contents, so calls whose work overlaps on the GPU
 * (different streams, or host threads) race; serialise them.  Asynchronous
 * on `stream`. */
dflash_status dflash_gemm_bf16_noalloc(const void* W, int N, int K, const void* X, const void* X_lo, int M,
                                       float* out, int splits, int* splits_used, int* status,
                                       dflash_stream stream);

/* Kernel timing classes of dflash_profile_read. */
#define DFLASH_PROF_PROJ 0      /* draft-layer projections (QKV, O, gate/up, down) */
#define DFLASH_PROF_LMHEAD 1    /* LM head with the fused argmax reduction */
#define DFLASH_PROF_INJECT 2    /* feature-fusion and K/V-injection projections */
#define DFLASH_PROF_ATTN 3      /* block attention (splits + merge) */
#define DFLASH_PROF_ROWWISE 4   /* row-wise kernels: norms, RoPE, SwiGLU, paging, merges */
#define DFLASH_PROF_ACCEPT 5    /* acceptance */
#define DFLASH_PROF_CLASSES 6

/* Turn per-launch timing on (1) or off (0).  While on, every launch of the
 * three calls is bracketed by CUDA events on its stream (host-side objects
 * only; no device memory). */
dflash_status dflash_profile_enable(dflash_ctx* ctx, int enable);

/* Synchronise `stream`, then add up the recorded launches per class:
 * ms[c] = total device time, launches[c] = number of kernel launches
 * (both arrays DFLASH_PROF_CLASSES long, host).  Clears the record. */
dflash_status dflash_profile_read(dflash_ctx* ctx, float* ms, int* launches, dflash_stream stream);

/* Synchronise `stream` and read the device status word (DFLASH_DEV_* bits).
 * Off the hot path. */
dflash_status dflash_get_status(dflash_ctx* ctx, int* device_status, dflash_stream stream);

/* Human-readable name of a status code. */
const char* dflash_status_string(dflash_status s);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H_ */

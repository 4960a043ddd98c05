// The libdflash C ABI (include/dflash.h): context set-up, workspace layout
// and the sequence of kernels behind dflash_inject_kv, dflash_draft_block and
// dflash_accept.  All device memory is the caller's; nothing here allocates.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "common.cuh"
#include "internal.h"
#include "kernels.cuh"

using namespace dflash;

namespace dflash {

bool prefer_max_smem(const void* kernel) {
  // a fixed table (no host heap) of (kernel, device) pairs already set: the
  // attribute belongs to the kernel on one device; the library has a few
  // dozen kernel instances
  static std::mutex mu;
  static const void* done[512];
  static int done_dev[512];
  static int n_done = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_done; ++i)
    if (done[i] == kernel && done_dev[i] == dev) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
      cudaSuccess)
    return false;
  if (n_done < 512) {
    done[n_done] = kernel;
    done_dev[n_done++] = dev;
  }
  return true;
}

}  // namespace dflash

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// bytes of an activation / feature element: bf16 for DFLASH_BF16 and
// DFLASH_BF16_W8 (whose E4M3 weights are one byte), fp32 otherwise
int elem_bytes(const dflash_config& g) { return g.dtype == DFLASH_F32 ? 4 : 2; }
// q and the KV pool: fp16 for bf16 workloads, fp32 for fp32 workloads
int kv_elem_bytes(const dflash_config& g) { return g.dtype == DFLASH_F32 ? 4 : 2; }

int ceil_div(int a, int b) { return (a + b - 1) / b; }
// Split count of one draft-side GEMM for M activation rows (hi/lo inputs).
int draft_splits(const dflash_config& g, int M, int N, int K, int num_sms, int max_ctas = 0) {
  if (g.dtype == DFLASH_F32) return 1;
  const int bn = gemm_bn(M, true, g.dtype == DFLASH_BF16_W8);
  return gemm_splits(ceil_div(N, kTileN) * ceil_div(M, bn), gemm_kb(K), bn, true, num_sms, max_ctas,
                     g.dtype == DFLASH_BF16_W8);
}
// Split count of an inject-side GEMM: independent of the row count (sized
// for a 32-row tile), so a row's result does not depend on how many rows
// share the call.
int inject_splits(const dflash_config& g, int N, int K, bool split, int num_sms) {
  if (g.dtype == DFLASH_F32) return 1;
  return gemm_splits(ceil_div(N, kTileN), gemm_kb(K), 32, split, num_sms, 0, g.dtype == DFLASH_BF16_W8);
}

// Rows of the packed gate/up weight: groups of 64 features, 64 gate rows then
// the 64 matching up rows, the last group zero-padded.
int gu_rows(int F) { return 128 * ceil_div(F, 64); }

int attn_max_splits_for(const dflash_config& g, int num_sms) {
  const int max_keys = g.max_pages_per_seq * kPage + kBlockK;
  const int by_sms = ceil_div(2 * num_sms, g.n_kv_heads);
  return std::max(1, std::min(by_sms, ceil_div(max_keys, 32)));
}

bool config_ok(const dflash_config* g) {
  if (g == nullptr) return false;
  if (g->dtype != DFLASH_F32 && g->dtype != DFLASH_BF16 && g->dtype != DFLASH_BF16_W8) return false;
  if (g->block_k != kBlockK || g->page_size != kPage) return false;
  if (g->n_layers < 1 || g->hidden < 8 || g->n_q_heads < 1 || g->n_kv_heads < 1) return false;
  if (g->n_q_heads % g->n_kv_heads != 0) return false;
  const int G = g->n_q_heads / g->n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return false;
  if (g->head_dim != 32 && g->head_dim != 64 && g->head_dim != 128) return false;
  if (g->dtype != DFLASH_F32 && g->head_dim == 32) return false;  // the fp16 attention tiles 64-wide
  if (g->ffn < 8 || g->vocab < 2 || g->mask_id < 0 || g->mask_id >= g->vocab) return false;
  if (g->n_taps < 1 || g->tap_width < 1) return false;
  if (g->max_batch < 1 || g->max_batch > 4096 || g->max_pages_per_seq < 1 || g->n_pages < 1) return false;
  if (g->max_rows < 1 || g->max_inject_rows < g->max_rows) return false;
  if (!(g->rope_theta > 0.f) || !(g->rms_eps >= 0.f)) return false;
  // TMA row strides must be multiples of 16 bytes; vector row copies need 16 bytes
  // (E4M3 weight rows: one byte an element)
  const int q = g->dtype == DFLASH_BF16_W8 ? 16 : elem_bytes(*g) == 2 ? 8 : 4;
  const int F = g->n_taps * g->tap_width;
  if (g->hidden % q || F % q || g->ffn % q || (g->n_q_heads * g->head_dim) % q) return false;
  return true;
}

struct Carve {
  char* base;
  size_t off = 0;
  void* take(size_t bytes) {
    void* p = base ? base + off : nullptr;
    off += align_up(bytes);
    return p;
  }
};

// Lays the workspace out (base == nullptr: just measure).
size_t layout(const dflash_config& g, int num_sms, dflash_ctx* c, char* base) {
  Carve w{base};
  const int e = elem_bytes(g);
  const size_t R = g.max_inject_rows, M = static_cast<size_t>(g.max_batch) * kBlockK;
  const int d = g.hidden, F = g.ffn, qd = g.n_q_heads * g.head_dim, kvd = g.n_kv_heads * g.head_dim;
  const int Fin = g.n_taps * g.tap_width, V = g.vocab, L = g.n_layers;
  const int n_lm_tiles = ceil_div(V, kTileN);
  const int rope_rows = g.max_pages_per_seq * kPage + kBlockK;
  const int Ngu = gu_rows(F), Nkv = 2 * L * kvd, Nqkv = qd + 2 * kvd;
  // fp32 projection outputs: the FC output u; for fp32 workloads also the
  // staging of every projection before its epilogue
  size_t yf = R * d;
  if (g.dtype == DFLASH_F32)
    yf = std::max({yf, R * static_cast<size_t>(Nkv), M * static_cast<size_t>(std::max({Nqkv, Ngu, d}))});
  const int G = g.n_q_heads / g.n_kv_heads;
  const int amax = attn_max_splits_for(g, num_sms);
  const size_t attn_rows = static_cast<size_t>(g.max_batch) * g.n_kv_heads * amax * G * kBlockK;

  int* status = static_cast<int*>(w.take(sizeof(int) * 8));
  auto free_ring = static_cast<int32_t*>(w.take(sizeof(int32_t) * g.n_pages));
  auto row_seq = static_cast<int32_t*>(w.take(sizeof(int32_t) * R));
  auto row_pos = static_cast<int32_t*>(w.take(sizeof(int32_t) * R));
  auto row_src = static_cast<int32_t*>(w.take(sizeof(int32_t) * R));
  auto blk_row = static_cast<int32_t*>(w.take(sizeof(int32_t) * g.max_batch));
  auto blk_len = static_cast<int32_t*>(w.take(sizeof(int32_t) * g.max_batch));
  auto attn_order = static_cast<int32_t*>(w.take(sizeof(int32_t) * g.max_batch));
  auto rcos = static_cast<float*>(w.take(sizeof(float) * rope_rows * (g.head_dim / 2)));
  auto rsin = static_cast<float*>(w.take(sizeof(float) * rope_rows * (g.head_dim / 2)));
  const bool lo = g.dtype != DFLASH_F32;  // GEMM inputs carry a second bf16 term
  void* fc_in = w.take(R * Fin * e);
  void* h_fused = w.take(R * d * e);
  void* h_lo = lo ? w.take(R * d * e) : nullptr;
  auto y = static_cast<float*>(w.take(sizeof(float) * yf));
  auto x = static_cast<float*>(w.take(sizeof(float) * M * d));
  void* a = w.take(M * d * e);
  void* a_lo = lo ? w.take(M * d * e) : nullptr;
  void* q = w.take(M * qd * kv_elem_bytes(g));
  void* o = w.take(M * qd * e);
  void* o_lo = lo ? w.take(M * qd * e) : nullptr;
  void* act = w.take(M * F * e);
  void* act_lo = lo ? w.take(M * F * e) : nullptr;
  auto attn_o = static_cast<float*>(w.take(sizeof(float) * attn_rows * g.head_dim));
  auto attn_ml = static_cast<float*>(w.take(sizeof(float) * attn_rows * 2));
  auto lm_mx = static_cast<float*>(w.take(sizeof(float) * M * n_lm_tiles));
  auto lm_se = static_cast<float*>(w.take(sizeof(float) * M * n_lm_tiles));
  auto lm_idx = static_cast<int32_t*>(w.take(sizeof(int32_t) * M * n_lm_tiles));
  float* logits_ws = g.dtype == DFLASH_F32 ? static_cast<float*>(w.take(sizeof(float) * M * V)) : nullptr;
  auto tok1 = static_cast<int32_t*>(w.take(sizeof(int32_t) * M));
  auto conf1 = static_cast<float*>(w.take(sizeof(float) * M));
  auto commit = static_cast<int32_t*>(w.take(sizeof(int32_t) * M));
  const size_t d_tiles = ceil_div(d, kTileN);
  auto ss_x = static_cast<float*>(w.take(sizeof(float) * d_tiles * M));
  auto ss_h = static_cast<float*>(w.take(sizeof(float) * d_tiles * R));
  const size_t Mc = M / 2;  // S = 2: the uncommitted half of the block rows
  void* ac = lo ? w.take(Mc * d * e) : nullptr;
  void* ac_lo = lo ? w.take(Mc * d * e) : nullptr;
  auto ss_c = lo ? static_cast<float*>(w.take(sizeof(float) * d_tiles * Mc)) : nullptr;
  auto crow = lo ? static_cast<int32_t*>(w.take(sizeof(int32_t) * Mc)) : nullptr;
  // the persistent projection kernel's split tail (it serves 256 rows and more)
  const bool pers = g.dtype == DFLASH_BF16 && std::max(R, M) >= 256;
  auto pers_ws = pers ? static_cast<float*>(w.take(sizeof(float) * num_sms * 128 * 128)) : nullptr;
  auto pers_cnt = pers ? static_cast<int*>(w.take(sizeof(int) * num_sms)) : nullptr;
  if (c != nullptr) {
    c->status = status;
    c->scal = status + 4;
    c->free_ring = free_ring;
    c->row_seq = row_seq;
    c->row_pos = row_pos;
    c->row_src = row_src;
    c->blk_row = blk_row;
    c->blk_len = blk_len;
    c->attn_order = attn_order;
    c->rope_cos = rcos;
    c->rope_sin = rsin;
    c->rope_rows = rope_rows;
    c->fc_in = fc_in;
    c->h_fused = h_fused;
    c->h_lo = h_lo;
    c->y = y;
    c->x = x;
    c->a = a;
    c->a_lo = a_lo;
    c->q = q;
    c->o = o;
    c->o_lo = o_lo;
    c->act = act;
    c->act_lo = act_lo;
    c->attn_o = attn_o;
    c->attn_ml = attn_ml;
    c->attn_max_splits = amax;
    c->lm = LmPartials{lm_mx, lm_se, lm_idx, n_lm_tiles};
    c->logits_ws = logits_ws;
    c->tok1 = tok1;
    c->conf1 = conf1;
    c->commit = commit;
    c->ss_x = ss_x;
    c->ss_h = ss_h;
    c->ac = ac;
    c->ac_lo = ac_lo;
    c->ss_c = ss_c;
    c->crow = crow;
    c->pers_ws = pers_ws;
    c->pers_cnt = pers_cnt;
  }
  return w.off;
}

int device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  return n;
}

#define DF_CHECK(call)                               \
  do {                                               \
    if ((call) != cudaSuccess) return DFLASH_ERR_CUDA; \
  } while (0)

#define DF_RUN(call)                  \
  do {                                \
    const dflash_status st_ = (call); \
    if (st_ != DFLASH_OK) return st_; \
  } while (0)

// Row scales of layer l's E4M3 projection weights, or null (bf16 weights).
const float* w_row_scale(const std::vector<const float*>& v, int l) { return v.empty() ? nullptr : v[l]; }

dflash_status run_gemm(dflash_ctx* c, const void* W, const float* w_scale, int N, int K, const void* X,
                       const void* X_lo, int M,
                       int M_alloc, int splits, const int* m_valid, const EpiArgs& epi, cudaStream_t s,
                       const NextGemm& next = NextGemm{}) {
  GemmLaunch g{};
  g.W = W;
  g.X = X;
  g.X_lo = X_lo;
  g.N = N;
  g.K = K;
  g.M = M;
  g.M_alloc = M_alloc;
  g.splits = c->cfg.dtype != DFLASH_F32 ? splits : 1;
  g.out = c->cfg.dtype != DFLASH_F32 ? nullptr : c->y;  // fp32 staging (bf16: epilogues write directly)
  g.w_scale = w_scale;
  g.split_stride = static_cast<long long>(M) * N;
  g.ldo = N;
  g.m_valid = m_valid;
  g.epi = epi;
  g.next = next;
  DF_CHECK(gemm_launch(c, g, s));
  return DFLASH_OK;
}

// The projection after a launch, for the L2 prefetch of its weights (only the
// latency-bound attention issues one: between projections HBM is busy and
// the prefetch would only compete).
NextGemm next_gemm(const void* W, int N, int K, int M, int splits, long long budget) {
  NextGemm n;
  n.W = W;
  n.N = N;
  n.K = K;
  n.M = M;
  n.split = true;
  n.splits = splits;
  n.budget_bytes = budget;
  return n;
}

EpiArgs epi_base(dflash_ctx* c, int kind, int M, int N) {
  EpiArgs e{};
  e.kind = kind;
  e.M = M;
  e.N = N;
  e.Hq = c->cfg.n_q_heads;
  e.Hkv = c->cfg.n_kv_heads;
  e.dh = c->cfg.head_dim;
  e.rope_cos = c->rope_cos;
  e.rope_sin = c->rope_sin;
  return e;
}

// Folded RMSNorm over the hidden size (epilogue.cuh), consumer side: the
// projection's input is g . z and its output rows are scaled by 1 / RMS(z).
void norm_in(dflash_ctx* c, EpiArgs& e, const float* ss, int ss_ld) {
  e.ss_in = ss;
  e.ss_tiles = ceil_div(c->cfg.hidden, kTileN);
  e.norm_dim_inv = 1.f / static_cast<float>(c->cfg.hidden);
  e.eps = c->cfg.rms_eps;
  e.ss_ld = ss_ld;
}
// Producer side: the stored rows z also become the next input g . z (hi, lo)
// with their partial sums of squares.
void norm_out(EpiArgs& e, void* hi, void* lo, const void* gain, float* ss, int ss_ld) {
  e.nx_hi = hi;
  e.nx_lo = lo;
  e.nx_gain = gain;
  e.ss_out = ss;
  e.ss_ld = ss_ld;
}

char* pool_layer(void* pool, const dflash_ctx* c, int layer) {
  const long long per_layer = static_cast<long long>(c->pool_pages) * c->cfg.n_kv_heads * kPage * c->cfg.head_dim;
  return static_cast<char*>(pool) + per_layer * layer * c->kv_elem;
}

// Brackets the launches between its construction and destruction with a
// pair of events of one timing class (no-op unless profiling is on).
struct ProfScope {
  dflash_ctx* c;
  cudaStream_t s;
  int cls, launches;
  cudaEvent_t a = nullptr;
  static cudaEvent_t get(dflash_ctx* c) {
    if (!c->prof_pool.empty()) {
      cudaEvent_t e = c->prof_pool.back();
      c->prof_pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
  }
  ProfScope(dflash_ctx* c_, int cls_, int launches_, cudaStream_t s_) : c(c_), s(s_), cls(cls_), launches(launches_) {
    if (!c->prof_on) return;
    a = get(c);
    if (a != nullptr) cudaEventRecord(a, s);
  }
  void close() {
    if (a == nullptr) return;
    cudaEvent_t b = get(c);
    if (b != nullptr) {
      cudaEventRecord(b, s);
      c->prof_live.push_back({a, b, cls, launches});
    } else {
      c->prof_pool.push_back(a);
    }
    a = nullptr;
  }
  ~ProfScope() { close(); }
};

}  // namespace

extern "C" {

const char* dflash_status_string(dflash_status s) {
  switch (s) {
    case DFLASH_OK: return "ok";
    case DFLASH_ERR_INVALID_ARG: return "invalid argument";
    case DFLASH_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case DFLASH_ERR_POOL_EXHAUSTED: return "KV page pool exhausted";
    case DFLASH_ERR_CUDA: return "CUDA error";
    case DFLASH_ERR_STATE: return "device status word set";
    case DFLASH_ERR_WORKSPACE: return "workspace or pool buffer too small";
    case DFLASH_ERR_TOO_LARGE: return "request exceeds the fixed scratch of the no-allocation entry point";
    case DFLASH_ERR_CAPTURE: return "not allowed in the context's capture state";
  }
  return "unknown";
}

size_t dflash_workspace_size(const dflash_config* cfg) {
  if (!config_ok(cfg)) return 0;
  return layout(*cfg, device_sms(), nullptr, nullptr);
}

size_t dflash_kv_pool_size(const dflash_config* cfg) {
  if (!config_ok(cfg)) return 0;
  return 2ull * cfg->n_layers * (cfg->n_pages + cfg->max_batch) * cfg->n_kv_heads * kPage * cfg->head_dim *
         kv_elem_bytes(*cfg);
}

dflash_status dflash_create(const dflash_config* cfg, const dflash_weights* w, void* kv_pool, size_t kv_pool_bytes,
                            int32_t* page_table, int32_t* seq_len, void* workspace, size_t workspace_bytes,
                            dflash_ctx** out) {
  if (out == nullptr) return DFLASH_ERR_INVALID_ARG;
  *out = nullptr;
  if (cfg == nullptr || w == nullptr || kv_pool == nullptr || page_table == nullptr || seq_len == nullptr ||
      workspace == nullptr)
    return DFLASH_ERR_INVALID_ARG;
  if (!config_ok(cfg)) return DFLASH_ERR_UNSUPPORTED_SHAPE;
  if (w->w_fc == nullptr || w->g_fc == nullptr || w->embed == nullptr || w->g_final == nullptr ||
      w->w_lm == nullptr || w->w_kv_inject == nullptr || w->w_qkv == nullptr || w->w_o == nullptr ||
      w->w_gu == nullptr || w->w_down == nullptr || w->g_in == nullptr || w->g_post == nullptr)
    return DFLASH_ERR_INVALID_ARG;
  for (int l = 0; l < cfg->n_layers; ++l)
    if (w->w_qkv[l] == nullptr || w->w_o[l] == nullptr || w->w_gu[l] == nullptr || w->w_down[l] == nullptr ||
        w->g_in[l] == nullptr || w->g_post[l] == nullptr)
      return DFLASH_ERR_INVALID_ARG;
  if (cfg->dtype == DFLASH_BF16_W8) {
    if (w->s_fc == nullptr || w->s_lm == nullptr || w->s_kv_inject == nullptr || w->s_qkv == nullptr ||
        w->s_o == nullptr || w->s_gu == nullptr || w->s_down == nullptr)
      return DFLASH_ERR_INVALID_ARG;
    for (int l = 0; l < cfg->n_layers; ++l)
      if (w->s_qkv[l] == nullptr || w->s_o[l] == nullptr || w->s_gu[l] == nullptr || w->s_down[l] == nullptr)
        return DFLASH_ERR_INVALID_ARG;
  }
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign != 0 || reinterpret_cast<uintptr_t>(kv_pool) % 16 != 0)
    return DFLASH_ERR_INVALID_ARG;
  const int sms = device_sms();
  if (workspace_bytes < layout(*cfg, sms, nullptr, nullptr) || kv_pool_bytes < dflash_kv_pool_size(cfg))
    return DFLASH_ERR_WORKSPACE;

  dflash_ctx* c = new (std::nothrow) dflash_ctx();
  if (c == nullptr) return DFLASH_ERR_INVALID_ARG;
  c->cfg = *cfg;
  c->elem = elem_bytes(*cfg);
  c->num_sms = sms;
  c->w_fc = w->w_fc;
  c->g_fc = w->g_fc;
  c->embed = w->embed;
  c->g_final = w->g_final;
  c->w_lm = w->w_lm;
  c->w_kv_inj = w->w_kv_inject;
  c->key_offset = w->key_offset;
  c->w_qkv.assign(w->w_qkv, w->w_qkv + cfg->n_layers);
  c->w_o.assign(w->w_o, w->w_o + cfg->n_layers);
  c->w_gu.assign(w->w_gu, w->w_gu + cfg->n_layers);
  c->w_down.assign(w->w_down, w->w_down + cfg->n_layers);
  c->g_in.assign(w->g_in, w->g_in + cfg->n_layers);
  c->g_post.assign(w->g_post, w->g_post + cfg->n_layers);
  if (cfg->dtype == DFLASH_BF16_W8) {
    c->s_fc = w->s_fc;
    c->s_lm = w->s_lm;
    c->s_kv_inj = w->s_kv_inject;
    c->s_qkv.assign(w->s_qkv, w->s_qkv + cfg->n_layers);
    c->s_o.assign(w->s_o, w->s_o + cfg->n_layers);
    c->s_gu.assign(w->s_gu, w->s_gu + cfg->n_layers);
    c->s_down.assign(w->s_down, w->s_down + cfg->n_layers);
  }
  {
    const char* env = std::getenv("DFLASH_PDL");
    c->pdl = env == nullptr || std::strcmp(env, "0") != 0;
  }
  c->pool_pages = cfg->n_pages + cfg->max_batch;
  c->kv_elem = kv_elem_bytes(*cfg);
  const size_t half_pool = dflash_kv_pool_size(cfg) / 2;
  c->pool_k = kv_pool;
  c->pool_v = static_cast<char*>(kv_pool) + half_pool;
  c->page_table = page_table;
  c->seq_len = seq_len;
  layout(*cfg, sms, c, static_cast<char*>(workspace));
  // zero the pool once: attention multiplies masked (zero-probability) slots
  // by their values, which must therefore be finite
  if (cudaMemsetAsync(kv_pool, 0, dflash_kv_pool_size(cfg), nullptr) != cudaSuccess ||
      (c->pers_cnt != nullptr && cudaMemsetAsync(c->pers_cnt, 0, sizeof(int) * sms, nullptr) != cudaSuccess) ||
      launch_rope_table(c, nullptr) != cudaSuccess || launch_reset(c, nullptr) != cudaSuccess ||
      cudaStreamSynchronize(nullptr) != cudaSuccess) {
    delete c;
    return DFLASH_ERR_CUDA;
  }
  *out = c;
  return DFLASH_OK;
}

dflash_status dflash_destroy(dflash_ctx* ctx) {
  if (ctx == nullptr) return DFLASH_ERR_INVALID_ARG;
  if (ctx->capturing) {  // leave the stream usable: drop the unfinished recording
    cudaGraph_t g = nullptr;
    if (cudaStreamEndCapture(ctx->capture, &g) == cudaSuccess && g != nullptr) cudaGraphDestroy(g);
  }
  for (auto& r : ctx->prof_live) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : ctx->prof_pool) cudaEventDestroy(e);
  delete ctx;
  return DFLASH_OK;
}

dflash_status dflash_reset(dflash_ctx* ctx, dflash_stream stream) {
  if (ctx == nullptr) return DFLASH_ERR_INVALID_ARG;
  DF_CHECK(launch_reset(ctx, stream));
  if (ctx->pers_cnt != nullptr)
    DF_CHECK(cudaMemsetAsync(ctx->pers_cnt, 0, sizeof(int) * ctx->num_sms, static_cast<cudaStream_t>(stream)));
  return DFLASH_OK;
}

dflash_status dflash_release(dflash_ctx* ctx, int b, dflash_stream stream) {
  if (ctx == nullptr || b < 0 || b >= ctx->cfg.max_batch) return DFLASH_ERR_INVALID_ARG;
  DF_CHECK(launch_release(ctx, b, stream));
  return DFLASH_OK;
}

dflash_status dflash_truncate(dflash_ctx* ctx, int b, int new_len, dflash_stream stream) {
  if (ctx == nullptr || b < 0 || b >= ctx->cfg.max_batch || new_len < 0) return DFLASH_ERR_INVALID_ARG;
  DF_CHECK(launch_truncate(ctx, b, new_len, stream));
  return DFLASH_OK;
}

dflash_status dflash_inject_kv(dflash_ctx* ctx, const void* feats, const int32_t* n_rows, int first_seq, int B,
                               int max_rows, dflash_stream stream) {
  if (ctx == nullptr || feats == nullptr || n_rows == nullptr) return DFLASH_ERR_INVALID_ARG;
  const dflash_config& g = ctx->cfg;
  if (B < 1 || first_seq < 0 || first_seq + B > g.max_batch || max_rows < 1) return DFLASH_ERR_INVALID_ARG;
  if (max_rows > g.max_rows || static_cast<long long>(B) * max_rows > g.max_inject_rows)
    return DFLASH_ERR_UNSUPPORTED_SHAPE;
  if (reinterpret_cast<uintptr_t>(feats) % 16 != 0) return DFLASH_ERR_INVALID_ARG;
  cudaStream_t s = stream;
  const int rows = B * max_rows;
  const int d = g.hidden, Fin = g.n_taps * g.tap_width, kvd = g.n_kv_heads * g.head_dim;
  const int Nkv = 2 * g.n_layers * kvd;
  {
    ProfScope p(ctx, DFLASH_PROF_ROWWISE, 2, s);
    DF_CHECK(launch_alloc(ctx, n_rows, first_seq, B, max_rows, s));
    DF_CHECK(launch_gather_rows(ctx, feats, rows, s));
  }
  const int R = g.max_inject_rows;
  const int s_fc = inject_splits(g, d, Fin, false, ctx->num_sms);
  {
    // u = W_fc f; the fused hidden state RMSNorm(u) * g_fc is folded into the
    // K/V projection below
    ProfScope p(ctx, DFLASH_PROF_INJECT, 1, s);
    EpiArgs e = epi_base(ctx, EPI_STORE, rows, d);
    e.m_valid = ctx->scal;
    norm_out(e, ctx->h_fused, ctx->h_lo, ctx->g_fc, ctx->ss_h, R);
    DF_RUN(run_gemm(ctx, ctx->w_fc, ctx->s_fc, d, Fin, ctx->fc_in, nullptr, rows, R, s_fc, ctx->scal, e, s));
  }
  const int s_kv = inject_splits(g, Nkv, d, true, ctx->num_sms);
  {
    ProfScope p(ctx, DFLASH_PROF_INJECT, 1, s);
    EpiArgs e = epi_base(ctx, EPI_KV_INJECT, rows, Nkv);
    norm_in(ctx, e, ctx->ss_h, R);
    e.m_valid = ctx->scal;
    e.pool_k = ctx->pool_k;
    e.pool_v = ctx->pool_v;
    e.layer_stride = static_cast<long long>(ctx->pool_pages) * g.n_kv_heads * kPage * g.head_dim;
    e.row_seq = ctx->row_seq;
    e.row_pos = ctx->row_pos;
    e.page_table = ctx->page_table;
    e.max_pages = g.max_pages_per_seq;
    e.key_offset = ctx->key_offset;
    DF_RUN(run_gemm(ctx, ctx->w_kv_inj, ctx->s_kv_inj, Nkv, d, ctx->h_fused, ctx->h_lo, rows, R, s_kv, ctx->scal, e, s));
  }
  return DFLASH_OK;
}

dflash_status dflash_draft_block(dflash_ctx* ctx, int B, int S, int32_t* draft_tokens, float* conf, float* logits,
                                 int32_t* committed, dflash_stream stream) {
  if (ctx == nullptr || draft_tokens == nullptr) return DFLASH_ERR_INVALID_ARG;
  const dflash_config& g = ctx->cfg;
  if (B < 1 || B > g.max_batch || (S != 1 && S != 2)) return DFLASH_ERR_INVALID_ARG;
  cudaStream_t s = stream;
  const int M = B * kBlockK, Mmax = g.max_batch * kBlockK;
  const int d = g.hidden, F = g.ffn, qd = g.n_q_heads * g.head_dim, kvd = g.n_kv_heads * g.head_dim;
  const int Nqkv = qd + 2 * kvd, Ngu = gu_rows(F);
  const int sms = ctx->num_sms;
  // at most one QKV CTA per SM, so that the attention CTAs (launched early)
  // find room beside them and stream the context while QKV runs
  const int s_qkv = draft_splits(g, M, Nqkv, d, sms, sms);
  const int s_o = draft_splits(g, M, d, qd, sms);
  const int s_gu = draft_splits(g, M, Ngu, d, sms);
  const int s_dn = draft_splits(g, M, d, F, sms);
  const int a_sp = attn_splits(ctx, B);
  // with more attention CTAs than SMs, the sequences start longest context
  // first (the order is written by the embedding kernel of each pass)
  int32_t* order = g.dtype != DFLASH_F32 && B * g.n_kv_heads * a_sp > sms ? ctx->attn_order : nullptr;
  AttnSrc asrc;
  asrc.order = order;
  for (int pass = 0; pass < S; ++pass) {
    {
      ProfScope p(ctx, DFLASH_PROF_ROWWISE, 1, s);
      DF_CHECK(launch_embed(ctx, M, pass == 1, order, s));
    }
    // every pre-norm runs folded: the producing epilogue writes g . x and the
    // sums of squares of x (ss_x), the consuming projection scales its rows
    for (int l = 0; l < g.n_layers; ++l) {
      {
        ProfScope p(ctx, DFLASH_PROF_PROJ, 1, s);
        EpiArgs e = epi_base(ctx, EPI_QKV, M, Nqkv);
        norm_in(ctx, e, ctx->ss_x, Mmax);
        e.q = ctx->q;
        e.pool_k = pool_layer(ctx->pool_k, ctx, l);
        e.pool_v = pool_layer(ctx->pool_v, ctx, l);
        e.block_page0 = g.n_pages;
        e.seq_len = ctx->seq_len;
        DF_RUN(run_gemm(ctx, ctx->w_qkv[l], w_row_scale(ctx->s_qkv, l), Nqkv, d, ctx->a, ctx->a_lo, M, Mmax, s_qkv, nullptr, e, s));
      }
      {
        ProfScope p(ctx, DFLASH_PROF_ATTN, g.dtype != DFLASH_F32 ? 1 : 2, s);
        // attention is latency-bound: it streams all of the O projection's
        // weights beyond that kernel's ring into L2
        DF_CHECK(launch_attention(ctx, l, B, a_sp, s, next_gemm(ctx->w_o[l], d, qd, M, s_o, 1ll << 40), asrc));
      }
      {
        ProfScope p(ctx, DFLASH_PROF_PROJ, 1, s);
        EpiArgs e = epi_base(ctx, EPI_RESIDUAL, M, d);
        e.out = ctx->x;
        norm_out(e, ctx->a, ctx->a_lo, ctx->g_post[l], ctx->ss_x, Mmax);
        DF_RUN(run_gemm(ctx, ctx->w_o[l], w_row_scale(ctx->s_o, l), d, qd, ctx->o, ctx->o_lo, M, Mmax, s_o, nullptr, e, s));
      }
      {
        ProfScope p(ctx, DFLASH_PROF_PROJ, 1, s);
        EpiArgs e = epi_base(ctx, EPI_SWIGLU, M, Ngu);
        norm_in(ctx, e, ctx->ss_x, Mmax);
        e.act_hi = ctx->act;
        e.act_lo = ctx->act_lo;
        e.F = F;
        DF_RUN(run_gemm(ctx, ctx->w_gu[l], w_row_scale(ctx->s_gu, l), Ngu, d, ctx->a, ctx->a_lo, M, Mmax, s_gu, nullptr, e, s));
      }
      {
        ProfScope p(ctx, DFLASH_PROF_PROJ, 1, s);
        EpiArgs e = epi_base(ctx, EPI_RESIDUAL, M, d);
        e.out = ctx->x;
        norm_out(e, ctx->a, ctx->a_lo, l + 1 < g.n_layers ? ctx->g_in[l + 1] : ctx->g_final, ctx->ss_x, Mmax);
        DF_RUN(run_gemm(ctx, ctx->w_down[l], w_row_scale(ctx->s_down, l), d, F, ctx->act, ctx->act_lo, M, Mmax, s_dn, nullptr, e, s));
      }
    }
    // the second pass needs the LM head on its uncommitted rows only: they
    // are compacted first (a logits store puts each row back in its place)
    const bool compact = pass == 1 && g.dtype != DFLASH_F32;
    if (compact) {
      ProfScope pc(ctx, DFLASH_PROF_ROWWISE, 1, s);
      DF_CHECK(launch_compact_rows(ctx, B, Mmax, s));
    }
    const int Mc = g.max_batch * kBlockK / 2;
    EpiArgs fin = epi_base(ctx, EPI_NONE, compact ? M / 2 : M, g.vocab);  // the final norm, folded into the LM head
    norm_in(ctx, fin, compact ? ctx->ss_c : ctx->ss_x, compact ? Mc : Mmax);
    const int32_t* skip = pass == 1 && !compact ? ctx->commit : nullptr;
    ProfScope plm(ctx, DFLASH_PROF_LMHEAD, g.dtype != DFLASH_F32 ? 1 : 2, s);
    if (g.dtype != DFLASH_F32) {
      GemmLaunch lm{};
      lm.W = ctx->w_lm;
      lm.w_scale = ctx->s_lm;
      lm.X = compact ? ctx->ac : ctx->a;
      lm.X_lo = compact ? ctx->ac_lo : ctx->a_lo;
      lm.N = g.vocab;
      lm.K = d;
      lm.M = compact ? M / 2 : M;
      lm.M_alloc = compact ? Mc : Mmax;
      lm.splits = 1;
      lm.lm = ctx->lm;
      lm.logits = logits;
      lm.ld_logits = g.vocab;
      lm.skip_rows = skip;
      lm.logits_rows = compact ? ctx->crow : nullptr;
      lm.epi = fin;
      DF_CHECK(gemm_launch(ctx, lm, s));
    } else {
      GemmLaunch lm{};
      lm.W = ctx->w_lm;
      lm.X = ctx->a;
      lm.N = g.vocab;
      lm.K = d;
      lm.M = M;
      lm.M_alloc = Mmax;
      lm.splits = 1;
      lm.out = ctx->logits_ws;
      lm.ldo = g.vocab;
      DF_CHECK(gemm_launch(ctx, lm, s));
      DF_CHECK(launch_logits_tiles(ctx, M, logits, skip, fin, s));
    }
    plm.close();
    ProfScope pm(ctx, DFLASH_PROF_ROWWISE, S == 2 && pass == 0 ? 2 : 1, s);
    if (S == 1) {
      DF_CHECK(launch_lm_merge(ctx, M, nullptr, draft_tokens, conf, s));
    } else if (pass == 0) {
      DF_CHECK(launch_lm_merge(ctx, M, nullptr, ctx->tok1, ctx->conf1, s));
      DF_CHECK(launch_commit(ctx, B, s));
    } else {
      DF_CHECK(launch_lm_merge(ctx, M, ctx->commit, draft_tokens, conf, s, compact));
    }
  }
  if (committed != nullptr) {
    if (S == 2)
      DF_CHECK(cudaMemcpyAsync(committed, ctx->commit, sizeof(int32_t) * M, cudaMemcpyDeviceToDevice, s));
    else
      DF_CHECK(cudaMemsetAsync(committed, 0, sizeof(int32_t) * M, s));
  }
  return DFLASH_OK;
}

dflash_status dflash_accept(dflash_ctx* ctx, int mode, int B, const int32_t* draft_tokens,
                            const int32_t* target_tokens, const float* target_logits, const float* draft_probs,
                            float temperature, uint64_t seed, uint64_t round, int32_t* accept_len, int32_t* emitted,
                            int32_t* n_emit, dflash_stream stream) {
  if (ctx == nullptr || draft_tokens == nullptr || accept_len == nullptr || emitted == nullptr || n_emit == nullptr)
    return DFLASH_ERR_INVALID_ARG;
  if (B < 1 || B > ctx->cfg.max_batch) return DFLASH_ERR_INVALID_ARG;
  cudaStream_t s = stream;
  if (mode == 0) {
    if (target_tokens == nullptr) return DFLASH_ERR_INVALID_ARG;
    ProfScope p(ctx, DFLASH_PROF_ACCEPT, 1, s);
    DF_CHECK(launch_accept_greedy(B, kBlockK, draft_tokens, target_tokens, accept_len, emitted, n_emit, ctx->pdl, s));
    return DFLASH_OK;
  }
  if (mode != 1 || target_logits == nullptr || !(temperature > 0.f)) return DFLASH_ERR_INVALID_ARG;
  ProfScope p(ctx, DFLASH_PROF_ACCEPT, 1, s);
  int* round_ctr = round == DFLASH_ROUND_DEVICE ? ctx->status + 2 : nullptr;
  DF_CHECK(launch_accept_stochastic(B, kBlockK, ctx->cfg.vocab, draft_tokens, target_logits, draft_probs,
                                    temperature, seed, round, round_ctr, accept_len, emitted, n_emit, ctx->num_sms,
                                    ctx->pdl, s));
  return DFLASH_OK;
}

dflash_status dflash_block_attention(dflash_ctx* ctx, int layer, int NB, const int32_t* seq, const int32_t* ctx_len,
                                     const void* q, const void* k_blk, const void* v_blk, float* out,
                                     dflash_stream stream) {
  if (ctx == nullptr || seq == nullptr || ctx_len == nullptr || q == nullptr || k_blk == nullptr ||
      v_blk == nullptr || out == nullptr)
    return DFLASH_ERR_INVALID_ARG;
  const dflash_config& g = ctx->cfg;
  if (g.dtype == DFLASH_F32) return DFLASH_ERR_UNSUPPORTED_SHAPE;  // the fp16-pool (tcgen05) attention only
  if (layer < 0 || layer >= g.n_layers || NB < 1 || NB > g.max_batch) return DFLASH_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(q) % 16 || reinterpret_cast<uintptr_t>(k_blk) % 16 ||
      reinterpret_cast<uintptr_t>(v_blk) % 16)
    return DFLASH_ERR_INVALID_ARG;
  ProfScope p(ctx, DFLASH_PROF_ATTN, 3, stream);
  DF_CHECK(launch_block_attention(ctx, layer, NB, seq, ctx_len, q, k_blk, v_blk, out, stream));
  return DFLASH_OK;
}

dflash_status dflash_gemm_bf16(const void* W, int N, int K, const void* X, const void* X_lo, int M, float* out,
                               int splits, int* splits_used, int* status, dflash_stream stream) {
  if (W == nullptr || X == nullptr || out == nullptr || status == nullptr || N < 1 || K < 8 || K % 8 || M < 1 ||
      splits < 1)
    return DFLASH_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(W) % 16 || reinterpret_cast<uintptr_t>(X) % 16 ||
      reinterpret_cast<uintptr_t>(X_lo) % 16)
    return DFLASH_ERR_INVALID_ARG;
  dflash_ctx tmp;
  tmp.cfg = dflash_config{};
  tmp.cfg.dtype = DFLASH_BF16;
  tmp.status = status;
  tmp.num_sms = device_sms();
  const int n_kb = gemm_kb(K);
  const int want = std::min(splits, n_kb);
  const int per = (n_kb + want - 1) / want;
  const int s_used = (n_kb + per - 1) / per;
  if (splits_used != nullptr) *splits_used = s_used;
  GemmLaunch g{};
  g.W = W;
  g.X = X;
  g.X_lo = X_lo;
  g.N = N;
  g.K = K;
  g.M = M;
  g.M_alloc = M;
  g.splits = s_used;
  g.out = out;
  g.split_stride = static_cast<long long>(M) * N;
  g.ldo = N;
  DF_CHECK(gemm_launch(&tmp, g, stream));
  return DFLASH_OK;
}

dflash_status dflash_gemm_w8(const void* W, const float* w_scale, int N, int K, const void* X, const void* X_lo, int M, float* out,
                               int splits, int* splits_used, int* status, dflash_stream stream) {
  if (W == nullptr || w_scale == nullptr || X == nullptr || out == nullptr || status == nullptr || N < 1 || K < 16 ||
      K % 16 || M < 1 || splits < 1)
    return DFLASH_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(W) % 16 || reinterpret_cast<uintptr_t>(X) % 16 ||
      reinterpret_cast<uintptr_t>(X_lo) % 16)
    return DFLASH_ERR_INVALID_ARG;
  dflash_ctx tmp;
  tmp.cfg = dflash_config{};
  tmp.cfg.dtype = DFLASH_BF16_W8;
  tmp.status = status;
  const int n_kb = gemm_kb(K);
  const int s_used = gemm_normalize_splits(n_kb, std::min(splits, n_kb), true);
  if (splits_used != nullptr) *splits_used = s_used;
  GemmLaunch g{};
  g.W = W;
  g.X = X;
  g.X_lo = X_lo;
  g.N = N;
  g.K = K;
  g.M = M;
  g.M_alloc = M;
  g.splits = s_used;
  g.out = out;
  g.split_stride = static_cast<long long>(M) * N;
  g.ldo = N;
  g.w_scale = w_scale;
  DF_CHECK(gemm_launch(&tmp, g, stream));
  return DFLASH_OK;
}

dflash_status dflash_graph_begin(dflash_ctx* ctx, dflash_stream stream) {
  if (ctx == nullptr || stream == nullptr) return DFLASH_ERR_INVALID_ARG;
  if (ctx->capturing || ctx->prof_on) return DFLASH_ERR_CAPTURE;
  DF_CHECK(cudaStreamBeginCapture(stream, cudaStreamCaptureModeThreadLocal));
  ctx->capturing = true;
  ctx->capture = stream;
  return DFLASH_OK;
}

dflash_status dflash_graph_end(dflash_ctx* ctx, dflash_stream stream, dflash_graph** out) {
  if (ctx == nullptr || out == nullptr) return DFLASH_ERR_INVALID_ARG;
  *out = nullptr;
  if (!ctx->capturing || stream != ctx->capture) return DFLASH_ERR_CAPTURE;
  ctx->capturing = false;
  ctx->capture = nullptr;
  cudaGraph_t g = nullptr;
  if (cudaStreamEndCapture(stream, &g) != cudaSuccess || g == nullptr) {
    if (g != nullptr) cudaGraphDestroy(g);
    cudaGetLastError();
    return DFLASH_ERR_CUDA;
  }
  cudaGraphExec_t x = nullptr;
  if (cudaGraphInstantiate(&x, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    cudaGetLastError();
    return DFLASH_ERR_CUDA;
  }
  auto* r = new (std::nothrow) dflash_graph{g, x};
  if (r == nullptr) {
    cudaGraphExecDestroy(x);
    cudaGraphDestroy(g);
    return DFLASH_ERR_CUDA;
  }
  *out = r;
  return DFLASH_OK;
}

dflash_status dflash_graph_launch(dflash_graph* graph, dflash_stream stream) {
  if (graph == nullptr) return DFLASH_ERR_INVALID_ARG;
  DF_CHECK(cudaGraphLaunch(graph->exec, stream));
  return DFLASH_OK;
}

dflash_status dflash_graph_destroy(dflash_graph* graph) {
  if (graph == nullptr) return DFLASH_ERR_INVALID_ARG;
  cudaGraphExecDestroy(graph->exec);
  cudaGraphDestroy(graph->graph);
  delete graph;
  return DFLASH_OK;
}

dflash_status dflash_profile_enable(dflash_ctx* ctx, int enable) {
  if (ctx == nullptr) return DFLASH_ERR_INVALID_ARG;
  if (ctx->capturing) return DFLASH_ERR_CAPTURE;
  ctx->prof_on = enable != 0;
  return DFLASH_OK;
}

dflash_status dflash_profile_read(dflash_ctx* ctx, float* ms, int* launches, dflash_stream stream) {
  if (ctx == nullptr || ms == nullptr || launches == nullptr) return DFLASH_ERR_INVALID_ARG;
  if (ctx->capturing) return DFLASH_ERR_CAPTURE;
  for (int i = 0; i < DFLASH_PROF_CLASSES; ++i) {
    ms[i] = 0.f;
    launches[i] = 0;
  }
  DF_CHECK(cudaStreamSynchronize(stream));
  for (auto& r : ctx->prof_live) {
    float t = 0.f;
    if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&t, r.a, r.b) == cudaSuccess) {
      ms[r.cls] += t;
      launches[r.cls] += r.launches;
    }
    ctx->prof_pool.push_back(r.a);
    ctx->prof_pool.push_back(r.b);
  }
  ctx->prof_live.clear();
  return DFLASH_OK;
}

dflash_status dflash_get_status(dflash_ctx* ctx, int* device_status, dflash_stream stream) {
  if (ctx == nullptr || device_status == nullptr) return DFLASH_ERR_INVALID_ARG;
  if (ctx->capturing) return DFLASH_ERR_CAPTURE;
  DF_CHECK(cudaMemcpyAsync(device_status, ctx->status, sizeof(int), cudaMemcpyDeviceToHost, stream));
  DF_CHECK(cudaStreamSynchronize(stream));
  return DFLASH_OK;
}

}  // extern "C"

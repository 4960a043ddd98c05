// Paged draft KV cache bookkeeping, all on the device so that a round needs
// no host synchronisation ("The systems side: Spec V2" in the stable-lab
// chapter: KV allocation overlapped with GPU work instead of a host round
// trip).
//
// Free list: a ring of page ids (free_ring) with head and count in scal[1],
// scal[2].  An append serves sequences in index order; sequence b takes
// ceil((len_b + n_b)/16) - ceil(len_b/16) pages from the head.  If the total
// need exceeds the free count nothing changes and the status word records
// the exhaustion.  The cache stores only injected context (the DFlash Guide,
// "Zero Redundant KV Caching"), so rejected drafts never need a rollback.
#include "common.cuh"
#include "kernels.cuh"

namespace dflash {

__global__ void k_reset(int* status, int* scal, int32_t* free_ring, int P, int32_t* page_table, int n_pt,
                        int32_t* seq_len, int B) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x, stride = gridDim.x * blockDim.x;
  for (int i = t; i < P; i += stride) free_ring[i] = i;
  for (int i = t; i < n_pt; i += stride) page_table[i] = -1;
  for (int i = t; i < B; i += stride) seq_len[i] = 0;
  if (t == 0) {
    status[0] = 0;
    status[2] = 0;  // device round counter of the stochastic accept, and its arrivals
    status[3] = 0;
    scal[0] = 0;
    scal[1] = 0;
    scal[2] = P;
  }
}

__global__ void k_release(int b, int* scal, int32_t* free_ring, int P, int32_t* page_table, int max_pages,
                          int32_t* seq_len) {
  if (threadIdx.x != 0) return;
  const int n = (seq_len[b] + kPage - 1) / kPage;
  int head = scal[1], count = scal[2];
  for (int j = 0; j < n; ++j) {
    free_ring[(head + count) % P] = page_table[b * max_pages + j];
    page_table[b * max_pages + j] = -1;
    ++count;
  }
  scal[2] = count;
  seq_len[b] = 0;
}

// Shorten sequence b to new_len tokens (no-op if it is not longer): pages
// past ceil(new_len/16) go to the tail of the free list in table order.
__global__ void k_truncate(int b, int new_len, int* scal, int32_t* free_ring, int P, int32_t* page_table,
                           int max_pages, int32_t* seq_len) {
  if (threadIdx.x != 0) return;
  const int len = seq_len[b];
  if (new_len >= len || new_len < 0) return;
  const int keep = (new_len + kPage - 1) / kPage, n = (len + kPage - 1) / kPage;
  int head = scal[1], count = scal[2];
  for (int j = keep; j < n; ++j) {
    free_ring[(head + count) % P] = page_table[b * max_pages + j];
    page_table[b * max_pages + j] = -1;
    ++count;
  }
  scal[2] = count;
  seq_len[b] = new_len;
}

// One CTA.  The threads bring every sequence's row count and length into
// shared memory, thread 0 plans the append from there (prefix sums of rows
// and of new pages, the checks), and the threads then write the page-table
// entries, the row map of the compacted rows and the lengths in parallel.
__global__ void k_alloc(const int32_t* __restrict__ n_rows, int first_seq, int B, int max_rows, int P, int max_pages,
                        int32_t* seq_len, int32_t* page_table, int32_t* free_ring, int* scal, int32_t* row_seq,
                        int32_t* row_pos, int32_t* row_src, int* status) {
  extern __shared__ int s_off[];  // [B + 1] row offsets, [B] old lengths, [B] row counts, [B] new-page offsets
  int* s_len = s_off + B + 1;
  int* s_n = s_len + B;
  int* s_pg = s_n + B;
  __shared__ int s_ok, s_head;
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i < B; i += blockDim.x) {
    s_n[i] = n_rows[i];
    s_len[i] = seq_len[first_seq + i];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int bad = 0, total_need = 0, rows = 0;
    for (int i = 0; i < B; ++i) {
      const int n = s_n[i], len = s_len[i];
      s_off[i] = rows;
      s_pg[i] = total_need;
      if (n < 0 || n > max_rows) {
        bad |= ST_BAD_ROWS;
        continue;
      }
      rows += n;
      const int p_old = (len + kPage - 1) / kPage, p_new = (len + n + kPage - 1) / kPage;
      if (p_new > max_pages) bad |= ST_SEQ_TOO_LONG;
      total_need += p_new - p_old;
    }
    s_off[B] = rows;
    const int head = scal[1], count = scal[2];
    if (!bad && total_need > count) bad |= ST_POOL_EXHAUSTED;
    if (bad) {
      atomicOr(status, bad);
      scal[0] = 0;
      s_ok = 0;
    } else {
      scal[1] = (head + total_need) % P;
      scal[2] = count - total_need;
      scal[0] = rows;
      s_head = head;
      s_ok = 1;
    }
  }
  __syncthreads();
  if (!s_ok) return;
  // sequence i's new pages take the free ring's entries from head + s_pg[i] on
  for (int i = threadIdx.x; i < B; i += blockDim.x) {
    const int b = first_seq + i, len = s_len[i], n = s_n[i];
    const int p_old = (len + kPage - 1) / kPage, p_new = (len + n + kPage - 1) / kPage;
    for (int j = p_old; j < p_new; ++j)
      page_table[b * max_pages + j] = free_ring[(s_head + s_pg[i] + (j - p_old)) % P];
  }
  for (int i = 0; i < B; ++i) {
    const int n = s_off[i + 1] - s_off[i];
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
      const int r = s_off[i] + j;
      row_seq[r] = first_seq + i;
      row_pos[r] = s_len[i] + j;
      row_src[r] = i * max_rows + j;
    }
  }
  for (int i = threadIdx.x; i < B; i += blockDim.x) seq_len[first_seq + i] = s_len[i] + (s_off[i + 1] - s_off[i]);
}

// cos/sin of pos * theta^(-2i/dh), computed in double and stored as fp32.
__global__ void k_rope_table(float* cosb, float* sinb, int rows, int half, int head_dim, double theta) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= rows * half) return;
  const int pos = t / half, i = t % half;
  const double inv = pow(theta, -2.0 * i / head_dim);
  double sn, cs;
  sincos(static_cast<double>(pos) * inv, &sn, &cs);
  cosb[t] = static_cast<float>(cs);
  sinb[t] = static_cast<float>(sn);
}

cudaError_t launch_reset(dflash_ctx* c, cudaStream_t s) {
  const auto& g = c->cfg;
  k_reset<<<64, 256, 0, s>>>(c->status, c->scal, c->free_ring, g.n_pages, c->page_table,
                             g.max_batch * g.max_pages_per_seq, c->seq_len, g.max_batch);
  return cudaGetLastError();
}

cudaError_t launch_release(dflash_ctx* c, int b, cudaStream_t s) {
  k_release<<<1, 32, 0, s>>>(b, c->scal, c->free_ring, c->cfg.n_pages, c->page_table, c->cfg.max_pages_per_seq,
                             c->seq_len);
  return cudaGetLastError();
}

cudaError_t launch_truncate(dflash_ctx* c, int b, int new_len, cudaStream_t s) {
  k_truncate<<<1, 32, 0, s>>>(b, new_len, c->scal, c->free_ring, c->cfg.n_pages, c->page_table,
                              c->cfg.max_pages_per_seq, c->seq_len);
  return cudaGetLastError();
}

cudaError_t launch_alloc(dflash_ctx* c, const int32_t* n_rows, int first_seq, int B, int max_rows, cudaStream_t s) {
  const size_t smem = sizeof(int) * (4 * B + 1);
  return launch_k(k_alloc, dim3(1), dim3(256), smem, s, dim3(1), c->pdl, n_rows, first_seq, B, max_rows,
                  c->cfg.n_pages, c->cfg.max_pages_per_seq, c->seq_len, c->page_table, c->free_ring, c->scal,
                  c->row_seq, c->row_pos, c->row_src, c->status);
}

cudaError_t launch_rope_table(dflash_ctx* c, cudaStream_t s) {
  const int half = c->cfg.head_dim / 2;
  const int n = c->rope_rows * half;
  k_rope_table<<<(n + 255) / 256, 256, 0, s>>>(c->rope_cos, c->rope_sin, c->rope_rows, half, c->cfg.head_dim,
                                               static_cast<double>(c->cfg.rope_theta));
  return cudaGetLastError();
}

}  // namespace dflash

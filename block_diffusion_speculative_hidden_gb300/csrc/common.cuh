// Device-side helpers shared by the libdflash kernels (sm_103a).
//
// Inline PTX wrappers for the Blackwell data path used by the GEMMs:
// mbarrier phase tracking, TMA tiled loads (cp.async.bulk.tensor), the
// tcgen05 tensor-memory allocator, tcgen05.mma (kind::f16, bf16 in, fp32
// accumulate in TMEM), tcgen05.commit and tcgen05.ld.  Every spin-wait is
// bounded by wall-clock time (%globaltimer) and reports a timeout in the
// device status word instead of hanging.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dflash {

// Sticky bits of the device status word.
enum : int {
  ST_POOL_EXHAUSTED = 1,   // an inject needed more free pages than the pool had
  ST_SEQ_TOO_LONG = 2,     // a sequence would exceed max_pages_per_seq
  ST_WAIT_TIMEOUT = 4,     // a bounded device wait gave up
  ST_BAD_TOKEN = 8,        // a token id outside [0, vocab)
  ST_BAD_ROWS = 16,        // an n_rows entry outside [0, max_rows]
  ST_BAD_BLOCK = 32,       // a training block's sequence or prefix length out of range
};

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr int kBlockK = 16;  // draft block size K
constexpr int kPage = 16;    // tokens per KV page

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Orders this thread's view of global memory (generic proxy) before its
// later async-proxy accesses of it (bulk copies).
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbarrier_arrive_one(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait that may suspend the thread until the phase completes, for at
// most `hint_ns` (a waiting warp then takes no issue slots)
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same wait polling without suspending (test_wait): for the one thread
// that feeds a pipeline, whose reaction time is the pipeline's bubble.
// Gives up after kWaitLimitNs, sets ST_WAIT_TIMEOUT and returns false.
__device__ __forceinline__ bool mbar_wait_spin(uint64_t* bar, uint32_t parity, int* status) {
  if (mbar_test_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test_wait(bar, parity)) return true;
    if ((it & 255u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, ST_WAIT_TIMEOUT);
      return false;
    }
  }
}
// Waits for the phase with the given parity to complete.  Gives up after
// kWaitLimitNs, sets ST_WAIT_TIMEOUT and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_hint(bar, parity, 20000u)) return true;
    if ((it & 15u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, ST_WAIT_TIMEOUT);
      return false;
    }
  }
}

// ----------------------------------------------------------------- programmatic dependent launch
// Every kernel of the inject / draft chain is launched so that it may start
// while its stream predecessor is still running.  The rule that keeps this
// race-free everywhere in the library:
//   - before pdl_wait() a kernel touches only data that its immediate
//     predecessor neither writes nor reads back (weights, tensor maps, the
//     context pages of the KV pool, its own shared memory);
//   - pdl_trigger() (which lets the successor start) comes after pdl_wait()
//     in every CTA, so when a kernel starts, every kernel before its
//     predecessor has completed.
// pdl_wait() returns once the predecessor grid has completed and its memory
// is visible; without a programmatic dependency both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ----------------------------------------------------------------- clusters / DSMEM
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA in the cluster arrives and waits (release /
// acquire): shared-memory writes before it are visible to the whole cluster.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The two halves of cluster_sync_all, for work between arriving and waiting.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
// Arrive without ordering this thread's earlier memory operations (loads
// still in flight do not delay it); for barriers that only order progress,
// e.g. "every CTA of the cluster is past its main loop".
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory location in cluster CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Arrive (release, cluster scope) on the mbarrier at the same shared-memory
// offset in cluster CTA `rank`.
__device__ __forceinline__ void mbar_remote_arrive(uint64_t* local_bar, uint32_t rank) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(dsmem_map(smem_u32(local_bar), rank))
               : "memory");
}
__device__ __forceinline__ void fence_acq_rel_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }
// Bounded wait (as mbar_wait) with acquire at cluster scope: what the
// arriving CTA wrote before its release-arrive is visible afterwards.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, int* status) {
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
        : "memory");
    if (ok) return true;
    if ((it & 15u) == 15u && globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, ST_WAIT_TIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
// Bulk copy of `bytes` (a multiple of 16) from this CTA's shared memory to
// the same-offset shared memory of cluster CTA `rank`, completing as
// transaction bytes on that CTA's mbarrier `bar` (same offset as ours).
__device__ __forceinline__ void bulk_copy_smem_to_rank(uint32_t dst_local, uint32_t src_local, uint32_t bytes,
                                                       uint64_t* bar, uint32_t rank) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dsmem_map(dst_local, rank)),
      "r"(src_local), "r"(bytes), "r"(dsmem_map(smem_u32(bar), rank))
      : "memory");
}
// Bulk copy global memory -> this CTA's shared memory (16-byte aligned
// addresses, a multiple of 16 bytes), completing as transaction bytes on
// the mbarrier `bar`.
__device__ __forceinline__ void bulk_load_global(uint32_t dst_local, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst_local),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
// Bulk copy shared memory -> global memory (the copy engine reads the
// source asynchronously; 16-byte aligned addresses, a multiple of 16 bytes),
// with an L2 cache policy; completes in this thread's bulk async-group.
__device__ __forceinline__ void bulk_store_global(void* dst, uint32_t src_local, uint32_t bytes, uint64_t policy) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
               "r"(src_local), "r"(bytes), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until the copy engine has read the sources of this thread's bulk copies.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void st_dsmem_f2(uint32_t addr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// ----------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 2-D tiled load of the box at (x = inner coordinate, y = row) into shared
// memory; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// Same, with an L2 eviction-priority hint (policy from createpolicy).
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ----------------------------------------------------------------- L2 prefetch of the next projection
// The next projection's weight k-blocks that its CTAs read right after
// their shared-memory ring, in its CTA geometry (grid x = 128-row weight
// tiles, grid z = k-splits).  A kernel whose own HBM streaming is done (a
// projection past its last load, the latency-bound attention) pulls them
// into L2, so that HBM keeps streaming through its tail.
struct L2Plan {
  int ctas;          // weight tiles x splits of the next projection (0: nothing)
  int n_tiles;       // its 128-row weight tiles
  int kb_per_split;  // its k-blocks per split
  int n_kb;          // its k-blocks in total
  int first;         // first k-block (within a split) to prefetch: its ring holds the ones before
  int count;         // k-blocks per weight tile and split to prefetch
};

__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

// This CTA's share of the plan (one thread issues it).
__device__ __forceinline__ void l2_prefetch_plan(const CUtensorMap* map, const L2Plan& pl) {
  const int G = gridDim.x * gridDim.y * gridDim.z;
  const int me = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  for (int j = me; j < pl.ctas; j += G) {
    const int x = j % pl.n_tiles, z = j / pl.n_tiles;
    const int kb0 = z * pl.kb_per_split, kb1 = min(pl.n_kb, kb0 + pl.kb_per_split);
    for (int i = pl.first; i < pl.first + pl.count && kb0 + i < kb1; ++i)
      tma_prefetch_l2_2d(map, (kb0 + i) * 64, x * 128);
  }
}

// ----------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 inputs, fp32 accumulator.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]^T, bf16 inputs, fp32 accumulator.  A
// (M = 128 rows x 16 k) sits in TMEM: row i in lane i, k-pairs packed into
// 32-bit columns (element 2j in the low half of column j).
__device__ __forceinline__ void tc_mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns from registers; lane i of the warp
// writes TMEM lane (taddr.lane + i).  The warp must be converged; call
// tc_wait_st() before signalling that the columns are written.
__device__ __forceinline__ void tc_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns from registers (as tc_st_32x32b_x32).
__device__ __forceinline__ void tc_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// 32 lanes x 8 consecutive 32-bit columns from registers.
__device__ __forceinline__ void tc_st_32x32b_x8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Four E4M3 codes (bytes of q, lowest byte first) -> four bf16 values as two
// bf16x2 words (lower code in the low half).  A code c = s.eeee.mmm becomes
// the bf16 bit pattern s at bit 15 and eeee.mmm at bits 4-10: a bf16 with
// exponent field eeee and mantissa mmm0000, whose value is exactly the
// code's value times 2^-120 (bf16's exponent bias is 127, E4M3's 7, and
// bf16's subnormals line up with E4M3's: m/8 * 2^-126 against m/8 * 2^-6).
// One bf16 multiply by 2^120 then restores the value; it is exact, since the
// result has 4 significant bits and lies in bf16's normal range.  Integer
// and bf16x2 instructions only, no conversion instructions.
__device__ __forceinline__ void e4m3x4_to_bf16x4(uint32_t q, uint32_t& w0, uint32_t& w1) {
  const uint32_t x0 = __byte_perm(q, 0u, 0x1404);  // bytes [0, c0, 0, c1]
  const uint32_t x1 = __byte_perm(q, 0u, 0x3424);  // bytes [0, c2, 0, c3]
  const uint32_t y0 = ((x0 & 0x7F007F00u) >> 4) | (x0 & 0x80008000u);
  const uint32_t y1 = ((x1 & 0x7F007F00u) >> 4) | (x1 & 0x80008000u);
  constexpr uint32_t k2p120 = 0x7B807B80u;  // bf16x2 {2^120, 2^120}
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(w0) : "r"(y0), "r"(k2p120));
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(w1) : "r"(y1), "r"(k2p120));
}

// Arrive once on `bar` when every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns; lane i of the warp gets TMEM lane
// (taddr.lane + i).  The warp must be converged.
__device__ __forceinline__ void tc_ld_32x32b_x16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor for a K-major operand tile whose rows are
// 128 bytes (64 bf16) written by TMA with 128-byte swizzling: 8-row groups
// 1024 bytes apart (stride byte offset), leading byte offset unused,
// descriptor version 1 (bits 46-48), swizzle mode 2 = 128B (bits 61-63).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Shared-memory matrix descriptor with 128-byte swizzling and explicit
// leading / stride byte offsets.  K-major operands: rows of 128 bytes, 8-row
// groups `sbo` apart (lbo unused).  MN-major operands: 64 MN-elements per
// 128-byte row, K rows 128 bytes apart, 8-row K groups `sbo` apart and the
// next 64 MN-elements `lbo` bytes away.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16 with fp16 A and B (format
// 0) and an fp32 accumulator; b_mn: B is MN-major (bit 16).
__host__ __device__ constexpr uint32_t mma_idesc_f16_f32(int m, int n, bool b_mn) {
  return (1u << 4) | (b_mn ? (1u << 16) : 0u) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// tcgen05.ld without the trailing wait: several loads may be in flight; call
// tc_wait_ld() before using any of the registers.
__device__ __forceinline__ void tc_ld_32x32b_x16_nw(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits
// 4-5 = 1), A and B bf16 (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 =
// 0), N/8 at bits 17-22, M/16 at bits 24-28.
__host__ __device__ constexpr uint32_t mma_idesc_bf16_f32(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// ----------------------------------------------------------------- scalar helpers
template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <>
__device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// An activation that feeds a tensor-core GEMM.  fp32 workloads store the
// value; bf16 workloads store the exact two-term split hi = bf16(v),
// lo = bf16(v - hi), which the GEMM consumes as two MMAs (|v - hi - lo| is
// within 2^-17 |v|).
template <typename T>
struct ActOut;
template <>
struct ActOut<float> {
  float* hi;
  float* lo;  // unused
  __device__ __forceinline__ void put(long long i, float v) const { hi[i] = v; }
};
template <>
struct ActOut<__nv_bfloat16> {
  __nv_bfloat16* hi;
  __nv_bfloat16* lo;
  __device__ __forceinline__ void put(long long i, float v) const {
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    hi[i] = h;
    lo[i] = __float2bfloat16_rn(v - __bfloat162float(h));
  }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum over blockDim.x threads (multiple of 32, <= 1024); result in all threads.
__device__ __forceinline__ float block_sum(float v, float* scratch32) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) scratch32[warp] = v;
  __syncthreads();
  float t = lane < nw ? scratch32[lane] : 0.f;
  return warp_sum(t);
}

}  // namespace dflash

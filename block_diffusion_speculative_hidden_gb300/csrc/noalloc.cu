// dflash_gemm_bf16_noalloc: the projection kernel for callers that cannot
// allocate device memory.
//
// Some callers of this library must not call cudaMalloc themselves or have
// it called for them: processes whose device memory is handed in full to
// another allocator up front (a framework's caching allocator or a serving
// engine's KV pool reserve nearly all of HBM, so a stray allocation fails or
// fragments it), and code that must not pay cudaMalloc's implicit device-wide
// synchronisation.  The regular dflash_gemm_bf16 writes split-K partials to
// a buffer the caller provides; this variant keeps them in a fixed array in
// the library's own device memory instead, and the caller passes only the
// inputs and the output.
//
// The array is a file-scope __device__ object: every GPU that loads the
// library holds it until the process exits.  Host code cannot use its name
// as a device address, so the first call on each device looks the address up
// with cudaGetSymbolAddress (with that device current) and caches it.
#include "common.cuh"
#include "internal.h"

namespace {

using namespace dflash;

constexpr size_t kScratchFloats = size_t(2) << 20;  // 8 MiB
constexpr size_t kReservedFloats = 64;              // slot 0: the status word
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

float* g_scratch_addr[kMaxDevices] = {};  // per device, set on first use

__global__ void k_sum_splits(const float* __restrict__ part, long long plane, int splits, float* __restrict__ out) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= plane) return;
  float v = part[i];
  for (int s = 1; s < splits; ++s) v += part[s * plane + i];
  out[i] = v;
}

}  // namespace

extern "C" dflash_status dflash_gemm_bf16_noalloc(const void* W, int N, int K, const void* X, const void* X_lo,
                                                  int M, float* out, int splits, int* splits_used, int* status,
                                                  dflash_stream stream) {
  if (W == nullptr || X == nullptr || out == nullptr || N < 1 || K < 8 || K % 8 || M < 1 || splits < 1)
    return DFLASH_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(W) % 16 || reinterpret_cast<uintptr_t>(X) % 16 ||
      reinterpret_cast<uintptr_t>(X_lo) % 16)
    return DFLASH_ERR_INVALID_ARG;
  const int n_kb = gemm_kb(K);
  const int want = splits < n_kb ? splits : n_kb;
  const int per = (n_kb + want - 1) / want;
  const int s_used = (n_kb + per - 1) / per;
  const long long plane = static_cast<long long>(M) * N;
  if (static_cast<unsigned long long>(s_used) * plane > kScratchFloats - kReservedFloats)
    return DFLASH_ERR_TOO_LARGE;  // nothing enqueued
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DFLASH_ERR_CUDA;
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return DFLASH_ERR_CUDA;
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  float* scratch = g_scratch_addr[dev];
  // with no caller status word, the kernel's flags go to the array's
  // reserved slot, which nothing reads back: such a call does not report a
  // device-side failure (the header says so)
  int* st = status != nullptr ? status : reinterpret_cast<int*>(scratch);
  if (status == nullptr && cudaMemsetAsync(st, 0, sizeof(int), stream) != cudaSuccess) return DFLASH_ERR_CUDA;
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
  g.out = scratch + kReservedFloats;  // every [split][m][n] element is written before it is read
  g.split_stride = plane;
  g.ldo = N;
  if (gemm_launch_uncached(st, g, stream) != cudaSuccess) return DFLASH_ERR_CUDA;
  const int threads = 256;
  k_sum_splits<<<static_cast<unsigned>((plane + threads - 1) / threads), threads, 0, stream>>>(
      scratch + kReservedFloats, plane, s_used, out);
  if (cudaGetLastError() != cudaSuccess) return DFLASH_ERR_CUDA;
  return DFLASH_OK;
}

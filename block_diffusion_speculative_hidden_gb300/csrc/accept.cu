// Lossless acceptance (the DFlash Guide, "The Cost Breakdown of Speculative
// Rounds": the longest valid prefix tau <= gamma is accepted; the stable-lab
// chapter: the output distribution is exactly the target's).
//
// Greedy: one warp per sequence; lane i compares d_i with y_i, a ballot finds
// the first mismatch.
//
// Stochastic: one CTA per sequence walks the block.  Per position it makes
// one pass over the target logits row for its max and sum of exponentials,
// tests u_i < min(1, p_i(d_i)/q_i(d_i)), and on the first reject (or at the
// bonus position) draws from max(0, p - q) by an exponential race,
// argmax_v r(v) / -ln U_v.  Uniforms come from Philox4x32-10 (Salmon et al.,
// SC'11) keyed by the seed, counter (v, i | stream << 16, b, round).
#include "common.cuh"
#include "kernels.cuh"

namespace dflash {

__global__ void k_accept_greedy(int B, int K, const int32_t* __restrict__ d, const int32_t* __restrict__ y,
                                int32_t* tau_out, int32_t* emitted, int32_t* n_emit) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  const bool mis = lane < K && d[b * K + lane] != y[b * (K + 1) + lane];
  const unsigned mask = __ballot_sync(0xffffffffu, mis);
  const int tau = mask ? __ffs(mask) - 1 : K;
  if (lane <= K) emitted[b * (K + 1) + lane] = lane <= tau ? y[b * (K + 1) + lane] : -1;
  if (lane == 0) {
    tau_out[b] = tau;
    n_emit[b] = tau + 1;
  }
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
    k.x += 0x9E3779B9u;
    k.y += 0xBB67AE85u;
  }
  return c;
}

// ((x >> 9) + 1/2) * 2^-23: exact in fp32, strictly inside (0, 1)
__device__ __forceinline__ float uniform_u32(uint32_t x) {
  return (static_cast<float>(x >> 9) + 0.5f) * 1.1920928955078125e-07f;
}

__device__ __forceinline__ float rng_uniform(uint2 key, uint32_t rnd, uint32_t b, uint32_t i, uint32_t stream,
                                             uint32_t v) {
  return uniform_u32(philox4x32_10(make_uint4(v, i | (stream << 16), b, rnd), key).x);
}

// argmax over (key, v) with ties to the lower v
__device__ __forceinline__ void better(float& k, int& v, float ok, int ov) {
  if (ok > k || (ok == k && ov < v)) {
    k = ok;
    v = ov;
  }
}

constexpr int kAccThreads = 1024;

__global__ void __launch_bounds__(kAccThreads) k_accept_stochastic(int K, int V, const int32_t* __restrict__ d,
                                                                   const float* __restrict__ z,
                                                                   const float* __restrict__ q, float invT,
                                                                   uint2 key, uint32_t rnd_host,
                                                                   int* round_ctr, int32_t* tau_out,
                                                                   int32_t* emitted, int32_t* n_emit) {
  __shared__ float s_a[32], s_b[32], s_c[32];
  __shared__ int s_i[32], s_j[32];
  __shared__ uint32_t s_rnd;
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // round_ctr (nullable): [0] the device round counter, [1] CTAs done with it
  if (tid == 0)
    s_rnd = round_ctr != nullptr ? static_cast<uint32_t>(*reinterpret_cast<volatile int*>(round_ctr)) : rnd_host;
  __syncthreads();
  const uint32_t rnd = s_rnd;
  int tau = K;
  for (int i = 0; i <= K; ++i) {
    const float* row = z + (static_cast<long long>(b) * (K + 1) + i) * V;
    // pass 1: max and sum of exp of z / T
    float m = -INFINITY, s = 0.f;
    for (int v = tid; v < V; v += kAccThreads) {
      const float x = row[v] * invT;
      if (x > m) {
        s = s * expf(m - x) + 1.f;
        m = x;
      } else {
        s += expf(x - m);
      }
    }
    for (int o = 16; o > 0; o >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, m, o), os = __shfl_xor_sync(0xffffffffu, s, o);
      const float nm = fmaxf(m, om);
      s = (m > -INFINITY ? s * expf(m - nm) : 0.f) + (om > -INFINITY ? os * expf(om - nm) : 0.f);
      m = nm;
    }
    __syncthreads();
    if (lane == 0) {
      s_a[warp] = m;
      s_b[warp] = s;
    }
    __syncthreads();
    if (warp == 0) {
      m = s_a[lane];
      s = s_b[lane];
      for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, o), os = __shfl_xor_sync(0xffffffffu, s, o);
        const float nm = fmaxf(m, om);
        s = (m > -INFINITY ? s * expf(m - nm) : 0.f) + (om > -INFINITY ? os * expf(om - nm) : 0.f);
        m = nm;
      }
      if (lane == 0) {
        s_a[0] = m;
        s_b[0] = s;
      }
    }
    __syncthreads();
    const float M = s_a[0], S = s_b[0];
    const float* qrow = q != nullptr && i < K ? q + (static_cast<long long>(b) * K + i) * V : nullptr;
    int dv = -1;
    if (i < K) {
      dv = d[b * K + i];
      bool acc = false;
      if (dv >= 0 && dv < V) {
        const float pd = expf(row[dv] * invT - M) / S;
        const float qd = qrow != nullptr ? qrow[dv] : 1.f;
        const float u = rng_uniform(key, rnd, b, i, 0, 0);
        acc = qd > 0.f ? (u < fminf(1.f, pd / qd)) : true;
      }
      if (acc) {
        if (tid == 0) emitted[b * (K + 1) + i] = dv;
        continue;
      }
    }
    // exponential race over r(v) = max(0, p(v) - q(v)) (point mass: p with d zeroed),
    // falling back to p when r has no mass
    float kr = -INFINITY, kp = -INFINITY, rsum = 0.f;
    int vr = 0x7fffffff, vp = 0x7fffffff;
    for (int v = tid; v < V; v += kAccThreads) {
      const float pv = expf(row[v] * invT - M) / S;
      float r = pv;
      if (i < K) r = qrow != nullptr ? fmaxf(0.f, pv - qrow[v]) : (v == dv ? 0.f : pv);
      const float e = -logf(rng_uniform(key, rnd, b, i, 1, v));
      if (r > 0.f) better(kr, vr, r / e, v);
      if (pv > 0.f) better(kp, vp, pv / e, v);
      rsum += r;
    }
    for (int o = 16; o > 0; o >>= 1) {
      better(kr, vr, __shfl_xor_sync(0xffffffffu, kr, o), __shfl_xor_sync(0xffffffffu, vr, o));
      better(kp, vp, __shfl_xor_sync(0xffffffffu, kp, o), __shfl_xor_sync(0xffffffffu, vp, o));
      rsum += __shfl_xor_sync(0xffffffffu, rsum, o);
    }
    __syncthreads();
    if (lane == 0) {
      s_a[warp] = kr;
      s_i[warp] = vr;
      s_b[warp] = kp;
      s_j[warp] = vp;
      s_c[warp] = rsum;
    }
    __syncthreads();
    if (warp == 0) {
      kr = s_a[lane];
      vr = s_i[lane];
      kp = s_b[lane];
      vp = s_j[lane];
      rsum = s_c[lane];
      for (int o = 16; o > 0; o >>= 1) {
        better(kr, vr, __shfl_xor_sync(0xffffffffu, kr, o), __shfl_xor_sync(0xffffffffu, vr, o));
        better(kp, vp, __shfl_xor_sync(0xffffffffu, kp, o), __shfl_xor_sync(0xffffffffu, vp, o));
        rsum += __shfl_xor_sync(0xffffffffu, rsum, o);
      }
      if (lane == 0) emitted[b * (K + 1) + i] = rsum > 0.f ? vr : vp;
    }
    tau = i < K ? i : K;
    break;
  }
  for (int j = tau + 1 + tid; j <= K; j += kAccThreads) emitted[b * (K + 1) + j] = -1;
  if (tid == 0) {
    tau_out[b] = tau;
    n_emit[b] = tau + 1;
    // every CTA read the counter before it arrives, so the last to arrive
    // may advance it for the next call
    if (round_ctr != nullptr) {
      __threadfence();
      if (atomicAdd(round_ctr + 1, 1) == static_cast<int>(gridDim.x) - 1) {
        round_ctr[1] = 0;
        atomicAdd(round_ctr, 1);
        __threadfence();
      }
    }
  }
}

cudaError_t launch_accept_greedy(int B, int K, const int32_t* d, const int32_t* y, int32_t* tau, int32_t* emitted,
                                 int32_t* n_emit, bool pdl, cudaStream_t s) {
  return launch_k(k_accept_greedy, dim3((B + 3) / 4), dim3(128), 0, s, dim3(1), pdl, B, K, d, y, tau, emitted,
                  n_emit);
}

cudaError_t launch_accept_stochastic(int B, int K, int V, const int32_t* d, const float* z, const float* q,
                                     float temperature, uint64_t seed, uint64_t round, int* round_ctr,
                                     int32_t* tau, int32_t* emitted, int32_t* n_emit, bool pdl, cudaStream_t s) {
  const uint2 key = make_uint2(static_cast<uint32_t>(seed & 0xffffffffu), static_cast<uint32_t>(seed >> 32));
  return launch_k(k_accept_stochastic, dim3(B), dim3(kAccThreads), 0, s, dim3(1), pdl, K, V, d, z, q,
                  1.0f / temperature, key, static_cast<uint32_t>(round & 0xffffffffu), round_ctr, tau, emitted,
                  n_emit);
}

}  // namespace dflash

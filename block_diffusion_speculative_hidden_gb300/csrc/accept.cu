// Lossless acceptance (the DFlash Guide, "The Cost Breakdown of Speculative
// Rounds": the longest valid prefix tau <= gamma is accepted; the stable-lab
// chapter: the output distribution is exactly the target's).
//
// Greedy: one warp per sequence; lane i compares d_i with y_i, a ballot finds
// the first mismatch.
//
// Stochastic: a thread-block cluster of C CTAs per sequence walks the block
// position by position, each CTA over its own slice of the vocabulary.  Per
// position every CTA reduces its slice of the target logits row to (max, sum
// of exponentials), the CTAs exchange those over distributed shared memory
// and every CTA combines them in rank order, so all hold the same softmax
// normaliser and take the same decision u_i < min(1, p_i(d_i)/q_i(d_i)).
// An accept moves to the next position; the first reject (or the bonus
// position after K accepts) runs one more pass over the slice: an
// exponential race argmax_v r(v) / -ln U_v over r = max(0, p - q), merged the
// same way, ties to the lowest v.  Rows past the first reject are never
// read.  Uniforms come from Philox4x32-10 (Salmon et al., SC'11) keyed by the
// seed, counter (v >> 2, i | stream << 16, b, round), word v & 3: one Philox
// block gives the race keys of four consecutive vocabulary entries.
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

// argmax over (key, v) with ties to the lower v
__device__ __forceinline__ void better(float& k, int& v, float ok, int ov) {
  if (ok > k || (ok == k && ov < v)) {
    k = ok;
    v = ov;
  }
}

// online (max, sum of exp(x - max)) of a set of values, merged with another
__device__ __forceinline__ void ms_merge(float& m, float& s, float om, float os) {
  const float nm = fmaxf(m, om);
  s = (m > -INFINITY ? s * expf(m - nm) : 0.f) + (om > -INFINITY ? os * expf(om - nm) : 0.f);
  m = nm;
}

constexpr int kAccThreads = 256;
constexpr int kAccWarps = kAccThreads / 32;
constexpr int kUnroll = 4;  // vocabulary groups a thread loads at once in the normaliser pass

// The four logits of vocabulary group g (entries 4g .. 4g + 3), scaled by
// 1/T; entries at or past v_end read as -inf.  `vec`: the row is 16-byte
// aligned, so whole groups load as one float4.
__device__ __forceinline__ void load_group(const float* row, int g, int v_end, bool vec, float invT, float (&x)[4]) {
  const int v = 4 * g;
  if (vec && v + 3 < v_end) {
    const float4 t = __ldg(reinterpret_cast<const float4*>(row + v));
    x[0] = t.x * invT;
    x[1] = t.y * invT;
    x[2] = t.z * invT;
    x[3] = t.w * invT;
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = v + j < v_end ? __ldg(row + v + j) * invT : -INFINITY;
  }
}

// One cluster of C CTAs per sequence (the cluster's CTAs are consecutive in
// x); CTA `rank` owns vocabulary groups [g0, g1) (four entries a group).
__global__ void __launch_bounds__(kAccThreads) k_accept_stochastic(int K, int V, int groups_per_cta,
                                                                   const int32_t* __restrict__ d,
                                                                   const float* __restrict__ z,
                                                                   const float* __restrict__ q, float invT,
                                                                   uint2 key, uint32_t rnd_host, int* round_ctr,
                                                                   int32_t* tau_out, int32_t* emitted,
                                                                   int32_t* n_emit) {
  // exchanged over distributed shared memory: per position this CTA's
  // (max, sum) of its slice, and its race result
  __shared__ float s_ms[kBlockK + 1][2];
  __shared__ float s_race_k[2], s_race_sum;
  __shared__ int s_race_v[2];
  __shared__ float s_wa[kAccWarps], s_wb[kAccWarps], s_wc[kAccWarps];
  __shared__ int s_wi[kAccWarps], s_wj[kAccWarps];
  __shared__ float s_M, s_S;
  __shared__ int s_dec;  // 1: the draft at this position is accepted
  __shared__ uint32_t s_rnd;
  pdl_wait();
  pdl_trigger();
  const int C = static_cast<int>(cluster_nctarank());
  const int rank = static_cast<int>(cluster_ctarank());
  const int b = blockIdx.x / C, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_groups = (V + 3) / 4;
  const int g0 = min(n_groups, rank * groups_per_cta), g1 = min(n_groups, g0 + groups_per_cta);
  // round_ctr (nullable): [0] the device round counter, [1] CTAs done with it
  if (tid == 0)
    s_rnd = round_ctr != nullptr ? static_cast<uint32_t>(*reinterpret_cast<volatile int*>(round_ctr)) : rnd_host;
  __syncthreads();
  const uint32_t rnd = s_rnd;
  int tau = K;
  for (int i = 0; i <= K; ++i) {
    const float* row = z + (static_cast<long long>(b) * (K + 1) + i) * V;
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    // pass 1: (max, sum of exp) of z / T over this CTA's slice, four groups
    // of a thread loaded before any is used (loads in flight, not one at a
    // time)
    float m = -INFINITY, sm = 0.f;
    for (int g = g0 + tid; g < g1; g += kUnroll * kAccThreads) {
      float x[kUnroll][4];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (g + u * kAccThreads < g1) {
          load_group(row, g + u * kAccThreads, V, vec, invT, x[u]);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) x[u][j] = -INFINITY;
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        float bm = fmaxf(fmaxf(x[u][0], x[u][1]), fmaxf(x[u][2], x[u][3]));
        if (bm == -INFINITY) continue;
        float bs = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) bs += x[u][j] == -INFINITY ? 0.f : expf(x[u][j] - bm);
        ms_merge(m, sm, bm, bs);
      }
    }
    for (int o = 16; o > 0; o >>= 1) ms_merge(m, sm, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, sm, o));
    if (lane == 0) {
      s_wa[warp] = m;
      s_wb[warp] = sm;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kAccWarps; ++w) ms_merge(m, sm, s_wa[w], s_wb[w]);
      s_ms[i][0] = m;
      s_ms[i][1] = sm;
    }
    // every CTA's slice is reduced: combine them in rank order
    cluster_arrive();
    cluster_wait();
    if (tid == 0) {
      float M = -INFINITY, S = 0.f;
      for (int r = 0; r < C; ++r)
        ms_merge(M, S, ld_dsmem_f32(dsmem_map(smem_u32(&s_ms[i][0]), r)), ld_dsmem_f32(dsmem_map(smem_u32(&s_ms[i][1]), r)));
      s_M = M;
      s_S = S;
      int acc = 0, dv = -1;
      if (i < K) {
        dv = d[b * K + i];
        if (dv >= 0 && dv < V) {
          const float pd = expf(__ldg(row + dv) * invT - M) / S;
          const float qd = q != nullptr ? __ldg(q + (static_cast<long long>(b) * K + i) * V + dv) : 1.f;
          const float u = uniform_u32(philox4x32_10(make_uint4(0u, static_cast<uint32_t>(i), b, rnd), key).x);
          acc = qd > 0.f ? (u < fminf(1.f, pd / qd) ? 1 : 0) : 1;
        }
        if (acc && rank == 0) emitted[b * (K + 1) + i] = dv;
      }
      s_dec = acc;
    }
    __syncthreads();
    if (s_dec) continue;
    // the first reject, or the bonus position: exponential race over
    // r(v) = max(0, p(v) - q(v)) (point mass: p with d zeroed), falling
    // back to p when r has no mass.  With the point-mass q (and at the bonus
    // position) r is p off d, so the keys drop the common factor 1/S (an
    // argmax does not see it), no second race over p is run (it could only
    // differ from the first at d) and r has no mass only when no entry but d
    // has any probability, when the fallback draws d itself.
    const float M = s_M, invS = 1.f / s_S;
    const int dv = i < K ? d[b * K + i] : -1;
    const float* qrow = q != nullptr && i < K ? q + (static_cast<long long>(b) * K + i) * V : nullptr;
    const bool pmass = qrow == nullptr;
    float kr = -INFINITY, kp = -INFINITY, rsum = 0.f;
    int vr = 0x7fffffff, vp = 0x7fffffff;
    // two groups a step: their loads and their Philox blocks are independent
    for (int g = g0 + tid; g < g1; g += 2 * kAccThreads) {
      float x[2][4];
      uint4 w[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int gu = g + u * kAccThreads;
        if (gu < g1) {
          load_group(row, gu, V, vec, invT, x[u]);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) x[u][j] = -INFINITY;
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u)
        w[u] = philox4x32_10(
            make_uint4(static_cast<uint32_t>(g + u * kAccThreads), static_cast<uint32_t>(i) | (1u << 16), b, rnd), key);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int gu = g + u * kAccThreads;
        if (gu >= g1) break;
        const uint32_t wv[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int v = 4 * gu + j;
          if (v >= V) break;
          const float inv_e = __frcp_rn(-logf(uniform_u32(wv[j])));  // 1 / E_v
          if (pmass) {
            const float pv = expf(x[u][j] - M);  // p(v) S
            if (pv > 0.f && v != dv) better(kr, vr, pv * inv_e, v);
          } else {
            const float pv = expf(x[u][j] - M) * invS;
            const float r = fmaxf(0.f, pv - __ldg(qrow + v));
            if (r > 0.f) better(kr, vr, r * inv_e, v);
            if (pv > 0.f) better(kp, vp, pv * inv_e, v);
            rsum += r;
          }
        }
      }
    }
    for (int o = 16; o > 0; o >>= 1) {
      better(kr, vr, __shfl_xor_sync(0xffffffffu, kr, o), __shfl_xor_sync(0xffffffffu, vr, o));
      better(kp, vp, __shfl_xor_sync(0xffffffffu, kp, o), __shfl_xor_sync(0xffffffffu, vp, o));
      rsum += __shfl_xor_sync(0xffffffffu, rsum, o);
    }
    if (lane == 0) {
      s_wa[warp] = kr;
      s_wi[warp] = vr;
      s_wb[warp] = kp;
      s_wj[warp] = vp;
      s_wc[warp] = rsum;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kAccWarps; ++w) {
        better(kr, vr, s_wa[w], s_wi[w]);
        better(kp, vp, s_wb[w], s_wj[w]);
        rsum += s_wc[w];
      }
      s_race_k[0] = kr;
      s_race_v[0] = vr;
      s_race_k[1] = kp;
      s_race_v[1] = vp;
      s_race_sum = rsum;
    }
    cluster_arrive();
    cluster_wait();
    if (tid == 0 && rank == 0) {
      float KR = -INFINITY, KP = -INFINITY, RS = 0.f;
      int VR = 0x7fffffff, VP = 0x7fffffff;
      for (int r = 0; r < C; ++r) {
        better(KR, VR, ld_dsmem_f32(dsmem_map(smem_u32(&s_race_k[0]), r)),
               static_cast<int>(__float_as_uint(ld_dsmem_f32(dsmem_map(smem_u32(&s_race_v[0]), r)))));
        better(KP, VP, ld_dsmem_f32(dsmem_map(smem_u32(&s_race_k[1]), r)),
               static_cast<int>(__float_as_uint(ld_dsmem_f32(dsmem_map(smem_u32(&s_race_v[1]), r)))));
        RS += ld_dsmem_f32(dsmem_map(smem_u32(&s_race_sum), r));
      }
      // point mass: r has mass iff some entry other than d won a key
      emitted[b * (K + 1) + i] = pmass ? (KR > -INFINITY ? VR : dv) : (RS > 0.f ? VR : VP);
    }
    tau = i < K ? i : K;
    break;
  }
  if (rank == 0) {
    for (int j = tau + 1 + tid; j <= K; j += kAccThreads) emitted[b * (K + 1) + j] = -1;
    if (tid == 0) {
      tau_out[b] = tau;
      n_emit[b] = tau + 1;
    }
  }
  if (tid == 0 && round_ctr != nullptr) {
    // every CTA read the counter before it arrives, so the last to arrive
    // may advance it for the next call
    __threadfence();
    if (atomicAdd(round_ctr + 1, 1) == static_cast<int>(gridDim.x) - 1) {
      round_ctr[1] = 0;
      atomicAdd(round_ctr, 1);
      __threadfence();
    }
  }
  // no CTA leaves while a peer may still read its shared memory
  cluster_arrive();
  cluster_wait();
}

cudaError_t launch_accept_greedy(int B, int K, const int32_t* d, const int32_t* y, int32_t* tau, int32_t* emitted,
                                 int32_t* n_emit, bool pdl, cudaStream_t s) {
  return launch_k(k_accept_greedy, dim3((B + 3) / 4), dim3(128), 0, s, dim3(1), pdl, B, K, d, y, tau, emitted,
                  n_emit);
}

cudaError_t launch_accept_stochastic(int B, int K, int V, const int32_t* d, const float* z, const float* q,
                                     float temperature, uint64_t seed, uint64_t round, int* round_ctr,
                                     int32_t* tau, int32_t* emitted, int32_t* n_emit, int num_sms, bool pdl,
                                     cudaStream_t s) {
  const uint2 key = make_uint2(static_cast<uint32_t>(seed & 0xffffffffu), static_cast<uint32_t>(seed >> 32));
  // CTAs per sequence: enough clusters to cover every SM about four times, at
  // most 8 (a portable cluster), each slice at least 512 groups
  const int n_groups = (V + 3) / 4;
  int C = 1;
  while (C < 8 && B * C < 4 * num_sms && n_groups / (2 * C) >= 512) C *= 2;
  const int per = (n_groups + C - 1) / C;
  return launch_k(k_accept_stochastic, dim3(B * C), dim3(kAccThreads), 0, s, dim3(C), pdl, K, V, per, d, z, q,
                  1.0f / temperature, key, static_cast<uint32_t>(round & 0xffffffffu), round_ctr, tau, emitted,
                  n_emit);
}

}  // namespace dflash

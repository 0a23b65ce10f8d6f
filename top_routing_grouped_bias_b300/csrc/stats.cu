// Routing side statistics of one routing decision.
//
// Pages: "MOE 专家选择与路由机制" §五 (load-balancing loss N * sum_i f_i P_i with
// f_i the share of assignments to expert i and P_i its mean router
// probability; router z-loss, the mean squared log-sum-exp of the logits) and
// §十三 (per-expert load and routing entropy are the quantities to monitor).
//
// Router probabilities are softmax(z) for a softmax router and the sigmoid
// scores divided by their per-token sum for a sigmoid router.
//
// Two launches, deterministic (fixed summation order, integer counts):
//   partial  one block per 64 tokens: the block's logits are staged in shared
//            memory (64 x N floats, or chunks of 16384 floats for N > 256)
//            with wide coalesced loads; then per-token max / normaliser /
//            lse^2 / entropy (warp per token, which also overwrites the token's
//            staged logits with its probabilities), per-expert probability
//            sums in token order and assignment counts
//   final    a warp per quantity column (P_e, counts_e, lse^2, entropy) sums
//            the block partials in block order; the last block to finish
//            (an atomic ticket, no waiting) forms L_bal from the written
//            P_e and f_e in a fixed order, and writes
//            [L_bal, L_z, entropy, P_0..P_{N-1}, f_0..f_{N-1}]
#include <math.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kTok = kStatsTokensPerBlock;  // 64 tokens per block

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

constexpr int kStageFloats = 16384;  // logits staged per pass: 64 KB
constexpr int kMaxExpertPasses = 4;  // N <= 1024 experts, 256 per pass

// Tokens of one staged chunk: the whole 64-token block for N <= 256.
inline int stats_chunk(int N) { return N * kTok <= kStageFloats ? kTok : kStageFloats / N; }

__global__ void __launch_bounds__(256, 4) stats_partial_kernel(StatsArgs a, int chunk) {
  __shared__ float s_lse2[kTok], s_ent[kTok];
  __shared__ float s_part[256];
  extern __shared__ __align__(16) unsigned char stats_smem[];
  const int N = a.N;
  float* s_z = reinterpret_cast<float*>(stats_smem);  // [chunk][N]
  int* s_cnt = reinterpret_cast<int*>(stats_smem + static_cast<size_t>(chunk) * N * 4);  // [N]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool softmax = a.score == MOE_SCORE_SOFTMAX;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTok;
  const int nvalid = a.T - t0 < kTok ? static_cast<int>(a.T - t0) : kTok;
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.ticket = 0u;  // read by the final kernel
  for (int e = threadIdx.x; e < N; e += blockDim.x) s_cnt[e] = 0;
  // tokens past T add nothing to the loss sums
  for (int lt = nvalid + static_cast<int>(threadIdx.x); lt < kTok; lt += blockDim.x) {
    s_lse2[lt] = 0.f;
    s_ent[lt] = 0.f;
  }
  // per-expert probability sums: with few experts several threads share an
  // expert, each summing every ns-th token in order; the slices are then
  // added in slice order (fixed order, deterministic)
  const int ns = N >= 256 ? 1 : (256 / N < 32 ? 256 / N : 32);
  const int epp = 256 / ns;  // experts per pass
  const int sl = threadIdx.x / epp, ecol = threadIdx.x % epp;
  float acc[kMaxExpertPasses];
#pragma unroll
  for (int p = 0; p < kMaxExpertPasses; ++p) acc[p] = 0.f;

  for (int c0 = 0; c0 < nvalid; c0 += chunk) {
    const int nt = nvalid - c0 < chunk ? nvalid - c0 : chunk;
    const float* src = a.logits + (t0 + c0) * N;
    const int nf = nt * N;
    __syncthreads();  // the previous chunk is fully consumed
    // ---- stage nt contiguous rows: eight 16-byte loads in flight per thread
    int done = 0;
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
      const float4* s4 = reinterpret_cast<const float4*>(src);
      float4* d4 = reinterpret_cast<float4*>(s_z);
      const int n4 = nf >> 2;
      for (int i0 = threadIdx.x; i0 < n4; i0 += 256 * 8) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (i0 + 256 * u < n4) v[u] = s4[i0 + 256 * u];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (i0 + 256 * u < n4) d4[i0 + 256 * u] = v[u];
      }
      done = n4 << 2;
    }
    for (int i = done + threadIdx.x; i < nf; i += 256) s_z[i] = src[i];
    __syncthreads();

    // ---- per-token statistics, a warp per token; each token's row of the
    // staged tile is then overwritten in place by its probabilities p_e
    for (int lt = warp; lt < nt; lt += 8) {
      float* z = s_z + lt * N;
      float m = -INFINITY;
      for (int e = lane; e < N; e += 32) m = fmaxf(m, z[e]);
      m = warp_max_f(m);
      float se = 0.f, sze = 0.f, ssig = 0.f;
      for (int e = lane; e < N; e += 32) {
        const float ze = z[e];
        const float ex = expf(ze - m);
        se += ex;
        sze += ex * (ze - m);
        if (!softmax) ssig += 1.f / (1.f + expf(-ze));
        else z[e] = ex;  // the softmax numerator, divided below
      }
      se = warp_sum_f(se);
      sze = warp_sum_f(sze);
      const float lse = m + logf(se);
      float norm, ent;
      if (softmax) {
        norm = se;
        ent = logf(se) - sze / se;  // -sum p log p with log p = z - m - log(se)
        for (int e = lane; e < N; e += 32) z[e] = z[e] / se;
      } else {
        norm = warp_sum_f(ssig);
        float h = 0.f;
        for (int e = lane; e < N; e += 32) {
          const float p = 1.f / (1.f + expf(-z[e])) / norm;
          if (p > 0.f) h -= p * logf(p);
          z[e] = p;
        }
        ent = warp_sum_f(h);
      }
      if (lane == 0) {
        s_lse2[c0 + lt] = lse * lse;
        s_ent[c0 + lt] = ent;
      }
    }
    __syncthreads();

    // ---- per-expert probability sums over this chunk's tokens, in order
    // (the p_e written above: the same values as exp(z - m) / se, or the
    // sigmoid over its token sum)
#pragma unroll
    for (int p = 0; p < kMaxExpertPasses; ++p) {
      const int e = p * epp + ecol;
      if (e < N && sl < ns) {
        int lt = c0 + (sl - c0 % ns + ns) % ns;  // first token of slice sl
#pragma unroll 8
        for (; lt < c0 + nt; lt += ns) acc[p] += s_z[(lt - c0) * N + e];
      }
    }
  }
  __syncthreads();
  // assignment counts (integers: order-independent)
  for (int i = threadIdx.x; i < kTok * a.k; i += blockDim.x) {
    const int64_t t = t0 + i / a.k;
    if (t < a.T) {
      const int e = a.idx[t0 * a.k + i];
      if (e >= 0 && e < N) atomicAdd(&s_cnt[e], 1);
    }
  }
  __syncthreads();
  // row-major [2N + 2][blocks]: each quantity's partials over the blocks
  // are contiguous for the final reduction
  const size_t nbk = gridDim.x;
  float* P = a.partial + blockIdx.x;
#pragma unroll
  for (int p = 0; p < kMaxExpertPasses; ++p) {
    if (p * epp >= N) break;
    s_part[threadIdx.x] = acc[p];
    __syncthreads();
    if (static_cast<int>(threadIdx.x) < epp && p * epp + static_cast<int>(threadIdx.x) < N) {
      float tot = 0.f;
      for (int q = 0; q < ns; ++q) tot += s_part[q * epp + threadIdx.x];
      P[(p * epp + threadIdx.x) * nbk] = tot;
    }
    __syncthreads();
  }
  for (int e = threadIdx.x; e < N; e += blockDim.x) P[(N + e) * nbk] = static_cast<float>(s_cnt[e]);
  if (threadIdx.x == 0) {
    float l2 = 0.f, en = 0.f;
    for (int lt = 0; lt < kTok; ++lt) {
      l2 += s_lse2[lt];
      en += s_ent[lt];
    }
    P[(2 * N) * nbk] = l2;
    P[(2 * N + 1) * nbk] = en;
  }
}

constexpr int kFinalWarps = 8;

// A warp per column c of the partials: c < N the probability sums of expert
// c, N <= c < 2N the counts of expert c - N, then lse^2 and entropy. Each lane
// adds its blocks (lane, lane + 32, ...) in block order, sixteen loads in
// flight, then a fixed butterfly. The last block to finish forms L_bal from
// the written P_e and f_e: lane l adds f_e * P_e over e = l, l + 32, ... in
// order, then the same butterfly. Deterministic.
__global__ void __launch_bounds__(kFinalWarps * 32) stats_final_kernel(StatsArgs a, int nb) {
  __shared__ bool s_last;
  const int N = a.N;
  const int lane = threadIdx.x & 31;
  const int c = blockIdx.x * kFinalWarps + (threadIdx.x >> 5);
  const size_t nbk = static_cast<size_t>(nb);
  const float invT = 1.f / static_cast<float>(a.T);
  const float invTk = 1.f / (static_cast<float>(a.T) * static_cast<float>(a.k));
  if (c < 2 * N + 2) {
    const float* pc = a.partial + c * nbk;
    float sum = 0.f;
    for (int b0 = lane; b0 < nb; b0 += 32 * 16) {
      float v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int b = b0 + 32 * u;
        v[u] = b < nb ? pc[b] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) sum += v[u];
    }
    sum = warp_sum_f(sum);
    if (lane == 0) {
      if (c < N) a.out[3 + c] = sum * invT;                     // P_e
      else if (c < 2 * N) a.out[3 + c] = sum * invTk;           // f_e
      else a.out[1 + (c - 2 * N)] = sum * invT;                 // L_z, entropy
    }
  }
  // the last block to finish sees every other block's writes
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(a.ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last || threadIdx.x >= 32) return;
  __threadfence();
  float local = 0.f;
  for (int e = lane; e < N; e += 32) local += __ldcg(a.out + 3 + N + e) * __ldcg(a.out + 3 + e);
  local = warp_sum_f(local);
  if (lane == 0) a.out[0] = static_cast<float>(N) * local;
}

}  // namespace

cudaError_t launch_route_stats(const StatsArgs& in, cudaStream_t stream) {
  if (in.T == 0) return cudaMemsetAsync(in.out, 0, sizeof(float) * (3 + 2 * in.N), stream);
  const int nb = static_cast<int>((in.T + kTok - 1) / kTok);
  StatsArgs a = in;
  a.ticket = reinterpret_cast<unsigned*>(a.partial + static_cast<size_t>(nb) * (2 * a.N + 2));
  const int chunk = stats_chunk(a.N);
  const size_t smem = static_cast<size_t>(chunk) * a.N * 4 + static_cast<size_t>(a.N) * 4;
  cudaError_t err = cudaFuncSetAttribute(stats_partial_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  stats_partial_kernel<<<nb, 256, smem, stream>>>(a, chunk);
  const int cols = 2 * a.N + 2;
  stats_final_kernel<<<(cols + kFinalWarps - 1) / kFinalWarps, kFinalWarps * 32, 0, stream>>>(a, nb);
  return cudaGetLastError();
}

}  // namespace moe

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
//   partial  one block per 64 tokens: per-token max / normaliser / lse^2 /
//            entropy (warp per token), then per-expert probability sums in
//            token order and assignment counts
//   final    one block: sums the block partials (a warp per expert column,
//            fixed order) and writes
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

__global__ void __launch_bounds__(256) stats_partial_kernel(StatsArgs a) {
  __shared__ float s_m[kTok], s_norm[kTok], s_lse2[kTok], s_ent[kTok];
  extern __shared__ int s_cnt[];  // [N]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;
  const bool softmax = a.score == MOE_SCORE_SOFTMAX;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTok;
  for (int e = threadIdx.x; e < N; e += blockDim.x) s_cnt[e] = 0;
  for (int lt = warp; lt < kTok; lt += 8) {
    const int64_t t = t0 + lt;
    if (t >= a.T) {
      if (lane == 0) { s_m[lt] = 0.f; s_norm[lt] = 1.f; s_lse2[lt] = 0.f; s_ent[lt] = 0.f; }
      continue;
    }
    const float* z = a.logits + t * N;
    float m = -INFINITY;
    for (int e = lane; e < N; e += 32) m = fmaxf(m, z[e]);
    m = warp_max_f(m);
    float se = 0.f, sze = 0.f, ssig = 0.f;
    for (int e = lane; e < N; e += 32) {
      const float ex = expf(z[e] - m);
      se += ex;
      sze += ex * (z[e] - m);
      if (!softmax) ssig += 1.f / (1.f + expf(-z[e]));
    }
    se = warp_sum_f(se);
    sze = warp_sum_f(sze);
    const float lse = m + logf(se);
    float norm, ent;
    if (softmax) {
      norm = se;
      ent = logf(se) - sze / se;  // -sum p log p with log p = z - m - log(se)
    } else {
      norm = warp_sum_f(ssig);
      float h = 0.f;
      for (int e = lane; e < N; e += 32) {
        const float p = 1.f / (1.f + expf(-z[e])) / norm;
        if (p > 0.f) h -= p * logf(p);
      }
      ent = warp_sum_f(h);
    }
    if (lane == 0) {
      s_m[lt] = m;
      s_norm[lt] = norm;
      s_lse2[lt] = lse * lse;
      s_ent[lt] = ent;
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
  // per-expert probability sums: with few experts several threads share an
  // expert, each summing every ns-th token in order; the slices are then
  // added in slice order (fixed order, deterministic)
  const int ns = N >= 256 ? 1 : (256 / N < 32 ? 256 / N : 32);
  __shared__ float s_part[256];
  for (int e0 = 0; e0 < N; e0 += 256 / ns) {
    const int e = e0 + threadIdx.x % (256 / ns);
    const int sl = threadIdx.x / (256 / ns);
    float acc = 0.f;
    if (e < N && sl < ns) {
      // tokens of this block, in order; loads of eight of them in flight
      const int lt_end = a.T - t0 < kTok ? static_cast<int>(a.T - t0) : kTok;
#pragma unroll 8
      for (int lt = sl; lt < lt_end; lt += ns) {
        const float z = a.logits[(t0 + lt) * N + e];
        acc += softmax ? expf(z - s_m[lt]) / s_norm[lt] : 1.f / (1.f + expf(-z)) / s_norm[lt];
      }
    }
    s_part[threadIdx.x] = acc;
    __syncthreads();
    if (threadIdx.x < 256 / ns && e0 + static_cast<int>(threadIdx.x) < N) {
      float tot = 0.f;
      for (int q = 0; q < ns; ++q) tot += s_part[q * (256 / ns) + threadIdx.x];
      P[(e0 + threadIdx.x) * nbk] = tot;
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

// One block: a warp per expert column (lanes take every 32nd block, in block
// order, then a fixed butterfly), the same for the two loss sums, and a fixed
// block reduction for L_bal. Deterministic.
__global__ void __launch_bounds__(1024) stats_final_kernel(StatsArgs a, int nb) {
  __shared__ float red[32];
  __shared__ float l2en[2];
  const int N = a.N;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const size_t nbk = static_cast<size_t>(nb);
  const float invT = 1.f / static_cast<float>(a.T);
  const float invTk = 1.f / (static_cast<float>(a.T) * static_cast<float>(a.k));
  float local = 0.f;  // lane 0 of each warp: sum of its experts' f_e P_e
  for (int e = w; e < N; e += nw) {
    float ps = 0.f, cs = 0.f;
    const float* pp = a.partial + e * nbk;
    const float* pc = a.partial + (N + e) * nbk;
    for (int b0 = lane; b0 < nb; b0 += 256) {
      // eight of this lane's blocks loaded before they are added, in order
      float vp[8], vc[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int b = b0 + 32 * u;
        vp[u] = b < nb ? pp[b] : 0.f;
        vc[u] = b < nb ? pc[b] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        ps += vp[u];
        cs += vc[u];
      }
    }
    ps = warp_sum_f(ps);
    cs = warp_sum_f(cs);
    const float Pe = ps * invT, fe = cs * invTk;
    if (lane == 0) {
      a.out[3 + e] = Pe;
      a.out[3 + N + e] = fe;
      local += fe * Pe;
    }
  }
  if (w == nw - 1) {
    float l2 = 0.f, en = 0.f;
    const float* pl = a.partial + (2 * N) * nbk;
    const float* pe = a.partial + (2 * N + 1) * nbk;
    for (int b0 = lane; b0 < nb; b0 += 256) {
      float vl[8], ve[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int b = b0 + 32 * u;
        vl[u] = b < nb ? pl[b] : 0.f;
        ve[u] = b < nb ? pe[b] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        l2 += vl[u];
        en += ve[u];
      }
    }
    l2 = warp_sum_f(l2);
    en = warp_sum_f(en);
    if (lane == 0) {
      l2en[0] = l2;
      l2en[1] = en;
    }
  }
  if (lane == 0) red[w] = local;
  __syncthreads();
  if (w == 0) {
    float v = lane < nw ? red[lane] : 0.f;
    v = warp_sum_f(v);
    if (lane == 0) {
      a.out[0] = static_cast<float>(N) * v;
      a.out[1] = l2en[0] * invT;
      a.out[2] = l2en[1] * invT;
    }
  }
}

}  // namespace

cudaError_t launch_route_stats(const StatsArgs& a, cudaStream_t stream) {
  if (a.T == 0) return cudaMemsetAsync(a.out, 0, sizeof(float) * (3 + 2 * a.N), stream);
  const int nb = static_cast<int>((a.T + kTok - 1) / kTok);
  stats_partial_kernel<<<nb, 256, a.N * sizeof(int), stream>>>(a);
  stats_final_kernel<<<1, 1024, 0, stream>>>(a, nb);
  return cudaGetLastError();
}

}  // namespace moe

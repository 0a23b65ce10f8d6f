// Router: logits, scores, top-k selection and gates, one warp per token.
// The logits come from one of three sources: this kernel's own dot products
// (fp32 inputs, N > 256), logits given by the caller, or the partial logits of
// the split tcgen05 GEMM (bf16 from h, N <= 256; grouped_gemm.cu, kLogits),
// which are added here slice by slice in slice order. Selection and gates are
// the same code for all three.
//
// Pages: "MOE 专家选择与路由机制" §二 (z = W_r h + b_r; softmax; TopK; renormalise
// over the selected experts); "MoE：router 怎样选 expert" (softmax over the
// selected logits; sigmoid scores; Switch top-1 without renormalisation);
// "拆解 MoE" (per-expert bias steers selection).
//
// Selection rule: experts are taken in descending selection score; equal
// scores go to the lower index. Without a selection bias the score is monotone
// in the logit for both softmax and sigmoid, so selection compares logits
// directly (no rounding of exp can merge two distinct logits). With a bias the
// selection score is p + bias in fp32.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;

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

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int n = 8;
  __device__ static void load(const __nv_bfloat16* p, float (&f)[8]) {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 t = __bfloat1622float2(b[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
};
template <>
struct Vec<float> {
  static constexpr int n = 4;
  __device__ static void load(const float* p, float (&f)[4]) {
    float4 u = *reinterpret_cast<const float4*>(p);
    f[0] = u.x; f[1] = u.y; f[2] = u.z; f[3] = u.w;
  }
};

// smem per warp: z[N] and (with a bias) q[N].
template <typename T>
__global__ void __launch_bounds__(kRouteWarps * 32) route_warp_kernel(RouteArgs a) {
  extern __shared__ float route_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kRouteWarps + warp;
  if (t >= a.T) return;
  const int N = a.N, k = a.k;
  const bool has_bias = a.sel_bias != nullptr;
  float* z = route_smem + static_cast<size_t>(warp) * N * ((has_bias || a.n_group > 1) ? 2 : 1);
  float* q = z + N;

  // ---- logits ----
  if (a.h != nullptr) {
    constexpr int V = Vec<T>::n;
    const T* hrow = static_cast<const T*>(a.h) + t * a.d;
    const T* W = static_cast<const T*>(a.W_r);
    for (int e0 = 0; e0 < N; e0 += 8) {
      const int ne = min(8, N - e0);
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      for (int c = lane * V; c < a.d; c += 32 * V) {
        float hv[V];
        Vec<T>::load(hrow + c, hv);
#pragma unroll
        for (int ee = 0; ee < 8; ++ee) {
          if (ee < ne) {
            float wv[V];
            Vec<T>::load(W + static_cast<size_t>(e0 + ee) * a.d + c, wv);
#pragma unroll
            for (int i = 0; i < V; ++i) acc[ee] = fmaf(hv[i], wv[i], acc[ee]);
          }
        }
      }
#pragma unroll
      for (int ee = 0; ee < 8; ++ee) acc[ee] = warp_sum(acc[ee]);
      if (lane == 0) {
        for (int ee = 0; ee < ne; ++ee)
          z[e0 + ee] = acc[ee] + (a.b_r != nullptr ? a.b_r[e0 + ee] : 0.f);
      }
    }
  } else if (a.partials != nullptr) {
    // slices added in slice order, four loads in flight
    const size_t slice = static_cast<size_t>(a.T) * a.ld_partial;
    const float* zp = a.partials + static_cast<size_t>(t) * a.ld_partial;
    for (int e = lane; e < N; e += 32) {
      float v = 0.f;
      for (int sl = 0; sl < a.n_partials; sl += 4) {
        float w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) w[u] = sl + u < a.n_partials ? zp[(sl + u) * slice + e] : 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (sl + u < a.n_partials) v += w[u];
      }
      z[e] = v + (a.b_r != nullptr ? a.b_r[e] : 0.f);
    }
  } else {
    const float* zin = a.logits_in + t * N;
    for (int e = lane; e < N; e += 32) z[e] = zin[e];
  }
  __syncwarp();
  if (a.logits_out != nullptr) {
    float* zo = a.logits_out + t * N;
    for (int e = lane; e < N; e += 32) zo[e] = z[e];
  }

  // ---- softmax statistics (global max, sum of exp) ----
  float m = -INFINITY;
  for (int e = lane; e < N; e += 32) m = fmaxf(m, z[e]);
  m = warp_max(m);
  float s = 0.f;
  if (a.score == MOE_SCORE_SOFTMAX) {
    for (int e = lane; e < N; e += 32) s += expf(z[e] - m);
    s = warp_sum(s);
  }

  // ---- selection score ----
  // with group-limited selection the group scores are sums/maxima of the
  // scores themselves, so q = p (+ bias) is formed even without a bias
  const bool grouped = a.n_group > 1;
  const float* sel = z;
  if (has_bias || grouped) {
    for (int e = lane; e < N; e += 32) {
      const float p = a.score == MOE_SCORE_SOFTMAX ? expf(z[e] - m) / s : 1.f / (1.f + expf(-z[e]));
      q[e] = p + (has_bias ? a.sel_bias[e] : 0.f);
    }
    __syncwarp();
    sel = q;
  }

  // ---- group-limited selection: keep the topk_group best groups ----
  uint32_t gkeep = 0xffffffffu;
  int gs = N;
  if (grouped) {
    gs = N / a.n_group;
    float gscore = -INFINITY;
    if (lane < a.n_group) {
      const float* sg = sel + lane * gs;
      if (a.group_rule == 0) {
        for (int i = 0; i < gs; ++i) gscore = fmaxf(gscore, sg[i]);
      } else {
        float tv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) tv[j] = -INFINITY;
        for (int i = 0; i < gs; ++i) {
          float v = sg[i];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (j < a.top_m && v > tv[j]) {
              const float t = tv[j];
              tv[j] = v;
              v = t;
            }
          }
        }
        gscore = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < a.top_m) gscore += tv[j];
      }
    }
    gkeep = 0;
    for (int r = 0; r < a.topk_group; ++r) {
      const bool cand = lane < a.n_group && !((gkeep >> lane) & 1u);
      float best = cand ? gscore : -INFINITY;
      int best_g = cand ? lane : 0x7fffffff;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int og = __shfl_xor_sync(0xffffffffu, best_g, o);
        if (ov > best || (ov == best && og < best_g)) {
          best = ov;
          best_g = og;
        }
      }
      if (best_g < 32) gkeep |= 1u << best_g;
    }
  }

  // ---- top-k: k rounds of a warp arg-max, lowest index on ties ----
  // bit i of `avail`: expert lane + 32 i can still be taken (not yet taken,
  // and its group kept)
  uint32_t avail = 0;
  for (int i = 0, e = lane; e < N; ++i, e += 32)
    if (!grouped || ((gkeep >> (e / gs)) & 1u)) avail |= 1u << i;  // masked group: -inf
  int my_sel = -1;     // lane j < k keeps the expert of slot j
  for (int r = 0; r < k; ++r) {
    float best = -INFINITY;
    int best_e = 0x7fffffff;
    for (int i = 0, e = lane; e < N; ++i, e += 32) {
      if (!((avail >> i) & 1u)) continue;
      const float v = sel[e];
      if (v > best || (v == best && e < best_e)) {
        best = v;
        best_e = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oe = __shfl_xor_sync(0xffffffffu, best_e, o);
      if (ov > best || (ov == best && oe < best_e)) {
        best = ov;
        best_e = oe;
      }
    }
    if (best_e == 0x7fffffff) best_e = 0;  // only reachable with NaN inputs
    if ((best_e & 31) == lane) avail &= ~(1u << (best_e >> 5));
    if (lane == r) my_sel = best_e;
  }

  // ---- gates ----
  const bool mine = lane < k;
  const float zsel = mine ? z[my_sel] : -INFINITY;
  float g = 0.f;
  if (a.score == MOE_SCORE_SOFTMAX) {
    if (a.norm == MOE_NORM_SELECTED) {
      const float ms = warp_max(zsel);
      const float num = mine ? expf(zsel - ms) : 0.f;
      const float den = warp_sum(num);
      g = num / den;
    } else {
      g = mine ? expf(zsel - m) / s : 0.f;
    }
  } else {
    const float sg = mine ? 1.f / (1.f + expf(-zsel)) : 0.f;
    if (a.norm == MOE_NORM_SELECTED) {
      const float den = warp_sum(sg);
      g = sg / den;
    } else {
      g = sg;
    }
  }
  if (mine) {
    a.idx[t * k + lane] = my_sel;
    a.gate[t * k + lane] = g;
  }
}

}  // namespace

cudaError_t launch_route(const RouteArgs& in, cudaStream_t stream) {
  if (in.T == 0) return cudaSuccess;
  RouteArgs a = in;
  if (route_on_tensor_cores(in)) {
    // one slice: the GEMM routes in its epilogue
    if (route_split(in.T, in.d, in.N).splits == 1 && in.n_group <= 1)
      return launch_route_mma(in, stream);
    // split partial logits on the tensor cores, selection below from them
    if (in.partials == nullptr) return cudaErrorInvalidValue;
    const cudaError_t e = launch_route_logits(in, stream);
    if (e != cudaSuccess) return e;
    const RouteSplit rs = route_split(in.T, in.d, in.N);
    a.h = nullptr;
    a.W_r = nullptr;
    a.logits_in = nullptr;
    a.n_partials = rs.splits;
    a.ld_partial = rs.n_pad;
  } else {
    a.partials = nullptr;
  }
  const bool two = a.sel_bias != nullptr || a.n_group > 1;
  const size_t smem = static_cast<size_t>(kRouteWarps) * a.N * (two ? 2 : 1) * sizeof(float);
  const unsigned grid = static_cast<unsigned>((a.T + kRouteWarps - 1) / kRouteWarps);
  cudaError_t err;
  if (a.dtype == MOE_F32) {
    err = cudaFuncSetAttribute(route_warp_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    route_warp_kernel<float><<<grid, kRouteWarps * 32, smem, stream>>>(a);
  } else {
    err = cudaFuncSetAttribute(route_warp_kernel<__nv_bfloat16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    route_warp_kernel<__nv_bfloat16><<<grid, kRouteWarps * 32, smem, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace moe

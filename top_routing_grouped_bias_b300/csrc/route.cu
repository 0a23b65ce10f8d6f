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
//
// Layout: lane l of the token's warp holds experts l + 32 i in registers
// (EPL slots, the smallest of 1, 2, 4, ..., 32 with 32 EPL >= N), so every
// per-expert pass is an unrolled register loop. Group-limited selection
// ("MoE：router 怎样选 expert", group section): groups of N / n_group
// consecutive experts; when that size divides 32 a group is an aligned lane
// segment and its max or top-2 sum comes from butterfly merges inside the
// segment, otherwise one lane per group scans its group in shared memory.
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

// One warp per token.  Expert e = lane + 32 i lives in register slot i of
// its lane (i < EPL, 32 EPL >= N; slots past N hold -inf and are never
// available).  Shared memory per warp: z[N] (read back for the gates) and,
// with a bias or groups, q[N] (for a group pass over groups that are not lane
// segments).
template <typename T, int EPL>
__global__ void __launch_bounds__(kRouteWarps * 32) route_warp_kernel(RouteArgs a) {
  extern __shared__ float route_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kRouteWarps + warp;
  if (t >= a.T) return;
  const int N = a.N, k = a.k;
  const bool has_bias = a.sel_bias != nullptr;
  const bool grouped = a.n_group > 1;
  float* z = route_smem + static_cast<size_t>(warp) * N * ((has_bias || grouped) ? 2 : 1);
  float* q = z + N;

  // ---- logits ----
  float zr[EPL];
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
    __syncwarp();
#pragma unroll
    for (int i = 0; i < EPL; ++i) zr[i] = lane + 32 * i < N ? z[lane + 32 * i] : -INFINITY;
  } else {
    if (a.partials != nullptr) {
      // slices added in slice order; U slices of every slot in flight
      constexpr int U = EPL >= 8 ? 1 : 8 / EPL;
      const size_t slice = static_cast<size_t>(a.T) * a.ld_partial;
      const float* zp = a.partials + static_cast<size_t>(t) * a.ld_partial + lane;
      float acc[EPL];
#pragma unroll
      for (int i = 0; i < EPL; ++i) acc[i] = 0.f;
      for (int sl = 0; sl < a.n_partials; sl += U) {
        float w[EPL][U];
#pragma unroll
        for (int i = 0; i < EPL; ++i)
#pragma unroll
          for (int u = 0; u < U; ++u)
            w[i][u] = lane + 32 * i < N && sl + u < a.n_partials ? zp[(sl + u) * slice + 32 * i] : 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
#pragma unroll
          for (int u = 0; u < U; ++u)
            if (sl + u < a.n_partials) acc[i] += w[i][u];
      }
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        zr[i] = e < N ? acc[i] + (a.b_r != nullptr ? a.b_r[e] : 0.f) : -INFINITY;
      }
    } else {
      const float* zin = a.logits_in + t * N;
#pragma unroll
      for (int i = 0; i < EPL; ++i) zr[i] = lane + 32 * i < N ? zin[lane + 32 * i] : -INFINITY;
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane + 32 * i < N) z[lane + 32 * i] = zr[i];
  }
  if (a.logits_out != nullptr) {
    float* zo = a.logits_out + t * N;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane + 32 * i < N) zo[lane + 32 * i] = zr[i];
  }

  // ---- softmax statistics (global max, sum of exp) ----
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < EPL; ++i) m = fmaxf(m, zr[i]);
  m = warp_max(m);
  float ex[EPL];
  float s = 0.f;
  if (a.score == MOE_SCORE_SOFTMAX) {
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      ex[i] = 0.f;
      if (lane + 32 * i < N) {
        ex[i] = expf(zr[i] - m);
        s += ex[i];
      }
    }
    s = warp_sum(s);
  }

  // ---- selection score ----
  // with group-limited selection the group scores are sums/maxima of the
  // scores themselves, so q = p (+ bias) is formed even without a bias
  int gs = N;
  int m_top = 1;
  bool seg = false;  // every group is an aligned lane segment of one 32-expert chunk
  if (grouped) {
    gs = N / a.n_group;
    m_top = a.group_rule == 0 ? 1 : a.top_m;
    seg = 32 % gs == 0 && m_top <= 2;
  }
  float sr[EPL];
  if (has_bias || grouped) {
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      sr[i] = -INFINITY;
      if (e < N) {
        const float p = a.score == MOE_SCORE_SOFTMAX ? ex[i] / s : 1.f / (1.f + expf(-zr[i]));
        sr[i] = p + (has_bias ? a.sel_bias[e] : 0.f);
        if (grouped && !seg) q[e] = sr[i];
      }
    }
    if (grouped && !seg) __syncwarp();
  } else {
#pragma unroll
    for (int i = 0; i < EPL; ++i) sr[i] = zr[i];
  }

  // ---- group-limited selection: keep the topk_group best groups ----
  // group score = max, or the sum of the top_m selection scores taken in
  // descending order; lane g < n_group ends up with group g's score
  uint32_t gkeep = 0xffffffffu;
  if (grouped) {
    float gscore = -INFINITY;
    if (seg) {
      // the segment's top-2 list by butterfly merges within the segment
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        if (32 * i >= N) break;
        float t0 = sr[i];
        float t1 = -INFINITY;
        for (int o = gs >> 1; o > 0; o >>= 1) {
          const float u0 = __shfl_xor_sync(0xffffffffu, t0, o);
          if (m_top == 2) {
            const float u1 = __shfl_xor_sync(0xffffffffu, t1, o);
            t1 = fmaxf(fminf(t0, u0), fmaxf(t1, u1));
          }
          t0 = fmaxf(t0, u0);
        }
        const float sc = a.group_rule == 0 ? t0 : (m_top == 1 ? 0.f + t0 : (0.f + t0) + t1);
        const float v = __shfl_sync(0xffffffffu, sc, (lane * gs) & 31);
        if (lane < a.n_group && (lane * gs) >> 5 == i) gscore = v;
      }
    } else if (lane < a.n_group) {
      const float* sg = q + lane * gs;
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
            if (j < m_top && v > tv[j]) {
              const float tt = tv[j];
              tv[j] = v;
              v = tt;
            }
          }
        }
        gscore = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < m_top) gscore += tv[j];
      }
    }
    // group g is kept when fewer than topk_group groups precede it in the
    // order (score descending, index ascending)
    int rank = 0;
    for (int h = 0; h < a.n_group; ++h) {
      const float sh = __shfl_sync(0xffffffffu, gscore, h);
      if (sh > gscore || (sh == gscore && h < lane)) ++rank;
    }
    gkeep = __ballot_sync(0xffffffffu, lane < a.n_group && rank < a.topk_group);
  }

  // ---- top-k: k rounds of a warp arg-max, lowest index on ties ----
  // bit i of `avail`: slot i can still be taken (a real expert, not yet
  // taken, its group kept)
  uint32_t avail = 0;
  if (!grouped) {
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane + 32 * i < N) avail |= 1u << i;
  } else if (seg) {
    const int per = 32 / gs, lg = lane / gs;  // group of slot i: i * per + lg
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane + 32 * i < N && ((gkeep >> (i * per + lg)) & 1u)) avail |= 1u << i;
  } else {
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < N && ((gkeep >> (e / gs)) & 1u)) avail |= 1u << i;
    }
  }
  __syncwarp();  // z[] of every lane is visible before the gates read it
  int my_sel = -1;     // lane j < k keeps the expert of slot j
  for (int r = 0; r < k; ++r) {
    float best = -INFINITY;
    int best_e = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const float v = sr[i];
      const int e = lane + 32 * i;
      if (((avail >> i) & 1u) && (v > best || (v == best && e < best_e))) {
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

template <typename T, int EPL>
cudaError_t launch_selection(const RouteArgs& a, unsigned grid, size_t smem, cudaStream_t stream) {
  const cudaError_t err = cudaFuncSetAttribute(
      route_warp_kernel<T, EPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  route_warp_kernel<T, EPL><<<grid, kRouteWarps * 32, smem, stream>>>(a);
  return cudaGetLastError();
}

// register slots per lane: the smallest of 1, 2, 4, 8, 16, 32 with 32 EPL >= N
template <typename T>
cudaError_t launch_selection(const RouteArgs& a, unsigned grid, size_t smem, cudaStream_t stream) {
  if (a.N <= 32) return launch_selection<T, 1>(a, grid, smem, stream);
  if (a.N <= 64) return launch_selection<T, 2>(a, grid, smem, stream);
  if (a.N <= 128) return launch_selection<T, 4>(a, grid, smem, stream);
  if (a.N <= 256) return launch_selection<T, 8>(a, grid, smem, stream);
  if (a.N <= 512) return launch_selection<T, 16>(a, grid, smem, stream);
  return launch_selection<T, 32>(a, grid, smem, stream);
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
  if (a.dtype == MOE_F32) return launch_selection<float>(a, grid, smem, stream);
  return launch_selection<__nv_bfloat16>(a, grid, smem, stream);
}

}  // namespace moe

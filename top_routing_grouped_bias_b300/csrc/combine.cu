// Combine: weighted scatter-ADD of the expert outputs back to their tokens.
//
// Pages: "MoE：router 怎样选 expert", 选好以后 (outputs are weighted and added,
// not overwritten or concatenated); "【大模型】MoE（专家混合模型）简介" §3 ④
// (restore token order, fuse by router weight); "MOE 专家选择与路由机制" §八
// (shared-expert term).
//
//   out[t] = y_shared[t] + sum_{j<k} gate[t,j] * y_rows[inv[t*k+j]]
//
// A warp takes one token at a time and reads its k rows and gates once; its
// lanes stride over the row's 16-byte vectors. fp32 accumulation in slot
// order (deterministic), rounded once to the output dtype.
#include <cuda_bf16.h>

#include "internal.h"

namespace moe {
namespace {

__device__ __forceinline__ void unpack(const uint4& u, float (&f)[8], __nv_bfloat16*) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(b[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ void unpack(const uint4& u, float (&f)[4], float*) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ uint4 pack(const float (&f)[8], __nv_bfloat16*) {
  uint4 u;
  __nv_bfloat162* b = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) b[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}
__device__ __forceinline__ uint4 pack(const float (&f)[4], float*) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                    __float_as_uint(f[3]));
}

// A warp per token (warps stride over the tokens): lanes < k fetch the
// token's rows and gates once and share them by shuffles; the warp then walks
// the row's 16-byte vectors 32 * U at a time (lane l takes v0 + l + 32 u), so
// that U loads per slot and lane, for two slots at a time, are in flight,
// accumulating in slot order.
constexpr int kCombineU = 4;

// `wpt` warps share a token (small batches): warp part p of a token takes the
// row's chunks of 32 * U vectors p, p + wpt, ...; each output vector still
// comes from one lane with the same slot-order arithmetic.
// kPair: two slots per step (k >= 2); top-1 keeps one, which needs fewer
// registers and so more warps per SM. U: vectors per slot and lane per step
// (two slots of U = 2 keep the registers low enough for four blocks per SM
// when every warp has a token of its own; small batches, with several warps
// per token, take U = 4).
template <typename T, bool kPair, int U>
__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a, int wpt) {
  constexpr int V = 16 / sizeof(T);
  const int nvec = a.d / V;
  const uint4* Y = static_cast<const uint4*>(a.y_rows);
  const uint4* S = static_cast<const uint4*>(a.y_shared);
  uint4* O = static_cast<uint4*>(a.out);
  const int64_t R = a.T * a.k;
  const int lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int part = static_cast<int>(gw % wpt);
  const int64_t tokens_per_pass = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5) / wpt;
  for (int64_t t = gw / wpt; t < a.T; t += tokens_per_pass) {
    // slot `lane`: first vector of its row (-1 = none; only rows moe_dispatch
    // wrote are read) and its gate
    int64_t my_row = -1;
    float my_g = 0.f;
    if (lane < a.k) {
      const int64_t r = a.inv[t * a.k + lane];
      if (r >= 0 && r < R) {
        my_row = r * nvec;
        my_g = a.gate[t * a.k + lane];
      }
    }
    // the same trip count on every lane: the shuffles below need the whole warp
    for (int v0 = part * 32 * U; v0 < nvec; v0 += wpt * 32 * U) {
      float acc[U][V];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + lane + 32 * u;
        if (S != nullptr && v < nvec) {
          unpack(S[t * nvec + v], acc[u], static_cast<T*>(nullptr));
        } else {
#pragma unroll
          for (int q = 0; q < V; ++q) acc[u][q] = 0.f;
        }
      }
      if constexpr (kPair) {
        // two slots per step: both rows' loads are in flight before either is
        // accumulated, and slot j is still added before slot j + 1
        for (int j = 0; j < a.k; j += 2) {
          const bool two = j + 1 < a.k;  // the same for the whole warp
          const int64_t row0 = __shfl_sync(0xffffffffu, my_row, j);
          const float g0 = __shfl_sync(0xffffffffu, my_g, j);
          int64_t row1 = __shfl_sync(0xffffffffu, my_row, two ? j + 1 : j);
          const float g1 = __shfl_sync(0xffffffffu, my_g, two ? j + 1 : j);
          if (!two) row1 = -1;
          uint4 y0[U], y1[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int v = v0 + lane + 32 * u;
            if (row0 >= 0 && v < nvec) y0[u] = Y[row0 + v];
            if (row1 >= 0 && v < nvec) y1[u] = Y[row1 + v];
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            if (v0 + lane + 32 * u < nvec) {
              float f[V];
              if (row0 >= 0) {
                unpack(y0[u], f, static_cast<T*>(nullptr));
#pragma unroll
                for (int q = 0; q < V; ++q) acc[u][q] = fmaf(g0, f[q], acc[u][q]);
              }
              if (row1 >= 0) {
                unpack(y1[u], f, static_cast<T*>(nullptr));
#pragma unroll
                for (int q = 0; q < V; ++q) acc[u][q] = fmaf(g1, f[q], acc[u][q]);
              }
            }
          }
        }
      } else {
        for (int j = 0; j < a.k; ++j) {
          const int64_t row = __shfl_sync(0xffffffffu, my_row, j);
          const float g = __shfl_sync(0xffffffffu, my_g, j);
          if (row < 0) continue;
          uint4 y[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int v = v0 + lane + 32 * u;
            if (v < nvec) y[u] = Y[row + v];
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            if (v0 + lane + 32 * u < nvec) {
              float f[V];
              unpack(y[u], f, static_cast<T*>(nullptr));
#pragma unroll
              for (int q = 0; q < V; ++q) acc[u][q] = fmaf(g, f[q], acc[u][q]);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + lane + 32 * u;
        if (v < nvec) O[t * nvec + v] = pack(acc[u], static_cast<T*>(nullptr));
      }
    }
  }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  // a warp per token; on batches too small to give every SM a block of 8
  // warps, up to one warp per chunk of 32 * U vectors of the row
  const int V = a.dtype == MOE_F32 ? 4 : 8;
  const int64_t chunks = (a.d / V + 32 * kCombineU - 1) / (32 * kCombineU);
  const int64_t target = static_cast<int64_t>(num_sms()) * 8;
  int64_t wpt = (target + a.T - 1) / a.T;
  if (wpt > chunks) wpt = chunks;
  if (wpt < 1) wpt = 1;
  // 8 warps per block, up to 8 blocks per SM; the grid holds whole tokens
  const int64_t need = (a.T * wpt + 7) / 8;
  int64_t blocks = static_cast<int64_t>(num_sms()) * 8;
  blocks = blocks / wpt * wpt;  // 8 * blocks warps: a multiple of wpt
  if (blocks < wpt) blocks = wpt;
  const unsigned grid = static_cast<unsigned>(need < blocks ? need : blocks);
  const int w = static_cast<int>(wpt);
  if (a.dtype == MOE_F32) {
    if (a.k >= 2 && w == 1)
      combine_kernel<float, true, 2><<<grid, 256, 0, stream>>>(a, w);
    else if (a.k >= 2)
      combine_kernel<float, true, 4><<<grid, 256, 0, stream>>>(a, w);
    else
      combine_kernel<float, false, kCombineU><<<grid, 256, 0, stream>>>(a, w);
  } else {
    if (a.k >= 2 && w == 1)
      combine_kernel<__nv_bfloat16, true, 2><<<grid, 256, 0, stream>>>(a, w);
    else if (a.k >= 2)
      combine_kernel<__nv_bfloat16, true, 4><<<grid, 256, 0, stream>>>(a, w);
    else
      combine_kernel<__nv_bfloat16, false, kCombineU><<<grid, 256, 0, stream>>>(a, w);
  }
  return cudaGetLastError();
}

}  // namespace moe

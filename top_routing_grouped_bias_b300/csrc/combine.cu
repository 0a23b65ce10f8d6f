// Combine: weighted scatter-ADD of the expert outputs back to their tokens.
//
// Pages: "MoE：router 怎样选 expert", 选好以后 (outputs are weighted and added,
// not overwritten or concatenated); "【大模型】MoE（专家混合模型）简介" §3 ④
// (restore token order, fuse by router weight); "MOE 专家选择与路由机制" §八
// (shared-expert term).
//
//   out[t] = y_shared[t] + sum_{j<k} gate[t,j] * y_rows[inv[t*k+j]]
//
// One thread per 16-byte vector of out; fp32 accumulation in slot order
// (deterministic), rounded once to the output dtype.
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

template <typename T>
__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
  constexpr int V = 16 / sizeof(T);
  const int nvec = a.d / V;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= a.T * nvec) return;
  const int64_t t = i / nvec;
  const int v = static_cast<int>(i - t * nvec);
  const uint4* Y = static_cast<const uint4*>(a.y_rows);
  float acc[V];
  if (a.y_shared != nullptr) {
    unpack(static_cast<const uint4*>(a.y_shared)[i], acc, static_cast<T*>(nullptr));
  } else {
#pragma unroll
    for (int q = 0; q < V; ++q) acc[q] = 0.f;
  }
  for (int j = 0; j < a.k; ++j) {
    const int64_t row = a.inv[t * a.k + j];
    if (row < 0 || row >= a.T * a.k) continue;  // only rows moe_dispatch wrote are read
    const float g = a.gate[t * a.k + j];
    float y[V];
    unpack(Y[row * nvec + v], y, static_cast<T*>(nullptr));
#pragma unroll
    for (int q = 0; q < V; ++q) acc[q] = fmaf(g, y[q], acc[q]);
  }
  static_cast<uint4*>(a.out)[i] = pack(acc, static_cast<T*>(nullptr));
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  const int V = a.dtype == MOE_F32 ? 4 : 8;
  const int64_t total = a.T * (a.d / V);
  const unsigned grid = static_cast<unsigned>((total + 255) / 256);
  if (a.dtype == MOE_F32)
    combine_kernel<float><<<grid, 256, 0, stream>>>(a);
  else
    combine_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace moe

// Combine: weighted scatter-ADD of the expert outputs back to their tokens.
//
// Pages: "MoE：router 怎样选 expert", 选好以后 (outputs are weighted and added,
// not overwritten or concatenated); "【大模型】MoE（专家混合模型）简介" §3 ④
// (restore token order, fuse by router weight); "MOE 专家选择与路由机制" §八
// (shared-expert term).
//
//   out[t] = y_shared[t] + sum_{j<k} gate[t,j] * y_rows[inv[t*k+j]]
//
// A block takes one token at a time (blocks stride over the tokens) and reads
// its k rows and gates once; its threads stride over the row's 16-byte
// vectors. fp32 accumulation in slot order (deterministic), rounded once to
// the output dtype.
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
  const uint4* Y = static_cast<const uint4*>(a.y_rows);
  const uint4* S = static_cast<const uint4*>(a.y_shared);
  uint4* O = static_cast<uint4*>(a.out);
  const int64_t R = a.T * a.k;
  // the token's rows (first vector, -1 = none) and gates in slot order; only
  // rows moe_dispatch wrote are read
  __shared__ int64_t rows[kMaxTopK];
  __shared__ float g[kMaxTopK];
  for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
    __syncthreads();  // the previous token's rows are no longer read
    if (threadIdx.x < a.k) {
      const int64_t r = a.inv[t * a.k + threadIdx.x];
      const bool ok = r >= 0 && r < R;
      rows[threadIdx.x] = ok ? r * nvec : -1;
      g[threadIdx.x] = ok ? a.gate[t * a.k + threadIdx.x] : 0.f;
    }
    __syncthreads();
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      float acc[V];
      if (S != nullptr) {
        unpack(S[t * nvec + v], acc, static_cast<T*>(nullptr));
      } else {
#pragma unroll
        for (int q = 0; q < V; ++q) acc[q] = 0.f;
      }
#pragma unroll 4
      for (int j = 0; j < a.k; ++j) {
        if (rows[j] >= 0) {
          float y[V];
          unpack(Y[rows[j] + v], y, static_cast<T*>(nullptr));
#pragma unroll
          for (int q = 0; q < V; ++q) acc[q] = fmaf(g[j], y[q], acc[q]);
        }
      }
      O[t * nvec + v] = pack(acc, static_cast<T*>(nullptr));
    }
  }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  const int64_t blocks = static_cast<int64_t>(num_sms()) * 8;
  const unsigned grid = static_cast<unsigned>(a.T < blocks ? a.T : blocks);
  if (a.dtype == MOE_F32)
    combine_kernel<float><<<grid, 256, 0, stream>>>(a);
  else
    combine_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace moe

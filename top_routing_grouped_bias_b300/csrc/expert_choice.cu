// Expert Choice routing: every expert picks the C tokens with the highest
// router score for it, and a token is served by every expert that picked it.
//
// Pages: "MOE 专家选择与路由机制" §九 routing table (Expert Choice: each expert
// selects a fixed number of tokens; fixed expert load, variable experts per
// token); "MoE：router 怎样选 expert", last section (expert picks tokens).
//
// Kernels (the expert FFN itself is the grouped GEMM pair, with exactly C rows
// per expert):
//   ec_scores   p = softmax (or sigmoid) of each token's logits, written
//               transposed [N, T] through a shared-memory tile
//   ec_select   one block per expert: radix select (4 x 8-bit digits of the
//               fp32 bit pattern, non-negative keys) finds the C-th largest
//               score; tokens above it are taken, ties at it go to the lower
//               token index; a block-wide scan writes the picked tokens in
//               ascending order to rows [e*C, e*C + C), their gates, and the
//               token-by-expert choice matrix used by the combine
//   ec_gather   x_disp[r] = h[row_token[r]] (16-byte vectors)
//   ec_combine  out[t] = y_shared[t] + sum over experts e in order of
//               gate * y_rows[row(t, e)], fp32 accumulation, one rounding
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"

namespace moe {
namespace {

__device__ __forceinline__ float wsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float wmax(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// 32 tokens per block (one warp per token for the row statistics), then the
// [32 x N] tile goes out transposed with consecutive tokens per expert.
__global__ void __launch_bounds__(256) ec_scores_kernel(EcArgs a) {
  extern __shared__ float tile[];  // [32][N + 1]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N, ld = N + 1;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * 32;
  for (int lt = warp; lt < 32; lt += 8) {
    const int64_t t = t0 + lt;
    if (t >= a.T) break;
    const float* z = a.logits + t * N;
    if (a.score == MOE_SCORE_SOFTMAX) {
      float m = -INFINITY;
      for (int e = lane; e < N; e += 32) m = fmaxf(m, z[e]);
      m = wmax(m);
      float s = 0.f;
      for (int e = lane; e < N; e += 32) s += expf(z[e] - m);
      s = wsum(s);
      for (int e = lane; e < N; e += 32) tile[lt * ld + e] = expf(z[e] - m) / s;
    } else {
      for (int e = lane; e < N; e += 32) tile[lt * ld + e] = 1.f / (1.f + expf(-z[e]));
    }
  }
  __syncthreads();
  const int nt = a.T - t0 < 32 ? static_cast<int>(a.T - t0) : 32;
  for (int i = threadIdx.x; i < N * 32; i += blockDim.x) {
    const int e = i >> 5, lt = i & 31;
    if (lt < nt) a.scores_t[static_cast<int64_t>(e) * a.T + t0 + lt] = tile[lt * ld + e];
  }
}

__global__ void __launch_bounds__(1024) ec_select_kernel(EcArgs a) {
  __shared__ unsigned int hist[256];
  __shared__ unsigned int s_digit, s_rem;
  __shared__ int s_gt[1024], s_eq[1024];
  const int e = blockIdx.x;
  const int64_t T = a.T;
  const int C = a.C;
  const float* key_f = a.scores_t + static_cast<int64_t>(e) * T;
  const unsigned int* key = reinterpret_cast<const unsigned int*>(key_f);
  // ---- radix select of the C-th largest key (non-negative floats order as unsigned) ----
  unsigned int prefix = 0, mask = 0, rem = static_cast<unsigned int>(C);
  if (C > 0) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      for (int64_t t = threadIdx.x; t < T; t += blockDim.x) {
        const unsigned int k = key[t];
        if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        unsigned int cum = 0;
        int d = 255;
        for (; d > 0; --d) {
          if (cum + hist[d] >= rem) break;
          cum += hist[d];
        }
        s_digit = static_cast<unsigned int>(d);
        s_rem = rem - cum;
      }
      __syncthreads();
      prefix |= s_digit << shift;
      mask |= 255u << shift;
      rem = s_rem;
      __syncthreads();
    }
  }
  // prefix = key of the C-th largest; rem = ties at it still to take (C > 0)
  const unsigned int thr = prefix;
  // ---- picked tokens in ascending order: contiguous chunk per thread ----
  const int64_t chunk = (T + blockDim.x - 1) / blockDim.x;
  const int64_t lo = threadIdx.x * chunk, hi = lo + chunk < T ? lo + chunk : T;
  int gt = 0, eq = 0;
  if (C > 0)
    for (int64_t t = lo; t < hi; ++t) {
      const unsigned int k = key[t];
      gt += k > thr;
      eq += k == thr;
    }
  s_gt[threadIdx.x] = gt;
  s_eq[threadIdx.x] = eq;
  __syncthreads();
  if (threadIdx.x == 0) {  // exclusive scans (1024 entries, once per expert)
    int rg = 0, re = 0;
    for (int i = 0; i < static_cast<int>(blockDim.x); ++i) {
      const int g = s_gt[i], q = s_eq[i];
      s_gt[i] = rg;
      s_eq[i] = re;
      rg += g;
      re += q;
    }
  }
  __syncthreads();
  if (C == 0) return;
  int gbefore = s_gt[threadIdx.x], ebefore = s_eq[threadIdx.x];
  const int take_eq = static_cast<int>(rem);
  for (int64_t t = lo; t < hi; ++t) {
    const unsigned int k = key[t];
    bool pick = false;
    int pos = 0;
    if (k > thr) {
      pick = true;
      pos = gbefore + min(ebefore, take_eq);
      ++gbefore;
    } else if (k == thr) {
      if (ebefore < take_eq) {
        pick = true;
        pos = gbefore + ebefore;
      }
      ++ebefore;
    }
    if (pick) {
      const int64_t row = static_cast<int64_t>(e) * C + pos;
      a.row_token[row] = static_cast<int32_t>(t);
      a.row_gate[row] = key_f[t];
      a.choice[t * a.N + e] = static_cast<int32_t>(row + 1);
      if (a.tokens_out) a.tokens_out[row] = static_cast<int32_t>(t);
      if (a.gates_out) a.gates_out[row] = key_f[t];
    }
  }
}

__global__ void ec_offsets_kernel(int32_t* offsets, int N, int C) {
  for (int e = threadIdx.x; e <= N; e += blockDim.x) offsets[e] = e * C;
}

// A block copies one picked row at a time (blocks stride over the rows), its
// threads striding over the row's 16-byte vectors.
__global__ void __launch_bounds__(256) ec_gather_kernel(EcArgs a, int64_t rows, int nvec) {
  const uint4* H = static_cast<const uint4*>(a.h);
  uint4* X = static_cast<uint4*>(a.x_disp);
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const int64_t t = a.row_token[r];
    const uint4* src = H + t * nvec;
    uint4* dst = X + r * nvec;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) dst[v] = src[v];
  }
}

template <typename T>
struct Pack;
template <>
struct Pack<__nv_bfloat16> {
  static constexpr int n = 8;
  __device__ static void load(const uint4& u, float* f) {
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(b[i]);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  }
  __device__ static uint4 store(const float* f) {
    uint4 u;
    __nv_bfloat162* b = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) b[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return u;
  }
};
template <>
struct Pack<float> {
  static constexpr int n = 4;
  __device__ static void load(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
  __device__ static uint4 store(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

// A block takes one token at a time: its threads first compact the token's
// chosen experts (ascending e, warp ballots) into a list of (row, gate) in
// shared memory, then stride over the row's 16-byte vectors and add the
// listed rows in that order.
template <typename T>
__global__ void __launch_bounds__(256) ec_combine_kernel(EcArgs a) {
  constexpr int V = Pack<T>::n;
  extern __shared__ int ec_smem[];
  int* rows = ec_smem;                                        // [N]
  float* gts = reinterpret_cast<float*>(ec_smem + a.N);       // [N]
  __shared__ int warp_cnt[8];
  __shared__ int n_sel;
  const int nvec = a.d / V;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint4* Y = static_cast<const uint4*>(a.y_rows);
  const uint4* S = static_cast<const uint4*>(a.y_shared);
  uint4* O = static_cast<uint4*>(a.out);
  for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
    const int32_t* ch = a.choice + t * a.N;
    __syncthreads();  // the previous token's list is no longer read
    if (threadIdx.x == 0) n_sel = 0;
    __syncthreads();
    for (int e0 = 0; e0 < a.N; e0 += 256) {
      const int e = e0 + threadIdx.x;
      const int32_t c = e < a.N ? ch[e] : 0;
      const unsigned m = __ballot_sync(0xffffffffu, c > 0);
      if (lane == 0) warp_cnt[w] = __popc(m);
      __syncthreads();
      int before = n_sel;
      for (int q = 0; q < w; ++q) before += warp_cnt[q];
      if (c > 0) {
        const int pos = before + __popc(m & ((1u << lane) - 1u));
        rows[pos] = c - 1;
        gts[pos] = a.row_gate[c - 1];
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        int tot = 0;
        for (int q = 0; q < 8; ++q) tot += warp_cnt[q];
        n_sel += tot;
      }
      __syncthreads();
    }
    const int cnt = n_sel;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      float acc[V];
      if (S != nullptr) {
        Pack<T>::load(S[t * nvec + v], acc);
      } else {
#pragma unroll
        for (int q = 0; q < V; ++q) acc[q] = 0.f;
      }
#pragma unroll 4
      for (int i = 0; i < cnt; ++i) {
        float y[V];
        Pack<T>::load(Y[static_cast<int64_t>(rows[i]) * nvec + v], y);
        const float g = gts[i];
#pragma unroll
        for (int q = 0; q < V; ++q) acc[q] = fmaf(g, y[q], acc[q]);
      }
      O[t * nvec + v] = Pack<T>::store(acc);
    }
  }
}

}  // namespace

cudaError_t launch_ec_select(const EcArgs& a, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  cudaError_t err = cudaMemsetAsync(a.choice, 0, sizeof(int32_t) * a.T * a.N, stream);
  if (err != cudaSuccess) return err;
  const size_t tile = sizeof(float) * 32 * (a.N + 1);
  err = cudaFuncSetAttribute(ec_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(tile));
  if (err != cudaSuccess) return err;
  ec_scores_kernel<<<static_cast<unsigned>((a.T + 31) / 32), 256, tile, stream>>>(a);
  ec_select_kernel<<<a.N, 1024, 0, stream>>>(a);
  ec_offsets_kernel<<<1, 1024, 0, stream>>>(a.offsets, a.N, a.C);
  const int vec = a.dtype == MOE_F32 ? 4 : 8;
  const int nvec = a.d / vec;
  const int64_t rows = static_cast<int64_t>(a.N) * a.C;
  if (rows > 0) {
    const int64_t blocks = static_cast<int64_t>(num_sms()) * 8;
    ec_gather_kernel<<<static_cast<unsigned>(rows < blocks ? rows : blocks), 256, 0, stream>>>(
        a, rows, nvec);
  }
  return cudaGetLastError();
}

cudaError_t launch_ec_combine(const EcArgs& a, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  const int64_t blocks = static_cast<int64_t>(num_sms()) * 8;
  const unsigned grid = static_cast<unsigned>(a.T < blocks ? a.T : blocks);
  const size_t smem = static_cast<size_t>(a.N) * (sizeof(int) + sizeof(float));
  if (a.dtype == MOE_F32)
    ec_combine_kernel<float><<<grid, 256, smem, stream>>>(a);
  else
    ec_combine_kernel<__nv_bfloat16><<<grid, 256, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace moe

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
//               fp32 bit pattern, non-negative keys; warp-aggregated
//               histogram counts) finds the C-th largest score; tokens above
//               it are taken, ties at it go to the lower token index; block
//               scans over rounds of tokens write the picked tokens in
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

// Exclusive block scan of two counts at once (blockDim.x = 1024 = 32 warps);
// also returns the block totals. Uses `ws` [64] of shared memory.
__device__ __forceinline__ void block_scan2(int g, int q, int& gx, int& qx, int& gt, int& qt,
                                            int* ws) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int gi = g, qi = q;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int vg = __shfl_up_sync(0xffffffffu, gi, o);
    const int vq = __shfl_up_sync(0xffffffffu, qi, o);
    if (lane >= o) {
      gi += vg;
      qi += vq;
    }
  }
  if (lane == 31) {
    ws[w] = gi;
    ws[32 + w] = qi;
  }
  __syncthreads();
  if (w == 0) {
    const int vg = ws[lane], vq = ws[32 + lane];
    int sg = vg, sq = vq;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ug = __shfl_up_sync(0xffffffffu, sg, o);
      const int uq = __shfl_up_sync(0xffffffffu, sq, o);
      if (lane >= o) {
        sg += ug;
        sq += uq;
      }
    }
    ws[lane] = sg - vg;       // exclusive prefix of the warps
    ws[32 + lane] = sq - vq;
    if (lane == 31) {
      ws[64] = sg;            // totals
      ws[65] = sq;
    }
  }
  __syncthreads();
  gx = ws[w] + gi - g;
  qx = ws[32 + w] + qi - q;
  gt = ws[64];
  qt = ws[65];
  __syncthreads();  // ws is reused by the next call
}

constexpr int kEcUnroll = 8;  // rounds of keys loaded per thread at once

// One block (1024 threads) per expert.
__global__ void __launch_bounds__(1024) ec_select_kernel(EcArgs a) {
  __shared__ unsigned int hist[256];
  __shared__ unsigned int s_digit, s_rem;
  __shared__ int scan_ws[66];
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int64_t T = a.T;
  const int C = a.C;
  if (C == 0) return;
  const float* key_f = a.scores_t + static_cast<int64_t>(e) * T;
  const unsigned int* key = reinterpret_cast<const unsigned int*>(key_f);
  // ---- radix select of the C-th largest key (non-negative floats order as
  // unsigned): 4 passes of 8-bit digits; each warp adds one count per distinct
  // digit among its lanes (scores cluster, so per-lane atomics would collide) ----
  unsigned int prefix = 0, mask = 0, rem = static_cast<unsigned int>(C);
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int64_t t0 = 0; t0 < T; t0 += static_cast<int64_t>(blockDim.x) * kEcUnroll) {
      unsigned int kk[kEcUnroll];
#pragma unroll
      for (int u = 0; u < kEcUnroll; ++u) {  // kEcUnroll rounds of loads in flight
        const int64_t t = t0 + static_cast<int64_t>(u) * blockDim.x + threadIdx.x;
        kk[u] = t < T ? key[t] : 0u;
      }
#pragma unroll
      for (int u = 0; u < kEcUnroll; ++u) {
        const int64_t t = t0 + static_cast<int64_t>(u) * blockDim.x + threadIdx.x;
        const bool in = t < T && (kk[u] & mask) == prefix;
        const unsigned int digit = in ? (kk[u] >> shift) & 255u : 256u;  // 256: not counted
        const unsigned int peers = __match_any_sync(0xffffffffu, digit);
        if (in && lane == __ffs(peers) - 1)
          atomicAdd(&hist[digit], static_cast<unsigned int>(__popc(peers)));
      }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // digit holding the rem-th largest: lane l sums bins [8l, 8l + 8), a
      // suffix scan over lanes (from digit 255 down) finds the bin
      unsigned int part = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) part += hist[lane * 8 + i];
      unsigned int suf = part;  // sum over lanes >= lane
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned int v = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += v;
      }
      const unsigned int above = suf - part;  // keys in bins of higher lanes
      // the lane whose chunk contains the boundary: above < rem <= above + part
      const bool mine = above < rem && rem <= suf;
      if (mine) {
        unsigned int cum = above;
        int d = lane * 8 + 7;
        for (; d > lane * 8; --d) {
          if (cum + hist[d] >= rem) break;
          cum += hist[d];
        }
        s_digit = static_cast<unsigned int>(d);
        s_rem = rem - cum;
      }
    }
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= 255u << shift;
    rem = s_rem;
    __syncthreads();
  }
  // prefix = key of the C-th largest; rem = ties at it still to take
  const unsigned int thr = prefix;
  const int take_eq = static_cast<int>(rem);
  // ---- picked tokens in ascending order: rounds of blockDim tokens, block
  // scans of the above-threshold and tie flags give each pick its position ----
  int g_run = 0, q_run = 0;
  for (int64_t t0 = 0; t0 < T; t0 += static_cast<int64_t>(blockDim.x) * kEcUnroll) {
    unsigned int kk[kEcUnroll];
#pragma unroll
    for (int u = 0; u < kEcUnroll; ++u) {
      const int64_t t = t0 + static_cast<int64_t>(u) * blockDim.x + threadIdx.x;
      kk[u] = t < T ? key[t] : 0u;
    }
    for (int u = 0; u < kEcUnroll; ++u) {  // rounds in token order
      const int64_t t = t0 + static_cast<int64_t>(u) * blockDim.x + threadIdx.x;
      const int g = t < T && kk[u] > thr, q = t < T && kk[u] == thr;
      int gx, qx, gt, qt;
      block_scan2(g, q, gx, qx, gt, qt, scan_ws);
      const int gb = g_run + gx, eb = q_run + qx;
      bool pick = false;
      int pos = 0;
      if (g) {
        pick = true;
        pos = gb + min(eb, take_eq);
      } else if (q && eb < take_eq) {
        pick = true;
        pos = gb + eb;
      }
      if (pick) {
        const int64_t row = static_cast<int64_t>(e) * C + pos;
        const float gv = __uint_as_float(kk[u]);
        a.row_token[row] = static_cast<int32_t>(t);
        a.row_gate[row] = gv;
        a.choice[t * a.N + e] = static_cast<int32_t>(row + 1);
        if (a.tokens_out) a.tokens_out[row] = static_cast<int32_t>(t);
        if (a.gates_out) a.gates_out[row] = gv;
      }
      g_run += gt;
      q_run += qt;
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

// A warp per token: its lanes compact the token's chosen experts (ascending
// e, warp ballots) into the warp's list of (row, gate) in shared memory, then
// stride over the row's 16-byte vectors and add the listed rows in that order.
// Eight tokens per block, no block-wide barrier: every warp of the SM has its
// own token's loads in flight.
constexpr int kEcCombineWarps = 8;

template <typename T>
__global__ void __launch_bounds__(kEcCombineWarps * 32) ec_combine_kernel(EcArgs a) {
  constexpr int V = Pack<T>::n;
  extern __shared__ int ec_smem[];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int* rows = ec_smem + static_cast<size_t>(w) * 2 * a.N;      // [N]
  float* gts = reinterpret_cast<float*>(rows + a.N);           // [N]
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kEcCombineWarps + w;
  if (t >= a.T) return;
  const int nvec = a.d / V;
  const uint4* Y = static_cast<const uint4*>(a.y_rows);
  const uint4* S = static_cast<const uint4*>(a.y_shared);
  uint4* O = static_cast<uint4*>(a.out);
  const int32_t* ch = a.choice + t * a.N;
  int cnt = 0;
  for (int e0 = 0; e0 < a.N; e0 += 32) {
    const int e = e0 + lane;
    const int32_t c = e < a.N ? ch[e] : 0;
    const unsigned m = __ballot_sync(0xffffffffu, c > 0);
    if (c > 0) {
      const int pos = cnt + __popc(m & ((1u << lane) - 1u));
      rows[pos] = c - 1;
      gts[pos] = a.row_gate[c - 1];
    }
    cnt += __popc(m);
  }
  __syncwarp();
  // each lane's vectors v0, v0 + 32, ... (up to kEcU of them) are loaded
  // together for every listed row; each element adds the rows in list order
  constexpr int kEcU = 8;
  for (int v0 = lane; v0 < nvec; v0 += 32 * kEcU) {
    float acc[kEcU][V];
#pragma unroll
    for (int u = 0; u < kEcU; ++u) {
      const int v = v0 + 32 * u;
      if (S != nullptr && v < nvec) {
        Pack<T>::load(S[t * nvec + v], acc[u]);
      } else {
#pragma unroll
        for (int q = 0; q < V; ++q) acc[u][q] = 0.f;
      }
    }
    for (int i = 0; i < cnt; ++i) {
      const int64_t rb = static_cast<int64_t>(rows[i]) * nvec;
      const float g = gts[i];
      uint4 raw[kEcU];
#pragma unroll
      for (int u = 0; u < kEcU; ++u)
        if (v0 + 32 * u < nvec) raw[u] = Y[rb + v0 + 32 * u];
#pragma unroll
      for (int u = 0; u < kEcU; ++u) {
        if (v0 + 32 * u < nvec) {
          float y[V];
          Pack<T>::load(raw[u], y);
#pragma unroll
          for (int q = 0; q < V; ++q) acc[u][q] = fmaf(g, y[q], acc[u][q]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kEcU; ++u)
      if (v0 + 32 * u < nvec) O[t * nvec + v0 + 32 * u] = Pack<T>::store(acc[u]);
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
  const unsigned grid = static_cast<unsigned>((a.T + kEcCombineWarps - 1) / kEcCombineWarps);
  const size_t smem = static_cast<size_t>(kEcCombineWarps) * a.N * (sizeof(int) + sizeof(float));
  cudaError_t err;
  if (a.dtype == MOE_F32) {
    err = cudaFuncSetAttribute(ec_combine_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    ec_combine_kernel<float><<<grid, kEcCombineWarps * 32, smem, stream>>>(a);
  } else {
    err = cudaFuncSetAttribute(ec_combine_kernel<__nv_bfloat16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    ec_combine_kernel<__nv_bfloat16><<<grid, kEcCombineWarps * 32, smem, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace moe

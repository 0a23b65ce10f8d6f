// Dispatch: regroup the (token, slot) pairs by expert and gather their rows.
//
// Pages: "MOE 专家选择与路由机制" §三 Token Dispatch (pairs of one expert are
// listed together, tokens ascending); "【大模型】MoE（专家混合模型）简介" §3 ②.
//
// Deterministic counting sort in three launches plus the gather (one launch
// plus the gather for small batches: dispatch_small_kernel below), no atomics
// on the ordering:
//   1. count    per block of 256 tokens, per-expert pair counts -> base[e][b]
//               (expert-major, so that each expert's column is contiguous)
//   2. scan     a block per expert column: base[e][b] = sum_{b' < b} count[b'][e],
//               counts[e] = sum_b (capped at the capacity when one is set)
//   3. permute  per block: for each warp and expert the mask of lanes holding
//               it, scan of the masks' counts over warps (plus the block's
//               base); rank = base + warp prefix + lower lanes holding e;
//               row = offsets[e] + rank, or inv = -1 when rank >= capacity,
//               with offsets = exclusive scan of counts over e (every block;
//               block 0 writes them). Writes row_token and inv.
//   4. gather   a warp per token at a time, up to eight 16-byte vectors of
//               the row per lane in flight (batches of 8192 tokens or more;
//               smaller ones a block per token, a thread per vector): reads
//               h[t] once, writes it to the token's k rows.
// The row of (t, e) is offsets[e] + #{t' < t : e in S_t'}, i.e. rows are
// ordered by (expert, token).
#include <cuda_bf16.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kTB = kDispatchTokensPerBlock;  // 256 tokens, 8 warps
constexpr int kWarps = kTB / 32;

__global__ void __launch_bounds__(kTB) dispatch_count_kernel(DispatchArgs a) {
  extern __shared__ int hist[];  // [N]
  for (int e = threadIdx.x; e < a.N; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kTB + threadIdx.x;
  if (t < a.T) {
    // all of the token's loads first, then the counting (a load per slot
    // followed by its atomic would wait out each load's latency in turn)
    int e[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) e[j] = j < a.k ? a.idx[t * a.k + j] : 0;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j >= a.k) break;
      if (e[j] >= 0 && e[j] < a.N)
        atomicAdd(&hist[e[j]], 1);
      else if (a.status != nullptr)
        atomicCAS(a.status, 0, MOE_ERR_DEVICE_CHECK);
    }
  }
  __syncthreads();
  // expert-major: base[e][b] for the scan's contiguous per-expert columns
  for (int e = threadIdx.x; e < a.N; e += blockDim.x)
    a.block_base[static_cast<size_t>(e) * gridDim.x + blockIdx.x] = hist[e];
}

// One block per expert column: the exclusive running sum of the expert's
// pair counts over the token blocks (base[e][b] = pairs of e in blocks
// before b), and its total, capped at the capacity when one is set, written
// to counts[e]. The offsets (a scan over the N totals) are left to the
// permute kernel, whose every block needs them.
__global__ void __launch_bounds__(kTB) dispatch_scan_kernel(DispatchArgs a, int nb) {
  __shared__ int warp_sums[kWarps];
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int* col = a.block_base + static_cast<size_t>(e) * nb;
  int carry = 0;
  for (int b0 = 0; b0 < nb; b0 += kTB) {
    const int b = b0 + static_cast<int>(threadIdx.x);
    const int c = b < nb ? col[b] : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    int before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int ws = warp_sums[w];
      before += w < warp ? ws : 0;
      all += ws;
    }
    if (b < nb) col[b] = carry + before + incl - c;
    carry += all;
    __syncthreads();  // warp_sums is rewritten by the next step
  }
  // rows kept for this expert: all of them, or its first `capacity` pairs
  if (threadIdx.x == 0)
    a.counts[e] = a.cap_enabled && carry > a.capacity ? static_cast<int>(a.capacity) : carry;
}

__global__ void __launch_bounds__(kTB) dispatch_permute_kernel(DispatchArgs a) {
  extern __shared__ int sm[];
  __shared__ int warp_sums[kWarps];
  const int N = a.N, k = a.k;
  unsigned* lanes = reinterpret_cast<unsigned*>(sm);   // [kWarps][N]: lanes holding e
  int* wbase = sm + kWarps * N;                        // [kWarps][N]: rank base of the warp
  int* sidx = sm + 2 * kWarps * N;                     // [kWarps][32][k]
  int* off = sidx + kWarps * 32 * k;                   // [N + 1]: first row of each expert
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kWarps * N; i += blockDim.x) lanes[i] = 0u;
  // offsets: exclusive scan of the capped totals over the experts, each
  // thread a contiguous chunk of them (every block; block 0 writes them out)
  {
    const int per = (N + kTB - 1) / kTB;
    const int lo = static_cast<int>(threadIdx.x) * per, hi = min(N, lo + per);
    int local = 0;
    for (int e = lo; e < hi; ++e) local += a.counts[e];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    int run = incl - local;
    for (int w = 0; w < warp; ++w) run += warp_sums[w];
    for (int e = lo; e < hi; ++e) {
      off[e] = run;
      if (blockIdx.x == 0) a.offsets[e] = run;
      run += a.counts[e];
    }
    if (hi == N && lo < hi) {
      off[N] = run;
      if (blockIdx.x == 0) a.offsets[N] = run;
    }
  }
  __syncthreads();
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kTB + threadIdx.x;
  const bool valid = t < a.T;
  int* my_idx = sidx + (warp * 32 + lane) * k;
  {
    int ev[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) ev[j] = (valid && j < k) ? a.idx[t * k + j] : -1;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j >= k) break;
      int e = ev[j];
      if (e < 0 || e >= N) e = -1;  // out-of-range indices were flagged by the count pass
      my_idx[j] = e;
      if (e >= 0) atomicOr(&lanes[warp * N + e], 1u << lane);
    }
  }
  __syncthreads();
  // per expert: exclusive scan over warps of their pair counts, plus the
  // block's rank base (the number of the expert's pairs in earlier blocks)
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    int run = a.block_base[static_cast<size_t>(e) * gridDim.x + blockIdx.x];
    for (int w = 0; w < kWarps; ++w) {
      wbase[w * N + e] = run;
      run += __popc(lanes[w * N + e]);
    }
  }
  __syncthreads();
  // A token never repeats an expert, so the pairs of expert e before (t, j)
  // inside the warp are the lower lanes holding e: rank = warp base + their
  // count; rows end up ordered by (expert, token).
  if (valid) {
    const unsigned below = (1u << lane) - 1u;
    for (int j = 0; j < k; ++j) {
      const int e = my_idx[j];
      if (e < 0) {
        a.inv[t * k + j] = -1;
        continue;
      }
      const int rank = wbase[warp * N + e] + __popc(lanes[warp * N + e] & below);
      if (a.cap_enabled && rank >= a.capacity) {
        a.inv[t * k + j] = -1;  // beyond the expert's capacity: dropped
        continue;
      }
      const int row = off[e] + rank;
      a.row_token[row] = static_cast<int32_t>(t);
      a.inv[t * k + j] = row;
    }
  }
}

// Small batches (T*k <= kSmallPairs pairs and ceil(T/32) * N <= kSmallMasks):
// count, scan and permute in ONE block of 1024 threads instead of three
// launches. Tokens form groups of 32 (one warp's lanes); the block
//   1. copies idx to shared memory and records, per (group g, expert e), the
//      mask of lanes whose token holds e (a ballot per expert when N <= 32,
//      else shared-memory ORs);
//   2. scans each expert's masks over the groups (a warp per expert, shuffle
//      scans): base[g][e] = pairs of e in groups before g, count[e] = total;
//   3. scans the (capped) counts over experts into offsets;
//   4. ranks each pair: base[g][e] + lower lanes of its group holding e.
// Same rows, in the same (expert, token) order, as the multi-block path.
constexpr int kSmallThreads = 1024;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int64_t kSmallPairs = 16384;
constexpr int64_t kSmallMasks = 8192;

__global__ void __launch_bounds__(kSmallThreads) dispatch_small_kernel(DispatchArgs a) {
  extern __shared__ int sm[];
  const int N = a.N, k = a.k;
  const int64_t T = a.T, P = T * k;
  const int G = static_cast<int>((T + 31) / 32);
  int* sidx = sm;                                                  // [T*k]
  unsigned* masks = reinterpret_cast<unsigned*>(sidx + P);         // [G][N]
  int* base = reinterpret_cast<int*>(masks + static_cast<size_t>(G) * N);  // [G][N]
  int* tot = base + static_cast<size_t>(G) * N;                    // [N]
  int* off = tot + N;                                              // [N + 1]
  __shared__ int warp_sums[kSmallWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // copy idx first (read-only loads, all in flight together), check it from
  // shared memory afterwards: a flag write between the loads would order them
  for (int64_t i0 = threadIdx.x; i0 < P; i0 += 8 * kSmallThreads) {
    int v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t i = i0 + u * kSmallThreads;
      v[u] = i < P ? __ldg(a.idx + i) : 0;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t i = i0 + u * kSmallThreads;
      if (i < P) sidx[i] = v[u];
    }
  }
  for (int64_t i = threadIdx.x; i < static_cast<int64_t>(G) * N; i += kSmallThreads) masks[i] = 0u;
  __syncthreads();
  if (a.status != nullptr) {
    bool bad = false;
    for (int64_t i = threadIdx.x; i < P; i += kSmallThreads) bad |= sidx[i] < 0 || sidx[i] >= N;
    if (bad) atomicCAS(a.status, 0, MOE_ERR_DEVICE_CHECK);
  }
  // 1. lane masks per (group, expert): with N <= 32 one ballot per expert
  //    over each lane's set of experts, else shared-memory ORs
  const unsigned below = (1u << lane) - 1u;
  for (int g = warp; g < G; g += kSmallWarps) {
    const int64_t t = static_cast<int64_t>(g) * 32 + lane;
    if (N <= 32) {
      unsigned mine = 0u;
      for (int j = 0; j < k; ++j) {
        const int e = t < T ? sidx[t * k + j] : -1;
        if (e >= 0 && e < N) mine |= 1u << e;
      }
      for (int e = 0; e < N; ++e) {
        const unsigned m = __ballot_sync(0xffffffffu, (mine >> e) & 1u);
        if (lane == 0) masks[static_cast<size_t>(g) * N + e] = m;
      }
    } else if (t < T) {
      for (int j = 0; j < k; ++j) {
        const int e = sidx[t * k + j];
        if (e >= 0 && e < N) atomicOr(&masks[static_cast<size_t>(g) * N + e], 1u << lane);
      }
    }
  }
  __syncthreads();
  // 2. per expert: exclusive scan of its pair counts over the groups
  for (int e = warp; e < N; e += kSmallWarps) {
    int carry = 0;
    for (int g0 = 0; g0 < G; g0 += 32) {
      const int g = g0 + lane;
      const int c = g < G ? __popc(masks[static_cast<size_t>(g) * N + e]) : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (g < G) base[static_cast<size_t>(g) * N + e] = carry + incl - c;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    // rows kept for this expert: all of them, or its first `capacity` pairs
    if (lane == 0) tot[e] = a.cap_enabled && carry > a.capacity ? static_cast<int>(a.capacity) : carry;
  }
  __syncthreads();
  // 3. exclusive scan of tot over experts: each thread a contiguous chunk
  {
    const int per = (N + kSmallThreads - 1) / kSmallThreads;
    const int lo = threadIdx.x * per, hi = min(N, lo + per);
    int local = 0;
    for (int e = lo; e < hi; ++e) local += tot[e];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int v = warp_sums[lane];
      int inc = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
      }
      warp_sums[lane] = inc - v;
    }
    __syncthreads();
    int run = warp_sums[warp] + incl - local;
    for (int e = lo; e < hi; ++e) {
      off[e] = run;
      a.counts[e] = tot[e];
      a.offsets[e] = run;
      run += tot[e];
    }
    if (hi == N && lo < hi) {
      off[N] = run;
      a.offsets[N] = run;
    }
  }
  __syncthreads();
  // 4. ranks, rows and the inverse index
  for (int g = warp; g < G; g += kSmallWarps) {
    const int64_t t = static_cast<int64_t>(g) * 32 + lane;
    if (t >= T) continue;
    for (int j = 0; j < k; ++j) {
      const int e = sidx[t * k + j];
      if (e < 0 || e >= N) {
        a.inv[t * k + j] = -1;
        continue;
      }
      const size_t ge = static_cast<size_t>(g) * N + e;
      const int rank = base[ge] + __popc(masks[ge] & below);
      if (a.cap_enabled && rank >= a.capacity) {
        a.inv[t * k + j] = -1;  // beyond the expert's capacity: dropped
        continue;
      }
      const int row = off[e] + rank;
      a.row_token[row] = static_cast<int32_t>(t);
      a.inv[t * k + j] = row;
    }
  }
}

// Gather: a block takes one token at a time (blocks stride over the tokens);
// its threads stride over the row's 16-byte vectors, read each from h once
// and write it to the token's k dispatched rows (coalesced along d).
// Small batches: a block per token at a time, a thread per 16-byte vector
// of the row (more threads per token than a warp).
template <typename T>
__global__ void __launch_bounds__(256) dispatch_gather_block_kernel(DispatchArgs a) {
  const int nvec = a.d * static_cast<int>(sizeof(T)) / 16;
  const uint4* H = static_cast<const uint4*>(a.h);
  uint4* X = static_cast<uint4*>(a.x_disp);
  const int64_t R = a.T * a.k;
  __shared__ int64_t rows[kMaxTopK];  // first vector of each kept row, -1 = none
  for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
    __syncthreads();  // the previous token's rows are no longer read
    if (threadIdx.x < a.k) {
      const int64_t r = a.inv[t * a.k + threadIdx.x];
      rows[threadIdx.x] = (r >= 0 && r < R) ? r * nvec : -1;
    }
    __syncthreads();
    const uint4* src = H + t * nvec;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      const uint4 val = src[v];
      for (int j = 0; j < a.k; ++j)
        if (rows[j] >= 0) X[rows[j] + v] = val;
    }
  }
}

constexpr int kGatherU = 8;
// From this many tokens the warp-per-token gather has enough warps to keep
// every SM busy (measured: 8192 and 65536 tokens faster, 4096 slower than a
// block per token).
constexpr int64_t kGatherWarpMinTokens = 8192;

template <typename T>
__global__ void __launch_bounds__(256) dispatch_gather_warp_kernel(DispatchArgs a) {
  // a warp per token (warps stride over the tokens): lanes < k read the
  // token's rows once and pass them round by shuffles; each lane loads up to
  // kGatherU 16-byte vectors of h[t] before storing them to the k rows
  constexpr int U = kGatherU;
  const int nvec = a.d * static_cast<int>(sizeof(T)) / 16;
  const uint4* H = static_cast<const uint4*>(a.h);
  uint4* X = static_cast<uint4*>(a.x_disp);
  const int64_t R = a.T * a.k;
  const int lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t nw = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t t = gw; t < a.T; t += nw) {
    int64_t my_row = -1;  // first vector of slot `lane`'s row, -1 = none
    if (lane < a.k) {
      const int64_t r = a.inv[t * a.k + lane];
      my_row = (r >= 0 && r < R) ? r * nvec : -1;
    }
    const uint4* src = H + t * nvec;
    // the same trip count on every lane: the shuffles below need the whole warp
    for (int v0 = 0; v0 < nvec; v0 += 32 * U) {
      uint4 val[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + lane + 32 * u;
        if (v < nvec) val[u] = src[v];
      }
      for (int j = 0; j < a.k; ++j) {
        const int64_t row = __shfl_sync(0xffffffffu, my_row, j);
        if (row < 0) continue;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + lane + 32 * u;
          if (v < nvec) X[row + v] = val[u];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t stream) {
  if (a.T == 0) {
    cudaError_t e1 = cudaMemsetAsync(a.counts, 0, sizeof(int32_t) * a.N, stream);
    if (e1 != cudaSuccess) return e1;
    return cudaMemsetAsync(a.offsets, 0, sizeof(int32_t) * (a.N + 1), stream);
  }
  const int64_t pairs = a.T * a.k;
  const int64_t groups = (a.T + 31) / 32;
  if (pairs <= kSmallPairs && groups * a.N <= kSmallMasks) {
    const size_t smem = sizeof(int) * (static_cast<size_t>(pairs) + 2 * static_cast<size_t>(groups) * a.N +
                                       2 * static_cast<size_t>(a.N) + 1);
    cudaError_t err = cudaFuncSetAttribute(dispatch_small_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    dispatch_small_kernel<<<1, kSmallThreads, smem, stream>>>(a);
  } else {
    const int nb = static_cast<int>((a.T + kTB - 1) / kTB);
    dispatch_count_kernel<<<nb, kTB, a.N * sizeof(int), stream>>>(a);
    dispatch_scan_kernel<<<a.N, kTB, 0, stream>>>(a, nb);
    const size_t smem = sizeof(int) * (2 * static_cast<size_t>(kWarps) * a.N + kWarps * 32 * a.k +
                                       static_cast<size_t>(a.N) + 1);
    cudaError_t err = cudaFuncSetAttribute(dispatch_permute_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    dispatch_permute_kernel<<<nb, kTB, smem, stream>>>(a);
  }
  if (a.x_disp != nullptr) {
    const int64_t blocks = static_cast<int64_t>(num_sms()) * 8;
    if (a.T >= kGatherWarpMinTokens) {
      // a warp per token, 8 warps per block, up to 8 blocks per SM
      const int64_t need = (a.T + 7) / 8;
      const unsigned grid = static_cast<unsigned>(need < blocks ? need : blocks);
      if (a.dtype == MOE_F32)
        dispatch_gather_warp_kernel<float><<<grid, 256, 0, stream>>>(a);
      else
        dispatch_gather_warp_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(a);
    } else {
      const unsigned grid = static_cast<unsigned>(a.T < blocks ? a.T : blocks);
      if (a.dtype == MOE_F32)
        dispatch_gather_block_kernel<float><<<grid, 256, 0, stream>>>(a);
      else
        dispatch_gather_block_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(a);
    }
  }
  return cudaGetLastError();
}

}  // namespace moe

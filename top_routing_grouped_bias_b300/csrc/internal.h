// Internal launch interfaces shared by the host API and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 16;
constexpr int kDispatchTokensPerBlock = 256;
constexpr int kStatsTokensPerBlock = 64;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline int elem_size(int dtype) { return dtype == MOE_F32 ? 4 : 2; }

// The router's logits GEMM (bf16 from h, N <= 256) splits the reduction over
// d into S slices when the batch has fewer 128-token tiles than there are
// SMs to stream h: S = min(max(1, 148 / tiles), max(1, ceil(d / 64) / 4)),
// each slice a whole number of (at least four) 64-element blocks, none empty. The plan depends on
// (T, d) only, so the partial sums and their order are the same on every
// device. Each slice writes fp32 partial logits [T, n_pad] (n_pad = N rounded
// up to 16); the selection kernel adds the slices in slice order.
constexpr int kRouteSplitTarget = 148;
struct RouteSplit {
  int splits, kb_per_split, n_pad;
};
inline RouteSplit route_split(int64_t T, int d, int N) {
  RouteSplit r{};
  const int64_t tiles = (T + 127) / 128;
  const int kb_total = (d + 63) / 64;
  int64_t s = tiles > 0 ? kRouteSplitTarget / tiles : 1;
  const int64_t s_max = kb_total / 4 > 1 ? kb_total / 4 : 1;
  if (s > s_max) s = s_max;
  if (s < 1) s = 1;
  r.kb_per_split = static_cast<int>((kb_total + s - 1) / s);
  r.splits = (kb_total + r.kb_per_split - 1) / r.kb_per_split;
  r.n_pad = (N + 15) / 16 * 16;
  return r;
}

// Workspace layout. Every region starts on a 256-byte boundary. The entry
// points use the prefixes they need: route [status, route_part], dispatch
// [status .. block_base], expert FFN [status .. act_sh], forward everything.
struct WsLayout {
  size_t status, route_part, block_base, stats, act, act_sh, offsets, counts, row_token, inv,
      x_disp, y_rows, y_sh, logits, ec_scores, ec_choice;
  size_t end_route, end_dispatch, end_ffn, total;
};

inline WsLayout ws_layout(const moe_config& c) {
  WsLayout L{};
  const size_t e = static_cast<size_t>(elem_size(c.dtype));
  const size_t T = static_cast<size_t>(c.T), R = T * static_cast<size_t>(c.k);
  const size_t nb = (T + kDispatchTokensPerBlock - 1) / kDispatchTokensPerBlock;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  L.status = take(256);
  // partial logits of the split router GEMM (bf16 from h, N <= 256)
  const RouteSplit rs = route_split(c.T, c.d, c.N);
  const bool tc_router = c.dtype == MOE_BF16 && c.N <= 256;
  L.route_part = take(tc_router ? static_cast<size_t>(rs.splits) * T * rs.n_pad * 4 : 0);
  L.end_route = o;
  L.block_base = take(nb * static_cast<size_t>(c.N) * 4);
  const size_t nbs = (T + kStatsTokensPerBlock - 1) / kStatsTokensPerBlock;
  // block partials [2N + 2][nbs], then the final reduction's ticket counter
  L.stats = take(nbs * (2 * static_cast<size_t>(c.N) + 2) * 4 + 4);
  L.end_dispatch = o;
  L.act = take(R * static_cast<size_t>(c.ffn) * e);
  L.act_sh = take(T * static_cast<size_t>(c.ffn_shared) * e);
  L.end_ffn = o;
  L.offsets = take(static_cast<size_t>(c.N + 1) * 4);
  L.counts = take(static_cast<size_t>(c.N) * 4);
  L.row_token = take(R * 4);
  L.inv = take(R * 4);
  L.x_disp = take(R * static_cast<size_t>(c.d) * e);
  L.y_rows = take(R * static_cast<size_t>(c.d) * e);
  L.y_sh = take(c.ffn_shared > 0 ? T * static_cast<size_t>(c.d) * e : 0);
  L.logits = take(T * static_cast<size_t>(c.N) * 4);
  L.ec_scores = take(T * static_cast<size_t>(c.N) * 4);
  L.ec_choice = take(T * static_cast<size_t>(c.N) * 4);
  L.total = o;
  return L;
}

// ---- route ----
struct RouteArgs {
  const void* h;
  const void* W_r;
  const float* b_r;
  const float* sel_bias;
  const float* logits_in;
  float* logits_out;
  int32_t* idx;
  float* gate;
  int32_t* status;  // device status word or null
  // tensor-core router: scratch for the split partial logits [splits][T][n_pad]
  // (route_split); the selection reads n_partials slices of row stride ld_partial
  float* partials;
  int32_t n_partials, ld_partial;
  int64_t T;
  int32_t d, N, k, score, norm, dtype;
  // group-limited selection (n_group <= 1: off)
  int32_t n_group, topk_group, group_rule, top_m;
};
cudaError_t launch_route(const RouteArgs& a, cudaStream_t stream);
// Router on the tensor cores (bf16, N <= 256, from h). With one slice in
// route_split(T, d, N) a single GEMM does the routing in its epilogue
// (launch_route_mma); otherwise the split GEMM writes the partial logits to
// a.partials (launch_route_logits) and the selection runs in route.cu.
bool route_on_tensor_cores(const RouteArgs& a);
cudaError_t launch_route_mma(const RouteArgs& a, cudaStream_t stream);
cudaError_t launch_route_logits(const RouteArgs& a, cudaStream_t stream);

// ---- dispatch ----
struct DispatchArgs {
  const void* h;
  const int32_t* idx;
  int32_t* counts;
  int32_t* offsets;
  int32_t* row_token;
  int32_t* inv;
  void* x_disp;
  int32_t* block_base;  // scratch [nb * N]
  int32_t* status;      // device status word (index checks)
  int64_t T;
  int32_t d, N, k, dtype;
  int32_t cap_enabled;  // 0 (value-initialised default): dropless
  int64_t capacity;     // rows kept per expert when cap_enabled
};
cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t stream);

// ---- grouped GEMM (gate/up with SwiGLU epilogue, and down) ----
struct FfnArgs {
  const void* x_disp;
  const int32_t* offsets;
  const void* W_gate;
  const void* W_up;
  const void* W_down;
  void* y_rows;
  const void* h;
  const void* Ws_gate;
  const void* Ws_up;
  const void* Ws_down;
  void* y_shared;
  void* act;     // [T*k, F]
  void* act_sh;  // [T, F_sh]
  int32_t* status;
  int64_t T;
  int32_t d, N, k, F, F_sh, dtype;
  int64_t rows;  // dispatched rows when not T*k (0 = T*k)
  // top-1 without a shared expert: fuse the combine into the down pass
  const int32_t* scatter_token;  // row -> token, or null
  const float* scatter_gate;     // [T]
  void* scatter_out;             // [T, d]
  // gate/up A operand straight from h by dispatched-row index (no x_disp)
  const int32_t* gather_rows;    // row -> token, or null
};
cudaError_t launch_expert_ffn(const FfnArgs& a, cudaStream_t stream);

// ---- combine ----
struct CombineArgs {
  const void* y_rows;
  const int32_t* inv;
  const float* gate;
  const void* y_shared;
  void* out;
  int64_t T;
  int32_t d, k, dtype;
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream);

// ---- routing side statistics ----
struct StatsArgs {
  const float* logits;  // [T, N]
  const int32_t* idx;   // [T, k]
  float* out;           // [3 + 2N]
  float* partial;       // scratch [2N + 2][nb], then one uint32 ticket
  unsigned* ticket;     // set by the launcher: the word after the partials
  int64_t T;
  int32_t N, k, score;
};
cudaError_t launch_route_stats(const StatsArgs& a, cudaStream_t stream);

// ---- expert-choice routing ----
struct EcArgs {
  const float* logits;  // [T, N]
  float* scores_t;      // [N, T] scratch
  int32_t* choice;      // [T, N] scratch: row + 1 of (token, expert), 0 = not picked
  int32_t* row_token;   // [N * C]
  float* row_gate;      // [N * C]
  int32_t* offsets;     // [N + 1]
  int32_t* tokens_out;  // [N, C] or null
  float* gates_out;     // [N, C] or null
  const void* h;
  void* x_disp;         // [N * C, d]
  const void* y_rows;   // [N * C, d]
  const void* y_shared; // [T, d] or null
  void* out;            // [T, d]
  int64_t T;
  int32_t d, N, C, score, dtype;
};
cudaError_t launch_ec_select(const EcArgs& a, cudaStream_t stream);
cudaError_t launch_ec_combine(const EcArgs& a, cudaStream_t stream);

cudaError_t launch_selftest_wait(int32_t* status, uint64_t budget_ns, cudaStream_t stream);

int num_sms();

}  // namespace moe

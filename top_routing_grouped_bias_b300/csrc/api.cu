// Host side of the C ABI declared in include/moe.h: argument validation,
// workspace carving and the launch sequence of each entry point.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "internal.h"

using namespace moe;

namespace {

// NVTX range around each stage and entry point for timeline tools, enabled
// by MOE_NVTX=1 in the environment (read once per process); otherwise no
// NVTX call is made.
bool nvtx_enabled() {
  static const bool on = [] {
    const char* v = getenv("MOE_NVTX");
    return v != nullptr && v[0] == '1';
  }();
  return on;
}
struct NvtxRange {
  bool on;
  explicit NvtxRange(const char* name) : on(nvtx_enabled()) {
    if (on) nvtxRangePushA(name);
  }
  ~NvtxRange() {
    if (on) nvtxRangePop();
  }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Pure host checks of a config; no CUDA calls.
moe_status check_config(const moe_config* c) {
  if (c == nullptr) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->T > (int64_t(1) << 31) / 16) return MOE_ERR_INVALID_ARG;
  if (c->d < 1 || c->N < 1 || c->N > kMaxExperts) return MOE_ERR_INVALID_ARG;
  if (c->k < 1 || c->k > c->N || c->k > kMaxTopK) return MOE_ERR_INVALID_ARG;
  if (c->ffn < 1 || c->ffn_shared < 0) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_BF16 && c->dtype != MOE_F32) return MOE_ERR_INVALID_ARG;
  if (c->score != MOE_SCORE_SOFTMAX && c->score != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (c->norm != MOE_NORM_SELECTED && c->norm != MOE_NORM_NONE) return MOE_ERR_INVALID_ARG;
  const int vec = c->dtype == MOE_F32 ? 4 : 8;  // elements per 16 bytes
  if (c->d % vec != 0 || c->ffn % vec != 0 || c->ffn_shared % vec != 0) return MOE_ERR_INVALID_ARG;
  // dispatched rows and B-operand rows must index with int32 on the device
  const int64_t R = c->T * c->k;
  if (R * int64_t(c->d) >= (int64_t(1) << 40)) return MOE_ERR_INVALID_ARG;
  if (int64_t(c->N) * c->ffn >= (int64_t(1) << 31) || int64_t(c->N) * c->d >= (int64_t(1) << 31))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

bool ok_tensor(const void* p) { return p != nullptr && aligned(p, 16); }
bool ok_f32(const void* p) { return p != nullptr && aligned(p, 4); }
bool ok_opt_f32(const void* p) { return p == nullptr || aligned(p, 4); }

moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<uint8_t*>(ws) + off);
}

moe_status route_impl(const moe_config* cfg, const void* h, const void* W_r, const float* b_r,
                      const float* sel_bias, const float* logits_in, float* logits_out,
                      int32_t* idx, float* gate, int32_t* status, float* partials,
                      cudaStream_t stream) {
  NvtxRange nvtx_range("moe.route");
  if (h != nullptr) {
    if (!ok_tensor(h) || !ok_tensor(W_r)) return MOE_ERR_INVALID_ARG;
  } else if (!ok_f32(logits_in)) {
    return MOE_ERR_INVALID_ARG;
  }
  if (!ok_f32(idx) || !ok_f32(gate) || !ok_opt_f32(b_r) || !ok_opt_f32(sel_bias) ||
      !ok_opt_f32(logits_out))
    return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  RouteArgs a{};
  a.h = h; a.W_r = W_r; a.b_r = b_r; a.sel_bias = sel_bias; a.logits_in = logits_in;
  a.logits_out = logits_out; a.idx = idx; a.gate = gate; a.T = cfg->T; a.d = cfg->d;
  a.N = cfg->N; a.k = cfg->k; a.score = cfg->score; a.norm = cfg->norm; a.dtype = cfg->dtype;
  a.status = status;
  a.partials = partials;
  if (route_on_tensor_cores(a) && partials == nullptr) return MOE_ERR_WORKSPACE;
  return from_cuda(launch_route(a, stream));
}

// The router's partial-logit scratch when the workspace holds it, else null.
float* route_scratch(const moe_config* cfg, void* ws, size_t ws_bytes) {
  const WsLayout L = ws_layout(*cfg);
  if (ws == nullptr || ws_bytes < L.end_route || !aligned(ws, 256)) return nullptr;
  return at<float>(ws, L.route_part);
}

moe_status dispatch_impl(const moe_config* cfg, const void* h, const int32_t* idx, int32_t* counts,
                         int32_t* offsets, int32_t* row_token, int32_t* inv, void* x_disp,
                         void* ws, const WsLayout& L, cudaStream_t stream,
                         int64_t capacity = -1) {
  NvtxRange nvtx_range("moe.dispatch");
  if (!ok_f32(idx) || !ok_f32(counts) || !ok_f32(offsets) || !ok_f32(row_token) || !ok_f32(inv))
    return MOE_ERR_INVALID_ARG;
  if (x_disp != nullptr && (!ok_tensor(x_disp) || !ok_tensor(h))) return MOE_ERR_INVALID_ARG;
  DispatchArgs a{};
  a.h = h; a.idx = idx; a.counts = counts; a.offsets = offsets; a.row_token = row_token;
  a.inv = inv; a.x_disp = x_disp; a.block_base = at<int32_t>(ws, L.block_base);
  a.status = at<int32_t>(ws, L.status);
  a.T = cfg->T; a.d = cfg->d; a.N = cfg->N; a.k = cfg->k; a.dtype = cfg->dtype;
  a.cap_enabled = capacity >= 0 ? 1 : 0;
  a.capacity = capacity;
  return from_cuda(launch_dispatch(a, stream));
}

moe_status ffn_impl(const moe_config* cfg, const void* x_disp, const int32_t* offsets,
                    const void* W_gate, const void* W_up, const void* W_down, void* y_rows,
                    const void* h, const void* Ws_gate, const void* Ws_up, const void* Ws_down,
                    void* y_shared, void* ws, const WsLayout& L, cudaStream_t stream,
                    const int32_t* scatter_token = nullptr, const float* scatter_gate = nullptr,
                    void* scatter_out = nullptr, const int32_t* gather_rows = nullptr) {
  NvtxRange nvtx_range("moe.expert_ffn");
  const bool a_ok = gather_rows != nullptr ? ok_tensor(h) && ok_f32(gather_rows) : ok_tensor(x_disp);
  if (!a_ok || !ok_f32(offsets) || !ok_tensor(W_gate) || !ok_tensor(W_up) ||
      !ok_tensor(W_down) || !ok_tensor(y_rows))
    return MOE_ERR_INVALID_ARG;
  if (cfg->ffn_shared > 0 && (!ok_tensor(h) || !ok_tensor(Ws_gate) || !ok_tensor(Ws_up) ||
                              !ok_tensor(Ws_down) || !ok_tensor(y_shared)))
    return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  FfnArgs a{};
  a.x_disp = x_disp; a.offsets = offsets; a.W_gate = W_gate; a.W_up = W_up; a.W_down = W_down;
  a.y_rows = y_rows; a.h = h; a.Ws_gate = Ws_gate; a.Ws_up = Ws_up; a.Ws_down = Ws_down;
  a.y_shared = y_shared; a.act = at<void>(ws, L.act); a.act_sh = at<void>(ws, L.act_sh);
  a.status = at<int32_t>(ws, L.status);
  a.T = cfg->T; a.d = cfg->d; a.N = cfg->N; a.k = cfg->k; a.F = cfg->ffn; a.F_sh = cfg->ffn_shared;
  a.dtype = cfg->dtype;
  a.scatter_token = scatter_token;
  a.scatter_gate = scatter_gate;
  a.scatter_out = scatter_out;
  a.gather_rows = gather_rows;
  return from_cuda(launch_expert_ffn(a, stream));
}

moe_status combine_impl(const moe_config* cfg, const void* y_rows, const int32_t* inv,
                        const float* gate, const void* y_shared, void* out, cudaStream_t stream) {
  NvtxRange nvtx_range("moe.combine");
  if (!ok_tensor(y_rows) || !ok_f32(inv) || !ok_f32(gate) || !ok_tensor(out))
    return MOE_ERR_INVALID_ARG;
  if (y_shared != nullptr && !ok_tensor(y_shared)) return MOE_ERR_INVALID_ARG;
  CombineArgs a{};
  a.y_rows = y_rows; a.inv = inv; a.gate = gate; a.y_shared = y_shared; a.out = out;
  a.T = cfg->T; a.d = cfg->d; a.k = cfg->k; a.dtype = cfg->dtype;
  return from_cuda(launch_combine(a, stream));
}

bool ws_ok(void* ws, size_t ws_bytes, size_t need) {
  return ws != nullptr && aligned(ws, 256) && ws_bytes >= need;
}

}  // namespace

extern "C" {

size_t moe_workspace_size(const moe_config* cfg) {
  if (check_config(cfg) != MOE_OK) return 0;
  return ws_layout(*cfg).total;
}

moe_status moe_route(const moe_config* cfg, const void* h, const void* W_r, const float* b_r,
                     const float* sel_bias, const float* logits_in, float* logits_out,
                     int32_t* idx, float* gate, void* ws, size_t ws_bytes, cudaStream_t stream) {
  moe_status s = check_config(cfg);
  if (s != MOE_OK) return s;
  // the status word records device-side failures of the router's bounded
  // waits; the tensor-core router also keeps its partial logits there
  int32_t* status = (ws != nullptr && ws_bytes >= 256 && aligned(ws, 256))
                        ? static_cast<int32_t*>(ws) : nullptr;
  return route_impl(cfg, h, W_r, b_r, sel_bias, logits_in, logits_out, idx, gate, status,
                    route_scratch(cfg, ws, ws_bytes), stream);
}

moe_status moe_dispatch(const moe_config* cfg, const void* h, const int32_t* idx, int32_t* counts,
                        int32_t* offsets, int32_t* row_token, int32_t* inv, void* x_disp, void* ws,
                        size_t ws_bytes, cudaStream_t stream) {
  moe_status s = check_config(cfg);
  if (s != MOE_OK) return s;
  const WsLayout L = ws_layout(*cfg);
  if (!ws_ok(ws, ws_bytes, L.end_dispatch)) return MOE_ERR_WORKSPACE;
  return dispatch_impl(cfg, h, idx, counts, offsets, row_token, inv, x_disp, ws, L, stream);
}

moe_status moe_expert_ffn(const moe_config* cfg, const void* x_disp, const int32_t* offsets,
                          const void* W_gate, const void* W_up, const void* W_down, void* y_rows,
                          const void* h, const void* Ws_gate, const void* Ws_up,
                          const void* Ws_down, void* y_shared, void* ws, size_t ws_bytes,
                          cudaStream_t stream) {
  moe_status s = check_config(cfg);
  if (s != MOE_OK) return s;
  const WsLayout L = ws_layout(*cfg);
  if (!ws_ok(ws, ws_bytes, L.end_ffn)) return MOE_ERR_WORKSPACE;
  return ffn_impl(cfg, x_disp, offsets, W_gate, W_up, W_down, y_rows, h, Ws_gate, Ws_up, Ws_down,
                  y_shared, ws, L, stream);
}

moe_status moe_expert_ffn_gather(const moe_config* cfg, const void* h, const int32_t* row_token,
                                 const int32_t* offsets, const void* W_gate, const void* W_up,
                                 const void* W_down, void* y_rows, const void* Ws_gate,
                                 const void* Ws_up, const void* Ws_down, void* y_shared, void* ws,
                                 size_t ws_bytes, cudaStream_t stream) {
  moe_status s = check_config(cfg);
  if (s != MOE_OK) return s;
  if (cfg->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (row_token == nullptr) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*cfg);
  if (!ws_ok(ws, ws_bytes, L.end_ffn)) return MOE_ERR_WORKSPACE;
  return ffn_impl(cfg, nullptr, offsets, W_gate, W_up, W_down, y_rows, h, Ws_gate, Ws_up, Ws_down,
                  y_shared, ws, L, stream, nullptr, nullptr, nullptr, row_token);
}

moe_status moe_combine(const moe_config* cfg, const void* y_rows, const int32_t* inv,
                       const float* gate, const void* y_shared, void* out, cudaStream_t stream) {
  moe_status s = check_config(cfg);
  if (s != MOE_OK) return s;
  if (cfg->T == 0) return MOE_OK;
  return combine_impl(cfg, y_rows, inv, gate, y_shared, out, stream);
}

namespace {
moe_status forward_impl(const moe_config* cfg, int64_t capacity, const void* h, const void* W_r,
                        const float* b_r, const float* sel_bias, const void* W_gate,
                        const void* W_up, const void* W_down, const void* Ws_gate,
                        const void* Ws_up, const void* Ws_down, void* out, float* logits_out,
                        int32_t* idx, float* gate, int32_t* counts, void* ws, size_t ws_bytes,
                        cudaStream_t stream) {
  NvtxRange nvtx_range("moe.forward");
  moe_status s = check_config(cfg);
  if (s != MOE_OK) return s;
  if (!ok_tensor(h) || !ok_tensor(W_r) || !ok_tensor(W_gate) || !ok_tensor(W_up) ||
      !ok_tensor(W_down) || !ok_tensor(out) || !ok_f32(idx) || !ok_f32(gate) ||
      !ok_opt_f32(counts) || !ok_opt_f32(logits_out))
    return MOE_ERR_INVALID_ARG;
  if (cfg->ffn_shared > 0 && (!ok_tensor(Ws_gate) || !ok_tensor(Ws_up) || !ok_tensor(Ws_down)))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*cfg);
  if (!ws_ok(ws, ws_bytes, L.total)) return MOE_ERR_WORKSPACE;
  if (cfg->T == 0) return MOE_OK;
  int32_t* cnt = counts != nullptr ? counts : at<int32_t>(ws, L.counts);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* row_token = at<int32_t>(ws, L.row_token);
  int32_t* inv = at<int32_t>(ws, L.inv);
  void* x_disp = at<void>(ws, L.x_disp);
  void* y_rows = at<void>(ws, L.y_rows);
  void* y_sh = cfg->ffn_shared > 0 ? at<void>(ws, L.y_sh) : nullptr;

  s = route_impl(cfg, h, W_r, b_r, sel_bias, nullptr, logits_out, idx, gate,
                 at<int32_t>(ws, L.status), at<float>(ws, L.route_part), stream);
  if (s != MOE_OK) return s;
  // The dispatched copy feeds the gate/up pass with one 16 KB TMA box per
  // stage; reading the rows from h by index (gather4, moe_expert_ffn_gather)
  // saves the copy but issues 32 loads per stage and runs ~2.5x slower.
  const int32_t* gather = nullptr;
  s = dispatch_impl(cfg, h, idx, cnt, offsets, row_token, inv, x_disp, ws, L, stream, capacity);
  if (s != MOE_OK) return s;
  // top-1 without a shared expert: out[t] = g_t * E(h_t) is written by the
  // down pass itself (one scaled store per row, no y_rows round trip);
  // tokens whose only pair was dropped (capacity) are cleared first
  const bool fuse = cfg->k == 1 && cfg->ffn_shared == 0;
  if (fuse) {
    if (capacity >= 0) {
      const size_t bytes = static_cast<size_t>(cfg->T) * cfg->d * elem_size(cfg->dtype);
      if (cudaMemsetAsync(out, 0, bytes, stream) != cudaSuccess) return MOE_ERR_CUDA;
    }
    return ffn_impl(cfg, x_disp, offsets, W_gate, W_up, W_down, y_rows, h, Ws_gate, Ws_up,
                    Ws_down, y_sh, ws, L, stream, row_token, gate, out, gather);
  }
  s = ffn_impl(cfg, x_disp, offsets, W_gate, W_up, W_down, y_rows, h, Ws_gate, Ws_up, Ws_down,
               y_sh, ws, L, stream, nullptr, nullptr, nullptr, gather);
  if (s != MOE_OK) return s;
  return combine_impl(cfg, y_rows, inv, gate, y_sh, out, stream);
}
}  // namespace

moe_status moe_route_grouped(const moe_config* cfg, const moe_group_config* grp, const void* h,
                             const void* W_r, const float* b_r, const float* sel_bias,
                             const float* logits_in, float* logits_out, int32_t* idx,
                             float* gate, void* ws, size_t ws_bytes, cudaStream_t stream) {
  NvtxRange nvtx_range("moe.route_grouped");
  moe_status s = check_config(cfg);
  if (s != MOE_OK) return s;
  if (grp == nullptr) return MOE_ERR_INVALID_ARG;
  const int N = cfg->N;
  if (grp->n_group < 1 || grp->n_group > 32 || N % grp->n_group != 0) return MOE_ERR_INVALID_ARG;
  const int gs = N / grp->n_group;
  if (grp->topk_group < 1 || grp->topk_group > grp->n_group) return MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(grp->topk_group) * gs < cfg->k) return MOE_ERR_INVALID_ARG;
  if (grp->rule != 0 && grp->rule != 1) return MOE_ERR_INVALID_ARG;
  if (grp->rule == 1 && (grp->top_m < 1 || grp->top_m > 8 || grp->top_m > gs))
    return MOE_ERR_INVALID_ARG;
  if (!ok_f32(idx) || !ok_f32(gate) || !ok_opt_f32(b_r) || !ok_opt_f32(sel_bias) ||
      !ok_opt_f32(logits_out))
    return MOE_ERR_INVALID_ARG;
  if (h != nullptr ? (!ok_tensor(h) || !ok_tensor(W_r)) : !ok_f32(logits_in))
    return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  RouteArgs a{};
  a.h = h; a.W_r = W_r; a.b_r = b_r; a.sel_bias = sel_bias; a.logits_in = logits_in;
  a.logits_out = logits_out; a.idx = idx; a.gate = gate; a.T = cfg->T; a.d = cfg->d;
  a.N = N; a.k = cfg->k; a.score = cfg->score; a.norm = cfg->norm; a.dtype = cfg->dtype;
  a.n_group = grp->n_group; a.topk_group = grp->topk_group; a.group_rule = grp->rule;
  a.top_m = grp->top_m;
  int32_t* status = (ws != nullptr && ws_bytes >= 256 && aligned(ws, 256))
                        ? static_cast<int32_t*>(ws) : nullptr;
  a.status = status;
  // bf16 from h: logits on the tensor cores, then the group pass and the
  // selection in the warp-per-token kernel from the partial logits
  a.partials = route_scratch(cfg, ws, ws_bytes);
  if (route_on_tensor_cores(a) && a.partials == nullptr) return MOE_ERR_WORKSPACE;
  return from_cuda(launch_route(a, stream));
}

moe_status moe_route_stats(const moe_config* cfg, const float* logits, const int32_t* idx,
                           float* stats, void* ws, size_t ws_bytes, cudaStream_t stream) {
  NvtxRange nvtx_range("moe.route_stats");
  moe_status s = check_config(cfg);
  if (s != MOE_OK) return s;
  if (!ok_f32(logits) || !ok_f32(idx) || !ok_f32(stats)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*cfg);
  if (!ws_ok(ws, ws_bytes, L.end_dispatch)) return MOE_ERR_WORKSPACE;
  StatsArgs a{};
  a.logits = logits; a.idx = idx; a.out = stats; a.partial = at<float>(ws, L.stats);
  a.T = cfg->T; a.N = cfg->N; a.k = cfg->k; a.score = cfg->score;
  return from_cuda(launch_route_stats(a, stream));
}

moe_status moe_forward(const moe_config* cfg, const void* h, const void* W_r, const float* b_r,
                       const float* sel_bias, const void* W_gate, const void* W_up,
                       const void* W_down, const void* Ws_gate, const void* Ws_up,
                       const void* Ws_down, void* out, float* logits_out, int32_t* idx,
                       float* gate, int32_t* counts, void* ws, size_t ws_bytes,
                       cudaStream_t stream) {
  return forward_impl(cfg, -1, h, W_r, b_r, sel_bias, W_gate, W_up, W_down, Ws_gate, Ws_up,
                      Ws_down, out, logits_out, idx, gate, counts, ws, ws_bytes, stream);
}

moe_status moe_forward_capacity(const moe_config* cfg, int64_t capacity, const void* h,
                                const void* W_r, const float* b_r, const float* sel_bias,
                                const void* W_gate, const void* W_up, const void* W_down,
                                const void* Ws_gate, const void* Ws_up, const void* Ws_down,
                                void* out, float* logits_out, int32_t* idx, float* gate,
                                int32_t* counts, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (capacity < 0 || capacity > (int64_t(1) << 31)) return MOE_ERR_INVALID_ARG;
  return forward_impl(cfg, capacity, h, W_r, b_r, sel_bias, W_gate, W_up, W_down, Ws_gate, Ws_up,
                      Ws_down, out, logits_out, idx, gate, counts, ws, ws_bytes, stream);
}

moe_status moe_dispatch_capacity(const moe_config* cfg, int64_t capacity, const void* h,
                                 const int32_t* idx, int32_t* counts, int32_t* offsets,
                                 int32_t* row_token, int32_t* inv, void* x_disp, void* ws,
                                 size_t ws_bytes, cudaStream_t stream) {
  moe_status s = check_config(cfg);
  if (s != MOE_OK) return s;
  if (capacity < 0 || capacity > (int64_t(1) << 31)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*cfg);
  if (!ws_ok(ws, ws_bytes, L.end_dispatch)) return MOE_ERR_WORKSPACE;
  return dispatch_impl(cfg, h, idx, counts, offsets, row_token, inv, x_disp, ws, L, stream,
                       capacity);
}

moe_status moe_forward_expert_choice(const moe_config* cfg, int64_t capacity, const void* h,
                                     const void* W_r, const float* b_r, const void* W_gate,
                                     const void* W_up, const void* W_down, const void* Ws_gate,
                                     const void* Ws_up, const void* Ws_down, void* out,
                                     float* logits_out, int32_t* tokens_out, float* gates_out,
                                     void* ws, size_t ws_bytes, cudaStream_t stream) {
  NvtxRange nvtx_range("moe.forward_expert_choice");
  moe_status s = check_config(cfg);
  if (s != MOE_OK) return s;
  if (capacity < 0 || capacity > cfg->T || capacity * cfg->N > cfg->T * cfg->k)
    return MOE_ERR_INVALID_ARG;
  if (!ok_tensor(h) || !ok_tensor(W_r) || !ok_tensor(W_gate) || !ok_tensor(W_up) ||
      !ok_tensor(W_down) || !ok_tensor(out) || !ok_opt_f32(logits_out) ||
      !ok_opt_f32(tokens_out) || !ok_opt_f32(gates_out) || !ok_opt_f32(b_r))
    return MOE_ERR_INVALID_ARG;
  if (cfg->ffn_shared > 0 && (!ok_tensor(Ws_gate) || !ok_tensor(Ws_up) || !ok_tensor(Ws_down)))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*cfg);
  if (!ws_ok(ws, ws_bytes, L.total)) return MOE_ERR_WORKSPACE;
  if (cfg->T == 0) return MOE_OK;
  float* z = logits_out != nullptr ? logits_out : at<float>(ws, L.logits);
  // logits through the router (its top-k output goes to scratch)
  s = route_impl(cfg, h, W_r, b_r, nullptr, nullptr, z, at<int32_t>(ws, L.row_token),
                 at<float>(ws, L.inv), at<int32_t>(ws, L.status), at<float>(ws, L.route_part),
                 stream);
  if (s != MOE_OK) return s;
  EcArgs e{};
  e.logits = z;
  e.scores_t = at<float>(ws, L.ec_scores);
  e.choice = at<int32_t>(ws, L.ec_choice);
  e.row_token = at<int32_t>(ws, L.row_token);
  e.row_gate = at<float>(ws, L.inv);
  e.offsets = at<int32_t>(ws, L.offsets);
  e.tokens_out = tokens_out;
  e.gates_out = gates_out;
  e.h = h;
  e.x_disp = at<void>(ws, L.x_disp);
  e.y_rows = at<void>(ws, L.y_rows);
  e.y_shared = cfg->ffn_shared > 0 ? at<void>(ws, L.y_sh) : nullptr;
  e.out = out;
  e.T = cfg->T; e.d = cfg->d; e.N = cfg->N; e.C = static_cast<int32_t>(capacity);
  e.score = cfg->score; e.dtype = cfg->dtype;
  s = from_cuda(launch_ec_select(e, stream));
  if (s != MOE_OK) return s;
  if (capacity > 0 || cfg->ffn_shared > 0) {
    FfnArgs a{};
    a.x_disp = e.x_disp; a.offsets = e.offsets; a.W_gate = W_gate; a.W_up = W_up;
    a.W_down = W_down; a.y_rows = at<void>(ws, L.y_rows); a.h = h; a.Ws_gate = Ws_gate;
    a.Ws_up = Ws_up; a.Ws_down = Ws_down; a.y_shared = const_cast<void*>(e.y_shared);
    a.act = at<void>(ws, L.act); a.act_sh = at<void>(ws, L.act_sh);
    a.status = at<int32_t>(ws, L.status);
    a.T = cfg->T; a.d = cfg->d; a.N = cfg->N; a.k = cfg->k; a.F = cfg->ffn;
    a.F_sh = cfg->ffn_shared; a.dtype = cfg->dtype;
    a.rows = capacity * cfg->N > 0 ? capacity * cfg->N : 1;
    s = from_cuda(launch_expert_ffn(a, stream));
    if (s != MOE_OK) return s;
  }
  return from_cuda(launch_ec_combine(e, stream));
}

moe_status moe_read_status(void* ws, size_t ws_bytes, int32_t* device_status, cudaStream_t stream) {
  if (ws == nullptr || ws_bytes < 256 || device_status == nullptr) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, ws, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(ws, 0, sizeof(v)) != cudaSuccess) return MOE_ERR_CUDA;
  *device_status = v;
  return MOE_OK;
}

moe_status moe_selftest_wait_timeout(uint64_t budget_ns, void* ws, size_t ws_bytes,
                                     cudaStream_t stream) {
  if (ws == nullptr || ws_bytes < 256 || !aligned(ws, 256)) return MOE_ERR_WORKSPACE;
  if (budget_ns > 1000000000ull) budget_ns = 1000000000ull;
  return from_cuda(launch_selftest_wait(static_cast<int32_t*>(ws), budget_ns, stream));
}

moe_status moe_expert_capacity(int64_t T, int32_t k, int32_t N, double capacity_factor,
                               int64_t* capacity) {
  if (capacity == nullptr || T < 0 || N < 1 || k < 1 || k > N) return MOE_ERR_INVALID_ARG;
  if (!(capacity_factor >= 0.0) || capacity_factor > 1e30) return MOE_ERR_INVALID_ARG;  // NaN too
  // ((cf * T) * k) / N in double precision, in this order, rounded up
  const double c = ceil(capacity_factor * static_cast<double>(T) * static_cast<double>(k) /
                        static_cast<double>(N));
  if (c > 2147483648.0) return MOE_ERR_INVALID_ARG;
  *capacity = static_cast<int64_t>(c);
  return MOE_OK;
}

const char* moe_status_string(int32_t status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK";
    default: return "MOE_UNKNOWN_STATUS";
  }
}

}  // extern "C"

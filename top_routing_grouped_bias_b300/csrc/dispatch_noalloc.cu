// Dispatch for callers that cannot allocate device memory.
//
// moe_dispatch needs a caller-provided workspace for its per-block expert
// histograms. Some callers have no way to provide one: a plain C or C++ host
// program that embeds this library without a framework and its memory pool,
// or a runtime that forbids device allocation once it is running (for
// instance because an allocation can synchronise the whole device or fail
// under a fixed memory budget). For them, moe_dispatch_noalloc runs the same
// dispatch kernels with the histograms held in a fixed-size array that is
// part of the library's own device image: loading the library on a GPU
// reserves it there until the process exits. The caller still passes every
// input and output buffer.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"

namespace moe {
namespace {

// Capacity of the histogram scratch, in int32 entries: one entry per
// (block of 256 tokens, expert), i.e. ceil(T / 256) * N <= 262144
// (for example T = 65536 tokens with up to 1024 experts).
constexpr size_t kNoallocHistInts = size_t(1) << 18;

// The per-block histograms (1 MiB). There is no status word: nothing could
// read one back from here, so index checks skip bad entries silently.
static __device__ __align__(256) int32_t g_dispatch_scratch[kNoallocHistInts];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx_id[kMaxDevices] = {};

// cuCtxGetCurrent and cuCtxGetId through the runtime's driver entry-point
// query (no link against the driver library).
template <typename Fn>
Fn driver_fn(const char* name, int version) {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &ptr, version, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<Fn>(ptr);
  return nullptr;
}

// Unique id of the current context (ids are never reused, unlike context
// handles); 0 when there is no current context yet.
bool current_ctx_id(unsigned long long* id) {
  static auto get_ctx = driver_fn<PFN_cuCtxGetCurrent_v4000>("cuCtxGetCurrent", 4000);
  static auto get_id = driver_fn<PFN_cuCtxGetId_v12000>("cuCtxGetId", 12000);
  if (get_ctx == nullptr || get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return false;
  *id = 0;
  return ctx == nullptr || get_id(ctx, id) == CUDA_SUCCESS;
}

// The array's device address on the current device. Host code cannot use the
// array's name as a device pointer (it names a host-side stand-in), so the
// address is looked up with the device current and cached together with the
// id of the context it belongs to. A device reset (or any new primary
// context) loads the module again, possibly at another address: the next
// call sees a new context id and looks the address up again.
moe_status scratch_on_current_device(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  unsigned long long id = 0;
  if (!current_ctx_id(&id)) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr || id == 0 || g_scratch_ctx_id[dev] != id) {
    void* p = nullptr;
    // sets up the device's primary context first when there is none yet
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    if (!current_ctx_id(&id) || id == 0) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = static_cast<int32_t*>(p);
    g_scratch_ctx_id[dev] = id;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

bool aligned_to(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace
}  // namespace moe

extern "C" moe_status moe_dispatch_noalloc(const moe_config* cfg, const void* h,
                                           const int32_t* idx, int32_t* counts, int32_t* offsets,
                                           int32_t* row_token, int32_t* inv, void* x_disp,
                                           cudaStream_t stream) {
  using namespace moe;
  // moe_workspace_size returns 0 exactly when the config is invalid.
  if (moe_workspace_size(cfg) == 0) return MOE_ERR_INVALID_ARG;
  auto ok_i32 = [](const void* p) { return p != nullptr && aligned_to(p, 4); };
  if (!ok_i32(idx) || !ok_i32(counts) || !ok_i32(offsets) || !ok_i32(row_token) || !ok_i32(inv))
    return MOE_ERR_INVALID_ARG;
  if (x_disp != nullptr &&
      (h == nullptr || !aligned_to(h, 16) || !aligned_to(x_disp, 16)))
    return MOE_ERR_INVALID_ARG;
  const int64_t nb = (cfg->T + kDispatchTokensPerBlock - 1) / kDispatchTokensPerBlock;
  if (static_cast<size_t>(nb) * static_cast<size_t>(cfg->N) > kNoallocHistInts)
    return MOE_ERR_WORKSPACE;  // beyond the fixed scratch capacity
  int32_t* scratch = nullptr;
  moe_status s = scratch_on_current_device(&scratch);
  if (s != MOE_OK) return s;
  // The array keeps the previous call's contents; nothing needs clearing:
  // the count pass overwrites every histogram entry the later passes read.
  DispatchArgs a{};
  a.h = h;
  a.idx = idx;
  a.counts = counts;
  a.offsets = offsets;
  a.row_token = row_token;
  a.inv = inv;
  a.x_disp = x_disp;
  a.block_base = scratch;
  a.status = nullptr;  // no read-out on this path: bad indices are skipped
  a.T = cfg->T;
  a.d = cfg->d;
  a.N = cfg->N;
  a.k = cfg->k;
  a.dtype = cfg->dtype;
  return launch_dispatch(a, stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

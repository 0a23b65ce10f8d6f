// Grouped GEMM for the expert FFNs on the 5th-generation tensor cores.
//
// Pages: "MOE 专家选择与路由机制" §一 (E_i(h) = W_down (SiLU(W_gate h) ⊙ W_up h))
// and §十二 (Grouped GEMM for many small per-expert matrices);
// "【大模型】MoE（专家混合模型）简介" §3 ③ and §8 (Grouped GEMM kernel).
//
// One persistent launch per pass runs every expert's rows (a "group") plus,
// optionally, one dense group (the shared expert over all tokens):
//   pass A (kSwiGLU): act = SiLU(x W_gate^T) ⊙ (x W_up^T)     [rows, F]
//   pass B (kDown):   y   = act W_down^T                       [rows, d]
// Group sizes live on the device (dispatch offsets); the host never syncs.
//
// CTA = 6 warps, one CTA per SM:
//   warp 0      TMA producer: A tile [128 x 128 B] and B tile [256 x 128 B]
//               per stage, 128-byte swizzle, 4-stage mbarrier ring
//   warp 1      tcgen05.mma issuer (one thread), M=128 N=256, fp32 in TMEM;
//               owns the 512-column TMEM allocation (2 accumulators)
//   warps 2..5  epilogue: tcgen05.ld from TMEM, SiLU⊙up or plain convert,
//               16-byte stores; double-buffered accumulators let the epilogue
//               of one tile overlap the MMAs of the next
// The CTAs share the tiles round-robin, over the fewest CTAs that finish in
// the same number of rounds (a weight-bound pass then has no last round on a
// few SMs). The CTA-pair kernel further down covers batches with many rows
// per expert (256-row tiles, 128-byte row-segment stores).
// For pass A the B tile stacks 128 rows of W_gate over the same 128 rows of
// W_up, so one N=256 MMA produces the gate half (columns 0..127) and the up
// half (128..255) of a 128-column output tile.
//
// Light experts (groups of at most 96 rows) run their tiles with swapped
// operands: the same shared-memory stage, but the two 128-row weight halves
// (W_gate / W_up, or the two halves of the 256-row W_down tile) are the A
// operands of two M=128 MMAs and the group's rows are the B operand with N =
// rows rounded up to 16, loaded as 32-row boxes. Accumulator columns [0, N)
// and [128, 128 + N) hold the two products, transposed (TMEM lane = output
// column); the epilogue writes them back row by row. Such tiles stream their
// weights from HBM for few rows; the swap keeps them from also issuing a
// zero-padded 128 x 256 MMA per K-step.
//
// Two more instances are the router: logits = h W_r^T for 128 tokens per tile
// with all N <= 256 experts in one accumulator.
//   kRoute   (a split plan of one reduction slice: at least 75 token tiles,
//            or d <= 448) does the whole routing in
//            its epilogue: each thread takes one token's logit row from TMEM
//            and computes softmax / sigmoid, the selection bias, the top-k
//            with the lowest-index tie-break and the gates, overlapped with
//            the next tile's MMAs. Up to 128 experts a tile is 256 tokens, two
//            128-row halves that share each K-step's W_r load.
//   kLogits  (smaller batches) splits the reduction over d into slices (one
//            work unit per tile and slice) so that enough SMs stream h; each
//            unit writes its fp32 partial logits and the warp-per-token
//            selection kernel (route.cu) adds the slices in slice order.
//
// Tiles of one group are ordered in bands of at most 16 m-tiles: inside a band
// the n-tiles advance slowest, so CTAs running side by side share one weight
// slice (and the band's activations) through L2.
//
// Every mbarrier wait is bounded (wall-clock budget). On expiry the kernel
// records MOE_ERR_TIMEOUT in the status word, lets the other roles stop, waits
// (bounded) for its own TMA loads and MMAs in flight, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

#ifndef MOE_GEMM_STAGES
#define MOE_GEMM_STAGES 4
#endif
#ifndef MOE_PAIR_STAGES
#define MOE_PAIR_STAGES 6
#endif
#ifndef MOE_PAIR_MIN_ROWS
#define MOE_PAIR_MIN_ROWS 256
#endif

constexpr int kBM = 128;
constexpr int kStages = MOE_GEMM_STAGES;
constexpr int kThreads = 192;
constexpr uint32_t kAccCols = 256;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxGroups = kMaxExperts + 1;
constexpr int kBandMax = 16;
constexpr uint32_t kStageA = kBM * 128;   // 128 rows x 128 B
constexpr uint32_t kStageB = 256 * 128;   // 256 rows x 128 B
constexpr uint32_t kStageBytes = kStageA + kStageB;
constexpr size_t kDynSmem = static_cast<size_t>(kStages) * kStageBytes + 1024;
constexpr uint64_t kWaitBudgetNs = 4000000000ull;   // 4 s per wait
constexpr int kPairMinRowsPerExpert = MOE_PAIR_MIN_ROWS;
constexpr uint64_t kDrainBudgetNs = 200000000ull;   // 0.2 s
// Groups of at most this many rows run with swapped operands (see the
// header comment): their rows are loaded as 32-row boxes.
#ifndef MOE_SWAP_MAX_ROWS
#define MOE_SWAP_MAX_ROWS 96
#endif
constexpr int kSwapMaxRows = MOE_SWAP_MAX_ROWS;
constexpr int kSwapBoxRows = 32;
constexpr uint32_t kSwapBoxBytes = kSwapBoxRows * 128;
// CTA-pair kernel: last tiles of at most this many rows run swapped.
#ifndef MOE_PAIR_SWAP_ROWS
#define MOE_PAIR_SWAP_ROWS 64
#endif
constexpr int kPairSwapRows = MOE_PAIR_SWAP_ROWS;

enum { kSwiGLU = 0, kDown = 1, kRoute = 2, kLogits = 3 };

// Router epilogue arguments (kRoute only).
struct RouteEpi {
  const float* b_r;       // [N] or null
  const float* sel_bias;  // [N] or null
  float* logits_out;      // [T, N] or null
  int32_t* idx;           // [T, k]
  float* gate;            // [T, k]
  int32_t N, k, score, norm;
};

struct GemmParams {
  const int32_t* offsets;  // [n_routed + 1] row offsets of the routed groups
  int32_t n_routed;
  int32_t rows_routed;     // rows of the routed operand (offsets[n_routed] <= this)
  int32_t rows_shared;     // rows of the dense group (0 = none)
  int32_t K;               // reduction width of the routed groups
  int32_t K_shared;        // reduction width of the dense group
  int32_t n_out;           // output columns of the routed groups
  int32_t n_out_shared;    // output columns of the dense group
  void* out;               // [sum rows, n_out]
  void* out_shared;        // [rows_shared, n_out_shared]
  int32_t* status;
  uint64_t budget_ns;
  RouteEpi re;
  // kLogits: fp32 partial logits [k_splits][rows_routed][n_out]; work unit u
  // is token tile u / k_splits and reduction slice u % k_splits of
  // kb_per_split 64-element blocks
  float* partials;
  int32_t k_splits, kb_per_split;
  // Down pass with top-1 routing and no shared expert: the combine is a
  // scaled scatter, so the epilogue writes gate * y to the token's output row
  // (out = [T, n_out]) instead of writing y_rows. Null: plain y_rows.
  const int32_t* scatter_token;  // dispatched row -> token
  const float* scatter_gate;     // [T] gate of each token's single slot
  // Gate/up pass reading the routed rows straight from h: A0 is then h with
  // a 1-row box and dispatched row r is h[gather_rows[r]] (TMA gather4).
  // Null: A0 is the dispatched copy x_disp.
  const int32_t* gather_rows;
  // kRoute: 128-row halves per token tile (1, or 2 when N <= 128: 256 tokens
  // per tile share each K-step's W_r operand)
  int32_t row_halves;
};

struct TileInfo {
  int g, m_blk, n_blk, row0, rows, ncols, b_row0, num_kb;
  // swapped tile (0 = no): MMA width N over the tile's valid rows, rounded
  // up to 16; rv = valid rows of the tile
  int nr, rv;
};

// Decides whether a tile of the 1-CTA kernel runs with swapped operands:
// bf16 gate/up or down passes, routed groups of at most kSwapMaxRows rows in
// all (light experts, whose tiles stream weights for few rows). The tails of
// larger groups keep the plain tile: measured, their swapped form (more TMA
// loads per stage, scalar epilogue stores) was slower.
// Whether routed group g of the pair kernel runs its last tile, of `tail`
// rows, with swapped operands (see the pair kernel's header comment).
template <int MODE>
__device__ __forceinline__ bool pair_swap_tail(int g, int tail, const GemmParams& p) {
  return (MODE == kSwiGLU || MODE == kDown) && g < p.n_routed && tail > 0 && tail <= kPairSwapRows;
}

template <int MODE, typename T>
__device__ __forceinline__ void set_swap(TileInfo& ti, const GemmParams& p) {
  ti.rv = min(kBM, ti.rows - ti.m_blk * kBM);
  ti.nr = 0;
  if constexpr ((MODE == kSwiGLU || MODE == kDown) && sizeof(T) == 2) {
    if (ti.g < p.n_routed && ti.rows <= kSwapMaxRows && ti.rv > 0)
      ti.nr = (ti.rv + 15) / 16 * 16;
  }
}

template <int BN, int BK, int BM = kBM>
__device__ __forceinline__ TileInfo decode_tile(int tile, const int* tile_start, const int* grp_off,
                                                int G, const GemmParams& p) {
  int lo = 0, hi = G;  // tile_start[lo] <= tile < tile_start[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_start[mid] <= tile) lo = mid; else hi = mid;
  }
  TileInfo ti;
  ti.g = lo;
  if (lo < p.n_routed) {
    ti.row0 = grp_off[lo];
    ti.rows = grp_off[lo + 1] - grp_off[lo];
    ti.ncols = p.n_out;
    ti.b_row0 = lo * p.n_out;
    ti.num_kb = (p.K + BK - 1) / BK;
  } else {
    ti.row0 = 0;
    ti.rows = p.rows_shared;
    ti.ncols = p.n_out_shared;
    ti.b_row0 = 0;
    ti.num_kb = (p.K_shared + BK - 1) / BK;
  }
  const int mt = (ti.rows + BM - 1) / BM;
  const int nt = (ti.ncols + BN - 1) / BN;
  const int nbands0 = (mt + kBandMax * kBM / BM - 1) / (kBandMax * kBM / BM);
  const int band_sz = (mt + nbands0 - 1) / nbands0;
  const int l = tile - tile_start[lo];
  const int band = l / (band_sz * nt);
  const int r = l - band * band_sz * nt;
  const int bs = min(band_sz, mt - band * band_sz);
  ti.n_blk = r / bs;
  ti.m_blk = band * band_sz + (r - ti.n_blk * bs);
  return ti;
}

// kRoute work unit: token tile `tile` of the single routed operand.
__device__ __forceinline__ TileInfo route_tile(int tile, const GemmParams& p) {
  TileInfo ti;
  ti.g = 0;
  ti.m_blk = tile;
  ti.n_blk = 0;
  ti.row0 = 0;
  ti.rows = p.rows_routed;
  ti.ncols = p.n_out;
  ti.b_row0 = 0;
  ti.num_kb = (p.K + 63) / 64;
  ti.nr = 0;
  ti.rv = 0;
  return ti;
}

// kLogits work unit: token tile and reduction slice; kb0 = first K block.
__device__ __forceinline__ TileInfo logits_tile(int unit, const GemmParams& p, int& split,
                                                int& kb0) {
  TileInfo ti;
  split = unit % p.k_splits;
  ti.g = 0;
  ti.m_blk = unit / p.k_splits;
  ti.n_blk = 0;
  ti.row0 = 0;
  ti.rows = p.rows_routed;
  ti.ncols = p.n_out;
  ti.b_row0 = 0;
  kb0 = split * p.kb_per_split;
  const int kb_total = (p.K + 63) / 64;
  ti.num_kb = min(p.kb_per_split, kb_total - kb0);
  return ti;
}

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kDrainBudgetNs) return false;
  }
  return true;
}

// TMEM -> registers, 32 columns of this warp's 32 lanes, waiting in the same
// asm block so that no use of the results can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld32_sync(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Store 32 consecutive values; `valid` = columns left in the output row
// (a multiple of the 16-byte vector width).
__device__ __forceinline__ void store32(__nv_bfloat16* dst, const float (&f)[32], int valid) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (q * 8 < valid) {
      uint4 u;
      __nv_bfloat162* b = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
      for (int i = 0; i < 4; ++i) b[i] = __floats2bfloat162_rn(f[q * 8 + 2 * i], f[q * 8 + 2 * i + 1]);
      *reinterpret_cast<uint4*>(dst + q * 8) = u;
    }
  }
}
// 32 fp32 values as 16 bf16x2 words (round to nearest even).
__device__ __forceinline__ void pack_bf16x32(const float (&f)[32], uint32_t* w) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
}

// One exchange step of a 4 x 4 transpose of 32-byte pieces inside each group
// of four lanes: a lane whose bit `m` is clear keeps piece i0 and receives
// the partner's piece i0 into slot i1; a lane with the bit set keeps piece i1
// and receives the partner's piece i1 into slot i0.
template <int M>
__device__ __forceinline__ void exchange_pieces(uint32_t (&w)[32], bool bit) {
#pragma unroll
  for (int i0 = 0; i0 < 4; ++i0) {
    if (i0 & M) continue;
    const int i1 = i0 | M;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const uint32_t send = bit ? w[8 * i0 + t] : w[8 * i1 + t];
      const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, M);
      if (bit)
        w[8 * i0 + t] = recv;
      else
        w[8 * i1 + t] = recv;
    }
  }
}

// A warp holds 32 rows x 64 bf16 columns, one row per lane, as four 32-byte
// pieces w[8q, 8q + 8). After a 4 x 4 transpose of the pieces inside each
// group of four lanes, lane 4g + q holds piece q of rows 4g .. 4g + 3, and
// each of four 32-byte stores per lane writes whole 128-byte row segments
// (eight rows per instruction) instead of one 16-byte piece of 32 rows.
// `row_ptr` is this lane's output row at the block's first column (null for
// a row past the tile), 32-byte aligned; `valid` = columns left in the rows,
// a multiple of 16.
__device__ __forceinline__ void store_rows64(uint32_t (&w)[32], __nv_bfloat16* row_ptr,
                                             int valid, int lane) {
  exchange_pieces<1>(w, (lane & 1) != 0);
  exchange_pieces<2>(w, (lane & 2) != 0);
  const int q = lane & 3;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(__shfl_sync(
        0xffffffffu, reinterpret_cast<uintptr_t>(row_ptr), (lane & ~3) | r));
    if (dst != nullptr && q * 16 < valid)
      asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + q * 16),
                   "r"(w[8 * r]), "r"(w[8 * r + 1]), "r"(w[8 * r + 2]), "r"(w[8 * r + 3]),
                   "r"(w[8 * r + 4]), "r"(w[8 * r + 5]), "r"(w[8 * r + 6]), "r"(w[8 * r + 7])
                   : "memory");
  }
}

__device__ __forceinline__ void store32(float* dst, const float (&f)[32], int valid) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    if (q * 4 < valid)
      *reinterpret_cast<float4*>(dst + q * 4) = make_float4(f[q * 4], f[q * 4 + 1], f[q * 4 + 2], f[q * 4 + 3]);
  }
}

// Keeps the KT best (score, index) pairs in descending order. Candidates
// arrive in ascending expert order and displace only on a strictly larger
// score, so equal scores keep the lower index first.
template <int KT>
struct TopK {
  float v[KT];
  float z[KT];
  int i[KT];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      v[j] = -INFINITY;
      z[j] = 0.f;
      i[j] = 0x7fffffff;
    }
  }
  __device__ __forceinline__ void push(float q, int e, float ze) {
    if (!(q > v[KT - 1])) return;
    v[KT - 1] = q;
    i[KT - 1] = e;
    z[KT - 1] = ze;
#pragma unroll
    for (int j = KT - 1; j > 0; --j) {
      if (v[j] > v[j - 1]) {
        const float tv = v[j]; v[j] = v[j - 1]; v[j - 1] = tv;
        const float tz = z[j]; z[j] = z[j - 1]; z[j - 1] = tz;
        const int ti = i[j]; i[j] = i[j - 1]; i[j - 1] = ti;
      }
    }
  }
};

// One thread = one token: its logits are TMEM lane `row_in_tile`, columns
// [0, N). Passes over TMEM: (A) logits, their max, and without a bias the
// top-k on the logits (softmax and sigmoid are monotone); (B) softmax
// denominator when needed; (C) with a bias, the top-k on p + bias.
template <int KT>
__device__ __forceinline__ void route_epilogue(uint32_t tbase, int64_t row, bool valid, int n_pad,
                                               const RouteEpi& r) {
  const int N = r.N;
  const bool bias = r.sel_bias != nullptr;
  const bool softmax = r.score == MOE_SCORE_SOFTMAX;
  TopK<KT> top;
  top.init();
  float m = -INFINITY;
  float* zrow = r.logits_out != nullptr ? r.logits_out + row * N : nullptr;
  if (softmax && !bias && r.norm == MOE_NORM_NONE) {
    // selection on z alone and gates p_i = exp(z_i - m) / sum_j exp(z_j - m):
    // one pass over the accumulator, the sum of exponentials kept relative
    // to the running maximum and rescaled when a chunk raises it
    float s = 0.f;
#pragma unroll 1
    for (int c = 0; c < n_pad; c += 32) {
      uint32_t v[32];
      tmem_ld32_sync(tbase + c, v);
      if (valid) {
        float z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = c + i;
          z[i] = e < N ? __uint_as_float(v[i]) + (r.b_r != nullptr ? r.b_r[e] : 0.f) : -INFINITY;
          if (e < N && zrow != nullptr) zrow[e] = z[i];
        }
        float cm[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          cm[i] = fmaxf(fmaxf(z[4 * i], z[4 * i + 1]), fmaxf(z[4 * i + 2], z[4 * i + 3]));
        const float mc = fmaxf(fmaxf(fmaxf(cm[0], cm[1]), fmaxf(cm[2], cm[3])),
                               fmaxf(fmaxf(cm[4], cm[5]), fmaxf(cm[6], cm[7])));
        if (mc > m) {
          s *= __expf(m - mc);  // 0 on the first chunk (m = -inf)
          m = mc;
        }
        float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 32; ++i) part[i & 3] += __expf(z[i] - m);
        s += (part[0] + part[1]) + (part[2] + part[3]);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c + i < N) top.push(z[i], c + i, z[i]);
      }
    }
    if (!valid) return;
    const int k = r.k;
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      if (j < k) {
        r.idx[row * k + j] = top.i[j] == 0x7fffffff ? 0 : top.i[j];
        r.gate[row * k + j] = expf(top.z[j] - m) / s;
      }
    }
    return;
  }
#pragma unroll 1
  for (int c = 0; c < n_pad; c += 32) {
    uint32_t v[32];
    tmem_ld32_sync(tbase + c, v);
    if (valid) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int e = c + i;
        if (e < N) {
          const float z = __uint_as_float(v[i]) + (r.b_r != nullptr ? r.b_r[e] : 0.f);
          if (zrow != nullptr) zrow[e] = z;
          m = fmaxf(m, z);
          if (!bias) top.push(z, e, z);
        }
      }
    }
  }
  float s = 0.f;
  if (softmax && (bias || r.norm == MOE_NORM_NONE)) {
#pragma unroll 1
    for (int c = 0; c < n_pad; c += 32) {
      uint32_t v[32];
      tmem_ld32_sync(tbase + c, v);
      if (valid) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = c + i;
          if (e < N) {
            const float z = __uint_as_float(v[i]) + (r.b_r != nullptr ? r.b_r[e] : 0.f);
            s += expf(z - m);
          }
        }
      }
    }
  }
  if (bias) {
#pragma unroll 1
    for (int c = 0; c < n_pad; c += 32) {
      uint32_t v[32];
      tmem_ld32_sync(tbase + c, v);
      if (valid) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = c + i;
          if (e < N) {
            const float z = __uint_as_float(v[i]) + (r.b_r != nullptr ? r.b_r[e] : 0.f);
            const float pe = softmax ? expf(z - m) / s : 1.f / (1.f + expf(-z));
            top.push(pe + r.sel_bias[e], e, z);
          }
        }
      }
    }
  }
  if (!valid) return;
  const int k = r.k;
  float g[KT];
  float den = 0.f;
  if (softmax && r.norm == MOE_NORM_SELECTED) {
    float ms = -INFINITY;
#pragma unroll
    for (int j = 0; j < KT; ++j)
      if (j < k) ms = fmaxf(ms, top.z[j]);
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      g[j] = j < k ? expf(top.z[j] - ms) : 0.f;
      den += g[j];
    }
  } else if (softmax) {
#pragma unroll
    for (int j = 0; j < KT; ++j) g[j] = j < k ? expf(top.z[j] - m) / s : 0.f;
  } else {
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      g[j] = j < k ? 1.f / (1.f + expf(-top.z[j])) : 0.f;
      den += g[j];
    }
  }
  const bool renorm = r.norm == MOE_NORM_SELECTED;
#pragma unroll
  for (int j = 0; j < KT; ++j) {
    if (j < k) {
      r.idx[row * k + j] = top.i[j] == 0x7fffffff ? 0 : top.i[j];
      r.gate[row * k + j] = renorm ? g[j] / den : g[j];
    }
  }
}

// Epilogue of a swapped tile. Accumulator columns [0, nr) hold D0 = W0 X^T
// and [128, 128 + nr) hold D1 = W1 X^T, with W0/W1 the two 128-row halves of
// the stage's weight tile and X the tile's rows. Thread `lane_row` owns weight
// row lane_row of both halves:
//   gate/up: act[r][col0 + lane_row] = SiLU(D0[lane_row][r]) * D1[lane_row][r]
//   down:    y[r][col0 + lane_row] = D0, y[r][col0 + 128 + lane_row] = D1
//            (or gate * y into the token's output row when the combine is fused)
template <int MODE>
__device__ __forceinline__ void swap_epilogue(uint32_t tbase, const TileInfo& ti, int lane_row,
                                              const GemmParams& p) {
  using bf = __nv_bfloat16;
  constexpr int BN = MODE == kSwiGLU ? 128 : 256;
  const int c0 = ti.n_blk * BN + lane_row;
  const int c1 = c0 + 128;
  const int r0 = ti.row0 + ti.m_blk * kBM;  // first row of the tile in the routed operand
#pragma unroll 1
  for (int c = 0; c < ti.nr; c += 32) {
    uint32_t d0[32], d1[32];
    tmem_ld32_sync(tbase + c, d0);
    tmem_ld32_sync(tbase + kAccCols / 2 + c, d1);
    // fused combine: lane l reads the token and gate of the chunk's row c + l
    // once; the rows' values are then passed round by shuffles
    int lane_tok = 0;
    float lane_gate = 1.f;
    if (MODE == kDown && p.scatter_token != nullptr && c + (lane_row & 31) < ti.rv) {
      lane_tok = p.scatter_token[r0 + c + (lane_row & 31)];
      lane_gate = p.scatter_gate[lane_tok];
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int r = c + j;
      int tok = 0;
      float scale = 1.f;
      if (MODE == kDown && p.scatter_token != nullptr) {
        tok = __shfl_sync(0xffffffffu, lane_tok, j);
        scale = __shfl_sync(0xffffffffu, lane_gate, j);
      }
      if (r < ti.rv) {
        const float v0 = __uint_as_float(d0[j]);
        const float v1 = __uint_as_float(d1[j]);
        if (MODE == kSwiGLU) {
          if (c0 < ti.ncols)
            static_cast<bf*>(p.out)[static_cast<size_t>(r0 + r) * p.n_out + c0] =
                __float2bfloat16_rn(__fdividef(v0, 1.0f + __expf(-v0)) * v1);
        } else {
          const size_t base = p.scatter_token != nullptr ? static_cast<size_t>(tok) * p.n_out
                                                         : static_cast<size_t>(r0 + r) * p.n_out;
          bf* o = static_cast<bf*>(p.out) + base;
          if (c0 < ti.ncols) o[c0] = __float2bfloat16_rn(v0 * scale);
          if (c1 < ti.ncols) o[c1] = __float2bfloat16_rn(v1 * scale);
        }
      }
    }
  }
}

template <int MODE, typename T, int KT = 1>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap mapA0,
                        const __grid_constant__ CUtensorMap mapB0,
                        const __grid_constant__ CUtensorMap mapB0u,
                        const __grid_constant__ CUtensorMap mapA1,
                        const __grid_constant__ CUtensorMap mapB1,
                        const __grid_constant__ CUtensorMap mapB1u,
                        const __grid_constant__ CUtensorMap mapAs, const GemmParams p) {
  constexpr int BK = 128 / static_cast<int>(sizeof(T));   // elements per 128-byte row
  constexpr int BN = MODE == kSwiGLU ? 128 : 256;         // output columns per tile
  // kRoute / kLogits: one accumulator of n_out = N rounded up to 16 columns
  constexpr bool kRouter = MODE == kRoute || MODE == kLogits;
  const int mma_n = kRouter ? p.n_out : 256;
  const uint32_t idesc = make_idesc(kBM, mma_n, sizeof(T) == 2 ? 1u : 2u);
  // kRoute with two halves: a tile is 256 tokens, A0 in the A region, A1 and
  // W_r in the B region; one W_r load per K-step serves both, accumulated
  // into columns [0, n) and [128, 128 + n)
  const int halves = MODE == kRoute ? p.row_halves : 1;
  const uint32_t stage_tx = kRouter ? kStageA * static_cast<uint32_t>(halves) +
                                          static_cast<uint32_t>(mma_n) * 128u
                                    : kStageBytes;

  extern __shared__ uint8_t dyn_smem[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ int tile_start[kMaxGroups + 1];
  __shared__ int grp_off[kMaxGroups + 1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.n_routed + (p.rows_shared > 0 ? 1 : 0);
  volatile int* abort_v = &abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 128);
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&mapA0);
      tma_prefetch_desc(&mapB0);
      if (MODE == kSwiGLU) tma_prefetch_desc(&mapB0u);
    }
    if (kRouter) {
      if (lane == 0) { grp_off[0] = 0; grp_off[1] = p.rows_routed; }
    } else {
      for (int g = lane; g <= p.n_routed; g += 32) grp_off[g] = p.offsets[g];
    }
    __syncwarp();
    // offsets must start at 0, never decrease and end inside the operand
    bool bad = lane == 0 && (grp_off[0] != 0 || grp_off[p.n_routed] > p.rows_routed);
    for (int g = lane; g < p.n_routed; g += 32) bad |= grp_off[g + 1] < grp_off[g];
    bad = __any_sync(0xffffffffu, bad);
    if (bad) {
      if (lane == 0 && p.status != nullptr) atomicCAS(p.status, 0, MOE_ERR_DEVICE_CHECK);
      for (int g = lane; g <= p.n_routed; g += 32) grp_off[g] = 0;
      __syncwarp();
    }
    int carry = 0;
    for (int g0 = 0; g0 < G; g0 += 32) {
      const int g = g0 + lane;
      int tiles = 0;
      if (g < G) {
        const int rows = g < p.n_routed ? grp_off[g + 1] - grp_off[g] : p.rows_shared;
        const int ncols = g < p.n_routed ? p.n_out : p.n_out_shared;
        tiles = ((rows + kBM * halves - 1) / (kBM * halves)) *
                (MODE == kLogits ? p.k_splits : (ncols + BN - 1) / BN);
      }
      int incl = tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (g < G) tile_start[g] = carry + incl - tiles;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tile_start[G] = carry;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;
  const int total = tile_start[G];
  // Equal shares: the fewest CTAs that finish in the same number of rounds
  // take all the tiles (CTA c: tiles c, c + stride, ...), so that a pass
  // bound by reading its weights ends without a last round on a few SMs
  // (896 tiles: 128 CTAs x 7 instead of 148 x 6 plus 8).
  const int rounds = (total + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
  const int stride = rounds > 0 ? (total + rounds - 1) / rounds : static_cast<int>(gridDim.x);
  const int first = static_cast<int>(blockIdx.x) < stride ? static_cast<int>(blockIdx.x) : total;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Lane 0 waits for free stages, arms the barriers and issues the tiled
    // loads; when the routed rows come from h by index, every lane issues one
    // gather4 (4 of the tile's 128 rows) per stage.
    int stage = 0;
    uint32_t phase = 0, issued_mask = 0, issued_par = 0;
    bool ok = true;
    for (int tile = first; tile < total && ok; tile += stride) {
      int split = 0, kb0 = 0;
      TileInfo ti = MODE == kLogits  ? logits_tile(tile, p, split, kb0)
                    : MODE == kRoute ? route_tile(tile, p)
                                     : decode_tile<BN, BK>(tile, tile_start, grp_off, G, p);
      set_swap<MODE, T>(ti, p);
      const bool dense = ti.g >= p.n_routed;
      const bool gather = MODE == kSwiGLU && p.gather_rows != nullptr && !dense;
      const int nbox = ti.nr > 0 ? (ti.rv + kSwapBoxRows - 1) / kSwapBoxRows : 0;
      const uint32_t tile_tx = ti.nr > 0 ? kStageB + static_cast<uint32_t>(nbox) * kSwapBoxBytes
                                         : stage_tx;
      const void* mA = dense ? static_cast<const void*>(&mapA1) : static_cast<const void*>(&mapA0);
      const void* mB = dense ? static_cast<const void*>(&mapB1) : static_cast<const void*>(&mapB0);
      const void* mBu = dense ? static_cast<const void*>(&mapB1u) : static_cast<const void*>(&mapB0u);
      const int a_row = ti.row0 + ti.m_blk * kBM * halves;
      const int b_row = ti.b_row0 + ti.n_blk * BN;
      int g4[4] = {0, 0, 0, 0};
      if (gather) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          // rows past the routed rows repeat the last one (their results are masked)
          const int r = min(a_row + lane * 4 + i, grp_off[p.n_routed] - 1);
          g4[i] = p.gather_rows[r];
        }
      }
      for (int kb = 0; kb < ti.num_kb; ++kb) {
        bool w = true;
        if (lane == 0) {
          w = mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, abort_v, p.status, p.budget_ns,
                                MOE_ERR_TIMEOUT);
          if (w) mbar_arrive_expect_tx(&full_bar[stage], tile_tx);
        }
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) {
          ok = false;
          break;
        }
        uint8_t* sA = smem + stage * kStageBytes;
        uint8_t* sB = sA + kStageA;
        // gathered rows: one gather4 (4 rows) per lane, over the 32-row boxes
        // of a swapped tile or the whole 128-row tile
        if (gather && (ti.nr == 0 || lane < nbox * (kSwapBoxRows / 4)))
          tma_gather4(sA + lane * 512, mA, &full_bar[stage], (kb0 + kb) * BK, g4[0], g4[1], g4[2],
                      g4[3]);
        if (lane == 0) {
          if (ti.nr > 0 && !gather) {
            // the tile's valid rows as 32-row boxes, stacked like one taller box
            for (int b = 0; b < nbox; ++b)
              tma_load_2d(sA + b * kSwapBoxBytes, &mapAs, &full_bar[stage], (kb0 + kb) * BK,
                          a_row + b * kSwapBoxRows);
          } else if (!gather) {
            tma_load_2d(sA, mA, &full_bar[stage], (kb0 + kb) * BK, a_row);
          }
          if (MODE == kSwiGLU) {
            tma_load_2d(sB, mB, &full_bar[stage], (kb0 + kb) * BK, b_row);
            tma_load_2d(sB + kStageB / 2, mBu, &full_bar[stage], (kb0 + kb) * BK, b_row);
          } else if (MODE == kRoute && halves == 2) {
            tma_load_2d(sB, mA, &full_bar[stage], (kb0 + kb) * BK, a_row + kBM);
            tma_load_2d(sB + kStageA, mB, &full_bar[stage], (kb0 + kb) * BK, b_row);
          } else {
            tma_load_2d(sB, mB, &full_bar[stage], (kb0 + kb) * BK, b_row);
          }
          issued_mask |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        }
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) {
      for (int s = 0; s < kStages; ++s)
        if ((issued_mask >> s) & 1u) drain_wait(&full_bar[s], (issued_par >> s) & 1u);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = first; tile < total && ok; tile += stride) {
        int split = 0, kb0 = 0;
        TileInfo ti = MODE == kLogits  ? logits_tile(tile, p, split, kb0)
                      : MODE == kRoute ? route_tile(tile, p)
                                       : decode_tile<BN, BK>(tile, tile_start, grp_off, G, p);
        set_swap<MODE, T>(ti, p);
        const uint32_t idesc_swap = make_idesc(kBM, ti.nr > 0 ? ti.nr : 16, 1u);
        if (!mbar_wait_bounded(&tempty_bar[acc], acc_phase ^ 1u, abort_v, p.status, p.budget_ns,
                               MOE_ERR_TIMEOUT)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * kAccCols;
        for (int kb = 0; kb < ti.num_kb; ++kb) {
          if (!mbar_wait_bounded(&full_bar[stage], phase, abort_v, p.status, p.budget_ns,
                                 MOE_ERR_TIMEOUT)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * kStageBytes);
          const uint32_t b_addr = a_addr + kStageA;
          if (ti.nr > 0) {
            // swapped: the two 128-row weight halves of the B stage are the
            // A operands, the tile's rows the (narrow) B operand
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t xd = sw128_kmajor_desc(a_addr + kk * 32);
              const uint64_t w0 = sw128_kmajor_desc(b_addr + kk * 32);
              const uint64_t w1 = sw128_kmajor_desc(b_addr + kStageB / 2 + kk * 32);
              const uint32_t accum = (kb | kk) != 0 ? 1u : 0u;
              mma_f16(d_tmem, w0, xd, idesc_swap, accum);
              mma_f16(d_tmem + kAccCols / 2, w1, xd, idesc_swap, accum);
            }
          } else {
            const bool two = MODE == kRoute && halves == 2;
            const uint32_t w_addr = two ? b_addr + kStageA : b_addr;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = sw128_kmajor_desc(a_addr + kk * 32);
              const uint64_t bd = sw128_kmajor_desc(w_addr + kk * 32);
              const uint32_t accum = (kb | kk) != 0 ? 1u : 0u;
              if (sizeof(T) == 2)
                mma_f16(d_tmem, ad, bd, idesc, accum);
              else
                mma_tf32(d_tmem, ad, bd, idesc, accum);
              if (two)
                mma_f16(d_tmem + kAccCols / 2, sw128_kmajor_desc(b_addr + kk * 32), bd, idesc,
                        accum);
            }
          }
          mma_commit(&empty_bar[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&tfull_bar[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        mma_commit(&drain_bar);
        drain_wait(&drain_bar, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
    const int row_in_tile = quad * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = first; tile < total; tile += stride) {
      int split = 0, kb0 = 0;
      TileInfo ti = MODE == kLogits  ? logits_tile(tile, p, split, kb0)
                    : MODE == kRoute ? route_tile(tile, p)
                                     : decode_tile<BN, BK>(tile, tile_start, grp_off, G, p);
      set_swap<MODE, T>(ti, p);
      const int row = ti.m_blk * kBM * halves + row_in_tile;
      const bool row_ok = row < ti.rows;
      const int col0 = ti.n_blk * BN;
      const int cols_left = ti.ncols - col0;
      const bool dense = ti.g >= p.n_routed;
      T* out = dense ? static_cast<T*>(p.out_shared) + static_cast<size_t>(row) * p.n_out_shared
                     : static_cast<T*>(p.out) + static_cast<size_t>(ti.row0 + row) * p.n_out;
      float scale = 1.f;
      // the fused combine's token and gate are read before the wait for the
      // accumulator, so that their latency overlaps it
      if (MODE == kDown && p.scatter_token != nullptr && !dense && row_ok && ti.nr == 0) {
        const int tok = p.scatter_token[ti.row0 + row];
        scale = p.scatter_gate[tok];
        out = static_cast<T*>(p.out) + static_cast<size_t>(tok) * p.n_out;
      }
      out += col0;
      if (!mbar_wait_bounded(&tfull_bar[acc], acc_phase, abort_v, p.status, p.budget_ns,
                             MOE_ERR_TIMEOUT))
        break;
      tc_fence_after();
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc) * kAccCols;
      if (ti.nr > 0) {
        // swapped tile: this thread's TMEM lane is one output column (a row
        // of the weight tile), its TMEM columns are the tile's rows
        swap_epilogue<MODE>(tbase, ti, row_in_tile, p);
      } else if (MODE == kRoute) {
#pragma unroll 1
        for (int h = 0; h < halves; ++h)  // the tile's 128-row halves
          route_epilogue<KT>(tbase + h * (kAccCols / 2), row + h * kBM, row + h * kBM < ti.rows,
                             p.n_out, p.re);
      } else if (MODE == kLogits) {
        // this unit's partial logits, rows of the tile x n_out columns
        float* dst = p.partials +
                     (static_cast<size_t>(split) * p.rows_routed + static_cast<size_t>(row)) * p.n_out;
#pragma unroll 1
        for (int c = 0; c < p.n_out; c += 32) {
          uint32_t v[32];
          tmem_ld32_sync(tbase + c, v);
          if (row_ok) {
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
            store32(dst + c, f, p.n_out - c);
          }
        }
      } else if (MODE == kSwiGLU) {
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t gr[32], ur[32];
          tmem_ld32_sync(tbase + c, gr);
          tmem_ld32_sync(tbase + 128 + c, ur);
          if (row_ok && c < cols_left) {
            float act[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float gv = __uint_as_float(gr[i]);
              const float uv = __uint_as_float(ur[i]);
              act[i] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
            }
            store32(out + c, act, cols_left - c);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
          uint32_t v[32];
          tmem_ld32_sync(tbase + c, v);
          if (row_ok && c < cols_left) {
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]) * scale;
            store32(out + c, f, cols_left - c);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty_bar[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// CTA-pair variant (tcgen05.mma.cta_group::2): a cluster of two CTAs on two SMs
// computes one 256-row tile. Each CTA loads its own 128 rows of A and one half
// of the 256-row B tile (pass A: CTA 0 the W_gate rows, CTA 1 the W_up rows;
// pass B: one 128-row half of W_down each), so each SM fetches 32 KB per
// K-step instead of 48 KB for the same tensor-core work. The leader CTA (rank
// 0) issues the MMAs for the pair; both CTAs' TMA loads count on the leader's
// full barrier, the leader's commits arrive on both CTAs' empty and
// accumulator-full barriers, and both CTAs' epilogue threads arrive on the
// leader's accumulator-empty barrier. Each CTA drains its own 128 TMEM lanes.
//
// Short tails. A routed group whose last 256-row tile holds at most
// kPairSwapRows rows runs that tile with swapped operands: the weights are
// the M=256 side of the pair MMA (128 weight rows per CTA) and the tail rows
// the B operand, N = tail rounded up to 16, split N/2 per CTA (one 32-row box
// in a third 4 KB region of the stage). Pass A: CTA r holds W_gate rows
// f0 + 128 r + [0,128) in the A region and the same W_up rows in the B region;
// two MMAs give gate and up of those columns for every tail row in the
// accumulator's columns [0, N) and [128, 128 + N), so one swapped tile covers
// 256 output columns (a plain pass-A tile covers 128). Pass B: CTA r holds
// W_down rows c0 + 128 r + [0,128); one MMA covers the tile's 256 output
// columns. TMEM lane = output column; the epilogue writes back row by row.
// A tail of 4..64 rows no longer costs a 256 x 256 MMA per K-step.
//
// Two K-steps per stage (KS = 2): when every reduction width is a multiple of
// 64, each operand is also described as a 3-D tensor [K / 64][rows][64] and
// one TMA load brings 2 x 64 columns of 128 (or 32) rows: the two canonical
// K-major blocks of two K-steps, one after the other. Half the load
// instructions for the same bytes; three stages of 72 KB instead of six of
// 36 KB.
constexpr uint32_t kPairStepA = 128 * 128;          // A rows of one K-step
constexpr uint32_t kPairStepB = 128 * 128;          // B rows of one K-step
constexpr uint32_t kPairStepX = kSwapBoxBytes;      // tail rows of a swapped tile
template <int KS>
struct PairStage {
  static constexpr int kStages = KS == 1 ? MOE_PAIR_STAGES : 3;
  static constexpr uint32_t A = KS * kPairStepA, B = KS * kPairStepB, X = KS * kPairStepX;
  static constexpr uint32_t kBytes = A + B + X;
  static constexpr size_t kDynSmem = static_cast<size_t>(kStages) * kBytes + 1024;
};
constexpr int kPairMaxStages = MOE_PAIR_STAGES > 3 ? MOE_PAIR_STAGES : 3;
#ifndef MOE_PAIR_TWO_K
#define MOE_PAIR_TWO_K 1
#endif
constexpr bool kPairTwoK = MOE_PAIR_TWO_K != 0;
static_assert(kPairSwapRows <= 2 * kSwapBoxRows, "a CTA's half of a swapped tail fits one box");

// Epilogue of a swapped tail of the pair kernel. Accumulator columns [0, N)
// hold W0 X^T and (pass A) [128, 128 + N) hold W1 X^T, with W0 / W1 this
// CTA's 128 rows of W_gate / W_up (pass A) or of W_down (pass B) and X the
// tile's rows; thread `lane_row` owns output column
// o = 256 n_blk + 128 rank + lane_row:
//   gate/up: act[r][o] = SiLU(W_gate X^T) * (W_up X^T)
//   down:    y[r][o] = W_down X^T (or gate * y into the token's row when the
//            combine is fused)
template <int MODE>
__device__ __forceinline__ void pair_swap_epilogue(uint32_t tbase, const TileInfo& ti,
                                                   int lane_row, int rank,
                                                   const GemmParams& p) {
  using bf = __nv_bfloat16;
  const int o = ti.n_blk * 256 + rank * 128 + lane_row;
  const int r0 = ti.row0 + ti.m_blk * 256;
#pragma unroll 1
  for (int c = 0; c < ti.nr; c += 32) {
    uint32_t d0[32], d1[32];
    tmem_ld32_sync(tbase + c, d0);
    if (MODE == kSwiGLU) tmem_ld32_sync(tbase + kAccCols / 2 + c, d1);
    // fused combine: lane l reads the token and gate of the chunk's row c + l
    // once; the rows' values are then passed round by shuffles
    int lane_tok = 0;
    float lane_gate = 1.f;
    if (MODE == kDown && p.scatter_token != nullptr && c + (lane_row & 31) < ti.rv) {
      lane_tok = p.scatter_token[r0 + c + (lane_row & 31)];
      lane_gate = p.scatter_gate[lane_tok];
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int r = c + j;
      int tok = 0;
      float scale = 1.f;
      if (MODE == kDown && p.scatter_token != nullptr) {
        tok = __shfl_sync(0xffffffffu, lane_tok, j);
        scale = __shfl_sync(0xffffffffu, lane_gate, j);
      }
      if (r < ti.rv && o < ti.ncols) {
        const float v0 = __uint_as_float(d0[j]);
        if (MODE == kSwiGLU) {
          const float v1 = __uint_as_float(d1[j]);
          static_cast<bf*>(p.out)[static_cast<size_t>(r0 + r) * p.n_out + o] =
              __float2bfloat16_rn(__fdividef(v0, 1.0f + __expf(-v0)) * v1);
        } else {
          const size_t base = p.scatter_token != nullptr ? static_cast<size_t>(tok) * p.n_out
                                                         : static_cast<size_t>(r0 + r) * p.n_out;
          static_cast<bf*>(p.out)[base + o] = __float2bfloat16_rn(v0 * scale);
        }
      }
    }
  }
}

// Tile `tile` of the pair kernel: the band-ordered plain tiles of each group,
// then (for a swapped tail) its n-tiles of the swapped form. ti.nr = MMA N of
// a swapped tail (0 for a plain tile), ti.rv = valid rows of the tile.
template <int MODE, int BN, int BK>
__device__ __forceinline__ TileInfo decode_pair_tile(int tile, const int* tile_start,
                                                     const int* grp_off, int G,
                                                     const GemmParams& p) {
  constexpr int BM = 256;
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_start[mid] <= tile) lo = mid; else hi = mid;
  }
  TileInfo ti;
  ti.g = lo;
  if (lo < p.n_routed) {
    ti.row0 = grp_off[lo];
    ti.rows = grp_off[lo + 1] - grp_off[lo];
    ti.ncols = p.n_out;
    ti.b_row0 = lo * p.n_out;
    ti.num_kb = (p.K + BK - 1) / BK;
  } else {
    ti.row0 = 0;
    ti.rows = p.rows_shared;
    ti.ncols = p.n_out_shared;
    ti.b_row0 = 0;
    ti.num_kb = (p.K_shared + BK - 1) / BK;
  }
  const int tail = ti.rows % BM;
  const bool swap = pair_swap_tail<MODE>(lo, tail, p);
  const int mt = ti.rows / BM + (tail > 0 && !swap ? 1 : 0);  // plain m-tiles
  const int nt = (ti.ncols + BN - 1) / BN;
  const int l = tile - tile_start[lo];
  ti.nr = 0;
  if (l >= mt * nt) {
    // swapped tail: n-tiles of 256 output columns (pass A) or BN (pass B)
    ti.m_blk = ti.rows / BM;
    ti.n_blk = l - mt * nt;
    ti.rv = tail;
    ti.nr = (tail + 15) / 16 * 16;
    return ti;
  }
  const int nbands0 = (mt + kBandMax * kBM / BM - 1) / (kBandMax * kBM / BM);
  const int band_sz = (mt + nbands0 - 1) / nbands0;
  const int band = l / (band_sz * nt);
  const int r = l - band * band_sz * nt;
  const int bs = min(band_sz, mt - band * band_sz);
  ti.n_blk = r / bs;
  ti.m_blk = band * band_sz + (r - ti.n_blk * bs);
  ti.rv = min(BM, ti.rows - ti.m_blk * BM);
  return ti;
}

template <int MODE, int KS>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap mapA0,
                             const __grid_constant__ CUtensorMap mapB0,
                             const __grid_constant__ CUtensorMap mapB0u,
                             const __grid_constant__ CUtensorMap mapA1,
                             const __grid_constant__ CUtensorMap mapB1,
                             const __grid_constant__ CUtensorMap mapB1u,
                             const __grid_constant__ CUtensorMap mapAs, const GemmParams p) {
  using T = __nv_bfloat16;
  using PS = PairStage<KS>;
  constexpr int kPairStages = PS::kStages;
  constexpr uint32_t kPairStageA = PS::A, kPairStageB = PS::B, kPairStageBytes = PS::kBytes;
  constexpr int BK = 64;
  constexpr int BM = 256;                                  // rows per pair tile
  constexpr int BN = MODE == kSwiGLU ? 128 : 256;
  const uint32_t idesc = make_idesc(BM, 256, 1u);

  extern __shared__ uint8_t dyn_smem[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full_bar[kPairMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kPairMaxStages];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ int tile_start[kMaxGroups + 1];
  __shared__ int grp_off[kMaxGroups + 1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int G = p.n_routed + (p.rows_shared > 0 ? 1 : 0);
  volatile int* abort_v = &abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 256);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&tmem_base_sh, kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&mapA0);
      tma_prefetch_desc(&mapB0);
      if (MODE == kSwiGLU) tma_prefetch_desc(&mapB0u);
    }
    for (int g = lane; g <= p.n_routed; g += 32) grp_off[g] = p.offsets[g];
    __syncwarp();
    bool bad = lane == 0 && (grp_off[0] != 0 || grp_off[p.n_routed] > p.rows_routed);
    for (int g = lane; g < p.n_routed; g += 32) bad |= grp_off[g + 1] < grp_off[g];
    bad = __any_sync(0xffffffffu, bad);
    if (bad) {
      if (lane == 0 && p.status != nullptr) atomicCAS(p.status, 0, MOE_ERR_DEVICE_CHECK);
      for (int g = lane; g <= p.n_routed; g += 32) grp_off[g] = 0;
      __syncwarp();
    }
    int carry = 0;
    for (int g0 = 0; g0 < G; g0 += 32) {
      const int g = g0 + lane;
      int tiles = 0;
      if (g < G) {
        const int rows = g < p.n_routed ? grp_off[g + 1] - grp_off[g] : p.rows_shared;
        const int ncols = g < p.n_routed ? p.n_out : p.n_out_shared;
        const int nt = (ncols + BN - 1) / BN;
        if (pair_swap_tail<MODE>(g, rows % BM, p))
          tiles = (rows / BM) * nt + (MODE == kSwiGLU ? (ncols + 255) / 256 : nt);
        else
          tiles = ((rows + BM - 1) / BM) * nt;
      }
      int incl = tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (g < G) tile_start[g] = carry + incl - tiles;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tile_start[G] = carry;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // barriers of both CTAs initialised before any cross-CTA use
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;
  const int total = tile_start[G];
  const int cluster_id = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = cluster_id; tile < total && ok; tile += n_clusters) {
      const TileInfo ti = decode_pair_tile<MODE, BN, BK>(tile, tile_start, grp_off, G, p);
      const bool dense = ti.g >= p.n_routed;
      const bool gather = MODE == kSwiGLU && p.gather_rows != nullptr && !dense;
      const bool swapped = ti.nr > 0;
      // bytes per stage of both CTAs: plain tiles A + B; swapped tails the
      // weight rows (both halves in pass A, one in pass B) and the tail box
      const uint32_t tile_tx =
          KS * (swapped ? 2 * ((MODE == kSwiGLU ? kPairStepA + kPairStepB : kPairStepA) + kPairStepX)
                        : 2 * (kPairStepA + kPairStepB));
      const int n_stages = (ti.num_kb + KS - 1) / KS;
      const void* mA = dense ? static_cast<const void*>(&mapA1) : static_cast<const void*>(&mapA0);
      const void* mB;
      int b_row;
      if (MODE == kSwiGLU) {
        // CTA 0 holds the W_gate half of B, CTA 1 the W_up half
        mB = leader ? (dense ? static_cast<const void*>(&mapB1) : static_cast<const void*>(&mapB0))
                    : (dense ? static_cast<const void*>(&mapB1u) : static_cast<const void*>(&mapB0u));
        b_row = ti.b_row0 + ti.n_blk * BN;
      } else {
        mB = dense ? static_cast<const void*>(&mapB1) : static_cast<const void*>(&mapB0);
        b_row = ti.b_row0 + ti.n_blk * BN + static_cast<int>(rank) * 128;
      }
      // a swapped tail: CTA r holds tail rows [r N/2, r N/2 + 32) and weight
      // rows 128 r + [0,128) of the tile's 256 output columns
      const int a_row = swapped ? ti.row0 + ti.m_blk * BM + static_cast<int>(rank) * (ti.nr / 2)
                                : ti.row0 + ti.m_blk * BM + static_cast<int>(rank) * 128;
      const int w_row = ti.b_row0 + ti.n_blk * 256 + static_cast<int>(rank) * 128;
      int g4[4] = {0, 0, 0, 0};
      if (gather) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = min(a_row + lane * 4 + i, grp_off[p.n_routed] - 1);
          g4[i] = p.gather_rows[r];
        }
      }
      for (int ks = 0; ks < n_stages; ++ks) {
        const int kb = ks * KS;  // first 64-column block of the stage
        bool w = true;
        if (lane == 0)
          w = mbar_wait_bounded_cluster(&empty_bar[stage], phase ^ 1u, abort_v, p.status,
                                        p.budget_ns, MOE_ERR_TIMEOUT);
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) {
          ok = false;
          break;
        }
        uint8_t* sA = smem + stage * kPairStageBytes;
        uint8_t* sB = sA + kPairStageA;
        uint8_t* sX = sB + kPairStageB;
        const uint32_t full_leader = mapa_shared(smem_u32(&full_bar[stage]), 0);
        if (lane == 0 && leader) mbar_arrive_expect_tx(&full_bar[stage], tile_tx);
        __syncwarp();
        // one load of a tiled operand: a 2-D box (KS = 1) or the 3-D box of
        // the stage's two 64-column blocks (KS = 2)
        auto load = [&](uint8_t* dst, const void* map, int row) {
          if (KS == 1)
            tma_load_2d_pair(dst, map, full_leader, kb * BK, row);
          else
            tma_load_3d_pair(dst, map, full_leader, 0, row, kb);
        };
        if (swapped) {
          // tail rows into the X region (a 32-row box, or 8 gather4 lanes per block)
          if (gather) {
            if (lane < kSwapBoxRows / 4)
              for (int c = 0; c < KS; ++c)
                tma_gather4_pair(sX + c * kPairStepX + lane * 512, mA, full_leader, (kb + c) * BK,
                                 g4[0], g4[1], g4[2], g4[3]);
          } else if (lane == 0) {
            load(sX, &mapAs, a_row);
          }
          if (lane == 0) {
            if (MODE == kSwiGLU) {
              load(sA, &mapB0, w_row);    // W_gate rows
              load(sB, &mapB0u, w_row);   // W_up rows
            } else {
              load(sA, &mapB0, w_row);    // W_down rows
            }
          }
        } else {
          if (gather)
            for (int c = 0; c < KS; ++c)
              tma_gather4_pair(sA + c * kPairStepA + lane * 512, mA, full_leader, (kb + c) * BK,
                               g4[0], g4[1], g4[2], g4[3]);
          if (lane == 0) {
            if (!gather) load(sA, mA, a_row);
            load(sB, mB, b_row);
          }
        }
        if (++stage == kPairStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) {
      // let loads already issued land before the CTA can leave
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 2000000ull) {
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------- MMA issuer (leader)
    if (lane == 0 && leader) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = cluster_id; tile < total && ok; tile += n_clusters) {
        const TileInfo ti = decode_pair_tile<MODE, BN, BK>(tile, tile_start, grp_off, G, p);
        const uint32_t idesc_swap = make_idesc(BM, ti.nr > 0 ? ti.nr : 16, 1u);
        if (!mbar_wait_bounded_cluster(&tempty_bar[acc], acc_phase ^ 1u, abort_v, p.status,
                                       p.budget_ns, MOE_ERR_TIMEOUT)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * kAccCols;
        const int n_stages = (ti.num_kb + KS - 1) / KS;
        for (int ks = 0; ks < n_stages; ++ks) {
          if (!mbar_wait_bounded_cluster(&full_bar[stage], phase, abort_v, p.status, p.budget_ns,
                                         MOE_ERR_TIMEOUT)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * kPairStageBytes);
          const uint32_t b_addr = a_addr + kPairStageA;
          // a last stage of KS = 2 past the reduction width holds zero-filled
          // columns (their products add nothing)
#pragma unroll
          for (int c = 0; c < KS; ++c) {
            const uint32_t ac = a_addr + c * kPairStepA, bc = b_addr + c * kPairStepB;
            if (ti.nr > 0) {
              // swapped tail: weights (A region; W_up in the B region) x tail rows
              const uint32_t xc = b_addr + kPairStageB + c * kPairStepX;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t xd = sw128_kmajor_desc(xc + kk * 32);
                const uint32_t accum = (ks | c | kk) != 0 ? 1u : 0u;
                mma_f16_pair(d_tmem, sw128_kmajor_desc(ac + kk * 32), xd, idesc_swap, accum);
                if (MODE == kSwiGLU)
                  mma_f16_pair(d_tmem + kAccCols / 2, sw128_kmajor_desc(bc + kk * 32), xd,
                               idesc_swap, accum);
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = sw128_kmajor_desc(ac + kk * 32);
                const uint64_t bd = sw128_kmajor_desc(bc + kk * 32);
                mma_f16_pair(d_tmem, ad, bd, idesc, (ks | c | kk) != 0 ? 1u : 0u);
              }
            }
          }
          mma_commit_pair(&empty_bar[stage], 0x3);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair(&tfull_bar[acc], 0x3);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        // wait (bounded) for the MMAs already issued
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int row_in_tile = quad * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = cluster_id; tile < total; tile += n_clusters) {
      const TileInfo ti = decode_pair_tile<MODE, BN, BK>(tile, tile_start, grp_off, G, p);
      const int row = ti.m_blk * BM + static_cast<int>(rank) * 128 + row_in_tile;
      const bool row_ok = row < ti.rows;
      const int col0 = ti.n_blk * BN;
      const int cols_left = ti.ncols - col0;
      const bool dense = ti.g >= p.n_routed;
      T* out = dense ? static_cast<T*>(p.out_shared) + static_cast<size_t>(row) * p.n_out_shared
                     : static_cast<T*>(p.out) + static_cast<size_t>(ti.row0 + row) * p.n_out;
      float scale = 1.f;
      // the fused combine's token and gate are read before the wait for the
      // accumulator, so that their latency overlaps it
      if (MODE == kDown && p.scatter_token != nullptr && !dense && row_ok && ti.nr == 0) {
        const int tok = p.scatter_token[ti.row0 + row];
        scale = p.scatter_gate[tok];
        out = static_cast<T*>(p.out) + static_cast<size_t>(tok) * p.n_out;
      }
      out += col0;
      if (!mbar_wait_bounded_cluster(&tfull_bar[acc], acc_phase, abort_v, p.status, p.budget_ns,
                                     MOE_ERR_TIMEOUT))
        break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(acc) * kAccCols;
      // whole 128-byte row segments per store when every row starts on a
      // 32-byte boundary
      const bool wide = ((dense ? p.n_out_shared : p.n_out) & 15) == 0 &&
                        (reinterpret_cast<uintptr_t>(dense ? p.out_shared : p.out) & 31) == 0;
      if (ti.nr > 0) {
        // swapped tail: TMEM lane = output column 256 n + 128 rank + lane_row
        pair_swap_epilogue<MODE>(tbase, ti, row_in_tile, static_cast<int>(rank), p);
      } else if (wide) {
        constexpr int kCols = MODE == kSwiGLU ? 128 : 256;
#pragma unroll 1
        for (int c = 0; c < kCols; c += 64) {
          uint32_t w[32];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float f[32];
            if (MODE == kSwiGLU) {
              uint32_t gr[32], ur[32];
              tmem_ld32_sync(tbase + c + 32 * h, gr);
              tmem_ld32_sync(tbase + 128 + c + 32 * h, ur);
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const float gv = __uint_as_float(gr[i]);
                f[i] = __fdividef(gv, 1.0f + __expf(-gv)) * __uint_as_float(ur[i]);
              }
            } else {
              uint32_t v[32];
              tmem_ld32_sync(tbase + c + 32 * h, v);
#pragma unroll
              for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]) * scale;
            }
            pack_bf16x32(f, w + 16 * h);
          }
          if (c < cols_left)  // the same for the whole warp
            store_rows64(w, row_ok ? out + c : nullptr, cols_left - c, lane);
        }
      } else if (MODE == kSwiGLU) {
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t gr[32], ur[32];
          tmem_ld32_sync(tbase + c, gr);
          tmem_ld32_sync(tbase + 128 + c, ur);
          if (row_ok && c < cols_left) {
            float act[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float gv = __uint_as_float(gr[i]);
              const float uv = __uint_as_float(ur[i]);
              act[i] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
            }
            store32(out + c, act, cols_left - c);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
          uint32_t v[32];
          tmem_ld32_sync(tbase + c, v);
          if (row_ok && c < cols_left) {
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]) * scale;
            store32(out + c, f, cols_left - c);
          }
        }
      }
      tc_fence_before();
      mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while its peer may still signal its barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// One CTA, one thread: waits on an mbarrier nothing arrives on, bounded.
__global__ void selftest_wait_kernel(int32_t* status, uint64_t budget_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  mbar_init(&bar, 1);
  abort_flag = 0;
  fence_mbar_init();
  volatile int* ab = &abort_flag;
  (void)mbar_wait_bounded(&bar, 0, ab, status, budget_ns, MOE_ERR_TIMEOUT);
}

// ------------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// Row-major [rows, inner] tensor, box = [box_rows, 128 bytes], 128-byte swizzle,
// zero fill outside the tensor.
bool make_map(CUtensorMap* m, const void* ptr, int dtype, uint64_t inner, uint64_t rows,
              uint32_t box_rows) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const uint64_t es = static_cast<uint64_t>(elem_size(dtype));
  cuuint64_t gdim[2] = {inner, rows};
  cuuint64_t gstride[1] = {inner * es};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / es), box_rows};
  cuuint32_t estr[2] = {1, 1};
  // fp32 operands are rounded to tf32 by the TMA unit on the way to shared memory
  const CUtensorMapDataType dt =
      dtype == MOE_F32 ? CU_TENSOR_MAP_DATA_TYPE_TFLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUresult r = enc(m, dt, 2, const_cast<void*>(ptr), gdim, gstride, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The same row-major [rows, inner] tensor as a 3-D tensor [inner / 64][rows][64]
// (dims innermost first: 64 elements, rows, 64-element blocks), box = 64 x
// box_rows x 2 with the 128-byte swizzle: one load brings two 64-column blocks
// of box_rows rows, each block a contiguous K-major tile. Needs inner % 64 == 0
// (a block must not run into the next row); returns false when the driver
// does not accept the description.
bool make_map_2k(CUtensorMap* m, const void* ptr, int dtype, uint64_t inner, uint64_t rows,
                 uint32_t box_rows) {
  auto enc = encode_fn();
  if (enc == nullptr || dtype != MOE_BF16 || inner % 64 != 0) return false;
  cuuint64_t gdim[3] = {64, rows, inner / 64};
  cuuint64_t gstride[2] = {inner * 2, 128};
  cuuint32_t box[3] = {64, box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), gdim,
                         gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int MODE, typename T, int KT = 1>
cudaError_t launch_gemm(const CUtensorMap* maps, const GemmParams& p, int grid, cudaStream_t stream) {
  auto kern = grouped_gemm_kernel<MODE, T, KT>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kDynSmem));
  if (err != cudaSuccess) return err;
  kern<<<grid, kThreads, kDynSmem, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5],
                                              maps[6], p);
  return cudaGetLastError();
}

int tiles_bound(int64_t rows_routed, int n_groups, int64_t n_out, int BN, int64_t rows_dense,
                int64_t n_out_dense, int BM = kBM) {
  int64_t b = (rows_routed / BM + n_groups) * ((n_out + BN - 1) / BN);
  if (rows_dense > 0) b += ((rows_dense + BM - 1) / BM) * ((n_out_dense + BN - 1) / BN);
  return static_cast<int>(b < 1 ? 1 : (b > (1 << 30) ? (1 << 30) : b));
}

// Clusters of two CTAs that can be resident at once (one CTA per SM), cached
// per device and kernel instance (`slot`).
int pair_clusters(const void* kern, cudaLaunchConfig_t cfg, int slot) {
  static int cache[64][4] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cache[dev][slot] > 0) return cache[dev][slot];
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = num_sms() / 2;
  }
  if (dev >= 0 && dev < 64) cache[dev][slot] = n;
  return n;
}

template <int MODE, int KS>
cudaError_t launch_gemm_pair(const CUtensorMap* maps, const GemmParams& p, int pair_tiles,
                             cudaStream_t stream) {
  auto kern = grouped_gemm_pair_kernel<MODE, KS>;
  constexpr size_t kPairDynSmem = PairStage<KS>::kDynSmem;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kPairDynSmem));
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kPairDynSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2, 1, 1);
  int clusters = pair_clusters(reinterpret_cast<const void*>(kern), cfg,
                               (MODE == kSwiGLU ? 0 : 1) + (KS == 2 ? 2 : 0));
  if (clusters > pair_tiles) clusters = pair_tiles;
  if (clusters < 1) clusters = 1;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  err = cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5],
                           maps[6], p);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

cudaError_t launch_expert_ffn(const FfnArgs& a, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  const int64_t R = a.rows > 0 ? a.rows : a.T * a.k;
  const bool sh = a.F_sh > 0;
  const int sms = num_sms();
  CUtensorMap m[7];

  // pass A: act = SiLU(x Wg^T) * (x Wu^T); x is the dispatched copy, or the
  // rows of h picked by index (gather4, 1-row box) when gather_rows is given.
  // m[6]: x in 32-row boxes for the swapped tiles (not used when gathering)
  const bool gather = a.gather_rows != nullptr;
  if (gather) {
    if (!make_map(&m[0], a.h, a.dtype, a.d, a.T, 1)) return cudaErrorInvalidValue;
    m[6] = m[0];
  } else if (!make_map(&m[0], a.x_disp, a.dtype, a.d, R, kBM) ||
             !make_map(&m[6], a.x_disp, a.dtype, a.d, R, kSwapBoxRows)) {
    return cudaErrorInvalidValue;
  }
  if (!make_map(&m[1], a.W_gate, a.dtype, a.d, static_cast<uint64_t>(a.N) * a.F, 128)) return cudaErrorInvalidValue;
  if (!make_map(&m[2], a.W_up, a.dtype, a.d, static_cast<uint64_t>(a.N) * a.F, 128)) return cudaErrorInvalidValue;
  if (sh) {
    if (!make_map(&m[3], a.h, a.dtype, a.d, a.T, kBM)) return cudaErrorInvalidValue;
    if (!make_map(&m[4], a.Ws_gate, a.dtype, a.d, a.F_sh, 128)) return cudaErrorInvalidValue;
    if (!make_map(&m[5], a.Ws_up, a.dtype, a.d, a.F_sh, 128)) return cudaErrorInvalidValue;
  } else {
    m[3] = m[0]; m[4] = m[1]; m[5] = m[2];
  }
  GemmParams pa{};
  pa.offsets = a.offsets;
  pa.n_routed = a.N;
  pa.rows_routed = static_cast<int32_t>(R);
  pa.rows_shared = sh ? static_cast<int32_t>(a.T) : 0;
  pa.K = a.d;
  pa.K_shared = a.d;
  pa.n_out = a.F;
  pa.n_out_shared = a.F_sh;
  pa.out = a.act;
  pa.out_shared = a.act_sh;
  pa.status = a.status;
  pa.budget_ns = kWaitBudgetNs;
  pa.gather_rows = a.gather_rows;
  // CTA pairs (256-row tiles) pay off when experts hold many rows on average;
  // with few rows per expert the 128-row tiles waste less of the MMA.
  const bool pair = a.dtype == MOE_BF16 && R >= static_cast<int64_t>(kPairMinRowsPerExpert) * a.N;
  // CTA pairs with two K-steps per stage when every reduction width is a
  // multiple of 64 and the driver accepts the 3-D descriptions (else one)
  const bool widths_2k = kPairTwoK && a.d % 64 == 0 && a.F % 64 == 0 && a.F_sh % 64 == 0;
  cudaError_t err;
  if (pair) {
    const int bound = tiles_bound(R, a.N, a.F, 128, sh ? a.T : 0, a.F_sh, 256);
    CUtensorMap m2[7];
    bool two_k = widths_2k &&
                 make_map_2k(&m2[1], a.W_gate, a.dtype, a.d, static_cast<uint64_t>(a.N) * a.F, 128) &&
                 make_map_2k(&m2[2], a.W_up, a.dtype, a.d, static_cast<uint64_t>(a.N) * a.F, 128);
    if (two_k && gather) {
      m2[0] = m[0];  // gather4 reads the 2-D map, one load per 64-column block
      m2[6] = m[0];
    } else if (two_k) {
      two_k = make_map_2k(&m2[0], a.x_disp, a.dtype, a.d, R, kBM) &&
              make_map_2k(&m2[6], a.x_disp, a.dtype, a.d, R, kSwapBoxRows);
    }
    if (two_k && sh) {
      two_k = make_map_2k(&m2[3], a.h, a.dtype, a.d, a.T, kBM) &&
              make_map_2k(&m2[4], a.Ws_gate, a.dtype, a.d, a.F_sh, 128) &&
              make_map_2k(&m2[5], a.Ws_up, a.dtype, a.d, a.F_sh, 128);
    } else if (two_k) {
      m2[3] = m2[0]; m2[4] = m2[1]; m2[5] = m2[2];
    }
    err = two_k ? launch_gemm_pair<kSwiGLU, 2>(m2, pa, bound, stream)
                : launch_gemm_pair<kSwiGLU, 1>(m, pa, bound, stream);
  } else {
    int grid = tiles_bound(R, a.N, a.F, 128, sh ? a.T : 0, a.F_sh);
    if (grid > sms) grid = sms;
    err = a.dtype == MOE_F32 ? launch_gemm<kSwiGLU, float>(m, pa, grid, stream)
                             : launch_gemm<kSwiGLU, __nv_bfloat16>(m, pa, grid, stream);
  }
  if (err != cudaSuccess) return err;

  // pass B: y = act Wd^T
  if (!make_map(&m[0], a.act, a.dtype, a.F, R, kBM) ||
      !make_map(&m[6], a.act, a.dtype, a.F, R, kSwapBoxRows))
    return cudaErrorInvalidValue;
  // a CTA pair splits the 256 B rows of a down tile 128/128 between its CTAs
  const uint32_t down_box = pair ? 128 : 256;
  if (!make_map(&m[1], a.W_down, a.dtype, a.F, static_cast<uint64_t>(a.N) * a.d, down_box))
    return cudaErrorInvalidValue;
  m[2] = m[1];
  if (sh) {
    if (!make_map(&m[3], a.act_sh, a.dtype, a.F_sh, a.T, kBM)) return cudaErrorInvalidValue;
    if (!make_map(&m[4], a.Ws_down, a.dtype, a.F_sh, a.d, down_box)) return cudaErrorInvalidValue;
    m[5] = m[4];
  } else {
    m[3] = m[0]; m[4] = m[1]; m[5] = m[1];
  }
  GemmParams pb = pa;
  pb.gather_rows = nullptr;
  pb.scatter_token = a.scatter_token;
  pb.scatter_gate = a.scatter_gate;
  pb.K = a.F;
  pb.K_shared = a.F_sh;
  pb.n_out = a.d;
  pb.n_out_shared = a.d;
  pb.out = a.scatter_token != nullptr ? a.scatter_out : a.y_rows;
  pb.out_shared = a.y_shared;
  if (pair) {
    const int bound = tiles_bound(R, a.N, a.d, 256, sh ? a.T : 0, a.d, 256);
    CUtensorMap m2[7];
    bool two_k = widths_2k &&
                 make_map_2k(&m2[0], a.act, a.dtype, a.F, R, kBM) &&
                 make_map_2k(&m2[6], a.act, a.dtype, a.F, R, kSwapBoxRows) &&
                 make_map_2k(&m2[1], a.W_down, a.dtype, a.F, static_cast<uint64_t>(a.N) * a.d, 128);
    m2[2] = m2[1];
    if (two_k && sh) {
      two_k = make_map_2k(&m2[3], a.act_sh, a.dtype, a.F_sh, a.T, kBM) &&
              make_map_2k(&m2[4], a.Ws_down, a.dtype, a.F_sh, a.d, 128);
      m2[5] = m2[4];
    } else if (two_k) {
      m2[3] = m2[0]; m2[4] = m2[1]; m2[5] = m2[1];
    }
    return two_k ? launch_gemm_pair<kDown, 2>(m2, pb, bound, stream)
                 : launch_gemm_pair<kDown, 1>(m, pb, bound, stream);
  }
  int grid = tiles_bound(R, a.N, a.d, 256, sh ? a.T : 0, a.d);
  if (grid > sms) grid = sms;
  return a.dtype == MOE_F32 ? launch_gemm<kDown, float>(m, pb, grid, stream)
                            : launch_gemm<kDown, __nv_bfloat16>(m, pb, grid, stream);
}

bool route_on_tensor_cores(const RouteArgs& a) {
  return a.h != nullptr && a.dtype == MOE_BF16 && a.N <= 256;
}

cudaError_t launch_route_logits(const RouteArgs& a, cudaStream_t stream) {
  const RouteSplit rs = route_split(a.T, a.d, a.N);
  CUtensorMap m[7];
  if (!make_map(&m[0], a.h, a.dtype, a.d, a.T, kBM)) return cudaErrorInvalidValue;
  if (!make_map(&m[1], a.W_r, a.dtype, a.d, a.N, static_cast<uint32_t>(rs.n_pad)))
    return cudaErrorInvalidValue;
  m[2] = m[1]; m[3] = m[0]; m[4] = m[1]; m[5] = m[1]; m[6] = m[0];
  GemmParams p{};
  p.offsets = nullptr;
  p.n_routed = 1;
  p.rows_routed = static_cast<int32_t>(a.T);
  p.rows_shared = 0;
  p.K = a.d;
  p.K_shared = a.d;
  p.n_out = rs.n_pad;
  p.n_out_shared = 0;
  p.status = a.status;
  p.budget_ns = kWaitBudgetNs;
  p.partials = a.partials;
  p.k_splits = rs.splits;
  p.kb_per_split = rs.kb_per_split;
  const int64_t units = (a.T + kBM - 1) / kBM * rs.splits;
  const int grid = static_cast<int>(units < num_sms() ? units : num_sms());
  return launch_gemm<kLogits, __nv_bfloat16>(m, p, grid, stream);
}

cudaError_t launch_route_mma(const RouteArgs& a, cudaStream_t stream) {
  const int n_pad = (a.N + 15) / 16 * 16;
  CUtensorMap m[7];
  if (!make_map(&m[0], a.h, a.dtype, a.d, a.T, kBM)) return cudaErrorInvalidValue;
  if (!make_map(&m[1], a.W_r, a.dtype, a.d, a.N, static_cast<uint32_t>(n_pad)))
    return cudaErrorInvalidValue;
  m[2] = m[1]; m[3] = m[0]; m[4] = m[1]; m[5] = m[1]; m[6] = m[0];
  GemmParams p{};
  p.offsets = nullptr;
  p.n_routed = 1;
  p.rows_routed = static_cast<int32_t>(a.T);
  p.rows_shared = 0;
  p.K = a.d;
  p.K_shared = a.d;
  p.n_out = n_pad;
  p.n_out_shared = 0;
  p.status = a.status;
  p.budget_ns = kWaitBudgetNs;
  p.re.b_r = a.b_r;
  p.re.sel_bias = a.sel_bias;
  p.re.logits_out = a.logits_out;
  p.re.idx = a.idx;
  p.re.gate = a.gate;
  p.re.N = a.N;
  p.re.k = a.k;
  p.re.score = a.score;
  p.re.norm = a.norm;
  // up to 128 experts: 256-token tiles, two halves sharing each W_r load
  p.row_halves = n_pad <= 128 ? 2 : 1;
  int grid = static_cast<int>((a.T + kBM * p.row_halves - 1) / (kBM * p.row_halves));
  if (grid > num_sms()) grid = num_sms();
  using bf = __nv_bfloat16;
  if (a.k <= 1) return launch_gemm<kRoute, bf, 1>(m, p, grid, stream);
  if (a.k <= 2) return launch_gemm<kRoute, bf, 2>(m, p, grid, stream);
  if (a.k <= 4) return launch_gemm<kRoute, bf, 4>(m, p, grid, stream);
  if (a.k <= 8) return launch_gemm<kRoute, bf, 8>(m, p, grid, stream);
  return launch_gemm<kRoute, bf, 16>(m, p, grid, stream);
}

cudaError_t launch_selftest_wait(int32_t* status, uint64_t budget_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 1, 0, stream>>>(status, budget_ns);
  return cudaGetLastError();
}

}  // namespace moe

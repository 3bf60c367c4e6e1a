// C-ABI layer of the fused LM-head library: argument checks, the workspace
// layout, TMA tensor maps, the chunk loop and launch-level profiling.
// Every kernel it launches is one of this library's own (rowops.cu and the
// four tcgen05 GEMM instantiations).
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "../../include/lmhead.h"
#include "internal.h"

namespace lmhead {
namespace {

constexpr int kDhMaxSplit = 4;  // most K parts of a dHidden tile (partial buffers)
static_assert(kDhMaxSplit <= 4, "the dHidden reduction sums at most four partials");
constexpr int kDhSplitFillPct = 85;  // split only when fewer worker slots than this are busy
// Raster blocks of the vocabulary projections (kFwd, kDz): 32 MB of bf16 Hc
// rows, but never fewer than 4096 rows.  The block stays in L2 (together with
// the vocabulary tiles in flight) while W streams past once per block; measured
// on the fwd + bwd step, 4096-row blocks beat 3072, 6144 and 8192 rows at
// H = 4096 and H = 5120, and 6400-row blocks beat 4096 rows at H = 2560.
constexpr int64_t kRowBlockBytes = 32ll << 20;
constexpr int64_t kRowBlockMinRows = 4096;

// Row tiles per raster block for tiles of tile_m rows and chunks of C rows
// (a block never exceeds the chunk, so block x column tiles fits an int).
int row_block_tiles(int H, int tile_m, int64_t C) {
  int64_t rows = kRowBlockBytes / (2ll * H) / tile_m * tile_m;
  if (rows < kRowBlockMinRows) rows = kRowBlockMinRows;
  if (rows > C) rows = C;
  return static_cast<int>((rows + tile_m - 1) / tile_m);
}

inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
inline int64_t cdiv(int64_t x, int64_t m) { return (x + m - 1) / m; }

// ------------------------------------------------------------ workspace
// Regions are 256-byte aligned offsets from the workspace base.
struct Layout {
  int64_t C = 0;        // rows per chunk (multiple of 256)
  int64_t num_vt = 0;   // 256-wide vocab tiles
  int64_t dz_ld = 0;    // row stride of the dZ chunk buffer (elements)
  size_t hdr = 0, counts = 0, idx = 0, yc = 0, v0 = 0, v1 = 0, v2 = 0, v3 = 0, p4 = 0, hc = 0,
         part = 0, dz = 0, dhp = 0, tflags = 0, tlist = 0, lvalid = 0, total = 0;
};

Layout make_layout(int64_t N, int H, int V, int chunk_rows) {
  Layout L;
  int64_t c = chunk_rows > 0 ? chunk_rows : LMHEAD_DEFAULT_CHUNK_ROWS;
  if (c > N) c = N;
  L.C = round_up(c < 1 ? 1 : c, 256);
  L.num_vt = cdiv(V, kBN);
  L.dz_ld = round_up(V, 8);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += static_cast<size_t>(round_up(static_cast<int64_t>(bytes), 256));
    return at;
  };
  L.hdr = take(256);
  L.counts = take(static_cast<size_t>(cdiv(N, 4096) + 1) * 4);
  // per-compact-row arrays hold up to N rounded up to 256 rows (the rows of
  // the active tiles in block-sparse mode)
  const size_t NP = static_cast<size_t>(round_up(N, 256));
  const size_t T = NP / 256;
  L.idx = take(NP * 4);
  L.yc = take(NP * 4);
  L.v0 = take(NP * 4);
  L.v1 = take(NP * 4);
  L.v2 = take(NP * 4);
  L.v3 = take(NP * 4);
  L.p4 = take(NP * 16);
  L.hc = take(static_cast<size_t>(L.C) * H * 2);
  L.part = take(static_cast<size_t>(L.num_vt) * L.C * 16);
  L.dz = take(static_cast<size_t>(L.C) * L.dz_ld * 2);
  L.dhp = take(static_cast<size_t>(kDhMaxSplit) * L.C * H * 4);
  L.tflags = take(T + 1);
  L.tlist = take((T + 1) * 4);
  L.lvalid = take(NP);
  L.total = off;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// ------------------------------------------------------------ profiling
enum Kind : int {
  kKindBuildKeep = 0, kKindCompact, kKindGatherRows, kKindGemmFwd, kKindMerge, kKindExpand,
  kKindGatherVec, kKindZeroRows, kKindGemmDz, kKindGemmDh, kKindGemmDw, kKindSlsFwd,
  kKindSlsBwd, kKindMergeShards, kKindDhReduce, kNumKinds
};
const char* kKindNames[kNumKinds] = {"build_keep", "compact",  "gather_rows", "gemm_fwd",
                                     "merge",      "expand",   "gather_vec",  "zero_rows",
                                     "gemm_dz",    "gemm_dh",  "gemm_dw",     "sls_fwd",
                                     "sls_bwd",    "merge_shards", "dh_reduce"};

std::atomic<int64_t> g_launches{0};
std::mutex g_prof_mu;
bool g_prof_on = false;
struct Rec {
  int kind;
  cudaEvent_t a, b;
};
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Brackets one kernel launch: counts it and, when profiling is on, records
// an event pair around it on the launching stream.
class Launch {
 public:
  Launch(int kind, cudaStream_t s, int nkernels = 1) : kind_(kind), s_(s) {
    g_launches.fetch_add(nkernels);
    std::lock_guard<std::mutex> g(g_prof_mu);
    if (g_prof_on) {
      a_ = take_event();
      b_ = take_event();
      cudaEventRecord(a_, s_);
    }
  }
  ~Launch() {
    std::lock_guard<std::mutex> g(g_prof_mu);
    if (a_ != nullptr) {
      cudaEventRecord(b_, s_);
      g_recs.push_back({kind_, a_, b_});
    }
  }

 private:
  int kind_;
  cudaStream_t s_;
  cudaEvent_t a_ = nullptr, b_ = nullptr;
};

// NVTX range over an entry point or a chunk (visible in Nsight timelines).
class Range {
 public:
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
};

// ------------------------------------------------------------ tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Host-side fault injection for tests: LMHEAD_FAULT names a site --
//   "tensor_map"  tensor-map encoding fails          (call returns ECUDA)
//   "launch"      the first GEMM launch is refused    (call returns ECUDA)
//   "stall"       the GEMM producer issues no loads   (device status ETIMEOUT)
// Nothing here touches the GPU in a way that can fault or hang it.
bool fault_at(const char* site) {
  const char* e = std::getenv("LMHEAD_FAULT");
  return e != nullptr && std::strcmp(e, site) == 0;
}

// 2-D tensor map over a row-major [rows, cols] matrix of bf16 (or fp32 with
// `f32`) with row stride `ld` elements; boxes of [box_rows, box_cols] with the
// 128-byte swizzle (box_cols * element size == 128).  Loads of out-of-range
// elements read zero; stores and reductions skip them.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld,
              int box_rows, int box_cols, bool f32 = false) {
  if (fault_at("tensor_map")) return false;
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const int64_t esize = f32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * esize)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------ device info
struct DevInfo {
  int sms = 0;
  bool ok = false;
};

DevInfo device_info() {
  static DevInfo cache[64];
  static bool have[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DevInfo{};
  std::lock_guard<std::mutex> g(mu);
  if (!have[dev]) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cache[dev].sms = sms;
    cache[dev].ok = (major == 10 && minor == 3);
    have[dev] = true;
  }
  return cache[dev];
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define LM_CHECK_PTRS(...)                                \
  do {                                                    \
    if (!device_ptrs_ok({__VA_ARGS__})) return LMHEAD_EINVAL; \
  } while (0)

lmhead_status cuda_status(cudaError_t e) { return e == cudaSuccess ? LMHEAD_OK : LMHEAD_ECUDA; }

// Clears the status word and the timeout record of the workspace header
// (status[0] and status[3]; Nk and the tile count in between are rewritten
// by every call that reads them).
cudaError_t clear_status(int* status, cudaStream_t s) {
  return cudaMemsetAsync(status, 0, 4 * sizeof(int), s);
}

#define LM_TRY(expr)                                  \
  do {                                                \
    cudaError_t e_ = (expr);                          \
    if (e_ != cudaSuccess) return LMHEAD_ECUDA;       \
  } while (0)

lmhead_status check_sizes(int64_t N, int H, int V) {
  if (N < 0 || N > (int64_t{1} << 31) - 1024) return LMHEAD_EINVAL;
  if (H < 8 || (H % 8) != 0 || V < 1) return LMHEAD_EINVAL;
  return LMHEAD_OK;
}

lmhead_status check_ws(void* ws, size_t ws_bytes, const Layout& L) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return LMHEAD_EINVAL;
  if (ws_bytes < L.total) return LMHEAD_EWORKSPACE;
  return LMHEAD_OK;
}

lmhead_status run_compact(const uint8_t* keep, const int64_t* targets, int64_t N,
                          int64_t V_valid, int64_t t_offset, int32_t* idx, int32_t* yc,
                          int32_t* d_nk, int32_t* counts, int* status, cudaStream_t s) {
  if (N == 0) {
    LM_TRY(cudaMemsetAsync(d_nk, 0, sizeof(int32_t), s));
    return LMHEAD_OK;
  }
  Launch l(kKindCompact, s, 2);
  LM_TRY(launch_compact(keep, targets, N, V_valid, t_offset, idx, yc, d_nk, counts, status, s));
  return LMHEAD_OK;
}

int gemm_grid(int64_t tiles) {
  const int sms = device_info().sms;
  return static_cast<int>(tiles < sms ? (tiles < 1 ? 1 : tiles) : sms);
}

// GEMM variant of one contraction.  By default the projections (kFwd, kDz)
// run on CTA pairs with 256 x 256 tiles and double-buffered accumulators
// (K = H is short and their epilogue (an exponential per logit) is long, so
// it must hide behind the MMAs of the next tile), and dHidden and dW on CTA
// pairs with 256 x 512 tiles (K = V, K = the chunk's rows: one 512-column
// accumulator released in halves, a quarter fewer operand bytes per FLOP) when
// H spans an even number of 256-column tiles (H = 2560, 4096, 5120, ...).
// Measured on the fwd + bwd step under the power cap (same-box A/B): the
// half-kept 64K-token step 95.3 ms against 95.6 (dHidden alone on wide
// tiles) and 96.8 (all on 256 x 256), long context 259.5 / 264.7 / 272.4 ms;
// the projections on wide tiles lose 7% each.
//   LMHEAD_GEMM = "single" (one-CTA kernel, 128 x 256 tiles), "pair" or
//     "wide" puts every contraction on one variant;
//   LMHEAD_WIDE = a comma-separated subset of "fwd,dz,dh,dw" replaces the
//     default set of contractions on 512-column tiles (when LMHEAD_GEMM is
//     unset; "none" for the empty set).
enum class GemmVariant { kSingle, kPair, kWide };

bool listed(const char* list, const char* name) {
  const size_t n = std::strlen(name);
  for (const char* p = list; *p != 0;) {
    const char* e = std::strchr(p, ',');
    const size_t len = e != nullptr ? static_cast<size_t>(e - p) : std::strlen(p);
    if (len == n && std::strncmp(p, name, n) == 0) return true;
    if (e == nullptr) break;
    p = e + 1;
  }
  return false;
}

GemmVariant gemm_variant(int mode, int H) {
  const char* e = std::getenv("LMHEAD_GEMM");
  if (e != nullptr && std::strcmp(e, "single") == 0) return GemmVariant::kSingle;
  if (e != nullptr && std::strcmp(e, "pair") == 0) return GemmVariant::kPair;
  if (e != nullptr && std::strcmp(e, "wide") == 0) return GemmVariant::kWide;
  static const char* kNames[4] = {"fwd", "dz", "dh", "dw"};
  const char* w = std::getenv("LMHEAD_WIDE");
  if (w != nullptr) return listed(w, kNames[mode]) ? GemmVariant::kWide : GemmVariant::kPair;
  // dHidden and dW tile the H columns: with an odd number of 256-column tiles
  // the last 512-column tile would spend half its MMAs on columns past H
  const bool h_even = cdiv(H, kBN) % 2 == 0;
  return (mode == kDh || mode == kDw) && h_even ? GemmVariant::kWide : GemmVariant::kPair;
}

// Rows and columns of one tile of the selected variant.
inline int tile_rows(GemmVariant v) { return v == GemmVariant::kSingle ? kBM : 256; }
inline int tile_cols(GemmVariant v) { return v == GemmVariant::kWide ? 2 * kBN : kBN; }

// Most K parts of a dHidden tail tile (work_schedule): LMHEAD_DH_SPLIT =
// 1 .. 4 (default 4; 1 never splits).
int dh_max_split() {
  const char* e = std::getenv("LMHEAD_DH_SPLIT");
  if (e == nullptr) return kDhMaxSplit;
  const int v = std::atoi(e);
  return v < 1 ? 1 : (v > kDhMaxSplit ? kDhMaxSplit : v);
}

// Launches one contraction on the selected variant.  m_upper bounds the rows
// of D (the chunk for kFwd/kDz/kDh, V for kDw); b_single / b_pair are the B
// maps for the one-CTA and CTA-pair variants (they differ only for K-major
// B); c is the output map of kDz / kDw (the other contractions do not read
// it).  *workers receives the number of persistent workers launched (CTA
// pairs or CTAs), which the dHidden schedule depends on.
template <int MODE>
cudaError_t run_gemm(GemmVariant v, const CUtensorMap& a, const CUtensorMap& b_single,
                     const CUtensorMap& b_pair, const CUtensorMap& c, const TcGemmParams& p,
                     int64_t m_upper, int64_t n, cudaStream_t s, int* workers = nullptr) {
  if (fault_at("launch")) return cudaErrorLaunchFailure;
  const int share = MODE == kDh ? p.max_split : 1;  // K parts a dHidden tile may be cut into
  if (v == GemmVariant::kPair || v == GemmVariant::kWide) {
    const int64_t tiles = cdiv(m_upper, 256) * cdiv(n, tile_cols(v)) * share;
    const int64_t pairs = device_info().sms / 2;
    const int64_t w = tiles < pairs ? (tiles < 1 ? 1 : tiles) : pairs;
    if (workers != nullptr) *workers = static_cast<int>(w);
    return v == GemmVariant::kWide
               ? launch_tc_gemm_pair<MODE, 2>(a, b_pair, c, p, static_cast<int>(2 * w), s)
               : launch_tc_gemm_pair<MODE, 1>(a, b_pair, c, p, static_cast<int>(2 * w), s);
  }
  const int grid = gemm_grid(cdiv(m_upper, kBM) * cdiv(n, kBN) * share);
  if (workers != nullptr) *workers = grid;
  return launch_tc_gemm<MODE>(a, b_single, c, p, grid, s);
}

// Forward over the vocabulary rows held in `weight` ([V, H]).  For the whole
// vocabulary (partial == nullptr) it writes logprob / entropy / lse; for a
// shard starting at vocabulary row t_offset it writes the shard's per-row
// (m, s, u, t) partials instead.  Targets are checked against [0, V_valid).
lmhead_status fwd_impl(const void* hidden, const void* weight, const int64_t* targets,
                       const uint8_t* keep, int64_t N, int H, int V, int want_entropy,
                       float* logprob, float* entropy, float* lse, float4* partial,
                       int64_t t_offset, int64_t V_valid, int chunk_rows, void* workspace,
                       size_t ws_bytes, lmhead_stream_t stream, bool blocksparse = false) {
  lmhead_status st = check_sizes(N, H, V);
  if (st != LMHEAD_OK) return st;
  if (hidden == nullptr || weight == nullptr || targets == nullptr)
    return LMHEAD_EINVAL;
  if (partial == nullptr &&
      (logprob == nullptr || lse == nullptr || (want_entropy && entropy == nullptr)))
    return LMHEAD_EINVAL;
  if (!aligned16(hidden) || !aligned16(weight)) return LMHEAD_EINVAL;
  const Layout L = make_layout(N, H, V, chunk_rows);
  st = check_ws(workspace, ws_bytes, L);
  if (st != LMHEAD_OK) return st;
  if (N == 0) return LMHEAD_OK;
  if (!device_info().ok) return LMHEAD_EUNSUPPORTED;
  LM_CHECK_PTRS(hidden, weight, targets, keep, logprob, entropy, lse, partial, workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Range range("lmhead_fwd");

  int* status = at<int>(workspace, L.hdr);
  int32_t* d_nk = status + 1;
  int32_t* idx = at<int32_t>(workspace, L.idx);
  int32_t* yc = at<int32_t>(workspace, L.yc);
  float* lp_c = at<float>(workspace, L.v0);
  float* ent_c = at<float>(workspace, L.v1);
  float* lse_c = at<float>(workspace, L.v2);
  float4* raw_c = partial != nullptr ? at<float4>(workspace, L.p4) : nullptr;
  __nv_bfloat16* hc = at<__nv_bfloat16>(workspace, L.hc);
  float4* part = at<float4>(workspace, L.part);

  LM_TRY(clear_status(status, s));
  uint8_t* lvalid = blocksparse ? at<uint8_t>(workspace, L.lvalid) : nullptr;
  int32_t* tile_list = at<int32_t>(workspace, L.tlist);
  if (blocksparse) {
    Launch l(kKindCompact, s, 4);
    LM_TRY(launch_tile_scan(keep, targets, N, V_valid, t_offset, at<uint8_t>(workspace, L.tflags),
                            tile_list, status + 2, at<int32_t>(workspace, L.counts), idx, yc,
                            lvalid, d_nk, status, s));
    st = LMHEAD_OK;
  } else {
    st = run_compact(keep, targets, N, V_valid, t_offset, idx, yc, d_nk,
                     at<int32_t>(workspace, L.counts), status, s);
  }
  if (st != LMHEAD_OK) return st;

  const GemmVariant gv = gemm_variant(kFwd, H);
  CUtensorMap ma, mb, mb2;
  if (!(blocksparse ? make_map(&ma, hidden, N, H, H, kBM, 64)
                    : make_map(&ma, hc, L.C, H, H, kBM, 64)) ||
      !make_map(&mb, weight, V, H, H, kBN, 64) ||
      !make_map(&mb2, weight, V, H, H, 128, 64))
    return LMHEAD_ECUDA;

  TcGemmParams p{};
  p.d_nk = d_nk;
  p.chunk_rows = static_cast<int>(L.C);
  p.V = V;
  p.H = H;
  p.n_rows = N;
  p.group_m = row_block_tiles(H, tile_rows(gv), L.C);
  p.group_n = 16;
  p.status = status;
  p.stall = fault_at("stall") ? 1 : 0;
  p.tile_list = blocksparse ? tile_list : nullptr;
  p.lvalid = lvalid;
  p.targets_c = yc;
  p.want_entropy = want_entropy ? 1 : 0;
  p.part = part;

  const int64_t max_chunks = cdiv(N, L.C);
  for (int64_t c = 0; c < max_chunks; ++c) {
    Range chunk_range("chunk");
    if (!blocksparse) {
      Launch l(kKindGatherRows, s);
      LM_TRY(launch_gather_rows(static_cast<const __nv_bfloat16*>(hidden), idx, d_nk,
                                static_cast<int>(c), static_cast<int>(L.C), H, hc, N, status,
                                s));
    }
    p.chunk_index = static_cast<int>(c);
    {
      Launch l(kKindGemmFwd, s);
      LM_TRY(run_gemm<kFwd>(gv, ma, mb, mb2, ma, p, L.C, V, s));
    }
    {
      Launch l(kKindMerge, s);
      LM_TRY(launch_merge(part, static_cast<int>(L.num_vt), d_nk, static_cast<int>(c),
                          static_cast<int>(L.C), p.want_entropy, lp_c, ent_c, lse_c, raw_c, s));
    }
  }
  {
    Launch l(kKindExpand, s);
    if (partial != nullptr) {
      LM_TRY(launch_expand4(keep, idx, d_nk, N, raw_c, partial, status, s));
    } else {
      LM_TRY(launch_expand3(keep, idx, d_nk, N, lp_c, want_entropy ? ent_c : nullptr, lse_c,
                            logprob, want_entropy ? entropy : nullptr, lse, lvalid, status,
                            s));
    }
  }
  return LMHEAD_OK;
}

// Backward over the vocabulary rows held in `weight` ([V, H], starting at
// vocabulary row t_offset; lse and entropy are the whole vocabulary's).
// dhidden receives this shard's dZ W (the whole hidden gradient when the shard
// is the whole vocabulary); dweight is the shard's [V, H] gradient.
lmhead_status bwd_impl(const void* hidden, const void* weight, const int64_t* targets,
                       const uint8_t* keep, int64_t N, int H, int V, int64_t t_offset,
                       int64_t V_valid, const float* lse, const float* entropy,
                       const float* grad_logprob, const float* grad_entropy, void* dhidden,
                       float* dweight, int dw_accumulate, int chunk_rows, void* workspace,
                       size_t ws_bytes, lmhead_stream_t stream, bool blocksparse = false) {
  lmhead_status st = check_sizes(N, H, V);
  if (st != LMHEAD_OK) return st;
  if (hidden == nullptr || weight == nullptr || targets == nullptr || lse == nullptr ||
      grad_logprob == nullptr || dhidden == nullptr || dweight == nullptr ||
      (grad_entropy != nullptr && entropy == nullptr))
    return LMHEAD_EINVAL;
  if (!aligned16(hidden) || !aligned16(weight) || !aligned16(dhidden) || !aligned16(dweight))
    return LMHEAD_EINVAL;
  const Layout L = make_layout(N, H, V, chunk_rows);
  st = check_ws(workspace, ws_bytes, L);
  if (st != LMHEAD_OK) return st;
  if (!device_info().ok) return LMHEAD_EUNSUPPORTED;
  LM_CHECK_PTRS(hidden, weight, targets, keep, lse, entropy, grad_logprob, grad_entropy, dhidden,
                dweight, workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Range range("lmhead_bwd");
  if (N == 0) {
    if (!dw_accumulate)
      LM_TRY(cudaMemsetAsync(dweight, 0, static_cast<size_t>(V) * H * sizeof(float), s));
    return LMHEAD_OK;
  }

  int* status = at<int>(workspace, L.hdr);
  int32_t* d_nk = status + 1;
  int32_t* idx = at<int32_t>(workspace, L.idx);
  int32_t* yc = at<int32_t>(workspace, L.yc);
  float* lse_c = at<float>(workspace, L.v0);
  float* ent_c = at<float>(workspace, L.v1);
  float* glp_c = at<float>(workspace, L.v2);
  float* gent_c = at<float>(workspace, L.v3);
  __nv_bfloat16* hc = at<__nv_bfloat16>(workspace, L.hc);
  __nv_bfloat16* dz = at<__nv_bfloat16>(workspace, L.dz);

  LM_TRY(clear_status(status, s));
  uint8_t* lvalid = blocksparse ? at<uint8_t>(workspace, L.lvalid) : nullptr;
  int32_t* tile_list = at<int32_t>(workspace, L.tlist);
  if (blocksparse) {
    Launch l(kKindCompact, s, 4);
    LM_TRY(launch_tile_scan(keep, targets, N, V_valid, t_offset, at<uint8_t>(workspace, L.tflags),
                            tile_list, status + 2, at<int32_t>(workspace, L.counts), idx, yc,
                            lvalid, d_nk, status, s));
    st = LMHEAD_OK;
  } else {
    st = run_compact(keep, targets, N, V_valid, t_offset, idx, yc, d_nk,
                     at<int32_t>(workspace, L.counts), status, s);
  }
  if (st != LMHEAD_OK) return st;
  {
    Launch l(kKindGatherVec, s);
    LM_TRY(launch_gather_vec(idx, d_nk, N, lse, grad_entropy ? entropy : nullptr, grad_logprob,
                             grad_entropy, lse_c, ent_c, glp_c, gent_c, status, s));
  }
  if (keep != nullptr) {
    Launch l(kKindZeroRows, s);
    LM_TRY(launch_zero_skipped_rows(keep, N, H, static_cast<__nv_bfloat16*>(dhidden), s));
  }

  const GemmVariant gv_dz = gemm_variant(kDz, H);
  const GemmVariant gv_dh = gemm_variant(kDh, H);
  const GemmVariant gv_dw = gemm_variant(kDw, H);
  CUtensorMap m_hc_k, m_w_k, m_w_k2, m_dz_k, m_w_mn, m_dz_mn, m_hc_mn, m_dz_out, m_dw_out;
  const void* rows_src = blocksparse ? hidden : static_cast<const void*>(hc);
  const int64_t rows_n = blocksparse ? N : L.C;
  if (!make_map(&m_hc_k, rows_src, rows_n, H, H, kBM, 64) ||  // A of kDz (K-major)
      !make_map(&m_w_k, weight, V, H, H, kBN, 64) ||       // B of kDz (K-major)
      !make_map(&m_w_k2, weight, V, H, H, 128, 64) ||      // B of kDz, CTA pairs
      !make_map(&m_dz_k, dz, L.C, V, L.dz_ld, kBM, 64) ||  // A of kDh (K-major)
      !make_map(&m_w_mn, weight, V, H, H, 64, 64) ||       // B of kDh (MN-major boxes)
      !make_map(&m_dz_mn, dz, L.C, V, L.dz_ld, 64, 64) ||  // A of kDw (MN-major boxes)
      !make_map(&m_hc_mn, rows_src, rows_n, H, H, 64, 64) ||  // B of kDw (MN-major boxes)
      !make_map(&m_dz_out, dz, L.C, V, L.dz_ld, 32, 64) ||   // output of kDz
      !make_map(&m_dw_out, dweight, V, H, H, 32, 32, true))   // output of kDw (fp32)
    return LMHEAD_ECUDA;

  TcGemmParams p{};
  p.d_nk = d_nk;
  p.chunk_rows = static_cast<int>(L.C);
  p.V = V;
  p.H = H;
  p.n_rows = N;
  p.status = status;
  p.stall = fault_at("stall") ? 1 : 0;
  p.targets_c = yc;
  p.idx = idx;
  p.tile_list = blocksparse ? tile_list : nullptr;
  p.lvalid = lvalid;
  p.lse_c = lse_c;
  p.ent_c = ent_c;
  p.glp_c = glp_c;
  p.gent_c = grad_entropy ? gent_c : nullptr;
  p.want_entropy = grad_entropy ? 1 : 0;
  p.dhidden = static_cast<__nv_bfloat16*>(dhidden);
  p.dh_part = at<float>(workspace, L.dhp);
  p.max_split = dh_max_split();
  p.split_fill_pct = kDhSplitFillPct;
  int dh_workers = 0;

  const int64_t max_chunks = cdiv(N, L.C);
  for (int64_t c = 0; c < max_chunks; ++c) {
    Range chunk_range("chunk");
    p.chunk_index = static_cast<int>(c);
    if (!blocksparse) {
      Launch l(kKindGatherRows, s);
      LM_TRY(launch_gather_rows(static_cast<const __nv_bfloat16*>(hidden), idx, d_nk,
                                static_cast<int>(c), static_cast<int>(L.C), H, hc, N, status,
                                s));
    }
    {
      Launch l(kKindGemmDz, s);
      p.group_m = row_block_tiles(H, tile_rows(gv_dz), L.C);
      p.group_n = 16;
      LM_TRY(run_gemm<kDz>(gv_dz, m_hc_k, m_w_k, m_w_k2, m_dz_out, p, L.C, V, s));
    }
    {
      Launch l(kKindGemmDh, s);
      p.group_m = 0;
      p.group_n = static_cast<int>(cdiv(H, tile_cols(gv_dh)));  // all column tiles per row tile
      LM_TRY(run_gemm<kDh>(gv_dh, m_dz_k, m_w_mn, m_w_mn, m_dz_k, p, L.C, H, s, &dh_workers));
    }
    {
      Launch l(kKindDhReduce, s);
      LM_TRY(launch_dh_reduce(p.dh_part, d_nk, static_cast<int>(c), static_cast<int>(L.C), H,
                              tile_rows(gv_dh), tile_cols(gv_dh),
                              dh_workers, static_cast<int>(cdiv(V, kBK)),
                              p.max_split, p.split_fill_pct, idx, lvalid,
                              static_cast<__nv_bfloat16*>(dhidden), N, status, s));
    }
    {
      Launch l(kKindGemmDw, s);
      p.group_m = 0;
      p.group_n = static_cast<int>(cdiv(H, tile_cols(gv_dw)));  // all column tiles per row tile
      p.beta = (c > 0 || dw_accumulate) ? 1 : 0;
      LM_TRY(run_gemm<kDw>(gv_dw, m_dz_mn, m_hc_mn, m_hc_mn, m_dw_out, p, V, H, s));
    }
  }
  return LMHEAD_OK;
}

}  // namespace

int device_sm_count() { return device_info().sms; }

}  // namespace lmhead

using namespace lmhead;

extern "C" {

size_t lmhead_workspace_size(int64_t N, int H, int V, int want_entropy, int chunk_rows) {
  (void)want_entropy;
  if (N < 0 || H < 1 || V < 1) return 0;
  return make_layout(N, H, V, chunk_rows).total;
}

lmhead_status lmhead_build_keep_mask(const float* loss_mask, const float* ce_weight,
                                     const float* kl_weight, const int32_t* seq_offsets,
                                     int32_t n_seq, int64_t N, uint8_t* keep,
                                     lmhead_stream_t stream) {
  if (N < 0 || n_seq < 0 || seq_offsets == nullptr || keep == nullptr) return LMHEAD_EINVAL;
  if (N == 0) return LMHEAD_OK;
  if (!device_info().ok) return LMHEAD_EUNSUPPORTED;
  LM_CHECK_PTRS(loss_mask, ce_weight, kl_weight, seq_offsets, keep);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Launch l(kKindBuildKeep, s);
  return cuda_status(launch_build_keep(loss_mask, ce_weight, kl_weight, seq_offsets, n_seq, N,
                                       keep, s));
}

lmhead_status lmhead_compact(const uint8_t* keep, const int64_t* targets, int64_t N, int V,
                             int32_t* idx, int32_t* targets_c, int32_t* d_nk, void* workspace,
                             size_t ws_bytes, lmhead_stream_t stream) {
  if (N < 0 || V < 1 || targets == nullptr || idx == nullptr || targets_c == nullptr ||
      d_nk == nullptr)
    return LMHEAD_EINVAL;
  const Layout L = make_layout(N, 8, V, 256);
  const size_t need = L.counts + static_cast<size_t>(round_up((cdiv(N, 4096) + 1) * 4, 256));
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return LMHEAD_EINVAL;
  if (ws_bytes < need) return LMHEAD_EWORKSPACE;
  if (!device_info().ok) return LMHEAD_EUNSUPPORTED;
  LM_CHECK_PTRS(keep, targets, idx, targets_c, d_nk, workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = at<int>(workspace, L.hdr);
  LM_TRY(clear_status(status, s));
  return run_compact(keep, targets, N, V, 0, idx, targets_c, d_nk,
                     at<int32_t>(workspace, L.counts), status, s);
}

lmhead_status lmhead_fwd(const void* hidden, const void* weight, const int64_t* targets,
                         const uint8_t* keep, int64_t N, int H, int V, int want_entropy,
                         float* logprob, float* entropy, float* lse, int chunk_rows,
                         void* workspace, size_t ws_bytes, lmhead_stream_t stream) {
  return fwd_impl(hidden, weight, targets, keep, N, H, V, want_entropy, logprob, entropy, lse,
                  nullptr, 0, V, chunk_rows, workspace, ws_bytes, stream);
}

lmhead_status lmhead_bwd(const void* hidden, const void* weight, const int64_t* targets,
                         const uint8_t* keep, int64_t N, int H, int V, const float* lse,
                         const float* entropy, const float* grad_logprob,
                         const float* grad_entropy, void* dhidden, float* dweight,
                         int dw_accumulate, int chunk_rows, void* workspace, size_t ws_bytes,
                         lmhead_stream_t stream) {
  return bwd_impl(hidden, weight, targets, keep, N, H, V, 0, V, lse, entropy, grad_logprob,
                  grad_entropy, dhidden, dweight, dw_accumulate, chunk_rows, workspace, ws_bytes,
                  stream);
}

lmhead_status lmhead_fwd_blocksparse(const void* hidden, const void* weight,
                                     const int64_t* targets, const uint8_t* keep, int64_t N,
                                     int H, int V, int want_entropy, float* logprob,
                                     float* entropy, float* lse, int chunk_rows, void* workspace,
                                     size_t ws_bytes, lmhead_stream_t stream) {
  return fwd_impl(hidden, weight, targets, keep, N, H, V, want_entropy, logprob, entropy, lse,
                  nullptr, 0, V, chunk_rows, workspace, ws_bytes, stream, true);
}

lmhead_status lmhead_bwd_blocksparse(const void* hidden, const void* weight,
                                     const int64_t* targets, const uint8_t* keep, int64_t N,
                                     int H, int V, const float* lse, const float* entropy,
                                     const float* grad_logprob, const float* grad_entropy,
                                     void* dhidden, float* dweight, int dw_accumulate,
                                     int chunk_rows, void* workspace, size_t ws_bytes,
                                     lmhead_stream_t stream) {
  return bwd_impl(hidden, weight, targets, keep, N, H, V, 0, V, lse, entropy, grad_logprob,
                  grad_entropy, dhidden, dweight, dw_accumulate, chunk_rows, workspace, ws_bytes,
                  stream, true);
}

lmhead_status lmhead_fwd_shard(const void* hidden, const void* weight_shard,
                               const int64_t* targets, const uint8_t* keep, int64_t N, int H,
                               int V_shard, int64_t v_begin, int64_t V_total, int want_entropy,
                               float* partials, int chunk_rows, void* workspace,
                               size_t ws_bytes, lmhead_stream_t stream) {
  if (partials == nullptr || v_begin < 0 || V_shard < 1 || v_begin + V_shard > V_total)
    return LMHEAD_EINVAL;
  if ((reinterpret_cast<uintptr_t>(partials) & 15u) != 0) return LMHEAD_EINVAL;
  return fwd_impl(hidden, weight_shard, targets, keep, N, H, V_shard, want_entropy, nullptr,
                  nullptr, nullptr, reinterpret_cast<float4*>(partials), v_begin, V_total,
                  chunk_rows, workspace, ws_bytes, stream);
}

lmhead_status lmhead_merge_shards(const float* partials, int num_shards, const uint8_t* keep,
                                  int64_t N, int want_entropy, float* logprob, float* entropy,
                                  float* lse, lmhead_stream_t stream) {
  if (N < 0 || num_shards < 1 || partials == nullptr || logprob == nullptr || lse == nullptr ||
      (want_entropy && entropy == nullptr) || (reinterpret_cast<uintptr_t>(partials) & 15u) != 0)
    return LMHEAD_EINVAL;
  if (N == 0) return LMHEAD_OK;
  if (!device_info().ok) return LMHEAD_EUNSUPPORTED;
  LM_CHECK_PTRS(partials, keep, logprob, entropy, lse);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Launch l(kKindMergeShards, s);
  return cuda_status(launch_merge_shards(reinterpret_cast<const float4*>(partials), num_shards,
                                         keep, N, want_entropy ? 1 : 0, logprob,
                                         want_entropy ? entropy : nullptr, lse, s));
}

lmhead_status lmhead_bwd_shard(const void* hidden, const void* weight_shard,
                               const int64_t* targets, const uint8_t* keep, int64_t N, int H,
                               int V_shard, int64_t v_begin, int64_t V_total, const float* lse,
                               const float* entropy, const float* grad_logprob,
                               const float* grad_entropy, void* dhidden_partial,
                               float* dweight_shard, int dw_accumulate, int chunk_rows,
                               void* workspace, size_t ws_bytes, lmhead_stream_t stream) {
  if (v_begin < 0 || V_shard < 1 || v_begin + V_shard > V_total) return LMHEAD_EINVAL;
  return bwd_impl(hidden, weight_shard, targets, keep, N, H, V_shard, v_begin, V_total, lse,
                  entropy, grad_logprob, grad_entropy, dhidden_partial, dweight_shard,
                  dw_accumulate, chunk_rows, workspace, ws_bytes, stream);
}

lmhead_status lmhead_expand(const float* src, const int32_t* idx, const int32_t* d_nk, int64_t N,
                            float* dst, int32_t* d_status, lmhead_stream_t stream) {
  if (N < 0 || src == nullptr || idx == nullptr || d_nk == nullptr || dst == nullptr)
    return LMHEAD_EINVAL;
  if (N == 0) return LMHEAD_OK;
  if (!device_info().ok) return LMHEAD_EUNSUPPORTED;
  LM_CHECK_PTRS(src, idx, d_nk, dst, d_status);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Launch l(kKindExpand, s);
  return cuda_status(launch_expand(src, idx, d_nk, N, dst, d_status, s));
}

lmhead_status lmhead_selective_log_softmax_fwd(const void* logits, int logits_dtype, int64_t ld,
                                               const int64_t* targets, const uint8_t* keep,
                                               int64_t N, int V, int want_entropy,
                                               float* logprob, float* entropy, float* lse,
                                               int32_t* d_status, lmhead_stream_t stream) {
  if (N < 0 || N > 2147483647LL || V < 1 || ld < V || (logits_dtype != 0 && logits_dtype != 1))
    return LMHEAD_EINVAL;
  if (logits == nullptr || targets == nullptr || logprob == nullptr || lse == nullptr ||
      (want_entropy && entropy == nullptr))
    return LMHEAD_EINVAL;
  if (N == 0) return LMHEAD_OK;
  if (!device_info().ok) return LMHEAD_EUNSUPPORTED;
  LM_CHECK_PTRS(logits, targets, keep, logprob, entropy, lse, d_status);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Range range("lmhead_selective_log_softmax_fwd");
  Launch l(kKindSlsFwd, s);
  return cuda_status(launch_sls_fwd(logits, logits_dtype, ld, targets, keep, N, V,
                                    want_entropy ? 1 : 0, logprob, want_entropy ? entropy : nullptr,
                                    lse, d_status, s));
}

lmhead_status lmhead_selective_log_softmax_bwd(const void* logits, int logits_dtype, int64_t ld,
                                               const int64_t* targets, const uint8_t* keep,
                                               int64_t N, int V, const float* lse,
                                               const float* entropy, const float* grad_logprob,
                                               const float* grad_entropy, void* dlogits,
                                               int64_t ld_out, int32_t* d_status,
                                               lmhead_stream_t stream) {
  if (N < 0 || N > 2147483647LL || V < 1 || ld < V || ld_out < V ||
      (logits_dtype != 0 && logits_dtype != 1))
    return LMHEAD_EINVAL;
  if (logits == nullptr || targets == nullptr || lse == nullptr || grad_logprob == nullptr ||
      dlogits == nullptr || (grad_entropy != nullptr && entropy == nullptr) || dlogits == logits)
    return LMHEAD_EINVAL;
  if (N == 0) return LMHEAD_OK;
  if (!device_info().ok) return LMHEAD_EUNSUPPORTED;
  LM_CHECK_PTRS(logits, targets, keep, lse, entropy, grad_logprob, grad_entropy, dlogits,
                d_status);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Range range("lmhead_selective_log_softmax_bwd");
  Launch l(kKindSlsBwd, s);
  return cuda_status(launch_sls_bwd(logits, logits_dtype, ld, targets, keep, N, V, lse, entropy,
                                    grad_logprob, grad_entropy, dlogits, ld_out, d_status, s));
}

const int32_t* lmhead_workspace_kept_rows(const void* workspace) {
  if (workspace == nullptr) return nullptr;
  return reinterpret_cast<const int32_t*>(static_cast<const char*>(workspace) + sizeof(int32_t));
}

lmhead_status lmhead_get_status(const void* workspace, lmhead_stream_t stream) {
  if (workspace == nullptr) return LMHEAD_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return LMHEAD_ECUDA;
  int h = 0;
  if (cudaMemcpy(&h, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return LMHEAD_ECUDA;
  return static_cast<lmhead_status>(h);
}

int32_t lmhead_get_timeout_record(const void* workspace, lmhead_stream_t stream) {
  if (workspace == nullptr) return -1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
  int32_t h = 0;
  if (cudaMemcpy(&h, static_cast<const int32_t*>(workspace) + 3, sizeof(int32_t),
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return -1;
  return h;
}

const char* lmhead_strerror(lmhead_status status) {
  switch (status) {
    case LMHEAD_OK: return "ok";
    case LMHEAD_EINVAL: return "invalid argument";
    case LMHEAD_EWORKSPACE: return "workspace too small";
    case LMHEAD_ETARGET: return "target outside [0, V) on a kept row";
    case LMHEAD_ECUDA: return "CUDA runtime error";
    case LMHEAD_ETIMEOUT: return "device pipeline wait timed out";
    case LMHEAD_EUNSUPPORTED: return "device is not an sm_103 GPU";
    case LMHEAD_EBOUNDS: return "an index outside its array was skipped";
  }
  return "unknown status";
}

void lmhead_profile_enable(int on) {
  std::lock_guard<std::mutex> g(g_prof_mu);
  g_prof_on = on != 0;
}

int lmhead_profile_kinds(void) { return kNumKinds; }

const char* lmhead_profile_kind_name(int kind) {
  return (kind >= 0 && kind < kNumKinds) ? kKindNames[kind] : "";
}

lmhead_status lmhead_profile_read(int64_t* launches, double* total_ms) {
  if (launches == nullptr || total_ms == nullptr) return LMHEAD_EINVAL;
  std::lock_guard<std::mutex> g(g_prof_mu);
  for (int k = 0; k < kNumKinds; ++k) {
    launches[k] = 0;
    total_ms[k] = 0.0;
  }
  lmhead_status st = LMHEAD_OK;
  for (const Rec& r : g_recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess ||
        cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
      st = LMHEAD_ECUDA;
    launches[r.kind] += 1;
    total_ms[r.kind] += ms;
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  g_recs.clear();
  return st;
}

int64_t lmhead_launch_count(void) { return g_launches.load(); }

const char* lmhead_version(void) {
#ifdef LMHEAD_DEBUG
  return "lmhead-gb300 0.1.0 (sm_103a, tcgen05, debug index checks)";
#else
  return "lmhead-gb300 0.1.0 (sm_103a, tcgen05)";
#endif
}

}  // extern "C"

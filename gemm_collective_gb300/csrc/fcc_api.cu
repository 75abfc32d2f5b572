// fcc_api.cu -- the C ABI of libfcc: argument checks, tensor maps, workspace,
// algorithm selection (fused / unfused / InterDecom / copy engine) and the
// device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cctype>
#include <chrono>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <random>
#include <string>

#include "fcc.h"
#include "fcc_internal.h"

namespace fcc {

// Device status word: kernels record the first device-side error here.
__device__ int g_status_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultTimeoutNs = 1000ull * 1000 * 1000;  // 1 s
constexpr int kGemmBN = 256;
constexpr int kMaxChunks = 64;
constexpr int kSideStreams = 4;

std::atomic<uint64_t> g_launches{0};
std::mutex g_mu;

struct DeviceState {
  bool init = false;
  int sms = 0;
  int* status = nullptr;
  void* pool = nullptr;
  size_t pool_bytes = 0;
  void* host = nullptr;  // pinned host memory for values a call reads back
  size_t host_bytes = 0;
  cudaStream_t side[kSideStreams] = {};
  cudaEvent_t ev[kMaxChunks + kSideStreams + 2] = {};
};
DeviceState g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

fcc_status cuda_fail(cudaError_t e) { return e == cudaSuccess ? FCC_OK : FCC_ERR_CUDA; }

fcc_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FCC_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.init) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FCC_ERR_CUDA;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status_word) != cudaSuccess)
      return FCC_ERR_CUDA;
    for (int i = 0; i < kSideStreams; ++i)
      if (cudaStreamCreateWithFlags(&d.side[i], cudaStreamNonBlocking) != cudaSuccess)
        return FCC_ERR_CUDA;
    for (auto& e : d.ev)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return FCC_ERR_CUDA;
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return FCC_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.init = true;
  }
  *out = &d;
  return FCC_OK;
}

// Encoded tensor maps, keyed by everything the encoding depends on (address,
// shape, box): an encoding is a pure function of these, so a cached map is
// exactly the one a new encode would give, whatever happened to the memory in
// between.  Calls on the same buffers (every step of a training or serving
// loop) skip the driver's encode.  Direct-mapped, 1024 entries.
struct MapKey {
  const void* ptr;
  int64_t rows, cols;
  uint32_t box_rows;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && rows == o.rows && cols == o.cols && box_rows == o.box_rows;
  }
};
struct MapEntry {
  bool used = false;
  MapKey key{};
  CUtensorMap map{};
};
constexpr int kMapCache = 1024;
MapEntry g_maps[kMapCache];
std::mutex g_map_mu;

size_t map_slot(const MapKey& k) {
  uint64_t h = reinterpret_cast<uintptr_t>(k.ptr) * 0x9E3779B97F4A7C15ull;
  h ^= static_cast<uint64_t>(k.rows) * 0xC2B2AE3D27D4EB4Full;
  h ^= static_cast<uint64_t>(k.cols) * 0x165667B19E3779F9ull;
  h ^= static_cast<uint64_t>(k.box_rows) * 0x27D4EB2F165667C5ull;
  return static_cast<size_t>((h >> 32) % kMapCache);
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix, box [box_rows, 64],
// 128-byte swizzle, zero fill out of bounds.
fcc_status make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols,
                    uint32_t box_rows) {
  const MapKey key{ptr, rows, cols, box_rows};
  const size_t slot = map_slot(key);
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_maps[slot].used && g_maps[slot].key == key) {
      *m = g_maps[slot].map;
      return FCC_OK;
    }
  }
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return FCC_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_map_mu);
  g_maps[slot].used = true;
  g_maps[slot].key = key;
  g_maps[slot].map = *m;
  return FCC_OK;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool ptrs_ok(const void* const* arr, int n) {
  if (arr == nullptr) return false;
  for (int i = 0; i < n; ++i)
    if (!aligned16(arr[i])) return false;
  return true;
}

unsigned long long timeout_of(const fcc_opts* o) {
  if (o != nullptr && o->timeout_ns > 0) return static_cast<unsigned long long>(o->timeout_ns);
  const int64_t env = env_defaults().timeout_ns;
  return env > 0 ? static_cast<unsigned long long>(env) : kDefaultTimeoutNs;
}

fcc_algo algo_of(const fcc_opts* o) {
  if (o == nullptr || o->algo == FCC_ALGO_AUTO) {
    const fcc_algo env = env_defaults().algo;
    return env != FCC_ALGO_AUTO ? env : FCC_ALGO_FUSED;
  }
  return o->algo;
}

// opts->chunks, else FCC_CHUNKS, else 0 (the cost model decides).
int chunks_of(const fcc_opts* o) {
  if (o != nullptr && o->chunks > 0) return o->chunks;
  return env_defaults().chunks;
}

}  // namespace

// The strategy for FCC_ALGO_AUTO, from measurements on GB300 (8 ranks, bf16):
//  * GEMM + RS / AR and AG + GEMM: the fused kernel beat the plain GEMM +
//    reduce, the InterDecom pipeline and the copy-engine path at every shape
//    measured (8192 x 8192 x 3584: 2.10-2.31 ms against 2.47-3.41 ms), and the
//    2-rank 256 x 256 x 128 call is one launch.
//  * GEMV + AR: the fused kernel ends with one CTA per column group adding
//    the group's `splits` partials, a serial tail that grows with the splits:
//    with 9 splits (N = 8192, K = 3584) fused 81.7 us against 83.0 us for the
//    plain per-rank GEMM + reduce kernel; with 19 splits (N = 4096) 54.8 us
//    against 45.5 us.  So the plain form is chosen from 16 splits on.
fcc_algo choose_algo(fcc_op op, int R, int64_t M, int64_t N, int64_t K, int sms, int max_ctas) {
  (void)M;
  // FCC_ALGO in the environment replaces the rule below.
  if (env_defaults().algo != FCC_ALGO_AUTO) return env_defaults().algo;
  if (op == FCC_OP_GEMV_AR) {
    int groups = 0, splits = 0;
    gemv_shape(N, R, K, sms, max_ctas, &groups, &splits);
    return splits >= 16 ? FCC_ALGO_UNFUSED : FCC_ALGO_FUSED;
  }
  //  * Embedding + All-to-All: the fused kernel (each pooled row stored
  //    straight into its sample's rank).  With eight rows in flight a warp it
  //    took 1133-1140 us at 8 ranks x 64 tables of 65536 x 128, 2048 samples
  //    a rank, bags of 32, against 1304-1308 us for pooling into a staging
  //    buffer and the exchange kernel (two boxes).  (With four rows in
  //    flight the two forms were within the box-to-box spread, and the
  //    staged one was kept.)
  return FCC_ALGO_FUSED;
}

namespace {

bool deterministic_of(const fcc_opts* o) {
  if (o != nullptr) return o->deterministic != 0;
  return env_defaults().deterministic != 0;  // (-1, unset: deterministic)
}

// Tensor-core tile shape (CTAs per cluster): a CTA pair per 256-row tile
// unless the rows are few (one CTA per 128-row tile), or the caller's shape.
// Automatic tile shape: CTA pairs (256 x 256 tiles) when the rows exceed 128
// and the 128 x 256 single-CTA tiles would not all fit in one round on the
// CTAs available (`ctas`).  At one round or less every CTA runs one tile
// either way, and the single CTAs skip the pair's cluster launch and
// handshakes: 5.8 against 7.3 us for the 2-rank 256 x 256 x 128 reduce-scatter.
int choose_cg(const fcc_opts* o, int64_t rows, int64_t single_tiles, int ctas) {
  if (o != nullptr && (o->cta_pair == 1 || o->cta_pair == 2)) return o->cta_pair;
  return (rows > kBM && single_tiles > ctas) ? 2 : 1;
}

// opts->cta_pair: 0 (automatic), 1 or 2.
bool tile_shape_ok(const fcc_opts* o) {
  return o == nullptr || o->cta_pair == 0 || o->cta_pair == 1 || o->cta_pair == 2;
}

int grid_for(const DeviceState* d, const fcc_opts* o, int64_t units) {
  int g = d->sms;
  if (o != nullptr && o->max_ctas > 0) g = std::min(g, o->max_ctas);
  if (units < g) g = static_cast<int>(std::max<int64_t>(units, 1));
  return g;
}

size_t align_up(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace: the caller's, else the internal pool (grown with cudaMalloc).
fcc_status get_workspace(DeviceState* d, const fcc_opts* o, size_t bytes, void** out) {
  *out = nullptr;
  if (bytes == 0) return FCC_OK;
  if (o != nullptr && o->workspace != nullptr) {
    if (o->workspace_bytes < bytes || !aligned16(o->workspace)) return FCC_ERR_WORKSPACE;
    *out = o->workspace;
    return FCC_OK;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (d->pool_bytes < bytes) {
    if (d->pool != nullptr) {
      if (cudaFree(d->pool) != cudaSuccess) return FCC_ERR_CUDA;
      d->pool = nullptr;
      d->pool_bytes = 0;
    }
    if (cudaMalloc(&d->pool, bytes) != cudaSuccess) return FCC_ERR_CUDA;
    d->pool_bytes = bytes;
  }
  *out = d->pool;
  return FCC_OK;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Common GEMM problem checks.  K and N must keep TMA row strides 16-byte aligned.
fcc_status check_gemm(int R, const void* const* A, const void* const* B, int64_t M, int64_t N,
                      int64_t K, fcc_dtype in) {
  if (R < 1 || R > FCC_MAX_RANKS) return FCC_ERR_INVALID;
  if (M <= 0 || N <= 0 || K <= 0) return FCC_ERR_INVALID;
  if (K % 8 != 0 || N % 8 != 0) return FCC_ERR_INVALID;
  if (M > (1ll << 31) - 1 || N > (1ll << 31) - 1 || K > (1ll << 31) - 1) return FCC_ERR_INVALID;
  if (!ptrs_ok(A, R) || !ptrs_ok(B, R)) return FCC_ERR_INVALID;
  if (in != FCC_BF16 && in != FCC_F16 && in != FCC_F32) return FCC_ERR_INVALID;
  if (in != FCC_BF16) return FCC_ERR_UNSUPPORTED;
  return FCC_OK;
}

fcc_status check_out_dtype(fcc_dtype out) {
  if (out == FCC_BF16 || out == FCC_F32) return FCC_OK;
  if (out == FCC_F16) return FCC_ERR_UNSUPPORTED;
  return FCC_ERR_INVALID;
}

// Fills the GEMM parameters shared by all modes.
fcc_status gemm_params(GemmParams& p, DeviceState* d, int mode, int R, const void* const* A,
                       const void* const* B, void* const* out, int nout, int64_t M, int64_t N,
                       int64_t K, int64_t Ms, int64_t m_begin, int64_t m_end, int out_f32,
                       const fcc_opts* o) {
  std::memset(&p, 0, sizeof(p));
  const int64_t a_rows = (mode == MODE_AG) ? Ms : M;
  for (int r = 0; r < R; ++r) {
    fcc_status s = make_map(&p.mapA[r], A[r], a_rows, K, kBM);
    if (s != FCC_OK) return s;
    s = make_map(&p.mapB[r], B[r], K, N, kBK);
    if (s != FCC_OK) return s;
  }
  for (int i = 0; i < nout; ++i) p.out[i] = out[i];
  p.R = R;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.Ms = static_cast<int>(Ms);
  p.m_begin = static_cast<int>(m_begin);
  p.m_end = static_cast<int>(m_end);
  p.kb_per_rank = static_cast<int>(cdiv(K, kBK));
  p.out_f32 = out_f32;
  // Raster groups of 8 m-tiles (the ordered RS / AR: 2.007 against 2.052 ms
  // with 16 and 2.162 with 32 at the 8-rank workload; the AllGather sets 8
  // below as well).
  p.group_m = 8;
  p.status = d->status;
  p.timeout_ns = timeout_of(o);
  p.phase_ns = o != nullptr ? reinterpret_cast<unsigned long long*>(o->phase_ns) : nullptr;
  const int tn = static_cast<int>(cdiv(N, kGemmBN));
  const int64_t rows = (mode == MODE_AG) ? Ms : (mode == MODE_PARTIAL ? m_end - m_begin : M);
  // 128-row tiles of the launch (as the switch below counts them for p.cg = 1)
  int64_t single_tiles = cdiv(rows, kBM) * tn;
  if (mode == MODE_PARTIAL || mode == MODE_RS_PUSH || mode == MODE_AR_PUSH) single_tiles *= R;
  if (mode == MODE_AG) single_tiles *= static_cast<int64_t>(R) * R;
  p.cg = choose_cg(o, rows, single_tiles, grid_for(d, o, INT64_MAX));
  const int64_t tm = static_cast<int64_t>(kBM) * p.cg;
  switch (mode) {
    case MODE_RS:
    case MODE_AR:
      p.tiles_m = static_cast<int>(cdiv(M, tm));
      p.tiles_n = tn;
      p.num_tiles = p.tiles_m * p.tiles_n;
      p.k_iters = R * p.kb_per_rank;
      break;
    case MODE_RS_PUSH:
    case MODE_AR_PUSH:
      p.tiles_m = static_cast<int>(cdiv(M, tm));
      p.tiles_n = tn;
      p.num_tiles = R * p.tiles_m * p.tiles_n;
      p.k_iters = p.kb_per_rank;
      break;
    case MODE_PARTIAL:
      p.tiles_m = static_cast<int>(cdiv(m_end - m_begin, tm));
      p.tiles_n = tn;
      p.num_tiles = R * p.tiles_m * p.tiles_n;
      p.k_iters = p.kb_per_rank;
      break;
    case MODE_AG:
      p.tiles_m = R * static_cast<int>(cdiv(Ms, tm));
      p.tiles_n = R * tn;
      p.num_tiles = p.tiles_m * p.tiles_n;
      p.k_iters = p.kb_per_rank;
      break;
    default:
      return FCC_ERR_INVALID;
  }
  p.split_first = p.num_tiles;  // no half tiles unless run_gemm makes them
  return FCC_OK;
}

// Clusters (CTAs or CTA pairs) that run tiles at the same time.
int gemm_slots(const GemmParams& p, DeviceState* d, const fcc_opts* o) {
  return std::max(1, std::min(grid_for(d, o, INT64_MAX) / p.cg, gemm_max_clusters(p.cg)));
}

// Tiles of the last round that a fused deterministic RS / AR launch splits
// in K (0: none): the last round holds at most half a round, after at least
// one full round, and the K loop has two iterations or more.
int ksplit_tiles(const GemmParams& p, int slots) {
  const int rem = p.num_tiles % slots;
  return (rem > 0 && 2 * rem <= slots && p.num_tiles > slots && p.k_iters >= 2) ? rem : 0;
}

// Ids of the calls that split tiles in K: unique within the process and, by
// a random start, across processes that share a caller's workspace.
std::atomic<unsigned long long> g_call_id{0};
std::once_flag g_call_id_once;
unsigned long long next_call_id() {
  std::call_once(g_call_id_once, [] {
    std::random_device rd;
    const unsigned long long salt = (static_cast<unsigned long long>(rd()) << 32) ^ rd() ^
        static_cast<unsigned long long>(
            std::chrono::steady_clock::now().time_since_epoch().count());
    g_call_id.store(salt | 1ull);
  });
  return g_call_id.fetch_add(2);  // odd: never the zero of fresh memory
}

fcc_status run_gemm(const GemmParams& p0, int mode, DeviceState* d, const fcc_opts* o,
                    cudaStream_t st) {
  if (p0.num_tiles <= 0) return FCC_OK;
  GemmParams p = p0;
  // Tiles go round-robin over `slots` CTAs (CTA pairs).  When the last round
  // would hold at most half a round of tiles, each of those tiles runs as two
  // halves on two slots, so the round takes about half a tile's time: for a
  // fused deterministic RS / AR given split workspace (p.split_ws), K halves
  // whose partial sums meet in the epilogue (a 128-column half tile costs
  // 0.81 of a whole one on the tensor cores, a K half 0.5); otherwise
  // 128-column halves, which keep the tile's whole K loop, so the results
  // are unchanged.
  const int slots = gemm_slots(p, d, o);
  const int rem = p.num_tiles % slots;
  p.split_first = p.num_tiles;
  const int kt = (mode == MODE_RS || mode == MODE_AR) && p.split_ws != nullptr
                     ? ksplit_tiles(p, slots) : 0;
  if ((mode == MODE_RS || mode == MODE_AR || mode == MODE_AG || mode == MODE_PARTIAL) &&
      rem > 0 && 2 * rem <= slots) {
    p.split_first = p.num_tiles - rem;
    p.num_tiles += rem;
    if (kt == rem) {
      p.ksplit = 1;
      p.k_half = (p.k_iters + 1) / 2;
      p.split_flags = reinterpret_cast<unsigned long long*>(
          reinterpret_cast<char*>(p.split_ws) + ksplit_ws_bytes(kt, p.cg) -
          static_cast<size_t>(kt) * p.cg * 8);
      p.call_id = next_call_id();
    }
  }
  // Grid in CTAs: one cluster per slot, at most one per work item.
  const int grid = p.cg * static_cast<int>(std::min<int64_t>(slots, p.num_tiles));
  // Release the next launch at the start for the fused GEMMs of several
  // rounds (the 8-rank AllGather + GEMM: 2.03-2.08 ms that way against
  // 2.09-2.18 ms released late), late for the per-rank GEMMs of the baselines
  // (a reduce or gather kernel follows: the 8-rank GEMV + AllReduce baseline
  // took 91 us with the reduce resident beside its GEMM, 83 us without) and
  // for launches of one round or less (2-rank 256x256x128 RS: 5.5 against
  // 5.7 us).
  p.trigger_late = (mode == MODE_PARTIAL || p.num_tiles <= slots) ? 1 : 0;
  cudaError_t e = launch_gemm(p, mode, p.cg, grid, st);
  if (e != cudaSuccess) return FCC_ERR_CUDA;
  g_launches.fetch_add(1);
  return FCC_OK;
}

// ------------------------------------------------------------ layouts
struct RankSumPlan {
  size_t partial_bytes = 0;  // R x M x N f32
  size_t recv_bytes = 0;     // CE: R x M x N f32
  size_t acc_bytes = 0;      // push: M x N f32
  size_t ticket_bytes = 0;
  size_t total() const {
    return align_up(partial_bytes) + align_up(recv_bytes) + align_up(acc_bytes) +
           align_up(ticket_bytes);
  }
};

RankSumPlan rank_sum_plan(int R, int64_t M, int64_t N, bool out_f32, const fcc_opts* o) {
  RankSumPlan pl;
  const fcc_algo a = algo_of(o);
  const size_t mn = static_cast<size_t>(M) * static_cast<size_t>(N);
  if (a == FCC_ALGO_FUSED) {
    if (!deterministic_of(o) && !out_f32) {
      pl.acc_bytes = mn * 4;
      // one counter per (tile, CTA): enough for either tile shape
      pl.ticket_bytes = static_cast<size_t>((cdiv(M, kBM) + 1) * cdiv(N, kGemmBN)) * 4;
    }
  } else {
    pl.partial_bytes = static_cast<size_t>(R) * mn * 4;
    if (a == FCC_ALGO_CE) pl.recv_bytes = static_cast<size_t>(R) * mn * 4;
  }
  return pl;
}

// Rows per InterDecom chunk, a multiple of `align` (a tile height).
int64_t chunk_rows(int64_t M, int chunks, int64_t align = kBM) {
  int64_t rows = cdiv(M, chunks);
  return cdiv(rows, align) * align;
}

// Default model constants for the chunk count when the caller gives none:
// sustained tensor rate, copy bandwidth and per-chunk overhead on a GB300.
constexpr double kModelTcFlops = 1.6e15;
constexpr double kModelBytesPerS = 6.0e12;
constexpr double kModelAlphaS = 6.0e-6;

int model_chunks(int R, int64_t M, int64_t N, int64_t K, int out_bytes) {
  const double G = 2.0 * R * static_cast<double>(M) * N * K / kModelTcFlops;
  const double X = (static_cast<double>(R) * M * N * 4 + static_cast<double>(M) * N * out_bytes) /
                   kModelBytesPerS;
  const int maxc = static_cast<int>(std::min<int64_t>(kMaxChunks, cdiv(M, kBM)));
  return fcc_interdecom_chunks(G, X, kModelAlphaS, maxc);
}

// AllGather + GEMM: G = the R per-rank GEMMs over all M gathered rows, X = the
// gather (M x K bf16 read once and written once); chunks of 256-row tiles.
int ag_model_chunks(int R, int64_t M, int64_t N, int64_t K) {
  const double G = 2.0 * R * static_cast<double>(M) * N * K / kModelTcFlops;
  const double X = 2.0 * static_cast<double>(M) * K * 2 / kModelBytesPerS;
  const int maxc = static_cast<int>(std::min<int64_t>(kMaxChunks, cdiv(M, 2 * kBM)));
  return fcc_interdecom_chunks(G, X, kModelAlphaS, maxc);
}

// Sum over ranks (RS or AR) through partial GEMM + reduce: UNFUSED, INTERDECOM, CE.
fcc_status rank_sum_unfused(int R, const void* const* A, const void* const* B, void* const* out,
                            int nout, bool per_shard, int64_t M, int64_t N, int64_t K,
                            int out_f32, const fcc_opts* o, DeviceState* d, void* ws,
                            const RankSumPlan& pl, cudaStream_t st) {
  const fcc_algo algo = algo_of(o);
  float* P[FCC_MAX_RANKS];
  char* base = static_cast<char*>(ws);
  for (int r = 0; r < R; ++r) P[r] = reinterpret_cast<float*>(base) + static_cast<size_t>(r) * M * N;
  float* recv[FCC_MAX_RANKS];
  char* recv_base = base + align_up(pl.partial_bytes);
  for (int r = 0; r < R; ++r)
    recv[r] = reinterpret_cast<float*>(recv_base) + static_cast<size_t>(r) * M * N;
  const int64_t Ms = per_shard ? M / R : M;
  void* Pv[FCC_MAX_RANKS];
  for (int r = 0; r < R; ++r) Pv[r] = P[r];

  if (algo == FCC_ALGO_UNFUSED || algo == FCC_ALGO_CE) {
    GemmParams p;
    fcc_status s = gemm_params(p, d, MODE_PARTIAL, R, A, B, Pv, R, M, N, K, Ms, 0, M, 1, o);
    if (s != FCC_OK) return s;
    s = run_gemm(p, MODE_PARTIAL, d, o, st);
    if (s != FCC_OK) return s;
    const float* const* src = P;
    if (algo == FCC_ALGO_CE) {
      // Copy-engine movement of every partial shard to its owner (R x R copies),
      // spread over side streams; the reduction itself still needs SMs.
      cudaEvent_t fork = d->ev[kMaxChunks];
      if (cudaEventRecord(fork, st) != cudaSuccess) return FCC_ERR_CUDA;
      for (int i = 0; i < kSideStreams; ++i)
        if (cudaStreamWaitEvent(d->side[i], fork, 0) != cudaSuccess) return FCC_ERR_CUDA;
      const int64_t rows = per_shard ? Ms : M;
      const int nshards = per_shard ? R : 1;
      int q = 0;
      for (int j = 0; j < nshards; ++j) {
        for (int r = 0; r < R; ++r) {
          const size_t off = static_cast<size_t>(j) * rows * N;
          const size_t bytes = static_cast<size_t>(rows) * N * 4;
          if (cudaMemcpyAsync(recv[r] + off, P[r] + off, bytes, cudaMemcpyDeviceToDevice,
                              d->side[q % kSideStreams]) != cudaSuccess)
            return FCC_ERR_CUDA;
          ++q;
        }
      }
      for (int i = 0; i < kSideStreams; ++i) {
        if (cudaEventRecord(d->ev[kMaxChunks + 1 + i], d->side[i]) != cudaSuccess) return FCC_ERR_CUDA;
        if (cudaStreamWaitEvent(st, d->ev[kMaxChunks + 1 + i], 0) != cudaSuccess) return FCC_ERR_CUDA;
      }
      src = recv;
    }
    if (cuda_fail(launch_reduce_shards(src, R, out, nout, per_shard ? 1 : 0, M, N, Ms, 0, M,
                                       out_f32, st)) != FCC_OK)
      return FCC_ERR_CUDA;
    return FCC_OK;
  }

  // INTERDECOM: GEMM of row chunk i on the caller stream overlaps the reduce
  // of chunk i-1 on a side stream.
  int chunks = chunks_of(o) > 0 ? chunks_of(o) : model_chunks(R, M, N, K, out_f32 ? 4 : 2);
  chunks = std::max(1, std::min(chunks, kMaxChunks));
  const int64_t rows = chunk_rows(M, chunks);
  cudaStream_t side = d->side[0];
  int i = 0;
  for (int64_t m0 = 0; m0 < M; m0 += rows, ++i) {
    const int64_t m1 = std::min(M, m0 + rows);
    GemmParams p;
    fcc_status s = gemm_params(p, d, MODE_PARTIAL, R, A, B, Pv, R, M, N, K, Ms, m0, m1, 1, o);
    if (s != FCC_OK) return s;
    s = run_gemm(p, MODE_PARTIAL, d, o, st);
    if (s != FCC_OK) return s;
    if (cudaEventRecord(d->ev[i], st) != cudaSuccess) return FCC_ERR_CUDA;
    if (cudaStreamWaitEvent(side, d->ev[i], 0) != cudaSuccess) return FCC_ERR_CUDA;
    if (cuda_fail(launch_reduce_shards(P, R, out, nout, per_shard ? 1 : 0, M, N, Ms, m0, m1,
                                       out_f32, side)) != FCC_OK)
      return FCC_ERR_CUDA;
  }
  cudaEvent_t join = d->ev[kMaxChunks + kSideStreams + 1];
  if (cudaEventRecord(join, side) != cudaSuccess) return FCC_ERR_CUDA;
  if (cudaStreamWaitEvent(st, join, 0) != cudaSuccess) return FCC_ERR_CUDA;
  return FCC_OK;
}

fcc_status rank_sum_call(int R, const void* const* A, const void* const* B, void* const* out,
                         bool per_shard, int64_t M, int64_t N, int64_t K, fcc_dtype in,
                         fcc_dtype out_dtype, const fcc_opts* o, cudaStream_t st) {
  fcc_status s = check_gemm(R, A, B, M, N, K, in);
  if (s != FCC_OK) return s;
  if (per_shard && M % R != 0) return FCC_ERR_INVALID;
  if ((s = check_out_dtype(out_dtype)) != FCC_OK) return s;
  if (!ptrs_ok(out, R)) return FCC_ERR_INVALID;
  const fcc_algo algo = algo_of(o);
  if (algo != FCC_ALGO_FUSED && algo != FCC_ALGO_UNFUSED && algo != FCC_ALGO_INTERDECOM &&
      algo != FCC_ALGO_CE)
    return FCC_ERR_INVALID;
  if (!tile_shape_ok(o)) return FCC_ERR_INVALID;
  DeviceState* d = nullptr;
  if ((s = device_state(&d)) != FCC_OK) return s;
  const int out_f32 = out_dtype == FCC_F32 ? 1 : 0;
  const RankSumPlan pl = rank_sum_plan(R, M, N, out_f32, o);
  void* ws = nullptr;
  if ((s = get_workspace(d, o, pl.total(), &ws)) != FCC_OK) return s;
  const int64_t Ms = per_shard ? M / R : M;

  if (algo != FCC_ALGO_FUSED)
    return rank_sum_unfused(R, A, B, out, R, per_shard, M, N, K, out_f32, o, d, ws, pl, st);

  if (deterministic_of(o)) {
    const int mode = per_shard ? MODE_RS : MODE_AR;
    GemmParams p;
    if ((s = gemm_params(p, d, mode, R, A, B, out, R, M, N, K, Ms, 0, M, out_f32, o)) != FCC_OK)
      return s;
    // The last round's K halves need room for their partial sums; a caller's
    // workspace too small for them leaves the column halves instead.
    const int kt = ksplit_tiles(p, gemm_slots(p, d, o));
    if (kt > 0) {
      const size_t sb = ksplit_ws_bytes(kt, p.cg);
      const bool caller = o != nullptr && o->workspace != nullptr;
      if (!caller || (o->workspace_bytes >= sb && aligned16(o->workspace))) {
        void* sws = nullptr;
        if ((s = get_workspace(d, o, sb, &sws)) != FCC_OK) return s;
        p.split_ws = static_cast<float*>(sws);
      }
    }
    return run_gemm(p, mode, d, o, st);
  }

  // Push mode: every (rank, tile) adds its f32 result into the owner's buffer.
  const int mode = per_shard ? MODE_RS_PUSH : MODE_AR_PUSH;
  GemmParams p;
  if ((s = gemm_params(p, d, mode, R, A, B, out, R, M, N, K, Ms, 0, M, out_f32, o)) != FCC_OK)
    return s;
  if (out_f32) {
    // Accumulate in place: zero the destinations first.
    if (per_shard) {
      for (int j = 0; j < R; ++j)
        if (cudaMemsetAsync(out[j], 0, static_cast<size_t>(Ms) * N * 4, st) != cudaSuccess)
          return FCC_ERR_CUDA;
    } else if (cudaMemsetAsync(out[0], 0, static_cast<size_t>(M) * N * 4, st) != cudaSuccess) {
      return FCC_ERR_CUDA;
    }
  } else {
    char* base = static_cast<char*>(ws);
    p.acc_ws = reinterpret_cast<float*>(base);
    p.tickets = reinterpret_cast<int*>(base + align_up(pl.acc_bytes));
    if (cudaMemsetAsync(ws, 0, pl.total(), st) != cudaSuccess) return FCC_ERR_CUDA;
  }
  if ((s = run_gemm(p, mode, d, o, st)) != FCC_OK) return s;
  if (!per_shard && out_f32) {
    for (int r = 1; r < R; ++r)
      if (cudaMemcpyAsync(out[r], out[0], static_cast<size_t>(M) * N * 4, cudaMemcpyDeviceToDevice,
                          st) != cudaSuccess)
        return FCC_ERR_CUDA;
  }
  return FCC_OK;
}

// ---------------------------------------------------------------- GEMV
struct GemvPlan {
  int groups = 0, splits = 0;
  size_t partial_bytes = 0;
  size_t ticket_bytes = 0;
  size_t total() const { return align_up(partial_bytes) + align_up(ticket_bytes); }
};

GemvPlan gemv_plan(int R, int64_t M, int64_t N, int64_t K, int sms, const fcc_opts* o) {
  GemvPlan g;
  gemv_shape(N, R, K, sms, o != nullptr ? o->max_ctas : 0, &g.groups, &g.splits);
  g.partial_bytes = gemv_partial_bytes(g.groups, g.splits, M);
  g.ticket_bytes = static_cast<size_t>(g.groups) * 4;
  return g;
}

}  // namespace

const EnvDefaults& env_defaults() {
  static EnvDefaults e;
  static std::once_flag once;
  std::call_once(once, [] {
    auto integer = [](const char* name, long long lo, long long hi, long long* out) {
      const char* v = std::getenv(name);
      if (v == nullptr || *v == 0) return false;
      char* end = nullptr;
      const long long n = std::strtoll(v, &end, 10);
      if (end == nullptr || *end != 0 || n < lo || n > hi) return false;
      *out = n;
      return true;
    };
    if (const char* v = std::getenv("FCC_ALGO")) {
      std::string a(v);
      for (char& c : a) c = static_cast<char>(std::tolower(static_cast<unsigned char>(c)));
      if (a == "fused") e.algo = FCC_ALGO_FUSED;
      else if (a == "unfused") e.algo = FCC_ALGO_UNFUSED;
      else if (a == "interdecom") e.algo = FCC_ALGO_INTERDECOM;
      else if (a == "ce") e.algo = FCC_ALGO_CE;
    }
    long long n = 0;
    if (integer("FCC_DETERMINISTIC", 0, 1, &n)) e.deterministic = static_cast<int>(n);
    if (integer("FCC_CHUNKS", 1, kMaxChunks, &n)) e.chunks = static_cast<int>(n);
    if (integer("FCC_TIMEOUT_MS", 1, 3600 * 1000, &n)) e.timeout_ns = n * 1000 * 1000;
  });
  return e;
}

int* device_status_ptr() {
  DeviceState* d = nullptr;
  return device_state(&d) == FCC_OK ? d->status : nullptr;
}

int device_sm_count() {
  DeviceState* d = nullptr;
  return device_state(&d) == FCC_OK ? d->sms : 1;
}

uint64_t bump_launch_count(uint64_t n) { return g_launches.fetch_add(n) + n; }

}  // namespace fcc

using namespace fcc;

extern "C" {

fcc_status fcc_gemm_rs(int R, const void* const* A, const void* const* B, void* const* out_shard,
                       int64_t M, int64_t N, int64_t K, fcc_dtype in, fcc_dtype out,
                       const fcc_opts* opts, fcc_stream_t stream) {
  return rank_sum_call(R, A, B, out_shard, true, M, N, K, in, out, opts,
                       reinterpret_cast<cudaStream_t>(stream));
}

fcc_status fcc_gemm_ar(int R, const void* const* A, const void* const* B, void* const* out,
                       int64_t M, int64_t N, int64_t K, fcc_dtype in, fcc_dtype out_dtype,
                       const fcc_opts* opts, fcc_stream_t stream) {
  return rank_sum_call(R, A, B, out, false, M, N, K, in, out_dtype, opts,
                       reinterpret_cast<cudaStream_t>(stream));
}

fcc_status fcc_gemv_ar(int R, const void* const* A, const void* const* B, void* const* out,
                       int64_t M, int64_t N, int64_t K, fcc_dtype in, fcc_dtype out_dtype,
                       const fcc_opts* opts, fcc_stream_t stream) {
  fcc_status s = check_gemm(R, A, B, M, N, K, in);
  if (s != FCC_OK) return s;
  if (M > 16) return FCC_ERR_INVALID;
  if ((s = check_out_dtype(out_dtype)) != FCC_OK) return s;
  if (!ptrs_ok(out, R)) return FCC_ERR_INVALID;
  DeviceState* d = nullptr;
  if ((s = device_state(&d)) != FCC_OK) return s;
  // AUTO resolves here; the copy carries the choice to the planning helpers,
  // which read the algorithm from the options themselves.
  fcc_opts chosen;
  if (opts != nullptr) {
    chosen = *opts;
  } else {
    std::memset(&chosen, 0, sizeof(chosen));
    chosen.deterministic = 1;
  }
  if (chosen.algo == FCC_ALGO_AUTO)
    chosen.algo = choose_algo(FCC_OP_GEMV_AR, R, M, N, K, d->sms, chosen.max_ctas);
  opts = &chosen;
  const fcc_algo algo = chosen.algo;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int out_f32 = out_dtype == FCC_F32 ? 1 : 0;
  if (algo != FCC_ALGO_FUSED) {
    if (algo == FCC_ALGO_INTERDECOM) return FCC_ERR_UNSUPPORTED;  // one 8-row chunk: nothing to split
    if (algo != FCC_ALGO_UNFUSED && algo != FCC_ALGO_CE) return FCC_ERR_INVALID;
    const RankSumPlan pl = rank_sum_plan(R, M, N, out_f32, opts);
    void* ws = nullptr;
    if ((s = get_workspace(d, opts, pl.total(), &ws)) != FCC_OK) return s;
    return rank_sum_unfused(R, A, B, out, R, false, M, N, K, out_f32, opts, d, ws, pl, st);
  }
  const GemvPlan g = gemv_plan(R, M, N, K, d->sms, opts);
  // The splits of a column group sum through distributed shared memory when
  // they fit on the device as clusters (no partials or tickets in memory);
  // otherwise the last arriving CTA of a group sums the partials.
  const bool cluster = gemv_cluster_fits(g.groups, g.splits);
  void* ws = nullptr;
  if (!cluster && (s = get_workspace(d, opts, g.total(), &ws)) != FCC_OK) return s;
  GemvParams p;
  std::memset(&p, 0, sizeof(p));
  for (int r = 0; r < R; ++r) {
    if ((s = make_map(&p.mapA[r], A[r], M, K, kGemvTok)) != FCC_OK) return s;
    if ((s = make_map(&p.mapB[r], B[r], K, N, kBK)) != FCC_OK) return s;
    p.out[r] = out[r];
  }
  p.R = R;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.kb_per_rank = static_cast<int>(cdiv(K, kBK));
  p.groups = g.groups;
  p.splits = g.splits;
  p.gen = next_gemv_gen();
  p.out_f32 = out_f32;
  p.partials = static_cast<float*>(ws);
  p.tickets = reinterpret_cast<int*>(static_cast<char*>(ws) + align_up(g.partial_bytes));
  p.status = d->status;
  p.timeout_ns = timeout_of(opts);
  p.cluster = cluster ? 1 : 0;
  if (cluster) {
    p.partials = nullptr;
    p.tickets = nullptr;
  } else if ((opts == nullptr || opts->workspace == nullptr) && g.groups <= kMaxGemvGroups) {
    // Library-held tickets: consistent across calls without clearing.
    if ((s = gemv_internal_tickets(&p.tickets)) != FCC_OK) return s;
  } else if (cudaMemsetAsync(p.tickets, 0, g.ticket_bytes, st) != cudaSuccess) {
    return FCC_ERR_CUDA;  // caller workspace may hold anything: start the tickets at zero
  }
  if (launch_gemv(p, g.groups * g.splits, st) != cudaSuccess) return FCC_ERR_CUDA;
  g_launches.fetch_add(1);
  return FCC_OK;
}

fcc_status fcc_ag_gemm(int R, const void* const* X_shard, const void* const* B, void* const* out,
                       void* const* gathered, int64_t M, int64_t N, int64_t K, fcc_dtype in,
                       fcc_dtype out_dtype, const fcc_opts* opts, fcc_stream_t stream) {
  fcc_status s = check_gemm(R, X_shard, B, M, N, K, in);
  if (s != FCC_OK) return s;
  if (M % R != 0) return FCC_ERR_INVALID;
  if ((s = check_out_dtype(out_dtype)) != FCC_OK) return s;
  if (!ptrs_ok(out, R)) return FCC_ERR_INVALID;
  if (gathered != nullptr)
    for (int r = 0; r < R; ++r)
      if (gathered[r] != nullptr && !aligned16(gathered[r])) return FCC_ERR_INVALID;
  const fcc_algo algo = algo_of(opts);
  if (algo != FCC_ALGO_FUSED && algo != FCC_ALGO_UNFUSED && algo != FCC_ALGO_INTERDECOM &&
      algo != FCC_ALGO_CE)
    return FCC_ERR_INVALID;
  if (!tile_shape_ok(opts)) return FCC_ERR_INVALID;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DeviceState* d = nullptr;
  if ((s = device_state(&d)) != FCC_OK) return s;
  const int64_t Ms = M / R;
  const int out_f32 = out_dtype == FCC_F32 ? 1 : 0;

  if (algo == FCC_ALGO_FUSED) {
    GemmParams p;
    if ((s = gemm_params(p, d, MODE_AG, R, X_shard, B, out, R, M, N, K, Ms, 0, M, out_f32,
                         opts)) != FCC_OK)
      return s;
    if ((s = run_gemm(p, MODE_AG, d, opts, st)) != FCC_OK) return s;
    // The gathered copies are an optional output: materialise them after the GEMM
    // has read the shards in place.
    if (gathered != nullptr) {
      for (int r = 0; r < R; ++r)
        if (gathered[r] != nullptr &&
            cuda_fail(launch_gather_rows(X_shard, R, Ms, K, gathered[r], st)) != FCC_OK)
          return FCC_ERR_CUDA;
    }
    return FCC_OK;
  }

  // Unfused: gather X (SM copy kernel or copy engines), then one GEMM per rank;
  // InterDecom: the same in row chunks, gather and GEMM pipelined.
  void* ws = nullptr;
  const bool have_g = gathered != nullptr && gathered[0] != nullptr;
  const size_t xbytes = static_cast<size_t>(M) * K * 2;
  if (!have_g) {
    if ((s = get_workspace(d, opts, xbytes, &ws)) != FCC_OK) return s;
  }
  void* g0 = have_g ? gathered[0] : ws;
  const void* Ag[FCC_MAX_RANKS];
  for (int r = 0; r < R; ++r) Ag[r] = g0;
  if (algo == FCC_ALGO_INTERDECOM) {
    // Row chunks of the gathered X: every chunk's gather is queued on a side
    // stream at once, and the GEMM of chunk i (rows [m0, m1) of every rank's
    // output) runs on the caller's stream after chunk i's gather, so chunk
    // i+1's gather overlaps chunk i's GEMM.  Chunks are whole 256-row tiles.
    int chunks = chunks_of(opts) > 0 ? chunks_of(opts) : ag_model_chunks(R, M, N, K);
    chunks = std::max(1, std::min(chunks, kMaxChunks));
    const int64_t rows = chunk_rows(M, chunks, 2 * kBM);
    cudaStream_t side = d->side[0];
    cudaEvent_t fork = d->ev[kMaxChunks];
    if (cudaEventRecord(fork, st) != cudaSuccess || cudaStreamWaitEvent(side, fork, 0) != cudaSuccess)
      return FCC_ERR_CUDA;
    int i = 0;
    for (int64_t m0 = 0; m0 < M; m0 += rows, ++i) {
      const int64_t m1 = std::min(M, m0 + rows);
      if (cuda_fail(launch_gather_rows_range(X_shard, R, Ms, K, g0, m0, m1, side)) != FCC_OK)
        return FCC_ERR_CUDA;
      if (cudaEventRecord(d->ev[i], side) != cudaSuccess ||
          cudaStreamWaitEvent(st, d->ev[i], 0) != cudaSuccess)
        return FCC_ERR_CUDA;
      GemmParams p;
      if ((s = gemm_params(p, d, MODE_PARTIAL, R, Ag, B, out, R, M, N, K, M, m0, m1, out_f32,
                           opts)) != FCC_OK)
        return s;
      if ((s = run_gemm(p, MODE_PARTIAL, d, opts, st)) != FCC_OK) return s;
    }
  } else {
    if (algo == FCC_ALGO_CE) {
      for (int sh = 0; sh < R; ++sh)
        if (cudaMemcpyAsync(static_cast<char*>(g0) + static_cast<size_t>(sh) * Ms * K * 2,
                            X_shard[sh], static_cast<size_t>(Ms) * K * 2,
                            cudaMemcpyDeviceToDevice, st) != cudaSuccess)
          return FCC_ERR_CUDA;
    } else if (cuda_fail(launch_gather_rows(X_shard, R, Ms, K, g0, st)) != FCC_OK) {
      return FCC_ERR_CUDA;
    }
    GemmParams p;
    if ((s = gemm_params(p, d, MODE_PARTIAL, R, Ag, B, out, R, M, N, K, M, 0, M, out_f32,
                         opts)) != FCC_OK)
      return s;
    if ((s = run_gemm(p, MODE_PARTIAL, d, opts, st)) != FCC_OK) return s;
  }
  if (have_g) {
    for (int r = 1; r < R; ++r)
      if (gathered[r] != nullptr &&
          cudaMemcpyAsync(gathered[r], g0, xbytes, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return FCC_ERR_CUDA;
  }
  return FCC_OK;
}

size_t fcc_workspace_size(fcc_op op, int R, int64_t M, int64_t N, int64_t K,
                          const fcc_opts* opts) {
  (void)K;
  if (R < 1 || R > FCC_MAX_RANKS || M <= 0 || N <= 0) return 0;
  switch (op) {
    case FCC_OP_GEMM_RS:
    case FCC_OP_GEMM_AR: {
      // bf16 vs f32 output only matters for the push mode; report the larger.
      size_t bytes = rank_sum_plan(R, M, N, false, opts).total();
      if (algo_of(opts) == FCC_ALGO_FUSED && deterministic_of(opts)) {
        // The K halves of the last round: at most half a round of tiles.
        int sms = 0, dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
          sms = 256;
        int ctas = sms;
        if (opts != nullptr && opts->max_ctas > 0) ctas = std::min(ctas, opts->max_ctas);
        const int64_t single = cdiv(M, kBM) * cdiv(N, kGemmBN);
        const int cg = choose_cg(opts, M, single, ctas);
        const int64_t tiles = cdiv(M, static_cast<int64_t>(kBM) * cg) * cdiv(N, kGemmBN);
        const int64_t half_round = std::max(1, ctas / cg) / 2;
        const int64_t kt = std::min(tiles, half_round);
        if (kt > 0) bytes += align_up(ksplit_ws_bytes(static_cast<int>(kt), cg));
      }
      return bytes;
    }
    case FCC_OP_GEMV_AR: {
      const bool automatic = opts == nullptr || opts->algo == FCC_ALGO_AUTO;
      fcc_opts plain;
      if (opts != nullptr) {
        plain = *opts;
      } else {
        std::memset(&plain, 0, sizeof(plain));
        plain.deterministic = 1;
      }
      plain.algo = FCC_ALGO_UNFUSED;
      const size_t unfused = rank_sum_plan(R, M, N, false, &plain).total();
      if (!automatic && opts->algo != FCC_ALGO_FUSED) return rank_sum_plan(R, M, N, false, opts).total();
      int sms = 0, dev = 0;
      if (cudaGetDevice(&dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 256;
      const size_t fused = gemv_plan(R, M, N, K, sms, opts).total();
      // AUTO may take either form (per shape): room for both.
      return automatic ? std::max(fused, unfused) : fused;
    }
    case FCC_OP_AG_GEMM:
      return algo_of(opts) == FCC_ALGO_FUSED ? 0 : static_cast<size_t>(M) * K * 2;
  }
  return 0;
}

fcc_status fcc_stream_status(fcc_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FCC_ERR_CUDA;
  DeviceState* d = nullptr;
  fcc_status s = device_state(&d);
  if (s != FCC_OK) return s;
  int v = 0;
  if (cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FCC_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return FCC_ERR_CUDA;
  }
  return static_cast<fcc_status>(v);
}

const char* fcc_status_string(fcc_status s) {
  switch (s) {
    case FCC_OK: return "ok";
    case FCC_ERR_INVALID: return "invalid argument";
    case FCC_ERR_UNSUPPORTED: return "unsupported";
    case FCC_ERR_CUDA: return "CUDA error";
    case FCC_ERR_CAPACITY: return "receive capacity exceeded";
    case FCC_ERR_TIMEOUT: return "device wait timed out";
    case FCC_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

double fcc_interdecom_time(double G, double X, double alpha, int chunks) {
  if (chunks < 1) chunks = 1;
  return std::max(G, X) + std::min(G, X) / chunks + chunks * alpha;
}

fcc_algo fcc_choose_algo(fcc_op op, int R, int64_t M, int64_t N, int64_t K, int sms,
                         int max_ctas) {
  if (sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      sms = 152;
    }
  }
  // (M, N, K describe the GEMM operators; the embedding's choice needs none)
  if (op != FCC_OP_EMBEDDING_A2A && (R < 1 || R > FCC_MAX_RANKS || N <= 0 || K <= 0))
    return FCC_ALGO_FUSED;
  return choose_algo(op, R, M, N, K, sms, max_ctas);
}

int fcc_interdecom_chunks(double G, double X, double alpha, int max_chunks) {
  if (max_chunks < 1) max_chunks = 1;
  if (!(G > 0) || !(X > 0)) return 1;
  if (!(alpha > 0)) return max_chunks;
  const double c = std::sqrt(std::min(G, X) / alpha);
  int lo = static_cast<int>(std::floor(c));
  int hi = lo + 1;
  lo = std::max(1, std::min(lo, max_chunks));
  hi = std::max(1, std::min(hi, max_chunks));
  return fcc_interdecom_time(G, X, alpha, hi) < fcc_interdecom_time(G, X, alpha, lo) ? hi : lo;
}

uint64_t fcc_launch_count(void) { return g_launches.load(); }

const char* fcc_version(void) { return "0.1.0"; }

fcc_status fcc_test_wait_timeout(int64_t timeout_ns, fcc_stream_t stream) {
  if (timeout_ns <= 0) return FCC_ERR_INVALID;
  DeviceState* d = nullptr;
  fcc_status s = device_state(&d);
  if (s != FCC_OK) return s;
  return cuda_fail(launch_wait_probe(d->status, static_cast<unsigned long long>(timeout_ns),
                                     reinterpret_cast<cudaStream_t>(stream)));
}

// Test support: a 1-rank 384 x 256 x 128 reduce-scatter (zeros) on two single
// CTAs, so its three 128-row tiles take a round of two and a last tile split
// in K; the second K half waits for a call id the first half never writes,
// so its bounded wait runs out after timeout_ns.
fcc_status fcc_test_ksplit_wait_timeout(int64_t timeout_ns, fcc_stream_t stream) {
  if (timeout_ns <= 0) return FCC_ERR_INVALID;
  DeviceState* d = nullptr;
  fcc_status s = device_state(&d);
  if (s != FCC_OK) return s;
  constexpr int64_t kM = 384, kN = 256, kK = 128;
  const size_t a_bytes = static_cast<size_t>(kM) * kK * 2, b_bytes = static_cast<size_t>(kK) * kN * 2,
               o_bytes = static_cast<size_t>(kM) * kN * 4, w_bytes = ksplit_ws_bytes(1, 1);
  const size_t total = align_up(a_bytes) + align_up(b_bytes) + align_up(o_bytes) + align_up(w_bytes);
  fcc_opts o;
  std::memset(&o, 0, sizeof(o));
  o.algo = FCC_ALGO_FUSED;
  o.deterministic = 1;
  o.max_ctas = 2;
  o.cta_pair = 1;
  o.timeout_ns = timeout_ns;
  void* ws = nullptr;
  if ((s = get_workspace(d, nullptr, total, &ws)) != FCC_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, total, st) != cudaSuccess) return FCC_ERR_CUDA;
  char* base = static_cast<char*>(ws);
  const void* A[1] = {base};
  const void* B[1] = {base + align_up(a_bytes)};
  void* out[1] = {base + align_up(a_bytes) + align_up(b_bytes)};
  GemmParams p;
  if ((s = gemm_params(p, d, MODE_RS, 1, A, B, out, 1, kM, kN, kK, kM, 0, kM, 1, &o)) != FCC_OK)
    return s;
  if (p.cg != 1 || ksplit_tiles(p, gemm_slots(p, d, &o)) != 1) return FCC_ERR_UNSUPPORTED;
  p.split_ws = reinterpret_cast<float*>(base + align_up(a_bytes) + align_up(b_bytes) +
                                        align_up(o_bytes));
  p.flag_skew = 2;  // (call ids are odd: the skewed one is never written)
  return run_gemm(p, MODE_RS, d, &o, st);
}

}  // extern "C"

// ------------------------------------------------------------------------
// Helpers for entry points that must not create streams, events or pools:
// they only look up what already exists (driver entry point, symbol addresses).
namespace fcc {

fcc_status light_encoder_ready() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode != nullptr) return FCC_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return FCC_ERR_CUDA;
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  return FCC_OK;
}

fcc_status light_make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols,
                          uint32_t box_rows) {
  fcc_status s = light_encoder_ready();
  if (s != FCC_OK) return s;
  return make_map(m, ptr, rows, cols, box_rows);
}

fcc_status light_status_word(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FCC_ERR_CUDA;
  static int* cached[kMaxDevices] = {};
  std::lock_guard<std::mutex> lk(g_mu);
  if (cached[dev] == nullptr) {
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&cached[dev]), g_status_word) != cudaSuccess)
      return FCC_ERR_CUDA;
  }
  *out = cached[dev];
  return FCC_OK;
}

fcc_status light_check_gemm(int R, const void* const* A, const void* const* B, int64_t M,
                            int64_t N, int64_t K, fcc_dtype in) {
  return check_gemm(R, A, B, M, N, K, in);
}

void count_launch() { g_launches.fetch_add(1); }

}  // namespace fcc

// ------------------------------------------------------------------------
// Host helpers shared with the other translation units (MoE entry point).
namespace fcc {

fcc_status internal_prepare(const fcc_opts* o, size_t ws_bytes, void** ws, int** status,
                            int* sms, unsigned long long* timeout_ns) {
  DeviceState* d = nullptr;
  fcc_status s = device_state(&d);
  if (s != FCC_OK) return s;
  if ((s = get_workspace(d, o, ws_bytes, ws)) != FCC_OK) return s;
  *status = d->status;
  *sms = (o != nullptr && o->max_ctas > 0) ? std::min(d->sms, o->max_ctas) : d->sms;
  *timeout_ns = timeout_of(o);
  return FCC_OK;
}

fcc_status internal_make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols,
                             uint32_t box_rows) {
  return make_map(m, ptr, rows, cols, box_rows);
}

fcc_status internal_streams_events(cudaStream_t* side, int nside, cudaEvent_t* ev, int nev) {
  DeviceState* d = nullptr;
  fcc_status s = device_state(&d);
  if (s != FCC_OK) return s;
  if (nside > kSideStreams || nev > kMaxChunks + kSideStreams + 2) return FCC_ERR_INVALID;
  for (int i = 0; i < nside; ++i) side[i] = d->side[i];
  for (int i = 0; i < nev; ++i) ev[i] = d->ev[i];
  return FCC_OK;
}

fcc_status internal_host_buffer(size_t bytes, void** out) {
  DeviceState* d = nullptr;
  fcc_status s = device_state(&d);
  if (s != FCC_OK) return s;
  std::lock_guard<std::mutex> lk(g_mu);
  if (d->host_bytes < bytes) {
    if (d->host != nullptr && cudaFreeHost(d->host) != cudaSuccess) return FCC_ERR_CUDA;
    d->host = nullptr;
    d->host_bytes = 0;
    if (cudaHostAlloc(&d->host, bytes, cudaHostAllocDefault) != cudaSuccess) return FCC_ERR_CUDA;
    d->host_bytes = bytes;
  }
  *out = d->host;
  return FCC_OK;
}

fcc_status internal_side_stream(cudaStream_t* side, cudaEvent_t* ev, int n) {
  DeviceState* d = nullptr;
  fcc_status s = device_state(&d);
  if (s != FCC_OK) return s;
  if (n > 8) return FCC_ERR_INVALID;
  *side = d->side[1];
  for (int i = 0; i < n; ++i) ev[i] = d->ev[kMaxChunks - 8 + i];
  return FCC_OK;
}

}  // namespace fcc

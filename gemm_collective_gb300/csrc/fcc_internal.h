// fcc_internal.h -- declarations shared by the libfcc translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "fcc.h"

namespace fcc {

// Sets a kernel's dynamic shared-memory limit once per device (the attribute
// belongs to the device's context) instead of on every launch; `done` is the
// kernel's own flag array.  A failed attempt is retried on the next launch.
template <class Kernel>
cudaError_t smem_attr_once(bool (&done)[64], Kernel kern, int bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = -1;
  if (dev >= 0 && done[dev]) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0) done[dev] = true;
  return e;
}

// Resident blocks per SM of `kern` with `threads` threads and no dynamic
// shared memory, looked up once per device (`cache` is the kernel's own).
template <class Kernel>
int blocks_per_sm_once(int (&cache)[64], Kernel kern, int threads) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = -1;
  if (dev >= 0 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, 0) != cudaSuccess || n < 1)
    return 1;
  if (dev >= 0) cache[dev] = n;
  return n;
}

// Launches kern<<<grid, block, smem, st>>>(args...) with programmatic stream
// serialization (and a cluster of `cluster` CTAs when > 1): the launch may
// overlap the previous kernel on `st`, so every thread of `kern` must call
// ptx::griddep_wait() before it touches global memory.
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, unsigned cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

constexpr int kBM = 128;       // output tile rows (one TMEM lane per row)
constexpr int kBK = 64;        // K per pipeline stage (128 bytes of bf16: one swizzle row)
constexpr int kGemmThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kCopyWarps = 2;      // grouped mode: warps 6-7 stage the expert rows
constexpr int kGemvTok = 16;   // GEMV: token rows per TMA box (M <= 16)

enum GemmMode : int {
  MODE_RS = 0,         // reduce-scatter, ordered tile-owner accumulation over ranks
  MODE_AR = 1,         // all-reduce: the same, stored to every rank's buffer
  MODE_PARTIAL = 2,    // plain per-rank GEMM: out[r] = A_r @ B_r over a row window
  MODE_AG = 3,         // all-gather + GEMM: A tile from the owning shard
  MODE_RS_PUSH = 4,    // reduce-scatter, push: red.add of each rank's tile into the owner
  MODE_AR_PUSH = 5,    // all-reduce, push
  MODE_GROUPED = 6,    // MoE grouped expert GEMM over a device-built tile table
};

struct GemmParams {
  CUtensorMap mapA[FCC_MAX_RANKS];
  CUtensorMap mapB[FCC_MAX_RANKS];
  void* out[FCC_MAX_RANKS];
  int R;
  int M, N, K;          // GEMM extents (RS/AR: all rows; AG: gathered rows; PARTIAL: rows of A_r)
  int Ms;               // rows per shard (RS, AG)
  int m_begin, m_end;   // row window (PARTIAL; others 0..M)
  int tiles_m, tiles_n; // tile grid of one rank's output
  int num_tiles;        // work items: whole tiles, then the halves from split_first on
  int split_first;      // RS/AR/AG/PARTIAL: first half-tile item (= num_tiles: none)
  int k_iters;          // pipeline stages per tile
  int kb_per_rank;      // ceil(K / kBK)
  int out_f32;          // output storage: 1 = f32, 0 = bf16
  int group_m;          // raster group height (tiles)
  int* status;
  unsigned long long timeout_ns;
  float* acc_ws;        // push mode with bf16 output: f32 accumulation rows (M x N)
  int* tickets;         // push mode with bf16 output: per (tile, CTA of the pair) counters
  int cg;               // host side: CTAs per cluster (1 or 2)
  unsigned long long* phase_ns;  // NULL, or 4 per CTA: span, epilogue busy, MMA wait, tiles
  // When the next kernel on the stream may launch (programmatic launch):
  // 0 = once this kernel has started (its set-up then overlaps our run),
  // 1 = once each CTA's last accumulator is complete (a small next kernel then
  // does not sit resident beside this one for its whole run).
  int trigger_late;
  // RS / AR, ksplit = 1: the work items from split_first on are the K halves
  // of the last round's tiles (k iterations [0, k_half) and [k_half, k_iters)),
  // not column halves.  The first half stores its f32 partial (one 128 x 256
  // block per CTA of the pair) to split_ws and then sets the tile's flag to
  // the call's id; the second half waits for the flag, adds the partial to
  // its own accumulator and stores the result.  A flag left by another call
  // holds another id, so the flags need no clearing between calls.
  int ksplit;
  int k_half;
  float* split_ws;                    // [split tiles][CG][128][256] f32, then the flags
  unsigned long long* split_flags;    // [split tiles][CG]
  unsigned long long call_id;
  unsigned long long flag_skew;       // test support: the second half waits for call_id + this
};

// Bytes of the K-split workspace for `tiles` split tiles of `cg` CTAs each.
inline size_t ksplit_ws_bytes(int tiles, int cg) {
  const size_t part = static_cast<size_t>(tiles) * cg * 128 * 256 * 4;
  return part + static_cast<size_t>(tiles) * cg * 8;
}

struct GemvParams {
  CUtensorMap mapA[FCC_MAX_RANKS];  // [M, K], box of 16 rows (rows past M read as zeros)
  CUtensorMap mapB[FCC_MAX_RANKS];  // [K, N]
  void* out[FCC_MAX_RANKS];
  int R, M, N, K;
  int kb_per_rank;
  int groups;           // column groups of 512 columns: ceil(N / 512)
  int splits;           // CTAs per group (parts of the R*K range); grid = groups * splits
  int out_f32;
  float* partials;      // [groups * splits][M][512]
  int* tickets;         // [groups]: (generation << 8) | arrivals
  unsigned gen;         // call generation, 1..2^24-1 (never 0: zeroed tickets are "old")
  int* status;
  unsigned long long timeout_ns;
  int cluster;          // 1: a column group's splits are one cluster and sum through
                        // distributed shared memory (no partials, no tickets)
};

// Launchers (return cudaSuccess or the launch error).
// Grouped expert GEMM (MoE): tile t belongs to expert e with
// tile_start[e] <= t < tile_start[e+1]; the expert's rows are
// [expert_base[e], expert_base[e] + expert_rows[e]) of rank e/Eloc's receive
// buffers.  The tile table is written on the device by the dispatch kernels.
struct GroupedParams {
  CUtensorMap mapA[FCC_MAX_RANKS];     // recv_x[d]: [cap, H]
  CUtensorMap mapB[FCC_MAX_EXPERTS];   // W_e: [H, F]
  void* out[FCC_MAX_RANKS];            // recv_y[d]: [cap, F]
  int R, E, Eloc;
  int N, K;                            // F, H
  int tiles_n;                         // ceil(F / 256)
  int kb_per_rank;                     // ceil(H / 64)
  int out_f32;
  const int* tile_start;               // [E + 1]
  const int* expert_base;              // [E]
  const int* expert_rows;              // [E] (clamped to the receive capacity)
  int e_lo, e_hi;                      // this launch covers the tiles of experts [e_lo, e_hi)
  int* status;
  unsigned long long timeout_ns;
  // Gather mode (gather = 1): the A rows are read straight from the source
  // tokens instead of from a staged copy.  Every mapA[d] is then the map of
  // the sources' concatenated [R*T, H] matrix with a box one row high, and row
  // i of rank d's receive order is its row recv_src[d][i] (= s*T + t).
  const int* recv_src[FCC_MAX_RANKS];  // [cap] per receiving rank
  int gather;
  // In-kernel staging (stage_copy = 1): the kernel's copy warps write row i of
  // receiving rank d's order, source row recv_src[d][i] of src_x, to row i of
  // stage_x[d] (the buffer mapA[d] maps), one (expert, m tile) unit after
  // another in tile order.  ready[u] counts the rows of unit u written so far
  // (u = tile_start[e] / tiles_n + m); the TMA producer waits for a unit's
  // count to reach its rows before loading them.  ready[] and copy_cursor are
  // zero at launch.
  const void* src_x[FCC_MAX_RANKS];    // [T, H] per source rank
  void* stage_x[FCC_MAX_RANKS];        // [cap, H] per receiving rank
  int T;                               // tokens per source rank
  int* ready;                          // [units]
  int* copy_cursor;                    // next chunk of rows to claim
  int stage_copy;
  unsigned long long* phase_ns;        // NULL, or 4 per CTA (as GemmParams)
  int trigger_late;                    // as GemmParams
};

// cg = 1: one CTA per 128 x 256 tile; cg = 2: a CTA pair (cluster of 2) per
// 256 x 256 tile.  grid is in CTAs (a multiple of cg).
cudaError_t launch_gemm(const GemmParams& p, int mode, int cg, int grid, cudaStream_t st);
cudaError_t launch_grouped_gemm(const GroupedParams& p, int cg, int grid, cudaStream_t st);
// Clusters of cg CTAs of the GEMM kernel that fit on the current device at once.
int gemm_max_clusters(int cg);
cudaError_t launch_gemv(const GemvParams& p, int grid, cudaStream_t st);
// Whether the cluster form of the GEMV's final sum fits the current device.
bool gemv_cluster_fits(int groups, int splits);
int gemv_smem_bytes();
// GEMV grid shape for N columns and R*K rows over `sms` SMs (max_ctas 0 = no cap).
void gemv_shape(int64_t N, int R, int64_t K, int sms, int max_ctas, int* groups, int* splits);
size_t gemv_partial_bytes(int groups, int splits, int64_t M);
constexpr int kMaxGemvGroups = 1024;  // column groups with library-held tickets
unsigned next_gemv_gen();
// Device address of the library's GEMV ticket array on the current device.
fcc_status gemv_internal_tickets(int** out);

// Elementwise helpers (fcc_aux.cu).
// out_j rows [row_begin,row_end) of shard j = sum_r P[r] rows, P[r] is [M, N] f32.
cudaError_t launch_reduce_shards(const float* const* P, int R, void* const* out, int nout,
                                 int per_shard, int64_t M, int64_t N, int64_t Ms,
                                 int64_t row_begin, int64_t row_end, int out_f32,
                                 cudaStream_t st);
// dst = [X_0; ...; X_{R-1}] (each X_s is [Ms, K] bf16), all rows or rows
// [row_begin, row_end) of the gathered [R*Ms, K] matrix.
cudaError_t launch_gather_rows(const void* const* X, int R, int64_t Ms, int64_t K, void* dst,
                               cudaStream_t st);
cudaError_t launch_gather_rows_range(const void* const* X, int R, int64_t Ms, int64_t K,
                                     void* dst, int64_t row_begin, int64_t row_end,
                                     cudaStream_t st);
cudaError_t launch_wait_probe(int* status, unsigned long long timeout_ns, cudaStream_t st);

// Shared host helpers (fcc_api.cu).
int* device_status_ptr();
int device_sm_count();
uint64_t bump_launch_count(uint64_t n);

}  // namespace fcc

namespace fcc {
// Look-up-only helpers (no streams, events or device memory are created).
fcc_status light_encoder_ready();
fcc_status light_make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols,
                          uint32_t box_rows);
fcc_status light_status_word(int** out);
fcc_status light_check_gemm(int R, const void* const* A, const void* const* B, int64_t M,
                            int64_t N, int64_t K, fcc_dtype in);
void count_launch();
}  // namespace fcc

namespace fcc {
// Device state, workspace (caller's or the pool), status word, usable SM count
// and the wait limit for a call; the tensor-map encoder is ready afterwards.
fcc_status internal_prepare(const fcc_opts* o, size_t ws_bytes, void** ws, int** status,
                            int* sms, unsigned long long* timeout_ns);
// 2-D bf16 tensor map, box [box_rows, 64], 128-byte swizzle (after internal_prepare).
fcc_status internal_make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols,
                             uint32_t box_rows);
// A side stream and n <= 8 events of the current device (after internal_prepare).
fcc_status internal_side_stream(cudaStream_t* side, cudaEvent_t* ev, int n);
// The device's side streams 0..nside-1 (nside <= 4) and events 0..nev-1
// (nev <= 70), shared with the InterDecom paths of the other operators.
fcc_status internal_streams_events(cudaStream_t* side, int nside, cudaEvent_t* ev, int nev);
// A pinned host buffer of at least `bytes` for the current device (grown with
// cudaHostAlloc; valid until the next call that asks for more).
fcc_status internal_host_buffer(size_t bytes, void** out);
// The algorithm FCC_ALGO_AUTO runs (the strategy selector, fcc_api.cu).
fcc_algo choose_algo(fcc_op op, int R, int64_t M, int64_t N, int64_t K, int sms, int max_ctas);
// Defaults from the environment, read once (fcc.h, fcc_opts): the algorithm
// that replaces FCC_ALGO_AUTO (FCC_ALGO_AUTO when unset), the deterministic
// setting of calls without opts (-1 when unset), the InterDecom chunk count
// (0 when unset) and the device wait limit (0 when unset).
struct EnvDefaults {
  fcc_algo algo = FCC_ALGO_AUTO;
  int deterministic = -1;
  int chunks = 0;
  int64_t timeout_ns = 0;
};
const EnvDefaults& env_defaults();
}  // namespace fcc

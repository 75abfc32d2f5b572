// fcc_gemm.cu -- persistent tcgen05 GEMM with collective epilogues (sm_103a).
//
// Persistent kernel: every SM runs one CTA that loops over output tiles.
// Warp 0 streams A and B tiles with TMA into a shared-memory ring; warp 1
// issues tcgen05.mma (bf16 x bf16 -> f32) into one of two TMEM accumulators;
// warps 2-5 drain the other accumulator with tcgen05.ld and perform the
// collective step in the epilogue, so the stores of tile i overlap the MMAs of
// tile i+1.
//
// Two shapes (template parameter CG):
//   CG = 1  one CTA per 128 x 256 tile, tcgen05.mma.cta_group::1 (M = 128),
//           4-stage ring of 48 KiB (A 128x64 + B 64x256).
//   CG = 2  a CTA pair (cluster of 2 on neighbouring SMs) per 256 x 256 tile,
//           tcgen05.mma.cta_group::2 (M = 256) issued by the pair's leader;
//           each CTA loads its 128 rows of A and its 128 columns of B into its
//           own shared memory, so each SM keeps a 7-stage ring of 32 KiB and
//           reads half the B bytes per MMA.  Each CTA's TMEM holds its 128 rows.
//
// The collective step per mode (the fused operators of the mKernel article's
// kernel list and of the SC24 paper's abstract, where each workgroup ships
// its result to the owner as soon as its tile is done):
//   MODE_RS       the tile's K loop runs over (rank 0..R-1) x K, so the one
//                 accumulator holds sum_r A_r B_r for the tile in a fixed
//                 rank order; the owner shard receives one store per element.
//   MODE_AR       the same sum, stored into every rank's buffer.
//   MODE_RS_PUSH  each (rank, tile) is its own work item; its f32 result is
//   MODE_AR_PUSH  added into the owner's f32 buffer with red.global.add.v4.f32;
//                 for bf16 outputs the last arriving rank (ticket) converts.
//   MODE_AG       the A tile is read straight from the shard that owns its rows
//                 (the gather), the B tile and output from the column's rank.
//   MODE_PARTIAL  plain per-rank GEMM over a row window (unfused baselines).
//   MODE_GROUPED  MoE expert GEMM over a tile table built on the device.
//                 With in-kernel staging, two more warps (6-7) copy each
//                 expert's rows from the source tokens into the receive
//                 buffers (the all-to-all) while the tensor cores work on the
//                 units already copied; the TMA producer waits, per tile, for
//                 its unit's row count.
//
// Shared memory operand layouts (128-byte swizzle, as written by TMA):
//   A stage  [128 rows][64 k]   K-major: row m at m*128 B, 8-row groups 1 KiB apart
//   B stage  boxes of [64 k][64 n] MN-major: box i at i*8 KiB, k-row at k*128 B
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "fcc_internal.h"
#include "fcc_ptx.cuh"

namespace fcc {
namespace {

constexpr int kBN = 256;                            // tile columns
constexpr uint32_t kABytes = kBM * kBK * 2;         // 16 KiB per CTA and stage
constexpr uint32_t kBBoxBytes = kBK * 64 * 2;       // 8 KiB: [64 k][64 n]
constexpr uint32_t kTmemCols = 2 * kBN;             // double-buffered accumulator
constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;  // unwinding limit after an abort

// Grouped mode: tile_start[0..E], expert_rows[0..E), expert_base[0..E) copied
// into shared memory once per CTA, so finding a tile's expert (a binary search)
// costs no global-memory round trips on the producer's or the MMA warp's path;
// then the copy warps' chunk prefix [0..E].
constexpr int kTabInts = 4 * FCC_MAX_EXPERTS + 2;
constexpr int kCopyRows = 4;  // rows per claimed chunk of the in-kernel staging copy

template <int MODE>
constexpr int threads_of() {
  return MODE == MODE_GROUPED ? kGemmThreads + 32 * kCopyWarps : kGemmThreads;
}

// CG = CTAs per cluster: 1 (one CTA per 128x256 tile) or 2 (a CTA pair per
// 256x256 tile).  Every TMA load goes to the issuing CTA's own shared memory.
// Ring depth on CTA pairs: five stages for the ordered RS and AR (8-rank
// RS 1.98-2.09 ms against 2.01-2.09 with seven, on three boxes, with lower
// DRAM reads, 4.6 against 5.4 GB; AR 2.05-2.08 against 2.05-2.13; four or
// three stages were slower), seven for the others: the AllGather + GEMM
// (1.99-2.01 against 1.99-2.02 ms with five) and the MoE expert GEMM, whose
// 64-deep K loops and in-kernel row copy want the deeper ring (561 us
// against 566 with six and 585 with five).
template <int CG, bool kShallow = false>
struct Cfg {
  static_assert(CG == 1 || CG == 2, "one CTA or a CTA pair per tile");
  static constexpr int kPairCtas = CG;                      // CTAs of one MMA
  static constexpr int kTileM = kBM * kPairCtas;            // rows of one (pair) tile
  static constexpr int kBNcta = kBN / kPairCtas;            // B columns this CTA holds
  static constexpr int kStages = CG >= 2 ? (kShallow ? 5 : 7) : 4;
  static constexpr uint32_t kBBytes = kBK * kBNcta * 2;     // 32 or 16 KiB
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kTileM, kBN, false, true);
  // A tile whose columns end in the first half of its 256 runs 128 wide.
  static constexpr uint32_t kIdescNarrow = ptx::idesc_bf16_f32(kTileM, kBN / 2, false, true);
  // Grouped mode, CTA pair: an expert's last unit of at most 128 rows runs
  // as an M = 128 pair MMA (64 rows from each CTA), at half the MMA work.
  static constexpr uint32_t kIdescShort = ptx::idesc_bf16_f32(128, kBN, false, true);
  static constexpr uint32_t kIdescShortNarrow = ptx::idesc_bf16_f32(128, kBN / 2, false, true);
  // ... + barriers + flags + the grouped mode's expert tables.
  static constexpr int kSmem = 1024 + kStages * static_cast<int>(kStageBytes) +
                               (2 * kStages + 5) * 8 + 16 + kTabInts * 4;
  static_assert(kSmem <= 232448, "shared memory per CTA");
};

struct Tile {
  int rank;    // rank whose A/B feed the tile (PARTIAL/PUSH/AG-B), -1 = all ranks
  int shard;   // AG: shard that owns the A rows; GROUPED: receiving rank
  int mt, nt;  // tile indices within one rank's output (GROUPED: within the expert)
  int expert;  // GROUPED: expert of the tile
  int row0;    // GROUPED: first receive-buffer row of the tile
  int rows;    // GROUPED: valid rows of the tile
  int half;    // -1: the whole 256-column tile; 0 / 1: its first / second 128 columns
  int kpart;   // -1: the whole K loop; 0 / 1: its first / second half (RS / AR)
  int slot;    // kpart >= 0: the tile's index among the last round's split tiles
  int m128;    // GROUPED on CTA pairs: 1 = at most 128 rows, run as an M = 128 pair MMA
};

__device__ __forceinline__ void raster(int t, int tiles_m, int tiles_n, int group, int& mt,
                                       int& nt) {
  const int per_group = group * tiles_n;
  const int g = t / per_group;
  const int first = g * group;
  const int gm = min(group, tiles_m - first);
  const int local = t - g * per_group;
  mt = first + local % gm;
  nt = local / gm;
}

template <int MODE, class P>
__device__ __forceinline__ int num_tiles_of(const P& p, const int* tab) {
  if constexpr (MODE == MODE_GROUPED) {
    // Tiles of experts [e_lo, e_hi); the table is written by the dispatch kernels.
    return tab[p.e_hi] - tab[p.e_lo];
  } else {
    return p.num_tiles;
  }
}

template <int MODE, class P>
__device__ __forceinline__ int k_iters_of(const P& p) {
  if constexpr (MODE == MODE_GROUPED) {
    return p.kb_per_rank;
  } else {
    return p.k_iters;
  }
}

template <int MODE, int TM, class P>
__device__ __forceinline__ Tile tile_of(const P& p, int t, const int* tab) {
  Tile tl;
  tl.rank = -1;
  tl.shard = 0;
  tl.expert = 0;
  tl.row0 = 0;
  tl.rows = 0;
  tl.half = -1;
  tl.kpart = -1;
  tl.slot = 0;
  tl.m128 = 0;
  if constexpr (MODE == MODE_RS || MODE == MODE_AR || MODE == MODE_AG || MODE == MODE_PARTIAL) {
    // Work items from split_first on are halves of the last round's tiles
    // (two per tile), so that round takes about half a tile's time: K halves
    // (RS / AR with ksplit), else 128-column halves.
    if (t >= p.split_first) {
      const int h = t - p.split_first;
      t = p.split_first + (h >> 1);
      bool ks = false;
      if constexpr (MODE == MODE_RS || MODE == MODE_AR) ks = p.ksplit != 0;
      if (ks) {
        tl.kpart = h & 1;
        tl.slot = h >> 1;
      } else {
        tl.half = h & 1;
      }
    }
  }
  if constexpr (MODE == MODE_GROUPED) {
    // Expert of tile t: the last e with tile_start[e] <= t (binary search).
    const int* ts = tab;                   // tile_start
    const int* rows = tab + p.E + 1;       // expert_rows
    const int* base = tab + 2 * p.E + 1;   // expert_base
    t += ts[p.e_lo];
    int lo = p.e_lo, hi = p.e_hi - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ts[mid] <= t)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int e = lo;
    const int rows_e = rows[e];
    const int tm = (rows_e + TM - 1) / TM;
    const int lt = t - ts[e];
    // m fastest: CTAs running at the same time share the expert's weight slab.
    tl.mt = lt % tm;
    tl.nt = lt / tm;
    tl.expert = e;
    tl.shard = e / p.Eloc;
    tl.row0 = base[e] + tl.mt * TM;
    tl.rows = min(TM, rows_e - tl.mt * TM);
    tl.m128 = (TM == 2 * kBM && tl.rows <= kBM) ? 1 : 0;
  } else if constexpr (MODE == MODE_RS || MODE == MODE_AR) {
    raster(t, p.tiles_m, p.tiles_n, p.group_m, tl.mt, tl.nt);
  } else if constexpr (MODE == MODE_AG) {
    // tiles_m = R * (tiles per shard), tiles_n = R * (tiles per rank)
    int gm, gn;
    raster(t, p.tiles_m, p.tiles_n, p.group_m, gm, gn);
    const int mt_per_shard = p.tiles_m / p.R;
    const int nt_per_rank = p.tiles_n / p.R;
    tl.shard = gm / mt_per_shard;
    tl.mt = gm - tl.shard * mt_per_shard;
    tl.rank = gn / nt_per_rank;
    tl.nt = gn - tl.rank * nt_per_rank;
  } else {
    const int per_rank = p.tiles_m * p.tiles_n;
    tl.rank = t / per_rank;
    raster(t - tl.rank * per_rank, p.tiles_m, p.tiles_n, p.group_m, tl.mt, tl.nt);
  }
  return tl;
}

// ----------------------------------------------------------------- epilogue
// Stores 32 consecutive f32 accumulator columns of one row.
__device__ __forceinline__ void store_row_chunk(void* row_ptr, int col, int N, int out_f32,
                                                const uint32_t (&v)[32]) {
  if (out_f32) {
    float* dst = reinterpret_cast<float*>(row_ptr) + col;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      if (col + 4 * g + 4 <= N)
        ptx::st_global_v4(dst + 4 * g, v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
    }
  } else {
    uint16_t* dst = reinterpret_cast<uint16_t*>(row_ptr) + col;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      if (col + 8 * g + 8 <= N) {
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h)
          w[h] = ptx::pack_bf16x2(__uint_as_float(v[8 * g + 2 * h]),
                                  __uint_as_float(v[8 * g + 2 * h + 1]));
        ptx::st_global_v4(dst + 8 * g, w[0], w[1], w[2], w[3]);
      }
    }
  }
}

// Stores a warp's 32 x 32 block of results as bf16; lane i holds the 32
// accumulator columns of its row i.  Four shuffle rounds per eight rows hand
// each lane one 16-byte piece of another lane's row, so that every store
// instruction writes eight whole 64-byte row pieces (four lanes a row), not
// a 16-byte piece of each of 32 rows.  emit(src, k, piece) stores piece k
// (columns 8k .. 8k+7 of the block) of lane src's row; every lane calls it
// (it may shuffle).
template <class Emit>
__device__ __forceinline__ void store_block_bf16(const uint32_t (&v)[32], int lane, Emit&& emit) {
  uint4 w[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    w[g].x = ptx::pack_bf16x2(__uint_as_float(v[8 * g]), __uint_as_float(v[8 * g + 1]));
    w[g].y = ptx::pack_bf16x2(__uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3]));
    w[g].z = ptx::pack_bf16x2(__uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5]));
    w[g].w = ptx::pack_bf16x2(__uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7]));
  }
  const int k = lane & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int src = 8 * j + (lane >> 2);
    uint4 piece = w[0];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint4 x;
      x.x = __shfl_sync(0xffffffffu, w[kk].x, src);
      x.y = __shfl_sync(0xffffffffu, w[kk].y, src);
      x.z = __shfl_sync(0xffffffffu, w[kk].z, src);
      x.w = __shfl_sync(0xffffffffu, w[kk].w, src);
      if (kk == k) piece = x;
    }
    emit(src, k, piece);
  }
}

__device__ __forceinline__ void red_row_chunk(float* row_ptr, int col, int N,
                                              const uint32_t (&v)[32]) {
  float* dst = row_ptr + col;
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    if (col + 4 * g + 4 <= N)
      ptx::red_add_v4_f32(dst + 4 * g, __uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]),
                          __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3]));
  }
}

template <int MODE, int CG, class P>
__global__ void __launch_bounds__(threads_of<MODE>(), 1) gemm_kernel(const __grid_constant__ P p) {
  using C = Cfg<CG, MODE == MODE_RS || MODE == MODE_AR>;
  constexpr int kStages = C::kStages;
  constexpr int TM = C::kTileM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kStages * C::kBBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* bcast = reinterpret_cast<volatile int*>(tmem_slot + 2);
  int* tab = reinterpret_cast<int*>(tmem_slot + 4);  // grouped mode: expert tables

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr bool kPair = CG == 2;                      // tcgen05 cta_group::2 MMAs
  const uint32_t cta = kPair ? ptx::cluster_ctarank() : 0u;  // 0 = the pair's leader (issues the MMAs)
  constexpr uint32_t lead = 0;                          // cluster rank of the pair's leader
  // Work units (tiles) go round-robin over clusters.
  const int pair = blockIdx.x / CG;
  const int npairs = gridDim.x / CG;

  // Gather mode (MoE without a staged copy): the producer warp fetches the A
  // rows from the source tokens with TMA gather4.
  bool gather = false;
  if constexpr (MODE == MODE_GROUPED) gather = p.gather != 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&tfull[b], 1);
      ptx::mbar_init(&tempty[b], 4 * C::kPairCtas);  // every epilogue warp of the pair
    }
    ptx::mbar_init(mma_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int r = 0; r < p.R; ++r) {
      ptx::tma_prefetch_desc(&p.mapA[r]);
      if constexpr (MODE != MODE_GROUPED) ptx::tma_prefetch_desc(&p.mapB[r]);
    }
  }
  const int k_iters = k_iters_of<MODE>(p);
  // Narrow tile: a half tile, or one whose output columns end in the first
  // half of its 256, so the B loads, the MMA width and the epilogue are halved.
  auto narrow = [&](const Tile& tl) { return tl.half >= 0 || p.N - tl.nt * kBN <= kBN / 2; };
  auto col_base = [&](const Tile& tl) { return tl.nt * kBN + (tl.half > 0 ? kBN / 2 : 0); };
  // The tile's k iterations [it_lo, it_hi).
  auto k_lo = [&](const Tile& tl) {
    if constexpr (MODE == MODE_RS || MODE == MODE_AR) return tl.kpart == 1 ? p.k_half : 0;
    return 0;
  };
  auto k_hi = [&](const Tile& tl) {
    if constexpr (MODE == MODE_RS || MODE == MODE_AR) return tl.kpart == 0 ? p.k_half : k_iters;
    return k_iters;
  };
  if (warp == 1) {
    if constexpr (kPair) {
      ptx::tmem_alloc_pair(tmem_slot, kTmemCols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(tmem_slot, kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  if constexpr (kPair) {
    ptx::cluster_sync_all();  // the peer's barriers exist before anyone signals them
  } else {
    __syncthreads();
  }
  ptx::tc_fence_after();
  // Launched with programmatic stream serialization: the set-up above touches
  // no global memory (the tensor maps are kernel parameters), so it may
  // overlap the previous kernel on the stream; everything below waits for it.
  // The next kernel's launch is released here, or (trigger_late) once this
  // CTA's last accumulator is complete, in the epilogue below.
  ptx::griddep_wait();
  if (!p.trigger_late) ptx::griddep_launch_dependents();
  if constexpr (MODE == MODE_GROUPED) {
    // The tables were written by the dispatch kernels before this launch.
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) tab[i] = __ldcg(p.tile_start + i);
    for (int i = threadIdx.x; i < p.E; i += blockDim.x) {
      tab[p.E + 1 + i] = __ldcg(p.expert_rows + i);
      tab[2 * p.E + 1 + i] = __ldcg(p.expert_base + i);
    }
    __syncthreads();
  }
  const uint32_t tmem_base = *tmem_slot;
  const ptx::Waiter W{abort_flag, p.status, p.timeout_ns};
  const int num_tiles = num_tiles_of<MODE>(p, tab);  // (tables loaded)
  // Phase timing (optional): this CTA's span, its epilogue's busy time and
  // its MMA warp's wait for an accumulator the epilogue still holds.
  unsigned long long* const times = p.phase_ns != nullptr ? p.phase_ns + 4ull * blockIdx.x
                                                          : nullptr;
  const uint64_t t_begin = times != nullptr ? ptx::globaltimer() : 0;

  if (warp == 0 && gather) {
    // ----------------------------------------------- producer, gather mode
    // The whole warp.  Row i of receiving rank d's order is row recv_src[d][i]
    // of the sources' concatenated [R*T, H] token matrix (mapA, a box one row
    // high), so lane q fetches rows 4q..4q+3 of this CTA's 128 A rows with one
    // TMA gather4 per stage: four 128-byte row pieces, swizzled like a tiled
    // box, counted on the same full barrier as the B tile that lane 0 loads.
    if constexpr (MODE == MODE_GROUPED) {
      uint32_t stage = 0, phase = 0;
      uint32_t issued = 0, last_parity = 0;
      bool ok = true;
      const CUtensorMap* ma = &p.mapA[0];
      for (int t = pair; t < num_tiles && ok; t += npairs) {
        const Tile tl = tile_of<MODE, TM>(p, t, tab);
        const int bn_cta = narrow(tl) ? C::kBNcta / 2 : C::kBNcta;
        const int b_col = col_base(tl) + static_cast<int>(cta) * bn_cta;
        const uint32_t stage_bytes = kABytes + static_cast<uint32_t>(bn_cta) * kBK * 2;
        // Source rows of this lane's four A rows; padding rows read row 0 (their
        // results are never stored).
        int y[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int local = static_cast<int>(cta) * (tl.m128 ? kBM / 2 : kBM) + 4 * lane + i;
          y[i] = local < tl.rows ? __ldcg(p.recv_src[tl.shard] + tl.row0 + local) : 0;
        }
        for (int it = 0; it < k_iters; ++it) {
          int good = 1;
          if (lane == 0) good = W.wait(&empty[stage], phase ^ 1u) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, good, 0)) {
            ok = false;
            break;
          }
          const CUtensorMap* mb = &p.mapB[tl.expert];
          uint8_t* a_dst = sA + stage * kABytes + lane * (4 * 128);
          uint8_t* b_dst = sB + stage * C::kBBytes;
          if constexpr (kPair) {
            const uint32_t bar = ptx::mapa(ptx::smem_addr(&full[stage]), lead);
            if (lane == 0) {
              if (cta == 0) ptx::mbar_arrive_expect_tx(&full[stage], 2 * stage_bytes);
              for (int i = 0; i < bn_cta / 64; ++i)
                ptx::tma_load_2d_pair(b_dst + i * kBBoxBytes, mb, bar, b_col + 64 * i, it * kBK);
            }
            __syncwarp();
            ptx::tma_gather4_pair(a_dst, ma, bar, it * kBK, y[0], y[1], y[2], y[3]);
          } else {
            if (lane == 0) {
              ptx::mbar_arrive_expect_tx(&full[stage], stage_bytes);
              for (int i = 0; i < bn_cta / 64; ++i)
                ptx::tma_load_2d(b_dst + i * kBBoxBytes, mb, &full[stage], b_col + 64 * i,
                                 it * kBK);
            }
            __syncwarp();
            ptx::tma_gather4(a_dst, ma, &full[stage], it * kBK, y[0], y[1], y[2], y[3]);
          }
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort_flag && cta == 0 && lane == 0) {
        for (int s = 0; s < kStages; ++s)
          if (issued & (1u << s)) W.drain(&full[s], (last_parity >> s) & 1u, kDrainNs);
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t issued = 0, last_parity = 0;
      bool ok = true;
      for (int t = pair; t < num_tiles && ok; t += npairs) {
        const Tile tl = tile_of<MODE, TM>(p, t, tab);
        int a_row;
        if constexpr (MODE == MODE_GROUPED) {
          a_row = tl.row0;
        } else if constexpr (MODE == MODE_PARTIAL) {
          a_row = p.m_begin + tl.mt * TM;
        } else {
          a_row = tl.mt * TM;
        }
        // this CTA's half of the rows (an M = 128 pair tile: 64 rows each; the
        // 128-row box then also loads 64 rows the MMA does not read)
        a_row += static_cast<int>(cta) * (tl.m128 ? kBM / 2 : kBM);
        const int bn_cta = narrow(tl) ? C::kBNcta / 2 : C::kBNcta;  // B columns of this CTA
        const int b_col = col_base(tl) + static_cast<int>(cta) * bn_cta;
        const uint32_t stage_bytes = kABytes + static_cast<uint32_t>(bn_cta) * kBK * 2;
        if constexpr (MODE == MODE_GROUPED) {
          if (p.stage_copy) {
            // The unit's rows are written by the copy warps (of any CTA):
            // wait for its count, then order the TMA reads after it.
            const int u = tab[tl.expert] / p.tiles_n + tl.mt;
            if (!W.wait_geq(p.ready + u, tl.rows)) {
              ok = false;
              break;
            }
            ptx::fence_proxy_async_global();
          }
        }
        const int it_lo = k_lo(tl), it_hi = k_hi(tl);
        int r = ((tl.rank >= 0) ? tl.rank : 0) + it_lo / p.kb_per_rank;
        int kb = it_lo % p.kb_per_rank;
        for (int it = it_lo; it < it_hi; ++it) {
          if (!W.wait(&empty[stage], phase ^ 1u)) {
            ok = false;
            break;
          }
          const CUtensorMap* ma =
              (MODE == MODE_AG || MODE == MODE_GROUPED) ? &p.mapA[tl.shard] : &p.mapA[r];
          const CUtensorMap* mb = (MODE == MODE_GROUPED) ? &p.mapB[tl.expert] : &p.mapB[r];
          uint8_t* a_dst = sA + stage * kABytes;
          uint8_t* b_dst = sB + stage * C::kBBytes;
          if constexpr (kPair) {
            // Both CTAs' bytes are counted on the leader's full barrier.
            const uint32_t bar = ptx::mapa(ptx::smem_addr(&full[stage]), lead);
            if (cta == 0) ptx::mbar_arrive_expect_tx(&full[stage], 2 * stage_bytes);
            ptx::tma_load_2d_pair(a_dst, ma, bar, kb * kBK, a_row);
            for (int i = 0; i < bn_cta / 64; ++i)
              ptx::tma_load_2d_pair(b_dst + i * kBBoxBytes, mb, bar, b_col + 64 * i, kb * kBK);
          } else {
            ptx::mbar_arrive_expect_tx(&full[stage], stage_bytes);
            ptx::tma_load_2d(a_dst, ma, &full[stage], kb * kBK, a_row);
            for (int i = 0; i < bn_cta / 64; ++i)
              ptx::tma_load_2d(b_dst + i * kBBoxBytes, mb, &full[stage], b_col + 64 * i,
                               kb * kBK);
          }
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
          if (++kb == p.kb_per_rank) {
            kb = 0;
            ++r;  // only MODE_RS / MODE_AR iterate past one rank
          }
        }
      }
      if (*abort_flag && cta == 0) {
        // Loads still in flight write into shared memory: let them land.  (In a
        // pair every load is counted on the leader's barriers, so the leader
        // drains them before the final pair barrier releases its peer.)
        for (int s = 0; s < kStages; ++s)
          if (issued & (1u << s)) W.drain(&full[s], (last_parity >> s) & 1u, kDrainNs);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issue
    if (lane == 0 && cta == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t acc = 0, acc_phase = 0;
      bool any = false, ok = true;
      uint64_t waited = 0;
      for (int t = pair; t < num_tiles && ok; t += npairs) {
        const Tile tm_ = tile_of<MODE, TM>(p, t, tab);
        const uint32_t idesc = tm_.m128 ? (narrow(tm_) ? C::kIdescShortNarrow : C::kIdescShort)
                                        : (narrow(tm_) ? C::kIdescNarrow : C::kIdesc);
        const uint64_t w0 = times != nullptr ? ptx::globaltimer() : 0;
        if (!W.wait(&tempty[acc], acc_phase ^ 1u)) break;
        if (times != nullptr) waited += ptx::globaltimer() - w0;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kBN;
        const int it_lo = k_lo(tm_), it_hi = k_hi(tm_);
        for (int it = it_lo; it < it_hi; ++it) {
          if (!W.wait(&full[stage], phase)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_addr = ptx::smem_addr(sA + stage * kABytes);
          const uint32_t b_addr = ptx::smem_addr(sB + stage * C::kBBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // A: K-major, advance 16 elements (32 B) inside the swizzled row.
            const uint64_t ad = ptx::smem_desc_sw128(a_addr + kk * 32, 16, 1024);
            // B: MN-major, advance 16 k-rows (2 KiB); 64-wide n atoms 8 KiB apart.
            const uint64_t bd = ptx::smem_desc_sw128(b_addr + kk * 2048, kBBoxBytes, 1024);
            if constexpr (kPair)
              ptx::mma_f16_pair(d_tmem, ad, bd, idesc, (it > it_lo || kk > 0) ? 1u : 0u);
            else
              ptx::mma_f16(d_tmem, ad, bd, idesc, (it > it_lo || kk > 0) ? 1u : 0u);
          }
          if constexpr (kPair)
            // Frees the stage in both CTAs of the pair.
            ptx::mma_commit_pair_arrive_ctas(&empty[stage], 0x3);
          else
            ptx::mma_commit(&empty[stage]);
          any = true;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (kPair)
          ptx::mma_commit_pair_arrive_ctas(&tfull[acc], 0x3);
        else
          ptx::mma_commit(&tfull[acc]);
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (any) {
        if constexpr (kPair)
          ptx::mma_commit_pair(mma_done);
        else
          ptx::mma_commit(mma_done);
        W.drain(mma_done, 0, kDrainNs);
      }
      if (times != nullptr) times[2] = waited;
    }
  } else if (warp >= kGemmThreads / 32) {
    // ------------------------------------------- staging copy (grouped mode)
    if constexpr (MODE == MODE_GROUPED) {
      if (p.stage_copy) {
        const int* rows_t = tab + p.E + 1;
        const int* base_t = tab + 2 * p.E + 1;
        int* cstart = tab + 3 * p.E + 1;  // chunks of experts before e, from e_lo
        const int cw = warp - kGemmThreads / 32;
        if (cw == 0 && lane == 0) {
          int acc = 0;
          for (int e = p.e_lo; e < p.e_hi; ++e) {
            cstart[e] = acc;
            acc += (rows_t[e] + kCopyRows - 1) / kCopyRows;
          }
          cstart[p.e_hi] = acc;
        }
        ptx::named_barrier_sync(2, 32 * kCopyWarps);
        const int total = cstart[p.e_hi];
        const int vec = p.K / 8;  // 16-byte vectors per row
        constexpr int kV = 16;    // vectors in flight per lane
        int c = 0;
        if (lane == 0) c = atomicAdd(p.copy_cursor, 1);
        c = __shfl_sync(0xffffffffu, c, 0);
        while (c < total) {
          // The next chunk's claim is in flight while this one is copied.
          int c_next = 0;
          if (lane == 0) c_next = atomicAdd(p.copy_cursor, 1);
          // expert of chunk c: the last e with cstart[e] <= c
          int lo = p.e_lo, hi = p.e_hi - 1;
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (cstart[mid] <= c)
              lo = mid;
            else
              hi = mid - 1;
          }
          const int e = lo;
          const int r0 = (c - cstart[e]) * kCopyRows;  // first row within the expert
          const int n = min(kCopyRows, rows_t[e] - r0);
          const int d = e / p.Eloc;
          // Lane i < n finds row i's source; every lane then prefetches its share
          // of the chunk's source rows into L2 (128-byte lines, the load path's
          // own prefetch), so only the chunk's first row waits for DRAM.
          const uint4* my_src = nullptr;
          if (lane < n) {
            const int src = __ldcg(p.recv_src[d] + base_t[e] + r0 + lane);
            const int s = src / p.T;
            my_src = reinterpret_cast<const uint4*>(p.src_x[s]) +
                     static_cast<long long>(src - s * p.T) * vec;
          }
          for (int i = 1; i < n; ++i) {
            const char* rp = reinterpret_cast<const char*>(
                __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(my_src), i));
            for (int off = lane * 128; off < vec * 16; off += 32 * 128) ptx::prefetch_l2(rp + off);
          }
          for (int i = 0; i < n; ++i) {
            const int row = base_t[e] + r0 + i;
            const uint4* sp = reinterpret_cast<const uint4*>(
                __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(my_src), i));
            uint4* dp = reinterpret_cast<uint4*>(p.stage_x[d]) + static_cast<long long>(row) * vec;
            for (int v0 = 0; v0 < vec; v0 += 32 * kV) {
              uint4 x[kV];
#pragma unroll
              for (int j = 0; j < kV; ++j) {
                const int v = v0 + 32 * j + lane;
                if (v < vec) x[j] = __ldg(sp + v);  // (read-only path: 602.6 against 608.3 us)
              }
#pragma unroll
              for (int j = 0; j < kV; ++j) {
                const int v = v0 + 32 * j + lane;
                if (v < vec) dp[v] = x[j];
              }
            }
          }
          // Publish: every lane's stores, then the unit's count (release).
          ptx::fence_proxy_async_global();
          __syncwarp();
          if (lane == 0) {
            __threadfence();
            atomicAdd(p.ready + tab[e] / p.tiles_n + r0 / TM, n);
          }
          c = __shfl_sync(0xffffffffu, c_next, 0);
        }
      }
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row_in_tile = static_cast<int>(cta) * kBM + q * 32 + lane;  // row of the pair tile
    const uint32_t tempty_leader0 = kPair ? ptx::mapa(ptx::smem_addr(&tempty[0]), lead) : 0u;
    uint32_t acc = 0, acc_phase = 0;
    uint64_t busy = 0;
    int tiles_done = 0;
    for (int t = pair; t < num_tiles; t += npairs) {
      const Tile tl = tile_of<MODE, TM>(p, t, tab);
      const bool failed = !W.wait(&tfull[acc], acc_phase);
      if (p.trigger_late && t + npairs >= num_tiles && warp == 2 && lane == 0)
        ptx::griddep_launch_dependents();
      const uint64_t e0 = times != nullptr ? ptx::globaltimer() : 0;
      if constexpr (MODE == MODE_RS_PUSH || MODE == MODE_AR_PUSH) {
        // The four epilogue warps meet at named barriers below: stop together.
        if (ptx::named_barrier_or(1, 128, failed)) break;
      } else if constexpr (MODE == MODE_RS || MODE == MODE_AR) {
        // (so do they for a K half of the last round)
        if (tl.kpart >= 0) {
          if (ptx::named_barrier_or(1, 128, failed)) break;
        } else if (failed) {
          break;
        }
      } else {
        if (failed) break;
      }
      ptx::tc_fence_after();

      // Destination row(s) for this thread.
      bool row_ok;
      void* rowp = nullptr;
      int64_t grow = 0;  // global row (RS/AR/PUSH)
      const int esz = p.out_f32 ? 4 : 2;
      if constexpr (MODE == MODE_RS || MODE == MODE_RS_PUSH) {
        grow = static_cast<int64_t>(tl.mt) * TM + row_in_tile;
        row_ok = grow < p.M;
        if (row_ok) {
          const int j = static_cast<int>(grow / p.Ms);
          rowp = static_cast<char*>(p.out[j]) + (grow - static_cast<int64_t>(j) * p.Ms) * p.N * esz;
        }
      } else if constexpr (MODE == MODE_AR || MODE == MODE_AR_PUSH) {
        grow = static_cast<int64_t>(tl.mt) * TM + row_in_tile;
        row_ok = grow < p.M;
      } else if constexpr (MODE == MODE_AG) {
        const int64_t local = static_cast<int64_t>(tl.mt) * TM + row_in_tile;
        row_ok = local < p.Ms;
        grow = static_cast<int64_t>(tl.shard) * p.Ms + local;
        if (row_ok) rowp = static_cast<char*>(p.out[tl.rank]) + grow * p.N * esz;
      } else if constexpr (MODE == MODE_GROUPED) {
        // An M = 128 pair tile: this CTA's 64 rows are in TMEM lanes 0-63 for
        // the first half of the tile's columns and again in lanes 64-127 for
        // the second half.
        const int rit = tl.m128 ? static_cast<int>(cta) * (kBM / 2) + ((q * 32 + lane) & 63)
                                : row_in_tile;
        row_ok = rit < tl.rows;
        grow = static_cast<int64_t>(tl.row0) + rit;
        if (row_ok) rowp = static_cast<char*>(p.out[tl.shard]) + grow * p.N * esz;
      } else {  // MODE_PARTIAL
        grow = static_cast<int64_t>(p.m_begin) + static_cast<int64_t>(tl.mt) * TM + row_in_tile;
        row_ok = grow < p.m_end;
        if (row_ok) rowp = static_cast<char*>(p.out[tl.rank]) + grow * p.N * esz;
      }

      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kBN;
      const int ncols = narrow(tl) ? kBN / 2 : kBN;  // the tile's columns
      // accumulator columns written: an M = 128 pair tile holds half of them
      // per lane, lanes 64-127 the second half
      const int cend = tl.m128 ? ncols / 2 : ncols;
      const int col0 = col_base(tl) + ((tl.m128 && q >= 2) ? ncols / 2 : 0);
      auto release_acc = [&]() {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (kPair)
            ptx::mbar_arrive_cluster(tempty_leader0 + acc * 8);
          else
            ptx::mbar_arrive(&tempty[acc]);
        }
      };
      // Stores accumulator columns [c, c + 32) of this thread's row (v).
      auto store_cols = [&](int c, const uint32_t (&v)[32]) {
        const int col = col0 + c;
        if (col >= p.N) return;
        // bf16 results as whole 64-byte row pieces per store: the 8-rank
        // GEMM + AllReduce (eight copies of every tile) went from 2.33 to
        // 2.16 ms, the MoE expert GEMM from 579-584 to 574 us; the RS did
        // not move and the AllGather + GEMM lost 15 us, so it keeps the
        // per-row stores.
        if constexpr (MODE == MODE_AR || MODE == MODE_RS || MODE == MODE_GROUPED) {
          if (!p.out_f32) {
            const int ok = row_ok ? 1 : 0;
            if constexpr (MODE == MODE_AR) {
              store_block_bf16(v, lane, [&](int src, int k, const uint4& x) {
                const long long srow = __shfl_sync(0xffffffffu, static_cast<long long>(grow), src);
                if (__shfl_sync(0xffffffffu, ok, src) && col + 8 * k + 8 <= p.N)
                  for (int r = 0; r < p.R; ++r)
                    ptx::st_global_v4(static_cast<uint16_t*>(p.out[r]) + srow * p.N + col + 8 * k,
                                      x.x, x.y, x.z, x.w);
              });
            } else {
              store_block_bf16(v, lane, [&](int src, int k, const uint4& x) {
                const unsigned long long sp =
                    __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(rowp), src);
                if (__shfl_sync(0xffffffffu, ok, src) && col + 8 * k + 8 <= p.N)
                  ptx::st_global_v4(reinterpret_cast<uint16_t*>(sp) + col + 8 * k, x.x, x.y, x.z,
                                    x.w);
              });
            }
            return;
          }
        }
        if (!row_ok) return;
        if constexpr (MODE == MODE_AR) {
          for (int r = 0; r < p.R; ++r)
            store_row_chunk(static_cast<char*>(p.out[r]) + grow * p.N * esz, col, p.N, p.out_f32, v);
        } else if constexpr (MODE == MODE_RS_PUSH || MODE == MODE_AR_PUSH) {
          float* dst;
          if (p.out_f32) {
            if constexpr (MODE == MODE_RS_PUSH)
              dst = reinterpret_cast<float*>(rowp);
            else
              dst = reinterpret_cast<float*>(p.out[0]) + grow * p.N;  // copied to others later
          } else {
            dst = p.acc_ws + grow * p.N;
          }
          red_row_chunk(dst, col, p.N, v);
        } else {
          store_row_chunk(rowp, col, p.N, p.out_f32, v);
        }
      };

      bool ksplit_tile = false;
      if constexpr (MODE == MODE_RS || MODE == MODE_AR) ksplit_tile = tl.kpart >= 0;
      if (!ksplit_tile) {
#pragma unroll 1
        for (int c = 0; c < cend; c += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(taddr + c, v);
          ptx::tmem_ld_wait();
          // Accumulator fully read: hand it back to the MMA warp early.
          if (c == cend - 32) release_acc();
          store_cols(c, v);
        }
      } else if constexpr (MODE == MODE_RS || MODE == MODE_AR) {
        // A K half of a last-round tile (the only tile of its slot in that
        // round).  Its partner half runs on another slot at the same time.
        const int lrow = q * 32 + lane;  // TMEM lane = row of this CTA's 128
        // The first half's partial of this CTA's 128 rows: block slot * CG + cta.
        const size_t blk = static_cast<size_t>(tl.slot) * CG + cta;
        float* const part = p.split_ws + blk * (static_cast<size_t>(kBM) * kBN) +
                            static_cast<size_t>(lrow) * kBN;
        unsigned long long* flag = p.split_flags + blk;
        if (tl.kpart == 0) {
          // First half: the f32 partial out, then the flag (release).
          float* dst = part;
#pragma unroll 1
          for (int c = 0; c < cend; c += 32) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(taddr + c, v);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int g = 0; g < 8; ++g)
              ptx::st_global_v4(dst + c + 4 * g, v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
          }
          __threadfence();
          ptx::named_barrier_sync(1, 128);
          if (threadIdx.x == 64) ptx::st_release_gpu_u64(flag, p.call_id);
        } else {
          // Second half: wait for the first half's partial (bounded), add it to
          // this accumulator and store the sums.  f32 addition is commutative,
          // so the result does not depend on which half finished first.
          if (threadIdx.x == 64) *bcast = W.wait_eq(flag, p.call_id + p.flag_skew) ? 1 : 0;
          ptx::named_barrier_sync(1, 128);
          if (*bcast) {
            const float* src = part;
#pragma unroll 1
            for (int c = 0; c < cend; c += 32) {
              uint32_t v[32];
              ptx::tmem_ld_32x32b_x32(taddr + c, v);
              ptx::tmem_ld_wait();
#pragma unroll
              for (int g = 0; g < 8; ++g) {
                const float4 f = __ldcg(reinterpret_cast<const float4*>(src + c + 4 * g));
                v[4 * g] = __float_as_uint(__uint_as_float(v[4 * g]) + f.x);
                v[4 * g + 1] = __float_as_uint(__uint_as_float(v[4 * g + 1]) + f.y);
                v[4 * g + 2] = __float_as_uint(__uint_as_float(v[4 * g + 2]) + f.z);
                v[4 * g + 3] = __float_as_uint(__uint_as_float(v[4 * g + 3]) + f.w);
              }
              store_cols(c, v);
            }
          }
          ptx::named_barrier_sync(1, 128);  // (bcast is read before any reuse)
        }
        release_acc();
      }

      if constexpr (MODE == MODE_RS_PUSH || MODE == MODE_AR_PUSH) {
        if (!p.out_f32) {
          // Last of the R contributions to this CTA's rows of the output tile
          // converts them to bf16 (one ticket per tile and CTA of the pair).
          __threadfence();
          ptx::named_barrier_sync(1, 128);
          if (threadIdx.x == 64) {
            const int tid = (tl.mt * p.tiles_n + tl.nt) * CG + static_cast<int>(cta);
            const int prev = atomicAdd(&p.tickets[tid], 1);
            *bcast = (prev == p.R - 1) ? 1 : 0;
            if (prev == p.R - 1) p.tickets[tid] = 0;
          }
          ptx::named_barrier_sync(1, 128);
          if (*bcast) {
            __threadfence();
            if (row_ok) {
              const float* src = p.acc_ws + grow * p.N;
#pragma unroll 1
              for (int c = 0; c < kBN; c += 32) {
                const int col = col0 + c;
                if (col >= p.N) break;
                uint32_t v[32];
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                  if (col + i + 4 <= p.N) {
                    const float4 f = __ldcg(reinterpret_cast<const float4*>(src + col + i));
                    v[i] = __float_as_uint(f.x);
                    v[i + 1] = __float_as_uint(f.y);
                    v[i + 2] = __float_as_uint(f.z);
                    v[i + 3] = __float_as_uint(f.w);
                  }
                }
                if constexpr (MODE == MODE_RS_PUSH) {
                  store_row_chunk(rowp, col, p.N, 0, v);
                } else {
                  for (int r = 0; r < p.R; ++r)
                    store_row_chunk(static_cast<char*>(p.out[r]) + grow * p.N * 2, col, p.N, 0, v);
                }
              }
            }
          }
          ptx::named_barrier_sync(1, 128);
        }
      }
      if (times != nullptr) {
        busy += ptx::globaltimer() - e0;
        ++tiles_done;
      }
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (times != nullptr && warp == 2 && lane == 0) {
      times[1] = busy;
      times[3] = static_cast<unsigned long long>(tiles_done);
    }
  }

  __syncwarp();
  ptx::tc_fence_before();
  if constexpr (kPair) {
    // The leader's MMAs read the peer's shared memory and write the peer's TMEM:
    // neither CTA frees anything before both are done.
    ptx::cluster_sync_all();
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    if constexpr (kPair)
      ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
  if (times != nullptr && threadIdx.x == 0) {
    times[0] = ptx::globaltimer() - t_begin;
    if (kPair && cta != 0) times[2] = 0;  // the peer issues no MMAs
  }
}

template <int MODE, int CG, class P>
cudaError_t launch_mode(const P& p, int grid, cudaStream_t st) {
  auto kern = gemm_kernel<MODE, CG, P>;
  static bool attr_set[64] = {};
  constexpr int kSmem = Cfg<CG, MODE == MODE_RS || MODE == MODE_AR>::kSmem;
  const cudaError_t e = smem_attr_once(attr_set, kern, kSmem);
  if (e != cudaSuccess) return e;
  // CTA pairs launch as clusters of two; a single CTA is its own cluster.
  return launch_pdl(kern, dim3(grid, 1, 1), dim3(threads_of<MODE>(), 1, 1), kSmem, st,
                    CG == 2 ? 2u : 1u, p);
}

template <int CG>
cudaError_t launch_cg(const GemmParams& p, int mode, int grid, cudaStream_t st) {
  switch (mode) {
    case MODE_RS: return launch_mode<MODE_RS, CG, GemmParams>(p, grid, st);
    case MODE_AR: return launch_mode<MODE_AR, CG, GemmParams>(p, grid, st);
    case MODE_PARTIAL: return launch_mode<MODE_PARTIAL, CG, GemmParams>(p, grid, st);
    case MODE_AG: return launch_mode<MODE_AG, CG, GemmParams>(p, grid, st);
    case MODE_RS_PUSH: return launch_mode<MODE_RS_PUSH, CG, GemmParams>(p, grid, st);
    case MODE_AR_PUSH: return launch_mode<MODE_AR_PUSH, CG, GemmParams>(p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

namespace {
template <int CG>
int query_max_clusters() {
  auto kern = gemm_kernel<MODE_RS, CG, GemmParams>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<CG, true>::kSmem) !=
      cudaSuccess)
    return 0;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(std::max(CG, (sms / CG) * CG)), 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg<CG, true>::kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}
}  // namespace

int gemm_max_clusters(int cg) {
  constexpr int kDevs = 16;
  static int cache[kDevs][3] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) dev = 0;
  const int k = cg == 2 ? 2 : 1;
  if (cache[dev][k] == 0) {
    int n = k == 2 ? query_max_clusters<2>() : query_max_clusters<1>();
    // (no answer: one cluster per group of k SMs)
    if (n <= 0) {
      int sms = 0;
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      n = std::max(1, sms / k);
    }
    cache[dev][k] = n;
  }
  return cache[dev][k];
}

cudaError_t launch_gemm(const GemmParams& p, int mode, int cg, int grid, cudaStream_t st) {
  if (cg == 2) return launch_cg<2>(p, mode, grid, st);
  if (cg == 1) return launch_cg<1>(p, mode, grid, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_grouped_gemm(const GroupedParams& p, int cg, int grid, cudaStream_t st) {
  if (cg == 2) return launch_mode<MODE_GROUPED, 2, GroupedParams>(p, grid, st);
  if (cg == 1) return launch_mode<MODE_GROUPED, 1, GroupedParams>(p, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace fcc

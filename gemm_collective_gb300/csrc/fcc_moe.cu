// fcc_moe.cu -- MoE route, dispatch (all-to-all) and grouped expert GEMM (sm_103a).
//
// The MoE Dispatch + GEMM kernel of the mKernel article's fused-kernel list
// (and the GEMM + All-to-All operator for MoE in the SC24 paper's abstract),
// over R virtual ranks in one GPU:
//   1. route_kernel   eight threads per token: top-k experts by logit (ties
//                     to the lower index), softmax gates, and a per-chunk
//                     expert histogram (chunk = 128 tokens of one source rank).
//   2. place_kernel   one CTA per chunk: its per-expert prefix over the
//                     chunks before it (a fixed order) and every expert's
//                     count, each CTA summing the whole histogram itself; then
//                     the stable rank of each of its assignments within its
//                     expert (warp match + popc, then a prefix over the CTA's
//                     warps), i.e. its receive row; writes recv_src.  CTA 0
//                     also writes each expert's first row in its receiving
//                     rank's buffer and the grouped GEMM's tile table, and the
//                     first CTA of each source rank its send counts.  Past 512
//                     chunks the same integers come from two kernels:
//                     offsets_kernel (one CTA per expert scans its histogram;
//                     the last to finish derives the tables) and rank_kernel.
//   4. the all-to-all row movement, into the caller's recv_x or into
//                     workspace.  By default the grouped GEMM's own copy warps
//                     move each (expert, m tile) unit of rows, in tile order,
//                     while its tensor cores work on the units already moved,
//                     and its TMA producer waits for a unit's row count before
//                     loading it.  With FCC_ALGO_UNFUSED (the unfused
//                     baseline) copy_kernel does it first, one warp per token
//                     (each token row read once, written to each of its
//                     receive rows).
//   5. the persistent tcgen05 GEMM in grouped mode: tiles over
//                     (expert, m tile, n tile) from the device tile table.
//                     With FCC_ALGO_FUSED and the sources one [R*T, H]
//                     array, the GEMM's producer warp fetches each A row
//                     straight from its source token with TMA gather4
//                     (recv_src gives the row), so no staged copy precedes
//                     it; a requested recv_x is then written by the copy on
//                     a second stream, beside the GEMM.
// No atomics decide any position, so every index output is bit-exact and
// repeatable; the host never waits for the counts.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "fcc.h"
#include "fcc_internal.h"
#include "fcc_ptx.cuh"

namespace fcc {
namespace {

constexpr int kChunkTok = 128;   // tokens per chunk (one source rank per chunk)
constexpr int kMoeBN = 256;      // grouped GEMM tile width (the GEMM's BN)

struct MoeArgs {
  const void* X[FCC_MAX_RANKS];       // [T, H] bf16 per source rank
  const float* logits[FCC_MAX_RANKS]; // [T, E]
  int32_t* idx[FCC_MAX_RANKS];        // [T, topk]
  float* gate[FCC_MAX_RANKS];         // [T, topk]
  void* recv_x[FCC_MAX_RANKS];        // [cap, H] per receiving rank
  int32_t* recv_src[FCC_MAX_RANKS];   // [cap]
  int R, E, Eloc, topk;
  int T, H;
  int cap;
  int chunks_per_rank;
  int tiles_n;
  int tile_m;             // rows per grouped-GEMM tile
  int32_t* chunk_counts;  // [E][nchunks]
  int32_t* chunk_off;     // [E][nchunks]
  int32_t* expert_counts; // [E] (caller's output)
  int32_t* send_counts;   // [R][R] (caller's output)
  int32_t* expert_base;   // [E]
  int32_t* expert_rows;   // [E], clamped to cap
  int32_t* tile_start;    // [E + 1]
  int32_t* row_of;        // [R*T*topk]: receive row of each assignment, -1 if dropped
  int32_t* ready;         // in-kernel staging: rows copied per (expert, m tile) unit
  int32_t* copy_cursor;   // in-kernel staging: next chunk to claim
  int32_t* offsets_ticket;  // CTAs of offsets_kernel done (the router zeroes it)
  // Copy-engine dispatch: per source rank s a send buffer of its kept rows in
  // (expert, token, slot) order; srcoff[s][e] = assignments to e from the
  // sources before s (srcoff[R][e] = all of e's); send_base[s][e] = the first
  // send row of (s, e); plan[s][e] = {send row, receive row, rows} of the
  // (s, e) run, which is contiguous on both sides.
  void* send[FCC_MAX_RANKS];
  int32_t* ce_srcoff;     // [R + 1][E]
  int32_t* ce_send_base;  // [R][E]
  int32_t* ce_plan;       // [R][E][3]
  int* status;
};

// Grid: one CTA per chunk of 128 tokens (of one source rank), eight threads
// per token (1024 threads; at most 32 registers, so two CTAs fit an SM and
// the 256 chunks of 8 x 4096 tokens run in one wave: 7.4-7.8 us, against
// 9.0-9.2 us with four threads a token).  Thread q of a token scans its
// eighth of the E logits for its own top two (a strictly larger logit
// replaces, so an equal logit keeps the lower expert index); the eight
// partial lists are merged by xor shuffles (the same total order: larger
// logit, then lower index), so all eight hold the token's top two and its
// largest logit m.  The softmax denominator sum_e exp(l_e - m) is summed per
// thread in expert order, then over the eight threads in a fixed shuffle
// tree.  The per-chunk expert histogram is counted in shared memory and
// stored expert-major (chunk_counts[e][chunk]) for the scan.
constexpr int kRouteSub = 8;  // threads per token

struct Cand {
  float v;
  int i;
};

// a ranks before b: larger logit, or equal logit and lower expert index.
__device__ __forceinline__ bool better(const Cand& a, const Cand& b) {
  return a.v > b.v || (a.v == b.v && a.i < b.i);
}

__global__ void __launch_bounds__(kChunkTok * kRouteSub, 2) route_kernel(const MoeArgs a) {
  ptx::griddep_wait();  // launched with programmatic stream serialization
  ptx::griddep_launch_dependents();
  __shared__ int hist[FCC_MAX_EXPERTS];
  const int chunk = blockIdx.x;
  const int s = chunk / a.chunks_per_rank;
  const int t0 = (chunk - s * a.chunks_per_rank) * kChunkTok;
  const int E = a.E;
  if (chunk == 0 && threadIdx.x == 0) *a.offsets_ticket = 0;  // (read after this grid ends)
  if (threadIdx.x < FCC_MAX_EXPERTS) hist[threadIdx.x] = 0;
  __syncthreads();
  const int t = t0 + static_cast<int>(threadIdx.x) / kRouteSub;
  const int q = threadIdx.x % kRouteSub;
  const bool live = t < a.T;  // (whole 8-thread groups: the shuffles stay uniform)
  const int per = (E + kRouteSub - 1) / kRouteSub;
  const int e_lo = min(E, q * per), e_hi = min(E, e_lo + per);
  const float* row = a.logits[s] + static_cast<long long>(live ? t : t0) * E;
  const float neg_inf = __int_as_float(0xff800000);
  Cand c0{neg_inf, E}, c1{neg_inf, E};  // (index E: no expert; loses every comparison)
  float x[FCC_MAX_EXPERTS / kRouteSub];
#pragma unroll
  for (int k = 0; k < FCC_MAX_EXPERTS / kRouteSub; ++k)
    x[k] = (live && e_lo + k < e_hi) ? __ldcs(row + e_lo + k) : neg_inf;
#pragma unroll
  for (int k = 0; k < FCC_MAX_EXPERTS / kRouteSub; ++k) {
    if (e_lo + k >= e_hi) break;
    const Cand c{x[k], e_lo + k};
    if (better(c, c0)) {
      c1 = c0;
      c0 = c;
    } else if (better(c, c1)) {
      c1 = c;
    }
  }
#pragma unroll
  for (int off = kRouteSub / 2; off > 0; off >>= 1) {
    Cand b0, b1;
    b0.v = __shfl_xor_sync(0xffffffffu, c0.v, off);
    b0.i = __shfl_xor_sync(0xffffffffu, c0.i, off);
    b1.v = __shfl_xor_sync(0xffffffffu, c1.v, off);
    b1.i = __shfl_xor_sync(0xffffffffu, c1.i, off);
    if (better(b0, c0)) {
      c1 = better(b1, c0) ? b1 : c0;
      c0 = b0;
    } else if (better(b0, c1)) {
      c1 = b0;
    }
  }
  const float m = c0.v;
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < FCC_MAX_EXPERTS / kRouteSub; ++k)
    if (e_lo + k < e_hi) sum += expf(x[k] - m);
#pragma unroll
  for (int off = kRouteSub / 2; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (live && q == 0) {
    const long long o = static_cast<long long>(t) * a.topk;
    a.idx[s][o] = c0.i;
    a.gate[s][o] = 1.0f / sum;  // exp(m - m) = 1
    atomicAdd(&hist[c0.i], 1);  // a count: order does not matter
    if (a.topk > 1) {
      a.idx[s][o + 1] = c1.i;
      a.gate[s][o + 1] = expf(c1.v - m) / sum;
      atomicAdd(&hist[c1.i], 1);
    }
  }
  __syncthreads();
  if (threadIdx.x < E)
    a.chunk_counts[static_cast<long long>(threadIdx.x) * a.R * a.chunks_per_rank + chunk] =
        hist[threadIdx.x];
}

// The grouped GEMM's tile table from the experts' kept rows (warp 0: the
// exclusive prefix of the experts' tiles, two experts a lane), then the
// in-kernel staging counters' reset (the whole CTA), which start at zero for
// every call.  rows[] is in shared memory, written before a barrier.
__device__ __forceinline__ void write_tiles(const MoeArgs& a, const int* rows, int* units_s) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    const int ea = 2 * lane, eb = 2 * lane + 1;
    const int ta = ea < a.E ? ((rows[ea] + a.tile_m - 1) / a.tile_m) * a.tiles_n : 0;
    const int tb = eb < a.E ? ((rows[eb] + a.tile_m - 1) / a.tile_m) * a.tiles_n : 0;
    int incl = ta + tb;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    const int excl = incl - ta - tb;
    if (ea < a.E) a.tile_start[ea] = excl;
    if (eb < a.E) a.tile_start[eb] = excl + ta;
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) {
      a.tile_start[a.E] = total;
      *units_s = total / a.tiles_n;  // (m tile units in all)
    }
  }
  if (a.ready != nullptr) {
    __syncthreads();
    const int units = *units_s;
    for (int u = threadIdx.x; u < units; u += blockDim.x) a.ready[u] = 0;
    if (threadIdx.x == 0) *a.copy_cursor = 0;
  }
}

// One CTA of 256 threads per expert e after the router: the exclusive prefix
// of e's histogram over the chunks, in chunk order (source rank, then token),
// so chunk_off[e][c] is the number of assignments to e that precede chunk c
// in (s, t, slot) order (integer sums in a fixed order of warp shuffles);
// and e's count.  The last CTA to finish (a ticket the router zeroed) then
// computes each expert's first row in its receiving rank's buffer and its
// kept rows (capacity), the send counts and the grouped GEMM's tile table.
__global__ void __launch_bounds__(256) offsets_kernel(const MoeArgs a) {
  ptx::griddep_wait();  // launched with programmatic stream serialization
  ptx::griddep_launch_dependents();
  __shared__ int wsum[8];
  __shared__ int last_s;
  __shared__ int counts[FCC_MAX_EXPERTS];
  __shared__ int rows[FCC_MAX_EXPERTS];
  __shared__ int srcoff[FCC_MAX_RANKS + 1][FCC_MAX_EXPERTS];  // prefix at each source's first chunk
  __shared__ int units_s;
  const int nchunks = a.R * a.chunks_per_rank;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  {
    const int e = blockIdx.x;
    const int32_t* cc = a.chunk_counts + static_cast<long long>(e) * nchunks;  // expert-major
    int carry = 0;
    for (int c0 = 0; c0 < nchunks; c0 += 256) {
      const int c = c0 + static_cast<int>(threadIdx.x);
      const int v = c < nchunks ? __ldcg(cc + c) : 0;
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      if (lane == 31) wsum[warp] = incl;
      __syncthreads();
      int before = carry + incl - v, total = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        if (w < warp) before += wsum[w];
        total += wsum[w];
      }
      if (c < nchunks) a.chunk_off[static_cast<long long>(e) * nchunks + c] = before;
      carry += total;
      __syncthreads();
    }
    if (threadIdx.x == 0) a.expert_counts[e] = carry;
  }
  // The last CTA to arrive sees every expert's prefix and count.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last_s = atomicAdd(a.offsets_ticket, 1) == a.E - 1 ? 1 : 0;
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  for (int i = threadIdx.x; i < a.E; i += blockDim.x) {
    counts[i] = __ldcg(a.expert_counts + i);
    srcoff[a.R][i] = counts[i];
  }
  for (int i = threadIdx.x; i < a.R * a.E; i += blockDim.x) {
    const int s = i / a.E, f = i - (i / a.E) * a.E;
    srcoff[s][f] = __ldcg(a.chunk_off + static_cast<long long>(f) * nchunks + s * a.chunks_per_rank);
  }
  __syncthreads();
  const int e = threadIdx.x;
  if (e < a.E) {
    const int d = e / a.Eloc;
    long long base = 0;
    for (int f = d * a.Eloc; f < e; ++f) base += counts[f];
    const long long room = static_cast<long long>(a.cap) - base;
    const int kept = static_cast<int>(max(0ll, min(static_cast<long long>(counts[e]), room)));
    a.expert_base[e] = static_cast<int>(min(base, static_cast<long long>(a.cap)));
    a.expert_rows[e] = kept;
    rows[e] = kept;
    if (e == (d + 1) * a.Eloc - 1 && base + counts[e] > a.cap && a.status != nullptr)
      atomicCAS(a.status, 0, FCC_ERR_CAPACITY);
  }
  // send_counts[s][d]: assignments from source rank s to the experts of rank d,
  // read off the prefix at the boundaries of s's chunks.
  if (e < a.R * a.R) {
    const int s = e / a.R, d = e - (e / a.R) * a.R;
    int sum = 0;
    for (int f = d * a.Eloc; f < (d + 1) * a.Eloc; ++f) sum += srcoff[s + 1][f] - srcoff[s][f];
    a.send_counts[e] = sum;
  }
  __syncthreads();
  write_tiles(a, rows, &units_s);
}

// The expert of assignment threadIdx.x of a chunk (token t0 + i/topk, slot
// i%topk), or -1 past the chunk's assignments (at most 256: topk <= 2).
__device__ __forceinline__ int chunk_expert(const MoeArgs& a, int chunk) {
  const int s = chunk / a.chunks_per_rank;
  const int t0 = (chunk - s * a.chunks_per_rank) * kChunkTok;
  const int n_assign = (min(a.T, t0 + kChunkTok) - t0) * a.topk;
  const int i = threadIdx.x;
  return i < n_assign ? a.idx[s][static_cast<long long>(t0) * a.topk + i] : -1;
}

// Receive rows of one chunk's assignments.  Thread i < 256 of the CTA holds
// assignment i of the chunk, whose expert e (chunk_expert) the caller
// loaded, so warps 0-7 hold consecutive runs in (t, slot) order.  pre[e] =
// assignments to e in earlier chunks, base[e] = e's first row in its
// receiving rank's buffer, rows[e] = e's kept rows; all three in shared
// memory, written before the call (its first barrier orders them).  The rank
// within the chunk is the warp-match rank plus a prefix over the lower
// warps, so each expert's rows follow (s, t, slot) order.
__device__ __forceinline__ void rank_chunk(const MoeArgs& a, int chunk, int e, const int* pre,
                                           const int* base, const int* rows,
                                           int (*cnt)[FCC_MAX_EXPERTS]) {
  const int s = chunk / a.chunks_per_rank;
  const int t0 = (chunk - s * a.chunks_per_rank) * kChunkTok;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 8 * FCC_MAX_EXPERTS; i += blockDim.x) (&cnt[0][0])[i] = 0;
  __syncthreads();
  const int i = threadIdx.x;
  const bool valid = e >= 0;
  int rank_in_warp = 0;
  if (warp < 8) {
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    rank_in_warp = __popc(peers & ((1u << lane) - 1u));
    if (valid && rank_in_warp == 0) cnt[warp][e] = __popc(peers);
  }
  __syncthreads();
  // exclusive prefix over the warps, per expert
  if (threadIdx.x < a.E) {
    int run = 0;
    for (int w = 0; w < 8; ++w) {
      const int c = cnt[w][threadIdx.x];
      cnt[w][threadIdx.x] = run;
      run += c;
    }
  }
  __syncthreads();
  if (valid) {
    const int pos = pre[e] + cnt[warp][e] + rank_in_warp;
    const int d = e / a.Eloc;
    const int row = base[e] + pos;
    const bool kept = pos < rows[e];
    const long long gidx = (static_cast<long long>(s) * a.T + t0) * a.topk + i;
    a.row_of[gidx] = kept ? row : -1;
    if (kept) a.recv_src[d][row] = s * a.T + t0 + i / a.topk;
  }
}

// One CTA of 256 threads per chunk, after offsets_kernel.
__global__ void __launch_bounds__(256) rank_kernel(const MoeArgs a) {
  ptx::griddep_wait();  // launched with programmatic stream serialization
  ptx::griddep_launch_dependents();
  __shared__ int cnt[8][FCC_MAX_EXPERTS];
  __shared__ int pre[FCC_MAX_EXPERTS], base[FCC_MAX_EXPERTS], rows[FCC_MAX_EXPERTS];
  const int chunk = blockIdx.x;
  const long long nchunks = static_cast<long long>(a.R) * a.chunks_per_rank;
  const int my_e = chunk_expert(a, chunk);
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
    pre[e] = a.chunk_off[e * nchunks + chunk];
    base[e] = a.expert_base[e];
    rows[e] = a.expert_rows[e];
  }
  rank_chunk(a, chunk, my_e, pre, base, rows, cnt);
}

// Offsets and ranks in one kernel after the router, for up to
// kPlaceMaxChunks chunks: one CTA of 1024 threads per chunk.  Every CTA sums
// the whole chunk histogram itself (16 threads an expert, then a fixed xor
// tree), which gives its chunk's per-expert prefix and every expert's total,
// so no CTA waits for another; the chunk's ranks follow as in rank_kernel.
// CTA 0 also writes the experts' counts, first rows and kept rows, the tile
// table and the staging counters' reset, and the first CTA of each source
// rank s writes row s of send_counts.  The same integers as offsets_kernel +
// rank_kernel, in fewer launches; the histogram is read once per chunk, so
// past the limit the two-kernel form is used.
constexpr int kPlaceMaxChunks = 512;
constexpr int kPlaceSub = 16;  // threads per expert

__global__ void __launch_bounds__(FCC_MAX_EXPERTS * kPlaceSub) place_kernel(const MoeArgs a) {
  ptx::griddep_wait();  // launched with programmatic stream serialization
  ptx::griddep_launch_dependents();
  __shared__ int cnt[8][FCC_MAX_EXPERTS];
  __shared__ int pre[FCC_MAX_EXPERTS], tot[FCC_MAX_EXPERTS], src_sum[FCC_MAX_EXPERTS];
  __shared__ int base[FCC_MAX_EXPERTS], rows[FCC_MAX_EXPERTS];
  __shared__ int units_s;
  const int nchunks = a.R * a.chunks_per_rank;
  const int chunk = blockIdx.x;
  const int s = chunk / a.chunks_per_rank;
  const int s_lo = s * a.chunks_per_rank, s_hi = s_lo + a.chunks_per_rank;
  const int my_e = chunk_expert(a, chunk);  // (in flight during the histogram pass)
  const int e = threadIdx.x / kPlaceSub, j = threadIdx.x % kPlaceSub;
  int p = 0, n = 0, ns = 0;  // before this chunk, all chunks, chunks of source s
  if (e < a.E) {
    const int32_t* cc = a.chunk_counts + static_cast<long long>(e) * nchunks;  // expert-major
    for (int c = j; c < nchunks; c += kPlaceSub) {
      const int v = __ldcg(cc + c);
      n += v;
      if (c < chunk) p += v;
      if (c >= s_lo && c < s_hi) ns += v;
    }
  }
#pragma unroll
  for (int off = kPlaceSub / 2; off > 0; off >>= 1) {
    p += __shfl_xor_sync(0xffffffffu, p, off);
    n += __shfl_xor_sync(0xffffffffu, n, off);
    ns += __shfl_xor_sync(0xffffffffu, ns, off);
  }
  if (j == 0 && e < a.E) {
    pre[e] = p;
    tot[e] = n;
    src_sum[e] = ns;
  }
  __syncthreads();
  if (threadIdx.x < a.E) {
    const int f = threadIdx.x, d = f / a.Eloc;
    long long b = 0;
    for (int g = d * a.Eloc; g < f; ++g) b += tot[g];
    const long long room = static_cast<long long>(a.cap) - b;
    const int kept = static_cast<int>(max(0ll, min(static_cast<long long>(tot[f]), room)));
    base[f] = static_cast<int>(min(b, static_cast<long long>(a.cap)));
    rows[f] = kept;
    a.chunk_off[static_cast<long long>(f) * nchunks + chunk] = pre[f];
    if (chunk == 0) {
      a.expert_counts[f] = tot[f];
      a.expert_base[f] = base[f];
      a.expert_rows[f] = kept;
      if (f == (d + 1) * a.Eloc - 1 && b + tot[f] > a.cap && a.status != nullptr)
        atomicCAS(a.status, 0, FCC_ERR_CAPACITY);
    }
  }
  if (chunk == s_lo && threadIdx.x < a.R) {
    // send_counts[s][d]: assignments from source rank s to the experts of rank d
    const int d = threadIdx.x;
    int sum = 0;
    for (int f = d * a.Eloc; f < (d + 1) * a.Eloc; ++f) sum += src_sum[f];
    a.send_counts[s * a.R + d] = sum;
  }
  __syncthreads();
  if (chunk == 0) write_tiles(a, rows, &units_s);
  rank_chunk(a, chunk, my_e, pre, base, rows, cnt);
}

// One warp per token: read the token's row once (16-byte loads) and write it to
// each of its receive rows.
__global__ void __launch_bounds__(256) copy_kernel(const MoeArgs a) {
  ptx::griddep_wait();  // launched with programmatic stream serialization
  ptx::griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const long long ntok = static_cast<long long>(a.R) * a.T;
  const int vec = a.H / 8;  // uint4 per row
  for (long long g = blockIdx.x * static_cast<long long>(blockDim.x >> 5) + (threadIdx.x >> 5);
       g < ntok; g += warps) {
    const int s = static_cast<int>(g / a.T);
    const int t = static_cast<int>(g - static_cast<long long>(s) * a.T);
    int row = -1, d = 0;
    if (lane < a.topk) {
      row = a.row_of[g * a.topk + lane];
      d = a.idx[s][static_cast<long long>(t) * a.topk + lane] / a.Eloc;
    }
    const int row0 = __shfl_sync(0xffffffffu, row, 0);
    const int d0 = __shfl_sync(0xffffffffu, d, 0);
    const int row1 = __shfl_sync(0xffffffffu, row, 1);
    const int d1 = __shfl_sync(0xffffffffu, d, 1);
    const uint4* src = reinterpret_cast<const uint4*>(a.X[s]) + static_cast<long long>(t) * vec;
    uint4* dst0 = row0 >= 0 ? reinterpret_cast<uint4*>(a.recv_x[d0]) +
                                  static_cast<long long>(row0) * vec
                            : nullptr;
    uint4* dst1 = (a.topk > 1 && row1 >= 0) ? reinterpret_cast<uint4*>(a.recv_x[d1]) +
                                                  static_cast<long long>(row1) * vec
                                            : nullptr;
    for (int v = lane; v < vec; v += 32) {
      const uint4 x = __ldcs(src + v);
      if (dst0 != nullptr) dst0[v] = x;
      if (dst1 != nullptr) dst1[v] = x;
    }
  }
}

// Rows of experts [e_lo, e_hi) of their receiving ranks' orders, one warp per
// receive row: row i of expert e on rank d = e / Eloc is source row
// recv_src[d][i] (= s*T + t).  The InterDecom baseline moves one expert range
// per chunk with it, on a side stream ahead of that range's GEMM.
__global__ void __launch_bounds__(256) copy_expert_rows_kernel(const MoeArgs a, int e_lo,
                                                               int e_hi) {
  __shared__ int pre[FCC_MAX_EXPERTS + 1];  // rows of the range's experts before e
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int e = e_lo; e < e_hi; ++e) {
      pre[e - e_lo] = acc;
      acc += a.expert_rows[e];
    }
    pre[e_hi - e_lo] = acc;
  }
  __syncthreads();
  const int total = pre[e_hi - e_lo];
  const int lane = threadIdx.x & 31;
  const int vec = a.H / 8;  // uint4 per row
  constexpr int kV = 8;     // vectors in flight per lane
  const int warps = gridDim.x * (blockDim.x >> 5);
  for (int g = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); g < total; g += warps) {
    int lo = 0, hi = e_hi - e_lo - 1;  // the last expert whose first row is <= g
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= g)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int e = e_lo + lo;
    const int d = e / a.Eloc;
    const int row = a.expert_base[e] + (g - pre[lo]);
    const int src = a.recv_src[d][row];
    const int s = src / a.T;
    const int t = src - s * a.T;
    const uint4* sp = reinterpret_cast<const uint4*>(a.X[s]) + static_cast<long long>(t) * vec;
    uint4* dp = reinterpret_cast<uint4*>(a.recv_x[d]) + static_cast<long long>(row) * vec;
    for (int v0 = 0; v0 < vec; v0 += 32 * kV) {
      uint4 x[kV];
#pragma unroll
      for (int j = 0; j < kV; ++j) {
        const int v = v0 + 32 * j + lane;
        if (v < vec) x[j] = __ldcg(sp + v);
      }
#pragma unroll
      for (int j = 0; j < kV; ++j) {
        const int v = v0 + 32 * j + lane;
        if (v < vec) dp[v] = x[j];
      }
    }
  }
}

// Copy-engine dispatch, step 1 (one CTA of 64 threads, after offsets_kernel):
// the (source rank, expert) runs.  Source s's assignments to expert e are, in
// both orders, one contiguous run: rows srcoff[s][e] .. srcoff[s + 1][e] of
// e's receive rows (receive order is (expert, s, t, slot)), and, packed on
// the sending side in (expert, t, slot) order, rows send_base[s][e] on of
// s's send buffer.  Only the kept rows (within the receive capacity) are
// packed and moved; they are a prefix of each run.
__global__ void __launch_bounds__(64) ce_plan_kernel(const MoeArgs a) {
  ptx::griddep_wait();  // launched with programmatic stream serialization
  ptx::griddep_launch_dependents();
  __shared__ int off[FCC_MAX_RANKS + 1][FCC_MAX_EXPERTS];
  __shared__ int kept[FCC_MAX_RANKS][FCC_MAX_EXPERTS];
  const int e = threadIdx.x;
  if (e < a.E) {
    for (int s = 0; s <= a.R; ++s) {
      off[s][e] = s < a.R ? a.chunk_off[static_cast<long long>(e) * a.R * a.chunks_per_rank +
                                        s * a.chunks_per_rank]
                          : a.expert_counts[e];
      a.ce_srcoff[s * a.E + e] = off[s][e];
    }
    for (int s = 0; s < a.R; ++s)
      kept[s][e] = max(0, min(off[s + 1][e] - off[s][e], a.expert_rows[e] - off[s][e]));
  }
  __syncthreads();
  if (e < a.R) {
    int acc = 0;
    for (int f = 0; f < a.E; ++f) {
      a.ce_send_base[e * a.E + f] = acc;
      int32_t* pl = a.ce_plan + 3 * (e * a.E + f);
      pl[0] = acc;                            // first send row
      pl[1] = a.expert_base[f] + off[e][f];   // first receive row on rank f / Eloc
      pl[2] = kept[e][f];                     // rows
      acc += kept[e][f];
    }
  }
}

// Copy-engine dispatch, step 2 (after rank_kernel): each source rank packs its
// kept rows into its own send buffer (a copy inside the rank; nothing crosses
// ranks here), one warp per token, the token's row read once.
__global__ void __launch_bounds__(256) ce_pack_kernel(const MoeArgs a) {
  ptx::griddep_wait();  // launched with programmatic stream serialization
  ptx::griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const long long ntok = static_cast<long long>(a.R) * a.T;
  const int vec = a.H / 8;
  for (long long g = blockIdx.x * static_cast<long long>(blockDim.x >> 5) + (threadIdx.x >> 5);
       g < ntok; g += warps) {
    const int s = static_cast<int>(g / a.T);
    const int t = static_cast<int>(g - static_cast<long long>(s) * a.T);
    int srow = -1;
    if (lane < a.topk) {
      const int row = a.row_of[g * a.topk + lane];
      if (row >= 0) {
        const int e = a.idx[s][static_cast<long long>(t) * a.topk + lane];
        // rank of the assignment within its (s, e) run
        const int k = row - a.expert_base[e] - a.ce_srcoff[s * a.E + e];
        srow = a.ce_send_base[s * a.E + e] + k;
      }
    }
    const int r0 = __shfl_sync(0xffffffffu, srow, 0);
    const int r1 = __shfl_sync(0xffffffffu, srow, 1);
    const uint4* src = reinterpret_cast<const uint4*>(a.X[s]) + static_cast<long long>(t) * vec;
    uint4* dst0 = r0 >= 0 ? reinterpret_cast<uint4*>(a.send[s]) + static_cast<long long>(r0) * vec
                          : nullptr;
    uint4* dst1 = (a.topk > 1 && r1 >= 0)
                      ? reinterpret_cast<uint4*>(a.send[s]) + static_cast<long long>(r1) * vec
                      : nullptr;
    for (int v = lane; v < vec; v += 32) {
      const uint4 x = __ldcs(src + v);
      if (dst0 != nullptr) dst0[v] = x;
      if (dst1 != nullptr) dst1[v] = x;
    }
  }
}

struct MoePlan {
  int chunks_per_rank = 0;
  int nchunks = 0;
  size_t off_stage = 0;  // staged rows when the caller passes no recv_x ([R][cap][H] bf16)
  size_t off_chunk_counts = 0, off_chunk_off = 0, off_base = 0, off_rows = 0, off_tiles = 0,
         off_row_of = 0, off_ready = 0, off_cursor = 0, off_ticket = 0, total = 0;
  // copy-engine dispatch: tables and the send buffers ([R][T*topk][H] bf16)
  size_t off_ce_srcoff = 0, off_ce_send_base = 0, off_ce_plan = 0, off_send = 0;
};

size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// The expert GEMM gathers its rows from the sources (no staged copy on its
// path) when FCC_ALGO_FUSED asks for it and the sources are one [R*T, H]
// array (X[s] = X[0] + s*T*H elements).  TMA gather4 moves 4 rows of 128 bytes
// per request, and on sm_103a its request rate, not memory, bounds that GEMM
// (about 2.7x the staged form on the 8 x 4096-token, 64-expert workload), so
// the default stages the rows with one streaming copy and loads whole tiles.
bool moe_gathers(const fcc_opts* o, int R, const void* const* X, int64_t T, int64_t H) {
  if (o == nullptr || o->algo != FCC_ALGO_FUSED) return false;
  const char* x0 = static_cast<const char*>(X[0]);
  for (int s = 1; s < R; ++s)
    if (static_cast<const char*>(X[s]) != x0 + static_cast<int64_t>(s) * T * H * 2) return false;
  return true;
}

MoePlan moe_plan(int R, int64_t T, int E, int topk, int64_t H = 0, int64_t cap = 0,
                 bool stage_in_workspace = false, bool ce = false) {
  MoePlan p;
  p.chunks_per_rank = static_cast<int>((T + kChunkTok - 1) / kChunkTok);
  p.nchunks = R * p.chunks_per_rank;
  size_t off = 0;
  p.off_chunk_counts = off;
  off += up256(static_cast<size_t>(p.nchunks) * E * 4);
  p.off_chunk_off = off;
  off += up256(static_cast<size_t>(p.nchunks) * E * 4);
  p.off_base = off;
  off += up256(static_cast<size_t>(E) * 4);
  p.off_rows = off;
  off += up256(static_cast<size_t>(E) * 4);
  p.off_tiles = off;
  off += up256(static_cast<size_t>(E + 1) * 4);
  p.off_row_of = off;
  off += up256(static_cast<size_t>(R) * T * topk * 4);
  // (expert, m tile) units: at most one partial tile per expert beyond
  // assignments / 128 full ones, and the rows are at most the assignments.
  p.off_ready = off;
  off += up256((static_cast<size_t>(R) * T * topk / 128 + E + 1) * 4);
  p.off_cursor = off;
  off += 256;
  p.off_ticket = off;
  off += 256;
  p.off_ce_srcoff = off;
  off += up256(static_cast<size_t>(R + 1) * E * 4);
  p.off_ce_send_base = off;
  off += up256(static_cast<size_t>(R) * E * 4);
  p.off_ce_plan = off;
  off += up256(static_cast<size_t>(R) * E * 3 * 4);
  p.off_stage = off;
  if (stage_in_workspace) off += up256(static_cast<size_t>(R) * cap * H * 2);
  p.off_send = off;
  if (ce) off += up256(static_cast<size_t>(R) * T * topk * H * 2);
  p.total = off;
  return p;
}

// Default model constants for the InterDecom chunk count (as for the GEMMs):
// sustained tensor rate, copy bandwidth and per-chunk overhead on a GB300.
// G = the expert GEMMs, X = the row copy (each receive row read and written);
// chunks are expert ranges, at most E.
int moe_model_chunks(int R, int64_t T, int64_t H, int64_t F, int E, int topk) {
  const double rows = static_cast<double>(R) * T * topk;
  const double G = 2.0 * rows * H * F / 1.6e15;
  const double X = 2.0 * rows * H * 2 / 6.0e12;
  return fcc_interdecom_chunks(G, X, 6.0e-6, E);
}

bool al(const void* p, uintptr_t a) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

fcc_status check_moe(int R, const void* const* X, const float* const* logits,
                     const void* const* W, int64_t T, int64_t H, int64_t F, int E, int topk,
                     void* const* recv_x, void* const* recv_y, int64_t cap,
                     int32_t* const* topk_idx, float* const* topk_gate, int32_t* expert_counts,
                     int32_t* send_counts, int32_t* const* recv_src, fcc_dtype in,
                     fcc_dtype out_dtype, const fcc_opts* opts) {
  if (R < 1 || R > FCC_MAX_RANKS || E < R || E > FCC_MAX_EXPERTS || E % R != 0)
    return FCC_ERR_INVALID;
  if (topk < 1 || topk > 2 || topk > E) return FCC_ERR_INVALID;
  if (T < 1 || H < 8 || F < 8 || H % 8 != 0 || F % 8 != 0 || cap < 1) return FCC_ERR_INVALID;
  if (T > (1ll << 28) || H > (1ll << 30) || F > (1ll << 30) || cap > (1ll << 30) ||
      static_cast<int64_t>(R) * T * topk > (1ll << 30))
    return FCC_ERR_INVALID;
  if (X == nullptr || logits == nullptr || W == nullptr || recv_y == nullptr ||
      topk_idx == nullptr || topk_gate == nullptr || recv_src == nullptr ||
      !al(expert_counts, 4) || !al(send_counts, 4))
    return FCC_ERR_INVALID;
  for (int r = 0; r < R; ++r) {
    if (!al(X[r], 16) || !al(logits[r], 4) || !al(recv_y[r], 16) || !al(topk_idx[r], 4) ||
        !al(topk_gate[r], 4) || !al(recv_src[r], 4))
      return FCC_ERR_INVALID;
    if (recv_x != nullptr && !al(recv_x[r], 16)) return FCC_ERR_INVALID;
  }
  for (int e = 0; e < E; ++e)
    if (!al(W[e], 16)) return FCC_ERR_INVALID;
  if (in != FCC_BF16 && in != FCC_F16 && in != FCC_F32) return FCC_ERR_INVALID;
  if (in != FCC_BF16) return FCC_ERR_UNSUPPORTED;
  if (out_dtype != FCC_BF16 && out_dtype != FCC_F32)
    return out_dtype == FCC_F16 ? FCC_ERR_UNSUPPORTED : FCC_ERR_INVALID;
  if (opts != nullptr && opts->cta_pair != 0 && opts->cta_pair != 1 && opts->cta_pair != 2)
    return FCC_ERR_INVALID;
  if (opts != nullptr && (opts->algo < FCC_ALGO_AUTO || opts->algo > FCC_ALGO_CE))
    return FCC_ERR_INVALID;
  return FCC_OK;
}

}  // namespace
}  // namespace fcc

using namespace fcc;

extern "C" {

size_t fcc_moe_workspace_size(int R, int64_t T, int64_t H, int64_t F, int E, int topk,
                              int64_t cap, const fcc_opts* opts) {
  (void)F;
  if (R < 1 || R > FCC_MAX_RANKS || T < 1 || E < 1 || E > FCC_MAX_EXPERTS || topk < 1)
    return 0;
  // Upper bound: includes room to stage the rows (recv_x NULL, and the
  // sources not one array or another algorithm than the gather asked for),
  // and with FCC_ALGO_CE the send buffers.
  const bool ce = opts != nullptr && opts->algo == FCC_ALGO_CE;
  return moe_plan(R, T, E, topk, H, cap, true, ce).total;
}

fcc_status fcc_moe_dispatch_gemm(int R, const void* const* X, const float* const* logits,
                                 const void* const* W, int64_t T, int64_t H, int64_t F, int E,
                                 int topk, void* const* recv_x, void* const* recv_y,
                                 int64_t cap, int32_t* const* topk_idx,
                                 float* const* topk_gate, int32_t* expert_counts,
                                 int32_t* send_counts, int32_t* const* recv_src, fcc_dtype in,
                                 fcc_dtype out_dtype, const fcc_opts* opts,
                                 fcc_stream_t stream) {
  fcc_status s = check_moe(R, X, logits, W, T, H, F, E, topk, recv_x, recv_y, cap, topk_idx,
                           topk_gate, expert_counts, send_counts, recv_src, in, out_dtype, opts);
  if (s != FCC_OK) return s;
  fcc_algo algo = opts != nullptr ? opts->algo : FCC_ALGO_AUTO;
  if (algo == FCC_ALGO_AUTO) algo = env_defaults().algo;  // (FCC_ALGO; AUTO when unset)
  const bool gather = moe_gathers(opts, R, X, T, H);
  const bool interdecom = algo == FCC_ALGO_INTERDECOM;
  const bool ce = algo == FCC_ALGO_CE;
  const bool unfused = algo == FCC_ALGO_UNFUSED;
  // AUTO / FUSED: the rows are moved by the GEMM's own copy warps (or, for
  // FUSED with one source array, gathered by its TMA).  The baselines move
  // them first: UNFUSED with one copy kernel, INTERDECOM with one copy kernel
  // per expert range on a side stream ahead of that range's GEMM, CE with the
  // copy engines.
  const bool baseline = unfused || interdecom || ce;
  const bool stage_ws = !gather && recv_x == nullptr;
  const bool copy_in_gemm = !gather && !baseline;
  const MoePlan plan = moe_plan(R, T, E, topk, H, cap, stage_ws, ce);
  void* ws = nullptr;
  int* status = nullptr;
  int sms = 0;
  unsigned long long timeout_ns = 0;
  if ((s = internal_prepare(opts, plan.total, &ws, &status, &sms, &timeout_ns)) != FCC_OK)
    return s;
  char* base = static_cast<char*>(ws);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  MoeArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int r = 0; r < R; ++r) {
    a.X[r] = X[r];
    a.logits[r] = logits[r];
    a.idx[r] = topk_idx[r];
    a.gate[r] = topk_gate[r];
    a.recv_x[r] = recv_x != nullptr
                      ? recv_x[r]
                      : (stage_ws ? static_cast<char*>(ws) + plan.off_stage +
                                        static_cast<size_t>(r) * cap * H * 2
                                  : nullptr);
    a.recv_src[r] = recv_src[r];
    if (ce) a.send[r] = base + plan.off_send + static_cast<size_t>(r) * T * topk * H * 2;
  }
  a.R = R;
  a.E = E;
  a.Eloc = E / R;
  a.topk = topk;
  a.T = static_cast<int>(T);
  a.H = static_cast<int>(H);
  a.cap = static_cast<int>(cap);
  a.chunks_per_rank = plan.chunks_per_rank;
  a.tiles_n = static_cast<int>((F + kMoeBN - 1) / kMoeBN);
  const int cg = (opts != nullptr && opts->cta_pair == 1) ? 1 : 2;
  a.tile_m = kBM * cg;
  a.chunk_counts = reinterpret_cast<int32_t*>(base + plan.off_chunk_counts);
  a.chunk_off = reinterpret_cast<int32_t*>(base + plan.off_chunk_off);
  a.expert_counts = expert_counts;
  a.send_counts = send_counts;
  a.expert_base = reinterpret_cast<int32_t*>(base + plan.off_base);
  a.expert_rows = reinterpret_cast<int32_t*>(base + plan.off_rows);
  a.tile_start = reinterpret_cast<int32_t*>(base + plan.off_tiles);
  a.row_of = reinterpret_cast<int32_t*>(base + plan.off_row_of);
  a.ready = copy_in_gemm ? reinterpret_cast<int32_t*>(base + plan.off_ready) : nullptr;
  a.copy_cursor = copy_in_gemm ? reinterpret_cast<int32_t*>(base + plan.off_cursor) : nullptr;
  a.offsets_ticket = reinterpret_cast<int32_t*>(base + plan.off_ticket);
  a.ce_srcoff = reinterpret_cast<int32_t*>(base + plan.off_ce_srcoff);
  a.ce_send_base = reinterpret_cast<int32_t*>(base + plan.off_ce_send_base);
  a.ce_plan = reinterpret_cast<int32_t*>(base + plan.off_ce_plan);
  a.status = status;

  GroupedParams g;
  std::memset(&g, 0, sizeof(g));
  for (int d = 0; d < R; ++d) {
    if (gather)
      s = d == 0 ? internal_make_map(&g.mapA[0], X[0], R * T, H, 1) : FCC_OK;
    else
      s = internal_make_map(&g.mapA[d], a.recv_x[d], cap, H, kBM);
    if (s != FCC_OK) return s;
    if (gather) g.mapA[d] = g.mapA[0];
    g.recv_src[d] = recv_src[d];
    g.out[d] = recv_y[d];
  }
  for (int e = 0; e < E; ++e)
    if ((s = internal_make_map(&g.mapB[e], W[e], H, F, kBK)) != FCC_OK) return s;
  g.R = R;
  g.E = E;
  g.Eloc = E / R;
  g.N = static_cast<int>(F);
  g.K = static_cast<int>(H);
  g.tiles_n = a.tiles_n;
  g.kb_per_rank = static_cast<int>((H + kBK - 1) / kBK);
  g.out_f32 = out_dtype == FCC_F32 ? 1 : 0;
  g.tile_start = a.tile_start;
  g.expert_base = a.expert_base;
  g.expert_rows = a.expert_rows;
  g.e_lo = 0;
  g.e_hi = E;
  g.status = status;
  g.timeout_ns = timeout_ns;
  g.phase_ns = opts != nullptr ? reinterpret_cast<unsigned long long*>(opts->phase_ns) : nullptr;
  // Release the next launch (a combine, or the next call's router) when the
  // expert GEMM's last accumulators are complete: 581-588 against 590-591 us
  // released at the start.
  g.trigger_late = 1;
  g.gather = gather ? 1 : 0;
  if (copy_in_gemm) {
    for (int r = 0; r < R; ++r) {
      g.src_x[r] = X[r];
      g.stage_x[r] = a.recv_x[r];
    }
    g.T = static_cast<int>(T);
    g.ready = a.ready;
    g.copy_cursor = a.copy_cursor;
    g.stage_copy = 1;
  }

  // The chain on `st` launches with programmatic stream serialization: each
  // kernel's launch overlaps the one before it, and waits for it in-kernel.
  // Up to kPlaceMaxChunks chunks, the offsets and ranks are one kernel.
  const bool place = plan.nchunks <= kPlaceMaxChunks;
  if (launch_pdl(route_kernel, dim3(plan.nchunks), dim3(kChunkTok * kRouteSub), 0, st, 1u, a) !=
      cudaSuccess)
    return FCC_ERR_CUDA;
  if (place) {
    if (launch_pdl(place_kernel, dim3(plan.nchunks), dim3(FCC_MAX_EXPERTS * kPlaceSub), 0, st,
                   1u, a) != cudaSuccess)
      return FCC_ERR_CUDA;
  } else if (launch_pdl(offsets_kernel, dim3(E), dim3(256), 0, st, 1u, a) != cudaSuccess ||
             launch_pdl(rank_kernel, dim3(plan.nchunks), dim3(256), 0, st, 1u, a) !=
                 cudaSuccess) {
    return FCC_ERR_CUDA;
  }
  uint64_t launches = place ? 2 : 3;
  const int grid = std::max(cg, (sms / cg) * cg);

  if (interdecom) {
    // Chunks are expert ranges [i*E/c, (i+1)*E/c): every range's row copy is
    // queued on a side stream at once, and range i's grouped GEMM runs on the
    // caller's stream after range i's copy, so range i+1's copy overlaps
    // range i's GEMM.  c from opts->chunks or the chunk model.
    int chunks = (opts != nullptr && opts->chunks > 0) ? opts->chunks
                 : (env_defaults().chunks > 0 ? env_defaults().chunks
                                              : moe_model_chunks(R, T, H, F, E, topk));
    chunks = std::max(1, std::min(chunks, E));
    cudaStream_t side = nullptr;
    cudaEvent_t ev[FCC_MAX_EXPERTS + 1];
    if ((s = internal_streams_events(&side, 1, ev, chunks + 1)) != FCC_OK) return s;
    if (cudaEventRecord(ev[chunks], st) != cudaSuccess ||
        cudaStreamWaitEvent(side, ev[chunks], 0) != cudaSuccess)
      return FCC_ERR_CUDA;
    for (int i = 0; i < chunks; ++i) {
      const int e_lo = i * E / chunks, e_hi = (i + 1) * E / chunks;
      if (e_lo == e_hi) continue;
      copy_expert_rows_kernel<<<std::max(1, sms) * 4, 256, 0, side>>>(a, e_lo, e_hi);
      if (cudaGetLastError() != cudaSuccess) return FCC_ERR_CUDA;
      if (cudaEventRecord(ev[i], side) != cudaSuccess ||
          cudaStreamWaitEvent(st, ev[i], 0) != cudaSuccess)
        return FCC_ERR_CUDA;
      g.e_lo = e_lo;
      g.e_hi = e_hi;
      if (launch_grouped_gemm(g, cg, grid, st) != cudaSuccess) return FCC_ERR_CUDA;
      launches += 2;
    }
  } else if (ce) {
    // The (source rank, expert) runs are contiguous on both sides once each
    // source packs its rows (an SM copy within the rank); the exchange itself
    // is one cudaMemcpyAsync per run on the copy engines.  The run sizes are
    // data-dependent, so the host reads them back first: this form
    // synchronises the stream (as a copy-engine all-to-all with variable
    // splits needs the split sizes on the host).
    if (launch_pdl(ce_plan_kernel, dim3(1), dim3(64), 0, st, 1u, a) != cudaSuccess ||
        launch_pdl(ce_pack_kernel, dim3(std::max(1, sms) * 4), dim3(256), 0, st, 1u, a) !=
            cudaSuccess)
      return FCC_ERR_CUDA;
    launches += 2;
    const size_t plan_bytes = static_cast<size_t>(R) * E * 3 * 4;
    int32_t* hp = nullptr;
    if ((s = internal_host_buffer(plan_bytes, reinterpret_cast<void**>(&hp))) != FCC_OK) return s;
    if (cudaMemcpyAsync(hp, a.ce_plan, plan_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return FCC_ERR_CUDA;
    constexpr int kCeStreams = 4;
    cudaStream_t side[kCeStreams];
    cudaEvent_t ev[kCeStreams + 1];
    if ((s = internal_streams_events(side, kCeStreams, ev, kCeStreams + 1)) != FCC_OK) return s;
    if (cudaEventRecord(ev[kCeStreams], st) != cudaSuccess) return FCC_ERR_CUDA;
    for (int i = 0; i < kCeStreams; ++i)
      if (cudaStreamWaitEvent(side[i], ev[kCeStreams], 0) != cudaSuccess) return FCC_ERR_CUDA;
    const size_t row_bytes = static_cast<size_t>(H) * 2;
    int q = 0;
    for (int src = 0; src < R; ++src) {
      for (int e = 0; e < E; ++e) {
        const int32_t* pl = hp + 3 * (src * E + e);
        const int64_t send_row = pl[0], recv_row = pl[1], rows = pl[2];
        if (rows == 0) continue;
        // The runs come from this call's own kernels; a run outside its
        // buffers would be a library fault: refuse it rather than copy.
        if (rows < 0 || send_row < 0 || recv_row < 0 || send_row + rows > T * topk ||
            recv_row + rows > cap)
          return FCC_ERR_CUDA;
        if (cudaMemcpyAsync(static_cast<char*>(a.recv_x[e / a.Eloc]) + recv_row * row_bytes,
                            static_cast<const char*>(a.send[src]) + send_row * row_bytes,
                            rows * row_bytes, cudaMemcpyDeviceToDevice,
                            side[q++ % kCeStreams]) != cudaSuccess)
          return FCC_ERR_CUDA;
      }
    }
    for (int i = 0; i < kCeStreams; ++i)
      if (cudaEventRecord(ev[i], side[i]) != cudaSuccess ||
          cudaStreamWaitEvent(st, ev[i], 0) != cudaSuccess)
        return FCC_ERR_CUDA;
    if (launch_grouped_gemm(g, cg, grid, st) != cudaSuccess) return FCC_ERR_CUDA;
    launches += 1;
  } else {
    // With the gather the copy (only for a requested recv_x) runs beside the
    // GEMM on a side stream: both only read what the dispatch kernels wrote.
    const bool copy = !gather || recv_x != nullptr;
    const bool side_copy = copy && gather;
    cudaStream_t side = nullptr;
    cudaEvent_t ev[2] = {};
    if (side_copy) {
      if ((s = internal_side_stream(&side, ev, 2)) != FCC_OK) return s;
      if (cudaEventRecord(ev[0], st) != cudaSuccess ||
          cudaStreamWaitEvent(side, ev[0], 0) != cudaSuccess)
        return FCC_ERR_CUDA;
    }
    if (copy && !copy_in_gemm) {
      if (launch_pdl(copy_kernel, dim3(std::max(1, sms) * 4), dim3(256), 0,
                     side_copy ? side : st, 1u, a) != cudaSuccess)
        return FCC_ERR_CUDA;
      launches += 1;
    }
    if (side_copy && cudaEventRecord(ev[1], side) != cudaSuccess) return FCC_ERR_CUDA;
    if (launch_grouped_gemm(g, cg, grid, st) != cudaSuccess) return FCC_ERR_CUDA;
    if (side_copy && cudaStreamWaitEvent(st, ev[1], 0) != cudaSuccess) return FCC_ERR_CUDA;
    launches += 1;
  }
  bump_launch_count(launches);
  return FCC_OK;
}

// Test support: the grouped expert GEMM (with in-kernel staging) on a table
// of one expert, one 256-row unit holding one row, and one 256-column tile,
// whose copy cursor starts past the last chunk: the copy warps claim nothing,
// so the unit's row counter stays at zero and the TMA producers' bounded wait
// for it runs out after timeout_ns.  The kernel then records FCC_ERR_TIMEOUT,
// unwinds (no loads or MMAs were issued), frees its tensor memory and exits.
fcc_status fcc_test_grouped_wait_timeout(int64_t timeout_ns, fcc_stream_t stream) {
  if (timeout_ns <= 0) return FCC_ERR_INVALID;
  constexpr int kRows = 256, kH = 64, kF = 256;
  // ints: tile_start[2], expert_rows[1], expert_base[1], ready[1], cursor, recv_src[1]
  constexpr size_t kInts = 256;
  constexpr size_t kA = static_cast<size_t>(kRows) * kH * 2, kB = static_cast<size_t>(kH) * kF * 2,
                   kOut = static_cast<size_t>(kRows) * kF * 2;
  void* ws = nullptr;
  int* status = nullptr;
  int sms = 0;
  unsigned long long tmo = 0;
  fcc_status s = internal_prepare(nullptr, kInts + kA + kB + kOut, &ws, &status, &sms, &tmo);
  if (s != FCC_OK) return s;
  char* base = static_cast<char*>(ws);
  int32_t* ints = reinterpret_cast<int32_t*>(base);
  void* A = base + kInts;
  void* Bw = base + kInts + kA;
  void* out = base + kInts + kA + kB;
  static const int32_t host_ints[8] = {0, 1, /*rows*/ 1, /*base*/ 0, /*ready*/ 0,
                                       /*cursor*/ 1 << 30, /*recv_src*/ 0, 0};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, kInts + kA + kB + kOut, st) != cudaSuccess ||
      cudaMemcpyAsync(ints, host_ints, sizeof(host_ints), cudaMemcpyHostToDevice, st) !=
          cudaSuccess)
    return FCC_ERR_CUDA;
  GroupedParams g;
  std::memset(&g, 0, sizeof(g));
  if ((s = internal_make_map(&g.mapA[0], A, kRows, kH, kBM)) != FCC_OK) return s;
  if ((s = internal_make_map(&g.mapB[0], Bw, kH, kF, kBK)) != FCC_OK) return s;
  g.out[0] = out;
  g.R = 1;
  g.E = 1;
  g.Eloc = 1;
  g.N = kF;
  g.K = kH;
  g.tiles_n = 1;
  g.kb_per_rank = 1;
  g.tile_start = ints;
  g.expert_rows = ints + 2;
  g.expert_base = ints + 3;
  g.e_lo = 0;
  g.e_hi = 1;
  g.status = status;
  g.timeout_ns = static_cast<unsigned long long>(timeout_ns);
  g.recv_src[0] = ints + 6;
  g.src_x[0] = A;
  g.stage_x[0] = A;
  g.T = 1;
  g.ready = ints + 4;
  g.copy_cursor = ints + 5;
  g.stage_copy = 1;
  if (launch_grouped_gemm(g, 2, 2, st) != cudaSuccess) return FCC_ERR_CUDA;
  bump_launch_count(1);
  return FCC_OK;
}

}  // extern "C"

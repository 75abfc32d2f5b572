// fcc_gemv.cu -- GEMV + AllReduce for the decode shape (sm_103a).
//
// Y = sum_r A_r @ B_r with A_r [M <= 16, K] (tokens) and B_r [K, N]; Y is
// written to every rank's buffer (SC24 paper, abstract: the GEMV + AllReduce
// operator for Transformers).  The work is a stream of B bytes from HBM.  The
// grid is (column groups of 512) x (splits of the rank-and-K range K' = R*K),
// about one persistent CTA per SM; the CTAs of one split read the same rows of
// B across all groups at the same time, so B is read in whole rows.
//
// Each stage is one 64-row block of 256 columns (32 KiB, four TMA boxes) plus
// the 16 token rows of that block (2 KiB, one TMA box; rows past M read as
// zeros).  One tcgen05.mma per 16 k (M = 128 rows, N = 256 columns)
// accumulates into one of the group's two TMEM accumulators; TMEM lane t holds
// token t's row.  The MMA's A operand is 128 rows, of which only the first 16
// are loaded: rows 16-127 read whatever shared memory follows (later stages),
// and each output row depends on its own A row only, so those lanes hold
// values nobody reads.  The stage thus costs 34 KiB instead of 48; five
// stages (160 KiB of B in flight) measured faster than six.
//
// Cross-CTA sum: each CTA writes its f32 partial rows for the group to its
// own workspace slot and takes the group's ticket; the last to arrive adds the
// group's partials in split order (a fixed order, so the result is
// repeatable) and stores the sum to all R output buffers.  No CTA waits on
// another.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "fcc_internal.h"
#include "fcc_ptx.cuh"

namespace fcc {
namespace {

constexpr int kGroupCols = 512;                 // columns per CTA group (two accumulators)
constexpr int kStageCols = 256;                 // columns per pipeline stage (UMMA N)
constexpr int kTok = kGemvTok;                  // token rows loaded per stage (M <= 16)
constexpr int kTokStep = 8;                     // tokens per step of the final sum
constexpr int kMaxClusterSplits = 16;           // splits a column group's cluster may hold
// Five stages: 76.2 us at the 8-rank decode workload against 77.9 with six
// (four: 76.1).
constexpr int kStages = 5;
constexpr uint32_t kBBox = kBK * 64 * 2;        // [64 k][64 n] bf16 = 8 KiB
constexpr uint32_t kBStage = 4 * kBBox;         // 32 KiB: [64 k][256 n]
constexpr uint32_t kAStage = kTok * kBK * 2;    // 2 KiB: [16 rows][64 k], rows >= M zero
constexpr uint32_t kStageBytes = kBStage + kAStage;
constexpr uint32_t kTmemCols = 512;             // 2 accumulators x 256 columns
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kBM, kStageCols, /*a_mn=*/false, /*b_mn=*/true);
constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + (2 * kStages + 4) * 8 + 16;
// The MMA reads 128 A rows (16 KiB) from each A stage: for the last one they
// run on into the B stages, which must therefore follow within the buffer.
static_assert((kStages - 1) * kAStage + kBM * kBK * 2 <= kStages * kStageBytes,
              "A operand read past the stages");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

__global__ void __launch_bounds__(kGemmThreads, 1) gemv_ar_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;                          // kStages x 2 KiB (MMA reads 16 KiB from each)
  uint8_t* sB = smem + kStages * kAStage;      // kStages x 32 KiB
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kStages * kBStage);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* mma_done = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* bcast = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = blockIdx.x / p.splits;              // column group
  const int split = blockIdx.x - g * p.splits;      // part of the K' range
  const int kbt = p.R * p.kb_per_rank;              // 64-row blocks of K'
  const int kb0 = static_cast<int>(static_cast<long long>(kbt) * split / p.splits);
  const int kb1 = static_cast<int>(static_cast<long long>(kbt) * (split + 1) / p.splits);
  const int col0 = g * kGroupCols;
  const int ncols = min(kGroupCols, p.N - col0);
  const int nstage_cols = (ncols + kStageCols - 1) / kStageCols;  // accumulators in use

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(tfull, 1);
    ptx::mbar_init(mma_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int r = 0; r < p.R; ++r) {
      ptx::tma_prefetch_desc(&p.mapA[r]);
      ptx::tma_prefetch_desc(&p.mapB[r]);
    }
    // The first stages' weights into L2 while the previous kernel may still
    // run: an L2 prefetch returns nothing to this CTA, so it cannot see data
    // older than the loads after the wait below, which read through L2.
    int kbi = kb0, sc = 0;
    for (int i = 0; i < kStages && kbi < kb1; ++i) {
      const int r = kbi / p.kb_per_rank;
      const int kb = kbi - r * p.kb_per_rank;
#pragma unroll
      for (int b = 0; b < kStageCols / 64; ++b)
        ptx::tma_prefetch_2d(&p.mapB[r], col0 + sc * kStageCols + 64 * b, kb * kBK);
      if (++sc == nstage_cols) {
        sc = 0;
        ++kbi;
      }
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // Launched with programmatic stream serialization: the set-up above touches
  // no global memory (the tensor maps are kernel parameters), so it may
  // overlap the previous kernel on the stream; everything below waits for it.
  // The next kernel's launch is released once the accumulators are complete
  // (epilogue below), so a small next kernel does not sit beside this one.
  ptx::griddep_wait();
  const uint32_t tmem_base = *tmem_slot;
  const ptx::Waiter W{abort_flag, p.status, p.timeout_ns};

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t keep = ptx::policy_evict_last();    // token rows are re-read by every group
      uint32_t stage = 0, phase = 0, issued = 0, last_parity = 0;
      bool ok = true;
      for (int kbi = kb0; kbi < kb1 && ok; ++kbi) {
        const int r = kbi / p.kb_per_rank;
        const int kb = kbi - r * p.kb_per_rank;
        for (int sc = 0; sc < nstage_cols; ++sc) {
          if (!W.wait(&empty[stage], phase ^ 1u)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&full[stage], kStageBytes);
          ptx::tma_load_2d_hint(sA + stage * kAStage, &p.mapA[r], &full[stage], kb * kBK, 0,
                                keep);
          uint8_t* b_dst = sB + stage * kBStage;
#pragma unroll
          for (int i = 0; i < kStageCols / 64; ++i)
            ptx::tma_load_2d(b_dst + i * kBBox, &p.mapB[r], &full[stage],
                             col0 + sc * kStageCols + 64 * i, kb * kBK);
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort_flag) {
        for (int s = 0; s < kStages; ++s)
          if (issued & (1u << s)) W.drain(&full[s], (last_parity >> s) & 1u, kDrainNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool any = false, ok = true;
      for (int kbi = kb0; kbi < kb1 && ok; ++kbi) {
        for (int sc = 0; sc < nstage_cols; ++sc) {
          if (!W.wait(&full[stage], phase)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_addr = ptx::smem_addr(sA + stage * kAStage);
          const uint32_t b_addr = ptx::smem_addr(sB + stage * kBStage);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // A = the token rows (zero past M, unread lanes past 16): K-major, 32 B per 16 k.
            const uint64_t ad = ptx::smem_desc_sw128(a_addr + kk * 32, 16, 1024);
            // B = 256 columns: MN-major, 16 k-rows per step, 64-column atoms 8 KiB apart.
            const uint64_t bd = ptx::smem_desc_sw128(b_addr + kk * 2048, kBBox, 1024);
            ptx::mma_f16(tmem_base + sc * kStageCols, ad, bd, kIdesc,
                         (kbi > kb0 || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit(&empty[stage]);
          any = true;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (ok && any) ptx::mma_commit(tfull);
      if (any) {
        ptx::mma_commit(mma_done);
        W.drain(mma_done, 0, kDrainNs);
      }
    }
  } else {
    // Epilogue.  TMEM lane t holds token t's row, so the warp reading lanes
    // 0-31 (warp 4) copies the tokens' partial rows; all four warps then take
    // the group's ticket together and, if last, sum the group.
    const int q = warp & 3;
    const int ep_tid = threadIdx.x - 64;
    const bool failed = (kb1 <= kb0) || !W.wait(tfull, 0);
    if (ep_tid == 0) ptx::griddep_launch_dependents();
    if (p.cluster) {
      // Cluster form: the partial rows stay in this CTA's shared memory (the
      // stages are free once the accumulators are complete); the cluster
      // sums them below.  A CTA that failed leaves its rows unwritten (the
      // status word holds the error).
      if (!failed && q == 0) {
        ptx::tc_fence_after();
        float* part = reinterpret_cast<float*>(sB) + lane * kGroupCols;
        for (int sc = 0; sc < nstage_cols; ++sc) {
#pragma unroll 1
          for (int c = 0; c < kStageCols; c += 32) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(tmem_base + sc * kStageCols + c, v);
            ptx::tmem_ld_wait();
            if (lane < p.M) {
              float4* d = reinterpret_cast<float4*>(part + sc * kStageCols + c);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                d[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                   __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
            }
          }
        }
      }
    } else if (!ptx::named_barrier_or(1, 128, failed)) {  // the epilogue warps stop together
      ptx::tc_fence_after();
      if (q == 0) {
        float* part = p.partials + (static_cast<long long>(blockIdx.x) * p.M + lane) * kGroupCols;
        for (int sc = 0; sc < nstage_cols; ++sc) {
#pragma unroll 1
          for (int c = 0; c < kStageCols; c += 32) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(tmem_base + sc * kStageCols + c, v);
            ptx::tmem_ld_wait();
            if (lane < p.M) {
              float4* d = reinterpret_cast<float4*>(part + sc * kStageCols + c);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                d[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                   __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
            }
          }
        }
      }
      __threadfence();
      ptx::named_barrier_sync(1, 128);
      if (ep_tid == 0) {
        // Ticket = (call generation << 8) | arrivals.  A value left by an
        // earlier call has another generation and counts as zero, so the
        // tickets need no clearing between calls.  Each CAS that fails means
        // another CTA of the group got in: at most `splits` retries.
        unsigned* tk = reinterpret_cast<unsigned*>(p.tickets + g);
        const unsigned gen = p.gen & 0xFFFFFFu;
        unsigned cur = *reinterpret_cast<volatile unsigned*>(tk), nv;
        while (true) {
          const unsigned cnt = ((cur >> 8) == gen) ? (cur & 0xFFu) : 0u;
          nv = (gen << 8) | (cnt + 1u);
          const unsigned prev = atomicCAS(tk, cur, nv);
          if (prev == cur) break;
          cur = prev;
        }
        *bcast = ((nv & 0xFFu) == static_cast<unsigned>(p.splits)) ? 1 : 0;
      }
      ptx::named_barrier_sync(1, 128);
      if (*bcast) {
        // Last of the group: sum the splits' partials in split order; each
        // thread handles 4 consecutive columns (one 16-byte load per partial)
        // of up to 8 tokens at a time, three splits per step, so 24 loads are
        // in flight instead of one: this sum is the kernel's serial tail.
        __threadfence();
        const int c = ep_tid * 4;
        if (c < ncols) {
          const float* base = p.partials + static_cast<long long>(g) * p.splits * p.M * kGroupCols;
          auto part = [&](int sp, int t) {
            return __ldcg(reinterpret_cast<const float4*>(
                base + (static_cast<long long>(sp) * p.M + t) * kGroupCols + c));
          };
          auto add = [](float4& a, const float4& x) {
            a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
          };
          for (int t0 = 0; t0 < p.M; t0 += kTokStep) {
            const int nt = min(kTokStep, p.M - t0);
            float4 acc[kTokStep];
#pragma unroll
            for (int i = 0; i < kTokStep; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            int sp = 0;
            for (; sp + 3 <= p.splits; sp += 3) {
              float4 x0[kTokStep], x1[kTokStep], x2[kTokStep];
#pragma unroll
              for (int i = 0; i < kTokStep; ++i)
                if (i < nt) {
                  x0[i] = part(sp, t0 + i);
                  x1[i] = part(sp + 1, t0 + i);
                  x2[i] = part(sp + 2, t0 + i);
                }
#pragma unroll
              for (int i = 0; i < kTokStep; ++i)
                if (i < nt) {  // (split order: sp, sp + 1, sp + 2)
                  add(acc[i], x0[i]);
                  add(acc[i], x1[i]);
                  add(acc[i], x2[i]);
                }
            }
            for (; sp < p.splits; ++sp) {
#pragma unroll
              for (int i = 0; i < kTokStep; ++i)
                if (i < nt) add(acc[i], part(sp, t0 + i));
            }
#pragma unroll
            for (int i = 0; i < kTokStep; ++i) {
              if (i >= nt) break;
              const long long o = static_cast<long long>(t0 + i) * p.N + col0 + c;
              for (int r = 0; r < p.R; ++r) {
                if (p.out_f32) {
                  *reinterpret_cast<float4*>(static_cast<float*>(p.out[r]) + o) = acc[i];
                } else {
                  uint2 w;
                  w.x = ptx::pack_bf16x2(acc[i].x, acc[i].y);
                  w.y = ptx::pack_bf16x2(acc[i].z, acc[i].w);
                  *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out[r]) + o) = w;
                }
              }
            }
          }
        }
      }
    }
  }

  __syncwarp();
  ptx::tc_fence_before();
  if (p.cluster) {
    // Every CTA of the column group's cluster holds its partial rows; CTA i
    // (cluster rank i = split i) adds the splits' values of its slice of the
    // group's columns in split order (the same additions, in the same order,
    // as the ticket form's last arriver) and stores the sums to all R
    // outputs.  The second cluster barrier keeps each CTA's shared memory
    // alive until its peers have read it.
    ptx::cluster_sync_all();
    const int nsp = p.splits;
    const int rank = static_cast<int>(ptx::cluster_ctarank());
    const int cw = ((kGroupCols + nsp - 1) / nsp + 3) & ~3;  // a slice: whole float4s
    const int c_lo = min(ncols, rank * cw), c_hi = min(ncols, c_lo + cw);
    const int nvec = (c_hi - c_lo) / 4;
    const uint32_t part0 = ptx::smem_addr(sB);
    for (int item = threadIdx.x; item < p.M * nvec; item += blockDim.x) {
      const int t = item / nvec;
      const int c = c_lo + (item - t * nvec) * 4;
      const uint32_t off = part0 + static_cast<uint32_t>((t * kGroupCols + c) * 4);
      float4 x[kMaxClusterSplits];  // every split's value in flight, then added in order
#pragma unroll
      for (int sp = 0; sp < kMaxClusterSplits; ++sp)
        if (sp < nsp) x[sp] = ptx::ld_shared_cluster_f4(ptx::mapa(off, static_cast<uint32_t>(sp)));
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int sp = 0; sp < kMaxClusterSplits; ++sp) {
        if (sp < nsp) {
          acc.x += x[sp].x;
          acc.y += x[sp].y;
          acc.z += x[sp].z;
          acc.w += x[sp].w;
        }
      }
      const long long o = static_cast<long long>(t) * p.N + col0 + c;
      for (int r = 0; r < p.R; ++r) {
        if (p.out_f32) {
          *reinterpret_cast<float4*>(static_cast<float*>(p.out[r]) + o) = acc;
        } else {
          uint2 w;
          w.x = ptx::pack_bf16x2(acc.x, acc.y);
          w.y = ptx::pack_bf16x2(acc.z, acc.w);
          *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out[r]) + o) = w;
        }
      }
    }
    ptx::cluster_sync_all();
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

int gemv_smem_bytes() { return kSmemBytes; }

cudaError_t launch_gemv(const GemvParams& p, int grid, cudaStream_t st) {
  static bool attr_set[64] = {};
  const cudaError_t e = smem_attr_once(attr_set, gemv_ar_kernel, kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(gemv_ar_kernel, dim3(grid, 1, 1), dim3(kGemmThreads, 1, 1), kSmemBytes, st,
                    p.cluster ? static_cast<unsigned>(p.splits) : 1u, p);
}

// Whether `groups` clusters of `splits` GEMV CTAs (one per SM) fit on the
// current device at once, so the cluster form of the final sum runs in one
// wave; looked up once per device and split count.
bool gemv_cluster_fits(int groups, int splits) {
  if (splits < 2 || splits > kMaxClusterSplits) return false;
  static int cache[64][kMaxClusterSplits + 1] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lk(mu);
  int& n = cache[dev][splits];
  if (n == 0) {
    n = -1;
    if (cudaFuncSetAttribute(gemv_ar_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) == cudaSuccess &&
        cudaFuncSetAttribute(gemv_ar_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(splits * groups), 1, 1);
      cfg.blockDim = dim3(kGemmThreads, 1, 1);
      cfg.dynamicSmemBytes = kSmemBytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int c = 0;
      if (cudaOccupancyMaxActiveClusters(&c, gemv_ar_kernel, &cfg) == cudaSuccess) n = c;
    }
    cudaGetLastError();  // (a refused query leaves no sticky error)
  }
  return n >= groups;
}

// Arrival tickets of the default path (no caller workspace): a library array,
// zero at load, that the generation-stamped tickets keep consistent without
// clearing (one entry per column group).
__device__ unsigned g_gemv_tickets[kMaxGemvGroups];

std::atomic<unsigned> g_gemv_gen{0};

unsigned next_gemv_gen() {
  return (g_gemv_gen.fetch_add(1) % 0xFFFFFEu) + 1u;  // 1 .. 2^24 - 2, never 0
}

fcc_status gemv_internal_tickets(int** out) {
  static int* cached[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FCC_ERR_CUDA;
  std::lock_guard<std::mutex> lk(mu);
  if (cached[dev] == nullptr &&
      cudaGetSymbolAddress(reinterpret_cast<void**>(&cached[dev]), g_gemv_tickets) != cudaSuccess)
    return FCC_ERR_CUDA;
  *out = cached[dev];
  return FCC_OK;
}

// Grid shape: groups = ceil(N / 512) column groups, `splits` CTAs per group
// (about one CTA per SM in total, at most one per 64-row block of K').
void gemv_shape(int64_t N, int R, int64_t K, int sms, int max_ctas, int* groups, int* splits) {
  const int g = static_cast<int>((N + kGroupCols - 1) / kGroupCols);
  const long long kbt = static_cast<long long>(R) * ((K + kBK - 1) / kBK);
  int ctas = sms;
  if (max_ctas > 0 && max_ctas < ctas) ctas = max_ctas;
  long long s = ctas / g;
  if (s < 1) s = 1;
  if (s > kbt) s = kbt;
  if (s > 255) s = 255;  // ticket arrivals are counted in 8 bits
  *groups = g;
  *splits = static_cast<int>(s);
}

size_t gemv_partial_bytes(int groups, int splits, int64_t M) {
  return static_cast<size_t>(groups) * splits * M * kGroupCols * 4;
}

}  // namespace fcc

// ---------------------------------------------------------------------------
// fcc_gemv_ar_static: the same GEMV + AllReduce kernel with its scratch (the
// per-CTA partial sums and the per-group arrival tickets) in a fixed device
// array of this file instead of caller or pool memory, for callers that cannot
// allocate device memory.  The array lives on every GPU that loads the library
// until the process exits.
#include <mutex>

namespace fcc {
namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB in total
constexpr size_t kStaticTicketBytes = 4096;              // tickets: up to 1024 groups

__device__ __align__(256) unsigned char g_gemv_static_scratch[kStaticScratchBytes];

struct StaticScratchDev {
  bool ready = false;
  unsigned char* ptr = nullptr;  // device address of g_gemv_static_scratch
  int sms = 0;
};
StaticScratchDev g_static_dev[64];
std::mutex g_static_mu;

// Once per device, with that device current: look up the array's device
// address (host code cannot use the symbol itself as a pointer) and the SM count.
fcc_status static_scratch_for_current_device(unsigned char** ptr, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FCC_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_static_mu);
  StaticScratchDev& s = g_static_dev[dev];
  if (!s.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_gemv_static_scratch) != cudaSuccess || p == nullptr)
      return FCC_ERR_CUDA;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FCC_ERR_CUDA;
    s.ptr = static_cast<unsigned char*>(p);
    s.sms = n;
    s.ready = true;
  }
  *ptr = s.ptr;
  *sms = s.sms;
  return FCC_OK;
}

}  // namespace
}  // namespace fcc

extern "C" fcc_status fcc_gemv_ar_static(int R, const void* const* A, const void* const* B,
                                         void* const* out, int64_t M, int64_t N, int64_t K,
                                         fcc_dtype in, fcc_dtype out_dtype, const fcc_opts* opts,
                                         fcc_stream_t stream) {
  using namespace fcc;
  fcc_status s = light_check_gemm(R, A, B, M, N, K, in);
  if (s != FCC_OK) return s;
  if (M > kTok) return FCC_ERR_INVALID;
  if (out_dtype != FCC_BF16 && out_dtype != FCC_F32)
    return out_dtype == FCC_F16 ? FCC_ERR_UNSUPPORTED : FCC_ERR_INVALID;
  if (out == nullptr) return FCC_ERR_INVALID;
  for (int r = 0; r < R; ++r)
    if (out[r] == nullptr || (reinterpret_cast<uintptr_t>(out[r]) & 15u) != 0)
      return FCC_ERR_INVALID;
  // The same status as fcc_gemv_ar for a value outside the enum; the valid
  // unfused forms need allocated partials, which this entry point has not.
  if (opts != nullptr && (opts->algo < FCC_ALGO_AUTO || opts->algo > FCC_ALGO_CE))
    return FCC_ERR_INVALID;
  if (opts != nullptr && opts->algo != FCC_ALGO_AUTO && opts->algo != FCC_ALGO_FUSED)
    return FCC_ERR_UNSUPPORTED;

  unsigned char* scratch = nullptr;
  int sms = 0;
  if ((s = static_scratch_for_current_device(&scratch, &sms)) != FCC_OK) return s;
  int* status = nullptr;
  if ((s = light_status_word(&status)) != FCC_OK) return s;

  int groups = 0, splits = 0;
  gemv_shape(N, R, K, sms, opts != nullptr ? opts->max_ctas : 0, &groups, &splits);
  // Size limit of the static array: one ticket per column group (4 KiB), and
  // one partial (M x 512 f32 = M x 2 KiB) per CTA and group in the remaining
  // 4 MiB - 4 KiB = 2046 x 2 KiB, i.e. ceil(N / 512) * M <= 2046; fewer CTAs
  // per group are used when the default number does not fit.
  const size_t room = kStaticScratchBytes - kStaticTicketBytes;
  const size_t per_split = gemv_partial_bytes(groups, 1, M);
  if (static_cast<size_t>(groups) * 4 > kStaticTicketBytes || per_split > room)
    return FCC_ERR_WORKSPACE;
  if (static_cast<size_t>(splits) * per_split > room) splits = static_cast<int>(room / per_split);

  GemvParams p;
  std::memset(&p, 0, sizeof(p));
  for (int r = 0; r < R; ++r) {
    if ((s = light_make_map(&p.mapA[r], A[r], M, K, kTok)) != FCC_OK) return s;
    if ((s = light_make_map(&p.mapB[r], B[r], K, N, kBK)) != FCC_OK) return s;
    p.out[r] = out[r];
  }
  p.R = R;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.kb_per_rank = static_cast<int>((K + kBK - 1) / kBK);
  p.groups = groups;
  p.splits = splits;
  p.gen = next_gemv_gen();
  p.out_f32 = out_dtype == FCC_F32 ? 1 : 0;
  p.tickets = reinterpret_cast<int*>(scratch);
  p.partials = reinterpret_cast<float*>(scratch + kStaticTicketBytes);
  p.status = status;
  p.timeout_ns = (opts != nullptr && opts->timeout_ns > 0)
                     ? static_cast<unsigned long long>(opts->timeout_ns)
                     : 1000ull * 1000 * 1000;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the tickets must start at zero.
  if (cudaMemsetAsync(p.tickets, 0, static_cast<size_t>(groups) * 4, st) != cudaSuccess)
    return FCC_ERR_CUDA;
  if (launch_gemv(p, groups * splits, st) != cudaSuccess) return FCC_ERR_CUDA;
  count_launch();
  return FCC_OK;
}

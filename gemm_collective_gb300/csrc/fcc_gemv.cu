// fcc_gemv.cu -- GEMV + AllReduce for the decode shape (sm_103a).
//
// Y = sum_r A_r @ B_r with A_r [M <= 16, K] (tokens) and B_r [K, N]; Y is
// written to every rank's buffer (SC24 paper, abstract: the GEMV + AllReduce
// operator for Transformers).  The work is a stream of B bytes from HBM, so
// the kernel is built to keep HBM busy: every SM runs one persistent CTA that
// streams its contiguous share of (column slab, rank, k block) units through a
// 10-stage TMA ring.  The multiply runs on the tensor cores with the roles
// swapped (D^T = B^T A^T): the 128-column B slab is the M=128 operand
// (MN-major in shared memory), the tokens padded to 16 rows by TMA's
// out-of-bounds zero fill are the N=16 operand, and the f32 accumulator sits
// in TMEM, one lane per output column.
//
// Cross-CTA sum: a slab's K' = R*K range is split over consecutive CTAs
// (stream-K).  Each CTA writes its f32 partial for the slab to its own
// workspace slot and takes a ticket; the last to arrive adds the partials in
// CTA order (a fixed order, so the result is repeatable) and stores the sum to
// all R output buffers.  Nothing waits on another CTA.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>

#include "fcc_internal.h"
#include "fcc_ptx.cuh"

namespace fcc {
namespace {

constexpr int kSlab = 128;                      // output columns per slab (UMMA M)
constexpr int kTok = 16;                        // padded tokens (UMMA N)
constexpr int kStages = 10;
constexpr uint32_t kBBox = kBK * 64 * 2;        // [64 k][64 n] bf16 = 8 KiB
constexpr uint32_t kBStage = 2 * kBBox;         // 16 KiB: [64 k][128 n]
constexpr uint32_t kAStage = kTok * kBK * 2;    // 2 KiB: [16 tokens][64 k]
constexpr uint32_t kStageBytes = kBStage + kAStage;
constexpr uint32_t kTmemCols = 32;              // 2 accumulators x 16 columns
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kSlab, kTok, /*a_mn=*/true, /*b_mn=*/false);
constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + (2 * kStages + 5) * 8 + 16;

__device__ __forceinline__ int owner_of(long long u, long long U, int G) {
  // CTA b covers units [floor(b*U/G), floor((b+1)*U/G)); the owner of u is the
  // largest b whose range starts at or before u.
  return static_cast<int>(((u + 1) * G - 1) / U);
}

__global__ void __launch_bounds__(kGemmThreads, 1) gemv_ar_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sB = smem;                          // kStages x 16 KiB
  uint8_t* sA = smem + kStages * kBStage;      // kStages x 2 KiB
  uint64_t* bars = reinterpret_cast<uint64_t*>(sA + kStages * kAStage);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* bcast = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const long long U = p.units;
  const long long u0 = U * blockIdx.x / G;
  const long long u1 = U * (blockIdx.x + 1) / G;
  const int per_slab = p.R * p.kb_per_rank;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&tfull[b], 1);
      ptx::mbar_init(&tempty[b], 4);
    }
    ptx::mbar_init(mma_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int r = 0; r < p.R; ++r) {
      ptx::tma_prefetch_desc(&p.mapA[r]);
      ptx::tma_prefetch_desc(&p.mapB[r]);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const ptx::Waiter W{abort_flag, p.status, p.timeout_ns};

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t keep = ptx::policy_evict_last();    // A rows are re-read by every slab
      const uint64_t stream = ptx::policy_evict_first(); // B is read exactly once
      uint32_t stage = 0, phase = 0, issued = 0, last_parity = 0;
      for (long long u = u0; u < u1; ++u) {
        const int slab = static_cast<int>(u / per_slab);
        const int rem = static_cast<int>(u - static_cast<long long>(slab) * per_slab);
        const int r = rem / p.kb_per_rank;
        const int kb = rem - r * p.kb_per_rank;
        if (!W.wait(&empty[stage], phase ^ 1u)) break;
        ptx::mbar_arrive_expect_tx(&full[stage], kStageBytes);
        uint8_t* b_dst = sB + stage * kBStage;
        ptx::tma_load_2d_hint(b_dst, &p.mapB[r], &full[stage], slab * kSlab, kb * kBK, stream);
        ptx::tma_load_2d_hint(b_dst + kBBox, &p.mapB[r], &full[stage], slab * kSlab + 64,
                              kb * kBK, stream);
        ptx::tma_load_2d_hint(sA + stage * kAStage, &p.mapA[r], &full[stage], kb * kBK, 0, keep);
        issued |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (*abort_flag) {
        for (int s = 0; s < kStages; ++s)
          if (issued & (1u << s)) W.drain(&full[s], (last_parity >> s) & 1u, kDrainNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool any = false, ok = true;
      long long u = u0;
      while (u < u1 && ok) {
        const int slab = static_cast<int>(u / per_slab);
        const long long seg_end = min(u1, static_cast<long long>(slab + 1) * per_slab);
        if (!W.wait(&tempty[acc], acc_phase ^ 1u)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kTok;
        for (long long v = u; v < seg_end; ++v) {
          if (!W.wait(&full[stage], phase)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t b_addr = ptx::smem_addr(sB + stage * kBStage);
          const uint32_t a_addr = ptx::smem_addr(sA + stage * kAStage);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // UMMA A = B^T slab: MN-major, 16 k-rows per step (2 KiB); n atoms 8 KiB apart.
            const uint64_t ad = ptx::smem_desc_sw128(b_addr + kk * 2048, kBBox, 1024);
            // UMMA B = tokens: K-major rows of 128 B, advance 32 B per 16 k.
            const uint64_t bd = ptx::smem_desc_sw128(a_addr + kk * 32, 16, 1024);
            ptx::mma_f16(d_tmem, ad, bd, kIdesc, (v > u || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit(&empty[stage]);
          any = true;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(&tfull[acc]);
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
        u = seg_end;
      }
      if (any) {
        ptx::mma_commit(mma_done);
        W.drain(mma_done, 0, kDrainNs);
      }
    }
  } else {
    // Epilogue: one thread per output column of the slab.
    const int q = warp & 3;
    const int n_local = q * 32 + lane;
    const int ep_tid = threadIdx.x - 64;
    uint32_t acc = 0, acc_phase = 0;
    long long u = u0;
    while (u < u1) {
      const int slab = static_cast<int>(u / per_slab);
      const long long seg_end = min(u1, static_cast<long long>(slab + 1) * per_slab);
      const bool failed = !W.wait(&tfull[acc], acc_phase);
      if (ptx::named_barrier_or(1, 128, failed)) break;  // the epilogue warps stop together
      ptx::tc_fence_after();
      uint32_t v[8], w[8];
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kTok;
      ptx::tmem_ld_32x32b_x8(taddr, v);
      ptx::tmem_ld_32x32b_x8(taddr + 8, w);
      ptx::tmem_ld_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tempty[acc]);

      const int slot = blockIdx.x + slab;
      float* part = p.partials + static_cast<long long>(slot) * kTok * kSlab;
#pragma unroll
      for (int t = 0; t < 8; ++t)
        if (t < p.M) part[t * kSlab + n_local] = __uint_as_float(v[t]);
#pragma unroll
      for (int t = 0; t < 8; ++t)
        if (t + 8 < p.M) part[(t + 8) * kSlab + n_local] = __uint_as_float(w[t]);
      __threadfence();
      ptx::named_barrier_sync(1, 128);
      const int first = owner_of(static_cast<long long>(slab) * per_slab, U, G);
      const int last = owner_of(static_cast<long long>(slab + 1) * per_slab - 1, U, G);
      if (ep_tid == 0) {
        const int prev = atomicAdd(&p.tickets[slab], 1);
        const int is_last = (prev == last - first) ? 1 : 0;
        if (is_last) p.tickets[slab] = 0;
        *bcast = is_last;
      }
      ptx::named_barrier_sync(1, 128);
      if (*bcast) {
        __threadfence();
        const int col = slab * kSlab + n_local;
        if (col < p.N) {
          for (int t = 0; t < p.M; ++t) {
            float s = 0.f;
            for (int c = first; c <= last; ++c)
              s += __ldcg(p.partials + (static_cast<long long>(c + slab) * kTok + t) * kSlab + n_local);
            for (int r = 0; r < p.R; ++r) {
              if (p.out_f32) {
                reinterpret_cast<float*>(p.out[r])[static_cast<long long>(t) * p.N + col] = s;
              } else {
                reinterpret_cast<uint16_t*>(p.out[r])[static_cast<long long>(t) * p.N + col] =
                    static_cast<uint16_t>(ptx::pack_bf16x2(s, 0.f) & 0xFFFFu);
              }
            }
          }
        }
      }
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
      u = seg_end;
    }
  }

  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

int gemv_smem_bytes() { return kSmemBytes; }

cudaError_t launch_gemv(const GemvParams& p, int grid, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(gemv_ar_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  gemv_ar_kernel<<<grid, kGemmThreads, kSmemBytes, st>>>(p);
  return cudaGetLastError();
}

}  // namespace fcc

// ---------------------------------------------------------------------------
// fcc_gemv_ar_static: the same GEMV + AllReduce kernel with its scratch (the
// per-CTA partial sums and the per-slab arrival tickets) in a fixed device
// array of this file instead of caller or pool memory, for callers that cannot
// allocate device memory.  The array lives on every GPU that loads the library
// until the process exits.
#include <mutex>

namespace fcc {
namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB in total
constexpr size_t kStaticTicketBytes = 4096;              // tickets: up to 1024 slabs
constexpr size_t kSlotBytes = size_t(kTok) * kSlab * 4;  // one partial: 16 x 128 f32

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
  if (opts != nullptr && opts->algo != FCC_ALGO_AUTO && opts->algo != FCC_ALGO_FUSED)
    return FCC_ERR_UNSUPPORTED;

  unsigned char* scratch = nullptr;
  int sms = 0;
  if ((s = static_scratch_for_current_device(&scratch, &sms)) != FCC_OK) return s;
  int* status = nullptr;
  if ((s = light_status_word(&status)) != FCC_OK) return s;

  const int slabs = static_cast<int>((N + kSlab - 1) / kSlab);
  const int kb = static_cast<int>((K + kBK - 1) / kBK);
  const long long units = static_cast<long long>(slabs) * R * kb;
  int grid = sms;
  if (opts != nullptr && opts->max_ctas > 0 && opts->max_ctas < grid) grid = opts->max_ctas;
  if (units < grid) grid = static_cast<int>(units);
  // Size limit of the static array: tickets for every slab, one partial slot
  // per (slab, contributing CTA) pair, of which there are at most slabs + grid.
  if (static_cast<size_t>(slabs) * 4 > kStaticTicketBytes ||
      static_cast<size_t>(slabs + grid) * kSlotBytes > kStaticScratchBytes - kStaticTicketBytes)
    return FCC_ERR_WORKSPACE;

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
  p.kb_per_rank = kb;
  p.slabs = slabs;
  p.units = units;
  p.out_f32 = out_dtype == FCC_F32 ? 1 : 0;
  p.tickets = reinterpret_cast<int*>(scratch);
  p.partials = reinterpret_cast<float*>(scratch + kStaticTicketBytes);
  p.status = status;
  p.timeout_ns = (opts != nullptr && opts->timeout_ns > 0)
                     ? static_cast<unsigned long long>(opts->timeout_ns)
                     : 1000ull * 1000 * 1000;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the tickets must start at zero.
  if (cudaMemsetAsync(p.tickets, 0, static_cast<size_t>(slabs) * 4, st) != cudaSuccess)
    return FCC_ERR_CUDA;
  if (launch_gemv(p, grid, st) != cudaSuccess) return FCC_ERR_CUDA;
  count_launch();
  return FCC_OK;
}

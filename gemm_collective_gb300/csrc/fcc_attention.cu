// fcc_attention.cu -- Ring attention over R sequence shards, tcgen05 (sm_103a).
//
// The mKernel article lists Ring Attention among its fused kernels: the
// sequence is split over R ranks, each rank's queries attend to the keys and
// values of every shard as the ring brings them round.  Here the R shards are
// buffers of one GPU and a CTA walks the key/value blocks in ring order
// (its own shard first, then r+1, r+2, ...), reading each block straight from
// the shard that holds it: the ring's transfers are the CTA's own loads.
//
// One CTA per (rank, head, 128-query tile); d = 128.  One pass over the
// key/value blocks of 128 positions, softmax with a lazily raised maximum:
//   S = Q K^T (tcgen05, M = N = K = 128, f32 in TMEM); each row keeps the
//   maximum m it exponentiates against and raises it only when a block's
//   maximum exceeds it by more than 8 (log2 units), so p = 2^(s c - m c)
//   stays <= 2^8; raising it rescales the row's O accumulator (in TMEM) and
//   its sum l by 2^(m_old c - m_new c) while no P V is in flight;
//   P (bf16) is written into TMEM over the S columns it came from and is the
//   A operand of O_c += P_c V_c (tcgen05, A from TMEM, O_c in TMEM, c the key
//   half); at the end, with m = max(m_0, m_1) and f_c = 2^(m_c c - m c),
//   O = (f_0 O_0 + f_1 O_1) / (f_0 l_0 + f_1 l_1).
//
// Warps: 0 = TMA producer (Q once, then a ring of four 32 KiB slots filled
// K_0, V_0, K_1, V_1, ...), 1 = MMA issue (S_{i+1} is issued before P_i is
// ready, so the tensor core works while the softmax runs; S_{i+2} reuses
// S_i's columns and is issued after P_i V_i, which the tensor core runs
// first), 2-9 = softmax and
// output (two warps per TMEM lane quarter of 32 query rows, one for each half
// of a block's key columns).  Each half keeps its own row maximum, sum and
// O accumulator, so the halves never wait on each other inside the walk;
// they are combined once, at the end.  Shared memory (128-byte swizzle throughout):
//   Q   [128 q][128 d]    K-major, two 64-column atoms of 16 KiB
//   K_j [128 keys][128 d] K-major (the B operand of Q K^T)
//   V_j [128 keys][128 d] MN-major B operand of P V: two 64-column atoms
// TMEM: S double buffer (2 x 128 columns; P_i in bf16 pairs over the first
// 32 columns of each half of S_i's) and O_0, O_1 (128 columns each).  No P in
// shared memory: the tensor core's shared-memory reads are Q, K and V only.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>

#include "fcc.h"
#include "fcc_internal.h"
#include "fcc_ptx.cuh"

namespace fcc {
namespace {

constexpr int kD = 128;                          // head dimension
constexpr int kBQ = 128;                         // query rows per CTA (MMA M)
constexpr int kBKV = 128;                        // keys per block
constexpr int kSlots = 4;                        // operand ring: 32 KiB slots (5, 6 measured the same)
constexpr uint32_t kAtom = 128 * 128;            // 16 KiB: [128 rows][64 bf16]
constexpr uint32_t kTile = 2 * kAtom;            // 32 KiB: [128][128] bf16
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256;       // S buffers at 0 and 128, O_0 at 256, O_1 at 384
constexpr float kRaise = 8.f;                    // raise the maximum past this (log2 units)
constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;
// S = Q K^T: both operands K-major.  O += P V: A K-major, B (V) MN-major.
constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(kBQ, kBKV, false, false);
constexpr uint32_t kIdescO = ptx::idesc_bf16_f32(kBQ, kD, false, true);
// Q, the ring, then the barriers and 4 words.
constexpr int kBars = 1 + 2 * kSlots + 2 + 1 + 1 + 2;
constexpr int kHalf = kBKV / 2;                  // key columns of a block per softmax warp
constexpr int kSoftmax = 8;                      // softmax warps: two per TMEM lane quarter
constexpr int kThreads = 64 + 32 * kSoftmax;     // warps 0-1 + the softmax warps
constexpr int kSmem = 1024 + kTile * (1 + kSlots) + kBars * 8 + 16;
static_assert(kSmem <= 232448, "shared memory per CTA");

struct AttnParams {
  CUtensorMap mapQ[FCC_MAX_RANKS];   // [S, H*d] bf16, box {64, 128}
  CUtensorMap mapK[FCC_MAX_RANKS];
  CUtensorMap mapV[FCC_MAX_RANKS];
  void* out[FCC_MAX_RANKS];          // [S, H, d]
  int R, S, H;
  int qtiles;                        // ceil(S / 128)
  int kvb;                           // key blocks per shard: ceil(S / 128)
  int causal;
  int out_f32;
  float scale_log2;                  // log2(e) / sqrt(d)
  int* status;
  unsigned long long timeout_ns;
};

// The key blocks a CTA visits, in ring order: block i of the walk is block
// i % kvb of shard (r + i / kvb) % R.  With the causal mask a block whose
// first position lies past the tile's last query is skipped (every role
// applies the same test, so the barrier counts agree).
struct Walk {
  int r, kvb, R, S, causal;
  long long q_last;                  // global position of the tile's last query row
  __device__ __forceinline__ int total() const { return R * kvb; }
  __device__ __forceinline__ int shard(int i) const { return (r + i / kvb) % R; }
  __device__ __forceinline__ int row0(int i) const { return (i % kvb) * kBKV; }
  __device__ __forceinline__ bool visible(int i) const {
    if (!causal) return true;
    return static_cast<long long>(shard(i)) * S + row0(i) <= q_last;
  }
};

// K-major SW128 operand of 128 rows x 128 elements (two 64-element atoms):
// descriptor of the 16-element K step kk.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int kk) {
  return ptx::smem_desc_sw128(base + (kk >> 2) * kAtom + (kk & 3) * 32, 16, 1024);
}
// MN-major SW128 operand (V: keys down, d across in two 64-column atoms 16 KiB
// apart): descriptor of the 16-key K step kk.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, int kk) {
  return ptx::smem_desc_sw128(base + kk * 2048, kAtom, 1024);
}


__global__ void __launch_bounds__(kThreads, 1) ring_attention_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sR = sQ + kTile;                    // ring slot s: sR + s * kTile
  uint64_t* bars = reinterpret_cast<uint64_t*>(sR + kSlots * kTile);
  uint64_t* q_full = bars;
  uint64_t* r_full = bars + 1;                 // [kSlots]
  uint64_t* r_empty = r_full + kSlots;         // [kSlots]
  uint64_t* s_full = r_empty + kSlots;         // [2]
  uint64_t* p_full = s_full + 2;
  uint64_t* p_empty = p_full + 1;
  uint64_t* o_full = p_empty + 1;
  uint64_t* mma_done = o_full + 1;             // kBars barriers in all
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // The halves' (m, l) rows, [2][2][128], over Q's tile: written only after
  // a softmax warp's walk, when every S = Q K^T has completed.
  float* red = reinterpret_cast<float*>(sQ);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA -> (rank, head, query tile), in reverse: with the causal mask the
  // last ranks' last tiles see the most keys, and launching them first keeps
  // them out of the final wave.
  const int bid = static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x);
  const int per_rank = p.H * p.qtiles;
  const int r = bid / per_rank;
  const int h = (bid - r * per_rank) / p.qtiles;
  const int qt = bid - r * per_rank - h * p.qtiles;
  Walk walk;
  walk.r = r;
  walk.kvb = p.kvb;
  walk.R = p.R;
  walk.S = p.S;
  walk.causal = p.causal;
  walk.q_last = static_cast<long long>(r) * p.S + min(p.S, (qt + 1) * kBQ) - 1;
  const int nwalk = walk.total();

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    for (int i = 0; i < kSlots; ++i) {
      ptx::mbar_init(&r_full[i], 1);
      ptx::mbar_init(&r_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) ptx::mbar_init(&s_full[i], 1);
    ptx::mbar_init(p_full, kSoftmax);
    ptx::mbar_init(p_empty, 1);
    ptx::mbar_init(o_full, 1);
    ptx::mbar_init(mma_done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&p.mapQ[r]);
    for (int i = 0; i < p.R; ++i) {
      ptx::tma_prefetch_desc(&p.mapK[i]);
      ptx::tma_prefetch_desc(&p.mapV[i]);
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
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t iss = 0, par = 0;                // slots with loads in flight (abort drain)
      bool ok = true;
      ptx::mbar_arrive_expect_tx(q_full, kTile);
      for (int b = 0; b < 2; ++b)
        ptx::tma_load_2d(sQ + b * kAtom, &p.mapQ[r], q_full, h * kD + 64 * b, qt * kBQ);
      int u = 0;                                // ring position: K_j at 2j, V_j at 2j + 1
      auto load = [&](const CUtensorMap* map, int y) -> bool {
        const int st = u % kSlots;
        const uint32_t ph = (u / kSlots) & 1u;
        if (!W.wait(&r_empty[st], ph ^ 1u)) return false;
        ptx::mbar_arrive_expect_tx(&r_full[st], kTile);
        for (int b = 0; b < 2; ++b)
          ptx::tma_load_2d(sR + st * kTile + b * kAtom, map, &r_full[st], h * kD + 64 * b, y);
        iss |= 1u << st;
        par = (par & ~(1u << st)) | (ph << st);
        ++u;
        return true;
      };
      for (int i = 0; i < nwalk && ok; ++i) {
        if (!walk.visible(i)) continue;
        const int sh = walk.shard(i);
        const int y = walk.row0(i);
        ok = load(&p.mapK[sh], y) && load(&p.mapV[sh], y);
      }
      if (*abort_flag) {
        W.drain(q_full, 0, kDrainNs);
        for (int st = 0; st < kSlots; ++st)
          if (iss & (1u << st)) W.drain(&r_full[st], (par >> st) & 1u, kDrainNs);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issue
    if (lane == 0) {
      bool ok = W.wait(q_full, 0);
      const uint32_t qa = ptx::smem_addr(sQ);
      int kpos = 0, vpos = 1, n = 0, m = 0;    // next key / value ring positions, S, P uses
      bool any = false;
      // S_n = Q K^T from the next key slot into S buffer n & 1; the key slot is
      // free once the product is done.  The buffer's last reader, P_{n-2} V,
      // was issued before (it waited for the softmax to finish with S_{n-2}),
      // and the tensor core runs this thread's MMAs in issue order.
      auto issue_s = [&]() -> bool {
        const int st = kpos % kSlots;
        if (!W.wait(&r_full[st], (kpos / kSlots) & 1u)) return false;
        const int b = n & 1;
        ptx::tc_fence_after();
        const uint32_t ka = ptx::smem_addr(sR + st * kTile);
        const uint32_t d_tmem = tmem_base + kColS + b * kBKV;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          ptx::mma_f16(d_tmem, desc_kmajor(qa, kk), desc_kmajor(ka, kk), kIdescS,
                       kk > 0 ? 1u : 0u);
        ptx::mma_commit(&s_full[b]);
        ptx::mma_commit(&r_empty[st]);
        ++n;
        kpos += 2;
        any = true;
        return true;
      };
      // O_c += P_m V_m over key half c, once the softmax warps have written
      // P_m into TMEM (and, where a row's maximum was raised, rescaled O_c).
      // Keys 16 kk of P_m: S buffer m & 1, half c = kk / 4, 8 columns a step.
      auto issue_pv = [&]() -> bool {
        const int st = vpos % kSlots;
        if (!W.wait(&r_full[st], (vpos / kSlots) & 1u)) return false;
        if (!W.wait(p_full, m & 1u)) return false;
        ptx::tc_fence_after();
        const uint32_t va = ptx::smem_addr(sR + st * kTile);
        const uint32_t p_tmem = tmem_base + kColS + (m & 1) * kBKV;
#pragma unroll
        for (int kk = 0; kk < kBKV / 16; ++kk)
          ptx::mma_f16_tmem_a(tmem_base + kColO + (kk / 4) * kD,
                              p_tmem + (kk / 4) * kHalf + (kk % 4) * 8, desc_mnmajor(va, kk),
                              kIdescO, (m > 0 || kk % 4 > 0) ? 1u : 0u);
        ptx::mma_commit(p_empty);
        ptx::mma_commit(&r_empty[st]);
        ++m;
        vpos += 2;
        return true;
      };
      // S_{i+1} goes in before P_i is awaited.
      bool pending = false;
      for (int i = 0; i < nwalk && ok; ++i) {
        if (!walk.visible(i)) continue;
        if (!(ok = issue_s())) break;
        if (pending && !(ok = issue_pv())) break;
        pending = true;
      }
      if (ok && pending) ok = issue_pv();
      if (ok) ptx::mma_commit(o_full);
      if (any) {
        ptx::mma_commit(mma_done);
        W.drain(mma_done, 0, kDrainNs);
      }
    }
  } else {
    // ------------------------------------------------- softmax and output
    // Warp w reads TMEM lane quarter w % 4 (32 query rows) and key columns
    // [64 c, 64 c + 64) of each block, c = (w - 2) / 4; its rows' maximum m_c,
    // sum l_c and accumulator O_c (TMEM columns kColO + 128 c) cover those keys.
    const int q = warp & 3;                     // TMEM lane quarter of this warp
    const int half = (warp - 2) >> 2;           // key column half
    const int c0 = half * kHalf;
    const int row = q * 32 + lane;              // query row of the tile
    const long long qpos = static_cast<long long>(r) * p.S + qt * kBQ + row;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t o_own = lane_addr + kColO + half * kD;
    // Lane 0 waits, the warp follows (the warp stops as one).
    auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
      int good = 1;
      if (lane == 0) good = W.wait(bar, parity) ? 1 : 0;
      return __shfl_sync(0xffffffffu, good, 0) != 0;
    };
    // The last valid column of block i for this row (keys past the shard's
    // end, and with the mask past the row's own position, are out).
    auto last_col = [&](int i) -> int {
      const int r0 = walk.row0(i);
      int c = min(kBKV, p.S - r0) - 1;
      if (p.causal) {
        const long long lim = qpos - (static_cast<long long>(walk.shard(i)) * p.S + r0);
        c = static_cast<int>(min(static_cast<long long>(c), lim));
      }
      return c;                                 // -1: nothing valid
    };
    bool ok = true;
    int n = 0;                                  // S buffers consumed (= P buffers written)
    float m_used = -INFINITY;                   // the maximum this half's p is taken against
    float l = 0.f;                              // this half's sum of p
    for (int i = 0; i < nwalk; ++i) {
      if (!walk.visible(i)) continue;
      const int b = n & 1;
      // A failed wait ends this warp's walk; the others' waits then end on
      // the abort flag or their own limit (no barrier inside the walk).
      if (!wait_warp(&s_full[b], (n >> 1) & 1u)) {
        ok = false;
        break;
      }
      uint32_t v[kHalf];
      const int cmax = last_col(i) - c0;        // in this half's columns
      ptx::tc_fence_after();
      ptx::tmem_ld_32x32b_x32(lane_addr + kColS + b * kBKV + c0,
                              *reinterpret_cast<uint32_t(*)[32]>(v));
      ptx::tmem_ld_32x32b_x32(lane_addr + kColS + b * kBKV + c0 + 32,
                              *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      ptx::tmem_ld_wait();
      float bm = -INFINITY;
      if (cmax >= kHalf - 1) {
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // four short chains
#pragma unroll
        for (int k = 0; k < kHalf; k += 2)
          mx[(k / 2) & 3] = ptx::max3(mx[(k / 2) & 3], __uint_as_float(v[k]),
                                      __uint_as_float(v[k + 1]));
        bm = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      } else {
#pragma unroll
        for (int k = 0; k < kHalf; ++k)
          if (k <= cmax) bm = fmaxf(bm, __uint_as_float(v[k]));
      }
      // Raise the maximum when this block's exceeds it by more than kRaise.
      const bool raise = bm * p.scale_log2 > m_used * p.scale_log2 + kRaise;
      const float m_new = raise ? bm : m_used;
      const float corr = ptx::ex2_approx((m_used - m_new) * p.scale_log2);  // 0 at the start
      if (raise) l *= (m_used == -INFINITY) ? 0.f : corr;
      m_used = m_new;
      const float msc = m_used * p.scale_log2;
      uint32_t pk[kHalf / 2];                   // bf16 pairs of p
      float ls[4] = {0.f, 0.f, 0.f, 0.f};       // four partial sums of this block's p
      if (cmax >= kHalf - 1) {
        const uint64_t c2 = ptx::f32x2_pack(p.scale_log2, p.scale_log2);
        const uint64_t n2 = ptx::f32x2_pack(-msc, -msc);
        uint64_t s2[4] = {0, 0, 0, 0};          // four chains of packed partial sums
#pragma unroll
        for (int k = 0; k < kHalf; k += 2) {
          float y0, y1;
          const uint64_t x2 = ptx::f32x2_pack(__uint_as_float(v[k]), __uint_as_float(v[k + 1]));
          ptx::f32x2_unpack(ptx::f32x2_fma(x2, c2, n2), y0, y1);   // s c - m c, two at once
          const float p0 = ptx::ex2_approx(y0);
          const float p1 = ptx::ex2_approx(y1);
          s2[(k / 2) & 3] = ptx::f32x2_add(s2[(k / 2) & 3], ptx::f32x2_pack(p0, p1));
          pk[k / 2] = ptx::pack_bf16x2(p0, p1);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float a0, a1;
          ptx::f32x2_unpack(s2[j], a0, a1);
          ls[j] = a0 + a1;
        }
      } else {
#pragma unroll
        for (int k = 0; k < kHalf; k += 2) {
          float p0 = ptx::ex2_approx(fmaf(__uint_as_float(v[k]), p.scale_log2, -msc));
          float p1 = ptx::ex2_approx(fmaf(__uint_as_float(v[k + 1]), p.scale_log2, -msc));
          if (k > cmax) p0 = 0.f;
          if (k + 1 > cmax) p1 = 0.f;
          ls[(k / 2) & 3] += p0 + p1;
          pk[k / 2] = ptx::pack_bf16x2(p0, p1);
        }
      }
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      // P_n over the first 32 columns of this half of S_n (read above; the
      // other half's warp reads and writes only its own columns).
      ptx::tmem_st_32x32b_x32(lane_addr + kColS + b * kBKV + c0, pk);
      // Rows whose maximum was raised rescale their O_c (after the first
      // block, when it holds earlier blocks' sums) once P_{n-1} V, the last
      // product on O_c, is done.  P_{n-2} V finished before S_n did and P_n V
      // waits for this warp, so the wait sees phase n - 1 of p_empty or n.
      if (n > 0 && __any_sync(0xffffffffu, raise)) {
        if (!wait_warp(p_empty, (n & 1u) ^ 1u)) {
          ptx::tmem_st_wait();
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const float f = raise ? corr : 1.f;
#pragma unroll 1
        for (int c = 0; c < kD; c += 32) {
          uint32_t o[32];
          ptx::tmem_ld_32x32b_x32(o_own + c, o);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
          ptx::tmem_st_32x32b_x32(o_own + c, o);
        }
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();                   // the tensor core reads P_n, adds to O_c
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(p_full);
      ++n;
    }
    // Combine the halves: each publishes its (m_c, l_c); both form the same
    // factors f_c = 2^(m_c c - m c) and denominator f_0 l_0 + f_1 l_1.
    red[half * kBQ + row] = m_used;
    red[(2 + half) * kBQ + row] = l;
    if (ptx::named_barrier_or(1, 32 * kSoftmax, !ok)) ok = false;
    const float m0 = red[row], m1 = red[kBQ + row];
    const float l0 = red[2 * kBQ + row], l1 = red[3 * kBQ + row];
    const float mm = fmaxf(m0, m1);
    const float f0 = m0 == -INFINITY ? 0.f : ptx::ex2_approx((m0 - mm) * p.scale_log2);
    const float f1 = m1 == -INFINITY ? 0.f : ptx::ex2_approx((m1 - mm) * p.scale_log2);
    // Output: this half's 64 columns of (f_0 O_0 + f_1 O_1) / l, for rows
    // inside the shard.
    if (ok && wait_warp(o_full, 0)) {
      ptx::tc_fence_after();
      const int grow = qt * kBQ + row;
      const float inv = 1.f / (l0 * f0 + l1 * f1);
      const float g0 = f0 * inv, g1 = f1 * inv;
      char* dst = static_cast<char*>(p.out[r]) +
                  (static_cast<long long>(grow) * p.H + h) * kD * (p.out_f32 ? 4 : 2);
#pragma unroll 1
      for (int c = c0; c < c0 + kHalf; c += 32) {
        uint32_t a[32], v[32];
        ptx::tmem_ld_32x32b_x32(lane_addr + kColO + c, a);
        ptx::tmem_ld_32x32b_x32(lane_addr + kColO + kD + c, v);
        ptx::tmem_ld_wait();
        float x[32];
#pragma unroll
        for (int k = 0; k < 32; ++k)
          x[k] = fmaf(__uint_as_float(a[k]), g0, __uint_as_float(v[k]) * g1);
        if (grow < p.S) {
          if (p.out_f32) {
            float4* o = reinterpret_cast<float4*>(dst) + c / 4;
#pragma unroll
            for (int k = 0; k < 32; k += 4) o[k / 4] = make_float4(x[k], x[k + 1], x[k + 2], x[k + 3]);
          } else {
            uint4* o = reinterpret_cast<uint4*>(dst) + c / 8;
#pragma unroll
            for (int k = 0; k < 32; k += 8) {
              uint4 w;
              w.x = ptx::pack_bf16x2(x[k], x[k + 1]);
              w.y = ptx::pack_bf16x2(x[k + 2], x[k + 3]);
              w.z = ptx::pack_bf16x2(x[k + 4], x[k + 5]);
              w.w = ptx::pack_bf16x2(x[k + 6], x[k + 7]);
              o[k / 8] = w;
            }
          }
        }
      }
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
}  // namespace fcc

using namespace fcc;

extern "C" {

fcc_status fcc_ring_attention(int R, const void* const* Q, const void* const* K,
                              const void* const* V, void* const* O, int64_t S, int H, int64_t d,
                              int causal, fcc_dtype in, fcc_dtype out_dtype, const fcc_opts* opts,
                              fcc_stream_t stream) {
  if (R < 1 || R > FCC_MAX_RANKS || S < 1 || S > (1ll << 30) || H < 1 || H > 1024 || d < 1)
    return FCC_ERR_INVALID;
  if (static_cast<int64_t>(R) * H * ((S + kBQ - 1) / kBQ) > (1ll << 31) - 1)
    return FCC_ERR_INVALID;
  if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr) return FCC_ERR_INVALID;
  for (int r = 0; r < R; ++r)
    for (const void* ptr : {Q[r], K[r], V[r], static_cast<const void*>(O[r])})
      if (ptr == nullptr || (reinterpret_cast<uintptr_t>(ptr) & 15u)) return FCC_ERR_INVALID;
  if ((in != FCC_BF16 && in != FCC_F16 && in != FCC_F32) ||
      (out_dtype != FCC_BF16 && out_dtype != FCC_F16 && out_dtype != FCC_F32))
    return FCC_ERR_INVALID;
  if (in != FCC_BF16 || out_dtype == FCC_F16 || d != kD) return FCC_ERR_UNSUPPORTED;
  if (opts != nullptr && opts->algo != FCC_ALGO_AUTO && opts->algo != FCC_ALGO_FUSED)
    return FCC_ERR_UNSUPPORTED;

  void* ws = nullptr;
  int* status = nullptr;
  int sms = 0;
  unsigned long long timeout_ns = 0;
  fcc_status s = internal_prepare(opts, 0, &ws, &status, &sms, &timeout_ns);
  if (s != FCC_OK) return s;
  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  for (int r = 0; r < R; ++r) {
    if ((s = internal_make_map(&p.mapQ[r], Q[r], S, static_cast<int64_t>(H) * kD, kBQ)) != FCC_OK ||
        (s = internal_make_map(&p.mapK[r], K[r], S, static_cast<int64_t>(H) * kD, kBKV)) != FCC_OK ||
        (s = internal_make_map(&p.mapV[r], V[r], S, static_cast<int64_t>(H) * kD, kBKV)) != FCC_OK)
      return s;
    p.out[r] = O[r];
  }
  p.R = R;
  p.S = static_cast<int>(S);
  p.H = H;
  p.qtiles = static_cast<int>((S + kBQ - 1) / kBQ);
  p.kvb = static_cast<int>((S + kBKV - 1) / kBKV);
  p.causal = causal ? 1 : 0;
  p.out_f32 = out_dtype == FCC_F32 ? 1 : 0;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(kD)));
  p.status = status;
  p.timeout_ns = timeout_ns;

  if (cudaFuncSetAttribute(ring_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmem) != cudaSuccess)
    return FCC_ERR_CUDA;
  const unsigned grid = static_cast<unsigned>(R * H * p.qtiles);
  ring_attention_kernel<<<grid, kThreads, kSmem, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  if (cudaGetLastError() != cudaSuccess) return FCC_ERR_CUDA;
  bump_launch_count(1);
  return FCC_OK;
}

}  // extern "C"

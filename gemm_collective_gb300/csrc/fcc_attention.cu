// fcc_attention.cu -- Ring attention over R sequence shards, tcgen05 (sm_103a).
//
// The mKernel article lists Ring Attention among its fused kernels: the
// sequence is split over R ranks, each rank's queries attend to the keys and
// values of every shard as the ring brings them round.  Here the R shards are
// buffers of one GPU and a CTA walks the key/value blocks in ring order
// (its own shard first, then r+1, r+2, ...), reading each block straight from
// the shard that holds it: the ring's transfers are the CTA's own loads.
//
// One CTA per (rank, head, pair of 128-query tiles A and B); d = 128.  One
// pass over the key/value blocks of 128 positions, softmax with a lazily
// raised maximum:
//   S_t = Q_t K^T (tcgen05, M = N = K = 128, f32 in TMEM) for tile t; each
//   row keeps the maximum m it exponentiates against and raises it only when
//   a block's maximum exceeds it by more than 8 (log2 units), so
//   p = 2^(s c - m c) stays <= 2^8; raising it rescales the row's O_t
//   accumulator (in TMEM) and its sum l by 2^(m_old c - m_new c);
//   P (bf16) is written into TMEM over the first 64 columns of S_t and is the
//   A operand of O_t += P V (tcgen05, A from TMEM); at the end O_t / l.
// Past a tile's first block, a whole (unmasked) block is exponentiated
// against the current maximum 32 columns at a time while the next 32 come
// from TMEM, its maximum taken along the way; only a block whose maximum
// calls for a raise starts over from S (still in TMEM) in the general form.
// One softmax thread owns one query row and all 128 columns of a block, so
// no two threads share a row's maximum or sum.  The two tiles take turns on
// the tensor core: while tile A's softmax runs, the tensor core computes tile
// B's S and P V, and the other way round.
//
// Warps: 0 = TMA producer (Q_A and Q_B once, then a ring of four 32 KiB
// slots filled K_0, V_0, K_1, V_1, ...), 1 = MMA issue, in the order
// P_A(j-1) V, S_A(j), P_B(j-1) V, S_B(j) for each block j (a tile's next S is
// issued after its P V, and the tensor core runs one thread's MMAs in issue
// order, so S_t(j) may reuse the columns P_t(j-1) occupied and, once S_t(j)
// is complete, O_t holds no P V in flight), 2-5 = softmax and output of tile
// A, 6-9 = tile B (warp w reads TMEM lane quarter w % 4: 32 query rows).
// Shared memory (128-byte swizzle throughout):
//   Q_t [128 q][128 d]    K-major, two 64-column atoms of 16 KiB
//   K_j [128 keys][128 d] K-major (the B operand of Q K^T)
//   V_j [128 keys][128 d] MN-major B operand of P V: two 64-column atoms
// TMEM: S_A, S_B at columns 0 and 128 (P_t in bf16 pairs over the first 64
// of S_t's), O_A, O_B at 256 and 384.
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
constexpr int kBQ = 128;                         // query rows per tile (MMA M)
constexpr int kBKV = 128;                        // keys per block
constexpr int kSlots = 4;                        // operand ring: 32 KiB slots
constexpr uint32_t kAtom = 128 * 128;            // 16 KiB: [128 rows][64 bf16]
constexpr uint32_t kTile = 2 * kAtom;            // 32 KiB: [128][128] bf16
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;                  // S_t at 128 t, O_t at 256 + 128 t
constexpr float kRaise = 8.f;                    // raise the maximum past this (log2 units)
constexpr uint64_t kDrainNs = 50ull * 1000 * 1000;
// S = Q K^T: both operands K-major.  O += P V: A K-major, B (V) MN-major.
constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(kBQ, kBKV, false, false);
constexpr uint32_t kIdescO = ptx::idesc_bf16_f32(kBQ, kD, false, true);
// Q_A, Q_B, the ring, then the barriers and 4 words.
constexpr int kBars = 1 + 2 * kSlots + 2 + 2 + 1 + 1;
constexpr int kThreads = 320;                    // warps 0-1 + two groups of four softmax warps
constexpr int kSmem = 1024 + kTile * (2 + kSlots) + kBars * 8 + 16;
static_assert(kSmem <= 232448, "shared memory per CTA");

struct AttnParams {
  CUtensorMap mapQ[FCC_MAX_RANKS];   // [S, H*d] bf16, box {64, 128}
  CUtensorMap mapK[FCC_MAX_RANKS];
  CUtensorMap mapV[FCC_MAX_RANKS];
  void* out[FCC_MAX_RANKS];          // [S, H, d]
  int R, S, H;
  int qtiles;                        // ceil(S / 128)
  int qpairs;                        // ceil(qtiles / 2)
  int kvb;                           // key blocks per shard: ceil(S / 128)
  int causal;
  int out_f32;
  float scale_log2;                  // log2(e) / sqrt(d)
  int* status;
  unsigned long long timeout_ns;
};

// The key blocks a CTA visits, in ring order: block i of the walk is block
// i % kvb of shard (r + i / kvb) % R.  Tile t sees block i unless the tile
// lies past the shard's end or, with the causal mask, the block's first
// position lies past the tile's last query.  In ring order those blocks form
// two runs: the own shard's first blocks (walk indices [0, own_end[t]), up to
// the tile's diagonal) and, from walk index other_begin on, the shards before
// this one (causal: shards 0 .. r-1, at walk indices [(R - r) kvb, R kvb);
// without the mask every block, other_begin = kvb).  Every role walks only
// those runs and applies the same test, so the barrier counts agree; the
// blocks in between (the shards past this one) cost nothing.
struct Walk {
  int r, kvb, R, S, causal;
  bool valid[2];                     // the tile holds rows of the shard
  long long q_last[2];               // global position of the tile's last query row
  int own_end[2];                    // own-shard blocks [0, own_end[t]) are visible to tile t
  int other_begin;                   // walk indices from here on are visible to valid tiles
  __device__ __forceinline__ int total() const { return R * kvb; }
  __device__ __forceinline__ int shard(int i) const { return (r + i / kvb) % R; }
  __device__ __forceinline__ int row0(int i) const { return (i % kvb) * kBKV; }
  __device__ __forceinline__ bool visible(int i, int t) const {
    return valid[t] && (i < own_end[t] || i >= other_begin);
  }
  __device__ __forceinline__ bool visible_a(int i) const { return visible(i, 0); }
  __device__ __forceinline__ bool visible_b(int i) const { return visible(i, 1); }
  // The walk index after i among the blocks visible to a tile whose own-shard
  // run ends at `end` (for both tiles: the larger end).
  __device__ __forceinline__ int next(int i, int end) const {
    return (i + 1 == end && end < other_begin) ? other_begin : i + 1;
  }
  __device__ __forceinline__ int first(int end) const { return end > 0 ? 0 : other_begin; }
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

// tcgen05.wait::ld tied to the 32 registers one 32x32b.x32 load filled, so
// the compiler keeps every use of them after the wait while arithmetic on
// other registers may run between the load and the wait.
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&v)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                 "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                 "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]),
                 "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]),
                 "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]),
                 "+r"(v[30]), "+r"(v[31])
               :
               : "memory");
}

__global__ void __launch_bounds__(kThreads, 1) ring_attention_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                          // Q_t: sQ + t * kTile
  uint8_t* sR = sQ + 2 * kTile;                // ring slot s: sR + s * kTile
  uint64_t* bars = reinterpret_cast<uint64_t*>(sR + kSlots * kTile);
  uint64_t* q_full = bars;
  uint64_t* r_full = bars + 1;                 // [kSlots]
  uint64_t* r_empty = r_full + kSlots;         // [kSlots]
  uint64_t* s_full = r_empty + kSlots;         // [2]: S_t complete
  uint64_t* p_full = s_full + 2;               // [2]: P_t written (and O_t rescaled)
  uint64_t* o_full = p_full + 2;
  uint64_t* mma_done = o_full + 1;             // kBars barriers in all
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA -> (rank, head, tile pair), in reverse: with the causal mask the
  // last ranks' last tiles see the most keys, and launching them first keeps
  // them out of the final wave.
  const int bid = static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x);
  const int per_rank = p.H * p.qpairs;
  const int r = bid / per_rank;
  const int h = (bid - r * per_rank) / p.qpairs;
  const int qp = bid - r * per_rank - h * p.qpairs;
  Walk walk;
  walk.r = r;
  walk.kvb = p.kvb;
  walk.R = p.R;
  walk.S = p.S;
  walk.causal = p.causal;
  for (int t = 0; t < 2; ++t) {
    const int qt = 2 * qp + t;
    const int last_local = min(p.S, (qt + 1) * kBQ) - 1;  // the tile's last query row
    walk.valid[t] = qt < p.qtiles;
    walk.q_last[t] = static_cast<long long>(r) * p.S + last_local;
    walk.own_end[t] = !walk.valid[t] ? 0 : (p.causal ? min(p.kvb, last_local / kBKV + 1) : p.kvb);
  }
  walk.other_begin = p.causal ? (p.R - r) * p.kvb : p.kvb;
  const int nwalk = walk.total();
  const int own_end_u = max(walk.own_end[0], walk.own_end[1]);  // either tile's run

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    for (int i = 0; i < kSlots; ++i) {
      ptx::mbar_init(&r_full[i], 1);
      ptx::mbar_init(&r_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(&s_full[t], 1);
      ptx::mbar_init(&p_full[t], 4);           // the tile's four softmax warps
    }
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
      const int ntiles = walk.valid[1] ? 2 : 1;
      ptx::mbar_arrive_expect_tx(q_full, kTile * ntiles);
      for (int t = 0; t < ntiles; ++t)
        for (int b = 0; b < 2; ++b)
          ptx::tma_load_2d(sQ + t * kTile + b * kAtom, &p.mapQ[r], q_full, h * kD + 64 * b,
                           (2 * qp + t) * kBQ);
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
      for (int i = walk.first(own_end_u); i < nwalk && ok; i = walk.next(i, own_end_u)) {
        if (!walk.visible_a(i) && !walk.visible_b(i)) continue;
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
      int np[2] = {0, 0};                       // P V products issued per tile
      int pend[2] = {-1, -1};                   // block (walk ordinal) whose P V is next
      bool any = false;
      // S_t = Q_t K_j^T from the key slot of walk ordinal j.
      auto issue_s = [&](int t, int j) {
        const uint32_t qa = ptx::smem_addr(sQ + t * kTile);
        const uint32_t ka = ptx::smem_addr(sR + ((2 * j) % kSlots) * kTile);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          ptx::mma_f16(tmem_base + t * kBKV, desc_kmajor(qa, kk), desc_kmajor(ka, kk), kIdescS,
                       kk > 0 ? 1u : 0u);
        ptx::mma_commit(&s_full[t]);
        any = true;
      };
      // O_t += P_t V_j once tile t's softmax warps have written P_t (and
      // rescaled O_t where a row's maximum was raised).  P_t: 8 TMEM columns
      // per 16 keys.
      auto issue_pv = [&](int t, int j) -> bool {
        const int pos = 2 * j + 1;
        if (!W.wait(&r_full[pos % kSlots], (pos / kSlots) & 1u)) return false;
        if (!W.wait(&p_full[t], np[t] & 1u)) return false;
        ptx::tc_fence_after();
        const uint32_t va = ptx::smem_addr(sR + (pos % kSlots) * kTile);
#pragma unroll
        for (int kk = 0; kk < kBKV / 16; ++kk)
          ptx::mma_f16_tmem_a(tmem_base + kColO + t * kD, tmem_base + t * kBKV + kk * 8,
                              desc_mnmajor(va, kk), kIdescO, (np[t] > 0 || kk > 0) ? 1u : 0u);
        ++np[t];
        return true;
      };
      int j = 0;                                // walk ordinal of the blocks either tile sees
      for (int i = walk.first(own_end_u); i < nwalk && ok; i = walk.next(i, own_end_u)) {
        const bool vis_a = walk.visible_a(i), vis_b = walk.visible_b(i);
        if (!vis_a && !vis_b) continue;
        const int pos = 2 * j;
        if (!(ok = W.wait(&r_full[pos % kSlots], (pos / kSlots) & 1u))) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok) break;
          if (pend[t] >= 0) {
            ok = issue_pv(t, pend[t]);
            pend[t] = -1;
          }
          if (ok && (t == 0 ? vis_a : vis_b)) {
            issue_s(t, j);
            pend[t] = j;
          }
        }
        if (!ok) break;
        // K_j is free once both tiles' S are done; V_{j-1} once both P V are.
        ptx::mma_commit(&r_empty[pos % kSlots]);
        if (j > 0) ptx::mma_commit(&r_empty[(pos - 1) % kSlots]);
        ++j;
      }
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (ok && pend[t] >= 0) ok = issue_pv(t, pend[t]);
      if (ok) ptx::mma_commit(o_full);
      if (any) {
        ptx::mma_commit(mma_done);
        W.drain(mma_done, 0, kDrainNs);
      }
    }
  } else {
    // ------------------------------------------------- softmax and output
    // Warp w serves tile (w - 2) / 4 and TMEM lane quarter w % 4; its thread
    // `lane` owns query row 32 (w % 4) + lane of the tile: all 128 columns of
    // each block, its maximum m, its sum l and its row of O_t.
    const int t = (warp - 2) >> 2;
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int grow = (2 * qp + t) * kBQ + row;  // row within the shard
    const long long qpos = static_cast<long long>(r) * p.S + grow;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t s_addr = lane_addr + t * kBKV;          // S_t, and P_t over its first 64
    const uint32_t o_addr = lane_addr + kColO + t * kD;    // O_t
    const bool t_valid = t == 0 ? walk.valid[0] : walk.valid[1];
    const int t_end = t == 0 ? walk.own_end[0] : walk.own_end[1];
    // The whole warp waits (every lane polls the barrier, so the warp never
    // splits around a one-lane spin: 3.53 -> 3.37 ms without the mask, 1.86 ->
    // 1.71 ms with it), and stops as one.
    auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, W.wait(bar, parity) ? 1 : 0) != 0;
    };
    // The last valid column of the block at row r0 of shard sh (keys past the
    // shard's end, and with the mask past the row's own position, are out).
    auto last_col = [&](int sh, int r0) -> int {
      int c = min(kBKV, p.S - r0) - 1;
      if (p.causal) {
        const long long lim = qpos - (static_cast<long long>(sh) * p.S + r0);
        c = static_cast<int>(min(static_cast<long long>(c), lim));
      }
      return c;                                 // -1: nothing valid
    };
    bool ok = true;
    int n = 0;                                  // blocks of this tile done
    float m_used = -INFINITY;                   // the maximum p is taken against
    float l = 0.f;                              // the row's sum of p
    // The walk visits only this tile's visible blocks (next() skips the
    // rest); the block's shard and row follow the walk index step by step.
    const int i0 = t_valid ? walk.first(t_end) : nwalk;
    int sh = i0 < nwalk ? walk.shard(i0) : 0, r0 = i0 < nwalk ? walk.row0(i0) : 0;
    for (int i = i0; i < nwalk; ) {
      // A failed wait ends this warp's walk; the others' waits then end on
      // the abort flag or their own limit (no barrier inside the walk).
      if (!wait_warp(&s_full[t], n & 1u)) {
        ok = false;
        break;
      }
      const int cmax = last_col(sh, r0);
      uint32_t vb[2][32];                       // two 32-column chunks of S in flight
      bool done = false;
      ptx::tc_fence_after();
      // The form is chosen for the whole warp (the TMEM loads and stores
      // and the vote below are warp-collective): with the mask, cmax differs
      // from row to row on a diagonal block.
      if (n > 0 && __all_sync(0xffffffffu, cmax >= kBKV - 1)) {
        // Speculative form, for a whole block once the row has a maximum:
        // each 32-column chunk of S is exponentiated against the current
        // maximum while the next chunk is still coming from TMEM, and the
        // block's maximum is taken along the way.  P is stored only if no
        // row's block maximum exceeds its current one by more than kRaise
        // (rare past a tile's first block); otherwise the general form below
        // starts over from S, still intact in TMEM, with the same result.
        const float msc = m_used * p.scale_log2;
        const uint64_t c2 = ptx::f32x2_pack(p.scale_log2, p.scale_log2);
        const uint64_t n2 = ptx::f32x2_pack(-msc, -msc);
        uint64_t s2[4] = {0, 0, 0, 0};          // four chains of packed partial sums (a half)
        float ls[4] = {0.f, 0.f, 0.f, 0.f};     // the halves' sums, as the general form adds them
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        uint32_t pk[64];                        // bf16 pairs of p, the whole block
        ptx::tmem_ld_32x32b_x32(s_addr, vb[0]);
        tmem_ld_wait_regs(vb[0]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (c < 3) ptx::tmem_ld_32x32b_x32(s_addr + 32 * (c + 1), vb[(c + 1) & 1]);
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            const float x0 = __uint_as_float(vb[c & 1][k]), x1 = __uint_as_float(vb[c & 1][k + 1]);
            mx[(k / 2) & 3] = ptx::max3(mx[(k / 2) & 3], x0, x1);
            float y0, y1;
            ptx::f32x2_unpack(ptx::f32x2_fma(ptx::f32x2_pack(x0, x1), c2, n2), y0, y1);
            const float p0 = ptx::ex2_approx(y0);
            const float p1 = ptx::ex2_approx(y1);
            s2[(k / 2) & 3] = ptx::f32x2_add(s2[(k / 2) & 3], ptx::f32x2_pack(p0, p1));
            pk[16 * c + k / 2] = ptx::pack_bf16x2(p0, p1);
          }
          if (c & 1) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              float a0, a1;
              ptx::f32x2_unpack(s2[j], a0, a1);
              ls[j] += a0 + a1;
              s2[j] = 0;
            }
          }
          if (c < 3) tmem_ld_wait_regs(vb[(c + 1) & 1]);
        }
        const float bm = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        if (!__any_sync(0xffffffffu, bm * p.scale_log2 > msc + kRaise)) {
          ptx::tmem_st_32x32b_x32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(pk));
          ptx::tmem_st_32x32b_x32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(pk + 32));
          l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
          done = true;
        }
      }
      if (!done) {  // warp-uniform: decided by __any_sync
        // General form: the block's maximum over the valid columns, then the
        // exponentials, in two passes over S in TMEM (a chunk at a time).
        float bm = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          ptx::tmem_ld_32x32b_x32(s_addr + 32 * c, vb[c & 1]);
          tmem_ld_wait_regs(vb[c & 1]);
          if (cmax >= kBKV - 1) {
            float mx[4] = {bm, -INFINITY, -INFINITY, -INFINITY};  // four short chains
#pragma unroll
            for (int k = 0; k < 32; k += 2)
              mx[(k / 2) & 3] = ptx::max3(mx[(k / 2) & 3], __uint_as_float(vb[c & 1][k]),
                                          __uint_as_float(vb[c & 1][k + 1]));
            bm = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k)
              if (32 * c + k <= cmax) bm = fmaxf(bm, __uint_as_float(vb[c & 1][k]));
          }
        }
        // Raise the maximum when this block's exceeds it by more than kRaise.
        const bool raise = bm * p.scale_log2 > m_used * p.scale_log2 + kRaise;
        const float m_new = raise ? bm : m_used;
        const float corr = ptx::ex2_approx((m_used - m_new) * p.scale_log2);  // 0 at the start
        if (raise) l *= (m_used == -INFINITY) ? 0.f : corr;
        m_used = m_new;
        const float msc = m_used * p.scale_log2;
        float ls[4] = {0.f, 0.f, 0.f, 0.f};     // four partial sums of this block's p
        // Two halves of 64 scores; each half's 32 bf16 pairs of p go to TMEM
        // over columns its scores came from (read just before).
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          ptx::tmem_ld_32x32b_x32(s_addr + 64 * hf, vb[0]);
          ptx::tmem_ld_32x32b_x32(s_addr + 64 * hf + 32, vb[1]);
          tmem_ld_wait_regs(vb[0]);
          tmem_ld_wait_regs(vb[1]);
          uint32_t pk[32];                      // bf16 pairs of p
          if (cmax >= kBKV - 1) {
            const uint64_t c2 = ptx::f32x2_pack(p.scale_log2, p.scale_log2);
            const uint64_t n2 = ptx::f32x2_pack(-msc, -msc);
            uint64_t s2[4] = {0, 0, 0, 0};      // four chains of packed partial sums
#pragma unroll
            for (int k = 0; k < 64; k += 2) {
              float y0, y1;
              const uint64_t x2 = ptx::f32x2_pack(__uint_as_float(vb[k >> 5][k & 31]),
                                                  __uint_as_float(vb[k >> 5][(k & 31) + 1]));
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
              ls[j] += a0 + a1;
            }
          } else {
#pragma unroll
            for (int k = 0; k < 64; k += 2) {
              const int kv = 64 * hf + k;
              float p0 = ptx::ex2_approx(fmaf(__uint_as_float(vb[k >> 5][k & 31]), p.scale_log2, -msc));
              float p1 = ptx::ex2_approx(fmaf(__uint_as_float(vb[k >> 5][(k & 31) + 1]), p.scale_log2, -msc));
              if (kv > cmax) p0 = 0.f;
              if (kv + 1 > cmax) p1 = 0.f;
              ls[(k / 2) & 3] += p0 + p1;
              pk[k / 2] = ptx::pack_bf16x2(p0, p1);
            }
          }
          ptx::tmem_st_32x32b_x32(s_addr + 32 * hf, pk);
        }
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        // Rows whose maximum was raised rescale their O_t (after the first
        // block, when it holds earlier blocks' sums).  S_t of this block was
        // issued after the last P_t V, so O_t has no product in flight until
        // P_t is signalled.
        if (n > 0 && __any_sync(0xffffffffu, raise)) {
          const float f = raise ? corr : 1.f;
#pragma unroll 1
          for (int c = 0; c < kD; c += 32) {
            uint32_t o[32];
            ptx::tmem_ld_32x32b_x32(o_addr + c, o);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
            ptx::tmem_st_32x32b_x32(o_addr + c, o);
          }
        }
      }
      ptx::tmem_st_wait();                      // P_t (and a rescaled O_t) in place
      ptx::tc_fence_before();                   // the tensor core reads P_t, adds to O_t
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&p_full[t]);
      ++n;
      const int i_next = walk.next(i, t_end);
      if (i_next == i + 1) {
        r0 += kBKV;
        if (r0 >= walk.kvb * kBKV) {
          r0 = 0;
          sh = sh + 1 == p.R ? 0 : sh + 1;
        }
      } else if (i_next < nwalk) {
        sh = walk.shard(i_next);
        r0 = walk.row0(i_next);
      }
      i = i_next;
    }
    // Output: the row of O_t / l, for rows inside the shard.
    if (ok && t_valid && wait_warp(o_full, 0)) {
      ptx::tc_fence_after();
      const float inv = 1.f / l;
      char* dst = static_cast<char*>(p.out[r]) +
                  (static_cast<long long>(grow) * p.H + h) * kD * (p.out_f32 ? 4 : 2);
#pragma unroll 1
      for (int c = 0; c < kD; c += 32) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(o_addr + c, v);
        ptx::tmem_ld_wait();
        if (grow < p.S) {
          if (p.out_f32) {
            float4* o = reinterpret_cast<float4*>(dst) + c / 4;
#pragma unroll
            for (int k = 0; k < 32; k += 4)
              o[k / 4] = make_float4(__uint_as_float(v[k]) * inv, __uint_as_float(v[k + 1]) * inv,
                                     __uint_as_float(v[k + 2]) * inv,
                                     __uint_as_float(v[k + 3]) * inv);
          } else {
            uint4* o = reinterpret_cast<uint4*>(dst) + c / 8;
#pragma unroll
            for (int k = 0; k < 32; k += 8) {
              uint4 w;
              w.x = ptx::pack_bf16x2(__uint_as_float(v[k]) * inv, __uint_as_float(v[k + 1]) * inv);
              w.y = ptx::pack_bf16x2(__uint_as_float(v[k + 2]) * inv,
                                     __uint_as_float(v[k + 3]) * inv);
              w.z = ptx::pack_bf16x2(__uint_as_float(v[k + 4]) * inv,
                                     __uint_as_float(v[k + 5]) * inv);
              w.w = ptx::pack_bf16x2(__uint_as_float(v[k + 6]) * inv,
                                     __uint_as_float(v[k + 7]) * inv);
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
  p.qpairs = (p.qtiles + 1) / 2;
  p.kvb = static_cast<int>((S + kBKV - 1) / kBKV);
  p.causal = causal ? 1 : 0;
  p.out_f32 = out_dtype == FCC_F32 ? 1 : 0;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(kD)));
  p.status = status;
  p.timeout_ns = timeout_ns;

  static bool attr_set[64] = {};
  if (smem_attr_once(attr_set, ring_attention_kernel, kSmem) != cudaSuccess) return FCC_ERR_CUDA;
  const unsigned grid = static_cast<unsigned>(R * H * p.qpairs);
  ring_attention_kernel<<<grid, kThreads, kSmem, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  if (cudaGetLastError() != cudaSuccess) return FCC_ERR_CUDA;
  bump_launch_count(1);
  return FCC_OK;
}

}  // extern "C"

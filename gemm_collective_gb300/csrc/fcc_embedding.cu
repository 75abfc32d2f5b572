// fcc_embedding.cu -- Embedding + All-to-All (DLRM pooled lookups), sm_103a.
//
// The SC24 paper's embedding + All-to-All operator: each table's owner pools
// (sums) the bag of rows of every sample of the global batch, and the
// all-to-all sends each pooled vector to the rank that holds the sample.  In
// the fused form one kernel does both: a warp pools one bag and stores the
// result straight into the sample's rank buffer, so the pooled vectors never
// make a round trip through a staging buffer.
//
// The work is a random gather of table rows (D = 128 bf16: 256-byte rows),
// done table by table so that a table's rows are served from L2 once read.
// A warp loads its bag's indices 32 at a time (one per lane) and passes them
// round by shuffles; 32 / (D/8) rows are read per step (16 bytes a lane),
// eight steps unrolled, so a warp has up to sixteen rows in flight (the fused
// form 1222 -> 1135 us against four steps at 8 x 64 tables of 65536 x 128;
// twelve or sixteen steps spilled and ran near twice as long).
// The row groups' f32 partial sums are added by a fixed shuffle tree: the
// result is repeatable.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "fcc.h"
#include "fcc_internal.h"
#include "fcc_ptx.cuh"

namespace fcc {
namespace {

struct EmbArgs {
  const uint16_t* tables[FCC_MAX_TABLES];   // [V, D] bf16
  const int32_t* offsets[FCC_MAX_TABLES];   // [R*Bl + 1]
  const int32_t* indices[FCC_MAX_TABLES];   // [nnz]
  void* out[FCC_MAX_RANKS];                 // fused: [Bl, ntables, D] per rank
  void* pooled;                             // staged: [ntables, R*Bl, D]
  int* status;
  long long V;
  int R, ntables, D, Bl;
  int out_f32;
};

// Pools bag (t, g) and stores its D values at dst (bf16 or f32).
__device__ __forceinline__ void pool_bag(const EmbArgs& a, int t, long long g, char* dst,
                                         int lane) {
  const int vecs = a.D / 8;                       // 16-byte vectors per row
  const int rp = vecs >= 32 ? 1 : 32 / vecs;      // rows per step
  const int grp = lane / vecs;                    // this lane's row in the step
  const int32_t* off = a.offsets[t];
  const int k0 = __ldg(off + g), k1 = __ldg(off + g + 1);
  const int nnz = __ldg(off + static_cast<long long>(a.R) * a.Bl);  // the table's index count
  const uint4* tab = reinterpret_cast<const uint4*>(a.tables[t]);
  bool bad = k1 < k0 || k0 < 0 || k1 > nnz;
  const int kend = bad ? k0 : k1;
  for (int vbase = 0; vbase < vecs; vbase += 32) {  // D > 256: 32 vectors at a time
    const int v = vbase + (vecs >= 32 ? lane : lane % vecs);
    const bool lane_on = (vecs >= 32) ? v < vecs : grp < rp;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int kb = k0; kb < kend; kb += 32) {
      // The next (up to) 32 indices of the bag, one per lane.
      int my = 0;
      if (kb + lane < kend) {
        my = __ldg(a.indices[t] + kb + lane);
        if (my < 0 || my >= a.V) {
          bad = true;
          my = -1;
        }
      }
      const int n = min(32, kend - kb);
      constexpr int kUnroll = 8;
      for (int j0 = 0; j0 < n; j0 += rp * kUnroll) {
        uint4 q[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int j = j0 + u * rp + grp;
          const int row = __shfl_sync(0xffffffffu, my, min(j, 31));
          q[u] = make_uint4(0, 0, 0, 0);
          if (lane_on && j < n && row >= 0)
            q[u] = __ldg(tab + static_cast<long long>(row) * vecs + v);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            acc[2 * h] += __uint_as_float(w[h] << 16);
            acc[2 * h + 1] += __uint_as_float(w[h] & 0xFFFF0000u);
          }
        }
      }
    }
    // Row groups 0..rp-1 hold partial sums of the same columns: a fixed tree
    // (group i takes group i + s at step s) leaves the total in group 0.
    for (int st = 1; st < rp; st <<= 1) {
      const int src = lane + st * vecs;
      const bool take = (grp % (2 * st)) == 0 && grp + st < rp;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float o = __shfl_sync(0xffffffffu, acc[k], src < 32 ? src : lane);
        if (take) acc[k] += o;
      }
    }
    if (lane_on && (vecs >= 32 || grp == 0)) {
      if (a.out_f32) {
        float4* p = reinterpret_cast<float4*>(dst) + 2 * v;
        __stcs(p, make_float4(acc[0], acc[1], acc[2], acc[3]));
        __stcs(p + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
      } else {
        uint4 o;
        o.x = ptx::pack_bf16x2(acc[0], acc[1]);
        o.y = ptx::pack_bf16x2(acc[2], acc[3]);
        o.z = ptx::pack_bf16x2(acc[4], acc[5]);
        o.w = ptx::pack_bf16x2(acc[6], acc[7]);
        __stcs(reinterpret_cast<uint4*>(dst) + v, o);
      }
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0 && a.status != nullptr)
    atomicCAS(a.status, 0, static_cast<int>(FCC_ERR_INVALID));
}

// A walk over (table t, sample g = r * Bl + b) in steps of a fixed number of
// items, table-major, without a division per step: the step is split once
// into whole tables, whole ranks and samples, and each step adds those with
// carries (fused form 1284-1297 -> 1246-1262 us at 8 x 64 tables of 65536 x
// 128, against two 64-bit divisions per bag).
struct ItemWalk {
  int t, r, b;                 // current item
  int st, sr, sb;              // the step in tables, ranks and samples
  int R, Bl;
  __device__ __forceinline__ void init(long long it, long long step, int R_, int Bl_) {
    R = R_;
    Bl = Bl_;
    const long long nsamp = static_cast<long long>(R) * Bl;
    t = static_cast<int>(it / nsamp);
    const long long g = it - static_cast<long long>(t) * nsamp;
    r = static_cast<int>(g / Bl);
    b = static_cast<int>(g - static_cast<long long>(r) * Bl);
    st = static_cast<int>(step / nsamp);
    const long long sg = step - static_cast<long long>(st) * nsamp;
    sr = static_cast<int>(sg / Bl);
    sb = static_cast<int>(sg - static_cast<long long>(sr) * Bl);
  }
  __device__ __forceinline__ void advance() {
    b += sb;                   // < 2 Bl
    r += sr;
    t += st;
    if (b >= Bl) {
      b -= Bl;
      ++r;
    }
    if (r >= R) {              // r < 2 R
      r -= R;
      ++t;
    }
  }
  __device__ __forceinline__ long long g() const { return static_cast<long long>(r) * Bl + b; }
};

// STAGED = false: bag (t, g) -> out[g / Bl][g % Bl][t] (the fused all-to-all);
// STAGED = true: -> pooled[t][g] (each owner's local result).
template <bool STAGED>
__global__ void __launch_bounds__(256) embedding_kernel(const EmbArgs a) {
  const int lane = threadIdx.x & 31;
  const long long nsamp = static_cast<long long>(a.R) * a.Bl;
  const long long items = nsamp * a.ntables;
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const long long esz = a.out_f32 ? 4 : 2;
  long long it = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (it >= items) return;
  ItemWalk w;
  w.init(it, nwarps, a.R, a.Bl);
  for (; it < items; it += nwarps, w.advance()) {
    // Table-major order: the warps running at once gather from one table,
    // which stays in L2 while its bags are pooled (random indices reuse its
    // rows many times), whichever buffer the vectors go to.  (Interleaving
    // 4, 8 or 16 tables, so that consecutive bags fill adjacent output rows,
    // measured slower: the larger live set costs L2 hits.)
    const long long g = w.g();
    char* dst;
    if constexpr (STAGED) {
      dst = static_cast<char*>(a.pooled) + (static_cast<long long>(w.t) * nsamp + g) * a.D * esz;
    } else {
      dst = static_cast<char*>(a.out[w.r]) +
            (static_cast<long long>(w.b) * a.ntables + w.t) * a.D * esz;
    }
    pool_bag(a, w.t, g, dst, lane);
  }
}

// Staged form's exchange: pooled[t][g] -> out[g / Bl][g % Bl][t], 16 bytes a thread.
__global__ void __launch_bounds__(256) a2a_permute_kernel(const EmbArgs a) {
  const long long esz = a.out_f32 ? 4 : 2;
  const long long vec_per_row = a.D * esz / 16;
  const long long nsamp = static_cast<long long>(a.R) * a.Bl;
  const long long total = static_cast<long long>(a.ntables) * nsamp * vec_per_row;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = i / vec_per_row;              // = t * nsamp + g
    const long long c = i - row * vec_per_row;
    const int t = static_cast<int>(row / nsamp);
    const long long g = row - static_cast<long long>(t) * nsamp;
    const int r = static_cast<int>(g / a.Bl);
    const long long b = g - static_cast<long long>(r) * a.Bl;
    const uint4 x = __ldcs(reinterpret_cast<const uint4*>(a.pooled) + i);
    __stcs(reinterpret_cast<uint4*>(static_cast<char*>(a.out[r]) +
                                    (b * a.ntables + t) * a.D * esz) + c, x);
  }
}

}  // namespace
}  // namespace fcc

using namespace fcc;

namespace {

bool emb_al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t emb_ws_bytes(int R, int ntables, int64_t D, int64_t Bl, fcc_dtype out_dtype,
                    fcc_algo algo) {
  if (algo != FCC_ALGO_UNFUSED && algo != FCC_ALGO_CE) return 0;
  const size_t esz = out_dtype == FCC_F32 ? 4 : 2;
  return (static_cast<size_t>(ntables) * R * Bl * D * esz + 255) & ~static_cast<size_t>(255);
}

fcc_algo emb_algo(const fcc_opts* o) {
  return (o == nullptr || o->algo == FCC_ALGO_AUTO) ? choose_algo(FCC_OP_EMBEDDING_A2A, 0, 0, 0,
                                                                  0, 0, 0)
                                                    : o->algo;
}

}  // namespace

extern "C" {

size_t fcc_embedding_workspace_size(int R, int ntables, int64_t D, int64_t Bl,
                                    fcc_dtype out_dtype, const fcc_opts* opts) {
  if (R < 1 || R > FCC_MAX_RANKS || ntables < 1 || D < 1 || Bl < 1) return 0;
  return emb_ws_bytes(R, ntables, D, Bl, out_dtype, emb_algo(opts));
}

fcc_status fcc_embedding_a2a(int R, int ntables, const void* const* tables, int64_t V,
                             int64_t D, int64_t Bl, const int32_t* const* offsets,
                             const int32_t* const* indices, void* const* out, fcc_dtype in,
                             fcc_dtype out_dtype, const fcc_opts* opts, fcc_stream_t stream) {
  if (R < 1 || R > FCC_MAX_RANKS || ntables < R || ntables > FCC_MAX_TABLES ||
      ntables % R != 0)
    return FCC_ERR_INVALID;
  if (V < 1 || V > (1ll << 31) - 1 || D < 8 || D % 8 != 0 || D > 4096 || Bl < 1 ||
      static_cast<int64_t>(R) * Bl > (1ll << 30))
    return FCC_ERR_INVALID;
  if (tables == nullptr || offsets == nullptr || indices == nullptr || out == nullptr)
    return FCC_ERR_INVALID;
  for (int t = 0; t < ntables; ++t)
    if (tables[t] == nullptr || offsets[t] == nullptr || indices[t] == nullptr ||
        !emb_al16(tables[t]) || (reinterpret_cast<uintptr_t>(offsets[t]) & 3u) ||
        (reinterpret_cast<uintptr_t>(indices[t]) & 3u))
      return FCC_ERR_INVALID;
  for (int r = 0; r < R; ++r)
    if (out[r] == nullptr || !emb_al16(out[r])) return FCC_ERR_INVALID;
  if ((in != FCC_BF16 && in != FCC_F16 && in != FCC_F32) ||
      (out_dtype != FCC_BF16 && out_dtype != FCC_F16 && out_dtype != FCC_F32))
    return FCC_ERR_INVALID;
  if (in != FCC_BF16 || out_dtype == FCC_F16) return FCC_ERR_UNSUPPORTED;
  const fcc_algo algo = emb_algo(opts);
  if (algo == FCC_ALGO_INTERDECOM) return FCC_ERR_UNSUPPORTED;
  if (algo != FCC_ALGO_FUSED && algo != FCC_ALGO_UNFUSED && algo != FCC_ALGO_CE)
    return FCC_ERR_INVALID;

  void* ws = nullptr;
  int* status = nullptr;
  int sms = 0;
  unsigned long long timeout_ns = 0;
  fcc_status s = internal_prepare(opts, emb_ws_bytes(R, ntables, D, Bl, out_dtype, algo), &ws,
                                  &status, &sms, &timeout_ns);
  if (s != FCC_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  EmbArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int t = 0; t < ntables; ++t) {
    a.tables[t] = static_cast<const uint16_t*>(tables[t]);
    a.offsets[t] = offsets[t];
    a.indices[t] = indices[t];
  }
  for (int r = 0; r < R; ++r) a.out[r] = out[r];
  a.pooled = ws;
  a.status = status;
  a.V = V;
  a.R = R;
  a.ntables = ntables;
  a.D = static_cast<int>(D);
  a.Bl = static_cast<int>(Bl);
  a.out_f32 = out_dtype == FCC_F32 ? 1 : 0;

  // A persistent grid of the warps that fit at once (each loops over bags).
  auto kern = algo == FCC_ALGO_FUSED ? embedding_kernel<false> : embedding_kernel<true>;
  static int occ[2][64] = {};
  const int per_sm = blocks_per_sm_once(occ[algo == FCC_ALGO_FUSED ? 0 : 1], kern, 256);
  const long long bags = static_cast<long long>(R) * Bl * ntables;
  const long long blocks = std::min<long long>((bags + 7) / 8, static_cast<long long>(sms) * per_sm);
  kern<<<static_cast<unsigned>(std::max<long long>(1, blocks)), 256, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return FCC_ERR_CUDA;
  uint64_t launches = 1;
  if (algo == FCC_ALGO_UNFUSED) {
    a2a_permute_kernel<<<std::max(1, sms) * 8, 256, 0, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return FCC_ERR_CUDA;
    ++launches;
  } else if (algo == FCC_ALGO_CE) {
    // One strided copy per (table, destination rank): Bl rows of D values.
    const size_t esz = a.out_f32 ? 4 : 2;
    const size_t row = static_cast<size_t>(D) * esz;
    for (int t = 0; t < ntables; ++t)
      for (int r = 0; r < R; ++r) {
        const char* src = static_cast<const char*>(ws) +
                          (static_cast<size_t>(t) * R * Bl + static_cast<size_t>(r) * Bl) * row;
        char* dst = static_cast<char*>(out[r]) + static_cast<size_t>(t) * row;
        if (cudaMemcpy2DAsync(dst, static_cast<size_t>(ntables) * row, src, row, row,
                              static_cast<size_t>(Bl), cudaMemcpyDeviceToDevice, st) !=
            cudaSuccess)
          return FCC_ERR_CUDA;
      }
  }
  bump_launch_count(launches);
  return FCC_OK;
}

}  // extern "C"

// fcc_combine.cu -- MoE combine: the return all-to-all and the gate-weighted
// top-k sum (sm_103a).
//
// The direction back to the token owners of the SC24 paper's GEMM + All-to-All
// operator for MoE: token t of source rank s collects the expert outputs of
// its top-k assignments from the receiving ranks and adds them, each scaled by
// its gate.  Three kernels:
//   0. clear_loc_kernel  loc[*] = -1.
//   1. locate_kernel  one thread per receive row (rank d, row i): the row's
//                     expert from the prefix of d's local expert counts, its
//                     token from recv_src, its slot from the token's top-k
//                     list; writes loc[token][slot] = d*cap + i.
//   2. combine_kernel one warp per token (a persistent grid): reads each of its
//                     (at most two) rows once, 16 bytes per lane and four
//                     steps in flight, adds gate * row in slot order in f32
//                     and stores the token's output row once.
// The rows move once each way (HBM bound: recv rows read, outputs written);
// no atomics, so the result is repeatable.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "fcc.h"
#include "fcc_internal.h"
#include "fcc_ptx.cuh"

namespace fcc {
namespace {

struct CombineArgs {
  const void* recv_y[FCC_MAX_RANKS];      // [cap, F] per receiving rank
  const int32_t* idx[FCC_MAX_RANKS];      // [T, topk] per source rank
  const float* gate[FCC_MAX_RANKS];       // [T, topk]
  const int32_t* recv_src[FCC_MAX_RANKS]; // [cap]
  const int32_t* counts;                  // [E]
  void* y[FCC_MAX_RANKS];                 // [T, F] per source rank
  int32_t* loc;                           // [R*T*topk]: d*cap + row, -1 = not received
  long long cap;
  int R, E, Eloc, topk, T, F;
  int in_f32, out_f32;
};

// loc[*] = -1 (a slot stays -1 unless locate_kernel finds its row).
__global__ void __launch_bounds__(256) clear_loc_kernel(const CombineArgs a) {
  ptx::griddep_wait();  // launched with programmatic stream serialization
  ptx::griddep_launch_dependents();
  const long long n = static_cast<long long>(a.R) * a.T * a.topk;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    a.loc[i] = -1;
}

__global__ void __launch_bounds__(256) locate_kernel(const CombineArgs a) {
  ptx::griddep_wait();  // launched with programmatic stream serialization
  ptx::griddep_launch_dependents();
  const long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g >= static_cast<long long>(a.R) * a.cap) return;
  const int d = static_cast<int>(g / a.cap);
  const long long i = g - static_cast<long long>(d) * a.cap;
  // Expert of row i: rank d holds its local experts' rows in expert order.
  long long start = 0;
  int e = -1;
  for (int l = 0; l < a.Eloc; ++l) {
    const long long c = __ldg(a.counts + d * a.Eloc + l);
    if (i < start + c) {
      e = d * a.Eloc + l;
      break;
    }
    start += c;
  }
  if (e < 0) return;  // past the rows this rank received
  const int src = __ldg(a.recv_src[d] + i);
  if (src < 0 || src >= a.R * a.T) return;
  const int s = src / a.T;
  const int t = src - s * a.T;
  for (int j = 0; j < a.topk; ++j) {
    if (__ldg(a.idx[s] + static_cast<long long>(t) * a.topk + j) == e) {
      a.loc[static_cast<long long>(src) * a.topk + j] = static_cast<int32_t>(g);
      break;
    }
  }
}

// One 16-byte vector of a row: 8 bf16 values, or 4 f32 values.  Rows are
// held raw while in flight (4 registers a vector) and widened at use.
__device__ __forceinline__ void widen_bf16(const uint4& q, float (&x)[8]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    x[2 * h] = __uint_as_float(w[h] << 16);
    x[2 * h + 1] = __uint_as_float(w[h] & 0xFFFF0000u);
  }
}

// Output vector v of the token: 8 values (bf16 rows) or 4 (f32 rows).
template <bool IN_F32>
__device__ __forceinline__ void store_vec(char* out, int v, int out_f32, const float* acc) {
  constexpr int kN = IN_F32 ? 4 : 8;
  if (out_f32) {
    float4* p = reinterpret_cast<float4*>(out) + (IN_F32 ? v : 2 * v);
    __stcs(p, make_float4(acc[0], acc[1], acc[2], acc[3]));
    if (kN == 8) __stcs(p + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
  } else if (kN == 8) {
    uint4 q;
    q.x = ptx::pack_bf16x2(acc[0], acc[1]);
    q.y = ptx::pack_bf16x2(acc[2], acc[3]);
    q.z = ptx::pack_bf16x2(acc[4], acc[5]);
    q.w = ptx::pack_bf16x2(acc[6], acc[7]);
    __stcs(reinterpret_cast<uint4*>(out) + v, q);
  } else {
    uint2 q;
    q.x = ptx::pack_bf16x2(acc[0], acc[1]);
    q.y = ptx::pack_bf16x2(acc[2], acc[3]);
    __stcs(reinterpret_cast<uint2*>(out) + v, q);
  }
}

template <bool IN_F32>
__global__ void __launch_bounds__(256) combine_kernel(const CombineArgs a) {
  ptx::griddep_wait();  // launched with programmatic stream serialization
  ptx::griddep_launch_dependents();
  constexpr int kN = IN_F32 ? 4 : 8;      // values per 16-byte vector
  constexpr int kUnroll = 4;              // vectors per lane in flight, per row
  const int lane = threadIdx.x & 31;
  const long long ntok = static_cast<long long>(a.R) * a.T;
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const int vecs = a.F / kN;
  const long long in_row = static_cast<long long>(a.F) * (IN_F32 ? 4 : 2);
  for (long long tok = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       tok < ntok; tok += nwarps) {
    const int s = static_cast<int>(tok / a.T);
    const int t = static_cast<int>(tok - static_cast<long long>(s) * a.T);
    // Lane j < topk fetches slot j's receive row and gate; the warp shares them.
    const uint4* row = nullptr;
    float g = 0.f;
    if (lane < a.topk) {
      const int l = a.loc[tok * a.topk + lane];
      if (l >= 0) {
        const int d = static_cast<int>(l / a.cap);
        const long long i = l - static_cast<long long>(d) * a.cap;
        row = reinterpret_cast<const uint4*>(static_cast<const char*>(a.recv_y[d]) + i * in_row);
        g = __ldg(a.gate[s] + static_cast<long long>(t) * a.topk + lane);
      }
    }
    const uint4* row0 = reinterpret_cast<const uint4*>(
        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(row), 0));
    const uint4* row1 = reinterpret_cast<const uint4*>(
        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(row), 1));
    const float g0 = __shfl_sync(0xffffffffu, g, 0);
    const float g1 = __shfl_sync(0xffffffffu, g, 1);
    if (a.topk < 2) row1 = nullptr;
    char* out = static_cast<char*>(a.y[s]) + static_cast<long long>(t) * a.F * (a.out_f32 ? 4 : 2);
    // All loads of a step (kUnroll vectors of both rows) are issued before the
    // first use: 8 x 16 bytes per lane in flight.
    for (int v0 = lane; v0 < vecs; v0 += 32 * kUnroll) {
      uint4 q0[kUnroll], q1[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + 32 * u;
        q0[u] = make_uint4(0, 0, 0, 0);
        q1[u] = make_uint4(0, 0, 0, 0);
        if (v < vecs) {
          if (row0 != nullptr) q0[u] = __ldcs(row0 + v);
          if (row1 != nullptr) q1[u] = __ldcs(row1 + v);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + 32 * u;
        if (v >= vecs) break;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float x[8];
        if (row0 != nullptr) {
          if constexpr (IN_F32) {
            x[0] = __uint_as_float(q0[u].x); x[1] = __uint_as_float(q0[u].y);
            x[2] = __uint_as_float(q0[u].z); x[3] = __uint_as_float(q0[u].w);
          } else {
            widen_bf16(q0[u], x);
          }
#pragma unroll
          for (int k = 0; k < kN; ++k) acc[k] += g0 * x[k];
        }
        if (row1 != nullptr) {
          if constexpr (IN_F32) {
            x[0] = __uint_as_float(q1[u].x); x[1] = __uint_as_float(q1[u].y);
            x[2] = __uint_as_float(q1[u].z); x[3] = __uint_as_float(q1[u].w);
          } else {
            widen_bf16(q1[u], x);
          }
#pragma unroll
          for (int k = 0; k < kN; ++k) acc[k] += g1 * x[k];
        }
        store_vec<IN_F32>(out, v, a.out_f32, acc);
      }
    }
  }
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t combine_ws_bytes(int R, int64_t T, int topk) {
  return (static_cast<size_t>(R) * static_cast<size_t>(T) * topk * 4 + 255) & ~size_t(255);
}

}  // namespace
}  // namespace fcc

using namespace fcc;

extern "C" {

size_t fcc_moe_combine_workspace_size(int R, int64_t T, int topk) {
  if (R < 1 || R > FCC_MAX_RANKS || T < 1 || topk < 1 || topk > 2) return 0;
  return combine_ws_bytes(R, T, topk);
}

fcc_status fcc_moe_combine(int R, const void* const* recv_y, int64_t cap, int64_t T, int64_t F,
                           int E, int topk, const int32_t* const* topk_idx,
                           const float* const* topk_gate, const int32_t* const* recv_src,
                           const int32_t* expert_counts, void* const* y, fcc_dtype in,
                           fcc_dtype out_dtype, const fcc_opts* opts, fcc_stream_t stream) {
  if (R < 1 || R > FCC_MAX_RANKS || E < R || E > FCC_MAX_EXPERTS || E % R != 0)
    return FCC_ERR_INVALID;
  if (topk < 1 || topk > 2 || topk > E || T < 1 || F < 8 || F % 8 != 0 || cap < 1)
    return FCC_ERR_INVALID;
  if (T > (1ll << 28) || F > (1ll << 30) || cap > (1ll << 30) ||
      static_cast<int64_t>(R) * cap > (1ll << 31) - 1 ||
      static_cast<int64_t>(R) * T * topk > (1ll << 30))
    return FCC_ERR_INVALID;
  if (recv_y == nullptr || topk_idx == nullptr || topk_gate == nullptr ||
      recv_src == nullptr || expert_counts == nullptr || y == nullptr)
    return FCC_ERR_INVALID;
  for (int r = 0; r < R; ++r)
    if (recv_y[r] == nullptr || topk_idx[r] == nullptr || topk_gate[r] == nullptr ||
        recv_src[r] == nullptr || y[r] == nullptr || !al16(recv_y[r]) || !al16(y[r]))
      return FCC_ERR_INVALID;
  if ((in != FCC_BF16 && in != FCC_F16 && in != FCC_F32) ||
      (out_dtype != FCC_BF16 && out_dtype != FCC_F16 && out_dtype != FCC_F32))
    return FCC_ERR_INVALID;
  if (in == FCC_F16 || out_dtype == FCC_F16) return FCC_ERR_UNSUPPORTED;
  if (opts != nullptr && opts->algo != FCC_ALGO_AUTO && opts->algo != FCC_ALGO_FUSED &&
      opts->algo != FCC_ALGO_UNFUSED)
    return FCC_ERR_UNSUPPORTED;

  void* ws = nullptr;
  int* status = nullptr;
  int sms = 0;
  unsigned long long timeout_ns = 0;
  fcc_status s = internal_prepare(opts, combine_ws_bytes(R, T, topk), &ws, &status, &sms,
                                  &timeout_ns);
  if (s != FCC_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  CombineArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int r = 0; r < R; ++r) {
    a.recv_y[r] = recv_y[r];
    a.idx[r] = topk_idx[r];
    a.gate[r] = topk_gate[r];
    a.recv_src[r] = recv_src[r];
    a.y[r] = y[r];
  }
  a.counts = expert_counts;
  a.loc = static_cast<int32_t*>(ws);
  a.cap = cap;
  a.R = R;
  a.E = E;
  a.Eloc = E / R;
  a.topk = topk;
  a.T = static_cast<int>(T);
  a.F = static_cast<int>(F);
  a.in_f32 = in == FCC_F32 ? 1 : 0;
  a.out_f32 = out_dtype == FCC_F32 ? 1 : 0;

  // Three kernels chained with programmatic stream serialization (each one's
  // launch overlaps the one before it; each waits for it in-kernel).
  const long long slots = static_cast<long long>(R) * T * topk;
  const unsigned clear_blocks =
      static_cast<unsigned>(std::min<long long>((slots + 255) / 256, 4ll * std::max(1, sms)));
  if (launch_pdl(clear_loc_kernel, dim3(clear_blocks), dim3(256), 0, st, 1u, a) != cudaSuccess)
    return FCC_ERR_CUDA;
  const long long rows = static_cast<long long>(R) * cap;
  if (launch_pdl(locate_kernel, dim3(static_cast<unsigned>((rows + 255) / 256)), dim3(256), 0, st,
                 1u, a) != cudaSuccess)
    return FCC_ERR_CUDA;
  // A persistent grid of the blocks that fit at once (warps loop over tokens).
  auto kern = a.in_f32 ? combine_kernel<true> : combine_kernel<false>;
  static int occ[2][64] = {};
  const int per_sm = blocks_per_sm_once(occ[a.in_f32], kern, 256);
  const long long ntok = static_cast<long long>(R) * T;
  const long long blocks =
      std::min<long long>((ntok + 7) / 8, static_cast<long long>(sms) * per_sm);
  if (launch_pdl(kern, dim3(static_cast<unsigned>(std::max<long long>(1, blocks))), dim3(256), 0,
                 st, 1u, a) != cudaSuccess)
    return FCC_ERR_CUDA;
  bump_launch_count(3);
  return FCC_OK;
}

}  // extern "C"

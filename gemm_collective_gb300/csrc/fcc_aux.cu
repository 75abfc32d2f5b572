// fcc_aux.cu -- bandwidth kernels for the unfused baselines and the gather
// copy, plus the bounded-wait probe used to test timeout reporting.
#include <cuda_runtime.h>

#include "fcc_internal.h"
#include "fcc_ptx.cuh"

namespace fcc {
namespace {

struct ReduceArgs {
  const float* P[FCC_MAX_RANKS];
  void* out[FCC_MAX_RANKS];
  int R;
  int nout;        // RS: one output per shard; AR: nout replicas of the full rows
  int per_shard;   // 1 = RS (row goes to its shard), 0 = AR (row goes to every output)
  long long N, Ms, row_begin, row_end;
  int out_f32;
};

// Each thread sums 8 consecutive columns of one row over the R partials,
// in rank order 0..R-1, and stores them (f32 or bf16).
__global__ void __launch_bounds__(256) reduce_shards_kernel(const ReduceArgs a) {
  ptx::griddep_wait();  // launched with programmatic stream serialization
  ptx::griddep_launch_dependents();
  const long long groups_per_row = a.N / 8;
  const long long total = (a.row_end - a.row_begin) * groups_per_row;
  for (long long g = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; g < total;
       g += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = a.row_begin + g / groups_per_row;
    const long long col = (g % groups_per_row) * 8;
    float s[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] = 0.f;
    for (int r = 0; r < a.R; ++r) {
      const float4* src = reinterpret_cast<const float4*>(a.P[r] + row * a.N + col);
      const float4 x = __ldcs(src);
      const float4 y = __ldcs(src + 1);
      s[0] += x.x; s[1] += x.y; s[2] += x.z; s[3] += x.w;
      s[4] += y.x; s[5] += y.y; s[6] += y.z; s[7] += y.w;
    }
    const int first = a.per_shard ? static_cast<int>(row / a.Ms) : 0;
    const int count = a.per_shard ? 1 : a.nout;
    const long long drow = a.per_shard ? row - static_cast<long long>(first) * a.Ms : row;
    for (int o = first; o < first + count; ++o) {
      if (a.out_f32) {
        float4* d = reinterpret_cast<float4*>(static_cast<float*>(a.out[o]) + drow * a.N + col);
        d[0] = make_float4(s[0], s[1], s[2], s[3]);
        d[1] = make_float4(s[4], s[5], s[6], s[7]);
      } else {
        uint4 w;
        w.x = ptx::pack_bf16x2(s[0], s[1]);
        w.y = ptx::pack_bf16x2(s[2], s[3]);
        w.z = ptx::pack_bf16x2(s[4], s[5]);
        w.w = ptx::pack_bf16x2(s[6], s[7]);
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out[o]) + drow * a.N + col) = w;
      }
    }
  }
}

struct GatherArgs {
  const void* X[FCC_MAX_RANKS];
  void* dst;
  int R;
  long long Ms, K;
  long long row_begin, row_end;  // rows of the gathered matrix to write
};

// dst rows [row_begin, row_end) of [X_0; X_1; ...] with 16-byte copies (K % 8 == 0).
__global__ void __launch_bounds__(256) gather_rows_kernel(const GatherArgs a) {
  ptx::griddep_wait();  // launched with programmatic stream serialization
  ptx::griddep_launch_dependents();
  const long long vec_per_row = a.K / 8;
  const long long per_shard = a.Ms * vec_per_row;
  const long long first = a.row_begin * vec_per_row;
  const long long total = (a.row_end - a.row_begin) * vec_per_row;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long g = first + i;
    const int s = static_cast<int>(g / per_shard);
    const long long off = g - s * per_shard;
    const uint4 v = __ldcs(reinterpret_cast<const uint4*>(a.X[s]) + off);
    reinterpret_cast<uint4*>(a.dst)[g] = v;
  }
}

// Waits on an mbarrier that nothing completes, with the library's bounded
// wait: the wait runs out after `timeout_ns`, the status word records
// FCC_ERR_TIMEOUT and the kernel returns.
__global__ void wait_probe_kernel(int* status, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const ptx::Waiter W{&abort_flag, status, timeout_ns};
    W.wait(&bar, 0);
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_reduce_shards(const float* const* P, int R, void* const* out, int nout,
                                 int per_shard, int64_t M, int64_t N, int64_t Ms,
                                 int64_t row_begin, int64_t row_end, int out_f32,
                                 cudaStream_t st) {
  (void)M;
  ReduceArgs a{};
  for (int r = 0; r < R; ++r) a.P[r] = P[r];
  for (int o = 0; o < nout; ++o) a.out[o] = out[o];
  a.R = R;
  a.nout = nout;
  a.per_shard = per_shard;
  a.N = N;
  a.Ms = Ms;
  a.row_begin = row_begin;
  a.row_end = row_end;
  a.out_f32 = out_f32;
  const long long work = (row_end - row_begin) * (N / 8);
  if (work <= 0) return cudaSuccess;
  const int sms = device_sm_count();
  long long blocks = (work + 255) / 256;
  const long long cap = static_cast<long long>(sms) * 8;
  if (blocks > cap) blocks = cap;
  bump_launch_count(1);
  return launch_pdl(reduce_shards_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1u,
                    a);
}

cudaError_t launch_gather_rows(const void* const* X, int R, int64_t Ms, int64_t K, void* dst,
                               cudaStream_t st) {
  return launch_gather_rows_range(X, R, Ms, K, dst, 0, static_cast<int64_t>(R) * Ms, st);
}

cudaError_t launch_gather_rows_range(const void* const* X, int R, int64_t Ms, int64_t K,
                                     void* dst, int64_t row_begin, int64_t row_end,
                                     cudaStream_t st) {
  GatherArgs a{};
  for (int r = 0; r < R; ++r) a.X[r] = X[r];
  a.dst = dst;
  a.R = R;
  a.Ms = Ms;
  a.K = K;
  a.row_begin = row_begin;
  a.row_end = row_end;
  const long long work = (row_end - row_begin) * (K / 8);
  if (work <= 0) return cudaSuccess;
  const int sms = device_sm_count();
  long long blocks = (work + 255) / 256;
  const long long cap = static_cast<long long>(sms) * 8;
  if (blocks > cap) blocks = cap;
  bump_launch_count(1);
  return launch_pdl(gather_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1u,
                    a);
}

cudaError_t launch_wait_probe(int* status, unsigned long long timeout_ns, cudaStream_t st) {
  wait_probe_kernel<<<1, 32, 0, st>>>(status, timeout_ns);
  bump_launch_count(1);
  return cudaGetLastError();
}

}  // namespace fcc

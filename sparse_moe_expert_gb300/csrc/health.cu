// Expert health: page "Qwen3.5-MoE与Qwen3-MoE架构差异深度解析", section 6 (a
// serving-side "MoE health" check built on two numbers per time window: the
// expert activated least often, and the standard deviation of all experts'
// activation counts) and section 4.2 (per-expert activation counts of a
// batch).  A layer call's counts are the expert_counts its grouping writes;
// a window sums them in int64 on the device, and one small kernel reduces
// the window to the least-activated expert, the mean and the standard
// deviation, so the monitor reads back three numbers per window.
#include <climits>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kHealthThreads = 1024;  // one thread per expert, E <= 1024

__global__ void counts_accumulate_kernel(const int32_t* __restrict__ counts, int E,
                                         long long* __restrict__ window) {
  pdl_wait();
  pdl_trigger();
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x)
    window[e] += counts[e];
}

// One CTA.  The sum of the counts is exact (int64); mean = sum / E and the
// population variance sum_e (c_e - mean)^2 / E in fp64, each sum in a fixed
// order (xor butterfly within a warp, then the warps in order).  The least
// count wins, equal counts the lower expert id.
__global__ void __launch_bounds__(kHealthThreads)
    expert_health_kernel(const long long* __restrict__ window, int E, int32_t* least,
                         double* mean_std) {
  pdl_wait();
  pdl_trigger();
  __shared__ long long wsum[32];
  __shared__ double wsq[32];
  __shared__ long long wmin[32];
  __shared__ int wid[32];
  __shared__ double mean_sh;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const bool on = t < E;
  const long long c = on ? window[t] : 0;

  long long s = c;
  long long mn = on ? c : LLONG_MAX;
  int id = on ? t : INT_MAX;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
    const long long om = __shfl_xor_sync(0xFFFFFFFFu, mn, off);
    const int oi = __shfl_xor_sync(0xFFFFFFFFu, id, off);
    if (om < mn || (om == mn && oi < id)) {
      mn = om;
      id = oi;
    }
  }
  if (lane == 0) {
    wsum[warp] = s;
    wmin[warp] = mn;
    wid[warp] = id;
  }
  __syncthreads();
  if (t == 0) {
    long long total = 0, best = LLONG_MAX;
    int best_id = INT_MAX;
    for (int w = 0; w < kHealthThreads / 32; ++w) {
      total += wsum[w];
      if (wmin[w] < best || (wmin[w] == best && wid[w] < best_id)) {
        best = wmin[w];
        best_id = wid[w];
      }
    }
    mean_sh = (double)total / (double)E;
    *least = best_id;
  }
  __syncthreads();
  const double d = on ? (double)c - mean_sh : 0.0;
  double q = d * d;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) q += __shfl_xor_sync(0xFFFFFFFFu, q, off);
  if (lane == 0) wsq[warp] = q;
  __syncthreads();
  if (t == 0) {
    double v = 0.0;
    for (int w = 0; w < kHealthThreads / 32; ++w) v += wsq[w];
    mean_std[0] = mean_sh;
    mean_std[1] = sqrt(v / (double)E);
  }
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_expert_counts_accumulate(const int32_t* expert_counts, int E,
                                                     int64_t* window_counts,
                                                     moe_stream_t stream) {
  using namespace moe_host;
  if (E < 1 || E > 1024 || !expert_counts || !window_counts) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(window_counts) & 7u) return MOE_ERR_INVALID_ARG;
  const int threads = 256;
  return launch(moe::counts_accumulate_kernel, (E + threads - 1) / threads, threads, 0,
                reinterpret_cast<cudaStream_t>(stream), expert_counts, E,
                reinterpret_cast<long long*>(window_counts));
}

extern "C" moe_status_t moe_expert_health(const int64_t* window_counts, int E,
                                          int32_t* least_expert, double* mean_std,
                                          moe_stream_t stream) {
  using namespace moe_host;
  if (E < 1 || E > 1024 || !window_counts || !least_expert || !mean_std)
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(window_counts) | reinterpret_cast<uintptr_t>(mean_std)) & 7u)
    return MOE_ERR_INVALID_ARG;
  return launch(moe::expert_health_kernel, 1, moe::kHealthThreads, 0,
                reinterpret_cast<cudaStream_t>(stream),
                reinterpret_cast<const long long*>(window_counts), E, least_expert, mean_std);
}

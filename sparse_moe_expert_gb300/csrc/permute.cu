// Permute: stable counting sort of the (token, slot) assignments by expert.
//
// Page "oMLX MoE gate/up 融合优化：qwen35_moe_gate_up 实现剖析", section
// 如何验证正确性 (the sorted branch that groups token indices by expert before
// the gathered product); page "Qwen3.5-MoE与Qwen3-MoE架构差异深度解析",
// section 4.2 (per-expert activation counts).
//
// CTAs of 1024 threads, each owning a contiguous range of assignments
// (a multiple of 1024).  Every CTA counts all assignments per expert with
// shared-memory atomics into per-warp histograms (integer, so
// order-independent), the ones before its range separately, and scans the
// totals into the offsets.
// It then places its own range chunk by chunk in ascending order; inside a
// chunk an assignment's rank among equal experts is its rank within its warp
// (__match_any_sync) plus the counts of the same expert in lower warps of the
// chunk (a per-expert column scan over the 32 warp histograms) plus the
// number before the chunk (earlier CTAs' ranges and earlier chunks).  The
// result is unique: for each expert, its assignments in ascending
// a = t*kmax + j.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kPermuteThreads = 1024;
constexpr int kPermuteWarps = kPermuteThreads / 32;

struct PermuteParams {
  const int32_t* ids;
  const int32_t* k_dev;
  int T, kmax, E;
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted;
  int32_t* inv_pos;
  int capacity;  // most assignments an expert keeps (INT32_MAX: no limit)
  unsigned int* err;
};

__global__ void __launch_bounds__(kPermuteThreads) permute_kernel(PermuteParams p, int per_block) {
  extern __shared__ int smem_i[];
  pdl_wait();
  pdl_trigger();
  const int E = p.E;
  int* cnt = smem_i;              // [E]
  int* off = cnt + E;             // [E]
  int* run = off + E;             // [E] placed before the current chunk
  int* tot = run + E;             // [E] this chunk's count
  int* wcnt = tot + E;            // [32][E] per-warp histograms / prefixes
  __shared__ int warp_sums[kPermuteWarps];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = *p.k_dev;
  const int slots = p.T * p.kmax;
  const int lo = blockIdx.x * per_block;
  const int hi = min(slots, lo + per_block);

  for (int i = tid; i < E; i += kPermuteThreads) { cnt[i] = 0; run[i] = 0; }
  for (int i = tid; i < kPermuteWarps * E; i += kPermuteThreads) wcnt[i] = 0;
  __syncthreads();

  // expert of assignment a, or -1 (slot j >= k, or an id outside [0, E))
  auto expert_of = [&](int a, bool report) -> int {
    if (a >= slots || a % p.kmax >= k) return -1;
    const int v = __ldg(p.ids + a);
    if (v >= 0 && v < E) return v;
    if (report) raise_device_error(p.err, MOE_DEVERR_BAD_EXPERT);
    return -1;
  };

  // counts: per-warp histogram rows (plain shared atomics, each warp on its
  // own row) of [0, lo), summed into run[], then of [lo, slots), summed
  // with run[] into cnt[] (the total).
  for (int pass = 0; pass < 2; ++pass) {
    const int from = pass == 0 ? 0 : lo, to = pass == 0 ? lo : slots;
    int* row = wcnt + warp * E;
    for (int base = from; base < to; base += 4 * kPermuteThreads) {
      int eb[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int a = base + u * kPermuteThreads + tid;
        eb[u] = a < to ? expert_of(a, blockIdx.x == 0) : -1;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (eb[u] >= 0) atomicAdd(row + eb[u], 1);
    }
    __syncthreads();
    for (int x = tid; x < E; x += kPermuteThreads) {
      int sum = 0;
      for (int w = 0; w < kPermuteWarps; ++w) {
        sum += wcnt[w * E + x];
        wcnt[w * E + x] = 0;
      }
      if (pass == 0) run[x] = sum;
      else cnt[x] = run[x] + sum;
    }
    __syncthreads();
  }

  // exclusive scan of the kept counts -> off (E <= 1024 = blockDim)
  {
    int v = tid < E ? min(cnt[tid], p.capacity) : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int ws = warp_sums[lane];
      int wincl = ws;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xFFFFFFFFu, wincl, o);
        if (lane >= o) wincl += n;
      }
      warp_sums[lane] = wincl - ws;  // exclusive prefix of warp totals
    }
    __syncthreads();
    if (tid < E) {
      int excl = incl - v + warp_sums[warp];
      off[tid] = excl;
      if (blockIdx.x == 0) {
        p.counts[tid] = v;
        p.offsets[tid] = excl;
        if (tid == E - 1) p.offsets[E] = excl + v;
      }
    }
  }
  __syncthreads();

  // stable scatter of [lo, hi), chunk by chunk
  for (int base = lo; base < hi; base += kPermuteThreads) {
    const int a = base + tid;
    const int e = a < hi ? expert_of(a, false) : -1;
    if (a < hi && e < 0) p.inv_pos[a] = -1;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    const int rank_in_warp = __popc(peers & lanemask_lt());
    const bool leader = (peers & lanemask_lt()) == 0u;
    if (e >= 0 && leader) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    for (int x = tid; x < E; x += kPermuteThreads) {
      int running = 0;
      for (int w = 0; w < kPermuteWarps; ++w) {
        int c = wcnt[w * E + x];
        wcnt[w * E + x] = running;
        running += c;
      }
      tot[x] = running;
    }
    __syncthreads();
    if (e >= 0) {
      // rank of a among its expert's assignments, in ascending a
      const int rank = run[e] + wcnt[warp * E + e] + rank_in_warp;
      if (rank < p.capacity) {
        const int pos = off[e] + rank;
        p.sorted[pos] = (int32_t)a;
        p.inv_pos[a] = pos;
      } else {
        p.inv_pos[a] = MOE_DROPPED;  // the expert's capacity is full
      }
    }
    __syncthreads();
    for (int x = tid; x < E; x += kPermuteThreads) {
      run[x] += tot[x];
      for (int w = 0; w < kPermuteWarps; ++w) wcnt[w * E + x] = 0;
    }
    __syncthreads();
  }
  // with a capacity, sorted rows past the kept total hold assignment 0 (a
  // valid one), so consumers of T*k sorted rows stay in bounds
  if (p.capacity != INT32_MAX && blockIdx.x == 0) {
    int kept = 0;
    for (int x = 0; x < E; ++x) kept += min(cnt[x], p.capacity);
    for (int i = kept + tid; i < p.T * k; i += kPermuteThreads) p.sorted[i] = 0;
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

namespace {

moe_status_t permute_impl(const int32_t* topk_ids, const int32_t* k_dev, int T, int kmax, int E,
                          int capacity, int32_t* expert_counts, int32_t* expert_offsets,
                          int32_t* sorted_assign, int32_t* inv_pos, moe_stream_t stream) {
  using namespace moe_host;
  if (T < 0 || E < 1 || E > 1024 || kmax < 1 || kmax > 16) return MOE_ERR_INVALID_ARG;
  if ((int64_t)T * kmax > (1 << 24)) return MOE_ERR_INVALID_ARG;
  if (!k_dev || !expert_counts || !expert_offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_ids || !sorted_assign || !inv_pos)) return MOE_ERR_INVALID_ARG;
  PermuteParams p;
  p.ids = topk_ids;
  p.k_dev = k_dev;
  p.T = T;
  p.kmax = kmax;
  p.E = E;
  p.counts = expert_counts;
  p.offsets = expert_offsets;
  p.sorted = sorted_assign;
  p.inv_pos = inv_pos;
  p.capacity = capacity;
  p.err = device_error_word();
  size_t smem = (size_t)(4 + kPermuteWarps) * E * sizeof(int);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  // ranges of whole 1024-assignment chunks; every CTA also reads all ids
  // once to count, so the CTA count stays moderate
  const int slots = T * kmax;
  const int chunks = slots > 0 ? (slots + kPermuteThreads - 1) / kPermuteThreads : 1;
  const int nb0 = chunks < 64 ? chunks : 64;
  const int per_block = (chunks + nb0 - 1) / nb0 * kPermuteThreads;
  const int nb = slots > 0 ? (slots + per_block - 1) / per_block : 1;
  return launch(permute_kernel, nb, kPermuteThreads, smem, reinterpret_cast<cudaStream_t>(stream),
                p, per_block);
}

}  // namespace

extern "C" moe_status_t moe_permute(const int32_t* topk_ids, const int32_t* k_dev, int T,
                                    int kmax, int E, int32_t* expert_counts,
                                    int32_t* expert_offsets, int32_t* sorted_assign,
                                    int32_t* inv_pos, moe_stream_t stream) {
  return permute_impl(topk_ids, k_dev, T, kmax, E, INT32_MAX, expert_counts, expert_offsets,
                      sorted_assign, inv_pos, stream);
}

extern "C" moe_status_t moe_permute_capped(const int32_t* topk_ids, const int32_t* k_dev, int T,
                                           int kmax, int E, int capacity,
                                           int32_t* expert_counts, int32_t* expert_offsets,
                                           int32_t* sorted_assign, int32_t* inv_pos,
                                           moe_stream_t stream) {
  if (capacity < 0) return MOE_ERR_INVALID_ARG;
  return permute_impl(topk_ids, k_dev, T, kmax, E, capacity, expert_counts, expert_offsets,
                      sorted_assign, inv_pos, stream);
}

// ---- token rows in expert order ------------------------------------------

namespace moe {
namespace {

constexpr int kRowsThreads = 256;
constexpr int kRowsUnroll = 4;

// x_sorted[r] = x[sorted[r] / kmax] for r < T*k, one warp per row, 16-byte
// vectors, kRowsUnroll loads in flight per lane.
__global__ void __launch_bounds__(kRowsThreads) permute_rows_kernel(
    const uint4* __restrict__ x, const int32_t* __restrict__ sorted,
    const int32_t* __restrict__ k_dev, int T, int kmax, int vec_per_row,
    uint4* __restrict__ out, unsigned int* err) {
  moe::pdl_wait();
  moe::pdl_trigger();
  const int k = min(max(*k_dev, 0), kmax);
  const int64_t rows = (int64_t)T * k;
  const int lane = threadIdx.x & 31;
  const int64_t wstride = (int64_t)gridDim.x * (kRowsThreads / 32);
  for (int64_t r = (int64_t)blockIdx.x * (kRowsThreads / 32) + (threadIdx.x >> 5); r < rows;
       r += wstride) {
    const int a = __ldg(sorted + r);
    if (a < 0 || a >= T * kmax) {
      if (lane == 0) raise_device_error(err, MOE_DEVERR_BAD_INDEX);
      continue;
    }
    const uint4* src = x + (int64_t)(a / kmax) * vec_per_row;
    uint4* dst = out + r * vec_per_row;
    for (int c0 = 0; c0 < vec_per_row; c0 += 32 * kRowsUnroll) {
      uint4 v[kRowsUnroll];
#pragma unroll
      for (int u = 0; u < kRowsUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < vec_per_row) v[u] = ldg_nc_v4(src + c);
      }
#pragma unroll
      for (int u = 0; u < kRowsUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < vec_per_row) dst[c] = v[u];
      }
    }
  }
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_permute_rows(const uint16_t* x, const int32_t* sorted_assign,
                                         const int32_t* k_dev, int T, int kmax, int H,
                                         uint16_t* x_sorted, moe_stream_t stream) {
  using namespace moe_host;
  if (T < 0 || kmax < 1 || kmax > 16 || (int64_t)T * kmax > (1 << 24)) return MOE_ERR_INVALID_ARG;
  if (H <= 0 || H % 8 != 0 || !k_dev) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  const void* ptrs[] = {x, sorted_assign, x_sorted};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)T * kmax;
  const int64_t warps_per_block = moe::kRowsThreads / 32;
  int64_t grid = (rows + warps_per_block - 1) / warps_per_block;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (grid > cap) grid = cap;
  return launch(moe::permute_rows_kernel, (int)grid, moe::kRowsThreads, 0,
                reinterpret_cast<cudaStream_t>(stream), reinterpret_cast<const uint4*>(x),
                sorted_assign, k_dev, T, kmax, H / 8, reinterpret_cast<uint4*>(x_sorted),
                device_error_word());
}

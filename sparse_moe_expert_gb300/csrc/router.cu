// Router: logits, softmax, entropy, top-k ids and weights, the batch's k.
//
// Page "Qwen3.5 Block在llama.cpp中的映射与优化原理", section 4.1 (linear
// router without bias, softmax, top-k); page "Qwen3.5-MoE与Qwen3-MoE架构差异
// 深度解析", sections 2.1-2.2 (top-k routing, entropy-aware k per batch).
//
// Kernel 1 (router_topk_kernel): a CTA takes up to kTokensPerCta tokens.
//   Phase A: every warp computes (token, expert) logits four at a time; lane
//   l owns the 8-element chunks c = l, l+32, ... of H and chains single-
//   rounding FMAs over them, then the 32 lane partials are combined by an
//   xor butterfly (16, 8, 4, 2, 1).  This is the fixed summation order that
//   makes the ids reproducible bit for bit.
//   Phase B: one warp per token: max, softmax sums, entropy, top-kmax by
//   repeated warp argmax (ties to the lower id), weights.
// Kernel 2 (router_finalize_kernel, or inline when one CTA covers the batch):
//   mean entropy over the batch in a fixed reduction order, the batch's k,
//   and for the adaptive rule the normalisation of the chosen k weights.
#include <cuda_fp16.h>
#include <math.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kRouterThreads = 512;
constexpr int kRouterWarps = kRouterThreads / 32;
constexpr int kTokensPerCta = 16;
constexpr int kMaxExperts = 1024;
constexpr int kFinalizeThreads = 256;

struct RouterParams {
  const uint16_t* x;
  const float* w;
  const float* bias;
  float inv_temp;
  int T, H, E, k_fixed, kmax;
  float thr1, thr2;
  int renorm;
  int32_t* ids;
  float* topw;
  int32_t* k_dev;
  float* mean_ent;
  float* ws_ent;  // [T] per-token entropy
  float* ws_sum;  // [T] softmax denominator over all experts
  unsigned int* err;
};

// The adaptive rule's largest k.
constexpr int kAdaptiveMaxK = 3;

__device__ __forceinline__ bool better(float v2, int i2, float v1, int i1) {
  // is (v2, i2) preferred over (v1, i1)?  larger value, then lower id
  if (i2 < 0) return false;
  if (i1 < 0) return true;
  return v2 > v1 || (v2 == v1 && i2 < i1);
}

// Batch mean entropy, k, and (adaptive) weight normalisation.  Run by one CTA.
__device__ void finalize_batch(const RouterParams& p) {
  __shared__ float part[kFinalizeThreads];
  __shared__ int k_sh;
  const int tid = threadIdx.x;
  const int nthr = blockDim.x < kFinalizeThreads ? blockDim.x : kFinalizeThreads;
  if (tid < nthr) {
    float acc = 0.0f;
    for (int t = tid; t < p.T; t += nthr) acc = __fadd_rn(acc, p.ws_ent[t]);
    part[tid] = acc;
  }
  __syncthreads();
  // fixed pairwise tree over the per-thread partials
  for (int w = nthr; w > 1;) {
    int half = (w + 1) >> 1;
    if (tid + half < w) part[tid] = __fadd_rn(part[tid], part[tid + half]);
    __syncthreads();
    w = half;
  }
  if (tid == 0) {
    float hbar = p.T > 0 ? __fdiv_rn(part[0], (float)p.T) : 0.0f;
    int k = p.k_fixed;
    if (k == 0) k = hbar < p.thr1 ? 1 : (hbar < p.thr2 ? 2 : 3);
    *p.k_dev = k;
    *p.mean_ent = hbar;
    k_sh = k;
  }
  __syncthreads();
  if (p.k_fixed != 0) return;
  const int k = k_sh;
  for (int t = tid; t < p.T; t += blockDim.x) {
    float ez[kAdaptiveMaxK];
    float denom = 0.0f;
    for (int j = 0; j < kAdaptiveMaxK; ++j) ez[j] = p.topw[(int64_t)t * p.kmax + j];
    if (p.renorm) {
      for (int j = 0; j < k; ++j) denom = __fadd_rn(denom, ez[j]);
    } else {
      denom = p.ws_sum[t];
    }
    for (int j = 0; j < p.kmax; ++j) {
      int64_t o = (int64_t)t * p.kmax + j;
      if (j < k) {
        p.topw[o] = __fdiv_rn(ez[j], denom);
      } else {
        p.topw[o] = 0.0f;
        p.ids[o] = -1;
      }
    }
  }
}

__global__ void __launch_bounds__(kRouterThreads) router_topk_kernel(RouterParams p) {
  extern __shared__ float logits_s[];  // [kTokensPerCta][E]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * kTokensPerCta;
  const int nt = min(kTokensPerCta, p.T - t0);
  const int E = p.E, H = p.H;
  const int nchunks = H >> 3;
  const int npairs = nt * E;

  // ---- Phase A: logits ---------------------------------------------------
  for (int base = warp * 4; base < npairs; base += kRouterWarps * 4) {
    float acc[4];
    const uint4* xrow[4];
    const float4* wrow[4];
    int tl[4], ex[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      int pidx = min(base + q, npairs - 1);
      tl[q] = pidx % nt;
      ex[q] = pidx / nt;
      xrow[q] = reinterpret_cast<const uint4*>(p.x + (int64_t)(t0 + tl[q]) * H);
      wrow[q] = reinterpret_cast<const float4*>(p.w + (int64_t)ex[q] * H);
      acc[q] = 0.0f;
    }
    for (int c = lane; c < nchunks; c += 32) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 xv = __ldg(xrow[q] + c);
        float4 w0 = __ldg(wrow[q] + 2 * c), w1 = __ldg(wrow[q] + 2 * c + 1);
        float2 x01 = bf16x2_to_f32x2(xv.x), x23 = bf16x2_to_f32x2(xv.y);
        float2 x45 = bf16x2_to_f32x2(xv.z), x67 = bf16x2_to_f32x2(xv.w);
        float a = acc[q];
        a = fmaf(x01.x, w0.x, a);
        a = fmaf(x01.y, w0.y, a);
        a = fmaf(x23.x, w0.z, a);
        a = fmaf(x23.y, w0.w, a);
        a = fmaf(x45.x, w1.x, a);
        a = fmaf(x45.y, w1.y, a);
        a = fmaf(x67.x, w1.z, a);
        a = fmaf(x67.y, w1.w, a);
        acc[q] = a;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1)
        acc[q] = __fadd_rn(acc[q], __shfl_xor_sync(0xFFFFFFFFu, acc[q], off));
    }
    if (lane == 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (base + q < npairs) {
          float v = acc[q];
          if (p.bias) v = __fadd_rn(v, __ldg(p.bias + ex[q]));
          v = __fmul_rn(v, p.inv_temp);
          logits_s[tl[q] * E + ex[q]] = v;
        }
      }
    }
  }
  __syncthreads();

  // ---- Phase B: softmax, entropy, top-k per token (one warp per token) ---
  const bool adaptive = p.k_fixed == 0;
  const int nsel = adaptive ? kAdaptiveMaxK : p.k_fixed;
  for (int tl = warp; tl < nt; tl += kRouterWarps) {
    const float* row = logits_s + tl * E;
    const int t = t0 + tl;
    float m = -INFINITY;
    for (int e = lane; e < E; e += 32) m = fmaxf(m, row[e]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    float s = 0.0f, s1 = 0.0f;
    for (int e = lane; e < E; e += 32) {
      float z = __fsub_rn(row[e], m);
      float ez = expf(z);
      s = __fadd_rn(s, ez);
      s1 = __fadd_rn(s1, __fmul_rn(ez, z));
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, off));
      s1 = __fadd_rn(s1, __shfl_xor_sync(0xFFFFFFFFu, s1, off));
    }
    const float ent = __fsub_rn(logf(s), __fdiv_rn(s1, s));

    // top-nsel by repeated warp argmax; lane owns e = lane + 32*j
    unsigned int taken = 0u;
    int sel[16];
    float selz[16];
    for (int r = 0; r < nsel; ++r) {
      float bv = -INFINITY;
      int bi = -1;
      for (int j = 0, e = lane; e < E; ++j, e += 32) {
        if (taken & (1u << j)) continue;
        float v = row[e];
        if (better(v, e, bv, bi)) { bv = v; bi = e; }
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
        int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if (bi >= 0 && (bi & 31) == lane) taken |= 1u << (bi >> 5);
      sel[r] = bi;
      selz[r] = expf(__fsub_rn(bv, m));
    }
    if (lane == 0) {
      int32_t* idr = p.ids + (int64_t)t * p.kmax;
      float* wr = p.topw + (int64_t)t * p.kmax;
      if (adaptive) {
        // weights are normalised once the batch's k is known
        for (int j = 0; j < p.kmax; ++j) {
          idr[j] = j < nsel ? sel[j] : -1;
          wr[j] = j < nsel ? selz[j] : 0.0f;
        }
      } else {
        float denom = 0.0f;
        if (p.renorm) {
          for (int j = 0; j < nsel; ++j) denom = __fadd_rn(denom, selz[j]);
        } else {
          denom = s;
        }
        for (int j = 0; j < p.kmax; ++j) {
          idr[j] = j < nsel ? sel[j] : -1;
          wr[j] = j < nsel ? __fdiv_rn(selz[j], denom) : 0.0f;
        }
      }
      p.ws_ent[t] = ent;
      p.ws_sum[t] = s;
    }
  }

  if (gridDim.x == 1) {
    __syncthreads();
    finalize_batch(p);
  }
}

__global__ void __launch_bounds__(kFinalizeThreads) router_finalize_kernel(RouterParams p) {
  finalize_batch(p);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_router_workspace_size(int T) {
  if (T < 0) return 0;
  size_t per = ((size_t)T * sizeof(float) + 255) / 256 * 256;
  return 2 * per + 256;
}

extern "C" moe_status_t moe_router_topk(const uint16_t* x, const float* w_router,
                                        const float* logit_bias, float inv_temperature, int T,
                                        int H, int E, int k_fixed, int kmax, float thr1,
                                        float thr2, int renormalize, int32_t* topk_ids,
                                        float* topk_w, int32_t* k_dev, float* mean_entropy,
                                        void* workspace, size_t workspace_bytes,
                                        moe_stream_t stream) {
  using namespace moe_host;
  if (T < 0 || H <= 0 || H % 64 != 0 || E < 1 || E > kMaxExperts || kmax < 1 || kmax > 16)
    return MOE_ERR_INVALID_ARG;
  if ((int64_t)T * kmax > (1 << 24)) return MOE_ERR_INVALID_ARG;
  if (k_fixed < 0 || k_fixed > kmax || k_fixed > E) return MOE_ERR_INVALID_ARG;
  if (k_fixed == 0 && (kmax < kAdaptiveMaxK || E < kAdaptiveMaxK)) return MOE_ERR_INVALID_ARG;
  if (!(thr1 <= thr2)) return MOE_ERR_INVALID_ARG;
  if (!k_dev || !mean_entropy || !workspace) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !w_router || !topk_ids || !topk_w)) return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < moe_router_workspace_size(T)) return MOE_ERR_INVALID_ARG;
  if ((x && !aligned16(x)) || (w_router && !aligned16(w_router)) || !aligned16(workspace))
    return MOE_ERR_INVALID_ARG;
  if (logit_bias && (reinterpret_cast<uintptr_t>(logit_bias) & 3u)) return MOE_ERR_INVALID_ARG;

  RouterParams p;
  p.x = x;
  p.w = w_router;
  p.bias = logit_bias;
  p.inv_temp = inv_temperature;
  p.T = T;
  p.H = H;
  p.E = E;
  p.k_fixed = k_fixed;
  p.kmax = kmax;
  p.thr1 = thr1;
  p.thr2 = thr2;
  p.renorm = renormalize ? 1 : 0;
  p.ids = topk_ids;
  p.topw = topk_w;
  p.k_dev = k_dev;
  p.mean_ent = mean_entropy;
  size_t per = ((size_t)T * sizeof(float) + 255) / 256 * 256;
  p.ws_ent = reinterpret_cast<float*>(workspace);
  p.ws_sum = reinterpret_cast<float*>(reinterpret_cast<char*>(workspace) + per);
  p.err = device_error_word();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  const int nblocks = (T + kTokensPerCta - 1) / kTokensPerCta;
  if (nblocks > 0) {
    size_t smem = (size_t)kTokensPerCta * E * sizeof(float);
    if (smem > 48 * 1024) {
      if (cudaFuncSetAttribute(router_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem) != cudaSuccess)
        return MOE_ERR_CUDA;
    }
    router_topk_kernel<<<nblocks, kRouterThreads, smem, st>>>(p);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
  }
  if (nblocks != 1) {
    router_finalize_kernel<<<1, kFinalizeThreads, 0, st>>>(p);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// ---------------------------------------------------------------------------
// moe_router_topk_noalloc: the same router for callers that cannot allocate.
//
// Some callers of this layer have no way to obtain device memory on demand:
// a model runner that reserves the whole device pool for itself at start-up
// and hands plugins only the tensors of their inputs and outputs, or a
// deployment that forbids allocation after initialisation because
// cudaMalloc can synchronize the device and stall a latency-bound decode
// loop.  This entry point needs nothing beyond its inputs and outputs: the
// per-token scratch (entropy and softmax denominator, two floats per token)
// lives in the file-scope array below, sized for
// MOE_ROUTER_NOALLOC_MAX_TOKENS tokens (512 KiB).  Every GPU that loads the
// library holds the array until the process exits.
//
// Host code must not pass the array's name to a kernel: on the host it is
// only a stand-in symbol.  Its device address is looked up once per device,
// with that device current, by the first call on that device
// (cudaGetSymbolAddress); make that first call before any stream capture.
// All calls share the array and it keeps the last call's contents; nothing
// in it needs to start at zero, because every entry a call reads was written
// earlier by the same call.  Calls whose executions overlap on the GPU (two
// streams, say) race on the array and must be ordered by the caller.
// ---------------------------------------------------------------------------
#include <mutex>

static __device__ __align__(256) float g_router_noalloc_scratch[2 * MOE_ROUTER_NOALLOC_MAX_TOKENS];

namespace {

constexpr int kNoallocMaxDevices = 64;
float* g_noalloc_scratch_ptr[kNoallocMaxDevices];
std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device.
moe_status_t noalloc_scratch(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kNoallocMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_router_noalloc_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    g_noalloc_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" moe_status_t moe_router_topk_noalloc(const uint16_t* x, const float* w_router,
                                                const float* logit_bias, float inv_temperature,
                                                int T, int H, int E, int k_fixed, int kmax,
                                                float thr1, float thr2, int renormalize,
                                                int32_t* topk_ids, float* topk_w, int32_t* k_dev,
                                                float* mean_entropy, moe_stream_t stream) {
  using namespace moe_host;
  if (T > MOE_ROUTER_NOALLOC_MAX_TOKENS) return MOE_ERR_INVALID_ARG;
  if (T < 0 || H <= 0 || H % 64 != 0 || E < 1 || E > kMaxExperts || kmax < 1 || kmax > 16)
    return MOE_ERR_INVALID_ARG;
  if (k_fixed < 0 || k_fixed > kmax || k_fixed > E) return MOE_ERR_INVALID_ARG;
  if (k_fixed == 0 && (kmax < kAdaptiveMaxK || E < kAdaptiveMaxK)) return MOE_ERR_INVALID_ARG;
  if (!(thr1 <= thr2)) return MOE_ERR_INVALID_ARG;
  if (!k_dev || !mean_entropy) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !w_router || !topk_ids || !topk_w)) return MOE_ERR_INVALID_ARG;
  if ((x && !aligned16(x)) || (w_router && !aligned16(w_router))) return MOE_ERR_INVALID_ARG;
  if (logit_bias && (reinterpret_cast<uintptr_t>(logit_bias) & 3u)) return MOE_ERR_INVALID_ARG;

  float* scratch = nullptr;
  const moe_status_t sst = noalloc_scratch(&scratch);
  if (sst != MOE_OK) return sst;

  RouterParams p;
  p.x = x;
  p.w = w_router;
  p.bias = logit_bias;
  p.inv_temp = inv_temperature;
  p.T = T;
  p.H = H;
  p.E = E;
  p.k_fixed = k_fixed;
  p.kmax = kmax;
  p.thr1 = thr1;
  p.thr2 = thr2;
  p.renorm = renormalize ? 1 : 0;
  p.ids = topk_ids;
  p.topw = topk_w;
  p.k_dev = k_dev;
  p.mean_ent = mean_entropy;
  p.ws_ent = scratch;
  p.ws_sum = scratch + MOE_ROUTER_NOALLOC_MAX_TOKENS;
  p.err = device_error_word();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  const int nblocks = (T + kTokensPerCta - 1) / kTokensPerCta;
  if (nblocks > 0) {
    size_t smem = (size_t)kTokensPerCta * E * sizeof(float);
    if (smem > 48 * 1024) {
      if (cudaFuncSetAttribute(router_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem) != cudaSuccess)
        return MOE_ERR_CUDA;
    }
    router_topk_kernel<<<nblocks, kRouterThreads, smem, st>>>(p);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
  }
  if (nblocks != 1) {
    router_finalize_kernel<<<1, kFinalizeThreads, 0, st>>>(p);
    if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

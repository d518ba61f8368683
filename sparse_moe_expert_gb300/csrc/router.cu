// Router: logits, softmax, entropy, top-k ids and weights, the batch's k.
//
// Page "Qwen3.5 Block在llama.cpp中的映射与优化原理", section 4.1 (linear
// router without bias, softmax, top-k); page "Qwen3.5-MoE与Qwen3-MoE架构差异
// 深度解析", sections 2.1-2.2 (top-k routing, entropy-aware k per batch).
//
// Kernel 1 (router_topk_kernel): a cluster of 8 CTAs takes a group of up to
// 32 tokens (16 when E > 256); CTA r of the cluster computes the logits of
// experts [r*E/8, (r+1)*E/8) and stores them into the leader CTA's shared
// memory (distributed shared memory), so the router weights are streamed by
// eight SMs at once.
//   Phase A: the fixed summation order that makes the ids reproducible bit
//   for bit: lane l of a warp owns the 8-element chunks c = l, l+32, ... of
//   H and chains single-rounding FMAs over them; the 32 lane partials are
//   combined by an xor butterfly (16, 8, 4, 2, 1).  A warp computes a tile
//   of 8 tokens x 4 experts at once (one token x one expert for groups of
//   fewer than 8 tokens), each (token, expert) value in that same order.
//   Small groups (the cluster's router-weight slice and token rows fit in
//   shared memory, e.g. decode): each CTA first brings them in with bulk
//   copies (one round trip to memory instead of one per 8-element chunk) and
//   runs the same chains from shared memory.
//   Phase B (leader CTA): one warp per token: max, softmax sums, entropy,
//   top-kmax by repeated warp argmax (ties to the lower id), weights.
// Kernel 2 (router_finalize_kernel, or inline when one cluster covers the
// batch): mean entropy over the batch in a fixed reduction order, the
// batch's k, and for the adaptive rule the normalisation of the chosen k
// weights.
#include <cuda_fp16.h>
#include <math.h>

#include "async.cuh"
#include "common.cuh"

namespace moe {
namespace {

constexpr int kRouterThreads = 512;
constexpr int kRouterWarps = kRouterThreads / 32;
constexpr int kRouterCluster = 8;  // CTAs per token group, splitting the experts
// Batches of many token groups use clusters of 4 (twice the experts per CTA):
// clusters of 8 CTAs at one CTA per SM leave a fifth of the SMs without a
// whole cluster's room.
constexpr int kRouterClusterWide = 4;
constexpr int kMaxExperts = 1024;

// Tokens per cluster: the leader holds [tokens][E] fp32 logits.
__host__ __device__ constexpr int router_group_tokens(int E) { return E <= 256 ? 32 : 16; }
constexpr int kFinalizeThreads = 256;
// Shared memory a CTA may stage for the small-batch path.
constexpr size_t kRouterStageBytes = 200 * 1024;

struct RouterParams {
  const uint16_t* x;
  const float* w;
  const float* bias;
  float inv_temp;
  int T, H, E, k_fixed, kmax;
  float thr1, thr2;
  int renorm;
  int smem_stage;  // bulk-copy the weight slice and token rows to shared memory
  int tpc;         // tokens per cluster (token group)
  int groups;      // > 0: group-limited selection, the best expert of each of
                   // `groups` groups of E / groups consecutive ids (k = groups)
  int32_t* ids;
  float* topw;
  int32_t* k_dev;
  float* mean_ent;
  float* ws_ent;  // [T] per-token entropy
  float* ws_sum;  // [T] softmax denominator over all experts
  // fused permute (one cluster covers the batch): outputs of moe_permute, or
  // null when a separate permute follows
  int32_t* pm_counts;
  int32_t* pm_offsets;
  int32_t* pm_sorted;
  int32_t* pm_inv_pos;
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

// The stable counting sort of moe_permute, run by the leader CTA once the
// batch's k is known (T * kmax <= blockDim, E <= 256).  Same result: for each
// expert, its assignments a = t * kmax + j (j < k) in ascending a.  `sm`
// holds at least (warps + 1) * E ints.
__device__ void fused_permute(const RouterParams& p, int* sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int E = p.E, slots = p.T * p.kmax;
  const int k = *p.k_dev;
  int* wh = sm;                 // [warp][E]: counts, then exclusive prefixes over warps
  int* off = wh + nwarps * E;   // [E]: totals, then offsets
  for (int i = tid; i < nwarps * E; i += blockDim.x) wh[i] = 0;
  __syncthreads();
  const int a = tid;
  int e = -1;
  if (a < slots && a % p.kmax < k) {
    const int v = p.ids[a];
    if (v >= 0 && v < E) e = v;
    else raise_device_error(p.err, MOE_DEVERR_BAD_EXPERT);
  }
  const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
  const int rank = __popc(peers & lanemask_lt());
  if (e >= 0 && rank == 0) wh[warp * E + e] = __popc(peers);
  __syncthreads();
  for (int x = tid; x < E; x += blockDim.x) {
    int run = 0;
    for (int w = 0; w < nwarps; ++w) {
      const int c = wh[w * E + x];
      wh[w * E + x] = run;
      run += c;
    }
    off[x] = run;
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int x0 = 0; x0 < E; x0 += 32) {
      const int x = x0 + lane;
      const int v = x < E ? off[x] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
      }
      if (x < E) {
        const int excl = carry + incl - v;
        off[x] = excl;
        p.pm_counts[x] = v;
        p.pm_offsets[x] = excl;
      }
      carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) p.pm_offsets[E] = carry;
  }
  __syncthreads();
  if (a < slots) {
    if (e >= 0) {
      const int pos = off[e] + wh[warp * E + e] + rank;
      p.pm_sorted[pos] = a;
      p.pm_inv_pos[a] = pos;
    } else {
      p.pm_inv_pos[a] = -1;
    }
  }
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(r)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}

// One 8-element chunk of the TM token rows and TN expert rows.
template <int TM, int TN>
struct RouterChunk {
  uint4 x[TM];
  float4 wa[TN], wb[TN];
};

template <int TM, int TN, bool SMEM>
__device__ __forceinline__ void load_chunk(RouterChunk<TM, TN>& d, const uint4* const (&xr)[TM],
                                           const float4* const (&wr)[TN], int c) {
#pragma unroll
  for (int m = 0; m < TM; ++m) d.x[m] = SMEM ? xr[m][c] : __ldg(xr[m] + c);
#pragma unroll
  for (int n = 0; n < TN; ++n) {
    d.wa[n] = SMEM ? wr[n][2 * c] : __ldg(wr[n] + 2 * c);
    d.wb[n] = SMEM ? wr[n][2 * c + 1] : __ldg(wr[n] + 2 * c + 1);
  }
}

// acc[m][n] = fma chain over the chunk's elements h = 0..7, in order.
template <int TM, int TN>
__device__ __forceinline__ void fma_chunk(float (&acc)[TM][TN], const RouterChunk<TM, TN>& d) {
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    float xf[TM], wf[TN];
#pragma unroll
    for (int m = 0; m < TM; ++m) {
      const uint32_t word = h < 2 ? d.x[m].x : h < 4 ? d.x[m].y : h < 6 ? d.x[m].z : d.x[m].w;
      xf[m] = (h & 1) ? __uint_as_float(word & 0xFFFF0000u) : __uint_as_float(word << 16);
    }
#pragma unroll
    for (int n = 0; n < TN; ++n) {
      const float4& q = h < 4 ? d.wa[n] : d.wb[n];
      const int hh = h & 3;
      wf[n] = hh == 0 ? q.x : hh == 1 ? q.y : hh == 2 ? q.z : q.w;
    }
#pragma unroll
    for (int m = 0; m < TM; ++m)
#pragma unroll
      for (int n = 0; n < TN; ++n) acc[m][n] = fmaf(xf[m], wf[n], acc[m][n]);
  }
}

// The xor butterfly (16, 8, 4, 2, 1) of 32 values per lane, as a reduce-
// scatter: at each step a lane keeps the half of its values that its bit
// selects and adds the partner's copy of that half.  Every sum is the one
// the full butterfly forms (a + b = b + a exactly), and lane l ends with the
// total of value l.
__device__ __forceinline__ float butterfly_scatter32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 16, c = 32; off >= 1; off >>= 1, c >>= 1) {
    const bool hi = (lane & off) != 0;
#pragma unroll
    for (int j = 0; j < c / 2; ++j) {
      const float keep = hi ? v[j + c / 2] : v[j];
      const float send = hi ? v[j] : v[j + c / 2];
      v[j] = __fadd_rn(keep, __shfl_xor_sync(0xFFFFFFFFu, send, off));
    }
  }
  return v[0];
}

// Logits of tokens [t0, t0+nt) x experts [e_lo, e_lo+ne) in warp tiles of
// TM tokens x TN experts, stored (after bias and temperature) into the
// leader's [token][E] array at cluster address `lead`.  SMEM: the token rows
// and weight rows are xs = x[t0 ..] and ws = w[e_lo ..] in shared memory.
template <int TM, int TN, bool SMEM>
__device__ __forceinline__ void router_logit_tiles(const RouterParams& p, int t0, int nt, int e_lo,
                                                   int ne, uint32_t lead, const uint16_t* xs,
                                                   const float* ws) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int H = p.H, E = p.E;
  const int nchunks = H >> 3;
  const int mtiles = (nt + TM - 1) / TM, ntiles = (ne + TN - 1) / TN;
  for (int tile = warp; tile < mtiles * ntiles; tile += kRouterWarps) {
    const int tm = tile % mtiles, tn = tile / mtiles;  // neighbouring warps share experts
    const uint4* xr[TM];
    const float4* wr[TN];
#pragma unroll
    for (int m = 0; m < TM; ++m)
      xr[m] = reinterpret_cast<const uint4*>(
          SMEM ? xs + (int64_t)min(tm * TM + m, nt - 1) * H
               : p.x + (int64_t)(t0 + min(tm * TM + m, nt - 1)) * H);
#pragma unroll
    for (int n = 0; n < TN; ++n)
      wr[n] = reinterpret_cast<const float4*>(
          SMEM ? ws + (int64_t)min(tn * TN + n, ne - 1) * H
               : p.w + (int64_t)(e_lo + min(tn * TN + n, ne - 1)) * H);
    constexpr bool kPacked = TM * TN == 32 && TM % 2 == 0;
    if constexpr (kPacked) {
      float2 acc2[TM / 2][TN];
#pragma unroll
      for (int m = 0; m < TM / 2; ++m)
#pragma unroll
        for (int n = 0; n < TN; ++n) acc2[m][n] = make_float2(0.0f, 0.0f);
      // chunks c = lane, lane+32, ...
#pragma unroll 1
      for (int c = lane; c < nchunks; c += 32) {
        // the chunk's token values, then its weights in two halves (h 0-3,
        // then 4-7), so fewer registers hold loaded data at once
        uint4 xv[TM];
        float4 wv[TN];
#pragma unroll
        for (int m = 0; m < TM; ++m) xv[m] = SMEM ? xr[m][c] : __ldg(xr[m] + c);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int n = 0; n < TN; ++n) wv[n] = SMEM ? wr[n][2 * c + half] : __ldg(wr[n] + 2 * c + half);
#pragma unroll
          for (int hh = 0; hh < 4; ++hh) {
            const int h = half * 4 + hh;
            float2 xp[TM / 2];
#pragma unroll
            for (int m = 0; m < TM; ++m) {
              const uint32_t word = h < 2 ? xv[m].x : h < 4 ? xv[m].y : h < 6 ? xv[m].z : xv[m].w;
              const float f = (h & 1) ? __uint_as_float(word & 0xFFFF0000u) : __uint_as_float(word << 16);
              if (m & 1) xp[m >> 1].y = f;
              else xp[m >> 1].x = f;
            }
#pragma unroll
            for (int n = 0; n < TN; ++n) {
              const float w = hh == 0 ? wv[n].x : hh == 1 ? wv[n].y : hh == 2 ? wv[n].z : wv[n].w;
              const float2 wp = make_float2(w, w);
#pragma unroll
              for (int mp = 0; mp < TM / 2; ++mp) acc2[mp][n] = __ffma2_rn(xp[mp], wp, acc2[mp][n]);
            }
          }
        }
      }
      // lane m*TN+n ends with the butterfly total of (m, n)
      float v[32];
#pragma unroll
      for (int m = 0; m < TM; ++m)
#pragma unroll
        for (int n = 0; n < TN; ++n) v[m * TN + n] = (m & 1) ? acc2[m >> 1][n].y : acc2[m >> 1][n].x;
      float tot = butterfly_scatter32(v);
      const int m = lane / TN, n = lane % TN;
      const int tl = tm * TM + m, el = tn * TN + n;
      if (tl < nt && el < ne) {
        const int e = e_lo + el;
        if (p.bias) tot = __fadd_rn(tot, __ldg(p.bias + e));
        tot = __fmul_rn(tot, p.inv_temp);
        st_cluster_f32(lead + (uint32_t)(tl * E + e) * 4u, tot);
      }
      continue;
    }
    float acc[TM][TN];
#pragma unroll
    for (int m = 0; m < TM; ++m)
#pragma unroll
      for (int n = 0; n < TN; ++n) acc[m][n] = 0.0f;
    // chunks c = lane, lane+32, ...
#pragma unroll(TM * TN == 1 ? 4 : 1)
    for (int c = lane; c < nchunks; c += 32) {
      RouterChunk<TM, TN> b;
      load_chunk<TM, TN, SMEM>(b, xr, wr, c);
      fma_chunk(acc, b);
    }
    // every lane ends with the butterfly total; lane m*TN+n stores (m, n)
#pragma unroll
    for (int m = 0; m < TM; ++m)
#pragma unroll
      for (int n = 0; n < TN; ++n) {
        float v = acc[m][n];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
          v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
        const int tl = tm * TM + m, el = tn * TN + n;
        if (lane == ((m * TN + n) & 31) && tl < nt && el < ne) {
          const int e = e_lo + el;
          if (p.bias) v = __fadd_rn(v, __ldg(p.bias + e));
          v = __fmul_rn(v, p.inv_temp);
          st_cluster_f32(lead + (uint32_t)(tl * E + e) * 4u, v);
        }
      }
  }
}

// Phase B for tokens [t0, t0 + nt) whose logits are in `logits_s`
// ([token][E], shared memory): softmax, entropy and top-k, one warp per
// token (warps 0 .. nwarps - 1 of the CTA).
__device__ void router_phase_b(const RouterParams& p, const float* logits_s, int t0, int nt,
                               int nwarps) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int E = p.E;
  const bool adaptive = p.k_fixed == 0;
  const int nsel = adaptive ? kAdaptiveMaxK : p.k_fixed;
  for (int tl = warp; tl < nt; tl += nwarps) {
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
    // grouped: round r takes the best expert of group r (page "Qwen3.5
    // Block在llama.cpp中的映射与优化原理", section 1.1), then the winners are
    // ordered as top-k orders its choice (larger logit, then lower id)
    const int gsz = p.groups > 0 ? E / p.groups : E;
    unsigned int taken = 0u;
    int sel[16];
    float selz[16], selv[16];
    for (int r = 0; r < nsel; ++r) {
      float bv = -INFINITY;
      int bi = -1;
      for (int j = 0, e = lane; e < E; ++j, e += 32) {
        if (taken & (1u << j)) continue;
        if (p.groups > 0 && e / gsz != r) continue;
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
      selv[r] = bv;
    }
    if (p.groups > 0 && lane == 0) {
      for (int i = 1; i < nsel; ++i)  // insertion sort: logit descending, id ascending
        for (int j = i; j > 0 && better(selv[j], sel[j], selv[j - 1], sel[j - 1]); --j) {
          const float tv = selv[j], tz = selz[j];
          const int ti = sel[j];
          selv[j] = selv[j - 1];
          selz[j] = selz[j - 1];
          sel[j] = sel[j - 1];
          selv[j - 1] = tv;
          selz[j - 1] = tz;
          sel[j - 1] = ti;
        }
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

}

template <int CL>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(kRouterThreads)
    router_topk_kernel(RouterParams p) {
  extern __shared__ __align__(16) float logits_s[];  // leader: [group tokens][E]
  __shared__ __align__(8) uint64_t stage_bar;
  const int E = p.E;
  const int tpc = p.tpc;
  const int t0 = (blockIdx.x / CL) * tpc;
  const int nt = min(tpc, p.T - t0);
  const uint32_t rank = cluster_ctarank();
  const int e_lo = (int)rank * E / CL;
  const int ne = ((int)rank + 1) * E / CL - e_lo;

  // ---- Phase A: logits (every CTA of the cluster, into the leader) -------
  // staged copies of the weight slice and token rows sit after the logits
  float* ws_s = logits_s + tpc * E;
  uint16_t* xs_s = reinterpret_cast<uint16_t*>(ws_s + (size_t)((E + CL - 1) / CL) * p.H);
  bool staged_ok = true;
  if (p.smem_stage) {
    if (threadIdx.x == 0) {
      mbar_init(&stage_bar, 1);
      fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && ne > 0) {
      const uint32_t wbytes = (uint32_t)ne * p.H * 4u, xbytes = (uint32_t)nt * p.H * 2u;
      mbar_arrive_expect_tx(&stage_bar, wbytes + xbytes);
      // one copy per weight row (no kernel of this library writes router
      // weights, so they are read before the wait on the previous kernel)
      for (int e = 0; e < ne; ++e)
        bulk_g2s(ws_s + (size_t)e * p.H, p.w + (int64_t)(e_lo + e) * p.H, (uint32_t)p.H * 4u,
                 &stage_bar);
    }
  }
  pdl_wait();
  pdl_trigger();
  if (p.smem_stage && threadIdx.x == 0 && ne > 0)
    bulk_g2s(xs_s, p.x + (int64_t)t0 * p.H, (uint32_t)nt * p.H * 2u, &stage_bar);  // token rows
  cluster_sync();  // the leader's shared memory is live before remote stores
  const uint32_t lead = cluster_map(logits_s, 0);
  if (p.smem_stage && ne > 0) {
    staged_ok = mbar_wait(&stage_bar, 0, kWaitBudgetCycles);
    if (!staged_ok && threadIdx.x == 0) raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
  }
  if (ne > 0 && staged_ok) {
    // tiles of 8 tokens x 4 experts unless that leaves fewer than 4 warps
    // busy; then 8 tokens x 1 expert (more warps on a small group; each
    // re-reads the token rows, which costs more than idle warps otherwise)
    const bool wide_tiles = ((nt + 7) / 8) * ((ne + 3) / 4) >= 4;
    if (p.smem_stage) {
      if (nt >= 8 && wide_tiles) router_logit_tiles<8, 4, true>(p, t0, nt, e_lo, ne, lead, xs_s, ws_s);
      else if (nt >= 8) router_logit_tiles<8, 1, true>(p, t0, nt, e_lo, ne, lead, xs_s, ws_s);
      else router_logit_tiles<1, 1, true>(p, t0, nt, e_lo, ne, lead, xs_s, ws_s);
    } else {
      if (nt >= 8 && wide_tiles)
        router_logit_tiles<8, 4, false>(p, t0, nt, e_lo, ne, lead, nullptr, nullptr);
      else if (nt >= 8)
        router_logit_tiles<8, 1, false>(p, t0, nt, e_lo, ne, lead, nullptr, nullptr);
      else router_logit_tiles<1, 1, false>(p, t0, nt, e_lo, ne, lead, nullptr, nullptr);
    }
  }
  cluster_sync();  // all logits of the group are in the leader
  if (rank != 0) return;

  // ---- Phase B: softmax, entropy, top-k per token (one warp per token) ---
  router_phase_b(p, logits_s, t0, nt, kRouterWarps);

  if (gridDim.x == CL) {
    __syncthreads();
    finalize_batch(p);
    if (p.pm_sorted) {
      __syncthreads();
      fused_permute(p, reinterpret_cast<int*>(logits_s));  // the logits are no longer needed
    }
  }
}

// The batch finalize; with the grouping requested (E <= 256, T kmax <= the
// CTA's threads) the stable counting sort follows in the same CTA.
constexpr int kFinalizePermuteThreads = 512;
__global__ void __launch_bounds__(kFinalizePermuteThreads) router_finalize_kernel(RouterParams p) {
  __shared__ int fp_scratch[(kFinalizePermuteThreads / 32 + 1) * 256];
  pdl_wait();
  pdl_trigger();
  finalize_batch(p);
  if (p.pm_sorted) {
    __syncthreads();
    fused_permute(p, fp_scratch);
  }
}

// ---------------------------------------------------------------------------
// Small batches (decode: up to kSmallMaxT tokens).  The router weight is
// spread over a cluster of up to 16 CTAs instead of 8, one warp per expert,
// so each SM brings in E / 16 weight rows (16 KB each for H 4096) before the
// previous kernel ends; the token rows follow once it has.  Each warp runs
// the canonical chains for its expert and every token, the leader CTA
// receives the logits through distributed shared memory and does phase B,
// the batch finalize and the fused grouping.
constexpr int kSmallMaxT = 8;
constexpr size_t kSmallStageBytes = 160 * 1024;  // weight rows + token rows per CTA
// with the leader's logits (T E floats) or the grouping's scratch ((warps + 1) E ints)
constexpr size_t kSmallMaxSmem = 200 * 1024;

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Order-preserving map of fp32 values onto uint32 (larger value, larger key).
__device__ __forceinline__ uint32_t f32_key(float v) {
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_f32(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Phase B, the batch finalize and the grouping of a small batch in one warp
// (T <= kSmallMaxT tokens, E <= 256, T * kmax <= 32): the results of
// router_phase_b, finalize_batch and fused_permute (sums in the same
// orders), with the selections in registers and shared memory and no
// CTA-wide barriers.  Maxima and argmaxima use the warp's hardware
// reductions on order-preserving keys (equal logits: the lower id).  The
// batch mean entropy is the pairwise tree over 32 slots, zeros past T.
// `scratch` is the logits' region: the counts and offsets (2 E words) take
// its start once the logits are no longer needed, the selected ids and
// weights (2 T kmax words) lie past max(2 E, T E) words.
__device__ void router_tail_warp(const RouterParams& p, const float* logits_s, int* scratch) {
  constexpr int kEL = 8;  // logits per lane
  const int lane = threadIdx.x & 31;
  const int E = p.E, T = p.T, kmax = p.kmax;
  const bool adaptive = p.k_fixed == 0;
  const int nsel = adaptive ? kAdaptiveMaxK : p.k_fixed;
  const int gsz = p.groups > 0 ? E / p.groups : E;
  int* ids_s = scratch + max(2 * E, T * E);                    // [T * kmax], past the logits
  float* w_s = reinterpret_cast<float*>(ids_s + T * kmax);     // [T * kmax]
  float ent_mine = 0.0f;  // lane t: token t's entropy
  float sum_mine = 0.0f;  // lane t: token t's softmax denominator
  for (int t = 0; t < T; ++t) {
    const float* row = logits_s + t * E;
    float lv[kEL];
#pragma unroll
    for (int j = 0; j < kEL; ++j) lv[j] = lane + 32 * j < E ? row[lane + 32 * j] : -INFINITY;
    float ml = -INFINITY;
#pragma unroll
    for (int j = 0; j < kEL; ++j) ml = fmaxf(ml, lv[j]);
    const float m = key_f32(__reduce_max_sync(0xFFFFFFFFu, f32_key(ml)));
    float sm = 0.0f, s1 = 0.0f;
#pragma unroll
    for (int j = 0; j < kEL; ++j) {
      if (lane + 32 * j < E) {
        const float z = __fsub_rn(lv[j], m);
        const float ez = expf(z);
        sm = __fadd_rn(sm, ez);
        s1 = __fadd_rn(s1, __fmul_rn(ez, z));
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      sm = __fadd_rn(sm, __shfl_xor_sync(0xFFFFFFFFu, sm, off));
      s1 = __fadd_rn(s1, __shfl_xor_sync(0xFFFFFFFFu, s1, off));
    }
    const float ent = __fsub_rn(logf(sm), __fdiv_rn(s1, sm));
    // top-nsel by repeated warp argmax (grouped: round r within group r)
    unsigned taken = 0u;
    int my_id = -1;
    float my_v = -INFINITY;
    for (int r = 0; r < nsel; ++r) {
      float bv = -INFINITY;
      int bi = 0x7FFFFFFF;
#pragma unroll
      for (int j = 0; j < kEL; ++j) {
        const int e = lane + 32 * j;
        if (e < E && !(taken & (1u << j)) && (p.groups <= 0 || e / gsz == r) &&
            (lv[j] > bv || bi == 0x7FFFFFFF)) {
          bv = lv[j];
          bi = e;
        }
      }
      const uint32_t mk = __reduce_max_sync(0xFFFFFFFFu, bi == 0x7FFFFFFF ? 0u : f32_key(bv));
      const int wi = (int)__reduce_min_sync(
          0xFFFFFFFFu, (bi != 0x7FFFFFFF && f32_key(bv) == mk) ? (unsigned)bi : 0x7FFFFFFFu);
      if ((wi & 31) == lane) taken |= 1u << (wi >> 5);
      if (lane == r) {
        my_id = wi;
        my_v = key_f32(mk);
      }
    }
    const float my_z = lane < nsel ? expf(__fsub_rn(my_v, m)) : 0.0f;
    // output slot of lane r's winner: its rank in the top-k order (larger
    // logit, then lower id); the rounds of plain top-k are already in it
    int slot = lane;
    if (p.groups > 0) {
      slot = 0;
      for (int q = 0; q < nsel; ++q) {
        const float qv = __shfl_sync(0xFFFFFFFFu, my_v, q);
        const int qi = __shfl_sync(0xFFFFFFFFu, my_id, q);
        if (q != lane && better(qv, qi, my_v, my_id)) ++slot;
      }
    }
    // the selected exponentials in slot order, summed in that order
    float denom = 0.0f;
    if (!adaptive) {
      if (p.renorm) {
        for (int j = 0; j < nsel; ++j) {
          const unsigned src = __ballot_sync(0xFFFFFFFFu, lane < nsel && slot == j);
          denom = __fadd_rn(denom, __shfl_sync(0xFFFFFFFFu, my_z, __ffs(src) - 1));
        }
      } else {
        denom = sm;
      }
    }
    if (lane < nsel) {
      ids_s[t * kmax + slot] = my_id;
      w_s[t * kmax + slot] = adaptive ? my_z : __fdiv_rn(my_z, denom);
    } else if (lane < kmax) {
      ids_s[t * kmax + lane] = -1;
      w_s[t * kmax + lane] = 0.0f;
    }
    if (lane == t) {
      ent_mine = ent;
      sum_mine = sm;
    }
  }
  __syncwarp();
  // batch mean entropy and k
  float acc = lane < T ? ent_mine : 0.0f;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_down_sync(0xFFFFFFFFu, acc, off));
  const float hbar = __fdiv_rn(__shfl_sync(0xFFFFFFFFu, acc, 0), (float)T);
  int k = p.k_fixed;
  if (k == 0) k = hbar < p.thr1 ? 1 : (hbar < p.thr2 ? 2 : 3);
  if (adaptive) {
    // the chosen k weights of every token renormalised (or over all experts)
    for (int t = 0; t < T; ++t) {
      const float ez = lane < kmax ? w_s[t * kmax + lane] : 0.0f;
      float den = 0.0f;
      if (p.renorm) {
        for (int j = 0; j < k; ++j) den = __fadd_rn(den, __shfl_sync(0xFFFFFFFFu, ez, j));
      } else {
        den = __shfl_sync(0xFFFFFFFFu, sum_mine, t);
      }
      __syncwarp();
      if (lane < kmax) {
        if (lane < k) {
          w_s[t * kmax + lane] = __fdiv_rn(ez, den);
        } else {
          w_s[t * kmax + lane] = 0.0f;
          ids_s[t * kmax + lane] = -1;
        }
      }
    }
  }
  __syncwarp();
  // outputs
  const int slots = T * kmax;
  for (int a = lane; a < slots; a += 32) {
    p.ids[a] = ids_s[a];
    p.topw[a] = w_s[a];
  }
  if (lane < T) {
    p.ws_ent[lane] = ent_mine;
    p.ws_sum[lane] = sum_mine;
  }
  if (lane == 0) {
    *p.k_dev = k;
    *p.mean_ent = hbar;
  }
  if (!p.pm_sorted) return;
  // the stable counting sort of moe_permute: counts, offsets, sorted rows
  int* cnt = scratch;
  int* off = scratch + E;
  for (int x = lane; x < E; x += 32) cnt[x] = 0;
  __syncwarp();
  const int a = lane;
  int e = -1;
  if (a < slots && a % kmax < k) {
    const int v = ids_s[a];
    if (v >= 0 && v < E) e = v;
    else raise_device_error(p.err, MOE_DEVERR_BAD_EXPERT);
  }
  if (e >= 0) atomicAdd(&cnt[e], 1);
  __syncwarp();
  const int chunk = (E + 31) / 32;
  const int x0 = min(E, lane * chunk), x1 = min(E, x0 + chunk);
  int run = 0;
  for (int x = x0; x < x1; ++x) run += cnt[x];
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  int pos0 = incl - run;
  for (int x = x0; x < x1; ++x) {
    const int c = cnt[x];
    off[x] = pos0;
    p.pm_counts[x] = c;
    p.pm_offsets[x] = pos0;
    pos0 += c;
  }
  if (lane == 31) p.pm_offsets[E] = incl;
  __syncwarp();
  const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
  const int rank = __popc(peers & lanemask_lt());
  if (a < slots) {
    if (e >= 0) {
      const int pos = off[e] + rank;
      p.pm_sorted[pos] = a;
      p.pm_inv_pos[a] = pos;
    } else {
      p.pm_inv_pos[a] = -1;
    }
  }
}

__global__ void __launch_bounds__(512, 1) router_small_kernel(RouterParams p, int lg_floats) {
  extern __shared__ __align__(16) float rs_smem[];
  float* logits_s = rs_smem;                 // leader: [T][E]; then the grouping's scratch
  float* ws_s = rs_smem + lg_floats;         // this CTA's weight rows [ne][H]
  __shared__ __align__(8) uint64_t wbar, xbar;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int E = p.E, H = p.H, nt = p.T;
  const uint32_t rank = cluster_ctarank();
  const int CL = (int)(gridDim.x);  // one cluster
  const int e_lo = (int)rank * E / CL;
  const int ne = ((int)rank + 1) * E / CL - e_lo;
  uint16_t* xs_s = reinterpret_cast<uint16_t*>(ws_s + (size_t)ne * H);
  cluster_arrive_relaxed();  // this CTA is running (waited for before remote stores)
  if (threadIdx.x == 0) {
    mbar_init(&wbar, 1);
    mbar_init(&xbar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && ne > 0) {
    // the weight rows: no kernel of this library writes router weights, so
    // they are read before the wait on the previous kernel
    mbar_arrive_expect_tx(&wbar, (uint32_t)ne * H * 4u);
    for (int e = 0; e < ne; ++e)
      bulk_g2s(ws_s + (size_t)e * H, p.w + (int64_t)(e_lo + e) * H, (uint32_t)H * 4u, &wbar);
  }
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0 && ne > 0) {
    mbar_arrive_expect_tx(&xbar, (uint32_t)nt * H * 2u);
    bulk_g2s(xs_s, p.x, (uint32_t)nt * H * 2u, &xbar);
  }
  bool ok = true;
  if (ne > 0) {
    ok = mbar_wait(&wbar, 0, kWaitBudgetCycles) && mbar_wait(&xbar, 0, kWaitBudgetCycles);
    if (!ok && lane == 0) raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
  }
  cluster_wait();
  const uint32_t lead = cluster_map(logits_s, 0);
  // ---- logits: warp w takes experts e_lo + w, + nwarps, ...; lane l the
  // chunks l, l + 32, ... of every token, in the canonical order
  const int nchunks = H >> 3;
  for (int el = warp; ok && el < ne; el += nwarps) {
    const float4* wr = reinterpret_cast<const float4*>(ws_s + (size_t)el * H);
    const int e = e_lo + el;
    const float bias = p.bias ? __ldg(p.bias + e) : 0.0f;
    for (int t = 0; t < nt; ++t) {
      const uint4* xr = reinterpret_cast<const uint4*>(xs_s + (size_t)t * H);
      float acc = 0.0f;
      for (int c = lane; c < nchunks; c += 32) {
        const float4 wa = wr[2 * c], wb = wr[2 * c + 1];
        const uint4 xv = xr[c];
        const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          const float xf = (h & 1) ? __uint_as_float(xw[h >> 1] & 0xFFFF0000u)
                                   : __uint_as_float(xw[h >> 1] << 16);
          acc = fmaf(xf, wv[h], acc);
        }
      }
      float v = acc;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
      if (lane == 0) {
        if (p.bias) v = __fadd_rn(v, bias);
        v = __fmul_rn(v, p.inv_temp);
        st_cluster_f32(lead + (uint32_t)(t * E + e) * 4u, v);
      }
    }
  }
  cluster_sync();  // every logit is in the leader
  if (rank != 0) return;
  if (E <= 256 && nt * p.kmax <= 32) {
    if (warp == 0) router_tail_warp(p, logits_s, reinterpret_cast<int*>(logits_s));
    return;
  }
  router_phase_b(p, logits_s, 0, nt, nwarps);
  __syncthreads();
  finalize_batch(p);
  if (p.pm_sorted) {
    __syncthreads();
    fused_permute(p, reinterpret_cast<int*>(logits_s));  // the logits are no longer needed
  }
}

// The cluster size for the small-batch router: 16 CTAs where the device can
// co-schedule such a cluster and E >= 16, else 8 (or E when smaller).
int small_router_cluster(int E, int threads, size_t smem) {
  static int can16[moe_host::kMaxCachedDevices] = {};  // 0 unknown, 1 yes, -1 no
  const int dev = moe_host::device_index();
  if (E >= 16 && can16[dev] == 0) {
    can16[dev] = -1;
    // the occupancy query honours the kernel's shared-memory limit: raise it
    // to the most this launcher asks for first
    if (cudaFuncSetAttribute(router_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmallMaxSmem) == cudaSuccess &&
        cudaFuncSetAttribute(router_small_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed,
                             1) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(16);
      cfg.blockDim = dim3(threads);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 16;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, router_small_kernel, &cfg) == cudaSuccess && n > 0)
        can16[dev] = 1;
    }
    cudaGetLastError();
  }
  if (E >= 16 && can16[dev] > 0) return 16;
  return E >= 8 ? 8 : E;
}

// Launches the small-batch router if the batch qualifies; false: use the
// general kernels.
bool launch_router_small(const RouterParams& p, cudaStream_t st, moe_status_t* status) {
  if (p.T < 1 || p.T > kSmallMaxT || p.groups < 0) return false;
  const int wcl = p.E >= 16 ? 16 : (p.E >= 8 ? 8 : p.E);  // widest cluster considered
  const int ne_max = (p.E + 7) / 8;                        // experts per CTA at 8 CTAs
  const size_t stage = (size_t)ne_max * p.H * 4 + (size_t)p.T * p.H * 2;
  if (stage > kSmallStageBytes) return false;
  // the leader's logits, then the grouping's scratch ((warps + 1) E ints)
  const int warps_max = (p.E + 7) / 8 > 16 ? 16 : (p.E + 7) / 8;
  if (p.pm_sorted && (p.T * p.kmax > 32 * warps_max || p.E > 256)) return false;
  int cl = 0;
  for (int pass = 0; pass < 2; ++pass) {
    const int c = pass == 0 ? wcl : (wcl == 16 ? 8 : wcl);
    const int ne = (p.E + c - 1) / c;
    const int warps = ne > 16 ? 16 : (ne < 1 ? 1 : ne);
    // the leader's logits, the block grouping's scratch, or the one-warp
    // tail's scratch (counts, offsets, ids and weights)
    int lg = p.T > warps + 1 ? p.T * p.E : (warps + 1) * p.E;
    lg = max(lg, max(2 * p.E, p.T * p.E) + 2 * p.T * p.kmax);
    lg = (lg + 3) & ~3;  // the weight rows after it start 16-byte aligned
    const size_t smem = (size_t)lg * 4 + (size_t)ne * p.H * 4 + (size_t)p.T * p.H * 2;
    if (pass == 0) {
      const int got = small_router_cluster(p.E, warps * 32, smem);
      if (got != c) continue;
    }
    if (p.pm_sorted && p.T * p.kmax > warps * 32) return false;
    cl = c;
    static bool set_max[moe_host::kMaxCachedDevices] = {};
    const int dev = moe_host::device_index();
    if (smem > kSmallMaxSmem) return false;
    if (!set_max[dev]) {
      if (cudaFuncSetAttribute(router_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kSmallMaxSmem) != cudaSuccess) {
        *status = MOE_ERR_CUDA;
        return true;
      }
      set_max[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cl);
    cfg.blockDim = dim3(warps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = moe_host::pdl_enabled() ? 2 : 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, router_small_kernel, p, lg);
    if (e != cudaSuccess) cudaGetLastError();
    *status = e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    return true;
  }
  return false;
}

// Kernel 1 over ceil(T / group) clusters, then the batch finalize unless a
// single cluster did it inline.
// Tokens per cluster: one group of 32 (16 when E > 256) for small batches;
// for larger ones groups as small as 8 tokens, so that the clusters cover the
// SMs (a 64-token batch takes 8 clusters rather than 2).
int router_tokens_per_group(int T, int E) {
  const int base = router_group_tokens(E);
  if (T <= base) return base;
  const int want = (int)(((int64_t)T * kRouterCluster + moe_host::sm_count() - 1) /
                         moe_host::sm_count());
  int tpc = 8;
  while (tpc < want && tpc < base) tpc <<= 1;
  return tpc;
}

// Large batches (at least 8 tokens per SM): one CTA per token group with
// every expert, so a warp walks several tiles of the same token rows and
// the group's logits, softmax and top-k stay in its own shared memory.  The
// group size (32, 16 or 8 tokens) minimises waves x tokens per group.
int router_single_cta_tokens(int T, int E) {
  const int sms = moe_host::sm_count();
  if ((int64_t)T < 8LL * sms) return 0;
  int best = 0;
  int64_t best_cost = 0;
  for (int tpc = router_group_tokens(E); tpc >= 8; tpc >>= 1) {
    const int64_t groups = (T + tpc - 1) / tpc;
    const int64_t cost = (groups + sms - 1) / sms * tpc;
    if (best == 0 || cost < best_cost) {
      best = tpc;
      best_cost = cost;
    }
  }
  return best;
}

moe_status_t launch_router(const RouterParams& p, cudaStream_t st) {
  using namespace moe_host;
  moe_status_t small_status = MOE_OK;
  if (launch_router_small(p, st, &small_status)) return small_status;
  const int single_tpc = router_single_cta_tokens(p.T, p.E);
  const int tpc = single_tpc ? single_tpc : router_tokens_per_group(p.T, p.E);
  const int ngroups = (p.T + tpc - 1) / tpc;
  if (ngroups > 0 && single_tpc) {
    const size_t smem = (size_t)tpc * p.E * sizeof(float);
    RouterParams q = p;
    q.tpc = tpc;
    q.smem_stage = 0;
    auto kern = router_topk_kernel<1>;
    static size_t set_max1[kMaxCachedDevices] = {};
    const int dev = device_index();
    if (smem > 48 * 1024 && smem > set_max1[dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess)
        return MOE_ERR_CUDA;
      set_max1[dev] = smem;
    }
    if (launch(kern, ngroups, kRouterThreads, smem, st, q) != MOE_OK) return MOE_ERR_CUDA;
  } else if (ngroups > 0) {
    size_t smem = (size_t)tpc * p.E * sizeof(float);
    // more token groups than a wave of 8-CTA clusters fills: clusters of 4
    const bool wide = (int64_t)ngroups * kRouterCluster > sm_count();
    const int cl = wide ? kRouterClusterWide : kRouterCluster;
    // small batches: the per-CTA weight slice and the token rows in shared memory
    const int ne_max = (p.E + cl - 1) / cl;
    const int nt_max = p.T < tpc ? p.T : tpc;
    const size_t staged = smem + (size_t)ne_max * p.H * 4 + (size_t)nt_max * p.H * 2;
    RouterParams q = p;
    q.tpc = tpc;
    q.smem_stage = (ngroups == 1 && staged <= kRouterStageBytes) ? 1 : 0;
    if (q.smem_stage) smem = staged;
    auto kern = wide ? router_topk_kernel<kRouterClusterWide> : router_topk_kernel<kRouterCluster>;
    static size_t set_max[2][kMaxCachedDevices] = {};  // per kernel and device
    const int dev = device_index();
    if (smem > 48 * 1024 && smem > set_max[wide][dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess)
        return MOE_ERR_CUDA;
      set_max[wide][dev] = smem;
    }
    if (launch(kern, ngroups * cl, kRouterThreads, smem, st, q) != MOE_OK) return MOE_ERR_CUDA;
  }
  if (ngroups != 1) {
    // the grouping rides along when the caller asked for it (route_impl
    // checks that it fits one CTA)
    RouterParams q = p;
    q.tpc = tpc;
    const int threads = q.pm_sorted ? kFinalizePermuteThreads : kFinalizeThreads;
    if (launch(router_finalize_kernel, 1, threads, 0, st, q) != MOE_OK) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" size_t moe_router_workspace_size(int T) {
  if (T < 0) return 0;
  size_t per = ((size_t)T * sizeof(float) + 255) / 256 * 256;
  return 2 * per + 256;
}

namespace {

// Validates the router arguments and fills the kernel parameters.
moe_status_t router_params(const uint16_t* x, const float* w_router, const float* logit_bias,
                           float inv_temperature, int T, int H, int E, int k_fixed, int kmax,
                           float thr1, float thr2, int renormalize, int32_t* topk_ids,
                           float* topk_w, int32_t* k_dev, float* mean_entropy, void* workspace,
                           size_t workspace_bytes, RouterParams* out) {
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

  RouterParams p{};
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
  p.smem_stage = 0;
  p.groups = 0;
  p.ids = topk_ids;
  p.topw = topk_w;
  p.k_dev = k_dev;
  p.mean_ent = mean_entropy;
  size_t per = ((size_t)T * sizeof(float) + 255) / 256 * 256;
  p.ws_ent = reinterpret_cast<float*>(workspace);
  p.ws_sum = reinterpret_cast<float*>(reinterpret_cast<char*>(workspace) + per);
  p.pm_counts = p.pm_offsets = p.pm_sorted = p.pm_inv_pos = nullptr;
  p.err = device_error_word();
  *out = p;
  return MOE_OK;
}

}  // namespace

extern "C" moe_status_t moe_router_topk(const uint16_t* x, const float* w_router,
                                        const float* logit_bias, float inv_temperature, int T,
                                        int H, int E, int k_fixed, int kmax, float thr1,
                                        float thr2, int renormalize, int32_t* topk_ids,
                                        float* topk_w, int32_t* k_dev, float* mean_entropy,
                                        void* workspace, size_t workspace_bytes,
                                        moe_stream_t stream) {
  RouterParams p{};
  const moe_status_t s = router_params(x, w_router, logit_bias, inv_temperature, T, H, E, k_fixed,
                                       kmax, thr1, thr2, renormalize, topk_ids, topk_w, k_dev,
                                       mean_entropy, workspace, workspace_bytes, &p);
  if (s != MOE_OK) return s;
  return launch_router(p, reinterpret_cast<cudaStream_t>(stream));
}

namespace {

moe_status_t route_impl(const uint16_t* x, const float* w_router, const float* logit_bias,
                        float inv_temperature, int T, int H, int E, int k_fixed, int kmax,
                        float thr1, float thr2, int renormalize, int32_t* topk_ids,
                        float* topk_w, int32_t* k_dev, float* mean_entropy, void* workspace,
                        size_t workspace_bytes, int32_t* expert_counts, int32_t* expert_offsets,
                        int32_t* sorted_assign, int32_t* inv_pos, int groups,
                        moe_stream_t stream) {
  RouterParams p{};
  moe_status_t s = router_params(x, w_router, logit_bias, inv_temperature, T, H, E, k_fixed,
                                 kmax, thr1, thr2, renormalize, topk_ids, topk_w, k_dev,
                                 mean_entropy, workspace, workspace_bytes, &p);
  if (s != MOE_OK) return s;
  if (groups < 0 || (groups > 0 && (E % groups != 0 || k_fixed != groups)))
    return MOE_ERR_INVALID_ARG;
  p.groups = groups;
  if (!expert_counts || !expert_offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!sorted_assign || !inv_pos)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the grouping inside the router's launches when it fits one CTA: the
  // leader of a single cluster, or the batch finalize of several clusters
  if (T > 0 && E <= 256 && T * kmax <= kRouterThreads) {
    p.pm_counts = expert_counts;
    p.pm_offsets = expert_offsets;
    p.pm_sorted = sorted_assign;
    p.pm_inv_pos = inv_pos;
    return launch_router(p, st);
  }
  s = launch_router(p, st);
  if (s != MOE_OK) return s;
  return moe_permute(topk_ids, k_dev, T, kmax, E, expert_counts, expert_offsets, sorted_assign,
                     inv_pos, stream);
}

}  // namespace

extern "C" moe_status_t moe_route(const uint16_t* x, const float* w_router,
                                  const float* logit_bias, float inv_temperature, int T, int H,
                                  int E, int k_fixed, int kmax, float thr1, float thr2,
                                  int renormalize, int32_t* topk_ids, float* topk_w,
                                  int32_t* k_dev, float* mean_entropy, void* workspace,
                                  size_t workspace_bytes, int32_t* expert_counts,
                                  int32_t* expert_offsets, int32_t* sorted_assign,
                                  int32_t* inv_pos, moe_stream_t stream) {
  return route_impl(x, w_router, logit_bias, inv_temperature, T, H, E, k_fixed, kmax, thr1, thr2,
                    renormalize, topk_ids, topk_w, k_dev, mean_entropy, workspace,
                    workspace_bytes, expert_counts, expert_offsets, sorted_assign, inv_pos, 0,
                    stream);
}

extern "C" moe_status_t moe_route_grouped(const uint16_t* x, const float* w_router,
                                          const float* logit_bias, float inv_temperature, int T,
                                          int H, int E, int n_groups, int kmax, int renormalize,
                                          int32_t* topk_ids, float* topk_w, int32_t* k_dev,
                                          float* mean_entropy, void* workspace,
                                          size_t workspace_bytes, int32_t* expert_counts,
                                          int32_t* expert_offsets, int32_t* sorted_assign,
                                          int32_t* inv_pos, moe_stream_t stream) {
  if (n_groups < 1) return MOE_ERR_INVALID_ARG;
  return route_impl(x, w_router, logit_bias, inv_temperature, T, H, E, n_groups, kmax, 1.2f,
                    2.5f, renormalize, topk_ids, topk_w, k_dev, mean_entropy, workspace,
                    workspace_bytes, expert_counts, expert_offsets, sorted_assign, inv_pos,
                    n_groups, stream);
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

  RouterParams p{};
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
  p.smem_stage = 0;
  p.groups = 0;
  p.ids = topk_ids;
  p.topw = topk_w;
  p.k_dev = k_dev;
  p.mean_ent = mean_entropy;
  p.ws_ent = scratch;
  p.ws_sum = scratch + MOE_ROUTER_NOALLOC_MAX_TOKENS;
  p.err = device_error_word();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  return launch_router(p, st);
}

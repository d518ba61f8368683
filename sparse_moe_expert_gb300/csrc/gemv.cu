// Grouped GEMV on CUDA cores: the decode / small-batch path of the two
// quantized products (gate_up with the SiLU(gate)*up epilogue, and down).
//
// Page "oMLX MoE gate/up 融合优化：qwen35_moe_gate_up 实现剖析", 融合原理 and
// 实现剖析 ④ (one gathered product with the [gate; up] matrix, split, SwitchGLU
// activation, down projection); page "Qwen3.5 Block在llama.cpp中的映射与优化
// 原理", section 4.2 (only the routed experts' weights are touched).
//
// Work: an item is (active expert, block of 8 warps x 4 weight rows).  The
// CTAs of a persistent grid take equal contiguous ranges of the item list.
// A CTA stages the activations of up to MT rows of the expert's segment in
// shared memory as fp32 (with per-segment sums, see below) and every warp
// streams its 4 weight rows once with 128-bit non-allocating loads,
// prefetching the next segment, and applies them to all staged tokens.
//
// Dequantization in registers.  A lane takes a 16-byte segment of a row
// (32 four-bit or 16 eight-bit codes).  Per group of 64 elements
//   sum_i x_i (s q_i + b) = s * sum_i x_i q_i + b * sum_i x_i,
// so only sum x_i q_i needs the codes.  A code is moved into the top of a
// float mantissa by one shift and one LOP3: the bit pattern 0x3F800000 |
// (q << p) is the float 1 + q * 2^(p-23), exact, and x * (1 + q 2^(p-23)) is
// exact in fp32 as well.  Starting the accumulator at -sum x (staged with the
// activations) leaves 2^(p-23) * sum x q.  Codes of adjacent elements sit at
// two positions of one shifted word (4-bit: p = 14 and 18) and are combined
// with one packed fp32x2 FMA.  Every row is reduced in the same order (lane
// segments ascending, then an xor butterfly), whatever rows it is computed
// with, so the fused gate_up product equals the separate gate and up products
// bit for bit.
#include <cuda_fp16.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;
constexpr int kRowsPerWarp = 4;

enum GemvMode { kSwiglu = 0, kRaw = 1 };
enum ActKind { kActXbf16 = 0, kActF32 = 1, kActBf16 = 2 };

struct GemvParams {
  const void* act;  // x [T, K] bf16 (gathered by token) or h [rows, K] (by sorted row)
  int act_kind;
  const int32_t* sorted;   // sorted_assign (kActXbf16)
  const int32_t* offsets;  // [E+1]
  int kmax, E, K;
  int n_rows;  // weight rows per expert
  int n_out;   // output columns: n_rows/2 (SWIGLU) or n_rows
  const uint32_t* wq;
  const uint16_t* ws;
  const uint16_t* wb;
  void* out;
  int out_dtype;
  int items_per_expert;
  int units_per_item;
  unsigned int* err;
};

template <int BITS>
struct Seg {
  static constexpr int kElems = 128 / BITS;       // elements per 16-byte segment
  static constexpr int kVec4 = kElems / 4;        // float4 vectors per segment
  static constexpr int kSegsPerGroup = 64 / kElems;
};

// sum_i x_i q_i over one segment, given the segment's staged activations
// (fp32, natural order) and acc0 = (-sum of even-position x, -sum of odd x).
template <int BITS>
__device__ __forceinline__ float seg_dot(const uint4& w, const float* x, float2 acc) {
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
  if constexpr (BITS == 4) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t v = words[i];
      const uint32_t sh[4] = {v << 14, v << 6, v >> 2, v >> 10};
#pragma unroll
      for (int pq = 0; pq < 4; ++pq) {
        float a = __uint_as_float((sh[pq] & 0x0003C000u) | 0x3F800000u);  // 1 + q_even/512
        float b = __uint_as_float((sh[pq] & 0x003C0000u) | 0x3F800000u);  // 1 + q_odd/32
        acc = ffma2(make_float2(a, b), make_float2(x[8 * i + 2 * pq], x[8 * i + 2 * pq + 1]), acc);
      }
    }
    return fmaf(512.0f, acc.x, 32.0f * acc.y);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t v = words[i];
      float a0 = __uint_as_float(((v << 15) & 0x007F8000u) | 0x3F800000u);  // 1 + byte0/256
      float b0 = __uint_as_float(((v << 7) & 0x007F8000u) | 0x3F800000u);   // 1 + byte1/256
      float a1 = __uint_as_float(((v >> 1) & 0x007F8000u) | 0x3F800000u);   // 1 + byte2/256
      float b1 = __uint_as_float(((v >> 9) & 0x007F8000u) | 0x3F800000u);   // 1 + byte3/256
      acc = ffma2(make_float2(a0, b0), make_float2(x[4 * i], x[4 * i + 1]), acc);
      acc = ffma2(make_float2(a1, b1), make_float2(x[4 * i + 2], x[4 * i + 3]), acc);
    }
    return 256.0f * (acc.x + acc.y);
  }
}

template <int BITS, int MODE, int MT>
__global__ void __launch_bounds__(kGemvThreads, 2) gemv_qmm_kernel(GemvParams p) {
  using S = Seg<BITS>;
  extern __shared__ __align__(16) float gsm[];
  const int K = p.K;
  const int nseg = K / S::kElems;
  float* xs = gsm;                                        // [MT][K] swizzled
  float2* xsum = reinterpret_cast<float2*>(gsm + MT * K);  // [MT][nseg]
  __shared__ int act_e[1024];
  __shared__ int n_act_sh;
  // what is staged in xs; every thread keeps the same copy
  int tag_e = -1, tag_r0 = -1, tag_nt = 0;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E;

  // active experts in id order
  if (tid == 0) n_act_sh = 0;
  __syncthreads();
  for (int base = 0; base < E; base += kGemvThreads) {
    const int e = base + tid;
    const bool act = e < E && (p.offsets[e + 1] - p.offsets[e]) > 0;
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, act);
    __shared__ int wtot[kGemvWarps];
    if (lane == 0) wtot[warp] = __popc(bal);
    __syncthreads();
    int before = n_act_sh;
    for (int w = 0; w < warp; ++w) before += wtot[w];
    if (act) act_e[before + __popc(bal & lanemask_lt())] = e;
    __syncthreads();
    if (tid == 0) {
      int s = 0;
      for (int w = 0; w < kGemvWarps; ++w) s += wtot[w];
      n_act_sh += s;
    }
    __syncthreads();
  }
  const int n_act = n_act_sh;
  const int64_t n_items = (int64_t)n_act * p.items_per_expert;
  const int64_t it0 = n_items * blockIdx.x / gridDim.x;
  const int64_t it1 = n_items * (blockIdx.x + 1) / gridDim.x;

  const int ngroups = K / 64;
  const int64_t row_words = (int64_t)K * BITS / 32;
  const int half = p.n_rows / 2;

  for (int64_t it = it0; it < it1; ++it) {
    const int e = act_e[it / p.items_per_expert];
    const int ub = (int)(it % p.items_per_expert);
    const int seg_lo = p.offsets[e];
    const int m = p.offsets[e + 1] - seg_lo;

    // this warp's 4 weight rows and output columns
    int wrow[kRowsPerWarp];
    int ocol[kRowsPerWarp];
    bool ovalid[kRowsPerWarp];
    if (MODE == kSwiglu) {
      const int u0 = ub * p.units_per_item + warp * 2;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int u = u0 + q;
        const int uc = u < p.n_out ? u : p.n_out - 1;
        wrow[q] = uc;            // gate row
        wrow[2 + q] = half + uc; // up row
        ocol[q] = u;
        ovalid[q] = u < p.n_out;
        ocol[2 + q] = u;
        ovalid[2 + q] = false;
      }
    } else {
      const int r0 = ub * p.units_per_item + warp * kRowsPerWarp;
#pragma unroll
      for (int q = 0; q < kRowsPerWarp; ++q) {
        const int r = r0 + q;
        wrow[q] = r < p.n_rows ? r : p.n_rows - 1;
        ocol[q] = r;
        ovalid[q] = r < p.n_rows;
      }
    }
    const uint4* wptr[kRowsPerWarp];
    const uint16_t* sptr[kRowsPerWarp];
    const uint16_t* bptr[kRowsPerWarp];
#pragma unroll
    for (int q = 0; q < kRowsPerWarp; ++q) {
      const int64_t grow = (int64_t)e * p.n_rows + wrow[q];
      wptr[q] = reinterpret_cast<const uint4*>(p.wq + grow * row_words);
      sptr[q] = p.ws + grow * ngroups;
      bptr[q] = p.wb + grow * ngroups;
    }

    for (int tc = 0; tc < m; tc += MT) {
      const int nt = min(MT, m - tc);
      const int r0 = seg_lo + tc;
      // ---- stage activations (skipped when already staged) ----
      bool same = false;
      if (p.act_kind == kActXbf16) {
        // tokens of the staged rows equal those of these rows?
        same = tag_nt == nt && tag_e >= 0;
        if (same) {
          for (int t = 0; t < nt; ++t)
            same = same && (p.sorted[tag_r0 + t] / p.kmax) == (p.sorted[r0 + t] / p.kmax);
        }
      } else {
        same = tag_r0 == r0 && tag_nt == nt;
      }
      if (!same) {
        __syncthreads();  // everyone is done with the previous staging
        for (int idx = tid; idx < nt * nseg; idx += kGemvThreads) {
          const int t = idx / nseg, sg = idx - t * nseg;
          float v[S::kElems];
          if (p.act_kind == kActXbf16) {
            const int tok = p.sorted[r0 + t] / p.kmax;
            const uint4* src = reinterpret_cast<const uint4*>(
                static_cast<const uint16_t*>(p.act) + (int64_t)tok * K + sg * S::kElems);
#pragma unroll
            for (int c = 0; c < S::kElems / 8; ++c) {
              uint4 u = __ldg(src + c);
              float2 a = bf16x2_to_f32x2(u.x), b = bf16x2_to_f32x2(u.y);
              float2 cc = bf16x2_to_f32x2(u.z), d = bf16x2_to_f32x2(u.w);
              v[8 * c + 0] = a.x; v[8 * c + 1] = a.y; v[8 * c + 2] = b.x; v[8 * c + 3] = b.y;
              v[8 * c + 4] = cc.x; v[8 * c + 5] = cc.y; v[8 * c + 6] = d.x; v[8 * c + 7] = d.y;
            }
          } else if (p.act_kind == kActF32) {
            const float4* src = reinterpret_cast<const float4*>(
                static_cast<const float*>(p.act) + (int64_t)(r0 + t) * K + sg * S::kElems);
#pragma unroll
            for (int c = 0; c < S::kVec4; ++c) {
              float4 u = __ldg(src + c);
              v[4 * c] = u.x; v[4 * c + 1] = u.y; v[4 * c + 2] = u.z; v[4 * c + 3] = u.w;
            }
          } else {
            const uint4* src = reinterpret_cast<const uint4*>(
                static_cast<const uint16_t*>(p.act) + (int64_t)(r0 + t) * K + sg * S::kElems);
#pragma unroll
            for (int c = 0; c < S::kElems / 8; ++c) {
              uint4 u = __ldg(src + c);
              float2 a = bf16x2_to_f32x2(u.x), b = bf16x2_to_f32x2(u.y);
              float2 cc = bf16x2_to_f32x2(u.z), d = bf16x2_to_f32x2(u.w);
              v[8 * c + 0] = a.x; v[8 * c + 1] = a.y; v[8 * c + 2] = b.x; v[8 * c + 3] = b.y;
              v[8 * c + 4] = cc.x; v[8 * c + 5] = cc.y; v[8 * c + 6] = d.x; v[8 * c + 7] = d.y;
            }
          }
          float se = 0.0f, so = 0.0f;
#pragma unroll
          for (int i = 0; i < S::kElems; i += 2) { se += v[i]; so += v[i + 1]; }
          float4* dst = reinterpret_cast<float4*>(xs + (int64_t)t * K + sg * S::kElems);
#pragma unroll
          for (int c = 0; c < S::kVec4; ++c)
            dst[(c + sg) % S::kVec4] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
          xsum[t * nseg + sg] = make_float2(-se, -so);
        }
        __syncthreads();
        tag_e = e;
        tag_r0 = r0;
        tag_nt = nt;
      }

      // ---- stream the weights ----
      float tot[kRowsPerWarp][MT];
#pragma unroll
      for (int q = 0; q < kRowsPerWarp; ++q)
#pragma unroll
        for (int t = 0; t < MT; ++t) tot[q][t] = 0.0f;

      uint4 wn[kRowsPerWarp];
      if (lane < nseg) {
#pragma unroll
        for (int q = 0; q < kRowsPerWarp; ++q) wn[q] = ldg_nc_v4(wptr[q] + lane);
      }
      for (int sg = lane; sg < nseg; sg += 32) {
        uint4 wc[kRowsPerWarp];
#pragma unroll
        for (int q = 0; q < kRowsPerWarp; ++q) wc[q] = wn[q];
        if (sg + 32 < nseg) {
#pragma unroll
          for (int q = 0; q < kRowsPerWarp; ++q) wn[q] = ldg_nc_v4(wptr[q] + sg + 32);
        }
        const int g = sg / S::kSegsPerGroup;
        float sc[kRowsPerWarp], bi[kRowsPerWarp];
#pragma unroll
        for (int q = 0; q < kRowsPerWarp; ++q) {
          sc[q] = f16_bits_to_f32(__ldg(sptr[q] + g));
          bi[q] = f16_bits_to_f32(__ldg(bptr[q] + g));
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          if (t < nt) {
            float xv[S::kElems];
            const float4* src = reinterpret_cast<const float4*>(xs + (int64_t)t * K + sg * S::kElems);
#pragma unroll
            for (int c = 0; c < S::kVec4; ++c) {
              float4 u = src[(c + sg) % S::kVec4];
              xv[4 * c] = u.x; xv[4 * c + 1] = u.y; xv[4 * c + 2] = u.z; xv[4 * c + 3] = u.w;
            }
            const float2 ns = xsum[t * nseg + sg];
            const float xsum_seg = -(ns.x + ns.y);
#pragma unroll
            for (int q = 0; q < kRowsPerWarp; ++q) {
              const float sxq = seg_dot<BITS>(wc[q], xv, ns);
              tot[q][t] = fmaf(sc[q], sxq, fmaf(bi[q], xsum_seg, tot[q][t]));
            }
          }
        }
      }
      // ---- reduce across lanes (fixed xor butterfly) and store ----
#pragma unroll
      for (int q = 0; q < kRowsPerWarp; ++q)
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1)
            tot[q][t] = __fadd_rn(tot[q][t], __shfl_xor_sync(0xFFFFFFFFu, tot[q][t], off));
      if (lane == 0) {
        for (int t = 0; t < nt; ++t) {
          const int64_t r = r0 + t;
          if (MODE == kSwiglu) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              if (!ovalid[q]) continue;
              const float hv = swiglu_f32(tot[q][t], tot[2 + q][t]);
              if (p.out_dtype == MOE_DTYPE_BF16)
                static_cast<uint16_t*>(p.out)[r * p.n_out + ocol[q]] = f32_to_bf16_rne(hv);
              else
                static_cast<float*>(p.out)[r * p.n_out + ocol[q]] = hv;
            }
          } else {
#pragma unroll
            for (int q = 0; q < kRowsPerWarp; ++q)
              if (ovalid[q]) static_cast<float*>(p.out)[r * p.n_out + ocol[q]] = tot[q][t];
          }
        }
      }
    }
  }
}

template <int BITS, int MODE, int MT>
moe_status_t launch_gemv(const GemvParams& p, int max_active, cudaStream_t st) {
  using S = Seg<BITS>;
  auto kern = gemv_qmm_kernel<BITS, MODE, MT>;
  const int nseg = p.K / S::kElems;
  const size_t smem = (size_t)MT * p.K * sizeof(float) + (size_t)MT * nseg * sizeof(float2);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
  }
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kGemvThreads, smem) !=
          cudaSuccess ||
      occ < 1)
    return MOE_ERR_CUDA;
  const int64_t items = (int64_t)max_active * p.items_per_expert;
  const int64_t slots = (int64_t)moe_host::sm_count() * occ;
  if (items <= 0) return MOE_OK;
  const int64_t per = (items + slots - 1) / slots;
  const int grid = (int)((items + per - 1) / per);
  kern<<<grid, kGemvThreads, smem, st>>>(p);
  return moe_host::launch_status();
}

template <int MODE>
moe_status_t dispatch_gemv(const GemvParams& p, int bits, int max_active, cudaStream_t st) {
  // MT: tokens staged at a time, bounded by ~100 KB of shared memory
  const int K = p.K;
  if (bits == 4) {
    if (K <= 6144) return launch_gemv<4, MODE, 4>(p, max_active, st);
    if (K <= 12288) return launch_gemv<4, MODE, 2>(p, max_active, st);
    return launch_gemv<4, MODE, 1>(p, max_active, st);
  } else {
    if (K <= 6144) return launch_gemv<8, MODE, 4>(p, max_active, st);
    if (K <= 12288) return launch_gemv<8, MODE, 2>(p, max_active, st);
    return launch_gemv<8, MODE, 1>(p, max_active, st);
  }
}

}  // namespace

// Entry used by the C-ABI wrappers (api.cu).
moe_status_t gemv_qmm(const void* act, int act_kind, const int32_t* sorted,
                      const int32_t* offsets, int T, int kmax, int E, int K, int n_rows,
                      bool swiglu, const uint32_t* wq, const uint16_t* ws, const uint16_t* wb,
                      int bits, void* out, int out_dtype, cudaStream_t st) {
  GemvParams p;
  p.act = act;
  p.act_kind = act_kind;
  p.sorted = sorted;
  p.offsets = offsets;
  p.kmax = kmax;
  p.E = E;
  p.K = K;
  p.n_rows = n_rows;
  p.n_out = swiglu ? n_rows / 2 : n_rows;
  p.wq = wq;
  p.ws = ws;
  p.wb = wb;
  p.out = out;
  p.out_dtype = out_dtype;
  p.units_per_item = swiglu ? kGemvWarps * 2 : kGemvWarps * kRowsPerWarp;
  p.items_per_expert = (p.n_out + p.units_per_item - 1) / p.units_per_item;
  p.err = moe_host::device_error_word();
  const int64_t slots = (int64_t)T * kmax;
  const int max_active = (int)(slots < E ? slots : E);
  if (max_active == 0) return MOE_OK;
  return swiglu ? dispatch_gemv<kSwiglu>(p, bits, max_active, st)
                : dispatch_gemv<kRaw>(p, bits, max_active, st);
}

}  // namespace moe

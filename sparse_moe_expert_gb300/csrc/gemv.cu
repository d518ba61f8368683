// Grouped GEMV on CUDA cores: the decode / small-batch path of the two
// quantized products (gate_up with the SiLU(gate)*up epilogue, and down).
//
// Page "oMLX MoE gate/up 融合优化：qwen35_moe_gate_up 实现剖析", 融合原理 and
// 实现剖析 ④ (one gathered product with the [gate; up] matrix, split, SwitchGLU
// activation, down projection); page "Qwen3.5 Block在llama.cpp中的映射与优化
// 原理", section 4.2 (only the routed experts' weights are touched).
//
// Work.  An item is (active expert, block of 8 warps x 4 weight rows); the
// CTAs of a persistent grid (two per SM) take equal contiguous ranges of the
// item list.  A CTA stages the activations of up to MT rows of the expert's
// segment in shared memory; each warp streams its 4 weight rows once with
// 128-bit loads (one segment ahead) and applies them to every staged token;
// lane partials are combined by a fixed xor butterfly.  SWIGLU warps hold
// gate rows n, n+1 and up rows n, n+1, so the activation is applied in
// registers.
//
// Dequantization in registers.  Per group of 64 elements
//   sum_i x_i (s q_i + b) = s * sum_i x_i q_i + b * sum_i x_i,
// so only sum x_i q_i needs the codes.  One shift and one LOP3 turn two codes
// of a word into the bf16 pair (128 + q_j, 128 + q_{j+4}) (exact: bf16 holds
// 128..255), each half feeding one fp32-accumulating bf16 FMA
// (fma.rn.f32.bf16) against the bf16 activation.  Activations are staged per
// token in that pair order together with their sums X per 32 codes, so
// sum x q = sum x (128 + q) - 128 X.  8-bit codes are read as two 4-bit codes
// (low, high) against activations (x, 16 x), exact in bf16.  Every row is
// reduced in the same order whatever rows it is computed with, so the fused
// gate_up product equals the separate gate and up products bit for bit.
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
struct Width {
  static constexpr int kNibPerElem = BITS / 4;            // 1 or 2
  static constexpr int kSegPerGroup = 64 * kNibPerElem / 32;  // 2 or 4
};

// acc += a_half * b_half for the low (hi = false) or high halves of two
// registers holding bf16 pairs; fp32 accumulation.
__device__ __forceinline__ void bf16_fma(float& acc, uint32_t a_pair, uint32_t b_pair, bool hi) {
  unsigned short a_lo, a_hi, b_lo, b_hi;
  asm("mov.b32 {%0,%1}, %2;" : "=h"(a_lo), "=h"(a_hi) : "r"(a_pair));
  asm("mov.b32 {%0,%1}, %2;" : "=h"(b_lo), "=h"(b_hi) : "r"(b_pair));
  if (hi)
    asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(acc) : "h"(a_hi), "h"(b_hi));
  else
    asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(acc) : "h"(a_lo), "h"(b_lo));
}

// Stage the activations of `nt` rows starting at sorted row r0 into xs (bf16
// pairs in code-pair order, 16 words per 32-nibble segment, vectors rotated
// by segment to avoid bank conflicts) and their per-segment sums.
template <int BITS>
__device__ void stage_activations(const GemvParams& p, int r0, int nt, uint32_t* xs, float2* xsum,
                                  int NK, int nseg_row) {
  const int K = p.K;
  for (int idx = threadIdx.x; idx < nt * nseg_row; idx += kGemvThreads) {
    const int t = idx / nseg_row, sg = idx - t * nseg_row;
    const int64_t r = r0 + t;
    uint32_t v[32];  // bf16 bits of the 32 nibble-order activation values
    if (BITS == 4) {
      const int k0 = sg * 32;
      if (p.act_kind == kActF32) {
        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.act) + r * K + k0);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 u = __ldg(src + c);
          v[4 * c] = f32_to_bf16_rne(u.x);
          v[4 * c + 1] = f32_to_bf16_rne(u.y);
          v[4 * c + 2] = f32_to_bf16_rne(u.z);
          v[4 * c + 3] = f32_to_bf16_rne(u.w);
        }
      } else {
        const int64_t row = p.act_kind == kActXbf16 ? (int64_t)(__ldg(p.sorted + r) / p.kmax) : r;
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.act) + row * K + k0);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 u = __ldg(src + c);
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            v[8 * c + 2 * q] = w4[q] & 0xFFFFu;
            v[8 * c + 2 * q + 1] = w4[q] >> 16;
          }
        }
      }
    } else {
      // 8-bit: 16 elements; nibble 2i <- x_i, nibble 2i+1 <- 16 x_i
      const int k0 = sg * 16;
      float xf[16];
      if (p.act_kind == kActF32) {
        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.act) + r * K + k0);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float4 u = __ldg(src + c);
          xf[4 * c] = bf16_bits_to_f32(f32_to_bf16_rne(u.x));
          xf[4 * c + 1] = bf16_bits_to_f32(f32_to_bf16_rne(u.y));
          xf[4 * c + 2] = bf16_bits_to_f32(f32_to_bf16_rne(u.z));
          xf[4 * c + 3] = bf16_bits_to_f32(f32_to_bf16_rne(u.w));
        }
      } else {
        const int64_t row = p.act_kind == kActXbf16 ? (int64_t)(__ldg(p.sorted + r) / p.kmax) : r;
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.act) + row * K + k0);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint4 u = __ldg(src + c);
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = bf16x2_to_f32x2(w4[q]);
            xf[8 * c + 2 * q] = f.x;
            xf[8 * c + 2 * q + 1] = f.y;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        v[2 * i] = __float_as_uint(xf[i]) >> 16;
        v[2 * i + 1] = __float_as_uint(16.0f * xf[i]) >> 16;
      }
    }
    float sum = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) sum += bf16_bits_to_f32(v[i]);
    float esum = sum;
    if (BITS == 8) {
      esum = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; i += 2) esum += bf16_bits_to_f32(v[i]);
    }
    uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)t * (NK / 2) + (size_t)sg * 16);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 o;
      o.x = v[8 * c + 0] | (v[8 * c + 4] << 16);
      o.y = v[8 * c + 1] | (v[8 * c + 5] << 16);
      o.z = v[8 * c + 2] | (v[8 * c + 6] << 16);
      o.w = v[8 * c + 3] | (v[8 * c + 7] << 16);
      dst[(c + (sg >> 1)) & 3] = o;
    }
    xsum[t * nseg_row + sg] = make_float2(sum, esum);
  }
}

template <int BITS, int MODE, int MT>
__global__ void __launch_bounds__(kGemvThreads, MT == 1 ? 3 : 2) gemv_qmm_kernel(GemvParams p) {
  using W = Width<BITS>;
  extern __shared__ __align__(16) unsigned char gsm[];
  const int K = p.K;
  const int NK = K * W::kNibPerElem;  // nibbles per row
  const int nseg = NK / 32;           // 16-byte code segments per row
  const int ngroups = K / 64;
  uint32_t* xs = reinterpret_cast<uint32_t*>(gsm);                          // [MT][NK/2]
  float2* xsum = reinterpret_cast<float2*>(gsm + (size_t)MT * (NK / 2) * 4);  // [MT][nseg]
  __shared__ int act_e[1024];
  __shared__ int n_act_sh;
  __shared__ int wtot[kGemvWarps];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E;

  // active experts in id order
  if (tid == 0) n_act_sh = 0;
  __syncthreads();
  for (int base = 0; base < E; base += kGemvThreads) {
    const int e = base + tid;
    const bool act = e < E && (__ldg(p.offsets + e + 1) - __ldg(p.offsets + e)) > 0;
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, act);
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
  const int64_t row_u4 = (int64_t)NK / 32;  // uint4 per row
  const int half = p.n_rows / 2;

  // A pass applies one item's rows to one chunk of at most MT of its
  // tokens.  Passes follow each other without a gap: the first segment of
  // the next pass is loaded during the last segment of the current one.
  struct Pass {
    int it, tc, seg_lo, m;
    int col0;                // first output column of this warp
    int grow[kRowsPerWarp];  // weight rows (global index e*n_rows + row)
  };
  auto make_pass = [&](int it, int tc, Pass& ps) {
    ps.it = it;
    ps.tc = tc;
    const int e = act_e[it / p.items_per_expert];
    const int ub = it % p.items_per_expert;
    ps.seg_lo = __ldg(p.offsets + e);
    ps.m = __ldg(p.offsets + e + 1) - ps.seg_lo;
    const int base = e * p.n_rows;
    if (MODE == kSwiglu) {
      ps.col0 = ub * p.units_per_item + warp * 2;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int u = ps.col0 + q;
        const int uc = u < p.n_out ? u : p.n_out - 1;
        ps.grow[q] = base + uc;             // gate row
        ps.grow[2 + q] = base + half + uc;  // up row
      }
    } else {
      ps.col0 = ub * p.units_per_item + warp * kRowsPerWarp;
#pragma unroll
      for (int q = 0; q < kRowsPerWarp; ++q) {
        const int r = ps.col0 + q;
        ps.grow[q] = base + (r < p.n_rows ? r : p.n_rows - 1);
      }
    }
  };
  // codes, scale and bias of segment sg of the pass's rows
  uint4 wn[kRowsPerWarp];
  uint16_t sn[kRowsPerWarp], bn[kRowsPerWarp];
  auto load_segment = [&](const Pass& ps, int sg) {
    const int g = sg / W::kSegPerGroup;
#pragma unroll
    for (int q = 0; q < kRowsPerWarp; ++q) {
      const int64_t grow = ps.grow[q];
      wn[q] = ldg_nc_v4(reinterpret_cast<const uint4*>(p.wq) + grow * row_u4 + sg);
      sn[q] = __ldg(p.ws + grow * ngroups + g);
      bn[q] = __ldg(p.wb + grow * ngroups + g);
    }
  };

  // what is staged in xs (every thread keeps the same copy)
  int tag_r0 = -1, tag_nt = -1;

  if (it0 >= it1) return;
  Pass cur, nxt;
  make_pass((int)it0, 0, cur);
  if (lane < nseg) load_segment(cur, lane);
  for (;;) {
    // the pass after this one
    bool has_next = true;
    if (cur.tc + MT < cur.m) {
      nxt = cur;
      nxt.tc = cur.tc + MT;
    } else if (cur.it + 1 < it1) {
      make_pass(cur.it + 1, 0, nxt);
    } else {
      has_next = false;
    }
    const int nt = min(MT, cur.m - cur.tc);
    const int r0 = cur.seg_lo + cur.tc;
    // ---- stage the activations when they changed ----
    bool same = tag_nt == nt;
    if (same) {
      if (p.act_kind == kActXbf16) {
        for (int t = 0; t < nt; ++t)
          same = same && (__ldg(p.sorted + tag_r0 + t) / p.kmax) == (__ldg(p.sorted + r0 + t) / p.kmax);
      } else {
        same = tag_r0 == r0;
      }
    }
    if (!same) {
      __syncthreads();  // everyone is done with the previous staging
      stage_activations<BITS>(p, r0, nt, xs, xsum, NK, nseg);
      __syncthreads();
      tag_r0 = r0;
      tag_nt = nt;
    }

    // ---- stream the weights ----
    float tot[kRowsPerWarp][MT];
#pragma unroll
    for (int q = 0; q < kRowsPerWarp; ++q)
#pragma unroll
      for (int t = 0; t < MT; ++t) tot[q][t] = 0.0f;

    for (int sg = lane; sg < nseg; sg += 32) {
      uint4 wc[kRowsPerWarp];
      float sc[kRowsPerWarp], bi[kRowsPerWarp];
#pragma unroll
      for (int q = 0; q < kRowsPerWarp; ++q) {
        wc[q] = wn[q];
        sc[q] = f16_bits_to_f32(sn[q]);
        bi[q] = f16_bits_to_f32(bn[q]);
      }
      if (sg + 32 < nseg)
        load_segment(cur, sg + 32);
      else if (has_next)
        load_segment(nxt, lane);
      const uint4* xsrc0 = reinterpret_cast<const uint4*>(xs + (size_t)sg * 16);
      const int rot = sg >> 1;
#pragma unroll
      for (int q = 0; q < kRowsPerWarp; ++q) {
        // code pairs (128 + q_j, 128 + q_{j+4}) of this row's segment
        uint32_t ep[16];
        const uint32_t w4[4] = {wc[q].x, wc[q].y, wc[q].z, wc[q].w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) ep[4 * i + j] = ((w4[i] >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          if (t < nt) {
            const uint4* xsrc = xsrc0 + (size_t)t * (NK / 8);
            uint32_t xp[16];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint4 u = xsrc[(c + rot) & 3];
              xp[4 * c] = u.x;
              xp[4 * c + 1] = u.y;
              xp[4 * c + 2] = u.z;
              xp[4 * c + 3] = u.w;
            }
            const float2 X = xsum[t * nseg + sg];
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              bf16_fma(a0, ep[i], xp[i], false);
              bf16_fma(a1, ep[i], xp[i], true);
            }
            const float sxq = fmaf(-128.0f, X.x, a0 + a1);
            tot[q][t] = fmaf(sc[q], sxq, fmaf(bi[q], X.y, tot[q][t]));
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
            const int col = cur.col0 + q;
            if (col >= p.n_out) continue;
            const float hv = swiglu_f32(tot[q][t], tot[2 + q][t]);
            if (p.out_dtype == MOE_DTYPE_BF16)
              static_cast<uint16_t*>(p.out)[r * p.n_out + col] = f32_to_bf16_rne(hv);
            else
              static_cast<float*>(p.out)[r * p.n_out + col] = hv;
          }
        } else {
#pragma unroll
          for (int q = 0; q < kRowsPerWarp; ++q) {
            const int col = cur.col0 + q;
            if (col >= p.n_rows) continue;
            if (p.out_dtype == MOE_DTYPE_BF16)
              static_cast<uint16_t*>(p.out)[r * p.n_out + col] = f32_to_bf16_rne(tot[q][t]);
            else
              static_cast<float*>(p.out)[r * p.n_out + col] = tot[q][t];
          }
        }
      }
    }
    if (!has_next) break;
    cur = nxt;
  }
}

template <int BITS, int MODE, int MT>
moe_status_t launch_gemv(const GemvParams& p, int max_active, cudaStream_t st) {
  auto kern = gemv_qmm_kernel<BITS, MODE, MT>;
  const int NK = p.K * (BITS / 4);
  const size_t smem = (size_t)MT * (NK / 2) * 4 + (size_t)MT * (NK / 32) * sizeof(float2);
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
  if (items <= 0) return MOE_OK;
  const int64_t slots = (int64_t)moe_host::sm_count() * occ;
  const int64_t per = (items + slots - 1) / slots;
  const int grid = (int)((items + per - 1) / per);
  kern<<<grid, kGemvThreads, smem, st>>>(p);
  return moe_host::launch_status();
}

template <int MODE>
moe_status_t dispatch_gemv(const GemvParams& p, int bits, int max_tokens, int max_active,
                           cudaStream_t st) {
  // MT: tokens applied per pass over the weights, at most the tokens an expert
  // can have (max_tokens) and bounded by shared memory
  const int NK = p.K * (bits / 4);
  int mt = NK <= 6144 ? 4 : (NK <= 12288 ? 2 : 1);
  if (max_tokens < mt) mt = max_tokens <= 1 ? 1 : 2;
  if (bits == 4) {
    if (mt == 4) return launch_gemv<4, MODE, 4>(p, max_active, st);
    if (mt == 2) return launch_gemv<4, MODE, 2>(p, max_active, st);
    return launch_gemv<4, MODE, 1>(p, max_active, st);
  } else {
    if (mt == 4) return launch_gemv<8, MODE, 4>(p, max_active, st);
    if (mt == 2) return launch_gemv<8, MODE, 2>(p, max_active, st);
    return launch_gemv<8, MODE, 1>(p, max_active, st);
  }
}

}  // namespace

bool gemv_stream_supported(int bits, int K, int E);
moe_status_t gemv_stream_qmm(const void* act, int act_kind, const int32_t* sorted,
                             const int32_t* offsets, int T, int kmax, int E, int K, int n_rows,
                             bool swiglu, const uint32_t* wq, const uint16_t* ws,
                             const uint16_t* wb, int bits, void* out, int out_dtype, bool early,
                             KGate gate, cudaStream_t st);
moe_status_t gemv_bits_qmm(const void* act, int act_kind, const int32_t* sorted,
                           const int32_t* offsets, int T, int kmax, int E, int K, int n_rows,
                           bool swiglu, const uint32_t* wq, const uint16_t* ws, const uint16_t* wb,
                           int bits, void* out, int out_dtype, cudaStream_t st);

// Entry used by the C-ABI wrappers (api.cu).  5- and 6-bit codes take their
// own kernel (gemv_bits.cu); 4- and 8-bit rows that are whole 128-byte
// blocks of codes (4-bit K a multiple of 256, 8-bit of 128) the streamed
// kernel (gemv_stream.cu); other rows this file's kernel.  Only the streamed
// kernel takes a k gate.
moe_status_t gemv_qmm(const void* act, int act_kind, const int32_t* sorted,
                      const int32_t* offsets, int T, int kmax, int E, int K, int n_rows,
                      bool swiglu, const uint32_t* wq, const uint16_t* ws, const uint16_t* wb,
                      int bits, void* out, int out_dtype, bool early, KGate gate,
                      cudaStream_t st) {
  if (bits == 5 || bits == 6) {
    if (gate.k != nullptr) return MOE_ERR_UNSUPPORTED;
    return gemv_bits_qmm(act, act_kind, sorted, offsets, T, kmax, E, K, n_rows, swiglu, wq, ws, wb,
                         bits, out, out_dtype, st);
  }
  if (gemv_stream_supported(bits, K, E))
    return gemv_stream_qmm(act, act_kind, sorted, offsets, T, kmax, E, K, n_rows, swiglu, wq, ws,
                           wb, bits, out, out_dtype, early, gate, st);
  if (gate.k != nullptr) return MOE_ERR_UNSUPPORTED;
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
  // an expert's segment holds at most one row per token (its k ids are distinct)
  const int max_tokens = T;
  return swiglu ? dispatch_gemv<kSwiglu>(p, bits, max_tokens, max_active, st)
                : dispatch_gemv<kRaw>(p, bits, max_tokens, max_active, st);
}

}  // namespace moe

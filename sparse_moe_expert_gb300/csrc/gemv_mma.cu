// Grouped GEMV for 4-bit codes with warp-level MMAs: the decode / small-batch
// path of the two quantized products.
//
// Page "oMLX MoE gate/up 融合优化：qwen35_moe_gate_up 实现剖析", 融合原理 and
// 实现剖析 ④ (one gathered product with the [gate; up] matrix, split, SwitchGLU
// activation, down projection); page "Qwen3.5 Block在llama.cpp中的映射与优化
// 原理", section 4.2 (only the routed experts' weights are read).
//
// Per group of 64 elements of a weight row (scale s, bias b):
//   sum_i x_i (s q_i + b) = s * (sum_i (128 + q_i) x_i - 128 X) + b * X,
// X = sum_i x_i.  One shift and one LOP3 turn two codes of a word into the
// bf16 pair (128 + q_j, 128 + q_{j+4}) (exact); those pairs are the A
// fragments of mma.sync.m16n8k16 (bf16 x bf16 -> fp32) straight from
// registers, so a warp forms P = sum_i (128 + q_i) x_i for 16 rows and up to
// 8 tokens with one MMA per 256 codes.  CUDA cores then apply s and b per
// group and sum the groups in order.
//
// Fragment mapping.  Lane (g, t) = (lane / 4, lane % 4) holds rows g and g+8
// of the 16-row tile.  In each group it loads words 2t and 2t+1 (8 bytes) of
// both rows; word 2t+w feeds the two MMAs of window w: MMA m takes nibble
// pairs (2m, 2m+4) and (2m+1, 2m+5) of it.  The token values are staged in
// that same order (B fragments, one 8-byte read per lane per MMA).
//
// Work.  A CTA item is (active expert, chunk of up to MT tokens, 16-row
// tile); SWIGLU tiles are 8 gate rows and the 8 up rows of the same
// features, so the activation is applied in registers.  The CTA's 8 warps
// split the item's groups (in quads of 4) and their partial sums are added
// in warp order through shared memory.  Codes and scales are prefetched
// several groups ahead, across item boundaries.  Every row is reduced in the
// same order whatever rows it shares a tile with, so the fused gate_up
// product equals the separate gate and up products bit for bit.
#include <cuda_fp16.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kMvThreads = 256;
constexpr int kMvWarps = kMvThreads / 32;

enum MvMode { kMvSwiglu = 0, kMvRaw = 1 };

struct MvParams {
  const uint16_t* act;     // x [T, K] bf16 (kind 0, through sorted) or rows [A, K] (kind 2)
  int act_kind;
  const int32_t* sorted;
  const int32_t* offsets;  // [E+1]
  const uint32_t* wq;      // codes [E, n_rows, K/8]
  const uint16_t* ws;      // [E, n_rows, K/64]
  const uint16_t* wb;
  void* out;
  int out_dtype;
  int kmax, E, K, n_rows, n_out;
  int tiles_per_chunk;     // 16-row tiles per (expert, token chunk)
  unsigned int* err;
};

__device__ __forceinline__ uint2 ldg_nc_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Weight row (within the expert) of tile row r of 16-row tile mt.
template <int MODE>
__device__ __forceinline__ int mv_weight_row(const MvParams& p, int mt, int r) {
  if (MODE == kMvSwiglu) {
    const int f = mt * 8 + (r & 7);
    return r < 8 ? f : (p.n_rows >> 1) + f;
  }
  return mt * 16 + r;
}

template <int MODE, int MT>
__global__ void __launch_bounds__(kMvThreads, 1) gemv_mma_kernel(MvParams p) {
  extern __shared__ __align__(16) unsigned char mv_smem[];
  const int ngroups = p.K / 64;
  const int nquads = ngroups / 4;
  // B fragments: [group][window 2][mma 2][token MT][t 4] as uint2 (two bf16 pairs)
  uint2* xs = reinterpret_cast<uint2*>(mv_smem);
  float* xsum = reinterpret_cast<float*>(xs + (size_t)ngroups * 16 * MT);  // [group][MT]
  float* part = xsum + (size_t)ngroups * MT;  // [warp][16 rows][8 tokens] partial sums
  __shared__ int act_e[1024];
  __shared__ int n_act_sh;
  __shared__ int wtot[kMvWarps];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  // active experts in id order and their token chunks
  if (tid == 0) n_act_sh = 0;
  __syncthreads();
  for (int base = 0; base < p.E; base += kMvThreads) {
    const int e = base + tid;
    const bool act = e < p.E && (__ldg(p.offsets + e + 1) - __ldg(p.offsets + e)) > 0;
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, act);
    if (lane == 0) wtot[warp] = __popc(bal);
    __syncthreads();
    int before = n_act_sh;
    for (int w = 0; w < warp; ++w) before += wtot[w];
    if (act) act_e[before + __popc(bal & lanemask_lt())] = e;
    __syncthreads();
    if (tid == 0) {
      int s = 0;
      for (int w = 0; w < kMvWarps; ++w) s += wtot[w];
      n_act_sh += s;
    }
    __syncthreads();
  }
  const int n_act = n_act_sh;
  // items: for each active expert, its chunks of MT tokens x tiles; counted
  // by one pass (every thread computes the same list position)
  // chunk counts are per expert, so items are enumerated expert by expert
  int64_t n_items = 0;
  for (int a = 0; a < n_act; ++a) {
    const int e = act_e[a];
    const int m = __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
    n_items += (int64_t)((m + MT - 1) / MT) * p.tiles_per_chunk;
  }
  const int64_t it0 = n_items * blockIdx.x / gridDim.x;
  const int64_t it1 = n_items * (blockIdx.x + 1) / gridDim.x;
  if (it0 >= it1) return;

  // this warp's quads of every item: [q0, q1)
  const int q0 = nquads * warp / kMvWarps, q1 = nquads * (warp + 1) / kMvWarps;
  const int64_t row_words = p.K / 8;

  // item -> (expert, chunk start, tile)
  struct Item {
    int e, seg_lo, m, c0, nt, mt;
  };
  auto item_at = [&](int64_t it) {
    Item r;
    int a = 0;
    int64_t acc = 0;
    for (;; ++a) {
      const int e = act_e[a];
      const int m = __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
      const int64_t n = (int64_t)((m + MT - 1) / MT) * p.tiles_per_chunk;
      if (it < acc + n || a == n_act - 1) {
        const int local = (int)(it - acc);
        r.e = e;
        r.seg_lo = __ldg(p.offsets + e);
        r.m = m;
        const int ch = local / p.tiles_per_chunk;
        r.mt = local - ch * p.tiles_per_chunk;
        r.c0 = ch * MT;
        r.nt = min(MT, m - r.c0);
        return r;
      }
      acc += n;
    }
  };

  // codes, scales and biases of (item, quad) for rows g and g+8 of the
  // tile; a ring of two quads (8 groups) in flight
  struct Quad {
    uint2 c0[4], c1[4];   // words 2t, 2t+1 of each group, rows g and g+8
    uint2 s0, s1, b0, b1; // 4 groups of scale / bias, rows g and g+8
  };
  int64_t la_it = it0;
  int la_q = q0;
  Item la_item = item_at(it0);
  int64_t la_r0 = 0, la_r1 = 0;  // global weight rows
  auto la_rows = [&]() {
    int w0 = mv_weight_row<MODE>(p, la_item.mt, g), w1 = mv_weight_row<MODE>(p, la_item.mt, g + 8);
    if (w0 >= p.n_rows) w0 = p.n_rows - 1;  // rows past the matrix: any valid row
    if (w1 >= p.n_rows) w1 = p.n_rows - 1;
    la_r0 = (int64_t)la_item.e * p.n_rows + w0;
    la_r1 = (int64_t)la_item.e * p.n_rows + w1;
  };
  la_rows();
  auto la_fetch = [&](Quad& d) {
    if (la_it >= it1 || q0 >= q1) return;
    const int g0q = la_q * 4;
    const uint32_t* c0p = p.wq + la_r0 * row_words + 2 * t + 8 * g0q;
    const uint32_t* c1p = p.wq + la_r1 * row_words + 2 * t + 8 * g0q;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      d.c0[i] = ldg_nc_v2(c0p + 8 * i);
      d.c1[i] = ldg_nc_v2(c1p + 8 * i);
    }
    d.s0 = __ldg(reinterpret_cast<const uint2*>(p.ws + la_r0 * ngroups + g0q));
    d.s1 = __ldg(reinterpret_cast<const uint2*>(p.ws + la_r1 * ngroups + g0q));
    d.b0 = __ldg(reinterpret_cast<const uint2*>(p.wb + la_r0 * ngroups + g0q));
    d.b1 = __ldg(reinterpret_cast<const uint2*>(p.wb + la_r1 * ngroups + g0q));
    if (++la_q == q1) {
      la_q = q0;
      if (++la_it < it1) {
        la_item = item_at(la_it);
        la_rows();
      }
    }
  };
  Quad ring0, ring1;
  la_fetch(ring0);
  la_fetch(ring1);
  int64_t qc = 0;  // quads consumed

  int tag_e = -1, tag_c0 = -1;  // staged activations
  for (int64_t it = it0; it < it1; ++it) {
    const Item ci = item_at(it);
    // ---- stage the activations of (expert, chunk) when they changed ----
    if (ci.e != tag_e || ci.c0 != tag_c0) {
      __syncthreads();  // everyone is done with the previous staging
      // B fragments: lane t' of group grp, window w, mma m holds token n's
      // elements (e0, e0+4) and (e0+1, e0+5), e0 = 8 (2 t' + w) + 2 m
      for (int idx = tid; idx < ngroups * 16 * MT; idx += kMvThreads) {
        const int tt = idx & 3, n = (idx >> 2) % MT, wm = (idx / (4 * MT)) & 3, grp = idx / (16 * MT);
        const int w = wm >> 1, mm = wm & 1;
        const int n_src = n < ci.nt ? n : 0;
        const int64_t r = ci.seg_lo + ci.c0 + n_src;
        const int64_t row = p.act_kind == 0 ? (int64_t)(__ldg(p.sorted + r) / p.kmax) : r;
        const uint16_t* xr = p.act + row * p.K + grp * 64 + 8 * (2 * tt + w) + 2 * mm;
        const uint32_t b0 = (uint32_t)__ldg(xr) | ((uint32_t)__ldg(xr + 4) << 16);
        const uint32_t b1 = (uint32_t)__ldg(xr + 1) | ((uint32_t)__ldg(xr + 5) << 16);
        xs[idx] = make_uint2(b0, b1);
      }
      // per-group sums X of each token, a fixed lane tree per (group, token)
      for (int idx = warp; idx < ngroups * MT; idx += kMvWarps) {
        const int grp = idx / MT, n = idx - grp * MT;
        const int n_src = n < ci.nt ? n : 0;
        const int64_t r = ci.seg_lo + ci.c0 + n_src;
        const int64_t row = p.act_kind == 0 ? (int64_t)(__ldg(p.sorted + r) / p.kmax) : r;
        const uint16_t* xr = p.act + row * p.K + grp * 64;
        float v = __fadd_rn(bf16_bits_to_f32(__ldg(xr + 2 * lane)),
                            bf16_bits_to_f32(__ldg(xr + 2 * lane + 1)));
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
        if (lane == 0) xsum[idx] = v;
      }
      __syncthreads();
      tag_e = ci.e;
      tag_c0 = ci.c0;
    }

    // ---- this warp's quads of the item ----
    // acc[0..1]: row g, tokens 2t, 2t+1; acc[2..3]: row g+8
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const int na = 2 * t < MT ? 2 * t : MT - 1, nb = 2 * t + 1 < MT ? 2 * t + 1 : MT - 1;
    const int bn = g < MT ? g : MT - 1;  // B column (token) of this lane
    auto process = [&](const Quad& cur, int quad) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int grp = quad * 4 + i;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        const uint2* xg = xs + (size_t)grp * 16 * MT;
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          const uint32_t va = w ? cur.c0[i].y : cur.c0[i].x, vc = w ? cur.c1[i].y : cur.c1[i].x;
#pragma unroll
          for (int mm = 0; mm < 2; ++mm) {
            uint32_t af[4];
            af[0] = ((va >> (8 * mm)) & 0x000F000Fu) | 0x43004300u;
            af[1] = ((vc >> (8 * mm)) & 0x000F000Fu) | 0x43004300u;
            af[2] = ((va >> (8 * mm + 4)) & 0x000F000Fu) | 0x43004300u;
            af[3] = ((vc >> (8 * mm + 4)) & 0x000F000Fu) | 0x43004300u;
            const uint2 bv = xg[((w * 2 + mm) * MT + bn) * 4 + t];
            mma_bf16_16816(d, af, bv.x, bv.y);
          }
        }
        const uint32_t sw0 = i < 2 ? cur.s0.x : cur.s0.y, sw1 = i < 2 ? cur.s1.x : cur.s1.y;
        const uint32_t bw0 = i < 2 ? cur.b0.x : cur.b0.y, bw1 = i < 2 ? cur.b1.x : cur.b1.y;
        const int sh = (i & 1) * 16;
        const float s0 = f16_bits_to_f32((uint16_t)(sw0 >> sh)), s1 = f16_bits_to_f32((uint16_t)(sw1 >> sh));
        const float bb0 = f16_bits_to_f32((uint16_t)(bw0 >> sh)), bb1 = f16_bits_to_f32((uint16_t)(bw1 >> sh));
        const float Xa = xsum[grp * MT + na], Xb = xsum[grp * MT + nb];
        acc[0] = fmaf(s0, fmaf(-128.0f, Xa, d[0]), fmaf(bb0, Xa, acc[0]));
        acc[1] = fmaf(s0, fmaf(-128.0f, Xb, d[1]), fmaf(bb0, Xb, acc[1]));
        acc[2] = fmaf(s1, fmaf(-128.0f, Xa, d[2]), fmaf(bb1, Xa, acc[2]));
        acc[3] = fmaf(s1, fmaf(-128.0f, Xb, d[3]), fmaf(bb1, Xb, acc[3]));
      }
    };
    // the older ring entry is consumed in place, then refilled
    for (int quad = q0; quad < q1; ++quad, ++qc) {
      if (qc & 1) {
        process(ring1, quad);
        la_fetch(ring1);
      } else {
        process(ring0, quad);
        la_fetch(ring0);
      }
    }
    // ---- add the warps' partials in warp order and store ----
    float* pw = part + (size_t)warp * 128;
    pw[g * 8 + 2 * t] = acc[0];
    pw[g * 8 + 2 * t + 1] = acc[1];
    pw[(g + 8) * 8 + 2 * t] = acc[2];
    pw[(g + 8) * 8 + 2 * t + 1] = acc[3];
    __syncthreads();
    if (tid < 128) {
      const int row = tid >> 3, n = tid & 7;  // tile row, token
      float v = part[row * 8 + n];
      for (int w = 1; w < kMvWarps; ++w) v = __fadd_rn(v, part[(size_t)w * 128 + row * 8 + n]);
      part[(size_t)kMvWarps * 128 + row * 8 + n] = v;
    }
    __syncthreads();
    if (tid < 64) {
      const int row = tid >> 3, n = tid & 7;  // row (< 8 for SWIGLU: the feature)
      const float* tot = part + (size_t)kMvWarps * 128;
      if (n < ci.nt) {
        const int64_t orow = (int64_t)ci.seg_lo + ci.c0 + n;
        if (MODE == kMvSwiglu) {
          const int f = ci.mt * 8 + row;
          if (f < p.n_out) {
            const float hv = swiglu_f32(tot[row * 8 + n], tot[(row + 8) * 8 + n]);
            if (p.out_dtype == MOE_DTYPE_BF16)
              static_cast<uint16_t*>(p.out)[orow * p.n_out + f] = f32_to_bf16_rne(hv);
            else
              static_cast<float*>(p.out)[orow * p.n_out + f] = hv;
          }
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int col = ci.mt * 16 + row + 8 * h;
            if (col < p.n_rows) static_cast<float*>(p.out)[orow * p.n_out + col] = tot[(row + 8 * h) * 8 + n];
          }
        }
      }
    }
    // the next item's partials overwrite part[] only after everyone read it
    __syncthreads();
  }
}

template <int MODE, int MT>
moe_status_t launch_gemv_mma(const MvParams& p, int64_t max_items, cudaStream_t st) {
  auto kern = gemv_mma_kernel<MODE, MT>;
  const int ngroups = p.K / 64;
  const size_t smem = (size_t)ngroups * 16 * MT * sizeof(uint2) + (size_t)ngroups * MT * 4 +
                      (size_t)(kMvWarps + 1) * 128 * 4;
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
  }
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kMvThreads, smem) != cudaSuccess ||
      occ < 1)
    return MOE_ERR_CUDA;
  if (max_items <= 0) return MOE_OK;
  const int64_t slots = (int64_t)moe_host::sm_count() * occ;
  const int grid = (int)(max_items < slots ? max_items : slots);
  kern<<<grid, kMvThreads, smem, st>>>(p);
  return moe_host::launch_status();
}

}  // namespace

// 4-bit codes, K a multiple of 256, activations bf16 (kind 0 or 2), and
// more than one token per launch (one token streams faster through the
// CUDA-core kernel, which keeps more loads in flight per SM).
bool gemv_mma_supported(int act_kind, int K, int bits, int T) {
  return bits == 4 && K % 256 == 0 && (act_kind == 0 || act_kind == 2) && T > 1;
}

moe_status_t gemv_mma_qmm(const void* act, int act_kind, const int32_t* sorted,
                          const int32_t* offsets, int T, int kmax, int E, int K, int n_rows,
                          bool swiglu, const uint32_t* wq, const uint16_t* ws, const uint16_t* wb,
                          void* out, int out_dtype, cudaStream_t st) {
  MvParams p;
  p.act = static_cast<const uint16_t*>(act);
  p.act_kind = act_kind;
  p.sorted = sorted;
  p.offsets = offsets;
  p.wq = wq;
  p.ws = ws;
  p.wb = wb;
  p.out = out;
  p.out_dtype = out_dtype;
  p.kmax = kmax;
  p.E = E;
  p.K = K;
  p.n_rows = n_rows;
  p.n_out = swiglu ? n_rows / 2 : n_rows;
  p.tiles_per_chunk = swiglu ? (p.n_out + 7) / 8 : (n_rows + 15) / 16;
  p.err = moe_host::device_error_word();
  const int64_t A = (int64_t)T * kmax;
  if (A == 0) return MOE_OK;
  const int64_t max_active = A < E ? A : E;
  // an expert's segment holds at most one row per token; tokens per chunk by
  // the largest possible segment
  const int mt_need = T < 8 ? T : 8;
  const int MT = mt_need <= 1 ? 1 : mt_need <= 2 ? 2 : mt_need <= 4 ? 4 : 8;
  // items: chunks of every possible segment x tiles (an upper bound)
  const int64_t max_chunks = max_active + (A + MT - 1) / MT;
  const int64_t max_items = max_chunks * p.tiles_per_chunk;
  switch (MT) {
    case 1:
      return swiglu ? launch_gemv_mma<kMvSwiglu, 1>(p, max_items, st)
                    : launch_gemv_mma<kMvRaw, 1>(p, max_items, st);
    case 2:
      return swiglu ? launch_gemv_mma<kMvSwiglu, 2>(p, max_items, st)
                    : launch_gemv_mma<kMvRaw, 2>(p, max_items, st);
    case 4:
      return swiglu ? launch_gemv_mma<kMvSwiglu, 4>(p, max_items, st)
                    : launch_gemv_mma<kMvRaw, 4>(p, max_items, st);
    default:
      return swiglu ? launch_gemv_mma<kMvSwiglu, 8>(p, max_items, st)
                    : launch_gemv_mma<kMvRaw, 8>(p, max_items, st);
  }
}

}  // namespace moe

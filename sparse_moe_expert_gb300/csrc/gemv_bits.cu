// Grouped GEMV for 5- and 6-bit affine codes: the two quantized products
// when the codes are not 4 or 8 bits wide.
//
// Page "oMLX MoE gate/up 融合优化：qwen35_moe_gate_up 实现剖析", 如何验证正确性
// (its test list covers the 5-, 6- and 8-bit families besides 4-bit) and
// 融合原理 (the gathered product with the [gate; up] matrix, split,
// SwitchGLU activation, down projection).
//
// Codes.  A row's codes form one little-endian bit stream over its uint32
// words: element i sits at bits [b i, b i + b).  A group of 64 codes is 2b
// whole words (10 for 5 bits, 12 for 6), so groups start on word
// boundaries and a row's scales and biases index groups as for 4 and 8 bits.
//
// Work.  An item is (active expert, chunk of up to MT of its tokens, block
// of 12 weight features); the persistent CTAs take equal contiguous ranges
// of the item list, so a CTA walks the feature blocks of one chunk after the
// other.  The chunk's token values are staged once in shared memory as fp32
// ([token][K]; bf16 rounding for fp32 rows, as the other GEMV paths apply)
// and stay there while the CTA's items keep to that chunk.  While a CTA
// computes an item it asks L2 for the code, scale and bias lines of its next
// item, so the weight loads of that item find their lines in L2.
// Warp w of an item computes feature f = 12 block + w: for SwiGLU its gate
// row f and up row n_out + f, else row f.  Lane l takes codes 2l and 2l + 1
// of every group (one funnel shift over the group's words brings both),
// dequantizes them in fp32 (s q + b, s and b exact from fp16) and
// accumulates them against each token's two values; the 32 lane partials are
// added by a fixed xor butterfly.  A row's value depends only on its own
// codes, scales, biases and the tokens, so the fused gate_up product equals
// the separate gate and up products bit for bit.
#include <cuda_fp16.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kBtThreads = 384;
constexpr int kBtWarps = kBtThreads / 32;  // features per item
constexpr int kBtMaxTokens = 8;            // tokens per chunk (at most)
constexpr int kBtMaxE = 1024;
constexpr size_t kBtMaxStage = 200 * 1024;  // staged token bytes (at most)

enum BtMode { kBtSwiglu = 0, kBtRaw = 1 };
enum BtAct { kBtActX = 0, kBtActF32 = 1, kBtActBf16 = 2 };

struct BtParams {
  const void* act;  // x [T, K] bf16 (gathered by token), or h [rows, K] (by sorted row)
  int act_kind;
  const int32_t* sorted;   // sorted_assign (kBtActX)
  const int32_t* offsets;  // [E+1]
  int T, kmax, E, K;
  int n_rows;  // weight rows per expert
  int n_out;   // output columns: n_rows / 2 (SWIGLU) or n_rows
  int blocks;  // feature blocks of kBtWarps per (expert, chunk)
  int mt;      // tokens per chunk
  const uint32_t* wq;
  const uint16_t* ws;
  const uint16_t* wb;
  void* out;
  int out_dtype;
  unsigned int* err;
};

// Activation value k of row `row` as fp32 (bf16 rounding for fp32 rows, as
// the other GEMV paths apply).
__device__ __forceinline__ float bt_act(const BtParams& p, int64_t row, int64_t k) {
  if (p.act_kind == kBtActF32)
    return bf16_bits_to_f32(f32_to_bf16_rne(__ldg(static_cast<const float*>(p.act) + row * p.K + k)));
  return bf16_bits_to_f32(__ldg(static_cast<const uint16_t*>(p.act) + row * p.K + k));
}

__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

template <int BITS, int MODE, int MT>
__global__ void __launch_bounds__(kBtThreads, 1) gemv_bits_kernel(BtParams p) {
  constexpr int kGroupWords = 2 * BITS;  // 64 codes of a group
  constexpr uint32_t kMask = (1u << BITS) - 1u;
  constexpr int kRows = MODE == kBtSwiglu ? 2 : 1;
  extern __shared__ float bt_x[];  // staged tokens [mt][K]
  __shared__ int act_e[kBtMaxE + 1], act_lo[kBtMaxE + 1], act_m[kBtMaxE + 1], act_base[kBtMaxE + 1];
  __shared__ int n_act_sh;
  __shared__ int wtot[kBtWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int mt = MT;  // tokens per chunk (p.mt)
  pdl_wait();
  pdl_trigger();

  // active experts in id order, with segment start and length
  if (tid == 0) n_act_sh = 0;
  __syncthreads();
  for (int base = 0; base < p.E; base += kBtThreads) {
    const int e = base + tid;
    int lo = 0, m = 0;
    if (e < p.E) {
      lo = __ldg(p.offsets + e);
      m = __ldg(p.offsets + e + 1) - lo;
    }
    const bool act = m > 0;
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, act);
    if (lane == 0) wtot[warp] = __popc(bal);
    __syncthreads();
    int before = n_act_sh;
    for (int w = 0; w < warp; ++w) before += wtot[w];
    if (act) {
      const int a = before + __popc(bal & lanemask_lt());
      act_e[a] = e;
      act_lo[a] = lo;
      act_m[a] = m;
    }
    __syncthreads();
    if (tid == 0) {
      int s = 0;
      for (int w = 0; w < kBtWarps; ++w) s += wtot[w];
      n_act_sh += s;
    }
    __syncthreads();
  }
  const int n_act = n_act_sh;
  // items before each active expert: chunks of mt tokens x feature blocks
  if (warp == 0) {
    int carry = 0;
    for (int a0 = 0; a0 < n_act; a0 += 32) {
      const int a = a0 + lane;
      int v = a < n_act ? ((act_m[a] + mt - 1) / mt) * p.blocks : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, v, off);
        if (lane >= off) v += y;
      }
      if (a < n_act) act_base[a + 1] = carry + v;
      carry += __shfl_sync(0xFFFFFFFFu, v, 31);
    }
    if (lane == 0) act_base[0] = 0;
  }
  __syncthreads();
  const int64_t n_items = act_base[n_act];
  const int64_t it0 = n_items * blockIdx.x / gridDim.x;
  const int64_t it1 = n_items * (blockIdx.x + 1) / gridDim.x;
  const int ngroups = p.K / 64;
  const int64_t row_words = (int64_t)p.K * BITS / 32;
  // this lane's codes 2 lane, 2 lane + 1 of a group: bits [2 lane b, 2 lane b + 2b)
  const int bit0 = 2 * lane * BITS;
  const int w0 = bit0 >> 5, sh = bit0 & 31;

  struct Item {
    int a, c, blk;
  };
  auto item_at = [&](int64_t it) {
    int lo = 0, hi = n_act - 1;  // last a with act_base[a] <= it
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (act_base[mid] <= it) lo = mid;
      else hi = mid - 1;
    }
    Item r;
    r.a = lo;
    const int local = (int)(it - act_base[lo]);
    r.c = local / p.blocks;
    r.blk = local - r.c * p.blocks;
    return r;
  };
  // L2 lines of an item's code rows, scales and biases (every thread a share)
  auto prefetch_item = [&](const Item& q) {
    const int64_t ebase = (int64_t)act_e[q.a] * p.n_rows;
    const int f0 = q.blk * kBtWarps;
    const int nf = min(kBtWarps, p.n_out - f0);
    for (int r = 0; r < kRows; ++r) {
      const int64_t row0 = ebase + (r == 0 ? f0 : p.n_out + f0);
      const char* cb = reinterpret_cast<const char*>(p.wq + row0 * row_words);
      const int64_t cbytes = (int64_t)nf * row_words * 4;
      for (int64_t o = (int64_t)tid * 128; o < cbytes; o += (int64_t)kBtThreads * 128)
        prefetch_l2(cb + o);
      const int64_t sbytes = (int64_t)nf * ngroups * 2;
      const char* sb = reinterpret_cast<const char*>(p.ws + row0 * ngroups);
      const char* bb = reinterpret_cast<const char*>(p.wb + row0 * ngroups);
      for (int64_t o = (int64_t)tid * 128; o < sbytes; o += (int64_t)kBtThreads * 128) {
        prefetch_l2(sb + o);
        prefetch_l2(bb + o);
      }
    }
  };

  int st_a = -1, st_c = -1;
  for (int64_t it = it0; it < it1; ++it) {
    const Item cur = item_at(it);
    const int lo_tok = act_lo[cur.a] + cur.c * mt;  // first sorted row of the chunk
    const int nt = min(mt, act_m[cur.a] - cur.c * mt);
    if (cur.a != st_a || cur.c != st_c) {
      // stage the chunk's token values (every warp is past the previous item)
      __syncthreads();
#pragma unroll 1
      for (int n = 0; n < MT; ++n) {
        float* dst = bt_x + (size_t)n * p.K;
        if (n < nt) {
          const int r = lo_tok + n;
          const int64_t row =
              p.act_kind == kBtActX ? (int64_t)(__ldg(p.sorted + r) / p.kmax) : (int64_t)r;
          for (int k = tid; k < p.K; k += kBtThreads) dst[k] = bt_act(p, row, k);
        } else {
          for (int k = tid; k < p.K; k += kBtThreads) dst[k] = 0.0f;
        }
      }
      __syncthreads();
      st_a = cur.a;
      st_c = cur.c;
    }
    if (it + 1 < it1) prefetch_item(item_at(it + 1));
    const int f = cur.blk * kBtWarps + warp;  // this warp's feature
    if (f >= p.n_out) continue;
    const int64_t ebase = (int64_t)act_e[cur.a] * p.n_rows;
    int64_t wrow[kRows];
    wrow[0] = ebase + f;
    if (MODE == kBtSwiglu) wrow[kRows - 1] = ebase + p.n_out + f;
    float acc[kRows][MT];
#pragma unroll
    for (int q = 0; q < kRows; ++q)
#pragma unroll
      for (int n = 0; n < MT; ++n) acc[q][n] = 0.0f;
    // this lane's pair of staged values: token n, group g at xs[n K / 2 + 32 g]
    const float2* xs = reinterpret_cast<const float2*>(bt_x) + lane;
    const int kh = p.K >> 1;
    // scales and biases of 32 groups per load (lane l holds group g32 + l);
    // code words in batches of kGb groups, the next batch loaded while the
    // current one is computed
    constexpr int kGb = 4;
    uint32_t sv[kRows] = {}, bv[kRows] = {};
    uint32_t wlo[kGb][kRows], whi[kGb][kRows], nlo[kGb][kRows], nhi[kGb][kRows];
    auto load_batch = [&](int g0, uint32_t (&lo)[kGb][kRows], uint32_t (&hi)[kGb][kRows]) {
#pragma unroll
      for (int j = 0; j < kGb; ++j)
#pragma unroll
        for (int q = 0; q < kRows; ++q) {
          lo[j][q] = hi[j][q] = 0u;
          if (g0 + j < ngroups) {
            const uint32_t* gw = p.wq + wrow[q] * row_words + (int64_t)(g0 + j) * kGroupWords;
            lo[j][q] = __ldg(gw + w0);
            if (w0 + 1 < kGroupWords) hi[j][q] = __ldg(gw + w0 + 1);
          }
        }
    };
    load_batch(0, wlo, whi);
    for (int g0 = 0; g0 < ngroups; g0 += kGb) {
      if ((g0 & 31) == 0) {
#pragma unroll
        for (int q = 0; q < kRows; ++q) {
          const int gl = g0 + lane;
          sv[q] = gl < ngroups ? __ldg(p.ws + wrow[q] * ngroups + gl) : 0u;
          bv[q] = gl < ngroups ? __ldg(p.wb + wrow[q] * ngroups + gl) : 0u;
        }
      }
      if (g0 + kGb < ngroups) load_batch(g0 + kGb, nlo, nhi);
#pragma unroll
      for (int j = 0; j < kGb; ++j) {
        const int g = g0 + j;
        if (g >= ngroups) break;
        float2 xv[MT];
        const float2* xg = xs + g * 32;
#pragma unroll
        for (int n = 0; n < MT; ++n) xv[n] = xg[n * kh];
#pragma unroll
        for (int q = 0; q < kRows; ++q) {
          const uint32_t v = __funnelshift_r(wlo[j][q], whi[j][q], sh);
          const float q0 = (float)(v & kMask), q1 = (float)((v >> BITS) & kMask);
          const float s = f16_bits_to_f32((uint16_t)__shfl_sync(0xFFFFFFFFu, sv[q], g & 31));
          const float b = f16_bits_to_f32((uint16_t)__shfl_sync(0xFFFFFFFFu, bv[q], g & 31));
          const float d0 = fmaf(s, q0, b), d1 = fmaf(s, q1, b);
#pragma unroll
          for (int n = 0; n < MT; ++n) acc[q][n] = fmaf(d1, xv[n].y, fmaf(d0, xv[n].x, acc[q][n]));
        }
      }
#pragma unroll
      for (int j = 0; j < kGb; ++j)
#pragma unroll
        for (int q = 0; q < kRows; ++q) {
          wlo[j][q] = nlo[j][q];
          whi[j][q] = nhi[j][q];
        }
    }
    // the 32 lane partials of every row and token, by a fixed xor butterfly
#pragma unroll
    for (int q = 0; q < kRows; ++q)
#pragma unroll
      for (int n = 0; n < MT; ++n)
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
          acc[q][n] = __fadd_rn(acc[q][n], __shfl_xor_sync(0xFFFFFFFFu, acc[q][n], off));
#pragma unroll
    for (int n = 0; n < MT; ++n) {
      if (lane != n || n >= nt) continue;
      const int64_t orow = (int64_t)lo_tok + n;
      if (MODE == kBtSwiglu) {
        const float hv = swiglu_f32(acc[0][n], acc[kRows - 1][n]);
        if (p.out_dtype == MOE_DTYPE_BF16)
          static_cast<uint16_t*>(p.out)[orow * p.n_out + f] = f32_to_bf16_rne(hv);
        else
          static_cast<float*>(p.out)[orow * p.n_out + f] = hv;
      } else if (p.out_dtype == MOE_DTYPE_BF16) {
        static_cast<uint16_t*>(p.out)[orow * p.n_out + f] = f32_to_bf16_rne(acc[0][n]);
      } else {
        static_cast<float*>(p.out)[orow * p.n_out + f] = acc[0][n];
      }
    }
  }
}

template <int BITS, int MODE, int MT>
moe_status_t launch_bits_mt(const BtParams& p, cudaStream_t st) {
  auto kern = gemv_bits_kernel<BITS, MODE, MT>;
  const size_t smem = (size_t)p.mt * p.K * sizeof(float);
  // the static arrays count against the same limit: raise it for any size
  static size_t set_max[moe_host::kMaxCachedDevices] = {};  // per device
  const int dev = moe_host::device_index();
  if (smem > set_max[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    set_max[dev] = smem;
  }
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kBtThreads, smem) != cudaSuccess ||
      occ < 1)
    return MOE_ERR_CUDA;
  return moe_host::launch(kern, occ * moe_host::sm_count(), kBtThreads, smem, st, p);
}

template <int BITS, int MODE>
moe_status_t launch_bits(const BtParams& p, cudaStream_t st) {
  switch (p.mt) {
    case 8: return launch_bits_mt<BITS, MODE, 8>(p, st);
    case 4: return launch_bits_mt<BITS, MODE, 4>(p, st);
    case 2: return launch_bits_mt<BITS, MODE, 2>(p, st);
    default: return launch_bits_mt<BITS, MODE, 1>(p, st);
  }
}

}  // namespace

moe_status_t gemv_bits_qmm(const void* act, int act_kind, const int32_t* sorted,
                           const int32_t* offsets, int T, int kmax, int E, int K, int n_rows,
                           bool swiglu, const uint32_t* wq, const uint16_t* ws, const uint16_t* wb,
                           int bits, void* out, int out_dtype, cudaStream_t st) {
  if ((bits != 5 && bits != 6) || K % 64 != 0 || E > kBtMaxE) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)T * kmax == 0) return MOE_OK;
  BtParams p;
  p.act = act;
  p.act_kind = act_kind;
  p.sorted = sorted;
  p.offsets = offsets;
  p.T = T;
  p.kmax = kmax;
  p.E = E;
  p.K = K;
  p.n_rows = n_rows;
  p.n_out = swiglu ? n_rows / 2 : n_rows;
  p.blocks = (p.n_out + kBtWarps - 1) / kBtWarps;
  // tokens per chunk: an expert holds at most T rows, and the staged values
  // must fit in shared memory
  int mt = 1;
  while (mt < kBtMaxTokens && mt < T && (size_t)(2 * mt) * K * sizeof(float) <= kBtMaxStage)
    mt <<= 1;
  if ((size_t)mt * K * sizeof(float) > kBtMaxStage) return MOE_ERR_UNSUPPORTED;
  p.mt = mt;
  p.wq = wq;
  p.ws = ws;
  p.wb = wb;
  p.out = out;
  p.out_dtype = out_dtype;
  p.err = moe_host::device_error_word();
  if ((int64_t)p.blocks * ((int64_t)T * kmax + E) >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  if (bits == 5)
    return swiglu ? launch_bits<5, kBtSwiglu>(p, st) : launch_bits<5, kBtRaw>(p, st);
  return swiglu ? launch_bits<6, kBtSwiglu>(p, st) : launch_bits<6, kBtRaw>(p, st);
}

}  // namespace moe

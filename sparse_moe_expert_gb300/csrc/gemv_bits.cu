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
// Arithmetic.  Per group of 64 elements of a row (scale s, bias b):
//   sum_i x_i (s q_i + b) = s * sum_i q_i x_i + b * X,   X = sum_i x_i.
// sum q x runs on the tensor cores (mma.sync.m16n8k16, fp16 x fp16 -> fp32):
// two codes OR-ed into the two halves of a 32-bit word are the fp16
// subnormals (q0, q1) * 2^-24, exact, and the token values are staged as
// fp16 x * 2^e with one power of two per token and group chosen so that the
// group's max |x| 2^e lies in [2^14, 2^15) (exact for bf16 values in range).
// One MMA step takes, in lane (g, t), codes 16t + 4s .. 16t + 4s + 3 of the
// group (s = 0..3) for A and the same elements of token g for B, so each
// lane reads one contiguous run of 16 codes (16b bits of the group's words,
// brought to bit 0 by funnel shifts) and 16 contiguous token values.  The
// four steps give P = 2^(e-24) sum q x for 16 rows x 8 tokens; CUDA cores
// add s 2^(24-e) P and b X per group.
//
// Work.  An item is (active expert, chunk of up to MT of its tokens, block
// of 16 row tiles); each of the 16 warps takes one tile of 16 rows (SwiGLU:
// 8 gate rows and the 8 up rows of the same features) over the whole row,
// so a row's value is reduced in one fixed order whatever rows share its
// tile, and the fused gate_up product equals the separate gate and up
// products bit for bit.  The chunk's token fragments are staged once in
// shared memory and stay while the CTA's items keep to that chunk.  Each
// warp streams its rows' codes, scales and biases through a ring of
// shared-memory stages filled by cp.async one stage (four groups) ahead.
#include <cuda_fp16.h>

#include "async.cuh"
#include "common.cuh"

namespace moe {
namespace {

constexpr int kBtThreads = 512;
constexpr int kBtWarps = kBtThreads / 32;  // row tiles per item
constexpr int kBtMaxTokens = 8;            // tokens per chunk (the MMA's n)
constexpr int kBtMaxE = 1024;
constexpr size_t kBtMaxSmem = 225 * 1024;  // dynamic shared memory (at most)

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
  int blocks;  // item blocks of kBtWarps row tiles per (expert, chunk)
  int mt;      // tokens per chunk
  const uint32_t* wq;
  const uint16_t* ws;
  const uint16_t* wb;
  void* out;
  int out_dtype;
  unsigned int* err;
};

// Ring of a warp: two slots (with 16 warps, deeper rings measured slower:
// the cp.async copies in flight compete with the shared memory for the
// SM's L1 storage), each holding kRingGroups groups of its 16 rows: the
// codes, one row after another at a stride of 8b + 4 words (44 for 5 bits,
// 52 for 6: 16-byte aligned, and the words that the 8 rows x 4 run offsets
// of one read touch fall in 32 distinct banks), then per row the 4 scales
// and the 4 biases (16 bytes).
constexpr int kRingGroups = 4;
__host__ __device__ constexpr int bt_ring_depth(int) { return 2; }
__host__ __device__ constexpr int bt_ring_row_words(int bits) { return kRingGroups * 2 * bits + 4; }
__host__ __device__ constexpr int bt_ring_codes_bytes(int bits) { return 16 * bt_ring_row_words(bits) * 4; }
__host__ __device__ constexpr int bt_ring_slot_bytes(int bits) { return bt_ring_codes_bytes(bits) + 16 * 16; }

// Shared memory: the active-expert lists [4][E + 1] ints; staged tokens, fp16
// values [mt][K + 8] (16 bytes of padding per token row keep the fragment
// loads free of bank conflicts), then (X, 2^(24-e)) per group and token
// [K / 64][mt2]; then the warps' code rings.
__host__ __device__ inline int bt_xs_stride(int K) { return K + 8; }
__host__ __device__ inline size_t bt_act_bytes(int E) { return ((size_t)4 * (E + 1) * 4 + 15) & ~(size_t)15; }
__host__ __device__ inline size_t bt_stage_bytes(int K, int mt) {
  const int mt2 = mt < 2 ? 2 : mt;
  return (size_t)mt * bt_xs_stride(K) * 2 + (size_t)(K / 64) * mt2 * 8;
}
__host__ __device__ inline size_t bt_smem_bytes(int bits, int K, int mt, int E) {
  return bt_act_bytes(E) + bt_stage_bytes(K, mt) + (size_t)kBtWarps * bt_ring_depth(bits) * bt_ring_slot_bytes(bits);
}

// 8 or 16 bytes global -> shared, asynchronous (completion by cp.async groups).
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// the two fp16 numbers of a word (low half first) as floats
__device__ __forceinline__ void half2_bits_to_f32(uint32_t w, float& lo, float& hi) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
  lo = f.x;
  hi = f.y;
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// d = A B (+ d when acc)
__device__ __forceinline__ void mma_bt(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                       uint32_t a3, uint32_t b0, uint32_t b1, bool acc) {
  if (acc)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// Codes 2j and 2j + 1 of a lane's run (its bits from bit 0 of n[0..2]) as
// the fp16 subnormal pair (q_2j, q_2j+1) 2^-24.
template <int BITS>
__device__ __forceinline__ uint32_t bt_pair(const uint32_t (&n)[3], int j) {
  constexpr uint32_t kMask = (1u << BITS) - 1u;
  const int pos = 2 * j * BITS;  // compile-time after unrolling
  const int wi = pos >> 5, sh = pos & 31;
  const uint32_t lo = n[wi], hi = wi + 1 < 3 ? n[wi + 1] : 0u;
  const uint32_t v = sh == 0 ? lo : __funnelshift_r(lo, hi, sh);
  // q0 from bits 0.., q1 moved from bit BITS to bit 16
  return (v & kMask) | ((v << (16 - BITS)) & (kMask << 16));
}

template <int BITS, int MODE, int MT>
__global__ void __launch_bounds__(kBtThreads, 1) gemv_bits_kernel(BtParams p) {
  constexpr int kGroupWords = 2 * BITS;  // 64 codes of a group
  constexpr int mt = MT;
  constexpr int mt2 = MT < 2 ? 2 : MT;
  constexpr int kTileRows = 16;  // SWIGLU: 8 features (gate rows, then up rows)
  constexpr int kRing = bt_ring_depth(BITS);
  extern __shared__ __align__(16) unsigned char bt_smem[];
  __shared__ int n_act_sh;
  __shared__ int wtot[kBtWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ngroups = p.K / 64;
  const int xs_stride = bt_xs_stride(p.K);
  int* act_e = reinterpret_cast<int*>(bt_smem);
  int* act_lo = act_e + (p.E + 1);
  int* act_m = act_lo + (p.E + 1);
  int* act_base = act_m + (p.E + 1);
  unsigned char* stage_base = bt_smem + bt_act_bytes(p.E);
  uint16_t* xh = reinterpret_cast<uint16_t*>(stage_base);  // [mt][xs_stride] fp16
  float2* xsum = reinterpret_cast<float2*>(stage_base + (size_t)mt * xs_stride * 2);  // [G][mt2]
  unsigned char* ring = stage_base + bt_stage_bytes(p.K, mt) +
                        (size_t)warp * bt_ring_depth(BITS) * bt_ring_slot_bytes(BITS);  // this warp's ring
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
  // items before each active expert: chunks of mt tokens x item blocks
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
  const int64_t row_words = (int64_t)p.K * BITS / 32;
  const int g = lane >> 2, t = lane & 3;
  // this lane's run of 16 codes of a group: bits [16 t b, 16 t b + 16 b)
  const int run_w0 = (16 * t * BITS) >> 5, run_sh = (16 * t * BITS) & 31;

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
  int st_a = -1, st_c = -1;
  for (int64_t it = it0; it < it1; ++it) {
    const Item cur = item_at(it);
    const int lo_tok = act_lo[cur.a] + cur.c * mt;  // first sorted row of the chunk
    const int nt = min(mt, act_m[cur.a] - cur.c * mt);
    if (cur.a != st_a || cur.c != st_c) {
      // stage the chunk's tokens (every warp is past the previous item): per
      // (token, group) one thread loads the 64 values, finds the power of
      // two, the sum (in element order) and the scaled fp16 values
      __syncthreads();
      for (int i = tid; i < mt2 * ngroups; i += kBtThreads) {
        const int n = i / ngroups, G = i - n * ngroups;
        uint32_t v[32];  // 64 bf16 values, two per word
#pragma unroll
        for (int w = 0; w < 32; ++w) v[w] = 0u;
        if (n < nt) {
          const int r = lo_tok + n;
          const int64_t row =
              p.act_kind == kBtActX ? (int64_t)(__ldg(p.sorted + r) / p.kmax) : (int64_t)r;
          if (p.act_kind == kBtActF32) {
            const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.act) +
                                                                row * p.K + (int64_t)G * 64);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const float4 f = __ldg(src + q);
              v[2 * q] = (uint32_t)f32_to_bf16_rne(f.x) | ((uint32_t)f32_to_bf16_rne(f.y) << 16);
              v[2 * q + 1] = (uint32_t)f32_to_bf16_rne(f.z) | ((uint32_t)f32_to_bf16_rne(f.w) << 16);
            }
          } else {
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.act) +
                                                              row * p.K + (int64_t)G * 64);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint4 u = __ldg(src + q);
              v[4 * q] = u.x;
              v[4 * q + 1] = u.y;
              v[4 * q + 2] = u.z;
              v[4 * q + 3] = u.w;
            }
          }
        }
        float mx = 0.0f, xsm = 0.0f;
#pragma unroll
        for (int w = 0; w < 32; ++w) {
          const float f0 = __uint_as_float(v[w] << 16), f1 = __uint_as_float(v[w] & 0xFFFF0000u);
          mx = fmaxf(mx, fmaxf(fabsf(f0), fabsf(f1)));
          xsm += f0;
          xsm += f1;
        }
        const int E8 = (int)((__float_as_uint(mx) >> 23) & 0xFFu);
        int e = mx == 0.0f ? 0 : (E8 == 0 ? 100 : 141 - E8);
        e = e < -100 ? -100 : (e > 100 ? 100 : e);
        const float sc = __uint_as_float((uint32_t)(127 + e) << 23);
        if (n < mt) {
          uint4* dst = reinterpret_cast<uint4*>(xh + (size_t)n * xs_stride + G * 64);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            uint32_t hw[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t w = v[4 * q + j];
              const __half2 h2 = __floats2half2_rn(__uint_as_float(w << 16) * sc,
                                                   __uint_as_float(w & 0xFFFF0000u) * sc);
              hw[j] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            dst[q] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          }
        }
        xsum[(size_t)G * mt2 + n] = make_float2(xsm, __uint_as_float((uint32_t)(151 - e) << 23));
      }
      __syncthreads();
      st_a = cur.a;
      st_c = cur.c;
    }
    const int tile = cur.blk * kBtWarps + warp;
    const int first = MODE == kBtSwiglu ? tile * 8 : tile * kTileRows;  // feature | row
    const int limit = MODE == kBtSwiglu ? p.n_out : p.n_rows;
    if (first >= limit) continue;  // past the matrix (warp-uniform)
    const int64_t ebase = (int64_t)act_e[cur.a] * p.n_rows;
    // MMA rows g and g + 8: gate and up rows of feature first + g (SWIGLU),
    // else rows first + g and first + g + 8; rows past the matrix read a
    // valid row and their results are dropped
    const int64_t last = ebase + p.n_rows - 1;
    // B columns past the chunk repeat one of its tokens (never read back)
    const int bn = min(g, mt - 1);
    const uint4* xq = reinterpret_cast<const uint4*>(xh + (size_t)bn * xs_stride + 16 * t);
    const float2* xsp = xsum + (t < (mt2 >> 1) ? 2 * t : mt2 - 2);
    float as[4] = {0.f, 0.f, 0.f, 0.f}, ab[4] = {0.f, 0.f, 0.f, 0.f};
    // The tile streams through the warp's ring: stage q holds groups
    // 4q .. 4q + 3 of the 16 rows (ring row r is MMA row r: rows 0-7 the
    // rows g of the lanes, 8-15 their rows g + 8), copied with cp.async
    // kRing - 1 stages ahead of its use.  When the groups of a row are a
    // multiple of 4 (every row and stage start is then 16-byte aligned for
    // the codes and 8-byte aligned for the scales) a stage is 16-byte code
    // copies and one 8-byte scale or bias copy per lane; otherwise 8-byte
    // code copies with the words past the row end taken from its start
    // (unused), and the scales loaded and stored in order, the group index
    // clamped to the row.
    constexpr int kRowWords = bt_ring_row_words(BITS);
    constexpr int kSegWords = kRingGroups * kGroupWords;  // a row's code words of one stage
    constexpr int kRow16 = kSegWords / 4;                 // its 16-byte copies
    constexpr int kLane16 = 16 * kRow16 / 32;             // a lane's per stage
    static_assert(16 * kRow16 % 32 == 0, "copies split evenly over the lanes");
    const int nst = (ngroups + kRingGroups - 1) / kRingGroups;
    const bool whole = (ngroups & (kRingGroups - 1)) == 0;
    auto ring_row = [&](int r) -> int64_t {  // weight row of ring row r
      return r < 8 ? min(ebase + first + r, last)
                   : min(MODE == kBtSwiglu ? ebase + p.n_out + first + (r - 8) : ebase + first + r, last);
    };
    const uint32_t* csrc[kLane16];  // copy i of the lane: words cw .. cw + 3 of ring row r
    int cdst[kLane16];
#pragma unroll
    for (int i = 0; i < kLane16; ++i) {
      const int c = lane + 32 * i;
      const int r = c / kRow16, cw = (c - r * kRow16) * 4;
      csrc[i] = p.wq + ring_row(r) * row_words + cw;
      cdst[i] = (r * kRowWords + cw) * 4;
    }
    // scale copy of the lane: ring row lane / 2, scales (even lane) or biases
    const int sr = lane >> 1;
    const uint16_t* ssrc = ((lane & 1) ? p.wb : p.ws) + ring_row(sr) * ngroups;
    const int sdst = bt_ring_codes_bytes(BITS) + sr * 16 + (lane & 1) * 8;
    auto issue = [&](int q) {
      if (q < nst) {
        unsigned char* slot = ring + (size_t)(q % kRing) * bt_ring_slot_bytes(BITS);
        const int G0 = q * kRingGroups;
        if (whole) {
#pragma unroll
          for (int i = 0; i < kLane16; ++i) cp_async16(slot + cdst[i], csrc[i] + (int64_t)G0 * kGroupWords);
          cp_async8(slot + sdst, ssrc + G0);
        } else {
          for (int c = lane; c < 16 * (kSegWords / 2); c += 32) {
            const int r = c / (kSegWords / 2), cw = (c - r * (kSegWords / 2)) * 2;
            const int64_t w = (int64_t)G0 * kGroupWords + cw;
            cp_async8(slot + (r * kRowWords + cw) * 4, p.wq + ring_row(r) * row_words + (w < row_words ? w : 0));
          }
          uint16_t v[kRingGroups];
#pragma unroll
          for (int j = 0; j < kRingGroups; ++j) v[j] = __ldg(ssrc + min(G0 + j, ngroups - 1));
          *reinterpret_cast<uint2*>(slot + sdst) =
              make_uint2((uint32_t)v[0] | ((uint32_t)v[1] << 16), (uint32_t)v[2] | ((uint32_t)v[3] << 16));
        }
      }
      cp_async_commit();  // one group per stage, empty or not
    };
#pragma unroll
    for (int q = 0; q < kRing - 1; ++q) issue(q);
    for (int q = 0; q < nst; ++q) {
      issue(q + kRing - 1);
      cp_async_wait<kRing - 1>();  // stage q has landed (this lane's copies) ...
      __syncwarp();                // ... and every lane's
      const unsigned char* slot = ring + (size_t)(q % kRing) * bt_ring_slot_bytes(BITS);
      const uint32_t* rlo = reinterpret_cast<const uint32_t*>(slot) + g * kRowWords + run_w0;
      const uint32_t* rhi = reinterpret_cast<const uint32_t*>(slot) + (8 + g) * kRowWords + run_w0;
      const uint4 sbl = *reinterpret_cast<const uint4*>(slot + bt_ring_codes_bytes(BITS) + g * 16);
      const uint4 sbh = *reinterpret_cast<const uint4*>(slot + bt_ring_codes_bytes(BITS) + (8 + g) * 16);
      // scales (s) and biases (b) of the stage's 4 groups, rows g and g + 8
      float sl[4], sh[4], bl[4], bh[4];
      half2_bits_to_f32(sbl.x, sl[0], sl[1]);
      half2_bits_to_f32(sbl.y, sl[2], sl[3]);
      half2_bits_to_f32(sbl.z, bl[0], bl[1]);
      half2_bits_to_f32(sbl.w, bl[2], bl[3]);
      half2_bits_to_f32(sbh.x, sh[0], sh[1]);
      half2_bits_to_f32(sbh.y, sh[2], sh[3]);
      half2_bits_to_f32(sbh.z, bh[0], bh[1]);
      half2_bits_to_f32(sbh.w, bh[2], bh[3]);
#pragma unroll
      for (int j = 0; j < kRingGroups; ++j) {
        const int G = q * kRingGroups + j;
        if (G < ngroups) {
          const float s0 = sl[j], s1 = sh[j], b0 = bl[j], b1 = bh[j];
          uint32_t w[6];
#pragma unroll
          for (int i = 0; i < 3; ++i) {
            w[i] = rlo[j * kGroupWords + i];
            w[3 + i] = rhi[j * kGroupWords + i];
          }
          // this lane's run of 16 codes, from bit 0
          uint32_t rl[3], rh[3];
          rl[0] = __funnelshift_r(w[0], w[1], run_sh);
          rl[1] = __funnelshift_r(w[1], w[2], run_sh);
          rl[2] = w[2] >> run_sh;
          rh[0] = __funnelshift_r(w[3], w[4], run_sh);
          rh[1] = __funnelshift_r(w[4], w[5], run_sh);
          rh[2] = w[5] >> run_sh;
          const uint4 xa = xq[(size_t)G * 8], xb = xq[(size_t)G * 8 + 1];  // 16 fp16 values
          const uint32_t xf[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
          float d[4];
#pragma unroll
          for (int s = 0; s < 4; ++s)
            mma_bt(d, bt_pair<BITS>(rl, 2 * s), bt_pair<BITS>(rh, 2 * s),
                   bt_pair<BITS>(rl, 2 * s + 1), bt_pair<BITS>(rh, 2 * s + 1), xf[2 * s],
                   xf[2 * s + 1], s > 0);
          const float4 X = *reinterpret_cast<const float4*>(xsp + (size_t)G * mt2);  // tokens 2t, 2t+1
          as[0] = fmaf(s0 * X.y, d[0], as[0]);
          as[1] = fmaf(s0 * X.w, d[1], as[1]);
          as[2] = fmaf(s1 * X.y, d[2], as[2]);
          as[3] = fmaf(s1 * X.w, d[3], as[3]);
          ab[0] = fmaf(b0, X.x, ab[0]);
          ab[1] = fmaf(b0, X.z, ab[1]);
          ab[2] = fmaf(b1, X.x, ab[2]);
          ab[3] = fmaf(b1, X.z, ab[3]);
        }
      }
      __syncwarp();  // the slot is rewritten by the next iteration's copies
    }
    // lane (g, t): MMA rows g and g + 8, tokens 2t and 2t + 1
    const float v0 = as[0] + ab[0], v1 = as[1] + ab[1], v2 = as[2] + ab[2], v3 = as[3] + ab[3];
    const int n0 = 2 * t, n1 = 2 * t + 1;
    if (MODE == kBtSwiglu) {
      const int f = first + g;
      if (f < p.n_out) {
        const float h0 = swiglu_f32(v0, v2), h1 = swiglu_f32(v1, v3);
        if (n0 < nt) {
          const int64_t oi = (int64_t)(lo_tok + n0) * p.n_out + f;
          if (p.out_dtype == MOE_DTYPE_BF16) static_cast<uint16_t*>(p.out)[oi] = f32_to_bf16_rne(h0);
          else static_cast<float*>(p.out)[oi] = h0;
        }
        if (n1 < nt) {
          const int64_t oi = (int64_t)(lo_tok + n1) * p.n_out + f;
          if (p.out_dtype == MOE_DTYPE_BF16) static_cast<uint16_t*>(p.out)[oi] = f32_to_bf16_rne(h1);
          else static_cast<float*>(p.out)[oi] = h1;
        }
      }
    } else {
      const float vv[4] = {v0, v1, v2, v3};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = first + g + (i >> 1) * 8, n = 2 * t + (i & 1);
        if (r < p.n_rows && n < nt) {
          const int64_t oi = (int64_t)(lo_tok + n) * p.n_out + r;
          if (p.out_dtype == MOE_DTYPE_BF16) static_cast<uint16_t*>(p.out)[oi] = f32_to_bf16_rne(vv[i]);
          else static_cast<float*>(p.out)[oi] = vv[i];
        }
      }
    }
  }
}

template <int BITS, int MODE, int MT>
moe_status_t launch_bits_mt(const BtParams& p, cudaStream_t st) {
  auto kern = gemv_bits_kernel<BITS, MODE, MT>;
  const size_t smem = bt_smem_bytes(BITS, p.K, MT, p.E);
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
  // item blocks: 16 row tiles of 16 rows (SWIGLU: 8 features each)
  p.blocks = swiglu ? (p.n_out + kBtWarps * 8 - 1) / (kBtWarps * 8)
                    : (n_rows + kBtWarps * 16 - 1) / (kBtWarps * 16);
  // tokens per chunk: an expert holds at most T rows, and the staged values
  // must fit in shared memory
  int mt = 1;
  while (mt < kBtMaxTokens && mt < T && bt_smem_bytes(bits, K, 2 * mt, E) <= kBtMaxSmem) mt <<= 1;
  if (bt_smem_bytes(bits, K, mt, E) > kBtMaxSmem) return MOE_ERR_UNSUPPORTED;
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

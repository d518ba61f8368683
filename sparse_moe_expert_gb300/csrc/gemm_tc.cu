// Grouped GEMM on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators, TMA-fed tiles): the prefill / batched path of the two
// quantized products.
//
// Page "oMLX MoE gate/up 融合优化：qwen35_moe_gate_up 实现剖析", 融合原理 and
// 实现剖析 ④ (one product with the [gate; up] matrix per expert, split, SiLU
// activation, down projection); page "Qwen3.5 Block在llama.cpp中的映射与优化
// 原理", section 4.2 (each expert only sees the tokens routed to it).
//
// Orientation: weights are the MMA's A operand (M = 128 rows of an expert),
// the expert's tokens are B (N = 128 tokens of its segment), K = the
// contraction axis, so D[m, n] lands in TMEM lane m, column n.  A SWIGLU tile
// holds two accumulators, gate rows n0..n0+127 and up rows I+n0..I+n0+127,
// so the epilogue has both halves of an output in the same thread.
//
// One CTA per SM, persistent over the tiles (active expert, m-tile, n-tile);
// n-tiles of the same weights are adjacent so neighbouring CTAs share them in
// L2.  Warp roles:
//   warp 5      loader: per k-block of 64, TMA loads the packed codes of the
//               tile's rows (2D tensor map) and the token tile: a 4-row gather
//               (tile::gather4) of the token rows of x for gate_up, a 2D tile
//               of h for down, both 128-byte swizzled as the MMA expects;
//   warps 6-13  dequant: read the codes from shared memory, w = s*q + b in
//               fp32 (packed FMA), round to bf16, write the A tile in the
//               128-byte-swizzled K-major layout, proxy fence, arrive;
//   warp 4      MMA: one thread issues tcgen05.mma (kind::f16, bf16 x bf16 ->
//               fp32) per 16-wide K slice, commits stage release and
//               accumulator completion to mbarriers;
//   warps 0-3   epilogue: tcgen05.ld of the accumulator, SiLU(gate)*up or raw,
//               store.  TMEM accumulators are double-buffered.
// Every mbarrier wait is bounded; a wait that runs out sets
// MOE_DEVERR_TIMEOUT, the CTA stops issuing, drains what is in flight and
// frees its TMEM.
#include <cuda.h>
#include <cuda_fp16.h>

#include <mutex>

#include "async.cuh"
#include "common.cuh"

namespace moe {
namespace {

constexpr int BM = 128;  // weight rows per accumulator
constexpr int BN = 128;  // tokens per tile
constexpr int BK = 64;   // contraction per stage = one scale group = one 128-B swizzle atom
constexpr int kEpiWarps = 4, kMmaWarp = 4, kLoadWarp = 5, kDeqWarp0 = 6, kDeqWarps = 8;
constexpr int kTcThreads = (kDeqWarp0 + kDeqWarps) * 32;  // 448
constexpr int kTileBytes = BM * BK * 2;                   // 16 KB bf16 tile (A or B)
constexpr int kMaxStages = 8;

enum TcMode { kTcSwiglu = 0, kTcRaw = 1 };
enum TcAct { kTcGatherX = 0, kTcRowsH = 1 };

struct TcParams {
  const int32_t* sorted;   // sorted_assign (gate_up)
  const int32_t* offsets;  // [E+1]
  const uint16_t* ws;      // scales  [E, n_rows, K/64]
  const uint16_t* wb;      // biases
  void* out;
  int out_dtype;
  int kmax, E, K, n_rows, n_out;
  int stages;
  int n_mt;  // m-tiles per expert
  unsigned int* err;
};

// ---- tcgen05 / TMA helpers ------------------------------------------------

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int c0, int c1,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// Four rows r0..r3 (each one box of 64 columns) into 4 consecutive 128-byte rows.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* tm, int col, int r0,
                                            int r1, int r2, int r3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
      "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulation.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once all tcgen05 operations issued so far by this thread complete.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart.  Start address must be in a 1024-byte aligned atom.
__device__ __forceinline__ uint64_t smem_desc_sw128(const void* p) {
  const uint64_t addr = smem_u32(p);
  uint64_t d = (addr >> 4) & 0x3FFFull;  // start address
  d |= 1ull << 16;                       // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;      // stride byte offset: 8 rows x 128 B
  d |= 1ull << 46;                       // descriptor version
  d |= 2ull << 61;                       // swizzle: 128 B
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// ---- tile schedule ----------------------------------------------------------

struct TileInfo {
  int e, seg_lo, m, mt, nt;
};

// tile_start[a] = first tile of active expert a (exclusive prefix), n_act entries + 1.
__device__ __forceinline__ TileInfo tile_info(const TcParams& p, const int* act_e,
                                              const int* tile_start, int n_act, int t) {
  int lo = 0, hi = n_act - 1;
  while (lo < hi) {  // last a with tile_start[a] <= t
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  TileInfo ti;
  ti.e = act_e[lo];
  ti.seg_lo = __ldg(p.offsets + ti.e);
  ti.m = __ldg(p.offsets + ti.e + 1) - ti.seg_lo;
  const int nnt = (ti.m + BN - 1) / BN;
  const int local = t - tile_start[lo];
  ti.mt = local / nnt;
  ti.nt = local % nnt;
  return ti;
}

// Weight row (within the expert) of accumulator `acc`, tile row r.
template <int MODE>
__device__ __forceinline__ int tile_weight_row(const TcParams& p, int mt, int acc, int r) {
  return MODE == kTcSwiglu ? acc * (p.n_rows / 2) + mt * BM + r : mt * BM + r;
}

template <int BITS, int MODE, int ACT>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_qmm_kernel(const __grid_constant__ CUtensorMap tm_codes,
                  const __grid_constant__ CUtensorMap tm_act, TcParams p) {
  constexpr int NACC = MODE == kTcSwiglu ? 2 : 1;
  constexpr int RAW_ROW_BYTES = BK * BITS / 8;          // code bytes per row per stage
  constexpr int RAW_BYTES = BM * RAW_ROW_BYTES;         // per accumulator
  constexpr int STAGE_BYTES = NACC * kTileBytes + kTileBytes + NACC * RAW_BYTES;
  constexpr uint32_t TMEM_COLS = NACC * BN * 2;         // double-buffered accumulators

  extern __shared__ __align__(1024) unsigned char tc_smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t raw_full[kMaxStages], a_full[kMaxStages], empty_bar[kMaxStages];
  __shared__ uint64_t tmem_full[2], tmem_empty[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int act_e[1024];
  __shared__ int tile_start[1025];
  __shared__ int n_act_sh;
  __shared__ int tok_table[BN];
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = p.stages;
  const int nkb = p.K / BK;

  // ---- set-up: barriers, TMEM, active experts and their tile ranges ----
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&a_full[s], kDeqWarps);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], kEpiWarps);
    }
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&tmem_base_sh, TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 0) {
    int n = 0, t = 0;
    for (int e = 0; e < p.E; ++e) {
      const int m = __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
      if (m > 0) {
        act_e[n] = e;
        tile_start[n] = t;
        t += p.n_mt * ((m + BN - 1) / BN);
        ++n;
      }
    }
    tile_start[n] = t;
    n_act_sh = n;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;
  const int n_act = n_act_sh;
  const int n_tiles = n_act > 0 ? tile_start[n_act] : 0;

  unsigned char* stage_base = smem;
  auto stage_a = [&](int s, int acc) { return stage_base + (size_t)s * STAGE_BYTES + acc * kTileBytes; };
  auto stage_b = [&](int s) { return stage_base + (size_t)s * STAGE_BYTES + NACC * kTileBytes; };
  auto stage_raw = [&](int s, int acc) {
    return stage_base + (size_t)s * STAGE_BYTES + (NACC + 1) * kTileBytes + acc * RAW_BYTES;
  };

  if (warp == kLoadWarp) {
    // =============================== loader ===============================
    int64_t issued = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      const TileInfo ti = tile_info(p, act_e, tile_start, n_act, t);
      if (ACT == kTcGatherX) {
        // token of each column of this tile (invalid columns repeat the first token)
        for (int n = lane; n < BN; n += 32) {
          const int col = ti.nt * BN + n;
          const int r = ti.seg_lo + (col < ti.m ? col : 0);
          tok_table[n] = __ldg(p.sorted + r) / p.kmax;
        }
        __syncwarp();
      }
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = (int)(issued % S);
        const uint32_t round = (uint32_t)(issued / S);
        if (!mbar_wait(&empty_bar[s], (round & 1u) ^ 1u, kWaitBudgetCycles) || abort_flag) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&raw_full[s], NACC * RAW_BYTES + kTileBytes);
          const int code_col = kb * (BK * BITS / 32);  // in uint32 words
#pragma unroll
          for (int acc = 0; acc < NACC; ++acc) {
            const int row = ti.e * p.n_rows + tile_weight_row<MODE>(p, ti.mt, acc, 0);
            tma_load_2d(stage_raw(s, acc), &tm_codes, code_col, row, &raw_full[s]);
          }
          if (ACT == kTcGatherX) {
            for (int g = 0; g < BN / 4; ++g)
              tma_gather4(stage_b(s) + g * 512, &tm_act, kb * BK, tok_table[4 * g],
                          tok_table[4 * g + 1], tok_table[4 * g + 2], tok_table[4 * g + 3],
                          &raw_full[s]);
          } else {
            tma_load_2d(stage_b(s), &tm_act, kb * BK, ti.seg_lo + ti.nt * BN, &raw_full[s]);
          }
        }
        __syncwarp();
        ++issued;
      }
      __syncwarp();
    }
    if (!ok) {
      if (lane == 0) {
        raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
        abort_flag = 1;
        const int64_t from = issued > S ? issued - S : 0;
        for (int64_t j = from; j < issued; ++j)
          mbar_wait(&raw_full[j % S], (uint32_t)((j / S) & 1), kWaitBudgetCycles);
      }
    }
  } else if (warp >= kDeqWarp0) {
    // =============================== dequant ===============================
    const int dt = tid - kDeqWarp0 * 32;  // 0..255
    // SWIGLU: one row of one accumulator per thread; RAW: half a row per thread
    const int acc = MODE == kTcSwiglu ? dt >> 7 : 0;
    const int r = dt & 127;
    const int khalf = MODE == kTcSwiglu ? -1 : (dt >> 7);  // RAW: which 32 of the 64 columns
    const int ngroups = p.K / 64;
    int64_t consumed = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      const TileInfo ti = tile_info(p, act_e, tile_start, n_act, t);
      int wrow = tile_weight_row<MODE>(p, ti.mt, acc, r);
      if (wrow >= p.n_rows) wrow = p.n_rows - 1;  // rows past the matrix: any valid scale
      const int64_t grow = (int64_t)ti.e * p.n_rows + wrow;
      const uint16_t* sp = p.ws + grow * ngroups;
      const uint16_t* bp = p.wb + grow * ngroups;
      uint16_t s_next = __ldg(sp), b_next = __ldg(bp);
      for (int kb = 0; kb < nkb; ++kb) {
        const float sc = f16_bits_to_f32(s_next), bi = f16_bits_to_f32(b_next);
        if (kb + 1 < nkb) {
          s_next = __ldg(sp + kb + 1);
          b_next = __ldg(bp + kb + 1);
        }
        const int s = (int)(consumed % S);
        const uint32_t round = (uint32_t)(consumed / S);
        if (!mbar_wait(&raw_full[s], round & 1u, kWaitBudgetCycles) || abort_flag) {
          ok = false;
          break;
        }
        const unsigned char* raw = stage_raw(s, acc) + r * RAW_ROW_BYTES;
        unsigned char* atile = stage_a(s, acc);
        if (BITS == 4) {
          // 8 codes per word; a word becomes one 16-byte chunk of 8 bf16
          const float2 mul = make_float2(512.0f * sc, 32.0f * sc);
          const float2 add = make_float2(bi - 512.0f * sc, bi - 32.0f * sc);
          const int c0 = MODE == kTcSwiglu ? 0 : khalf * 4;
          const int nc = MODE == kTcSwiglu ? 8 : 4;
          for (int c = c0; c < c0 + nc; c += 4) {
            const uint4 q4 = *reinterpret_cast<const uint4*>(raw + c * 4);
            const uint32_t wv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t v = wv[i];
              const uint32_t sh[4] = {v << 14, v << 6, v >> 2, v >> 10};
              uint32_t o[4];
#pragma unroll
              for (int pq = 0; pq < 4; ++pq) {
                // (1 + q_even/512, 1 + q_odd/32), then w = s*q + b exactly in fp32
                const float2 f = make_float2(__uint_as_float((sh[pq] & 0x0003C000u) | 0x3F800000u),
                                             __uint_as_float((sh[pq] & 0x003C0000u) | 0x3F800000u));
                const float2 w = __ffma2_rn(f, mul, add);
                o[pq] = pack_bf16x2(w.x, w.y);
              }
              *reinterpret_cast<uint4*>(atile + sw128_offset(r, c + i)) =
                  make_uint4(o[0], o[1], o[2], o[3]);
            }
          }
        } else {
          // 4 codes per word; two words become one 16-byte chunk
          const float2 mul = make_float2(256.0f * sc, 256.0f * sc);
          const float2 add = make_float2(bi - 256.0f * sc, bi - 256.0f * sc);
          const int c0 = MODE == kTcSwiglu ? 0 : khalf * 4;
          const int nc = MODE == kTcSwiglu ? 8 : 4;
          for (int c = c0; c < c0 + nc; c += 2) {
            const uint4 q4 = *reinterpret_cast<const uint4*>(raw + c * 8);
            const uint32_t wv[4] = {q4.x, q4.y, q4.z, q4.w};
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t v = wv[i];
              const float2 f0 = make_float2(__uint_as_float(((v << 15) & 0x007F8000u) | 0x3F800000u),
                                            __uint_as_float(((v << 7) & 0x007F8000u) | 0x3F800000u));
              const float2 f1 = make_float2(__uint_as_float(((v >> 1) & 0x007F8000u) | 0x3F800000u),
                                            __uint_as_float(((v >> 9) & 0x007F8000u) | 0x3F800000u));
              const float2 w0 = __ffma2_rn(f0, mul, add);
              const float2 w1 = __ffma2_rn(f1, mul, add);
              o[2 * i] = pack_bf16x2(w0.x, w0.y);
              o[2 * i + 1] = pack_bf16x2(w1.x, w1.y);
            }
            *reinterpret_cast<uint4*>(atile + sw128_offset(r, c)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(atile + sw128_offset(r, c + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[s]);
        ++consumed;
      }
    }
    if (!ok && lane == 0) {
      raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
      abort_flag = 1;
    }
  } else if (warp == kMmaWarp) {
    // ================================= MMA =================================
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(BM, BN);
      int64_t consumed = 0;
      int j = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++j) {
        const int buf = j & 1;
        if (!mbar_wait(&tmem_empty[buf], (uint32_t)(((j >> 1) & 1) ^ 1), kWaitBudgetCycles) ||
            abort_flag) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem_base + (uint32_t)(buf * NACC * BN);
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = (int)(consumed % S);
          const uint32_t round = (uint32_t)(consumed / S);
          if (!mbar_wait(&a_full[s], round & 1u, kWaitBudgetCycles) ||
              !mbar_wait(&raw_full[s], round & 1u, kWaitBudgetCycles) || abort_flag) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bdesc = smem_desc_sw128(stage_b(s));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
#pragma unroll
            for (int acc = 0; acc < NACC; ++acc) {
              const uint64_t adesc = smem_desc_sw128(stage_a(s, acc));
              // K advance inside the swizzle atom: 16 elements = 32 bytes
              umma_bf16(d0 + acc * BN, adesc + 2 * kk, bdesc + 2 * kk, idesc,
                        (kb | kk) != 0 ? 1u : 0u);
            }
          }
          umma_commit(&empty_bar[s]);
          ++consumed;
        }
        if (!ok) break;
        umma_commit(&tmem_full[buf]);
      }
      if (!ok) {
        raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
        abort_flag = 1;
      }
      // wait for the last MMAs of this thread before TMEM is released
      __shared__ uint64_t drain_bar;
      mbar_init(&drain_bar, 1);
      fence_barrier_init();
      umma_commit(&drain_bar);
      mbar_wait(&drain_bar, 0, kWaitBudgetCycles);
    }
    __syncwarp();
  } else {
    // =============================== epilogue ===============================
    int j = 0;
    bool ok = true;
    const int m = warp * 32 + lane;  // accumulator row = TMEM lane
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++j) {
      const TileInfo ti = tile_info(p, act_e, tile_start, n_act, t);
      const int buf = j & 1;
      if (!mbar_wait(&tmem_full[buf], (uint32_t)((j >> 1) & 1), kWaitBudgetCycles) || abort_flag) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int col = ti.mt * BM + m;  // output column
      const bool col_ok = col < p.n_out;
      const int nvalid = min(BN, ti.m - ti.nt * BN);
      const uint32_t lane_addr = tmem_base + ((uint32_t)(warp * 32) << 16) + (uint32_t)(buf * NACC * BN);
      for (int n0 = 0; n0 < BN; n0 += 16) {
        uint32_t g[16], u[16];
        tmem_ld16(lane_addr + n0, g);
        if (MODE == kTcSwiglu) tmem_ld16(lane_addr + BN + n0, u);
        tmem_ld_wait();
        if (col_ok) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (n0 + i < nvalid) {
              const int64_t row = (int64_t)ti.seg_lo + ti.nt * BN + n0 + i;
              if (MODE == kTcSwiglu) {
                const float hv = swiglu_f32(__uint_as_float(g[i]), __uint_as_float(u[i]));
                if (p.out_dtype == MOE_DTYPE_BF16)
                  static_cast<uint16_t*>(p.out)[row * p.n_out + col] = f32_to_bf16_rne(hv);
                else
                  static_cast<float*>(p.out)[row * p.n_out + col] = hv;
              } else {
                static_cast<float*>(p.out)[row * p.n_out + col] = __uint_as_float(g[i]);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tmem_empty[buf]);
    }
    if (!ok && lane == 0) {
      raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
      abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ---- host side ----------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                 uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                 CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BITS, int MODE, int ACT>
moe_status_t launch_tc(const CUtensorMap& tmc, const CUtensorMap& tma, TcParams p,
                       int64_t max_tiles, cudaStream_t st) {
  constexpr int NACC = MODE == kTcSwiglu ? 2 : 1;
  constexpr int STAGE_BYTES = NACC * kTileBytes + kTileBytes + NACC * BM * BK * BITS / 8;
  const size_t budget = 200 * 1024;
  int stages = (int)(budget / STAGE_BYTES);
  if (stages > 6) stages = 6;
  if (stages < 2) return MOE_ERR_UNSUPPORTED;
  p.stages = stages;
  const size_t smem = (size_t)stages * STAGE_BYTES + 1024;  // + alignment slack
  auto kern = tc_qmm_kernel<BITS, MODE, ACT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  const int64_t sms = moe_host::sm_count();
  const int grid = (int)(max_tiles < sms ? max_tiles : sms);
  if (grid <= 0) return MOE_OK;
  kern<<<grid, kTcThreads, smem, st>>>(tmc, tma, p);
  return moe_host::launch_status();
}

}  // namespace

bool tc_available() { return encode_fn() != nullptr; }

moe_status_t tc_qmm(const void* act, int act_kind, const int32_t* sorted,
                    const int32_t* offsets, int T, int kmax, int E, int K, int n_rows,
                    bool swiglu, const uint32_t* wq, const uint16_t* ws, const uint16_t* wb,
                    int bits, void* out, int out_dtype, cudaStream_t st) {
  // act_kind: 0 = x bf16 [T, K] gathered by token, 2 = h bf16 [T*kmax, K] by sorted row
  if (act_kind != 0 && act_kind != 2) return MOE_ERR_UNSUPPORTED;
  if (K % BK != 0 || n_rows % 64 != 0) return MOE_ERR_INVALID_ARG;
  const bool gather = act_kind == 0;
  const int64_t A = (int64_t)T * kmax;
  if (A == 0) return MOE_OK;
  CUtensorMap tmc, tma;
  const uint64_t row_words = (uint64_t)K * bits / 32;
  if (!make_map_2d(&tmc, CU_TENSOR_MAP_DATA_TYPE_UINT32, wq, row_words, (uint64_t)E * n_rows,
                   row_words * 4, BK * bits / 32, BM, CU_TENSOR_MAP_SWIZZLE_NONE))
    return MOE_ERR_CUDA;
  if (gather) {
    if (!make_map_2d(&tma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, act, K, (uint64_t)T,
                     (uint64_t)K * 2, BK, 1, CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  } else {
    if (!make_map_2d(&tma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, act, K, (uint64_t)A,
                     (uint64_t)K * 2, BK, BN, CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  }
  TcParams p;
  p.sorted = sorted;
  p.offsets = offsets;
  p.ws = ws;
  p.wb = wb;
  p.out = out;
  p.out_dtype = out_dtype;
  p.kmax = kmax;
  p.E = E;
  p.K = K;
  p.n_rows = n_rows;
  p.n_out = swiglu ? n_rows / 2 : n_rows;
  p.n_mt = (p.n_out + BM - 1) / BM;
  p.stages = 2;
  p.err = moe_host::device_error_word();
  // upper bound of the tile count: every expert that can be active, plus one
  // partial n-tile each
  const int64_t max_active = A < E ? A : E;
  const int64_t max_tiles = (int64_t)p.n_mt * (max_active + (A + BN - 1) / BN);
  if (bits == 4) {
    if (swiglu) return gather ? launch_tc<4, kTcSwiglu, kTcGatherX>(tmc, tma, p, max_tiles, st)
                              : launch_tc<4, kTcSwiglu, kTcRowsH>(tmc, tma, p, max_tiles, st);
    return gather ? launch_tc<4, kTcRaw, kTcGatherX>(tmc, tma, p, max_tiles, st)
                  : launch_tc<4, kTcRaw, kTcRowsH>(tmc, tma, p, max_tiles, st);
  }
  if (swiglu) return gather ? launch_tc<8, kTcSwiglu, kTcGatherX>(tmc, tma, p, max_tiles, st)
                            : launch_tc<8, kTcSwiglu, kTcRowsH>(tmc, tma, p, max_tiles, st);
  return gather ? launch_tc<8, kTcRaw, kTcGatherX>(tmc, tma, p, max_tiles, st)
                : launch_tc<8, kTcRaw, kTcRowsH>(tmc, tma, p, max_tiles, st);
}

}  // namespace moe

// Grouped GEMM on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators, TMA-fed tiles): the prefill / batched path of the two
// quantized products.
//
// Page "oMLX MoE gate/up 融合优化：qwen35_moe_gate_up 实现剖析", 融合原理 and
// 实现剖析 ④ (one product with the [gate; up] matrix per expert, split, SiLU
// activation, down projection); page "Qwen3.5 Block在llama.cpp中的映射与优化
// 原理", section 4.2 (each expert only sees the tokens routed to it).
//
// Orientation: weights are the MMA's A operand (M = 128 rows), the expert's
// tokens are B (N = up to 256 tokens of its segment), K = the contraction
// axis, so D[m, n] lands in TMEM lane m, column n.
//   RAW tile:    A rows = 128 consecutive weight rows.
//   SWIGLU tile: A rows 0..63 = gate rows f0..f0+63, rows 64..127 = the up
//                rows of the same 64 features, so one accumulator holds both
//                halves of 64 outputs and TMEM (512 columns) still fits two
//                accumulators of 256 tokens for double buffering.
// A segment of m tokens is cut into ceil(m/256) tiles of equal size (rounded
// up to 16, the MMA's N granularity); the MMA's N is set per tile.  Each
// dequantized weight tile thus feeds up to 256 tokens, so the dequantization
// (CUDA cores) costs less than the MMA time it feeds.
//
// One CTA per SM, persistent over the tiles (active expert, m-tile, n-tile);
// n-tiles of the same weights are adjacent so neighbouring CTAs share them in
// L2.  Warp roles:
//   warp 5      loader: per k-block of 64, TMA loads the token tile: 4-row
//               gathers (tile::gather4) of the token rows of x, or 64-row 2D
//               boxes of rows already in sorted order (h, or x permuted),
//               128-byte swizzled as the MMA expects; all 32 lanes issue;
//   code warp   TMA-loads the packed codes of the tile's 128 rows,
//               128 bytes of each row per slot (4 k-blocks of 4-bit codes,
//               2 of 8-bit), two 64-row boxes with the 128-byte swizzle,
//               into a ring of 16 KB slots; bulk copies keep far more bytes
//               in flight than per-thread loads of 16-64 bytes per row could;
//   warps 6..   dequant (8 warps for 4-bit codes, 16 for 8-bit; the code
//               warp comes after them): each thread reads its row slice of
//               the codes from
//               the slot and loads the row's scale and bias into registers
//               a few A stages ahead, then w = s*q + b in fp32 (packed FMA),
//               rounds to bf16, writes the A tile in the 128-byte-swizzled
//               K-major layout, proxy fence, arrive;
//   warp 4      MMA: one thread issues tcgen05.mma (kind::f16, bf16 x bf16 ->
//               fp32) per 16-wide K slice, commits stage release and
//               accumulator completion to mbarriers;
//   warps 0-3   epilogue: tcgen05.ld of the accumulator, then raw fp32 stores
//               or SiLU(gate)*up (gate and up lanes sit in different warps:
//               warp pairs swap half of their columns through shared memory).
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

constexpr int BM = 128;        // accumulator rows = TMEM lanes
constexpr int BN = 256;        // most tokens per tile
constexpr int BK = 64;         // contraction per stage = one scale group = one 128-B swizzle atom
constexpr int kHalfRows = 64;  // SWIGLU: gate rows, then up rows, per A tile
constexpr int kBoxRows = 64;   // rows per 2D TMA box (codes and token rows)
constexpr int kEpiWarps = 4, kMmaWarp = 4, kLoadWarp = 5, kDeqWarp0 = 6;
// Dequant warps: 8 for 4-bit codes, 16 for 8-bit (twice the code bytes per
// weight to convert; measured: 16 warps speed up the 8-bit products and slow
// the 4-bit ones).  The code warp follows them.
__host__ __device__ constexpr int deq_warps(int bits) { return bits == 8 ? 16 : 8; }
__host__ __device__ constexpr int code_warp(int bits) { return kDeqWarp0 + deq_warps(bits); }
__host__ __device__ constexpr int tc_threads(int bits) { return (code_warp(bits) + 1) * 32; }
constexpr int kATileBytes = BM * BK * 2;                  // 16 KB bf16 weight tile
// k-blocks per A stage: each stage ends with a proxy fence and an arrival
// by every dequant thread, so two k-blocks per stage (measured on the
// prefill gate_up product: 308 us with two slots of two k-blocks, 392 us
// with three slots of one)
constexpr int kKbPerA = 2;
constexpr int kAStageBytes = kKbPerA * kATileBytes;       // 32 KB
constexpr int kBRowBytes = BK * 2;                         // one token row of a k-block
constexpr int kCodeRowBytes = 128;                         // code bytes of a row per code slot
constexpr int kCodeSlotBytes = BM * kCodeRowBytes;         // 16 KB
constexpr int kMaxCodeSlots = 8;
constexpr int kMaxStages = 8;
constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators of up to 256 columns
// A stages of scales and biases in flight per dequant thread (registers)
constexpr int kScaleLookahead = 4;

enum TcMode { kTcSwiglu = 0, kTcRaw = 1 };
enum TcAct { kTcGatherX = 0, kTcRowsH = 1 };

struct TcParams {
  const int32_t* sorted;   // sorted_assign (gate_up)
  const int32_t* offsets;  // [E+1]
  const uint32_t* wq;      // codes   [E, n_rows, K*bits/32]
  const uint16_t* ws;      // scales  [E, n_rows, K/64]
  const uint16_t* wb;      // biases
  void* out;
  int out_dtype;
  int kmax, E, K, n_rows, n_out;
  int a_stages;  // ring of dequantized weight stages (kKbPerA k-blocks each)
  int b_stages;  // ring of TMA-loaded token tiles (one k-block each)
  int c_stages;  // ring of TMA-loaded code slots (kCodeRowBytes of each row)
  int bn_cap;    // most tokens per tile (a multiple of 16, at most BN)
  int n_mt;         // m-tiles per expert
  KGate gate;       // k-gated launch (gate.k null: always runs)
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
// tcgen05.mma and tcgen05.commit are issued by one thread.  The MMA warp
// runs its loop converged (all lanes wait, walk the tiles and form the
// descriptors, which stay warp-uniform) and the lane that elect.sync picks,
// the lowest one every time, issues.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once all tcgen05 operations issued so far by the elected
// lane complete (the whole warp executes it, converged).
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
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

// Bounded wait whose outcome is the same in every lane of the warp (a wait
// that runs out in one lane counts as run out for all), so warp-collective
// instructions after it are never reached by part of a warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity,
                                          const volatile int* abort_flag) {
  const bool ok = mbar_wait_sleep(bar, parity, kWaitBudgetCycles) && *abort_flag == 0;
  return __all_sync(0xffffffffu, ok);
}

// Position in a ring of n stages: slot index and the parity of the current
// pass, advanced incrementally (no division in the pipelined loops).
struct Ring {
  int idx = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++idx == n) {
      idx = 0;
      phase ^= 1u;
    }
  }
};

// ---- tile schedule ----------------------------------------------------------

struct TileInfo {
  int e, seg_lo, mt;
  int tok0;  // first token of the tile within the segment
  int nv;    // tokens in the tile
  int nmma;  // MMA N: nv rounded up to 16
};

__device__ __forceinline__ int ntiles_of(int m, int cap) { return (m + cap - 1) / cap; }

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
  const int m = __ldg(p.offsets + ti.e + 1) - ti.seg_lo;
  const int nnt = ntiles_of(m, p.bn_cap);
  const int tsz = (((m + nnt - 1) / nnt) + 15) & ~15;  // <= bn_cap, and (nnt-1)*tsz < m
  const int local = t - tile_start[lo];
  ti.mt = local / nnt;
  const int nt = local - ti.mt * nnt;
  ti.tok0 = nt * tsz;
  ti.nv = min(tsz, m - ti.tok0);
  ti.nmma = (ti.nv + 15) & ~15;
  return ti;
}

// Weight row (within the expert) of A-tile row r of m-tile mt.
template <int MODE>
__device__ __forceinline__ int tile_weight_row(const TcParams& p, int mt, int r) {
  if (MODE == kTcSwiglu)
    return r < kHalfRows ? mt * kHalfRows + r : (p.n_rows >> 1) + mt * kHalfRows + r - kHalfRows;
  return mt * BM + r;
}

// One CTA per SM: 15 warps (4-bit) or 23 warps (8-bit) share the register
// file, so at most 128 or 88 registers per thread.
template <int BITS, int MODE, int ACT>
__global__ void __launch_bounds__(tc_threads(BITS), 1)
    tc_qmm_kernel(const __grid_constant__ CUtensorMap tm_act,
                  const __grid_constant__ CUtensorMap tm_codes, TcParams p) {
  if (k_gate_closed(p.gate.k, p.gate.lo, p.gate.hi, false)) return;
  // dequant work split: DQ_SLICES threads per A row, BK / DQ_SLICES codes of
  // each k-block each
  constexpr int kDeqWarps = deq_warps(BITS);
  constexpr int kCodeWarp = code_warp(BITS);
  constexpr int DQ_SLICES = kDeqWarps * 32 / BM;  // 2 | 4
  constexpr int DQ_CHUNKS = 8 / DQ_SLICES;        // 16-byte bf16 chunks per thread per k-block
  constexpr int KB_WORDS = BK * BITS / 32;         // code words of one row per k-block
  constexpr int CW = KB_WORDS / DQ_SLICES;         // code words per thread per k-block
  constexpr int KB_BYTES = BK * BITS / 8;          // code bytes of a row per k-block: 32 | 64
  constexpr int KPC = kCodeRowBytes / KB_BYTES;    // k-blocks per code slot: 4 | 2
  constexpr int PD = kScaleLookahead;              // A stages of scales in flight
  static_assert(CW * 4 == 8 || CW % 4 == 0, "a thread reads 8 bytes or whole 16-byte chunks");
  static_assert(KPC % kKbPerA == 0, "a code slot holds whole A stages");

  extern __shared__ __align__(1024) unsigned char tc_smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  // A ring (dequantized weights, kKbPerA k-blocks per stage): a_full arrived
  // by the dequant warps, a_empty committed by the MMAs.  B ring (token
  // tiles, one k-block per slot): b_full counts the TMA bytes, b_empty is
  // committed by the MMAs.  The MMA thread waits on both, so the dequant
  // warps run ahead of the token tiles and neither ring waits on the other.
  __shared__ uint64_t a_full[kMaxStages], a_empty[kMaxStages];
  __shared__ uint64_t b_full[kMaxStages], b_empty[kMaxStages];
  __shared__ uint64_t c_full[kMaxCodeSlots], c_empty[kMaxCodeSlots];
  __shared__ uint64_t tmem_full[2], tmem_empty[2];
  __shared__ uint64_t xfull[2][2][2];  // SWIGLU exchange: [pair][buffer][writer half]
  __shared__ uint64_t drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int act_e[1024];
  __shared__ int tile_start[1025];
  __shared__ int n_act_sh;
  __shared__ float xbuf[MODE == kTcSwiglu ? 2 * 2 * 2 * 16 * 32 : 1];
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int SA = p.a_stages, SB = p.b_stages, SC = p.c_stages;
  const int nkb = p.K / BK;
  const int nas = (nkb + kKbPerA - 1) / kKbPerA;  // A stages per tile

  // ---- set-up: barriers, TMEM, active experts and their tile ranges ----
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < SA; ++s) {
      mbar_init(&a_full[s], kDeqWarps);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int s = 0; s < SC; ++s) {
      mbar_init(&c_full[s], 1);
      mbar_init(&c_empty[s], kDeqWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], kEpiWarps);
    }
    for (int i = 0; i < 8; ++i) mbar_init(&xfull[i >> 2][(i >> 1) & 1][i & 1], 1);
    mbar_init(&drain_bar, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  // the set-up above overlaps the end of the previous kernel of the stream
  pdl_wait();
  pdl_trigger();
  // tiles of each expert, all threads at once (tile_start[e] holds expert
  // e's count), then one warp compacts the active experts in id order with
  // their first tiles (an active entry a <= e is written only after the
  // warp has read the counts of its 32 experts)
  for (int e = tid; e < p.E; e += blockDim.x) {
    const int m = __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
    tile_start[e] = m > 0 ? p.n_mt * ntiles_of(m, p.bn_cap) : 0;
  }
  __syncthreads();
  if (warp == 0) {
    int n = 0, t = 0;
    for (int base = 0; base < p.E; base += 32) {
      const int e = base + lane;
      const int c = e < p.E ? tile_start[e] : 0;
      __syncwarp();
      const unsigned act = __ballot_sync(0xFFFFFFFFu, c > 0);
      int incl = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += y;
      }
      if (c > 0) {
        const int a = n + __popc(act & lanemask_lt());
        act_e[a] = e;
        tile_start[a] = t + incl - c;
      }
      n += __popc(act);
      t += __shfl_sync(0xFFFFFFFFu, incl, 31);
      __syncwarp();
    }
    if (lane == 0) {
      tile_start[n] = t;
      n_act_sh = n;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;
  const int n_act = n_act_sh;
  const int n_tiles = n_act > 0 ? tile_start[n_act] : 0;

  const int b_tile_bytes = p.bn_cap * kBRowBytes;
  unsigned char* a_base = smem;                                     // SA * kAStageBytes
  unsigned char* c_base = smem + (size_t)SA * kAStageBytes;         // SC * kCodeSlotBytes
  unsigned char* b_base = c_base + (size_t)SC * kCodeSlotBytes;     // SB * b_tile_bytes
  // k-block h of A stage s: a 128 x 64 K-major SW128 tile
  auto stage_a = [&](int s, int h) { return a_base + (size_t)s * kAStageBytes + h * kATileBytes; };
  auto stage_b = [&](int s) { return b_base + (size_t)s * b_tile_bytes; };
  auto stage_c = [&](int s) { return c_base + (size_t)s * kCodeSlotBytes; };

  if (warp == kLoadWarp) {
    // =============================== loader ===============================
    int64_t issued = 0;
    Ring ring;  // B ring
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      const TileInfo ti = tile_info(p, act_e, tile_start, n_act, t);
      // this lane's gathers: groups g = lane and lane + 32 of 4 token rows
      // (columns past the tile repeat its first token)
      const int ngroups = ti.nmma / 4;
      int tok[8];
      if (ACT == kTcGatherX) {
        const int first = ti.seg_lo + ti.tok0;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int n = 4 * (lane + 32 * h) + i;
            tok[4 * h + i] = __ldg(p.sorted + first + (n < ti.nv ? n : 0)) / p.kmax;
          }
      }
      const int nbox = (ti.nmma + kBoxRows - 1) / kBoxRows;
      const uint32_t bytes = ACT == kTcGatherX ? (uint32_t)ti.nmma * (BK * 2)
                                               : (uint32_t)nbox * (kBoxRows * BK * 2);
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = ring.idx;
        if (!warp_wait(&b_empty[s], ring.phase ^ 1u, &abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&b_full[s], bytes);
        __syncwarp();
        if (ACT == kTcGatherX) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int g = lane + 32 * h;
            if (g < ngroups)
              tma_gather4(stage_b(s) + g * 4 * (BK * 2), &tm_act, kb * BK, tok[4 * h],
                          tok[4 * h + 1], tok[4 * h + 2], tok[4 * h + 3], &b_full[s]);
          }
        } else if (lane < nbox) {
          tma_load_2d(stage_b(s) + lane * (kBoxRows * BK * 2), &tm_act, kb * BK,
                      ti.seg_lo + ti.tok0 + lane * kBoxRows, &b_full[s]);
        }
        __syncwarp();
        ++issued;
        ring.next(SB);
      }
    }
    if (!ok && lane == 0) {
      raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
      abort_flag = 1;
      // the last min(issued, SB) slots may still have copies in flight
      Ring r = ring;
      for (int64_t j = 0; j < issued && j < SB; ++j) {
        r.idx = r.idx == 0 ? SB - 1 : r.idx - 1;
        if (r.idx == SB - 1) r.phase ^= 1u;
        mbar_wait(&b_full[r.idx], r.phase, kWaitBudgetCycles);
      }
    }
  } else if (warp == kCodeWarp) {
    // ============================== code loader ==============================
    // per tile: ceil(nkb / KPC) slots, each the next kCodeRowBytes of the
    // tile's 128 rows (A rows 0-63 and 64-127 as two 64-row boxes; rows past
    // the matrix come back zero, rows of the next expert are never stored)
    int64_t issued = 0;
    Ring ring;  // code ring
    bool ok = true;
    const int nslot = (nkb + KPC - 1) / KPC;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      const TileInfo ti = tile_info(p, act_e, tile_start, n_act, t);
      const int r0 = tile_weight_row<MODE>(p, ti.mt, 0);
      const int r1 = tile_weight_row<MODE>(p, ti.mt, kHalfRows);
      const int g0 = ti.e * p.n_rows;  // E * n_rows < 2^31 (checked on the host)
      for (int c = 0; c < nslot; ++c) {
        const int sc = ring.idx;
        if (!warp_wait(&c_empty[sc], ring.phase ^ 1u, &abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&c_full[sc], (uint32_t)kCodeSlotBytes);
          tma_load_2d(stage_c(sc), &tm_codes, c * kCodeRowBytes, g0 + r0, &c_full[sc]);
          tma_load_2d(stage_c(sc) + kHalfRows * kCodeRowBytes, &tm_codes, c * kCodeRowBytes,
                      g0 + r1, &c_full[sc]);
        }
        __syncwarp();
        ++issued;
        ring.next(SC);
      }
    }
    if (!ok && lane == 0) {
      raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
      abort_flag = 1;
      // the last min(issued, SC) slots may still have copies in flight
      Ring r = ring;
      for (int64_t j = 0; j < issued && j < SC; ++j) {
        r.idx = r.idx == 0 ? SC - 1 : r.idx - 1;
        if (r.idx == SC - 1) r.phase ^= 1u;
        mbar_wait(&c_full[r.idx], r.phase, kWaitBudgetCycles);
      }
    }
  } else if (warp >= kDeqWarp0) {
    // =============================== dequant ===============================
    const int dt = tid - kDeqWarp0 * 32;
    const int r = dt / DQ_SLICES;                  // A-tile row 0 .. 127
    const int slice = dt % DQ_SLICES;
    const int c0 = slice * DQ_CHUNKS;              // first 16-byte bf16 chunk of this thread
    const int ngroups = p.K / 64;
    // this CTA's A stages in order, (its tiles) x (A stages of the tile); the
    // scales and biases of A stage st + PD are loaded while stage st is
    // converted; the codes come from the code ring
    const int my_tiles = blockIdx.x < n_tiles ? (n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int nst = my_tiles * nas;  // < 2^31: tiles and k-blocks are bounded by int sizes
    struct Ahead {
      uint32_t sb[kKbPerA];   // scale | bias << 16 of each k-block
      int nkb;                // k-blocks in the stage (the last of a tile may have fewer)
    };
    int la_t = blockIdx.x, la_kb = 0;
    const uint16_t* la_sp = nullptr;
    const uint16_t* la_bp = nullptr;
    auto la_fetch = [&](Ahead& d) {
      if (la_t >= n_tiles) {
        d.nkb = 0;
#pragma unroll
        for (int h = 0; h < kKbPerA; ++h) d.sb[h] = 0u;
        return;
      }
      if (la_kb == 0) {
        const TileInfo ti = tile_info(p, act_e, tile_start, n_act, la_t);
        int wrow = tile_weight_row<MODE>(p, ti.mt, r);
        if (wrow >= p.n_rows) wrow = p.n_rows - 1;  // rows past the matrix: any valid row
        const int64_t grow = (int64_t)ti.e * p.n_rows + wrow;
        la_sp = p.ws + grow * ngroups;
        la_bp = p.wb + grow * ngroups;
      }
      d.nkb = min(kKbPerA, nkb - la_kb);
#pragma unroll
      for (int h = 0; h < kKbPerA; ++h) {
        const int kb = h < d.nkb ? la_kb + h : la_kb;  // a missing second k-block repeats the first
        d.sb[h] = (uint32_t)__ldg(la_sp + kb) | ((uint32_t)__ldg(la_bp + kb) << 16);
      }
      la_kb += d.nkb;
      if (la_kb == nkb) {
        la_kb = 0;
        la_t += gridDim.x;
      }
    };
    // the ring is indexed by the unrolled position u, so each slot keeps its
    // own registers while its loads are in flight
    Ahead ahead[PD];
#pragma unroll
    for (int i = 0; i < PD; ++i) la_fetch(ahead[i]);
    // this thread's CW code words of k-block j of a code slot: row r, bytes
    // j * KB_BYTES + slice * CW * 4 on, 16-byte chunks 128-byte swizzled
    auto load_codes = [&](const unsigned char* slot, int j, uint32_t (&w)[CW]) {
      const int byte0 = j * KB_BYTES + slice * CW * 4;
      const unsigned char* row = slot + r * kCodeRowBytes;
      if constexpr (CW * 4 >= 16) {
#pragma unroll
        for (int v = 0; v < CW / 4; ++v) {
          const int ch = byte0 / 16 + v;
          const uint4 t = *reinterpret_cast<const uint4*>(row + ((ch ^ (r & 7)) << 4));
          w[4 * v] = t.x;
          w[4 * v + 1] = t.y;
          w[4 * v + 2] = t.z;
          w[4 * v + 3] = t.w;
        }
      } else {
        const int ch = byte0 / 16;
        const uint2 t = *reinterpret_cast<const uint2*>(row + ((ch ^ (r & 7)) << 4) + (byte0 & 15));
        w[0] = t.x;
        w[1] = t.y;
      }
    };

    Ring ra, rc;  // A ring, code ring
    int akb = 0;      // k-block (within the tile) of the next A stage
    bool ok = true;
    for (int st0 = 0; st0 < nst && ok; st0 += PD) {
#pragma unroll
      for (int u = 0; u < PD; ++u) {
        if (st0 + u < nst && ok) {
          const Ahead sbc = ahead[u];
          la_fetch(ahead[u]);
          // the stage's codes: a new slot starts every KPC k-blocks
          if (akb % KPC == 0 && !warp_wait(&c_full[rc.idx], rc.phase, &abort_flag)) {
            ok = false;
            break;
          }
          struct {
            uint32_t q[kKbPerA][CW];
            uint32_t sb[kKbPerA];
            int nkb;
          } cur;
          const unsigned char* cslot = stage_c(rc.idx);
#pragma unroll
          for (int h = 0; h < kKbPerA; ++h) {
            cur.sb[h] = sbc.sb[h];
            if (h < sbc.nkb) {
              load_codes(cslot, (akb + h) % KPC, cur.q[h]);
            } else {
#pragma unroll
              for (int v = 0; v < CW; ++v) cur.q[h][v] = 0u;
            }
          }
          cur.nkb = sbc.nkb;
          const int sa = ra.idx;
          {
            if (!warp_wait(&a_empty[sa], ra.phase ^ 1u, &abort_flag)) ok = false;
          }
          if (ok) {
#pragma unroll
            for (int h = 0; h < kKbPerA; ++h) {
              if (h < cur.nkb) {
                const float sc = __half2float(__ushort_as_half((uint16_t)(cur.sb[h] & 0xFFFFu)));
                const float bi = __half2float(__ushort_as_half((uint16_t)(cur.sb[h] >> 16)));
                unsigned char* atile = stage_a(sa, h);
                if (BITS == 4) {
                  // one 32-bit word = 8 codes = one 16-byte bf16 chunk
                  const float2 mul = make_float2(512.0f * sc, 32.0f * sc);
                  const float2 add = make_float2(bi - 512.0f * sc, bi - 32.0f * sc);
#pragma unroll
                  for (int i = 0; i < DQ_CHUNKS; ++i) {
                    const uint32_t v = cur.q[h][i];
                    const uint32_t sh[4] = {v << 14, v << 6, v >> 2, v >> 10};
                    uint32_t o[4];
#pragma unroll
                    for (int pq = 0; pq < 4; ++pq) {
                      // (1 + q_even/512, 1 + q_odd/32), then w = s*q + b in fp32
                      const float2 f =
                          make_float2(__uint_as_float((sh[pq] & 0x0003C000u) | 0x3F800000u),
                                      __uint_as_float((sh[pq] & 0x003C0000u) | 0x3F800000u));
                      const float2 w = __ffma2_rn(f, mul, add);
                      o[pq] = pack_bf16x2(w.x, w.y);
                    }
                    *reinterpret_cast<uint4*>(atile + sw128_offset(r, c0 + i)) =
                        make_uint4(o[0], o[1], o[2], o[3]);
                  }
                } else {
                  // one 32-bit word = 4 codes; two words = one 16-byte bf16 chunk
                  const float2 mul = make_float2(256.0f * sc, 256.0f * sc);
                  const float2 add = make_float2(bi - 256.0f * sc, bi - 256.0f * sc);
#pragma unroll
                  for (int i = 0; i < DQ_CHUNKS; i += 2) {
                    const uint32_t wv[4] = {cur.q[h][2 * i], cur.q[h][2 * i + 1], cur.q[h][2 * i + 2],
                                            cur.q[h][2 * i + 3]};
                    uint32_t o[8];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                      const uint32_t v = wv[jj];
                      const float2 f0 = make_float2(__uint_as_float(((v << 15) & 0x007F8000u) | 0x3F800000u),
                                                    __uint_as_float(((v << 7) & 0x007F8000u) | 0x3F800000u));
                      const float2 f1 = make_float2(__uint_as_float(((v >> 1) & 0x007F8000u) | 0x3F800000u),
                                                    __uint_as_float(((v >> 9) & 0x007F8000u) | 0x3F800000u));
                      const float2 w0 = __ffma2_rn(f0, mul, add);
                      const float2 w1 = __ffma2_rn(f1, mul, add);
                      o[2 * jj] = pack_bf16x2(w0.x, w0.y);
                      o[2 * jj + 1] = pack_bf16x2(w1.x, w1.y);
                    }
                    *reinterpret_cast<uint4*>(atile + sw128_offset(r, c0 + i)) =
                        make_uint4(o[0], o[1], o[2], o[3]);
                    *reinterpret_cast<uint4*>(atile + sw128_offset(r, c0 + i + 1)) =
                        make_uint4(o[4], o[5], o[6], o[7]);
                  }
                }
              }
            }
            fence_proxy_async_smem();
            // the code slot is released once its last k-block is converted
            akb += cur.nkb;
            const bool tile_end = akb == nkb;
            if (akb % KPC == 0 || tile_end) {
              __syncwarp();
              if (lane == 0) mbar_arrive(&c_empty[rc.idx]);
              rc.next(SC);
            }
            if (tile_end) akb = 0;
            if (lane == 0) mbar_arrive(&a_full[sa]);
            ra.next(SA);
          }
        }
      }
    }
    if (!ok && lane == 0) {
      raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
      abort_flag = 1;
    }
  } else if (warp == kMmaWarp) {
    // ================================= MMA =================================
    // the whole warp, converged; every wait's outcome is agreed by the warp
    int64_t it = 0;
    Ring ra, rb;  // A ring, B ring
    int j = 0;
    bool ok = true;
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      const bool got = mbar_wait_sleep(bar, parity, kWaitBudgetCycles);
      return __all_sync(0xFFFFFFFFu, got);
    };
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++j) {
      const TileInfo ti = tile_info(p, act_e, tile_start, n_act, t);
      const uint32_t idesc = idesc_bf16(BM, ti.nmma);
      const int buf = j & 1;
      {
        if (!wait_all(&tmem_empty[buf], (uint32_t)(((j >> 1) & 1) ^ 1))) ok = false;
      }
      if (__any_sync(0xFFFFFFFFu, !ok || abort_flag != 0)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d0 = tmem_base + (uint32_t)(buf * BN);
      for (int as = 0, kb = 0; as < nas; ++as, ra.next(SA)) {
        const int sa = ra.idx;
        {
          if (!wait_all(&a_full[sa], ra.phase)) ok = false;
        }
        if (!ok) break;
        // operand visibility: the dequant writers' proxy fence and release
        // arrivals acquired by the wait above; the token tile's TMA
        // transaction count by the wait below
#pragma unroll
        for (int h = 0; h < kKbPerA; ++h) {
          if (kb < nkb && (h == 0 || as * kKbPerA + h < nkb)) {
            {
              if (!wait_all(&b_full[rb.idx], rb.phase)) ok = false;
            }
            if (!ok) break;
            const uint64_t adesc = smem_desc_sw128(stage_a(sa, h));
            const uint64_t bdesc = smem_desc_sw128(stage_b(rb.idx));
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)  // K advance in the swizzle atom: 32 bytes
              umma_bf16(d0, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
            umma_commit(&b_empty[rb.idx]);
            rb.next(SB);
            ++kb;
            ++it;
          }
        }
        if (!ok) break;
        umma_commit(&a_empty[sa]);
      }
      if (!ok) break;
      umma_commit(&tmem_full[buf]);
    }
    if (!ok && lane == 0) {
      raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
      abort_flag = 1;
    }
    // wait for the warp's last MMAs before TMEM is released (a commit with
    // no MMA issued before it is not relied on to arrive)
    if (it > 0) {
      umma_commit(&drain_bar);
      mbar_wait(&drain_bar, 0, kWaitBudgetCycles);
    }
    __syncwarp();
  } else {
    // =============================== epilogue ===============================
    int j = 0;
    uint32_t xs = 0;  // SWIGLU exchange steps so far
    bool ok = true;
    const int pair = warp & 1, hi = warp >> 1;  // SWIGLU: hi = 0 holds gate lanes, 1 up lanes
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++j) {
      const TileInfo ti = tile_info(p, act_e, tile_start, n_act, t);
      const int buf = j & 1;
      {
        if (!warp_wait(&tmem_full[buf], (uint32_t)((j >> 1) & 1), &abort_flag)) ok = false;
      }
      if (!ok) break;
      tc_fence_after();
      const int64_t row0 = (int64_t)ti.seg_lo + ti.tok0;  // output row of tile column 0
      const uint32_t lane_addr =
          tmem_base + ((uint32_t)(warp * 32) << 16) + (uint32_t)(buf * BN);
      if (MODE == kTcRaw) {
        const int col = ti.mt * BM + warp * 32 + lane;
        const bool col_ok = col < p.n_out;
        const int64_t stride = p.n_out;
        const bool bf16_out = p.out_dtype == MOE_DTYPE_BF16;
        // element (row n0 + i, col) of the output, fp32 or rounded to bf16
        auto put = [&](int64_t oi, uint32_t v) {
          if (bf16_out)
            static_cast<uint16_t*>(p.out)[oi] = f32_to_bf16_rne(__uint_as_float(v));
          else
            static_cast<float*>(p.out)[oi] = __uint_as_float(v);
        };
        for (int n0 = 0; n0 < ti.nv; n0 += 32) {
          uint32_t a[16], b[16];
          tmem_ld16(lane_addr + n0, a);
          tmem_ld16(lane_addr + n0 + 16, b);
          tmem_ld_wait();
          if (col_ok) {
            const int64_t o0 = (row0 + n0) * stride + col;
            if (n0 + 32 <= ti.nv) {
#pragma unroll
              for (int i = 0; i < 16; ++i) put(o0 + i * stride, a[i]);
#pragma unroll
              for (int i = 0; i < 16; ++i) put(o0 + (16 + i) * stride, b[i]);
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i)
                if (n0 + i < ti.nv) put(o0 + i * stride, a[i]);
#pragma unroll
              for (int i = 0; i < 16; ++i)
                if (n0 + 16 + i < ti.nv) put(o0 + (16 + i) * stride, b[i]);
            }
          }
        }
      } else {
        // gate lane f (warp pair, hi = 0) and up lane f (hi = 1) hold the two
        // halves of feature f.  Per step both load two 16-column chunks; the
        // gate warp finishes the first chunk, the up warp the second, each
        // after receiving the partner's half of it through shared memory
        // (double-buffered: a buffer is rewritten only after the partner's
        // next arrival, which follows its reads).
        const int f = ti.mt * kHalfRows + pair * 32 + lane;
        const bool f_ok = f < p.n_out;
        for (int c = 0; c * 16 < ti.nv; c += 2, ++xs) {
          uint32_t a[16], b[16];
          tmem_ld16(lane_addr + c * 16, a);
          tmem_ld16(lane_addr + c * 16 + 16, b);
          tmem_ld_wait();
          const int xb = (int)(xs & 1u);
          float* mine = xbuf + ((pair * 2 + xb) * 2 + hi) * (16 * 32);
          const float* theirs = xbuf + ((pair * 2 + xb) * 2 + (hi ^ 1)) * (16 * 32);
#pragma unroll
          for (int i = 0; i < 16; ++i) mine[i * 32 + lane] = __uint_as_float(hi == 0 ? b[i] : a[i]);
          __syncwarp();
          if (lane == 0) mbar_arrive(&xfull[pair][xb][hi]);
          if (!warp_wait(&xfull[pair][xb][hi ^ 1], (xs >> 1) & 1u, &abort_flag)) {
            ok = false;
            break;
          }
          const int chunk = c + hi;
          if (f_ok) {
            const int64_t stride = p.n_out;
            const int64_t first = (row0 + chunk * 16) * stride + f;
            const int nrem = ti.nv - chunk * 16;  // valid rows of this chunk (may be <= 0)
            float hv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float other = theirs[i * 32 + lane];
              const float g = hi == 0 ? __uint_as_float(a[i]) : other;
              const float u = hi == 0 ? other : __uint_as_float(b[i]);
              hv[i] = swiglu_f32(g, u);
            }
            if (p.out_dtype == MOE_DTYPE_BF16) {
              uint16_t* q = static_cast<uint16_t*>(p.out) + first;
#pragma unroll
              for (int i = 0; i < 16; ++i, q += stride)
                if (i < nrem) *q = f32_to_bf16_rne(hv[i]);
            } else {
              float* q = static_cast<float*>(p.out) + first;
#pragma unroll
              for (int i = 0; i < 16; ++i, q += stride)
                if (i < nrem) *q = hv[i];
            }
          }
          __syncwarp();
        }
        if (!ok) break;
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
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, kTmemCols);
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
moe_status_t launch_tc(const CUtensorMap& tma, const CUtensorMap& tmc, TcParams p,
                       int64_t max_tiles, cudaStream_t st) {
  auto kern = tc_qmm_kernel<BITS, MODE, ACT>;
  // opt-in shared memory left beside the static part
  static const long avail = [kern] {
    cudaFuncAttributes fa;
    int dev = 0, optin = 0;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
      return 0L;
    return (long)optin - (long)fa.sharedSizeBytes - 1024;
  }();
  // ring depths: two A stages, code slots for about 8 k-blocks, and as many
  // token-tile slots as fit (fewer code slots, down to 2, while fewer than 4
  // token tiles fit: each token tile is in flight from its TMA issue to the
  // end of its MMAs, so their count sets how many k-blocks overlap)
  const long b_tile = (long)p.bn_cap * kBRowBytes;
  const long kpc = kCodeRowBytes / (BK * BITS / 8);
  const long a_stages = 2;
  long c_stages = (8 + kpc - 1) / kpc;
  if (c_stages < 2) c_stages = 2;
  auto fit_b = [&] { return (avail - a_stages * kAStageBytes - c_stages * kCodeSlotBytes) / b_tile; };
  long b_stages = fit_b();
  while (b_stages < 4 && c_stages > 2) {
    --c_stages;
    b_stages = fit_b();
  }
  if (b_stages > kMaxStages) b_stages = kMaxStages;
  if (b_stages < 2) return MOE_ERR_UNSUPPORTED;
  p.a_stages = (int)a_stages;
  p.b_stages = (int)b_stages;
  p.c_stages = (int)c_stages;
  const size_t smem = (size_t)a_stages * kAStageBytes + (size_t)c_stages * kCodeSlotBytes +
                      (size_t)b_stages * b_tile + 1024;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  const int64_t sms = moe_host::sm_count();
  const int grid = (int)(max_tiles < sms ? max_tiles : sms);
  if (grid <= 0) return MOE_OK;
  return moe_host::launch(kern, grid, tc_threads(BITS), smem, st, tma, tmc, p);
}

}  // namespace

bool tc_available() { return encode_fn() != nullptr; }

// 2D tensor map for other kernels of the library (the small-batch path).
bool make_tensor_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                        uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                        CUtensorMapSwizzle sw) {
  return make_map_2d(m, dt, base, inner, outer, row_bytes, box_inner, box_outer, sw);
}

// 3D tensor map (the streamed GEMV's code boxes); strides in bytes of dims 1, 2.
bool make_tensor_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base,
                        const uint64_t (&dims)[3], const uint64_t (&strides)[2],
                        const uint32_t (&box)[3], CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  const cuuint64_t str[2] = {strides[0], strides[1]};
  const cuuint32_t bx[3] = {box[0], box[1], box[2]};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), d, str, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

moe_status_t tc_qmm(const void* act, int act_kind, const int32_t* sorted,
                    const int32_t* offsets, int T, int kmax, int E, int K, int n_rows,
                    bool swiglu, const uint32_t* wq, const uint16_t* ws, const uint16_t* wb,
                    int bits, void* out, int out_dtype, KGate gate, cudaStream_t st) {
  // act_kind: 0 = x bf16 [T, K] gathered by token, 2 = h bf16 [T*kmax, K] by sorted row
  if (act_kind != 0 && act_kind != 2) return MOE_ERR_UNSUPPORTED;
  if (K % BK != 0 || n_rows % 64 != 0) return MOE_ERR_INVALID_ARG;
  if ((int64_t)K * bits / 8 < kCodeRowBytes) return MOE_ERR_UNSUPPORTED;  // one code box per row
  if (E > 1024) return MOE_ERR_UNSUPPORTED;
  const bool gather = act_kind == 0;
  const int64_t A = (int64_t)T * kmax;
  if (A == 0) return MOE_OK;
  CUtensorMap tma;
  if (gather) {
    if (!make_map_2d(&tma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, act, K, (uint64_t)T,
                     (uint64_t)K * 2, BK, 1, CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  } else {
    if (!make_map_2d(&tma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, act, K, (uint64_t)A,
                     (uint64_t)K * 2, BK, kBoxRows, CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  }
  TcParams p;
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
  p.n_mt = swiglu ? (p.n_out + kHalfRows - 1) / kHalfRows : (p.n_out + BM - 1) / BM;
  p.a_stages = 2;
  p.b_stages = 2;
  p.c_stages = 2;
  // tokens per tile: near the mean segment length, so that a weight tile is
  // dequantized about once per expert while small segments keep small token
  // tiles (more token-tile slots fit)
  const int64_t mean = A / E;
  p.bn_cap = mean <= 32 ? 64 : (mean <= 64 ? 128 : BN);
  p.gate = gate;
  p.err = moe_host::device_error_word();
  // codes: [E * n_rows rows][K * bits / 8 bytes], 64-row boxes of 128 bytes
  if ((int64_t)E * n_rows >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  const uint64_t row_bytes = (uint64_t)K * bits / 8;
  CUtensorMap tmc;
  if (!make_map_2d(&tmc, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, row_bytes, (uint64_t)E * n_rows,
                   row_bytes, kCodeRowBytes, kHalfRows, CU_TENSOR_MAP_SWIZZLE_128B))
    return MOE_ERR_CUDA;
  // upper bound of the tile count: every expert that can be active, plus one
  // partial n-tile each
  const int64_t max_active = A < E ? A : E;
  const int64_t max_tiles = (int64_t)p.n_mt * (max_active + (A + p.bn_cap - 1) / p.bn_cap);
  if (bits == 4) {
    if (swiglu) return gather ? launch_tc<4, kTcSwiglu, kTcGatherX>(tma, tmc, p, max_tiles, st)
                              : launch_tc<4, kTcSwiglu, kTcRowsH>(tma, tmc, p, max_tiles, st);
    return gather ? launch_tc<4, kTcRaw, kTcGatherX>(tma, tmc, p, max_tiles, st)
                  : launch_tc<4, kTcRaw, kTcRowsH>(tma, tmc, p, max_tiles, st);
  }
  if (swiglu) return gather ? launch_tc<8, kTcSwiglu, kTcGatherX>(tma, tmc, p, max_tiles, st)
                            : launch_tc<8, kTcSwiglu, kTcRowsH>(tma, tmc, p, max_tiles, st);
  return gather ? launch_tc<8, kTcRaw, kTcGatherX>(tma, tmc, p, max_tiles, st)
                : launch_tc<8, kTcRaw, kTcRowsH>(tma, tmc, p, max_tiles, st);
}

}  // namespace moe

// Grouped GEMM for few tokens per expert (decode, small batches) on the
// 5th-generation tensor cores, with the packed codes in tensor memory.
//
// Page "oMLX MoE gate/up 融合优化：qwen35_moe_gate_up 实现剖析", 融合原理 and
// 实现剖析 ④ (one product with the [gate; up] matrix per expert, split, SiLU
// activation, down projection); page "Qwen3.5 Block在llama.cpp中的映射与优化
// 原理", section 4.2 (only the routed experts' weights are read).
//
// Per group of 64 elements of a weight row (scale s, bias b):
//   sum_i x_i (s q_i + b) = s * (sum_i (128 + q_i) x_i - 128 X) + b * X,
// X = sum_i x_i.  The tensor cores compute P = sum_i (128 + q_i) x_i with
// the codes as they are: one shift and one LOP3 turn two codes of a word
// into a bf16 pair (128 + q_j, 128 + q_{j+4}) (exact), written straight into
// tensor memory, which is the MMA's A operand (no shared-memory round trip
// for the weights).  Each group's P lands in its own accumulator columns;
// CUDA cores apply s and b per group and sum the groups in order.  8-bit
// codes are read as two 4-bit codes (low, high) against (x, 16 x) (exact in
// bf16), i.e. twice the contraction length with X' = 17 X.
//
// Tile: 128 weight rows x up to 16 tokens of one expert's segment.  The
// MMA's K order inside each 8-nibble word is (j, j+4) for j = 0..3; the
// token tile is staged in that same order.  SWIGLU tiles interleave, in each
// 32-lane quarter, 16 gate rows and the 16 up rows of the same features, so
// the activation needs one warp shuffle.
//
// Warp roles (one CTA per SM, persistent over the tiles):
//   warp 6      codes: TMA copies of each k-block's 128 rows x 32 bytes
//               into a 16-slot shared-memory ring (eight 16-row boxes);
//   warps 8-15  convert: lane = weight row (warp % 4 selects the lane
//               quarter it may write), even / odd k-blocks by warp half;
//               codes from the ring become bf16 pairs, tcgen05.st into the
//               A slot of the stage ring;
//   warp 7      tokens: stages the tile's tokens per k-block (plain loads
//               issued for 8 k-blocks at once, reordered, 128-byte swizzle)
//               into the B slot of the stage ring;
//   warps 4-5   MMA: tcgen05.mma kind::f16, A from tensor memory, B from
//               shared memory, one accumulator region per group; warp 4
//               takes the even groups, warp 5 the odd ones, so the tensor
//               pipe stays fed while one of them waits;
//   warps 0-3   epilogue: per-group X sums of the tile, then per group
//               acc += s (P - 128 m X) + b X, activation and stores.
// Every wait is bounded; a wait that runs out sets MOE_DEVERR_TIMEOUT and
// the CTA drains what is in flight and frees its tensor memory.
#include <cuda.h>
#include <cuda_fp16.h>

#include "async.cuh"
#include "common.cuh"

// Optional per-role cycle accounting (compiled in only with -DMOE_TCS_TRACE).
#ifdef MOE_TCS_TRACE
__device__ unsigned long long g_tcs_trace[16];
#define TCS_T0() const long long tcs_t0_ = clock64()
#define TCS_ACC(var) var += clock64() - tcs_t0_
#define TCS_FLUSH(slot, var) atomicAdd(&g_tcs_trace[slot], (unsigned long long)(var))
#else
#define TCS_T0()
#define TCS_ACC(var)
#define TCS_FLUSH(slot, var) ((void)(var))
#endif

namespace moe {
bool make_tensor_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                        uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                        CUtensorMapSwizzle sw);
bool tc_available();
namespace {

constexpr int kSmEpiWarps = 4, kSmMmaWarp0 = 4, kSmMmaWarps = 2, kSmCodeWarp = 6, kSmStageWarp = 7;
constexpr int kSmConvWarp0 = 8, kSmConvWarps = 8;
constexpr int kSmThreads = (kSmConvWarp0 + kSmConvWarps) * 32;  // 512
constexpr int kSmBM = 128;       // weight rows per tile = TMEM lanes
constexpr int kSmBN = 16;        // tokens per tile (MMA N)
constexpr int kSmCells = 32;     // A cells (bf16 pairs) per row per k-block = 64 nibbles
constexpr int kSmS = 8;          // stage ring: A slot (TMEM columns 32 s ..) + B slot (smem)
constexpr int kSmSC = 16;        // codes ring (shared memory), 128 rows x 32 B per slot
constexpr int kSmCSlotBytes = kSmBM * 32;
constexpr int kSmStageBatch = 8; // k-blocks whose token values are loaded together
constexpr int kSmGC = 8;         // groups per accumulator chunk
constexpr int kSmAccCol0 = 256;  // accumulators: two chunks of kSmGC x 16 columns
constexpr int kSmBSlotBytes = kSmBN * 128;
constexpr uint32_t kSmTmemCols = 512;

enum SmMode { kSmSwiglu = 0, kSmRaw = 1 };

struct SmParams {
  const uint16_t* act;     // x [T, K] (kind 0) or rows in sorted order [A, K] (kind 2), bf16
  int act_kind;
  const int32_t* sorted;   // sorted_assign (kind 0)
  const int32_t* offsets;  // [E+1]
  const uint32_t* wq;      // codes [E, n_rows, K*bits/32]
  const uint16_t* ws;      // scales [E, n_rows, K/64]
  const uint16_t* wb;
  void* out;
  int out_dtype;
  int kmax, E, K, n_rows, n_out, n_mt;
  unsigned int* err;
};

__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit_sm(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_sm(void* dst, const CUtensorMap* tm, int c0, int c1,
                                               uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem_sm() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before_sm() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sm() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld16_sm(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait_sm() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ uint64_t smem_desc_sw128_sm(const void* p) {
  const uint64_t addr = smem_u32(p);
  uint64_t d = (addr >> 4) & 0x3FFFull;
  d |= 1ull << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}
__device__ __forceinline__ uint32_t sw128_off_sm(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// Bounded wait with one outcome for the whole warp.
__device__ __forceinline__ bool sm_warp_wait(uint64_t* bar, uint32_t parity,
                                             const volatile int* abort_flag) {
  const bool ok = mbar_wait_sleep(bar, parity, kWaitBudgetCycles) && *abort_flag == 0;
  return __all_sync(0xffffffffu, ok);
}

struct SmRing {
  int idx = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++idx == n) {
      idx = 0;
      phase ^= 1u;
    }
  }
};

struct SmTile {
  int e, seg_lo, mt, t0, nt;
};

// tile_start[a]: first tile of active expert a; tiles of an expert are its
// m-tiles x token chunks (token chunk fastest).
__device__ __forceinline__ SmTile sm_tile(const SmParams& p, const int* act_e, const int* tile_start,
                                          int n_act, int t) {
  int lo = 0, hi = n_act - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  SmTile ti;
  ti.e = act_e[lo];
  ti.seg_lo = __ldg(p.offsets + ti.e);
  const int m = __ldg(p.offsets + ti.e + 1) - ti.seg_lo;
  const int nch = (m + kSmBN - 1) / kSmBN;
  const int local = t - tile_start[lo];
  ti.mt = local / nch;
  const int ch = local - ti.mt * nch;
  ti.t0 = ch * kSmBN;
  ti.nt = min(kSmBN, m - ti.t0);
  return ti;
}

// Weight row (within the expert) of tile row r (= TMEM lane).
template <int MODE>
__device__ __forceinline__ int sm_weight_row(const SmParams& p, int mt, int r) {
  if (MODE == kSmSwiglu) {
    const int q = r >> 5, l = r & 31;
    const int f = mt * 64 + q * 16 + (l & 15);
    return l < 16 ? f : (p.n_rows >> 1) + f;
  }
  return mt * kSmBM + r;
}

// Source row of activations of token slot n of a tile.
__device__ __forceinline__ int64_t sm_act_row(const SmParams& p, const SmTile& ti, int n) {
  const int r = ti.seg_lo + ti.t0 + n;
  return p.act_kind == 0 ? (int64_t)(__ldg(p.sorted + r) / p.kmax) : (int64_t)r;
}

template <int BITS, int MODE>
__global__ void __launch_bounds__(kSmThreads, 1)
    tc_small_kernel(const __grid_constant__ CUtensorMap tm_codes, SmParams p) {
  constexpr int KPG = BITS / 4;      // k-blocks (64 nibbles) per group of 64 elements
  constexpr float kMult = BITS == 4 ? 1.0f : 17.0f;

  extern __shared__ __align__(1024) unsigned char sm_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
  // codes ring: c_full (TMA bytes), c_empty (the 4 converter warps read it)
  __shared__ uint64_t c_full[kSmSC], c_empty[kSmSC];
  // stage ring: full once the 4 converter warps and the token stager have
  // written its A and B slots; empty once its MMAs completed
  __shared__ uint64_t full[kSmS], empty[kSmS];
  __shared__ uint64_t acc_full[2], acc_empty[2], xs_bar[2];
  __shared__ uint64_t drain_bar[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int act_e[1024];
  __shared__ int tile_start[1025];
  __shared__ int n_act_sh;
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ngroups = p.K / 64;
  const int nkb = ngroups * KPG;
  const int nchunks = (ngroups + kSmGC - 1) / kSmGC;

  unsigned char* cring = smem;                                        // kSmSC x 4 KB codes
  unsigned char* bring = cring + kSmSC * kSmCSlotBytes;               // kSmS x 2 KB tokens
  float* xsum = reinterpret_cast<float*>(bring + kSmS * kSmBSlotBytes);  // [2][ngroups][16]

  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < kSmSC; ++s) {
      mbar_init(&c_full[s], 1);
      mbar_init(&c_empty[s], 4);
    }
    for (int s = 0; s < kSmS; ++s) {
      mbar_init(&full[s], 5);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], kSmMmaWarps);
      mbar_init(&acc_empty[b], kSmEpiWarps);
      mbar_init(&xs_bar[b], kSmEpiWarps);
      mbar_init(&drain_bar[b], 1);
    }
    fence_barrier_init();
  }
  if (warp == kSmMmaWarp0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base_sh)),
                 "r"(kSmTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    int n = 0, t = 0;
    for (int e = 0; e < p.E; ++e) {
      const int m = __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
      if (m > 0) {
        act_e[n] = e;
        tile_start[n] = t;
        t += p.n_mt * ((m + kSmBN - 1) / kSmBN);
        ++n;
      }
    }
    tile_start[n] = t;
    n_act_sh = n;
  }
  tc_fence_before_sm();
  __syncthreads();
  tc_fence_after_sm();
  const uint32_t tmem_base = tmem_base_sh;
  const int n_act = n_act_sh;
  const int n_tiles = n_act > 0 ? tile_start[n_act] : 0;

  if (warp == kSmCodeWarp) {
    // ========================= codes: TMA issue =========================
    // lane b < 8 copies tile rows 16b .. 16b+15 of each k-block (SWIGLU:
    // quarter b/2, gate rows for even b, up rows for odd b)
    SmRing rc;
    int64_t issued = 0;
    bool ok = true;
    long long w_code = 0;
    const long long t_code0 = clock64();
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      const SmTile ti = sm_tile(p, act_e, tile_start, n_act, t);
      int wrow0 = sm_weight_row<MODE>(p, ti.mt, 16 * (lane & 7));
      const int crow = (int)((int64_t)ti.e * p.n_rows + wrow0);
      for (int kb = 0; kb < nkb && ok; ++kb) {
        TCS_T0();
        if (!sm_warp_wait(&c_empty[rc.idx], rc.phase ^ 1u, &abort_flag)) {
          ok = false;
          break;
        }
        TCS_ACC(w_code);
        if (lane == 0) mbar_arrive_expect_tx(&c_full[rc.idx], kSmCSlotBytes);
        __syncwarp();
        if (lane < 8)
          tma_load_2d_sm(cring + rc.idx * kSmCSlotBytes + lane * 512, &tm_codes, kb * 8, crow,
                         &c_full[rc.idx]);
        __syncwarp();
        ++issued;
        rc.next(kSmSC);
      }
    }
    if (lane == 0) {
      TCS_FLUSH(2, w_code);
      TCS_FLUSH(3, clock64() - t_code0);
    }
    if (!ok && lane == 0) {
      raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
      abort_flag = 1;
      SmRing r = rc;  // the last min(issued, SC) slots may still be in flight
      for (int64_t j = 0; j < issued && j < kSmSC; ++j) {
        r.idx = r.idx == 0 ? kSmSC - 1 : r.idx - 1;
        if (r.idx == kSmSC - 1) r.phase ^= 1u;
        mbar_wait(&c_full[r.idx], r.phase, kWaitBudgetCycles);
      }
    }
  } else if (warp >= kSmConvWarp0) {
    // ============================== convert ==============================
    const int quarter = warp & 3;                 // TMEM lanes this warp may write
    const int par = (warp - kSmConvWarp0) >> 2;   // k-blocks of this parity
    const int r = quarter * 32 + lane;            // tile row = TMEM lane
    const int my_tiles = blockIdx.x < n_tiles ? (n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int64_t total_kb = (int64_t)my_tiles * nkb;
    const int64_t own = total_kb > par ? (total_kb - par + 1) / 2 : 0;
    SmRing rc, ra;  // codes ring and stage ring positions of k-block i = par + 2 j
    rc.idx = par;
    ra.idx = par;
    bool ok = true;
    long long w_conv_wait = 0, w_conv_code = 0;
    const long long t_conv0 = clock64();
    for (int64_t j = 0; j < own && ok; ++j) {
      {
        TCS_T0();
        if (!sm_warp_wait(&c_full[rc.idx], rc.phase, &abort_flag)) ok = false;
        TCS_ACC(w_conv_code);
      }
      if (!ok) break;
      const uint4* src = reinterpret_cast<const uint4*>(cring + rc.idx * kSmCSlotBytes + r * 32);
      const uint4 c0 = src[0], c1 = src[1];
      __syncwarp();
      if (lane == 0) mbar_arrive(&c_empty[rc.idx]);
      rc.next(kSmSC);
      rc.next(kSmSC);
      const uint32_t wv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      uint32_t cell[kSmCells];
#pragma unroll
      for (int w = 0; w < 8; ++w)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
          cell[4 * w + jj] = ((wv[w] >> (4 * jj)) & 0x000F000Fu) | 0x43004300u;
      {
        TCS_T0();
        if (!sm_warp_wait(&empty[ra.idx], ra.phase ^ 1u, &abort_flag)) ok = false;
        TCS_ACC(w_conv_wait);
      }
      if (!ok) break;
      tc_fence_after_sm();
      tmem_st32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(ra.idx * kSmCells), cell);
      tmem_st_wait();
      tc_fence_before_sm();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[ra.idx]);
      ra.next(kSmS);
      ra.next(kSmS);
    }
    if (lane == 0) {
      TCS_FLUSH(0, w_conv_wait);
      TCS_FLUSH(1, clock64() - t_conv0);
      TCS_FLUSH(12, w_conv_code);
    }
    if (!ok && lane == 0) {
      raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
      abort_flag = 1;
    }
  } else if (warp == kSmStageWarp) {
    // ========================= tokens: B staging =========================
    // lane l fills B positions 2l, 2l+1 of a k-block: word w = l / 4,
    // nibbles j = l % 4 and j + 4 of that word.  The values of up to 4 tokens
    // of kSmStageBatch k-blocks are loaded before any is stored.
    const int w = lane >> 2, j = lane & 3;
    float m0 = 1.0f;
    int d0, d1;  // element offsets of the two nibbles within a k-block's words
    if (BITS == 4) {
      d0 = 8 * w + j;
      d1 = 8 * w + j + 4;
    } else {
      d0 = 4 * w + (j >> 1);
      d1 = 4 * w + 2 + (j >> 1);
      m0 = (j & 1) ? 16.0f : 1.0f;
    }
    constexpr int KB_ELEMS = 64 / KPG;  // elements per k-block
    SmRing rb;
    bool ok = true;
    long long w_stage = 0;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      const SmTile ti = sm_tile(p, act_e, tile_start, n_act, t);
      for (int kb0 = 0; kb0 < nkb && ok; kb0 += kSmStageBatch) {
        const int nb = min(kSmStageBatch, nkb - kb0);
        for (int n0 = 0; n0 < ti.nt && ok; n0 += 4) {
          uint16_t v0[kSmStageBatch][4], v1[kSmStageBatch][4];
          const uint16_t* xr[4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            xr[q] = p.act + sm_act_row(p, ti, n0 + q < ti.nt ? n0 + q : n0) * p.K;
#pragma unroll
          for (int u = 0; u < kSmStageBatch; ++u)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int e = (kb0 + (u < nb ? u : 0)) * KB_ELEMS;
              v0[u][q] = __ldg(xr[q] + e + d0);
              v1[u][q] = __ldg(xr[q] + e + d1);
            }
          // slots of these k-blocks: the first token group waits for them,
          // the last one publishes them
          const bool last_group = n0 + 4 >= ti.nt;
          SmRing r = rb;
#pragma unroll
          for (int u = 0; u < kSmStageBatch; ++u) {
            if (u < nb && ok) {
              if (n0 == 0) {
                TCS_T0();
                if (!sm_warp_wait(&empty[r.idx], r.phase ^ 1u, &abort_flag)) ok = false;
                TCS_ACC(w_stage);
              }
              if (ok) {
                unsigned char* slot = bring + r.idx * kSmBSlotBytes;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  if (n0 + q < ti.nt) {
                    const float x0 = bf16_bits_to_f32(v0[u][q]) * m0;
                    const float x1 = bf16_bits_to_f32(v1[u][q]) * m0;
                    const uint32_t v = (__float_as_uint(x0) >> 16) | (__float_as_uint(x1) & 0xFFFF0000u);
                    *reinterpret_cast<uint32_t*>(slot + sw128_off_sm(n0 + q, lane >> 2) + (lane & 3) * 4) = v;
                  }
                }
                if (last_group) {
                  fence_proxy_async_smem_sm();
                  __syncwarp();
                  if (lane == 0) mbar_arrive(&full[r.idx]);
                }
              }
              r.next(kSmS);
            }
          }
          if (last_group) rb = r;
        }
      }
    }
    if (lane == 0) TCS_FLUSH(14, w_stage);
    if (!ok && lane == 0) {
      raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
      abort_flag = 1;
    }
  } else if (warp == kSmMmaWarp0 || warp == kSmMmaWarp0 + 1) {
    // ================================= MMA =================================
    // warp m issues the MMAs of the groups g with g % 2 == m (their own
    // accumulator columns), so one warp's MMAs run while the other waits
    const int m = warp - kSmMmaWarp0;
    if (lane == 0) {
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kSmBN >> 3) << 17) |
                             ((uint32_t)(kSmBM >> 4) << 24);
      SmRing ra;
      int64_t issued = 0;
      int chunk_no = 0;
      bool ok = true;
      long long w_mma_acc = 0, w_mma_full = 0, w_mma_issue = 0;
      const long long t_mma0 = clock64();
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
        for (int c = 0; c < nchunks && ok; ++c, ++chunk_no) {
          const int buf = chunk_no & 1;
          {
            TCS_T0();
            if (!mbar_wait_sleep(&acc_empty[buf], (uint32_t)(((chunk_no >> 1) & 1) ^ 1),
                                 kWaitBudgetCycles) ||
                abort_flag)
              ok = false;
            TCS_ACC(w_mma_acc);
          }
          if (!ok) break;
          tc_fence_after_sm();
          const int g1 = min(ngroups, (c + 1) * kSmGC);
          bool any = false;
          for (int g = c * kSmGC; g < g1 && ok; ++g) {
            if ((g & 1) != m) {  // the other warp's group: skip its stages
              for (int h = 0; h < KPG; ++h) ra.next(kSmS);
              continue;
            }
            const uint32_t d = tmem_base + (uint32_t)(kSmAccCol0 + buf * kSmGC * kSmBN +
                                                      (g - c * kSmGC) * kSmBN);
            for (int h = 0; h < KPG; ++h) {
              {
                TCS_T0();
                if (!mbar_wait_sleep(&full[ra.idx], ra.phase, kWaitBudgetCycles)) ok = false;
                TCS_ACC(w_mma_full);
              }
              if (!ok) break;
              TCS_T0();
              tc_fence_after_sm();
              const uint32_t a = tmem_base + (uint32_t)(ra.idx * kSmCells);
              const uint64_t bd = smem_desc_sw128_sm(bring + ra.idx * kSmBSlotBytes);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)  // K = 16 per MMA: 8 cells of A, 32 bytes of B
                umma_bf16_tmem_a(d, a + 8 * kk, bd + 2 * kk, idesc, (h | kk) != 0 ? 1u : 0u);
              umma_commit_sm(&empty[ra.idx]);
              TCS_ACC(w_mma_issue);
              ra.next(kSmS);
              ++issued;
              any = true;
            }
          }
          if (!ok) break;
          // this warp's MMAs of the chunk (if any) complete, then the arrival
          if (any) umma_commit_sm(&acc_full[buf]);
          else mbar_arrive(&acc_full[buf]);
        }
      }
      if (!ok) {
        raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
        abort_flag = 1;
      }
      if (issued > 0) {
        umma_commit_sm(&drain_bar[m]);
        mbar_wait(&drain_bar[m], 0, kWaitBudgetCycles);
      }
      if (m == 0) {
        TCS_FLUSH(4, w_mma_acc);
        TCS_FLUSH(5, w_mma_full);
        TCS_FLUSH(7, clock64() - t_mma0);
        TCS_FLUSH(8, issued);
        TCS_FLUSH(6, w_mma_issue);
      }
    }
    __syncwarp();
  } else if (warp < kSmEpiWarps) {
    // ============================== epilogue ==============================
    const int quarter = warp;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
    int chunk_no = 0, tile_no = 0;
    bool ok = true;
    long long w_epi_acc = 0, w_epi_xs = 0;
    const long long t_epi0 = clock64();
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++tile_no) {
      const SmTile ti = sm_tile(p, act_e, tile_start, n_act, t);
      const int xb = tile_no & 1;
      float* xs = xsum + (size_t)xb * ngroups * kSmBN;
      // X sums of the tile's tokens per group (warp w: groups w, w+4, ...),
      // a fixed lane tree
      for (int g = quarter; g < ngroups; g += kSmEpiWarps) {
        for (int n = 0; n < ti.nt; ++n) {
          const uint16_t* xr = p.act + sm_act_row(p, ti, n) * p.K + g * 64;
          float v = __fadd_rn(bf16_bits_to_f32(__ldg(xr + 2 * lane)),
                              bf16_bits_to_f32(__ldg(xr + 2 * lane + 1)));
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1)
            v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
          if (lane == 0) xs[g * kSmBN + n] = v;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&xs_bar[xb]);
      {
        TCS_T0();
        if (!sm_warp_wait(&xs_bar[xb], (uint32_t)((tile_no >> 1) & 1), &abort_flag)) ok = false;
        TCS_ACC(w_epi_xs);
      }
      if (!ok) break;
      int wrow = sm_weight_row<MODE>(p, ti.mt, r);
      const bool row_ok = wrow < p.n_rows;  // RAW output row exists
      if (wrow >= p.n_rows) wrow = p.n_rows - 1;
      const int64_t grow = (int64_t)ti.e * p.n_rows + wrow;
      const uint16_t* sp = p.ws + grow * ngroups;
      const uint16_t* bp = p.wb + grow * ngroups;
      float acc[kSmBN];
#pragma unroll
      for (int n = 0; n < kSmBN; ++n) acc[n] = 0.0f;
      // scales of the next chunk are in flight while one is applied
      uint16_t sv[kSmGC], bv[kSmGC];
      auto load_scales = [&](int c, uint16_t (&s_)[kSmGC], uint16_t (&b_)[kSmGC]) {
        const int g0 = c * kSmGC, g1 = min(ngroups, g0 + kSmGC);
#pragma unroll
        for (int i = 0; i < kSmGC; ++i) {
          const int g = min(g0 + i, g1 - 1);
          s_[i] = __ldg(sp + g);
          b_[i] = __ldg(bp + g);
        }
      };
      load_scales(0, sv, bv);
      for (int c = 0; c < nchunks && ok; ++c, ++chunk_no) {
        const int buf = chunk_no & 1;
        const int g0 = c * kSmGC, g1 = min(ngroups, g0 + kSmGC);
        uint16_t svn[kSmGC], bvn[kSmGC];
        load_scales(c + 1 < nchunks ? c + 1 : c, svn, bvn);
        {
          TCS_T0();
          if (!sm_warp_wait(&acc_full[buf], (uint32_t)((chunk_no >> 1) & 1), &abort_flag)) ok = false;
          TCS_ACC(w_epi_acc);
        }
        if (!ok) break;
        tc_fence_after_sm();
#pragma unroll
        for (int i = 0; i < kSmGC; i += 2) {
          uint32_t d0[16], d1[16];
          const uint32_t col = lane_base + (uint32_t)(kSmAccCol0 + buf * kSmGC * kSmBN + i * kSmBN);
          tmem_ld16_sm(col, d0);
          tmem_ld16_sm(col + kSmBN, d1);
          tmem_ld_wait_sm();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (g0 + i + h < g1) {
              const uint32_t* d = h == 0 ? d0 : d1;
              const float s = f16_bits_to_f32(sv[i + h]), b = f16_bits_to_f32(bv[i + h]);
              const float* xg = xs + (g0 + i + h) * kSmBN;
#pragma unroll
              for (int n = 0; n < kSmBN; ++n) {
                if (n < ti.nt) {
                  const float X = xg[n];
                  const float dq = fmaf(-128.0f * kMult, X, __uint_as_float(d[n]));
                  acc[n] = fmaf(s, dq, fmaf(b, X, acc[n]));
                }
              }
            }
          }
        }
        tc_fence_before_sm();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
#pragma unroll
        for (int i = 0; i < kSmGC; ++i) {
          sv[i] = svn[i];
          bv[i] = bvn[i];
        }
      }
      if (!ok) break;
      // outputs
      const int64_t orow0 = (int64_t)ti.seg_lo + ti.t0;
      if (MODE == kSmSwiglu) {
        const int f = ti.mt * 64 + quarter * 16 + (lane & 15);
#pragma unroll
        for (int n = 0; n < kSmBN; ++n) {
          const float u = __shfl_down_sync(0xFFFFFFFFu, acc[n], 16);
          if (lane < 16 && n < ti.nt && f < p.n_out) {
            const float hv = swiglu_f32(acc[n], u);
            if (p.out_dtype == MOE_DTYPE_BF16)
              static_cast<uint16_t*>(p.out)[(orow0 + n) * p.n_out + f] = f32_to_bf16_rne(hv);
            else
              static_cast<float*>(p.out)[(orow0 + n) * p.n_out + f] = hv;
          }
        }
      } else if (row_ok) {
#pragma unroll
        for (int n = 0; n < kSmBN; ++n)
          if (n < ti.nt) static_cast<float*>(p.out)[(orow0 + n) * p.n_out + wrow] = acc[n];
      }
    }
    if (lane == 0 && warp == 0) {
      TCS_FLUSH(9, w_epi_acc);
      TCS_FLUSH(10, w_epi_xs);
      TCS_FLUSH(11, clock64() - t_epi0);
    }
    if (!ok && lane == 0) {
      raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
      abort_flag = 1;
    }
  }

  tc_fence_before_sm();
  __syncthreads();
  tc_fence_after_sm();
  if (warp == kSmMmaWarp0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kSmTmemCols)
                 : "memory");
}

template <int BITS, int MODE>
moe_status_t launch_tc_small(const CUtensorMap& tmc, const SmParams& p, int64_t max_tiles,
                             cudaStream_t st) {
  auto kern = tc_small_kernel<BITS, MODE>;
  const size_t smem = (size_t)kSmSC * kSmCSlotBytes + (size_t)kSmS * kSmBSlotBytes +
                      2 * (size_t)(p.K / 64) * kSmBN * 4 + 1024;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  const int64_t sms = moe_host::sm_count();
  const int grid = (int)(max_tiles < sms ? max_tiles : sms);
  if (grid <= 0) return MOE_OK;
  kern<<<grid, kSmThreads, smem, st>>>(tmc, p);
  return moe_host::launch_status();
}

}  // namespace

moe_status_t tc_small_qmm(const void* act, int act_kind, const int32_t* sorted,
                          const int32_t* offsets, int T, int kmax, int E, int K, int n_rows,
                          bool swiglu, const uint32_t* wq, const uint16_t* ws, const uint16_t* wb,
                          int bits, void* out, int out_dtype, cudaStream_t st) {
  // act_kind: 0 = x bf16 [T, K] through sorted_assign, 2 = bf16 rows in sorted order
  if (act_kind != 0 && act_kind != 2) return MOE_ERR_UNSUPPORTED;
  if (K % 64 != 0 || n_rows % 64 != 0 || E > 1024) return MOE_ERR_INVALID_ARG;
  if (K / 64 > 1024) return MOE_ERR_UNSUPPORTED;  // X sums of two tiles fit shared memory
  const int64_t A = (int64_t)T * kmax;
  if (A == 0) return MOE_OK;
  SmParams p;
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
  p.n_mt = swiglu ? (p.n_out + 63) / 64 : (n_rows + kSmBM - 1) / kSmBM;
  p.err = moe_host::device_error_word();
  const int64_t max_active = A < E ? A : E;
  const int64_t max_tiles = (int64_t)p.n_mt * (max_active + (A + kSmBN - 1) / kSmBN);
  // codes: [E * n_rows rows, K*bits/32 words], boxes of 16 rows x 8 words
  if (!tc_available()) return MOE_ERR_UNSUPPORTED;
  CUtensorMap tmc;
  const uint64_t row_words = (uint64_t)K * bits / 32;
  if (!make_tensor_map_2d(&tmc, CU_TENSOR_MAP_DATA_TYPE_UINT32, wq, row_words,
                          (uint64_t)E * n_rows, row_words * 4, 8, 16, CU_TENSOR_MAP_SWIZZLE_NONE))
    return MOE_ERR_CUDA;
  if (bits == 4)
    return swiglu ? launch_tc_small<4, kSmSwiglu>(tmc, p, max_tiles, st)
                  : launch_tc_small<4, kSmRaw>(tmc, p, max_tiles, st);
  return swiglu ? launch_tc_small<8, kSmSwiglu>(tmc, p, max_tiles, st)
                : launch_tc_small<8, kSmRaw>(tmc, p, max_tiles, st);
}

}  // namespace moe

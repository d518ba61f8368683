// Streamed grouped GEMV with warp-level MMAs: the decode / small-batch path
// of the two quantized products.
//
// Page "oMLX MoE gate/up 融合优化：qwen35_moe_gate_up 实现剖析", 融合原理 and
// 实现剖析 ④ (one gathered product with the [gate; up] matrix, split, SwitchGLU
// activation, down projection); page "Qwen3.5 Block在llama.cpp中的映射与优化
// 原理", section 4.2 (only the routed experts' weights are read).
//
// Arithmetic.  Per group of 64 elements of a weight row (scale s, bias b):
//   sum_i x_i (s q_i + b) = s * sum_i q_i x_i + b * X,   X = sum_i x_i.
// The codes enter the tensor cores unconverted: a 4-bit code word masked with
// 0x000F000F, read as two fp16 values, is exactly (q_j, q_{j+4}) * 2^-24 (fp16
// subnormals); masked with 0x00F000F0 it is (16 q_{j+1}, 16 q_{j+5}) * 2^-24,
// so those slots take the token values divided by 16; an 8-bit word masked
// with 0x00FF00FF is (c_0, c_2) * 2^-24.  One or two integer instructions per
// A register, then mma.sync.m16n8k16 (fp16 x fp16 -> fp32).  The token
// values are staged as fp16 x * 2^e, one power of two per token and group
// chosen so that the group's max |x| 2^e lies in [2^14, 2^15): exact for
// bf16 values in range.  So one MMA forms P = 2^(e-24) sum q x over 16 k for
// 16 weight rows and up to 8 tokens, with no offset to cancel; CUDA cores
// accumulate (s 2^(24-e)) P and b X per group.
//
// Data movement.  A tile is 16 weight rows (SWIGLU: 8 gate rows and the 8 up
// rows of the same features) of one active expert, applied to a chunk of up
// to 8 of its tokens.  A stage is 2 KB of codes of each of the tile's rows
// plus their fp16 scales and biases.  One CTA of 19 warps per SM:
//   warp 16     producer: TMA (cp.async.bulk.tensor, 128-byte swizzle) loads
//               the codes of each stage into a ring of shared-memory slots;
//   warp 17     its lanes copy the stage's scales and biases with cp.async,
//               whose completion arrives on the same slot mbarrier;
//   warps 0-15  consumers: each takes one of 16 slots of a tile's groups
//               (128 contiguous code bytes of every stage; the warp of a
//               slot rotates from tile to tile), converts the codes in
//               registers and issues the MMAs;
//               the token values are staged once per (expert, chunk) in the
//               B-fragment order, with their group sums;
//   warp 18     epilogue: adds the 16 slot partials of each row of a tile
//               (slots 0-7 and 8-15 each in order, then the two halves) and
//               writes SiLU(gate) * up or the raw fp32 rows.
// Each CTA takes an equal contiguous range of the tile list (expert-major),
// so the weight stream of the whole GPU is split evenly across the SMs.
//
// Every row is reduced in the same order whatever rows it shares a tile
// with (a fixed group -> slot assignment, slot partials added in slot
// order), so the fused gate_up product equals the separate gate and up
// products bit for bit.  Every mbarrier wait is bounded; a wait that runs
// out sets MOE_DEVERR_TIMEOUT, the CTA stops and the producer waits for the
// copies it has in flight.
#include <cuda.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "async.cuh"
#include "common.cuh"

namespace moe {

bool make_tensor_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base,
                        const uint64_t (&dims)[3], const uint64_t (&strides)[2],
                        const uint32_t (&box)[3], CUtensorMapSwizzle sw);
bool tc_available();

namespace {

constexpr int kSvConsumers = 16;
constexpr int kSvThreads = (kSvConsumers + 3) * 32;
constexpr int kSvProducer = kSvConsumers;      // codes (TMA)
constexpr int kSvScaler = kSvConsumers + 1;    // scales and biases (cp.async)
constexpr int kSvEpilogue = kSvConsumers + 2;
constexpr int kSvRowChunk = 2048;               // code bytes of one row per stage
constexpr int kSvCodeBytes = 16 * kSvRowChunk;  // codes of one stage
constexpr int kSvHalfBytes = 8 * kSvRowChunk;   // tile rows 0-7 | rows 8-15
constexpr int kSvBoxes = kSvRowChunk / 128;     // 128-byte blocks per row and stage
constexpr int kSvMaxStages = 8;
constexpr int kSvMaxRedSlots = 4;

// Result slots between consumers and epilogue: more when they are small.
__host__ __device__ constexpr int sv_red_slots(int mts) { return mts == 1 ? 4 : 2; }
constexpr int kSvMaxE = 1024;
constexpr int kSvMaxTokens = 8;  // tokens per pass (the n of one MMA)

enum SvMode { kSvSwiglu = 0, kSvRaw = 1 };
enum SvAct { kSvActX = 0, kSvActF32 = 1, kSvActBf16 = 2 };

template <int BITS>
struct SvShape {
  static constexpr int kGroupBytes = 32 * BITS / 4;       // codes of one row per group
  static constexpr int kLaneWords = kGroupBytes / 16;     // per lane, row and group: 2 | 4
  static constexpr int kGpc = kSvRowChunk / kGroupBytes;  // groups per stage: 32 | 16
  static constexpr int kGpw = kGpc / kSvConsumers;        // groups per consumer warp
  static constexpr int kScaleRow = kGpc * 2 + 16;         // padded bytes per scale row
  using ScaleVec = typename std::conditional<BITS == 4, uint2, uint32_t>::type;  // kGpw halves
  static constexpr int kScaleBytes = 2 * 16 * kScaleRow;  // scales and biases of 16 rows
};

struct SvParams {
  const void* act;
  int act_kind;
  const int32_t* sorted;
  const int32_t* offsets;  // [E+1]
  const uint16_t* ws;      // [E, n_rows, K/64]
  const uint16_t* wb;
  void* out;
  int out_dtype;
  int T, kmax, E, K, n_rows, n_out;
  int mts;       // tokens per pass: 1, 2, 4 or 8
  int stages;    // ring slots
  int rt;        // row tiles per (expert, token chunk)
  int scale_cw;  // cp.async width for scales and biases: 4, 8 or 16 bytes
  int early;     // offsets and weights final before the previous kernel ends:
                 // stream them before waiting on it (activations after)
  KGate gate;    // k-gated launch (gate.k null: always runs)
  unsigned int* err;
};

struct SvLayout {
  uint32_t codes, scales, x, xsum, red, act, bars, total;
};

// Shared-memory carve-up, from a 1024-byte aligned base.
__host__ __device__ inline SvLayout sv_layout(int bits, int K, int mts, int stages, int E,
                                              bool dual) {
  const int ngroups = K / 64;
  const int gpc = kSvRowChunk / (8 * bits);
  const int scale_bytes = (dual ? 2 : 1) * 2 * 16 * (gpc * 2 + 16);
  const int mts2 = mts < 2 ? 2 : mts;
  SvLayout L;
  uint32_t o = 0;
  L.codes = o;
  o += (uint32_t)stages * kSvCodeBytes;
  L.scales = o;
  o += (uint32_t)stages * scale_bytes;
  L.x = o;
  o += (uint32_t)ngroups * 2 * mts * 4 * 16;
  L.xsum = o;
  o += (uint32_t)ngroups * mts2 * 8;
  L.red = o;
  o += (uint32_t)sv_red_slots(mts) * kSvConsumers * mts * 16 * 4;
  L.act = o;
  o += (uint32_t)4 * (E + 1) * 4;
  o = (o + 7u) & ~7u;
  L.bars = o;
  o += (uint32_t)(2 * stages + 2 * kSvMaxRedSlots + 2) * 8;
  L.total = o;
  return L;
}

struct SvRing {
  int idx;
  uint32_t phase;
  __device__ __forceinline__ void next(int n) {
    if (++idx == n) {
      idx = 0;
      phase ^= 1u;
    }
  }
};

// Bounded wait of a whole warp; a waiting thread sleeps in the barrier
// (woken when the phase completes) instead of spinning on issue slots that
// the working warps of its SM sub-partition need.
__device__ __forceinline__ bool sv_wait(uint64_t* bar, uint32_t parity) {
  bool ok = mbar_test(bar, parity);
  if (!ok) {
    const long long t0 = clock64();
    while (!(ok = mbar_test_sleep(bar, parity, 1000u)))
      if (clock64() - t0 > kWaitBudgetCycles) break;
  }
  return __all_sync(0xFFFFFFFFu, ok);
}

// One 3D box: 32 code words x 8 rows x 8 consecutive 128-byte blocks of the
// rows (8 KB), written as [block][row][128 B] with the 128-byte swizzle.
__device__ __forceinline__ void tma_load_3d_sv(void* dst, const CUtensorMap* tm, int row, int kblk,
                                               uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(0), "r"(row), "r"(kblk), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void cp_async_sv(void* dst, const void* src, int width) {
  if (width == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
  else if (width == 8)
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}

// Arrives on `bar` once every cp.async this thread issued before has landed.
__device__ __forceinline__ void cp_async_arrive_sv(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void cp_async_wait_all_sv() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// d = A B (zero accumulator in)
__device__ __forceinline__ void mma_sv0(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

__device__ __forceinline__ void mma_sv(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                       uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Half i of a packed vector of fp16 scales, as fp32.
__device__ __forceinline__ float sv_half(uint32_t v, int i) {
  const __half2 h = *reinterpret_cast<const __half2*>(&v);
  return (i & 1) ? __high2float(h) : __low2float(h);
}
__device__ __forceinline__ float sv_half(uint2 v, int i) { return sv_half(i < 2 ? v.x : v.y, i); }

// Walk over the tile list: active expert a, token chunk c, row tile rt.
struct SvCursor {
  int a, c, rt, nch;
};

// GATED: a k-gated launch (p.gate); a separate instantiation, since even an
// untaken gate check at the top cost the single-token kernels 3 %.
// DUAL: rows of at most 8 blocks (1024 bytes): a tile is 32 rows (SWIGLU:
// 16 gate rows and the 16 up rows of the same features), held as two
// 16-row halves of a stage (four boxes of 8 rows x 8 blocks); consumer
// warps 0-7 take the group slots of half 0 and warps 8-15 those of half 1,
// so a short row keeps twice as many warps busy and a stage carries twice
// the rows.
template <int BITS, int MODE, bool ONE, bool GATED, bool DUAL>
__global__ void __launch_bounds__(kSvThreads, 1)
    gemv_stream_kernel(const __grid_constant__ CUtensorMap tm_codes, SvParams p) {
  using S = SvShape<BITS>;
  // bytes between the two 8-row boxes of a 16-row half, and scale bytes per stage
  constexpr int kHalfOff = DUAL ? 8 * 1024 : kSvHalfBytes;
  constexpr int kScaleStage = (DUAL ? 2 : 1) * S::kScaleBytes;
  constexpr int kRowsPerTile = DUAL ? 32 : 16;
  if constexpr (GATED) {
    if (k_gate_closed(p.gate.k, p.gate.lo, p.gate.hi, p.early != 0)) return;
  }
  extern __shared__ __align__(16) unsigned char sv_raw[];
  unsigned char* sm = sv_raw + ((1024u - (smem_u32(sv_raw) & 1023u)) & 1023u);
  const SvLayout L = sv_layout(BITS, p.K, p.mts, p.stages, p.E, DUAL);
  unsigned char* codes = sm + L.codes;
  unsigned char* scales = sm + L.scales;
  uint4* xs = reinterpret_cast<uint4*>(sm + L.x);      // [G][half][n][t] B fragments
  float2* xsum = reinterpret_cast<float2*>(sm + L.xsum);  // [G][mts2] (X, 2^(24-e))
  float* red = reinterpret_cast<float*>(sm + L.red);       // [slot][warp][n][16 rows]
  int* act_e = reinterpret_cast<int*>(sm + L.act);
  int* act_lo = act_e + (p.E + 1);
  int* act_m = act_lo + (p.E + 1);
  int* act_base = act_m + (p.E + 1);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* empty = full + p.stages;
  uint64_t* red_full = empty + p.stages;
  const int rslots = sv_red_slots(ONE ? 1 : p.mts);
  uint64_t* red_empty = red_full + rslots;
  uint64_t* xbar = red_empty + rslots;  // consumer-only barrier (two phases per restage)
  __shared__ int n_act_sh;
  __shared__ int wtot[kSvThreads / 32];
  __shared__ volatile int abort_flag;
  __shared__ int st_tok[kSvMaxTokens];
  __shared__ int st_nt;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int stages = p.stages;
  const int mts = ONE ? 1 : p.mts;
  const int mts2 = mts < 2 ? 2 : mts;
  const int ngroups = p.K / 64;

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 33);  // the producer's expect_tx + one cp.async arrival per lane
      mbar_init(&empty[s], kSvConsumers);
    }
    for (int r = 0; r < rslots; ++r) {
      mbar_init(&red_full[r], kSvConsumers);
      mbar_init(&red_empty[r], 1);
    }
    mbar_init(xbar, kSvConsumers);
    n_act_sh = 0;
    abort_flag = 0;
    st_nt = -1;
    fence_barrier_init();
  }
  __syncthreads();
  // the previous kernel of the stream: waited for here unless the offsets and
  // weights may be read while it finishes (then each role waits before it
  // reads activations or writes results, and every thread waits before exit)
  if (!p.early) pdl_wait();
  pdl_trigger();

  // active experts in id order, with segment start and length
  for (int base = 0; base < p.E; base += kSvThreads) {
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
      for (int w = 0; w < kSvThreads / 32; ++w) s += wtot[w];
      n_act_sh += s;
    }
    __syncthreads();
  }
  const int n_act = n_act_sh;
  // tiles before each active expert
  if (warp == 0) {
    int carry = 0;
    for (int a0 = 0; a0 < n_act; a0 += 32) {
      const int a = a0 + lane;
      int v = a < n_act ? ((act_m[a] + mts - 1) / mts) * p.rt : 0;
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
  const int n_tiles = act_base[n_act];
  const int u0 = (int)((int64_t)n_tiles * blockIdx.x / gridDim.x);
  const int u1 = (int)((int64_t)n_tiles * (blockIdx.x + 1) / gridDim.x);
  if (u0 >= u1) {
    pdl_wait();
    return;
  }

  auto cursor_at = [&](int u) {
    int lo = 0, hi = n_act - 1;  // last a with act_base[a] <= u
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (act_base[mid] <= u) lo = mid;
      else hi = mid - 1;
    }
    SvCursor cu;
    cu.a = lo;
    const int local = u - act_base[lo];
    cu.c = local / p.rt;
    cu.rt = local - cu.c * p.rt;
    cu.nch = (act_m[lo] + mts - 1) / mts;
    return cu;
  };
  auto cursor_next = [&](SvCursor& cu) {
    if (++cu.rt == p.rt) {
      cu.rt = 0;
      if (++cu.c == cu.nch) {
        cu.c = 0;
        ++cu.a;
        cu.nch = cu.a < n_act ? (act_m[cu.a] + mts - 1) / mts : 0;
      }
    }
  };
  const int row_words = p.K * BITS / 32;
  const int nck = (row_words + kSvRowChunk / 4 - 1) / (kSvRowChunk / 4);  // stages per tile

  if (warp == kSvProducer || warp == kSvScaler) {
    // ======================== producers (codes | scales) ======================
    // Both walk the same stages; a slot is full once the TMA bytes have landed
    // and every cp.async lane of the scale warp has arrived.
    const bool codes_warp = warp == kSvProducer;
    const int64_t tot_rows = (int64_t)p.E * p.n_rows;
    SvRing ring{0, 0u};
    bool ok = true;
    int64_t issued = 0;
    SvCursor cu = cursor_at(u0);
    const int arr = lane >> 4, srow = lane & 15;  // this lane's scale row
    for (int u = u0; u < u1 && ok; ++u, cursor_next(cu)) {
      const int64_t ebase = (int64_t)act_e[cu.a] * p.n_rows;
      // first rows of the tile's 8-row boxes: half h takes boxes 2h, 2h + 1
      int64_t rb[4];
      if (MODE == kSvSwiglu) {
        rb[0] = ebase + (int64_t)cu.rt * (kRowsPerTile / 2);
        rb[1] = rb[0] + p.n_out;
        rb[2] = rb[0] + 8;
        rb[3] = rb[1] + 8;
      } else {
        rb[0] = ebase + (int64_t)cu.rt * kRowsPerTile;
        rb[1] = rb[0] + 8;
        rb[2] = rb[0] + 16;
        rb[3] = rb[0] + 24;
      }
      for (int ch = 0; ch < nck; ++ch) {
        if (abort_flag || !sv_wait(&empty[ring.idx], ring.phase ^ 1u)) {
          ok = false;
          break;
        }
        if (codes_warp) {
          unsigned char* cdst = codes + (size_t)ring.idx * kSvCodeBytes;
          if (lane == 0) {
            // blocks past the row end are zero-filled and still counted
            mbar_arrive_expect_tx(&full[ring.idx], (uint32_t)kSvCodeBytes);
            if (DUAL) {
#pragma unroll
              for (int b = 0; b < 4; ++b)
                tma_load_3d_sv(cdst + b * 8192, &tm_codes, (int)rb[b], 0, &full[ring.idx]);
            } else {
              tma_load_3d_sv(cdst, &tm_codes, (int)rb[0], ch * kSvBoxes, &full[ring.idx]);
              tma_load_3d_sv(cdst + kSvHalfBytes, &tm_codes, (int)rb[1], ch * kSvBoxes,
                             &full[ring.idx]);
            }
          }
          __syncwarp();
        } else {
          const int g0 = ch * S::kGpc;
          const int gbytes = 2 * min(S::kGpc, ngroups - g0);
#pragma unroll
          for (int h = 0; h < (DUAL ? 2 : 1); ++h) {
            const int64_t grow = srow < 8 ? rb[2 * h] + srow : rb[2 * h + 1] + (srow - 8);
            if (grow < tot_rows) {
              const uint16_t* srcrow = (arr ? p.wb : p.ws) + grow * ngroups;
              unsigned char* sdst = scales + (size_t)ring.idx * kScaleStage + h * S::kScaleBytes +
                                    (arr * 16 + srow) * S::kScaleRow;
              const unsigned char* src = reinterpret_cast<const unsigned char*>(srcrow + g0);
              for (int o = 0; o < gbytes; o += p.scale_cw)
                cp_async_sv(sdst + o, src + o, p.scale_cw);
            }
          }
          cp_async_arrive_sv(&full[ring.idx]);
        }
        ++issued;
        ring.next(stages);
      }
    }
    if (!codes_warp) cp_async_wait_all_sv();
    pdl_wait();
    if (!ok && lane == 0) {
      raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
      abort_flag = 1;
      if (codes_warp) {
        // the last min(issued, stages) slots may still have copies in flight
        SvRing r = ring;
        for (int64_t j = 0; j < issued && j < stages; ++j) {
          r.idx = r.idx == 0 ? stages - 1 : r.idx - 1;
          if (r.idx == stages - 1) r.phase ^= 1u;
          mbar_wait(&full[r.idx], r.phase, kWaitBudgetCycles);
        }
      }
    }
  } else if (warp < kSvConsumers) {
    // ================================ consumers ===============================
    pdl_wait();
    const int g = lane >> 2, t = lane & 3;
    // shared-memory row of MMA row g (rows 0,4 | 2,6 | 1,5 | 3,7 per quarter
    // warp keep the swizzled code reads free of bank conflicts)
    const int rr = ((g & 1) << 2) | (g & 2) | ((g >> 2) & 1);
    const int ctid = tid;  // 0 .. 511
    SvRing ring{0, 0u}, rs{0, 0u};
    uint32_t xphase = 0;
    bool ok = true;
    int st_a = -1, st_c = -1;

    auto consumer_sync = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(xbar);
      const bool r = sv_wait(xbar, xphase);
      xphase ^= 1u;
      return r;
    };
    // the 16 token values (bf16 bits) of lane t of group G of staged token n
    auto load16 = [&](int r0, int n, int G, int tq, uint32_t (&v)[16]) {
      const int64_t col = (int64_t)G * 64 + tq * 16;
      if (p.act_kind == kSvActF32) {
        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.act) +
                                                            (int64_t)(r0 + n) * p.K + col);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 f = __ldg(src + q);
          v[4 * q] = f32_to_bf16_rne(f.x);
          v[4 * q + 1] = f32_to_bf16_rne(f.y);
          v[4 * q + 2] = f32_to_bf16_rne(f.z);
          v[4 * q + 3] = f32_to_bf16_rne(f.w);
        }
      } else {
        // x by token (a single-token call has only token 0), or h by sorted row
        const int64_t row = p.act_kind == kSvActX
                                ? (p.T == 1 ? 0 : (int64_t)(__ldg(p.sorted + r0 + n) / p.kmax))
                                : (int64_t)(r0 + n);
        const uint4* src =
            reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.act) + row * p.K + col);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint4 w = __ldg(src + q);
          const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            v[8 * q + 2 * i] = w4[i] & 0xFFFFu;
            v[8 * q + 2 * i + 1] = w4[i] >> 16;
          }
        }
      }
    };
    // stage the token values of (expert a, chunk c) in B-fragment order: per
    // group of 64 values one power of two 2^e with max |x| 2^e in [2^14,
    // 2^15) (found by the 4 lanes that hold the group), fp16 x 2^e (4-bit
    // odd-MMA slots x 2^(e-4): their codes read as 16 q), and per group the
    // sum X of x and the factor 2^(24-e) that undoes the scalings
    auto stage_x = [&](int a, int c) -> bool {
      const int lo = act_lo[a], m = act_m[a];
      const int nt = min(mts, m - c * mts);
      const int r0 = lo + c * mts;
      // everyone is done with the staged values (nothing staged before the first)
      if (st_a >= 0 && !consumer_sync()) return false;
      // a single-token pass reads only token 0's values and sums (the B
      // fragments' other columns and xsum's second entry are never used)
      const int total = ngroups * (ONE ? 1 : mts2) * 4;
      for (int base = 0; base < total; base += kSvConsumers * 32) {
        const int idx = base + ctid;
        const bool valid = idx < total;
        const int tq = idx & 3;
        const int rest = idx >> 2;
        const int n = rest / ngroups;
        const int G = rest - n * ngroups;
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0u;
        if (valid && n < nt) load16(r0, n, G, tq, v);
        float mx = 0.0f, xb = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float f = bf16_bits_to_f32(v[i]);
          mx = fmaxf(mx, fabsf(f));
          xb += f;
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
        xb += __shfl_xor_sync(0xFFFFFFFFu, xb, 1);
        xb += __shfl_xor_sync(0xFFFFFFFFu, xb, 2);
        const int E = (int)((__float_as_uint(mx) >> 23) & 0xFFu);
        int e = mx == 0.0f ? 0 : (E == 0 ? 100 : 141 - E);
        e = e < -100 ? -100 : (e > 100 ? 100 : e);
        const float sc = __uint_as_float((uint32_t)(127 + e) << 23);
        const float sc16 = __uint_as_float((uint32_t)(123 + e) << 23);
        uint32_t h[16], h16[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float f = bf16_bits_to_f32(v[i]);
          h[i] = __half_as_ushort(__float2half_rn(f * sc));
          h16[i] = BITS == 4 ? __half_as_ushort(__float2half_rn(f * sc16)) : 0u;
        }
        uint32_t regs[8];
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
          if (BITS == 4) {
            const uint32_t* src = (mm & 1) ? h16 : h;
            regs[2 * mm] = src[mm] | (src[mm + 4] << 16);
            regs[2 * mm + 1] = src[8 + mm] | (src[12 + mm] << 16);
          } else {
            const int pp = mm >> 1, r = mm & 1;
            regs[2 * mm] = h[8 * pp + r] | (h[8 * pp + r + 2] << 16);
            regs[2 * mm + 1] = h[8 * pp + 4 + r] | (h[8 * pp + 6 + r] << 16);
          }
        }
        if (valid && n < mts) {
#pragma unroll
          for (int q = 0; q < 2; ++q)
            xs[(((size_t)G * 2 + q) * mts + n) * 4 + tq] =
                make_uint4(regs[4 * q], regs[4 * q + 1], regs[4 * q + 2], regs[4 * q + 3]);
        }
        if (valid && tq == 0)
          xsum[(size_t)G * mts2 + n] =
              make_float2(xb, __uint_as_float((uint32_t)(151 - e) << 23));
      }
      if (ctid < kSvMaxTokens) {
        const int n = ctid;
        st_tok[n] = (n < nt && p.act_kind == kSvActX)
                        ? (p.T == 1 ? 0 : __ldg(p.sorted + r0 + n) / p.kmax)
                        : -1;
      }
      if (ctid == 0) st_nt = nt;
      return consumer_sync();
    };

    // Group slots.  Logical slot wl takes the groups jb .. jb + kGpw - 1
    // (jb = kGpw wl) of every stage of a tile and its partial sums go to
    // reduction slot wl, so each row is summed in the same order whichever
    // warp holds which slot.  The physical warp of a slot rotates from tile
    // to tile: the last stage of a tile is partial when a row is not a whole
    // number of stages (an 11008-code row fills 11 of 16 slots there, a
    // 1536-code one 6), and the rotation spreads the idle slots over the
    // warps.  kGpw groups are 128 bytes of a row, so slot wl's code offsets
    // in a slot are slot 0's plus wl 1024.
    int coff[S::kGpw];
#pragma unroll
    for (int i = 0; i < S::kGpw; ++i) {
      const int o = i * S::kGroupBytes + t * (S::kGroupBytes / 4);
      coff[i] = (o >> 7) * 1024 + rr * 128 + ((((o >> 4) & 7) ^ rr) << 4) + (o & 15);
    }
    static_assert(S::kGpw * S::kGroupBytes == 128, "a slot's groups span one 128-byte block");
    const int last_groups = ngroups - (nck - 1) * S::kGpc;
    const int rot_step = (last_groups + S::kGpw - 1) / S::kGpw;  // busy slots of the last stage
    // DUAL: warps 0-7 hold the slots of half 0, warps 8-15 those of half 1,
    // rotating within their eight
    const int half = DUAL ? warp >> 3 : 0;
    // B column g of a lane: token g, or a copy of a staged token for the
    // columns past the chunk (their results are never read)
    const int bn = ONE ? 0 : min(g, mts - 1);
    SvCursor cu = cursor_at(u0);
    for (int u = u0; u < u1 && ok; ++u, cursor_next(cu)) {
      if (cu.a != st_a || cu.c != st_c) {
        bool need = true;
        if (p.act_kind == kSvActX && st_a >= 0) {
          const int lo = act_lo[cu.a], m = act_m[cu.a];
          const int nt = min(mts, m - cu.c * mts);
          const int r0 = lo + cu.c * mts;
          need = nt != st_nt;
          for (int n = 0; n < nt && !need; ++n)
            need = (p.T == 1 ? 0 : __ldg(p.sorted + r0 + n) / p.kmax) != st_tok[n];
        }
        if (need && !stage_x(cu.a, cu.c)) {
          ok = false;
          break;
        }
        st_a = cu.a;
        st_c = cu.c;
      }
      const int wl = DUAL ? ((warp & 7) + u * rot_step) & 7 : (warp + u * rot_step) & (kSvConsumers - 1);
      const int jb = S::kGpw * wl;
      const int soff = rr * S::kScaleRow + jb * 2;
      // sums of s * P (P = 2^(e-24) sum q x) and of b * X, rows g and g + 8;
      // ONE: token 0 only, else tokens 2t and 2t + 1
      float as[4] = {0.0f, 0.0f, 0.0f, 0.0f}, ab[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      for (int ch = 0; ch < nck; ++ch) {
        if (abort_flag || !sv_wait(&full[ring.idx], ring.phase)) {
          ok = false;
          break;
        }
        const unsigned char* cst =
            codes + (size_t)ring.idx * kSvCodeBytes + half * 16384 + wl * 1024;
        const int g0 = ch * S::kGpc;
        const int nv = min(S::kGpw, ngroups - g0 - jb);  // this warp's groups in the stage
        if (nv > 0) {
          // scales and biases of rows g and g + 8 of the warp's groups, one load each
          const unsigned char* sp =
              scales + (size_t)ring.idx * kScaleStage + half * S::kScaleBytes + soff;
          typename S::ScaleVec sv[4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            sv[q] = *reinterpret_cast<const typename S::ScaleVec*>(sp + q * 8 * S::kScaleRow);
          const int G0 = g0 + jb;
          const uint4* xq = xs + (((size_t)G0 * 2 * mts + bn) * 4 + t);
          const float2* xsp = xsum + (size_t)G0 * mts2 + (ONE ? 0 : 2 * min(t, (mts2 >> 1) - 1));
          auto group = [&](int i) {
            // this lane's codes of rows g and g + 8 (128-byte swizzled boxes)
            uint32_t a0[S::kLaneWords], a1[S::kLaneWords];
            if constexpr (BITS == 4) {
              const uint2 v0 = *reinterpret_cast<const uint2*>(cst + coff[i]);
              const uint2 v1 = *reinterpret_cast<const uint2*>(cst + kHalfOff + coff[i]);
              a0[0] = v0.x;
              a0[1] = v0.y;
              a1[0] = v1.x;
              a1[1] = v1.y;
            } else {
              const uint4 v0 = *reinterpret_cast<const uint4*>(cst + coff[i]);
              const uint4 v1 = *reinterpret_cast<const uint4*>(cst + kHalfOff + coff[i]);
              a0[0] = v0.x;
              a0[1] = v0.y;
              a0[2] = v0.z;
              a0[3] = v0.w;
              a1[0] = v1.x;
              a1[1] = v1.y;
              a1[2] = v1.z;
              a1[3] = v1.w;
            }
            uint4 xb[2];
            const uint4* xqi = xq + (size_t)i * 2 * mts * 4;
            xb[0] = xqi[0];
            xb[1] = xqi[(size_t)mts * 4];
            // the words shifted right by 8 bits
            uint32_t a0h[S::kLaneWords], a1h[S::kLaneWords];
#pragma unroll
            for (int w = 0; w < S::kLaneWords; ++w) {
              a0h[w] = a0[w] >> 8;
              a1h[w] = a1[w] >> 8;
            }
            float d[4];
#pragma unroll
            for (int mm = 0; mm < 4; ++mm) {
              uint32_t af[4];
              if constexpr (BITS == 4) {
                // fp16 subnormal pairs: (q_m, q_{m+4}) 2^-24, odd m as 16 q
                const uint32_t mask = (mm & 1) ? 0x00F000F0u : 0x000F000Fu;
                af[0] = (mm >= 2 ? a0h[0] : a0[0]) & mask;
                af[1] = (mm >= 2 ? a1h[0] : a1[0]) & mask;
                af[2] = (mm >= 2 ? a0h[1] : a0[1]) & mask;
                af[3] = (mm >= 2 ? a1h[1] : a1[1]) & mask;
              } else {
                // 8-bit: bytes (c_r, c_{r+2}) of words 2p, 2p + 1
                const int pp = mm >> 1;
                af[0] = ((mm & 1) ? a0h[2 * pp] : a0[2 * pp]) & 0x00FF00FFu;
                af[1] = ((mm & 1) ? a1h[2 * pp] : a1[2 * pp]) & 0x00FF00FFu;
                af[2] = ((mm & 1) ? a0h[2 * pp + 1] : a0[2 * pp + 1]) & 0x00FF00FFu;
                af[3] = ((mm & 1) ? a1h[2 * pp + 1] : a1[2 * pp + 1]) & 0x00FF00FFu;
              }
              const uint4 bq = xb[mm >> 1];
              const uint32_t b0 = (mm & 1) ? bq.z : bq.x, b1 = (mm & 1) ? bq.w : bq.y;
              if (mm == 0)
                mma_sv0(d, af, b0, b1);
              else
                mma_sv(d, af, b0, b1);
            }
            const float s0 = sv_half(sv[0], i), s1 = sv_half(sv[1], i);
            const float b0 = sv_half(sv[2], i), b1 = sv_half(sv[3], i);
            if (ONE) {
              const float2 X = xsp[(size_t)i * mts2];  // (sum x, 2^(24-e))
              as[0] = fmaf(s0 * X.y, d[0], as[0]);
              as[2] = fmaf(s1 * X.y, d[2], as[2]);
              ab[0] = fmaf(b0, X.x, ab[0]);
              ab[2] = fmaf(b1, X.x, ab[2]);
            } else {
              const float4 X = *reinterpret_cast<const float4*>(xsp + (size_t)i * mts2);
              as[0] = fmaf(s0 * X.y, d[0], as[0]);
              as[1] = fmaf(s0 * X.w, d[1], as[1]);
              as[2] = fmaf(s1 * X.y, d[2], as[2]);
              as[3] = fmaf(s1 * X.w, d[3], as[3]);
              ab[0] = fmaf(b0, X.x, ab[0]);
              ab[1] = fmaf(b0, X.z, ab[1]);
              ab[2] = fmaf(b1, X.x, ab[2]);
              ab[3] = fmaf(b1, X.z, ab[3]);
            }
          };
          if (nv == S::kGpw) {
#pragma unroll
            for (int i = 0; i < S::kGpw; ++i) group(i);
          } else {
#pragma unroll
            for (int i = 0; i < S::kGpw; ++i)
              if (i < nv) group(i);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[ring.idx]);
        ring.next(stages);
      }
      if (!ok) break;
      // this warp's partial sums of the tile to the epilogue
      if (abort_flag || !sv_wait(&red_empty[rs.idx], rs.phase ^ 1u)) {
        ok = false;
        break;
      }
      float* rd = red + ((size_t)rs.idx * kSvConsumers + half * 8 + wl) * mts * 16;
      const int n0 = 2 * t, n1 = 2 * t + 1;
      if (n0 < mts) {
        rd[n0 * 16 + rr] = as[0] + ab[0];
        rd[n0 * 16 + 8 + rr] = as[2] + ab[2];
      }
      if (!ONE && n1 < mts) {
        rd[n1 * 16 + rr] = as[1] + ab[1];
        rd[n1 * 16 + 8 + rr] = as[3] + ab[3];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_full[rs.idx]);
      rs.next(rslots);
    }
    if (!ok && lane == 0) {
      raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
      abort_flag = 1;
    }
  } else if (warp == kSvEpilogue) {
    // ================================ epilogue ================================
    pdl_wait();
    SvRing rs{0, 0u};
    bool ok = true;
    SvCursor cu = cursor_at(u0);
    for (int u = u0; u < u1; ++u, cursor_next(cu)) {
      if (abort_flag) {
        ok = false;
        break;
      }
      const bool got = mbar_wait(&red_full[rs.idx], rs.phase, kWaitBudgetCycles);
      if (!__all_sync(0xFFFFFFFFu, got)) {
        ok = false;
        break;
      }
      const int m = act_m[cu.a];
      const int nt = min(mts, m - cu.c * mts);
      const int64_t row0 = (int64_t)act_lo[cu.a] + (int64_t)cu.c * mts;
      const float* rd = red + (size_t)rs.idx * kSvConsumers * mts * 16;
      // A row's value is (slot partials 0..7, added in order) + (slots
      // 8..15, in order), whatever rows and tokens share its tile.  DUAL:
      // half h's rows take slots 8h .. 8h + 7 in order (its rows are at most
      // 8 blocks, so the other slots of a 16-slot tile would hold zeros).
      if constexpr (DUAL) {
        if (ONE) {
          // lane l: half l >> 4, its row l & 15
          const int ri = lane & 15, hh = lane >> 4;
          float v = 0.0f;
#pragma unroll
          for (int w = 0; w < 8; ++w) v += rd[(hh * 8 + w) * 16 + ri];
          if (MODE == kSvSwiglu) {
            const float up = __shfl_sync(0xFFFFFFFFu, v, (lane & 16) | 8 | (lane & 7));
            const int col = cu.rt * 16 + hh * 8 + ri;
            if (ri < 8 && col < p.n_out) {
              const float hv = swiglu_f32(v, up);
              const int64_t oi = row0 * p.n_out + col;
              if (p.out_dtype == MOE_DTYPE_BF16)
                static_cast<uint16_t*>(p.out)[oi] = f32_to_bf16_rne(hv);
              else
                static_cast<float*>(p.out)[oi] = hv;
            }
          } else {
            const int col = cu.rt * 32 + hh * 16 + ri;
            if (col < p.n_rows) {
              const int64_t oi = row0 * p.n_out + col;
              if (p.out_dtype == MOE_DTYPE_BF16)
                static_cast<uint16_t*>(p.out)[oi] = f32_to_bf16_rne(v);
              else
                static_cast<float*>(p.out)[oi] = v;
            }
          }
        } else {
          // lane l: token l / 4, rows 4 (l & 3) .. + 3 of each half
          const int n = lane >> 2, q = lane & 3;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (n < nt) {
              const float4* r4 = reinterpret_cast<const float4*>(rd) + n * 4 + q;
#pragma unroll
              for (int w = 0; w < 8; ++w) {
                const float4 pl = r4[(size_t)(hh * 8 + w) * mts * 4];
                v.x += pl.x;
                v.y += pl.y;
                v.z += pl.z;
                v.w += pl.w;
              }
            }
            if (MODE == kSvSwiglu) {
              float4 up;
              up.x = __shfl_xor_sync(0xFFFFFFFFu, v.x, 2);
              up.y = __shfl_xor_sync(0xFFFFFFFFu, v.y, 2);
              up.z = __shfl_xor_sync(0xFFFFFFFFu, v.z, 2);
              up.w = __shfl_xor_sync(0xFFFFFFFFu, v.w, 2);
              const int col0 = cu.rt * 16 + hh * 8 + q * 4;
              if (n < nt && q < 2 && col0 < p.n_out) {
                const float4 hv = make_float4(swiglu_f32(v.x, up.x), swiglu_f32(v.y, up.y),
                                              swiglu_f32(v.z, up.z), swiglu_f32(v.w, up.w));
                const int64_t oi = (row0 + n) * p.n_out + col0;
                if (p.out_dtype == MOE_DTYPE_BF16)
                  *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + oi) = make_uint2(
                      (uint32_t)f32_to_bf16_rne(hv.x) | ((uint32_t)f32_to_bf16_rne(hv.y) << 16),
                      (uint32_t)f32_to_bf16_rne(hv.z) | ((uint32_t)f32_to_bf16_rne(hv.w) << 16));
                else
                  *reinterpret_cast<float4*>(static_cast<float*>(p.out) + oi) = hv;
              }
            } else {
              const int col0 = cu.rt * 32 + hh * 16 + q * 4;
              if (n < nt && col0 < p.n_rows) {
                const int64_t oi = (row0 + n) * p.n_out + col0;
                if (p.out_dtype == MOE_DTYPE_BF16)
                  *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + oi) = make_uint2(
                      (uint32_t)f32_to_bf16_rne(v.x) | ((uint32_t)f32_to_bf16_rne(v.y) << 16),
                      (uint32_t)f32_to_bf16_rne(v.z) | ((uint32_t)f32_to_bf16_rne(v.w) << 16));
                else
                  *reinterpret_cast<float4*>(static_cast<float*>(p.out) + oi) = v;
              }
            }
          }
        }
      } else if (ONE) {
        // lane l: tile row l & 15, slots 8 (l >> 4) .. + 7
        const int ri = lane & 15, wh = (lane >> 4) * 8;
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) v += rd[(wh + w) * 16 + ri];
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
        if (MODE == kSvSwiglu) {
          const float up = __shfl_sync(0xFFFFFFFFu, v, (lane & 7) + 8);
          const int col = cu.rt * 8 + lane;
          if (lane < 8 && col < p.n_out) {
            const float hv = swiglu_f32(v, up);
            const int64_t oi = row0 * p.n_out + col;
            if (p.out_dtype == MOE_DTYPE_BF16)
              static_cast<uint16_t*>(p.out)[oi] = f32_to_bf16_rne(hv);
            else
              static_cast<float*>(p.out)[oi] = hv;
          }
        } else {
          const int col = cu.rt * 16 + lane;
          if (lane < 16 && col < p.n_rows) {
            const int64_t oi = row0 * p.n_out + col;
            if (p.out_dtype == MOE_DTYPE_BF16)
              static_cast<uint16_t*>(p.out)[oi] = f32_to_bf16_rne(v);
            else
              static_cast<float*>(p.out)[oi] = v;
          }
        }
      } else {
        // lane l: token l / 4, tile rows 4 (l & 3) .. + 3
        const int n = lane >> 2, q = lane & 3;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (n < nt) {
          const float4* r4 = reinterpret_cast<const float4*>(rd) + n * 4 + q;
          float4 hi = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
          for (int w = 0; w < 8; ++w) {
            const float4 pl = r4[(size_t)w * mts * 4], ph = r4[(size_t)(w + 8) * mts * 4];
            v.x += pl.x;
            v.y += pl.y;
            v.z += pl.z;
            v.w += pl.w;
            hi.x += ph.x;
            hi.y += ph.y;
            hi.z += ph.z;
            hi.w += ph.w;
          }
          v.x += hi.x;
          v.y += hi.y;
          v.z += hi.z;
          v.w += hi.w;
        }
        if (MODE == kSvSwiglu) {
          // gate rows 0-7 in quads 0 and 1, the up rows of the same features
          // in quads 2 and 3
          float4 up;
          up.x = __shfl_xor_sync(0xFFFFFFFFu, v.x, 2);
          up.y = __shfl_xor_sync(0xFFFFFFFFu, v.y, 2);
          up.z = __shfl_xor_sync(0xFFFFFFFFu, v.z, 2);
          up.w = __shfl_xor_sync(0xFFFFFFFFu, v.w, 2);
          const int col0 = cu.rt * 8 + q * 4;
          if (n < nt && q < 2 && col0 < p.n_out) {
            const float4 hv = make_float4(swiglu_f32(v.x, up.x), swiglu_f32(v.y, up.y),
                                          swiglu_f32(v.z, up.z), swiglu_f32(v.w, up.w));
            const int64_t oi = (row0 + n) * p.n_out + col0;
            if (p.out_dtype == MOE_DTYPE_BF16)
              *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + oi) = make_uint2(
                  (uint32_t)f32_to_bf16_rne(hv.x) | ((uint32_t)f32_to_bf16_rne(hv.y) << 16),
                  (uint32_t)f32_to_bf16_rne(hv.z) | ((uint32_t)f32_to_bf16_rne(hv.w) << 16));
            else
              *reinterpret_cast<float4*>(static_cast<float*>(p.out) + oi) = hv;
          }
        } else {
          const int col0 = cu.rt * 16 + q * 4;
          if (n < nt && col0 < p.n_rows) {
            const int64_t oi = (row0 + n) * p.n_out + col0;
            if (p.out_dtype == MOE_DTYPE_BF16)
              *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + oi) = make_uint2(
                  (uint32_t)f32_to_bf16_rne(v.x) | ((uint32_t)f32_to_bf16_rne(v.y) << 16),
                  (uint32_t)f32_to_bf16_rne(v.z) | ((uint32_t)f32_to_bf16_rne(v.w) << 16));
            else
              *reinterpret_cast<float4*>(static_cast<float*>(p.out) + oi) = v;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_empty[rs.idx]);
      rs.next(rslots);
    }
    if (!ok && lane == 0) {
      raise_device_error(p.err, MOE_DEVERR_TIMEOUT);
      abort_flag = 1;
    }
  }
}

template <int BITS, int MODE, bool ONE, bool GATED, bool DUAL>
moe_status_t launch_stream_kernel(const CUtensorMap& tm, const SvParams& p, int smem,
                                  cudaStream_t st) {
  auto kern = gemv_stream_kernel<BITS, MODE, ONE, GATED, DUAL>;
  static int set_max[moe_host::kMaxCachedDevices] = {};  // per device
  const int dev = moe_host::device_index();
  if (smem > set_max[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    set_max[dev] = smem;
  }
  return moe_host::launch(kern, moe_host::sm_count(), kSvThreads, smem, st, tm, p);
}

template <int BITS, int MODE>
moe_status_t launch_stream(const CUtensorMap& tm, SvParams p, bool dual, cudaStream_t st) {
  static int optin = -1, static_smem = 0;
  if (optin < 0) {
    int dev = 0, v = 0;
    cudaFuncAttributes fa;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, gemv_stream_kernel<BITS, MODE, false, false, false>) !=
            cudaSuccess)
      return MOE_ERR_CUDA;
    static_smem = (int)fa.sharedSizeBytes;
    optin = v;
  }
  const long budget = (long)optin - static_smem - 1024;
  // tokens per pass: as many as fit beside at least 3 ring slots (a pass of
  // 8 tokens with 3 slots beats two passes of 4 with 4 slots: each pass
  // streams the expert's rows again)
  int stages = 0;
  for (;;) {
    stages = kSvMaxStages;
    while (stages >= 2 && (long)sv_layout(BITS, p.K, p.mts, stages, p.E, dual).total > budget)
      --stages;
    if (stages >= 3 || p.mts == 1) break;
    p.mts >>= 1;
  }
  if (stages < 2) return MOE_ERR_UNSUPPORTED;
  p.stages = stages;
  const int smem = (int)sv_layout(BITS, p.K, p.mts, stages, p.E, dual).total + 1024;
  if (p.gate.k != nullptr)
    return launch_stream_kernel<BITS, MODE, false, true, false>(tm, p, smem, st);
  if (dual)
    return p.mts == 1 ? launch_stream_kernel<BITS, MODE, true, false, true>(tm, p, smem, st)
                      : launch_stream_kernel<BITS, MODE, false, false, true>(tm, p, smem, st);
  return p.mts == 1 ? launch_stream_kernel<BITS, MODE, true, false, false>(tm, p, smem, st)
                    : launch_stream_kernel<BITS, MODE, false, false, false>(tm, p, smem, st);
}

}  // namespace

// 4- or 8-bit codes with rows a whole number of 128-byte blocks (K a multiple
// of 256 for 4-bit, 128 for 8-bit), E at most 1024.
bool gemv_stream_supported(int bits, int K, int E) {
  return (bits == 4 || bits == 8) && K % (bits == 4 ? 256 : 128) == 0 && E <= kSvMaxE &&
         tc_available();
}

moe_status_t gemv_stream_qmm(const void* act, int act_kind, const int32_t* sorted,
                             const int32_t* offsets, int T, int kmax, int E, int K, int n_rows,
                             bool swiglu, const uint32_t* wq, const uint16_t* ws,
                             const uint16_t* wb, int bits, void* out, int out_dtype, bool early,
                             KGate gate, cudaStream_t st) {
  if (!gemv_stream_supported(bits, K, E)) return MOE_ERR_UNSUPPORTED;
  if (!moe_host::aligned16(act) || !moe_host::aligned16(wq)) return MOE_ERR_INVALID_ARG;
  const int64_t A = (int64_t)T * kmax;
  if (A == 0) return MOE_OK;
  SvParams p;
  p.act = act;
  p.act_kind = act_kind;
  p.sorted = sorted;
  p.offsets = offsets;
  p.ws = ws;
  p.wb = wb;
  p.out = out;
  p.out_dtype = out_dtype;
  p.T = T;
  p.kmax = kmax;
  p.E = E;
  p.K = K;
  p.n_rows = n_rows;
  p.n_out = swiglu ? n_rows / 2 : n_rows;
  // rows of at most 8 blocks (ungated launches): 32-row tiles of two halves
  const uint64_t row_words = (uint64_t)K * bits / 32;
  const bool dual = row_words <= 8 * 32 && gate.k == nullptr;
  p.rt = swiglu ? (p.n_out + (dual ? 15 : 7)) / (dual ? 16 : 8)
                : (n_rows + (dual ? 31 : 15)) / (dual ? 32 : 16);
  // an expert's segment holds at most one row per token
  int mts = 1;
  while (mts < kSvMaxTokens && mts < T) mts <<= 1;
  p.mts = mts;
  p.stages = 0;
  const int ngroups = K / 64;
  const uintptr_t sa = reinterpret_cast<uintptr_t>(ws) | reinterpret_cast<uintptr_t>(wb);
  if (sa & 3u) return MOE_ERR_INVALID_ARG;
  p.scale_cw = (ngroups % 8 == 0 && (sa & 15u) == 0) ? 16
               : (ngroups % 4 == 0 && (sa & 7u) == 0) ? 8
                                                      : 4;
  p.early = early ? 1 : 0;
  p.gate = gate;
  p.err = moe_host::device_error_word();
  // tile count bound (int32 positions)
  const int64_t max_tiles = (int64_t)p.rt * (A + E);
  if (max_tiles >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
  // codes as [128-byte block][row][32 words]: boxes of 8 rows x 16 blocks
  // (a row's share of a stage), or 8 rows x 8 blocks for the DUAL tiles
  const uint64_t dims[3] = {32, (uint64_t)E * n_rows, row_words / 32};
  const uint64_t strides[2] = {row_words * 4, 128};
  const uint32_t box[3] = {32, 8, (uint32_t)(dual ? 8 : kSvBoxes)};
  CUtensorMap tm;
  if (!make_tensor_map_3d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT32, wq, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B))
    return MOE_ERR_CUDA;
  if (bits == 4)
    return swiglu ? launch_stream<4, kSvSwiglu>(tm, p, dual, st)
                  : launch_stream<4, kSvRaw>(tm, p, dual, st);
  return swiglu ? launch_stream<8, kSvSwiglu>(tm, p, dual, st)
                : launch_stream<8, kSvRaw>(tm, p, dual, st);
}

}  // namespace moe

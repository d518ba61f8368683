// Shared device helpers of libmoe_gb300 (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_gb300.h"

namespace moe {

constexpr int kGroup = 64;  // elements per scale/bias group

// Kernels report data problems (MOE_DEVERR_* bits) into the per-device error
// word whose address the launcher passes in; moe_get_device_error reads it.
__device__ __forceinline__ void raise_device_error(unsigned int* err, unsigned int bit) {
  if (err) atomicOr(err, bit);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t v16) {
  return __uint_as_float(v16 << 16);
}

// Two bf16 packed in one word -> two floats (low half first).
__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// fp32 -> bf16, round to nearest even (one hardware conversion).
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

// SiLU(gate) * up, the SwitchGLU activation, in fp32: g / (1 + e^-g) * u
// with the hardware exponential and reciprocal (a few ulp of fp32, far below
// the bf16 rounding of h that follows).  For g -> -inf, e^-g overflows to inf
// and the quotient is 0, the limit of SiLU.  Every path that produces h
// (fused epilogues and the separate swiglu kernel) calls this one function,
// so the fused and unfused results agree bit for bit.
__device__ __forceinline__ float swiglu_f32(float g, float u) {
  const float sig_den = __fadd_rn(1.0f, __expf(-g));
  return __fmul_rn(__fdividef(g, sig_den), u);
}

// Packed fp32x2 fused multiply-add (Blackwell FFMA2): d = a * b + c, lane-wise.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long ra, rb, rc, rd;
  asm("mov.b64 %0, {%1,%2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1,%2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1,%2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  float2 d;
  asm("mov.b64 {%0,%1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint16_t ldg_u16(const uint16_t* p) { return __ldg(p); }

// Programmatic dependent launch.  pdl_wait() returns once the kernel this
// one was launched behind has finished and its memory is visible (at once
// when there is no such dependency); every thread waits before it reads
// what an earlier kernel of the stream wrote or overwrites what one reads.
// pdl_trigger() lets the next kernel of the stream be scheduled before this
// one ends; it is called only after this kernel's own pdl_wait(), so a
// dependent that starts early still sees every kernel before this one done.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// A k-gated launch: the product runs only if lo <= *k (the routing k on the
// device) <= hi; otherwise its kernel returns at once.  An adaptive-k layer
// queues both kernel families, each gated on the k values it serves.
struct KGate {
  const int32_t* k;  // null: not gated
  int lo, hi;
};

// True if a gated kernel must return.  It waits for the previous kernel first
// (right away, or before returning when `early` lets it read k ahead of that
// wait), so whatever runs after it sees every earlier kernel completed.
__device__ __forceinline__ bool k_gate_closed(const int32_t* k, int lo, int hi, bool early) {
  if (k == nullptr) return false;
  if (!early) pdl_wait();
  const int kv = *reinterpret_cast<const volatile int32_t*>(k);
  if (kv >= lo && kv <= hi) return false;
  if (early) pdl_wait();
  return true;
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

}  // namespace moe

// Host-side helpers shared by the launchers.
namespace moe_host {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Streaming multiprocessor count of the current device (cached per device).
int sm_count();
// The current device's index, for per-device caches of launch settings
// (kernel attributes are set per device); 0 .. kMaxCachedDevices - 1.
constexpr int kMaxCachedDevices = 64;
int device_index();

// Device address of the current device's error word (nullptr on failure).
unsigned int* device_error_word();

inline moe_status_t launch_status() {
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Whether kernels are launched with programmatic stream serialization (the
// environment variable MOE_GB300_PDL=0 turns it off; read once).
bool pdl_enabled();

// Launch `kern` on `st`, allowed to start while the previous kernel of the
// stream finishes (when PDL is enabled); the kernel calls moe::pdl_wait()
// before it touches data of earlier kernels.
template <typename... KArgs, typename... Args>
inline moe_status_t launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace moe_host

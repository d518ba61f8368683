// C-ABI entry points of libmoe_gb300 that are not defined next to their
// kernels: status strings, the two quantized products (path selection and
// argument checks) and the device error word.
#include <atomic>
#include <cstdlib>
#include <mutex>

#include "async.cuh"
#include "common.cuh"

namespace moe {
moe_status_t gemv_qmm(const void* act, int act_kind, const int32_t* sorted,
                      const int32_t* offsets, int T, int kmax, int E, int K, int n_rows,
                      bool swiglu, const uint32_t* wq, const uint16_t* ws, const uint16_t* wb,
                      int bits, void* out, int out_dtype, bool early, KGate gate,
                      cudaStream_t st);
moe_status_t tc_qmm(const void* act, int act_kind, const int32_t* sorted,
                    const int32_t* offsets, int T, int kmax, int E, int K, int n_rows,
                    bool swiglu, const uint32_t* wq, const uint16_t* ws, const uint16_t* wb,
                    int bits, void* out, int out_dtype, KGate gate, cudaStream_t st);
moe_status_t gemv_bits_qmm(const void* act, int act_kind, const int32_t* sorted,
                           const int32_t* offsets, int T, int kmax, int E, int K, int n_rows,
                           bool swiglu, const uint32_t* wq, const uint16_t* ws, const uint16_t* wb,
                           int bits, void* out, int out_dtype, cudaStream_t st);
bool tc_available();
}  // namespace moe

namespace {

constexpr int kMaxDevices = 64;

// Per-device error word.  Kernels receive its address; it lives for the
// lifetime of the loaded module.
__device__ unsigned int g_moe_device_error;

struct DeviceCache {
  int sm = 0;
  unsigned int* err = nullptr;
};
DeviceCache g_cache[kMaxDevices];
std::mutex g_cache_mu;

DeviceCache& cache_for_current() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
  return g_cache[dev];
}

// Average tokens per expert above which the tensor-core path wins.
constexpr int kTcMinTokensPerExpert = 24;

}  // namespace

namespace moe_host {

int sm_count() {
  DeviceCache& c = cache_for_current();
  if (c.sm == 0) {
    std::lock_guard<std::mutex> lk(g_cache_mu);
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 1;
    c.sm = n;
  }
  return c.sm;
}

// -1 until first use: then the environment variable MOE_GB300_PDL ("0" turns
// programmatic dependent launch off), or the value moe_set_launch_overlap set.
std::atomic<int> g_pdl{-1};

bool pdl_enabled() {
  int v = g_pdl.load(std::memory_order_relaxed);
  if (v < 0) {
    const char* e = getenv("MOE_GB300_PDL");
    v = (e && e[0] == '0') ? 0 : 1;
    int expected = -1;
    g_pdl.compare_exchange_strong(expected, v);
    v = g_pdl.load(std::memory_order_relaxed);
  }
  return v != 0;
}

int device_index() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxCachedDevices) dev = 0;
  return dev;
}

unsigned int* device_error_word() {
  DeviceCache& c = cache_for_current();
  if (c.err == nullptr) {
    std::lock_guard<std::mutex> lk(g_cache_mu);
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_moe_device_error) == cudaSuccess)
      c.err = static_cast<unsigned int*>(p);
  }
  return c.err;
}

}  // namespace moe_host

extern "C" const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_INCOMPATIBLE: return "gate and up cannot be fused";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE: return "device-side check failed";
  }
  return "unknown status";
}

extern "C" int moe_abi_version(void) { return 2; }

extern "C" int moe_set_launch_overlap(int enable) {
  const int prev = moe_host::pdl_enabled() ? 1 : 0;
  moe_host::g_pdl.store(enable ? 1 : 0, std::memory_order_relaxed);
  return prev;
}

// The tensor-core path also needs rows of at least 128 code bytes (K * bits / 8)
// and 4- or 8-bit codes; 5- and 6-bit codes always take the GEMV family.
static int pick_path(int path, int T, int kmax, int E, int K, int bits) {
  if (path != MOE_PATH_AUTO) return path;
  if (bits != 4 && bits != 8) return MOE_PATH_GEMV;
  const int64_t per_expert = (int64_t)T * kmax / E;
  return (per_expert >= kTcMinTokensPerExpert && (int64_t)K * bits / 8 >= 128 &&
          moe::tc_available())
             ? MOE_PATH_TC
             : MOE_PATH_GEMV;
}

// `path` = kernel family (low byte) | MOE_PATH_FLAG_WEIGHTS_EARLY (where
// allowed) | an optional k gate (MOE_PATH_K_RANGE: explicit GEMV or TC only).
static bool split_path(int path, int kmax, const int32_t* k_dev, bool allow_early, int& family,
                       bool& early, moe::KGate& gate) {
  const unsigned u = (unsigned)path;
  const unsigned known = 0xFFu | MOE_PATH_FLAG_WEIGHTS_EARLY | MOE_PATH_FLAG_K_GATED |
                         (0xFFu << 16) | (0x7Fu << 24);
  if (u & ~known) return false;
  early = (u & MOE_PATH_FLAG_WEIGHTS_EARLY) != 0;
  if (early && !allow_early) return false;
  family = (int)(u & 0xFFu);
  if (family < MOE_PATH_AUTO || family > MOE_PATH_TC) return false;
  gate = moe::KGate{nullptr, 0, 0};
  if (u & MOE_PATH_FLAG_K_GATED) {
    const int lo = (int)((u >> 16) & 0xFFu), hi = (int)((u >> 24) & 0x7Fu);
    if (lo < 1 || hi < lo || hi > kmax) return false;
    if (family != MOE_PATH_GEMV && family != MOE_PATH_TC) return false;
    gate = moe::KGate{k_dev, lo, hi};
  } else if (u >> 16) {
    return false;  // a range without the flag
  }
  return true;
}

static bool common_shape_ok(int T, int kmax, int E) {
  return T >= 0 && kmax >= 1 && kmax <= 16 && E >= 1 && E <= 1024 &&
         (int64_t)T * kmax <= (1 << 24);
}

extern "C" moe_status_t moe_gate_up_qmm(const uint16_t* x, const int32_t* sorted_assign,
                                        const int32_t* expert_offsets, const int32_t* k_dev,
                                        int T, int kmax, int E, int H, int n_rows,
                                        const uint32_t* w_q, const uint16_t* w_s,
                                        const uint16_t* w_b, int bits, int epilogue,
                                        int out_dtype, void* out, int path,
                                        moe_stream_t stream) {
  using namespace moe_host;
  if (!common_shape_ok(T, kmax, E)) return MOE_ERR_INVALID_ARG;
  if (H <= 0 || H % 64 != 0 || n_rows <= 0 || n_rows % 64 != 0) return MOE_ERR_INVALID_ARG;
  if (bits != 4 && bits != 5 && bits != 6 && bits != 8) return MOE_ERR_UNSUPPORTED;
  if (epilogue != MOE_EPILOGUE_RAW && epilogue != MOE_EPILOGUE_SWIGLU) return MOE_ERR_INVALID_ARG;
  if (out_dtype != MOE_DTYPE_F32 && out_dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
  if (epilogue == MOE_EPILOGUE_RAW && out_dtype != MOE_DTYPE_F32) return MOE_ERR_UNSUPPORTED;
  if (epilogue == MOE_EPILOGUE_SWIGLU && n_rows % 2 != 0) return MOE_ERR_INVALID_ARG;
  int family = 0;
  bool early = false;
  moe::KGate gate{nullptr, 0, 0};
  if (!split_path(path, kmax, k_dev, false, family, early, gate)) return MOE_ERR_INVALID_ARG;
  if (H > 49152) return MOE_ERR_UNSUPPORTED;
  if (!expert_offsets || !k_dev) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  const void* ptrs[] = {x, w_q, w_s, w_b, out};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (sorted_assign && !aligned16(sorted_assign)) return MOE_ERR_INVALID_ARG;
  // x by token through sorted_assign (kind 0), or rows already in sorted order (kind 2)
  const int act_kind = sorted_assign ? 0 : 2;
  const bool swiglu = epilogue == MOE_EPILOGUE_SWIGLU;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int p = pick_path(family, T, kmax, E, H, bits);
  if (p == MOE_PATH_TC) {
    if (!moe::tc_available() || (bits != 4 && bits != 8)) return MOE_ERR_UNSUPPORTED;
    return moe::tc_qmm(x, act_kind, sorted_assign, expert_offsets, T, kmax, E, H, n_rows, swiglu,
                       w_q, w_s, w_b, bits, out, out_dtype, gate, st);
  }
  return moe::gemv_qmm(x, act_kind, sorted_assign, expert_offsets, T, kmax, E, H, n_rows, swiglu,
                       w_q, w_s, w_b, bits, out, out_dtype, false, gate, st);
}

extern "C" moe_status_t moe_down_qmm(const void* h, int h_dtype, const int32_t* expert_offsets,
                                     const int32_t* k_dev, int T, int kmax, int E, int I, int H,
                                     const uint32_t* w_q, const uint16_t* w_s,
                                     const uint16_t* w_b, int bits, void* y, int y_dtype,
                                     int path, moe_stream_t stream) {
  using namespace moe_host;
  if (!common_shape_ok(T, kmax, E)) return MOE_ERR_INVALID_ARG;
  if (I <= 0 || I % 64 != 0 || H <= 0 || H % 64 != 0) return MOE_ERR_INVALID_ARG;
  if (bits != 4 && bits != 5 && bits != 6 && bits != 8) return MOE_ERR_UNSUPPORTED;
  if (h_dtype != MOE_DTYPE_F32 && h_dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
  if (y_dtype != MOE_DTYPE_F32 && y_dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
  int family = 0;
  bool early = false;
  moe::KGate gate{nullptr, 0, 0};
  if (!split_path(path, kmax, k_dev, true, family, early, gate)) return MOE_ERR_INVALID_ARG;
  if (I > 49152) return MOE_ERR_UNSUPPORTED;
  if (!expert_offsets || !k_dev) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  const void* ptrs[] = {h, w_q, w_s, w_b, y};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  const int act_kind = h_dtype == MOE_DTYPE_F32 ? 1 : 2;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int p = pick_path(family, T, kmax, E, I, bits);
  if (p == MOE_PATH_TC) {
    if (!moe::tc_available() || (bits != 4 && bits != 8)) return MOE_ERR_UNSUPPORTED;
    return moe::tc_qmm(h, act_kind, nullptr, expert_offsets, T, kmax, E, I, H, false, w_q, w_s,
                       w_b, bits, y, y_dtype, gate, st);
  }
  return moe::gemv_qmm(h, act_kind, nullptr, expert_offsets, T, kmax, E, I, H, false, w_q, w_s,
                       w_b, bits, y, y_dtype, early, gate, st);
}

namespace {

// One thread waits on an mbarrier nothing arrives on, for at most `budget`
// cycles, with the library's bounded wait, and reports the timeout.
__global__ void wait_timeout_selftest_kernel(unsigned int* err, long long budget) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    moe::mbar_init(&bar, 1);
    moe::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !moe::mbar_wait(&bar, 0, budget))
    moe::raise_device_error(err, MOE_DEVERR_TIMEOUT);
}

}  // namespace

extern "C" moe_status_t moe_selftest_wait_timeout(uint32_t budget_cycles, moe_stream_t stream) {
  if (budget_cycles < 1 || budget_cycles > 100000000u) return MOE_ERR_INVALID_ARG;
  unsigned int* err = moe_host::device_error_word();
  if (!err) return MOE_ERR_CUDA;
  wait_timeout_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      err, (long long)budget_cycles);
  return moe_host::launch_status();
}

extern "C" moe_status_t moe_get_device_error(uint32_t* flags, int clear, moe_stream_t stream) {
  if (!flags) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  unsigned int* word = moe_host::device_error_word();
  if (!word) return MOE_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyAsync(&v, word, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (clear && cudaMemsetAsync(word, 0, sizeof v, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  *flags = v;
  return MOE_OK;
}

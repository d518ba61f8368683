// Memory-bound helpers of the layer: the weighted combine back to token order,
// the stand-alone SwitchGLU activation, and the gate/up concatenation.
#include <cuda_fp16.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kEwThreads = 256;

// out[t, m] = bf16( sum_{j<k} w[t, j] * y[inv_pos[t*kmax + j], m] ), fp32, j ascending.
// Page "Qwen3.5 Block在llama.cpp中的映射与优化原理", section 4.2 (weighted sum of
// the chosen experts' outputs).  One thread per V consecutive m of one token:
// V = 4 for fp32 y (one 16-byte load per row), 8 for bf16 y (also 16 bytes).
template <bool BF16_Y>
__global__ void __launch_bounds__(kEwThreads) combine_kernel(const void* __restrict__ y,
                                                             const int32_t* __restrict__ inv_pos,
                                                             const float* __restrict__ topk_w,
                                                             const int32_t* __restrict__ k_dev,
                                                             int T, int kmax, int H,
                                                             uint16_t* __restrict__ out,
                                                             unsigned int* err) {
  constexpr int V = BF16_Y ? 8 : 4;
  pdl_wait();
  pdl_trigger();
  const int k = *k_dev;
  const int vec_per_row = H / V;
  const int64_t total = (int64_t)T * vec_per_row;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / vec_per_row);
    const int v = (int)(i - (int64_t)t * vec_per_row);
    float acc[V];
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = 0.0f;
    // four slots at a time: their indices, weights and rows are all loaded
    // before the sums, which still run in ascending j
    constexpr int kJ = 4;
    for (int j0 = 0; j0 < k; j0 += kJ) {
      int r[kJ];
      float w[kJ];
      uint4 q[kJ];
#pragma unroll
      for (int jj = 0; jj < kJ; ++jj) {
        const int j = j0 + jj;
        r[jj] = j < k ? __ldg(inv_pos + (int64_t)t * kmax + j) : MOE_DROPPED;
        w[jj] = j < k ? __ldg(topk_w + (int64_t)t * kmax + j) : 0.0f;
      }
#pragma unroll
      for (int jj = 0; jj < kJ; ++jj) {
        q[jj] = make_uint4(0u, 0u, 0u, 0u);
        if (r[jj] >= 0) {
          if constexpr (BF16_Y)
            q[jj] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(y) +
                                                         (int64_t)r[jj] * H) + v);
          else
            q[jj] = __ldg(reinterpret_cast<const uint4*>(static_cast<const float*>(y) +
                                                         (int64_t)r[jj] * H) + v);
        } else if (r[jj] != MOE_DROPPED) {
          raise_device_error(err, MOE_DEVERR_BAD_INDEX);
        }
      }
#pragma unroll
      for (int jj = 0; jj < kJ; ++jj) {
        if (r[jj] < 0) continue;  // dropped by its expert's capacity, or past k
        float yv[V];
        const uint32_t q4[4] = {q[jj].x, q[jj].y, q[jj].z, q[jj].w};
        if constexpr (BF16_Y) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            yv[2 * e] = __uint_as_float(q4[e] << 16);
            yv[2 * e + 1] = __uint_as_float(q4[e] & 0xFFFF0000u);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) yv[e] = __uint_as_float(q4[e]);
        }
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = fmaf(w[jj], yv[e], acc[e]);
      }
    }
    uint32_t o[V / 2];
#pragma unroll
    for (int e = 0; e < V / 2; ++e)
      o[e] = (uint32_t)f32_to_bf16_rne(acc[2 * e]) | ((uint32_t)f32_to_bf16_rne(acc[2 * e + 1]) << 16);
    if constexpr (BF16_Y)
      reinterpret_cast<uint4*>(out + (int64_t)t * H)[v] = make_uint4(o[0], o[1], o[2], o[3]);
    else
      reinterpret_cast<uint2*>(out + (int64_t)t * H)[v] = make_uint2(o[0], o[1]);
  }
}

// h[r, n] = SiLU(gate[r, n]) * up[r, n] for rows r < T*k.
__global__ void __launch_bounds__(kEwThreads) swiglu_kernel(const float* __restrict__ gate,
                                                            const float* __restrict__ up,
                                                            const int32_t* __restrict__ k_dev,
                                                            int T, int I, int out_dtype,
                                                            void* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t rows = (int64_t)T * (*k_dev);
  const int64_t total = rows * I;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float h = swiglu_f32(__ldg(gate + i), __ldg(up + i));
    if (out_dtype == MOE_DTYPE_BF16)
      static_cast<uint16_t*>(out)[i] = f32_to_bf16_rne(h);
    else
      static_cast<float*>(out)[i] = h;
  }
}

// Concatenate per expert: dst[e] = [src_a[e]; src_b[e]], each block `blk` bytes.
__global__ void __launch_bounds__(kEwThreads) concat_kernel(const uint4* __restrict__ a,
                                                            const uint4* __restrict__ b,
                                                            uint4* __restrict__ dst, int E,
                                                            int64_t blk16) {
  const int64_t total = (int64_t)E * 2 * blk16;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = i / (2 * blk16);
    const int64_t r = i - e * 2 * blk16;
    dst[i] = r < blk16 ? a[e * blk16 + r] : b[e * blk16 + (r - blk16)];
  }
}

int grid_for(int64_t work) {
  const int64_t per_cta = kEwThreads;
  int64_t g = (work + per_cta - 1) / per_cta;
  const int64_t cap = (int64_t)moe_host::sm_count() * 8;
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_combine(const void* y, int y_dtype, const int32_t* inv_pos,
                                    const float* topk_w, const int32_t* k_dev, int T, int kmax,
                                    int H, uint16_t* out, moe_stream_t stream) {
  using namespace moe_host;
  if (T < 0 || H <= 0 || H % 64 != 0 || kmax < 1 || kmax > 16) return MOE_ERR_INVALID_ARG;
  if ((int64_t)T * kmax > (1 << 24)) return MOE_ERR_INVALID_ARG;
  if (y_dtype != MOE_DTYPE_F32 && y_dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
  if (!k_dev) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!y || !inv_pos || !topk_w || !out || !aligned16(y) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (y_dtype == MOE_DTYPE_BF16)
    return launch(combine_kernel<true>, grid_for((int64_t)T * H / 8), kEwThreads, 0, st, y,
                  inv_pos, topk_w, k_dev, T, kmax, H, out, device_error_word());
  return launch(combine_kernel<false>, grid_for((int64_t)T * H / 4), kEwThreads, 0, st, y,
                inv_pos, topk_w, k_dev, T, kmax, H, out, device_error_word());
}

extern "C" moe_status_t moe_swiglu(const float* gate, const float* up, const int32_t* k_dev,
                                   int T, int kmax, int I, int out_dtype, void* out,
                                   moe_stream_t stream) {
  using namespace moe_host;
  if (T < 0 || I <= 0 || I % 64 != 0 || kmax < 1 || kmax > 16) return MOE_ERR_INVALID_ARG;
  if ((int64_t)T * kmax > (1 << 24)) return MOE_ERR_INVALID_ARG;
  if (out_dtype != MOE_DTYPE_F32 && out_dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
  if (!k_dev) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!gate || !up || !out || !aligned16(gate) || !aligned16(up) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  return launch(swiglu_kernel, grid_for((int64_t)T * kmax * I), kEwThreads, 0,
                reinterpret_cast<cudaStream_t>(stream), gate, up, k_dev, T, I, out_dtype, out);
}

extern "C" moe_status_t moe_pack_gate_up(const moe_qdesc_t* gd, const moe_qdesc_t* ud,
                                         const uint32_t* gate_q, const uint16_t* gate_s,
                                         const uint16_t* gate_b, const uint32_t* up_q,
                                         const uint16_t* up_s, const uint16_t* up_b, int E,
                                         uint32_t* gu_q, uint16_t* gu_s, uint16_t* gu_b,
                                         moe_stream_t stream) {
  using namespace moe_host;
  if (!gd || !ud || E < 1) return MOE_ERR_INVALID_ARG;
  // Eligibility, page "oMLX MoE gate/up 融合优化：qwen35_moe_gate_up 实现剖析",
  // 实现剖析 ②: same projection type, group size, bits and mode, same presence
  // of a bias, same shape and dtype -- otherwise the layer stays unfused.
  if (gd->quantized != ud->quantized || gd->bits != ud->bits ||
      gd->group_size != ud->group_size || gd->mode != ud->mode || gd->has_bias != ud->has_bias ||
      gd->rows != ud->rows || gd->cols != ud->cols || gd->scale_dtype != ud->scale_dtype)
    return MOE_ERR_INCOMPATIBLE;
  if (gd->quantized != 1 || (gd->bits != 4 && gd->bits != 5 && gd->bits != 6 && gd->bits != 8) ||
      gd->group_size != 64 ||
      gd->mode != MOE_QMODE_AFFINE || gd->has_bias != 0 || gd->scale_dtype != MOE_SCALE_F16)
    return MOE_ERR_UNSUPPORTED;
  const int I = gd->rows, H = gd->cols;
  if (I <= 0 || H <= 0 || I % 64 != 0 || H % 64 != 0) return MOE_ERR_INVALID_ARG;
  const void* ptrs[9] = {gate_q, gate_s, gate_b, up_q, up_s, up_b, gu_q, gu_s, gu_b};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t q_blk = (int64_t)I * H * gd->bits / 8;   // bytes of one expert's codes
  const int64_t s_blk = (int64_t)I * (H / 64) * 2;       // bytes of one expert's scales
  concat_kernel<<<grid_for(E * 2 * q_blk / 16), kEwThreads, 0, st>>>(
      reinterpret_cast<const uint4*>(gate_q), reinterpret_cast<const uint4*>(up_q),
      reinterpret_cast<uint4*>(gu_q), E, q_blk / 16);
  if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
  concat_kernel<<<grid_for(E * 2 * s_blk / 16), kEwThreads, 0, st>>>(
      reinterpret_cast<const uint4*>(gate_s), reinterpret_cast<const uint4*>(up_s),
      reinterpret_cast<uint4*>(gu_s), E, s_blk / 16);
  if (launch_status() != MOE_OK) return MOE_ERR_CUDA;
  concat_kernel<<<grid_for(E * 2 * s_blk / 16), kEwThreads, 0, st>>>(
      reinterpret_cast<const uint4*>(gate_b), reinterpret_cast<const uint4*>(up_b),
      reinterpret_cast<uint4*>(gu_b), E, s_blk / 16);
  return launch_status();
}

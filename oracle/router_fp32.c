/*
 * Oracle: router logits of the sparse-MoE layer in fp32 with one fixed
 * summation order.  TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).
 *
 * The router is a bias-free linear layer, logits[t, e] = x[t] . W[e]
 * (page "Qwen3.5 Block在llama.cpp中的映射与优化原理", section 4.1: the
 * router is a linear layer followed by a softmax and a top-k).  Top-k picks
 * expert ids from these logits, so the ids are only reproducible if every
 * implementation adds the H products in the same order.  The order fixed
 * for this layer is:
 *   - split the H products into chunks of 8 consecutive elements; chunk c
 *     belongs to partial sum p[c mod 32];
 *   - each partial sum starts at +0 and takes its chunks in ascending order,
 *     elements in ascending order, one fused multiply-add (fmaf, a single
 *     rounding) per product;
 *   - the 32 partial sums are combined pairwise: for off = 16, 8, 4, 2, 1,
 *     p[l] <- p[l] + p[l xor off]; the result is p[0];
 *   - then the optional per-expert logit bias is added, and the sum is
 *     multiplied by the inverse temperature.
 * Written plainly, one product at a time.  Compile without FP contraction.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static float bf16_to_f32(uint16_t v) {
  uint32_t u = (uint32_t)v << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

int oracle_router_logits(const uint16_t* x, const float* w, const float* logit_bias,
                         float inv_temperature, int T, int H, int E, float* logits) {
  if (H % 8 != 0 || T < 0 || E <= 0) return -1;
  const int nchunks = H / 8;
  for (int t = 0; t < T; ++t) {
    const uint16_t* xt = x + (int64_t)t * H;
    for (int e = 0; e < E; ++e) {
      const float* we = w + (int64_t)e * H;
      float p[32];
      for (int l = 0; l < 32; ++l) {
        float acc = 0.0f;
        for (int c = l; c < nchunks; c += 32)
          for (int i = 0; i < 8; ++i) {
            int h = 8 * c + i;
            acc = fmaf(bf16_to_f32(xt[h]), we[h], acc);
          }
        p[l] = acc;
      }
      for (int off = 16; off >= 1; off >>= 1) {
        float q[32];
        for (int l = 0; l < 32; ++l) q[l] = p[l] + p[l ^ off];
        memcpy(p, q, sizeof p);
      }
      float v = p[0];
      if (logit_bias) v = v + logit_bias[e];
      v = v * inv_temperature;
      logits[(int64_t)t * E + e] = v;
    }
  }
  return 0;
}

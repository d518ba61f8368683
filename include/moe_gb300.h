/*
 * moe_gb300.h -- C ABI of libmoe_gb300.so, the forward pass of a quantized
 * sparse-MoE SwitchGLU layer on one GB300 GPU (sm_103a).
 *
 * The layer, for T tokens x[T, H], E experts and k experts per token:
 *   1. router logits  l = x . W_r^T (+ logit bias) * inverse temperature
 *   2. softmax, top-k expert ids and routing weights; k is fixed or picked
 *      per batch from the mean softmax entropy (top-1/2/3)
 *   3. the (token, slot) assignments grouped by expert
 *   4. one product with the concatenated [gate; up] affine-quantized matrix
 *      of each expert, then h = SiLU(gate) * up
 *   5. the down projection y = h . W_d^T
 *   6. out[t] = sum_j w[t, j] * y[t, j]
 *
 * Pages the declarations cite:
 *   [A] "Qwen3.5 Block在llama.cpp中的映射与优化原理" (mokono.cn/news/2993189)
 *   [B] "Qwen3.5-MoE与Qwen3-MoE架构差异深度解析" (jsqmd.com/news/1062166)
 *   [C] "oMLX MoE gate/up 融合优化：qwen35_moe_gate_up 实现剖析" (xdnf.cn/news/169715)
 *
 * Conventions shared by every call
 * --------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller; the library
 *   never allocates, frees or retains them.  Calls enqueue work on `stream`
 *   (a cudaStream_t passed as void*; NULL = the legacy default stream) and
 *   return without synchronizing, except moe_get_device_error.
 * - Arguments are checked before anything is launched; a failed check
 *   returns an error code and enqueues nothing.  A launch failure returns
 *   MOE_ERR_CUDA.  Problems found by the kernels themselves (an expert id
 *   out of range, a bounded wait that ran out) set bits of a per-device
 *   error word, read with moe_get_device_error.
 * - Tensors are dense, row-major, with the shapes given below.  Every
 *   pointer must be 16-byte aligned.
 * - bf16 and fp16 values travel as their raw 16-bit patterns (uint16_t).
 * - Packed codes: a row of `cols` b-bit codes (b = 4, 5, 6 or 8) is one
 *   little-endian bit stream over uint32 words: element i occupies bits
 *   [b*i, b*i + b) of the row (for 4 and 8 bits: word i/(32/b), bit
 *   b*(i mod (32/b))).  A group of 64 codes is 2b whole words.  5- and 6-bit
 *   codes take the GEMV family only (MOE_PATH_TC returns MOE_ERR_UNSUPPORTED)
 *   and no k gate.
 *   Dequantized weight = scale * code + bias, where scale and bias are fp16
 *   and shared by 64 consecutive elements of the row (group size 64 along
 *   the contraction axis).  Page [C], section 融合原理.
 * - Limits: H % 64 == 0, I % 64 == 0, 1 <= E <= 1024, 1 <= kmax <= 16,
 *   0 <= T, T * kmax <= 2^24.
 * - Assignment numbering: slot j of token t is assignment a = t*kmax + j.
 *   Only slots j < k (k read from the device scalar k_dev) exist.  After
 *   moe_permute, "sorted row r" is the r-th assignment in expert-grouped
 *   order (r < T*k).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null/misaligned pointer or shape outside the limits */
  MOE_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement */
  MOE_ERR_INCOMPATIBLE = 3, /* gate and up cannot be fused (moe_pack_gate_up) */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  MOE_ERR_TIMEOUT = 5,      /* a bounded device-side wait ran out */
  MOE_ERR_DEVICE = 6        /* a kernel rejected its data (see moe_get_device_error) */
} moe_status_t;

enum { MOE_DTYPE_F32 = 0, MOE_DTYPE_BF16 = 1 };
enum { MOE_EPILOGUE_RAW = 0, MOE_EPILOGUE_SWIGLU = 1 };
/* Kernel family for the two quantized products. */
enum {
  MOE_PATH_AUTO = 0, /* chosen from the mean tokens per expert, T*kmax/E */
  MOE_PATH_GEMV = 1, /* CUDA-core grouped GEMV: decode and small batches */
  MOE_PATH_TC = 2    /* tcgen05 grouped GEMM (TMEM accumulators), many tokens per expert */
};
/* ------------------------------------------------------------------------
 * moe_set_launch_overlap -- whether later launches of this library may
 * overlap the end of the previous kernel of their stream (programmatic
 * dependent launch, on by default; the environment variable MOE_GB300_PDL=0
 * sets the default off).  Results do not depend on it; per-kernel timings
 * taken with events between kernels are cleaner with it off.  Returns the
 * previous setting.  Not synchronized with launches in flight on other
 * threads.
 * ---------------------------------------------------------------------- */
int moe_set_launch_overlap(int enable);

/* Flag OR-ed into the `path` argument of moe_down_qmm.  Kernels of this
 * library are launched with programmatic stream serialization: a kernel may
 * start while the previous kernel of the stream finishes, and waits for it
 * before it reads activations or writes results.  With this flag the down
 * product also reads expert_offsets and streams its weights before that
 * wait.  Set it only when the kernel issued just before the call on the
 * stream writes neither expert_offsets nor the down weights (in the layer
 * sequence that kernel is the gate_up product). */
enum { MOE_PATH_FLAG_WEIGHTS_EARLY = 0x100 };
/* k-gated launch, OR-ed into the `path` of moe_gate_up_qmm or moe_down_qmm
 * with an explicit MOE_PATH_GEMV or MOE_PATH_TC: the product runs only if
 * lo <= *k_dev <= hi (1 <= lo <= hi <= kmax); otherwise its kernel returns
 * without reading or writing anything but k_dev.  It still waits for the
 * kernel ahead of it on the stream, so the stream's order holds.  With the
 * adaptive k of page [B] section 2.2 the host does not know k when it
 * queues a layer; queuing both kernel families, each gated on the k values
 * it is faster for, lets the device pick per call without a host round trip.
 * Only the streamed GEMV (4-bit K a multiple of 256, 8-bit of 128) and the
 * tensor-core kernel take a gate (else MOE_ERR_UNSUPPORTED). */
enum { MOE_PATH_FLAG_K_GATED = 0x200 };
#define MOE_PATH_K_RANGE(lo, hi) (MOE_PATH_FLAG_K_GATED | ((lo) << 16) | ((hi) << 24))
/* Device error word bits (moe_get_device_error). */
enum { MOE_DEVERR_BAD_EXPERT = 1u, MOE_DEVERR_TIMEOUT = 2u, MOE_DEVERR_BAD_INDEX = 4u };
/* inv_pos value of an assignment that its expert's capacity turned away
 * (moe_permute_capped); moe_combine skips it. */
enum { MOE_DROPPED = -2 };

typedef void* moe_stream_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* moe_status_string(moe_status_t status);

/* Version of this ABI; bumps on any incompatible change. */
int moe_abi_version(void);

/* ------------------------------------------------------------------------
 * moe_pack_gate_up -- fuse an expert layer's gate and up projections.
 *
 * Page [C], 融合原理 and 实现剖析 ② ③: the codes, scales and biases of gate
 * and up are concatenated along the OUTPUT axis, gate first, so that one
 * product with the [E, 2*I, H] matrix yields both halves; because affine
 * codes carry their scale and bias per output row, the fused product equals
 * the two separate ones bit for bit.  Fusion is allowed only when gate and
 * up describe the same kind of projection: same quantized flag, bits, group
 * size and mode, same presence of a linear bias, same shape and scale dtype.
 *
 * gate_desc, up_desc  host pointers to the two descriptors.
 * gate_q, up_q        uint32 [E, I, H*bits/32] codes.
 * gate_s/b, up_s/b    fp16 [E, I, H/64] scales and biases.
 * gu_q                out: uint32 [E, 2*I, H*bits/32]; rows [0, I) gate,
 *                     rows [I, 2I) up, per expert.
 * gu_s, gu_b          out: fp16 [E, 2*I, H/64].
 * Returns MOE_ERR_INCOMPATIBLE (nothing written) when the descriptors
 * differ -- the caller keeps the unfused path; MOE_ERR_UNSUPPORTED for a
 * descriptor this library cannot run (not quantized, bits not 4/5/6/8, group
 * not 64, mode not affine, a linear bias, scale dtype not fp16).
 * ---------------------------------------------------------------------- */
enum { MOE_QMODE_AFFINE = 0 };
enum { MOE_SCALE_F16 = 0, MOE_SCALE_BF16 = 1, MOE_SCALE_F32 = 2 };
typedef struct moe_qdesc {
  int32_t quantized;   /* 1 = affine-quantized projection, 0 = dense */
  int32_t bits;        /* code width */
  int32_t group_size;  /* elements sharing one scale/bias */
  int32_t mode;        /* MOE_QMODE_* */
  int32_t has_bias;    /* projection has a linear bias */
  int32_t rows;        /* output features (I) */
  int32_t cols;        /* input features (H) */
  int32_t scale_dtype; /* MOE_SCALE_* */
} moe_qdesc_t;

moe_status_t moe_pack_gate_up(const moe_qdesc_t* gate_desc, const moe_qdesc_t* up_desc,
                              const uint32_t* gate_q, const uint16_t* gate_s,
                              const uint16_t* gate_b, const uint32_t* up_q,
                              const uint16_t* up_s, const uint16_t* up_b, int E,
                              uint32_t* gu_q, uint16_t* gu_s, uint16_t* gu_b,
                              moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_router_topk -- router logits, softmax, top-k ids and weights, and the
 * batch's k.
 *
 * Page [A], section 4.1: logits = linear(x, W_r) without bias, softmax over
 * experts, top-k.  Page [B], sections 2.1-2.2: top-k routing; in adaptive
 * mode one k per batch from the Shannon entropy of the routing distribution:
 * mean over tokens of H_t = -sum_e p_te ln p_te (nats, softmax over all E
 * after bias and temperature); H < thr1 -> 1, thr1 <= H < thr2 -> 2,
 * otherwise 3 (the page's thresholds are 1.2 and 2.5).
 *
 * Logits are fp32 with one fixed summation order so that ids are exactly
 * reproducible: chunks of 8 consecutive h go round-robin to 32 partial sums
 * (chunk c -> partial c mod 32), each accumulated in ascending h with
 * single-rounding fused multiply-adds from +0; the partials are combined by
 * p[l] += p[l xor o] for o = 16, 8, 4, 2, 1; then + logit_bias[e], then
 * * inv_temperature.  The k largest logits are chosen (equal logits: lower
 * expert id first), largest first.  Weight j = exp(l_j - max)/D with D the
 * sum over the chosen k (renormalize = 1) or over all E (renormalize = 0).
 *
 * x            bf16 [T, H].
 * w_router     fp32 [E, H].
 * logit_bias   fp32 [E], or NULL.
 * k_fixed      1..kmax, or 0 for the adaptive rule (needs kmax >= 3).
 * topk_ids     out: int32 [T, kmax]; slots j >= k hold -1.
 * topk_w       out: fp32 [T, kmax]; slots j >= k hold 0.
 * k_dev        out: int32 scalar, the batch's k (read by later calls).
 * mean_entropy out: fp32 scalar, the batch-mean entropy (0 when T = 0).
 * workspace    device scratch of moe_router_workspace_size(T) bytes.
 * ---------------------------------------------------------------------- */
size_t moe_router_workspace_size(int T);

moe_status_t moe_router_topk(const uint16_t* x, const float* w_router, const float* logit_bias,
                             float inv_temperature, int T, int H, int E, int k_fixed, int kmax,
                             float thr1, float thr2, int renormalize, int32_t* topk_ids,
                             float* topk_w, int32_t* k_dev, float* mean_entropy,
                             void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_router_topk_noalloc -- moe_router_topk for callers that cannot
 * allocate device memory.
 *
 * No page describes this call; it exists for integration only.  Some callers
 * cannot get device memory on demand: a model runner that reserves the whole
 * device pool at start-up and gives a plugged-in layer only its input and
 * output tensors, or a deployment that forbids allocation after start-up
 * because cudaMalloc can synchronize the device in the middle of a
 * latency-bound decode loop.  This call takes no workspace; its scratch is a
 * static device array inside the library holding 2 floats per token for up
 * to MOE_ROUTER_NOALLOC_MAX_TOKENS tokens (512 KiB), kept by every GPU that
 * loads the library until the process exits.  It allocates nothing.
 *
 * Arguments, outputs and results are those of moe_router_topk without
 * workspace/workspace_bytes.  T > MOE_ROUTER_NOALLOC_MAX_TOKENS returns
 * MOE_ERR_INVALID_ARG and launches nothing.  The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress) with that
 * device current; make that first call before any stream capture.  All calls
 * share the array: calls whose executions overlap on the GPU race, so the
 * caller must order them (one stream, or events).  Nothing in the array
 * needs clearing between calls.  The looked-up address belongs to the
 * device's current context: after cudaDeviceReset the library's cached
 * device addresses (this array's and the error word's of
 * moe_get_device_error) are stale, so no entry point of the library may be
 * called on that device again in the same process.
 * ---------------------------------------------------------------------- */
#define MOE_ROUTER_NOALLOC_MAX_TOKENS 65536

moe_status_t moe_router_topk_noalloc(const uint16_t* x, const float* w_router,
                                     const float* logit_bias, float inv_temperature, int T,
                                     int H, int E, int k_fixed, int kmax, float thr1, float thr2,
                                     int renormalize, int32_t* topk_ids, float* topk_w,
                                     int32_t* k_dev, float* mean_entropy, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_permute -- group the assignments by expert (stable counting sort).
 *
 * Page [C], 如何验证正确性 (the sorted branch that groups token indices by
 * expert before the gathered product) and page [B], section 4.2 (per-expert
 * activation counts).  For each expert e in id order, the assignments
 * a = t*kmax + j (j < k) routed to e, in ascending a.
 *
 * topk_ids        int32 [T, kmax] (from moe_router_topk).
 * k_dev           int32 scalar.
 * expert_counts   out: int32 [E].
 * expert_offsets  out: int32 [E+1], exclusive prefix sum of the counts.
 * sorted_assign   out: int32 [T*kmax]; entries [0, T*k) hold the grouped
 *                 assignments, the rest is left untouched.
 * inv_pos         out: int32 [T*kmax]; inv_pos[a] = sorted row of a, or -1
 *                 for slots j >= k.
 * An id outside [0, E) is skipped and sets MOE_DEVERR_BAD_EXPERT.
 * ---------------------------------------------------------------------- */
moe_status_t moe_permute(const int32_t* topk_ids, const int32_t* k_dev, int T, int kmax, int E,
                         int32_t* expert_counts, int32_t* expert_offsets,
                         int32_t* sorted_assign, int32_t* inv_pos, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_permute_capped -- moe_permute with an expert capacity.
 *
 * Page [B], sections 4.3 and 5.2 (expert_capacity: a limit on the tokens an
 * expert takes per batch).  Each expert keeps at most `capacity` of its
 * assignments, those of the lowest a = t*kmax + j, in the same stable order
 * as moe_permute; the others get inv_pos = MOE_DROPPED, contribute nothing
 * to the combine, and the kept weights are not renormalised.
 * expert_counts and expert_offsets describe the kept assignments only;
 * sorted_assign entries past offsets[E] (up to T*k) hold 0, a valid
 * assignment, so consumers of T*k sorted rows stay in bounds.
 * capacity >= 0 (0 drops everything).
 * ---------------------------------------------------------------------- */
moe_status_t moe_permute_capped(const int32_t* topk_ids, const int32_t* k_dev, int T, int kmax,
                                int E, int capacity, int32_t* expert_counts,
                                int32_t* expert_offsets, int32_t* sorted_assign,
                                int32_t* inv_pos, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_route -- moe_router_topk followed by moe_permute, as one call.
 *
 * The two calls above in sequence (their passages), with their arguments and
 * outputs.  When one cluster of the router covers the batch (T <= 32 tokens
 * for E <= 256), E <= 256 and T*kmax <= 512, the router's leader CTA sorts
 * the assignments itself once the batch's k is known: one launch instead of
 * two, the same outputs bit for bit.  Otherwise the two kernels are launched
 * one after the other.  Argument errors of either call return
 * MOE_ERR_INVALID_ARG before anything is launched.
 * ---------------------------------------------------------------------- */
moe_status_t moe_route(const uint16_t* x, const float* w_router, const float* logit_bias,
                       float inv_temperature, int T, int H, int E, int k_fixed, int kmax,
                       float thr1, float thr2, int renormalize, int32_t* topk_ids, float* topk_w,
                       int32_t* k_dev, float* mean_entropy, void* workspace,
                       size_t workspace_bytes, int32_t* expert_counts, int32_t* expert_offsets,
                       int32_t* sorted_assign, int32_t* inv_pos, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_route_grouped -- moe_route with group-limited selection.
 *
 * Page [A], section 1.1: the E experts form n_groups groups of E / n_groups
 * consecutive ids and each token takes the best expert of every group, so
 * k = n_groups.  Within a group the larger logit wins, equal logits go to
 * the lower id; the chosen ids are listed larger logit first (equal logits:
 * lower id first), as moe_router_topk lists its top-k.  Weights, entropy,
 * k_dev and the expert grouping are those of moe_route with k_fixed =
 * n_groups.  E must be a multiple of n_groups and n_groups <= kmax <= 16.
 * ---------------------------------------------------------------------- */
moe_status_t moe_route_grouped(const uint16_t* x, const float* w_router, const float* logit_bias,
                               float inv_temperature, int T, int H, int E, int n_groups,
                               int kmax, int renormalize, int32_t* topk_ids, float* topk_w,
                               int32_t* k_dev, float* mean_entropy, void* workspace,
                               size_t workspace_bytes, int32_t* expert_counts,
                               int32_t* expert_offsets, int32_t* sorted_assign,
                               int32_t* inv_pos, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_permute_rows -- the token rows in expert order.
 *
 * Page [C], 如何验证正确性 (the sorted branch: token rows are gathered into
 * expert order before the gathered product).  x_sorted[r] = x[t] with
 * t = sorted_assign[r] / kmax, for sorted rows r < T*k; an exact copy.
 *
 * x               bf16 [T, H] (H a multiple of 8), 16-byte aligned.
 * sorted_assign   int32 [T*kmax] from moe_permute.
 * k_dev           int32 scalar (clamped to [0, kmax]).
 * x_sorted        out: bf16 [T*kmax, H], 16-byte aligned; rows >= T*k are
 *                 not written.  The caller owns all buffers.
 * An entry outside [0, T*kmax) leaves its row unwritten and sets
 * MOE_DEVERR_BAD_INDEX.
 * ---------------------------------------------------------------------- */
moe_status_t moe_permute_rows(const uint16_t* x, const int32_t* sorted_assign,
                              const int32_t* k_dev, int T, int kmax, int H, uint16_t* x_sorted,
                              moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_gate_up_qmm -- the fused gate_up product over expert segments.
 *
 * Page [C], 融合原理 and 实现剖析 ④: one gathered quantized product with the
 * [gate; up] matrix instead of two, split into halves, then the SwitchGLU
 * activation SiLU(gate) * up, SiLU(z) = z / (1 + exp(-z)); page [A], section
 * 4.2: only the experts a token was routed to are evaluated.
 *
 * For sorted row r (expert e, token t = sorted_assign[r] / kmax) and matrix
 * row n: acc[r, n] = sum_h x[t, h] * (s[e, n, h/64] * code[e, n, h] +
 * b[e, n, h/64]) in fp32.
 *   epilogue RAW:    out fp32 [T*kmax, n_rows], out[r, n] = acc[r, n].
 *   epilogue SWIGLU: n_rows even, half = n_rows/2; out [T*kmax, half] of
 *                    out_dtype, out[r, n] = SiLU(acc[r, n]) * acc[r, half+n].
 * Rows r >= T*k are not written.  Calling RAW on the gate-only and up-only
 * matrices (n_rows = I each) gives, bit for bit, the two halves of RAW on
 * the fused matrix; moe_swiglu then reproduces the SWIGLU epilogue exactly.
 *
 * x               bf16 [T, H], read through sorted_assign; or, with
 *                 sorted_assign = NULL, bf16 [T*kmax, H] already in sorted
 *                 row order (moe_permute_rows), row r read for sorted row r.
 *                 Both forms give bitwise the same result.
 * sorted_assign, expert_offsets, k_dev  from moe_permute / moe_router_topk.
 * w_q             uint32 [E, n_rows, H*bits/32]; w_s, w_b fp16 [E, n_rows, H/64].
 * bits            4, 5, 6 or 8 (5 and 6: the GEMV family, no k gate).
 * path            MOE_PATH_*, optionally | MOE_PATH_K_RANGE(lo, hi).
 * ---------------------------------------------------------------------- */
moe_status_t moe_gate_up_qmm(const uint16_t* x, const int32_t* sorted_assign,
                             const int32_t* expert_offsets, const int32_t* k_dev, int T,
                             int kmax, int E, int H, int n_rows, const uint32_t* w_q,
                             const uint16_t* w_s, const uint16_t* w_b, int bits, int epilogue,
                             int out_dtype, void* out, int path, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_down_qmm -- the down projection over expert segments.
 *
 * Page [C], 实现剖析 ④ (down_proj after the activation) and page [A],
 * section 4.2.  For sorted row r in expert e's segment and output m:
 * y[r, m] = sum_i h[r, i] * (s[e, m, i/64] * code[e, m, i] + b[e, m, i/64]),
 * fp32 accumulation.
 *
 * h         [T*kmax, I] of h_dtype (MOE_DTYPE_F32 or MOE_DTYPE_BF16), rows in
 *           sorted order (as written by moe_gate_up_qmm).
 * w_q       uint32 [E, H, I*bits/32]; w_s, w_b fp16 [E, H, I/64].
 * y         out: [T*kmax, H] of y_dtype, sorted order; rows >= T*k not
 *           written.  MOE_DTYPE_F32 stores the fp32 sums; MOE_DTYPE_BF16
 *           stores each sum rounded to bf16 (nearest even), bit for bit the
 *           rounding of the fp32 result, at half the bytes written here and
 *           read again by moe_combine.
 * path      MOE_PATH_*, optionally | MOE_PATH_FLAG_WEIGHTS_EARLY and/or
 *           | MOE_PATH_K_RANGE(lo, hi).
 * ---------------------------------------------------------------------- */
moe_status_t moe_down_qmm(const void* h, int h_dtype, const int32_t* expert_offsets,
                          const int32_t* k_dev, int T, int kmax, int E, int I, int H,
                          const uint32_t* w_q, const uint16_t* w_s, const uint16_t* w_b,
                          int bits, void* y, int y_dtype, int path, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Expert health.  Page [B], section 6: a serving-side "MoE health" check on
 * two numbers per time window (one minute there): the expert activated least
 * often, and the standard deviation of all experts' activation counts (an
 * alert when it stays above 20 for five windows in a row); section 4.2 counts
 * activations per expert with a bincount of the routed expert ids.  Here a
 * call's activations of expert e are expert_counts[e] as the grouping writes
 * it (moe_permute, moe_route, moe_permute_capped: the assignments the expert
 * runs).  The window and the alert rule live in the caller
 * (sparse_moe_expert_gb300.ExpertHealthMonitor).
 *
 * moe_expert_counts_accumulate: window_counts[e] += expert_counts[e], e < E.
 *   expert_counts   int32 [E] (device); window_counts int64 [E] (device,
 *   8-byte aligned, zeroed by the caller when a window opens).
 * moe_expert_health: over c = window_counts[0..E):
 *   *least_expert = the e of the smallest c_e (equal counts: the lower e);
 *   mean_std[0] = sum(c) / E; mean_std[1] = sqrt(sum((c_e - mean)^2) / E)
 *   (population standard deviation), in fp64, sums in a fixed order.
 *   least_expert int32 scalar, mean_std double [2] (device, 8-byte aligned).
 * 1 <= E <= 1024 (else MOE_ERR_INVALID_ARG).  Both are asynchronous on
 * `stream`; the caller owns every buffer.
 * ---------------------------------------------------------------------- */
moe_status_t moe_expert_counts_accumulate(const int32_t* expert_counts, int E,
                                          int64_t* window_counts, moe_stream_t stream);
moe_status_t moe_expert_health(const int64_t* window_counts, int E, int32_t* least_expert,
                               double* mean_std, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_combine -- routing-weighted sum back to token order.
 *
 * Page [A], section 4.2: y[t] = sum_k w_k * expert_out_k.  Here
 * out[t, m] = bf16_rne( sum_{j<k} topk_w[t, j] * y[inv_pos[t*kmax+j], m] ),
 * accumulated in fp32 in ascending j.  A slot with inv_pos = MOE_DROPPED
 * (expert capacity) is skipped.
 *
 * y        [T*kmax, H] of y_dtype (MOE_DTYPE_F32 or MOE_DTYPE_BF16, as
 *          moe_down_qmm wrote it), sorted order; bf16 values enter the sum
 *          as their exact fp32 values.
 * out      out: bf16 [T, H].
 * ---------------------------------------------------------------------- */
moe_status_t moe_combine(const void* y, int y_dtype, const int32_t* inv_pos,
                         const float* topk_w, const int32_t* k_dev, int T, int kmax, int H,
                         uint16_t* out, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_swiglu -- the activation on its own, for the unfused two-product path.
 *
 * Page [C], 实现剖析 ④.  out[r, n] = SiLU(gate[r, n]) * up[r, n] for rows
 * r < T*k, with exactly the arithmetic of the SWIGLU epilogue.
 * gate, up   fp32 [T*kmax, I] (RAW outputs of the gate-only and up-only
 *            products).  out: [T*kmax, I] of out_dtype.
 * ---------------------------------------------------------------------- */
moe_status_t moe_swiglu(const float* gate, const float* up, const int32_t* k_dev, int T,
                        int kmax, int I, int out_dtype, void* out, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_get_device_error -- read (and optionally clear) the device error word
 * of the current device.  Synchronizes `stream` first.  *flags receives an
 * OR of MOE_DEVERR_* bits.
 * ---------------------------------------------------------------------- */
moe_status_t moe_get_device_error(uint32_t* flags, int clear, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_selftest_wait_timeout -- check of the bounded device waits.
 *
 * No page has a counterpart: every wait in the library's kernels gives up
 * after a bounded number of SM clock cycles, reports MOE_DEVERR_TIMEOUT in
 * the device error word and lets its kernel end, so a stalled pipeline is
 * reported instead of hanging the GPU.  This call launches one small CTA
 * whose thread waits, with the same wait routine, on an mbarrier that no
 * thread ever arrives on, for at most `budget_cycles` cycles (1 ..
 * 100,000,000, about 50 ms at 2 GHz), then sets MOE_DEVERR_TIMEOUT.  It lets
 * a caller check that a wait which runs out is reported and that the
 * context stays usable.  Asynchronous on `stream`.
 * ---------------------------------------------------------------------- */
moe_status_t moe_selftest_wait_timeout(uint32_t budget_cycles, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */

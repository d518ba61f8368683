/*
 * Seeded synthetic inputs for the quantized sparse-MoE layer forward.
 *
 * This file generates inputs only: normal draws, bf16 rounding of
 * activations, and the min-max affine quantizer that turns float expert
 * weights into packed codes with fp16 scale and bias per group of 64.
 * It holds none of the layer's arithmetic (no dequantization, no matmul,
 * no routing); both the oracle and the CUDA library consume its output.
 *
 * Random numbers come from a counter-based generator: element i of stream
 * (seed, stream) is a pure function of (seed, stream, i), so any slice of a
 * tensor can be generated on its own and in parallel.  64 random bits per
 * pair of elements come from the splitmix64 finaliser (Steele, Lea, Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014) applied to
 * a mixed counter; the pair is turned into two N(0,1) draws by the
 * Box-Muller transform.
 *
 * Packing convention (shared with every consumer): a row of `cols` b-bit
 * codes is stored as uint32 words, element i of the row in word i/(32/b) at
 * bit offset b*(i mod (32/b)), little-endian.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t mix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(mix64(seed) ^ (stream * 0xD6E8FEB86659FD93ull));
}

/* Two N(0,1) draws for pair index p of a stream. */
static inline void normal_pair(uint64_t key, uint64_t p, double* z0, double* z1) {
  uint64_t r = mix64(key ^ mix64(p));
  double u1 = ((double)(r >> 32) + 1.0) * (1.0 / 4294967296.0); /* (0, 1] */
  double u2 = (double)(r & 0xFFFFFFFFull) * (1.0 / 4294967296.0); /* [0, 1) */
  double rad = sqrt(-2.0 * log(u1));
  double ang = 6.283185307179586476925286766559 * u2;
  *z0 = rad * cos(ang);
  *z1 = rad * sin(ang);
}

static inline double normal_at(uint64_t key, uint64_t i) {
  double z0, z1;
  normal_pair(key, i >> 1, &z0, &z1);
  return (i & 1) ? z1 : z0;
}

static inline uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static inline float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* float -> bf16, round to nearest even (finite inputs). */
static inline uint16_t f32_to_bf16(float f) {
  uint32_t u = f32_bits(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* float -> IEEE binary16, round to nearest even, with subnormals. */
static uint16_t f32_to_f16(float f) {
  uint32_t u = f32_bits(f);
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  uint32_t a = u & 0x7FFFFFFFu;
  if (a >= 0x7F800000u) return (uint16_t)(sign | 0x7C00u | (a > 0x7F800000u ? 0x200u : 0u));
  if (a >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u); /* rounds to inf */
  int e = (int)(a >> 23) - 127;
  uint32_t mant = (a & 0x7FFFFFu) | 0x800000u;
  if (e >= -14) { /* normal half */
    uint32_t h = ((uint32_t)(e + 15) << 10) | ((mant >> 13) & 0x3FFu);
    uint32_t rem = mant & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;
    return (uint16_t)(sign | h);
  }
  if (e < -25) return sign; /* below half the smallest subnormal */
  /* subnormal: value = mant * 2^(e-23); unit = 2^-24 */
  int shift = -e - 1; /* 14..24: mant >> (shift) gives units of 2^-24 */
  uint32_t h = mant >> shift;
  uint32_t rem = mant & ((1u << shift) - 1u);
  uint32_t halfway = 1u << (shift - 1);
  if (rem > halfway || (rem == halfway && (h & 1u))) h += 1u;
  return (uint16_t)(sign | h);
}

static float f16_to_f32(uint16_t h) {
  uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
  uint32_t e = (h >> 10) & 0x1Fu, m = h & 0x3FFu;
  if (e == 0) {
    float v = (float)m * (1.0f / 16777216.0f);
    return sign ? -v : v;
  }
  if (e == 31) return bits_f32(sign | 0x7F800000u | (m << 13));
  return bits_f32(sign | ((e + 112u) << 23) | (m << 13));
}

/* ---- plain fills ------------------------------------------------------- */

void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t start, int64_t n,
                      double sigma, float* out) {
  uint64_t key = stream_key(seed, stream);
  for (int64_t j = 0; j < n; ++j) out[j] = (float)(sigma * normal_at(key, start + (uint64_t)j));
}

void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t start, int64_t n,
                       double sigma, uint16_t* out) {
  uint64_t key = stream_key(seed, stream);
  for (int64_t j = 0; j < n; ++j)
    out[j] = f32_to_bf16((float)(sigma * normal_at(key, start + (uint64_t)j)));
}

/* ---- quantized weights ------------------------------------------------- */

typedef struct {
  uint64_t key;
  int64_t row0, row1; /* absolute rows [row0, row1) of the flattened [E*rows] matrix */
  int64_t out_row0;   /* absolute row that output index 0 corresponds to */
  int cols, bits;
  double sigma;
  uint32_t* q;
  uint16_t *s, *b;
  float* w_out; /* optional: the float weights before quantization */
} qjob_t;

static void quantize_rows(const qjob_t* j) {
  const int G = 64;
  const int words = j->cols * j->bits / 32;
  const int groups = j->cols / G;
  const uint32_t qmax = (1u << j->bits) - 1u;
  float w[64];
  for (int64_t r = j->row0; r < j->row1; ++r) {
    const int64_t o = r - j->out_row0;
    uint32_t* qrow = j->q + o * (int64_t)words;
    memset(qrow, 0, sizeof(uint32_t) * (size_t)words);
    for (int g = 0; g < groups; ++g) {
      uint64_t base = (uint64_t)r * (uint64_t)j->cols + (uint64_t)g * G;
      float mn = 0.f, mx = 0.f;
      for (int i = 0; i < G; i += 2) {
        double z0, z1;
        normal_pair(j->key, (base + (uint64_t)i) >> 1, &z0, &z1);
        w[i] = (float)(j->sigma * z0);
        w[i + 1] = (float)(j->sigma * z1);
      }
      mn = w[0]; mx = w[0];
      for (int i = 1; i < G; ++i) { if (w[i] < mn) mn = w[i]; if (w[i] > mx) mx = w[i]; }
      uint16_t sh = f32_to_f16((mx - mn) / (float)qmax);
      uint16_t bh = f32_to_f16(mn);
      float sf = f16_to_f32(sh), bf = f16_to_f32(bh);
      j->s[o * (int64_t)groups + g] = sh;
      j->b[o * (int64_t)groups + g] = bh;
      for (int i = 0; i < G; ++i) {
        uint32_t qi = 0;
        if (sf > 0.f) {
          float v = nearbyintf((w[i] - bf) / sf);
          if (v < 0.f) v = 0.f;
          if (v > (float)qmax) v = (float)qmax;
          qi = (uint32_t)v;
        }
        /* element col at bits [bits*col, bits*col + bits) of the row's
           little-endian bit stream (whole in one word for 4 and 8 bits) */
        const int col = g * G + i;
        const int64_t pos = (int64_t)col * j->bits;
        const int wi = (int)(pos >> 5), off = (int)(pos & 31);
        qrow[wi] |= qi << off;
        if (off + j->bits > 32) qrow[wi + 1] |= qi >> (32 - off);
        if (j->w_out) j->w_out[o * (int64_t)j->cols + col] = w[i];
      }
    }
  }
}

static void* quantize_thread(void* arg) { quantize_rows((const qjob_t*)arg); return NULL; }

/*
 * Fill rows [row0, row0+nrows) of a stream of weights with N(0, sigma)
 * draws (row-major, `cols` per row), quantize each group of 64 consecutive
 * columns with min-max affine codes: scale = fp16((max-min)/(2^bits-1)),
 * bias = fp16(min), code = clamp(rint((w-bias)/scale), 0, 2^bits-1) using the
 * fp16-rounded scale and bias (scale 0 gives code 0).  Outputs are indexed
 * from row0: q[(r-row0)*cols*bits/32], s/b[(r-row0)*cols/64].  bits is 4,
 * 5, 6 or 8; a row's codes form one little-endian bit stream over its
 * uint32 words (a 64-code group is 2*bits whole words).
 */
int synth_quantized(uint64_t seed, uint64_t stream, int64_t row0, int64_t nrows, int cols,
                    int bits, double sigma, uint32_t* q, uint16_t* s, uint16_t* b,
                    float* w_out, int nthreads) {
  if ((bits != 4 && bits != 5 && bits != 6 && bits != 8) || cols % 64 != 0 || nrows < 0)
    return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > nrows) nthreads = nrows > 0 ? (int)nrows : 1;
  uint64_t key = stream_key(seed, stream);
  qjob_t jobs[256];
  pthread_t th[256];
  int started[256];
  for (int t = 0; t < nthreads; ++t) {
    int64_t a = nrows * t / nthreads, e = nrows * (t + 1) / nthreads;
    jobs[t].key = key;
    jobs[t].row0 = row0 + a;
    jobs[t].row1 = row0 + e;
    jobs[t].out_row0 = row0;
    jobs[t].cols = cols;
    jobs[t].bits = bits;
    jobs[t].sigma = sigma;
    jobs[t].q = q;
    jobs[t].s = s;
    jobs[t].b = b;
    jobs[t].w_out = w_out;
  }
  for (int t = 0; t < nthreads; ++t) {
    started[t] = (nthreads > 1) && pthread_create(&th[t], NULL, quantize_thread, &jobs[t]) == 0;
    if (!started[t]) quantize_rows(&jobs[t]);
  }
  for (int t = 0; t < nthreads; ++t)
    if (started[t]) pthread_join(th[t], NULL);
  return 0;
}

/*
 * Seeded synthetic inputs for the blockwise-FP8 routed-MoE layer.
 *
 * This file generates DATA only.  It holds none of the layer's arithmetic:
 * no routing, no dequantisation, no expert FFN.  Both the CPU oracle and the
 * CUDA library read the bytes it writes.
 *
 * Random numbers are counter based, so every element depends only on
 * (seed, tensor id, element index) and the result is the same for any thread
 * count:
 *   key      = splitmix64(splitmix64(seed) ^ (tensor_id * 0xD1B54A32D192ED03))
 *   pair j   : b1 = splitmix64(key + 2j), b2 = splitmix64(key + 2j + 1)
 *              u1 = ((b1 >> 11) + 1) * 2^-53   in (0, 1]
 *              u2 =  (b2 >> 11)      * 2^-53   in [0, 1)
 *              z[2j]   = sqrt(-2 ln u1) * cos(2 pi u2)
 *              z[2j+1] = sqrt(-2 ln u1) * sin(2 pi u2)      (Box-Muller)
 * splitmix64 is Steele, Lea and Flood's SplitMix64 finaliser (2014).
 *
 * Weight matrices are quantised per 128x128 block to e4m3 ("fn" variant:
 * bias 7, no infinities, max 448) with one f32 scale per block:
 *   scale = absmax / 448 (f32), or 1 if the block is all zero,
 *   code  = e4m3_rne(clamp(v / scale, -448, 448)).
 * This is the weight format the dragon.c page states under "Precision"
 * (e4m3 with 128x128 blockwise f32 scales).
 *
 * The FP4 expert format (NVFP4, the Qwen post's experts) is generated from
 * the same normal streams: per expert matrix a global f32 scale
 * g = absmax / (6 * 448) (1 if all zero); per 16 consecutive values of a row
 * an e4m3 block scale s = e4m3_rne(block absmax / (6 g)); codes
 * e2m1_rne(clamp(v / (s g), -6, 6)) (0 where s is 0), two per byte, the
 * even element in the low nibble.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static inline uint64_t splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t gen_stream_key(uint64_t seed, uint64_t tensor_id) {
  return splitmix64(splitmix64(seed) ^ (tensor_id * 0xD1B54A32D192ED03ull));
}

static inline void normal_pair(uint64_t key, uint64_t j, double *z0, double *z1) {
  const double two_m53 = 1.1102230246251565e-16; /* 2^-53 */
  uint64_t b1 = splitmix64(key + 2 * j);
  uint64_t b2 = splitmix64(key + 2 * j + 1);
  double u1 = (double)((b1 >> 11) + 1) * two_m53;
  double u2 = (double)(b2 >> 11) * two_m53;
  double r = sqrt(-2.0 * log(u1));
  double a = 6.283185307179586 * u2;
  *z0 = r * cos(a);
  *z1 = r * sin(a);
}

/* Standard normal number i of a stream (exported for tests). */
double gen_normal_at(uint64_t seed, uint64_t tensor_id, uint64_t i) {
  double z0, z1;
  normal_pair(gen_stream_key(seed, tensor_id), i >> 1, &z0, &z1);
  return (i & 1) ? z1 : z0;
}

/* f32 -> bf16 bits, round to nearest even (inputs here are finite). */
static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* f32 -> e4m3 ("fn") code, round to nearest even, saturating at +-448. */
uint8_t gen_e4m3_encode(float y) {
  double a = fabs((double)y);
  uint8_t sign = signbit(y) ? 0x80 : 0x00;
  if (isnan(y)) return 0x7F;
  if (a >= 448.0) return sign | 0x7E;
  if (a < 0.015625) { /* below 2^-6: subnormal grid of step 2^-9 */
    double m = nearbyint(a * 512.0);  /* 0..8; 8 is the smallest normal */
    return sign | (uint8_t)m;
  }
  int ex;
  double fr = frexp(a, &ex); /* a = fr * 2^ex, fr in [0.5, 1) */
  int e = ex - 1;            /* a in [2^e, 2^(e+1)), e in [-6, 8] */
  double mant = fr * 2.0;    /* [1, 2) */
  double m = nearbyint((mant - 1.0) * 8.0);
  if (m >= 8.0) { m = 0.0; e += 1; }
  int code = ((e + 7) << 3) | (int)m;
  if (code > 0x7E) code = 0x7E;
  return sign | (uint8_t)code;
}

void gen_e4m3_encode_array(const float *in, int64_t n, uint8_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = gen_e4m3_encode(in[i]);
}

/* e4m3 ("fn") code -> value (finite codes only). */
static double e4m3_decode(uint8_t c) {
  int e = (c >> 3) & 0xF, m = c & 7;
  double v = e == 0 ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
  return (c & 0x80) ? -v : v;
}

/* f32 -> e2m1 code (sign bit 3; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 are
 * codes 0..7), round to nearest with ties to the even code, saturating at
 * +-6. */
uint8_t gen_e2m1_encode(float y) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  const uint8_t sign = signbit(y) ? 0x8 : 0x0;
  const double a = fabs((double)y);
  if (a >= 6.0) return sign | 7;
  int best = 0;
  for (int c = 1; c < 8; ++c) {
    const double d = fabs(a - mag[c]), db = fabs(a - mag[best]);
    if (d < db || (d == db && (c & 1) == 0)) best = c;
  }
  return sign | (uint8_t)best;
}

/* ---------------------------------------------------------------- threads */

typedef struct {
  int kind; /* 0 = f32, 1 = bf16, 2 = blockwise e4m3, 3 = nvfp4 (one expert per unit) */
  uint64_t key;
  int64_t lo, hi; /* work range: elements (kinds 0, 1) or blocks (kind 2) */
  double std;
  float *out_f32;
  uint16_t *out_bf16;
  /* blockwise */
  int64_t R, C;
  uint8_t *codes;
  float *scales;
  /* nvfp4 */
  uint8_t *bscales;
  float *gscales;
} job_t;

static void run_flat(job_t *j) {
  int64_t i = j->lo;
  while (i < j->hi) {
    double z[2];
    normal_pair(j->key, (uint64_t)i >> 1, &z[0], &z[1]);
    for (int s = (int)(i & 1); s < 2 && i < j->hi; ++s, ++i) {
      float v = (float)(j->std * z[s]);
      if (j->kind == 0) j->out_f32[i] = v;
      else j->out_bf16[i] = f32_to_bf16_rne(v);
    }
  }
}

static void run_blocks(job_t *j) {
  const int64_t rb_n = j->R / 128, cb_n = j->C / 128;
  float *buf = (float *)malloc(128 * 128 * sizeof(float));
  for (int64_t b = j->lo; b < j->hi; ++b) {
    int64_t e = b / (rb_n * cb_n);
    int64_t rb = (b / cb_n) % rb_n;
    int64_t cb = b % cb_n;
    float amax = 0.0f;
    for (int r = 0; r < 128; ++r) {
      int64_t row = rb * 128 + r;
      uint64_t base = (uint64_t)((e * j->R + row) * j->C + cb * 128); /* even */
      for (int c = 0; c < 128; c += 2) {
        double z0, z1;
        normal_pair(j->key, (base + (uint64_t)c) >> 1, &z0, &z1);
        float v0 = (float)(j->std * z0), v1 = (float)(j->std * z1);
        buf[r * 128 + c] = v0;
        buf[r * 128 + c + 1] = v1;
        float a0 = fabsf(v0), a1 = fabsf(v1);
        if (a0 > amax) amax = a0;
        if (a1 > amax) amax = a1;
      }
    }
    float scale = (amax > 0.0f) ? amax / 448.0f : 1.0f;
    j->scales[(e * rb_n + rb) * cb_n + cb] = scale;
    for (int r = 0; r < 128; ++r) {
      int64_t row = rb * 128 + r;
      uint8_t *dst = j->codes + (e * j->R + row) * j->C + cb * 128;
      for (int c = 0; c < 128; ++c) dst[c] = gen_e4m3_encode(buf[r * 128 + c] / scale);
    }
  }
  free(buf);
}

/* Experts [lo, hi) of an nvfp4 matrix set; element (e, r, c) is normal
 * number (e*R + r)*C + c of the stream, as in run_blocks. */
static void run_nvfp4(job_t *j) {
  const int64_t R = j->R, C = j->C;
  for (int64_t e = j->lo; e < j->hi; ++e) {
    const uint64_t base = (uint64_t)(e * R * C); /* even: C is a multiple of 16 */
    float amax = 0.0f;
    for (uint64_t i = 0; i < (uint64_t)(R * C); i += 2) {
      double z0, z1;
      normal_pair(j->key, (base + i) >> 1, &z0, &z1);
      const float a0 = fabsf((float)(j->std * z0)), a1 = fabsf((float)(j->std * z1));
      if (a0 > amax) amax = a0;
      if (a1 > amax) amax = a1;
    }
    const float g = amax > 0.0f ? amax / (6.0f * 448.0f) : 1.0f;
    j->gscales[e] = g;
    for (int64_t r = 0; r < R; ++r) {
      for (int64_t c0 = 0; c0 < C; c0 += 16) {
        float v[16], bmax = 0.0f;
        for (int c = 0; c < 16; c += 2) {
          double z0, z1;
          normal_pair(j->key, (base + (uint64_t)(r * C + c0 + c)) >> 1, &z0, &z1);
          v[c] = (float)(j->std * z0);
          v[c + 1] = (float)(j->std * z1);
        }
        for (int c = 0; c < 16; ++c)
          if (fabsf(v[c]) > bmax) bmax = fabsf(v[c]);
        const uint8_t sc = gen_e4m3_encode(bmax / (6.0f * g));
        j->bscales[(e * R + r) * (C / 16) + c0 / 16] = sc;
        const double sv = e4m3_decode(sc) * (double)g;
        uint8_t *dst = j->codes + (e * R + r) * (C / 2) + c0 / 2;
        for (int c = 0; c < 16; c += 2) {
          const uint8_t q0 = sv > 0.0 ? gen_e2m1_encode((float)(v[c] / sv)) : 0;
          const uint8_t q1 = sv > 0.0 ? gen_e2m1_encode((float)(v[c + 1] / sv)) : 0;
          dst[c / 2] = (uint8_t)(q0 | (q1 << 4));
        }
      }
    }
  }
}

static void *thread_main(void *arg) {
  job_t *j = (job_t *)arg;
  if (j->kind == 3) run_nvfp4(j);
  else if (j->kind == 2) run_blocks(j);
  else run_flat(j);
  return NULL;
}

static int run_parallel(job_t proto, int64_t total, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > total) nthreads = total > 0 ? (int)total : 1;
  pthread_t th[256];
  job_t jobs[256];
  int joinable[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = proto;
    jobs[t].lo = total * t / nthreads;
    jobs[t].hi = total * (t + 1) / nthreads;
    joinable[t] = pthread_create(&th[t], NULL, thread_main, &jobs[t]) == 0;
    if (!joinable[t]) thread_main(&jobs[t]); /* run it on this thread */
  }
  for (int t = 0; t < nthreads; ++t)
    if (joinable[t]) pthread_join(th[t], NULL);
  return 0;
}

/* out[i] = f32(std * z_i), i in [0, n). */
int gen_normal_f32(uint64_t seed, uint64_t tensor_id, int64_t n, double std, float *out,
                   int nthreads) {
  job_t p;
  memset(&p, 0, sizeof p);
  p.kind = 0;
  p.key = gen_stream_key(seed, tensor_id);
  p.std = std;
  p.out_f32 = out;
  return run_parallel(p, n, nthreads);
}

/* out[i] = bf16_rne(f32(std * z_i)). */
int gen_normal_bf16(uint64_t seed, uint64_t tensor_id, int64_t n, double std, uint16_t *out,
                    int nthreads) {
  job_t p;
  memset(&p, 0, sizeof p);
  p.kind = 1;
  p.key = gen_stream_key(seed, tensor_id);
  p.std = std;
  p.out_bf16 = out;
  return run_parallel(p, n, nthreads);
}

/* E matrices of R x C values f32(std * z), z indexed (e*R + r)*C + c,
 * quantised per 128x128 block: codes [E,R,C] u8, scales [E,R/128,C/128] f32. */
int gen_blockwise_e4m3(uint64_t seed, uint64_t tensor_id, int64_t E, int64_t R, int64_t C,
                       double std, uint8_t *codes, float *scales, int nthreads) {
  if (R % 128 != 0 || C % 128 != 0 || E < 0) return -1;
  job_t p;
  memset(&p, 0, sizeof p);
  p.kind = 2;
  p.key = gen_stream_key(seed, tensor_id);
  p.std = std;
  p.R = R;
  p.C = C;
  p.codes = codes;
  p.scales = scales;
  return run_parallel(p, E * (R / 128) * (C / 128), nthreads);
}

/* E matrices of R x C values f32(std * z) in the FP4 expert format:
 * codes [E,R,C/2] u8 (two e2m1 per byte, even element low), block scales
 * [E,R,C/16] e4m3 codes, global scales [E] f32.  C % 16 == 0. */
int gen_nvfp4(uint64_t seed, uint64_t tensor_id, int64_t E, int64_t R, int64_t C, double std,
              uint8_t *codes, uint8_t *bscales, float *gscales, int nthreads) {
  if (C % 16 != 0 || R <= 0 || E < 0) return -1;
  job_t p;
  memset(&p, 0, sizeof p);
  p.kind = 3;
  p.key = gen_stream_key(seed, tensor_id);
  p.std = std;
  p.R = R;
  p.C = C;
  p.codes = codes;
  p.bscales = bscales;
  p.gscales = gscales;
  return run_parallel(p, E, nthreads);
}

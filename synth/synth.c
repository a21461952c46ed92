/*
 * Seeded synthetic inputs for the routed-expert FFN layer.
 *
 * This module only draws random numbers and lays bytes out in the canonical
 * expert-major order; it holds none of the layer's arithmetic (no dequant,
 * no router, no softmax, no FFN). Both the CPU oracle (via the tests) and the
 * CUDA library (via the tests and the benchmark) receive exactly these bytes.
 *
 * Generator: a counter-based hash. Every value is a pure function of
 * (seed, stream, counter), so any slice of any tensor can be regenerated
 * independently and in parallel. The mixing function is the splitmix64
 * finaliser (Steele, Lea, Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014), applied twice.
 *
 * Distributions (the workload recipe):
 *   x        ~ N(0,1) by Box-Muller in double, rounded to fp32 (RN) and then
 *              to bf16 (round to nearest even).
 *   W_router ~ N(0, 1/d), rounded to fp32.
 *   codes    uniform bytes, i.e. two independent uniform 4-bit codes per byte.
 *   scales   uniform integer exponent byte in [lo, hi] inclusive.
 *   bias     Zipf(s) log-probabilities over a seeded random permutation of
 *            ranks: b[e] = -s * ln(rank(e)), rank a permutation of 1..E.
 *   affine experts (group 64, `bits`-bit codes): codes uniform bits; per
 *            group a bf16 scale 2^e (1 + m/128), e uniform in {-9, -8, -7},
 *            m uniform in 0..127, and a bf16 bias
 *            -scale (2^bits - 1) / 2 (0.75 + 0.5u'), u, u' uniform in (0, 1),
 *            so the weights of a group straddle zero as a quantised
 *            zero-mean row does.
 *
 * Build flags must keep floating point contraction off (-ffp-contract=off)
 * so the same seed gives the same bits on x86-64 and AArch64.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define SYNTH_STREAM_X 1ULL
#define SYNTH_STREAM_ROUTER 2ULL
#define SYNTH_STREAM_BIAS 3ULL
#define SYNTH_STREAM_CODES 4ULL
#define SYNTH_STREAM_SCALES 5ULL
#define SYNTH_STREAM_SHARED_GATE 6ULL
#define SYNTH_STREAM_AFFINE 7ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(seed * 0x9E3779B97F4A7C15ULL + stream * 0xD1B54A32D192ED03ULL + 0x2545F4914F6CDD1DULL);
}
static inline uint64_t draw(uint64_t key, uint64_t ctr) {
  return mix64(key ^ (ctr * 0x9E3779B97F4A7C15ULL + 0x632BE59BD9B4E019ULL));
}

/* One 64-bit draw for (seed, stream, counter). */
uint64_t synth_u64(uint64_t seed, uint64_t stream, uint64_t ctr) { return draw(stream_key(seed, stream), ctr); }

/* Uniform double in the open interval (0, 1). */
static inline double u01(uint64_t r) { return ((double)(r >> 11) + 0.5) * (1.0 / 9007199254740992.0); }

/* One standard normal from two draws (counters 2i and 2i+1), Box-Muller cosine branch. */
static double normal_at(uint64_t seed, uint64_t stream, uint64_t i) {
  double u1 = u01(synth_u64(seed, stream, 2 * i));
  double u2 = u01(synth_u64(seed, stream, 2 * i + 1));
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925 * u2);
}

static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* x: [T][d] bf16 bit patterns. */
void synth_x(uint64_t seed, int T, int d, uint16_t* x) {
  size_t n = (size_t)T * (size_t)d;
  for (size_t i = 0; i < n; ++i) x[i] = f32_to_bf16_rne((float)normal_at(seed, SYNTH_STREAM_X, i));
}

/* W_router: [E][d] fp32, N(0, 1/d). */
void synth_router(uint64_t seed, int E, int d, float* w) {
  size_t n = (size_t)E * (size_t)d;
  double sd = 1.0 / sqrt((double)d);
  for (size_t i = 0; i < n; ++i) w[i] = (float)(normal_at(seed, SYNTH_STREAM_ROUTER, i) * sd);
}

/* Shared-expert gate row w_sg: [d] fp32, N(0, 1/d) (the router's distribution). */
void synth_shared_gate(uint64_t seed, int d, float* w) {
  double sd = 1.0 / sqrt((double)d);
  for (int i = 0; i < d; ++i) w[i] = (float)(normal_at(seed, SYNTH_STREAM_SHARED_GATE, (uint64_t)i) * sd);
}

/* Zipf(s) log-probability bias over a seeded permutation of ranks 1..E. */
void synth_bias_zipf(uint64_t seed, int E, double s, float* b) {
  int rank[4096];
  if (E > 4096) return;
  for (int e = 0; e < E; ++e) rank[e] = e + 1;
  for (int i = E - 1; i > 0; --i) { /* Fisher-Yates */
    uint64_t r = synth_u64(seed, SYNTH_STREAM_BIAS, (uint64_t)i);
    int j = (int)(((r >> 32) * (uint64_t)(i + 1)) >> 32);
    int t = rank[i]; rank[i] = rank[j]; rank[j] = t;
  }
  for (int e = 0; e < E; ++e) b[e] = (float)(-s * log((double)rank[e]));
}

/* Uniform code bytes: byte i of stream `stream` is byte (i % 8) of draw i / 8. */
void synth_code_bytes(uint64_t seed, uint64_t stream, size_t n, uint8_t* out) {
  uint64_t key = stream_key(seed, (SYNTH_STREAM_CODES << 40) ^ stream);
  size_t whole = n / 8;
  for (size_t c = 0; c < whole; ++c) {
    uint64_t r = draw(key, c);
    uint8_t b[8];
    for (int j = 0; j < 8; ++j) b[j] = (uint8_t)(r >> (8 * j)); /* byte order fixed, host-independent */
    memcpy(out + 8 * c, b, 8);
  }
  if (n % 8) {
    uint64_t r = draw(key, whole);
    for (size_t i = 8 * whole; i < n; ++i) out[i] = (uint8_t)(r >> (8 * (i % 8)));
  }
}

/* Uniform exponent bytes in [lo, hi]. */
void synth_scale_bytes(uint64_t seed, uint64_t stream, size_t n, int lo, int hi, uint8_t* out) {
  uint64_t span = (uint64_t)(hi - lo + 1);
  uint64_t key = stream_key(seed, (SYNTH_STREAM_SCALES << 40) ^ stream);
  for (size_t i = 0; i < n; ++i) {
    uint64_t r = draw(key, i);
    out[i] = (uint8_t)(lo + (int)(((r >> 32) * span) >> 32));
  }
}

/*
 * All experts of one layer in the canonical expert-major layout:
 * expert j in [0, E) has ffn F, the shared expert (j == E, present when S > 0)
 * has ffn S. Per expert: codes = gate/up [2f][d/2] then down [d][f/2];
 * scales = gate/up [2f][d/32] then down [d][f/32]. Expert j's bytes are drawn
 * from stream j, so they do not depend on E or on the other experts.
 */
typedef struct {
  uint64_t seed;
  int d, F, S, E, lo, hi;
  uint8_t* codes;
  uint8_t* scales;
  int first, stride;
} synth_job;

static size_t code_bytes_of(int d, int f) { return (size_t)3 * (size_t)f * (size_t)d / 2; }
static size_t scale_bytes_of(int d, int f) { return (size_t)3 * (size_t)f * (size_t)d / 32; }

static void* synth_experts_worker(void* arg) {
  synth_job* j = (synth_job*)arg;
  int n = j->E + (j->S > 0 ? 1 : 0);
  for (int e = j->first; e < n; e += j->stride) {
    int f = (e < j->E) ? j->F : j->S;
    size_t co = (size_t)e * code_bytes_of(j->d, j->F);
    size_t so = (size_t)e * scale_bytes_of(j->d, j->F);
    synth_code_bytes(j->seed, (uint64_t)e, code_bytes_of(j->d, f), j->codes + co);
    synth_scale_bytes(j->seed, (uint64_t)e, scale_bytes_of(j->d, f), j->lo, j->hi, j->scales + so);
  }
  return NULL;
}

int synth_experts(uint64_t seed, int d, int F, int S, int E, int lo, int hi, uint8_t* codes, uint8_t* scales,
                  int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  synth_job jobs[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = (synth_job){seed, d, F, S, E, lo, hi, codes, scales, t, nthreads};
    if (t > 0 && pthread_create(&th[t], NULL, synth_experts_worker, &jobs[t]) != 0) return -1;
  }
  synth_experts_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  return 0;
}

/*
 * Affine group-64 experts in their canonical layout: per expert (ffn f) the
 * codes of the gate/up rows [2f][d] then of the down rows [d][f] (each row a
 * little-endian stream of `bits`-bit fields), then the bf16 scales of gate/up
 * [2f][d/64] and of down [d][f/64], then the bf16 biases in the same order.
 * Expert j (the shared one is j == E) draws from stream j of its own key, so
 * its bytes do not depend on E or on the other experts.
 */
static size_t affine_bytes_of(int d, int f, int bits) {
  size_t n = (size_t)3 * (size_t)f * (size_t)d;
  return n * (size_t)bits / 8 + n / 16;
}

void synth_affine_expert(uint64_t seed, uint64_t stream, int d, int f, int bits, uint8_t* out) {
  size_t n = (size_t)3 * (size_t)f * (size_t)d, code_bytes = n * (size_t)bits / 8, groups = n / 64;
  synth_code_bytes(seed, (SYNTH_STREAM_AFFINE << 32) ^ stream, code_bytes, out);
  uint64_t key = stream_key(seed, (SYNTH_STREAM_AFFINE << 40) ^ stream);
  uint8_t* sc = out + code_bytes;
  uint8_t* bi = sc + 2 * groups;
  double half_range = 0.5 * (double)((1 << bits) - 1);
  for (size_t g = 0; g < groups; ++g) {
    uint64_t r = draw(key, g);
    double u = ((double)(r >> 40) + 0.5) * (1.0 / 16777216.0);
    double v = ((double)(r & 0xFFFFFFULL) + 0.5) * (1.0 / 16777216.0);
    /* scale: bf16 2^e (1 + m / 128), e uniform in {-9, -8, -7}, m uniform in 0..127 (built exactly) */
    int e2 = -9 + (int)(u * 3.0);
    uint16_t s16 = (uint16_t)(((uint32_t)(127 + e2) << 7) | (uint32_t)((r >> 24) & 0x7F));
    uint32_t sbits = (uint32_t)s16 << 16;
    float s32;
    memcpy(&s32, &sbits, 4);
    uint16_t b16 = f32_to_bf16_rne((float)(-(double)s32 * half_range * (0.75 + 0.5 * v)));
    sc[2 * g] = (uint8_t)(s16 & 0xFF);
    sc[2 * g + 1] = (uint8_t)(s16 >> 8);
    bi[2 * g] = (uint8_t)(b16 & 0xFF);
    bi[2 * g + 1] = (uint8_t)(b16 >> 8);
  }
}

typedef struct {
  uint64_t seed;
  int d, F, S, E, bits;
  uint8_t* out;
  int first, stride;
} synth_affine_job;

static void* synth_affine_worker(void* arg) {
  synth_affine_job* j = (synth_affine_job*)arg;
  int n = j->E + (j->S > 0 ? 1 : 0);
  for (int e = j->first; e < n; e += j->stride) {
    int f = (e < j->E) ? j->F : j->S;
    synth_affine_expert(j->seed, (uint64_t)e, j->d, f, j->bits, j->out + (size_t)e * affine_bytes_of(j->d, j->F, j->bits));
  }
  return NULL;
}

int synth_experts_affine(uint64_t seed, int d, int F, int S, int E, int bits, uint8_t* out, int nthreads) {
  if (bits < 1 || bits > 8 || d % 64 || F % 64 || S % 64) return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  synth_affine_job jobs[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = (synth_affine_job){seed, d, F, S, E, bits, out, t, nthreads};
    if (t > 0 && pthread_create(&th[t], NULL, synth_affine_worker, &jobs[t]) != 0) return -1;
  }
  synth_affine_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  return 0;
}

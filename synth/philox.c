/* Seeded synthetic inputs: counter-based normal draws.
 *
 * Philox-4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
 * SC'11) turns a 128-bit counter and a 64-bit key into four 32-bit words; the Box-Muller
 * transform turns two uniforms into two standard normals.  Because the draw for element i depends
 * only on (seed, stream, i), any thread count gives the same bytes.
 *
 * This module only makes inputs.  It contains none of the decode step's arithmetic, and both the
 * oracle side and the GPU side of every test consume the same buffers it writes.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

static void philox4x32_10(uint32_t ctr[4], uint32_t k0, uint32_t k1) {
  for (int round = 0; round < 10; ++round) {
    uint64_t p0 = (uint64_t)PHILOX_M0 * ctr[0];
    uint64_t p1 = (uint64_t)PHILOX_M1 * ctr[2];
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ ctr[1] ^ k0;
    uint32_t n2 = hi0 ^ ctr[3] ^ k1;
    ctr[0] = n0;
    ctr[1] = lo1;
    ctr[2] = n2;
    ctr[3] = lo0;
    k0 += PHILOX_W0;
    k1 += PHILOX_W1;
  }
}

/* Four standard normals for block `blk` of stream `stream` under `seed`. */
static void normals4(uint64_t seed, uint64_t stream, uint64_t blk, double out[4]) {
  uint32_t c[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), (uint32_t)stream,
                   (uint32_t)(stream >> 32)};
  philox4x32_10(c, (uint32_t)seed, (uint32_t)(seed >> 32));
  const double two_pi = 6.283185307179586476925286766559;
  const double inv32 = 1.0 / 4294967296.0;
  for (int h = 0; h < 2; ++h) {
    double u1 = ((double)c[2 * h] + 1.0) * inv32; /* (0, 1] */
    double u2 = (double)c[2 * h + 1] * inv32;     /* [0, 1) */
    double rad = sqrt(-2.0 * log(u1));
    out[2 * h] = rad * cos(two_pi * u2);
    out[2 * h + 1] = rad * sin(two_pi * u2);
  }
}

typedef struct {
  uint64_t seed, stream, offset;
  int64_t begin, end;
  double mean, stdev;
  float* out;
} normal_job;

static void* normal_worker(void* arg) {
  normal_job* j = (normal_job*)arg;
  double buf[4];
  uint64_t cached = UINT64_MAX;
  for (int64_t i = j->begin; i < j->end; ++i) {
    uint64_t g = j->offset + (uint64_t)i;
    uint64_t blk = g >> 2;
    if (blk != cached) {
      normals4(j->seed, j->stream, blk, buf);
      cached = blk;
    }
    j->out[i] = (float)(j->mean + j->stdev * buf[g & 3]);
  }
  return 0;
}

/* out[i] = fp32(mean + stdev * N(offset + i)), i in [0, n). */
int synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double mean,
                     double stdev, float* out, int nthreads) {
  if (n <= 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 64) nthreads = 64;
  if (n < (int64_t)1 << 16) nthreads = 1;
  pthread_t th[64];
  normal_job jobs[64];
  int64_t chunk = ((n + nthreads - 1) / nthreads + 3) & ~(int64_t)3;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    int64_t b = (int64_t)t * chunk, e = b + chunk;
    if (b >= n) break;
    if (e > n) e = n;
    jobs[t] = (normal_job){seed, stream, offset, b, e, mean, stdev, out};
    if (t == 0) continue;
    if (pthread_create(&th[t], 0, normal_worker, &jobs[t]) != 0) return 1;
    started = t;
  }
  normal_worker(&jobs[0]);
  for (int t = 1; t <= started; ++t) pthread_join(th[t], 0);
  return 0;
}

typedef struct {
  const float* in;
  uint16_t* out;
  int64_t begin, end;
} bf16_job;

static void* bf16_worker(void* arg) {
  bf16_job* j = (bf16_job*)arg;
  for (int64_t i = j->begin; i < j->end; ++i) {
    uint32_t u;
    memcpy(&u, &j->in[i], 4);
    /* round to nearest even on the upper 16 bits (inputs are finite) */
    u += 0x7FFFu + ((u >> 16) & 1u);
    j->out[i] = (uint16_t)(u >> 16);
  }
  return 0;
}

/* bf16 round-to-nearest-even of finite fp32 values. */
int synth_f32_to_bf16(const float* in, int64_t n, uint16_t* out, int nthreads) {
  if (n <= 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 64) nthreads = 64;
  if (n < (int64_t)1 << 16) nthreads = 1;
  pthread_t th[64];
  bf16_job jobs[64];
  int64_t chunk = (n + nthreads - 1) / nthreads;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    int64_t b = (int64_t)t * chunk, e = b + chunk;
    if (b >= n) break;
    if (e > n) e = n;
    jobs[t] = (bf16_job){in, out, b, e};
    if (t == 0) continue;
    if (pthread_create(&th[t], 0, bf16_worker, &jobs[t]) != 0) return 1;
    started = t;
  }
  bf16_worker(&jobs[0]);
  for (int t = 1; t <= started; ++t) pthread_join(th[t], 0);
  return 0;
}

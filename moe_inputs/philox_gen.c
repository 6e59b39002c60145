/*
 * Seeded synthetic-input generator shared by the CUDA path's tests/bench and
 * by the CPU oracle.  It holds none of the MoE method's arithmetic: it only
 * turns (seed, tensor id, element index) into numbers.
 *
 * Generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
 * numbers: as easy as 1, 2, 3", SC'11), counter-based.  Element i of a tensor
 * uses counter block i/4 and lane i%4; key = (seed, tensor_id).
 * Normals: Box-Muller in double on lane pairs (0,1) and (2,3).
 * bf16 values: double -> float (RN) -> bf16 (round to nearest even).
 *
 * Built as a plain C shared library (gcc -O2 -fopenmp); every entry point is
 * pure and thread-safe, parallelised over elements with OpenMP.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

static inline void philox_round(uint32_t c[4], uint32_t k0, uint32_t k1) {
  uint64_t p0 = (uint64_t)PHILOX_M0 * (uint64_t)c[0];
  uint64_t p1 = (uint64_t)PHILOX_M1 * (uint64_t)c[2];
  uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
  uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
  uint32_t n0 = hi1 ^ c[1] ^ k0;
  uint32_t n2 = hi0 ^ c[3] ^ k1;
  c[0] = n0;
  c[1] = lo1;
  c[2] = n2;
  c[3] = lo0;
}

/* One Philox4x32-10 block: ten rounds, the key bumped by the Weyl constants
 * between rounds. */
void moe_inputs_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
  uint32_t k0 = key[0], k1 = key[1];
  for (int r = 0; r < 10; ++r) {
    philox_round(c, k0, k1);
    k0 += PHILOX_W0;
    k1 += PHILOX_W1;
  }
  memcpy(out, c, sizeof(c));
}

static inline void block_for(uint64_t seed, uint32_t tensor_id, uint64_t blk, uint32_t out[4]) {
  uint32_t ctr[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), 0u, 0u};
  uint32_t key[2] = {(uint32_t)seed ^ (uint32_t)(seed >> 32), tensor_id};
  moe_inputs_philox4x32_10(ctr, key, out);
}

static inline double u01(uint32_t a) { return ((double)a + 0.5) * (1.0 / 4294967296.0); }

static inline double normal_at(uint64_t seed, uint32_t tensor_id, uint64_t i) {
  uint32_t r[4];
  block_for(seed, tensor_id, i >> 2, r);
  unsigned lane = (unsigned)(i & 3u);
  unsigned pair = lane & 2u;
  double u1 = u01(r[pair]), u2 = u01(r[pair + 1]);
  double rad = sqrt(-2.0 * log(u1));
  double th = 6.283185307179586476925286766559 * u2;
  return (lane & 1u) ? rad * sin(th) : rad * cos(th);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* out[i] = uniform u32 stream (raw Philox words), i < n. */
void moe_inputs_u32(uint64_t seed, uint32_t tensor_id, int64_t n, uint32_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < (n + 3) / 4; ++b) {
    uint32_t r[4];
    block_for(seed, tensor_id, (uint64_t)b, r);
    for (int j = 0; j < 4; ++j) {
      int64_t i = b * 4 + j;
      if (i < n) out[i] = r[j];
    }
  }
}

/* The four normals of counter block blk: z[j] = normal_at(seed, tensor_id, 4*blk + j), one Philox
 * block and one Box-Muller pair per two elements instead of one each per element. */
static inline void normal4_at(uint64_t seed, uint32_t tensor_id, uint64_t blk, double z[4]) {
  uint32_t r[4];
  block_for(seed, tensor_id, blk, r);
  for (unsigned pair = 0; pair < 4; pair += 2) {
    double u1 = u01(r[pair]), u2 = u01(r[pair + 1]);
    double rad = sqrt(-2.0 * log(u1));
    double th = 6.283185307179586476925286766559 * u2;
    z[pair] = rad * cos(th);
    z[pair + 1] = rad * sin(th);
  }
}

/* out[i - start] = bf16(mean + std * z_i), z_i ~ N(0,1), for start <= i < start + n: a slice of the
 * tensor's stream (element i always uses counter block i/4, lane i%4). */
void moe_inputs_normal_bf16_range(uint64_t seed, uint32_t tensor_id, int64_t start, int64_t n, double mean,
                                  double stdv, uint16_t* out) {
  const int64_t b0 = start / 4, b1 = (start + n + 3) / 4;
#pragma omp parallel for schedule(static)
  for (int64_t b = b0; b < b1; ++b) {
    double z[4];
    normal4_at(seed, tensor_id, (uint64_t)b, z);
    for (int j = 0; j < 4; ++j) {
      const int64_t i = b * 4 + j;
      if (i >= start && i < start + n) out[i - start] = f32_to_bf16_rne((float)(mean + stdv * z[j]));
    }
  }
}

/* out[i] = bf16(mean + std * z_i), z_i ~ N(0,1). */
void moe_inputs_normal_bf16(uint64_t seed, uint32_t tensor_id, int64_t n, double mean, double stdv,
                            uint16_t* out) {
  moe_inputs_normal_bf16_range(seed, tensor_id, 0, n, mean, stdv, out);
}

/* out[i] = float(mean + std * z_i). */
void moe_inputs_normal_f32(uint64_t seed, uint32_t tensor_id, int64_t n, double mean, double stdv,
                           float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    out[i] = (float)(mean + stdv * normal_at(seed, tensor_id, (uint64_t)i));
  }
}

/* Router logits on a 2^-q grid: out[t*E+e] = RNE_{2^-q}(z_{t,e} + off[e]), in
 * double, then converted to float (exact for the magnitudes generated). */
void moe_inputs_grid_logits(uint64_t seed, uint32_t tensor_id, int64_t T, int64_t E, const double* off,
                            int q, float* out) {
  const double s = ldexp(1.0, q);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < T * E; ++i) {
    double v = normal_at(seed, tensor_id, (uint64_t)i) + (off ? off[i % E] : 0.0);
    out[i] = (float)(nearbyint(v * s) / s);
  }
}

/*
 * Seeded synthetic inputs shared by the CUDA path's tests/benchmarks and by
 * the CPU oracle.  This file holds no arithmetic of the tensor relational
 * algebra method: it only turns (seed, tensor id, element index) into a number.
 *
 * Generator: Philox-4x32 with 10 rounds, the counter-based generator of
 * Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3"
 * (SC'11).  One bijection of a 128-bit counter under a 64-bit key:
 *   round:  (c0,c1,c2,c3) -> (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2),
 *                            hi(M0*c0) ^ c3 ^ k1, lo(M0*c0))
 *   key bump between rounds: k0 += W0, k1 += W1
 * with M0 = 0xD2511F53, M1 = 0xCD9E8D57, W0 = 0x9E3779B9, W1 = 0xBB67AE85.
 *
 * Stream layout used everywhere in this repository:
 *   key     = (seed, tensor_id)
 *   counter = (element_index low 32 bits, element_index high 32 bits, 0, 0)
 * where element_index is the row-major position in the dense tensor.
 *
 * Uniform U[lo,hi):  u = (r0 >> 8) * 2^-24,  value = lo + (hi-lo)*u
 * Normal N(mu,sigma): Box-Muller, cosine branch, one normal per counter:
 *   u1 = ((r0 >> 8) + 1) * 2^-24 in (0,1],  u2 = (r1 >> 8) * 2^-24
 *   z  = sqrt(-2 ln u1) * cos(2 pi u2),     value = mu + sigma*z
 * Values are formed in double and rounded once to fp32 (round to nearest
 * even).  BF16 values are the fp32 value rounded to nearest even in bf16.
 *
 * Built with -ffp-contract=off so that x86-64 and aarch64 hosts produce the
 * same fp32 values for the uniform stream (the normal stream also depends on
 * the host libm's log/cos).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

void dg_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += PHILOX_W0;
            k1 += PHILOX_W1;
        }
        uint64_t p0 = (uint64_t)PHILOX_M0 * (uint64_t)c0;
        uint64_t p1 = (uint64_t)PHILOX_M1 * (uint64_t)c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

static inline void draw(uint32_t seed, uint32_t tensor, uint64_t idx, uint32_t r[4]) {
    uint32_t ctr[4] = {(uint32_t)idx, (uint32_t)(idx >> 32), 0u, 0u};
    uint32_t key[2] = {seed, tensor};
    dg_philox4x32_10(ctr, key, r);
}

static const double TWO_M24 = 1.0 / 16777216.0;
static const double TWO_PI = 6.283185307179586476925286766559;

static inline double uniform01(const uint32_t r[4]) { return (double)(r[0] >> 8) * TWO_M24; }

static inline double std_normal(const uint32_t r[4]) {
    double u1 = ((double)(r[0] >> 8) + 1.0) * TWO_M24;
    double u2 = (double)(r[1] >> 8) * TWO_M24;
    return sqrt(-2.0 * log(u1)) * cos(TWO_PI * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) return (uint16_t)((b >> 16) | 0x40u); /* quiet NaN */
    uint32_t lsb = (b >> 16) & 1u;
    b += 0x7FFFu + lsb;
    return (uint16_t)(b >> 16);
}

void dg_fill_uniform_f32(uint32_t seed, uint32_t tensor, int64_t n, double lo, double hi, float* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint32_t r[4];
        draw(seed, tensor, (uint64_t)i, r);
        out[i] = (float)(lo + (hi - lo) * uniform01(r));
    }
}

void dg_fill_normal_f32(uint32_t seed, uint32_t tensor, int64_t n, double mu, double sigma, float* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint32_t r[4];
        draw(seed, tensor, (uint64_t)i, r);
        out[i] = (float)(mu + sigma * std_normal(r));
    }
}

void dg_fill_uniform_bf16(uint32_t seed, uint32_t tensor, int64_t n, double lo, double hi, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint32_t r[4];
        draw(seed, tensor, (uint64_t)i, r);
        out[i] = f32_to_bf16_rne((float)(lo + (hi - lo) * uniform01(r)));
    }
}

void dg_fill_normal_bf16(uint32_t seed, uint32_t tensor, int64_t n, double mu, double sigma, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint32_t r[4];
        draw(seed, tensor, (uint64_t)i, r);
        out[i] = f32_to_bf16_rne((float)(mu + sigma * std_normal(r)));
    }
}

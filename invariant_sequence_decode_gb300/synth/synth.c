/*
 * synth.c - seeded, counter-based synthetic inputs for the batched decode step.
 *
 * This file generates INPUTS only (weights, scales, activations, KV caches,
 * lengths).  It holds none of the decode step's arithmetic, so the GPU path
 * and the CPU oracle can both be fed from it without sharing any of the
 * computation they are compared on.
 *
 * Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014): state advances by the golden-ratio gamma
 * 0x9E3779B97F4A7C15 and each output is the state passed through the
 * variant-13 mixer (xor-shift 30, multiply 0xBF58476D1CE4E5B9, xor-shift 27,
 * multiply 0x94D049BB133111EB, xor-shift 31).  Element i of a tensor is the
 * mixer applied to key + (i + 1) * gamma, so any element can be produced
 * independently of the others (the array is generated in parallel).
 *
 * Distributions (all floating steps are single IEEE double operations, so a
 * numpy restatement reproduces every bit):
 *   int8 uniform on [-127, 127]   : (h >> 32) % 255 - 127
 *   approx. normal N(mu, sigma)   : S = sum of the four 16-bit fields of h,
 *                                   z = ((S - 131070) / 65536) * sqrt(3),
 *                                   x = mu + sigma * z      (Irwin-Hall, n=4)
 *   q8_0 weight scale             : fp16( |sigma * z| / 127 )
 *   integer uniform on [lo, hi]   : lo + (h >> 32) % (hi - lo + 1)
 */
#include <stdint.h>
#include <stddef.h>

#define SM_GAMMA 0x9E3779B97F4A7C15ULL
#define SQRT3 1.7320508075688772

static inline uint64_t sm_mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Stream key of tensor `tensor` under `seed`. */
uint64_t synth_key(uint64_t seed, uint64_t tensor)
{
    return sm_mix(sm_mix(seed * SM_GAMMA + 0x243F6A8885A308D3ULL) ^ (tensor * 0xD1B54A32D192ED03ULL));
}

static inline uint64_t sm_at(uint64_t key, uint64_t i)
{
    return sm_mix(key + (i + 1) * SM_GAMMA);
}

static inline double sm_z(uint64_t h)
{
    int64_t s = (int64_t)(h & 0xFFFF) + (int64_t)((h >> 16) & 0xFFFF) +
                (int64_t)((h >> 32) & 0xFFFF) + (int64_t)(h >> 48);
    double z = (double)(s - 131070) / 65536.0;
    return z * SQRT3;
}

void synth_u64(uint64_t seed, uint64_t tensor, uint64_t off, int64_t n, uint64_t* out)
{
    uint64_t key = synth_key(seed, tensor);
#pragma omp parallel for schedule(static) if (n > (1 << 20))
    for (int64_t i = 0; i < n; ++i) out[i] = sm_at(key, off + (uint64_t)i);
}

void synth_int8(uint64_t seed, uint64_t tensor, uint64_t off, int64_t n, int8_t* out)
{
    uint64_t key = synth_key(seed, tensor);
#pragma omp parallel for schedule(static) if (n > (1 << 20))
    for (int64_t i = 0; i < n; ++i) {
        uint64_t h = sm_at(key, off + (uint64_t)i);
        out[i] = (int8_t)((int)((h >> 32) % 255u) - 127);
    }
}

void synth_normal_f64(uint64_t seed, uint64_t tensor, uint64_t off, int64_t n,
                      double mu, double sigma, double* out)
{
    uint64_t key = synth_key(seed, tensor);
#pragma omp parallel for schedule(static) if (n > (1 << 20))
    for (int64_t i = 0; i < n; ++i) {
        double sz = sigma * sm_z(sm_at(key, off + (uint64_t)i));
        out[i] = mu + sz;
    }
}

void synth_normal_f32(uint64_t seed, uint64_t tensor, uint64_t off, int64_t n,
                      double mu, double sigma, float* out)
{
    uint64_t key = synth_key(seed, tensor);
#pragma omp parallel for schedule(static) if (n > (1 << 20))
    for (int64_t i = 0; i < n; ++i) {
        double sz = sigma * sm_z(sm_at(key, off + (uint64_t)i));
        out[i] = (float)(mu + sz);
    }
}

void synth_normal_f16(uint64_t seed, uint64_t tensor, uint64_t off, int64_t n,
                      double mu, double sigma, _Float16* out)
{
    uint64_t key = synth_key(seed, tensor);
#pragma omp parallel for schedule(static) if (n > (1 << 20))
    for (int64_t i = 0; i < n; ++i) {
        double sz = sigma * sm_z(sm_at(key, off + (uint64_t)i));
        out[i] = (_Float16)(mu + sz);
    }
}

void synth_q8_scale_f16(uint64_t seed, uint64_t tensor, uint64_t off, int64_t n,
                        double sigma, _Float16* out)
{
    uint64_t key = synth_key(seed, tensor);
#pragma omp parallel for schedule(static) if (n > (1 << 20))
    for (int64_t i = 0; i < n; ++i) {
        double sz = sigma * sm_z(sm_at(key, off + (uint64_t)i));
        if (sz < 0) sz = -sz;
        out[i] = (_Float16)(sz / 127.0);
    }
}

void synth_int_uniform(uint64_t seed, uint64_t tensor, uint64_t off, int64_t n,
                       int64_t lo, int64_t hi, int64_t* out)
{
    uint64_t key = synth_key(seed, tensor);
    uint64_t span = (uint64_t)(hi - lo + 1);
    for (int64_t i = 0; i < n; ++i) {
        uint64_t h = sm_at(key, off + (uint64_t)i);
        out[i] = lo + (int64_t)((h >> 32) % span);
    }
}

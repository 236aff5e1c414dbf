/*
 * Seeded synthetic inputs for the ternary linear layer and its optimizer step.
 *
 * This module is shared by the CUDA path's tests/bench and by the CPU oracle's
 * tests.  It holds only random-number generation and input formatting (fp64 ->
 * fp32 -> bf16 rounding of the drawn values); none of the layer's arithmetic.
 *
 * Generator: a counter-based splitmix64 stream.  Tensor `tid` of a workload
 * with seed `seed` has key k = mix(seed ^ (tid * G)) with G = 0x9E3779B97F4A7C15,
 * and its draw number j is d(j) = mix(k + (j + 1) * G), where mix is the
 * splitmix64 finaliser (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014).  Element i of every tensor uses draws 2i and
 * 2i + 1 only, so any element can be regenerated on its own (random access) and
 * a slice [start, start + n) equals the same slice of the whole tensor.
 *
 *   uniform u in [0,1)   : (d >> 11) * 2^-53
 *   normal               : Box-Muller, cosine branch, sqrt(-2 ln(1 - u1)) cos(2 pi u2)
 *   integer in [lo, hi]  : lo + (((d >> 32) * (hi - lo + 1)) >> 32)   (Lemire's
 *                          multiply-shift; bias below (hi-lo+1) / 2^32)
 *   forced zero          : draw 2i is a uniform; u < p gives 0, draw 2i+1 the value
 *   bf16                 : fp64 -> fp32 (round to nearest even) -> bf16 (round to
 *                          nearest even on the upper 16 bits)
 *
 * Threads: every entry point splits [start, start+n) over up to `nthreads`
 * pthreads; the result does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>
#include <unistd.h>

#define SYN_GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t syn_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t synth_key(uint64_t seed, uint64_t tid) { return syn_mix(seed ^ (tid * SYN_GOLDEN)); }

static inline uint64_t syn_draw(uint64_t key, uint64_t j) { return syn_mix(key + (j + 1) * SYN_GOLDEN); }

static inline double syn_unit(uint64_t d) { return (double)(d >> 11) * (1.0 / 9007199254740992.0); }

static inline double syn_normal(uint64_t key, uint64_t i) {
    double u1 = syn_unit(syn_draw(key, 2 * i));
    double u2 = syn_unit(syn_draw(key, 2 * i + 1));
    return sqrt(-2.0 * log(1.0 - u1)) * cos(6.283185307179586476925286766559 * u2);
}

static inline uint16_t syn_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u = u + 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

enum { K_NORMAL_BF16, K_NORMAL_F32, K_UNIFORM_F32, K_INT8 };

typedef struct {
    int kind;
    uint64_t key;
    double a, b, p;
    int64_t lo, hi;
    int64_t start, n;
    void* out;
} syn_job;

static void syn_run(const syn_job* j, int64_t i0, int64_t i1) {
    for (int64_t t = i0; t < i1; ++t) {
        uint64_t i = (uint64_t)(j->start + t);
        switch (j->kind) {
        case K_NORMAL_BF16:
            ((uint16_t*)j->out)[t] = syn_f32_to_bf16((float)(j->a + j->b * syn_normal(j->key, i)));
            break;
        case K_NORMAL_F32:
            ((float*)j->out)[t] = (float)(j->a + j->b * syn_normal(j->key, i));
            break;
        case K_UNIFORM_F32:
            ((float*)j->out)[t] = (float)(j->a + (j->b - j->a) * syn_unit(syn_draw(j->key, 2 * i)));
            break;
        case K_INT8: {
            int8_t v;
            if (j->p > 0.0 && syn_unit(syn_draw(j->key, 2 * i)) < j->p) {
                v = 0;
            } else {
                uint64_t hi32 = syn_draw(j->key, 2 * i + 1) >> 32;
                uint64_t span = (uint64_t)(j->hi - j->lo + 1);
                v = (int8_t)(j->lo + (int64_t)((hi32 * span) >> 32));
            }
            ((int8_t*)j->out)[t] = v;
            break;
        }
        }
    }
}

typedef struct {
    const syn_job* job;
    int64_t i0, i1;
} syn_slice;

static void* syn_thread(void* arg) {
    const syn_slice* s = (const syn_slice*)arg;
    syn_run(s->job, s->i0, s->i1);
    return NULL;
}

#define SYN_MAX_THREADS 64

static void syn_parallel(const syn_job* j, int nthreads) {
    if (j->n <= 0) return;
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads > SYN_MAX_THREADS) nthreads = SYN_MAX_THREADS;
    if (nthreads < 1 || j->n < 65536) nthreads = 1;
    if (nthreads == 1) {
        syn_run(j, 0, j->n);
        return;
    }
    pthread_t th[SYN_MAX_THREADS];
    int live[SYN_MAX_THREADS];
    syn_slice sl[SYN_MAX_THREADS];
    for (int t = 0; t < nthreads; ++t) {
        sl[t].job = j;
        sl[t].i0 = j->n * t / nthreads;
        sl[t].i1 = j->n * (t + 1) / nthreads;
        live[t] = pthread_create(&th[t], NULL, syn_thread, &sl[t]) == 0;
        if (!live[t]) syn_run(j, sl[t].i0, sl[t].i1); /* no thread: do the slice here */
    }
    for (int t = 0; t < nthreads; ++t)
        if (live[t]) pthread_join(th[t], NULL);
}

void synth_normal_bf16(uint64_t seed, uint64_t tid, double mean, double std, int64_t start, int64_t n,
                       uint16_t* out, int nthreads) {
    syn_job j = {K_NORMAL_BF16, synth_key(seed, tid), mean, std, 0.0, 0, 0, start, n, out};
    syn_parallel(&j, nthreads);
}

void synth_normal_f32(uint64_t seed, uint64_t tid, double mean, double std, int64_t start, int64_t n,
                      float* out, int nthreads) {
    syn_job j = {K_NORMAL_F32, synth_key(seed, tid), mean, std, 0.0, 0, 0, start, n, out};
    syn_parallel(&j, nthreads);
}

void synth_uniform_f32(uint64_t seed, uint64_t tid, double lo, double hi, int64_t start, int64_t n,
                       float* out, int nthreads) {
    syn_job j = {K_UNIFORM_F32, synth_key(seed, tid), lo, hi, 0.0, 0, 0, start, n, out};
    syn_parallel(&j, nthreads);
}

void synth_int8(uint64_t seed, uint64_t tid, int64_t lo, int64_t hi, double zero_prob, int64_t start,
                int64_t n, int8_t* out, int nthreads) {
    syn_job j = {K_INT8, synth_key(seed, tid), 0.0, 0.0, zero_prob, lo, hi, start, n, out};
    syn_parallel(&j, nthreads);
}

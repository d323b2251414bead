/*
 * synthgen/synth.c — seeded, counter-based synthetic gradient generators.
 *
 * This module only draws input values. It contains none of the allreduce
 * arithmetic (no combining, no rounding to a reduced precision, no chunking);
 * it is shared by the CUDA path's tests/benchmark and by the CPU oracle's
 * callers, and imports neither.
 *
 * Every value is a pure function of (seed, element index), so any element of
 * any rank can be regenerated on its own, on any machine, in any thread split:
 *
 *   h(seed, k)  = SplitMix64 output for state (seed << 40) + k
 *                 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 *                 generators", OOPSLA 2014: one increment by the golden gamma,
 *                 then the 64-bit variant-13 finaliser)
 *   U(seed, k)  = ((h >> 11) + 0.5) * 2^-53          uniform on the open (0,1)
 *   normal(i)   = sqrt(-2 ln U(seed,2i)) * cos(2 pi U(seed,2i+1))   (Box–Muller,
 *                 Box & Muller 1958, cosine branch only)
 *   value(i)    = sigma * normal(i), times `outlier_scale` when the independent
 *                 stream U(seed ^ 0x5bd1e995, i) < outlier_p; rounded to fp32
 *                 by the C double->float conversion (round to nearest even).
 *   uniform(i)  = lo + (hi - lo) * U(seed, i)
 *   int(i)      = lo + (h(seed, i) mod (hi - lo + 1))      (inclusive range)
 *
 * Rank r of a workload uses seed = base + r.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>

#define SG_PI 3.14159265358979323846

static inline uint64_t sg_splitmix64(uint64_t state)
{
    uint64_t z = state + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t sg_hash(uint64_t seed, uint64_t k)
{
    return sg_splitmix64((seed << 40) + k);
}

static inline double sg_u01(uint64_t h)
{
    return ((double)(h >> 11) + 0.5) * 0x1.0p-53;
}

static inline double sg_normal(uint64_t seed, uint64_t i)
{
    double u1 = sg_u01(sg_hash(seed, 2 * i));
    double u2 = sg_u01(sg_hash(seed, 2 * i + 1));
    return sqrt(-2.0 * log(u1)) * cos(2.0 * SG_PI * u2);
}

/* kinds */
enum { SG_NORMAL = 0, SG_UNIFORM = 1, SG_INT = 2 };

typedef struct {
    int kind;
    void *out;            /* float* for NORMAL/UNIFORM, int32_t* for INT */
    uint64_t first;       /* global index of out[0] */
    size_t n;
    uint64_t seed;
    double a, b;          /* NORMAL: sigma, unused; UNIFORM/INT: lo, hi */
    double outlier_p, outlier_scale;
} sg_job;

static void sg_run(const sg_job *j, size_t lo, size_t hi)
{
    if (j->kind == SG_NORMAL) {
        float *o = (float *)j->out;
        uint64_t oseed = j->seed ^ 0x5bd1e995ull;
        for (size_t t = lo; t < hi; ++t) {
            uint64_t i = j->first + t;
            double v = j->a * sg_normal(j->seed, i);
            if (j->outlier_p > 0.0 && sg_u01(sg_hash(oseed, i)) < j->outlier_p)
                v *= j->outlier_scale;
            o[t] = (float)v;
        }
    } else if (j->kind == SG_UNIFORM) {
        float *o = (float *)j->out;
        for (size_t t = lo; t < hi; ++t) {
            uint64_t i = j->first + t;
            o[t] = (float)(j->a + (j->b - j->a) * sg_u01(sg_hash(j->seed, i)));
        }
    } else {
        int32_t *o = (int32_t *)j->out;
        int64_t ilo = (int64_t)j->a, ihi = (int64_t)j->b;
        uint64_t span = (uint64_t)(ihi - ilo) + 1u;
        for (size_t t = lo; t < hi; ++t) {
            uint64_t i = j->first + t;
            o[t] = (int32_t)(ilo + (int64_t)(sg_hash(j->seed, i) % span));
        }
    }
}

typedef struct { const sg_job *j; size_t lo, hi; } sg_slice;

static void *sg_thread(void *p)
{
    const sg_slice *s = (const sg_slice *)p;
    sg_run(s->j, s->lo, s->hi);
    return NULL;
}

static void sg_parallel(const sg_job *j, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads == 1 || j->n < 65536) { sg_run(j, 0, j->n); return; }
    pthread_t th[256];
    sg_slice sl[256];
    size_t per = (j->n + (size_t)nthreads - 1) / (size_t)nthreads;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        size_t lo = (size_t)t * per, hi = lo + per;
        if (lo >= j->n) break;
        if (hi > j->n) hi = j->n;
        sl[t].j = j; sl[t].lo = lo; sl[t].hi = hi;
        if (pthread_create(&th[t], NULL, sg_thread, &sl[t]) != 0) {
            sg_run(j, lo, hi);          /* could not start a thread: do it here */
            sl[t].j = NULL;
        }
        started = t + 1;
    }
    for (int t = 0; t < started; ++t)
        if (sl[t].j) pthread_join(th[t], NULL);
}

/* sigma * N(0,1) with optional outliers, elements [first, first+n) of stream `seed`. */
void synth_normal_f32(float *out, uint64_t first, size_t n, uint64_t seed, double sigma,
                      double outlier_p, double outlier_scale, int nthreads)
{
    sg_job j = {SG_NORMAL, out, first, n, seed, sigma, 0.0, outlier_p, outlier_scale};
    sg_parallel(&j, nthreads);
}

/* uniform on (lo, hi) */
void synth_uniform_f32(float *out, uint64_t first, size_t n, uint64_t seed, double lo, double hi,
                       int nthreads)
{
    sg_job j = {SG_UNIFORM, out, first, n, seed, lo, hi, 0.0, 0.0};
    sg_parallel(&j, nthreads);
}

/* integers uniform on [lo, hi] inclusive */
void synth_uniform_i32(int32_t *out, uint64_t first, size_t n, uint64_t seed, int64_t lo, int64_t hi,
                       int nthreads)
{
    sg_job j = {SG_INT, out, first, n, seed, (double)lo, (double)hi, 0.0, 0.0};
    sg_parallel(&j, nthreads);
}

/* exposed for the generator's own tests */
uint64_t synth_splitmix64(uint64_t state) { return sg_splitmix64(state); }

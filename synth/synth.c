/*
 * Seeded synthetic input generators for the sublayer-boundary workloads.
 *
 * This file draws random numbers and nothing else: it holds none of the
 * boundary's arithmetic (no norm, no residual scaling, no rounding to BF16).
 * It produces FP32 values; the caller converts them to BF16 storage.
 *
 * Every value is a pure function of (seed, stream, index): the generator is
 * counter based, so any slice of a tensor can be regenerated on its own and
 * the same bytes reach both the CUDA path and the CPU oracle.
 *
 *   key(seed, stream)  = mix(mix(seed + G) ^ (stream * C + G))
 *   word(key, i)       = mix(key + (i + 1) * G)          (splitmix64 step i)
 *   uniform(key, i)    = ((word >> 11) + 0.5) * 2^-53     in (0, 1)
 *   normal(key, j)     = Box-Muller on uniforms 2*(j/2), 2*(j/2)+1:
 *                        sqrt(-2 ln u1) * (j even ? cos : sin)(2 pi u2)
 *   t3_unit(key, j)    = Z / sqrt(V) with Z = normal(key, 2j),
 *                        V = -2 ln U + normal(key, 2j+1)^2 (chi-square, 3 dof),
 *                        U = uniform(key', j); Z/sqrt(V/3) is Student-t(3),
 *                        whose variance is 3, so Z/sqrt(V) has unit variance.
 *   bernoulli(key,j,p) = word(key, j) < p * 2^64
 *
 * mix() is the splitmix64 finaliser (Steele, Lea, Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014); G = 0x9E3779B97F4A7C15.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static uint64_t mix(uint64_t z) {
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ULL;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBULL;
    z ^= z >> 31;
    return z;
}

static uint64_t make_key(uint64_t seed, uint64_t stream) {
    return mix(mix(seed + GOLDEN) ^ (stream * 0xD1B54A32D192ED03ULL + GOLDEN));
}

static uint64_t word_at(uint64_t key, uint64_t i) { return mix(key + (i + 1) * GOLDEN); }

static double uniform_at(uint64_t key, uint64_t i) {
    return ((double)(word_at(key, i) >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static double normal_at(uint64_t key, uint64_t j) {
    const double two_pi = 6.283185307179586476925286766559;
    uint64_t p = j >> 1;
    double u1 = uniform_at(key, 2 * p);
    double u2 = uniform_at(key, 2 * p + 1);
    double rad = sqrt(-2.0 * log(u1));
    return (j & 1) ? rad * sin(two_pi * u2) : rad * cos(two_pi * u2);
}

static double t3_unit_at(uint64_t key, uint64_t key_u, uint64_t j) {
    double z = normal_at(key, 2 * j);
    double g = normal_at(key, 2 * j + 1);
    double v = -2.0 * log(uniform_at(key_u, j)) + g * g;
    return z / sqrt(v);
}

/* ---- threading: split [0, count) into contiguous chunks ---------------- */

enum { K_NORMAL = 0, K_T3 = 1, K_BERNOULLI = 2, K_TOPK = 3 };

typedef struct {
    int kind;
    uint64_t key, key2;
    uint64_t start, lo, hi; /* absolute index = start + i for i in [lo, hi) */
    double a, b;            /* kind-specific parameters */
    int k;                  /* top-k width for K_TOPK */
    void* out;
} job_t;

static void run_job(job_t* jb) {
    for (uint64_t i = jb->lo; i < jb->hi; ++i) {
        uint64_t j = jb->start + i;
        switch (jb->kind) {
        case K_NORMAL:
            ((float*)jb->out)[i] = (float)(jb->b + jb->a * normal_at(jb->key, j));
            break;
        case K_T3:
            ((float*)jb->out)[i] = (float)t3_unit_at(jb->key, jb->key2, j);
            break;
        case K_BERNOULLI: {
            /* p * 2^64, saturated; p in [0, 1] */
            double thr = jb->a * 18446744073709551616.0;
            uint64_t w = word_at(jb->key, j);
            ((uint8_t*)jb->out)[i] = (thr >= 18446744073709551615.0) ? 1 : ((double)w < thr);
            break;
        }
        case K_TOPK: {
            /* row j: z_k ~ N(0,1); s_k = logistic(z_k); w_k = scale * s_k / sum(s) */
            double s[64], tot = 0.0;
            int k = jb->k;
            for (int q = 0; q < k; ++q) {
                double z = normal_at(jb->key, j * (uint64_t)k + (uint64_t)q);
                s[q] = 1.0 / (1.0 + exp(-z));
                tot += s[q];
            }
            for (int q = 0; q < k; ++q)
                ((float*)jb->out)[i * (uint64_t)k + (uint64_t)q] = (float)(jb->a * s[q] / tot);
            break;
        }
        }
    }
}

static void* thread_main(void* p) {
    run_job((job_t*)p);
    return NULL;
}

static void run_parallel(job_t proto, uint64_t count, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((uint64_t)nthreads > count) nthreads = count ? (int)count : 1;
    job_t jobs[256];
    pthread_t tid[256];
    uint64_t per = count / (uint64_t)nthreads, rem = count % (uint64_t)nthreads, lo = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = proto;
        jobs[t].lo = lo;
        jobs[t].hi = lo + per + ((uint64_t)t < rem ? 1 : 0);
        lo = jobs[t].hi;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, thread_main, &jobs[t]) != 0) break;
        started = t;
    }
    run_job(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tid[t], NULL);
    for (int t = started + 1; t < nthreads; ++t) run_job(&jobs[t]); /* thread creation failed */
}

/* ---- exported API --------------------------------------------------------- */

/* out[i] = offset + scale * normal(start + i), i in [0, count) */
void synth_normal(uint64_t seed, uint64_t stream, uint64_t start, uint64_t count,
                  double scale, double offset, float* out, int nthreads) {
    job_t jb = {K_NORMAL, make_key(seed, stream), 0, start, 0, 0, scale, offset, 0, out};
    run_parallel(jb, count, nthreads);
}

/* out[i] = t3_unit(start + i): Student-t with 3 degrees of freedom scaled to unit variance */
void synth_student_t3_unit(uint64_t seed, uint64_t stream, uint64_t start, uint64_t count,
                           float* out, int nthreads) {
    job_t jb = {K_T3, make_key(seed, stream), make_key(seed, stream ^ 0x5555555555555555ULL),
                start, 0, 0, 0.0, 0.0, 0, out};
    run_parallel(jb, count, nthreads);
}

/* out[i] = 1 with probability p (counter-hash threshold), else 0 */
void synth_bernoulli(uint64_t seed, uint64_t stream, uint64_t start, uint64_t count, double p,
                     uint8_t* out, int nthreads) {
    job_t jb = {K_BERNOULLI, make_key(seed, stream), 0, start, 0, 0, p, 0.0, 0, out};
    run_parallel(jb, count, nthreads);
}

/* Routing weights for rows [row_start, row_start + rows): out[r, q] for q < k (k <= 64):
 * z ~ N(0,1), s = 1 / (1 + exp(-z)) in double, w = scale * s / sum_q s, stored as float. */
int synth_topk_weights(uint64_t seed, uint64_t stream, uint64_t row_start, uint64_t rows, int k,
                       double scale, float* out, int nthreads) {
    if (k < 1 || k > 64) return -1;
    job_t jb = {K_TOPK, make_key(seed, stream), 0, row_start, 0, 0, scale, 0.0, k, out};
    run_parallel(jb, rows, nthreads);
    return 0;
}

/* raw splitmix words, for tests of the generator itself */
void synth_words(uint64_t seed, uint64_t stream, uint64_t start, uint64_t count, uint64_t* out) {
    uint64_t key = make_key(seed, stream);
    for (uint64_t i = 0; i < count; ++i) out[i] = word_at(key, start + i);
}

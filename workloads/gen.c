/*
 * Seeded synthetic input generators shared by the CPU oracle and the CUDA path.
 *
 * This file holds no attention arithmetic.  It only turns (seed, stream,
 * counter) into numbers:
 *   - splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
 *     generators", OOPSLA 2014), evaluated in counter form: output k of a
 *     stream whose state starts at s is mix(s + (k+1)*0x9E3779B97F4A7C15);
 *   - uniform doubles on [0,1) from the top 53 bits;
 *   - standard normals by the Box-Muller transform (Box & Muller, 1958),
 *     rounded to float and then to bfloat16 with round-to-nearest-even.
 *
 * Every function is a pure function of (seed, stream, index), so any range of
 * indices can be produced independently and by several threads; the result
 * does not depend on the thread count or on the machine (compile with
 * -ffp-contract=off so no fused multiply-add changes a rounding).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Starting state of stream `stream` under `seed`. */
static inline uint64_t stream_state(uint64_t seed, uint64_t stream) {
    return mix64(mix64(seed + GOLDEN) ^ mix64((stream + 1) * 0xD1B54A32D192ED03ULL));
}

/* Output number k (k = 0, 1, ...) of the splitmix64 sequence started at s. */
static inline uint64_t at(uint64_t s, uint64_t k) { return mix64(s + (k + 1) * GOLDEN); }

static inline double u01(uint64_t x) { return (double)(x >> 11) * (1.0 / 9007199254740992.0); }

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* Normal deviate number `e` of the stream: pairs (2p, 2p+1) share one
 * Box-Muller draw (cos for the even member, sin for the odd one). */
static inline double normal_at(uint64_t s, uint64_t e) {
    uint64_t p = e >> 1;
    double u1 = (double)((at(s, 2 * p) >> 11) + 1) * (1.0 / 9007199254740992.0); /* (0,1] */
    double u2 = u01(at(s, 2 * p + 1));
    double r = sqrt(-2.0 * log(u1));
    double th = 6.283185307179586476925286766559 * u2;
    return (e & 1) ? r * sin(th) : r * cos(th);
}

typedef struct {
    uint64_t state, offset;
    int64_t lo, hi;
    void *out;
    int what;
} job_t;

static void *worker(void *arg) {
    job_t *j = (job_t *)arg;
    for (int64_t i = j->lo; i < j->hi; ++i) {
        uint64_t e = j->offset + (uint64_t)i;
        if (j->what == 0)
            ((uint16_t *)j->out)[i] = f32_to_bf16_rne((float)normal_at(j->state, e));
        else if (j->what == 1)
            ((double *)j->out)[i] = u01(at(j->state, e));
        else
            ((uint64_t *)j->out)[i] = at(j->state, e);
    }
    return 0;
}

static void run(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, void *out, int what,
                int threads) {
    if (n <= 0) return;
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if (n < 65536) threads = 1;
    pthread_t tid[256];
    job_t jobs[256];
    uint64_t st = stream_state(seed, stream);
    for (int t = 0; t < threads; ++t) {
        jobs[t].state = st;
        jobs[t].offset = offset;
        jobs[t].lo = n * t / threads;
        jobs[t].hi = n * (t + 1) / threads;
        jobs[t].out = out;
        jobs[t].what = what;
    }
    int started = 0;
    for (int t = 1; t < threads; ++t)
        if (pthread_create(&tid[t], 0, worker, &jobs[t]) == 0) started = t;
        else { worker(&jobs[t]); }
    worker(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tid[t], 0);
}

/* out[i] = bf16 bits of N(0,1) deviate number (offset + i) of (seed, stream). */
void bsgen_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, uint16_t *out,
                       int threads) {
    run(seed, stream, offset, n, out, 0, threads);
}

/* out[i] = uniform double on [0,1), number (offset + i) of (seed, stream). */
void bsgen_uniform01(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double *out,
                     int threads) {
    run(seed, stream, offset, n, out, 1, threads);
}

/* out[i] = raw 64-bit output number (offset + i) of (seed, stream). */
void bsgen_u64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, uint64_t *out,
               int threads) {
    run(seed, stream, offset, n, out, 2, threads);
}

/*
 * Seeded synthetic inputs for the chunked linear cross-entropy workloads:
 * the fast C twin of the numpy definition in lce_inputs/__init__.py.
 *
 * This file holds no arithmetic of the loss itself.  It only turns
 * (seed, tensor id, element index) into a bf16 value, so that the oracle
 * and the GPU library can be fed the very same bits, and so that the
 * oracle can regenerate any sampled row of a tensor without generating
 * the rest of it.
 *
 * Stream: counter-based SplitMix64 (Steele, Lea and Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014).  Draw n of
 * stream `key` is mix64(key + (n + 1) * GAMMA), i.e. the (n+1)-th output
 * of a SplitMix64 generator whose state starts at `key`.
 * Normals: the Box-Muller transform (Box and Muller, 1958).  Pair k uses
 * draws 2k and 2k+1; element 2k takes r*cos(theta), element 2k+1 takes
 * r*sin(theta).
 * Rounding: sigma * normal in double -> float32 (round to nearest even)
 * -> bf16 (round to nearest even), the same as torch's
 * .to(float32).to(bfloat16).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t lce_inputs_stream_key(uint64_t seed, uint64_t tensor_id) {
    return mix64(mix64(seed + GAMMA) ^ (tensor_id * 0xD1B54A32D192ED03ULL));
}

static inline uint64_t draw(uint64_t key, uint64_t n) {
    return mix64(key + (n + 1) * GAMMA);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u) /* inf / nan: keep, quiet nan */
        return (uint16_t)((u >> 16) | ((u & 0x007FFFFFu) ? 0x40u : 0u));
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

static void normal_pair(uint64_t key, uint64_t k, double* c, double* s) {
    const double two_pi = 6.283185307179586476925286766559;
    double u1 = 1.0 - (double)(draw(key, 2 * k) >> 11) * 0x1.0p-53;     /* (0, 1] */
    double u2 = (double)(draw(key, 2 * k + 1) >> 11) * 0x1.0p-53;       /* [0, 1) */
    double r = sqrt(-2.0 * log(u1));
    double t = two_pi * u2;
    *c = r * cos(t);
    *s = r * sin(t);
}

typedef struct {
    uint64_t key, start, count;
    double sigma;
    uint16_t* out;
} job_t;

static void* run_job(void* p) {
    job_t* j = (job_t*)p;
    uint64_t e = j->start, end = j->start + j->count;
    while (e < end) {
        double c, s;
        uint64_t k = e >> 1;
        normal_pair(j->key, k, &c, &s);
        if ((e & 1) == 0) {
            j->out[e - j->start] = f32_to_bf16_rne((float)(j->sigma * c));
            ++e;
            if (e < end) {
                j->out[e - j->start] = f32_to_bf16_rne((float)(j->sigma * s));
                ++e;
            }
        } else {
            j->out[e - j->start] = f32_to_bf16_rne((float)(j->sigma * s));
            ++e;
        }
    }
    return NULL;
}

/* Fill out[0..count) with elements start..start+count-1 of the normal
 * stream (seed, tensor_id) scaled by sigma, rounded to bf16.  Returns 0,
 * or -1 when a worker thread could not be started. */
int lce_inputs_normal_bf16(uint64_t seed, uint64_t tensor_id, uint64_t start,
                           uint64_t count, double sigma, uint16_t* out,
                           int threads) {
    enum { MAXT = 256 };
    if (threads < 1) threads = 1;
    if (threads > MAXT) threads = MAXT;
    if ((uint64_t)threads > count / 65536 + 1) threads = (int)(count / 65536 + 1);
    uint64_t key = lce_inputs_stream_key(seed, tensor_id);
    job_t jobs[MAXT];
    pthread_t tids[MAXT];
    int created[MAXT];
    uint64_t per = (count + threads - 1) / threads;
    int rc = 0, njobs = 0;
    for (int t = 0; t < threads; ++t) {
        uint64_t b = (uint64_t)t * per;
        if (b >= count) break;
        jobs[t].key = key;
        jobs[t].start = start + b;
        jobs[t].count = count - b < per ? count - b : per;
        jobs[t].sigma = sigma;
        jobs[t].out = out + b;
        njobs = t + 1;
    }
    /* job 0 runs on the calling thread; a job whose thread cannot be
     * started runs there too */
    for (int t = 1; t < njobs; ++t) {
        created[t] = pthread_create(&tids[t], NULL, run_job, &jobs[t]) == 0;
        if (!created[t]) rc = -1;
    }
    if (njobs > 0) run_job(&jobs[0]);
    for (int t = 1; t < njobs; ++t) {
        if (created[t])
            pthread_join(tids[t], NULL);
        else
            run_job(&jobs[t]);
    }
    return rc;
}

/* Raw 64-bit draws n = start..start+count-1 of stream (seed, tensor_id). */
void lce_inputs_u64(uint64_t seed, uint64_t tensor_id, uint64_t start,
                    uint64_t count, uint64_t* out) {
    uint64_t key = lce_inputs_stream_key(seed, tensor_id);
    for (uint64_t i = 0; i < count; ++i) out[i] = draw(key, start + i);
}

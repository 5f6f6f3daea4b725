/* Multithreaded fill for the seeded synthetic input generator (synth.py holds the
 * definition and a numpy implementation of the same stream; tests check that both give
 * identical bits). Counter-based: element i depends only on (key, i), so threads split the
 * index range freely. Inputs only: none of the attention method's arithmetic is here.
 *
 * SplitMix64 output function: Steele, Lea, Flood, OOPSLA 2014. Box-Muller transform:
 * Box and Muller, Ann. Math. Statist. 1958. Build with -ffp-contract=off.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define G 0x9E3779B97F4A7C15ULL

static uint64_t mix64(uint64_t z) {
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ULL;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBULL;
    z ^= z >> 31;
    return z;
}

static double normal_at(uint64_t key, uint64_t i) {
    const uint64_t j = i >> 1;
    const uint64_t h1 = mix64(key + (2 * j + 1) * G);
    const uint64_t h2 = mix64(key + (2 * j + 2) * G);
    const double u1 = ((double)(h1 >> 11) + 0.5) * 0x1.0p-53;
    const double u2 = (double)(h2 >> 11) * 0x1.0p-53;
    const double r = sqrt(-2.0 * log(u1));
    const double phi = (2.0 * 3.141592653589793) * u2;
    return (i & 1) ? r * sin(phi) : r * cos(phi);
}

static uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0;
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

typedef struct {
    uint64_t key, start, count;
    double mean, std;
    void* out;
    int bf16;
} job_t;

static void put(job_t* jb, uint64_t k, double z) {
    const float v = (float)(jb->mean + jb->std * z);
    if (jb->bf16) ((uint16_t*)jb->out)[k] = f32_to_bf16(v);
    else ((float*)jb->out)[k] = v;
}

static void* run(void* arg) {
    job_t* jb = (job_t*)arg;
    uint64_t k = 0;
    if (jb->count && ((jb->start + k) & 1)) { put(jb, k, normal_at(jb->key, jb->start + k)); ++k; }
    for (; k + 1 < jb->count; k += 2) {            /* whole Box-Muller pairs */
        const uint64_t j = (jb->start + k) >> 1;
        const uint64_t h1 = mix64(jb->key + (2 * j + 1) * G);
        const uint64_t h2 = mix64(jb->key + (2 * j + 2) * G);
        const double u1 = ((double)(h1 >> 11) + 0.5) * 0x1.0p-53;
        const double u2 = (double)(h2 >> 11) * 0x1.0p-53;
        const double r = sqrt(-2.0 * log(u1));
        const double phi = (2.0 * 3.141592653589793) * u2;
        put(jb, k, r * cos(phi));
        put(jb, k + 1, r * sin(phi));
    }
    if (k < jb->count) put(jb, k, normal_at(jb->key, jb->start + k));
    return 0;
}

static void fill(uint64_t key, uint64_t start, uint64_t count, double mean, double std, void* out,
                 int bf16, int threads) {
    if (threads < 1) threads = 1;
    if (threads > 64) threads = 64;
    if (count < (1u << 16)) threads = 1;
    pthread_t th[64];
    job_t jobs[64];
    const uint64_t per = (count + threads - 1) / threads;
    int started = 0;
    for (int t = 0; t < threads; ++t) {
        const uint64_t s = per * t;
        if (s >= count) break;
        jobs[t].key = key;
        jobs[t].start = start + s;
        jobs[t].count = (s + per <= count) ? per : count - s;
        jobs[t].mean = mean;
        jobs[t].std = std;
        jobs[t].out = bf16 ? (void*)((uint16_t*)out + s) : (void*)((float*)out + s);
        jobs[t].bf16 = bf16;
        if (pthread_create(&th[t], 0, run, &jobs[t]) != 0) { run(&jobs[t]); th[t] = 0; }
        ++started;
    }
    for (int t = 0; t < started; ++t)
        if (th[t]) pthread_join(th[t], 0);
}

void synth_normal_bf16(uint64_t key, uint64_t start, uint64_t count, double mean, double std,
                       uint16_t* out, int threads) {
    fill(key, start, count, mean, std, out, 1, threads);
}

void synth_normal_f32(uint64_t key, uint64_t start, uint64_t count, double mean, double std,
                      float* out, int threads) {
    fill(key, start, count, mean, std, out, 0, threads);
}

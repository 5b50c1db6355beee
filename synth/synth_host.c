/*
 * Host side of the synthetic input generator (see gen.h): fills whole ranges
 * with a few threads, or gathers single elements by index.  Built with
 * -ffp-contract=off; the only floating-point operations are one double
 * multiply and the double->float conversion, both IEEE round-to-nearest.
 */
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#include "gen.h"

static inline float syn_to_f32(const syn_stream_t* st, uint64_t n) {
    return (float)syn_value(st, n);
}

static inline uint16_t syn_to_bf16(const syn_stream_t* st, uint64_t n) {
    float f = syn_to_f32(st, n);
    uint32_t b;
    memcpy(&b, &f, 4);
    return syn_f32bits_to_bf16(b);
}

static inline uint16_t syn_to_f16(const syn_stream_t* st, uint64_t n) {
    float f = syn_to_f32(st, n);
    uint32_t b;
    memcpy(&b, &f, 4);
    return syn_f32bits_to_f16(b);
}

typedef struct {
    syn_stream_t st;
    int64_t start, lo, hi;
    void* out;
    int is_bf16;   /* 1: bf16, 2: fp16, 0: fp32 */
} job_t;

static void* worker(void* arg) {
    job_t* j = (job_t*)arg;
    if (j->is_bf16 == 1) {
        uint16_t* o = (uint16_t*)j->out;
        for (int64_t i = j->lo; i < j->hi; ++i) o[i] = syn_to_bf16(&j->st, (uint64_t)(j->start + i));
    } else if (j->is_bf16 == 2) {
        uint16_t* o = (uint16_t*)j->out;
        for (int64_t i = j->lo; i < j->hi; ++i) o[i] = syn_to_f16(&j->st, (uint64_t)(j->start + i));
    } else {
        float* o = (float*)j->out;
        for (int64_t i = j->lo; i < j->hi; ++i) o[i] = syn_to_f32(&j->st, (uint64_t)(j->start + i));
    }
    return NULL;
}

#define SYN_MAX_THREADS 256

static void fill(const syn_stream_t* st, int64_t start, int64_t n, void* out, int is_bf16, int nthreads) {
    if (n <= 0) return;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > SYN_MAX_THREADS) nthreads = SYN_MAX_THREADS;
    if (n < 65536) nthreads = 1;
    job_t jobs[SYN_MAX_THREADS];
    pthread_t th[SYN_MAX_THREADS];
    int running[SYN_MAX_THREADS];
    int64_t chunk = (n + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].st = *st;
        jobs[t].start = start;
        jobs[t].lo = (int64_t)t * chunk < n ? (int64_t)t * chunk : n;
        jobs[t].hi = jobs[t].lo + chunk < n ? jobs[t].lo + chunk : n;
        jobs[t].out = out;
        jobs[t].is_bf16 = is_bf16;
        running[t] = 0;
        if (t > 0 && jobs[t].lo < jobs[t].hi)
            running[t] = pthread_create(&th[t], NULL, worker, &jobs[t]) == 0;
        if (t > 0 && !running[t]) worker(&jobs[t]);  /* inline if no thread */
    }
    worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (running[t]) pthread_join(th[t], NULL);
}

/* Fill out[0..n) with elements start..start+n-1 of the stream. */
void synth_fill_bf16(const syn_stream_t* st, int64_t start, int64_t n, uint16_t* out, int nthreads) {
    fill(st, start, n, out, 1, nthreads);
}

void synth_fill_f32(const syn_stream_t* st, int64_t start, int64_t n, float* out, int nthreads) {
    fill(st, start, n, out, 0, nthreads);
}

void synth_fill_f16(const syn_stream_t* st, int64_t start, int64_t n, uint16_t* out, int nthreads) {
    fill(st, start, n, out, 2, nthreads);
}

void synth_gather_f16(const syn_stream_t* st, const int64_t* idx, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = syn_to_f16(st, (uint64_t)idx[i]);
}

uint16_t synth_f32bits_to_f16(uint32_t b) { return syn_f32bits_to_f16(b); }

/* out[i] = element idx[i] of the stream. */
void synth_gather_bf16(const syn_stream_t* st, const int64_t* idx, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = syn_to_bf16(st, (uint64_t)idx[i]);
}

void synth_gather_f32(const syn_stream_t* st, const int64_t* idx, int64_t n, float* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = syn_to_f32(st, (uint64_t)idx[i]);
}

/* Raw pieces, for the generator's own tests. */
uint64_t synth_mix64(uint64_t z) { return syn_mix64(z); }
double synth_normal(uint64_t key, uint64_t n) { return syn_normal(key, n); }
int synth_is_outlier(uint64_t key_out, uint64_t n, uint32_t thr) { return syn_is_outlier(key_out, n, thr); }

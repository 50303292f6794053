/*
 * Multithreaded CPU baseline: a blocked three-phase int32 exclusive add-scan
 * on the host's cores (POSIX threads).
 *
 * TEST INFRASTRUCTURE ONLY, like oracle.c beside it: the benchmark times it
 * as a CPU baseline and the tests check it against the serial oracle.  It is
 * not the oracle (parity is always judged against the serial definition in
 * oracle.c) and shares no code with the CUDA library.
 *
 * The scheme is the multi-block scan of geek-doc.cn "并行前缀和 scan ..."
 * section 四 and lpnh.cn "并行扫描" section 3.2, with CPU threads in place
 * of thread blocks:
 *   1. every thread sums its contiguous chunk;
 *   2. one thread turns the chunk sums into exclusive chunk offsets;
 *   3. every thread scans its chunk serially from its offset.
 * lpnh.cn section 5.1 advises tasks of at least 16 KB, so a chunk holds at
 * least 4,096 elements and fewer threads run on small inputs.  int32
 * addition wraps modulo 2^32 (computed in uint32_t), as in the oracle.
 */
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>

#define MT_MIN_CHUNK 4096u   /* elements: 16 KB of int32 */
#define MT_MAX_THREADS 256

struct mt_job {
    const int32_t *x;
    int32_t *y;
    size_t begin, end;
    uint32_t sum;      /* phase 1 result */
    uint32_t offset;   /* phase 2 result, phase 3 input */
};

static void *mt_sum(void *arg)
{
    struct mt_job *j = (struct mt_job *)arg;
    uint32_t s = 0;
    for (size_t i = j->begin; i < j->end; ++i) s += (uint32_t)j->x[i];
    j->sum = s;
    return NULL;
}

static void *mt_scan(void *arg)
{
    struct mt_job *j = (struct mt_job *)arg;
    uint32_t acc = j->offset;
    for (size_t i = j->begin; i < j->end; ++i) {
        j->y[i] = (int32_t)acc;
        acc += (uint32_t)j->x[i];
    }
    return NULL;
}

/* Runs fn on every job: jobs 1 .. threads-1 on their own threads, job 0 and
 * any job whose thread could not be started on the calling thread. */
static void mt_run(void *(*fn)(void *), struct mt_job *jobs, int threads)
{
    pthread_t tid[MT_MAX_THREADS];
    int ok[MT_MAX_THREADS] = {0};
    for (int t = 1; t < threads; ++t) ok[t] = pthread_create(&tid[t], NULL, fn, &jobs[t]) == 0;
    fn(&jobs[0]);
    for (int t = 1; t < threads; ++t) {
        if (ok[t])
            pthread_join(tid[t], NULL);
        else
            fn(&jobs[t]);
    }
}

/* y[i] = x[0] + ... + x[i-1] (wrapping), y[0] = 0, on up to `threads`
 * threads; returns the number of chunks (threads) used. */
int mt_scan_excl_add_i32(const int32_t *x, int32_t *y, size_t n, int threads)
{
    if (threads < 1) threads = 1;
    if (threads > MT_MAX_THREADS) threads = MT_MAX_THREADS;
    size_t most = n / MT_MIN_CHUNK;
    if (most < 1) most = 1;
    if ((size_t)threads > most) threads = (int)most;
    struct mt_job jobs[MT_MAX_THREADS];
    const size_t chunk = (n + (size_t)threads - 1) / (size_t)threads;
    for (int t = 0; t < threads; ++t) {
        size_t b = (size_t)t * chunk, e = b + chunk;
        if (b > n) b = n;
        if (e > n) e = n;
        jobs[t].x = x;
        jobs[t].y = y;
        jobs[t].begin = b;
        jobs[t].end = e;
        jobs[t].sum = 0;
        jobs[t].offset = 0;
    }
    mt_run(mt_sum, jobs, threads);                   /* 1. chunk sums */
    uint32_t run = 0;                                /* 2. chunk offsets */
    for (int t = 0; t < threads; ++t) {
        jobs[t].offset = run;
        run += jobs[t].sum;
    }
    mt_run(mt_scan, jobs, threads);                  /* 3. chunk scans */
    return threads;
}

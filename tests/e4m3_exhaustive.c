/*
 * e4m3_exhaustive.c -- test helper: the oracle's E4M3 encoder checked on every
 * one of the 2^32 binary32 bit patterns ("Engines for the card you have",
 * section "One checkpoint, many engines": an FP8 key/value cache; the format
 * is OCP E4M3: bias 7, largest finite value 448, no infinities, S.1111.111 is
 * NaN, and the store rounds to nearest with ties to even and saturates).
 *
 * Compiled together with oracle/oracle.c by tests/test_oracle_e4m3_exhaustive.py
 * and called through ctypes.  For each pattern x it checks, against the
 * decoder (itself pinned code by code against the OCP field definition):
 *   [0] NaN in           -> code 0x7F
 *   [1] not NaN in       -> a finite code, with x's sign bit
 *   [2] |x| >= 448 or inf -> +-448 (0x7E / 0xFE)
 *   [3] |x| < 448        -> the code is a nearest finite value: no neighbour
 *                           code (one up, one down) is strictly closer
 *   [4] exact ties       -> the even code
 *   [5] monotone         -> for x >= +0 in increasing order, the codes never
 *                           decrease (positive codes increase with value)
 *   [6] symmetric        -> code(-x) == code(x) | 0x80
 * and decode -> encode gives back every finite code ([7]).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

uint8_t oracle_e4m3_from_f32(float x);
double oracle_e4m3_to_f64(uint8_t code);

enum { N_CHECKS = 8 };

static double g_val[256];

static float f32_of(uint32_t u)
{
    float f;
    memcpy(&f, &u, 4);
    return f;
}

typedef struct {
    uint64_t begin, end; /* pattern range [begin, end) within 0 .. 2^32 */
    uint64_t bad[N_CHECKS];
    uint32_t first_bad[N_CHECKS];
} job_t;

static void note(job_t *j, int k, uint32_t u)
{
    if (j->bad[k]++ == 0)
        j->first_bad[k] = u;
}

static void *run(void *arg)
{
    job_t *j = (job_t *)arg;
    int prev = -1; /* code of the previous positive pattern (monotonicity) */
    if (j->begin > 0 && j->begin <= 0x7f800000u)
        prev = oracle_e4m3_from_f32(f32_of((uint32_t)(j->begin - 1)));
    for (uint64_t p = j->begin; p < j->end; ++p) {
        const uint32_t u = (uint32_t)p;
        const float x = f32_of(u);
        const uint8_t c = oracle_e4m3_from_f32(x);
        if (isnan(x)) {
            if (c != 0x7f)
                note(j, 0, u);
            continue;
        }
        const uint8_t mag = c & 0x7f;
        if (mag == 0x7f || (c & 0x80) != ((u >> 31) ? 0x80 : 0x00))
            note(j, 1, u);
        const double a = fabs((double)x);
        if (a >= 448.0) {
            if (mag != 0x7e)
                note(j, 2, u);
        } else if (mag <= 0x7e) {
            const double d = fabs(a - g_val[mag]);
            const double dn = mag > 0 ? fabs(a - g_val[mag - 1]) : INFINITY;
            const double up = mag < 0x7e ? fabs(a - g_val[mag + 1]) : INFINITY;
            if (dn < d || up < d)
                note(j, 3, u);
            if ((dn == d || up == d) && (mag & 1))
                note(j, 4, u);
        }
        if (u <= 0x7f800000u) {
            if ((int)mag < prev)
                note(j, 5, u);
            prev = mag;
        }
        if (u < 0x80000000u) {
            const uint8_t cn = oracle_e4m3_from_f32(-x);
            if (cn != (uint8_t)(c | 0x80))
                note(j, 6, u);
        }
    }
    return NULL;
}

/* Run every check over all 2^32 patterns on n_threads threads.  bad[k] gets
 * the number of patterns failing check k, first_bad[k] the first of them. */
void e4m3_exhaustive(int n_threads, uint64_t *bad, uint32_t *first_bad)
{
    for (int c = 0; c < 256; ++c)
        g_val[c] = oracle_e4m3_to_f64((uint8_t)c);
    if (n_threads < 1)
        n_threads = 1;
    if (n_threads > 256)
        n_threads = 256;
    const uint64_t total = 1ull << 32;
    const int n_jobs = 1024; /* small pieces, handed out round robin to the threads */
    static job_t jobs[1024];
    for (int i = 0; i < n_jobs; ++i) {
        memset(&jobs[i], 0, sizeof(job_t));
        jobs[i].begin = total / n_jobs * i;
        jobs[i].end = total / n_jobs * (i + 1);
    }
    for (int base = 0; base < n_jobs; base += n_threads) {
        pthread_t th[256];
        int n = n_jobs - base < n_threads ? n_jobs - base : n_threads;
        for (int t = 0; t < n; ++t)
            pthread_create(&th[t], NULL, run, &jobs[base + t]);
        for (int t = 0; t < n; ++t)
            pthread_join(th[t], NULL);
    }
    for (int k = 0; k < N_CHECKS; ++k) {
        bad[k] = 0;
        first_bad[k] = 0;
    }
    for (int i = 0; i < n_jobs; ++i)
        for (int k = 0; k < N_CHECKS; ++k)
            if (jobs[i].bad[k]) {
                if (bad[k] == 0)
                    first_bad[k] = jobs[i].first_bad[k];
                bad[k] += jobs[i].bad[k];
            }
    /* [7] decode -> encode identity on the 254 finite codes */
    for (int c = 0; c < 256; ++c) {
        if ((c & 0x7f) == 0x7f)
            continue;
        if (oracle_e4m3_from_f32((float)g_val[c]) != c) {
            if (bad[7]++ == 0)
                first_bad[7] = (uint32_t)c;
        }
    }
}

/*
 * synth.c -- seeded, counter-addressable synthetic input generator.
 *
 * Holds no arithmetic of the attention method itself: it only draws numbers
 * and shapes their distributions (normal, unit-norm rows, -c*softplus,
 * sigmoid, scaled normal) and rounds them to the storage type.  Both the
 * test-side oracle and the CUDA library receive inputs made here.
 *
 * Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014), used as a counter-based generator:
 * draw(key, n) is the (n+1)-th output of a SplitMix64 sequence seeded with
 * `key`, so any element of any tensor can be produced on its own.  A normal
 * variate is made from two draws by the Box-Muller transform (Box and Muller,
 * 1958).  Values are computed in double, cast to float (round to nearest even)
 * and, for bf16 storage, rounded again to the upper 16 bits with
 * round-to-nearest-even on the float's bit pattern.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>
#include <unistd.h>

#define SPLITMIX_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Key of an independent stream: (seed, stream id) -> 64-bit SplitMix64 seed. */
uint64_t synth_stream_key(uint64_t seed, uint64_t stream)
{
    return mix64(mix64(seed + SPLITMIX_GAMMA) ^ (stream * SPLITMIX_GAMMA + 0x632BE59BD9B4E019ULL));
}

static inline uint64_t draw(uint64_t key, uint64_t n) { return mix64(key + (n + 1) * SPLITMIX_GAMMA); }

/* Standard normal number n of the stream (Box-Muller, cosine branch). */
static inline double normal_at(uint64_t key, uint64_t n)
{
    const uint64_t x1 = draw(key, 2 * n), x2 = draw(key, 2 * n + 1);
    const double u1 = ((double)(x1 >> 11) + 1.0) * 0x1.0p-53; /* (0, 1] */
    const double u2 = (double)(x2 >> 11) * 0x1.0p-53;         /* [0, 1) */
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925 * u2);
}

static inline uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

enum { SYNTH_NORMAL = 0, SYNTH_UNIT_ROWS = 1, SYNTH_NEG_SOFTPLUS = 2, SYNTH_SIGMOID = 3 };

typedef struct {
    int kind;
    uint64_t key;
    int64_t row0, row_step, nrows, D;
    double scale;
    float *out_f32;
    uint16_t *out_bf16;
    int64_t m_begin, m_end;
} rows_job;

static void rows_range(const rows_job *J)
{
    double tmp[4096];
    for (int64_t m = J->m_begin; m < J->m_end; ++m) {
        const uint64_t base = (uint64_t)((J->row0 + m * J->row_step) * J->D);
        double ss = 0.0;
        for (int64_t i = 0; i < J->D; ++i) {
            const double z = normal_at(J->key, base + (uint64_t)i);
            double x;
            switch (J->kind) {
            case SYNTH_UNIT_ROWS: x = z; ss += z * z; break;
            case SYNTH_NEG_SOFTPLUS: /* -scale * log(1 + e^z), evaluated without overflow */
                x = -J->scale * (z > 0 ? z + log1p(exp(-z)) : log1p(exp(z)));
                break;
            case SYNTH_SIGMOID: x = 1.0 / (1.0 + exp(-z)); break;
            default: x = J->scale * z; break;
            }
            tmp[i] = x;
        }
        if (J->kind == SYNTH_UNIT_ROWS) {
            const double inv = 1.0 / sqrt(ss);
            for (int64_t i = 0; i < J->D; ++i) tmp[i] *= inv;
        }
        for (int64_t i = 0; i < J->D; ++i) {
            const float f = (float)tmp[i];
            if (J->out_f32) J->out_f32[m * J->D + i] = f;
            if (J->out_bf16) J->out_bf16[m * J->D + i] = f32_to_bf16_rne(f);
        }
    }
}

static void *rows_worker(void *arg)
{
    rows_range((const rows_job *)arg);
    return NULL;
}

/*
 * Fill nrows rows of D values.  Output row m is logical row r = row0 + m*row_step
 * of the tensor, whose element i is stream element r*D + i.  Either output may be
 * NULL.  Returns 0, or -1 for D outside [1, 4096].
 */
int synth_rows(int kind, uint64_t key, int64_t row0, int64_t row_step, int64_t nrows, int64_t D,
               double scale, float *out_f32, uint16_t *out_bf16, int nthreads)
{
    if (D < 1 || D > 4096 || nrows < 0) return -1;
    if (nthreads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = c > 0 ? (int)c : 1;
    }
    if (nthreads > 64) nthreads = 64;
    if (nrows * D < (1 << 16)) nthreads = 1;
    rows_job jobs[64];
    pthread_t tid[64];
    int joined[64];
    for (int t = 0; t < nthreads; ++t) {
        rows_job *J = &jobs[t];
        J->kind = kind; J->key = key; J->row0 = row0; J->row_step = row_step; J->nrows = nrows;
        J->D = D; J->scale = scale; J->out_f32 = out_f32; J->out_bf16 = out_bf16;
        J->m_begin = nrows * t / nthreads;
        J->m_end = nrows * (t + 1) / nthreads;
        joined[t] = 0;
        if (nthreads == 1 || pthread_create(&tid[t], NULL, rows_worker, J) != 0)
            rows_range(J); /* no thread: do this share inline */
        else
            joined[t] = 1;
    }
    for (int t = 0; t < nthreads; ++t)
        if (joined[t]) pthread_join(tid[t], NULL);
    return 0;
}

/* n uniform integers in [lo, hi] (inclusive) from draws 0..n-1 of the stream. */
void synth_uniform_ints(uint64_t key, int64_t n, int64_t lo, int64_t hi, int64_t *out)
{
    const uint64_t span = (uint64_t)(hi - lo) + 1u;
    for (int64_t m = 0; m < n; ++m)
        out[m] = lo + (int64_t)(draw(key, (uint64_t)m) % span);
}

/* Host side of the seeded synthetic-input generator (see synth_core.h).
 * Bulk fills are split over pthreads by index range; every element depends
 * only on (key, index), so the thread count never changes the bytes. */
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include "synth_core.h"

typedef struct {
  int kind;
  void* out;
  uint64_t begin, end;   /* element or block range of this thread */
  uint64_t key;
  double a, b;           /* std / lo,hi / dlo,dhi */
  uint64_t cols;         /* row length for per-row scales */
  const double* row_scale;
  uint64_t block0;       /* counter offset of the first block */
} job_t;

enum { K_NORMAL_BF16 = 0, K_UNIFORM_F32 = 1, K_Q2K = 2, K_Q3K = 3 };

static void* run_job(void* p) {
  job_t* j = (job_t*)p;
  for (uint64_t i = j->begin; i < j->end; ++i) {
    switch (j->kind) {
      case K_NORMAL_BF16: {
        double s = j->a;
        if (j->row_scale) s *= j->row_scale[i / j->cols];
        ((uint16_t*)j->out)[i] = syn_f64_to_bf16(syn_normal(j->key, i) * s);
        break;
      }
      case K_UNIFORM_F32:
        ((float*)j->out)[i] = (float)syn_affine(j->a, j->b, syn_unit(syn_draw(j->key, i)));
        break;
      case K_Q2K:
        syn_q2k_block((uint8_t*)j->out + i * 84ULL, j->key, j->block0 + i, j->a, j->b);
        break;
      case K_Q3K:
        syn_q3k_block((uint8_t*)j->out + i * 110ULL, j->key, j->block0 + i, j->a, j->b);
        break;
    }
  }
  return NULL;
}

static void run_parallel(job_t base, uint64_t n, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((uint64_t)nthreads > n) nthreads = n ? (int)n : 1;
  pthread_t th[256];
  job_t jobs[256];
  uint64_t per = (n + (uint64_t)nthreads - 1) / (uint64_t)nthreads;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = base;
    jobs[t].begin = per * (uint64_t)t;
    jobs[t].end = jobs[t].begin + per > n ? n : jobs[t].begin + per;
    if (jobs[t].begin > n) jobs[t].begin = n;
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, run_job, &jobs[t]);
  run_job(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
}

uint64_t syn_stream_key(uint64_t seed, uint32_t layer, uint32_t tensor, uint32_t expert) {
  return syn_key(seed, layer, tensor, expert);
}

uint64_t syn_draw_u64(uint64_t key, uint64_t i) { return syn_draw(key, i); }

uint16_t syn_half_bits(double v) { return syn_f64_to_f16(v); }

/* bf16 of std * row_scale[row] * N(0,1); row_scale may be NULL */
void syn_fill_normal_bf16(uint16_t* out, uint64_t n, uint64_t cols, uint64_t key, double std_,
                          const double* row_scale, int nthreads) {
  job_t j;
  memset(&j, 0, sizeof j);
  j.kind = K_NORMAL_BF16; j.out = out; j.key = key; j.a = std_; j.cols = cols ? cols : 1;
  j.row_scale = row_scale;
  run_parallel(j, n, nthreads);
}

void syn_fill_uniform_f32(float* out, uint64_t n, uint64_t key, double lo, double hi, int nthreads) {
  job_t j;
  memset(&j, 0, sizeof j);
  j.kind = K_UNIFORM_F32; j.out = out; j.key = key; j.a = lo; j.b = hi;
  run_parallel(j, n, nthreads);
}

void syn_fill_q2k(uint8_t* out, uint64_t nblocks, uint64_t block0, uint64_t key, double dlo,
                  double dhi, int nthreads) {
  job_t j;
  memset(&j, 0, sizeof j);
  j.kind = K_Q2K; j.out = out; j.key = key; j.a = dlo; j.b = dhi; j.block0 = block0;
  run_parallel(j, nblocks, nthreads);
}

void syn_fill_q3k(uint8_t* out, uint64_t nblocks, uint64_t block0, uint64_t key, double dlo,
                  double dhi, int nthreads) {
  job_t j;
  memset(&j, 0, sizeof j);
  j.kind = K_Q3K; j.out = out; j.key = key; j.a = dlo; j.b = dhi; j.block0 = block0;
  run_parallel(j, nblocks, nthreads);
}

/* Fisher-Yates shuffle of 0..n-1: step i (from n-1 down to 1) swaps i with
 * j = floor(hi32(draw i) * (i+1) / 2^32). */
void syn_permutation(int32_t* out, int32_t n, uint64_t key) {
  for (int32_t i = 0; i < n; ++i) out[i] = i;
  for (int32_t i = n - 1; i >= 1; --i) {
    uint64_t r = syn_draw(key, (uint64_t)i) >> 32;
    int32_t j = (int32_t)((r * (uint64_t)(i + 1)) >> 32);
    int32_t t = out[i]; out[i] = out[j]; out[j] = t;
  }
}

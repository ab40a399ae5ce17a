/*
 * synth_host.c -- host filler for the seeded synthetic inputs.
 *
 * Fills elements [e0, e1) of a tensor described by a synth_spec into `out`
 * (out[i] holds element e0 + i), splitting the range over POSIX threads.
 * The per-element value is defined in synth_core.h and is bit-identical to
 * the device filler in synth_dev.cu.  Built with -ffp-contract=off so that
 * the multiply and the add of each element are separately rounded.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "synth_core.h"

typedef struct {
  const synth_spec* sp;
  void* out;
  int64_t e0, begin, end;
} synth_job;

static void* synth_worker(void* arg) {
  const synth_job* j = (const synth_job*)arg;
  const synth_spec* sp = j->sp;
  for (int64_t e = j->begin; e < j->end; ++e) {
    float v = synth_value(sp, (uint64_t)e);
    int64_t i = e - j->e0;
    if (sp->dtype == SYNTH_F32) {
      ((float*)j->out)[i] = v;
    } else if (sp->dtype == SYNTH_BF16) {
      ((uint16_t*)j->out)[i] = synth_f32_to_bf16(v);
    } else {
      ((uint16_t*)j->out)[i] = synth_f32_to_f16(v);
    }
  }
  return NULL;
}

/* Returns 0 on success, -1 on a bad argument. */
int synth_fill_host(int32_t dtype, void* out, int64_t e0, int64_t e1, int64_t d,
                    int64_t rows_per_head, int64_t S, const float* bias,
                    const int32_t* attempt, uint32_t seed, uint32_t tid, int32_t nthreads) {
  if (!out || e1 < e0 || d <= 0) return -1;
  if (dtype != SYNTH_F32 && dtype != SYNTH_BF16 && dtype != SYNTH_F16) return -1;
  if (bias && (rows_per_head <= 0 || S <= 0)) return -1;
  synth_spec sp;
  memset(&sp, 0, sizeof sp);
  sp.d = d;
  sp.rows_per_head = rows_per_head > 0 ? rows_per_head : 1;
  sp.S = S > 0 ? S : 1;
  sp.bias = bias;
  sp.attempt = attempt;
  sp.seed = seed;
  sp.tid = tid;
  sp.dtype = dtype;
  int64_t n = e1 - e0;
  if (nthreads < 1) nthreads = 1;
  if (n < (int64_t)nthreads * 65536) nthreads = (int32_t)(n / 65536) + 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  int joinable[256];
  synth_job jobs[256];
  int64_t per = (n + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    int64_t b = e0 + (int64_t)t * per;
    jobs[t].sp = &sp;
    jobs[t].out = out;
    jobs[t].e0 = e0;
    jobs[t].begin = b < e1 ? b : e1;
    jobs[t].end = b + per < e1 ? b + per : e1;
    joinable[t] = 0;
  }
  for (int t = 1; t < nthreads; ++t) {
    if (jobs[t].begin >= jobs[t].end) continue;
    if (pthread_create(&th[t], NULL, synth_worker, &jobs[t]) == 0)
      joinable[t] = 1;
    else
      synth_worker(&jobs[t]);
  }
  synth_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t)
    if (joinable[t]) pthread_join(th[t], NULL);
  return 0;
}

/* One raw Philox4x32-10 block, for known-answer tests of the generator. */
void synth_philox_block(const uint32_t* ctr, const uint32_t* key, uint32_t* out) {
  synth_philox4x32_10(ctr, key, out);
}

/* Single conversions, for tests of the rounding helpers. */
void synth_round_f32(const float* in, int64_t n, int32_t dtype, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i)
    out[i] = dtype == SYNTH_BF16 ? synth_f32_to_bf16(in[i]) : synth_f32_to_f16(in[i]);
}

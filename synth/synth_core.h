/*
 * synth_core.h -- seeded, counter-based synthetic input values.
 *
 * This header is the whole arithmetic of the input generator.  It is
 * compiled twice: by gcc into the host filler (synth_host.c) and by nvcc
 * into the device filler (synth_dev.cu).  Both use only integer operations
 * plus one IEEE fp32 multiply and one fp32 add per element, with FMA
 * contraction disabled, so the host and the device produce bit-identical
 * tensors.  Nothing here computes any step of the attention method: no
 * summaries, scores, selections or softmax.
 *
 * Value of element e of a tensor with (seed, tensor id, attempt):
 *   r[0..7] = the eight 16-bit halves of Philox4x32-10(counter = {e_lo, e_hi,
 *             0, 0}, key = {seed, tid | attempt << 8})
 *             (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
 *             as 1, 2, 3", SC'11 -- the Philox-4x32 bijection, 10 rounds)
 *   z       = (sum r - 262140) * (fl32(sqrt(1.5)) * 2^-16)
 *             i.e. an Irwin-Hall sum of eight uniforms (r_i + 1/2)/2^16,
 *             centred and scaled to unit variance: an approximately N(0,1)
 *             value in [-4.9, 4.9] that needs no transcendental function.
 *   v       = z + bias            (fp32, only where a bias table is given)
 *   stored  = v rounded once to the storage type (fp32, or bf16 / fp16 by
 *             round-to-nearest-even).
 */
#ifndef SYNTH_CORE_H
#define SYNTH_CORE_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYNTH_FN static __host__ __device__ __forceinline__
#else
#define SYNTH_FN static inline
#endif

enum { SYNTH_F32 = 0, SYNTH_BF16 = 1, SYNTH_F16 = 2 };

/* Philox-4x32 constants: the two round multipliers and the two Weyl key
 * increments given with the generator's definition. */
#define SYNTH_PHILOX_M0 0xD2511F53u
#define SYNTH_PHILOX_M1 0xCD9E8D57u
#define SYNTH_PHILOX_W0 0x9E3779B9u
#define SYNTH_PHILOX_W1 0xBB67AE85u

SYNTH_FN void synth_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                                  uint32_t out[4]) {
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += SYNTH_PHILOX_W0;
      k1 += SYNTH_PHILOX_W1;
    }
    uint64_t p0 = (uint64_t)SYNTH_PHILOX_M0 * (uint64_t)c0;
    uint64_t p1 = (uint64_t)SYNTH_PHILOX_M1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* fl32(sqrt(1.5)) * 2^-16, written as an exact hexadecimal float. */
#define SYNTH_SCALE_BITS 0x379cc471u

SYNTH_FN float synth_bits_to_f32(uint32_t u) {
  union { uint32_t u; float f; } c;
  c.u = u;
  return c.f;
}

SYNTH_FN uint32_t synth_f32_to_bits(float f) {
  union { uint32_t u; float f; } c;
  c.f = f;
  return c.u;
}

/* The unbiased fp32 base value of element e (before any bias). */
SYNTH_FN float synth_base_value(uint64_t e, uint32_t seed, uint32_t tid, uint32_t attempt) {
  uint32_t ctr[4] = {(uint32_t)e, (uint32_t)(e >> 32), 0u, 0u};
  uint32_t key[2] = {seed, (tid & 0xffu) | (attempt << 8)};
  uint32_t r[4];
  synth_philox4x32_10(ctr, key, r);
  int32_t s = 0;
  for (int i = 0; i < 4; ++i) s += (int32_t)(r[i] & 0xffffu) + (int32_t)(r[i] >> 16);
  float centred = (float)(s - 262140); /* |.| <= 262140 < 2^24: exact */
#if defined(__CUDA_ARCH__)
  return __fmul_rn(centred, synth_bits_to_f32(SYNTH_SCALE_BITS));
#else
  return centred * synth_bits_to_f32(SYNTH_SCALE_BITS);
#endif
}

SYNTH_FN float synth_add(float a, float b) {
#if defined(__CUDA_ARCH__)
  return __fadd_rn(a, b);
#else
  return a + b;
#endif
}

/* fp32 -> bf16, round to nearest even (finite inputs; NaN kept quiet). */
SYNTH_FN uint16_t synth_f32_to_bf16(float f) {
  uint32_t u = synth_f32_to_bits(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* fp32 -> IEEE binary16, round to nearest even, subnormals included. */
SYNTH_FN uint16_t synth_f32_to_f16(float f) {
  uint32_t x = synth_f32_to_bits(f);
  uint32_t sign = (x >> 16) & 0x8000u;
  uint32_t ax = x & 0x7fffffffu;
  if (ax > 0x7f800000u) return (uint16_t)(sign | 0x7e00u);    /* NaN */
  if (ax >= 0x47800000u) return (uint16_t)(sign | 0x7c00u);   /* >= 2^16: inf */
  if (ax < 0x38800000u) {                                     /* < 2^-14 */
    if (ax < 0x33000000u) return (uint16_t)sign;              /* <= 2^-25 */
    uint32_t e = ax >> 23;
    uint32_t m = (ax & 0x7fffffu) | 0x800000u;
    uint32_t s = 126u - e;                                    /* 14..24 */
    uint32_t q = m >> s;
    uint32_t rem = m & ((1u << s) - 1u);
    uint32_t half = 1u << (s - 1u);
    if (rem > half || (rem == half && (q & 1u))) q += 1u;
    return (uint16_t)(sign | q);
  }
  uint32_t e = ax >> 23;
  uint32_t m23 = ax & 0x7fffffu;
  uint32_t h = ((e - 112u) << 10) | (m23 >> 13);
  uint32_t rem = m23 & 0x1fffu;
  if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;
  return (uint16_t)(sign | h);
}

/*
 * Layout of a fill: a tensor whose rows have `d` elements.  The optional
 * per-row attempt array redraws single rows; the optional bias table adds
 * bias[(head * nb + (t / S)) * d + c] where row = head * rows_per_head + t,
 * nb = ceil(rows_per_head / S).
 */
typedef struct {
  int64_t d;              /* elements per row */
  int64_t rows_per_head;  /* rows per head, for the bias lookup */
  int64_t S;              /* rows per bias block (span length) */
  const float* bias;      /* nullable */
  const int32_t* attempt; /* nullable, indexed by global row */
  uint32_t seed;
  uint32_t tid;
  int32_t dtype;          /* SYNTH_F32 / SYNTH_BF16 / SYNTH_F16 */
} synth_spec;

SYNTH_FN float synth_value(const synth_spec* sp, uint64_t e) {
  uint64_t row = e / (uint64_t)sp->d;
  uint64_t c = e - row * (uint64_t)sp->d;
  uint32_t attempt = sp->attempt ? (uint32_t)sp->attempt[row] : 0u;
  float v = synth_base_value(e, sp->seed, sp->tid, attempt);
  if (sp->bias) {
    uint64_t head = row / (uint64_t)sp->rows_per_head;
    uint64_t t = row - head * (uint64_t)sp->rows_per_head;
    uint64_t nb = ((uint64_t)sp->rows_per_head + (uint64_t)sp->S - 1) / (uint64_t)sp->S;
    uint64_t bi = (head * nb + t / (uint64_t)sp->S) * (uint64_t)sp->d + c;
    v = synth_add(v, sp->bias[bi]);
  }
  return v;
}

#endif /* SYNTH_CORE_H */

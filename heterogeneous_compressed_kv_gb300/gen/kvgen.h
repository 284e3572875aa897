/*
 * kvgen.h -- seeded, counter-based synthetic input generator.
 *
 * This module produces the synthetic K / V / indexer-key / query tensors,
 * gate logits and request lengths that drive both the CUDA path and the
 * CPU oracle.  It holds none of the KV-cache method's arithmetic: it only
 * turns (seed, stream, index) into a number, identically on host and device,
 * so that a 64 GiB workload can be generated on the GPU and any sampled
 * element regenerated on the CPU without copying it.
 *
 * Definition (all integer arithmetic is modulo 2^64):
 *   mix64(z)        : the splitmix64 output mixer (Steele, Lea, Flood,
 *                     "Fast splittable pseudorandom number generators",
 *                     OOPSLA 2014; constants as published with Java 8's
 *                     SplittableRandom / Vigna's splitmix64.c):
 *                       z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
 *                       z = (z ^ (z >> 27)) * 0x94D049BB133111EB
 *                       z =  z ^ (z >> 31)
 *   base(seed, s)   = mix64(seed ^ mix64(s + G)),  G = 0x9E3779B97F4A7C15
 *   u64(base, i)    = mix64(base + (i + 1) * G)   -- the i-th splitmix64
 *                     output of a generator whose state starts at `base`
 *   normal(base, i) = ((c0 + c1 + c2 + c3) * 2^-16 - 2) * fl(sqrt(3))
 *                     where c_k are the four 16-bit chunks of u64(base, i):
 *                     an Irwin-Hall(4) stand-in for N(0,1) (mean 0, variance
 *                     1, support +-2*sqrt(3)).  Every step is exact in fp32
 *                     except the final IEEE multiply, so host and device
 *                     produce the same bits.
 *   bf16 inputs     : normal() rounded to nearest-even bfloat16.
 *
 * Stream ids name a tensor: kind << 56 | layer << 40 | request.
 */
#ifndef KVGEN_H
#define KVGEN_H

#include <stdint.h>
#include <string.h>

#ifdef __CUDACC__
#define KVGEN_HD __host__ __device__ __forceinline__
#else
#define KVGEN_HD static inline
#endif

#define KVGEN_GOLDEN 0x9E3779B97F4A7C15ULL
#define KVGEN_SQRT3F 0x1.bb67aep+0f /* fl(sqrt(3)) = 0x3FDDB3D7 */

/* tensor kinds used in stream ids */
enum {
  KVGEN_K = 1,        /* new-token keys      [layer][request][pos][H][d]      */
  KVGEN_V = 2,        /* new-token values    [layer][request][pos][H][d]      */
  KVGEN_IDXK = 3,     /* new-token indexer keys [layer][request][pos][Ih][Id] */
  KVGEN_Q = 4,        /* decode queries      [layer][request][step][H][d]     */
  KVGEN_QIDX = 5,     /* indexer queries     [layer][request][step][Ih][Id]   */
  KVGEN_GATE_CSA = 6, /* gate logits         [layer][H][m]                    */
  KVGEN_GATE_HCA = 7, /* gate logits         [layer][H][m']                   */
  KVGEN_GATE_IDX = 8, /* gate logits         [layer][Ih][m]                   */
  KVGEN_LEN = 9,      /* request lengths / churn draws                        */
};

/* output formats: float; uint16 bfloat16 bits; (host only) float holding the
 * bfloat16-rounded value */
enum { KVGEN_OUT_F32 = 0, KVGEN_OUT_BF16 = 1, KVGEN_OUT_BF16_F32 = 2 };

KVGEN_HD uint64_t kvgen_stream_id(uint64_t kind, uint64_t layer, uint64_t request) {
  return (kind << 56) | ((layer & 0xFFFFull) << 40) | (request & 0xFFFFFFFFFFull);
}

KVGEN_HD uint64_t kvgen_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

KVGEN_HD uint64_t kvgen_base(uint64_t seed, uint64_t stream) {
  return kvgen_mix64(seed ^ kvgen_mix64(stream + KVGEN_GOLDEN));
}

KVGEN_HD uint64_t kvgen_u64(uint64_t base, uint64_t i) {
  return kvgen_mix64(base + (i + 1ull) * KVGEN_GOLDEN);
}

KVGEN_HD float kvgen_normal(uint64_t base, uint64_t i) {
  uint64_t u = kvgen_u64(base, i);
  uint32_t s = (uint32_t)(u & 0xFFFFu) + (uint32_t)((u >> 16) & 0xFFFFu) +
               (uint32_t)((u >> 32) & 0xFFFFu) + (uint32_t)(u >> 48);
  float c = (float)s * 0x1p-16f - 2.0f; /* exact: a multiple of 2^-16 in [-2, 2) */
#ifdef __CUDA_ARCH__
  return __fmul_rn(c, KVGEN_SQRT3F);
#else
  return c * KVGEN_SQRT3F;
#endif
}

/* round-to-nearest-even fp32 -> bfloat16 bits (inputs are finite) */
KVGEN_HD uint16_t kvgen_bf16_bits(float x) {
  uint32_t u;
#ifdef __CUDA_ARCH__
  u = __float_as_uint(x);
#else
  memcpy(&u, &x, 4);
#endif
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* One contiguous run of generated values: values index0 .. index0+count-1
 * of stream `stream`, written to out + out_offset elements. */
typedef struct kvgen_run {
  uint64_t stream;
  int64_t index0;
  int64_t count;
  int64_t out_offset;
} kvgen_run;

#ifdef __cplusplus
extern "C" {
#endif

/* Fill a host buffer.  out_dtype: KVGEN_OUT_F32 (float), KVGEN_OUT_BF16
 * (uint16 bfloat16 bits) or KVGEN_OUT_BF16_F32 (float holding the bfloat16
 * value).  Returns 0, or -1 on a bad argument. */
int kvgen_fill_host(void* out, int out_dtype, uint64_t seed, int n_runs, const kvgen_run* runs);

/* Fill a device buffer on `stream` (a cudaStream_t, NULL = legacy default).
 * `runs` is a host array; it is copied into kernel parameters, so it may be
 * reused as soon as the call returns.  Returns 0, -1 on a bad argument,
 * -6 on a CUDA launch error. */
int kvgen_fill_device(void* out, int out_dtype, uint64_t seed, int n_runs, const kvgen_run* runs,
                      void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVGEN_H */

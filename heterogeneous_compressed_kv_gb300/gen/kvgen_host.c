/* kvgen_host.c -- host side of the seeded input generator (see kvgen.h). */
#include "kvgen.h"

int kvgen_fill_host(void* out, int out_dtype, uint64_t seed, int n_runs, const kvgen_run* runs) {
  if (!out || n_runs < 0 || (n_runs > 0 && !runs)) return -1;
  if (out_dtype != KVGEN_OUT_F32 && out_dtype != KVGEN_OUT_BF16 && out_dtype != KVGEN_OUT_BF16_F32) return -1;
  for (int r = 0; r < n_runs; ++r) {
    const kvgen_run* run = &runs[r];
    if (run->count < 0 || run->index0 < 0 || run->out_offset < 0) return -1;
    uint64_t base = kvgen_base(seed, run->stream);
    if (out_dtype == KVGEN_OUT_F32) {
      float* o = (float*)out + run->out_offset;
      for (int64_t i = 0; i < run->count; ++i) o[i] = kvgen_normal(base, (uint64_t)(run->index0 + i));
    } else if (out_dtype == KVGEN_OUT_BF16) {
      uint16_t* o = (uint16_t*)out + run->out_offset;
      for (int64_t i = 0; i < run->count; ++i)
        o[i] = kvgen_bf16_bits(kvgen_normal(base, (uint64_t)(run->index0 + i)));
    } else {
      uint32_t* o = (uint32_t*)out + run->out_offset;
      for (int64_t i = 0; i < run->count; ++i)
        o[i] = (uint32_t)kvgen_bf16_bits(kvgen_normal(base, (uint64_t)(run->index0 + i))) << 16;
    }
  }
  return 0;
}

/* Raw 64-bit draws (lengths, churn choices). */
int kvgen_u64_host(uint64_t* out, uint64_t seed, uint64_t stream, int64_t index0, int64_t count) {
  if (!out || index0 < 0 || count < 0) return -1;
  uint64_t base = kvgen_base(seed, stream);
  for (int64_t i = 0; i < count; ++i) out[i] = kvgen_u64(base, (uint64_t)(index0 + i));
  return 0;
}

/* kvgen_device.cu -- device side of the seeded input generator (see kvgen.h).
 * Bit-identical to kvgen_fill_host: the same integer mixer, exact fp32 steps
 * and one IEEE multiply (__fmul_rn), then round-to-nearest-even bf16. */
#include <cuda_runtime.h>
#include "kvgen.h"

namespace {

constexpr int kMaxRunsPerLaunch = 512;

struct FillParams {
  void* out;
  int out_dtype;
  int n_runs;
  uint64_t seed;
  kvgen_run runs[kMaxRunsPerLaunch];
};

__global__ void __launch_bounds__(256) kvgen_fill_kernel(const __grid_constant__ FillParams p) {
  const kvgen_run run = p.runs[blockIdx.y];
  const uint64_t base = kvgen_base(p.seed, run.stream);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  if (p.out_dtype == KVGEN_OUT_F32) {
    float* o = (float*)p.out + run.out_offset;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < run.count; i += stride)
      o[i] = kvgen_normal(base, (uint64_t)(run.index0 + i));
  } else {
    uint16_t* o = (uint16_t*)p.out + run.out_offset;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < run.count; i += stride)
      o[i] = kvgen_bf16_bits(kvgen_normal(base, (uint64_t)(run.index0 + i)));
  }
}

}  // namespace

extern "C" int kvgen_fill_device(void* out, int out_dtype, uint64_t seed, int n_runs, const kvgen_run* runs,
                                 void* stream) {
  if (!out || n_runs < 0 || (n_runs > 0 && !runs)) return -1;
  if (out_dtype != KVGEN_OUT_F32 && out_dtype != KVGEN_OUT_BF16) return -1;
  cudaStream_t s = (cudaStream_t)stream;
  for (int r0 = 0; r0 < n_runs; r0 += kMaxRunsPerLaunch) {
    FillParams p;
    p.out = out;
    p.out_dtype = out_dtype;
    p.seed = seed;
    p.n_runs = n_runs - r0 < kMaxRunsPerLaunch ? n_runs - r0 : kMaxRunsPerLaunch;
    int64_t maxc = 0;
    for (int r = 0; r < p.n_runs; ++r) {
      p.runs[r] = runs[r0 + r];
      if (p.runs[r].count < 0 || p.runs[r].index0 < 0 || p.runs[r].out_offset < 0) return -1;
      if (p.runs[r].count > maxc) maxc = p.runs[r].count;
    }
    if (maxc == 0) continue;
    int64_t bx = (maxc + 255) / 256;
    if (bx > 4096) bx = 4096;
    dim3 grid((unsigned)bx, (unsigned)p.n_runs);
    kvgen_fill_kernel<<<grid, 256, 0, s>>>(p);
    if (cudaGetLastError() != cudaSuccess) return -6;
  }
  return 0;
}

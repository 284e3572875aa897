// kvpool_image.cu -- block copies between the arena (block part planes,
// window rings) and page-locked host memory read or written over the host
// link: prefix images ("Ch 12 Inference framework: heterogeneous KV
// scheduling" s3: the compressed block cache restored by an async copy
// instead of a prefill; "V4 disk prefix cache": the window stored or not per
// SWA policy) and HiSparse offload / fetch of CSA entries ("V4 KV Layout"
// ESS / HiSparse table), with the moved blocks' table, location and activity
// writes.
#include "device_util.cuh"

namespace kvp {
namespace {

constexpr int kImageThreads = 256;
constexpr int kUnitsPerThread = kImagePieceBytes / 16 / kImageThreads;  // 4
static_assert(kUnitsPerThread * 16 * kImageThreads == kImagePieceBytes, "piece = whole units per thread");

// zero the bytes of a 16-byte unit from byte `from` on
__device__ __forceinline__ uint4 zero_tail(uint4 v, int from) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int lo = 4 * i;
    if (from <= lo) w[i] = 0u;
    else if (from < lo + 4) w[i] &= (1u << (8 * (from - lo))) - 1u;
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Each CTA copies pieces of kImagePieceBytes (grid-stride); a piece lies in
// one segment.  Every thread issues its loads of a piece before its stores,
// so a CTA keeps 16 KB in flight over the link.
__global__ void __launch_bounds__(kImageThreads) image_copy_kernel(const __grid_constant__ ImageParams P) {
  pdl_start();
  const PoolDesc& pd = P.pool;
  const int tid = threadIdx.x;
  // bookkeeping of the moved blocks: table row, locations, activity stamps
  int32_t* row = reinterpret_cast<int32_t*>(pd.arena + pd.table) + (int64_t)P.dst * pd.max_bpr;
  int32_t* loc = reinterpret_cast<int32_t*>(pd.arena + pd.csa_loc);
  uint32_t* stamp = reinterpret_cast<uint32_t*>(pd.arena + pd.last_used);
  for (int r = blockIdx.x; r < P.n_runs; r += gridDim.x) {
    const ImageRun u = P.runs[r];
    if (u.cnt < 0 || u.id0 < 0 || u.id0 + u.cnt > pd.max_blocks || (u.b0 >= 0 && u.b0 + u.cnt > pd.max_bpr)) {
      if (tid == 0) flag_error(pd, kErrBadBlock);
      continue;
    }
    for (int i = tid; i < u.cnt; i += blockDim.x) {
      if (u.b0 >= 0) row[u.b0 + i] = u.id0 + i;
      if (u.loc_dir != 0) loc[u.id0 + i] = u.loc0 + i * u.loc_dir;
      if (u.stamp) stamp[u.id0 + i] = P.epoch;
    }
  }
  for (int64_t piece = blockIdx.x; piece < P.n_pieces; piece += gridDim.x) {
    int lo = 0, hi = P.n_segs - 1;  // the segment holding this piece
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (P.piece_base[mid] <= piece) lo = mid;
      else hi = mid - 1;
    }
    const ImageSeg& S = P.segs[lo];
    const int64_t off0 = (piece - P.piece_base[lo]) * kImagePieceBytes;
    const int64_t n = min((int64_t)kImagePieceBytes, S.bytes - off0);
    const uint8_t* src = reinterpret_cast<const uint8_t*>(S.src) + off0;
    uint8_t* dst = reinterpret_cast<uint8_t*>(S.dst) + off0;
    uint4 v[kUnitsPerThread];
#pragma unroll
    for (int k = 0; k < kUnitsPerThread; ++k) {
      const int64_t u = (int64_t)(k * kImageThreads + tid) * 16;
      if (u < n) v[k] = S.src_host ? *reinterpret_cast<const uint4*>(src + u) : ld_stream16(src + u);
    }
#pragma unroll
    for (int k = 0; k < kUnitsPerThread; ++k) {
      const int64_t u = (int64_t)(k * kImageThreads + tid) * 16;
      if (u < n) {
        uint4 x = v[k];
        if (S.mask_row > 0) {
          const int r = (int)((off0 + u) % S.mask_row);
          if (r + 16 > S.mask_valid) x = zero_tail(x, S.mask_valid - r);
        }
        *reinterpret_cast<uint4*>(dst + u) = x;
      }
    }
  }
}

// One thread waits on a barrier that expects an arrival nothing makes: the
// bounded wait gives up after its limit and sets the wait flag.
__global__ void wait_selftest_kernel(const PoolDesc pd) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  mbar_fence_init();
  mbar_wait(&bar, 0, pd);
}

}  // namespace

int launch_wait_selftest(const PoolDesc& pd, void* stream) {
  wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(pd);
  return (int)cudaGetLastError();
}

int launch_image(const ImageParams& p, void* stream, int* n_kernels) {
  if (p.n_pieces <= 0 && p.n_runs <= 0) return 0;
  if (p.n_segs < 0 || p.n_segs > kMaxImageSegs || p.n_runs < 0 || p.n_runs > kMaxImageRuns ||
      (p.n_pieces > 0 && p.n_segs == 0))
    return (int)cudaErrorInvalidValue;
  const int64_t work = p.n_pieces > p.n_runs ? p.n_pieces : p.n_runs;
  const int64_t cap = (int64_t)kImageCtasPerSm * (p.n_sms > 0 ? p.n_sms : 1);  // at most 8 CTAs per SM
  const int ctas = (int)(work < cap ? work : cap);
  launch_kernel(true, image_copy_kernel, dim3(ctas), dim3(kImageThreads), 0, reinterpret_cast<cudaStream_t>(stream),
                p);
  *n_kernels += 1;
  return (int)cudaGetLastError();
}

}  // namespace kvp

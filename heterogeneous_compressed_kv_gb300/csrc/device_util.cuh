// device_util.cuh -- small device helpers for the kvpool kernels: number
// formats, bounded mbarrier waits, 1-D bulk (TMA) copies and L2 hints, loads.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "kvpool_internal.h"

namespace kvp {

// ---------------------------------------------------------------------------
// number formats
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// The short-float conversions below are the sm_100-family PTX instructions
// (round to nearest even, saturating to the largest finite value); the first
// operand of a packed conversion goes to the high half.

// two e4m3 codes (the low byte first) -> f16x2; exact
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(two));
  return h;
}

// e4m3 code pair -> exact fp32 values (every e4m3 value is exact in f16 and f32)
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t two) {
  const uint32_t h = e4m3x2_to_f16x2(two);
  return make_float2(__half2float(__ushort_as_half((uint16_t)(h & 0xFFFFu))),
                     __half2float(__ushort_as_half((uint16_t)(h >> 16))));
}

// two fp32 -> two e4m3 codes (a in the low byte), saturate to +-448
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(r) : "f"(a), "f"(b));
  return r;
}

// two fp32 -> two e2m1 codes in one byte (a in the low nibble), saturate to +-6
__device__ __forceinline__ uint8_t f32x2_to_e2m1x2(float a, float b) {
  uint16_t r;
  asm("{.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\tmov.b16 %0, {t, 0};}" : "=h"(r) : "f"(a), "f"(b));
  return (uint8_t)r;
}

// the four bytes of w (eight e2m1 codes, the low byte first) -> four f16x2
// words; the bytes are taken apart inside one asm block
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t* h) {
  asm("{.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// fp4 scale of a vector with absolute maximum amax: bf16(amax / 6), 1 if 0
__device__ __forceinline__ uint16_t fp4_scale_bits(float amax) {
  uint16_t s = f32_to_bf16_bits(__fdiv_rn(amax, 6.0f));
  return s == 0 ? (uint16_t)0x3F80 : s;
}

// fp8 scale of a vector with absolute maximum amax: bf16(amax / 448), 1 if 0
__device__ __forceinline__ uint16_t fp8_scale_bits(float amax) {
  uint16_t s = f32_to_bf16_bits(__fdiv_rn(amax, 448.0f));
  return s == 0 ? (uint16_t)0x3F80 : s;
}

// orderable key of a score: larger score -> larger key; -0 folds to +0
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: every kernel of this library starts with
// pdl_start(), which lets the next kernel in the stream be scheduled (it
// still waits for this grid to finish before touching memory) and waits for
// the previous kernel in the stream to finish and flush.  Every CTA calls it
// before any early exit, so a grid never completes before its predecessor.
// Without the launch attribute both instructions are no-ops.  The attribute
// is set where an early start hides launch latency on the critical path
// (append, indexer scores, the one-CTA select, the [selected CSA] attention
// part, merge); the two-pass select and the [HCA | window] part launch
// without it: their early-started CTAs held SM resources that the work
// beside them needed (measured slower).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_start() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// request of a CTA: requests are ordered by their first CTA index (score
// CTAs: which 0, select CTAs: which 1); the last request whose base <= cta
// ---------------------------------------------------------------------------
__device__ __forceinline__ int find_req(const AttendParams& P, int cta, int which) {
  int lo = 0, hi = P.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    const int base = which == 0 ? P.reqs[mid].score_base : P.reqs[mid].key_base;
    if (base <= cta) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// ---------------------------------------------------------------------------
// error word
// ---------------------------------------------------------------------------
__device__ __forceinline__ void flag_error(const PoolDesc& p, uint32_t f) {
  atomicOr(reinterpret_cast<uint32_t*>(p.arena + p.err), f);
}

// ---------------------------------------------------------------------------
// mbarrier + bulk copy (sm_90+ PTX), with time-limited waits
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// order this thread's (and, after a warp/CTA barrier, its peers') generic
// shared-memory accesses before later async-proxy (bulk copy) accesses
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

// Wait for the phase with the given parity to complete; false (and the error
// flag set) if it has not completed within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const PoolDesc& p) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) {
      flag_error(p, kErrWaitTimeout);
      return false;
    }
  }
}

// L2 policy for data read once (a stream through the cache): its lines are
// the first evicted, so it does not push out what later kernels read again
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D bulk copy global -> shared of data read once (evict-first in L2)
__device__ __forceinline__ void bulk_g2s_stream(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

// ---------------------------------------------------------------------------
// streaming loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ld_nc16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

}  // namespace kvp

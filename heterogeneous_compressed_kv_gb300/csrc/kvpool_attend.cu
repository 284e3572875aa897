// kvpool_attend.cu -- split-K decode attention over the three sources and the
// split merge ("Why does V4 split pools? ..." s4: attention reads compressed
// Classical entries sparsely (CSA top-k) and densely (HCA) plus the exact
// local State window; one softmax over all of them).
//
// A request's sources are one virtual list [selected CSA entries | HCA
// entries | window tokens]; every source is one contiguous entry of
// entry_bytes ([K | V] codes, fp8 scales), so a 1-D bulk copy (TMA) moves it
// into shared memory wherever it lives (a shared block, the request's
// staging block or its window ring); entries that follow each other in
// memory move in one copy.  A CTA takes one split of the list: its producer
// warp streams the split's entries through a ring of stages guarded by
// mbarriers (lane e copies entry e of a stage); consumer threads (16 dims of
// one head each) run an online softmax in the log2 domain and write a
// partial (max, sum, output) per head.  Scores: with an fp8 cache and a bf16
// query, tensor-core MMAs on the e4m3 codes (the query split into two exact
// e4m3 pieces); otherwise mixed-precision FMAs (f16 or bf16 products, exact
// in fp32) when the query is exactly representable, plain fp32 FMAs if not.
// fp8 values are weighted by p * scale rounded to f16.  A merge kernel
// combines the partials.  All waits are time-limited.
#include <algorithm>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_util.cuh"
#include "kvpool_internal.h"

namespace kvp {
namespace {

constexpr int kStages = 4;
// the stages' full and empty barriers sit in front of the staged entries
constexpr int kBarBytes = 64;
static_assert(2 * kStages * (int)sizeof(uint64_t) <= kBarBytes, "the barriers must fit in front of the stages");
constexpr int kMaxSplitLen = 1024;
constexpr int kUnroll = 4;  // entries per online-softmax update

__device__ __forceinline__ int find_split_req(const AttendParams& P, int cta, int part) {
  int lo = 0, hi = P.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((part ? P.reqs[mid].cta_base1 : P.reqs[mid].cta_base0) <= cta) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Device address of virtual source v of request R: an entry in the arena,
// or (HiSparse) an offloaded CSA entry in its host slot, through the host
// pool's device alias.  Reading a sealed block's CSA entry stamps the block
// with this call's epoch (HiSparse activity).
template <bool HS>
__device__ __forceinline__ uint64_t source_addr(const AttendParams& P, int i, const AttendReq& R, int v) {
  const PoolDesc& pd = P.pool;
  const LayerDesc& L = P.layer;
  const int32_t* table = reinterpret_cast<const int32_t*>(pd.arena + pd.table) + (int64_t)R.slot * pd.max_bpr;
  const uint64_t ring = reinterpret_cast<uint64_t>(pd.arena + L.ring + (int64_t)R.slot * L.ring_req_bytes);
  if (v < R.k) {
    const int32_t e = P.sel[(int64_t)i * P.sel_stride + v];
    if (e < 0 || e >= R.n_cand) {
      flag_error(pd, kErrBadIndex);
      return ring;
    }
    const int CB = pd.csa_per_block;
    const int seg = e / CB;
    const int64_t in_block = (int64_t)(e % CB) * pd.entry_bytes;
    if (seg >= R.n_sealed)  // the request's open block
      return reinterpret_cast<uint64_t>(pd.arena + L.csa_pool +
                                        (int64_t)(pd.csa_staging_base + R.slot) * L.csa_stride + in_block);
    const int32_t bid = table[seg];
    if (bid < 0 || bid >= pd.max_blocks) {
      flag_error(pd, kErrBadBlock);
      return ring;
    }
    int32_t loc = bid;
    if constexpr (HS) {
      loc = reinterpret_cast<const int32_t*>(pd.arena + pd.csa_loc)[bid];
      reinterpret_cast<uint32_t*>(pd.arena + pd.last_used)[bid] = P.epoch;
      if (loc < 0) {
        const int64_t h = -1 - (int64_t)loc;
        if (!pd.host_pool || (h + 1) * pd.host_slot_bytes > pd.host_pool_bytes) {
          flag_error(pd, kErrBadBlock);
          return ring;
        }
        return reinterpret_cast<uint64_t>(pd.host_pool + h * pd.host_slot_bytes + L.csa_host_off + in_block);
      }
      if (loc >= pd.csa_staging_base) {
        flag_error(pd, kErrBadBlock);
        return ring;
      }
    }
    return reinterpret_cast<uint64_t>(pd.arena + L.csa_pool + (int64_t)loc * L.csa_stride + in_block);
  }
  v -= R.k;
  if (v < R.n_hca) {
    const int32_t bid = table[v];
    if (bid < 0 || bid >= pd.max_blocks) {
      flag_error(pd, kErrBadBlock);
      return ring;
    }
    return reinterpret_cast<uint64_t>(pd.arena + L.hca_pool + (int64_t)bid * L.hca_stride);
  }
  v -= R.n_hca;
  const int64_t pos = R.length - R.w + v;
  return ring + (uint64_t)((pos % pd.n_win) * pd.entry_bytes);
}

// ---- shared-memory loads and number formats of the consumer loop ----------
// A bf16 consumer thread (TPH threads per head of TPH * 16 dims) owns dims
// [8r, 8r + 8) and [TPH * 8 + 8r, TPH * 8 + 8r + 8) of its head, r = its rank
// in the head: the second run starts TPH * 16 bytes after the first.  (16
// contiguous dims per thread put neighbouring threads 32 bytes apart: two
// shared-memory wavefronts per quarter-warp instead of one.)  Other caches
// keep 16 contiguous dims per thread.
template <int TPH>
constexpr int kRun2Bytes = TPH * 16;
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
// four e4m3 codes -> two f16x2 words (exact)
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}
// c0 += lo(a) * lo(b), c1 += hi(a) * hi(b): f16 (or bf16) operands, products
// exact in fp32, fp32 accumulation
__device__ __forceinline__ void fma_f16x2(uint32_t a, uint32_t b, float& c0, float& c1) {
  asm("{.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\tfma.rn.f32.f16 %1, ah, bh, %1;}"
      : "+f"(c0), "+f"(c1)
      : "r"(a), "r"(b));
}
__device__ __forceinline__ void fma_bf16x2(uint32_t a, uint32_t b, float& c0, float& c1) {
  asm("{.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %0;\n\tfma.rn.f32.bf16 %1, ah, bh, %1;}"
      : "+f"(c0), "+f"(c1)
      : "r"(a), "r"(b));
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float f16lo_to_f32(uint32_t w) { return __half2float(__ushort_as_half((uint16_t)(w & 0xFFFFu))); }
__device__ __forceinline__ float f16hi_to_f32(uint32_t w) { return __half2float(__ushort_as_half((uint16_t)(w >> 16))); }

// Dot product of the query's 16 dims with 16 key values at shared address a.
// FAST: the query is exact in the mixed-precision operand type (f16 for an
// fp8 cache, bf16 for a bf16 cache) and qw holds it as pairs; otherwise qf.
// bf16: the thread's dims are two runs of 8, the second B2 bytes after the
// first (so that neighbouring threads read neighbouring 16-byte words).
template <int CACHE, bool FAST, int B2>
__device__ __forceinline__ float dot16(uint32_t a, const uint32_t* qw, const float* qf) {
  float c0 = 0.0f, c1 = 0.0f;
  if constexpr (CACHE == KVPOOL_FP8_E4M3) {
    const uint4 r = lds128(a);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t lo, hi;
      e4m3x4_to_f16x4(w[i], lo, hi);
      if constexpr (FAST) {
        fma_f16x2(lo, qw[2 * i], c0, c1);
        fma_f16x2(hi, qw[2 * i + 1], c0, c1);
      } else {
        c0 = fmaf(qf[4 * i], f16lo_to_f32(lo), c0);
        c1 = fmaf(qf[4 * i + 1], f16hi_to_f32(lo), c1);
        c0 = fmaf(qf[4 * i + 2], f16lo_to_f32(hi), c0);
        c1 = fmaf(qf[4 * i + 3], f16hi_to_f32(hi), c1);
      }
    }
  } else if constexpr (CACHE == KVPOOL_BF16) {
    const uint4 r0 = lds128(a), r1 = lds128(a + B2);
    const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if constexpr (FAST) {
        fma_bf16x2(w[i], qw[i], c0, c1);
      } else {
        c0 = fmaf(qf[2 * i], bf16_bits_to_f32(w[i] & 0xFFFFu), c0);
        c1 = fmaf(qf[2 * i + 1], __uint_as_float(w[i] & 0xFFFF0000u), c1);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 r = lds128(a + 16 * i);
      c0 = fmaf(qf[4 * i], __uint_as_float(r.x), c0);
      c1 = fmaf(qf[4 * i + 1], __uint_as_float(r.y), c1);
      c0 = fmaf(qf[4 * i + 2], __uint_as_float(r.z), c0);
      c1 = fmaf(qf[4 * i + 3], __uint_as_float(r.w), c1);
    }
  }
  return c0 + c1;
}

// o[0..16) += weight * (16 values at shared address a; bf16: two runs of 8,
// B2 bytes apart).  fp8: the weight is p times the entry's V scale rounded to
// f16, so its products with the f16 values are exact; bf16 / fp32: p in fp32.
template <int CACHE, int B2>
__device__ __forceinline__ void acc16(uint32_t a, float wgt, float* o) {
  if constexpr (CACHE == KVPOOL_FP8_E4M3) {
    const uint32_t h = __half_as_ushort(__float2half_rn(wgt));
    const uint32_t h2 = h | (h << 16);
    const uint4 r = lds128(a);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t lo, hi;
      e4m3x4_to_f16x4(w[i], lo, hi);
      fma_f16x2(lo, h2, o[4 * i], o[4 * i + 1]);
      fma_f16x2(hi, h2, o[4 * i + 2], o[4 * i + 3]);
    }
  } else if constexpr (CACHE == KVPOOL_BF16) {
    const uint4 r0 = lds128(a), r1 = lds128(a + B2);
    const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      o[2 * i] = fmaf(wgt, bf16_bits_to_f32(w[i] & 0xFFFFu), o[2 * i]);
      o[2 * i + 1] = fmaf(wgt, __uint_as_float(w[i] & 0xFFFF0000u), o[2 * i + 1]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 r = lds128(a + 16 * i);
      o[4 * i] = fmaf(wgt, __uint_as_float(r.x), o[4 * i]);
      o[4 * i + 1] = fmaf(wgt, __uint_as_float(r.y), o[4 * i + 1]);
      o[4 * i + 2] = fmaf(wgt, __uint_as_float(r.z), o[4 * i + 2]);
      o[4 * i + 3] = fmaf(wgt, __uint_as_float(r.w), o[4 * i + 3]);
    }
  }
}

// Online-softmax update over NU entries starting at shared address a0
// (entries ES bytes apart): scores in the log2 domain, then the weighted V.
template <int CACHE, bool FAST, int TPH, int NU>
__device__ __forceinline__ void update(uint32_t a0, uint32_t ES, uint32_t koff, uint32_t voff, uint32_t soff,
                                       float qscale, const uint32_t* qw, const float* qf, float& m_run,
                                       float& l_run, float* o) {
  float sc[NU], vsc[NU];
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    const uint32_t a = a0 + u * ES;
    float d = dot16<CACHE, FAST, kRun2Bytes<TPH>>(a + koff, qw, qf);
#pragma unroll
    for (int off = TPH / 2; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    if constexpr (CACHE == KVPOOL_FP8_E4M3) {
      const uint32_t s2 = lds32(a + soff);  // K scale (low half), V scale (high half)
      sc[u] = d * (qscale * bf16_bits_to_f32(s2 & 0xFFFFu));
      vsc[u] = __uint_as_float(s2 & 0xFFFF0000u);
    } else {
      sc[u] = d * qscale;
      vsc[u] = 1.0f;
    }
  }
  float mx = m_run;
#pragma unroll
  for (int u = 0; u < NU; ++u) mx = fmaxf(mx, sc[u]);
  const float corr = ex2(m_run - mx);
  l_run *= corr;
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j] *= corr;
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    const float p = ex2(sc[u] - mx);
    l_run += p;
    acc16<CACHE, kRun2Bytes<TPH>>(a0 + u * ES + voff, p * vsc[u], o);
  }
  m_run = mx;
}

// ---- tensor-core scores: fp8 cache, bf16 query, head_dim 128 --------------
// q.k of 4 entries x 4 heads is one m16n8k32 e4m3 MMA per 32 dims: A rows are
// (head, entry) key rows straight from the staged entries, B columns are
// (head, piece) query pieces.  A head's bf16 query scaled by 2^s (largest
// magnitude in [128, 256)) is the exact sum of two e4m3 numbers per element
// (8 significant bits = 4 + 4) for elements down to 2^-2 after scaling;
// smaller ones keep their bits above 2^-10 (an error below 2^-17 of the
// head's largest element).  Products of e4m3 values are exact.

// Query pieces of this warp's 4 heads as the B fragments of the 4 MMAs of a
// 128-dim head (bq[4c + r]: chunk c of 64 dims), and the factor that undoes
// the scaling (times log2(e) / sqrt(d)).  Lane L holds the 16 query values
// of head L / 8, dims 16 (L % 8) ...; the MMA k index is permuted so that a
// lane's A bytes of one row are 16 contiguous dims.
__device__ __forceinline__ void q_pieces_fp8(const float* qf, int lane, float qscale, uint32_t* bq, float& fq) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(qf[j]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  int sh = amax > 0.0f ? 7 - ((int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127) : 0;
  sh = max(-126, min(126, sh));
  const float up = __uint_as_float((uint32_t)(127 + sh) << 23);
  fq = qscale * __uint_as_float((uint32_t)(127 - sh) << 23);
  uint32_t p0[4], p1[4];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float x0 = qf[2 * j] * up, x1 = qf[2 * j + 1] * up;
    const uint16_t c1 = f32x2_to_e4m3x2(x0, x1);
    const float2 v1 = e4m3x2_to_f32x2(c1);
    const uint16_t c2 = f32x2_to_e4m3x2(x0 - v1.x, x1 - v1.y);
    if (j & 1) {
      p0[j >> 1] |= (uint32_t)c1 << 16;
      p1[j >> 1] |= (uint32_t)c2 << 16;
    } else {
      p0[j >> 1] = c1;
      p1[j >> 1] = c2;
    }
  }
  // B lane (g, t), chunk c: piece g & 1 of head g >> 1, dims 64c + 16t + [0, 16)
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int src = 8 * (g >> 1) + 4 * c + t;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint32_t a = __shfl_sync(0xffffffffu, p0[r], src);
      const uint32_t b = __shfl_sync(0xffffffffu, p1[r], src);
      bq[4 * c + r] = (g & 1) ? b : a;
    }
  }
}

__device__ __forceinline__ void mma_e4m3(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Online-softmax update over NU (<= 4) entries starting at shared address a0:
// MMA scores (rows of entries past NU repeat the last one and are ignored),
// then the weighted V on CUDA cores.  arow: this lane's A row offset in an
// entry ((4 warp + g / 4) * 128 + 16 t).
template <int NU>
__device__ __forceinline__ void update_tc(uint32_t a0, uint32_t ES, uint32_t arow, uint32_t voff, uint32_t soff,
                                          int lane, const uint32_t* bq, float fq, float& m_run, float& l_run,
                                          float* o) {
  const uint32_t ra = a0 + (uint32_t)min((lane >> 2) & 3, NU - 1) * ES + arow;  // row g
  const uint32_t rb = ra + 256;                                                 // row g + 8: head + 2
  float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const uint4 lo = lds128(ra + 64 * c), hi = lds128(rb + 64 * c);
    mma_e4m3(d, lo.x, hi.x, lo.y, hi.y, bq[4 * c], bq[4 * c + 1]);
    mma_e4m3(d, lo.z, hi.z, lo.w, hi.w, bq[4 * c + 2], bq[4 * c + 3]);
  }
  // lane (g, t) holds head t, entry g & 3 when t & 1 == g / 4 (both pieces summed)
  const float u = (lane & 3) < 2 ? d[0] + d[1] : d[2] + d[3];
  const int hh = lane >> 3;  // this lane's head in the V phase
  float sc[NU], vsc[NU];
#pragma unroll
  for (int e = 0; e < NU; ++e) {
    const float dot = __shfl_sync(0xffffffffu, u, 16 * (hh & 1) + 4 * e + hh);
    const uint32_t s2 = lds32(a0 + e * ES + soff);  // K scale (low half), V scale (high half)
    sc[e] = dot * (fq * bf16_bits_to_f32(s2 & 0xFFFFu));
    vsc[e] = __uint_as_float(s2 & 0xFFFF0000u);
  }
  float mx = m_run;
#pragma unroll
  for (int e = 0; e < NU; ++e) mx = fmaxf(mx, sc[e]);
  const float corr = ex2(m_run - mx);
  l_run *= corr;
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j] *= corr;
#pragma unroll
  for (int e = 0; e < NU; ++e) {
    const float p = ex2(sc[e] - mx);
    l_run += p;
    acc16<KVPOOL_FP8_E4M3, 0>(a0 + e * ES + voff, p * vsc[e], o);
  }
  m_run = mx;
}

__device__ __forceinline__ void consume_stage_tc(uint32_t base, int ne, uint32_t ES, uint32_t arow, uint32_t voff,
                                                 uint32_t soff, int lane, const uint32_t* bq, float fq, float& m_run,
                                                 float& l_run, float* o) {
  int e0 = 0;
  for (; e0 + 4 <= ne; e0 += 4) update_tc<4>(base + e0 * ES, ES, arow, voff, soff, lane, bq, fq, m_run, l_run, o);
  switch (ne - e0) {
    case 3: update_tc<3>(base + e0 * ES, ES, arow, voff, soff, lane, bq, fq, m_run, l_run, o); break;
    case 2: update_tc<2>(base + e0 * ES, ES, arow, voff, soff, lane, bq, fq, m_run, l_run, o); break;
    case 1: update_tc<1>(base + e0 * ES, ES, arow, voff, soff, lane, bq, fq, m_run, l_run, o); break;
    default: break;
  }
}

// Online-softmax updates over the ne entries of one stage, kUnroll at a time.
template <int CACHE, bool FAST, int TPH>
__device__ __forceinline__ void consume_stage(uint32_t base, int ne, uint32_t ES, uint32_t koff, uint32_t voff,
                                              uint32_t soff, float qscale, const uint32_t* qw, const float* qf,
                                              float& m_run, float& l_run, float* o) {
  int e0 = 0;
  for (; e0 + kUnroll <= ne; e0 += kUnroll)
    update<CACHE, FAST, TPH, kUnroll>(base + e0 * ES, ES, koff, voff, soff, qscale, qw, qf, m_run, l_run, o);
  switch (ne - e0) {
    case 3: update<CACHE, FAST, TPH, 3>(base + e0 * ES, ES, koff, voff, soff, qscale, qw, qf, m_run, l_run, o); break;
    case 2: update<CACHE, FAST, TPH, 2>(base + e0 * ES, ES, koff, voff, soff, qscale, qw, qf, m_run, l_run, o); break;
    case 1: update<CACHE, FAST, TPH, 1>(base + e0 * ES, ES, koff, voff, soff, qscale, qw, qf, m_run, l_run, o); break;
    default: break;
  }
}

// TPH: consumer threads per head (head_dim / 16); each owns 16 dims.  One
// CTA per split: a producer warp streams the split's entries through a ring
// of kStages stages (lane e copies entry e of a stage; entries that follow
// each other in memory go in one copy); the consumer threads run the online
// softmax and write the split's partial.
template <int IN, int CACHE, int TPH, bool HS>
__global__ void __launch_bounds__(kAttendThreadsMax, 2) attend_kernel(const __grid_constant__ AttendParams P,
                                                                      int e_stage, int part) {
  pdl_start();
  extern __shared__ __align__(128) uint8_t smem[];
  const PoolDesc& pd = P.pool;
  const int HD = pd.HD;
  const int n_act = HD / 16;                  // consumer threads with work
  const int n_cons = (n_act + 31) / 32 * 32;  // whole consumer warps
  const int tid = threadIdx.x;
  const uint32_t ES = (uint32_t)pd.entry_bytes;
  const uint32_t stage_bytes = (uint32_t)e_stage * ES;
  const int i = find_split_req(P, blockIdx.x, part);
  const AttendReq& R = P.reqs[i];
  const int split = blockIdx.x - (part ? R.cta_base1 : R.cta_base0);
  // part 0 covers virtual sources [k, k + n_hca + w), part 1 covers [0, k)
  const int lo = part ? 0 : R.k, hi = part ? R.k : R.k + R.n_hca + R.w;
  const int len = part ? R.split_len1 : R.split_len0;
  const int v0 = lo + split * len;
  const int cnt = min(hi, v0 + len) - v0;
  const int n_st = (cnt + e_stage - 1) / e_stage;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kStages;
  uint8_t* stage_mem = smem + kBarBytes;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], n_cons / 32);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (tid >= n_cons) {
    // ---- producer warp: source addresses 32 at a time, one batch ahead ----
    const int lane = tid & 31;
    const uint64_t hbase = reinterpret_cast<uint64_t>(pd.host_pool), hbytes = (uint64_t)pd.host_pool_bytes;
    const uint64_t l2pol = l2_evict_first_policy();
    uint64_t cur = lane < cnt ? source_addr<HS>(P, i, R, v0 + lane) : 0;
    uint64_t nxt = 32 + lane < cnt ? source_addr<HS>(P, i, R, v0 + 32 + lane) : 0;
    int batch = 0;
    bool ok = true;
    int issued = 0;
    for (int st = 0; st < n_st; ++st) {
      const int s = st % kStages;
      if (lane == 0 && st >= kStages && !mbar_wait(&empty[s], ((st / kStages) - 1) & 1, pd)) ok = false;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const int e0 = st * e_stage;
      const int ne = min(e_stage, cnt - e0);
      if constexpr (!HS) {
        if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)ne * ES);
        __syncwarp();
      }
      const int x = e0 + lane;
      const uint64_t ac = __shfl_sync(0xffffffffu, cur, x & 31);
      const uint64_t an = __shfl_sync(0xffffffffu, nxt, x & 31);
      const uint64_t a = (x >> 5) == batch ? ac : an;
      // offloaded entries (HiSparse): the warp loads them from host memory
      // into the stage before the stage's arrival releases it
      const bool hst = HS && lane < ne && a - hbase < hbytes;
      const uint32_t hmask = HS ? __ballot_sync(0xffffffffu, hst) : 0u;
      if (HS && hmask) {
        constexpr int kLd = 8;
        const int units = (int)(ES / 16);
        for (uint32_t mk = hmask; mk; mk &= mk - 1) {
          const int j = __ffs(mk) - 1;
          const uint4* src = reinterpret_cast<const uint4*>(__shfl_sync(0xffffffffu, a, j));
          uint4* dst = reinterpret_cast<uint4*>(stage_mem + (size_t)s * stage_bytes + (size_t)j * ES);
          for (int u0 = 0; u0 < units; u0 += 32 * kLd) {
            uint4 t[kLd];
#pragma unroll
            for (int k = 0; k < kLd; ++k) {
              const int u = u0 + k * 32 + lane;
              if (u < units) t[k] = src[u];
            }
#pragma unroll
            for (int k = 0; k < kLd; ++k) {
              const int u = u0 + k * 32 + lane;
              if (u < units) dst[u] = t[k];
            }
          }
        }
        fence_proxy_async();  // before later bulk copies into this stage
        __syncwarp();
      }
      if constexpr (HS) {
        if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(ne - __popc(hmask)) * ES);
        __syncwarp();
      }
      // lane e starts a copy unless entry e - 1 ends right where entry e begins
      const uint64_t prev = __shfl_up_sync(0xffffffffu, a, 1);
      const bool prev_host = lane > 0 && ((hmask >> (lane - 1)) & 1u);
      const bool start = lane < ne && !hst && (lane == 0 || prev_host || a != prev + (uint64_t)ES);
      const uint32_t starts = __ballot_sync(0xffffffffu, start);
      if (start) {
        const uint32_t later = (starts | hmask) & ~((2u << lane) - 1u);
        const int end = later ? __ffs(later) - 1 : ne;
        bulk_g2s_stream(stage_mem + (size_t)s * stage_bytes + (size_t)lane * ES, reinterpret_cast<const void*>(a),
                        (uint32_t)(end - lane) * ES, &full[s], l2pol);
      }
      if (((e0 + ne) >> 5) != batch) {  // the next stage starts in the next batch
        ++batch;
        cur = nxt;
        const int y = (batch + 1) * 32 + lane;
        nxt = y < cnt ? source_addr<HS>(P, i, R, v0 + y) : 0;
      }
      issued = st + 1;
    }
    // on every exit path, wait (time-limited) for this CTA's copies still in
    // flight, so the CTA never ends while bulk copies land in its shared
    // memory: a consumer whose wait ran out may already have left
    if (lane == 0)
      for (int t = max(0, issued - kStages); t < issued; ++t) mbar_wait(&full[t % kStages], (t / kStages) & 1, pd);
    return;
  }

  // ---- consumers: head h, dims [dA, dA + 8) and [dB, dB + 8) ----
  // (bf16: two runs TPH * 8 dims apart; otherwise dB = dA + 8)
  constexpr bool kRuns = CACHE == KVPOOL_BF16;
  const int lane = tid & 31;
  const bool act = tid < n_act;
  const int h = act ? tid / TPH : 0;
  const int rk = act ? tid % TPH : 0;
  const int dA = kRuns ? 8 * rk : 16 * rk;
  const int dB = kRuns ? TPH * 8 + 8 * rk : dA + 8;
  // scores in the log2 domain: dot(q, k) * log2(e) / sqrt(d) (* fp8 K scale)
  const float qscale = 1.4426950408889634f * rsqrtf((float)pd.head_dim);
  const uint32_t koff = (uint32_t)((h * pd.head_dim + dA) * pd.vs);
  const uint32_t voff = (uint32_t)(HD * pd.vs) + koff;
  const uint32_t soff = (uint32_t)(2 * HD * pd.vs);
  const uint32_t stage0 = smem_addr(stage_mem);
  // the thread's 16 query values; the mixed-precision path needs them exact in
  // its operand type (decided per warp: every lane or none)
  float qf[16];
  uint32_t qw[8];
  int exact = 1;
  const uint8_t* qrow = reinterpret_cast<const uint8_t*>(P.q) + ((int64_t)(P.row0 + i) * HD + h * pd.head_dim) * pd.isz;
  const uint8_t* qa = qrow + dA * pd.isz;
  const uint8_t* qb = qrow + dB * pd.isz;
  if constexpr (IN == KVPOOL_F32) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 r = *reinterpret_cast<const uint4*>((c < 2 ? qa : qb) + 16 * (c & 1));
      qf[4 * c] = __uint_as_float(r.x);
      qf[4 * c + 1] = __uint_as_float(r.y);
      qf[4 * c + 2] = __uint_as_float(r.z);
      qf[4 * c + 3] = __uint_as_float(r.w);
    }
  } else {
    const uint4 r0 = *reinterpret_cast<const uint4*>(qa), r1 = *reinterpret_cast<const uint4*>(qb);
    const uint32_t wq[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      qf[2 * j] = bf16_bits_to_f32(wq[j] & 0xFFFFu);
      qf[2 * j + 1] = __uint_as_float(wq[j] & 0xFFFF0000u);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t lo16 = 0, hi16 = 0;
    if constexpr (CACHE == KVPOOL_FP8_E4M3) {
      const __half a = __float2half_rn(qf[2 * j]), b = __float2half_rn(qf[2 * j + 1]);
      exact &= (__half2float(a) == qf[2 * j]) && (__half2float(b) == qf[2 * j + 1]);
      lo16 = __half_as_ushort(a);
      hi16 = __half_as_ushort(b);
    } else if constexpr (CACHE == KVPOOL_BF16) {
      lo16 = f32_to_bf16_bits(qf[2 * j]);
      hi16 = f32_to_bf16_bits(qf[2 * j + 1]);
      exact &= (bf16_bits_to_f32(lo16) == qf[2 * j]) && (bf16_bits_to_f32(hi16) == qf[2 * j + 1]);
    } else {
      exact = 0;
    }
    qw[j] = lo16 | (hi16 << 16);
  }
  const bool fast = __all_sync(0xffffffffu, exact) != 0;
  // tensor-core scores: fp8 cache, bf16 query, 128-dim heads in groups of 4
  // (warp w: heads 4w .. 4w + 3)
  constexpr bool kTC = CACHE == KVPOOL_FP8_E4M3 && IN == KVPOOL_BF16 && TPH == 8;
  const bool tc = kTC && pd.heads % 4 == 0;
  const uint32_t arow = (uint32_t)((4 * (tid >> 5) + (lane >> 4)) * 128 + 16 * (lane & 3));
  uint32_t bq[8];
  float fq = 0.0f;
  if (tc) q_pieces_fp8(qf, lane, qscale, bq, fq);

  float m_run = -INFINITY, l_run = 0.0f, o[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j] = 0.0f;
  for (int st = 0; st < n_st; ++st) {
    const int s = st % kStages;
    if (!mbar_wait(&full[s], (st / kStages) & 1, pd)) break;
    const uint32_t base = stage0 + (uint32_t)s * stage_bytes;
    const int ne = min(e_stage, cnt - st * e_stage);
    if (tc)
      consume_stage_tc(base, ne, ES, arow, voff, soff, lane, bq, fq, m_run, l_run, o);
    else if (fast)
      consume_stage<CACHE, true, TPH>(base, ne, ES, koff, voff, soff, qscale, qw, qf, m_run, l_run, o);
    else
      consume_stage<CACHE, false, TPH>(base, ne, ES, koff, voff, soff, qscale, qw, qf, m_run, l_run, o);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (act) {
    const int64_t pslot = R.part_base + (part ? R.n_split0 : 0) + split;
    float* po = P.part_o + pslot * HD + h * pd.head_dim;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      reinterpret_cast<float4*>(po + (j < 2 ? dA : dB))[j & 1] =
          make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
    if (rk == 0) {
      float* ml = P.part_ml + (pslot * pd.heads + h) * 2;
      ml[0] = m_run;
      ml[1] = l_run;
    }
  }
}

// Merge of the split partials of one (request, head): o = sum_s 2^(m_s - M) o_s
// / sum_s 2^(m_s - M) l_s.  Warp w of the CTA's nw warps merges splits w,
// w + nw, ... into its own running (max, sum, output) in one pass -- every
// split's loads are independent of the running state, so they are all in
// flight together -- lane l owning dims [4l, 4l + 4); the warps' states are
// then merged through shared memory.  nw is sized to the split count (about
// four splits per warp, at most kCombineWarps).
constexpr int kCombineWarps = 32;
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const __grid_constant__ AttendParams P) {
  pdl_start();
  __shared__ float red_o[kCombineWarps][128];
  __shared__ float red_m[kCombineWarps], red_l[kCombineWarps];
  const int i = blockIdx.x, h = blockIdx.y;
  const AttendReq& R = P.reqs[i];
  const PoolDesc& pd = P.pool;
  const int d = pd.head_dim;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_split = R.n_split0 + R.n_split1;
  // the select passes that read this request's histogram are done: clear it
  // for the next call
  if (h == 0 && P.layer.has_csa) {
    uint32_t* gh = P.hist + (int64_t)i * kHistBins;
    for (int b = threadIdx.x; b < kHistBins; b += blockDim.x) gh[b] = 0u;
  }
  const bool on = 4 * lane < d;
  const int nw = blockDim.x >> 5;
  float m = -INFINITY, l = 0.0f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int s = warp; s < n_split; s += nw) {
    const int64_t gs = R.part_base + s;
    const float2 ml = *reinterpret_cast<const float2*>(P.part_ml + (gs * pd.heads + h) * 2);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (on) v = *reinterpret_cast<const float4*>(P.part_o + gs * pd.HD + h * d + 4 * lane);
    const bool empty = ml.x == -INFINITY;  // an empty split weighs nothing
    const float mn = empty ? m : fmaxf(m, ml.x);
    const float a = m == mn ? 1.0f : exp2f(m - mn);
    const float b = empty ? 0.0f : exp2f(ml.x - mn);
    l = fmaf(ml.y, b, l * a);
    acc.x = fmaf(v.x, b, acc.x * a);
    acc.y = fmaf(v.y, b, acc.y * a);
    acc.z = fmaf(v.z, b, acc.z * a);
    acc.w = fmaf(v.w, b, acc.w * a);
    m = mn;
  }
  if (on) {
    red_o[warp][4 * lane] = acc.x;
    red_o[warp][4 * lane + 1] = acc.y;
    red_o[warp][4 * lane + 2] = acc.z;
    red_o[warp][4 * lane + 3] = acc.w;
  }
  if (lane == 0) {
    red_m[warp] = m;
    red_l[warp] = l;
  }
  __syncthreads();
  if (threadIdx.x < d) {
    float M = -INFINITY;
    for (int w = 0; w < nw; ++w) M = fmaxf(M, red_m[w]);
    float num = 0.0f, den = 0.0f;
    for (int w = 0; w < nw; ++w) {
      if (red_m[w] == -INFINITY) continue;
      const float f = exp2f(red_m[w] - M);
      num = fmaf(red_o[w][threadIdx.x], f, num);
      den = fmaf(red_l[w], f, den);
    }
    P.out[((int64_t)(P.row0 + i) * pd.heads + h) * d + threadIdx.x] = num / den;
  }
}

template <int IN, int CACHE>
int launch_attend_t(const AttendParams& p, cudaStream_t s, int e_stage, size_t smem, int part, int ctas) {
  const int threads = (p.pool.HD / 16 + 31) / 32 * 32 + 32;
  auto go = [&](auto k, size_t* set) {
    if (*set < smem) {
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      *set = smem;
    }
    // part 1 follows the select on the critical path: programmatic dependent
    // launch (long context 178.4 -> 177.3 us per step)
    launch_kernel(part == 1, k, dim3(ctas), dim3(threads), smem, s, p, e_stage, part);
  };
  static size_t set[4] = {0, 0, 0, 0};
  // only part 1 (selected CSA entries) can meet an offloaded entry
  const bool hs = p.pool.hisparse != 0 && part == 1;
  if (p.pool.head_dim == 128) {
    if (hs) go(attend_kernel<IN, CACHE, 8, true>, &set[0]);
    else go(attend_kernel<IN, CACHE, 8, false>, &set[1]);
  } else if (p.pool.head_dim == 64) {
    if (hs) go(attend_kernel<IN, CACHE, 4, true>, &set[2]);
    else go(attend_kernel<IN, CACHE, 4, false>, &set[3]);
  } else {
    return (int)cudaErrorInvalidValue;
  }
  return (int)cudaGetLastError();
}

}  // namespace

// entries per pipeline stage: about 16 KiB, at most 8
int attend_stage_entries(const PoolDesc& pd) {
  const int e = (int)(16448 / pd.entry_bytes);
  return e < 1 ? 1 : (e > 8 ? 8 : e);
}

size_t attend_smem_bytes(const PoolDesc& pd) {
  return kBarBytes + (size_t)kStages * attend_stage_entries(pd) * pd.entry_bytes;
}

int attend_max_split_len() { return kMaxSplitLen; }

int launch_attend(const AttendParams& p, int part, int ctas, void* stream, int* n_kernels) {
  if (ctas <= 0) return 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int e_stage = attend_stage_entries(p.pool);
  const size_t smem = attend_smem_bytes(p.pool);
  *n_kernels += 1;
  const int key = p.pool.in_dtype * 3 + p.pool.cache_dtype;
  switch (key) {
    case KVPOOL_F32 * 3 + KVPOOL_F32: return launch_attend_t<KVPOOL_F32, KVPOOL_F32>(p, s, e_stage, smem, part, ctas);
    case KVPOOL_F32 * 3 + KVPOOL_BF16: return launch_attend_t<KVPOOL_F32, KVPOOL_BF16>(p, s, e_stage, smem, part, ctas);
    case KVPOOL_F32 * 3 + KVPOOL_FP8_E4M3:
      return launch_attend_t<KVPOOL_F32, KVPOOL_FP8_E4M3>(p, s, e_stage, smem, part, ctas);
    case KVPOOL_BF16 * 3 + KVPOOL_F32: return launch_attend_t<KVPOOL_BF16, KVPOOL_F32>(p, s, e_stage, smem, part, ctas);
    case KVPOOL_BF16 * 3 + KVPOOL_BF16: return launch_attend_t<KVPOOL_BF16, KVPOOL_BF16>(p, s, e_stage, smem, part, ctas);
    case KVPOOL_BF16 * 3 + KVPOOL_FP8_E4M3:
      return launch_attend_t<KVPOOL_BF16, KVPOOL_FP8_E4M3>(p, s, e_stage, smem, part, ctas);
    default: return (int)cudaErrorInvalidValue;
  }
}

int launch_combine(const AttendParams& p, void* stream, int* n_kernels) {
  if (p.n <= 0) return 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int max_split = 1;
  for (int i = 0; i < p.n; ++i) max_split = std::max(max_split, p.reqs[i].n_split0 + p.reqs[i].n_split1);
  // enough threads for the output row (head_dim), about four splits per warp
  const int nw = std::min(kCombineWarps, std::max((p.pool.head_dim + 31) / 32, (max_split + 3) / 4));
  launch_kernel(true, combine_kernel, dim3(p.n, p.pool.heads), dim3(nw * 32), 0, s, p);
  *n_kernels += 1;
  return (int)cudaGetLastError();
}

}  // namespace kvp

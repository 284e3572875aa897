// kvpool_append.cu -- fused append / compress / seal kernel and the
// share-prefix window fill.
//
// One CTA handles one (request, block segment, slice of the 2*H*d K/V
// values, layer) of an append call ("Why does V4 split pools? ..." s4: a new
// token enters the tail; when a 4-group or a 128-group completes it is
// compressed into a CSA or HCA entry; the SWA window slides).
//
// The compressor is an fp32 chain acc = fma(alpha_i, x_i, acc) over a group's
// tokens in position order.  Instead of keeping the tail's raw tokens and
// re-reading them when a group completes, the kernel carries the chain's
// running value: inside one call in registers, across calls in a per-request
// fp32 accumulator in the State region.  The chain order is unchanged, so the
// entry is bit-identical to compressing the stored tail at the end; the tail's
// raw tokens themselves remain visible to attention through the SWA window
// (the window is a whole number of blocks, so it always covers the tail).
#include <cuda_runtime.h>

#include "device_util.cuh"
#include "kvpool_internal.h"

namespace kvp {
namespace {

constexpr int kVpt = 8;  // consecutive values per thread

// 16 bytes from a shared-memory address
__device__ __forceinline__ uint4 lds16(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}

template <int IN>
struct InTraits;
template <>
struct InTraits<KVPOOL_F32> {
  static constexpr int kBytes = 4;
  struct Raw {
    uint4 a, b;
  };
  __device__ static Raw load(const uint8_t* p) { return Raw{ld_nc16(p), ld_nc16(p + 16)}; }
  __device__ static void unpack(const Raw& r, float* x) {
    x[0] = __uint_as_float(r.a.x); x[1] = __uint_as_float(r.a.y); x[2] = __uint_as_float(r.a.z);
    x[3] = __uint_as_float(r.a.w); x[4] = __uint_as_float(r.b.x); x[5] = __uint_as_float(r.b.y);
    x[6] = __uint_as_float(r.b.z); x[7] = __uint_as_float(r.b.w);
  }
  __device__ static void load8(const uint8_t* p, float* x) { unpack(load(p), x); }
  __device__ static void load8_sa(uint32_t a, float* x) { unpack(Raw{lds16(a), lds16(a + 16)}, x); }
};
template <>
struct InTraits<KVPOOL_BF16> {
  static constexpr int kBytes = 2;
  using Raw = uint4;
  __device__ static Raw load(const uint8_t* p) { return ld_nc16(p); }
  __device__ static void unpack(const Raw& a, float* x) {
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
      x[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
    }
  }
  __device__ static void load8(const uint8_t* p, float* x) { unpack(load(p), x); }
  __device__ static void load8_sa(uint32_t a, float* x) { unpack(lds16(a), x); }
};

// Store 8 fp32 values (already scaled for fp8) as cache codes at dst.
template <int CACHE>
__device__ __forceinline__ void store8(uint8_t* dst, const float* x, float inv_unused);

template <>
__device__ __forceinline__ void store8<KVPOOL_F32>(uint8_t* dst, const float* x, float) {
  uint4 a = make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]), __float_as_uint(x[3]));
  uint4 b = make_uint4(__float_as_uint(x[4]), __float_as_uint(x[5]), __float_as_uint(x[6]), __float_as_uint(x[7]));
  *reinterpret_cast<uint4*>(dst) = a;
  *reinterpret_cast<uint4*>(dst + 16) = b;
}
template <>
__device__ __forceinline__ void store8<KVPOOL_BF16>(uint8_t* dst, const float* x, float) {
  // two values per conversion (round to nearest even; the first operand goes
  // to the high half)
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[i]) : "f"(x[2 * i + 1]), "f"(x[2 * i]));
  *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
}
template <>
__device__ __forceinline__ void store8<KVPOOL_FP8_E4M3>(uint8_t* dst, const float* x, float s) {
  // code = e4m3_rn_satfinite(x / s), s the bf16 scale widened to fp32
  uint32_t w[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(x[4 * i], s), __fdiv_rn(x[4 * i + 1], s));
    const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(x[4 * i + 2], s), __fdiv_rn(x[4 * i + 3], s));
    w[i] = lo | (hi << 16);
  }
  *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
}

__device__ __forceinline__ float amax8(const float* x) {
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < kVpt; ++i) a = fmaxf(a, fabsf(x[i]));
  return a;
}

// Block-wide maxima of three per-thread values (K half, V half, indexer).
__device__ __forceinline__ float3 block_max3(float a, float b, float c, float* sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
    c = fmaxf(c, __shfl_xor_sync(0xffffffffu, c, o));
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();
  if (l == 0) {
    sh[3 * w] = a;
    sh[3 * w + 1] = b;
    sh[3 * w + 2] = c;
  }
  __syncthreads();
  float3 r = make_float3(0.f, 0.f, 0.f);
  for (int i = 0; i < nw; ++i) {
    r.x = fmaxf(r.x, sh[3 * i]);
    r.y = fmaxf(r.y, sh[3 * i + 1]);
    r.z = fmaxf(r.z, sh[3 * i + 2]);
  }
  return r;
}

// Write one K/V entry (CSA entry, HCA entry or window token) of which this
// thread holds 8 consecutive fp32 values starting at v0 of [K | V]; all
// threads of the CTA call it together.  For fp8, K and V get one scale each
// (amax over the half / 448, rounded to bf16).
template <int CACHE>
__device__ __forceinline__ void write_entry(uint8_t* entry, const PoolDesc& pd, int v0, int half, int hv,
                                            const float* x, float* sh) {
  if constexpr (CACHE == KVPOOL_FP8_E4M3) {
    const float a = amax8(x);
    const float3 r = block_max3(half == 0 ? a : 0.f, half == 1 ? a : 0.f, 0.f, sh);
    const uint16_t sb = fp8_scale_bits(half == 0 ? r.x : r.y);
    store8<CACHE>(entry + v0, x, bf16_bits_to_f32(sb));
    if (hv == 0) *reinterpret_cast<uint16_t*>(entry + 2 * pd.HD + 2 * half) = sb;
    if (v0 == 0) {
      uint32_t* pad = reinterpret_cast<uint32_t*>(entry + 2 * pd.HD + 4);
      pad[0] = 0u;
      pad[1] = 0u;
      pad[2] = 0u;
    }
  } else {
    store8<CACHE>(entry + (int64_t)v0 * pd.vs, x, 1.0f);
  }
}

// Indexer entry: 8 values at xv0 of the [Ih][Id] key, stored chunk-major in
// the block's indexer part `base`.
template <int CACHE>
__device__ __forceinline__ void write_idx(uint8_t* base, const PoolDesc& pd, int slot, int xv0, const float* x,
                                          float s) {
  const int CB = pd.csa_per_block;
  if constexpr (CACHE == KVPOOL_FP8_E4M3) {
    const int c = xv0 / 16, within = xv0 % 16;
    store8<CACHE>(base + ((int64_t)c * CB + slot) * 16 + within, x, s);
  } else if constexpr (CACHE == KVPOOL_BF16) {
    const int c = xv0 / 8;
    store8<CACHE>(base + ((int64_t)c * CB + slot) * 16, x, 1.0f);
  } else {
    const int c = xv0 / 4;  // two chunks
    uint4 a = make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]), __float_as_uint(x[3]));
    uint4 b = make_uint4(__float_as_uint(x[4]), __float_as_uint(x[5]), __float_as_uint(x[6]), __float_as_uint(x[7]));
    *reinterpret_cast<uint4*>(base + ((int64_t)c * CB + slot) * 16) = a;
    *reinterpret_cast<uint4*>(base + ((int64_t)(c + 1) * CB + slot) * 16) = b;
  }
}

// FP4 indexer entry: 8 values at xv0 as 4 bytes of e2m1 pairs (element 2j in
// the low nibble) inside chunk xv0 / 32 of the block's indexer part.
__device__ __forceinline__ void write_idx_fp4(uint8_t* base, const PoolDesc& pd, int slot, int xv0, const float* x,
                                              float s) {
  uint32_t w = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w |= (uint32_t)f32x2_to_e2m1x2(__fdiv_rn(x[2 * i], s), __fdiv_rn(x[2 * i + 1], s)) << (8 * i);
  *reinterpret_cast<uint32_t*>(base + ((int64_t)(xv0 / 32) * pd.csa_per_block + slot) * 16 + (xv0 % 32) / 2) = w;
}

constexpr int kTokGroup = 8;
__device__ __forceinline__ void ld8f(const float* p, float* x) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void st8f(float* p, const float* x) {
  reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}  // tokens whose loads are issued together

// ---------------------------------------------------------------------------
// Staged token rows (long units, e.g. prefill chunks): the unit's input rows
// -- this CTA's span of each K and V row and, for slice 0, each indexer row --
// stream through a ring of kAppendStages shared-memory stages of
// P.stage_tokens tokens, filled by 1-D bulk copies (one copy for all tokens of
// a stage where the span is the whole row, else one per token, issued by the
// lanes of warp 0).  token(t, x, y) then runs for every token in order with
// the thread's values read from shared memory -- the same per-token work and
// order as the direct loads, so every stored value is identical.  Returns
// false (the same in every thread) if a wait ran out; the copies still in
// flight are waited for (time-limited) first.
// ---------------------------------------------------------------------------
constexpr int kAppendStages = 4;
constexpr int kAppendRingOffset = 128;  // the stages' barriers sit in front of the ring

template <int IN, typename F>
__device__ bool staged_tokens(const AppendParams& P, const AppendUnit& u, int layer, int slice, int HD, int XD,
                              bool idx_thread, int half, int hv, int xv0, F&& token) {
  extern __shared__ __align__(128) uint8_t ring[];
  constexpr int isz = InTraits<IN>::kBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring);
  uint8_t* stages = ring + kAppendRingOffset;
  const PoolDesc& pd = P.pool;
  const int tid = threadIdx.x, lane = tid & 31;
  const int cv0 = slice * blockDim.x * kVpt, cv1 = cv0 + blockDim.x * kVpt;  // this CTA's values of [K | V]
  const int k_lo = min(cv0, HD), k_hi = min(cv1, HD);
  const int v_lo = max(cv0, HD) - HD, v_hi = max(cv1, HD) - HD;
  const int kb = (k_hi - k_lo) * isz, vb = (v_hi - v_lo) * isz;
  const int xb = (slice == 0 && P.layers[layer].has_csa && u.role != kUnitHca) ? XD * isz : 0;
  const int TS = P.stage_tokens;
  const int tok_bytes = kb + vb + xb;
  const int64_t stage_bytes = (int64_t)TS * tok_bytes;
  const int n_tok = u.t1 - u.t0;
  const int n_st = (n_tok + TS - 1) / TS;
  const int64_t row0 = (int64_t)layer * P.rows + u.in_row;
  const uint8_t* kin = reinterpret_cast<const uint8_t*>(P.k) + row0 * HD * isz + (int64_t)k_lo * isz;
  const uint8_t* vin = reinterpret_cast<const uint8_t*>(P.v) + row0 * HD * isz + (int64_t)v_lo * isz;
  const uint8_t* xin = xb ? reinterpret_cast<const uint8_t*>(P.idx_k) + row0 * XD * isz : nullptr;
  if (tid == 0) {
    for (int s = 0; s < kAppendStages; ++s) mbar_init(&full[s], 1);
    mbar_fence_init();
  }
  __syncthreads();
  const uint64_t l2pol = l2_evict_first_policy();  // the input rows are read once
  auto issue = [&](int st) {  // warp 0: stage st into slot st % kAppendStages
    const int s = st % kAppendStages;
    const int j0 = st * TS, nt = min(TS, n_tok - j0);
    uint8_t* dst = stages + (int64_t)s * stage_bytes;
    if (lane == 0) {
      fence_proxy_async();  // the CTA's reads of the slot come before the copies that overwrite it
      mbar_arrive_expect_tx(&full[s], (uint32_t)(nt * tok_bytes));
    }
    __syncwarp();
    if (kb) {
      if (kb == HD * isz) {
        if (lane == 0) bulk_g2s_stream(dst, kin + (int64_t)j0 * kb, (uint32_t)(nt * kb), &full[s], l2pol);
      } else {
        for (int j = lane; j < nt; j += 32) bulk_g2s_stream(dst + j * kb, kin + (int64_t)(j0 + j) * HD * isz, kb, &full[s], l2pol);
      }
    }
    if (vb) {
      uint8_t* dv = dst + (int64_t)TS * kb;
      if (vb == HD * isz) {
        if (lane == 0) bulk_g2s_stream(dv, vin + (int64_t)j0 * vb, (uint32_t)(nt * vb), &full[s], l2pol);
      } else {
        for (int j = lane; j < nt; j += 32) bulk_g2s_stream(dv + j * vb, vin + (int64_t)(j0 + j) * HD * isz, vb, &full[s], l2pol);
      }
    }
    if (xb && lane == 0) bulk_g2s_stream(dst + (int64_t)TS * (kb + vb), xin + (int64_t)j0 * xb, (uint32_t)(nt * xb), &full[s], l2pol);
  };
  // the thread's values in a stage: shared-memory addresses of token 0 and
  // the step from one token to the next
  const uint32_t stage_sa = smem_addr(stages);
  const uint32_t x_off = (uint32_t)(half == 0 ? (hv - k_lo) * isz : TS * kb + (hv - v_lo) * isz);
  const uint32_t x_step = (uint32_t)(half == 0 ? kb : vb);
  const uint32_t y_off = (uint32_t)(TS * (kb + vb) + xv0 * isz);
  if (tid < 32)
    for (int st = 0; st < n_st && st < kAppendStages; ++st) issue(st);
  for (int st = 0; st < n_st; ++st) {
    const int s = st % kAppendStages;
    const bool got = mbar_wait(&full[s], (st / kAppendStages) & 1, pd);
    if (__syncthreads_or(!got)) {  // drain the copies still in flight, then give up
      if (tid == 0)
        for (int k = st; k < n_st && k < st + kAppendStages; ++k)
          mbar_wait(&full[k % kAppendStages], (k / kAppendStages) & 1, pd);
      return false;
    }
    const int nt = min(TS, n_tok - st * TS);
    uint32_t px = stage_sa + (uint32_t)(s * stage_bytes) + x_off, py = stage_sa + (uint32_t)(s * stage_bytes) + y_off;
    int t = u.t0 + st * TS;
    // two tokens per iteration: the next token's shared-memory loads issue
    // while this one's chains run (four measured no better)
#pragma unroll 2
    for (int j = 0; j < nt; ++j, px += x_step, py += (uint32_t)xb, ++t) {
      float x[kVpt], y[kVpt];
      InTraits<IN>::load8_sa(px, x);
      if (idx_thread) InTraits<IN>::load8_sa(py, y);
      token(t, x, y);
    }
    __syncthreads();  // every thread is done with slot s
    if (tid < 32 && st + kAppendStages < n_st) issue(st + kAppendStages);
  }
  return true;
}

// PT: per-token indexer keys (the pool's idx_per_token), a separate
// instantiation so the per-entry path keeps its registers
// STAGED: the unit's tokens arrive through staged_tokens (long units) instead
// of direct loads of kTokGroup tokens at a time.
template <int IN, int CACHE, bool PT, bool STAGED>
__global__ void __launch_bounds__(512) append_kernel(const __grid_constant__ AppendParams P) {
  pdl_start();
  __shared__ float sh[3 * 16];
  const PoolDesc& pd = P.pool;
  const AppendUnit u = P.units[blockIdx.x];
  const int slice = blockIdx.y;
  const int layer = blockIdx.z;
  const LayerDesc& L = P.layers[layer];
  const int tid = threadIdx.x;
  const int HD = pd.HD, XD = pd.XD, m = pd.m, mp = pd.m_prime;
  constexpr int isz = InTraits<IN>::kBytes;

  if (u.slot < 0 || u.slot >= pd.max_requests || u.seg < 0 || u.seg >= pd.max_bpr + 1 ||
      u.block_id >= pd.max_blocks || u.t0 < 0 || u.t1 > mp || u.t0 > u.t1 ||
      (u.block_id >= 0 && (u.csa_slot < 0 || u.csa_slot >= pd.csa_staging_base))) {
    if (tid == 0) flag_error(pd, kErrBadIndex);
    return;
  }

  // Seal copy CTAs (slices n_slices ..): the CSA / indexer entries that
  // earlier calls staged move into the sealing block, spread over
  // copy_slices CTAs of the unit (this call's own entries go to the block
  // directly).
  if (slice >= P.n_slices) {
    if (u.role == kUnitCsa || u.block_id < 0 || !L.has_csa || u.t0 < (PT ? 1 : m)) return;
    const int cs = slice - P.n_slices, ncs = P.copy_slices;
    const int n_copy = u.t0 / m;
    const int CB = pd.csa_per_block;
    const int32_t sid = pd.staging_base + u.slot;
    const uint8_t* stg_csa = pd.arena + L.csa_pool + (int64_t)(pd.csa_staging_base + u.slot) * L.csa_stride;
    uint8_t* dst_csa = pd.arena + L.csa_pool + (int64_t)u.csa_slot * L.csa_stride;
    const uint8_t* stg_idx = pd.arena + L.idx_pool + (int64_t)sid * L.idx_stride;
    uint8_t* dst_idx = pd.arena + L.idx_pool + (int64_t)u.block_id * L.idx_stride;
    const int64_t units = (int64_t)n_copy * pd.entry_bytes / 16;  // CSA entries, 16-byte units
    for (int64_t o = (int64_t)cs * blockDim.x + tid; o < units; o += (int64_t)ncs * blockDim.x)
      reinterpret_cast<uint4*>(dst_csa)[o] = reinterpret_cast<const uint4*>(stg_csa)[o];
    // indexer keys: of the staged entries, or with per-token keys of the
    // staged tokens (key e in run e / CB, slot e % CB)
    const int n_keys = PT ? u.t0 : n_copy;
    for (int64_t k = (int64_t)cs * blockDim.x + tid; k < (int64_t)pd.idx_chunks * n_keys; k += (int64_t)ncs * blockDim.x) {
      const int c = (int)(k / n_keys), e = (int)(k % n_keys);
      const int64_t o = (int64_t)(e / CB) * L.idx_run + ((int64_t)c * CB + e % CB) * 16;
      *reinterpret_cast<uint4*>(dst_idx + o) = *reinterpret_cast<const uint4*>(stg_idx + o);
    }
    const bool scaled = pd.idx_dtype == KVPOOL_FP8_E4M3 || pd.idx_dtype == KVPOOL_FP4_E2M1;
    if (scaled && cs == 0)
      for (int e = tid; e < n_keys; e += blockDim.x) {
        const int64_t o = (int64_t)(e / CB) * L.idx_run + L.idx_scale_off + 2 * (e % CB);
        *reinterpret_cast<uint16_t*>(dst_idx + o) = *reinterpret_cast<const uint16_t*>(stg_idx + o);
      }
    return;
  }

  const int v0 = (slice * blockDim.x + tid) * kVpt;  // my values in [K | V]
  const int half = v0 >= HD ? 1 : 0;
  const int hv = v0 - half * HD;
  const int h = hv / pd.head_dim;
  // the parts of the unit this CTA does (one layer's kinds decide the rest)
  const bool do_hca = L.has_hca && u.role != kUnitCsa;
  const bool do_csa = L.has_csa && u.role != kUnitHca;
  const bool do_win = u.role != kUnitHca;
  const bool idx_thread = do_csa && slice == 0 && tid * kVpt < XD;
  const bool idx_fp4 = pd.idx_dtype == KVPOOL_FP4_E2M1;
  const bool idx_scaled = idx_fp4 || pd.idx_dtype == KVPOOL_FP8_E4M3;
  const int xv0 = tid * kVpt;
  const int g = idx_thread ? xv0 / pd.idx_dim : 0;

  const uint8_t* in_kv = reinterpret_cast<const uint8_t*>(half ? P.v : P.k) +
                         ((int64_t)layer * P.rows + u.in_row) * HD * isz + (int64_t)hv * isz;
  const uint8_t* in_x = idx_thread ? reinterpret_cast<const uint8_t*>(P.idx_k) +
                                         ((int64_t)layer * P.rows + u.in_row) * XD * isz + (int64_t)xv0 * isz
                                   : nullptr;

  float* acc_base = reinterpret_cast<float*>(pd.arena + L.acc + (int64_t)u.slot * L.acc_req_bytes);
  float* acc_c_ptr = acc_base + v0;
  float* acc_x_ptr = acc_base + 2 * HD + xv0;
  float* acc_h_ptr = acc_base + 2 * HD + XD + v0;
  const float* a_csa = reinterpret_cast<const float*>(pd.arena + L.alpha_csa) + h * m;
  const float* a_hca = reinterpret_cast<const float*>(pd.arena + L.alpha_hca) + h * mp;
  const float* a_idx = reinterpret_cast<const float*>(pd.arena + L.alpha_idx) + g * m;

  float acc_c[kVpt], acc_h[kVpt], acc_x[kVpt];
#pragma unroll
  for (int j = 0; j < kVpt; ++j) acc_c[j] = acc_h[j] = acc_x[j] = 0.0f;
  if (do_hca && u.t0 > 0) {
    ld8f(acc_h_ptr, acc_h);
  }
  if (do_csa && (u.t0 % m) != 0) {
    ld8f(acc_c_ptr, acc_c);
    if (idx_thread) {
      ld8f(acc_x_ptr, acc_x);
    }
  }

  const int32_t dst_block = u.block_id >= 0 ? u.block_id : pd.staging_base + u.slot;
  // CSA entries go to the block's CSA slot (its id without HiSparse)
  const int32_t csa_slot = u.block_id >= 0 ? u.csa_slot : pd.csa_staging_base + u.slot;
  uint8_t* blk_csa = pd.arena + L.csa_pool + (int64_t)csa_slot * L.csa_stride;
  uint8_t* blk_idx = pd.arena + L.idx_pool + (int64_t)dst_block * L.idx_stride;
  uint8_t* blk_hca = pd.arena + L.hca_pool + (int64_t)dst_block * L.hca_stride;
  uint8_t* ring = pd.arena + L.ring + (int64_t)u.slot * L.ring_req_bytes;
  const int64_t seg_pos0 = (int64_t)u.seg * mp;

  // The tokens come in order from u.t0, so the per-token positions are
  // counters rather than divisions: tm = t % m, tq = t / m, and for per-token
  // keys tk = t % CB, tr = t / CB.  The window is a whole number of blocks, so
  // a segment's tokens never wrap the ring: slot = (segment start mod n_win) + t.
  int tm = u.t0 % m, tq = u.t0 / m;
  int tk = u.t0 % pd.csa_per_block, tr = u.t0 / pd.csa_per_block;
  // the gates of the current token: HCA by position, CSA / indexer by the
  // position in the group (advanced with the counters)
  const float* pa_h = a_hca + u.t0;
  const float* pa_c = a_csa + tm;
  const float* pa_x = a_idx + tm;
  const int64_t ring_base = seg_pos0 % pd.n_win;

  // the per-token work (window, compressor chains, completed entries); x: this
  // thread's kVpt input values of token t, y: its indexer values (idx threads)
  auto token = [&](int t, const float* x, const float* y) {
    if (do_hca) {
      const float a = __ldg(pa_h);
#pragma unroll
      for (int j = 0; j < kVpt; ++j) acc_h[j] = __fmaf_rn(a, x[j], acc_h[j]);
    }
    if (do_csa) {
      const float a = __ldg(pa_c);
#pragma unroll
      for (int j = 0; j < kVpt; ++j) acc_c[j] = __fmaf_rn(a, x[j], acc_c[j]);
      if constexpr (PT) {
        // the token's own indexer key, at key t % CB of run t / CB; the
        // indexer threads are the first XD / 8 lanes of warp 0
        if (slice == 0 && tid < 32) {
          float s = 1.0f;
          uint8_t* run = blk_idx + (int64_t)tr * L.idx_run;
          const int key = tk;
          if (idx_scaled) {
            float a = idx_thread ? amax8(y) : 0.0f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
            const uint16_t sb = idx_fp4 ? fp4_scale_bits(a) : fp8_scale_bits(a);
            s = bf16_bits_to_f32(sb);
            if (idx_thread && xv0 == 0) *reinterpret_cast<uint16_t*>(run + L.idx_scale_off + 2 * key) = sb;
          }
          if (idx_thread) {
            if (idx_fp4) write_idx_fp4(run, pd, key, xv0, y, s);
            else write_idx<CACHE>(run, pd, key, xv0, y, s);
          }
        }
      } else if (idx_thread) {
        const float b = __ldg(pa_x);
#pragma unroll
        for (int j = 0; j < kVpt; ++j) acc_x[j] = __fmaf_rn(b, y[j], acc_x[j]);
      }
      if (tm == m - 1) {  // a CSA group completes: entry slot (t+1)/m - 1 = t / m of the block
        const int slot = tq;
        write_entry<CACHE>(blk_csa + (int64_t)slot * pd.entry_bytes, pd, v0, half, hv, acc_c, sh);
        float s = 1.0f;
        if (idx_scaled && !PT) {  // uniform over the CTA: block-wide amax of the indexer entry
          const float3 r = block_max3(0.f, 0.f, idx_thread ? amax8(acc_x) : 0.f, sh);
          const uint16_t sb = idx_fp4 ? fp4_scale_bits(r.z) : fp8_scale_bits(r.z);
          s = bf16_bits_to_f32(sb);
          if (idx_thread && xv0 == 0) *reinterpret_cast<uint16_t*>(blk_idx + L.idx_scale_off + 2 * slot) = sb;
        }
        if (idx_thread && !PT) {
          if (idx_fp4) write_idx_fp4(blk_idx, pd, slot, xv0, acc_x, s);
          else write_idx<CACHE>(blk_idx, pd, slot, xv0, acc_x, s);
        }
#pragma unroll
        for (int j = 0; j < kVpt; ++j) acc_c[j] = acc_x[j] = 0.0f;
      }
    }
    if (do_win && t >= u.ring_from)  // the token enters the SWA window
      write_entry<CACHE>(ring + (ring_base + t) * pd.entry_bytes, pd, v0, half, hv, x, sh);
    ++pa_h;
    ++pa_c;
    ++pa_x;
    if (++tm == m) {
      tm = 0;
      pa_c = a_csa;
      pa_x = a_idx;
      ++tq;
    }
    if constexpr (PT) {
      if (++tk == pd.csa_per_block) {
        tk = 0;
        ++tr;
      }
    }
  };

  bool ok = true;
  if constexpr (!STAGED) {
    using Raw = typename InTraits<IN>::Raw;
    for (int tb = u.t0; tb < u.t1; tb += kTokGroup) {
      const int n = min(kTokGroup, u.t1 - tb);
      Raw xr[kTokGroup], yr[kTokGroup];
#pragma unroll
      for (int gi = 0; gi < kTokGroup; ++gi) {
        if (gi < n) {
          xr[gi] = InTraits<IN>::load(in_kv + (int64_t)(tb - u.t0 + gi) * HD * isz);
          if (idx_thread) yr[gi] = InTraits<IN>::load(in_x + (int64_t)(tb - u.t0 + gi) * XD * isz);
        }
      }
#pragma unroll
      for (int gi = 0; gi < kTokGroup; ++gi) {
        if (gi >= n) break;
        float x[kVpt], y[kVpt];
        InTraits<IN>::unpack(xr[gi], x);
        if (idx_thread) InTraits<IN>::unpack(yr[gi], y);
        token(tb + gi, x, y);
      }
    }
  } else {
    ok = staged_tokens<IN>(P, u, layer, slice, HD, XD, idx_thread, half, hv, xv0, token);
  }
  if (!ok) return;  // a wait ran out: the error word says so, nothing more is written

  if (do_hca && u.t1 == mp) {  // the HCA group completes with the block
    if (u.block_id < 0) {
      if (tid == 0) flag_error(pd, kErrBadBlock);
    } else {
      write_entry<CACHE>(blk_hca, pd, v0, half, hv, acc_h, sh);
    }
  }
  if (do_hca && u.t1 < mp) {
    st8f(acc_h_ptr, acc_h);
  }
  if (do_csa && (u.t1 % m) != 0) {
    st8f(acc_c_ptr, acc_c);
    if (idx_thread) {
      st8f(acc_x_ptr, acc_x);
    }
  }

  if (u.block_id >= 0 && slice == 0 && layer == 0 && tid == 0) {
    reinterpret_cast<int32_t*>(pd.arena + pd.table)[(int64_t)u.slot * pd.max_bpr + u.seg] = u.block_id;
    if (pd.hisparse) {  // the new block's CSA location and activity stamp
      reinterpret_cast<int32_t*>(pd.arena + pd.csa_loc)[u.block_id] = u.csa_slot;
      reinterpret_cast<uint32_t*>(pd.arena + pd.last_used)[u.block_id] = P.epoch;
    }
  }
}

// share_prefix: blockIdx.x = window token, blockIdx.y = slice, blockIdx.z = layer;
// the CTA (0, 0, 0) also copies the shared block ids into dst's table row
// (src >= 0; a restored prefix image writes its own ids).
template <int IN, int CACHE>
__global__ void __launch_bounds__(512) share_kernel(const __grid_constant__ ShareParams P) {
  pdl_start();
  __shared__ float sh[3 * 16];
  const PoolDesc& pd = P.pool;
  const int tok = blockIdx.x, slice = blockIdx.y, layer = blockIdx.z;
  const LayerDesc& L = P.layers[layer];
  const int HD = pd.HD;
  constexpr int isz = InTraits<IN>::kBytes;
  const int v0 = (slice * blockDim.x + threadIdx.x) * kVpt;
  const int half = v0 >= HD ? 1 : 0;
  const int hv = v0 - half * HD;
  if (P.src >= 0 && blockIdx.x == 0 && slice == 0 && layer == 0) {
    int32_t* table = reinterpret_cast<int32_t*>(pd.arena + pd.table);
    for (int b = threadIdx.x; b < P.n_blocks; b += blockDim.x)
      table[(int64_t)P.dst * pd.max_bpr + b] = table[(int64_t)P.src * pd.max_bpr + b];
  }
  float x[kVpt];
  const uint8_t* src = reinterpret_cast<const uint8_t*>(half ? P.win_v : P.win_k) +
                       ((int64_t)layer * P.w + tok) * HD * isz + (int64_t)hv * isz;
  InTraits<IN>::load8(src, x);
  const int64_t pos = P.n_tokens - P.w + tok;
  uint8_t* ring = pd.arena + L.ring + (int64_t)P.dst * L.ring_req_bytes;
  write_entry<CACHE>(ring + (pos % pd.n_win) * pd.entry_bytes, pd, v0, half, hv, x, sh);
}


int append_threads(const PoolDesc& pd, int n_slices) { return 2 * pd.HD / kVpt / n_slices; }

constexpr int kAppendStageBudget = 48 * 1024;  // bytes of one stage of the staged path

}  // namespace

// CTAs that split one unit's 2*H*d values (8 per thread): one CTA up to 256
// threads; fp8 needs each half (K, V) inside one CTA for its scale.
int append_slices(const PoolDesc& pd) {
  const int chunks = 2 * pd.HD / kVpt;
  if (chunks <= 256) return 1;
  if (pd.cache_dtype == KVPOOL_FP8_E4M3) return 2;
  return chunks / 256;
}

// Slices of the staged path: the same as the direct path, so a CTA's span of
// a K or V row is the whole row (one bulk copy moves all tokens of a stage);
// finer slices of 64 threads measured slower (1 KB copies, 4 warps per SM).
int append_slices_staged(const PoolDesc& pd) { return append_slices(pd); }

// Bytes one token takes in a stage (the widest slice: slice 0 also stages the
// indexer row), tokens per stage, and the dynamic shared memory of the ring.
static int append_token_bytes(const PoolDesc& pd, int n_slices) {
  return (2 * pd.HD / n_slices) * pd.isz + pd.XD * pd.isz;
}
int append_stage_tokens(const PoolDesc& pd, int n_slices) {
  const int tb = append_token_bytes(pd, n_slices);
  int ts = 32;
  while (ts > 1 && ts * tb > kAppendStageBudget) ts /= 2;
  return ts;
}
static size_t append_staged_smem(const PoolDesc& pd, int n_slices, int ts) {
  return (size_t)kAppendRingOffset + (size_t)kAppendStages * ts * append_token_bytes(pd, n_slices);
}

int launch_append(const AppendParams& p, int n_layers, void* stream, int* n_kernels) {
  if (p.n_units <= 0) return 0;
  const int want = p.staged ? append_slices_staged(p.pool) : append_slices(p.pool);
  if (p.n_slices != want) return (int)cudaErrorInvalidValue;
  if (p.staged && (p.stage_tokens < 1 || p.stage_tokens != append_stage_tokens(p.pool, p.n_slices)))
    return (int)cudaErrorInvalidValue;
  const int threads = append_threads(p.pool, p.n_slices);
  if (p.copy_slices < 0) return (int)cudaErrorInvalidValue;
  dim3 grid(p.n_units, p.n_slices + p.copy_slices, n_layers);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t smem = p.staged ? append_staged_smem(p.pool, p.n_slices, p.stage_tokens) : 0;
  const int key = p.pool.in_dtype * 3 + p.pool.cache_dtype;
  // the four instantiations of one dtype pair: (per-entry | per-token keys) x (direct | staged)
  auto go = [&](auto k_entry, auto k_token, auto k_entry_st, auto k_token_st) {
    if (p.staged) {
      // the ring needs more than the default dynamic shared memory; staged
      // launches move whole prefill chunks, so the attribute is simply set
      // before each one
      auto k = p.pool.idx_per_token ? k_token_st : k_entry_st;
      cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      return launch_kernel(true, k, grid, dim3(threads), smem, s, p);
    } else {
      return launch_kernel(true, p.pool.idx_per_token ? k_token : k_entry, grid, dim3(threads), 0, s, p);
    }
  };
  cudaError_t e = cudaSuccess;
#define KVP_APPEND_KERNELS(I, C) \
  append_kernel<I, C, false, false>, append_kernel<I, C, true, false>, append_kernel<I, C, false, true>, \
      append_kernel<I, C, true, true>
  switch (key) {
    case KVPOOL_F32 * 3 + KVPOOL_F32: e = go(KVP_APPEND_KERNELS(KVPOOL_F32, KVPOOL_F32)); break;
    case KVPOOL_F32 * 3 + KVPOOL_BF16: e = go(KVP_APPEND_KERNELS(KVPOOL_F32, KVPOOL_BF16)); break;
    case KVPOOL_F32 * 3 + KVPOOL_FP8_E4M3: e = go(KVP_APPEND_KERNELS(KVPOOL_F32, KVPOOL_FP8_E4M3)); break;
    case KVPOOL_BF16 * 3 + KVPOOL_F32: e = go(KVP_APPEND_KERNELS(KVPOOL_BF16, KVPOOL_F32)); break;
    case KVPOOL_BF16 * 3 + KVPOOL_BF16: e = go(KVP_APPEND_KERNELS(KVPOOL_BF16, KVPOOL_BF16)); break;
    case KVPOOL_BF16 * 3 + KVPOOL_FP8_E4M3: e = go(KVP_APPEND_KERNELS(KVPOOL_BF16, KVPOOL_FP8_E4M3)); break;
    default: return (int)cudaErrorInvalidValue;
  }
#undef KVP_APPEND_KERNELS
  *n_kernels += 1;
  return (int)(e != cudaSuccess ? e : cudaGetLastError());
}

int launch_share(const ShareParams& p, int n_layers, void* stream, int* n_kernels) {
  if (p.w <= 0) return 0;
  const int n_slices = append_slices(p.pool);
  const int threads = append_threads(p.pool, n_slices);
  dim3 grid(p.w, n_slices, n_layers);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int key = p.pool.in_dtype * 3 + p.pool.cache_dtype;
  switch (key) {
    case KVPOOL_F32 * 3 + KVPOOL_F32: launch_kernel(true, share_kernel<KVPOOL_F32, KVPOOL_F32>, grid, dim3(threads), 0, s, p); break;
    case KVPOOL_F32 * 3 + KVPOOL_BF16: launch_kernel(true, share_kernel<KVPOOL_F32, KVPOOL_BF16>, grid, dim3(threads), 0, s, p); break;
    case KVPOOL_F32 * 3 + KVPOOL_FP8_E4M3: launch_kernel(true, share_kernel<KVPOOL_F32, KVPOOL_FP8_E4M3>, grid, dim3(threads), 0, s, p); break;
    case KVPOOL_BF16 * 3 + KVPOOL_F32: launch_kernel(true, share_kernel<KVPOOL_BF16, KVPOOL_F32>, grid, dim3(threads), 0, s, p); break;
    case KVPOOL_BF16 * 3 + KVPOOL_BF16: launch_kernel(true, share_kernel<KVPOOL_BF16, KVPOOL_BF16>, grid, dim3(threads), 0, s, p); break;
    case KVPOOL_BF16 * 3 + KVPOOL_FP8_E4M3: launch_kernel(true, share_kernel<KVPOOL_BF16, KVPOOL_FP8_E4M3>, grid, dim3(threads), 0, s, p); break;
    default: return (int)cudaErrorInvalidValue;
  }
  *n_kernels += 1;
  return (int)cudaGetLastError();
}

}  // namespace kvp

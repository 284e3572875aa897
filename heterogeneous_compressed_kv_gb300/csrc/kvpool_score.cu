// kvpool_score.cu -- lightning-indexer scores of every CSA entry
// ("V4 KV Layout: Classical + State dual pool", Classical KV cache table:
// CSA entries are read top-k sparse; the State cache table: the indexer keeps
// light K-only vectors for that choice).
//
// One warp per block of csa_per_block (= 32) entries; lane e owns entry e and
// runs the fixed-order fp32 chain
//   acc = fma(q_idx[v], key_e[v], acc), v = 0 .. Ih*Id-1
// (times the entry's bf16 scale for fp8 and FP4).  The indexer keys of a
// block are stored 16-byte-chunk-major, so chunk c of the warp's 32 entries is
// one 512-byte coalesced read.  Scores become orderable uint32 keys; a CTA
// histograms their top 11 bits in shared memory and adds its histogram to the
// request's (the first radix digit of the top-k select).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "device_util.cuh"
#include "kvpool_internal.h"

namespace kvp {
namespace {

// One 16-byte chunk of an indexer key folded into the score chain, in order;
// q points at the chunk's query values in shared memory (16-byte aligned).
template <int CACHE>
struct IdxChunk;

template <>
struct IdxChunk<KVPOOL_F32> {
  static constexpr int kVals = 4;
  __device__ static float chain(const uint4& c, const float* q, float acc) {
    const float4 a = *reinterpret_cast<const float4*>(q);
    acc = __fmaf_rn(a.x, __uint_as_float(c.x), acc);
    acc = __fmaf_rn(a.y, __uint_as_float(c.y), acc);
    acc = __fmaf_rn(a.z, __uint_as_float(c.z), acc);
    acc = __fmaf_rn(a.w, __uint_as_float(c.w), acc);
    return acc;
  }
};
template <>
struct IdxChunk<KVPOOL_BF16> {
  static constexpr int kVals = 8;
  __device__ static float chain(const uint4& c, const float* q, float acc) {
    const float4 a = *reinterpret_cast<const float4*>(q), b = *reinterpret_cast<const float4*>(q + 4);
    const float qq[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = __fmaf_rn(qq[2 * i], bf16_bits_to_f32(w[i] & 0xFFFFu), acc);
      acc = __fmaf_rn(qq[2 * i + 1], bf16_bits_to_f32(w[i] >> 16), acc);
    }
    return acc;
  }
};
template <>
struct IdxChunk<KVPOOL_FP8_E4M3> {
  static constexpr int kVals = 16;
  __device__ static float chain(const uint4& c, const float* q, float acc) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 qq = *reinterpret_cast<const float4*>(q + 4 * i);
      const float2 a = e4m3x2_to_f32x2((uint16_t)(w[i] & 0xFFFFu));
      const float2 b = e4m3x2_to_f32x2((uint16_t)(w[i] >> 16));
      acc = __fmaf_rn(qq.x, a.x, acc);
      acc = __fmaf_rn(qq.y, a.y, acc);
      acc = __fmaf_rn(qq.z, b.x, acc);
      acc = __fmaf_rn(qq.w, b.y, acc);
    }
    return acc;
  }
};

template <>
struct IdxChunk<KVPOOL_FP4_E2M1> {  // 32 e2m1 values, element 2j in the low nibble of byte j
  static constexpr int kVals = 32;
  __device__ static float chain(const uint4& c, const float* q, float acc) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t hw[4];
      e2m1x8_to_f16x2x4(w[i], hw);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t h = hw[b];
        const int v = 8 * i + 2 * b;
        acc = __fmaf_rn(q[v], __half2float(__ushort_as_half((uint16_t)(h & 0xFFFFu))), acc);
        acc = __fmaf_rn(q[v + 1], __half2float(__ushort_as_half((uint16_t)(h >> 16))), acc);
      }
    }
    return acc;
  }
};

// Fast chains: the same fixed-order fp32 chain with the products taken by the
// mixed-precision FMA (f16 x f16 + f32 or bf16 x bf16 + f32; a product of two
// f16 or two bf16 values is exact in fp32 and the FMA rounds once, so every
// step equals fmaf on the widened operands).  qh holds the query as f16 (fp8
// keys, which convert exactly to f16) or bf16 (bf16 keys) pairs.
template <int CACHE>
struct IdxChunkFast;

// acc = fma(hi(a), hi(b), fma(lo(a), lo(b), acc)): two chain steps on the
// halves of two f16 (or bf16) pairs, low half first; the halves are taken
// apart inside one asm block so no extraction instructions are emitted
__device__ __forceinline__ float chain2_f16(uint32_t a, uint32_t b, float acc) {
  asm("{.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\tfma.rn.f32.f16 %0, ah, bh, %0;}"
      : "+f"(acc)
      : "r"(a), "r"(b));
  return acc;
}
__device__ __forceinline__ float chain2_bf16(uint32_t a, uint32_t b, float acc) {
  asm("{.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %0;\n\tfma.rn.f32.bf16 %0, ah, bh, %0;}"
      : "+f"(acc)
      : "r"(a), "r"(b));
  return acc;
}

template <>
struct IdxChunkFast<KVPOOL_FP8_E4M3> {  // 16 keys per chunk, q as 16 f16
  __device__ static float chain(const uint4& c, const uint32_t* qh, float acc) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    const uint4 qa = *reinterpret_cast<const uint4*>(qh), qb = *reinterpret_cast<const uint4*>(qh + 4);
    const uint32_t q[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = chain2_f16(e4m3x2_to_f16x2((uint16_t)(w[i] & 0xFFFFu)), q[2 * i], acc);
      acc = chain2_f16(e4m3x2_to_f16x2((uint16_t)(w[i] >> 16)), q[2 * i + 1], acc);
    }
    return acc;
  }
};
template <>
struct IdxChunkFast<KVPOOL_BF16> {  // 8 keys per chunk, q as 8 bf16
  __device__ static float chain(const uint4& c, const uint32_t* qh, float acc) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    const uint4 qa = *reinterpret_cast<const uint4*>(qh);
    const uint32_t q[4] = {qa.x, qa.y, qa.z, qa.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) acc = chain2_bf16(w[i], q[i], acc);
    return acc;
  }
};
template <>
struct IdxChunkFast<KVPOOL_FP4_E2M1> {  // 32 keys per chunk, q as 32 f16
  __device__ static float chain(const uint4& c, const uint32_t* qh, float acc) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 qv = *reinterpret_cast<const uint4*>(qh + 4 * i);
      const uint32_t q[4] = {qv.x, qv.y, qv.z, qv.w};
      uint32_t h[4];
      e2m1x8_to_f16x2x4(w[i], h);
#pragma unroll
      for (int b = 0; b < 4; ++b) acc = chain2_f16(h[b], q[b], acc);
    }
    return acc;
  }
};
template <>
struct IdxChunkFast<KVPOOL_F32> {  // unused: fp32 keys take the fp32 chain
  __device__ static float chain(const uint4&, const uint32_t*, float acc) { return acc; }
};

// ---------------------------------------------------------------------------
// score kernel.  Every warp streams its own blocks: lane 0 issues a 1-D bulk
// copy of a block's indexer section (keys + fp8 scales, contiguous) into one
// of the warp's R shared-memory slots; the warp waits on that slot's
// mbarrier, copies its keys into registers (lane e = entry e), refills the
// slot with the warp's next-but-(R-1) block, and runs the chains.  Warp w of
// a CTA takes the CTA's blocks w, w + W, w + 2W, ...; a slot's barrier is only
// waited on by its own warp, in order, so every parity wait is exact.
// ---------------------------------------------------------------------------
// Warps per score CTA: more warps keep more fixed-order chains in flight (the
// chain is latency-bound: one dependent FMA per key value).  FP4 blocks are
// small enough for 20 warps with 2 slots each (FP4 scoring is bound by its
// instruction stream rather than its copies: 20 warps 67.6 -> 65.4 us at
// 8 x 1M, 24 no better); fp8 blocks take 16 warps with one slot each (a warp
// moves its block's keys into registers and refills the slot before running
// its chains, so the copy of its next block is in flight meanwhile: 16 copies
// per SM); the 16 KiB bf16 blocks fit 8 warps.
template <int IDX>
struct ScoreShape {
  static constexpr int kWarps = IDX == KVPOOL_FP4_E2M1 ? 20 : IDX == KVPOOL_FP8_E4M3 ? 16 : 8;
  static constexpr int kRegChunks = IDX == KVPOOL_FP4_E2M1 ? 8 : 16;  // key chunks held in registers
};
constexpr int kScoreMaxWarps = 20;
constexpr int kScoreMaxRing = 3;                      // slots per warp
constexpr int kScoreMaxSlots = kScoreMaxWarps * kScoreMaxRing;
constexpr int kScoreMaxGates = 64;  // per-token keys: idx_heads * m gates in shared memory
constexpr int kScoreStageBudget = 140 * 1024;         // shared memory for slots: two per warp measured as fast as three
constexpr int kScoreStageBudgetFp4 = 176 * 1024;      // FP4: 20 warps x 2 slots of 4,160 bytes
__host__ __device__ constexpr int score_warps(int idx_dtype) {
  return idx_dtype == KVPOOL_FP4_E2M1 ? 20 : idx_dtype == KVPOOL_FP8_E4M3 ? 16 : 8;
}

// PT: per-token indexer keys.  A segment is then one run of csa_per_block
// tokens (csa_per_block / m entries) instead of one block; lane t scores
// token t: each head's fp32 chain times the token's scale, an fp32 FMA chain
// over the heads with the entry's gates alpha_idx[j][t % m], and the entry's
// first lane adds its m tokens in order.
template <int IN, int CACHE, bool PT>
__global__ void __launch_bounds__(ScoreShape<CACHE>::kWarps * 32, 1) score_kernel(const __grid_constant__ AttendParams P, int stage_bytes,
                                                                 int ring, int stage_off) {
  pdl_start();
  extern __shared__ __align__(128) uint8_t sm[];
  const PoolDesc& pd = P.pool;
  const LayerDesc& L = P.layer;
  const int XD = pd.XD;
  const int CW = blockDim.x >> 5;  // warps (fewer than kWarps when a block's keys are large)
  constexpr int KCH = ScoreShape<CACHE>::kRegChunks;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm);
  float* q_sh = reinterpret_cast<float*>(sm + 8 * kScoreMaxSlots);
  uint16_t* qh_sh = reinterpret_cast<uint16_t*>(q_sh + XD);  // q as f16 (fp8 keys) or bf16 (bf16 keys)
  uint32_t* hist = reinterpret_cast<uint32_t*>(qh_sh + XD);
  uint8_t* slots = sm + stage_off;

  const int i = find_req(P, blockIdx.x, 0);
  const AttendReq& R = P.reqs[i];
  const int CB = pd.csa_per_block;
  const int m = pd.m;
  const int EPS = PT ? CB / m : CB;  // entries per segment
  const int nseg = (R.n_cand + EPS - 1) / EPS;
  __shared__ float a_sh[kScoreMaxGates];  // per-token keys: the indexer gates [Ih][m]
  if (PT) {
    const float* ag = reinterpret_cast<const float*>(pd.arena + L.alpha_idx);
    for (int v = threadIdx.x; v < pd.idx_heads * m && v < kScoreMaxGates; v += blockDim.x) a_sh[v] = ag[v];
  }
  const int seg_begin = (blockIdx.x - R.score_base) * P.segs_per_cta;
  const int seg_end = min(nseg, seg_begin + P.segs_per_cta);
  const int n_st = max(0, seg_end - seg_begin);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // this warp's blocks: st = warp + j * CW, j = 0 .. mine-1
  const int mine = warp < n_st ? (n_st - 1 - warp) / CW + 1 : 0;
  const int32_t* table = reinterpret_cast<const int32_t*>(pd.arena + pd.table) + (int64_t)R.slot * pd.max_bpr;
  const int32_t staging = pd.staging_base + R.slot;
  auto block_id = [&](int jj) -> int32_t {  // id of this warp's jj-th block (any lane)
    const int seg = seg_begin + warp + jj * CW;
    const int blk = PT ? seg / m : seg;
    if (jj >= mine || blk >= R.n_sealed) return staging;
    const int32_t bid = table[blk];
    if (bid < 0 || bid >= pd.max_blocks) {
      flag_error(pd, kErrBadBlock);
      return staging;  // read something valid; the error word reports it
    }
    return bid;
  };
  // block ids 32 at a time, one batch ahead of their use (lane x holds block
  // batch*32 + x); requests come in increasing order
  int32_t id_cur = block_id(lane), id_nxt = block_id(32 + lane);
  int id_batch = 0;
  auto src_of = [&](int jj) -> const uint8_t* {  // all lanes call it
    while ((jj >> 5) > id_batch) {
      ++id_batch;
      id_cur = id_nxt;
      id_nxt = block_id((id_batch + 1) * 32 + lane);
    }
    const int32_t bid = __shfl_sync(0xffffffffu, id_cur, jj & 31);
    const int run = PT ? (seg_begin + warp + jj * CW) % m : 0;
    return pd.arena + L.idx_pool + (int64_t)bid * L.idx_stride + (int64_t)run * L.idx_run;
  };
  const uint64_t l2pol = l2_evict_first_policy();
  uint64_t* my_full = full + warp * ring;
  uint8_t* my_slots = slots + (int64_t)warp * ring * stage_bytes;
  // every warp initialises its own barriers and starts its first copies
  // before the query is loaded (the copies need neither the query nor the
  // other warps)
  if (lane == 0) {
    for (int s = 0; s < ring; ++s) mbar_init(&my_full[s], 1);
    mbar_fence_init();
  }
  __syncwarp();
  for (int jj = 0; jj < mine && jj < ring; ++jj) {
    const uint8_t* src = src_of(jj);
    if (lane == 0) {
      mbar_arrive_expect_tx(&my_full[jj], (uint32_t)stage_bytes);
      bulk_g2s_stream(my_slots + (int64_t)jj * stage_bytes, src, (uint32_t)stage_bytes, &my_full[jj], l2pol);
    }
  }

  // the histogram and the query (its loads overlap the first copies)
  for (int b = tid; b < kHistBins; b += blockDim.x) hist[b] = 0u;
  // the fast chain needs the query exactly in the keys' 16-bit format
  int exact = CACHE != KVPOOL_F32;
  for (int v = tid; v < XD; v += blockDim.x) {
    const int64_t row = (int64_t)(P.row0 + i) * XD + v;
    const float qv = IN == KVPOOL_F32 ? reinterpret_cast<const float*>(P.q_idx)[row]
                                      : bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(P.q_idx)[row]);
    q_sh[v] = qv;
    if (CACHE == KVPOOL_FP8_E4M3 || CACHE == KVPOOL_FP4_E2M1) {
      const __half hq = __float2half_rn(qv);
      qh_sh[v] = __half_as_ushort(hq);
      exact &= __half2float(hq) == qv;
    } else if (CACHE == KVPOOL_BF16) {
      const uint16_t bq = f32_to_bf16_bits(qv);
      qh_sh[v] = bq;
      exact &= bf16_bits_to_f32(bq) == qv;
    }
  }
  const bool fast = __syncthreads_and(exact) != 0;

  constexpr int V = IdxChunk<CACHE>::kVals;
  const int n_chunks = pd.idx_chunks;
  const int key_bytes = CB * (int)pd.idx_entry_bytes;
  uint32_t* keys = P.keys + (int64_t)i * P.key_stride;
  const uint32_t* qh = reinterpret_cast<const uint32_t*>(qh_sh);
  int j = 0;
  for (; j < mine; ++j) {
    const int slot = j % ring;
    bool got = mbar_wait(&my_full[slot], (j / ring) & 1, pd);
    if (PT) got = __all_sync(0xffffffffu, got);  // the lanes exchange scores below
    if (!got) break;
    const uint8_t* stg = my_slots + (int64_t)slot * stage_bytes;
    const int64_t T = (int64_t)(seg_begin + warp + j * CW) * CB + lane;  // entry, or token (PT)
    const int64_t E = PT ? T / m : T;
    const bool valid = lane < CB && E < R.n_cand;
    const int cph = n_chunks / pd.idx_heads;  // chunks per indexer head
    const int ti = lane % m;                  // the token's place in its entry (PT)
    float acc = 0.0f;
    float scale = 1.0f;
    if (n_chunks <= KCH) {
      // the lane's key into registers, then the slot takes the next block
      uint4 ch[KCH];
#pragma unroll
      for (int c = 0; c < KCH; ++c)
        if (c < n_chunks && valid) ch[c] = *reinterpret_cast<const uint4*>(stg + ((int64_t)c * CB + lane) * 16);
      if ((CACHE == KVPOOL_FP8_E4M3 || CACHE == KVPOOL_FP4_E2M1) && valid)
        scale = bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(stg + key_bytes + 2 * lane));
      __syncwarp();
      if (j + ring < mine) {
        const uint8_t* src = src_of(j + ring);
        if (lane == 0) {
          fence_proxy_async();  // the warp's reads of the slot come before the copy that overwrites it
          mbar_arrive_expect_tx(&my_full[slot], (uint32_t)stage_bytes);
          bulk_g2s_stream(my_slots + (int64_t)slot * stage_bytes, src, (uint32_t)stage_bytes, &my_full[slot], l2pol);
        }
      }
      if (valid && PT) {  // per head: chain, times the token's scale, into the gate chain
        float d = 0.0f;
        int left = cph;               // chunks left in the current head
        const float* ga = a_sh + ti;  // the gate of the current head
        auto head_done = [&]() {
          if (--left == 0) {
            if constexpr (CACHE == KVPOOL_FP8_E4M3 || CACHE == KVPOOL_FP4_E2M1) d = __fmul_rn(d, scale);
            acc = __fmaf_rn(*ga, d, acc);
            ga += m;
            d = 0.0f;
            left = cph;
          }
        };
        if (fast) {
#pragma unroll
          for (int c = 0; c < KCH; ++c)
            if (c < n_chunks) {
              d = IdxChunkFast<CACHE>::chain(ch[c], qh + c * (V / 2), d);
              head_done();
            }
        } else {
#pragma unroll
          for (int c = 0; c < KCH; ++c)
            if (c < n_chunks) {
              d = IdxChunk<CACHE>::chain(ch[c], q_sh + c * V, d);
              head_done();
            }
        }
      } else if (valid) {
        if (fast) {
#pragma unroll
          for (int c = 0; c < KCH; ++c)
            if (c < n_chunks) acc = IdxChunkFast<CACHE>::chain(ch[c], qh + c * (V / 2), acc);
        } else {
#pragma unroll
          for (int c = 0; c < KCH; ++c)
            if (c < n_chunks) acc = IdxChunk<CACHE>::chain(ch[c], q_sh + c * V, acc);
        }
      }
    } else {
      if (valid) {
        if (CACHE == KVPOOL_FP8_E4M3 || CACHE == KVPOOL_FP4_E2M1)
          scale = bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(stg + key_bytes + 2 * lane));
        float d = 0.0f;
        int left = cph;
        const float* ga = a_sh + ti;
        for (int c = 0; c < n_chunks; ++c) {
          const uint4 chk = *reinterpret_cast<const uint4*>(stg + ((int64_t)c * CB + lane) * 16);
          if (PT) {
            d = fast ? IdxChunkFast<CACHE>::chain(chk, qh + c * (V / 2), d) : IdxChunk<CACHE>::chain(chk, q_sh + c * V, d);
            if (--left == 0) {
              if constexpr (CACHE == KVPOOL_FP8_E4M3 || CACHE == KVPOOL_FP4_E2M1) d = __fmul_rn(d, scale);
              acc = __fmaf_rn(*ga, d, acc);
              ga += m;
              d = 0.0f;
              left = cph;
            }
          } else {
            acc = fast ? IdxChunkFast<CACHE>::chain(chk, qh + c * (V / 2), acc)
                       : IdxChunk<CACHE>::chain(chk, q_sh + c * V, acc);
          }
        }
      }
      __syncwarp();
      if (j + ring < mine) {
        const uint8_t* src = src_of(j + ring);
        if (lane == 0) {
          fence_proxy_async();  // the warp's reads of the slot come before the copy that overwrites it
          mbar_arrive_expect_tx(&my_full[slot], (uint32_t)stage_bytes);
          bulk_g2s_stream(my_slots + (int64_t)slot * stage_bytes, src, (uint32_t)stage_bytes, &my_full[slot], l2pol);
        }
      }
    }
    if constexpr (PT) {  // the entry's first lane adds its m tokens in order
      float sum = acc;
      for (int k = 1; k < m; ++k) sum += __shfl_sync(0xffffffffu, acc, (lane + k) & 31);
      if (valid && ti == 0) {
        const uint32_t key = score_key(sum);
        keys[E] = key;
        atomicAdd(&hist[key >> 21], 1u);
      }
    } else if (valid) {
      if constexpr (CACHE == KVPOOL_FP8_E4M3 || CACHE == KVPOOL_FP4_E2M1) acc = __fmul_rn(acc, scale);
      const uint32_t key = score_key(acc);
      keys[E] = key;
      atomicAdd(&hist[key >> 21], 1u);
    }
  }
  if (j < mine && lane == 0) {  // a wait gave up: drain this warp's copies still in flight
    for (int jj = j; jj < mine && jj < j + ring; ++jj) mbar_wait(&my_full[jj % ring], (jj / ring) & 1, pd);
  }
  __syncthreads();
  uint32_t* gh = P.hist + (int64_t)i * kHistBins;
  for (int b = tid; b < kHistBins; b += blockDim.x)
    if (hist[b]) atomicAdd(&gh[b], hist[b]);
}

}  // namespace

// Score CTAs of a launch, and the shared-memory plan of the score kernel.
int score_stage_plan(const PoolDesc& pd, int* stage_bytes, int* ring, int* stage_off, int* warps, size_t* smem) {
  // one block's indexer part: keys, then (fp8) scales; the same size as the
  // indexer plane's stride
  *stage_bytes = pd.csa_per_block * (int)pd.idx_entry_bytes +
                 (pd.idx_dtype == KVPOOL_FP8_E4M3 || pd.idx_dtype == KVPOOL_FP4_E2M1
                      ? (2 * pd.csa_per_block + 15) / 16 * 16
                      : 0);
  // fewer warps when even one slot per warp would overrun the budget (large
  // fp32 or bf16 indexer entries)
  const int budget = pd.idx_dtype == KVPOOL_FP4_E2M1 ? kScoreStageBudgetFp4 : kScoreStageBudget;
  *warps = std::max(1, std::min(score_warps(pd.idx_dtype), budget / *stage_bytes));
  *ring = std::max(1, std::min(kScoreMaxRing, budget / (*warps * *stage_bytes)));
  *stage_off = (8 * kScoreMaxSlots + 6 * pd.XD + 4 * kHistBins + 127) / 128 * 128;
  *smem = (size_t)*stage_off + (size_t)*warps * *ring * *stage_bytes;
  return 0;
}

template <int IN, int CACHE, bool PT>
static int launch_score_t(const AttendParams& p, cudaStream_t s) {
  int sb, ns, so, nw;
  size_t smem;
  score_stage_plan(p.pool, &sb, &ns, &so, &nw, &smem);
  auto k = score_kernel<IN, CACHE, PT>;
  static size_t set = 0;
  if (set < smem) {
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    set = smem;
  }
  launch_kernel(true, k, dim3(p.total_score_ctas), dim3(nw * 32), smem, s, p, sb, ns, so);
  return 0;
}

int launch_score(const AttendParams& p, void* stream, int* n_kernels) {
  if (p.total_score_ctas <= 0) return 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the score kernel reads indexer entries only: it is specialised on their type
  const int key = p.pool.in_dtype * 4 + p.pool.idx_dtype;
  if (p.pool.idx_per_token) {  // per-token keys
    switch (key) {
      case KVPOOL_F32 * 4 + KVPOOL_F32: launch_score_t<KVPOOL_F32, KVPOOL_F32, true>(p, s); break;
      case KVPOOL_F32 * 4 + KVPOOL_BF16: launch_score_t<KVPOOL_F32, KVPOOL_BF16, true>(p, s); break;
      case KVPOOL_F32 * 4 + KVPOOL_FP8_E4M3: launch_score_t<KVPOOL_F32, KVPOOL_FP8_E4M3, true>(p, s); break;
      case KVPOOL_F32 * 4 + KVPOOL_FP4_E2M1: launch_score_t<KVPOOL_F32, KVPOOL_FP4_E2M1, true>(p, s); break;
      case KVPOOL_BF16 * 4 + KVPOOL_F32: launch_score_t<KVPOOL_BF16, KVPOOL_F32, true>(p, s); break;
      case KVPOOL_BF16 * 4 + KVPOOL_BF16: launch_score_t<KVPOOL_BF16, KVPOOL_BF16, true>(p, s); break;
      case KVPOOL_BF16 * 4 + KVPOOL_FP8_E4M3: launch_score_t<KVPOOL_BF16, KVPOOL_FP8_E4M3, true>(p, s); break;
      case KVPOOL_BF16 * 4 + KVPOOL_FP4_E2M1: launch_score_t<KVPOOL_BF16, KVPOOL_FP4_E2M1, true>(p, s); break;
      default: return (int)cudaErrorInvalidValue;
    }
    *n_kernels += 1;
    return (int)cudaGetLastError();
  }
  switch (key) {
    case KVPOOL_F32 * 4 + KVPOOL_F32: launch_score_t<KVPOOL_F32, KVPOOL_F32, false>(p, s); break;
    case KVPOOL_F32 * 4 + KVPOOL_BF16: launch_score_t<KVPOOL_F32, KVPOOL_BF16, false>(p, s); break;
    case KVPOOL_F32 * 4 + KVPOOL_FP8_E4M3: launch_score_t<KVPOOL_F32, KVPOOL_FP8_E4M3, false>(p, s); break;
    case KVPOOL_F32 * 4 + KVPOOL_FP4_E2M1: launch_score_t<KVPOOL_F32, KVPOOL_FP4_E2M1, false>(p, s); break;
    case KVPOOL_BF16 * 4 + KVPOOL_F32: launch_score_t<KVPOOL_BF16, KVPOOL_F32, false>(p, s); break;
    case KVPOOL_BF16 * 4 + KVPOOL_BF16: launch_score_t<KVPOOL_BF16, KVPOOL_BF16, false>(p, s); break;
    case KVPOOL_BF16 * 4 + KVPOOL_FP8_E4M3: launch_score_t<KVPOOL_BF16, KVPOOL_FP8_E4M3, false>(p, s); break;
    case KVPOOL_BF16 * 4 + KVPOOL_FP4_E2M1: launch_score_t<KVPOOL_BF16, KVPOOL_FP4_E2M1, false>(p, s); break;
    default: return (int)cudaErrorInvalidValue;
  }
  *n_kernels += 1;
  return (int)cudaGetLastError();
}

}  // namespace kvp

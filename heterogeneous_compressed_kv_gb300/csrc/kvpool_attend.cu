// kvpool_attend.cu -- split-K decode attention over the three sources and the
// split merge ("Why does V4 split pools? ..." s4: attention reads compressed
// Classical entries sparsely (CSA top-k) and densely (HCA) plus the exact
// local State window; one softmax over all of them).
//
// A request's sources are one virtual list [selected CSA entries | HCA
// entries | window tokens]; every source is one contiguous entry of
// entry_bytes ([K | V] codes, fp8 scales), so one 1-D bulk copy (TMA) moves
// it into shared memory wherever it lives (a shared block, the request's
// staging block or its window ring).  A CTA takes one split of the list: its
// producer warp streams the split's entries through a ring of stages guarded
// by mbarriers; consumer threads (8 dims of one head each) run an online
// softmax in the log2 domain and write a partial (max, sum, output) per head.
// Consumer thread = 16 dims of one head; q.k takes mixed-precision FMAs
// (f16 or bf16 products, exact in fp32) when the query is exactly
// representable; fp8 values are weighted by p * scale rounded to f16.
// A merge kernel combines the partials.  All waits are time-limited.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_util.cuh"
#include "kvpool_internal.h"

namespace kvp {
namespace {

constexpr int kStages = 4;
constexpr int kMaxSplitLen = 1024;

__device__ __forceinline__ int find_split_req(const AttendParams& P, int cta, int part) {
  int lo = 0, hi = P.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((part ? P.reqs[mid].cta_base1 : P.reqs[mid].cta_base0) <= cta) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Byte offset (from the arena) of virtual source v of request R.
__device__ __forceinline__ int64_t source_offset(const AttendParams& P, int i, const AttendReq& R, int v) {
  const PoolDesc& pd = P.pool;
  const LayerDesc& L = P.layer;
  const int32_t* table = reinterpret_cast<const int32_t*>(pd.arena + pd.table) + (int64_t)R.slot * pd.max_bpr;
  const int64_t ring = L.ring + (int64_t)R.slot * L.ring_req_bytes;
  if (v < R.k) {
    const int32_t e = P.sel[(int64_t)i * P.sel_stride + v];
    if (e < 0 || e >= R.n_cand) {
      flag_error(pd, kErrBadIndex);
      return ring;
    }
    const int CB = pd.csa_per_block;
    const int seg = e / CB;
    const int32_t bid = seg < R.n_sealed ? table[seg] : pd.staging_base + R.slot;
    if (seg < R.n_sealed && (bid < 0 || bid >= pd.max_blocks)) {
      flag_error(pd, kErrBadBlock);
      return ring;
    }
    return L.csa_pool + (int64_t)bid * L.csa_stride + (int64_t)(e % CB) * pd.entry_bytes;
  }
  v -= R.k;
  if (v < R.n_hca) {
    const int32_t bid = table[v];
    if (bid < 0 || bid >= pd.max_blocks) {
      flag_error(pd, kErrBadBlock);
      return ring;
    }
    return L.hca_pool + (int64_t)bid * L.hca_stride;
  }
  v -= R.n_hca;
  const int64_t pos = R.length - R.w + v;
  return ring + (pos % pd.n_win) * pd.entry_bytes;
}

__device__ __forceinline__ float fma_f16(uint16_t a, uint16_t b, float c) {
  float d;
  asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fma_bf16(uint16_t a, uint16_t b, float c) {
  float d;
  asm("fma.rn.f32.bf16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
  return d;
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)two));
  return h;
}
__device__ __forceinline__ float f16_to_f32(uint32_t h) { return __half2float(__ushort_as_half((uint16_t)h)); }

// Sixteen consecutive cache values of one entry (K or V part of one head) in
// shared memory: as f16 pairs (fp8), bf16 pairs, or fp32.
template <int CACHE>
struct Row16;
template <>
struct Row16<KVPOOL_FP8_E4M3> {  // 16 B -> 8 f16x2 words
  __device__ static void load(const uint8_t* p, uint32_t* w) {
    const uint4 a = *reinterpret_cast<const uint4*>(p);
    const uint32_t b[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[2 * i] = e4m3x2_to_f16x2(b[i] & 0xFFFFu);
      w[2 * i + 1] = e4m3x2_to_f16x2(b[i] >> 16);
    }
  }
};
template <>
struct Row16<KVPOOL_BF16> {  // 32 B -> 8 bf16x2 words
  __device__ static void load(const uint8_t* p, uint32_t* w) {
    const uint4 a = *reinterpret_cast<const uint4*>(p), b = *reinterpret_cast<const uint4*>(p + 16);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  }
};
template <>
struct Row16<KVPOOL_F32> {  // 64 B -> 16 fp32 bit patterns
  __device__ static void load(const uint8_t* p, uint32_t* w) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 a = *reinterpret_cast<const uint4*>(p + 16 * i);
      w[4 * i] = a.x; w[4 * i + 1] = a.y; w[4 * i + 2] = a.z; w[4 * i + 3] = a.w;
    }
  }
};

// value j (0..15) of a loaded row as fp32
template <int CACHE>
__device__ __forceinline__ float row_value(const uint32_t* w, int j) {
  if constexpr (CACHE == KVPOOL_F32) return __uint_as_float(w[j]);
  else if constexpr (CACHE == KVPOOL_BF16) return bf16_bits_to_f32((j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xFFFFu));
  else return f16_to_f32((j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xFFFFu));
}

// TPH: consumer threads per head (head_dim / 16); each owns 16 dims
template <int IN, int CACHE, int TPH>
__global__ void __launch_bounds__(kAttendThreadsMax) attend_kernel(const __grid_constant__ AttendParams P, int e_stage,
                                                                   int part) {
  extern __shared__ __align__(128) uint8_t smem[];
  const PoolDesc& pd = P.pool;
  const int HD = pd.HD;
  const int n_act = HD / 16;                    // consumer threads with work
  const int n_cons = (n_act + 31) / 32 * 32;    // whole consumer warps
  const int n_cons_warps = n_cons / 32;
  const int tid = threadIdx.x;
  const int i = find_split_req(P, blockIdx.x, part);
  const AttendReq& R = P.reqs[i];
  const int split = blockIdx.x - (part ? R.cta_base1 : R.cta_base0);
  // part 0 covers virtual sources [k, k + n_hca + w), part 1 covers [0, k)
  const int lo = part ? 0 : R.k, hi = part ? R.k : R.k + R.n_hca + R.w;
  const int len = part ? R.split_len1 : R.split_len0;
  const int v0 = lo + split * len;
  const int v1 = min(hi, v0 + len);
  const int cnt = v1 - v0;
  const int64_t ES = pd.entry_bytes;
  const int64_t pslot = R.part_base + (part ? R.n_split0 : 0) + split;  // partial slot

  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kStages;
  uint8_t* stage_mem = smem + 64;
  const int64_t stage_bytes = (int64_t)e_stage * ES;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], n_cons_warps);
    }
    mbar_fence_init();
  }
  // consumer: head h, dims [dd0, dd0 + 16); the query row of this thread
  const bool act = tid < n_act;
  const int h = act ? tid / TPH : 0;
  const int dd0 = act ? (tid % TPH) * 16 : 0;
  float qf[16];
  uint32_t qw[8];  // the query as f16 pairs (fp8 cache) or bf16 pairs (bf16 cache)
  int exact = 1;
  if (tid < n_cons) {
    const int64_t base = (int64_t)(P.row0 + i) * HD + h * pd.head_dim + dd0;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      qf[j] = IN == KVPOOL_F32 ? reinterpret_cast<const float*>(P.q)[base + j]
                               : bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(P.q)[base + j]);
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
  }
  const bool fast = __syncthreads_and(tid < n_cons ? exact : 1) != 0;

  const int n_st = (cnt + e_stage - 1) / e_stage;
  if (tid >= n_cons) {
    // producer warp: lanes compute source addresses 32 at a time, one batch
    // ahead of the copies; lane 0 issues the bulk copies of each stage
    const int lane = tid - n_cons;
    int64_t cur = lane < cnt ? source_offset(P, i, R, v0 + lane) : 0;
    int64_t nxt = 32 + lane < cnt ? source_offset(P, i, R, v0 + 32 + lane) : 0;
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
      if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(ne * ES));
      uint8_t* dst = stage_mem + s * stage_bytes;
      for (int e = 0; e < ne; ++e) {
        const int x = e0 + e;
        if ((x >> 5) != batch) {  // next batch of addresses; start the one after it
          batch = x >> 5;
          cur = nxt;
          const int y = (batch + 1) * 32 + lane;
          nxt = y < cnt ? source_offset(P, i, R, v0 + y) : 0;
        }
        const int64_t a = __shfl_sync(0xffffffffu, cur, x & 31);
        if (lane == 0) bulk_g2s(dst + e * ES, pd.arena + a, (uint32_t)ES, &full[s]);
      }
      issued = st + 1;
    }
    if (!ok && lane == 0)  // drain the copies still in flight before leaving
      for (int st = max(0, issued - kStages); st < issued; ++st) mbar_wait(&full[st % kStages], (st / kStages) & 1, pd);
    return;
  }

  // scores in the log2 domain: dot(q, k) * log2(e) / sqrt(d) (* fp8 K scale)
  const float qscale = 1.4426950408889634f * rsqrtf((float)pd.head_dim);
  float m_run = -INFINITY, l_run = 0.0f, o[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j] = 0.0f;
  const int koff = (h * pd.head_dim + dd0) * pd.vs;
  const int voff = HD * pd.vs + koff;

  for (int st = 0; st < n_st; ++st) {
    const int s = st % kStages;
    if (!mbar_wait(&full[s], (st / kStages) & 1, pd)) break;
    const uint8_t* base = stage_mem + s * stage_bytes;
    const int ne = min(e_stage, cnt - st * e_stage);
    for (int e0 = 0; e0 < ne; e0 += 4) {
      float sc[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        sc[u] = -INFINITY;
        if (e0 + u < ne) {
          const uint8_t* ent = base + (e0 + u) * ES;
          uint32_t kw[16];
          Row16<CACHE>::load(ent + koff, kw);
          float d = 0.0f;
          if (CACHE == KVPOOL_FP8_E4M3 && fast) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              d = fma_f16((uint16_t)(kw[j] & 0xFFFFu), (uint16_t)(qw[j] & 0xFFFFu), d);
              d = fma_f16((uint16_t)(kw[j] >> 16), (uint16_t)(qw[j] >> 16), d);
            }
          } else if (CACHE == KVPOOL_BF16 && fast) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              d = fma_bf16((uint16_t)(kw[j] & 0xFFFFu), (uint16_t)(qw[j] & 0xFFFFu), d);
              d = fma_bf16((uint16_t)(kw[j] >> 16), (uint16_t)(qw[j] >> 16), d);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) d = fmaf(qf[j], row_value<CACHE>(kw, j), d);
          }
#pragma unroll
          for (int off = TPH / 2; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
          float f = qscale;
          if constexpr (CACHE == KVPOOL_FP8_E4M3) f *= bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(ent + 2 * HD));
          sc[u] = d * f;
        }
      }
      const float mx = fmaxf(fmaxf(m_run, fmaxf(sc[0], sc[1])), fmaxf(sc[2], sc[3]));
      const float corr = exp2f(m_run - mx);
      l_run *= corr;
#pragma unroll
      for (int j = 0; j < 16; ++j) o[j] *= corr;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (e0 + u < ne) {
          const uint8_t* ent = base + (e0 + u) * ES;
          const float p = exp2f(sc[u] - mx);
          l_run += p;
          uint32_t vw[16];
          Row16<CACHE>::load(ent + voff, vw);
          if constexpr (CACHE == KVPOOL_FP8_E4M3) {
            // weight times the V scale, rounded to f16; products with the f16
            // values are exact, accumulation fp32
            const float ps = p * bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(ent + 2 * HD + 2));
            const uint16_t ph = __half_as_ushort(__float2half_rn(ps));
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              o[2 * j] = fma_f16((uint16_t)(vw[j] & 0xFFFFu), ph, o[2 * j]);
              o[2 * j + 1] = fma_f16((uint16_t)(vw[j] >> 16), ph, o[2 * j + 1]);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] = fmaf(p, row_value<CACHE>(vw, j), o[j]);
          }
        }
      }
      m_run = mx;
    }
    __syncwarp();
    if ((tid & 31) == 0) mbar_arrive(&empty[s]);
  }

  if (act) {
    float* po = P.part_o + pslot * HD + h * pd.head_dim + dd0;
#pragma unroll
    for (int j = 0; j < 4; ++j) reinterpret_cast<float4*>(po)[j] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
    if (dd0 == 0) {
      float* ml = P.part_ml + (pslot * pd.heads + h) * 2;
      ml[0] = m_run;
      ml[1] = l_run;
    }
  }
}

// Merge of the split partials of one (request, head): o = sum_s 2^(m_s - M) o_s
// / sum_s 2^(m_s - M) l_s.  Warp w merges splits w, w + 32, ... with its own
// running maximum (one round of loads in flight), lane l owns dims
// [4l, 4l + 4); the 32 warp results are merged through shared memory.
constexpr int kCombineWarps = 32;
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const __grid_constant__ AttendParams P) {
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
  float m = -INFINITY, l = 0.0f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int s = warp; s < n_split; s += kCombineWarps) {
    const int64_t gs = R.part_base + s;
    const float2 ml = *reinterpret_cast<const float2*>(P.part_ml + (gs * pd.heads + h) * 2);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (on) v = *reinterpret_cast<const float4*>(P.part_o + gs * pd.HD + h * d + 4 * lane);
    if (ml.x == -INFINITY) continue;  // an empty split
    const float mn = fmaxf(m, ml.x);
    const float a = exp2f(m - mn), b = exp2f(ml.x - mn);
    l = l * a + ml.y * b;
    acc.x = acc.x * a + v.x * b;
    acc.y = acc.y * a + v.y * b;
    acc.z = acc.z * a + v.z * b;
    acc.w = acc.w * a + v.w * b;
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
    for (int w = 0; w < kCombineWarps; ++w) M = fmaxf(M, red_m[w]);
    float num = 0.0f, den = 0.0f;
    for (int w = 0; w < kCombineWarps; ++w) {
      if (red_m[w] == -INFINITY) continue;
      const float wt = exp2f(red_m[w] - M);
      num = fmaf(red_o[w][threadIdx.x], wt, num);
      den = fmaf(red_l[w], wt, den);
    }
    P.out[((int64_t)(P.row0 + i) * pd.heads + h) * d + threadIdx.x] = num / den;
  }
}

template <int IN, int CACHE>
int launch_attend_t(const AttendParams& p, cudaStream_t s, int e_stage, size_t smem, int part, int ctas) {
  const int threads = (p.pool.HD / 16 + 31) / 32 * 32 + 32;
  if (p.pool.head_dim == 128) {
    auto k = attend_kernel<IN, CACHE, 8>;
    static size_t set8 = 0;
    if (set8 < smem) {
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      set8 = smem;
    }
    k<<<ctas, threads, smem, s>>>(p, e_stage, part);
  } else if (p.pool.head_dim == 64) {
    auto k = attend_kernel<IN, CACHE, 4>;
    static size_t set4 = 0;
    if (set4 < smem) {
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      set4 = smem;
    }
    k<<<ctas, threads, smem, s>>>(p, e_stage, part);
  } else {
    return (int)cudaErrorInvalidValue;
  }
  return (int)cudaGetLastError();
}

}  // namespace

// entries per pipeline stage: about 16 KiB of entries, at most 8
int attend_stage_entries(const PoolDesc& pd) {
  int e = (int)(16384 / pd.entry_bytes);
  return e < 1 ? 1 : (e > 8 ? 8 : e);
}

size_t attend_smem_bytes(const PoolDesc& pd) {
  return 64 + (size_t)kStages * attend_stage_entries(pd) * pd.entry_bytes;
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
  combine_kernel<<<dim3(p.n, p.pool.heads), kCombineWarps * 32, 0, s>>>(p);
  *n_kernels += 1;
  return (int)cudaGetLastError();
}

}  // namespace kvp

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
// A merge kernel combines the partials.  All waits are time-limited.
#include <cuda_runtime.h>

#include "device_util.cuh"
#include "kvpool_internal.h"

namespace kvp {
namespace {

constexpr int kStages = 3;
constexpr int kMaxSplitLen = 1024;

__device__ __forceinline__ int find_split_req(const AttendParams& P, int cta) {
  int lo = 0, hi = P.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P.reqs[mid].split_base <= cta) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

template <int CACHE>
struct KV8;
template <>
struct KV8<KVPOOL_F32> {
  __device__ static void load(const uint8_t* p, float* x) {
    const uint4 a = *reinterpret_cast<const uint4*>(p), b = *reinterpret_cast<const uint4*>(p + 16);
    x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y); x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
    x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y); x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
  }
};
template <>
struct KV8<KVPOOL_BF16> {
  __device__ static void load(const uint8_t* p, float* x) {
    const uint4 a = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
      x[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
    }
  }
};
template <>
struct KV8<KVPOOL_FP8_E4M3> {
  __device__ static void load(const uint8_t* p, float* x) {
    const uint2 a = *reinterpret_cast<const uint2*>(p);
    const uint32_t w[2] = {a.x, a.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float2 lo = e4m3x2_to_f32x2((uint16_t)(w[i] & 0xFFFFu));
      const float2 hi = e4m3x2_to_f32x2((uint16_t)(w[i] >> 16));
      x[4 * i] = lo.x;
      x[4 * i + 1] = lo.y;
      x[4 * i + 2] = hi.x;
      x[4 * i + 3] = hi.y;
    }
  }
};

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
    return L.block_pool + (int64_t)bid * L.block_bytes + L.csa_off + (int64_t)(e % CB) * pd.entry_bytes;
  }
  v -= R.k;
  if (v < R.n_hca) {
    const int32_t bid = table[v];
    if (bid < 0 || bid >= pd.max_blocks) {
      flag_error(pd, kErrBadBlock);
      return ring;
    }
    return L.block_pool + (int64_t)bid * L.block_bytes + L.hca_off;
  }
  v -= R.n_hca;
  const int64_t pos = R.length - R.w + v;
  return ring + (pos % pd.n_win) * pd.entry_bytes;
}

// TPH: consumer threads per head (head_dim / 8)
template <int IN, int CACHE, int TPH>
__global__ void __launch_bounds__(kAttendThreadsMax) attend_kernel(const __grid_constant__ AttendParams P, int e_stage) {
  extern __shared__ __align__(128) uint8_t smem[];
  const PoolDesc& pd = P.pool;
  const int HD = pd.HD;
  const int n_cons = HD / 8;  // consumer threads
  const int n_cons_warps = n_cons / 32;
  const int tid = threadIdx.x;
  const int i = find_split_req(P, blockIdx.x);
  const AttendReq& R = P.reqs[i];
  const int split = blockIdx.x - R.split_base;
  const int n_src = R.k + R.n_hca + R.w;
  const int v0 = split * R.split_len;
  const int v1 = min(n_src, v0 + R.split_len);
  const int cnt = v1 - v0;
  const int64_t ES = pd.entry_bytes;

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
  // zero this request's select histogram for the next call (the select
  // passes that read it ran before this kernel)
  if (split == 0 && P.layer.has_csa) {
    uint32_t* gh = P.hist + (int64_t)i * kHistBins;
    for (int b = tid; b < kHistBins; b += blockDim.x) gh[b] = 0u;
  }
  __syncthreads();

  const int n_st = (cnt + e_stage - 1) / e_stage;
  if (tid >= n_cons) {
    // producer warp: lanes compute source addresses 32 at a time, one batch
    // ahead of the copies; lane 0 issues the bulk copies of each stage
    const int lane = tid - n_cons;
    if (lane >= 32) return;
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

  // consumer: head h, dims [dd0, dd0 + 8)
  const int h = tid / TPH;
  const int dd0 = (tid % TPH) * 8;
  const float qscale = 1.4426950408889634f * rsqrtf((float)pd.head_dim);  // log2(e) / sqrt(d)
  float q[8];
  {
    const int64_t base = (int64_t)(P.row0 + i) * HD + h * pd.head_dim + dd0;
    if constexpr (IN == KVPOOL_F32) {
      const float* qp = reinterpret_cast<const float*>(P.q) + base;
#pragma unroll
      for (int j = 0; j < 8; ++j) q[j] = qp[j] * qscale;
    } else {
      const uint4 a = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(P.q) + base);
      const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        q[2 * j] = bf16_bits_to_f32(w[j] & 0xFFFFu) * qscale;
        q[2 * j + 1] = bf16_bits_to_f32(w[j] >> 16) * qscale;
      }
    }
  }
  float m_run = -INFINITY, l_run = 0.0f, o[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) o[j] = 0.0f;
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
          float kx[8];
          KV8<CACHE>::load(ent + koff, kx);
          float d = 0.0f;
#pragma unroll
          for (int j = 0; j < 8; ++j) d = fmaf(q[j], kx[j], d);
#pragma unroll
          for (int off = TPH / 2; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
          if constexpr (CACHE == KVPOOL_FP8_E4M3) d *= bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(ent + 2 * HD));
          sc[u] = d;
        }
      }
      const float mx = fmaxf(fmaxf(m_run, fmaxf(sc[0], sc[1])), fmaxf(sc[2], sc[3]));
      const float corr = exp2f(m_run - mx);
      l_run *= corr;
#pragma unroll
      for (int j = 0; j < 8; ++j) o[j] *= corr;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (e0 + u < ne) {
          const uint8_t* ent = base + (e0 + u) * ES;
          float p = exp2f(sc[u] - mx);
          l_run += p;
          if constexpr (CACHE == KVPOOL_FP8_E4M3) p *= bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(ent + 2 * HD + 2));
          float vx[8];
          KV8<CACHE>::load(ent + voff, vx);
#pragma unroll
          for (int j = 0; j < 8; ++j) o[j] = fmaf(p, vx[j], o[j]);
        }
      }
      m_run = mx;
    }
    __syncwarp();
    if ((tid & 31) == 0) mbar_arrive(&empty[s]);
  }

  float* po = P.part_o + (int64_t)blockIdx.x * HD + h * pd.head_dim + dd0;
  reinterpret_cast<float4*>(po)[0] = make_float4(o[0], o[1], o[2], o[3]);
  reinterpret_cast<float4*>(po)[1] = make_float4(o[4], o[5], o[6], o[7]);
  if (dd0 == 0) {
    float* ml = P.part_ml + ((int64_t)blockIdx.x * pd.heads + h) * 2;
    ml[0] = m_run;
    ml[1] = l_run;
  }
}

// Merge of the split partials of one (request, head): o = sum_s 2^(m_s - M) o_s
// / sum_s 2^(m_s - M) l_s.  Warp w takes splits w, w + 8, ...; lane l owns
// dims [4l, 4l + 4).
constexpr int kCombineWarps = 8;
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const __grid_constant__ AttendParams P) {
  __shared__ float red_o[kCombineWarps][128];
  __shared__ float red_l[kCombineWarps];
  __shared__ float sM;
  const int i = blockIdx.x, h = blockIdx.y;
  const AttendReq& R = P.reqs[i];
  const PoolDesc& pd = P.pool;
  const int d = pd.head_dim;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // M: max over the splits' running maxima of this head
  float m = -INFINITY;
  for (int s = threadIdx.x; s < R.n_split; s += blockDim.x)
    m = fmaxf(m, P.part_ml[((int64_t)(R.split_base + s) * pd.heads + h) * 2]);
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red_l[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = -INFINITY;
    for (int w = 0; w < kCombineWarps; ++w) M = fmaxf(M, red_l[w]);
    sM = M;
  }
  __syncthreads();
  const float M = sM;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float l = 0.0f;
  const bool on = 4 * lane < d;
#pragma unroll 4
  for (int s = warp; s < R.n_split; s += kCombineWarps) {
    const int64_t gs = R.split_base + s;
    const float2 ml = *reinterpret_cast<const float2*>(P.part_ml + (gs * pd.heads + h) * 2);
    const float wgt = exp2f(ml.x - M);
    l = fmaf(ml.y, wgt, l);
    if (on) {
      const float4 v = *reinterpret_cast<const float4*>(P.part_o + gs * pd.HD + h * d + 4 * lane);
      acc.x = fmaf(v.x, wgt, acc.x);
      acc.y = fmaf(v.y, wgt, acc.y);
      acc.z = fmaf(v.z, wgt, acc.z);
      acc.w = fmaf(v.w, wgt, acc.w);
    }
  }
  __syncthreads();
  if (on) {
    red_o[warp][4 * lane] = acc.x;
    red_o[warp][4 * lane + 1] = acc.y;
    red_o[warp][4 * lane + 2] = acc.z;
    red_o[warp][4 * lane + 3] = acc.w;
  }
  if (lane == 0) red_l[warp] = l;
  __syncthreads();
  if (threadIdx.x < d) {
    float num = 0.0f, den = 0.0f;
    for (int w = 0; w < kCombineWarps; ++w) {
      num += red_o[w][threadIdx.x];
      den += red_l[w];
    }
    P.out[((int64_t)(P.row0 + i) * pd.heads + h) * d + threadIdx.x] = num / den;
  }
}

template <int IN, int CACHE>
int launch_attend_t(const AttendParams& p, cudaStream_t s, int e_stage, size_t smem) {
  const int threads = p.pool.HD / 8 + 32;
  if (p.pool.head_dim == 128) {
    auto k = attend_kernel<IN, CACHE, 16>;
    static size_t set16 = 0;
    if (set16 < smem) {
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      set16 = smem;
    }
    k<<<p.total_splits, threads, smem, s>>>(p, e_stage);
  } else if (p.pool.head_dim == 64) {
    auto k = attend_kernel<IN, CACHE, 8>;
    static size_t set8 = 0;
    if (set8 < smem) {
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      set8 = smem;
    }
    k<<<p.total_splits, threads, smem, s>>>(p, e_stage);
  } else {
    return (int)cudaErrorInvalidValue;
  }
  return (int)cudaGetLastError();
}

}  // namespace

// entries per pipeline stage: about 32 KiB of entries, at most 16
int attend_stage_entries(const PoolDesc& pd) {
  int e = (int)(32768 / pd.entry_bytes);
  return e < 1 ? 1 : (e > 16 ? 16 : e);
}

size_t attend_smem_bytes(const PoolDesc& pd) {
  return 64 + (size_t)kStages * attend_stage_entries(pd) * pd.entry_bytes;
}

int attend_max_split_len() { return kMaxSplitLen; }

int launch_attend(const AttendParams& p, void* stream, int* n_kernels) {
  if (p.total_splits <= 0) return 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int e_stage = attend_stage_entries(p.pool);
  const size_t smem = attend_smem_bytes(p.pool);
  *n_kernels += 1;
  const int key = p.pool.in_dtype * 3 + p.pool.cache_dtype;
  switch (key) {
    case KVPOOL_F32 * 3 + KVPOOL_F32: return launch_attend_t<KVPOOL_F32, KVPOOL_F32>(p, s, e_stage, smem);
    case KVPOOL_F32 * 3 + KVPOOL_BF16: return launch_attend_t<KVPOOL_F32, KVPOOL_BF16>(p, s, e_stage, smem);
    case KVPOOL_F32 * 3 + KVPOOL_FP8_E4M3: return launch_attend_t<KVPOOL_F32, KVPOOL_FP8_E4M3>(p, s, e_stage, smem);
    case KVPOOL_BF16 * 3 + KVPOOL_F32: return launch_attend_t<KVPOOL_BF16, KVPOOL_F32>(p, s, e_stage, smem);
    case KVPOOL_BF16 * 3 + KVPOOL_BF16: return launch_attend_t<KVPOOL_BF16, KVPOOL_BF16>(p, s, e_stage, smem);
    case KVPOOL_BF16 * 3 + KVPOOL_FP8_E4M3: return launch_attend_t<KVPOOL_BF16, KVPOOL_FP8_E4M3>(p, s, e_stage, smem);
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

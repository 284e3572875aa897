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
// The combine kernel merges the partials.  All waits are time-limited.
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
  int64_t* addr = reinterpret_cast<int64_t*>(smem + 64);
  uint8_t* stage_mem = smem + 64 + kMaxSplitLen * 8;
  const int64_t stage_bytes = (int64_t)e_stage * ES;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], n_cons_warps);
    }
    mbar_fence_init();
  }
  // zero this request's select histograms for the next call (they were
  // consumed by the select passes that ran before this kernel)
  if (split == 0 && P.layer.has_csa) {
    uint32_t* gh = P.hist + (int64_t)i * 3 * kHistBins;
    for (int b = tid; b < 3 * kHistBins; b += blockDim.x) gh[b] = 0u;
  }
  for (int v = tid; v < cnt; v += blockDim.x) addr[v] = source_offset(P, i, R, v0 + v);
  __syncthreads();

  const int n_st = (cnt + e_stage - 1) / e_stage;
  if (tid >= n_cons) {
    // producer warp: one lane issues the bulk copies of each stage
    if (tid == n_cons) {
      int issued = 0;
      bool ok = true;
      for (int st = 0; st < n_st; ++st) {
        const int s = st % kStages;
        if (st >= kStages && !mbar_wait(&empty[s], ((st / kStages) - 1) & 1, pd)) {
          ok = false;
          break;
        }
        const int e0 = st * e_stage;
        const int ne = min(e_stage, cnt - e0);
        mbar_arrive_expect_tx(&full[s], (uint32_t)(ne * ES));
        uint8_t* dst = stage_mem + s * stage_bytes;
        for (int e = 0; e < ne; ++e) bulk_g2s(dst + e * ES, pd.arena + addr[e0 + e], (uint32_t)ES, &full[s]);
        issued = st + 1;
      }
      if (!ok) {  // drain the copies still in flight before leaving
        for (int st = max(0, issued - kStages); st < issued; ++st) mbar_wait(&full[st % kStages], (st / kStages) & 1, pd);
      }
    }
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

  const int gsplit = blockIdx.x;
  float* po = P.part_o + (int64_t)gsplit * HD + h * pd.head_dim + dd0;
#pragma unroll
  for (int j = 0; j < 8; ++j) po[j] = o[j];
  if (dd0 == 0) {
    float* ml = P.part_ml + ((int64_t)gsplit * pd.heads + h) * 2;
    ml[0] = m_run;
    ml[1] = l_run;
  }
}

// grid (n requests, heads); head_dim threads
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ AttendParams P) {
  const int i = blockIdx.x, h = blockIdx.y, j = threadIdx.x;
  const AttendReq& R = P.reqs[i];
  const PoolDesc& pd = P.pool;
  float M = -INFINITY;
  for (int s = 0; s < R.n_split; ++s) M = fmaxf(M, P.part_ml[((int64_t)(R.split_base + s) * pd.heads + h) * 2]);
  float den = 0.0f, num = 0.0f;
  for (int s = 0; s < R.n_split; ++s) {
    const int64_t gs = R.split_base + s;
    const float* ml = P.part_ml + (gs * pd.heads + h) * 2;
    const float w = exp2f(ml[0] - M);
    den = fmaf(ml[1], w, den);
    num = fmaf(P.part_o[gs * pd.HD + h * pd.head_dim + j], w, num);
  }
  P.out[((int64_t)(P.row0 + i) * pd.heads + h) * pd.head_dim + j] = num / den;
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
  return 64 + (size_t)kMaxSplitLen * 8 + (size_t)kStages * attend_stage_entries(pd) * pd.entry_bytes;
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
  dim3 grid(p.n, p.pool.heads);
  combine_kernel<<<grid, p.pool.head_dim, 0, s>>>(p);
  *n_kernels += 1;
  return (int)cudaGetLastError();
}

}  // namespace kvp

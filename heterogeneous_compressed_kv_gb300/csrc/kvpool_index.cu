// kvpool_index.cu -- lightning-indexer scores of every CSA entry and the
// top-k selection over them ("V4 KV Layout: Classical + State dual pool",
// Classical KV cache table: CSA entries are read top-k sparse; the State cache
// table: the indexer keeps light K-only vectors for that choice).
//
// score:  one warp per block of csa_per_block (= 32) entries; lane e owns
//         entry e and runs the fixed-order fp32 chain
//           acc = fma(q_idx[v], key_e[v], acc), v = 0 .. Ih*Id-1
//         (times the entry's bf16 scale for fp8).  The indexer keys of a
//         block are stored 16-byte-chunk-major, so chunk c of the warp's 32
//         entries is one 512-byte coalesced read.  Scores become orderable
//         uint32 keys; a CTA histograms their top 11 bits in shared memory.
// select: three 11/11/10-bit radix passes find the k-th largest key T and
//         how many keys equal to T are taken (lowest indices first); a count
//         pass and an emit pass with ordered block scans then write the
//         selected indices in ascending order.  No pass waits on another
//         CTA; passes are separate launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <new>

#include "device_util.cuh"
#include "kvpool_internal.h"

namespace kvp {
namespace {

__device__ __forceinline__ int find_req(const AttendParams& P, int cta, int which) {
  // requests are ordered by their first CTA index; binary search the last
  // request whose base <= cta
  int lo = 0, hi = P.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    const int base = which == 0 ? P.reqs[mid].score_base : P.reqs[mid].key_base;
    if (base <= cta) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

template <int CACHE>
struct IdxChunk;

template <>
struct IdxChunk<KVPOOL_F32> {
  static constexpr int kVals = 4;
  __device__ static float chain(const uint4& c, const float* q, float acc) {
    acc = __fmaf_rn(q[0], __uint_as_float(c.x), acc);
    acc = __fmaf_rn(q[1], __uint_as_float(c.y), acc);
    acc = __fmaf_rn(q[2], __uint_as_float(c.z), acc);
    acc = __fmaf_rn(q[3], __uint_as_float(c.w), acc);
    return acc;
  }
};
template <>
struct IdxChunk<KVPOOL_BF16> {
  static constexpr int kVals = 8;
  __device__ static float chain(const uint4& c, const float* q, float acc) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = __fmaf_rn(q[2 * i], bf16_bits_to_f32(w[i] & 0xFFFFu), acc);
      acc = __fmaf_rn(q[2 * i + 1], bf16_bits_to_f32(w[i] >> 16), acc);
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
      const float2 a = e4m3x2_to_f32x2((uint16_t)(w[i] & 0xFFFFu));
      const float2 b = e4m3x2_to_f32x2((uint16_t)(w[i] >> 16));
      acc = __fmaf_rn(q[4 * i + 0], a.x, acc);
      acc = __fmaf_rn(q[4 * i + 1], a.y, acc);
      acc = __fmaf_rn(q[4 * i + 2], b.x, acc);
      acc = __fmaf_rn(q[4 * i + 3], b.y, acc);
    }
    return acc;
  }
};

constexpr int kScoreThreads = 256;
constexpr int kChunkBatch = 8;  // 16-byte chunks loaded together per lane

template <int IN, int CACHE>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(const __grid_constant__ AttendParams P) {
  extern __shared__ float q_sh[];  // [XD] fp32 indexer query
  __shared__ uint32_t hist[kHistBins];
  const PoolDesc& pd = P.pool;
  const LayerDesc& L = P.layer;
  const int i = find_req(P, blockIdx.x, 0);
  const AttendReq& R = P.reqs[i];
  const int CB = pd.csa_per_block;
  const int nseg = (R.n_cand + CB - 1) / CB;
  const int seg0 = (blockIdx.x - R.score_base) * kScoreSegsPerCta;
  const int seg1 = min(nseg, seg0 + kScoreSegsPerCta);

  for (int b = threadIdx.x; b < kHistBins; b += blockDim.x) hist[b] = 0u;
  const int XD = pd.XD;
  for (int v = threadIdx.x; v < XD; v += blockDim.x) {
    const int64_t row = (int64_t)(P.row0 + i) * XD + v;
    q_sh[v] = IN == KVPOOL_F32 ? reinterpret_cast<const float*>(P.q_idx)[row]
                               : bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(P.q_idx)[row]);
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int V = IdxChunk<CACHE>::kVals;
  const int n_chunks = pd.idx_chunks;
  const int32_t* table = reinterpret_cast<const int32_t*>(pd.arena + pd.table) + (int64_t)R.slot * pd.max_bpr;
  uint32_t* keys = P.keys + (int64_t)i * P.key_stride;

  for (int seg = seg0 + warp; seg < seg1; seg += kScoreThreads / 32) {
    int32_t bid = seg < R.n_sealed ? table[seg] : pd.staging_base + R.slot;
    if (seg < R.n_sealed && (bid < 0 || bid >= pd.max_blocks)) {
      if (lane == 0) flag_error(pd, kErrBadBlock);
      continue;
    }
    const uint8_t* sec = pd.arena + L.block_pool + (int64_t)bid * L.block_bytes;
    const uint8_t* kbase = sec + L.idx_off;
    for (int e0 = 0; e0 < CB; e0 += 32) {
      const int e = e0 + lane;
      const int64_t E = (int64_t)seg * CB + e;
      const bool valid = e < CB && E < R.n_cand;
      float acc = 0.0f;
      if (valid) {
        for (int c0 = 0; c0 < n_chunks; c0 += kChunkBatch) {
          uint4 ch[kChunkBatch];
#pragma unroll
          for (int b = 0; b < kChunkBatch; ++b)
            if (c0 + b < n_chunks) ch[b] = ld_stream16(kbase + ((int64_t)(c0 + b) * CB + e) * 16);
#pragma unroll
          for (int b = 0; b < kChunkBatch; ++b)
            if (c0 + b < n_chunks) acc = IdxChunk<CACHE>::chain(ch[b], q_sh + (c0 + b) * V, acc);
        }
        if constexpr (CACHE == KVPOOL_FP8_E4M3) {
          const uint16_t sb = *reinterpret_cast<const uint16_t*>(sec + L.idx_scale_off + 2 * e);
          acc = __fmul_rn(acc, bf16_bits_to_f32(sb));
        }
        const uint32_t key = score_key(acc);
        keys[E] = key;
        atomicAdd(&hist[key >> 21], 1u);
      }
    }
  }
  __syncthreads();
  uint32_t* gh = P.hist + (int64_t)i * 3 * kHistBins;
  for (int b = threadIdx.x; b < kHistBins; b += blockDim.x)
    if (hist[b]) atomicAdd(&gh[b], hist[b]);
}

// ---------------------------------------------------------------------------
// radix select
// ---------------------------------------------------------------------------
constexpr int kSelThreads = 256;
constexpr int kItems = kSelectKeysPerCta / kSelThreads;  // 16 keys per thread

// Block-wide: the digit d (bin index) at which the count of keys in bins
// above d is < k and the count in bins >= d is >= k, and k - (count above d).
__device__ void find_digit(const uint32_t* h, int nbins, uint32_t k, uint32_t* sh, uint32_t* d_out,
                           uint32_t* k_out) {
  // thread t owns bins [t*per, (t+1)*per), per = nbins / 256
  const int per = nbins / kSelThreads;
  const int t = threadIdx.x;
  uint32_t own = 0;
  for (int b = 0; b < per; ++b) own += h[t * per + b];
  // inclusive suffix sum over threads (high bins first) via shared memory
  sh[t] = own;
  __syncthreads();
  for (int off = 1; off < kSelThreads; off <<= 1) {
    const uint32_t add = (t + off < kSelThreads) ? sh[t + off] : 0u;
    __syncthreads();
    sh[t] += add;
    __syncthreads();
  }
  const uint32_t incl = sh[t];          // keys in bins >= t*per
  const uint32_t above = incl - own;    // keys in bins >= (t+1)*per
  if (above < k && incl >= k) {
    uint32_t acc = above;
    for (int b = per - 1; b >= 0; --b) {
      const uint32_t c = h[t * per + b];
      if (acc + c >= k) {
        *d_out = (uint32_t)(t * per + b);
        *k_out = k - acc;
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

struct Thresh {
  uint32_t T, need;
};

// Recompute the select state from the global histograms of request i.
// level: how many radix levels are complete (1, 2 or 3).
__device__ void select_state(const AttendParams& P, int i, int level, uint32_t* sh, uint32_t* out /*[4]*/) {
  const AttendReq& R = P.reqs[i];
  const uint32_t* gh = P.hist + (int64_t)i * 3 * kHistBins;
  __shared__ uint32_t st[6];
  if (threadIdx.x == 0) st[0] = st[1] = st[2] = st[3] = st[4] = st[5] = 0;
  __syncthreads();
  find_digit(gh, kHistBins, (uint32_t)R.k, sh, &st[0], &st[1]);
  if (level >= 2) find_digit(gh + kHistBins, kHistBins, st[1], sh, &st[2], &st[3]);
  if (level >= 3) find_digit(gh + 2 * kHistBins, 1024, st[3], sh, &st[4], &st[5]);
  out[0] = st[0];
  out[1] = st[2];
  out[2] = st[4];
  out[3] = level == 1 ? st[1] : level == 2 ? st[3] : st[5];
  __syncthreads();
}

__global__ void __launch_bounds__(kSelThreads) select_hist_kernel(const __grid_constant__ AttendParams P, int level) {
  __shared__ uint32_t sh[kSelThreads];
  __shared__ uint32_t hist[kHistBins];
  const int i = find_req(P, blockIdx.x, 1);
  const AttendReq& R = P.reqs[i];
  if (R.select_all || R.k == 0) return;
  const int64_t k0 = (int64_t)(blockIdx.x - R.key_base) * kSelectKeysPerCta;
  if (k0 >= R.n_cand) return;
  const int64_t k1 = min((int64_t)R.n_cand, k0 + kSelectKeysPerCta);
  uint32_t s[4];
  select_state(P, i, level - 1, sh, s);
  for (int b = threadIdx.x; b < kHistBins; b += blockDim.x) hist[b] = 0u;
  __syncthreads();
  const uint32_t* keys = P.keys + (int64_t)i * P.key_stride;
  for (int64_t e = k0 + threadIdx.x; e < k1; e += blockDim.x) {
    const uint32_t key = keys[e];
    if (level == 2) {
      if ((key >> 21) == s[0]) atomicAdd(&hist[(key >> 10) & 2047u], 1u);
    } else {
      if ((key >> 10) == ((s[0] << 11) | s[1])) atomicAdd(&hist[key & 1023u], 1u);
    }
  }
  __syncthreads();
  uint32_t* gh = P.hist + (int64_t)i * 3 * kHistBins + (level - 1) * kHistBins;
  const int nb = level == 2 ? kHistBins : 1024;
  for (int b = threadIdx.x; b < nb; b += blockDim.x)
    if (hist[b]) atomicAdd(&gh[b], hist[b]);
}

__device__ __forceinline__ Thresh final_thresh(const AttendParams& P, int i, uint32_t* sh) {
  uint32_t s[4];
  select_state(P, i, 3, sh, s);
  return Thresh{(s[0] << 21) | (s[1] << 10) | s[2], s[3]};
}

// counts[i][chunk] = (keys > T, keys == T) in the chunk
__global__ void __launch_bounds__(kSelThreads) select_count_kernel(const __grid_constant__ AttendParams P) {
  __shared__ uint32_t sh[kSelThreads];
  __shared__ uint32_t red[2];
  const int i = find_req(P, blockIdx.x, 1);
  const AttendReq& R = P.reqs[i];
  if (R.select_all || R.k == 0) return;
  const int chunk = blockIdx.x - R.key_base;
  const int64_t k0 = (int64_t)chunk * kSelectKeysPerCta;
  if (k0 >= R.n_cand) return;
  const int64_t k1 = min((int64_t)R.n_cand, k0 + kSelectKeysPerCta);
  const Thresh th = final_thresh(P, i, sh);
  if (threadIdx.x == 0) red[0] = red[1] = 0;
  __syncthreads();
  const uint32_t* keys = P.keys + (int64_t)i * P.key_stride;
  uint32_t gt = 0, eq = 0;
  for (int64_t e = k0 + threadIdx.x; e < k1; e += blockDim.x) {
    const uint32_t key = keys[e];
    gt += key > th.T;
    eq += key == th.T;
  }
  atomicAdd(&red[0], gt);
  atomicAdd(&red[1], eq);
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t* c = P.counts + ((int64_t)i * P.max_key_ctas + chunk) * 2;
    c[0] = red[0];
    c[1] = red[1];
  }
}

// exclusive block scan of one value per thread; returns the block total
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* sh, uint32_t* total) {
  const int t = threadIdx.x;
  sh[t] = v;
  __syncthreads();
  for (int off = 1; off < kSelThreads; off <<= 1) {
    const uint32_t add = t >= off ? sh[t - off] : 0u;
    __syncthreads();
    sh[t] += add;
    __syncthreads();
  }
  const uint32_t incl = sh[t];
  *total = sh[kSelThreads - 1];
  __syncthreads();
  return incl - v;
}

__global__ void __launch_bounds__(kSelThreads) select_emit_kernel(const __grid_constant__ AttendParams P) {
  __shared__ uint32_t sh[kSelThreads];
  const int i = find_req(P, blockIdx.x, 1);
  const AttendReq& R = P.reqs[i];
  const int chunk = blockIdx.x - R.key_base;
  const int64_t k0 = (int64_t)chunk * kSelectKeysPerCta;
  int32_t* sel = P.sel + (int64_t)i * P.sel_stride;
  int32_t* tko = P.topk_out ? P.topk_out + (int64_t)(P.row0 + i) * P.top_k : nullptr;
  if (chunk == 0 && tko)
    for (int j = R.k + threadIdx.x; j < P.top_k; j += blockDim.x) tko[j] = -1;
  if (R.k == 0 || k0 >= R.n_cand) return;
  const int64_t k1 = min((int64_t)R.n_cand, k0 + kSelectKeysPerCta);
  if (R.select_all) {
    for (int64_t e = k0 + threadIdx.x; e < k1; e += blockDim.x) {
      sel[e] = (int32_t)e;
      if (tko) tko[e] = (int32_t)e;
    }
    return;
  }
  const Thresh th = final_thresh(P, i, sh);
  // totals of earlier chunks of this request
  uint32_t base_gt = 0, base_eq = 0;
  const uint32_t* cnt = P.counts + (int64_t)i * P.max_key_ctas * 2;
  for (int c = 0; c < chunk; ++c) {
    base_gt += cnt[2 * c];
    base_eq += cnt[2 * c + 1];
  }
  const uint32_t* keys = P.keys + (int64_t)i * P.key_stride;
  // each thread owns kItems consecutive keys of the chunk
  const int64_t my0 = k0 + (int64_t)threadIdx.x * kItems;
  uint32_t kk[kItems];
  uint32_t n_gt = 0, n_eq = 0;
#pragma unroll
  for (int j = 0; j < kItems; ++j) {
    kk[j] = (my0 + j < k1) ? keys[my0 + j] : 0u;
    const bool in = my0 + j < k1;
    n_gt += in && kk[j] > th.T;
    n_eq += in && kk[j] == th.T;
  }
  uint32_t tot;
  const uint32_t pre_gt = block_excl_scan(n_gt, sh, &tot);
  const uint32_t pre_eq = block_excl_scan(n_eq, sh, &tot);
  uint32_t eq_rank = base_eq + pre_eq;  // equal keys before my first one
  uint32_t gt_rank = base_gt + pre_gt;
#pragma unroll
  for (int j = 0; j < kItems; ++j) {
    const int64_t e = my0 + j;
    if (e >= k1) break;
    bool take = false;
    if (kk[j] > th.T) {
      take = true;
    } else if (kk[j] == th.T) {
      take = eq_rank < th.need;
    }
    if (take) {
      const uint32_t pos = gt_rank + min(eq_rank, th.need);
      if (pos < (uint32_t)R.k) {
        sel[pos] = (int32_t)e;
        if (tko) tko[pos] = (int32_t)e;
      } else {
        flag_error(P.pool, kErrBadIndex);
      }
    }
    if (kk[j] > th.T) ++gt_rank;
    if (kk[j] == th.T) ++eq_rank;
  }
}

}  // namespace

int launch_score(const AttendParams& p, void* stream, int* n_kernels) {
  if (p.total_score_ctas <= 0) return 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t smem = sizeof(float) * p.pool.XD;
  const int key = p.pool.in_dtype * 3 + p.pool.cache_dtype;
  switch (key) {
    case KVPOOL_F32 * 3 + KVPOOL_F32: score_kernel<KVPOOL_F32, KVPOOL_F32><<<p.total_score_ctas, kScoreThreads, smem, s>>>(p); break;
    case KVPOOL_F32 * 3 + KVPOOL_BF16: score_kernel<KVPOOL_F32, KVPOOL_BF16><<<p.total_score_ctas, kScoreThreads, smem, s>>>(p); break;
    case KVPOOL_F32 * 3 + KVPOOL_FP8_E4M3: score_kernel<KVPOOL_F32, KVPOOL_FP8_E4M3><<<p.total_score_ctas, kScoreThreads, smem, s>>>(p); break;
    case KVPOOL_BF16 * 3 + KVPOOL_F32: score_kernel<KVPOOL_BF16, KVPOOL_F32><<<p.total_score_ctas, kScoreThreads, smem, s>>>(p); break;
    case KVPOOL_BF16 * 3 + KVPOOL_BF16: score_kernel<KVPOOL_BF16, KVPOOL_BF16><<<p.total_score_ctas, kScoreThreads, smem, s>>>(p); break;
    case KVPOOL_BF16 * 3 + KVPOOL_FP8_E4M3: score_kernel<KVPOOL_BF16, KVPOOL_FP8_E4M3><<<p.total_score_ctas, kScoreThreads, smem, s>>>(p); break;
    default: return (int)cudaErrorInvalidValue;
  }
  *n_kernels += 1;
  return (int)cudaGetLastError();
}

int launch_select(const AttendParams& p, void* stream, int* n_kernels) {
  if (p.total_key_ctas <= 0) return 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  bool any_radix = false;
  for (int i = 0; i < p.n; ++i) any_radix |= (!p.reqs[i].select_all && p.reqs[i].k > 0);
  if (any_radix) {
    select_hist_kernel<<<p.total_key_ctas, kSelThreads, 0, s>>>(p, 2);
    select_hist_kernel<<<p.total_key_ctas, kSelThreads, 0, s>>>(p, 3);
    select_count_kernel<<<p.total_key_ctas, kSelThreads, 0, s>>>(p);
    *n_kernels += 3;
  }
  select_emit_kernel<<<p.total_key_ctas, kSelThreads, 0, s>>>(p);
  *n_kernels += 1;
  return (int)cudaGetLastError();
}

}  // namespace kvp

// ===========================================================================
// Top-k over a caller's score matrix with no allocation: the scratch (keys,
// radix histograms, per-chunk counts, the selected list, an error word) is a
// file-scope device array owned by this library.  The design pages have no
// counterpart of this entry point; it exists for callers that can only hand
// over an input and an output buffer.
// ===========================================================================
namespace kvp {
namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;  // 16 MiB, held by every device that loads the library
static __device__ __align__(256) uint8_t g_topk_scratch[kStaticScratchBytes];

// device address of g_topk_scratch, looked up once per device
constexpr int kMaxDevices = 64;
static void* g_scratch_addr[kMaxDevices];
static std::mutex g_scratch_mu;

// scores -> orderable keys and the first radix histogram (top 11 bits)
__global__ void __launch_bounds__(kSelThreads) static_keys_kernel(const __grid_constant__ AttendParams P,
                                                                  const float* __restrict__ scores, int64_t ld) {
  __shared__ uint32_t hist[kHistBins];
  const int i = find_req(P, blockIdx.x, 1);
  const AttendReq& R = P.reqs[i];
  const int64_t k0 = (int64_t)(blockIdx.x - R.key_base) * kSelectKeysPerCta;
  const int64_t k1 = min((int64_t)R.n_cand, k0 + kSelectKeysPerCta);
  for (int b = threadIdx.x; b < kHistBins; b += blockDim.x) hist[b] = 0u;
  __syncthreads();
  uint32_t* keys = P.keys + (int64_t)i * P.key_stride;
  for (int64_t e = k0 + threadIdx.x; e < k1; e += blockDim.x) {
    const uint32_t key = score_key(scores[(int64_t)i * ld + e]);
    keys[e] = key;
    atomicAdd(&hist[key >> 21], 1u);
  }
  __syncthreads();
  uint32_t* gh = P.hist + (int64_t)i * 3 * kHistBins;
  for (int b = threadIdx.x; b < kHistBins; b += blockDim.x)
    if (hist[b]) atomicAdd(&gh[b], hist[b]);
}

}  // namespace
}  // namespace kvp

extern "C" int kvpool_topk_static(const float* d_scores, int32_t n_rows, int32_t n_cols, int32_t top_k,
                                  int32_t* d_topk_out, void* stream) {
  using namespace kvp;
  if (n_rows < 0 || n_cols < 0 || top_k < 0) return KVPOOL_ERR_INVALID_ARG;
  if (n_rows == 0 || top_k == 0) return KVPOOL_OK;
  if (!d_scores || !d_topk_out || n_rows > kMaxAttendReqs) return KVPOOL_ERR_INVALID_ARG;
  // scratch plan: [error word | hist | counts | selected | keys], each 256-B aligned
  const int64_t chunks = std::max<int64_t>(1, ((int64_t)n_cols + kSelectKeysPerCta - 1) / kSelectKeysPerCta);
  auto up = [](int64_t x) { return (x + 255) / 256 * 256; };
  const int64_t off_hist = 256;
  const int64_t off_counts = off_hist + up(4LL * n_rows * 3 * kHistBins);
  const int64_t off_sel = off_counts + up(8LL * n_rows * chunks);
  const int64_t off_keys = off_sel + up(4LL * n_rows * top_k);
  const int64_t need = off_keys + up(4LL * n_rows * n_cols);
  if (need > (int64_t)kStaticScratchBytes) return KVPOOL_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVPOOL_ERR_CUDA;
  uint8_t* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_topk_scratch) != cudaSuccess || !ptr) return KVPOOL_ERR_CUDA;
      g_scratch_addr[dev] = ptr;
    }
    base = static_cast<uint8_t*>(g_scratch_addr[dev]);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the error word and the histograms must start at zero; the rest is overwritten
  if (cudaMemsetAsync(base, 0, (size_t)off_counts, s) != cudaSuccess) return KVPOOL_ERR_CUDA;

  AttendParams* P = new (std::nothrow) AttendParams();
  if (!P) return KVPOOL_ERR_INVALID_ARG;
  P->pool.arena = base;
  P->pool.err = 0;
  P->topk_out = d_topk_out;
  P->top_k = top_k;
  P->n = n_rows;
  P->row0 = 0;
  P->keys = reinterpret_cast<uint32_t*>(base + off_keys);
  P->key_stride = n_cols;
  P->hist = reinterpret_cast<uint32_t*>(base + off_hist);
  P->counts = reinterpret_cast<uint32_t*>(base + off_counts);
  P->max_key_ctas = (int32_t)chunks;
  P->sel = reinterpret_cast<int32_t*>(base + off_sel);
  P->sel_stride = top_k;
  for (int i = 0; i < n_rows; ++i) {
    AttendReq& R = P->reqs[i];
    R = AttendReq{};
    R.n_cand = n_cols;
    R.k = std::min(top_k, n_cols);
    R.select_all = R.k == n_cols ? 1 : 0;
    R.key_base = (int32_t)(i * chunks);
  }
  P->total_key_ctas = (int32_t)(n_rows * chunks);
  int rc = 0;
  bool radix = false;
  for (int i = 0; i < n_rows; ++i) radix |= !P->reqs[i].select_all && P->reqs[i].k > 0;
  if (radix) {
    static_keys_kernel<<<P->total_key_ctas, kSelThreads, 0, s>>>(*P, d_scores, n_cols);
    rc = (int)cudaGetLastError();
  }
  int nk = 0;
  if (rc == 0) rc = launch_select(*P, stream, &nk);
  delete P;
  return rc == 0 ? KVPOOL_OK : KVPOOL_ERR_CUDA;
}

// kvpool_select.cu -- the top-k selection over the indexer scores ("V4 KV
// Layout: Classical + State dual pool", Classical KV cache table: CSA entries
// are read top-k sparse): the k largest orderable keys of each request, ties
// to the lower index, written in ascending index order.
//
// The k-th largest key T is found by three radix digits (11, 11 and 10 bits);
// the first comes from the histogram the score kernel built.  Three shapes:
//  - at most 4096 candidates per request: one CTA per request keeps the keys
//    in registers and does everything (select_small_kernel);
//  - more: one CTA per 4096-key chunk lists its keys in buckets >= the first
//    digit, the request's last CTA (atomic count) finds T from the lists and
//    writes the selection from them (select_list_kernel);
//  - a request of more than 16 chunks when the select has the GPU to itself:
//    one thread-block cluster per request, digit histograms summed through
//    distributed shared memory (select_cluster_kernel).
// No CTA waits on another except through a cluster barrier.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <new>

#include "device_util.cuh"
#include "kvpool_internal.h"

namespace cg = cooperative_groups;

namespace kvp {
namespace {

// ---------------------------------------------------------------------------
// radix select
// ---------------------------------------------------------------------------
constexpr int kSelThreads = 256;
constexpr int kItems = kSelectKeysPerCta / kSelThreads;  // 16 keys per thread
constexpr uint32_t kCandCache = 4096;                    // listed candidates kept in shared memory

// Block-wide (NT threads): the digit d (bin index) at which the
// count of keys in bins above d is < k and the count in bins >= d is >= k,
// and k - (count above d).  Thread t owns bins [t*per, (t+1)*per); suffix
// sums run over warp shuffles, then across the 8 warps.
template <int NT = kSelThreads>
__device__ void find_digit(const uint32_t* h, int nbins, uint32_t k, uint32_t* sh, uint32_t* d_out,
                           uint32_t* k_out) {
  const int per = nbins / NT;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  uint32_t own = 0;
  for (int b = 0; b < per; ++b) own += h[t * per + b];
  // inclusive suffix sum within the warp (higher lanes own higher bins)
  uint32_t suf = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_down_sync(0xffffffffu, suf, o);
    if (lane + o < 32) suf += v;
  }
  if (lane == 0) sh[warp] = suf;  // warp total
  __syncthreads();
  uint32_t above_warps = 0;
  for (int w = warp + 1; w < NT / 32; ++w) above_warps += sh[w];
  const uint32_t incl = suf + above_warps;  // keys in bins >= t*per
  const uint32_t above = incl - own;        // keys in bins >= (t+1)*per
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

// exclusive block scan of one value per thread; returns the block total
template <int NT = kSelThreads>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* sh, uint32_t* total) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  __syncthreads();
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  uint32_t before = 0, tot = 0;
  for (int w = 0; w < NT / 32; ++w) {
    if (w < warp) before += sh[w];
    tot += sh[w];
  }
  *total = tot;
  return before + inc - v;
}

// kItems consecutive keys of thread t (chunk-local), from global memory
__device__ __forceinline__ int load_items(const uint32_t* keys, int64_t my0, int64_t kend, uint32_t* kk) {
  const int n = (int)max((int64_t)0, min((int64_t)kItems, kend - my0));
  if (n == kItems) {
#pragma unroll
    for (int q = 0; q < kItems / 4; ++q) {
      const uint4 v = *reinterpret_cast<const uint4*>(keys + my0 + 4 * q);
      kk[4 * q] = v.x;
      kk[4 * q + 1] = v.y;
      kk[4 * q + 2] = v.z;
      kk[4 * q + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < kItems; ++j) kk[j] = j < n ? keys[my0 + j] : 0u;
  }
  return n;
}

// Multi-chunk requests (one CTA per 4096 keys): the whole select in one
// launch.  The first digit d1 of the k-th largest key follows from the score
// histogram; every CTA lists its keys in buckets >= d1 (fewer than k lie
// above d1, plus the boundary bucket) as (key, index) pairs, in index order,
// in its chunk's region of the candidate buffer.  The request's last CTA
// (atomic count after a fence) concatenates the lists in chunk order, which
// is ascending index order, takes the two remaining digits from histograms of
// the listed keys, and writes the selection -- keys above the threshold T and
// the first `need` keys equal to it -- with block scans over the lists.  No
// CTA waits on another, and no pass reads all keys twice.  The lists are
// usually a few thousand pairs; when the scores tie massively the boundary
// bucket holds most keys and the last CTA works through all of them (slower,
// still exact).
__device__ __forceinline__ int list_chunk_of(const uint32_t* coff, int n_chunks, uint32_t t) {
  // the chunk c whose list holds element t: coff[c] <= t < coff[c + 1]
  int lo = 0, hi = n_chunks - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (coff[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kSelThreads) select_list_kernel(const __grid_constant__ AttendParams P) {
  pdl_start();
  __shared__ uint32_t sh[kSelThreads];
  __shared__ uint32_t st[8];
  __shared__ uint32_t h2[kHistBins];
  __shared__ uint32_t coff[kMaxKeyCtasPerReq + 1];
  __shared__ uint2 cs[kCandCache];
  __shared__ int is_last;
  const int i = find_req(P, blockIdx.x, 1);
  const AttendReq& R = P.reqs[i];
  const int chunk = blockIdx.x - R.key_base;
  const int n_chunks = (R.n_cand + kSelectKeysPerCta - 1) / kSelectKeysPerCta;
  const int64_t k0 = (int64_t)chunk * kSelectKeysPerCta;
  int32_t* sel = P.sel + (int64_t)i * P.sel_stride;
  int32_t* tko = P.topk_out ? P.topk_out + (int64_t)(P.row0 + i) * P.top_k : nullptr;
  const int tid = threadIdx.x;
  if (chunk == 0 && tko)
    for (int j = R.k + tid; j < P.top_k; j += blockDim.x) tko[j] = -1;
  if (R.k == 0 || k0 >= R.n_cand) return;
  const int64_t kend = min((int64_t)R.n_cand, k0 + kSelectKeysPerCta);
  if (R.select_all) {
    for (int64_t e = k0 + tid; e < kend; e += blockDim.x) {
      sel[e] = (int32_t)e;
      if (tko) tko[e] = (int32_t)e;
    }
    return;
  }
  uint32_t* sync = P.sync + (int64_t)i * 4;
  uint2* cand = P.cand + (int64_t)i * P.key_stride;
  uint32_t* cnt = P.counts + ((int64_t)i * P.max_key_ctas) * 2;
  const uint32_t* keys = P.keys + (int64_t)i * P.key_stride;

  uint32_t kk[kItems];
  const int64_t my0 = k0 + (int64_t)tid * kItems;
  const int n_mine = load_items(keys, my0, kend, kk);
  find_digit(P.hist + (int64_t)i * kHistBins, kHistBins, (uint32_t)R.k, sh, &st[0], &st[1]);
  const uint32_t d1 = st[0], k1 = st[1];
  const uint32_t lo_key = d1 << 21;  // the smallest key of bucket d1
  uint32_t c = 0;
#pragma unroll
  for (int j = 0; j < kItems; ++j) c += (j < n_mine && kk[j] >= lo_key) ? 1u : 0u;
  uint32_t listed;
  uint32_t pos = block_excl_scan(c, sh, &listed);
  uint2* lst = cand + k0;  // this chunk's region: room for every key of the chunk
#pragma unroll
  for (int j = 0; j < kItems; ++j)
    if (j < n_mine && kk[j] >= lo_key) lst[pos++] = make_uint2(kk[j], (uint32_t)(my0 + j));
  if (tid == 0) {
    cnt[2 * chunk] = listed;
    __threadfence();
    is_last = atomicAdd(&sync[1], 1u) == (uint32_t)(n_chunks - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // ---- the last CTA: the lists' offsets, in chunk order ----
  uint32_t n_list;
  {
    const uint32_t len = tid < n_chunks ? __ldcg(&cnt[2 * tid]) : 0u;
    const uint32_t off = block_excl_scan(len, sh, &n_list);  // n_chunks <= kMaxKeyCtasPerReq = kSelThreads
    if (tid < n_chunks) coff[tid] = off;
  }
  __syncthreads();
  // element t of the concatenated list (every thread of the CTA may call it)
  auto at_global = [&](uint32_t t) -> uint2 {
    const int cc = list_chunk_of(coff, n_chunks, t);
    return __ldcg(&cand[(int64_t)cc * kSelectKeysPerCta + (t - coff[cc])]);
  };
  const uint32_t n_cached = min(n_list, kCandCache);
  for (uint32_t t0 = 0; t0 < n_cached; t0 += 4 * kSelThreads) {  // four loads in flight per thread
    uint2 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t t = t0 + u * kSelThreads + tid;
      if (t < n_cached) v[u] = at_global(t);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t t = t0 + u * kSelThreads + tid;
      if (t < n_cached) cs[t] = v[u];
    }
  }
  for (int b = tid; b < kHistBins; b += kSelThreads) h2[b] = 0u;
  __syncthreads();
  auto at = [&](uint32_t t) -> uint2 { return t < n_cached ? cs[t] : at_global(t); };
  // second digit: the next 11 bits of the listed keys in bucket d1
  for (uint32_t t = tid; t < n_list; t += kSelThreads) {
    const uint32_t key = at(t).x;
    if ((key >> 21) == d1) atomicAdd(&h2[(key >> 10) & 2047u], 1u);
  }
  __syncthreads();
  find_digit(h2, kHistBins, k1, sh, &st[3], &st[4]);
  const uint32_t pre = (d1 << 11) | st[3], k2 = st[4];
  for (int b = tid; b < 1024; b += kSelThreads) h2[b] = 0u;
  __syncthreads();
  // third digit: the low 10 bits of the listed keys with that prefix
  for (uint32_t t = tid; t < n_list; t += kSelThreads) {
    const uint32_t key = at(t).x;
    if ((key >> 10) == pre) atomicAdd(&h2[key & 1023u], 1u);
  }
  __syncthreads();
  find_digit(h2, 1024, k2, sh, &st[5], &st[6]);
  const uint32_t T = (pre << 10) | st[5], need = st[6];
  // ordered emission: tiles of kItems consecutive list elements per thread; a
  // selected key's position is the number of keys > T before it plus
  // min(keys == T before it, need)
  uint32_t gt_base = 0, eq_base = 0;
  for (uint32_t t0 = 0; t0 < n_list; t0 += kSelThreads * kItems) {
    const uint32_t my = t0 + (uint32_t)tid * kItems;
    uint2 v[kItems];
    uint32_t n_gt = 0, n_eq = 0;
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
      v[j] = my + j < n_list ? at(my + j) : make_uint2(0u, 0u);
      n_gt += (my + j < n_list && v[j].x > T) ? 1u : 0u;
      n_eq += (my + j < n_list && v[j].x == T) ? 1u : 0u;
    }
    uint32_t tot_gt, tot_eq;
    uint32_t gt_rank = gt_base + block_excl_scan(n_gt, sh, &tot_gt);
    uint32_t eq_rank = eq_base + block_excl_scan(n_eq, sh, &tot_eq);
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
      if (my + j >= n_list) break;
      const bool g = v[j].x > T, q = v[j].x == T;
      if (g || (q && eq_rank < need)) {
        const uint32_t p = gt_rank + min(eq_rank, need);
        const uint32_t e = v[j].y;
        if (p < (uint32_t)R.k && e < (uint32_t)R.n_cand) {
          sel[p] = (int32_t)e;
          if (tko) tko[p] = (int32_t)e;
        } else {
          flag_error(P.pool, kErrBadIndex);
        }
      }
      if (g) ++gt_rank;
      if (q) ++eq_rank;
    }
    gt_base += tot_gt;
    eq_base += tot_eq;
  }
  if (tid == 0) sync[1] = 0u;  // ready for the next call
}

// The whole select for a launch whose requests have at most
// kSelectKeysPerCta candidates each: one CTA per request keeps the keys in
// registers and takes the three radix digits of the k-th largest key from
// shared-memory histograms (the first from the score histogram), then writes
// the selection in ascending index order: keys above the threshold T and the
// first `need` keys equal to it.
__global__ void __launch_bounds__(kSelThreads) select_small_kernel(const __grid_constant__ AttendParams P) {
  pdl_start();
  __shared__ uint32_t sh[kSelThreads];
  __shared__ uint32_t st[8];
  __shared__ uint32_t h2[kHistBins];
  const int i = blockIdx.x;
  const AttendReq& R = P.reqs[i];
  int32_t* sel = P.sel + (int64_t)i * P.sel_stride;
  int32_t* tko = P.topk_out ? P.topk_out + (int64_t)(P.row0 + i) * P.top_k : nullptr;
  if (tko)
    for (int j = R.k + threadIdx.x; j < P.top_k; j += blockDim.x) tko[j] = -1;
  if (R.k == 0) return;
  if (R.select_all || R.n_cand > kSelectKeysPerCta) {  // (the host only sends requests that fit)
    for (int e = threadIdx.x; e < R.k; e += blockDim.x) {
      sel[e] = e;
      if (tko) tko[e] = e;
    }
    if (!R.select_all && threadIdx.x == 0) flag_error(P.pool, kErrBadShape);
    return;
  }
  const int tid = threadIdx.x;
  const uint32_t* keys = P.keys + (int64_t)i * P.key_stride;
  uint32_t kk[kItems];
  const int64_t my0 = (int64_t)tid * kItems;
  const int n_mine = load_items(keys, my0, R.n_cand, kk);
  // first digit: from the score histogram
  find_digit(P.hist + (int64_t)i * kHistBins, kHistBins, (uint32_t)R.k, sh, &st[0], &st[1]);
  const uint32_t d1 = st[0], k1 = st[1];
  // second digit: the next 11 bits of the keys in bucket d1
  for (int b = tid; b < kHistBins; b += kSelThreads) h2[b] = 0u;
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kItems; ++j)
    if (j < n_mine && (kk[j] >> 21) == d1) atomicAdd(&h2[(kk[j] >> 10) & 2047u], 1u);
  __syncthreads();
  find_digit(h2, kHistBins, k1, sh, &st[2], &st[3]);
  const uint32_t d2 = st[2], k2 = st[3];
  const uint32_t pre = (d1 << 11) | d2;
  // third digit: the low 10 bits of the keys with that prefix
  for (int b = tid; b < 1024; b += kSelThreads) h2[b] = 0u;
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kItems; ++j)
    if (j < n_mine && (kk[j] >> 10) == pre) atomicAdd(&h2[kk[j] & 1023u], 1u);
  __syncthreads();
  find_digit(h2, 1024, k2, sh, &st[4], &st[5]);
  const uint32_t T = (pre << 10) | st[4], need = st[5];
  uint32_t n_gt = 0, n_eq = 0;
#pragma unroll
  for (int j = 0; j < kItems; ++j) {
    n_gt += j < n_mine && kk[j] > T;
    n_eq += j < n_mine && kk[j] == T;
  }
  uint32_t tot;
  uint32_t gt_rank = block_excl_scan(n_gt, sh, &tot);
  uint32_t eq_rank = block_excl_scan(n_eq, sh, &tot);
#pragma unroll
  for (int j = 0; j < kItems; ++j) {
    if (j >= n_mine) break;
    const int64_t e = my0 + j;
    if (kk[j] > T || (kk[j] == T && eq_rank < need)) {
      const uint32_t pos = gt_rank + min(eq_rank, need);
      if (pos < (uint32_t)R.k) {
        sel[pos] = (int32_t)e;
        if (tko) tko[pos] = (int32_t)e;
      } else {
        flag_error(P.pool, kErrBadIndex);
      }
    }
    if (kk[j] > T) ++gt_rank;
    if (kk[j] == T) ++eq_rank;
  }
}

// ---------------------------------------------------------------------------
// Cluster select: one thread-block cluster of C CTAs (16, or 8 where a
// 16-CTA cluster cannot be resident) per request.  CTA r of the cluster
// holds keys [r*chunk, (r+1)*chunk) of its request in shared memory.  The
// first radix digit d1 of the k-th largest key comes from the score
// histogram; one pass over the keys lists those in buckets >= d1 (fewer than
// k above d1, plus the boundary bucket) and histograms the boundary bucket's
// next digit; the other two digits come from histograms summed across the
// cluster through distributed shared memory, and the listed keys alone give
// the counts and, in ascending index order, the selection, placed by the
// cluster-wide exclusive prefix of (keys > T, keys == T).  One launch, no
// global atomics, no CTA waiting on a counter.
// Every exit before the first cluster barrier depends on the request only, so
// either all CTAs of a cluster reach each barrier or none does.
// ---------------------------------------------------------------------------
constexpr int kSelCThreads = 512;
constexpr int kSelClusterMax = 16;

// Sum of the cluster's local histograms h (nb bins, nb a multiple of the
// cluster size) into hred of every CTA: CTA r first sums the slice
// [r*nb/C, (r+1)*nb/C) over the cluster into hpart, then every CTA gathers
// the C slices.  Called by every thread of every CTA of the cluster.
__device__ void cluster_hist_sum(cg::cluster_group& cl, uint32_t* h, uint32_t* hpart, uint32_t* hred, int nb) {
  const int C = (int)cl.num_blocks();
  const int r = (int)cl.block_rank();
  const int per = nb / C;
  cl.sync();  // every local histogram is complete
  for (int t = threadIdx.x; t < per; t += blockDim.x) {
    uint32_t v = 0;
#pragma unroll 4
    for (int c = 0; c < C; ++c) v += cl.map_shared_rank(h, c)[r * per + t];
    hpart[t] = v;
  }
  cl.sync();  // every slice is summed, and no CTA reads a peer's h any more
  for (int b = threadIdx.x; b < nb; b += blockDim.x) hred[b] = cl.map_shared_rank(hpart, b / per)[b % per];
  __syncthreads();
}

__global__ void __launch_bounds__(kSelCThreads) select_cluster_kernel(const __grid_constant__ AttendParams P,
                                                                      int cap_keys) {
  pdl_start();
  extern __shared__ __align__(16) uint32_t ks[];  // this CTA's keys [cap_keys], then 16-bit list slots [cap_keys]
  __shared__ __align__(16) uint32_t h[kHistBins];
  __shared__ __align__(16) uint32_t hred[kHistBins];
  __shared__ uint32_t hpart[kHistBins / 8];
  __shared__ uint32_t sh[32];
  __shared__ uint32_t st[8];
  __shared__ uint32_t wgt[kSelCThreads / 32], weq[kSelCThreads / 32];
  __shared__ uint32_t tot[2];
  cg::cluster_group cl = cg::this_cluster();
  const int C = (int)cl.num_blocks();
  const int r = (int)cl.block_rank();
  const int i = (int)(blockIdx.x / C);
  const AttendReq& R = P.reqs[i];
  int32_t* sel = P.sel + (int64_t)i * P.sel_stride;
  int32_t* tko = P.topk_out ? P.topk_out + (int64_t)(P.row0 + i) * P.top_k : nullptr;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gtid = r * kSelCThreads + tid, gstride = C * kSelCThreads;
  if (tko)
    for (int j = R.k + gtid; j < P.top_k; j += gstride) tko[j] = -1;
  if (R.k == 0) return;
  const int64_t chunk = (((int64_t)R.n_cand + C - 1) / C + 3) & ~(int64_t)3;  // a multiple of 4 keys
  if (R.select_all || chunk > cap_keys) {  // (the host sends only requests that fit)
    for (int e = gtid; e < R.k; e += gstride) {
      sel[e] = e;
      if (tko) tko[e] = e;
    }
    if (!R.select_all && gtid == 0) flag_error(P.pool, kErrBadShape);
    return;
  }
  const int64_t c0 = (int64_t)r * chunk;
  const int nk = (int)max((int64_t)0, min((int64_t)R.n_cand, c0 + chunk) - c0);
  // keys and the score histogram -> shared memory, eight 16-byte loads in
  // flight per thread (c0 is a multiple of 4; key rows are 16-byte aligned)
  const uint4* keys4 = reinterpret_cast<const uint4*>(P.keys + (int64_t)i * P.key_stride + c0);
  const uint4* hist4 = reinterpret_cast<const uint4*>(P.hist + (int64_t)i * kHistBins);
  uint4* ks4 = reinterpret_cast<uint4*>(ks);
  const int n4 = nk >> 2;
  constexpr int kHist4 = kHistBins / 4;
  {
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int q = j * kSelCThreads + tid;
      if (q < kHist4) v[j] = hist4[q];
      else if (q - kHist4 < n4) v[j] = keys4[q - kHist4];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int q = j * kSelCThreads + tid;
      if (q < kHist4) reinterpret_cast<uint4*>(hred)[q] = v[j];
      else if (q - kHist4 < n4) ks4[q - kHist4] = v[j];
    }
  }
  for (int q0 = 8 * kSelCThreads - kHist4; q0 < n4; q0 += 8 * kSelCThreads) {
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int q = q0 + j * kSelCThreads + tid;
      if (q < n4) v[j] = keys4[q];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int q = q0 + j * kSelCThreads + tid;
      if (q < n4) ks4[q] = v[j];
    }
  }
  for (int e = (n4 << 2) + tid; e < nk; e += kSelCThreads) ks[e] = P.keys[(int64_t)i * P.key_stride + c0 + e];
  for (int b = tid; b < kHistBins; b += kSelCThreads) h[b] = 0u;
  __syncthreads();
  // first digit: from the score histogram (the same in every CTA)
  find_digit<kSelCThreads>(hred, kHistBins, (uint32_t)R.k, sh, &st[0], &st[1]);
  const uint32_t d1 = st[0], k1 = st[1];
  // one pass over the keys: each warp owns a run of consecutive keys and
  // lists, in index order, the local indices of its keys in buckets >= d1
  // (fewer than k of them lie above d1: the list is short); the keys in
  // bucket d1 also count into the histogram of their next 11 bits
  constexpr int kWarps = kSelCThreads / 32;
  const int seg = ((nk + kWarps - 1) / kWarps + 127) & ~127;
  const int w0 = min(nk, warp * seg), w1 = min(nk, w0 + seg);
  uint16_t* lst = reinterpret_cast<uint16_t*>(ks + cap_keys) + w0;
  uint32_t n_list = 0;
  for (int e0 = w0; e0 < w1; e0 += 128) {
    const int e = e0 + lane * 4;
    uint32_t kv[4];
    if (e + 3 < w1) {
      const uint4 v = ks4[e >> 2];
      kv[0] = v.x;
      kv[1] = v.y;
      kv[2] = v.z;
      kv[3] = v.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) kv[j] = e + j < w1 ? ks[e + j] : 0u;
    }
    bool fl[4];
    uint32_t c = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool valid = e + j < w1;
      const uint32_t b = kv[j] >> 21;
      if (valid && b == d1) atomicAdd(&h[(kv[j] >> 10) & 2047u], 1u);
      fl[j] = valid && b >= d1;
      c += fl[j] ? 1u : 0u;
    }
    uint32_t inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += u;
    }
    uint32_t pos = n_list + inc - c;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (fl[j]) lst[pos++] = (uint16_t)(e + j);
    n_list += __shfl_sync(0xffffffffu, inc, 31);
  }
  cluster_hist_sum(cl, h, hpart, hred, kHistBins);
  find_digit<kSelCThreads>(hred, kHistBins, k1, sh, &st[2], &st[3]);
  const uint32_t pre = (d1 << 11) | st[2], k2 = st[3];
  // third digit: the low 10 bits of the listed keys with that prefix
  for (int b = tid; b < 1024; b += kSelCThreads) h[b] = 0u;
  __syncthreads();
  for (uint32_t t = lane; t < n_list; t += 32) {
    const uint32_t key = ks[lst[t]];
    if ((key >> 10) == pre) atomicAdd(&h[key & 1023u], 1u);
  }
  cluster_hist_sum(cl, h, hpart, hred, 1024);
  find_digit<kSelCThreads>(hred, 1024, k2, sh, &st[4], &st[5]);
  const uint32_t T = (pre << 10) | st[4], need = st[5];
  // each warp's counts of (> T, == T): all of them are on its list
  uint32_t n_gt = 0, n_eq = 0;
  for (uint32_t t = lane; t < n_list; t += 32) {
    const uint32_t key = ks[lst[t]];
    n_gt += key > T ? 1u : 0u;
    n_eq += key == T ? 1u : 0u;
  }
  n_gt = __reduce_add_sync(0xffffffffu, n_gt);
  n_eq = __reduce_add_sync(0xffffffffu, n_eq);
  if (lane == 0) {
    wgt[warp] = n_gt;
    weq[warp] = n_eq;
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t a = 0, b = 0;
    for (int w = 0; w < kWarps; ++w) {
      a += wgt[w];
      b += weq[w];
    }
    tot[0] = a;
    tot[1] = b;
  }
  cl.sync();  // every CTA's totals are visible to the cluster
  if (warp == 0) {  // this CTA's exclusive prefix over the lower ranks
    uint32_t a = 0, b = 0;
    if (lane < r) {
      const uint32_t* t = cl.map_shared_rank(tot, lane);
      a = t[0];
      b = t[1];
    }
    a = __reduce_add_sync(0xffffffffu, a);
    b = __reduce_add_sync(0xffffffffu, b);
    if (lane == 0) {
      st[6] = a;
      st[7] = b;
    }
  }
  __syncthreads();
  uint32_t gt_rank = st[6], eq_rank = st[7];
  for (int w = 0; w < warp; ++w) {
    gt_rank += wgt[w];
    eq_rank += weq[w];
  }
  // ordered emission over the list: a selected key's position is the number
  // of keys > T before it plus min(keys == T before it, need)
  const uint32_t lt = (1u << lane) - 1u;
  for (uint32_t t0 = 0; t0 < n_list; t0 += 32) {
    const uint32_t t = t0 + lane;
    const uint32_t e = t < n_list ? lst[t] : 0u;
    const uint32_t key = t < n_list ? ks[e] : 0u;
    const bool g = t < n_list && key > T, q = t < n_list && key == T;
    const uint32_t gm = __ballot_sync(0xffffffffu, g), qm = __ballot_sync(0xffffffffu, q);
    const uint32_t eqb = eq_rank + __popc(qm & lt);
    if (g || (q && eqb < need)) {
      const uint32_t pos = gt_rank + __popc(gm & lt) + min(eqb, need);
      if (pos < (uint32_t)R.k) {
        sel[pos] = (int32_t)(c0 + e);
        if (tko) tko[pos] = (int32_t)(c0 + e);
      } else {
        flag_error(P.pool, kErrBadIndex);
      }
    }
    gt_rank += __popc(gm);
    eq_rank += __popc(qm);
  }
  cl.sync();  // no CTA leaves while a peer may still read its totals
}

}  // namespace

namespace {

// Cluster size and shared-memory key capacity of the cluster select on the
// current device: 16 CTAs per cluster where a 16-CTA cluster with the largest
// key buffer can be resident, else 8, else none (the two-pass select runs).
struct ClusterShape {
  int ctas = 0;
  int cap_keys = 0;
};
constexpr int kClusterKeyBytes = 180 * 1024;  // 6 bytes per key: the key and a list slot
constexpr int kShapeDevices = 64;

ClusterShape cluster_shape() {
  static std::mutex mu;
  static bool done[kShapeDevices];
  static ClusterShape shape[kShapeDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kShapeDevices) return {};
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    done[dev] = true;
    ClusterShape c;
    if (cudaFuncSetAttribute(select_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kClusterKeyBytes) ==
            cudaSuccess &&
        cudaFuncSetAttribute(select_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess) {
      for (int n : {kSelClusterMax, 8}) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(n);
        cfg.blockDim = dim3(kSelCThreads);
        cfg.dynamicSmemBytes = kClusterKeyBytes;
        cudaLaunchAttribute a[1];
        a[0].id = cudaLaunchAttributeClusterDimension;
        a[0].val.clusterDim.x = n;
        a[0].val.clusterDim.y = 1;
        a[0].val.clusterDim.z = 1;
        cfg.attrs = a;
        cfg.numAttrs = 1;
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, select_cluster_kernel, &cfg) == cudaSuccess && active > 0) {
          c.ctas = n;
          c.cap_keys = std::min(kClusterKeyBytes / 6, 65535);  // list slots hold 16-bit indices
          break;
        }
      }
    }
    (void)cudaGetLastError();  // a refused attribute or query leaves the two-pass select
    shape[dev] = c;
  }
  return shape[dev];
}

}  // namespace

int launch_select(const AttendParams& p, void* stream, int* n_kernels, bool alone) {
  if (p.total_key_ctas <= 0) return 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // one select CTA per request (at most kSelectKeysPerCta candidates each):
  // the whole select in one pass
  if (p.total_key_ctas == p.n) {
    launch_kernel(true, select_small_kernel, dim3(p.n), dim3(kSelThreads), 0, s, p);
    *n_kernels += 1;
    return (int)cudaGetLastError();
  }
  // requests of more than one cluster's worth of 4096-key chunks, when the
  // select has the GPU to itself: one cluster per request, its keys in the
  // CTAs' shared memory
  int64_t max_cand = 0;
  for (int i = 0; i < p.n; ++i)
    if (!p.reqs[i].select_all && p.reqs[i].k > 0) max_cand = std::max<int64_t>(max_cand, p.reqs[i].n_cand);
  const ClusterShape cs = alone ? cluster_shape() : ClusterShape{};
  if (cs.ctas > 0 && max_cand > (int64_t)cs.ctas * kSelectKeysPerCta) {
    const int64_t chunk = ((max_cand + cs.ctas - 1) / cs.ctas + 3) & ~(int64_t)3;
    if (chunk <= cs.cap_keys) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(p.n * cs.ctas));
      cfg.blockDim = dim3(kSelCThreads);
      cfg.dynamicSmemBytes = (size_t)chunk * 6;
      cfg.stream = s;
      cudaLaunchAttribute a[1];
      a[0].id = cudaLaunchAttributeClusterDimension;
      a[0].val.clusterDim.x = (unsigned)cs.ctas;
      a[0].val.clusterDim.y = 1;
      a[0].val.clusterDim.z = 1;
      cfg.attrs = a;
      cfg.numAttrs = 1;
      cudaLaunchKernelEx(&cfg, select_cluster_kernel, p, (int)chunk);
      *n_kernels += 1;
      return (int)cudaGetLastError();
    }
  }
  // every other shape: one CTA per 4096-key chunk, the request's last CTA
  // finishes it (launched without programmatic dependent launch: its
  // early-started CTAs would hold SM room that the attention beside it needs)
  launch_kernel(false, select_list_kernel, dim3(p.total_key_ctas), dim3(kSelThreads), 0, s, p);
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
  pdl_start();
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
  uint32_t* gh = P.hist + (int64_t)i * kHistBins;
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
  if ((!d_scores && n_cols > 0) || !d_topk_out || n_rows > kMaxAttendReqs) return KVPOOL_ERR_INVALID_ARG;
  // scratch plan: [error word | hist | sync | thresholds | counts | selected | keys | candidates]
  const int64_t chunks = std::max<int64_t>(1, ((int64_t)n_cols + kSelectKeysPerCta - 1) / kSelectKeysPerCta);
  if (chunks > kMaxKeyCtasPerReq) return KVPOOL_ERR_INVALID_ARG;
  auto up = [](int64_t x) { return (x + 255) / 256 * 256; };
  const int64_t off_hist = 256;
  const int64_t off_sync = off_hist + up(4LL * n_rows * kHistBins);
  const int64_t off_thr = off_sync + up(16LL * n_rows);
  const int64_t off_counts = off_thr + up(8LL * n_rows);
  const int64_t off_sel = off_counts + up(8LL * n_rows * chunks);
  const int64_t stride = ((int64_t)n_cols + 3) / 4 * 4;  // 16-byte aligned key rows
  const int64_t off_keys = off_sel + up(4LL * n_rows * top_k);
  const int64_t off_cand = off_keys + up(4LL * n_rows * stride);
  const int64_t need = off_cand + up(8LL * n_rows * stride);
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
  // the error word, the histograms and the sync counters must start at zero;
  // everything else is written before it is read
  if (cudaMemsetAsync(base, 0, (size_t)off_thr, s) != cudaSuccess) return KVPOOL_ERR_CUDA;

  AttendParams* P = new (std::nothrow) AttendParams();
  if (!P) return KVPOOL_ERR_INVALID_ARG;
  P->pool.arena = base;
  P->pool.err = 0;
  P->topk_out = d_topk_out;
  P->top_k = top_k;
  P->n = n_rows;
  P->row0 = 0;
  P->keys = reinterpret_cast<uint32_t*>(base + off_keys);
  P->key_stride = stride;
  P->hist = reinterpret_cast<uint32_t*>(base + off_hist);
  P->counts = reinterpret_cast<uint32_t*>(base + off_counts);
  P->max_key_ctas = (int32_t)chunks;
  P->sel = reinterpret_cast<int32_t*>(base + off_sel);
  P->sel_stride = top_k;
  P->cand = reinterpret_cast<uint2*>(base + off_cand);
  P->sync = reinterpret_cast<uint32_t*>(base + off_sync);
  P->thr = reinterpret_cast<uint32_t*>(base + off_thr);
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
    launch_kernel(false, static_keys_kernel, dim3(P->total_key_ctas), dim3(kSelThreads), 0, s, *P, d_scores, (int64_t)n_cols);
    rc = (int)cudaGetLastError();
  }
  int nk = 0;
  if (rc == 0) rc = launch_select(*P, stream, &nk, true);
  delete P;
  return rc == 0 ? KVPOOL_OK : KVPOOL_ERR_CUDA;
}

extern "C" int kvpool_topk_static_check(void* stream, uint32_t* h_flags) {
  using namespace kvp;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVPOOL_ERR_CUDA;
  uint32_t word = 0;
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    base = g_scratch_addr[dev];
  }
  if (base) {  // no call on this device yet: nothing can have been flagged
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return KVPOOL_ERR_CUDA;
    if (cudaMemcpy(&word, base, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return KVPOOL_ERR_CUDA;
  }
  if (h_flags) *h_flags = word;
  return word == 0 ? KVPOOL_OK : KVPOOL_ERR_DEVICE_CHECK;
}

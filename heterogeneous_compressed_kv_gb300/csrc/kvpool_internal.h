// kvpool_internal.h -- shared definitions of the kvpool host runtime and its
// CUDA kernels (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>

#include "kvpool.h"

namespace kvp {

constexpr int kMaxLayers = 16;
constexpr size_t kMaxDynSmem = 232448;  // dynamic shared memory one CTA may opt into (227 KiB)
constexpr int kHistBins = 2048;          // radix digit of the top-k select (11 bits)
constexpr int kMaxKeyCtasPerReq = 256;   // select chunks per request (1M candidates)
constexpr int kSelectKeysPerCta = 4096;  // keys handled by one select CTA
constexpr int kMaxAppendUnits = 512;     // units per append launch
constexpr int kMaxAttendReqs = 256;      // requests per attend-side launch
constexpr int kAttendThreadsMax = 288;   // 8 consumer warps (16 dims each) + 1 producer warp

// device error word flags
enum : uint32_t {
  kErrWaitTimeout = 1u << 0,  // an mbarrier wait passed its time limit
  kErrBadBlock = 1u << 1,     // block id out of range
  kErrBadIndex = 1u << 2,     // entry / slot index out of range
  kErrBadShape = 1u << 3,     // launch shape inconsistent with the pool
};

// Byte offsets of one layer inside the arena (see kvpool.h for the layout).
struct LayerDesc {
  int32_t kind;
  int32_t has_csa, has_hca;
  // one plane per part, indexed by block id (ids >= staging_base are the
  // requests' private staging blocks): CSA entries, indexer keys (+ fp8
  // scales at idx_scale_off inside a block's part), HCA entry
  int64_t csa_pool, csa_stride;
  int64_t idx_pool, idx_stride, idx_scale_off;
  int64_t idx_run;  // bytes of one run of csa_per_block keys (+ scales); a block part holds idx_runs runs
  int64_t hca_pool, hca_stride;
  int64_t ring, ring_req_bytes;
  int64_t acc, acc_req_bytes;  // acc: CSA [2HD] f32, idx [XD] f32, HCA [2HD] f32
  int64_t alpha_csa, alpha_hca, alpha_idx;  // f32 [H][m], [H][m'], [Ih][m]
  int64_t csa_host_off;  // HiSparse: this layer's CSA entries inside a host slot
};

// Everything a kernel needs to know about the pool (passed by value).
struct PoolDesc {
  uint8_t* arena;
  int32_t m, m_prime, n_win;
  int32_t heads, head_dim, idx_heads, idx_dim, HD, XD;
  int32_t in_dtype, cache_dtype, vs, isz;  // cache value bytes, input value bytes
  int32_t idx_dtype;                       // indexer entries: cache_dtype or KVPOOL_FP4_E2M1
  int32_t csa_per_block, idx_chunks;       // idx_chunks: 16-B chunks per indexer key
  int32_t idx_per_token, idx_runs;         // per-token keys: m runs of csa_per_block keys per block, else 1 run
  int64_t entry_bytes, idx_entry_bytes;
  int32_t max_blocks, max_requests, max_bpr, staging_base;
  int64_t table;  // int32 [max_requests][max_bpr]
  int64_t err;    // uint32
  // HiSparse: CSA entries of a sealed block at its location (csa_loc[id]:
  // >= 0 a CSA plane slot, < 0 host slot -1-loc); without it the location is
  // the id.  Staging CSA slots start at csa_staging_base.
  int32_t hisparse, csa_staging_base;
  int64_t csa_loc, last_used;  // int32 / uint32 [max_blocks]
  uint8_t* host_pool;          // device alias of the host slots (or null)
  int64_t host_slot_bytes, host_pool_bytes;
};

// ---- append ---------------------------------------------------------------
// One (request, block segment) touched by an append call: positions
// seg*m' + t for t in [t0, t1).
// A unit's work: all of it, or -- units of many tokens in a launch too small
// to fill the GPU -- the HCA chain over all its tokens (plus the seal copies)
// in one CTA and the CSA / indexer chains and window writes over a range of
// whole CSA groups in each of several others.
enum : int16_t { kUnitAll = 0, kUnitHca = 1, kUnitCsa = 2 };

struct AppendUnit {
  int32_t slot;      // request slot
  int32_t seg;       // block index within the request
  int16_t t0, t1;    // token range inside the segment
  int16_t ring_from; // first t written to the window (t1 if none)
  int16_t role;      // kUnitAll, or one part of a unit split over CTAs (kUnitHca / kUnitCsa)
  int32_t in_row;    // input row of the token at t0
  int32_t block_id;  // id the segment seals into in this call, or -1
  int32_t csa_slot;  // CSA plane slot of that block (its id without HiSparse)
};

struct AppendParams {
  PoolDesc pool;
  LayerDesc layers[kMaxLayers];
  const void* k;
  const void* v;
  const void* idx_k;
  int64_t rows;  // T: rows per layer in the inputs
  int32_t n_units;
  int32_t n_slices;  // CTAs that split one unit's 2*H*d values
  int32_t copy_slices;  // further CTAs per unit that copy a sealing block's staged entries (0: none seal)
  uint32_t epoch;    // HiSparse activity stamp of the blocks sealed here
  int32_t staged;        // tokens arrive through shared-memory stages (long units)
  int32_t stage_tokens;  // tokens per stage of the staged path
  AppendUnit units[kMaxAppendUnits];
};

// share_prefix: window fill of dst + table row copy (src < 0: window only,
// for a prefix image restored without its window)
struct ShareParams {
  PoolDesc pool;
  LayerDesc layers[kMaxLayers];
  const void* win_k;
  const void* win_v;
  int32_t dst, src, n_blocks, w;
  int64_t n_tokens;
};

// ---- block copies: prefix images, HiSparse offload and fetch ------------------
// One contiguous copy: a run of adjacent block parts, a piece of a window
// ring, between the arena, a host image and the host slots.  The bytes of
// each mask_row-long row from mask_valid on are written as zeros (the
// padding after the indexer scales, on export); mask_row 0 means no mask.
struct ImageSeg {
  uint64_t src, dst;  // device addresses (a host buffer's device alias)
  int64_t bytes;      // multiple of 16
  int32_t mask_row, mask_valid;
  int32_t src_host;   // the source is host memory
  int32_t pad;
};
// bookkeeping writes for blocks id0 + i, i < cnt: table[dst][b0 + i] = id0 + i
// (b0 >= 0), csa_loc[id0 + i] = loc0 + i * loc_dir (loc_dir != 0), and
// last_used[id0 + i] = epoch (stamp)
struct ImageRun {
  int32_t b0, id0, cnt, loc0;
  int16_t loc_dir, stamp;
};
constexpr int kMaxImageSegs = 64;
constexpr int kMaxImageRuns = 64;
constexpr int kImagePieceBytes = 16384;  // bytes one CTA copies per step
constexpr int kImageCtasPerSm = 8;       // resident copy CTAs per SM (256 threads each)

struct ImageParams {
  PoolDesc pool;
  int32_t dst;         // request slot whose table row the runs fill
  uint32_t epoch;      // activity stamp of the runs' blocks
  int32_t n_sms;       // multiprocessors of the device (sizes the grid)
  int32_t pad_;
  int32_t n_segs, n_runs;
  int64_t n_pieces;    // pieces of kImagePieceBytes over all segments
  int64_t piece_base[kMaxImageSegs + 1];  // first piece of each segment
  ImageSeg segs[kMaxImageSegs];
  ImageRun runs[kMaxImageRuns];
};

// ---- decode attention -----------------------------------------------------
struct AttendReq {
  int32_t slot;
  int32_t n_sealed;   // sealed blocks of the request
  int32_t n_cand;     // CSA entries N_c (0 for layers without CSA)
  int32_t k;          // min(top_k, N_c)
  int32_t n_hca;      // HCA entries attended (0 for layers without HCA)
  int32_t w;          // window tokens
  int64_t length;     // L
  int32_t select_all; // k == N_c: every CSA entry is selected
  int32_t score_base; // first score CTA of this request
  int32_t key_base;   // first select CTA of this request
  // attention: part 0 = [HCA entries | window] (needs no top-k), part 1 =
  // [selected CSA entries]; each part is split into chunks of its split_len
  int32_t split_len0, split_len1;  // sources per split of each part
  int32_t n_split0, n_split1;
  int32_t cta_base0, cta_base1;  // first attention CTA (split) of this request in each part's launch
  int32_t part_base;             // first partial slot; part 1 follows part 0
};

struct AttendParams {
  PoolDesc pool;
  LayerDesc layer;
  const void* q;
  const void* q_idx;
  float* out;
  int32_t* topk_out;
  int32_t top_k;
  uint32_t epoch;            // HiSparse activity stamp of this call
  int32_t n;                 // requests in this launch
  int32_t row0;              // first row of q / out for this launch
  int32_t total_score_ctas, total_key_ctas;
  int32_t total_ctas0, total_ctas1;  // attention CTAs (= splits) of part 0 and part 1
  int32_t segs_per_cta;      // block segments scored by one score CTA
  int32_t src_lo, src_hi;    // attention sources [lo, hi) of the virtual list this launch covers
  // scratch (device pointers)
  uint32_t* keys;            // [rows][key_stride] orderable score keys
  int64_t key_stride;        // max_cand
  uint32_t* hist;            // [rows][kHistBins] first radix digit histogram
  uint32_t* counts;          // [rows][max_key_ctas][2] (keys > T, keys == T) per select chunk
  int32_t max_key_ctas;
  uint2* cand;               // [rows][key_stride] (key, index) of the boundary bucket
  uint32_t* sync;            // [rows][4]: candidates, select CTAs done, pad, pad
  uint32_t* thr;             // [rows][2] (T, keys == T taken)
  int32_t* sel;              // [rows][sel_stride]
  int32_t sel_stride;
  float* part_o;             // [max_splits][HD]
  float* part_ml;            // [max_splits][H][2]
  AttendReq reqs[kMaxAttendReqs];
};

// ---- launchers (implemented in the .cu files; return cudaError_t as int) --
// Each launcher adds the number of kernels it launched to *n_kernels.
int launch_append(const AppendParams& p, int n_layers, void* stream, int* n_kernels);
int append_slices(const PoolDesc& pd);         // CTAs per unit, direct token loads
int append_slices_staged(const PoolDesc& pd);  // CTAs per unit, staged token rows
int append_stage_tokens(const PoolDesc& pd, int n_slices);
int launch_share(const ShareParams& p, int n_layers, void* stream, int* n_kernels);
int launch_image(const ImageParams& p, void* stream, int* n_kernels);
int launch_wait_selftest(const PoolDesc& pd, void* stream);
int launch_score(const AttendParams& p, void* stream, int* n_kernels);
// the score kernel's shared-memory plan: one block's indexer bytes per slot,
// slots per warp, the slots' offset, warps per CTA and the dynamic bytes
int score_stage_plan(const PoolDesc& pd, int* stage_bytes, int* ring, int* stage_off, int* warps, size_t* smem);
size_t attend_smem_bytes(const PoolDesc& pd);
// alone: nothing else runs on the GPU beside the select, so it may take one
// thread-block cluster per large request (a cluster waits for 16 SMs with room
// at once, which attention CTAs running beside it would hold)
int launch_select(const AttendParams& p, void* stream, int* n_kernels, bool alone);
int launch_attend(const AttendParams& p, int part, int ctas, void* stream, int* n_kernels);
int launch_combine(const AttendParams& p, void* stream, int* n_kernels);

}  // namespace kvp

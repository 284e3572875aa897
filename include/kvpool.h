/*
 * kvpool.h -- C ABI of a GPU-resident two-pool KV cache (DeepSeek-V4 style:
 * a Classical/Block pool of immutable, lcm-aligned compressed blocks plus a
 * per-request State pool), built for one GB300 (sm_103a).
 *
 * What the library computes, per decode step and attention layer, follows
 * these design pages (cited by title and section):
 *   [P1] "Why does V4 split pools? How do block alignment and the tail buffer
 *        work together" -- s1.1 (Classical holds only full, immutable
 *        compressed entries; State holds the tail and the SWA window), s1.2
 *        (CSA: every m = 4 tokens -> 1 entry, read top-k sparse; HCA: every
 *        m' = 128 tokens -> 1 entry, read densely), s2.2 (block = lcm(m, m')
 *        = 128 tokens = 32 CSA + 1 HCA entries; L = 128q + r), s3.1 (tails of
 *        at most 3 / 127 tokens), s4 (one decode step: token into the tail,
 *        compress when a group fills, SWA slides, attention reads Classical
 *        entries sparsely/densely plus the exact local window).
 *   [P2] "V4 KV Layout: Classical + State dual pool" -- Classical KV cache
 *        and State cache tables; the lightning indexer's light K vectors.
 *   [P3] "Ch 12 Inference framework: heterogeneous KV scheduling" -- s2.1
 *        (one State block per request, freed whole), s2.2 (Block cache shared
 *        across requests by refcount), Figure 12-1 (a block id spans all
 *        layers; each block holds CSA indexer KV, CSA main KV and HCA KV).
 *   [P4] "V4 disk prefix cache" -- Zero SWA caching: on a prefix hit only
 *        the compressed blocks are reused and the window is recomputed.
 * The pages give no compressor, score or attention formula.  This library
 * fixes them as follows (the same definitions as the CPU oracle):
 *   compressor   entry[h][j] = fp32 chain acc = fma(alpha[h][i], x_i[h][j], acc)
 *                over the group's tokens i = 0..m-1 (m' for HCA) from +0,
 *                alpha = softmax of the caller's gate logits (double, rounded
 *                to fp32); K and V share alpha; indexer entries use their own
 *                gates per indexer head;
 *   score        s_e = fp32 chain fma(q_idx[v], key_e[v], acc) over the flat
 *                indexer (head, dim) order from +0, times the entry scale
 *                (fp8 cache);
 *   top-k        k = min(top_k, number of CSA entries), by (score desc,
 *                index asc), -0 == +0;
 *   attention    one softmax with scale 1/sqrt(head_dim) over [selected CSA
 *                entries, every HCA entry, the SWA window] (no masking; the
 *                window includes the token appended in this step), fp32.
 *
 * Conventions (all entry points):
 *   - Device pointers ("d_") are read/written in stream order on `stream`
 *     (a cudaStream_t; NULL = the legacy default stream).  Host pointers
 *     ("h_") are read before the call returns.
 *   - The caller owns the device arena (kvpool_required_bytes bytes, 256-B
 *     aligned), every input and every output.  The library owns the layout
 *     inside the arena and all host metadata.
 *   - Every call validates its whole batch and reserves blocks on the host
 *     before launching anything; a call that returns an error has changed
 *     nothing.  No call synchronizes with the device except
 *     kvpool_check_device and kvpool_profile_read.
 *   - A pool is not thread safe; drive it from one host thread and one
 *     stream.  No exception crosses this ABI.
 */
#ifndef KVPOOL_H
#define KVPOOL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ---- */
enum {
  KVPOOL_OK = 0,
  KVPOOL_ERR_INVALID_ARG = -1,     /* bad size, pointer, dtype or combination */
  KVPOOL_ERR_OUT_OF_BLOCKS = -2,   /* the Classical pool has too few free blocks */
  KVPOOL_ERR_OUT_OF_REQUESTS = -3, /* every request slot is in use */
  KVPOOL_ERR_BAD_REQUEST = -4,     /* request id out of range or not allocated */
  KVPOOL_ERR_NOT_SHAREABLE = -5,   /* prefix not whole sealed blocks, or dst not fresh */
  KVPOOL_ERR_CUDA = -6,            /* a CUDA runtime call failed (see kvpool_last_error) */
  KVPOOL_ERR_DEVICE_CHECK = -7,    /* a kernel flagged a bounds or wait-limit violation */
  KVPOOL_ERR_CAPACITY = -8,        /* a request would exceed max_blocks_per_request */
  KVPOOL_ERR_BAD_IMAGE = -9,       /* a prefix image is malformed or from another config */
};

/* ---- element types ---- */
enum {
  KVPOOL_F32 = 0,
  KVPOOL_BF16 = 1,
  KVPOOL_FP8_E4M3 = 2, /* cache only: e4m3 codes + one bf16 scale per K half, V half, indexer entry */
  KVPOOL_FP4_E2M1 = 3, /* indexer entries only (kvpool_config.idx_fp4): two e2m1 codes per byte (element
                          2j in the low nibble) + one bf16 scale = bf16(amax / 6), 1 if that is 0 */
};

/* ---- layer kinds (Figure 12-1 lists SWA, CSA and HCA layers) ---- */
enum {
  KVPOOL_SWA_ONLY = 0, /* window only */
  KVPOOL_CSA = 1,      /* CSA top-k + window */
  KVPOOL_HCA = 2,      /* HCA dense + window */
  KVPOOL_CSA_HCA = 3,  /* all three sources */
};

enum { KVPOOL_FLAG_NO_DEVICE = 1u }; /* bookkeeping only: no arena, no launches (host tests) */

typedef struct kvpool_config {
  int32_t m;          /* CSA group (4); must divide m_prime so lcm(m, m') = m' */
  int32_t m_prime;    /* HCA group (128) = block length in tokens */
  int32_t n_win;      /* SWA window in tokens; a positive multiple of m_prime */
  int32_t heads;      /* attention heads (queries and cache alike) */
  int32_t head_dim;   /* 64 or 128 */
  int32_t idx_heads;  /* lightning-indexer heads */
  int32_t idx_dim;    /* lightning-indexer head dim */
  int32_t in_dtype;   /* KVPOOL_F32 or KVPOOL_BF16: new K/V/indexer keys and queries */
  int32_t cache_dtype;/* KVPOOL_F32, KVPOOL_BF16 or KVPOOL_FP8_E4M3 */
  int32_t n_layers;
  const int32_t* layer_kinds;     /* [n_layers] */
  int32_t max_requests;           /* request slots (State blocks) */
  int32_t max_blocks;             /* Classical blocks (ids 0 .. max_blocks-1) */
  int32_t max_blocks_per_request; /* block-table row length */
  int32_t max_batch;              /* most requests in one append or decode_attend call */
  int32_t max_top_k;              /* largest top_k a decode_attend call may ask for */
  const float* gate_csa;          /* [n_layers][heads][m] gate logits (read at create) */
  const float* gate_hca;          /* [n_layers][heads][m_prime] */
  const float* gate_idx;          /* [n_layers][idx_heads][m] */
  uint32_t flags;                 /* KVPOOL_FLAG_* */
  int32_t idx_fp4;                /* 1: indexer entries in FP4 (KVPOOL_FP4_E2M1), 0: in cache_dtype.
                                     FP4 needs idx_heads * idx_dim to be a multiple of 32.  ([P3] s2.2
                                     gives the lightning indexer FP4 keys.) */
  int32_t csa_hot_slots;          /* HiSparse: GPU slots for sealed blocks' CSA entries (0 = off: a
                                     block's CSA entries stay with the block id; else <= max_blocks) */
  int32_t csa_host_slots;         /* HiSparse: host slots for offloaded blocks' CSA entries (0 if off) */
  int32_t idx_per_token;          /* 1: the indexer keeps one key per token (m' per block, the
                                     block figure's "128 indexer K") instead of one per CSA entry;
                                     entry e's score is sum_i sum_j alpha_idx[j][i] * <q_j, key of
                                     token m*e+i, head j> (fixed order: per token, each head's fp32
                                     chain times the token's scale, an fp32 chain over heads with
                                     the gates, then the m tokens added in order).  Needs
                                     idx_heads * idx_dim <= 256. */
} kvpool_config;

typedef struct kvpool kvpool_t;

/* Arena bytes a config needs (0 if the config is invalid). */
size_t kvpool_required_bytes(const kvpool_config* cfg);

/* Create a pool in the caller's device arena.  Validates cfg ([P1] s2.2:
 * m | m'; [P3] s2.2: the window is a whole number of blocks; heads * head_dim
 * a multiple of 256 up to 4096; idx_heads * idx_dim a multiple of 16 up to
 * 2048 and at most 2 * heads * head_dim; one block's indexer keys (score
 * kernel) and four stages of entries (attention kernel) small enough to stage
 * in one CTA's 227 KiB of shared memory), computes the
 * gates' softmax on the host and uploads them, and clears the device error
 * word, in stream order on `stream`.  d_arena must stay allocated until
 * kvpool_destroy.  With KVPOOL_FLAG_NO_DEVICE, d_arena must be NULL and the
 * pool only keeps bookkeeping.  Errors: INVALID_ARG, CUDA. */
int kvpool_create(const kvpool_config* cfg, void* d_arena, size_t arena_bytes, void* stream, kvpool_t** out);
int kvpool_destroy(kvpool_t* pool);

/* Take the smallest free request slot; its State block is empty (length 0).
 * [P3] s2.1.  Errors: OUT_OF_REQUESTS. */
int kvpool_alloc_request(kvpool_t* pool, int32_t* req_out);

/* Release a request: its State block whole, and one reference on each of its
 * sealed blocks (a block id returns to the free set at refcount 0).  [P3]
 * s2.1, s2.2.  Errors: BAD_REQUEST. */
int kvpool_free_request(kvpool_t* pool, int32_t req);

/* Zero SWA prefix reuse ([P4], [P3] s2.2): the fresh request dst references
 * (refcount + 1) the first n_tokens / m' sealed blocks of src and takes
 * length n_tokens.  d_win_k, d_win_v: [n_layers][w][heads][head_dim] in
 * in_dtype, w = min(n_tokens, n_win): the caller's recomputed K/V of
 * positions n_tokens-w .. n_tokens-1, written into dst's window.  Errors:
 * BAD_REQUEST (dst/src invalid or equal), INVALID_ARG (n_tokens <= 0 or a
 * NULL window), NOT_SHAREABLE (n_tokens not a multiple of m', beyond src's
 * sealed blocks, or dst not fresh), CUDA. */
int kvpool_share_prefix(kvpool_t* pool, int32_t dst, int32_t src, int64_t n_tokens, const void* d_win_k,
                        const void* d_win_v, void* stream);

/* ---- prefix images: sealed blocks in host memory ----
 * "Ch 12 Inference framework: heterogeneous KV scheduling" s3 (disk-resident
 * KV: the compressed block cache is serialized, and a prefix hit brings it
 * back with an async copy instead of a prefill) and s3.1, with "V4 disk
 * prefix cache" (SWA policies: Full, Periodic checkpointing, Zero).  Here the
 * store is page-locked host memory; the copies run as kernels that read and
 * write it over the host link.
 *
 * An image holds the first n_tokens / m' sealed blocks of a request
 * (n_tokens a positive multiple of m') and, with KVPOOL_IMAGE_WINDOW, the
 * SWA window at length n_tokens, which the pool holds only while the
 * request's length is n_tokens (a checkpoint; at a multiple p of m' this is
 * Periodic checkpointing).  Without the window a restore takes the caller's
 * recomputed window tokens (Zero SWA).  Byte layout, little-endian:
 *   header, 64 B: u32 magic 0x4950564B ("KVPI"), u32 version 1, u64 config
 *     fingerprint, i64 n_tokens, i32 n_blocks, i32 w (window tokens in the
 *     image, 0 if none), u64 block-section bytes, u64 window-section bytes,
 *     u64 total bytes, u64 0;
 *   block section: for each layer in order, for each part the layer has (CSA
 *     entries, indexer keys, HCA entry) the n_blocks blocks' part in table
 *     order, each exactly as stored in the part's plane (kvpool_layer_layout:
 *     csa/idx/hca_block_bytes), with the zero padding after the indexer
 *     scales forced to zero;
 *   window section: for each layer the tokens at positions n_tokens - w ..
 *     n_tokens - 1, one entry_bytes record each (w = min(n_tokens, n_win)).
 * The fingerprint is FNV-1a 64 over the little-endian int32 fields m, m',
 * n_win, heads, head_dim, idx_heads, idx_dim, in_dtype, cache_dtype, idx_fp4 +
 * 2 * idx_per_token, n_layers, then per layer its kind and the fp32 bits of the gate logits it
 * uses (CSA then indexer if it has CSA, HCA if it has HCA).  Images need each
 * indexer key to be whole 16-byte chunks (when a layer has CSA).
 *
 * The image buffer is caller-owned page-locked host memory (cudaHostAlloc,
 * or cudaHostRegister'd with cudaHostRegisterMapped), 16-byte aligned. */
#define KVPOOL_IMAGE_WINDOW 1u

/* FNV-1a 64 of the pool's config record (see above). */
uint64_t kvpool_fingerprint(const kvpool_t* pool);

/* Bytes of the image of an n_tokens prefix with `flags`; -1 if n_tokens is
 * not a positive multiple of m' or the config has no image layout. */
int64_t kvpool_image_bytes(const kvpool_t* pool, int64_t n_tokens, uint32_t flags);

/* Write the image of request req's first n_tokens tokens into h_image
 * (capacity bytes).  The header is written by the host during the call; the
 * blocks and window are copied by a kernel in stream order on `stream`, so
 * the image is complete when the stream reaches that point.  Errors:
 * BAD_REQUEST, NOT_SHAREABLE (n_tokens not a multiple of m', beyond req's
 * sealed blocks, or the window asked for at a length other than req's),
 * INVALID_ARG (unknown flag, capacity below kvpool_image_bytes, a buffer that
 * is not page-locked host memory or not 16-byte aligned, no image layout),
 * CUDA. */
int kvpool_export_prefix(kvpool_t* pool, int32_t req, int64_t n_tokens, uint32_t flags, void* h_image,
                         int64_t capacity, void* stream);

/* Restore an image into the fresh request dst: its blocks get new ids (the
 * smallest free ids, in image order, refcount 1), dst's table and length
 * n_tokens are set, and its window comes from the image, or, for an image
 * without one, from d_win_k / d_win_v ([n_layers][w][heads][head_dim] in
 * in_dtype, w = min(n_tokens, n_win), 16-byte aligned device memory: the
 * recomputed K/V of positions n_tokens - w .. n_tokens - 1, as for
 * kvpool_share_prefix); give NULL windows with an image that has one.  The
 * host reads the header during the call (the image must be complete by
 * then); a kernel copies the rest in stream order.  Errors: BAD_IMAGE
 * (magic, version, fingerprint or sizes wrong, bytes too small),
 * NOT_SHAREABLE (dst not fresh), CAPACITY, OUT_OF_BLOCKS, INVALID_ARG
 * (windows missing or given when the image has one, buffer not page-locked
 * or aligned), BAD_REQUEST, CUDA; an error leaves the pool unchanged. */
int kvpool_import_prefix(kvpool_t* pool, int32_t dst, const void* h_image, int64_t bytes, const void* d_win_k,
                         const void* d_win_v, void* stream);

/* ---- HiSparse: inactive CSA entries off the GPU ----
 * "V4 KV Layout: Classical + State dual pool" (ESS / HiSparse table: HiSparse
 * moves inactive C4 entries of the Classical pool off the GPU, on top of the
 * layout) and "Why does V4 split pools? ..." s1 / s3.2 (only full, immutable
 * blocks move; the SWA window stays resident).  With csa_hot_slots > 0 a
 * sealed block's CSA entries (every layer's) live in one of csa_hot_slots
 * GPU slots or, once offloaded, in one of csa_host_slots slots of a
 * caller-owned page-locked host pool; its indexer keys and HCA entry never
 * move (the indexer scans every key, and every HCA entry is read, each step).
 * Slots are taken smallest-free when a block seals, is restored or fetched
 * (hot) and when it is offloaded (host); they return when the block is freed.
 * Attention reads a selected entry of an offloaded block straight from host
 * memory.  Activity: every kvpool_decode_attend call advances the pool's
 * epoch by one; a call on a CSA layer stamps each block holding a selected
 * entry with that epoch, and sealing, restoring or fetching a block stamps the
 * current epoch.  A block is inactive after `idle` epochs without a stamp.
 * Placement never changes a value: outputs are bit-identical whether or not
 * blocks are offloaded.  All of this is in stream order on `stream`. */

/* Bytes of one host slot: the CSA entries of one block over all CSA layers. */
int64_t kvpool_host_slot_bytes(const kvpool_t* pool);

/* Give the pool its host slots: h_pool page-locked (mapped) host memory of at
 * least csa_host_slots * kvpool_host_slot_bytes bytes, 16-byte aligned,
 * owned by the caller and kept until kvpool_destroy.  Needed before the first
 * offload.  Errors: INVALID_ARG (HiSparse off, too small, not page-locked or
 * aligned, already set while blocks are offloaded). */
int kvpool_set_host_pool(kvpool_t* pool, void* h_pool, int64_t bytes);

/* Move the CSA entries of the resident sealed blocks h_ids[0..n) to host
 * slots (taken in the given order), freeing their GPU slots.  Errors:
 * INVALID_ARG (HiSparse off, no host pool, an id that is free, offloaded or
 * repeated), OUT_OF_BLOCKS (too few free host slots), CUDA; an error changes
 * nothing. */
int kvpool_offload(kvpool_t* pool, int32_t n, const int32_t* h_ids, void* stream);

/* Bring offloaded blocks back to GPU slots (and stamp them).  Errors:
 * INVALID_ARG (an id that is free, resident or repeated), OUT_OF_BLOCKS (too
 * few free GPU slots), CUDA. */
int kvpool_fetch(kvpool_t* pool, int32_t n, const int32_t* h_ids, void* stream);

/* Where block id's CSA entries are (host bookkeeping, no synchronization):
 * *loc >= 0 a GPU slot, < 0 host slot -1 - *loc (without HiSparse *loc is
 * the id).  Errors: INVALID_ARG (a free block). */
int kvpool_block_location(const kvpool_t* pool, int32_t block_id, int32_t* loc);

/* Decode calls so far (the current epoch). */
uint32_t kvpool_epoch(const kvpool_t* pool);

/* Synchronize `stream` and write the activity stamps of blocks h_ids[0..n)
 * to h_last_used.  Errors: INVALID_ARG (HiSparse off, a free block), CUDA. */
int kvpool_block_activity(kvpool_t* pool, int32_t n, const int32_t* h_ids, uint32_t* h_last_used, void* stream);

/* Synchronize `stream` and list the resident sealed blocks with epoch -
 * stamp >= idle, ascending ids, up to cap of them into h_ids; returns how
 * many there are (negative: an error: INVALID_ARG with HiSparse off, CUDA). */
int32_t kvpool_inactive_blocks(kvpool_t* pool, uint32_t idle, int32_t* h_ids, int32_t cap, void* stream);

/* Append new tokens ([P1] s3, s4): for request h_req_ids[i], h_n_new[i]
 * tokens.  d_k, d_v: [n_layers][T][heads][head_dim], d_idx_k:
 * [n_layers][T][idx_heads][idx_dim] (may be NULL when no layer has CSA), all
 * in_dtype, T = sum(h_n_new), rows in batch order then position order.  Each
 * token enters its request's SWA window (rounded to the cache dtype) and
 * tail; every completed m-group forms a CSA entry and an indexer entry, every
 * completed m'-group forms an HCA entry and seals the block, which gets the
 * smallest free block id (requests in batch order, then positions) and is
 * immutable from then on.  Errors: INVALID_ARG (n < 0, n > max_batch,
 * negative counts, duplicate ids, NULL inputs with T > 0), BAD_REQUEST,
 * CAPACITY, OUT_OF_BLOCKS, CUDA. */
int kvpool_append(kvpool_t* pool, int32_t n, const int32_t* h_req_ids, const int32_t* h_n_new, const void* d_k,
                  const void* d_v, const void* d_idx_k, void* stream);

/* Decode attention of one layer for n requests ([P1] s4, [P2] Classical KV
 * cache table): score every CSA entry with the indexer, keep the top_k, and
 * attend over [selected CSA entries | all HCA entries | SWA window] in one
 * softmax.  d_q: [n][heads][head_dim], d_q_idx: [n][idx_heads][idx_dim] (may
 * be NULL for layers without CSA), both in_dtype.  d_out: [n][heads][head_dim]
 * fp32.  d_topk_out: [n][top_k] int32 or NULL: the selected CSA entry indices
 * in ascending order, padded with -1.  Errors: INVALID_ARG (layer, n > max_batch,
 * top_k < 0 or > max_top_k, NULL pointers, an empty request), BAD_REQUEST,
 * CUDA. */
int kvpool_decode_attend(kvpool_t* pool, int32_t layer, int32_t n, const int32_t* h_req_ids, const void* d_q,
                         const void* d_q_idx, int32_t top_k, float* d_out, int32_t* d_topk_out, void* stream);

/* Top-k selection over a caller's score matrix that allocates nothing.  The
 * design pages have no counterpart of this entry point: it is the indexer's
 * selection step (same rule as decode_attend: k = min(top_k, n_cols) largest
 * scores, ties to the lower index, -0 == +0, ascending indices padded with
 * -1) offered on its own to callers that cannot allocate device memory: a
 * plugin that only receives its input and output buffers from a host
 * framework that owns every allocation (and gives the plugin no allocator),
 * or a serving loop whose device memory is budgeted once at start-up and must
 * not fail or stall on an allocation in the middle of a step.
 * d_scores: [n_rows][n_cols] fp32 (finite) on the device (may be NULL when
 * n_cols is 0: every row is then all -1); d_topk_out: [n_rows][top_k] int32.  Its scratch (sort keys, radix histograms, counts)
 * is a file-scope 16 MiB device array in this library, present on every GPU
 * that loads it until the process exits: n_rows <= 256, n_cols <= 1,048,576 and
 * 12*n_rows*n_cols + 4*n_rows*top_k + 8.5 KiB*n_rows (+ small) <= 16 MiB,
 * else INVALID_ARG.  No cudaMalloc, cudaFree or allocating library routine is
 * called.  Rows of more than 65,536 columns are selected by one 16-CTA
 * thread-block cluster each (8 where 16 cannot be resident; a cluster starts
 * only when that many SMs have room at once, so work running beside the call
 * delays it); smaller rows by 4096-column chunks or one CTA per row.  The first call on a device looks up that
 * device's address of the array and the cluster shape (for the current
 * device).
 * Every call shares the array and clears what must start at zero; calls that
 * overlap on the GPU (other streams, other host threads) race.  Errors:
 * INVALID_ARG, CUDA; kernel-side errors land in the array's error word, which
 * kvpool_topk_static_check reads. */
int kvpool_topk_static(const float* d_scores, int32_t n_rows, int32_t n_cols, int32_t top_k, int32_t* d_topk_out,
                       void* stream);

/* Device-side error flags of the last kvpool_topk_static call on the current
 * device (the kvpool_check_device bits: 8 = a launch shape the kernels
 * refused, 4 = an index out of range).  Synchronizes `stream` first, then
 * copies the word to *h_flags (may be NULL).  Allocates nothing.  Returns OK
 * when the word is zero, DEVICE_CHECK when a flag is set (the output of that
 * call is not a valid top-k), CUDA on a CUDA error.  Call it before the next
 * kvpool_topk_static, which clears the word. */
int kvpool_topk_static_check(void* stream, uint32_t* h_flags);

/* ---- host-side queries (no device access) ---- */
typedef struct kvpool_info {
  int64_t length;   /* tokens appended (or shared) so far */
  int64_t n_csa;    /* floor(length / m)  CSA entries (sealed + staged) */
  int64_t n_hca;    /* floor(length / m') HCA entries (all sealed) */
  int32_t csa_tail; /* length mod m  (<= m-1)  */
  int32_t hca_tail; /* length mod m' (<= m'-1) */
  int32_t n_blocks; /* sealed blocks in the block table */
  int32_t window;   /* tokens in the SWA window: min(length, n_win) */
} kvpool_info;

/* Fill *info and up to cap block ids (table order).  Errors: BAD_REQUEST. */
int kvpool_request_info(const kvpool_t* pool, int32_t req, kvpool_info* info, int32_t* h_block_ids,
                        int32_t cap);
/* Refcount of a block id (0 = free), or INVALID_ARG. */
int kvpool_block_refcount(const kvpool_t* pool, int32_t block_id);
/* Number of free Classical blocks. */
int kvpool_free_block_count(const kvpool_t* pool);

/* ---- arena layout (byte offsets from d_arena) ----
 * Entry (CSA entry, HCA entry, window token), entry_bytes long:
 *   K codes [heads][head_dim], V codes [heads][head_dim] in the cache dtype,
 *   then for fp8 a bf16 K scale, a bf16 V scale and 12 zero bytes.
 * Indexer keys of a block: runs of csa_per_block keys (one run; with
 *   idx_per_token, m runs of consecutive tokens, idx_block_bytes / m bytes
 *   each): 16-byte chunk c of key e of a run at (c * csa_per_block + e) * 16
 *   from the run's start (chunk-major, so a warp reading chunk c of 32
 *   consecutive keys reads 512 contiguous bytes); fp8 / FP4 scales
 *   [csa_per_block] bf16 at idx_scale_offset from the run's start.
 * Block parts of a layer, each in its own plane: CSA entries [csa_per_block]
 *   at csa_offset + s * csa_block_bytes where s is the block's location (its
 *   id without HiSparse, its GPU slot with it; an offloaded block's CSA
 *   entries are at its host slot * host_slot_bytes + csa_host_offset in the
 *   host pool), indexer keys (then fp8 / FP4 scales at idx_scale_offset) at
 *   idx_offset + b * idx_block_bytes, the HCA entry at hca_offset + b *
 *   hca_block_bytes, b the block id; absent parts have offset -1.  Ids
 *   staging_base + r (r a request slot) are request r's private staging
 *   blocks (its open block); its CSA staging slot is csa_staging_base + r.
 *   A request's blocks, allocated in order, make its indexer keys and HCA
 *   entries contiguous runs.
 * HiSparse: int32 locations [max_blocks] at csa_loc_offset and uint32
 *   activity stamps [max_blocks] at activity_offset.
 * Window of request r: ring_offset + r * ring_request_bytes, token at
 *   position p in slot p mod n_win.
 * Compressor accumulators of request r (fp32): acc_offset + r * acc_request_bytes:
 *   CSA [2][heads][head_dim], indexer [idx_heads][idx_dim], HCA [2][heads][head_dim].
 * Block table: int32 [max_requests][max_blocks_per_request] at table_offset. */
typedef struct kvpool_layer_layout {
  int32_t kind;
  int32_t pad;
  int64_t csa_offset, csa_block_bytes;
  int64_t idx_offset, idx_block_bytes, idx_scale_offset;
  int64_t hca_offset, hca_block_bytes;
  int64_t ring_offset, ring_request_bytes;
  int64_t acc_offset, acc_request_bytes;
  int64_t csa_host_offset; /* this layer's CSA entries inside a host slot (-1 without CSA) */
} kvpool_layer_layout;

typedef struct kvpool_layout {
  int64_t entry_bytes;     /* bytes of one K/V entry or window token */
  int64_t idx_entry_bytes; /* bytes of one indexer key (without scale) */
  int32_t csa_per_block;   /* m' / m */
  int32_t staging_base;    /* = max_blocks */
  int64_t table_offset;
  int64_t error_offset;    /* uint32 device error word */
  int64_t total_bytes;
  int32_t csa_staging_base; /* CSA plane slot of request 0's staging block */
  int32_t csa_hot_slots;    /* 0 without HiSparse */
  int64_t host_slot_bytes;  /* 0 without HiSparse */
  int64_t csa_loc_offset, activity_offset;
} kvpool_layout;

/* Layout of the pool and (if layer_out != NULL) of one layer. */
int kvpool_get_layout(const kvpool_t* pool, kvpool_layout* out, int32_t layer, kvpool_layer_layout* layer_out);

/* Synchronize `stream`, read and clear the device error word.  Returns OK,
 * DEVICE_CHECK (a kernel met an out-of-range index or a wait limit; *word_out
 * gets the flags), or CUDA. */
int kvpool_check_device(kvpool_t* pool, void* stream, uint32_t* word_out);

/* Self-test of the bounded waits (the failure detection of the kernels):
 * one CTA waits, in stream order, on a barrier that nothing completes; after
 * the wait limit (1 s) it sets the wait flag in the device error word and
 * returns, leaving the context usable.  kvpool_check_device then reports
 * DEVICE_CHECK with flag 1.  No memory other than the error word is touched.
 * Errors: INVALID_ARG (a pool without device memory), CUDA. */
int kvpool_wait_selftest(kvpool_t* pool, void* stream);

/* ---- profiling: CUDA events around each launch, on the launch stream ---- */
enum {
  KVPOOL_KERNEL_APPEND = 0,  /* fused append / compress / seal */
  KVPOOL_KERNEL_SCORE = 1,   /* indexer scores + first radix histogram */
  KVPOOL_KERNEL_SELECT = 2,  /* top-k radix select passes and emit */
  KVPOOL_KERNEL_ATTEND = 3,  /* split-K attention over the three sources */
  KVPOOL_KERNEL_COMBINE = 4, /* split-K merge */
  KVPOOL_KERNEL_IMAGE = 5,   /* prefix image copies (export / import) */
  KVPOOL_KERNEL_COUNT = 6
};
#define KVPOOL_PROFILE_ALL ((1 << KVPOOL_KERNEL_COUNT) - 1)
/* With this bit in the mask every launch of every kind also adds its kernel
 * count and algorithmic bytes to its kind's totals, with no events (its time
 * is not measured): accounting that leaves the launches' timing untouched. */
#define KVPOOL_PROFILE_COUNT (1 << 16)
/* Record events around the launches of the kernel kinds whose bit is set in
 * kinds (bit k = KVPOOL_KERNEL_k; KVPOOL_PROFILE_ALL for every kind), and with
 * KVPOOL_PROFILE_COUNT count every launch; 0 disables recording.  A non-zero
 * mask resets the totals and the timeline.
 * Each recorded launch adds two event records to its stream. */
int kvpool_profile_enable(kvpool_t* pool, int kinds);
/* Synchronize and report, for one kernel kind, the summed device time of its
 * launches since profiling was enabled, the launch count and the algorithmic
 * bytes those launches had to move (inputs read + outputs written, scratch
 * excluded). */
int kvpool_profile_read(kvpool_t* pool, int32_t kernel, double* ms_total, int64_t* launches, int64_t* bytes);

/* Synchronize and write, for up to cap launch records since profiling was
 * enabled, (kernel kind, start ms, end ms) triples relative to the first
 * recorded event (h_out: [cap][3] float), in launch order, across the
 * caller's stream and the pool's side stream; returns the number of records
 * or a negative error.  Reading it does not reset the totals. */
int kvpool_profile_timeline(kvpool_t* pool, int32_t cap, float* h_out);

/* Last error message of this pool (never NULL). */
const char* kvpool_last_error(const kvpool_t* pool);

#ifdef __cplusplus
}
#endif
#endif /* KVPOOL_H */

/*
 * kvoracle.h -- CPU oracle for the DeepSeek-V4 two-pool (Classical + State)
 * KV cache decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-threaded model of
 * what the GPU path computes, written from the design pages and used to
 * check it.  Only the tests, the smoke check and the benchmark's CPU
 * baseline leg may load it; the product library never links or calls it,
 * and it shares no code with the CUDA path (the seeded input generator,
 * which holds none of the method's arithmetic, is the one module both use,
 * and only in the test harness).
 *
 * Sources (page title, section):
 *   [P1] "Why does V4 split pools? How do block alignment and the tail
 *        buffer work together": s1.1 pool table, s1.2 CSA m=4 / HCA m'=128,
 *        s2.2 lcm block alignment and L = 128q + r, s2.3 the L = 130
 *        example, s3.1 tail lengths, s3.3 tail vs SWA, s4 one decode step.
 *   [P2] "V4 KV Layout: Classical + State dual pool": Classical KV cache
 *        table (lcm alignment, immutable, CSA top-k sparse read, HCA dense
 *        read of ~L/128 entries), State cache table (SWA, tail, indexer).
 *   [P3] "Ch 12 Inference framework: heterogeneous KV scheduling": glossary
 *        (State / Block cache, lcm blocks, 32 CSA + 1 HCA per block), s2.1
 *        State cache per request, s2.2 Block cache with refcounted sharing,
 *        Figure 12-1 (one block id spans all layers).
 *   [P4] "V4 disk prefix cache": Zero SWA caching (recompute the window on a
 *        prefix hit).
 *
 * Where the pages are silent the oracle takes these readings:
 *   - compressor: entry = fp32 chain acc = fmaf(alpha_i, x_i, acc), i = 0..m-1
 *     from acc = +0, alpha = softmax of seeded per-(layer, head, position)
 *     gate logits computed in double and rounded to fp32; K and V share alpha;
 *     the indexer key has its own gates per indexer head;
 *   - CSA / indexer entries are formed at every completed 4-group and staged
 *     in the request's State until their 128-token block seals;
 *   - indexer score = fp32 chain over the flat (head, dim) order of
 *     fmaf(q_idx, key, acc) from +0, times the entry's scale for fp8;
 *   - top-k: k = min(top_k, #CSA entries), order (score desc, index asc),
 *     returned as ascending indices padded with -1;
 *   - attention: one softmax (scale 1/sqrt(d)) over [selected CSA entries,
 *     all HCA entries, the SWA window] concatenated with no masking; the
 *     window includes the token just appended; computed here in double;
 *   - fp8 e4m3 cache: one bf16 scale per K half, per V half and per indexer
 *     entry: scale = bf16_rn(amax / 448) (1 when that is 0), code =
 *     e4m3_rn_satfinite(x / scale);
 *   - block ids: smallest free id, drawn when a block seals, requests in
 *     batch order then tokens in order; one id spans every layer;
 *   - share_prefix shares whole sealed blocks only and takes the caller's
 *     recomputed window (the Zero SWA policy).
 */
#ifndef KVORACLE_H
#define KVORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { KVO_F32 = 0, KVO_BF16 = 1, KVO_FP8 = 2, KVO_FP4 = 3 /* indexer entries only */ };
enum { KVO_SWA_ONLY = 0, KVO_CSA = 1, KVO_HCA = 2, KVO_CSA_HCA = 3 };
enum {
  KVO_OK = 0,
  KVO_ERR_INVALID_ARG = -1,
  KVO_ERR_OUT_OF_BLOCKS = -2,
  KVO_ERR_OUT_OF_REQUESTS = -3,
  KVO_ERR_BAD_REQUEST = -4,
  KVO_ERR_NOT_SHAREABLE = -5,
  KVO_ERR_CAPACITY = -8, /* a request would exceed max_blocks_per_request */
};

typedef struct kvo_config {
  int32_t m, m_prime, n_win;
  int32_t heads, head_dim, idx_heads, idx_dim;
  int32_t in_dtype, cache_dtype;
  int32_t n_layers;
  const int32_t* layer_kinds;
  int32_t max_requests, max_blocks, max_blocks_per_request;
  const float* gate_csa; /* logits [n_layers][heads][m]       */
  const float* gate_hca; /* logits [n_layers][heads][m_prime] */
  const float* gate_idx; /* logits [n_layers][idx_heads][m]   */
  int32_t idx_fp4;       /* 1: indexer entries in FP4 (e2m1 + one bf16 scale), 0: in the cache dtype */
  /* HiSparse placement of sealed blocks' CSA entries: GPU-resident ("hot")
   * slots and host slots; csa_hot_slots 0 = no HiSparse (every block's CSA
   * entries stay where the block is) */
  int32_t csa_hot_slots, csa_host_slots;
  /* 1: the indexer keeps one key per token (m' per block) instead of one per
   * CSA entry; an entry's score combines its m tokens' scores with the
   * entry's indexer gates (kvo_score_tokens) */
  int32_t idx_per_token;
} kvo_config;

typedef struct kvo kvo_t;

/* ---- scalar codecs (pinned against library casts in the tests) ---- */
uint16_t kvo_bf16_from_f32(float x);
float kvo_f32_from_bf16(uint16_t b);
uint8_t kvo_e4m3_from_f32(float x); /* round to nearest even, saturate to +-448 */
float kvo_f32_from_e4m3(uint8_t c);
uint8_t kvo_e2m1_from_f32(float x); /* 4-bit code: round to nearest even, saturate to +-6 */
float kvo_f32_from_e2m1(uint8_t c);

/* softmax of n logits, computed in double, rounded to fp32 */
void kvo_softmax_f32(const float* logits, int n, float* alpha);

/* Encode n fp32 values: codes are 4/2/1 bytes per value (f32 bits, bf16
 * bits, e4m3) or two e2m1 codes per byte (FP4, element 2j in the low
 * nibble); fp8 and fp4 write one bf16 scale to *scale (amax / 448, amax / 6;
 * 1 if that is 0). */
void kvo_encode(int dtype, const float* x, int n, uint8_t* code, uint16_t* scale);
/* Exact value of element i of an encoded vector (fp8 multiplies its scale). */
double kvo_decode(int dtype, const uint8_t* code, const uint16_t* scale, int i);

/* ---- the method's steps as pure functions ---- */
/* entry (K half then V half, [2][heads][head_dim]) from cnt tokens laid out
 * [cnt][2][heads][head_dim] (fp32 values of the inputs), gates of `layer`,
 * kind 1 = CSA (cnt = m), 2 = HCA (cnt = m_prime).  code: 2*H*d*vsize bytes,
 * scale: 2 bf16. */
int kvo_compress_kv(const kvo_t* o, int layer, int kind, const float* tokens, uint8_t* code, uint16_t* scale);
/* indexer entry ([idx_heads][idx_dim]) from m tokens' indexer keys */
int kvo_compress_idx(const kvo_t* o, int layer, const float* keys, uint8_t* code, uint16_t* scale);
/* indexer score of one encoded indexer entry */
float kvo_score(const kvo_t* o, const uint8_t* code, const uint16_t* scale, const float* q_idx);
/* indexer score of a CSA entry from its m tokens' encoded keys (per-token
 * indexer keys; codes [m][Ih*Id*vsize] and scales [m] contiguous), gates of
 * `layer`: token i's head-j dot D = fmaf chain over idx_dim from +0 (times
 * the token's scale for fp8 / FP4), p_i = fmaf chain over heads of
 * alpha_idx[j][i] * D, score = ((p_0 + p_1) + p_2) + ... in token order.
 * By linearity this is the per-entry score of the uncompressed keys. */
float kvo_score_tokens(const kvo_t* o, int layer, const uint8_t* codes, const uint16_t* scales, const float* q_idx);
/* top-k over n scores: writes k = min(top_k, n) ascending indices, then -1 up to top_k */
int kvo_topk(const float* scores, int64_t n, int top_k, int32_t* out);
/* attention of q ([heads][head_dim]) over n_src encoded entries laid out
 * contiguously (codes [n_src][2*H*d*vsize], scales [n_src][2]); out [H][d] */
int kvo_attend_sources(const kvo_t* o, int64_t n_src, const uint8_t* codes, const uint16_t* scales,
                       const float* q, double* out);

/* ---- the stateful two-pool cache ---- */
int kvo_create(const kvo_config* cfg, kvo_t** out);
void kvo_destroy(kvo_t* o);
int kvo_alloc_request(kvo_t* o, int32_t* req);
int kvo_free_request(kvo_t* o, int32_t req);
/* k, v: [n_layers][T][heads][head_dim]; idx_k: [n_layers][T][idx_heads][idx_dim];
 * T = sum(n_new); rows in batch order then position order (fp32 values). */
int kvo_append(kvo_t* o, int n, const int32_t* req_ids, const int32_t* n_new, const float* k, const float* v,
               const float* idx_k);
/* win_k, win_v: [n_layers][w][heads][head_dim], w = min(n_tokens, n_win): the
 * keys/values of positions n_tokens-w .. n_tokens-1 */
int kvo_share_prefix(kvo_t* o, int32_t dst, int32_t src, int64_t n_tokens, const float* win_k, const float* win_v);
/* q: [n][heads][head_dim]; q_idx: [n][idx_heads][idx_dim]; out: [n][heads][head_dim];
 * topk: [n][top_k] or NULL */
int kvo_decode_attend(kvo_t* o, int layer, int n, const int32_t* req_ids, const float* q, const float* q_idx,
                      int top_k, double* out, int32_t* topk);

/* ---- inspection ---- */
typedef struct kvo_info {
  int64_t length, n_csa, n_hca;
  int32_t csa_tail, hca_tail, n_blocks, window;
} kvo_info;
int kvo_request_info(const kvo_t* o, int32_t req, kvo_info* info, int32_t* block_ids, int32_t cap);
int kvo_block_refcount(const kvo_t* o, int32_t block_id);
int kvo_free_block_count(const kvo_t* o);
/* kind: 1 CSA entry, 2 HCA entry, 3 indexer entry; slot within the block */
int kvo_block_entry(const kvo_t* o, int layer, int32_t block_id, int kind, int slot, uint8_t* code, uint16_t* scale);
/* CSA / indexer entry e of a request (sealed or staged) */
int kvo_request_entry(const kvo_t* o, int layer, int32_t req, int kind, int64_t e, uint8_t* code, uint16_t* scale);
/* window token at absolute position pos (must be in the window) */
int kvo_window_token(const kvo_t* o, int layer, int32_t req, int64_t pos, uint8_t* code, uint16_t* scale);
/* all indexer scores of a request: out[n_csa] */
int kvo_request_scores(const kvo_t* o, int layer, int32_t req, const float* q_idx, float* out);
/* ---- prefix images ([P3] s3 disk-resident KV cache: the compressed block
 * cache serialized and brought back by an async copy, skipping the prefill;
 * [P3] s3.1 and [P4] SWA policies: Full / Periodic checkpoint / Zero) ----
 * An image holds the first n_tokens / m' sealed blocks of a request (n_tokens
 * a multiple of m'), optionally followed by the SWA window at n_tokens (a
 * checkpoint, taken when the request's length is n_tokens).  Byte layout,
 * little-endian:
 *   header (64 B): u32 magic "KVPI", u32 version 1, u64 fingerprint of the
 *     pool's config, i64 n_tokens, i32 n_blocks, i32 w = window tokens in
 *     the image (0 without a window), u64 bytes of the block section, u64
 *     bytes of the window section, u64 total bytes, u64 zero;
 *   block section: for each layer in order, for each part the layer has
 *     (CSA entries, indexer keys, HCA entry), that part of the n_blocks
 *     blocks in table order;
 *   window section: for each layer, the w window tokens at positions
 *     n_tokens - w .. n_tokens - 1.
 *   A K/V entry (CSA, HCA, window token) is its codes (K half, V half), then
 *   for fp8 the bf16 K and V scales and 12 zero bytes.  A block's indexer
 *   part is one run per CB = m'/m keys (one run, or m runs with per-token
 *   keys, tokens in order): the run's keys 16-byte chunk by chunk (byte j
 *   of key e at ((j / 16) * CB + e) * 16 + j % 16), then for fp8 / FP4 keys
 *   the CB bf16 scales, zero-padded to a multiple of 16 bytes.  Images need each
 *   indexer key to be whole 16-byte chunks (when a layer has CSA); other
 *   configs are refused (INVALID_ARG, image bytes -1).
 * The fingerprint is FNV-1a (64-bit) over the little-endian int32 fields m,
 * m', n_win, heads, head_dim, idx_heads, idx_dim, in_dtype, cache_dtype,
 * idx_fp4 + 2 * idx_per_token, n_layers, then per layer its kind followed by the fp32 bits of
 * its gate logits (CSA then indexer if the layer has CSA; HCA if it has HCA).
 */
#define KVO_IMAGE_WINDOW 1u
#define KVO_ERR_BAD_IMAGE (-9)
uint64_t kvo_fnv1a64(const uint8_t* bytes, int64_t n);
uint64_t kvo_fingerprint(const kvo_t* o);
/* bytes of the image of an n_tokens prefix (-1 if n_tokens is not a positive multiple of m') */
int64_t kvo_image_bytes(const kvo_t* o, int64_t n_tokens, uint32_t flags);
/* Write the image; with KVO_IMAGE_WINDOW, n_tokens must be the request's length.
 * Errors: BAD_REQUEST, NOT_SHAREABLE (not whole sealed blocks, or the window
 * asked for at another length), INVALID_ARG (capacity too small). */
int kvo_export_prefix(const kvo_t* o, int32_t req, int64_t n_tokens, uint32_t flags, uint8_t* image, int64_t cap);
/* Restore an image into the fresh request dst: new block ids (smallest free, in
 * image order), length n_tokens, empty tails; the window from the image, else
 * ([P4] Zero SWA) from win_k / win_v [n_layers][w][heads][head_dim] fp32
 * values of the recomputed tokens (w = min(n_tokens, n_win)), which must then
 * be given.  Errors: BAD_IMAGE (magic, version, fingerprint, sizes),
 * NOT_SHAREABLE (dst not fresh), CAPACITY, OUT_OF_BLOCKS, INVALID_ARG. */
int kvo_import_prefix(kvo_t* o, int32_t dst, const uint8_t* image, int64_t bytes, const float* win_k,
                      const float* win_v);
/* ---- HiSparse: offload of inactive CSA entries ("V4 KV Layout" ESS /
 * HiSparse table: inactive C4 entries of the Classical pool move off the GPU;
 * "Why does V4 split pools?" s1, s3.2: only full, immutable blocks are
 * moved).  Reading: a sealed block's CSA entries (every layer's) live in a
 * hot slot or a host slot, taken smallest-free when the block seals (or is
 * restored or fetched) and when it is offloaded; indexer keys and the HCA
 * entry never move.  Activity: every decode_attend call advances the epoch
 * by one; a call on a CSA layer stamps each block holding a selected entry
 * with that epoch (a sealing, restore or fetch stamps the current epoch).  A
 * block is inactive after `idle` epochs without a stamp.  Placement never
 * changes a value. ---- */
/* loc: >= 0 hot slot, < 0 host slot -1-loc; INVALID_ARG for a free block */
int kvo_block_location(const kvo_t* o, int32_t block_id, int32_t* loc, uint32_t* last_used);
uint32_t kvo_epoch(const kvo_t* o);
/* resident sealed blocks with epoch - last_used >= idle, ascending; returns the count (<= cap written) */
int kvo_inactive_blocks(const kvo_t* o, uint32_t idle, int32_t* ids, int32_t cap);
/* Move the CSA entries of resident blocks to host slots (in the given order).
 * Errors: INVALID_ARG (HiSparse off, a free, offloaded or repeated id),
 * OUT_OF_BLOCKS (too few host slots); an error changes nothing. */
int kvo_offload(kvo_t* o, int n, const int32_t* ids);
/* Bring offloaded blocks back to hot slots.  Errors: INVALID_ARG (not
 * offloaded, repeated), OUT_OF_BLOCKS (too few hot slots). */
int kvo_fetch(kvo_t* o, int n, const int32_t* ids);
int kvo_value_bytes(int dtype);
/* bytes of n encoded values (FP4: two per byte) */
int64_t kvo_code_bytes(int dtype, int64_t n);

#ifdef __cplusplus
}
#endif
#endif /* KVORACLE_H */

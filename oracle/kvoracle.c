/*
 * kvoracle.c -- CPU oracle of the two-pool KV cache decode step.
 * TEST INFRASTRUCTURE ONLY (see kvoracle.h for sources and readings).
 *
 * Plain C99, single-threaded, no blocking or fusion: each function follows
 * the step it models in the order the pages give it.  Floating point that
 * decides a stored code or an index (compressor, fp8/bf16 rounding, indexer
 * score) is done in fp32 with explicit fmaf in a fixed order, because those
 * values must agree bit for bit with the GPU; the attention output, which is
 * compared within a tolerance, is computed in double.
 */
#include "kvoracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* scalar codecs                                                        */
/* ------------------------------------------------------------------ */

uint16_t kvo_bf16_from_f32(float x) {
  /* keep the top 16 bits, rounding the dropped 16 to nearest, ties to even */
  uint32_t u;
  memcpy(&u, &x, 4);
  uint32_t upper = u >> 16, lower = u & 0xFFFFu;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return (uint16_t)upper;
}

float kvo_f32_from_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* e4m3 (OCP FP8 "E4M3FN"): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
 * no infinities; largest finite 448 = 1.75 * 2^8; smallest normal 2^-6;
 * subnormals are multiples of 2^-9.  Round to nearest, ties to even, and
 * saturate anything that rounds beyond 448 to 448. */
uint8_t kvo_e4m3_from_f32(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
  float a = fabsf(x);
  if (a >= 448.0f) return sign | 0x7E;
  int E = (int)((u >> 23) & 0xFFu) - 127; /* unbiased exponent of x */
  if (E < -6) {                            /* below the smallest normal 2^-6 */
    float q = nearbyintf(a * 512.0f);      /* units of 2^-9 (exact scaling); 8 = smallest normal */
    return (uint8_t)(sign | (uint8_t)q);
  }
  uint32_t pb = (uint32_t)(127 + 3 - E) << 23; /* 2^(3-E) */
  float p2;
  memcpy(&p2, &pb, 4);
  float q = nearbyintf(a * p2); /* significand in eighths, 8 .. 16 (exact scaling, then ties-to-even) */
  if (q == 16.0f) {
    q = 8.0f;
    E += 1;
  }
  if (E > 8 || (E == 8 && q > 14.0f)) return sign | 0x7E;
  return (uint8_t)(sign | (uint8_t)(((E + 7) << 3) | ((int)q - 8)));
}

float kvo_f32_from_e4m3(uint8_t c) {
  int E = (c >> 3) & 15, M = c & 7;
  double v = (E == 0) ? ldexp((double)M, -9) : ldexp((double)(8 + M), E - 10);
  return (float)((c & 0x80) ? -v : v);
}

/* e2m1 (OCP MX FP4): 1 sign, 2 exponent (bias 1), 1 mantissa bit; the
 * magnitudes 0, 0.5 (subnormal), 1, 1.5, 2, 3, 4, 6; no infinities or NaN.
 * The nearest magnitude wins, a tie goes to the even code (mantissa bit 0),
 * anything at or beyond 6 saturates to 6; the sign bit is the sign of x. */
static const float kE2m1[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

uint8_t kvo_e2m1_from_f32(float x) {
  const uint8_t sign = signbit(x) ? 8 : 0;
  const float a = fabsf(x);
  if (a >= 6.0f) return sign | 7;
  int best = 0;
  for (int c = 1; c < 8; ++c) {
    const float d = fabsf(a - kE2m1[c]), db = fabsf(a - kE2m1[best]);
    if (d < db || (d == db && (c & 1) == 0)) best = c;
  }
  return (uint8_t)(sign | best);
}

float kvo_f32_from_e2m1(uint8_t c) {
  const float v = kE2m1[c & 7];
  return (c & 8) ? -v : v;
}

void kvo_softmax_f32(const float* g, int n, float* alpha) {
  double mx = g[0];
  for (int i = 1; i < n; ++i)
    if (g[i] > mx) mx = g[i];
  double* e = (double*)malloc(sizeof(double) * (size_t)n);
  double sum = 0.0;
  for (int i = 0; i < n; ++i) {
    e[i] = exp((double)g[i] - mx);
    sum += e[i];
  }
  for (int i = 0; i < n; ++i) alpha[i] = (float)(e[i] / sum);
  free(e);
}

int kvo_value_bytes(int dtype) { return dtype == KVO_F32 ? 4 : dtype == KVO_BF16 ? 2 : 1; }

int64_t kvo_code_bytes(int dtype, int64_t n) { return dtype == KVO_FP4 ? (n + 1) / 2 : n * kvo_value_bytes(dtype); }

void kvo_encode(int dtype, const float* x, int n, uint8_t* code, uint16_t* scale) {
  if (dtype == KVO_F32) {
    memcpy(code, x, 4 * (size_t)n);
  } else if (dtype == KVO_BF16) {
    for (int i = 0; i < n; ++i) {
      uint16_t b = kvo_bf16_from_f32(x[i]);
      memcpy(code + 2 * (size_t)i, &b, 2);
    }
  } else {
    const float top = dtype == KVO_FP4 ? 6.0f : 448.0f;
    float amax = 0.0f;
    for (int i = 0; i < n; ++i)
      if (fabsf(x[i]) > amax) amax = fabsf(x[i]);
    uint16_t sb = kvo_bf16_from_f32(amax / top);
    if (sb == 0) sb = 0x3F80; /* 1.0 */
    float s = kvo_f32_from_bf16(sb);
    if (dtype == KVO_FP4) {
      for (int i = 0; i < (n + 1) / 2; ++i) code[i] = 0;
      for (int i = 0; i < n; ++i) code[i / 2] |= (uint8_t)(kvo_e2m1_from_f32(x[i] / s) << (4 * (i & 1)));
    } else {
      for (int i = 0; i < n; ++i) code[i] = kvo_e4m3_from_f32(x[i] / s);
    }
    *scale = sb;
  }
}

/* value of element i without the fp8 scale (the code's own value) */
static float raw_value(int dtype, const uint8_t* code, int i) {
  if (dtype == KVO_F32) {
    float f;
    memcpy(&f, code + 4 * (size_t)i, 4);
    return f;
  }
  if (dtype == KVO_BF16) {
    uint16_t b;
    memcpy(&b, code + 2 * (size_t)i, 2);
    return kvo_f32_from_bf16(b);
  }
  if (dtype == KVO_FP4) return kvo_f32_from_e2m1((uint8_t)((code[i / 2] >> (4 * (i & 1))) & 15));
  return kvo_f32_from_e4m3(code[i]);
}

double kvo_decode(int dtype, const uint8_t* code, const uint16_t* scale, int i) {
  double v = raw_value(dtype, code, i);
  if (dtype == KVO_FP8 || dtype == KVO_FP4) v *= (double)kvo_f32_from_bf16(*scale);
  return v;
}

/* ------------------------------------------------------------------ */
/* oracle state                                                         */
/* ------------------------------------------------------------------ */

typedef struct layer_sec { /* one layer's share of a Classical block (or of a request's staging) */
  uint8_t* csa_code;
  uint16_t* csa_scale; /* [CB][esz], [CB][2] */
  uint8_t* idx_code;
  uint16_t* idx_scale; /* [CB][xsz], [CB]    */
  uint8_t* hca_code;
  uint16_t hca_scale[2];
} layer_sec;

typedef struct block {
  int refcount;
  layer_sec* layers;  /* allocated on first use, kept */
  int32_t loc;        /* HiSparse: >= 0 hot slot, < 0 host slot -1-loc */
  uint32_t last_used; /* epoch of the last selection of one of its CSA entries */
} block;

typedef struct req_layer {
  uint8_t* win_code;
  uint16_t* win_scale; /* [W][esz], [W][2]; position p lives in slot p % W */
  float* tail_kv;      /* [m'][2*H*d] raw tokens since the last block boundary */
  int tail_len;
  float* tail_idx; /* [m][Ih*Id] raw indexer keys since the last CSA boundary */
  int tail_idx_len;
  layer_sec stage;  /* CSA / indexer entries of the open block */
  uint8_t* hca_new; /* HCA entry formed this token, moved into the block at seal */
  uint16_t hca_new_scale[2];
} req_layer;

typedef struct request {
  int active;
  int64_t L;
  int n_sealed;
  int32_t* table;     /* [max_blocks_per_request] */
  req_layer* layers;  /* allocated on first use, kept */
} request;

struct kvo {
  kvo_config c;
  int32_t* kinds;
  int HD, XD, CB, esz, xsz, vs;
  int XB; /* indexer keys per block section: CB (one per CSA entry) or m' (one per token) */
  int idx_dtype; /* indexer entries: the cache dtype, or KVO_FP4 */
  float* alpha_csa; /* [n_layers][H][m]  */
  float* alpha_hca; /* [n_layers][H][m'] */
  float* alpha_idx; /* [n_layers][Ih][m] */
  block* blocks;
  int n_free_blocks;
  int block_hint; /* no free id below this */
  uint64_t fingerprint; /* of the config, for prefix images */
  int hisparse;         /* HiSparse placement on */
  uint8_t* hot_used;    /* [csa_hot_slots] */
  uint8_t* host_used;   /* [csa_host_slots] */
  int hot_free, host_free;
  uint32_t epoch;       /* decode_attend calls so far */
  request* reqs;
};

static int has_csa(const kvo_t* o, int l) { return o->kinds[l] == KVO_CSA || o->kinds[l] == KVO_CSA_HCA; }
static int has_hca(const kvo_t* o, int l) { return o->kinds[l] == KVO_HCA || o->kinds[l] == KVO_CSA_HCA; }

static void sec_alloc(const kvo_t* o, layer_sec* s) {
  s->csa_code = (uint8_t*)calloc((size_t)o->CB, (size_t)o->esz);
  s->csa_scale = (uint16_t*)calloc((size_t)o->CB * 2, 2);
  s->idx_code = (uint8_t*)calloc((size_t)o->XB, (size_t)o->xsz);
  s->idx_scale = (uint16_t*)calloc((size_t)o->XB, 2);
  s->hca_code = (uint8_t*)calloc(1, (size_t)o->esz);
  s->hca_scale[0] = s->hca_scale[1] = 0;
}

static void sec_free(layer_sec* s) {
  free(s->csa_code);
  free(s->csa_scale);
  free(s->idx_code);
  free(s->idx_scale);
  free(s->hca_code);
}

/* FNV-1a, 64-bit (Fowler, Noll, Vo): h = offset basis; for each byte
 * h = (h xor byte) * prime, modulo 2^64 */
uint64_t kvo_fnv1a64(const uint8_t* bytes, int64_t n) {
  uint64_t h = 0xcbf29ce484222325ull;
  for (int64_t i = 0; i < n; ++i) {
    h ^= bytes[i];
    h *= 0x100000001b3ull;
  }
  return h;
}

typedef struct hasher {
  uint64_t h;
} hasher;

static void hash_bytes(hasher* x, const uint8_t* b, int n) {
  for (int i = 0; i < n; ++i) {
    x->h ^= b[i];
    x->h *= 0x100000001b3ull;
  }
}

static void hash_i32(hasher* x, int32_t v) {
  uint32_t u = (uint32_t)v;
  uint8_t b[4] = {(uint8_t)u, (uint8_t)(u >> 8), (uint8_t)(u >> 16), (uint8_t)(u >> 24)};
  hash_bytes(x, b, 4);
}

static void hash_f32s(hasher* x, const float* f, int64_t n) {
  for (int64_t i = 0; i < n; ++i) {
    uint32_t u;
    memcpy(&u, &f[i], 4);
    hash_i32(x, (int32_t)u);
  }
}

/* the canonical config record of prefix images (see kvoracle.h) */
static uint64_t config_fingerprint(const kvo_config* c) {
  hasher x = {0xcbf29ce484222325ull};
  const int32_t f[11] = {c->m,       c->m_prime,  c->n_win,       c->heads,   c->head_dim, c->idx_heads,
                         c->idx_dim, c->in_dtype, c->cache_dtype, c->idx_fp4 | (c->idx_per_token << 1),
                         c->n_layers};
  for (int i = 0; i < 11; ++i) hash_i32(&x, f[i]);
  for (int l = 0; l < c->n_layers; ++l) {
    const int k = c->layer_kinds[l];
    hash_i32(&x, k);
    if (k == KVO_CSA || k == KVO_CSA_HCA) {
      hash_f32s(&x, c->gate_csa + (size_t)l * c->heads * c->m, (int64_t)c->heads * c->m);
      hash_f32s(&x, c->gate_idx + (size_t)l * c->idx_heads * c->m, (int64_t)c->idx_heads * c->m);
    }
    if (k == KVO_HCA || k == KVO_CSA_HCA)
      hash_f32s(&x, c->gate_hca + (size_t)l * c->heads * c->m_prime, (int64_t)c->heads * c->m_prime);
  }
  return x.h;
}

int kvo_create(const kvo_config* cfg, kvo_t** out) {
  if (!cfg || !out) return KVO_ERR_INVALID_ARG;
  const kvo_config* c = cfg;
  if (c->m < 1 || c->m_prime < c->m || c->m_prime % c->m != 0) return KVO_ERR_INVALID_ARG;
  /* lcm(m, m') = m' when m | m'; the window is a whole number of blocks */
  if (c->n_win < c->m_prime || c->n_win % c->m_prime != 0) return KVO_ERR_INVALID_ARG;
  if (c->heads < 1 || c->head_dim < 1 || c->idx_heads < 1 || c->idx_dim < 1) return KVO_ERR_INVALID_ARG;
  if (c->in_dtype != KVO_F32 && c->in_dtype != KVO_BF16) return KVO_ERR_INVALID_ARG;
  if (c->cache_dtype < KVO_F32 || c->cache_dtype > KVO_FP8) return KVO_ERR_INVALID_ARG;
  if (c->idx_fp4 != 0 && c->idx_fp4 != 1) return KVO_ERR_INVALID_ARG;
  if (c->idx_per_token != 0 && c->idx_per_token != 1) return KVO_ERR_INVALID_ARG;
  if (c->n_layers < 1 || !c->layer_kinds) return KVO_ERR_INVALID_ARG;
  if (c->max_requests < 1 || c->max_blocks < 1 || c->max_blocks_per_request < 1) return KVO_ERR_INVALID_ARG;
  for (int l = 0; l < c->n_layers; ++l)
    if (c->layer_kinds[l] < KVO_SWA_ONLY || c->layer_kinds[l] > KVO_CSA_HCA) return KVO_ERR_INVALID_ARG;

  kvo_t* o = (kvo_t*)calloc(1, sizeof(kvo_t));
  o->c = *c;
  o->kinds = (int32_t*)malloc(sizeof(int32_t) * (size_t)c->n_layers);
  memcpy(o->kinds, c->layer_kinds, sizeof(int32_t) * (size_t)c->n_layers);
  o->c.layer_kinds = o->kinds;
  o->HD = c->heads * c->head_dim;
  o->XD = c->idx_heads * c->idx_dim;
  o->CB = c->m_prime / c->m; /* CSA entries per block */
  o->XB = c->idx_per_token ? c->m_prime : o->CB;
  o->vs = kvo_value_bytes(c->cache_dtype);
  o->esz = 2 * o->HD * o->vs;
  o->idx_dtype = c->idx_fp4 ? KVO_FP4 : c->cache_dtype;
  o->xsz = (int)kvo_code_bytes(o->idx_dtype, o->XD);

  /* gates: alpha = softmax over the group's positions, per layer and head */
  o->alpha_csa = (float*)calloc((size_t)c->n_layers * c->heads * c->m, sizeof(float));
  o->alpha_hca = (float*)calloc((size_t)c->n_layers * c->heads * c->m_prime, sizeof(float));
  o->alpha_idx = (float*)calloc((size_t)c->n_layers * c->idx_heads * c->m, sizeof(float));
  for (int l = 0; l < c->n_layers; ++l) {
    if (has_csa(o, l)) {
      if (!c->gate_csa || !c->gate_idx) {
        kvo_destroy(o);
        return KVO_ERR_INVALID_ARG;
      }
      for (int h = 0; h < c->heads; ++h) {
        size_t off = ((size_t)l * c->heads + h) * c->m;
        kvo_softmax_f32(c->gate_csa + off, c->m, o->alpha_csa + off);
      }
      for (int g = 0; g < c->idx_heads; ++g) {
        size_t off = ((size_t)l * c->idx_heads + g) * c->m;
        kvo_softmax_f32(c->gate_idx + off, c->m, o->alpha_idx + off);
      }
    }
    if (has_hca(o, l)) {
      if (!c->gate_hca) {
        kvo_destroy(o);
        return KVO_ERR_INVALID_ARG;
      }
      for (int h = 0; h < c->heads; ++h) {
        size_t off = ((size_t)l * c->heads + h) * c->m_prime;
        kvo_softmax_f32(c->gate_hca + off, c->m_prime, o->alpha_hca + off);
      }
    }
  }
  o->blocks = (block*)calloc((size_t)c->max_blocks, sizeof(block));
  o->n_free_blocks = c->max_blocks;
  o->block_hint = 0;
  o->reqs = (request*)calloc((size_t)c->max_requests, sizeof(request));
  o->fingerprint = config_fingerprint(c);
  o->hisparse = c->csa_hot_slots > 0;
  if (c->csa_hot_slots < 0 || c->csa_host_slots < 0 || (!o->hisparse && c->csa_host_slots > 0)) {
    kvo_destroy(o);
    return KVO_ERR_INVALID_ARG;
  }
  o->hot_used = (uint8_t*)calloc((size_t)c->csa_hot_slots + 1, 1);
  o->host_used = (uint8_t*)calloc((size_t)c->csa_host_slots + 1, 1);
  o->hot_free = c->csa_hot_slots;
  o->host_free = c->csa_host_slots;
  *out = o;
  return KVO_OK;
}

void kvo_destroy(kvo_t* o) {
  if (!o) return;
  free(o->hot_used);
  free(o->host_used);
  if (o->blocks) {
    for (int b = 0; b < o->c.max_blocks; ++b) {
      if (!o->blocks[b].layers) continue;
      for (int l = 0; l < o->c.n_layers; ++l) sec_free(&o->blocks[b].layers[l]);
      free(o->blocks[b].layers);
    }
    free(o->blocks);
  }
  if (o->reqs) {
    for (int r = 0; r < o->c.max_requests; ++r) {
      request* q = &o->reqs[r];
      free(q->table);
      if (!q->layers) continue;
      for (int l = 0; l < o->c.n_layers; ++l) {
        req_layer* rl = &q->layers[l];
        free(rl->win_code);
        free(rl->win_scale);
        free(rl->tail_kv);
        free(rl->tail_idx);
        free(rl->hca_new);
        sec_free(&rl->stage);
      }
      free(q->layers);
    }
    free(o->reqs);
  }
  free(o->alpha_csa);
  free(o->alpha_hca);
  free(o->alpha_idx);
  free(o->kinds);
  free(o);
}

/* ------------------------------------------------------------------ */
/* the method's steps                                                   */
/* ------------------------------------------------------------------ */

/* Compressor: a fixed-order fp32 chain over the group's tokens, then the
 * cache-dtype encoding of the K half and of the V half. */
int kvo_compress_kv(const kvo_t* o, int layer, int kind, const float* tokens, uint8_t* code, uint16_t* scale) {
  if (layer < 0 || layer >= o->c.n_layers || (kind != 1 && kind != 2)) return KVO_ERR_INVALID_ARG;
  int cnt = kind == 1 ? o->c.m : o->c.m_prime;
  const float* alpha = kind == 1 ? o->alpha_csa + (size_t)layer * o->c.heads * o->c.m
                                 : o->alpha_hca + (size_t)layer * o->c.heads * o->c.m_prime;
  int HD = o->HD, W2 = 2 * HD;
  float* acc = (float*)malloc(sizeof(float) * (size_t)W2);
  for (int v = 0; v < W2; ++v) {
    int h = (v % HD) / o->c.head_dim;
    float a = 0.0f;
    for (int i = 0; i < cnt; ++i) a = fmaf(alpha[(size_t)h * cnt + i], tokens[(size_t)i * W2 + v], a);
    acc[v] = a;
  }
  scale[0] = scale[1] = 0;
  kvo_encode(o->c.cache_dtype, acc, HD, code, &scale[0]);
  kvo_encode(o->c.cache_dtype, acc + HD, HD, code + (size_t)HD * o->vs, &scale[1]);
  free(acc);
  return KVO_OK;
}

int kvo_compress_idx(const kvo_t* o, int layer, const float* keys, uint8_t* code, uint16_t* scale) {
  if (layer < 0 || layer >= o->c.n_layers) return KVO_ERR_INVALID_ARG;
  int m = o->c.m, XD = o->XD;
  const float* alpha = o->alpha_idx + (size_t)layer * o->c.idx_heads * m;
  float* acc = (float*)malloc(sizeof(float) * (size_t)XD);
  for (int v = 0; v < XD; ++v) {
    int g = v / o->c.idx_dim;
    float a = 0.0f;
    for (int i = 0; i < m; ++i) a = fmaf(alpha[(size_t)g * m + i], keys[(size_t)i * XD + v], a);
    acc[v] = a;
  }
  *scale = 0;
  kvo_encode(o->idx_dtype, acc, XD, code, scale);
  free(acc);
  return KVO_OK;
}

float kvo_score(const kvo_t* o, const uint8_t* code, const uint16_t* scale, const float* q_idx) {
  float a = 0.0f;
  for (int v = 0; v < o->XD; ++v) a = fmaf(q_idx[v], raw_value(o->idx_dtype, code, v), a);
  if (o->idx_dtype == KVO_FP8 || o->idx_dtype == KVO_FP4) a = a * kvo_f32_from_bf16(*scale);
  return a;
}

float kvo_score_tokens(const kvo_t* o, int layer, const uint8_t* codes, const uint16_t* scales, const float* q_idx) {
  const int m = o->c.m, Ih = o->c.idx_heads, Id = o->c.idx_dim;
  const float* alpha = o->alpha_idx + (size_t)layer * Ih * m;
  const int scaled = o->idx_dtype == KVO_FP8 || o->idx_dtype == KVO_FP4;
  float s = 0.0f;
  for (int i = 0; i < m; ++i) {
    const uint8_t* code = codes + (size_t)i * o->xsz;
    float p = 0.0f;
    for (int j = 0; j < Ih; ++j) {
      float d = 0.0f;
      for (int v = j * Id; v < (j + 1) * Id; ++v) d = fmaf(q_idx[v], (float)raw_value(o->idx_dtype, code, v), d);
      if (scaled) d = d * kvo_f32_from_bf16(scales[i]);
      p = fmaf(alpha[(size_t)j * m + i], d, p);
    }
    s = i == 0 ? p : s + p;
  }
  return s;
}

typedef struct cand {
  float s;
  int64_t i;
} cand;

static int cand_cmp(const void* pa, const void* pb) {
  const cand* a = (const cand*)pa;
  const cand* b = (const cand*)pb;
  if (a->s > b->s) return -1; /* higher score first; -0 == +0 here */
  if (a->s < b->s) return 1;
  return (a->i < b->i) ? -1 : (a->i > b->i); /* tie: lower index first */
}

static int i32_cmp(const void* pa, const void* pb) {
  int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  return (a > b) - (a < b);
}

int kvo_topk(const float* scores, int64_t n, int top_k, int32_t* out) {
  if (n < 0 || top_k < 0) return KVO_ERR_INVALID_ARG;
  int64_t k = n < top_k ? n : top_k;
  if (k > 0) {
    cand* c = (cand*)malloc(sizeof(cand) * (size_t)n);
    for (int64_t i = 0; i < n; ++i) {
      c[i].s = scores[i];
      c[i].i = i;
    }
    qsort(c, (size_t)n, sizeof(cand), cand_cmp);
    for (int64_t j = 0; j < k; ++j) out[j] = (int32_t)c[j].i;
    free(c);
    qsort(out, (size_t)k, sizeof(int32_t), i32_cmp);
  }
  for (int64_t j = k; j < top_k; ++j) out[j] = -1;
  return KVO_OK;
}

/* value v of an encoded K/V entry: K half uses scale[0], V half scale[1] */
static double entry_value(const kvo_t* o, const uint8_t* code, const uint16_t* scale, int v) {
  return kvo_decode(o->c.cache_dtype, code, scale + (v >= o->HD ? 1 : 0), v);
}

int kvo_attend_sources(const kvo_t* o, int64_t n_src, const uint8_t* codes, const uint16_t* scales,
                       const float* q, double* out) {
  if (n_src <= 0) return KVO_ERR_INVALID_ARG;
  int d = o->c.head_dim, HD = o->HD;
  double* z = (double*)malloc(sizeof(double) * (size_t)n_src);
  for (int h = 0; h < o->c.heads; ++h) {
    double mx = -INFINITY;
    for (int64_t s = 0; s < n_src; ++s) {
      const uint8_t* c = codes + (size_t)s * o->esz;
      const uint16_t* sc = scales + 2 * (size_t)s;
      double dot = 0.0;
      for (int j = 0; j < d; ++j) dot += (double)q[h * d + j] * entry_value(o, c, sc, h * d + j);
      z[s] = dot / sqrt((double)d);
      if (z[s] > mx) mx = z[s];
    }
    double den = 0.0;
    for (int64_t s = 0; s < n_src; ++s) den += exp(z[s] - mx);
    for (int j = 0; j < d; ++j) {
      double num = 0.0;
      for (int64_t s = 0; s < n_src; ++s) {
        const uint8_t* c = codes + (size_t)s * o->esz;
        const uint16_t* sc = scales + 2 * (size_t)s;
        num += exp(z[s] - mx) * entry_value(o, c, sc, HD + h * d + j);
      }
      out[h * d + j] = num / den;
    }
  }
  free(z);
  return KVO_OK;
}

/* ------------------------------------------------------------------ */
/* requests and blocks                                                  */
/* ------------------------------------------------------------------ */

static int req_ok(const kvo_t* o, int32_t r) { return r >= 0 && r < o->c.max_requests && o->reqs[r].active; }

int kvo_alloc_request(kvo_t* o, int32_t* out) {
  if (!o || !out) return KVO_ERR_INVALID_ARG;
  for (int32_t r = 0; r < o->c.max_requests; ++r) {
    request* q = &o->reqs[r];
    if (q->active) continue;
    if (!q->layers) {
      q->table = (int32_t*)calloc((size_t)o->c.max_blocks_per_request, sizeof(int32_t));
      q->layers = (req_layer*)calloc((size_t)o->c.n_layers, sizeof(req_layer));
      for (int l = 0; l < o->c.n_layers; ++l) {
        req_layer* rl = &q->layers[l];
        rl->win_code = (uint8_t*)calloc((size_t)o->c.n_win, (size_t)o->esz);
        rl->win_scale = (uint16_t*)calloc((size_t)o->c.n_win * 2, 2);
        rl->tail_kv = (float*)calloc((size_t)o->c.m_prime * 2 * o->HD, sizeof(float));
        rl->tail_idx = (float*)calloc((size_t)o->c.m * o->XD, sizeof(float));
        rl->hca_new = (uint8_t*)calloc(1, (size_t)o->esz);
        sec_alloc(o, &rl->stage);
      }
    }
    q->active = 1;
    q->L = 0;
    q->n_sealed = 0;
    for (int l = 0; l < o->c.n_layers; ++l) {
      q->layers[l].tail_len = 0;
      q->layers[l].tail_idx_len = 0;
    }
    *out = r;
    return KVO_OK;
  }
  return KVO_ERR_OUT_OF_REQUESTS;
}

static int32_t block_take(kvo_t* o) { /* smallest free id */
  for (int32_t b = o->block_hint; b < o->c.max_blocks; ++b) {
    if (o->blocks[b].refcount == 0) {
      o->blocks[b].refcount = 1;
      o->n_free_blocks -= 1;
      o->block_hint = b + 1;
      if (!o->blocks[b].layers) {
        o->blocks[b].layers = (layer_sec*)calloc((size_t)o->c.n_layers, sizeof(layer_sec));
        for (int l = 0; l < o->c.n_layers; ++l) sec_alloc(o, &o->blocks[b].layers[l]);
      }
      return b;
    }
  }
  return -1; /* callers check n_free_blocks first */
}

/* HiSparse slots: smallest free; without HiSparse a block's CSA entries stay
 * with the block (location = its id) */
static int32_t hot_take(kvo_t* o) {
  for (int32_t i = 0; i < o->c.csa_hot_slots; ++i)
    if (!o->hot_used[i]) {
      o->hot_used[i] = 1;
      o->hot_free -= 1;
      return i;
    }
  return -1; /* callers check hot_free first */
}

static int32_t host_take(kvo_t* o) {
  for (int32_t i = 0; i < o->c.csa_host_slots; ++i)
    if (!o->host_used[i]) {
      o->host_used[i] = 1;
      o->host_free -= 1;
      return i;
    }
  return -1;
}

static void loc_release(kvo_t* o, int32_t loc) {
  if (!o->hisparse) return;
  if (loc >= 0) {
    o->hot_used[loc] = 0;
    o->hot_free += 1;
  } else {
    o->host_used[-1 - loc] = 0;
    o->host_free += 1;
  }
}

/* a block id just taken (sealed or restored): its CSA entries go to a hot slot */
static void place_new_block(kvo_t* o, int32_t b) {
  o->blocks[b].loc = o->hisparse ? hot_take(o) : b;
  o->blocks[b].last_used = o->epoch;
}

static void block_release(kvo_t* o, int32_t b) {
  o->blocks[b].refcount -= 1;
  if (o->blocks[b].refcount == 0) {
    o->n_free_blocks += 1;
    if (b < o->block_hint) o->block_hint = b;
    loc_release(o, o->blocks[b].loc);
  }
}

int kvo_free_request(kvo_t* o, int32_t r) {
  if (!o) return KVO_ERR_INVALID_ARG;
  if (!req_ok(o, r)) return KVO_ERR_BAD_REQUEST;
  request* q = &o->reqs[r];
  for (int s = 0; s < q->n_sealed; ++s) block_release(o, q->table[s]);
  q->active = 0;
  q->L = 0;
  q->n_sealed = 0;
  return KVO_OK;
}

/* window: the token at position pos goes to slot pos % W, overwriting the
 * token that has just left the window ([P1] s4: the oldest drops) */
static void window_put(kvo_t* o, req_layer* rl, int64_t pos, const float* kv) {
  int64_t slot = pos % o->c.n_win;
  uint8_t* code = rl->win_code + (size_t)slot * o->esz;
  uint16_t* sc = rl->win_scale + 2 * (size_t)slot;
  sc[0] = sc[1] = 0;
  kvo_encode(o->c.cache_dtype, kv, o->HD, code, &sc[0]);
  kvo_encode(o->c.cache_dtype, kv + o->HD, o->HD, code + (size_t)o->HD * o->vs, &sc[1]);
}

/* One new token of one request through one layer, in the order of [P1] s4:
 * into the tail; compress when a group completes.  Returns nothing; sealing
 * (which spans all layers) is done by the caller. */
static void token_into_layer(kvo_t* o, request* q, int l, const float* kv, const float* idx) {
  req_layer* rl = &q->layers[l];
  int HD2 = 2 * o->HD;
  int64_t pos = q->L; /* position of this token */
  if (has_csa(o, l) || has_hca(o, l)) {
    memcpy(rl->tail_kv + (size_t)rl->tail_len * HD2, kv, sizeof(float) * (size_t)HD2);
    rl->tail_len += 1;
  }
  if (has_csa(o, l)) {
    if (o->c.idx_per_token) { /* the token's own indexer key, at its place in the block */
      int slot = (int)(pos % o->c.m_prime);
      kvo_encode(o->idx_dtype, idx, o->XD, rl->stage.idx_code + (size_t)slot * o->xsz, rl->stage.idx_scale + slot);
    } else {
      memcpy(rl->tail_idx + (size_t)rl->tail_idx_len * o->XD, idx, sizeof(float) * (size_t)o->XD);
      rl->tail_idx_len += 1;
    }
    if ((pos + 1) % o->c.m == 0) { /* a CSA group of m tokens is complete */
      int64_t g = (pos + 1) / o->c.m - 1;
      int slot = (int)(g % o->CB);
      const float* group = rl->tail_kv + (size_t)(rl->tail_len - o->c.m) * HD2;
      kvo_compress_kv(o, l, 1, group, rl->stage.csa_code + (size_t)slot * o->esz, rl->stage.csa_scale + 2 * slot);
      if (!o->c.idx_per_token)
        kvo_compress_idx(o, l, rl->tail_idx, rl->stage.idx_code + (size_t)slot * o->xsz, rl->stage.idx_scale + slot);
      rl->tail_idx_len = 0;
    }
  }
  if (has_hca(o, l) && (pos + 1) % o->c.m_prime == 0) /* an HCA group of m' tokens is complete */
    kvo_compress_kv(o, l, 2, rl->tail_kv, rl->hca_new, rl->hca_new_scale);
  if ((pos + 1) % o->c.m_prime == 0) rl->tail_len = 0; /* block boundary: the tail empties */
  window_put(o, rl, pos, kv);
}

/* the block of m' tokens ending at the current length is complete: give it
 * the smallest free id and move the staged entries in ([P1] s2.2, [P3] s2.2) */
static void seal_block(kvo_t* o, request* q) {
  int32_t id = block_take(o);
  place_new_block(o, id);
  block* b = &o->blocks[id];
  for (int l = 0; l < o->c.n_layers; ++l) {
    req_layer* rl = &q->layers[l];
    layer_sec* dst = &b->layers[l];
    if (has_csa(o, l)) {
      memcpy(dst->csa_code, rl->stage.csa_code, (size_t)o->CB * o->esz);
      memcpy(dst->csa_scale, rl->stage.csa_scale, (size_t)o->CB * 2 * 2);
      memcpy(dst->idx_code, rl->stage.idx_code, (size_t)o->XB * o->xsz);
      memcpy(dst->idx_scale, rl->stage.idx_scale, (size_t)o->XB * 2);
    }
    if (has_hca(o, l)) {
      memcpy(dst->hca_code, rl->hca_new, (size_t)o->esz);
      dst->hca_scale[0] = rl->hca_new_scale[0];
      dst->hca_scale[1] = rl->hca_new_scale[1];
    }
  }
  q->table[q->n_sealed] = id;
  q->n_sealed += 1;
}

static int any_csa(const kvo_t* o) {
  for (int l = 0; l < o->c.n_layers; ++l)
    if (has_csa(o, l)) return 1;
  return 0;
}

int kvo_append(kvo_t* o, int n, const int32_t* req_ids, const int32_t* n_new, const float* k, const float* v,
               const float* idx_k) {
  if (!o || n < 0 || (n > 0 && (!req_ids || !n_new))) return KVO_ERR_INVALID_ARG;
  /* validate the whole batch before changing anything */
  int64_t T = 0, seals = 0;
  for (int i = 0; i < n; ++i) {
    if (!req_ok(o, req_ids[i])) return KVO_ERR_BAD_REQUEST;
    if (n_new[i] < 0) return KVO_ERR_INVALID_ARG;
    for (int j = 0; j < i; ++j)
      if (req_ids[j] == req_ids[i]) return KVO_ERR_INVALID_ARG;
    int64_t L0 = o->reqs[req_ids[i]].L, L1 = L0 + n_new[i];
    if (L1 / o->c.m_prime > o->c.max_blocks_per_request) return KVO_ERR_CAPACITY;
    T += n_new[i];
    seals += L1 / o->c.m_prime - L0 / o->c.m_prime;
  }
  if (T > 0 && (!k || !v || (any_csa(o) && !idx_k))) return KVO_ERR_INVALID_ARG;
  if (seals > o->n_free_blocks || (o->hisparse && seals > o->hot_free)) return KVO_ERR_OUT_OF_BLOCKS;

  int HD = o->HD, XD = o->XD;
  float* kv = (float*)malloc(sizeof(float) * 2 * (size_t)HD);
  int64_t row = 0;
  for (int i = 0; i < n; ++i) {
    request* q = &o->reqs[req_ids[i]];
    for (int t = 0; t < n_new[i]; ++t, ++row) {
      for (int l = 0; l < o->c.n_layers; ++l) {
        /* gather this token's K and V into one [2][H][d] row */
        memcpy(kv, k + ((size_t)l * T + row) * HD, sizeof(float) * (size_t)HD);
        memcpy(kv + HD, v + ((size_t)l * T + row) * HD, sizeof(float) * (size_t)HD);
        const float* idx = has_csa(o, l) ? idx_k + ((size_t)l * T + row) * XD : NULL;
        token_into_layer(o, q, l, kv, idx);
      }
      q->L += 1;
      if (q->L % o->c.m_prime == 0) seal_block(o, q);
    }
  }
  free(kv);
  return KVO_OK;
}

int kvo_share_prefix(kvo_t* o, int32_t dst, int32_t src, int64_t n_tokens, const float* win_k, const float* win_v) {
  if (!o) return KVO_ERR_INVALID_ARG;
  if (!req_ok(o, dst) || !req_ok(o, src) || dst == src) return KVO_ERR_BAD_REQUEST;
  if (n_tokens <= 0) return KVO_ERR_INVALID_ARG;
  request* s = &o->reqs[src];
  request* d = &o->reqs[dst];
  if (n_tokens % o->c.m_prime != 0 || n_tokens / o->c.m_prime > s->n_sealed) return KVO_ERR_NOT_SHAREABLE;
  if (d->L != 0) return KVO_ERR_NOT_SHAREABLE;
  if (!win_k || !win_v) return KVO_ERR_INVALID_ARG;
  int nb = (int)(n_tokens / o->c.m_prime);
  for (int b = 0; b < nb; ++b) {
    d->table[b] = s->table[b];
    o->blocks[s->table[b]].refcount += 1;
  }
  d->n_sealed = nb;
  d->L = n_tokens;
  int64_t w = n_tokens < o->c.n_win ? n_tokens : o->c.n_win;
  int HD = o->HD;
  float* kv = (float*)malloc(sizeof(float) * 2 * (size_t)HD);
  for (int l = 0; l < o->c.n_layers; ++l) {
    req_layer* rl = &d->layers[l];
    rl->tail_len = 0;
    rl->tail_idx_len = 0;
    for (int64_t t = 0; t < w; ++t) {
      memcpy(kv, win_k + ((size_t)l * w + t) * HD, sizeof(float) * (size_t)HD);
      memcpy(kv + HD, win_v + ((size_t)l * w + t) * HD, sizeof(float) * (size_t)HD);
      window_put(o, rl, n_tokens - w + t, kv);
    }
  }
  free(kv);
  return KVO_OK;
}

/* CSA or indexer entry e of a request: in a sealed block or still staged */
static void locate_entry(const kvo_t* o, int l, const request* q, int kind, int64_t e, const uint8_t** code,
                         const uint16_t** scale) {
  int64_t seg = e / o->CB;
  int slot = (int)(e % o->CB);
  const layer_sec* sec = seg < q->n_sealed ? &o->blocks[q->table[seg]].layers[l] : &q->layers[l].stage;
  if (kind == 1) {
    *code = sec->csa_code + (size_t)slot * o->esz;
    *scale = sec->csa_scale + 2 * slot;
  } else { /* per-token keys: the entry's first token; its m tokens follow */
    const int ks = o->c.idx_per_token ? slot * o->c.m : slot;
    *code = sec->idx_code + (size_t)ks * o->xsz;
    *scale = sec->idx_scale + ks;
  }
}

/* indexer score of a CSA entry located by locate_entry (kind 3) */
static float entry_score(const kvo_t* o, int l, const uint8_t* code, const uint16_t* scale, const float* q_idx) {
  return o->c.idx_per_token ? kvo_score_tokens(o, l, code, scale, q_idx) : kvo_score(o, code, scale, q_idx);
}

int kvo_decode_attend(kvo_t* o, int layer, int n, const int32_t* req_ids, const float* q, const float* q_idx,
                      int top_k, double* out, int32_t* topk) {
  if (!o || layer < 0 || layer >= o->c.n_layers || n < 0 || top_k < 0) return KVO_ERR_INVALID_ARG;
  if (n > 0 && (!req_ids || !q || !out || (has_csa(o, layer) && !q_idx))) return KVO_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    if (!req_ok(o, req_ids[i])) return KVO_ERR_BAD_REQUEST;
    if (o->reqs[req_ids[i]].L == 0) return KVO_ERR_INVALID_ARG;
  }
  int HD = o->HD, XD = o->XD;
  o->epoch += 1; /* this call's epoch */
  for (int i = 0; i < n; ++i) {
    const request* r = &o->reqs[req_ids[i]];
    int64_t N_c = has_csa(o, layer) ? r->L / o->c.m : 0;
    int64_t N_h = has_hca(o, layer) ? r->L / o->c.m_prime : 0;
    int64_t w = r->L < o->c.n_win ? r->L : o->c.n_win;
    int64_t kk = N_c < top_k ? N_c : top_k;
    int32_t* sel = (int32_t*)malloc(sizeof(int32_t) * (size_t)(top_k > 0 ? top_k : 1));
    if (N_c > 0) {
      float* s = (float*)malloc(sizeof(float) * (size_t)N_c);
      for (int64_t e = 0; e < N_c; ++e) {
        const uint8_t* c;
        const uint16_t* sc;
        locate_entry(o, layer, r, 3, e, &c, &sc);
        s[e] = entry_score(o, layer, c, sc, q_idx + (size_t)i * XD);
      }
      kvo_topk(s, N_c, top_k, sel);
      free(s);
    } else {
      for (int j = 0; j < top_k; ++j) sel[j] = -1;
    }
    if (topk)
      for (int j = 0; j < top_k; ++j) topk[(size_t)i * top_k + j] = sel[j];
    for (int64_t j = 0; j < kk; ++j) { /* activity: the blocks of the selected sealed entries */
      const int64_t seg = sel[j] / o->CB;
      if (seg < r->n_sealed) o->blocks[r->table[seg]].last_used = o->epoch;
    }
    /* sources: [selected CSA entries | every HCA entry | the window] */
    int64_t n_src = kk + N_h + w;
    uint8_t* codes = (uint8_t*)malloc((size_t)n_src * o->esz);
    uint16_t* scales = (uint16_t*)malloc((size_t)n_src * 2 * 2);
    int64_t s = 0;
    for (int64_t j = 0; j < kk; ++j, ++s) {
      const uint8_t* c;
      const uint16_t* sc;
      locate_entry(o, layer, r, 1, sel[j], &c, &sc);
      memcpy(codes + (size_t)s * o->esz, c, (size_t)o->esz);
      memcpy(scales + 2 * (size_t)s, sc, 4);
    }
    for (int64_t t = 0; t < N_h; ++t, ++s) {
      const layer_sec* sec = &o->blocks[r->table[t]].layers[layer];
      memcpy(codes + (size_t)s * o->esz, sec->hca_code, (size_t)o->esz);
      memcpy(scales + 2 * (size_t)s, sec->hca_scale, 4);
    }
    for (int64_t p = r->L - w; p < r->L; ++p, ++s) {
      int64_t slot = p % o->c.n_win;
      memcpy(codes + (size_t)s * o->esz, r->layers[layer].win_code + (size_t)slot * o->esz, (size_t)o->esz);
      memcpy(scales + 2 * (size_t)s, r->layers[layer].win_scale + 2 * (size_t)slot, 4);
    }
    kvo_attend_sources(o, n_src, codes, scales, q + (size_t)i * HD, out + (size_t)i * HD);
    free(codes);
    free(scales);
    free(sel);
  }
  return KVO_OK;
}

/* ------------------------------------------------------------------ */
/* inspection                                                           */
/* ------------------------------------------------------------------ */

int kvo_request_info(const kvo_t* o, int32_t r, kvo_info* info, int32_t* ids, int32_t cap) {
  if (!o || !info) return KVO_ERR_INVALID_ARG;
  if (!req_ok(o, r)) return KVO_ERR_BAD_REQUEST;
  const request* q = &o->reqs[r];
  info->length = q->L;
  info->n_csa = q->L / o->c.m;
  info->n_hca = q->L / o->c.m_prime;
  info->csa_tail = (int32_t)(q->L % o->c.m);
  info->hca_tail = (int32_t)(q->L % o->c.m_prime);
  info->n_blocks = q->n_sealed;
  info->window = (int32_t)(q->L < o->c.n_win ? q->L : o->c.n_win);
  if (ids)
    for (int32_t s = 0; s < q->n_sealed && s < cap; ++s) ids[s] = q->table[s];
  return KVO_OK;
}

int kvo_block_refcount(const kvo_t* o, int32_t b) {
  if (!o || b < 0 || b >= o->c.max_blocks) return KVO_ERR_INVALID_ARG;
  return o->blocks[b].refcount;
}

int kvo_free_block_count(const kvo_t* o) { return o ? o->n_free_blocks : KVO_ERR_INVALID_ARG; }

int kvo_block_entry(const kvo_t* o, int l, int32_t b, int kind, int slot, uint8_t* code, uint16_t* scale) {
  if (!o || l < 0 || l >= o->c.n_layers || b < 0 || b >= o->c.max_blocks) return KVO_ERR_INVALID_ARG;
  if (o->blocks[b].refcount == 0 || !o->blocks[b].layers) return KVO_ERR_INVALID_ARG;
  const layer_sec* sec = &o->blocks[b].layers[l];
  if (kind == 1 && has_csa(o, l) && slot >= 0 && slot < o->CB) {
    memcpy(code, sec->csa_code + (size_t)slot * o->esz, (size_t)o->esz);
    memcpy(scale, sec->csa_scale + 2 * slot, 4);
  } else if (kind == 2 && has_hca(o, l) && slot == 0) {
    memcpy(code, sec->hca_code, (size_t)o->esz);
    memcpy(scale, sec->hca_scale, 4);
  } else if (kind == 3 && has_csa(o, l) && slot >= 0 && slot < o->XB) {
    memcpy(code, sec->idx_code + (size_t)slot * o->xsz, (size_t)o->xsz);
    scale[0] = sec->idx_scale[slot];
  } else {
    return KVO_ERR_INVALID_ARG;
  }
  return KVO_OK;
}

int kvo_request_entry(const kvo_t* o, int l, int32_t r, int kind, int64_t e, uint8_t* code, uint16_t* scale) {
  if (!o || l < 0 || l >= o->c.n_layers || (kind != 1 && kind != 3) || !has_csa(o, l)) return KVO_ERR_INVALID_ARG;
  if (!req_ok(o, r)) return KVO_ERR_BAD_REQUEST;
  const request* q = &o->reqs[r];
  if (kind == 3 && o->c.idx_per_token) { /* per-token keys: e is a token position */
    if (e < 0 || e >= q->L) return KVO_ERR_INVALID_ARG;
    const int64_t seg = e / o->c.m_prime;
    const int slot = (int)(e % o->c.m_prime);
    const layer_sec* sec = seg < q->n_sealed ? &o->blocks[q->table[seg]].layers[l] : &q->layers[l].stage;
    memcpy(code, sec->idx_code + (size_t)slot * o->xsz, (size_t)o->xsz);
    scale[0] = sec->idx_scale[slot];
    return KVO_OK;
  }
  if (e < 0 || e >= q->L / o->c.m) return KVO_ERR_INVALID_ARG;
  const uint8_t* c;
  const uint16_t* sc;
  locate_entry(o, l, q, kind, e, &c, &sc);
  if (kind == 1) {
    memcpy(code, c, (size_t)o->esz);
    memcpy(scale, sc, 4);
  } else {
    memcpy(code, c, (size_t)o->xsz);
    scale[0] = sc[0];
  }
  return KVO_OK;
}

int kvo_window_token(const kvo_t* o, int l, int32_t r, int64_t pos, uint8_t* code, uint16_t* scale) {
  if (!o || l < 0 || l >= o->c.n_layers) return KVO_ERR_INVALID_ARG;
  if (!req_ok(o, r)) return KVO_ERR_BAD_REQUEST;
  const request* q = &o->reqs[r];
  if (pos < 0 || pos >= q->L || pos < q->L - o->c.n_win) return KVO_ERR_INVALID_ARG;
  int64_t slot = pos % o->c.n_win;
  memcpy(code, q->layers[l].win_code + (size_t)slot * o->esz, (size_t)o->esz);
  memcpy(scale, q->layers[l].win_scale + 2 * (size_t)slot, 4);
  return KVO_OK;
}

int kvo_request_scores(const kvo_t* o, int l, int32_t r, const float* q_idx, float* out) {
  if (!o || l < 0 || l >= o->c.n_layers || !has_csa(o, l)) return KVO_ERR_INVALID_ARG;
  if (!req_ok(o, r)) return KVO_ERR_BAD_REQUEST;
  const request* q = &o->reqs[r];
  for (int64_t e = 0; e < q->L / o->c.m; ++e) {
    const uint8_t* c;
    const uint16_t* sc;
    locate_entry(o, l, q, 3, e, &c, &sc);
    out[e] = entry_score(o, l, c, sc, q_idx);
  }
  return KVO_OK;
}

/* ------------------------------------------------------------------ */
/* prefix images ([P3] s3, s3.1; [P4])                                   */
/* ------------------------------------------------------------------ */

uint64_t kvo_fingerprint(const kvo_t* o) { return o ? o->fingerprint : 0; }

static int64_t round16(int64_t x) { return (x + 15) / 16 * 16; }
static int idx_has_scale(const kvo_t* o) { return o->idx_dtype == KVO_FP8 || o->idx_dtype == KVO_FP4; }
/* bytes of one K/V entry record: codes, then fp8 scales and zero padding */
static int64_t entry_rec(const kvo_t* o) { return o->esz + (o->c.cache_dtype == KVO_FP8 ? 16 : 0); }
/* one run of CB indexer keys: codes chunk-major, then fp8 / FP4 scales padded
 * to 16 bytes; a block holds XB / CB runs (one, or m with per-token keys) */
static int64_t idx_run(const kvo_t* o) {
  return (int64_t)o->CB * o->xsz + (idx_has_scale(o) ? round16(2 * (int64_t)o->CB) : 0);
}
static int64_t idx_part(const kvo_t* o) { return (int64_t)(o->XB / o->CB) * idx_run(o); }
/* bytes of one block's parts summed over the layers */
static int64_t block_rec(const kvo_t* o) {
  int64_t b = 0;
  for (int l = 0; l < o->c.n_layers; ++l) {
    if (has_csa(o, l)) b += o->CB * entry_rec(o) + idx_part(o);
    if (has_hca(o, l)) b += entry_rec(o);
  }
  return b;
}

static void put_u32(uint8_t* p, uint32_t v) {
  for (int i = 0; i < 4; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
static void put_u64(uint8_t* p, uint64_t v) {
  for (int i = 0; i < 8; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
static uint32_t get_u32(const uint8_t* p) {
  uint32_t v = 0;
  for (int i = 0; i < 4; ++i) v |= (uint32_t)p[i] << (8 * i);
  return v;
}
static uint64_t get_u64(const uint8_t* p) {
  uint64_t v = 0;
  for (int i = 0; i < 8; ++i) v |= (uint64_t)p[i] << (8 * i);
  return v;
}

static const uint32_t kImageMagic = 0x4950564Bu; /* "KVPI" */

/* the chunk-by-chunk indexer layout needs whole 16-byte chunks per key */
static int image_ok(const kvo_t* o) { return !any_csa(o) || o->xsz % 16 == 0; }

int64_t kvo_image_bytes(const kvo_t* o, int64_t n_tokens, uint32_t flags) {
  if (!o || !image_ok(o) || n_tokens <= 0 || n_tokens % o->c.m_prime != 0) return -1;
  const int64_t nb = n_tokens / o->c.m_prime;
  const int64_t w = (flags & KVO_IMAGE_WINDOW) ? (n_tokens < o->c.n_win ? n_tokens : o->c.n_win) : 0;
  return 64 + nb * block_rec(o) + w * entry_rec(o) * o->c.n_layers;
}

/* one K/V entry record from codes + scales */
static void entry_to_rec(const kvo_t* o, const uint8_t* code, const uint16_t* scale, uint8_t* rec) {
  memcpy(rec, code, (size_t)o->esz);
  if (o->c.cache_dtype == KVO_FP8) {
    uint8_t* t = rec + o->esz;
    memset(t, 0, 16);
    t[0] = (uint8_t)scale[0];
    t[1] = (uint8_t)(scale[0] >> 8);
    t[2] = (uint8_t)scale[1];
    t[3] = (uint8_t)(scale[1] >> 8);
  }
}

static void rec_to_entry(const kvo_t* o, const uint8_t* rec, uint8_t* code, uint16_t* scale) {
  memcpy(code, rec, (size_t)o->esz);
  if (o->c.cache_dtype == KVO_FP8) {
    const uint8_t* t = rec + o->esz;
    scale[0] = (uint16_t)(t[0] | (t[1] << 8));
    scale[1] = (uint16_t)(t[2] | (t[3] << 8));
  } else {
    scale[0] = scale[1] = 0;
  }
}

/* a block's indexer part: keys chunk by chunk, then the scales */
static void idx_to_part(const kvo_t* o, const layer_sec* s, uint8_t* part) {
  memset(part, 0, (size_t)idx_part(o));
  for (int q = 0; q < o->XB / o->CB; ++q) {
    uint8_t* run = part + q * idx_run(o);
    for (int e = 0; e < o->CB; ++e)
      for (int j = 0; j < o->xsz; ++j)
        run[((int64_t)(j / 16) * o->CB + e) * 16 + j % 16] = s->idx_code[(size_t)(q * o->CB + e) * o->xsz + j];
    if (idx_has_scale(o)) {
      uint8_t* t = run + (int64_t)o->CB * o->xsz;
      for (int e = 0; e < o->CB; ++e) {
        t[2 * e] = (uint8_t)s->idx_scale[q * o->CB + e];
        t[2 * e + 1] = (uint8_t)(s->idx_scale[q * o->CB + e] >> 8);
      }
    }
  }
}

static void part_to_idx(const kvo_t* o, const uint8_t* part, layer_sec* s) {
  for (int q = 0; q < o->XB / o->CB; ++q) {
    const uint8_t* run = part + q * idx_run(o);
    for (int e = 0; e < o->CB; ++e)
      for (int j = 0; j < o->xsz; ++j)
        s->idx_code[(size_t)(q * o->CB + e) * o->xsz + j] = run[((int64_t)(j / 16) * o->CB + e) * 16 + j % 16];
    const uint8_t* t = run + (int64_t)o->CB * o->xsz;
    for (int e = 0; e < o->CB; ++e)
      s->idx_scale[q * o->CB + e] = idx_has_scale(o) ? (uint16_t)(t[2 * e] | (t[2 * e + 1] << 8)) : 0;
  }
}

int kvo_export_prefix(const kvo_t* o, int32_t req, int64_t n_tokens, uint32_t flags, uint8_t* image, int64_t cap) {
  if (!o || !image || (flags & ~KVO_IMAGE_WINDOW) || !image_ok(o)) return KVO_ERR_INVALID_ARG;
  if (!req_ok(o, req)) return KVO_ERR_BAD_REQUEST;
  const request* q = &o->reqs[req];
  if (n_tokens <= 0 || n_tokens % o->c.m_prime != 0 || n_tokens / o->c.m_prime > q->n_sealed)
    return KVO_ERR_NOT_SHAREABLE;
  if ((flags & KVO_IMAGE_WINDOW) && n_tokens != q->L) return KVO_ERR_NOT_SHAREABLE;
  const int64_t total = kvo_image_bytes(o, n_tokens, flags);
  if (cap < total) return KVO_ERR_INVALID_ARG;
  const int64_t nb = n_tokens / o->c.m_prime, E = entry_rec(o), X = idx_part(o);
  const int64_t w = (flags & KVO_IMAGE_WINDOW) ? (n_tokens < o->c.n_win ? n_tokens : o->c.n_win) : 0;

  memset(image, 0, 64);
  put_u32(image, kImageMagic);
  put_u32(image + 4, 1);
  put_u64(image + 8, o->fingerprint);
  put_u64(image + 16, (uint64_t)n_tokens);
  put_u32(image + 24, (uint32_t)nb);
  put_u32(image + 28, (uint32_t)w);
  put_u64(image + 32, (uint64_t)(nb * block_rec(o)));
  put_u64(image + 40, (uint64_t)(w * E * o->c.n_layers));
  put_u64(image + 48, (uint64_t)total);

  uint8_t* p = image + 64;
  for (int l = 0; l < o->c.n_layers; ++l) {
    if (has_csa(o, l)) {
      for (int64_t b = 0; b < nb; ++b) {
        const layer_sec* s = &o->blocks[q->table[b]].layers[l];
        for (int e = 0; e < o->CB; ++e, p += E) entry_to_rec(o, s->csa_code + (size_t)e * o->esz, s->csa_scale + 2 * e, p);
      }
      for (int64_t b = 0; b < nb; ++b, p += X) idx_to_part(o, &o->blocks[q->table[b]].layers[l], p);
    }
    if (has_hca(o, l))
      for (int64_t b = 0; b < nb; ++b, p += E) {
        const layer_sec* s = &o->blocks[q->table[b]].layers[l];
        entry_to_rec(o, s->hca_code, s->hca_scale, p);
      }
  }
  for (int l = 0; l < o->c.n_layers && w > 0; ++l) {
    const req_layer* rl = &q->layers[l];
    for (int64_t pos = n_tokens - w; pos < n_tokens; ++pos, p += E) {
      const int64_t slot = pos % o->c.n_win;
      entry_to_rec(o, rl->win_code + (size_t)slot * o->esz, rl->win_scale + 2 * slot, p);
    }
  }
  return KVO_OK;
}

int kvo_import_prefix(kvo_t* o, int32_t dst, const uint8_t* image, int64_t bytes, const float* win_k,
                      const float* win_v) {
  if (!o || !image || !image_ok(o)) return KVO_ERR_INVALID_ARG;
  if (!req_ok(o, dst)) return KVO_ERR_BAD_REQUEST;
  if (bytes < 64 || get_u32(image) != kImageMagic || get_u32(image + 4) != 1 || get_u64(image + 8) != o->fingerprint)
    return KVO_ERR_BAD_IMAGE;
  const int64_t n_tokens = (int64_t)get_u64(image + 16);
  const int64_t nb = (int64_t)get_u32(image + 24), w = (int64_t)get_u32(image + 28);
  const uint32_t flags = w > 0 ? KVO_IMAGE_WINDOW : 0;
  const int64_t total = kvo_image_bytes(o, n_tokens, flags);
  const int64_t w_full = n_tokens < o->c.n_win ? n_tokens : o->c.n_win;
  if (total < 0 || nb != n_tokens / o->c.m_prime || (w != 0 && w != w_full) || bytes < total ||
      get_u64(image + 48) != (uint64_t)total || get_u64(image + 32) != (uint64_t)(nb * block_rec(o)) ||
      get_u64(image + 40) != (uint64_t)(w * entry_rec(o) * o->c.n_layers))
    return KVO_ERR_BAD_IMAGE;
  request* q = &o->reqs[dst];
  if (q->L != 0) return KVO_ERR_NOT_SHAREABLE;
  if (w == 0 && (!win_k || !win_v)) return KVO_ERR_INVALID_ARG;
  if (nb > o->c.max_blocks_per_request) return KVO_ERR_CAPACITY;
  if (nb > o->n_free_blocks || (o->hisparse && nb > o->hot_free)) return KVO_ERR_OUT_OF_BLOCKS;

  const int64_t E = entry_rec(o), X = idx_part(o);
  for (int64_t b = 0; b < nb; ++b) {
    q->table[b] = block_take(o);
    place_new_block(o, q->table[b]);
  }
  q->n_sealed = (int)nb;
  q->L = n_tokens;
  const uint8_t* p = image + 64;
  for (int l = 0; l < o->c.n_layers; ++l) {
    req_layer* rl = &q->layers[l];
    rl->tail_len = 0;
    rl->tail_idx_len = 0;
    if (has_csa(o, l)) {
      for (int64_t b = 0; b < nb; ++b) {
        layer_sec* s = &o->blocks[q->table[b]].layers[l];
        for (int e = 0; e < o->CB; ++e, p += E) rec_to_entry(o, p, s->csa_code + (size_t)e * o->esz, s->csa_scale + 2 * e);
      }
      for (int64_t b = 0; b < nb; ++b, p += X) part_to_idx(o, p, &o->blocks[q->table[b]].layers[l]);
    }
    if (has_hca(o, l))
      for (int64_t b = 0; b < nb; ++b, p += E) {
        layer_sec* s = &o->blocks[q->table[b]].layers[l];
        rec_to_entry(o, p, s->hca_code, s->hca_scale);
      }
  }
  if (w > 0) {
    for (int l = 0; l < o->c.n_layers; ++l) {
      req_layer* rl = &q->layers[l];
      for (int64_t pos = n_tokens - w; pos < n_tokens; ++pos, p += E) {
        const int64_t slot = pos % o->c.n_win;
        rec_to_entry(o, p, rl->win_code + (size_t)slot * o->esz, rl->win_scale + 2 * slot);
      }
    }
  } else { /* Zero SWA: the caller's recomputed window goes through the cache encoding */
    float* kv = (float*)malloc(sizeof(float) * 2 * (size_t)o->HD);
    for (int l = 0; l < o->c.n_layers; ++l)
      for (int64_t t = 0; t < w_full; ++t) {
        memcpy(kv, win_k + ((size_t)l * w_full + t) * o->HD, sizeof(float) * (size_t)o->HD);
        memcpy(kv + o->HD, win_v + ((size_t)l * w_full + t) * o->HD, sizeof(float) * (size_t)o->HD);
        window_put(o, &q->layers[l], n_tokens - w_full + t, kv);
      }
    free(kv);
  }
  return KVO_OK;
}

/* ------------------------------------------------------------------ */
/* HiSparse placement                                                   */
/* ------------------------------------------------------------------ */

int kvo_block_location(const kvo_t* o, int32_t b, int32_t* loc, uint32_t* last_used) {
  if (!o || b < 0 || b >= o->c.max_blocks || o->blocks[b].refcount == 0) return KVO_ERR_INVALID_ARG;
  if (loc) *loc = o->blocks[b].loc;
  if (last_used) *last_used = o->blocks[b].last_used;
  return KVO_OK;
}

uint32_t kvo_epoch(const kvo_t* o) { return o ? o->epoch : 0; }

int kvo_inactive_blocks(const kvo_t* o, uint32_t idle, int32_t* ids, int32_t cap) {
  if (!o || cap < 0 || (cap > 0 && !ids)) return KVO_ERR_INVALID_ARG;
  int n = 0;
  for (int32_t b = 0; b < o->c.max_blocks; ++b) {
    const block* x = &o->blocks[b];
    if (x->refcount == 0 || x->loc < 0 || o->epoch - x->last_used < idle) continue;
    if (n < cap) ids[n] = b;
    ++n;
  }
  return n;
}

/* a list of distinct live block ids, all resident (want_hot) or all offloaded */
static int ids_ok(const kvo_t* o, int n, const int32_t* ids, int want_hot) {
  if (!o->hisparse || n < 0 || (n > 0 && !ids)) return 0;
  for (int i = 0; i < n; ++i) {
    const int32_t b = ids[i];
    if (b < 0 || b >= o->c.max_blocks || o->blocks[b].refcount == 0) return 0;
    if ((o->blocks[b].loc >= 0) != want_hot) return 0;
    for (int j = 0; j < i; ++j)
      if (ids[j] == b) return 0;
  }
  return 1;
}

int kvo_offload(kvo_t* o, int n, const int32_t* ids) {
  if (!o || !ids_ok(o, n, ids, 1)) return KVO_ERR_INVALID_ARG;
  if (n > o->host_free) return KVO_ERR_OUT_OF_BLOCKS;
  for (int i = 0; i < n; ++i) {
    block* x = &o->blocks[ids[i]];
    const int32_t h = host_take(o);
    loc_release(o, x->loc);
    x->loc = -1 - h;
  }
  return KVO_OK;
}

int kvo_fetch(kvo_t* o, int n, const int32_t* ids) {
  if (!o || !ids_ok(o, n, ids, 0)) return KVO_ERR_INVALID_ARG;
  if (n > o->hot_free) return KVO_ERR_OUT_OF_BLOCKS;
  for (int i = 0; i < n; ++i) {
    block* x = &o->blocks[ids[i]];
    const int32_t h = hot_take(o);
    loc_release(o, x->loc);
    x->loc = h;
    x->last_used = o->epoch;
  }
  return KVO_OK;
}

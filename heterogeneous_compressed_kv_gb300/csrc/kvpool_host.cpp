// kvpool_host.cpp -- host runtime of the two-pool KV cache: configuration,
// arena layout, block allocator with refcounts, request lifecycle, and the
// launch plans of append / share_prefix / decode_attend.
//
// Bookkeeping follows "Why does V4 split pools? ..." (s2.2: blocks of
// lcm(m, m') tokens; s3.1: tails; s4: one decode step) and "Ch 12 Inference
// framework: heterogeneous KV scheduling" (s2.1: one State block per request,
// freed whole; s2.2: Block cache shared by refcount).  The host never reads
// device memory: every launch carries the per-request lengths, block ids and
// work split it needs in its kernel parameters.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <memory>
#include <new>
#include <cstddef>
#include <set>
#include <string>
#include <vector>

#include "kvpool.h"
#include "kvpool_internal.h"

namespace kvp {
int attend_max_split_len();
}  // namespace kvp

using namespace kvp;

namespace {

constexpr int kMaxSplits = 4096;
// CTA targets per launch, in CTAs per SM (the SM count comes from the device):
// attention CTAs of a part that has the GPU to itself: 3 per SM, of which 2
// are resident at a time (registers); 1.5 waves of shorter splits measured a
// little faster than one wave of longer ones (long context 178.8 vs 180.6 us)
constexpr int kAttendCtasPerSm = 3;
// CTAs of the [HCA | window] part beside the select: 2 per SM, one wave
// (1.5 or 1 per SM left room for the select but the step took 190 / 213 us)
constexpr int kPart0CtasPerSm = 2;
constexpr int kScoreCtasPerSm = 1;      // CTAs of the score kernel (1 per SM, one wave)
constexpr int kSealCopySlices = 8;      // CTAs per sealing unit that copy its staged entries
constexpr int kStagedMinTokens = 16;    // an append call with a unit this long ...
constexpr int kStagedMaxCtasPerSm = 1;  // ... and at most this many CTAs per SM takes the staged path
constexpr int kSplitMinTokens = 64;     // a unit this long in a launch that leaves SMs idle ...
constexpr int kMaxCsaParts = 4;         // ... spreads its CSA groups over up to this many CTAs

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
int value_bytes(int dtype) { return dtype == KVPOOL_F32 ? 4 : dtype == KVPOOL_BF16 ? 2 : 1; }
bool kind_has_csa(int k) { return k == KVPOOL_CSA || k == KVPOOL_CSA_HCA; }

// algorithmic bytes of one indexer entry: its codes and (fp8, fp4) its scale
int64_t idx_algo_bytes(const PoolDesc& pd) {
  const bool scaled = pd.idx_dtype == KVPOOL_FP8_E4M3 || pd.idx_dtype == KVPOOL_FP4_E2M1;
  return pd.idx_entry_bytes + (scaled ? 2 : 0);
}
bool kind_has_hca(int k) { return k == KVPOOL_HCA || k == KVPOOL_CSA_HCA; }

// The smallest run length in [lo, hi] for which the CTAs sum_i ceil(work_i /
// len) fit `cap` (one wave); lo when no length does (more pieces of work than
// CTAs) .  The count falls as the length grows, so a bisection finds it.
int64_t fit_one_wave(const std::vector<int64_t>& work, int64_t lo, int64_t hi, int64_t cap) {
  auto ctas = [&](int64_t len) {
    int64_t c = 0;
    for (int64_t w : work) c += (w + len - 1) / len;
    return c;
  };
  if (lo >= hi || ctas(lo) <= cap || ctas(hi) > cap) return lo;
  while (hi - lo > 1) {  // ctas(lo) > cap >= ctas(hi)
    const int64_t mid = lo + (hi - lo) / 2;
    if (ctas(mid) <= cap) hi = mid;
    else lo = mid;
  }
  return hi;
}

struct Layout {
  PoolDesc pd;
  LayerDesc layers[kMaxLayers];
  int64_t hist, sync, thr, keys, cand, counts, sel, part_o, part_ml;
  int64_t key_stride;
  int32_t max_key_ctas, sel_stride, n_attend_rows;
  int64_t total;
};

// Validate a configuration and compute the arena layout.  Returns "" on
// success or the reason it is refused.
std::string plan_layout(const kvpool_config* c, Layout* out) {
  if (!c) return "config is NULL";
  if (c->m < 1 || c->m_prime < c->m || c->m_prime % c->m != 0)
    return "m must divide m_prime (block = lcm(m, m') = m')";
  if (c->m_prime > 32767) return "m_prime too large";
  if (c->m_prime / c->m > 32) return "at most 32 CSA entries per block";
  if (c->n_win < c->m_prime || c->n_win % c->m_prime != 0) return "n_win must be a positive multiple of m_prime";
  if (c->heads < 1 || (c->head_dim != 64 && c->head_dim != 128)) return "head_dim must be 64 or 128";
  if (c->idx_heads < 1 || c->idx_dim < 1) return "indexer dims must be positive";
  if (c->in_dtype != KVPOOL_F32 && c->in_dtype != KVPOOL_BF16) return "in_dtype must be F32 or BF16";
  if (c->cache_dtype < KVPOOL_F32 || c->cache_dtype > KVPOOL_FP8_E4M3) return "bad cache_dtype";
  if (c->n_layers < 1 || c->n_layers > kMaxLayers || !c->layer_kinds) return "n_layers must be 1..16";
  if (c->max_requests < 1 || c->max_blocks < 1 || c->max_blocks_per_request < 1 || c->max_batch < 1 ||
      c->max_top_k < 0)
    return "capacities must be positive";
  const int HD = c->heads * c->head_dim, XD = c->idx_heads * c->idx_dim;
  if (HD % 256 != 0 || HD > 4096) return "heads * head_dim must be a multiple of 256, at most 4096";
  if (XD % 16 != 0 || XD > 8 * 256) return "idx_heads * idx_dim must be a multiple of 16, at most 2048";
  if (XD > 2 * HD) return "idx_heads * idx_dim must be at most 2 * heads * head_dim";
  if (c->idx_fp4 != 0 && c->idx_fp4 != 1) return "idx_fp4 must be 0 or 1";
  if (c->idx_fp4 && XD % 32 != 0) return "FP4 indexer entries need idx_heads * idx_dim to be a multiple of 32";
  if (c->idx_per_token != 0 && c->idx_per_token != 1) return "idx_per_token must be 0 or 1";
  if (c->idx_per_token && XD > 256) return "per-token indexer keys need idx_heads * idx_dim <= 256";
  if (c->idx_per_token && c->idx_heads * c->m > 64) return "per-token indexer keys need idx_heads * m <= 64";
  if (c->idx_per_token && ((c->idx_fp4 ? c->idx_dim / 2 : c->idx_dim * value_bytes(c->cache_dtype)) % 16 != 0))
    return "per-token indexer keys need each head's key to be whole 16-byte chunks";
  if (c->csa_hot_slots < 0 || c->csa_host_slots < 0 || c->csa_hot_slots > c->max_blocks ||
      (c->csa_hot_slots == 0 && c->csa_host_slots > 0))
    return "HiSparse slots: 0 <= csa_hot_slots <= max_blocks, host slots only with hot slots";
  const int vs = value_bytes(c->cache_dtype);
  bool any_csa = false;
  for (int l = 0; l < c->n_layers; ++l) {
    const int k = c->layer_kinds[l];
    if (k < KVPOOL_SWA_ONLY || k > KVPOOL_CSA_HCA) return "bad layer kind";
    any_csa |= kind_has_csa(k);
    if (kind_has_csa(k) && (!c->gate_csa || !c->gate_idx)) return "gate_csa and gate_idx are required";
    if (kind_has_hca(k) && !c->gate_hca) return "gate_hca is required";
  }

  Layout L{};
  PoolDesc& pd = L.pd;
  pd.m = c->m;
  pd.m_prime = c->m_prime;
  pd.n_win = c->n_win;
  pd.heads = c->heads;
  pd.head_dim = c->head_dim;
  pd.idx_heads = c->idx_heads;
  pd.idx_dim = c->idx_dim;
  pd.HD = HD;
  pd.XD = XD;
  pd.in_dtype = c->in_dtype;
  pd.cache_dtype = c->cache_dtype;
  pd.vs = vs;
  pd.isz = value_bytes(c->in_dtype);
  pd.csa_per_block = c->m_prime / c->m;
  pd.idx_dtype = c->idx_fp4 ? KVPOOL_FP4_E2M1 : c->cache_dtype;
  pd.idx_entry_bytes = c->idx_fp4 ? (int64_t)XD / 2 : (int64_t)XD * vs;
  pd.idx_chunks = (int32_t)(pd.idx_entry_bytes / 16);
  pd.idx_per_token = c->idx_per_token;
  pd.idx_runs = c->idx_per_token ? c->m : 1;
  pd.entry_bytes = 2LL * HD * vs + (c->cache_dtype == KVPOOL_FP8_E4M3 ? 16 : 0);
  pd.max_blocks = c->max_blocks;
  pd.max_requests = c->max_requests;
  pd.max_bpr = c->max_blocks_per_request;
  pd.staging_base = c->max_blocks;
  pd.hisparse = c->csa_hot_slots > 0 ? 1 : 0;
  pd.csa_staging_base = pd.hisparse ? c->csa_hot_slots : c->max_blocks;

  int64_t cur = 0;
  pd.err = cur;
  cur += 256;
  pd.table = cur;
  cur = round_up(cur + 4LL * c->max_requests * c->max_blocks_per_request, 256);
  pd.csa_loc = cur;
  cur = round_up(cur + 4LL * c->max_blocks, 256);
  pd.last_used = cur;
  cur = round_up(cur + 4LL * c->max_blocks, 256);
  pd.host_slot_bytes = 0;
  const int CB = pd.csa_per_block;
  for (int l = 0; l < c->n_layers; ++l) {
    LayerDesc& d = L.layers[l];
    d.kind = c->layer_kinds[l];
    d.has_csa = kind_has_csa(d.kind);
    d.has_hca = kind_has_hca(d.kind);
    d.alpha_csa = cur;
    cur = round_up(cur + 4LL * c->heads * c->m, 256);
    d.alpha_hca = cur;
    cur = round_up(cur + 4LL * c->heads * c->m_prime, 256);
    d.alpha_idx = cur;
    cur = round_up(cur + 4LL * c->idx_heads * c->m, 256);
    const int64_t n_ids = (int64_t)c->max_blocks + c->max_requests;
    const int64_t n_csa_slots = (int64_t)pd.csa_staging_base + c->max_requests;
    d.csa_pool = d.idx_pool = d.hca_pool = d.idx_scale_off = d.csa_host_off = -1;
    d.csa_stride = d.idx_stride = d.hca_stride = d.idx_run = 0;
    if (d.has_csa) {
      d.csa_stride = CB * pd.entry_bytes;
      d.csa_pool = cur;
      cur = round_up(cur + d.csa_stride * n_csa_slots, 256);
      if (pd.hisparse) {
        d.csa_host_off = pd.host_slot_bytes;
        pd.host_slot_bytes += d.csa_stride;
      }
      d.idx_run = CB * pd.idx_entry_bytes;
      if (pd.idx_dtype == KVPOOL_FP8_E4M3 || pd.idx_dtype == KVPOOL_FP4_E2M1) {
        d.idx_scale_off = d.idx_run;
        d.idx_run += round_up(2LL * CB, 16);
      }
      d.idx_stride = d.idx_run * pd.idx_runs;
      d.idx_pool = cur;
      cur = round_up(cur + d.idx_stride * n_ids, 256);
    }
    if (d.has_hca) {
      d.hca_stride = pd.entry_bytes;
      d.hca_pool = cur;
      cur = round_up(cur + d.hca_stride * n_ids, 256);
    }
    d.ring_req_bytes = round_up((int64_t)c->n_win * pd.entry_bytes, 256);
    d.ring = cur;
    cur += d.ring_req_bytes * c->max_requests;
    d.acc_req_bytes = (d.has_csa || d.has_hca) ? round_up(4LL * (4LL * HD + XD), 256) : 0;
    d.acc = cur;
    cur += d.acc_req_bytes * c->max_requests;
  }
  // decode-attention scratch
  L.n_attend_rows = std::min(c->max_batch, kMaxAttendReqs);
  L.key_stride = round_up((int64_t)(c->max_blocks_per_request + 1) * CB, 16);  // 16-byte aligned rows
  L.max_key_ctas = (int32_t)((L.key_stride + kSelectKeysPerCta - 1) / kSelectKeysPerCta);
  L.sel_stride = std::max(1, c->max_top_k);
  if (L.max_key_ctas > kMaxKeyCtasPerReq) return "max_blocks_per_request too large for the top-k select";
  // zero-initialised part: histograms and sync counters
  L.hist = cur;
  cur = round_up(cur + 4LL * L.n_attend_rows * kHistBins, 256);
  L.sync = cur;
  cur = round_up(cur + 16LL * L.n_attend_rows, 256);
  L.thr = cur;
  cur = round_up(cur + 8LL * L.n_attend_rows, 256);
  L.keys = cur;
  cur = round_up(cur + 4LL * L.n_attend_rows * L.key_stride, 256);
  L.cand = cur;
  cur = round_up(cur + 8LL * L.n_attend_rows * L.key_stride, 256);
  L.counts = cur;
  cur = round_up(cur + 8LL * L.n_attend_rows * L.max_key_ctas, 256);
  L.sel = cur;
  cur = round_up(cur + 4LL * L.n_attend_rows * L.sel_stride, 256);
  L.part_o = cur;
  cur = round_up(cur + 4LL * kMaxSplits * HD, 256);
  L.part_ml = cur;
  cur = round_up(cur + 8LL * kMaxSplits * c->heads, 256);
  L.total = cur;
  // the kernels' shared-memory plans must fit one CTA of an sm_100-family SM
  if (any_csa) {
    int sb = 0, ring = 0, so = 0, nw = 0;
    size_t smem = 0;
    score_stage_plan(pd, &sb, &ring, &so, &nw, &smem);
    if (smem > kMaxDynSmem) return "indexer blocks too large for the score kernel's shared memory";
  }
  if (attend_smem_bytes(pd) > kMaxDynSmem) return "entries too large for the attention kernel's shared memory";
  *out = L;
  return "";
}

// alpha = softmax(logits) over n positions, in double, rounded to fp32
void softmax_rows(const float* g, int rows, int n, std::vector<float>* out) {
  out->resize((size_t)rows * n);
  std::vector<double> e(n);
  for (int r = 0; r < rows; ++r) {
    const float* x = g + (size_t)r * n;
    double mx = x[0];
    for (int i = 1; i < n; ++i) mx = x[i] > mx ? x[i] : mx;
    double sum = 0.0;
    for (int i = 0; i < n; ++i) {
      e[i] = std::exp((double)x[i] - mx);
      sum += e[i];
    }
    for (int i = 0; i < n; ++i) (*out)[(size_t)r * n + i] = (float)(e[i] / sum);
  }
}

// FNV-1a 64 (Fowler, Noll, Vo) over the prefix-image config record:
// little-endian int32 m, m', n_win, heads, head_dim, idx_heads, idx_dim,
// in_dtype, cache_dtype, idx_fp4 + 2 * idx_per_token, n_layers, then per layer its kind and the
// fp32 bits of the gate logits it uses (CSA then indexer; HCA).  A gate array
// that is NULL (a pool without device memory) adds nothing.
struct Fnv1a {
  uint64_t h = 0xcbf29ce484222325ull;
  void u32(uint32_t v) {
    for (int i = 0; i < 4; ++i) {
      h ^= (v >> (8 * i)) & 0xFFu;
      h *= 0x100000001b3ull;
    }
  }
  void floats(const float* f, int64_t n) {
    if (!f) return;
    for (int64_t i = 0; i < n; ++i) {
      uint32_t u;
      std::memcpy(&u, f + i, 4);
      u32(u);
    }
  }
};

uint64_t config_fingerprint(const kvpool_config* c) {
  Fnv1a x;
  const int32_t f[11] = {c->m,       c->m_prime,  c->n_win,       c->heads,   c->head_dim, c->idx_heads,
                         c->idx_dim, c->in_dtype, c->cache_dtype, c->idx_fp4 | (c->idx_per_token << 1),
                         c->n_layers};
  for (int32_t v : f) x.u32((uint32_t)v);
  for (int l = 0; l < c->n_layers; ++l) {
    const int k = c->layer_kinds[l];
    x.u32((uint32_t)k);
    if (kind_has_csa(k)) {
      x.floats(c->gate_csa ? c->gate_csa + (size_t)l * c->heads * c->m : nullptr, (int64_t)c->heads * c->m);
      x.floats(c->gate_idx ? c->gate_idx + (size_t)l * c->idx_heads * c->m : nullptr, (int64_t)c->idx_heads * c->m);
    }
    if (kind_has_hca(k))
      x.floats(c->gate_hca ? c->gate_hca + (size_t)l * c->heads * c->m_prime : nullptr,
               (int64_t)c->heads * c->m_prime);
  }
  return x.h;
}

constexpr uint32_t kImageMagic = 0x4950564Bu;  // "KVPI"
constexpr int64_t kImageHeader = 64;

struct Request {
  bool active = false;
  int64_t length = 0;
  std::vector<int32_t> table;
};

struct ProfileSlot {
  cudaEvent_t a, b;
  int kernel;
  int n_kernels;
  int64_t bytes;
};

}  // namespace

struct kvpool {
  kvpool_config cfg{};
  // kernel parameter blocks, reused by every call (a call fills the header
  // and the entries it launches with; nothing else is read)
  std::unique_ptr<AppendParams> append_params;
  std::unique_ptr<AttendParams> attend_params;
  std::vector<int32_t> kinds;
  uint32_t flags = 0;
  uint64_t fingerprint = 0;  // of the config, for prefix images
  Layout lay{};
  uint8_t* arena = nullptr;
  int n_sms = 152;  // multiprocessors of the pool's device (queried at create)
  std::vector<int32_t> refcount;
  std::set<int32_t> free_blocks;
  std::set<int32_t> free_slots;
  std::vector<Request> reqs;
  // HiSparse: where each live block's CSA entries are (>= 0 GPU slot, < 0
  // host slot -1-loc; the id without HiSparse), the free slots, the epoch
  std::vector<int32_t> loc;
  std::set<int32_t> hot_free, host_free;
  uint32_t epoch = 0;
  uint8_t* host_pool = nullptr;  // device alias of the caller's host slots
  int64_t host_pool_bytes = 0;
  std::string err;
  // second stream for the attention part that needs no top-k, and the events
  // that fork it from / join it back to the caller's stream
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  // profiling
  int profiling = 0;  // mask of the kernel kinds whose launches are recorded
  std::vector<ProfileSlot> prof;
  std::vector<cudaEvent_t> event_pool;
  double prof_ms[KVPOOL_KERNEL_COUNT] = {};
  int64_t prof_launches[KVPOOL_KERNEL_COUNT] = {};
  int64_t prof_bytes[KVPOOL_KERNEL_COUNT] = {};

  bool device() const { return !(flags & KVPOOL_FLAG_NO_DEVICE); }
  int fail(int code, const std::string& msg) {
    err = msg;
    return code;
  }
  int cuda_fail(cudaError_t e, const char* where) {
    err = std::string(where) + ": " + cudaGetErrorString(e);
    return KVPOOL_ERR_CUDA;
  }
  bool req_ok(int32_t r) const { return r >= 0 && r < cfg.max_requests && reqs[r].active; }
  bool hisparse() const { return lay.pd.hisparse != 0; }
  // location of a block id just taken (sealed or restored): a GPU slot
  int32_t take_hot(int32_t id) {
    if (!hisparse()) return id;
    const int32_t h = *hot_free.begin();
    hot_free.erase(hot_free.begin());
    return h;
  }
  void release_loc(int32_t l) {
    if (!hisparse()) return;
    if (l >= 0) hot_free.insert(l);
    else host_free.insert(-1 - l);
  }
  // the device address of the CSA part of layer d of a block at location l
  uint64_t csa_addr(const LayerDesc& d, int32_t l) const {
    if (l >= 0) return reinterpret_cast<uint64_t>(arena + d.csa_pool + (int64_t)l * d.csa_stride);
    return reinterpret_cast<uint64_t>(host_pool + (int64_t)(-1 - l) * lay.pd.host_slot_bytes + d.csa_host_off);
  }

  // ---- profiling helpers ----
  cudaEvent_t take_event() {
    if (!event_pool.empty()) {
      cudaEvent_t e = event_pool.back();
      event_pool.pop_back();
      return e;
    }
    cudaEvent_t e;
    cudaEventCreate(&e);
    return e;
  }
  // run f(&n_kernels), recording events around it when profiling
  template <class F>
  int launch(int kernel, int64_t bytes, void* stream, F&& f) {
    ProfileSlot s{};
    const bool rec = (profiling >> kernel) & 1;
    if (rec) {
      s.a = take_event();
      s.b = take_event();
      s.kernel = kernel;
      s.bytes = bytes;
      cudaEventRecord(s.a, (cudaStream_t)stream);
    }
    int nk = 0;
    const int rc = f(&nk);
    if (rec) {
      cudaEventRecord(s.b, (cudaStream_t)stream);
      s.n_kernels = nk;
      prof.push_back(s);
    } else if (profiling & KVPOOL_PROFILE_COUNT) {  // counted without events
      prof_launches[kernel] += nk;
      prof_bytes[kernel] += bytes;
    }
    return rc;
  }
  std::vector<float> timeline;  // (kind, start, end) since profiling was enabled
  cudaEvent_t t0 = nullptr;     // first event of the timeline (kept out of the pool)
  void settle_profile() {
    for (auto& s : prof) {
      cudaEventSynchronize(s.b);
      float ms = 0.f;
      cudaEventElapsedTime(&ms, s.a, s.b);
      prof_ms[s.kernel] += ms;
      prof_launches[s.kernel] += s.n_kernels;
      prof_bytes[s.kernel] += s.bytes;
      if (!t0) t0 = s.a;
      float a = 0.f, b = 0.f;
      cudaEventElapsedTime(&a, t0, s.a);
      cudaEventElapsedTime(&b, t0, s.b);
      timeline.push_back((float)s.kernel);
      timeline.push_back(a);
      timeline.push_back(b);
      if (s.a != t0) event_pool.push_back(s.a);
      event_pool.push_back(s.b);
    }
    prof.clear();
  }
};

extern "C" {

size_t kvpool_required_bytes(const kvpool_config* cfg) {
  Layout L;
  if (!plan_layout(cfg, &L).empty()) return 0;
  return (size_t)L.total;
}

int kvpool_create(const kvpool_config* cfg, void* d_arena, size_t arena_bytes, void* stream, kvpool_t** out) {
  if (!out) return KVPOOL_ERR_INVALID_ARG;
  *out = nullptr;
  Layout L;
  if (!plan_layout(cfg, &L).empty()) return KVPOOL_ERR_INVALID_ARG;
  const bool no_dev = (cfg->flags & KVPOOL_FLAG_NO_DEVICE) != 0;
  if (no_dev ? d_arena != nullptr : (!d_arena || arena_bytes < (size_t)L.total)) return KVPOOL_ERR_INVALID_ARG;
  if (!no_dev && (reinterpret_cast<uintptr_t>(d_arena) % 256) != 0) return KVPOOL_ERR_INVALID_ARG;

  kvpool* p = new (std::nothrow) kvpool();
  if (!p) return KVPOOL_ERR_INVALID_ARG;
  p->cfg = *cfg;
  p->kinds.assign(cfg->layer_kinds, cfg->layer_kinds + cfg->n_layers);
  p->cfg.layer_kinds = p->kinds.data();
  p->fingerprint = config_fingerprint(&p->cfg);
  p->cfg.gate_csa = p->cfg.gate_hca = p->cfg.gate_idx = nullptr;
  p->flags = cfg->flags;
  p->lay = L;
  p->arena = static_cast<uint8_t*>(d_arena);
  p->lay.pd.arena = p->arena;
  p->refcount.assign(cfg->max_blocks, 0);
  p->loc.assign(cfg->max_blocks, 0);
  for (int32_t h = 0; h < cfg->csa_hot_slots; ++h) p->hot_free.insert(p->hot_free.end(), h);
  for (int32_t h = 0; h < cfg->csa_host_slots; ++h) p->host_free.insert(p->host_free.end(), h);
  for (int32_t b = 0; b < cfg->max_blocks; ++b) p->free_blocks.insert(p->free_blocks.end(), b);
  for (int32_t r = 0; r < cfg->max_requests; ++r) p->free_slots.insert(p->free_slots.end(), r);
  p->reqs.resize(cfg->max_requests);

  if (!no_dev) {
    cudaStream_t s = (cudaStream_t)stream;
    // launch shapes are sized in CTAs per SM of the device the arena lives on
    int dev = 0, sms = 0;
    cudaError_t de = cudaGetDevice(&dev);
    if (de == cudaSuccess) de = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (de != cudaSuccess || sms < 1) { int rc = p->cuda_fail(de != cudaSuccess ? de : cudaErrorInvalidDevice, "device query"); delete p; return rc; }
    p->n_sms = sms;
    // gates: softmax on the host, one upload per layer and kind
    std::vector<float> a;
    for (int l = 0; l < cfg->n_layers; ++l) {
      const LayerDesc& d = L.layers[l];
      if (d.has_csa) {
        softmax_rows(cfg->gate_csa + (size_t)l * cfg->heads * cfg->m, cfg->heads, cfg->m, &a);
        cudaError_t e = cudaMemcpy(p->arena + d.alpha_csa, a.data(), a.size() * 4, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) { int rc = p->cuda_fail(e, "gate upload"); delete p; return rc; }
        softmax_rows(cfg->gate_idx + (size_t)l * cfg->idx_heads * cfg->m, cfg->idx_heads, cfg->m, &a);
        e = cudaMemcpy(p->arena + d.alpha_idx, a.data(), a.size() * 4, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) { int rc = p->cuda_fail(e, "gate upload"); delete p; return rc; }
      }
      if (d.has_hca) {
        softmax_rows(cfg->gate_hca + (size_t)l * cfg->heads * cfg->m_prime, cfg->heads, cfg->m_prime, &a);
        cudaError_t e = cudaMemcpy(p->arena + d.alpha_hca, a.data(), a.size() * 4, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) { int rc = p->cuda_fail(e, "gate upload"); delete p; return rc; }
      }
    }
    // error word and select histograms start at zero
    cudaError_t e = cudaMemsetAsync(p->arena + L.pd.err, 0, 256, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p->arena + L.hist, 0, (size_t)(L.thr - L.hist), s);
    if (e != cudaSuccess) { int rc = p->cuda_fail(e, "arena init"); delete p; return rc; }
    e = cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_join, cudaEventDisableTiming);
    if (e != cudaSuccess) { int rc = p->cuda_fail(e, "side stream"); kvpool_destroy(p); return rc; }
  }
  *out = p;
  return KVPOOL_OK;
}

int kvpool_destroy(kvpool_t* p) {
  if (!p) return KVPOOL_ERR_INVALID_ARG;
  for (auto& s : p->prof) {
    cudaEventDestroy(s.a);
    cudaEventDestroy(s.b);
  }
  for (auto e : p->event_pool) cudaEventDestroy(e);
  if (p->t0) cudaEventDestroy(p->t0);
  if (p->ev_fork) cudaEventDestroy(p->ev_fork);
  if (p->ev_join) cudaEventDestroy(p->ev_join);
  if (p->side) cudaStreamDestroy(p->side);
  delete p;
  return KVPOOL_OK;
}

int kvpool_alloc_request(kvpool_t* p, int32_t* req_out) {
  if (!p || !req_out) return KVPOOL_ERR_INVALID_ARG;
  if (p->free_slots.empty()) return p->fail(KVPOOL_ERR_OUT_OF_REQUESTS, "no free request slot");
  const int32_t r = *p->free_slots.begin();
  p->free_slots.erase(p->free_slots.begin());
  Request& q = p->reqs[r];
  q.active = true;
  q.length = 0;
  q.table.clear();
  *req_out = r;
  return KVPOOL_OK;
}

static void release_block(kvpool_t* p, int32_t b) {
  if (--p->refcount[b] == 0) {
    p->free_blocks.insert(b);
    p->release_loc(p->loc[b]);
  }
}

int kvpool_free_request(kvpool_t* p, int32_t r) {
  if (!p) return KVPOOL_ERR_INVALID_ARG;
  if (!p->req_ok(r)) return p->fail(KVPOOL_ERR_BAD_REQUEST, "free_request: bad request id");
  Request& q = p->reqs[r];
  for (int32_t b : q.table) release_block(p, b);
  q.table.clear();
  q.active = false;
  q.length = 0;
  p->free_slots.insert(r);
  return KVPOOL_OK;
}

int kvpool_share_prefix(kvpool_t* p, int32_t dst, int32_t src, int64_t n_tokens, const void* d_win_k,
                        const void* d_win_v, void* stream) {
  if (!p) return KVPOOL_ERR_INVALID_ARG;
  if (!p->req_ok(dst) || !p->req_ok(src) || dst == src) return p->fail(KVPOOL_ERR_BAD_REQUEST, "share_prefix: bad ids");
  if (n_tokens <= 0) return p->fail(KVPOOL_ERR_INVALID_ARG, "share_prefix: n_tokens <= 0");
  const int mp = p->cfg.m_prime;
  Request& s = p->reqs[src];
  Request& d = p->reqs[dst];
  if (n_tokens % mp != 0 || n_tokens / mp > (int64_t)s.table.size())
    return p->fail(KVPOOL_ERR_NOT_SHAREABLE, "share_prefix: prefix is not whole sealed blocks of src");
  if (d.length != 0) return p->fail(KVPOOL_ERR_NOT_SHAREABLE, "share_prefix: dst is not fresh");
  if (!d_win_k || !d_win_v) {
    if (p->device()) return p->fail(KVPOOL_ERR_INVALID_ARG, "share_prefix: NULL window");
  }
  const int nb = (int)(n_tokens / mp);
  const int w = (int)std::min<int64_t>(n_tokens, p->cfg.n_win);
  if (p->device()) {
    if ((reinterpret_cast<uintptr_t>(d_win_k) | reinterpret_cast<uintptr_t>(d_win_v)) % 16 != 0)
      return p->fail(KVPOOL_ERR_INVALID_ARG, "share_prefix: window not 16-byte aligned");
    ShareParams sp{};
    sp.pool = p->lay.pd;
    std::memcpy(sp.layers, p->lay.layers, sizeof(sp.layers));
    sp.win_k = d_win_k;
    sp.win_v = d_win_v;
    sp.dst = dst;
    sp.src = src;
    sp.n_blocks = nb;
    sp.w = w;
    sp.n_tokens = n_tokens;
    const int rc = p->launch(KVPOOL_KERNEL_APPEND, 0, stream, [&](int* nk) { return launch_share(sp, p->cfg.n_layers, stream, nk); });
    if (rc != 0) return p->cuda_fail((cudaError_t)rc, "share_prefix launch");
  }
  d.table.assign(s.table.begin(), s.table.begin() + nb);
  for (int32_t b : d.table) p->refcount[b] += 1;
  d.length = n_tokens;
  return KVPOOL_OK;
}

}  // extern "C"

// ---- block copies: prefix images, HiSparse offload and fetch -----------------
namespace {

bool image_layout_ok(const kvpool_t* p) {
  for (int k : p->kinds)
    if (kind_has_csa(k) && p->lay.pd.idx_entry_bytes % 16 != 0) return false;
  return true;
}

int64_t image_window_tokens(const kvpool_t* p, int64_t n_tokens, uint32_t flags) {
  return (flags & KVPOOL_IMAGE_WINDOW) ? std::min<int64_t>(n_tokens, p->cfg.n_win) : 0;
}

// bytes of one block's parts, summed over the layers
int64_t image_block_bytes(const kvpool_t* p) {
  int64_t b = 0;
  for (int l = 0; l < p->cfg.n_layers; ++l) {
    const LayerDesc& d = p->lay.layers[l];
    if (d.has_csa) b += d.csa_stride + d.idx_stride;
    if (d.has_hca) b += d.hca_stride;
  }
  return b;
}

void put_le(uint8_t* dst, uint64_t v, int n) {
  for (int i = 0; i < n; ++i) dst[i] = (uint8_t)(v >> (8 * i));
}
uint64_t get_le(const uint8_t* src, int n) {
  uint64_t v = 0;
  for (int i = 0; i < n; ++i) v |= (uint64_t)src[i] << (8 * i);
  return v;
}

// Append a copy, merged into the previous one when both ends continue it.
void add_copy(std::vector<ImageSeg>* segs, uint64_t src, uint64_t dst, int64_t bytes, bool src_host, int32_t mask_row = 0,
              int32_t mask_valid = 0) {
  if (!segs->empty()) {
    ImageSeg& g = segs->back();
    if (g.src + (uint64_t)g.bytes == src && g.dst + (uint64_t)g.bytes == dst && g.mask_row == mask_row &&
        g.mask_valid == mask_valid && (g.src_host != 0) == src_host) {
      g.bytes += bytes;
      return;
    }
  }
  segs->push_back(ImageSeg{src, dst, bytes, mask_row, mask_valid, src_host ? 1 : 0, 0});
}

// Append the bookkeeping writes for block ids[i] at locs[i] (table index
// b0 + i when b0 >= 0), merged into runs of consecutive ids and locations.
void add_runs(std::vector<ImageRun>* runs, const std::vector<int32_t>& ids, const std::vector<int32_t>& locs, int32_t b0,
              bool write_loc, bool stamp) {
  for (size_t i = 0; i < ids.size();) {
    size_t e = i + 1;
    const int dir = write_loc && e < ids.size() && locs[e] == locs[i] - 1 ? -1 : 1;
    while (e < ids.size() && ids[e] == ids[e - 1] + 1 && (!write_loc || locs[e] == locs[e - 1] + dir)) ++e;
    runs->push_back(ImageRun{b0 >= 0 ? b0 + (int32_t)i : -1, ids[i], (int32_t)(e - i), locs[i],
                             (int16_t)(write_loc ? dir : 0), (int16_t)(stamp ? 1 : 0)});
    i = e;
  }
}

// The copies between the pool and an image: per layer and part, the blocks
// (ids, CSA entries at locs) in table order, then the window ring pieces.
// to_image: pool -> image, else image -> pool.
void image_segments(const kvpool_t* p, const std::vector<int32_t>& ids, const std::vector<int32_t>& locs, int32_t slot,
                    int64_t n_tokens, int64_t w, uint64_t image, bool to_image, std::vector<ImageSeg>* segs) {
  const int64_t nb = (int64_t)ids.size();
  const PoolDesc& pd = p->lay.pd;
  const uint64_t arena = reinterpret_cast<uint64_t>(p->arena);
  uint64_t img = image + kImageHeader;
  auto add = [&](uint64_t pool_addr, bool pool_host, int64_t bytes, int32_t mask_row, int32_t mask_valid) {
    if (to_image) add_copy(segs, pool_addr, img, bytes, pool_host, mask_row, mask_valid);
    else add_copy(segs, img, pool_addr, bytes, true);
    img += bytes;
  };
  const bool idx_scaled = pd.idx_dtype == KVPOOL_FP8_E4M3 || pd.idx_dtype == KVPOOL_FP4_E2M1;
  for (int l = 0; l < p->cfg.n_layers; ++l) {
    const LayerDesc& d = p->lay.layers[l];
    if (d.has_csa) {
      for (int64_t b = 0; b < nb; ++b) add(p->csa_addr(d, locs[b]), locs[b] < 0, d.csa_stride, 0, 0);
      // the padding after each run's scales is written as zeros
      const int64_t valid = d.idx_scale_off + 2LL * pd.csa_per_block;
      const int32_t mvalid = idx_scaled && valid < d.idx_run ? (int32_t)valid : 0;
      for (int64_t b = 0; b < nb; ++b)
        add(arena + d.idx_pool + (uint64_t)ids[b] * d.idx_stride, false, d.idx_stride, mvalid ? (int32_t)d.idx_run : 0,
            mvalid);
    }
    if (d.has_hca)
      for (int64_t b = 0; b < nb; ++b) add(arena + d.hca_pool + (uint64_t)ids[b] * d.hca_stride, false, d.hca_stride, 0, 0);
  }
  for (int l = 0; l < p->cfg.n_layers && w > 0; ++l) {
    const LayerDesc& d = p->lay.layers[l];
    const uint64_t ring = arena + d.ring + (uint64_t)slot * d.ring_req_bytes;
    const int64_t s0 = (n_tokens - w) % pd.n_win;
    const int64_t first = std::min<int64_t>(w, pd.n_win - s0);
    add(ring + (uint64_t)s0 * pd.entry_bytes, false, first * pd.entry_bytes, 0, 0);
    if (w > first) add(ring, false, (w - first) * pd.entry_bytes, 0, 0);
  }
}

// Launch the copies in batches of kMaxImageSegs copies and kMaxImageRuns
// bookkeeping runs.
int launch_block_copies(kvpool_t* p, int32_t dst, const std::vector<ImageSeg>& segs, const std::vector<ImageRun>& runs,
                        int64_t bytes, void* stream) {
  const size_t n_launch = std::max((segs.size() + kMaxImageSegs - 1) / kMaxImageSegs,
                                   (runs.size() + kMaxImageRuns - 1) / kMaxImageRuns);
  for (size_t i = 0; i < n_launch; ++i) {
    ImageParams ip{};
    ip.pool = p->lay.pd;
    ip.dst = dst;
    ip.epoch = p->epoch;
    ip.n_sms = p->n_sms;
    const size_t s0 = i * kMaxImageSegs, s1 = std::min(segs.size(), s0 + kMaxImageSegs);
    ip.n_segs = s1 > s0 ? (int32_t)(s1 - s0) : 0;
    int64_t pieces = 0;
    for (int32_t k = 0; k < ip.n_segs; ++k) {
      ip.segs[k] = segs[s0 + k];
      ip.piece_base[k] = pieces;
      pieces += (ip.segs[k].bytes + kImagePieceBytes - 1) / kImagePieceBytes;
    }
    ip.piece_base[ip.n_segs] = pieces;
    ip.n_pieces = pieces;
    const size_t r0 = i * kMaxImageRuns, r1 = std::min(runs.size(), r0 + kMaxImageRuns);
    ip.n_runs = r1 > r0 ? (int32_t)(r1 - r0) : 0;
    for (int32_t k = 0; k < ip.n_runs; ++k) ip.runs[k] = runs[r0 + k];
    const int rc = p->launch(KVPOOL_KERNEL_IMAGE, i == 0 ? 2 * bytes : 0, stream,
                             [&](int* nk) { return launch_image(ip, stream, nk); });
    if (rc != 0) return rc;
  }
  return 0;
}

// Device alias of a page-locked, mapped host buffer, or nullptr (pageable
// memory included, even where the GPU could reach it through the host's page
// tables).
uint8_t* host_alias(const void* h) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
    cudaGetLastError();  // clear the (non-sticky) error
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
  return static_cast<uint8_t*>(a.devicePointer);
}

// distinct live block ids, all resident (want_hot) or all offloaded
bool hisparse_ids_ok(const kvpool_t* p, int32_t n, const int32_t* ids, bool want_hot) {
  if (!p->hisparse() || n < 0 || (n > 0 && !ids)) return false;
  std::set<int32_t> seen;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t b = ids[i];
    if (b < 0 || b >= p->cfg.max_blocks || p->refcount[b] == 0) return false;
    if ((p->loc[b] >= 0) != want_hot || !seen.insert(b).second) return false;
  }
  return true;
}

// Move blocks' CSA entries to new locations (host slots or GPU slots).
int move_blocks(kvpool_t* p, int32_t n, const int32_t* ids, const std::vector<int32_t>& to, bool stamp, void* stream) {
  if (!p->device() || n == 0) return 0;
  std::vector<ImageSeg> segs;
  for (int l = 0; l < p->cfg.n_layers; ++l) {
    const LayerDesc& d = p->lay.layers[l];
    if (!d.has_csa) continue;
    for (int32_t i = 0; i < n; ++i)
      add_copy(&segs, p->csa_addr(d, p->loc[ids[i]]), p->csa_addr(d, to[i]), d.csa_stride, p->loc[ids[i]] < 0);
  }
  std::vector<ImageRun> runs;
  add_runs(&runs, std::vector<int32_t>(ids, ids + n), to, -1, true, stamp);
  return launch_block_copies(p, 0, segs, runs, (int64_t)n * p->lay.pd.host_slot_bytes, stream);
}

}  // namespace

extern "C" {

uint64_t kvpool_fingerprint(const kvpool_t* p) { return p ? p->fingerprint : 0; }

int64_t kvpool_image_bytes(const kvpool_t* p, int64_t n_tokens, uint32_t flags) {
  if (!p || !image_layout_ok(p) || (flags & ~KVPOOL_IMAGE_WINDOW) || n_tokens <= 0 || n_tokens % p->cfg.m_prime != 0)
    return -1;
  const int64_t nb = n_tokens / p->cfg.m_prime, w = image_window_tokens(p, n_tokens, flags);
  return kImageHeader + nb * image_block_bytes(p) + w * p->lay.pd.entry_bytes * p->cfg.n_layers;
}

int kvpool_export_prefix(kvpool_t* p, int32_t req, int64_t n_tokens, uint32_t flags, void* h_image, int64_t capacity,
                         void* stream) {
  if (!p) return KVPOOL_ERR_INVALID_ARG;
  if (!h_image || (flags & ~KVPOOL_IMAGE_WINDOW) || !image_layout_ok(p))
    return p->fail(KVPOOL_ERR_INVALID_ARG, "export_prefix: bad arguments");
  if (!p->req_ok(req)) return p->fail(KVPOOL_ERR_BAD_REQUEST, "export_prefix: bad request id");
  const Request& q = p->reqs[req];
  const int mp = p->cfg.m_prime;
  if (n_tokens <= 0 || n_tokens % mp != 0 || n_tokens / mp > (int64_t)q.table.size())
    return p->fail(KVPOOL_ERR_NOT_SHAREABLE, "export_prefix: prefix is not whole sealed blocks");
  if ((flags & KVPOOL_IMAGE_WINDOW) && n_tokens != q.length)
    return p->fail(KVPOOL_ERR_NOT_SHAREABLE, "export_prefix: the window exists only at the request's length");
  const int64_t total = kvpool_image_bytes(p, n_tokens, flags);
  if (capacity < total) return p->fail(KVPOOL_ERR_INVALID_ARG, "export_prefix: capacity too small");
  if (reinterpret_cast<uintptr_t>(h_image) % 16 != 0)
    return p->fail(KVPOOL_ERR_INVALID_ARG, "export_prefix: image not 16-byte aligned");
  uint8_t* d_image = nullptr;
  if (p->device() && !(d_image = host_alias(h_image)))
    return p->fail(KVPOOL_ERR_INVALID_ARG, "export_prefix: image is not page-locked host memory");
  const int64_t nb = n_tokens / mp, w = image_window_tokens(p, n_tokens, flags);
  const int64_t block_sec = nb * image_block_bytes(p), win_sec = w * p->lay.pd.entry_bytes * p->cfg.n_layers;

  uint8_t* h = static_cast<uint8_t*>(h_image);
  std::memset(h, 0, kImageHeader);
  put_le(h, kImageMagic, 4);
  put_le(h + 4, 1, 4);
  put_le(h + 8, p->fingerprint, 8);
  put_le(h + 16, (uint64_t)n_tokens, 8);
  put_le(h + 24, (uint64_t)nb, 4);
  put_le(h + 28, (uint64_t)w, 4);
  put_le(h + 32, (uint64_t)block_sec, 8);
  put_le(h + 40, (uint64_t)win_sec, 8);
  put_le(h + 48, (uint64_t)total, 8);
  if (!p->device()) return KVPOOL_OK;  // bookkeeping-only pool: the header alone

  std::vector<int32_t> ids(q.table.begin(), q.table.begin() + nb), locs(nb);
  for (int64_t b = 0; b < nb; ++b) locs[b] = p->loc[ids[b]];
  std::vector<ImageSeg> segs;
  image_segments(p, ids, locs, req, n_tokens, w, reinterpret_cast<uint64_t>(d_image), true, &segs);
  const int rc = launch_block_copies(p, req, segs, {}, block_sec + win_sec, stream);
  if (rc != 0) return p->cuda_fail((cudaError_t)rc, "export_prefix launch");
  return KVPOOL_OK;
}

int kvpool_import_prefix(kvpool_t* p, int32_t dst, const void* h_image, int64_t bytes, const void* d_win_k,
                         const void* d_win_v, void* stream) {
  if (!p) return KVPOOL_ERR_INVALID_ARG;
  if (!h_image || !image_layout_ok(p)) return p->fail(KVPOOL_ERR_INVALID_ARG, "import_prefix: bad arguments");
  if (!p->req_ok(dst)) return p->fail(KVPOOL_ERR_BAD_REQUEST, "import_prefix: bad request id");
  const uint8_t* h = static_cast<const uint8_t*>(h_image);
  if (bytes < kImageHeader || get_le(h, 4) != kImageMagic || get_le(h + 4, 4) != 1 ||
      get_le(h + 8, 8) != p->fingerprint)
    return p->fail(KVPOOL_ERR_BAD_IMAGE, "import_prefix: not an image of this pool's config");
  const int mp = p->cfg.m_prime;
  const int64_t n_tokens = (int64_t)get_le(h + 16, 8);
  const int64_t nb = (int64_t)get_le(h + 24, 4), w = (int64_t)get_le(h + 28, 4);
  const uint32_t flags = w > 0 ? KVPOOL_IMAGE_WINDOW : 0u;
  const int64_t total = kvpool_image_bytes(p, n_tokens, flags);
  if (total < 0 || nb != n_tokens / mp || (w != 0 && w != std::min<int64_t>(n_tokens, p->cfg.n_win)) ||
      bytes < total || get_le(h + 48, 8) != (uint64_t)total ||
      get_le(h + 32, 8) != (uint64_t)(nb * image_block_bytes(p)) ||
      get_le(h + 40, 8) != (uint64_t)(w * p->lay.pd.entry_bytes * p->cfg.n_layers))
    return p->fail(KVPOOL_ERR_BAD_IMAGE, "import_prefix: inconsistent sizes");
  Request& d = p->reqs[dst];
  if (d.length != 0) return p->fail(KVPOOL_ERR_NOT_SHAREABLE, "import_prefix: dst is not fresh");
  const bool zero_swa = w == 0;
  if (p->device() && zero_swa != (d_win_k && d_win_v))
    return p->fail(KVPOOL_ERR_INVALID_ARG, zero_swa ? "import_prefix: the image has no window: give one"
                                                    : "import_prefix: the image has a window: give NULL windows");
  if (p->device() && zero_swa &&
      ((reinterpret_cast<uintptr_t>(d_win_k) | reinterpret_cast<uintptr_t>(d_win_v)) % 16) != 0)
    return p->fail(KVPOOL_ERR_INVALID_ARG, "import_prefix: window not 16-byte aligned");
  if (nb > p->cfg.max_blocks_per_request) return p->fail(KVPOOL_ERR_CAPACITY, "import_prefix: prefix too long");
  if (nb > (int64_t)p->free_blocks.size() || (p->hisparse() && nb > (int64_t)p->hot_free.size()))
    return p->fail(KVPOOL_ERR_OUT_OF_BLOCKS, "import_prefix: out of blocks");
  if (reinterpret_cast<uintptr_t>(h_image) % 16 != 0)
    return p->fail(KVPOOL_ERR_INVALID_ARG, "import_prefix: image not 16-byte aligned");
  uint8_t* d_image = nullptr;
  if (p->device() && !(d_image = host_alias(h_image)))
    return p->fail(KVPOOL_ERR_INVALID_ARG, "import_prefix: image is not page-locked host memory");

  // the smallest free ids (and GPU slots), in image order; taken only once
  // the launches succeeded, so an error leaves the pool unchanged
  std::vector<int32_t> ids, locs;
  auto it = p->free_blocks.begin();
  auto ht = p->hot_free.begin();
  for (int64_t b = 0; b < nb; ++b, ++it) {
    ids.push_back(*it);
    locs.push_back(p->hisparse() ? *ht++ : *it);
  }
  if (p->device()) {
    std::vector<ImageSeg> segs;
    image_segments(p, ids, locs, dst, n_tokens, w, reinterpret_cast<uint64_t>(d_image), false, &segs);
    std::vector<ImageRun> runs;
    add_runs(&runs, ids, locs, 0, p->hisparse(), p->hisparse());
    const int64_t moved = nb * image_block_bytes(p) + w * p->lay.pd.entry_bytes * p->cfg.n_layers;
    int rc = launch_block_copies(p, dst, segs, runs, moved, stream);
    if (rc == 0 && zero_swa) {  // Zero SWA: the recomputed window through the cache encoding
      ShareParams sp{};
      sp.pool = p->lay.pd;
      std::memcpy(sp.layers, p->lay.layers, sizeof(sp.layers));
      sp.win_k = d_win_k;
      sp.win_v = d_win_v;
      sp.dst = dst;
      sp.src = -1;
      sp.n_blocks = 0;
      sp.w = (int)std::min<int64_t>(n_tokens, p->cfg.n_win);
      sp.n_tokens = n_tokens;
      rc = p->launch(KVPOOL_KERNEL_IMAGE, 0, stream, [&](int* nk) { return launch_share(sp, p->cfg.n_layers, stream, nk); });
    }
    if (rc != 0) return p->cuda_fail((cudaError_t)rc, "import_prefix launch");
  }
  for (int64_t b = 0; b < nb; ++b) {
    p->free_blocks.erase(ids[b]);
    if (p->hisparse()) p->hot_free.erase(locs[b]);
    p->refcount[ids[b]] = 1;
    p->loc[ids[b]] = locs[b];
  }
  d.table = ids;
  d.length = n_tokens;
  return KVPOOL_OK;
}

// ---- HiSparse ----
int64_t kvpool_host_slot_bytes(const kvpool_t* p) { return p ? p->lay.pd.host_slot_bytes : -1; }

int kvpool_set_host_pool(kvpool_t* p, void* h_pool, int64_t bytes) {
  if (!p) return KVPOOL_ERR_INVALID_ARG;
  if (!p->hisparse()) return p->fail(KVPOOL_ERR_INVALID_ARG, "set_host_pool: HiSparse is off");
  if (!h_pool || bytes < (int64_t)p->cfg.csa_host_slots * p->lay.pd.host_slot_bytes ||
      reinterpret_cast<uintptr_t>(h_pool) % 16 != 0)
    return p->fail(KVPOOL_ERR_INVALID_ARG, "set_host_pool: too small or not 16-byte aligned");
  if ((int32_t)p->host_free.size() != p->cfg.csa_host_slots)
    return p->fail(KVPOOL_ERR_INVALID_ARG, "set_host_pool: blocks are offloaded to the current pool");
  uint8_t* d = nullptr;
  if (p->device() && !(d = host_alias(h_pool)))
    return p->fail(KVPOOL_ERR_INVALID_ARG, "set_host_pool: not page-locked host memory");
  p->host_pool = d;
  p->host_pool_bytes = bytes;
  p->lay.pd.host_pool = d;
  p->lay.pd.host_pool_bytes = bytes;
  return KVPOOL_OK;
}

int kvpool_offload(kvpool_t* p, int32_t n, const int32_t* h_ids, void* stream) {
  if (!p) return KVPOOL_ERR_INVALID_ARG;
  if (!hisparse_ids_ok(p, n, h_ids, true)) return p->fail(KVPOOL_ERR_INVALID_ARG, "offload: bad block ids");
  if (p->device() && !p->host_pool) return p->fail(KVPOOL_ERR_INVALID_ARG, "offload: no host pool");
  if (n > (int32_t)p->host_free.size()) return p->fail(KVPOOL_ERR_OUT_OF_BLOCKS, "offload: out of host slots");
  std::vector<int32_t> to;
  auto it = p->host_free.begin();
  for (int32_t i = 0; i < n; ++i, ++it) to.push_back(-1 - *it);
  const int rc = move_blocks(p, n, h_ids, to, false, stream);
  if (rc != 0) return p->cuda_fail((cudaError_t)rc, "offload launch");
  for (int32_t i = 0; i < n; ++i) {
    p->host_free.erase(-1 - to[i]);
    p->release_loc(p->loc[h_ids[i]]);
    p->loc[h_ids[i]] = to[i];
  }
  return KVPOOL_OK;
}

int kvpool_fetch(kvpool_t* p, int32_t n, const int32_t* h_ids, void* stream) {
  if (!p) return KVPOOL_ERR_INVALID_ARG;
  if (!hisparse_ids_ok(p, n, h_ids, false)) return p->fail(KVPOOL_ERR_INVALID_ARG, "fetch: bad block ids");
  if (n > (int32_t)p->hot_free.size()) return p->fail(KVPOOL_ERR_OUT_OF_BLOCKS, "fetch: out of GPU slots");
  std::vector<int32_t> to;
  auto it = p->hot_free.begin();
  for (int32_t i = 0; i < n; ++i, ++it) to.push_back(*it);
  const int rc = move_blocks(p, n, h_ids, to, true, stream);
  if (rc != 0) return p->cuda_fail((cudaError_t)rc, "fetch launch");
  for (int32_t i = 0; i < n; ++i) {
    p->hot_free.erase(to[i]);
    p->release_loc(p->loc[h_ids[i]]);
    p->loc[h_ids[i]] = to[i];
  }
  return KVPOOL_OK;
}

int kvpool_block_location(const kvpool_t* p, int32_t b, int32_t* loc) {
  if (!p || !loc || b < 0 || b >= p->cfg.max_blocks || p->refcount[b] == 0) return KVPOOL_ERR_INVALID_ARG;
  *loc = p->loc[b];
  return KVPOOL_OK;
}

uint32_t kvpool_epoch(const kvpool_t* p) { return p ? p->epoch : 0; }

}  // extern "C"

namespace {
// every block's activity stamp, read back after synchronizing the stream
int read_activity(kvpool_t* p, std::vector<uint32_t>* out, void* stream) {
  out->assign(p->cfg.max_blocks, 0);
  cudaError_t e = cudaMemcpyAsync(out->data(), p->arena + p->lay.pd.last_used, 4ull * p->cfg.max_blocks,
                                  cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  return (int)e;
}
}  // namespace

extern "C" {

int kvpool_block_activity(kvpool_t* p, int32_t n, const int32_t* h_ids, uint32_t* h_last_used, void* stream) {
  if (!p) return KVPOOL_ERR_INVALID_ARG;
  if (!p->hisparse() || !p->device() || n < 0 || (n > 0 && (!h_ids || !h_last_used)))
    return p->fail(KVPOOL_ERR_INVALID_ARG, "block_activity: bad arguments");
  for (int32_t i = 0; i < n; ++i)
    if (h_ids[i] < 0 || h_ids[i] >= p->cfg.max_blocks || p->refcount[h_ids[i]] == 0)
      return p->fail(KVPOOL_ERR_INVALID_ARG, "block_activity: a free block");
  std::vector<uint32_t> a;
  const int rc = read_activity(p, &a, stream);
  if (rc != 0) return p->cuda_fail((cudaError_t)rc, "block_activity");
  for (int32_t i = 0; i < n; ++i) h_last_used[i] = a[h_ids[i]];
  return KVPOOL_OK;
}

int32_t kvpool_inactive_blocks(kvpool_t* p, uint32_t idle, int32_t* h_ids, int32_t cap, void* stream) {
  if (!p) return KVPOOL_ERR_INVALID_ARG;
  if (!p->hisparse() || !p->device() || cap < 0 || (cap > 0 && !h_ids))
    return p->fail(KVPOOL_ERR_INVALID_ARG, "inactive_blocks: bad arguments");
  std::vector<uint32_t> a;
  const int rc = read_activity(p, &a, stream);
  if (rc != 0) return p->cuda_fail((cudaError_t)rc, "inactive_blocks");
  int32_t n = 0;
  for (int32_t b = 0; b < p->cfg.max_blocks; ++b) {
    if (p->refcount[b] == 0 || p->loc[b] < 0 || p->epoch - a[b] < idle) continue;
    if (n < cap) h_ids[n] = b;
    ++n;
  }
  return n;
}

int kvpool_append(kvpool_t* p, int32_t n, const int32_t* h_req_ids, const int32_t* h_n_new, const void* d_k,
                  const void* d_v, const void* d_idx_k, void* stream) {
  if (!p || n < 0 || (n > 0 && (!h_req_ids || !h_n_new))) return KVPOOL_ERR_INVALID_ARG;
  if (n > p->cfg.max_batch) return p->fail(KVPOOL_ERR_INVALID_ARG, "append: n > max_batch");
  const int mp = p->cfg.m_prime, W = p->cfg.n_win;
  int64_t T = 0, seals = 0;
  for (int i = 0; i < n; ++i) {
    if (!p->req_ok(h_req_ids[i])) return p->fail(KVPOOL_ERR_BAD_REQUEST, "append: bad request id");
    if (h_n_new[i] < 0) return p->fail(KVPOOL_ERR_INVALID_ARG, "append: negative count");
    for (int j = 0; j < i; ++j)
      if (h_req_ids[j] == h_req_ids[i]) return p->fail(KVPOOL_ERR_INVALID_ARG, "append: duplicate request id");
    const int64_t L0 = p->reqs[h_req_ids[i]].length, L1 = L0 + h_n_new[i];
    if (L1 / mp > p->cfg.max_blocks_per_request) return p->fail(KVPOOL_ERR_CAPACITY, "append: request too long");
    T += h_n_new[i];
    seals += L1 / mp - L0 / mp;
  }
  bool any_csa = false;
  for (int k : p->kinds) any_csa |= kind_has_csa(k);
  if (T > 0 && p->device() && (!d_k || !d_v || (any_csa && !d_idx_k)))
    return p->fail(KVPOOL_ERR_INVALID_ARG, "append: NULL input");
  if (T > INT32_MAX / 2) return p->fail(KVPOOL_ERR_INVALID_ARG, "append: too many tokens in one call");
  if (p->device() && ((reinterpret_cast<uintptr_t>(d_k) | reinterpret_cast<uintptr_t>(d_v) |
                       reinterpret_cast<uintptr_t>(d_idx_k)) % 16) != 0)
    return p->fail(KVPOOL_ERR_INVALID_ARG, "append: inputs must be 16-byte aligned");
  if (seals > (int64_t)p->free_blocks.size() || (p->hisparse() && seals > (int64_t)p->hot_free.size()))
    return p->fail(KVPOOL_ERR_OUT_OF_BLOCKS, "append: out of blocks");

  // reserve block ids: smallest free, requests in batch order, then positions;
  // with HiSparse each also takes the smallest free GPU slot for its CSA entries
  std::vector<std::vector<int32_t>> new_ids(n), new_locs(n);
  for (int i = 0; i < n; ++i) {
    const int64_t L0 = p->reqs[h_req_ids[i]].length, L1 = L0 + h_n_new[i];
    for (int64_t s = L0 / mp; s < L1 / mp; ++s) {
      const int32_t id = *p->free_blocks.begin();
      p->free_blocks.erase(p->free_blocks.begin());
      new_ids[i].push_back(id);
      new_locs[i].push_back(p->take_hot(id));
    }
  }

  int rc = 0;
  if (p->device() && T > 0) {
    // build the units: one per (request, block segment touched)
    std::vector<AppendUnit> phase1, phase2;
    int64_t row = 0;
    for (int i = 0; i < n; ++i) {
      const int32_t slot = h_req_ids[i];
      const int64_t L0 = p->reqs[slot].length, L1 = L0 + h_n_new[i];
      if (L1 == L0) continue;
      const int64_t s_first = L0 / mp, s_last = (L1 - 1) / mp;
      const int64_t ring_from_abs = std::max(L0, L1 - W);
      const bool split = s_last > s_first && (L0 % mp) != 0 && (L1 % mp) != 0;
      for (int64_t s = s_first; s <= s_last; ++s) {
        AppendUnit u{};
        u.slot = slot;
        u.seg = (int32_t)s;
        const int64_t a = std::max(L0, s * mp), b = std::min(L1, (s + 1) * mp);
        u.t0 = (int16_t)(a - s * mp);
        u.t1 = (int16_t)(b - s * mp);
        u.ring_from = (int16_t)(std::min<int64_t>(std::max(ring_from_abs, a), b) - s * mp);
        u.in_row = (int32_t)(row + (a - L0));
        u.block_id = (s < L1 / mp) ? new_ids[i][(size_t)(s - L0 / mp)] : -1;
        u.csa_slot = (s < L1 / mp) ? new_locs[i][(size_t)(s - L0 / mp)] : -1;
        (split && s == s_first ? phase1 : phase2).push_back(u);
      }
      row += h_n_new[i];
    }
    // a launch of few long units (a prefill chunk of one request) would leave
    // most SMs idle while each CTA walks its unit's tokens in order: such a
    // unit becomes one CTA for its HCA chain over all its tokens and `parts`
    // CTAs for its CSA / indexer groups and window tokens (ranges of whole CSA
    // groups; only the first may start and only the last may end inside a
    // group, so every State accumulator has one reader and one writer)
    {
      const int m = p->cfg.m;
      const int64_t base = (int64_t)(phase1.size() + phase2.size()) * append_slices(p->lay.pd) * p->cfg.n_layers;
      // (two CTAs per SM with half-size stages, or a split into the HCA chain
      // and one CSA part, measured slower: the CTAs that share an SM take
      // longer than the unsplit unit)
      const int parts = base > 0 ? (int)std::min<int64_t>(kMaxCsaParts, p->n_sms / base - 1) : 0;
      if (parts >= 2) {
        for (auto* list : {&phase1, &phase2}) {
          std::vector<AppendUnit> out;
          for (const AppendUnit& u : *list) {
            const int len = u.t1 - u.t0;
            if (len < kSplitMinTokens || ((u.t0 % m) != 0 && (u.t1 % m) != 0)) {
              out.push_back(u);
              continue;
            }
            AppendUnit hu = u;
            hu.role = kUnitHca;
            out.push_back(hu);
            int a = u.t0;
            for (int k = 1; k <= parts && a < u.t1; ++k) {
              const int b = k == parts ? (int)u.t1 : std::min<int>(u.t1, (u.t0 + (len * k + parts - 1) / parts + m - 1) / m * m);
              if (b <= a) continue;
              AppendUnit cu = u;
              cu.role = kUnitCsa;
              cu.t0 = (int16_t)a;
              cu.t1 = (int16_t)b;
              cu.in_row = u.in_row + (a - u.t0);
              out.push_back(cu);
              a = b;
            }
          }
          *list = std::move(out);
        }
      }
    }
    if (!p->append_params) p->append_params.reset(new AppendParams());
    AppendParams* ap = p->append_params.get();
    std::memset(static_cast<void*>(ap), 0, offsetof(AppendParams, units));
    ap->pool = p->lay.pd;
    std::memcpy(ap->layers, p->lay.layers, sizeof(ap->layers));
    ap->k = d_k;
    ap->v = d_v;
    ap->idx_k = d_idx_k;
    ap->rows = T;
    // units of many tokens (prefill chunks) in a launch too small to fill the
    // GPU stream their rows through shared memory (several stages in flight per
    // CTA); otherwise every thread loads its tokens directly, kTokGroup at a
    // time (enough in flight once there are a few CTAs per SM)
    int64_t longest = 0, ctas = 0;
    for (const auto* list : {&phase1, &phase2})
      for (const AppendUnit& u : *list) longest = std::max<int64_t>(longest, u.t1 - u.t0);
    ctas = (int64_t)(phase1.size() + phase2.size()) * append_slices(p->lay.pd) * p->cfg.n_layers;
    ap->staged = (longest >= kStagedMinTokens && ctas <= (int64_t)kStagedMaxCtasPerSm * p->n_sms) ? 1 : 0;
    ap->n_slices = ap->staged ? append_slices_staged(p->lay.pd) : append_slices(p->lay.pd);
    ap->stage_tokens = ap->staged ? append_stage_tokens(p->lay.pd, ap->n_slices) : 0;
    ap->epoch = p->epoch;
    // algorithmic bytes: inputs read + window tokens and new entries written
    const PoolDesc& pd = p->lay.pd;
    const int64_t fp8 = pd.cache_dtype == KVPOOL_FP8_E4M3 ? 1 : 0;
    const int64_t entry_algo = 2LL * pd.HD * pd.vs + 4 * fp8, idx_algo = idx_algo_bytes(pd);
    int64_t bytes = 0;
    for (int l = 0; l < p->cfg.n_layers; ++l) {
      const LayerDesc& d = p->lay.layers[l];
      bytes += T * 2LL * pd.HD * pd.isz + (d.has_csa ? T * (int64_t)pd.XD * pd.isz : 0);
      for (int i = 0; i < n; ++i) {
        const int64_t L0 = p->reqs[h_req_ids[i]].length, L1 = L0 + h_n_new[i];
        bytes += std::min<int64_t>(h_n_new[i], W) * entry_algo;
        if (d.has_csa) bytes += (L1 / p->cfg.m - L0 / p->cfg.m) * (entry_algo + idx_algo);
        if (d.has_hca) bytes += (L1 / mp - L0 / mp) * entry_algo;
      }
    }
    for (auto* list : {&phase1, &phase2}) {
      for (size_t o = 0; o < list->size() && rc == 0; o += kMaxAppendUnits) {
        ap->n_units = (int32_t)std::min<size_t>(kMaxAppendUnits, list->size() - o);
        std::memcpy(ap->units, list->data() + o, sizeof(AppendUnit) * ap->n_units);
        // a unit that seals a block with entries staged by earlier calls gets
        // copy CTAs for them
        ap->copy_slices = 0;
        for (int32_t k = 0; k < ap->n_units; ++k)
          if (any_csa && ap->units[k].role != kUnitCsa && ap->units[k].block_id >= 0 &&
              ap->units[k].t0 >= (p->cfg.idx_per_token ? 1 : p->cfg.m))
            ap->copy_slices = kSealCopySlices;  // staged entries (or per-token keys) move into the block
        rc = p->launch(KVPOOL_KERNEL_APPEND, bytes, stream, [&](int* nk) { return launch_append(*ap, p->cfg.n_layers, stream, nk); });
        bytes = 0;
      }
    }
  }
  if (rc != 0) {  // undo the reservation: nothing changes on error
    for (auto& v : new_ids)
      for (int32_t id : v) p->free_blocks.insert(id);
    for (auto& v : new_locs)
      for (int32_t l : v) p->release_loc(l);
    return p->cuda_fail((cudaError_t)rc, "append launch");
  }
  for (int i = 0; i < n; ++i) {
    Request& q = p->reqs[h_req_ids[i]];
    for (size_t j = 0; j < new_ids[i].size(); ++j) {
      const int32_t id = new_ids[i][j];
      p->refcount[id] = 1;
      p->loc[id] = new_locs[i][j];
      q.table.push_back(id);
    }
    q.length += h_n_new[i];
  }
  return KVPOOL_OK;
}

int kvpool_decode_attend(kvpool_t* p, int32_t layer, int32_t n, const int32_t* h_req_ids, const void* d_q,
                         const void* d_q_idx, int32_t top_k, float* d_out, int32_t* d_topk_out, void* stream) {
  if (!p) return KVPOOL_ERR_INVALID_ARG;
  if (layer < 0 || layer >= p->cfg.n_layers || n < 0 || top_k < 0)
    return p->fail(KVPOOL_ERR_INVALID_ARG, "decode_attend: bad layer, n or top_k");
  if (n > p->cfg.max_batch) return p->fail(KVPOOL_ERR_INVALID_ARG, "decode_attend: n > max_batch");
  if (top_k > p->cfg.max_top_k) return p->fail(KVPOOL_ERR_INVALID_ARG, "decode_attend: top_k > max_top_k");
  const LayerDesc& Ld = p->lay.layers[layer];
  if (n > 0 && (!h_req_ids || !d_q || !d_out || (Ld.has_csa && !d_q_idx)))
    return p->fail(KVPOOL_ERR_INVALID_ARG, "decode_attend: NULL pointer");
  for (int i = 0; i < n; ++i) {
    if (!p->req_ok(h_req_ids[i])) return p->fail(KVPOOL_ERR_BAD_REQUEST, "decode_attend: bad request id");
    if (p->reqs[h_req_ids[i]].length == 0) return p->fail(KVPOOL_ERR_INVALID_ARG, "decode_attend: empty request");
  }
  if (!p->device()) return p->fail(KVPOOL_ERR_INVALID_ARG, "decode_attend: pool has no device");
  if (n == 0) return KVPOOL_OK;
  if (reinterpret_cast<uintptr_t>(d_q) % 16 != 0) return p->fail(KVPOOL_ERR_INVALID_ARG, "decode_attend: q not 16-byte aligned");

  const PoolDesc& pd = p->lay.pd;
  const int CB = pd.csa_per_block;
  const int EPS = pd.idx_per_token ? CB / p->cfg.m : CB;  // CSA entries per score segment (a block, or a run of tokens)
  const int max_split_len = attend_max_split_len();
  if (!p->attend_params) p->attend_params.reset(new AttendParams());
  AttendParams* ap = p->attend_params.get();
  int rc = 0;
  p->epoch += 1;  // this call's epoch (HiSparse activity)
  for (int g0 = 0; g0 < n && rc == 0; g0 += kMaxAttendReqs) {
    const int gn = std::min(kMaxAttendReqs, n - g0);
    AttendParams& P = *ap;
    std::memset(static_cast<void*>(ap), 0, offsetof(AttendParams, reqs));
    P.pool = pd;
    P.layer = Ld;
    P.epoch = p->epoch;
    P.q = d_q;
    P.q_idx = d_q_idx;
    P.out = d_out;
    P.topk_out = d_topk_out;
    P.top_k = top_k;
    P.n = gn;
    P.row0 = g0;
    P.keys = reinterpret_cast<uint32_t*>(p->arena + p->lay.keys);
    P.key_stride = p->lay.key_stride;
    P.hist = reinterpret_cast<uint32_t*>(p->arena + p->lay.hist);
    P.counts = reinterpret_cast<uint32_t*>(p->arena + p->lay.counts);
    P.max_key_ctas = p->lay.max_key_ctas;
    P.sel = reinterpret_cast<int32_t*>(p->arena + p->lay.sel);
    P.cand = reinterpret_cast<uint2*>(p->arena + p->lay.cand);
    P.sync = reinterpret_cast<uint32_t*>(p->arena + p->lay.sync);
    P.thr = reinterpret_cast<uint32_t*>(p->arena + p->lay.thr);
    P.sel_stride = p->lay.sel_stride;
    P.part_o = reinterpret_cast<float*>(p->arena + p->lay.part_o);
    P.part_ml = reinterpret_cast<float*>(p->arena + p->lay.part_ml);
    // algorithmic bytes: codes + scales actually needed (layout padding excluded)
    const int64_t fp8 = pd.cache_dtype == KVPOOL_FP8_E4M3 ? 1 : 0;
    const int64_t entry_algo = 2LL * pd.HD * pd.vs + 4 * fp8;
    const int64_t idx_algo = idx_algo_bytes(pd);
    int64_t total_src = 0, total_segs = 0;
    int score_ctas = 0, key_ctas = 0;
    int64_t score_bytes = 0, attend_bytes = 0, out_bytes = 0;
    std::vector<int64_t> req_segs;  // segments each request has scored
    for (int i = 0; i < gn; ++i) {
      const Request& q = p->reqs[h_req_ids[g0 + i]];
      const int32_t n_cand = Ld.has_csa ? (int32_t)(q.length / p->cfg.m) : 0;
      const int32_t k = std::min(top_k, n_cand);
      if (k != n_cand && k > 0) {
        total_segs += (n_cand + EPS - 1) / EPS;
        req_segs.push_back((n_cand + EPS - 1) / EPS);
      }
    }
    // a score CTA takes a run of one request's segments; every request rounds
    // its CTA count up, so lengthen the runs until the CTAs fit one wave
    const int64_t score_target = (int64_t)kScoreCtasPerSm * p->n_sms;
    const int64_t attend_target = (int64_t)kAttendCtasPerSm * p->n_sms;
    const int64_t spc0 = std::min<int64_t>(4096, std::max<int64_t>(8, (total_segs + score_target - 1) / score_target));
    P.segs_per_cta = (int32_t)fit_one_wave(req_segs, spc0, 4096, score_target);
    for (int i = 0; i < gn; ++i) {
      const Request& q = p->reqs[h_req_ids[g0 + i]];
      AttendReq& R = P.reqs[i];
      R = AttendReq{};
      R.slot = h_req_ids[g0 + i];
      R.length = q.length;
      R.n_sealed = (int32_t)q.table.size();
      R.n_cand = Ld.has_csa ? (int32_t)(q.length / p->cfg.m) : 0;
      R.k = std::min(top_k, R.n_cand);
      R.select_all = (R.k == R.n_cand) ? 1 : 0;
      R.n_hca = Ld.has_hca ? (int32_t)(q.length / p->cfg.m_prime) : 0;
      R.w = (int32_t)std::min<int64_t>(q.length, p->cfg.n_win);
      R.score_base = score_ctas;
      const int nseg = (R.n_cand + EPS - 1) / EPS;
      if (!R.select_all && R.k > 0) {
        score_ctas += (nseg + P.segs_per_cta - 1) / P.segs_per_cta;
        score_bytes += (int64_t)R.n_cand * pd.idx_runs * idx_algo + (int64_t)nseg * 4 + (int64_t)pd.XD * pd.isz;
      }
      R.key_base = key_ctas;
      // select CTAs: one per 4096 candidates; at least one when topk_out needs its -1 padding
      if (Ld.has_csa || d_topk_out)
        key_ctas += std::max(1, (int)((R.n_cand + kSelectKeysPerCta - 1) / kSelectKeysPerCta));
      total_src += (int64_t)R.k + R.n_hca + R.w;
      attend_bytes += ((int64_t)R.k + R.n_hca + R.w) * entry_algo + ((int64_t)R.k + R.n_hca) * 4 +
                      (int64_t)pd.HD * pd.isz;
    }
    out_bytes = (int64_t)gn * pd.HD * 4;
    // each part is cut into splits, one CTA each, sized to fill the GPU
    int64_t src0 = 0, src1 = 0;
    for (int i = 0; i < gn; ++i) {
      src0 += (int64_t)P.reqs[i].n_hca + P.reqs[i].w;
      src1 += P.reqs[i].k;
    }
    // part 0 runs beside the select on the side stream when both parts have
    // work: two CTAs per SM leave room for the select and part 1
    const bool forked = Ld.has_csa && src1 > 0;
    const int64_t target0 = forked ? (int64_t)kPart0CtasPerSm * p->n_sms : attend_target;
    int64_t len0 = std::min<int64_t>(max_split_len, std::max<int64_t>(16, (src0 + target0 - 1) / target0));
    int64_t len1 = std::min<int64_t>(max_split_len, std::max<int64_t>(16, (src1 + attend_target - 1) / attend_target));
    // every request rounds its split count up: lengthen the splits until the
    // CTAs fit one wave (a few CTAs past it would double the part's time)
    std::vector<int64_t> src_0(gn), src_1(gn);
    for (int i = 0; i < gn; ++i) {
      src_0[i] = (int64_t)P.reqs[i].n_hca + P.reqs[i].w;
      src_1[i] = P.reqs[i].k;
    }
    len0 = fit_one_wave(src_0, len0, max_split_len, target0);
    len1 = fit_one_wave(src_1, len1, max_split_len, attend_target);
    int splits0 = 0, splits1 = 0, parts = 0;
    for (int pass = 0; pass < 2; ++pass) {
      splits0 = splits1 = parts = 0;
      for (int i = 0; i < gn; ++i) {
        AttendReq& R = P.reqs[i];
        R.split_len0 = (int32_t)len0;
        R.split_len1 = (int32_t)len1;
        R.n_split0 = (int32_t)(((int64_t)R.n_hca + R.w + len0 - 1) / len0);
        R.n_split1 = (int32_t)(((int64_t)R.k + len1 - 1) / len1);
        R.cta_base0 = splits0;
        R.cta_base1 = splits1;
        R.part_base = parts;
        splits0 += R.n_split0;
        splits1 += R.n_split1;
        parts += R.n_split0 + R.n_split1;
      }
      if (parts <= kMaxSplits) break;
      len0 = len1 = max_split_len;
    }
    if (parts > kMaxSplits) {
      rc = -1;
      p->fail(KVPOOL_ERR_INVALID_ARG, "decode_attend: too many attention splits");
      break;
    }
    const int ctas0 = splits0, ctas1 = splits1;
    P.total_score_ctas = score_ctas;
    P.total_key_ctas = key_ctas;
    P.total_ctas0 = ctas0;
    P.total_ctas1 = ctas1;
    int64_t bytes1 = 0;
    for (int i = 0; i < gn; ++i) bytes1 += (int64_t)P.reqs[i].k * (entry_algo + 4);
    const int64_t bytes0 = attend_bytes - bytes1;
    // [HCA | window] attention needs no top-k: after the indexer scan (which
    // wants every SM) it runs on the side stream, beside the latency-bound
    // select passes; the [selected CSA] part follows the select
    const bool fork = Ld.has_csa && ctas0 > 0 && ctas1 > 0;
    void* s0 = fork ? (void*)p->side : stream;
    if (rc == 0 && Ld.has_csa)
      rc = p->launch(KVPOOL_KERNEL_SCORE, score_bytes, stream, [&](int* nk) { return launch_score(P, stream, nk); });
    if (rc == 0 && fork) {
      cudaError_t e = cudaEventRecord(p->ev_fork, (cudaStream_t)stream);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(p->side, p->ev_fork, 0);
      if (e != cudaSuccess) rc = (int)e;
    }
    if (rc == 0)
      rc = p->launch(KVPOOL_KERNEL_ATTEND, bytes0, s0, [&](int* nk) { return launch_attend(P, 0, ctas0, s0, nk); });
    if (rc == 0 && key_ctas > 0)
      rc = p->launch(KVPOOL_KERNEL_SELECT, 0, stream, [&](int* nk) { return launch_select(P, stream, nk, !fork); });
    if (rc == 0)
      rc = p->launch(KVPOOL_KERNEL_ATTEND, bytes1, stream, [&](int* nk) { return launch_attend(P, 1, ctas1, stream, nk); });
    if (fork) {
      cudaError_t e = cudaEventRecord(p->ev_join, p->side);
      if (e == cudaSuccess) e = cudaStreamWaitEvent((cudaStream_t)stream, p->ev_join, 0);
      if (e != cudaSuccess && rc == 0) rc = (int)e;
    }
    if (rc == 0) rc = p->launch(KVPOOL_KERNEL_COMBINE, out_bytes, stream, [&](int* nk) { return launch_combine(P, stream, nk); });
  }
  if (rc != 0) p->epoch -= 1;
  if (rc == -1) return KVPOOL_ERR_INVALID_ARG;
  if (rc != 0) return p->cuda_fail((cudaError_t)rc, "decode_attend launch");
  return KVPOOL_OK;
}

int kvpool_request_info(const kvpool_t* p, int32_t r, kvpool_info* info, int32_t* ids, int32_t cap) {
  if (!p || !info) return KVPOOL_ERR_INVALID_ARG;
  if (!p->req_ok(r)) return KVPOOL_ERR_BAD_REQUEST;
  const Request& q = p->reqs[r];
  info->length = q.length;
  info->n_csa = q.length / p->cfg.m;
  info->n_hca = q.length / p->cfg.m_prime;
  info->csa_tail = (int32_t)(q.length % p->cfg.m);
  info->hca_tail = (int32_t)(q.length % p->cfg.m_prime);
  info->n_blocks = (int32_t)q.table.size();
  info->window = (int32_t)std::min<int64_t>(q.length, p->cfg.n_win);
  if (ids)
    for (int32_t s = 0; s < (int32_t)q.table.size() && s < cap; ++s) ids[s] = q.table[s];
  return KVPOOL_OK;
}

int kvpool_block_refcount(const kvpool_t* p, int32_t b) {
  if (!p || b < 0 || b >= p->cfg.max_blocks) return KVPOOL_ERR_INVALID_ARG;
  return p->refcount[b];
}

int kvpool_free_block_count(const kvpool_t* p) { return p ? (int)p->free_blocks.size() : KVPOOL_ERR_INVALID_ARG; }

int kvpool_get_layout(const kvpool_t* p, kvpool_layout* out, int32_t layer, kvpool_layer_layout* lo) {
  if (!p || !out) return KVPOOL_ERR_INVALID_ARG;
  const Layout& L = p->lay;
  out->entry_bytes = L.pd.entry_bytes;
  out->idx_entry_bytes = L.pd.idx_entry_bytes;
  out->csa_per_block = L.pd.csa_per_block;
  out->staging_base = L.pd.staging_base;
  out->table_offset = L.pd.table;
  out->error_offset = L.pd.err;
  out->total_bytes = L.total;
  out->csa_staging_base = L.pd.csa_staging_base;
  out->csa_hot_slots = p->cfg.csa_hot_slots;
  out->host_slot_bytes = L.pd.host_slot_bytes;
  out->csa_loc_offset = L.pd.csa_loc;
  out->activity_offset = L.pd.last_used;
  if (lo) {
    if (layer < 0 || layer >= p->cfg.n_layers) return KVPOOL_ERR_INVALID_ARG;
    const LayerDesc& d = L.layers[layer];
    lo->kind = d.kind;
    lo->pad = 0;
    lo->csa_offset = d.csa_pool;
    lo->csa_block_bytes = d.csa_stride;
    lo->idx_offset = d.idx_pool;
    lo->idx_block_bytes = d.idx_stride;
    lo->idx_scale_offset = d.idx_scale_off;
    lo->hca_offset = d.hca_pool;
    lo->hca_block_bytes = d.hca_stride;
    lo->ring_offset = d.ring;
    lo->ring_request_bytes = d.ring_req_bytes;
    lo->acc_offset = d.acc;
    lo->acc_request_bytes = d.acc_req_bytes;
    lo->csa_host_offset = d.csa_host_off;
  }
  return KVPOOL_OK;
}

int kvpool_wait_selftest(kvpool_t* p, void* stream) {
  if (!p) return KVPOOL_ERR_INVALID_ARG;
  if (!p->device()) return p->fail(KVPOOL_ERR_INVALID_ARG, "wait_selftest: pool has no device");
  const int rc = launch_wait_selftest(p->lay.pd, stream);
  if (rc != 0) return p->cuda_fail((cudaError_t)rc, "wait_selftest launch");
  return KVPOOL_OK;
}

int kvpool_check_device(kvpool_t* p, void* stream, uint32_t* word_out) {
  if (!p) return KVPOOL_ERR_INVALID_ARG;
  if (!p->device()) {
    if (word_out) *word_out = 0;
    return KVPOOL_OK;
  }
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t w = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(&w, p->arena + p->lay.pd.err, 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && w != 0) e = cudaMemset(p->arena + p->lay.pd.err, 0, 4);
  if (e != cudaSuccess) return p->cuda_fail(e, "check_device");
  if (word_out) *word_out = w;
  if (w != 0) return p->fail(KVPOOL_ERR_DEVICE_CHECK, "a kernel flagged an out-of-range index or a wait limit");
  return KVPOOL_OK;
}

int kvpool_profile_enable(kvpool_t* p, int kinds) {
  if (!p || (kinds & ~(KVPOOL_PROFILE_ALL | KVPOOL_PROFILE_COUNT))) return KVPOOL_ERR_INVALID_ARG;
  if (kinds) {
    p->settle_profile();
    p->timeline.clear();
    if (p->t0) {
      p->event_pool.push_back(p->t0);
      p->t0 = nullptr;
    }
    for (int k = 0; k < KVPOOL_KERNEL_COUNT; ++k) {
      p->prof_ms[k] = 0;
      p->prof_launches[k] = 0;
      p->prof_bytes[k] = 0;
    }
  }
  p->profiling = p->device() ? kinds : 0;
  return KVPOOL_OK;
}

int kvpool_profile_read(kvpool_t* p, int32_t kernel, double* ms_total, int64_t* launches, int64_t* bytes) {
  if (!p || kernel < 0 || kernel >= KVPOOL_KERNEL_COUNT) return KVPOOL_ERR_INVALID_ARG;
  p->settle_profile();
  if (ms_total) *ms_total = p->prof_ms[kernel];
  if (launches) *launches = p->prof_launches[kernel];
  if (bytes) *bytes = p->prof_bytes[kernel];
  return KVPOOL_OK;
}

int kvpool_profile_timeline(kvpool_t* p, int32_t cap, float* h_out) {
  if (!p || cap < 0 || (cap > 0 && !h_out)) return KVPOOL_ERR_INVALID_ARG;
  p->settle_profile();
  const int32_t n = (int32_t)std::min<size_t>((size_t)cap, p->timeline.size() / 3);
  std::memcpy(h_out, p->timeline.data(), sizeof(float) * 3 * (size_t)n);
  return n;
}

const char* kvpool_last_error(const kvpool_t* p) { return p ? p->err.c_str() : "NULL pool"; }

}  // extern "C"

// C ABI of libinjectscale.so: the GPU fact store, argument validation and
// the launch sequences of the retrieval and injection calls.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "injectscale.h"
#include "internal.h"

using namespace isk;

// Launch helpers shared by every kernel launch (declared in internal.h).
namespace isk {

void prefer_max_shared(const void* kern) {
  static std::mutex mu;
  static const void* done_kern[64];
  static int done_dev[64];
  static int n_done = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_done; ++i)
    if (done_kern[i] == kern && done_dev[i] == dev) return;
  cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                       (int)cudaSharedmemCarveoutMaxShared);
  if (n_done < 64) {
    done_kern[n_done] = kern;
    done_dev[n_done] = dev;
    ++n_done;
  }
}

cudaError_t ensure_dynamic_smem(const void* kern, size_t bytes) {
  static std::mutex mu;
  static const void* kern_set[64];
  static int dev_set[64];
  static size_t bytes_set[64];
  static int n_set = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  int slot = -1;
  for (int i = 0; i < n_set; ++i)
    if (kern_set[i] == kern && dev_set[i] == dev) slot = i;
  if (slot >= 0 && bytes_set[slot] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  if (slot < 0 && n_set < 64) slot = n_set++;
  if (slot >= 0) {
    kern_set[slot] = kern;
    dev_set[slot] = dev;
    bytes_set[slot] = bytes;
  }
  return cudaSuccess;
}

}  // namespace isk

namespace {

thread_local std::string g_err;

is_status_t fail(is_status_t s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

// On failure the runtime's pending error is read and cleared too, so that a
// failed launch is reported by this call and not again by a later one.
#define CUDA_TRY(expr)                                                                  \
  do {                                                                                  \
    cudaError_t e_ = (expr);                                                            \
    if (e_ != cudaSuccess) {                                                            \
      cudaGetLastError();                                                               \
      return fail(IS_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e_));         \
    }                                                                                   \
  } while (0)

int dtype_bytes(int dt) { return dt == IS_F32 ? 4 : 2; }
bool valid_kv_dtype(int dt) { return dt == IS_F32 || dt == IS_BF16 || dt == IS_F16; }
bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

class DeviceGuard {
 public:
  explicit DeviceGuard(int dev) {
    cudaGetDevice(&prev_);
    if (prev_ != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != prev_) cudaSetDevice(prev_);
  }

 private:
  int prev_ = 0;
};

struct EventPair {
  cudaEvent_t a, b;
};

}  // namespace

// Facts written to the device but not yet visible to retrieval: their embedding
// rows, tiles and arena tokens follow the store's current counters.
struct PendingFacts {
  int32_t user = -1;
  int32_t n = 0;
  int64_t f0 = 0, tok0 = 0, tokens = 0;
  int32_t max_len = 0;
  int32_t tiles_used = 0;
  std::vector<int32_t> rows, new_tiles;
};

// is_retrieve_and_inject_host: calls whose staged inputs fit in this many
// bytes run on the mapped buffer with no copies (a Llama-3.1-8B request, 3 KB,
// gains about 4 us a call); larger ones copy (a 100-request batch with its
// block tables, 250 KB, lost about 19 us reading them over the host link).
constexpr size_t kMappedStageBytes = 16384;

struct is_store {
  is_store_config_t cfg{};
  int device = 0;
  int num_sms = 0;
  int elt = 0;
  int emb_elt = 0;
  int64_t row_bytes = 0;          // H * D * elt
  int64_t tok_bytes = 0;          // L * 2 * row_bytes
  int64_t max_tiles = 0;
  int64_t score_stride = 0;
  int32_t seg_stride = 0;

  uint8_t* kv = nullptr;
  int64_t* fact_tok = nullptr;
  int32_t* fact_len = nullptr;
  int32_t* fact_user = nullptr;
  uint8_t* emb = nullptr;
  float* emb_inv_norm = nullptr;
  int32_t* tile_fact = nullptr;
  int32_t* tile_len = nullptr;    // length of the fact of each embedding row
  int4* user_meta = nullptr;      // {tile list offset, tiles, facts, first tile if consecutive else -1}
  int32_t* user_tiles = nullptr;
  int64_t* tile_tok = nullptr;    // arena token of the fact of each embedding row
  int64_t* fact_src = nullptr;    // plan: arena token of each planned fact [R][seg_stride]
  float* scores = nullptr;
  int64_t* ids_tmp = nullptr;
  float* scores_tmp = nullptr;
  int32_t* fact_seg_off = nullptr;
  int32_t* n_ids = nullptr;
  int32_t* seg_len_tmp = nullptr;
  int32_t* rows_tmp = nullptr;
  uint32_t* status = nullptr;
  int32_t* arrive = nullptr;      // per-query arrival counters of the retrieval kernel
  uint32_t* hist = nullptr;       // per-query cosine-bin counts of the retrieval kernel (left zeroed)
  // batched (tensor-core) retrieval
  __half* qg = nullptr;           // [max_queries][E] queries packed in group order
  float* q_inv = nullptr;
  int32_t* qperm = nullptr;
  int4* groups = nullptr;
  int32_t* counts = nullptr;
  alignas(64) unsigned char map_emb[128];
  alignas(64) unsigned char map_q[128];
  bool batched_ok = false;
  int32_t retrieval_mode = IS_RETRIEVAL_AUTO;
  uint64_t wait_ns = kWaitBudgetNs;   // budget of each pipeline wait (is_set_wait_budget)
  // segment plan of the last injecting call (reused by is_inject_layer)
  int32_t plan_R = 0;
  const int32_t* plan_seg_len = nullptr;
  int64_t scratch_bytes = 0;

  int64_t n_facts = 0, n_tokens = 0;
  int32_t n_tiles = 0;
  int32_t max_len = 0;
  std::vector<std::vector<int32_t>> user_tiles_h;
  std::vector<int32_t> user_nfacts_h;
  std::vector<int32_t> tile_rows_h;
  int32_t max_user_tiles = 0;
  int64_t max_user_facts = 0;

  // rotation table of the last RoPE parameters seen
  bool turns_valid = false;
  is_rope_params_t turns_key{};
  RopeTurns turns{};

  // open Context-Window Encoding capture
  bool cap_open = false;
  int64_t cap_src_tokens = 0;
  std::vector<uint8_t> cap_layers;
  int64_t* cap_seg = nullptr;     // [IS_MAX_CAPTURE_FACTS][2] {first source token, first arena token}
  uint32_t* work_ctr = nullptr;   // [kCtrBlockWords]: the inject kernel's chunk counters (two sets,
                                  // alternate launches), then its CTA arrival counter
  int work_parity = 0;
  PendingFacts cap_pending;

  // staging of is_retrieve_and_inject_host: a mapped page-locked host buffer
  // and (for inputs above kMappedStageBytes) a device buffer, inputs then
  // outputs, grown on demand
  uint8_t* stage_h = nullptr;
  uint8_t* stage_d = nullptr;
  size_t stage_d_bytes = 0;
  size_t stage_bytes = 0;
  // completion word of the mapped-buffer calls: the inject kernel's last CTA
  // stores the call's sequence number here (done_armed: the next inject
  // launch does so)
  uint32_t* done_h = nullptr;
  uint32_t done_seq = 0;
  bool done_armed = false;

  bool timing = false;
  std::vector<EventPair> pending[IS_NUM_STAGES];
  std::vector<cudaEvent_t> event_pool;
  double total_ms[IS_NUM_STAGES] = {};
  int64_t launches[IS_NUM_STAGES] = {};
};

namespace {

template <typename P>
is_status_t dev_alloc(P** p, size_t bytes, const char* what) {
  void* v = nullptr;
  cudaError_t e = cudaMalloc(&v, bytes > 0 ? bytes : 16);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(IS_ERR_OOM, "cudaMalloc(%zu bytes) for %s failed: %s", bytes, what,
                cudaGetErrorString(e));
  }
  *p = static_cast<P*>(v);
  return IS_OK;
}

// Page-locked host memory for the arena, mapped into the device's address
// space; *p is the device-side address (equal to the host one under UVA).
is_status_t host_alloc(uint8_t** p, size_t bytes) {
  void* h = nullptr;
  cudaError_t e = cudaHostAlloc(&h, bytes > 0 ? bytes : 16, cudaHostAllocMapped | cudaHostAllocPortable);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(IS_ERR_OOM, "cudaHostAlloc(%zu bytes) for the host K/V arena failed: %s", bytes,
                cudaGetErrorString(e));
  }
  void* d = nullptr;
  e = cudaHostGetDevicePointer(&d, h, 0);
  if (e != cudaSuccess || d != h) {
    cudaGetLastError();
    cudaFreeHost(h);
    return fail(IS_ERR_UNSUPPORTED, "host K/V arena is not mapped at its host address");
  }
  *p = static_cast<uint8_t*>(d);
  return IS_OK;
}

void free_store(is_store_t* s) {
  if (s->kv && s->cfg.kv_placement == IS_KV_HOST) {
    cudaFreeHost(s->kv);
    s->kv = nullptr;
  }
  if (s->stage_h) cudaFreeHost(s->stage_h);
  if (s->stage_d) cudaFree(s->stage_d);
  if (s->done_h) cudaFreeHost(s->done_h);
  s->stage_h = s->stage_d = nullptr;
  s->done_h = nullptr;
  void* ptrs[] = {s->kv, s->fact_tok, s->fact_len, s->fact_user, s->emb, s->emb_inv_norm,
                  s->tile_fact, s->tile_len, s->user_meta, s->tile_tok, s->fact_src, s->user_tiles, s->scores,
                  s->ids_tmp, s->scores_tmp, s->fact_seg_off, s->n_ids, s->seg_len_tmp,
                  s->rows_tmp, s->status, s->arrive, s->qg, s->q_inv, s->qperm, s->groups, s->counts,
                  s->cap_seg, s->work_ctr, s->hist};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  for (int st = 0; st < IS_NUM_STAGES; ++st)
    for (auto& ev : s->pending[st]) {
      cudaEventDestroy(ev.a);
      cudaEventDestroy(ev.b);
    }
  for (auto ev : s->event_pool) cudaEventDestroy(ev);
  delete s;
}

cudaEvent_t take_event(is_store_t* s) {
  if (!s->event_pool.empty()) {
    cudaEvent_t e = s->event_pool.back();
    s->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Brackets one launch with events when timing is enabled.
struct StageTimer {
  StageTimer(is_store_t* s, int stage, cudaStream_t st) : s_(s), stage_(stage), st_(st) {
    if (s_->timing) {
      ev_.a = take_event(s_);
      ev_.b = take_event(s_);
      cudaEventRecord(ev_.a, st_);
    }
  }
  ~StageTimer() {
    if (s_->timing) {
      cudaEventRecord(ev_.b, st_);
      s_->pending[stage_].push_back(ev_);
    }
  }
  is_store_t* s_;
  int stage_;
  cudaStream_t st_;
  EventPair ev_{};
};

void rope_inv_freq(const is_rope_params_t& r, int D, double* out) {
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < D / 2; ++i) {
    double w = std::pow(r.theta, -(2.0 * i) / D);
    if (r.scaling == 1) {
      const double lam = two_pi / w;
      const double high_wavelen = r.original_max_pos / r.high_freq_factor;
      const double low_wavelen = r.original_max_pos / r.low_freq_factor;
      if (lam > low_wavelen) {
        w = w / r.factor;
      } else if (lam >= high_wavelen) {
        const double s = (r.original_max_pos / lam - r.low_freq_factor) /
                         (r.high_freq_factor - r.low_freq_factor);
        w = (1.0 - s) * w / r.factor + s * w;
      }
    }
    out[i] = w;
  }
}

is_status_t check_rope(const is_rope_params_t* r, int D, int kv_dtype) {
  if (!r) return fail(IS_ERR_INVALID_ARG, "rope params are NULL");
  if (!(r->theta > 1.0) || !std::isfinite(r->theta))
    return fail(IS_ERR_INVALID_ARG, "rope theta must be finite and > 1");
  if (r->style != 0 && r->style != 1) return fail(IS_ERR_INVALID_ARG, "rope style must be 0 or 1");
  if (r->scaling == 1) {
    if (!(r->factor > 0) || !(r->low_freq_factor > 0) ||
        !(r->high_freq_factor > r->low_freq_factor) || r->original_max_pos <= 0)
      return fail(IS_ERR_INVALID_ARG, "bad Llama-3.1 scaling parameters");
  } else if (r->scaling != 0) {
    return fail(IS_ERR_INVALID_ARG, "rope scaling must be 0 or 1");
  }
  const int ve = 16 / dtype_bytes(kv_dtype);
  const int vecs = r->style == 0 ? D / 2 / ve : D / ve;
  if (vecs < 1 || vecs > 32)
    return fail(IS_ERR_UNSUPPORTED, "head_dim %d with this dtype/style needs %d vectors per %s", D,
                vecs, r->style == 0 ? "half head (max 32)" : "head (max 32)");
  return IS_OK;
}

bool same_rope(const is_rope_params_t& a, const is_rope_params_t& b) {
  return a.theta == b.theta && a.style == b.style && a.scaling == b.scaling && a.factor == b.factor &&
         a.low_freq_factor == b.low_freq_factor && a.high_freq_factor == b.high_freq_factor &&
         a.original_max_pos == b.original_max_pos;
}

RopeTurns make_turns(const is_rope_params_t& r, int D) {
  RopeTurns t;
  std::memset(&t, 0, sizeof t);
  double w[kMaxHalfDim];
  rope_inv_freq(r, D, w);
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < D / 2; ++i) {
    const double turns = w[i] / two_pi;
    t.hi[i] = (float)turns;
    t.lo[i] = (float)(turns - (double)t.hi[i]);
  }
  return t;
}

is_status_t check_cache(const is_store_t* s, const is_cache_desc_t* c, const void* kv_cache) {
  if (!c || !kv_cache) return fail(IS_ERR_INVALID_ARG, "cache descriptor or kv_cache is NULL");
  if (c->block_size <= 0 || c->num_blocks <= 0)
    return fail(IS_ERR_INVALID_ARG, "block_size and num_blocks must be > 0");
  if (c->dtype == IS_FP8_E4M3) {
    if (s->cfg.kv_dtype != IS_BF16 && s->cfg.kv_dtype != IS_F16)
      return fail(IS_ERR_UNSUPPORTED, "an FP8 cache takes a bf16 or fp16 store");
    if (!(c->k_scale > 0.f) || !(c->v_scale > 0.f) || !std::isfinite(c->k_scale) || !std::isfinite(c->v_scale))
      return fail(IS_ERR_INVALID_ARG, "FP8 cache scales must be finite and > 0");
  } else if (c->dtype != s->cfg.kv_dtype) {
    return fail(IS_ERR_INVALID_ARG, "cache dtype %d differs from the store's kv dtype %d", c->dtype,
                s->cfg.kv_dtype);
  }
  if (((uintptr_t)kv_cache & 15) != 0) return fail(IS_ERR_INVALID_ARG, "kv_cache must be 16-byte aligned");
  return IS_OK;
}

// Bytes of one (layer, K or V) row of the cache and of one layer of the cache.
int64_t cache_row_bytes(const is_store_t* s, const is_cache_desc_t* c) {
  return c->dtype == IS_FP8_E4M3 ? s->row_bytes / s->elt : s->row_bytes;
}
int64_t cache_layer_bytes(const is_store_t* s, const is_cache_desc_t* c) {
  return 2LL * c->num_blocks * c->block_size * cache_row_bytes(s, c);
}

is_status_t upload_user_index(is_store_t* s, cudaStream_t st) {
  const int U = s->cfg.max_users;
  std::vector<int4> meta(U);
  std::vector<int32_t> tiles;
  tiles.reserve(s->n_tiles);
  for (int u = 0; u < U; ++u) {
    const std::vector<int32_t>& ut = s->user_tiles_h[u];
    bool consecutive = !ut.empty();
    for (size_t i = 1; i < ut.size() && consecutive; ++i) consecutive = ut[i] == ut[i - 1] + 1;
    meta[u] = make_int4((int32_t)tiles.size(), (int32_t)ut.size(), s->user_nfacts_h[u],
                        consecutive ? ut[0] : -1);
    tiles.insert(tiles.end(), ut.begin(), ut.end());
  }
  CUDA_TRY(cudaMemcpyAsync(s->user_meta, meta.data(), meta.size() * sizeof(int4), cudaMemcpyHostToDevice, st));
  if (!tiles.empty())
    CUDA_TRY(cudaMemcpyAsync(s->user_tiles, tiles.data(), tiles.size() * 4, cudaMemcpyHostToDevice, st));
  CUDA_TRY(cudaStreamSynchronize(st));   // host vectors die on return
  return IS_OK;
}

}  // namespace

void isk::set_last_error_message(const char* msg) { g_err = msg ? msg : ""; }

extern "C" {

const char* is_last_error_message(void) { return g_err.c_str(); }

const char* is_status_string(is_status_t s) {
  switch (s) {
    case IS_OK: return "IS_OK";
    case IS_ERR_INVALID_ARG: return "IS_ERR_INVALID_ARG";
    case IS_ERR_OOM: return "IS_ERR_OOM";
    case IS_ERR_CAPACITY: return "IS_ERR_CAPACITY";
    case IS_ERR_OUT_OF_RANGE: return "IS_ERR_OUT_OF_RANGE";
    case IS_ERR_CUDA: return "IS_ERR_CUDA";
    case IS_ERR_TIMEOUT: return "IS_ERR_TIMEOUT";
    case IS_ERR_DEVICE: return "IS_ERR_DEVICE";
    case IS_ERR_UNSUPPORTED: return "IS_ERR_UNSUPPORTED";
  }
  return "IS_ERR_UNKNOWN";
}

is_status_t is_rope_frequencies(const is_rope_params_t* rope, int32_t head_dim, double* out) {
  if (!rope || !out) return fail(IS_ERR_INVALID_ARG, "NULL argument");
  if (head_dim < 2 || head_dim > IS_MAX_HEAD_DIM || head_dim % 2)
    return fail(IS_ERR_INVALID_ARG, "head_dim must be even and <= %d", IS_MAX_HEAD_DIM);
  is_status_t st = check_rope(rope, head_dim, IS_BF16);
  if (st != IS_OK && st != IS_ERR_UNSUPPORTED) return st;
  rope_inv_freq(*rope, head_dim, out);
  return IS_OK;
}

is_status_t is_store_create(const is_store_config_t* config, int device, cudaStream_t stream,
                            is_store_t** out) {
  if (!config || !out) return fail(IS_ERR_INVALID_ARG, "NULL config or out");
  *out = nullptr;
  is_store_config_t c = *config;
  if (c.num_layers <= 0 || c.num_kv_heads <= 0 || c.head_dim <= 0 || c.emb_dim <= 0)
    return fail(IS_ERR_INVALID_ARG, "layers, kv heads, head_dim and emb_dim must be > 0");
  if (!valid_kv_dtype(c.kv_dtype)) return fail(IS_ERR_INVALID_ARG, "bad kv_dtype %d", c.kv_dtype);
  if (c.emb_dtype != IS_F16 && c.emb_dtype != IS_F32)
    return fail(IS_ERR_INVALID_ARG, "emb_dtype must be IS_F16 or IS_F32");
  if (c.max_facts <= 0 || c.max_tokens <= 0 || c.max_users <= 0)
    return fail(IS_ERR_INVALID_ARG, "max_facts, max_tokens and max_users must be > 0");
  if (c.max_facts >= (int64_t)INT32_MAX)
    return fail(IS_ERR_INVALID_ARG, "max_facts must be < 2^31");
  if (c.max_queries == 0) c.max_queries = 64;
  if (c.max_k == 0) c.max_k = 256;
  if (c.max_requests == 0) c.max_requests = c.max_queries;
  if (c.max_facts_per_user <= 0 || c.max_facts_per_user > c.max_facts) c.max_facts_per_user = c.max_facts;
  if (c.max_facts_per_user > IS_MAX_FACTS_PER_USER) c.max_facts_per_user = IS_MAX_FACTS_PER_USER;
  if (c.max_queries < 1 || c.max_queries > IS_MAX_QUERIES)
    return fail(IS_ERR_INVALID_ARG, "max_queries must be in [1, %d]", IS_MAX_QUERIES);
  if (c.max_k < 1 || c.max_k > IS_MAX_K) return fail(IS_ERR_INVALID_ARG, "max_k must be in [1, %d]", IS_MAX_K);
  if (c.max_requests < 1 || c.max_requests > IS_MAX_REQUESTS)
    return fail(IS_ERR_INVALID_ARG, "max_requests must be in [1, %d]", IS_MAX_REQUESTS);
  if (c.kv_placement != IS_KV_DEVICE && c.kv_placement != IS_KV_HOST)
    return fail(IS_ERR_INVALID_ARG, "kv_placement must be IS_KV_DEVICE or IS_KV_HOST");
  if (c.reserved != 0) return fail(IS_ERR_INVALID_ARG, "reserved config field must be 0");
  if (c.emb_dim % 8 != 0) return fail(IS_ERR_UNSUPPORTED, "emb_dim must be a multiple of 8");
  const int D = c.head_dim;
  if (!is_pow2(D) || D < 16 || D > IS_MAX_HEAD_DIM)
    return fail(IS_ERR_UNSUPPORTED, "head_dim must be a power of two in [16, %d]", IS_MAX_HEAD_DIM);
  const int elt = dtype_bytes(c.kv_dtype);
  const int64_t row_bytes = (int64_t)c.num_kv_heads * D * elt;
  if (row_bytes % 512 != 0 || !inject_shape_ok((int)row_bytes, std::max(c.max_requests, c.max_queries)))
    return fail(IS_ERR_UNSUPPORTED,
                "num_kv_heads * head_dim * elt (%lld B) must be a multiple of 512 and at most 32 KiB",
                (long long)row_bytes);

  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
    cudaGetLastError();
    return fail(IS_ERR_CUDA, "no CUDA device");
  }
  if (device < 0 || device >= ndev) return fail(IS_ERR_INVALID_ARG, "device %d out of range", device);
  DeviceGuard g(device);
  if (c.kv_placement == IS_KV_HOST) {
    int can_map = 0;
    cudaDeviceGetAttribute(&can_map, cudaDevAttrCanMapHostMemory, device);
    if (!can_map) return fail(IS_ERR_UNSUPPORTED, "device %d cannot map host memory", device);
  }

  is_store_t* s = new is_store_t();
  s->cfg = c;
  s->device = device;
  cudaDeviceGetAttribute(&s->num_sms, cudaDevAttrMultiProcessorCount, device);
  s->elt = elt;
  s->emb_elt = dtype_bytes(c.emb_dtype);
  s->row_bytes = row_bytes;
  s->tok_bytes = (int64_t)c.num_layers * 2 * row_bytes;
  s->max_tiles = (c.max_facts + kTile - 1) / kTile + c.max_users;
  s->score_stride = (c.max_facts_per_user + kTile - 1) / kTile * kTile;
  s->seg_stride = c.max_k + 1;
  s->user_tiles_h.assign(c.max_users, {});
  s->user_nfacts_h.assign(c.max_users, 0);

  is_status_t st = IS_OK;
  const size_t Q = c.max_queries, R = std::max(c.max_requests, c.max_queries);
#define ALLOC(ptr, bytes, what)                              \
  if ((st = dev_alloc(&s->ptr, (bytes), what)) != IS_OK) {    \
    free_store(s);                                           \
    return st;                                               \
  }
  if (c.kv_placement == IS_KV_HOST) {
    if ((st = host_alloc(&s->kv, (size_t)c.max_tokens * s->tok_bytes)) != IS_OK) {
      free_store(s);
      return st;
    }
  } else {
    ALLOC(kv, (size_t)c.max_tokens * s->tok_bytes, "K/V arena");
  }
  ALLOC(fact_tok, (size_t)c.max_facts * 8, "fact offsets");
  ALLOC(fact_len, (size_t)c.max_facts * 4, "fact lengths");
  ALLOC(fact_user, (size_t)c.max_facts * 4, "fact users");
  ALLOC(emb, (size_t)s->max_tiles * kTile * c.emb_dim * s->emb_elt, "embedding tiles");
  ALLOC(emb_inv_norm, (size_t)s->max_tiles * kTile * 4, "embedding norms");
  ALLOC(tile_fact, (size_t)s->max_tiles * kTile * 4, "tile fact ids");
  ALLOC(tile_len, (size_t)s->max_tiles * kTile * 4, "tile fact lengths");
  ALLOC(user_meta, (size_t)c.max_users * sizeof(int4), "user records");
  ALLOC(user_tiles, (size_t)s->max_tiles * 4, "user tiles");
  ALLOC(tile_tok, (size_t)s->max_tiles * kTile * 8, "tile fact tokens");
  ALLOC(scores, Q * s->score_stride * 4, "score scratch");
  ALLOC(ids_tmp, Q * c.max_k * 8, "id scratch");
  ALLOC(scores_tmp, Q * c.max_k * 4, "top-k score scratch");
  ALLOC(fact_seg_off, R * s->seg_stride * 4, "segment plan");
  ALLOC(fact_src, R * s->seg_stride * 8, "segment sources");
  ALLOC(n_ids, R * 4, "fact counts");
  ALLOC(seg_len_tmp, R * 4, "segment lengths");
  ALLOC(rows_tmp, (size_t)c.max_facts * 4, "row list");
  ALLOC(status, 4, "status word");
  ALLOC(arrive, Q * 4, "arrival counters");
  ALLOC(hist, Q * kCosBins * 4, "cosine bins");
  ALLOC(qg, Q * (size_t)c.emb_dim * 2, "packed queries");
  ALLOC(q_inv, Q * 4, "query norms");
  ALLOC(qperm, Q * 4, "query order");
  ALLOC(groups, Q * sizeof(int4), "query groups");
  ALLOC(counts, 8, "group counts");
  ALLOC(cap_seg, (size_t)std::min<int64_t>(c.max_facts, IS_MAX_CAPTURE_FACTS) * 16, "capture segments");
  ALLOC(work_ctr, kCtrBlockWords * 4, "inject chunk counters");
#undef ALLOC
  s->scratch_bytes = (int64_t)(Q * s->score_stride * 4 + Q * c.max_k * 12 + Q * kCosBins * 4 +
                               R * (s->seg_stride * 4 + 8) + (size_t)c.max_facts * 4 + 4);
  cudaError_t e = cudaMemsetAsync(s->status, 0, 4, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(s->user_meta, 0, (size_t)c.max_users * sizeof(int4), stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(s->arrive, 0, Q * 4, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(s->hist, 0, Q * kCosBins * 4, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(s->work_ctr, 0, kCtrBlockWords * 4, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    free_store(s);
    return fail(IS_ERR_CUDA, "store initialisation failed: %s", cudaGetErrorString(e));
  }
  // Tensor maps for the batched path (fp16 embeddings only).
  if (c.emb_dtype == IS_F16 && operand_map_bytes() <= sizeof(s->map_emb))
    s->batched_ok = make_operand_map(s->map_emb, s->emb, c.emb_dim, s->max_tiles * kTile, 128) &&
                    make_operand_map(s->map_q, s->qg, c.emb_dim, (int64_t)Q, 64);
  *out = s;
  return IS_OK;
}

is_status_t is_store_destroy(is_store_t* s) {
  if (!s) return fail(IS_ERR_INVALID_ARG, "NULL store");
  DeviceGuard g(s->device);
  cudaDeviceSynchronize();
  free_store(s);
  return IS_OK;
}

is_status_t is_store_info(const is_store_t* s, is_store_info_t* out) {
  if (!s || !out) return fail(IS_ERR_INVALID_ARG, "NULL argument");
  out->n_facts = s->n_facts;
  out->n_tokens = s->n_tokens;
  out->n_tiles = s->n_tiles;
  out->max_user_tiles = s->max_user_tiles;
  out->max_user_facts = s->max_user_facts;
  out->kv_bytes = s->cfg.max_tokens * s->tok_bytes;
  out->emb_bytes = s->max_tiles * kTile * s->cfg.emb_dim * s->emb_elt;
  out->scratch_bytes = s->scratch_bytes;
  out->num_sms = s->num_sms;
  out->kv_placement = s->cfg.kv_placement;
  return IS_OK;
}

// Validates n facts of one user and writes everything but their K/V: the
// embedding rows (and their norms), the per-fact table and the row -> fact
// map.  Nothing becomes visible until commit_facts.  Synchronous.
static is_status_t stage_facts(is_store_t* s, int32_t user, int32_t n, const int32_t* lengths,
                               const void* emb, cudaStream_t stream, PendingFacts* pf) {
  if (user < 0 || user >= s->cfg.max_users)
    return fail(IS_ERR_OUT_OF_RANGE, "user %d outside [0, %d)", user, s->cfg.max_users);
  int64_t tokens = 0;
  int32_t max_len = 0;
  for (int i = 0; i < n; ++i) {
    if (lengths[i] <= 0) return fail(IS_ERR_INVALID_ARG, "fact %d has length %d", i, lengths[i]);
    tokens += lengths[i];
    max_len = std::max(max_len, lengths[i]);
  }
  if (s->n_facts + n > s->cfg.max_facts)
    return fail(IS_ERR_CAPACITY, "store holds %lld of %lld facts; %d more do not fit",
                (long long)s->n_facts, (long long)s->cfg.max_facts, n);
  if (s->n_tokens + tokens > s->cfg.max_tokens)
    return fail(IS_ERR_CAPACITY, "store holds %lld of %lld tokens; %lld more do not fit",
                (long long)s->n_tokens, (long long)s->cfg.max_tokens, (long long)tokens);
  if ((int64_t)s->user_nfacts_h[user] + n > s->cfg.max_facts_per_user)
    return fail(IS_ERR_CAPACITY, "user %d would exceed max_facts_per_user", user);

  // Embedding rows: fill the user's last tile, then fresh tiles.
  std::vector<int32_t> rows(n);
  int32_t tiles_used = s->n_tiles;
  std::vector<int32_t> new_tiles;
  {
    int32_t last = s->user_tiles_h[user].empty() ? -1 : s->user_tiles_h[user].back();
    int32_t fill = last >= 0 ? s->tile_rows_h[last] : kTile;
    for (int i = 0; i < n; ++i) {
      if (fill == kTile) {
        if (tiles_used >= s->max_tiles) return fail(IS_ERR_CAPACITY, "embedding tiles exhausted");
        last = tiles_used++;
        new_tiles.push_back(last);
        fill = 0;
      }
      rows[i] = last * kTile + fill++;
    }
  }
  DeviceGuard g(s->device);
  // Embeddings, one copy per run of consecutive rows.
  const size_t erow = (size_t)s->cfg.emb_dim * s->emb_elt;
  for (int i = 0; i < n;) {
    int j = i + 1;
    while (j < n && rows[j] == rows[j - 1] + 1) ++j;
    CUDA_TRY(cudaMemcpyAsync(s->emb + (size_t)rows[i] * erow, (const uint8_t*)emb + (size_t)i * erow,
                             (size_t)(j - i) * erow, cudaMemcpyDefault, stream));
    i = j;
  }
  // Per-fact metadata and the row -> fact map.
  std::vector<int64_t> tok(n);
  std::vector<int32_t> users(n, user), fids(n);
  int64_t acc = s->n_tokens;
  for (int i = 0; i < n; ++i) {
    tok[i] = acc;
    acc += lengths[i];
    fids[i] = (int32_t)(s->n_facts + i);
  }
  const int64_t f0 = s->n_facts;
  CUDA_TRY(cudaMemcpyAsync(s->fact_tok + f0, tok.data(), (size_t)n * 8, cudaMemcpyHostToDevice, stream));
  CUDA_TRY(cudaMemcpyAsync(s->fact_len + f0, lengths, (size_t)n * 4, cudaMemcpyHostToDevice, stream));
  CUDA_TRY(cudaMemcpyAsync(s->fact_user + f0, users.data(), (size_t)n * 4, cudaMemcpyHostToDevice, stream));
  for (int i = 0; i < n;) {
    int j = i + 1;
    while (j < n && rows[j] == rows[j - 1] + 1) ++j;
    CUDA_TRY(cudaMemcpyAsync(s->tile_fact + rows[i], fids.data() + i, (size_t)(j - i) * 4,
                             cudaMemcpyHostToDevice, stream));
    CUDA_TRY(cudaMemcpyAsync(s->tile_len + rows[i], lengths + i, (size_t)(j - i) * 4,
                             cudaMemcpyHostToDevice, stream));
    CUDA_TRY(cudaMemcpyAsync(s->tile_tok + rows[i], tok.data() + i, (size_t)(j - i) * 8,
                             cudaMemcpyHostToDevice, stream));
    i = j;
  }
  CUDA_TRY(cudaMemcpyAsync(s->rows_tmp, rows.data(), (size_t)n * 4, cudaMemcpyHostToDevice, stream));
  CUDA_TRY(launch_emb_norms(s->emb, s->cfg.emb_dtype, s->cfg.emb_dim, s->rows_tmp, n,
                            s->emb_inv_norm, stream));
  CUDA_TRY(cudaStreamSynchronize(stream));
  pf->user = user;
  pf->n = n;
  pf->f0 = f0;
  pf->tok0 = s->n_tokens;
  pf->tokens = tokens;
  pf->max_len = max_len;
  pf->tiles_used = tiles_used;
  pf->rows = std::move(rows);
  pf->new_tiles = std::move(new_tiles);
  return IS_OK;
}

// Makes staged facts (whose K/V are in place) visible to retrieval.
static is_status_t commit_facts(is_store_t* s, const PendingFacts& pf, int64_t* ids_out, cudaStream_t stream) {
  const int32_t user = pf.user;
  for (int32_t t : pf.new_tiles) {
    s->user_tiles_h[user].push_back(t);
    s->tile_rows_h.push_back(0);
  }
  for (int i = 0; i < pf.n; ++i) s->tile_rows_h[pf.rows[i] / kTile] = pf.rows[i] % kTile + 1;
  s->n_tiles = pf.tiles_used;
  s->user_nfacts_h[user] += pf.n;
  s->max_user_tiles = std::max<int32_t>(s->max_user_tiles, (int32_t)s->user_tiles_h[user].size());
  s->max_user_facts = std::max<int64_t>(s->max_user_facts, s->user_nfacts_h[user]);
  s->max_len = std::max(s->max_len, pf.max_len);
  s->n_facts += pf.n;
  s->n_tokens += pf.tokens;
  if (ids_out)
    for (int i = 0; i < pf.n; ++i) ids_out[i] = pf.f0 + i;
  DeviceGuard g(s->device);
  return upload_user_index(s, stream);
}

is_status_t is_store_add_facts(is_store_t* s, int32_t user, int32_t n, const int32_t* lengths,
                               const void* k, const void* v, const void* emb, int64_t* ids_out,
                               cudaStream_t stream) {
  if (!s) return fail(IS_ERR_INVALID_ARG, "NULL store");
  if (n <= 0 || !lengths || !k || !v || !emb)
    return fail(IS_ERR_INVALID_ARG, "n must be > 0 and lengths, k, v, emb non-NULL");
  if (s->cap_open) return fail(IS_ERR_INVALID_ARG, "a capture is open; end or abort it first");
  PendingFacts pf;
  is_status_t st = stage_facts(s, user, n, lengths, emb, stream, &pf);
  if (st != IS_OK) return st;
  DeviceGuard g(s->device);
  const int L = s->cfg.num_layers;
  // K and V into the token-major arena [T][L][2][H][D].
  uint8_t* dst = s->kv + (size_t)pf.tok0 * s->tok_bytes;
  CUDA_TRY(cudaMemcpy2DAsync(dst, 2 * s->row_bytes, k, s->row_bytes, s->row_bytes,
                             (size_t)pf.tokens * L, cudaMemcpyDefault, stream));
  CUDA_TRY(cudaMemcpy2DAsync(dst + s->row_bytes, 2 * s->row_bytes, v, s->row_bytes, s->row_bytes,
                             (size_t)pf.tokens * L, cudaMemcpyDefault, stream));
  CUDA_TRY(cudaStreamSynchronize(stream));
  return commit_facts(s, pf, ids_out, stream);
}

// ---------------------------------------------------------------------------
// Context-Window Encoding capture.

is_status_t is_store_capture_begin(is_store_t* s, int32_t user, int32_t n, const int32_t* window,
                                   const int32_t* lengths, const void* emb, cudaStream_t stream) {
  if (!s) return fail(IS_ERR_INVALID_ARG, "NULL store");
  if (s->cap_open) return fail(IS_ERR_INVALID_ARG, "a capture is already open");
  if (n <= 0 || !window || !lengths || !emb)
    return fail(IS_ERR_INVALID_ARG, "n must be > 0 and window, lengths, emb non-NULL");
  if (n > IS_MAX_CAPTURE_FACTS)
    return fail(IS_ERR_UNSUPPORTED, "at most %d facts per capture", IS_MAX_CAPTURE_FACTS);
  if (s->n_facts + n > s->cfg.max_facts)
    return fail(IS_ERR_CAPACITY, "store holds %lld of %lld facts; %d more do not fit",
                (long long)s->n_facts, (long long)s->cfg.max_facts, n);
  std::vector<int64_t> seg(2 * (size_t)n);      // per fact: {source token of its first fact token, its first arena token}
  int64_t src = 0, dst = s->n_tokens;
  for (int i = 0; i < n; ++i) {
    if (window[i] < 0) return fail(IS_ERR_INVALID_ARG, "fact %d has window %d", i, window[i]);
    if (lengths[i] <= 0) return fail(IS_ERR_INVALID_ARG, "fact %d has length %d", i, lengths[i]);
    src += window[i];
    seg[2 * i] = src;
    seg[2 * i + 1] = dst;
    src += lengths[i];
    dst += lengths[i];
  }
  if (src > (int64_t)INT32_MAX) return fail(IS_ERR_UNSUPPORTED, "a capture may span at most 2^31-1 tokens");
  PendingFacts pf;
  is_status_t st = stage_facts(s, user, n, lengths, emb, stream, &pf);
  if (st != IS_OK) return st;
  DeviceGuard g(s->device);
  CUDA_TRY(cudaMemcpyAsync(s->cap_seg, seg.data(), seg.size() * 8, cudaMemcpyHostToDevice, stream));
  CUDA_TRY(cudaStreamSynchronize(stream));
  s->cap_pending = pf;
  s->cap_src_tokens = src;
  s->cap_layers.assign(s->cfg.num_layers, 0);
  s->cap_open = true;
  return IS_OK;
}

is_status_t is_store_capture_layer(is_store_t* s, int32_t layer, const void* k_pre_rope, const void* v,
                                   cudaStream_t stream) {
  if (!s) return fail(IS_ERR_INVALID_ARG, "NULL store");
  if (!s->cap_open) return fail(IS_ERR_INVALID_ARG, "no capture is open");
  if (layer < 0 || layer >= s->cfg.num_layers)
    return fail(IS_ERR_OUT_OF_RANGE, "layer %d outside [0, %d)", layer, s->cfg.num_layers);
  if (s->cap_layers[layer]) return fail(IS_ERR_INVALID_ARG, "layer %d was already captured", layer);
  if (!k_pre_rope || !v) return fail(IS_ERR_INVALID_ARG, "k_pre_rope or v is NULL");
  if ((((uintptr_t)k_pre_rope) | ((uintptr_t)v)) & 15)
    return fail(IS_ERR_INVALID_ARG, "k_pre_rope and v must be 16-byte aligned");
  DeviceGuard g(s->device);
  CaptureArgs ca{};
  ca.k = static_cast<const uint8_t*>(k_pre_rope);
  ca.v = static_cast<const uint8_t*>(v);
  ca.kv = s->kv;
  ca.seg = s->cap_seg;
  ca.n = s->cap_pending.n;
  ca.tok0 = s->cap_pending.tok0;
  ca.tokens = s->cap_pending.tokens;
  ca.L = s->cfg.num_layers;
  ca.layer = layer;
  ca.row_bytes = (int32_t)s->row_bytes;
  CUDA_TRY(launch_capture_layer(ca, LaunchCfg{stream, s->num_sms, false}));
  s->cap_layers[layer] = 1;
  return IS_OK;
}

is_status_t is_store_capture_end(is_store_t* s, int64_t* ids_out, cudaStream_t stream) {
  if (!s) return fail(IS_ERR_INVALID_ARG, "NULL store");
  if (!s->cap_open) return fail(IS_ERR_INVALID_ARG, "no capture is open");
  s->cap_open = false;
  for (int l = 0; l < s->cfg.num_layers; ++l)
    if (!s->cap_layers[l]) return fail(IS_ERR_INVALID_ARG, "layer %d was not captured; capture dropped", l);
  DeviceGuard g(s->device);
  CUDA_TRY(cudaStreamSynchronize(stream));
  return commit_facts(s, s->cap_pending, ids_out, stream);
}

is_status_t is_store_capture_abort(is_store_t* s) {
  if (!s) return fail(IS_ERR_INVALID_ARG, "NULL store");
  s->cap_open = false;
  return IS_OK;
}

// ---------------------------------------------------------------------------

static is_status_t check_retrieve(is_store_t* s, int32_t Q, const int32_t* users, const void* q_emb,
                                  int32_t k) {
  if (!s) return fail(IS_ERR_INVALID_ARG, "NULL store");
  if (Q < 1 || Q > s->cfg.max_queries)
    return fail(IS_ERR_INVALID_ARG, "Q=%d outside [1, %d]", Q, s->cfg.max_queries);
  if (k < 1 || k > s->cfg.max_k) return fail(IS_ERR_OUT_OF_RANGE, "k=%d outside [1, %d]", k, s->cfg.max_k);
  if (!users || !q_emb) return fail(IS_ERR_INVALID_ARG, "users or q_emb is NULL");
  if (((uintptr_t)q_emb & 15) != 0) return fail(IS_ERR_INVALID_ARG, "q_emb must be 16-byte aligned");
  return IS_OK;
}

static is_status_t run_retrieval(is_store_t* s, int32_t Q, const int32_t* users, const void* q_emb,
                                 int32_t k, int64_t* ids, float* scores, const int32_t* seg_start,
                                 int32_t* seg_len, const int32_t* block_table, int32_t max_blocks,
                                 cudaStream_t stream, int32_t* seg_len_copy = nullptr) {
  const LaunchCfg cfg{stream, s->num_sms, false};     // first kernel: stream order
  SimArgs sa{};
  sa.emb = s->emb;
  sa.emb_inv_norm = s->emb_inv_norm;
  sa.user_meta = s->user_meta;
  sa.user_tiles = s->user_tiles;
  sa.users = users;
  sa.q_emb = q_emb;
  sa.scores = s->scores;
  sa.score_stride = s->score_stride;
  sa.status = s->status;
  sa.Q = Q;
  sa.E = s->cfg.emb_dim;
  sa.max_users = s->cfg.max_users;
  const bool batched = s->batched_ok &&
                       (s->retrieval_mode == IS_RETRIEVAL_BATCHED ||
                        (s->retrieval_mode == IS_RETRIEVAL_AUTO && Q >= 32 && s->max_user_facts >= 1024));
  TopkArgs ta{};
  ta.scores = s->scores;
  ta.score_stride = s->score_stride;
  ta.users = users;
  ta.user_meta = s->user_meta;
  ta.user_tiles = s->user_tiles;
  ta.tile_fact = s->tile_fact;
  ta.tile_len = s->tile_len;
  ta.tile_tok = s->tile_tok;
  ta.fact_tok = s->fact_tok;
  ta.fact_src = seg_start ? s->fact_src : nullptr;
  ta.block_table = block_table;
  ta.max_blocks = max_blocks;
  ta.fact_len = s->fact_len;
  ta.seg_start = seg_start;
  ta.ids_out = ids;
  ta.scores_out = scores;
  ta.n_ids_out = seg_start ? s->n_ids : nullptr;
  ta.fact_seg_off = seg_start ? s->fact_seg_off : nullptr;
  ta.seg_stride = s->seg_stride;
  ta.seg_len = seg_start ? seg_len : nullptr;
  ta.seg_len_copy = seg_start ? seg_len_copy : nullptr;
  ta.status = s->status;
  ta.Q = Q;
  ta.k = k;
  ta.max_users = s->cfg.max_users;
  ta.hist = batched ? nullptr : s->hist;
  if (!batched) {
    StageTimer tm(s, IS_STAGE_SIMILARITY, stream);
    CUDA_TRY(launch_retrieve(sa, ta, s->cfg.emb_dtype, s->max_user_tiles, s->max_user_facts, s->arrive,
                             cfg));
    return IS_OK;
  }
  GroupArgs ga{};
  ga.users = users;
  ga.q_emb = q_emb;
  ga.Q = Q;
  ga.E = s->cfg.emb_dim;
  ga.user_meta = s->user_meta;
  ga.max_users = s->cfg.max_users;
  ga.qg = s->qg;
  ga.q_inv = s->q_inv;
  ga.qperm = s->qperm;
  ga.groups = s->groups;
  ga.counts = s->counts;
  ga.status = s->status;
  GemmArgs gg{};
  gg.groups = s->groups;
  gg.counts = s->counts;
  gg.qperm = s->qperm;
  gg.q_inv = s->q_inv;
  gg.user_meta = s->user_meta;
  gg.user_tiles = s->user_tiles;
  gg.emb_inv_norm = s->emb_inv_norm;
  gg.scores = s->scores;
  gg.score_stride = s->score_stride;
  gg.E = s->cfg.emb_dim;
  gg.status = s->status;
  gg.wait_ns = s->wait_ns;
  const LaunchCfg dep{stream, s->num_sms, true};
  {
    StageTimer tm(s, IS_STAGE_PLAN, stream);
    CUDA_TRY(launch_group(ga, cfg));
  }
  {
    StageTimer tm(s, IS_STAGE_SIMILARITY, stream);
    CUDA_TRY(launch_sim_gemm(gg, s->map_emb, s->map_q, Q, s->max_user_tiles, dep));
  }
  {
    StageTimer tm(s, IS_STAGE_TOPK, stream);
    CUDA_TRY(launch_topk_batched(ta, Q, s->cfg.max_users, s->max_user_facts, dep));
  }
  return IS_OK;
}

is_status_t is_retrieve_topk(is_store_t* s, int32_t Q, const int32_t* users, const void* q_emb,
                             int32_t k, int64_t* ids_out, float* scores_out, cudaStream_t stream) {
  is_status_t st = check_retrieve(s, Q, users, q_emb, k);
  if (st != IS_OK) return st;
  if (!ids_out || !scores_out) return fail(IS_ERR_INVALID_ARG, "ids_out or scores_out is NULL");
  DeviceGuard g(s->device);
  return run_retrieval(s, Q, users, q_emb, k, ids_out, scores_out, nullptr, nullptr, nullptr, 0, stream);
}

static is_status_t check_inject_common(is_store_t* s, int32_t R, const int32_t* seg_start,
                                       const is_rope_params_t* rope, const int32_t* block_table,
                                       int32_t max_blocks, const is_cache_desc_t* cache,
                                       void* kv_cache, int32_t facts_per_request) {
  if (!seg_start || !block_table) return fail(IS_ERR_INVALID_ARG, "seg_start or block_table is NULL");
  if (max_blocks < 1) return fail(IS_ERR_INVALID_ARG, "max_blocks_per_seq must be >= 1");
  is_status_t st = check_cache(s, cache, kv_cache);
  if (st != IS_OK) return st;
  st = check_rope(rope, s->cfg.head_dim, s->cfg.kv_dtype);
  if (st != IS_OK) return st;
  const int64_t bound = (int64_t)R * facts_per_request * std::max(1, s->max_len);
  if (bound >= (int64_t)INT32_MAX)
    return fail(IS_ERR_UNSUPPORTED, "a call may inject up to %lld tokens; the limit is 2^31-1",
                (long long)bound);
  return IS_OK;
}

// Layers [layer0, layer0 + n_layers) into a cache whose consecutive layers are
// layer_stride bytes apart (kv_cache points at layer layer0's K block).
static is_status_t launch_injection(is_store_t* s, int32_t R, const int64_t* ids, int32_t ids_stride,
                                    const int32_t* seg_len, const int32_t* seg_start,
                                    const is_rope_params_t* rope, const int32_t* block_table,
                                    int32_t max_blocks, const is_cache_desc_t* cache, void* kv_cache,
                                    int64_t* slot_mapping, cudaStream_t stream, int32_t layer0,
                                    int32_t n_layers, int64_t layer_stride, bool after_plan,
                                    void* const* layer_caches = nullptr) {
  InjectArgs a{};
  a.kv = s->kv;
  a.fact_tok = s->fact_tok;
  a.fact_len = s->fact_len;
  a.fact_user = s->fact_user;
  a.n_facts = s->n_facts;
  a.ids = ids;
  a.ids_stride = ids_stride;
  a.fact_src = s->fact_src;
  a.n_ids = s->n_ids;
  a.fact_seg_off = s->fact_seg_off;
  a.seg_stride = s->seg_stride;
  a.seg_len = seg_len;
  a.seg_start = seg_start;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.cache = static_cast<uint8_t*>(kv_cache);
  if (layer_caches) {
    a.per_layer = 1;
    for (int i = 0; i < n_layers; ++i) a.layer_cache[i] = static_cast<uint8_t*>(layer_caches[i]);
  }
  a.block_size = cache->block_size;
  a.num_blocks = cache->num_blocks;
  a.slot_mapping = slot_mapping;
  a.status = s->status;
  a.R = R;
  a.L = s->cfg.num_layers;
  a.layer0 = layer0;
  a.n_layers = n_layers;
  a.layer_stride = layer_stride;
  a.row_bytes = (int32_t)s->row_bytes;
  a.cache_row_bytes = (int32_t)cache_row_bytes(s, cache);
  a.wait_ns = s->wait_ns;
  a.work_ctr = s->work_ctr + (size_t)s->work_parity * kPoolCtrWords;
  a.work_ctr_next = s->work_ctr + (size_t)(s->work_parity ^ 1) * kPoolCtrWords;
  if (s->done_armed) {
    a.done_ctr = s->work_ctr + kDoneCtrWord;
    a.host_done = s->done_h;
    a.done_seq = s->done_seq;
  }
  a.k_inv = (float)(1.0 / (double)cache->k_scale);
  a.v_inv = (float)(1.0 / (double)cache->v_scale);
  const int ve = 16 / s->elt;
  a.half_vecs = s->cfg.head_dim / 2 / ve;
  a.head_vecs = s->cfg.head_dim / ve;
  // The rotation table of the last RoPE parameters is kept: serving loops pass
  // the same parameters on every call.
  if (!s->turns_valid || !same_rope(s->turns_key, *rope)) {
    s->turns = make_turns(*rope, s->cfg.head_dim);
    s->turns_key = *rope;
    s->turns_valid = true;
  }
  const RopeTurns& rt = s->turns;
  // A programmatic dependent launch only right after this call's own planning
  // (or retrieval) kernel: the inject kernel reads the caller's starts and
  // block table before its dependency wait, which is safe only when the
  // kernel before it does not write them.  A call that reuses an earlier plan
  // follows whatever the caller queued, so it launches in plain stream order.
  const LaunchCfg cfg{stream, s->num_sms, after_plan};
  StageTimer tm(s, IS_STAGE_INJECT, stream);
  CUDA_TRY(launch_inject(a, rt, s->cfg.kv_dtype, rope->style, s->cfg.kv_placement == IS_KV_HOST,
                         cache->dtype == IS_FP8_E4M3, cfg));
  s->work_parity ^= 1;
  return IS_OK;
}

// Arguments of the planning kernel for an explicit fact list.
static PlanArgs make_plan_args(is_store_t* s, int32_t R, const int64_t* fact_ids, const int32_t* n_ids,
                               int32_t ids_stride, const int32_t* users, const int32_t* seg_start,
                               const int32_t* block_table, int32_t max_blocks, int32_t* seg_len) {
  PlanArgs p{};
  p.ids = fact_ids;
  p.ids_stride = ids_stride;
  p.n_ids_in = n_ids;
  p.users = users;
  p.seg_start = seg_start;
  p.fact_len = s->fact_len;
  p.fact_user = s->fact_user;
  p.fact_tok = s->fact_tok;
  p.n_facts = s->n_facts;
  p.n_ids_out = s->n_ids;
  p.fact_seg_off = s->fact_seg_off;
  p.fact_src = s->fact_src;
  p.block_table = block_table;
  p.max_blocks = max_blocks;
  p.seg_stride = s->seg_stride;
  p.seg_len = seg_len;
  p.status = s->status;
  p.R = R;
  return p;
}

is_status_t is_inject(is_store_t* s, int32_t R, const int64_t* fact_ids, const int32_t* n_ids,
                      int32_t ids_stride, const int32_t* users, const int32_t* seg_start,
                      const is_rope_params_t* rope, const int32_t* block_table, int32_t max_blocks,
                      const is_cache_desc_t* cache, void* kv_cache, int32_t* seg_len_out,
                      int64_t* slot_mapping_out, cudaStream_t stream) {
  if (!s) return fail(IS_ERR_INVALID_ARG, "NULL store");
  if (R < 1 || R > s->cfg.max_requests)
    return fail(IS_ERR_INVALID_ARG, "R=%d outside [1, %d]", R, s->cfg.max_requests);
  if (ids_stride < 1 || ids_stride > s->cfg.max_k)
    return fail(IS_ERR_OUT_OF_RANGE, "ids_stride=%d outside [1, %d]", ids_stride, s->cfg.max_k);
  if (!fact_ids || !n_ids) return fail(IS_ERR_INVALID_ARG, "fact_ids or n_ids is NULL");
  is_status_t st = check_inject_common(s, R, seg_start, rope, block_table, max_blocks, cache, kv_cache,
                                       ids_stride);
  if (st != IS_OK) return st;
  DeviceGuard g(s->device);
  int32_t* seg_len = seg_len_out ? seg_len_out : s->seg_len_tmp;
  const PlanArgs p = make_plan_args(s, R, fact_ids, n_ids, ids_stride, users, seg_start, block_table,
                                    max_blocks, seg_len);
  {
    StageTimer tm(s, IS_STAGE_PLAN, stream);
    CUDA_TRY(launch_plan(p, LaunchCfg{stream, s->num_sms, false}));
  }
  s->plan_R = R;
  s->plan_seg_len = seg_len;
  return launch_injection(s, R, fact_ids, ids_stride, seg_len, seg_start, rope, block_table, max_blocks,
                          cache, kv_cache, slot_mapping_out, stream, 0, s->cfg.num_layers,
                          cache_layer_bytes(s, cache), true);
}

is_status_t is_inject_layers(is_store_t* s, int32_t layer0, int32_t n_layers, int32_t R,
                             const int64_t* fact_ids, const int32_t* n_ids, int32_t ids_stride,
                             const int32_t* users, const int32_t* seg_start, const is_rope_params_t* rope,
                             const int32_t* block_table, int32_t max_blocks, const is_cache_desc_t* cache,
                             void* const* layer_caches, int32_t* seg_len_out, int64_t* slot_mapping_out,
                             cudaStream_t stream) {
  if (!s) return fail(IS_ERR_INVALID_ARG, "NULL store");
  if (n_layers < 1 || n_layers > IS_MAX_LAYERS_PER_CALL)
    return fail(IS_ERR_OUT_OF_RANGE, "n_layers=%d outside [1, %d]", n_layers, IS_MAX_LAYERS_PER_CALL);
  if (layer0 < 0 || (int64_t)layer0 + n_layers > s->cfg.num_layers)
    return fail(IS_ERR_OUT_OF_RANGE, "layers [%d, %lld) outside [0, %d)", layer0,
                (long long)layer0 + n_layers, s->cfg.num_layers);
  if (R < 1 || R > s->cfg.max_requests)
    return fail(IS_ERR_INVALID_ARG, "R=%d outside [1, %d]", R, s->cfg.max_requests);
  if (!layer_caches) return fail(IS_ERR_INVALID_ARG, "layer_caches is NULL");
  const int32_t stride_for_bound = fact_ids ? ids_stride : s->cfg.max_k;
  is_status_t st = check_inject_common(s, R, seg_start, rope, block_table, max_blocks, cache, layer_caches[0],
                                       stride_for_bound);
  if (st != IS_OK) return st;
  for (int i = 1; i < n_layers; ++i)
    if ((st = check_cache(s, cache, layer_caches[i])) != IS_OK) return st;
  DeviceGuard g(s->device);
  const int32_t* seg_len = nullptr;
  if (fact_ids) {
    if (ids_stride < 1 || ids_stride > s->cfg.max_k)
      return fail(IS_ERR_OUT_OF_RANGE, "ids_stride=%d outside [1, %d]", ids_stride, s->cfg.max_k);
    if (!n_ids) return fail(IS_ERR_INVALID_ARG, "n_ids is NULL");
    int32_t* out = seg_len_out ? seg_len_out : s->seg_len_tmp;
    const PlanArgs p = make_plan_args(s, R, fact_ids, n_ids, ids_stride, users, seg_start, block_table,
                                      max_blocks, out);
    {
      StageTimer tm(s, IS_STAGE_PLAN, stream);
      CUDA_TRY(launch_plan(p, LaunchCfg{stream, s->num_sms, false}));
    }
    s->plan_R = R;
    s->plan_seg_len = out;
    seg_len = out;
  } else {
    if (s->plan_R != R || !s->plan_seg_len)
      return fail(IS_ERR_INVALID_ARG, "no segment plan of %d requests to reuse", R);
    seg_len = s->plan_seg_len;
  }
  return launch_injection(s, R, nullptr, 0, seg_len, seg_start, rope, block_table, max_blocks, cache,
                          layer_caches[0], slot_mapping_out, stream, layer0, n_layers, 0, fact_ids != nullptr,
                          layer_caches);
}

is_status_t is_inject_layer(is_store_t* s, int32_t layer, int32_t R, const int64_t* fact_ids,
                            const int32_t* n_ids, int32_t ids_stride, const int32_t* users,
                            const int32_t* seg_start, const is_rope_params_t* rope,
                            const int32_t* block_table, int32_t max_blocks, const is_cache_desc_t* cache,
                            void* layer_cache, int32_t* seg_len_out, int64_t* slot_mapping_out,
                            cudaStream_t stream) {
  if (s && (layer < 0 || layer >= s->cfg.num_layers))
    return fail(IS_ERR_OUT_OF_RANGE, "layer %d outside [0, %d)", layer, s->cfg.num_layers);
  void* const caches[1] = {layer_cache};
  return is_inject_layers(s, layer, 1, R, fact_ids, n_ids, ids_stride, users, seg_start, rope, block_table,
                          max_blocks, cache, caches, seg_len_out, slot_mapping_out, stream);
}

is_status_t is_retrieve_and_inject(is_store_t* s, int32_t Q, const int32_t* users, const void* q_emb,
                                   int32_t k, const int32_t* seg_start, const is_rope_params_t* rope,
                                   const int32_t* block_table, int32_t max_blocks,
                                   const is_cache_desc_t* cache, void* kv_cache, int64_t* ids_out,
                                   float* scores_out, int32_t* seg_len_out, int64_t* slot_mapping_out,
                                   cudaStream_t stream) {
  is_status_t st = check_retrieve(s, Q, users, q_emb, k);
  if (st != IS_OK) return st;
  if (Q > s->cfg.max_requests && Q > s->cfg.max_queries)
    return fail(IS_ERR_INVALID_ARG, "Q exceeds the store's request capacity");
  st = check_inject_common(s, Q, seg_start, rope, block_table, max_blocks, cache, kv_cache, k);
  if (st != IS_OK) return st;
  DeviceGuard g(s->device);
  int64_t* ids = ids_out ? ids_out : s->ids_tmp;
  float* scores = scores_out ? scores_out : s->scores_tmp;
  // The plan's segment lengths stay in the store, so a later layer call can
  // reuse the plan whatever becomes of the caller's arrays; the top-k writes
  // them to seg_len_out as well (device or mapped host memory).
  int32_t* seg_len = s->seg_len_tmp;
  st = run_retrieval(s, Q, users, q_emb, k, ids, scores, seg_start, seg_len, block_table, max_blocks,
                     stream, seg_len_out);
  if (st != IS_OK) return st;
  s->plan_R = Q;
  s->plan_seg_len = seg_len;
  return launch_injection(s, Q, ids, k, seg_len, seg_start, rope, block_table, max_blocks, cache,
                          kv_cache, slot_mapping_out, stream, 0, s->cfg.num_layers,
                          cache_layer_bytes(s, cache), true);
}

is_status_t is_retrieve_and_inject_host(is_store_t* s, int32_t Q, const int32_t* users, const void* q_emb,
                                        int32_t k, const int32_t* seg_start, const is_rope_params_t* rope,
                                        const int32_t* block_table, int32_t max_blocks,
                                        const is_cache_desc_t* cache, void* kv_cache, int64_t* ids_out,
                                        float* scores_out, int32_t* seg_len_out, cudaStream_t stream) {
  if (!s) return fail(IS_ERR_INVALID_ARG, "NULL store");
  if (Q < 1 || Q > s->cfg.max_queries)
    return fail(IS_ERR_INVALID_ARG, "Q=%d outside [1, %d]", Q, s->cfg.max_queries);
  if (k < 1 || k > s->cfg.max_k) return fail(IS_ERR_OUT_OF_RANGE, "k=%d outside [1, %d]", k, s->cfg.max_k);
  if (!users || !q_emb || !seg_start || !block_table)
    return fail(IS_ERR_INVALID_ARG, "users, q_emb, seg_start or block_table is NULL");
  if (max_blocks < 1) return fail(IS_ERR_INVALID_ARG, "max_blocks_per_seq=%d must be >= 1", max_blocks);
  auto up = [](size_t b) { return (b + 255) & ~(size_t)255; };
  const size_t emb_elt = s->cfg.emb_dtype == IS_F16 ? 2 : 4;
  const size_t b_users = up((size_t)Q * 4), b_q = up((size_t)Q * s->cfg.emb_dim * emb_elt);
  const size_t b_start = up((size_t)Q * 4), b_bt = up((size_t)Q * max_blocks * 4);
  const size_t b_ids = up((size_t)Q * k * 8), b_sc = up((size_t)Q * k * 4), b_len = up((size_t)Q * 4);
  const size_t in_bytes = b_users + b_q + b_start + b_bt, out_bytes = b_ids + b_sc + b_len;
  const size_t bytes = in_bytes + out_bytes;
  // Small inputs are read by the kernels straight from the mapped buffer and
  // the outputs written back into it: no copy-engine transfer on the call's
  // path.  Larger inputs (the block tables of many requests, which the inject
  // kernel reads once per chunk) cross the host link once, in one copy to the
  // device buffer, and the outputs return in one copy.
  const bool mapped = in_bytes <= kMappedStageBytes;
  DeviceGuard g(s->device);
  if (bytes > s->stage_bytes || (!mapped && s->stage_d_bytes < bytes)) {
    CUDA_TRY(cudaStreamSynchronize(stream));
    if (bytes > s->stage_bytes) {
      if (s->stage_h) cudaFreeHost(s->stage_h);
      s->stage_h = nullptr;
      s->stage_bytes = 0;
      void* h = nullptr;
      void* d = nullptr;
      if (cudaHostAlloc(&h, bytes, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
        cudaGetLastError();
        return fail(IS_ERR_OOM, "cudaHostAlloc(%zu bytes) for host staging failed", bytes);
      }
      if (cudaHostGetDevicePointer(&d, h, 0) != cudaSuccess || d != h) {
        cudaGetLastError();
        cudaFreeHost(h);
        return fail(IS_ERR_UNSUPPORTED, "host staging is not mapped at its host address");
      }
      s->stage_h = static_cast<uint8_t*>(h);
      s->stage_bytes = bytes;
    }
    if (!mapped && s->stage_d_bytes < bytes) {
      if (s->stage_d) cudaFree(s->stage_d);
      s->stage_d = nullptr;
      s->stage_d_bytes = 0;
      void* d = nullptr;
      if (cudaMalloc(&d, s->stage_bytes) != cudaSuccess) {
        cudaGetLastError();
        return fail(IS_ERR_OOM, "cudaMalloc(%zu bytes) for device staging failed", s->stage_bytes);
      }
      s->stage_d = static_cast<uint8_t*>(d);
      s->stage_d_bytes = s->stage_bytes;
    }
  }
  if (mapped && !s->done_h) {
    void* w = nullptr;
    if (cudaHostAlloc(&w, 128, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
      cudaGetLastError();
      return fail(IS_ERR_OOM, "cudaHostAlloc of the completion word failed");
    }
    void* wd = nullptr;
    if (cudaHostGetDevicePointer(&wd, w, 0) != cudaSuccess || wd != w) {
      cudaGetLastError();
      cudaFreeHost(w);
      return fail(IS_ERR_UNSUPPORTED, "the completion word is not mapped at its host address");
    }
    s->done_h = static_cast<uint32_t*>(w);
    *reinterpret_cast<volatile uint32_t*>(s->done_h) = 0u;
  }
  uint8_t* h = s->stage_h;
  std::memcpy(h, users, (size_t)Q * 4);
  std::memcpy(h + b_users, q_emb, (size_t)Q * s->cfg.emb_dim * emb_elt);
  std::memcpy(h + b_users + b_q, seg_start, (size_t)Q * 4);
  std::memcpy(h + b_users + b_q + b_start, block_table, (size_t)Q * max_blocks * 4);
  uint8_t* d = mapped ? h : s->stage_d;
  if (!mapped) CUDA_TRY(cudaMemcpyAsync(d, h, in_bytes, cudaMemcpyHostToDevice, stream));
  uint8_t* hout = h + in_bytes;
  uint8_t* dout = d + in_bytes;
  // Mapped buffer: the inject kernel, the call's last, stores this call's
  // sequence number into the completion word once all its writes are done,
  // and the top-k wrote the outputs into the buffer before that kernel's
  // dependency wait released.
  uint32_t seq = 0;
  if (mapped) {
    seq = s->done_seq + 1 == 0 ? 1 : s->done_seq + 1;
    s->done_seq = seq;
    s->done_armed = true;
  }
  is_status_t st = is_retrieve_and_inject(
      s, Q, reinterpret_cast<const int32_t*>(d), d + b_users, k, reinterpret_cast<const int32_t*>(d + b_users + b_q),
      rope, reinterpret_cast<const int32_t*>(d + b_users + b_q + b_start), max_blocks, cache, kv_cache,
      reinterpret_cast<int64_t*>(dout), reinterpret_cast<float*>(dout + b_ids),
      reinterpret_cast<int32_t*>(dout + b_ids + b_sc), nullptr, stream);
  s->done_armed = false;
  if (st != IS_OK) {
    cudaStreamSynchronize(stream);              // the staged inputs stay in use until the kernels ran
    return st;
  }
  if (!mapped) CUDA_TRY(cudaMemcpyAsync(hout, dout, out_bytes, cudaMemcpyDeviceToHost, stream));
  // The caller is blocked until the outputs arrive, so the thread spins: on
  // the completion word (mapped calls), which it sees about 1.7 us before
  // the stream reports the work done, with a look at the stream every 1024
  // polls so that a failed launch still ends the wait; else on the stream
  // (sleeping in cudaStreamSynchronize wakes about 1 us later).
  cudaError_t qe = cudaSuccess;
  if (mapped) {
    const volatile uint32_t* word = s->done_h;
    for (uint32_t polls = 1; *word != seq; ++polls) {
      if ((polls & 1023u) != 0) continue;
      const cudaError_t e = cudaStreamQuery(stream);
      if (e != cudaErrorNotReady) {
        qe = e;
        break;
      }
    }
  } else {
    while ((qe = cudaStreamQuery(stream)) == cudaErrorNotReady) {
    }
  }
  if (qe != cudaSuccess) return fail(IS_ERR_CUDA, "stream: %s", cudaGetErrorString(qe));
  if (ids_out) std::memcpy(ids_out, hout, (size_t)Q * k * 8);
  if (scores_out) std::memcpy(scores_out, hout + b_ids, (size_t)Q * k * 4);
  if (seg_len_out) std::memcpy(seg_len_out, hout + b_ids + b_sc, (size_t)Q * 4);
  return IS_OK;
}

struct is_host_call {
  is_store_t* s;
  int32_t Q, k, max_blocks;
  const int32_t* users;
  const void* q_emb;
  const int32_t* seg_start;
  const int32_t* block_table;
  is_rope_params_t rope;
  is_cache_desc_t cache;
  void* kv_cache;
  int64_t* ids;
  float* scores;
  int32_t* seg_len;
  cudaStream_t stream;
};

is_status_t is_host_call_prepare(is_store_t* s, int32_t Q, const int32_t* users, const void* q_emb, int32_t k,
                                 const int32_t* seg_start, const is_rope_params_t* rope,
                                 const int32_t* block_table, int32_t max_blocks, const is_cache_desc_t* cache,
                                 void* kv_cache, int64_t* ids_out, float* scores_out, int32_t* seg_len_out,
                                 cudaStream_t stream, is_host_call_t** call_out) {
  if (!call_out) return fail(IS_ERR_INVALID_ARG, "call_out is NULL");
  *call_out = nullptr;
  if (!s) return fail(IS_ERR_INVALID_ARG, "NULL store");
  if (Q < 1 || Q > s->cfg.max_queries)
    return fail(IS_ERR_INVALID_ARG, "Q=%d outside [1, %d]", Q, s->cfg.max_queries);
  if (k < 1 || k > s->cfg.max_k) return fail(IS_ERR_OUT_OF_RANGE, "k=%d outside [1, %d]", k, s->cfg.max_k);
  if (!users || !q_emb || !seg_start || !block_table || !rope || !cache || !kv_cache)
    return fail(IS_ERR_INVALID_ARG, "users, q_emb, seg_start, block_table, rope, cache or kv_cache is NULL");
  if (max_blocks < 1) return fail(IS_ERR_INVALID_ARG, "max_blocks_per_seq=%d must be >= 1", max_blocks);
  is_host_call_t* c = new (std::nothrow) is_host_call_t();
  if (!c) return fail(IS_ERR_OOM, "host call object");
  *c = is_host_call_t{s, Q, k, max_blocks, users, q_emb, seg_start, block_table, *rope, *cache, kv_cache,
                      ids_out, scores_out, seg_len_out, stream};
  *call_out = c;
  return IS_OK;
}

is_status_t is_host_call_run(is_host_call_t* c) {
  if (!c) return fail(IS_ERR_INVALID_ARG, "NULL host call");
  return is_retrieve_and_inject_host(c->s, c->Q, c->users, c->q_emb, c->k, c->seg_start, &c->rope,
                                     c->block_table, c->max_blocks, &c->cache, c->kv_cache, c->ids, c->scores,
                                     c->seg_len, c->stream);
}

is_status_t is_host_call_destroy(is_host_call_t* c) {
  delete c;
  return IS_OK;
}

is_status_t is_get_status(is_store_t* s, cudaStream_t stream, uint32_t* bits_out) {
  if (!s || !bits_out) return fail(IS_ERR_INVALID_ARG, "NULL argument");
  DeviceGuard g(s->device);
  uint32_t bits = 0;
  CUDA_TRY(cudaMemcpyAsync(&bits, s->status, 4, cudaMemcpyDeviceToHost, stream));
  CUDA_TRY(cudaMemsetAsync(s->status, 0, 4, stream));
  CUDA_TRY(cudaStreamSynchronize(stream));
  *bits_out = bits;
  if (bits & IS_ST_TIMEOUT) return fail(IS_ERR_TIMEOUT, "a device wait timed out (bits 0x%x)", bits);
  if (bits) return fail(IS_ERR_DEVICE, "device status bits 0x%x", bits);
  return IS_OK;
}

is_status_t is_set_retrieval_mode(is_store_t* s, int32_t mode) {
  if (!s) return fail(IS_ERR_INVALID_ARG, "NULL store");
  if (mode != IS_RETRIEVAL_AUTO && mode != IS_RETRIEVAL_PER_QUERY && mode != IS_RETRIEVAL_BATCHED)
    return fail(IS_ERR_INVALID_ARG, "unknown retrieval mode %d", mode);
  if (mode == IS_RETRIEVAL_BATCHED && !s->batched_ok)
    return fail(IS_ERR_UNSUPPORTED, "the batched path needs fp16 embeddings and tensor maps");
  s->retrieval_mode = mode;
  return IS_OK;
}

is_status_t is_set_wait_budget(is_store_t* s, int64_t budget_ns) {
  if (!s) return fail(IS_ERR_INVALID_ARG, "NULL store");
  if (budget_ns < 0 || budget_ns > (int64_t)kWaitBudgetNs)
    return fail(IS_ERR_INVALID_ARG, "budget_ns must be in [0, %llu]", (unsigned long long)kWaitBudgetNs);
  s->wait_ns = (uint64_t)budget_ns;
  return IS_OK;
}

is_status_t is_set_timing(is_store_t* s, int32_t enable) {
  if (!s) return fail(IS_ERR_INVALID_ARG, "NULL store");
  s->timing = enable != 0;
  return IS_OK;
}

static is_status_t collect_timing(is_store_t* s) {
  for (int st = 0; st < IS_NUM_STAGES; ++st) {
    for (auto& ev : s->pending[st]) {
      CUDA_TRY(cudaEventSynchronize(ev.b));
      float ms = 0.f;
      CUDA_TRY(cudaEventElapsedTime(&ms, ev.a, ev.b));
      s->total_ms[st] += ms;
      s->launches[st] += 1;
      s->event_pool.push_back(ev.a);
      s->event_pool.push_back(ev.b);
    }
    s->pending[st].clear();
  }
  return IS_OK;
}

is_status_t is_get_timing(is_store_t* s, int32_t stage, double* total_ms, int64_t* launches) {
  if (!s || !total_ms || !launches) return fail(IS_ERR_INVALID_ARG, "NULL argument");
  if (stage < 0 || stage >= IS_NUM_STAGES) return fail(IS_ERR_INVALID_ARG, "bad stage %d", stage);
  DeviceGuard g(s->device);
  is_status_t st = collect_timing(s);
  if (st != IS_OK) return st;
  *total_ms = s->total_ms[stage];
  *launches = s->launches[stage];
  return IS_OK;
}

is_status_t is_reset_timing(is_store_t* s) {
  if (!s) return fail(IS_ERR_INVALID_ARG, "NULL store");
  DeviceGuard g(s->device);
  is_status_t st = collect_timing(s);
  for (int i = 0; i < IS_NUM_STAGES; ++i) {
    s->total_ms[i] = 0;
    s->launches[i] = 0;
  }
  return st;
}

}  // extern "C"

// Host side of the C ABI declared in include/kvq.h: configuration checks,
// the packed layout inside the caller's buffer, split planning and launch
// dispatch. No device memory is allocated here.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <atomic>
#include <cstring>
#include <string>
#include <vector>

#include "kvq_internal.h"

namespace {

thread_local std::string g_err;

kvq_status fail(kvq_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
kvq_status fail(kvq_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

kvq_status cuda_fail(cudaError_t e, const char* what) {
  return fail(KVQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Kernels launch on the current device, which must be the one that holds the
// cache (a launch elsewhere would fault on the cache's addresses).
kvq_status check_device(const kvq_cache* h);

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

int codes_per_word(int bits) { return bits == 3 ? 10 : 32 / bits; }

int words_per_row(int bits) {
  const int cpw = codes_per_word(bits);
  return (kvq::kHeadDim + cpw - 1) / cpw;
}

// Byte layout of one layer; all offsets relative to the layer base.
struct TensorPlan {
  int64_t codes_off = 0, codes_sb = 0;
  int64_t meta_off = 0, meta_sb = 0;
  int64_t resid_off = 0, resid_sb = 0;
  int64_t rp_off = 0, rp_sb = 0;
  int64_t col_off = 0, col_sb = 0;
  int64_t val_off = 0, val_sb = 0;
  int meta_bytes = 0;
  int words = 0;
};

// One layer: its code widths and tensors, offsets relative to the layer base.
struct LayerPlan {
  int k_bits = 0, v_bits = 0;
  TensorPlan k, v;
  int64_t sink_k_off = 0, sink_v_off = 0, sink_sb = 0;  // fp16 sink tokens [n][sink_tokens][D]
  int64_t ctr_off = 0;  // uint32 split-merge counters [n_streams]
  int64_t base = 0;     // from the start of the buffer
};

struct Plan {
  int capacity = 0;
  int64_t n_streams = 0;
  std::vector<LayerPlan> layer;
  int64_t header_bytes = 256;
  int64_t total = 0;
};

kvq_status check_tensor(const char* name, int bits, int mode, int group, bool is_k) {
  if (bits != 3 && bits != 4 && bits != 8)
    return fail(KVQ_ERR_INVALID_ARG, "%s_bits must be 3, 4 or 8 (got %d)", name, bits);
  if (mode < KVQ_SYM_PER_TOKEN || mode > KVQ_CODEBOOK_PER_TOKEN)
    return fail(KVQ_ERR_INVALID_ARG, "%s_mode %d is not a kvq_mode", name, mode);
  if (mode == KVQ_CODEBOOK_PER_TOKEN && bits != 4)
    return fail(KVQ_ERR_UNSUPPORTED, "codebook groups are supported at 4 bits only");
  if (mode == KVQ_ASYM_PER_CHANNEL) {
    if (!is_k)
      return fail(KVQ_ERR_UNSUPPORTED, "per-channel grouping is supported for keys only");
    if (group != 64 && group != 128 && group != 256)
      return fail(KVQ_ERR_UNSUPPORTED, "%s_group (tokens per block) must be 64, 128 or 256 (got %d)",
                  name, group);
    return KVQ_OK;
  }
  if (mode == KVQ_SYM_PER_TOKEN && bits != 8)
    return fail(KVQ_ERR_UNSUPPORTED, "symmetric groups are supported at 8 bits only");
  if (mode == KVQ_CODEBOOK_PER_TOKEN && group < 16)
    return fail(KVQ_ERR_UNSUPPORTED, "codebook groups must span at least 16 channels");
  if (group != 16 && group != 32 && group != 64 && group != 128)
    return fail(KVQ_ERR_INVALID_ARG, "%s_group must be 16, 32, 64 or 128 channels (got %d)", name,
                group);
  if (group != kvq::kHeadDim && group % codes_per_word(bits) != 0)
    return fail(KVQ_ERR_UNSUPPORTED,
                "%s_group %d is not a multiple of the %d codes per word (3-bit groups must span "
                "the whole row)",
                name, group, codes_per_word(bits));
  return KVQ_OK;
}

kvq_status check_config(const kvq_config* c, const int32_t* layer_bits = nullptr) {
  if (!c) return fail(KVQ_ERR_INVALID_ARG, "config is NULL");
  if (c->num_layers < 1 || c->batch < 1 || c->num_kv_heads < 1 || c->max_seq < 1)
    return fail(KVQ_ERR_INVALID_ARG, "num_layers, batch, num_kv_heads and max_seq must be >= 1");
  if (c->head_dim != kvq::kHeadDim)
    return fail(KVQ_ERR_UNSUPPORTED, "head_dim must be 128 (got %d)", c->head_dim);
  if (c->max_seq > (1 << 24))
    return fail(KVQ_ERR_UNSUPPORTED, "max_seq above 16M tokens is not supported");
  if ((int64_t)c->batch * c->num_kv_heads > 65535)
    return fail(KVQ_ERR_UNSUPPORTED, "batch * num_kv_heads must be <= 65535");
  if (c->outliers_per_row < 0 || c->outliers_per_row > kvq::kMaxOutliers)
    return fail(KVQ_ERR_INVALID_ARG, "outliers_per_row must be in [0, %d]", kvq::kMaxOutliers);
  if (c->sink_tokens < 0 || c->sink_tokens > kvq::kMaxSinkTokens || c->sink_tokens >= c->max_seq)
    return fail(KVQ_ERR_INVALID_ARG, "sink_tokens must be in [0, %d] and below max_seq", kvq::kMaxSinkTokens);
  kvq_status s = check_tensor("k", c->k_bits, c->k_mode, c->k_group, true);
  if (s != KVQ_OK) return s;
  s = check_tensor("v", c->v_bits, c->v_mode, c->v_group, false);
  if (s != KVQ_OK) return s;
  const bool kcb = c->k_mode == KVQ_CODEBOOK_PER_TOKEN, vcb = c->v_mode == KVQ_CODEBOOK_PER_TOKEN;
  if (kcb != vcb) return fail(KVQ_ERR_UNSUPPORTED, "codebook codes are supported for keys and values together");
  if (kcb) {
    if (c->outliers_per_row != 0) return fail(KVQ_ERR_UNSUPPORTED, "codebook codes take no outliers");
    float mx = 0.0f;
    for (int i = 0; i < 16; ++i) {
      __half_raw hr;
      hr.x = c->codebook[i];
      const float f = __half2float(__half(hr));
      if (!std::isfinite(f)) return fail(KVQ_ERR_INVALID_ARG, "codebook level %d is not finite", i);
      mx = std::fmax(mx, std::fabs(f));
    }
    if (!(mx > 0.0f)) return fail(KVQ_ERR_INVALID_ARG, "the codebook has no nonzero level");
    // distinct levels closer than max|level| / 65536 could tie with a level
    // that is not next to the quantized value after fp32 rounding; the search
    // table of the quantizer assumes they do not
    float lv[16];
    for (int i = 0; i < 16; ++i) {
      __half_raw hr;
      hr.x = c->codebook[i];
      lv[i] = __half2float(__half(hr));
    }
    std::sort(lv, lv + 16);
    for (int i = 1; i < 16; ++i)
      if (lv[i] != lv[i - 1] && (double)lv[i] - (double)lv[i - 1] < (double)mx / 65536.0)
        return fail(KVQ_ERR_UNSUPPORTED, "codebook levels %g and %g are closer than max|level| / 65536",
                    (double)lv[i - 1], (double)lv[i]);
  }
  if (!layer_bits) return s;
  for (int l = 0; l < c->num_layers; ++l) {
    s = check_tensor("layer k", layer_bits[2 * l], c->k_mode, c->k_group, true);
    if (s == KVQ_OK) s = check_tensor("layer v", layer_bits[2 * l + 1], c->v_mode, c->v_group, false);
    if (s != KVQ_OK) {
      const std::string m = kvq_last_error();
      return fail(s, "layer %d: %s", l, m.c_str());
    }
  }
  return KVQ_OK;
}

void plan_tensor(const kvq_config& c, int bits, int cap, bool is_k, int64_t* cursor, TensorPlan* t) {
  const int mode = is_k ? c.k_mode : c.v_mode;
  const int group = is_k ? c.k_group : c.v_group;
  const int64_t n = (int64_t)c.batch * c.num_kv_heads;
  const int D = kvq::kHeadDim;
  t->words = words_per_row(bits);
  t->meta_bytes = (mode == KVQ_SYM_PER_TOKEN || mode == KVQ_CODEBOOK_PER_TOKEN) ? 2 : 4;
  auto take = [&](int64_t stream_bytes, int64_t* off, int64_t* sb) {
    *sb = round_up(stream_bytes, 16);
    *off = *cursor;
    *cursor = round_up(*cursor + n * *sb, 256);
  };
  take((int64_t)cap * t->words * 4, &t->codes_off, &t->codes_sb);
  if (mode == KVQ_ASYM_PER_CHANNEL) {
    take((int64_t)(cap / group) * D * 4, &t->meta_off, &t->meta_sb);
    take((int64_t)group * D * 2, &t->resid_off, &t->resid_sb);
  } else {
    take((int64_t)cap * (D / group) * t->meta_bytes, &t->meta_off, &t->meta_sb);
  }
  if (c.outliers_per_row > 0) {
    take((int64_t)(cap + 4) * 4, &t->rp_off, &t->rp_sb);
    take((int64_t)cap * c.outliers_per_row * 2, &t->col_off, &t->col_sb);
    take((int64_t)cap * c.outliers_per_row * 2, &t->val_off, &t->val_sb);
  }
}

// layer_bits: NULL (every layer takes c.k_bits / c.v_bits) or [num_layers][2].
Plan make_plan(const kvq_config& c, const int32_t* layer_bits = nullptr) {
  Plan p;
  int64_t gran = kvq::kTile;
  if (c.k_mode == KVQ_ASYM_PER_CHANNEL && c.k_group > gran) gran = c.k_group;
  p.capacity = (int)round_up(c.max_seq, gran);
  p.n_streams = (int64_t)c.batch * c.num_kv_heads;
  p.layer.resize(c.num_layers);
  int64_t base = p.header_bytes;
  for (int l = 0; l < c.num_layers; ++l) {
    LayerPlan& lp = p.layer[l];
    lp.k_bits = layer_bits ? layer_bits[2 * l] : c.k_bits;
    lp.v_bits = layer_bits ? layer_bits[2 * l + 1] : c.v_bits;
    int64_t cursor = 0;
    plan_tensor(c, lp.k_bits, p.capacity, true, &cursor, &lp.k);
    plan_tensor(c, lp.v_bits, p.capacity, false, &cursor, &lp.v);
    if (c.sink_tokens > 0) {
      lp.sink_sb = round_up((int64_t)c.sink_tokens * kvq::kHeadDim * 2, 256);
      lp.sink_k_off = cursor;
      cursor += p.n_streams * lp.sink_sb;
      lp.sink_v_off = cursor;
      cursor += p.n_streams * lp.sink_sb;
    }
    lp.ctr_off = cursor;
    cursor = round_up(cursor + p.n_streams * 4, 256);
    lp.base = base;
    base += cursor;
  }
  p.total = base;
  return p;
}

}  // namespace

struct kvq_cache {
  kvq_config cfg;
  Plan plan;
  unsigned char* base = nullptr;
  size_t bytes = 0;
  std::vector<int> len;
  int splits_override = 0;
  int sm_count = 0;
  int device = 0;  // device that holds the buffer; launches need it current
  std::vector<cudaEvent_t> step_events;  // kvq_decode_step: one per layer + 1, made on first use
  std::vector<std::vector<int32_t>> seq;  // per layer: the batch rows' own lengths (empty: all `len`)
  float cb_thr[16] = {};                 // codebook search table (codebook codes only)
  uint8_t cb_code[16] = {};

  ~kvq_cache() {
    for (cudaEvent_t e : step_events)
      if (e) cudaEventDestroy(e);
  }
};

namespace {

kvq_status check_device(const kvq_cache* h) {
  int dev = -1;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != h->device)
    return fail(KVQ_ERR_INVALID_ARG, "the current device is %d but the cache lives on device %d", dev,
                h->device);
  return KVQ_OK;
}

kvq::TensorDev tensor_dev(const kvq_cache* h, int layer, bool is_k) {
  const kvq_config& c = h->cfg;
  const LayerPlan& lp = h->plan.layer[layer];
  const TensorPlan& t = is_k ? lp.k : lp.v;
  unsigned char* lb = h->base + lp.base;
  kvq::TensorDev d;
  d.bits = is_k ? lp.k_bits : lp.v_bits;
  d.mode = is_k ? c.k_mode : c.v_mode;
  d.group = is_k ? c.k_group : c.v_group;
  d.words = t.words;
  d.meta_bytes = t.meta_bytes;
  d.codes = reinterpret_cast<uint32_t*>(lb + t.codes_off);
  d.codes_sstride = t.codes_sb / 4;
  d.meta = lb + t.meta_off;
  d.meta_sstride = t.meta_sb;
  d.resid = d.mode == KVQ_ASYM_PER_CHANNEL ? reinterpret_cast<__half*>(lb + t.resid_off) : nullptr;
  d.resid_sstride = t.resid_sb / 2;
  const bool out = c.outliers_per_row > 0;
  d.rowptr = out ? reinterpret_cast<int32_t*>(lb + t.rp_off) : nullptr;
  d.rowptr_sstride = t.rp_sb / 4;
  d.col = out ? reinterpret_cast<uint16_t*>(lb + t.col_off) : nullptr;
  d.val = out ? reinterpret_cast<__half*>(lb + t.val_off) : nullptr;
  d.out_sstride = t.col_sb / 2;
  return d;
}

kvq::LayerDev layer_dev(const kvq_cache* h, int layer) {
  kvq::LayerDev L;
  L.k = tensor_dev(h, layer, true);
  L.v = tensor_dev(h, layer, false);
  L.n_streams = (int)h->plan.n_streams;
  L.num_kv_heads = h->cfg.num_kv_heads;
  L.capacity = h->plan.capacity;
  L.outliers = h->cfg.outliers_per_row;
  L.status = reinterpret_cast<uint32_t*>(h->base);
  const LayerPlan& lp = h->plan.layer[layer];
  L.counters = reinterpret_cast<uint32_t*>(h->base + lp.base + lp.ctr_off);
  L.in_rows = 0;
  L.sink_tokens = h->cfg.sink_tokens;
  L.sink_k = h->cfg.sink_tokens ? reinterpret_cast<__half*>(h->base + lp.base + lp.sink_k_off) : nullptr;
  L.sink_v = h->cfg.sink_tokens ? reinterpret_cast<__half*>(h->base + lp.base + lp.sink_v_off) : nullptr;
  std::memcpy(L.codebook, h->cfg.codebook, sizeof L.codebook);
  std::memcpy(L.cb_thr, h->cb_thr, sizeof L.cb_thr);
  std::memcpy(L.cb_code, h->cb_code, sizeof L.cb_code);
  return L;
}

// The streams of batch row b alone (its num_kv_heads streams) as a layer:
// every per-stream array starts at the row's first stream.
kvq::LayerDev row_view(const kvq::LayerDev& L, int b) {
  kvq::LayerDev R = L;
  const int64_t s0 = (int64_t)b * L.num_kv_heads;
  for (kvq::TensorDev* T : {&R.k, &R.v}) {
    T->codes += s0 * T->codes_sstride;
    T->meta += s0 * T->meta_sstride;
    if (T->resid) T->resid += s0 * T->resid_sstride;
    if (T->rowptr) T->rowptr += s0 * T->rowptr_sstride;
    if (T->col) T->col += s0 * T->out_sstride;
    if (T->val) T->val += s0 * T->out_sstride;
  }
  R.n_streams = L.num_kv_heads;
  return R;
}

// Tokens of a layer held as sinks, and the tokens after them (the coded rows).
int sink_len(const kvq_config& c, int len) { return len < c.sink_tokens ? len : c.sink_tokens; }
int coded_len(const kvq_config& c, int len) { return len - sink_len(c, len); }

// fp16 rows [0, rows) of every stream of a [n][src_rows][D] input (or of a
// single [n][D] row, src_rows = 1) into the sink array at row `at`.
cudaError_t copy_sink_rows(const kvq::LayerDev& L, __half* dst, const void* src, int src_rows, int at, int rows,
                           cudaStream_t st) {
  const size_t row = (size_t)kvq::kHeadDim * 2;
  return cudaMemcpy2DAsync(dst + (size_t)at * kvq::kHeadDim, (size_t)L.sink_tokens * row, src, (size_t)src_rows * row,
                           (size_t)rows * row, (size_t)L.n_streams, cudaMemcpyDeviceToDevice, st);
}

int k_quant_len(const kvq_config& c, int len) {
  if (c.k_mode != KVQ_ASYM_PER_CHANNEL) return len;
  return len / c.k_group * c.k_group;
}

// Splits of the sequence: every (stream, split) is one CTA of equal work.
// With `slots` CTAs resident on the GPU at once, the time of a launch is
// about waves * (rows per CTA + fixed cost), waves = ceil(CTAs / slots), plus
// the merge of a stream's partials by its last CTA (one round of loads per
// 16 partials); the split count minimizing it balances wave quantization
// against short CTAs and long merges.
// lens: the batch rows' own lengths (variable lengths), or NULL when every
// row holds `len` tokens. With variable lengths a row of n tiles keeps
// ceil(n / tps) CTAs busy; the others of its grid row find no tiles.
void plan_splits(const kvq_cache* h, int len, int slots, int* splits, int* tiles_per_split,
                 const int32_t* lens = nullptr) {
  const int ntiles = (len + kvq::kTile - 1) / kvq::kTile;
  if (h->splits_override > 0) {
    int want = h->splits_override < ntiles ? h->splits_override : ntiles;
    int tps = (ntiles + want - 1) / want;
    *tiles_per_split = tps;
    *splits = (ntiles + tps - 1) / tps;
    return;
  }
  const int64_t n = h->plan.n_streams;
  if (slots < 1) slots = 1;
  const double fixed_rows = 192.0;  // pipeline fill, query load and merge, in rows
  double best = 1e300;
  int best_s = 1, best_tps = ntiles;
  const int s_max = ntiles < 4096 ? ntiles : 4096;
  for (int s = 1; s <= s_max; ++s) {
    const int tps = (ntiles + s - 1) / s;
    const int s2 = (ntiles + tps - 1) / tps;
    if (s2 != s) continue;  // same shape as a smaller s
    int64_t ctas = n * s2;
    double empty_rows = 0.0;  // CTAs past a short row still load the query and write an empty partial
    if (lens) {  // only the CTAs that hold tiles of their row do the work
      ctas = 0;
      for (int b = 0; b < h->cfg.batch; ++b)
        ctas += (int64_t)h->cfg.num_kv_heads * (((lens[b] + kvq::kTile - 1) / kvq::kTile + tps - 1) / tps);
      empty_rows = 96.0 * (double)(n * s2 - ctas) / (double)slots;
    }
    const int64_t waves = (ctas + slots - 1) / slots;
    const double merge_rows = s2 > 1 ? 48.0 * (double)((s2 + 15) / 16) : 0.0;
    const double t = (double)waves * ((double)tps * kvq::kTile + fixed_rows) + merge_rows + empty_rows;
    if (t < best * 0.999) {
      best = t;
      best_s = s2;
      best_tps = tps;
    }
  }
  *splits = best_s;
  *tiles_per_split = best_tps;
}

// Workspace bytes of the sink partials (at the front of the workspace).
size_t sink_part_bytes(const kvq_cache* h, int num_q_heads) {
  if (h->cfg.sink_tokens == 0) return 0;
  return (size_t)round_up((int64_t)h->cfg.batch * num_q_heads * kvq::kSinkPartRow * 4, 256);
}

size_t workspace_for(const kvq_cache* h, int num_q_heads, int splits) {
  const int64_t rows = (int64_t)h->cfg.batch * num_q_heads;
  return (size_t)(rows * splits * kvq::kHeadDim * 4 + round_up(rows * splits * 2 * 4, 256) + 256);
}

kvq_status check_layer(const kvq_cache* h, int layer) {
  if (!h) return fail(KVQ_ERR_INVALID_ARG, "cache handle is NULL");
  if (layer < 0 || layer >= h->cfg.num_layers)
    return fail(KVQ_ERR_INVALID_ARG, "layer %d out of range [0, %d)", layer, h->cfg.num_layers);
  return KVQ_OK;
}

}  // namespace

namespace kvq {
void set_error_message(const char* msg) { g_err = msg ? msg : ""; }

uint32_t* cache_status_word(kvq_cache* h) { return reinterpret_cast<uint32_t*>(h->base); }

kvq_status cache_device_is_current(const kvq_cache* h) { return check_device(h); }

static std::atomic<uint64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
}  // namespace kvq

extern "C" {

kvq_status kvq_cache_bytes_per_layer(const kvq_config* cfg, const int32_t* layer_bits, size_t* bytes) {
  if (!bytes) return fail(KVQ_ERR_INVALID_ARG, "bytes is NULL");
  kvq_status s = check_config(cfg, layer_bits);
  if (s != KVQ_OK) return s;
  *bytes = (size_t)make_plan(*cfg, layer_bits).total;
  return KVQ_OK;
}

kvq_status kvq_cache_bytes(const kvq_config* cfg, size_t* bytes) {
  return kvq_cache_bytes_per_layer(cfg, nullptr, bytes);
}

kvq_status kvq_cache_create_per_layer(const kvq_config* cfg, const int32_t* layer_bits, void* dev_buf,
                                      size_t bytes, void* stream, kvq_cache** out) {
  if (!out) return fail(KVQ_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  kvq_status s = check_config(cfg, layer_bits);
  if (s != KVQ_OK) return s;
  if (!dev_buf) return fail(KVQ_ERR_INVALID_ARG, "dev_buf is NULL");
  if (!aligned(dev_buf, 256)) return fail(KVQ_ERR_INVALID_ARG, "dev_buf must be 256-byte aligned");
  Plan p = make_plan(*cfg, layer_bits);
  if ((int64_t)bytes < p.total)
    return fail(KVQ_ERR_BUFFER_TOO_SMALL, "cache buffer has %zu bytes, needs %lld", bytes,
                (long long)p.total);
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, dev_buf);
  if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes");
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
    return fail(KVQ_ERR_INVALID_ARG, "dev_buf is not device memory");
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, attr.device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  e = cudaMemsetAsync(dev_buf, 0, (size_t)p.total, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  kvq_cache* h = new kvq_cache;
  h->cfg = *cfg;
  if (cfg->k_mode == KVQ_CODEBOOK_PER_TOKEN) kvq::codebook_search_table(cfg->codebook, h->cb_thr, h->cb_code);
  h->plan = p;
  h->base = static_cast<unsigned char*>(dev_buf);
  h->bytes = bytes;
  h->len.assign(cfg->num_layers, 0);
  h->seq.assign(cfg->num_layers, std::vector<int32_t>());
  h->sm_count = sms > 0 ? sms : 1;
  h->device = attr.device;
  *out = h;
  return KVQ_OK;
}

kvq_status kvq_cache_create(const kvq_config* cfg, void* dev_buf, size_t bytes, void* stream,
                            kvq_cache** out) {
  return kvq_cache_create_per_layer(cfg, nullptr, dev_buf, bytes, stream, out);
}

kvq_status kvq_cache_destroy(kvq_cache* cache) {
  delete cache;
  return KVQ_OK;
}

kvq_status kvq_prefill_quantize(kvq_cache* h, int32_t layer, const void* k, const void* v,
                                int32_t seq_len, void* stream) {
  kvq_status s = check_layer(h, layer);
  if (s != KVQ_OK) return s;
  s = check_device(h);
  if (s != KVQ_OK) return s;
  if (seq_len < 0) return fail(KVQ_ERR_INVALID_ARG, "seq_len must be >= 0");
  if (seq_len > h->cfg.max_seq)
    return fail(KVQ_ERR_CAPACITY, "seq_len %d exceeds max_seq %d", seq_len, h->cfg.max_seq);
  if (seq_len > 0) {
    if (!k || !v) return fail(KVQ_ERR_INVALID_ARG, "k and v must not be NULL");
    if (!aligned(k, 16) || !aligned(v, 16))
      return fail(KVQ_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  }
  kvq::LayerDev L = layer_dev(h, layer);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int ns = sink_len(h->cfg, seq_len), nq = seq_len - ns;
  if (ns > 0) {  // the first tokens stay in fp16
    cudaError_t e = copy_sink_rows(L, L.sink_k, k, seq_len, 0, ns, st);
    if (e == cudaSuccess) e = copy_sink_rows(L, L.sink_v, v, seq_len, 0, ns, st);
    if (e != cudaSuccess) return cuda_fail(e, "sink copy");
  }
  L.in_rows = seq_len;
  const __half* kq = seq_len > 0 ? static_cast<const __half*>(k) + (size_t)ns * kvq::kHeadDim : nullptr;
  const __half* vq = seq_len > 0 ? static_cast<const __half*>(v) + (size_t)ns * kvq::kHeadDim : nullptr;
  cudaError_t e = kvq::launch_prefill(L, kq, vq, nq, st);
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  if (nq > 0) kvq::count_launches(1);
  h->len[layer] = seq_len;
  h->seq[layer].clear();
  return KVQ_OK;
}

kvq_status kvq_prefill_quantize_varlen(kvq_cache* h, int32_t layer, const void* k, const void* v,
                                       int32_t seq_len, const int32_t* lens, void* stream) {
  kvq_status s = check_layer(h, layer);
  if (s != KVQ_OK) return s;
  const kvq_config& c = h->cfg;
  if (c.sink_tokens > 0) return fail(KVQ_ERR_UNSUPPORTED, "variable lengths are not combined with sink tokens");
  if (c.batch > kvq::kMaxVarlenBatch)
    return fail(KVQ_ERR_UNSUPPORTED, "variable lengths take at most %d batch rows", kvq::kMaxVarlenBatch);
  if (!lens) return fail(KVQ_ERR_INVALID_ARG, "lens must not be NULL");
  int mx = 0;
  for (int b = 0; b < c.batch; ++b) {
    if (lens[b] < 1 || lens[b] > seq_len)
      return fail(KVQ_ERR_INVALID_ARG, "lens[%d] = %d must be in [1, seq_len = %d]", b, lens[b], seq_len);
    mx = lens[b] > mx ? lens[b] : mx;
  }
  if (c.k_mode == KVQ_ASYM_PER_CHANNEL) {
    // per-channel key blocks start at each row's first token: one prefill per
    // batch row over its own tokens (its key blocks and fp16 residual)
    s = check_device(h);
    if (s != KVQ_OK) return s;
    if (seq_len > c.max_seq) return fail(KVQ_ERR_CAPACITY, "seq_len %d exceeds max_seq %d", seq_len, c.max_seq);
    if (!k || !v) return fail(KVQ_ERR_INVALID_ARG, "k and v must not be NULL");
    if (!aligned(k, 16) || !aligned(v, 16)) return fail(KVQ_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
    const kvq::LayerDev L = layer_dev(h, layer);
    const size_t row_elems = (size_t)c.num_kv_heads * seq_len * kvq::kHeadDim;
    for (int b = 0; b < c.batch; ++b) {
      kvq::LayerDev Lb = row_view(L, b);
      Lb.in_rows = seq_len;
      const cudaError_t e = kvq::launch_prefill(Lb, static_cast<const __half*>(k) + b * row_elems,
                                                static_cast<const __half*>(v) + b * row_elems, lens[b],
                                                static_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
      kvq::count_launches(1);
    }
  } else {
    // rows are coded independently: the padded rows past a batch row's length
    // are coded too and overwritten by that row's later appends
    s = kvq_prefill_quantize(h, layer, k, v, seq_len, stream);
    if (s != KVQ_OK) return s;
  }
  h->seq[layer].assign(lens, lens + c.batch);
  h->len[layer] = mx;
  return KVQ_OK;
}

kvq_status kvq_append_quantize(kvq_cache* h, int32_t layer, const void* k, const void* v,
                               void* stream) {
  kvq_status s = check_layer(h, layer);
  if (s != KVQ_OK) return s;
  s = check_device(h);
  if (s != KVQ_OK) return s;
  if (!k || !v) return fail(KVQ_ERR_INVALID_ARG, "k and v must not be NULL");
  if (!aligned(k, 16) || !aligned(v, 16))
    return fail(KVQ_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  const int pos = h->len[layer];
  if (pos >= h->cfg.max_seq)
    return fail(KVQ_ERR_CAPACITY, "layer %d is full (%d tokens)", layer, pos);
  kvq::LayerDev L = layer_dev(h, layer);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::vector<int32_t>& sq = h->seq[layer];
  if (!sq.empty()) {  // variable lengths: each batch row appends at its own length
    kvq::VarPos vp;
    std::memset(&vp, 0, sizeof vp);
    vp.on = 1;
    vp.hkv = h->cfg.num_kv_heads;
    vp.rows = h->cfg.batch;
    for (int b = 0; b < h->cfg.batch; ++b) vp.pos[b] = sq[b];
    cudaError_t e = kvq::launch_append(L, static_cast<const __half*>(k), static_cast<const __half*>(v), pos, vp, st);
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
    kvq::count_launches(1);
    int mx = 0;
    for (int32_t& x : sq) mx = ++x > mx ? x : mx;
    h->len[layer] = mx;
    return KVQ_OK;
  }
  if (pos < h->cfg.sink_tokens) {  // a sink token: kept in fp16 as it is
    cudaError_t e = copy_sink_rows(L, L.sink_k, k, 1, pos, 1, st);
    if (e == cudaSuccess) e = copy_sink_rows(L, L.sink_v, v, 1, pos, 1, st);
    if (e != cudaSuccess) return cuda_fail(e, "sink copy");
  } else {
    kvq::VarPos none;
    none.on = 0;
    none.hkv = 1;
    cudaError_t e = kvq::launch_append(L, static_cast<const __half*>(k), static_cast<const __half*>(v),
                                       pos - h->cfg.sink_tokens, none, st);
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
    kvq::count_launches(1);
  }
  h->len[layer] = pos + 1;
  return KVQ_OK;
}

kvq_status kvq_decode_workspace_bytes(const kvq_cache* h, int32_t num_q_heads, size_t* bytes) {
  if (!h || !bytes) return fail(KVQ_ERR_INVALID_ARG, "NULL argument");
  if (num_q_heads < 1) return fail(KVQ_ERR_INVALID_ARG, "num_q_heads must be >= 1");
  const int hkv = h->cfg.num_kv_heads;
  // the largest need over the layers (their code widths may differ)
  size_t need = 0;
  bool split = false;
  for (int l = 0; l < h->cfg.num_layers; ++l) {
    kvq::LayerDev L = layer_dev(h, l);
    if (num_q_heads % hkv == 0 && kvq::decode_pipe_supported(L, num_q_heads / hkv)) {
      const size_t b = kvq::decode_pipe_workspace_max(L, num_q_heads / hkv, h->sm_count);
      if (b > need) need = b;
    }
    split = true;  // the split decode serves every layer with variable lengths
  }
  if (split) {
    const int max_splits = h->plan.capacity / kvq::kTile;  // one tile per split at most
    const size_t b = workspace_for(h, num_q_heads, max_splits);
    if (b > need) need = b;
  }
  *bytes = need + sink_part_bytes(h, num_q_heads);
  return KVQ_OK;
}

kvq_status kvq_decode_attention(kvq_cache* h, int32_t layer, const void* q, int32_t num_q_heads,
                                float softmax_scale, void* out, int32_t out_dtype,
                                void* workspace, size_t ws_bytes, void* stream) {
  kvq_status s = check_layer(h, layer);
  if (s != KVQ_OK) return s;
  s = check_device(h);
  if (s != KVQ_OK) return s;
  if (!q || !out || !workspace) return fail(KVQ_ERR_INVALID_ARG, "q, out and workspace must not be NULL");
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(workspace, 16))
    return fail(KVQ_ERR_INVALID_ARG, "q, out and workspace must be 16-byte aligned");
  if (out_dtype != KVQ_F32 && out_dtype != KVQ_F16)
    return fail(KVQ_ERR_INVALID_ARG, "out_dtype must be KVQ_F32 or KVQ_F16");
  const int hkv = h->cfg.num_kv_heads;
  if (num_q_heads < hkv || num_q_heads % hkv != 0)
    return fail(KVQ_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d",
                num_q_heads, hkv);
  const int gqa = num_q_heads / hkv;
  int len = h->len[layer];
  if (len == 0) return fail(KVQ_ERR_INVALID_ARG, "layer %d is empty: attention is undefined", layer);
  kvq::LayerDev L = layer_dev(h, layer);
  if (!kvq::decode_supported(L, gqa))
    return fail(KVQ_ERR_UNSUPPORTED, "no decode kernel for this codec pair with %d query heads per kv-head",
                gqa);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  // fp16 sink tokens first: their attention is merged into the decode's output
  // (or is the output when no token is coded yet)
  const int nsink = sink_len(h->cfg, len), ncoded = len - nsink;
  const size_t sink_ws = sink_part_bytes(h, num_q_heads);
  if (ws_bytes < sink_ws)
    return fail(KVQ_ERR_BUFFER_TOO_SMALL, "workspace has %zu bytes, needs %zu", ws_bytes, sink_ws);
  float* sink_part = nullptr;
  if (nsink > 0) {
    sink_part = static_cast<float*>(workspace);
    cudaError_t e = kvq::launch_sink_attention(L, static_cast<const __half*>(q), num_q_heads, scale_log2, nsink,
                                               sink_part, ncoded == 0 ? out : nullptr, out_dtype, st);
    if (e != cudaSuccess) return cuda_fail(e, "sink attention launch");
    if (ncoded == 0) return KVQ_OK;
  }
  workspace = static_cast<unsigned char*>(workspace) + sink_ws;
  ws_bytes -= sink_ws;
  len = ncoded;
  kvq::DecodeArgs a;
  std::memset(&a, 0, sizeof a);
  a.gqa = gqa;
  a.num_q_heads = num_q_heads;
  a.sink_part = sink_part;
  if (!h->seq[layer].empty()) {  // variable lengths: each batch row its own tokens
    a.varlen = 1;
    for (int b = 0; b < h->cfg.batch; ++b) a.lens[b] = h->seq[layer][b];
  }
  if (kvq::decode_pipe_supported(L, gqa) && !a.varlen) {  // stream-K cuts equal-length streams
    const kvq::PipePlan pp = kvq::plan_decode_pipe(L, len, gqa, h->sm_count, h->splits_override);
    if (ws_bytes < pp.ws_bytes)
      return fail(KVQ_ERR_BUFFER_TOO_SMALL, "workspace has %zu bytes, needs %zu", ws_bytes, pp.ws_bytes);
    a.q = static_cast<const __half*>(q);
    a.out = out;
    a.out_dtype = out_dtype;
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    a.length = len;
    a.k_quant_len = k_quant_len(h->cfg, len);
    a.part_o = static_cast<float*>(workspace);
    cudaError_t e = kvq::launch_decode_pipe(L, a, pp, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return KVQ_OK;
  }
  int occ = 0;
  a.occupancy_out = &occ;
  cudaError_t e = kvq::launch_decode(L, a, st);
  if (e != cudaSuccess) return cuda_fail(e, "decode occupancy query");
  a.occupancy_out = nullptr;
  int splits = 1, tps = 1;
  plan_splits(h, len, h->sm_count * (occ > 0 ? occ : 1), &splits, &tps, a.varlen ? a.lens : nullptr);
  const size_t need = workspace_for(h, num_q_heads, splits);
  if (ws_bytes < need)
    return fail(KVQ_ERR_BUFFER_TOO_SMALL, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  a.q = static_cast<const __half*>(q);
  a.out = out;
  a.out_dtype = out_dtype;
  a.num_q_heads = num_q_heads;
  a.gqa = gqa;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.length = len;
  a.k_quant_len = k_quant_len(h->cfg, len);
  a.splits = splits;
  a.tiles_per_split = tps;
  const int64_t rows = (int64_t)h->cfg.batch * num_q_heads;
  a.part_o = static_cast<float*>(workspace);
  a.part_ml = a.part_o + rows * splits * kvq::kHeadDim;
  e = kvq::launch_decode(L, a, st);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return KVQ_OK;
}

kvq_status kvq_prefill_attention(kvq_cache* h, int32_t layer, const void* q, int32_t chunk, int32_t num_q_heads,
                                 float softmax_scale, void* out, int32_t out_dtype, void* stream) {
  kvq_status s = check_layer(h, layer);
  if (s != KVQ_OK) return s;
  s = check_device(h);
  if (s != KVQ_OK) return s;
  if (!q || !out) return fail(KVQ_ERR_INVALID_ARG, "q and out must not be NULL");
  if (!aligned(q, 16) || !aligned(out, 16)) return fail(KVQ_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  if (out_dtype != KVQ_F32 && out_dtype != KVQ_F16)
    return fail(KVQ_ERR_INVALID_ARG, "out_dtype must be KVQ_F32 or KVQ_F16");
  const int hkv = h->cfg.num_kv_heads;
  if (num_q_heads < hkv || num_q_heads % hkv != 0)
    return fail(KVQ_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d", num_q_heads, hkv);
  const int len = h->len[layer];
  if (len == 0) return fail(KVQ_ERR_INVALID_ARG, "layer %d is empty: attention is undefined", layer);
  if (chunk < 1 || chunk > len)
    return fail(KVQ_ERR_INVALID_ARG, "chunk %d must be in [1, %d] (the tokens cached)", chunk, len);
  const std::vector<int32_t>& sq = h->seq[layer];
  for (int32_t x : sq)  // variable lengths: every row's chunk is its own last `chunk` positions
    if (chunk > x) return fail(KVQ_ERR_INVALID_ARG, "chunk %d exceeds a batch row of %d tokens", chunk, x);
  if ((int64_t)chunk * (num_q_heads / hkv) > ((int64_t)1 << 30))
    return fail(KVQ_ERR_INVALID_ARG, "chunk * query heads per kv-head is too large");
  kvq::PrefillAttnArgs a;
  std::memset(&a, 0, sizeof a);
  a.q = static_cast<const __half*>(q);
  a.out = out;
  a.out_dtype = out_dtype;
  a.num_q_heads = num_q_heads;
  a.G = num_q_heads / hkv;
  a.chunk = chunk;
  a.length = len;
  a.sink_len = sink_len(h->cfg, len);
  a.kq = k_quant_len(h->cfg, coded_len(h->cfg, len));
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  if (!sq.empty()) {
    a.varlen = 1;
    for (int b = 0; b < h->cfg.batch; ++b) a.lens[b] = sq[b];
  }
  const kvq::LayerDev L = layer_dev(h, layer);
  const cudaError_t e = kvq::launch_prefill_attention(L, a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "prefill attention launch");
  kvq::count_launches(1);
  return KVQ_OK;
}

kvq_status kvq_decode_step(kvq_cache* h, const void* const* q, const void* const* k1, const void* const* v1,
                           int32_t num_q_heads, float softmax_scale, void* const* out, int32_t out_dtype,
                           void* workspace, size_t ws_bytes, void* stream, void* aux_stream) {
  if (!h) return fail(KVQ_ERR_INVALID_ARG, "cache handle is NULL");
  kvq_status s = check_device(h);
  if (s != KVQ_OK) return s;
  if (!q || !k1 || !v1 || !out) return fail(KVQ_ERR_INVALID_ARG, "q, k1, v1 and out must not be NULL");
  const int nl = h->cfg.num_layers;
  for (int l = 0; l < nl; ++l) {  // refuse the whole step before enqueuing any of it
    if (!q[l] || !k1[l] || !v1[l] || !out[l])
      return fail(KVQ_ERR_INVALID_ARG, "layer %d: q, k1, v1 and out must not be NULL", l);
    if (h->len[l] >= h->cfg.max_seq) return fail(KVQ_ERR_CAPACITY, "layer %d is full (%d tokens)", l, h->len[l]);
  }
  size_t need = 0;
  s = kvq_decode_workspace_bytes(h, num_q_heads, &need);
  if (s != KVQ_OK) return s;
  if (ws_bytes < need) return fail(KVQ_ERR_BUFFER_TOO_SMALL, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  cudaStream_t main_st = static_cast<cudaStream_t>(stream);
  cudaStream_t aux = static_cast<cudaStream_t>(aux_stream);
  if (aux && aux != main_st && h->step_events.empty()) {
    h->step_events.assign(nl + 1, nullptr);
    for (auto& e : h->step_events) {
      const cudaError_t ce = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
      if (ce != cudaSuccess) return cuda_fail(ce, "cudaEventCreateWithFlags");
    }
  }
  const bool two = aux && aux != main_st;
  if (two) {  // the step's appends start after everything already on `stream`
    cudaError_t ce = cudaEventRecord(h->step_events[nl], main_st);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(aux, h->step_events[nl], 0);
    if (ce != cudaSuccess) return cuda_fail(ce, "step ordering");
  }
  for (int l = 0; l < nl; ++l) {
    s = kvq_append_quantize(h, l, k1[l], v1[l], two ? aux : main_st);
    if (s != KVQ_OK) return s;
    if (two) {  // layer l's decode waits for layer l's append only
      cudaError_t ce = cudaEventRecord(h->step_events[l], aux);
      if (ce == cudaSuccess) ce = cudaStreamWaitEvent(main_st, h->step_events[l], 0);
      if (ce != cudaSuccess) return cuda_fail(ce, "step ordering");
    }
    s = kvq_decode_attention(h, l, q[l], num_q_heads, softmax_scale, out[l], out_dtype, workspace, ws_bytes,
                             main_st);
    if (s != KVQ_OK) return s;
  }
  return KVQ_OK;
}

kvq_status kvq_cache_set_decode_splits(kvq_cache* h, int32_t splits) {
  if (!h) return fail(KVQ_ERR_INVALID_ARG, "cache handle is NULL");
  if (splits < 0) return fail(KVQ_ERR_INVALID_ARG, "splits must be >= 0");
  h->splits_override = splits;
  return KVQ_OK;
}

kvq_status kvq_cache_get_layout(const kvq_cache* h, int32_t layer, kvq_layout* o) {
  kvq_status s = check_layer(h, layer);
  if (s != KVQ_OK) return s;
  if (!o) return fail(KVQ_ERR_INVALID_ARG, "out is NULL");
  std::memset(o, 0, sizeof *o);
  const int len = h->len[layer];
  kvq::LayerDev L = layer_dev(h, layer);
  o->capacity = h->plan.capacity;
  o->length = len;
  o->k_quantized_len = k_quant_len(h->cfg, coded_len(h->cfg, len));
  o->k_resid_len = coded_len(h->cfg, len) - o->k_quantized_len;
  o->sink_tokens = h->cfg.sink_tokens;
  o->sink_len = sink_len(h->cfg, len);
  o->sink_stream_bytes = h->plan.layer[layer].sink_sb;
  o->k_sink = L.sink_k;
  o->v_sink = L.sink_v;
  const LayerPlan& lp = h->plan.layer[layer];
  o->k_words_per_row = lp.k.words;
  o->v_words_per_row = lp.v.words;
  o->k_meta_entry_bytes = lp.k.meta_bytes;
  o->v_meta_entry_bytes = lp.v.meta_bytes;
  o->k_codes_stream_bytes = lp.k.codes_sb;
  o->v_codes_stream_bytes = lp.v.codes_sb;
  o->k_meta_stream_bytes = lp.k.meta_sb;
  o->v_meta_stream_bytes = lp.v.meta_sb;
  o->k_resid_stream_bytes = lp.k.resid_sb;
  o->out_rowptr_stream_bytes = lp.k.rp_sb;
  o->out_col_stream_bytes = lp.k.col_sb;
  o->out_val_stream_bytes = lp.k.val_sb;
  o->k_codes = L.k.codes;
  o->k_meta = L.k.meta;
  o->k_resid = L.k.resid;
  o->v_codes = L.v.codes;
  o->v_meta = L.v.meta;
  o->k_out_rowptr = L.k.rowptr;
  o->k_out_col = L.k.col;
  o->k_out_val = L.k.val;
  o->v_out_rowptr = L.v.rowptr;
  o->v_out_col = L.v.col;
  o->v_out_val = L.v.val;
  return KVQ_OK;
}

kvq_status kvq_cache_length(const kvq_cache* h, int32_t layer, int32_t* len) {
  kvq_status s = check_layer(h, layer);
  if (s != KVQ_OK) return s;
  if (!len) return fail(KVQ_ERR_INVALID_ARG, "len is NULL");
  *len = h->len[layer];
  return KVQ_OK;
}

kvq_status kvq_cache_seq_lengths(const kvq_cache* h, int32_t layer, int32_t* lens) {
  kvq_status s = check_layer(h, layer);
  if (s != KVQ_OK) return s;
  if (!lens) return fail(KVQ_ERR_INVALID_ARG, "lens is NULL");
  for (int b = 0; b < h->cfg.batch; ++b) lens[b] = h->seq[layer].empty() ? h->len[layer] : h->seq[layer][b];
  return KVQ_OK;
}

kvq_status kvq_cache_status(kvq_cache* h, void* stream, uint32_t* word) {
  if (!h) return fail(KVQ_ERR_INVALID_ARG, "cache handle is NULL");
  const kvq_status ds = check_device(h);
  if (ds != KVQ_OK) return ds;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  uint32_t w = 0;
  e = cudaMemcpy(&w, h->base, sizeof w, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy status");
  if (w != 0) {
    e = cudaMemset(h->base, 0, sizeof w);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset status");
    // a decode that gave up may have left split-merge counters set
    for (int l = 0; l < h->cfg.num_layers; ++l) {
      e = cudaMemset(h->base + h->plan.layer[l].base + h->plan.layer[l].ctr_off, 0,
                     (size_t)h->plan.n_streams * 4);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemset counters");
    }
  }
  if (word) *word = w;
  if (w & kvq::kStatusTimeout) return fail(KVQ_ERR_TIMEOUT, "a bounded device wait gave up (status 0x%x)", w);
  if (w) return fail(KVQ_ERR_DEVICE_STATUS, "device status word 0x%x", w);
  return KVQ_OK;
}

const char* kvq_last_error(void) { return g_err.c_str(); }

uint64_t kvq_kernel_launches(void) { return kvq::g_launches.load(std::memory_order_relaxed); }

int32_t kvq_version(void) { return 100; }

}  // extern "C"

// Host side of libdflash: argument validation, state and workspace layout,
// and the launch sequence of each entry point. See include/dflash.h for the
// contract of every function.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <new>
#include <vector>

#include "internal.h"

namespace dfl {

static std::atomic<long long> g_launches{0};
void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
int cuda_status(cudaError_t e) { return e == cudaSuccess ? DFLASH_OK : DFLASH_E_CUDA; }

namespace {
struct TraceRec {
  const char* name;
  cudaEvent_t a, b;
  double bytes, flops;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<TraceRec> g_trace;
std::vector<cudaEvent_t> g_event_pool;
size_t g_event_next = 0;

cudaEvent_t next_event() {
  if (g_event_next == g_event_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_event_pool.push_back(e);
  }
  return g_event_pool[g_event_next++];
}
}  // namespace

TraceScope::TraceScope(cudaStream_t s, const char* name, double bytes, double flops) : st(s), idx(-1) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (!g_trace_on) return;
  cudaEvent_t a = next_event(), b = next_event();
  if (!a || !b) return;
  if (cudaEventRecord(a, s) != cudaSuccess) return;
  g_trace.push_back(TraceRec{name, a, b, bytes, flops});
  idx = static_cast<int>(g_trace.size()) - 1;
}

TraceScope::~TraceScope() {
  if (idx < 0) return;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (idx < static_cast<int>(g_trace.size())) cudaEventRecord(g_trace[idx].b, st);
}

// Bump allocator over caller-owned memory; with base == nullptr it only sizes.
struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  template <class T>
  T* take(size_t count) {
    off = (off + 255) & ~size_t(255);
    T* r = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return r;
  }
};

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace dfl

using namespace dfl;

struct LayerMaps {
  CUtensorMap q, k, v, o, gate, up, down;
};

struct dflash_handle {
  dflash_config cfg;
  int device = 0;
  int num_sms = 0;
  const __nv_bfloat16* fc = nullptr;
  const __nv_bfloat16* hidden_norm = nullptr;
  const __nv_bfloat16* norm = nullptr;
  const __nv_bfloat16* embed = nullptr;
  const __nv_bfloat16* conv_norm = nullptr;  // two-tap convolution (conv_groups > 0)
  const __nv_bfloat16* conv_proj = nullptr;
  std::vector<dflash_layer_weights> layers;
  CUtensorMap fc_map, embed_map;
  std::vector<LayerMaps> maps;
};

struct dflash_state {
  dflash_handle* h = nullptr;
  int S = 0;
  int R = 0;
  int* lens = nullptr;
  int* status = nullptr;
  float2* rope = nullptr;
  __nv_bfloat16* ring = nullptr;
  std::vector<__nv_bfloat16*> kc, vc;
  std::vector<int> cap, window;
  std::vector<CUtensorMap> kmap, vmap;  // per-layer cache maps of the cluster attention
  std::vector<int64_t> host_len;
};

namespace {

constexpr int kFusePass = 4096;       // rows per fc / inject pass of a fill
constexpr int kDecodeRegimeN = 1024;  // up to this many tokens a GEMM uses the fixed split-K

int head_threads_ok(int d) { return d == 32 || d == 64 || d == 128; }

// Split-K of a GEMM plan (M, K, N and the dual flag set):
//  * up to invariant_n tokens, the split is fixed by the weight's shape
//    (cluster split-K), so a row's result does not depend on the batch it
//    runs in: the drafter's GEMMs keep this up to kInvariantN tokens (four
//    streams' blocks), the fill GEMMs (fc, K/V injection) up to
//    kDecodeRegimeN rows, so a fill resumed after a truncate rebuilds the
//    same cache;
//  * up to kDecodeRegimeN tokens, throughput: 128-token tiles unless the
//    weight alone gives two waves of 256-token tiles (a wide tile's epilogue
//    costs about as much as its MMAs, and two accumulators in tensor memory
//    let a CTA's next tile run under it), no split when the tiles
//    already cover half the SMs, else the smallest split reaching 3/4 of them
//    (global partials, persistent CTAs, at least 8 reduction blocks a chunk);
//  * above, no split.
constexpr int kInvariantN = 64;
constexpr int kInvariantStreams = kInvariantN / DFLASH_BLOCK;  // four streams of a draft call

void set_split(const dflash_handle* h, GemmPlan& p, int invariant_n = kInvariantN) {
  p.no_cluster = false;
  p.bn = 0;
  if (p.N > kDecodeRegimeN) {
    p.ksplit = 1;
    return;
  }
  const int m_tiles = p.M / kTileM, kb = p.K / kTileK;
  if (p.N <= invariant_n) {
    p.ksplit = gemm_choose_ksplit(m_tiles, kb, h->num_sms);
    return;
  }
  // wide weights (the LM head) have tiles for many waves at 256 columns
  if (m_tiles * ((p.N + 255) / 256) < 2 * h->num_sms) p.bn = 128;
  const int BN = plan_bn(p);
  const int tiles = m_tiles * ((p.N + BN - 1) / BN);
  // fewer tiles than half the SMs: the largest split (<= 4, at least eight
  // reduction blocks a chunk) whose CTAs still fit one wave at one CTA an SM.
  // The chunks of a tile form a cluster, so its epilogue (up to 128 columns
  // of heads, residual or SwiGLU work) is shared by the ranks instead of
  // falling to the last chunk to finish (DFlash2 geometry, 128 tokens: the
  // Q/K/V launch 56 -> 29 us, each O and down launch 32 -> 24 us).
  int ks = 1;
  if (2 * tiles < h->num_sms) {
    while (ks < 4 && tiles * (ks + 1) <= h->num_sms && kb / (ks + 1) >= 8) ++ks;
  }
  p.ksplit = ks;
  p.no_cluster = false;
}

int attn_chunk(int cap) { return cap <= 8192 ? 256 : 512; }

int layer_cap(const dflash_config& c, int l, int R) {
  return c.layer_kind[l] == DFLASH_LAYER_SLIDING ? std::min(c.sliding_window, R) : R;
}

}  // namespace

extern "C" {

const char* dflash_strerror(int code) {
  switch (code) {
    case DFLASH_OK: return "ok";
    case DFLASH_E_INVALID_ARG: return "invalid argument";
    case DFLASH_E_TAPS_RANGE: return "tap count or tap layer out of range";
    case DFLASH_E_TAPS_REPEATED: return "a target layer is tapped twice";
    case DFLASH_E_CAUSAL: return "a causal draft is refused";
    case DFLASH_E_SHAPE: return "unsupported shape";
    case DFLASH_E_CAPACITY: return "position past the ring capacity";
    case DFLASH_E_WORKSPACE: return "workspace or state memory too small or misaligned";
    case DFLASH_E_CUDA: return "CUDA error";
    case DFLASH_E_TIMEOUT: return "a device-side wait timed out";
    case DFLASH_E_DEVICE_FAULT: return "the device flagged bad input";
    case DFLASH_E_UNSUPPORTED: return "unsupported device or driver";
    default: return "unknown status";
  }
}

int64_t dflash_launch_count(void) { return g_launches.load(); }

int dflash_trace_enable(int on) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (on) {
    g_trace.clear();
    g_event_next = 0;
  }
  g_trace_on = on != 0;
  return DFLASH_OK;
}

int dflash_trace_count(void) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  return static_cast<int>(g_trace.size());
}

int dflash_trace_get(int i, const char** name, float* ms, double* bytes, double* flops) {
  TraceRec r;
  {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (i < 0 || i >= static_cast<int>(g_trace.size())) return DFLASH_E_INVALID_ARG;
    r = g_trace[i];
  }
  if (cudaEventSynchronize(r.b) != cudaSuccess) return DFLASH_E_CUDA;
  float t = 0.f;
  if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return DFLASH_E_CUDA;
  if (name) *name = r.name;
  if (ms) *ms = t;
  if (bytes) *bytes = r.bytes;
  if (flops) *flops = r.flops;
  return DFLASH_OK;
}

int dflash_config_validate(const dflash_config* c) {
  if (!c) return DFLASH_E_INVALID_ARG;
  if (c->n_taps < 1 || c->n_taps > DFLASH_MAX_TAPS) return DFLASH_E_TAPS_RANGE;
  for (int i = 0; i < c->n_taps; ++i) {
    if (c->tap_layers[i] < 0 || c->tap_layers[i] >= c->target_layers) return DFLASH_E_TAPS_RANGE;
    for (int j = 0; j < i; ++j)
      if (c->tap_layers[j] == c->tap_layers[i]) return DFLASH_E_TAPS_REPEATED;
  }
  if (c->causal != 0) return DFLASH_E_CAUSAL;
  if (c->variant != DFLASH_VARIANT_V1 && c->variant != DFLASH_VARIANT_2) return DFLASH_E_SHAPE;
  if (c->block != DFLASH_BLOCK) return DFLASH_E_SHAPE;
  if (c->n_layers < 1 || c->n_layers > DFLASH_MAX_LAYERS) return DFLASH_E_SHAPE;
  if (c->n_q_heads < 1 || c->n_kv_heads < 1 || c->n_q_heads % c->n_kv_heads) return DFLASH_E_SHAPE;
  if (c->n_q_heads / c->n_kv_heads > 8) return DFLASH_E_SHAPE;
  if (!head_threads_ok(c->head_dim)) return DFLASH_E_SHAPE;
  if (c->hidden != c->n_q_heads * c->head_dim) return DFLASH_E_SHAPE;
  if (c->hidden % 128 || c->ffn < 128 || c->ffn % 128 || (c->n_kv_heads * c->head_dim) % 128) return DFLASH_E_SHAPE;
  if (c->vocab < 128 || c->vocab % 128) return DFLASH_E_SHAPE;
  if (c->mask_token < 0 || c->mask_token >= c->vocab) return DFLASH_E_SHAPE;
  if (!(c->rope_theta > 0.f) || !(c->rms_eps >= 0.f)) return DFLASH_E_SHAPE;
  for (int l = 0; l < c->n_layers; ++l) {
    if (c->layer_kind[l] != DFLASH_LAYER_FULL && c->layer_kind[l] != DFLASH_LAYER_SLIDING) return DFLASH_E_SHAPE;
    if (c->layer_kind[l] == DFLASH_LAYER_SLIDING && c->sliding_window <= 0) return DFLASH_E_SHAPE;
  }
  if (c->conv_groups != 0) {
    // the v1 layout has no conv tensor [TF1851 item 1]
    if (c->variant == DFLASH_VARIANT_V1) return DFLASH_E_SHAPE;
    if (c->conv_groups < 0 || c->conv_groups > kMaxConvGroups || c->hidden % c->conv_groups ||
        (c->hidden / c->conv_groups) % 16)
      return DFLASH_E_SHAPE;
  }
  return DFLASH_OK;
}

const char* dflash_kind(const dflash_config* c) {
  if (!c) return nullptr;
  return c->variant == DFLASH_VARIANT_V1 ? "DFlash" : "DFlash2";
}

int64_t dflash_tap_row_bytes(const dflash_config* c) {
  if (!c) return -1;
  const int64_t H = c->hidden, N = c->n_taps;
  return c->variant == DFLASH_VARIANT_V1 ? (2 * N + 2) * H * 2 : N * H * 2;
}

int64_t dflash_fused_row_bytes(const dflash_config* c) {
  if (!c) return -1;
  return static_cast<int64_t>(c->hidden) * 2;
}

// ---------------------------------------------------------------- handle
int dflash_create(const dflash_config* cfg, const dflash_weights* w, dflash_handle** out) {
  if (!cfg || !w || !out) return DFLASH_E_INVALID_ARG;
  *out = nullptr;
  int rc = dflash_config_validate(cfg);
  if (rc) return rc;
  const void* ptrs[] = {w->fc, w->hidden_norm, w->norm, w->embed};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return DFLASH_E_INVALID_ARG;
  if (!w->layers) return DFLASH_E_INVALID_ARG;
  if (cfg->conv_groups > 0 && (!w->conv_norm || !w->conv_proj || !aligned16(w->conv_norm) || !aligned16(w->conv_proj)))
    return DFLASH_E_INVALID_ARG;
  for (int l = 0; l < cfg->n_layers; ++l) {
    const dflash_layer_weights& L = w->layers[l];
    const void* lp[] = {L.input_norm, L.q_proj, L.k_proj, L.v_proj, L.o_proj, L.q_norm,
                        L.k_norm,     L.post_norm, L.gate_proj, L.up_proj, L.down_proj};
    for (const void* p : lp)
      if (!p || !aligned16(p)) return DFLASH_E_INVALID_ARG;
  }
  int dev = 0, major = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DFLASH_E_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return DFLASH_E_CUDA;
  if (major != 10) return DFLASH_E_UNSUPPORTED;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DFLASH_E_CUDA;

  dflash_handle* h = new (std::nothrow) dflash_handle();
  if (!h) return DFLASH_E_INVALID_ARG;
  h->cfg = *cfg;
  h->device = dev;
  h->num_sms = sms;
  h->fc = static_cast<const __nv_bfloat16*>(w->fc);
  h->hidden_norm = static_cast<const __nv_bfloat16*>(w->hidden_norm);
  h->norm = static_cast<const __nv_bfloat16*>(w->norm);
  h->embed = static_cast<const __nv_bfloat16*>(w->embed);
  if (cfg->conv_groups > 0) {
    h->conv_norm = static_cast<const __nv_bfloat16*>(w->conv_norm);
    h->conv_proj = static_cast<const __nv_bfloat16*>(w->conv_proj);
  }
  h->layers.assign(w->layers, w->layers + cfg->n_layers);
  const int64_t H = cfg->hidden, N = cfg->n_taps, d = cfg->head_dim, F = cfg->ffn, V = cfg->vocab;
  const int64_t qd = cfg->n_q_heads * d, kvd = cfg->n_kv_heads * d;
  rc = encode_kmajor_map(&h->fc_map, w->fc, H, N * H, N * H, kTileM);
  if (!rc) rc = encode_kmajor_map(&h->embed_map, w->embed, V, H, H, kTileM);
  h->maps.resize(cfg->n_layers);
  for (int l = 0; l < cfg->n_layers && !rc; ++l) {
    const dflash_layer_weights& L = w->layers[l];
    LayerMaps& m = h->maps[l];
    rc = encode_kmajor_map(&m.q, L.q_proj, qd, H, H, kTileM);
    if (!rc) rc = encode_kmajor_map(&m.k, L.k_proj, kvd, H, H, kTileM);
    if (!rc) rc = encode_kmajor_map(&m.v, L.v_proj, kvd, H, H, kTileM);
    if (!rc) rc = encode_kmajor_map(&m.o, L.o_proj, H, qd, qd, kTileM);
    if (!rc) rc = encode_kmajor_map(&m.gate, L.gate_proj, F, H, H, kTileM);
    if (!rc) rc = encode_kmajor_map(&m.up, L.up_proj, F, H, H, kTileM);
    if (!rc) rc = encode_kmajor_map(&m.down, L.down_proj, H, F, F, kTileM);
  }
  if (rc) {
    delete h;
    return rc;
  }
  *out = h;
  return DFLASH_OK;
}

int dflash_destroy(dflash_handle* h) {
  delete h;
  return DFLASH_OK;
}

// ---------------------------------------------------------------- state
static size_t state_layout(const dflash_handle* h, int S, int R, void* base, dflash_state* st) {
  const dflash_config& c = h->cfg;
  Carver cv(base);
  int* lens = cv.take<int>(S);
  int* status = cv.take<int>(4);
  float2* rope = cv.take<float2>(static_cast<size_t>(R + DFLASH_BLOCK) * (c.head_dim / 2));
  __nv_bfloat16* ring = cv.take<__nv_bfloat16>(static_cast<size_t>(S) * R * c.hidden);
  if (st) {
    st->lens = lens;
    st->status = status;
    st->rope = rope;
    st->ring = ring;
    st->kc.assign(c.n_layers, nullptr);
    st->vc.assign(c.n_layers, nullptr);
    st->cap.assign(c.n_layers, 0);
    st->window.assign(c.n_layers, 0);
  }
  for (int l = 0; l < c.n_layers; ++l) {
    const int cap = layer_cap(c, l, R);
    const size_t n = static_cast<size_t>(S) * c.n_kv_heads * cap * c.head_dim;
    __nv_bfloat16* k = cv.take<__nv_bfloat16>(n);
    __nv_bfloat16* v = cv.take<__nv_bfloat16>(n);
    if (st) {
      st->kc[l] = k;
      st->vc[l] = v;
      st->cap[l] = cap;
      st->window[l] = c.layer_kind[l] == DFLASH_LAYER_SLIDING ? cap : 0;
    }
  }
  return cv.off;
}

int dflash_state_bytes(const dflash_handle* h, int streams, int ring_capacity, size_t* bytes) {
  if (!h || !bytes || streams < 1 || ring_capacity < 1) return DFLASH_E_INVALID_ARG;
  *bytes = state_layout(h, streams, ring_capacity, nullptr, nullptr);
  return DFLASH_OK;
}

int dflash_state_init(dflash_handle* h, void* dev_mem, size_t bytes, int streams, int ring_capacity,
                      dflash_stream_t stream, dflash_state** out) {
  if (!h || !dev_mem || !out || streams < 1 || ring_capacity < 1) return DFLASH_E_INVALID_ARG;
  *out = nullptr;
  if ((reinterpret_cast<uintptr_t>(dev_mem) & 255u) != 0) return DFLASH_E_WORKSPACE;
  if (state_layout(h, streams, ring_capacity, nullptr, nullptr) > bytes) return DFLASH_E_WORKSPACE;
  dflash_state* st = new (std::nothrow) dflash_state();
  if (!st) return DFLASH_E_INVALID_ARG;
  st->h = h;
  st->S = streams;
  st->R = ring_capacity;
  state_layout(h, streams, ring_capacity, dev_mem, st);
  st->host_len.assign(streams, 0);
  st->kmap.resize(h->cfg.n_layers);
  st->vmap.resize(h->cfg.n_layers);
  if (h->cfg.head_dim == 128) {
    for (int l = 0; l < h->cfg.n_layers; ++l) {
      const int rc = attention_cluster_maps(&st->kmap[l], &st->vmap[l], st->kc[l], st->vc[l],
                                            streams * h->cfg.n_kv_heads, st->cap[l]);
      if (rc) {
        delete st;
        return rc;
      }
    }
  }
  // RoPE table: angle pos * theta^(-2i/d), evaluated in double precision
  const int d = h->cfg.head_dim, half = d / 2;
  const size_t npos = static_cast<size_t>(ring_capacity) + DFLASH_BLOCK;
  std::vector<float2> tab(npos * half);
  std::vector<double> inv(half);
  for (int i = 0; i < half; ++i) inv[i] = pow(static_cast<double>(h->cfg.rope_theta), -2.0 * i / d);
  for (size_t p = 0; p < npos; ++p)
    for (int i = 0; i < half; ++i) {
      const double a = static_cast<double>(p) * inv[i];
      tab[p * half + i] = make_float2(static_cast<float>(cos(a)), static_cast<float>(sin(a)));
    }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(st->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(st->lens, 0, sizeof(int) * streams, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(st->status, 0, sizeof(int) * 4, s);
  // caches start at zero: attention tiles may read (and mask) slots not yet written
  for (int l = 0; l < h->cfg.n_layers && e == cudaSuccess; ++l) {
    const size_t n = static_cast<size_t>(streams) * h->cfg.n_kv_heads * st->cap[l] * h->cfg.head_dim * 2;
    e = cudaMemsetAsync(st->kc[l], 0, n, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(st->vc[l], 0, n, s);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);  // the host table goes out of scope
  if (e != cudaSuccess) {
    delete st;
    return DFLASH_E_CUDA;
  }
  *out = st;
  return DFLASH_OK;
}

int dflash_state_free(dflash_state* st) {
  delete st;
  return DFLASH_OK;
}

int dflash_state_length(const dflash_state* st, int s, int64_t* len) {
  if (!st || !len || s < 0 || s >= st->S) return DFLASH_E_INVALID_ARG;
  *len = st->host_len[s];
  return DFLASH_OK;
}

int dflash_state_ring(const dflash_state* st, void** ring) {
  if (!st || !ring) return DFLASH_E_INVALID_ARG;
  *ring = st->ring;
  return DFLASH_OK;
}

int dflash_state_cache(const dflash_state* st, int layer, void** k, void** v, int* cap) {
  if (!st || !k || !v || !cap || layer < 0 || layer >= static_cast<int>(st->kc.size())) return DFLASH_E_INVALID_ARG;
  *k = st->kc[layer];
  *v = st->vc[layer];
  *cap = st->cap[layer];
  return DFLASH_OK;
}

int dflash_device_status(dflash_state* st, dflash_stream_t stream, int32_t* out) {
  if (!st || !out) return DFLASH_E_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, st->status, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(st->status, 0, sizeof(int), s);
  if (e != cudaSuccess) return DFLASH_E_CUDA;
  *out = v;
  if (v & DFLASH_STATUS_TIMEOUT) return DFLASH_E_TIMEOUT;
  if (v) return DFLASH_E_DEVICE_FAULT;
  return DFLASH_OK;
}

int dflash_state_wait_probe(dflash_state* st, int64_t cycles, dflash_stream_t stream) {
  if (!st || cycles < 0 || cycles > 10000000000ll) return DFLASH_E_INVALID_ARG;
  return launch_wait_probe(st->status, static_cast<long long>(cycles), reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- fusion
namespace {

struct FuseWs {
  int* counters;
  int* row_stream;
  int* row_pos;
  int* row_end;
  float* y;
  float* ss;      // [H/128][rows of the pass]: sums of squares of y, published by the fc GEMM
  float* kv_raw;  // [rows of the pass][2 * layers of a K/V pass * n_kv * d]: raw K/V of wide fills
  __nv_bfloat16* fused;
  float* partial;
  size_t bytes;
};

// GEMM plans of one fill pass of `rows` rows (fc, and K/V injection of the
// layers in [l0, l1)).
GemmPlan fc_plan(const dflash_handle* h, int rows) {
  const dflash_config& c = h->cfg;
  GemmPlan p;
  p.n_aseg = 1;
  p.a_maps[0] = &h->fc_map;
  p.a_rows[0] = c.hidden;
  p.n_b = c.n_taps;
  p.Kp = c.hidden;
  p.M = c.hidden;
  p.N = rows;
  p.K = c.n_taps * c.hidden;
  set_split(h, p, kDecodeRegimeN);
  p.epi = EPI_STORE_F32;
  p.epi_args.ldo = c.hidden;
  p.name = "gemm.fc";
  return p;
}

GemmPlan kv_plan(const dflash_handle* h, const dflash_state* st, int rows, int l0, int l1, bool sliding_only) {
  const dflash_config& c = h->cfg;
  GemmPlan p;
  const int kvd = c.n_kv_heads * c.head_dim;
  int n = 0;
  for (int l = l0; l < l1; ++l) {
    if (sliding_only && c.layer_kind[l] != DFLASH_LAYER_SLIDING) continue;
    for (int kv = 0; kv < 2; ++kv) {
      p.a_maps[n] = kv == 0 ? &h->maps[l].k : &h->maps[l].v;
      p.a_rows[n] = kvd;
      HeadSeg& sg = p.epi_args.seg[n];
      sg.kind = kv == 0 ? HEAD_K : HEAD_V;
      sg.heads = c.n_kv_heads;
      sg.cap = st ? st->cap[l] : 0;
      sg.window = st ? st->window[l] : 0;
      sg.gain = kv == 0 ? static_cast<const __nv_bfloat16*>(h->layers[l].k_norm) : nullptr;
      sg.dst = st ? (kv == 0 ? st->kc[l] : st->vc[l]) : nullptr;
      ++n;
    }
  }
  p.n_aseg = n;
  p.n_b = 1;
  p.Kp = c.hidden;
  p.M = n * kvd;
  p.N = rows;
  p.K = c.hidden;
  set_split(h, p, kDecodeRegimeN);
  p.epi = EPI_HEADS;
  p.epi_args.head_dim = c.head_dim;
  p.epi_args.eps = c.rms_eps;
  p.epi_args.pos_mode = 1;
  p.name = "gemm.kv_inject";
  return p;
}

int layers_per_kv_pass() { return kMaxASeg / 2; }

// A wide fill's fc GEMM whose tiles leave the last wave at most half full
// runs as two launches: the row tiles that fill whole waves, then the rest
// with their reduction split so that they still cover the SMs (4096 rows of
// the 9B shape: 3 waves + a half-filled fourth -> 3 waves + one of half-K
// units: 0.78 -> 0.71 ms). (On the K/V projections, whose last wave holds 16
// of 1536 tiles, the extra launch cost more than it saved.) Returns the
// first row tile of the tail (0: no split) and its split.
int tail_split(const dflash_handle* h, const GemmPlan& p, int& ks_tail) {
  ks_tail = 1;
  if (p.N <= kDecodeRegimeN || p.ksplit != 1) return 0;
  const int m_tiles = p.M / kTileM, BN = plan_bn(p), sms = h->num_sms;
  const int n_tiles = (p.N + BN - 1) / BN;
  const int tiles = m_tiles * n_tiles, full = tiles / sms, rem = tiles - full * sms;
  if (full < 1 || rem == 0 || 2 * rem > sms) return 0;
  const int msplit = full * sms / n_tiles;
  if (msplit <= 0 || msplit >= m_tiles) return 0;
  const int kb = p.K / kTileK;
  int ks = std::min(4, sms / ((m_tiles - msplit) * n_tiles));
  while (ks > 1 && kb / ks < 8) --ks;
  if (ks < 2) return 0;
  ks_tail = ks;
  return msplit;
}

// Launches p (a wide fill's fc GEMM), as two launches when tail_split says so;
// advances the counter cursor past what they used.
int launch_wide(const dflash_handle* h, GemmPlan p, float* partial, int*& counters, int* status, cudaStream_t s) {
  int ks_tail = 1;
  const int msplit = tail_split(h, p, ks_tail);
  GemmPlan tail = p;
  if (msplit > 0) {
    p.M = msplit * kTileM;
    tail.m_tile0 = msplit;
    tail.M -= msplit * kTileM;
    tail.ksplit = ks_tail;
    tail.no_cluster = true;
  }
  int rc = gemm_launch(p, partial, counters, status, h->num_sms, s);
  if (rc) return rc;
  counters += gemm_counter_count(p);
  if (msplit > 0) {
    rc = gemm_launch(tail, partial, counters, status, h->num_sms, s);
    if (rc) return rc;
    counters += gemm_counter_count(tail);
  }
  return DFLASH_OK;
}

size_t fuse_ws_layout(const dflash_handle* h, int rows, void* base, FuseWs* ws) {
  const dflash_config& c = h->cfg;
  const int pass = std::min(std::max(rows, 1), kFusePass);
  size_t counters = gemm_counter_count(fc_plan(h, pass));
  size_t partial = gemm_partial_bytes(fc_plan(h, pass));
  // a split fc tail: at most one wave of units of at most 256 columns
  if (pass > kDecodeRegimeN)
    partial = std::max(partial, static_cast<size_t>(h->num_sms) * 256 * kTileM * sizeof(float));
  for (int l0 = 0; l0 < c.n_layers; l0 += layers_per_kv_pass()) {
    const GemmPlan kp = kv_plan(h, nullptr, pass, l0, std::min(c.n_layers, l0 + layers_per_kv_pass()), false);
    counters += gemm_counter_count(kp);
    partial = std::max(partial, gemm_partial_bytes(kp));
  }
  Carver cv(base);
  FuseWs w{};
  w.counters = cv.take<int>(counters * ((rows + pass - 1) / pass + 1));
  w.row_stream = cv.take<int>(std::max(rows, 1));
  w.row_pos = cv.take<int>(std::max(rows, 1));
  w.row_end = cv.take<int>(std::max(rows, 1));
  w.y = cv.take<float>(static_cast<size_t>(pass) * c.hidden);
  w.ss = cv.take<float>(static_cast<size_t>(pass) * (c.hidden / kTileM));
  w.kv_raw = pass > kDecodeRegimeN
                 ? cv.take<float>(static_cast<size_t>(pass) * 2 * std::min(c.n_layers, layers_per_kv_pass()) *
                                  c.n_kv_heads * c.head_dim)
                 : nullptr;
  w.fused = cv.take<__nv_bfloat16>(static_cast<size_t>(pass) * c.hidden);
  w.partial = cv.take<float>(partial / sizeof(float) + 1);
  w.bytes = cv.off;
  if (ws) *ws = w;
  return cv.off;
}

// K/V injection for `rows` fused rows already in `fused` (rows tables in ws).
// Up to kDecodeRegimeN rows the GEMM's epilogue applies k_norm, RoPE and the
// cache scatter; wider passes (no split-K, many tiles a CTA) write the raw
// projections to kv_raw and an elementwise kernel does that work with the
// whole GPU, with the same arithmetic.
int inject_kv(dflash_handle* h, dflash_state* st, const __nv_bfloat16* fused, const int* row_stream,
              const int* row_pos, const int* row_end, int rows, bool sliding_only, int*& counters, float* partial,
              float* kv_raw, cudaStream_t s) {
  const dflash_config& c = h->cfg;
  for (int l0 = 0; l0 < c.n_layers; l0 += layers_per_kv_pass()) {
    GemmPlan kp = kv_plan(h, st, rows, l0, std::min(c.n_layers, l0 + layers_per_kv_pass()), sliding_only);
    if (kp.n_aseg == 0) continue;
    kp.b_ptr[0] = fused;
    kp.ldb = c.hidden;
    const bool split = kv_raw != nullptr && rows > kDecodeRegimeN;
    KvSegs segs{};
    if (split) {
      segs.n = kp.n_aseg;
      int64_t col = 0;
      segs.head0[0] = 0;
      for (int i = 0; i < kp.n_aseg; ++i) {
        const HeadSeg& sg = kp.epi_args.seg[i];
        segs.col0[i] = col;
        segs.heads[i] = sg.heads;
        segs.cap[i] = sg.cap;
        segs.window[i] = sg.window;
        segs.gain[i] = sg.kind == HEAD_V ? nullptr : sg.gain;
        segs.dst[i] = sg.dst;
        segs.head0[i + 1] = segs.head0[i] + sg.heads;
        col += kp.a_rows[i];
      }
      kp.epi = EPI_STORE_F32;
      kp.epi_args.out = kv_raw;
      kp.epi_args.ldo = kp.M;
      kp.name = "gemm.kv_inject";
    } else {
      kp.epi_args.row_stream = row_stream;
      kp.epi_args.row_pos = row_pos;
      kp.epi_args.row_end = row_end;
      kp.epi_args.rope = st->rope;
    }
    int rc = gemm_launch(kp, partial, counters, st->status, h->num_sms, s);
    if (rc) return rc;
    counters += gemm_counter_count(kp);
    if (split) {
      rc = launch_kv_rows(kv_raw, kp.M, segs, row_stream, row_pos, row_end, st->rope, c.head_dim, c.rms_eps, rows, s);
      if (rc) return rc;
    }
  }
  return DFLASH_OK;
}

}  // namespace

int dflash_fuse_workspace_bytes(const dflash_handle* h, int rows, size_t* bytes) {
  if (!h || !bytes || rows < 0) return DFLASH_E_INVALID_ARG;
  *bytes = fuse_ws_layout(h, rows, nullptr, nullptr);
  return DFLASH_OK;
}

int dflash_fuse_taps(dflash_handle* h, dflash_state* st, const void* const* planes, int64_t plane_row_stride,
                     int nseg, const int32_t* seg_stream, const int64_t* seg_start, const int32_t* seg_rows,
                     int flags, void* ws, size_t ws_bytes, dflash_stream_t stream) {
  if (!h || !st || !planes || !seg_stream || !seg_start || !seg_rows || !ws) return DFLASH_E_INVALID_ARG;
  if (st->h != h || nseg < 1 || nseg > 256 || (flags & ~DFLASH_FUSE_INJECT_KV)) return DFLASH_E_INVALID_ARG;
  const dflash_config& c = h->cfg;
  if (plane_row_stride < c.hidden || (plane_row_stride * 2) % 16) return DFLASH_E_SHAPE;
  for (int i = 0; i < c.n_taps; ++i)
    if (!planes[i] || !aligned16(planes[i])) return DFLASH_E_INVALID_ARG;
  int rows = 0;
  std::vector<int> seen(st->S, 0);
  std::vector<int> packed(3 * nseg);
  for (int i = 0; i < nseg; ++i) {
    const int s = seg_stream[i];
    if (s < 0 || s >= st->S || seen[s] || seg_rows[i] < 1) return DFLASH_E_INVALID_ARG;
    seen[s] = 1;
    if (seg_start[i] != st->host_len[s]) return DFLASH_E_INVALID_ARG;  // append only
    if (seg_start[i] + seg_rows[i] > st->R) return DFLASH_E_CAPACITY;
    packed[3 * i] = s;
    packed[3 * i + 1] = static_cast<int>(seg_start[i]);
    packed[3 * i + 2] = seg_rows[i];
    rows += seg_rows[i];
  }
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return DFLASH_E_WORKSPACE;
  FuseWs w{};
  if (fuse_ws_layout(h, rows, ws, &w) > ws_bytes) return DFLASH_E_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool inject = (flags & DFLASH_FUSE_INJECT_KV) != 0;

  // one launch: the row tables, every split-K counter of this call cleared,
  // and (with K/V injection) the new stream lengths, which no kernel of this
  // call reads (the K/V epilogue places rows by their table positions)
  const size_t counters_bytes = reinterpret_cast<char*>(w.row_stream) - reinterpret_cast<char*>(w.counters);
  int rc = launch_prep_rows(w.row_stream, w.row_pos, w.row_end, inject ? st->lens : nullptr, nseg, rows,
                            packed.data(), w.counters, static_cast<int>(counters_bytes / sizeof(int)), s);
  if (rc) return rc;
  int* counters = w.counters;
  for (int r0 = 0; r0 < rows; r0 += kFusePass) {
    const int n = std::min(kFusePass, rows - r0);
    GemmPlan fp = fc_plan(h, n);
    for (int i = 0; i < c.n_taps; ++i)
      fp.b_ptr[i] = static_cast<const __nv_bfloat16*>(planes[i]) + static_cast<int64_t>(r0) * plane_row_stride;
    fp.ldb = plane_row_stride;
    fp.epi_args.out = w.y;
    fp.epi_args.ss_out = w.ss;
    fp.epi_args.ss_ld = n;
    rc = launch_wide(h, fp, w.partial, counters, st->status, s);
    if (rc) return rc;
    rc = launch_hidden_norm(st->ring, w.fused, w.y, w.ss, h->hidden_norm, w.row_stream + r0, w.row_pos + r0, n,
                            c.hidden, st->R, c.rms_eps, s);
    if (rc) return rc;
    if (inject) {
      rc = inject_kv(h, st, w.fused, w.row_stream + r0, w.row_pos + r0, w.row_end + r0, n, false, counters,
                     w.partial, w.kv_raw, s);
      if (rc) return rc;
    }
  }
  if (inject)
    for (int i = 0; i < nseg; ++i) st->host_len[seg_stream[i]] = seg_start[i] + seg_rows[i];
  return DFLASH_OK;
}

int dflash_state_truncate(dflash_handle* h, dflash_state* st, int s_id, int64_t new_len, void* ws, size_t ws_bytes,
                          dflash_stream_t stream) {
  if (!h || !st || st->h != h || s_id < 0 || s_id >= st->S) return DFLASH_E_INVALID_ARG;
  const int64_t old_len = st->host_len[s_id];
  if (new_len < 0 || new_len > old_len) return DFLASH_E_INVALID_ARG;
  const dflash_config& c = h->cfg;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // sliding caches: positions [new_len - W, old_len - W) were overwritten by
  // the dropped rows (same ring slots) and are rebuilt from the fused ring
  bool any_sliding = false;
  for (int l = 0; l < c.n_layers; ++l) any_sliding |= c.layer_kind[l] == DFLASH_LAYER_SLIDING;
  const int64_t W = std::min<int64_t>(c.sliding_window, st->R);
  const int64_t lo = std::max<int64_t>(0, new_len - W);
  const int64_t hi = std::min<int64_t>(new_len, old_len - W);
  int packed[3] = {s_id, static_cast<int>(new_len), 0};
  if (any_sliding && hi > lo) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return DFLASH_E_WORKSPACE;
    const int n = static_cast<int>(hi - lo);
    FuseWs w{};
    if (fuse_ws_layout(h, n, ws, &w) > ws_bytes) return DFLASH_E_WORKSPACE;
    const size_t counters_bytes = reinterpret_cast<char*>(w.row_stream) - reinterpret_cast<char*>(w.counters);
    int seg[3] = {s_id, static_cast<int>(lo), n};
    int rc = launch_prep_rows(w.row_stream, w.row_pos, w.row_end, nullptr, 1, n, seg, w.counters,
                              static_cast<int>(counters_bytes / sizeof(int)), s);
    if (rc) return rc;
    int* counters = w.counters;
    for (int r0 = 0; r0 < n; r0 += kFusePass) {
      const int m = std::min(kFusePass, n - r0);
      const __nv_bfloat16* rows = st->ring + (static_cast<int64_t>(s_id) * st->R + lo + r0) * c.hidden;
      rc = inject_kv(h, st, rows, w.row_stream + r0, w.row_pos + r0, w.row_end + r0, m, true, counters,
                     w.partial, w.kv_raw, s);
      if (rc) return rc;
    }
  }
  const int rc = launch_prep_rows(nullptr, nullptr, nullptr, st->lens, 1, 0, packed, nullptr, 0, s);
  if (rc) return rc;
  st->host_len[s_id] = new_len;
  return DFLASH_OK;
}

// ---------------------------------------------------------------- drafting
namespace {

struct DraftWs {
  int* counters;
  size_t n_counters;
  float* X;
  __nv_bfloat16* hbuf;  // bf16 normalised rows, the B operand after each RMSNorm
  float* ss;            // [H/128][T] per-part sums of squares of the residual rows (every writer of X publishes them)
  __nv_bfloat16* Q;
  __nv_bfloat16* Kb;
  __nv_bfloat16* Vb;
  __nv_bfloat16* attn;
  __nv_bfloat16* mid;
  float* part_o;
  float* part_ml;
  float* partial;
  __nv_bfloat16* logits;
  float* cand_v;  // LM-head per-tile top-k candidates, [rows][V/128][8]
  int* cand_i;
  float* conv_z;  // two-tap convolution logits [T][2 * groups]
};

int max_nchunk(const dflash_state* st) {
  int m = 1;
  for (size_t l = 0; l < st->cap.size(); ++l) m = std::max(m, (st->cap[l] + attn_chunk(st->cap[l]) - 1) / attn_chunk(st->cap[l]));
  return m;
}

void layer_plans(const dflash_handle* h, int l, int T, GemmPlan& qkv, GemmPlan& o, GemmPlan& gu, GemmPlan& dn) {
  const dflash_config& c = h->cfg;
  const int qd = c.n_q_heads * c.head_dim, kvd = c.n_kv_heads * c.head_dim;
  const LayerMaps& m = h->maps[l];
  qkv = GemmPlan();
  qkv.n_aseg = 3;
  qkv.a_maps[0] = &m.q;
  qkv.a_maps[1] = &m.k;
  qkv.a_maps[2] = &m.v;
  qkv.a_rows[0] = qd;
  qkv.a_rows[1] = kvd;
  qkv.a_rows[2] = kvd;
  qkv.n_b = 1;
  qkv.Kp = c.hidden;
  qkv.M = qd + 2 * kvd;
  qkv.N = T;
  qkv.K = c.hidden;
  set_split(h, qkv);
  qkv.epi = EPI_HEADS;
  qkv.name = "gemm.qkv";
  o = GemmPlan();
  o.n_aseg = 1;
  o.a_maps[0] = &m.o;
  o.a_rows[0] = c.hidden;
  o.n_b = 1;
  o.Kp = qd;
  o.M = c.hidden;
  o.N = T;
  o.K = qd;
  set_split(h, o);
  o.epi = EPI_RESID;
  o.name = "gemm.o";
  gu = GemmPlan();
  gu.n_aseg = 1;
  gu.a_maps[0] = &m.gate;
  gu.a_rows[0] = c.ffn;
  gu.a2_map = &m.up;
  gu.n_b = 1;
  gu.Kp = c.hidden;
  gu.M = c.ffn;
  gu.N = T;
  gu.K = c.hidden;
  set_split(h, gu);
  gu.epi = EPI_SWIGLU;
  gu.name = "gemm.gate_up";
  dn = GemmPlan();
  dn.n_aseg = 1;
  dn.a_maps[0] = &m.down;
  dn.a_rows[0] = c.hidden;
  dn.n_b = 1;
  dn.Kp = c.ffn;
  dn.M = c.hidden;
  dn.N = T;
  dn.K = c.ffn;
  set_split(h, dn);
  dn.epi = EPI_RESID;
  dn.name = "gemm.down";
}

GemmPlan lm_plan(const dflash_handle* h, int rows) {
  const dflash_config& c = h->cfg;
  GemmPlan p;
  p.n_aseg = 1;
  p.a_maps[0] = &h->embed_map;
  p.a_rows[0] = c.vocab;
  p.n_b = 1;
  p.Kp = c.hidden;
  p.M = c.vocab;
  p.N = rows;
  p.K = c.hidden;
  set_split(h, p);
  p.epi = EPI_STORE_BF16;
  p.epi_args.ldo = c.vocab;
  p.name = "gemm.lm_head";
  return p;
}

size_t draft_ws_layout(const dflash_handle* h, const dflash_state* st, int S, bool need_logits, void* base,
                       DraftWs* out) {
  const dflash_config& c = h->cfg;
  const int T = S * DFLASH_BLOCK;
  const int qd = c.n_q_heads * c.head_dim, kvd = c.n_kv_heads * c.head_dim;
  size_t counters = 0, partial = 0;
  for (int l = 0; l < c.n_layers; ++l) {
    GemmPlan a, b, g, d;
    layer_plans(h, l, T, a, b, g, d);
    for (const GemmPlan* p : {&a, &b, &g, &d}) {
      counters += gemm_counter_count(*p);
      partial = std::max(partial, gemm_partial_bytes(*p));
    }
  }
  const GemmPlan lp = lm_plan(h, S * (DFLASH_BLOCK - 1));
  counters += gemm_counter_count(lp);
  partial = std::max(partial, gemm_partial_bytes(lp));
  const int nch = max_nchunk(st);
  Carver cv(base);
  DraftWs w{};
  w.counters = cv.take<int>(counters);
  w.n_counters = counters;
  w.X = cv.take<float>(static_cast<size_t>(T) * c.hidden);
  w.hbuf = cv.take<__nv_bfloat16>(static_cast<size_t>(T) * c.hidden);
  w.ss = cv.take<float>(static_cast<size_t>(T) * (c.hidden / kTileM));
  w.Q = cv.take<__nv_bfloat16>(static_cast<size_t>(T) * qd);
  w.Kb = cv.take<__nv_bfloat16>(static_cast<size_t>(T) * kvd);
  w.Vb = cv.take<__nv_bfloat16>(static_cast<size_t>(T) * kvd);
  w.attn = cv.take<__nv_bfloat16>(static_cast<size_t>(T) * qd);
  w.mid = cv.take<__nv_bfloat16>(static_cast<size_t>(T) * c.ffn);
  w.part_o = cv.take<float>(static_cast<size_t>(S) * c.n_q_heads * nch * 16 * c.head_dim);
  w.part_ml = cv.take<float>(static_cast<size_t>(S) * c.n_q_heads * nch * 16 * 2);
  w.partial = cv.take<float>(partial / sizeof(float) + 1);
  w.logits = need_logits ? cv.take<__nv_bfloat16>(static_cast<size_t>(S) * (DFLASH_BLOCK - 1) * c.vocab) : nullptr;
  const size_t ncand = static_cast<size_t>(S) * (DFLASH_BLOCK - 1) * (c.vocab / kTileM) * 8;
  w.cand_v = cv.take<float>(ncand);
  w.cand_i = cv.take<int>(ncand);
  w.conv_z = cv.take<float>(static_cast<size_t>(T) * 2 * std::max(c.conv_groups, 1));
  if (out) *out = w;
  return cv.off;
}

}  // namespace

int dflash_draft_workspace_bytes(const dflash_handle* h, const dflash_state* st, int s_count, int need_logits,
                                 size_t* bytes) {
  if (!h || !st || !bytes || s_count < 1) return DFLASH_E_INVALID_ARG;
  *bytes = draft_ws_layout(h, st, s_count, need_logits != 0, nullptr, nullptr);
  return DFLASH_OK;
}

namespace {

// The RMSNorm gain of stage g's input norm (input_norm of layer g/2 for an
// attention half, post_norm for an MLP half).
const __nv_bfloat16* stage_gain(const dflash_handle* h, int g) {
  const dflash_layer_weights& L = h->layers[g >> 1];
  return static_cast<const __nv_bfloat16*>((g & 1) ? L.post_norm : L.input_norm);
}

// Stage g's input RMSNorm of X into w.hbuf (rstd from the sums in w.ss),
// which the stage's first GEMM `p` reads.
int stage_norm(dflash_handle* h, int g, GemmPlan& p, const float* X, const DraftWs& w, int T, cudaStream_t s) {
  const dflash_config& c = h->cfg;
  p.n_b = 1;
  p.ldb = c.hidden;
  p.b_ptr[0] = w.hbuf;
  return launch_rmsnorm_rows(w.hbuf, X, stage_gain(h, g), w.ss, T, T, c.hidden, c.rms_eps, 0, s);
}

// A residual add that also leaves the new rows' sums of squares in w.ss.
void resid_add(EpiArgs& e, float* X, const dflash_config& c, const DraftWs& w, int T) {
  e.out = X;
  e.ldo = c.hidden;
  e.ss_out = w.ss;
  e.ss_ld = T;
}

// Stages [g0, g1) of the block forward on the fp32 residual X [16*s_count, H]
// whose per-part sums of squares are in w.ss: stage 2l is layer l's
// attention half (input norm, QKV, attention, O-proj added to X), stage 2l+1
// its MLP half (post norm, SwiGLU, down added to X). Each residual add
// leaves the sums of squares of the new rows for the next stage's norm;
// first_ready: stage g0's normalised rows are in w.hbuf already.
int run_stages(dflash_handle* h, dflash_state* st, int s_begin, int s_count, int g0, int g1, float* X,
               const DraftWs& w, int*& counters, cudaStream_t s, bool first_ready = false) {
  bool ready = first_ready;
  const dflash_config& c = h->cfg;
  const int T = s_count * DFLASH_BLOCK;
  const int qd = c.n_q_heads * c.head_dim, kvd = c.n_kv_heads * c.head_dim;
  const int nch = max_nchunk(st);
  int rc = DFLASH_OK;
  for (int g = g0; g < g1; ++g) {
    const int l = g >> 1;
    const dflash_layer_weights& L = h->layers[l];
    GemmPlan qkv, o, gu, dn;
    layer_plans(h, l, T, qkv, o, gu, dn);
    if (g & 1) {
      // post-attention RMSNorm -> SwiGLU -> down projection added to the residual
      if (ready) {
        gu.n_b = 1;
        gu.ldb = c.hidden;
        gu.b_ptr[0] = w.hbuf;
      } else {
        rc = stage_norm(h, g, gu, X, w, T, s);
        if (rc) return rc;
      }
      gu.epi_args.out = w.mid;
      gu.epi_args.ldo = c.ffn;
      rc = gemm_launch(gu, w.partial, counters, st->status, h->num_sms, s);
      if (rc) return rc;
      counters += gemm_counter_count(gu);
      dn.b_ptr[0] = w.mid;
      dn.ldb = c.ffn;
      resid_add(dn.epi_args, X, c, w, T);
      ready = false;
      rc = gemm_launch(dn, w.partial, counters, st->status, h->num_sms, s);
      if (rc) return rc;
      counters += gemm_counter_count(dn);
      continue;
    }
    // input RMSNorm -> QKV with q_norm / k_norm + RoPE at positions C..C+15
    if (ready) {
      qkv.n_b = 1;
      qkv.ldb = c.hidden;
      qkv.b_ptr[0] = w.hbuf;
    } else {
      rc = stage_norm(h, g, qkv, X, w, T, s);
      if (rc) return rc;
    }
    EpiArgs& e = qkv.epi_args;
    e.head_dim = c.head_dim;
    e.eps = c.rms_eps;
    e.pos_mode = 0;
    e.s_begin = s_begin;
    e.lens = st->lens;
    e.rope = st->rope;
    e.seg[0] = HeadSeg{HEAD_Q, c.n_q_heads, 0, 0, static_cast<const __nv_bfloat16*>(L.q_norm), w.Q};
    e.seg[1] = HeadSeg{HEAD_K, c.n_kv_heads, 0, 0, static_cast<const __nv_bfloat16*>(L.k_norm), w.Kb};
    e.seg[2] = HeadSeg{HEAD_V, c.n_kv_heads, 0, 0, nullptr, w.Vb};
    rc = gemm_launch(qkv, w.partial, counters, st->status, h->num_sms, s);
    if (rc) return rc;
    counters += gemm_counter_count(qkv);
    // attention over the layer's window of context + the block
    AttnArgs a{};
    a.Q = w.Q;
    a.Kb = w.Kb;
    a.Vb = w.Vb;
    a.Kc = st->kc[l];
    a.Vc = st->vc[l];
    a.lens = st->lens;
    a.s_begin = s_begin;
    a.cap = st->cap[l];
    a.window = st->window[l];
    a.nq = c.n_q_heads;
    a.nkv = c.n_kv_heads;
    a.d = c.head_dim;
    a.chunk = attn_chunk(st->cap[l]);
    a.nchunk = nch;
    a.part_o = w.part_o;
    a.part_ml = w.part_ml;
    a.out = w.attn;
    {
      double keys = 0.0;
      for (int i = 0; i < s_count; ++i) {
        const int64_t C = st->host_len[s_begin + i];
        keys += static_cast<double>(st->window[l] > 0 ? std::min<int64_t>(C, st->window[l]) : C) + DFLASH_BLOCK;
      }
      a.trace_bytes = keys * kvd * 2.0 * 2.0 + 2.0 * T * qd * 2.0;
    }
    a.err = st->status;
    // more than four streams whose (stream, kv head) pairs fit one wave of
    // SMs: the tensor-memory kernel, one 128-row MMA per kv head's query
    // group (the DFlash2 geometry, 8 streams x 8 kv heads: 0.74 ms a draft
    // with the cluster kernel, 0.29 ms). Up to four streams the
    // batch-invariant 8-way split of the cluster kernel stays; with more
    // pairs than SMs the cluster kernel's finer key split balanced uneven
    // contexts better when the tensor-memory kernel still took 64-key tiles
    // (32 streams of the 9B shape: 0.77 ms against 0.79-0.85 ms a round).
    if (s_count > kInvariantStreams && s_count * a.nkv <= h->num_sms && attention_tc_supported(a))
      rc = launch_attention_tc(a, st->kmap[l], st->vmap[l], s_count, h->num_sms, s);
    else
      rc = attention_cluster_supported(a) ? launch_attention_cluster(a, st->kmap[l], st->vmap[l], s_count, s)
                                          : launch_attention(a, s_count, s);
    if (rc) return rc;
    // O projection added to the residual
    o.b_ptr[0] = w.attn;
    o.ldb = qd;
    resid_add(o.epi_args, X, c, w, T);
    ready = false;
    rc = gemm_launch(o, w.partial, counters, st->status, h->num_sms, s);
    if (rc) return rc;
    counters += gemm_counter_count(o);
  }
  return DFLASH_OK;
}

// DFlash2's two-tap dynamic convolution on the residual X (sums of squares
// in w.ss), leaving the new rows' sums of squares in w.ss for the final norm.
int run_conv(dflash_handle* h, int s_count, float* X, const DraftWs& w, cudaStream_t s) {
  const dflash_config& c = h->cfg;
  const int T = s_count * DFLASH_BLOCK;
  int rc = launch_rmsnorm_rows(w.hbuf, X, h->conv_norm, w.ss, T, T, c.hidden, c.rms_eps, 0, s);
  if (!rc) rc = launch_block_conv(X, w.hbuf, w.conv_z, h->conv_proj, s_count, c.hidden, c.conv_groups, s);
  if (!rc) rc = launch_row_sumsq(w.ss, X, T, c.hidden, s);
  return rc;
}

// Final norm on the 15 mask rows of every stream (sums of squares of X in
// w.ss), shared LM head, top-k.
int run_head(dflash_handle* h, int* status, int s_count, const float* X, const DraftWs& w, __nv_bfloat16* logits,
             int32_t* topk_ids, float* topk_vals, int k, int*& counters, cudaStream_t s) {
  const dflash_config& c = h->cfg;
  const int rows = s_count * (DFLASH_BLOCK - 1);
  int rc = launch_rmsnorm_rows(w.hbuf, X, h->norm, w.ss, s_count * DFLASH_BLOCK, rows, c.hidden, c.rms_eps, 1, s);
  if (rc) return rc;
  GemmPlan lp = lm_plan(h, rows);
  lp.b_ptr[0] = w.hbuf;
  lp.ldb = c.hidden;
  lp.epi_args.out = logits;
  // top-k up to 8 of a single stream's 15 rows: the LM head's epilogue ranks
  // each 128-id tile (hidden under its weight stream), a small kernel merges
  // the tiles' lists. Wider heads are compute-bound and their epilogues would
  // rank 16 column chunks a tile: there a vocabulary scan after the GEMM is
  // cheaper.
  const bool fused_topk = topk_ids != nullptr && k <= 8 && plan_bn(lp) == 16;
  if (fused_topk) {
    lp.epi_args.cand_k = k;
    lp.epi_args.cand_v = w.cand_v;
    lp.epi_args.cand_i = w.cand_i;
  }
  rc = gemm_launch(lp, w.partial, counters, status, h->num_sms, s);
  if (rc) return rc;
  counters += gemm_counter_count(lp);
  if (fused_topk)
    rc = launch_topk_merge(w.cand_v, w.cand_i, rows, c.vocab / kTileM, k, topk_ids, topk_vals, s);
  else if (topk_ids)
    rc = launch_topk(logits, rows, c.vocab, k, 1.0f, nullptr, topk_ids, topk_vals, nullptr, s);
  return rc;
}

int check_draft_args(dflash_handle* h, dflash_state* st, int s_begin, int s_count, const void* ws, int32_t* topk_ids,
                     float* topk_vals, int k, const void* logits_out) {
  if (!h || !st || st->h != h || !ws) return DFLASH_E_INVALID_ARG;
  if (s_count < 1 || s_begin < 0 || s_begin + s_count > st->S) return DFLASH_E_INVALID_ARG;
  const bool do_topk = topk_ids != nullptr || topk_vals != nullptr;
  if (do_topk && (!topk_ids || !topk_vals || k < 1 || k > DFLASH_MAX_TOPK)) return DFLASH_E_INVALID_ARG;
  if (logits_out && !aligned16(logits_out)) return DFLASH_E_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return DFLASH_E_WORKSPACE;
  return DFLASH_OK;
}

}  // namespace

int dflash_draft_block(dflash_handle* h, dflash_state* st, int s_begin, int s_count, const int32_t* anchor_ids,
                       void* logits_out, int32_t* topk_ids, float* topk_vals, int k, void* ws, size_t ws_bytes,
                       dflash_stream_t stream) {
  int rc = check_draft_args(h, st, s_begin, s_count, ws, topk_ids, topk_vals, k, logits_out);
  if (rc) return rc;
  if (!anchor_ids) return DFLASH_E_INVALID_ARG;
  const dflash_config& c = h->cfg;
  DraftWs w{};
  if (draft_ws_layout(h, st, s_count, logits_out == nullptr, ws, &w) > ws_bytes) return DFLASH_E_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  __nv_bfloat16* logits = logits_out ? static_cast<__nv_bfloat16*>(logits_out) : w.logits;
  // the embedding launch also writes the first layer's input norm
  rc = launch_embed(w.X, w.ss, h->embed, anchor_ids, s_count, c.hidden, c.vocab, c.mask_token, st->status, w.counters,
                    static_cast<int>(w.n_counters), w.hbuf, stage_gain(h, 0), c.rms_eps, s);
  if (rc) return rc;
  int* counters = w.counters;
  rc = run_stages(h, st, s_begin, s_count, 0, 2 * c.n_layers, w.X, w, counters, s, true);
  if (rc) return rc;
  if (c.conv_groups > 0) {
    rc = run_conv(h, s_count, w.X, w, s);
    if (rc) return rc;
  }
  return run_head(h, st->status, s_count, w.X, w, logits, topk_ids, topk_vals, k, counters, s);
}

int dflash_draft_conv(dflash_handle* h, dflash_state* st, int s_count, float* X, void* ws, size_t ws_bytes,
                      dflash_stream_t stream) {
  int rc = check_draft_args(h, st, 0, s_count, ws, nullptr, nullptr, 0, nullptr);
  if (rc) return rc;
  if (!X || !aligned16(X) || h->cfg.conv_groups <= 0) return DFLASH_E_INVALID_ARG;
  DraftWs w{};
  if (draft_ws_layout(h, st, s_count, false, ws, &w) > ws_bytes) return DFLASH_E_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rc = launch_row_sumsq(w.ss, X, s_count * DFLASH_BLOCK, h->cfg.hidden, s);
  if (rc) return rc;
  return run_conv(h, s_count, X, w, s);
}

int dflash_draft_stages(dflash_handle* h, dflash_state* st, int s_begin, int s_count, int stage0, int stage1,
                        float* X, void* ws, size_t ws_bytes, dflash_stream_t stream) {
  int rc = check_draft_args(h, st, s_begin, s_count, ws, nullptr, nullptr, 0, nullptr);
  if (rc) return rc;
  if (!X || !aligned16(X) || stage0 < 0 || stage1 < stage0 || stage1 > 2 * h->cfg.n_layers)
    return DFLASH_E_INVALID_ARG;
  DraftWs w{};
  if (draft_ws_layout(h, st, s_count, false, ws, &w) > ws_bytes) return DFLASH_E_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(w.counters, 0, w.n_counters * sizeof(int), s) != cudaSuccess) return DFLASH_E_CUDA;
  int* counters = w.counters;
  if (stage1 == stage0) return DFLASH_OK;
  rc = launch_row_sumsq(w.ss, X, s_count * DFLASH_BLOCK, h->cfg.hidden, s);
  if (rc) return rc;
  return run_stages(h, st, s_begin, s_count, stage0, stage1, X, w, counters, s);
}

int dflash_draft_head(dflash_handle* h, dflash_state* st, int s_count, const float* X, void* logits_out,
                      int32_t* topk_ids, float* topk_vals, int k, void* ws, size_t ws_bytes, dflash_stream_t stream) {
  int rc = check_draft_args(h, st, 0, s_count, ws, topk_ids, topk_vals, k, logits_out);
  if (rc) return rc;
  if (!X || !aligned16(X) || !logits_out) return DFLASH_E_INVALID_ARG;
  DraftWs w{};
  if (draft_ws_layout(h, st, s_count, false, ws, &w) > ws_bytes) return DFLASH_E_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(w.counters, 0, w.n_counters * sizeof(int), s) != cudaSuccess) return DFLASH_E_CUDA;
  int* counters = w.counters;
  rc = launch_row_sumsq(w.ss, X, s_count * DFLASH_BLOCK, h->cfg.hidden, s);
  if (rc) return rc;
  return run_head(h, st->status, s_count, X, w, static_cast<__nv_bfloat16*>(logits_out), topk_ids, topk_vals, k,
                  counters, s);
}

// ---------------------------------------------------------------- top-k / verify
int dflash_topk(const void* logits, int rows, int vocab, int k, float temperature, const float* uniforms,
                int32_t* ids, float* vals, int32_t* sampled, dflash_stream_t stream) {
  if (rows == 0 && vocab >= 8 && vocab % 8 == 0 && k >= 0 && k <= DFLASH_MAX_TOPK) return DFLASH_OK;
  if (!logits || rows < 0 || vocab < 8 || vocab % 8 || k < 0 || k > DFLASH_MAX_TOPK) return DFLASH_E_INVALID_ARG;
  if (k > 0 && (!ids || !vals)) return DFLASH_E_INVALID_ARG;
  if ((uniforms == nullptr) != (sampled == nullptr)) return DFLASH_E_INVALID_ARG;
  if (uniforms && !(temperature > 0.f)) return DFLASH_E_INVALID_ARG;
  if (!aligned16(logits)) return DFLASH_E_INVALID_ARG;
  if (k == 0 && !uniforms) return DFLASH_OK;
  return launch_topk(static_cast<const __nv_bfloat16*>(logits), rows, vocab, k, uniforms ? temperature : 1.0f,
                     uniforms, ids, vals, sampled, reinterpret_cast<cudaStream_t>(stream));
}

int dflash_draft_stop(const void* logits, int streams, int vocab, float temperature, float min_p, float* conf,
                      int32_t* draft_len, dflash_stream_t stream) {
  if (streams < 0 || vocab < 8 || vocab % 8) return DFLASH_E_INVALID_ARG;
  if (streams == 0) return DFLASH_OK;
  if (!logits || !conf || !draft_len || !aligned16(logits)) return DFLASH_E_INVALID_ARG;
  if (!(temperature > 0.f) || !(min_p >= 0.f && min_p <= 1.f)) return DFLASH_E_INVALID_ARG;
  return launch_draft_stop(static_cast<const __nv_bfloat16*>(logits), streams, vocab, temperature, min_p, conf,
                           draft_len, reinterpret_cast<cudaStream_t>(stream));
}

int dflash_verify_workspace_bytes(int mode, int streams, int vocab, size_t* bytes) {
  if (!bytes || streams < 0 || vocab < 8) return DFLASH_E_INVALID_ARG;
  if (mode == DFLASH_VERIFY_GREEDY) *bytes = 0;
  else if (mode == DFLASH_VERIFY_SAMPLE) *bytes = static_cast<size_t>(streams) * 31 * 2 * sizeof(float);
  else return DFLASH_E_INVALID_ARG;
  return DFLASH_OK;
}

int dflash_verify(int mode, int streams, int vocab, const int32_t* draft_ids, int draft_ld, const void* target_logits,
                  const void* draft_logits, const float* uniforms, float temperature, int32_t* accept_len,
                  int32_t* out_tokens, void* ws, size_t ws_bytes, dflash_stream_t stream) {
  if (streams < 0 || vocab < 8 || vocab % 8 || !draft_ids || draft_ld < 1 || !target_logits || !accept_len ||
      !out_tokens)
    return DFLASH_E_INVALID_ARG;
  if (!aligned16(target_logits)) return DFLASH_E_INVALID_ARG;
  if (streams == 0) return DFLASH_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (mode == DFLASH_VERIFY_GREEDY) {
    return launch_verify_greedy(streams, vocab, draft_ids, draft_ld, static_cast<const __nv_bfloat16*>(target_logits),
                                accept_len, out_tokens, s);
  }
  if (mode != DFLASH_VERIFY_SAMPLE) return DFLASH_E_INVALID_ARG;
  if (!draft_logits || !uniforms || !(temperature > 0.f) || !aligned16(draft_logits)) return DFLASH_E_INVALID_ARG;
  if (streams > DFLASH_MAX_SAMPLE_STREAMS) return DFLASH_E_INVALID_ARG;
  size_t need = 0;
  dflash_verify_workspace_bytes(mode, streams, vocab, &need);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 15u)) return DFLASH_E_WORKSPACE;
  return launch_verify_sample(streams, vocab, draft_ids, draft_ld, static_cast<const __nv_bfloat16*>(target_logits),
                              static_cast<const __nv_bfloat16*>(draft_logits), uniforms, temperature, accept_len,
                              out_tokens, static_cast<float*>(ws), s);
}

}  // extern "C"

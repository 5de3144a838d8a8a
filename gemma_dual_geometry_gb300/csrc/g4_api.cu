// C-ABI front end of libg4attn: argument validation, shared-KV source
// resolution, the float32 RoPE frequency table, and kernel dispatch.
// Declarations and the contract of every entry point: include/g4attn.h.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <string>

#include "../../include/g4attn.h"
#include "g4_internal.h"

namespace {

thread_local std::string g_last_error;

g4_status fail(g4_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
g4_status fail(g4_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

g4_status ok() {
  g_last_error.clear();
  return G4_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_hd(int hd) { return hd == 64 || hd == 128 || hd == 256 || hd == 512; }

// Device error word: a kernel that gives up a bounded wait records a code here.
__device__ int g_device_error = 0;

// Its device address, looked up once per device (with that device current)
// under a lock, so host threads driving different GPUs each get their own.
int* device_error_ptr() {
  static std::mutex mu;
  static int* addr[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<int*>(p);
  }
  return addr[dev];
}

g4_status check_params(const g4_layer_params* p) {
  if (p == nullptr) return fail(G4_ERR_INVALID_ARG, "params is NULL");
  if (p->layer_type != G4_SLIDING && p->layer_type != G4_FULL)
    return fail(G4_ERR_INVALID_ARG, "layer_type %d is neither G4_SLIDING nor G4_FULL", p->layer_type);
  if (p->dtype != G4_F32 && p->dtype != G4_BF16) return fail(G4_ERR_INVALID_ARG, "dtype %d unknown", p->dtype);
  if (!supported_hd(p->head_dim))
    return fail(G4_ERR_UNSUPPORTED, "head_dim %d not supported (64, 128, 256, 512)", p->head_dim);
  if (p->n_heads < 1 || p->n_kv_heads < 1 || p->n_heads % p->n_kv_heads != 0)
    return fail(G4_ERR_INVALID_ARG, "n_heads %d must be a positive multiple of n_kv_heads %d", p->n_heads,
                p->n_kv_heads);
  const int g = p->n_heads / p->n_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8)
    return fail(G4_ERR_UNSUPPORTED, "GQA group %d not supported (1, 2, 4, 8)", g);
  if (g * p->head_dim > 2048)
    return fail(G4_ERR_UNSUPPORTED, "GQA group %d x head_dim %d exceeds 2048", g, p->head_dim);
  if (p->layer_type == G4_SLIDING && p->window < 1)
    return fail(G4_ERR_INVALID_ARG, "sliding layer needs window >= 1 (got %d)", p->window);
  if (!(p->theta > 0.0f) || !isfinite(p->theta)) return fail(G4_ERR_INVALID_ARG, "theta must be finite and > 0");
  if (!(p->rotary_fraction >= 0.0f && p->rotary_fraction <= 1.0f))
    return fail(G4_ERR_INVALID_ARG, "rotary_fraction must lie in [0, 1]");
  if (!(p->eps >= 0.0f) || !isfinite(p->eps)) return fail(G4_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (!(p->attn_scale > 0.0f) || !isfinite(p->attn_scale))
    return fail(G4_ERR_INVALID_ARG, "attn_scale must be finite and > 0");
  return G4_OK;
}

// Resolves the cache a layer reads and checks that it matches the layer.
g4_status resolve_src(const g4_layer_params* p, const g4_kv_cache* caches, int n_layers, int layer,
                      const g4_kv_cache** out) {
  if (caches == nullptr) return fail(G4_ERR_INVALID_ARG, "caches is NULL");
  if (layer < 0 || layer >= n_layers) return fail(G4_ERR_INVALID_ARG, "layer %d outside [0, %d)", layer, n_layers);
  const int src = p->kv_share_src < 0 ? layer : p->kv_share_src;
  if (src >= n_layers) return fail(G4_ERR_INVALID_ARG, "kv_share_src %d outside [0, %d)", src, n_layers);
  const g4_kv_cache* c = &caches[src];
  if (c->k == nullptr || c->v == nullptr)
    return fail(G4_ERR_INVALID_ARG, "cache of layer %d (read by layer %d) has NULL k or v", src, layer);
  if (c->layer_type != p->layer_type || c->head_dim != p->head_dim || c->n_kv_heads != p->n_kv_heads ||
      c->dtype != p->dtype)
    return fail(G4_ERR_SHARE_MISMATCH,
                "layer %d (type %d, head_dim %d, n_kv %d, dtype %d) cannot read the cache of layer %d "
                "(type %d, head_dim %d, n_kv %d, dtype %d)",
                layer, p->layer_type, p->head_dim, p->n_kv_heads, p->dtype, src, c->layer_type, c->head_dim,
                c->n_kv_heads, c->dtype);
  if (c->max_len < 1 || c->batch < 1) return fail(G4_ERR_INVALID_ARG, "cache of layer %d has no rows", src);
  if (c->ring != 0 && c->ring != 1) return fail(G4_ERR_INVALID_ARG, "cache of layer %d: ring %d is neither 0 nor 1", src, c->ring);
  if (c->ring) {
    // A ring keeps the last max_len positions: only a sliding layer's window
    // fits in one, and the window itself must fit.
    if (c->layer_type != G4_SLIDING)
      return fail(G4_ERR_INVALID_ARG, "cache of layer %d is a ring but not a sliding layer's", src);
    if (c->max_len < p->window)
      return fail(G4_ERR_CAPACITY, "ring cache of layer %d has %d rows, fewer than the window %d", src, c->max_len,
                  p->window);
  }
  if (!aligned16(c->k) || !aligned16(c->v))
    return fail(G4_ERR_INVALID_ARG, "cache of layer %d is not 16-byte aligned", src);
  *out = c;
  return G4_OK;
}

g4_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(G4_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Scratch for g4_attn_decode_noalloc: a fixed array in device global memory,
// created when the library's device code is loaded on a GPU and held until the
// process exits.  Host code must not hand `g_noalloc_scratch` itself to a
// kernel (on the host it only names the symbol); noalloc_scratch() looks up
// its device address once per device.
constexpr size_t kNoAllocScratchBytes = G4_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

void* noalloc_scratch(cudaError_t* e) {
  static std::mutex mu;
  static void* addr[128] = {};
  int dev = 0;
  *e = cudaGetDevice(&dev);
  if (*e != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 128) {
    *e = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    *e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // with this device current
    if (*e != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" {

int32_t g4_kv_share_src(int32_t n_layers, int32_t n_shared, const int32_t* is_sliding, int32_t layer) {
  if (n_layers < 1 || n_shared < 0 || n_shared >= n_layers || is_sliding == nullptr || layer < 0 ||
      layer >= n_layers)
    return -2;
  const int first_shared = n_layers - n_shared;
  if (layer < first_shared) return -1;
  const int src = first_shared - (is_sliding[layer] ? 2 : 1);
  return src < 0 ? -2 : src;
}

g4_status g4_kv_append_normrope(const g4_layer_params* params, const g4_kv_cache* caches, int32_t n_layers,
                                int32_t layer, const void* q_in, const void* k_in, const void* v_in,
                                const float* q_norm_w, const float* k_norm_w, const int32_t* positions, int32_t B,
                                int32_t T, void* q_out, void* stream) {
  g4_status st = check_params(params);
  if (st != G4_OK) return st;
  if (B < 0 || T < 0) return fail(G4_ERR_INVALID_ARG, "B %d and T %d must be >= 0", B, T);
  if (q_in == nullptr || q_out == nullptr || q_norm_w == nullptr || positions == nullptr)
    return fail(G4_ERR_INVALID_ARG, "q_in, q_out, q_norm_w and positions must be non-NULL");
  if (!aligned16(q_in) || !aligned16(q_out) || !aligned16(q_norm_w))
    return fail(G4_ERR_INVALID_ARG, "q_in, q_out and q_norm_w must be 16-byte aligned");
  const bool shared = params->kv_share_src >= 0;
  g4::AppendArgs a;
  memset(&a, 0, sizeof(a));
  if (shared) {
    if (k_in != nullptr || v_in != nullptr || k_norm_w != nullptr)
      return fail(G4_ERR_INVALID_ARG, "layer %d shares the cache of layer %d: k_in, v_in and k_norm_w must be NULL",
                  layer, params->kv_share_src);
    if (layer < 0 || layer >= n_layers) return fail(G4_ERR_INVALID_ARG, "layer %d outside [0, %d)", layer, n_layers);
  } else {
    if (k_in == nullptr || v_in == nullptr || k_norm_w == nullptr)
      return fail(G4_ERR_INVALID_ARG, "layer %d owns its cache: k_in, v_in and k_norm_w must be non-NULL", layer);
    if (!aligned16(k_in) || !aligned16(v_in) || !aligned16(k_norm_w))
      return fail(G4_ERR_INVALID_ARG, "k_in, v_in and k_norm_w must be 16-byte aligned");
    const g4_kv_cache* c = nullptr;
    st = resolve_src(params, caches, n_layers, layer, &c);
    if (st != G4_OK) return st;
    if (c->batch < B) return fail(G4_ERR_CAPACITY, "cache batch %d < B %d", c->batch, B);
    a.cache_k = c->k;
    a.cache_v = c->v;
    a.max_len = c->max_len;
    a.ring = c->ring;
    a.k_in = k_in;
    a.v_in = v_in;
    a.k_w = k_norm_w;
  }
  if (B == 0 || T == 0) return ok();
  a.q_in = q_in;
  a.q_w = q_norm_w;
  a.positions = positions;
  a.q_out = q_out;
  a.B = B;
  a.T = T;
  a.H = params->n_heads;
  a.Hkv = params->n_kv_heads;
  a.hd = params->head_dim;
  a.eps = params->eps;
  const int nrows = a.H + (shared ? 0 : 2 * a.Hkv);
  // Tokens at the same t of up to 8 sequences share a CTA (and, when their
  // positions agree, one cos/sin table); small launches split the rows.
  a.tok_per_cta = T >= 16 ? (B < 8 ? B : 8) : 1;
  const long long ctas = static_cast<long long>(T) * ((B + a.tok_per_cta - 1) / a.tok_per_cta);
  a.rows_per_cta = ctas >= 1024 ? nrows : 4;
  // inv_freq[j] = theta^(-2j/hd) in float64, stored as float32; zero past the rotated pairs.
  const int half = a.hd / 2;
  int n_rot = static_cast<int>(floor(static_cast<double>(a.hd) * static_cast<double>(params->rotary_fraction) / 2.0));
  if (n_rot > half) n_rot = half;
  a.n_rot = n_rot;
  for (int j = 0; j < half; ++j)
    a.inv_freq[j] = j < n_rot ? static_cast<float>(pow(static_cast<double>(params->theta), -2.0 * j / a.hd)) : 0.0f;
  return cuda_status(g4::launch_append(a, params->dtype, static_cast<cudaStream_t>(stream)), "append launch");
}

g4_status g4_attn_prefill(const g4_layer_params* params, const g4_kv_cache* caches, int32_t n_layers,
                          int32_t layer, const void* q, const int32_t* q_start_pos, int32_t B, int32_t T,
                          void* out, void* stream) {
  g4_status st = check_params(params);
  if (st != G4_OK) return st;
  if (B < 0 || T < 0) return fail(G4_ERR_INVALID_ARG, "B %d and T %d must be >= 0", B, T);
  if (q == nullptr || out == nullptr || q_start_pos == nullptr)
    return fail(G4_ERR_INVALID_ARG, "q, out and q_start_pos must be non-NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(G4_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  const g4_kv_cache* c = nullptr;
  st = resolve_src(params, caches, n_layers, layer, &c);
  if (st != G4_OK) return st;
  if (c->batch < B) return fail(G4_ERR_CAPACITY, "cache batch %d < B %d", c->batch, B);
  if (c->ring) {
    // Every key of the chunk's windows must still be in the ring after the
    // chunk's own T rows went in: T + window - 1 positions.
    if (static_cast<long long>(T) + params->window - 1 > c->max_len)
      return fail(G4_ERR_CAPACITY, "ring cache of %d rows cannot hold the %d + %d - 1 keys a chunk of T = %d needs",
                  c->max_len, T, params->window, T);
    if (params->dtype == G4_BF16 && c->max_len % 128 != 0)
      return fail(G4_ERR_UNSUPPORTED, "bf16 prefill on a ring cache needs max_len a multiple of 128 (got %d)",
                  c->max_len);
  } else if (T > c->max_len) {
    return fail(G4_ERR_CAPACITY, "T %d exceeds the cache length %d", T, c->max_len);
  }
  if (B == 0 || T == 0) return ok();
  int* err = device_error_ptr();
  if (err == nullptr) return fail(G4_ERR_CUDA, "cannot resolve the device error word");
  const float scale_log2 = params->attn_scale * 1.4426950408889634f;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (params->dtype == G4_BF16) {
    g4::PrefillTcArgs a;
    memset(&a, 0, sizeof(a));
    a.q = q;
    a.ck = c->k;
    a.cv = c->v;
    a.out = out;
    a.q_start = q_start_pos;
    a.err = err;
    a.B = B;
    a.T = T;
    a.H = params->n_heads;
    a.Hkv = params->n_kv_heads;
    a.hd = params->head_dim;
    a.max_len = c->max_len;
    a.ring = c->ring;
    a.sliding = params->layer_type == G4_SLIDING;
    a.window = params->window;
    a.scale_log2 = scale_log2;
    return cuda_status(g4::launch_prefill_tc(a, s), "tcgen05 prefill launch");
  }
  g4::AttnSimtArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.ck = c->k;
  a.cv = c->v;
  a.out = out;
  a.base = q_start_pos;
  a.err = err;
  a.mode = 1;
  a.B = B;
  a.T = T;
  a.H = params->n_heads;
  a.Hkv = params->n_kv_heads;
  a.hd = params->head_dim;
  a.max_len = c->max_len;
  a.ring = c->ring;
  a.sliding = params->layer_type == G4_SLIDING;
  a.window = params->window;
  a.len_cap = c->max_len;
  a.chunk = a.sliding ? params->window : c->max_len;
  a.nsplit = 1;
  a.scale_log2 = scale_log2;
  return cuda_status(g4::launch_attn_simt(a, params->dtype, s), "float32 prefill launch");
}

g4_status g4_attn_encoder(const g4_layer_params* params, const g4_kv_cache* caches, int32_t n_layers,
                          int32_t layer, const void* q, int32_t B, int32_t T, void* out, void* stream) {
  g4_status st = check_params(params);
  if (st != G4_OK) return st;
  if (B < 0 || T < 0) return fail(G4_ERR_INVALID_ARG, "B %d and T %d must be >= 0", B, T);
  if (q == nullptr || out == nullptr) return fail(G4_ERR_INVALID_ARG, "q and out must be non-NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(G4_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  const g4_kv_cache* c = nullptr;
  st = resolve_src(params, caches, n_layers, layer, &c);
  if (st != G4_OK) return st;
  if (c->ring)
    return fail(G4_ERR_INVALID_ARG, "the encoder reads the sequence's keys at rows 0 .. T-1: a ring cache cannot hold them");
  if (c->batch < B) return fail(G4_ERR_CAPACITY, "cache batch %d < B %d", c->batch, B);
  if (T > c->max_len) return fail(G4_ERR_CAPACITY, "T %d exceeds the cache length %d", T, c->max_len);
  if (B == 0 || T == 0) return ok();
  int* err = device_error_ptr();
  if (err == nullptr) return fail(G4_ERR_CUDA, "cannot resolve the device error word");
  const bool sliding = params->layer_type == G4_SLIDING;
  // A window of T or more keys reaches every key; capping it keeps i + window
  // in range.
  const int window = sliding ? (params->window < T ? params->window : T) : 0;
  const float scale_log2 = params->attn_scale * 1.4426950408889634f;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (params->dtype == G4_BF16) {
    g4::PrefillTcArgs a;
    memset(&a, 0, sizeof(a));
    a.q = q;
    a.ck = c->k;
    a.cv = c->v;
    a.out = out;
    a.q_start = nullptr;  // unused: token t sits at position t
    a.err = err;
    a.B = B;
    a.T = T;
    a.H = params->n_heads;
    a.Hkv = params->n_kv_heads;
    a.hd = params->head_dim;
    a.max_len = c->max_len;
    a.sliding = sliding;
    a.window = window;
    a.bidir = 1;
    a.scale_log2 = scale_log2;
    return cuda_status(g4::launch_prefill_tc(a, s), "tcgen05 encoder launch");
  }
  g4::AttnSimtArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.ck = c->k;
  a.cv = c->v;
  a.out = out;
  a.err = err;
  a.mode = 2;
  a.B = B;
  a.T = T;
  a.H = params->n_heads;
  a.Hkv = params->n_kv_heads;
  a.hd = params->head_dim;
  a.max_len = c->max_len;
  a.sliding = sliding;
  a.window = window;
  a.len_cap = c->max_len;
  // one split holds a query's whole key range (2 window + 1 keys at most, T at most)
  a.chunk = sliding && 2LL * window + 1 < T ? 2 * window + 1 : T;
  a.nsplit = 1;
  a.scale_log2 = scale_log2;
  return cuda_status(g4::launch_attn_simt(a, params->dtype, s), "float32 encoder launch");
}

size_t g4_attn_decode_workspace_size(const g4_layer_params* params, int32_t B, int32_t max_seq_len) {
  if (check_params(params) != G4_OK || B < 1 || max_seq_len < 1) return 0;
  return g4::decode_plan(params->dtype, params->layer_type == G4_SLIDING, params->window, params->head_dim, params->n_heads,
                         params->n_kv_heads, B, max_seq_len)
      .ws_bytes;
}

}  // extern "C"

namespace {

// Shared by g4_attn_decode and g4_decode_step: validation, split plan and launch.
// q is normed+roped (fused == false) or the raw projection (fused == true, with
// k_in / v_in / weights and the RoPE table of the layer).
// With clear_tickets the splits' arrival counters in the workspace are
// zeroed on the stream right before the launch, after every check passed
// (the built-in scratch of g4_attn_decode_noalloc; a caller's workspace is
// left zeroed by the previous call instead).
g4_status decode_common(const g4_layer_params* params, const g4_kv_cache* caches, int32_t n_layers, int32_t layer,
                        const void* q, const void* k_in, const void* v_in, const float* q_norm_w,
                        const float* k_norm_w, bool fused, const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                        void* out, void* workspace, size_t workspace_bytes, void* stream,
                        bool clear_tickets = false) {
  g4_status st = check_params(params);
  if (st != G4_OK) return st;
  if (B < 0) return fail(G4_ERR_INVALID_ARG, "B %d must be >= 0", B);
  if (q == nullptr || out == nullptr || seq_lens == nullptr)
    return fail(G4_ERR_INVALID_ARG, "q, out and seq_lens must be non-NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(G4_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  const bool shared = params->kv_share_src >= 0;
  if (fused) {
    if (q_norm_w == nullptr || !aligned16(q_norm_w))
      return fail(G4_ERR_INVALID_ARG, "q_norm_w must be non-NULL and 16-byte aligned");
    if (shared && (k_in != nullptr || v_in != nullptr || k_norm_w != nullptr))
      return fail(G4_ERR_INVALID_ARG, "layer %d shares the cache of layer %d: k_in, v_in and k_norm_w must be NULL",
                  layer, params->kv_share_src);
    if (!shared && (k_in == nullptr || v_in == nullptr || k_norm_w == nullptr))
      return fail(G4_ERR_INVALID_ARG, "layer %d owns its cache: k_in, v_in and k_norm_w must be non-NULL", layer);
    if (!shared && (!aligned16(k_in) || !aligned16(v_in) || !aligned16(k_norm_w)))
      return fail(G4_ERR_INVALID_ARG, "k_in, v_in and k_norm_w must be 16-byte aligned");
  }
  const g4_kv_cache* c = nullptr;
  st = resolve_src(params, caches, n_layers, layer, &c);
  if (st != G4_OK) return st;
  if (c->batch < B) return fail(G4_ERR_CAPACITY, "cache batch %d < B %d", c->batch, B);
  if (max_seq_len < 1 || (!c->ring && max_seq_len > c->max_len))
    return fail(G4_ERR_CAPACITY, "max_seq_len %d outside [1, cache length %d]", max_seq_len, c->max_len);
  if (B == 0) return ok();
  const g4::DecodePlan plan = g4::decode_plan(params->dtype, params->layer_type == G4_SLIDING, params->window, params->head_dim,
                                              params->n_heads, params->n_kv_heads, B, max_seq_len);
  if (workspace_bytes < plan.ws_bytes)
    return fail(G4_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", workspace_bytes, plan.ws_bytes);
  if (plan.ws_bytes > 0 && (workspace == nullptr || !aligned16(workspace)))
    return fail(G4_ERR_INVALID_ARG, "workspace must be non-NULL and 16-byte aligned");
  int* err = device_error_ptr();
  if (err == nullptr) return fail(G4_ERR_CUDA, "cannot resolve the device error word");
  g4::AttnSimtArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.ck = c->k;
  a.cv = c->v;
  a.out = out;
  a.base = seq_lens;
  a.err = err;
  a.mode = 0;
  a.B = B;
  a.T = 1;
  a.H = params->n_heads;
  a.Hkv = params->n_kv_heads;
  a.hd = params->head_dim;
  a.max_len = c->max_len;
  a.ring = c->ring;
  a.sliding = params->layer_type == G4_SLIDING;
  a.window = params->window;
  a.len_cap = max_seq_len;
  a.chunk = plan.chunk;
  a.nsplit = plan.nsplit;
  a.scale_log2 = params->attn_scale * 1.4426950408889634f;
  if (plan.nsplit > 1) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.ws_o = reinterpret_cast<float*>(ws);
    a.ws_m = reinterpret_cast<float*>(ws + plan.o_bytes);
    a.ws_l = reinterpret_cast<float*>(ws + plan.o_bytes + plan.m_bytes);
    a.tickets = reinterpret_cast<unsigned*>(ws + plan.o_bytes + 2 * plan.m_bytes);
    if (clear_tickets) {
      const cudaError_t e = cudaMemsetAsync(a.tickets, 0, plan.t_bytes, static_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) return cuda_status(e, "clearing the decode scratch's arrival counters");
    }
  }
  if (fused) {
    a.fused = 1;
    a.q_w = q_norm_w;
    a.eps = params->eps;
    if (!shared) {
      a.k_raw = k_in;
      a.v_raw = v_in;
      a.k_w = k_norm_w;
      a.cache_k = caches[layer].k;
      a.cache_v = caches[layer].v;
    }
    const int half = a.hd / 2;
    int n_rot =
        static_cast<int>(floor(static_cast<double>(a.hd) * static_cast<double>(params->rotary_fraction) / 2.0));
    if (n_rot > half) n_rot = half;
    a.n_rot = n_rot;
    for (int j = 0; j < half; ++j)
      a.inv_freq[j] =
          j < n_rot ? static_cast<float>(pow(static_cast<double>(params->theta), -2.0 * j / a.hd)) : 0.0f;
  }
  if (plan.win)
    return cuda_status(g4::launch_decode_win(a, static_cast<cudaStream_t>(stream)), "windowed decode launch");
  return cuda_status(g4::launch_attn_simt(a, params->dtype, static_cast<cudaStream_t>(stream)), "decode launch");
}

}  // namespace

extern "C" {

g4_status g4_attn_decode(const g4_layer_params* params, const g4_kv_cache* caches, int32_t n_layers, int32_t layer,
                         const void* q, const int32_t* seq_lens, int32_t B, int32_t max_seq_len, void* out,
                         void* workspace, size_t workspace_bytes, void* stream) {
  return decode_common(params, caches, n_layers, layer, q, nullptr, nullptr, nullptr, nullptr, false, seq_lens, B,
                       max_seq_len, out, workspace, workspace_bytes, stream);
}

g4_status g4_decode_step(const g4_layer_params* params, const g4_kv_cache* caches, int32_t n_layers, int32_t layer,
                         const void* q_in, const void* k_in, const void* v_in, const float* q_norm_w,
                         const float* k_norm_w, const int32_t* seq_lens, int32_t B, int32_t max_seq_len, void* out,
                         void* workspace, size_t workspace_bytes, void* stream) {
  return decode_common(params, caches, n_layers, layer, q_in, k_in, v_in, q_norm_w, k_norm_w, true, seq_lens, B,
                       max_seq_len, out, workspace, workspace_bytes, stream);
}

g4_status g4_attn_decode_noalloc(const g4_layer_params* params, const g4_kv_cache* caches, int32_t n_layers,
                                 int32_t layer, const void* q, const int32_t* seq_lens, int32_t B,
                                 int32_t max_seq_len, void* out, void* stream) {
  g4_status st = check_params(params);
  if (st != G4_OK) return st;
  if (B >= 1 && max_seq_len >= 1) {
    const g4::DecodePlan plan = g4::decode_plan(params->dtype, params->layer_type == G4_SLIDING, params->window,
                                                params->head_dim, params->n_heads, params->n_kv_heads, B,
                                                max_seq_len);
    if (plan.ws_bytes > kNoAllocScratchBytes)
      return fail(G4_ERR_WORKSPACE,
                  "this decode needs %zu bytes of scratch, more than the %zu bytes built into the library for "
                  "g4_attn_decode_noalloc; call g4_attn_decode with a caller-allocated workspace instead",
                  plan.ws_bytes, kNoAllocScratchBytes);
  }
  cudaError_t e = cudaSuccess;
  void* scratch = noalloc_scratch(&e);
  if (scratch == nullptr) return fail(G4_ERR_CUDA, "cannot resolve the built-in decode scratch: %s", cudaGetErrorString(e));
  // Same kernels and split plan as g4_attn_decode, with the split partials in
  // the built-in array.  The partials are written before they are read; the
  // splits' arrival counters must start at zero, so decode_common clears them
  // once every argument has been checked, just before the launch.
  return decode_common(params, caches, n_layers, layer, q, nullptr, nullptr, nullptr, nullptr, false, seq_lens, B,
                       max_seq_len, out, scratch, kNoAllocScratchBytes, stream, /*clear_tickets=*/true);
}

g4_status g4_qkv_project_append(const g4_layer_params* params, const g4_kv_cache* caches, int32_t n_layers,
                                int32_t layer, const void* x, int32_t D, const void* w_qkv, const float* q_norm_w,
                                const float* k_norm_w, const int32_t* positions, int32_t B, int32_t T, void* q_out,
                                void* stream) {
  g4_status st = check_params(params);
  if (st != G4_OK) return st;
  if (params->dtype != G4_BF16)
    return fail(G4_ERR_UNSUPPORTED, "the fused projection runs on the bf16 tensor cores only");
  if (B < 0 || T < 0) return fail(G4_ERR_INVALID_ARG, "B %d and T %d must be >= 0", B, T);
  if (D < 64 || D % 64 != 0) return fail(G4_ERR_UNSUPPORTED, "D %d must be a positive multiple of 64", D);
  if (x == nullptr || w_qkv == nullptr || q_norm_w == nullptr || positions == nullptr || q_out == nullptr)
    return fail(G4_ERR_INVALID_ARG, "x, w_qkv, q_norm_w, positions and q_out must be non-NULL");
  if (!aligned16(x) || !aligned16(w_qkv) || !aligned16(q_out) || !aligned16(q_norm_w))
    return fail(G4_ERR_INVALID_ARG, "x, w_qkv, q_norm_w and q_out must be 16-byte aligned");
  const bool shared = params->kv_share_src >= 0;
  g4::GemmArgs a;
  memset(&a, 0, sizeof(a));
  if (shared) {
    if (k_norm_w != nullptr)
      return fail(G4_ERR_INVALID_ARG, "layer %d shares the cache of layer %d: k_norm_w must be NULL", layer,
                  params->kv_share_src);
    if (layer < 0 || layer >= n_layers) return fail(G4_ERR_INVALID_ARG, "layer %d outside [0, %d)", layer, n_layers);
  } else {
    if (k_norm_w == nullptr || !aligned16(k_norm_w))
      return fail(G4_ERR_INVALID_ARG, "layer %d owns its cache: k_norm_w must be non-NULL and 16-byte aligned", layer);
    const g4_kv_cache* c = nullptr;
    st = resolve_src(params, caches, n_layers, layer, &c);
    if (st != G4_OK) return st;
    if (c->batch < B) return fail(G4_ERR_CAPACITY, "cache batch %d < B %d", c->batch, B);
    a.cache_k = c->k;
    a.cache_v = c->v;
    a.max_len = c->max_len;
    a.ring = c->ring;
    a.k_w = k_norm_w;
  }
  const long long M = static_cast<long long>(B) * T;
  if (M == 0) return ok();
  if (M > 0x7fffffffLL - 128) return fail(G4_ERR_INVALID_ARG, "B * T too large");
  const int hd = params->head_dim;
  a.epi = 0;
  a.M = static_cast<int>(M);
  a.K = D;
  a.N = (params->n_heads + (shared ? 0 : 2 * params->n_kv_heads)) * hd;
  a.B = B;
  a.T = T;
  a.H = params->n_heads;
  a.Hkv = params->n_kv_heads;
  a.hd = hd;
  a.eps = params->eps;
  a.eps_in = params->eps;
  a.q_w = q_norm_w;
  a.positions = positions;
  a.q_out = q_out;
  const int half = hd / 2;
  int n_rot = static_cast<int>(floor(static_cast<double>(hd) * static_cast<double>(params->rotary_fraction) / 2.0));
  if (n_rot > half) n_rot = half;
  a.n_rot = n_rot;
  for (int j = 0; j < half; ++j)
    a.inv_freq[j] = j < n_rot ? static_cast<float>(pow(static_cast<double>(params->theta), -2.0 * j / hd)) : 0.0f;
  int* err = device_error_ptr();
  if (err == nullptr) return fail(G4_ERR_CUDA, "cannot resolve the device error word");
  a.err = err;
  return cuda_status(g4::launch_gemm_tc(a, x, w_qkv, static_cast<cudaStream_t>(stream)), "projection launch");
}

g4_status g4_attn_out_residual(const void* ao, int32_t M, int32_t K, const void* w_o, int32_t D,
                               const float* post_norm_w, float eps, const void* h, void* out, void* stream) {
  if (M < 0) return fail(G4_ERR_INVALID_ARG, "M %d must be >= 0", M);
  if (K < 64 || K % 64 != 0) return fail(G4_ERR_UNSUPPORTED, "K %d must be a positive multiple of 64", K);
  if (D < 256 || D % 256 != 0 || D > 2048)
    return fail(G4_ERR_UNSUPPORTED, "D %d must be a multiple of 256 in [256, 2048]", D);
  if (!(eps >= 0.0f) || !isfinite(eps)) return fail(G4_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (ao == nullptr || w_o == nullptr || post_norm_w == nullptr || h == nullptr || out == nullptr)
    return fail(G4_ERR_INVALID_ARG, "ao, w_o, post_norm_w, h and out must be non-NULL");
  if (!aligned16(ao) || !aligned16(w_o) || !aligned16(h) || !aligned16(out))
    return fail(G4_ERR_INVALID_ARG, "ao, w_o, h and out must be 16-byte aligned");
  if (M == 0) return ok();
  if (M > 0x7fffffff - 128) return fail(G4_ERR_INVALID_ARG, "M too large");
  int* err = device_error_ptr();
  if (err == nullptr) return fail(G4_ERR_CUDA, "cannot resolve the device error word");
  g4::GemmArgs a;
  memset(&a, 0, sizeof(a));
  a.epi = 1;
  a.M = M;
  a.K = K;
  a.N = D;
  a.err = err;
  a.eps = eps;
  a.h = h;
  a.out = out;
  a.post_w = post_norm_w;
  return cuda_status(g4::launch_gemm_tc(a, ao, w_o, static_cast<cudaStream_t>(stream)), "o_proj launch");
}

const char* g4_last_error(void) { return g_last_error.c_str(); }

int32_t g4_take_device_error(void) {
  int* p = device_error_ptr();
  if (p == nullptr) return -1;
  int v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
  const int zero = 0;
  if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return -1;
  return v;
}

}  // extern "C"

/*
 * g4attn.h -- C ABI of the GB300 (sm_103a) Gemma-4 E-series dual-geometry
 * attention path.
 *
 * The path, per layer of an attention-only stack:
 *   1. g4_kv_append_normrope: per-head RMSNorm of q and k (plain x-hat * w,
 *      eps inside the mean), weight-less RMSNorm of v, rotate_half RoPE on q
 *      and k, and the write of k and v into the layer's KV cache.
 *   2. g4_attn_prefill / g4_attn_decode: causal GQA softmax attention with
 *      score scale attn_scale (1.0 for Gemma-4), windowed on sliding layers,
 *      over the cache of the layer itself or, on a shared-KV tail layer, of
 *      its source layer.  g4_attn_encoder: the bidirectional (encoder) form.
 *
 * Sources (page title + item):
 *   cortiq-engine g4e.rs: `rms`, `rms_plain`, `G4eGlobals` (inv_freq tables,
 *     window counted with the current token), `G4eLayer` (kv_share_src,
 *     sliding, hd),
 *     `g4e_forward` attention block.
 *   ferrox-models gemma4_engine.rs: `Gemma4Hparams` (head_dim per type,
 *     has_kv, kv_reuse_layer, rope_theta_for, attention_scale = 1.0),
 *     `forward_token_on_worker` (norm per head, RoPE, push, windowed /
 *     unwindowed causal GQA attention, shared-KV head_dim check).
 *   taconite-embeddinggemma2 model.rs: `rope_half`, `text_attention`
 *     (rotate_half pairing, head grouping kh = hh / group).
 *   turbospark-runtime gemma4/attn.rs: `encode_gemma4_layer_attn_and_router`
 *     (RMS_EPS = 1e-6, rotated_pairs, kv_start = seq_len - sliding_window).
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers owned by the caller; the
 *     library allocates no device memory and keeps no state between calls
 *     except a thread-local error message, one device-side error word (see
 *     g4_take_device_error), the built-in scratch of g4_attn_decode_noalloc
 *     and 64 pairs of work-item counters of the bf16 prefill (see
 *     g4_attn_prefill), all of them static device variables.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL is the legacy default stream).  A call that returns G4_OK has only
 *     enqueued work.
 *   - Host-detectable errors return a status before anything is launched;
 *     nothing is written then.  g4_last_error() gives the message.
 *   - Device-side values (positions, lengths) cannot be checked on the host.
 *     Kernels clamp them so that no access leaves the buffers; rows with
 *     out-of-contract values get unspecified contents.
 *   - Pointers to q/k/v/out/cache must be 16-byte aligned.
 *   - dtype is per layer and covers q_in/k_in/v_in, the cache, q_out and the
 *     attention output alike: G4_F32 (float) or G4_BF16 (bfloat16, RNE on
 *     every store).  Norm weights are always float32.  Arithmetic is float32
 *     with float32 accumulation (bf16 tensor-core inputs in bf16 prefill).
 */
#ifndef G4ATTN_H
#define G4ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  G4_OK = 0,
  G4_ERR_INVALID_ARG = 1,    /* null / misaligned pointer, bad size or field      */
  G4_ERR_UNSUPPORTED = 2,    /* head_dim or GQA group not built                    */
  G4_ERR_SHARE_MISMATCH = 3, /* shared layer's source cache has another type,
                                head_dim, kv-head count or dtype                   */
  G4_ERR_CAPACITY = 4,       /* batch or length larger than the cache              */
  G4_ERR_WORKSPACE = 5,      /* decode workspace too small                         */
  G4_ERR_CUDA = 6            /* a CUDA runtime/driver call or launch failed        */
} g4_status;

typedef enum { G4_SLIDING = 0, G4_FULL = 1 } g4_layer_type;
typedef enum { G4_F32 = 0, G4_BF16 = 1 } g4_dtype;

/*
 * Per-layer attention hyperparameters (ferrox-models `Gemma4Hparams`,
 * cortiq-engine `G4eLayer`).
 *   layer_type      G4_SLIDING or G4_FULL.
 *   head_dim        this layer's head width: head_dim on sliding layers,
 *                   global_head_dim on full layers.  64, 128, 256 or 512.
 *   n_heads         query heads H; n_kv_heads Hkv divides it and the group
 *                   H / Hkv is 1, 2, 4 or 8 (with group * head_dim <= 2048).
 *   window          sliding window in tokens, current token included (a key
 *                   j is visible from query i iff j <= i and i - j < window).
 *                   Must be >= 1 on sliding layers; ignored on full layers.
 *   theta           RoPE base (local theta on sliding, model theta on full).
 *   rotary_fraction fraction of the head that is rotated: the first
 *                   floor(head_dim * rotary_fraction / 2) pairs rotate with
 *                   inv_freq[j] = theta^(-2j / head_dim); the other pairs have
 *                   inv_freq 0 (identity).  1.0 on sliding layers, the
 *                   partial-rotary factor (e.g. 0.25) on full layers.
 *   eps             RMSNorm epsilon (1e-6), added to the mean square.
 *   attn_scale      score scale, > 0 (Gemma-4: 1.0).
 *   kv_share_src    -1 if the layer owns its cache, else the index of the
 *                   layer whose cache it reads (see g4_kv_share_src).
 *   dtype           g4_dtype of every tensor of the layer.
 */
typedef struct {
  int32_t layer_type;
  int32_t head_dim;
  int32_t n_heads;
  int32_t n_kv_heads;
  int32_t window;
  float theta;
  float rotary_fraction;
  float eps;
  float attn_scale;
  int32_t kv_share_src;
  int32_t dtype;
} g4_layer_params;

/*
 * One layer's KV cache, caller-owned device memory, layout
 * k[batch][n_kv_heads][max_len][head_dim] (same for v): rows of head_dim
 * contiguous.  Layers that read another layer's cache may leave their entry
 * zeroed.
 *   ring = 0  linear cache: position p lives in row p, positions < max_len.
 *   ring = 1  sliding-window ring buffer (turbospark-runtime gemma4 decode:
 *             `ring_capacity`, `active_ring`): position p lives in row
 *             p mod max_len, any p >= 0, so the cache keeps the last max_len
 *             positions.  Only on a G4_SLIDING cache, with max_len >= the
 *             layer's window (G4_ERR_INVALID_ARG / G4_ERR_CAPACITY otherwise).
 *             A ring of `window` rows serves decode; a prefill chunk of T
 *             tokens needs max_len >= T + window - 1 (see g4_attn_prefill).
 */
typedef struct {
  void* k;
  void* v;
  int32_t layer_type;
  int32_t head_dim;
  int32_t n_kv_heads;
  int32_t max_len;
  int32_t batch;
  int32_t dtype;
  int32_t ring;
} g4_kv_cache;

/*
 * Shared-KV routing (ferrox-models `Gemma4Hparams::kv_reuse_layer`;
 * cortiq-engine g4e.rs module doc).  With first_shared = n_layers - n_shared:
 * returns -1 for layer < first_shared (owns its cache), first_shared - 2 for a
 * sliding tail layer and first_shared - 1 for a full tail layer.
 * is_sliding[n_layers] holds 1 for sliding layers.  Returns -2 on invalid
 * arguments (n_layers < 1, n_shared outside [0, n_layers), layer out of range,
 * NULL is_sliding, or a source index < 0).  Host only.
 */
int32_t g4_kv_share_src(int32_t n_layers, int32_t n_shared, const int32_t* is_sliding, int32_t layer);

/*
 * Step a4: fused norm -> RoPE -> KV append for B*T tokens of one layer.
 *   q_in       [B][T][n_heads][head_dim]      raw q projections
 *   k_in, v_in [B][T][n_kv_heads][head_dim]   raw k / v projections; must be
 *              NULL on a shared layer (kv_share_src >= 0), non-NULL otherwise.
 *              A full layer whose v projection is its k projection
 *              (turbospark-runtime gemma4 `attention_k_eq_v`) passes the raw
 *              k as v_in too; v is then the weight-less norm of the raw k.
 *   q_norm_w   [head_dim] float32 weight shared by all q heads
 *   k_norm_w   [head_dim] float32 weight shared by all k heads (NULL on a
 *              shared layer).  v has no weight.
 *   positions  [B][T] int32: the RoPE position of each token and the cache row
 *              it is written to (row = position on a linear cache, position
 *              mod max_len on a ring).  Negative positions, and positions
 *              >= max_len of a linear cache, are not written.
 *   q_out      [B][T][n_heads][head_dim] normed + roped q; may equal q_in.
 * The layer's cache is caches[layer] (n_layers entries).  Writes exactly the
 * rows k[b][*][row(positions[b][t])][*] and v[...] for every (b, t); nothing
 * else in the cache changes.  Two tokens of one call that map to the same
 * ring row leave either one there.  RoPE angles are pos * inv_freq[j] with
 * inv_freq held in float32 and the angle reduced in float64.
 */
g4_status g4_kv_append_normrope(const g4_layer_params* params, const g4_kv_cache* caches, int32_t n_layers,
                                int32_t layer, const void* q_in, const void* k_in, const void* v_in,
                                const float* q_norm_w, const float* k_norm_w, const int32_t* positions,
                                int32_t B, int32_t T, void* q_out, void* stream);

/*
 * Step a5 (+ a7): prefill attention of T new tokens per sequence.
 *   q            [B][T][n_heads][head_dim], normed + roped (g4_kv_append_normrope's q_out)
 *   q_start_pos  [B] int32 device: token t of sequence b sits at position
 *                q_start_pos[b] + t; the cache of the source layer must
 *                already hold positions [0, q_start_pos[b] + T).  On a ring
 *                cache those are the last max_len of them, and every key the
 *                chunk needs is still there when max_len >= T + window - 1
 *                (checked: G4_ERR_CAPACITY); a bf16 ring also needs max_len
 *                a multiple of 128, the key tile (G4_ERR_UNSUPPORTED).
 *   out          [B][T][n_heads][head_dim]
 * Reads caches[src], src = kv_share_src < 0 ? layer : kv_share_src, which must
 * match the layer's type, head_dim, n_kv_heads and dtype
 * (G4_ERR_SHARE_MISMATCH otherwise).  bf16 runs on the tcgen05 tensor cores
 * (bf16 operands, float32 accumulation, P rounded to bf16); f32 runs on CUDA
 * cores in float32.  The bf16 kernel is persistent: its CTAs draw work items
 * from a counter pair the library keeps in device memory, one of 64 taken in
 * turn per call and cleared by the launch when it ends; so at most 64 bf16
 * prefill launches may be in flight at the same time (any streams).  A CUDA
 * graph keeps the pair it was captured with: replays of one graph, or of two
 * graphs whose prefill captures were a multiple of 64 calls apart, must not
 * overlap.
 */
g4_status g4_attn_prefill(const g4_layer_params* params, const g4_kv_cache* caches, int32_t n_layers,
                          int32_t layer, const void* q, const int32_t* q_start_pos, int32_t B, int32_t T,
                          void* out, void* stream);

/*
 * Bidirectional (encoder) attention, the form of taconite-embeddinggemma2
 * model.rs `text_attention`: no causal mask; a key j is visible from query i
 * iff |i - j| <= window on a sliding layer (the window counts keys on each
 * side, the token itself in the middle), every key on a full layer.
 *   q    [B][T][n_heads][head_dim], normed + roped at positions 0 .. T-1
 *        (g4_kv_append_normrope's q_out with positions[b][t] = t)
 *   out  [B][T][n_heads][head_dim]
 * The keys and values are the same T tokens, rows [0, T) of caches[src]
 * (appended by g4_kv_append_normrope at positions 0 .. T-1; src as in
 * g4_attn_prefill).  A ring cache is refused (G4_ERR_INVALID_ARG); T must
 * not exceed max_len (G4_ERR_CAPACITY).  Score scale attn_scale.  bf16 runs
 * on the tcgen05 tensor cores, f32 on CUDA cores, like g4_attn_prefill (the
 * bf16 kernel takes one of the same 64 work-item counter pairs).
 */
g4_status g4_attn_encoder(const g4_layer_params* params, const g4_kv_cache* caches, int32_t n_layers,
                          int32_t layer, const void* q, int32_t B, int32_t T, void* out, void* stream);

/*
 * Workspace bytes g4_attn_decode / g4_decode_step need for this layer, batch
 * and bound on the sequence lengths (0 means no workspace is needed).
 */
size_t g4_attn_decode_workspace_size(const g4_layer_params* params, int32_t B, int32_t max_seq_len);

/*
 * Step a6 (+ a7): one query token per sequence (decode).
 *   q            [B][n_heads][head_dim], normed + roped
 *   seq_lens     [B] int32 device: keys per sequence INCLUDING the new token,
 *                which sits at position seq_lens[b] - 1 (append it first).
 *                Values are clamped into [1, max_seq_len].
 *   max_seq_len  host-side upper bound of seq_lens, 1..cache max_len (any
 *                value >= 1 on a ring cache); it sizes the split-KV grid and
 *                the workspace.
 *   out          [B][n_heads][head_dim]
 *   workspace    device scratch of at least g4_attn_decode_workspace_size()
 *                bytes (may be NULL when that is 0); caller-owned, 16-byte
 *                aligned.  Zero-fill it once before its first use: it holds
 *                arrival counters that every call leaves at zero again.
 * Sliding layers read keys [max(0, L - window), L), full layers [0, L).  The
 * key range is split across CTAs (split-KV); the CTA that finishes last for a
 * (sequence, kv head) merges the splits with log-sum-exp weights.  Calls
 * sharing a workspace must not overlap on the GPU.
 */
g4_status g4_attn_decode(const g4_layer_params* params, const g4_kv_cache* caches, int32_t n_layers,
                         int32_t layer, const void* q, const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                         void* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Steps a4 + a6 (+ a7) in one launch: the decode step of one layer from the
 * new token's raw projections.  Same result as g4_kv_append_normrope with
 * positions[b] = seq_lens[b] - 1 (T = 1) followed by g4_attn_decode on its
 * q_out, without the q_out round trip through memory:
 *   q_in         [B][n_heads][head_dim] raw q of the new token
 *   k_in, v_in   [B][n_kv_heads][head_dim] raw k / v (NULL on a shared layer;
 *                the same pointer twice for attention_k_eq_v, as above)
 *   q_norm_w, k_norm_w  float32 [head_dim] (k_norm_w NULL on a shared layer)
 * On a layer that owns its cache the new k / v rows are written to position
 * seq_lens[b] - 1 of caches[layer] (row seq_lens[b] - 1, or that mod max_len
 * on a ring, which overwrites a key the window no longer sees).  Other
 * arguments as g4_attn_decode.
 */
g4_status g4_decode_step(const g4_layer_params* params, const g4_kv_cache* caches, int32_t n_layers, int32_t layer,
                         const void* q_in, const void* k_in, const void* v_in, const float* q_norm_w,
                         const float* k_norm_w, const int32_t* seq_lens, int32_t B, int32_t max_seq_len, void* out,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * The step before the path, fused into it: the q / k / v projections of one
 * layer for B*T tokens, their input RMSNorm, and the per-head norm / RoPE /
 * KV append of g4_kv_append_normrope, on the tcgen05 tensor cores
 * (cortiq-engine g4e.rs `g4e_forward`: `rms(h, attn_norm)`, then `matvec`
 * with wq / wk / wv, then the per-head norm, RoPE and `append`;
 * turbospark-runtime gemma4/attn.rs writes the projections straight into the
 * KV slot and norms / ropes them there).  bf16 only (G4_ERR_UNSUPPORTED for
 * float32 layers).
 *   x        [B][T][D] bf16: the layer input (residual stream), D a multiple
 *            of 64.
 *   w_qkv    [N][D] bf16, N = (n_heads + 2 n_kv_heads) * head_dim rows: the
 *            rows of Wq, then Wk, then Wv (n_heads * head_dim rows, Wq only,
 *            on a shared layer), each column k multiplied by the attention-norm
 *            weight attn_norm_w[k] (folded in once by the caller, as
 *            taconite-embeddinggemma2 model.rs folds RMSNorm weights into its
 *            GEMM operands).  The kernel applies the rest of the input norm,
 *            the row scale (mean(x^2) + eps)^-1/2 with the layer's eps.
 *   q_norm_w, k_norm_w, positions, q_out  as g4_kv_append_normrope (k_norm_w
 *            NULL on a shared layer).
 * q = (x scale) Wq^T etc. accumulate in float32 from bf16 products; the
 * per-head norm, RoPE and the bf16 rounding (to nearest even) follow in
 * float32.  So the stored values are those of g4_kv_append_normrope on the
 * exact projections to within one bf16 unit in the last place, where the
 * float32 accumulation lands next to a rounding boundary.  Writes q_out and
 * the cache rows of the tokens' positions (positions outside a linear cache
 * are not written), nothing else.  The launch takes one 128-token x
 * head_dim output tile per CTA.
 */
g4_status g4_qkv_project_append(const g4_layer_params* params, const g4_kv_cache* caches, int32_t n_layers,
                                int32_t layer, const void* x, int32_t D, const void* w_qkv, const float* q_norm_w,
                                const float* k_norm_w, const int32_t* positions, int32_t B, int32_t T, void* q_out,
                                void* stream);

/*
 * The step after the path: o_proj, the post-attention RMSNorm and the
 * residual add (cortiq-engine g4e.rs `g4e_forward`: `wo`, then the sandwich
 * norm `rms(.., post_attn_norm)` added to the hidden state; ferrox-models
 * gemma4_engine.rs `forward_token_on_worker`: `o_proj`, `post_attn_norm`,
 * residual), on the tcgen05 tensor cores, bf16:
 *   out[m][:] = h[m][:] + rmsnorm(ao[m][:] . w_o^T, post_norm_w, eps)
 *   ao           [M][K] bf16: attention output rows (K = n_heads * head_dim,
 *                a multiple of 64), e.g. g4_attn_prefill's out as [B*T][H*hd]
 *   w_o          [D][K] bf16
 *   post_norm_w  [D] float32; eps added to the mean square
 *   h            [M][D] bf16 residual stream; out [M][D] bf16 (may equal h)
 * D must be a multiple of 256 and at most 2048 (G4_ERR_UNSUPPORTED): the
 * norm's row sum is formed by one thread-block cluster of D / 256 CTAs.
 * Accumulation and the norm in float32; out rounded to nearest even.
 */
g4_status g4_attn_out_residual(const void* ao, int32_t M, int32_t K, const void* w_o, int32_t D,
                               const float* post_norm_w, float eps, const void* h, void* out, void* stream);

/*
 * Bytes of device scratch built into the library for g4_attn_decode_noalloc
 * (8 MiB).  Every GPU that loads the library holds this array until the
 * process exits.
 */
#define G4_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

/*
 * g4_attn_decode without a workspace argument, for callers that cannot
 * allocate device memory: code that is handed only its input and output
 * buffers (a plugin or custom op inside a host framework that owns every
 * allocation), or a serving loop that must not call cudaMalloc because it
 * synchronises the device and can fail mid-request.  (The pages have no
 * counterpart: this is an interface choice of this library.)
 *
 * Arguments, results and error codes are those of g4_attn_decode; the
 * split-KV partials go to a fixed array of G4_NOALLOC_SCRATCH_BYTES inside
 * the library instead of a caller's workspace.  A call whose split plan
 * (g4_attn_decode_workspace_size) exceeds that size returns
 * G4_ERR_WORKSPACE and launches nothing.  The call allocates nothing.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls share the one array and it keeps the last call's
 * contents; each call clears the part that must start at zero (the splits'
 * arrival counters, an asynchronous memset on `stream`) once its arguments
 * have passed every check, just before its launch, so a refused call writes
 * nothing.  Calls whose kernels overlap on the GPU (different streams, or
 * several threads) race on the array and must be serialised by the caller.
 */
g4_status g4_attn_decode_noalloc(const g4_layer_params* params, const g4_kv_cache* caches, int32_t n_layers,
                                 int32_t layer, const void* q, const int32_t* seq_lens, int32_t B,
                                 int32_t max_seq_len, void* out, void* stream);

/* Thread-local message of the last non-OK status ("" if none). */
const char* g4_last_error(void);

/*
 * Reads and clears the device-side error word (synchronises the device).
 * Nonzero means a kernel gave up a bounded wait (code 1), or found its
 * shared memory not 1024-byte aligned (code 2, the tensor-core prefill needs
 * that for its swizzled tiles), and returned early; its outputs are then
 * unspecified.  Returns -1 if the read itself failed.
 */
int32_t g4_take_device_error(void);

#ifdef __cplusplus
}
#endif

#endif /* G4ATTN_H */

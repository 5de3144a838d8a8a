// Step a4: fused per-head RMSNorm -> rotate_half RoPE -> KV-cache append.
//
// cortiq-engine g4e.rs `g4e_forward` (attention block): q heads are normed
// with q_norm and roped; on a layer that owns its cache, k heads are normed
// with k_norm and roped, v heads get the weight-less norm (`rms_plain`), and
// both are appended at the token's position.  ferrox-models
// gemma4_engine.rs `forward_token_on_worker` does the same per head
// (`rms_norm_per_head`, `apply_rope`, `cache.push`).  turbospark-runtime
// gemma4/attn.rs writes the projections straight into the cache slot and
// norms/ropes them there, which is the fusion done here.
//
// One CTA (4 warps) per token handles rows_per_cta of its H + 2*Hkv head
// rows; one warp per head row.  The token's cos/sin table (head_dim / 2
// pairs, double-float) is built once per CTA from angle = pos * inv_freq[j]
// with inv_freq a float32 table.  Pairs j >= n_rot (zero inv_freq) are left
// unrotated, so those dims are the normed input.  bf16 stores are the
// correctly rounded real results (g4_normrope.cuh).
//
// Lane l of a warp owns elements [l*E, l*E + E) of the lower half and the
// same offsets of the upper half (E = head_dim / 64), so each rotate_half
// pair (j, j + head_dim/2) sits in one lane.
#include "g4_device.cuh"
#include "g4_internal.h"
#include "g4_normrope.cuh"

namespace g4 {
namespace {

template <typename T, int HD>
__global__ void __launch_bounds__(128) append_normrope_kernel(const __grid_constant__ AppendArgs a) {
  constexpr int HALF = HD / 2;
  constexpr int E = HD / 64;
  constexpr bool kBF16 = sizeof(T) == 2;
  __shared__ DF s_cos[HALF];
  __shared__ DF s_sin[HALF];

  pdl_wait();
  pdl_trigger();
  const int tok = blockIdx.x;  // b * T + t
  const int b = tok / a.T;
  const int pos = a.positions[tok];

  for (int j = threadIdx.x; j < HALF; j += blockDim.x) {
    DF c = {1.0f, 0.0f}, s = {0.0f, 0.0f};
    if (j < a.n_rot) sincos_df(pos, a.inv_freq[j], c, s);
    s_cos[j] = c;
    s_sin[j] = s;
  }
  __syncthreads();

  const bool owns = a.k_in != nullptr;
  const int nrows = a.H + (owns ? 2 * a.Hkv : 0);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row0 = blockIdx.y * a.rows_per_cta;
  const int row1 = min(nrows, row0 + a.rows_per_cta);
  const bool pos_ok = pos >= 0 && pos < a.max_len;

  for (int row = row0 + warp; row < row1; row += 4) {
    const T* src;
    T* dst;
    const float* w;
    bool rope;
    if (row < a.H) {  // q head
      const size_t off = (static_cast<size_t>(tok) * a.H + row) * HD;
      src = static_cast<const T*>(a.q_in) + off;
      dst = static_cast<T*>(a.q_out) + off;
      w = a.q_w;
      rope = true;
    } else {
      const bool is_k = row < a.H + a.Hkv;
      const int kvh = is_k ? row - a.H : row - a.H - a.Hkv;
      if (!pos_ok) continue;
      src = static_cast<const T*>(is_k ? a.k_in : a.v_in) + (static_cast<size_t>(tok) * a.Hkv + kvh) * HD;
      dst = static_cast<T*>(is_k ? a.cache_k : a.cache_v) +
            ((static_cast<size_t>(b) * a.Hkv + kvh) * a.max_len + pos) * HD;
      w = is_k ? a.k_w : nullptr;
      rope = is_k;
    }
    float x[2 * E], wl[E], wh[E];
    load_elems<E>(src + lane * E, x);
    load_elems<E>(src + HALF + lane * E, x + E);
    if (w != nullptr) {
      load_elems<E>(w + lane * E, wl);
      load_elems<E>(w + HALF + lane * E, wh);
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) wl[i] = wh[i] = 1.0f;
    }
    const DF r = inv_rms_df(row_sumsq_df<2 * E>(x), HD, a.eps);
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const int j = lane * E + i;
      const bool rot = rope && j < a.n_rot;
      normrope_pair<kBF16>(x[i], wl[i], x[E + i], wh[i], r, rot, s_cos[j], s_sin[j], x[i], x[E + i]);
    }
    store_elems<E>(dst + lane * E, x);
    store_elems<E>(dst + HALF + lane * E, x + E);
  }
}

template <typename Kern>
cudaError_t launch_pdl(Kern kern, dim3 grid, cudaStream_t s, const AppendArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(128);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T>
cudaError_t launch_t(const AppendArgs& a, cudaStream_t s) {
  const int nrows = a.H + (a.k_in ? 2 * a.Hkv : 0);
  dim3 grid(a.B * a.T, (nrows + a.rows_per_cta - 1) / a.rows_per_cta);
  switch (a.hd) {
    case 64: return launch_pdl(append_normrope_kernel<T, 64>, grid, s, a);
    case 128: return launch_pdl(append_normrope_kernel<T, 128>, grid, s, a);
    case 256: return launch_pdl(append_normrope_kernel<T, 256>, grid, s, a);
    case 512: return launch_pdl(append_normrope_kernel<T, 512>, grid, s, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, int dtype, cudaStream_t s) {
  return dtype == 1 ? launch_t<__nv_bfloat16>(a, s) : launch_t<float>(a, s);
}

}  // namespace g4

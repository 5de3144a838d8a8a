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
// One CTA (4 warps) handles the tokens at one t of up to tok_per_cta
// consecutive sequences, rows_per_cta of each token's H + 2*Hkv head rows;
// one warp per head row.  The cos/sin table (head_dim / 2 pairs,
// double-float) is built per distinct position from angle = pos *
// inv_freq[j] with inv_freq a float32 table.  Pairs j >= n_rot (zero inv_freq) are left
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
  constexpr float kErrY = normrope_err_y<2 * E>();
  constexpr float kErrRot = normrope_err_rot<2 * E>(kDFTrigErrUnits);
  __shared__ DF s_cos[HALF];
  __shared__ DF s_sin[HALF];

  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x % a.T;
  const int b0 = (blockIdx.x / a.T) * a.tok_per_cta;
  const int b1 = min(a.B, b0 + a.tok_per_cta);
  const bool owns = a.k_in != nullptr;
  const int nrows = a.H + (owns ? 2 * a.Hkv : 0);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row0 = blockIdx.y * a.rows_per_cta;
  const int row1 = min(nrows, row0 + a.rows_per_cta);
  const int nr = row1 - row0;

  auto build_table = [&](int pos) {
    for (int j = threadIdx.x; j < HALF; j += blockDim.x) {
      DF c = {1.0f, 0.0f}, s = {0.0f, 0.0f};
      if (j < a.n_rot) sincos_df(pos, a.inv_freq[j], c, s);
      s_cos[j] = c;
      s_sin[j] = s;
    }
  };

  // Where head row `row` of token (b, t) comes from and goes to.
  struct RowRef {
    const T* src;
    T* dst;
    const float* w;
    bool rope;
    bool valid;
  };
  auto row_ref = [&](int b, int row) -> RowRef {
    const int tok = b * a.T + t;
    const int pos = a.positions[tok];
    RowRef rr;
    if (row < a.H) {  // q head
      const size_t off = (static_cast<size_t>(tok) * a.H + row) * HD;
      rr.src = static_cast<const T*>(a.q_in) + off;
      rr.dst = static_cast<T*>(a.q_out) + off;
      rr.w = a.q_w;
      rr.rope = true;
      rr.valid = true;
    } else {
      const bool is_k = row < a.H + a.Hkv;
      const int kvh = is_k ? row - a.H : row - a.H - a.Hkv;
      rr.valid = pos >= 0 && pos < a.max_len;  // k / v need a cache slot
      rr.src = static_cast<const T*>(is_k ? a.k_in : a.v_in) + (static_cast<size_t>(tok) * a.Hkv + kvh) * HD;
      rr.dst = static_cast<T*>(is_k ? a.cache_k : a.cache_v) +
               ((static_cast<size_t>(b) * a.Hkv + kvh) * a.max_len + (rr.valid ? pos : 0)) * HD;
      rr.w = is_k ? a.k_w : nullptr;
      rr.rope = is_k;
    }
    return rr;
  };
  auto load_row = [&](const RowRef& rr, float* x) {
    if (!rr.valid) return;
    load_elems<E>(rr.src + lane * E, x);
    load_elems<E>(rr.src + HALF + lane * E, x + E);
  };
  auto compute_store = [&](const RowRef& rr, const float* x) {
    if (!rr.valid) return;
    float wl[E], wh[E], o[2 * E];
    if (rr.w != nullptr) {
      load_elems<E>(rr.w + lane * E, wl);
      load_elems<E>(rr.w + HALF + lane * E, wh);
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) wl[i] = wh[i] = 1.0f;
    }
    const float r = inv_rms_f32(row_sumsq_f32<2 * E>(x), HD, a.eps);
    uint32_t need = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const int j = lane * E + i;
      const bool rot = rr.rope && j < a.n_rot;
      bool na, nb;
      normrope_pair_fast(x[i], wl[i], x[E + i], wh[i], r, rot, rot ? s_cos[j].h : 1.0f, rot ? s_sin[j].h : 0.0f,
                         kErrY, kErrRot, o[i], o[E + i], na, nb);
      need |= (na ? 1u : 0u) << i;
      need |= (nb ? 1u : 0u) << (E + i);
    }
    if constexpr (kBF16) {
      if (__any_sync(0xffffffffu, need != 0)) {
        // Some value of this row lies too close to a bf16 rounding boundary
        // for the float32 evaluation; decide it in double-float.
        const DF rd = inv_rms_df(row_sumsq_df<2 * E>(x), HD, a.eps);
#pragma unroll
        for (int i = 0; i < E; ++i) {
          const int j = lane * E + i;
          const bool rot = rr.rope && j < a.n_rot;
          if (need & (1u << i)) o[i] = normrope_exact_bf16(x[i], wl[i], x[E + i], wh[i], rd, rot, true, s_cos[j], s_sin[j]);
          if (need & (1u << (E + i)))
            o[E + i] = normrope_exact_bf16(x[E + i], wh[i], x[i], wl[i], rd, rot, false, s_cos[j], s_sin[j]);
        }
      }
    }
    store_elems<E>(rr.dst + lane * E, o);
    store_elems<E>(rr.dst + HALF + lane * E, o + E);
  };

  // One cos/sin table serves every token of the CTA when their positions
  // agree (the usual prefill case); otherwise tokens go one at a time.
  const int p0 = a.positions[b0 * a.T + t];
  bool same = true;
  for (int b = b0 + 1; b < b1; ++b) same = same && a.positions[b * a.T + t] == p0;
  if (same) {
    build_table(p0);
    __syncthreads();
    for (int idx = warp; idx < (b1 - b0) * nr; idx += 4) {
      const RowRef rr = row_ref(b0 + idx / nr, row0 + idx % nr);
      float x[2 * E];
      load_row(rr, x);
      compute_store(rr, x);
    }
  } else {
    for (int b = b0; b < b1; ++b) {
      if (b > b0) __syncthreads();
      build_table(a.positions[b * a.T + t]);
      __syncthreads();
      for (int row = row0 + warp; row < row1; row += 4) {
        const RowRef rr = row_ref(b, row);
        float x[2 * E];
        load_row(rr, x);
        compute_store(rr, x);
      }
    }
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
  dim3 grid(a.T * ((a.B + a.tok_per_cta - 1) / a.tok_per_cta), (nrows + a.rows_per_cta - 1) / a.rows_per_cta);
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

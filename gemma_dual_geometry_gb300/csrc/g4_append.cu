// Step a4: fused per-head RMSNorm -> rotate_half RoPE -> KV-cache append.
//
// cortiq-engine g4e.rs `g4e_forward` (attention block): q heads are normed
// with q_norm and roped; on a layer that owns its cache, k heads are normed
// with k_norm and roped, v heads get the weight-less norm (`rms_plain`), and
// both are appended at the token's position.  ferrox-models
// gemma4_engine.rs `forward_token_on_worker` does the same per head
// (`rms_norm_per_head`, `apply_rope`, `cache.push`).  turbospark-runtime
// gemma4/attn.rs writes the projections straight into the cache slot and
// norms/ropes them there, which is the fusion done here.  A token at
// position p goes to cache row p, or p mod max_len on a sliding-window ring.
//
// One CTA (4 warps) handles the tokens at one t of up to tok_per_cta
// consecutive sequences, rows_per_cta of each token's H + 2*Hkv head rows;
// one warp per head row.  The cos/sin table (head_dim / 2 pairs,
// double-float) is built per distinct position from angle = pos *
// inv_freq[j] with inv_freq a float32 table.  Pairs j >= n_rot (zero inv_freq) are left
// unrotated, so those dims are the normed input.  bf16 stores are the
// correctly rounded real results (g4_normrope.cuh), decided in three stages:
//   1. float32 for the whole row (packed float32x2 products), with Ziv's test
//      of each value against its error bound; in the synthetic workloads
//      about one row in five has a value the test leaves open;
//   2. for those values only, lane by lane: the float32 inverse rms times the
//      row's inner products in double-float, whose error is the inverse
//      rms's alone; this leaves open about one row in twenty to thirty;
//   3. the row's sum of squares in double-float (error-free splitting) and a
//      double-float inverse rms, which decide the rest.
//
// Lane l of a warp owns elements [l*E, l*E + E) of the lower half and the
// same offsets of the upper half (E = head_dim / 64), so each rotate_half
// pair (j, j + head_dim/2) sits in one lane.  Each warp loads its next row
// before it computes the current one.
#include <type_traits>

#include "g4_device.cuh"
#include "g4_internal.h"
#include "g4_normrope.cuh"

namespace g4 {
namespace {

// The bits of a lane's E consecutive elements of one half of a head row.
template <typename T, int E>
struct HalfBits;
template <int E>
struct HalfBits<float, E> {
  float v[E];
};
template <int E>
struct HalfBits<__nv_bfloat16, E> {
  uint32_t v[(E + 1) / 2];
};

template <int E>
__device__ __forceinline__ void load_bits(const float* p, HalfBits<float, E>& h) {
  load_elems<E>(p, h.v);
}
template <int E>
__device__ __forceinline__ void load_bits(const __nv_bfloat16* p, HalfBits<__nv_bfloat16, E>& h) {
  if constexpr (E == 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    h.v[0] = v.x; h.v[1] = v.y; h.v[2] = v.z; h.v[3] = v.w;
  } else if constexpr (E == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    h.v[0] = v.x; h.v[1] = v.y;
  } else if constexpr (E == 2) {
    h.v[0] = *reinterpret_cast<const uint32_t*>(p);
  } else {
    h.v[0] = *reinterpret_cast<const uint16_t*>(p);
  }
}

template <int E>
__device__ __forceinline__ void unpack_bits(const HalfBits<float, E>& h, float* x) {
#pragma unroll
  for (int i = 0; i < E; ++i) x[i] = h.v[i];
}
template <int E>
__device__ __forceinline__ void unpack_bits(const HalfBits<__nv_bfloat16, E>& h, float* x) {
  if constexpr (E == 1) {
    x[0] = bf16_lo(h.v[0]);
  } else {
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
      x[2 * i] = bf16_lo(h.v[i]);
      x[2 * i + 1] = bf16_hi(h.v[i]);
    }
  }
}

// y = (x * r) * w elementwise (w == nullptr: y = x * r), two elements per
// packed float32x2 instruction; each product is rounded as its own float op.
template <int E>
__device__ __forceinline__ void scale_elems(float* y, const float* x, float r, const float* w) {
  if constexpr (E % 2 == 0) {
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      float2 t = __fmul2_rn(make_float2(x[i], x[i + 1]), make_float2(r, r));
      if (w != nullptr) t = __fmul2_rn(t, make_float2(w[i], w[i + 1]));
      y[i] = t.x;
      y[i + 1] = t.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) y[i] = w != nullptr ? (x[i] * r) * w[i] : x[i] * r;
  }
}

// rotate_half on the lane's pairs: oa = ya c - yb s, ob = yb c + ya s, each
// as one fma over one rounded product.
template <int E>
__device__ __forceinline__ void rotate_elems(float* oa, float* ob, const float* ya, const float* yb, const float* c,
                                             const float* s) {
  if constexpr (E % 2 == 0) {
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      const float2 a2 = make_float2(ya[i], ya[i + 1]);
      const float2 b2 = make_float2(yb[i], yb[i + 1]);
      const float2 c2 = make_float2(c[i], c[i + 1]);
      const float2 ra = __ffma2_rn(a2, c2, __fmul2_rn(b2, make_float2(-s[i], -s[i + 1])));
      const float2 rb = __ffma2_rn(b2, c2, __fmul2_rn(a2, make_float2(s[i], s[i + 1])));
      oa[i] = ra.x; oa[i + 1] = ra.y;
      ob[i] = rb.x; ob[i + 1] = rb.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      oa[i] = fmaf(ya[i], c[i], yb[i] * -s[i]);
      ob[i] = fmaf(yb[i], c[i], ya[i] * s[i]);
    }
  }
}

// True when no bf16 rounding boundary lies within e of v (so v's own bf16
// rounding is that of every value within e of it).
__device__ __forceinline__ bool bf16_decided(float v, float e) { return fabsf(v - bf16_midpoint(v)) > e; }

template <typename T, int HD>
__global__ void __launch_bounds__(128, HD >= 512 ? 5 : 8) append_normrope_kernel(const __grid_constant__ AppendArgs a) {
  constexpr int HALF = HD / 2;
  constexpr int E = HD / 64;
  constexpr bool kBF16 = sizeof(T) == 2;
  constexpr float kErrY = normrope_err_y<2 * E>();
  constexpr float kErrAB = normrope_err_pair(kDFTrigErrUnits);
  constexpr float kErrO = normrope_err_out<2 * E>();
  constexpr float kErrR = normrope_err_r<2 * E>();
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
  if (nr <= 0) return;

  // Error-bound multipliers of this lane's outputs on a roped row (bound =
  // kA |y_self| + kB |y_other| + kO |o|): the rotation bound where the lane's
  // pairs rotate, the plain one where none does.  A lane straddling n_rot
  // takes the rotation bound for all its pairs, which also covers the plain ones.
  const bool lane_plain = lane * E >= a.n_rot;
  const float kA = lane_plain ? kErrY : kErrAB;
  const float kB = lane_plain ? 0.0f : kErrAB;
  const float kO = lane_plain ? 0.0f : kErrO;
  const bool all_rot = __all_sync(0xffffffffu, (lane + 1) * E <= a.n_rot);

  // This lane's cos / sin (float parts; 1 / 0 past n_rot), built per position.
  float cr[E], sr[E];
  auto build_table = [&](int pos) {
    for (int j = threadIdx.x; j < HALF; j += blockDim.x) {
      DF c = {1.0f, 0.0f}, s = {0.0f, 0.0f};
      if (j < a.n_rot) sincos_df(pos, a.inv_freq[j], c, s);
      s_cos[j] = c;
      s_sin[j] = s;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < E; ++i) {
      cr[i] = s_cos[lane * E + i].h;
      sr[i] = s_sin[lane * E + i].h;
    }
  };

  // Where head row `row` of token (b, t) at position pos comes from and goes to.
  struct RowRef {
    const T* src;
    T* dst;
    const float* w;
    bool rope;
    bool valid;
  };
  auto row_ref = [&](int b, int row, int pos) -> RowRef {
    const int tok = b * a.T + t;
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
      // k / v need a cache row: the position itself, or on a sliding-window
      // ring the position modulo its capacity.
      rr.valid = pos >= 0 && (a.ring || pos < a.max_len);
      const int crow = !rr.valid ? 0 : (a.ring ? pos % a.max_len : pos);
      rr.src = static_cast<const T*>(is_k ? a.k_in : a.v_in) + (static_cast<size_t>(tok) * a.Hkv + kvh) * HD;
      rr.dst = static_cast<T*>(is_k ? a.cache_k : a.cache_v) +
               ((static_cast<size_t>(b) * a.Hkv + kvh) * a.max_len + crow) * HD;
      rr.w = is_k ? a.k_w : nullptr;
      rr.rope = is_k;
    }
    return rr;
  };
  auto load_row = [&](const RowRef& rr, HalfBits<T, E>& lo, HalfBits<T, E>& hi) {
    if (!rr.valid) return;
    load_bits<E>(rr.src + lane * E, lo);
    load_bits<E>(rr.src + HALF + lane * E, hi);
  };

  // Values of row rr that the float32 evaluation could not decide (bit k of
  // need: element k of the lane's 2E, lower half first), evaluated again in
  // double-float from the row's inverse rms rd and stored over the fast ones.
  // One element per pass, so the loop stays short for the usual 0-2 bits.
  auto fix_elems = [&](const RowRef& rr, uint32_t need, DF rd) {
#pragma unroll 1
    while (need != 0) {
      const int k = __ffs(need) - 1;
      need &= need - 1;
      const bool lower = k < E;
      const int j = lane * E + (lower ? k : k - E);
      const int self = lower ? j : HALF + j, other = lower ? HALF + j : j;
      const float xs = static_cast<float>(rr.src[self]);
      float v;
      if (rr.rope) {
        const float xo = static_cast<float>(rr.src[other]);
        const float ws = rr.w != nullptr ? rr.w[self] : 1.0f, wo = rr.w != nullptr ? rr.w[other] : 1.0f;
        v = normrope_exact_bf16_inl(xs, ws, xo, wo, rd, j < a.n_rot, lower, s_cos[j], s_sin[j]);
      } else {
        v = df_round_bf16(df_mul_f(rd, xs));
      }
      rr.dst[self] = static_cast<T>(v);
    }
  };

  // Second stage for the values of row rr the float32 evaluation left open
  // (bits of need, as for fix_elems): the same float inverse rms r times the
  // row's inner products in double-float.  That value is off from the exact
  // one by r's own error (and 2^-40 of the terms), much less than the float32
  // evaluation, so it decides most of them; the bits still open are returned.
  auto refine = [&](const RowRef& rr, uint32_t need, float r) -> uint32_t {
    uint32_t open = 0;
#pragma unroll 1
    while (need != 0) {
      const int k = __ffs(need) - 1;
      need &= need - 1;
      const bool lower = k < E;
      const int j = lane * E + (lower ? k : k - E);
      const int self = lower ? j : HALF + j, other = lower ? HALF + j : j;
      const float xs = static_cast<float>(rr.src[self]);
      DF inner = {xs, 0.0f};
      float mag = fabsf(xs);
      if (rr.rope) {
        const float ws = rr.w != nullptr ? rr.w[self] : 1.0f;
        inner = two_prod(xs, ws);
        mag = fabsf(inner.h);
        if (j < a.n_rot) {
          const float xo = static_cast<float>(rr.src[other]);
          const float wo = rr.w != nullptr ? rr.w[other] : 1.0f;
          const DF po = two_prod(xo, wo);
          mag += fabsf(po.h);
          inner = df_add(df_mul(inner, s_cos[j]), df_mul(po, lower ? df_neg(s_sin[j]) : s_sin[j]));
        }
      }
      const DF v = df_mul_f(inner, r);
      const float e = fmaf(kErrR, fabsf(v.h), 0x1.0p-40f * r * mag);
      if (fabsf((v.h - bf16_midpoint(v.h)) + v.l) > e)
        rr.dst[self] = static_cast<T>(df_round_bf16(v));
      else
        open |= 1u << k;
    }
    return open;
  };

  // One row: float32 evaluation, stored.  For bf16, a value whose rounding
  // the float32 evaluation cannot decide (Ziv's test against its error bound)
  // is then decided in double-float (refine, then fix_elems).  all_rot (warp-uniform):
  // every lane's pairs rotate, so both outputs of a pair share one bound.
  auto do_row = [&](const RowRef& rr, const HalfBits<T, E>& lo, const HalfBits<T, E>& hi, auto all_rot_tag) {
    [[maybe_unused]] constexpr bool kAllRot = decltype(all_rot_tag)::value;
    if (!rr.valid) return;
    float x[2 * E], o[2 * E];
    unpack_bits<E>(lo, x);
    unpack_bits<E>(hi, x + E);
    const float sf = row_sumsq_f32<2 * E>(x);
    const float r = inv_rms_f32(sf, HD, a.eps);
    [[maybe_unused]] uint32_t need = 0;
    if (rr.rope) {
      float wl[E], wh[E], ya[E], yb[E];
      if (rr.w != nullptr) {
        load_elems<E>(rr.w + lane * E, wl);
        load_elems<E>(rr.w + HALF + lane * E, wh);
      } else {
#pragma unroll
        for (int i = 0; i < E; ++i) wl[i] = wh[i] = 1.0f;
      }
      scale_elems<E>(ya, x, r, wl);
      scale_elems<E>(yb, x + E, r, wh);
      rotate_elems<E>(o, o + E, ya, yb, cr, sr);
      if constexpr (kBF16) {
#pragma unroll
        for (int i = 0; i < E; ++i) {
          const float aa = fabsf(ya[i]), ab = fabsf(yb[i]);
          float ea, eb;
          if constexpr (kAllRot) {
            const float shared = kErrAB * (aa + ab);
            ea = fmaf(kErrO, fabsf(o[i]), shared);
            eb = fmaf(kErrO, fabsf(o[E + i]), shared);
          } else {
            ea = fmaf(kO, fabsf(o[i]), fmaf(kB, ab, kA * aa));
            eb = fmaf(kO, fabsf(o[E + i]), fmaf(kB, aa, kA * ab));
          }
          need |= (bf16_decided(o[i], ea) ? 0u : 1u) << i;
          need |= (bf16_decided(o[E + i], eb) ? 0u : 1u) << (E + i);
        }
      }
    } else {  // v head: weight-less norm, no rotation
      scale_elems<E>(o, x, r, nullptr);
      scale_elems<E>(o + E, x + E, r, nullptr);
      if constexpr (kBF16) {
#pragma unroll
        for (int k = 0; k < 2 * E; ++k) need |= (bf16_decided(o[k], kErrY * fabsf(o[k])) ? 0u : 1u) << k;
      }
    }
    store_elems<E>(rr.dst + lane * E, o);
    store_elems<E>(rr.dst + HALF + lane * E, o + E);
    if constexpr (kBF16) {
      if (__any_sync(0xffffffffu, need != 0)) {
        need = refine(rr, need, r);
        if (__any_sync(0xffffffffu, need != 0))
          fix_elems(rr, need, inv_rms_df(row_sumsq_split<2 * E, HD>(x, sf), HD, a.eps));
      }
    }
  };

  // Rows of tokens [bA, bB) (all at position pos), flattened in (b, row)
  // order; warp w takes items w, w + 4, ...  The next item's loads are issued
  // before the current one is computed.
  auto run = [&](int bA, int bB, int pos) {
    int b = bA, row = row0 + warp;
    while (row >= row1 && b < bB) { row -= nr; ++b; }
    RowRef rr = {};
    HalfBits<T, E> lo, hi;
    if (b < bB) {
      rr = row_ref(b, row, pos);
      load_row(rr, lo, hi);
    }
    while (b < bB) {
      int bn = b, rn = row + 4;
      while (rn >= row1 && bn < bB) { rn -= nr; ++bn; }
      RowRef rrn = {};
      HalfBits<T, E> lon, hin;
      if (bn < bB) {
        rrn = row_ref(bn, rn, pos);
        load_row(rrn, lon, hin);
      }
      if (all_rot)
        do_row(rr, lo, hi, std::true_type());
      else
        do_row(rr, lo, hi, std::false_type());
      b = bn;
      row = rn;
      rr = rrn;
      lo = lon;
      hi = hin;
    }
  };

  // One cos/sin table serves every token of the CTA when their positions
  // agree (the usual prefill case); otherwise tokens go one at a time.
  const int p0 = a.positions[b0 * a.T + t];
  bool same = true;
  for (int b = b0 + 1; b < b1; ++b) same = same && a.positions[b * a.T + t] == p0;
  if (same) {
    build_table(p0);
    run(b0, b1, p0);
  } else {
    for (int b = b0; b < b1; ++b) {
      if (b > b0) __syncthreads();  // every warp is done with the previous table
      const int pos = a.positions[b * a.T + t];
      build_table(pos);
      run(b, b + 1, pos);
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

// Per-head RMSNorm + rotate_half RoPE of one element pair, with the bf16
// stored value rounded correctly from the real-number result.
//
// What is computed (cortiq-engine g4e.rs `rms` / `rms_plain`, taconite
// model.rs `rope_half`): for a head row x of width hd with weight w,
//   y_d  = x_d * (mean(x^2) + eps)^(-1/2) * w_d          (w = 1 for V)
//   y'_j = y_j cos(p f_j) - y_{j+hd/2} sin(p f_j)
//   y'_{j+hd/2} = y_{j+hd/2} cos(p f_j) + y_j sin(p f_j)  for j < n_rot
// with f_j the float32 inverse frequency and p the token position.
//
// Storing y' as bf16 is a rounding decision, and a one-ulp difference in a
// stored q or k moves a score of a scale-1.0 softmax enough to change an
// attention output by more than its own rounding.  So the stored bf16 value
// is the round-to-nearest-even of the exact result:
//   * a float32 evaluation runs first, with a bound on its error; when no
//     bf16 rounding boundary lies within that bound of the float32 value, its
//     rounding is the correct one (Ziv's rounding test);
//   * otherwise a double-float evaluation decides: values carried as an
//     unevaluated sum of two floats, built from Dekker's exact product (one
//     fma) and Knuth's two-sum, accurate to about 2^-44 relative.  It runs
//     for about one element in a thousand (rotated values whose two terms
//     nearly cancel make up most of them).
// cos / sin in double-float come from an exact p * f, Cody-Waite reduction
// by a three-float pi/2 and Taylor polynomials on [-pi/4, pi/4].
#pragma once

#include "g4_device.cuh"

namespace g4 {

// h + l with |l| <= ulp(h) / 2.
struct DF {
  float h, l;
};

// a + b = s + e exactly (Knuth).
__device__ __forceinline__ DF two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  return {s, (a - (s - bb)) + (b - bb)};
}

// a + b = s + e exactly when |a| >= |b| or a == 0 (Dekker).
__device__ __forceinline__ DF fast_two_sum(float a, float b) {
  const float s = a + b;
  return {s, b - (s - a)};
}

// a * b = p + e exactly (the fma returns the product's rounding error).
__device__ __forceinline__ DF two_prod(float a, float b) {
  const float p = a * b;
  return {p, fmaf(a, b, -p)};
}

__device__ __forceinline__ DF df_add(DF a, DF b) {
  const DF s = two_sum(a.h, b.h);
  return fast_two_sum(s.h, s.l + (a.l + b.l));
}

__device__ __forceinline__ DF df_add_f(DF a, float b) {
  const DF s = two_sum(a.h, b);
  return fast_two_sum(s.h, s.l + a.l);
}

__device__ __forceinline__ DF df_mul(DF a, DF b) {
  const DF p = two_prod(a.h, b.h);
  return fast_two_sum(p.h, fmaf(a.h, b.l, fmaf(a.l, b.h, p.l)));
}

__device__ __forceinline__ DF df_mul_f(DF a, float b) {
  const DF p = two_prod(a.h, b);
  return fast_two_sum(p.h, fmaf(a.l, b, p.l));
}

__device__ __forceinline__ DF df_neg(DF a) { return {-a.h, -a.l}; }

// The exact bf16 round-to-nearest-even of h + l, returned as a float.
__device__ __forceinline__ float df_round_bf16(DF v) {
  const uint32_t b = __float_as_uint(v.h);
  if ((b & 0xFFFFu) == 0x8000u && v.l != 0.0f) {
    // h sits exactly on a bf16 midpoint: the sign of l decides.
    const bool away = (v.l > 0.0f) == (v.h > 0.0f);
    return __uint_as_float((b & 0xFFFF0000u) + (away ? 0x10000u : 0u));
  }
  return __bfloat162float(__float2bfloat16_rn(v.h));
}

// The bf16 rounding boundary of v's bf16 interval (same sign and binade as v,
// so v - mid is exact).
__device__ __forceinline__ float bf16_midpoint(float v) {
  return __uint_as_float((__float_as_uint(v) & 0xFFFF0000u) | 0x8000u);
}

constexpr int ilog2c(int x) { return x <= 1 ? 0 : 1 + ilog2c(x / 2); }

// Row sum of squares in float32: pairwise over the lane's N elements, then
// the 32-lane butterfly (every lane ends with the same value).  Relative
// error at most (log2 N + 5) u, u = 2^-24.
template <int N>
__device__ __forceinline__ float row_sumsq_f32(const float* x) {
  float v[N];
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = x[i] * x[i];
#pragma unroll
  for (int w = N / 2; w >= 1; w /= 2)
#pragma unroll
    for (int i = 0; i < w; ++i) v[i] += v[i + w];
  float s = v[0];
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// Bound, in units of u, on the relative error of y = fl(fl(x r) w) with
// r = rsqrt_rn(fl(S / hd + eps)) and S from row_sumsq_f32<N>: the sum, the
// eps addition (halved by the root), the correctly rounded root, two products.
template <int N>
constexpr float norm_err_units() {
  return (ilog2c(N) + 6) * 0.5f + 3.0f;
}

// Row sum of squares in double-float over the lane's n elements, then over
// the 32 lanes of the warp (every lane ends with the same value).
template <int N>
__device__ __forceinline__ DF row_sumsq_df(const float* x) {
  float hi = 0.0f, lo = 0.0f;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const DF p = two_prod(x[i], x[i]);
    const DF t = two_sum(hi, p.h);
    hi = t.h;
    lo += t.l + p.l;
  }
  DF s = fast_two_sum(hi, lo);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const DF t = {__shfl_xor_sync(0xffffffffu, s.h, o), __shfl_xor_sync(0xffffffffu, s.l, o)};
    s = df_add(s, t);  // symmetric in its arguments, so all lanes agree
  }
  return s;
}

// The same row sum in double-float, cheaper, for rows whose squares are exact
// in float (bf16 elements) and whose float32 sum sf (row_sumsq_f32) is known.
// Two error-free splittings against powers of two (Rump, Ogita and Oishi's
// ExtractScalar): each square p = q1 + q2 + p2 exactly, q1 a multiple of
// ulp(s1), q2 of ulp(s2) / 2, with s1 >= 2 sf and s2 = s1 2^(log2 HD - 23).
// Every partial sum of the q1 (and of the q2) is then exact in float, and the
// p2 are small enough (|p2| <= s2 2^-24) that their float sum is off by less
// than 2^-46 of the row sum.  Rows outside [2^-60, 2^124) take row_sumsq_df.
template <int N, int HD>
__device__ __forceinline__ DF row_sumsq_split(const float* x, float sf) {
  if (!(sf >= 0x1.0p-60f && sf < 0x1.0p+124f)) return row_sumsq_df<N>(x);
  const float s1 = __uint_as_float((__float_as_uint(sf) & 0x7F800000u) + (2u << 23));  // 2^(e+2) > 2 sf
  const float s2 = s1 * (static_cast<float>(HD) * 0x1.0p-23f);
  float a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
  if constexpr (N % 2 == 0) {
    float2 c1 = make_float2(0.0f, 0.0f), c2 = c1, c3 = c1;
    const float2 ps1 = make_float2(s1, s1), ns1 = make_float2(-s1, -s1);
    const float2 ps2 = make_float2(s2, s2), ns2 = make_float2(-s2, -s2);
    const float2 m1 = make_float2(-1.0f, -1.0f);
#pragma unroll
    for (int i = 0; i < N; i += 2) {
      const float2 v = make_float2(x[i], x[i + 1]);
      const float2 p = __fmul2_rn(v, v);
      const float2 q1 = __fadd2_rn(__fadd2_rn(ps1, p), ns1);
      const float2 r1 = __ffma2_rn(q1, m1, p);
      const float2 q2 = __fadd2_rn(__fadd2_rn(ps2, r1), ns2);
      const float2 r2 = __ffma2_rn(q2, m1, r1);
      c1 = __fadd2_rn(c1, q1);
      c2 = __fadd2_rn(c2, q2);
      c3 = __fadd2_rn(c3, r2);
    }
    a1 = c1.x + c1.y;
    a2 = c2.x + c2.y;
    a3 = c3.x + c3.y;
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const float p = x[i] * x[i];
      const float q1 = (s1 + p) - s1;
      const float r1 = p - q1;
      const float q2 = (s2 + r1) - s2;
      a1 += q1;
      a2 += q2;
      a3 += r1 - q2;
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    a1 += __shfl_xor_sync(0xffffffffu, a1, o);
    a2 += __shfl_xor_sync(0xffffffffu, a2, o);
    a3 += __shfl_xor_sync(0xffffffffu, a3, o);
  }
  return df_add_f(fast_two_sum(a1, a2), a3);
}

// (sumsq / hd + eps)^(-1/2) in double-float: one Newton step on rsqrtf.
__device__ __forceinline__ DF inv_rms_df(DF sumsq, int hd, float eps) {
  const float inv_hd = 1.0f / static_cast<float>(hd);  // hd is a power of two: exact
  const DF ms = df_add_f(DF{sumsq.h * inv_hd, sumsq.l * inv_hd}, eps);
  const float r0 = rsqrtf(ms.h);
  const DF t = df_mul(ms, two_prod(r0, r0));  // ms * r0^2, close to 1
  const float d = (1.0f - t.h) - t.l;         // 1 - t.h is exact there
  return fast_two_sum(r0, r0 * (0.5f * d));
}

// p * f (p an integer position, f a float32 frequency) reduced to r in
// [-pi/4, pi/4] (+ a rounding of k) in double-float, and its quadrant k mod 4.
__device__ __forceinline__ DF reduce_angle_df(int p, float f, int& quadrant) {
  DF r;
  if (p < (1 << 24) && p > -(1 << 24)) {
    // theta = p * f exactly (p is exact in float); k = nearest multiple of pi/2
    const DF th = two_prod(static_cast<float>(p), f);
    const float k = rintf(th.h * 0x1.45f306p-1f);  // 2 / pi
    // pi/2 = P1 + P2 + P3 (+ < 1e-23)
    constexpr float P1 = 0x1.921fb6p+0f, P2 = -0x1.777a5cp-25f, P3 = -0x1.ee59dap-50f;
    const DF a = two_prod(k, P1);
    const float r_hi = th.h - a.h;  // exact: th.h and k * P1 are within a factor of two (or k = 0)
    DF e = two_sum(th.l, -a.l);
    e = df_add(e, df_neg(two_prod(k, P2)));
    e = df_add_f(e, -k * P3);
    r = df_add_f(e, r_hi);
    quadrant = static_cast<int>(k) & 3;
  } else {
    // positions beyond float's exact integers: reduce in float64
    const double th = static_cast<double>(p) * static_cast<double>(f);
    const double k = rint(th * 0.63661977236758134308);
    const double rd = fma(-k, 1.5707963267948966192e0, th) - k * 6.123233995736766036e-17;
    r.h = static_cast<float>(rd);
    r.l = static_cast<float>(rd - static_cast<double>(r.h));
    quadrant = static_cast<int>(fmod(k, 4.0) + 4.0) & 3;
  }
  return r;
}

// The two polynomials of sincos_df on the reduced angle r (z = r^2):
// sin r = r + r z S(z) and cos r = 1 - z/2 + z^2 C(z), with the Taylor
// coefficients 1/n! in double-float and the tail (< 2^-30 of the result) in float.
__device__ __forceinline__ DF sin_poly_df(DF r, DF z) {
  const float zh = z.h;
  // S(z) = -1/3! + z/5! - z^2/7! + z^3/9! - z^4/11! + z^5/13! - z^6/15!
  float ts = fmaf(zh, -0x1.ae7f3ep-41f, 0x1.612462p-33f);
  ts = fmaf(zh, ts, -0x1.ae6456p-26f);
  DF S = df_add(df_mul_f(z, ts), DF{0x1.71de3ap-19f, 0x1.55b1ccp-45f});
  S = df_add(df_mul(z, S), DF{-0x1.a01a02p-13f, 0x1.7f97fap-39f});
  S = df_add(df_mul(z, S), DF{0x1.111112p-7f, -0x1.dddddep-32f});
  S = df_add(df_mul(z, S), DF{-0x1.555556p-3f, 0x1.555556p-28f});
  return df_add(r, df_mul(df_mul(r, z), S));
}
__device__ __forceinline__ DF cos_poly_df(DF z) {
  const float zh = z.h;
  // C(z) = 1/4! - z/6! + z^2/8! - z^3/10! + z^4/12! - z^5/14! + z^6/16!
  float tc = fmaf(zh, 0x1.ae7f3ep-45f, -0x1.93974ap-37f);
  tc = fmaf(zh, tc, 0x1.1eed8ep-29f);
  DF Cz = df_add(df_mul_f(z, tc), DF{-0x1.27e4fcp-22f, 0x1.10ec14p-47f});
  Cz = df_add(df_mul(z, Cz), DF{0x1.a01a02p-16f, -0x1.7f97fap-42f});
  Cz = df_add(df_mul(z, Cz), DF{-0x1.6c16c2p-10f, 0x1.27d27ep-35f});
  Cz = df_add(df_mul(z, Cz), DF{0x1.555556p-5f, -0x1.555556p-30f});
  return df_add(df_add_f(DF{-0.5f * z.h, -0.5f * z.l}, 1.0f), df_mul(df_mul(z, z), Cz));
}

// cos and sin of p * f in double-float (absolute error about 2^-47).
__device__ __forceinline__ void sincos_df(int p, float f, DF& c_out, DF& s_out) {
  int quadrant;
  const DF r = reduce_angle_df(p, f, quadrant);
  const DF z = df_mul(r, r);
  const DF sn = sin_poly_df(r, z);
  const DF cs = cos_poly_df(z);
  // theta = k pi/2 + r
  switch (quadrant) {
    case 0: c_out = cs; s_out = sn; break;
    case 1: c_out = df_neg(sn); s_out = cs; break;
    case 2: c_out = df_neg(cs); s_out = df_neg(sn); break;
    default: c_out = sn; s_out = df_neg(cs); break;
  }
}

// Half of sincos_df, for two threads sharing one angle: part 0 evaluates the
// cosine polynomial, part 1 the sine one; the result is cos (p f) when
// to_cos is set on return, else sin (p f).  Same values as sincos_df.
__device__ __forceinline__ DF sincos_df_part(int p, float f, int part, bool& to_cos) {
  int quadrant;
  const DF r = reduce_angle_df(p, f, quadrant);
  const DF z = df_mul(r, r);
  const DF v = part == 0 ? cos_poly_df(z) : sin_poly_df(r, z);
  // cos poly: cos for quadrants 0 (+), 2 (-); sin for 1 (+), 3 (-).
  // sin poly: sin for quadrants 0 (+), 2 (-); cos for 1 (-), 3 (+).
  to_cos = (part == 0) == ((quadrant & 1) == 0);
  const bool neg = part == 0 ? quadrant >= 2 : (quadrant == 1 || quadrant == 2);
  return neg ? df_neg(v) : v;
}

// Error of a double-float table's float part: at most u (+ 2^-47).
constexpr float kDFTrigErrUnits = 1.0f;

// Exact value of one output of a pair, rounded to bf16: y_self * c +- y_other
// * s on a rotated pair (sign - for the lower element), else y_self.
__device__ __forceinline__ float normrope_exact_bf16_inl(float x_self, float w_self, float x_other, float w_other, DF r,
                                                         bool rot, bool lower, DF c, DF s) {
  const DF ys = df_mul_f(df_mul_f(r, x_self), w_self);
  if (!rot) return df_round_bf16(ys);
  const DF yo = df_mul_f(df_mul_f(r, x_other), w_other);
  return df_round_bf16(df_add(df_mul(ys, c), df_mul(yo, lower ? df_neg(s) : s)));
}
static __device__ __noinline__ float normrope_exact_bf16(float x_self, float w_self, float x_other, float w_other, DF r,
                                                         bool rot, bool lower, DF c, DF s) {
  return normrope_exact_bf16_inl(x_self, w_self, x_other, w_other, r, rot, lower, c, s);
}

// Float32 evaluation of one pair (lower a = element j, upper b = element
// j + hd/2) with row inverse rms r, cos / sin c, s.  Sets need_a / need_b
// when the float32 value cannot decide the bf16 rounding.  Bounds: err_y |y|
// for an unrotated output; err_ab (|ya| + |yb|) + err_o |o| for a rotated one
// (normrope_err_pair, normrope_err_out).
__device__ __forceinline__ void normrope_pair_fast(float xa, float wa, float xb, float wb, float r, bool rot, float c,
                                                   float s, float err_y, float err_ab, float err_o, float& oa,
                                                   float& ob, bool& need_a, bool& need_b) {
  const float ya = (xa * r) * wa;
  const float yb = (xb * r) * wb;
  float ea, eb;
  if (rot) {
    oa = fmaf(ya, c, -(yb * s));
    ob = fmaf(yb, c, ya * s);
    const float shared = err_ab * (fabsf(ya) + fabsf(yb));
    ea = fmaf(err_o, fabsf(oa), shared);
    eb = fmaf(err_o, fabsf(ob), shared);
  } else {
    oa = ya;
    ob = yb;
    ea = err_y * fabsf(ya);
    eb = err_y * fabsf(yb);
  }
  need_a = !(fabsf(oa - bf16_midpoint(oa)) > ea);
  need_b = !(fabsf(ob - bf16_midpoint(ob)) > eb);
}

// Bounds for normrope_pair_fast with N elements per lane and the cos / sin
// error trig_units.  To first order the error of a plain output is
// norm_err_units u |y|; that of a rotated one, ya c - yb s with c, s off by
// trig_units u relative, the product yb s and the fma each rounded once, is
// at most (norm_err_units + trig_units + 2) u (|ya c| + |yb s|), so (as
// |c|, |s| <= 1) at most that times |ya| + |yb|.  The factor 1 + 2^-4 covers the second-order terms (below 2^-40
// relative), the rounding of the bound itself and |y| standing for the exact
// normed value (both below 2^-19 relative).
constexpr float kBoundMargin = 1.0625f;
template <int N>
constexpr float normrope_err_y() {
  return kBoundMargin * norm_err_units<N>() * 0x1.0p-24f;
}
template <int N>
constexpr float normrope_err_rot(float trig_units) {
  return kBoundMargin * (norm_err_units<N>() + trig_units + 2.0f) * 0x1.0p-24f;
}

// A sharper bound for a rotated output, split by where the error comes from.
// With r_f the float32 inverse rms as computed, let O' = r_f (xa wa c - xb wb
// s) in exact arithmetic.  The float32 evaluation is within (3 + trig_units) u
// (|ya| + |yb|) of O' (two roundings in each y, the table's cos / sin, the
// product yb s) plus u |o| (the fma); O' is within (norm_err_units - 2) u |o|
// of the exact value, r_f's own relative error being the sum's, the eps
// addition's and the root's.  So the bound is
//   normrope_err_pair * (|ya| + |yb|) + normrope_err_out * |o|,
// never above normrope_err_rot * (|ya| + |yb|) and about half of it on average.
constexpr float normrope_err_pair(float trig_units) { return kBoundMargin * (3.0f + trig_units) * 0x1.0p-24f; }
template <int N>
constexpr float normrope_err_out() {
  return kBoundMargin * (norm_err_units<N>() - 1.0f) * 0x1.0p-24f;
}
// Bound (times |o|) on the error of r_f times an inner product evaluated in
// double-float: r_f's relative error alone.
template <int N>
constexpr float normrope_err_r() {
  return kBoundMargin * (norm_err_units<N>() - 2.0f) * 0x1.0p-24f;
}

// Inverse rms of a row in float32 (all lanes), from row_sumsq_f32.
__device__ __forceinline__ float inv_rms_f32(float sumsq, int hd, float eps) {
  return __frsqrt_rn(fmaf(sumsq, 1.0f / static_cast<float>(hd), eps));
}

// ---------------------------------------------------------------- whole rows
// A head row held by one warp: lane l owns pieces l + 32c (c < NPC) of PE
// consecutive elements (16-byte pieces where the row is wide enough).

// Lane l's elements of a row: pieces l + 32c (c < NPC) of PE elements.
template <typename T, int NPC, int PE>
__device__ __forceinline__ void load_row(const T* row, int lane, float* f) {
#pragma unroll
  for (int c = 0; c < NPC; ++c) load_elems<PE>(row + (lane + 32 * c) * PE, f + c * PE);
}

template <typename T, int NPC, int PE>
__device__ __forceinline__ void store_row(T* row, int lane, const float* f) {
#pragma unroll
  for (int c = 0; c < NPC; ++c) store_elems<PE>(row + (lane + 32 * c) * PE, f + c * PE);
}

template <int N>
__device__ __forceinline__ void to_f2(const float* f, float2 (&x)[N / 2]) {
#pragma unroll
  for (int i = 0; i < N / 2; ++i) x[i] = make_float2(f[2 * i], f[2 * i + 1]);
}

template <typename T, int NPC, int PE>
__device__ __forceinline__ void load_row_f2(const T* row, int lane, float2 (&x)[NPC * PE / 2]) {
  float f[NPC * PE];
  load_row<T, NPC, PE>(row, lane, f);
  to_f2<NPC * PE>(f, x);
}

// Round through the storage type (what a stored row would hold).
template <typename T>
__device__ __forceinline__ float through(float x) {
  if constexpr (sizeof(T) == 2) {
    return __bfloat162float(__float2bfloat16_rn(x));
  } else {
    return x;
  }
}

// RMSNorm (optional weight) then rotate_half RoPE of one row held in the lane
// layout above (f: the row's raw values; wf: the lane's weights, or ones for
// a row without weight), at position pos; the partner
// of element d is d +- HD/2, which is the same lane (NPC >= 2) or lane ^ 16
// (NPC == 1).  bf16 results are the correctly rounded real values
// (g4_normrope.cuh), the ones the append kernel stores, decided in three
// stages as there: float32 with Ziv's test; the float inverse rms times the
// inner products in double-float for the values left open; the row's
// double-float inverse rms for the rest.  s_cos / s_sin hold cos and sin of
// the HD/2 pairs.
template <typename T, int HD, int NPC, int PE>
__device__ __forceinline__ void norm_rope_row(float* f, const float* wf, bool rope, const DF* s_cos, const DF* s_sin,
                                              int n_rot, float eps, int lane) {
  constexpr int EL = NPC * PE;
  constexpr bool kBF16 = sizeof(T) == 2;
  constexpr float kErrY = normrope_err_y<EL>();
  constexpr float kErrAB = normrope_err_pair(kDFTrigErrUnits);
  constexpr float kErrO = normrope_err_out<EL>();
  constexpr float kErrR = normrope_err_r<EL>();
  const float sf = row_sumsq_f32<EL>(f);
  const float r = inv_rms_f32(sf, HD, eps);
  // raw partner values and weights
  float fp[EL], wp[EL];
  if constexpr (NPC >= 2) {
#pragma unroll
    for (int c = 0; c < NPC; ++c)
#pragma unroll
      for (int e = 0; e < PE; ++e) {
        fp[c * PE + e] = f[((c + NPC / 2) % NPC) * PE + e];
        wp[c * PE + e] = wf[((c + NPC / 2) % NPC) * PE + e];
      }
  } else {
#pragma unroll
    for (int e = 0; e < PE; ++e) {
      fp[e] = __shfl_xor_sync(0xffffffffu, f[e], 16);
      wp[e] = __shfl_xor_sync(0xffffffffu, wf[e], 16);
    }
  }
  // Each element's own output only, the same float32 operations as
  // normrope_pair_fast's output of that side (ya, yb rounded products, one
  // fma with the partner's product; the same bounds), with the rotation's
  // sign selected rather than branched on: with one row half per lane group
  // (NPC == 1) a branch on the half ran both sides in every warp.
  float o[EL];
  uint32_t need = 0;
#pragma unroll
  for (int c = 0; c < NPC; ++c) {
#pragma unroll
    for (int e = 0; e < PE; ++e) {
      const int i = c * PE + e;
      const int d = (lane + 32 * c) * PE + e;
      const bool lower = d < HD / 2;
      const int j = lower ? d : d - HD / 2;
      const bool rot = rope && j < n_rot;
      const float ys = (f[i] * r) * wf[i];
      float oi, ei;
      if (rot) {
        const float cj = s_cos[j].h, sj = s_sin[j].h;
        const float yo = (fp[i] * r) * wp[i];
        const float po = yo * sj;
        oi = fmaf(ys, cj, lower ? -po : po);
        ei = fmaf(kErrO, fabsf(oi), kErrAB * (fabsf(ys) + fabsf(yo)));
      } else {
        oi = ys;
        ei = kErrY * fabsf(ys);
      }
      o[i] = oi;
      need |= (fabsf(oi - bf16_midpoint(oi)) > ei ? 0u : 1u) << i;
    }
  }
  if constexpr (kBF16) {
    if (__any_sync(0xffffffffu, need != 0)) {
      // Stage 2, lane by lane, one open value per pass.  The operands come
      // from the registers (a select over the lane's elements keeps the
      // arrays in registers; reloading them from memory put an L2 round trip
      // on every pass).
      uint32_t open = 0;
#pragma unroll 1
      for (uint32_t left = need; left != 0; left &= left - 1) {
        const int i = __ffs(left) - 1;
        const int d = (lane + 32 * (i / PE)) * PE + i % PE;
        const bool lower = d < HD / 2;
        const int j = lower ? d : d - HD / 2;
        float xs = 0.0f, ws = 1.0f, xo = 0.0f, wo = 1.0f;
#pragma unroll
        for (int k = 0; k < EL; ++k)
          if (k == i) {
            xs = f[k];
            ws = wf[k];
            xo = fp[k];
            wo = wp[k];
          }
        DF inner = two_prod(xs, ws);
        float mag = fabsf(inner.h);
        if (rope && j < n_rot) {
          const DF po = two_prod(xo, wo);
          mag += fabsf(po.h);
          inner = df_add(df_mul(inner, s_cos[j]), df_mul(po, lower ? df_neg(s_sin[j]) : s_sin[j]));
        }
        const DF v = df_mul_f(inner, r);
        if (fabsf((v.h - bf16_midpoint(v.h)) + v.l) > fmaf(kErrR, fabsf(v.h), 0x1.0p-40f * r * mag)) {
          const float val = df_round_bf16(v);
#pragma unroll
          for (int k = 0; k < EL; ++k)
            if (k == i) o[k] = val;
        } else {
          open |= 1u << i;
        }
      }
      // Stage 3: the row's double-float inverse rms.
      if (__any_sync(0xffffffffu, open != 0)) {
        const DF rd = inv_rms_df(row_sumsq_split<EL, HD>(f, sf), HD, eps);
#pragma unroll
        for (int c = 0; c < NPC; ++c) {
#pragma unroll
          for (int e = 0; e < PE; ++e) {
            const int i = c * PE + e;
            if (open & (1u << i)) {
              const int d = (lane + 32 * c) * PE + e;
              const bool lower = d < HD / 2;
              const int j = lower ? d : d - HD / 2;
              o[i] = normrope_exact_bf16(f[i], wf[i], fp[i], wp[i], rd, rope && j < n_rot, lower, s_cos[j], s_sin[j]);
            }
          }
        }
      }
    }
  }
  // the stored value (certified float32 values still need their rounding)
#pragma unroll
  for (int i = 0; i < EL; ++i) f[i] = through<T>(o[i]);
}

}  // namespace g4

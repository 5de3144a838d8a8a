// Steps a6 (decode) and a5 in float32: causal GQA softmax attention on CUDA
// cores, split over the key range (split-KV), HBM-bound.
//
// Semantics (cortiq-engine g4e.rs `attend_all_heads(q, caches[src], ..., 1.0,
// window, ...)`; ferrox-models gemma4_engine.rs `causal_gqa_attention[_windowed]`;
// turbospark-runtime gemma4/attn.rs `kv_start = seq_len - sliding_window`):
// query head h reads kv head h / G (G = H / Hkv, contiguous groups as in
// taconite `text_attention`), keys [kstart, L) with kstart = L - window on
// sliding layers and 0 on full layers, scores scaled by attn_scale (1.0).
// On a sliding-window ring cache (turbospark-runtime gemma4 decode:
// `ring_capacity`) key position p is row p mod max_len, and a stage whose
// keys cross the ring's last row is two copies.  Mode 2 (float32 encoder,
// taconite-embeddinggemma2 `text_attention`): query t of a sequence sees its
// keys [t - window, t + window] (sliding) or all T, with no causal mask.
//
// Work decomposition: one CTA per (split, kv head, query row).  All G query
// heads of the kv head share every K/V row the CTA streams, so each key row
// is read from HBM once per query row.  Each of the 4 warps (8 when the
// launch fits one CTA per SM) owns a ring of 2-3 shared-memory stages filled
// by non-tensor bulk copies
// (cp.async.bulk, one K and one V copy per stage, completing on the stage's
// mbarrier); stages of the CTA's key range go to the warps round-robin.
//
// Inside a warp, lane l owns HD/32 elements of every row (16-byte pieces
// l, l+32, ... so shared-memory reads are conflict-free).  For a batch of
// KB = min(16/G, 4 KB of rows) keys the lane forms KB*G partial dot products
// with packed f32x2 FMAs, a butterfly reduce-scatter turns the KB*G partials
// of 32 lanes into KB*G full scores, the scores go through shared memory so
// every lane holds all of them, and the online softmax (log2 domain; q is
// pre-scaled by attn_scale*log2(e)) and the P.V update run redundantly per
// lane with no further shuffles.  Warps merge their (m, l, o) through shared
// memory.  With one split the CTA writes the normalised output; otherwise it
// writes an un-normalised partial, takes a ticket from an atomic counter,
// and the CTA that takes the last ticket of its (query row, kv head) merges
// all partials with log-sum-exp weights and writes the output (no CTA ever
// waits for another).
//
// The FUSED variant (decode step) starts from the new token's raw q / k / v:
// every CTA norms and ropes its q heads itself, and the CTA whose split holds
// position L-1 norms/ropes the new k and v (cortiq-engine `rms`, `rms_plain`,
// rotate_half as in taconite `rope_half`), stores them into the cache row
// L-1, and uses them as its last key -- the append and the attention of one
// decode step in a single launch.
#include <math.h>
#include <string.h>

#include "g4_device.cuh"
#include "g4_internal.h"
#include "g4_normrope.cuh"

namespace g4 {
namespace {

constexpr int kNPMax = 16;        // partial scores per reduce-scatter batch, at most
constexpr int kStageMaxB = 4096;  // bytes of K (and of V) a reduce batch may span



constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// d = a * b + c on two packed floats (one f32x2 instruction).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  unsigned long long ua, ub, uc, ud;
  memcpy(&ua, &a, 8);
  memcpy(&ub, &b, 8);
  memcpy(&uc, &c, 8);
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(ud) : "l"(ua), "l"(ub), "l"(uc));
  float2 d;
  memcpy(&d, &ud, 8);
  return d;
}

// 2^x with the hardware approximation (inputs here are <= 0; -inf gives 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Sum of v[i] over the 32 lanes, scattered: lane l returns the total of index
// l >> (5 - log2(NP)).  NP is a power of two in [2, 32].
template <int NP>
__device__ __forceinline__ float reduce_scatter(float (&v)[NP], int lane) {
#pragma unroll
  for (int n = NP, o = 16; n > 1; n >>= 1, o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = up ? v[i] : v[i + n / 2];
      const float keep = up ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float r = v[0];
#pragma unroll
  for (int o = 16 >> ilog2(NP); o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  return r;
}

template <typename T, int HD, int G, int NW_>
struct SimtCfg {
  static constexpr int NW = NW_;                     // warps per CTA
  static constexpr int ES = sizeof(T);
  static constexpr int EL = HD / 32;                 // elements per lane per row
  static constexpr int CHE = 16 / ES;                // elements per 16-byte piece
  static constexpr int PE = EL < CHE ? EL : CHE;     // elements per piece a lane reads
  static constexpr int NPC = EL / PE;                // pieces per lane per row
  static constexpr int ROWB = HD * ES;               // bytes per cache row
  static constexpr int KB_G = kNPMax / G;
  static constexpr int KB_B = kStageMaxB / ROWB;
  static constexpr int KB = KB_G < KB_B ? KB_G : KB_B;  // keys per reduce batch
  static constexpr int NP = KB * G;                  // partial scores per batch (2..16)
  static constexpr int NB = (KB * ROWB >= 2048) ? 1 : 2048 / (KB * ROWB);  // batches per stage
  static constexpr int SK = KB * NB;                 // keys per stage
  static constexpr int STAGE_B = SK * ROWB;          // bytes of K (and of V) per stage
  // G*HD = 2048 needs ~180 registers for q and o alone: two CTAs per SM with
  // three stages per warp; narrower heads fit three CTAs with two stages.  The
  // 8-warp CTA serves launches of at most one CTA per SM.
  static constexpr int NST = (G * HD >= 2048) ? 3 : 2;   // stages per warp
  static constexpr int MINB = NW > 4 ? 1 : (G * HD >= 2048) ? 2 : 3;  // CTAs per SM the register budget aims for
  static constexpr int RING_B = NW * NST * 2 * STAGE_B;
  static constexpr int MERGE_B = NW * G * (HD + 2) * 4;
  static constexpr int AREA_B = RING_B > MERGE_B ? RING_B : MERGE_B;
  // after the area: barriers, per-warp score buffers, cos/sin table, merge weights, flag
  static constexpr int BAR_OFF = AREA_B;
  static constexpr int SC_OFF = BAR_OFF + NW * NST * 8;
  static constexpr int SA_OFF = SC_OFF + NW * kNPMax * 4;
  static constexpr int COS_OFF = SA_OFF + NW * 8 * 4;
  static constexpr int W_OFF = COS_OFF + HD * 8;  // cos and sin of HD/2 pairs, double-float
  static constexpr int FLAG_OFF = W_OFF + G * kMaxSplits * 4;
  static constexpr int QN_OFF = FLAG_OFF + 16;  // normed q of the G heads (fused step)
  static constexpr int KN_OFF = QN_OFF + G * HD * ES;  // normed new k and v (fused step)
  static constexpr int SMEM_B = KN_OFF + 2 * HD * ES;
  static_assert(NP >= 2 && NP <= 16 && (NP & (NP - 1)) == 0, "reduce batch");
  static_assert(SMEM_B <= 232448, "shared memory budget");
};

template <typename T, int HD, int G, bool FUSED, int NW>
__global__ void __launch_bounds__(NW * 32, (SimtCfg<T, HD, G, NW>::MINB))
    attn_simt_kernel(const __grid_constant__ AttnSimtArgs a) {
  using C = SimtCfg<T, HD, G, NW>;
  constexpr int EL2 = C::EL / 2;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  float* sc_all = reinterpret_cast<float*>(smem + C::SC_OFF);
  float* sa_all = reinterpret_cast<float*>(smem + C::SA_OFF);
  DF* s_cos = reinterpret_cast<DF*>(smem + C::COS_OFF);
  DF* s_sin = s_cos + HD / 2;
  float* s_w = reinterpret_cast<float*>(smem + C::W_OFF);
  int* s_flag = reinterpret_cast<int*>(smem + C::FLAG_OFF);

  const int split = blockIdx.x % a.nsplit;
  const int rest = blockIdx.x / a.nsplit;
  const int kvh = rest % a.Hkv;
  const int bt = rest / a.Hkv;  // b * T + t
  const int b = bt / a.T;
  const int t = bt % a.T;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint64_t* wbar = bars + warp * C::NST;
  // With 8 warps and 1 KB rows the last warp (which has no norm row when
  // G <= 6) sets up every warp's stage barriers and issues their first stages
  // (48 copies, which take microseconds to issue), so the others go straight
  // to the cos/sin table; they first touch the barriers after the CTA barrier
  // that ends the table.  Otherwise each warp does its own.
  constexpr bool kIssuer = NW > 4 && HD >= 512;
  if (kIssuer ? (warp == NW - 1 && lane == 0) : lane == 0) {
    for (int i = 0; i < (kIssuer ? NW : 1) * C::NST; ++i) mbar_init(smem_u32(&(kIssuer ? bars : wbar)[i]), 1);
    fence_mbar_init();
  }
  __syncwarp();
  pdl_wait();
  pdl_trigger();

  // Query position and visible key range [kbeg, L).
  int L, kbeg;
  if (!FUSED && a.mode == 2) {
    // encoder: token t of the sequence's T keys, no causal mask (the host
    // caps the window at T)
    kbeg = a.sliding ? max(0, t - a.window) : 0;
    L = a.sliding ? min(a.T, t + a.window + 1) : a.T;
  } else {
    if (a.mode == 0) {
      L = min(max(a.base[b], 1), a.len_cap);
    } else if (a.ring) {
      L = max(a.base[b] + t, 0) + 1;  // every position has a row in a ring
    } else {
      L = min(max(a.base[b] + t, 0), a.max_len - 1) + 1;
    }
    kbeg = a.sliding ? max(0, L - a.window) : 0;
  }
  const int k0 = kbeg + split * a.chunk;
  const int k1 = min(L, k0 + a.chunk);
  // FUSED: the CTA holding position L-1 computes that key itself.
  const bool new_key = FUSED && a.k_raw != nullptr && (L - 1 >= k0) && (L - 1 < k1);
  const int k1c = new_key ? L - 1 : k1;  // keys streamed from the cache
  const int nkeys = max(0, k1c - k0);
  const int nstages = (nkeys + C::SK - 1) / C::SK;

  uint8_t* ring = smem + warp * (C::NST * 2 * C::STAGE_B);
  float* sc = sc_all + warp * kNPMax;
  float* sa = sa_all + warp * 8;
  bool aborted = false;
  // After a reduce-scatter, lane l holds the score of entry idx = l >> kSh
  // (key idx / G, head idx % G); it keeps the softmax state (m, l) of head hh.
  constexpr int kSh = 5 - ilog2(C::NP);
  const int hh = (lane >> kSh) & (G - 1);

  const size_t head_base = (static_cast<size_t>(b) * a.Hkv + kvh) * a.max_len;
  const T* gk = static_cast<const T*>(a.ck) + head_base * HD;
  const T* gv = static_cast<const T*>(a.cv) + head_base * HD;

  // stage st_idx of warp w's ring into its buffer buf
  auto issue_for = [&](int w, int st_idx, int buf) {
    const int kk0 = k0 + st_idx * C::SK;
    const int n = min(C::SK, k1c - kk0);
    const uint32_t bytes = static_cast<uint32_t>(n) * C::ROWB;
    const uint32_t bar = smem_u32(&bars[w * C::NST + buf]);
    uint8_t* rw = smem + w * (C::NST * 2 * C::STAGE_B);
    const uint32_t dk = smem_u32(rw + buf * 2 * C::STAGE_B);
    const uint32_t dv = dk + C::STAGE_B;
    mbar_arrive_expect_tx(bar, 2 * bytes);
    if (!a.ring) {
      bulk_g2s(dk, gk + static_cast<size_t>(kk0) * HD, bytes, bar);
      bulk_g2s(dv, gv + static_cast<size_t>(kk0) * HD, bytes, bar);
    } else {
      // Positions kk0 .. kk0+n-1 sit in rows r0 .. (wrapping to row 0 once
      // the ring's end is reached, at most once since n <= max_len).
      const int r0 = kk0 % a.max_len;
      const int n0 = min(n, a.max_len - r0);
      const uint32_t b0 = static_cast<uint32_t>(n0) * C::ROWB;
      bulk_g2s(dk, gk + static_cast<size_t>(r0) * HD, b0, bar);
      bulk_g2s(dv, gv + static_cast<size_t>(r0) * HD, b0, bar);
      if (n0 < n) {
        bulk_g2s(dk + b0, gk, bytes - b0, bar);
        bulk_g2s(dv + b0, gv, bytes - b0, bar);
      }
    }
  };
  auto issue = [&](int st_idx, int buf) { issue_for(warp, st_idx, buf); };

  // (lane w of the issuing warp issues warp w's stages)
  if (kIssuer ? (warp == NW - 1 && lane < NW) : lane == 0) {
    const int w = kIssuer ? lane : warp;
    for (int i = 0; i < C::NST; ++i) {
      const int st = w + i * NW;
      if (st < nstages) issue_for(w, st, i);
    }
  }
  // (the fused step's table ends with a CTA barrier; the plain one needs its own)
  if constexpr (kIssuer && !FUSED) __syncthreads();

  if constexpr (FUSED) {
    // cos/sin of the new token's position (two threads per rotated pair, one
    // per polynomial), then its q heads -- and on the CTA that holds position
    // L-1 the new k and v -- normed and roped, one row per warp, into shared
    // memory (k and v also into the cache row L-1).
    const int pos = L - 1;
    const int njobs = G + (new_key ? 2 : 0);
    // Row `job` of the jobs: q head job (< G), then the new k and v.
    struct Job {
      const T* src;
      T* dst_g;
      const float* w;
      bool rope;
    };
    auto job_of = [&](int job) -> Job {
      Job j;
      if (job < G) {
        j.src = static_cast<const T*>(a.q) + (static_cast<size_t>(bt) * a.H + kvh * G + job) * HD;
        j.dst_g = nullptr;
        j.w = a.q_w;
        j.rope = true;
      } else {
        const bool is_k = job == G;
        j.src = static_cast<const T*>(is_k ? a.k_raw : a.v_raw) + (static_cast<size_t>(b) * a.Hkv + kvh) * HD;
        const int row = a.ring ? (L - 1) % a.max_len : L - 1;
        j.dst_g = static_cast<T*>(is_k ? a.cache_k : a.cache_v) + (head_base + row) * HD;
        j.w = is_k ? a.k_w : nullptr;
        j.rope = is_k;
      }
      return j;
    };
    auto load_job = [&](const Job& j, float* f, float* wf) {
      load_row<T, C::NPC, C::PE>(j.src, lane, f);
      if (j.w != nullptr) {
        load_row<float, C::NPC, C::PE>(j.w, lane, wf);
      } else {
#pragma unroll
        for (int i = 0; i < C::EL; ++i) wf[i] = 1.0f;
      }
    };
    // The warp's first row is loaded before the table is built, so the two overlap.
    float f[C::EL], wf[C::EL];
    if (warp < njobs) load_job(job_of(warp), f, wf);
    constexpr int kTableThreads = (kIssuer ? NW - 1 : NW) * 32;
    for (int idx = threadIdx.x; idx < HD && threadIdx.x < kTableThreads; idx += kTableThreads) {
      const int j = idx >> 1, part = idx & 1;
      if (j < a.n_rot) {
        bool to_cos;
        const DF v = sincos_df_part(pos, a.inv_freq[j], part, to_cos);
        (to_cos ? s_cos : s_sin)[j] = v;
      } else if (part == 0) {
        s_cos[j] = DF{1.0f, 0.0f};
      } else {
        s_sin[j] = DF{0.0f, 0.0f};
      }
    }
    __syncthreads();
    T* s_qn = reinterpret_cast<T*>(smem + C::QN_OFF);
    T* s_kn = reinterpret_cast<T*>(smem + C::KN_OFF);
    for (int job = warp; job < njobs; job += NW) {
      const Job j = job_of(job);
      if (job != warp) load_job(j, f, wf);
      norm_rope_row<T, HD, C::NPC, C::PE>(f, wf, j.rope, s_cos, s_sin, a.n_rot, a.eps, lane);
      store_row<T, C::NPC, C::PE>(job < G ? s_qn + job * HD : s_kn + (job - G) * HD, lane, f);
      if (j.dst_g != nullptr) store_row<T, C::NPC, C::PE>(j.dst_g, lane, f);
    }
    __syncthreads();
  }

  // q of the G heads, pre-scaled into the log2 domain.
  float2 q2[G][EL2];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const T* qrow = FUSED ? reinterpret_cast<const T*>(smem + C::QN_OFF) + h * HD
                          : static_cast<const T*>(a.q) + (static_cast<size_t>(bt) * a.H + kvh * G + h) * HD;
    float f[C::EL];
    load_row<T, C::NPC, C::PE>(qrow, lane, f);
#pragma unroll
    for (int i = 0; i < C::EL; ++i) f[i] *= a.scale_log2;
    to_f2<C::EL>(f, q2[h]);
  }

  float m_l = -INFINITY, l_l = 0.0f;  // softmax state of head hh (log2 domain)
  float2 o2[G][EL2];
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int i = 0; i < EL2; ++i) o2[h][i] = make_float2(0.0f, 0.0f);
  }

  if constexpr (FUSED) {
    // The new key (normed above) goes first, into the last warp's state.
    if (new_key && warp == NW - 1) {
      const T* s_kn = reinterpret_cast<const T*>(smem + C::KN_OFF);
      float2 kx[EL2], vx[EL2];
      load_row_f2<T, C::NPC, C::PE>(s_kn, lane, kx);
      load_row_f2<T, C::NPC, C::PE>(s_kn + HD, lane, vx);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < EL2; ++i) acc = fma2(q2[h][i], kx[i], acc);
        const float s = warp_sum(acc.x + acc.y);
        const float m_h = __shfl_sync(0xffffffffu, m_l, h << kSh);
        const float m_new = fmaxf(m_h, s);
        const float alpha = (m_h == -INFINITY) ? 0.0f : ex2(m_h - m_new);
        const float pn = ex2(s - m_new);
        if (hh == h) {
          l_l = l_l * alpha + pn;
          m_l = m_new;
        }
        const float2 pp = make_float2(pn, pn);
#pragma unroll
        for (int i = 0; i < EL2; ++i) {
          o2[h][i].x *= alpha;
          o2[h][i].y *= alpha;
          o2[h][i] = fma2(pp, vx[i], o2[h][i]);
        }
      }
    }
  }

  int consumed = 0;  // stages this warp has finished (for draining after an abort)
  for (int it = 0;; ++it) {
    const int st_idx = warp + it * NW;
    if (st_idx >= nstages) break;
    const int buf = it % C::NST;
    if (!warp_wait(smem_u32(&wbar[buf]), (it / C::NST) & 1, a.err)) {
      aborted = true;
      break;
    }
    const int n = min(C::SK, k1c - (k0 + st_idx * C::SK));
    const T* sk = reinterpret_cast<const T*>(ring + buf * 2 * C::STAGE_B);
    const T* sv = reinterpret_cast<const T*>(ring + buf * 2 * C::STAGE_B + C::STAGE_B);

#pragma unroll 1
    for (int nb = 0; nb < C::NB; ++nb) {
      const int kb0 = nb * C::KB;
      if (kb0 >= n) break;
      // Partial dot products: part[key * G + h].
      float part[C::NP];
#pragma unroll
      for (int key = 0; key < C::KB; ++key) {
        float2 kx[EL2];
        load_row_f2<T, C::NPC, C::PE>(sk + (kb0 + key) * HD, lane, kx);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int i = 0; i < EL2; ++i) acc = fma2(q2[h][i], kx[i], acc);
          part[key * G + h] = acc.x + acc.y;
        }
      }
      // Softmax of this batch: each lane exponentiates its own entry; batch
      // max and sum per head run over the lanes of the same head (key bits).
      const float s = reduce_scatter<C::NP>(part, lane);
      const int key_l = (lane >> kSh) / G;
      const float s_me = (kb0 + key_l < n) ? s : -INFINITY;
      float mb = s_me;
#pragma unroll
      for (int o = 1 << (kSh + ilog2(G)); o < 32; o <<= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
      const float m_new = fmaxf(m_l, mb);
      const float alpha = (m_l == -INFINITY) ? 0.0f : ex2(m_l - m_new);
      const float p_l = ex2(s_me - m_new);
      float ps = p_l;
#pragma unroll
      for (int o = 1 << (kSh + ilog2(G)); o < 32; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l_l = l_l * alpha + ps;
      m_l = m_new;
      if ((lane & ((1 << kSh) - 1)) == 0) {
        sc[lane >> kSh] = p_l;
        if (key_l == 0) sa[hh] = alpha;
      }
      __syncwarp();
      float p[C::KB][G];
#pragma unroll
      for (int i = 0; i < C::NP; ++i) p[i / G][i % G] = sc[i];
      float al[G];
#pragma unroll
      for (int h = 0; h < G; ++h) al[h] = sa[h];
      __syncwarp();
#pragma unroll
      for (int h = 0; h < G; ++h) {
        if (al[h] != 1.0f) {
#pragma unroll
          for (int i = 0; i < EL2; ++i) {
            o2[h][i].x *= al[h];
            o2[h][i].y *= al[h];
          }
        }
      }
      // o += p . v
#pragma unroll
      for (int key = 0; key < C::KB; ++key) {
        if (kb0 + key < n) {
          float2 vx[EL2];
          load_row_f2<T, C::NPC, C::PE>(sv + (kb0 + key) * HD, lane, vx);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float2 pp = make_float2(p[key][h], p[key][h]);
#pragma unroll
            for (int i = 0; i < EL2; ++i) o2[h][i] = fma2(pp, vx[i], o2[h][i]);
          }
        }
      }
    }
    __syncwarp();
    consumed = it + 1;
    const int next = st_idx + C::NST * NW;
    if (lane == 0 && next < nstages) issue(next, buf);
  }

  // After an abort, wait (bounded) for copies this warp still has in flight.
  if (aborted) {
    for (int it = consumed;; ++it) {
      const int st_idx = warp + it * NW;
      if (st_idx >= nstages || it >= consumed + C::NST) break;
      warp_wait(smem_u32(&wbar[it % C::NST]), (it / C::NST) & 1, nullptr);
    }
  }

  __syncthreads();

  // Merge the warps' (m, l, o) through shared memory (the ring is free now).
  float* ms = reinterpret_cast<float*>(smem);          // [NW][G]
  float* ls = ms + NW * G;                            // [NW][G]
  float* os = ls + NW * G;                            // [NW][G][HD]
  if ((lane & ((1 << kSh) - 1)) == 0 && (lane >> kSh) < G) {
    ms[warp * G + hh] = m_l;
    ls[warp * G + hh] = l_l;
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float* orow = os + (warp * G + h) * HD;
#pragma unroll
    for (int c = 0; c < C::NPC; ++c) {
      float f[C::PE];
#pragma unroll
      for (int e = 0; e < C::PE; e += 2) {
        f[e] = o2[h][(c * C::PE + e) / 2].x;
        f[e + 1] = o2[h][(c * C::PE + e) / 2].y;
      }
      store_elems<C::PE>(orow + (lane + 32 * c) * C::PE, f);
    }
  }
  __syncthreads();

  for (int idx = threadIdx.x; idx < G * HD; idx += blockDim.x) {
    const int h = idx / HD;
    const int d = idx % HD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, ms[w * G + h]);
    float O = 0.0f, Ls = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float mw = ms[w * G + h];
        if (mw != -INFINITY) {
          const float f = ex2(mw - M);
          O += f * os[(w * G + h) * HD + d];
          Ls += f * ls[w * G + h];
        }
      }
    }
    const int head = kvh * G + h;
    if (a.nsplit == 1) {
      const float val = (Ls > 0.0f) ? O / Ls : 0.0f;
      T* dst = static_cast<T*>(a.out) + (static_cast<size_t>(bt) * a.H + head) * HD + d;
      store_elems<1>(dst, &val);
    } else {
      const size_t pidx = (static_cast<size_t>(bt) * a.H + head) * a.nsplit + split;
      a.ws_o[pidx * HD + d] = O;
      if (d == 0) {
        a.ws_m[pidx] = M;
        a.ws_l[pidx] = Ls;
      }
    }
  }
  if (a.nsplit == 1) return;

  // Ticket: the CTA that completes the set of splits of this (row, kv head)
  // merges them.  Writers publish their partial before taking a ticket.
  __threadfence();
  __syncthreads();
  unsigned* ticket = a.tickets + static_cast<size_t>(bt) * a.Hkv + kvh;
  if (threadIdx.x == 0) *s_flag = (atomicAdd(ticket, 1u) == static_cast<unsigned>(a.nsplit - 1)) ? 1 : 0;
  __syncthreads();
  if (*s_flag == 0) return;
  __threadfence();
  if (a.nsplit <= 8) {
    // Each thread owns float4 groups of the G*HD outputs and merges the (at
    // most 8) splits with log-sum-exp weights, all of its loads -- running
    // maxima, denominators and partial outputs -- in flight at once.
    constexpr int NG4 = G * HD / 4;                        // float4 groups
    constexpr int PER = (NG4 + NW * 32 - 1) / (NW * 32);  // groups per thread
    const size_t pbase = (static_cast<size_t>(bt) * a.H + kvh * G) * a.nsplit;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int g4i = threadIdx.x + i * NW * 32;
      if (g4i >= NG4) break;
      const int h = (g4i * 4) / HD;
      const int d = (g4i * 4) % HD;
      const size_t prow = pbase + static_cast<size_t>(h) * a.nsplit;  // (head h, split 0)
      float mv[8], lv[8];
      float4 ov[8];
      float M = -INFINITY;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        mv[u] = -INFINITY;
        if (u < a.nsplit) {
          mv[u] = __ldcg(a.ws_m + prow + u);
          lv[u] = __ldcg(a.ws_l + prow + u);
          ov[u] = __ldcg(reinterpret_cast<const float4*>(a.ws_o + (prow + u) * HD + d));
        }
        M = fmaxf(M, mv[u]);
      }
      float Ls = 0.0f;
      float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (mv[u] != -INFINITY) {
          const float w = exp2f(mv[u] - M);
          Ls = fmaf(w, lv[u], Ls);
          acc.x = fmaf(w, ov[u].x, acc.x);
          acc.y = fmaf(w, ov[u].y, acc.y);
          acc.z = fmaf(w, ov[u].z, acc.z);
          acc.w = fmaf(w, ov[u].w, acc.w);
        }
      }
      const float inv = Ls > 0.0f ? 1.0f / Ls : 0.0f;
      T* dst = static_cast<T*>(a.out) + (static_cast<size_t>(bt) * a.H + kvh * G + h) * HD + d;
      const float f[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
      store_elems<4>(dst, f);
    }
  } else {
    // More splits: the log-sum-exp weights per head first (into shared
    // memory), then every partial output load of a round in flight.
    for (int h = warp; h < G; h += NW) {
      const size_t p0 = (static_cast<size_t>(bt) * a.H + kvh * G + h) * a.nsplit;
      float M = -INFINITY;
      for (int s = lane; s < a.nsplit; s += 32) M = fmaxf(M, __ldcg(a.ws_m + p0 + s));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      float Ls = 0.0f;
      for (int s = lane; s < a.nsplit; s += 32) {
        const float ms_ = __ldcg(a.ws_m + p0 + s);
        const float w = (ms_ == -INFINITY) ? 0.0f : exp2f(ms_ - M);
        s_w[h * kMaxSplits + s] = w;
        Ls += w * __ldcg(a.ws_l + p0 + s);
      }
      Ls = warp_sum(Ls);
      const float inv = Ls > 0.0f ? 1.0f / Ls : 0.0f;
      __syncwarp();
      for (int s = lane; s < a.nsplit; s += 32) s_w[h * kMaxSplits + s] *= inv;
    }
    __syncthreads();
    // Each thread owns float4 groups of the G*HD outputs and keeps many loads in
    // flight: 8 splits x up to 4 groups per round.
    constexpr int NG4 = G * HD / 4;                        // float4 groups
    constexpr int PER = (NG4 + NW * 32 - 1) / (NW * 32);  // groups per thread
    float4 acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const size_t pbase = (static_cast<size_t>(bt) * a.H + kvh * G) * a.nsplit;
    for (int s0 = 0; s0 < a.nsplit; s0 += 8) {
      float4 v[PER][8];
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int g4i = threadIdx.x + i * NW * 32;
        const int h = (g4i * 4) / HD;
        const int d = (g4i * 4) % HD;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int sp = s0 + u;
          v[i][u] = (g4i < NG4 && sp < a.nsplit)
                        ? __ldcg(reinterpret_cast<const float4*>(a.ws_o + ((pbase + static_cast<size_t>(h) * a.nsplit +
                                                                             sp) * HD + d)))
                        : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
      }
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int g4i = threadIdx.x + i * NW * 32;
        const int h = g4i < NG4 ? (g4i * 4) / HD : 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float w = (s0 + u < a.nsplit) ? s_w[h * kMaxSplits + s0 + u] : 0.0f;
          acc[i].x = fmaf(w, v[i][u].x, acc[i].x);
          acc[i].y = fmaf(w, v[i][u].y, acc[i].y);
          acc[i].z = fmaf(w, v[i][u].z, acc[i].z);
          acc[i].w = fmaf(w, v[i][u].w, acc[i].w);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int g4i = threadIdx.x + i * NW * 32;
      if (g4i < NG4) {
        const int h = (g4i * 4) / HD;
        const int d = (g4i * 4) % HD;
        T* dst = static_cast<T*>(a.out) + (static_cast<size_t>(bt) * a.H + kvh * G + h) * HD + d;
        const float f[4] = {acc[i].x, acc[i].y, acc[i].z, acc[i].w};
        store_elems<4>(dst, f);
      }
    }
  }
  if (threadIdx.x == 0) *ticket = 0u;  // ready for the next call
}

template <typename Kern>
cudaError_t launch_pdl(Kern kern, unsigned grid, unsigned block, size_t smem, cudaStream_t s,
                       const AttnSimtArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T, int HD, int G, bool FUSED, int NW>
cudaError_t launch_simt_hgfw(const AttnSimtArgs& a, long long nblk, cudaStream_t s) {
  using C = SimtCfg<T, HD, G, NW>;
  const cudaError_t e = set_smem_limit_once<attn_simt_kernel<T, HD, G, FUSED, NW>>(C::SMEM_B);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_simt_kernel<T, HD, G, FUSED, NW>, static_cast<unsigned>(nblk), NW * 32, C::SMEM_B, s, a);
}

// A launch that fits one CTA per SM (short sliding windows, small batches)
// is latency-bound: its CTAs take 8 warps, so each warp streams half as many
// stages.  Larger launches keep 4 warps and several CTAs per SM.
template <typename T, int HD, int G, bool FUSED>
cudaError_t launch_simt_hgf(const AttnSimtArgs& a, cudaStream_t s) {
  const long long nblk = static_cast<long long>(a.nsplit) * a.Hkv * a.B * a.T;
  if (nblk <= sm_count()) return launch_simt_hgfw<T, HD, G, FUSED, 8>(a, nblk, s);
  return launch_simt_hgfw<T, HD, G, FUSED, 4>(a, nblk, s);
}

template <typename T, int HD, int G>
cudaError_t launch_simt_hg(const AttnSimtArgs& a, cudaStream_t s) {
  return a.fused ? launch_simt_hgf<T, HD, G, true>(a, s) : launch_simt_hgf<T, HD, G, false>(a, s);
}

template <typename T, int HD>
cudaError_t launch_simt_h(const AttnSimtArgs& a, cudaStream_t s) {
  const int G = a.H / a.Hkv;
  switch (G) {
    case 1: return launch_simt_hg<T, HD, 1>(a, s);
    case 2: return launch_simt_hg<T, HD, 2>(a, s);
    case 4: return launch_simt_hg<T, HD, 4>(a, s);
    case 8:
      if constexpr (HD <= 256) return launch_simt_hg<T, HD, 8>(a, s);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_simt_t(const AttnSimtArgs& a, cudaStream_t s) {
  switch (a.hd) {
    case 64: return launch_simt_h<T, 64>(a, s);
    case 128: return launch_simt_h<T, 128>(a, s);
    case 256: return launch_simt_h<T, 256>(a, s);
    case 512: return launch_simt_h<T, 512>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_attn_simt(const AttnSimtArgs& a, int dtype, cudaStream_t s) {
  return dtype == 1 ? launch_simt_t<__nv_bfloat16>(a, s) : launch_simt_t<float>(a, s);
}

int sm_count() {
  static int cached[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) {
    cudaGetLastError();
    return 152;  // GB300
  }
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 152;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

DecodePlan decode_plan(int dtype, int sliding, int window, int hd, int H, int Hkv, int B, int max_seq_len) {
  DecodePlan p;
  const int span = sliding ? (max_seq_len < window ? max_seq_len : window) : max_seq_len;
  if (decode_win_eligible(dtype, hd, H / Hkv, span, B * Hkv)) {
    p.win = 1;
    p.chunk = 64;
    p.nsplit = decode_win_splits(span);
    p.o_bytes = p.m_bytes = p.t_bytes = p.ws_bytes = 0;
    return p;
  }
  p.win = 0;
  const int units = B * Hkv;
  const int G = H / Hkv;
  // CTA slots of one wave: SMs x CTAs per SM (two for G*hd >= 2048, else three).
  const int slots = sm_count() * ((G * hd >= 2048) ? 2 : 3);
  // Splits: at least 64 keys each, and at most sqrt(span / 8) so that the
  // final merge (nsplit partials of G*hd floats) stays small next to the keys
  // each split streams; within that, a whole number of waves (4 down to 1).
  const int by_len = (span + 63) / 64;
  int by_merge = static_cast<int>(sqrt(static_cast<double>(span) / 8.0));
  if (by_merge < 4) by_merge = 4;
  int cap = by_len < by_merge ? by_len : by_merge;
  if (cap > kMaxSplits) cap = kMaxSplits;
  if (cap < 1) cap = 1;
  int nsplit = 0;
  if (units * 2 <= sm_count()) {
    // Few (row, kv head) units: one 8-warp CTA per SM, as many splits as fit
    // one wave, so each CTA streams a long key range and the per-CTA work
    // (norm, merges) is paid as few times as possible.
    nsplit = sm_count() / units;
    if (nsplit > cap) nsplit = cap;
  }
  for (int m = 4; m >= 1 && nsplit == 0; --m) {
    const int ns = static_cast<int>((static_cast<long long>(m) * slots) / units);
    if (ns >= 1 && ns <= cap) nsplit = ns;
  }
  if (nsplit == 0) {
    const int want = (slots + units - 1) / units;
    nsplit = want < cap ? want : cap;
  }
  if (nsplit < 1) nsplit = 1;
  int chunk = (span + nsplit - 1) / nsplit;
  chunk = (chunk + 15) / 16 * 16;
  nsplit = (span + chunk - 1) / chunk;
  p.chunk = chunk;
  p.nsplit = nsplit;
  if (nsplit <= 1) {
    p.o_bytes = p.m_bytes = p.t_bytes = p.ws_bytes = 0;
  } else {
    const size_t np = static_cast<size_t>(B) * H * nsplit;
    p.o_bytes = (np * hd * 4 + 255) / 256 * 256;
    p.m_bytes = (np * 4 + 255) / 256 * 256;
    p.t_bytes = (static_cast<size_t>(B) * Hkv * 4 + 255) / 256 * 256;
    p.ws_bytes = p.o_bytes + 2 * p.m_bytes + p.t_bytes;
  }
  return p;
}

}  // namespace g4

// Step a6 (bf16) for short key spans: decode attention over at most 512 keys
// per (sequence, kv head) -- a sliding layer's window, or any layer early in
// a sequence -- with the splits of a (sequence, kv head) merged inside a
// thread-block cluster.
//
// Semantics as in g4_attn_simt.cu (turbospark-runtime gemma4/attn.rs decode:
// keys [kv_start, seq_len) with kv_start = seq_len - sliding_window on sliding
// layers, score scale attn_scale; query head h reads kv head h / (H / Hkv) as
// in taconite-embeddinggemma2 `text_attention`), and the FUSED form appends
// the new token first (cortiq-engine g4e.rs `g4e_forward`: q and k RMS-normed
// with their weights and roped, v normed without weight; k and v written to
// the cache at position L - 1).
//
// Why a second decode kernel: a window of 512 keys is 8 KB of K and V per
// (sequence, kv head) row of 256 bf16 values; streamed through the general
// split-KV kernel it takes a chain of dependent phases (per-warp online
// softmax over 4-key batches, a warp merge, partials through global memory,
// an arrival ticket and a last-CTA merge) that costs far more than the bytes.
// Here the chain is short:
//   * a cluster of NS CTAs per (sequence, kv head), CTA r holding keys
//     [r * 64, r * 64 + 64) of the span: it issues one bulk copy for its K
//     rows and one for its V rows (two each where a ring cache wraps) before
//     anything else, so the copies are in flight during the norm;
//   * fused: cos / sin of the new position in double-float (all threads), the
//     G q rows and, on the CTA holding position L - 1, the new k and v rows
//     normed and roped (one warp per row, the correctly rounded bf16 values
//     of g4_normrope.cuh); k and v go to the cache row and into the CTA's own
//     K / V rows in shared memory, so the new key is scored like the others;
//   * scores of all 64 keys at once: 16 lanes per key (8 for head_dim 64), each
//     lane a 16- or 32-element slice of the key row against the G query slices
//     it holds in registers, the 16-byte pieces read in a rotated order so
//     that the 8 lanes of a shared-memory phase hit 8 distinct bank groups;
//     a reduce-scatter over the key's lanes leaves one head's score per lane;
//   * softmax per head by one warp over the 64 scores (log2 domain, q pre-
//     scaled by attn_scale * log2 e), then P.V by all threads (a dim pair and
//     a slice of the keys each, V read along its rows), the slices summed
//     through shared memory: the CTA's (max, sum, unnormalised output);
//   * the cluster merges the NS partials through distributed shared memory
//     (CTA r owns 1/NS of the G x head_dim outputs and reads the peers'
//     maxima, sums and outputs with ld.shared::cluster), with one cluster
//     barrier before the merge and one before exit.  No global scratch and no
//     arrival counter.
#include <math.h>
#include <string.h>

#include "g4_device.cuh"
#include "g4_internal.h"
#include "g4_normrope.cuh"

namespace g4 {
namespace {

constexpr int kWinKeys = 64;    // keys per CTA
constexpr int kWinThreads = 256;
constexpr int kWinWarps = 8;

template <int HD, int G>
struct WinCfg {
  static constexpr int ROWB = HD * 2;                 // bytes per bf16 row
  static constexpr int LPK = HD >= 128 ? 16 : 8;      // lanes per key in the score pass
  static constexpr int CPL = HD / (8 * LPK);          // 16-byte pieces per lane per key row (1 or 2)
  static constexpr int KPW = 32 / LPK;                // keys per warp per pass
  static constexpr int KPP = kWinWarps * KPW;         // keys per pass
  static constexpr int NPASS = kWinKeys / KPP;
  static constexpr int NDP = HD / 2;                  // dim pairs in the P.V pass
  static constexpr int NKS = kWinThreads / NDP;       // key slices in the P.V pass
  static constexpr int KPS = kWinKeys / NKS;          // keys per slice
  // row layout of the norm (one warp per row), as in g4_normrope.cuh
  static constexpr int EL = HD / 32;
  static constexpr int PE = EL < 8 ? EL : 8;
  static constexpr int NPC = EL / PE;
  // shared memory (bytes)
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + kWinKeys * ROWB;
  static constexpr int QF_OFF = V_OFF + kWinKeys * ROWB;   // [G][HD] f32 query, pre-scaled
  static constexpr int S_OFF = QF_OFF + G * HD * 4;        // [G][64] scores
  static constexpr int P_OFF = S_OFF + G * kWinKeys * 4;   // [64][G] probabilities
  static constexpr int ML_OFF = P_OFF + kWinKeys * G * 4;  // [G] max, [G] sum
  static constexpr int O_OFF = ML_OFF + (2 * G * 4 + 64 + 15) / 16 * 16;  // [G][HD] partial output (16-byte aligned)
  static constexpr int TAB_OFF = O_OFF + G * HD * 4;       // cos, sin of HD/2 pairs (double-float)
  // the cluster leader's receive area: every CTA's partial (output, max, sum)
  static constexpr int RO_OFF = TAB_OFF + HD * 8;           // [8][G][HD] f32
  static constexpr int RM_OFF = RO_OFF + kMaxWinSplits * G * HD * 4;  // [8][G] max
  static constexpr int RL_OFF = RM_OFF + kMaxWinSplits * G * 4;       // [8][G] sum
  static constexpr int BAR_OFF = RL_OFF + kMaxWinSplits * G * 4;
  static constexpr int SMEM_B = BAR_OFF + 16;
  static constexpr int RED_B = NKS * G * HD * 4;           // P.V slice sums, over the K and V rows
  static_assert(RED_B <= 2 * kWinKeys * ROWB, "slice sums fit in the K / V area");
  static_assert(NPASS * KPP == kWinKeys && NKS * KPS == kWinKeys, "tiling");
  static_assert(G <= LPK && G <= kWinWarps, "one head per lane of a key group, one softmax warp per head");
  static constexpr int MINB = G * HD >= 2048 ? 1 : 2;      // CTAs per SM the registers aim for
};

__device__ __forceinline__ float2 fma2w(float2 a, float2 b, float2 c) {
  unsigned long long ua, ub, uc, ud;
  memcpy(&ua, &a, 8);
  memcpy(&ub, &b, 8);
  memcpy(&uc, &c, 8);
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(ud) : "l"(ua), "l"(ub), "l"(uc));
  float2 d;
  memcpy(&d, &ud, 8);
  return d;
}

// Sum over the LPK lanes of a key group of v[i], scattered: lane l of the
// group returns the total of index (l mod LPK) >> log2(LPK / NP).
template <int NP, int LPK>
__device__ __forceinline__ float group_reduce_scatter(float (&v)[NP], int lane) {
  int o = LPK / 2;
#pragma unroll
  for (int n = NP; n > 1; n >>= 1, o >>= 1) {
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
  for (; o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  return r;
}


// Arrive on the cluster barrier without ordering (start of the kernel), and
// the matching wait: after it every CTA of the cluster has started, so its
// shared memory may be written by its peers.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void st_cluster_f32x2(uint32_t addr, float2 v) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(v.x), "f"(v.y) : "memory");
}

template <int HD, int G, bool FUSED>
__global__ void __launch_bounds__(kWinThreads, (WinCfg<HD, G>::MINB))
    decode_win_kernel(const __grid_constant__ AttnSimtArgs a) {
  using C = WinCfg<HD, G>;
  using T = __nv_bfloat16;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sK = smem + C::K_OFF;
  uint8_t* sV = smem + C::V_OFF;
  float* qf = reinterpret_cast<float*>(smem + C::QF_OFF);
  float* s_sc = reinterpret_cast<float*>(smem + C::S_OFF);
  float* s_p = reinterpret_cast<float*>(smem + C::P_OFF);
  float* s_m = reinterpret_cast<float*>(smem + C::ML_OFF);
  float* s_l = s_m + G;
  float* s_o = reinterpret_cast<float*>(smem + C::O_OFF);
  DF* s_cos = reinterpret_cast<DF*>(smem + C::TAB_OFF);
  DF* s_sin = s_cos + HD / 2;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);

  const int ns = a.nsplit;
  const int split = blockIdx.x % ns;  // == the CTA's rank in its cluster
  const int unit = blockIdx.x / ns;
  const int kvh = unit % a.Hkv;
  const int b = unit / a.Hkv;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(bar), 1);
    fence_mbar_init();
  }
  if (a.nsplit > 1) cluster_arrive_relaxed();  // waited for before the first store to a peer

  const size_t head_base = (static_cast<size_t>(b) * a.Hkv + kvh) * a.max_len;
  const T* gk = static_cast<const T*>(a.ck) + head_base * HD;
  const T* gv = static_cast<const T*>(a.cv) + head_base * HD;
  // Keys [kbeg, L) of the sequence; this CTA holds [k0, k0 + n) of them.
  auto first_key = [&](int Lx) { return (a.sliding ? max(0, Lx - a.window) : 0) + split * kWinKeys; };
  auto n_keys = [&](int Lx) { return max(0, min(Lx, first_key(Lx) + kWinKeys) - first_key(Lx)); };
  // cos / sin of position p (all threads; the pairs past n_rot are the identity)
  auto build_table = [&](int p) {
    for (int idx = threadIdx.x; idx < HD; idx += kWinThreads) {
      const int j = idx >> 1, part = idx & 1;
      if (j < a.n_rot) {
        bool to_cos;
        const DF v = sincos_df_part(p, a.inv_freq[j], part, to_cos);
        (to_cos ? s_cos : s_sin)[j] = v;
      } else if (part == 0) {
        s_cos[j] = DF{1.0f, 0.0f};
      } else {
        s_sin[j] = DF{0.0f, 0.0f};
      }
    }
  };

  // ---- while the previous kernel on the stream may still be running
  // (programmatic dependent launch): a speculative read of the sequence's
  // length, the L2 prefetch of the K / V rows it implies and (fused) the
  // cos / sin table of its position.  The prefetch only warms the cache, and
  // the table is rebuilt below unless the length read after the wait agrees,
  // so nothing read here reaches a result.
  const int L_spec = min(max(a.base[b], 1), a.len_cap);
  if (threadIdx.x == 0) {
    const int k0s = first_key(L_spec);
    const int ns_ = n_keys(L_spec);
    if (ns_ > 0) {
      if (!a.ring) {
        prefetch_l2_bulk(gk + static_cast<size_t>(k0s) * HD, static_cast<uint32_t>(ns_) * C::ROWB);
        prefetch_l2_bulk(gv + static_cast<size_t>(k0s) * HD, static_cast<uint32_t>(ns_) * C::ROWB);
      } else {
        const int r0 = k0s % a.max_len;
        const int n0 = min(ns_, a.max_len - r0);
        prefetch_l2_bulk(gk + static_cast<size_t>(r0) * HD, static_cast<uint32_t>(n0) * C::ROWB);
        prefetch_l2_bulk(gv + static_cast<size_t>(r0) * HD, static_cast<uint32_t>(n0) * C::ROWB);
        if (n0 < ns_) {
          prefetch_l2_bulk(gk, static_cast<uint32_t>(ns_ - n0) * C::ROWB);
          prefetch_l2_bulk(gv, static_cast<uint32_t>(ns_ - n0) * C::ROWB);
        }
      }
    }
  }
  if constexpr (FUSED) {
    // the rows the norm reads: the G raw q rows, the new k and v rows, the
    // weights (one 16-byte-multiple prefetch each, by otherwise idle lanes)
    if (warp == kWinWarps - 1 && lane < G + 4) {
      const void* src = nullptr;
      uint32_t bytes = C::ROWB;
      if (lane < G) {
        src = static_cast<const T*>(a.q) + (static_cast<size_t>(b) * a.H + kvh * G + lane) * HD;
      } else if (lane < G + 2) {
        const void* raw = lane == G ? a.k_raw : a.v_raw;
        if (raw != nullptr) src = static_cast<const T*>(raw) + (static_cast<size_t>(b) * a.Hkv + kvh) * HD;
      } else {
        src = lane == G + 2 ? static_cast<const void*>(a.q_w) : static_cast<const void*>(a.k_w);
        bytes = HD * 4;
      }
      if (src != nullptr) prefetch_l2_bulk(src, bytes);
    }
    build_table(L_spec - 1);
  }
  pdl_wait();
  pdl_trigger();

  const int L = min(max(a.base[b], 1), a.len_cap);
  const int k0 = first_key(L);
  const int nvalid = n_keys(L);
  const int k1 = k0 + nvalid;
  // FUSED on a layer that owns its cache: the new key is normed here, not read.
  const bool new_key = FUSED && a.k_raw != nullptr && L - 1 >= k0 && L - 1 < k1;
  const int ncopy = new_key ? nvalid - 1 : nvalid;
  __syncthreads();  // barrier initialised, table built
  if constexpr (FUSED) {
    if (L != L_spec) {  // the length changed under the speculative read: rebuild the table
      build_table(L - 1);
      __syncthreads();
    }
  }
  // The copies are issued by the last warp, which the norm below leaves idle
  // for G <= 5 (issuing them costs a lane several hundred cycles, which would
  // otherwise delay that lane's warp and the norm's barrier).
  if (warp == kWinWarps - 1 && lane == 0) {
    const uint32_t bytes = static_cast<uint32_t>(max(ncopy, 0)) * C::ROWB;
    mbar_arrive_expect_tx(smem_u32(bar), 2 * bytes);
    if (bytes > 0) {
      const uint32_t dk = smem_u32(sK), dv = smem_u32(sV);
      if (!a.ring) {
        bulk_g2s(dk, gk + static_cast<size_t>(k0) * HD, bytes, smem_u32(bar));
        bulk_g2s(dv, gv + static_cast<size_t>(k0) * HD, bytes, smem_u32(bar));
      } else {
        // positions k0 .. k0 + ncopy - 1 in rows r0 .. (wrapping once at most)
        const int r0 = k0 % a.max_len;
        const int n0 = min(ncopy, a.max_len - r0);
        const uint32_t b0 = static_cast<uint32_t>(n0) * C::ROWB;
        bulk_g2s(dk, gk + static_cast<size_t>(r0) * HD, b0, smem_u32(bar));
        bulk_g2s(dv, gv + static_cast<size_t>(r0) * HD, b0, smem_u32(bar));
        if (n0 < ncopy) {
          bulk_g2s(dk + b0, gk, bytes - b0, smem_u32(bar));
          bulk_g2s(dv + b0, gv, bytes - b0, smem_u32(bar));
        }
      }
    }
  }

  // ---- the query (and the new key / value): normed rows into shared memory
  if constexpr (FUSED) {
    const int njobs = G + (new_key ? 2 : 0);
    auto src_of = [&](int job) -> const T* {
      if (job < G) return static_cast<const T*>(a.q) + (static_cast<size_t>(b) * a.H + kvh * G + job) * HD;
      return static_cast<const T*>(job == G ? a.k_raw : a.v_raw) + (static_cast<size_t>(b) * a.Hkv + kvh) * HD;
    };
    auto w_of = [&](int job) -> const float* { return job < G ? a.q_w : (job == G ? a.k_w : nullptr); };
    auto load_job = [&](int job, float* f, float* wf) {
      load_row<T, C::NPC, C::PE>(src_of(job), lane, f);
      const float* w = w_of(job);
      if (w != nullptr) {
        load_row<float, C::NPC, C::PE>(w, lane, wf);
      } else {
#pragma unroll
        for (int i = 0; i < C::EL; ++i) wf[i] = 1.0f;
      }
    };
    float f[C::EL], wf[C::EL];
    for (int job = warp; job < njobs; job += kWinWarps) {
      load_job(job, f, wf);
      norm_rope_row<T, HD, C::NPC, C::PE>(f, wf, job <= G, s_cos, s_sin, a.n_rot, a.eps, lane);
      if (job < G) {
        float g[C::EL];
#pragma unroll
        for (int i = 0; i < C::EL; ++i) g[i] = f[i] * a.scale_log2;
        store_row<float, C::NPC, C::PE>(qf + job * HD, lane, g);
      } else {
        // the new key / value: into the cache row of position L - 1 and this CTA's row of it
        const int row = a.ring ? (L - 1) % a.max_len : L - 1;
        T* dst = static_cast<T*>(job == G ? a.cache_k : a.cache_v) + (head_base + row) * HD;
        store_row<T, C::NPC, C::PE>(dst, lane, f);
        store_row<T, C::NPC, C::PE>(reinterpret_cast<T*>((job == G ? sK : sV) + (L - 1 - k0) * C::ROWB), lane, f);
      }
    }
  } else {
    if (warp < G) {
      float f[C::EL];
      load_row<T, C::NPC, C::PE>(static_cast<const T*>(a.q) + (static_cast<size_t>(b) * a.H + kvh * G + warp) * HD,
                                 lane, f);
#pragma unroll
      for (int i = 0; i < C::EL; ++i) f[i] *= a.scale_log2;
      store_row<float, C::NPC, C::PE>(qf + warp * HD, lane, f);
    }
  }
  __syncthreads();

  // ---- scores: key group of LPK lanes, lane part p holds CPL 16-byte pieces
  const int part = lane % C::LPK;
  const int rot = C::CPL > 1 ? (part >> 2) & 1 : 0;  // piece order (bank groups)
  float2 qr[G][C::CPL][4];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int c = 0; c < C::CPL; ++c) {
      const int pc = (c + rot) & (C::CPL - 1);
      const float4* src = reinterpret_cast<const float4*>(qf + h * HD + (part * C::CPL + pc) * 8);
      const float4 x0 = src[0], x1 = src[1];
      qr[h][c][0] = make_float2(x0.x, x0.y);
      qr[h][c][1] = make_float2(x0.z, x0.w);
      qr[h][c][2] = make_float2(x1.x, x1.y);
      qr[h][c][3] = make_float2(x1.z, x1.w);
    }
  bool ok = warp_wait(smem_u32(bar), 0, a.err);
  constexpr int kSh = ilog2c(C::LPK / G);
  // All passes' partial dot products first (independent accumulators), then
  // their reduce-scatters, so that the passes' dependency chains overlap.
  float part_s[C::NPASS][G];
#pragma unroll
  for (int pass = 0; pass < C::NPASS; ++pass) {
    const int key = pass * C::KPP + warp * C::KPW + lane / C::LPK;
    const int kr = key < nvalid ? key : 0;  // keys past the valid ones read row 0 and are dropped below
    float2 acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int c = 0; c < C::CPL; ++c) {
      const int pc = (c + rot) & (C::CPL - 1);
      const uint4 kw = *reinterpret_cast<const uint4*>(sK + kr * C::ROWB + (part * C::CPL + pc) * 16);
      const float2 k0v = make_float2(bf16_lo(kw.x), bf16_hi(kw.x));
      const float2 k1v = make_float2(bf16_lo(kw.y), bf16_hi(kw.y));
      const float2 k2v = make_float2(bf16_lo(kw.z), bf16_hi(kw.z));
      const float2 k3v = make_float2(bf16_lo(kw.w), bf16_hi(kw.w));
#pragma unroll
      for (int h = 0; h < G; ++h) {
        acc[h] = fma2w(qr[h][c][0], k0v, acc[h]);
        acc[h] = fma2w(qr[h][c][1], k1v, acc[h]);
        acc[h] = fma2w(qr[h][c][2], k2v, acc[h]);
        acc[h] = fma2w(qr[h][c][3], k3v, acc[h]);
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) part_s[pass][h] = key < nvalid ? acc[h].x + acc[h].y : 0.0f;
  }
#pragma unroll
  for (int pass = 0; pass < C::NPASS; ++pass) {
    const int key = pass * C::KPP + warp * C::KPW + lane / C::LPK;
    const float sc = group_reduce_scatter<G, C::LPK>(part_s[pass], lane);
    if ((part & ((1 << kSh) - 1)) == 0) s_sc[(part >> kSh) * kWinKeys + key] = sc;
  }
  __syncthreads();

  // ---- softmax per head (warp h), over this CTA's keys
  if (ns > 1) cluster_wait();  // every CTA of the cluster has started
  if (warp < G) {
    const int h = warp;
    const float v0 = (ok && lane < nvalid) ? s_sc[h * kWinKeys + lane] : -INFINITY;
    const float v1 = (ok && lane + 32 < nvalid) ? s_sc[h * kWinKeys + lane + 32] : -INFINITY;
    float m = fmaxf(v0, v1);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float p0 = m == -INFINITY ? 0.0f : ex2_approx(v0 - m);
    const float p1 = m == -INFINITY ? 0.0f : ex2_approx(v1 - m);
    const float l = warp_sum(p0 + p1);
    s_p[lane * G + h] = p0;
    s_p[(lane + 32) * G + h] = p1;
    if (lane == 0) {
      s_m[h] = m;
      s_l[h] = l;
      if (ns > 1) {
        // this CTA's max and sum go straight to the cluster leader's receive area
        st_cluster_f32(peer_addr(smem_u32(smem + C::RM_OFF) + (split * G + h) * 4, 0), m);
        st_cluster_f32(peer_addr(smem_u32(smem + C::RL_OFF) + (split * G + h) * 4, 0), l);
      }
    }
  }
  __syncthreads();

  // ---- P.V: thread = (dim pair, key slice)
  {
    const int dp = threadIdx.x % C::NDP;
    const int ks = threadIdx.x / C::NDP;
    // every key of the slice, unrolled, four accumulator sets (key index mod
    // 4); keys past this CTA's valid ones read nothing (their rows may hold
    // anything, and their probabilities are zero)
    constexpr int NA = C::KPS >= 4 ? 4 : C::KPS;  // accumulator sets (keys kk mod NA)
    float2 acc[NA][G];
#pragma unroll
    for (int u = 0; u < NA; ++u)
#pragma unroll
      for (int h = 0; h < G; ++h) acc[u][h] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int kk = 0; kk < C::KPS; ++kk) {
      const int key = ks * C::KPS + kk;
      const uint32_t vw = key < nvalid ? *reinterpret_cast<const uint32_t*>(sV + key * C::ROWB + dp * 4) : 0u;
      const float2 vv = make_float2(bf16_lo(vw), bf16_hi(vw));
      float pk[G];
      if constexpr (G % 4 == 0) {
#pragma unroll
        for (int i = 0; i < G / 4; ++i) {
          const float4 x = reinterpret_cast<const float4*>(s_p + key * G)[i];
          pk[4 * i] = x.x; pk[4 * i + 1] = x.y; pk[4 * i + 2] = x.z; pk[4 * i + 3] = x.w;
        }
      } else {
#pragma unroll
        for (int h = 0; h < G; ++h) pk[h] = s_p[key * G + h];
      }
#pragma unroll
      for (int h = 0; h < G; ++h) acc[kk % NA][h] = fma2w(make_float2(pk[h], pk[h]), vv, acc[kk % NA][h]);
    }
    float2 accs[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      accs[h] = acc[0][h];
#pragma unroll
      for (int u = 1; u < NA; ++u) accs[h] = make_float2(accs[h].x + acc[u][h].x, accs[h].y + acc[u][h].y);
    }
    __syncthreads();  // every K / V read is done: the area takes the slice sums
    float2* red = reinterpret_cast<float2*>(smem);  // [NKS][G][HD/2]
#pragma unroll
    for (int h = 0; h < G; ++h) red[(ks * G + h) * C::NDP + dp] = accs[h];
  }
  __syncthreads();
  // The slice sums: this CTA's unnormalised output.  With one CTA it is
  // normalised and written here; in a cluster every CTA stores it into its
  // slot of the leader's receive area, one cluster barrier publishes the
  // slots (release / acquire), and the leader merges them.
  T* out = static_cast<T*>(a.out) + (static_cast<size_t>(b) * a.H + kvh * G) * HD;
  const uint32_t slot_o = peer_addr(smem_u32(smem + C::RO_OFF) + split * G * HD * 4, 0);
  for (int idx = threadIdx.x; idx < G * C::NDP; idx += kWinThreads) {
    const float2* red = reinterpret_cast<const float2*>(smem);
    float2 sum = red[idx];
#pragma unroll
    for (int ks = 1; ks < C::NKS; ++ks) {
      const float2 x = red[ks * G * C::NDP + idx];
      sum.x += x.x;
      sum.y += x.y;
    }
    if (ns == 1)
      reinterpret_cast<float2*>(s_o)[idx] = sum;  // [G][HD]
    else
      st_cluster_f32x2(slot_o + idx * 8, sum);
  }
  if (ns == 1) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * HD; idx += kWinThreads) {
      const float l = s_l[idx / HD];
      const float val = l > 0.0f ? s_o[idx] / l : 0.0f;
      store_elems<1>(out + idx, &val);
    }
  } else {
    cluster_sync_all();
    if (split == 0) {
      const float* ro = reinterpret_cast<const float*>(smem + C::RO_OFF);
      const float* rm = reinterpret_cast<const float*>(smem + C::RM_OFF);
      const float* rl = reinterpret_cast<const float*>(smem + C::RL_OFF);
      // log-sum-exp weight of each (split, head), normalised: all G x ns of
      // them at once, the splits of a head on 8 consecutive lanes of warps
      // 0-1 (ns <= 8, G <= 8), reduced with shuffles
      float* wts = s_sc;  // [ns][G] (the scores are no longer needed)
      static_assert(kMaxWinSplits == 8, "8 lanes per head");
      if (threadIdx.x < 64) {
        const int h = threadIdx.x >> 3, r = threadIdx.x & 7;
        const bool have = h < G && r < ns;
        const float mr = have ? rm[r * G + h] : -INFINITY;
        float M = mr;
#pragma unroll
        for (int o = 4; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float w = mr == -INFINITY ? 0.0f : ex2_approx(mr - M);
        float den = have ? w * rl[r * G + h] : 0.0f;
#pragma unroll
        for (int o = 4; o >= 1; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        if (have) wts[r * G + h] = den > 0.0f ? w / den : 0.0f;
      }
      __syncthreads();
      // four consecutive outputs per thread (G x HD is a multiple of 4 and
      // every partial is 16-byte aligned)
      for (int idx = threadIdx.x * 4; idx < G * HD; idx += kWinThreads * 4) {
        const int h = idx / HD;
        float val[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int r = 0; r < ns; ++r) {
          const float w = wts[r * G + h];
          const float4 x = *reinterpret_cast<const float4*>(ro + r * G * HD + idx);
          val[0] = fmaf(w, x.x, val[0]);
          val[1] = fmaf(w, x.y, val[1]);
          val[2] = fmaf(w, x.z, val[2]);
          val[3] = fmaf(w, x.w, val[3]);
        }
        store_elems<4>(out + idx, val);
      }
    }
  }
  // A copy wait that gave up: wait (bounded) once more for the copies still
  // in flight before the CTA's shared memory goes away.
  if (!ok) warp_wait(smem_u32(bar), 0, nullptr);
}

template <int HD, int G, bool FUSED>
cudaError_t launch_win_hgf(const AttnSimtArgs& a, cudaStream_t s) {
  using C = WinCfg<HD, G>;
  const cudaError_t e = set_smem_limit_once<decode_win_kernel<HD, G, FUSED>>(C::SMEM_B);
  if (e != cudaSuccess) return e;
  const long long nblk = static_cast<long long>(a.nsplit) * a.Hkv * a.B;
  if (nblk <= 0 || nblk > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nblk));
  cfg.blockDim = dim3(kWinThreads);
  cfg.dynamicSmemBytes = C::SMEM_B;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(a.nsplit);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, decode_win_kernel<HD, G, FUSED>, a);
}

template <int HD, int G>
cudaError_t launch_win_hg(const AttnSimtArgs& a, cudaStream_t s) {
  return a.fused ? launch_win_hgf<HD, G, true>(a, s) : launch_win_hgf<HD, G, false>(a, s);
}

template <int HD>
cudaError_t launch_win_h(const AttnSimtArgs& a, cudaStream_t s) {
  switch (a.H / a.Hkv) {
    case 1: return launch_win_hg<HD, 1>(a, s);
    case 2: return launch_win_hg<HD, 2>(a, s);
    case 4: return launch_win_hg<HD, 4>(a, s);
    case 8: return launch_win_hg<HD, 8>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool decode_win_eligible(int dtype, int hd, int group, int span, int units) {
  if (dtype != 1 || !(hd == 64 || hd == 128 || hd == 256) || span < 1 || span > kMaxWinSplits * kWinKeys) return false;
  // One wave of CTAs at most (two per SM, one for group x head_dim 2048): with
  // more, the clusters start over several waves and the split-KV kernel,
  // whose CTAs stream long key ranges, is faster.
  const long long ctas = static_cast<long long>(units) * decode_win_splits(span);
  return ctas <= static_cast<long long>(sm_count()) * (group * hd >= 2048 ? 1 : 2);
}

int decode_win_splits(int span) { return (span + kWinKeys - 1) / kWinKeys; }

cudaError_t launch_decode_win(const AttnSimtArgs& a, cudaStream_t s) {
  if (a.nsplit < 1 || a.nsplit > kMaxWinSplits || a.chunk != kWinKeys || a.mode != 0 || a.T != 1)
    return cudaErrorInvalidValue;
  switch (a.hd) {
    case 64: return launch_win_h<64>(a, s);
    case 128: return launch_win_h<128>(a, s);
    case 256: return launch_win_h<256>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace g4

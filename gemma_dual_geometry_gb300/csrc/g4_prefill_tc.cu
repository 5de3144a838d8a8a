// Step a5 in bf16: causal GQA flash attention on the tcgen05 tensor cores.
//
// Semantics as in g4_attn_simt.cu (cortiq-engine g4e.rs `attend_all_heads`
// with scale 1.0 and the sliding window, ferrox-models gemma4_engine.rs
// `causal_gqa_attention[_windowed]`): o_i = sum_j softmax_j(scale q_i.k_j) v_j
// over keys j <= i (and i - j < window on sliding layers), query head h
// reading kv head h / (H / Hkv).
//
// One CTA computes a 128-query-row tile of one (sequence, head) and, for
// head_dim 512, one 256-wide half of the output columns (two CTAs per tile
// then recompute the same scores; TMEM holds 512 f32 columns per SM and a
// 128 x 512 accumulator alone would fill it).  Warp roles (192 threads):
//   warp 0      TMA producer: the Q tile once, then K chunks (128 keys x 64
//               dims) and V chunks (VK keys x DV dims) through a ring of
//               16 KB shared-memory slots, 128-byte swizzled.
//   warp 1      allocates TMEM and issues tcgen05.mma (one elected lane):
//                 S[j%2] = Q K_j^T      (M=128, N=128, K=head_dim; A, B from
//                                        shared memory, K-major)
//                 O     += P_j V_j      (M=128, N=DV,  K=128; A = P_j from
//                                        TMEM, B = V_j MN-major)
//               in the order QK_0, QK_1, PV_0, QK_2, PV_1, ... so the score
//               MMA of the next tile overlaps the softmax of this one.
//   warps 2-5   softmax, one query row per thread (TMEM lane = row): load S
//               with tcgen05.ld, mask (causal / window / keys past the cache),
//               online softmax in the log2 domain with the running maximum
//               raised only when it grows by more than 2^8 (the stale maximum
//               is exact for O / l), rescale the O row in TMEM when it is
//               raised, and write P as bf16 over the first 64 columns of the
//               same S buffer; finally O / l to global memory.  The row sum
//               l adds the bf16-rounded P values, the weights the PV MMA
//               really applies, so a row dominated by one key returns that
//               key's value without the rounding error of P.
// TMEM columns: S0/P0 [0,128), S1/P1 [128,256), O [256, 256 + DV).
// The MMAs of one thread execute in issue order, so QK_{j+2} (issued after
// PV_j) overwrites P_j only after PV_j has read it; no barrier is needed
// between them.  Barriers come in pairs indexed by tile parity (j % 2), which
// keeps each phase unambiguous for waiters that skip phases.
// Key tiles wholly outside every row's band are never loaded.
#include <math.h>

#include "g4_device.cuh"
#include "g4_internal.h"

namespace g4 {
namespace {

constexpr int kBM = 128;       // query rows per CTA
constexpr int kBN = 128;       // keys per tile
constexpr int kSlotB = 16384;  // ring slot bytes
constexpr int kThreads = 192;
constexpr int kMaxSlots = 12;
constexpr int kSmemMax = 232448;  // opt-in shared memory per block
constexpr float kRescaleLog2 = 8.0f;

template <int HD>
struct TcCfg {
  static constexpr int DV = HD < 256 ? HD : 256;  // output columns per CTA
  static constexpr int NDH = HD / DV;             // CTAs per (tile, head)
  static constexpr int QCH = HD / 64;             // 64-dim chunks of Q and of a K tile
  static constexpr int VK = 8192 / DV;            // keys per V chunk (VK * DV * 2 = 16 KB)
  static constexpr int VCH = kBN / VK;            // V chunks per tile
  static constexpr int Q_OFF = 0;
  static constexpr int RING_OFF = Q_OFF + QCH * kSlotB;
  static constexpr int BAR_B = 512;
  static constexpr int NSLOT_FIT = (kSmemMax - 1024 - BAR_B - RING_OFF) / kSlotB;
  static constexpr int NSLOT = NSLOT_FIT < kMaxSlots ? NSLOT_FIT : kMaxSlots;
  static constexpr int BAR_OFF = RING_OFF + NSLOT * kSlotB;
  static constexpr int SMEM_B = 1024 + BAR_OFF + BAR_B;  // + alignment slack
  static_assert(NSLOT >= 4, "ring depth");
  static_assert(SMEM_B <= kSmemMax, "shared memory budget");
};

struct TcBars {
  uint64_t q_full;
  uint64_t s_full[2];  // QK_j complete (tile parity)
  uint64_t p_full[2];  // P_j written to TMEM by all 128 softmax threads
  uint64_t o_done[2];  // PV_j complete
  uint64_t drain;
  uint64_t full[kMaxSlots];
  uint64_t empty[kMaxSlots];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(TcBars) <= 512, "barrier block");

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ PrefillTcArgs a) {
  using C = TcCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  TcBars* bars = reinterpret_cast<TcBars*>(smem + C::BAR_OFF);
  const uint32_t sQ = smem_u32(smem + C::Q_OFF);
  const uint32_t sRing = smem_u32(smem + C::RING_OFF);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();

  // Block -> (q tile, sequence, head, output half); heaviest (last) tiles first.
  const int nqt = (a.T + kBM - 1) / kBM;
  int idx = blockIdx.x;
  const int dh = idx % C::NDH;
  idx /= C::NDH;
  const int h = idx % a.H;
  idx /= a.H;
  const int b = idx % a.B;
  const int qt = nqt - 1 - idx / a.B;
  const int kvh = h / (a.H / a.Hkv);

  const int q_start = a.q_start[b];
  const int q0 = qt * kBM;
  const int valid_rows = min(kBM, a.T - q0);
  const int qpos_first = q_start + q0;
  const int qpos_last = qpos_first + valid_rows - 1;
  const int Lk = min(q_start + a.T, a.max_len);  // cache rows holding keys
  const int kend = min(qpos_last + 1, Lk);
  const int kbeg = a.sliding ? max(0, qpos_first - a.window + 1) : 0;
  const int kt_begin = kbeg / kBN;
  const int ntiles = max(0, (kend + kBN - 1) / kBN - kt_begin);

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->q_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->s_full[i]), 1);
      mbar_init(smem_u32(&bars->p_full[i]), 128);
      mbar_init(smem_u32(&bars->o_done[i]), 1);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(smem_u32(&bars->full[i]), 1);
      mbar_init(smem_u32(&bars->empty[i]), 1);
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t tmem_O = tmem + 256;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int seq = 0;
    if (lane == 0 && ntiles > 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      const uint32_t qb = smem_u32(&bars->q_full);
      mbar_arrive_expect_tx(qb, C::QCH * kSlotB);
      for (int c = 0; c < C::QCH; ++c) tma_load_4d(sQ + c * kSlotB, &tm_q, c * 64, h, q0, b, qb);
    }
    bool ok = true;
    auto acquire = [&](int& slot) -> bool {
      slot = seq % C::NSLOT;
      const uint32_t par = ((seq / C::NSLOT) & 1) ^ 1;
      return warp_wait(smem_u32(&bars->empty[slot]), par, a.err, abort);
    };
    auto load_k = [&](int kt) {
      for (int c = 0; c < C::QCH && ok; ++c) {
        int slot;
        if (!acquire(slot)) { ok = false; break; }
        if (lane == 0) {
          const uint32_t fb = smem_u32(&bars->full[slot]);
          mbar_arrive_expect_tx(fb, kSlotB);
          tma_load_4d(sRing + slot * kSlotB, &tm_k, c * 64, kt * kBN, kvh, b, fb);
        }
        __syncwarp();
        ++seq;
      }
    };
    auto load_v = [&](int kt) {
      for (int c = 0; c < C::VCH && ok; ++c) {
        int slot;
        if (!acquire(slot)) { ok = false; break; }
        if (lane == 0) {
          const uint32_t fb = smem_u32(&bars->full[slot]);
          mbar_arrive_expect_tx(fb, kSlotB);
          for (int dc = 0; dc < C::DV / 64; ++dc)
            tma_load_4d(sRing + slot * kSlotB + dc * C::VK * 128, &tm_v, dh * C::DV + dc * 64,
                        kt * kBN + c * C::VK, kvh, b, fb);
        }
        __syncwarp();
        ++seq;
      }
    };
    if (ntiles > 0) {
      load_k(kt_begin);
      for (int j = 0; j < ntiles && ok; ++j) {
        if (j + 1 < ntiles) load_k(kt_begin + j + 1);
        load_v(kt_begin + j);
      }
      // Copies still in flight must land before the CTA may exit.
      warp_wait(smem_u32(&bars->q_full), 0, nullptr);
      for (int s = max(0, seq - C::NSLOT); s < seq; ++s)
        warp_wait(smem_u32(&bars->full[s % C::NSLOT]), (s / C::NSLOT) & 1, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (ntiles > 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, C::DV, 0, 1);
      int seq = 0;
      bool ok = warp_wait(smem_u32(&bars->q_full), 0, a.err, abort);
      tc_fence_after();
      auto mma_qk = [&](int j) {
        const int sb = j & 1;
        const uint32_t dS = tmem + sb * kBN;
        for (int c = 0; c < C::QCH; ++c) {
          const int slot = seq % C::NSLOT;
          if (!warp_wait(smem_u32(&bars->full[slot]), (seq / C::NSLOT) & 1, a.err, abort)) { ok = false; return; }
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = smem_desc_sw128(sQ + c * kSlotB + kk * 32, 16, 1024);
              const uint64_t bd = smem_desc_sw128(sRing + slot * kSlotB + kk * 32, 16, 1024);
              tc_mma_ss(dS, ad, bd, idesc_qk, (c > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(smem_u32(&bars->empty[slot]));
          }
          __syncwarp();
          ++seq;
        }
        if (lane == 0) tc_commit(smem_u32(&bars->s_full[sb]));
        __syncwarp();
      };
      auto mma_pv = [&](int j) {
        const int sb = j & 1;
        if (!warp_wait(smem_u32(&bars->p_full[sb]), (j >> 1) & 1, a.err, abort)) { ok = false; return; }
        tc_fence_after();
        const int kt = kt_begin + j;
        const uint32_t tP = tmem + sb * kBN;  // P_j: 128 keys as 64 packed columns
        for (int c = 0; c < C::VCH; ++c) {
          const int slot = seq % C::NSLOT;
          if (!warp_wait(smem_u32(&bars->full[slot]), (seq / C::NSLOT) & 1, a.err, abort)) { ok = false; return; }
          // Rows of keys past the cache's filled length may hold anything
          // (even NaN, and 0 * NaN = NaN); zero them before they meet P.
          const int key0 = kt * kBN + c * C::VK;
          const int nvalid = min(C::VK, max(0, Lk - key0));
          if (nvalid < C::VK) {
            uint8_t* slot_ptr = smem + C::RING_OFF + slot * kSlotB;
            const int nbad = C::VK - nvalid;
            for (int i = lane; i < (C::DV / 64) * nbad * 8; i += 32) {
              const int dc = i / (nbad * 8);
              const int rr = (i / 8) % nbad + nvalid;
              const int pc = i % 8;
              *reinterpret_cast<uint4*>(slot_ptr + dc * C::VK * 128 + rr * 128 + pc * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < C::VK / 16; ++kk) {
              const int kp = c * C::VK + kk * 16;  // key offset inside the tile
              const uint64_t bd = smem_desc_sw128(sRing + slot * kSlotB + kk * 2048, C::VK * 128, 1024);
              tc_mma_ts(tmem_O, tP + kp / 2, bd, idesc_pv, (j > 0 || c > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(smem_u32(&bars->empty[slot]));
          }
          __syncwarp();
          ++seq;
        }
        if (lane == 0) tc_commit(smem_u32(&bars->o_done[sb]));
        __syncwarp();
      };
      if (ok) mma_qk(0);
      for (int j = 0; j < ntiles && ok; ++j) {
        if (j + 1 < ntiles) mma_qk(j + 1);
        if (ok) mma_pv(j);
      }
      // Every MMA issued so far completes before TMEM is released.
      if (lane == 0) tc_commit(smem_u32(&bars->drain));
      __syncwarp();
      warp_wait(smem_u32(&bars->drain), 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int qpos = qpos_first + r;
    const bool row_valid = r < valid_rows;
    const float c2 = a.scale_log2;  // > 0 (checked on the host)
    float m = -INFINITY;  // exponent base in log2 units: a stale running maximum
    float l = 0.0f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int sb = j & 1;
      if (!warp_wait(smem_u32(&bars->s_full[sb]), (j >> 1) & 1, a.err, abort)) { ok = false; break; }
      tc_fence_after();
      float s[kBN];
      {
        uint32_t r0[32], r1[32], r2[32], r3[32];
        const uint32_t tS = tmem + lane_off + sb * kBN;
        tmem_ld32(tS, r0);
        tmem_ld32(tS + 32, r1);
        tmem_ld32(tS + 64, r2);
        tmem_ld32(tS + 96, r3);
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = __uint_as_float(r0[i]);
          s[32 + i] = __uint_as_float(r1[i]);
          s[64 + i] = __uint_as_float(r2[i]);
          s[96 + i] = __uint_as_float(r3[i]);
        }
      }

      const int k0 = (kt_begin + j) * kBN;
      const bool all_vis = row_valid && (k0 + kBN - 1 <= qpos) && (k0 + kBN <= Lk) &&
                           (!a.sliding || qpos - k0 < a.window);
      if (!all_vis) {
#pragma unroll
        for (int n = 0; n < kBN; ++n) {
          const int kp = k0 + n;
          const bool vis = row_valid && kp <= qpos && kp < Lk && (!a.sliding || qpos - kp < a.window);
          if (!vis) s[n] = -INFINITY;
        }
      }
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int n = 0; n < kBN; ++n) mx[n & 3] = fmaxf(mx[n & 3], s[n]);
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * c2;
      float alpha = 1.0f;
      bool rescale = false;
      float m_use = m;
      if (m == -INFINITY) {
        m_use = mt;  // nothing accumulated yet (O row is zero or unwritten)
      } else if (mt - m > kRescaleLog2) {
        m_use = mt;
        alpha = ex2_approx(m - mt);
        rescale = true;
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // A row of this warp raises its base (only after a tile with a
        // visible key, so j > 0): PV_{j-1} must be complete before the O
        // rows are scaled; PV_j is not issued until P_j below is published.
        if (!warp_wait(smem_u32(&bars->o_done[(j - 1) & 1]), ((j - 1) >> 1) & 1, a.err, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float f = rescale ? alpha : 1.0f;
#pragma unroll 1
        for (int cc = 0; cc < C::DV / 32; ++cc) {
          uint32_t rr[32];
          tmem_ld32(tmem_O + lane_off + cc * 32, rr);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * f);
          tmem_st32(tmem_O + lane_off + cc * 32, rr);
        }
        tc_wait_st();
      }
      const float nb = (m_use == -INFINITY) ? 0.0f : -m_use;
      uint32_t p0[32], p1[32];
      float sa[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const uint32_t w0 = pack_bf16x2(ex2_approx(fmaf(s[2 * i], c2, nb)), ex2_approx(fmaf(s[2 * i + 1], c2, nb)));
        const uint32_t w1 =
            pack_bf16x2(ex2_approx(fmaf(s[64 + 2 * i], c2, nb)), ex2_approx(fmaf(s[64 + 2 * i + 1], c2, nb)));
        p0[i] = w0;
        p1[i] = w1;
        sa[0] += bf16_lo(w0);
        sa[1] += bf16_hi(w0);
        sa[2] += bf16_lo(w1);
        sa[3] += bf16_hi(w1);
      }
      tmem_st32(tmem + lane_off + sb * kBN, p0);
      tmem_st32(tmem + lane_off + sb * kBN + 32, p1);
      l = l * alpha + ((sa[0] + sa[1]) + (sa[2] + sa[3]));
      m = m_use;
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars->p_full[sb]));
    }
    if (ntiles > 0 && ok) {
      const int jl = ntiles - 1;
      if (warp_wait(smem_u32(&bars->o_done[jl & 1]), (jl >> 1) & 1, a.err, abort)) {
        tc_fence_after();
        const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) +
                             (((static_cast<size_t>(b) * a.T + q0 + r) * a.H + h) * HD + dh * C::DV);
#pragma unroll 1
        for (int cc = 0; cc < C::DV / 32; ++cc) {
          uint32_t rr[32];
          tmem_ld32(tmem_O + lane_off + cc * 32, rr);
          tc_wait_ld();
          if (row_valid) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(rr[8 * i + 0]) * inv_l, __uint_as_float(rr[8 * i + 1]) * inv_l);
              v.y = pack_bf16x2(__uint_as_float(rr[8 * i + 2]) * inv_l, __uint_as_float(rr[8 * i + 3]) * inv_l);
              v.z = pack_bf16x2(__uint_as_float(rr[8 * i + 4]) * inv_l, __uint_as_float(rr[8 * i + 5]) * inv_l);
              v.w = pack_bf16x2(__uint_as_float(rr[8 * i + 6]) * inv_l, __uint_as_float(rr[8 * i + 7]) * inv_l);
              reinterpret_cast<uint4*>(dst + cc * 32)[i] = v;
            }
          }
        }
      }
    } else if (ntiles == 0 && r < valid_rows) {
      // No visible key (only reachable with out-of-contract positions).
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) +
                           (((static_cast<size_t>(b) * a.T + q0 + r) * a.H + h) * HD + dh * C::DV);
      for (int i = 0; i < C::DV / 8; ++i) reinterpret_cast<uint4*>(dst)[i] = make_uint4(0, 0, 0, 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// bf16 4-D tensor map, dims innermost first, 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap* m, const void* base, const cuuint64_t dims[4], const cuuint64_t strides_bytes[3],
              const cuuint32_t box[4]) {
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) return false;
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides_bytes, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int HD>
cudaError_t launch_hd(const PrefillTcArgs& a, cudaStream_t s) {
  using C = TcCfg<HD>;
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(prefill_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_B);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  CUtensorMap mq, mk, mv;
  const cuuint64_t row_b = static_cast<cuuint64_t>(HD) * 2;
  {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(a.H),
                                static_cast<cuuint64_t>(a.T), static_cast<cuuint64_t>(a.B)};
    const cuuint64_t str[3] = {row_b, row_b * a.H, row_b * a.H * a.T};
    const cuuint32_t box[4] = {64, 1, kBM, 1};
    if (!make_map(&mq, a.q, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(a.max_len),
                                static_cast<cuuint64_t>(a.Hkv), static_cast<cuuint64_t>(a.B)};
    const cuuint64_t str[3] = {row_b, row_b * a.max_len, row_b * a.max_len * a.Hkv};
    const cuuint32_t boxk[4] = {64, kBN, 1, 1};
    const cuuint32_t boxv[4] = {64, static_cast<cuuint32_t>(C::VK), 1, 1};
    if (!make_map(&mk, a.ck, dims, str, boxk)) return cudaErrorInvalidValue;
    if (!make_map(&mv, a.cv, dims, str, boxv)) return cudaErrorInvalidValue;
  }
  const int nqt = (a.T + kBM - 1) / kBM;
  const long long nblk = static_cast<long long>(nqt) * a.H * a.B * C::NDH;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nblk));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM_B;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<HD>, mq, mk, mv, a);
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillTcArgs& a, cudaStream_t s) {
  switch (a.hd) {
    case 64: return launch_hd<64>(a, s);
    case 128: return launch_hd<128>(a, s);
    case 256: return launch_hd<256>(a, s);
    case 512: return launch_hd<512>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace g4

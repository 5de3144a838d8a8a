// The steps before and after the attention path, on the tcgen05 tensor cores:
// a bf16 GEMM out = A . Bw^T with float32 accumulation in TMEM whose epilogue
// is the surrounding per-row work.
//
//   epi 0, the q / k / v projections fused into the append (cortiq-engine
//     g4e.rs `g4e_forward`: `rms(h, attn_norm)`, then `matvec` with wq / wk /
//     wv, then the per-head norm and RoPE of q and k and the cache append;
//     turbospark-runtime gemma4/attn.rs writes the projections straight into
//     the KV slot and norms / ropes them there).  A = the layer input x
//     [M = B*T][K = D]; Bw = the q, k and v projection rows stacked, [N][D],
//     with the attention-norm weight folded into their columns (taconite-
//     embeddinggemma2 model.rs multiplies RMSNorm weights into its GEMM
//     operands the same way), so the input RMSNorm leaves only a per-row
//     scale (mean(x^2) + eps)^-1/2, which the epilogue warps compute from the
//     A tiles as they stream through shared memory.  The N tile is one head
//     (head_dim columns): q heads, then k heads, then v heads.  Each
//     epilogue thread owns one token row of the head: it forms y = scale *
//     acc, the head's RMSNorm (with q_norm / k_norm, none on v), rotate_half
//     RoPE on q and k (the pair j, j + head_dim/2 sits in the same thread),
//     and stores bf16 (round to nearest even) to q_out or the cache row of
//     the token's position (position mod max_len on a ring).
//   epi 1, o_proj + post-attention norm + residual (cortiq-engine g4e.rs
//     `g4e_forward` sandwich norm; ferrox-models gemma4_engine.rs
//     `forward_token_on_worker`: `o_proj`, `post_attn_norm`, added to
//     `hidden`).  A = attention output rows [M][H*hd], Bw = Wo [D][H*hd].  The
//     norm runs over a row's D columns, which a cluster of D / 256 CTAs
//     (256 columns each) holds between them: each thread sums its row's
//     squares over its 256 columns, the sums meet through distributed shared
//     memory, and every CTA writes h + y (sum/D + eps)^-1/2 w for its columns.
//
// One CTA per 128 x BN output tile (BN = head_dim or 256), 192 threads:
//   warp 0       TMA producer (one lane): per 64-wide K step the A box
//                (128 rows x 64) and the Bw box(es) (<= 256 rows x 64), 128-byte
//                swizzled, into a ring of stages;
//   warp 1       allocates TMEM; one lane issues the MMAs (M = 128, N <= 256,
//                K = 16; both operands K-major from shared memory) and
//                commits each stage back to the producer;
//   warps 2-5    epilogue, one TMEM lane quarter each (thread = tile row):
//                during the main loop (epi 0) the row sums of squares of A;
//                then the accumulator through tcgen05.ld, 32 columns at a time.
// Tiles are ordered with N fastest, so the CTAs working at the same time
// share their A rows in L2; the Bw operand (a few tens of MB) stays in L2.
#include <math.h>

#include <mutex>

#include "g4_device.cuh"
#include "g4_internal.h"
#include "g4_normrope.cuh"

namespace g4 {
namespace {

constexpr int kGM = 128;         // rows per tile
constexpr int kGK = 64;          // K per stage: one 128-byte swizzled row per tile row
constexpr int kGThreads = 192;
constexpr int kGSmemMax = 232448;

template <int BN>
struct GemmCfg {
  static constexpr int A_B = kGM * kGK * 2;               // 16 KB
  static constexpr int B_B = BN * kGK * 2;                // BN x 128 B
  static constexpr int STAGE_B = A_B + B_B;
  static constexpr int BAR_B = 4096;  // barriers (1 KB), then the epilogue's weight row (<= 512 floats)
  // Tiles of up to 256 columns run two CTAs per SM (TMEM: 2 x 256 columns),
  // so one CTA's epilogue overlaps the other's main loop; 512 columns fill
  // TMEM and take the SM alone.
  static constexpr int CTAS_PER_SM = BN <= 256 ? 2 : 1;
  static constexpr int SMEM_BUDGET = CTAS_PER_SM == 2 ? 113 * 1024 : kGSmemMax;
  static constexpr int NST_FIT = (SMEM_BUDGET - BAR_B) / STAGE_B;
  static constexpr int NSTAGE = NST_FIT > 6 ? 6 : NST_FIT;
  static constexpr int BAR_OFF = NSTAGE * STAGE_B;
  static constexpr int SMEM_B = BAR_OFF + BAR_B;
  static constexpr int MMA_N = BN > 256 ? 256 : BN;       // N of one MMA
  static constexpr int NMMA = BN / MMA_N;                 // MMAs per 16-wide K substep
  static constexpr int NBOX = NMMA;                       // Bw boxes per stage (<= 256 rows each)
  static constexpr uint32_t TMEM_COLS = BN < 32 ? 32 : BN;
  static_assert(NSTAGE >= 2, "stages");
  static_assert(MMA_N % 16 == 0 && MMA_N >= 16, "MMA N");
};

struct GemmBars {
  uint64_t full[6];
  uint64_t empty[6];
  uint64_t acc_full;
  uint32_t tmem_base;
  int abort;
  float red[kGM];  // epi 1: this CTA's per-row sums of squares (read by the cluster)
};
static_assert(sizeof(GemmBars) <= 1024, "barrier block");

// The 128 epilogue threads meet (named barrier 1).
__device__ __forceinline__ void epilogue_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// cos and sin of pos * f in float32, to about 2^-21 absolute (the stored
// values are bf16, 2^-9 relative): the product split exactly into hi + lo
// (one fma), Cody-Waite reduction by 2 pi in three parts (C1 has 8
// significant bits, so k C1 is exact for |k| < 2^16, i.e. angles below
// 4 x 10^5 rad; the other two parts take the rest of 2 pi), then the
// hardware sine / cosine on [-pi, pi].  Positions at or above 2^24 (not
// exact in float) reduce in float64.
__device__ __forceinline__ void rope_cos_sin(int pos, float f, float& c, float& s) {
  constexpr float kInv2Pi = 0x1.45f306p-3f;
  constexpr float C1 = 0x1.92p+2f, C2 = 0x1.fb5444p-10f, C3 = 0x1.68c234p-37f;  // C1 + C2 + C3 = 2 pi (to 4e-19)
  float r;
  if (pos < (1 << 24)) {
    const float p = static_cast<float>(pos);
    const float hi = p * f;
    const float lo = fmaf(p, f, -hi);
    const float k = rintf(hi * kInv2Pi);
    r = fmaf(-k, C1, hi);
    r = fmaf(-k, C2, r);
    r = fmaf(-k, C3, r) + lo;
  } else {
    const double th = static_cast<double>(pos) * static_cast<double>(f);
    const double k = rint(th * 0.15915494309189533577);
    r = static_cast<float>(fma(-k, 6.2831853071795864769, th));
  }
  __sincosf(r, &s, &c);
}

template <int BN, int EPI>
__global__ void __launch_bounds__(kGThreads, (GemmCfg<BN>::CTAS_PER_SM))
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const __grid_constant__ GemmArgs a) {
  using C = GemmCfg<BN>;
  extern __shared__ __align__(1024) uint8_t smem[];
  GemmBars* bars = reinterpret_cast<GemmBars*>(smem + C::BAR_OFF);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_tile = blockIdx.x;
  const int m0 = blockIdx.y * kGM;
  const int n0 = n_tile * BN;
  const int nk = a.K / kGK;
  // 128-byte swizzled tiles need 1024-byte alignment: a block without it
  // records the error and skips its work (every thread still meets the
  // barriers below).
  const bool aligned = (smem_u32(smem) & 1023u) == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NSTAGE; ++i) {
      mbar_init(smem_u32(&bars->full[i]), 1);
      // released by the MMA commit and, in epi 0, by the four epilogue warps
      // once they have summed the A rows' squares
      mbar_init(smem_u32(&bars->empty[i]), EPI == 0 ? 5 : 1);
    }
    mbar_init(smem_u32(&bars->acc_full), 1);
    bars->abort = aligned ? 0 : 1;
    fence_mbar_init();
    if (!aligned) atomicExch(a.err, kErrSmemAlign);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  pdl_trigger();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t sbase = smem_u32(smem);
  auto sA = [&](int s) { return sbase + s * C::STAGE_B; };
  auto sB = [&](int s) { return sbase + s * C::STAGE_B + C::A_B; };

  float row_sq = 0.0f;  // epilogue thread: its row's sum of squares (of A in epi 0, of the tile in epi 1)
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The warp runs the loop converged; one elected lane posts each stage's
    // byte count and issues its copies.
    if (aligned) {
      if (elect_one()) {
        prefetch_tensormap(&tm_a);
        prefetch_tensormap(&tm_b);
      }
      __syncwarp();
      int issued = 0;
      for (int k = 0; k < nk; ++k) {
        const int s = k % C::NSTAGE;
        const uint32_t ph = (k / C::NSTAGE) & 1;
        if (k >= C::NSTAGE && !warp_wait(smem_u32(&bars->empty[s]), ph ^ 1u, a.err, abort)) break;
        const uint32_t fb = smem_u32(&bars->full[s]);
        if (elect_one()) {
          mbar_arrive_expect_tx(fb, C::STAGE_B);
          tma_load_2d(sA(s), &tm_a, k * kGK, m0, fb);
#pragma unroll
          for (int bx = 0; bx < C::NBOX; ++bx)
            tma_load_2d(sB(s) + bx * C::MMA_N * 128, &tm_b, k * kGK, n0 + bx * C::MMA_N, fb);
        }
        __syncwarp();
        issued = k + 1;
      }
      // copies still in flight must land before the CTA may exit
      for (int k = issued > C::NSTAGE ? issued - C::NSTAGE : 0; k < issued; ++k)
        warp_wait(smem_u32(&bars->full[k % C::NSTAGE]), (k / C::NSTAGE) & 1, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The warp runs the loop converged and one elected lane issues each MMA
    // and commit (run by one lane inside a lane test, the loop issued MMAs
    // slower than the tensor pipe executes them).
    if (aligned) {
      constexpr uint32_t idesc = idesc_bf16_f32(kGM, C::MMA_N, 0, 0);
      bool ok = true;
      for (int k = 0; k < nk && ok; ++k) {
        const int s = k % C::NSTAGE;
        if (!warp_wait(smem_u32(&bars->full[s]), (k / C::NSTAGE) & 1, a.err, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = smem_desc_sw128(sA(s), 16, 1024);
        const uint64_t bd = smem_desc_sw128(sB(s), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kGK / 16; ++kk)
#pragma unroll
          for (int nm = 0; nm < C::NMMA; ++nm)
            tc_mma_ss_elect(tmem + nm * C::MMA_N, ad + 2 * kk, bd + 2 * kk + nm * ((C::MMA_N * 128) >> 4), idesc,
                            (k > 0 || kk > 0) ? 1u : 0u);
        tc_commit_elect(smem_u32(&bars->empty[s]));
      }
      // acc_full: every MMA issued has completed (also on the way out after
      // an abort, so TMEM is not released under a running MMA)
      tc_commit_elect(smem_u32(&bars->acc_full));
      warp_wait(smem_u32(&bars->acc_full), 0, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;  // tile row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = aligned;
    // this tile's weight row into shared memory (read by every thread per
    // column): the head's q_norm / k_norm weight (epi 0; none on v heads),
    // the post-attention norm weight of the tile's columns (epi 1)
    {
      float* s_w = reinterpret_cast<float*>(smem + C::BAR_OFF + 1024);
      const float* wsrc = nullptr;
      if constexpr (EPI == 0) {
        wsrc = n_tile < a.H ? a.q_w : (n_tile < a.H + a.Hkv ? a.k_w : nullptr);
      } else {
        wsrc = a.post_w + n0;
      }
      const int t = threadIdx.x - 64;
      for (int i = t; i < BN; i += 128) s_w[i] = wsrc != nullptr ? wsrc[i] : 1.0f;
      epilogue_sync();
    }
    if constexpr (EPI == 0) {
      // the input RMSNorm's sum of squares of row m, from the A tiles in flight
      for (int k = 0; k < nk && ok; ++k) {
        const int s = k % C::NSTAGE;
        if (!warp_wait(smem_u32(&bars->full[s]), (k / C::NSTAGE) & 1, a.err, abort)) {
          ok = false;
          break;
        }
        // row m's 128 bytes: 16-byte pieces at (piece ^ (m & 7)); the order
        // of the pieces does not matter for the sum
        const uint8_t* row = smem + s * C::STAGE_B + m * 128;
        float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll
        for (int pc = 0; pc < 8; ++pc) {
          const uint4 w = *reinterpret_cast<const uint4*>(row + pc * 16);
          const float x0 = bf16_lo(w.x), x1 = bf16_hi(w.x), x2 = bf16_lo(w.y), x3 = bf16_hi(w.y);
          const float x4 = bf16_lo(w.z), x5 = bf16_hi(w.z), x6 = bf16_lo(w.w), x7 = bf16_hi(w.w);
          acc0 = fmaf(x0, x0, fmaf(x1, x1, fmaf(x2, x2, fmaf(x3, x3, acc0))));
          acc1 = fmaf(x4, x4, fmaf(x5, x5, fmaf(x6, x6, fmaf(x7, x7, acc1))));
        }
        row_sq += acc0 + acc1;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->empty[s]));
      }
    }
    if (ok && !warp_wait(smem_u32(&bars->acc_full), 0, a.err, abort)) ok = false;
    tc_fence_after();
    const int gm = m0 + m;
    const bool row_valid = gm < a.M;
    if constexpr (EPI == 0) {
      if (ok) {
        const int hd = BN;
        const int hn = n_tile;  // head: q heads, then k heads, then v heads
        const int kind = hn < a.H ? 0 : (hn < a.H + a.Hkv ? 1 : 2);
        const float* s_w = reinterpret_cast<const float*>(smem + C::BAR_OFF + 1024);  // ones on v heads
        const bool rope = kind < 2;
        // input norm row scale, then this head's sum of squares of acc
        const float rx = __frsqrt_rn(fmaf(row_sq, 1.0f / static_cast<float>(a.K), a.eps_in));
        float ss = 0.0f;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + c * 32, r);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ss = fmaf(__uint_as_float(r[i]), __uint_as_float(r[i]), ss);
        }
        // y = rx acc; the head's norm: (mean(y^2) + eps)^-1/2
        const float inv = __frsqrt_rn(fmaf(rx * rx, ss * (1.0f / static_cast<float>(hd)), a.eps));
        const float scale = rx * inv;
        // destination row
        __nv_bfloat16* dst = nullptr;
        int pos = 0;
        if (row_valid) {
          const int b = gm / a.T;
          pos = a.positions[gm];
          if (kind == 0) {
            dst = static_cast<__nv_bfloat16*>(a.q_out) + (static_cast<size_t>(gm) * a.H + hn) * hd;
          } else if (pos >= 0 && (a.ring || pos < a.max_len)) {
            const int kvh = hn - a.H - (kind == 2 ? a.Hkv : 0);
            const int row = a.ring ? pos % a.max_len : pos;
            dst = static_cast<__nv_bfloat16*>(kind == 1 ? a.cache_k : a.cache_v) +
                  ((static_cast<size_t>(b) * a.Hkv + kvh) * a.max_len + row) * hd;
          }
        }
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
          uint32_t lo[32], hi[32];
          tmem_ld32(tmem + lane_off + c * 32, lo);
          tmem_ld32(tmem + lane_off + BN / 2 + c * 32, hi);
          tc_wait_ld();
          uint32_t plo[16], phi[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float oa[2], ob[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int j = c * 32 + i + e;
              const float ya = __uint_as_float(lo[i + e]) * scale * s_w[j];
              const float yb = __uint_as_float(hi[i + e]) * scale * s_w[j + BN / 2];
              if (rope && j < a.n_rot) {
                float cj, sj;
                rope_cos_sin(pos, a.inv_freq[j], cj, sj);
                oa[e] = fmaf(ya, cj, -(yb * sj));
                ob[e] = fmaf(yb, cj, ya * sj);
              } else {
                oa[e] = ya;
                ob[e] = yb;
              }
            }
            plo[i / 2] = pack_bf16x2(oa[0], oa[1]);
            phi[i / 2] = pack_bf16x2(ob[0], ob[1]);
          }
          if (dst != nullptr) {
            uint4* dl = reinterpret_cast<uint4*>(dst + c * 32);
            uint4* dh = reinterpret_cast<uint4*>(dst + BN / 2 + c * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              dl[q] = make_uint4(plo[4 * q], plo[4 * q + 1], plo[4 * q + 2], plo[4 * q + 3]);
              dh[q] = make_uint4(phi[4 * q], phi[4 * q + 1], phi[4 * q + 2], phi[4 * q + 3]);
            }
          }
        }
      }
    } else {
      // epi 1, first half: this CTA's share of the row's sum of squares
      if (ok) {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + c * 32, r);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) row_sq = fmaf(__uint_as_float(r[i]), __uint_as_float(r[i]), row_sq);
        }
      }
      bars->red[m] = row_sq;
    }
  }

  if constexpr (EPI == 1) {
    // the cluster's CTAs hold the row's other columns: their sums meet here
    const uint32_t csize = gridDim.x;  // one cluster spans the N tiles of a row block
    cluster_sync_all();
    if (warp >= 2) {
      const int quarter = warp & 3;
      const int m = quarter * 32 + lane;
      const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
      const int gm = m0 + m;
      float tot = 0.0f;
      const uint32_t my = smem_u32(&bars->red[m]);
      for (uint32_t r = 0; r < csize; ++r) tot += ld_cluster_f32(peer_addr(my, r));
      const float rn = __frsqrt_rn(fmaf(tot, 1.0f / static_cast<float>(a.N), a.eps));
      const bool live = *abort == 0;
      if (live) {
        const float* s_w = reinterpret_cast<const float*>(smem + C::BAR_OFF + 1024);
        const bool rv = gm < a.M;
        const uint4* hrow = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.h) +
                                                           static_cast<size_t>(rv ? gm : 0) * a.N + n0);
        uint4* orow = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) +
                                               static_cast<size_t>(rv ? gm : 0) * a.N + n0);
        // the residual's 32-column pieces, one piece ahead of the columns in use
        uint4 hcur[4], hnext[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) hcur[q] = rv ? hrow[q] : make_uint4(0, 0, 0, 0);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          if (c + 1 < BN / 32) {
#pragma unroll
            for (int q = 0; q < 4; ++q) hnext[q] = rv ? hrow[(c + 1) * 4 + q] : make_uint4(0, 0, 0, 0);
          }
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + c * 32, r);
          tc_wait_ld();
          if (rv) {
            uint32_t ov[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t hw[4] = {hcur[q].x, hcur[q].y, hcur[q].z, hcur[q].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int i = q * 8 + e * 2;
                const float y0 = fmaf(__uint_as_float(r[i]) * rn, s_w[c * 32 + i], bf16_lo(hw[e]));
                const float y1 = fmaf(__uint_as_float(r[i + 1]) * rn, s_w[c * 32 + i + 1], bf16_hi(hw[e]));
                ov[q * 4 + e] = pack_bf16x2(y0, y1);
              }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
              orow[c * 4 + q] = make_uint4(ov[4 * q], ov[4 * q + 1], ov[4 * q + 2], ov[4 * q + 3]);
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) hcur[q] = hnext[q];
        }
      }
    }
    cluster_sync_all();  // the peers have read this CTA's row sums
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 [rows][K] row-major, K contiguous: boxes of 64 K-elements (128 bytes,
// swizzled) x box_rows rows; rows past the end read as zero.
bool make_map_2d(CUtensorMap* m, const void* base, int rows, int K, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kGK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int EPI>
cudaError_t launch_bn(const GemmArgs& a, const void* A, const void* Bw, cudaStream_t s) {
  using C = GemmCfg<BN>;
  cudaError_t e = set_smem_limit_once<gemm_tc_kernel<BN, EPI>>(C::SMEM_B);
  if (e != cudaSuccess) return e;
  CUtensorMap ma, mb;
  if (!make_map_2d(&ma, A, a.M, a.K, kGM)) return cudaErrorInvalidValue;
  if (!make_map_2d(&mb, Bw, a.N, a.K, C::MMA_N)) return cudaErrorInvalidValue;
  const int ntn = a.N / BN;
  const int ntm = (a.M + kGM - 1) / kGM;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ntn), static_cast<unsigned>(ntm));
  cfg.blockDim = dim3(kGThreads);
  cfg.dynamicSmemBytes = C::SMEM_B;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int nattr = 1;
  if (EPI == 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(ntn);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    nattr = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, EPI>, ma, mb, a);
}

}  // namespace

cudaError_t launch_gemm_tc(const GemmArgs& a, const void* A, const void* Bw, cudaStream_t s) {
  if (a.M < 1 || a.K < kGK || a.K % kGK != 0) return cudaErrorInvalidValue;
  if (a.epi == 0) {
    switch (a.hd) {
      case 64: return launch_bn<64, 0>(a, A, Bw, s);
      case 128: return launch_bn<128, 0>(a, A, Bw, s);
      case 256: return launch_bn<256, 0>(a, A, Bw, s);
      case 512: return launch_bn<512, 0>(a, A, Bw, s);
      default: return cudaErrorInvalidValue;
    }
  }
  if (a.N % 256 != 0 || a.N / 256 > 8) return cudaErrorInvalidValue;
  return launch_bn<256, 1>(a, A, Bw, s);
}

}  // namespace g4

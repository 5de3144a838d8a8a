// Step a5 in bf16: causal GQA flash attention on the tcgen05 tensor cores.
//
// Semantics as in g4_attn_simt.cu (cortiq-engine g4e.rs `attend_all_heads`
// with scale 1.0 and the sliding window, ferrox-models gemma4_engine.rs
// `causal_gqa_attention[_windowed]`): o_i = sum_j softmax_j(scale q_i.k_j) v_j
// over keys j <= i (and i - j < window on sliding layers), query head h
// reading kv head h / (H / Hkv).
//
// The BIDIR instantiation is the encoder form (taconite-embeddinggemma2
// model.rs `text_attention`): the T tokens of a sequence are both queries
// and keys (cache rows 0..T-1), with no causal mask, and key j is visible
// from query i iff |i - j| <= window on a sliding layer.  Only the tile
// range of a work item and the visible interval of a row differ.  On a
// sliding-window ring cache (max_len rows, a multiple of the 128-key tile)
// key position p is row p mod max_len; the masks stay in positions.
//
// A work item is a 128-query-row tile of one (sequence, head) and, for
// head_dim 512, one 256-wide half of the output columns (two items per tile
// then recompute the same scores; TMEM holds 512 f32 columns per SM and a
// 128 x 512 accumulator alone would fill it).  Items run in (sequence, kv
// head) groups, heaviest query tiles first, so the CTAs in flight share their
// K / V in L2.  The kernel is persistent: one CTA per SM takes items one
// after another from a global counter (the producer draws them and passes
// them on through a 4-entry queue in shared memory), with its barriers, ring and TMEM
// running on from item to item, so the next item's Q and first K parts load
// while the current one finishes.  Warp roles (320 threads):
//   warp 0      TMA producer (converged; one elected lane issues): the Q
//               tile, then K parts (128 keys x 64..256 dims) and V parts
//               (64..128 keys x DV dims) as 5-D boxes, one request per
//               32-64 KB (a request costs the SM about the same whatever its
//               size), through a ring of slots, 128-byte swizzled.
//   warp 1      allocates TMEM and runs the MMA issue loop converged; one
//               elected lane issues every tcgen05.mma from precomputed
//               descriptors:
//                 S[j%2] = Q K_j^T      (M=128, N=128, K=head_dim; A, B from
//                                        shared memory, K-major)
//                 O     += P_j V_j      (M=128, N=DV,  K=128; A = P_j from
//                                        TMEM, B = V_j MN-major)
//               in the order QK_0, QK_1, PV_0, QK_2, PV_1, ... so the score
//               MMA of the next tile overlaps the softmax of this one.
//   warps 2-9   softmax: two warps per TMEM lane quarter (a warp may only
//               touch its quarter's 32 lanes), each thread half a query row
//               (64 of the 128 score columns; TMEM lane = row): load the
//               whole S row with tcgen05.ld (both threads of a row find the
//               same maximum), mask (one visible key interval per row:
//               causal end, window start, keys past the cache), online
//               softmax in the log2 domain with the running maximum raised
//               only when it grows by more than 2^64 (the stale maximum is
//               exact for O / l), rescale its half of the O row in TMEM when
//               it is raised, and write its P half as bf16 over the S buffer
//               (packed: 32 columns), once the other warp of the quarter has
//               read the row too (P lands on S columns both warps read).
//               The row sum l adds the bf16-rounded P
//               values, the weights the PV MMA really applies, so a row
//               dominated by one key returns that key's value without the
//               rounding error of P; the two halves' sums meet in shared
//               memory once, at the end.  Epilogue: O / l as bf16 into the
//               ring slots of the item's last V parts (swizzled like the
//               output tensor map), TMA stores, then those slots are freed.
// TMEM columns: S0/P0 [0,128), S1/P1 [128,256), O [256, 256 + DV).
// The MMAs of one thread execute in issue order, so QK_{j+2} (issued after
// PV_j) overwrites P_j only after PV_j has read it; no barrier is needed
// between them.  Barriers come in pairs indexed by tile parity (j % 2), which
// keeps each phase unambiguous for waiters that skip phases.
// Key tiles wholly outside every row's band are never loaded.
#include <math.h>

#include <mutex>

#include "g4_device.cuh"
#include "g4_internal.h"

namespace g4 {
namespace {

constexpr int kBM = 128;       // query rows per CTA
constexpr int kBN = 128;       // keys per tile
constexpr int kChunkB = 16384;  // 128 rows x 64 bf16, one 128-byte-swizzled block
constexpr int kThreads = 320;  // 10 warps
constexpr int kMaxSlots = 12;
constexpr int kSmemMax = 232448;  // opt-in shared memory per block
// The exponent base of a row is raised only when a tile's maximum exceeds it
// by more than 2^64: P <= 2^64 in bf16 and O <= 2^64 * keys * |v| in f32 stay
// far from overflow, and rescaling O (a TMEM round trip) becomes rare.
constexpr float kRescaleLog2 = 64.0f;

template <int HD>
struct TcCfg {
  static constexpr int DV = HD < 256 ? HD : 256;  // output columns per CTA
  static constexpr int NDH = HD / DV;             // CTAs per (tile, head)
  static constexpr int QCH = HD / 64;             // 64-dim chunks of Q and of a K tile
  // A TMA request costs the SM about 576 cycles whatever its size up to
  // 32 KB (64 KB: ~900), so tiles move as few large multi-dimensional boxes:
  // a K part is 128 keys x CPP 64-dim chunks, a V part VKP keys x DV dims.
  static constexpr int KPARTS = HD == 512 ? 4 : 1;
  static constexpr int CPP = QCH / KPARTS;          // 64-dim chunks per K part
  static constexpr int KPB = CPP * kChunkB;         // K part bytes
  static constexpr int VKP = HD == 512 ? 64 : 128;  // keys per V part
  static constexpr int VPARTS = kBN / VKP;
  static constexpr int VPB = VKP * DV * 2;          // V part bytes
  static constexpr int SLOTB = KPB > VPB ? KPB : VPB;
  // The output tile (DV / 64 chunks) is staged in the slots of the last V
  // parts of the item: CPS chunks per slot, OSLOTS slots.
  static constexpr int CPS = SLOTB / kChunkB;
  static constexpr int OSLOTS = (DV / 64) / CPS;
  static constexpr int Q_OFF = 0;
  static constexpr int RING_OFF = Q_OFF + QCH * kChunkB;
  static constexpr int BAR_B = 3072;
  static constexpr int NSLOT_FIT = (kSmemMax - BAR_B - RING_OFF) / SLOTB;
  static constexpr int NSLOT = NSLOT_FIT < kMaxSlots ? NSLOT_FIT : kMaxSlots;
  static constexpr int BAR_OFF = RING_OFF + NSLOT * SLOTB;
  static constexpr int SMEM_B = BAR_OFF + BAR_B;
  static_assert(NSLOT >= 2, "ring depth");
  static_assert(SMEM_B <= kSmemMax, "shared memory budget");
  static_assert(VKP % 16 == 0 && kBN % VKP == 0 && QCH % KPARTS == 0, "tiling");
  static_assert(SLOTB % kChunkB == 0 && (DV / 64) % CPS == 0 && OSLOTS >= 1 && OSLOTS <= VPARTS &&
                    OSLOTS < NSLOT && VPB == SLOTB,
                "output staging in the ring");
};

struct TcBars {
  uint64_t q_full;     // the current item's Q tile has landed (one phase per item)
  uint64_t q_free;     // every QK MMA of the current item is complete (Q may be replaced)
  uint64_t s_full[2];  // QK_j complete (tile parity)
  uint64_t p_full[2];  // P_j written to TMEM by all 128 softmax threads
  uint64_t o_done[2];  // PV_j complete
  uint64_t drain;
  uint64_t sum_full[4];  // [lane quarter]: both row-sum shares written
  uint64_t s_read[4];    // [lane quarter]: both warps have S_j in registers (P_j may overwrite it)
  uint64_t full[kMaxSlots];
  uint64_t empty[kMaxSlots];
  uint64_t it_full[4];   // work-item queue entry written (by the producer)
  uint64_t it_empty[4];  // entry read by the MMA issuer and the softmax warps
  int items[4];          // work-item queue: item index, or -1 when none is left
  uint32_t tmem_base;
  int abort;
  float red[2][kBM];  // [column half][row]: row-sum shares
};
static_assert(sizeof(TcBars) <= 3072, "barrier block");

// All 256 softmax threads meet (named barrier 1) and learn whether any of
// them passed a nonzero flag.
__device__ __forceinline__ bool softmax_sync_any(int flag) {
  uint32_t any;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, 256, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(any)
      : "r"(flag)
      : "memory");
  return any != 0;
}

// Work item -> (output half, q head of the group, q tile, kv head, sequence)
// and the key tiles it needs.  Items run in (sequence, kv head) groups so the
// CTAs working at the same time share one K / V in L2; within a group the
// heaviest (last) query tiles come first.
struct TcItem {
  int dh, h, kvh, b;
  int q0, valid_rows, qpos_first, Lk, kt_begin, ntiles;
};

template <int NDH, bool BIDIR>
__device__ __forceinline__ TcItem tc_item(const PrefillTcArgs& a, int it, int nqt) {
  TcItem w;
  const int grp = a.H / a.Hkv;
  int idx = it;
  w.dh = idx % NDH;
  idx /= NDH;
  const int hq = idx % grp;
  idx /= grp;
  const int qt = nqt - 1 - idx % nqt;
  idx /= nqt;
  w.kvh = idx % a.Hkv;
  w.b = idx / a.Hkv;
  w.h = w.kvh * grp + hq;
  const int q_start = BIDIR ? 0 : a.q_start[w.b];
  w.q0 = qt * kBM;
  w.valid_rows = min(kBM, a.T - w.q0);
  w.qpos_first = q_start + w.q0;
  const int qpos_last = w.qpos_first + w.valid_rows - 1;
  int kbeg, kend;
  if constexpr (BIDIR) {
    // Encoder: the sequence's own T keys, no causal mask; query i sees
    // [i - window, i + window] on a sliding layer (window <= T here).
    w.Lk = a.T;
    kbeg = a.sliding ? max(0, w.qpos_first - a.window) : 0;
    kend = a.sliding ? min(qpos_last + a.window + 1, w.Lk) : w.Lk;
  } else {
    // keys held: positions [0, Lk) (a ring holds the last max_len of them)
    w.Lk = a.ring ? q_start + a.T : min(q_start + a.T, a.max_len);
    kend = min(qpos_last + 1, w.Lk);
    kbeg = a.sliding ? max(0, w.qpos_first - a.window + 1) : 0;
  }
  w.kt_begin = kbeg / kBN;
  w.ntiles = max(0, (kend + kBN - 1) / kBN - w.kt_begin);
  return w;
}

template <int HD, bool BIDIR>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                      const __grid_constant__ PrefillTcArgs a) {
  using C = TcCfg<HD>;
  // 128-byte-swizzled tiles need 1024-byte alignment; the declaration asks
  // for it, and a block that does not get it reports and does nothing.
  extern __shared__ __align__(1024) uint8_t smem[];
  // The last CTA to finish clears the launch's work-item counters for the
  // next launch that uses them (every CTA has drawn its last item by then).
  auto release_counters = [&]() {
    if (threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(a.item_ctr + 1, 1u) == gridDim.x - 1) {
        __threadfence();
        atomicExch(a.item_ctr, 0u);
        atomicExch(a.item_ctr + 1, 0u);
      }
    }
  };
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicExch(a.err, kErrSmemAlign);
    release_counters();
    return;
  }
  TcBars* bars = reinterpret_cast<TcBars*>(smem + C::BAR_OFF);
  const uint32_t sQ = smem_u32(smem + C::Q_OFF);
  const uint32_t sRing = smem_u32(smem + C::RING_OFF);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();

  const int nqt = (a.T + kBM - 1) / kBM;
  const int nitems = nqt * a.H * a.B * C::NDH;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->q_full), 1);
    mbar_init(smem_u32(&bars->q_free), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->s_full[i]), 1);
      mbar_init(smem_u32(&bars->p_full[i]), 256);
      mbar_init(smem_u32(&bars->o_done[i]), 1);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    for (int qq = 0; qq < 4; ++qq) mbar_init(smem_u32(&bars->sum_full[qq]), 64);
    for (int qq = 0; qq < 4; ++qq) mbar_init(smem_u32(&bars->s_read[qq]), 64);
    for (int i = 0; i < C::NSLOT; ++i) mbar_init(smem_u32(&bars->full[i]), 1);
    for (int i = 0; i < C::NSLOT; ++i) mbar_init(smem_u32(&bars->empty[i]), 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(smem_u32(&bars->it_full[i]), 1);
      mbar_init(smem_u32(&bars->it_empty[i]), 2);
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
    // The warp runs the loop converged; one elected lane draws the work items
    // and issues every copy.  The ring runs on across work items: the next
    // item's Q is loaded once the last QK MMA of the current one has read the
    // old Q, and its first K parts go into whatever slots are free while the
    // current item finishes.
    {
      if (elect_one()) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
      }
      __syncwarp();
      const uint32_t qb = smem_u32(&bars->q_full);
      bool ok = true;
      int seq = 0;
      int slot = 0;        // ring slot of the next part
      uint32_t phase = 0;  // parity of that slot's current use
      int nq = 0;          // items whose Q has been requested
      auto advance = [&]() {
        ++seq;
        if (++slot == C::NSLOT) {
          slot = 0;
          phase ^= 1u;
        }
      };
      for (int n = 0; ok; ++n) {
        // next work item into queue entry n % 4 (once both readers are done with its last use)
        const int e = n & 3;
        if (n >= 4 && !warp_wait(smem_u32(&bars->it_empty[e]), ((n >> 2) - 1) & 1, a.err, abort)) break;
        unsigned got = 0;
        if (lane == 0) got = atomicAdd(a.item_ctr, 1u);
        got = __shfl_sync(0xffffffffu, got, 0);
        const int it = got < static_cast<unsigned>(nitems) ? static_cast<int>(got) : -1;
        if (lane == 0) {
          *reinterpret_cast<volatile int*>(&bars->items[e]) = it;
          mbar_arrive(smem_u32(&bars->it_full[e]));
        }
        __syncwarp();
        if (it < 0) break;
        const TcItem w = tc_item<C::NDH, BIDIR>(a, it, nqt);
        if (w.ntiles == 0) continue;
        if (nq > 0 && !warp_wait(smem_u32(&bars->q_free), (nq - 1) & 1, a.err, abort)) break;
        // Q tile: 128 rows x QCH chunks in one request (two for head_dim 512)
        constexpr int QREQ = C::QCH > 4 ? 2 : 1;
        if (elect_one()) {
          mbar_arrive_expect_tx(qb, C::QCH * kChunkB);
#pragma unroll
          for (int r = 0; r < QREQ; ++r)
            tma_load_5d(sQ + r * (C::QCH / QREQ) * kChunkB, &tm_q, 0, w.q0, r * (C::QCH / QREQ), w.h, w.b, qb);
        }
        __syncwarp();
        ++nq;
        // Cache row of a key tile's first position: on a ring of max_len
        // rows (a multiple of the 128-key tile, so no tile wraps) the
        // position modulo max_len.
        auto tile_row = [&](int kt) { return a.ring ? (kt * kBN) % a.max_len : kt * kBN; };
        auto load_k = [&](int kt) {
          const int kr = tile_row(kt);
          for (int p2 = 0; p2 < C::KPARTS && ok; ++p2) {
            if (!warp_wait(smem_u32(&bars->empty[slot]), phase ^ 1u, a.err, abort)) { ok = false; break; }
            const uint32_t fb = smem_u32(&bars->full[slot]);
            if (elect_one()) {
              mbar_arrive_expect_tx(fb, C::KPB);
              tma_load_5d(sRing + slot * C::SLOTB, &tm_k, 0, kr, p2 * C::CPP, w.kvh, w.b, fb);
            }
            __syncwarp();
            advance();
          }
        };
        auto load_v = [&](int kt) {
          const int kr = tile_row(kt);
          for (int p2 = 0; p2 < C::VPARTS && ok; ++p2) {
            if (!warp_wait(smem_u32(&bars->empty[slot]), phase ^ 1u, a.err, abort)) { ok = false; break; }
            const uint32_t fb = smem_u32(&bars->full[slot]);
            if (elect_one()) {
              mbar_arrive_expect_tx(fb, C::VPB);
              tma_load_5d(sRing + slot * C::SLOTB, &tm_v, 0, kr + p2 * C::VKP, w.dh * (C::DV / 64), w.kvh, w.b,
                          fb);
            }
            __syncwarp();
            advance();
          }
        };
        load_k(w.kt_begin);
        for (int j = 0; j < w.ntiles && ok; ++j) {
          if (j + 1 < w.ntiles) load_k(w.kt_begin + j + 1);
          load_v(w.kt_begin + j);
        }
      }
      // Copies still in flight must land before the CTA may exit.
      if (nq > 0) warp_wait(qb, (nq - 1) & 1, nullptr);
      for (int s2 = max(0, seq - C::NSLOT); s2 < seq; ++s2)
        warp_wait(smem_u32(&bars->full[s2 % C::NSLOT]), (s2 / C::NSLOT) & 1, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop converged (waits included) and one
    // elected lane issues each tcgen05.mma and commit: the loop's descriptor
    // and ring arithmetic stays warp-uniform, and issue keeps ahead of the
    // tensor pipe (run by one lane inside a lane test, the loop issued each
    // MMA slower than the pipe executes it).  Tile parities run on across
    // items (J counts every tile of the CTA).
    {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, C::DV, 0, 1);
      bool ok = true;
      // Descriptors are built once; a slot, a 64-dim chunk or a 16-element
      // K step only moves the start address (16-byte units in the low bits,
      // which stay below 2^14 for any shared-memory address).  Building them
      // per instruction costs the issue loop more cycles than the MMA.
      const uint64_t dq0 = smem_desc_sw128(sQ, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(sRing, 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(sRing, C::VKP * 128, 1024);
      // Ring state, advanced incrementally: the issue loop's own instruction
      // latency sits between MMAs of 64 cycles, so there is no division,
      // modulo or multiply on this path.
      int slot = 0;        // ring slot of the next part
      uint32_t phase = 0;  // parity of that slot's current use
      uint32_t soff = 0;   // slot * SLOTB in descriptor units (16 bytes)
      const uint32_t full0 = smem_u32(&bars->full[0]);
      const uint32_t empty0 = smem_u32(&bars->empty[0]);
      auto advance = [&]() {
        soff += C::SLOTB >> 4;
        if (++slot == C::NSLOT) {
          slot = 0;
          phase ^= 1u;
          soff = 0;
        }
      };
      auto release = [&]() {
        tc_commit_elect(empty0 + slot * 8);
        advance();
      };
      int J = 0;   // tiles of earlier items
      int nq = 0;  // items started
      for (int n = 0; ok; ++n) {
        const int e = n & 3;
        if (!warp_wait(smem_u32(&bars->it_full[e]), (n >> 2) & 1, a.err, abort)) break;
        const int it = *reinterpret_cast<volatile int*>(&bars->items[e]);
        if (lane == 0) mbar_arrive(smem_u32(&bars->it_empty[e]));
        __syncwarp();
        if (it < 0) break;
        const TcItem w = tc_item<C::NDH, BIDIR>(a, it, nqt);
        if (w.ntiles == 0) continue;
        if (!warp_wait(smem_u32(&bars->q_full), nq & 1, a.err, abort)) break;
        ++nq;
        tc_fence_after();
        auto mma_qk = [&](int j) {
          const int sb = (J + j) & 1;
          const uint32_t dS = tmem + sb * kBN;
          uint64_t ad = dq0;
#pragma unroll 1
          for (int p2 = 0; p2 < C::KPARTS; ++p2) {
            if (!warp_wait(full0 + slot * 8, phase, a.err, abort)) { ok = false; return; }
            tc_fence_after();
            uint64_t bd = dk0 + soff;
#pragma unroll
            for (int c = 0; c < C::CPP; ++c) {
              tc_mma_ss_elect(dS, ad, bd, idesc_qk, (p2 > 0 || c > 0) ? 1u : 0u);
              tc_mma_ss_elect(dS, ad + 2, bd + 2, idesc_qk, 1u);
              tc_mma_ss_elect(dS, ad + 4, bd + 4, idesc_qk, 1u);
              tc_mma_ss_elect(dS, ad + 6, bd + 6, idesc_qk, 1u);
              ad += kChunkB >> 4;
              bd += kChunkB >> 4;
            }
            release();
          }
          tc_commit_elect(smem_u32(&bars->s_full[sb]));
          // after the item's last QK, the Q area may take the next item's Q
          if (j == w.ntiles - 1) tc_commit_elect(smem_u32(&bars->q_free));
        };
        auto mma_pv = [&](int j) {
          const int sb = (J + j) & 1;
          if (!warp_wait(smem_u32(&bars->p_full[sb]), ((J + j) >> 1) & 1, a.err, abort)) { ok = false; return; }
          tc_fence_after();
          const int kt = w.kt_begin + j;
          uint32_t ta = tmem + sb * kBN;  // P_j: 128 keys as 64 packed columns
          const bool last = j == w.ntiles - 1;
#pragma unroll 1
          for (int p2 = 0; p2 < C::VPARTS; ++p2) {
            if (!warp_wait(full0 + slot * 8, phase, a.err, abort)) { ok = false; return; }
            // Rows of keys past the cache's filled length may hold anything
            // (even NaN, and 0 * NaN = NaN); zero them before they meet P
            // (only in the part holding the end of the keys).
            const int key0 = kt * kBN + p2 * C::VKP;
            if (key0 + C::VKP > w.Lk) {
              const int nvalid = max(0, w.Lk - key0);
              uint8_t* slot_ptr = smem + C::RING_OFF + slot * C::SLOTB;
              const int nbad = C::VKP - nvalid;
              for (int i = lane; i < (C::DV / 64) * nbad * 8; i += 32) {
                const int dc = i / (nbad * 8);
                const int rr = (i / 8) % nbad + nvalid;
                const int pc = i % 8;
                *reinterpret_cast<uint4*>(slot_ptr + dc * C::VKP * 128 + rr * 128 + pc * 16) = make_uint4(0, 0, 0, 0);
              }
              fence_proxy_async_smem();
              __syncwarp();
            }
            tc_fence_after();
            const uint64_t bd = dv0 + soff;
#pragma unroll
            for (int kk = 0; kk < C::VKP / 16; ++kk)
              tc_mma_ts_elect(tmem_O, ta + kk * 8, bd + static_cast<uint64_t>(kk * 128), idesc_pv,
                        (j > 0 || p2 > 0 || kk > 0) ? 1u : 0u);
            ta += C::VKP / 2;
            // The item's last OSLOTS V parts stay held: the epilogue stages
            // O there and frees them after its store has read them.
            if (last && p2 >= C::VPARTS - C::OSLOTS)
              advance();
            else
              release();
          }
          tc_commit_elect(smem_u32(&bars->o_done[sb]));
        };
        mma_qk(0);
        for (int j = 0; j < w.ntiles && ok; ++j) {
          if (j + 1 < w.ntiles) mma_qk(j + 1);
          if (ok) mma_pv(j);
        }
        J += w.ntiles;
      }
      // Every MMA issued so far completes before TMEM is released.
      tc_commit_elect(smem_u32(&bars->drain));
      warp_wait(smem_u32(&bars->drain), 0, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // which 64 of the 128 score columns
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c2 = a.scale_log2;  // > 0 (checked on the host)
    constexpr int kHB = kBN / 2;    // score columns per thread
    constexpr int kDVH = C::DV / 2; // O columns per thread
    constexpr int kParts = C::KPARTS + C::VPARTS;  // ring parts per key tile
    int J = 0;      // tiles of earlier items
    int nq = 0;     // items done
    int parts = 0;  // ring parts of earlier items
    for (int n = 0;; ++n) {
      const int e = n & 3;
      const int it = warp_wait(smem_u32(&bars->it_full[e]), (n >> 2) & 1, a.err, abort)
                         ? *reinterpret_cast<volatile int*>(&bars->items[e])
                         : -1;
      if (it < 0) {
        // no item left (or a wait gave up): every softmax thread leaves here
        // or at the end of an item, together
        softmax_sync_any(1);
        break;
      }
      const TcItem w = tc_item<C::NDH, BIDIR>(a, it, nqt);
      const int ntiles = w.ntiles;
      if (ntiles == 0) {
        // No visible key (only reachable with out-of-contract positions).
        if (r < w.valid_rows) {
          __nv_bfloat16* dst =
              static_cast<__nv_bfloat16*>(a.out) +
              (((static_cast<size_t>(w.b) * a.T + w.q0 + r) * a.H + w.h) * HD + w.dh * C::DV + half * kDVH);
          for (int i = 0; i < kDVH / 8; ++i) reinterpret_cast<uint4*>(dst)[i] = make_uint4(0, 0, 0, 0);
        }
        const bool stop0 = softmax_sync_any(*abort);
        if (warp == 2 && lane == 0 && !stop0) mbar_arrive(smem_u32(&bars->it_empty[e]));
        __syncwarp();
        if (stop0) break;
        continue;
      }
      const int qpos = w.qpos_first + r;
      const bool row_valid = r < w.valid_rows;
      float m = -INFINITY;  // exponent base in log2 units: a stale running maximum
      float l = 0.0f;       // this half's share of the row sum
      bool ok = true;
      for (int j = 0; j < ntiles; ++j) {
        const int sb = (J + j) & 1;
        if (!warp_wait(smem_u32(&bars->s_full[sb]), ((J + j) >> 1) & 1, a.err, abort)) { ok = false; break; }
        tc_fence_after();
        float s[kHB];
        float mt;
        {
          // the whole row: both threads of a row take the same maximum
          uint32_t r0[32], r1[32], o0[32], o1[32];
          const uint32_t tS = tmem + lane_off + sb * kBN;
          tmem_ld32(tS + half * kHB, r0);
          tmem_ld32(tS + half * kHB + 32, r1);
          tmem_ld32(tS + (1 - half) * kHB, o0);
          tmem_ld32(tS + (1 - half) * kHB + 32, o1);
          tc_wait_ld();
          // P_j goes over S_j, partly over the other warp's half of the row,
          // which that warp reads too: tell it this warp's reads are done.
          mbar_arrive(smem_u32(&bars->s_read[quarter]));
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            s[i] = __uint_as_float(r0[i]);
            s[32 + i] = __uint_as_float(r1[i]);
          }
          const int kr = (w.kt_begin + j) * kBN;
          const bool row_vis =
              BIDIR ? row_valid && (kr + kBN <= w.Lk) &&
                          (!a.sliding || (qpos - kr <= a.window && kr + kBN - 1 - qpos <= a.window))
                    : row_valid && (kr + kBN - 1 <= qpos) && (kr + kBN <= w.Lk) &&
                          (!a.sliding || qpos - kr < a.window);
          const int k0 = kr + half * kHB;
          const int k1 = kr + (1 - half) * kHB;
          float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          if (row_vis) {
#pragma unroll
            for (int n = 0; n < 32; ++n) {
              mx[n & 3] = fmaxf(mx[n & 3], fmaxf(s[n], s[32 + n]));
              mx[(n + 2) & 3] = fmaxf(mx[(n + 2) & 3], fmaxf(__uint_as_float(o0[n]), __uint_as_float(o1[n])));
            }
          } else {
            // The row's visible keys are one interval [vlo, vhi): causal end,
            // the cache's filled length and (sliding) the window start; in
            // the encoder form the window's two ends and the sequence end.
            const int vlo = a.sliding ? max(0, qpos - a.window + (BIDIR ? 0 : 1)) : 0;
            const int vhi = !row_valid ? 0
                            : BIDIR    ? (a.sliding ? min(qpos + a.window + 1, w.Lk) : w.Lk)
                                       : min(qpos + 1, w.Lk);
            const unsigned span = static_cast<unsigned>(max(0, vhi - vlo));
            const int lo0 = vlo - k0, lo1 = vlo - k1;
#pragma unroll
            for (int n = 0; n < kHB; ++n) {
              if (static_cast<unsigned>(n - lo0) >= span) s[n] = -INFINITY;
              mx[n & 3] = fmaxf(mx[n & 3], s[n]);
            }
#pragma unroll
            for (int n = 0; n < 32; ++n) {
              const float v0 = static_cast<unsigned>(n - lo1) < span ? __uint_as_float(o0[n]) : -INFINITY;
              const float v1 = static_cast<unsigned>(n + 32 - lo1) < span ? __uint_as_float(o1[n]) : -INFINITY;
              mx[n & 3] = fmaxf(mx[n & 3], fmaxf(v0, v1));
            }
          }
          mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * c2;
        }
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
          if (!warp_wait(smem_u32(&bars->o_done[(J + j - 1) & 1]), ((J + j - 1) >> 1) & 1, a.err, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float f = rescale ? alpha : 1.0f;
#pragma unroll 1
          for (int cc = 0; cc < kDVH / 32; ++cc) {
            uint32_t rr[32];
            const uint32_t tO = tmem_O + lane_off + half * kDVH + cc * 32;
            tmem_ld32(tO, rr);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * f);
            tmem_st32(tO, rr);
          }
          tc_wait_st();
        }
        const float nb = (m_use == -INFINITY) ? 0.0f : -m_use;
        uint32_t p[32];
        float sa[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t pw = pack_bf16x2(ex2_approx(fmaf(s[2 * i], c2, nb)), ex2_approx(fmaf(s[2 * i + 1], c2, nb)));
          p[i] = pw;
          sa[(2 * i) & 3] += bf16_lo(pw);
          sa[(2 * i + 1) & 3] += bf16_hi(pw);
        }
        if (!warp_wait(smem_u32(&bars->s_read[quarter]), (J + j) & 1, a.err, abort)) {
          ok = false;
          break;
        }
        tmem_st32(tmem + lane_off + sb * kBN + half * (kHB / 2), p);
        l = l * alpha + ((sa[0] + sa[1]) + (sa[2] + sa[3]));
        m = m_use;
        tc_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars->p_full[sb]));
      }
      if (ok) {
        // the full row sum: both halves' shares
        bars->red[half][r] = l;
        mbar_arrive(smem_u32(&bars->sum_full[quarter]));
        ok = warp_wait(smem_u32(&bars->sum_full[quarter]), nq & 1, a.err, abort);
        l = bars->red[0][r] + bars->red[1][r];
      }
      // Epilogue: O / l as bf16, in the chunk-major 128-byte-swizzled layout of
      // the output tensor map, into the ring slots of the item's last V parts
      // (free once the last PV has completed), then TMA stores of the tile.
      // Rows past T fall outside the map and are not written.
      const int last_part = parts + ntiles * kParts - 1;  // ring sequence number
      auto oslot = [&](int k) { return (last_part - (C::OSLOTS - 1) + k) % C::NSLOT; };
      if (ok) {
        const int jl = J + ntiles - 1;
        if (warp_wait(smem_u32(&bars->o_done[jl & 1]), (jl >> 1) & 1, a.err, abort)) {
          tc_fence_after();
          const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
          constexpr int NCC = kDVH / 32;
          uint32_t rr[NCC][32];
#pragma unroll
          for (int cc = 0; cc < NCC; ++cc) tmem_ld32(tmem_O + lane_off + half * kDVH + cc * 32, rr[cc]);
          tc_wait_ld();
#pragma unroll
          for (int cc = 0; cc < NCC; ++cc) {
            // 32 columns = half a 64-column chunk: pieces (16 bytes) p0 .. p0 + 3
            const int col = half * kDVH + cc * 32;
            const int ch = col / 64;
            const uint32_t row_addr = sRing + oslot(ch / C::CPS) * C::SLOTB + (ch % C::CPS) * kChunkB + r * 128;
            const int p0 = (col % 64) / 8;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t x = pack_bf16x2(__uint_as_float(rr[cc][8 * i + 0]) * inv_l, __uint_as_float(rr[cc][8 * i + 1]) * inv_l);
              const uint32_t y = pack_bf16x2(__uint_as_float(rr[cc][8 * i + 2]) * inv_l, __uint_as_float(rr[cc][8 * i + 3]) * inv_l);
              const uint32_t z = pack_bf16x2(__uint_as_float(rr[cc][8 * i + 4]) * inv_l, __uint_as_float(rr[cc][8 * i + 5]) * inv_l);
              const uint32_t q = pack_bf16x2(__uint_as_float(rr[cc][8 * i + 6]) * inv_l, __uint_as_float(rr[cc][8 * i + 7]) * inv_l);
              const uint32_t addr = row_addr + (((p0 + i) ^ (r & 7)) * 16);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z), "r"(q)
                           : "memory");
            }
          }
          fence_proxy_async_smem();
        } else {
          ok = false;
        }
      }
      // All 256 softmax threads meet here on every path, and all leave the
      // item loop together if any wait anywhere gave up.
      const bool stop = softmax_sync_any(!ok || *abort);
      if (warp == 2 && lane == 0 && !stop) {
#pragma unroll
        for (int k = 0; k < C::OSLOTS; ++k)
          tma_store_5d(&tm_o, sRing + oslot(k) * C::SLOTB, 0, w.q0, w.dh * (C::DV / 64) + k * C::CPS, w.h, w.b);
        bulk_commit_group();
        bulk_wait_read_all();  // the slots must not be refilled before the stores have read them
#pragma unroll
        for (int k = 0; k < C::OSLOTS; ++k) mbar_arrive(smem_u32(&bars->empty[oslot(k)]));
      }
      if (warp == 2 && lane == 0 && !stop) mbar_arrive(smem_u32(&bars->it_empty[e]));
      __syncwarp();
      if (stop) break;
      J += ntiles;
      parts += ntiles * kParts;
      ++nq;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  release_counters();
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

// bf16 5-D tensor map, dims innermost first, 128-byte swizzle, zero fill out
// of bounds.  Dim 0 is 64 consecutive elements (one 128-byte row), dim 1 the
// rows (tokens or keys), dim 2 the 64-element chunks of a head, so a box of
// (64, rows, chunks) lands in shared memory as chunk-major 128-byte rows:
// the layout the MMA descriptors read.
bool make_map(CUtensorMap* m, const void* base, const cuuint64_t dims[5], const cuuint64_t strides_bytes[4],
              const cuuint32_t box[5]) {
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) return false;
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides_bytes, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int HD, bool BIDIR>
cudaError_t launch_hd(const PrefillTcArgs& a, cudaStream_t s) {
  using C = TcCfg<HD>;
  const cudaError_t e = set_smem_limit_once<prefill_tc_kernel<HD, BIDIR>>(C::SMEM_B);
  if (e != cudaSuccess) return e;
  CUtensorMap mq, mk, mv, mo;
  const cuuint64_t row_b = static_cast<cuuint64_t>(HD) * 2;
  constexpr cuuint32_t kQBoxChunks = C::QCH > 4 ? C::QCH / 2 : C::QCH;
  {
    // q [B][T][H][hd]: (element, token, chunk, head, sequence)
    const cuuint64_t dims[5] = {64, static_cast<cuuint64_t>(a.T), static_cast<cuuint64_t>(C::QCH),
                                static_cast<cuuint64_t>(a.H), static_cast<cuuint64_t>(a.B)};
    const cuuint64_t str[4] = {row_b * a.H, 128, row_b, row_b * a.H * a.T};
    const cuuint32_t box[5] = {64, kBM, kQBoxChunks, 1, 1};
    if (!make_map(&mq, a.q, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    // cache [B][Hkv][max_len][hd]: (element, key, chunk, kv head, sequence)
    const cuuint64_t dims[5] = {64, static_cast<cuuint64_t>(a.max_len), static_cast<cuuint64_t>(C::QCH),
                                static_cast<cuuint64_t>(a.Hkv), static_cast<cuuint64_t>(a.B)};
    const cuuint64_t str[4] = {row_b, 128, row_b * a.max_len, row_b * a.max_len * a.Hkv};
    const cuuint32_t boxk[5] = {64, kBN, C::CPP, 1, 1};
    const cuuint32_t boxv[5] = {64, C::VKP, C::DV / 64, 1, 1};
    if (!make_map(&mk, a.ck, dims, str, boxk)) return cudaErrorInvalidValue;
    if (!make_map(&mv, a.cv, dims, str, boxv)) return cudaErrorInvalidValue;
  }
  {
    // out [B][T][H][hd], written DV columns (DV / 64 chunks) at a time
    const cuuint64_t dims[5] = {64, static_cast<cuuint64_t>(a.T), static_cast<cuuint64_t>(C::QCH),
                                static_cast<cuuint64_t>(a.H), static_cast<cuuint64_t>(a.B)};
    const cuuint64_t str[4] = {row_b * a.H, 128, row_b, row_b * a.H * a.T};
    const cuuint32_t box[5] = {64, kBM, C::CPS, 1, 1};
    if (!make_map(&mo, a.out, dims, str, box)) return cudaErrorInvalidValue;
  }
  // One persistent CTA per SM (shared memory and TMEM allow no more), each
  // drawing work items from the launch's counter pair until none is left.
  const int nqt = (a.T + kBM - 1) / kBM;
  const long long nitems = static_cast<long long>(nqt) * a.H * a.B * C::NDH;
  if (nitems > 0x7fffffffLL) return cudaErrorInvalidValue;
  const long long nblk = nitems < sm_count() ? nitems : sm_count();
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
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<HD, BIDIR>, mq, mk, mv, mo, a);
}

}  // namespace

// Work-item counters of the persistent prefill, one pair per launch in flight
// (launches take the pairs in turn, so up to kCtrSlots launches may overlap).
constexpr int kCtrSlots = 64;
__device__ unsigned g_prefill_ctr[kCtrSlots][2];

cudaError_t launch_prefill_tc(const PrefillTcArgs& a_in, cudaStream_t s) {
  static std::mutex mu;
  static unsigned* base[128] = {};
  static unsigned next_slot = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  PrefillTcArgs a = a_in;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (base[dev] == nullptr) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_prefill_ctr);
      if (e != cudaSuccess) return e;
      base[dev] = static_cast<unsigned*>(p);
    }
    a.item_ctr = base[dev] + 2 * (next_slot++ % kCtrSlots);
  }
  if (a.bidir) {
    switch (a.hd) {
      case 64: return launch_hd<64, true>(a, s);
      case 128: return launch_hd<128, true>(a, s);
      case 256: return launch_hd<256, true>(a, s);
      case 512: return launch_hd<512, true>(a, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (a.hd) {
    case 64: return launch_hd<64, false>(a, s);
    case 128: return launch_hd<128, false>(a, s);
    case 256: return launch_hd<256, false>(a, s);
    case 512: return launch_hd<512, false>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace g4

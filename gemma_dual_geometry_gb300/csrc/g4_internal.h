// Internal launch interface between the C-ABI front end (g4_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

namespace g4 {

// Raises kernel Kern's dynamic shared-memory limit to `bytes` on the current
// device.  The attribute belongs to the device, so it is set once per device
// (and per kernel: Kern is a template argument), under a lock.
template <auto Kern>
cudaError_t set_smem_limit_once(int bytes) {
  static std::mutex mu;
  static bool done[128] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  return cudaSuccess;
}

constexpr int kMaxHalf = 256;  // head_dim / 2 for the widest supported head (512)

// Step a4: norm -> RoPE -> cache append.
struct AppendArgs {
  const void* q_in;
  const void* k_in;  // null on a shared layer
  const void* v_in;
  const float* q_w;
  const float* k_w;
  const int32_t* positions;  // [B*T]
  void* q_out;
  void* cache_k;  // [B][Hkv][max_len][hd]
  void* cache_v;
  int B, T, H, Hkv, hd, max_len;
  int ring;          // 1: position p goes to row p mod max_len (sliding-window ring)
  int rows_per_cta;  // head rows (of H + 2 Hkv) handled per CTA
  int tok_per_cta;   // tokens (same t, consecutive b) handled per CTA
  int n_rot;         // rotated pairs; inv_freq[j] == 0 for j >= n_rot
  float eps;
  float inv_freq[kMaxHalf];
};
cudaError_t launch_append(const AppendArgs& a, int dtype, cudaStream_t s);

// Steps a5 (float32) and a6: split-KV softmax attention on CUDA cores.
// mode 0 (decode): one query per sequence at position base[b] - 1, keys
//   [kstart, base[b]); mode 1 (prefill): query t at position base[b] + t;
// mode 2 (encoder, not fused): query t of a sequence of T tokens whose keys
//   are rows [0, T), keys [t - window, t + window] (sliding) or all T.
// With fused set (decode only), q / k_raw / v_raw are the new token's raw
// projections: each CTA norms and ropes its q heads, and the CTA whose split
// holds position L-1 norms/ropes the new k and v, writes them to the cache
// row L-1 and uses them as the last key (the append of step a4 in the same
// launch).
struct AttnSimtArgs {
  const void* q;    // [B][T][H][hd] (raw when fused)
  const void* ck;   // [B][Hkv][max_len][hd]
  const void* cv;
  void* out;        // [B][T][H][hd]
  const int32_t* base;
  float* ws_o;      // [B*T][H][nsplit][hd] partial outputs (nsplit > 1)
  float* ws_m;      // [B*T][H][nsplit] running max (log2 domain)
  float* ws_l;      // [B*T][H][nsplit] softmax denominators
  unsigned* tickets;  // [B*T][Hkv] arrival counters of the splits (zero between calls)
  int* err;
  int mode;
  int B, T, H, Hkv, hd, max_len;
  int ring;         // 1: key position p is row p mod max_len (sliding-window ring)
  int sliding, window;
  int len_cap;      // decode: lengths clamped to [1, len_cap]
  int chunk;        // keys per split
  int nsplit;
  float scale_log2;  // attn_scale * log2(e)
  // fused append of the new token
  int fused;
  const void* k_raw;  // [B][Hkv][hd], null on a shared layer
  const void* v_raw;
  const float* q_w;
  const float* k_w;
  void* cache_k;      // the layer's own cache (written at row L-1)
  void* cache_v;
  float eps;
  int n_rot;
  float inv_freq[kMaxHalf];
};
cudaError_t launch_attn_simt(const AttnSimtArgs& a, int dtype, cudaStream_t s);

// Step a5 (bf16): tcgen05 flash prefill.
struct PrefillTcArgs {
  const void* q;     // [B][T][H][hd] bf16
  const void* ck;    // [B][Hkv][max_len][hd] bf16
  const void* cv;
  void* out;         // [B][T][H][hd] bf16
  const int32_t* q_start;  // [B]
  int* err;
  int B, T, H, Hkv, hd, max_len;
  int ring;          // 1: key position p is row p mod max_len (max_len a multiple of 128)
  int sliding, window;
  int bidir;         // 1: encoder form -- rows [0, T) hold the sequence's keys, no causal
                     //    mask, |i - j| <= window on sliding layers; q_start unused
  float scale_log2;
  unsigned* item_ctr;  // [2]: next work item, CTAs done (zero between launches; set by the launcher)
};
cudaError_t launch_prefill_tc(const PrefillTcArgs& a, cudaStream_t s);

// Step a6 (bf16) for key spans of at most kMaxWinSplits x 64 keys per
// (sequence, kv head): one cluster of 64-key CTAs per (sequence, kv head),
// merged through distributed shared memory; no workspace.  Takes the
// AttnSimtArgs of a decode (mode 0, T = 1) with chunk = 64 and nsplit =
// decode_win_splits(span).  Used when its CTAs fit one wave
// (decode_win_eligible, units = batch x kv heads).
constexpr int kMaxWinSplits = 8;
bool decode_win_eligible(int dtype, int hd, int group, int span, int units);
int decode_win_splits(int span);
cudaError_t launch_decode_win(const AttnSimtArgs& a, cudaStream_t s);

// The projections around the path on the tcgen05 tensor cores: a bf16 GEMM
// out[M][N] = A[M][K] . Bw[N][K]^T (both operands K-major) whose epilogue is
//   epi 0: the q / k / v projections of a layer (A = the layer input x, Bw =
//          the stacked q, k, v rows with the attention-norm weight folded in):
//          the input RMSNorm's row scale, then per head the norm / RoPE / bf16
//          store of g4_kv_append_normrope (q to q_out, k and v to the cache);
//   epi 1: o_proj (A = attention output rows, Bw = Wo): the post-attention
//          RMSNorm over the N = D columns of a row (one cluster of CTAs per
//          row block) and the residual add, out = h + norm(A Bw^T) w.
struct GemmArgs {
  int epi;
  int M, N, K;
  int* err;
  // epi 0
  int B, T, H, Hkv, hd, max_len, ring, n_rot;
  float eps;       // per-head norm eps (epi 0) / post-attention norm eps (epi 1)
  float eps_in;    // input RMSNorm eps (epi 0)
  const float* q_w;
  const float* k_w;
  const int32_t* positions;  // [M]
  void* q_out;               // [M][H][hd]
  void* cache_k;             // [B][Hkv][max_len][hd]
  void* cache_v;
  float inv_freq[kMaxHalf];
  // epi 1
  const void* h;             // [M][N] residual
  void* out;                 // [M][N]
  const float* post_w;       // [N]
};
cudaError_t launch_gemm_tc(const GemmArgs& a, const void* A, const void* Bw, cudaStream_t s);

// Decode split plan shared by the workspace query and the launch.
// Workspace layout: ws_o, then ws_m, ws_l, tickets, each 256-byte aligned.
// win = 1: the windowed cluster kernel (launch_decode_win), no workspace.
constexpr int kMaxSplits = 128;
struct DecodePlan {
  int chunk;
  int nsplit;
  int win;
  size_t o_bytes, m_bytes, t_bytes;  // sizes of the four regions (ws_m and ws_l share m_bytes)
  size_t ws_bytes;
};
DecodePlan decode_plan(int dtype, int sliding, int window, int hd, int H, int Hkv, int B, int max_seq_len);
int sm_count();  // SMs of the current device

}  // namespace g4

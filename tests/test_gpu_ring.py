"""Parity of the sliding-window ring-buffer cache (g4_kv_cache.ring = 1)
against the float64 oracle's ring (``ring_slot`` / ``ring_rows``, pinned to
the linear-cache attention in test_oracle_pins.py).

A ring of C rows keeps position p in row p mod C.  The tests run sequences
well past C, so every kernel meets the wrap: the append (rows p mod C), the
tcgen05 prefill (key tiles at rows (128 t) mod C), the float32 prefill and
the split-KV decode (key stages split where the ring wraps), and the fused
decode step (the new row at (L-1) mod C).

Tolerances are those of the linear cache: stored rows (append) bf16 bit for
bit, f32 within 1e-4; attention bf16 max-abs 2e-2 and rel-L2 5e-3, f32
max-abs 1e-4.  Rings start NaN-filled: a row the oracle does not hold and
that a kernel read into a result would poison it, and after every call the
whole ring is compared with the oracle's, NaN rows included.
"""

import numpy as np
import pytest
import torch

from gemma_dual_geometry_gb300 import build as g4build
from gemma_dual_geometry_gb300 import g4attn as G
from gemma_dual_geometry_gb300 import workloads as W
from oracle import g4_oracle as O

from gpu_common import DEV, assert_attn_close, f64, geometry, nan_cache, oracle_lp, params_of

pytestmark = pytest.mark.gpu

S = W.SLIDING


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    g4build.build()
    G.lib()
    yield
    assert G.g4_take_device_error() == 0


def assert_ring_equal(gpu, ref, dtype, what):
    """Whole ring against the oracle's: NaN where neither wrote, stored values
    elsewhere (bf16 bit for bit, f32 within 1e-4)."""
    g = f64(gpu)
    nan_g, nan_r = np.isnan(g), np.isnan(ref)
    assert np.array_equal(nan_g, nan_r), f"{what}: written rows differ ({(nan_g != nan_r).sum()} values)"
    if dtype == W.BF16:
        bad = g[~nan_g] != ref[~nan_r]
        assert not bad.any(), f"{what}: {bad.sum()} stored values differ"
    elif (~nan_g).any():
        err = np.max(np.abs(g[~nan_g] - ref[~nan_r]))
        assert err <= 1e-4, f"{what}: max abs {err}"


class RingSeq:
    """B sequences streamed through one sliding layer whose cache is a ring of
    ``cap`` rows, on the GPU (C ABI) and in the oracle side by side.
    Sequence b starts ``off[b]`` positions ahead (a history chunk)."""

    def __init__(self, geo, B, cap, off, seed):
        self.geo, self.B, self.cap = geo, B, cap
        self.hd, self.H, self.Hkv, self.dt = geo["head_dim"], geo["n_heads"], geo["n_kv_heads"], geo["dtype"]
        self.seed = seed
        self.qw = W.norm_weight(self.hd, seed + 1)
        self.kw = W.norm_weight(self.hd, seed + 2)
        self.ck = nan_cache(B, self.Hkv, cap, self.hd, self.dt)
        self.cv = nan_cache(B, self.Hkv, cap, self.hd, self.dt)
        self.table = G.cache_table(1)
        G.set_cache(self.table, 0, self.ck, self.cv, S, self.hd, self.Hkv, cap, B, self.dt, ring=True)
        self.p = params_of(geo)
        self.lp = oracle_lp(geo)
        self.ok = np.full((B, self.Hkv, cap, self.hd), np.nan)
        self.ov = np.full((B, self.Hkv, cap, self.hd), np.nan)
        self.len = np.zeros(B, dtype=np.int64)  # positions appended so far
        self.calls = 0
        off = np.asarray(off, dtype=np.int64)
        if off.max() > 0:
            # history: sequence b appends positions [0, off[b]); the rest of
            # the chunk carries position -1, which is not written
            t = np.arange(int(off.max()))[None, :]
            pos = np.where(t < off[:, None], t, -1)
            self._append(pos)
            self.len = off.copy()

    def _inputs(self, T):
        self.calls += 1
        s = self.seed + 100 * self.calls
        B, H, Hkv, hd, dt = self.B, self.H, self.Hkv, self.hd, self.dt
        return (W.normal((B, T, H, hd), s + 1, dt), W.normal((B, T, Hkv, hd), s + 2, dt),
                W.normal((B, T, Hkv, hd), s + 3, dt))

    def _append(self, pos):
        """Append tokens at positions pos [B, T] on both sides; returns
        (gpu q_out, oracle q_out)."""
        B, T = pos.shape
        q, k, v = self._inputs(T)
        qd = q.to(DEV)
        q_out = torch.empty_like(qd)
        G.g4_kv_append_normrope(self.p, self.table, 0, qd, k.to(DEV), v.to(DEV), self.qw.to(DEV), self.kw.to(DEV),
                                torch.tensor(pos, dtype=torch.int32, device=DEV), B, T, q_out)
        # the oracle writes only the positions >= 0 (the GPU skips the rest)
        oq = np.zeros((B, T, self.H, self.hd))
        for b in range(B):
            keep = pos[b] >= 0
            if keep.any():
                oq[b:b + 1, keep] = O.kv_append_normrope(
                    self.lp, f64(q[b:b + 1, keep]), f64(k[b:b + 1, keep]), f64(v[b:b + 1, keep]), f64(self.qw),
                    f64(self.kw), pos[b:b + 1, keep], self.ok[b:b + 1], self.ov[b:b + 1], ring=True)
        torch.cuda.synchronize()
        assert_ring_equal(self.ck, self.ok, self.dt, "ring k after append")
        assert_ring_equal(self.cv, self.ov, self.dt, "ring v after append")
        return q_out, oq, (q, k, v)

    def prefill(self, T):
        """Append a chunk of T tokens per sequence, then prefill attention."""
        pos = self.len[:, None] + np.arange(T)[None, :]
        q_out, oq, _ = self._append(pos)
        out = torch.empty_like(q_out)
        qs = torch.tensor(self.len, dtype=torch.int32, device=DEV)
        G.g4_attn_prefill(self.p, self.table, 0, q_out, qs, self.B, T, out)
        torch.cuda.synchronize()
        self.len = self.len + T
        # the attention oracle on the GPU's own q_out (bit-equal to the
        # oracle's for bf16, checked) and the oracle's ring (equal to the GPU's)
        gq = f64(q_out)
        if self.dt == W.BF16:
            assert np.array_equal(gq, oq)
        ref = O.attention(gq, self.ok, self.ov, pos, self.len, self.Hkv, S, self.geo["window"],
                          self.geo["attn_scale"], ring=True)
        return f64(out), ref

    def decode(self, fused, max_seq_len=None):
        """One decode step per sequence (the new token at position len)."""
        B, H, Hkv, hd = self.B, self.H, self.Hkv, self.hd
        L = self.len + 1
        msl = int(max_seq_len or L.max())
        wsb = G.g4_attn_decode_workspace_size(self.p, B, msl)
        ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=DEV)
        out = torch.empty((B, H, hd), dtype=W.torch_dtype(self.dt), device=DEV)
        sl = torch.tensor(L, dtype=torch.int32, device=DEV)
        pos = (L - 1)[:, None]
        if fused:
            q, k, v = self._inputs(1)
            G.g4_decode_step(self.p, self.table, 0, q.to(DEV).view(B, H, hd), k.to(DEV).view(B, Hkv, hd),
                             v.to(DEV).view(B, Hkv, hd), self.qw.to(DEV), self.kw.to(DEV), sl, B, msl, out, ws, wsb)
            oq = O.kv_append_normrope(self.lp, f64(q), f64(k), f64(v), f64(self.qw), f64(self.kw), pos, self.ok,
                                      self.ov, ring=True)
            torch.cuda.synchronize()
            assert_ring_equal(self.ck, self.ok, self.dt, "ring k after decode step")
            assert_ring_equal(self.cv, self.ov, self.dt, "ring v after decode step")
        else:
            q_out, oq, _ = self._append(pos)
            G.g4_attn_decode(self.p, self.table, 0, q_out.view(B, H, hd), sl, B, msl, out, ws, wsb)
            torch.cuda.synchronize()
        self.len = L
        ref = O.attention(oq, self.ok, self.ov, pos, L, Hkv, S, self.geo["window"], self.geo["attn_scale"], ring=True)
        return f64(out), ref[:, 0]


def test_ring_bf16_chunked_prefill_then_decode_past_the_wrap():
    # 1024-row ring, window 512: chunks of 384 tokens (384 + 511 <= 1024)
    # carry both sequences round the ring more than once; sequence 1 runs 77
    # positions ahead, so its tiles and stages sit at other ring offsets.
    geo = geometry(S, 256, H=8, Hkv=2, window=512)
    r = RingSeq(geo, B=2, cap=1024, off=[0, 77], seed=900)
    for c in range(6):
        gpu, ref = r.prefill(384)
        assert_attn_close(gpu, ref, W.BF16, f"ring prefill chunk {c}")
    for step in range(3):
        gpu, ref = r.decode(fused=step != 1)
        assert_attn_close(gpu, ref, W.BF16, f"ring decode step {step}")
    assert r.len.max() > 2 * r.cap


def test_ring_bf16_prefill_chunk_filling_the_ring_exactly():
    # T + window - 1 == capacity: the first query's oldest key sits in the
    # row the chunk's last token is about to reach
    geo = geometry(S, 256, H=4, Hkv=2, window=129)
    r = RingSeq(geo, B=2, cap=256, off=[5, 200], seed=910)
    for c in range(4):
        gpu, ref = r.prefill(128)
        assert_attn_close(gpu, ref, W.BF16, f"exact-fit ring prefill chunk {c}")


def test_ring_f32_prefill_and_decode_with_unaligned_capacity():
    # float32 runs the CUDA-core kernel for prefill too; a 35-row ring is no
    # multiple of the key stage, so stages wrap mid-way
    geo = geometry(S, 64, H=4, Hkv=2, window=16, dtype=W.F32)
    r = RingSeq(geo, B=3, cap=35, off=[0, 3, 34], seed=920)
    for c in range(4):
        gpu, ref = r.prefill(20)
        assert_attn_close(gpu, ref, W.F32, f"f32 ring prefill chunk {c}")
    for step in range(4):
        gpu, ref = r.decode(fused=step % 2 == 0)
        assert_attn_close(gpu, ref, W.F32, f"f32 ring decode step {step}")


@pytest.mark.parametrize("dtype", [W.BF16, W.F32])
def test_ring_of_one_window_decode_at_many_wrap_offsets(dtype):
    # The smallest ring (capacity = window) serves decode.  Each sequence's
    # history is a random ring at its own length, so the window's wrap falls
    # at a different key (and split) in each; lengths below the capacity
    # leave unwritten (NaN) rows that must not be read.
    W_ = 512
    geo = geometry(S, 256, H=8, Hkv=2, window=W_, dtype=dtype)
    lens = np.array([1, 2, 300, 511, 512, 513, 700, 1024, 1025, 4097, 5000, 123457])
    B = len(lens)
    for fused in (True, False):
        r = RingSeq(geo, B=B, cap=W_, off=[0] * B, seed=930 + int(fused))
        hist_k = W.normal((B, 2, W_, 256), 931, dtype)
        hist_v = W.normal((B, 2, W_, 256), 932, dtype)
        for b, L in enumerate(lens):
            n = L - 1  # positions already in the sequence
            if n < W_:
                hist_k[b, :, n:] = float("nan")
                hist_v[b, :, n:] = float("nan")
        r.ck.copy_(hist_k.to(DEV))
        r.cv.copy_(hist_v.to(DEV))
        r.ok, r.ov = f64(hist_k), f64(hist_v)
        r.len = lens - 1
        for step in range(2):
            gpu, ref = r.decode(fused=fused, max_seq_len=200000)
            assert_attn_close(gpu, ref, dtype, f"ring decode fused={fused} step {step}")

"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and the float64 oracle on the same seeded inputs.

The oracle always starts from the raw inputs (q/k/v projections, norm
weights, positions, prefilled cache rows); it never reads anything the CUDA
path produced.
"""

import numpy as np
import torch

from gemma_dual_geometry_gb300 import g4attn as G
from gemma_dual_geometry_gb300 import workloads as W
from oracle import g4_oracle as O

DEV = "cuda"


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def params_of(geo, src=-1):
    return G.layer_params(geo["layer_type"], geo["head_dim"], geo["n_heads"], geo["n_kv_heads"], geo["window"],
                          geo["theta"], geo["rotary_fraction"], geo["eps"], geo["attn_scale"], src, geo["dtype"])


def oracle_lp(geo, src=-1):
    d = dict(geo)
    d["kv_share_src"] = src
    return d


def geometry(layer_type, head_dim, H=8, Hkv=2, window=512, theta=None, frac=None, dtype=W.BF16):
    if theta is None:
        theta = 1e4 if layer_type == W.SLIDING else 1e6
    if frac is None:
        frac = 1.0 if layer_type == W.SLIDING else 0.25
    return dict(layer_type=layer_type, head_dim=head_dim, n_heads=H, n_kv_heads=Hkv,
                window=window if layer_type == W.SLIDING else 0, theta=theta, rotary_fraction=frac,
                eps=W.EPS, attn_scale=W.ATTN_SCALE, dtype=dtype)


def nan_cache(B, Hkv, Lmax, hd, dtype):
    return torch.full((B, Hkv, Lmax, hd), float("nan"), dtype=W.torch_dtype(dtype), device=DEV)


def assert_stored_close(gpu, ref, dtype, what=""):
    """Stored values of the append against the oracle's: bf16 bit for bit
    (both sides round the exact normed / roped value to nearest even), f32
    within max-abs 1e-4."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(gpu)), what
    if dtype == W.BF16:
        bad = gpu != ref
        assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} values differ, e.g. {gpu[bad][:4]} vs {ref[bad][:4]}"
    else:
        err = np.max(np.abs(gpu - ref)) if gpu.size else 0.0
        assert err <= 1e-4, f"{what}: max abs {err}"


def attn_errors(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    max_abs = float(np.max(np.abs(gpu - ref))) if gpu.size else 0.0
    rel_l2 = float(np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-30))
    return max_abs, rel_l2


def assert_attn_close(gpu, ref, dtype, what=""):
    """Attention output tolerances: f32 max-abs 1e-4; bf16 max-abs 2e-2 and rel-L2 5e-3.

    ``ref`` is the oracle's exact (float64, unrounded) output, so the bound
    covers the storage rounding of the stored value (half an ulp) plus the
    computation error.  Comparing against a separately rounded reference
    would count a full ulp (1/32 for |o| in [4, 8)) whenever the two land on
    either side of a rounding boundary."""
    assert np.all(np.isfinite(np.asarray(gpu))), f"{what}: non-finite output"
    max_abs, rel_l2 = attn_errors(gpu, ref)
    if dtype == W.BF16:
        assert max_abs <= 2e-2 and rel_l2 <= 5e-3, f"{what}: max_abs {max_abs:.3e} rel_l2 {rel_l2:.3e}"
    else:
        assert max_abs <= 1e-4, f"{what}: max_abs {max_abs:.3e}"
    return max_abs, rel_l2


class LayerRun:
    """One layer's prefill through the C ABI: append (+ optional earlier chunk) then attention."""

    def __init__(self, geo, B, T, Lmax, q_start, seed, prior=True):
        self.geo, self.B, self.T, self.Lmax = geo, B, T, Lmax
        self.q_start = np.asarray(q_start, dtype=np.int64)
        hd, H, Hkv, dt = geo["head_dim"], geo["n_heads"], geo["n_kv_heads"], geo["dtype"]
        self.Tp = int(self.q_start.max()) if prior else 0
        # raw inputs on the CPU (seeded); the earlier chunk first
        self.prior = None
        if self.Tp > 0:
            self.prior = dict(q=W.normal((B, self.Tp, H, hd), seed + 11, dt),
                              k=W.normal((B, self.Tp, Hkv, hd), seed + 12, dt),
                              v=W.normal((B, self.Tp, Hkv, hd), seed + 13, dt))
        self.x = dict(q=W.normal((B, T, H, hd), seed + 1, dt), k=W.normal((B, T, Hkv, hd), seed + 2, dt),
                      v=W.normal((B, T, Hkv, hd), seed + 3, dt), q_norm_w=W.norm_weight(hd, seed + 4),
                      k_norm_w=W.norm_weight(hd, seed + 5))

    def positions(self):
        return self.q_start[:, None] + np.arange(self.T)[None, :]

    def prior_positions(self):
        # t < q_start[b] goes to row t; the rest is pushed past the cache (not written)
        t = np.arange(self.Tp)[None, :]
        return np.where(t < self.q_start[:, None], t, self.Lmax + 5)

    def run_gpu(self, table=None, layer=0):
        g, B, T = self.geo, self.B, self.T
        hd, Hkv, dt = g["head_dim"], g["n_kv_heads"], g["dtype"]
        self.ck = nan_cache(B, Hkv, self.Lmax, hd, dt)
        self.cv = nan_cache(B, Hkv, self.Lmax, hd, dt)
        if table is None:
            table = G.cache_table(1)
        G.set_cache(table, layer, self.ck, self.cv, g["layer_type"], hd, Hkv, self.Lmax, B, dt)
        self.table = table
        p = params_of(g)
        qw = self.x["q_norm_w"].to(DEV)
        kw = self.x["k_norm_w"].to(DEV)
        if self.prior is not None:
            pq = self.prior["q"].to(DEV)
            pos = torch.tensor(self.prior_positions(), dtype=torch.int32, device=DEV)
            G.g4_kv_append_normrope(p, table, layer, pq, self.prior["k"].to(DEV), self.prior["v"].to(DEV), qw, kw,
                                    pos, B, self.Tp, torch.empty_like(pq))
        q = self.x["q"].to(DEV)
        self.q_out = torch.empty_like(q)
        pos = torch.tensor(self.positions(), dtype=torch.int32, device=DEV)
        G.g4_kv_append_normrope(p, table, layer, q, self.x["k"].to(DEV), self.x["v"].to(DEV), qw, kw, pos, B, T,
                                self.q_out)
        self.out = torch.empty_like(q)
        qs = torch.tensor(self.q_start, dtype=torch.int32, device=DEV)
        G.g4_attn_prefill(p, table, layer, self.q_out, qs, B, T, self.out)
        torch.cuda.synchronize()
        return self

    def run_oracle(self):
        g, B = self.geo, self.B
        hd, Hkv = g["head_dim"], g["n_kv_heads"]
        lp = oracle_lp(g)
        ck = np.zeros((B, Hkv, self.Lmax, hd))
        cv = np.zeros((B, Hkv, self.Lmax, hd))
        qw, kw = f64(self.x["q_norm_w"]), f64(self.x["k_norm_w"])
        if self.prior is not None:
            # only the rows t < q_start[b] of the earlier chunk reach the cache
            for b in range(B):
                n = int(self.q_start[b])
                if n == 0:
                    continue
                O.kv_append_normrope(lp, f64(self.prior["q"][b:b + 1, :n]), f64(self.prior["k"][b:b + 1, :n]),
                                     f64(self.prior["v"][b:b + 1, :n]), qw, kw, np.arange(n)[None, :],
                                     ck[b:b + 1], cv[b:b + 1])
        pos = self.positions()
        self.o_q = O.kv_append_normrope(lp, f64(self.x["q"]), f64(self.x["k"]), f64(self.x["v"]), qw, kw, pos, ck, cv)
        self.o_ck, self.o_cv = ck, cv
        self.o_out = O.attention(self.o_q, ck, cv, pos, self.q_start + self.T, Hkv, g["layer_type"],
                                 g["window"], g["attn_scale"])
        return self


def run_decode(geo, lens, Lmax, seed, max_seq_len=None, fused=False, return_cache=False):
    """Cache rows [0, L-1) prefilled with N(0,1), the new token appended at
    L-1, rows >= L NaN; then decode through the C ABI -- append + decode, or
    the fused decode step.  Returns (gpu_out, oracle_out, workspace_bytes)
    (+ (gpu k cache, gpu v cache, oracle k, oracle v) with return_cache)."""
    B = len(lens)
    hd, H, Hkv, dt = geo["head_dim"], geo["n_heads"], geo["n_kv_heads"], geo["dtype"]
    lens = np.asarray(lens, dtype=np.int64)
    pk = W.normal((B, Hkv, Lmax, hd), seed + 1, dt)
    pv = W.normal((B, Hkv, Lmax, hd), seed + 2, dt)
    for b in range(B):
        pk[b, :, lens[b] - 1:] = float("nan")
        pv[b, :, lens[b] - 1:] = float("nan")
    x = dict(q=W.normal((B, 1, H, hd), seed + 3, dt), k=W.normal((B, 1, Hkv, hd), seed + 4, dt),
             v=W.normal((B, 1, Hkv, hd), seed + 5, dt), qw=W.norm_weight(hd, seed + 6), kw=W.norm_weight(hd, seed + 7))
    ck, cv = pk.to(DEV), pv.to(DEV)
    table = G.cache_table(1)
    G.set_cache(table, 0, ck, cv, geo["layer_type"], hd, Hkv, Lmax, B, dt)
    p = params_of(geo)
    q = x["q"].to(DEV)
    msl = int(max_seq_len or lens.max())
    wsb = G.g4_attn_decode_workspace_size(p, B, msl)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=DEV)
    out = torch.empty((B, H, hd), dtype=W.torch_dtype(dt), device=DEV)
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    if fused:
        G.g4_decode_step(p, table, 0, q.view(B, H, hd), x["k"].to(DEV).view(B, Hkv, hd),
                         x["v"].to(DEV).view(B, Hkv, hd), x["qw"].to(DEV), x["kw"].to(DEV), sl, B, msl, out, ws, wsb)
    else:
        q_out = torch.empty_like(q)
        pos = torch.tensor(lens - 1, dtype=torch.int32, device=DEV).view(B, 1)
        G.g4_kv_append_normrope(p, table, 0, q, x["k"].to(DEV), x["v"].to(DEV), x["qw"].to(DEV), x["kw"].to(DEV),
                                pos, B, 1, q_out)
        G.g4_attn_decode(p, table, 0, q_out.view(B, H, hd), sl, B, msl, out, ws, wsb)
    torch.cuda.synchronize()
    # oracle: same prefilled rows, its own append of the new token
    lp = oracle_lp(geo)
    ok, ov = f64(pk), f64(pv)
    oq = O.kv_append_normrope(lp, f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["qw"]), f64(x["kw"]),
                              (lens - 1)[:, None], ok, ov)
    ref = O.attention(oq, ok, ov, (lens - 1)[:, None], lens, Hkv, geo["layer_type"], geo["window"], 1.0)
    if return_cache:
        return f64(out), ref[:, 0], wsb, (ck, cv, ok, ov)
    return f64(out), ref[:, 0], wsb

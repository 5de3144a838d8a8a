"""Parity of the bidirectional (encoder) attention, g4_attn_encoder, against
the float64 oracle's ``attention_bidirectional`` (taconite-embeddinggemma2
``model.rs``: ``text_attention``; pinned in test_oracle_pins.py by SDPA with
a band mask, loops and reversal symmetry).

The tokens' q/k/v go through g4_kv_append_normrope at positions 0..T-1 (its
stores checked bit for bit against the oracle's append for bf16), then the
encoder attention runs on the GPU's q_out and cache, and the oracle on the
same values.  Tolerances as for the causal path: bf16 max-abs 2e-2 and
rel-L2 5e-3, f32 max-abs 1e-4, against the oracle's exact output.  Cache
rows past T hold NaN, so a key read past the sequence poisons the result.
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

S, F = W.SLIDING, W.FULL


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    g4build.build()
    G.lib()
    yield
    assert G.g4_take_device_error() == 0


def run_encoder(geo, B, T, seed, Lmax=None):
    hd, H, Hkv, dt = geo["head_dim"], geo["n_heads"], geo["n_kv_heads"], geo["dtype"]
    Lmax = Lmax or T + 37
    x = dict(q=W.normal((B, T, H, hd), seed + 1, dt), k=W.normal((B, T, Hkv, hd), seed + 2, dt),
             v=W.normal((B, T, Hkv, hd), seed + 3, dt), qw=W.norm_weight(hd, seed + 4),
             kw=W.norm_weight(hd, seed + 5))
    ck = nan_cache(B, Hkv, Lmax, hd, dt)
    cv = nan_cache(B, Hkv, Lmax, hd, dt)
    table = G.cache_table(1)
    G.set_cache(table, 0, ck, cv, geo["layer_type"], hd, Hkv, Lmax, B, dt)
    p = params_of(geo)
    q = x["q"].to(DEV)
    q_out = torch.empty_like(q)
    pos_np = np.broadcast_to(np.arange(T)[None, :], (B, T))
    pos = torch.tensor(pos_np, dtype=torch.int32, device=DEV)
    G.g4_kv_append_normrope(p, table, 0, q, x["k"].to(DEV), x["v"].to(DEV), x["qw"].to(DEV), x["kw"].to(DEV), pos,
                            B, T, q_out)
    out = torch.empty_like(q)
    G.g4_attn_encoder(p, table, 0, q_out, B, T, out)
    torch.cuda.synchronize()
    # the append against the oracle's (bit for bit in bf16)
    ok = np.zeros((B, Hkv, Lmax, hd))
    ov = np.zeros((B, Hkv, Lmax, hd))
    oq = O.kv_append_normrope(oracle_lp(geo), f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["qw"]), f64(x["kw"]),
                              pos_np, ok, ov)
    gq, gk, gv = f64(q_out), f64(ck), f64(cv)
    if dt == W.BF16:
        assert np.array_equal(gq, oq)
        assert np.array_equal(gk[:, :, :T], ok[:, :, :T]) and np.array_equal(gv[:, :, :T], ov[:, :, :T])
    assert np.isnan(gk[:, :, T:]).all() and np.isnan(gv[:, :, T:]).all()
    ref = O.attention_bidirectional(gq, gk, gv, T, Hkv, geo["layer_type"], geo["window"], geo["attn_scale"])
    # the table holds raw device pointers: the cache tensors must stay alive
    # as long as it is used (a later launch on it would read freed memory)
    run_encoder.last = dict(table=table, q_out=q_out, out=out, caches=(ck, cv))
    return f64(out), ref


ENCODER_CASES = [
    # dtype, layer type, head_dim, window, B, T
    (W.BF16, S, 256, 512, 2, 2048),   # several items per persistent CTA, windows wider than a tile
    (W.BF16, S, 256, 100, 2, 1000),   # window narrower than a tile, ragged T
    (W.BF16, S, 256, 1, 1, 300),      # the token and its two neighbours
    (W.BF16, F, 512, 0, 2, 700),      # global layer: every key (two O halves per query tile)
    (W.BF16, S, 128, 64, 3, 257),
    (W.BF16, F, 64, 0, 2, 129),
    (W.F32, S, 64, 16, 2, 77),
    (W.F32, F, 128, 0, 2, 60),
]


@pytest.mark.parametrize("dtype,lt,hd,window,B,T", ENCODER_CASES)
def test_encoder_parity(dtype, lt, hd, window, B, T):
    geo = geometry(lt, hd, H=8 if hd <= 256 else 4, Hkv=2, window=window, theta=1e4 if lt == S else 1e6, frac=1.0,
                   dtype=dtype)
    gpu, ref = run_encoder(geo, B, T, seed=1200 + hd + T)
    assert_attn_close(gpu, ref, dtype, f"encoder {lt} hd {hd} W {window} T {T}")


def test_encoder_single_token_and_window_reaching_every_key():
    # T = 1: each head returns its kv head's v row (as stored)
    geo = geometry(S, 256, H=8, Hkv=2, window=512, frac=1.0)
    gpu, ref = run_encoder(geo, 3, 1, seed=1300)
    assert_attn_close(gpu, ref, W.BF16, "encoder T=1")
    # a sliding window of T - 1 or more sees every key: same as the global form
    for window in (299, 300, 5000):
        geo_s = geometry(S, 256, H=8, Hkv=2, window=window, frac=1.0)
        g_s, ref_s = run_encoder(geo_s, 2, 300, seed=1301)
        geo_f = dict(geo_s, layer_type=F, window=0)
        g_f, ref_f = run_encoder(geo_f, 2, 300, seed=1301)
        assert np.array_equal(ref_s, ref_f)
        assert_attn_close(g_s, ref_s, W.BF16, f"encoder W={window}")
        assert np.array_equal(g_s, g_f)   # same kernel, same visible keys, same arithmetic


def test_encoder_last_row_is_the_causal_window_one_wider():
    # The last token sees [T-1-W, T-1] in the encoder form and with a causal
    # window of W + 1: the same keys in the same tiles, so the tcgen05
    # prefill's last rows equal the encoder's bit for bit.  The first token
    # differs: the causal form sees key 0 alone there (o = v_0).
    B, T, Wn = 2, 600, 200
    geo = geometry(S, 256, H=8, Hkv=2, window=Wn, frac=1.0)
    gpu, ref = run_encoder(geo, B, T, seed=1302)
    assert_attn_close(gpu, ref, W.BF16, "encoder")
    r = run_encoder.last
    p_causal = params_of(dict(geo, window=Wn + 1))
    out_c = torch.empty_like(r["out"])
    qs = torch.zeros(B, dtype=torch.int32, device=DEV)
    G.g4_attn_prefill(p_causal, r["table"], 0, r["q_out"], qs, B, T, out_c)
    torch.cuda.synchronize()
    oc = f64(out_c)
    assert np.array_equal(oc[:, T - 1], gpu[:, T - 1])
    assert np.abs(oc[:, 0] - gpu[:, 0]).max() > 0.1

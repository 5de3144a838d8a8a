"""attention_k_eq_v through the C ABI: a full layer whose v projection is
its k projection (turbospark-runtime gemma4: ``v_name`` is ``k_name`` when
``is_full && arch.attention_k_eq_v``) passes its raw k as v_in as well.

The append and the fused decode step then store v = the weight-less norm of
the raw k (unroped) next to the normed, roped k; checked against the
float64 oracle's append of the same raw k as both inputs (bf16 bit for bit)
and its attention over those rows (max-abs 2e-2, rel-L2 5e-3).
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

F = W.FULL


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    g4build.build()
    G.lib()
    yield
    assert G.g4_take_device_error() == 0


def test_k_eq_v_append_then_fused_decode_step():
    geo = geometry(F, 512, H=4, Hkv=2)
    hd, H, Hkv, dt = 512, 4, 2, W.BF16
    B, T, Lmax = 3, 40, 64
    q = W.normal((B, T, H, hd), 1401, dt)
    k = W.normal((B, T, Hkv, hd), 1402, dt)
    qw, kw = W.norm_weight(hd, 1403), W.norm_weight(hd, 1404)
    ck = nan_cache(B, Hkv, Lmax, hd, dt)
    cv = nan_cache(B, Hkv, Lmax, hd, dt)
    table = G.cache_table(1)
    G.set_cache(table, 0, ck, cv, F, hd, Hkv, Lmax, B, dt)
    p = params_of(geo)
    lp = oracle_lp(geo)
    pos_np = np.broadcast_to(np.arange(T)[None, :], (B, T))
    kd = k.to(DEV)
    q_out = torch.empty((B, T, H, hd), dtype=W.torch_dtype(dt), device=DEV)
    G.g4_kv_append_normrope(p, table, 0, q.to(DEV), kd, kd, qw.to(DEV), kw.to(DEV),
                            torch.tensor(pos_np, dtype=torch.int32, device=DEV), B, T, q_out)
    ok = np.full((B, Hkv, Lmax, hd), np.nan)
    ov = np.full((B, Hkv, Lmax, hd), np.nan)
    oq = O.kv_append_normrope(lp, f64(q), f64(k), f64(k), f64(qw), f64(kw), pos_np, ok, ov)
    torch.cuda.synchronize()
    assert np.array_equal(f64(q_out), oq)
    assert np.array_equal(f64(ck), ok, equal_nan=True)
    assert np.array_equal(f64(cv), ov, equal_nan=True)

    # one decode step with the raw k of the new token as its raw v too
    L = T + 1
    q1 = W.normal((B, 1, H, hd), 1405, dt)
    k1 = W.normal((B, 1, Hkv, hd), 1406, dt)
    sl = torch.full((B,), L, dtype=torch.int32, device=DEV)
    wsb = G.g4_attn_decode_workspace_size(p, B, L)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=DEV)
    out = torch.empty((B, H, hd), dtype=W.torch_dtype(dt), device=DEV)
    k1d = k1.to(DEV).view(B, Hkv, hd)
    G.g4_decode_step(p, table, 0, q1.to(DEV).view(B, H, hd), k1d, k1d, qw.to(DEV), kw.to(DEV), sl, B, L, out, ws,
                     wsb)
    pos1 = np.full((B, 1), T)
    oq1 = O.kv_append_normrope(lp, f64(q1), f64(k1), f64(k1), f64(qw), f64(kw), pos1, ok, ov)
    ref = O.attention(oq1, ok, ov, pos1, np.full(B, L), Hkv, F, 0, 1.0)
    torch.cuda.synchronize()
    assert np.array_equal(f64(ck), ok, equal_nan=True)
    assert np.array_equal(f64(cv), ov, equal_nan=True)
    assert_attn_close(f64(out), ref[:, 0], dt, "k_eq_v decode step")

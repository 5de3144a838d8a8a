"""g4_attn_decode_noalloc: decode attention for callers that cannot allocate.

Some callers of this library are handed only their input and output buffers
-- a plugin inside a host framework that owns every device allocation, or a
serving loop that must not call cudaMalloc mid-request because it
synchronises the device and can fail.  For them the library carries a fixed
8 MiB scratch array in device memory and g4_attn_decode_noalloc uses it in
place of the caller's workspace.  These tests call it through the C ABI and
check it against g4_attn_decode (with a caller-allocated workspace) on two
calls in a row, the second overwriting what the first left in the shared
array: bit for bit, since both run the same kernels with the same split plan,
and both against the float64 oracle.  A plan larger than the array is
refused before anything is launched or written.

This file is collected last on purpose, and passes both alone in a fresh
process and after the other tests.
"""

import numpy as np
import pytest
import torch

from gemma_dual_geometry_gb300 import build as g4build
from gemma_dual_geometry_gb300 import g4attn as G
from gemma_dual_geometry_gb300 import workloads as W
from oracle import g4_oracle as O

from gpu_common import DEV, assert_attn_close, f64, geometry, oracle_lp, params_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    g4build.build()
    G.lib()
    yield
    assert G.g4_take_device_error() == 0


def _decode_inputs(geo, lens, Lmax, seed):
    """Cache with rows [0, L-1) drawn N(0,1), the new token appended at L-1
    through the C ABI, rows >= L NaN; returns what a decode call needs and the
    oracle's output computed from the same raw inputs (its own append)."""
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
    q_out = torch.empty_like(q)
    pos = torch.tensor(lens - 1, dtype=torch.int32, device=DEV).view(B, 1)
    G.g4_kv_append_normrope(p, table, 0, q, x["k"].to(DEV), x["v"].to(DEV), x["qw"].to(DEV), x["kw"].to(DEV), pos,
                            B, 1, q_out)
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    # the oracle: same prefilled rows, its own append of the new token
    ok, ov = f64(pk), f64(pv)
    oq = O.kv_append_normrope(oracle_lp(geo), f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["qw"]), f64(x["kw"]),
                              (lens - 1)[:, None], ok, ov)
    ref = O.attention(oq, ok, ov, (lens - 1)[:, None], lens, Hkv, geo["layer_type"], geo["window"], 1.0)[:, 0]
    return dict(p=p, table=table, q=q_out.view(B, H, hd), sl=sl, B=B, msl=int(lens.max()), keep=(ck, cv),
                out_shape=(B, H, hd), tdt=W.torch_dtype(dt), dtype=dt, ref=ref)


def _with_workspace(x):
    wsb = G.g4_attn_decode_workspace_size(x["p"], x["B"], x["msl"])
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=DEV)
    out = torch.empty(x["out_shape"], dtype=x["tdt"], device=DEV)
    G.g4_attn_decode(x["p"], x["table"], 0, x["q"], x["sl"], x["B"], x["msl"], out, ws, wsb)
    torch.cuda.synchronize()
    return out, wsb


def _no_alloc(x):
    out = torch.empty(x["out_shape"], dtype=x["tdt"], device=DEV)
    G.g4_attn_decode_noalloc(x["p"], x["table"], 0, x["q"], x["sl"], x["B"], x["msl"], out)
    torch.cuda.synchronize()
    return out


def test_no_alloc_decode_matches_workspace_decode_on_two_calls_in_a_row():
    # call 1: full layer, head_dim 512, ragged lengths (many splits)
    a = _decode_inputs(geometry(W.FULL, 512), [1, 130, 2047, 3000, 777], 3008, seed=41)
    # call 2: sliding layer, head_dim 256, a window of 1024 keys (spans above
    # 512 keys go through the split kernel and its scratch), other lengths
    b = _decode_inputs(geometry(W.SLIDING, 256, window=1024), [5, 600, 2500], 2504, seed=42)
    ref_a, ws_a = _with_workspace(a)
    ref_b, ws_b = _with_workspace(b)
    assert ws_a > 0 and ws_b > 0          # both plans really use split-KV scratch
    got_a = _no_alloc(a)
    got_b = _no_alloc(b)                  # overwrites what call 1 left in the array
    for got, ws_out, x in ((got_a, ref_a, a), (got_b, ref_b, b)):
        # same kernels, same split plan: the same bits
        assert torch.equal(got, ws_out), "no-alloc decode differs from the workspace decode"
        assert_attn_close(f64(got), x["ref"], x["dtype"], "no-alloc decode vs oracle")
    # and once more on the first inputs, after the second call
    assert torch.equal(_no_alloc(a), ref_a)


def test_no_alloc_decode_refuses_plans_beyond_its_scratch():
    # many sequences of one kv head (group 8, head_dim 256): find a batch
    # whose split plan needs more partials than the built-in array holds
    geo = geometry(W.SLIDING, 256, H=8, Hkv=1, window=1024)
    p = params_of(geo)
    L = 1024
    B = next(b for b in range(64, 4096, 8) if G.g4_attn_decode_workspace_size(p, b, L) > G.G4_NOALLOC_SCRATCH_BYTES)
    # real device buffers of the declared shapes, so that a regression in the
    # size check fails this assertion instead of touching memory it should not
    dt = W.torch_dtype(W.BF16)
    ck = torch.zeros((B, 1, L, 256), dtype=dt, device=DEV)
    cv = torch.zeros_like(ck)
    q = torch.zeros((B, 8, 256), dtype=dt, device=DEV)
    sl = torch.full((B,), L, dtype=torch.int32, device=DEV)
    out = torch.full((B, 8, 256), 7.0, dtype=dt, device=DEV)
    table = G.cache_table(1)
    G.set_cache(table, 0, ck, cv, W.SLIDING, 256, 1, L, B, W.BF16)
    torch.cuda.synchronize()
    with pytest.raises(G.G4Error) as e:
        G.g4_attn_decode_noalloc(p, table, 0, q, sl, B, L, out)
    assert e.value.status == G.G4_ERR_WORKSPACE
    assert "built into the library" in str(e.value)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())       # nothing was launched

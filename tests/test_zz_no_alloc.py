"""g4_attn_decode_noalloc: decode attention for callers that cannot allocate.

Some callers of this library are handed only their input and output buffers
-- a plugin inside a host framework that owns every device allocation, or a
serving loop that must not call cudaMalloc mid-request because it
synchronises the device and can fail.  For them the library carries a fixed
8 MiB scratch array in device memory and g4_attn_decode_noalloc uses it in
place of the caller's workspace.  These tests call it through the C ABI and
check it against g4_attn_decode (with a caller-allocated workspace) on two
calls in a row, the second overwriting what the first left in the shared
array, and that a plan larger than the array is refused before any launch.

This file is collected last on purpose, and passes both alone in a fresh
process and after the other tests.
"""

import numpy as np
import pytest
import torch

from gemma_dual_geometry_gb300 import build as g4build
from gemma_dual_geometry_gb300 import g4attn as G
from gemma_dual_geometry_gb300 import workloads as W

from gpu_common import DEV, assert_attn_close, f64, geometry, params_of

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
    through the C ABI, rows >= L NaN; returns what a decode call needs."""
    B = len(lens)
    hd, H, Hkv, dt = geo["head_dim"], geo["n_heads"], geo["n_kv_heads"], geo["dtype"]
    lens = np.asarray(lens, dtype=np.int64)
    ck = W.normal((B, Hkv, Lmax, hd), seed + 1, dt)
    cv = W.normal((B, Hkv, Lmax, hd), seed + 2, dt)
    for b in range(B):
        ck[b, :, lens[b] - 1:] = float("nan")
        cv[b, :, lens[b] - 1:] = float("nan")
    ck, cv = ck.to(DEV), cv.to(DEV)
    table = G.cache_table(1)
    G.set_cache(table, 0, ck, cv, geo["layer_type"], hd, Hkv, Lmax, B, dt)
    p = params_of(geo)
    q = W.normal((B, 1, H, hd), seed + 3, dt).to(DEV)
    q_out = torch.empty_like(q)
    pos = torch.tensor(lens - 1, dtype=torch.int32, device=DEV).view(B, 1)
    G.g4_kv_append_normrope(p, table, 0, q, W.normal((B, 1, Hkv, hd), seed + 4, dt).to(DEV),
                            W.normal((B, 1, Hkv, hd), seed + 5, dt).to(DEV), W.norm_weight(hd, seed + 6).to(DEV),
                            W.norm_weight(hd, seed + 7).to(DEV), pos, B, 1, q_out)
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    return dict(p=p, table=table, q=q_out.view(B, H, hd), sl=sl, B=B, msl=int(lens.max()), keep=(ck, cv),
                out_shape=(B, H, hd), tdt=W.torch_dtype(dt), dtype=dt)


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
    # call 2: sliding layer, head_dim 256, other shapes and lengths
    b = _decode_inputs(geometry(W.SLIDING, 256, window=512), [5, 600, 2500], 2504, seed=42)
    ref_a, ws_a = _with_workspace(a)
    ref_b, ws_b = _with_workspace(b)
    assert ws_a > 0 and ws_b > 0          # both plans really use split-KV scratch
    got_a = _no_alloc(a)
    got_b = _no_alloc(b)                  # overwrites what call 1 left in the array
    for got, ref, x in ((got_a, ref_a, a), (got_b, ref_b, b)):
        assert_attn_close(f64(got), f64(ref), x["dtype"], "no-alloc decode vs workspace decode")
    # and once more on the first inputs, after the second call
    assert_attn_close(f64(_no_alloc(a)), f64(ref_a), a["dtype"], "repeat")


def test_no_alloc_decode_refuses_plans_beyond_its_scratch():
    # many sequences of one kv head (group 8, head_dim 256): find a batch
    # whose split plan needs more partials than the built-in array holds
    geo = geometry(W.SLIDING, 256, H=8, Hkv=1, window=1024)
    p = params_of(geo)
    B = next(b for b in range(64, 4096, 8) if G.g4_attn_decode_workspace_size(p, b, 1024) > G.G4_NOALLOC_SCRATCH_BYTES)
    fake = 0x7f0000000000
    table = G.cache_table(1)
    G.set_cache(table, 0, fake, fake + 4096, W.SLIDING, 256, 1, 1024, B, W.BF16)
    with pytest.raises(G.G4Error) as e:
        G.g4_attn_decode_noalloc(p, table, 0, fake, fake, B, 1024, fake, stream=0)
    assert e.value.status == G.G4_ERR_WORKSPACE
    assert "built into the library" in str(e.value)

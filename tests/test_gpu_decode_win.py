"""Decode attention over short key spans (at most 512 keys per (sequence,
kv head): sliding windows, and full layers early in a sequence) in bf16,
which runs on the windowed cluster kernel: one cluster of 64-key CTAs per
(sequence, kv head), merged through distributed shared memory, no workspace.

Checked against the float64 oracle (its own append of the new token from the
same raw inputs) at every GQA group and head width the kernel is built for,
at lengths on both sides of the 64-key CTA boundaries and of the window, in
the plain and the fused (append + attention) forms; the fused form's new
cache rows bit for bit.
"""

import numpy as np
import pytest
import torch

from gemma_dual_geometry_gb300 import build as g4build
from gemma_dual_geometry_gb300 import g4attn as G
from gemma_dual_geometry_gb300 import workloads as W

from gpu_common import assert_attn_close, assert_stored_close, f64, geometry, params_of, run_decode

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


CASES = [
    # (layer type, head_dim, H, Hkv, window, lengths)
    (S, 256, 8, 2, 512, [1, 2, 63, 64, 65, 511, 512, 513, 700, 4097]),
    (S, 256, 16, 2, 512, [1, 64, 300, 512, 1000]),      # group 8
    (S, 256, 2, 2, 512, [1, 129, 512, 513]),            # group 1
    (S, 256, 4, 2, 100, [1, 99, 100, 101, 250]),        # group 2, window not a multiple of 64
    (S, 128, 8, 2, 200, [1, 63, 199, 200, 201, 1000]),
    (S, 128, 16, 2, 64, [1, 63, 64, 65, 300]),          # one 64-key CTA
    (S, 64, 16, 2, 16, [1, 15, 16, 17, 400]),           # group 8, head_dim 64
    (S, 64, 4, 1, 1, [1, 2, 50]),                       # window of one key
    (F, 256, 8, 2, 0, [1, 64, 65, 300, 500]),           # full layer, lengths <= 512
    (F, 128, 8, 2, 0, [5, 128, 511]),
]


@pytest.mark.parametrize("lt,hd,H,Hkv,window,lens", CASES)
@pytest.mark.parametrize("fused", [False, True])
def test_windowed_decode_against_oracle(lt, hd, H, Hkv, window, lens, fused):
    geo = geometry(lt, hd, H=H, Hkv=Hkv, window=window)
    Lmax = max(lens) + 8
    msl = max(lens)
    p = params_of(geo)
    span = min(msl, window) if lt == S else msl
    assert span <= 512 and G.g4_attn_decode_workspace_size(p, len(lens), msl) == 0
    gpu, ref, wsb, (ck, cv, ok, ov) = run_decode(geo, lens, Lmax, seed=900 + hd + H + int(fused), fused=fused,
                                                 return_cache=True)
    assert wsb == 0
    assert_attn_close(gpu, ref, W.BF16, f"windowed decode {'step' if fused else ''}")
    if fused:
        for b, L in enumerate(lens):
            assert_stored_close(f64(ck[b, :, L - 1]), ok[b, :, L - 1], W.BF16, "new k row")
            assert_stored_close(f64(cv[b, :, L - 1]), ov[b, :, L - 1], W.BF16, "new v row")
            assert torch.isnan(ck[b, :, L:]).all() and torch.isnan(cv[b, :, L:]).all()


def test_windowed_decode_one_full_wave_and_repeat_is_deterministic():
    # 19 sequences x 2 kv heads x 8 CTAs = 304 CTAs, the most the cluster
    # kernel takes (two per SM): every output row against the oracle, and two
    # calls give the same bits
    geo = geometry(S, 256, H=8, Hkv=2, window=512)
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(1, 6000, size=17)] + [4097, 4224]
    assert G.g4_attn_decode_workspace_size(params_of(geo), len(lens), max(lens)) == 0
    gpu, ref, _ = run_decode(geo, lens, max(lens) + 4, seed=77, fused=True)
    assert_attn_close(gpu, ref, W.BF16, "windowed decode, 19 sequences")
    gpu2, _, _ = run_decode(geo, lens, max(lens) + 4, seed=77, fused=True)
    assert np.array_equal(gpu, gpu2)

"""Split-KV decode at the benchmark's unit counts: 8 sequences x 2 kv heads =
16 (sequence, kv head) units, which the decode plan splits 9 ways (one
8-warp CTA per SM, 144 CTAs), and 24 units split 6 ways.  Ragged lengths
leave many splits with no key at all, so the merge must weigh empty
partials at zero.  Groups 1, 2 and 4, head_dim 256 and 512; outputs against
the float64 oracle, the fused step's appended rows bit for bit, and two runs
against each other.
"""

import numpy as np
import pytest
import torch

from gemma_dual_geometry_gb300 import workloads as W

from gpu_common import assert_attn_close, assert_stored_close, f64, geometry, run_decode

pytestmark = pytest.mark.gpu

F = W.FULL
RAGGED = [4097, 100, 2000, 3500, 1, 64, 577, 4096]

CASES = [
    # head_dim, H, Hkv, lengths (B = len(lengths), units = B * Hkv)
    (512, 8, 2, RAGGED),                                 # 16 units x 9 splits, group 4 (the benchmark's full layer)
    (512, 4, 2, [3000] * 8),                             # group 2
    (512, 2, 2, [1, 2, 3000, 1500, 700, 2999, 64, 65]),  # group 1
    (256, 8, 2, [2048, 1, 1000, 2047, 513, 64, 1999, 1500]),
    (512, 8, 2, [1200] * 12),                            # 24 units x 6 splits
]


@pytest.mark.parametrize("hd,H,Hkv,lens", CASES)
def test_split_decode_matches_oracle(hd, H, Hkv, lens):
    geo = geometry(F, hd, H=H, Hkv=Hkv)
    gpu, ref, _ = run_decode(geo, lens, max(lens) + 8, seed=hd + H + len(lens))
    assert_attn_close(gpu, ref, W.BF16, f"split decode hd={hd} H={H} Hkv={Hkv}")


def test_split_decode_step_appends_and_attends():
    geo = geometry(F, 512)
    Lmax = max(RAGGED) + 8
    gpu, ref, _, (ck, cv, ok, ov) = run_decode(geo, RAGGED, Lmax, seed=77, fused=True, return_cache=True)
    assert_attn_close(gpu, ref, W.BF16, "split decode step")
    for b, L in enumerate(RAGGED):
        assert_stored_close(f64(ck[b, :, L - 1]), ok[b, :, L - 1], W.BF16, "new k row")
        assert_stored_close(f64(cv[b, :, L - 1]), ov[b, :, L - 1], W.BF16, "new v row")
        assert torch.isnan(ck[b, :, L:]).all() and torch.isnan(cv[b, :, L:]).all()


def test_split_decode_is_deterministic():
    geo = geometry(F, 512)
    a, _, _ = run_decode(geo, RAGGED, max(RAGGED) + 8, seed=5)
    b, _, _ = run_decode(geo, RAGGED, max(RAGGED) + 8, seed=5)
    assert np.array_equal(a, b)

"""The steps around the path on the tcgen05 tensor cores, against the float64
oracle on the same seeded inputs:

* g4_qkv_project_append: the layer input x times the q / k / v projection
  rows (attention-norm weight folded in), the input RMSNorm's row scale, and
  the per-head norm / RoPE / append (oracle: ``qkv_projection`` then
  ``kv_append_normrope``).  The projections accumulate in float32, so a
  stored bf16 value may differ from the oracle's correctly rounded one by one
  unit in the last place where the float32 sum lands next to a rounding
  boundary: every stored value is within one ulp, at least 99 % are equal
  bit for bit, and cache rows of positions not in the call stay untouched.
* g4_attn_out_residual: h + rmsnorm(ao Wo^T) (oracle ``attn_output_residual``)
  within max-abs 2e-2 and rel-L2 5e-3, the bf16 attention tolerances.
"""

import numpy as np
import pytest
import torch

from gemma_dual_geometry_gb300 import build as g4build
from gemma_dual_geometry_gb300 import g4attn as G
from gemma_dual_geometry_gb300 import workloads as W
from oracle import g4_oracle as O

from gpu_common import DEV, attn_errors, f64, geometry, nan_cache, oracle_lp, params_of

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


def _bf16(a):
    """float64 array -> bf16 torch tensor (the oracle's own rounding, exact values)."""
    return torch.from_numpy(O.round_bf16(a)).to(torch.bfloat16)


def _within_one_ulp(gpu, ref, what):
    """Every value within one bf16 ulp of the oracle's, plus 2^-16 absolute:
    a rotated output y_j cos - y_{j+hd/2} sin that nearly cancels carries the
    float32 error of its two terms (relative to |y_j| + |y_{j+hd/2}|, about 1),
    not of its own small magnitude.  At least 99 % equal bit for bit."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(gpu)), what
    ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(ref), 2.0 ** -126))[1] - 8)
    d = np.abs(gpu - ref)
    bad = d > ulp + 2.0 ** -16
    if bad.any():
        i = np.argsort(-(d - ulp).ravel())[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} values off by more than one ulp + 2^-16, e.g. gpu "
                             f"{gpu.ravel()[i]} ref {ref.ravel()[i]}")
    same = float(np.mean(gpu == ref))
    assert same >= 0.99, f"{what}: only {same:.4f} equal bit for bit"
    return same


PROJ_CASES = [
    # layer type, head_dim, D, B, T, q_start, shared, ring
    (S, 256, 512, 2, 200, [0, 37], False, False),
    (F, 512, 2048, 1, 130, [5], False, False),
    (S, 128, 256, 3, 64, [0, 0, 100], False, False),
    (F, 64, 128, 2, 129, [0, 3], False, False),
    (S, 256, 512, 2, 150, [0, 0], True, False),       # shared layer: q only
    (S, 256, 512, 2, 100, [600, 1000], False, True),  # ring of 512 rows past its wrap
]


@pytest.mark.parametrize("lt,hd,D,B,T,q_start,shared,ring", PROJ_CASES)
def test_qkv_project_append_against_oracle(lt, hd, D, B, T, q_start, shared, ring):
    geo = geometry(lt, hd, H=8, Hkv=2, window=512)
    H, Hkv, dt = 8, 2, W.BF16
    seed = 3000 + hd + D + T
    x = W.normal((B, T, D), seed + 1, dt)
    a = f64(W.norm_weight(D, seed + 2))
    N = (H + (0 if shared else 2 * Hkv)) * hd
    w = f64(W.normal((N, D), seed + 3, W.F32)) / np.sqrt(D)
    w_f = O.round_bf16(w * a[None, :])                     # attention-norm weight folded in, bf16
    qw, kw = W.norm_weight(hd, seed + 4), W.norm_weight(hd, seed + 5)
    pos = np.asarray(q_start)[:, None] + np.arange(T)[None, :]
    Lmax = 512 if ring else int(pos.max()) + 9
    ck = nan_cache(B, Hkv, Lmax, hd, dt)
    cv = nan_cache(B, Hkv, Lmax, hd, dt)
    table = G.cache_table(2)
    G.set_cache(table, 0, ck, cv, lt, hd, Hkv, Lmax, B, dt, ring=ring)
    layer = 1 if shared else 0
    p = params_of(geo, src=0 if shared else -1)
    q_out = torch.empty((B, T, H, hd), dtype=torch.bfloat16, device=DEV)
    G.g4_qkv_project_append(p, table, layer, x.to(DEV), D, _bf16(w_f).to(DEV), qw.to(DEV),
                            None if shared else kw.to(DEV), torch.tensor(pos, dtype=torch.int32, device=DEV), B, T,
                            q_out)
    torch.cuda.synchronize()
    # oracle: the plain definition on the same (folded, bf16) weights
    q, k, v = O.qkv_projection(f64(x), None, w_f[:H * hd], None if shared else w_f[H * hd:(H + Hkv) * hd],
                               None if shared else w_f[(H + Hkv) * hd:], geo["eps"])
    q = q.reshape(B, T, H, hd)
    ok = np.full((B, Hkv, Lmax, hd), np.nan)
    ov = np.full((B, Hkv, Lmax, hd), np.nan)
    lp = oracle_lp(geo, src=0 if shared else -1)
    oq = O.kv_append_normrope(lp, q, None if shared else k.reshape(B, T, Hkv, hd),
                              None if shared else v.reshape(B, T, Hkv, hd), f64(qw), None if shared else f64(kw),
                              pos, ok, ov, ring=ring)
    _within_one_ulp(f64(q_out), oq, "q_out")
    gk, gv = f64(ck), f64(cv)
    if shared:
        assert np.isnan(gk).all() and np.isnan(gv).all()   # a shared layer writes no cache row
    else:
        written = ~np.isnan(ok[:, 0, :, 0])                  # rows the oracle's append wrote
        for b in range(B):
            rows = np.nonzero(written[b])[0]
            _within_one_ulp(gk[b][:, rows], ok[b][:, rows], "k rows")
            _within_one_ulp(gv[b][:, rows], ov[b][:, rows], "v rows")
            others = np.nonzero(~written[b])[0]
            assert np.isnan(gk[b][:, others]).all() and np.isnan(gv[b][:, others]).all()


OUT_CASES = [
    # M, K, D
    (300, 512, 256),
    (257, 2048, 2048),
    (128, 4096, 512),
    (1, 64, 2048),
]


@pytest.mark.parametrize("M,K,D", OUT_CASES)
@pytest.mark.parametrize("in_place", [False, True])
def test_attn_out_residual_against_oracle(M, K, D, in_place):
    seed = 4000 + M + K + D
    ao = W.normal((M, K), seed + 1, W.BF16)
    wo = W.normal((D, K), seed + 2, W.F32) / np.sqrt(K)
    wo_b = wo.to(torch.bfloat16)
    post = W.norm_weight(D, seed + 3)
    h = W.normal((M, D), seed + 4, W.BF16)
    hd_ = h.to(DEV)
    out = hd_ if in_place else torch.empty_like(hd_)
    G.g4_attn_out_residual(ao.to(DEV), M, K, wo_b.to(DEV), D, post.to(DEV), W.EPS, hd_, out)
    torch.cuda.synchronize()
    ref = O.attn_output_residual(f64(h), f64(ao), f64(wo_b), f64(post), W.EPS)
    max_abs, rel = attn_errors(f64(out), ref)
    assert np.all(np.isfinite(f64(out)))
    assert max_abs <= 2e-2 and rel <= 5e-3, f"max_abs {max_abs:.3e} rel_l2 {rel:.3e}"

"""Parity of the CUDA path (through the C ABI) against the float64 oracle.

Tolerances (fixed by the specification of the path):
  * append: bf16 stores equal, bit for bit, to the oracle's correctly rounded
    values; f32 within 1e-4;
    cache rows not addressed by a position stay bit-for-bit untouched (caches
    start NaN-filled, which also makes any read past the filled length poison
    the attention output).
  * attention, against the oracle's exact float64 output: f32 max-abs 1e-4;
    bf16 max-abs 2e-2 and rel-L2 5e-3.
"""

import numpy as np
import pytest
import torch

from gemma_dual_geometry_gb300 import build as g4build
from gemma_dual_geometry_gb300 import g4attn as G
from gemma_dual_geometry_gb300 import workloads as W
from oracle import g4_oracle as O

from gpu_common import (DEV, LayerRun, assert_attn_close, assert_stored_close, f64, geometry, nan_cache,
                        oracle_lp, params_of, run_decode)

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


# ---------------------------------------------------------------- a1-a4 append

APPEND_CASES = [(S, 64, 1e4, 1.0), (F, 128, 1e6, 0.25), (S, 256, 1e4, 1.0), (F, 512, 1e6, 0.25)]


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("lt,hd,theta,frac", APPEND_CASES)
def test_append_parity_and_exact_rows(dtype, lt, hd, theta, frac):
    geo = geometry(lt, hd, theta=theta, frac=frac, dtype=dtype)
    r = LayerRun(geo, B=3, T=37, Lmax=300, q_start=[0, 100, 263], seed=100 + hd, prior=False).run_gpu()
    r.run_oracle()
    assert_stored_close(f64(r.q_out), r.o_q, dtype, "q_out")
    ck, cv = f64(r.ck), f64(r.cv)
    written = np.zeros((3, 300), bool)
    for b in range(3):
        written[b, r.positions()[b]] = True
    mask = np.broadcast_to(written[:, None, :, None], ck.shape)
    assert_stored_close(ck[mask], r.o_ck[mask], dtype, "cache k")
    assert_stored_close(cv[mask], r.o_cv[mask], dtype, "cache v")
    # every other row is still the NaN sentinel, bit for bit
    ity = torch.int16 if dtype == W.BF16 else torch.int32
    sentinel = torch.full((1,), float("nan"), dtype=W.torch_dtype(dtype)).view(ity).item()
    for c in (r.ck, r.cv):
        raw = c.view(ity).cpu().numpy()
        assert np.all(raw[~mask] == sentinel)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("lt,hd", [(S, 256), (F, 512)])
def test_append_rope_at_long_positions(dtype, lt, hd):
    # positions up to 131071: p * inv_freq is formed exactly and reduced by a three-part pi/2
    geo = geometry(lt, hd, dtype=dtype)
    B, T, Lmax = 1, 24, 131072
    r = LayerRun(geo, B=B, T=T, Lmax=Lmax, q_start=[Lmax - T], seed=7, prior=False).run_gpu()
    r.run_oracle()
    assert_stored_close(f64(r.q_out), r.o_q, dtype, "q_out")
    p0 = int(r.positions()[0, 0])
    assert_stored_close(f64(r.ck[0, :, p0:p0 + T]), r.o_ck[0, :, p0:p0 + T], dtype, "k rows")
    assert_stored_close(f64(r.cv[0, :, p0:p0 + T]), r.o_cv[0, :, p0:p0 + T], dtype, "v rows")


@pytest.mark.parametrize("lt,hd", [(S, 256), (F, 512)])
def test_append_bf16_bit_exact_on_many_rows(lt, hd):
    # ~6M stored values: several thousand of them land close enough to a bf16
    # rounding boundary that the float32 evaluation cannot decide them
    geo = geometry(lt, hd, H=8, Hkv=2)
    r = LayerRun(geo, B=2, T=512, Lmax=1100, q_start=[0, 517], seed=900 + hd, prior=False).run_gpu()
    r.run_oracle()
    assert_stored_close(f64(r.q_out), r.o_q, W.BF16, "q_out")
    for b in range(2):
        p0 = int(r.q_start[b])
        assert_stored_close(f64(r.ck[b, :, p0:p0 + 512]), r.o_ck[b, :, p0:p0 + 512], W.BF16, "k rows")
        assert_stored_close(f64(r.cv[b, :, p0:p0 + 512]), r.o_cv[b, :, p0:p0 + 512], W.BF16, "v rows")


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("lt,hd", [(S, 256), (F, 512)])
def test_append_q_rope_at_positions_beyond_float_integers(dtype, lt, hd):
    # q is normed and roped at any position (only k / v need a cache slot);
    # positions from 2^24 on take the float64 reduction
    geo = geometry(lt, hd, dtype=dtype)
    pos_list = [2 ** 24 - 1, 2 ** 24, 2 ** 24 + 1, 2 ** 24 + 12345, 2 ** 29 + 3, 2 ** 30 + 7, 2 ** 31 - 1, 99999999]
    B, T, H = 1, len(pos_list), geo["n_heads"]
    q = W.normal((B, T, H, hd), 31, dtype)
    qw = W.norm_weight(hd, 32)
    p = params_of(geo, src=0)   # shared layer: q only
    tab = G.cache_table(2)
    out = torch.empty_like(q, device=DEV)
    pos = torch.tensor([pos_list], dtype=torch.int32, device=DEV)
    G.g4_kv_append_normrope(p, tab, 1, q.to(DEV), None, None, qw.to(DEV), None, pos, B, T, out)
    torch.cuda.synchronize()
    ref = O.store(O.normrope_q(f64(q), f64(qw), np.array([pos_list]), hd, geo["theta"], geo["rotary_fraction"],
                               geo["eps"]), dtype)
    assert_stored_close(f64(out), ref, dtype, "q_out")


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_append_zero_tail_is_bitwise_unrotated(dtype):
    # full layer, 64 of 256 pairs rotate: the other dims must equal the
    # position-0 output (RoPE at position 0 is the identity) bit for bit
    geo = geometry(F, 512, dtype=dtype)
    B, T = 1, 16
    x = W.normal((B, 1, 8, 512), 5, dtype).repeat(1, T, 1, 1).contiguous().to(DEV)
    w = W.norm_weight(512, 6).to(DEV)
    p = params_of(geo, src=0)   # shared layer: q only
    tab = G.cache_table(2)
    out = torch.empty_like(x)
    pos = torch.tensor([[0, 1, 2, 3, 100, 1000, 4095, 4096, 10000, 65535, 65536, 100000, 131071, 7, 9, 11]],
                       dtype=torch.int32, device=DEV)
    G.g4_kv_append_normrope(p, tab, 1, x, None, None, w, None, pos, B, T, out)
    torch.cuda.synchronize()
    o = out.view(torch.int16 if dtype == W.BF16 else torch.int32).cpu().numpy()[0]
    tail = np.r_[64:256, 320:512]
    assert np.all(o[:, :, tail] == o[0:1, :, tail])
    assert not np.all(o[:, :, :64] == o[0:1, :, :64])


# ---------------------------------------------------------------- a5 prefill

PREFILL_CASES = [
    # dtype, type, hd, window, B, T, q_start
    (W.BF16, S, 256, 512, 1, 700, [0]),
    (W.BF16, F, 512, 0, 1, 300, [0]),
    (W.BF16, S, 64, 40, 2, 200, [0, 37]),
    (W.BF16, F, 128, 0, 2, 150, [5, 0]),
    (W.BF16, S, 256, 100, 2, 333, [0, 129]),
    (W.BF16, F, 512, 0, 2, 129, [200, 0]),
    (W.BF16, S, 512, 1, 1, 130, [0]),
    (W.F32, S, 64, 16, 1, 64, [0]),
    (W.F32, F, 128, 0, 2, 90, [0, 11]),
    (W.F32, F, 512, 0, 1, 50, [3]),
    (W.F32, S, 256, 7, 1, 40, [0]),
    # more work items (query tile x head x output half) than a GB300 has SMs,
    # ragged lengths and query offsets in one launch
    (W.BF16, S, 256, 512, 4, 1000, [0, 37, 500, 1024]),
    (W.BF16, F, 512, 0, 3, 700, [0, 300, 1111]),
]


@pytest.mark.parametrize("dtype,lt,hd,window,B,T,q_start", PREFILL_CASES)
def test_prefill_parity(dtype, lt, hd, window, B, T, q_start):
    geo = geometry(lt, hd, window=window, dtype=dtype)
    Lmax = max(q_start) + T + 64
    r = LayerRun(geo, B, T, Lmax, q_start, seed=1000 + hd + T).run_gpu()
    r.run_oracle()
    assert_attn_close(f64(r.out), r.o_out, dtype, "prefill")


def test_prefill_gqa_group_8():
    geo = geometry(S, 128, H=16, Hkv=2, window=60)
    r = LayerRun(geo, 1, 260, 300, [0], seed=31).run_gpu()
    r.run_oracle()
    assert_attn_close(f64(r.out), r.o_out, W.BF16, "prefill g8")


def test_prefill_window_covering_everything_equals_full():
    # a sliding layer whose window covers all keys reproduces the full layer bit for bit
    geo_s = geometry(S, 256, window=100000)
    geo_f = geometry(F, 256, theta=1e4, frac=1.0)
    a = LayerRun(geo_s, 1, 400, 400, [0], seed=5).run_gpu()
    b = LayerRun(geo_f, 1, 400, 400, [0], seed=5).run_gpu()
    assert torch.equal(a.q_out, b.q_out)
    assert torch.equal(a.out, b.out)


def test_shared_layer_reads_source_cache_bitwise():
    # layer 1 shares layer 0's cache: its output equals prefill run directly
    # on layer 0's cache with the same q, and its append writes nothing
    geo = geometry(S, 256, window=300)
    table = G.cache_table(2)
    r = LayerRun(geo, 2, 300, 400, [0, 50], seed=9).run_gpu(table=table, layer=0)
    ck_before = r.ck.clone()
    q1 = W.normal((2, 300, 8, 256), 77, W.BF16).to(DEV)
    w1 = W.norm_weight(256, 78).to(DEV)
    p1 = params_of(geo, src=0)
    q1_out = torch.empty_like(q1)
    pos = torch.tensor(r.positions(), dtype=torch.int32, device=DEV)
    G.g4_kv_append_normrope(p1, table, 1, q1, None, None, w1, None, pos, 2, 300, q1_out)
    qs = torch.tensor(r.q_start, dtype=torch.int32, device=DEV)
    o_shared = torch.empty_like(q1)
    G.g4_attn_prefill(p1, table, 1, q1_out, qs, 2, 300, o_shared)
    o_direct = torch.empty_like(q1)
    G.g4_attn_prefill(params_of(geo), table, 0, q1_out, qs, 2, 300, o_direct)
    torch.cuda.synchronize()
    assert torch.equal(o_shared, o_direct)
    assert torch.equal(ck_before.view(torch.int16), r.ck.view(torch.int16))


def test_tiny_fp32_stack_against_oracle():
    cfg = W.CONFIGS["tiny_fp32_stack"]
    B, T, n = cfg["B"], cfg["T"], len(cfg["types"])
    is_s = [t == S for t in cfg["types"]]
    srcs = [G.g4_kv_share_src(n, cfg["n_shared"], is_s, l) for l in range(n)]
    assert srcs == [-1, -1, 0, 1]
    table = G.cache_table(n)
    layers, inputs, outs, keep = [], [], [], []
    pos = torch.arange(T, dtype=torch.int32, device=DEV).repeat(B, 1)
    qs = torch.zeros(B, dtype=torch.int32, device=DEV)
    for l in range(n):
        geo = W.layer_geometry(cfg, l)
        x = W.layer_inputs(cfg, l, T, srcs[l] < 0)
        layers.append(oracle_lp(geo, srcs[l]))
        inputs.append({k: f64(v) for k, v in x.items()})
        hd = geo["head_dim"]
        if srcs[l] < 0:
            ck = nan_cache(B, cfg["Hkv"], T, hd, W.F32)
            cv = nan_cache(B, cfg["Hkv"], T, hd, W.F32)
            keep += [ck, cv]
            G.set_cache(table, l, ck, cv, geo["layer_type"], hd, cfg["Hkv"], T, B, W.F32)
        dev = {k: v.to(DEV) for k, v in x.items()}
        q_out = torch.empty_like(dev["q"])
        G.g4_kv_append_normrope(params_of(geo, srcs[l]), table, l, dev["q"], dev.get("k"), dev.get("v"),
                                dev["q_norm_w"], dev.get("k_norm_w"), pos, B, T, q_out)
        o = torch.empty_like(dev["q"])
        G.g4_attn_prefill(params_of(geo, srcs[l]), table, l, q_out, qs, B, T, o)
        outs.append(o)
    torch.cuda.synchronize()
    ref, _ = O.run_stack_prefill(layers, inputs, B, T, T)
    for l in range(n):
        assert_attn_close(f64(outs[l]), ref[l], W.F32, f"layer {l}")


# ---------------------------------------------------------------- a6 decode

DECODE_CASES = [
    (W.BF16, F, 512, 0, 2, [1, 2, 127, 128, 129, 1000, 2047, 3000]),
    (W.BF16, S, 256, 512, 2, [1, 5, 511, 512, 513, 1300, 2999, 3000]),
    (W.BF16, S, 128, 200, 2, [1, 199, 200, 201, 1000]),
    (W.BF16, F, 64, 0, 2, [3, 64, 900]),
    (W.F32, F, 128, 0, 2, [1, 77, 700, 1500]),
    (W.F32, S, 64, 16, 2, [1, 15, 16, 17, 400]),
    (W.F32, F, 512, 0, 2, [2, 600]),
]


@pytest.mark.parametrize("dtype,lt,hd,window,Hkv,lens", DECODE_CASES)
def test_decode_parity(dtype, lt, hd, window, Hkv, lens):
    geo = geometry(lt, hd, H=4 * Hkv, Hkv=Hkv, window=window, dtype=dtype)
    gpu, ref, _ = run_decode(geo, lens, max(lens) + 8, seed=500 + hd)
    assert_attn_close(gpu, ref, dtype, "decode")


def test_decode_gqa_group_8_and_1():
    for H, Hkv, hd in ((16, 2, 64), (2, 2, 512), (4, 2, 256)):
        geo = geometry(F, hd, H=H, Hkv=Hkv)
        gpu, ref, _ = run_decode(geo, [1, 333, 1025], 1100, seed=H + hd)
        assert_attn_close(gpu, ref, W.BF16, f"decode H={H} Hkv={Hkv}")


def test_decode_split_and_single_split_agree_with_oracle():
    # the same lengths through one split (small bound) and many splits (large bound)
    geo = geometry(F, 256, theta=1e6)
    g1, ref, w1 = run_decode(geo, [40, 64], 100, seed=3, max_seq_len=64)     # one 64-key split
    g2, ref2, w2 = run_decode(geo, [40, 64], 6000, seed=3, max_seq_len=6000)
    assert w1 == 0 and w2 > 0
    assert_attn_close(g1, ref, W.BF16, "one split")
    assert_attn_close(g2, ref2, W.BF16, "many splits")


# ---------------------------------------------------------------- a4 + a6 fused decode step

@pytest.mark.parametrize("dtype,lt,hd,window,Hkv,lens", DECODE_CASES)
def test_decode_step_parity_and_appended_rows(dtype, lt, hd, window, Hkv, lens):
    geo = geometry(lt, hd, H=4 * Hkv, Hkv=Hkv, window=window, dtype=dtype)
    Lmax = max(lens) + 8
    gpu, ref, _, (ck, cv, ok, ov) = run_decode(geo, lens, Lmax, seed=700 + hd, fused=True, return_cache=True)
    assert_attn_close(gpu, ref, dtype, "decode step")
    # the new rows were written at L-1 (the oracle's append, bit for bit); rows >= L are untouched NaN
    for b, L in enumerate(lens):
        assert_stored_close(f64(ck[b, :, L - 1]), ok[b, :, L - 1], dtype, "new k row")
        assert_stored_close(f64(cv[b, :, L - 1]), ov[b, :, L - 1], dtype, "new v row")
        assert torch.isnan(ck[b, :, L:]).all() and torch.isnan(cv[b, :, L:]).all()


def test_decode_step_shared_layer_and_gqa_groups():
    # group 8 and group 1; and a shared layer reading the source cache
    for H, Hkv, hd in ((16, 2, 64), (2, 2, 512)):
        geo = geometry(F, hd, H=H, Hkv=Hkv)
        gpu, ref, _ = run_decode(geo, [1, 333, 1025], 1100, seed=H + hd + 1, fused=True)
        assert_attn_close(gpu, ref, W.BF16, f"decode step H={H} Hkv={Hkv}")
    geo = geometry(S, 256, window=300)
    B, Hkv, H, hd, Lmax = 3, 2, 8, 256, 700
    lens = np.array([1, 299, 650])
    ck = W.normal((B, Hkv, Lmax, hd), 81, W.BF16).to(DEV)
    cv = W.normal((B, Hkv, Lmax, hd), 82, W.BF16).to(DEV)
    table = G.cache_table(2)
    G.set_cache(table, 0, ck, cv, S, hd, Hkv, Lmax, B, W.BF16)
    q = W.normal((B, H, hd), 83, W.BF16).to(DEV)
    qw = W.norm_weight(hd, 84).to(DEV)
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    p1 = params_of(geo, src=0)
    wsb = G.g4_attn_decode_workspace_size(p1, B, Lmax)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=DEV)
    before = ck.clone()
    o_step = torch.empty_like(q)
    G.g4_decode_step(p1, table, 1, q, None, None, qw, None, sl, B, Lmax, o_step, ws, wsb)
    q_out = torch.empty_like(q)
    G.g4_kv_append_normrope(p1, table, 1, q.view(B, 1, H, hd), None, None, qw, None, (sl - 1).view(B, 1), B, 1,
                            q_out.view(B, 1, H, hd))
    o_ref = torch.empty_like(q)
    G.g4_attn_decode(p1, table, 1, q_out, sl, B, Lmax, o_ref, ws, wsb)
    torch.cuda.synchronize()
    assert torch.equal(before.view(torch.int16), ck.view(torch.int16))    # a shared layer writes nothing
    assert_attn_close(f64(o_step), f64(o_ref), W.BF16, "shared-layer decode step vs append + decode")

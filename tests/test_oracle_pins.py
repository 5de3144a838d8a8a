"""Pins of the float64 oracle against facts that do not come from the oracle.

Each test uses something other than the oracle's own formula: a closed form,
an invariant, a library routine computing the same textbook operation, brute
force over explicit loops, or the worked example the pages print
(ferrox-models ``gemma4_engine.rs`` test ``layer_routing_swa_and_shared_kv``).
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import g4_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rng(seed=0):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- bf16 rounding

def test_round_bf16_matches_torch_on_float32_values():
    # torch's float32 -> bfloat16 conversion is round-to-nearest-even; on
    # values exactly representable in float32 it is the correctly rounded one.
    x = rng(1).standard_normal(200000).astype(np.float32) * np.float32(3.0)
    x = np.concatenate([x, np.float32([1e-30, -7e-39, 3e38, 65504.0, 0.0, -0.0])])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_bf16(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_round_bf16_ties_to_even():
    ulp = 2.0 ** -7  # bf16 spacing on [1, 2)
    assert O.round_bf16(1.0 + ulp / 2) == 1.0               # tie -> even (1.0)
    assert O.round_bf16(1.0 + 3 * ulp / 2) == 1.0 + 2 * ulp  # tie -> even
    assert O.round_bf16(1.0 + ulp / 2 + 2.0 ** -40) == 1.0 + ulp  # just above tie
    assert O.round_bf16(-(1.0 + ulp / 2)) == -1.0


# ---------------------------------------------------------------- RMSNorm (a1, a2)

def test_rms_norm_constant_vector_closed_form():
    # x = c * 1: mean(x^2) = c^2, so y = w * c / sqrt(c^2 + eps)
    for c in (0.5, -3.0, 1e-4):
        for eps in (1e-6, 1e-2):
            w = np.linspace(0.5, 1.5, 64)
            y = O.rms_norm(np.full(64, c), w, eps)
            assert np.allclose(y, w * c / math.sqrt(c * c + eps), rtol=1e-14, atol=0)


def test_rms_norm_weight_is_plain_not_one_plus_w():
    x = rng(2).standard_normal(128)
    xhat = O.rms_norm(x, None, 1e-6)
    assert np.allclose(O.rms_norm(x, np.zeros(128), 1e-6), 0.0)   # 1+w would give xhat
    assert np.allclose(O.rms_norm(x, np.full(128, 2.0), 1e-6), 2 * xhat, rtol=1e-15)


def test_rms_norm_unit_weight_mean_square():
    # with w = 1 the output mean square is ms / (ms + eps): pins eps inside the mean
    x = rng(3).standard_normal((50, 256)) * 1e-3
    eps = 1e-6
    ms = np.mean(x * x, axis=-1)
    y = O.rms_norm(x, np.ones(256), eps)
    assert np.allclose(np.mean(y * y, axis=-1), ms / (ms + eps), rtol=1e-12)


def test_rms_norm_matches_torch_library():
    x = rng(4).standard_normal((7, 3, 512))
    w = 1 + 0.1 * rng(5).standard_normal(512)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (512,), torch.from_numpy(w), eps=1e-6).numpy()
    assert np.allclose(O.rms_norm(x, w, 1e-6), ref, rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- RoPE (a3)

def test_inv_freq_closed_forms():
    inv = O.rope_inv_freq(64, 1e4, 1.0)
    assert inv.dtype == np.float32 and inv.shape == (32,)
    assert inv[0] == 1.0
    assert inv[16] == np.float32(0.01)                  # 1e4 ** (-32/64) = 1e-2
    assert np.all(inv > 0) and np.all(np.diff(inv) < 0)
    # constant ratio theta^(-2/hd) between neighbours
    r = inv[1:].astype(np.float64) / inv[:-1]
    assert np.allclose(r, 1e4 ** (-2 / 64), rtol=2e-7)


def test_inv_freq_proportional_partial_rotary():
    # full layer: global head dim 512, fraction 0.25 -> 64 rotated pairs of 256,
    # frequencies over the FULL width (denominator 512), zero tail
    inv = O.rope_inv_freq(512, 1e6, 0.25)
    assert inv.shape == (256,)
    assert np.count_nonzero(inv) == 64
    assert np.all(inv[64:] == 0)
    assert inv[32] == np.float32(1e6 ** (-64 / 512))
    # tiny config's full layer: hd 128, fraction .25 -> 16 pairs
    assert np.count_nonzero(O.rope_inv_freq(128, 1e6, 0.25)) == 16
    # floor, not round: 100 * 0.25 / 2 = 12.5 -> 12
    assert O.rotated_pairs(100, 0.25) == 12


def test_rope_matches_complex_rotation():
    # rotate_half on (j, j + hd/2) is multiplication of z_j = x_j + i x_{j+h}
    # by exp(i * pos * w_j)
    hd = 128
    x = rng(6).standard_normal((5, hd))
    pos = np.array([0, 1, 17, 4095, 131071])
    inv = O.rope_inv_freq(hd, 1e4, 1.0)
    y = O.rope_rotate_half(x, pos, inv)
    z = x[:, :hd // 2] + 1j * x[:, hd // 2:]
    zr = z * np.exp(1j * pos[:, None] * inv.astype(np.float64)[None, :])
    assert np.allclose(y[:, :hd // 2], zr.real, rtol=0, atol=1e-12)
    assert np.allclose(y[:, hd // 2:], zr.imag, rtol=0, atol=1e-12)


def test_rope_basis_vector_and_sign():
    hd, j, pos = 64, 3, 5
    inv = O.rope_inv_freq(hd, 1e4, 1.0)
    x = np.zeros(hd)
    x[j] = 1.0
    y = O.rope_rotate_half(x, pos, inv)
    a = pos * float(inv[j])
    assert y[j] == pytest.approx(math.cos(a), abs=1e-15)
    assert y[j + hd // 2] == pytest.approx(math.sin(a), abs=1e-15)   # + sin on the upper half
    x = np.zeros(hd)
    x[j + hd // 2] = 1.0
    y = O.rope_rotate_half(x, pos, inv)
    assert y[j] == pytest.approx(-math.sin(a), abs=1e-15)
    assert y[j + hd // 2] == pytest.approx(math.cos(a), abs=1e-15)


def test_rope_identity_at_pos0_and_zero_tail():
    x = rng(7).standard_normal((3, 512))
    inv = O.rope_inv_freq(512, 1e6, 0.25)
    assert np.array_equal(O.rope_rotate_half(x, 0, inv), x)
    y = O.rope_rotate_half(x, 98765, inv)
    tail = np.r_[64:256, 256 + 64:512]
    assert np.array_equal(y[:, tail], x[:, tail])          # bitwise unrotated
    assert not np.allclose(y[:, :64], x[:, :64])


def test_rope_norm_preserving_and_relative():
    hd = 256
    inv = O.rope_inv_freq(hd, 1e4, 1.0)
    q, k = rng(8).standard_normal((2, hd))
    y = O.rope_rotate_half(q, 1234, inv)
    pn = lambda v: v[:hd // 2] ** 2 + v[hd // 2:] ** 2
    assert np.allclose(pn(y), pn(q), rtol=1e-12)
    # <rope(q, p+s), rope(k, p'+s)> depends only on p - p'
    d0 = O.rope_rotate_half(q, 40, inv) @ O.rope_rotate_half(k, 7, inv)
    d1 = O.rope_rotate_half(q, 40 + 900, inv) @ O.rope_rotate_half(k, 7 + 900, inv)
    assert d0 == pytest.approx(d1, rel=1e-9, abs=1e-9)


# ---------------------------------------------------------------- attention (a5, a6)

def _cache_from(k, v, Lmax=None):
    # k, v [B, L, Hkv, hd] -> cache layout [B, Hkv, Lmax, hd]
    B, L, Hkv, hd = k.shape
    Lmax = Lmax or L
    ck = np.zeros((B, Hkv, Lmax, hd))
    cv = np.zeros((B, Hkv, Lmax, hd))
    ck[:, :, :L] = np.transpose(k, (0, 2, 1, 3))
    cv[:, :, :L] = np.transpose(v, (0, 2, 1, 3))
    return ck, cv


@pytest.mark.parametrize("layer_type,window", [(O.FULL, 0), (O.SLIDING, 5), (O.SLIDING, 1)])
def test_attention_matches_torch_sdpa(layer_type, window):
    # library routine: torch SDPA in float64 with an explicit boolean mask,
    # scale 1.0 and kv heads repeated to query heads (h -> h // g)
    B, T, H, Hkv, hd = 2, 13, 4, 2, 32
    r = rng(9)
    q = r.standard_normal((B, T, H, hd))
    k = r.standard_normal((B, T, Hkv, hd))
    v = r.standard_normal((B, T, Hkv, hd))
    ck, cv = _cache_from(k, v, Lmax=T + 3)
    ck[:, :, T:] = np.nan     # rows past kv_len are never read
    pos = np.broadcast_to(np.arange(T), (B, T))
    got = O.attention(q, ck, cv, pos, np.full(B, T), Hkv, layer_type, window, 1.0)
    i = torch.arange(T)[:, None]
    j = torch.arange(T)[None, :]
    mask = j <= i
    if layer_type == O.SLIDING:
        mask = mask & (i - j < window)
    qt = torch.from_numpy(q).permute(0, 2, 1, 3)
    kt = torch.from_numpy(k).permute(0, 2, 1, 3).repeat_interleave(H // Hkv, dim=1)
    vt = torch.from_numpy(v).permute(0, 2, 1, 3).repeat_interleave(H // Hkv, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=1.0)
    assert np.allclose(got, ref.permute(0, 2, 1, 3).numpy(), rtol=1e-12, atol=1e-12)


def test_attention_brute_force_loops():
    # explicit loops with math.exp, tiny sizes
    B, T, H, Hkv, hd, W = 1, 7, 2, 1, 4, 3
    r = rng(10)
    q = r.standard_normal((B, T, H, hd))
    k = r.standard_normal((B, T, Hkv, hd))
    v = r.standard_normal((B, T, Hkv, hd))
    ck, cv = _cache_from(k, v)
    pos = np.arange(T)[None, :]
    for lt in (O.FULL, O.SLIDING):
        got = O.attention(q, ck, cv, pos, [T], Hkv, lt, W, 1.0)
        for t in range(T):
            for h in range(H):
                js = [j for j in range(T) if j <= t and (lt == O.FULL or t - j < W)]
                sc = [sum(q[0, t, h, d] * k[0, j, 0, d] for d in range(hd)) for j in js]
                mx = max(sc)
                ws = [math.exp(s - mx) for s in sc]
                z = sum(ws)
                exp = [sum(w * v[0, j, 0, d] for w, j in zip(ws, js)) / z for d in range(hd)]
                assert np.allclose(got[0, t, h], exp, rtol=1e-12, atol=1e-13)


def test_window_covering_everything_is_full_attention():
    B, T, H, Hkv, hd = 1, 20, 2, 2, 16
    r = rng(11)
    q = r.standard_normal((B, T, H, hd))
    ck, cv = _cache_from(r.standard_normal((B, T, Hkv, hd)), r.standard_normal((B, T, Hkv, hd)))
    pos = np.arange(T)[None, :]
    full = O.attention(q, ck, cv, pos, [T], Hkv, O.FULL, 0)
    for W in (T, T + 1, 10 * T):
        assert np.array_equal(O.attention(q, ck, cv, pos, [T], Hkv, O.SLIDING, W), full)
    assert not np.allclose(O.attention(q, ck, cv, pos, [T], Hkv, O.SLIDING, T - 1), full)


def test_probs_sum_to_one_and_single_visible_key():
    r = rng(12)
    keys = r.standard_normal((30, 8)) * 5
    for qp in (0, 5, 29):
        for lt, W in ((O.FULL, 0), (O.SLIDING, 4), (O.SLIDING, 1)):
            p = O.attention_probs(r.standard_normal(8), keys, np.arange(30), qp, lt, W, 1.0)
            assert p.sum() == pytest.approx(1.0, abs=1e-14)
            assert np.all(p[qp + 1:] == 0)
    # T = 1 or W = 1: output is exactly the current token's v
    B, T, H, Hkv, hd = 1, 9, 2, 1, 8
    q = r.standard_normal((B, T, H, hd))
    k = r.standard_normal((B, T, Hkv, hd))
    v = r.standard_normal((B, T, Hkv, hd))
    ck, cv = _cache_from(k, v)
    o = O.attention(q, ck, cv, np.arange(T)[None, :], [T], Hkv, O.SLIDING, 1)
    for h in range(H):
        assert np.array_equal(o[0, :, h], v[0, :, 0])


def test_equal_keys_give_mean_of_visible_values():
    # identical keys -> uniform weights -> mean of exactly the visible v rows,
    # which pins the window edge (q - k < W, current token included)
    T, hd, W = 12, 4, 5
    k = np.ones((1, T, 1, hd))
    v = np.arange(T, dtype=np.float64)[None, :, None, None] * np.ones((1, T, 1, hd))
    ck, cv = _cache_from(k, v)
    q = np.ones((1, T, 1, hd))
    o = O.attention(q, ck, cv, np.arange(T)[None, :], [T], 1, O.SLIDING, W)
    for t in range(T):
        lo = max(0, t - W + 1)
        assert o[0, t, 0, 0] == pytest.approx(np.mean(np.arange(lo, t + 1)), abs=1e-13)
    o = O.attention(q, ck, cv, np.arange(T)[None, :], [T], 1, O.FULL, 0)
    assert np.allclose(o[0, :, 0, 0], [t / 2 for t in range(T)], atol=1e-13)


def test_score_scale_is_one_closed_form():
    # two visible keys with scores 0 and a: weight of the second = sigmoid(a)
    hd = 16
    q = np.zeros(hd)
    q[0] = 1.5
    keys = np.zeros((2, hd))
    keys[1, 0] = 2.0          # score 3.0 at scale 1.0 (a 1/sqrt(hd) scale would give 0.75)
    p = O.attention_probs(q, keys, np.arange(2), 1, O.FULL, 0, 1.0)
    assert p[1] == pytest.approx(1 / (1 + math.exp(-3.0)), rel=1e-14)


def test_gqa_head_mapping_contiguous_groups():
    # v constant per kv head = its index; output of q head h = h // (H/Hkv)
    B, T, H, Hkv, hd = 1, 6, 8, 2, 8
    r = rng(13)
    q = r.standard_normal((B, T, H, hd))
    k = r.standard_normal((B, T, Hkv, hd))
    v = np.zeros((B, T, Hkv, hd))
    v[:, :, 1, :] = 1.0
    ck, cv = _cache_from(k, v)
    o = O.attention(q, ck, cv, np.arange(T)[None, :], [T], Hkv, O.FULL, 0)
    for h in range(H):
        assert np.allclose(o[0, :, h], h // 4, atol=1e-14)


def test_one_hot_dominant_key():
    hd = 32
    r = rng(14)
    keys = r.standard_normal((10, hd))
    q = keys[6] * 10.0
    vals = r.standard_normal((10, hd))
    p = O.attention_probs(q, keys, np.arange(10), 9, O.FULL, 0, 1.0)
    assert p[6] > 1 - 1e-12
    assert np.allclose(p @ vals, vals[6], atol=1e-10)


def test_attention_rows_equals_dense():
    B, T, H, Hkv, hd = 2, 11, 4, 2, 16
    r = rng(15)
    q = r.standard_normal((B, T, H, hd))
    ck, cv = _cache_from(r.standard_normal((B, T, Hkv, hd)), r.standard_normal((B, T, Hkv, hd)))
    pos = np.broadcast_to(np.arange(T), (B, T))
    dense = O.attention(q, ck, cv, pos, [T, T], Hkv, O.SLIDING, 4)
    rows = [(1, 10, 3), (0, 0, 0), (1, 4, 1)]
    got = O.attention_rows(q, ck, cv, rows, pos, [T, T], Hkv, O.SLIDING, 4)
    for i, (b, t, h) in enumerate(rows):
        assert np.allclose(got[i], dense[b, t, h], rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- routing (a7)

def test_kv_share_src_pages_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "p2_layer_routing.json")))
    n, ns, per = g["n_layers"], g["n_shared"], g["swa_period"]
    is_swa = [(i + 1) % per != 0 for i in range(n)]
    for l, e in g["expect"]["is_swa"].items():
        assert is_swa[int(l)] == e
    for l, e in g["expect"]["has_kv"].items():
        assert (O.kv_share_src(n, ns, is_swa, int(l)) < 0) == e
    for l, e in g["expect"]["kv_reuse_layer"].items():
        assert O.kv_share_src(n, ns, is_swa, int(l)) == e


def test_kv_share_src_stack_configs():
    # 42 layers, 5 sliding : 1 full, last 18 shared -> sources 22 (S) and 23 (F)
    is_swa = [(i + 1) % 6 != 0 for i in range(42)]
    srcs = {O.kv_share_src(42, 18, is_swa, l) for l in range(24, 42)}
    assert srcs == {22, 23}
    for l in range(24, 42):
        s = O.kv_share_src(42, 18, is_swa, l)
        assert is_swa[s] == is_swa[l]
    assert all(O.kv_share_src(42, 18, is_swa, l) == -1 for l in range(24))


# ---------------------------------------------------------------- append (a4)

def test_append_writes_exact_slots_and_shared_writes_nothing():
    B, T, H, Hkv, hd, Lmax = 2, 3, 4, 2, 64, 10
    r = rng(16)
    lp = dict(head_dim=hd, theta=1e4, rotary_fraction=1.0, eps=1e-6, dtype=O.BF16, kv_share_src=-1)
    q = r.standard_normal((B, T, H, hd))
    k = r.standard_normal((B, T, Hkv, hd))
    v = r.standard_normal((B, T, Hkv, hd))
    qw = 1 + 0.1 * r.standard_normal(hd)
    kw = 1 + 0.1 * r.standard_normal(hd)
    pos = np.array([[2, 3, 4], [7, 8, 9]])
    ck = np.full((B, Hkv, Lmax, hd), 1234.5)
    cv = np.full((B, Hkv, Lmax, hd), 1234.5)
    q_out = O.kv_append_normrope(lp, q, k, v, qw, kw, pos, ck, cv)
    written = np.zeros((B, Lmax), bool)
    for b in range(B):
        written[b, pos[b]] = True
    assert np.all(ck[~written[:, None, :].repeat(Hkv, 1)] == 1234.5)
    # v: weight-less norm, no rope -> every row has mean square ~ 1
    vrow = cv[0, 1, 3]
    assert np.mean(vrow ** 2) == pytest.approx(1.0, rel=1e-2)
    # stored values are bf16
    for b in range(B):
        rows = ck[b][:, pos[b]]
        assert np.array_equal(O.round_bf16(rows), rows)
    assert np.array_equal(O.round_bf16(q_out), q_out)
    # shared layer: q normed/roped the same, cache untouched
    ck2 = np.full_like(ck, 7.0)
    lp2 = dict(lp, kv_share_src=0)
    q2 = O.kv_append_normrope(lp2, q, None, None, qw, None, pos, ck2, ck2)
    assert np.array_equal(q2, q_out)
    assert np.all(ck2 == 7.0)


def test_stack_shared_layer_reads_source_cache():
    # a shared layer's output equals attention computed directly on the
    # source layer's cache with the shared layer's own q
    B, T, H, Hkv = 1, 10, 4, 2
    r = rng(17)
    layers, inputs = [], []
    types = [O.SLIDING, O.FULL, O.SLIDING, O.FULL]
    for li, lt in enumerate(types):
        hd = 64 if lt == O.SLIDING else 128
        src = O.kv_share_src(4, 2, [t == O.SLIDING for t in types], li)
        lp = dict(layer_type=lt, head_dim=hd, n_heads=H, n_kv_heads=Hkv, window=4,
                  theta=1e4 if lt == O.SLIDING else 1e6, rotary_fraction=1.0 if lt == O.SLIDING else 0.25,
                  eps=1e-6, attn_scale=1.0, kv_share_src=src, dtype=O.F32)
        layers.append(lp)
        x = dict(q=r.standard_normal((B, T, H, hd)), q_norm_w=1 + 0.1 * r.standard_normal(hd))
        if src < 0:
            x.update(k=r.standard_normal((B, T, Hkv, hd)), v=r.standard_normal((B, T, Hkv, hd)),
                     k_norm_w=1 + 0.1 * r.standard_normal(hd))
        inputs.append(x)
    outs, caches = O.run_stack_prefill(layers, inputs, B, T, T)
    assert [lp["kv_share_src"] for lp in layers] == [-1, -1, 0, 1]
    for li in (2, 3):
        lp = layers[li]
        pos = np.arange(T)[None, :]
        qn = O.store(O.normrope_q(inputs[li]["q"], inputs[li]["q_norm_w"], pos, lp["head_dim"], lp["theta"],
                                  lp["rotary_fraction"], lp["eps"]), lp["dtype"])
        ck, cv = caches[lp["kv_share_src"]]
        direct = O.store(O.attention(qn, ck, cv, pos, [T], Hkv, lp["layer_type"], lp["window"]), lp["dtype"])
        assert np.array_equal(outs[li], direct)


# ------------------------------------------------- sliding-window ring cache

def test_ring_rows_keep_the_last_capacity_positions():
    # A FIFO of bounded length is an independent model of "the ring keeps the
    # last C positions": after each append its content must be exactly the
    # resident set the oracle reports, each held in a distinct row.
    import collections
    for cap in (1, 3, 5, 8):
        fifo = collections.deque(maxlen=cap)
        for n in range(1, 4 * cap + 3):
            fifo.append(n - 1)
            pos, rows = O.ring_rows(n, cap)
            assert list(pos) == list(fifo)
            assert len(set(rows.tolist())) == len(rows)
            assert all(0 <= r < cap for r in rows)
            # the row the newest position went to is the one it overwrote
            if n > cap:
                assert O.ring_slot(n - 1, cap) == O.ring_slot(n - 1 - cap, cap)


def test_ring_append_holds_what_a_linear_cache_holds():
    # Appending the same tokens in chunks to a linear cache and to a ring of
    # capacity C: every resident position's row in the ring is bit-equal to
    # that position's row in the linear cache (same arithmetic, other slot).
    B, Hkv, H, hd, cap, N = 2, 2, 4, 64, 7, 19
    r = rng(31)
    lp = dict(head_dim=hd, theta=1e4, rotary_fraction=1.0, eps=1e-6, dtype=O.BF16, kv_share_src=-1)
    q = r.standard_normal((B, N, H, hd))
    k = r.standard_normal((B, N, Hkv, hd))
    v = r.standard_normal((B, N, Hkv, hd))
    qw = 1 + 0.1 * r.standard_normal(hd)
    kw = 1 + 0.1 * r.standard_normal(hd)
    lin_k = np.zeros((B, Hkv, N, hd))
    lin_v = np.zeros((B, Hkv, N, hd))
    ring_k = np.full((B, Hkv, cap, hd), 99.0)
    ring_v = np.full((B, Hkv, cap, hd), 99.0)
    start = 0
    for T in (5, 1, 1, 6, 1, 5):
        sl = slice(start, start + T)
        pos = np.broadcast_to(np.arange(start, start + T)[None, :], (B, T))
        q1 = O.kv_append_normrope(lp, q[:, sl], k[:, sl], v[:, sl], qw, kw, pos, lin_k, lin_v)
        q2 = O.kv_append_normrope(lp, q[:, sl], k[:, sl], v[:, sl], qw, kw, pos, ring_k, ring_v, ring=True)
        assert np.array_equal(q1, q2)
        start += T
        rpos, rrows = O.ring_rows(start, cap)
        for p, row in zip(rpos, rrows):
            assert np.array_equal(ring_k[:, :, row], lin_k[:, :, p])
            assert np.array_equal(ring_v[:, :, row], lin_v[:, :, p])
        # rows not yet reached keep their old content
        for row in range(start, cap):
            assert np.all(ring_k[:, :, row] == 99.0)
    assert start == N


@pytest.mark.parametrize("window,extra", [(4, 0), (4, 3), (1, 0)])
def test_ring_attention_equals_linear_attention(window, extra):
    # Prefill chunks and single-token decode steps on a sliding layer: with a
    # ring of capacity T_chunk + W - 1 (+ extra) the attention output equals
    # the one on a linear cache holding every position (the linear form is
    # pinned above by SDPA and by brute-force loops).  Not bitwise: the ring
    # form sums over fewer masked (zero) terms.
    B, Hkv, H, hd = 2, 2, 4, 64
    chunks = (6, 1, 1, 1, 6, 2, 1)
    N = sum(chunks)
    cap = max(chunks) + window - 1 + extra
    r = rng(32 + window + extra)
    lp = dict(head_dim=hd, theta=1e4, rotary_fraction=1.0, eps=1e-6, dtype=O.F32, kv_share_src=-1)
    q = r.standard_normal((B, N, H, hd))
    k = r.standard_normal((B, N, Hkv, hd))
    v = r.standard_normal((B, N, Hkv, hd))
    qw = 1 + 0.1 * r.standard_normal(hd)
    kw = 1 + 0.1 * r.standard_normal(hd)
    lin = (np.zeros((B, Hkv, N, hd)), np.zeros((B, Hkv, N, hd)))
    ring = (np.full((B, Hkv, cap, hd), np.nan), np.full((B, Hkv, cap, hd), np.nan))
    start = 0
    for T in chunks:
        sl = slice(start, start + T)
        pos = np.broadcast_to(np.arange(start, start + T)[None, :], (B, T))
        qo = O.kv_append_normrope(lp, q[:, sl], k[:, sl], v[:, sl], qw, kw, pos, *lin)
        O.kv_append_normrope(lp, q[:, sl], k[:, sl], v[:, sl], qw, kw, pos, *ring, ring=True)
        start += T
        kv_len = np.full(B, start)
        o_lin = O.attention(qo, *lin, pos, kv_len, Hkv, O.SLIDING, window)
        o_ring = O.attention(qo, *ring, pos, kv_len, Hkv, O.SLIDING, window, ring=True)
        assert np.all(np.isfinite(o_ring))
        np.testing.assert_allclose(o_ring, o_lin, rtol=0, atol=1e-12)
        rows = [(b, t, h) for b in range(B) for t in range(T) for h in range(H)]
        o_rows = O.attention_rows(qo, *ring, rows, pos, kv_len, Hkv, O.SLIDING, window, ring=True)
        np.testing.assert_allclose(o_rows, o_lin.reshape(-1, hd), rtol=0, atol=1e-12)


def test_ring_too_small_or_on_a_full_layer_is_refused():
    B, Hkv, H, hd, W, T = 1, 1, 1, 64, 4, 5
    r = rng(33)
    q = r.standard_normal((B, T, H, hd))
    cap = T + W - 2  # one row short: the first query's oldest key is gone
    ck = r.standard_normal((B, Hkv, cap, hd))
    pos = np.arange(10, 10 + T)[None, :]
    with pytest.raises(ValueError):
        O.attention(q, ck, ck, pos, [10 + T], Hkv, O.SLIDING, W, ring=True)
    # one more row suffices
    ck2 = r.standard_normal((B, Hkv, cap + 1, hd))
    O.attention(q, ck2, ck2, pos, [10 + T], Hkv, O.SLIDING, W, ring=True)
    with pytest.raises(ValueError):
        O.attention(q, ck2, ck2, pos, [10 + T], Hkv, O.FULL, W, ring=True)
    with pytest.raises(ValueError):
        O.ring_slot(-1, 4)


# ------------------------------------------- bidirectional (encoder) attention

@pytest.mark.parametrize("layer_type,window", [(O.FULL, 0), (O.SLIDING, 4), (O.SLIDING, 0), (O.SLIDING, 30)])
def test_bidirectional_matches_torch_sdpa_band_mask(layer_type, window):
    # library routine: torch SDPA in float64, no causal mask, the band
    # |i - j| <= W as an explicit boolean mask on sliding layers
    B, T, H, Hkv, hd = 2, 17, 4, 2, 32
    r = rng(40 + window)
    q = r.standard_normal((B, T, H, hd))
    k = r.standard_normal((B, T, Hkv, hd))
    v = r.standard_normal((B, T, Hkv, hd))
    ck, cv = _cache_from(k, v, Lmax=T + 5)
    ck[:, :, T:] = np.nan     # rows past T are never read
    cv[:, :, T:] = np.nan
    got = O.attention_bidirectional(q, ck, cv, T, Hkv, layer_type, window, 1.0)
    i = torch.arange(T)[:, None]
    j = torch.arange(T)[None, :]
    mask = torch.ones(T, T, dtype=torch.bool)
    if layer_type == O.SLIDING:
        mask = (i - j).abs() <= window
    qt = torch.from_numpy(q).permute(0, 2, 1, 3)
    kt = torch.from_numpy(k).permute(0, 2, 1, 3).repeat_interleave(H // Hkv, dim=1)
    vt = torch.from_numpy(v).permute(0, 2, 1, 3).repeat_interleave(H // Hkv, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=1.0)
    assert np.allclose(got, ref.permute(0, 2, 1, 3).numpy(), rtol=1e-12, atol=1e-12)


def test_bidirectional_brute_force_loops():
    # explicit loops over the key interval [i - W, i + W] clipped to the sequence
    B, T, H, Hkv, hd, W = 1, 9, 2, 1, 4, 2
    r = rng(41)
    q = r.standard_normal((B, T, H, hd))
    k = r.standard_normal((B, T, Hkv, hd))
    v = r.standard_normal((B, T, Hkv, hd))
    ck, cv = _cache_from(k, v)
    for lt in (O.FULL, O.SLIDING):
        got = O.attention_bidirectional(q, ck, cv, T, Hkv, lt, W)
        for t in range(T):
            lo, hi = (max(0, t - W), min(T, t + W + 1)) if lt == O.SLIDING else (0, T)
            for h in range(H):
                js = list(range(lo, hi))
                sc = [sum(q[0, t, h, d] * k[0, j, 0, d] for d in range(hd)) for j in js]
                mx = max(sc)
                ws = [math.exp(s - mx) for s in sc]
                z = sum(ws)
                exp = [sum(w * v[0, j, 0, d] for w, j in zip(ws, js)) / z for d in range(hd)]
                assert np.allclose(got[0, t, h], exp, rtol=1e-12, atol=1e-13)


def test_bidirectional_is_symmetric_under_reversal():
    # The band is symmetric: reversing the tokens reverses the output.  A
    # causal or one-sided mask fails this.
    B, T, H, Hkv, hd, W = 2, 15, 2, 2, 16, 3
    r = rng(42)
    q = r.standard_normal((B, T, H, hd))
    k = r.standard_normal((B, T, Hkv, hd))
    v = r.standard_normal((B, T, Hkv, hd))
    ck, cv = _cache_from(k, v)
    rk, rv = _cache_from(k[:, ::-1], v[:, ::-1])
    for lt in (O.FULL, O.SLIDING):
        fwd = O.attention_bidirectional(q, ck, cv, T, Hkv, lt, W)
        bwd = O.attention_bidirectional(q[:, ::-1], rk, rv, T, Hkv, lt, W)
        assert np.allclose(bwd[:, ::-1], fwd, rtol=1e-12, atol=1e-12)


def test_bidirectional_window_special_cases():
    B, T, H, Hkv, hd = 1, 12, 4, 2, 16
    r = rng(43)
    q = r.standard_normal((B, T, H, hd))
    k = r.standard_normal((B, T, Hkv, hd))
    v = r.standard_normal((B, T, Hkv, hd))
    ck, cv = _cache_from(k, v)
    # W = 0: each token sees itself alone, o_i = v_i
    o0 = O.attention_bidirectional(q, ck, cv, T, Hkv, O.SLIDING, 0)
    for h in range(H):
        assert np.allclose(o0[0, :, h], v[0, :, h // 2], rtol=0, atol=1e-15)
    # a window reaching every key (W >= T - 1) is the global layer
    full = O.attention_bidirectional(q, ck, cv, T, Hkv, O.FULL, 0)
    assert np.array_equal(O.attention_bidirectional(q, ck, cv, T, Hkv, O.SLIDING, T - 1), full)
    assert not np.allclose(O.attention_bidirectional(q, ck, cv, T, Hkv, O.SLIDING, T - 2), full)
    # the last token sees [T-1-W, T-1]: the causal window of W + 1 keys
    # (current included) at the same query -- the two conventions differ by one
    W = 4
    pos = np.arange(T)[None, :]
    bi = O.attention_bidirectional(q, ck, cv, T, Hkv, O.SLIDING, W)
    causal = O.attention(q, ck, cv, pos, [T], Hkv, O.SLIDING, W + 1)
    assert np.allclose(bi[0, T - 1], causal[0, T - 1], rtol=0, atol=1e-14)
    assert not np.allclose(bi[0, T - 1], O.attention(q, ck, cv, pos, [T], Hkv, O.SLIDING, W)[0, T - 1])


# --------------------------------- before / after the path: projections, residual

def test_qkv_projection_matches_torch_library():
    # library routines: torch rms_norm and linear in float64
    T, D, H, Hkv, hd = 5, 96, 4, 2, 16
    r = rng(50)
    x = r.standard_normal((T, D))
    nw = 1 + 0.1 * r.standard_normal(D)
    wq = r.standard_normal((H * hd, D)) / math.sqrt(D)
    wk = r.standard_normal((Hkv * hd, D)) / math.sqrt(D)
    wv = r.standard_normal((Hkv * hd, D)) / math.sqrt(D)
    q, k, v = O.qkv_projection(x, nw, wq, wk, wv, 1e-6)
    xt = torch.nn.functional.rms_norm(torch.from_numpy(x), (D,), torch.from_numpy(nw), 1e-6)
    for got, w in ((q, wq), (k, wk), (v, wv)):
        ref = torch.nn.functional.linear(xt, torch.from_numpy(w)).numpy()
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    # a shared layer projects q only
    q2, k2, v2 = O.qkv_projection(x, nw, wq, None, None, 1e-6)
    assert k2 is None and v2 is None and np.array_equal(q2, q)


def test_qkv_projection_selection_matrix_is_the_normed_input():
    # W = [I 0] picks the first outputs of the normed input exactly
    D, n = 40, 24
    r = rng(51)
    x = r.standard_normal((3, D))
    nw = 1 + 0.1 * r.standard_normal(D)
    sel = np.zeros((n, D))
    sel[np.arange(n), np.arange(n)] = 1.0
    q, _, _ = O.qkv_projection(x, nw, sel, None, None, 1e-6)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    assert np.allclose(q, (x / np.sqrt(ms + 1e-6) * nw)[:, :n], rtol=1e-14, atol=0)


def test_attn_output_residual_library_and_special_cases():
    T, D, HD = 4, 64, 48
    r = rng(52)
    h = r.standard_normal((T, D))
    ao = r.standard_normal((T, HD))
    wo = r.standard_normal((D, HD)) / math.sqrt(HD)
    pw = 1 + 0.1 * r.standard_normal(D)
    got = O.attn_output_residual(h, ao, wo, pw, 1e-6)
    a = torch.nn.functional.linear(torch.from_numpy(ao), torch.from_numpy(wo))
    ref = torch.from_numpy(h) + torch.nn.functional.rms_norm(a, (D,), torch.from_numpy(pw), 1e-6)
    assert np.allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)
    # a zero projection adds nothing (0 * (0 + eps)^-1/2 = 0)
    assert np.array_equal(O.attn_output_residual(h, ao, np.zeros_like(wo), pw, 1e-6), h)
    # with eps = 0 the added term ignores the scale of the attention output,
    # and with unit weight its mean square is 1
    g1 = O.attn_output_residual(h, ao, wo, np.ones(D), 0.0)
    g2 = O.attn_output_residual(h, 7.5 * ao, wo, np.ones(D), 0.0)
    assert np.allclose(g1, g2, rtol=0, atol=1e-12)
    assert np.allclose(np.mean((g1 - h) ** 2, axis=-1), 1.0, rtol=1e-12)


def test_k_eq_v_values_are_the_plain_norm_of_the_raw_k():
    # attention_k_eq_v (the v projection is the k projection): the layer's
    # raw v is its raw k, so each stored v row is the weight-less RMSNorm of
    # the raw k row (torch's rms_norm as the library routine), unroped, while
    # k is normed with its weight and roped as usual
    B, T, H, Hkv, hd, Lmax = 1, 3, 2, 2, 64, 8
    r = rng(60)
    lp = dict(head_dim=hd, theta=1e6, rotary_fraction=0.25, eps=1e-6, dtype=O.F32, kv_share_src=-1)
    q = r.standard_normal((B, T, H, hd))
    k = r.standard_normal((B, T, Hkv, hd))
    qw = 1 + 0.1 * r.standard_normal(hd)
    kw = 1 + 0.1 * r.standard_normal(hd)
    pos = np.array([[5, 6, 7]])
    ck = np.zeros((B, Hkv, Lmax, hd))
    cv = np.zeros((B, Hkv, Lmax, hd))
    O.kv_append_normrope(lp, q, k, k, qw, kw, pos, ck, cv)
    ref_v = torch.nn.functional.rms_norm(torch.from_numpy(k), (hd,), None, 1e-6).numpy()
    for t in range(T):
        assert np.allclose(cv[0, :, pos[0, t]], O.store(ref_v[0, t], O.F32), rtol=0, atol=1e-7)
        assert not np.allclose(ck[0, :, pos[0, t]], cv[0, :, pos[0, t]])


# ---------------------------------------------------------------- the norm -> RoPE composition

def _norm_then_rotate(x, w, pos, inv, eps, rotate=True):
    """Independent restatement: torch's rms_norm (the library routine, with
    the weight), then rotate_half as complex multiplication of
    x_j + i x_{j+hd/2} by exp(i pos inv_freq_j)."""
    hd = x.shape[-1]
    xn = torch.nn.functional.rms_norm(torch.from_numpy(np.asarray(x, np.float64)), (hd,),
                                      None if w is None else torch.from_numpy(np.asarray(w, np.float64)),
                                      eps).numpy()
    if not rotate:
        return xn
    z = xn[..., :hd // 2] + 1j * xn[..., hd // 2:]
    zr = z * np.exp(1j * np.asarray(pos, np.float64)[..., None] * inv.astype(np.float64))
    return np.concatenate([zr.real, zr.imag], axis=-1)


@pytest.mark.parametrize("hd,theta,frac", [(256, 1e4, 1.0), (512, 1e6, 0.25), (64, 1e4, 1.0), (128, 1e6, 0.25)])
@pytest.mark.parametrize("dtype", [O.F32, O.BF16])
def test_normrope_composition_norm_weight_then_rotation(hd, theta, frac, dtype):
    # The attention block of cortiq-engine g4e.rs `g4e_forward` and taconite
    # model.rs `text_attention`: q and k are RMS-normed with their own
    # weight (q_norm / k_norm) and then roped; v gets the weight-less norm
    # and no rotation.  Checked against torch's rms_norm followed by complex
    # rotation, on q / k / v rows at positions from 0 to 131071, through both
    # normrope_* and the append (which writes the cache and returns q_out).
    r = rng(70 + hd)
    B, T, H, Hkv, Lmax = 2, 3, 4, 2, 8
    eps = 1e-6
    q = r.standard_normal((B, T, H, hd))
    k = r.standard_normal((B, T, Hkv, hd))
    v = r.standard_normal((B, T, Hkv, hd))
    qw = 1 + 0.1 * r.standard_normal(hd)
    kw = 1 + 0.1 * r.standard_normal(hd)
    pos = np.array([[0, 9, 131071], [4096, 4098, 5]])  # distinct rows mod 8
    inv = O.rope_inv_freq(hd, theta, frac)
    ref_q = _norm_then_rotate(q, qw, pos[..., None], inv, eps)
    ref_k = _norm_then_rotate(k, kw, pos[..., None], inv, eps)
    ref_v = _norm_then_rotate(v, None, pos[..., None], inv, eps, rotate=False)
    # normrope_q / normrope_kv
    assert np.allclose(O.normrope_q(q, qw, pos, hd, theta, frac, eps), ref_q, rtol=0, atol=1e-12)
    kn, vn = O.normrope_kv(k, v, kw, pos, hd, theta, frac, eps)
    assert np.allclose(kn, ref_k, rtol=0, atol=1e-12)
    assert np.allclose(vn, ref_v, rtol=0, atol=1e-12)
    # the append: q_out with q's weight, cache k with k's weight, v unroped,
    # each rounded as stored (round_bf16 is pinned against torch above)
    lp = dict(head_dim=hd, theta=theta, rotary_fraction=frac, eps=eps, dtype=dtype, kv_share_src=-1)
    ck = np.zeros((B, Hkv, Lmax, hd))
    cv = np.zeros((B, Hkv, Lmax, hd))
    ring_cap = Lmax
    q_out = O.kv_append_normrope(lp, q, k, v, qw, kw, pos, ck, cv, ring=True)
    tol = 1e-6 if dtype == O.F32 else 2.0 ** -7
    assert np.allclose(q_out, ref_q, rtol=tol, atol=1e-6)
    for b in range(B):
        for t in range(T):
            row = int(pos[b, t]) % ring_cap
            assert np.allclose(ck[b, :, row], ref_k[b, t], rtol=tol, atol=1e-6)
            assert np.allclose(cv[b, :, row], ref_v[b, t], rtol=tol, atol=1e-6)
    # The mistakes this pin separates from the right composition: RoPE
    # before the weighted norm (the weight is per element, so the two do not
    # commute), the weights of q and k exchanged, v roped.
    rope_first = _norm_then_rotate(q, None, pos[..., None], inv, eps) * qw
    swapped_q = _norm_then_rotate(q, kw, pos[..., None], inv, eps)
    roped_v = _norm_then_rotate(v, None, pos[..., None], inv, eps)
    assert not np.allclose(rope_first, ref_q, rtol=0, atol=1e-3)
    assert not np.allclose(swapped_q, ref_q, rtol=0, atol=1e-3)
    assert not np.allclose(roped_v, ref_v, rtol=0, atol=1e-3)


def test_qkv_projection_with_the_norm_weight_folded_into_w():
    # rms(x, a) W^T = rms(x) (W diag(a))^T: the attention-norm weight may be
    # multiplied into the projection's columns (the form the fused projection
    # takes), exactly in float64
    r = rng(80)
    D, Nq, Nk = 64, 48, 16
    x = r.standard_normal((3, 5, D))
    a = 1 + 0.1 * r.standard_normal(D)
    wq, wk, wv = r.standard_normal((Nq, D)), r.standard_normal((Nk, D)), r.standard_normal((Nk, D))
    q1, k1, v1 = O.qkv_projection(x, a, wq, wk, wv, 1e-6)
    q2, k2, v2 = O.qkv_projection(x, None, wq * a, wk * a, wv * a, 1e-6)
    for u, w_ in ((q1, q2), (k1, k2), (v1, v2)):
        assert np.allclose(u, w_, rtol=1e-13, atol=1e-13)
    # and a shared layer projects q only
    q3, k3, v3 = O.qkv_projection(x, a, wq, None, None, 1e-6)
    assert k3 is None and v3 is None and np.array_equal(q3, q1)

"""Host-side tests of the C ABI (no GPU needed).

Loads libg4attn.so, checks that it exports every entry point the header
declares, and exercises the argument validation and the shared-KV routing,
none of which launches a kernel.
"""

import json
import os
import re
import subprocess

import pytest

from gemma_dual_geometry_gb300 import build as g4build
from gemma_dual_geometry_gb300 import g4attn as G
from oracle import g4_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "g4attn.h")
FAKE = 0x7f0000000000  # aligned, never dereferenced: validation fails first


@pytest.fixture(scope="module")
def L():
    g4build.build()
    return G.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(g4_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_are_all_exported(L):
    names = declared_functions()
    assert "g4_kv_append_normrope" in names and "g4_attn_prefill" in names and "g4_attn_decode" in names
    for n in names:
        assert hasattr(L, n), n
        assert n in G.SIGNATURES, n
    out = subprocess.run(["nm", "-D", "--defined-only", G.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (g4_[a-z0-9_]+)$", out, flags=re.M))
    assert exported == set(names)


def test_kv_share_src_worked_example(L):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "p2_layer_routing.json")))
    n, ns, per = g["n_layers"], g["n_shared"], g["swa_period"]
    is_swa = [(i + 1) % per != 0 for i in range(n)]
    for l, e in g["expect"]["kv_reuse_layer"].items():
        assert G.g4_kv_share_src(n, ns, is_swa, int(l)) == e
    for l, e in g["expect"]["has_kv"].items():
        assert (G.g4_kv_share_src(n, ns, is_swa, int(l)) == -1) == e


@pytest.mark.parametrize("n,ns,period", [(42, 18, 6), (4, 2, 2), (10, 4, 5), (35, 15, 5), (7, 0, 3)])
def test_kv_share_src_matches_oracle(L, n, ns, period):
    is_swa = [(i + 1) % period != 0 for i in range(n)]
    for l in range(n):
        assert G.g4_kv_share_src(n, ns, is_swa, l) == O.kv_share_src(n, ns, is_swa, l)


def test_kv_share_src_invalid(L):
    assert G.g4_kv_share_src(4, 4, [1, 1, 1, 1], 0) == -2
    assert G.g4_kv_share_src(4, 1, [1, 1, 1, 1], 4) == -2
    assert G.g4_kv_share_src(4, 1, [1, 1, 1, 1], -1) == -2
    assert G.g4_kv_share_src(2, 1, [1, 1], 1) == -2   # sliding tail would read layer -1
    assert L.g4_kv_share_src(4, 1, None, 0) == -2


def _params(**kw):
    d = dict(layer_type=G.G4_SLIDING, head_dim=256, n_heads=8, n_kv_heads=2, window=512, theta=1e4,
             rotary_fraction=1.0, eps=1e-6, attn_scale=1.0, kv_share_src=-1, dtype=G.G4_BF16)
    d.update(kw)
    return G.layer_params(**d)


def _table(entries):
    t = G.cache_table(len(entries))
    for i, e in enumerate(entries):
        if e is not None:
            G.set_cache(t, i, FAKE, FAKE + 4096, *e)
    return t


def _status(fn, *args):
    try:
        fn(*args)
        return G.G4_OK
    except G.G4Error as e:
        return e.status


def test_validation_errors(L):
    tab = _table([(G.G4_SLIDING, 256, 2, 100, 1, G.G4_BF16)])

    def pf(p, B=1, T=4):
        return _status(G.g4_attn_prefill, p, tab, 0, FAKE, FAKE, B, T, FAKE, 0)

    assert L.g4_attn_prefill(None, tab, 1, 0, FAKE, FAKE, 1, 4, FAKE, None) == G.G4_ERR_INVALID_ARG
    assert "params" in G.g4_last_error()
    assert pf(_params(head_dim=96)) == G.G4_ERR_UNSUPPORTED
    assert pf(_params(n_heads=12, n_kv_heads=2)) == G.G4_ERR_UNSUPPORTED       # group 6
    assert pf(_params(n_heads=8, n_kv_heads=1, head_dim=512)) == G.G4_ERR_UNSUPPORTED   # 8 x 512 > 2048
    assert pf(_params(n_heads=7, n_kv_heads=2)) == G.G4_ERR_INVALID_ARG
    assert pf(_params(window=0)) == G.G4_ERR_INVALID_ARG
    assert pf(_params(theta=0.0)) == G.G4_ERR_INVALID_ARG
    assert pf(_params(rotary_fraction=1.5)) == G.G4_ERR_INVALID_ARG
    assert pf(_params(attn_scale=-1.0)) == G.G4_ERR_INVALID_ARG
    assert pf(_params(dtype=7)) == G.G4_ERR_INVALID_ARG
    assert pf(_params(layer_type=G.G4_FULL)) == G.G4_ERR_SHARE_MISMATCH         # cache is sliding
    assert pf(_params(head_dim=512)) == G.G4_ERR_SHARE_MISMATCH
    assert pf(_params(dtype=G.G4_F32)) == G.G4_ERR_SHARE_MISMATCH
    assert pf(_params(n_heads=4, n_kv_heads=4)) == G.G4_ERR_SHARE_MISMATCH     # kv-head count differs
    assert pf(_params(), B=2) == G.G4_ERR_CAPACITY
    assert pf(_params(), T=101) == G.G4_ERR_CAPACITY
    assert pf(_params(), B=0) == G.G4_OK
    assert pf(_params(), T=0) == G.G4_OK
    # misaligned pointer
    assert _status(G.g4_attn_prefill, _params(), tab, 0, FAKE + 2, FAKE, 1, 4, FAKE, 0) == G.G4_ERR_INVALID_ARG
    # layer outside the table, source outside the table, source without a cache
    assert _status(G.g4_attn_prefill, _params(), tab, 1, FAKE, FAKE, 1, 4, FAKE, 0) == G.G4_ERR_INVALID_ARG
    assert pf(_params(kv_share_src=3)) == G.G4_ERR_INVALID_ARG
    tab2 = _table([(G.G4_SLIDING, 256, 2, 100, 1, G.G4_BF16), None])
    assert _status(G.g4_attn_prefill, _params(kv_share_src=1), tab2, 0, FAKE, FAKE, 1, 4, FAKE, 0) == \
        G.G4_ERR_INVALID_ARG


def test_append_validation(L):
    tab = _table([(G.G4_SLIDING, 256, 2, 100, 1, G.G4_BF16), None])

    def ap(p, layer, k, v, kw, B=1):
        return _status(G.g4_kv_append_normrope, p, tab, layer, FAKE, k, v, FAKE, kw, FAKE, B, 2, FAKE, 0)

    # an owning layer needs k, v and k_norm_w
    assert ap(_params(), 0, None, FAKE, FAKE) == G.G4_ERR_INVALID_ARG
    assert ap(_params(), 0, FAKE, FAKE, None) == G.G4_ERR_INVALID_ARG
    # a shared layer must not pass k / v / k_norm_w
    assert ap(_params(kv_share_src=0), 1, FAKE, FAKE, FAKE) == G.G4_ERR_INVALID_ARG
    assert ap(_params(kv_share_src=0), 1, None, None, None, B=0) == G.G4_OK
    assert ap(_params(), 0, FAKE, FAKE, FAKE, B=2) == G.G4_ERR_CAPACITY
    assert ap(_params(), 0, FAKE, FAKE, FAKE, B=0) == G.G4_OK
    assert ap(_params(head_dim=128), 0, FAKE, FAKE, FAKE) == G.G4_ERR_SHARE_MISMATCH


def test_decode_validation_and_workspace(L):
    tab = _table([(G.G4_FULL, 512, 2, 8192, 64, G.G4_BF16)])
    p = _params(layer_type=G.G4_FULL, head_dim=512, theta=1e6, rotary_fraction=0.25, window=0)
    need = G.g4_attn_decode_workspace_size(p, 64, 8192)
    assert need > 0 and need % 256 == 0

    def dec(B=64, maxlen=8192, ws=FAKE, wsb=need):
        return _status(G.g4_attn_decode, p, tab, 0, FAKE, FAKE, B, maxlen, FAKE, ws, wsb, 0)

    assert dec(wsb=need - 1) == G.G4_ERR_WORKSPACE
    assert dec(ws=None) == G.G4_ERR_INVALID_ARG
    assert dec(maxlen=8193) == G.G4_ERR_CAPACITY
    assert dec(maxlen=0) == G.G4_ERR_CAPACITY
    assert dec(B=65) == G.G4_ERR_CAPACITY
    assert dec(B=0) == G.G4_OK
    # a sliding layer whose window is no longer than the minimum split needs no workspace
    assert G.g4_attn_decode_workspace_size(_params(window=64), 64, 8192) == 0    # one 64-key split
    # bf16 spans of at most 512 keys (head_dim <= 256) merge their splits in a
    # cluster when its CTAs fit one wave: no workspace; longer windows, head_dim
    # 512, float32 and more (sequence, kv head) pairs use the split kernel's
    assert G.g4_attn_decode_workspace_size(_params(window=512), 8, 8192) == 0       # 16 clusters of 8
    assert G.g4_attn_decode_workspace_size(_params(layer_type=G.G4_FULL, window=0), 8, 512) == 0
    assert G.g4_attn_decode_workspace_size(_params(window=512), 64, 8192) > 0      # 1024 CTAs: split kernel
    assert G.g4_attn_decode_workspace_size(_params(window=1024), 8, 8192) > 0
    assert G.g4_attn_decode_workspace_size(_params(window=512, dtype=G.G4_F32), 8, 8192) > 0
    assert G.g4_attn_decode_workspace_size(_params(layer_type=G.G4_FULL, window=0), 8, 513) > 0
    assert L.g4_attn_decode_workspace_size(None, 64, 8192) == 0


def test_decode_step_validation(L):
    tab = _table([(G.G4_SLIDING, 256, 2, 100, 4, G.G4_BF16), None])

    def st(p, layer, k, v, kw, qw=FAKE, B=4):
        return _status(G.g4_decode_step, p, tab, layer, FAKE, k, v, qw, kw, FAKE, B, 100, FAKE, FAKE, 1 << 20, 0)

    assert st(_params(), 0, None, FAKE, FAKE) == G.G4_ERR_INVALID_ARG           # owner needs k/v/k_norm_w
    assert st(_params(), 0, FAKE, FAKE, FAKE, qw=None) == G.G4_ERR_INVALID_ARG  # q_norm_w required
    assert st(_params(kv_share_src=0), 1, FAKE, None, None) == G.G4_ERR_INVALID_ARG  # shared: no k/v
    assert st(_params(kv_share_src=0), 1, None, None, None, B=0) == G.G4_OK
    assert st(_params(), 0, FAKE, FAKE, FAKE, B=5) == G.G4_ERR_CAPACITY
    assert st(_params(head_dim=512), 0, FAKE, FAKE, FAKE) == G.G4_ERR_SHARE_MISMATCH


def test_ring_cache_validation(L):
    # Sliding-window ring caches: only on sliding layers, at least a window of
    # rows, and a prefill chunk must leave every key of its windows resident.
    W = 512
    def ring(max_len, lt=G.G4_SLIDING, hd=256, dt=G.G4_BF16, flag=1):
        t = _table([(lt, hd, 2, max_len, 1, dt)])
        t[0].ring = flag   # the raw field, so that values other than 0 / 1 reach the library
        return t

    full = _params(layer_type=G.G4_FULL, head_dim=512, theta=1e6, rotary_fraction=0.25, window=0)

    def pf(p, tab, T, B=1):   # B=0: every host check, no launch
        return _status(G.g4_attn_prefill, p, tab, 0, FAKE, FAKE, B, T, FAKE, 0)

    assert pf(_params(), ring(1024, flag=2), 4) == G.G4_ERR_INVALID_ARG
    assert pf(full, ring(1024, lt=G.G4_FULL, hd=512), 4) == G.G4_ERR_INVALID_ARG
    assert pf(_params(), ring(W - 1), 1) == G.G4_ERR_CAPACITY
    # T + W - 1 keys: 513 + 511 = 1024 fit a 1024-row ring, 514 do not
    assert pf(_params(), ring(1024), 514) == G.G4_ERR_CAPACITY
    assert pf(_params(), ring(1024), 0) == G.G4_OK
    # the bf16 prefill needs whole 128-key tiles in the ring; float32 does not
    assert pf(_params(), ring(1000), 0) == G.G4_ERR_UNSUPPORTED
    assert pf(_params(dtype=G.G4_F32), ring(1000, dt=G.G4_F32), 0) == G.G4_OK
    # with a one-token window a chunk may fill the whole ring, not more
    assert pf(_params(window=1), ring(256), 256, B=0) == G.G4_OK
    assert pf(_params(window=1), ring(256), 257) == G.G4_ERR_CAPACITY

    # decode: the sequence may be longer than the ring
    def dec(tab, maxlen, B=0):
        return _status(G.g4_attn_decode, _params(), tab, 0, FAKE, FAKE, B, maxlen, FAKE, FAKE, 1 << 30, 0)

    assert dec(ring(W), 100000) == G.G4_OK
    assert dec(ring(W, flag=0), 100000) == G.G4_ERR_CAPACITY
    assert dec(ring(W - 1), 100) == G.G4_ERR_CAPACITY

    # append: a ring is validated like any cache
    def ap(tab):
        return _status(G.g4_kv_append_normrope, _params(), tab, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 2,
                       FAKE, 0)

    assert ap(ring(W)) == G.G4_OK
    assert ap(ring(W - 1)) == G.G4_ERR_CAPACITY


def test_encoder_validation(L):
    tab = _table([(G.G4_SLIDING, 256, 2, 100, 2, G.G4_BF16)])

    def enc(p=None, tab=tab, B=2, T=4, q=FAKE, out=FAKE):
        return _status(G.g4_attn_encoder, p or _params(), tab, 0, q, B, T, out, 0)

    assert enc(B=0) == G.G4_OK
    assert enc(T=0) == G.G4_OK
    assert enc(B=3) == G.G4_ERR_CAPACITY
    assert enc(T=101, B=0) == G.G4_ERR_CAPACITY
    assert enc(T=-1) == G.G4_ERR_INVALID_ARG
    assert enc(q=None) == G.G4_ERR_INVALID_ARG
    assert enc(out=FAKE + 8) == G.G4_ERR_INVALID_ARG
    assert enc(_params(head_dim=512)) == G.G4_ERR_SHARE_MISMATCH
    assert enc(_params(window=0)) == G.G4_ERR_INVALID_ARG
    # the encoder reads rows 0 .. T-1: no ring
    ring = _table([(G.G4_SLIDING, 256, 2, 1024, 2, G.G4_BF16, True)])
    assert enc(tab=ring, B=0) == G.G4_ERR_INVALID_ARG
    assert "ring" in G.g4_last_error()


def test_tiny_config_literal_layer_types_are_rejected(L):
    # The tiny config's literal [S, S, S, F] with the last two layers shared
    # routes the full tail layer (head_dim 128) to layer 1, a sliding layer of
    # head_dim 64: the same-type rule forbids it, and the library says so.
    types = [G.G4_SLIDING, G.G4_SLIDING, G.G4_SLIDING, G.G4_FULL]
    src3 = G.g4_kv_share_src(4, 2, [t == G.G4_SLIDING for t in types], 3)
    assert src3 == 1
    tab = _table([(G.G4_SLIDING, 64, 2, 64, 1, G.G4_F32), (G.G4_SLIDING, 64, 2, 64, 1, G.G4_F32), None, None])
    p3 = _params(layer_type=G.G4_FULL, head_dim=128, n_heads=4, n_kv_heads=2, theta=1e6, rotary_fraction=0.25,
                 kv_share_src=src3, dtype=G.G4_F32)
    assert _status(G.g4_attn_prefill, p3, tab, 3, FAKE, FAKE, 1, 64, FAKE, 0) == G.G4_ERR_SHARE_MISMATCH
    assert "cannot read the cache of layer 1" in G.g4_last_error()


def test_binding_refuses_to_run_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(G, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(G, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        G.lib()


def test_projection_validation(L):
    # every call here is refused before a launch, or has no rows (B*T == 0 or
    # M == 0): the fake addresses are never dereferenced
    tab = _table([(G.G4_SLIDING, 256, 2, 100, 2, G.G4_BF16), None])

    def qkv(p=None, layer=0, x=FAKE, D=512, w=FAKE, kw=FAKE, B=2, T=4, q_out=FAKE, tab=tab):
        return _status(G.g4_qkv_project_append, p or _params(), tab, layer, x, D, w, FAKE, kw, FAKE, B, T, q_out, 0)

    assert qkv(B=0) == G.G4_OK
    assert qkv(T=0) == G.G4_OK
    assert qkv(D=100) == G.G4_ERR_UNSUPPORTED                       # not a multiple of 64
    assert qkv(D=0) == G.G4_ERR_UNSUPPORTED
    assert qkv(_params(dtype=G.G4_F32)) == G.G4_ERR_UNSUPPORTED      # tensor cores: bf16 only
    assert qkv(x=None) == G.G4_ERR_INVALID_ARG
    assert qkv(w=FAKE + 8) == G.G4_ERR_INVALID_ARG
    assert qkv(kw=None) == G.G4_ERR_INVALID_ARG                     # owning layer needs k_norm_w
    assert qkv(B=3) == G.G4_ERR_CAPACITY
    assert qkv(_params(head_dim=512)) == G.G4_ERR_SHARE_MISMATCH
    assert qkv(_params(kv_share_src=0), layer=1, kw=FAKE) == G.G4_ERR_INVALID_ARG   # shared: no k_norm_w
    assert qkv(_params(kv_share_src=0), layer=1, kw=None, B=0) == G.G4_OK

    def out(M=4, K=512, D=2048, eps=1e-6, ao=FAKE, w=FAKE, h=FAKE, o=FAKE):
        return _status(G.g4_attn_out_residual, ao, M, K, w, D, FAKE, eps, h, o, 0)

    assert out(M=0) == G.G4_OK
    assert out(M=-1) == G.G4_ERR_INVALID_ARG
    assert out(D=2304) == G.G4_ERR_UNSUPPORTED                      # row spans more than 8 CTAs
    assert out(D=300) == G.G4_ERR_UNSUPPORTED
    assert out(K=96) == G.G4_ERR_UNSUPPORTED
    assert out(eps=-1.0) == G.G4_ERR_INVALID_ARG
    assert out(h=None) == G.G4_ERR_INVALID_ARG
    assert out(o=FAKE + 4) == G.G4_ERR_INVALID_ARG

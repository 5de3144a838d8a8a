"""Plain float64 CPU oracle for the Gemma-4 E-series dual-geometry attention path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The CUDA library never calls it, and it shares no code with the CUDA
library: it takes numpy arrays and returns numpy arrays.

What it computes, and where each step comes from (page title + function):

* ``rms_norm``       -- plain x-hat * w RMSNorm, eps inside the mean
                        (cortiq-engine ``g4e.rs``: ``rms``; weight-less form
                        ``rms_plain`` for V).
* ``rope_inv_freq``  -- per-layer RoPE inverse frequencies: ``theta^(-2j/hd)``
                        for the rotated prefix, zero for the tail
                        (cortiq-engine ``g4e.rs``: ``G4eGlobals`` doc on
                        ``inv_freq_local`` / ``inv_freq_global``;
                        turbospark-runtime ``gemma4/attn.rs``:
                        ``rotated_pairs``).
* ``rope_rotate_half`` -- rotate_half ("neox") RoPE on pairs (j, j+hd/2)
                        (taconite-embeddinggemma2 ``model.rs``: ``rope_half``).
* ``kv_append_normrope`` -- norm -> RoPE on q and k, weight-less norm on v,
                        k/v written to the layer's cache at the token position
                        (cortiq-engine ``g4e.rs``: ``g4e_forward`` attention
                        block; ferrox-models ``gemma4_engine.rs``:
                        ``forward_token_on_worker``).
* ``attention``      -- causal GQA softmax attention, score scale 1.0,
                        sliding window with the current token included
                        (cortiq-engine ``g4e.rs``: ``attend_all_heads`` call with
                        scale 1.0 and ``window``; ferrox-models
                        ``causal_gqa_attention[_windowed]``; head grouping as in
                        taconite ``text_attention``: ``kh = hh / group``).
* ``ring_rows``      -- sliding-window ring-buffer cache: a sliding layer's
                        cache of capacity C keeps position p in row p mod C,
                        so only the last C positions stay resident
                        (turbospark-runtime ``gemma4`` decode: ``ring_capacity``
                        and ``active_ring`` passed to the attention next to
                        ``kv_start = seq_len - sliding_window``).
* ``attention_bidirectional`` -- the encoder form of the same attention
                        (taconite-embeddinggemma2 ``model.rs``:
                        ``text_attention``): no causal mask, and a sliding
                        layer sees the keys with |i - j| <= window.
* ``qkv_projection`` -- the step before the path: the layer input's RMSNorm
                        (attn_norm) and the q / k / v projections
                        (cortiq-engine ``g4e_forward``: ``rms(h, attn_norm)``
                        then ``matvec`` with wq / wk / wv; memra-engine
                        ``forward.rs``: ``rms_norm`` then the linear layers).
* ``attn_output_residual`` -- the step after it: o_proj, the
                        post-attention RMSNorm and the residual add
                        (cortiq-engine ``g4e_forward`` "sandwich"; ferrox-models
                        ``forward_token_on_worker``: ``o_proj``,
                        ``post_attn_norm``, add to ``hidden``).
* ``kv_share_src``   -- shared-KV routing of the tail layers
                        (ferrox-models ``Gemma4Hparams::kv_reuse_layer``;
                        cortiq-engine ``g4e.rs`` module doc on shared KV).

Everything is float64.  Inputs given as bf16 are widened exactly by the
caller.  Where the interface stores bf16 (the KV cache, q_out and the
attention output), ``round_bf16`` applies round-to-nearest-even to the float64
value, so the oracle's stored values are the correctly rounded ones.

Parity pins for every function live in ``tests/test_oracle_pins.py``.
"""

from __future__ import annotations

import math

import numpy as np

SLIDING = 0
FULL = 1

F32 = 0
BF16 = 1


# --------------------------------------------------------------------------
# Storage rounding
# --------------------------------------------------------------------------

def round_bf16(x):
    """Round float64 values to the nearest bfloat16 (ties to even).

    bfloat16 keeps 8 significant bits and float32's exponent range.  A
    finite x = m * 2**e with 0.5 <= |m| < 1 rounds to round(m * 2**8) * 2**(e-8)
    (numpy's ``np.round`` rounds half to even).  Values below the smallest
    normal (2**-126) use the subnormal quantum 2**-133.  The scaling by a
    power of two is exact, so the only rounding is the one ``np.round`` does.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    finite = np.isfinite(x) & (x != 0.0)
    xf = x[finite]
    m, e = np.frexp(xf)
    normal = np.abs(xf) >= 2.0 ** -126
    r = np.empty_like(xf)
    r[normal] = np.ldexp(np.round(np.ldexp(m[normal], 8)), e[normal] - 8)
    sub = ~normal
    r[sub] = np.round(xf[sub] / 2.0 ** -133) * 2.0 ** -133
    # overflow past the largest bfloat16 becomes infinity
    big = np.abs(r) > 3.3895313892515355e38
    r[big] = np.copysign(np.inf, r[big])
    out[finite] = r
    return out


def store(x, dtype):
    """Value as the interface stores it: float32 for F32, bfloat16 for BF16."""
    if dtype == BF16:
        return round_bf16(x)
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# a1 / a2: RMSNorm
# --------------------------------------------------------------------------

def rms_norm(x, w, eps):
    """y = x * (mean(x**2) + eps) ** -1/2 * w over the last axis, in float64.

    cortiq-engine ``g4e.rs``: ``rms`` (the weight multiplies as-is, it is not
    1 + w) and ``rms_plain`` (no weight, used for V).  ``w=None`` is the
    weight-less form.
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.sum(x * x, axis=-1, keepdims=True) / x.shape[-1]
    inv = (ms + eps) ** -0.5
    y = x * inv
    if w is not None:
        y = y * np.asarray(w, dtype=np.float64)
    return y


# --------------------------------------------------------------------------
# a3: RoPE
# --------------------------------------------------------------------------

def rotated_pairs(head_dim, rotary_fraction):
    """Number of rotated pairs: floor(head_dim * fraction / 2).

    turbospark-runtime ``gemma4/attn.rs``: ``rotated_pairs`` is
    ``(full_head_dim * partial_rotary_factor / 2.0) as u32`` (a truncation).
    A sliding layer rotates all head_dim/2 pairs (fraction 1.0).
    """
    return int(math.floor(float(head_dim) * float(rotary_fraction) / 2.0))


def rope_inv_freq(head_dim, theta, rotary_fraction):
    """float32 table of head_dim/2 inverse frequencies.

    inv_freq[j] = theta ** (-2j / head_dim) for j < rotated_pairs, else 0.
    The power is taken in float64 and rounded to float32 once, because the
    pages keep the table as ``Vec<f32>`` (cortiq-engine ``G4eGlobals``) and
    build it in f32 (taconite ``text_attention``).  The denominator is the
    full head width; a zero frequency leaves its pair unrotated, so the tail
    passes through unchanged (cortiq-engine ``g4e.rs``, the ``G4eGlobals``
    documentation of the global inverse-frequency table).
    """
    half = head_dim // 2
    n_rot = min(rotated_pairs(head_dim, rotary_fraction), half)
    inv = np.zeros(half, dtype=np.float32)
    th = float(theta)
    for j in range(n_rot):
        inv[j] = np.float32(th ** (-2.0 * j / head_dim))
    return inv


def rope_rotate_half(x, pos, inv_freq):
    """rotate_half RoPE on the last axis.

    For j < hd/2 with angle = pos * inv_freq[j] (float64):
        x'[j]      = x[j] cos - x[j+hd/2] sin
        x'[j+hd/2] = x[j+hd/2] cos + x[j] sin
    (taconite ``model.rs``: ``rope_half`` with the cos/sin table duplicated
    over both halves).  ``pos`` broadcasts against ``x.shape[:-1]``.
    """
    x = np.asarray(x, dtype=np.float64)
    hd = x.shape[-1]
    half = hd // 2
    ang = np.asarray(pos, dtype=np.float64)[..., None] * np.asarray(inv_freq, dtype=np.float32).astype(np.float64)
    c = np.cos(ang)
    s = np.sin(ang)
    a = x[..., :half]
    b = x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


# --------------------------------------------------------------------------
# a4: the fused norm -> RoPE -> KV append
# --------------------------------------------------------------------------

def normrope_q(q_in, q_norm_w, positions, head_dim, theta, rotary_fraction, eps):
    """Normed and roped q, float64.  q_in [..., H, hd]; positions [...]."""
    inv = rope_inv_freq(head_dim, theta, rotary_fraction)
    qn = rms_norm(q_in, q_norm_w, eps)
    return rope_rotate_half(qn, np.asarray(positions)[..., None], inv)


def normrope_kv(k_in, v_in, k_norm_w, positions, head_dim, theta, rotary_fraction, eps):
    """Normed + roped k and weight-less normed v, float64 (no RoPE on v)."""
    inv = rope_inv_freq(head_dim, theta, rotary_fraction)
    kn = rope_rotate_half(rms_norm(k_in, k_norm_w, eps), np.asarray(positions)[..., None], inv)
    vn = rms_norm(v_in, None, eps)
    return kn, vn


def kv_append_normrope(lp, q_in, k_in, v_in, q_norm_w, k_norm_w, positions, cache_k, cache_v, ring=False):
    """Step a4 for one layer and a batch of tokens.

    lp: dict with head_dim, theta, rotary_fraction, eps, dtype and
        kv_share_src (-1 when the layer owns its cache).
    q_in [B, T, H, hd]; k_in / v_in [B, T, Hkv, hd] or None on a shared
    layer; positions [B, T] (the cache slot and the RoPE position);
    cache_k / cache_v [B, Hkv, Lmax, hd] float64 arrays updated in place
    (ignored on a shared layer).  With ``ring`` the cache is a sliding-window
    ring of Lmax rows and position p goes to row p mod Lmax (``ring_rows``).

    Returns q_out [B, T, H, hd] as stored (bf16- or f32-rounded).
    Shared layers norm and rope q and write nothing
    (cortiq-engine ``g4e_forward``: the append sits under
    ``if lw.kv_share_src.is_none()``).
    """
    hd, th, fr, eps, dt = lp["head_dim"], lp["theta"], lp["rotary_fraction"], lp["eps"], lp["dtype"]
    positions = np.asarray(positions, dtype=np.int64)
    q_out = store(normrope_q(q_in, q_norm_w, positions, hd, th, fr, eps), dt)
    if lp.get("kv_share_src", -1) < 0:
        kn, vn = normrope_kv(k_in, v_in, k_norm_w, positions, hd, th, fr, eps)
        kn = store(kn, dt)
        vn = store(vn, dt)
        B, T = positions.shape
        cap = cache_k.shape[2]
        for b in range(B):
            for t in range(T):
                p = int(positions[b, t])
                row = ring_slot(p, cap) if ring else p
                cache_k[b, :, row, :] = kn[b, t]
                cache_v[b, :, row, :] = vn[b, t]
    return q_out


# --------------------------------------------------------------------------
# Sliding-window ring-buffer cache
# --------------------------------------------------------------------------

def ring_slot(pos, capacity):
    """Row of a ring cache of ``capacity`` rows that holds position ``pos``.

    The ring keeps every position in row pos mod capacity, so appending
    position p overwrites position p - capacity (turbospark-runtime
    ``gemma4`` decode: the attention gets the ring capacity once the sequence
    is longer than it, ``if ring > 0 && seq_len > ring``).
    """
    if capacity < 1 or pos < 0:
        raise ValueError("ring capacity must be >= 1 and positions >= 0")
    return pos % capacity


def ring_rows(kv_len, capacity):
    """Positions still resident in a ring after positions [0, kv_len) were
    appended in order, and the rows holding them: the last ``capacity``
    positions, (positions, rows) in position order."""
    pos = np.arange(max(0, kv_len - capacity), kv_len, dtype=np.int64)
    return pos, pos % capacity


def check_ring_covers(q_pos, kv_len, capacity, layer_type, window):
    """Raise unless every key a query needs is still resident in the ring.

    Only a sliding layer can use a ring (a full layer needs every earlier
    key).  The query at q_pos needs positions [max(0, q_pos - window + 1),
    q_pos]; the ring holds [max(0, kv_len - capacity), kv_len).  So a chunk
    of T new tokens appended before its attention needs
    capacity >= T + window - 1.
    """
    if layer_type != SLIDING:
        raise ValueError("a ring cache needs a sliding layer")
    first_resident = max(0, int(kv_len) - capacity)
    q_pos = np.asarray(q_pos, dtype=np.int64)
    need = np.maximum(0, q_pos - window + 1)
    if np.any(need < first_resident):
        raise ValueError("ring of %d rows no longer holds key %d that a query needs"
                         % (capacity, int(np.min(need))))


# --------------------------------------------------------------------------
# a5 / a6: causal GQA attention with score scale 1.0
# --------------------------------------------------------------------------

def visible(q_pos, k_pos, layer_type, window):
    """Key at position k_pos is visible from a query at q_pos.

    Causal (k <= q) on every layer; a sliding layer also needs q - k < window,
    i.e. the window is counted in tokens and the query's own token is one of
    them (cortiq-engine ``g4e.rs``, the ``G4eGlobals`` field documentation of
    the window; turbospark-runtime ``gemma4/attn.rs``, decode:
    ``kv_start = seq_len - sliding_window``).
    """
    q_pos = np.asarray(q_pos)
    k_pos = np.asarray(k_pos)
    vis = k_pos <= q_pos
    if layer_type == SLIDING:
        vis = vis & ((q_pos - k_pos) < window)
    return vis


def attention_probs(q_row, keys, k_pos, q_pos, layer_type, window, scale):
    """Softmax weights of one query row over ``keys`` [L, hd] (float64).

    scores = scale * q . k_j on visible keys, -inf elsewhere; softmax with the
    row maximum subtracted (taconite ``text_attention`` computes dot,
    ``softmax_``, then the weighted sum).
    """
    s = (keys @ np.asarray(q_row, dtype=np.float64)) * scale
    vis = visible(q_pos, k_pos, layer_type, window)
    s = np.where(vis, s, -np.inf)
    m = np.max(s)
    e = np.exp(s - m)
    return e / np.sum(e)


def key_rows(kv_len, capacity, ring):
    """(positions, cache rows) of the keys a sequence of kv_len tokens has:
    rows 0 .. kv_len-1 of a linear cache, the resident part of a ring."""
    if ring:
        return ring_rows(kv_len, capacity)
    pos = np.arange(kv_len, dtype=np.int64)
    return pos, pos


def attention(q, cache_k, cache_v, q_pos, kv_len, n_kv_heads, layer_type, window, scale=1.0, ring=False):
    """o[b, t, h] = sum_j softmax_j(scale * q[b,t,h] . k_j) v_j over visible j.

    q [B, T, H, hd] (already normed and roped); cache_k / cache_v
    [B, Hkv, Lmax, hd]; q_pos [B, T] positions of the queries; kv_len [B]
    number of positions holding keys (rows >= kv_len of a linear cache are
    never read; a ring cache, ``ring``, holds the last Lmax of them).
    Query head h reads kv head h // (H / Hkv).  Returns float64 [B, T, H, hd].
    """
    q = np.asarray(q, dtype=np.float64)
    B, T, H, hd = q.shape
    g = H // n_kv_heads
    out = np.zeros((B, T, H, hd), dtype=np.float64)
    q_pos = np.asarray(q_pos, dtype=np.int64)
    cap = cache_k.shape[2]
    for b in range(B):
        L = int(kv_len[b])
        if ring:
            check_ring_covers(q_pos[b], L, cap, layer_type, window)
        j, rows = key_rows(L, cap, ring)
        vis = visible(q_pos[b][:, None], j[None, :], layer_type, window)   # [T, keys]
        for h in range(H):
            kvh = h // g
            K = np.asarray(cache_k[b, kvh, rows], dtype=np.float64)
            V = np.asarray(cache_v[b, kvh, rows], dtype=np.float64)
            S = (q[b, :, h, :] @ K.T) * scale
            S = np.where(vis, S, -np.inf)
            m = np.max(S, axis=1, keepdims=True)
            P = np.exp(S - m)
            P = P / np.sum(P, axis=1, keepdims=True)
            out[b, :, h, :] = P @ V
    return out


def attention_rows(q, cache_k, cache_v, rows, q_pos, kv_len, n_kv_heads, layer_type, window, scale=1.0,
                   ring=False):
    """The same definition evaluated one output row at a time.

    rows: iterable of (b, t, h).  Returns float64 [len(rows), hd].  Used where
    the full output is too large for the CPU (sampled parity at full sizes).
    """
    q = np.asarray(q)
    H = q.shape[2]
    g = H // n_kv_heads
    cap = cache_k.shape[2]
    res = []
    for (b, t, h) in rows:
        L = int(kv_len[b])
        kvh = h // g
        if ring:
            check_ring_covers(q_pos[b, t], L, cap, layer_type, window)
        j, crow = key_rows(L, cap, ring)
        K = np.asarray(cache_k[b, kvh, crow], dtype=np.float64)
        V = np.asarray(cache_v[b, kvh, crow], dtype=np.float64)
        p = attention_probs(q[b, t, h], K, j, int(q_pos[b, t]), layer_type, window, scale)
        res.append(p @ V)
    return np.stack(res) if res else np.zeros((0, q.shape[-1]))


def visible_bidirectional(q_pos, k_pos, layer_type, window):
    """Key at k_pos is visible from a query at q_pos in the encoder form:
    every key on a global layer, |q - k| <= window on a sliding one
    (taconite-embeddinggemma2 ``text_attention``: keys lo..hi-1 with
    lo = i - win saturating at 0 and hi = min(i + win + 1, n); win is the
    sliding window, or n where the window cuts nothing off)."""
    q_pos = np.asarray(q_pos)
    k_pos = np.asarray(k_pos)
    vis = np.ones(np.broadcast(q_pos, k_pos).shape, dtype=bool)
    if layer_type == SLIDING:
        vis = np.abs(q_pos - k_pos) <= window
    return vis


def attention_bidirectional(q, cache_k, cache_v, T, n_kv_heads, layer_type, window, scale=1.0):
    """Encoder attention over one sequence of T tokens per batch entry.

    q [B, T, H, hd] (normed and roped at positions 0..T-1); the keys and
    values of the same tokens in cache rows [0, T) of cache_k / cache_v
    [B, Hkv, Lmax, hd].  o[b, i, h] = sum_j softmax_j(scale * q . k_j) v_j
    over the keys ``visible_bidirectional`` admits; head h reads kv head
    h // (H / Hkv).  Returns float64 [B, T, H, hd].
    """
    q = np.asarray(q, dtype=np.float64)
    B, Tq, H, hd = q.shape
    assert Tq == T
    g = H // n_kv_heads
    out = np.zeros((B, T, H, hd), dtype=np.float64)
    i = np.arange(T)
    vis = visible_bidirectional(i[:, None], i[None, :], layer_type, window)   # [T, T]
    for b in range(B):
        for h in range(H):
            kvh = h // g
            K = np.asarray(cache_k[b, kvh, :T], dtype=np.float64)
            V = np.asarray(cache_v[b, kvh, :T], dtype=np.float64)
            S = (q[b, :, h, :] @ K.T) * scale
            S = np.where(vis, S, -np.inf)
            m = np.max(S, axis=1, keepdims=True)
            P = np.exp(S - m)
            P = P / np.sum(P, axis=1, keepdims=True)
            out[b, :, h, :] = P @ V
    return out


# --------------------------------------------------------------------------
# Before and after the path: projections, post-attention norm, residual
# --------------------------------------------------------------------------

def qkv_projection(x, attn_norm_w, wq, wk, wv, eps):
    """Raw q / k / v of one layer from its input hidden state.

    x [..., D]; attn_norm_w [D]; wq [H*hd, D]; wk, wv [Hkv*hd, D] (None on a
    shared-KV layer, which projects q only).  xn = rms_norm(x, attn_norm_w)
    and q = wq xn, k = wk xn, v = wv xn (a row of W per output, as the pages'
    ``matvec`` / ``linear`` take it).  Returns (q, k, v), k and v None on a
    shared layer; the caller splits the last axis into heads.
    """
    xn = rms_norm(x, attn_norm_w, eps)
    q = xn @ np.asarray(wq, dtype=np.float64).T
    k = None if wk is None else xn @ np.asarray(wk, dtype=np.float64).T
    v = None if wv is None else xn @ np.asarray(wv, dtype=np.float64).T
    return q, k, v


def attn_output_residual(h, ao, wo, post_norm_w, eps):
    """h + rms_norm(wo ao, post_norm_w): the attention output [..., H*hd]
    projected back to the model width by wo [D, H*hd], normed with the
    post-attention weight [D] and added to the residual stream h [..., D]."""
    a = np.asarray(ao, dtype=np.float64) @ np.asarray(wo, dtype=np.float64).T
    return np.asarray(h, dtype=np.float64) + rms_norm(a, post_norm_w, eps)


# --------------------------------------------------------------------------
# a7: shared-KV routing
# --------------------------------------------------------------------------

def kv_share_src(n_layers, n_shared, is_sliding, layer):
    """Source layer of a shared-KV tail layer, or -1 for a layer that owns one.

    The last ``n_shared`` layers own no cache; a sliding one reads layer
    first_shared - 2 and a full one first_shared - 1
    (ferrox-models ``Gemma4Hparams::kv_reuse_layer``:
    ``n_layer_kv_from_start - if swa {2} else {1}``).
    """
    first_shared = n_layers - n_shared
    if layer < first_shared:
        return -1
    return first_shared - (2 if is_sliding[layer] else 1)


# --------------------------------------------------------------------------
# A whole attention-only stack (append then attention, layer by layer)
# --------------------------------------------------------------------------

def run_stack_prefill(layers, inputs, B, T, Lmax, q_start=0):
    """Prefill of an attention-only stack.

    layers: list of dicts (layer_type, head_dim, n_heads, n_kv_heads, window,
            theta, rotary_fraction, eps, attn_scale, kv_share_src, dtype).
    inputs: list of dicts per layer with q [B,T,H,hd], k, v (None if shared),
            q_norm_w, k_norm_w (None if shared); float64 arrays.
    Each layer is independent (no hidden state flows between layers); a
    shared layer reads its source layer's cache.
    Returns (outputs per layer as stored, caches per layer).
    """
    caches = [None] * len(layers)
    outs = []
    positions = np.broadcast_to(q_start + np.arange(T)[None, :], (B, T))
    for li, (lp, x) in enumerate(zip(layers, inputs)):
        hd, nkv = lp["head_dim"], lp["n_kv_heads"]
        if lp["kv_share_src"] < 0:
            caches[li] = (np.zeros((B, nkv, Lmax, hd)), np.zeros((B, nkv, Lmax, hd)))
            ck, cv = caches[li]
        else:
            ck = cv = None
        q_out = kv_append_normrope(lp, x["q"], x.get("k"), x.get("v"), x["q_norm_w"], x.get("k_norm_w"),
                                   positions, ck, cv)
        src = li if lp["kv_share_src"] < 0 else lp["kv_share_src"]
        sk, sv = caches[src]
        o = attention(q_out, sk, sv, positions, np.full(B, q_start + T), nkv, lp["layer_type"],
                      lp["window"], lp.get("attn_scale", 1.0))
        outs.append(store(o, lp["dtype"]))
    return outs, caches

"""Seeded synthetic workloads: shapes, seeds and value distributions only.

This module holds none of the attention arithmetic.  Both the CUDA path (via
the tests and the benchmark) and the float64 oracle are fed from here; neither
side generates its own inputs.

The five workloads are the ones the attention path is specified on:

* ``tiny_fp32_stack``  -- batch 1, prefill T=64, 4 layers, fp32.  Layer types are
  run as [S, F, S, F] with the last two shared (S reads 0, F reads 1); the
  literal [S, S, S, F] would route the full tail layer to a sliding source of
  another head width, which the same-type rule forbids.
* ``prefill_bf16``     -- batch 1, T=2048, one sliding and one full layer.
* ``decode_bf16``      -- batch 64, one new token each, KV lengths U[1024, 8192].
* ``stack42_bf16``     -- 42 layers (5 sliding : 1 full, last 18 shared), batch 8,
  prefill T=4096 then 128 decode steps.
* ``longctx_decode_bf16`` -- batch 4, KV length 131072 on the full layer plus a
  sliding layer.

``stack42_bf16_dec8`` is ``stack42_bf16`` with 8 decode steps, for launch lists
taken under a profiler; ``stack42_bf16_b2`` is the stack at batch 2, the small
case for counter captures.

Values: q/k/v and cache contents ~ N(0, 1); norm weights ~ 1 + 0.1 N(0, 1)
(float32).  bf16 workloads round the float32 draws to bf16 (torch's RNE cast).
"""

from __future__ import annotations

import torch

SLIDING, FULL = 0, 1
F32, BF16 = 0, 1

SLIDING_GEOM_BF16 = dict(head_dim=256, theta=1e4, rotary_fraction=1.0, window=512)
FULL_GEOM_BF16 = dict(head_dim=512, theta=1e6, rotary_fraction=0.25, window=0)

CONFIGS = {
    "tiny_fp32_stack": dict(
        B=1, T=64, H=4, Hkv=2, dtype=F32, seed=0,
        types=[SLIDING, FULL, SLIDING, FULL], n_shared=2,
        geom={SLIDING: dict(head_dim=64, theta=1e4, rotary_fraction=1.0, window=16),
              FULL: dict(head_dim=128, theta=1e6, rotary_fraction=0.25, window=0)}),
    "prefill_bf16": dict(
        B=1, T=2048, H=8, Hkv=2, dtype=BF16, seed=1,
        types=[SLIDING, FULL], n_shared=0,
        geom={SLIDING: SLIDING_GEOM_BF16, FULL: FULL_GEOM_BF16}),
    "decode_bf16": dict(
        B=64, L_lo=1024, L_hi=8192, H=8, Hkv=2, dtype=BF16, seed=2,
        types=[SLIDING, FULL], n_shared=0,
        geom={SLIDING: SLIDING_GEOM_BF16, FULL: FULL_GEOM_BF16}),
    "stack42_bf16": dict(
        B=8, T=4096, decode_steps=128, H=8, Hkv=2, dtype=BF16, seed=3,
        types=[FULL if (i + 1) % 6 == 0 else SLIDING for i in range(42)], n_shared=18,
        geom={SLIDING: SLIDING_GEOM_BF16, FULL: FULL_GEOM_BF16}),
    # The same 42-layer stack with an 8-step decode phase, for launch lists
    # under a profiler: every decode step launches the same kernels, so the
    # 128-step figures are the decode launches' times x 16.
    "stack42_bf16_dec8": dict(
        B=8, T=4096, decode_steps=8, H=8, Hkv=2, dtype=BF16, seed=3,
        types=[FULL if (i + 1) % 6 == 0 else SLIDING for i in range(42)], n_shared=18,
        geom={SLIDING: SLIDING_GEOM_BF16, FULL: FULL_GEOM_BF16}),
    # The stack at batch 2 with a 2-step decode phase: the small case that
    # counter captures under a profiler run on (about 2.5 GB on the device);
    # per-launch figures scale to batch 8 by the sequences processed.
    "stack42_bf16_b2": dict(
        B=2, T=4096, decode_steps=2, H=8, Hkv=2, dtype=BF16, seed=3,
        types=[FULL if (i + 1) % 6 == 0 else SLIDING for i in range(42)], n_shared=18,
        geom={SLIDING: SLIDING_GEOM_BF16, FULL: FULL_GEOM_BF16}),
    # decode_bf16 with the sliding layer's cache as a ring of one window
    # (512 rows instead of the longest length): same keys read per step
    "ring_decode_bf16": dict(
        B=64, L_lo=1024, L_hi=8192, H=8, Hkv=2, dtype=BF16, seed=2, ring=True,
        types=[SLIDING, FULL], n_shared=0,
        geom={SLIDING: SLIDING_GEOM_BF16, FULL: FULL_GEOM_BF16}),
    # bidirectional (encoder) attention over T tokens, both layer types; the
    # encoder page ropes every pair on both (rotary fraction 1.0)
    "encoder_bf16": dict(
        B=4, T=2048, H=8, Hkv=2, dtype=BF16, seed=5, encoder=True,
        types=[SLIDING, FULL], n_shared=0,
        geom={SLIDING: SLIDING_GEOM_BF16, FULL: dict(FULL_GEOM_BF16, rotary_fraction=1.0)}),
    # The steps around the path at the stack's prefill shape (8 sequences of
    # 4096 tokens), on a sliding and a full layer: the q / k / v projections
    # fused into the append (model width D = 2048: the pages print no hidden
    # size; 2048 is n_heads x the sliding head_dim), and o_proj with the
    # post-attention norm and the residual.
    "qkv_proj_bf16": dict(
        B=8, T=4096, D=2048, H=8, Hkv=2, dtype=BF16, seed=6, proj="qkv",
        types=[SLIDING, FULL], n_shared=0,
        geom={SLIDING: SLIDING_GEOM_BF16, FULL: FULL_GEOM_BF16}),
    "out_proj_bf16": dict(
        B=8, T=4096, D=2048, H=8, Hkv=2, dtype=BF16, seed=7, proj="out",
        types=[SLIDING, FULL], n_shared=0,
        geom={SLIDING: SLIDING_GEOM_BF16, FULL: FULL_GEOM_BF16}),
    "longctx_decode_bf16": dict(
        B=4, L=131072, H=8, Hkv=2, dtype=BF16, seed=4,
        types=[FULL, SLIDING], n_shared=0,
        geom={SLIDING: SLIDING_GEOM_BF16, FULL: FULL_GEOM_BF16}),
}

EPS = 1e-6
ATTN_SCALE = 1.0


def torch_dtype(dtype):
    return torch.bfloat16 if dtype == BF16 else torch.float32


def layer_geometry(cfg, layer):
    """Per-layer hyperparameters of a workload (type, head width, theta, ...)."""
    lt = cfg["types"][layer]
    g = cfg["geom"][lt]
    return dict(layer_type=lt, head_dim=g["head_dim"], n_heads=cfg["H"], n_kv_heads=cfg["Hkv"],
                window=g["window"], theta=g["theta"], rotary_fraction=g["rotary_fraction"],
                eps=EPS, attn_scale=ATTN_SCALE, dtype=cfg["dtype"])


def seed_for(base, layer, tensor, step=0):
    """Distinct, reproducible seed per (workload, layer, tensor, decode step)."""
    return ((base * 1_000_003 + layer) * 131 + tensor) * 10_007 + step


def normal(shape, seed, dtype, device="cpu"):
    """N(0,1) draws from a seeded torch generator on ``device``, cast to dtype."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return x.to(torch_dtype(dtype)) if dtype in (F32, BF16) else x.to(dtype)


def norm_weight(head_dim, seed):
    """Norm weight 1 + 0.1 N(0,1), float32, on the CPU."""
    g = torch.Generator()
    g.manual_seed(seed)
    return 1.0 + 0.1 * torch.randn(head_dim, generator=g, dtype=torch.float32)


def lengths(B, lo, hi, seed):
    """KV lengths uniform over the integers [lo, hi]."""
    g = torch.Generator()
    g.manual_seed(seed)
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int32)


def layer_inputs(cfg, layer, T, owns_cache, device="cpu", step=0, B=None):
    """Raw q/k/v of one layer for T tokens, and its norm weights.

    Returns dict(q [B,T,H,hd], k / v [B,T,Hkv,hd] (absent on a shared layer),
    q_norm_w [hd] f32, k_norm_w [hd] f32 (absent on a shared layer)).
    """
    geo = layer_geometry(cfg, layer)
    hd, H, Hkv, dt = geo["head_dim"], cfg["H"], cfg["Hkv"], cfg["dtype"]
    B = cfg["B"] if B is None else B
    s = cfg["seed"]
    out = dict(q=normal((B, T, H, hd), seed_for(s, layer, 0, step), dt, device),
               q_norm_w=norm_weight(hd, seed_for(s, layer, 3)))
    if owns_cache:
        out["k"] = normal((B, T, Hkv, hd), seed_for(s, layer, 1, step), dt, device)
        out["v"] = normal((B, T, Hkv, hd), seed_for(s, layer, 2, step), dt, device)
        out["k_norm_w"] = norm_weight(hd, seed_for(s, layer, 4))
    return out


def projection_inputs(cfg, layer, device="cpu"):
    """Inputs of the projection workloads: the layer input x [B*T][D] (qkv) or
    the attention output [B*T][H*hd] and residual h [B*T][D] (out), bf16 N(0,1);
    weights N(0,1)/sqrt(fan-in) rounded to bf16; norm weights 1 + 0.1 N(0,1)
    (the attention-norm weight folded into the q/k/v rows in float32, then
    rounded to bf16 once)."""
    geo = layer_geometry(cfg, layer)
    hd, H, Hkv, D = geo["head_dim"], cfg["H"], cfg["Hkv"], cfg["D"]
    M = cfg["B"] * cfg["T"]
    s = cfg["seed"]
    if cfg["proj"] == "qkv":
        N = (H + 2 * Hkv) * hd
        w = normal((N, D), seed_for(s, layer, 11), F32, device) / D ** 0.5
        a = norm_weight(D, seed_for(s, layer, 12)).to(device)
        return dict(x=normal((M, D), seed_for(s, layer, 10), BF16, device), w=(w * a[None, :]).to(torch.bfloat16),
                    q_norm_w=norm_weight(hd, seed_for(s, layer, 3)).to(device),
                    k_norm_w=norm_weight(hd, seed_for(s, layer, 4)).to(device))
    K = H * hd
    return dict(ao=normal((M, K), seed_for(s, layer, 13), BF16, device),
                w=(normal((D, K), seed_for(s, layer, 14), F32, device) / K ** 0.5).to(torch.bfloat16),
                post_w=norm_weight(D, seed_for(s, layer, 15)).to(device),
                h=normal((M, D), seed_for(s, layer, 16), BF16, device))


def cache_rows(cfg, layer, Lmax):
    """Rows of a layer's cache: Lmax, or one window for a sliding layer of a
    workload whose sliding caches are rings."""
    geo = layer_geometry(cfg, layer)
    if cfg.get("ring") and geo["layer_type"] == SLIDING:
        return geo["window"]
    return Lmax


def prefilled_cache(cfg, layer, Lmax, device="cpu", B=None):
    """A KV cache whose rows already hold N(0,1) values (decode workloads)."""
    geo = layer_geometry(cfg, layer)
    hd, Hkv, dt = geo["head_dim"], cfg["Hkv"], cfg["dtype"]
    B = cfg["B"] if B is None else B
    s = cfg["seed"]
    k = normal((B, Hkv, Lmax, hd), seed_for(s, layer, 5), dt, device)
    v = normal((B, Hkv, Lmax, hd), seed_for(s, layer, 6), dt, device)
    return k, v

"""Host-side driver of an attention-only layer stack over the C ABI.

Owns the device buffers of a stack (one KV cache per layer that owns one,
q_out scratch per head width, decode workspaces) and sequences the per-layer
calls: g4_kv_append_normrope then g4_attn_prefill / g4_attn_decode (or
g4_attn_encoder).  Sliding caches may be rings of one window.  Shared-KV
tail layers get no cache and read their source layer's
(cortiq-engine g4e.rs `g4e_forward`: `src = kv_share_src.unwrap_or(li)`).
Every step runs in the CUDA kernels; this module only allocates and calls.
"""

from __future__ import annotations

import torch

from . import g4attn as G
from . import workloads as W


class AttnStack:
    def __init__(self, cfg, Lmax, device="cuda", B=None):
        self.cfg = cfg
        self.B = cfg["B"] if B is None else B
        self.Lmax = Lmax
        self.device = torch.device(device)
        self.n = len(cfg["types"])
        is_s = [t == W.SLIDING for t in cfg["types"]]
        self.src = [G.g4_kv_share_src(self.n, cfg["n_shared"], is_s, l) for l in range(self.n)]
        if any(s == -2 for s in self.src):
            raise ValueError("invalid shared-KV routing for this stack")
        self.geo = [W.layer_geometry(cfg, l) for l in range(self.n)]
        self.params = [G.layer_params(g["layer_type"], g["head_dim"], g["n_heads"], g["n_kv_heads"], g["window"],
                                      g["theta"], g["rotary_fraction"], g["eps"], g["attn_scale"], self.src[l],
                                      g["dtype"]) for l, g in enumerate(self.geo)]
        self.table = G.cache_table(self.n)
        self.caches = {}
        tdt = W.torch_dtype(cfg["dtype"])
        for l, g in enumerate(self.geo):
            if self.src[l] < 0:
                # a ring (sliding layers of a ring workload) holds one window
                rows = W.cache_rows(cfg, l, Lmax)
                shape = (self.B, cfg["Hkv"], rows, g["head_dim"])
                k = torch.zeros(shape, dtype=tdt, device=self.device)
                v = torch.zeros(shape, dtype=tdt, device=self.device)
                self.caches[l] = (k, v)
                G.set_cache(self.table, l, k, v, g["layer_type"], g["head_dim"], cfg["Hkv"], rows, self.B,
                            cfg["dtype"], ring=bool(cfg.get("ring")) and g["layer_type"] == W.SLIDING)
        self.ws = {}
        for l, p in enumerate(self.params):
            nb = G.g4_attn_decode_workspace_size(p, self.B, Lmax)
            self.ws[l] = (torch.zeros(max(nb, 16), dtype=torch.uint8, device=self.device), nb)

    def owns(self, l):
        return self.src[l] < 0

    def cache_bytes(self):
        return sum(k.numel() * k.element_size() * 2 for k, _ in self.caches.values())

    def append(self, l, q, k, v, qw, kw, positions, T, q_out, stream=None):
        G.g4_kv_append_normrope(self.params[l], self.table, l, q, k, v, qw, kw, positions, self.B, T, q_out,
                                stream=stream)

    def prefill_attn(self, l, q_out, q_start, T, out, stream=None):
        G.g4_attn_prefill(self.params[l], self.table, l, q_out, q_start, self.B, T, out, stream=stream)

    def encoder_attn(self, l, q_out, T, out, stream=None):
        """Bidirectional attention over the T tokens appended at positions 0..T-1."""
        G.g4_attn_encoder(self.params[l], self.table, l, q_out, self.B, T, out, stream=stream)

    def decode_attn(self, l, q_out, seq_lens, max_seq_len, out, stream=None):
        ws, nb = self.ws[l]
        G.g4_attn_decode(self.params[l], self.table, l, q_out, seq_lens, self.B, max_seq_len, out, ws, nb,
                         stream=stream)

    def decode_step(self, l, q, k, v, qw, kw, seq_lens, max_seq_len, out, stream=None):
        """Fused append of the new token + decode attention (one launch)."""
        ws, nb = self.ws[l]
        G.g4_decode_step(self.params[l], self.table, l, q, k, v, qw, kw, seq_lens, self.B, max_seq_len, out, ws, nb,
                         stream=stream)

    def decode_launches(self, l):
        """Kernels one g4_attn_decode or g4_decode_step call launches."""
        return 1

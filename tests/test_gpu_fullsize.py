"""Parity at the full workload sizes, in the launch configuration bench.py times.

The CUDA side runs bench.py's own job objects (the same buffers, call order,
split plans and, for the stack, the captured decode graph).  The oracle side
regenerates every input from the seeded generators (on the device the job
drew them on, since torch's CPU and CUDA generators differ), copies it to the
host and recomputes the norm,
RoPE and cache rows from the raw projections itself:
  * single-layer prefill (B=1, T=2048): every output row of both layers;
  * decode (B=64, lengths 1024..8192): every (sequence, head) of both layers;
  * long-context decode (B=4, L=131072): every (sequence, head) of both layers;
  * the 42-layer stack (B=8, T=4096, then 128 decode steps): sampled prefill
    rows (first, last, both sides of the window edge, random) and every head
    of the last decode step, on owning, source and shared layers of both
    types, for the first and last sequence.
"""

import numpy as np
import pytest
import torch

import bench
from gemma_dual_geometry_gb300 import build as g4build
from gemma_dual_geometry_gb300 import g4attn as G
from gemma_dual_geometry_gb300 import workloads as W
from oracle import g4_oracle as O

from gpu_common import assert_attn_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    g4build.build()
    G.lib()
    yield
    assert G.g4_take_device_error() == 0


def _oracle_kv(geo, k, v, kw, positions):
    """Stored cache rows for raw k, v [T, Hkv, hd] at positions [T] (oracle)."""
    kn, vn = O.normrope_kv(k, v, kw, positions, geo["head_dim"], geo["theta"], geo["rotary_fraction"], geo["eps"])
    return O.store(kn, geo["dtype"]), O.store(vn, geo["dtype"])


def _oracle_q(geo, q, qw, positions):
    """Stored normed + roped queries for raw q [T, H, hd] at positions [T] (oracle)."""
    return O.store(O.normrope_q(q, qw, positions, geo["head_dim"], geo["theta"], geo["rotary_fraction"],
                                geo["eps"]), geo["dtype"])


def _row(geo, q_row, K, V, q_pos):
    p = O.attention_probs(q_row, K, np.arange(K.shape[0]), q_pos, geo["layer_type"], geo["window"],
                          geo["attn_scale"])
    return p @ V


def test_prefill_single_layer_full_size():
    cfg = W.CONFIGS["prefill_bf16"]
    job = bench.LayerJob(cfg, torch.device("cuda"))
    job.step()
    torch.cuda.synchronize()
    T, Hkv = cfg["T"], cfg["Hkv"]
    pos = np.arange(T)
    for l in range(job.n):
        geo = job.st.geo[l]
        x = W.layer_inputs(cfg, l, T, True, device="cuda")   # regenerated (same generator and device)
        kc, vc = _oracle_kv(geo, f64(x["k"][0]), f64(x["v"][0]), f64(x["k_norm_w"]), pos)
        qn = _oracle_q(geo, f64(x["q"][0]), f64(x["q_norm_w"]), pos)
        ck = np.transpose(kc, (1, 0, 2))[None]
        cv = np.transpose(vc, (1, 0, 2))[None]
        ref = O.attention(qn[None], ck, cv, pos[None, :], [T], Hkv, geo["layer_type"], geo["window"])
        assert_attn_close(f64(job.out[l]), ref, W.BF16, f"prefill layer {l}")


def _check_decode_job(cfg):
    job = bench.LayerJob(cfg, torch.device("cuda"))
    job.step()
    torch.cuda.synchronize()
    B, H, Hkv = cfg["B"], cfg["H"], cfg["Hkv"]
    g = H // Hkv
    for l in range(job.n):
        geo = job.st.geo[l]
        x = W.layer_inputs(cfg, l, 1, True, device="cuda")
        pk, pv = W.prefilled_cache(cfg, l, job.Lmax, device="cuda")   # the rows the job started from
        qw, kw = f64(x["q_norm_w"]), f64(x["k_norm_w"])
        out = f64(job.out[l])[:, 0]                                 # [B, H, hd]
        got, ref = [], []
        for b in range(B):
            L = job.L[b]
            qn = _oracle_q(geo, f64(x["q"][b]), qw, np.array([L - 1]))[0]       # [H, hd]
            kn, vn = _oracle_kv(geo, f64(x["k"][b]), f64(x["v"][b]), kw, np.array([L - 1]))
            for kvh in range(Hkv):
                K = f64(pk[b, kvh, :L])
                V = f64(pv[b, kvh, :L])
                K[L - 1] = kn[0, kvh]
                V[L - 1] = vn[0, kvh]
                for h in range(kvh * g, (kvh + 1) * g):
                    ref.append(_row(geo, qn[h], K, V, L - 1))
                    got.append(out[b, h])
        del pk, pv
        assert_attn_close(np.stack(got), np.stack(ref), W.BF16, f"{cfg['types']} decode layer {l}")


def test_decode_full_size():
    _check_decode_job(W.CONFIGS["decode_bf16"])


def test_long_context_decode_full_size():
    _check_decode_job(W.CONFIGS["longctx_decode_bf16"])


def test_stack_full_size_sampled_rows():
    cfg = W.CONFIGS["stack42_bf16"]
    job = bench.Job(cfg, torch.device("cuda"))
    B, T, H, Hkv, S = cfg["B"], cfg["T"], cfg["H"], cfg["Hkv"], cfg["decode_steps"]
    g = H // Hkv
    L = T + S
    # owning S and F, the two sources (22 S, 23 F), shared S and F, the last of each width
    layers = [0, 5, 22, 23, 24, 29, 40, 41]
    assert [job.st.src[l] for l in layers] == [-1, -1, -1, -1, 22, 23, 22, 23]
    # prefill in bench.py's order, keeping the sampled layers' outputs
    pf = {}
    for l in range(job.n):
        x, hd = job.X[l], job.st.geo[l]["head_dim"]
        job.st.append(l, x["q"], x.get("k"), x.get("v"), x["q_norm_w"], x.get("k_norm_w"), job.pos_pf, T,
                      job.qo[hd])
        job.st.prefill_attn(l, job.qo[hd], job.qs, T, job.out[hd])
        if l in layers:
            pf[l] = job.out[hd].cpu()
    # the 128 x 42 decode steps as bench.py times them (one CUDA graph), then
    # the last step once more, eagerly, keeping each sampled layer's output
    job.capture_decode()
    job.graph.replay()
    torch.cuda.synchronize()
    graph_last = {hd: t.clone() for hd, t in job.out_dec.items()}
    dec = {}
    s = S - 1
    for l in range(job.n):
        d, hd = job.D[l], job.st.geo[l]["head_dim"]
        job.st.decode_step(l, d["q"][s].view(B, H, hd), d["k"][s].view(B, Hkv, hd) if "k" in d else None,
                           d["v"][s].view(B, Hkv, hd) if "v" in d else None, job.X[l]["q_norm_w"],
                           job.X[l].get("k_norm_w"), job.sl_dec[s], job.Lmax, job.out_dec[hd])
        if l in layers:
            dec[l] = job.out_dec[hd].cpu()
    torch.cuda.synchronize()
    for hd, t in graph_last.items():
        last = max(l for l in range(job.n) if job.st.geo[l]["head_dim"] == hd)
        assert torch.equal(t.cpu(), dec[last]), f"graph replay vs eager last step, head_dim {hd}"

    rng = np.random.default_rng(11)
    for l in layers:
        geo = job.st.geo[l]
        src = job.st.src[l] if job.st.src[l] >= 0 else l
        gsrc = job.st.geo[src]
        xs = W.layer_inputs(cfg, src, T, True, device="cuda")   # regenerated (same generator and device)
        xl = W.layer_inputs(cfg, l, T, False, device="cuda")
        ds = {k: W.normal((S, B, 1, Hkv, gsrc["head_dim"]), W.seed_for(cfg["seed"], src, t), cfg["dtype"], "cuda")
              for k, t in (("k", 8), ("v", 9))}
        dq = W.normal((S, B, 1, H, geo["head_dim"]), W.seed_for(cfg["seed"], l, 7), cfg["dtype"], "cuda")
        kw, qw = f64(xs["k_norm_w"]), f64(xl["q_norm_w"])
        for b in (0, B - 1):
            kc, vc = _oracle_kv(gsrc, f64(xs["k"][b]), f64(xs["v"][b]), kw, np.arange(T))
            kd, vd = _oracle_kv(gsrc, f64(ds["k"][:, b, 0]), f64(ds["v"][:, b, 0]), kw, T + np.arange(S))
            K = np.concatenate([kc, kd])                       # [L, Hkv, hd]
            V = np.concatenate([vc, vd])
            qn = _oracle_q(geo, f64(xl["q"][b]), qw, np.arange(T))
            ts = sorted({0, 1, 511, 512, 513, T - 1, *rng.integers(0, T, 3).tolist()})
            hs = sorted({0, H - 1, int(rng.integers(0, H))})
            got = np.stack([f64(pf[l][b, t, h]) for t in ts for h in hs])
            ref = np.stack([_row(geo, qn[t, h], K[:t + 1, h // g], V[:t + 1, h // g], t) for t in ts for h in hs])
            assert_attn_close(got, ref, W.BF16, f"stack prefill layer {l} seq {b}")
            qd = _oracle_q(geo, f64(dq[s, b]), qw, np.array([L - 1]))[0]
            refd = np.stack([_row(geo, qd[h], K[:, h // g], V[:, h // g], L - 1) for h in range(H)])
            assert_attn_close(f64(dec[l][b]), refd, W.BF16, f"stack decode layer {l} seq {b}")

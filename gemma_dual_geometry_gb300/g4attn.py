"""ctypes binding of libg4attn.so (declared in include/g4attn.h).

Argument marshalling only: every step of the attention path runs in the CUDA
kernels behind the C ABI.  Tensor arguments may be torch tensors (their
``data_ptr()`` is passed) or raw integer device addresses.  The functions
keep the C names; a non-OK status raises ``G4Error`` with the library's
message.  There is no fallback: if the library is not built, ``lib()``
raises.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libg4attn.so")

G4_OK, G4_ERR_INVALID_ARG, G4_ERR_UNSUPPORTED, G4_ERR_SHARE_MISMATCH = 0, 1, 2, 3
G4_ERR_CAPACITY, G4_ERR_WORKSPACE, G4_ERR_CUDA = 4, 5, 6
G4_SLIDING, G4_FULL = 0, 1
G4_F32, G4_BF16 = 0, 1

STATUS_NAMES = {0: "G4_OK", 1: "G4_ERR_INVALID_ARG", 2: "G4_ERR_UNSUPPORTED", 3: "G4_ERR_SHARE_MISMATCH",
                4: "G4_ERR_CAPACITY", 5: "G4_ERR_WORKSPACE", 6: "G4_ERR_CUDA"}

_c_void_p = ctypes.c_void_p
_i32 = ctypes.c_int32


class G4LayerParams(ctypes.Structure):
    _fields_ = [("layer_type", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("window", ctypes.c_int32), ("theta", ctypes.c_float),
                ("rotary_fraction", ctypes.c_float), ("eps", ctypes.c_float), ("attn_scale", ctypes.c_float),
                ("kv_share_src", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class G4KVCache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("layer_type", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("max_len", ctypes.c_int32),
                ("batch", ctypes.c_int32), ("dtype", ctypes.c_int32), ("ring", ctypes.c_int32)]


_P = ctypes.POINTER
# Every function include/g4attn.h declares, with its ctypes signature.
SIGNATURES = {
    "g4_kv_share_src": (_i32, [_i32, _i32, _P(_i32), _i32]),
    "g4_kv_append_normrope": (_i32, [_P(G4LayerParams), _P(G4KVCache), _i32, _i32, _c_void_p, _c_void_p, _c_void_p,
                                     _c_void_p, _c_void_p, _c_void_p, _i32, _i32, _c_void_p, _c_void_p]),
    "g4_attn_prefill": (_i32, [_P(G4LayerParams), _P(G4KVCache), _i32, _i32, _c_void_p, _c_void_p, _i32, _i32,
                               _c_void_p, _c_void_p]),
    "g4_attn_encoder": (_i32, [_P(G4LayerParams), _P(G4KVCache), _i32, _i32, _c_void_p, _i32, _i32, _c_void_p,
                               _c_void_p]),
    "g4_attn_decode_workspace_size": (ctypes.c_size_t, [_P(G4LayerParams), _i32, _i32]),
    "g4_attn_decode": (_i32, [_P(G4LayerParams), _P(G4KVCache), _i32, _i32, _c_void_p, _c_void_p, _i32, _i32,
                              _c_void_p, _c_void_p, ctypes.c_size_t, _c_void_p]),
    "g4_decode_step": (_i32, [_P(G4LayerParams), _P(G4KVCache), _i32, _i32, _c_void_p, _c_void_p, _c_void_p,
                              _c_void_p, _c_void_p, _c_void_p, _i32, _i32, _c_void_p, _c_void_p, ctypes.c_size_t,
                              _c_void_p]),
    "g4_attn_decode_noalloc": (_i32, [_P(G4LayerParams), _P(G4KVCache), _i32, _i32, _c_void_p, _c_void_p, _i32,
                                      _i32, _c_void_p, _c_void_p]),
    "g4_qkv_project_append": (_i32, [_P(G4LayerParams), _P(G4KVCache), _i32, _i32, _c_void_p, _i32, _c_void_p,
                                     _c_void_p, _c_void_p, _c_void_p, _i32, _i32, _c_void_p, _c_void_p]),
    "g4_attn_out_residual": (_i32, [_c_void_p, _i32, _i32, _c_void_p, _i32, _c_void_p, ctypes.c_float, _c_void_p,
                                    _c_void_p, _c_void_p]),
    "g4_last_error": (ctypes.c_char_p, []),
    "g4_take_device_error": (_i32, []),
}

_lib = None


class G4Error(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with python -m gemma_dual_geometry_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream, *tensors):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    for t in tensors:
        if t is not None and not isinstance(t, int) and t.is_cuda:
            import torch
            return torch.cuda.current_stream(t.device).cuda_stream
    return None


def _check(status):
    if status != G4_OK:
        raise G4Error(status, lib().g4_last_error().decode())


def layer_params(layer_type, head_dim, n_heads, n_kv_heads, window=0, theta=1e4, rotary_fraction=1.0, eps=1e-6,
                 attn_scale=1.0, kv_share_src=-1, dtype=G4_BF16):
    return G4LayerParams(int(layer_type), int(head_dim), int(n_heads), int(n_kv_heads), int(window), float(theta),
                         float(rotary_fraction), float(eps), float(attn_scale), int(kv_share_src), int(dtype))


def cache_table(n_layers):
    """Zeroed array of n_layers g4_kv_cache entries."""
    return (G4KVCache * n_layers)()


def set_cache(table, layer, k, v, layer_type, head_dim, n_kv_heads, max_len, batch, dtype, ring=False):
    """Fill entry ``layer``; ``ring`` makes it a sliding-window ring of max_len rows."""
    table[layer] = G4KVCache(_ptr(k), _ptr(v), int(layer_type), int(head_dim), int(n_kv_heads), int(max_len),
                             int(batch), int(dtype), int(bool(ring)))


def g4_kv_share_src(n_layers, n_shared, is_sliding, layer):
    arr = (ctypes.c_int32 * n_layers)(*[1 if s else 0 for s in is_sliding])
    return lib().g4_kv_share_src(n_layers, n_shared, arr, layer)


def g4_kv_append_normrope(params, caches, layer, q_in, k_in, v_in, q_norm_w, k_norm_w, positions, B, T, q_out,
                          stream=None):
    _check(lib().g4_kv_append_normrope(ctypes.byref(params), caches, len(caches), layer, _ptr(q_in), _ptr(k_in),
                                       _ptr(v_in), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(positions), B, T,
                                       _ptr(q_out), _stream(stream, q_in)))


def g4_attn_prefill(params, caches, layer, q, q_start_pos, B, T, out, stream=None):
    _check(lib().g4_attn_prefill(ctypes.byref(params), caches, len(caches), layer, _ptr(q), _ptr(q_start_pos), B, T,
                                 _ptr(out), _stream(stream, q)))


def g4_attn_encoder(params, caches, layer, q, B, T, out, stream=None):
    _check(lib().g4_attn_encoder(ctypes.byref(params), caches, len(caches), layer, _ptr(q), B, T, _ptr(out),
                                 _stream(stream, q)))


def g4_attn_decode_workspace_size(params, B, max_seq_len):
    return int(lib().g4_attn_decode_workspace_size(ctypes.byref(params), B, max_seq_len))


def g4_attn_decode(params, caches, layer, q, seq_lens, B, max_seq_len, out, workspace=None, workspace_bytes=0,
                   stream=None):
    _check(lib().g4_attn_decode(ctypes.byref(params), caches, len(caches), layer, _ptr(q), _ptr(seq_lens), B,
                                max_seq_len, _ptr(out), _ptr(workspace), int(workspace_bytes), _stream(stream, q)))


def g4_decode_step(params, caches, layer, q_in, k_in, v_in, q_norm_w, k_norm_w, seq_lens, B, max_seq_len, out,
                   workspace=None, workspace_bytes=0, stream=None):
    _check(lib().g4_decode_step(ctypes.byref(params), caches, len(caches), layer, _ptr(q_in), _ptr(k_in), _ptr(v_in),
                                _ptr(q_norm_w), _ptr(k_norm_w), _ptr(seq_lens), B, max_seq_len, _ptr(out),
                                _ptr(workspace), int(workspace_bytes), _stream(stream, q_in)))


G4_NOALLOC_SCRATCH_BYTES = 8 << 20


def g4_attn_decode_noalloc(params, caches, layer, q, seq_lens, B, max_seq_len, out, stream=None):
    """g4_attn_decode with the library's built-in scratch instead of a workspace."""
    _check(lib().g4_attn_decode_noalloc(ctypes.byref(params), caches, len(caches), layer, _ptr(q), _ptr(seq_lens),
                                        B, max_seq_len, _ptr(out), _stream(stream, q)))


def g4_qkv_project_append(params, caches, layer, x, D, w_qkv, q_norm_w, k_norm_w, positions, B, T, q_out,
                          stream=None):
    """q/k/v projections of x (attention-norm weight folded into w_qkv) fused into the norm/RoPE/append."""
    _check(lib().g4_qkv_project_append(ctypes.byref(params), caches, len(caches), layer, _ptr(x), int(D),
                                       _ptr(w_qkv), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(positions), B, T,
                                       _ptr(q_out), _stream(stream, x)))


def g4_attn_out_residual(ao, M, K, w_o, D, post_norm_w, eps, h, out, stream=None):
    """out = h + rmsnorm(ao . w_o^T, post_norm_w, eps)."""
    _check(lib().g4_attn_out_residual(_ptr(ao), int(M), int(K), _ptr(w_o), int(D), _ptr(post_norm_w), float(eps),
                                      _ptr(h), _ptr(out), _stream(stream, ao)))


def g4_last_error():
    return lib().g4_last_error().decode()


def g4_take_device_error():
    return int(lib().g4_take_device_error())

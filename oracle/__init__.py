"""Double-precision CPU oracle for the decoder-step attention path.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg import this package; the CUDA library never
does, and the two share no code.  It wraps ``liboracle.so`` (oracle.c) with
numpy arrays in and out.  Every function returns float64 results computed
from the same f16 bytes the GPU reads.

Parity pins: every function here is pinned by the ``-m "not gpu"`` tests in
tests/test_oracle_pins.py (closed forms, brute force on tiny inputs, numpy's
independent binary16 conversion, invariants such as step == prefill row and
GQA == MHA with duplicated KV heads).  No function is left unpinned.

Layout: a cache row holds 2*Hkv*hd f16 (K of every KV head, then V of every
KV head); caches are C-contiguous ``uint16`` arrays whose leading axis is the
sequence (or source) axis.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None

_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64 = ctypes.c_int64
_int = ctypes.c_int
_dbl = ctypes.c_double


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        sig = {
            "orc_set_threads": (_int, [_int]),
            "orc_get_threads": (_int, []),
            "orc_f16_to_f64": (_dbl, [ctypes.c_uint16]),
            "orc_f64_to_f16": (ctypes.c_uint16, [_dbl]),
            "orc_f32_to_f16": (ctypes.c_uint16, [ctypes.c_float]),
            "orc_f16_decode_array": (None, [_u16p, _f64p, _i64]),
            "orc_f32_encode_array": (None, [_f32p, _u16p, _i64]),
            "orc_f64_encode_array": (None, [_f64p, _u16p, _i64]),
            "orc_attend_one": (None, [_f64p, _u16p, _u16p, _i64, _int, _int, _dbl, _f64p, _f64p]),
            "orc_kv_append": (_int, [_f32p, _f32p, _i64, _u16p, _i64, _i32p, _int, _int, _int, _int]),
            "orc_self_attn_step": (_int, [_f32p, _i64, _u16p, _i64, _i32p, _int, _int, _int, _int,
                                          _dbl, _f64p]),
            "orc_cross_attn_step": (_int, [_f32p, _i64, _u16p, _i64, _i32p, _int, _int, _int, _int,
                                           _int, _dbl, _f64p]),
            "orc_rmsnorm": (None, [_f64p, _f64p, _dbl, _int, _f64p]),
            "orc_rope_neox": (None, [_f64p, _int, _dbl, _dbl, _f64p]),
            "orc_gqa_step": (_int, [_f32p, _f32p, _f32p, _f32p, _f32p, _dbl, _dbl, _i32p, _u16p,
                                    _i64, _int, _int, _int, _int, _int, _dbl, _f64p]),
            "orc_kv_rearrange": (_int, [_u16p, _u16p, _i64, _i64, _int, _int, _int, _i32p, _i32p,
                                        _i32p, _int]),
            "orc_prefill_attn": (_int, [_u16p, _u16p, _u16p, _f32p, _f32p, _dbl, _dbl, _int, _int,
                                        _int, _int, _int, _dbl, _u16p, _i64, _int, _f64p, _u16p]),
            "orc_prefill_prep": (_int, [_u16p, _u16p, _u16p, _f32p, _f32p, _dbl, _dbl, _int, _int,
                                        _int, _int, _int, _u16p, _i64, _int, _u16p]),
            "orc_prefill_attn_rows": (None, [_u16p, _i32p, _int, _u16p, _int, _int, _int, _int,
                                             _dbl, _f64p]),
            "orc_mha_attn": (_int, [_u16p, _u16p, _u16p, _i32p, _int, _int, _int, _int, _dbl, _int,
                                    _u16p, _i64, _int, _f64p]),
            "orc_cross_kv_fill": (None, [_u16p, _u16p, _f32p, _int, _int, _int, _u16p, _i64]),
            "orc_layer_norm": (None, [_f32p, _i64, _f32p, _f32p, _dbl, _f64p]),
            "orc_gelu_erf": (_dbl, [_dbl]),
            "orc_silu": (_dbl, [_dbl]),
            "orc_linear": (None, [_f32p, _i64, _int, _int, _int, _f32p, _f32p, _dbl, _int, _u16p,
                                  _int, _f32p, _int, _f64p, _i64]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _p(a, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def _c(a, dtype):
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    if not a.flags.c_contiguous:
        raise ValueError("array must be C-contiguous")
    return a


def set_threads(n):
    """Number of host threads the attention loops may use (independent items)."""
    return _lib().orc_set_threads(int(n))


def get_threads():
    return _lib().orc_get_threads()


# ---------------------------------------------------------------- binary16 --

def f16_to_f64(bits):
    """binary16 bit patterns (uint16) -> exact float64 values."""
    bits = _c(np.ascontiguousarray(bits), np.uint16)
    out = np.empty(bits.shape, np.float64)
    _lib().orc_f16_decode_array(_p(bits, ctypes.c_uint16), _p(out, ctypes.c_double), bits.size)
    return out


def f32_to_f16(x):
    """float32 -> binary16 bits, IEEE round to nearest even, overflow to inf."""
    x = _c(np.ascontiguousarray(x), np.float32)
    out = np.empty(x.shape, np.uint16)
    _lib().orc_f32_encode_array(_p(x, ctypes.c_float), _p(out, ctypes.c_uint16), x.size)
    return out


def f64_to_f16(x):
    """float64 -> binary16 bits, one IEEE round to nearest even."""
    x = _c(np.ascontiguousarray(x), np.float64)
    out = np.empty(x.shape, np.uint16)
    _lib().orc_f64_encode_array(_p(x, ctypes.c_double), _p(out, ctypes.c_uint16), x.size)
    return out


# ------------------------------------------------------------- primitives --

def attend_one(q, k_rows, v_rows, scale):
    """softmax(scale * k_rows @ q) @ v_rows with k/v given as f16 [L, hd] rows."""
    q = np.ascontiguousarray(q, np.float64)
    k_rows = _c(np.ascontiguousarray(k_rows), np.uint16)
    v_rows = _c(np.ascontiguousarray(v_rows), np.uint16)
    L, hd = k_rows.shape
    both = np.concatenate([k_rows, v_rows], axis=1)  # one row = K then V
    z = np.empty(max(L, 1), np.float64)
    out = np.empty(hd, np.float64)
    _lib().orc_attend_one(_p(q, ctypes.c_double), _p(both, ctypes.c_uint16),
                          both[:, hd:].ctypes.data_as(_u16p), 2 * hd, L, hd, float(scale),
                          _p(z, ctypes.c_double), _p(out, ctypes.c_double))
    return out


def rmsnorm(x, w, eps):
    x = np.ascontiguousarray(x, np.float64)
    w = np.ascontiguousarray(w, np.float64)
    y = np.empty_like(x)
    _lib().orc_rmsnorm(_p(x, ctypes.c_double), _p(w, ctypes.c_double), float(eps), x.size,
                       _p(y, ctypes.c_double))
    return y


def rope_neox(x, pos, base):
    x = np.ascontiguousarray(x, np.float64)
    y = np.empty_like(x)
    _lib().orc_rope_neox(_p(x, ctypes.c_double), x.size, float(pos), float(base),
                         _p(y, ctypes.c_double))
    return y


# -------------------------------------------------------------- the steps --

def kv_append(k, v, cache, slot, kv_heads, head_dim, src_row_stride=None):
    """Write f16(k_b) || f16(v_b) into row slot[b] of cache[b] (in place).

    k, v: float32 [B, >=Hkv*hd] row-strided views (for example the k and v
    columns of [q|k|v] rows; row stride in floats = src_row_stride, default
    the view's own); cache: uint16 [B, capacity, row].
    Returns the number of sequences skipped for an out-of-range slot."""
    k = np.asarray(k)
    v = np.asarray(v)
    if k.dtype != np.float32 or v.dtype != np.float32:
        raise TypeError("k and v must be float32")
    if k.ndim != 2 or k.strides[1] != 4 or v.strides != k.strides:
        raise ValueError("k and v must be row-strided 2-D views with unit inner stride")
    cache = _c(cache, np.uint16)
    slot = _c(np.ascontiguousarray(slot, np.int32), np.int32)
    B, cap = cache.shape[0], cache.shape[1]
    stride = src_row_stride if src_row_stride is not None else k.strides[0] // 4
    return _lib().orc_kv_append(_p(k, ctypes.c_float), _p(v, ctypes.c_float), stride,
                                _p(cache, ctypes.c_uint16), cache[0].size, _p(slot, ctypes.c_int32),
                                B, kv_heads, head_dim, cap)


def self_attn_step(q, cache, lens, heads, head_dim, scale, q_stride=None):
    """Causal one-token self-attention; q float32 [B, >=H*hd], cache uint16
    [B, capacity, 2*H*hd], lens int32 [B] (keys incl. the new one).
    Returns (out float64 [B, H*hd], n_skipped)."""
    q = _c(q, np.float32)
    cache = _c(cache, np.uint16)
    lens = _c(np.ascontiguousarray(lens, np.int32), np.int32)
    B, cap = cache.shape[0], cache.shape[1]
    out = np.empty((B, heads * head_dim), np.float64)
    qs = q_stride if q_stride is not None else q.shape[-1]
    n = _lib().orc_self_attn_step(_p(q, ctypes.c_float), qs, _p(cache, ctypes.c_uint16),
                                  cache[0].size, _p(lens, ctypes.c_int32), B, heads, head_dim, cap,
                                  float(scale), _p(out, ctypes.c_double))
    return out, n


def cross_attn_step(q, cross, group, heads, head_dim, scale, q_stride=None):
    """Unmasked one-token cross-attention; cross uint16 [G, frames, 2*H*hd],
    group int32 [B] (source of each sequence).  Returns (out, n_skipped)."""
    q = _c(q, np.float32)
    cross = _c(cross, np.uint16)
    group = _c(np.ascontiguousarray(group, np.int32), np.int32)
    G, frames = cross.shape[0], cross.shape[1]
    B = group.shape[0]
    out = np.empty((B, heads * head_dim), np.float64)
    qs = q_stride if q_stride is not None else q.shape[-1]
    n = _lib().orc_cross_attn_step(_p(q, ctypes.c_float), qs, _p(cross, ctypes.c_uint16),
                                   cross[0].size, _p(group, ctypes.c_int32), B, G, heads, head_dim,
                                   frames, float(scale), _p(out, ctypes.c_double))
    return out, n


def gqa_step(q, k_new, v_new, q_norm_w, k_norm_w, eps, rope_base, n_past, cache, q_heads,
             kv_heads, head_dim, scale):
    """Fused RMSNorm + NeoX RoPE + append + GQA attention step (cache updated
    in place).  Returns (out float64 [B, Hq*hd], n_skipped)."""
    q = _c(q, np.float32)
    k_new = _c(k_new, np.float32)
    v_new = _c(v_new, np.float32)
    wq = _c(np.ascontiguousarray(q_norm_w, np.float32), np.float32)
    wk = _c(np.ascontiguousarray(k_norm_w, np.float32), np.float32)
    n_past = _c(np.ascontiguousarray(n_past, np.int32), np.int32)
    cache = _c(cache, np.uint16)
    B, cap = cache.shape[0], cache.shape[1]
    out = np.empty((B, q_heads * head_dim), np.float64)
    n = _lib().orc_gqa_step(_p(q, ctypes.c_float), _p(k_new, ctypes.c_float),
                            _p(v_new, ctypes.c_float), _p(wq, ctypes.c_float),
                            _p(wk, ctypes.c_float), float(eps), float(rope_base),
                            _p(n_past, ctypes.c_int32), _p(cache, ctypes.c_uint16), cache[0].size,
                            cap, B, q_heads, kv_heads, head_dim, float(scale),
                            _p(out, ctypes.c_double))
    return out, n


def kv_rearrange(src, dst, idx, lens_src, capacity):
    """Beam reorder.  src/dst uint16 [B, n_layers, capacity, row] (dst updated
    in place).  Returns (lens_dst int32 [B], n_skipped)."""
    src = _c(src, np.uint16)
    dst = _c(dst, np.uint16)
    idx = _c(np.ascontiguousarray(idx, np.int32), np.int32)
    lens_src = _c(np.ascontiguousarray(lens_src, np.int32), np.int32)
    B, n_layers, cap, row = src.shape
    lens_dst = np.zeros(B, np.int32)
    n = _lib().orc_kv_rearrange(_p(src, ctypes.c_uint16), _p(dst, ctypes.c_uint16), src[0].size,
                                src[0, 0].size, n_layers, row, capacity,
                                _p(idx, ctypes.c_int32), _p(lens_src, ctypes.c_int32),
                                _p(lens_dst, ctypes.c_int32), B)
    return lens_dst, n


def prefill_attn(q, k, v, q_norm_w, k_norm_w, eps, rope_base, q_heads, kv_heads, head_dim, scale,
                 cache):
    """Batched causal prefill.  q uint16 [B, T, Hq*hd], k/v uint16 [B, T, Hkv*hd];
    cache uint16 [B, capacity, 2*Hkv*hd] (rows [0,T) written in place).
    Returns (out float64 [B, T, Hq*hd], qhat uint16 [B, T, Hq*hd])."""
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    wq = _c(np.ascontiguousarray(q_norm_w, np.float32), np.float32)
    wk = _c(np.ascontiguousarray(k_norm_w, np.float32), np.float32)
    cache = _c(cache, np.uint16)
    B, T = q.shape[0], q.shape[1]
    cap = cache.shape[1]
    out = np.empty((B, T, q_heads * head_dim), np.float64)
    qhat = np.empty((B, T, q_heads * head_dim), np.uint16)
    rc = _lib().orc_prefill_attn(_p(q, ctypes.c_uint16), _p(k, ctypes.c_uint16),
                                 _p(v, ctypes.c_uint16), _p(wq, ctypes.c_float),
                                 _p(wk, ctypes.c_float), float(eps), float(rope_base), B, T,
                                 q_heads, kv_heads, head_dim, float(scale),
                                 _p(cache, ctypes.c_uint16), cache[0].size, cap,
                                 _p(out, ctypes.c_double), _p(qhat, ctypes.c_uint16))
    if rc != 0:
        raise ValueError("T exceeds the cache capacity")
    return out, qhat


def prefill_prep(q, k, v, q_norm_w, k_norm_w, eps, rope_base, q_heads, kv_heads, head_dim,
                 cache):
    """Prefill preparation only: cache rows [0,T) written in place (normed and
    roped K, V copied); returns qhat uint16 [B, T, Hq*hd]."""
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    wq = _c(np.ascontiguousarray(q_norm_w, np.float32), np.float32)
    wk = _c(np.ascontiguousarray(k_norm_w, np.float32), np.float32)
    cache = _c(cache, np.uint16)
    B, T = q.shape[0], q.shape[1]
    qhat = np.empty((B, T, q_heads * head_dim), np.uint16)
    rc = _lib().orc_prefill_prep(_p(q, ctypes.c_uint16), _p(k, ctypes.c_uint16),
                                 _p(v, ctypes.c_uint16), _p(wq, ctypes.c_float),
                                 _p(wk, ctypes.c_float), float(eps), float(rope_base), B, T,
                                 q_heads, kv_heads, head_dim, _p(cache, ctypes.c_uint16),
                                 cache[0].size, cache.shape[1], _p(qhat, ctypes.c_uint16))
    if rc != 0:
        raise ValueError("T exceeds the cache capacity")
    return qhat


def prefill_attn_rows(qhat_rows, t_of_row, seq_cache, q_heads, kv_heads, head_dim, head, scale):
    """Causal attention for selected query rows of one (sequence, head):
    qhat_rows uint16 [n, hd] (normed+roped f16 queries), t_of_row int32 [n],
    seq_cache uint16 [capacity, row] of that sequence.  Returns float64 [n, hd]."""
    qhat_rows = _c(np.ascontiguousarray(qhat_rows), np.uint16)
    t_of_row = _c(np.ascontiguousarray(t_of_row, np.int32), np.int32)
    seq_cache = _c(np.ascontiguousarray(seq_cache), np.uint16)
    n = t_of_row.shape[0]
    out = np.empty((n, head_dim), np.float64)
    _lib().orc_prefill_attn_rows(_p(qhat_rows, ctypes.c_uint16), _p(t_of_row, ctypes.c_int32), n,
                                 _p(seq_cache, ctypes.c_uint16), q_heads, kv_heads, head_dim, head,
                                 float(scale), _p(out, ctypes.c_double))
    return out


def mha_attn(q, k, v, heads, head_dim, scale, causal, lens=None, cache=None):
    """Multi-head attention of each sequence's positions among themselves
    (causal: the prompt prefill; unmasked: the encoder's self-attention).
    q, k, v uint16 [B, T, heads*hd]; lens int32 [B] or None (all T); cache
    uint16 [B, capacity, 2*heads*hd] or None (rows [0, lens[b]) get k || v in
    place).  Returns (out float64 [B, T, heads*hd] with rows past lens[b]
    left as NaN, number of sequences skipped for a bad length)."""
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    B, T = q.shape[0], q.shape[1]
    out = np.full((B, T, heads * head_dim), np.nan, np.float64)
    lp = None
    if lens is not None:
        lens = _c(np.ascontiguousarray(lens, np.int32), np.int32)
        lp = _p(lens, ctypes.c_int32)
    cp, cstride, cap = None, 0, 0
    if cache is not None:
        cache = _c(cache, np.uint16)
        cp, cstride, cap = _p(cache, ctypes.c_uint16), cache[0].size, cache.shape[1]
    n = _lib().orc_mha_attn(_p(q, ctypes.c_uint16), _p(k, ctypes.c_uint16), _p(v, ctypes.c_uint16),
                            lp, B, T, heads, head_dim, float(scale), 1 if causal else 0, cp,
                            cstride, cap, _p(out, ctypes.c_double))
    if n < 0:
        raise ValueError("T exceeds the cache capacity")
    return out, n


def cross_kv_fill(enc, w, bias_v, cross):
    """Cross K/V of one layer from the encoder output: enc uint16 [G, frames, d],
    w uint16 [2d, d], bias_v float32 [d]; cross uint16 [G, frames_cap, 2d] is
    written in place (rows [0, frames))."""
    enc = _c(enc, np.uint16)
    w = _c(w, np.uint16)
    bias_v = _c(np.ascontiguousarray(bias_v, np.float32), np.float32)
    cross = _c(cross, np.uint16)
    G, frames, d = enc.shape
    _lib().orc_cross_kv_fill(_p(enc, ctypes.c_uint16), _p(w, ctypes.c_uint16),
                             _p(bias_v, ctypes.c_float), G, frames, d,
                             _p(cross, ctypes.c_uint16), cross[0].size)


# ------------------------------------------- the dense steps of a layer --

LINEAR_MODES = {"store": 0, "residual": 1, "gelu": 2}


def layer_norm(x, g, b, eps=1e-5):
    """LayerNorm of each row of x (float32 [M, K]) with weight g and bias b
    (float32 [K]); float64 [M, K]."""
    x = _c(np.ascontiguousarray(x, np.float32), np.float32)
    g = _c(np.ascontiguousarray(g, np.float32), np.float32)
    b = _c(np.ascontiguousarray(b, np.float32), np.float32)
    x2 = x.reshape(-1, x.shape[-1])
    out = np.empty(x2.shape, np.float64)
    for m in range(x2.shape[0]):
        _lib().orc_layer_norm(_p(x2[m], ctypes.c_float), x2.shape[1], _p(g, ctypes.c_float),
                              _p(b, ctypes.c_float), float(eps), _p(out[m], ctypes.c_double))
    return out.reshape(x.shape)


def gelu_erf(v):
    """GELU, error-function form, elementwise on float64 values."""
    v = np.asarray(v, np.float64)
    f = _lib().orc_gelu_erf
    return np.vectorize(lambda t: f(float(t)), otypes=[np.float64])(v)


def silu(v):
    """SiLU v * sigmoid(v), elementwise on float64 values."""
    v = np.asarray(v, np.float64)
    f = _lib().orc_silu
    return np.vectorize(lambda t: f(float(t)), otypes=[np.float64])(v)


def linear(x, w, bias=None, mode="store", ln=None, eps=1e-5, y=None, rms=None, swiglu=False):
    """One dense step: a = LayerNorm(x) (ln = (g, b)), RMSNorm(x) (rms = g),
    silu(x[:, :K]) * x[:, K:] (swiglu) or x; v = a W^T + bias;
    mode "store" -> v, "residual" -> y + v, "gelu" -> gelu(v).

    x: float32 [M, K] ([M, 2K] with swiglu); w: uint16 (f16 bits) [N, K];
    bias: float32 [N] or None; y: the values the residual is added onto
    ([M, N]).  Returns float64 [M, N]."""
    x = _c(np.ascontiguousarray(x, np.float32), np.float32)
    w = _c(w, np.uint16)
    M = x.shape[0]
    N, K = w.shape
    if x.shape[1] != (2 * K if swiglu else K):
        raise ValueError("x must be [M, K] ([M, 2K] with swiglu) for w [N, K]")
    if sum(t is not None for t in (ln, rms)) + bool(swiglu) > 1:
        raise ValueError("one of ln, rms, swiglu at most")
    m = LINEAR_MODES[mode]
    out = np.zeros((M, N), np.float64)
    if m == 1:
        if y is None:
            raise ValueError("residual mode needs y")
        out[:] = np.asarray(y, np.float64)
    bp = None
    if bias is not None:
        bias = _c(np.ascontiguousarray(bias, np.float32), np.float32)
        bp = _p(bias, ctypes.c_float)
    gp = bq = None
    norm = 0
    if ln is not None:
        norm = 1
        g = _c(np.ascontiguousarray(ln[0], np.float32), np.float32)
        b = _c(np.ascontiguousarray(ln[1], np.float32), np.float32)
        gp, bq = _p(g, ctypes.c_float), _p(b, ctypes.c_float)
    elif rms is not None:
        norm = 2
        g = _c(np.ascontiguousarray(rms, np.float32), np.float32)
        gp = _p(g, ctypes.c_float)
    _lib().orc_linear(_p(x, ctypes.c_float), x.shape[1], M, K, norm, gp, bq, float(eps),
                      1 if swiglu else 0, _p(w, ctypes.c_uint16), N, bp, m,
                      _p(out, ctypes.c_double), N)
    return out


def whisper_decoder_layer_step(x, p, cache, lens, cross, group, heads, head_dim, eps=1e-5):
    """One Whisper decoder layer for one new token per sequence, in the order
    of "wavo 0.1.0, src/whisper/decoder.rs", Decoder::record_step:

      qkv = LN_self(x) W_qkv^T + b_qkv;  k, v -> cache row lens-1;
      x  += attend(q, own cache, lens) W_o^T + b_o;
      qx  = LN_cross(x) W_cq^T + b_cq;   x += attend(qx, cross) W_co^T + b_co;
      x  += gelu(LN_ffn(x) W_1^T + b_1) W_2^T + b_2.

    Each step computes in double; its result is stored as float32, as the
    pages' buffers (x, qkv, att, h) are f32, and the cache row as f16.
    x: float32 [B, d]; p: the layer's parameters (keys ln1_g, ln1_b, w_qkv,
    b_qkv, w_o, b_o, ln2_g, ln2_b, w_cq, b_cq, w_co, b_co, ln3_g, ln3_b,
    w_fc1, b_fc1, w_fc2, b_fc2; weights uint16 f16 bits [out, in], the rest
    float32); cache: uint16 [B, capacity, 2d] (row lens-1 written in place);
    lens: int32 [B] keys incl. the new token; cross: uint16 [G, frames, 2d];
    group: int32 [B].  Returns (x_out float32 [B, d], intermediates)."""
    d = heads * head_dim
    scale = head_dim ** -0.5
    f32 = np.float32
    x = np.ascontiguousarray(x, f32)
    lens = np.ascontiguousarray(lens, np.int32)
    qkv = linear(x, p["w_qkv"], p["b_qkv"], ln=(p["ln1_g"], p["ln1_b"]), eps=eps).astype(f32)
    kv_append(qkv[:, d:2 * d], qkv[:, 2 * d:], cache, lens - 1, heads, head_dim)
    att, _ = self_attn_step(qkv, cache, lens, heads, head_dim, scale, q_stride=3 * d)
    att = att.astype(f32)
    x1 = linear(att, p["w_o"], p["b_o"], mode="residual", y=x).astype(f32)
    qx = linear(x1, p["w_cq"], p["b_cq"], ln=(p["ln2_g"], p["ln2_b"]), eps=eps).astype(f32)
    attc, _ = cross_attn_step(qx, cross, group, heads, head_dim, scale)
    attc = attc.astype(f32)
    x2 = linear(attc, p["w_co"], p["b_co"], mode="residual", y=x1).astype(f32)
    h = linear(x2, p["w_fc1"], p["b_fc1"], mode="gelu", ln=(p["ln3_g"], p["ln3_b"]),
               eps=eps).astype(f32)
    x3 = linear(h, p["w_fc2"], p["b_fc2"], mode="residual", y=x2).astype(f32)
    return x3, {"qkv": qkv, "att": att, "x1": x1, "qx": qx, "attc": attc, "x2": x2, "h": h}


def qwen3_decoder_layer_step(x, p, cache, n_past, q_heads, kv_heads, head_dim, eps=1e-6,
                             rope_base=1e6):
    """One Qwen3-ASR decoder layer for one new token per sequence
    ("transcribe.cpp, src/arch/qwen3_asr/decoder.h", header comment and
    StepBuildBatched): pre-norm RMSNorm (eps 1e-6), the q/k/v projections,
    the GQA step (per-head Q/K RMSNorm, NeoX RoPE at base 1e6, K/V written at
    row n_past, attention over rows [0, n_past]), the output projection onto
    the residual, then RMSNorm and the SwiGLU MLP down(silu(gate(x)) * up(x))
    onto the residual.  No projection has a bias.

    Each step computes in double and stores its result as float32 (the
    buffers between steps are f32), the cache row as f16.  x: float32 [B, d];
    p: w_qkv [(Hq + 2 Hkv) hd, d] (q rows, then k, then v), w_o [d, Hq hd],
    w_gu [2 I, d] (gate rows, then up rows), w_down [d, I] (f16 bits),
    rms1, rms2 float32 [d], q_norm, k_norm float32 [hd]; cache: uint16
    [B, capacity, 2 Hkv hd] (row n_past written in place); n_past: int32 [B].
    Returns (x_out float32 [B, d], intermediates)."""
    f32 = np.float32
    x = np.ascontiguousarray(x, f32)
    nq, nk = q_heads * head_dim, kv_heads * head_dim
    qkv = linear(x, p["w_qkv"], None, rms=p["rms1"], eps=eps).astype(f32)
    q = np.ascontiguousarray(qkv[:, :nq])
    k = np.ascontiguousarray(qkv[:, nq:nq + nk])
    v = np.ascontiguousarray(qkv[:, nq + nk:])
    att, _ = gqa_step(q, k, v, p["q_norm"], p["k_norm"], eps, rope_base, n_past, cache, q_heads,
                      kv_heads, head_dim, head_dim ** -0.5)
    att = att.astype(f32)
    x1 = linear(att, p["w_o"], None, mode="residual", y=x).astype(f32)
    gu = linear(x1, p["w_gu"], None, rms=p["rms2"], eps=eps).astype(f32)
    x2 = linear(gu, p["w_down"], None, mode="residual", y=x1, swiglu=True).astype(f32)
    return x2, {"qkv": qkv, "att": att, "x1": x1, "gu": gu}


def build():
    """Compile liboracle.so (the checker) if it is missing or stale."""
    return _build.build()


__all__ = [
    "set_threads", "get_threads", "f16_to_f64", "f32_to_f16", "f64_to_f16", "attend_one",
    "rmsnorm", "rope_neox", "kv_append", "self_attn_step", "cross_attn_step", "gqa_step",
    "kv_rearrange", "prefill_prep", "prefill_attn", "prefill_attn_rows", "mha_attn", "cross_kv_fill",
    "layer_norm", "gelu_erf", "silu", "linear", "whisper_decoder_layer_step",
    "qwen3_decoder_layer_step", "build",
]

if os.environ.get("ORACLE_THREADS"):
    set_threads(int(os.environ["ORACLE_THREADS"]))

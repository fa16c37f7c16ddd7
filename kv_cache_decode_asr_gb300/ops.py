"""ctypes binding of libasrkv.so: the C entry points under the same names.

Each function takes torch tensors (device memory owned by the caller),
checks dtype/device/contiguity, and passes raw pointers, sizes and the
current CUDA stream to the C ABI.  All arithmetic happens in the library's
kernels; this module only marshals arguments.  A non-zero status raises
AsrError.  If libasrkv.so has not been built, every call raises: there is no
CPU fallback.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libasrkv.so")

ASR_OK = 0
STATUS = {0: "ASR_OK", 1: "ASR_ERR_INVALID_ARG", 2: "ASR_ERR_UNSUPPORTED",
          3: "ASR_ERR_MISALIGNED", 4: "ASR_ERR_ALIAS", 5: "ASR_ERR_WORKSPACE", 6: "ASR_ERR_CUDA",
          7: "ASR_ERR_SCRATCH_LIMIT"}
DEVERR_LEN, DEVERR_INDEX, DEVERR_BEAMS, DEVERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8
OP_SELF_ATTN, OP_CROSS_ATTN, OP_GQA_STEP, OP_PREFILL_ATTN = 1, 2, 3, 4
OP_MHA_PREFILL, OP_ENCODER_ATTN = 5, 6

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t

SIGNATURES = {
    "asr_kv_append": (_int, [_p, _p, _i64, _p, _i64, _p, _int, _int, _int, _int, _p, _p]),
    "asr_self_attn_step": (_int, [_p, _i64, _p, _i64, _p, _int, _int, _int, _int, _f, _p, _p, _sz,
                                  _p, _p]),
    "asr_self_attn_append_step": (_int, [_p, _i64, _p, _p, _i64, _p, _i64, _p, _int, _int, _int,
                                         _int, _f, _p, _p, _sz, _p, _p]),
    "asr_self_attn_reorder_append_step": (_int, [_p, _i64, _p, _p, _i64, _p, _p, _i64, _p, _p,
                                                 _p, _int, _int, _int, _int, _f, _p, _p, _sz, _p,
                                                 _p]),
    "asr_cross_attn_step": (_int, [_p, _i64, _p, _i64, _p, _int, _int, _int, _int, _int, _int, _f,
                                   _p, _p, _sz, _p, _p]),
    "asr_gqa_step": (_int, [_p, _i64, _p, _p, _i64, _p, _p, _f, _f, _p, _p, _i64, _int, _int, _int,
                            _int, _int,
                            _f, _p, _p, _sz, _p, _p]),
    "asr_kv_rearrange": (_int, [_p, _p, _i64, _i64, _int, _int, _int, _p, _p, _p, _int, _p, _p]),
    "asr_self_attn_step_noalloc": (_int, [_p, _i64, _p, _i64, _p, _int, _int, _int, _int, _f, _p,
                                          _p, _p]),
    "asr_noalloc_scratch_bytes": (_sz, []),
    "asr_prefill_attn": (_int, [_p, _p, _p, _p, _p, _f, _f, _int, _int, _int, _int, _int, _f, _p,
                                _i64, _int, _p, _p, _sz, _p, _p]),
    "asr_prefill_prep": (_int, [_p, _p, _p, _p, _p, _f, _f, _int, _int, _int, _int, _int, _p,
                                _i64, _int, _p, _sz, _p]),
    "asr_prefill_attention": (_int, [_int, _int, _int, _int, _int, _f, _p, _i64, _int, _p, _p,
                                     _sz, _p, _p]),
    "asr_mha_prefill": (_int, [_p, _p, _p, _p, _int, _int, _int, _int, _f, _p, _i64, _int, _p, _p,
                               _sz, _p, _p]),
    "asr_encoder_attn": (_int, [_p, _p, _p, _p, _int, _int, _int, _int, _f, _p, _p, _sz, _p, _p]),
    "asr_cross_kv_fill": (_int, [_p, _p, _p, _int, _int, _int, _p, _i64, _p, _p]),
    "asr_linear": (_int, [_p, _i64, _int, _p, _p, _f, _int, _p, _p, _int, _int, _int, _int, _p,
                          _i64, _p, _sz, _p, _p]),
    "asr_linear_workspace_size": (_sz, [_int, _int, _int]),
    "asr_workspace_size": (_sz, [_int, _int, _int, _int, _int, _int, _int]),
    "asr_status_string": (ctypes.c_char_p, [_int]),
    "asr_version": (_int, []),
    "asr_debug_stall_next_decode": (_int, [ctypes.c_uint64]),
    "asr_set_history_ready": (_int, [_int]),
}

_LIB = None


class AsrError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")


def load():
    """Load libasrkv.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(there is no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, dtype, name):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")


def _check(fn, st):
    if st != ASR_OK:
        raise AsrError(fn, st)


def asr_status_string(status):
    return load().asr_status_string(int(status)).decode()


def asr_version():
    return load().asr_version()


def asr_set_history_ready(ready):
    """Promise (ready=True) that the launch just before each decode-attention
    call of this thread writes none of its lengths, groups, norm weights or
    cached rows, so the call reads them before the grid dependency wait."""
    _check("asr_set_history_ready", load().asr_set_history_ready(1 if ready else 0))


def asr_debug_stall_next_decode(wait_ns):
    """Test support: the next decode-attention launch from this thread issues
    no copies, so its waits run out after wait_ns and it reports
    DEVERR_TIMEOUT (its outputs are undefined)."""
    _check("asr_debug_stall_next_decode", load().asr_debug_stall_next_decode(int(wait_ns)))


def asr_workspace_size(op, B, n_sources, max_beams, q_heads, head_dim, T=0):
    return load().asr_workspace_size(op, B, n_sources, max_beams, q_heads, head_dim, T)


def workspace(op, B, n_sources, max_beams, q_heads, head_dim, T=0, device=None):
    """A zero-filled, 256-byte-aligned workspace tensor for one entry point."""
    import torch
    n = asr_workspace_size(op, B, n_sources, max_beams, q_heads, head_dim, T)
    if n == 0:
        raise AsrError("asr_workspace_size", 1)
    return torch.zeros(n + 256, dtype=torch.uint8, device=device or "cuda")


def _ws_ptr(ws):
    """Pointer into ws rounded up to 256 bytes, and the bytes left."""
    base = ws.data_ptr()
    al = (base + 255) // 256 * 256
    return ctypes.c_void_p(al), ws.numel() - (al - base)


def asr_kv_append(k, v, cache, slot, kv_heads, head_dim, capacity, dev_err=None,
                  src_row_stride=None, stream=None):
    """k, v: f32 [B, >=Hkv*hd] views (row stride src_row_stride); cache: f16
    [B, seq_stride]-strided; slot: int32 [B]."""
    import torch
    _need(k, torch.float32, "k")
    _need(v, torch.float32, "v")
    _need(cache, torch.float16, "cache")
    _need(slot, torch.int32, "slot")
    B = slot.shape[0]
    stride = src_row_stride if src_row_stride is not None else k.stride(0)
    st = load().asr_kv_append(_ptr(k), _ptr(v), stride, _ptr(cache), cache.stride(0), _ptr(slot),
                              B, kv_heads, head_dim, capacity, _ptr(dev_err), _stream(stream))
    _check("asr_kv_append", st)


def asr_self_attn_step(q, cache, lens, heads, head_dim, capacity, scale, out, ws, dev_err=None,
                       stream=None):
    """q: f32 [B, >=H*hd] (row stride q.stride(0)); cache: f16 [B, ...] with
    seq stride cache.stride(0); lens: int32 [B]; out: f32 [B, H*hd]."""
    import torch
    _need(q, torch.float32, "q")
    _need(cache, torch.float16, "cache")
    _need(lens, torch.int32, "lens")
    _need(out, torch.float32, "out")
    B = lens.shape[0]
    wp, wn = _ws_ptr(ws)
    st = load().asr_self_attn_step(_ptr(q), q.stride(0), _ptr(cache), cache.stride(0), _ptr(lens),
                                   B, heads, head_dim, capacity, float(scale), _ptr(out), wp, wn,
                                   _ptr(dev_err), _stream(stream))
    _check("asr_self_attn_step", st)


def asr_self_attn_append_step(q, k_new, v_new, cache, lens, heads, head_dim, capacity, scale,
                              out, ws, dev_err=None, stream=None):
    """Fused append + self-attention.  q, k_new, v_new: f32 [B, >=H*hd] row
    views (k_new and v_new share one row stride); cache: f16, sequence stride
    cache.stride(0); lens: int32 [B]; out: f32 [B, H*hd]."""
    import torch
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (out, "out")):
        _need(t, torch.float32, n)
    _need(cache, torch.float16, "cache")
    _need(lens, torch.int32, "lens")
    if k_new.stride(0) != v_new.stride(0):
        raise ValueError("k_new and v_new must share the row stride")
    B = lens.shape[0]
    wp, wn = _ws_ptr(ws)
    st = load().asr_self_attn_append_step(_ptr(q), q.stride(0), _ptr(k_new), _ptr(v_new),
                                          k_new.stride(0), _ptr(cache), cache.stride(0),
                                          _ptr(lens), B, heads, head_dim, capacity, float(scale),
                                          _ptr(out), wp, wn, _ptr(dev_err), _stream(stream))
    _check("asr_self_attn_append_step", st)


def asr_self_attn_reorder_append_step(q, k_new, v_new, cache_src, cache_dst, idx, lens_src,
                                      lens_dst, heads, head_dim, capacity, scale, out, ws,
                                      dev_err=None, stream=None):
    """Beam reorder + append + self-attention of one layer.  cache_src,
    cache_dst: f16 caches with one sequence stride; idx, lens_src, lens_dst:
    int32 [B]; other arguments as asr_self_attn_append_step."""
    import torch
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (out, "out")):
        _need(t, torch.float32, n)
    _need(cache_src, torch.float16, "cache_src")
    _need(cache_dst, torch.float16, "cache_dst")
    for t, n in ((idx, "idx"), (lens_src, "lens_src"), (lens_dst, "lens_dst")):
        _need(t, torch.int32, n)
    if k_new.stride(0) != v_new.stride(0):
        raise ValueError("k_new and v_new must share the row stride")
    if cache_src.stride(0) != cache_dst.stride(0):
        raise ValueError("cache_src and cache_dst must share the sequence stride")
    B = idx.shape[0]
    wp, wn = _ws_ptr(ws)
    st = load().asr_self_attn_reorder_append_step(
        _ptr(q), q.stride(0), _ptr(k_new), _ptr(v_new), k_new.stride(0), _ptr(cache_src),
        _ptr(cache_dst), cache_src.stride(0), _ptr(idx), _ptr(lens_src), _ptr(lens_dst), B, heads,
        head_dim, capacity, float(scale), _ptr(out), wp, wn, _ptr(dev_err), _stream(stream))
    _check("asr_self_attn_reorder_append_step", st)


def asr_self_attn_step_noalloc(q, cache, lens, heads, head_dim, capacity, scale, out,
                               dev_err=None, stream=None):
    """Self-attention with the library's fixed scratch array instead of a
    workspace (for callers that cannot allocate one); arguments as
    asr_self_attn_step without ws."""
    import torch
    _need(q, torch.float32, "q")
    _need(cache, torch.float16, "cache")
    _need(lens, torch.int32, "lens")
    _need(out, torch.float32, "out")
    B = lens.shape[0]
    st = load().asr_self_attn_step_noalloc(_ptr(q), q.stride(0), _ptr(cache), cache.stride(0),
                                           _ptr(lens), B, heads, head_dim, capacity,
                                           float(scale), _ptr(out), _ptr(dev_err),
                                           _stream(stream))
    _check("asr_self_attn_step_noalloc", st)


def asr_noalloc_scratch_bytes():
    return load().asr_noalloc_scratch_bytes()


def asr_cross_attn_step(q, cross, group, G, max_beams, heads, head_dim, frames, scale, out, ws,
                        dev_err=None, stream=None):
    """q: f32 [B, >=H*hd] (row stride q.stride(0)); cross: f16 [G, >=frames,
    2*H*hd] (group stride cross.stride(0)); group: int32 [B], non-decreasing,
    at most max_beams sequences per group; out: f32 [B, H*hd]."""
    import torch
    _need(q, torch.float32, "q")
    _need(cross, torch.float16, "cross")
    _need(group, torch.int32, "group")
    _need(out, torch.float32, "out")
    B = group.shape[0]
    wp, wn = _ws_ptr(ws)
    st = load().asr_cross_attn_step(_ptr(q), q.stride(0), _ptr(cross), cross.stride(0),
                                    _ptr(group), B, G, max_beams, heads, head_dim, frames,
                                    float(scale), _ptr(out), wp, wn, _ptr(dev_err), _stream(stream))
    _check("asr_cross_attn_step", st)


def asr_gqa_step(q, k_new, v_new, q_norm_w, k_norm_w, eps, rope_base, n_past, cache, capacity,
                 q_heads, kv_heads, head_dim, scale, out, ws, dev_err=None, stream=None):
    """q: f32 [B, >=Hq*hd]; k_new, v_new: f32 [B, >=Hkv*hd] sharing one row
    stride (for instance the thirds of a fused q/k/v projection); q_norm_w,
    k_norm_w: f32 [hd]; n_past: int32 [B]; cache: f16 [B, capacity,
    2*Hkv*hd] (row n_past written); out: f32 [B, Hq*hd]."""
    import torch
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (q_norm_w, "q_norm_w"),
                 (k_norm_w, "k_norm_w"), (out, "out")):
        _need(t, torch.float32, n)
    _need(n_past, torch.int32, "n_past")
    _need(cache, torch.float16, "cache")
    B = n_past.shape[0]
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new")):
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError(f"{n} must be 2-D with unit inner stride")
    if k_new.stride(0) != v_new.stride(0):
        raise ValueError("k_new and v_new must share one row stride")
    wp, wn = _ws_ptr(ws)
    st = load().asr_gqa_step(_ptr(q), q.stride(0), _ptr(k_new), _ptr(v_new), k_new.stride(0),
                             _ptr(q_norm_w), _ptr(k_norm_w),
                             float(eps), float(rope_base), _ptr(n_past), _ptr(cache),
                             cache.stride(0), capacity, B, q_heads, kv_heads, head_dim,
                             float(scale), _ptr(out), wp, wn, _ptr(dev_err), _stream(stream))
    _check("asr_gqa_step", st)


def asr_prefill_attn(q, k, v, q_norm_w, k_norm_w, eps, rope_base, q_heads, kv_heads, head_dim,
                     scale, cache, capacity, out, ws, dev_err=None, stream=None):
    """q: f16 [B, T, Hq*hd]; k, v: f16 [B, T, Hkv*hd]; cache: f16 with sequence
    stride cache.stride(0); out: f32 [B, T, Hq*hd]; ws from
    workspace(OP_PREFILL_ATTN, B, kv_heads, 1, q_heads, head_dim, T)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (cache, "cache")):
        _need(t, torch.float16, n)
    for t, n in ((q_norm_w, "q_norm_w"), (k_norm_w, "k_norm_w"), (out, "out")):
        _need(t, torch.float32, n)
    B, T = q.shape[0], q.shape[1]
    wp, wn = _ws_ptr(ws)
    st = load().asr_prefill_attn(_ptr(q), _ptr(k), _ptr(v), _ptr(q_norm_w), _ptr(k_norm_w),
                                 float(eps), float(rope_base), B, T, q_heads, kv_heads, head_dim,
                                 float(scale), _ptr(cache), cache.stride(0), capacity, _ptr(out),
                                 wp, wn, _ptr(dev_err), _stream(stream))
    _check("asr_prefill_attn", st)


def asr_prefill_prep(q, k, v, q_norm_w, k_norm_w, eps, rope_base, q_heads, kv_heads, head_dim,
                     cache, capacity, ws, stream=None):
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (cache, "cache")):
        _need(t, torch.float16, n)
    B, T = q.shape[0], q.shape[1]
    wp, wn = _ws_ptr(ws)
    st = load().asr_prefill_prep(_ptr(q), _ptr(k), _ptr(v), _ptr(q_norm_w), _ptr(k_norm_w),
                                 float(eps), float(rope_base), B, T, q_heads, kv_heads, head_dim,
                                 _ptr(cache), cache.stride(0), capacity, wp, wn, _stream(stream))
    _check("asr_prefill_prep", st)


def asr_prefill_attention(B, T, q_heads, kv_heads, head_dim, scale, cache, capacity, out, ws,
                          dev_err=None, stream=None):
    import torch
    _need(cache, torch.float16, "cache")
    _need(out, torch.float32, "out")
    wp, wn = _ws_ptr(ws)
    st = load().asr_prefill_attention(B, T, q_heads, kv_heads, head_dim, float(scale), _ptr(cache),
                                      cache.stride(0), capacity, _ptr(out), wp, wn, _ptr(dev_err),
                                      _stream(stream))
    _check("asr_prefill_attention", st)


def asr_mha_prefill(q, k, v, heads, head_dim, scale, cache, capacity, out, ws, lens=None,
                    dev_err=None, stream=None):
    """q, k, v: f16 [B, T, heads*head_dim]; cache: f16 [B, capacity, 2*heads*head_dim];
    out: fp32 [B, T, heads*head_dim]; lens: int32 [B] or None."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (cache, "cache")):
        _need(t, torch.float16, n)
    _need(out, torch.float32, "out")
    if lens is not None:
        _need(lens, torch.int32, "lens")
    B, T = q.shape[0], q.shape[1]
    wp, wn = _ws_ptr(ws)
    st = load().asr_mha_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(lens), B, T, heads, head_dim,
                                float(scale), _ptr(cache), cache.stride(0), capacity, _ptr(out),
                                wp, wn, _ptr(dev_err), _stream(stream))
    _check("asr_mha_prefill", st)


def asr_encoder_attn(q, k, v, heads, head_dim, scale, out, ws, lens=None, dev_err=None,
                     stream=None):
    """q, k, v: f16 [B, T, heads*head_dim]; out: fp32 [B, T, heads*head_dim];
    lens: int32 [B] or None."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.float16, n)
    _need(out, torch.float32, "out")
    if lens is not None:
        _need(lens, torch.int32, "lens")
    B, T = q.shape[0], q.shape[1]
    wp, wn = _ws_ptr(ws)
    st = load().asr_encoder_attn(_ptr(q), _ptr(k), _ptr(v), _ptr(lens), B, T, heads, head_dim,
                                 float(scale), _ptr(out), wp, wn, _ptr(dev_err), _stream(stream))
    _check("asr_encoder_attn", st)


def asr_cross_kv_fill(enc, w, bias_v, cross, frames=None, dev_err=None, stream=None):
    """enc: f16 [G, frames, d]; w: f16 [2d, d]; bias_v: fp32 [d];
    cross: f16 [G, capacity, 2d] (rows [0, frames) written)."""
    import torch
    for t, n in ((enc, "enc"), (w, "w"), (cross, "cross")):
        _need(t, torch.float16, n)
    _need(bias_v, torch.float32, "bias_v")
    G, F, d = enc.shape
    st = load().asr_cross_kv_fill(_ptr(enc), _ptr(w), _ptr(bias_v), G, frames or F, d,
                                  _ptr(cross), cross.stride(0), _ptr(dev_err), _stream(stream))
    _check("asr_cross_kv_fill", st)


LINEAR_MODES = {"store": 0, "residual": 1, "gelu": 2}


def linear_workspace(M, N, K, device=None):
    """A zero-filled workspace for asr_linear on M x K activations and an
    N x K weight (None when the call needs none)."""
    import torch
    n = load().asr_linear_workspace_size(int(M), int(N), int(K))
    if n == 0:
        return None
    return torch.zeros(n + 256, dtype=torch.uint8, device=device or "cuda")


NORM_NONE, NORM_LAYER, NORM_RMS = 0, 1, 2
ACT_NONE, ACT_SWIGLU = 0, 1


def asr_linear(x, w, y, bias=None, ln=None, rms=None, eps=1e-5, swiglu=False, mode="store",
               ws=None, dev_err=None, stream=None):
    """y (fp32 [M, N], row-strided) = epilogue(norm(x) @ w^T + bias).

    x: fp32 [M, K] (row-strided, unit inner stride; [M, 2K] = [gate | up]
    with swiglu=True); w: f16 [N, K]; bias: fp32 [N] or None; ln: (g, b)
    fp32 [K] each for a LayerNorm, or rms: g fp32 [K] for an RMSNorm (at
    most one); mode "store", "residual" (y += ...) or "gelu"."""
    import torch
    _need(x, torch.float32, "x")
    _need(w, torch.float16, "w")
    _need(y, torch.float32, "y")
    if x.dim() != 2 or y.dim() != 2 or x.stride(1) != 1 or y.stride(1) != 1:
        raise ValueError("x and y must be 2-D with unit inner stride")
    if not w.is_contiguous():
        raise ValueError("w must be contiguous")
    M = x.shape[0]
    N, K = w.shape
    if x.shape[1] != (2 * K if swiglu else K) or y.shape[0] != M or y.shape[1] != N:
        raise ValueError("shapes do not match: x [M, K] ([M, 2K] with swiglu), w [N, K], y [M, N]")
    if ln is not None and rms is not None:
        raise ValueError("one norm at most")
    if bias is not None:
        _need(bias, torch.float32, "bias")
    norm, g, b = NORM_NONE, None, None
    if ln is not None:
        norm, (g, b) = NORM_LAYER, ln
        _need(g, torch.float32, "ln_g")
        _need(b, torch.float32, "ln_b")
    elif rms is not None:
        norm, g = NORM_RMS, rms
        _need(g, torch.float32, "rms_g")
    if ws is None:
        wp, wn = None, 0
    else:
        wp, wn = _ws_ptr(ws)
    st = load().asr_linear(_ptr(x), x.stride(0), norm, _ptr(g), _ptr(b), float(eps),
                           ACT_SWIGLU if swiglu else ACT_NONE, _ptr(w), _ptr(bias), M, N, K,
                           LINEAR_MODES[mode], _ptr(y), y.stride(0), wp, wn, _ptr(dev_err),
                           _stream(stream))
    _check("asr_linear", st)


def asr_kv_rearrange(src, dst, idx, lens_src, lens_dst, n_layers, row_elems, capacity,
                     layer_stride=None, dev_err=None, stream=None):
    """src, dst: f16 [B, n_layers, capacity, row] (or strided alike); idx,
    lens_src, lens_dst: int32 [B]."""
    import torch
    _need(src, torch.float16, "src")
    _need(dst, torch.float16, "dst")
    for t, n in ((idx, "idx"), (lens_src, "lens_src"), (lens_dst, "lens_dst")):
        _need(t, torch.int32, n)
    if src.stride(0) != dst.stride(0):
        raise ValueError("src and dst must share the sequence stride")
    B = idx.shape[0]
    ls = layer_stride if layer_stride is not None else (src.stride(1) if src.dim() > 2 else 0)
    st = load().asr_kv_rearrange(_ptr(src), _ptr(dst), src.stride(0), ls, n_layers, row_elems,
                                 capacity, _ptr(idx), _ptr(lens_src), _ptr(lens_dst), B,
                                 _ptr(dev_err), _stream(stream))
    _check("asr_kv_rearrange", st)

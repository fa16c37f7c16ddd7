"""GPU parity of the dense steps of a decoder layer (asr_linear) and of a
whole Whisper decoder layer composed through the C ABI, against the oracle.

Tolerance of asr_linear, from its arithmetic: per output (m, n)

    |gpu - oracle| <= 2^-14 * c * (sum_k |a_mk| |W_nk| + |bias_n|)
                      + 2^-22 * |y_old_mn| + 1e-7

with a the oracle's activation (LayerNorm-ed or not) and c = 1.13 for the
GELU (the largest slope of v * Phi(v)), else 1.  The activation reaches the
tensor cores as two f16 parts (relative error below 2^-21), the fp32
LayerNorm adds a few fp32 ulps, and the fp32 sums (at most a few hundred
accumulation steps per CTA, then one fp32 add per K split) stay far below
2^-14 of the magnitude sum; the residual add rounds once more to fp32.  A
wrong row, column, k offset or operand gives an error of the order of the
magnitude sum / sqrt(K), two orders of magnitude above the bound here.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from kv_cache_decode_asr_gb300 import ops  # noqa: E402
from kv_cache_decode_asr_gb300 import synthetic as syn  # noqa: E402

from gpu_util import (assert_attn_close, dev, host, host_u16, lo_plane_inputs,  # noqa: E402
                      new_err)

GELU_SLOPE = 1.13


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_decode_asr_gb300 import build
    build.build()
    ops.load()
    oracle.build()
    oracle.set_threads(8)


def dec16(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def linear_bound(a, w_bits, bias, mode, y_old=None):
    s = np.abs(a) @ np.abs(dec16(w_bits)).T
    if bias is not None:
        s = s + np.abs(bias.astype(np.float64))
    tol = 2.0 ** -14 * s * (GELU_SLOPE if mode == "gelu" else 1.0) + 1e-7
    if y_old is not None:
        tol = tol + 2.0 ** -22 * np.abs(y_old.astype(np.float64))
    return tol, s


def assert_linear_close(gpu, ref, tol, s, what):
    gpu = np.asarray(gpu, np.float64)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    err = np.abs(gpu - ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} outputs outside the bound; worst "
                           f"err/sum|a||w| = {float((err / s).max()):.3e}")
    return float((err / s).max())


# M sequences, N weight rows, K inputs, epilogue, LayerNorm, strided x and y
CASES = [
    (1, 1152, 384, "store", True, False),      # Whisper-tiny qkv, one sequence
    (32, 3840, 1280, "store", True, True),     # Large-Whisper qkv, 32 sequences, row strides
    (32, 1280, 1280, "residual", False, False),  # out-projection onto the stream
    (32, 5120, 1280, "gelu", True, False),     # fc1 + GELU
    (32, 1280, 5120, "residual", False, False),  # fc2 onto the stream
    (45, 200, 320, "store", True, False),      # ragged rows, partial last weight tile, K % 128 = 64
    (300, 384, 384, "gelu", True, False),      # two row tiles
    (5, 1536, 64, "residual", False, False),   # one K block: no K split
    (3, 100, 128, "store", True, False),       # fewer weight rows than one 128-row tile
    (4, 10240, 128, "gelu", True, False),      # 80 weight tiles, K split in two under the norm
]


# Activations whose low bits matter: each value is +-2^e (1 + j 2^-13), j in
# {3, 5}, so its f16 high part drops exactly 3 2^-13 2^e, which the f16
# remainder plane holds exactly.  The two planes together reach the tensor
# cores with no rounding, and what is left is the fp32 accumulation error
# (about 2^-22 of sum |a||W| measured on random data).  Without the remainder
# plane the error would be sum_k lo_k W_nk, about 3.7e-4 |a| sqrt(K) |W|, i.e.
# 2^-16.6 of sum |a||W| at K = 1280 and more at K = 128: the bound 2^-19
# sum |a||W| separates the two.
LO_PLANE_BOUND = 2.0 ** -19
LO_PLANE_CASES = [(32, 1280, 1280), (16, 2048, 2048), (8, 512, 128)]


@pytest.mark.parametrize("M,N,K", LO_PLANE_CASES)
def test_linear_keeps_the_activation_remainder(M, N, K):
    """The activation's low bits reach the product: error <= 2^-19 sum|a||W|."""
    x, w = lo_plane_inputs(M, N, K, 7700 + K)
    ref = oracle.linear(x, w, None, mode="store")
    s = np.abs(x.astype(np.float64)) @ np.abs(dec16(w)).T
    y_d = torch.full((M, N), float("nan"), device="cuda")
    err = new_err()
    ops.asr_linear(dev(x), dev(w), y_d, mode="store", ws=ops.linear_workspace(M, N, K),
                   dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    worst = assert_linear_close(host(y_d), ref, LO_PLANE_BOUND * s + 1e-7, s,
                                f"remainder plane M={M} N={N} K={K}")
    print(f"remainder plane M={M} N={N} K={K}: worst err / sum|a||w| = {worst:.2e}")


@pytest.mark.parametrize("M,N,K,mode,ln,strided", CASES)
def test_linear_matches_oracle(M, N, K, mode, ln, strided):
    seed = 7000 + M + N + K
    x = syn.host_normal_f32((M, K), seed, mean=0.3, std=1.5)
    w = (syn.host_normal_f32((N, K), seed + 1) * np.float32(K ** -0.5)).astype(
        np.float16).view(np.uint16)
    bias = syn.host_normal_f32(N, seed + 2, std=0.5)
    g = syn.host_normal_f32(K, seed + 3, mean=1.0, std=0.2)
    b = syn.host_normal_f32(K, seed + 4, std=0.2)
    y0 = syn.host_normal_f32((M, N), seed + 5)
    lnp = (g, b) if ln else None
    ref = oracle.linear(x, w, bias, mode=mode, ln=lnp, y=y0 if mode == "residual" else None)
    a = oracle.layer_norm(x, g, b) if ln else x.astype(np.float64)
    tol, s = linear_bound(a, w, bias, mode, y0 if mode == "residual" else None)

    if strided:
        xw = dev(np.concatenate([x, np.full((M, 64), np.nan, np.float32)], axis=1))
        x_d = xw[:, :K]
        yw = torch.full((M, N + 32), float("nan"), device="cuda")
        y_d = yw[:, :N]
    else:
        x_d = dev(x)
        y_d = torch.full((M, N), float("nan"), device="cuda")
    if mode == "residual":
        y_d.copy_(dev(y0))
    ws = ops.linear_workspace(M, N, K)
    err = new_err()
    ops.asr_linear(x_d, dev(w), y_d, bias=dev(bias), ln=(dev(g), dev(b)) if ln else None,
                   mode=mode, ws=ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    worst = assert_linear_close(host(y_d), ref, tol, s, f"M={M} N={N} K={K} {mode}")
    print(f"M={M} N={N} K={K} {mode}: worst err / sum|a||w| = {worst:.2e}")
    if strided:
        assert torch.isnan(yw[:, N:]).all()  # nothing written past N
    if ws is not None:
        assert int(ws.count_nonzero().item()) == 0  # the call leaves its workspace zero


def test_linear_no_bias_and_repeat():
    """No bias; the same call twice gives results within the bound both
    times (the workspace is reused as the first call left it)."""
    M, N, K = 17, 640, 1280
    x = syn.host_normal_f32((M, K), 7100)
    w = (syn.host_normal_f32((N, K), 7101) * np.float32(K ** -0.5)).astype(
        np.float16).view(np.uint16)
    ref = oracle.linear(x, w, None)
    tol, s = linear_bound(x.astype(np.float64), w, None, "store")
    ws = ops.linear_workspace(M, N, K)
    x_d, w_d = dev(x), dev(w)
    for _ in range(2):
        y = torch.full((M, N), float("nan"), device="cuda")
        ops.asr_linear(x_d, w_d, y, ws=ws)
        torch.cuda.synchronize()
        assert_linear_close(host(y), ref, tol, s, "no bias")


def test_linear_rejects_on_device_args():
    M, N, K = 4, 256, 128
    x = torch.zeros(M, K, device="cuda")
    w = torch.zeros(N, K, dtype=torch.float16, device="cuda")
    y = torch.zeros(M, N, device="cuda")
    need = ops.load().asr_linear_workspace_size(M, N, K)
    assert need > 256  # K is split: the call needs its workspace
    small = torch.zeros(512, dtype=torch.uint8, device="cuda")
    with pytest.raises(ops.AsrError):
        ops.asr_linear(x, w, y, ws=small)  # workspace too small
    with pytest.raises(ops.AsrError):
        ops.asr_linear(x, w, y)  # workspace missing
    with pytest.raises(ops.AsrError):
        big = torch.zeros(M, N + K, device="cuda")
        ops.asr_linear(big[:, :K], w, big[:, K:K + N])  # y overlaps x


# ------------------------------------------------ one whole decoder layer --

def _dev_params(p):
    return {k: dev(v) for k, v in p.items()}


def test_whisper_decoder_layer_matches_oracle():
    """Whisper-tiny layer (d 384, 6 heads x 64, MLP 1536), 5 sequences in two
    beam groups, self lengths up to the 448-slot capacity, 1500 cross frames.
    Each step is checked against the oracle on the GPU's own input to that
    step (the dense bound above, the attention tolerance, the cache row bit
    for bit), then the whole layer against the oracle's composed layer."""
    from kv_cache_decode_asr_gb300 import decoder
    B, H, hd, cap, F, inner = 5, 6, 64, 448, 1500, 1536
    d = H * hd
    p = syn.layer_params(d, inner, 7200)
    x0 = syn.host_normal_f32((B, d), 7300)
    lens = np.array([1, 448, 37, 200, 5], np.int32)
    group = np.array([0, 0, 0, 1, 1], np.int32)
    cache0 = syn.host_normal_f16bits((B, cap, 2 * d), 7301)
    cross = syn.host_normal_f16bits((2, F, 2 * d), 7302)

    pd = _dev_params(p)
    x = dev(x0)
    cache = dev(cache0)
    cross_d = dev(cross)
    lens_d, group_d = dev(lens), dev(group)
    bufs = decoder.DecoderBuffers(B, d, inner, H, hd, 2, 3)
    err = new_err()
    # run the steps one by one to keep every intermediate
    snaps = {}
    scale = hd ** -0.5
    wl = bufs.ws_lin
    ops.asr_linear(x, pd["w_qkv"], bufs.qkv, bias=pd["b_qkv"], ln=(pd["ln1_g"], pd["ln1_b"]),
                   ws=wl, dev_err=err)
    ops.asr_self_attn_append_step(bufs.qkv[:, :d], bufs.qkv[:, d:2 * d], bufs.qkv[:, 2 * d:],
                                  cache, lens_d, H, hd, cap, scale, bufs.att, bufs.ws_self,
                                  dev_err=err)
    ops.asr_linear(bufs.att, pd["w_o"], x, bias=pd["b_o"], mode="residual", ws=wl, dev_err=err)
    snaps["x1"] = x.clone()
    ops.asr_linear(x, pd["w_cq"], bufs.qx, bias=pd["b_cq"], ln=(pd["ln2_g"], pd["ln2_b"]), ws=wl,
                   dev_err=err)
    ops.asr_cross_attn_step(bufs.qx, cross_d, group_d, 2, 3, H, hd, F, scale, bufs.attc,
                            bufs.ws_cross, dev_err=err)
    ops.asr_linear(bufs.attc, pd["w_co"], x, bias=pd["b_co"], mode="residual", ws=wl,
                   dev_err=err)
    snaps["x2"] = x.clone()
    ops.asr_linear(x, pd["w_fc1"], bufs.h, bias=pd["b_fc1"], ln=(pd["ln3_g"], pd["ln3_b"]),
                   mode="gelu", ws=wl, dev_err=err)
    ops.asr_linear(bufs.h, pd["w_fc2"], x, bias=pd["b_fc2"], mode="residual", ws=wl,
                   dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    qkv, att, qx, attc, h = (host(t) for t in (bufs.qkv, bufs.att, bufs.qx, bufs.attc, bufs.h))
    x1, x2, x3 = host(snaps["x1"]), host(snaps["x2"]), host(x)
    cache_g = host_u16(cache)

    def dense(xin, wk, bk, mode, ln, y_old, got, what):
        lnp = (p[ln + "_g"], p[ln + "_b"]) if ln else None
        ref = oracle.linear(xin, p[wk], p[bk], mode=mode, ln=lnp, y=y_old)
        a = oracle.layer_norm(xin, *lnp) if ln else xin.astype(np.float64)
        tol, s = linear_bound(a, p[wk], p[bk], mode, y_old)
        assert_linear_close(got, ref, tol, s, what)

    dense(x0, "w_qkv", "b_qkv", "store", "ln1", None, qkv, "qkv")
    cache_ref = cache0.copy()
    oracle.kv_append(qkv[:, d:2 * d], qkv[:, 2 * d:], cache_ref, lens - 1, H, hd)
    assert np.array_equal(cache_g, cache_ref)
    att_ref, _ = oracle.self_attn_step(qkv, cache_ref, lens, H, hd, scale, q_stride=3 * d)
    assert_attn_close(att, att_ref, "self-attention")
    dense(att, "w_o", "b_o", "residual", None, x0, x1, "out-projection")
    dense(x1, "w_cq", "b_cq", "store", "ln2", None, qx, "cross query")
    attc_ref, _ = oracle.cross_attn_step(qx, cross, group, H, hd, scale)
    assert_attn_close(attc, attc_ref, "cross-attention")
    dense(attc, "w_co", "b_co", "residual", None, x1, x2, "cross out-projection")
    dense(x2, "w_fc1", "b_fc1", "gelu", "ln3", None, h, "fc1 + GELU")
    dense(h, "w_fc2", "b_fc2", "residual", None, x2, x3, "fc2")

    # the whole layer against the oracle's composition from the same inputs
    cache_o = cache0.copy()
    x_ref, _ = oracle.whisper_decoder_layer_step(x0, p, cache_o, lens, cross, group, H, hd)
    assert_attn_close(x3, x_ref, "whole layer")

    # and through the package's composition (same launches, one call)
    x_b = dev(x0)
    cache_b = dev(cache0)
    decoder.whisper_decoder_layer(x_b, pd, cache_b, lens_d, cross_d, group_d, F, bufs, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attn_close(host(x_b), x_ref, "whisper_decoder_layer")


# ------------------------------------------------ RMSNorm and SwiGLU inputs --

# M sequences, N weight rows, K inputs, epilogue, input kind
CASES_QWEN = [
    (16, 4096, 2048, "store", "rms"),        # Qwen3-ASR q/k/v: RMSNorm, K split, bulk reduction
    (16, 12288, 2048, "store", "rms"),       # gate/up: 96 weight tiles, one CTA per tile (no split)
    (16, 2048, 6144, "residual", "swiglu"),  # down: silu(gate) * up onto the stream
    (37, 300, 192, "gelu", "rms"),           # ragged rows and weight tile
    (5, 256, 128, "residual", "rms"),        # RMSNorm with a residual: the ticket path
    (300, 256, 128, "store", "rms"),         # two row tiles of 150 (> 128 rows: the scalar path)
    (7, 640, 320, "gelu", "swiglu"),
    (254, 256, 128, "residual", "swiglu"),   # wide rows: two row tiles so one k-block fits
    (4, 10240, 128, "store", "rms"),         # 80 weight tiles, K split in two under the norm
]


@pytest.mark.parametrize("M,N,K,mode,kind", CASES_QWEN)
def test_linear_rms_swiglu_matches_oracle(M, N, K, mode, kind):
    seed = 7400 + M + N + K
    xw = 2 * K if kind == "swiglu" else K
    x = syn.host_normal_f32((M, xw), seed, mean=0.2, std=1.4)
    w = (syn.host_normal_f32((N, K), seed + 1) * np.float32(K ** -0.5)).astype(
        np.float16).view(np.uint16)
    g = syn.host_normal_f32(K, seed + 3, mean=1.0, std=0.2)
    y0 = syn.host_normal_f32((M, N), seed + 5)
    res = mode == "residual"
    kw = {"rms": g} if kind == "rms" else {"swiglu": True}
    ref = oracle.linear(x, w, None, mode=mode, eps=1e-6, y=y0 if res else None, **kw)
    if kind == "rms":
        a = np.stack([oracle.rmsnorm(x[m].astype(np.float64), g.astype(np.float64), 1e-6)
                      for m in range(M)])
    else:
        a = oracle.silu(x[:, :K]) * x[:, K:].astype(np.float64)
    tol, s = linear_bound(a, w, None, mode, y0 if res else None)
    y_d = dev(y0) if res else torch.full((M, N), float("nan"), device="cuda")
    ws = ops.linear_workspace(M, N, K)
    err = new_err()
    dkw = {"rms": dev(g)} if kind == "rms" else {"swiglu": True}
    ops.asr_linear(dev(x), dev(w), y_d, mode=mode, eps=1e-6, ws=ws, dev_err=err, **dkw)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    worst = assert_linear_close(host(y_d), ref, tol, s, f"M={M} N={N} K={K} {mode} {kind}")
    print(f"M={M} N={N} K={K} {mode} {kind}: worst err / sum|a||w| = {worst:.2e}")
    if ws is not None:
        assert int(ws.count_nonzero().item()) == 0


def test_qwen3_decoder_layer_matches_oracle():
    """A Qwen3-ASR-shaped layer (16 Q / 8 KV heads of 128, d 256, MLP 384),
    3 sequences at n_past 0, 30 and 63 of a 64-row cache.  Each step against
    the oracle on the GPU's own input to it (the dense bound, the attention
    tolerance, the cache row bit for bit), then the whole layer."""
    from kv_cache_decode_asr_gb300 import decoder
    B, Hq, Hkv, hd, cap, d, inner = 3, 16, 8, 128, 64, 256, 384
    nq, nk = Hq * hd, Hkv * hd
    p = syn.qwen_layer_params(d, inner, Hq, Hkv, hd, 7500)
    x0 = syn.host_normal_f32((B, d), 7600)
    n_past = np.array([0, 30, 63], np.int32)
    cache0 = syn.host_normal_f16bits((B, cap, 2 * nk), 7601)
    pd = {k: dev(v) for k, v in p.items()}
    bufs = decoder.QwenDecoderBuffers(B, d, inner, Hq, Hkv, hd)
    x = dev(x0)
    cache = dev(cache0)
    np_d = dev(n_past)
    err = new_err()
    wl = bufs.ws_lin
    ops.asr_linear(x, pd["w_qkv"], bufs.qkv, rms=pd["rms1"], eps=1e-6, ws=wl, dev_err=err)
    ops.asr_gqa_step(bufs.qkv[:, :nq], bufs.qkv[:, nq:nq + nk], bufs.qkv[:, nq + nk:],
                     pd["q_norm"], pd["k_norm"], 1e-6, 1e6, np_d, cache, cap, Hq, Hkv, hd,
                     hd ** -0.5, bufs.att, bufs.ws_gqa, dev_err=err)
    ops.asr_linear(bufs.att, pd["w_o"], x, mode="residual", ws=wl, dev_err=err)
    x1 = host(x).copy()
    ops.asr_linear(x, pd["w_gu"], bufs.gu, rms=pd["rms2"], eps=1e-6, ws=wl, dev_err=err)
    ops.asr_linear(bufs.gu, pd["w_down"], x, swiglu=True, mode="residual", ws=wl, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    qkv, att, gu, x2 = host(bufs.qkv), host(bufs.att), host(bufs.gu), host(x)

    def dense(xin, wk, mode, rms, y_old, got, what, swiglu=False):
        ref = oracle.linear(xin, p[wk], None, mode=mode, eps=1e-6, y=y_old,
                            rms=p[rms] if rms else None, swiglu=swiglu)
        if rms:
            a = np.stack([oracle.rmsnorm(xin[m].astype(np.float64), p[rms].astype(np.float64),
                                         1e-6) for m in range(xin.shape[0])])
        elif swiglu:
            K = p[wk].shape[1]
            a = oracle.silu(xin[:, :K]) * xin[:, K:].astype(np.float64)
        else:
            a = xin.astype(np.float64)
        tol, s = linear_bound(a, p[wk], None, mode, y_old)
        assert_linear_close(got, ref, tol, s, what)

    dense(x0, "w_qkv", "store", "rms1", None, qkv, "q/k/v")
    cache_ref = cache0.copy()
    att_ref, _ = oracle.gqa_step(np.ascontiguousarray(qkv[:, :nq]),
                                 np.ascontiguousarray(qkv[:, nq:nq + nk]),
                                 np.ascontiguousarray(qkv[:, nq + nk:]), p["q_norm"], p["k_norm"],
                                 1e-6, 1e6, n_past, cache_ref, Hq, Hkv, hd, hd ** -0.5)
    assert_attn_close(att, att_ref, "GQA step")
    k_rows = host_u16(cache)[np.arange(B), n_past]
    assert np.array_equal(k_rows[:, nk:], cache_ref[np.arange(B), n_past][:, nk:])  # V bitwise
    dense(att, "w_o", "residual", None, x0, x1, "output projection")
    dense(x1, "w_gu", "store", "rms2", None, gu, "gate/up")
    dense(gu, "w_down", "residual", None, x1, x2, "SwiGLU down", swiglu=True)

    cache_o = cache0.copy()
    x_ref, _ = oracle.qwen3_decoder_layer_step(x0, p, cache_o, n_past, Hq, Hkv, hd)
    assert_attn_close(x2, x_ref, "whole layer")

    xb = dev(x0)
    cb = dev(cache0)
    decoder.qwen3_decoder_layer(xb, pd, cb, np_d, bufs, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attn_close(host(xb), x_ref, "qwen3_decoder_layer")


def test_linear_one_workspace_every_mode():
    """One workspace serves calls in every norm and input mode, back to back
    on one stream (each leaves it zero for the next)."""
    M, N, K = 9, 768, 512
    ws = ops.linear_workspace(M, N, K)
    assert ws is not None
    x = syn.host_normal_f32((M, 2 * K), 7700)
    w = (syn.host_normal_f32((N, K), 7701) * np.float32(K ** -0.5)).astype(
        np.float16).view(np.uint16)
    g = syn.host_normal_f32(K, 7702, mean=1.0, std=0.1)
    b = syn.host_normal_f32(K, 7703, std=0.1)
    bias = syn.host_normal_f32(N, 7704, std=0.1)
    xd, wd, gd, bd, biasd = dev(x), dev(w), dev(g), dev(b), dev(bias)
    xk = np.ascontiguousarray(x[:, :K])
    calls = [("ln", dict(ln=(gd, bd)), dict(ln=(g, b)), "store"),
             ("rms", dict(rms=gd), dict(rms=g), "gelu"),
             ("swiglu", dict(swiglu=True), dict(swiglu=True), "store"),
             ("plain", {}, {}, "gelu")]
    err = new_err()
    outs = []
    for name, dkw, okw, mode in calls:
        src = xd if name == "swiglu" else xd[:, :K]
        y = torch.full((M, N), float("nan"), device="cuda")
        ops.asr_linear(src, wd, y, bias=biasd, mode=mode, eps=1e-5, ws=ws, dev_err=err, **dkw)
        outs.append((name, okw, mode, y))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert int(ws.count_nonzero().item()) == 0
    for name, okw, mode, y in outs:
        xin = x if name == "swiglu" else xk
        ref = oracle.linear(xin, w, bias, mode=mode, eps=1e-5, **okw)
        if name == "ln":
            a = oracle.layer_norm(xk, g, b, eps=1e-5)
        elif name == "rms":
            a = np.stack([oracle.rmsnorm(xk[m].astype(np.float64), g.astype(np.float64), 1e-5)
                          for m in range(M)])
        elif name == "swiglu":
            a = oracle.silu(x[:, :K]) * x[:, K:].astype(np.float64)
        else:
            a = xk.astype(np.float64)
        tol, s = linear_bound(a, w, bias, mode)
        assert_linear_close(host(y), ref, tol, s, name)

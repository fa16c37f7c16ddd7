"""Host checks of the decoder-layer composition (no GPU needed).

`kv_cache_decode_asr_gb300.decoder` only orders calls of the C ABI.  These
tests replace its binding with a recorder and check, against the pages'
order of a layer (wavo Decoder::record_step for Whisper; transcribe.cpp
decoder.h for Qwen3-ASR), that every step is called once, in order, on the
right buffers, with the right norm, input and epilogue.
"""
import types

import numpy as np
import pytest

from kv_cache_decode_asr_gb300 import decoder


class Buf:
    """A stand-in tensor: a name and the column range it views."""

    def __init__(self, name, cols=None, rows=4, lo=0):
        self.name, self.cols, self.rows, self.lo = name, cols, rows, lo
        self.shape = (rows, cols, cols) if name == "cache" else (rows, cols)

    def __getitem__(self, idx):
        _, sl = idx
        lo = sl.start or 0
        hi = sl.stop if sl.stop is not None else self.cols
        return Buf(self.name, hi - lo, self.rows, self.lo + lo)

    def __repr__(self):
        return f"{self.name}[{self.lo}:{self.lo + (self.cols or 0)}]"


class Recorder:
    def __init__(self):
        self.calls = []

    def asr_linear(self, x, w, y, bias=None, ln=None, rms=None, eps=None, swiglu=False,
                   mode="store", ws=None, dev_err=None, stream=None):
        norm = "ln" if ln is not None else "rms" if rms is not None else None
        self.calls.append(("linear", repr(x), w, repr(y), bias, norm, swiglu, mode))

    def asr_self_attn_append_step(self, q, k, v, cache, lens, H, hd, cap, scale, out, ws,
                                  dev_err=None, stream=None):
        self.calls.append(("self", repr(q), repr(k), repr(v), repr(out)))

    def asr_cross_attn_step(self, q, cross, group, G, beams, H, hd, frames, scale, out, ws,
                            dev_err=None, stream=None):
        self.calls.append(("cross", repr(q), repr(out)))

    def asr_gqa_step(self, q, k, v, wq, wk, eps, base, n_past, cache, cap, Hq, Hkv, hd, scale,
                     out, ws, dev_err=None, stream=None):
        self.calls.append(("gqa", repr(q), repr(k), repr(v), wq, wk, repr(out)))


@pytest.fixture
def rec(monkeypatch):
    r = Recorder()
    monkeypatch.setattr(decoder, "ops", r)
    return r


def test_whisper_layer_order(rec):
    d = 8
    bufs = types.SimpleNamespace(d=d, heads=2, head_dim=4, n_sources=1, max_beams=1,
                                 qkv=Buf("qkv", 3 * d), att=Buf("att", d), qx=Buf("qx", d),
                                 attc=Buf("attc", d), h=Buf("h", 4 * d), ws_self=None,
                                 ws_cross=None, ws_lin=None)
    p = {k: k for k in ("w_qkv", "b_qkv", "w_o", "b_o", "w_cq", "b_cq", "w_co", "b_co", "w_fc1",
                        "b_fc1", "w_fc2", "b_fc2", "ln1_g", "ln1_b", "ln2_g", "ln2_b", "ln3_g",
                        "ln3_b")}
    x = Buf("x", d)
    decoder.whisper_decoder_layer(x, p, Buf("cache", 16), None, None, None, 1500, bufs)
    assert rec.calls == [
        ("linear", "x[0:8]", "w_qkv", "qkv[0:24]", "b_qkv", "ln", False, "store"),
        ("self", "qkv[0:8]", "qkv[8:16]", "qkv[16:24]", "att[0:8]"),
        ("linear", "att[0:8]", "w_o", "x[0:8]", "b_o", None, False, "residual"),
        ("linear", "x[0:8]", "w_cq", "qx[0:8]", "b_cq", "ln", False, "store"),
        ("cross", "qx[0:8]", "attc[0:8]"),
        ("linear", "attc[0:8]", "w_co", "x[0:8]", "b_co", None, False, "residual"),
        ("linear", "x[0:8]", "w_fc1", "h[0:32]", "b_fc1", "ln", False, "gelu"),
        ("linear", "h[0:32]", "w_fc2", "x[0:8]", "b_fc2", None, False, "residual"),
    ]
    assert len(rec.calls) == decoder.LAUNCHES_PER_LAYER


def test_qwen3_layer_order(rec):
    Hq, Hkv, hd, d, inner = 4, 2, 8, 16, 24
    nq, nk = Hq * hd, Hkv * hd
    bufs = types.SimpleNamespace(nq=nq, nk=nk, head_dim=hd, q_heads=Hq, kv_heads=Hkv,
                                 qkv=Buf("qkv", nq + 2 * nk), att=Buf("att", nq),
                                 gu=Buf("gu", 2 * inner), ws_gqa=None, ws_lin=None)
    p = {k: k for k in ("w_qkv", "w_o", "w_gu", "w_down", "rms1", "rms2", "q_norm", "k_norm")}
    x = Buf("x", d)
    decoder.qwen3_decoder_layer(x, p, Buf("cache", 64), None, bufs)
    assert rec.calls == [
        ("linear", "x[0:16]", "w_qkv", "qkv[0:64]", None, "rms", False, "store"),
        ("gqa", "qkv[0:32]", "qkv[32:48]", "qkv[48:64]", "q_norm", "k_norm", "att[0:32]"),
        ("linear", "att[0:32]", "w_o", "x[0:16]", None, None, False, "residual"),
        ("linear", "x[0:16]", "w_gu", "gu[0:48]", None, "rms", False, "store"),
        ("linear", "gu[0:48]", "w_down", "x[0:16]", None, None, True, "residual"),
    ]
    assert len(rec.calls) == decoder.QWEN_LAUNCHES_PER_LAYER


def test_synthetic_layer_params_shapes():
    from kv_cache_decode_asr_gb300 import synthetic as syn
    p = syn.layer_params(16, 64, 1)
    assert p["w_qkv"].shape == (48, 16) and p["w_fc2"].shape == (16, 64)
    assert np.all(p["b_qkv"][16:32] == 0)  # the key projection has no bias
    q = syn.qwen_layer_params(32, 48, 4, 2, 16, 2)
    assert q["w_qkv"].shape == (4 * 16 + 2 * 2 * 16, 32)
    assert q["w_gu"].shape == (96, 32) and q["w_down"].shape == (32, 48)
    assert q["w_o"].shape == (32, 64) and q["q_norm"].shape == (16,)

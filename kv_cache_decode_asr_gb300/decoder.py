"""The whole decoder step around the attention, composed from the library's
entry points (argument marshalling only: every step runs in the library's
kernels): the Whisper decoder layer and the Qwen3-ASR decoder layer.

Order of the steps ("wavo 0.1.0, src/whisper/decoder.rs",
Decoder::record_step), for one new token per sequence:

    qkv = LN_self(x) W_qkv^T + b_qkv        asr_linear (LayerNorm fused, Bias)
    cache row lens-1 <- f16(k, v); att      asr_self_attn_append_step
    x  += att W_o^T + b_o                   asr_linear (Residual)
    qx  = LN_cross(x) W_cq^T + b_cq         asr_linear (LayerNorm fused, Bias)
    attc = attend(qx, cross K/V)            asr_cross_attn_step
    x  += attc W_co^T + b_co                asr_linear (Residual)
    h   = gelu(LN_ffn(x) W_1^T + b_1)       asr_linear (LayerNorm fused, Gelu)
    x  += h W_2^T + b_2                     asr_linear (Residual)

Eight launches per layer.  Buffers: x fp32 [B, d] (the residual stream,
updated in place), qkv fp32 [B, 3d], att / qx / attc fp32 [B, d], h fp32
[B, inner].
"""
from . import ops


class DecoderBuffers:
    """Scratch of one decoder step: activations and the workspaces.

    One linear workspace serves every projection: each call leaves it zero
    and calls on one stream run one after another."""

    def __init__(self, B, d, inner, heads, head_dim, n_sources, max_beams, device=None):
        import torch
        device = device or "cuda"
        f32 = torch.float32
        self.B, self.d, self.inner = B, d, inner
        self.heads, self.head_dim = heads, head_dim
        self.n_sources, self.max_beams = n_sources, max_beams
        self.qkv = torch.zeros(B, 3 * d, dtype=f32, device=device)
        self.att = torch.zeros(B, d, dtype=f32, device=device)
        self.qx = torch.zeros(B, d, dtype=f32, device=device)
        self.attc = torch.zeros(B, d, dtype=f32, device=device)
        self.h = torch.zeros(B, inner, dtype=f32, device=device)
        self.ws_self = ops.workspace(ops.OP_SELF_ATTN, B, B, 1, heads, head_dim, device=device)
        self.ws_cross = ops.workspace(ops.OP_CROSS_ATTN, B, n_sources, max_beams, heads, head_dim,
                                      device=device)
        sizes = [(3 * d, d), (d, d), (inner, d), (d, inner)]
        need = max(ops.load().asr_linear_workspace_size(B, n, k) for n, k in sizes)
        self.ws_lin = (torch.zeros(need + 256, dtype=torch.uint8, device=device) if need else None)


def whisper_decoder_layer(x, p, cache, lens, cross, group, frames, bufs, eps=1e-5, dev_err=None,
                          stream=None):
    """One decoder layer on the new token of every sequence.

    x: fp32 [B, d], updated in place; p: the layer's parameters (w_qkv,
    w_o, w_cq, w_co, w_fc1, w_fc2 f16 [out, in]; b_* fp32 [out]; ln1_g ..
    ln3_b fp32 [d]); cache: f16 self cache [B, capacity, 2d] (sequence
    stride cache.stride(0)); lens: int32 [B] keys including the new token
    (its row is lens-1); cross: f16 [G, frames, 2d] (group stride
    cross.stride(0)); group: int32 [B]; bufs: DecoderBuffers."""
    d, H, hd = bufs.d, bufs.heads, bufs.head_dim
    scale = hd ** -0.5
    cap = cache.shape[1]
    wl = bufs.ws_lin
    qkv = bufs.qkv
    ops.asr_linear(x, p["w_qkv"], qkv, bias=p["b_qkv"], ln=(p["ln1_g"], p["ln1_b"]), eps=eps,
                   ws=wl, dev_err=dev_err, stream=stream)
    ops.asr_self_attn_append_step(qkv[:, :d], qkv[:, d:2 * d], qkv[:, 2 * d:], cache, lens, H, hd,
                                  cap, scale, bufs.att, bufs.ws_self, dev_err=dev_err,
                                  stream=stream)
    ops.asr_linear(bufs.att, p["w_o"], x, bias=p["b_o"], mode="residual", ws=wl, dev_err=dev_err,
                   stream=stream)
    ops.asr_linear(x, p["w_cq"], bufs.qx, bias=p["b_cq"], ln=(p["ln2_g"], p["ln2_b"]), eps=eps,
                   ws=wl, dev_err=dev_err, stream=stream)
    ops.asr_cross_attn_step(bufs.qx, cross, group, bufs.n_sources, bufs.max_beams, H, hd, frames,
                            scale, bufs.attc, bufs.ws_cross, dev_err=dev_err, stream=stream)
    ops.asr_linear(bufs.attc, p["w_co"], x, bias=p["b_co"], mode="residual", ws=wl,
                   dev_err=dev_err, stream=stream)
    ops.asr_linear(x, p["w_fc1"], bufs.h, bias=p["b_fc1"], ln=(p["ln3_g"], p["ln3_b"]), eps=eps,
                   mode="gelu", ws=wl, dev_err=dev_err, stream=stream)
    ops.asr_linear(bufs.h, p["w_fc2"], x, bias=p["b_fc2"], mode="residual", ws=wl,
                   dev_err=dev_err, stream=stream)


LAUNCHES_PER_LAYER = 8


# ------------------------------------------------------------- Qwen3-ASR --
#
# Order ("transcribe.cpp, src/arch/qwen3_asr/decoder.h", header comment and
# StepBuildBatched), for one new token per sequence at position n_past:
#
#     qkv = RMSNorm(x) [W_q | W_k | W_v]^T     asr_linear (RMSNorm fused, no bias)
#     q/k RMSNorm, RoPE, append, GQA           asr_gqa_step
#     x  += att W_o^T                          asr_linear (Residual)
#     gu  = RMSNorm(x) [W_gate | W_up]^T       asr_linear (RMSNorm fused)
#     x  += (silu(gate) * up) W_down^T         asr_linear (SwiGLU input, Residual)
#
# Five launches per layer.

class QwenDecoderBuffers:
    """Scratch of one Qwen3-ASR decoder step: qkv fp32 [B, (Hq + 2 Hkv) hd],
    att fp32 [B, Hq hd], gu fp32 [B, 2 inner] and the workspaces."""

    def __init__(self, B, d, inner, q_heads, kv_heads, head_dim, device=None):
        import torch
        device = device or "cuda"
        f32 = torch.float32
        self.B, self.d, self.inner = B, d, inner
        self.q_heads, self.kv_heads, self.head_dim = q_heads, kv_heads, head_dim
        nq, nk = q_heads * head_dim, kv_heads * head_dim
        self.nq, self.nk = nq, nk
        self.qkv = torch.zeros(B, nq + 2 * nk, dtype=f32, device=device)
        self.att = torch.zeros(B, nq, dtype=f32, device=device)
        self.gu = torch.zeros(B, 2 * inner, dtype=f32, device=device)
        self.ws_gqa = ops.workspace(ops.OP_GQA_STEP, B, B, 1, q_heads, head_dim, device=device)
        sizes = [(nq + 2 * nk, d), (d, nq), (2 * inner, d), (d, inner)]
        need = max(ops.load().asr_linear_workspace_size(B, n, k) for n, k in sizes)
        self.ws_lin = (torch.zeros(need + 256, dtype=torch.uint8, device=device) if need else None)


def qwen3_decoder_layer(x, p, cache, n_past, bufs, eps=1e-6, rope_base=1e6, dev_err=None,
                        stream=None):
    """One Qwen3-ASR decoder layer on the new token of every sequence.

    x: fp32 [B, d], updated in place; p: the layer's parameters (w_qkv,
    w_o, w_gu, w_down f16 [out, in]; rms1, rms2 fp32 [d]; q_norm, k_norm
    fp32 [head_dim]); cache: f16 [B, capacity, 2 Hkv hd] (row n_past
    written); n_past: int32 [B]; bufs: QwenDecoderBuffers."""
    nq, nk, hd = bufs.nq, bufs.nk, bufs.head_dim
    wl = bufs.ws_lin
    qkv = bufs.qkv
    ops.asr_linear(x, p["w_qkv"], qkv, rms=p["rms1"], eps=eps, ws=wl, dev_err=dev_err,
                   stream=stream)
    ops.asr_gqa_step(qkv[:, :nq], qkv[:, nq:nq + nk], qkv[:, nq + nk:], p["q_norm"], p["k_norm"],
                     eps, rope_base, n_past, cache, cache.shape[1], bufs.q_heads, bufs.kv_heads,
                     hd, hd ** -0.5, bufs.att, bufs.ws_gqa, dev_err=dev_err, stream=stream)
    ops.asr_linear(bufs.att, p["w_o"], x, mode="residual", ws=wl, dev_err=dev_err, stream=stream)
    ops.asr_linear(x, p["w_gu"], bufs.gu, rms=p["rms2"], eps=eps, ws=wl, dev_err=dev_err,
                   stream=stream)
    ops.asr_linear(bufs.gu, p["w_down"], x, swiglu=True, mode="residual", ws=wl,
                   dev_err=dev_err, stream=stream)


QWEN_LAUNCHES_PER_LAYER = 5

"""Seeded synthetic inputs for the decoder-step attention path.

This module only draws random numbers and lays them out; it holds none of the
path's arithmetic.  The same bytes feed the CUDA library and the CPU oracle.

Workloads (shapes of the pages' models; no weights or audio are needed):

* ``whisper_tiny_b1``      -- Whisper-tiny (d=384, 6 heads x 64, 4 decoder
  layers), one sequence, self cache of 448 slots filled to t=223 so the new
  token sits at 224 (225 keys), cross K/V of 1500 encoder frames.
* ``whisper_tiny_b64_beam5`` -- the same model, 64 sequences in 5-beam groups
  (group of sequence b is b // 5, so 13 groups, the last of 4 beams), self
  lengths uniform in [1, 448], cross K/V shared per group, a random beam
  permutation drawn within each group.
* ``whisper_large_b32``    -- Large-Whisper shape (d=1280, 20 heads x 64, 32
  decoder layers), 32 sequences, self lengths uniform in [1, 448], cross K/V of
  1500 frames per sequence.
* ``qwen3_asr_gqa_b16``    -- Qwen3-ASR decoder (28 layers, 16 Q / 8 KV heads of
  128), 16 sequences, n_past uniform in [1024, 4096], cache of 4224 slots,
  RMSNorm weights N(1, 0.1).
* ``qwen3_asr_prefill_b8`` -- the same decoder prefilling 8 prompts of 1536
  tokens (16 prefix + 1500 audio frames + 20 suffix).
* ``whisper_large_prefill_b32`` -- Large-Whisper decoder prompt prefill
  (20 heads x 64): 32 prompts of up to 448 tokens, lengths uniform in
  [1, 448], K/V written to a 448-slot self cache.
* ``whisper_large_encoder_b8`` -- Large-Whisper encoder self-attention (20
  heads x 64) over the 1500 frames of 8 utterances, unmasked.
* ``whisper_large_cross_fill_b32`` -- the cross K/V of one Large-Whisper
  decoder layer (d = 1280) from the encoder output of 32 utterances of 1500
  frames; weights N(0, 1/d), bias N(0, 1).
* ``whisper_large_decoder_step_b32`` -- the whole Large-Whisper decoder step
  around the attention (32 layers, d = 1280, 20 heads x 64, MLP 5120), 32
  sequences, self lengths uniform in [1, 448], 1500 cross frames: per layer
  LayerNorm + qkv, append + self-attention, out-projection, LayerNorm +
  cross query, cross-attention, cross out-projection, LayerNorm + fc1 + GELU,
  fc2.  Random weights (``layer_params``).

* ``qwen3_asr_decoder_step_b16`` -- the whole Qwen3-ASR decoder step around
  the GQA step (28 layers, 16 Q / 8 KV heads of 128, d = 2048, MLP 6144),
  16 sequences, n_past uniform in [1024, 4096]: per layer RMSNorm + q/k/v,
  the fused GQA step, the output projection, RMSNorm + gate/up, SwiGLU +
  down.  Random weights (``qwen_layer_params``).

Layer weights (``layer_params``): every projection N(0, 1/fan_in) stored as
f16, biases N(0, 0.1) with the key bias zero, LayerNorm weights N(1, 0.1) and
biases N(0, 0.1); the residual stream x starts N(0, 1).

Values: activations and caches N(0, 1); caches are stored as f16 (the fp32
draw rounded to nearest even).  Host draws use numpy's PCG64; device draws use
torch's generator for that device.
"""
import numpy as np

WORKLOADS = {
    "whisper_tiny_b1": dict(kind="whisper", B=1, d=384, heads=6, head_dim=64, layers=4,
                            capacity=448, frames=1500, beam=1, lens="fixed", fixed_len=225),
    "whisper_tiny_b64_beam5": dict(kind="whisper", B=64, d=384, heads=6, head_dim=64, layers=4,
                                   capacity=448, frames=1500, beam=5, lens="uniform",
                                   len_lo=1, len_hi=448, rearrange=True),
    "whisper_large_b32": dict(kind="whisper", B=32, d=1280, heads=20, head_dim=64, layers=32,
                              capacity=448, frames=1500, beam=1, lens="uniform",
                              len_lo=1, len_hi=448),
    "qwen3_asr_gqa_b16": dict(kind="gqa", B=16, layers=28, q_heads=16, kv_heads=8, head_dim=128,
                              capacity=4224, n_past_lo=1024, n_past_hi=4096, eps=1e-6,
                              rope_base=1e6, w_mean=1.0, w_std=0.1),
    "qwen3_asr_prefill_b8": dict(kind="prefill", B=8, T=1536, prefix=16, audio=1500, suffix=20,
                                 q_heads=16, kv_heads=8, head_dim=128, capacity=1536, eps=1e-6,
                                 rope_base=1e6, w_mean=1.0, w_std=0.1),
    "whisper_large_prefill_b32": dict(kind="mha_prefill", B=32, T=448, heads=20, head_dim=64,
                                      capacity=448, len_lo=1, len_hi=448),
    "whisper_large_encoder_b8": dict(kind="encoder", B=8, T=1500, heads=20, head_dim=64),
    "whisper_large_cross_fill_b32": dict(kind="cross_fill", G=32, frames=1500, d=1280),
    "whisper_large_decoder_step_b32": dict(kind="decoder_step", B=32, d=1280, heads=20,
                                           head_dim=64, inner=5120, layers=32, capacity=448,
                                           frames=1500, beam=1, len_lo=1, len_hi=448),
    "qwen3_asr_decoder_step_b16": dict(kind="qwen_decoder_step", B=16, layers=28, q_heads=16,
                                       kv_heads=8, head_dim=128, d=2048, inner=6144,
                                       capacity=4224, n_past_lo=1024, n_past_hi=4096, eps=1e-6,
                                       rope_base=1e6, w_mean=1.0, w_std=0.1),
}

# projections of one decoder layer: name, output size, input size (d units)
LAYER_PROJ = (("qkv", 3, 1), ("o", 1, 1), ("cq", 1, 1), ("co", 1, 1), ("fc1", "inner", 1),
              ("fc2", 1, "inner"))


def _proj_shapes(d, inner):
    size = lambda u: inner if u == "inner" else u * d
    return [(name, size(o), size(i)) for name, o, i in LAYER_PROJ]


def layer_params(d, inner, seed):
    """Host parameters of one decoder layer (numpy): w_* f16 bits [out, in],
    b_* float32 [out] (the key third of b_qkv zero), ln{1,2,3}_{g,b} float32 [d]."""
    p = {}
    for i, (name, n_out, n_in) in enumerate(_proj_shapes(d, inner)):
        w = host_normal_f32((n_out, n_in), seed + 2 * i, std=n_in ** -0.5)
        p["w_" + name] = w.astype(np.float16).view(np.uint16)
        p["b_" + name] = host_normal_f32(n_out, seed + 2 * i + 1, std=0.1)
    p["b_qkv"][d:2 * d] = 0
    for j in (1, 2, 3):
        p[f"ln{j}_g"] = host_normal_f32(d, seed + 20 + j, mean=1.0, std=0.1)
        p[f"ln{j}_b"] = host_normal_f32(d, seed + 30 + j, std=0.1)
    return p


def seed_for(workload_index, tensor_id):
    """Seed of tensor ``tensor_id`` of workload ``workload_index``."""
    return 1000 * int(workload_index) + int(tensor_id)


# ------------------------------------------------------------------ host --

def rng(seed):
    return np.random.Generator(np.random.PCG64(int(seed)))


def host_normal_f32(shape, seed, mean=0.0, std=1.0):
    """float32 N(mean, std) array."""
    x = rng(seed).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0 or mean != 0.0:
        x = (x * np.float32(std) + np.float32(mean)).astype(np.float32)
    return x


def host_normal_f16bits(shape, seed):
    """f16 N(0, 1) values as their binary16 bit patterns (uint16)."""
    return host_normal_f32(shape, seed).astype(np.float16).view(np.uint16)


def lens_uniform(B, lo, hi, seed):
    """int32 [B] drawn uniformly from the integers lo..hi inclusive."""
    return rng(seed).integers(lo, hi + 1, size=B, dtype=np.int64).astype(np.int32)


def beam_groups(B, beam):
    """Group (encoder source) of each sequence: consecutive runs of ``beam``."""
    return (np.arange(B, dtype=np.int32) // np.int32(beam)).astype(np.int32)


def beam_permutation(B, beam, seed):
    """A random permutation of the sequences that stays inside each beam group."""
    r = rng(seed)
    idx = np.arange(B, dtype=np.int32)
    for g0 in range(0, B, beam):
        g1 = min(g0 + beam, B)
        idx[g0:g1] = g0 + r.permutation(g1 - g0).astype(np.int32)
    return idx


# ---------------------------------------------------------------- device --

def dev_normal(shape, seed, device, dtype=None, mean=0.0, std=1.0):
    """torch tensor N(mean, std) drawn on ``device`` (fp32 draw, then cast)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0 or mean != 0.0:
        x.mul_(std).add_(mean)
    if dtype is not None and dtype != torch.float32:
        x = x.to(dtype)
    return x


def _qwen_shapes(d, inner, q_heads, kv_heads, head_dim):
    nq, nk = q_heads * head_dim, kv_heads * head_dim
    return [("qkv", nq + 2 * nk, d), ("o", d, nq), ("gu", 2 * inner, d), ("down", d, inner)]


def qwen_layer_params(d, inner, q_heads, kv_heads, head_dim, seed):
    """Host parameters of one Qwen3-ASR decoder layer (numpy): w_qkv (q rows,
    then k, then v), w_o, w_gu (gate rows, then up rows), w_down as f16 bits
    [out, in], each N(0, 1/fan_in); rms1, rms2 float32 [d] and q_norm, k_norm
    float32 [head_dim], N(1, 0.1).  No biases."""
    p = {}
    for i, (name, n_out, n_in) in enumerate(_qwen_shapes(d, inner, q_heads, kv_heads, head_dim)):
        w = host_normal_f32((n_out, n_in), seed + i, std=n_in ** -0.5)
        p["w_" + name] = w.astype(np.float16).view(np.uint16)
    p["rms1"] = host_normal_f32(d, seed + 10, mean=1.0, std=0.1)
    p["rms2"] = host_normal_f32(d, seed + 11, mean=1.0, std=0.1)
    p["q_norm"] = host_normal_f32(head_dim, seed + 12, mean=1.0, std=0.1)
    p["k_norm"] = host_normal_f32(head_dim, seed + 13, mean=1.0, std=0.1)
    return p


def dev_qwen_layer_params(n_layers, d, inner, q_heads, kv_heads, head_dim, seed, device):
    """qwen_layer_params of n_layers layers drawn on the device, stacked on a
    leading layer axis."""
    import torch
    p = {}
    for i, (name, n_out, n_in) in enumerate(_qwen_shapes(d, inner, q_heads, kv_heads, head_dim)):
        w = torch.empty(n_layers, n_out, n_in, dtype=torch.float16, device=device)
        dev_fill_normal_(w, seed + i)
        w.mul_(n_in ** -0.5)
        p["w_" + name] = w
    p["rms1"] = dev_normal((n_layers, d), seed + 10, device, mean=1.0, std=0.1)
    p["rms2"] = dev_normal((n_layers, d), seed + 11, device, mean=1.0, std=0.1)
    p["q_norm"] = dev_normal((n_layers, head_dim), seed + 12, device, mean=1.0, std=0.1)
    p["k_norm"] = dev_normal((n_layers, head_dim), seed + 13, device, mean=1.0, std=0.1)
    return p


def dev_layer_params(n_layers, d, inner, seed, device):
    """The parameters of n_layers decoder layers drawn on the device, stacked
    on a leading layer axis (weights f16, the rest fp32); same recipe as
    layer_params."""
    import torch
    p = {}
    for i, (name, n_out, n_in) in enumerate(_proj_shapes(d, inner)):
        w = torch.empty(n_layers, n_out, n_in, dtype=torch.float16, device=device)
        dev_fill_normal_(w, seed + 2 * i)
        w.mul_(n_in ** -0.5)
        p["w_" + name] = w
        p["b_" + name] = dev_normal((n_layers, n_out), seed + 2 * i + 1, device, std=0.1)
    p["b_qkv"][:, d:2 * d] = 0
    for j in (1, 2, 3):
        p[f"ln{j}_g"] = dev_normal((n_layers, d), seed + 20 + j, device, mean=1.0, std=0.1)
        p[f"ln{j}_b"] = dev_normal((n_layers, d), seed + 30 + j, device, std=0.1)
    return p


def dev_fill_normal_(t, seed, chunk_elems=1 << 28):
    """Fill an existing f16 (or f32) device tensor with N(0,1), in bounded chunks."""
    import torch
    flat = t.view(-1)
    g = torch.Generator(device=t.device)
    g.manual_seed(int(seed))
    for s in range(0, flat.numel(), chunk_elems):
        e = min(s + chunk_elems, flat.numel())
        flat[s:e] = torch.randn(e - s, generator=g, device=t.device, dtype=torch.float32).to(t.dtype)
    return t

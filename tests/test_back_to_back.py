"""Back-to-back launches of the tensor-core kernels.

Every kernel of the library is launched with programmatic dependent launch.
In a run of launches on one stream (or a CUDA graph) the next launch's CTAs
therefore start while the previous launch's last CTAs still run, and a CTA
can land on an SM the moment the previous launch's CTA there leaves.  These
tests run each tensor-core kernel (the dense step, the cross K/V fill, the
encoder attention, the multi-head prompt prefill and the GQA prefill) eight
times back to back on a side stream and in a captured graph replayed five
times, and check that no bounded wait of any launch runs out and that the
result is the one a single call gives: bit for bit where the kernel's sums
have a fixed order, and within a few fp32 roundings for the dense step,
whose K-split partial sums meet in an unspecified order.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from kv_cache_decode_asr_gb300 import ops  # noqa: E402
from kv_cache_decode_asr_gb300 import synthetic as syn  # noqa: E402

from gpu_util import dev, new_err  # noqa: E402

REPS, REPLAYS = 8, 5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_decode_asr_gb300 import build
    build.build()
    ops.load()


def _back_to_back(call, outs):
    """Results after REPS launches on a side stream, then after REPLAYS
    replays of a graph of REPS launches."""
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for _ in range(REPS):
            call(s)
    s.synchronize()
    eager = [o.clone() for o in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(REPS):
            call(s)
    with torch.cuda.stream(s):
        for _ in range(REPLAYS):
            g.replay()
    s.synchronize()
    return eager, [o.clone() for o in outs]


def _same_bits(a, b):
    """Equal bit patterns (NaN included) of two f16 or fp32 tensors."""
    as_int = {2: torch.int16, 4: torch.int32}[a.element_size()]
    return torch.equal(a.contiguous().view(as_int), b.contiguous().view(as_int))


LINEAR_CASES = [
    # M, N, K, norm, swiglu: the decoder shapes with the most K splits
    (32, 3840, 1280, "ln", False),    # Large-Whisper LayerNorm + qkv
    (16, 12288, 2048, "rms", False),  # Qwen3-ASR RMSNorm + gate/up (two waves)
    (16, 2048, 6144, None, True),     # Qwen3-ASR SwiGLU + down
    (32, 1280, 5120, None, False),    # Large-Whisper fc2
]


@pytest.mark.parametrize("M,N,K,norm,swiglu", LINEAR_CASES)
def test_linear_back_to_back(M, N, K, norm, swiglu):
    seed = 9100 + N
    x = dev(syn.host_normal_f32((M, 2 * K if swiglu else K), seed))
    w = dev((syn.host_normal_f32((N, K), seed + 1) * np.float32(K ** -0.5)).astype(
        np.float16).view(np.uint16))
    bias = dev(syn.host_normal_f32(N, seed + 2, std=0.5))
    g = dev(syn.host_normal_f32(K, seed + 3, mean=1.0, std=0.2))
    b = dev(syn.host_normal_f32(K, seed + 4, std=0.2))
    kw = {"ln": (g, b)} if norm == "ln" else ({"rms": g} if norm == "rms" else {})
    ws = ops.linear_workspace(M, N, K)
    err = new_err()
    y = torch.full((M, N), float("nan"), device="cuda")

    def call(stream=None):
        ops.asr_linear(x, w, y, bias=bias, swiglu=swiglu, mode="store", ws=ws, dev_err=err,
                       stream=stream, **kw)

    call()
    torch.cuda.synchronize()
    ref = y.clone()
    assert int(err.item()) == 0
    for got in _back_to_back(call, [y]):
        d = float((got[0] - ref).abs().max())
        scale = float(ref.abs().max())
        assert np.isfinite(d) and d <= 1e-5 * scale, f"M={M} N={N} K={K}: {d:.3e} of {scale:.3e}"
    assert int(err.item()) == 0
    if ws is not None:
        assert int(ws.count_nonzero().item()) == 0  # every launch left the workspace zero


def test_cross_fill_back_to_back():
    G, frames, d, cap = 2, 1500, 1280, 1504
    enc = dev(syn.host_normal_f16bits((G, frames, d), 9200))
    w = dev((syn.host_normal_f32((2 * d, d), 9201) * np.float32(d ** -0.5)).astype(
        np.float16).view(np.uint16))
    bias = dev(syn.host_normal_f32(d, 9202))
    cross = torch.zeros(G, cap, 2 * d, dtype=torch.float16, device="cuda")
    err = new_err()

    def call(stream=None):
        ops.asr_cross_kv_fill(enc, w, bias, cross, frames=frames, dev_err=err, stream=stream)

    call()
    torch.cuda.synchronize()
    ref = cross.clone()
    for got in _back_to_back(call, [cross]):
        assert _same_bits(got[0], ref)
    assert int(err.item()) == 0


def test_encoder_attn_back_to_back():
    B, T, H, hd = 2, 1500, 20, 64
    q, k, v = (dev(syn.host_normal_f16bits((B, T, H * hd), 9300 + i)) for i in range(3))
    out = torch.full((B, T, H * hd), float("nan"), device="cuda")
    ws = ops.workspace(ops.OP_ENCODER_ATTN, B, H, 1, H, hd, T)
    err = new_err()

    def call(stream=None):
        ops.asr_encoder_attn(q, k, v, H, hd, hd ** -0.5, out, ws, dev_err=err, stream=stream)

    call()
    torch.cuda.synchronize()
    ref = out.clone()
    for got in _back_to_back(call, [out]):
        assert _same_bits(got[0], ref)
    assert int(err.item()) == 0


def test_mha_prefill_back_to_back():
    """Per-sequence lengths (the V-transpose prep, then the attention)."""
    B, T, H, hd, cap = 6, 448, 20, 64, 448
    q, k, v = (dev(syn.host_normal_f16bits((B, T, H * hd), 9400 + i)) for i in range(3))
    lens = dev(np.array([1, 100, 128, 129, 300, 448], np.int32))
    cache = torch.zeros(B, cap, 2 * H * hd, dtype=torch.float16, device="cuda")
    out = torch.full((B, T, H * hd), float("nan"), device="cuda")
    ws = ops.workspace(ops.OP_MHA_PREFILL, B, H, 1, H, hd, T)
    err = new_err()

    def call(stream=None):
        ops.asr_mha_prefill(q, k, v, H, hd, hd ** -0.5, cache, cap, out, ws, lens=lens,
                            dev_err=err, stream=stream)

    call()
    torch.cuda.synchronize()
    ref_out, ref_cache = out.clone(), cache.clone()
    for got in _back_to_back(call, [out, cache]):
        assert _same_bits(got[0], ref_out)
        assert _same_bits(got[1], ref_cache)
    assert int(err.item()) == 0


def test_gqa_prefill_back_to_back():
    B, T, Hq, Hkv, HD, cap = 2, 640, 16, 8, 128, 640
    q = dev(syn.host_normal_f16bits((B, T, Hq * HD), 9500))
    k = dev(syn.host_normal_f16bits((B, T, Hkv * HD), 9501))
    v = dev(syn.host_normal_f16bits((B, T, Hkv * HD), 9502))
    wq = dev(syn.host_normal_f32(HD, 9503, 1.0, 0.1))
    wk = dev(syn.host_normal_f32(HD, 9504, 1.0, 0.1))
    cache = torch.zeros(B, cap, 2 * Hkv * HD, dtype=torch.float16, device="cuda")
    out = torch.full((B, T, Hq * HD), float("nan"), device="cuda")
    ws = ops.workspace(ops.OP_PREFILL_ATTN, B, Hkv, 1, Hq, HD, T)
    err = new_err()

    def call(stream=None):
        ops.asr_prefill_attn(q, k, v, wq, wk, 1e-6, 1e6, Hq, Hkv, HD, HD ** -0.5, cache, cap,
                             out, ws, dev_err=err, stream=stream)

    call()
    torch.cuda.synchronize()
    ref_out, ref_cache = out.clone(), cache.clone()
    for got in _back_to_back(call, [out, cache]):
        assert _same_bits(got[0], ref_out)
        assert _same_bits(got[1], ref_cache)
    assert int(err.item()) == 0

"""GPU parity of the batched causal prefill (tcgen05 path) against the oracle.

The cache rows written are compared bit for bit for V and within one f16 ulp
(plus the fp32 evaluation error of RMSNorm + RoPE) for the roped K; the
attention output with the fp32 attention tolerance.  Small cases compare
every output; the full Qwen3-ASR prefill (8 x 1536 tokens) compares sampled
rows that the oracle computes one by one from its own normed/roped queries.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from kv_cache_decode_asr_gb300 import ops  # noqa: E402
from kv_cache_decode_asr_gb300 import synthetic as syn  # noqa: E402

from gpu_util import assert_attn_close, dev, f16_ulp, host, host_u16, new_err  # noqa: E402

K_FP32_SLACK = 2e-6
HD = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_decode_asr_gb300 import build
    build.build()
    ops.load()
    oracle.build()
    oracle.set_threads(16)


def _inputs(B, T, Hq, Hkv, cap, seed):
    q = syn.host_normal_f16bits((B, T, Hq * HD), seed)
    k = syn.host_normal_f16bits((B, T, Hkv * HD), seed + 1)
    v = syn.host_normal_f16bits((B, T, Hkv * HD), seed + 2)
    wq = syn.host_normal_f32(HD, seed + 3, 1.0, 0.1)
    wk = syn.host_normal_f32(HD, seed + 4, 1.0, 0.1)
    cache0 = syn.host_normal_f16bits((B, cap, 2 * Hkv * HD), seed + 5)
    return q, k, v, wq, wk, cache0


def _run(q, k, v, wq, wk, cache0, Hq, Hkv):
    B, T = q.shape[0], q.shape[1]
    cap = cache0.shape[1]
    cache = dev(cache0)
    out = torch.full((B, T, Hq * HD), float("nan"), device="cuda")
    ws = ops.workspace(ops.OP_PREFILL_ATTN, B, Hkv, 1, Hq, HD, T)
    err = new_err()
    ops.asr_prefill_attn(dev(q), dev(k), dev(v), dev(wq), dev(wk), 1e-6, 1e6, Hq, Hkv, HD,
                         HD ** -0.5, cache, cap, out, ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return host(out), host_u16(cache)


def _check_cache(got, ref, cache0, T, Hkv):
    half = Hkv * HD
    assert np.array_equal(got[:, T:], cache0[:, T:])                 # rows past T untouched
    assert np.array_equal(got[:, :T, half:], ref[:, :T, half:])      # V copied bitwise
    kg = got[:, :T, :half].view(np.float16).astype(np.float64)
    kr = ref[:, :T, :half].view(np.float16).astype(np.float64)
    excess = np.abs(kg - kr) - f16_ulp(ref[:, :T, :half])
    assert excess.max() <= K_FP32_SLACK, f"roped K off by {excess.max():.3e} beyond 1 ulp"


@pytest.mark.parametrize("B,T,Hq,Hkv,cap", [
    (1, 128, 2, 1, 128),      # one tile, capacity == T
    (2, 200, 4, 2, 256),      # ragged second tile
    (1, 1, 2, 2, 8),          # a single token
    (3, 300, 16, 8, 320),     # the Qwen3-ASR head layout, three tiles
    (2, 384, 8, 8, 384),      # MHA, three full tiles
])
def test_prefill_matches_oracle(B, T, Hq, Hkv, cap):
    q, k, v, wq, wk, cache0 = _inputs(B, T, Hq, Hkv, cap, 700 + T + Hq)
    got, cache_gpu = _run(q, k, v, wq, wk, cache0, Hq, Hkv)
    ref_cache = cache0.copy()
    ref, _ = oracle.prefill_attn(q, k, v, wq, wk, 1e-6, 1e6, Hq, Hkv, HD, HD ** -0.5, ref_cache)
    _check_cache(cache_gpu, ref_cache, cache0, T, Hkv)
    assert_attn_close(got, ref, f"prefill B={B} T={T} Hq={Hq} Hkv={Hkv}")


def test_prefill_repeat_is_identical():
    B, T, Hq, Hkv, cap = 2, 256, 4, 2, 256
    q, k, v, wq, wk, cache0 = _inputs(B, T, Hq, Hkv, cap, 790)
    a, ca = _run(q, k, v, wq, wk, cache0, Hq, Hkv)
    b, cb = _run(q, k, v, wq, wk, cache0, Hq, Hkv)
    assert np.array_equal(a, b) and np.array_equal(ca, cb)


def test_prefill_full_qwen3_asr_sampled():
    """The full configuration (B=8, T=1536 = 16 prefix + 1500 audio + 20
    suffix, 16/8 heads of 128) in the launch configuration the benchmark
    times; sampled outputs computed one by one by the oracle."""
    cfg = syn.WORKLOADS["qwen3_asr_prefill_b8"]
    B, T, Hq, Hkv, cap = cfg["B"], cfg["T"], cfg["q_heads"], cfg["kv_heads"], cfg["capacity"]
    q, k, v, wq, wk, cache0 = _inputs(B, T, Hq, Hkv, cap, 800)
    got, cache_gpu = _run(q, k, v, wq, wk, cache0, Hq, Hkv)
    ref_cache = cache0.copy()
    qhat = oracle.prefill_prep(q, k, v, wq, wk, 1e-6, 1e6, Hq, Hkv, HD, ref_cache)
    _check_cache(cache_gpu, ref_cache, cache0, T, Hkv)
    r = syn.rng(801)
    ts = np.unique(np.concatenate([[0, 1, 15, 16, 127, 128, 129, 1515, 1535],
                                   r.integers(0, T, 23)])).astype(np.int32)
    for (b, h) in [(0, 0), (3, 5), (7, 15), (5, 8)]:
        rows = oracle.prefill_attn_rows(qhat[b, ts, h * HD:(h + 1) * HD], ts, ref_cache[b], Hq, Hkv,
                                        HD, h, HD ** -0.5)
        assert_attn_close(got[b, ts, h * HD:(h + 1) * HD], rows, f"prefill b={b} h={h}")
    # one (sequence, head) pair whole: every one of its 1536 rows, element-wise
    b, h = 2, 9
    all_t = np.arange(T, dtype=np.int32)
    rows = oracle.prefill_attn_rows(qhat[b, :, h * HD:(h + 1) * HD], all_t, ref_cache[b], Hq, Hkv,
                                    HD, h, HD ** -0.5)
    assert_attn_close(got[b, :, h * HD:(h + 1) * HD], rows, f"prefill b={b} h={h}, all rows")
    assert np.all(np.isfinite(got))

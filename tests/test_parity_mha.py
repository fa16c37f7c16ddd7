"""GPU parity of the multi-head prompt prefill and the encoder's unmasked
self-attention (tcgen05 path, head_dim 64 and 128, per-sequence lengths)
against the oracle.

Cache rows are compared bit for bit (they are copies); outputs with the fp32
attention tolerance.  Rows at or past a sequence's length must stay as they
were (NaN sentinels for out, the initial random bytes for the cache).  The
full-size cases compare sampled rows, which the oracle computes through its
one-query self and cross steps (pinned equal to rows of its prefill and
encoder attention).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from kv_cache_decode_asr_gb300 import ops  # noqa: E402
from kv_cache_decode_asr_gb300 import synthetic as syn  # noqa: E402

from gpu_util import assert_attn_close, dev, host, host_u16, new_err  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_decode_asr_gb300 import build
    build.build()
    ops.load()
    oracle.build()
    oracle.set_threads(16)


def _inputs(B, T, H, hd, seed):
    q = syn.host_normal_f16bits((B, T, H * hd), seed)
    k = syn.host_normal_f16bits((B, T, H * hd), seed + 1)
    v = syn.host_normal_f16bits((B, T, H * hd), seed + 2)
    return q, k, v


def _run_prefill(q, k, v, H, hd, lens, cache0):
    B, T = q.shape[0], q.shape[1]
    cap = cache0.shape[1]
    cache = dev(cache0)
    out = torch.full((B, T, H * hd), float("nan"), device="cuda")
    ws = ops.workspace(ops.OP_MHA_PREFILL, B, H, 1, H, hd, T)
    err = new_err()
    ops.asr_mha_prefill(dev(q), dev(k), dev(v), H, hd, hd ** -0.5, cache, cap, out, ws,
                        lens=None if lens is None else dev(lens), dev_err=err)
    torch.cuda.synchronize()
    return host(out), host_u16(cache), int(err.item())


def _run_encoder(q, k, v, H, hd, lens):
    B, T = q.shape[0], q.shape[1]
    out = torch.full((B, T, H * hd), float("nan"), device="cuda")
    ws = ops.workspace(ops.OP_ENCODER_ATTN, B, H, 1, H, hd, T)
    err = new_err()
    ops.asr_encoder_attn(dev(q), dev(k), dev(v), H, hd, hd ** -0.5, out, ws,
                         lens=None if lens is None else dev(lens), dev_err=err)
    torch.cuda.synchronize()
    return host(out), int(err.item())


def _lens_of(B, T, lens):
    return np.full(B, T, np.int32) if lens is None else np.asarray(lens, np.int32)


CASES = [
    (1, 128, 2, 64, None),                 # one tile
    (2, 200, 3, 64, [200, 77]),            # ragged tiles, a short sequence
    (3, 300, 6, 64, [1, 129, 300]),        # one token, a tile and a key past it, full
    (2, 384, 4, 128, [384, 250]),          # head_dim 128, three tiles
    (1, 1, 2, 64, None),                   # a single position
    (2, 260, 20, 64, [0, 260]),            # Whisper-large heads; an empty sequence
    (3, 128, 4, 64, [0, 0, 0]),            # every sequence empty: no work at all
    (37, 300, 5, 64, [(7 * i * i + 3 * i) % 301 for i in range(37)]),  # > 32 sequences
]


@pytest.mark.parametrize("B,T,H,hd,lens", CASES)
def test_mha_prefill_matches_oracle(B, T, H, hd, lens):
    q, k, v = _inputs(B, T, H, hd, 900 + T + H + hd)
    cap = T + 5
    cache0 = syn.host_normal_f16bits((B, cap, 2 * H * hd), 950 + T)
    got, cache_gpu, err = _run_prefill(q, k, v, H, hd, None if lens is None else np.array(lens, np.int32), cache0)
    assert err == 0
    ref_cache = cache0.copy()
    ref, bad = oracle.mha_attn(q, k, v, H, hd, hd ** -0.5, True, lens=lens, cache=ref_cache)
    assert bad == 0
    assert np.array_equal(cache_gpu, ref_cache)            # rows < L copied, the rest untouched
    L = _lens_of(B, T, lens)
    for b in range(B):
        assert np.all(np.isnan(got[b, L[b]:]))              # rows past the length not written
        if L[b]:
            assert_attn_close(got[b, :L[b]], ref[b, :L[b]], f"prefill b={b} T={T} H={H} hd={hd}")


@pytest.mark.parametrize("B,T,H,hd,lens", CASES)
def test_encoder_attn_matches_oracle(B, T, H, hd, lens):
    q, k, v = _inputs(B, T, H, hd, 1900 + T + H + hd)
    got, err = _run_encoder(q, k, v, H, hd, None if lens is None else np.array(lens, np.int32))
    assert err == 0
    ref, bad = oracle.mha_attn(q, k, v, H, hd, hd ** -0.5, False, lens=lens)
    assert bad == 0
    L = _lens_of(B, T, lens)
    for b in range(B):
        assert np.all(np.isnan(got[b, L[b]:]))
        if L[b]:
            assert_attn_close(got[b, :L[b]], ref[b, :L[b]], f"encoder b={b} T={T} H={H} hd={hd}")


def test_bad_length_is_flagged_and_skipped():
    B, T, H, hd = 2, 130, 2, 64
    q, k, v = _inputs(B, T, H, hd, 2990)
    got, err = _run_encoder(q, k, v, H, hd, np.array([T + 1, 64], np.int32))
    assert err & ops.DEVERR_LEN
    assert np.all(np.isnan(got[0]))
    ref, _ = oracle.mha_attn(q, k, v, H, hd, hd ** -0.5, False, lens=[0, 64])
    assert_attn_close(got[1, :64], ref[1, :64], "encoder beside a bad length")


def test_prefill_bad_length_is_flagged_and_skipped():
    """The prompt prefill with a length past T: flagged, that sequence
    skipped (no cache rows, output untouched), the other one correct."""
    B, T, H, hd, cap = 2, 200, 4, 64, 256
    q, k, v = _inputs(B, T, H, hd, 2993)
    cache0 = syn.host_normal_f16bits((B, cap, 2 * H * hd), 2994)
    got, cache_gpu, err = _run_prefill(q, k, v, H, hd, np.array([T + 1, 150], np.int32), cache0)
    assert err & ops.DEVERR_LEN
    assert np.all(np.isnan(got[0]))
    assert np.array_equal(cache_gpu[0], cache0[0])
    ref_cache = cache0.copy()
    ref, _ = oracle.mha_attn(q, k, v, H, hd, hd ** -0.5, True, lens=[0, 150], cache=ref_cache)
    assert_attn_close(got[1, :150], ref[1, :150], "prefill beside a bad length")
    assert np.array_equal(cache_gpu[1], ref_cache[1])


def test_repeat_is_identical():
    B, T, H, hd = 2, 300, 4, 64
    q, k, v = _inputs(B, T, H, hd, 2995)
    a, _ = _run_encoder(q, k, v, H, hd, None)
    b, _ = _run_encoder(q, k, v, H, hd, None)
    assert np.array_equal(a, b, equal_nan=True)


def test_encoder_full_whisper_large_sampled():
    """Whisper-large encoder self-attention, 1500 frames x 20 heads of 64 per
    sequence, in the launch configuration the benchmark times; sampled rows
    against the oracle's one-query cross step over all frames."""
    cfg = syn.WORKLOADS["whisper_large_encoder_b8"]
    B, T, H, hd = cfg["B"], cfg["T"], cfg["heads"], cfg["head_dim"]
    q, k, v = _inputs(B, T, H, hd, 3000)
    got, err = _run_encoder(q, k, v, H, hd, None)
    assert err == 0 and np.all(np.isfinite(got))
    r = syn.rng(3001)
    for b in (0, B - 1):
        ts = np.unique(np.concatenate([[0, 127, 128, 1499], r.integers(0, T, 12)]))
        cross = np.ascontiguousarray(np.concatenate([k[b:b + 1], v[b:b + 1]], axis=2))
        qt = q[b, ts].view(np.float16).astype(np.float32)
        ref, _ = oracle.cross_attn_step(qt, cross, np.zeros(len(ts), np.int32), H, hd, hd ** -0.5)
        assert_attn_close(got[b, ts], ref, f"encoder b={b}")


def test_prefill_full_whisper_large_sampled():
    """Whisper-large prompt prefill, 32 prompts of up to 448 tokens with
    lengths uniform in [1, 448], 20 heads of 64; the cache rows bit for bit
    and sampled rows against the oracle's one-token self step."""
    cfg = syn.WORKLOADS["whisper_large_prefill_b32"]
    B, T, H, hd, cap = cfg["B"], cfg["T"], cfg["heads"], cfg["head_dim"], cfg["capacity"]
    q, k, v = _inputs(B, T, H, hd, 3100)
    lens = syn.lens_uniform(B, cfg["len_lo"], cfg["len_hi"], 3101)
    cache0 = syn.host_normal_f16bits((B, cap, 2 * H * hd), 3102)
    got, cache_gpu, err = _run_prefill(q, k, v, H, hd, lens, cache0)
    assert err == 0
    ref_cache = cache0.copy()
    for b in range(B):
        L = lens[b]
        ref_cache[b, :L, :H * hd] = k[b, :L]
        ref_cache[b, :L, H * hd:] = v[b, :L]
    assert np.array_equal(cache_gpu, ref_cache)
    r = syn.rng(3103)
    for b in (0, 7, B - 1):
        L = int(lens[b])
        ts = np.unique(np.concatenate([[0, L - 1], r.integers(0, L, 8)]))
        qt = q[b, ts].view(np.float16).astype(np.float32)
        ref, _ = oracle.self_attn_step(qt, np.ascontiguousarray(np.repeat(ref_cache[b:b + 1], len(ts), 0)),
                                       (ts + 1).astype(np.int32), H, hd, hd ** -0.5)
        assert_attn_close(got[b, ts], ref, f"prefill b={b}")
        assert np.all(np.isnan(got[b, L:]))

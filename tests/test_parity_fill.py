"""GPU parity of the cross K/V fill (tcgen05 GEMM, bias and f16 pack) against
the oracle.

The oracle sums the f16 products in double and rounds once; the kernel sums
them in fp32 on the tensor cores, adds the bias in fp32 and rounds once.  The
two f16 results may differ by one step where the exact value lies near a
rounding boundary, and by the fp32 summation error, bounded here by 1e-3
(K up to 1280 terms of size about d^-1/2).  Rows past `frames` must keep
their bytes.  The full Large-Whisper fill (32 utterances x 1500 frames,
d = 1280) compares sampled rows, which the oracle computes as a batch of
their own (the rows are independent).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from kv_cache_decode_asr_gb300 import ops  # noqa: E402
from kv_cache_decode_asr_gb300 import synthetic as syn  # noqa: E402

from gpu_util import dev, f16_ulp, host_u16, new_err  # noqa: E402

SUM_SLACK = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_decode_asr_gb300 import build
    build.build()
    ops.load()
    oracle.build()
    oracle.set_threads(16)


def _inputs(G, frames, d, seed):
    enc = syn.host_normal_f16bits((G, frames, d), seed)
    w = (syn.host_normal_f32((2 * d, d), seed + 1) * np.float32(d ** -0.5)).astype(np.float16).view(np.uint16)
    bias = syn.host_normal_f32(d, seed + 2)
    return enc, w, bias


def _run(enc, w, bias, cross0, frames):
    cross = dev(cross0)
    err = new_err()
    ops.asr_cross_kv_fill(dev(enc), dev(w), dev(bias), cross, frames=frames, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return host_u16(cross)


def _assert_rows_close(got, ref, what):
    g = got.view(np.float16).astype(np.float64)
    r = ref.view(np.float16).astype(np.float64)
    excess = np.abs(g - r) - f16_ulp(ref)
    assert np.all(np.isfinite(g)), f"{what}: non-finite"
    assert excess.max() <= SUM_SLACK, f"{what}: {excess.max():.3e} beyond 1 f16 ulp"


@pytest.mark.parametrize("G,frames,cap,d", [
    (1, 128, 128, 128),     # one tile each way
    (2, 200, 208, 128),     # a ragged frame tile; rows past frames keep their bytes
    (1, 1500, 1500, 384),   # Whisper-tiny: three column tiles, six K steps
    (3, 70, 80, 256),       # a partial single tile, the V half in the second column tile
])
def test_fill_matches_oracle(G, frames, cap, d):
    enc, w, bias = _inputs(G, frames, d, 4000 + d + frames)
    cross0 = syn.host_normal_f16bits((G, cap, 2 * d), 4001)
    got = _run(enc, w, bias, cross0, frames)
    ref = cross0.copy()
    oracle.cross_kv_fill(enc, w, bias, ref)
    assert np.array_equal(got[:, frames:], cross0[:, frames:])
    _assert_rows_close(got[:, :frames], ref[:, :frames], f"fill G={G} frames={frames} d={d}")


def test_fill_identity_weights_are_exact():
    """[I | I] weights: K rows are the encoder rows bit for bit; V rows are
    f16(enc + bias)."""
    G, frames, d = 2, 130, 128
    enc, _, bias = _inputs(G, frames, d, 4100)
    eye = np.zeros((2 * d, d), np.float32)
    eye[np.arange(d), np.arange(d)] = 1
    eye[d + np.arange(d), np.arange(d)] = 1
    w = eye.astype(np.float16).view(np.uint16)
    got = _run(enc, w, bias, np.zeros((G, frames, 2 * d), np.uint16), frames)
    assert np.array_equal(got[..., :d], enc)
    want = (enc.view(np.float16).astype(np.float32) + bias).astype(np.float16).view(np.uint16)
    assert np.array_equal(got[..., d:], want)


def test_fill_full_whisper_large_sampled():
    cfg = syn.WORKLOADS["whisper_large_cross_fill_b32"]
    G, frames, d = cfg["G"], cfg["frames"], cfg["d"]
    enc, w, bias = _inputs(G, frames, d, 4200)
    got = _run(enc, w, bias, np.zeros((G, frames, 2 * d), np.uint16), frames)
    r = syn.rng(4201)
    for g in (0, 17, G - 1):
        ts = np.unique(np.concatenate([[0, 127, 128, 1499], r.integers(0, frames, 8)]))
        ref = np.zeros((1, len(ts), 2 * d), np.uint16)
        oracle.cross_kv_fill(np.ascontiguousarray(enc[g:g + 1, ts]), w, bias, ref)
        _assert_rows_close(got[g, ts], ref[0], f"fill g={g}")

"""GPU parity of the fused beam reorder + append + self-attention step.

The fused call must equal, byte for byte in the destination cache and the
destination lengths, the oracle's beam reorder ("mlx-bun whisper.ts",
WhisperKvCache.rearrange: take along the batch axis) followed by its append
of the new row; its output must match the oracle's self-attention over the
reordered cache within the attention tolerance of gpu_util.  Destination
caches start filled with a marker pattern, so rows the call must leave alone
(past each beam's length, and every row of a skipped beam) are checked too.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from kv_cache_decode_asr_gb300 import ops  # noqa: E402
from kv_cache_decode_asr_gb300 import synthetic as syn  # noqa: E402

from gpu_util import assert_attn_close, dev, host, host_u16, new_err  # noqa: E402

MARK = 0x1357


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_decode_asr_gb300 import build
    build.build()
    ops.load()
    oracle.build()
    oracle.set_threads(8)


def _oracle_step(qkv, src, dst0, idx, lens_src, H, hd, cap):
    """Oracle composition: reorder one layer, append row L-1, attend."""
    d = H * hd
    ref = dst0.copy()
    lens_dst, bad = oracle.kv_rearrange(src[:, None], ref[:, None], idx, lens_src, cap)
    ref = np.ascontiguousarray(ref)
    oracle.kv_append(qkv[:, d:2 * d], qkv[:, 2 * d:], ref, lens_dst - 1, H, hd)
    out, bad_attn = oracle.self_attn_step(qkv, ref, lens_dst, H, hd, hd ** -0.5, q_stride=3 * d)
    return ref, lens_dst, out, bad


def _run(qkv, src_d, dst_d, idx, lens_src, H, hd, cap, ws=None, err=None):
    B = idx.shape[0]
    d = H * hd
    q = dev(qkv)
    out = torch.full((B, d), float("nan"), device="cuda")
    lens_dst = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    if ws is None:
        ws = ops.workspace(ops.OP_SELF_ATTN, B, B, 1, H, hd)
    ops.asr_self_attn_reorder_append_step(q[:, :d], q[:, d:2 * d], q[:, 2 * d:], src_d, dst_d,
                                          dev(idx), dev(lens_src), lens_dst, H, hd, cap,
                                          hd ** -0.5, out, ws, dev_err=err)
    torch.cuda.synchronize()
    return host(out), host(lens_dst)


REORDER_CASES = [
    # B, H, hd, cap, beam
    (64, 6, 64, 448, 5),      # Whisper-tiny beam search, 13 groups of 5
    (32, 20, 64, 448, 4),     # Large-Whisper head count
    (7, 3, 128, 50, 3),       # head_dim 128, ragged groups
    (5, 2, 64, 12, 5),        # short caches: single tiles
    (1, 6, 64, 448, 1),
]


@pytest.mark.parametrize("B,H,hd,cap,beam", REORDER_CASES)
def test_reorder_step_matches_oracle(B, H, hd, cap, beam):
    seed = 500 + B + H
    d = H * hd
    qkv = syn.host_normal_f32((B, 3 * d), seed)
    src = syn.host_normal_f16bits((B, cap, 2 * d), seed + 1)
    lens_src = syn.lens_uniform(B, 1, cap, seed + 2)
    lens_src[0] = 1                   # a beam with no history row
    lens_src[-1] = cap                # a full cache
    idx = syn.beam_permutation(B, beam, seed + 3)
    if B > 2:
        idx[1] = idx[0]               # two beams continue one hypothesis
        idx[2] = B - 1                # and one continues the full cache
    dst0 = np.full_like(src, MARK)
    ref, lens_ref, out_ref, bad = _oracle_step(qkv, src, dst0, idx, lens_src, H, hd, cap)
    assert bad == 0
    err = new_err()
    dst = dev(dst0)
    got, lens_got = _run(qkv, dev(src), dst, idx, lens_src, H, hd, cap, err=err)
    assert np.array_equal(lens_got, lens_ref)
    assert np.array_equal(host_u16(dst), ref)
    assert_attn_close(got, out_ref, f"reorder+append+self B={B} H={H} hd={hd}")
    assert int(err.item()) == 0


def test_reorder_step_layer_slices_and_repeat():
    """One layer of [B][layers][cap][row] caches (the sequence stride spans
    the layers); other layers stay untouched; a second call on the same
    workspace gives the same bits and leaves the counters at zero."""
    B, nl, H, hd, cap, layer = 20, 3, 6, 64, 448, 1
    d = H * hd
    qkv = syn.host_normal_f32((B, 3 * d), 520)
    src = syn.host_normal_f16bits((B, nl, cap, 2 * d), 521)
    lens_src = syn.lens_uniform(B, 1, cap, 522)
    idx = syn.beam_permutation(B, 5, 523)
    dst0 = np.full_like(src, MARK)
    ref_l, lens_ref, out_ref, bad = _oracle_step(qkv, np.ascontiguousarray(src[:, layer]),
                                                 np.ascontiguousarray(dst0[:, layer]), idx,
                                                 lens_src, H, hd, cap)
    assert bad == 0
    ref = dst0.copy()
    ref[:, layer] = ref_l
    src_d = dev(src)
    dst_d = dev(dst0)
    ws = ops.workspace(ops.OP_SELF_ATTN, B, B, 1, H, hd)
    err = new_err()
    outs = []
    for _ in range(2):
        got, lens_got = _run(qkv, src_d[:, layer], dst_d[:, layer], idx, lens_src, H, hd, cap,
                             ws=ws, err=err)
        assert np.array_equal(lens_got, lens_ref)
        assert np.array_equal(host_u16(dst_d), ref)
        assert_attn_close(got, out_ref, "reorder on a layer slice")
        outs.append(got)
    assert np.array_equal(outs[0], outs[1])
    assert int(err.item()) == 0
    start = (ws.data_ptr() + 255) // 256 * 256 - ws.data_ptr()
    cnt = np.frombuffer(host(ws[start:start + 4 * B]).tobytes(), dtype=np.int32)
    assert np.all(cnt == 0)


def test_reorder_step_bad_entries_skipped():
    """An index outside [0, B) or a source length outside [1, capacity] skips
    the beam: output row zero, lens_dst 0, its destination rows untouched."""
    B, H, hd, cap = 6, 2, 64, 30
    d = H * hd
    qkv = syn.host_normal_f32((B, 3 * d), 530)
    src = syn.host_normal_f16bits((B, cap, 2 * d), 531)
    lens_src = np.array([3, 30, 31, 0, 5, 1], np.int32)
    idx = np.array([1, 2, 3, 6, -1, 4], np.int32)
    dst0 = np.full_like(src, MARK)
    ref, lens_ref, out_ref, bad = _oracle_step(qkv, src, dst0, idx, lens_src, H, hd, cap)
    assert bad == 4 and list(lens_ref) == [30, 0, 0, 0, 0, 5]
    err = new_err()
    dst = dev(dst0)
    got, lens_got = _run(qkv, dev(src), dst, idx, lens_src, H, hd, cap, err=err)
    assert np.array_equal(lens_got, lens_ref)
    assert np.array_equal(host_u16(dst), ref)
    assert np.all(got[1:5] == 0)
    assert_attn_close(got, out_ref, "reorder with bad entries")
    assert int(err.item()) == ops.DEVERR_LEN | ops.DEVERR_INDEX


def test_reorder_step_rejects_overlap():
    B, H, hd, cap = 4, 2, 64, 16
    d = H * hd
    q = torch.zeros(B, 3 * d, device="cuda")
    cache = torch.zeros(B, cap, 2 * d, dtype=torch.float16, device="cuda")
    idx = torch.arange(B, dtype=torch.int32, device="cuda")
    lens = torch.ones(B, dtype=torch.int32, device="cuda")
    out = torch.zeros(B, d, device="cuda")
    ws = ops.workspace(ops.OP_SELF_ATTN, B, B, 1, H, hd)
    with pytest.raises(ops.AsrError) as e:
        ops.asr_self_attn_reorder_append_step(q[:, :d], q[:, d:2 * d], q[:, 2 * d:], cache, cache,
                                              idx, lens, lens.clone(), H, hd, cap, 1.0, out, ws)
    assert e.value.status == 4      # ASR_ERR_ALIAS: destination rows over the source rows
    other = torch.zeros_like(cache)
    with pytest.raises(ops.AsrError) as e:
        ops.asr_self_attn_reorder_append_step(q[:, :d], q[:, d:2 * d], q[:, 2 * d:], cache, other,
                                              idx, lens, lens, H, hd, cap, 1.0, out, ws)
    assert e.value.status == 4      # lens_dst over lens_src

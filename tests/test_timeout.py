"""The bounded waits of the decode kernel give up cleanly.

asr_debug_stall_next_decode arms one launch whose producer issues no copies,
so its pipeline waits can never complete; they run out after a short limit
(1 ms here).  The kernel must then return (nothing hangs), report
ASR_DEVERR_TIMEOUT, leave its workspace counters at zero, and the next call
on the same workspace (or the same fixed scratch, for the workspace-free
entry point) must match the oracle again.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from kv_cache_decode_asr_gb300 import ops  # noqa: E402
from kv_cache_decode_asr_gb300 import synthetic as syn  # noqa: E402

from gpu_util import assert_attn_close, dev, host, new_err  # noqa: E402

LIMIT_NS = 1_000_000


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_decode_asr_gb300 import build
    build.build()
    ops.load()
    oracle.build()


def _counters_zero(ws, n_src, heads):
    base = ws.data_ptr()
    off = (base + 255) // 256 * 256 - base
    n = (n_src * heads * 4 + 255) // 256 * 256
    return int(ws[off:off + n].count_nonzero().item()) == 0


@pytest.mark.parametrize("B,H,hd,cap", [(16, 6, 64, 448), (4, 8, 128, 2048)])
def test_self_attn_stall_times_out_then_recovers(B, H, hd, cap):
    d = H * hd
    q = syn.host_normal_f32((B, d), 900 + B)
    cache = syn.host_normal_f16bits((B, cap, 2 * d), 901 + B)
    lens = syn.lens_uniform(B, cap // 2, cap, 902 + B)
    ref, _ = oracle.self_attn_step(q, cache, lens, H, hd, hd ** -0.5)
    q_d, cache_d, lens_d = dev(q), dev(cache), dev(lens)
    ws = ops.workspace(ops.OP_SELF_ATTN, B, B, 1, H, hd)
    out = torch.full((B, d), float("nan"), device="cuda")
    err = new_err()
    ops.asr_debug_stall_next_decode(LIMIT_NS)
    ops.asr_self_attn_step(q_d, cache_d, lens_d, H, hd, cap, hd ** -0.5, out, ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ops.DEVERR_TIMEOUT
    assert _counters_zero(ws, B, H)
    err = new_err()
    ops.asr_self_attn_step(q_d, cache_d, lens_d, H, hd, cap, hd ** -0.5, out, ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attn_close(host(out), ref, "self-attention after a stalled call")


def test_gqa_stall_times_out_then_recovers():
    B, Hq, Hkv, hd, cap = 4, 16, 8, 128, 4224
    r = syn.rng(910)
    q = syn.host_normal_f32((B, Hq * hd), 911)
    kn = syn.host_normal_f32((B, Hkv * hd), 912)
    vn = syn.host_normal_f32((B, Hkv * hd), 913)
    wq = (1.0 + 0.1 * r.standard_normal(hd)).astype(np.float32)
    wk = (1.0 + 0.1 * r.standard_normal(hd)).astype(np.float32)
    cache0 = syn.host_normal_f16bits((B, cap, 2 * Hkv * hd), 914)
    n_past = syn.lens_uniform(B, 1024, 4096, 915)
    ref_cache = cache0.copy()
    ref, _ = oracle.gqa_step(q, kn, vn, wq, wk, 1e-6, 1e6, n_past, ref_cache, Hq, Hkv, hd,
                             hd ** -0.5)
    args = [dev(t) for t in (q, kn, vn, wq, wk)]
    n_past_d, cache = dev(n_past), dev(cache0)
    ws = ops.workspace(ops.OP_GQA_STEP, B, B, 1, Hq, hd)
    out = torch.full((B, Hq * hd), float("nan"), device="cuda")
    err = new_err()
    ops.asr_debug_stall_next_decode(LIMIT_NS)
    ops.asr_gqa_step(*args, 1e-6, 1e6, n_past_d, cache, cap, Hq, Hkv, hd, hd ** -0.5, out, ws,
                     dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ops.DEVERR_TIMEOUT
    assert _counters_zero(ws, B, Hq)
    err = new_err()
    ops.asr_gqa_step(*args, 1e-6, 1e6, n_past_d, cache, cap, Hq, Hkv, hd, hd ** -0.5, out, ws,
                     dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attn_close(host(out), ref, "GQA step after a stalled call")


def test_cross_stall_times_out_then_recovers():
    B, G, mb, H, hd, frames = 10, 2, 5, 6, 64, 1500
    group = syn.beam_groups(B, mb)
    q = syn.host_normal_f32((B, H * hd), 920)
    cross = syn.host_normal_f16bits((G, frames, 2 * H * hd), 921)
    ref, _ = oracle.cross_attn_step(q, cross, group, H, hd, hd ** -0.5)
    q_d, cross_d, group_d = dev(q), dev(cross), dev(group)
    ws = ops.workspace(ops.OP_CROSS_ATTN, B, G, mb, H, hd)
    out = torch.full((B, H * hd), float("nan"), device="cuda")
    err = new_err()
    ops.asr_debug_stall_next_decode(LIMIT_NS)
    ops.asr_cross_attn_step(q_d, cross_d, group_d, G, mb, H, hd, frames, hd ** -0.5, out, ws,
                            dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ops.DEVERR_TIMEOUT
    assert _counters_zero(ws, G, H)
    err = new_err()
    ops.asr_cross_attn_step(q_d, cross_d, group_d, G, mb, H, hd, frames, hd ** -0.5, out, ws,
                            dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attn_close(host(out), ref, "cross-attention after a stalled call")


def test_noalloc_stall_times_out_then_recovers():
    B, H, hd, cap = 16, 6, 64, 448
    d = H * hd
    q = syn.host_normal_f32((B, d), 930)
    cache = syn.host_normal_f16bits((B, cap, 2 * d), 931)
    lens = syn.lens_uniform(B, 1, cap, 932)
    ref, _ = oracle.self_attn_step(q, cache, lens, H, hd, hd ** -0.5)
    q_d, cache_d, lens_d = dev(q), dev(cache), dev(lens)
    out = torch.full((B, d), float("nan"), device="cuda")
    err = new_err()
    ops.asr_debug_stall_next_decode(LIMIT_NS)
    ops.asr_self_attn_step_noalloc(q_d, cache_d, lens_d, H, hd, cap, hd ** -0.5, out, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ops.DEVERR_TIMEOUT
    err = new_err()
    ops.asr_self_attn_step_noalloc(q_d, cache_d, lens_d, H, hd, cap, hd ** -0.5, out, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attn_close(host(out), ref, "workspace-free call after a stalled call")


def test_stall_rejects_bad_limits():
    with pytest.raises(ops.AsrError):
        ops.asr_debug_stall_next_decode(0)
    with pytest.raises(ops.AsrError):
        ops.asr_debug_stall_next_decode(3_000_000_000)

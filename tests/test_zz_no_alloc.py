"""Self-attention without a caller workspace.

asr_self_attn_step_noalloc serves callers that cannot allocate device memory
for a workspace: a plugin whose host owns every allocation and forbids
allocating while it enqueues work, or a real-time audio thread that must not
wait on an allocator.  The library keeps that entry point's scratch in a
fixed array in device memory.  These tests call it through the C ABI and
check it against the ordinary entry point (which takes a workspace) and
against the CPU oracle, on two calls in a row with different inputs, so that
whatever the first call left in the shared array cannot leak into the
second.

This file is collected last, so a run that stops at the first failure has
already run every other test; it passes both alone and after the others.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from kv_cache_decode_asr_gb300 import ops  # noqa: E402
from kv_cache_decode_asr_gb300 import synthetic as syn  # noqa: E402

from gpu_util import assert_attn_close, dev, host, new_err  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_decode_asr_gb300 import build
    build.build()
    ops.load()
    oracle.build()


def _inputs(B, H, hd, cap, seed):
    q = syn.host_normal_f32((B, 3 * H * hd), seed)          # rows of a [q|k|v] buffer
    cache = syn.host_normal_f16bits((B, cap, 2 * H * hd), seed + 1)
    lens = syn.lens_uniform(B, 1, cap, seed + 2)
    return q, cache, lens


@pytest.mark.parametrize("B,H,hd,cap", [(16, 6, 64, 448), (7, 4, 128, 300)])
def test_noalloc_matches_workspace_entry_on_two_calls(B, H, hd, cap):
    d = H * hd
    for seed in (500, 600):   # two calls in a row, different inputs
        qh, ch, lh = _inputs(B, H, hd, cap, seed + B)
        q, cache, lens = dev(qh), dev(ch), dev(lh)
        ws = ops.workspace(ops.OP_SELF_ATTN, B, B, 1, H, hd)
        ref = torch.empty(B, d, device="cuda")
        ops.asr_self_attn_step(q[:, :d], cache, lens, H, hd, cap, hd ** -0.5, ref, ws)
        got = torch.full((B, d), float("nan"), device="cuda")
        err = new_err()
        ops.asr_self_attn_step_noalloc(q[:, :d], cache, lens, H, hd, cap, hd ** -0.5, got,
                                       dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_attn_close(host(got), host(ref), f"no-alloc call seed={seed}")
        want, skipped = oracle.self_attn_step(qh, ch, lh, H, hd, hd ** -0.5, q_stride=3 * d)
        assert skipped == 0
        assert_attn_close(host(got), want, f"no-alloc call seed={seed} vs oracle")


def test_noalloc_rejects_problems_beyond_the_scratch():
    lib = ops.load()
    B, H, hd, cap = 2048, 64, 128, 16
    need = ops.asr_workspace_size(ops.OP_SELF_ATTN, B, B, 1, H, hd)
    assert need > ops.asr_noalloc_scratch_bytes()
    P = ctypes.c_void_p
    # aligned stand-in pointers: the call is rejected before touching them
    st = lib.asr_self_attn_step_noalloc(P(0x10000), 3 * H * hd, P(0x20000), cap * 2 * H * hd,
                                        P(0x30000), B, H, hd, cap, ctypes.c_float(0.1),
                                        P(0x40000), None, None)
    assert st == 7
    assert lib.asr_status_string(st) == b"problem needs more scratch than the fixed scratch array"

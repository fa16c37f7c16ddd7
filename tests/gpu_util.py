"""Helpers for the GPU parity tests: host <-> device copies of the same bytes
and the tolerance check.

Tolerance for fp32 attention outputs (from the path's stated bar): the
maximum absolute error over the compared outputs must be <= 2e-3 AND that
maximum divided by max(1e-6, max |reference|) must be <= 1e-2.  The integer
and byte paths (append, rearrange, appended V rows) must match bit for bit.
"""
import numpy as np
import torch

from kv_cache_decode_asr_gb300 import synthetic as syn

ABS_TOL = 2e-3
REL_TOL = 1e-2


def dev(x):
    """numpy array -> CUDA tensor with the same bytes (uint16 travels as f16)."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
    return torch.from_numpy(x).cuda()


def host_u16(t):
    """f16 CUDA tensor -> uint16 bit patterns."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host(t):
    return t.detach().cpu().numpy()


def max_err(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    if gpu.size == 0:
        return 0.0, 0.0
    err = float(np.abs(gpu - ref).max())
    return err, err / max(1e-6, float(np.abs(ref).max()))


def assert_attn_close(gpu, ref, what=""):
    gpu = np.asarray(gpu, np.float64)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    err, rel = max_err(gpu, ref)
    assert err <= ABS_TOL and rel <= REL_TOL, f"{what}: max abs err {err:.3e}, rel {rel:.3e}"
    return err


def f16_ulp(bits):
    """Spacing of binary16 values at each (finite) pattern."""
    v = np.abs(bits.view(np.float16).astype(np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -14)))
    return 2.0 ** (e - 10)


def new_err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def lo_plane_inputs(M, N, K, seed):
    """Activations +-2^e (1 + j 2^-13), e in [-2, 2], j in {3, 5}: the f16
    high part of each drops exactly 3 2^-13 2^e.  Weights f16 N(0, 1/K)."""
    r = syn.rng(seed)
    e = r.integers(-2, 3, (M, K)).astype(np.float64)
    j = np.where(r.integers(0, 2, (M, K)) == 0, 3.0, 5.0)
    sgn = np.where(r.integers(0, 2, (M, K)) == 0, -1.0, 1.0)
    x = (sgn * 2.0 ** e * (1.0 + j * 2.0 ** -13)).astype(np.float32)
    w = (syn.host_normal_f32((N, K), seed + 1) * np.float32(K ** -0.5)).astype(
        np.float16).view(np.uint16)
    return x, w

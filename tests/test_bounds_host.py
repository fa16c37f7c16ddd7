"""The GPU parity bounds separate a correct kernel from plausible mistakes.

Run on the CPU: each test simulates, in numpy double precision, what a
kernel with one specific mistake would return on the GPU test's own inputs,
and checks that the GPU test's bound rejects it, while the exact result
(rounded as the kernel's design rounds it) passes.
"""
import numpy as np
import pytest

import oracle
from gpu_util import lo_plane_inputs

LO_PLANE_BOUND = 2.0 ** -19
LO_PLANE_CASES = [(32, 1280, 1280), (16, 2048, 2048), (8, 512, 128)]


@pytest.fixture(scope="module", autouse=True)
def _oracle():
    oracle.build()


def _dec16(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


@pytest.mark.parametrize("M,N,K", LO_PLANE_CASES)
def test_remainder_plane_bound_rejects_plain_f16_activations(M, N, K):
    x, w = lo_plane_inputs(M, N, K, 7700 + K)
    W = _dec16(w)
    a = x.astype(np.float64)
    hi = x.astype(np.float16).astype(np.float64)
    lo = (x - hi.astype(np.float32)).astype(np.float16).astype(np.float64)
    assert np.array_equal(hi + lo, a)          # the two planes hold x exactly
    ref = oracle.linear(x, w, None, mode="store")
    s = np.abs(a) @ np.abs(W).T
    bound = LO_PLANE_BOUND * s + 1e-7
    # the two-plane product, summed in fp32 per 16-wide step as a tensor core would
    two_plane = np.zeros((M, N), np.float32)
    for k0 in range(0, K, 16):
        part = (hi[:, k0:k0 + 16] + lo[:, k0:k0 + 16]) @ W[:, k0:k0 + 16].T
        two_plane = (two_plane + part.astype(np.float32)).astype(np.float32)
    assert np.all(np.abs(two_plane - ref) <= bound)
    # the mistake: the remainder plane dropped
    hi_only = hi @ W.T
    assert np.any(np.abs(hi_only - ref) > bound)
    assert float((np.abs(hi_only - ref) / s).max()) > 4 * LO_PLANE_BOUND

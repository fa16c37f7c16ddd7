"""GPU parity of the decode entry points against the CPU oracle.

Every case draws seeded inputs once, sends the same bytes to the CUDA library
(through the C ABI) and to the oracle, and compares: bit-exact for the append
and the rearrange, the attention tolerance of gpu_util for fp32 outputs.
Sizes span several tiles and ragged tails; the Whisper and Qwen3-ASR shaped
layers run at their full sizes.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from kv_cache_decode_asr_gb300 import ops  # noqa: E402
from kv_cache_decode_asr_gb300 import synthetic as syn  # noqa: E402

from gpu_util import assert_attn_close, dev, f16_ulp, host, host_u16, new_err  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_decode_asr_gb300 import build
    build.build()
    ops.load()
    oracle.build()
    oracle.set_threads(8)


# ------------------------------------------------------------- append ----

def test_append_bit_exact():
    B, H, hd, cap = 6, 6, 64, 16
    d = H * hd
    r = syn.rng(100)
    qkv = syn.host_normal_f32((B, 3 * d), 101)
    qkv[0, d:d + 40] *= 1e5          # overflow to +-inf
    qkv[1, d:d + 40] *= 1e-6         # subnormals
    qkv[2, 2 * d:2 * d + 8] = [65504, 65519.99, 65520, -65520, 6e-8, 3e-8, 0.0, -0.0]
    cache0 = r.integers(0, 65536, size=(B, cap, 2 * d)).astype(np.uint16)
    slot = np.array([0, 15, 3, 16, -1, 7], np.int32)
    ref = cache0.copy()
    skipped = oracle.kv_append(qkv[:, d:2 * d], qkv[:, 2 * d:], ref, slot, H, hd)
    assert skipped == 2
    qkv_d = dev(qkv)
    cache = dev(cache0)
    err = new_err()
    ops.asr_kv_append(qkv_d[:, d:2 * d], qkv_d[:, 2 * d:], cache, dev(slot), H, hd, cap,
                      dev_err=err)
    torch.cuda.synchronize()
    assert np.array_equal(host_u16(cache), ref)
    assert int(err.item()) == ops.DEVERR_LEN


def test_append_hd128_gqa_row():
    B, Hkv, hd, cap = 3, 8, 128, 9
    r = syn.rng(102)
    k = syn.host_normal_f32((B, Hkv * hd), 103)
    v = syn.host_normal_f32((B, Hkv * hd), 104)
    cache0 = r.integers(0, 65536, size=(B, cap, 2 * Hkv * hd)).astype(np.uint16)
    slot = np.array([8, 0, 4], np.int32)
    ref = cache0.copy()
    oracle.kv_append(k, v, ref, slot, Hkv, hd)
    cache = dev(cache0)
    ops.asr_kv_append(dev(k), dev(v), cache, dev(slot), Hkv, hd, cap)
    torch.cuda.synchronize()
    assert np.array_equal(host_u16(cache), ref)


# ---------------------------------------------------------- rearrange ----

@pytest.mark.parametrize("B,nl,cap,row,beam", [(7, 3, 20, 768, 3), (64, 4, 448, 768, 5),
                                               (32, 2, 448, 2560, 1)])
def test_rearrange_bit_exact(B, nl, cap, row, beam):
    r = syn.rng(110 + B)
    src = r.integers(0, 65536, size=(B, nl, cap, row)).astype(np.uint16)
    lens = syn.lens_uniform(B, 1, cap, 111 + B)
    lens[0] = 1
    lens[-1] = cap
    idx = syn.beam_permutation(B, beam, 112)
    if beam > 1:
        idx[1] = idx[0]
    dst0 = np.full_like(src, 0x1357)
    ref = dst0.copy()
    lens_ref, bad = oracle.kv_rearrange(src, ref, idx, lens, cap)
    assert bad == 0
    dst = dev(dst0)
    lens_dst = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    err = new_err()
    ops.asr_kv_rearrange(dev(src), dst, dev(idx), dev(lens), lens_dst, nl, row, cap, dev_err=err)
    torch.cuda.synchronize()
    assert np.array_equal(host_u16(dst), ref)
    assert np.array_equal(host(lens_dst), lens_ref)
    assert int(err.item()) == 0


def test_rearrange_bad_entries_skipped():
    B, nl, cap, row = 5, 2, 12, 64
    r = syn.rng(120)
    src = r.integers(0, 65536, size=(B, nl, cap, row)).astype(np.uint16)
    lens = np.array([3, 12, 13, 0, 5], np.int32)
    idx = np.array([1, 2, 3, 5, -1], np.int32)
    ref = np.zeros_like(src)
    lens_ref, bad = oracle.kv_rearrange(src, ref, idx, lens, cap)
    assert bad == 4
    dst = dev(np.zeros_like(src))
    lens_dst = torch.full((B,), 99, dtype=torch.int32, device="cuda")
    err = new_err()
    ops.asr_kv_rearrange(dev(src), dst, dev(idx), dev(lens), lens_dst, nl, row, cap, dev_err=err)
    torch.cuda.synchronize()
    assert np.array_equal(host_u16(dst), ref)
    assert np.array_equal(host(lens_dst), lens_ref)
    assert int(err.item()) == ops.DEVERR_LEN | ops.DEVERR_INDEX


# ------------------------------------------------------- self-attention --

SELF_CASES = [
    # B, H, hd, cap, lens (None = uniform in [1, cap])
    (1, 6, 64, 448, [225]),
    (3, 2, 64, 40, [1, 40, 17]),
    (5, 3, 128, 300, None),
    (64, 6, 64, 448, None),
    (2, 20, 64, 448, [448, 1]),
    (33, 1, 128, 70, None),
    (32, 20, 64, 448, None),
    (1, 1, 64, 1, [1]),
]


def _self_case(B, H, hd, cap, lens, seed, q_stride_mult=3):
    d = H * hd
    qkv = syn.host_normal_f32((B, q_stride_mult * d), seed)
    cache = syn.host_normal_f16bits((B, cap, 2 * d), seed + 1)
    if lens is None:
        lens = syn.lens_uniform(B, 1, cap, seed + 2)
    return qkv, cache, np.asarray(lens, np.int32)


def _run_self(qkv, cache, lens, H, hd, cap, err=None, ws=None, out=None):
    B = lens.shape[0]
    q = dev(qkv)
    if out is None:
        out = torch.full((B, H * hd), float("nan"), device="cuda")
    if ws is None:
        ws = ops.workspace(ops.OP_SELF_ATTN, B, B, 1, H, hd)
    ops.asr_self_attn_step(q[:, :H * hd], dev(cache), dev(lens), H, hd, cap, hd ** -0.5, out, ws,
                           dev_err=err)
    torch.cuda.synchronize()
    return host(out)


@pytest.mark.parametrize("B,H,hd,cap,lens", SELF_CASES)
def test_self_attn_matches_oracle(B, H, hd, cap, lens):
    qkv, cache, lens = _self_case(B, H, hd, cap, lens, 200 + B + H)
    err = new_err()
    got = _run_self(qkv, cache, lens, H, hd, cap, err=err)
    ref, bad = oracle.self_attn_step(qkv, cache, lens, H, hd, hd ** -0.5, q_stride=qkv.shape[1])
    assert bad == 0
    assert_attn_close(got, ref, f"self B={B} H={H} hd={hd}")
    assert int(err.item()) == 0


def test_self_attn_bad_lengths_zeroed():
    B, H, hd, cap = 4, 2, 64, 30
    qkv, cache, _ = _self_case(B, H, hd, cap, [1] * B, 230)
    lens = np.array([0, 30, 31, -5], np.int32)
    err = new_err()
    got = _run_self(qkv, cache, lens, H, hd, cap, err=err)
    ref, bad = oracle.self_attn_step(qkv, cache, lens, H, hd, hd ** -0.5, q_stride=qkv.shape[1])
    assert bad == 3
    assert np.all(got[[0, 2, 3]] == 0)
    assert_attn_close(got, ref, "self with bad lengths")
    assert int(err.item()) == ops.DEVERR_LEN


def test_self_attn_repeat_calls_identical():
    """The workspace counters return to zero: a second call on the same
    workspace gives the same bits."""
    B, H, hd, cap = 16, 6, 64, 448
    qkv, cache, lens = _self_case(B, H, hd, cap, None, 240)
    ws = ops.workspace(ops.OP_SELF_ATTN, B, B, 1, H, hd)
    a = _run_self(qkv, cache, lens, H, hd, cap, ws=ws)
    b = _run_self(qkv, cache, lens, H, hd, cap, ws=ws)
    assert np.array_equal(a, b)
    start = (ws.data_ptr() + 255) // 256 * 256 - ws.data_ptr()   # the pointer the call used
    cnt = np.frombuffer(host(ws[start:start + 4 * B]).tobytes(), dtype=np.int32)
    assert np.all(cnt == 0)


@pytest.mark.parametrize("B,H,hd,cap,lens", SELF_CASES + [(4, 2, 64, 30, [1, 2, 29, 30])])
def test_self_attn_append_step_matches_oracle(B, H, hd, cap, lens):
    """Fused append + attend: the cache bytes equal the oracle's append, the
    output the oracle's attention over rows [0, lens)."""
    qkv, cache0, lens = _self_case(B, H, hd, cap, lens, 260 + B + H)
    d = H * hd
    ref_cache = cache0.copy()
    oracle.kv_append(qkv[:, d:2 * d], qkv[:, 2 * d:], ref_cache, lens - 1, H, hd)
    ref, bad = oracle.self_attn_step(qkv, ref_cache, lens, H, hd, hd ** -0.5, q_stride=3 * d)
    assert bad == 0
    q = dev(qkv)
    cache = dev(cache0)
    out = torch.full((B, d), float("nan"), device="cuda")
    ws = ops.workspace(ops.OP_SELF_ATTN, B, B, 1, H, hd)
    err = new_err()
    for _ in range(2):   # a repeat rewrites the same row and returns the same output
        ops.asr_self_attn_append_step(q[:, :d], q[:, d:2 * d], q[:, 2 * d:], cache, dev(lens), H,
                                      hd, cap, hd ** -0.5, out, ws, dev_err=err)
        torch.cuda.synchronize()
        assert np.array_equal(host_u16(cache), ref_cache)
        assert_attn_close(host(out), ref, f"self+append B={B} H={H} hd={hd}")
    assert int(err.item()) == 0


def test_self_attn_append_bad_lengths():
    B, H, hd, cap = 3, 2, 64, 20
    qkv, cache0, _ = _self_case(B, H, hd, cap, [1] * B, 270)
    lens = np.array([0, 21, 5], np.int32)
    d = H * hd
    q = dev(qkv)
    cache = dev(cache0)
    out = torch.full((B, d), float("nan"), device="cuda")
    ws = ops.workspace(ops.OP_SELF_ATTN, B, B, 1, H, hd)
    err = new_err()
    ops.asr_self_attn_append_step(q[:, :d], q[:, d:2 * d], q[:, 2 * d:], cache, dev(lens), H, hd,
                                  cap, hd ** -0.5, out, ws, dev_err=err)
    torch.cuda.synchronize()
    got = host(out)
    assert np.all(got[:2] == 0) and int(err.item()) == ops.DEVERR_LEN
    ref_cache = cache0.copy()
    oracle.kv_append(qkv[2:, d:2 * d], qkv[2:, 2 * d:], ref_cache[2:], lens[2:] - 1, H, hd)
    assert np.array_equal(host_u16(cache), ref_cache)      # rows of bad sequences untouched


# ------------------------------------------------------ cross-attention --

CROSS_CASES = [
    # B, G, max_beams, H, hd, frames, group (None = b // beam)
    (1, 1, 1, 6, 64, 1500, None),
    (64, 13, 5, 6, 64, 1500, None),
    (10, 4, 4, 2, 64, 37, [0, 0, 0, 1, 1, 2, 2, 2, 2, 3]),
    (6, 3, 2, 4, 128, 300, [0, 0, 1, 1, 2, 2]),
    (32, 32, 1, 20, 64, 1500, None),
    (9, 2, 8, 1, 64, 5, [0] * 8 + [1]),
    (5, 7, 2, 3, 128, 250, [0, 2, 2, 5, 6]),   # groups with no beams are skipped
]


def _cross_case(B, G, H, hd, frames, seed):
    d = H * hd
    q = syn.host_normal_f32((B, d), seed)
    cross = syn.host_normal_f16bits((G, frames, 2 * d), seed + 1)
    return q, cross


def _run_cross(q, cross, group, G, mb, H, hd, frames, err=None):
    B = group.shape[0]
    out = torch.full((B, H * hd), float("nan"), device="cuda")
    ws = ops.workspace(ops.OP_CROSS_ATTN, B, G, mb, H, hd)
    ops.asr_cross_attn_step(dev(q), dev(cross), dev(group), G, mb, H, hd, frames, hd ** -0.5, out,
                            ws, dev_err=err)
    torch.cuda.synchronize()
    return host(out)


@pytest.mark.parametrize("B,G,mb,H,hd,frames,group", CROSS_CASES)
def test_cross_attn_matches_oracle(B, G, mb, H, hd, frames, group):
    if group is None:
        group = syn.beam_groups(B, mb)
    group = np.asarray(group, np.int32)
    q, cross = _cross_case(B, G, H, hd, frames, 300 + B + G)
    err = new_err()
    got = _run_cross(q, cross, group, G, mb, H, hd, frames, err=err)
    ref, bad = oracle.cross_attn_step(q, cross, group, H, hd, hd ** -0.5)
    assert bad == 0
    assert_attn_close(got, ref, f"cross B={B} G={G} beams={mb}")
    assert int(err.item()) == 0


def test_cross_attn_bad_groups():
    B, G, H, hd, frames = 6, 3, 2, 64, 50
    q, cross = _cross_case(B, G, H, hd, frames, 330)
    # group id out of range on the last sequence; group 0 has 3 members > max_beams 2
    group = np.array([0, 0, 0, 1, 2, 3], np.int32)
    err = new_err()
    got = _run_cross(q, cross, group, G, 2, H, hd, frames, err=err)
    ref, _ = oracle.cross_attn_step(q, cross, np.array([0, 0, 0, 1, 2, 0], np.int32), H, hd,
                                    hd ** -0.5)
    assert np.all(got[2] == 0) and np.all(got[5] == 0)
    assert_attn_close(got[[0, 1, 3, 4]], ref[[0, 1, 3, 4]], "cross valid rows")
    assert int(err.item()) == ops.DEVERR_INDEX | ops.DEVERR_BEAMS
    # groups not sorted: everything is zeroed and flagged
    err = new_err()
    got = _run_cross(q, cross, np.array([1, 0, 0, 1, 2, 2], np.int32), G, 2, H, hd, frames, err=err)
    assert np.all(got == 0) and int(err.item()) == ops.DEVERR_INDEX
    # a negative group id before the first group: only that sequence is
    # skipped, and the members of group 0 are the sequences that follow it
    group = np.array([-1, 0, 0, 1, 2, 2], np.int32)
    err = new_err()
    got = _run_cross(q, cross, group, G, 2, H, hd, frames, err=err)
    ref, _ = oracle.cross_attn_step(q, cross, np.array([0, 0, 0, 1, 2, 2], np.int32), H, hd,
                                    hd ** -0.5)
    assert np.all(got[0] == 0) and int(err.item()) == ops.DEVERR_INDEX
    assert_attn_close(got[1:], ref[1:], "cross after a negative group id")


# ----------------------------------------------------------- GQA step ----

# fp32 evaluation error of the normed + roped key before its f16 rounding:
# a few float32 roundings of terms of magnitude <= ~4 (8 * 2^-24 * 4 ~ 2e-6).
K_FP32_SLACK = 2e-6

GQA_CASES = [
    # B, Hq, Hkv, hd, cap, n_past (None = uniform in [1024, 4096])
    (4, 16, 8, 128, 300, [0, 1, 150, 299]),
    (3, 4, 2, 64, 90, [89, 0, 45]),
    (16, 16, 8, 128, 4224, None),
    (2, 8, 1, 128, 64, [63, 10]),
    (5, 6, 6, 64, 33, [1, 2, 3, 31, 32]),
]


def _gqa_case(B, Hq, Hkv, hd, cap, seed):
    q = syn.host_normal_f32((B, Hq * hd), seed)
    kn = syn.host_normal_f32((B, Hkv * hd), seed + 1)
    vn = syn.host_normal_f32((B, Hkv * hd), seed + 2)
    wq = syn.host_normal_f32(hd, seed + 3, 1.0, 0.1)
    wk = syn.host_normal_f32(hd, seed + 4, 1.0, 0.1)
    cache = syn.host_normal_f16bits((B, cap, 2 * Hkv * hd), seed + 5)
    return q, kn, vn, wq, wk, cache


def _run_gqa(q, kn, vn, wq, wk, n_past, cache, cap, Hq, Hkv, hd, err=None):
    B = n_past.shape[0]
    out = torch.full((B, Hq * hd), float("nan"), device="cuda")
    ws = ops.workspace(ops.OP_GQA_STEP, B, B, 1, Hq, hd)
    cache_d = dev(cache)
    ops.asr_gqa_step(dev(q), dev(kn), dev(vn), dev(wq), dev(wk), 1e-6, 1e6, dev(n_past), cache_d,
                     cap, Hq, Hkv, hd, hd ** -0.5, out, ws, dev_err=err)
    torch.cuda.synchronize()
    return host(out), host_u16(cache_d)


@pytest.mark.parametrize("B,Hq,Hkv,hd,cap,n_past", GQA_CASES)
def test_gqa_step_matches_oracle(B, Hq, Hkv, hd, cap, n_past):
    q, kn, vn, wq, wk, cache0 = _gqa_case(B, Hq, Hkv, hd, cap, 400 + B + Hq)
    if n_past is None:
        n_past = syn.lens_uniform(B, 1024, 4096, 409)
    n_past = np.asarray(n_past, np.int32)
    err = new_err()
    got, cache_gpu = _run_gqa(q, kn, vn, wq, wk, n_past, cache0, cap, Hq, Hkv, hd, err=err)
    ref_cache = cache0.copy()
    ref, bad = oracle.gqa_step(q, kn, vn, wq, wk, 1e-6, 1e6, n_past, ref_cache, Hq, Hkv, hd,
                               hd ** -0.5)
    assert bad == 0
    assert int(err.item()) == 0
    assert_attn_close(got, ref, f"gqa B={B} Hq={Hq} Hkv={Hkv} hd={hd}")
    half = Hkv * hd
    for b in range(B):
        p = n_past[b]
        other = np.ones(cap, bool)
        other[p] = False
        assert np.array_equal(cache_gpu[b, other], cache0[b, other])      # nothing else touched
        assert np.array_equal(cache_gpu[b, p, half:], ref_cache[b, p, half:])  # V bitwise
        kg = cache_gpu[b, p, :half].view(np.float16).astype(np.float64)
        kr = ref_cache[b, p, :half].view(np.float16).astype(np.float64)
        # K within 1 f16 ulp of the oracle's rounding plus the fp32 evaluation
        # error of RMSNorm + rotation (absolute: it scales with the operands,
        # |x^| <= ~4, not with a result that cancellation made small)
        excess = np.abs(kg - kr) - f16_ulp(ref_cache[b, p, :half])
        worst = int(np.argmax(excess))
        assert excess[worst] <= K_FP32_SLACK, (f"b={b} p={p} K elem {worst}: gpu {kg[worst]!r} "
                                               f"ref {kr[worst]!r}")


def test_gqa_bad_positions():
    B, Hq, Hkv, hd, cap = 3, 4, 2, 128, 20
    q, kn, vn, wq, wk, cache0 = _gqa_case(B, Hq, Hkv, hd, cap, 450)
    n_past = np.array([20, -1, 5], np.int32)
    err = new_err()
    got, cache_gpu = _run_gqa(q, kn, vn, wq, wk, n_past, cache0, cap, Hq, Hkv, hd, err=err)
    ref_cache = cache0.copy()
    ref, bad = oracle.gqa_step(q, kn, vn, wq, wk, 1e-6, 1e6, n_past, ref_cache, Hq, Hkv, hd,
                               hd ** -0.5)
    assert bad == 2 and int(err.item()) == ops.DEVERR_LEN
    assert np.all(got[:2] == 0)
    assert_attn_close(got, ref, "gqa with bad positions")
    assert np.array_equal(cache_gpu[:2], cache0[:2])


def test_history_ready_gives_the_same_bits():
    """asr_set_history_ready(1): self, self + append, cross and GQA calls read
    their lengths, groups and history before the grid dependency wait.  Here
    the launch before each call is a fill of its output or workspace, which
    the promise allows, and every result must equal the default order's bit
    for bit (the beam-reorder entry never starts early; its own tests run
    with the default)."""
    B, H, hd, cap = 24, 6, 64, 300
    qkv, cache, lens = _self_case(B, H, hd, cap, None, 4100)
    q, cross = _cross_case(20, 4, H, hd, 1500, 4110)
    group = np.array([i // 5 for i in range(20)], np.int32)
    gq = _gqa_case(16, 16, 8, 128, 512, 4120)
    n_past = syn.lens_uniform(16, 1, 500, 4130)
    d = H * hd

    def self_append():
        qd = dev(qkv)
        c = dev(cache)
        out = torch.full((B, d), float("nan"), device="cuda")
        ws = ops.workspace(ops.OP_SELF_ATTN, B, B, 1, H, hd)
        ops.asr_self_attn_append_step(qd[:, :d], qd[:, d:2 * d], qd[:, 2 * d:], c, dev(lens), H,
                                      hd, cap, hd ** -0.5, out, ws)
        torch.cuda.synchronize()
        return host(out), host_u16(c)

    def run_all():
        return (_run_self(qkv, cache, lens, H, hd, cap), self_append(),
                _run_cross(q, cross, group, 4, 5, H, hd, 1500),
                _run_gqa(*gq[:5], n_past, gq[5], 512, 16, 8, 128))

    base = run_all()
    try:
        ops.asr_set_history_ready(True)
        early = run_all()
    finally:
        ops.asr_set_history_ready(False)
    flat = lambda r: [np.asarray(x) for x in (r[0], *r[1], r[2], *r[3])]
    for a, b in zip(flat(base), flat(early)):
        assert a.dtype == b.dtype and np.array_equal(a.view(np.uint8), b.view(np.uint8))
    assert ops.load().asr_set_history_ready(2) != 0  # 0 or 1 only

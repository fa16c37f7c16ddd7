"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every entry point include/asrkv.h declares,
and reject bad arguments on the host before touching CUDA.  Pointers passed
here are never dereferenced: every case returns before any device work.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "asrkv.h")

OK, INVALID, UNSUP, MISAL, ALIAS, WS, CUDA = range(7)


@pytest.fixture(scope="module")
def lib():
    from kv_cache_decode_asr_gb300 import build, ops
    build.build()
    return ops.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(asr_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["asr_kv_append", "asr_self_attn_step", "asr_self_attn_append_step",
              "asr_cross_attn_step", "asr_gqa_step", "asr_prefill_attn", "asr_prefill_prep",
              "asr_prefill_attention",
              "asr_kv_rearrange", "asr_workspace_size", "asr_status_string", "asr_version"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from kv_cache_decode_asr_gb300 import ops
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in ops.SIGNATURES, name


def test_status_strings_and_version(lib):
    assert lib.asr_version() >= 100
    for s in range(8):
        assert lib.asr_status_string(s)
    assert lib.asr_status_string(0) == b"ok"
    assert lib.asr_status_string(99) == b"unknown status"


P = ctypes.c_void_p
A16 = P(0x10000)  # 16-byte aligned stand-in pointers (never dereferenced)
A16b = P(0x20000)
A16c = P(0x30000)
MIS = P(0x10004)


def test_append_rejects(lib):
    f = lib.asr_kv_append
    # B out of range, head_dim not a multiple of 8, too many heads
    assert f(A16, A16, 768, A16b, 448 * 768, A16c, -1, 6, 64, 448, None, None) == INVALID
    assert f(A16, A16, 768, A16b, 448 * 768, A16c, 1, 6, 60, 448, None, None) == UNSUP
    assert f(A16, A16, 768, A16b, 448 * 768, A16c, 1, 65, 64, 448, None, None) == UNSUP
    # B == 0 is a no-op
    assert f(None, None, 0, None, 0, None, 0, 6, 64, 448, None, None) == OK
    # NULL, stride too small, misaligned pointer / stride
    assert f(None, A16, 1152, A16b, 448 * 768, A16c, 1, 6, 64, 448, None, None) == INVALID
    assert f(A16, A16, 300, A16b, 448 * 768, A16c, 1, 6, 64, 448, None, None) == INVALID
    assert f(A16, A16, 1152, A16b, 447 * 768, A16c, 1, 6, 64, 448, None, None) == INVALID
    assert f(MIS, A16, 1152, A16b, 448 * 768, A16c, 1, 6, 64, 448, None, None) == MISAL
    assert f(A16, A16, 1154, A16b, 448 * 768, A16c, 1, 6, 64, 448, None, None) == MISAL
    assert f(A16, A16, 1152, A16b, 448 * 768 + 4, A16c, 1, 6, 64, 448, None, None) == MISAL


def test_self_attn_rejects(lib):
    f = lib.asr_self_attn_step
    row = 2 * 6 * 64
    args = lambda **kw: [kw.get("q", A16), kw.get("qs", 1152), A16b, kw.get("ss", 448 * row), A16c,
                         kw.get("B", 2), kw.get("H", 6), kw.get("hd", 64), kw.get("cap", 448),
                         ctypes.c_float(0.125), kw.get("out", P(0x40000)), P(0x50000),
                         ctypes.c_size_t(1 << 20), None, None]
    assert f(*args(hd=96)) == UNSUP
    assert f(*args(H=65)) == UNSUP
    assert f(*args(B=2049)) == INVALID
    assert f(*args(cap=0)) == INVALID
    assert f(*args(q=None)) == INVALID
    assert f(*args(qs=100)) == INVALID
    assert f(*args(ss=447 * row)) == INVALID
    assert f(*args(q=MIS)) == MISAL
    assert f(*args(qs=1154)) == MISAL
    assert f(*args(out=P(0x40008))) == MISAL
    assert f(*args(B=0)) == OK


def test_cross_attn_rejects(lib):
    f = lib.asr_cross_attn_step
    row = 2 * 6 * 64
    args = lambda **kw: [A16, 1152, A16b, kw.get("gs", 1500 * row), A16c, kw.get("B", 10),
                         kw.get("G", 2), kw.get("mb", 5), 6, kw.get("hd", 64), kw.get("fr", 1500),
                         ctypes.c_float(0.125), P(0x40000), P(0x50000), ctypes.c_size_t(1 << 20),
                         None, None]
    assert f(*args(mb=9)) == UNSUP
    assert f(*args(mb=0)) == INVALID
    assert f(*args(G=0)) == INVALID
    assert f(*args(fr=0)) == INVALID
    assert f(*args(hd=32)) == UNSUP
    assert f(*args(gs=1499 * row)) == INVALID
    assert f(*args(gs=1500 * row + 2)) == MISAL


def test_gqa_rejects(lib):
    f = lib.asr_gqa_step
    row = 2 * 8 * 128
    args = lambda **kw: [A16, kw.get("qs", 2048), A16, A16, kw.get("kvs", 1024), A16, A16,
                         ctypes.c_float(kw.get("eps", 1e-6)),
                         ctypes.c_float(kw.get("base", 1e6)), A16c, A16b, kw.get("ss", 4224 * row),
                         4224, 16, kw.get("hq", 16), kw.get("hkv", 8), kw.get("hd", 128),
                         ctypes.c_float(0.088), P(0x40000), P(0x50000), ctypes.c_size_t(1 << 20),
                         None, None]
    assert f(*args(hq=12)) == UNSUP          # 12 % 8 != 0
    assert f(*args(hq=72, hkv=8)) == UNSUP   # group of 9 query heads
    assert f(*args(base=0.0)) == INVALID
    assert f(*args(eps=-1.0)) == INVALID
    assert f(*args(ss=4223 * row)) == INVALID
    assert f(*args(hd=96)) == UNSUP
    assert f(*args(qs=2044)) == INVALID      # q rows narrower than 16 heads x 128
    assert f(*args(kvs=1026)) == MISAL       # k/v row stride not a multiple of 4


def test_rearrange_rejects(lib):
    f = lib.asr_kv_rearrange
    row, cap, nl = 768, 448, 4
    seq = nl * cap * row
    src = 0x100000
    base = lambda **kw: [P(kw.get("src", src)), P(kw.get("dst", src + 64 * seq * 2)),
                         kw.get("ss", seq), kw.get("ls", cap * row), kw.get("nl", nl),
                         kw.get("row", row), cap, A16, A16b, A16c, kw.get("B", 64), None, None]
    assert f(*base(dst=src + 10 * seq * 2)) == ALIAS           # overlapping buffers
    assert f(*base(ls=cap * row - 8)) == INVALID
    assert f(*base(ss=seq - 8)) == INVALID
    assert f(*base(row=770, ls=cap * 776, ss=nl * cap * 776)) == MISAL
    assert f(*base(row=4)) == INVALID
    assert f(*base(B=0)) == OK
    assert f(*base(nl=1100)) in (INVALID, UNSUP)


def test_prefill_rejects(lib):
    f = lib.asr_prefill_attn
    row = 2 * 8 * 128
    args = lambda **kw: [A16, A16, A16, A16, A16, ctypes.c_float(1e-6), ctypes.c_float(1e6),
                         kw.get("B", 8), kw.get("T", 1536), 16, kw.get("hkv", 8), kw.get("hd", 128),
                         ctypes.c_float(0.088), A16b, kw.get("ss", 1536 * row),
                         kw.get("cap", 1536), P(0x40000), P(0x50000), ctypes.c_size_t(1 << 30),
                         None, None]
    assert f(*args(hd=64)) == UNSUP
    assert f(*args(hkv=32)) == UNSUP
    assert f(*args(T=1537)) == INVALID          # T beyond the capacity
    assert f(*args(T=0)) == INVALID
    assert f(*args(ss=1536 * row - 8)) == INVALID
    assert f(*args(ss=1536 * row + 4)) == MISAL
    assert f(*args(B=0)) == OK


def test_linear_rejects(lib):
    f = lib.asr_linear
    x, w, y = P(0x100000), P(0x200000), P(0x900000)

    def args(**kw):
        return [kw.get("x", x), kw.get("xs", 1280), kw.get("norm", 0), kw.get("g", None),
                kw.get("b", None), ctypes.c_float(1e-5), kw.get("act", 0), w, None,
                kw.get("M", 32), kw.get("N", 3840), kw.get("K", 1280), kw.get("mode", 0),
                kw.get("y", y), kw.get("ys", 3840), None, ctypes.c_size_t(0), None, None]

    assert f(*args(K=1000)) == UNSUP           # K not a multiple of 64
    assert f(*args(mode=3)) == INVALID
    assert f(*args(N=0)) == INVALID
    assert f(*args(xs=1000)) == INVALID        # row stride below K
    assert f(*args(ys=100)) == INVALID
    assert f(*args(norm=1, g=P(0x300000))) == INVALID  # LayerNorm weight without its bias
    assert f(*args(norm=2)) == INVALID         # RMSNorm without its weight
    assert f(*args(norm=3)) == INVALID
    assert f(*args(act=2)) == INVALID
    assert f(*args(act=1, norm=2, g=P(0x300000))) == UNSUP  # SwiGLU input takes no norm
    assert f(*args(act=1)) == INVALID          # SwiGLU rows hold 2K values: stride 1280 < 2560
    assert f(*args(norm=2, g=P(0x300000), K=64, xs=64)) == UNSUP  # a norm needs K >= 128
    assert f(*args(x=P(0x100004))) == MISAL
    assert f(*args(xs=1282)) == MISAL
    assert f(*args(y=P(0x100000 + 64))) == ALIAS  # y overlaps x
    assert f(*args(M=0)) == OK


def test_binding_signatures_match_header():
    """Every entry point the header declares has a ctypes signature in the
    binding with the same number of arguments (catches drift of the ABI)."""
    from kv_cache_decode_asr_gb300 import ops
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    protos = re.findall(r"^\s*(?:int|size_t|const char\*)\s+(asr_\w+)\s*\(([^;]*?)\)\s*;", text,
                        re.M | re.S)
    assert protos
    for name, params in protos:
        params = params.strip()
        n = 0 if params in ("", "void") else params.count(",") + 1
        assert name in ops.SIGNATURES, f"{name} has no binding"
        assert len(ops.SIGNATURES[name][1]) == n, f"{name}: header {n} args, binding " \
            f"{len(ops.SIGNATURES[name][1])}"


def test_linear_wrapper_checks_before_the_library():
    """The Python wrapper of asr_linear rejects CPU tensors and mismatched
    shapes before it calls the library."""
    torch = pytest.importorskip("torch")
    from kv_cache_decode_asr_gb300 import ops
    x = torch.zeros(4, 128)
    w = torch.zeros(256, 128, dtype=torch.float16)
    y = torch.zeros(4, 256)
    with pytest.raises(ValueError):
        ops.asr_linear(x, w, y)  # not CUDA tensors
    with pytest.raises(TypeError):
        ops.asr_linear(x.double(), w, y)

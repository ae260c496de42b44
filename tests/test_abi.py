"""The C-ABI library loads without a GPU, exports every entry point include/kv_int4.h declares, and
rejects invalid arguments on the host (these calls return before any CUDA work)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kv_int4.h")


@pytest.fixture(scope="module")
def lib():
    from int4_token_head_kv_gb300._build import build_library
    return ctypes.CDLL(build_library())


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kv_int[248]_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 8
    assert {"kv_int2_write", "kv_int2_paged_attention", "kv_int2_row_bytes"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in kv_int4.h but not exported"


def test_host_side_validation(lib):
    lib.kv_int4_write.restype = ctypes.c_int
    lib.kv_int4_write.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                          ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p]
    fake = 1 << 20   # never dereferenced: every call below fails validation first
    # head size 96 is not built
    assert lib.kv_int4_write(fake, fake, 1, 4, 2, 96, fake, fake, fake, 8, 16, None) == 2
    # block size must be 16
    assert lib.kv_int4_write(fake, fake, 1, 4, 2, 128, fake, fake, fake, 8, 32, None) == 2
    # fp32 inputs are not a cache-write dtype
    assert lib.kv_int4_write(fake, fake, 2, 4, 2, 128, fake, fake, fake, 8, 16, None) == 2
    # negative sizes / null pointers
    assert lib.kv_int4_write(fake, fake, 1, -1, 2, 128, fake, fake, fake, 8, 16, None) == 1
    assert lib.kv_int4_write(None, fake, 1, 4, 2, 128, fake, fake, fake, 8, 16, None) == 1
    # misaligned input
    assert lib.kv_int4_write(fake + 2, fake, 1, 4, 2, 128, fake, fake, fake, 8, 16, None) == 3
    # nothing to do
    assert lib.kv_int4_write(None, None, 1, 0, 2, 128, None, None, None, 8, 16, None) == 0
    # the INT8 comparator's write validates the same way (no signs argument)
    lib.kv_int8_write.restype = ctypes.c_int
    lib.kv_int8_write.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                                          ctypes.c_int32, ctypes.c_void_p]
    assert lib.kv_int8_write(fake, fake, 1, 4, 2, 96, fake, fake, 8, 16, None) == 2
    assert lib.kv_int8_write(fake, fake, 1, 4, 2, 128, fake, fake, 8, 32, None) == 2
    assert lib.kv_int8_write(fake, fake, 1, -1, 2, 128, fake, fake, 8, 16, None) == 1
    assert lib.kv_int8_write(fake, None, 1, 4, 2, 128, fake, fake, 8, 16, None) == 1
    assert lib.kv_int8_write(fake, fake + 8, 1, 4, 2, 128, fake, fake, 8, 16, None) == 3
    assert lib.kv_int8_write(None, None, 1, 0, 2, 128, None, None, 8, 16, None) == 0
    lib.kv_int8_row_bytes.restype = ctypes.c_int32
    assert lib.kv_int8_row_bytes(128) == 132 and lib.kv_int8_row_bytes(64) == 68
    # the INT2 write takes the INT4 write's arguments and validates them the same way
    lib.kv_int2_write.restype = ctypes.c_int
    lib.kv_int2_write.argtypes = lib.kv_int4_write.argtypes
    assert lib.kv_int2_write(fake, fake, 1, 4, 2, 96, fake, fake, fake, 8, 16, None) == 2
    assert lib.kv_int2_write(fake, fake, 1, 4, 2, 128, fake, fake, fake, 8, 32, None) == 2
    assert lib.kv_int2_write(fake, fake, 1, 4, 2, 128, fake, None, fake, 8, 16, None) == 1   # signs required
    assert lib.kv_int2_write(fake, fake, 1, 4, 2, 128, fake, fake, fake + 4, 8, 16, None) == 3
    assert lib.kv_int2_write(None, None, 1, 0, 2, 128, None, None, None, 8, 16, None) == 0
    lib.kv_int2_row_bytes.restype = ctypes.c_int32
    assert lib.kv_int2_row_bytes(128) == 36 and lib.kv_int2_row_bytes(64) == 20


def test_attention_validation_and_workspace_policy(lib):
    f = lib.kv_int4_paged_attention
    f.restype = ctypes.c_int
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    f.argtypes = [vp, ctypes.c_int, i64, i32, vp, i64, i32, i32, i32, vp, i32, vp, vp, i32, i32, i32, ctypes.c_float,
                  vp, i32, vp, ctypes.c_int, vp, ctypes.c_size_t, vp]
    fake = 1 << 20
    base = dict(q=fake, qd=1, nq=2, hq=32, cache=fake, nb=64, h=8, d=128, bs=16, bt=fake, mb=4, sl=fake, qsl=fake,
                ns=2, mql=1, msl=64, scale=0.088, signs=fake, seg=0, out=fake, od=2, ws=None, wsb=0, st=None)

    def call(**kw):
        a = dict(base, **kw)
        return f(*a.values())

    assert call(h=3, hq=24) == 2           # kv heads must be a power of two <= 8
    assert call(hq=48) == 2                # q heads per kv head must be a power of two <= 8
    assert call(d=80) == 2
    assert call(seg=24) == 2               # segment length must be a multiple of 16
    assert call(q=None) == 1
    assert call(out=fake + 4) == 3
    lib.kv_int4_attention_workspace_bytes.restype = ctypes.c_size_t
    lib.kv_int4_attention_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.kv_int4_attention_segment_len.restype = i32
    lib.kv_int4_attention_segment_len.argtypes = [i32, i32, i32]
    ws = lib.kv_int4_attention_workspace_bytes

    def a256(x):
        return (x + 255) // 256 * 256

    # 8 seqs x 131072 tokens in segments of 4096: per sequence its first segment index, its first
    # prefill query tile and its rotated-query record (8 kv heads x 128 x 8 (G = 8) or 4 fp16x2 words, then Hq logit factors
    # and Hq query sums); per segment 8 warps x (1024 accumulators for G = 8, 512 otherwise) and
    # 8 (max, sum) pairs
    units = 8 * 32
    for hq, acc, qw in ((64, 1024, 8), (32, 512, 4)):
        rec = (8 * 128 * qw + 2 * hq) * 4
        assert ws(hq, 8, 128, 8, 131072, 4096) == (2 * a256(9 * 4) + a256(8 * rec) + a256(units * 8 * acc * 4)
                                                   + units * 8 * 16 * 4)
    assert ws(32, 8, 128, 0, 4096, 0) == 0          # no sequences
    assert ws(32, 3, 128, 8, 4096, 0) == 0          # heads do not group
    assert call(msl=131072, seg=4096, mb=8192) == 4   # workspace required but missing
    assert lib.kv_int4_attention_segment_len(8, 131072, 4096) == 4096
    auto = lib.kv_int4_attention_segment_len(8, 131072, 0)
    assert auto % 32 == 0 and 32 <= auto <= 4096
    assert lib.kv_int4_attention_segment_len(1, 16, 0) == 32     # floor: one block pair
    assert lib.kv_int4_attention_segment_len(4096, 1 << 20, 0) == 4096   # ceiling


def test_options_validation(lib):
    class Opts(ctypes.Structure):
        _fields_ = [("window_left", ctypes.c_int32), ("softcap", ctypes.c_float), ("alibi_slopes", ctypes.c_void_p),
                    ("qq_bias", ctypes.c_void_p), ("qq_bias_stride", ctypes.c_int32)]

    f = lib.kv_int4_paged_attention_ex
    f.restype = ctypes.c_int
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    f.argtypes = [vp, ctypes.c_int, i64, i32, vp, i64, i32, i32, i32, vp, i32, vp, vp, i32, i32, i32, ctypes.c_float,
                  vp, i32, vp, ctypes.c_int, vp, ctypes.c_size_t, vp, ctypes.POINTER(Opts)]
    fake = 1 << 20
    base = dict(q=fake, qd=1, nq=16, hq=32, cache=fake, nb=64, h=8, d=128, bs=16, bt=fake, mb=4, sl=fake, qsl=fake,
                ns=2, mql=8, msl=64, scale=0.088, signs=fake, seg=0, out=fake, od=2, ws=None, wsb=0, st=None)

    def call(opts, **kw):
        a = dict(base, **kw)
        return f(*a.values(), ctypes.byref(opts))

    assert call(Opts(-1, -1.0, None, None, 0)) == 1                 # negative softcap
    assert call(Opts(-1, float("nan"), None, None, 0)) == 1         # non-finite softcap
    assert call(Opts(-1, 0.0, None, fake, 7)) == 1                  # qq_bias rows shorter than the chunks
    assert call(Opts(-1, 0.0, None, fake, 8), q=None) == 1          # stride accepted, then the usual checks
    assert call(Opts(-1, 0.0, None, fake, 8), nq=0) == 0


def test_int8_attention_validation(lib):
    f = lib.kv_int8_paged_attention
    f.restype = ctypes.c_int
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    f.argtypes = [vp, ctypes.c_int, i64, i32, vp, i64, i32, i32, i32, vp, i32, vp, vp, i32, i32, i32, ctypes.c_float,
                  i32, vp, ctypes.c_int, vp, ctypes.c_size_t, vp]
    fake = 1 << 20
    base = dict(q=fake, qd=1, nq=2, hq=32, cache=fake, nb=64, h=8, d=128, bs=16, bt=fake, mb=4, sl=fake, qsl=fake,
                ns=2, mql=1, msl=64, scale=0.088, seg=0, out=fake, od=2, ws=None, wsb=0, st=None)

    def call(**kw):
        a = dict(base, **kw)
        return f(*a.values())

    assert call(mql=2) == 2                # decode only: a chunk of several queries is not built
    assert call(h=3, hq=24) == 2
    assert call(d=96) == 2
    assert call(cache=None) == 1
    assert call(q=fake + 8) == 3
    assert call(msl=131072, seg=4096, mb=8192) == 4   # the INT4 call's workspace, required and missing
    assert call(nq=0) == 0


def test_int2_attention_validation(lib):
    f = lib.kv_int2_paged_attention
    f.restype = ctypes.c_int
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    f.argtypes = [vp, ctypes.c_int, i64, i32, vp, i64, i32, i32, i32, vp, i32, vp, vp, i32, i32, i32, ctypes.c_float,
                  vp, i32, vp, ctypes.c_int, vp, ctypes.c_size_t, vp]
    fake = 1 << 20
    base = dict(q=fake, qd=1, nq=2, hq=32, cache=fake, nb=64, h=8, d=128, bs=16, bt=fake, mb=4, sl=fake, qsl=fake,
                ns=2, mql=1, msl=64, scale=0.088, signs=fake, seg=0, out=fake, od=2, ws=None, wsb=0, st=None)

    def call(**kw):
        a = dict(base, **kw)
        return f(*a.values())

    assert call(mql=2) == 2                # decode only
    assert call(h=3, hq=24) == 2
    assert call(d=96) == 2
    assert call(signs=None) == 1           # rotated: the signs are required
    assert call(cache=fake + 8) == 3
    assert call(msl=131072, seg=4096, mb=8192) == 4
    assert call(nq=0) == 0


def test_status_strings(lib):
    lib.kv_int4_status_string.restype = ctypes.c_char_p
    for s in range(6):
        assert lib.kv_int4_status_string(s)
    assert lib.kv_int4_status_string(99) == b"unknown status"


def test_package_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "int4_token_head_kv_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, flags=re.M), fn
                assert "kv_int4_oracle" not in src, fn


def test_binding_requires_one_device():
    # the binding launches on its tensors' device, so tensors on two devices are refused before any call
    import torch
    from int4_token_head_kv_gb300 import _one_device
    a, b = torch.empty(2), torch.empty(2, device="meta")
    assert _one_device(a, None, a) == a.device
    with pytest.raises(ValueError):
        _one_device(a, b)

"""The C-ABI library builds, loads and exports what include/pa.h declares (no GPU).

Only host-side argument checks are exercised here: each call below is rejected
before any CUDA call is made.
"""
import ctypes
import os
import re

import pytest

import paged_kv_cache_306_gb300 as pa
from paged_kv_cache_306_gb300 import _binding as B
from paged_kv_cache_306_gb300 import build as pa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(pa_\w+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    return B.load()


# Every pointer these tests pass lies inside a buffer the test owns: 1 MiB of zeroed
# device memory when a GPU is present, else host memory (without a device no kernel
# can launch).  A host-side check that stopped rejecting its case would then launch
# on memory that exists, never on a made-up address.
_BUF = {}


@pytest.fixture(scope="module", autouse=True)
def _owned_buffer():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        t = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
        _BUF["base"], _BUF["keep"] = t.data_ptr(), t
    else:
        raw = (ctypes.c_ubyte * ((1 << 20) + 256))()
        _BUF["base"], _BUF["keep"] = (ctypes.addressof(raw) + 255) // 256 * 256, raw
    yield
    _BUF.clear()


def A(off):
    """Byte `off` of the owned buffer (off 0 stands for a null pointer)."""
    assert 0 <= off < (1 << 20)
    return ctypes.c_void_p(_BUF["base"] + off) if off else ctypes.c_void_p(0)


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for n in ("pa_reshape_and_cache", "pa_copy_blocks", "pa_decode", "pa_decode_workspace_size",
              "pa_decode_plan_partition", "pa_get_device_error", "pa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    # nothing else with the pa_ prefix leaks out as a C symbol
    raw = ctypes.CDLL(B.LIB_PATH)
    assert raw.pa_decode is not None


def test_status_strings(lib):
    assert lib.pa_status_string(0) == b"PA_OK"
    assert lib.pa_status_string(4) == b"PA_ERR_WORKSPACE"
    assert lib.pa_status_string(99) == b"PA_ERR_UNKNOWN"


def _decode(lib, **kw):
    a = dict(out=8192, q=8192, k=8192, v=8192, bt=8192, mb=4, sl=8192, S=1, msl=16, H=4, Hkv=4, D=128, bs=16,
             nb=8, scale=0.1, ps=0, ws=None, wsb=0, dt=B.PA_F16)
    a.update(kw)
    return lib.pa_decode(A(a["out"]), A(a["q"]), A(a["k"]), A(a["v"]), A(a["bt"]), a["mb"], A(a["sl"]), a["S"],
                         a["msl"], a["H"], a["Hkv"], a["D"], a["bs"], a["nb"], a["scale"], a["ps"], A(a["ws"] or 0),
                         a["wsb"], a["dt"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(H=6, Hkv=4), B.PA_ERR_INVALID_ARG),           # heads not a multiple of kv heads
    (dict(D=96), B.PA_ERR_UNSUPPORTED),                 # head size outside {64, 128}
    (dict(bs=8), B.PA_ERR_UNSUPPORTED),                 # block size outside {16, 32}
    (dict(msl=65), B.PA_ERR_INVALID_ARG),               # max_seq_len beyond the table width
    (dict(msl=0), B.PA_ERR_INVALID_ARG),
    (dict(ps=24), B.PA_ERR_INVALID_ARG),                # partition not a multiple of block_size
    (dict(ps=-2), B.PA_ERR_INVALID_ARG),
    (dict(dt=7), B.PA_ERR_INVALID_ARG),
    (dict(nb=0), B.PA_ERR_INVALID_ARG),
    (dict(S=-1), B.PA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), B.PA_ERR_INVALID_ARG),
    (dict(q=8200), B.PA_ERR_ALIGNMENT),                 # q not 16-byte aligned
    (dict(bt=8194), B.PA_ERR_ALIGNMENT),
    (dict(q=0), B.PA_ERR_INVALID_ARG),                  # null pointer
])
def test_decode_rejects_bad_arguments_on_the_host(lib, kw, status):
    assert _decode(lib, **kw) == status
    assert lib.pa_last_error_message()


def test_decode_with_no_sequences_is_a_no_op(lib):
    assert _decode(lib, S=0, q=0, out=0) == B.PA_OK


def test_workspace_size_is_zero_for_arguments_decode_rejects(lib):
    assert lib.pa_decode_workspace_size(2, 8, 2, 96, 70, 16, 0, B.PA_F16) == 0     # head size
    assert lib.pa_decode_workspace_size(2, 8, 3, 128, 70, 16, 0, B.PA_F16) == 0    # heads vs kv heads
    assert lib.pa_decode_workspace_size(2, 8, 2, 128, 70, 16, 24, B.PA_F16) == 0   # partition not a block multiple
    assert lib.pa_decode_workspace_size(0, 8, 2, 128, 70, 16, 0, B.PA_F16) == 0    # nothing to do


def test_plan_rejects_what_decode_rejects(lib):
    assert lib.pa_decode_plan_partition(1, 6, 4, 128, 100, 16, B.PA_F16) == -1
    assert lib.pa_decode_plan_partition(1, 4, 4, 96, 100, 16, B.PA_F16) == -1


def test_write_path_rejects_bad_arguments_on_the_host(lib):
    st = lib.pa_reshape_and_cache(A(16), A(16), A(16), A(16), A(16), 4, 2, 60, 16, 8, B.PA_F16, None)
    assert st == B.PA_ERR_INVALID_ARG                   # head size not a multiple of x
    st = lib.pa_reshape_and_cache(A(16), A(16), A(24), A(16), A(16), 4, 2, 64, 16, 8, B.PA_F16, None)
    assert st == B.PA_ERR_ALIGNMENT
    st = lib.pa_reshape_and_cache(None, None, None, None, None, 0, 2, 64, 16, 8, B.PA_F16, None)
    assert st == B.PA_OK                                # nothing to write
    st = lib.pa_copy_blocks(A(16), A(16), A(12), 3, 2, 64, 16, 8, B.PA_F16, None)
    assert st == B.PA_ERR_ALIGNMENT
    st = lib.pa_copy_blocks(A(16), A(16), A(16), 3, 2, 64, 16, 8, 5, None)
    assert st == B.PA_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 4, 128, dtype=torch.float16)
    with pytest.raises(pa.PAError):
        pa.pa_decode(q, q, torch.zeros(1, 4, 16, 16, 8, dtype=torch.float16),
                     torch.zeros(1, 4, 128, 16, dtype=torch.float16), torch.zeros(1, 1, dtype=torch.int32),
                     torch.ones(1, dtype=torch.int32), 0.1, 1)


def _decode_scaled(lib, **kw):
    a = dict(out=8192, q=8192, k=8192, v=8192, bt=8192, mb=4, sl=8192, S=1, msl=16, H=4, Hkv=2, D=128, bs=16,
             nb=8, scale=0.1, ps=0, ws=None, wsb=0, qdt=B.PA_F16, cdt=B.PA_FP8_E4M3, ks=0.5, vs=0.25)
    a.update(kw)
    return lib.pa_decode_scaled(A(a["out"]), A(a["q"]), A(a["k"]), A(a["v"]), A(a["bt"]), a["mb"], A(a["sl"]),
                                a["S"], a["msl"], a["H"], a["Hkv"], a["D"], a["bs"], a["nb"], a["scale"], a["ps"],
                                A(a["ws"] or 0), a["wsb"], a["qdt"], a["cdt"], a["ks"], a["vs"], None)


def test_plain_decode_refuses_an_fp8_cache(lib):
    # the FP8 cache needs the query dtype and the scales: pa_decode_scaled
    assert _decode(lib, dt=B.PA_FP8_E4M3) == B.PA_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw,status", [
    (dict(qdt=B.PA_F32), B.PA_ERR_UNSUPPORTED),          # FP8 cache read by fp32 queries
    (dict(qdt=B.PA_FP8_E4M3), B.PA_ERR_UNSUPPORTED),
    (dict(qdt=9), B.PA_ERR_INVALID_ARG),
    (dict(ks=0.0), B.PA_ERR_INVALID_ARG),
    (dict(vs=-1.0), B.PA_ERR_INVALID_ARG),
    (dict(ks=float("inf")), B.PA_ERR_INVALID_ARG),
    (dict(vs=float("nan")), B.PA_ERR_INVALID_ARG),
    (dict(cdt=B.PA_F16, qdt=B.PA_BF16, ks=1.0, vs=1.0), B.PA_ERR_INVALID_ARG),   # 16-bit cache, other queries
    (dict(cdt=B.PA_F16, ks=0.5, vs=1.0), B.PA_ERR_INVALID_ARG),                  # 16-bit cache, scale != 1
    (dict(D=96), B.PA_ERR_UNSUPPORTED),
    (dict(ps=24), B.PA_ERR_INVALID_ARG),
    (dict(q=8200), B.PA_ERR_ALIGNMENT),
])
def test_scaled_decode_rejects_bad_arguments_on_the_host(lib, kw, status):
    assert _decode_scaled(lib, **kw) == status
    assert lib.pa_last_error_message()


def test_scaled_decode_with_no_sequences_is_a_no_op(lib):
    assert _decode_scaled(lib, S=0, q=0, out=0) == B.PA_OK


def test_scaled_write_rejects_bad_arguments_on_the_host(lib):
    F8, F16 = B.PA_FP8_E4M3, B.PA_F16

    def w(key_dt=F16, cache_dt=F8, ks=0.5, vs=0.5, D=128, key=16, T=4):
        return lib.pa_reshape_and_cache_scaled(A(key), A(16), A(16), A(16), A(16), T, 2, D, 16, 8, key_dt, cache_dt,
                                               ks, vs, None)
    assert w(key_dt=F8) == B.PA_ERR_UNSUPPORTED           # codes are not a source dtype
    assert w(ks=0.0) == B.PA_ERR_INVALID_ARG
    assert w(vs=float("nan")) == B.PA_ERR_INVALID_ARG
    assert w(D=72) == B.PA_ERR_INVALID_ARG                # x = 16 codes per K row chunk
    assert w(key=24) == B.PA_ERR_ALIGNMENT
    assert w(cache_dt=F16, ks=0.5) == B.PA_ERR_INVALID_ARG   # a 16-bit cache takes no scales
    assert w(cache_dt=F16, key_dt=B.PA_BF16, ks=1.0, vs=1.0) == B.PA_ERR_INVALID_ARG
    assert w(T=0) == B.PA_OK


def test_prefill_rejects_bad_arguments_on_the_host(lib):
    def pf(dt=B.PA_F16, D=128, bs=16, T=8, q=8192, S=2, msl=64, mb=4, H=8, Hkv=2):
        return lib.pa_prefill(A(8192), A(q), A(8192), A(8192), A(8192), mb, A(8192), A(8192), S, T, msl, H, Hkv, D,
                              bs, 64, 0.1, dt, None)
    assert pf(dt=B.PA_F32) == B.PA_ERR_UNSUPPORTED       # tensor-core prefill: 16-bit caches
    assert pf(dt=B.PA_FP8_E4M3) == B.PA_ERR_UNSUPPORTED
    assert pf(D=96) == B.PA_ERR_UNSUPPORTED
    assert pf(bs=8) == B.PA_ERR_UNSUPPORTED
    assert pf(T=-1) == B.PA_ERR_INVALID_ARG
    assert pf(msl=65) == B.PA_ERR_INVALID_ARG
    assert pf(H=6, Hkv=4) == B.PA_ERR_INVALID_ARG
    assert pf(q=8200) == B.PA_ERR_ALIGNMENT
    assert pf(T=0) == B.PA_OK and pf(S=0) == B.PA_OK
    # null pointers: the row-count check comes first, and without it the null check would refuse
    big = lib.pa_prefill(None, None, None, None, None, 4, None, None, 2, 8, 64, 8, 2, 128, 16, 1 << 27, 0.1,
                         B.PA_F16, None)
    assert big == B.PA_ERR_UNSUPPORTED     # 2^27 blocks x 2 kv heads x 128 dims: past the V tensor map's rows


def test_fused_step_rejects_bad_arguments_on_the_host(lib):
    def st(dt=B.PA_F16, key=8192, value=8192, sd=8192, npairs=1, S=1, D=128, bs=16, msl=16, q=8192):
        return lib.pa_decode_step(A(8192), A(q), A(key), A(value), A(8192), A(8192), A(sd), npairs, A(8192), 4,
                                  A(8192), S, msl, 4, 4, D, bs, 8, 0.1, 0, None, 0, dt, None)
    assert st(dt=B.PA_FP8_E4M3) == B.PA_ERR_UNSUPPORTED   # an FP8 cache is written by the scaled write
    assert st(dt=7) == B.PA_ERR_UNSUPPORTED
    assert st(npairs=-1) == B.PA_ERR_INVALID_ARG
    assert st(sd=0) == B.PA_ERR_INVALID_ARG                # pairs without an array
    assert st(sd=8196) == B.PA_ERR_ALIGNMENT
    assert st(key=0) == B.PA_ERR_INVALID_ARG
    assert st(value=8200) == B.PA_ERR_ALIGNMENT
    assert st(D=96) == B.PA_ERR_UNSUPPORTED                # the decode checks follow
    assert st(msl=65) == B.PA_ERR_INVALID_ARG
    assert st(q=8200) == B.PA_ERR_ALIGNMENT
    assert st(S=0, npairs=0, key=0, value=0, q=0) == B.PA_OK
    assert lib.pa_last_error_message()


def test_scaled_fused_step_rejects_bad_arguments_on_the_host(lib):
    def st(qdt=B.PA_F16, cdt=B.PA_FP8_E4M3, ks=0.5, vs=0.5, key=8192, S=1):
        return lib.pa_decode_step_scaled(A(8192), A(8192), A(key), A(8192), A(8192), A(8192), None, 0, A(8192), 4,
                                         A(8192), S, 16, 4, 4, 128, 16, 8, 0.1, 0, None, 0, qdt, cdt, ks, vs, None)
    assert st(qdt=B.PA_F32) == B.PA_ERR_UNSUPPORTED       # an FP8 pool is read by fp16 or bf16 queries
    assert st(ks=0.0) == B.PA_ERR_INVALID_ARG
    assert st(vs=float("inf")) == B.PA_ERR_INVALID_ARG
    assert st(cdt=B.PA_F16, ks=1.0, vs=1.0, qdt=B.PA_BF16) == B.PA_ERR_INVALID_ARG  # 16-bit pool: the query's dtype
    assert st(cdt=B.PA_F16, ks=0.5, vs=1.0) == B.PA_ERR_INVALID_ARG                 # and scales 1
    assert st(cdt=9) == B.PA_ERR_UNSUPPORTED
    assert st(key=8200) == B.PA_ERR_ALIGNMENT
    assert st(S=0, key=0) == B.PA_OK


def test_shared_decode_rejects_bad_arguments_on_the_host(lib):
    def sd(key=8192, value=8192, sd_=0, npairs=0, grp=8192, blk=8192, S=2, cdt=B.PA_F16, qdt=B.PA_F16, D=128):
        return lib.pa_decode_shared(A(8192), A(8192), A(key), A(value), A(8192), A(8192), A(sd_), npairs, A(8192), 4,
                                    A(8192), A(grp), A(blk), S, 16, 8, 2, D, 16, 8, 0.1, 0, None, 0, qdt, cdt, 1.0,
                                    1.0, None)
    assert sd(grp=0) == B.PA_ERR_INVALID_ARG                    # no group description
    assert sd(blk=0) == B.PA_ERR_INVALID_ARG
    assert sd(key=0) == B.PA_ERR_INVALID_ARG                    # key without value
    assert sd(key=0, value=0, npairs=1, sd_=8192) == B.PA_ERR_INVALID_ARG   # copies without a step
    assert sd(grp=8194) == B.PA_ERR_ALIGNMENT
    assert sd(cdt=9) == B.PA_ERR_UNSUPPORTED
    assert sd(D=96) == B.PA_ERR_UNSUPPORTED
    assert sd(S=0, grp=0, blk=0) == B.PA_OK
    assert lib.pa_decode_shared_workspace_size(4, 8, 2, 96, 64, 16, 0, B.PA_F16) == 0


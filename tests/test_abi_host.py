"""Host-side checks of the C ABI (no GPU needed).

The library must load on a machine without a GPU, export every function that
``include/gdn.h`` declares, and reject bad arguments on the host with the
documented status, before touching CUDA. Fault injection happens here, on the
host: bad sizes, null and misaligned pointers, unsupported head sizes and
chunk sizes, aliasing output.
"""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "gdn.h"
HEADERS = sorted((ROOT / "include").glob("*.h"))

OK, INVALID, UNSUPPORTED, MISALIGNED, CUDA = 0, -1, -2, -3, -4


def declared_functions(headers=None):
    names = set()
    for h in headers or HEADERS:
        text = re.sub(r"/\*.*?\*/", "", h.read_text(), flags=re.S)
        names.update(re.findall(
            r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(gdn_\w+)\s*\(",
            text, flags=re.M))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions([HEADER])
    for required in ("gdn_chunk_fwd", "gdn_chunk_fwd_f32", "gdn_chunk_fwd_ex",
                     "gdn_recurrent_step", "gdn_status_string",
                     "gdn_timing_enable", "gdn_timing_read"):
        assert required in names
    assert "gdn_selftest_mma" in declared_functions()


def test_library_loads_and_exports_every_declared_symbol(lib):
    so = lib.library()
    for name in declared_functions():
        assert hasattr(so, name), f"{name} declared in gdn.h but not exported"


def test_status_strings(lib):
    assert lib.gdn_status_string(OK) == "GDN_OK"
    assert lib.gdn_status_string(MISALIGNED) == "GDN_ERR_MISALIGNED"
    assert lib.gdn_status_string(12345) == "GDN_UNKNOWN_STATUS"


# Fake device addresses: never dereferenced because every call below fails a
# host check first.
A = 0x7F0000000000  # 16-byte aligned
ODD = A + 4


def chunk(so, q=A, k=A + 0x1000, v=A + 0x2000, g=A + 0x3000, beta=A + 0x4000,
          h0=None, out=A + 0x5000, hT=None, cu=None, B=1, H=1, T=64, dk=64,
          dv=64, C=64, **ex):
    if ex:
        return so.gdn_chunk_fwd_ex(q, k, v, g, beta, h0, out, hT, cu, B, H, T,
                                   dk, dv, C, ex.get("dtype", 0),
                                   ex.get("variant", 0), ex.get("path", 0),
                                   ex.get("sp_parts", 0), None)
    return so.gdn_chunk_fwd(q, k, v, g, beta, h0, out, hT, cu, B, H, T, dk, dv,
                            C, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), INVALID),
    (dict(out=None), INVALID),
    (dict(g=None), INVALID),
    (dict(B=-1), INVALID),
    (dict(H=0), INVALID),
    (dict(T=-5), INVALID),
    (dict(dk=96), UNSUPPORTED),
    (dict(dv=32), UNSUPPORTED),
    (dict(C=32), UNSUPPORTED),
    (dict(C=128), UNSUPPORTED),
    (dict(q=ODD), MISALIGNED),
    (dict(beta=ODD), MISALIGNED),
    (dict(h0=ODD), MISALIGNED),
    (dict(hT=ODD), MISALIGNED),
    (dict(cu=ODD, B=2), MISALIGNED),
    (dict(out=A), INVALID),              # out aliases q
    (dict(cu=A + 0x6000, B=0), INVALID),  # packed batch needs >= 1 sequence
    (dict(variant=7), INVALID),
    (dict(path=9), INVALID),
    (dict(path=0x300), INVALID),         # chain and scan both requested
    (dict(path=0x400), INVALID),         # unknown flag
    (dict(dtype=5), INVALID),
    (dict(sp_parts=-1), INVALID),
    (dict(dtype=1, path=2), UNSUPPORTED),  # tensor-core path is bf16 only
    (dict(dtype=1, path=3), UNSUPPORTED),
    (dict(dtype=1, path=4), UNSUPPORTED),
    (dict(dtype=1, path=5), UNSUPPORTED),
    (dict(path=5, dv=32), UNSUPPORTED),    # tensor-core shapes only
    (dict(path=5, dk=128, dv=128, sp_parts=3), UNSUPPORTED),  # no split
    (dict(path=6), INVALID),
])
def test_chunk_fwd_rejects_on_host(lib, kw, expect):
    assert chunk(lib.library(), **kw) == expect


def test_empty_batch_is_a_no_op(lib):
    assert chunk(lib.library(), B=0) == OK
    # T = 0 with dense batches: nothing to do, but arguments still checked
    assert chunk(lib.library(), T=0, dk=96) == UNSUPPORTED


@pytest.mark.parametrize("kw,expect", [
    (dict(N=-1), INVALID), (dict(H=0), INVALID), (dict(dk=80), UNSUPPORTED),
    (dict(state=None), INVALID), (dict(q=ODD), MISALIGNED),
    (dict(out=A), INVALID),
])
def test_recurrent_step_rejects_on_host(lib, kw, expect):
    a = dict(q=A, k=A + 0x100, v=A + 0x200, g=A + 0x300, beta=A + 0x400,
             state=A + 0x500, out=A + 0x600, N=2, H=2, dk=64, dv=64)
    a.update(kw)
    so = lib.library()
    rc = so.gdn_recurrent_step(a["q"], a["k"], a["v"], a["g"], a["beta"],
                               a["state"], a["out"], a["N"], a["H"], a["dk"],
                               a["dv"], None)
    assert rc == expect


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(1, 4, 1, 64, dtype=torch.bfloat16)
    gb = torch.zeros(1, 4, 1)
    with pytest.raises(ValueError, match="CUDA"):
        lib.gdn_chunk_fwd(x, x, x, gb, gb)


def test_launch_counter_is_monotone(lib):
    a = lib.kernel_counters()
    chunk(lib.library(), B=0)
    assert lib.kernel_counters() == a


def test_timing_switch_and_read_on_host(lib):
    """Per-kernel timing: switching and reading need no GPU while nothing
    has been timed; an unknown kernel family is rejected."""
    so = lib.library()
    n = ctypes.c_ulonglong(7)
    ms = ctypes.c_double(7.0)
    assert so.gdn_timing_enable(1) == OK
    for k in range(lib.GDN_KERNEL_COUNT):
        assert so.gdn_timing_read(k, ctypes.byref(n), ctypes.byref(ms)) == OK
        assert n.value == 0 and ms.value == 0.0
    assert so.gdn_timing_read(lib.GDN_KERNEL_COUNT, None, None) == INVALID
    assert so.gdn_timing_read(-1, None, None) == INVALID
    assert so.gdn_timing_enable(0) == OK
    assert lib.kernel_timings() == {}


def fused(so, q=A, k=A + 0x1000, v=A + 0x2000, a=A + 0x3000, b=A + 0x4000,
          h0=None, out=A + 0x5000, hT=None, cu=None, w=A + 0x7000,
          gate=A + 0x8000, eps=1e-6, B=1, H=1, T=64, dk=128, dv=128, C=64,
          path=0):
    return so.gdn_chunk_fwd_fused(q, k, v, a, b, h0, out, hT, cu, w, gate,
                                  ctypes.c_float(eps), B, H, T, dk, dv, C,
                                  path, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), INVALID),
    (dict(eps=-1.0), INVALID),
    (dict(eps=float("nan")), INVALID),
    (dict(dk=64), UNSUPPORTED),          # the tensor-core path's shapes only
    (dict(dv=32), UNSUPPORTED),
    (dict(w=ODD), MISALIGNED),
    (dict(gate=ODD), MISALIGNED),
    (dict(gate=A + 0x5000), INVALID),    # gate aliases out
    (dict(C=32), UNSUPPORTED),
    (dict(path=1), UNSUPPORTED),         # no fp32 CUDA-core fused path
    (dict(path=6), INVALID),
    (dict(path=-1), INVALID),
])
def test_fused_rejects_on_host(lib, kw, expect):
    assert fused(lib.library(), **kw) == expect


def test_fused_empty_batch_is_a_no_op(lib):
    assert fused(lib.library(), B=0) == OK


def kda(so, q=A, k=A + 0x1000, v=A + 0x2000, g=A + 0x3000, b=A + 0x4000,
        h0=None, out=A + 0x5000, hT=None, cu=None, B=1, H=1, T=16, dk=128,
        dv=128):
    return so.gdn_kda_fwd(q, k, v, g, b, h0, out, hT, cu, B, H, T, dk, dv, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(B=-1), INVALID), (dict(H=0), INVALID), (dict(T=-1), INVALID),
    (dict(q=None), INVALID), (dict(dk=96), UNSUPPORTED),
    (dict(dv=32), UNSUPPORTED), (dict(g=ODD), MISALIGNED),
    (dict(h0=ODD), MISALIGNED), (dict(out=A), INVALID),
    (dict(cu=A + 0x6000, B=0), INVALID),
])
def test_kda_rejects_on_host(lib, kw, expect):
    assert kda(lib.library(), **kw) == expect


def test_kda_empty_batch_is_a_no_op(lib):
    assert kda(lib.library(), B=0) == OK


def kda_ex(so, path=0, sp=0, **kw):
    a = dict(q=A, k=A + 0x1000, v=A + 0x2000, g=A + 0x3000, b=A + 0x4000,
             h0=None, out=A + 0x5000, hT=None, cu=None, B=1, H=1, T=16,
             dk=128, dv=128)
    a.update(kw)
    return so.gdn_kda_fwd_ex(a["q"], a["k"], a["v"], a["g"], a["b"], a["h0"],
                             a["out"], a["hT"], a["cu"], a["B"], a["H"],
                             a["T"], a["dk"], a["dv"], path, sp, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(path=-1), INVALID), (dict(path=6), INVALID),
    (dict(path=5), UNSUPPORTED),                 # single-launch form: GDN only
    (dict(path=0x300), INVALID), (dict(path=0x400), INVALID),
    (dict(path=3), UNSUPPORTED),                 # split chain: scalar gate only
    (dict(path=2, dk=64), UNSUPPORTED),          # chunk form: dk = 128 only
    (dict(path=4, dv=32), UNSUPPORTED),
    (dict(path=2, q=None), INVALID), (dict(path=2, out=A), INVALID),
    (dict(path=2, sp=-1), INVALID), (dict(path=2, g=ODD), MISALIGNED),
    (dict(path=0, dk=96), UNSUPPORTED), (dict(path=1, B=-1), INVALID),
])
def test_kda_ex_rejects_on_host(lib, kw, expect):
    assert kda_ex(lib.library(), **kw) == expect


@pytest.mark.parametrize("path", [0, 1, 2, 4])
def test_kda_ex_empty_batch_is_a_no_op(lib, path):
    assert kda_ex(lib.library(), path=path, B=0) == OK


def bwd(so, fn="gdn_chunk_bwd", **kw):
    a = dict(q=A, k=A + 0x1000, v=A + 0x2000, g=A + 0x3000, b=A + 0x4000,
             h0=None, do=A + 0x5000, dhT=None, dq=A + 0x6000, dk=A + 0x7000,
             dv=A + 0x8000, dg=A + 0x9000, db=A + 0xa000, dh0=None, cu=None,
             B=1, H=1, T=16, dk_=128, dv_=128)
    a.update(kw)
    extra = ((a.get("variant", 0),) if fn in ("gdn_chunk_bwd", "gdn_chunk_bwd_f32")
             else ())
    return getattr(so, fn)(a["q"], a["k"], a["v"], a["g"], a["b"], a["h0"],
                           a["do"], a["dhT"], a["dq"], a["dk"], a["dv"],
                           a["dg"], a["db"], a["dh0"], a["cu"], a["B"], a["H"],
                           a["T"], a["dk_"], a["dv_"], *extra, None)


@pytest.mark.parametrize("fn", ["gdn_chunk_bwd", "gdn_kda_bwd", "gdn_chunk_bwd_f32",
                                "gdn_chunk_bwd_chunked"])
@pytest.mark.parametrize("kw,expect", [
    (dict(B=-1), INVALID), (dict(H=0), INVALID), (dict(T=-1), INVALID),
    (dict(q=None), INVALID), (dict(do=None), INVALID), (dict(dg=None), INVALID),
    (dict(dk_=96), UNSUPPORTED), (dict(dv_=32), UNSUPPORTED),
    (dict(B=70000), UNSUPPORTED), (dict(g=ODD), MISALIGNED),
    (dict(dh0=ODD), MISALIGNED), (dict(dq=A), INVALID),
    (dict(dv=A + 0x5000), INVALID), (dict(cu=A + 0xb000, B=0), INVALID),
])
def test_bwd_rejects_on_host(lib, fn, kw, expect):
    assert bwd(lib.library(), fn, **kw) == expect


@pytest.mark.parametrize("fn", ["gdn_chunk_bwd", "gdn_chunk_bwd_f32"])
@pytest.mark.parametrize("variant", [-1, 2])
def test_chunk_bwd_rejects_unknown_gate_placement(lib, fn, variant):
    assert bwd(lib.library(), fn, variant=variant) == INVALID


@pytest.mark.parametrize("fn", ["gdn_chunk_bwd", "gdn_kda_bwd", "gdn_chunk_bwd_f32",
                                "gdn_chunk_bwd_chunked"])
def test_bwd_empty_batch_is_a_no_op(lib, fn):
    assert bwd(lib.library(), fn, B=0) == OK


def test_chunked_bwd_takes_dense_batches_only(lib):
    assert bwd(lib.library(), "gdn_chunk_bwd_chunked", cu=A + 0xb000) == UNSUPPORTED


def bwd_fused(so, **kw):
    a = dict(q=A, k=A + 0x1000, v=A + 0x2000, a=A + 0x3000, b=A + 0x4000,
             h0=None, cu=None, w=None, z=None, eps=1e-6, do=A + 0x5000,
             dhT=None, dq=A + 0x6000, dk=A + 0x7000, dv=A + 0x8000,
             da=A + 0x9000, db=A + 0xa000, dh0=None, dw=None, dz=None,
             B=1, H=1, T=16, dk_=128, dv_=128)
    a.update(kw)
    return so.gdn_chunk_bwd_fused(a["q"], a["k"], a["v"], a["a"], a["b"], a["h0"],
                                  a["cu"], a["w"], a["z"], a["eps"], a["do"],
                                  a["dhT"], a["dq"], a["dk"], a["dv"], a["da"],
                                  a["db"], a["dh0"], a["dw"], a["dz"], a["B"],
                                  a["H"], a["T"], a["dk_"], a["dv_"], None)


@pytest.mark.parametrize("kw,expect", [
    (dict(B=-1), INVALID), (dict(H=0), INVALID), (dict(eps=-1.0), INVALID),
    (dict(q=None), INVALID), (dict(da=None), INVALID), (dict(do=None), INVALID),
    (dict(dw=A + 0xb000), INVALID),              # dweight without a weight
    (dict(dz=A + 0xb000), INVALID),              # dgate without a gate
    (dict(dk_=96), UNSUPPORTED), (dict(dv_=32), UNSUPPORTED),
    (dict(a=ODD), MISALIGNED), (dict(w=ODD), MISALIGNED),
    (dict(dq=A), INVALID), (dict(cu=A + 0xb000, B=0), INVALID),
])
def test_bwd_fused_rejects_on_host(lib, kw, expect):
    assert bwd_fused(lib.library(), **kw) == expect


def test_bwd_fused_empty_batch_is_a_no_op(lib):
    assert bwd_fused(lib.library(), B=0) == OK

"""Thin ctypes binding of ``include/gdn.h`` (argument marshalling only).

Each function takes CUDA torch tensors, checks dtypes/shapes/contiguity,
passes raw device pointers and the current torch stream to the native entry
point of the same name, and raises ``GdnError`` on a negative status. Output
tensors are allocated with torch when not supplied (torch is the memory and
stream provider; every step of the computation runs in the library's
kernels). There is no CPU fallback: without the built library, or with a
non-CUDA tensor, these functions raise.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

from . import build as _build

GDN_OK = 0
GDN_GATE_BEFORE_PREDICT = 0
GDN_GATE_AFTER_PREDICT = 1
GDN_DTYPE_BF16 = 0
GDN_DTYPE_F32 = 1
GDN_PATH_AUTO = 0
GDN_PATH_SIMT = 1
GDN_PATH_TCGEN05 = 2
GDN_PATH_TCGEN05_SPLIT = 3
GDN_PATH_TCGEN05_WHOLE = 4
GDN_PATH_TCGEN05_FUSED = 5
GDN_SP_CHAIN = 0x100
GDN_SP_SCAN = 0x200
# kernel families for per-kernel timing (gdn_kernel_t)
GDN_KERNEL_CHUNK_PREP = 0
GDN_KERNEL_CHUNK_CHAIN = 1
GDN_KERNEL_CHUNK_SIMT = 2
GDN_KERNEL_SP_CHAIN = 3
GDN_KERNEL_DECODE = 4
GDN_KERNEL_CHUNK_OFFSETS = 5
GDN_KERNEL_CHUNK_CHAIN_WHOLE = 6
GDN_KERNEL_KDA = 7
GDN_KERNEL_KDA_PREP = 8
GDN_KERNEL_BWD = 9
GDN_KERNEL_BWD_FINALIZE = 10
GDN_KERNEL_CBWD_PREP = 11
GDN_KERNEL_CBWD_FWD = 12
GDN_KERNEL_CBWD_REV = 13
GDN_KERNEL_CBWD_GRAD = 14
GDN_KERNEL_CHUNK_FUSED = 15
GDN_KERNEL_COUNT = 16
KERNEL_NAMES = {
    GDN_KERNEL_CHUNK_PREP: "ut_prep_kernel",
    GDN_KERNEL_CHUNK_CHAIN: "chunk_tc_kernel",
    GDN_KERNEL_CHUNK_SIMT: "chunk_simt_kernel",
    GDN_KERNEL_SP_CHAIN: "sp_chain_kernel",
    GDN_KERNEL_DECODE: "decode_kernel",
    GDN_KERNEL_CHUNK_OFFSETS: "chunk_offsets_kernel",
    GDN_KERNEL_CHUNK_CHAIN_WHOLE: "chain_tx_kernel",
    GDN_KERNEL_KDA: "kda_kernel",
    GDN_KERNEL_KDA_PREP: "kda_prep_kernel",
    GDN_KERNEL_BWD: "bwd_kernel",
    GDN_KERNEL_BWD_FINALIZE: "bwd_finalize_kernel",
    GDN_KERNEL_CBWD_PREP: "cbwd_prep_kernel",
    GDN_KERNEL_CBWD_FWD: "cbwd_fwd_kernel",
    GDN_KERNEL_CBWD_REV: "cbwd_rev_kernel",
    GDN_KERNEL_CBWD_GRAD: "cbwd_grad_kernel",
    GDN_KERNEL_CHUNK_FUSED: "fused_chunk_kernel",
}

_lib = None


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {gdn_status_string(status)} ({status})")


def library_path() -> Path:
    return _build.LIB


def library():
    """The loaded ``libgdn_gb300.so`` (ctypes.CDLL) with typed entry points."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not path.exists():
        raise RuntimeError(
            f"native library {path} is missing: run "
            "`python -c 'import __graft_entry__ as g; g.build()'` first "
            "(there is no fallback implementation)")
    lib = ctypes.CDLL(str(path))
    vp, fp, ip = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
    i = ctypes.c_int
    chunk_args = [vp, vp, vp, fp, fp, fp, vp, fp, ip, i, i, i, i, i, i, vp]
    lib.gdn_chunk_fwd.argtypes = chunk_args
    lib.gdn_chunk_fwd.restype = i
    lib.gdn_chunk_fwd_f32.argtypes = chunk_args
    lib.gdn_chunk_fwd_f32.restype = i
    lib.gdn_chunk_fwd_ex.argtypes = chunk_args[:-1] + [i, i, i, i, vp]
    lib.gdn_chunk_fwd_ex.restype = i
    lib.gdn_recurrent_step.argtypes = [vp, vp, vp, fp, fp, fp, vp, i, i, i, i,
                                       vp]
    lib.gdn_recurrent_step.restype = i
    lib.gdn_kda_fwd.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, ip, i, i, i, i,
                                i, vp]
    lib.gdn_kda_fwd.restype = i
    lib.gdn_kda_fwd_ex.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, ip, i, i, i,
                                   i, i, i, i, vp]
    lib.gdn_kda_fwd_ex.restype = i
    bwd_args = [vp, vp, vp, fp, fp, fp, vp, fp, fp, fp, fp, fp, fp, fp, ip, i,
                i, i, i, i]
    lib.gdn_kda_bwd.argtypes = bwd_args + [vp]
    lib.gdn_kda_bwd.restype = i
    lib.gdn_chunk_bwd.argtypes = bwd_args + [i, vp]
    lib.gdn_chunk_bwd.restype = i
    lib.gdn_chunk_bwd_f32.argtypes = bwd_args + [i, vp]
    lib.gdn_chunk_bwd_f32.restype = i
    lib.gdn_chunk_bwd_chunked.argtypes = bwd_args + [vp]
    lib.gdn_chunk_bwd_chunked.restype = i
    lib.gdn_chunk_bwd_fused.argtypes = [vp, vp, vp, fp, fp, fp, ip, fp, vp,
                                        ctypes.c_float, vp, fp, fp, fp, fp, fp,
                                        fp, fp, fp, fp, i, i, i, i, i, vp]
    lib.gdn_chunk_bwd_fused.restype = i
    lib.gdn_device_status.argtypes = [vp]
    lib.gdn_device_status.restype = i
    lib.gdn_status_string.argtypes = [i]
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_version.restype = i
    lib.gdn_kernel_launches.restype = ctypes.c_ulonglong
    lib.gdn_selftest_mma.argtypes = [vp, vp, vp, i, i, i, i, i, i, vp]
    lib.gdn_selftest_mma.restype = i
    lib.gdn_chunk_fwd_fused.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, ip,
                                        fp, vp, ctypes.c_float, i, i, i, i,
                                        i, i, i, vp]
    lib.gdn_chunk_fwd_fused.restype = i
    lib.gdn_timing_enable.argtypes = [i]
    lib.gdn_timing_enable.restype = i
    lib.gdn_timing_read.argtypes = [i, ctypes.POINTER(ctypes.c_ulonglong),
                                    ctypes.POINTER(ctypes.c_double)]
    lib.gdn_timing_read.restype = i
    _lib = lib
    return lib


def gdn_status_string(status: int) -> str:
    return library().gdn_status_string(int(status)).decode()


def kernel_counters() -> int:
    """Kernels enqueued by the library so far in this process."""
    return int(library().gdn_kernel_launches())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, name, dtype, device):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (no CPU fallback)")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _shape(t, name, shape):
    """The kernels index by the sizes passed: a tensor of another shape would
    be read or written out of bounds, so it is refused here."""
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be {list(shape)}, got {list(t.shape)}")
    return t


def _chunk_call(fn_name, q, k, v, g, beta, h0, cu_seqlens, out, hT,
                output_final_state, C, stream, io_dtype, extra=()):
    fn = getattr(library(), fn_name)
    if extra:
        f0 = fn
        fn = (lambda *a: f0(*a[:-1], *extra, a[-1]))
    return _chunk_call_fn(fn, fn_name, q, k, v, g, beta, h0, cu_seqlens, out,
                          hT, output_final_state, C, stream, io_dtype)


def _chunk_call_fn(fn, fn_name, q, k, v, g, beta, h0, cu_seqlens, out, hT,
                   output_final_state, C, stream, io_dtype):
    dev = q.device
    _need(q, "q", io_dtype, None)
    _need(k, "k", io_dtype, dev)
    _need(v, "v", io_dtype, dev)
    _need(g, "g", torch.float32, dev)
    _need(beta, "beta", torch.float32, dev)
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q/k must be [B, T, H, dk] and v [B, T, H, dv]")
    Bt, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != (Bt, T, H):
        raise ValueError("q/k/v shapes disagree")
    if g.shape != (Bt, T, H) or beta.shape != (Bt, T, H):
        raise ValueError("g/beta must be [B, T, H]")
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
        if Bt != 1:
            raise ValueError("packed sequences are passed as [1, T, H, ...]")
        N = cu_seqlens.numel() - 1
    else:
        N = Bt
    if h0 is not None:
        _need(h0, "h0", torch.float32, dev)
        if h0.shape != (N, H, dk, dv):
            raise ValueError(f"h0 must be [{N}, {H}, {dk}, {dv}]")
    if out is None:
        out = torch.empty_like(v)
    else:
        _shape(_need(out, "out", io_dtype, dev), "out", v.shape)
    if hT is None and output_final_state:
        hT = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    elif hT is not None:
        _shape(_need(hT, "hT", torch.float32, dev), "hT", (N, H, dk, dv))
    with torch.cuda.device(dev):
        rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                _ptr(out), _ptr(hT), _ptr(cu_seqlens), N, H, T, dk, dv, C,
                _stream(stream))
    if rc != GDN_OK:
        raise GdnError(rc, fn_name)
    return out, hT


def gdn_chunk_fwd(q, k, v, g, beta, h0=None, cu_seqlens=None, *, out=None,
                  hT=None, output_final_state=True, C=64, stream=None):
    """bf16 chunkwise forward; returns (out bf16 like v, hT fp32 or None)."""
    return _chunk_call("gdn_chunk_fwd", q, k, v, g, beta, h0, cu_seqlens, out,
                       hT, output_final_state, C, stream, torch.bfloat16)


def gdn_chunk_fwd_f32(q, k, v, g, beta, h0=None, cu_seqlens=None, *, out=None,
                      hT=None, output_final_state=True, C=64, stream=None):
    """fp32 chunkwise forward; returns (out fp32, hT fp32 or None)."""
    return _chunk_call("gdn_chunk_fwd_f32", q, k, v, g, beta, h0, cu_seqlens,
                       out, hT, output_final_state, C, stream, torch.float32)


def gdn_chunk_fwd_ex(q, k, v, g, beta, h0=None, cu_seqlens=None, *, out=None,
                     hT=None, output_final_state=True, C=64,
                     variant=GDN_GATE_BEFORE_PREDICT, path=GDN_PATH_AUTO,
                     sp_parts=0, stream=None):
    """Chunkwise forward with explicit gate placement, kernel family and
    sequence-parallel split; q/k/v dtype (bf16 or fp32) selects the dtype."""
    dtype = {torch.bfloat16: GDN_DTYPE_BF16, torch.float32: GDN_DTYPE_F32}.get(
        q.dtype)
    if dtype is None:
        raise ValueError("q/k/v must be bf16 or fp32")
    return _chunk_call("gdn_chunk_fwd_ex", q, k, v, g, beta, h0, cu_seqlens,
                       out, hT, output_final_state, C, stream, q.dtype,
                       extra=(dtype, int(variant), int(path), int(sp_parts)))


def gdn_kda_fwd(q, k, v, g, beta, h0=None, cu_seqlens=None, *, out=None,
                hT=None, output_final_state=True, stream=None):
    """The delta rule with a per-channel decay, token by token: q, k bf16
    [B, T, H, dk], v bf16 [B, T, H, dv], g fp32 [B, T, H, dk] log-decays,
    beta fp32 [B, T, H]. Returns (out bf16 like v, hT fp32 [N, H, dk, dv] or
    None); ``hT`` may be ``h0`` (in-place state update)."""
    return _kda("gdn_kda_fwd", q, k, v, g, beta, h0, cu_seqlens, out, hT,
                output_final_state, stream, ())


def gdn_kda_fwd_ex(q, k, v, g, beta, h0=None, cu_seqlens=None, *, out=None,
                   hT=None, output_final_state=True, path=GDN_PATH_AUTO,
                   sp_parts=0, stream=None):
    """gdn_kda_fwd with a choice of kernels: ``path`` GDN_PATH_AUTO (the
    chunk form on the tensor cores where it applies), GDN_PATH_SIMT (token by
    token) or GDN_PATH_TCGEN05 (the chunk form), optionally or-ed with
    GDN_SP_CHAIN / GDN_SP_SCAN; ``sp_parts`` the sequence-parallel split of
    the chunk form (0: automatic)."""
    return _kda("gdn_kda_fwd_ex", q, k, v, g, beta, h0, cu_seqlens, out, hT,
                output_final_state, stream, (int(path), int(sp_parts)))


def gdn_kda_bwd(q, k, v, g, beta, h0, dout, dhT=None, cu_seqlens=None, *,
                want_dh0=True, stream=None):
    """Gradients of gdn_kda_fwd for L = sum(dout * out) + sum(dhT * hT):
    returns dict dq, dk [B, T, H, dk], dv [B, T, H, dv], dg [B, T, H, dk],
    dbeta [B, T, H] (fp32) and dh0 [N, H, dk, dv] (fp32, or None)."""
    return _bwd("gdn_kda_bwd", q, k, v, g, beta, h0, dout, dhT, cu_seqlens,
                want_dh0, stream, per_channel=True)


def gdn_chunk_bwd(q, k, v, g, beta, h0, dout, dhT=None, cu_seqlens=None, *,
                  variant=GDN_GATE_BEFORE_PREDICT, want_dh0=True, stream=None):
    """Gradients of gdn_chunk_fwd_ex (scalar gate; ``variant`` the forward's
    gate placement): as gdn_kda_bwd with g and dg [B, T, H]."""
    return _bwd("gdn_chunk_bwd", q, k, v, g, beta, h0, dout, dhT, cu_seqlens,
                want_dh0, stream, per_channel=False, extra=(int(variant),))


def gdn_chunk_bwd_chunked(q, k, v, g, beta, h0, dout, dhT=None, *,
                          want_dh0=True, stream=None):
    """gdn_chunk_bwd (decay before the prediction) through the chunk form:
    per-chunk UT/WY quantities, the chunks' entry states and exit gradients by
    two chains, then every chunk's gradients in parallel; dense batches only.
    Returns the dict of gdn_chunk_bwd."""
    return _bwd("gdn_chunk_bwd_chunked", q, k, v, g, beta, h0, dout, dhT,
                None, want_dh0, stream, per_channel=False)


def gdn_chunk_bwd_f32(q, k, v, g, beta, h0, dout, dhT=None, cu_seqlens=None,
                      *, variant=GDN_GATE_BEFORE_PREDICT, want_dh0=True,
                      stream=None):
    """gdn_chunk_bwd for fp32 q, k, v and dout."""
    return _bwd("gdn_chunk_bwd_f32", q, k, v, g, beta, h0, dout, dhT,
                cu_seqlens, want_dh0, stream, per_channel=False,
                extra=(int(variant),), in_dtype=torch.float32)


def gdn_chunk_bwd_fused(q, k, v, a, b, h0, dout, dhT=None, cu_seqlens=None, *,
                        norm_weight=None, gate=None, eps=1e-6, want_dh0=True,
                        stream=None):
    """Gradients of gdn_chunk_fwd_fused for L = sum(dout * out) + sum(dhT *
    hT): dict dq, dk, dv, da, db, dh0 (or None), dweight (with norm_weight,
    else None), dgate (with gate, else None); all fp32."""
    dev = q.device
    _need(q, "q", torch.bfloat16, None)
    for name, t in (("k", k), ("v", v), ("dout", dout)):
        _need(t, name, torch.bfloat16, dev)
    _need(a, "a", torch.float32, dev)
    _need(b, "b", torch.float32, dev)
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q/k must be [B, T, H, dk] and v/dout [B, T, H, dv]")
    Bt, T, H, dk = q.shape
    dv = v.shape[-1]
    _shape(k, "k", q.shape)
    _shape(v, "v", (Bt, T, H, dv))
    _shape(dout, "dout", v.shape)
    _shape(a, "a", (Bt, T, H))
    _shape(b, "b", (Bt, T, H))
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
        if Bt != 1:
            raise ValueError("packed sequences are passed as [1, T, H, ...]")
        N = cu_seqlens.numel() - 1
    else:
        N = Bt
    if norm_weight is not None:
        _shape(_need(norm_weight, "norm_weight", torch.float32, dev),
               "norm_weight", (dv,))
    if gate is not None:
        _shape(_need(gate, "gate", torch.bfloat16, dev), "gate", v.shape)
    for name, st in (("h0", h0), ("dhT", dhT)):
        if st is not None:
            _shape(_need(st, name, torch.float32, dev), name, (N, H, dk, dv))
    f32 = dict(dtype=torch.float32, device=dev)
    res = {"dq": torch.empty(q.shape, **f32), "dk": torch.empty(q.shape, **f32),
           "dv": torch.empty(v.shape, **f32), "da": torch.empty(a.shape, **f32),
           "db": torch.empty(b.shape, **f32),
           "dh0": torch.empty((N, H, dk, dv), **f32) if want_dh0 else None,
           "dweight": torch.empty((dv,), **f32) if norm_weight is not None else None,
           "dgate": torch.empty(v.shape, **f32) if gate is not None else None}
    with torch.cuda.device(dev):
        rc = library().gdn_chunk_bwd_fused(
            _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(h0),
            _ptr(cu_seqlens), _ptr(norm_weight), _ptr(gate), float(eps),
            _ptr(dout), _ptr(dhT), _ptr(res["dq"]), _ptr(res["dk"]),
            _ptr(res["dv"]), _ptr(res["da"]), _ptr(res["db"]),
            _ptr(res["dh0"]), _ptr(res["dweight"]), _ptr(res["dgate"]), N, H,
            T, dk, dv, _stream(stream))
    if rc != GDN_OK:
        raise GdnError(rc, "gdn_chunk_bwd_fused")
    return res


def _bwd(fn, q, k, v, g, beta, h0, dout, dhT, cu_seqlens, want_dh0, stream,
         per_channel, extra=(), in_dtype=torch.bfloat16):
    dev = q.device
    _need(q, "q", in_dtype, None)
    for name, t in (("k", k), ("v", v), ("dout", dout)):
        _need(t, name, in_dtype, dev)
    _need(g, "g", torch.float32, dev)
    _need(beta, "beta", torch.float32, dev)
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q/k must be [B, T, H, dk] and v/dout [B, T, H, dv]")
    Bt, T, H, dk = q.shape
    dv = v.shape[-1]
    gshape = q.shape if per_channel else q.shape[:3]
    if k.shape != q.shape or v.shape[:3] != (Bt, T, H) or dout.shape != v.shape:
        raise ValueError("q/k must be [B, T, H, dk], v/dout [B, T, H, dv]")
    if g.shape != gshape or beta.shape != (Bt, T, H):
        raise ValueError(f"g must be {tuple(gshape)} and beta [B, T, H]")
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
        if Bt != 1:
            raise ValueError("packed sequences are passed as [1, T, H, ...]")
        N = cu_seqlens.numel() - 1
    else:
        N = Bt
    for name, st in (("h0", h0), ("dhT", dhT)):
        if st is not None:
            _need(st, name, torch.float32, dev)
            if st.shape != (N, H, dk, dv):
                raise ValueError(f"{name} must be [{N}, {H}, {dk}, {dv}]")
    f32 = dict(dtype=torch.float32, device=dev)
    res = {"dq": torch.empty(q.shape, **f32), "dk": torch.empty(q.shape, **f32),
           "dv": torch.empty(v.shape, **f32), "dg": torch.empty(gshape, **f32),
           "dbeta": torch.empty(beta.shape, **f32),
           "dh0": torch.empty((N, H, dk, dv), **f32) if want_dh0 else None}
    with torch.cuda.device(dev):
        rc = getattr(library(), fn)(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
            _ptr(dout), _ptr(dhT), _ptr(res["dq"]), _ptr(res["dk"]),
            _ptr(res["dv"]), _ptr(res["dg"]), _ptr(res["dbeta"]),
            _ptr(res["dh0"]), _ptr(cu_seqlens), N, H, T, dk, dv, *extra,
            _stream(stream))
    if rc != GDN_OK:
        raise GdnError(rc, fn)
    return res


def _kda(fn, q, k, v, g, beta, h0, cu_seqlens, out, hT, output_final_state,
         stream, extra):
    dev = q.device
    _need(q, "q", torch.bfloat16, None)
    _need(k, "k", torch.bfloat16, dev)
    _need(v, "v", torch.bfloat16, dev)
    _need(g, "g", torch.float32, dev)
    _need(beta, "beta", torch.float32, dev)
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q/k/g must be [B, T, H, dk] and v [B, T, H, dv]")
    Bt, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != (Bt, T, H) or g.shape != q.shape:
        raise ValueError("q/k/g must be [B, T, H, dk] and v [B, T, H, dv]")
    if beta.shape != (Bt, T, H):
        raise ValueError("beta must be [B, T, H]")
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
        if Bt != 1:
            raise ValueError("packed sequences are passed as [1, T, H, ...]")
        N = cu_seqlens.numel() - 1
    else:
        N = Bt
    for name, st in (("h0", h0), ("hT", hT)):
        if st is not None:
            _need(st, name, torch.float32, dev)
            if st.shape != (N, H, dk, dv):
                raise ValueError(f"{name} must be [{N}, {H}, {dk}, {dv}]")
    if out is None:
        out = torch.empty_like(v)
    else:
        _shape(_need(out, "out", torch.bfloat16, dev), "out", v.shape)
    if hT is None and output_final_state:
        hT = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        rc = getattr(library(), fn)(_ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                      _ptr(beta), _ptr(h0), _ptr(out),
                                      _ptr(hT), _ptr(cu_seqlens), N, H, T, dk,
                                      dv, *extra, _stream(stream))
    if rc != GDN_OK:
        raise GdnError(rc, fn)
    return out, hT


def gdn_chunk_fwd_fused(q, k, v, a, b, h0=None, cu_seqlens=None, *,
                        norm_weight=None, gate=None, eps=1e-6, out=None,
                        hT=None, output_final_state=True, C=64,
                        path=GDN_PATH_AUTO, stream=None):
    """The forward pass with the steps either side fused: raw q, k (L2-
    normalised in the kernels), gate logits a (log alpha = -softplus(a)) and
    step logits b (beta = sigmoid(b)); output RMS-normalised over d_v and
    scaled by ``norm_weight`` [dv] fp32 when given, then gated by
    sigmoid(``gate``) (bf16, like v) when given. Returns (out bf16, hT)."""
    dev = q.device
    if norm_weight is not None:
        _need(norm_weight, "norm_weight", torch.float32, dev)
        if norm_weight.shape != (v.shape[-1],):
            raise ValueError("norm_weight must be [dv]")
    if gate is not None:
        _need(gate, "gate", torch.bfloat16, dev)
        if gate.shape != v.shape:
            raise ValueError("gate must have the shape of v")
    extra_ptrs = (_ptr(norm_weight), _ptr(gate), ctypes.c_float(float(eps)))

    class _Fn:  # argument order of gdn_chunk_fwd_fused
        def __init__(self, f):
            self.f = f

        def __call__(self, q_, k_, v_, a_, b_, h0_, out_, hT_, cu_, N, H, T,
                     dk, dv, C_, stream_):
            return self.f(q_, k_, v_, a_, b_, h0_, out_, hT_, cu_,
                          *extra_ptrs, N, H, T, dk, dv, C_, int(path),
                          stream_)

    lib = library()
    return _chunk_call_fn(_Fn(lib.gdn_chunk_fwd_fused), "gdn_chunk_fwd_fused",
                          q, k, v, a, b, h0, cu_seqlens, out, hT,
                          output_final_state, C, stream, torch.bfloat16)


def gdn_recurrent_step(q, k, v, g, beta, state, *, out=None, stream=None):
    """One decode token per (sequence, head); ``state`` is updated in place.
    q, k [N, H, dk] bf16, v [N, H, dv] bf16, g/beta [N, H] fp32, state
    [N, H, dk, dv] fp32. Returns out [N, H, dv] bf16."""
    dev = q.device
    _need(q, "q", torch.bfloat16, None)
    _need(k, "k", torch.bfloat16, dev)
    _need(v, "v", torch.bfloat16, dev)
    _need(g, "g", torch.float32, dev)
    _need(beta, "beta", torch.float32, dev)
    _need(state, "state", torch.float32, dev)
    if q.dim() != 3 or v.dim() != 3:
        raise ValueError("q/k must be [N, H, dk] and v [N, H, dv]")
    N, H, dk = q.shape
    dv = v.shape[-1]
    _shape(k, "k", q.shape)
    _shape(v, "v", (N, H, dv))
    _shape(g, "g", (N, H))
    _shape(beta, "beta", (N, H))
    if state.shape != (N, H, dk, dv):
        raise ValueError("state must be [N, H, dk, dv]")
    if out is None:
        out = torch.empty_like(v)
    else:
        _shape(_need(out, "out", torch.bfloat16, dev), "out", v.shape)
    with torch.cuda.device(dev):
        rc = library().gdn_recurrent_step(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
            _ptr(out), N, H, dk, dv, _stream(stream))
    if rc != GDN_OK:
        raise GdnError(rc, "gdn_recurrent_step")
    return out


def gdn_selftest_mma(A, B, *, a_mn=False, b_mn=False, b_stacked=False,
                     twice=False, a_tmem=False, stream=None):
    """D = A @ B (x2 when ``twice``) through one tcgen05 MMA sequence with the
    chunk kernel's shared-memory layouts. A bf16 [128, K], B bf16 [K, N];
    ``a_tmem`` places A in TMEM instead of shared memory."""
    dev = A.device
    _need(A, "A", torch.bfloat16, None)
    _need(B, "B", torch.bfloat16, dev)
    K, N = A.shape[1], B.shape[1]
    if A.shape != (128, K) or B.shape != (K, N):
        raise ValueError("A must be [128, K] and B [K, N]")
    D = torch.empty((128, N), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        rc = library().gdn_selftest_mma(_ptr(A), _ptr(B), _ptr(D), K, N,
                                        2 if a_tmem else int(a_mn),
                                        int(b_mn), int(b_stacked),
                                        int(twice), _stream(stream))
    if rc != GDN_OK:
        raise GdnError(rc, "gdn_selftest_mma")
    return D


def gdn_device_status(stream=None) -> int:
    """Synchronises ``stream`` and returns/clears the kernels' status word."""
    return int(library().gdn_device_status(_stream(stream)))


def gdn_timing_enable(on: bool) -> None:
    """Per-kernel device timing on/off (resets the accumulated totals)."""
    rc = library().gdn_timing_enable(1 if on else 0)
    if rc != GDN_OK:
        raise GdnError(rc, "gdn_timing_enable")


def gdn_timing_read(kernel: int):
    """(launches, total_ms) of one kernel family since timing was enabled;
    waits for the recorded events."""
    n = ctypes.c_ulonglong(0)
    ms = ctypes.c_double(0.0)
    rc = library().gdn_timing_read(int(kernel), ctypes.byref(n),
                                   ctypes.byref(ms))
    if rc != GDN_OK:
        raise GdnError(rc, "gdn_timing_read")
    return int(n.value), float(ms.value)


def kernel_timings():
    """{kernel name: (launches, total_ms)} for every family timed so far."""
    out = {}
    for k in range(GDN_KERNEL_COUNT):
        n, ms = gdn_timing_read(k)
        if n:
            out[KERNEL_NAMES[k]] = (n, ms)
    return out

"""Oracle for the Gated DeltaNet forward pass (fp64, CPU).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. It shares no code with the CUDA library and never imports it.

Two parts:

* ``forward`` -- the definition: a plain fp64 token loop written in C
  (``gdn_oracle.c``), parallel over (sequence, head) with OpenMP. This is the
  function every GPU result is compared with.
* ``oracle.chunked`` -- slower numpy restatements of the same map in the
  forms the pages derive (per-token affine maps and their composition, the
  WY/UT chunk form, the sequence-parallel correction, the Householder product
  sum). They exist only to pin ``forward`` from independent directions in the
  CPU tests; the GPU is never compared with them.
* ``oracle.sublayer`` -- the steps either side of the recurrence in fp64
  (L2 normalisation of q and k, the sigmoid / softplus gate activations, the
  RMS normalisation and sigmoid gate of the output) and ``fused_forward``,
  which wraps ``forward`` with them; pinned in
  ``tests/test_oracle_sublayer_pins.py``.
* ``oracle.kda`` -- the delta rule with a per-channel decay (KDA) in fp64,
  token by token; pinned in ``tests/test_oracle_kda_pins.py``.
* ``oracle.backward`` -- gradients of both (per-channel and scalar gate,
  decay before the prediction) by the reverse sweep of the token loop in
  fp64; pinned in ``tests/test_oracle_backward_pins.py`` (finite differences
  through the forward oracles, closed forms, automatic differentiation of an
  independent PyTorch forward).
* ``oracle.chunked_backward`` -- the same gradients chunk by chunk: the
  adjoint of each step of the chunk form (the algebra a chunked backward
  evaluates), pinned to ``oracle.backward`` at chunk sizes 1 to T in
  ``tests/test_oracle_chunk_backward_pins.py``.

Pins (all in ``tests/test_oracle_pins.py``): worked numbers of the illustrated
DeltaNet page (delta-rule 1.5/2.25/2.625, the 2-D example, prediction/error,
the GDN 3.7 gate-placement example, 1-D WY split, gate prefix ratio 0.1/0.8),
closed forms (beta = 0 pure decay, orthonormal-key overwrite, unit-key
interpolation, single-token rank-1 update), brute force at T <= 8, affine
composition and associativity, chunk-size invariance, the sequence-parallel
correction, resume through h0/hT and varlen packing. No function here is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "gdn_oracle.c"
_BUILD = _HERE / "_build"
_LIB_PATH = _BUILD / "libgdn_oracle.so"

G1 = 1  # decay, then correct (the GDN paragraph of the illustrated page)
G0 = 0  # correct against the undecayed state (the lqnn.cn page, section 1.2)


def build(force: bool = False) -> Path:
    """Compile the C oracle with gcc (-O2, OpenMP). Idempotent."""
    _BUILD.mkdir(exist_ok=True)
    if (not force and _LIB_PATH.exists()
            and _LIB_PATH.stat().st_mtime >= _SRC.stat().st_mtime):
        return _LIB_PATH
    tmp = _LIB_PATH.with_suffix(f".{os.getpid()}.tmp")
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           str(_SRC), "-o", str(tmp), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(str(_LIB_PATH))
        dp = ctypes.POINTER(ctypes.c_double)
        lib.gdn_oracle_forward.argtypes = [
            dp, dp, dp, dp, dp, dp, dp, dp, ctypes.POINTER(ctypes.c_int32),
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.gdn_oracle_forward.restype = ctypes.c_int
        lib.gdn_oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor (any dtype, incl. bf16)
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(_load().gdn_oracle_max_threads())


def forward(q, k, v, g, beta, h0=None, cu_seqlens=None, variant: int = G1,
            threads: int = 0):
    """fp64 token loop.

    q, k: [B, T, H, dk]; v: [B, T, H, dv]; g (log alpha), beta: [B, T, H];
    h0: [N, H, dk, dv] or None (zero state); cu_seqlens: int32 [N + 1] or None
    (then the tensors are [1, T, H, ...] and N sequences are packed).
    Accepts numpy arrays or CPU torch tensors of any float dtype; values are
    upcast exactly to fp64. Returns (out [B, T, H, dv], hT [N, H, dk, dv]) as
    float64 numpy arrays.
    """
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == q.shape and v.shape[:3] == (B, T, H)
    assert g.shape == (B, T, H) and beta.shape == (B, T, H)
    cu = None
    if cu_seqlens is not None:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        assert B == 1, "packed sequences are passed as [1, T, H, ...]"
        N, T_arg = cu.shape[0] - 1, T
    else:
        N, T_arg = B, T
    if h0 is not None:
        assert h0.shape == (N, H, dk, dv)
    out = np.zeros((B, T, H, dv), dtype=np.float64)
    hT = np.zeros((N, H, dk, dv), dtype=np.float64)
    rc = _load().gdn_oracle_forward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(out),
        _ptr(hT),
        None if cu is None else cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
        N, H, T_arg, dk, dv, int(variant), int(threads))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (rc={rc})")
    return out, hT


def recurrent_step(q, k, v, g, beta, state, variant: int = G1):
    """One token per (sequence, head) applied to ``state`` [N, H, dk, dv].

    q, k: [N, H, dk]; v: [N, H, dv]; g, beta: [N, H]. This is ``forward`` with
    T = 1; returns (out [N, H, dv], new_state) without touching the input.
    """
    q, k, v, g, beta, state = map(_f64, (q, k, v, g, beta, state))
    out, hT = forward(q[:, None], k[:, None], v[:, None], g[:, None],
                      beta[:, None], h0=state, variant=variant)
    return out[:, 0], hT

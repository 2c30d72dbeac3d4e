"""Gated DeltaNet chunkwise forward pass and decode step for GB300 (sm_103a).

The compute lives in a native library (``_lib/libgdn_gb300.so``) built from
``csrc/`` by ``build.build()``; ``abi`` is a thin ctypes binding with the same
entry-point names as ``include/gdn.h``. There is no CPU fallback: touching an
entry point without the built library raises.

``inputs`` (seeded synthetic data) is importable without the native library.
"""
from __future__ import annotations

_ABI_NAMES = (
    "gdn_chunk_fwd", "gdn_chunk_fwd_f32", "gdn_chunk_fwd_ex",
    "gdn_recurrent_step", "gdn_chunk_fwd_fused", "gdn_kda_fwd",
    "gdn_kda_fwd_ex", "gdn_kda_bwd", "gdn_chunk_bwd", "gdn_chunk_bwd_f32",
    "gdn_chunk_bwd_chunked",
    "gdn_chunk_bwd_fused",
    "GDN_GATE_BEFORE_PREDICT", "GDN_GATE_AFTER_PREDICT",
    "gdn_status_string",
    "GdnError", "library_path",
    "library", "kernel_counters", "gdn_device_status", "gdn_selftest_mma",
    "gdn_timing_enable", "gdn_timing_read", "kernel_timings",
    "GDN_KERNEL_CHUNK_PREP", "GDN_KERNEL_CHUNK_CHAIN", "GDN_KERNEL_CHUNK_SIMT",
    "GDN_KERNEL_SP_CHAIN", "GDN_KERNEL_DECODE", "GDN_KERNEL_CHUNK_OFFSETS",
    "GDN_KERNEL_CHUNK_CHAIN_WHOLE", "GDN_KERNEL_KDA", "GDN_KERNEL_KDA_PREP", "GDN_KERNEL_BWD", "GDN_KERNEL_BWD_FINALIZE",
    "GDN_KERNEL_CBWD_PREP", "GDN_KERNEL_CBWD_FWD", "GDN_KERNEL_CBWD_REV", "GDN_KERNEL_CBWD_GRAD",
    "GDN_KERNEL_CHUNK_FUSED",
    "GDN_KERNEL_COUNT",
    "KERNEL_NAMES",
    "GDN_PATH_AUTO", "GDN_PATH_SIMT", "GDN_PATH_TCGEN05",
    "GDN_PATH_TCGEN05_SPLIT", "GDN_PATH_TCGEN05_WHOLE",
    "GDN_PATH_TCGEN05_FUSED", "GDN_SP_CHAIN",
    "GDN_SP_SCAN",
)


def __getattr__(name):
    if name in _ABI_NAMES:
        from . import abi
        return getattr(abi, name)
    raise AttributeError(name)

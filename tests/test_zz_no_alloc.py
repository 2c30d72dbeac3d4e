"""The allocation-free sequence-parallel entry point.

gdn_chunk_fwd_sp_noalloc serves callers that cannot allocate device memory
while enqueueing work (an engine plugin with a fixed memory plan, a serving
loop under a fixed budget): it runs the sequence-parallel pass with its
workspace in a fixed device array owned by the library. These tests call it
through the C ABI and compare it with the allocating entry point
gdn_chunk_fwd_ex on the same inputs, twice in a row (the array keeps the
previous call's contents), within the parity tolerance used elsewhere.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from gated_deltanet_chunkwise_gb300 import inputs

TOL = {"f32": 1e-3, "bf16": 2e-2}
UNSUPPORTED, INVALID = -2, -1


def _bind(so):
    vp, i = ctypes.c_void_p, ctypes.c_int
    so.gdn_chunk_fwd_sp_noalloc.argtypes = [vp] * 9 + [i] * 9 + [vp]
    so.gdn_chunk_fwd_sp_noalloc.restype = i
    so.gdn_noalloc_scratch_bytes.argtypes = [i] * 5
    so.gdn_noalloc_scratch_bytes.restype = ctypes.c_ulonglong
    return so


def _noalloc(so, x, out, hT, parts, dtype_code, stream):
    B, T, H, dk = x["q"].shape
    dv = x["v"].shape[-1]
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return so.gdn_chunk_fwd_sp_noalloc(
        p(x["q"]), p(x["k"]), p(x["v"]), p(x["g"]), p(x["beta"]), p(x["h0"]),
        p(out), p(hT), None, B, H, T, dk, dv, 64, dtype_code, 0, parts,
        ctypes.c_void_p(stream.cuda_stream))


def test_rejects_requests_above_the_scratch_limit(lib):
    so = _bind(lib.library())
    limit = 32 << 20
    assert so.gdn_noalloc_scratch_bytes(1, 16, 128, 128, 8) <= limit
    assert so.gdn_noalloc_scratch_bytes(64, 16, 128, 128, 8) > limit
    a = 0x7F0000000000
    args = [a, a + 0x1000, a + 0x2000, a + 0x3000, a + 0x4000, None,
            a + 0x5000, None, None]
    # far too many (sequence, head, part) triples: refused before any launch
    assert so.gdn_chunk_fwd_sp_noalloc(*args, 64, 16, 4096, 128, 128, 64, 0,
                                       0, 8, None) == UNSUPPORTED
    assert so.gdn_chunk_fwd_sp_noalloc(*args, 1, 1, 256, 64, 64, 64, 0, 0, 1,
                                       None) == INVALID


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,parts", [("bf16", 4), ("f32", 3)])
def test_matches_allocating_entry_on_two_calls(lib, cuda_device, dtype,
                                               parts):
    so = _bind(lib.library())
    stream = torch.cuda.current_stream(cuda_device)
    code = 0 if dtype == "bf16" else 1
    for call, seed in enumerate((31, 32)):  # different data on each call
        d = inputs.chunk_inputs(2, 3, 64 * 9 + 40, 128, 128, dtype=dtype,
                                seed=seed, h0=True)
        x = {k: (None if v is None else v.to(cuda_device))
             for k, v in d.items()}
        ref_out, ref_hT = lib.gdn_chunk_fwd_ex(
            x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
            path=1, sp_parts=parts)
        out = torch.full_like(x["v"], float("nan"))
        hT = torch.full_like(ref_hT, float("nan"))
        rc = _noalloc(so, x, out, hT, parts, code, stream)
        assert rc == 0, lib.gdn_status_string(rc)
        torch.cuda.synchronize()
        for got, ref in ((out, ref_out), (hT, ref_hT)):
            g = got.double().cpu().numpy()
            r = ref.double().cpu().numpy()
            assert np.all(np.isfinite(g)), f"call {call}: unwritten output"
            err = np.max(np.abs(g - r)) / np.max(np.abs(r))
            assert err <= TOL[dtype], f"call {call}: rel err {err:.3e}"

"""The allocation-free sequence-parallel entry point.

gdn_chunk_fwd_sp_noalloc serves callers that cannot allocate device memory
while enqueueing work (an engine plugin with a fixed memory plan, a serving
loop under a fixed budget): it runs the sequence-parallel pass with its
workspace in a fixed device array owned by the library. These tests call it
through the C ABI on two calls in a row with different layouts (the array
keeps the previous call's contents) and compare each call with the
allocating entry point gdn_chunk_fwd_ex and with the fp64 oracle, within the
parity tolerance used elsewhere.

The file name sorts last so that pytest collects it last: the entry point is
an addition outside the method's own path, and if it fails, a run that stops
at the first failure (-x) has already run every other test. Nothing here
depends on the order: each test makes its own first call, and the tests pass
alone in a fresh process as well.
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


def test_rejects_requests_above_the_scratch_limit(lib):
    so = _bind(lib.library())
    limit = 32 << 20
    assert so.gdn_noalloc_scratch_bytes(1, 16, 128, 128, 8) <= limit
    assert so.gdn_noalloc_scratch_bytes(64, 16, 128, 128, 8) > limit
    # head dimensions the entry point does not serve size to 0 (no overflow)
    assert so.gdn_noalloc_scratch_bytes(1, 1, 1 << 20, 1 << 20, 8) == 0
    assert so.gdn_noalloc_scratch_bytes(1, 1, 96, 128, 8) == 0
    a = 0x7F0000000000
    args = [a, a + 0x1000, a + 0x2000, a + 0x3000, a + 0x4000, None,
            a + 0x5000, None, None]
    # far too many (sequence, head, part) triples: refused before any launch
    assert so.gdn_chunk_fwd_sp_noalloc(*args, 64, 16, 4096, 128, 128, 64, 0,
                                       0, 8, None) == UNSUPPORTED
    assert so.gdn_chunk_fwd_sp_noalloc(*args, 1, 1, 256, 64, 64, 64, 0, 0, 1,
                                       None) == INVALID


def _packed_inputs(dtype, seed):
    lens = [64 * 4 + 9, 64 * 7 + 33]  # both longer than two parts' chunks
    return inputs.chunk_inputs(len(lens), 3, 0, 128, 128, dtype=dtype,
                               seed=seed, h0=True, lengths=lens)


def _check(lib, so, d, parts, dtype, stream, dev, call):
    import oracle
    x = {k: (None if v is None else v.to(dev)) for k, v in d.items()}
    cu = x["cu_seqlens"]
    ref_out, ref_hT = lib.gdn_chunk_fwd_ex(
        x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], cu,
        path=1, sp_parts=parts)
    o_ref, h_ref = oracle.forward(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                  d["h0"], d["cu_seqlens"])
    out = torch.full_like(x["v"], float("nan"))
    hT = torch.full_like(ref_hT, float("nan"))
    B, T, H, dk = x["q"].shape
    dv = x["v"].shape[-1]
    N = cu.numel() - 1 if cu is not None else B
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = so.gdn_chunk_fwd_sp_noalloc(
        p(x["q"]), p(x["k"]), p(x["v"]), p(x["g"]), p(x["beta"]), p(x["h0"]),
        p(out), p(hT), p(cu), N, H, T, dk, dv, 64,
        0 if dtype == "bf16" else 1, 0, parts,
        ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0, lib.gdn_status_string(rc)
    torch.cuda.synchronize()
    assert lib.gdn_device_status() == 0
    for got, ref, exact in ((out, ref_out, o_ref), (hT, ref_hT, h_ref)):
        g = got.double().cpu().numpy()
        assert np.all(np.isfinite(g)), f"call {call}: unwritten output"
        r = ref.double().cpu().numpy()
        err = np.max(np.abs(g - r)) / np.max(np.abs(r))
        assert err <= TOL[dtype], f"call {call}: vs allocating entry {err:.3e}"
        err = np.max(np.abs(g - exact)) / np.max(np.abs(exact))
        assert err <= TOL[dtype], f"call {call}: vs oracle {err:.3e}"


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,parts", [("bf16", 4), ("f32", 3)])
def test_matches_allocating_entry_on_two_calls(lib, cuda_device, dtype,
                                               parts):
    so = _bind(lib.library())
    stream = torch.cuda.current_stream(cuda_device)
    for call, seed in enumerate((31, 32)):  # different data on each call
        d = inputs.chunk_inputs(2, 3, 64 * 9 + 40, 128, 128, dtype=dtype,
                                seed=seed, h0=True)
        _check(lib, so, d, parts, dtype, stream, cuda_device, call)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_large_call_then_smaller_packed_call(lib, cuda_device, dtype):
    # The first call fills more of the array (two sequences, five parts: the
    # correction chain runs) than the second reads (packed sequences, two
    # parts: no chain, the start states come from the split pass alone), at
    # other offsets; both are checked against the oracle.
    so = _bind(lib.library())
    stream = torch.cuda.current_stream(cuda_device)
    big = inputs.chunk_inputs(2, 3, 64 * 11 + 5, 128, 128, dtype=dtype,
                              seed=41, h0=True)
    _check(lib, so, big, 5, dtype, stream, cuda_device, 0)
    _check(lib, so, _packed_inputs(dtype, 42), 2, dtype, stream, cuda_device,
           1)

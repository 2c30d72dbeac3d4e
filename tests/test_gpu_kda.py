"""gdn_kda_fwd (per-channel decay) against the fp64 oracle (oracle/kda.py) on
the same seeded inputs, element by element.

Bound: max|X_gpu - X_ref| / max|X_ref| <= 2e-2, the bf16 bound of the chunk
path (the kernel keeps the state in fp32; its outputs are rounded to bf16).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import kda
from gated_deltanet_chunkwise_gb300 import inputs

pytestmark = pytest.mark.gpu
TOL = 2e-2


def rel_err(x, ref):
    x = x.detach().float().cpu().numpy() if hasattr(x, "detach") else x
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


def run(lib, dev, d, **kw):
    g = lambda t: None if t is None else t.to(dev)
    out = torch.full(d["v"].shape, float("nan"), dtype=torch.bfloat16, device=dev)
    o, hT = lib.gdn_kda_fwd(g(d["q"]), g(d["k"]), g(d["v"]), g(d["g"]),
                            g(d["beta"]), g(d["h0"]), g(d["cu_seqlens"]),
                            out=out, **kw)
    torch.cuda.synchronize(dev)
    assert lib.gdn_device_status() == 0
    return o, hT


def check(lib, dev, d):
    o, hT = run(lib, dev, d)
    o_ref, h_ref = kda.forward(d["q"], d["k"], d["v"], d["g"], d["beta"],
                               d["h0"], cu_seqlens=d["cu_seqlens"])
    assert rel_err(o, o_ref) <= TOL, rel_err(o, o_ref)
    assert rel_err(hT, h_ref) <= TOL, rel_err(hT, h_ref)


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("h0", [False, True])
def test_kda_matches_oracle(lib, cuda_device, dk, dv, h0):
    d = inputs.kda_inputs(2, 3, 77, dk, dv, seed=31, h0=h0)
    check(lib, cuda_device, d)


@pytest.mark.parametrize("T", [1, 15, 16, 17, 200])
def test_kda_lengths(lib, cuda_device, T):
    d = inputs.kda_inputs(1, 2, T, 128, 128, seed=32, h0=True)
    check(lib, cuda_device, d)


def test_kda_packed(lib, cuda_device):
    d = inputs.kda_inputs(0, 2, 0, 128, 64, seed=33, h0=True,
                          lengths=[40, 0, 1, 16, 129, 3])
    check(lib, cuda_device, d)


def test_kda_equal_channels_is_the_scalar_gate(lib, cuda_device):
    """One log-decay for every channel: the scalar-gate recurrence (decay
    before the prediction), checked against that oracle."""
    d = inputs.chunk_inputs(2, 2, 90, 128, 128, dtype="bf16", seed=34, h0=True)
    g1 = d["g"]
    d["g"] = g1[..., None].expand(*g1.shape, 128).contiguous()
    o, hT = run(lib, cuda_device, d)
    o_ref, h_ref = oracle.forward(d["q"], d["k"], d["v"], g1, d["beta"],
                                  d["h0"], variant=oracle.G1)
    assert rel_err(o, o_ref) <= TOL
    assert rel_err(hT, h_ref) <= TOL


def test_kda_decode_step_in_place(lib, cuda_device):
    """T = 1 with hT = h0: one token updates the state in place."""
    d = inputs.kda_inputs(4, 3, 1, 128, 128, seed=35, h0=True)
    g = lambda t: t.to(cuda_device)
    state = g(d["h0"])
    out = torch.empty_like(g(d["v"]))
    lib.gdn_kda_fwd(g(d["q"]), g(d["k"]), g(d["v"]), g(d["g"]), g(d["beta"]),
                    state, None, out=out, hT=state)
    torch.cuda.synchronize(cuda_device)
    o_ref, h_ref = kda.forward(d["q"], d["k"], d["v"], d["g"], d["beta"],
                               d["h0"])
    assert rel_err(out, o_ref) <= TOL
    assert rel_err(state, h_ref) <= TOL


def test_kda_invalid_packing_is_recorded(lib, cuda_device):
    d = inputs.kda_inputs(0, 2, 0, 64, 64, seed=36, lengths=[30, 20, 10])
    d["cu_seqlens"] = torch.tensor([0, 50, 30, 60], dtype=torch.int32)
    g = lambda t: None if t is None else t.to(cuda_device)
    lib.gdn_kda_fwd(g(d["q"]), g(d["k"]), g(d["v"]), g(d["g"]), g(d["beta"]),
                    None, g(d["cu_seqlens"]))
    torch.cuda.synchronize(cuda_device)
    assert lib.gdn_device_status() == -1  # GDN_ERR_INVALID_ARG

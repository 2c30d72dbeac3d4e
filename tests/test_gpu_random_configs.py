"""Seeded random configurations through the tensor-core forward (both chain
kernels, sequence-parallel splits and both sub-sequence combinations), the
chunk form of KDA and the backward pass, each against its fp64 oracle: a
sweep over shapes, packings, lengths around chunk and block boundaries and
initial states that the targeted tests do not enumerate.

Bounds as in the targeted tests: 2e-2 (bf16 outputs), 1e-3 (fp32 gradients).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import backward, kda
from gated_deltanet_chunkwise_gb300 import inputs

pytestmark = pytest.mark.gpu


def rel_err(x, ref):
    x = x.detach().float().cpu().numpy() if hasattr(x, "detach") else x
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


def draw(seed):
    rng = np.random.default_rng(seed)
    cfg = {"H": int(rng.integers(1, 4)), "dv": int(rng.choice([64, 128])),
           "h0": bool(rng.integers(0, 2))}
    if rng.integers(0, 2):
        n = int(rng.integers(1, 6))
        cfg["lengths"] = [int(x) for x in rng.choice(
            [0, 1, 15, 16, 17, 63, 64, 65, 100, 129, 200], size=n)]
        if sum(cfg["lengths"]) == 0:
            cfg["lengths"][0] = 33
        cfg["B"], cfg["T"] = 0, 0
    else:
        cfg["lengths"] = None
        cfg["B"] = int(rng.integers(1, 4))
        cfg["T"] = int(rng.choice([1, 63, 64, 65, 127, 128, 129, 257, 640]))
    cfg["path"] = int(rng.choice([2, 3, 4]))
    cfg["sp"] = int(rng.choice([0, 0, 2, 3, 5]))
    cfg["combine"] = int(rng.choice([0x100, 0x200]))
    return cfg


def kw(cfg):
    return dict(lengths=cfg["lengths"]) if cfg["lengths"] is not None else {}


@pytest.mark.parametrize("seed", range(24))
def test_forward_random(lib, cuda_device, seed):
    cfg = draw(1000 + seed)
    d = inputs.chunk_inputs(cfg["B"], cfg["H"], cfg["T"], 128, cfg["dv"],
                            dtype="bf16", seed=seed, h0=cfg["h0"], **kw(cfg))
    x = lambda t: None if t is None else t.to(cuda_device)
    # sp > 0 forces that many sub-sequences (parts past a short sequence's end
    # stay empty)
    path = cfg["path"] | (cfg["combine"] if cfg["sp"] else 0)
    o, hT = lib.gdn_chunk_fwd_ex(x(d["q"]), x(d["k"]), x(d["v"]), x(d["g"]),
                                 x(d["beta"]), x(d["h0"]), x(d["cu_seqlens"]),
                                 path=path, sp_parts=cfg["sp"])
    torch.cuda.synchronize(cuda_device)
    assert lib.gdn_device_status() == 0
    o_ref, h_ref = oracle.forward(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                  d["h0"], cu_seqlens=d["cu_seqlens"])
    assert rel_err(o, o_ref) <= 2e-2, cfg
    assert rel_err(hT, h_ref) <= 2e-2, cfg


@pytest.mark.parametrize("seed", range(16))
def test_kda_chunk_random(lib, cuda_device, seed):
    cfg = draw(2000 + seed)
    d = inputs.kda_inputs(cfg["B"], cfg["H"], cfg["T"], 128, cfg["dv"],
                          seed=seed, h0=cfg["h0"], **kw(cfg))
    x = lambda t: None if t is None else t.to(cuda_device)
    path = 2 | (cfg["combine"] if cfg["sp"] else 0)
    o, hT = lib.gdn_kda_fwd_ex(x(d["q"]), x(d["k"]), x(d["v"]), x(d["g"]),
                               x(d["beta"]), x(d["h0"]), x(d["cu_seqlens"]),
                               path=path, sp_parts=cfg["sp"])
    torch.cuda.synchronize(cuda_device)
    assert lib.gdn_device_status() == 0
    o_ref, h_ref = kda.forward(d["q"], d["k"], d["v"], d["g"], d["beta"],
                               d["h0"], cu_seqlens=d["cu_seqlens"])
    assert rel_err(o, o_ref) <= 2e-2, cfg
    assert rel_err(hT, h_ref) <= 2e-2, cfg


@pytest.mark.parametrize("seed", range(12))
def test_backward_random(lib, cuda_device, seed):
    cfg = draw(3000 + seed)
    after = bool(seed % 2)
    d = inputs.chunk_inputs(cfg["B"], cfg["H"], cfg["T"], 128, cfg["dv"],
                            dtype="bf16", seed=seed, h0=cfg["h0"], **kw(cfg))
    dout, dh = inputs.grad_inputs(d, seed=seed, dhT=bool(seed % 3))
    x = lambda t: None if t is None else t.to(cuda_device)
    got = lib.gdn_chunk_bwd(x(d["q"]), x(d["k"]), x(d["v"]), x(d["g"]),
                            x(d["beta"]), x(d["h0"]), x(dout), x(dh),
                            x(d["cu_seqlens"]),
                            variant=lib.GDN_GATE_AFTER_PREDICT if after
                            else lib.GDN_GATE_BEFORE_PREDICT)
    torch.cuda.synchronize(cuda_device)
    assert lib.gdn_device_status() == 0
    ref = backward.backward(d["q"], d["k"], d["v"], d["g"], d["beta"],
                            d["h0"], dout, dh, cu_seqlens=d["cu_seqlens"],
                            variant=oracle.G0 if after else oracle.G1)
    for n in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        assert rel_err(got[n], ref[n]) <= 1e-3, (n, cfg)

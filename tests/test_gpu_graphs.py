"""The entry points inside CUDA graphs: each call is captured once (after an
eager warm-up that performs the per-device set-up) and replayed on new
inputs copied into the captured buffers; every replay must reproduce the
eager call on the same inputs bit for bit (the kernels are deterministic),
and the decode step, whose state is updated in place, must advance by one
token per replay.
"""
import pytest
import torch

from gated_deltanet_chunkwise_gb300 import inputs

pytestmark = pytest.mark.gpu


def fill(static, d):
    for k, v in d.items():
        if v is not None and static.get(k) is not None:
            static[k].copy_(v)


def capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        res = fn()
    return g, res


def test_chunk_forward_replays(lib, cuda_device):
    dev = cuda_device
    first = inputs.chunk_inputs(2, 4, 300, 128, 128, dtype="bf16", seed=81, h0=True)
    static = {k: (None if v is None else v.to(dev)) for k, v in first.items()}
    out = torch.empty_like(static["v"])
    hT = torch.empty_like(static["h0"])
    call = lambda: lib.gdn_chunk_fwd(static["q"], static["k"], static["v"],
                                     static["g"], static["beta"], static["h0"],
                                     out=out, hT=hT)
    g, _ = capture(call)
    for seed in (82, 83):
        d = inputs.chunk_inputs(2, 4, 300, 128, 128, dtype="bf16", seed=seed, h0=True)
        fill(static, d)
        g.replay()
        torch.cuda.synchronize()
        got_o, got_h = out.clone(), hT.clone()
        call()
        torch.cuda.synchronize()
        assert torch.equal(got_o, out) and torch.equal(got_h, hT)
    assert lib.gdn_device_status() == 0


def test_kda_chunk_forward_replays(lib, cuda_device):
    dev = cuda_device
    first = inputs.kda_inputs(2, 3, 200, 128, 128, seed=84, h0=True)
    static = {k: (None if v is None else v.to(dev)) for k, v in first.items()}
    out = torch.empty_like(static["v"])
    hT = torch.empty_like(static["h0"])
    call = lambda: lib.gdn_kda_fwd_ex(static["q"], static["k"], static["v"],
                                      static["g"], static["beta"], static["h0"],
                                      out=out, hT=hT, path=2)
    g, _ = capture(call)
    d = inputs.kda_inputs(2, 3, 200, 128, 128, seed=85, h0=True)
    fill(static, d)
    g.replay()
    torch.cuda.synchronize()
    got_o, got_h = out.clone(), hT.clone()
    call()
    torch.cuda.synchronize()
    assert torch.equal(got_o, out) and torch.equal(got_h, hT)
    assert lib.gdn_device_status() == 0


def test_backward_replays(lib, cuda_device):
    dev = cuda_device
    first = inputs.chunk_inputs(1, 2, 150, 128, 128, dtype="bf16", seed=86, h0=True)
    dout, dhT = inputs.grad_inputs(first, seed=86)
    first["dout"], first["dhT"] = dout, dhT
    static = {k: (None if v is None else v.to(dev)) for k, v in first.items()}
    call = lambda: lib.gdn_chunk_bwd(static["q"], static["k"], static["v"],
                                     static["g"], static["beta"], static["h0"],
                                     static["dout"], static["dhT"])
    g, res = capture(call)
    d = inputs.chunk_inputs(1, 2, 150, 128, 128, dtype="bf16", seed=87, h0=True)
    d["dout"], d["dhT"] = inputs.grad_inputs(d, seed=87)
    fill(static, d)
    g.replay()
    torch.cuda.synchronize()
    got = {k: v.clone() for k, v in res.items()}
    eager = call()
    torch.cuda.synchronize()
    for k in got:
        assert torch.equal(got[k], eager[k]), k
    assert lib.gdn_device_status() == 0


def test_decode_step_replays_advance_the_state(lib, cuda_device):
    dev = cuda_device
    d = inputs.decode_inputs(8, 4, 128, 128, seed=88)
    static = {k: v.to(dev) for k, v in d.items()}
    out = torch.empty_like(static["v"])
    state0 = static["state"].clone()
    call = lambda: lib.gdn_recurrent_step(static["q"], static["k"], static["v"],
                                          static["g"], static["beta"],
                                          static["state"], out=out)
    g, _ = capture(call)
    static["state"].copy_(state0)  # the warm-up step advanced it
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    replayed = static["state"].clone()
    static["state"].copy_(state0)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    assert torch.equal(replayed, static["state"])
    assert lib.gdn_device_status() == 0


def test_fused_backward_replays(lib, cuda_device):
    """The fused-sublayer backward (five kernels and the backward kernel's two
    sweeps) replays bit for bit."""
    dev = cuda_device
    first = inputs.fused_inputs(1, 2, 150, 128, 128, seed=89, h0=True)
    first["dout"], first["dhT"] = inputs.grad_inputs(first, seed=89)
    static = {k: (None if v is None else v.to(dev)) for k, v in first.items()}
    call = lambda: lib.gdn_chunk_bwd_fused(
        static["q"], static["k"], static["v"], static["a"], static["b"],
        static["h0"], static["dout"], static["dhT"],
        norm_weight=static["norm_weight"], gate=static["gate"])
    g, res = capture(call)
    d = inputs.fused_inputs(1, 2, 150, 128, 128, seed=90, h0=True)
    d["dout"], d["dhT"] = inputs.grad_inputs(d, seed=90)
    fill(static, d)
    g.replay()
    torch.cuda.synchronize()
    got = {k: v.clone() for k, v in res.items() if v is not None}
    eager = call()
    torch.cuda.synchronize()
    for k in got:
        assert torch.equal(got[k], eager[k]), k
    assert lib.gdn_device_status() == 0

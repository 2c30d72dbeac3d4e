"""gdn_chunk_bwd_chunked (the backward pass through the chunk form: per-chunk
UT/WY quantities, a forward chain of entry states, a reverse chain of exit
gradients, then every chunk's gradients in parallel) against the fp64
gradient oracle (oracle/backward.py) on the same seeded inputs, element by
element; bound 1e-3 as for gdn_chunk_bwd (fp32 arithmetic on the exact bf16
inputs)."""
import numpy as np
import pytest
import torch

from oracle import backward
from gated_deltanet_chunkwise_gb300 import inputs

pytestmark = pytest.mark.gpu
TOL = 1e-3
GRADS = ("dq", "dk", "dv", "dg", "dbeta")


def rel_err(x, ref):
    x = x.detach().float().cpu().numpy()
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


def check(lib, dev, d, *, dhT=True, seed=0):
    dout, dh = inputs.grad_inputs(d, seed=seed, dhT=dhT)
    x = lambda t: None if t is None else t.to(dev)
    got = lib.gdn_chunk_bwd_chunked(x(d["q"]), x(d["k"]), x(d["v"]), x(d["g"]),
                                    x(d["beta"]), x(d["h0"]), x(dout), x(dh))
    torch.cuda.synchronize(dev)
    assert lib.gdn_device_status() == 0
    ref = backward.backward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"],
                            dout, dh, variant=1)
    errs = {n: rel_err(got[n], ref[n]) for n in GRADS + ("dh0",)}
    assert all(e <= TOL for e in errs.values()), errs


@pytest.mark.parametrize("dk,dv", [(128, 128), (128, 64), (64, 128), (64, 64)])
@pytest.mark.parametrize("h0", [False, True])
def test_chunked_bwd_matches_oracle(lib, cuda_device, dk, dv, h0):
    d = inputs.chunk_inputs(2, 2, 150, dk, dv, dtype="bf16", seed=91, h0=h0)
    check(lib, cuda_device, d, seed=3)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_chunked_bwd_lengths(lib, cuda_device, T):
    d = inputs.chunk_inputs(1, 3, T, 128, 128, dtype="bf16", seed=92, h0=True)
    check(lib, cuda_device, d, dhT=bool(T % 2), seed=4)


def test_chunked_bwd_agrees_with_the_token_sweep(lib, cuda_device):
    d = inputs.chunk_inputs(2, 4, 700, 128, 128, dtype="bf16", seed=93, h0=True)
    dout, dh = inputs.grad_inputs(d, seed=5)
    x = lambda t: None if t is None else t.to(cuda_device)
    args = (x(d["q"]), x(d["k"]), x(d["v"]), x(d["g"]), x(d["beta"]),
            x(d["h0"]), x(dout), x(dh))
    a = lib.gdn_chunk_bwd_chunked(*args)
    b = lib.gdn_chunk_bwd(*args)
    torch.cuda.synchronize(cuda_device)
    for n in GRADS + ("dh0",):
        ref = b[n].double().cpu().numpy()
        assert rel_err(a[n], ref) <= TOL, n


def test_chunked_bwd_bench_size_sampled(lib, cuda_device):
    """B=4, H=16, T=2048 (the backward bench workload); two (sequence, head)
    pairs against the oracle on their slices."""
    d = inputs.chunk_inputs(4, 16, 2048, 128, 128, dtype="bf16", seed=94)
    dout, _ = inputs.grad_inputs(d, seed=6, dhT=False)
    x = lambda t: None if t is None else t.to(cuda_device)
    got = lib.gdn_chunk_bwd_chunked(x(d["q"]), x(d["k"]), x(d["v"]), x(d["g"]),
                                    x(d["beta"]), None, x(dout), None)
    torch.cuda.synchronize(cuda_device)
    assert lib.gdn_device_status() == 0
    for n, h in ((0, 1), (3, 14)):
        sl = lambda t: t[n:n + 1, :, h:h + 1]
        ref = backward.backward(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["g"]),
                                sl(d["beta"]), None, sl(dout))
        for name in GRADS:
            assert rel_err(sl(got[name]), ref[name]) <= TOL, (name, n, h)
        assert rel_err(got["dh0"][n:n + 1, h:h + 1], ref["dh0"]) <= TOL

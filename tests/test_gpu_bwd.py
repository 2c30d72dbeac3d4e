"""The backward pass on the GPU (gdn_kda_bwd, gdn_chunk_bwd: bwd_kernel +
bwd_finalize_kernel) against the fp64 gradient oracle (oracle/backward.py)
on the same seeded inputs, element by element.

Bound: max|X_gpu - X_ref| / max|X_ref| <= 1e-3 for every gradient (the
kernels compute in fp32 from the same bf16 / fp32 inputs the oracle reads
exactly; nothing is rounded to bf16 on the way).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import backward
from gated_deltanet_chunkwise_gb300 import inputs

pytestmark = pytest.mark.gpu
TOL = 1e-3
GRADS = ("dq", "dk", "dv", "dg", "dbeta")


def rel_err(x, ref):
    x = x.detach().float().cpu().numpy()
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


def run_and_check(lib, dev, d, scalar, *, dhT=True, seed=0, after=False):
    """after: the gate placement that predicts with the undecayed state
    (GDN_GATE_AFTER_PREDICT; the oracle's G0)."""
    dout, dh = inputs.grad_inputs(d, seed=seed, dhT=dhT)
    x = lambda t: None if t is None else t.to(dev)
    args = (x(d["q"]), x(d["k"]), x(d["v"]), x(d["g"]), x(d["beta"]),
            x(d["h0"]), x(dout), x(dh), x(d["cu_seqlens"]))
    if scalar:
        got = lib.gdn_chunk_bwd(*args, variant=lib.GDN_GATE_AFTER_PREDICT if after
                                else lib.GDN_GATE_BEFORE_PREDICT)
    else:
        got = lib.gdn_kda_bwd(*args)
    torch.cuda.synchronize(dev)
    assert lib.gdn_device_status() == 0
    if scalar:
        ref = backward.backward(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                d["h0"], dout, dh, cu_seqlens=d["cu_seqlens"],
                                variant=oracle.G0 if after else oracle.G1)
    else:
        ref = backward.kda_backward(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                    d["h0"], dout, dh, cu_seqlens=d["cu_seqlens"])
    errs = {n: rel_err(got[n], ref[n]) for n in GRADS + ("dh0",)}
    assert all(e <= TOL for e in errs.values()), errs
    return errs


@pytest.mark.parametrize("dk,dv", [(128, 128), (128, 64), (64, 128), (64, 64)])
@pytest.mark.parametrize("h0", [False, True])
def test_kda_bwd_matches_oracle(lib, cuda_device, dk, dv, h0):
    d = inputs.kda_inputs(2, 2, 77, dk, dv, seed=61, h0=h0)
    run_and_check(lib, cuda_device, d, scalar=False, seed=1)


@pytest.mark.parametrize("T", [1, 15, 16, 17, 64, 200])
def test_scalar_bwd_lengths(lib, cuda_device, T):
    d = inputs.chunk_inputs(1, 2, T, 128, 128, dtype="bf16", seed=62, h0=True)
    run_and_check(lib, cuda_device, d, scalar=True, seed=2)


@pytest.mark.parametrize("T", [1, 17, 200])
def test_scalar_bwd_other_gate_placement(lib, cuda_device, T):
    d = inputs.chunk_inputs(2, 2, T, 128, 128, dtype="bf16", seed=68, h0=True)
    run_and_check(lib, cuda_device, d, scalar=True, seed=7, after=True)


def test_scalar_bwd_other_gate_placement_packed(lib, cuda_device):
    d = inputs.chunk_inputs(0, 2, 0, 128, 64, dtype="bf16", seed=69, h0=True,
                            lengths=[33, 0, 70, 5])
    run_and_check(lib, cuda_device, d, scalar=True, seed=8, after=True)


@pytest.mark.parametrize("after", [False, True])
@pytest.mark.parametrize("lengths", [None, [40, 0, 1, 129, 7]])
def test_f32_bwd_matches_oracle(lib, cuda_device, after, lengths):
    """fp32 q, k, v, dout (gdn_chunk_bwd_f32), dense and packed, both gate
    placements."""
    if lengths is None:
        d = inputs.chunk_inputs(2, 2, 97, 128, 128, dtype="f32", seed=71, h0=True)
    else:
        d = inputs.chunk_inputs(0, 2, 0, 128, 64, dtype="f32", seed=72, h0=True,
                                lengths=lengths)
    dout, dh = inputs.grad_inputs(d, seed=9)
    dout = dout.float()
    x = lambda t: None if t is None else t.to(cuda_device)
    got = lib.gdn_chunk_bwd_f32(x(d["q"]), x(d["k"]), x(d["v"]), x(d["g"]),
                                x(d["beta"]), x(d["h0"]), x(dout), x(dh),
                                x(d["cu_seqlens"]),
                                variant=lib.GDN_GATE_AFTER_PREDICT if after
                                else lib.GDN_GATE_BEFORE_PREDICT)
    torch.cuda.synchronize(cuda_device)
    assert lib.gdn_device_status() == 0
    ref = backward.backward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"],
                            dout, dh, cu_seqlens=d["cu_seqlens"],
                            variant=oracle.G0 if after else oracle.G1)
    errs = {n: rel_err(got[n], ref[n]) for n in GRADS + ("dh0",)}
    assert all(e <= TOL for e in errs.values()), errs


def test_scalar_bwd_without_dhT(lib, cuda_device):
    d = inputs.chunk_inputs(2, 3, 90, 128, 128, dtype="bf16", seed=63, h0=True)
    run_and_check(lib, cuda_device, d, scalar=True, dhT=False, seed=3)


@pytest.mark.parametrize("scalar", [True, False])
def test_bwd_packed(lib, cuda_device, scalar):
    lengths = [40, 0, 1, 16, 129, 3]
    if scalar:
        d = inputs.chunk_inputs(0, 2, 0, 128, 64, dtype="bf16", seed=64, h0=True,
                                lengths=lengths)
    else:
        d = inputs.kda_inputs(0, 2, 0, 128, 64, seed=64, h0=True, lengths=lengths)
    run_and_check(lib, cuda_device, d, scalar=scalar, seed=4)


def test_bwd_dh0_in_place_of_dhT(lib, cuda_device):
    """dh0 may be the dhT buffer: each state row is read before it is
    overwritten."""
    d = inputs.kda_inputs(2, 2, 50, 128, 128, seed=65, h0=True)
    dout, dh = inputs.grad_inputs(d, seed=5)
    dev = cuda_device
    x = lambda t: None if t is None else t.to(dev)
    buf = x(dh).clone()
    res = {n: torch.empty(s, dtype=torch.float32, device=dev) for n, s in
           (("dq", d["q"].shape), ("dk", d["q"].shape), ("dv", d["v"].shape),
            ("dg", d["q"].shape), ("dbeta", d["beta"].shape))}
    dd = {n: x(d[n]) for n in ("q", "k", "v", "g", "beta", "h0")}
    dd["dout"] = x(dout)  # (device copies kept alive through the call)
    P = lib.abi._ptr
    rc = lib.library().gdn_kda_bwd(
        *(P(dd[n]) for n in ("q", "k", "v", "g", "beta", "h0")), P(dd["dout"]),
        P(buf), *(P(res[n]) for n in GRADS), P(buf), None, 2, 2, 50, 128, 128,
        None)
    assert rc == 0
    torch.cuda.synchronize(dev)
    ref = backward.kda_backward(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                d["h0"], dout, dh)
    assert rel_err(buf, ref["dh0"]) <= TOL
    assert rel_err(res["dq"], ref["dq"]) <= TOL


def test_zero_dout_and_dhT_give_zero_gradients(lib, cuda_device):
    d = inputs.chunk_inputs(1, 2, 40, 128, 128, dtype="bf16", seed=66, h0=True)
    x = lambda t: None if t is None else t.to(cuda_device)
    dout = torch.zeros(d["v"].shape, dtype=torch.bfloat16)
    got = lib.gdn_chunk_bwd(x(d["q"]), x(d["k"]), x(d["v"]), x(d["g"]),
                            x(d["beta"]), x(d["h0"]), x(dout), None)
    torch.cuda.synchronize(cuda_device)
    for n in GRADS + ("dh0",):
        assert float(got[n].abs().max()) == 0.0, n


def test_bwd_bench_size_sampled(lib, cuda_device):
    """B=4, H=16, T=2048 (the bench workload) in the bench's launch
    configuration; two (sequence, head) pairs checked against the oracle
    (heads are independent, so the oracle runs on their slices only)."""
    d = inputs.chunk_inputs(4, 16, 2048, 128, 128, dtype="bf16", seed=67)
    dout, dh = inputs.grad_inputs(d, seed=6, dhT=False)
    x = lambda t: None if t is None else t.to(cuda_device)
    got = lib.gdn_chunk_bwd(x(d["q"]), x(d["k"]), x(d["v"]), x(d["g"]),
                            x(d["beta"]), None, x(dout), None)
    torch.cuda.synchronize(cuda_device)
    for n, h in ((0, 0), (3, 13)):
        sl = lambda t: t[n:n + 1, :, h:h + 1]
        ref = backward.backward(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["g"]),
                                sl(d["beta"]), None, sl(dout))
        for name in GRADS:
            assert rel_err(sl(got[name]), ref[name]) <= TOL, (name, n, h)
        assert rel_err(got["dh0"][n:n + 1, h:h + 1], ref["dh0"]) <= TOL


@pytest.mark.parametrize("weight,gate", [(True, True), (True, False),
                                         (False, True), (False, False)])
@pytest.mark.parametrize("dk,dv", [(128, 64), (128, 128), (64, 64), (64, 128)])
def test_fused_bwd_matches_oracle(lib, cuda_device, weight, gate, dk, dv):
    """gdn_chunk_bwd_fused against the fused-sublayer gradient oracle (raw q,
    k with lengths in [0.25, 4), gate and step logits, RMSNorm weight and
    output gate when present)."""
    d = inputs.fused_inputs(2, 2, 77, dk, dv, seed=73, h0=True, weight=weight,
                            gate=gate)
    dout, dh = inputs.grad_inputs(d, seed=10)
    x = lambda t: None if t is None else t.to(cuda_device)
    got = lib.gdn_chunk_bwd_fused(x(d["q"]), x(d["k"]), x(d["v"]), x(d["a"]),
                                  x(d["b"]), x(d["h0"]), x(dout), x(dh),
                                  norm_weight=x(d["norm_weight"]),
                                  gate=x(d["gate"]), eps=1e-6)
    torch.cuda.synchronize(cuda_device)
    assert lib.gdn_device_status() == 0
    ref = backward.fused_backward(d["q"], d["k"], d["v"], d["a"], d["b"],
                                  d["h0"], dout, dh, weight=d["norm_weight"],
                                  gate=d["gate"], eps=1e-6)
    names = ["dq", "dk", "dv", "da", "db", "dh0"]
    names += ["dweight"] if weight else []
    names += ["dgate"] if gate else []
    errs = {n: rel_err(got[n], ref[n]) for n in names}
    assert all(e <= TOL for e in errs.values()), errs


def test_fused_bwd_packed(lib, cuda_device):
    d = inputs.fused_inputs(0, 2, 0, 128, 128, seed=74, h0=True,
                            lengths=[30, 0, 70, 1])
    dout, dh = inputs.grad_inputs(d, seed=11)
    x = lambda t: None if t is None else t.to(cuda_device)
    got = lib.gdn_chunk_bwd_fused(x(d["q"]), x(d["k"]), x(d["v"]), x(d["a"]),
                                  x(d["b"]), x(d["h0"]), x(dout), x(dh),
                                  x(d["cu_seqlens"]),
                                  norm_weight=x(d["norm_weight"]),
                                  gate=x(d["gate"]), eps=1e-6)
    torch.cuda.synchronize(cuda_device)
    assert lib.gdn_device_status() == 0
    ref = backward.fused_backward(d["q"], d["k"], d["v"], d["a"], d["b"],
                                  d["h0"], dout, dh, cu_seqlens=d["cu_seqlens"],
                                  weight=d["norm_weight"], gate=d["gate"],
                                  eps=1e-6)
    for n in ("dq", "dk", "dv", "da", "db", "dh0", "dweight", "dgate"):
        assert rel_err(got[n], ref[n]) <= TOL, n


def test_fused_bwd_bench_size_sampled(lib, cuda_device):
    """The fused-sublayer backward at B=4, H=16, T=2048 (the bench workload:
    RMSNorm weight and output gate, no h0, no dhT) in the bench's launch
    configuration; two (sequence, head) pairs against the fused gradient
    oracle on their slices (the norm and gate act within a (token, head), so
    every gradient but dweight, a sum over all of them, depends on the slice
    alone; dweight is checked at the small sizes above)."""
    d = inputs.fused_inputs(4, 16, 2048, 128, 128, seed=75)
    dout, _ = inputs.grad_inputs(d, seed=12, dhT=False)
    x = lambda t: None if t is None else t.to(cuda_device)
    got = lib.gdn_chunk_bwd_fused(x(d["q"]), x(d["k"]), x(d["v"]), x(d["a"]),
                                  x(d["b"]), None, x(dout), None,
                                  norm_weight=x(d["norm_weight"]),
                                  gate=x(d["gate"]), want_dh0=True)
    torch.cuda.synchronize(cuda_device)
    assert lib.gdn_device_status() == 0
    for n, h in ((1, 2), (2, 15)):
        sl = lambda t: t[n:n + 1, :, h:h + 1]
        ref = backward.fused_backward(sl(d["q"]), sl(d["k"]), sl(d["v"]),
                                      sl(d["a"]), sl(d["b"]), None, sl(dout),
                                      weight=d["norm_weight"],
                                      gate=sl(d["gate"]))
        for name in ("dq", "dk", "dv", "da", "db", "dgate"):
            assert rel_err(sl(got[name]), ref[name]) <= TOL, (name, n, h)
        assert rel_err(got["dh0"][n:n + 1, h:h + 1], ref["dh0"]) <= TOL


def test_kda_bwd_bench_size_sampled(lib, cuda_device):
    """gdn_kda_bwd at B=4, H=16, T=2048 (the per-channel backward bench
    workload) in the bench's launch configuration; two (sequence, head)
    pairs against the oracle on their slices."""
    d = inputs.kda_inputs(4, 16, 2048, 128, 128, seed=68)
    dout, _ = inputs.grad_inputs(d, seed=7, dhT=False)
    x = lambda t: None if t is None else t.to(cuda_device)
    got = lib.gdn_kda_bwd(x(d["q"]), x(d["k"]), x(d["v"]), x(d["g"]),
                          x(d["beta"]), None, x(dout), None)
    torch.cuda.synchronize(cuda_device)
    assert lib.gdn_device_status() == 0
    for n, h in ((0, 5), (3, 11)):
        sl = lambda t: t[n:n + 1, :, h:h + 1]
        ref = backward.kda_backward(sl(d["q"]), sl(d["k"]), sl(d["v"]),
                                    sl(d["g"]), sl(d["beta"]), None, sl(dout))
        for name in GRADS:
            assert rel_err(sl(got[name]), ref[name]) <= TOL, (name, n, h)
        assert rel_err(got["dh0"][n:n + 1, h:h + 1], ref["dh0"]) <= TOL

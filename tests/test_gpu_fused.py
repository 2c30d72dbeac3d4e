"""gdn_chunk_fwd_fused against the fp64 oracle of the steps either side of
the recurrence (oracle/sublayer.py) on the same seeded raw inputs.

Bound: the bf16 tolerance of the chunk path, max|X_gpu - X_ref| /
max|X_ref| <= 2e-2, for the outputs (after normalisation and gate) and the
final states.
"""
import numpy as np
import pytest
import torch

from oracle import sublayer
from gated_deltanet_chunkwise_gb300 import inputs

pytestmark = pytest.mark.gpu
TOL = 2e-2
# both chain kernels of the tensor-core path: 64 state rows per CTA (two
# CTAs per head when dv = 128, a cluster pair for the fused epilogue) and
# 128 rows per CTA (the whole state in TMEM lanes)
CHAINS = [3, 4]
# and the single-launch form (preparation and chain in one cluster)
FUSED = 5


def rel_err(x, ref):
    x = x.detach().float().cpu().numpy() if hasattr(x, "detach") else x
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


def run(lib, dev, d, eps=1e-6, path=0):
    g = lambda t: None if t is None else t.to(dev)
    out = torch.full(d["v"].shape, float("nan"), dtype=torch.bfloat16, device=dev)
    o, hT = lib.gdn_chunk_fwd_fused(
        g(d["q"]), g(d["k"]), g(d["v"]), g(d["a"]), g(d["b"]), g(d["h0"]),
        g(d["cu_seqlens"]), norm_weight=g(d["norm_weight"]), gate=g(d["gate"]),
        eps=eps, out=out, path=path)
    torch.cuda.synchronize(dev)
    assert lib.gdn_device_status() == 0
    return o, hT


def check(lib, dev, d, eps=1e-6, path=0):
    o, hT = run(lib, dev, d, eps, path)
    o_ref, h_ref = sublayer.fused_forward(
        d["q"], d["k"], d["v"], d["a"], d["b"], d["h0"],
        cu_seqlens=d["cu_seqlens"], weight=d["norm_weight"], gate=d["gate"],
        eps=eps)
    assert rel_err(o, o_ref) <= TOL, rel_err(o, o_ref)
    assert rel_err(hT, h_ref) <= TOL, rel_err(hT, h_ref)


@pytest.mark.parametrize("path", CHAINS + [FUSED])
@pytest.mark.parametrize("dv", [64, 128])
@pytest.mark.parametrize("weight,gate", [(True, True), (True, False),
                                         (False, True), (False, False)])
def test_fused_matches_oracle(lib, cuda_device, dv, weight, gate, path):
    d = inputs.fused_inputs(2, 3, 200, 128, dv, seed=11, h0=True,
                            weight=weight, gate=gate)
    check(lib, cuda_device, d, path=path)


@pytest.mark.parametrize("path", CHAINS + [FUSED])
@pytest.mark.parametrize("T", [1, 63, 65, 130])
def test_fused_short_and_ragged(lib, cuda_device, T, path):
    d = inputs.fused_inputs(1, 2, T, 128, 128, seed=12)
    check(lib, cuda_device, d, path=path)


@pytest.mark.parametrize("path", CHAINS + [FUSED])
def test_fused_packed(lib, cuda_device, path):
    d = inputs.fused_inputs(0, 4, 0, 128, 128, seed=13, h0=True,
                            lengths=[70, 1, 0, 300, 64, 129])
    check(lib, cuda_device, d, path=path)


@pytest.mark.parametrize("path", [0] + CHAINS)
def test_fused_long_sequence_split(lib, cuda_device, path):
    # long enough for the automatic sequence-parallel split
    d = inputs.fused_inputs(1, 2, 6000, 128, 128, seed=14, h0=True)
    check(lib, cuda_device, d, path=path)


def test_fused_unit_inputs_reduce_to_the_plain_path(lib, cuda_device):
    """With a unit weight, no gate and eps = 0 every output row has unit RMS;
    the final state equals the plain entry point's on the normalised inputs."""
    d = inputs.fused_inputs(1, 2, 256, 128, 128, seed=15, weight=False,
                            gate=False)
    d["norm_weight"] = torch.ones(128)
    o, hT = run(lib, cuda_device, d, eps=0.0)
    ms = o.float().pow(2).mean(-1)
    assert torch.allclose(ms, torch.ones_like(ms), atol=2e-2)
    q, k, g, beta = sublayer.prologue(d["q"], d["k"], d["a"], d["b"])
    dev = cuda_device
    o2, h2 = lib.gdn_chunk_fwd(
        torch.from_numpy(q).to(torch.bfloat16).to(dev),
        torch.from_numpy(k).to(torch.bfloat16).to(dev), d["v"].to(dev),
        torch.from_numpy(g).float().to(dev), torch.from_numpy(beta).float().to(dev))
    torch.cuda.synchronize(dev)
    h_ref = h2.cpu().numpy().astype(np.float64)
    assert rel_err(hT, h_ref) <= TOL


def test_fused_bench_size_sampled(lib, cuda_device):
    """B=4, H=16, T=2048 (the fused bench workload) in the bench's launch
    configuration; two (sequence, head) pairs checked against the oracle
    (heads are independent and the norm weight is shared, so the oracle runs
    on their slices only)."""
    d = inputs.fused_inputs(4, 16, 2048, 128, 128, seed=12, h0=False)
    o, hT = run(lib, cuda_device, d)
    for n, h in ((0, 0), (2, 9)):
        sl = lambda t: None if t is None else t[n:n + 1, :, h:h + 1]
        o_ref, h_ref = sublayer.fused_forward(
            sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["a"]), sl(d["b"]), None,
            weight=d["norm_weight"], gate=sl(d["gate"]), eps=1e-6)
        assert rel_err(o[n:n + 1, :, h:h + 1], o_ref) <= TOL
        assert rel_err(hT[n:n + 1, h:h + 1], h_ref) <= TOL

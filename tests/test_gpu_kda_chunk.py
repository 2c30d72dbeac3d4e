"""The chunk form of KDA on the tensor cores (gdn_kda_fwd_ex, path
GDN_PATH_TCGEN05: kda_prep_kernel + the whole-state chain kernel) against the
fp64 oracle (oracle/kda.py, token by token) on the same seeded inputs,
element by element.

Bound: max|X_gpu - X_ref| / max|X_ref| <= 2e-2, the bf16 bound of the
scalar-gate chunk path (the same chain: bf16 operands, fp32 accumulators and
state, bf16 outputs).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import kda
from gated_deltanet_chunkwise_gb300 import inputs

pytestmark = pytest.mark.gpu
TOL = 2e-2
TC = 2           # GDN_PATH_TCGEN05
SP_CHAIN, SP_SCAN = 0x100, 0x200


def rel_err(x, ref):
    x = x.detach().float().cpu().numpy() if hasattr(x, "detach") else x
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


def run(lib, dev, d, path=TC, sp_parts=0):
    g = lambda t: None if t is None else t.to(dev)
    out = torch.full(d["v"].shape, float("nan"), dtype=torch.bfloat16, device=dev)
    o, hT = lib.gdn_kda_fwd_ex(g(d["q"]), g(d["k"]), g(d["v"]), g(d["g"]),
                               g(d["beta"]), g(d["h0"]), g(d["cu_seqlens"]),
                               out=out, path=path, sp_parts=sp_parts)
    torch.cuda.synchronize(dev)
    assert lib.gdn_device_status() == 0
    return o, hT


def check(lib, dev, d, **kw):
    o, hT = run(lib, dev, d, **kw)
    o_ref, h_ref = kda.forward(d["q"], d["k"], d["v"], d["g"], d["beta"],
                               d["h0"], cu_seqlens=d["cu_seqlens"])
    eo, eh = rel_err(o, o_ref), rel_err(hT, h_ref)
    assert eo <= TOL and eh <= TOL, (eo, eh)
    return eo, eh


@pytest.mark.parametrize("dv", [64, 128])
@pytest.mark.parametrize("h0", [False, True])
def test_kda_chunk_matches_oracle(lib, cuda_device, dv, h0):
    # two full chunks and a ragged one
    d = inputs.kda_inputs(2, 3, 64 * 2 + 37, 128, dv, seed=41, h0=h0)
    check(lib, cuda_device, d)


@pytest.mark.parametrize("T", [1, 15, 16, 17, 63, 64, 65, 128, 300])
def test_kda_chunk_lengths(lib, cuda_device, T):
    d = inputs.kda_inputs(1, 2, T, 128, 128, seed=42, h0=True)
    check(lib, cuda_device, d)


def test_kda_chunk_packed(lib, cuda_device):
    d = inputs.kda_inputs(0, 2, 0, 128, 64, seed=43, h0=True,
                          lengths=[40, 0, 1, 16, 129, 3, 200])
    check(lib, cuda_device, d)


def test_kda_chunk_auto_takes_the_chunk_form(lib, cuda_device):
    d = inputs.kda_inputs(1, 2, 150, 128, 128, seed=44, h0=True)
    lib.gdn_timing_enable(True)
    try:
        run(lib, cuda_device, d, path=0)
        t = lib.kernel_timings()
    finally:
        lib.gdn_timing_enable(False)
    # (a short sequence on few heads may also be split into sub-sequences:
    # one or two chain passes)
    assert t.get("kda_prep_kernel", (0, 0))[0] == 1
    assert t.get("chain_tx_kernel", (0, 0))[0] in (1, 2)
    assert "kda_kernel" not in t and "ut_prep_kernel" not in t


def test_kda_chunk_agrees_with_token_serial(lib, cuda_device):
    d = inputs.kda_inputs(2, 2, 257, 128, 128, seed=45, h0=True)
    o1, h1 = run(lib, cuda_device, d, path=TC)
    o2, h2 = run(lib, cuda_device, d, path=1)
    o_ref, h_ref = kda.forward(d["q"], d["k"], d["v"], d["g"], d["beta"],
                               d["h0"])
    assert rel_err(o1, o2.float().cpu().numpy()) <= 2 * TOL
    assert rel_err(h1, h2.cpu().numpy()) <= 2 * TOL
    assert rel_err(o1, o_ref) <= TOL and rel_err(o2, o_ref) <= TOL


def test_kda_chunk_equal_channels_is_the_scalar_gate(lib, cuda_device):
    """One log-decay for every channel: the scalar-gate recurrence (decay
    before the prediction), checked against that oracle."""
    d = inputs.chunk_inputs(2, 2, 150, 128, 128, dtype="bf16", seed=46, h0=True)
    g1 = d["g"]
    d["g"] = g1[..., None].expand(*g1.shape, 128).contiguous()
    o, hT = run(lib, cuda_device, d)
    o_ref, h_ref = oracle.forward(d["q"], d["k"], d["v"], g1, d["beta"],
                                  d["h0"], variant=oracle.G1)
    assert rel_err(o, o_ref) <= TOL
    assert rel_err(hT, h_ref) <= TOL


@pytest.mark.parametrize("where", ["first", "middle", "last"])
def test_kda_chunk_exact_fallback_for_steep_decays(lib, cuda_device, where):
    """A channel that decays by e^-100 at one token (2^-144, beyond the
    tables' 2^120 range within a 16-token block) sends its chunk to the exact
    pairwise sum; the result still matches the oracle."""
    d = inputs.kda_inputs(1, 2, 200, 128, 128, seed=47, h0=True)
    t = {"first": 1, "middle": 70, "last": 199}[where]
    d["g"][0, t, 0, 5] = -100.0
    d["g"][0, t, 1, 77] = -100.0
    check(lib, cuda_device, d)


def test_kda_chunk_zero_decay(lib, cuda_device):
    """g = 0 everywhere: the ungated delta rule."""
    d = inputs.kda_inputs(1, 2, 130, 128, 128, seed=48, h0=True)
    d["g"].zero_()
    check(lib, cuda_device, d)


@pytest.mark.parametrize("mode", [SP_CHAIN, SP_SCAN])
@pytest.mark.parametrize("parts", [2, 3, 5])
def test_kda_chunk_sequence_parallel(lib, cuda_device, mode, parts):
    d = inputs.kda_inputs(1, 2, 64 * 20 + 11, 128, 128, seed=49, h0=True)
    check(lib, cuda_device, d, path=TC | mode, sp_parts=parts)


def test_kda_chunk_in_place_state(lib, cuda_device):
    """hT = h0: the state buffer is read before it is overwritten."""
    d = inputs.kda_inputs(2, 2, 100, 128, 128, seed=50, h0=True)
    g = lambda t: t.to(cuda_device)
    state = g(d["h0"])
    out = torch.empty_like(g(d["v"]))
    lib.gdn_kda_fwd_ex(g(d["q"]), g(d["k"]), g(d["v"]), g(d["g"]),
                       g(d["beta"]), state, None, out=out, hT=state, path=TC)
    torch.cuda.synchronize(cuda_device)
    o_ref, h_ref = kda.forward(d["q"], d["k"], d["v"], d["g"], d["beta"],
                               d["h0"])
    assert rel_err(out, o_ref) <= TOL
    assert rel_err(state, h_ref) <= TOL


def test_kda_chunk_bench_size_sampled(lib, cuda_device):
    """B=4, H=16, T=2048 (the KDA bench workload) in the bench's launch
    configuration; two (sequence, head) pairs checked against the oracle
    (heads are independent, so the oracle runs on their slices only)."""
    d = inputs.kda_inputs(4, 16, 2048, 128, 128, seed=51, h0=False)
    o, hT = run(lib, cuda_device, d, path=0)
    for n, h in ((0, 0), (3, 11)):
        sl = lambda x: x[n:n + 1, :, h:h + 1]
        o_ref, h_ref = kda.forward(sl(d["q"]), sl(d["k"]), sl(d["v"]),
                                   sl(d["g"]), sl(d["beta"]))
        assert rel_err(o[n:n + 1, :, h:h + 1], o_ref) <= TOL
        assert rel_err(hT[n:n + 1, h:h + 1], h_ref) <= TOL


def test_kda_token_path_bench_size_sampled(lib, cuda_device):
    """The same workload through the token-by-token kernel (path
    GDN_PATH_SIMT, the bench's --kda-path serial line); two (sequence, head)
    pairs against the oracle on their slices."""
    d = inputs.kda_inputs(4, 16, 2048, 128, 128, seed=52, h0=False)
    o, hT = run(lib, cuda_device, d, path=1)
    for n, h in ((1, 4), (2, 15)):
        sl = lambda x: x[n:n + 1, :, h:h + 1]
        o_ref, h_ref = kda.forward(sl(d["q"]), sl(d["k"]), sl(d["v"]),
                                   sl(d["g"]), sl(d["beta"]))
        assert rel_err(o[n:n + 1, :, h:h + 1], o_ref) <= TOL
        assert rel_err(hT[n:n + 1, h:h + 1], h_ref) <= TOL

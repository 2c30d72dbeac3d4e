"""The binding refuses tensors whose shapes disagree with the sizes it
passes to the library (the kernels index by those sizes, so a mismatched
tensor would be read or written out of bounds): every entry point raises
ValueError before anything is enqueued."""
import pytest
import torch

from gated_deltanet_chunkwise_gb300 import inputs

pytestmark = pytest.mark.gpu


def on(d, dev):
    return {k: (None if v is None else v.to(dev)) for k, v in d.items()}


def test_forward_refuses_mismatched_outputs(lib, cuda_device):
    d = on(inputs.chunk_inputs(1, 2, 40, 64, 64, dtype="bf16", seed=1), cuda_device)
    bad_out = torch.empty((1, 2, 40, 64), dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(ValueError):
        lib.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], out=bad_out)
    bad_hT = torch.empty((1, 2, 64, 32), dtype=torch.float32, device=cuda_device)
    with pytest.raises(ValueError):
        lib.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], hT=bad_hT)
    with pytest.raises(ValueError):
        lib.gdn_chunk_fwd(d["q"], d["k"], d["v"][..., None], d["g"], d["beta"])


def test_kda_refuses_mismatched_out(lib, cuda_device):
    d = on(inputs.kda_inputs(1, 2, 40, 64, 64, seed=2), cuda_device)
    bad_out = torch.empty((1, 40, 2, 32), dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(ValueError):
        lib.gdn_kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], out=bad_out)


def test_fused_backward_refuses_mismatched_inputs(lib, cuda_device):
    d = on(inputs.fused_inputs(1, 2, 40, 64, 64, seed=3), cuda_device)
    dout = torch.zeros_like(d["v"])
    base = dict(norm_weight=d["norm_weight"], gate=d["gate"])
    cases = [
        dict(k=d["k"][:, :20]),
        dict(dout=dout[:, :, :1]),
        dict(a=d["a"][:, :10]),
        dict(norm_weight=d["norm_weight"][:32]),
        dict(gate=d["gate"][..., :32]),
        dict(h0=torch.zeros((1, 2, 64, 32), device=cuda_device)),
    ]
    for case in cases:
        args = dict(q=d["q"], k=d["k"], v=d["v"], a=d["a"], b=d["b"],
                    h0=None, dout=dout)
        kw = dict(base)
        for key, val in case.items():
            (args if key in args else kw)[key] = val
        with pytest.raises(ValueError):
            lib.gdn_chunk_bwd_fused(args["q"], args["k"], args["v"], args["a"],
                                    args["b"], args["h0"], args["dout"], **kw)


def test_decode_refuses_mismatched_inputs(lib, cuda_device):
    d = on(inputs.decode_inputs(4, 2, 64, 64, seed=4), cuda_device)
    with pytest.raises(ValueError):
        lib.gdn_recurrent_step(d["q"], d["k"][:2], d["v"], d["g"], d["beta"],
                               d["state"])
    with pytest.raises(ValueError):
        lib.gdn_recurrent_step(d["q"], d["k"], d["v"], d["g"][:, :1],
                               d["beta"], d["state"])
    bad_out = torch.empty((4, 2, 32), dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(ValueError):
        lib.gdn_recurrent_step(d["q"], d["k"], d["v"], d["g"], d["beta"],
                               d["state"], out=bad_out)

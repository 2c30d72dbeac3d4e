"""GPU parity at the full benchmark workload sizes, through the C ABI, in the
launch configuration the bench times (automatic kernel and split choice).

Workloads (seed 0, the input recipe of ``gated_deltanet_chunkwise_gb300.inputs``):
  W1  B=4, H=16, T=2048, dk=dv=128, C=64, bf16, zero initial state
  W2  B=1, H=16, T=65536, bf16 (sequence-parallel split chosen automatically)
  W3  32 packed sequences, lengths U{256..8192}, H=16, bf16, h0 ~ 0.1 N(0,1)
  W4  decode: N=512, H=32, dk=dv=128, fp32 state ~ 0.1 N(0,1), in place
The oracle finishes each of these in seconds on the host cores, so every
output element and every final state is compared.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_chunkwise_gb300 import inputs

from test_gpu_parity import rel_err, run_gpu

pytestmark = pytest.mark.gpu
TOL_BF16 = 2e-2


def _check_chunk(lib, dev, d):
    o_ref, h_ref = oracle.forward(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                  d["h0"], d["cu_seqlens"])
    out, hT = run_gpu(lib, d, dev, "bf16")
    eo, eh = rel_err(out, o_ref), rel_err(hT, h_ref)
    print(f"rel err out {eo:.3e} state {eh:.3e}")
    assert eo <= TOL_BF16 and eh <= TOL_BF16


def test_w1_dense_batch(lib, cuda_device):
    d = inputs.chunk_inputs(4, 16, 2048, 128, 128, dtype="bf16", seed=0)
    _check_chunk(lib, cuda_device, d)


def test_w2_long_sequence(lib, cuda_device):
    d = inputs.chunk_inputs(1, 16, 65536, 128, 128, dtype="bf16", seed=0)
    _check_chunk(lib, cuda_device, d)


def test_w3_packed_varlen(lib, cuda_device):
    d = inputs.chunk_inputs(32, 16, 0, 128, 128, dtype="bf16", seed=0,
                            h0=True, length_range=(256, 8192))
    _check_chunk(lib, cuda_device, d)


def test_w4_decode(lib, cuda_device):
    d = inputs.decode_inputs(512, 32, 128, 128, dtype="bf16", seed=0)
    o_ref, s_ref = oracle.recurrent_step(d["q"], d["k"], d["v"], d["g"],
                                         d["beta"], d["state"])
    x = {k: v.to(cuda_device) for k, v in d.items()}
    out = lib.gdn_recurrent_step(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                 x["state"])
    torch.cuda.synchronize()
    assert rel_err(out, o_ref) <= TOL_BF16
    assert rel_err(x["state"], s_ref) <= TOL_BF16

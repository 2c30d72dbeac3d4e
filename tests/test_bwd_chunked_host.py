"""The chunk-form backward's kernel bodies (csrc/bwd_chunked_body.cuh) run on
the host, compiled with g++ (tests/host/bwd_chunked_emu.cpp: one std::thread
per CUDA thread, a barrier per CTA; under AddressSanitizer, so an index that
leaves a buffer fails the test), against the fp64 gradient oracle: the
bodies' index arithmetic and algebra are checked without a GPU. The GPU
kernels instantiate the same bodies (tests/test_gpu_bwd_chunked.py)."""
import shutil
import subprocess
from pathlib import Path

import numpy as np
import pytest

from oracle import backward

ROOT = Path(__file__).resolve().parent.parent
SRC = ROOT / "tests" / "host" / "bwd_chunked_emu.cpp"
INC = ROOT / "gated_deltanet_chunkwise_gb300" / "csrc"


@pytest.fixture(scope="module")
def emu(tmp_path_factory):
    if shutil.which("g++") is None:
        pytest.skip("g++ is not available")
    exe = tmp_path_factory.mktemp("emu") / "bwd_chunked_emu"
    cmd = ["g++", "-std=c++20", "-O1", "-g", "-pthread", "-fsanitize=address",
           f"-I{INC}", str(SRC), "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0 and "sanitize" in r.stderr:
        cmd.remove("-fsanitize=address")
        r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    return exe


def run_case(emu, tmp_path, N, H, T, DK, DV, h0, dhT, seed, bf16=False):
    rng = np.random.default_rng(seed)
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    f32 = lambda x: np.ascontiguousarray(x, dtype=np.float32)
    q = f32(unit(rng.standard_normal((N, T, H, DK))))
    k = f32(unit(rng.standard_normal((N, T, H, DK))))
    v = f32(rng.standard_normal((N, T, H, DV)))
    g = f32(-np.log1p(np.exp(rng.standard_normal((N, T, H)))))
    beta = f32(1 / (1 + np.exp(-rng.standard_normal((N, T, H)))))
    dout = f32(rng.standard_normal((N, T, H, DV)))
    H0 = f32(0.1 * rng.standard_normal((N, H, DK, DV))) if h0 else None
    DH = f32(0.1 * rng.standard_normal((N, H, DK, DV))) if dhT else None
    if bf16:
        # round to bf16 (nearest even); the file holds the bit patterns and
        # the oracle reads the rounded values
        import torch
        def to_bf16(x):
            t = torch.from_numpy(x).to(torch.bfloat16)
            return t.view(torch.int16).numpy().view(np.uint16), t.float().numpy()
        (qb, q), (kb, k), (vb, v), (ob, dout) = map(to_bf16, (q, k, v, dout))
        for name, x in (("q", qb), ("k", kb), ("v", vb), ("dout", ob)):
            x.tofile(tmp_path / f"{name}.bin")
    else:
        for name, x in (("q", q), ("k", k), ("v", v), ("dout", dout)):
            x.tofile(tmp_path / f"{name}.bin")
    for name, x in (("g", g), ("beta", beta), ("h0", H0), ("dhT", DH)):
        if x is not None:
            x.tofile(tmp_path / f"{name}.bin")
    r = subprocess.run([str(emu), str(tmp_path), str(N), str(H), str(T),
                        str(DK), str(DV), str(int(h0)), str(int(dhT)),
                        str(int(bf16))],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    ref = backward.backward(q, k, v, g, beta, H0, dout, DH, variant=1)
    shapes = {"dq": q.shape, "dk": k.shape, "dv": v.shape, "dg": g.shape,
              "dbeta": beta.shape, "dh0": (N, H, DK, DV)}
    for name, shp in shapes.items():
        got = np.fromfile(tmp_path / f"{name}.bin", dtype=np.float32).reshape(shp)
        want = np.asarray(ref[name])
        err = np.max(np.abs(got - want)) / max(np.max(np.abs(want)), 1e-30)
        assert err < 1e-4, (name, err)


@pytest.mark.parametrize("N,H,T,DK,DV,h0,dhT", [
    (1, 1, 64, 64, 64, False, False),     # one whole chunk
    (2, 2, 150, 64, 64, True, True),      # ragged last chunk, two sequences
    (1, 1, 129, 128, 128, True, False),
    (1, 1, 200, 64, 128, False, True),
    (2, 1, 65, 128, 64, True, True),
    (1, 1, 1, 64, 64, True, True),        # a single token
])
def test_chunked_bwd_bodies_on_the_host(emu, tmp_path, N, H, T, DK, DV, h0, dhT):
    run_case(emu, tmp_path, N, H, T, DK, DV, h0, dhT, seed=T + DK + DV)


def test_chunked_bwd_bodies_read_bf16_inputs(emu, tmp_path):
    # the GPU entry point's input type: bf16 bit patterns widened in the loads
    run_case(emu, tmp_path, 2, 2, 100, 128, 64, True, True, seed=7, bf16=True)

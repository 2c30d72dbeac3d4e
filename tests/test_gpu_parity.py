"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Acceptance (per output tensor and per final state):
    max|X_gpu - X_ref| / max|X_ref| <= 1e-3 for fp32 inputs, <= 2e-2 for bf16.
Both sides read identical seeded inputs (bf16 values upcast exactly).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_chunkwise_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-3, "bf16": 2e-2}


def rel_err(x, ref):
    x = x.detach().cpu().double().numpy() if hasattr(x, "detach") else x
    denom = np.max(np.abs(ref))
    assert np.all(np.isfinite(x)), "non-finite values in the GPU result"
    return float(np.max(np.abs(x - ref)) / max(denom, 1e-30))


def to_dev(d, dev):
    return {k: (None if v is None else v.to(dev)) for k, v in d.items()}


def run_gpu(lib, d, dev, dtype, variant=0, path=0, sp_parts=0, poison=True):
    x = to_dev(d, dev)
    out = torch.empty_like(x["v"])
    N = x["h0"].shape[0] if x["h0"] is not None else (
        x["cu_seqlens"].numel() - 1 if x["cu_seqlens"] is not None
        else x["q"].shape[0])
    H, dk, dv = x["q"].shape[2], x["q"].shape[3], x["v"].shape[3]
    hT = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    if poison:  # unwritten elements would surface as NaN
        out.fill_(float("nan"))
        hT.fill_(float("nan"))
    lib.gdn_chunk_fwd_ex(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                         x["cu_seqlens"], out=out, hT=hT, variant=variant,
                         path=path, sp_parts=sp_parts)
    torch.cuda.synchronize()
    assert lib.gdn_device_status() == 0
    return out, hT


def oracle_variant(abi_variant):
    """The ABI numbers gate placements 0 = decay first, 1 = decay after the
    prediction; the oracle names them G1 and G0."""
    return oracle.G1 if abi_variant == 0 else oracle.G0


def check(lib, dev, d, dtype, variant=0, path=0, sp_parts=0):
    o_ref, h_ref = oracle.forward(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                  d["h0"], d["cu_seqlens"],
                                  variant=oracle_variant(variant))
    out, hT = run_gpu(lib, d, dev, dtype, variant, path, sp_parts)
    eo, eh = rel_err(out, o_ref), rel_err(hT, h_ref)
    assert eo <= TOL[dtype], f"output rel err {eo:.3e}"
    assert eh <= TOL[dtype], f"final-state rel err {eh:.3e}"
    return eo, eh


# ---- workload 0: B=1, H=1, T=256, dk=dv=64, fp32, gated and alpha = 1 ----
@pytest.mark.parametrize("gated", [True, False])
def test_small_fp32_gated_and_deltanet(lib, cuda_device, gated):
    d = inputs.chunk_inputs(1, 1, 256, 64, 64, dtype="f32", seed=0,
                            gated=gated)
    check(lib, cuda_device, d, "f32")


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ragged_multi_chunk_shapes(lib, cuda_device, dk, dv, dtype):
    # several chunks plus a ragged tail, nonzero initial states
    d = inputs.chunk_inputs(2, 3, 64 * 3 + 17, dk, dv, dtype=dtype, seed=1,
                            h0=True)
    check(lib, cuda_device, d, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gate_after_prediction_variant(lib, cuda_device, dtype):
    d = inputs.chunk_inputs(2, 2, 150, 64, 64, dtype=dtype, seed=2, h0=True)
    check(lib, cuda_device, d, dtype, variant=1)


@pytest.mark.parametrize("T", [1, 5, 63, 64, 65])
def test_short_and_boundary_lengths(lib, cuda_device, T):
    d = inputs.chunk_inputs(1, 2, T, 128, 128, dtype="f32", seed=3, h0=True)
    check(lib, cuda_device, d, "f32")


@pytest.mark.parametrize("parts", [2, 3, 5])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sequence_parallel_split_matches_oracle(lib, cuda_device, parts,
                                                dtype):
    d = inputs.chunk_inputs(2, 2, 64 * 9 + 40, 64, 128, dtype=dtype, seed=4,
                            h0=True)
    check(lib, cuda_device, d, dtype, sp_parts=parts)


def test_sequence_parallel_more_parts_than_chunks(lib, cuda_device):
    d = inputs.chunk_inputs(1, 2, 64 * 2 + 3, 64, 64, dtype="f32", seed=5,
                            h0=True)
    check(lib, cuda_device, d, "f32", sp_parts=6)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_packed_sequences_with_empty_and_short(lib, cuda_device, dtype):
    lengths = [70, 0, 1, 64, 200, 3]
    d = inputs.chunk_inputs(len(lengths), 2, 0, 128, 64, dtype=dtype, seed=6,
                            h0=True, lengths=lengths)
    check(lib, cuda_device, d, dtype)


def test_packed_sequences_sequence_parallel(lib, cuda_device):
    lengths = [300, 5, 640]
    d = inputs.chunk_inputs(len(lengths), 2, 0, 64, 64, dtype="f32", seed=7,
                            h0=True, lengths=lengths)
    check(lib, cuda_device, d, "f32", sp_parts=3)


# ---- sub-sequences combined by the associative scan (GDN_SP_SCAN) ----
SP_SCAN = 0x200


@pytest.mark.parametrize("parts", [3, 4, 6, 11])
@pytest.mark.parametrize("dtype,dk", [("f32", 64), ("f32", 128), ("bf16", 128)])
def test_sequence_parallel_scan_matches_oracle(lib, cuda_device, parts, dtype,
                                               dk):
    d = inputs.chunk_inputs(2, 2, 64 * 13 + 21, dk, 64, dtype=dtype, seed=19,
                            h0=True)
    check(lib, cuda_device, d, dtype, path=SP_SCAN, sp_parts=parts)


@pytest.mark.parametrize("path", [3, 4])
def test_sequence_parallel_scan_tensor_core(lib, cuda_device, path):
    d = inputs.chunk_inputs(1, 2, 64 * 19 + 40, 128, 128, dtype="bf16",
                            seed=20, h0=True)
    check(lib, cuda_device, d, "bf16", path=path | SP_SCAN, sp_parts=9)


def test_packed_sequences_scan(lib, cuda_device):
    lengths = [300, 5, 640, 0, 129]
    d = inputs.chunk_inputs(len(lengths), 2, 0, 64, 64, dtype="f32", seed=21,
                            h0=True, lengths=lengths)
    check(lib, cuda_device, d, "f32", path=SP_SCAN, sp_parts=7)


def test_resume_through_final_state(lib, cuda_device):
    d = inputs.chunk_inputs(2, 2, 300, 128, 128, dtype="f32", seed=8, h0=True)
    x = to_dev(d, cuda_device)
    o_all, h_all = lib.gdn_chunk_fwd_f32(x["q"], x["k"], x["v"], x["g"],
                                         x["beta"], x["h0"])
    t = 131
    part = lambda a, s: a[:, s].contiguous()
    o1, h1 = lib.gdn_chunk_fwd_f32(*(part(x[n], slice(0, t)) for n in
                                     ("q", "k", "v", "g", "beta")), x["h0"])
    o2, h2 = lib.gdn_chunk_fwd_f32(*(part(x[n], slice(t, None)) for n in
                                     ("q", "k", "v", "g", "beta")), h1)
    torch.cuda.synchronize()
    o_cat = torch.cat([o1, o2], 1)
    ref = o_all.double().cpu().numpy()
    assert rel_err(o_cat, ref) <= 1e-4
    assert rel_err(h2, h_all.double().cpu().numpy()) <= 1e-4


def test_invalid_packing_is_reported_on_device(lib, cuda_device):
    d = inputs.chunk_inputs(2, 1, 0, 64, 64, dtype="f32", seed=9,
                            lengths=[10, 20])
    x = to_dev(d, cuda_device)
    cu = torch.tensor([0, 25, 20], dtype=torch.int32, device=cuda_device)
    lib.gdn_device_status()  # clear
    lib.gdn_chunk_fwd_f32(x["q"], x["k"], x["v"], x["g"], x["beta"], None,
                          cu)
    assert lib.gdn_device_status() == -1
    assert lib.gdn_device_status() == 0  # cleared by the read


# ---- decode step ----
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 64), (64, 128), (128, 128)])
def test_recurrent_step_small(lib, cuda_device, dk, dv):
    d = inputs.decode_inputs(7, 3, dk, dv, seed=10)
    o_ref, s_ref = oracle.recurrent_step(d["q"], d["k"], d["v"], d["g"],
                                         d["beta"], d["state"])
    x = to_dev(d, cuda_device)
    out = lib.gdn_recurrent_step(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                 x["state"])
    torch.cuda.synchronize()
    assert rel_err(out, o_ref) <= TOL["bf16"]
    assert rel_err(x["state"], s_ref) <= 1e-5  # fp32 state, bf16 token


def test_recurrent_step_matches_chunk_path_single_token(lib, cuda_device):
    d = inputs.decode_inputs(4, 2, 128, 128, seed=11)
    x = to_dev(d, cuda_device)
    h0 = x["state"].clone()
    o_c, h_c = lib.gdn_chunk_fwd(x["q"][:, None].contiguous(),
                                 x["k"][:, None].contiguous(),
                                 x["v"][:, None].contiguous(),
                                 x["g"][:, None].contiguous(),
                                 x["beta"][:, None].contiguous(), h0)
    o_d = lib.gdn_recurrent_step(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                 x["state"])
    torch.cuda.synchronize()
    # the bf16 chunk path multiplies by a bf16 copy of the state, so the two
    # agree to the bf16 parity bound, not to fp32 rounding
    assert rel_err(x["state"], h_c.double().cpu().numpy()) <= TOL["bf16"]
    assert rel_err(o_d, o_c[:, 0].double().cpu().numpy()) <= TOL["bf16"]


# ---- tensor-core (tcgen05) path, forced ----
TC = 2
# its two chain kernels, forced: 64 state rows per CTA, 128 rows per CTA
CHAINS = [3, 4]
# the single-launch form (preparation and chain of a (sequence, head) in one
# cluster, no workspace), forced; it takes no sequence-parallel split
FUSED = 5


@pytest.mark.parametrize("path", [TC] + CHAINS + [FUSED])
@pytest.mark.parametrize("dv", [64, 128])
@pytest.mark.parametrize("variant", [0, 1])
def test_tensor_core_path(lib, cuda_device, dv, variant, path):
    d = inputs.chunk_inputs(2, 3, 64 * 4 + 29, 128, dv, dtype="bf16", seed=12,
                            h0=True)
    check(lib, cuda_device, d, "bf16", variant=variant, path=path)


@pytest.mark.parametrize("path", CHAINS + [FUSED])
def test_tensor_core_alpha_one_single_chunk(lib, cuda_device, path):
    d = inputs.chunk_inputs(1, 2, 64, 128, 128, dtype="bf16", seed=13,
                            gated=False)
    check(lib, cuda_device, d, "bf16", path=path)


@pytest.mark.parametrize("path", CHAINS + [FUSED])
@pytest.mark.parametrize("T", [1, 17, 63, 65, 128, 64 * 7 + 5])
def test_tensor_core_short_lengths(lib, cuda_device, T, path):
    d = inputs.chunk_inputs(2, 2, T, 128, 128, dtype="bf16", seed=14, h0=True)
    check(lib, cuda_device, d, "bf16", path=path)


@pytest.mark.parametrize("path", CHAINS)
@pytest.mark.parametrize("dv", [64, 128])
@pytest.mark.parametrize("parts", [2, 3, 5])
def test_tensor_core_sequence_parallel(lib, cuda_device, parts, dv, path):
    d = inputs.chunk_inputs(1, 2, 64 * 9 + 40, 128, dv, dtype="bf16", seed=15,
                            h0=True)
    check(lib, cuda_device, d, "bf16", path=path, sp_parts=parts)


@pytest.mark.parametrize("path", CHAINS + [FUSED])
def test_tensor_core_packed(lib, cuda_device, path):
    lengths = [70, 0, 1, 64, 200, 3, 129]
    d = inputs.chunk_inputs(len(lengths), 2, 0, 128, 128, dtype="bf16",
                            seed=16, h0=True, lengths=lengths)
    check(lib, cuda_device, d, "bf16", path=path)


@pytest.mark.parametrize("path", [1] + CHAINS + [FUSED])
def test_strong_gates_chunk_decay_beyond_fp32_range(lib, cuda_device, path):
    """Log-gates ~6x stronger than the workload's, so a chunk's total decay
    exceeds e^-87: the tensor-core kernel must switch from factored decays
    e^{G_r} e^{-G_j} to running products without overflow."""
    d = inputs.chunk_inputs(2, 2, 64 * 3 + 11, 128, 128, dtype="bf16",
                            seed=17, h0=True)
    d["g"] = d["g"] * 6.0
    check(lib, cuda_device, d, "bf16", path=path)


def test_mixed_gate_strength_across_chunks(lib, cuda_device):
    """Weak gates in one chunk, strong in the next: per-chunk path choice."""
    d = inputs.chunk_inputs(1, 2, 64 * 4, 128, 64, dtype="bf16", seed=18,
                            h0=True)
    d["g"][:, 64:128] *= 8.0
    d["g"][:, 192:] *= 5.0
    for path in CHAINS + [FUSED]:
        check(lib, cuda_device, d, "bf16", path=path)


@pytest.mark.gpu
def test_kernel_timing_counts_the_launches(lib, cuda_device):
    """Per-kernel timing sees exactly the launches of each path."""
    d = inputs.chunk_inputs(2, 4, 200, 128, 128, dtype="bf16", seed=5)
    lib.gdn_timing_enable(True)
    try:
        run_gpu(lib, d, cuda_device, "bf16", path=3, sp_parts=1)
        run_gpu(lib, d, cuda_device, "bf16", path=4, sp_parts=1)
        run_gpu(lib, d, cuda_device, "bf16", path=1, sp_parts=1)
        run_gpu(lib, d, cuda_device, "bf16", path=FUSED, sp_parts=1)
        t = lib.kernel_timings()
    finally:
        lib.gdn_timing_enable(False)
    assert t["ut_prep_kernel"][0] == 2
    assert t["chunk_tc_kernel"][0] == 1
    assert t["chain_tx_kernel"][0] == 1
    assert t["chunk_simt_kernel"][0] == 1
    assert t["fused_chunk_kernel"][0] == 1
    assert all(ms > 0 for _, ms in t.values())


@pytest.mark.parametrize("path", [TC] + CHAINS + [FUSED])
@pytest.mark.parametrize("dv", [64, 128])
def test_tensor_core_dk64(lib, cuda_device, dv, path):
    # d_k = 64 runs on the d_k = 128 kernels with the keys' and queries'
    # second 64 columns read as zeros: every state row and column beyond
    # d_k must stay out of h0 / hT and the split's workspace
    d = inputs.chunk_inputs(2, 3, 64 * 4 + 29, 64, dv, dtype="bf16", seed=20,
                            h0=True)
    check(lib, cuda_device, d, "bf16", variant=1 if path == 4 else 0,
          path=path)


@pytest.mark.parametrize("path", CHAINS)
@pytest.mark.parametrize("parts", [2, 5])
def test_tensor_core_dk64_sequence_parallel(lib, cuda_device, parts, path):
    d = inputs.chunk_inputs(1, 2, 64 * 9 + 40, 64, 128, dtype="bf16", seed=21,
                            h0=True)
    check(lib, cuda_device, d, "bf16", path=path, sp_parts=parts)


@pytest.mark.parametrize("path", CHAINS + [FUSED])
def test_tensor_core_dk64_packed(lib, cuda_device, path):
    lengths = [70, 0, 1, 64, 200, 3, 129]
    d = inputs.chunk_inputs(len(lengths), 2, 0, 64, 64, dtype="bf16",
                            seed=22, h0=True, lengths=lengths)
    check(lib, cuda_device, d, "bf16", path=path)


def test_fused_path_rejects_a_split(lib, cuda_device):
    d = to_dev(inputs.chunk_inputs(1, 2, 300, 128, 128, dtype="bf16", seed=6),
               cuda_device)
    with pytest.raises(lib.GdnError) as e:
        lib.gdn_chunk_fwd_ex(d["q"], d["k"], d["v"], d["g"], d["beta"],
                             path=FUSED, sp_parts=3)
    assert e.value.status == -2


@pytest.mark.parametrize("dv", [64, 128])
def test_fused_path_many_chunks_and_heads(lib, cuda_device, dv):
    # more (sequence, head) clusters than SMs hold at once, long enough that
    # every preparation group cycles its stage many times
    d = inputs.chunk_inputs(3, 40, 64 * 21 + 33, 128, dv, dtype="bf16",
                            seed=19, h0=True)
    check(lib, cuda_device, d, "bf16", path=FUSED)

"""Building blocks of the tensor-core kernel, checked on the device.

gdn_selftest_mma lays out A [128, K] and B [K, 64] in shared memory exactly as
the chunk kernel does (128-byte swizzle; K-major or M/N-major; a K-major B in
the first rows of a 128-row stacked tile), runs the tcgen05 MMA sequence with
the kernel's instruction descriptors and reads D back from TMEM. The
reference is the fp32 product of the same bf16 values.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

# (K, N, a_mn, b_mn, b_stacked): the operand forms of the chunk kernel's MMAs
CASES = [
    (128, 64, False, False, True),   # [K;Q] K^T         (K-major A, K-major B)
    (128, 64, False, True, False),   # [-W;Q^] S^T       (K-major A, N-major B)
    (64, 64, False, True, False),    # [T;0] V', [0;P] U (K-major A, N-major B)
    (64, 128, False, True, False),   # [T;T] K'          (N-major B, 2 blocks)
    (64, 64, True, True, False),     # Kbar^T U          (M-major A, N-major B)
    (128, 64, False, False, False),  # dense K-major B
    (64, 128, True, False, False),   # V^T [T_U;0]^T     (M-major A, K-major B)
]

# A in TMEM (bf16 pairs per column): the transposed chain's S and U operands
TMEM_CASES = [
    (128, 128, False),  # S [-W;Q_g]^T  (K-major B, 128 rows)
    (64, 128, True),    # U K_d         (N-major B, 2 blocks)
    (64, 64, False),    # U P^T         (K-major B)
    (128, 64, True),
]


@pytest.mark.parametrize("K,N,b_mn", TMEM_CASES)
@pytest.mark.parametrize("twice", [False, True])
def test_mma_a_in_tmem(lib, cuda_device, K, N, b_mn, twice):
    g = torch.Generator(device="cpu").manual_seed(K * 5 + N + b_mn)
    A = torch.randn(128, K, generator=g).to(torch.bfloat16)
    B = torch.randn(K, N, generator=g).to(torch.bfloat16)
    ref = (A.double() @ B.double()) * (2 if twice else 1)
    D = lib.gdn_selftest_mma(A.to(cuda_device), B.to(cuda_device),
                             a_tmem=True, b_mn=b_mn, twice=twice)
    torch.cuda.synchronize()
    err = (D.double().cpu() - ref).abs().max().item()
    assert err <= 1e-3 * ref.abs().max().item(), f"max abs err {err}"


@pytest.mark.parametrize("K,N,a_mn,b_mn,b_stacked", CASES)
@pytest.mark.parametrize("twice", [False, True])
def test_mma_layouts(lib, cuda_device, K, N, a_mn, b_mn, b_stacked, twice):
    g = torch.Generator(device="cpu").manual_seed(K * 7 + N + a_mn * 3 + b_mn)
    A = torch.randn(128, K, generator=g).to(torch.bfloat16)
    B = torch.randn(K, N, generator=g).to(torch.bfloat16)
    ref = (A.double() @ B.double()) * (2 if twice else 1)
    D = lib.gdn_selftest_mma(A.to(cuda_device), B.to(cuda_device), a_mn=a_mn,
                             b_mn=b_mn, b_stacked=b_stacked, twice=twice)
    torch.cuda.synchronize()
    err = (D.double().cpu() - ref).abs().max().item()
    assert err <= 1e-3 * ref.abs().max().item(), f"max abs err {err}"

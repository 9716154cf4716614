"""Tensor-core operand encodings used by the prefill kernel, on one tile:
shared-memory descriptors with the 128-byte swizzle (K-major and N-major),
A staged through tensor memory, and the instruction descriptor."""
import pytest
import torch


@pytest.mark.gpu
def test_selftest_umma_matches_torch(swa):
    g = torch.Generator(device="cuda").manual_seed(0)
    A = torch.randn(128, 128, generator=g, device="cuda").to(torch.bfloat16)
    Bk = torch.randn(128, 128, generator=g, device="cuda").to(torch.bfloat16)
    Bn = torch.randn(128, 128, generator=g, device="cuda").to(torch.bfloat16)
    D1, D2 = swa.selftest_umma(A, Bk, Bn)
    torch.cuda.synchronize()
    assert swa.device_status() == 0
    ref1 = A.double() @ Bk.double().T
    ref2 = A.double() @ Bn.double()
    assert (D1.double() - ref1).abs().max().item() < 1e-3
    assert (D2.double() - ref2).abs().max().item() < 1e-3

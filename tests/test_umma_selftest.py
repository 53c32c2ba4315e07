"""The tcgen05 descriptors the bf16 kernel uses, checked on one GEMM tile
against a host matmul of the same bf16 values (GPU)."""
import pytest
import torch

import masked_head_attention_gb300 as mha
from parity_util import randn


@pytest.mark.gpu
@pytest.mark.parametrize("variant,kn", [(0, 64), (0, 128), (1, 64), (1, 128), (2, 64), (2, 128)])
def test_umma_tile(variant, kn):
    seed = 100 * variant + kn
    if variant == 0:
        a = randn((128, kn), seed, dtype=torch.bfloat16)
        b = randn((128, kn), seed + 1, dtype=torch.bfloat16)
        ref = a.double() @ b.double().T
    else:
        a = randn((128, 128), seed, dtype=torch.bfloat16)
        b = randn((128, kn), seed + 1, dtype=torch.bfloat16)
        ref = a.double() @ b.double()
    c = torch.full(ref.shape, float("nan"), dtype=torch.float32, device="cuda")
    mha.selftest_umma(variant, kn, a.cuda(), b.cuda(), c)
    torch.cuda.synchronize()
    err = (c.cpu().double() - ref).abs().max().item()
    assert err < 1e-3, "variant %d kn %d: max abs %.3g" % (variant, kn, err)
    assert mha.device_status() == 0

"""GPU parity of the contraction GW = scale * g^T X on its own (through the C
ABI): the tcgen05 tensor-core kernel and the CUDA-core kernel against an
fp64 product of the same bf16 values. Only fp32 accumulation separates the
two, so the bound is 1e-5 normwise relative."""
import numpy as np
import pytest

import token_perturbation_estimator_gb300 as dust
from helpers import cuda, rel_fro

pytestmark = pytest.mark.gpu

SHAPES = [
    # T, d_in, d_out
    (64, 256, 128),        # one tile, one k-step
    (1000, 512, 2048),     # ragged T, split tokens
    (4096, 1024, 3072),
    (333, 72, 136),        # tails in every dimension
    (128, 8, 8),           # smallest tensor-core shape
    (16384, 512, 512),
    (77, 520, 264),
    # token-slice counts of the tensor-core kernel: up to 8 reduce inside a
    # thread-block cluster (uneven row blocks when 128 is not a multiple),
    # more through fp32 partials and a reduction kernel
    (8192, 512, 4096),     # 2 slices
    (4096, 512, 1152),     # 8 slices
    (2048, 512, 2560),     # 3 slices: row blocks of 43, 43, 42
    (2000, 256, 3840),     # 5 slices: row blocks of 26, the last 24
    (2000, 256, 2688),     # 7 slices: row blocks of 19, the last 14
    (16384, 256, 256),     # 64 slices: partials
    # 256-channel tiles (two accumulators), where every token slice keeps at
    # least 4096 tokens: 4 slices through partials; 5 slices with ragged
    # channels, inputs and tokens; one slice
    (16384, 1024, 2048),
    (24600, 520, 2056),
    (4096, 2048, 4096),
]


@pytest.mark.parametrize("T,d_in,d_out", SHAPES)
@pytest.mark.parametrize("force", [0, dust.FORCE_SIMT])
def test_contract_bf16(T, d_in, d_out, force):
    import torch
    dev = cuda()
    gen = torch.Generator().manual_seed(T + d_in + d_out)
    g = torch.randn((T, d_out), generator=gen).to(torch.bfloat16)
    X = torch.randn((T, d_in), generator=gen).to(torch.bfloat16)
    want = 0.5 * (g.double().numpy().T @ X.double().numpy())
    got = dust.dust_contract(g.to(dev), X.to(dev), 0.5, force).cpu().numpy()
    assert rel_fro(got, want) <= 1e-5
    # accumulate into an existing gradient
    base = torch.randn((d_out, d_in), generator=gen)
    acc = dust.dust_contract(g.to(dev), X.to(dev), 0.5, force | dust.ACCUMULATE,
                             gW=base.clone().to(dev)).cpu().numpy()
    assert rel_fro(acc, want + base.double().numpy()) <= 1e-5


def test_contract_f32_and_empty():
    import torch
    dev = cuda()
    gen = torch.Generator().manual_seed(5)
    g = torch.randn((300, 40), generator=gen)
    X = torch.randn((300, 24), generator=gen)
    got = dust.dust_contract(g.to(dev), X.to(dev)).cpu().numpy()
    assert rel_fro(got, g.double().numpy().T @ X.double().numpy()) <= 1e-6
    e = dust.dust_contract(torch.empty((0, 16), dtype=torch.bfloat16, device=dev),
                           torch.empty((0, 8), dtype=torch.bfloat16, device=dev))
    assert torch.count_nonzero(e).item() == 0


def test_contract_tensor_core_deterministic():
    import torch
    dev = cuda()
    gen = torch.Generator().manual_seed(9)
    g = torch.randn((8192, 2048), generator=gen).to(torch.bfloat16).to(dev)
    X = torch.randn((8192, 512), generator=gen).to(torch.bfloat16).to(dev)
    a = dust.dust_contract(g, X)
    b = dust.dust_contract(g, X)
    assert torch.equal(a, b)
    # 256-channel tiles, 4 token slices through fp32 partials
    g2 = torch.randn((16384, 2048), generator=gen).to(torch.bfloat16).to(dev)
    X2 = torch.randn((16384, 1024), generator=gen).to(torch.bfloat16).to(dev)
    assert torch.equal(dust.dust_contract(g2, X2), dust.dust_contract(g2, X2))
    assert dust.dust_last_error() == dust.OK

"""The Python binding checks dtypes and shapes before any C call: the C ABI
takes raw device pointers and sizes, so a float64 loss-change tensor would
be misread and an output of the wrong shape written past its end."""
import pytest

import token_perturbation_estimator_gb300 as dust
from helpers import cuda

pytestmark = pytest.mark.gpu


def test_binding_rejects_misshaped_buffers_before_launch():
    import torch
    dev = cuda()
    delta = torch.zeros((4, 100), device=dev)
    so = torch.tensor([0, 100], dtype=torch.int32, device=dev)
    with pytest.raises(ValueError):
        dust.dust_credit_scan(delta.double(), so, 0.5)
    with pytest.raises(ValueError):
        dust.dust_credit_scan(delta, so.long(), 0.5)
    with pytest.raises(ValueError):
        dust.dust_credit_scan(delta, so, 0.5, r=torch.empty((100, 3), device=dev))
    with pytest.raises(ValueError):
        dust.dust_credit_scan_noalloc(delta, so, 0.5, r=torch.empty((99, 4), device=dev))
    with pytest.raises(ValueError):
        dust.dust_error_estimate(torch.zeros((100, 4), dtype=torch.float64, device=dev), 64, 0,
                                 dust.GAUSSIAN, 0, 1e-3)

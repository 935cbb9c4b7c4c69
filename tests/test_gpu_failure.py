"""Failure detection on the GPU without a fault: a bounded device-side wait is
made to run out (an mbarrier no thread arrives at, via the library's test
hook). The kernel must return, dust_last_error must report DUST_ERR_TIMEOUT
once, and the context must stay usable: the next call is correct."""
import time

import numpy as np
import pytest

import token_perturbation_estimator_gb300 as dust
from helpers import cuda, rel_fro

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,d_in,d_out", [
    (128, 128, 256),    # one slice: direct write
    (2048, 128, 256),   # 8 slices reduced inside a cluster: every CTA times out together
    (4096, 256, 128),   # 16 slices: partials and the reduction kernel
])
def test_bounded_wait_timeout_is_reported_and_context_survives(T, d_in, d_out):
    import torch
    dev = cuda()
    gen = torch.Generator().manual_seed(3)
    g = torch.randn((T, d_out), generator=gen).to(torch.bfloat16).to(dev)
    X = torch.randn((T, d_in), generator=gen).to(torch.bfloat16).to(dev)
    want = g.double().cpu().numpy().T @ X.double().cpu().numpy()
    assert dust.dust_last_error() == dust.OK
    dust.lib().dust_debug_inject_timeout(1)
    t0 = time.time()
    dust.dust_contract(g, X)
    st = dust.dust_last_error()  # synchronises
    elapsed = time.time() - t0
    assert st == dust.ERR_TIMEOUT, dust.status_string(st)
    assert 0.5 < elapsed < 30.0
    assert dust.dust_last_error() == dust.OK  # cleared after reading
    # the hook is one-shot and the context is healthy: the next call is exact
    got = dust.dust_contract(g, X).cpu().numpy()
    assert dust.dust_last_error() == dust.OK
    assert rel_fro(got, want) <= 1e-5

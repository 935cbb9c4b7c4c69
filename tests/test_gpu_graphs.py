"""Repeated identical estimator calls replay a captured CUDA graph (the
second call with the same arguments captures, later ones launch it). The
graph must do exactly the direct launches' work on the buffers' current
contents: new values written into the same input buffers between replays
give the results of direct launches (profiling on: graphs bypassed), bit for
bit. (The host-buffer entry point always launches directly; its repeated
calls are checked the same way.)"""
import numpy as np
import pytest

import token_perturbation_estimator_gb300 as dust
from helpers import cuda, offsets_from_lengths, random_lengths

pytestmark = pytest.mark.gpu

T, D_IN, D_OUT, K = 8192, 256, 512, 8


def _direct(fn, *a, **kw):
    """One call with graphs bypassed (they are while profiling is on)."""
    dust.dust_profile_enable(True)
    try:
        return fn(*a, **kw)
    finally:
        dust.dust_profile_enable(False)
        dust.dust_profile_read()


def _fill(rng, X, delta):
    import torch
    X.copy_(torch.from_numpy(rng.standard_normal(tuple(X.shape)).astype(np.float32)))
    delta.copy_(torch.from_numpy((0.05 * rng.standard_normal(tuple(delta.shape)))
                                 .astype(np.float32)))


@pytest.mark.parametrize("flags", [dust.CENTER, dust.CENTER | dust.ANTITHETIC])
def test_replays_follow_buffer_contents_device(flags):
    import torch
    dev = cuda()
    rng = np.random.default_rng(31)
    so = torch.from_numpy(offsets_from_lengths(random_lengths(rng, T, 900))).to(dev)
    X = torch.empty((T, D_IN), dtype=torch.bfloat16, device=dev)
    delta = torch.empty((K, T), dtype=torch.float32, device=dev)
    gW = torch.empty((D_OUT, D_IN), dtype=torch.float32, device=dev)
    gW2 = torch.empty_like(gW)
    ws = torch.empty(dust.dust_estimate_gW_workspace(T, D_IN, D_OUT, K, dust.BF16, flags),
                     dtype=torch.uint8, device=dev)
    args = (D_OUT, so, 9, 1, 0, 1e-3, 0.9, 0.5, flags)
    for i in range(5):  # direct, capture, then three replays
        _fill(rng, X, delta)
        dust.dust_estimate_gW(X, delta, *args, gW=gW, workspace=ws)
        want = _direct(dust.dust_estimate_gW, X, delta, *args, gW=gW2, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(gW, want), i
    assert dust.dust_last_error() == dust.OK


def test_replays_follow_buffer_contents_host():
    import torch
    dev = cuda()
    rng = np.random.default_rng(32)
    so = torch.from_numpy(offsets_from_lengths(random_lengths(rng, T, 900)))
    Xh = torch.empty((T, D_IN), dtype=torch.bfloat16).pin_memory()
    dh = torch.empty((K, T), dtype=torch.float32).pin_memory()
    sh = so.pin_memory()
    gh = torch.empty((D_OUT, D_IN), dtype=torch.float32).pin_memory()
    Xd, dd, sd = torch.empty_like(Xh, device=dev), torch.empty_like(dh, device=dev), \
        torch.empty_like(sh, device=dev)
    gd = torch.empty((D_OUT, D_IN), dtype=torch.float32, device=dev)
    for i in range(5):
        _fill(rng, Xh, dh)
        dust.dust_estimate_gW_host(Xh, Xd, dh, dd, sh, sd, gh, gd, D_OUT, 9, 1, 0, 1e-3, 0.9,
                                   0.5, dust.CENTER)
        torch.cuda.synchronize()
        want = _direct(dust.dust_estimate_gW, Xh.to(dev), dh.to(dev), D_OUT, sh.to(dev), 9, 1,
                       0, 1e-3, 0.9, 0.5, dust.CENTER).cpu()
        assert torch.equal(gh, want), i
    assert dust.dust_last_error() == dust.OK

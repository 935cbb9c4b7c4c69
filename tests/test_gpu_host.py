"""The host-buffer entry point (dust_estimate_gW_host) against the device
entry point on the same inputs: X travels over an internal copy stream while
the scan and the weighting run, so the checks are that the result is the
device path's bit for bit, that back-to-back calls reusing the staging
buffers never see a half-copied X, and that accumulation and empty token
sets behave as on the device path."""
import numpy as np
import pytest

import token_perturbation_estimator_gb300 as dust
from helpers import cuda, offsets_from_lengths, random_lengths

pytestmark = pytest.mark.gpu


def _case(seed, T, d_in, d_out, K, bf16=True):
    import torch
    rng = np.random.default_rng(seed)
    so = offsets_from_lengths(random_lengths(rng, T, 600))
    X = torch.from_numpy(rng.standard_normal((T, d_in)).astype(np.float32))
    if bf16:
        X = X.to(torch.bfloat16)
    delta = torch.from_numpy((0.05 * rng.standard_normal((K, T))).astype(np.float32))
    return X, delta, torch.from_numpy(so)


def _host_call(X, delta, so, d_out, flags, gW_host=None, stage=None, stream=None):
    import torch
    dev = cuda()
    if stage is None:
        stage = (torch.empty_like(X, device=dev), torch.empty_like(delta, device=dev),
                 torch.empty_like(so, device=dev),
                 torch.empty((d_out, X.shape[1]), dtype=torch.float32, device=dev))
    if gW_host is None:
        gW_host = torch.empty((d_out, X.shape[1]), dtype=torch.float32).pin_memory()
    dust.dust_estimate_gW_host(X, stage[0], delta, stage[1], so, stage[2], gW_host, stage[3],
                               d_out, 21, 1, 0, 1e-3, 0.9, 0.5, flags, stream=stream)
    return gW_host, stage


@pytest.mark.parametrize("bf16", [True, False])
def test_host_path_matches_device_path(bf16):
    import torch
    dev = cuda()
    T, d_in, d_out, K = 6000, 256, 512, 8
    X, delta, so = _case(1, T, d_in, d_out, K, bf16)
    want = dust.dust_estimate_gW(X.to(dev), delta.to(dev), d_out, so.to(dev), 21, 1, 0, 1e-3,
                                 0.9, 0.5, dust.CENTER).cpu()
    got, _ = _host_call(X.pin_memory(), delta.pin_memory(), so.pin_memory(), d_out, dust.CENTER)
    torch.cuda.synchronize()
    assert dust.dust_last_error() == dust.OK
    assert torch.equal(got, want)


def test_host_path_back_to_back_reuses_staging():
    """Alternating inputs through one set of staging buffers on a user stream:
    each call's X copy starts only after the previous call's contraction has
    read the staged X, and each result is complete when the stream is."""
    import torch
    dev = cuda()
    T, d_in, d_out, K = 16384, 512, 2048, 8
    cases = [_case(s, T, d_in, d_out, K) for s in (2, 3)]
    wants = [dust.dust_estimate_gW(X.to(dev), d.to(dev), d_out, so.to(dev), 21, 1, 0, 1e-3, 0.9,
                                   0.5, dust.CENTER).cpu() for X, d, so in cases]
    pinned = [(X.pin_memory(), d.pin_memory(), so.pin_memory()) for X, d, so in cases]
    st = torch.cuda.Stream()
    stage = None
    outs = []
    for i in range(6):
        X, d, so = pinned[i % 2]
        out = torch.empty((d_out, d_in), dtype=torch.float32).pin_memory()
        out, stage = _host_call(X, d, so, d_out, dust.CENTER, gW_host=out, stage=stage, stream=st)
        outs.append(out)
    st.synchronize()
    assert dust.dust_last_error() == dust.OK
    for i, out in enumerate(outs):
        assert torch.equal(out, wants[i % 2]), i


def test_host_path_accumulate_and_empty():
    import torch
    dev = cuda()
    T, d_in, d_out, K = 4096, 128, 256, 4
    X, delta, so = _case(4, T, d_in, d_out, K)
    base = torch.randn((d_out, d_in))
    want = dust.dust_estimate_gW(X.to(dev), delta.to(dev), d_out, so.to(dev), 21, 1, 0, 1e-3,
                                 0.9, 0.5, dust.CENTER | dust.ACCUMULATE,
                                 gW=base.clone().to(dev)).cpu()
    acc = base.clone().pin_memory()
    got, _ = _host_call(X.pin_memory(), delta.pin_memory(), so.pin_memory(), d_out,
                        dust.CENTER | dust.ACCUMULATE, gW_host=acc)
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    # no tokens: GW is zeroed (or left as it was when accumulating)
    Xe = torch.empty((0, d_in), dtype=torch.bfloat16).pin_memory()
    de = torch.empty((K, 0), dtype=torch.float32).pin_memory()
    se = torch.zeros(1, dtype=torch.int32).pin_memory()
    z = torch.full((d_out, d_in), 7.0).pin_memory()
    got, _ = _host_call(Xe, de, se, d_out, dust.CENTER, gW_host=z)
    torch.cuda.synchronize()
    assert torch.count_nonzero(got).item() == 0


def _site(X, delta, so, d_out, seed, gamma, dev, pinned_gw=True):
    import torch
    T, d_in = X.shape
    K = delta.shape[0]
    ws = torch.empty(max(256, dust.dust_estimate_gW_workspace(T, d_in, d_out, K,
                                                              dust.BF16, dust.CENTER)),
                     dtype=torch.uint8, device=dev)
    gh = torch.full((d_out, d_in), float("nan"))
    return {"X_host": X.pin_memory(), "X_dev": torch.empty_like(X, device=dev),
            "delta_host": delta.pin_memory(), "delta_dev": torch.empty_like(delta, device=dev),
            "seq_host": so.pin_memory(), "seq_dev": torch.empty_like(so, device=dev),
            "gW_host": gh.pin_memory() if pinned_gw else gh,
            "gW_dev": torch.empty((d_out, d_in), dtype=torch.float32, device=dev),
            "workspace": ws, "seed": seed, "sigma": 1e-3, "gamma": gamma}


@pytest.mark.parametrize("pinned_gw", [True, False])
def test_host_sites_match_device_calls(pinned_gw):
    """Three layers of different shapes, decays and seeds in one pass, twice
    in a row on a user stream: each result equals the device entry point's
    for that site, bit for bit (mapped or copied-back ĜW)."""
    import torch
    dev = cuda()
    shapes = [(4096, 512, 1536, 32, 0.9), (4096, 512, 512, 32, 0.0), (2048, 256, 1024, 8, 0.0)]
    cases, wants = [], []
    for i, (T, d_in, d_out, K, gamma) in enumerate(shapes):
        X, delta, so = _case(10 + i, T, d_in, d_out, K)
        cases.append((X, delta, so, d_out, 100 + i, gamma))
        wants.append(dust.dust_estimate_gW(X.to(dev), delta.to(dev), d_out, so.to(dev), 100 + i,
                                           dust.GAUSSIAN, 0, 1e-3, gamma, 1.0,
                                           dust.CENTER).cpu())
    sites = [_site(*c, dev, pinned_gw) for c in cases]
    st = torch.cuda.Stream()
    for rep in range(2):
        for q in sites:
            q["gW_host"].fill_(float("nan"))
        dust.dust_estimate_gW_host_sites(sites, dust.GAUSSIAN, 0, 1.0, dust.CENTER, stream=st)
        st.synchronize()
        assert dust.dust_last_error() == dust.OK
        for i, (q, want) in enumerate(zip(sites, wants)):
            assert torch.equal(q["gW_host"], want), (rep, i)


def test_host_sites_reject_overlapping_staging():
    import torch
    dev = cuda()
    X, delta, so = _case(20, 1024, 256, 512, 8)
    a = _site(X, delta, so, 512, 1, 0.0, dev)
    b = _site(X, delta, so, 512, 2, 0.0, dev)
    b["X_dev"] = a["workspace"][: X.numel() * 2].view(torch.bfloat16).view(X.shape)
    with pytest.raises(dust.DustError) as e:
        dust.dust_estimate_gW_host_sites([a, b], dust.GAUSSIAN, 0)
    assert e.value.status == dust.ERR_INVALID_ARG


def test_host_sites_accumulate_and_empty_site():
    """Accumulating into existing host gradients (each site's GW_host is read
    before and written after), with an empty site (no tokens) in the middle,
    which leaves its accumulated gradient unchanged."""
    import torch
    dev = cuda()
    shapes = [(2048, 256, 512, 8, 0.9), (0, 256, 512, 8, 0.0), (3000, 128, 1024, 16, 0.0)]
    sites, wants = [], []
    for i, (T, d_in, d_out, K, gamma) in enumerate(shapes):
        if T:
            X, delta, so = _case(30 + i, T, d_in, d_out, K)
        else:
            X = torch.empty((0, d_in), dtype=torch.bfloat16)
            delta = torch.empty((K, 0), dtype=torch.float32)
            so = torch.zeros(1, dtype=torch.int32)
        base = torch.randn((d_out, d_in))
        if T:
            wants.append(dust.dust_estimate_gW(X.to(dev), delta.to(dev), d_out, so.to(dev),
                                               200 + i, dust.GAUSSIAN, 0, 1e-3, gamma, 1.0,
                                               dust.CENTER | dust.ACCUMULATE,
                                               gW=base.clone().to(dev)).cpu())
        else:
            wants.append(base.clone())
        q = _site(X, delta, so, d_out, 200 + i, gamma, dev)
        q["gW_host"].copy_(base)
        sites.append(q)
    dust.dust_estimate_gW_host_sites(sites, dust.GAUSSIAN, 0, 1.0,
                                     dust.CENTER | dust.ACCUMULATE)
    torch.cuda.synchronize()
    assert dust.dust_last_error() == dust.OK
    for i, (q, want) in enumerate(zip(sites, wants)):
        assert torch.equal(q["gW_host"], want), i

"""The multi-site device entry point (dust_estimate_gW_sites) against the
single-site one on the same inputs. Sites run on the library's compute lanes,
so the checks are that every result is the single-site call's bit for bit
(direct launches, the captured graph and its replays), that the lanes start
after the caller's earlier work and the caller's later work sees every
result, that sites may share read-only inputs but not what they write, and
that accumulation and empty sites behave as on the single-site path."""
import numpy as np
import pytest

import token_perturbation_estimator_gb300 as dust
from helpers import cuda, offsets_from_lengths, random_lengths

pytestmark = pytest.mark.gpu

# (T, d_in, d_out, K, gamma): scan and no-scan sites, both tile shapes of the
# contraction, narrow and wide weighting lanes, more sites than lanes
SHAPES = [(4096, 512, 1536, 32, 0.9), (4096, 512, 512, 32, 0.0), (4096, 512, 2048, 32, 0.0),
          (4096, 2048, 512, 32, 0.0), (3000, 256, 1024, 16, 0.5), (2048, 128, 256, 8, 0.0),
          (1000, 64, 192, 4, 0.0)]


def _inputs(seed, T, d_in, K, dev):
    import torch
    rng = np.random.default_rng(seed)
    X = torch.from_numpy(rng.standard_normal((T, d_in)).astype(np.float32))
    delta = torch.from_numpy((0.05 * rng.standard_normal((K, T))).astype(np.float32))
    so = torch.from_numpy(offsets_from_lengths(random_lengths(rng, T, 600)))
    return X.to(torch.bfloat16).to(dev), delta.to(dev), so.to(dev)


def _site(X, delta, so, d_out, seed, gamma, dev, sigma=1e-3):
    import torch
    T, d_in = X.shape
    K = delta.shape[0]
    ws = torch.empty(max(256, dust.dust_estimate_gW_workspace(T, d_in, d_out, K, dust.BF16,
                                                              dust.CENTER)),
                     dtype=torch.uint8, device=dev)
    return {"X": X, "delta": delta, "seq_offsets": so, "seed": seed, "sigma": sigma,
            "gamma": gamma, "workspace": ws,
            "gW": torch.full((d_out, d_in), float("nan"), device=dev)}


def _single(q, flags=dust.CENTER, gW=None):
    return dust.dust_estimate_gW(q["X"], q["delta"], q["gW"].shape[0], q["seq_offsets"],
                                 q["seed"], dust.GAUSSIAN, 0, q["sigma"], q["gamma"], 1.0, flags,
                                 gW=gW)


def _sites(dev):
    sites = []
    for i, (T, d_in, d_out, K, gamma) in enumerate(SHAPES):
        X, delta, so = _inputs(40 + i, T, d_in, K, dev)
        sites.append(_site(X, delta, so, d_out, 300 + i, gamma, dev))
    return sites


def test_sites_match_single_site_calls():
    """Seven sites of mixed shapes on a user stream, four calls in a row
    (direct launches, then the graph's capture, then two replays): every
    result equals dust_estimate_gW's for that site, bit for bit."""
    import torch
    dev = cuda()
    sites = _sites(dev)
    wants = [_single(q).cpu() for q in sites]
    st = torch.cuda.Stream()
    arr = dust.SiteArray(sites)
    for rep in range(4):
        for q in sites:
            q["gW"].fill_(float("nan"))
        torch.cuda.synchronize()  # the fills ran on the default stream
        dust.dust_estimate_gW_sites(arr, dust.GAUSSIAN, 0, 1.0, dust.CENTER, stream=st)
        st.synchronize()
        assert dust.dust_last_error() == dust.OK
        for i, (q, want) in enumerate(zip(sites, wants)):
            assert torch.equal(q["gW"].cpu(), want), (rep, i)


def test_sites_order_with_the_callers_stream():
    """The lanes start after what the stream already holds (here: the copy of
    every site's loss changes into place) and the stream's next work (a
    clone of every result) sees every site's result."""
    import torch
    dev = cuda()
    sites = _sites(dev)
    wants = [_single(q).cpu() for q in sites]
    real = [q["delta"].clone() for q in sites]
    st = torch.cuda.Stream()
    for rep in range(3):
        for q in sites:
            q["delta"].zero_()
            q["gW"].fill_(float("nan"))
        torch.cuda.synchronize()
        # a long-running fill just before the call, then the real loss changes
        with torch.cuda.stream(st):
            big = torch.empty(1 << 28, device=dev)
            big.fill_(1.0)
            for q, d in zip(sites, real):
                q["delta"].copy_(d)
            dust.dust_estimate_gW_sites(sites, dust.GAUSSIAN, 0, 1.0, dust.CENTER, stream=st)
            outs = [q["gW"].clone() for q in sites]
        st.synchronize()
        for i, (o, want) in enumerate(zip(outs, wants)):
            assert torch.equal(o.cpu(), want), (rep, i)


def test_sites_share_inputs_not_results():
    """Several sites reading one X, one delta and one offset array (Dust's
    loss changes are shared by every layer) are accepted and exact; two sites
    writing one workspace, or one site's result over another's input, are
    rejected before anything runs."""
    import torch
    dev = cuda()
    X, delta, so = _inputs(60, 4096, 512, 32, dev)
    sites = [_site(X, delta, so, d_out, 500 + i, g, dev)
             for i, (d_out, g) in enumerate([(1536, 0.9), (512, 0.0), (2048, 0.0), (512, 0.5)])]
    wants = [_single(q).cpu() for q in sites]
    dust.dust_estimate_gW_sites(sites, dust.GAUSSIAN, 0, 1.0, dust.CENTER)
    torch.cuda.synchronize()
    for i, (q, want) in enumerate(zip(sites, wants)):
        assert torch.equal(q["gW"].cpu(), want), i
    bad = [dict(q) for q in sites]
    bad[3]["workspace"] = bad[1]["workspace"]
    with pytest.raises(dust.DustError) as e:
        dust.dust_estimate_gW_sites(bad, dust.GAUSSIAN, 0, 1.0, dust.CENTER)
    assert e.value.status == dust.ERR_INVALID_ARG
    bad = [dict(q) for q in sites]
    bad[2]["gW"] = X.view(torch.float32).view(2048, 512)  # over the X every site reads
    with pytest.raises(dust.DustError) as e:
        dust.dust_estimate_gW_sites(bad, dust.GAUSSIAN, 0, 1.0, dust.CENTER)
    assert e.value.status == dust.ERR_INVALID_ARG


def test_sites_accumulate_and_empty_sites():
    """Accumulating into existing gradients, with a site of no tokens (its
    gradient left as it was) and a site with no outputs in the middle."""
    import torch
    dev = cuda()
    shapes = [(2048, 256, 512, 8, 0.9), (0, 256, 512, 8, 0.0), (1024, 128, 0, 8, 0.0),
              (3000, 128, 1024, 16, 0.0), (1500, 256, 768, 8, 0.0)]
    sites, wants = [], []
    for i, (T, d_in, d_out, K, gamma) in enumerate(shapes):
        if T:
            X, delta, so = _inputs(70 + i, T, d_in, K, dev)
        else:
            X = torch.empty((0, d_in), dtype=torch.bfloat16, device=dev)
            delta = torch.empty((K, 0), device=dev)
            so = torch.zeros(1, dtype=torch.int32, device=dev)
        q = _site(X, delta, so, d_out, 700 + i, gamma, dev)
        base = torch.randn((d_out, d_in), device=dev)
        q["gW"].copy_(base)
        if T and d_out:
            wants.append(_single(q, dust.CENTER | dust.ACCUMULATE, gW=base.clone()).cpu())
        else:
            wants.append(base.cpu())
        sites.append(q)
    dust.dust_estimate_gW_sites(sites, dust.GAUSSIAN, 0, 1.0, dust.CENTER | dust.ACCUMULATE)
    torch.cuda.synchronize()
    assert dust.dust_last_error() == dust.OK
    for i, (q, want) in enumerate(zip(sites, wants)):
        assert torch.equal(q["gW"].cpu(), want), i


def test_sites_graph_replay_reads_current_inputs():
    """A replayed call (same arguments) computes from the buffers' contents at
    launch time: new X and loss changes written in place give the single-site
    results for those new values."""
    import torch
    dev = cuda()
    sites = _sites(dev)[:4]
    arr = dust.SiteArray(sites)
    for _ in range(3):  # direct, capture, replay
        dust.dust_estimate_gW_sites(arr, dust.GAUSSIAN, 0, 1.0, dust.CENTER)
    torch.cuda.synchronize()
    for i, q in enumerate(sites):
        X, delta, _ = _inputs(90 + i, q["X"].shape[0], q["X"].shape[1], q["delta"].shape[0], dev)
        q["X"].copy_(X)
        q["delta"].copy_(delta)
    wants = [_single(q).cpu() for q in sites]
    dust.dust_estimate_gW_sites(arr, dust.GAUSSIAN, 0, 1.0, dust.CENTER)
    torch.cuda.synchronize()
    for i, (q, want) in enumerate(zip(sites, wants)):
        assert torch.equal(q["gW"].cpu(), want), i


@pytest.mark.parametrize("kind", [dust.RADEMACHER, dust.RADEMACHER_PACKED, dust.GAUSSIAN])
def test_sites_other_noises_antithetic_and_offset(kind):
    """Sign noises and Gaussians with antithetic pairs and a later draw range
    (draw_begin 6) and a scale: each site equals dust_estimate_gW's result."""
    import torch
    dev = cuda()
    shapes = [(4096, 512, 1024, 16, 0.9), (4096, 256, 512, 16, 0.0), (2048, 512, 2048, 8, 0.0),
              (3000, 128, 1024, 16, 0.5)]
    sites, wants = [], []
    flags = dust.CENTER | dust.ANTITHETIC
    for i, (T, d_in, d_out, K, gamma) in enumerate(shapes):
        X, delta, so = _inputs(110 + i, T, d_in, K, dev)
        q = _site(X, delta, so, d_out, 900 + i, gamma, dev)
        wants.append(dust.dust_estimate_gW(X, delta, d_out, so, q["seed"], kind, 6, q["sigma"],
                                           gamma, 0.25, flags).cpu())
        sites.append(q)
    dust.dust_estimate_gW_sites(sites, kind, 6, 0.25, flags)
    torch.cuda.synchronize()
    assert dust.dust_last_error() == dust.OK
    for i, (q, want) in enumerate(zip(sites, wants)):
        assert torch.equal(q["gW"].cpu(), want), i


def test_sites_fp32_inputs():
    """fp32 X (the CUDA-core contraction, which stays on the lanes): each site
    equals dust_estimate_gW's result."""
    import torch
    dev = cuda()
    shapes = [(2048, 256, 512, 8, 0.9), (1500, 192, 320, 8, 0.0), (1024, 128, 256, 4, 0.0)]
    sites, wants = [], []
    for i, (T, d_in, d_out, K, gamma) in enumerate(shapes):
        X, delta, so = _inputs(130 + i, T, d_in, K, dev)
        X = X.float()
        ws = torch.empty(max(256, dust.dust_estimate_gW_workspace(T, d_in, d_out, K, dust.F32,
                                                                  dust.CENTER)),
                         dtype=torch.uint8, device=dev)
        q = {"X": X, "delta": delta, "seq_offsets": so, "seed": 950 + i, "sigma": 1e-3,
             "gamma": gamma, "workspace": ws, "gW": torch.empty((d_out, d_in), device=dev)}
        wants.append(_single(q).cpu())
        sites.append(q)
    dust.dust_estimate_gW_sites(sites, dust.GAUSSIAN, 0, 1.0, dust.CENTER)
    torch.cuda.synchronize()
    for i, (q, want) in enumerate(zip(sites, wants)):
        assert torch.equal(q["gW"].cpu(), want), i


@pytest.mark.slow
def test_sweep_full_size_through_the_sites_call():
    """The headline configuration in the launch configuration the benchmark
    times: the sweep's 48 sites at full size (65,536 tokens, K = 32, inputs
    built as the benchmark builds them) in one dust_estimate_gW_sites call,
    the third call of the same arguments (a graph replay). Every site equals
    its single-site call bit for bit, and one layer's four sites match the
    oracle on 16 sampled ĜW entries each (bf16 inputs: 1e-2 relative)."""
    import torch
    import bench
    import oracle
    import workloads as wl
    from helpers import rel_fro
    dev = cuda()
    sites = wl.sweep_sites()
    qs = []
    for i, w in enumerate(sites):
        X, delta, so = bench.make_inputs_fast(w, dev, i)
        ws = torch.empty(dust.dust_estimate_gW_workspace(w.T, w.d_in, w.d_out, w.K, dust.BF16,
                                                         dust.CENTER),
                         dtype=torch.uint8, device=dev)
        qs.append({"X": X, "delta": delta, "seq_offsets": so, "seed": w.seed, "sigma": w.sigma,
                   "gamma": w.gamma, "workspace": ws,
                   "gW": torch.empty((w.d_out, w.d_in), device=dev)})
    arr = dust.SiteArray(qs)
    for _ in range(3):  # direct launches, capture, replay
        for q in qs:
            q["gW"].fill_(float("nan"))
        torch.cuda.synchronize()
        dust.dust_estimate_gW_sites(arr, dust.GAUSSIAN, 0, 1.0, dust.CENTER)
    torch.cuda.synchronize()
    assert dust.dust_last_error() == dust.OK
    got = [q["gW"].clone() for q in qs]
    for i, (w, q) in enumerate(zip(sites, qs)):
        want = dust.dust_estimate_gW(q["X"], q["delta"], w.d_out, q["seq_offsets"], w.seed,
                                     w.kind, 0, w.sigma, w.gamma, 1.0, dust.CENTER,
                                     workspace=q["workspace"])
        assert torch.equal(got[i], want), i
    rng = np.random.default_rng(12)
    for i in range(20, 24):  # layer 5: QKV, O, up, down
        w, q = sites[i], qs[i]
        X = q["X"].float().cpu().numpy()
        delta = q["delta"].cpu().numpy()
        so = q["seq_offsets"].cpu().numpy()
        chan = rng.integers(0, w.d_out, 16)
        col = rng.integers(0, w.d_in, 16)
        r = oracle.credit(delta, so, np.float32(w.gamma), oracle.CENTER)
        want = oracle.gW_entries(X, r, w.d_out, chan, col, w.seed, w.kind, 0,
                                 np.float32(w.sigma), 1.0, oracle.CENTER)
        g = got[i].double().cpu().numpy()
        assert np.all(np.isfinite(g))
        assert rel_fro(g[chan, col], want) <= 1e-2, i


def test_many_mixed_sites():
    """37 sites of mixed sizes (more than ten per lane), some with d_in or
    d_out not a multiple of 8 (the CUDA-core contraction, which stays on the
    lane), some with γ ≠ 0: every result equals its single-site call."""
    import torch
    dev = cuda()
    rng = np.random.default_rng(77)
    sites, wants = [], []
    for i in range(37):
        T = int(rng.integers(200, 1500))
        d_in = int(rng.choice([64, 128, 60, 256]))
        d_out = int(rng.choice([128, 256, 72, 100]))
        K = int(rng.choice([4, 8, 16]))
        gamma = float(rng.choice([0.0, 0.0, 0.9]))
        X, delta, so = _inputs(200 + i, T, d_in, K, dev)
        q = _site(X, delta, so, d_out, 1200 + i, gamma, dev)
        wants.append(_single(q).cpu())
        sites.append(q)
    for _ in range(2):
        for q in sites:
            q["gW"].fill_(float("nan"))
        torch.cuda.synchronize()
        dust.dust_estimate_gW_sites(sites, dust.GAUSSIAN, 0, 1.0, dust.CENTER)
        torch.cuda.synchronize()
        assert dust.dust_last_error() == dust.OK
        for i, (q, want) in enumerate(zip(sites, wants)):
            assert torch.equal(q["gW"].cpu(), want), i


def test_sites_from_two_host_threads():
    """Two host threads each calling dust_estimate_gW_sites on their own
    stream and buffers, several times: the calls share the library's lanes
    (their enqueues are serialised on the host) and every result equals its
    single-site call."""
    import threading
    import torch
    dev = cuda()
    groups, wants = [], []
    for gi in range(2):
        sites = []
        for i, (T, d_in, d_out, K, gamma) in enumerate(SHAPES[:4]):
            X, delta, so = _inputs(300 + 10 * gi + i, T, d_in, K, dev)
            sites.append(_site(X, delta, so, d_out, 1500 + 10 * gi + i, gamma, dev))
        wants.append([_single(q).cpu() for q in sites])
        groups.append(sites)
    torch.cuda.synchronize()
    errors = []

    def run(gi):
        try:
            st = torch.cuda.Stream()
            arr = dust.SiteArray(groups[gi])
            for _ in range(5):
                dust.dust_estimate_gW_sites(arr, dust.GAUSSIAN, 0, 1.0, dust.CENTER, stream=st)
            st.synchronize()
        except Exception as e:  # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(gi,)) for gi in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert dust.dust_last_error() == dust.OK
    for gi in range(2):
        for i, (q, want) in enumerate(zip(groups[gi], wants[gi])):
            assert torch.equal(q["gW"].cpu(), want), (gi, i)


@pytest.mark.parametrize("flags", [dust.CENTER, dust.CENTER | dust.ACCUMULATE])
def test_sites_wide_tiles_in_cluster(flags):
    """Sites whose contraction takes 256-channel tiles and reduces its token
    slices inside a cluster (16,384 tokens, 1024 -> 2048: 32 tiles, 4 slices of
    4096 tokens), next to one with 128-channel tiles, in the 32-register build
    of the lanes: each equals dust_estimate_gW's result (which takes the
    192-thread build), overwritten or accumulated."""
    import torch
    dev = cuda()
    shapes = [(16384, 1024, 2048, 8, 0.0), (16384, 1024, 2048, 8, 0.9), (16384, 512, 2048, 8, 0.0)]
    sites, wants = [], []
    for i, (T, d_in, d_out, K, gamma) in enumerate(shapes):
        X, delta, so = _inputs(160 + i, T, d_in, K, dev)
        q = _site(X, delta, so, d_out, 1700 + i, gamma, dev)
        base = torch.randn((d_out, d_in), device=dev)
        q["gW"].copy_(base)
        wants.append(_single(q, flags, gW=base.clone()).cpu())
        sites.append(q)
    torch.cuda.synchronize()
    dust.dust_estimate_gW_sites(sites, dust.GAUSSIAN, 0, 1.0, flags)
    torch.cuda.synchronize()
    assert dust.dust_last_error() == dust.OK
    for i, (q, want) in enumerate(zip(sites, wants)):
        assert torch.equal(q["gW"].cpu(), want), i

"""GPU parity of the reward weighting and of the whole estimator (through the
C ABI) against the fp64 oracle.

Tolerances: g within 1e-5 normwise relative (fp32 output); GW within 1e-5
relative Frobenius on the fp32 path and 1e-2 with bf16 X (g rounded to bf16
before the contraction on the tensor-core paths).
"""
import numpy as np
import pytest

import oracle
import token_perturbation_estimator_gb300 as dust
import workloads as wl
from helpers import bf16_round, cuda, offsets_from_lengths, random_lengths, rel_fro

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------ weighting --

W_CASES = [
    # K, T, d_out, kind, draw_begin, flags
    (1, 1, 1, 0, 0, 0),
    (4, 9, 7, 1, 0, 0),
    (8, 100, 256, 1, 8, dust.ANTITHETIC),
    (3, 257, 300, 0, 5, 0),
    (64, 64, 1000, 0, 0, 0),
    (65, 31, 513, 1, 123, 0),
    (16, 200, 2048, 1, 0, 0),
    (66, 77, 1024, 1, 4, dust.ANTITHETIC),  # two draw groups, ragged T
    (8, 77, 1024, 1, 4, 0),                 # 32 channels per lane (d_out % 1024 == 0)
    (16, 45, 2048, 1, 2, dust.ANTITHETIC),  # the same with 8 antithetic pairs
    (64, 50, 1024, 1, 3, 0),                # wide lanes, one whole group of 64 draws
    (128, 33, 1024, 1, 2, dust.ANTITHETIC),  # wide lanes, 64 base draws
    (100, 40, 1024, 1, 0, 0),               # more than 64 noise draws: narrow lanes
    (130, 17, 64, 0, 2, dust.ANTITHETIC),
    # packed signs: one 32-sign word per lane, 1024 channels per CTA
    (8, 100, 77, 3, 0, 0),            # a 13-channel last word
    (65, 33, 1000, 3, 5, 0),          # two draw groups, a ragged CTA
    (16, 64, 2048, 3, 2, dust.ANTITHETIC),
    (3, 5, 31, 3, 1, 0),              # narrower than one word
]


@pytest.mark.parametrize("K,T,d_out,kind,draw_begin,flags", W_CASES)
def test_error_estimate_parity(K, T, d_out, kind, draw_begin, flags):
    import torch
    dev = cuda()
    rng = np.random.default_rng(K + T + d_out)
    r = rng.standard_normal((T, K)).astype(np.float32)
    sigma = 1e-3
    g = dust.dust_error_estimate(torch.from_numpy(r).to(dev), d_out, 77, kind, draw_begin,
                                 sigma, flags)
    want = oracle.error_estimate(r.T, d_out, 77, kind, draw_begin, np.float32(sigma), flags)
    got = g.cpu().numpy()
    assert rel_fro(got, want) <= 1e-5
    gb = dust.dust_error_estimate(torch.from_numpy(r).to(dev), d_out, 77, kind, draw_begin,
                                  sigma, flags, g_dtype=torch.bfloat16)
    assert torch.equal(gb, g.to(torch.bfloat16))


# -------------------------------------------------------- whole estimator --

def _run(w, X, delta, so, flags, gamma=None, scale=1.0, draw_begin=0):
    import torch
    dev = cuda()
    Xd = torch.from_numpy(X).to(dev)
    if w.x_dtype == "bf16":
        Xd = Xd.to(torch.bfloat16)
    return dust.dust_estimate_gW(Xd, torch.from_numpy(delta).to(dev), w.d_out,
                                 torch.from_numpy(so).to(dev), w.seed, w.kind, draw_begin,
                                 w.sigma, w.gamma if gamma is None else gamma, scale, flags)


def _inputs(w, planted=True):
    so = wl.seq_offsets(w)
    X = wl.make_X(w)
    if w.x_dtype == "bf16":
        X = wl.to_bf16_exact(X)
    if planted:
        delta = oracle.planted_delta(wl.make_dplant(w), w.seed, w.kind, 0, w.K,
                                     np.float32(w.sigma), w.curvature,
                                     wl.make_eps(w)).astype(np.float32)
    else:
        delta = wl.marginal_delta(w)
    return X, delta, so


SMALL = [
    wl.TOY,
    wl.MLP_UP.scaled(n_seq=3, seq_len=100, d_in=72, d_out=136),
    wl.QKV_DECAY.scaled(n_seq=2, seq_len=300, d_in=64, d_out=192),
    wl.SQUARE_R.scaled(n_seq=4, seq_len=64, d_in=128, d_out=128, K=16),
    wl.SQUARE_G.scaled(n_seq=4, seq_len=64, d_in=120, d_out=40, K=16),
    wl.SQUARE_RP.scaled(n_seq=4, seq_len=64, d_in=128, d_out=200, K=16),
]

FORCE = [0, dust.FORCE_SIMT, dust.FORCE_UNFUSED, dust.FORCE_FUSED]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("force", FORCE)
def test_estimate_gW_small(w, force):
    X, delta, so = _inputs(w)
    flags = dust.CENTER | force
    xd = dust.BF16 if w.x_dtype == "bf16" else dust.F32
    try:
        path = dust.dust_estimate_gW_path(w.T, w.d_in, w.d_out, w.K, xd, flags)
    except dust.DustError as e:
        assert e.status == dust.ERR_UNSUPPORTED
        return
    if w.kind == dust.RADEMACHER_PACKED and force == dust.FORCE_FUSED:
        with pytest.raises(dust.DustError) as e:  # the fused kernel has no packed signs
            _run(w, X, delta, so, flags)
        assert e.value.status == dust.ERR_UNSUPPORTED
        return
    got = _run(w, X, delta, so, flags).double().cpu().numpy()
    want = oracle.estimate_gW(X, delta, w.d_out, so, w.seed, w.kind, 0, np.float32(w.sigma),
                              np.float32(w.gamma), 1.0, oracle.CENTER)
    tol = 1e-5 if w.x_dtype == "f32" else 1e-2
    assert rel_fro(got, want) <= tol, (path, rel_fro(got, want))


@pytest.mark.parametrize("T,K,max_len", [(70000, 2, 9000), (900, 260, 300)])
def test_estimate_gW_long_token_set_and_many_draws(T, K, max_len):
    """Many scan chunks (70,000 tokens) and many draws (260, past one
    weighting draw group): the chunk carries the weighting kernel folds in
    and the draw grouping both reach the oracle's estimate."""
    import torch
    dev = cuda()
    rng = np.random.default_rng(T + K)
    so = offsets_from_lengths(random_lengths(rng, T, max_len))
    d_in, d_out = 16, 24
    X = bf16_round(rng.standard_normal((T, d_in))).astype(np.float32)
    delta = (0.05 * rng.standard_normal((K, T))).astype(np.float32)
    got = dust.dust_estimate_gW(torch.from_numpy(X).to(dev).to(torch.bfloat16),
                                torch.from_numpy(delta).to(dev), d_out,
                                torch.from_numpy(so).to(dev), 13, 1, 0, 1e-3, 0.95, 1.0,
                                dust.CENTER).double().cpu().numpy()
    want = oracle.estimate_gW(X, delta, d_out, so, 13, 1, 0, np.float32(1e-3),
                              np.float32(0.95), 1.0, oracle.CENTER)
    assert rel_fro(got, want) <= 1e-2


def test_estimate_matches_brute_force_tiny():
    import torch
    dev = cuda()
    rng = np.random.default_rng(8)
    lengths = [5, 1, 9, 3]
    so = offsets_from_lengths(lengths)
    T, d_in, d_out, K = int(so[-1]), 6, 10, 4
    X = rng.standard_normal((T, d_in)).astype(np.float32)
    delta = rng.standard_normal((K, T)).astype(np.float32)
    for kind in (0, 1):
        got = dust.dust_estimate_gW(torch.from_numpy(X).to(dev), torch.from_numpy(delta).to(dev),
                                    d_out, torch.from_numpy(so).to(dev), 3, kind, 2, 0.01, 0.6,
                                    0.5, dust.CENTER).double().cpu().numpy()
        want = oracle.bruteforce_gW(X, delta, d_out, so, 3, kind, 2, np.float32(0.01),
                                    np.float32(0.6), 0.5, oracle.CENTER)
        assert rel_fro(got, want) <= 1e-5


def test_deterministic_and_accumulate():
    import torch
    dev = cuda()
    w = wl.MLP_UP.scaled(n_seq=4, seq_len=256, d_in=128, d_out=256)
    X, delta, so = _inputs(w, planted=False)
    a = _run(w, X, delta, so, dust.CENTER)
    b = _run(w, X, delta, so, dust.CENTER)
    assert torch.equal(a, b)
    base = torch.randn_like(a)
    acc = base.clone()
    Xd = torch.from_numpy(X).to(dev).to(torch.bfloat16)
    dust.dust_estimate_gW(Xd, torch.from_numpy(delta).to(dev), w.d_out,
                          torch.from_numpy(so).to(dev), w.seed, w.kind, 0, w.sigma, w.gamma,
                          1.0, dust.CENTER | dust.ACCUMULATE, gW=acc)
    assert torch.allclose(acc, base + a, rtol=1e-6, atol=1e-6 * a.abs().max().item())


def test_empty_token_set():
    import torch
    dev = cuda()
    X = torch.empty((0, 16), dtype=torch.bfloat16, device=dev)
    delta = torch.empty((4, 0), dtype=torch.float32, device=dev)
    so = torch.zeros(1, dtype=torch.int32, device=dev)
    gW = torch.full((8, 16), 3.0, device=dev)
    dust.dust_estimate_gW(X, delta, 8, so, 0, 1, 0, 1e-3, 0.0, 1.0, dust.CENTER, gW=gW)
    assert torch.count_nonzero(gW).item() == 0
    gW.fill_(3.0)
    dust.dust_estimate_gW(X, delta, 8, so, 0, 1, 0, 1e-3, 0.0, 1.0,
                          dust.CENTER | dust.ACCUMULATE, gW=gW)
    assert torch.all(gW == 3.0)


@pytest.mark.parametrize("gamma", [0.0, 0.9])
def test_antithetic_cancels_curvature_on_gpu(gamma):
    """GPU version of the even-order cancellation: with antithetic pairs the
    curvature term of the planted loss leaves GW unchanged (to rounding)."""
    import torch
    dev = cuda()
    rng = np.random.default_rng(21)
    T, d_in, d_out, K, sigma = 512, 32, 48, 8, 0.05
    so = offsets_from_lengths([200, 312])
    dp = rng.standard_normal((T, d_out))
    X = rng.standard_normal((T, d_in)).astype(np.float32)
    f = oracle.ANTITHETIC
    lin = oracle.planted_delta(dp, 4, 1, 0, K, sigma, curv=0.0, flags=f).astype(np.float32)
    quad = oracle.planted_delta(dp, 4, 1, 0, K, sigma, curv=1.0, flags=f).astype(np.float32)
    outs = []
    for d in (lin, quad):
        outs.append(dust.dust_estimate_gW(torch.from_numpy(X).to(dev), torch.from_numpy(d).to(dev),
                                          d_out, torch.from_numpy(so).to(dev), 4, 1, 0, sigma,
                                          gamma, 1.0, dust.CENTER | dust.ANTITHETIC)
                    .double().cpu().numpy())
    assert rel_fro(outs[1], outs[0]) <= 1e-4


def test_sequence_sharding_sums_to_whole():
    """Token sharding by whole sequences (the multi-GPU split): the scan never
    crosses a sequence and the hash uses global token indices, so per-shard
    estimates over the shards' rows sum to the unsharded estimate. Emulated
    here on one GPU with zero-padded shards."""
    import torch
    dev = cuda()
    rng = np.random.default_rng(22)
    lengths = [100, 60, 150, 90]
    so = offsets_from_lengths(lengths)
    T, d_in, d_out, K = int(so[-1]), 24, 40, 6
    X = rng.standard_normal((T, d_in)).astype(np.float32)
    delta = rng.standard_normal((K, T)).astype(np.float32)
    full = dust.dust_estimate_gW(torch.from_numpy(X).to(dev), torch.from_numpy(delta).to(dev),
                                 d_out, torch.from_numpy(so).to(dev), 9, 1, 0, 0.01, 0.9, 1.0,
                                 dust.CENTER)
    acc = torch.zeros_like(full)
    for lo, hi in ((0, 2), (2, 4)):
        Xs = np.zeros_like(X)
        t0, t1 = so[lo], so[hi]
        Xs[t0:t1] = X[t0:t1]
        dust.dust_estimate_gW(torch.from_numpy(Xs).to(dev), torch.from_numpy(delta).to(dev),
                              d_out, torch.from_numpy(so).to(dev), 9, 1, 0, 0.01, 0.9, 1.0,
                              dust.CENTER | dust.ACCUMULATE, gW=acc)
    assert rel_fro(acc.cpu().numpy(), full.cpu().numpy()) <= 1e-6


def test_draw_sharding_sums_to_whole():
    """Sharding by draws: each shard takes a range of absolute draw indices
    (draw_begin); the loss changes are centred once over all K draws and
    passed without DUST_CENTER, and each shard's estimate is scaled by its
    share of the draws, so the shards accumulate to the unsharded centred
    estimate."""
    import torch
    dev = cuda()
    rng = np.random.default_rng(23)
    so = offsets_from_lengths([120, 80, 200])
    T, d_in, d_out, K = int(so[-1]), 24, 40, 12
    X = torch.from_numpy(rng.standard_normal((T, d_in)).astype(np.float32)).to(dev)
    delta = rng.standard_normal((K, T)).astype(np.float32)
    sod = torch.from_numpy(so).to(dev)
    full = dust.dust_estimate_gW(X, torch.from_numpy(delta).to(dev), d_out, sod, 4, 1, 0, 0.01,
                                 0.9, 1.0, dust.CENTER)
    centred = (delta - delta.mean(axis=0, keepdims=True)).astype(np.float32)
    acc = torch.zeros_like(full)
    for d0, d1 in ((0, 4), (4, 10), (10, 12)):
        dust.dust_estimate_gW(X, torch.from_numpy(np.ascontiguousarray(centred[d0:d1])).to(dev),
                              d_out, sod, 4, 1, d0, 0.01, 0.9, (d1 - d0) / K, dust.ACCUMULATE,
                              gW=acc)
    assert rel_fro(acc.cpu().numpy(), full.cpu().numpy()) <= 1e-5


# ----------------------------------------------- full sizes, sampled entries --

FULL = [wl.TOY, wl.MLP_UP, wl.QKV_DECAY, wl.SQUARE_R, wl.SQUARE_G]


@pytest.mark.slow
@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_estimate_gW_full_size_sampled(w):
    """The measured workloads at full size, in the default launch
    configuration: 64 sampled GW entries against the oracle, each computed
    one by one from the full column of g."""
    planted = w.element_draws <= 1_000_000_000
    X, delta, so = _inputs(w, planted=planted)
    got = _run(w, X, delta, so, dust.CENTER).double().cpu().numpy()
    assert np.all(np.isfinite(got))
    rng = np.random.default_rng(3)
    n = 64
    chan = rng.integers(0, w.d_out, n)
    col = rng.integers(0, w.d_in, n)
    chan[:2] = [0, w.d_out - 1]
    col[:2] = [0, w.d_in - 1]
    r = oracle.credit(delta, so, np.float32(w.gamma), oracle.CENTER)
    want = oracle.gW_entries(X, r, w.d_out, chan, col, w.seed, w.kind, 0, np.float32(w.sigma),
                             1.0, oracle.CENTER)
    tol = 1e-5 if w.x_dtype == "f32" else 1e-2
    assert rel_fro(got[chan, col], want) <= tol


@pytest.mark.slow
@pytest.mark.parametrize("w", [wl.MLP_UP, wl.sweep_sites()[0]], ids=["mlp_up", "sweep_qkv"])
def test_fused_full_size_sampled(w):
    """The fused path (g tiles made in shared memory, never in HBM) at full
    size against the oracle: the up-projection the bench measures (16,384
    tokens, K 8, gamma 0) and the sweep's QKV site (65,536 tokens, K 32,
    gamma 0.9, through the scan's chunk carries), 64 sampled GW entries."""
    flags = dust.CENTER | dust.FORCE_FUSED
    assert dust.dust_estimate_gW_path(w.T, w.d_in, w.d_out, w.K, dust.BF16,
                                      flags) == dust.PATH_FUSED_TC
    X, delta, so = _inputs(w, planted=w.element_draws <= 1_000_000_000)
    got = _run(w, X, delta, so, flags).double().cpu().numpy()
    assert np.all(np.isfinite(got))
    rng = np.random.default_rng(5)
    n = 64
    chan = rng.integers(0, w.d_out, n)
    col = rng.integers(0, w.d_in, n)
    chan[:2] = [0, w.d_out - 1]
    col[:2] = [0, w.d_in - 1]
    r = oracle.credit(delta, so, np.float32(w.gamma), oracle.CENTER)
    want = oracle.gW_entries(X, r, w.d_out, chan, col, w.seed, w.kind, 0, np.float32(w.sigma),
                             1.0, oracle.CENTER)
    assert rel_fro(got[chan, col], want) <= 1e-2


# ------------------------------------------------- fused vs unfused paths --

FUSED_SHAPES = [
    # T, d_in, d_out, K, kind, gamma
    (1000, 264, 136, 8, 1, 0.9),    # two MMA halves (256 + 64), channel tail, ragged T
    (4096, 512, 2048, 8, 1, 0.0),   # the measured up-projection shape, shorter T
    (777, 40, 256, 5, 0, 0.5),      # one narrow MMA, Rademacher, odd K
    (2048, 512, 512, 32, 1, 0.9),
    (300, 128, 8, 3, 0, 0.0),       # a single 8-channel tile
    (1500, 96, 384, 64, 1, 0.98),   # the largest K of the fused kernel, unaligned carry rows
]


@pytest.mark.parametrize("T,d_in,d_out,K,kind,gamma", FUSED_SHAPES)
def test_fused_matches_unfused(T, d_in, d_out, K, kind, gamma):
    """The fused kernel makes the same bf16 g tiles as the weighting kernel
    (same draw order, same rounding) and contracts them in another order, so
    the two paths agree to fp32 summation error."""
    import torch
    dev = cuda()
    rng = np.random.default_rng(T + d_in + d_out + K)
    so = torch.from_numpy(offsets_from_lengths(random_lengths(rng, T, 300))).to(dev)
    X = torch.from_numpy(rng.standard_normal((T, d_in)).astype(np.float32)).to(torch.bfloat16).to(dev)
    delta = torch.from_numpy((0.05 * rng.standard_normal((K, T))).astype(np.float32)).to(dev)
    args = (d_out, so, 11, kind, 4, 1e-3, gamma, 0.5)
    assert dust.dust_estimate_gW_path(T, d_in, d_out, K, dust.BF16,
                                      dust.CENTER | dust.FORCE_FUSED) == dust.PATH_FUSED_TC
    a = dust.dust_estimate_gW(X, delta, *args, dust.CENTER | dust.FORCE_FUSED)
    b = dust.dust_estimate_gW(X, delta, *args, dust.CENTER | dust.FORCE_UNFUSED)
    torch.cuda.synchronize()
    assert dust.dust_last_error() == dust.OK
    assert rel_fro(a.cpu().numpy(), b.cpu().numpy()) <= 1e-5
    a2 = dust.dust_estimate_gW(X, delta, *args, dust.CENTER | dust.FORCE_FUSED)
    assert torch.equal(a, a2)
    base = torch.randn_like(a)
    acc = base.clone()
    dust.dust_estimate_gW(X, delta, *args, dust.CENTER | dust.FORCE_FUSED | dust.ACCUMULATE,
                          gW=acc)
    assert torch.allclose(acc, base + a, rtol=1e-6, atol=1e-6 * a.abs().max().item())


def test_fused_limits():
    assert dust.dust_estimate_gW_path(1024, 520, 256, 8, dust.BF16, dust.CENTER) == \
        dust.PATH_UNFUSED_TC
    with pytest.raises(dust.DustError):
        dust.dust_estimate_gW_path(1024, 512, 256, 65, dust.BF16, dust.CENTER | dust.FORCE_FUSED)
    with pytest.raises(dust.DustError):
        dust.dust_estimate_gW_path(1024, 520, 256, 8, dust.BF16, dust.CENTER | dust.FORCE_FUSED)
    with pytest.raises(dust.DustError):
        dust.dust_estimate_gW_path(1024, 64, 64, 8, dust.F32, dust.CENTER | dust.FORCE_FUSED)


def test_fused_rejects_packed_signs():
    """The fused kernel evaluates only Gaussian and per-channel signs: packed
    signs with DUST_FORCE_FUSED are refused before anything is enqueued."""
    import torch
    dev = cuda()
    X = torch.zeros((256, 64), dtype=torch.bfloat16, device=dev)
    delta = torch.zeros((4, 256), dtype=torch.float32, device=dev)
    so = torch.tensor([0, 256], dtype=torch.int32, device=dev)
    with pytest.raises(dust.DustError) as e:
        dust.dust_estimate_gW(X, delta, 64, so, 0, dust.RADEMACHER_PACKED, 0, 1e-3, 0.0, 1.0,
                              dust.CENTER | dust.FORCE_FUSED)
    assert e.value.status == dust.ERR_UNSUPPORTED


@pytest.mark.slow
@pytest.mark.parametrize("site", [0, 1, 2, 3], ids=["qkv", "o", "up", "down"])
def test_sweep_site_full_size_sampled(site):
    """One layer of the 12-layer sweep at full size (65,536 tokens, K = 32):
    QKV 512->1536 (gamma 0.9), O 512->512, up 512->2048, down 2048->512."""
    w = wl.sweep_sites()[site]
    X, delta, so = _inputs(w, planted=False)
    got = _run(w, X, delta, so, dust.CENTER).double().cpu().numpy()
    assert np.all(np.isfinite(got))
    rng = np.random.default_rng(11)
    n = 16
    chan = rng.integers(0, w.d_out, n)
    col = rng.integers(0, w.d_in, n)
    r = oracle.credit(delta, so, np.float32(w.gamma), oracle.CENTER)
    want = oracle.gW_entries(X, r, w.d_out, chan, col, w.seed, w.kind, 0, np.float32(w.sigma),
                             1.0, oracle.CENTER)
    assert rel_fro(got[chan, col], want) <= 1e-2


DIRECT_CASES = [
    # T, d_in, d_out, K, kind, flags, x dtype
    (4096, 512, 2048, 8, 1, dust.CENTER, "bf16"),
    (1003, 64, 200, 32, 0, dust.CENTER, "bf16"),               # the most draws read directly
    (1003, 64, 200, 33, 0, dust.CENTER, "bf16"),               # one more: through the scan
    (517, 64, 96, 65, 1, dust.CENTER, "bf16"),                 # two draw groups
    (777, 96, 320, 16, 3, dust.CENTER | dust.ANTITHETIC, "bf16"),
    (300, 40, 72, 6, 1, 0, "f32"),                              # no centring, fp32 path
    (129, 64, 64, 1, 0, dust.CENTER, "f32"),                    # K = 1: centring is a no-op
    (2003, 64, 1024, 16, 1, dust.CENTER | dust.ANTITHETIC, "bf16"),  # wide lanes, 8 pairs
    (500, 40, 1024, 8, 1, dust.CENTER, "f32"),                 # wide lanes, fp32 g
    (1500, 64, 2048, 32, 1, dust.CENTER, "bf16"),              # wide lanes, a draw in every lane
    (900, 64, 1024, 32, 1, dust.CENTER | dust.ANTITHETIC, "bf16"),  # wide lanes, 16 pairs
    (700, 64, 1024, 32, 3, dust.CENTER, "bf16"),               # packed signs, 32 draws
    (333, 48, 1000, 32, 1, dust.CENTER, "bf16"),               # narrow Gaussian lanes, staged
]


@pytest.mark.parametrize("T,d_in,d_out,K,kind,flags,xd", DIRECT_CASES)
def test_gamma_zero_skips_the_scan_bit_for_bit(T, d_in, d_out, K, kind, flags, xd):
    """With gamma = 0 the credit scan is the identity and dust_estimate_gW
    centres the loss changes inside the weighting kernel (no scan kernel).
    The result must equal, bit for bit, the staged path through the scan:
    dust_credit_scan -> dust_error_estimate -> dust_contract."""
    import torch
    dev = cuda()
    rng = np.random.default_rng(T + K + kind)
    so = torch.from_numpy(offsets_from_lengths(random_lengths(rng, T, 250))).to(dev)
    X = torch.from_numpy(rng.standard_normal((T, d_in)).astype(np.float32)).to(dev)
    if xd == "bf16":
        X = X.to(torch.bfloat16)
    delta = torch.from_numpy((0.05 * rng.standard_normal((K, T))).astype(np.float32)).to(dev)
    seed, draw_begin, sigma, scale = 21, 4, 1e-3, 0.5
    got = dust.dust_estimate_gW(X, delta, d_out, so, seed, kind, draw_begin, sigma, 0.0, scale,
                                flags)
    r = dust.dust_credit_scan(delta, so, 0.0, flags & dust.CENTER)
    g = dust.dust_error_estimate(r, d_out, seed, kind, draw_begin, sigma,
                                 flags & dust.ANTITHETIC, g_dtype=X.dtype)
    want = dust.dust_contract(g, X, scale)
    torch.cuda.synchronize()
    assert dust.dust_last_error() == dust.OK
    assert torch.equal(got, want)


@pytest.mark.parametrize("kind", [dust.GAUSSIAN, dust.RADEMACHER])
def test_error_estimate_highest_draw_indices(kind):
    """The weighting with the last legal draws (draw_begin + K = 2^31) and a
    64-bit seed, against the oracle."""
    import torch
    dev = cuda()
    rng = np.random.default_rng(31)
    K, T, d_out = 70, 40, 130
    db = (1 << 31) - K
    r = rng.standard_normal((T, K)).astype(np.float32)
    g = dust.dust_error_estimate(torch.from_numpy(r).to(dev), d_out, 2 ** 63 + 11, kind, db, 1e-2)
    want = oracle.error_estimate(r.T.copy(), d_out, 2 ** 63 + 11, kind, db, np.float32(1e-2), 0)
    assert rel_fro(g.cpu().numpy(), want) <= 1e-5

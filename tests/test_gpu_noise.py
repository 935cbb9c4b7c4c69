"""GPU parity of the noise generator and the jitter (through the C ABI).

Hash words and Rademacher signs must equal the fp64 oracle's bit for bit.
Gaussian values: the GPU evaluates Box-Muller in fp32 with the hardware
log2/sqrt/sin/cos (plus a series near u1 = 1), the oracle in fp64; the bound
|a_gpu - a| <= 1e-5 max(1, |a|) follows from those functions' documented
errors (about 2^-22 absolute for log2 and 2^-21.4 for sin/cos on [-pi, pi]).
"""
import numpy as np
import pytest

import oracle
import token_perturbation_estimator_gb300 as dust
from helpers import cuda

pytestmark = pytest.mark.gpu

SHAPES = [(0, 1, 1, 1), (3, 2, 37, 33), (0, 3, 129, 256), (1000, 2, 64, 1001), (7, 1, 513, 2)]


@pytest.mark.parametrize("draw_begin,n_draws,T,d_out", SHAPES)
@pytest.mark.parametrize("stream", [0, 1])
def test_raw_words_bit_exact(draw_begin, n_draws, T, d_out, stream):
    import torch
    dev = cuda()
    seed = 0xDEADBEEF12345 + draw_begin
    out = torch.empty((n_draws, T, d_out), dtype=torch.int32, device=dev)
    dust.dust_noise(out, seed, dust.RAW_WORDS, draw_begin, n_draws, T, d_out,
                    dust.WORD_STREAM1 if stream else 0)
    got = out.cpu().numpy().view(np.uint32)
    want = oracle.words(seed, draw_begin, n_draws, T, d_out, stream)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("draw_begin,n_draws,T,d_out", SHAPES)
@pytest.mark.parametrize("flags", [0, dust.ANTITHETIC])
@pytest.mark.parametrize("kind", [dust.RADEMACHER, dust.RADEMACHER_PACKED])
def test_rademacher_bit_exact(draw_begin, n_draws, T, d_out, flags, kind):
    import torch
    dev = cuda()
    out = torch.empty((n_draws, T, d_out), dtype=torch.float32, device=dev)
    dust.dust_noise(out, 42, kind, draw_begin, n_draws, T, d_out, flags)
    want = oracle.noise(42, kind, draw_begin, n_draws, T, d_out, flags)
    assert np.array_equal(out.cpu().numpy().astype(np.float64), want)


@pytest.mark.parametrize("draw_begin,n_draws,T,d_out", SHAPES + [(0, 4, 4096, 1024)])
@pytest.mark.parametrize("flags", [0, dust.ANTITHETIC])
def test_gaussian_within_bound(draw_begin, n_draws, T, d_out, flags):
    import torch
    dev = cuda()
    out = torch.empty((n_draws, T, d_out), dtype=torch.float32, device=dev)
    dust.dust_noise(out, 7, dust.GAUSSIAN, draw_begin, n_draws, T, d_out, flags)
    got = out.cpu().numpy().astype(np.float64)
    want = oracle.noise(7, oracle.GAUSSIAN, draw_begin, n_draws, T, d_out, flags)
    err = np.abs(got - want) / np.maximum(1.0, np.abs(want))
    assert err.max() <= 1e-5, float(err.max())


def test_bf16_output_is_rounded_fp32():
    import torch
    dev = cuda()
    for kind in (dust.RADEMACHER, dust.GAUSSIAN, dust.RADEMACHER_PACKED):
        a = torch.empty((2, 100, 77), dtype=torch.float32, device=dev)
        b = torch.empty((2, 100, 77), dtype=torch.bfloat16, device=dev)
        dust.dust_noise(a, 3, kind, 5, 2, 100, 77)
        dust.dust_noise(b, 3, kind, 5, 2, 100, 77)
        assert torch.equal(a.to(torch.bfloat16), b)


def test_counter_limit_two_pow_32():
    """T * d_out = 2^32 exactly: the largest accepted counter range. Sampled
    elements, including the last ones, match the oracle."""
    import torch
    dev = cuda()
    T, d_out = 1 << 22, 1024
    out = torch.empty((1, T, d_out), dtype=torch.bfloat16, device=dev)
    dust.dust_noise(out, 99, dust.RADEMACHER, 0, 1, T, d_out)
    rng = np.random.default_rng(0)
    t = np.concatenate([rng.integers(0, T, 2000), [T - 1, T - 1, 0]])
    c = np.concatenate([rng.integers(0, d_out, 2000), [d_out - 1, d_out - 2, 0]])
    got = out[0, torch.from_numpy(t).to(dev), torch.from_numpy(c).to(dev)].float().cpu().numpy()
    want = oracle.noise_at(np.zeros_like(t), t, c, 99, oracle.RADEMACHER, d_out)
    assert np.array_equal(got.astype(np.float64), want)
    del out
    with pytest.raises(dust.DustError):
        dust.dust_noise(torch.empty(1, device=dev), 99, dust.RADEMACHER, 0, 1, T + 1, d_out)


@pytest.mark.parametrize("kind", [0, 1, 3])
@pytest.mark.parametrize("flags", [0, dust.ANTITHETIC])
def test_jitter_f32(kind, flags):
    import torch
    dev = cuda()
    rng = np.random.default_rng(1)
    T, d_out, ld = 300, 130, 160
    base = rng.standard_normal((T, ld)).astype(np.float32)
    y = torch.from_numpy(base).to(dev)
    dust.dust_jitter_apply(y[:, :d_out], 11, kind, 3, 0.125, flags)
    got = y.cpu().numpy().astype(np.float64)
    want = oracle.jitter(base[:, :d_out], 11, kind, 3, 0.125, flags)
    assert np.max(np.abs(got[:, :d_out] - want)) <= 2e-6 + 1e-6 * np.abs(want).max()
    assert np.array_equal(got[:, d_out:], base[:, d_out:].astype(np.float64))


def test_jitter_bf16():
    import torch
    dev = cuda()
    rng = np.random.default_rng(2)
    T, d_out = 64, 96
    base = torch.from_numpy(rng.standard_normal((T, d_out)).astype(np.float32)).to(torch.bfloat16)
    y = base.to(dev)
    dust.dust_jitter_apply(y, 5, dust.GAUSSIAN, 1, 0.5)
    a = torch.empty((1, T, d_out), dtype=torch.float32, device=dev)
    dust.dust_noise(a, 5, dust.GAUSSIAN, 1, 1, T, d_out)
    # rounding of the fp32 sum to bf16: within one bf16 ulp of the oracle's sum
    want = base.double().numpy() + 0.5 * oracle.noise(5, 1, 1, 1, T, d_out)[0]
    got = y.double().cpu().numpy()
    assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -8 + 1e-6)

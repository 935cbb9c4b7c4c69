"""dust_credit_scan_noalloc: the credit scan for callers that cannot allocate
device memory (a plugin whose host framework's pooling allocator owns the
device, or a latency-critical loop where cudaMalloc/cudaFree may synchronise
the device). It keeps its scratch in a fixed array built into the library,
so the caller passes only inputs and outputs.

Checked through the C ABI against dust_credit_scan (which takes a caller
workspace), on two different calls in a row so that the second one runs on
the array as the first left it. This file is collected last on purpose.
"""
import ctypes as C

import numpy as np
import pytest

import token_perturbation_estimator_gb300 as dust
from helpers import cuda, offsets_from_lengths, random_lengths, rel_fro

pytestmark = pytest.mark.gpu


def _noalloc(L, delta, so, gamma, flags, r, stream):
    K, T = delta.shape
    return L.dust_credit_scan_noalloc(C.c_void_p(delta.data_ptr()), K, T,
                                      C.c_void_p(so.data_ptr()), so.numel() - 1, gamma, flags,
                                      C.c_void_p(r.data_ptr()), C.c_void_p(stream.cuda_stream))


def test_noalloc_scan_matches_workspace_scan_twice():
    import torch
    dev = cuda()
    L = dust.lib()
    assert L.dust_credit_scan_noalloc_capacity() == 8 << 20
    stream = torch.cuda.current_stream()
    cases = [(16, 5000, 700, 0.9, dust.CENTER), (7, 3001, 300, 0.5, 0)]
    for K, T, max_len, gamma, flags in cases:
        rng = np.random.default_rng(K * T)
        so = torch.from_numpy(offsets_from_lengths(random_lengths(rng, T, max_len))).to(dev)
        delta = torch.from_numpy((0.05 * rng.standard_normal((K, T))).astype(np.float32)).to(dev)
        want = dust.dust_credit_scan(delta, so, gamma, flags)
        r = torch.full((T, K), float("nan"), dtype=torch.float32, device=dev)
        st = _noalloc(L, delta, so, gamma, flags, r, stream)
        assert st == dust.OK, dust.status_string(st)
        torch.cuda.synchronize()
        assert dust.dust_last_error() == dust.OK
        got = r.cpu().numpy()
        ref = want.cpu().numpy()
        assert np.all(np.isfinite(got))
        assert rel_fro(got, ref) <= 1e-5


def test_noalloc_rejects_sizes_beyond_capacity():
    import torch
    dev = cuda()
    L = dust.lib()
    stream = torch.cuda.current_stream()
    K, T = 64, 1 << 21  # needs about 8 MiB for P plus 8 MiB of chunk summaries
    fake = torch.empty(16, device=dev)
    st = L.dust_credit_scan_noalloc(C.c_void_p(fake.data_ptr()), K, T,
                                    C.c_void_p(fake.data_ptr()), 1, 0.5, dust.CENTER,
                                    C.c_void_p(fake.data_ptr()), C.c_void_p(stream.cuda_stream))
    assert st == dust.ERR_RANGE
    assert dust.status_string(st).startswith("DUST_ERR_RANGE")

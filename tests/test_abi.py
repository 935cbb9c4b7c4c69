"""The C ABI library loads and exports what include/dust.h declares, and its
host-side argument checks reject bad calls before touching the GPU (CPU only:
every call here fails validation, so nothing is enqueued)."""
import ctypes as C

import pytest

import token_perturbation_estimator_gb300 as dust

NULL = C.c_void_p(0)


@pytest.fixture(scope="module")
def L():
    from token_perturbation_estimator_gb300 import build
    build.build()
    return dust.lib()


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


# Tests that pass fake device addresses: each call is meant to fail its host
# checks, but should a check ever let one through, no kernel may be launched
# on a made-up pointer, so they run only where there is no GPU.
fake_addresses = pytest.mark.skipif(_has_gpu(), reason="fake device addresses: CPU only")


def test_exports_every_declared_function(L):
    names = dust.header_functions()
    assert "dust_estimate_gW" in names and "dust_noise" in names and "dust_jitter_apply" in names
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for s in range(7):
        assert dust.status_string(s).startswith("DUST_")
    assert L.dust_version() >= 100


def _ws(L, T, d_in, d_out, K, xd, flags):
    n = C.c_size_t(0)
    st = L.dust_estimate_gW_workspace(C.byref(n), T, d_in, d_out, K, xd, flags)
    return st, n.value


def test_workspace_query_validation(L):
    assert _ws(L, 16384, 512, 2048, 8, dust.BF16, dust.CENTER)[0] == dust.OK
    assert _ws(L, 16384, 512, 2048, 8, dust.BF16, dust.CENTER)[1] > 0
    assert _ws(L, 16, 8, 8, 0, dust.BF16, 0)[0] == dust.ERR_INVALID_ARG          # K = 0
    assert _ws(L, 16, 8, 8, 9000, dust.BF16, 0)[0] == dust.ERR_RANGE             # K too big
    assert _ws(L, -1, 8, 8, 4, dust.BF16, 0)[0] == dust.ERR_INVALID_ARG
    assert _ws(L, 16, 8, 8, 4, 7, 0)[0] == dust.ERR_INVALID_ARG                  # dtype
    assert _ws(L, 16, 8, 8, 3, dust.BF16, dust.ANTITHETIC)[0] == dust.ERR_INVALID_ARG
    assert _ws(L, 16, 8, 8, 4, dust.BF16, 1 << 20)[0] == dust.ERR_INVALID_ARG    # unknown flag
    assert _ws(L, 16, 8, 8, 4, dust.BF16,
               dust.FORCE_FUSED | dust.FORCE_SIMT)[0] == dust.ERR_INVALID_ARG
    # T * d_out beyond the 32-bit hash counter
    assert _ws(L, (1 << 20) + 1, 8, 4096, 4, dust.BF16, 0)[0] == dust.ERR_RANGE
    assert _ws(L, 1 << 20, 8, 4096, 4, dust.BF16, 0)[0] == dust.OK


def _est(L, **kw):
    a = dict(X=NULL, xd=dust.BF16, T=64, d_in=16, delta=NULL, K=4, d_out=16, so=NULL, n_seq=1,
             seed=0, kind=dust.GAUSSIAN, db=0, sigma=1e-3, gamma=0.0, scale=1.0,
             flags=dust.CENTER, gW=NULL, ws=NULL, wsb=0)
    a.update(kw)
    return L.dust_estimate_gW(a["X"], a["xd"], a["T"], a["d_in"], a["delta"], a["K"],
                              a["d_out"], a["so"], a["n_seq"], a["seed"], a["kind"], a["db"],
                              a["sigma"], a["gamma"], a["scale"], a["flags"], a["gW"], a["ws"],
                              a["wsb"], NULL)


@fake_addresses
def test_estimate_rejects_bad_arguments(L):
    fake = C.c_void_p(1 << 20)
    assert _est(L) == dust.ERR_INVALID_ARG                      # null gW
    assert _est(L, gW=fake) == dust.ERR_INVALID_ARG             # null X / delta
    assert _est(L, gW=fake, sigma=0.0) == dust.ERR_INVALID_ARG
    assert _est(L, gW=fake, sigma=float("nan")) == dust.ERR_INVALID_ARG
    assert _est(L, gW=fake, gamma=1.5) == dust.ERR_INVALID_ARG
    assert _est(L, gW=fake, kind=dust.RAW_WORDS) == dust.ERR_INVALID_ARG
    assert _est(L, gW=fake, K=0) == dust.ERR_INVALID_ARG
    assert _est(L, gW=fake, db=-1) == dust.ERR_INVALID_ARG
    assert _est(L, gW=fake, db=(1 << 31) - 2) == dust.ERR_RANGE
    assert _est(L, gW=fake, n_seq=0) == dust.ERR_INVALID_ARG
    assert _est(L, gW=fake, n_seq=65) == dust.ERR_INVALID_ARG
    assert _est(L, gW=fake, flags=dust.ANTITHETIC, db=1) == dust.ERR_INVALID_ARG
    # all pointers present but no workspace
    assert _est(L, gW=fake, X=fake, delta=fake, so=fake) == dust.ERR_WORKSPACE
    # misaligned workspace
    assert _est(L, gW=fake, X=fake, delta=fake, so=fake, ws=C.c_void_p((1 << 20) + 4),
                wsb=1 << 30) == dust.ERR_WORKSPACE
    # empty layer: nothing to do, success without touching the device
    assert _est(L, d_out=0) == dust.OK


@fake_addresses
def test_noise_and_jitter_reject_bad_arguments(L):
    fake = C.c_void_p(1 << 20)
    assert L.dust_noise(fake, dust.F32, 0, dust.RAW_WORDS, 0, 1, 4, 4, 0, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_noise(fake, dust.U32, 0, dust.GAUSSIAN, 0, 1, 4, 4, 0, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_noise(fake, dust.F32, 0, 9, 0, 1, 4, 4, 0, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_noise(fake, dust.F32, 0, dust.GAUSSIAN, -1, 1, 4, 4, 0, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_noise(fake, dust.F32, 0, dust.GAUSSIAN, 0, 1, 1 << 23, 1 << 10, 0, NULL) == dust.ERR_RANGE
    assert L.dust_noise(NULL, dust.F32, 0, dust.GAUSSIAN, 0, 1, 4, 4, 0, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_noise(NULL, dust.F32, 0, dust.GAUSSIAN, 0, 0, 4, 4, 0, NULL) == dust.OK
    assert L.dust_jitter_apply(fake, dust.F32, 3, 4, 4, 0, dust.GAUSSIAN, 0, 1.0, 0, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_jitter_apply(NULL, dust.F32, 4, 4, 4, 0, dust.GAUSSIAN, 0, 1.0, 0, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_jitter_apply(fake, dust.U32, 4, 4, 4, 0, dust.GAUSSIAN, 0, 1.0, 0, NULL) == dust.ERR_INVALID_ARG


@fake_addresses
def test_scan_and_weighting_reject_bad_arguments(L):
    fake = C.c_void_p(1 << 20)
    assert L.dust_credit_scan(fake, 4, 8, fake, 1, 1.5, 1, fake, fake, 1 << 20, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_credit_scan(fake, 0, 8, fake, 1, 0.5, 1, fake, fake, 1 << 20, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_credit_scan(fake, 4, 8, fake, 1, 0.5, 1, fake, NULL, 0, NULL) == dust.ERR_WORKSPACE
    assert L.dust_error_estimate(fake, 4, 8, 8, 0, dust.GAUSSIAN, 0, 0.0, 0, fake, dust.F32, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_error_estimate(fake, 3, 8, 8, 0, dust.GAUSSIAN, 0, 1.0, dust.ANTITHETIC, fake, dust.F32, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_error_estimate(fake, 4, 8, 8, 0, dust.GAUSSIAN, 0, 1.0, 0, fake, dust.U32, NULL) == dust.ERR_INVALID_ARG


@fake_addresses
def test_packed_signs_accepted_where_values_are(L):
    """DUST_NOISE_RADEMACHER_PACKED is a value kind like the other two: it is
    refused as a word stream and as a U32 output, and unknown kinds (4) are
    refused everywhere."""
    fake = C.c_void_p(1 << 20)
    P = dust.RADEMACHER_PACKED
    assert L.dust_noise(fake, dust.U32, 0, P, 0, 1, 4, 4, 0, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_noise(fake, dust.F32, 0, P, 0, 1, 4, 4, dust.WORD_STREAM1, NULL) == \
        dust.ERR_INVALID_ARG
    assert L.dust_noise(NULL, dust.F32, 0, P, 0, 0, 4, 4, 0, NULL) == dust.OK
    assert L.dust_noise(fake, dust.F32, 0, 4, 0, 1, 4, 4, 0, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_jitter_apply(fake, dust.F32, 4, 0, 4, 0, P, 0, 1.0, 0, NULL) == dust.OK
    assert L.dust_jitter_apply(fake, dust.F32, 4, 4, 4, 0, 4, 0, 1.0, 0, NULL) == \
        dust.ERR_INVALID_ARG
    assert L.dust_jitter_apply(fake, dust.F32, 4, 4, 4, 0, dust.RAW_WORDS, 0, 1.0, 0, NULL) == \
        dust.ERR_INVALID_ARG
    assert L.dust_error_estimate(fake, 4, 0, 8, 0, P, 0, 1.0, 0, fake, dust.F32, NULL) == dust.OK
    assert L.dust_error_estimate(fake, 4, 8, 8, 0, 4, 0, 1.0, 0, fake, dust.F32, NULL) == \
        dust.ERR_INVALID_ARG


@fake_addresses
def test_scatter_and_embedding_estimator_validation(L):
    fake = C.c_void_p(1 << 20)
    n = C.c_size_t(0)
    assert L.dust_scatter_gE_workspace(C.byref(n), 16384, 4096, 512) == dust.OK
    assert n.value >= 8 * 4096 * 512
    assert L.dust_scatter_gE(fake, dust.U32, fake, 8, 4, 4, C.c_float(1.0), 0, fake, fake,
                             1 << 30, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_scatter_gE(fake, dust.F32, fake, 8, 4, 4, C.c_float(1.0), dust.CENTER, fake,
                             fake, 1 << 30, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_scatter_gE(fake, dust.F32, fake, 8, 4, 4, C.c_float(1.0), 0, fake, NULL, 0,
                             NULL) == dust.ERR_WORKSPACE
    assert L.dust_scatter_gE(fake, dust.F32, fake, 8, 4, 0, C.c_float(1.0), 0, NULL, NULL, 0,
                             NULL) == dust.OK
    assert L.dust_estimate_gE_workspace(C.byref(n), 16384, 512, 4096, 8) == dust.OK
    assert L.dust_estimate_gE(fake, 8, 4, fake, 4, 4, fake, 1, 0, dust.GAUSSIAN, 0,
                              C.c_float(0.0), C.c_float(0.0), C.c_float(1.0), 0, fake, fake,
                              1 << 30, NULL) == dust.ERR_INVALID_ARG  # sigma 0
    assert L.dust_estimate_gE(fake, 8, 4, fake, 3, 4, fake, 1, 0, dust.GAUSSIAN, 0,
                              C.c_float(1.0), C.c_float(0.0), C.c_float(1.0), dust.ANTITHETIC,
                              fake, fake, 1 << 30, NULL) == dust.ERR_INVALID_ARG  # odd K
    assert L.dust_estimate_gE(fake, 8, 4, fake, 4, 4, fake, 1, 0, dust.RAW_WORDS, 0,
                              C.c_float(1.0), C.c_float(0.0), C.c_float(1.0), 0, fake, fake,
                              1 << 30, NULL) == dust.ERR_INVALID_ARG


@fake_addresses
def test_forward_jitter_validation(L):
    """Argument checks of dust_forward_jitter that return before any launch."""
    fake = C.c_void_p(1 << 20)
    odd = C.c_void_p((1 << 20) + 8)  # not 16-byte aligned
    f = C.c_float

    def call(X=fake, W=fake, T=64, d_in=64, d_out=64, kind=dust.GAUSSIAN, draw_begin=0,
             n_draws=4, sigma=f(1e-3), flags=0, clean=1, Y=fake):
        return L.dust_forward_jitter(X, W, T, d_in, d_out, 7, kind, draw_begin, n_draws, sigma,
                                     flags, clean, Y, NULL)

    assert call(kind=dust.RAW_WORDS) == dust.ERR_INVALID_ARG
    assert call(kind=9) == dust.ERR_INVALID_ARG
    assert call(flags=dust.CENTER) == dust.ERR_INVALID_ARG
    assert call(clean=2) == dust.ERR_INVALID_ARG
    assert call(T=-1) == dust.ERR_INVALID_ARG
    assert call(sigma=f(float("nan"))) == dust.ERR_INVALID_ARG
    assert call(n_draws=8193) == dust.ERR_RANGE
    assert call(draw_begin=(1 << 31) - 2) == dust.ERR_RANGE
    assert call(T=1 << 27, d_out=64) == dust.ERR_RANGE  # T d_out > 2^32
    assert call(d_in=12) == dust.ERR_UNSUPPORTED
    assert call(d_out=20) == dust.ERR_UNSUPPORTED
    assert call(d_in=0) == dust.ERR_UNSUPPORTED
    assert call(Y=odd) == dust.ERR_UNSUPPORTED
    assert call(Y=NULL) == dust.ERR_INVALID_ARG
    # nothing to write: OK without touching the device
    assert call(T=0, X=NULL, Y=NULL) == dust.OK
    assert call(n_draws=0, clean=0, X=NULL, W=NULL, Y=NULL) == dust.OK


def test_binding_rejects_wrong_dtype_and_shape():
    """The binding checks dtypes and shapes before any C call: the C ABI takes
    raw pointers and sizes, so a float64 delta would be misread and an r of
    the wrong shape written past its end."""
    import torch
    with pytest.raises(ValueError, match="float32"):
        dust._scan_inputs(torch.zeros((4, 8), dtype=torch.float64), torch.zeros(2, dtype=torch.int32))
    with pytest.raises(ValueError, match="int32"):
        dust._scan_inputs(torch.zeros((4, 8)), torch.zeros(2, dtype=torch.int64))
    with pytest.raises(ValueError, match="dimensions"):
        dust._scan_inputs(torch.zeros(8), torch.zeros(2, dtype=torch.int32))
    with pytest.raises(ValueError, match="shape"):
        dust._expect(torch.zeros((8, 3)), "r", (torch.float32,), shape=(8, 4))
    dust._expect(torch.zeros((8, 4)), "r", (torch.float32,), shape=(8, 4))
    dust._expect(torch.zeros((8, 4), dtype=torch.bfloat16), "g",
                 (torch.float32, torch.bfloat16), shape=(8, 4))


@fake_addresses
def test_host_sites_validation_without_a_device(L):
    """Argument errors of the multi-site host entry point are found on the
    host before anything is enqueued: staging that overlaps another buffer,
    too many sites, a bad site argument, a null site array."""
    T, d_in, d_out, K = 1024, 256, 512, 8
    ws = C.c_size_t(0)
    assert L.dust_estimate_gW_workspace(C.byref(ws), T, d_in, d_out, K, dust.BF16,
                                        dust.CENTER) == dust.OK

    def site(base, seed):
        # fake, 256-aligned, disjoint device addresses from `base`
        return dust.HostSite(0x1000, base, T, d_in, d_out, 0x2000, base + (1 << 24), K,
                             0x3000, base + (2 << 24), 4, seed, 1e-3, 0.0, 0x4000,
                             base + (3 << 24), base + (4 << 24), ws.value)

    arr = (dust.HostSite * 2)(site(1 << 32, 1), site(2 << 32, 2))
    arr[1].X_dev = arr[0].workspace  # overlaps site 0's workspace
    call = lambda a, n: L.dust_estimate_gW_host_sites(C.cast(a, C.c_void_p), n, dust.BF16,
                                                       dust.GAUSSIAN, 0, 1.0, dust.CENTER, NULL)
    assert call(arr, 2) == dust.ERR_INVALID_ARG
    arr[1].X_dev = (2 << 32) + 64  # 16-byte aligned, disjoint again, but site 0's delta_dev
    arr[1].delta_dev = arr[0].delta_dev  # shared with a copy-stream write of site 1
    assert call(arr, 2) == dust.ERR_INVALID_ARG
    arr2 = (dust.HostSite * 1)(site(1 << 32, 1))
    arr2[0].ws_bytes = 16  # too small
    assert call(arr2, 1) == dust.ERR_WORKSPACE
    arr2[0].ws_bytes = ws.value
    arr2[0].sigma = 0.0
    assert call(arr2, 1) == dust.ERR_INVALID_ARG
    assert L.dust_estimate_gW_host_sites(NULL, 1, dust.BF16, dust.GAUSSIAN, 0, 1.0,
                                         dust.CENTER, NULL) == dust.ERR_INVALID_ARG
    assert call(arr2, 5000) == dust.ERR_RANGE


@fake_addresses
def test_pipe_probe_rejects_bad_arguments(L):
    ops = C.c_double(0.0)
    sink = C.c_void_p(1 << 32)
    assert L.dust_pipe_probe(7, 100, C.byref(ops), sink, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_pipe_probe(-1, 100, C.byref(ops), sink, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_pipe_probe(dust.PIPE_XU, 0, C.byref(ops), sink, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_pipe_probe(dust.PIPE_XU, 1 << 31, C.byref(ops), sink,
                             NULL) == dust.ERR_INVALID_ARG
    assert L.dust_pipe_probe(dust.PIPE_XU, 100, None, sink, NULL) == dust.ERR_INVALID_ARG
    assert L.dust_pipe_probe(dust.PIPE_XU, 100, C.byref(ops), NULL, NULL) == dust.ERR_INVALID_ARG


@fake_addresses
def test_host_sites_overlap_check_scales_to_many_sites(L):
    """4096 sites (the most one call takes) with one overlap between the first
    and the last: found before anything is enqueued, without a quadratic
    search over the call's buffers."""
    import time
    T, d_in, d_out, K = 256, 64, 64, 4
    ws = C.c_size_t(0)
    assert L.dust_estimate_gW_workspace(C.byref(ws), T, d_in, d_out, K, dust.BF16,
                                        dust.CENTER) == dust.OK
    n = 4096
    arr = (dust.HostSite * n)()
    for i in range(n):
        base = (1 << 40) + i * (1 << 24)  # 16 MiB apart, 256-aligned
        arr[i] = dust.HostSite(0x1000, base, T, d_in, d_out, 0x2000, base + (1 << 20), K,
                               0x3000, base + (2 << 20), 1, i, 1e-3, 0.0, 0x4000,
                               base + (3 << 20), base + (4 << 20), ws.value)
    arr[n - 1].X_dev = arr[0].workspace + 256
    t0 = time.perf_counter()
    st = L.dust_estimate_gW_host_sites(C.cast(arr, C.c_void_p), n, dust.BF16, dust.GAUSSIAN, 0,
                                       1.0, dust.CENTER, NULL)
    assert st == dust.ERR_INVALID_ARG
    assert time.perf_counter() - t0 < 2.0


def test_site_struct_matches_the_header():
    # dust_site is 13 eight-byte fields with no padding (its bytes key graphs)
    assert C.sizeof(dust.Site) == 13 * 8
    assert C.sizeof(dust.HostSite) == 17 * 8


@fake_addresses
def test_sites_validation_without_a_device(L):
    """Argument errors of the multi-site device entry point are found on the
    host before anything is enqueued: what a site writes (gW, workspace)
    overlapping any buffer of another site, too many sites, a bad site
    argument, a null site array. (Sharing read-only inputs between sites is
    accepted; that is checked on the GPU, with real buffers.)"""
    T, d_in, d_out, K = 1024, 256, 512, 8
    ws = C.c_size_t(0)
    assert L.dust_estimate_gW_workspace(C.byref(ws), T, d_in, d_out, K, dust.BF16,
                                        dust.CENTER) == dust.OK

    def site(base, seed):
        # fake, 256-aligned, disjoint device addresses from `base`
        return dust.Site(base, T, d_in, d_out, base + (1 << 24), K, base + (2 << 24), 4, seed,
                         1e-3, 0.0, base + (3 << 24), base + (4 << 24), ws.value)

    call = lambda a, n: L.dust_estimate_gW_sites(C.cast(a, C.c_void_p), n, dust.BF16,
                                                  dust.GAUSSIAN, 0, 1.0, dust.CENTER, NULL)
    arr = (dust.Site * 3)(site(1 << 32, 1), site(2 << 32, 2), site(3 << 32, 3))
    arr[2].workspace = arr[0].workspace  # two sites writing one workspace
    assert call(arr, 3) == dust.ERR_INVALID_ARG
    arr[2].workspace = (3 << 32) + (4 << 24)
    arr[1].gW = arr[2].X + 1024  # a site's result over another site's input
    assert call(arr, 3) == dust.ERR_INVALID_ARG
    arr[1].gW = (2 << 32) + (3 << 24)
    arr[0].X = arr[2].gW + 1024  # an input inside another site's result
    assert call(arr, 3) == dust.ERR_INVALID_ARG
    arr[0].X = 1 << 32
    arr[2].delta = arr[1].workspace + 4096  # an input inside another site's workspace
    assert call(arr, 3) == dust.ERR_INVALID_ARG
    one = (dust.Site * 1)(site(1 << 32, 1))
    one[0].ws_bytes = 16
    assert call(one, 1) == dust.ERR_WORKSPACE
    one[0].ws_bytes = ws.value
    one[0].gamma = 2.0
    assert call(one, 1) == dust.ERR_INVALID_ARG
    assert call(one, 0) == dust.OK  # nothing to do
    assert call(one, -1) == dust.ERR_INVALID_ARG
    assert call(one, 5000) == dust.ERR_RANGE
    assert L.dust_estimate_gW_sites(NULL, 2, dust.BF16, dust.GAUSSIAN, 0, 1.0, dust.CENTER,
                                    NULL) == dust.ERR_INVALID_ARG


@fake_addresses
def test_host_sites_reject_a_shared_workspace(L):
    """With several sites the host entry point computes them on concurrent
    lanes, so two sites may no longer share a workspace (or write into each
    other's buffers)."""
    T, d_in, d_out, K = 1024, 256, 512, 8
    ws = C.c_size_t(0)
    assert L.dust_estimate_gW_workspace(C.byref(ws), T, d_in, d_out, K, dust.BF16,
                                        dust.CENTER) == dust.OK

    def site(base, seed):
        return dust.HostSite(0x1000, base, T, d_in, d_out, 0x2000, base + (1 << 24), K,
                             0x3000, base + (2 << 24), 4, seed, 1e-3, 0.0, 0x4000,
                             base + (3 << 24), base + (4 << 24), ws.value)

    arr = (dust.HostSite * 2)(site(1 << 32, 1), site(2 << 32, 2))
    arr[1].workspace = arr[0].workspace
    call = lambda a, n: L.dust_estimate_gW_host_sites(C.cast(a, C.c_void_p), n, dust.BF16,
                                                       dust.GAUSSIAN, 0, 1.0, dust.CENTER, NULL)
    assert call(arr, 2) == dust.ERR_INVALID_ARG
    arr[1].workspace = (2 << 32) + (4 << 24)
    arr[1].gW_dev = arr[0].workspace + 512  # the last site's result (not copied out of order)
    assert call(arr, 2) == dust.ERR_INVALID_ARG


@fake_addresses
def test_sites_overlap_check_scales_to_many_sites(L):
    """4096 device sites sharing one delta and one offset array, with one
    conflict between the first and the last: found on the host in well under
    a second (sorted sweep, not a search over pairs)."""
    import time
    T, d_in, d_out, K = 256, 64, 64, 4
    ws = C.c_size_t(0)
    assert L.dust_estimate_gW_workspace(C.byref(ws), T, d_in, d_out, K, dust.BF16,
                                        dust.CENTER) == dust.OK
    n = 4096
    arr = (dust.Site * n)()
    delta, so = 1 << 39, (1 << 39) + (1 << 20)  # shared by every site
    for i in range(n):
        base = (1 << 40) + i * (1 << 24)
        arr[i] = dust.Site(base, T, d_in, d_out, delta, K, so, 1, i, 1e-3, 0.0,
                           base + (3 << 20), base + (4 << 20), ws.value)
    arr[n - 1].gW = arr[0].X + 256
    t0 = time.perf_counter()
    st = L.dust_estimate_gW_sites(C.cast(arr, C.c_void_p), n, dust.BF16, dust.GAUSSIAN, 0, 1.0,
                                  dust.CENTER, NULL)
    assert st == dust.ERR_INVALID_ARG
    assert time.perf_counter() - t0 < 2.0

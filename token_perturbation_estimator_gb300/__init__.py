"""Python binding of the GB300 Dust estimator library (``include/dust.h``).

Argument marshalling only: each function passes raw device pointers, sizes and
the current CUDA stream to the C ABI of ``lib/libdust_gb300.so``; every step
of the computation runs in that library's CUDA kernels. PyTorch supplies
device memory and streams. There is no fallback: if the library is missing
the import of a function raises.

Functions keep the C names: ``dust_noise``, ``dust_jitter_apply``,
``dust_forward_jitter``,
``dust_credit_scan``, ``dust_error_estimate``, ``dust_estimate_gW``,
``dust_estimate_gW_host``, ``dust_last_error`` (plus the workspace queries).
"""
from __future__ import annotations

import ctypes as C
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libdust_gb300.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "dust.h")

# dust_status
OK, ERR_INVALID_ARG, ERR_RANGE, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE = range(7)
# dust_noise_kind
RADEMACHER, GAUSSIAN, RAW_WORDS, RADEMACHER_PACKED = 0, 1, 2, 3
# dust_dtype
F32, BF16, U32 = 0, 1, 2
# flags
CENTER, ANTITHETIC, ACCUMULATE = 1, 2, 4
FORCE_UNFUSED, FORCE_FUSED, WORD_STREAM1, FORCE_SIMT = 8, 16, 32, 64
# dust_path
PATH_FUSED_TC, PATH_UNFUSED_TC, PATH_SIMT = 1, 2, 3


class DustError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__("%s: %s" % (where, status_string(status)))


_lib = None


def _signatures():
    i32, i64, u32, u64, f32 = C.c_int32, C.c_int64, C.c_uint32, C.c_uint64, C.c_float
    P, SZ, PSZ = C.c_void_p, C.c_size_t, C.POINTER(C.c_size_t)
    return {
        "dust_status_string": (C.c_char_p, [i32]),
        "dust_version": (i32, []),
        "dust_noise": (i32, [P, i32, u64, i32, i64, i64, i64, i64, u32, P]),
        "dust_jitter_apply": (i32, [P, i32, i64, i64, i64, u64, i32, i64, f32, u32, P]),
        "dust_credit_scan_workspace": (i32, [PSZ, i64, i64]),
        "dust_credit_scan": (i32, [P, i64, i64, P, i64, f32, u32, P, P, SZ, P]),
        "dust_error_estimate": (i32, [P, i64, i64, i64, u64, i32, i64, f32, u32, P, i32, P]),
        "dust_contract_workspace": (i32, [PSZ, i64, i64, i64, i32, u32]),
        "dust_contract": (i32, [P, P, i32, i64, i64, i64, f32, u32, P, P, SZ, P]),
        "dust_estimate_gW_workspace": (i32, [PSZ, i64, i64, i64, i64, i32, u32]),
        "dust_estimate_gW": (i32, [P, i32, i64, i64, P, i64, i64, P, i64, u64, i32, i64, f32,
                                   f32, f32, u32, P, P, SZ, P]),
        "dust_estimate_gW_path": (i32, [i64, i64, i64, i64, i32, u32]),
        "dust_estimate_gW_host": (i32, [P, P, i32, i64, i64, P, P, i64, i64, P, P, i64, u64,
                                        i32, i64, f32, f32, f32, u32, P, P, P, SZ, P]),
        "dust_last_error": (i32, [P]),
        "dust_estimate_gW_host_sites": (i32, [P, i64, i32, i32, i64, f32, u32, P]),
        "dust_estimate_gW_sites": (i32, [P, i64, i32, i32, i64, f32, u32, P]),
        "dust_estimate_gW_sites_lanes": (i32, []),
        "dust_credit_scan_noalloc_capacity": (SZ, []),
        "dust_credit_scan_noalloc": (i32, [P, i64, i64, P, i64, f32, u32, P, P]),
        "dust_forward_jitter": (i32, [P, P, i64, i64, i64, u64, i32, i64, i64, f32, u32, i32,
                                      P, P]),
        "dust_local_score": (i32, [P, i32, P, i32, i64, i64, i64, P, P]),
        "dust_scatter_gE_workspace": (i32, [PSZ, i64, i64, i64]),
        "dust_scatter_gE": (i32, [P, i32, P, i64, i64, i64, f32, u32, P, P, SZ, P]),
        "dust_estimate_gE_workspace": (i32, [PSZ, i64, i64, i64, i64]),
        "dust_estimate_gE": (i32, [P, i64, i64, P, i64, i64, P, i64, u64, i32, i64, f32, f32,
                                   f32, u32, P, P, SZ, P]),
        "dust_debug_inject_timeout": (i32, [i32]),
        "dust_pipe_probe": (i32, [i32, i64, C.POINTER(C.c_double), P, P]),
        "dust_pipe_probe_threads": (i32, []),
        "dust_profile_enable": (i32, [i32]),
        "dust_profile_read": (i32, [P, i32]),
    }


def lib():
    """The loaded C library. Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libdust_gb300.so is not built (run __graft_entry__.build() or "
                              "python token_perturbation_estimator_gb300/build.py)")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _signatures().items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def header_functions():
    """Names of the functions declared in include/dust.h."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dust_[a-zA-Z0-9_]+)\s*\(", text)))


def status_string(status: int) -> str:
    return lib().dust_status_string(int(status)).decode()


def _check(st, where):
    if st != OK:
        raise DustError(st, where)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else C.c_void_p(0)


def _dtype_code(t):
    import torch
    return {torch.float32: F32, torch.bfloat16: BF16, torch.int32: U32,
            torch.uint32: U32}[t.dtype]


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("expected a CUDA tensor")
        if t is not None and not t.is_contiguous():
            raise ValueError("expected a contiguous tensor")


def _expect(t, name, dtypes, shape=None, dim=None):
    """Raise ValueError unless tensor t has one of `dtypes` and, when given,
    exactly `shape` (a tuple) or `dim` dimensions: the C ABI takes raw pointers
    and sizes, so a tensor of another dtype or shape would be misread, or
    written past its end."""
    if t.dtype not in dtypes:
        raise ValueError("%s must be %s, got %s"
                         % (name, " or ".join(str(d) for d in dtypes), t.dtype))
    if dim is not None and t.dim() != dim:
        raise ValueError("%s must have %d dimensions, got shape %s"
                         % (name, dim, tuple(t.shape)))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def _scan_inputs(delta, seq_offsets):
    import torch
    _expect(delta, "delta", (torch.float32,), dim=2)
    _expect(seq_offsets, "seq_offsets", (torch.int32,), dim=1)


# ------------------------------------------------------------------ calls --

def dust_noise(out, seed, kind, draw_begin, n_draws, T, d_out, flags=0, stream=None):
    _need_cuda(out)
    _check(lib().dust_noise(_ptr(out), _dtype_code(out), seed, kind, draw_begin, n_draws, T,
                            d_out, flags, _stream(stream)), "dust_noise")
    return out


def dust_jitter_apply(y, seed, kind, draw, sigma, flags=0, stream=None):
    """y: CUDA tensor [T, d_out] (row stride may exceed d_out)."""
    if not y.is_cuda or y.dim() != 2 or y.stride(1) != 1:
        raise ValueError("y must be a CUDA [T, d_out] tensor with unit column stride")
    T, d_out = y.shape
    _check(lib().dust_jitter_apply(_ptr(y), _dtype_code(y), y.stride(0), T, d_out, seed, kind,
                                   draw, float(sigma), flags, _stream(stream)),
           "dust_jitter_apply")
    return y


def dust_forward_jitter(X, W, seed, kind, draw_begin, n_draws, sigma, flags=0, clean=False,
                        Y=None, stream=None):
    """X: CUDA bf16 [T, d_in]; W: CUDA bf16 [d_out, d_in]; returns Y bf16
    [clean + n_draws, T, d_out]: X W^T, then X W^T + sigma a^(draw_begin + k)."""
    import torch
    _need_cuda(X, W, Y)
    T, d_in = X.shape
    d_out = W.shape[0]
    if W.dim() != 2 or W.shape[1] != d_in:
        raise ValueError("W must be [d_out, d_in] matching X [T, d_in]")
    c = 1 if clean else 0
    if Y is None:
        Y = torch.empty((c + n_draws, T, d_out), dtype=torch.bfloat16, device=X.device)
    if X.dtype != torch.bfloat16 or W.dtype != torch.bfloat16 or Y.dtype != torch.bfloat16:
        raise ValueError("X, W and Y must be bf16")
    if tuple(Y.shape) != (c + n_draws, T, d_out):
        raise ValueError("Y must be [clean + n_draws, T, d_out]")
    _check(lib().dust_forward_jitter(_ptr(X), _ptr(W), T, d_in, d_out, seed, kind, draw_begin,
                                     n_draws, float(sigma), flags, c, _ptr(Y), _stream(stream)),
           "dust_forward_jitter")
    return Y


def dust_local_score(g, delta_o, out=None, stream=None):
    """g: CUDA [T, d] (f32 or bf16); delta_o: CUDA [K, T, d]; returns the loss
    changes delta f32 [K, T] = <g[t], delta_o[k, t]>."""
    import torch
    _need_cuda(g, delta_o, out)
    K, T, d = delta_o.shape
    if tuple(g.shape) != (T, d):
        raise ValueError("g must be [T, d] matching delta_o [K, T, d]")
    if out is None:
        out = torch.empty((K, T), dtype=torch.float32, device=delta_o.device)
    _check(lib().dust_local_score(_ptr(g), _dtype_code(g), _ptr(delta_o), _dtype_code(delta_o),
                                  K, T, d, _ptr(out), _stream(stream)), "dust_local_score")
    return out


def dust_scatter_gE(g, ids, V, scale=1.0, flags=0, gE=None, workspace=None, stream=None):
    """g: CUDA [T, d] (f32 or bf16); ids: CUDA int32 [T]; returns gE f32 [V, d]."""
    import torch
    _need_cuda(g, ids, gE)
    T, d = g.shape
    if gE is None:
        gE = torch.empty((V, d), dtype=torch.float32, device=g.device)
    n = C.c_size_t(0)
    _check(lib().dust_scatter_gE_workspace(C.byref(n), T, V, d), "dust_scatter_gE_workspace")
    if workspace is None:
        workspace = _workspace(n.value, g.device)
    _check(lib().dust_scatter_gE(_ptr(g), _dtype_code(g), _ptr(ids), T, d, V, float(scale),
                                 flags, _ptr(gE), _ptr(workspace), workspace.numel(),
                                 _stream(stream)), "dust_scatter_gE")
    return gE


def dust_estimate_gE(ids, delta, V, d, seq_offsets, seed, kind, draw_begin, sigma, gamma,
                     scale=1.0, flags=CENTER, gE=None, workspace=None, stream=None):
    """ids: CUDA int32 [T]; delta: f32 [K, T]; returns gE f32 [V, d]."""
    import torch
    _need_cuda(ids, delta, seq_offsets, gE)
    T = ids.numel()
    K = delta.shape[0]
    if gE is None:
        gE = torch.empty((V, d), dtype=torch.float32, device=ids.device)
    n = C.c_size_t(0)
    _check(lib().dust_estimate_gE_workspace(C.byref(n), T, d, V, K), "dust_estimate_gE_workspace")
    if workspace is None:
        workspace = _workspace(n.value, ids.device)
    _check(lib().dust_estimate_gE(_ptr(ids), T, V, _ptr(delta), K, d, _ptr(seq_offsets),
                                  seq_offsets.numel() - 1, seed, kind, draw_begin, float(sigma),
                                  float(gamma), float(scale), flags, _ptr(gE), _ptr(workspace),
                                  workspace.numel(), _stream(stream)), "dust_estimate_gE")
    return gE


def dust_credit_scan_workspace(K, T):
    n = C.c_size_t(0)
    _check(lib().dust_credit_scan_workspace(C.byref(n), K, T), "dust_credit_scan_workspace")
    return n.value


def _workspace(nbytes, device):
    import torch
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def dust_credit_scan(delta, seq_offsets, gamma, flags=CENTER, r=None, workspace=None,
                     stream=None):
    """delta: f32 [K, T]; seq_offsets: i32 [n_seq+1]; returns r f32 [T, K]."""
    import torch
    _need_cuda(delta, seq_offsets, r, workspace)
    _scan_inputs(delta, seq_offsets)
    K, T = delta.shape
    if r is None:
        r = torch.empty((T, K), dtype=torch.float32, device=delta.device)
    _expect(r, "r", (torch.float32,), shape=(T, K))
    need = dust_credit_scan_workspace(K, T)
    if workspace is None:
        workspace = _workspace(need, delta.device)
    _check(lib().dust_credit_scan(_ptr(delta), K, T, _ptr(seq_offsets), seq_offsets.numel() - 1,
                                  float(gamma), flags, _ptr(r), _ptr(workspace),
                                  workspace.numel(), _stream(stream)), "dust_credit_scan")
    return r


def dust_credit_scan_noalloc(delta, seq_offsets, gamma, flags=CENTER, r=None, stream=None):
    """As dust_credit_scan, with the library's built-in scratch array instead
    of a caller workspace (for callers that cannot allocate device memory).
    r must be passed in by such callers; it is allocated here only for
    convenience when omitted."""
    import torch
    _need_cuda(delta, seq_offsets, r)
    _scan_inputs(delta, seq_offsets)
    K, T = delta.shape
    if r is None:
        r = torch.empty((T, K), dtype=torch.float32, device=delta.device)
    _expect(r, "r", (torch.float32,), shape=(T, K))
    _check(lib().dust_credit_scan_noalloc(_ptr(delta), K, T, _ptr(seq_offsets),
                                          seq_offsets.numel() - 1, float(gamma), flags, _ptr(r),
                                          _stream(stream)), "dust_credit_scan_noalloc")
    return r


def dust_error_estimate(r, d_out, seed, kind, draw_begin, sigma, flags=0, g=None,
                        g_dtype=None, stream=None):
    """r: f32 [T, K]; returns g [T, d_out] (f32 unless g_dtype=torch.bfloat16)."""
    import torch
    _need_cuda(r, g)
    _expect(r, "r", (torch.float32,), dim=2)
    T, K = r.shape
    if g is None:
        g = torch.empty((T, d_out), dtype=g_dtype or torch.float32, device=r.device)
    _expect(g, "g", (torch.float32, torch.bfloat16), shape=(T, d_out))
    _check(lib().dust_error_estimate(_ptr(r), K, T, d_out, seed, kind, draw_begin, float(sigma),
                                     flags, _ptr(g), _dtype_code(g), _stream(stream)),
           "dust_error_estimate")
    return g


def dust_contract(g, X, scale=1.0, flags=0, gW=None, workspace=None, stream=None):
    """g: [T, d_out], X: [T, d_in], same dtype (bf16 or f32); returns
    gW f32 [d_out, d_in] = scale * g^T X."""
    import torch
    _need_cuda(g, X, gW)
    T, d_out = g.shape
    d_in = X.shape[1]
    dt = _dtype_code(X)
    if gW is None:
        gW = torch.empty((d_out, d_in), dtype=torch.float32, device=X.device)
    n = C.c_size_t(0)
    _check(lib().dust_contract_workspace(C.byref(n), T, d_in, d_out, dt, flags),
           "dust_contract_workspace")
    if workspace is None:
        workspace = _workspace(n.value, X.device)
    _check(lib().dust_contract(_ptr(g), _ptr(X), dt, T, d_in, d_out, float(scale), flags,
                               _ptr(gW), _ptr(workspace), workspace.numel(), _stream(stream)),
           "dust_contract")
    return gW


def dust_estimate_gW_workspace(T, d_in, d_out, K, x_dtype, flags=CENTER):
    n = C.c_size_t(0)
    _check(lib().dust_estimate_gW_workspace(C.byref(n), T, d_in, d_out, K, x_dtype, flags),
           "dust_estimate_gW_workspace")
    return n.value


def dust_estimate_gW_path(T, d_in, d_out, K, x_dtype, flags=CENTER):
    p = lib().dust_estimate_gW_path(T, d_in, d_out, K, x_dtype, flags)
    if p < 0:
        raise DustError(-p, "dust_estimate_gW_path")
    return p


def dust_estimate_gW(X, delta, d_out, seq_offsets, seed, kind, draw_begin, sigma, gamma,
                     scale=1.0, flags=CENTER, gW=None, workspace=None, stream=None):
    """X: [T, d_in] bf16 or f32; delta: f32 [K, T]; returns gW f32 [d_out, d_in]."""
    import torch
    _need_cuda(X, delta, seq_offsets, gW, workspace)
    _expect(X, "X", (torch.float32, torch.bfloat16), dim=2)
    _scan_inputs(delta, seq_offsets)
    T, d_in = X.shape
    K = delta.shape[0]
    _expect(delta, "delta", (torch.float32,), shape=(K, T))
    xd = _dtype_code(X)
    if gW is None:
        gW = torch.empty((d_out, d_in), dtype=torch.float32, device=X.device)
    _expect(gW, "gW", (torch.float32,), shape=(d_out, d_in))
    need = dust_estimate_gW_workspace(T, d_in, d_out, K, xd, flags)
    if workspace is None:
        workspace = _workspace(need, X.device)
    _check(lib().dust_estimate_gW(_ptr(X), xd, T, d_in, _ptr(delta), K, d_out,
                                  _ptr(seq_offsets), seq_offsets.numel() - 1, seed, kind,
                                  draw_begin, float(sigma), float(gamma), float(scale), flags,
                                  _ptr(gW), _ptr(workspace), workspace.numel(),
                                  _stream(stream)), "dust_estimate_gW")
    return gW


def dust_estimate_gW_host(X_host, X_dev, delta_host, delta_dev, seq_host, seq_dev, gW_host,
                          gW_dev, d_out, seed, kind, draw_begin, sigma, gamma, scale=1.0,
                          flags=CENTER, workspace=None, stream=None):
    """Host-buffer variant: *_host are CPU tensors (pinned for async copies),
    *_dev are CUDA staging tensors of the same shapes. The caller
    synchronises the stream before reading gW_host."""
    T, d_in = X_host.shape
    K = delta_host.shape[0]
    xd = _dtype_code(X_host)
    need = dust_estimate_gW_workspace(T, d_in, d_out, K, xd, flags)
    if workspace is None:
        workspace = _workspace(need, X_dev.device)
    _check(lib().dust_estimate_gW_host(
        _ptr(X_host), _ptr(X_dev), xd, T, d_in, _ptr(delta_host), _ptr(delta_dev), K, d_out,
        _ptr(seq_host), _ptr(seq_dev), seq_host.numel() - 1, seed, kind, draw_begin,
        float(sigma), float(gamma), float(scale), flags, _ptr(gW_host), _ptr(gW_dev),
        _ptr(workspace), workspace.numel(), _stream(stream)), "dust_estimate_gW_host")
    return gW_host


PIPE_XU, PIPE_ALU, PIPE_FMA, PIPE_ISSUE = 0, 1, 2, 3


def dust_pipe_probe(pipe, steps, sink, stream=None):
    """Enqueue one pipe-rate probe launch; returns the number of counted
    operations it performs (time it with CUDA events on `stream`). `sink`:
    CUDA float tensor of at least dust_pipe_probe_threads() elements."""
    _need_cuda(sink)
    if sink.numel() < dust_pipe_probe_threads():
        raise ValueError("sink must hold dust_pipe_probe_threads() floats")
    ops = C.c_double(0.0)
    _check(lib().dust_pipe_probe(int(pipe), int(steps), C.byref(ops), _ptr(sink),
                                 _stream(stream)), "dust_pipe_probe")
    return ops.value


def dust_pipe_probe_threads():
    n = lib().dust_pipe_probe_threads()
    if n < 0:
        raise DustError(-n, "dust_pipe_probe_threads")
    return n


class Site(C.Structure):
    """dust_site of include/dust.h: one layer of a multi-site device call."""
    _fields_ = [("X", C.c_void_p), ("T", C.c_int64), ("d_in", C.c_int64),
                ("d_out", C.c_int64), ("delta", C.c_void_p), ("K", C.c_int64),
                ("seq_offsets", C.c_void_p), ("n_seq", C.c_int64), ("seed", C.c_uint64),
                ("sigma", C.c_float), ("gamma", C.c_float), ("gW", C.c_void_p),
                ("workspace", C.c_void_p), ("ws_bytes", C.c_size_t)]


class SiteArray:
    """The marshalled site array of a dust_estimate_gW_sites call, built once
    from a list of dicts (see dust_estimate_gW_sites) and reusable while the
    tensors it points to live (it keeps references to them)."""

    def __init__(self, sites):
        import torch
        self.sites = list(sites)
        self.arr = (Site * max(1, len(self.sites)))()
        self.x_dtype = None
        for i, q in enumerate(self.sites):
            X, delta, so, gW, ws = q["X"], q["delta"], q["seq_offsets"], q["gW"], q["workspace"]
            _need_cuda(X, delta, so, gW, ws)
            _expect(X, "X", (torch.float32, torch.bfloat16), dim=2)
            T, d_in = X.shape
            _expect(delta, "delta", (torch.float32,), dim=2)
            K = delta.shape[0]
            _expect(delta, "delta", (torch.float32,), shape=(K, T))
            _expect(so, "seq_offsets", (torch.int32,), dim=1)
            _expect(gW, "gW", (torch.float32,), dim=2)
            d_out = gW.shape[0]
            _expect(gW, "gW", (torch.float32,), shape=(d_out, d_in))
            _expect(ws, "workspace", (torch.uint8,), dim=1)
            code = _dtype_code(X)
            if self.x_dtype is None:
                self.x_dtype = code
            elif code != self.x_dtype:
                raise ValueError("every site's X must have the same dtype")
            self.arr[i] = Site(_ptr(X), T, d_in, d_out, _ptr(delta), K, _ptr(so), so.numel() - 1,
                               int(q["seed"]), float(q["sigma"]), float(q["gamma"]), _ptr(gW),
                               _ptr(ws), ws.numel())


def dust_estimate_gW_sites(sites, kind, draw_begin, scale=1.0, flags=CENTER, stream=None):
    """Several layers on device buffers in one pass on the library's compute
    lanes (one site's contraction overlaps later sites' weighting).
    `sites`: a SiteArray, or a list of dicts with the CUDA tensors X [T, d_in]
    (bf16 or f32, one dtype for all), delta f32 [K, T], seq_offsets i32
    [n_seq+1], gW f32 [d_out, d_in] (written), a uint8 `workspace` of at least
    dust_estimate_gW_workspace bytes, and the scalars seed, sigma, gamma.
    Returns the gW tensors."""
    a = sites if isinstance(sites, SiteArray) else SiteArray(sites)
    _check(lib().dust_estimate_gW_sites(C.cast(a.arr, C.c_void_p), len(a.sites),
                                        BF16 if a.x_dtype is None else a.x_dtype, kind,
                                        draw_begin, float(scale), flags, _stream(stream)),
           "dust_estimate_gW_sites")
    return [q["gW"] for q in a.sites]


def dust_estimate_gW_sites_lanes():
    return int(lib().dust_estimate_gW_sites_lanes())


class HostSite(C.Structure):
    """dust_host_site of include/dust.h: one layer of a multi-site call."""
    _fields_ = [("X_host", C.c_void_p), ("X_dev", C.c_void_p), ("T", C.c_int64),
                ("d_in", C.c_int64), ("d_out", C.c_int64), ("delta_host", C.c_void_p),
                ("delta_dev", C.c_void_p), ("K", C.c_int64), ("seq_offsets_host", C.c_void_p),
                ("seq_dev", C.c_void_p), ("n_seq", C.c_int64), ("seed", C.c_uint64),
                ("sigma", C.c_float), ("gamma", C.c_float), ("gW_host", C.c_void_p),
                ("gW_dev", C.c_void_p), ("workspace", C.c_void_p), ("ws_bytes", C.c_size_t)]


def dust_estimate_gW_host_sites(sites, kind, draw_begin, scale=1.0, flags=CENTER, stream=None):
    """Several layers from host buffers in one pass (later sites' inputs are
    copied while earlier sites compute). `sites`: list of dicts with the CPU
    tensors X_host [T, d_in], delta_host f32 [K, T], seq_host i32 [n_seq+1],
    gW_host f32 [d_out, d_in] (pinned for overlap), the CUDA staging tensors
    X_dev, delta_dev, seq_dev, gW_dev of the same shapes, a CUDA uint8
    `workspace` and the scalars seed, sigma, gamma. All X share one dtype.
    The caller synchronises the stream before reading the gW_host tensors."""
    import torch
    arr = (HostSite * max(1, len(sites)))()
    xd = None
    for i, q in enumerate(sites):
        Xh, Xd = q["X_host"], q["X_dev"]
        _need_cuda(Xd, q["delta_dev"], q["seq_dev"], q["gW_dev"], q["workspace"])
        _expect(Xh, "X_host", (torch.float32, torch.bfloat16), dim=2)
        T, d_in = Xh.shape
        d_out = q["gW_host"].shape[0]
        K = q["delta_host"].shape[0]
        n_seq = q["seq_host"].numel() - 1
        _expect(Xd, "X_dev", (Xh.dtype,), shape=(T, d_in))
        for nm in ("delta_host", "delta_dev"):
            _expect(q[nm], nm, (torch.float32,), shape=(K, T))
        for nm in ("seq_host", "seq_dev"):
            _expect(q[nm], nm, (torch.int32,), shape=(n_seq + 1,))
        for nm in ("gW_host", "gW_dev"):
            _expect(q[nm], nm, (torch.float32,), shape=(d_out, d_in))
        code = _dtype_code(Xh)
        if xd is None:
            xd = code
        elif code != xd:
            raise ValueError("every site's X must have the same dtype")
        arr[i] = HostSite(_ptr(Xh), _ptr(Xd), T, d_in, d_out, _ptr(q["delta_host"]),
                          _ptr(q["delta_dev"]), K, _ptr(q["seq_host"]), _ptr(q["seq_dev"]),
                          n_seq, int(q["seed"]), float(q["sigma"]), float(q["gamma"]),
                          _ptr(q["gW_host"]), _ptr(q["gW_dev"]), _ptr(q["workspace"]),
                          q["workspace"].numel())
    _check(lib().dust_estimate_gW_host_sites(C.cast(arr, C.c_void_p), len(sites),
                                             BF16 if xd is None else xd, kind, draw_begin,
                                             float(scale), flags, _stream(stream)),
           "dust_estimate_gW_host_sites")
    return [q["gW_host"] for q in sites]


def dust_last_error(stream=None):
    return int(lib().dust_last_error(_stream(stream)))


class _ProfileEntry(C.Structure):
    _fields_ = [("name", C.c_char * 32), ("launches", C.c_int64), ("total_ms", C.c_double)]


def dust_profile_enable(on=True):
    _check(lib().dust_profile_enable(1 if on else 0), "dust_profile_enable")


def dust_profile_read():
    """{kernel family: (launches, total_ms)} since the last read."""
    buf = (_ProfileEntry * 32)()
    n = lib().dust_profile_read(C.cast(buf, C.c_void_p), 32)
    if n < 0:
        raise DustError(-n, "dust_profile_read")
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms))
            for i in range(n)}

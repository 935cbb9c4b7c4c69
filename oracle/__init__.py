"""Python face of the fp64 CPU oracle (``dust_oracle.c``).

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg import this package. It shares no
code with the CUDA library in ``token_perturbation_estimator_gb300`` and the
product path never imports it.

All arrays are numpy, C-contiguous. Floating-point inputs are converted to
float64 (bf16 and fp32 inputs are exact in fp64); outputs are float64.
Layouts follow the C file: delta, c, r are [K, T]; g is [T, d_out]; X is
[T, d_in]; GW is [d_out, d_in].
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

RADEMACHER = 0
GAUSSIAN = 1
RADEMACHER_PACKED = 3  # 32 signs per hash word
CENTER = 1
ANTITHETIC = 2

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        u32, u64, i32, i64, f64 = C.c_uint32, C.c_uint64, C.c_int32, C.c_int64, C.c_double
        P = C.c_void_p
        sig = {
            "dust_oracle_fmix32": (u32, [u32]),
            "dust_oracle_seed_key": (u32, [u64]),
            "dust_oracle_draw_key": (u32, [u64, i64, i32]),
            "dust_oracle_num_threads": (i32, []),
            "dust_oracle_set_threads": (None, [i32]),
            "dust_oracle_words": (None, [P, u64, i64, i64, i64, i64, i32]),
            "dust_oracle_noise": (None, [P, u64, i32, i64, i64, i64, i64, u32]),
            "dust_oracle_noise_at": (None, [P, P, P, P, i64, u64, i32, i64, u32]),
            "dust_oracle_center": (None, [P, i64, i64, u32, P]),
            "dust_oracle_scan": (None, [P, i64, i64, P, i64, f64, P]),
            "dust_oracle_error_estimate": (None, [P, i64, i64, i64, u64, i32, i64, f64, u32, P]),
            "dust_oracle_contract": (None, [P, P, i64, i64, i64, f64, P]),
            "dust_oracle_estimate_gW": (i32, [P, i64, i64, P, i64, i64, P, i64, u64, i32,
                                              i64, f64, f64, f64, u32, P]),
            "dust_oracle_error_rows": (None, [P, i64, i64, i64, P, i64, u64, i32, i64, f64,
                                              u32, P]),
            "dust_oracle_gW_entries": (None, [P, i64, i64, P, i64, i64, P, P, i64, u64, i32,
                                              i64, f64, f64, u32, P]),
            "dust_oracle_bruteforce_gW": (None, [P, i64, i64, P, i64, i64, P, i64, u64, i32,
                                                 i64, f64, f64, f64, u32, P]),
            "dust_oracle_jitter": (None, [P, i64, i64, i64, u64, i32, i64, f64, u32]),
            "dust_oracle_local_score": (None, [P, P, i64, i64, i64, P]),
            "dust_oracle_scatter_gE": (i64, [P, P, i64, i64, i64, f64, P]),
            "dust_oracle_forward_jitter": (None, [P, P, i64, i64, i64, u64, i32, i64, i64, f64,
                                                  u32, i32, P]),
            "dust_oracle_planted_delta": (None, [P, P, P, i64, i64, i64, u64, i32, i64, f64,
                                                 f64, u32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _i64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _p(a):
    return a.ctypes.data_as(C.c_void_p) if a is not None else None


def num_threads() -> int:
    return int(lib().dust_oracle_num_threads())


def set_threads(n: int) -> None:
    lib().dust_oracle_set_threads(int(n))


def fmix32(h: int) -> int:
    return int(lib().dust_oracle_fmix32(int(h) & 0xFFFFFFFF))


def seed_key(seed: int) -> int:
    return int(lib().dust_oracle_seed_key(int(seed)))


def draw_key(seed: int, i: int, s: int) -> int:
    return int(lib().dust_oracle_draw_key(int(seed), int(i), int(s)))


def words(seed, draw_begin, n_draws, T, d_out, stream=0):
    out = np.empty((n_draws, T, d_out), dtype=np.uint32)
    lib().dust_oracle_words(_p(out), seed, draw_begin, n_draws, T, d_out, stream)
    return out


def noise(seed, kind, draw_begin, n_draws, T, d_out, flags=0):
    out = np.empty((n_draws, T, d_out), dtype=np.float64)
    lib().dust_oracle_noise(_p(out), seed, kind, draw_begin, n_draws, T, d_out, flags)
    return out


def noise_at(draw, tok, chan, seed, kind, d_out, flags=0):
    draw, tok, chan = _i64(draw), _i64(tok), _i64(chan)
    out = np.empty(draw.shape[0], dtype=np.float64)
    lib().dust_oracle_noise_at(_p(out), _p(draw), _p(tok), _p(chan), draw.shape[0],
                               seed, kind, d_out, flags)
    return out


def center(delta, flags=CENTER):
    delta = _f64(delta)
    K, T = delta.shape
    out = np.empty_like(delta)
    lib().dust_oracle_center(_p(delta), K, T, flags, _p(out))
    return out


def scan(c, seq_offsets, gamma):
    c = _f64(c)
    K, T = c.shape
    so = _i32(seq_offsets)
    out = np.zeros_like(c)
    lib().dust_oracle_scan(_p(c), K, T, _p(so), so.shape[0] - 1, float(gamma), _p(out))
    return out


def credit(delta, seq_offsets, gamma, flags=CENTER):
    """Centre then scan: r [K, T]."""
    return scan(center(delta, flags), seq_offsets, gamma)


def error_estimate(r, d_out, seed, kind, draw_begin, sigma, flags=CENTER):
    r = _f64(r)
    K, T = r.shape
    out = np.empty((T, d_out), dtype=np.float64)
    lib().dust_oracle_error_estimate(_p(r), K, T, d_out, seed, kind, draw_begin,
                                     float(sigma), flags, _p(out))
    return out


def contract(g, X, scale=1.0):
    g, X = _f64(g), _f64(X)
    T, d_out = g.shape
    d_in = X.shape[1]
    out = np.empty((d_out, d_in), dtype=np.float64)
    lib().dust_oracle_contract(_p(g), _p(X), T, d_in, d_out, float(scale), _p(out))
    return out


def estimate_gW(X, delta, d_out, seq_offsets, seed, kind, draw_begin, sigma, gamma,
                scale=1.0, flags=CENTER):
    X, delta, so = _f64(X), _f64(delta), _i32(seq_offsets)
    T, d_in = X.shape
    K = delta.shape[0]
    out = np.empty((d_out, d_in), dtype=np.float64)
    rc = lib().dust_oracle_estimate_gW(_p(X), T, d_in, _p(delta), K, d_out, _p(so),
                                       so.shape[0] - 1, seed, kind, draw_begin, float(sigma),
                                       float(gamma), float(scale), flags, _p(out))
    if rc != 0:
        raise MemoryError("oracle scratch allocation failed")
    return out


def error_rows(r, d_out, toks, seed, kind, draw_begin, sigma, flags=CENTER):
    r, toks = _f64(r), _i64(toks)
    K, T = r.shape
    out = np.empty((toks.shape[0], d_out), dtype=np.float64)
    lib().dust_oracle_error_rows(_p(r), K, T, d_out, _p(toks), toks.shape[0], seed, kind,
                                 draw_begin, float(sigma), flags, _p(out))
    return out


def gW_entries(X, r, d_out, chan, col, seed, kind, draw_begin, sigma, scale=1.0,
               flags=CENTER):
    X, r, chan, col = _f64(X), _f64(r), _i64(chan), _i64(col)
    T, d_in = X.shape
    K = r.shape[0]
    out = np.empty(chan.shape[0], dtype=np.float64)
    lib().dust_oracle_gW_entries(_p(X), T, d_in, _p(r), K, d_out, _p(chan), _p(col),
                                 chan.shape[0], seed, kind, draw_begin, float(sigma),
                                 float(scale), flags, _p(out))
    return out


def bruteforce_gW(X, delta, d_out, seq_offsets, seed, kind, draw_begin, sigma, gamma,
                  scale=1.0, flags=CENTER):
    X, delta, so = _f64(X), _f64(delta), _i32(seq_offsets)
    T, d_in = X.shape
    K = delta.shape[0]
    out = np.empty((d_out, d_in), dtype=np.float64)
    lib().dust_oracle_bruteforce_gW(_p(X), T, d_in, _p(delta), K, d_out, _p(so),
                                    so.shape[0] - 1, seed, kind, draw_begin, float(sigma),
                                    float(gamma), float(scale), flags, _p(out))
    return out


def jitter(y, seed, kind, draw, sigma, flags=0):
    y = _f64(y).copy()
    T, d_out = y.shape
    lib().dust_oracle_jitter(_p(y), d_out, T, d_out, seed, kind, draw, float(sigma), flags)
    return y


def forward_jitter(X, W, seed, kind, draw_begin, n_draws, sigma, flags=0, clean=False):
    """y = X W^T and y + sigma a^(draw_begin + k) for k < n_draws, stacked
    [clean + n_draws][T][d_out] (slice 0 = y when clean)."""
    X = _f64(X)
    W = _f64(W)
    T, d_in = X.shape
    d_out = W.shape[0]
    assert W.shape == (d_out, d_in)
    c = 1 if clean else 0
    out = np.empty((c + n_draws, T, d_out), dtype=np.float64)
    lib().dust_oracle_forward_jitter(_p(X), _p(W), T, d_in, d_out, seed, kind, draw_begin,
                                     n_draws, float(sigma), flags, c, _p(out))
    return out


def scatter_gE(g, ids, V, scale=1.0):
    """gE[v] = scale * sum of g[t] over the tokens t with ids[t] == v, in token
    order; ids outside [0, V) are skipped (their count is returned too)."""
    g = _f64(g)
    T, d = g.shape
    ids = _i32(ids)
    assert ids.shape == (T,)
    out = np.empty((V, d), dtype=np.float64)
    bad = lib().dust_oracle_scatter_gE(_p(g), _p(ids), T, d, V, float(scale), _p(out))
    return out, int(bad)


def local_score(g, delta_o):
    """delta[k][s] = <g[s], delta_o[k][s]>: the loss change whose reduction is
    the page's local score c_s = -<g_s, delta_o_s>."""
    g = _f64(g)
    delta_o = _f64(delta_o)
    K, T, d = delta_o.shape
    assert g.shape == (T, d)
    out = np.empty((K, T), dtype=np.float64)
    lib().dust_oracle_local_score(_p(g), _p(delta_o), K, T, d, _p(out))
    return out


def planted_delta(dplant, seed, kind, draw_begin, n_draws, sigma, curv=1.0, eps=None,
                  flags=0):
    dplant = _f64(dplant)
    T, d_out = dplant.shape
    e = _f64(eps) if eps is not None else None
    out = np.empty((n_draws, T), dtype=np.float64)
    lib().dust_oracle_planted_delta(_p(out), _p(dplant), _p(e), n_draws, T, d_out, seed,
                                    kind, draw_begin, float(sigma), float(curv), flags)
    return out

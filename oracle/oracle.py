"""ctypes front end of the fp64 CPU oracle (``ssm_oracle.c``).

TEST INFRASTRUCTURE ONLY. Inputs may be numpy arrays or CPU torch tensors of any
float dtype; they are widened exactly to float64 (bf16 and fp32 values are
representable in fp64) and passed to the C routines. Outputs are float64 numpy
arrays. Nothing here does arithmetic of the method: it only marshals arguments.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import numpy as np

from . import build_oracle

_lib = None
_P = ctypes.POINTER(ctypes.c_double)


def _load():
    global _lib
    if _lib is None:
        path = build_oracle.build()
        lib = ctypes.CDLL(path)
        L, I = ctypes.c_long, ctypes.c_int
        lib.oracle_softplus.argtypes = [_P, _P, L]
        lib.oracle_silu.argtypes = [_P, _P, L]
        lib.oracle_causal_conv1d.argtypes = [_P, _P, _P, _P, _P, L, L, L, I, I, I]
        lib.oracle_selective_scan.argtypes = ([_P] * 8 + [I] + [_P, _P, I] + [_P, _P, _P, _P, _P, _P]
                                              + [L, L, L, L, I, I])
        lib.oracle_compose.argtypes = [_P, _P, _P, _P, _P, _P, L]
        lib.oracle_chunk_aggregates.argtypes = ([_P] * 5 + [I] + [_P, _P, I, _P, L, _P, _P]
                                                + [L, L, L, L, I, I])
        lib.oracle_state_update.argtypes = ([_P, _P] + [_P] * 8 + [I] + [_P, _P, I, _P] + [L, L, L, I, I])
        lib.oracle_selective_scan_bwd.argtypes = ([_P] * 8 + [I] + [_P] * 3 + [_P] * 9 + [L, L, L, L, I])
        lib.oracle_causal_conv1d_bwd.argtypes = [_P] * 9 + [L, L, L, I, I, I]
        lib.oracle_ssd.argtypes = [_P] * 7 + [I, _P, _P, _P] + [L] * 5 + [I]
        for f in ("oracle_softplus", "oracle_silu", "oracle_causal_conv1d", "oracle_selective_scan", "oracle_ssd",
                  "oracle_compose", "oracle_chunk_aggregates", "oracle_state_update", "oracle_selective_scan_bwd",
                  "oracle_causal_conv1d_bwd"):
            getattr(lib, f).restype = None
        _lib = lib
    return _lib


def _f64(a) -> Optional[np.ndarray]:
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(_P)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def softplus(x) -> np.ndarray:
    x = _f64(x)
    y = np.empty_like(x)
    _load().oracle_softplus(_ptr(x), _ptr(y), x.size)
    return y


def silu(x) -> np.ndarray:
    x = _f64(x)
    y = np.empty_like(x)
    _load().oracle_silu(_ptr(x), _ptr(y), x.size)
    return y


def causal_conv1d(x, w, bias=None, window=None, apply_silu: bool = True, nthreads: int = 1) -> np.ndarray:
    """x [batch, dim, L], w [dim, K], bias [dim] or None, window [batch, dim, K-1] or None."""
    x, w, bias, window = _f64(x), _f64(w), _f64(bias), _f64(window)
    batch, dim, L = x.shape
    K = w.shape[1]
    out = np.empty_like(x)
    _load().oracle_causal_conv1d(_ptr(x), _ptr(w), _ptr(bias), _ptr(window), _ptr(out), batch, dim, L, K,
                                 int(apply_silu), nthreads)
    return out


def causal_conv1d_bwd(x, w, dout, bias=None, window=None, apply_silu: bool = True, nthreads: int = 1) -> dict:
    """Gradients through causal_conv1d from dout = dL/dout: dict with dx [b, d, L], dw [d, K],
    dbias [d] (None without bias) and dwindow [b, d, K-1] (None without a window)."""
    x, w, dout, bias, window = _f64(x), _f64(w), _f64(dout), _f64(bias), _f64(window)
    batch, dim, L = x.shape
    K = w.shape[1]
    g = {"dx": np.empty_like(x), "dw": np.empty((dim, K)), "dbias": np.empty(dim) if bias is not None else None,
         "dwindow": np.empty((batch, dim, K - 1)) if (window is not None and K > 1) else None}
    _load().oracle_causal_conv1d_bwd(_ptr(x), _ptr(w), _ptr(bias), _ptr(window), _ptr(dout), _ptr(g["dx"]),
                                     _ptr(g["dwindow"]), _ptr(g["dw"]), _ptr(g["dbias"]), batch, dim, L, K,
                                     int(apply_silu), nthreads)
    return g


def selective_scan(x, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus: bool = True,
                   conv_w=None, conv_b=None, conv_init=None, h0=None, want_conv_state: bool = False,
                   want_trace: bool = False, nthreads: int = 1, reverse: bool = False,
                   zoh: bool = False) -> Tuple[np.ndarray, ...]:
    """Returns (out [b, d, L], h_last [b, d, N]) plus conv_state_out and/or h_trace [b, d, L, N] if asked.

    reverse: the backward scan of a bidirectional layer ("Mamba", ozercemkelahmet.com, "Bidirectional
    and multi-directional scans": one scan runs forward, one backward). It is the forward scan of
    the time-reversed stream, so it is computed as exactly that: the per-token inputs are re-indexed
    t -> L-1-t, the forward routine runs, and out / h_trace are re-indexed back. h0, conv_init and
    the returned h_last / conv_state_out belong to the reversed stream (conv_init[j] is the raw
    input at L+K-2-j; conv_state_out[j] is x at K-2-j).

    zoh: zero-order-hold input factor, Bbar = expm1(Delta A)/A * B, instead of Euler's Delta * B.
    """
    x, delta, A, B, C = _f64(x), _f64(delta), _f64(A), _f64(B), _f64(C)
    D, z, delta_bias, conv_w, conv_b, conv_init, h0 = map(_f64, (D, z, delta_bias, conv_w, conv_b, conv_init, h0))
    if reverse:
        flip = lambda a: None if a is None else np.ascontiguousarray(a[..., ::-1])
        x, delta, B, C, z = map(flip, (x, delta, B, C, z))
    batch, dim, L = x.shape
    N = A.shape[1]
    K = conv_w.shape[1] if conv_w is not None else 0
    out = np.empty((batch, dim, L))
    h_last = np.empty((batch, dim, N))
    cs = np.empty((batch, dim, max(K - 1, 0))) if (want_conv_state and K > 1) else None
    tr = np.empty((batch, dim, L, N)) if want_trace else None
    _load().oracle_selective_scan(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                  _ptr(delta_bias), int(delta_softplus), _ptr(conv_w), _ptr(conv_b), K,
                                  _ptr(conv_init), _ptr(h0), _ptr(out), _ptr(h_last), _ptr(cs), _ptr(tr),
                                  batch, dim, L, N, nthreads, int(zoh))
    if reverse:
        out = np.ascontiguousarray(out[..., ::-1])
        tr = None if tr is None else np.ascontiguousarray(tr[:, :, ::-1, :])
    res = [out, h_last]
    if want_conv_state:
        res.append(cs)
    if want_trace:
        res.append(tr)
    return tuple(res)


def selective_scan_bwd(u, delta, A, B, C, dout, D=None, z=None, delta_bias=None, delta_softplus: bool = True,
                       h0=None, dh_last=None, nthreads: int = 1) -> dict:
    """Gradients of a scalar loss through selective_scan (u given directly, Euler, forward in
    time) from dout = dL/dout and dh_last = dL/dh_last. Returns a dict with du, ddelta, dz (or
    None), dA [d, N], dB, dC [b, N, L], dD, ddelta_bias [d] (None when D / delta_bias are None)
    and dh0 [b, d, N]."""
    u, delta, A, B, C, dout = _f64(u), _f64(delta), _f64(A), _f64(B), _f64(C), _f64(dout)
    D, z, delta_bias, h0, dh_last = map(_f64, (D, z, delta_bias, h0, dh_last))
    batch, dim, L = u.shape
    N = A.shape[1]
    g = {"du": np.empty((batch, dim, L)), "ddelta": np.empty((batch, dim, L)),
         "dz": np.empty((batch, dim, L)) if z is not None else None, "dA": np.empty((dim, N)),
         "dB": np.empty((batch, N, L)), "dC": np.empty((batch, N, L)),
         "dD": np.empty(dim) if D is not None else None,
         "ddelta_bias": np.empty(dim) if delta_bias is not None else None, "dh0": np.empty((batch, dim, N))}
    _load().oracle_selective_scan_bwd(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                      _ptr(delta_bias), int(delta_softplus), _ptr(h0), _ptr(dout), _ptr(dh_last),
                                      _ptr(g["du"]), _ptr(g["ddelta"]), _ptr(g["dz"]), _ptr(g["dA"]), _ptr(g["dB"]),
                                      _ptr(g["dC"]), _ptr(g["dD"]), _ptr(g["ddelta_bias"]), _ptr(g["dh0"]),
                                      batch, dim, L, N, nthreads)
    return g


def compose(a1, b1, a2, b2) -> Tuple[np.ndarray, np.ndarray]:
    """(a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2), elementwise."""
    a1, b1, a2, b2 = map(_f64, (a1, b1, a2, b2))
    a = np.empty_like(a1)
    b = np.empty_like(a1)
    _load().oracle_compose(_ptr(a1), _ptr(b1), _ptr(a2), _ptr(b2), _ptr(a), _ptr(b), a1.size)
    return a, b


def chunk_aggregates(x, delta, A, B, delta_bias=None, delta_softplus: bool = True, conv_w=None, conv_b=None,
                     conv_init=None, chunk_len: int = 64, nthreads: int = 1,
                     zoh: bool = False) -> Tuple[np.ndarray, np.ndarray]:
    """Per-chunk aggregates (a, b), each [batch, dim, nchunks, N]."""
    x, delta, A, B = _f64(x), _f64(delta), _f64(A), _f64(B)
    delta_bias, conv_w, conv_b, conv_init = map(_f64, (delta_bias, conv_w, conv_b, conv_init))
    batch, dim, L = x.shape
    N = A.shape[1]
    K = conv_w.shape[1] if conv_w is not None else 0
    q = (L + chunk_len - 1) // chunk_len
    agg_a = np.empty((batch, dim, q, N))
    agg_b = np.empty((batch, dim, q, N))
    _load().oracle_chunk_aggregates(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(delta_bias),
                                    int(delta_softplus), _ptr(conv_w), _ptr(conv_b), K, _ptr(conv_init),
                                    chunk_len, _ptr(agg_a), _ptr(agg_b), batch, dim, L, N, nthreads, int(zoh))
    return agg_a, agg_b


def state_update(state, conv_state, x, delta, A, B, C, D=None, z=None, delta_bias=None,
                 delta_softplus: bool = True, conv_w=None, conv_b=None, nthreads: int = 1, zoh: bool = False):
    """One decode step. Returns (y [batch, dim], new state, new conv_state); the inputs are not modified.
    zoh: zero-order-hold input factor expm1(Delta A)/A instead of Delta."""
    state = _f64(state).copy()
    conv_state = _f64(conv_state).copy() if conv_state is not None else None
    x, delta, A, B, C = _f64(x), _f64(delta), _f64(A), _f64(B), _f64(C)
    D, z, delta_bias, conv_w, conv_b = map(_f64, (D, z, delta_bias, conv_w, conv_b))
    batch, dim = x.shape
    N = A.shape[1]
    K = conv_w.shape[1] if conv_w is not None else 0
    y = np.empty((batch, dim))
    _load().oracle_state_update(_ptr(state), _ptr(conv_state), _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                _ptr(D), _ptr(z), _ptr(delta_bias), int(delta_softplus), _ptr(conv_w),
                                _ptr(conv_b), K, _ptr(y), batch, dim, N, nthreads, int(zoh))
    return y, state, conv_state


def ssd(x, dt, A, B, C, D=None, dt_bias=None, dt_softplus: bool = True, h0=None,
        nthreads: int = 1) -> Tuple[np.ndarray, np.ndarray]:
    """Multi-head SSM with one scalar decay per head (the layer of the state-space duality).

    x [batch, L, H, P], dt [batch, L, H], A [H], B, C [batch, L, N], D and dt_bias [H],
    h0 [batch, H, P, N]. Returns (y [batch, L, H, P], h_last [batch, H, P, N])."""
    x, dt, A, B, C = _f64(x), _f64(dt), _f64(A), _f64(B), _f64(C)
    D, dt_bias, h0 = map(_f64, (D, dt_bias, h0))
    batch, L, H, P = x.shape
    N = B.shape[2]
    y = np.empty((batch, L, H, P))
    h_last = np.empty((batch, H, P, N))
    _load().oracle_ssd(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(dt_bias), int(dt_softplus),
                       _ptr(h0), _ptr(y), _ptr(h_last), batch, L, H, P, N, nthreads)
    return y, h_last

"""Python binding of libssm.so (argument marshalling only).

Each function takes CUDA torch tensors, checks shapes, dtypes and contiguity, and calls
the C entry point of the same name on the current torch stream with raw device pointers.
Every step of the computation runs in the library's kernels; nothing here computes.
The library must have been built (``__graft_entry__.build()`` or ``python -m
selective_state_space_145_b300.build``): a missing library raises, there is no fallback.
``select_library("debug")`` points every call at libssm_debug.so, the range-checked build
(``debug_bounds_status`` reads its error word).
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssm.so")
DEBUG_LIB_PATH = os.path.join(_HERE, "libssm_debug.so")
_LIB_KINDS = ("release", "debug")
_lib_kind = "release"
_loaded = {}

SSM_OK, SSM_ERR_INVALID_ARG, SSM_ERR_UNSUPPORTED, SSM_ERR_CUDA = 0, 1, 2, 3
SSM_F32, SSM_BF16 = 0, 1

_DTYPE_CODE = {torch.float32: SSM_F32, torch.bfloat16: SSM_BF16}

_lib = None

# Exported C symbols, as declared in include/ssm.h.
EXPORTS = ("ssm_version", "ssm_status_string", "ssm_causal_conv1d_fwd", "ssm_scan_default_chunk_len",
           "ssm_scan_workspace_bytes", "ssm_selective_scan_fwd", "ssm_selective_state_update",
           "ssm_selective_scan_fwd_noalloc", "ssm_scan_bwd_workspace_bytes", "ssm_selective_scan_bwd",
           "ssm_conv_bwd_workspace_bytes", "ssm_causal_conv1d_bwd", "ssm_ssd_workspace_bytes", "ssm_ssd_fwd",
           "ssm_set_test_hooks", "ssm_scan_aggregate_workspace_bytes", "ssm_selective_scan_aggregate",
           "ssm_scan_compose", "ssm_debug_bounds_status")

# Bits of the debug build's error word (include/ssm.h).
BOUNDS_SCAN, BOUNDS_DECODE, BOUNDS_CONV, BOUNDS_SEGMENT, BOUNDS_BACKWARD, BOUNDS_SSD = 1, 2, 4, 8, 16, 32

# Bytes of the fixed device scratch array ssm_selective_scan_fwd_noalloc uses (include/ssm.h).
NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024

# Option bits (include/ssm.h).
SCAN_REVERSE = 1
SCAN_ZOH = 2
SCAN_S4D_REAL = 4


class SSMError(RuntimeError):
    """A libssm call returned a non-OK status."""

    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")
        self.status = status


def select_library(kind: str) -> None:
    """Route every following call to libssm.so ("release", the default) or libssm_debug.so
    ("debug"). Both may stay loaded; each is loaded once."""
    global _lib, _lib_kind
    if kind not in _LIB_KINDS:
        raise ValueError(f"unknown library kind {kind!r}")
    _lib_kind = kind
    _lib = _loaded.get(kind)


def library_path() -> str:
    """Path of the library the calls go to."""
    return LIB_PATH if _lib_kind == "release" else DEBUG_LIB_PATH


def lib() -> ctypes.CDLL:
    """Load the selected library once; raise if it has not been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build the CUDA library first "
                               "(python -m selective_state_space_145_b300.build"
                               + (" --debug)" if _lib_kind == "debug" else ")"))
        L = ctypes.CDLL(path)
        vp, fp, i, sz, u = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint
        L.ssm_version.restype = i
        L.ssm_version.argtypes = []
        L.ssm_status_string.restype = ctypes.c_char_p
        L.ssm_status_string.argtypes = [i]
        L.ssm_causal_conv1d_fwd.restype = i
        L.ssm_causal_conv1d_fwd.argtypes = [vp, fp, fp, vp, vp, i, i, i, i, i, i, vp]
        L.ssm_scan_default_chunk_len.restype = i
        L.ssm_scan_default_chunk_len.argtypes = [i, i, i, i, i]
        L.ssm_scan_workspace_bytes.restype = sz
        L.ssm_scan_workspace_bytes.argtypes = [i, i, i, i, i, i]
        L.ssm_selective_scan_fwd.restype = i
        L.ssm_selective_scan_fwd.argtypes = ([vp, vp, fp, vp, vp, fp, vp, fp, i, fp, fp, i, vp, fp, vp, fp, vp]
                                             + [i] * 6 + [vp, sz, u, vp])
        L.ssm_selective_scan_fwd_noalloc.restype = i
        L.ssm_selective_scan_fwd_noalloc.argtypes = ([vp, vp, fp, vp, vp, fp, vp, fp, i, fp, fp, i, vp, fp, vp, fp, vp]
                                                     + [i] * 6 + [u, vp])
        L.ssm_conv_bwd_workspace_bytes.restype = sz
        L.ssm_conv_bwd_workspace_bytes.argtypes = [i, i, i, i, i]
        L.ssm_causal_conv1d_bwd.restype = i
        L.ssm_causal_conv1d_bwd.argtypes = [vp, fp, fp, vp, vp, i, vp, fp, fp, vp, i, i, i, i, i, vp, sz, vp]
        L.ssm_scan_bwd_workspace_bytes.restype = sz
        L.ssm_scan_bwd_workspace_bytes.argtypes = [i, i, i, i, i]
        L.ssm_selective_scan_bwd.restype = i
        L.ssm_selective_scan_bwd.argtypes = ([vp, vp, fp, vp, vp, fp, vp, fp, i, fp, vp, fp]
                                             + [vp, vp, vp, fp, fp, fp, fp, fp, fp] + [i] * 5 + [vp, sz, u, vp])
        L.ssm_set_test_hooks.restype = None
        L.ssm_set_test_hooks.argtypes = [u]
        L.ssm_ssd_workspace_bytes.restype = sz
        L.ssm_ssd_workspace_bytes.argtypes = [i] * 6
        L.ssm_ssd_fwd.restype = i
        L.ssm_ssd_fwd.argtypes = [vp, vp, fp, vp, vp, fp, fp, i, fp, vp, fp] + [i] * 6 + [vp, sz, vp]
        L.ssm_scan_aggregate_workspace_bytes.restype = sz
        L.ssm_scan_aggregate_workspace_bytes.argtypes = [i] * 5
        L.ssm_selective_scan_aggregate.restype = i
        L.ssm_selective_scan_aggregate.argtypes = ([vp, vp, fp, vp, fp, i, fp, fp, i, vp, fp, fp] + [i] * 5
                                                   + [vp, sz, u, vp])
        L.ssm_scan_compose.restype = i
        L.ssm_scan_compose.argtypes = [fp, fp, fp, fp, fp, i, i, i, i, vp]
        L.ssm_selective_state_update.restype = i
        L.ssm_selective_state_update.argtypes = [fp, vp, vp, vp, fp, vp, vp, fp, vp, fp, i, fp, fp, i, vp,
                                                 i, i, i, i, u, vp]
        L.ssm_debug_bounds_status.restype = i
        L.ssm_debug_bounds_status.argtypes = [ctypes.POINTER(ctypes.c_uint), i]
        _lib = L
        _loaded[_lib_kind] = L
    return _lib


def debug_bounds_status(clear: bool = True) -> int:
    """The debug library's error word (0: no checked access left its tensor), cleared when
    `clear`. Synchronises the device. Raises SSMError(SSM_ERR_UNSUPPORTED) on the release library."""
    word = ctypes.c_uint(0)
    _check("ssm_debug_bounds_status", lib().ssm_debug_bounds_status(ctypes.byref(word), 1 if clear else 0))
    return int(word.value)


def version() -> int:
    return lib().ssm_version()


def status_string(status: int) -> str:
    return lib().ssm_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != SSM_OK:
        raise SSMError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _io_code(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPE_CODE:
        raise TypeError(f"unsupported I/O dtype {t.dtype}; use float32 or bfloat16")
    return _DTYPE_CODE[t.dtype]


def _need(t: Optional[torch.Tensor], name: str, shape, dtype, device, optional=False):
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name}: expected device {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def ssm_causal_conv1d_fwd(x: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor] = None,
                          conv_init: Optional[torch.Tensor] = None, apply_silu: bool = True,
                          out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Causal depthwise conv1d (+SiLU). x [batch, dim, L] (f32/bf16), w [dim, K] f32."""
    batch, dim, L = x.shape
    K = w.shape[1]
    dev, io = x.device, x.dtype
    _need(x, "x", (batch, dim, L), io, dev)
    _need(w, "w", (dim, K), torch.float32, dev)
    _need(bias, "bias", (dim,), torch.float32, dev, optional=True)
    _need(conv_init, "conv_init", (batch, dim, K - 1), io, dev, optional=True)
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", (batch, dim, L), io, dev)
    st = lib().ssm_causal_conv1d_fwd(_ptr(x), _ptr(w), _ptr(bias), _ptr(conv_init), _ptr(out), batch, dim, L, K,
                                     int(bool(apply_silu)), _io_code(x), _stream(dev))
    _check("ssm_causal_conv1d_fwd", st)
    return out


def ssm_causal_conv1d_bwd(x: torch.Tensor, w: torch.Tensor, dout: torch.Tensor, bias: Optional[torch.Tensor] = None,
                          conv_init: Optional[torch.Tensor] = None, apply_silu: bool = True,
                          workspace: Optional[torch.Tensor] = None) -> dict:
    """Backward of ssm_causal_conv1d_fwd. Returns a dict with dx [batch, dim, L] (io dtype),
    dw [dim, K] and dbias [dim] (float32), and dconv_init [batch, dim, K-1] (io dtype; None
    without conv_init or for K = 1)."""
    batch, dim, L = x.shape
    K = w.shape[1]
    dev, io = x.device, x.dtype
    _need(x, "x", (batch, dim, L), io, dev)
    _need(w, "w", (dim, K), torch.float32, dev)
    _need(dout, "dout", (batch, dim, L), io, dev)
    _need(bias, "bias", (dim,), torch.float32, dev, optional=True)
    _need(conv_init, "conv_init", (batch, dim, K - 1), io, dev, optional=True)
    g = {"dx": torch.empty_like(x), "dw": torch.empty(dim, K, dtype=torch.float32, device=dev),
         "dbias": torch.empty(dim, dtype=torch.float32, device=dev),
         "dconv_init": torch.empty(batch, dim, K - 1, dtype=io, device=dev) if (conv_init is not None and K > 1)
         else None}
    need = int(lib().ssm_conv_bwd_workspace_bytes(batch, dim, L, K, _io_code(x)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    st = lib().ssm_causal_conv1d_bwd(_ptr(x), _ptr(w), _ptr(bias), _ptr(conv_init), _ptr(dout), int(bool(apply_silu)),
                                     _ptr(g["dx"]), _ptr(g["dw"]), _ptr(g["dbias"]), _ptr(g["dconv_init"]),
                                     batch, dim, L, K, _io_code(x), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(dev))
    _check("ssm_causal_conv1d_bwd", st)
    return g


def ssm_scan_default_chunk_len(batch: int, dim: int, seqlen: int, dstate: int, io: torch.dtype) -> int:
    return lib().ssm_scan_default_chunk_len(batch, dim, seqlen, dstate, _DTYPE_CODE[io])


def ssm_scan_workspace_bytes(batch: int, dim: int, seqlen: int, dstate: int, chunk_len: int,
                             io: torch.dtype) -> int:
    return int(lib().ssm_scan_workspace_bytes(batch, dim, seqlen, dstate, chunk_len, _DTYPE_CODE[io]))


def ssm_selective_scan_fwd(x: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                           C: torch.Tensor, D: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
                           delta_bias: Optional[torch.Tensor] = None, delta_softplus: bool = True,
                           conv_w: Optional[torch.Tensor] = None, conv_b: Optional[torch.Tensor] = None,
                           conv_init: Optional[torch.Tensor] = None, h0: Optional[torch.Tensor] = None,
                           return_last_state: bool = True, return_conv_state: bool = False,
                           d_conv: Optional[int] = None, chunk_len: int = 0,
                           workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                           h_last: Optional[torch.Tensor] = None,
                           conv_state_out: Optional[torch.Tensor] = None,
                           reverse: bool = False, zoh: bool = False,
                           s4d_real: bool = False) -> Tuple[torch.Tensor, ...]:
    """Selective scan forward. Returns (out, h_last) [+ conv_state_out when asked].

    x, delta, z: [batch, dim, L]; B, C: [batch, dstate, L] (all float32 or bfloat16, one dtype);
    A [dim, dstate], D / delta_bias / conv_b [dim], conv_w [dim, K], h0 [batch, dim, dstate]: float32.
    The workspace (if the chosen chunking needs one) is allocated here unless passed in.
    reverse: the backward scan (SSM_SCAN_REVERSE), the recurrence runs from t = L-1 to 0.
    zoh: zero-order-hold input term expm1(Delta A)/A B u (SSM_SCAN_ZOH) instead of Delta B u.
    s4d_real: the opt-in S4D-real path (SSM_SCAN_S4D_REAL): where A[d,n] = (n+1) A[d,0], Abar_n is
    taken as Abar_0^(n+1); checked per CTA, other A takes the generic path.
    """
    batch, dim, L = x.shape
    N = A.shape[1]
    dev, io = x.device, x.dtype
    K = conv_w.shape[1] if conv_w is not None else (d_conv or 0)
    _need(x, "x", (batch, dim, L), io, dev)
    _need(delta, "delta", (batch, dim, L), io, dev)
    _need(A, "A", (dim, N), torch.float32, dev)
    _need(B, "B", (batch, N, L), io, dev)
    _need(C, "C", (batch, N, L), io, dev)
    _need(D, "D", (dim,), torch.float32, dev, optional=True)
    _need(z, "z", (batch, dim, L), io, dev, optional=True)
    _need(delta_bias, "delta_bias", (dim,), torch.float32, dev, optional=True)
    if conv_w is not None:
        _need(conv_w, "conv_w", (dim, K), torch.float32, dev)
    _need(conv_b, "conv_b", (dim,), torch.float32, dev, optional=True)
    _need(conv_init, "conv_init", (batch, dim, K - 1), io, dev, optional=True)
    _need(h0, "h0", (batch, dim, N), torch.float32, dev, optional=True)
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", (batch, dim, L), io, dev)
    if return_last_state and h_last is None:
        h_last = torch.empty(batch, dim, N, dtype=torch.float32, device=dev)
    _need(h_last, "h_last", (batch, dim, N), torch.float32, dev, optional=True)
    if return_conv_state and conv_state_out is None:
        if K < 1:
            raise ValueError("return_conv_state needs a conv width (conv_w or d_conv)")
        conv_state_out = torch.empty(batch, dim, K - 1, dtype=io, device=dev)
    _need(conv_state_out, "conv_state_out", (batch, dim, K - 1), io, dev, optional=True)
    io_code = _io_code(x)
    need = ssm_scan_workspace_bytes(batch, dim, L, N, chunk_len, io)
    ws_bytes = 0
    if workspace is not None:
        ws_bytes = workspace.numel() * workspace.element_size()
    elif need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        ws_bytes = need
    st = lib().ssm_selective_scan_fwd(
        _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)),
        _ptr(conv_w), _ptr(conv_b), K, _ptr(conv_init), _ptr(h0), _ptr(out), _ptr(h_last), _ptr(conv_state_out),
        batch, dim, L, N, io_code, int(chunk_len), _ptr(workspace), ws_bytes,
        (SCAN_REVERSE if reverse else 0) | (SCAN_ZOH if zoh else 0) | (SCAN_S4D_REAL if s4d_real else 0),
        _stream(dev))
    _check("ssm_selective_scan_fwd", st)
    res = (out, h_last)
    if return_conv_state:
        res = res + (conv_state_out,)
    return res


def ssm_selective_scan_aggregate(x: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                                 delta_bias: Optional[torch.Tensor] = None, delta_softplus: bool = True,
                                 conv_w: Optional[torch.Tensor] = None, conv_b: Optional[torch.Tensor] = None,
                                 conv_init: Optional[torch.Tensor] = None, reverse: bool = False,
                                 zoh: bool = False) -> Tuple[torch.Tensor, torch.Tensor]:
    """Aggregate of one sequence segment: (S [batch, dim], h [batch, dim, dstate]), the sum of
    Delta over the segment and the state at its end from a zero state (include/ssm.h)."""
    batch, dim, L = x.shape
    N = A.shape[1]
    dev, io = x.device, x.dtype
    K = conv_w.shape[1] if conv_w is not None else 0
    _need(x, "x", (batch, dim, L), io, dev)
    _need(delta, "delta", (batch, dim, L), io, dev)
    _need(A, "A", (dim, N), torch.float32, dev)
    _need(B, "B", (batch, N, L), io, dev)
    _need(delta_bias, "delta_bias", (dim,), torch.float32, dev, optional=True)
    if conv_w is not None:
        _need(conv_w, "conv_w", (dim, K), torch.float32, dev)
    _need(conv_b, "conv_b", (dim,), torch.float32, dev, optional=True)
    _need(conv_init, "conv_init", (batch, dim, K - 1), io, dev, optional=True)
    S = torch.empty(batch, dim, dtype=torch.float32, device=dev)
    h = torch.empty(batch, dim, N, dtype=torch.float32, device=dev)
    need = int(lib().ssm_scan_aggregate_workspace_bytes(batch, dim, L, N, _io_code(x)))
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    st = lib().ssm_selective_scan_aggregate(
        _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(delta_bias), int(bool(delta_softplus)), _ptr(conv_w),
        _ptr(conv_b), K, _ptr(conv_init), _ptr(S), _ptr(h), batch, dim, L, N, _io_code(x), _ptr(ws), need,
        (SCAN_REVERSE if reverse else 0) | (SCAN_ZOH if zoh else 0), _stream(dev))
    _check("ssm_selective_scan_aggregate", st)
    return S, h


def ssm_scan_compose(S: torch.Tensor, b: torch.Tensor, A: torch.Tensor,
                     h0: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The state after segments with aggregates S [nseg, batch, dim], b [nseg, batch, dim, dstate]
    (in order), starting from h0 [batch, dim, dstate] (zeros when None)."""
    nseg, batch, dim = S.shape
    N = A.shape[1]
    dev = A.device
    _need(S, "S", (nseg, batch, dim), torch.float32, dev)
    _need(b, "b", (nseg, batch, dim, N), torch.float32, dev)
    _need(h0, "h0", (batch, dim, N), torch.float32, dev, optional=True)
    h = torch.empty(batch, dim, N, dtype=torch.float32, device=dev)
    _check("ssm_scan_compose", lib().ssm_scan_compose(_ptr(S), _ptr(b), _ptr(A), _ptr(h0), _ptr(h), nseg, batch, dim,
                                                      N, _stream(dev)))
    return h


def ssm_ssd_workspace_bytes(batch: int, seqlen: int, nheads: int, headdim: int, dstate: int, io) -> int:
    return int(lib().ssm_ssd_workspace_bytes(batch, seqlen, nheads, headdim, dstate, _DTYPE_CODE[io]))


def ssm_ssd_fwd(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, B: torch.Tensor, C: torch.Tensor,
                D: Optional[torch.Tensor] = None, dt_bias: Optional[torch.Tensor] = None, dt_softplus: bool = True,
                h0: Optional[torch.Tensor] = None, return_last_state: bool = True,
                workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                h_last: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Multi-head SSM with one decay per head (the state-space-duality layer). Returns (y, h_last).

    x [batch, L, nheads, headdim], dt [batch, L, nheads], B, C [batch, L, dstate] (bfloat16);
    A, D, dt_bias [nheads] and h0 [batch, nheads, headdim, dstate] float32. headdim 64, dstate 128.
    The workspace is allocated here unless passed in."""
    batch, L, H, P = x.shape
    N = B.shape[2]
    dev, io = x.device, x.dtype
    _need(x, "x", (batch, L, H, P), io, dev)
    _need(dt, "dt", (batch, L, H), io, dev)
    _need(A, "A", (H,), torch.float32, dev)
    _need(B, "B", (batch, L, N), io, dev)
    _need(C, "C", (batch, L, N), io, dev)
    _need(D, "D", (H,), torch.float32, dev, optional=True)
    _need(dt_bias, "dt_bias", (H,), torch.float32, dev, optional=True)
    _need(h0, "h0", (batch, H, P, N), torch.float32, dev, optional=True)
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", (batch, L, H, P), io, dev)
    if return_last_state and h_last is None:
        h_last = torch.empty(batch, H, P, N, dtype=torch.float32, device=dev)
    _need(h_last, "h_last", (batch, H, P, N), torch.float32, dev, optional=True)
    need = ssm_ssd_workspace_bytes(batch, L, H, P, N, io)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    st = lib().ssm_ssd_fwd(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(dt_bias),
                           int(bool(dt_softplus)), _ptr(h0), _ptr(out), _ptr(h_last), batch, L, H, P, N,
                           _io_code(x), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(dev))
    _check("ssm_ssd_fwd", st)
    return out, h_last


def ssm_scan_bwd_workspace_bytes(batch: int, dim: int, seqlen: int, dstate: int, io) -> int:
    return int(lib().ssm_scan_bwd_workspace_bytes(batch, dim, seqlen, dstate, _DTYPE_CODE[io]))


def ssm_selective_scan_bwd(u: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                           C: torch.Tensor, dout: torch.Tensor, D: Optional[torch.Tensor] = None,
                           z: Optional[torch.Tensor] = None, delta_bias: Optional[torch.Tensor] = None,
                           delta_softplus: bool = True, h0: Optional[torch.Tensor] = None,
                           dh_last: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None, grads: Optional[dict] = None) -> dict:
    """Backward pass of the forward-time Euler scan with u given directly. Returns a dict with
    du, ddelta, dz (None without z) in the io dtype and dA, dB, dC, dD, ddelta_bias, dh0 in
    float32 (dD / ddelta_bias None when D / delta_bias are None). ``grads``: a dict of the same
    keys to write into instead of allocating (a previous call's result)."""
    batch, dim, L = u.shape
    N = A.shape[1]
    dev, io = u.device, u.dtype
    for t, name, shape, dt in ((u, "u", (batch, dim, L), io), (delta, "delta", (batch, dim, L), io),
                               (A, "A", (dim, N), torch.float32), (B, "B", (batch, N, L), io),
                               (C, "C", (batch, N, L), io), (dout, "dout", (batch, dim, L), io)):
        _need(t, name, shape, dt, dev)
    _need(D, "D", (dim,), torch.float32, dev, optional=True)
    _need(z, "z", (batch, dim, L), io, dev, optional=True)
    _need(delta_bias, "delta_bias", (dim,), torch.float32, dev, optional=True)
    _need(h0, "h0", (batch, dim, N), torch.float32, dev, optional=True)
    _need(dh_last, "dh_last", (batch, dim, N), torch.float32, dev, optional=True)
    f32 = dict(dtype=torch.float32, device=dev)
    g = grads if grads is not None else {"du": torch.empty_like(u), "ddelta": torch.empty_like(u), "dz": torch.empty_like(u) if z is not None else None,
         "dA": torch.empty(dim, N, **f32), "dB": torch.empty(batch, N, L, **f32), "dC": torch.empty(batch, N, L, **f32),
         "dD": torch.empty(dim, **f32) if D is not None else None,
         "ddelta_bias": torch.empty(dim, **f32) if delta_bias is not None else None,
         "dh0": torch.empty(batch, dim, N, **f32)}
    for name, shape, dt in (("du", (batch, dim, L), io), ("ddelta", (batch, dim, L), io),
                            ("dA", (dim, N), torch.float32), ("dB", (batch, N, L), torch.float32),
                            ("dC", (batch, N, L), torch.float32), ("dh0", (batch, dim, N), torch.float32)):
        _need(g[name], name, shape, dt, dev)
    _need(g["dz"], "dz", (batch, dim, L), io, dev, optional=z is None)
    need = ssm_scan_bwd_workspace_bytes(batch, dim, L, N, io)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().ssm_selective_scan_bwd(
        _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)),
        _ptr(h0), _ptr(dout), _ptr(dh_last), _ptr(g["du"]), _ptr(g["ddelta"]), _ptr(g["dz"]), _ptr(g["dA"]),
        _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]), _ptr(g["ddelta_bias"]), _ptr(g["dh0"]),
        batch, dim, L, N, _io_code(u), _ptr(workspace), ws_bytes, 0, _stream(dev))
    _check("ssm_selective_scan_bwd", st)
    return g


def ssm_selective_state_update(state: torch.Tensor, conv_state: Optional[torch.Tensor], x: torch.Tensor,
                               delta: torch.Tensor, A: torch.Tensor, B: torch.Tensor, C: torch.Tensor,
                               D: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
                               delta_bias: Optional[torch.Tensor] = None, delta_softplus: bool = True,
                               conv_w: Optional[torch.Tensor] = None, conv_b: Optional[torch.Tensor] = None,
                               y: Optional[torch.Tensor] = None, zoh: bool = False) -> torch.Tensor:
    """One decode step; updates ``state`` [batch, dim, N] f32 and ``conv_state`` [batch, dim, K-1] in place.

    x, delta, z: [batch, dim]; B, C: [batch, N]. Returns y [batch, dim].
    """
    batch, dim = x.shape
    N = A.shape[1]
    dev, io = x.device, x.dtype
    K = conv_w.shape[1] if conv_w is not None else 0
    _need(state, "state", (batch, dim, N), torch.float32, dev)
    if conv_w is not None:
        _need(conv_w, "conv_w", (dim, K), torch.float32, dev)
        _need(conv_state, "conv_state", (batch, dim, K - 1), io, dev, optional=(K == 1))
    _need(x, "x", (batch, dim), io, dev)
    _need(delta, "delta", (batch, dim), io, dev)
    _need(A, "A", (dim, N), torch.float32, dev)
    _need(B, "B", (batch, N), io, dev)
    _need(C, "C", (batch, N), io, dev)
    _need(D, "D", (dim,), torch.float32, dev, optional=True)
    _need(z, "z", (batch, dim), io, dev, optional=True)
    _need(delta_bias, "delta_bias", (dim,), torch.float32, dev, optional=True)
    _need(conv_b, "conv_b", (dim,), torch.float32, dev, optional=True)
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", (batch, dim), io, dev)
    st = lib().ssm_selective_state_update(
        _ptr(state), _ptr(conv_state if conv_w is not None else None), _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
        _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)), _ptr(conv_w), _ptr(conv_b), K, _ptr(y),
        batch, dim, N, _io_code(x), SCAN_ZOH if zoh else 0, _stream(dev))
    _check("ssm_selective_state_update", st)
    return y

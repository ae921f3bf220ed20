"""Shared helpers of the GPU tests: tolerances, moving seeded inputs to the device, running
the CUDA path through the binding and the fp64 oracle on the same inputs (whole problems or
sampled channels)."""

from __future__ import annotations

import numpy as np
import torch

import oracle

# Elementwise |gpu - oracle| <= ATOL + RTOL * |oracle| (allclose convention), by I/O dtype:
# fp32 I/O rtol 1e-4 / atol 1e-5; bf16 I/O with fp32 state rtol 2e-2 / atol 1e-2.
TOL = {"f32": (1e-4, 1e-5), "bf16": (2e-2, 1e-2)}
SCAN_KEYS = ("x", "delta", "z", "B", "C")


def io_of(t: torch.Tensor) -> str:
    return "bf16" if t.dtype == torch.bfloat16 else "f32"


_BLOCK = 1 << 24  # elements compared per pass, so that full-size tensors need no large temporaries


def assert_close(got, ref, io: str, what: str):
    """Every element: |got - ref| <= atol + rtol |ref|. got may be a (device) tensor of any float
    dtype or an array; ref is the fp64 oracle result. Large tensors are compared block by block."""
    rtol, atol = TOL[io]
    if hasattr(got, "detach"):
        got = got.detach()
        shape = tuple(got.shape)
        flat_got = got.reshape(-1)
        take = lambda s, e: flat_got[s:e].float().cpu().double().numpy()
    else:
        arr = np.asarray(got, np.float64)
        shape = arr.shape
        flat_np = arr.reshape(-1)
        take = lambda s, e: flat_np[s:e]
    ref = np.asarray(ref, dtype=np.float64)
    assert shape == ref.shape, (what, shape, ref.shape)
    flat_ref = ref.reshape(-1)
    nbad, first, max_err = 0, None, 0.0
    for s in range(0, flat_ref.size, _BLOCK):
        e = min(flat_ref.size, s + _BLOCK)
        g, r = take(s, e), flat_ref[s:e]
        assert np.all(np.isfinite(g)), f"{what}: non-finite values"
        err = np.abs(g - r)
        max_err = max(max_err, float(err.max(initial=0.0)))
        bad = err > atol + rtol * np.abs(r)
        if bad.any():
            nbad += int(bad.sum())
            if first is None:
                j = int(np.argmax(bad))
                first = (np.unravel_index(s + j, shape), g[j], r[j])
    if nbad:
        i, gv, rv = first
        raise AssertionError(f"{what}: {nbad}/{flat_ref.size} outside rtol={rtol} atol={atol}; first at "
                             f"{tuple(int(v) for v in i)}: gpu={gv!r} oracle={rv!r}; max abs err {max_err:.3e}")


def to_dev(p: dict, dev) -> dict:
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in p.items()}


def gpu_scan(g: dict, chunk_len: int = 0, use_conv: bool = True, use_h0: bool = True, use_init: bool = True,
             return_conv_state: bool = False, delta_softplus: bool = True, **kw):
    import selective_state_space_145_b300 as ssm

    conv_w = g.get("conv_w") if use_conv else None
    return ssm.ssm_selective_scan_fwd(
        g["x"], g["delta"], g["A"], g["B"], g["C"], g.get("D"), g.get("z"), g.get("delta_bias"), delta_softplus,
        conv_w, g.get("conv_b") if use_conv else None, g.get("conv_init") if (use_conv and use_init) else None,
        g.get("h0") if use_h0 else None, return_conv_state=return_conv_state, chunk_len=chunk_len, **kw)


def oracle_scan(p: dict, use_conv: bool = True, use_h0: bool = True, use_init: bool = True,
                want_conv_state: bool = False, delta_softplus: bool = True, nthreads: int = 0,
                reverse: bool = False, zoh: bool = False):
    nthreads = nthreads or oracle.oracle.default_threads()
    return oracle.selective_scan(
        p["x"], p["delta"], p["A"], p["B"], p["C"], p.get("D"), p.get("z"), p.get("delta_bias"), delta_softplus,
        p.get("conv_w") if use_conv else None, p.get("conv_b") if use_conv else None,
        p.get("conv_init") if (use_conv and use_init) else None, p.get("h0") if use_h0 else None,
        want_conv_state=want_conv_state, nthreads=nthreads, reverse=reverse, zoh=zoh)


def channel_slice(p: dict, b: int, d: int) -> dict:
    """The inputs of one (b, d) channel as a batch-1, dim-1 problem."""
    q = {}
    for k, v in p.items():
        if v is None:
            q[k] = None
        elif k in ("x", "delta", "z", "h0", "conv_init"):
            q[k] = v[b:b + 1, d:d + 1]
        elif k in ("B", "C"):
            q[k] = v[b:b + 1]
        elif k in ("A", "D", "delta_bias", "conv_w", "conv_b"):
            q[k] = v[d:d + 1]
        else:
            q[k] = v
    return q


def sample_channels(batch: int, dim: int, n: int, seed: int):
    rng = np.random.default_rng(seed)
    flat = rng.choice(batch * dim, size=min(n, batch * dim), replace=False)
    return [(int(f // dim), int(f % dim)) for f in flat]

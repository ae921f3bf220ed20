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


def assert_close(got, ref, io: str, what: str):
    rtol, atol = TOL[io]
    got = got.detach().float().cpu().double().numpy() if hasattr(got, "detach") else np.asarray(got, np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside rtol={rtol} atol={atol}; first at {i}: "
                             f"gpu={got[i]!r} oracle={ref[i]!r}; max abs err {err.max():.3e}")


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

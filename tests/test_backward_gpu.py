"""GPU parity of the scan's backward pass (ssm_selective_scan_bwd) against the fp64 oracle's
adjoint, gradient by gradient, on seeded problems that span several channel tiles, several
16-step tiles, ragged tails and the optional terms.

Every element of every gradient is held to the scan's own per-element bounds,
|gpu - oracle| <= rtol |oracle| + atol: fp32 I/O rtol 1e-4 / atol 1e-5, bf16 I/O (du, ddelta, dz
rounded to bf16) rtol 2e-2 / atol 1e-2. With SSM_GRAD_REPORT set to a file path, each comparison
appends one JSON line with the largest ratio err / (rtol |oracle| + atol), and the same ratio
with atol scaled by the tensor's largest magnitude (the looser criterion sums with
cancellation would otherwise need).
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from selective_state_space_145_b300 import inputs
from ssm_testutil import TOL, to_dev

pytestmark = pytest.mark.gpu

GRADS = ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0")


def _assert_grad(got, ref, io, what):
    rtol, atol = TOL[io]
    got = got.detach().float().cpu().double().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    scale = max(float(np.abs(ref).max()) if ref.size else 0.0, 1e-30)
    err = np.abs(got - ref)
    _report(what, io, err, ref, rtol, atol, scale)
    bad = err > rtol * np.abs(ref) + atol
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside; first at {i}: gpu={got[i]!r} "
                             f"oracle={ref[i]!r}; max err {err.max():.3e}")


def _report(what, io, err, ref, rtol, atol, scale):
    """Per-element figures against rtol |ref| + atol, appended to $SSM_GRAD_REPORT if set."""
    path = os.environ.get("SSM_GRAD_REPORT")
    if not path or err.size == 0:
        return
    ratio = err / (rtol * np.abs(ref) + atol)
    rec = {"grad": what, "io": io, "n": int(err.size), "within_elem": float(np.mean(ratio <= 1.0)),
           "max_ratio_elem": float(ratio.max()), "max_err": float(err.max()), "scale": scale,
           "max_ratio_scaled": float((err / (rtol * np.abs(ref) + atol * scale)).max())}
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")


def _problem(batch, dim, L, N, io, seed, with_z=True, with_D=True, with_bias=True, with_h0=True):
    p = inputs.scan_inputs(batch, dim, L, N, 0, io, seed=seed, with_h0=with_h0, with_z=with_z, with_D=with_D,
                           random_A=True)
    if not with_bias:
        p["delta_bias"] = None
    g = torch.Generator().manual_seed(seed + 1)
    dout = torch.randn(batch, dim, L, generator=g).to(p["x"].dtype)
    dhl = torch.randn(batch, dim, N, generator=g)
    return p, dout, dhl


CASES = [
    # batch, dim, L, N, io, z, D, bias, h0, dh_last
    (2, 37, 50, 16, "f32", True, True, True, True, True),     # ragged tile, partial channel tile
    (1, 64, 96, 7, "f32", False, False, False, False, False),  # options off, N < 16
    (2, 70, 129, 16, "bf16", True, True, True, True, True),   # 3 channel tiles, ragged
    (3, 5, 1, 16, "f32", True, True, True, True, True),       # L = 1
    (2, 40, 100, 16, "f32", True, True, True, True, True),    # vector path, last tile of 4 steps
    (1, 33, 704, 5, "bf16", True, False, True, True, True),   # vector path, chunks, N < 16
    (2, 64, 264, 16, "bf16", False, True, False, False, True),  # vector path, no gate / bias / h0
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}_d{}_l{}_n{}_{}_z{}_D{}_bias{}_h0{}_dh{}".format(*c))
def test_backward_matches_oracle(cuda_device, case):
    import selective_state_space_145_b300 as ssm

    batch, dim, L, N, io, wz, wD, wb, wh, wdh = case
    p, dout, dhl = _problem(batch, dim, L, N, io, seed=7000 + dim + L, with_z=wz, with_D=wD, with_bias=wb,
                            with_h0=wh)
    g = to_dev(p, cuda_device)
    got = ssm.ssm_selective_scan_bwd(g["x"], g["delta"], g["A"], g["B"], g["C"], dout.to(cuda_device), g.get("D"),
                                     g.get("z"), g.get("delta_bias"), True, g.get("h0"),
                                     dhl.to(cuda_device) if wdh else None)
    ref = oracle.selective_scan_bwd(p["x"], p["delta"], p["A"], p["B"], p["C"], dout, p.get("D"), p.get("z"),
                                    p.get("delta_bias"), True, p.get("h0"), dhl if wdh else None,
                                    nthreads=oracle.oracle.default_threads())
    for k in GRADS:
        if ref[k] is None:
            assert got[k] is None, k
            continue
        _assert_grad(got[k], ref[k], io, k)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_backward_chunked_long(cuda_device, io):
    """Few channels and a long sequence: the backward pass cuts time into chunks (forward carries
    for the chunk-start states, adjoint carries for the chunk-end adjoints)."""
    import selective_state_space_145_b300 as ssm

    p, dout, dhl = _problem(2, 48, 700, 16, io, seed=77)
    g = to_dev(p, cuda_device)
    got = ssm.ssm_selective_scan_bwd(g["x"], g["delta"], g["A"], g["B"], g["C"], dout.to(cuda_device), g["D"], g["z"],
                                     g["delta_bias"], True, g["h0"], dhl.to(cuda_device))
    ref = oracle.selective_scan_bwd(p["x"], p["delta"], p["A"], p["B"], p["C"], dout, p["D"], p["z"],
                                    p["delta_bias"], True, p["h0"], dhl, nthreads=oracle.oracle.default_threads())
    for k in GRADS:
        _assert_grad(got[k], ref[k], io, k)


def test_backward_softplus_off_and_deterministic(cuda_device):
    import selective_state_space_145_b300 as ssm

    p, dout, dhl = _problem(2, 40, 64, 16, "f32", seed=71)
    # softplus off: Delta = delta + bias must stay positive for a decaying recurrence
    p["delta"] = (p["delta"].abs() * 0.2 + 0.01)
    p["delta_bias"] = torch.full_like(p["delta_bias"], 0.01)
    g = to_dev(p, cuda_device)
    args = (g["x"], g["delta"], g["A"], g["B"], g["C"], dout.to(cuda_device), g["D"], g["z"], g["delta_bias"], False,
            g["h0"], dhl.to(cuda_device))
    a1 = ssm.ssm_selective_scan_bwd(*args)
    a2 = ssm.ssm_selective_scan_bwd(*args)
    ref = oracle.selective_scan_bwd(p["x"], p["delta"], p["A"], p["B"], p["C"], dout, p["D"], p["z"],
                                    p["delta_bias"], False, p["h0"], dhl)
    for k in GRADS:
        _assert_grad(a1[k], ref[k], "f32", k)
        assert torch.equal(a1[k], a2[k]), f"{k} not deterministic"


def test_backward_empty_sequence(cuda_device):
    """L = 0: no per-token gradients; dh0 = dh_last and the parameter gradients are zero."""
    import selective_state_space_145_b300 as ssm

    p, dout, dhl = _problem(2, 8, 0, 16, "f32", seed=5)
    g = to_dev(p, cuda_device)
    got = ssm.ssm_selective_scan_bwd(g["x"], g["delta"], g["A"], g["B"], g["C"], dout.to(cuda_device), g["D"], g["z"],
                                     g["delta_bias"], True, g["h0"], dhl.to(cuda_device))
    torch.cuda.synchronize()
    assert torch.equal(got["dh0"].cpu(), dhl)
    assert float(got["dA"].abs().max()) == 0.0 and float(got["dD"].abs().max()) == 0.0


# ---------------------------------------------------------------- conv prologue backward

CONV_CASES = [
    # batch, dim, L, K, io, window, silu
    (2, 37, 1500, 4, "f32", True, True),     # two 1024-step segments, ragged
    (3, 20, 7, 3, "f32", True, False),       # short rows, no SiLU
    (2, 48, 2100, 4, "bf16", True, True),
    (1, 16, 2, 4, "f32", True, True),        # L < K-1: the window gradient from the first steps only
    (2, 9, 100, 1, "f32", False, True),      # K = 1: no window
    (1, 8, 0, 4, "f32", True, True),         # L = 0
]


@pytest.mark.parametrize("case", CONV_CASES, ids=lambda c: "b{}_d{}_l{}_k{}_{}_win{}_silu{}".format(*c))
def test_conv_backward_matches_oracle(cuda_device, case):
    import selective_state_space_145_b300 as ssm

    batch, dim, L, K, io, wwin, act = case
    gen = torch.Generator().manual_seed(900 + dim + L)
    dt = torch.bfloat16 if io == "bf16" else torch.float32
    x = torch.randn(batch, dim, L, generator=gen).to(dt)
    dout = torch.randn(batch, dim, L, generator=gen).to(dt)
    w = torch.rand(dim, K, generator=gen) - 0.5
    bias = torch.randn(dim, generator=gen)
    win = torch.randn(batch, dim, K - 1, generator=gen).to(dt) if (wwin and K > 1) else None
    got = ssm.ssm_causal_conv1d_bwd(x.to(cuda_device), w.to(cuda_device), dout.to(cuda_device), bias.to(cuda_device),
                                    win.to(cuda_device) if win is not None else None, apply_silu=act)
    ref = oracle.causal_conv1d_bwd(x, w, dout, bias, win, apply_silu=act)
    _assert_grad(got["dx"], ref["dx"], io, "dx")
    _assert_grad(got["dw"], ref["dw"], io, "dw")
    _assert_grad(got["dbias"], ref["dbias"], io, "dbias")
    if win is not None:
        _assert_grad(got["dconv_init"], ref["dwindow"], io, "dconv_init")


def test_block_backward_chain(cuda_device):
    """The fused block's gradient through this library: u = silu(conv(x)); scan backward on u
    gives du; the conv backward turns du into dx, dw, dbias. Checked against the oracle's
    two backward routines chained the same way."""
    import selective_state_space_145_b300 as ssm

    p = inputs.scan_inputs(2, 40, 300, 16, 4, "f32", seed=91, with_h0=True)
    gen = torch.Generator().manual_seed(92)
    dout = torch.randn(2, 40, 300, generator=gen)
    g = to_dev(p, cuda_device)
    u = ssm.ssm_causal_conv1d_fwd(g["x"], g["conv_w"], g["conv_b"])
    gs = ssm.ssm_selective_scan_bwd(u, g["delta"], g["A"], g["B"], g["C"], dout.to(cuda_device), g["D"], g["z"],
                                    g["delta_bias"], True, g["h0"], None)
    gc = ssm.ssm_causal_conv1d_bwd(g["x"], g["conv_w"], gs["du"], g["conv_b"])
    u_ref = oracle.causal_conv1d(p["x"], p["conv_w"], p["conv_b"])
    rs = oracle.selective_scan_bwd(u_ref, p["delta"], p["A"], p["B"], p["C"], dout, p["D"], p["z"], p["delta_bias"],
                                   True, p["h0"], None)
    rc = oracle.causal_conv1d_bwd(p["x"], p["conv_w"], rs["du"], p["conv_b"])
    _assert_grad(gc["dx"], rc["dx"], "f32", "dx")
    _assert_grad(gc["dw"], rc["dw"], "f32", "dconv_w")
    _assert_grad(gc["dbias"], rc["dbias"], "f32", "dconv_b")


@pytest.mark.parametrize("name", ["block_f32_b2_d1024_l1024_n16_k4", "block_bf16_b8_d2048_l2048_n16_k4",
                                  pytest.param("longscan_bf16_b1_d1536_l131072_n16", marks=pytest.mark.slow)])
def test_backward_workload_whole(cuda_device, name):
    """The backward pass on a block workload at full size, in the benchmark's configuration (x
    taken as the scan input u, the same seeded dout and dh_last): every element of every gradient
    against the fp64 adjoint at the per-element bounds."""
    import selective_state_space_145_b300 as ssm

    w = inputs.WORKLOADS[name]
    # the fp64 adjoint of the long scan holds about 11 GB of arrays on the host
    host_bytes = os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES")
    if w.batch * w.dim * w.seqlen > 1 << 28 and host_bytes < 32 << 30:
        pytest.skip("host memory below 32 GB for the fp64 adjoint of this workload")
    p = inputs.workload_inputs(w)
    gen = torch.Generator().manual_seed(w.seed + 7)
    dout = torch.randn(w.batch, w.dim, w.seqlen, generator=gen).to(p["x"].dtype)
    dhl = torch.randn(w.batch, w.dim, w.dstate, generator=gen)
    g = to_dev(p, cuda_device)
    got = ssm.ssm_selective_scan_bwd(g["x"], g["delta"], g["A"], g["B"], g["C"], dout.to(cuda_device), g["D"], g["z"],
                                     g["delta_bias"], True, g["h0"], dhl.to(cuda_device))
    got = {k: (v.cpu() if v is not None else None) for k, v in got.items()}
    del g
    torch.cuda.synchronize()
    ref = oracle.selective_scan_bwd(p["x"], p["delta"], p["A"], p["B"], p["C"], dout, p["D"], p["z"],
                                    p["delta_bias"], True, p["h0"], dhl, nthreads=oracle.oracle.default_threads())
    for k in GRADS:
        if ref[k] is None:
            assert got[k] is None, k
            continue
        _assert_grad(got[k], ref[k], w.io, k)
        ref[k] = None


@pytest.mark.parametrize("name", ["block_f32_b2_d1024_l1024_n16_k4", "block_bf16_b8_d2048_l2048_n16_k4"])
def test_conv_backward_workload_whole(cuda_device, name):
    """The conv prologue's backward on a block workload at full size (the workload's x, conv
    weights and window, a seeded dout): every element of dx, dconv_w, dconv_b and the window
    gradient against the oracle at the per-element bounds."""
    import selective_state_space_145_b300 as ssm

    w = inputs.WORKLOADS[name]
    p = inputs.workload_inputs(w)
    gen = torch.Generator().manual_seed(w.seed + 9)
    dout = torch.randn(w.batch, w.dim, w.seqlen, generator=gen).to(p["x"].dtype)
    win = p.get("conv_init")
    got = ssm.ssm_causal_conv1d_bwd(p["x"].to(cuda_device), p["conv_w"].to(cuda_device), dout.to(cuda_device),
                                    p["conv_b"].to(cuda_device), win.to(cuda_device) if win is not None else None)
    ref = oracle.causal_conv1d_bwd(p["x"], p["conv_w"], dout, p["conv_b"], win,
                                   nthreads=oracle.oracle.default_threads())
    _assert_grad(got["dx"], ref["dx"], w.io, "dx")
    _assert_grad(got["dw"], ref["dw"], w.io, "dconv_w")
    _assert_grad(got["dbias"], ref["dbias"], w.io, "dconv_b")
    if win is not None:
        _assert_grad(got["dconv_init"], ref["dwindow"], w.io, "dconv_init")

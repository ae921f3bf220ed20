"""GPU parity of the multi-head SSM with one decay per head (the state-space-duality layer, run on
the tcgen05 tensor cores), called through the C ABI, against the fp64 oracle on the same seeded
inputs: whole small problems (one chunk, several chunks, a ragged last chunk, one step, with and
without an initial state or softplus) and every head of the full-size workload. Tolerance is
the bf16-I/O bound: |gpu - oracle| <= 1e-2 + 2e-2 |oracle| on y and on the final state.
"""

import os

import numpy as np
import pytest
import torch

import oracle
from selective_state_space_145_b300 import inputs
from ssm_testutil import assert_close

pytestmark = pytest.mark.gpu


def _ssm():
    import selective_state_space_145_b300 as ssm

    return ssm


def _dev(p, dev):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in p.items()}


def _run(g, softplus=True, workspace=None):
    ssm = _ssm()
    batch, L, H, P = g["x"].shape
    N = g["B"].shape[2]
    if workspace is None:
        workspace = torch.zeros(max(1, ssm.ssm_ssd_workspace_bytes(batch, L, H, P, N, torch.bfloat16)),
                                dtype=torch.uint8, device=g["x"].device)
    y, hl = ssm.ssm_ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["dt_bias"], softplus, g["h0"],
                            workspace=workspace)
    torch.cuda.synchronize()
    if L > 0:
        assert int(workspace[:4].view(torch.int32).item()) == 0, "tensor-core wait ran out"
    return y, hl


CASES = [
    # batch, L, heads, with_h0
    (1, 128, 2, False),     # exactly one chunk
    (2, 300, 3, True),      # three chunks, ragged last chunk, initial state
    (1, 1, 1, True),        # one step
    (2, 1000, 2, False),    # eight chunks, ragged
    (3, 256, 5, True),      # two full chunks, odd head count
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}_l{}_h{}_h0{}".format(*c))
def test_ssd_matches_oracle(cuda_device, case):
    batch, L, H, with_h0 = case
    p = inputs.ssd_inputs(batch, L, H, seed=11 + L + H, with_h0=with_h0)
    y, hl = _run(_dev(p, cuda_device))
    ref, ref_h = oracle.ssd(p["x"], p["dt"], p["A"], p["B"], p["C"], p["D"], p["dt_bias"], True, p["h0"],
                            nthreads=oracle.oracle.default_threads())
    assert_close(y, ref, "bf16", "y")
    assert_close(hl, ref_h, "bf16", "h_last")


def test_ssd_softplus_off_and_no_skip(cuda_device):
    p = inputs.ssd_inputs(2, 260, 2, seed=5, with_h0=True, with_D=False)
    p["dt"] = (p["dt"].float().abs() * 0.05).to(torch.bfloat16)
    p["dt_bias"] = torch.full((2,), 0.01)
    y, hl = _run(_dev(p, cuda_device), softplus=False)
    ref, ref_h = oracle.ssd(p["x"], p["dt"], p["A"], p["B"], p["C"], None, p["dt_bias"], False, p["h0"])
    assert_close(y, ref, "bf16", "y")
    assert_close(hl, ref_h, "bf16", "h_last")


def test_ssd_without_bias_and_skip_pointers(cuda_device):
    """dt_bias and D absent (NULL at the ABI): the step is softplus(dt) and there is no skip term."""
    p = inputs.ssd_inputs(1, 256, 3, seed=17, with_h0=False, with_D=False)
    p["dt"] = (p["dt"].float() - 3.0).to(torch.bfloat16)   # softplus(dt) of the order of the workloads' steps
    p["dt_bias"] = None
    y, hl = _run(_dev(p, cuda_device))
    ref, ref_h = oracle.ssd(p["x"], p["dt"], p["A"], p["B"], p["C"], None, None, True, None)
    assert_close(y, ref, "bf16", "y")
    assert_close(hl, ref_h, "bf16", "h_last")


def test_ssd_deterministic_and_two_calls(cuda_device):
    p = inputs.ssd_inputs(2, 512, 2, seed=8, with_h0=True)
    g = _dev(p, cuda_device)
    y1, h1 = _run(g)
    y2, h2 = _run(g)
    assert torch.equal(y1, y2) and torch.equal(h1, h2)
    # two calls passing the state equal one call (the state is fp32 between calls)
    L1 = 200
    cut = lambda sl: {k: (v[:, sl].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in g.items()}
    ya, ha = _run(cut(slice(0, L1)))
    gb = cut(slice(L1, None))
    gb["h0"] = ha
    yb, hb = _run(gb)
    assert_close(torch.cat([ya, yb], dim=1), y1.float().cpu().double().numpy(), "bf16", "two calls")
    assert_close(hb, h1.cpu().double().numpy(), "bf16", "state after two calls")


def test_ssd_bounded_wait_reports_status(cuda_device):
    """Failure detection without a fault: with the SSM_TEST_SSD_SKIP_MMA hook no GEMM is issued,
    the kernel's wait for it runs out, it records status 1, frees its tensor memory and returns;
    the context stays usable and the next call is correct."""
    import time

    ssm = _ssm()
    p = inputs.ssd_inputs(1, 256, 1, seed=3)
    g = _dev(p, cuda_device)
    ws = torch.zeros(256, dtype=torch.uint8, device=cuda_device)
    ssm.lib().ssm_set_test_hooks(1)
    try:
        t0 = time.time()
        ssm.ssm_ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["dt_bias"], True, None, workspace=ws)
        torch.cuda.synchronize()
        waited = time.time() - t0
    finally:
        ssm.lib().ssm_set_test_hooks(0)
    assert int(ws[:4].view(torch.int32).item()) == 1
    assert waited < 30.0
    y, hl = _run(g)   # also checks that the status word is back to 0
    ref, ref_h = oracle.ssd(p["x"], p["dt"], p["A"], p["B"], p["C"], p["D"], p["dt_bias"], True, None)
    assert_close(y, ref, "bf16", "y after the timed-out call")
    assert_close(hl, ref_h, "bf16", "h_last after the timed-out call")


def test_ssd_empty(cuda_device):
    ssm = _ssm()
    p = _dev(inputs.ssd_inputs(2, 0, 3, seed=1, with_h0=True), cuda_device)
    y, hl = ssm.ssm_ssd_fwd(p["x"], p["dt"], p["A"], p["B"], p["C"], p["D"], p["dt_bias"], True, p["h0"])
    torch.cuda.synchronize()
    assert y.numel() == 0 and torch.equal(hl, p["h0"])
    p["h0"] = None
    y, hl = ssm.ssm_ssd_fwd(p["x"], p["dt"], p["A"], p["B"], p["C"], p["D"], p["dt_bias"], True, None)
    torch.cuda.synchronize()
    assert torch.count_nonzero(hl) == 0


def test_ssd_workload_every_head(cuda_device):
    """The full-size workload in the benchmark's launch configuration, every output and every
    final state against the oracle (4.3e9 state updates: well under a second on the host's
    cores)."""
    w = inputs.SSD_WORKLOADS["ssd_bf16_b8_l2048_h32_p64_n128"]
    p = inputs.ssd_workload_inputs(w)
    y, hl = _run(_dev(p, cuda_device))
    y, hl = y.cpu(), hl.cpu()
    ref, ref_h = oracle.ssd(p["x"], p["dt"], p["A"], p["B"], p["C"], p["D"], p["dt_bias"], True, None,
                            nthreads=os.cpu_count() or 1)
    assert_close(y, ref, "bf16", "y")
    assert_close(hl, ref_h, "bf16", "h_last")


def test_ssd_ragged_every_head(cuda_device):
    """The cp.async copy path (a sequence length that is not a multiple of the 128-step chunk)
    on a mid-size problem with an initial state: 16 chunks, a ragged last one, 32 heads; every
    output and every final state against the oracle."""
    p = inputs.ssd_inputs(2, 2000, 32, seed=2024, with_h0=True)
    y, hl = _run(_dev(p, cuda_device))
    ref, ref_h = oracle.ssd(p["x"], p["dt"], p["A"], p["B"], p["C"], p["D"], p["dt_bias"], True, p["h0"],
                            nthreads=os.cpu_count() or 1)
    assert_close(y.cpu(), ref, "bf16", "y")
    assert_close(hl.cpu(), ref_h, "bf16", "h_last")

"""The seeded input recipes (CPU): shapes, dtypes, determinism by seed and the stated
distributions, for the host draws and for the device draws used by the largest problems (drawn
here on the CPU device)."""

import math

import pytest
import torch

from selective_state_space_145_b300 import inputs


def _close(v, target, tol):
    assert abs(v - target) <= tol, (v, target)


def test_scan_recipe_moments_and_determinism():
    p = inputs.scan_inputs(2, 64, 512, 16, 4, "f32", seed=7, with_h0=True)
    q = inputs.scan_inputs(2, 64, 512, 16, 4, "f32", seed=7, with_h0=True)
    assert all(torch.equal(p[k], q[k]) for k in p if p[k] is not None)
    _close(p["x"].std().item(), 1.0, 0.02)
    _close(p["delta"].std().item(), 0.5, 0.01)
    _close(p["B"].mean().item(), 0.0, 0.02)
    assert torch.equal(p["A"], -torch.arange(1, 17, dtype=torch.float32).repeat(64, 1))
    dt = torch.nn.functional.softplus(p["delta_bias"].double())   # the bias is softplus^-1 of dt
    assert dt.min() >= 1e-3 * (1 - 1e-6) and dt.max() <= 0.1 * (1 + 1e-6)
    assert p["conv_w"].abs().max() <= 0.5 and torch.count_nonzero(p["conv_b"]) == 0


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_device_draws_keep_shapes_dtypes_and_distributions(io):
    dev = torch.device("cpu")
    p = inputs.scan_inputs_on(dev, 2, 32, 4096, 16, 4, io, seed=3)
    dt = inputs.IO_DTYPES[io]
    assert p["x"].shape == (2, 32, 4096) and p["x"].dtype == dt and p["B"].shape == (2, 16, 4096)
    assert p["A"].dtype == torch.float32 and p["conv_w"].shape == (32, 4)
    _close(p["x"].float().std().item(), 1.0, 0.02)
    _close(p["delta"].float().std().item(), 0.5, 0.01)
    q = inputs.scan_inputs_on(dev, 2, 32, 4096, 16, 4, io, seed=3)
    assert torch.equal(p["x"], q["x"]) and torch.equal(p["delta_bias"], q["delta_bias"])

    d = inputs.decode_inputs_on(dev, 64, 128, 16, 4, io, seed=4)
    assert d["state"].shape == (64, 128, 16) and d["state"].dtype == torch.float32
    assert d["conv_state"].shape == (64, 128, 3) and d["conv_state"].dtype == dt
    _close(d["state"].std().item(), 1.0, 0.02)

    s = inputs.ssd_inputs_on(dev, 2, 1024, 4, seed=5)
    assert s["x"].shape == (2, 1024, 4, 64) and s["B"].shape == (2, 1024, 128) and s["dt"].shape == (2, 1024, 4)
    assert s["x"].dtype == torch.bfloat16 and s["A"].dtype == torch.float32
    assert ((s["A"] <= -1.0) & (s["A"] >= -16.0)).all()
    _close(s["dt"].float().std().item(), 0.5, 0.02)


def test_ssd_recipe_matches_its_statement():
    p = inputs.ssd_inputs(2, 256, 8, seed=9, with_h0=True)
    assert p["h0"].shape == (2, 8, 64, 128)
    assert ((p["A"] <= -1.0) & (p["A"] >= -16.0)).all()
    dt0 = torch.nn.functional.softplus(p["dt_bias"].double())
    assert dt0.min() >= 1e-3 * (1 - 1e-6) and dt0.max() <= 0.1 * (1 + 1e-6)
    w = inputs.SSD_WORKLOADS["ssd_bf16_b8_l2048_h32_p64_n128"]
    assert w.updates == 8 * 2048 * 32 * 64 * 128 and w.d_model * w.expand == w.nheads * w.headdim
    assert math.isclose(inputs.WORKLOADS["block_bf16_b8_d2048_l2048_n16_k4"].dim, w.nheads * w.headdim)

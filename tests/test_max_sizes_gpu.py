"""GPU parity at the largest sizes: problems whose per-token tensors (or decode state) hold more
than 2^31 elements, so that every flat element index past 2^31 - 1 has to be formed in 64 bits.

The inputs are drawn on the device (same distributions as the host recipe, see
`inputs.scan_inputs_on` and its siblings); the oracle recomputes sampled channels or heads, which
are independent of the others, so each sampled slice is exact. The samples include the last
channels or heads, whose flat indices lie past 2^31, and the first ones. Tolerances are the
bf16-I/O bound of the other parity tests.
"""

import numpy as np
import pytest
import torch

import oracle
from selective_state_space_145_b300 import inputs
from ssm_testutil import assert_close

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

INT31 = 2 ** 31


def _ssm():
    import selective_state_space_145_b300 as ssm

    return ssm


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("chunk_len", [0, 4096], ids=["default_chunks", "chunks_4096"])
def test_scan_past_int32_indices(cuda_device, chunk_len):
    """bf16 prefill with the conv prologue and the gate, 8 x 8192 channels x 32800 steps: each of
    x, delta, z and out holds 2.15e9 elements. chunk_len 4096 adds nine chunks and their carries."""
    ssm = _ssm()
    batch, dim, L, N, K = 8, 8192, 32800, 16, 4
    assert batch * dim * L > INT31
    p = inputs.scan_inputs_on(cuda_device, batch, dim, L, N, K, "bf16", seed=2031)
    out, hl = ssm.ssm_selective_scan_fwd(p["x"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"],
                                         p["delta_bias"], True, p["conv_w"], p["conv_b"], None, None,
                                         chunk_len=chunk_len)
    torch.cuda.synchronize()
    # (b * dim + d) * L >= 2^31 for b = 7, d >= 8000
    chans = [(0, 0), (3, 4097), (7, 8000), (7, 8190), (7, 8191)]
    assert (chans[-1][0] * dim + chans[-1][1]) * L > INT31
    for b, d in chans:
        sl = lambda t: t[b:b + 1, d:d + 1].cpu()
        ref, ref_h = oracle.selective_scan(sl(p["x"]), sl(p["delta"]), p["A"][d:d + 1].cpu(), p["B"][b:b + 1].cpu(),
                                           p["C"][b:b + 1].cpu(), p["D"][d:d + 1].cpu(), sl(p["z"]),
                                           p["delta_bias"][d:d + 1].cpu(), True, p["conv_w"][d:d + 1].cpu(),
                                           p["conv_b"][d:d + 1].cpu())
        assert_close(out[b:b + 1, d:d + 1], ref, "bf16", f"out[{b},{d}]")
        assert_close(hl[b:b + 1, d:d + 1], ref_h, "bf16", f"h_last[{b},{d}]")
    del p, out, hl
    _free()


def test_decode_past_int32_indices(cuda_device):
    """One decode step of 4100 sequences x 32768 channels: the fp32 state [4100, 32768, 16] holds
    2.15e9 elements (8.6 GB), updated in place together with the conv window."""
    ssm = _ssm()
    batch, dim, N, K = 4100, 32768, 16, 4
    assert batch * dim * N > INT31
    p = inputs.decode_inputs_on(cuda_device, batch, dim, N, K, "bf16", seed=2032)
    # (b * dim + d) * N >= 2^31 for b >= 4096
    chans = [(0, 0), (2048, 100), (4096, 0), (4097, 5), (4099, 32767)]
    before = [(p["state"][b:b + 1, d:d + 1].cpu(), p["conv_state"][b:b + 1, d:d + 1].cpu()) for b, d in chans]
    y = ssm.ssm_selective_state_update(p["state"], p["conv_state"], p["x"], p["delta"], p["A"], p["B"], p["C"],
                                       p["D"], p["z"], p["delta_bias"], True, p["conv_w"], p["conv_b"])
    torch.cuda.synchronize()
    for (b, d), (st, win) in zip(chans, before):
        yr, st_r, win_r = oracle.state_update(st, win, p["x"][b:b + 1, d:d + 1].cpu(),
                                              p["delta"][b:b + 1, d:d + 1].cpu(), p["A"][d:d + 1].cpu(),
                                              p["B"][b:b + 1].cpu(), p["C"][b:b + 1].cpu(), p["D"][d:d + 1].cpu(),
                                              p["z"][b:b + 1, d:d + 1].cpu(), p["delta_bias"][d:d + 1].cpu(), True,
                                              p["conv_w"][d:d + 1].cpu(), p["conv_b"][d:d + 1].cpu())
        assert_close(y[b:b + 1, d:d + 1], yr, "bf16", f"y[{b},{d}]")
        assert_close(p["state"][b:b + 1, d:d + 1], st_r, "bf16", f"state[{b},{d}]")
        np.testing.assert_array_equal(p["conv_state"][b:b + 1, d:d + 1].float().cpu().numpy(), win_r)
    del p, y
    _free()


@pytest.mark.parametrize("L", [32896, 32900], ids=["tma_L32896", "ragged_L32900"])
def test_ssd_past_int32_indices(cuda_device, L):
    """State-space-duality layer, batch 16 x 64 heads of 64, state 128: x and y hold 2.16e9
    elements each. L = 32896 is a whole number of 128-step chunks (tensor-map copies); L = 32900
    ends in a ragged chunk (per-thread copies)."""
    ssm = _ssm()
    batch, H, P, N = 16, 64, 64, 128
    assert batch * L * H * P > INT31
    p = inputs.ssd_inputs_on(cuda_device, batch, L, H, P, N, seed=2033)
    ws = torch.zeros(256, dtype=torch.uint8, device=cuda_device)
    y, hl = ssm.ssm_ssd_fwd(p["x"], p["dt"], p["A"], p["B"], p["C"], p["D"], p["dt_bias"], True, None,
                            workspace=ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0, "tensor-core wait ran out"
    # ((b * L + t) * H + h) * P >= 2^31 for b = 15 and t past about 32700
    for b, h in ((0, 0), (15, 31), (15, 63)):
        sl = slice(h, h + 1)
        ref, ref_h = oracle.ssd(p["x"][b:b + 1, :, sl].cpu(), p["dt"][b:b + 1, :, sl].cpu(), p["A"][sl].cpu(),
                                p["B"][b:b + 1].cpu(), p["C"][b:b + 1].cpu(), p["D"][sl].cpu(),
                                p["dt_bias"][sl].cpu(), True, None)
        assert_close(y[b:b + 1, :, sl], ref, "bf16", f"y b{b} h{h}")
        assert_close(hl[b:b + 1, sl], ref_h, "bf16", f"h_last b{b} h{h}")
    del p, y, hl
    _free()


def test_backward_past_int32_indices(cuda_device):
    """Scan backward, bf16, 4 x 16384 channels x 32800 steps: u, delta, z, dout and the three
    per-token gradients hold 2.15e9 elements each, and the 8-step checkpoints 18 GB. Every
    per-channel gradient (du, ddelta, dz, dh0; dA, dD, ddelta_bias, which sum over the channel's
    sequences) of the sampled channels against the oracle; dB and dC sum over all channels and are
    covered by the smaller backward tests."""
    ssm = _ssm()
    batch, dim, L, N = 4, 16384, 32800, 16
    assert batch * dim * L > INT31
    p = inputs.scan_inputs_on(cuda_device, batch, dim, L, N, 0, "bf16", seed=2034)
    gen = torch.Generator(device=cuda_device).manual_seed(2035)
    dout = torch.randn(batch, dim, L, generator=gen, device=cuda_device).to(torch.bfloat16)
    dhl = torch.randn(batch, dim, N, generator=gen, device=cuda_device)
    g = ssm.ssm_selective_scan_bwd(p["x"], p["delta"], p["A"], p["B"], p["C"], dout, p["D"], p["z"], p["delta_bias"],
                                   True, None, dhl)
    torch.cuda.synchronize()
    # (b * dim + d) * L >= 2^31 for b = 3 and d past about 10000
    for d in (0, 8000, 16383):
        assert d < 16383 or (3 * dim + d) * L > INT31
        sl = lambda t: t[:, d:d + 1].cpu()
        ref = oracle.selective_scan_bwd(sl(p["x"]), sl(p["delta"]), p["A"][d:d + 1].cpu(), p["B"].cpu(), p["C"].cpu(),
                                        sl(dout), p["D"][d:d + 1].cpu(), sl(p["z"]), p["delta_bias"][d:d + 1].cpu(),
                                        True, None, sl(dhl), nthreads=oracle.oracle.default_threads())
        for k in ("du", "ddelta", "dz", "dh0"):
            assert_close(g[k][:, d:d + 1], ref[k], "bf16", f"{k}[:, {d}]")
        assert_close(g["dA"][d:d + 1], ref["dA"], "bf16", f"dA[{d}]")
        assert_close(g["dD"][d:d + 1], ref["dD"], "bf16", f"dD[{d}]")
        assert_close(g["ddelta_bias"][d:d + 1], ref["ddelta_bias"], "bf16", f"ddelta_bias[{d}]")
    del p, g, dout, dhl
    _free()

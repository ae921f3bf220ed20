"""Segment aggregates on the GPU: ssm_selective_scan_aggregate and ssm_scan_compose against the
oracle, and a sequence processed as segments in order, one after another on one GPU, the way the
sequence-split ranks do it (aggregate, compose the earlier segments, scan from the composed
state), against the oracle's scan of the whole sequence."""

import numpy as np
import pytest
import torch

import oracle
from selective_state_space_145_b300 import inputs
from ssm_testutil import assert_close, oracle_scan, to_dev

pytestmark = pytest.mark.gpu


def _ssm():
    import selective_state_space_145_b300 as ssm

    return ssm


@pytest.mark.parametrize("io,N,K,L", [("f32", 16, 4, 700), ("bf16", 16, 0, 5000), ("bf16", 32, 4, 333),
                                      ("f32", 7, 3, 1), ("bf16", 16, 4, 40000)])
def test_aggregate_matches_oracle(cuda_device, io, N, K, L):
    ssm = _ssm()
    p = inputs.scan_inputs(2, 45, L, N, K, io, seed=90 + L + N, with_conv_init=K > 1, random_A=True,
                           salient_frac=0.01)
    g = to_dev(p, cuda_device)
    S, h = ssm.ssm_selective_scan_aggregate(g["x"], g["delta"], g["A"], g["B"], g["delta_bias"], True, g["conv_w"],
                                            g["conv_b"], g["conv_init"])
    v = p["delta"].double().numpy() + p["delta_bias"].double().numpy()[None, :, None]
    S_ref = oracle.softplus(v).sum(axis=2)
    _, h_ref = oracle.selective_scan(p["x"], p["delta"], p["A"], p["B"], p["B"], None, None, p["delta_bias"], True,
                                     p["conv_w"], p["conv_b"], p["conv_init"], None)
    assert_close(S, S_ref, io, "sum of Delta")
    assert_close(h, h_ref, io, "end state from zero")


def test_compose_matches_oracle(cuda_device):
    ssm = _ssm()
    gen = torch.Generator().manual_seed(17)
    nseg, batch, dim, N = 5, 3, 40, 16
    S = torch.rand(nseg, batch, dim, generator=gen) * 2
    b = torch.randn(nseg, batch, dim, N, generator=gen)
    A = -torch.rand(dim, N, generator=gen) * 3
    h0 = torch.randn(batch, dim, N, generator=gen)
    got = ssm.ssm_scan_compose(S.to(cuda_device), b.to(cuda_device), A.to(cuda_device), h0.to(cuda_device))
    h = h0.double().numpy()
    for j in range(nseg):
        a = np.exp(A.double().numpy()[None] * S[j].double().numpy()[:, :, None])
        _, h = oracle.compose(np.ones_like(a), h, a, b[j].double().numpy())
    assert_close(got, h, "f32", "composed state")
    got0 = ssm.ssm_scan_compose(S[:0].to(cuda_device), b[:0].to(cuda_device), A.to(cuda_device), h0.to(cuda_device))
    assert torch.equal(got0, h0.to(cuda_device))  # no segment: the initial state


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_segments_in_order_equal_the_whole_scan(cuda_device, io):
    ssm = _ssm()
    L, cuts = 900, [0, 300, 302, 900]  # the middle segment is shorter than the conv window
    p = inputs.scan_inputs(2, 37, L, 16, 4, io, seed=71, with_h0=True, with_conv_init=True, random_A=True)
    g = to_dev(p, cuda_device)
    ref, ref_h = oracle_scan(p)
    K1 = 3
    S_list, b_list, outs = [], [], []
    stream_x = torch.cat([g["conv_init"], g["x"]], dim=2)   # the raw inputs with the window before them
    for r in range(len(cuts) - 1):
        t0, t1 = cuts[r], cuts[r + 1]
        seg = lambda t: t[..., t0:t1].contiguous()
        win = stream_x[:, :, t0:t0 + K1].contiguous()         # the last 3 raw inputs before t0
        S_r, b_r = ssm.ssm_selective_scan_aggregate(seg(g["x"]), seg(g["delta"]), g["A"], seg(g["B"]), g["delta_bias"],
                                                    True, g["conv_w"], g["conv_b"], win)
        h_in = ssm.ssm_scan_compose(torch.stack(S_list), torch.stack(b_list), g["A"], g["h0"]) if S_list else g["h0"]
        out, h_last = ssm.ssm_selective_scan_fwd(seg(g["x"]), seg(g["delta"]), g["A"], seg(g["B"]), seg(g["C"]),
                                                 g["D"], seg(g["z"]), g["delta_bias"], True, g["conv_w"], g["conv_b"],
                                                 win, h_in)
        S_list.append(S_r)
        b_list.append(b_r)
        outs.append(out)
    assert_close(torch.cat(outs, dim=2), ref, io, "segments vs whole")
    assert_close(h_last, ref_h, io, "final state")
    h_all = ssm.ssm_scan_compose(torch.stack(S_list), torch.stack(b_list), g["A"], g["h0"])
    assert_close(h_all, ref_h, io, "composed final state")

"""GPU parity of the opt-in S4D-real path (SSM_SCAN_S4D_REAL): where A[d,n] = (n+1) A[d,0] (the
pages' initialisation A = -(1..N)), the whole-channel kernels take Abar_n = Abar_0^(n+1) from one
exp2 and multiplies. Against the fp64 oracle at the scan's own bounds, on problems planned for the
whole-channel passes (chunked, many channels), forward and reverse, N = 16 and N < 16; the path
must differ from the generic one in rounding (so it ran), and must fall back to the generic one,
bit for bit, for the channels of any CTA whose A breaks the structure.
"""

import pytest
import torch

from selective_state_space_145_b300 import inputs
from ssm_testutil import assert_close, gpu_scan, oracle_scan, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    # batch, dim, L, N, K, io, chunk_len, reverse
    (2, 1000, 704, 16, 4, "bf16", 64, False),   # 11 chunks, conv, whole-channel passes
    (2, 1000, 333, 5, 0, "f32", 64, False),     # N < 16, ragged last chunk
    (1, 2048, 1000, 16, 0, "f32", 128, True),   # reverse
    (2, 1200, 257, 12, 3, "f32", 64, False),    # element-wise path (row not a 16-byte multiple)
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}_d{}_l{}_n{}_k{}_{}_cl{}_rev{}".format(*c))
def test_s4d_matches_oracle_and_takes_the_powers(cuda_device, case):
    batch, dim, L, N, K, io, cl, rev = case
    p = inputs.scan_inputs(batch, dim, L, N, K, io, seed=4400 + dim + L, with_h0=True, with_conv_init=K > 1,
                           salient_frac=0.01)
    g = to_dev(p, cuda_device)
    out_s, h_s = gpu_scan(g, chunk_len=cl, reverse=rev, s4d_real=True)
    out_g, h_g = gpu_scan(g, chunk_len=cl, reverse=rev)
    ref, refL = oracle_scan(p, reverse=rev)
    assert_close(out_s, ref, io, "out (S4D-real)")
    assert_close(h_s, refL, io, "h_last (S4D-real)")
    # the powers round differently from one exp2 per state: equal results would mean they never ran
    assert not torch.equal(h_s, h_g)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_s4d_falls_back_for_generic_A(cuda_device, io):
    """Random A breaks the structure in every CTA: the flag then computes exactly the generic path."""
    p = inputs.scan_inputs(2, 1000, 704, 16, 4, io, seed=4411, with_h0=True, random_A=True)
    g = to_dev(p, cuda_device)
    out_s, h_s = gpu_scan(g, chunk_len=64, s4d_real=True)
    out_g, h_g = gpu_scan(g, chunk_len=64)
    assert torch.equal(out_s, out_g) and torch.equal(h_s, h_g)


def test_s4d_one_channel_off_structure(cuda_device):
    """One channel's A off the structure by one ulp: its CTAs take the generic path (its results
    are the generic ones bit for bit), the other CTAs the powers; all against the oracle."""
    p = inputs.scan_inputs(2, 1000, 704, 16, 0, "f32", seed=4412, with_h0=True)
    bad = 517
    A = p["A"].clone()
    A[bad, 7] = torch.nextafter(A[bad, 7], torch.tensor(0.0))
    p["A"] = A
    g = to_dev(p, cuda_device)
    out_s, h_s = gpu_scan(g, chunk_len=64, s4d_real=True)
    out_g, h_g = gpu_scan(g, chunk_len=64)
    ref, refL = oracle_scan(p)
    assert_close(out_s, ref, "f32", "out (S4D-real, one channel off)")
    assert_close(h_s, refL, "f32", "h_last (S4D-real, one channel off)")
    assert torch.equal(out_s[:, bad], out_g[:, bad]) and torch.equal(h_s[:, bad], h_g[:, bad])
    assert not torch.equal(h_s, h_g)


def test_s4d_longscan_workload_whole(cuda_device):
    """The long-scan workload (A = -(n+1)) with the flag, every output against the oracle."""
    w = inputs.WORKLOADS["longscan_bf16_b1_d1536_l131072_n16"]
    p = inputs.workload_inputs(w)
    g = to_dev(p, cuda_device)
    out, hL = gpu_scan(g, s4d_real=True)
    torch.cuda.synchronize()
    del g
    ref, refL = oracle_scan(p)
    del p
    assert_close(out, ref, w.io, "long scan out (S4D-real)")
    del ref
    assert_close(hL, refL, w.io, "long scan h_last (S4D-real)")


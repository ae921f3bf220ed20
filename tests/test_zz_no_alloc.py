"""The selective scan for callers that cannot allocate device memory.

ssm_selective_scan_fwd_noalloc keeps the chunk-carry scratch in a fixed device array of the
library instead of a caller-provided workspace, for callers that own only their inputs and
outputs (a plugin interface that passes tensors but no workspace, or a serving loop that
must not call cudaMalloc). These tests call it through the C ABI, twice in a row, and check
each result against the fp64 oracle and against the ordinary entry point, within the
tolerances the other GPU tests use. This file is collected last on purpose.
"""

import ctypes

import pytest
import torch

import oracle
from selective_state_space_145_b300 import inputs
from ssm_testutil import TOL, assert_close, gpu_scan, oracle_scan, to_dev

pytestmark = pytest.mark.gpu


def _call_noalloc(g, out, h_last, chunk_len):
    import selective_state_space_145_b300 as ssm
    from selective_state_space_145_b300.ssm import _io_code

    L = ssm.lib()
    batch, dim, seqlen = g["x"].shape
    N = g["A"].shape[1]
    K = g["conv_w"].shape[1] if g.get("conv_w") is not None else 0
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.ssm_selective_scan_fwd_noalloc(
        p(g["x"]), p(g["delta"]), p(g["A"]), p(g["B"]), p(g["C"]), p(g["D"]), p(g["z"]), p(g["delta_bias"]), 1,
        p(g.get("conv_w")), p(g.get("conv_b")), K, p(g.get("conv_init")), p(g.get("h0")), p(out), p(h_last), None,
        batch, dim, seqlen, N, _io_code(g["x"]), chunk_len, 0, stream)


@pytest.mark.parametrize("io,chunk_len", [("f32", 64), ("bf16", 128), ("bf16", 0)])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(cuda_device, io, chunk_len):
    p = inputs.scan_inputs(2, 96, 640, 16, 4, io, seed=4242, with_h0=True, with_conv_init=True)
    g = to_dev(p, cuda_device)
    ref, ref_h = oracle_scan(p)
    ws_out, ws_h = gpu_scan(g, chunk_len=chunk_len)
    torch.cuda.synchronize()
    for call in range(2):  # the array keeps the last call's contents; a second call must not depend on them
        out = torch.full_like(g["x"], float("nan"))
        h_last = torch.full((2, 96, 16), float("nan"), device=cuda_device)
        assert _call_noalloc(g, out, h_last, chunk_len) == 0
        torch.cuda.synchronize()
        assert_close(out, ref, io, f"noalloc out, call {call}")
        assert_close(h_last, ref_h, io, f"noalloc h_last, call {call}")
        assert_close(out, ws_out.float().cpu().double().numpy(), io, f"noalloc vs workspace entry, call {call}")
        assert_close(h_last, ws_h.cpu().double().numpy(), io, f"noalloc vs workspace h_last, call {call}")


def test_noalloc_fits_default_chunks_to_its_array(cuda_device):
    """A problem whose default chunking would need more carry scratch than the fixed array: with
    chunk_len = 0 the call lowers the chunk count until the carries fit, and still gives the
    oracle's result (checked on sampled channels, the first and last among them) and the
    ordinary entry point's (checked on every element)."""
    import selective_state_space_145_b300 as ssm

    batch, dim, N = 1, 8192, 16
    L = 3072
    while ssm.ssm_scan_workspace_bytes(batch, dim, L, N, 0, torch.bfloat16) <= ssm.ssm.NOALLOC_SCRATCH_BYTES:
        L += 3072
        assert L <= 40 * 3072, "no problem of this shape needs more than the fixed array"
    g = inputs.scan_inputs_on(cuda_device, batch, dim, L, N, 0, "bf16", seed=77)
    ws_out, ws_h = gpu_scan(g)
    torch.cuda.synchronize()
    chans = [0, 1, 4095, 5000, dim - 1]
    for call in range(2):
        out = torch.full_like(g["x"], float("nan"))
        h_last = torch.full((batch, dim, N), float("nan"), device=cuda_device)
        assert _call_noalloc(g, out, h_last, 0) == 0
        torch.cuda.synchronize()
        rtol, atol = TOL["bf16"]
        assert torch.isfinite(out.float()).all()
        assert torch.allclose(out.float(), ws_out.float(), rtol=rtol, atol=atol), f"noalloc vs workspace, call {call}"
        assert torch.allclose(h_last, ws_h, rtol=rtol, atol=atol), f"noalloc h_last vs workspace, call {call}"
        for d in chans:
            sl = lambda t: t[:, d:d + 1].cpu()
            ref, ref_h = oracle.selective_scan(sl(g["x"]), sl(g["delta"]), g["A"][d:d + 1].cpu(), g["B"].cpu(),
                                               g["C"].cpu(), g["D"][d:d + 1].cpu(), sl(g["z"]),
                                               g["delta_bias"][d:d + 1].cpu(), True)
            assert_close(out[:, d:d + 1], ref, "bf16", f"noalloc out[0,{d}], call {call}")
            assert_close(h_last[:, d:d + 1], ref_h, "bf16", f"noalloc h_last[0,{d}], call {call}")
    del g, ws_out, ws_h
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_noalloc_rejects_scratch_beyond_its_maximum(cuda_device):
    import selective_state_space_145_b300 as ssm

    # 256 channels x 499 carries of 68 bytes each is beyond the fixed array: refused on the
    # host before any launch (the tensors still have the full size the call states)
    g = to_dev(inputs.scan_inputs(1, 256, 32000, 16, 0, "bf16", seed=1), cuda_device)
    need = ssm.ssm_scan_workspace_bytes(1, 256, 32000, 16, 64, torch.bfloat16)
    assert need > ssm.ssm.NOALLOC_SCRATCH_BYTES
    out = torch.empty_like(g["x"])
    h_last = torch.empty(1, 256, 16, device=cuda_device)
    assert _call_noalloc(g, out, h_last, 64) == 2  # SSM_ERR_UNSUPPORTED

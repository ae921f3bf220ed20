"""The selective scan for callers that cannot allocate device memory.

ssm_selective_scan_fwd_noalloc keeps the chunk-carry scratch in a fixed device array of the
library instead of a caller-provided workspace, for callers that own only their inputs and
outputs (a plugin interface that passes tensors but no workspace, or a serving loop that
must not call cudaMalloc). These tests call it through the C ABI and check that two calls in
a row give the result of the ordinary entry point, within the tolerances the other GPU tests
use. This file is collected last on purpose.
"""

import ctypes

import pytest
import torch

from selective_state_space_145_b300 import inputs
from ssm_testutil import assert_close, gpu_scan, to_dev

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
def test_noalloc_matches_workspace_entry_point_twice(cuda_device, io, chunk_len):
    p = inputs.scan_inputs(2, 96, 640, 16, 4, io, seed=4242, with_h0=True, with_conv_init=True)
    g = to_dev(p, cuda_device)
    ref_out, ref_h = gpu_scan(g, chunk_len=chunk_len)
    torch.cuda.synchronize()
    for _ in range(2):  # the array keeps the last call's contents; a second call must not depend on them
        out = torch.full_like(g["x"], float("nan"))
        h_last = torch.full((2, 96, 16), float("nan"), device=cuda_device)
        assert _call_noalloc(g, out, h_last, chunk_len) == 0
        torch.cuda.synchronize()
        assert_close(out, ref_out.float().cpu().double().numpy(), io, "noalloc out")
        assert_close(h_last, ref_h.cpu().double().numpy(), io, "noalloc h_last")


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

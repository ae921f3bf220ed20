"""The library's calls under CUDA graph capture: they launch on the caller's stream, allocate
nothing and make no host synchronisation, so a captured sequence replays to the same results
as eager calls (bit for bit: the kernels are deterministic)."""

import pytest
import torch

from selective_state_space_145_b300 import inputs
from ssm_testutil import to_dev

pytestmark = pytest.mark.gpu


def test_decode_steps_replay_from_a_graph(cuda_device):
    import selective_state_space_145_b300 as ssm

    q = inputs.decode_inputs(8, 512, 16, 4, "bf16", seed=3, steps=6)
    g = to_dev(q, cuda_device)
    state0, win0 = g["state"].clone(), g["conv_state"].clone()
    y = torch.empty(6, 8, 512, dtype=torch.bfloat16, device=cuda_device)

    def steps():
        for t in range(6):
            ssm.ssm_selective_state_update(g["state"], g["conv_state"], g["x"][t], g["delta"][t], g["A"], g["B"][t],
                                           g["C"][t], g["D"], g["z"][t], g["delta_bias"], True, g["conv_w"],
                                           g["conv_b"], y=y[t])

    steps()
    torch.cuda.synchronize()
    y_eager, s_eager, w_eager = y.clone(), g["state"].clone(), g["conv_state"].clone()
    g["state"].copy_(state0)
    g["conv_state"].copy_(win0)
    side = torch.cuda.Stream(cuda_device)
    side.wait_stream(torch.cuda.current_stream(cuda_device))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        steps()  # warm the kernels' one-time attribute setup outside the capture
        torch.cuda.synchronize()
        g["state"].copy_(state0)
        g["conv_state"].copy_(win0)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=side):
            steps()
    torch.cuda.synchronize()
    g["state"].copy_(state0)
    g["conv_state"].copy_(win0)
    y.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, y_eager)
    assert torch.equal(g["state"], s_eager)
    assert torch.equal(g["conv_state"], w_eager)


def test_chunked_scan_replays_from_a_graph(cuda_device):
    """The chunked forward (carry kernel, then main kernel) under capture."""
    import selective_state_space_145_b300 as ssm

    p = inputs.scan_inputs(2, 64, 1024, 16, 4, "f32", seed=9, with_h0=True)
    g = to_dev(p, cuda_device)
    ws = torch.empty(max(1, ssm.ssm_scan_workspace_bytes(2, 64, 1024, 16, 128, torch.float32)), dtype=torch.uint8,
                     device=cuda_device)
    out = torch.empty_like(g["x"])
    hl = torch.empty(2, 64, 16, device=cuda_device)

    def call():
        ssm.ssm_selective_scan_fwd(g["x"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"], g["delta_bias"], True,
                                   g["conv_w"], g["conv_b"], h0=g["h0"], chunk_len=128, workspace=ws, out=out,
                                   h_last=hl)

    call()
    torch.cuda.synchronize()
    o_eager, h_eager = out.clone(), hl.clone()
    side = torch.cuda.Stream(cuda_device)
    side.wait_stream(torch.cuda.current_stream(cuda_device))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            call()
    torch.cuda.synchronize()
    out.zero_()
    hl.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, o_eager) and torch.equal(hl, h_eager)

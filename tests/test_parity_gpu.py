"""GPU parity: the CUDA library, called through its C ABI (ctypes binding), against the fp64
CPU oracle on the same seeded inputs, element by element.

Small problems are compared whole; they span several time tiles, several channel tiles,
ragged tails, several chunks and the degenerate cases. The five synthetic workloads run at
full size in the launch configuration the benchmark uses and every output element is
compared with the oracle run on the whole workload.
"""

import numpy as np
import pytest
import torch

import oracle
from selective_state_space_145_b300 import inputs
from ssm_testutil import TOL, assert_close, gpu_scan, oracle_scan, to_dev

pytestmark = pytest.mark.gpu


def _ssm():
    import selective_state_space_145_b300 as ssm

    return ssm


# ---------------------------------------------------------------- whole small problems

SMALL = [
    # batch, dim, L, N, K, io, with_h0, with_init, random_A, chunk_len
    (1, 64, 256, 16, 0, "f32", False, False, False, 0),      # the small scan workload's shape
    (2, 37, 101, 16, 4, "f32", True, True, True, 0),         # ragged L (element-wise path), partial channel tile
    (2, 40, 96, 5, 3, "bf16", True, True, True, 0),          # N < 16, K < 4
    (3, 130, 200, 16, 4, "bf16", False, False, False, 64),   # 4 chunks, ragged last chunk
    (2, 33, 333, 7, 2, "f32", True, True, True, 64),         # chunks + ragged + odd N
    (1, 20000, 40, 16, 4, "bf16", True, False, False, 0),    # many channel tiles
    (2, 5000, 300, 16, 4, "f32", True, True, True, 128),     # many channel tiles, chunked
    (1, 3, 1, 1, 4, "f32", True, True, True, 0),             # L = 1, N = 1
    (1, 8, 3, 16, 4, "bf16", False, True, False, 0),         # L < K-1: the window comes from conv_init
    # more than 16 states: four lanes of 8 states per channel (main pass), two lanes of 16 (carry)
    (1, 40, 200, 17, 0, "f32", True, False, True, 0),        # N = 17, one chunk
    (2, 24, 333, 24, 3, "f32", True, True, True, 64),        # N = 24, chunks, ragged
    (2, 50, 300, 32, 4, "bf16", True, True, True, 128),      # N = 32, chunks, conv
    (1, 3000, 64, 32, 4, "bf16", False, False, False, 0),    # N = 32, many channel tiles
    (1, 1536, 8192, 32, 4, "bf16", True, True, False, 0),    # N = 32, long: the default plan's many chunks
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "b{}_d{}_l{}_n{}_k{}_{}_h0{}_ci{}_rA{}_cl{}".format(*c))
def test_scan_small_whole(cuda_device, case):
    batch, dim, L, N, K, io, h0, ci, rA, cl = case
    p = inputs.scan_inputs(batch, dim, L, N, K, io, seed=1000 + dim + L, with_h0=h0, with_conv_init=ci,
                           random_A=rA)
    g = to_dev(p, cuda_device)
    out, hL, cs = gpu_scan(g, chunk_len=cl, return_conv_state=K > 0, d_conv=K or None) if K > 0 else \
        (*gpu_scan(g, chunk_len=cl), None)
    ref, refL, *rest = oracle_scan(p, want_conv_state=K > 0)
    assert_close(out, ref, io, "out")
    assert_close(hL, refL, io, "h_last")
    if K > 1:
        # the raw-input window is moved bit for bit
        np.testing.assert_array_equal(cs.float().cpu().numpy(), rest[0])


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_scan_options_off(cuda_device, io):
    """No gate, no skip, no bias, softplus off (Delta = delta, positive), no conv."""
    p = inputs.scan_inputs(2, 70, 130, 16, 0, io, seed=5, with_z=False, with_D=False, random_A=True)
    p["delta_bias"] = None
    p["delta"] = (p["delta"].float().abs() * 0.2 + 0.01).to(p["delta"].dtype)
    g = to_dev(p, cuda_device)
    out, hL = gpu_scan(g, delta_softplus=False)
    ref, refL = oracle_scan(p, delta_softplus=False)
    assert_close(out, ref, io, "out")
    assert_close(hL, refL, io, "h_last")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_chunked_equals_unchunked(cuda_device, io):
    """The cross-chunk carry: every chunk length gives the oracle's result, and the same
    result as one chunk to within rounding."""
    p = inputs.scan_inputs(2, 48, 700, 16, 4, io, seed=77, with_h0=True, with_conv_init=True, salient_frac=0.02)
    g = to_dev(p, cuda_device)
    ref, refL = oracle_scan(p)
    one, one_h = gpu_scan(g, chunk_len=1 << 20)
    for cl in (64, 128, 192, 320):
        out, hL = gpu_scan(g, chunk_len=cl)
        assert_close(out, ref, io, f"out chunk_len={cl}")
        assert_close(hL, refL, io, f"h_last chunk_len={cl}")
        assert_close(out, one.float().cpu().double().numpy(), io, f"chunked vs whole cl={cl}")


def test_chunked_prompt_on_gpu(cuda_device):
    """Two GPU calls passing (h_last, conv window) equal one call (prompts processed in chunks)."""
    p = inputs.scan_inputs(2, 50, 257, 16, 4, "f32", seed=9, with_h0=True, with_conv_init=True)
    g = to_dev(p, cuda_device)
    full, hfull, csfull = gpu_scan(g, return_conv_state=True)
    L1 = 100
    g1 = {k: (v[..., :L1].contiguous() if k in ("x", "delta", "z", "B", "C") else v) for k, v in g.items()}
    o1, h1, cs1 = gpu_scan(g1, return_conv_state=True)
    g2 = {k: (v[..., L1:].contiguous() if k in ("x", "delta", "z", "B", "C") else v) for k, v in g.items()}
    g2["h0"], g2["conv_init"] = h1, cs1
    o2, h2, cs2 = gpu_scan(g2, return_conv_state=True)
    ref, refL = oracle_scan(p)
    assert_close(torch.cat([o1, o2], dim=-1), ref, "f32", "two calls vs oracle")
    assert_close(h2, refL, "f32", "h_last after two calls")
    assert torch.equal(cs2, csfull)


def test_empty_and_zero_length(cuda_device):
    ssm = _ssm()
    p = inputs.scan_inputs(2, 24, 0, 16, 4, "f32", seed=3, with_h0=True, with_conv_init=True)
    g = to_dev(p, cuda_device)
    out, hL, cs = gpu_scan(g, return_conv_state=True)
    torch.cuda.synchronize()
    assert out.numel() == 0
    assert torch.equal(hL, g["h0"])
    assert torch.equal(cs, g["conv_init"])
    # batch 0 / dim 0: nothing to do
    e = torch.empty(0, 8, 16, device=cuda_device)
    A = -torch.ones(8, 16, device=cuda_device)
    Bm = torch.empty(0, 16, 16, device=cuda_device)
    out, hL = ssm.ssm_selective_scan_fwd(e, e, A, Bm, Bm)
    assert out.shape == (0, 8, 16)


# ---------------------------------------------------------------- backward scan (SSM_SCAN_REVERSE)

REVERSE = [
    # batch, dim, L, N, K, io, with_h0, with_init, chunk_len
    (2, 37, 200, 16, 4, "f32", True, True, 0),       # ragged last tile, vector path, partial channel tile
    (1, 40, 100, 16, 4, "f32", True, True, 0),       # fp32 rows ending on a 4-step boundary
    (2, 40, 264, 16, 4, "bf16", True, True, 128),    # 3 chunks, ragged last chunk
    (2, 33, 101, 7, 3, "f32", True, True, 64),       # element-wise path (row not a whole 16 bytes), chunks
    (1, 70, 130, 16, 0, "bf16", True, False, 0),     # element-wise path, no conv
    (2, 64, 196, 16, 4, "f32", False, False, 64),    # chunks of 64, last chunk 4 steps
    (1, 8, 3, 16, 4, "bf16", False, True, 0),        # L < K-1: the window comes from conv_init
    (2, 30, 300, 32, 4, "bf16", True, True, 128),    # N = 32, chunks
    (1, 20, 97, 20, 0, "f32", True, False, 64),      # N = 20, element-wise path, chunks
]


@pytest.mark.parametrize("case", REVERSE, ids=lambda c: "b{}_d{}_l{}_n{}_k{}_{}_h0{}_ci{}_cl{}".format(*c))
def test_reverse_small_whole(cuda_device, case):
    batch, dim, L, N, K, io, h0, ci, cl = case
    p = inputs.scan_inputs(batch, dim, L, N, K, io, seed=3000 + dim + L, with_h0=h0, with_conv_init=ci,
                           random_A=True)
    g = to_dev(p, cuda_device)
    if K > 0:
        out, hL, cs = gpu_scan(g, chunk_len=cl, return_conv_state=True, d_conv=K, reverse=True)
        ref, refL, refcs = oracle_scan(p, want_conv_state=True, reverse=True)
    else:
        out, hL = gpu_scan(g, chunk_len=cl, reverse=True)
        ref, refL = oracle_scan(p, reverse=True)
    assert_close(out, ref, io, "out")
    assert_close(hL, refL, io, "h_last")
    if K > 1:
        np.testing.assert_array_equal(cs.float().cpu().numpy(), refcs)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_reverse_chunked_equals_unchunked(cuda_device, io):
    p = inputs.scan_inputs(2, 48, 700, 16, 4, io, seed=78, with_h0=True, with_conv_init=True, salient_frac=0.02)
    g = to_dev(p, cuda_device)
    ref, refL = oracle_scan(p, reverse=True)
    one, _ = gpu_scan(g, chunk_len=1 << 20, reverse=True)
    for cl in (64, 192, 320):
        out, hL = gpu_scan(g, chunk_len=cl, reverse=True)
        assert_close(out, ref, io, f"out chunk_len={cl}")
        assert_close(hL, refL, io, f"h_last chunk_len={cl}")
        assert_close(out, one.float().cpu().double().numpy(), io, f"chunked vs whole cl={cl}")


def test_reverse_split_on_gpu(cuda_device):
    """Two backward GPU calls, the later part first, passing (h_last, conv window), equal one."""
    p = inputs.scan_inputs(2, 50, 257, 16, 4, "f32", seed=10, with_h0=True, with_conv_init=True)
    g = to_dev(p, cuda_device)
    full, hfull, csfull = gpu_scan(g, return_conv_state=True, reverse=True)
    L1 = 100
    late = {k: (v[..., L1:].contiguous() if k in ("x", "delta", "z", "B", "C") else v) for k, v in g.items()}
    o2, h2, cs2 = gpu_scan(late, return_conv_state=True, reverse=True)
    early = {k: (v[..., :L1].contiguous() if k in ("x", "delta", "z", "B", "C") else v) for k, v in g.items()}
    early["h0"], early["conv_init"] = h2, cs2
    o1, h1, cs1 = gpu_scan(early, return_conv_state=True, reverse=True)
    ref, refL = oracle_scan(p, reverse=True)
    assert_close(torch.cat([o1, o2], dim=-1), ref, "f32", "two backward calls vs oracle")
    assert_close(h1, refL, "f32", "h_last after two backward calls")
    assert torch.equal(cs1, csfull)


def test_deterministic(cuda_device):
    p = inputs.scan_inputs(2, 64, 512, 16, 4, "bf16", seed=21, with_h0=True)
    g = to_dev(p, cuda_device)
    a1, h1 = gpu_scan(g, chunk_len=128)
    a2, h2 = gpu_scan(g, chunk_len=128)
    assert torch.equal(a1, a2) and torch.equal(h1, h2)


# ---------------------------------------------------------------- standalone conv

@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("L", [1, 37, 256])
def test_conv1d(cuda_device, io, K, L):
    ssm = _ssm()
    p = inputs.scan_inputs(2, 19, L, 4, K, io, seed=K * 100 + L, with_conv_init=True)
    g = to_dev(p, cuda_device)
    for silu in (True, False):
        for init in (True, False):
            y = ssm.ssm_causal_conv1d_fwd(g["x"], g["conv_w"], g["conv_b"], g["conv_init"] if init else None,
                                          apply_silu=silu)
            ref = oracle.causal_conv1d(p["x"], p["conv_w"], p["conv_b"], p["conv_init"] if init else None,
                                       apply_silu=silu)
            assert_close(y, ref, io, f"conv silu={silu} init={init}")


# ---------------------------------------------------------------- decode

DECODE_SMALL = [
    # batch, dim, N, K, io, steps
    (3, 50, 16, 4, "bf16", 5),
    (2, 33, 5, 2, "f32", 4),     # N not a multiple of 4: element-wise state path
    (4, 64, 16, 4, "f32", 3),
    (1, 7, 16, 1, "bf16", 2),    # K = 1: no window
    (2, 40, 17, 4, "f32", 3),    # more than 16 states: 8 states per thread
    (3, 33, 24, 3, "bf16", 4),
    (2, 70, 32, 4, "f32", 3),
]


@pytest.mark.parametrize("case", DECODE_SMALL, ids=lambda c: "b{}_d{}_n{}_k{}_{}_s{}".format(*c))
def test_decode_small(cuda_device, case):
    ssm = _ssm()
    batch, dim, N, K, io, steps = case
    q = inputs.decode_inputs(batch, dim, N, K, io, seed=batch * dim + N, steps=steps, random_A=True)
    g = to_dev(q, cuda_device)
    state, win = q["state"].double().numpy(), (q["conv_state"].double().numpy() if q["conv_state"] is not None else None)
    for t in range(steps):
        y = ssm.ssm_selective_state_update(g["state"], g["conv_state"], g["x"][t], g["delta"][t], g["A"], g["B"][t],
                                           g["C"][t], g["D"], g["z"][t], g["delta_bias"], True, g["conv_w"],
                                           g["conv_b"])
        yr, state, win = oracle.state_update(state, win, q["x"][t], q["delta"][t], q["A"], q["B"][t], q["C"][t], q["D"],
                                             q["z"][t], q["delta_bias"], True, q["conv_w"], q["conv_b"])
        assert_close(y, yr, io, f"y step {t}")
        assert_close(g["state"], state, io, f"state step {t}")
        if K > 1:
            np.testing.assert_array_equal(g["conv_state"].float().cpu().numpy(), win)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_recurrent_equals_parallel_on_gpu(cuda_device, io):
    """K decode steps from (state, window) equal one scan over the same K tokens with h0 = state
    and conv_init = window (recurrent and parallel mode agree)."""
    ssm = _ssm()
    batch, dim, N, K, T = 2, 40, 16, 4, 12
    p = inputs.scan_inputs(batch, dim, T, N, K, io, seed=31, with_h0=True, with_conv_init=True)
    g = to_dev(p, cuda_device)
    out, hL, cs = gpu_scan(g, return_conv_state=True)
    state, win = g["h0"].clone(), g["conv_init"].clone()
    ys = []
    for t in range(T):
        ys.append(ssm.ssm_selective_state_update(state, win, g["x"][..., t].contiguous(), g["delta"][..., t].contiguous(),
                                                 g["A"], g["B"][..., t].contiguous(), g["C"][..., t].contiguous(),
                                                 g["D"], g["z"][..., t].contiguous(), g["delta_bias"], True,
                                                 g["conv_w"], g["conv_b"]))
    yd = torch.stack(ys, dim=-1)
    rtol, atol = TOL[io]
    assert_close(yd, out.float().cpu().double().numpy(), io, "decode vs scan")
    assert_close(state, hL.cpu().double().numpy(), io, "decode state vs scan h_last")
    assert torch.equal(win, cs)


# ---------------------------------------------------------------- zero-order hold (SSM_SCAN_ZOH)

def _zoh_edge_A(A: torch.Tensor) -> torch.Tensor:
    """A with exact zeros and tiny magnitudes in some states, so the expm1 series branch,
    its boundary and the A = 0 limit are all exercised."""
    A = A.clone()
    N = A.shape[1]
    if N > 3:
        A[:, 0] = 0.0
        A[:, 1] = -1e-6
        A[:, 2] = -0.02
        A[:, 3] = 0.3   # a growing mode
    return A


ZOH = [
    # batch, dim, L, N, K, io, chunk_len, reverse
    (2, 37, 200, 16, 4, "f32", 0, False),
    (2, 40, 264, 16, 4, "bf16", 128, False),
    (2, 33, 101, 7, 3, "f32", 64, False),        # element-wise path, chunks, N < 16
    (2, 48, 300, 16, 4, "f32", 64, True),        # backward + ZOH, chunked
    (1, 70, 130, 16, 0, "bf16", 0, True),
    (2, 20, 200, 32, 4, "f32", 64, False),       # N = 32, chunks
]


@pytest.mark.parametrize("case", ZOH, ids=lambda c: "b{}_d{}_l{}_n{}_k{}_{}_cl{}_rev{}".format(*c))
def test_zoh_small_whole(cuda_device, case):
    batch, dim, L, N, K, io, cl, rev = case
    p = inputs.scan_inputs(batch, dim, L, N, K, io, seed=4000 + dim + L, with_h0=True, with_conv_init=K > 1,
                           random_A=True)
    p["A"] = _zoh_edge_A(p["A"])
    g = to_dev(p, cuda_device)
    out, hL = gpu_scan(g, chunk_len=cl, reverse=rev, zoh=True)
    ref, refL = oracle_scan(p, reverse=rev, zoh=True)
    assert_close(out, ref, io, "out")
    assert_close(hL, refL, io, "h_last")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_zoh_decode_matches_oracle_and_scan(cuda_device, io):
    """ZOH decode steps against the oracle, and against the ZOH scan over the same tokens."""
    ssm = _ssm()
    batch, dim, N, K, T = 2, 300, 16, 4, 6
    p = inputs.scan_inputs(batch, dim, T, N, K, io, seed=41, with_h0=True, with_conv_init=True, random_A=True)
    p["A"] = _zoh_edge_A(p["A"])
    g = to_dev(p, cuda_device)
    out, hL, cs = gpu_scan(g, return_conv_state=True, zoh=True)
    state, win = g["h0"].clone(), g["conv_init"].clone()
    ostate, owin = p["h0"].double().numpy(), p["conv_init"].double().numpy()
    ys = []
    for t in range(T):
        cols = {k: g[k][..., t].contiguous() for k in ("x", "delta", "B", "C", "z")}
        ys.append(ssm.ssm_selective_state_update(state, win, cols["x"], cols["delta"], g["A"], cols["B"], cols["C"],
                                                 g["D"], cols["z"], g["delta_bias"], True, g["conv_w"], g["conv_b"],
                                                 zoh=True))
        yr, ostate, owin = oracle.state_update(ostate, owin, p["x"][..., t], p["delta"][..., t], p["A"],
                                               p["B"][..., t], p["C"][..., t], p["D"], p["z"][..., t],
                                               p["delta_bias"], True, p["conv_w"], p["conv_b"], zoh=True)
        assert_close(ys[-1], yr, io, f"decode y step {t}")
        assert_close(state, ostate, io, f"decode state step {t}")
    assert_close(torch.stack(ys, dim=-1), out.float().cpu().double().numpy(), io, "ZOH decode vs ZOH scan")
    assert torch.equal(win, cs)


# ---------------------------------------------------------------- the five workloads, full size
# Every output element of every workload is compared with the oracle: the oracle runs on all host
# threads (about a second for the largest workload on a 16-core host), so no sampling is needed.

def _workload_scan_whole(name, cuda_device, reverse=False, zoh=False):
    w = inputs.WORKLOADS[name]
    p = inputs.workload_inputs(w)
    g = to_dev(p, cuda_device)
    out, hL = gpu_scan(g, reverse=reverse, zoh=zoh)   # default chunking: the launch configuration the benchmark times
    torch.cuda.synchronize()
    del g
    ref, refL = oracle_scan(p, reverse=reverse, zoh=zoh)
    del p
    assert_close(out, ref, w.io, f"{name} out")
    del ref
    assert_close(hL, refL, w.io, f"{name} h_last")


def test_workload_small_scan_whole(cuda_device):
    _workload_scan_whole("scan_f32_b1_d64_l256_n16", cuda_device)


def test_workload_block_f32_whole(cuda_device):
    _workload_scan_whole("block_f32_b2_d1024_l1024_n16_k4", cuda_device)


@pytest.mark.slow
def test_workload_block_bf16_whole(cuda_device):
    _workload_scan_whole("block_bf16_b8_d2048_l2048_n16_k4", cuda_device)


@pytest.mark.slow
def test_workload_longscan_bf16_whole(cuda_device):
    _workload_scan_whole("longscan_bf16_b1_d1536_l131072_n16", cuda_device)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["block_bf16_b8_d2048_l2048_n16_k4", "longscan_bf16_b1_d1536_l131072_n16"])
@pytest.mark.parametrize("mode", ["reverse", "zoh"])
def test_workload_options_whole(cuda_device, name, mode):
    """The backward-direction scan and the ZOH rule on the bf16 workloads at full size, in the
    launch configurations `bench.py --reverse` / `--zoh` time: every output against the oracle."""
    _workload_scan_whole(name, cuda_device, reverse=mode == "reverse", zoh=mode == "zoh")


@pytest.mark.slow
@pytest.mark.parametrize("zoh", [False, True], ids=["euler", "zoh"])
def test_workload_decode_whole(cuda_device, zoh):
    """The decode workload: 64 consecutive steps on every (sequence, channel); y of every step,
    the final state and the final window against the oracle stepping the same inputs (Euler, and
    the ZOH rule that `bench.py --zoh` times)."""
    ssm = _ssm()
    w = inputs.WORKLOADS["decode_bf16_b256_d5120_n16_k4_x64"]
    q = inputs.workload_inputs(w)
    g = to_dev(q, cuda_device)
    state = q["state"].double().numpy()
    win = q["conv_state"].double().numpy()
    for t in range(w.steps):
        y = ssm.ssm_selective_state_update(g["state"], g["conv_state"], g["x"][t], g["delta"][t], g["A"], g["B"][t],
                                           g["C"][t], g["D"], g["z"][t], g["delta_bias"], True, g["conv_w"],
                                           g["conv_b"], zoh=zoh)
        yr, state, win = oracle.state_update(state, win, q["x"][t], q["delta"][t], q["A"], q["B"][t], q["C"][t],
                                             q["D"], q["z"][t], q["delta_bias"], True, q["conv_w"], q["conv_b"],
                                             nthreads=oracle.oracle.default_threads(), zoh=zoh)
        assert_close(y, yr, "bf16", f"decode y step {t}")
    assert_close(g["state"], state, "bf16", "decode state after 64 steps")
    # the window holds raw inputs: moved bit for bit
    np.testing.assert_array_equal(g["conv_state"].float().cpu().numpy(), win)

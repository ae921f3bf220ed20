"""The small odd-shape parity cases again, through libssm_debug.so: the library compiled with
SSM_DEBUG_BOUNDS, in which every checked global access of the scan, segment, decode, conv
(forward and backward), scan-backward and state-space-duality kernels is range-tested against its tensor and an access outside it sets a bit of a device
error word instead of touching memory.

Each case must still match the fp64 oracle (the checks skip nothing on a correct call) and must
leave the error word at zero.
"""

import pytest

import test_backward_gpu as bwd
import test_parity_gpu as par
import test_s4d_gpu as s4d
import test_shard_gpu as seg
import test_ssd_gpu as ssd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_lib(cuda_device):
    import selective_state_space_145_b300 as ssm

    ssm.select_library("debug")
    assert ssm.library_path().endswith("libssm_debug.so")
    ssm.debug_bounds_status(clear=True)
    yield ssm
    ssm.select_library("release")


def _clean(ssm, what):
    word = ssm.debug_bounds_status(clear=True)
    assert word == 0, f"{what}: out-of-range accesses flagged (error word {word:#x})"


@pytest.mark.parametrize("case", par.SMALL, ids=lambda c: "b{}_d{}_l{}_n{}_k{}_{}_h0{}_ci{}_rA{}_cl{}".format(*c))
def test_debug_scan_small(debug_lib, cuda_device, case):
    par.test_scan_small_whole(cuda_device, case)
    _clean(debug_lib, "scan")


@pytest.mark.parametrize("case", par.REVERSE, ids=lambda c: "b{}_d{}_l{}_n{}_k{}_{}_h0{}_ci{}_cl{}".format(*c))
def test_debug_reverse_small(debug_lib, cuda_device, case):
    par.test_reverse_small_whole(cuda_device, case)
    _clean(debug_lib, "reverse scan")


@pytest.mark.parametrize("case", par.ZOH, ids=lambda c: "b{}_d{}_l{}_n{}_k{}_{}_cl{}_rev{}".format(*c))
def test_debug_zoh_small(debug_lib, cuda_device, case):
    par.test_zoh_small_whole(cuda_device, case)
    _clean(debug_lib, "ZOH scan")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_debug_chunked_and_options(debug_lib, cuda_device, io):
    par.test_chunked_equals_unchunked(cuda_device, io)
    par.test_scan_options_off(cuda_device, io)
    _clean(debug_lib, "chunked scan")


def test_debug_empty_and_split(debug_lib, cuda_device):
    par.test_empty_and_zero_length(cuda_device)
    par.test_chunked_prompt_on_gpu(cuda_device)
    _clean(debug_lib, "empty / split prompt")


@pytest.mark.parametrize("case", par.DECODE_SMALL, ids=lambda c: "b{}_d{}_n{}_k{}_{}_s{}".format(*c))
def test_debug_decode_small(debug_lib, cuda_device, case):
    par.test_decode_small(cuda_device, case)
    _clean(debug_lib, "decode")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("L", [1, 37, 256])
def test_debug_conv1d(debug_lib, cuda_device, io, K, L):
    par.test_conv1d(cuda_device, io, K, L)
    _clean(debug_lib, "conv")


@pytest.mark.parametrize("io,N,K,L", [("f32", 16, 4, 700), ("bf16", 32, 4, 333), ("f32", 7, 3, 1)])
def test_debug_segments(debug_lib, cuda_device, io, N, K, L):
    seg.test_aggregate_matches_oracle(cuda_device, io, N, K, L)
    seg.test_compose_matches_oracle(cuda_device)
    _clean(debug_lib, "segment aggregate / compose")


@pytest.mark.parametrize("case", bwd.CASES, ids=lambda c: "b{}_d{}_l{}_n{}_{}_z{}_D{}_bias{}_h0{}_dh{}".format(*c))
def test_debug_backward(debug_lib, cuda_device, case):
    bwd.test_backward_matches_oracle(cuda_device, case)
    _clean(debug_lib, "scan backward")


def test_debug_backward_chunked(debug_lib, cuda_device):
    bwd.test_backward_chunked_long(cuda_device, "bf16")
    bwd.test_backward_empty_sequence(cuda_device)
    _clean(debug_lib, "scan backward, chunked / empty")


@pytest.mark.parametrize("case", bwd.CONV_CASES, ids=lambda c: "b{}_d{}_l{}_k{}_{}_win{}_silu{}".format(*c))
def test_debug_conv_backward(debug_lib, cuda_device, case):
    bwd.test_conv_backward_matches_oracle(cuda_device, case)
    _clean(debug_lib, "conv backward")


@pytest.mark.parametrize("case", ssd.CASES, ids=lambda c: "b{}_l{}_h{}_h0{}".format(*c))
def test_debug_ssd(debug_lib, cuda_device, case):
    ssd.test_ssd_matches_oracle(cuda_device, case)
    _clean(debug_lib, "state-space duality")


@pytest.mark.parametrize("case", s4d.CASES, ids=lambda c: "b{}_d{}_l{}_n{}_k{}_{}_cl{}_rev{}".format(*c))
def test_debug_s4d_real(debug_lib, cuda_device, case):
    s4d.test_s4d_matches_oracle_and_takes_the_powers(cuda_device, case)
    _clean(debug_lib, "S4D-real scan")

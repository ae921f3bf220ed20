"""CPU-side checks of the C ABI: the library builds, loads, exports every symbol include/ssm.h
declares, and rejects bad arguments on the host before any launch (no GPU needed: every call
here returns from the argument checks)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from selective_state_space_145_b300 import build

    build.build()
    import selective_state_space_145_b300 as ssm

    return ssm.lib()


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "ssm.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"SSM_API\s+[\w\s\*]+?\b(ssm_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    decl = _declared_symbols()
    for name in ("ssm_causal_conv1d_fwd", "ssm_selective_scan_fwd", "ssm_selective_state_update"):
        assert name in decl


def test_library_exports_every_declared_symbol(L):
    import selective_state_space_145_b300 as ssm

    decl = _declared_symbols()
    assert sorted(ssm.EXPORTS) == decl
    for name in decl:
        assert hasattr(L, name), name


def test_version_and_status_strings(L):
    import selective_state_space_145_b300 as ssm

    assert ssm.version() >= 100
    assert ssm.status_string(0) == "SSM_OK"
    assert ssm.status_string(1) == "SSM_ERR_INVALID_ARG"
    assert ssm.status_string(2) == "SSM_ERR_UNSUPPORTED"
    assert ssm.status_string(3) == "SSM_ERR_CUDA"


# A non-null, 64 KiB-aligned address that is not device memory. Every call below is built to
# FAIL the host-side checks (or to be empty work), so nothing is ever launched with it.
FAKE = 0x10000


def _scan(L, **kw):
    a = dict(x=FAKE, delta=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, z=None, delta_bias=None, sp=1, conv_w=None,
             conv_b=None, d_conv=0, conv_init=None, h0=None, out=FAKE, h_last=None, cs_out=None, batch=1, dim=4,
             seqlen=8, dstate=16, io=0, chunk_len=0, ws=None, ws_bytes=0, flags=0)
    a.update(kw)
    return L.ssm_selective_scan_fwd(a["x"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["delta_bias"],
                                    a["sp"], a["conv_w"], a["conv_b"], a["d_conv"], a["conv_init"], a["h0"],
                                    a["out"], a["h_last"], a["cs_out"], a["batch"], a["dim"], a["seqlen"],
                                    a["dstate"], a["io"], a["chunk_len"], a["ws"], a["ws_bytes"], a["flags"], None)


def test_scan_argument_checks(L):
    assert _scan(L, x=None) == 1
    assert _scan(L, out=None) == 1
    assert _scan(L, seqlen=-1) == 1
    assert _scan(L, dstate=0) == 1
    assert _scan(L, dstate=33) == 2  # the forward scan holds up to 32 states
    assert _scan(L, io=7) == 2
    assert _scan(L, sp=2) == 1
    assert _scan(L, conv_w=FAKE, d_conv=5) == 2
    assert _scan(L, conv_w=FAKE, d_conv=0) == 1
    assert _scan(L, conv_b=FAKE) == 1              # conv bias without conv weight
    assert _scan(L, x=FAKE + 2) == 2               # misaligned fp32 pointer
    assert _scan(L, chunk_len=-5) == 1
    assert _scan(L, flags=8) == 1                  # unknown option bit
    assert _scan(L, flags=4, batch=0) == 0         # SSM_SCAN_S4D_REAL is a scan option
    assert _scan(L, flags=1, x=None) == 1          # reverse: same checks
    assert _scan(L, seqlen=1 << 20, chunk_len=64, batch=1, dim=4) == 1   # chunked: workspace missing
    # empty work: no launch, OK
    assert _scan(L, batch=0) == 0
    assert _scan(L, dim=0, x=None) == 0


def test_workspace_query(L):
    import selective_state_space_145_b300 as ssm
    import torch

    assert ssm.ssm_scan_workspace_bytes(1, 64, 256, 16, 256, torch.float32) == 0
    ws = ssm.ssm_scan_workspace_bytes(2, 100, 1000, 16, 64, torch.float32)
    q = (1000 + 63) // 64
    s_bytes = ((q - 1) * 200 * 4 + 255) // 256 * 256
    assert ws == s_bytes + (q - 1) * 200 * 16 * 4
    cl = ssm.ssm_scan_default_chunk_len(1, 1536, 131072, 16, torch.bfloat16)
    assert cl % 64 == 0 and 256 <= cl <= 131072


def test_backward_argument_checks(L):
    f = L.ssm_selective_scan_bwd
    # u, delta, A, B, C, D, z, bias, sp, h0, dout, dh_last, du, ddelta, dz, dA, dB, dC, dD, dbias, dh0,
    # batch, dim, seqlen, dstate, io, ws, ws_bytes, flags, stream
    base = [FAKE] * 5 + [None, None, None, 1, None, FAKE, None] + [FAKE, FAKE, None, FAKE, FAKE, FAKE, None, None,
                                                                     None] + [1, 4, 8, 16, 0, FAKE, 1 << 30, 0, None]
    for i, v, want in ((0, None, 1), (15, None, 1), (24, 17, 2), (25, 7, 2), (28, 1, 2), (28, 2, 2), (28, 4, 1),
                       (6, FAKE, 1), (27, 0, 1), (0, FAKE + 2, 2)):
        bad = list(base)
        bad[i] = v
        assert f(*bad) == want, (i, v)


def test_conv_backward_argument_checks(L):
    f = L.ssm_causal_conv1d_bwd
    # x, w, bias, conv_init, dout, silu, dx, dw, dbias, dconv_init, batch, dim, L, K, io, ws, ws_bytes, stream
    base = [FAKE, FAKE, None, None, FAKE, 1, FAKE, FAKE, None, None, 1, 4, 8, 4, 0, FAKE, 1 << 20, None]
    for i, v, want in ((0, None, 1), (7, None, 1), (13, 5, 2), (13, 0, 1), (5, 2, 1), (14, 9, 2), (16, 0, 1),
                       (0, FAKE + 2, 2)):
        bad = list(base)
        bad[i] = v
        assert f(*bad) == want, (i, v)


def test_decode_and_conv_argument_checks(L):
    f = L.ssm_selective_state_update
    base = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, 1, FAKE, None, 4, FAKE, 2, 8, 16, 1, 0, None]
    bad = list(base)
    bad[0] = None
    assert f(*bad) == 1                            # state missing
    bad = list(base)
    bad[17] = 33
    assert f(*bad) == 2                            # dstate > 32
    bad = list(base)
    bad[1] = None
    assert f(*bad) == 1                            # conv window missing with a conv
    bad = list(base)
    bad[13] = 6
    assert f(*bad) == 2                            # d_conv > 4
    for flags in (1, 4):                           # reverse has no decode form; unknown bit
        bad = list(base)
        bad[19] = flags
        assert f(*bad) == 1
    c = L.ssm_causal_conv1d_fwd
    assert c(None, FAKE, None, None, FAKE, 1, 4, 8, 4, 1, 0, None) == 1
    assert c(FAKE, FAKE, None, None, FAKE, 1, 4, 8, 0, 1, 0, None) == 1
    assert c(FAKE, FAKE, None, None, FAKE, 1, 4, 8, 5, 1, 0, None) == 2
    assert c(FAKE, FAKE, None, None, FAKE, 0, 4, 8, 4, 1, 0, None) == 0


def test_ssd_argument_checks_and_workspace(L):
    f = L.ssm_ssd_fwd
    # x, dt, A, B, C, D, dt_bias, softplus, h0, y, h_last, batch, L, H, P, N, io, ws, ws_bytes, stream
    base = [FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 1, None, FAKE, None, 2, 300, 4, 64, 128, 1, FAKE, 1 << 40, None]
    for i, v, want in ((16, 0, 2),        # fp32 I/O: the tensor-core path is bf16
                       (14, 32, 2),       # head dim other than 64
                       (15, 64, 2),       # state dim other than 128
                       (0, None, 1),      # x missing
                       (7, 2, 1),         # softplus flag not 0/1
                       (18, 128, 1),      # workspace too small
                       (17, None, 1),     # workspace missing
                       (0, FAKE + 2, 2),  # x not 16-byte aligned
                       (17, FAKE + 16, 2),  # workspace not 256-byte aligned
                       (11, 0, 0),        # no sequences: nothing to do
                       (13, 0, 0)):
        bad = list(base)
        bad[i] = v
        assert f(*bad) == want, (i, v)
    ws = L.ssm_ssd_workspace_bytes
    assert ws(2, 300, 4, 64, 128, 1) == 256                        # the status word
    assert ws(2, 300, 4, 64, 128, 0) == 0 and ws(2, 300, 4, 32, 128, 1) == 0


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import selective_state_space_145_b300.ssm as s

    monkeypatch.setattr(s, "_lib", None)
    monkeypatch.setattr(s, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        s.lib()


_C_PROGRAM = r"""
#include <stdio.h>
#include "ssm.h"
int main(void) {
  /* every call returns from the host-side checks: nothing touches a GPU */
  ssm_status st = ssm_selective_scan_fwd(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, NULL, NULL, 0, NULL,
                                         NULL, NULL, NULL, NULL, 1, 4, 8, 16, SSM_F32, 0, NULL, 0, 0u, NULL);
  printf("%d %s %s %zu %zu\n", ssm_version(), ssm_status_string(SSM_OK), ssm_status_string(st),
         ssm_ssd_workspace_bytes(1, 128, 1, 64, 128, SSM_BF16), ssm_ssd_workspace_bytes(1, 128, 1, 32, 128, SSM_BF16));
  return 0;
}
"""


def test_header_is_plain_c_and_links(L, tmp_path):
    """A C99 program (no C++, no torch) includes include/ssm.h under -pedantic -Werror, links
    libssm.so and calls it; the header also compiles as C++."""
    import shutil
    import subprocess

    import selective_state_space_145_b300 as ssm

    gcc = shutil.which("gcc")
    assert gcc, "gcc is part of the toolchain"
    src = tmp_path / "abi.c"
    src.write_text(_C_PROGRAM)
    libdir = os.path.dirname(ssm.LIB_PATH)
    exe = tmp_path / "abi"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(src), "-L", libdir, "-lssm", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert out == [str(ssm.version()), "SSM_OK", "SSM_ERR_INVALID_ARG", "256", "0"]
    gxx = shutil.which("g++")
    if gxx:
        subprocess.run([gxx, "-std=c++17", "-Wall", "-Wextra", "-Werror", "-x", "c++", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), str(src)], check=True)


def test_default_chunk_policy_one_wave_rule(L):
    """The default chunking on a 148-SM part with the resident CTAs the shared-memory limit
    allows (the figures the library assumes when no device answers). A main-pass CTA is one
    warp. With two lanes of 8 states per channel it covers 16 channels, and 7 bf16 or 5 fp32
    CTAs fit an SM; a problem whose CTAs then fill more than half a wave runs unchunked.
    Otherwise the sequence is split and the main pass takes whole channels per lane (two
    channels of 16 states per lane, 64 channels per CTA, 16-step tiles, 9 bf16 or 5 fp32 CTAs
    per SM): split only as far as the chunks' CTAs still fit one wave, in multiples of 64
    steps, and cut chunks of a split sequence to at most 3072 steps."""
    import selective_state_space_145_b300 as ssm
    import torch

    f32, bf16 = torch.float32, torch.bfloat16
    resident1 = {f32: 148 * 5, bf16: 148 * 9}
    # fp32 block workload: 128 two-lane CTAs fit easily -> split; 32 whole-channel CTAs, 23
    # chunks would fit a wave, the sequence allows 16 -> chunks of 64
    assert ssm.ssm_scan_default_chunk_len(2, 1024, 1024, 16, f32) == 64
    # bf16 block workload: 1024 two-lane CTAs already more than half a wave -> one chunk
    assert ssm.ssm_scan_default_chunk_len(8, 2048, 2048, 16, bf16) == 2048
    # long scan: 24 whole-channel CTAs, 55 chunks fit a wave -> 131072 / 55 rounded up to 64
    assert ssm.ssm_scan_default_chunk_len(1, 1536, 131072, 16, bf16) == 2432
    # small scan: 1 whole-channel CTA; 4 chunks of 64 steps (the sequence allows no more)
    assert ssm.ssm_scan_default_chunk_len(1, 64, 256, 16, f32) == 64
    for io in (f32, bf16):
        for batch, dim, L_ in ((1, 1536, 32768), (3, 700, 5000), (1, 33, 70000)):
            cl = ssm.ssm_scan_default_chunk_len(batch, dim, L_, 16, io)
            ctas = (dim + 63) // 64 * batch
            q = (L_ + cl - 1) // cl
            assert cl % 64 == 0 and cl <= max(3072, (L_ + 63) // 64 * 64)
            assert q == 1 or q * ctas <= resident1[io] or cl == 3072


def test_scan_workspace_stays_far_below_a_per_step_state(L):
    """Memory is linear in the sequence only through the chunk count: the default chunking's
    workspace holds (chunks - 1) carries of N + 1 floats per channel, never a state per step."""
    import selective_state_space_145_b300 as ssm
    import torch

    batch, dim, N = 1, 1536, 16
    prev = -1
    for L_ in (1024, 8192, 65536, 131072, 524288):
        cl = ssm.ssm_scan_default_chunk_len(batch, dim, L_, N, torch.bfloat16)
        ws = ssm.ssm_scan_workspace_bytes(batch, dim, L_, N, 0, torch.bfloat16)
        q = (L_ + cl - 1) // cl
        assert ws <= (q - 1) * batch * dim * (N + 1) * 4 + 256
        # a per-step state would be L x N floats; chunks of at least 64 steps keep the carries
        # (N + 1 floats per chunk) at least 64 N / (N + 1) ~ 60 times smaller
        assert ws * 50 < batch * dim * L_ * N * 4
        assert ws >= prev                                     # grows with L, at most linearly
        prev = ws


def test_release_library_has_no_bounds_checks(L):
    """ssm_debug_bounds_status answers SSM_ERR_UNSUPPORTED from the release library (no check
    compiled in, no CUDA call made) and rejects a NULL word or a bad clear flag."""
    word = ctypes.c_uint(7)
    assert L.ssm_debug_bounds_status(ctypes.byref(word), 0) == 2
    assert word.value == 7
    assert L.ssm_debug_bounds_status(None, 0) == 1
    assert L.ssm_debug_bounds_status(ctypes.byref(word), 2) == 1


def test_debug_library_builds_and_exports_every_symbol():
    """libssm_debug.so (SSM_DEBUG_BOUNDS) builds, loads beside the release library and exports
    the same entry points; its argument checks are the release library's."""
    from selective_state_space_145_b300 import build

    path = build.build(variant="debug")
    D = ctypes.CDLL(path)
    for name in _declared_symbols():
        assert hasattr(D, name), name
    D.ssm_version.restype = ctypes.c_int
    import selective_state_space_145_b300 as ssm

    assert D.ssm_version() == ssm.version()
    D.ssm_debug_bounds_status.restype = ctypes.c_int
    assert D.ssm_debug_bounds_status(None, 0) == 1  # host-side argument check, before any CUDA call
    D.ssm_scan_workspace_bytes.restype = ctypes.c_size_t
    assert D.ssm_scan_workspace_bytes(1, 1536, 131072, 16, 1, 0) == ssm.lib().ssm_scan_workspace_bytes(
        1, 1536, 131072, 16, 1, 0)


def test_library_selection_routes_the_binding():
    import selective_state_space_145_b300 as ssm

    try:
        ssm.select_library("debug")
        assert ssm.library_path() == ssm.DEBUG_LIB_PATH
        ssm.select_library("release")
        assert ssm.library_path() == ssm.LIB_PATH
        with pytest.raises(ValueError):
            ssm.select_library("fast")
    finally:
        ssm.select_library("release")
    with pytest.raises(ssm.SSMError, match="UNSUPPORTED"):
        ssm.debug_bounds_status()


def test_s4d_real_bit_only_on_the_scan(L):
    """SSM_SCAN_S4D_REAL is an option of ssm_selective_scan_fwd; the segment aggregate and the
    decode step refuse it on the host (SSM_ERR_INVALID_ARG)."""
    import selective_state_space_145_b300 as ssm

    assert ssm.SCAN_S4D_REAL == 4
    assert L.ssm_selective_scan_aggregate(None, None, None, None, None, 1, None, None, 0, None, None, None,
                                          1, 8, 16, 16, 0, None, 0, ssm.SCAN_S4D_REAL, None) == 1
    assert L.ssm_selective_state_update(None, None, None, None, None, None, None, None, None, None, 1, None, None, 0,
                                        None, 1, 8, 16, 0, ssm.SCAN_S4D_REAL, None) == 1

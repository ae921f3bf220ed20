"""Pins of the fp64 CPU oracle against what the pages and the mathematics fix.

Each test ties the oracle to something other than itself: a closed form, a
limit, brute-force products on tiny inputs, a library routine for a special
case, an invariant of the method, or a worked example. Together they are chosen
so that a dropped term, a wrong sign or index, or a transposed operand in the
oracle fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

RNG = np.random.default_rng(145)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(*shape):
    return RNG.standard_normal(shape)


def _neg_A(dim, N, lo=0.2, hi=2.0):
    return -RNG.uniform(lo, hi, size=(dim, N))


def _silu_lib(x):
    return F.silu(torch.as_tensor(x, dtype=torch.float64)).numpy()


# ---------------------------------------------------------------- library special cases

def test_softplus_matches_torch():
    # "Mamba" (ai360xpert.com), selection mechanism: Delta = softplus(.)
    x = np.concatenate([np.linspace(-60, 60, 2001), _rand(1000) * 5])
    ref = F.softplus(torch.as_tensor(x), beta=1.0, threshold=1e4).numpy()
    np.testing.assert_allclose(oracle.softplus(x), ref, rtol=5e-16, atol=0)


def test_silu_matches_torch():
    x = np.concatenate([np.linspace(-40, 40, 801), _rand(1000) * 4])
    np.testing.assert_allclose(oracle.silu(x), _silu_lib(x), rtol=4e-16, atol=1e-300)


@pytest.mark.parametrize("K", [2, 3, 4])
def test_causal_conv_matches_torch_conv1d(K):
    # "Overview of Mamba (SSM) Model", block: depthwise causal conv then SiLU.
    b, d, L = 2, 5, 19
    x, w, bias = _rand(b, d, L), _rand(d, K), _rand(d)
    ref = F.conv1d(torch.as_tensor(x), torch.as_tensor(w)[:, None, :], torch.as_tensor(bias),
                   padding=K - 1, groups=d)[..., :L].numpy()
    np.testing.assert_allclose(oracle.causal_conv1d(x, w, bias, apply_silu=False), ref, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(oracle.causal_conv1d(x, w, bias, apply_silu=True), _silu_lib(ref),
                               rtol=1e-14, atol=1e-14)
    # a supplied window plays the role of the inputs before t = 0
    win = _rand(b, d, K - 1)
    ref_w = F.conv1d(torch.as_tensor(np.concatenate([win, x], axis=-1)), torch.as_tensor(w)[:, None, :],
                     torch.as_tensor(bias), groups=d).numpy()
    np.testing.assert_allclose(oracle.causal_conv1d(x, w, bias, window=win, apply_silu=False), ref_w,
                               rtol=1e-14, atol=1e-14)


def test_scan_with_conv_equals_conv_then_scan():
    # the fused prologue is the library conv (+SiLU) followed by the plain scan
    b, d, L, N, K = 2, 3, 23, 4, 4
    x, delta, z = _rand(b, d, L), 0.5 * _rand(b, d, L), _rand(b, d, L)
    A, B, C, D, bias = _neg_A(d, N), _rand(b, N, L), _rand(b, N, L), _rand(d), _rand(d) - 2
    w, cb = RNG.uniform(-0.5, 0.5, (d, K)), _rand(d)
    u = _silu_lib(F.conv1d(torch.as_tensor(x), torch.as_tensor(w)[:, None, :], torch.as_tensor(cb),
                           padding=K - 1, groups=d)[..., :L].numpy())
    out1, h1 = oracle.selective_scan(x, delta, A, B, C, D, z, bias, True, w, cb)
    out2, h2 = oracle.selective_scan(u, delta, A, B, C, D, z, bias, True)
    np.testing.assert_allclose(out1, out2, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(h1, h2, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- closed forms

def test_lti_closed_form_convolution():
    """Delta, B, C constant in t: the scan is the LTI convolution
    y_t = sum_k (sum_n C_n Abar_n^k Delta B_n) u_{t-k} + sum_n C_n Abar_n^{t+1} h0_n + D u_t
    ("Mamba" ai360xpert.com: fixed-Delta SSM; "Mamba" ozercemkelahmet.com, step 1-2)."""
    b, d, L, N = 2, 3, 40, 4
    Delta = RNG.uniform(0.05, 0.6, (b, d))
    Bc, Cc = _rand(b, N), _rand(b, N)
    A, D, u, z, h0 = _neg_A(d, N), _rand(d), _rand(b, d, L), _rand(b, d, L), _rand(b, d, N)
    delta = np.repeat(Delta[:, :, None], L, axis=2)
    B = np.repeat(Bc[:, :, None], L, axis=2)
    C = np.repeat(Cc[:, :, None], L, axis=2)
    out, h_last = oracle.selective_scan(u, delta, A, B, C, D, z, None, False, h0=h0)
    ref = np.zeros((b, d, L))
    for bi in range(b):
        for di in range(d):
            Abar = np.exp(Delta[bi, di] * A[di])                                   # [N]
            kern = np.array([np.sum(Cc[bi] * Abar ** k * Delta[bi, di] * Bc[bi]) for k in range(L)])
            y = np.convolve(u[bi, di], kern)[:L] + D[di] * u[bi, di]
            y += np.array([np.sum(Cc[bi] * Abar ** (t + 1) * h0[bi, di]) for t in range(L)])
            ref[bi, di] = y * _silu_lib(z[bi, di])
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_lti_constant_input_geometric_sum():
    """Constant u, Delta, B: h_t[n] = Delta B_n u (1 - Abar_n^{t+1}) / (1 - Abar_n) from h = 0."""
    d, L, N = 3, 57, 5
    Delta = RNG.uniform(0.01, 0.3, (1, d))
    Bc, A = _rand(1, N), _neg_A(d, N)
    uval = 1.7
    u = np.full((1, d, L), uval)
    delta = np.repeat(Delta[:, :, None], L, axis=2)
    B = np.repeat(Bc[:, :, None], L, axis=2)
    C = _rand(1, N, L)
    _, _, trace = oracle.selective_scan(u, delta, A, B, C, None, None, None, False, want_trace=True)
    for di in range(d):
        Abar = np.exp(Delta[0, di] * A[di])
        for t in (0, 1, 10, L - 1):
            ref = Delta[0, di] * Bc[0] * uval * (1 - Abar ** (t + 1)) / (1 - Abar)
            np.testing.assert_allclose(trace[0, di, t], ref, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- limits of the step size

def test_small_delta_keeps_state():
    """Delta -> 0: Abar -> 1 and Bbar -> 0, so h_t = h0 and y_t = C_t.h0 + D u_t
    ("Mamba" ai360xpert.com: small Delta keeps the state; "Mamba" ozercemkelahmet.com step 3)."""
    b, d, L, N = 2, 3, 33, 4
    x, z, B, C = _rand(b, d, L), _rand(b, d, L), _rand(b, N, L), _rand(b, N, L)
    A, D, h0 = _neg_A(d, N), _rand(d), _rand(b, d, N)
    delta = np.full((b, d, L), -40.0)                     # softplus(-40) ~ 4.2e-18
    out, h_last = oracle.selective_scan(x, delta, A, B, C, D, z, np.zeros(d), True, h0=h0)
    np.testing.assert_allclose(h_last, h0, rtol=1e-15, atol=1e-15)
    ref = (np.einsum("bnt,bdn->bdt", C, h0) + D[None, :, None] * x) * _silu_lib(z)
    np.testing.assert_allclose(out, ref, rtol=1e-14, atol=1e-14)


def test_large_delta_forgets_past():
    """Large Delta with A <= -1: Abar ~ 0, so the output is memoryless:
    y_t = Delta u_t (C_t . B_t) + D u_t ("Mamba" ai360xpert.com: large Delta resets the state)."""
    b, d, L, N = 2, 3, 29, 4
    x, z, B, C = _rand(b, d, L), _rand(b, d, L), _rand(b, N, L), _rand(b, N, L)
    A, D, h0 = -1.0 - RNG.uniform(0, 1, (d, N)), _rand(d), _rand(b, d, N)
    delta = np.full((b, d, L), 40.0)
    out, h_last = oracle.selective_scan(x, delta, A, B, C, D, z, np.zeros(d), True, h0=h0)
    Delta = 40.0 + math.log1p(math.exp(-40.0))
    ref = (Delta * x * np.einsum("bnt,bnt->bt", C, B)[:, None, :] + D[None, :, None] * x) * _silu_lib(z)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(h_last, Delta * B[:, None, :, -1] * x[:, :, -1:], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- brute force

def _brute_force(x, delta, A, B, C, D, z, bias, w, cb, win, h0):
    """Unrolled: h_T = (prod_{r<=T} Abar_r) h0 + sum_s (prod_{r=s+1}^{T} Abar_r) Bbar_s u_s, scalars only."""
    b, d, L = x.shape
    N = A.shape[1]
    K = w.shape[1]
    out = np.zeros((b, d, L))
    hL = np.zeros((b, d, N))
    for bi in range(b):
        for di in range(d):
            stream = list(win[bi, di]) + list(x[bi, di])
            u = []
            for t in range(L):
                acc = sum(w[di, k] * stream[t + k] for k in range(K)) + cb[di]
                u.append(acc / (1.0 + math.exp(-acc)))
            Dl = [math.log1p(math.exp(delta[bi, di, t] + bias[di])) for t in range(L)]
            for T in range(L):
                y = 0.0
                for n in range(N):
                    Abar = [math.exp(Dl[r] * A[di, n]) for r in range(L)]
                    p0 = 1.0
                    for r in range(T + 1):
                        p0 *= Abar[r]
                    hT = p0 * h0[bi, di, n]
                    for s in range(T + 1):
                        p = 1.0
                        for r in range(s + 1, T + 1):
                            p *= Abar[r]
                        hT += p * Dl[s] * B[bi, n, s] * u[s]
                    y += C[bi, n, T] * hT
                    if T == L - 1:
                        hL[bi, di, n] = hT
                y += D[di] * u[T]
                out[bi, di, T] = y * z[bi, di, T] / (1.0 + math.exp(-z[bi, di, T]))
    return out, hL


def test_brute_force_tiny():
    b, d, L, N, K = 2, 3, 7, 3, 3
    x, delta, z = _rand(b, d, L), 0.8 * _rand(b, d, L), _rand(b, d, L)
    A, B, C, D, bias = _neg_A(d, N), _rand(b, N, L), _rand(b, N, L), _rand(d), _rand(d) - 1
    w, cb, win, h0 = RNG.uniform(-0.5, 0.5, (d, K)), _rand(d), _rand(b, d, K - 1), _rand(b, d, N)
    out, hL = oracle.selective_scan(x, delta, A, B, C, D, z, bias, True, w, cb, conv_init=win, h0=h0)
    ref, refL = _brute_force(x, delta, A, B, C, D, z, bias, w, cb, win, h0)
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(hL, refL, rtol=1e-13, atol=1e-13)


def _brute_force_backward(x, delta, A, B, C, D, z, bias, w, cb, ahead, h0):
    """The backward scan written directly, t = L-1 down to 0: the conv reads x at t .. t+K-1
    (w[K-1] on x_t, w[0] on x_{t+K-1}; positions past the end come from `ahead`, ahead[j]
    being the input at L+K-2-j), and h_t = exp(Delta_t A) h_{t+1} + Delta_t B_t u_t from
    h_L = h0. Scalars only, no re-indexing of arrays."""
    b, d, L = x.shape
    N = A.shape[1]
    K = w.shape[1]
    out = np.zeros((b, d, L))
    hL = np.zeros((b, d, N))
    for bi in range(b):
        for di in range(d):
            def xs(s):
                return x[bi, di, s] if s < L else ahead[bi, di, L + K - 2 - s]
            h = [h0[bi, di, n] for n in range(N)]
            for t in range(L - 1, -1, -1):
                acc = sum(w[di, k] * xs(t + K - 1 - k) for k in range(K)) + cb[di]
                u = acc / (1.0 + math.exp(-acc))
                Dl = math.log1p(math.exp(delta[bi, di, t] + bias[di]))
                y = 0.0
                for n in range(N):
                    h[n] = math.exp(Dl * A[di, n]) * h[n] + Dl * B[bi, n, t] * u
                    y += C[bi, n, t] * h[n]
                y += D[di] * u
                out[bi, di, t] = y * z[bi, di, t] / (1.0 + math.exp(-z[bi, di, t]))
            hL[bi, di] = h
    return out, hL


def test_backward_scan_brute_force():
    b, d, L, N, K = 2, 3, 9, 3, 4
    x, delta, z = _rand(b, d, L), 0.8 * _rand(b, d, L), _rand(b, d, L)
    A, B, C, D, bias = _neg_A(d, N), _rand(b, N, L), _rand(b, N, L), _rand(d), _rand(d) - 1
    w, cb, ahead, h0 = RNG.uniform(-0.5, 0.5, (d, K)), _rand(d), _rand(b, d, K - 1), _rand(b, d, N)
    out, hL, cs = oracle.selective_scan(x, delta, A, B, C, D, z, bias, True, w, cb, conv_init=ahead, h0=h0,
                                        want_conv_state=True, reverse=True)
    ref, refL = _brute_force_backward(x, delta, A, B, C, D, z, bias, w, cb, ahead, h0)
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(hL, refL, rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(cs, x[:, :, K - 2::-1])   # x at K-2, ..., 0


def test_backward_scan_split_equals_whole():
    """The backward scan over [0, L) equals the backward scan over [L1, L) followed by the one
    over [0, L1) started from its end state and raw-input window."""
    p = _problem()
    L = p["x"].shape[-1]
    full, hfull, csfull = oracle.selective_scan(**p, want_conv_state=True, reverse=True)
    for L1 in (1, 5, 13, L - 1):
        late = {k: (v[..., L1:] if k in ("x", "delta", "z", "B", "C") else v) for k, v in p.items()}
        out2, h2, cs2 = oracle.selective_scan(**late, want_conv_state=True, reverse=True)
        early = {k: (v[..., :L1] if k in ("x", "delta", "z", "B", "C") else v) for k, v in p.items()}
        early["h0"], early["conv_init"] = h2, cs2
        out1, h1, cs1 = oracle.selective_scan(**early, want_conv_state=True, reverse=True)
        np.testing.assert_array_equal(np.concatenate([out1, out2], axis=-1), full)
        np.testing.assert_array_equal(h1, hfull)
        np.testing.assert_array_equal(cs1, csfull)


# ---------------------------------------------------------------- zero-order hold (zoh=True)

def test_zoh_is_exact_for_piecewise_constant_input():
    """With a constant input u, B, A and h(0) = h0, the continuous system h' = A h + B u has
    h(T) = e^{A T} h0 + (B u / -A)(1 - e^{A T}). Zero-order hold is exact for inputs held
    constant over each step, so after steps of any lengths Delta_t the discrete state equals
    the solution at T = sum of Delta_t ("Mamba", ai360xpert.com, "Show Me the Code")."""
    b, d, L, N = 1, 3, 40, 5
    A = _neg_A(d, N, 0.05, 3.0)
    uval, Bval, h0 = 0.7, RNG.standard_normal(N), RNG.standard_normal((b, d, N))
    x = np.full((b, d, L), uval)
    B = np.repeat(Bval[None, :, None], L, axis=2).reshape(b, N, L)
    delta = RNG.uniform(0.01, 0.6, (b, d, L))                  # softplus off: Delta = delta
    C = np.zeros((b, N, L))
    _, hL, tr = oracle.selective_scan(x, delta, A, B, C, h0=h0, delta_softplus=False, want_trace=True, zoh=True)
    T = np.cumsum(delta, axis=-1)                             # [b, d, L]
    for t in (0, 7, L - 1):
        eAT = np.exp(A[None] * T[:, :, t:t + 1])              # [b, d, N]
        ref = eAT * h0 + (Bval[None, None, :] * uval / -A[None]) * (1.0 - eAT)
        np.testing.assert_allclose(tr[:, :, t, :], ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(hL, tr[:, :, -1, :], rtol=0, atol=0)


def test_zoh_tends_to_euler_as_A_vanishes():
    """expm1(Delta A)/A -> Delta as A -> 0: with A = -1e-9 both rules agree to ~1e-9 relative,
    and A = 0 exactly takes the limit."""
    p = _problem(L=30)
    for a in (-1e-9, 0.0):
        q = dict(p, A=np.full_like(p["A"], a))
        e_out, e_h = oracle.selective_scan(**q)
        z_out, z_h = oracle.selective_scan(**q, zoh=True)
        np.testing.assert_allclose(z_out, e_out, rtol=1e-7, atol=1e-9)
        np.testing.assert_allclose(z_h, e_h, rtol=1e-7, atol=1e-9)


def test_zoh_brute_force_tiny():
    """Scalar loop with Bbar = (1 - exp(Delta A)) / (-A) B written as the pages print it."""
    b, d, L, N = 1, 2, 6, 3
    x, delta, z = _rand(b, d, L), 0.8 * _rand(b, d, L), _rand(b, d, L)
    A, B, C, D, bias = _neg_A(d, N), _rand(b, N, L), _rand(b, N, L), _rand(d), _rand(d) - 1
    out, hL = oracle.selective_scan(x, delta, A, B, C, D, z, bias, True, zoh=True)
    for di in range(d):
        h = [0.0] * N
        for t in range(L):
            Dl = math.log1p(math.exp(delta[0, di, t] + bias[di]))
            y = 0.0
            for n in range(N):
                Ab = math.exp(Dl * A[di, n])
                h[n] = Ab * h[n] + (1.0 - Ab) / (-A[di, n]) * B[0, n, t] * x[0, di, t]
                y += C[0, n, t] * h[n]
            y += D[di] * x[0, di, t]
            ref = y * z[0, di, t] / (1.0 + math.exp(-z[0, di, t]))
            assert abs(out[0, di, t] - ref) <= 1e-12 * (1 + abs(ref))
        np.testing.assert_allclose(hL[0, di], h, rtol=1e-12, atol=1e-13)


def test_zoh_decode_equals_scan():
    """One ZOH decode step per token equals the ZOH scan over the same tokens."""
    p = _problem(L=6)
    out, hL, cs = oracle.selective_scan(**p, want_conv_state=True, zoh=True)
    state, win = p["h0"], p["conv_init"]
    for t in range(6):
        y, state, win = oracle.state_update(state, win, p["x"][..., t], p["delta"][..., t], p["A"], p["B"][..., t],
                                            p["C"][..., t], p["D"], p["z"][..., t], p["delta_bias"], True,
                                            p["conv_w"], p["conv_b"], zoh=True)
        np.testing.assert_allclose(y, out[..., t], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(state, hL, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(win, cs)


# ---------------------------------------------------------------- backward pass

def _bwd_problem(b=2, d=3, L=9, N=3):
    return dict(u=_rand(b, d, L), delta=0.7 * _rand(b, d, L), A=_neg_A(d, N), B=_rand(b, N, L),
                C=_rand(b, N, L), D=_rand(d), z=_rand(b, d, L), delta_bias=_rand(d) - 1.0, h0=_rand(b, d, N))


def _loss(p, dout, dhl):
    out, hL = oracle.selective_scan(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"], p["delta_bias"],
                                    True, h0=p["h0"])
    return float(np.sum(dout * out) + np.sum(dhl * hL))


def test_backward_matches_finite_differences():
    """Every gradient of L = sum(dout * out) + sum(dh_last * h_last) against central differences
    of the forward oracle, element by element."""
    p = _bwd_problem()
    dout, dhl = _rand(*p["u"].shape), _rand(*p["h0"].shape)
    g = oracle.selective_scan_bwd(p["u"], p["delta"], p["A"], p["B"], p["C"], dout, p["D"], p["z"],
                                  p["delta_bias"], True, p["h0"], dhl)
    names = {"u": "du", "delta": "ddelta", "z": "dz", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "delta_bias": "ddelta_bias", "h0": "dh0"}
    eps = 1e-6
    for key, gk in names.items():
        num = np.empty_like(p[key])
        for idx in np.ndindex(p[key].shape):
            q = {k: v.copy() for k, v in p.items()}
            q[key][idx] += eps
            lp = _loss(q, dout, dhl)
            q[key][idx] -= 2 * eps
            lm = _loss(q, dout, dhl)
            num[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g[gk], num, rtol=1e-6, atol=1e-7, err_msg=key)


def _torch_scan(u, delta, A, B, C, D, z, bias, h0):
    """The forward as tensor algebra over all channels at once (independent of the C oracle)."""
    Dl = F.softplus(delta + bias[None, :, None])                  # [b, d, L]
    h = h0
    ys = []
    for t in range(u.shape[-1]):
        Ab = torch.exp(Dl[:, :, t, None] * A[None])               # [b, d, N]
        h = Ab * h + Dl[:, :, t, None] * B[:, None, :, t] * u[:, :, t, None]
        ys.append((h * C[:, None, :, t]).sum(-1) + D[None] * u[:, :, t])
    y = torch.stack(ys, dim=-1)
    return y * F.silu(z), h


def test_backward_matches_autograd():
    """The oracle's gradients equal torch autograd through an independent fp64 forward."""
    p = _bwd_problem(b=2, d=4, L=17, N=5)
    dout, dhl = _rand(*p["u"].shape), _rand(*p["h0"].shape)
    tp = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in p.items()}
    out, hL = _torch_scan(tp["u"], tp["delta"], tp["A"], tp["B"], tp["C"], tp["D"], tp["z"], tp["delta_bias"],
                          tp["h0"])
    ((out * torch.tensor(dout)).sum() + (hL * torch.tensor(dhl)).sum()).backward()
    g = oracle.selective_scan_bwd(p["u"], p["delta"], p["A"], p["B"], p["C"], dout, p["D"], p["z"],
                                  p["delta_bias"], True, p["h0"], dhl)
    for key, gk in {"u": "du", "delta": "ddelta", "z": "dz", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
                    "delta_bias": "ddelta_bias", "h0": "dh0"}.items():
        np.testing.assert_allclose(g[gk], tp[key].grad.numpy(), rtol=1e-11, atol=1e-12, err_msg=key)


def test_conv_backward_matches_autograd_conv1d():
    """The conv backward against torch autograd through F.conv1d (groups = channels, left
    padding supplied by the window), with and without SiLU."""
    b, d, L, K = 2, 5, 13, 4
    x, w, bias, win, dout = _rand(b, d, L), RNG.uniform(-0.5, 0.5, (d, K)), _rand(d), _rand(b, d, K - 1), _rand(b, d, L)
    for act in (True, False):
        g = oracle.causal_conv1d_bwd(x, w, dout, bias, win, apply_silu=act)
        tx, tw, tb, twin = (torch.tensor(v, requires_grad=True) for v in (x, w, bias, win))
        y = F.conv1d(torch.cat([twin, tx], dim=-1), tw[:, None, :], tb, groups=d)
        if act:
            y = F.silu(y)
        (y * torch.tensor(dout)).sum().backward()
        np.testing.assert_allclose(g["dx"], tx.grad.numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(g["dw"], tw.grad.numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(g["dbias"], tb.grad.numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(g["dwindow"], twin.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_conv_backward_matches_finite_differences():
    b, d, L, K = 1, 3, 7, 3
    x, w, bias, win, dout = _rand(b, d, L), RNG.uniform(-0.5, 0.5, (d, K)), _rand(d), _rand(b, d, K - 1), _rand(b, d, L)
    g = oracle.causal_conv1d_bwd(x, w, dout, bias, win)
    p = {"x": x, "w": w, "bias": bias, "window": win}
    eps = 1e-6
    for key, gk in (("x", "dx"), ("w", "dw"), ("bias", "dbias"), ("window", "dwindow")):
        num = np.empty_like(p[key])
        for idx in np.ndindex(p[key].shape):
            q = {k: v.copy() for k, v in p.items()}
            q[key][idx] += eps
            lp = float(np.sum(dout * oracle.causal_conv1d(q["x"], q["w"], q["bias"], q["window"])))
            q[key][idx] -= 2 * eps
            lm = float(np.sum(dout * oracle.causal_conv1d(q["x"], q["w"], q["bias"], q["window"])))
            num[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g[gk], num, rtol=1e-6, atol=1e-8, err_msg=key)


# ---------------------------------------------------------------- invariants

def _problem(b=2, d=3, L=21, N=4, K=4):
    return dict(x=_rand(b, d, L), delta=0.7 * _rand(b, d, L), A=_neg_A(d, N), B=_rand(b, N, L), C=_rand(b, N, L),
                D=_rand(d), z=_rand(b, d, L), delta_bias=_rand(d) - 1.5, conv_w=RNG.uniform(-0.5, 0.5, (d, K)),
                conv_b=_rand(d), conv_init=_rand(b, d, K - 1), h0=_rand(b, d, N))


def test_chunked_prompt_equals_whole_prompt():
    """Processing a prompt in two calls that pass on (h, conv window) equals one call
    ("Mamba" ozercemkelahmet.com, deployment notes: chunks pass the state on)."""
    p = _problem()
    L = p["x"].shape[-1]
    full, hfull, csfull = oracle.selective_scan(**p, want_conv_state=True)
    for L1 in range(1, L):
        a = {k: (v[..., :L1] if k in ("x", "delta", "z", "B", "C") else v) for k, v in p.items()}
        out1, h1, cs1 = oracle.selective_scan(**a, want_conv_state=True)
        bpart = {k: (v[..., L1:] if k in ("x", "delta", "z", "B", "C") else v) for k, v in p.items()}
        bpart["h0"], bpart["conv_init"] = h1, cs1
        out2, h2, cs2 = oracle.selective_scan(**bpart, want_conv_state=True)
        np.testing.assert_array_equal(np.concatenate([out1, out2], axis=-1), full)
        np.testing.assert_array_equal(h2, hfull)
        np.testing.assert_array_equal(cs2, csfull)


def test_recurrent_mode_equals_parallel_mode():
    """K decode steps from (state, window) equal one scan over the same K tokens with
    h0 = state and the conv window as the inputs before t = 0
    ("Mamba" ozercemkelahmet.com, sanity checks: recurrent and parallel mode agree)."""
    p = _problem(L=9)
    out, hL, cs = oracle.selective_scan(**p, want_conv_state=True)
    state, window = p["h0"], p["conv_init"]
    for t in range(p["x"].shape[-1]):
        y, state, window = oracle.state_update(state, window, p["x"][..., t], p["delta"][..., t], p["A"],
                                               p["B"][..., t], p["C"][..., t], p["D"], p["z"][..., t],
                                               p["delta_bias"], True, p["conv_w"], p["conv_b"])
        np.testing.assert_array_equal(y, out[..., t])
    np.testing.assert_array_equal(state, hL)
    np.testing.assert_array_equal(window, cs)


def test_compose_is_function_composition_and_associative():
    n = 1000
    a1, a2, a3 = (RNG.uniform(0, 1, n) for _ in range(3))
    b1, b2, b3 = (_rand(n) for _ in range(3))
    h = _rand(n)
    a12, b12 = oracle.compose(a1, b1, a2, b2)
    # applying (a1, b1) then (a2, b2) to h
    np.testing.assert_allclose(a12 * h + b12, a2 * (a1 * h + b1) + b2, rtol=1e-14, atol=1e-14)
    left = oracle.compose(a12, b12, a3, b3)
    a23, b23 = oracle.compose(a2, b2, a3, b3)
    right = oracle.compose(a1, b1, a23, b23)
    np.testing.assert_allclose(left[0], right[0], rtol=1e-15, atol=0)
    np.testing.assert_allclose(left[1], right[1], rtol=1e-14, atol=1e-14)
    one, zero = np.ones(n), np.zeros(n)
    for got in (oracle.compose(one, zero, a1, b1), oracle.compose(a1, b1, one, zero)):
        np.testing.assert_array_equal(got[0], a1)
        np.testing.assert_array_equal(got[1], b1)


@pytest.mark.parametrize("chunk", [1, 4, 5, 8, 21, 64])
def test_chunk_carry_equals_sequential(chunk):
    """Chunk aggregates composed in order give the state at every chunk boundary, and each
    chunk rerun from that state reproduces the sequential output (the cross-chunk carry)."""
    p = _problem(L=21)
    L = p["x"].shape[-1]
    out, hL, trace = oracle.selective_scan(**p, want_trace=True)
    agg_a, agg_b = oracle.chunk_aggregates(p["x"], p["delta"], p["A"], p["B"], p["delta_bias"], True,
                                           p["conv_w"], p["conv_b"], p["conv_init"], chunk_len=chunk)
    h = p["h0"].copy()
    K = p["conv_w"].shape[1]
    stream = np.concatenate([p["conv_init"], p["x"]], axis=-1)
    for q in range(agg_a.shape[2]):
        t0, t1 = q * chunk, min(L, (q + 1) * chunk)
        sub = {k: (v[..., t0:t1] if k in ("x", "delta", "z", "B", "C") else v) for k, v in p.items()}
        sub["h0"], sub["conv_init"] = h, stream[..., t0:t0 + K - 1]
        o, _ = oracle.selective_scan(**sub)
        np.testing.assert_allclose(o, out[..., t0:t1], rtol=1e-12, atol=1e-12)
        h = agg_a[:, :, q] * h + agg_b[:, :, q]
        np.testing.assert_allclose(h, trace[:, :, t1 - 1], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(h, hL, rtol=1e-12, atol=1e-12)


def test_decay_is_monotone_without_input():
    """A < 0 and Delta > 0 give 0 < Abar < 1: with no input the state shrinks every step."""
    b, d, L, N = 1, 4, 50, 6
    x, delta = _rand(b, d, L), _rand(b, d, L)
    out, hL, trace = oracle.selective_scan(x, delta, _neg_A(d, N), np.zeros((b, N, L)), _rand(b, N, L),
                                           None, None, np.zeros(d), True, h0=_rand(b, d, N), want_trace=True)
    ratio = trace[:, :, 1:] / trace[:, :, :-1]
    assert np.all(ratio > 0) and np.all(ratio < 1)


def test_decode_window_shifts_raw_inputs():
    """The decode window keeps the last K-1 raw inputs, oldest first."""
    d, N, K = 3, 2, 4
    win = _rand(1, d, K - 1)
    xs = _rand(5, 1, d)
    state = np.zeros((1, d, N))
    for t in range(5):
        _, state, win2 = oracle.state_update(state, win, xs[t], np.zeros((1, d)), _neg_A(d, N), _rand(1, N),
                                             _rand(1, N), None, None, None, True, RNG.uniform(-1, 1, (d, K)), None)
        np.testing.assert_array_equal(win2, np.concatenate([win[..., 1:], xs[t][..., None]], axis=-1))
        win = win2


# ---------------------------------------------------------------- worked example

def test_scalar_walkthrough_golden():
    """The pages' scalar walk-through with the step sizes fixed by the fixture."""
    with open(os.path.join(GOLDEN, "scalar_walkthrough.json")) as f:
        g = json.load(f)
    L = len(g["inputs"])
    x = np.array(g["inputs"], dtype=np.float64).reshape(1, 1, L)
    Delta = np.array([math.log(v) for v in g["delta_as_log_of"]]).reshape(1, 1, L)
    A = np.array([[-g["a"]]])
    ones = np.ones((1, 1, L))
    out, hL, tr = oracle.selective_scan(x, Delta, A, ones, ones, None, None, None, False, want_trace=True)
    ln2 = math.log(2.0)
    expect = np.array([num / den * ln2 for num, den in g["state_over_ln2"]])
    np.testing.assert_allclose(tr[0, 0, :, 0], expect, rtol=1e-14, atol=0)
    np.testing.assert_allclose(out[0, 0], expect, rtol=1e-14, atol=0)

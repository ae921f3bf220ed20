"""Pins of the fp64 oracle of the multi-head SSM with one decay per head (the layer of the
state-space duality), against things other than itself:

* the dual view ("Mamba", ozercemkelahmet.com, "Mamba-2 and the dual view": the layer written as
  a masked matrix product with a decaying mask), computed here by brute force from that form;
* the selective-scan oracle, already pinned on its own, to which the layer reduces channel by
  channel (d = h*P + p, A[d, n] = A[h], delta[b, d, t] = dt[b, t, h]);
* closed forms: no decay (A = 0) gives prefix sums; a decay that wipes the state keeps only the
  current token; two calls passing the state equal one call; heads do not interact.
"""

import numpy as np
import pytest

import oracle


def _inputs(batch, L, H, P, N, seed, with_h0=True, A_scale=1.0):
    rng = np.random.default_rng(seed)
    return dict(
        x=rng.standard_normal((batch, L, H, P)),
        dt=0.5 * rng.standard_normal((batch, L, H)),
        A=-A_scale * rng.uniform(0.5, 4.0, H),
        B=rng.standard_normal((batch, L, N)),
        C=rng.standard_normal((batch, L, N)),
        D=rng.standard_normal(H),
        dt_bias=rng.uniform(-3.0, -1.0, H),
        h0=rng.standard_normal((batch, H, P, N)) if with_h0 else None,
    )


def _softplus(v):
    return np.maximum(v, 0) + np.log1p(np.exp(-np.abs(v)))


def _dual_form(p, softplus=True):
    """y_t = sum_{s<=t} (C_t . B_s) exp(A (c_t - c_s)) Delta_s x_s + exp(A c_t) C_t . H0 + D x_t,
    c_t = Delta_0 + ... + Delta_t: the masked (decaying) matrix product, one mask per head."""
    x, dt, A, B, C, D, bias, h0 = (p[k] for k in ("x", "dt", "A", "B", "C", "D", "dt_bias", "h0"))
    batch, L, H, P = x.shape
    N = B.shape[2]
    y = np.zeros_like(x)
    for b in range(batch):
        G = C[b] @ B[b].T                                   # [t, s] = C_t . B_s
        for h in range(H):
            v = dt[b, :, h] + bias[h]
            Delta = _softplus(v) if softplus else v
            c = np.cumsum(Delta)
            mask = np.tril(np.exp(A[h] * (c[:, None] - c[None, :])))
            M = G * mask * Delta[None, :]
            y[b, :, h, :] = M @ x[b, :, h, :] + D[h] * x[b, :, h, :]
            if h0 is not None:
                y[b, :, h, :] += np.exp(A[h] * c)[:, None] * (C[b] @ h0[b, h].T)
    return y


@pytest.mark.parametrize("softplus", [True, False])
def test_ssd_equals_dual_masked_matrix_form(softplus):
    p = _inputs(2, 37, 3, 5, 7, seed=1)
    if not softplus:
        p["dt"] = np.abs(p["dt"]) * 0.2
        p["dt_bias"] = np.full(3, 0.05)
    y, _ = oracle.ssd(**p, dt_softplus=softplus)
    ref = _dual_form(p, softplus)
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-11)


def test_ssd_reduces_to_selective_scan_per_channel():
    batch, L, H, P, N = 2, 29, 3, 4, 6
    p = _inputs(batch, L, H, P, N, seed=2)
    y, hl = oracle.ssd(**p)
    dim = H * P
    x6 = p["x"].reshape(batch, L, dim).transpose(0, 2, 1)                  # [b, d, t]
    delta6 = np.repeat(p["dt"], P, axis=2).transpose(0, 2, 1)             # dt of the channel's head
    A6 = np.repeat(p["A"], P)[:, None] * np.ones((1, N))
    D6, bias6 = np.repeat(p["D"], P), np.repeat(p["dt_bias"], P)
    B6, C6 = p["B"].transpose(0, 2, 1), p["C"].transpose(0, 2, 1)          # [b, n, t]
    h06 = p["h0"].reshape(batch, dim, N)
    out6, hl6 = oracle.selective_scan(x6, delta6, A6, B6, C6, D6, None, bias6, True, h0=h06)
    np.testing.assert_allclose(y, out6.transpose(0, 2, 1).reshape(batch, L, H, P), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(hl, hl6.reshape(batch, H, P, N), rtol=1e-12, atol=1e-12)


def test_ssd_no_decay_is_prefix_sum():
    p = _inputs(1, 23, 2, 3, 4, seed=3)
    p["A"] = np.zeros(2)
    y, hl = oracle.ssd(**p)
    Delta = _softplus(p["dt"] + p["dt_bias"])                              # [b, t, h]
    inc = Delta[..., None, None] * p["x"][..., :, None] * p["B"][:, :, None, None, :]   # [b, t, h, p, n]
    Hs = p["h0"][:, None] + np.cumsum(inc, axis=1)
    ref = np.einsum("bthpn,btn->bthp", Hs, p["C"]) + p["D"][None, None, :, None] * p["x"]
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(hl, Hs[:, -1], rtol=1e-11, atol=1e-11)


def test_ssd_full_decay_keeps_only_current_token():
    p = _inputs(1, 9, 2, 3, 4, seed=4)
    p["A"] = np.full(2, -1e4)
    p["dt_bias"] = np.full(2, 3.0)                                        # Delta ~ 3: exp(-3e4) = 0
    y, hl = oracle.ssd(**p)
    Delta = _softplus(p["dt"] + p["dt_bias"])
    cb = np.einsum("btn,btn->bt", p["C"], p["B"])
    ref = (Delta * cb[..., None])[..., None] * p["x"] + p["D"][None, None, :, None] * p["x"]
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    last = Delta[:, -1, :, None, None] * p["x"][:, -1, :, :, None] * p["B"][:, -1, None, None, :]
    np.testing.assert_allclose(hl, last, rtol=1e-12, atol=1e-12)


def test_ssd_two_calls_pass_the_state():
    p = _inputs(2, 40, 2, 3, 5, seed=5)
    y, hl = oracle.ssd(**p)
    L1 = 17
    cut = lambda a, sl: a[:, sl]
    p1 = dict(p, x=cut(p["x"], slice(0, L1)), dt=cut(p["dt"], slice(0, L1)), B=cut(p["B"], slice(0, L1)),
              C=cut(p["C"], slice(0, L1)))
    y1, h1 = oracle.ssd(**p1)
    p2 = dict(p, x=cut(p["x"], slice(L1, None)), dt=cut(p["dt"], slice(L1, None)), B=cut(p["B"], slice(L1, None)),
              C=cut(p["C"], slice(L1, None)), h0=h1)
    y2, h2 = oracle.ssd(**p2)
    np.testing.assert_allclose(np.concatenate([y1, y2], axis=1), y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(h2, hl, rtol=1e-12, atol=1e-12)


def test_ssd_heads_do_not_interact():
    p = _inputs(1, 15, 3, 2, 4, seed=6)
    y, _ = oracle.ssd(**p)
    q = dict(p)
    q["x"] = p["x"].copy()
    q["x"][:, :, 1, :] += 5.0
    q["dt"] = p["dt"].copy()
    q["dt"][:, :, 1] -= 1.0
    y2, _ = oracle.ssd(**q)
    np.testing.assert_array_equal(y[:, :, 0], y2[:, :, 0])
    np.testing.assert_array_equal(y[:, :, 2], y2[:, :, 2])
    assert not np.allclose(y[:, :, 1], y2[:, :, 1])


def test_ssd_constant_input_geometric_sum():
    """Constant x, dt, B, C over time: H_t = Delta x B^T (1 - a^(t+1)) / (1 - a) with a = exp(Delta A),
    so y_t = Delta (B . C) x (1 - a^(t+1)) / (1 - a) + D x (closed form, no recurrence)."""
    rng = np.random.default_rng(11)
    batch, L, H, P, N = 2, 50, 3, 4, 5
    x1 = rng.standard_normal((batch, 1, H, P))
    B1, C1 = rng.standard_normal((batch, 1, N)), rng.standard_normal((batch, 1, N))
    dt1 = 0.3 * rng.standard_normal((batch, 1, H))
    A = -rng.uniform(0.5, 3.0, H)
    D = rng.standard_normal(H)
    bias = rng.uniform(-3.0, -1.0, H)
    p = dict(x=np.repeat(x1, L, axis=1), dt=np.repeat(dt1, L, axis=1), A=A, B=np.repeat(B1, L, axis=1),
             C=np.repeat(C1, L, axis=1), D=D, dt_bias=bias, h0=None)
    y, hl = oracle.ssd(**p)
    Delta = _softplus(dt1[:, 0] + bias)                         # [b, h]
    a = np.exp(Delta * A)
    t = np.arange(L)[None, :, None]
    geo = (1.0 - a[:, None, :] ** (t + 1)) / (1.0 - a[:, None, :])      # [b, t, h]
    bc = np.einsum("bn,bn->b", B1[:, 0], C1[:, 0])[:, None, None]
    ref = (Delta[:, None, :] * bc * geo)[..., None] * x1 + D[None, None, :, None] * x1
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-12)
    hl_ref = (Delta * (1.0 - a ** L) / (1.0 - a))[:, :, None, None] * x1[:, 0, :, :, None] * B1[:, 0][:, None, None, :]
    np.testing.assert_allclose(hl, hl_ref, rtol=1e-11, atol=1e-12)

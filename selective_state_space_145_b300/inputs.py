"""Seeded synthetic inputs for the selective-scan (S6) hot path.

This module only draws numbers: it holds none of the scan's arithmetic, so the
CUDA path and the fp64 CPU oracle can both take their inputs from it and share
nothing else.

Recipe. One CPU ``torch.Generator`` per call, seeded explicitly; the draws are
made in float32 in this fixed order and then cast to the I/O dtype once:

* ``x``  ~ N(0, 1), shape [batch, dim, seqlen]. It is the scan input ``u``
  when there is no conv prologue, else the raw input of the causal conv.
* ``delta`` (the pre-activation of the step size) ~ N(0, 0.5^2), same shape.
  The per-channel bias is *not* added here: the op adds it (``delta_bias``).
* ``z`` (the gate branch) ~ N(0, 1), same shape.
* ``B``, ``C`` ~ N(0, 1), shape [batch, dstate, seqlen]: one input map and
  one output map per token, shared by every channel.
* ``D`` (the skip weight) ~ N(0, 1), shape [dim].
* ``dt`` log-uniform in [1e-3, 0.1], shape [dim]; ``delta_bias`` is the value
  whose softplus is ``dt``, i.e. ``dt + log(-expm1(-dt))``, so that the step
  size of a token with zero pre-activation is ``dt``.
* the conv weight ~ U(-0.5, 0.5), shape [dim, d_conv]; the conv bias is 0.
* optionally, "salient" time indices: a fraction of the positions of each
  batch element, drawn without replacement; ``delta`` is shifted by ``+4``
  there for every channel (rare tokens with a large step size).
* optionally ``h0`` ~ N(0, 1), shape [batch, dim, dstate], fp32.

``A[d, n] = -(n + 1)`` for every channel (the S4D-real initialisation,
``A = -exp(log(1..N))``), unless a test asks for random negative values.

Parameters (``A``, ``D``, ``delta_bias``, conv weight and bias) and states are
always float32; the per-token tensors take the I/O dtype.
"""

from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import torch

IO_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One named synthetic workload with its sizes and seed."""

    name: str
    kind: str            # "scan" (prefill) or "decode"
    io: str              # "f32" or "bf16"
    batch: int
    dim: int             # d_inner = expand * d_model
    seqlen: int          # tokens per sequence (1 for decode)
    dstate: int          # N
    d_conv: int          # 0 = no conv prologue
    seed: int
    salient_frac: float = 0.0
    steps: int = 1       # decode steps run back to back
    d_model: Optional[int] = None
    expand: Optional[int] = None

    @property
    def updates(self) -> int:
        """State updates (b, t, d, n) processed by one pass."""
        return self.batch * self.seqlen * self.dim * self.dstate * self.steps


# The five synthetic workloads the method is measured on.
WORKLOADS: Dict[str, Workload] = {w.name: w for w in [
    Workload("scan_f32_b1_d64_l256_n16", "scan", "f32", 1, 64, 256, 16, 0, seed=145000),
    Workload("block_f32_b2_d1024_l1024_n16_k4", "scan", "f32", 2, 1024, 1024, 16, 4, seed=145001,
             d_model=512, expand=2),
    Workload("block_bf16_b8_d2048_l2048_n16_k4", "scan", "bf16", 8, 2048, 2048, 16, 4, seed=145002,
             d_model=1024, expand=2),
    Workload("longscan_bf16_b1_d1536_l131072_n16", "scan", "bf16", 1, 1536, 131072, 16, 0, seed=145003,
             salient_frac=0.01),
    Workload("decode_bf16_b256_d5120_n16_k4_x64", "decode", "bf16", 256, 5120, 1, 16, 4, seed=145004,
             steps=64, d_model=2560, expand=2),
]}

# Listed in order of size; the first is small enough for the oracle to run whole.
WORKLOAD_ORDER = list(WORKLOADS)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _log_uniform(g: torch.Generator, n: int, lo: float, hi: float) -> torch.Tensor:
    r = torch.rand(n, generator=g, dtype=torch.float64)
    return torch.exp(torch.log(torch.tensor(lo, dtype=torch.float64))
                     + r * (torch.log(torch.tensor(hi, dtype=torch.float64))
                            - torch.log(torch.tensor(lo, dtype=torch.float64))))


def s4d_real_A(dim: int, dstate: int) -> torch.Tensor:
    """A[d, n] = -(n + 1), float32 [dim, dstate]."""
    return -torch.arange(1, dstate + 1, dtype=torch.float32).repeat(dim, 1).contiguous()


def random_negative_A(g: torch.Generator, dim: int, dstate: int) -> torch.Tensor:
    """A[d, n] = -exp(N(0, 0.5^2)): distinct negative values per (d, n), for tests."""
    return (-torch.exp(0.5 * torch.randn(dim, dstate, generator=g))).contiguous()


def scan_inputs(batch: int, dim: int, seqlen: int, dstate: int, d_conv: int = 0, io: str = "f32",
                seed: int = 0, salient_frac: float = 0.0, with_h0: bool = False,
                with_z: bool = True, with_D: bool = True, random_A: bool = False,
                with_conv_init: bool = False) -> Dict[str, Optional[torch.Tensor]]:
    """Draw one prefill problem on the CPU. Returns a dict of contiguous tensors.

    Keys: x, delta, z, B, C, D, delta_bias, A, conv_w, conv_b, conv_init, h0.
    ``conv_init`` [batch, dim, d_conv-1] is the raw input that precedes t = 0
    (zeros when absent); ``h0`` the initial state (zeros when absent).
    """
    g = _gen(seed)
    dt = IO_DTYPES[io]
    x = torch.randn(batch, dim, seqlen, generator=g)
    delta = 0.5 * torch.randn(batch, dim, seqlen, generator=g)
    z = torch.randn(batch, dim, seqlen, generator=g)
    Bm = torch.randn(batch, dstate, seqlen, generator=g)
    Cm = torch.randn(batch, dstate, seqlen, generator=g)
    D = torch.randn(dim, generator=g)
    dt_ = _log_uniform(g, dim, 1e-3, 0.1)
    delta_bias = (dt_ + torch.log(-torch.expm1(-dt_))).to(torch.float32)
    conv_w = conv_b = conv_init = None
    if d_conv > 0:
        conv_w = (torch.rand(dim, d_conv, generator=g) - 0.5).contiguous()
        conv_b = torch.zeros(dim, dtype=torch.float32)
    if salient_frac > 0.0:
        n_sal = max(1, int(round(salient_frac * seqlen)))
        for b in range(batch):
            idx = torch.randperm(seqlen, generator=g)[:n_sal]
            delta[b, :, idx] += 4.0
    h0 = torch.randn(batch, dim, dstate, generator=g) if with_h0 else None
    if d_conv > 0 and with_conv_init:
        conv_init = torch.randn(batch, dim, d_conv - 1, generator=g).to(dt).contiguous()
    A = random_negative_A(g, dim, dstate) if random_A else s4d_real_A(dim, dstate)
    return {
        "x": x.to(dt).contiguous(),
        "delta": delta.to(dt).contiguous(),
        "z": z.to(dt).contiguous() if with_z else None,
        "B": Bm.to(dt).contiguous(),
        "C": Cm.to(dt).contiguous(),
        "D": D.contiguous() if with_D else None,
        "delta_bias": delta_bias.contiguous(),
        "A": A,
        "conv_w": conv_w,
        "conv_b": conv_b,
        "conv_init": conv_init,
        "h0": h0.contiguous() if h0 is not None else None,
    }


def decode_inputs(batch: int, dim: int, dstate: int, d_conv: int = 4, io: str = "bf16", seed: int = 0,
                  steps: int = 1, random_A: bool = False) -> Dict[str, Optional[torch.Tensor]]:
    """Draw one decode problem: ``steps`` fresh tokens per sequence plus the starting state.

    Keys: x, delta, z [steps, batch, dim]; B, C [steps, batch, dstate]; D, delta_bias [dim];
    A [dim, dstate]; conv_w [dim, d_conv], conv_b [dim]; state [batch, dim, dstate] fp32;
    conv_state [batch, dim, d_conv-1] (the last d_conv-1 raw inputs, oldest first).
    """
    g = _gen(seed)
    dt = IO_DTYPES[io]
    x = torch.randn(steps, batch, dim, generator=g)
    delta = 0.5 * torch.randn(steps, batch, dim, generator=g)
    z = torch.randn(steps, batch, dim, generator=g)
    Bm = torch.randn(steps, batch, dstate, generator=g)
    Cm = torch.randn(steps, batch, dstate, generator=g)
    D = torch.randn(dim, generator=g)
    dt_ = _log_uniform(g, dim, 1e-3, 0.1)
    delta_bias = (dt_ + torch.log(-torch.expm1(-dt_))).to(torch.float32)
    conv_w = conv_b = None
    if d_conv > 0:
        conv_w = (torch.rand(dim, d_conv, generator=g) - 0.5).contiguous()
        conv_b = torch.zeros(dim, dtype=torch.float32)
    state = torch.randn(batch, dim, dstate, generator=g)
    conv_state = torch.randn(batch, dim, max(d_conv - 1, 0), generator=g).to(dt).contiguous() if d_conv > 0 else None
    A = random_negative_A(g, dim, dstate) if random_A else s4d_real_A(dim, dstate)
    return {
        "x": x.to(dt).contiguous(), "delta": delta.to(dt).contiguous(), "z": z.to(dt).contiguous(),
        "B": Bm.to(dt).contiguous(), "C": Cm.to(dt).contiguous(), "D": D.contiguous(),
        "delta_bias": delta_bias.contiguous(), "A": A, "conv_w": conv_w, "conv_b": conv_b,
        "state": state.contiguous(), "conv_state": conv_state,
    }


def workload_inputs(w: Workload) -> Dict[str, Optional[torch.Tensor]]:
    """Inputs of a named workload, drawn from its own seed."""
    if w.kind == "decode":
        return decode_inputs(w.batch, w.dim, w.dstate, w.d_conv, w.io, w.seed, steps=w.steps)
    return scan_inputs(w.batch, w.dim, w.seqlen, w.dstate, w.d_conv, w.io, w.seed,
                       salient_frac=w.salient_frac)


# ---- multi-head SSM with one decay per head (the state-space-duality layer)
#
# Recipe, one seeded CPU generator per call, float32 draws in this order, then the per-token
# tensors cast to bf16 once:
#   x ~ N(0, 1) [batch, L, nheads, headdim]; dt (step pre-activation) ~ N(0, 0.5^2) [batch, L, nheads];
#   B, C ~ N(0, 1) [batch, L, dstate] (one group: shared by every head); D ~ N(0, 1) [nheads];
#   per-head step dt0 log-uniform in [1e-3, 0.1] with dt_bias = dt0 + log(-expm1(-dt0));
#   A[h] = -U(1, 16) (one decay rate per head); optionally h0 ~ N(0, 1) [batch, nheads, headdim, dstate].
# The pages give no sizes for this layer; the workload below takes the bf16 block workload's model
# (d_model 1024, expand 2, so 2048 channels = 32 heads of 64) with a state of 128 per head.

@dataclasses.dataclass(frozen=True)
class SsdWorkload:
    """A named synthetic workload of the state-space-duality layer."""

    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    seed: int
    d_model: Optional[int] = None
    expand: Optional[int] = None
    kind: str = "ssd"
    io: str = "bf16"

    @property
    def updates(self) -> int:
        """State updates (b, t, h, p, n) of one pass."""
        return self.batch * self.seqlen * self.nheads * self.headdim * self.dstate


SSD_WORKLOADS: Dict[str, SsdWorkload] = {w.name: w for w in [
    SsdWorkload("ssd_bf16_b8_l2048_h32_p64_n128", 8, 2048, 32, 64, 128, seed=145005, d_model=1024, expand=2),
]}


def ssd_inputs(batch: int, seqlen: int, nheads: int, headdim: int = 64, dstate: int = 128, seed: int = 0,
               with_h0: bool = False, with_D: bool = True) -> Dict[str, Optional[torch.Tensor]]:
    """Draw one problem of the state-space-duality layer. Keys: x, dt, B, C (bf16), A, D, dt_bias, h0."""
    g = _gen(seed)
    x = torch.randn(batch, seqlen, nheads, headdim, generator=g)
    dt = 0.5 * torch.randn(batch, seqlen, nheads, generator=g)
    Bm = torch.randn(batch, seqlen, dstate, generator=g)
    Cm = torch.randn(batch, seqlen, dstate, generator=g)
    D = torch.randn(nheads, generator=g)
    dt0 = _log_uniform(g, nheads, 1e-3, 0.1)
    dt_bias = (dt0 + torch.log(-torch.expm1(-dt0))).to(torch.float32)
    A = -(1.0 + 15.0 * torch.rand(nheads, generator=g))
    h0 = torch.randn(batch, nheads, headdim, dstate, generator=g) if with_h0 else None
    bf = torch.bfloat16
    return {
        "x": x.to(bf).contiguous(), "dt": dt.to(bf).contiguous(), "B": Bm.to(bf).contiguous(),
        "C": Cm.to(bf).contiguous(), "A": A.contiguous(), "D": D.contiguous() if with_D else None,
        "dt_bias": dt_bias.contiguous(), "h0": h0.contiguous() if h0 is not None else None,
    }


def ssd_workload_inputs(w: SsdWorkload) -> Dict[str, Optional[torch.Tensor]]:
    return ssd_inputs(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.seed)


# ---- problems too large to draw on the host
#
# Same distributions and shapes as scan_inputs, decode_inputs and ssd_inputs, for tensors of
# billions of elements: the per-token tensors and states are drawn directly on `device`, in their
# storage dtype, by a generator of that device seeded with `seed`; the per-channel (or per-head)
# parameters are drawn on the host as above and then moved. The numbers differ from the host
# recipe's (another generator), the distributions do not.

def _dev_gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _dev_normal(g: torch.Generator, shape, dtype, device, scale: float = 1.0) -> torch.Tensor:
    t = torch.randn(shape, generator=g, dtype=dtype, device=device)
    return t.mul_(scale) if scale != 1.0 else t


def _channel_params(g: torch.Generator, dim: int, dstate: int, d_conv: int, device):
    D = torch.randn(dim, generator=g)
    dt_ = _log_uniform(g, dim, 1e-3, 0.1)
    delta_bias = (dt_ + torch.log(-torch.expm1(-dt_))).to(torch.float32)
    conv_w = (torch.rand(dim, d_conv, generator=g) - 0.5).contiguous() if d_conv > 0 else None
    conv_b = torch.zeros(dim, dtype=torch.float32) if d_conv > 0 else None
    mv = lambda t: None if t is None else t.to(device)
    return {"D": mv(D), "delta_bias": mv(delta_bias), "A": mv(s4d_real_A(dim, dstate)), "conv_w": mv(conv_w),
            "conv_b": mv(conv_b)}


def scan_inputs_on(device, batch: int, dim: int, seqlen: int, dstate: int, d_conv: int = 0, io: str = "bf16",
                   seed: int = 0) -> Dict[str, Optional[torch.Tensor]]:
    """A prefill problem drawn on `device` (keys of scan_inputs; no h0, no conv_init)."""
    gd = _dev_gen(seed, device)
    dt = IO_DTYPES[io]
    p = {
        "x": _dev_normal(gd, (batch, dim, seqlen), dt, device),
        "delta": _dev_normal(gd, (batch, dim, seqlen), dt, device, 0.5),
        "z": _dev_normal(gd, (batch, dim, seqlen), dt, device),
        "B": _dev_normal(gd, (batch, dstate, seqlen), dt, device),
        "C": _dev_normal(gd, (batch, dstate, seqlen), dt, device),
        "conv_init": None, "h0": None,
    }
    p.update(_channel_params(_gen(seed), dim, dstate, d_conv, device))
    return p


def decode_inputs_on(device, batch: int, dim: int, dstate: int, d_conv: int = 4, io: str = "bf16",
                     seed: int = 0) -> Dict[str, Optional[torch.Tensor]]:
    """One decode step drawn on `device`: x, delta, z [batch, dim]; B, C [batch, dstate];
    state [batch, dim, dstate] fp32; conv_state [batch, dim, d_conv-1]; parameters as decode_inputs."""
    gd = _dev_gen(seed, device)
    dt = IO_DTYPES[io]
    p = {
        "x": _dev_normal(gd, (batch, dim), dt, device),
        "delta": _dev_normal(gd, (batch, dim), dt, device, 0.5),
        "z": _dev_normal(gd, (batch, dim), dt, device),
        "B": _dev_normal(gd, (batch, dstate), dt, device),
        "C": _dev_normal(gd, (batch, dstate), dt, device),
        "state": _dev_normal(gd, (batch, dim, dstate), torch.float32, device),
        "conv_state": _dev_normal(gd, (batch, dim, d_conv - 1), dt, device) if d_conv > 1 else None,
    }
    p.update(_channel_params(_gen(seed), dim, dstate, d_conv, device))
    return p


def ssd_inputs_on(device, batch: int, seqlen: int, nheads: int, headdim: int = 64, dstate: int = 128,
                  seed: int = 0) -> Dict[str, Optional[torch.Tensor]]:
    """A problem of the state-space-duality layer drawn on `device` (keys of ssd_inputs, no h0)."""
    gd = _dev_gen(seed, device)
    bf = torch.bfloat16
    g = _gen(seed)
    D = torch.randn(nheads, generator=g)
    dt0 = _log_uniform(g, nheads, 1e-3, 0.1)
    dt_bias = (dt0 + torch.log(-torch.expm1(-dt0))).to(torch.float32)
    A = -(1.0 + 15.0 * torch.rand(nheads, generator=g))
    return {
        "x": _dev_normal(gd, (batch, seqlen, nheads, headdim), bf, device),
        "dt": _dev_normal(gd, (batch, seqlen, nheads), bf, device, 0.5),
        "B": _dev_normal(gd, (batch, seqlen, dstate), bf, device),
        "C": _dev_normal(gd, (batch, seqlen, dstate), bf, device),
        "A": A.to(device), "D": D.to(device), "dt_bias": dt_bias.to(device), "h0": None,
    }

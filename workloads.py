"""Seeded synthetic workloads for the gated delta-rule prefill and decode step.

This module only draws random inputs; it holds none of the method's arithmetic
and is shared by the tests, the benchmark and the smoke check (both the CUDA
path and the CPU oracle consume what it returns).

Recipe (one ``torch.Generator`` per workload, seeded with the workload's seed,
tensors drawn on the CPU in this fixed order: q, k, v, g_log, beta, state):

* q, k  ~ N(0, 1) in fp32, then divided by their L2 norm over the head dim
  (the "GDN CTE Kernel API Reference" Notes require L2-normalised q/k), then
  rounded to the compute dtype (round-to-nearest-even for bf16);
* v     ~ N(0, 1), rounded to the compute dtype;
* g_log ~ U(lo, hi) fp32 (a negative log-decay, Parameters / g_log);
* beta  = sigmoid(N(0, s)) fp32, in (0, 1) (Parameters / beta);
* state ~ N(0, sigma) fp32 [B, Hv, Dk, Dv] when the workload supplies one,
  otherwise the zero-start ("omitted") form is used.

``N(m, s)`` names a standard deviation ``s``.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "prefill" or "decode"
    B: int
    Hk: int
    Hv: int
    S: int
    Dk: int
    Dv: int
    dtype: str           # compute dtype of q/k/v/out: "f32" or "bf16"
    g_lo: float
    g_hi: float
    beta_std: float
    state_std: float     # 0.0 -> zero initial state (no state supplied)
    seed: int

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.Dk)

    @property
    def tokens(self) -> int:
        return self.B * self.S

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the method's benchmark plan.
TINY_PREFILL = Workload("prefill_b1_h2_s128_d64_f32", "prefill", 1, 2, 2, 128, 64, 64, "f32",
                        -0.5, -0.005, 1.0, 0.0, 0)
DECODE_STEP = Workload("decode_b64_hk16_hv32_d128_bf16", "decode", 64, 16, 32, 1, 128, 128, "bf16",
                       -0.5, -0.005, 1.0, 0.02, 1)
PREFILL = Workload("prefill_b4_hk16_hv32_s4096_d128_bf16", "prefill", 4, 16, 32, 4096, 128, 128, "bf16",
                   -0.5, -0.005, 1.0, 0.02, 2)
LONG_PREFILL = Workload("prefill_b1_hk16_hv32_s32768_d128_bf16", "prefill", 1, 16, 32, 32768, 128, 128,
                        "bf16", -0.5, -0.005, 1.0, 0.0, 3)
WIDE_GQA_PREFILL = Workload("prefill_b16_hk8_hv32_s2048_d128_bf16", "prefill", 16, 8, 32, 2048, 128, 128,
                            "bf16", -2.0, -0.001, 2.0, 0.05, 4)

ALL = [TINY_PREFILL, DECODE_STEP, PREFILL, LONG_PREFILL, WIDE_GQA_PREFILL]
BY_NAME = {w.name: w for w in ALL}


def make_inputs(w: Workload, device="cpu", pin: bool = False):
    """Draw the workload's tensors.  Returns a dict with q, k, v, g_log, beta,
    state (None for a zero start) and scale.  Values are drawn on the CPU so they
    do not depend on the device; they are then moved to ``device``."""
    gen = torch.Generator(device="cpu").manual_seed(w.seed)
    dt = w.torch_dtype

    def unit(shape):
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
        x = x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)
        return x.to(dt)

    q = unit((w.B, w.Hk, w.S, w.Dk))
    k = unit((w.B, w.Hk, w.S, w.Dk))
    v = torch.randn((w.B, w.Hv, w.S, w.Dv), generator=gen, dtype=torch.float32).to(dt)
    g = torch.rand((w.B, w.Hv, w.S), generator=gen, dtype=torch.float32) * (w.g_hi - w.g_lo) + w.g_lo
    beta = torch.sigmoid(torch.randn((w.B, w.Hv, w.S), generator=gen, dtype=torch.float32) * w.beta_std)
    state = None
    if w.state_std > 0.0:
        state = torch.randn((w.B, w.Hv, w.Dk, w.Dv), generator=gen, dtype=torch.float32) * w.state_std
    out = dict(q=q, k=k, v=v, g_log=g, beta=beta, state=state, scale=w.scale)
    for key in ("q", "k", "v", "g_log", "beta", "state"):
        t = out[key]
        if t is None:
            continue
        if pin:
            t = t.pin_memory()
        if device != "cpu":
            t = t.to(device)
        out[key] = t
    return out


# ------------------------------------------------------------------ conv1d
# The depthwise causal conv1d + SiLU in front of the recurrence ("GDN Conv1D
# Kernel API Reference").  Its channels are q|k|v packed: C = 2 * Hk * Dk +
# Hv * Dv = 8192 for the Hk = 16, Hv = 32, D = 128 heads above, with K = 4 taps.
# Recipe (one generator per workload, drawn on the CPU in this order):
#   mixed / x  ~ N(0, 1) [B, C, T], rounded to the activation dtype;
#   weight     ~ U(-1/sqrt(K), 1/sqrt(K)) fp32 [C, K] (a depthwise Conv1d's
#                default initialisation bound for a fan-in of K);
#   conv_state ~ N(0, 1) [B, C, K] in the activation dtype (decode only).

@dataclasses.dataclass(frozen=True)
class ConvWorkload:
    name: str
    kind: str            # "prefill" or "decode"
    B: int
    C: int
    T: int               # tokens (1 for the decode step)
    K: int               # taps
    dtype: str           # activation dtype of mixed / out / conv_state: "f32" or "bf16"
    seed: int

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def tokens(self) -> int:
        return self.B * self.T

    def with_(self, **kw) -> "ConvWorkload":
        return dataclasses.replace(self, **kw)


CONV_PREFILL = ConvWorkload("conv1d_prefill_b4_c8192_t4096_k4_bf16", "prefill", 4, 8192, 4096, 4, "bf16", 5)
CONV_DECODE = ConvWorkload("conv1d_decode_b64_c8192_k4_bf16", "decode", 64, 8192, 1, 4, "bf16", 6)


def make_conv_inputs(w: ConvWorkload, device="cpu", pin: bool = False):
    """Draw a conv1d workload's tensors: x [B, C, T], weight [C, K] fp32 and,
    for the decode step, conv_state [B, C, K]."""
    gen = torch.Generator(device="cpu").manual_seed(w.seed)
    x = torch.randn((w.B, w.C, w.T), generator=gen, dtype=torch.float32).to(w.torch_dtype)
    bound = 1.0 / math.sqrt(w.K)
    weight = (torch.rand((w.C, w.K), generator=gen, dtype=torch.float32) * 2.0 - 1.0) * bound
    state = None
    if w.kind == "decode":
        state = torch.randn((w.B, w.C, w.K), generator=gen, dtype=torch.float32).to(w.torch_dtype)
    out = dict(x=x, weight=weight, state=state)
    for key in ("x", "weight", "state"):
        t = out[key]
        if t is None:
            continue
        if pin:
            t = t.pin_memory()
        if device != "cpu":
            t = t.to(device)
        out[key] = t
    return out


# ------------------------------------------------------------------ gated decode step
# One token of the decode block's gated step: the post-conv q|k|v row, the output
# gate z, the raw gate inputs a, b and the per-head parameters.  Recipe (one
# generator per workload, drawn on the CPU in this order):
#   qkv   ~ N(0, 1) [B, 2 Hk Dk + Hv Dv]  (q, k are normalised by the kernel itself)
#   z     ~ N(0, 1) [B, Hv Dv];  a ~ N(0, 1), b ~ N(0, 1) [B, Hv]   (activation dtype)
#   A_log = log(U(1, 16)) [Hv];  dt ~ exp(U(log 1e-3, log 1e-1)), dt_bias = dt + log(1 - e^-dt)
#           (the inverse softplus of dt) [Hv];  norm_weight = 1 + 0.1 N(0, 1) [Dv]   (fp32)
#   state ~ N(0, sigma) [B, Hv, Dk, Dv] fp32.

@dataclasses.dataclass(frozen=True)
class GatedWorkload:
    name: str
    B: int
    Hk: int
    Hv: int
    Dk: int
    Dv: int
    dtype: str
    state_std: float
    seed: int

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.Dk)

    def with_(self, **kw) -> "GatedWorkload":
        return dataclasses.replace(self, **kw)


GATED_DECODE = GatedWorkload("gated_decode_b64_hk16_hv32_d128_bf16", 64, 16, 32, 128, 128, "bf16", 0.02, 7)


def make_gated_inputs(w: GatedWorkload, device="cpu"):
    gen = torch.Generator(device="cpu").manual_seed(w.seed)
    dt = w.torch_dtype
    rn = lambda *shape: torch.randn(shape, generator=gen, dtype=torch.float32)
    ru = lambda lo, hi, *shape: torch.rand(shape, generator=gen, dtype=torch.float32) * (hi - lo) + lo
    qkv = rn(w.B, 2 * w.Hk * w.Dk + w.Hv * w.Dv).to(dt)
    z = rn(w.B, w.Hv * w.Dv).to(dt)
    a = rn(w.B, w.Hv).to(dt)
    b = rn(w.B, w.Hv).to(dt)
    A_log = torch.log(ru(1.0, 16.0, w.Hv))
    dtv = torch.exp(ru(math.log(1e-3), math.log(1e-1), w.Hv))
    dt_bias = dtv + torch.log(-torch.expm1(-dtv))
    norm_weight = 1.0 + 0.1 * rn(w.Dv)
    state = rn(w.B, w.Hv, w.Dk, w.Dv) * w.state_std if w.state_std > 0 else None
    out = dict(qkv=qkv, z=z, a=a, b=b, A_log=A_log, dt_bias=dt_bias, norm_weight=norm_weight, state=state,
               scale=w.scale)
    if device != "cpu":
        out = {k: (v.to(device) if hasattr(v, "to") else v) for k, v in out.items()}
    return out


# ------------------------------------------------------------------ the gated prefill
# The prefill's inputs (make_inputs) plus the RMSNormGated inputs of every token, drawn
# from their own generator (seed + 500): z ~ N(0, 1) [B, Hv, S, Dv] in the compute dtype,
# norm_weight = 1 + 0.1 N(0, 1) [Dv] fp32.

def make_gate_inputs(w: Workload, device="cpu"):
    gen = torch.Generator(device="cpu").manual_seed(w.seed + 500)
    z = torch.randn((w.B, w.Hv, w.S, w.Dv), generator=gen, dtype=torch.float32).to(w.torch_dtype)
    norm_weight = 1.0 + 0.1 * torch.randn((w.Dv,), generator=gen, dtype=torch.float32)
    return dict(z=z.to(device), norm_weight=norm_weight.to(device))


# ------------------------------------------------------------------ the decode block
# The whole decode block without its output projection: the token's hidden state,
# the four input projections, the conv1d and the gated step.  Hidden size H = 2048.
# Recipe (one generator, drawn on the CPU in this order):
#   hidden ~ N(0, 1) [B, 1, H] bf16;  W_qkv, W_z, W_a, W_b ~ N(0, 1/H) bf16 ([H, N], so the
#   projections are O(1));  conv_weight ~ U(-1/sqrt(K), 1/sqrt(K)) fp32 [C, K];
#   conv_state ~ N(0, 1) bf16 [B, C, K];  A_log, dt_bias, norm_weight as the gated step;
#   state ~ N(0, 0.02) fp32.

@dataclasses.dataclass(frozen=True)
class BlockWorkload:
    name: str
    B: int
    H: int
    Hk: int
    Hv: int
    Dk: int
    Dv: int
    K: int
    seed: int

    @property
    def C(self) -> int:
        return 2 * self.Hk * self.Dk + self.Hv * self.Dv

    def with_(self, **kw) -> "BlockWorkload":
        return dataclasses.replace(self, **kw)


DECODE_BLOCK = BlockWorkload("decode_block_b64_h2048_hk16_hv32_d128_k4_bf16", 64, 2048, 16, 32, 128, 128, 4, 8)


def make_block_inputs(w: BlockWorkload, device="cpu"):
    gen = torch.Generator(device="cpu").manual_seed(w.seed)
    rn = lambda *shape: torch.randn(shape, generator=gen, dtype=torch.float32)
    ru = lambda lo, hi, *shape: torch.rand(shape, generator=gen, dtype=torch.float32) * (hi - lo) + lo
    bf = torch.bfloat16
    sd = 1.0 / math.sqrt(w.H)
    hidden = rn(w.B, 1, w.H).to(bf)
    W_qkv = (rn(w.H, w.C) * sd).to(bf)
    W_z = (rn(w.H, w.Hv * w.Dv) * sd).to(bf)
    W_a = (rn(w.H, w.Hv) * sd).to(bf)
    W_b = (rn(w.H, w.Hv) * sd).to(bf)
    bound = 1.0 / math.sqrt(w.K)
    conv_weight = (torch.rand((w.C, w.K), generator=gen, dtype=torch.float32) * 2.0 - 1.0) * bound
    conv_state = rn(w.B, w.C, w.K).to(bf)
    A_log = torch.log(ru(1.0, 16.0, w.Hv))
    dtv = torch.exp(ru(math.log(1e-3), math.log(1e-1), w.Hv))
    dt_bias = dtv + torch.log(-torch.expm1(-dtv))
    norm_weight = 1.0 + 0.1 * rn(w.Dv)
    state = rn(w.B, w.Hv, w.Dk, w.Dv) * 0.02
    out = dict(hidden=hidden, W_qkv=W_qkv, W_z=W_z, W_a=W_a, W_b=W_b, conv_weight=conv_weight,
               conv_state=conv_state, A_log=A_log, dt_bias=dt_bias, norm_weight=norm_weight, state=state)
    if device != "cpu":
        out = {k: v.to(device) for k, v in out.items()}
    return out

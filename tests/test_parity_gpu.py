"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Tolerances (the method's contract): fp32 compute, elementwise
|gpu - ref| <= 1e-4 (1 + |ref|); bf16 compute, relative L2 <= 1e-2 over the
output and over the final state.  Every case is seeded; the five benchmark
workloads run at full size, compared over every sequence of the whole tensors.
"""
import pytest
import torch

import gated_delta_rule_20_gb300 as gdn
import oracle  # noqa: E402
import workloads
from gpu_util import check, check_whole, oracle_for, rel_l2, run_prefill, to64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _status_clean():
    gdn.device_status(0, clear=True)
    yield
    assert gdn.device_status(0, clear=True) == 0, "a kernel reported a wait timeout"


def small(dtype, B=2, Hk=2, Hv=4, S=200, D=128, Dv=None, state=0.02, seed=0, g=(-0.5, -0.005), bs=1.0):
    return workloads.PREFILL.with_(B=B, Hk=Hk, Hv=Hv, S=S, Dk=D, Dv=Dv or D, dtype=dtype, state_std=state,
                                   seed=seed, g_lo=g[0], g_hi=g[1], beta_std=bs)


# ------------------------------------------------------------------ decode step
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dims", [(128, 128), (64, 64), (128, 37), (5, 130 // 2), (1, 1)])
@pytest.mark.parametrize("gqa", [1, 2, 4])
def test_decode_small(dtype, dims, gqa):
    Dk, Dv = dims
    w = workloads.DECODE_STEP.with_(B=3, Hk=2, Hv=2 * gqa, Dk=Dk, Dv=Dv, dtype=dtype, seed=100 + Dk + gqa)
    x = workloads.make_inputs(w, device=DEV)
    st = x["state"].clone()
    out, st = gdn.decode_step(x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], st)
    torch.cuda.synchronize()
    ro, rs = oracle_for(x)
    check(out, st, ro, rs, dtype == "bf16", "decode %s %s gqa%d" % (dtype, dims, gqa))


def test_decode_full_workload():
    """The decode workload at full size: B=64, Hk=16, Hv=32, Dk=Dv=128, bf16."""
    w = workloads.DECODE_STEP
    x = workloads.make_inputs(w, device=DEV)
    st = x["state"].clone()
    out, st = gdn.decode_step(x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], st)
    torch.cuda.synchronize()
    ro, rs = oracle_for(x)
    eo, es = check(out, st, ro, rs, True, "decode full")
    assert eo < 5e-3 and es < 1e-5  # out rounds once to bf16; the state stays fp32


def test_decode_zero_initial_state_full_size():
    """GDN_ZERO_INITIAL_STATE on the decode step (through the C ABI), at the full size so that
    every CTA of the streaming kernel walks several heads: equals the oracle from a zero state,
    and the state buffer's previous contents (NaN here) are never read."""
    from gated_delta_rule_20_gb300 import _binding as B
    w = workloads.DECODE_STEP
    x = workloads.make_inputs(w, device=DEV)
    st = torch.full_like(x["state"], float("nan"))
    out = torch.empty_like(x["v"])
    B._call("gdn_decode_step", x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], st, out, True, False, None)
    torch.cuda.synchronize()
    ro, rs = oracle.recurrence(x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], None)
    check(out, st, ro, rs, True, "decode zero start")


def test_decode_equals_prefill_at_one_token():
    w = small("bf16", S=1, seed=7)
    x = workloads.make_inputs(w, device=DEV)
    s1 = x["state"].clone()
    o1, s1 = gdn.decode_step(x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], s1)
    s2 = x["state"].clone()
    o2, s2 = gdn.prefill(x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], s2)
    torch.cuda.synchronize()
    ro, rs = oracle_for(x)
    check(o1, s1, ro, rs, True, "decode")
    check(o2, s2, ro, rs, True, "prefill S=1")


# ------------------------------------------------------------------ fp32 prefill (FFMA kernel)
def test_prefill_tiny_fp32_workload():
    """The tiny fp32 workload (B=1, Hk=Hv=2, S=128, D=64, zero start)."""
    x = workloads.make_inputs(workloads.TINY_PREFILL, device=DEV)
    out, st = run_prefill(x, guard=64)
    ro, rs = oracle_for(x)
    check(out, st, ro, rs, False, "tiny fp32")


@pytest.mark.parametrize("S", [1, 31, 32, 33, 100])
@pytest.mark.parametrize("dims", [(64, 64), (128, 128), (37, 19)])
@pytest.mark.parametrize("with_state", [False, True])
def test_prefill_fp32_shapes(S, dims, with_state):
    w = small("f32", B=1, Hk=1, Hv=2, S=S, D=dims[0], Dv=dims[1], state=0.3 if with_state else 0.0,
              seed=S + dims[0])
    x = workloads.make_inputs(w, device=DEV)
    out, st = run_prefill(x, guard=16)
    ro, rs = oracle_for(x)
    check(out, st, ro, rs, False, "fp32 S=%d %s" % (S, dims))


def test_prefill_fp32_strong_decay():
    w = small("f32", B=1, Hk=1, Hv=2, S=96, D=64, g=(-2.0, -0.001), bs=2.0, state=0.05, seed=5)
    x = workloads.make_inputs(w, device=DEV)
    out, st = run_prefill(x)
    ro, rs = oracle_for(x)
    check(out, st, ro, rs, False, "fp32 strong decay")


# ------------------------------------------------------------------ bf16 prefill (tensor-core kernel)
@pytest.mark.parametrize("S", [1, 17, 63, 64, 65, 128, 200, 333])
@pytest.mark.parametrize("gqa", [1, 2, 4])
def test_prefill_bf16_shapes(S, gqa):
    w = small("bf16", B=2, Hk=2, Hv=2 * gqa, S=S, seed=1000 + S * 7 + gqa)
    x = workloads.make_inputs(w, device=DEV)
    out, st = run_prefill(x, guard=128)
    ro, rs = oracle_for(x)
    check(out, st, ro, rs, True, "bf16 S=%d gqa=%d" % (S, gqa))


@pytest.mark.parametrize("S", [64, 150])
def test_prefill_bf16_zero_start(S):
    w = small("bf16", S=S, state=0.0, seed=77 + S)
    x = workloads.make_inputs(w, device=DEV)
    out, st = run_prefill(x, guard=128)
    ro, rs = oracle_for(x)
    check(out, st, ro, rs, True, "bf16 zero start")


def test_prefill_bf16_strong_decay_and_beta():
    w = small("bf16", S=256, g=(-2.0, -0.001), bs=2.0, state=0.05, seed=31)
    x = workloads.make_inputs(w, device=DEV)
    out, st = run_prefill(x)
    ro, rs = oracle_for(x)
    check(out, st, ro, rs, True, "bf16 strong decay")


def test_prefill_bf16_decay_beyond_factored_range():
    """Per-token log-decays of -2..-3.5: a 64-token chunk's decay range exceeds what the factored
    masks take (125 in log2 units), so every chunk evaluates exp(G_r - G_j) per element."""
    w = small("bf16", S=256, g=(-3.5, -2.0), bs=2.0, state=0.05, seed=32)
    x = workloads.make_inputs(w, device=DEV)
    out, st = run_prefill(x)
    ro, rs = oracle_for(x)
    check(out, st, ro, rs, True, "bf16 decay beyond the factored range")


def test_prefill_bf16_mixed_factored_and_exact_masks():
    """Chunks alternate between weak decay (factored masks) and very strong decay (per-element
    exponentials) inside one sequence, and across heads, with a ragged last chunk."""
    w = small("bf16", S=330, state=0.05, seed=33)
    x = workloads.make_inputs(w, device=DEV)
    gen = torch.Generator().manual_seed(33)
    g = -(0.005 + 0.5 * torch.rand(x["g_log"].shape, generator=gen))
    strong = -(2.0 + 1.5 * torch.rand(x["g_log"].shape, generator=gen))
    chunk = torch.arange(w.S) // 64
    pick = ((chunk[None, None, :] + torch.arange(w.Hv)[None, :, None]) % 2 == 1).expand_as(g)
    x["g_log"] = torch.where(pick, strong, g).float().to(DEV)
    out, st = run_prefill(x)
    ro, rs = oracle_for(x)
    check(out, st, ro, rs, True, "bf16 mixed mask forms")


def test_prefill_bf16_correlated_keys():
    """Keys that share a common direction make A large and the solve harder."""
    w = small("bf16", S=192, seed=41)
    x = workloads.make_inputs(w, device=DEV)
    g = torch.Generator().manual_seed(41)
    base = torch.randn(1, 1, 1, 128, generator=g)
    k = x["k"].float().cpu() + 0.8 * base / base.norm()
    k = (k / k.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    x["k"] = k.to(DEV)
    out, st = run_prefill(x)
    ro, rs = oracle_for(x)
    check(out, st, ro, rs, True, "bf16 correlated keys")


def test_prefill_tc_matches_ffma_kernel():
    """The two kernels agree on the same bf16 inputs."""
    w = small("bf16", S=130, seed=9)
    x = workloads.make_inputs(w, device=DEV)
    o1, s1 = run_prefill(x)
    o2, s2 = run_prefill(x, force_ffma=True)
    assert rel_l2(to64(o1), to64(o2)) < 1e-2
    assert rel_l2(to64(s1), to64(s2)) < 1e-2


def test_prefill_halves_chain_through_state():
    """Two calls chained through the in/out state equal one call."""
    w = small("bf16", S=256, seed=13)
    x = workloads.make_inputs(w, device=DEV)
    st = x["state"].clone()
    o_full, st_full = gdn.prefill(x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], st)
    m = 128
    st2 = x["state"].clone()
    part = lambda t, a, b: t[:, :, a:b].contiguous()
    oa, st2 = gdn.prefill(part(x["q"], 0, m), part(x["k"], 0, m), part(x["v"], 0, m), part(x["g_log"], 0, m),
                          part(x["beta"], 0, m), x["scale"], st2)
    ob, st2 = gdn.prefill(part(x["q"], m, 256), part(x["k"], m, 256), part(x["v"], m, 256),
                          part(x["g_log"], m, 256), part(x["beta"], m, 256), x["scale"], st2)
    torch.cuda.synchronize()
    ro, rs = oracle_for(x)
    check(torch.cat([oa, ob], dim=2), st2, ro, rs, True, "chained halves")
    check(o_full, st_full, ro, rs, True, "one pass")


def test_prefill_deterministic():
    w = small("bf16", S=200, seed=21)
    x = workloads.make_inputs(w, device=DEV)
    o1, s1 = run_prefill(x)
    o2, s2 = run_prefill(x)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


@pytest.mark.parametrize("B,Hk,Hv", [(4, 16, 32), (16, 8, 32)], ids=["one_wave", "several_waves"])
def test_prefill_deterministic_full_size(B, Hk, Hv):
    """One pass at a full-size shape (one wave of CTAs, and 512 sequences in several waves),
    repeated: bit-identical outputs and states, with the inputs of the first chunks warm in L2
    after the first call."""
    w = workloads.PREFILL.with_(B=B, Hk=Hk, Hv=Hv, S=2048, seed=22)
    x = workloads.make_inputs(w, device=DEV)
    o1, s1 = run_prefill(x)
    for _ in range(6):
        o2, s2 = run_prefill(x)
        assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_prefill_empty_sequence():
    w = small("bf16", S=0, seed=3)
    x = workloads.make_inputs(w, device=DEV)
    st = x["state"].clone()
    out, st = gdn.prefill(x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], st)
    torch.cuda.synchronize()
    assert out.numel() == 0 and torch.equal(st, x["state"])
    out, st0 = gdn.prefill(x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], None)
    torch.cuda.synchronize()
    assert (st0 == 0).all()


# ------------------------------------------------------------------ full-size workloads, whole tensors
def _full(w):
    """The workload at full size through gdn_prefill, compared with the fp64 oracle over
    every (batch, value head) sequence: relative L2 over the whole output and the whole
    final state (the oracle runs on all host cores, about a second per workload)."""
    x = workloads.make_inputs(w, device=DEV)
    st = x["state"].clone() if x["state"] is not None else None
    out, st = gdn.prefill(x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], st)
    torch.cuda.synchronize()
    assert gdn.device_status(0, clear=False) == 0
    ro, rs = oracle_for(x)
    return check_whole(out, st, ro, rs, w.name)


@pytest.mark.slow
def test_full_prefill_b4_s4096():
    _full(workloads.PREFILL)


@pytest.mark.slow
def test_full_long_prefill_s32768():
    _full(workloads.LONG_PREFILL)


@pytest.mark.slow
def test_full_long_prefill_s32768_single_pass():
    """The same long workload with GDN_SINGLE_PASS (one CTA per sequence, no split)."""
    w = workloads.LONG_PREFILL
    x = workloads.make_inputs(w, device=DEV)
    out, st = gdn.prefill(x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], None, single_pass=True)
    torch.cuda.synchronize()
    ro, rs = oracle_for(x)
    check_whole(out, st, ro, rs, w.name + " single pass")


@pytest.mark.slow
def test_full_wide_gqa_prefill():
    _full(workloads.WIDE_GQA_PREFILL)

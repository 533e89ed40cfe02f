"""The split prefill (gdn.h, gdn_prefill): on the tensor-core path, few long sequences are
split into segments; every later segment runs from a zero start and from the identity with
v = 0 (the chunk recurrence is affine in its start state), a combine step chains the maps
into the start states, and a correction adds the start state's part to the later segments'
outputs.  Checked here: parity with the fp64 oracle, agreement with the one-pass form
(GDN_SINGLE_PASS), a ragged last segment, zero and supplied start states, GQA, weak decay
(so that every segment's state map matters), strong decay, determinism, NaN-prefilled
outputs with guard bands, the caller's workspace, and replay in a CUDA graph."""
import pytest
import torch

import gated_delta_rule_20_gb300 as gdn
import workloads
from gpu_util import check_whole, oracle_for, rel_l2, to64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _status_clean():
    gdn.device_status(0, clear=True)
    yield
    assert gdn.device_status(0, clear=True) == 0, "a kernel reported a wait timeout"


def segments(w):
    """The segment count gdn_prefill picks for workload w on this GPU (1: one pass)."""
    return gdn.prefill_segments(w.B, w.Hk, w.Hv, w.S)


def starts(w):
    """The first token of every segment gdn_prefill picks for workload w on this GPU, then S."""
    return gdn.prefill_segment_starts(w.B, w.Hk, w.Hv, w.S)


# name, B, Hk, Hv, S, state std, log-decay range, beta std, seed; each case is compared with
# the oracle over the whole output and final-state tensors
CASES = [
    ("b1_hv2_s2000_state_ragged", 1, 1, 2, 2000, 0.02, (-0.5, -0.005), 1.0, 101),
    ("b1_hv1_s4608_zero_start", 1, 1, 1, 4608, 0.0, (-0.5, -0.005), 1.0, 102),
    ("b2_hk2_hv8_s3072_gqa4", 2, 2, 8, 3072, 0.05, (-0.5, -0.005), 1.0, 103),
    ("b1_hv2_s3000_weak_decay", 1, 1, 2, 3000, 0.05, (-0.01, -0.0001), 1.0, 104),
    ("b1_hk2_hv4_s2500_strong_decay", 1, 2, 4, 2500, 0.05, (-2.0, -0.001), 2.0, 105),
    # almost no decay: the state persists through every segment, so the maps carry it
    ("b1_hv2_s4096_almost_no_decay", 1, 1, 2, 4096, 0.05, (-1e-4, -1e-6), 1.0, 107),
    # 50 sequences: two segments, 150 CTAs in one wave
    ("b2_hk5_hv25_s4096_two_segments", 2, 5, 25, 4096, 0.02, (-0.5, -0.005), 1.0, 106),
    # 64 sequences: the runs take two waves of CTAs
    ("b2_hk4_hv32_s8192_two_waves", 2, 4, 32, 8192, 0.02, (-0.5, -0.005), 1.0, 108),
]


def _inputs(case):
    _, B, Hk, Hv, S, st, g, bs, seed = case
    w = workloads.PREFILL.with_(B=B, Hk=Hk, Hv=Hv, S=S, dtype="bf16", state_std=st, seed=seed, g_lo=g[0],
                                g_hi=g[1], beta_std=bs)
    return w, workloads.make_inputs(w, device=DEV)


def _run(x, single_pass=False):
    st = x["state"].clone() if x["state"] is not None else None
    out, st = gdn.prefill(x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], st, single_pass=single_pass)
    torch.cuda.synchronize()
    return out, st


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_split_prefill_matches_oracle(case):
    w, x = _inputs(case)
    if segments(w) < 2:  # every case splits on a 152-SM GB300
        pytest.skip("not split on this GPU")
    out, st = _run(x)
    ro, rs = oracle_for(x)
    check_whole(out, st, ro, rs, case[0])


@pytest.mark.parametrize("case", CASES[:4], ids=[c[0] for c in CASES[:4]])
def test_split_prefill_agrees_with_one_pass(case):
    w, x = _inputs(case)
    o1, s1 = _run(x)
    o2, s2 = _run(x, single_pass=True)
    assert rel_l2(to64(o1), to64(o2)) < 1e-2
    assert rel_l2(to64(s1), to64(s2)) < 1e-2
    # segment 0 runs from the real start state in both forms, on the same kernel and tokens
    L = starts(w)[1]
    assert 0 < L < w.S
    assert torch.equal(o1[:, :, :L], o2[:, :, :L])


def test_split_prefill_is_taken():
    """With weak decay a segment's start state still matters at its end, so the start states
    the combine step derives differ in rounding from the one-pass chain: the later segments'
    outputs differ bit-wise (within the tolerance above).  (With the workloads' stronger
    decay the start state fades below fp32 resolution inside a segment, and both forms can
    agree bit for bit.)"""
    w, x = _inputs(CASES[3])
    o1, _ = _run(x)
    o2, _ = _run(x, single_pass=True)
    assert not torch.equal(o1, o2)


def test_split_prefill_writes_every_output_once():
    """Outputs pre-filled with NaN and guard elements around out and state: the split form
    writes every output element (no NaN left) and nothing outside the buffers."""
    from gpu_util import run_prefill
    _, x = _inputs(CASES[0])
    out, st = run_prefill(x, guard=256)
    o2, s2 = _run(x)
    assert torch.equal(out, o2) and torch.equal(st, s2)


def test_split_prefill_deterministic():
    _, x = _inputs(CASES[0])
    o1, s1 = _run(x)
    o2, s2 = _run(x)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_split_prefill_deterministic_over_many_waves():
    """A split whose runs take several waves of CTAs (32 sequences, later segments paired on
    the same inputs), repeated: every output and state bit-identical.  Catches ordering races
    inside a CTA that only show when a run's first input load lands early (from L2) -- such
    a race perturbs a segment's first chunks by less than the parity tolerance."""
    w = workloads.LONG_PREFILL.with_(S=8192, seed=31)
    assert segments(w) > 1
    x = workloads.make_inputs(w, device=DEV)
    ref_out, ref_st = _run(x)
    for _ in range(10):
        out, st = _run(x)
        assert torch.equal(out, ref_out) and torch.equal(st, ref_st)


def test_split_prefill_graph_replay():
    """The split form (its stream-ordered scratch included) captured in a CUDA graph and
    replayed gives the eager result bit for bit."""
    _, x = _inputs(CASES[0])
    o_ref, s_ref = _run(x)
    st = x["state"].clone()
    out = torch.empty_like(o_ref)

    def call():
        gdn.prefill(x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], st, out)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside the capture
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for _ in range(2):
        st.copy_(x["state"])
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, o_ref) and torch.equal(st, s_ref)


def test_caller_workspace_matches_own_scratch():
    """gdn_prefill_ws: a split prefill with the caller's scratch gives bit-identical results, a
    one-pass shape needs none, and a workspace one 16-byte step too small is refused before
    anything runs."""
    w = workloads.LONG_PREFILL.with_(S=8192, seed=31)
    assert segments(w) > 1
    need = gdn.prefill_workspace_bytes(w.B, w.Hk, w.Hv, w.S, w.Dk, w.Dv)
    P, s1, heads = segments(w), starts(w)[1], w.B * w.Hv
    # 3 (P - 1) states per sequence, one identity, the zero v tile, C after segment 0 (bf16)
    assert need == (3 * (P - 1) * heads * 128 * 128 + 128 * 128) * 4 + 64 * 128 * 2 + heads * (w.S - s1) * 128 * 2
    assert gdn.prefill_workspace_bytes(w.B, w.Hk, w.Hv, w.S, w.Dk, w.Dv, single_pass=True) == 0
    assert gdn.prefill_workspace_bytes(4, 16, 32, 4096, 128, 128) == 0  # one pass
    x = workloads.make_inputs(w, device=DEV)
    ref_out, ref_st = _run(x)
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device=DEV)  # stale contents must not matter
    for _ in range(2):  # twice in a row with the same workspace
        out, st = gdn.prefill(x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], None, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(st, ref_st)
    small = ws[: need - 16]
    out = torch.full_like(ref_out, float("nan"))
    with pytest.raises(gdn.GdnError) as e:
        gdn.prefill(x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], None, out, workspace=small)
    assert e.value.code == gdn.GDN_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all(), "a refused call launched work"

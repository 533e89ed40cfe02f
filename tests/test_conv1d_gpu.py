"""GPU parity of the depthwise causal conv1d + SiLU (``gdn_conv1d_prefill`` /
``gdn_conv1d_decode``, "GDN Conv1D Kernel API Reference") against the fp64
oracle ``oracle.conv1d``, through the C ABI.

Bars: the new conv_state is a copy of raw tokens, so it must be bit-exact.
Outputs meet the stated floating-point bars (bf16: relative L2 <= 1e-2; fp32:
|d| <= 1e-4 (1 + |ref|)) and, as a tighter check, every bf16 output is within
one bf16 rounding of the fp64 value: |d| <= 2^-8 |ref| + 1e-5 (the fp32 FIR and
SiLU add ~1e-6 relative before the final round-to-nearest, which costs at most
2^-9 relative)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import conv1d as oc  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import gated_delta_rule_20_gb300 as g
    g.lib()
    return g


def _inputs(B, C, T, K, dtype, seed, decode=False):
    w = workloads.ConvWorkload("t", "decode" if decode else "prefill", B, C, T, K, dtype, seed)
    return workloads.make_conv_inputs(w, device="cuda")


def _check_out(gpu, ref, dtype, what):
    g = gpu.double().cpu().numpy()
    d = g - ref
    assert np.isfinite(g).all(), what + ": non-finite output"
    if dtype == "bf16":
        rel = np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30)
        assert rel <= 1e-2, "%s: rel L2 %.3e" % (what, rel)
        bad = np.abs(d) > 2.0 ** -8 * np.abs(ref) + 1e-5
        assert not bad.any(), "%s: %d elements beyond one bf16 rounding, worst |d| %.3e" % (
            what, bad.sum(), np.abs(d).max())
    else:
        bad = np.abs(d) > 1e-4 * (1.0 + np.abs(ref))
        assert not bad.any(), "%s: %d elements beyond 1e-4 (1 + |ref|)" % (what, bad.sum())


def _run_prefill(gdn, x, w, misalign=False):
    if misalign:  # an unaligned view forces the scalar path
        buf = torch.empty(x.numel() + 1, dtype=x.dtype, device=x.device)
        xv = buf[1:].view(x.shape)
        xv.copy_(x)
        obuf = torch.full((x.numel() + 1,), float("nan"), dtype=x.dtype, device=x.device)
        out = obuf[1:].view(x.shape)
        out, st = gdn.conv1d_prefill(xv, w, out=out)
    else:
        out = torch.full_like(x, float("nan"))
        out, st = gdn.conv1d_prefill(x, w, out=out)
    torch.cuda.synchronize()
    return out, st


SHAPES = [(1, 8, 1, 4), (2, 16, 3, 4), (2, 64, 64, 4), (1, 128, 100, 3), (2, 256, 1024, 4), (1, 32, 17, 1),
          (1, 64, 96, 8), (3, 40, 8, 4), (1, 24, 200, 7)]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,C,T,K", SHAPES)
def test_prefill_shapes(gdn, B, C, T, K, dtype):
    x = _inputs(B, C, T, K, dtype, seed=B * 1000 + C + T + K)
    out, st = _run_prefill(gdn, x["x"], x["weight"])
    ref, ref_st = oc.conv1d_prefill(x["x"], x["weight"])
    _check_out(out, ref, dtype, "prefill %s" % ((B, C, T, K, dtype),))
    assert torch.equal(st.cpu(), torch.from_numpy(ref_st).to(st.dtype)), "conv_state is not the raw tail"


@pytest.mark.parametrize("B,C,T,K", [(2, 64, 64, 4), (1, 32, 100, 4)])
def test_prefill_unaligned_takes_the_scalar_path(gdn, B, C, T, K):
    x = _inputs(B, C, T, K, "bf16", seed=7)
    out, st = _run_prefill(gdn, x["x"], x["weight"], misalign=True)
    ref, ref_st = oc.conv1d_prefill(x["x"], x["weight"])
    _check_out(out, ref, "bf16", "unaligned prefill")
    assert torch.equal(st.cpu(), torch.from_numpy(ref_st).to(st.dtype))


def test_prefill_no_tokens_zeroes_the_state(gdn):
    x = torch.empty((2, 16, 0), dtype=torch.bfloat16, device="cuda")
    w = torch.ones((16, 4), dtype=torch.float32, device="cuda")
    st = torch.full((2, 16, 4), 3.0, dtype=torch.bfloat16, device="cuda")
    _, st = gdn.conv1d_prefill(x, w, conv_state=st)
    torch.cuda.synchronize()
    assert torch.count_nonzero(st).item() == 0


def test_prefill_empty_batch_is_a_noop(gdn):
    x = torch.empty((0, 16, 32), dtype=torch.bfloat16, device="cuda")
    w = torch.ones((16, 4), dtype=torch.float32, device="cuda")
    out, st = gdn.conv1d_prefill(x, w)
    torch.cuda.synchronize()
    assert out.numel() == 0 and st.numel() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,C,K", [(1, 8, 4), (4, 300, 4), (64, 8192, 4), (2, 50, 1), (3, 33, 8)])
def test_decode_shapes(gdn, B, C, K, dtype):
    x = _inputs(B, C, 1, K, dtype, seed=B + C + K, decode=True)
    st_in = x["state"].clone()
    out, st = gdn.conv1d_decode(x["x"], x["weight"], x["state"])
    torch.cuda.synchronize()
    ref, ref_st = oc.conv1d_decode(x["x"], st_in, x["weight"])
    _check_out(out, ref, dtype, "decode %s" % ((B, C, K, dtype),))
    assert torch.equal(st.cpu(), torch.from_numpy(ref_st).to(st.dtype)), "window not shifted exactly"


def test_decode_chain_matches_the_prefill_oracle(gdn):
    """Nine decode steps from a zero window == the prefill of the nine tokens."""
    B, C, T, K = 2, 96, 9, 4
    x = _inputs(B, C, T, K, "bf16", seed=99)
    st = torch.zeros((B, C, K), dtype=torch.bfloat16, device="cuda")
    outs = []
    for t in range(T):
        o, st = gdn.conv1d_decode(x["x"][:, :, t:t + 1].contiguous(), x["weight"], st)
        outs.append(o)
    torch.cuda.synchronize()
    ref, ref_st = oc.conv1d_prefill(x["x"], x["weight"])
    _check_out(torch.cat(outs, dim=2), ref, "bf16", "decode chain")
    assert torch.equal(st.cpu(), torch.from_numpy(ref_st).to(st.dtype))


def test_full_size_prefill_sampled(gdn):
    """The benchmark workload (B=4, C=8192, T=4096, K=4), as the bench launches it;
    64 channels sampled (channels are independent FIRs)."""
    w = workloads.CONV_PREFILL
    x = workloads.make_conv_inputs(w, device="cuda")
    out, st = _run_prefill(gdn, x["x"], x["weight"])
    ch = np.random.default_rng(0).choice(w.C, 64, replace=False)
    ch_t = torch.from_numpy(ch).cuda()
    ref, ref_st = oc.conv1d_prefill(x["x"].index_select(1, ch_t), x["weight"].index_select(0, ch_t))
    _check_out(out.index_select(1, ch_t), ref, "bf16", "full-size prefill")
    assert torch.equal(st.index_select(1, ch_t).cpu(), torch.from_numpy(ref_st).to(st.dtype))
    assert gdn.device_status(0) == 0

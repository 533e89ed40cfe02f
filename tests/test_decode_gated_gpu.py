"""GPU parity of the gated single-token step (``gdn_decode_gated``) against the
fp64 oracle ``oracle.gated_decode``, through the C ABI.

Bars (the stated ones): bf16 compute, relative L2 <= 1e-2 on out and on the
final state; fp32 compute, |d| <= 1e-4 (1 + |ref|) elementwise."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import gated_decode as og  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import gated_delta_rule_20_gb300 as g
    g.lib()
    return g


def _check(gpu, ref, dtype, what):
    g = gpu.double().cpu().numpy()
    assert np.isfinite(g).all(), what + ": non-finite"
    if dtype == "bf16":
        rel = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30)
        assert rel <= 1e-2, "%s: rel L2 %.3e" % (what, rel)
    else:
        bad = np.abs(g - ref) > 1e-4 * (1.0 + np.abs(ref))
        assert not bad.any(), "%s: %d elements beyond 1e-4 (1 + |ref|), worst %.3e" % (
            what, bad.sum(), np.abs(g - ref).max())


def _run(gdn, w, zero_state=False):
    x = workloads.make_gated_inputs(w.with_(state_std=0.0 if zero_state else w.state_std), device="cuda")
    st = torch.full((w.B, w.Hv, w.Dk, w.Dv), float("nan") if zero_state else 0.0, dtype=torch.float32,
                    device="cuda") if zero_state else x["state"].clone()
    out, st = gdn.decode_gated(x["qkv"], x["z"], x["a"], x["b"], x["A_log"], x["dt_bias"], x["norm_weight"],
                               x["scale"], st, w.Hk, w.Hv, w.Dk, w.Dv, zero_initial_state=zero_state)
    torch.cuda.synchronize()
    ref_out, ref_st = og.decode_gated(x["qkv"], x["z"], x["a"], x["b"], x["A_log"], x["dt_bias"],
                                      x["norm_weight"], x["scale"], None if zero_state else x["state"],
                                      w.Hk, w.Hv, w.Dk, w.Dv)
    return out, st, ref_out, ref_st


SHAPES = [(1, 1, 1, 128, 128), (2, 2, 4, 64, 64), (3, 1, 3, 32, 48), (2, 2, 2, 128, 100), (2, 4, 8, 17, 128),
          (5, 2, 6, 128, 128)]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,Hk,Hv,Dk,Dv", SHAPES)
def test_gated_shapes(gdn, B, Hk, Hv, Dk, Dv, dtype):
    w = workloads.GatedWorkload("t", B, Hk, Hv, Dk, Dv, dtype, 0.05, B * 100 + Hv * 10 + Dk + Dv)
    out, st, ro, rs = _run(gdn, w)
    _check(out, ro, dtype, "out %s" % ((B, Hk, Hv, Dk, Dv, dtype),))
    _check(st, rs, dtype, "state %s" % ((B, Hk, Hv, Dk, Dv, dtype),))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gated_zero_initial_state(gdn, dtype):
    w = workloads.GatedWorkload("t", 3, 2, 4, 128, 128, dtype, 0.0, 21)
    out, st, ro, rs = _run(gdn, w, zero_state=True)
    _check(out, ro, dtype, "zero-start out")
    _check(st, rs, dtype, "zero-start state")


def test_gated_full_size(gdn):
    """The decode block's size (B=64, Hk=16, Hv=32, D=128, bf16), every head."""
    out, st, ro, rs = _run(gdn, workloads.GATED_DECODE)
    _check(out, ro, "bf16", "full-size out")
    _check(st, rs, "bf16", "full-size state")

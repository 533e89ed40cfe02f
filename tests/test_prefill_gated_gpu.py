"""GPU parity of the RMSNormGated row pass (``gdn_rmsnorm_gated``) and of the gated
prefill (``gdn_prefill_gated``: the prefill, then the pass on its output) against
the fp64 oracles ``oracle.gated_decode.rms_norm_gated`` and
``oracle.prefill_gated``, through the C ABI.

Bars: fp32 |gpu - ref| <= 1e-4 (1 + |ref|) elementwise; bf16 relative L2 <= 1e-2
(the gated prefill rounds the recurrence's output to bf16 before the norm, as its
two launches hand it over in the output buffer)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import gated_decode as og  # noqa: E402
from oracle import prefill_gated as opg  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import gated_delta_rule_20_gb300 as g
    g.lib()
    return g


def _check(got, ref, dtype, what):
    g = got.double().cpu().numpy()
    assert np.isfinite(g).all(), what
    if dtype == "f32":
        err = np.abs(g - ref) / (1.0 + np.abs(ref))
        assert err.max() <= 1e-4, "%s: max scaled error %.3e" % (what, err.max())
    else:
        rel = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30)
        assert rel <= 1e-2, "%s: rel L2 %.3e" % (what, rel)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("rows,D", [(1000, 128), (37, 48), (5, 1), (3, 256)])
@pytest.mark.parametrize("in_place", [False, True])
def test_rmsnorm_gated(gdn, dtype, rows, D, in_place):
    gen = torch.Generator().manual_seed(rows * 7 + D)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    x = (3.0 * torch.randn((rows, D), generator=gen)).to(dt).cuda()
    z = torch.randn((rows, D), generator=gen).to(dt).cuda()
    w = (1.0 + 0.1 * torch.randn((D,), generator=gen)).cuda()
    ref = og.rms_norm_gated(x, z, w)
    out = gdn.rmsnorm_gated(x, z, w, out=x if in_place else None)
    torch.cuda.synchronize()
    _check(out, ref, dtype, "rmsnorm rows=%d D=%d" % (rows, D))


CASES = [workloads.TINY_PREFILL,
         workloads.PREFILL.with_(B=1, Hk=1, Hv=2, S=200, seed=31),
         workloads.PREFILL.with_(B=2, Hk=2, Hv=4, S=130, state_std=0.0, seed=32),
         # two long sequences: the prefill runs split into segments
         workloads.PREFILL.with_(B=1, Hk=1, Hv=2, S=1800, seed=33)]


@pytest.mark.parametrize("w", CASES, ids=lambda w: "%s_b%d_hv%d_s%d" % (w.dtype, w.B, w.Hv, w.S))
def test_prefill_gated(gdn, w):
    x = workloads.make_inputs(w, device="cuda")
    gz = workloads.make_gate_inputs(w, device="cuda")
    st = x["state"].clone() if x["state"] is not None else None
    out, st = gdn.prefill_gated(x["q"], x["k"], x["v"], x["g_log"], x["beta"], gz["z"], gz["norm_weight"],
                                x["scale"], st)
    torch.cuda.synchronize()
    ry, rs = opg.prefill_gated(x["q"], x["k"], x["v"], x["g_log"], x["beta"], gz["z"], gz["norm_weight"], x["scale"],
                               x["state"])
    _check(out, ry, w.dtype, "gated prefill out")
    _check(st, rs, "f32" if w.dtype == "f32" else "bf16", "gated prefill state")
    assert gdn.device_status(0) == 0


def test_prefill_gated_full_size(gdn):
    """The bench's size (B=4, Hk=16, Hv=32, S=4096, bf16, tcgen05 path), compared with the
    oracle over every (batch, value head) sequence: relative L2 over the whole gated output
    and the whole final state."""
    from gpu_util import check_whole
    w = workloads.PREFILL
    x = workloads.make_inputs(w, device="cuda")
    gz = workloads.make_gate_inputs(w, device="cuda")
    out, st = gdn.prefill_gated(x["q"], x["k"], x["v"], x["g_log"], x["beta"], gz["z"], gz["norm_weight"],
                                x["scale"], x["state"].clone())
    torch.cuda.synchronize()
    ry, rs = opg.prefill_gated(x["q"], x["k"], x["v"], x["g_log"], x["beta"], gz["z"], gz["norm_weight"], x["scale"],
                               x["state"])
    check_whole(out, st, ry, rs, "full-size gated prefill")
    assert gdn.device_status(0) == 0

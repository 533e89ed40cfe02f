"""GPU parity of the decode block without its output projection
(``gdn_decode_block``: input projections on tcgen05, conv1d decode, gated step)
against the fp64 oracle ``oracle.decode_block``, through the C ABI.

The GPU rounds every inter-stage activation (the projections, the conv output)
to bf16, as the page's bf16 activations do; the oracle keeps them exact.  The
bar is the stated bf16 one: relative L2 <= 1e-2 on out, on the new conv window
and on the new state."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import decode_block as ob  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import gated_delta_rule_20_gb300 as g
    g.lib()
    return g


def _rel(g, ref):
    g = g.double().cpu().numpy()
    assert np.isfinite(g).all()
    return np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30)


# (B, H, Hk, Hv, Dk, Dv, K): C = 2 Hk Dk + Hv Dv, value_dim and Hv multiples of 8
SHAPES = [(2, 128, 2, 8, 64, 64, 4), (5, 192, 4, 8, 32, 48, 3), (130, 256, 1, 8, 128, 128, 4),
          (1, 64, 2, 8, 16, 8, 1), (64, 2048, 16, 32, 128, 128, 4)]


@pytest.mark.parametrize("B,H,Hk,Hv,Dk,Dv,K", SHAPES)
def test_block(gdn, B, H, Hk, Hv, Dk, Dv, K):
    w = workloads.BlockWorkload("t", B, H, Hk, Hv, Dk, Dv, K, seed=B + H + Hv + Dk + K)
    x = workloads.make_block_inputs(w, device="cuda")
    cst, st = x["conv_state"].clone(), x["state"].clone()
    out, cst, st = gdn.decode_block(x["hidden"], x["W_qkv"], x["W_z"], x["W_a"], x["W_b"], x["conv_weight"], cst,
                                    x["A_log"], x["dt_bias"], x["norm_weight"], st, Hk, Hv, Dk, Dv)
    torch.cuda.synchronize()
    ro, rc, rs = ob.decode_block(x["hidden"], x["W_qkv"], x["W_z"], x["W_a"], x["W_b"], x["conv_weight"],
                                 x["conv_state"], x["A_log"], x["dt_bias"], x["norm_weight"], x["state"],
                                 Hk, Hv, Dk, Dv)
    for what, g, r in (("out", out, ro), ("conv_state", cst, rc), ("state", st, rs)):
        e = _rel(g, r)
        assert e <= 1e-2, "%s %s: rel L2 %.3e" % (what, (B, H, Hk, Hv, Dk, Dv, K), e)
    assert gdn.device_status(0) == 0


def test_block_workspace_too_small_is_refused(gdn):
    w = workloads.BlockWorkload("t", 2, 128, 2, 8, 64, 64, 4, seed=3)
    x = workloads.make_block_inputs(w, device="cuda")
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(gdn.GdnError) as e:
        gdn.decode_block(x["hidden"], x["W_qkv"], x["W_z"], x["W_a"], x["W_b"], x["conv_weight"], x["conv_state"],
                         x["A_log"], x["dt_bias"], x["norm_weight"], x["state"], 2, 8, 64, 64, workspace=ws)
    assert e.value.code == gdn.GDN_ERR_DIMS


def test_block_three_tokens_in_a_row(gdn):
    """Three calls back to back on one stream, each feeding the next through the conv
    window and the state: the gated step of a call starts while that call's projections
    still run, so this checks that it reads their outputs, and the previous call's state,
    only once they are complete."""
    w = workloads.BlockWorkload("t", 64, 2048, 16, 32, 128, 128, 4, seed=21)
    x = workloads.make_block_inputs(w, device="cuda")
    gen = torch.Generator(device="cpu").manual_seed(22)
    hiddens = [x["hidden"]] + [torch.randn(x["hidden"].shape, generator=gen).to(torch.bfloat16).cuda()
                               for _ in range(2)]
    cst, st = x["conv_state"].clone(), x["state"].clone()
    outs = []
    for h in hiddens:
        out, cst, st = gdn.decode_block(h, x["W_qkv"], x["W_z"], x["W_a"], x["W_b"], x["conv_weight"], cst,
                                        x["A_log"], x["dt_bias"], x["norm_weight"], st, 16, 32, 128, 128)
        outs.append(out.clone())
    torch.cuda.synchronize()
    rc, rs = x["conv_state"], x["state"]
    for i, h in enumerate(hiddens):
        ro, rc, rs = ob.decode_block(h, x["W_qkv"], x["W_z"], x["W_a"], x["W_b"], x["conv_weight"], rc,
                                     x["A_log"], x["dt_bias"], x["norm_weight"], rs, 16, 32, 128, 128)
        e = _rel(outs[i], ro)
        assert e <= 1e-2, "token %d: out rel L2 %.3e" % (i, e)
    assert _rel(cst, rc) <= 1e-2 and _rel(st, rs) <= 1e-2
    assert gdn.device_status(0) == 0

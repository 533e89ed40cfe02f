"""The library's calls under CUDA-graph stream capture (the way a serving loop
replays a decode step): a captured decode block (two launches, the second a
programmatic dependent of the first), decode step and prefill, replayed, give
the same results as the same calls run eagerly on copies of the inputs."""
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import gated_delta_rule_20_gb300 as g
    g.lib()
    return g


def _replay_vs_eager(capture_fn, eager_fn, n_replays=3):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside the capture (attributes, status words)
        capture_fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        capture_fn()
    for _ in range(n_replays):
        g.replay()
        eager_fn()
    torch.cuda.synchronize()


def test_decode_block_graph(gdn):
    w = workloads.DECODE_BLOCK.with_(seed=41)
    x = workloads.make_block_inputs(w, device="cuda")
    ws = torch.empty(gdn.decode_block_workspace_bytes(w.B, w.H, w.Hk, w.Hv, w.Dk, w.Dv, w.K), dtype=torch.uint8,
                     device="cuda")
    ws2 = torch.empty_like(ws)
    a = dict(cst=x["conv_state"].clone(), st=x["state"].clone(), out=torch.empty(w.B, 1, w.Hv * w.Dv,
                                                                                    dtype=torch.bfloat16, device="cuda"))
    b = dict(cst=x["conv_state"].clone(), st=x["state"].clone(), out=torch.empty_like(a["out"]))

    def call(t, wsp):
        gdn.decode_block(x["hidden"], x["W_qkv"], x["W_z"], x["W_a"], x["W_b"], x["conv_weight"], t["cst"],
                         x["A_log"], x["dt_bias"], x["norm_weight"], t["st"], w.Hk, w.Hv, w.Dk, w.Dv, out=t["out"],
                         workspace=wsp)

    _replay_vs_eager(lambda: call(a, ws), lambda: call(b, ws2))
    # the warm-up ran on a only: b is one step behind, so bring it level
    call(b, ws2)
    torch.cuda.synchronize()
    for k in ("out", "cst", "st"):
        assert torch.equal(a[k], b[k]), k
    assert gdn.device_status(0) == 0


def test_decode_and_prefill_graph(gdn):
    wd = workloads.DECODE_STEP.with_(seed=42)
    xd = workloads.make_inputs(wd, device="cuda")
    sa, sb = xd["state"].clone(), xd["state"].clone()
    oa, ob = torch.empty_like(xd["v"]), torch.empty_like(xd["v"])
    dec = lambda st, o: gdn.decode_step(xd["q"], xd["k"], xd["v"], xd["g_log"], xd["beta"], xd["scale"], st, o)
    _replay_vs_eager(lambda: dec(sa, oa), lambda: dec(sb, ob))
    dec(sb, ob)
    torch.cuda.synchronize()
    assert torch.equal(oa, ob) and torch.equal(sa, sb)

    wp = workloads.PREFILL.with_(B=1, Hk=2, Hv=4, S=300, seed=43)
    xp = workloads.make_inputs(wp, device="cuda")
    pa, pb = xp["state"].clone(), xp["state"].clone()
    qa, qb = torch.empty_like(xp["v"]), torch.empty_like(xp["v"])
    pre = lambda st, o: gdn.prefill(xp["q"], xp["k"], xp["v"], xp["g_log"], xp["beta"], xp["scale"], st, o)
    _replay_vs_eager(lambda: pre(pa, qa), lambda: pre(pb, qb))
    pre(pb, qb)
    torch.cuda.synchronize()
    assert torch.equal(qa, qb) and torch.equal(pa, pb)
    assert gdn.device_status(0) == 0

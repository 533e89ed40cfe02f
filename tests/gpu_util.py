"""Helpers shared by the GPU tests: run the library and the oracle on the same
seeded inputs and compare with the tolerances of the method's contract."""
import numpy as np
import torch

import gated_delta_rule_20_gb300 as gdn
import oracle

# fp32 compute: elementwise |gpu - ref| <= 1e-4 (1 + |ref|).
F32_ATOL = 1e-4
# bf16 compute: relative L2 error <= 1e-2 over out and over the final state.
BF16_REL_L2 = 1e-2


def rel_l2(a, ref):
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(a - ref) / max(np.linalg.norm(ref), 1e-300))


def to64(t):
    return t.detach().to("cpu").double().numpy()


def sample_heads(x, heads, G):
    """Inputs of the listed (b, h) sequences, stacked as a batch of Hk = Hv = 1."""
    def pick(t, kv):
        if t is None:
            return None
        rows = [t[b, (h // G) if kv else h] for (b, h) in heads]
        return torch.stack(rows).unsqueeze(1)
    return dict(q=pick(x["q"], True), k=pick(x["k"], True), v=pick(x["v"], False),
                g_log=pick(x["g_log"], False), beta=pick(x["beta"], False), state=pick(x["state"], False))


def oracle_for(x, heads=None, G=None):
    if heads is None:
        return oracle.recurrence(x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], x["state"])
    s = sample_heads(x, heads, G)
    o, st = oracle.recurrence(s["q"], s["k"], s["v"], s["g_log"], s["beta"], x["scale"], s["state"])
    return o[:, 0], st[:, 0]


def check(out, state, ref_out, ref_state, bf16, what=""):
    o, s = to64(out), to64(state)
    assert np.isfinite(o).all() and np.isfinite(s).all(), what + ": non-finite values"
    if bf16:
        eo, es = rel_l2(o, ref_out), rel_l2(s, ref_state)
        assert eo <= BF16_REL_L2, "%s: out rel L2 %.3e" % (what, eo)
        assert es <= BF16_REL_L2, "%s: state rel L2 %.3e" % (what, es)
        return eo, es
    bo = np.abs(o - ref_out) - F32_ATOL * (1.0 + np.abs(ref_out))
    bs = np.abs(s - ref_state) - F32_ATOL * (1.0 + np.abs(ref_state))
    assert bo.max() <= 0, "%s: out max excess %.3e" % (what, bo.max())
    assert bs.max() <= 0, "%s: state max excess %.3e" % (what, bs.max())
    return float(np.abs(o - ref_out).max()), float(np.abs(s - ref_state).max())


def check_whole(out, state, ref_out, ref_state, what=""):
    """bf16 contract over the WHOLE tensors: relative L2 of out and of the final state,
    each taken over every element of every (batch, value head) sequence.  The worst
    per-sequence relative L2 is printed as a diagnostic (not asserted: a sequence whose
    reference output is tiny can have a large relative error that the contract allows)."""
    o, s = to64(out), to64(state)
    assert np.isfinite(o).all() and np.isfinite(s).all(), what + ": non-finite values"
    eo, es = rel_l2(o, ref_out), rel_l2(s, ref_state)
    n = o.shape[0] * o.shape[1]

    def worst(a, ref):
        d = np.linalg.norm((a - ref).reshape(n, -1), axis=1)
        r = np.maximum(np.linalg.norm(np.asarray(ref).reshape(n, -1), axis=1), 1e-300)
        i = int(np.argmax(d / r))
        return float(d[i] / r[i]), divmod(i, o.shape[1])

    wo, io = worst(o, ref_out)
    ws, is_ = worst(s, ref_state)
    print("%s: %d sequences; out rel L2 %.3e (worst sequence %.3e at (b, h) = %s); "
          "state rel L2 %.3e (worst %.3e at %s)" % (what, n, eo, wo, io, es, ws, is_))
    assert eo <= BF16_REL_L2, "%s: out rel L2 %.3e" % (what, eo)
    assert es <= BF16_REL_L2, "%s: state rel L2 %.3e" % (what, es)
    return eo, es


def run_prefill(x, force_ffma=False, guard=0):
    """Call the library; outputs are pre-filled with NaN so an unwritten element
    shows, and optional guard elements around out and state must stay untouched."""
    q = x["q"]
    B, Hk, S, Dk = q.shape
    Hv, Dv = x["v"].shape[1], x["v"].shape[3]
    n_out = B * Hv * S * Dv
    out_buf = torch.full((n_out + 2 * guard,), float("nan"), dtype=q.dtype, device=q.device)
    st_buf = torch.full((B * Hv * Dk * Dv + 2 * guard,), 7.25, dtype=torch.float32, device=q.device)
    out = out_buf[guard:guard + n_out].view(B, Hv, S, Dv)
    state = st_buf[guard:guard + B * Hv * Dk * Dv].view(B, Hv, Dk, Dv)
    zero = x["state"] is None
    if not zero:
        state.copy_(x["state"])
    from gated_delta_rule_20_gb300 import _binding
    _binding._call("gdn_prefill", x["q"], x["k"], x["v"], x["g_log"], x["beta"], x["scale"], state, out, zero,
                   force_ffma, None)
    torch.cuda.synchronize()
    if guard:
        assert torch.isnan(out_buf[:guard].float()).all() and torch.isnan(out_buf[-guard:].float()).all()
        assert (st_buf[:guard] == 7.25).all() and (st_buf[-guard:] == 7.25).all()
    return out, state

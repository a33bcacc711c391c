"""gdn_chunked_prefill_noalloc: the chunked prefill on the library's static
per-device scratch instead of a caller workspace.  (None of the reference
pages has this entry point; it is checked against the workspace entry point,
which the other chunked tests check against the oracle, and against the
oracle directly.)"""
import ctypes

import numpy as np
import pytest
import torch

from gated_delta_rule_gate_gb300 import _native as N
from gated_delta_rule_gate_gb300 import api

FAKE = 0x100000  # 256-byte aligned, never dereferenced by the host
SCRATCH = 768 << 20


def _problem(**over):
    p = N.GdnProblem()
    p.batch, p.total_tokens, p.seq_len = 1, 64, 0
    p.num_heads_q, p.num_heads_v, p.head_dim_k, p.head_dim_v = 1, 1, 128, 128
    p.num_state_rows = 0
    p.act_dtype, p.decay_dtype, p.beta_dtype = N.DTYPE_F16, N.DTYPE_F32, N.DTYPE_F32
    p.rule, p.flags, p.scale, p.state_update_capacity = N.RULES["gated_delta"], 0, 0.0, 0
    for f in ("q", "k", "v", "o", "decay", "beta", "final_state"):
        setattr(p, f, FAKE)
    for k, v in over.items():
        setattr(p, k, v)
    return p


def test_exported_and_declared():
    assert hasattr(N.load(), "gdn_chunked_prefill_noalloc")
    assert "gdn_chunked_prefill_noalloc" in N.EXPORTS


def test_oversize_rejected_on_the_host():
    """A problem whose workspace exceeds the 768 MiB scratch is refused before
    anything is enqueued (no GPU needed)."""
    lib = N.load()
    p = _problem(batch=4, total_tokens=4 * 32768, num_heads_q=32, num_heads_v=32)
    need = lib.gdn_chunked_prefill_workspace_size(ctypes.byref(p), 64)
    assert need > SCRATCH
    assert lib.gdn_chunked_prefill_noalloc(ctypes.byref(p), 64, None) == N.GDN_ERR_WORKSPACE
    assert "static scratch" in N.last_error_message()
    # the same argument checks as the workspace entry point come first
    bad = _problem(head_dim_k=12, head_dim_v=9)
    assert lib.gdn_chunked_prefill_noalloc(ctypes.byref(bad), 64, None) == N.GDN_ERR_UNSUPPORTED


def _noalloc_like(p, d, o1, f1, rule):
    """Runs the problem already run through the workspace entry point (o1, f1)
    through the no-alloc entry point into fresh outputs."""
    o2 = torch.full_like(o1, float("nan"))
    f2 = torch.full_like(f1, float("nan"))
    prob = api.make_problem(q=d["q"], k=d["k"], v=d["v"], o=o2, final_state=f2, rule=rule,
                            decay=d.get("decay"), beta=d.get("beta"), gate_bias=d.get("gate_bias"),
                            gate_scale=d.get("gate_scale"), cu_seqlens=d.get("cu_seqlens"),
                            initial_state=d.get("initial_state"), batch=p["batch"],
                            l2norm_k=p.get("l2norm_k", False), beta_sigmoid=p.get("beta_sigmoid", False),
                            decay_per_key=p.get("decay_per_key", False))
    api.gdn_chunked_prefill_noalloc(prob)
    return o2, f2


@pytest.mark.gpu
@pytest.mark.parametrize("rule,per_key", [("gated_delta", False), ("delta", False), ("linear", False),
                                          ("gdn2", True)])
def test_same_result_as_the_workspace_entry_point(rule, per_key):
    """Two no-alloc calls in a row (different problems, the second reusing the
    scratch the first left behind), each bit-exact against the workspace entry
    point; the first also against the oracle."""
    import oracle
    import workloads
    from gpu_helpers import o_flat, rel_err, run
    extra = dict(decay_per_key=True, gate_dtype="f32", write_gate=True) if per_key else {}
    pa = workloads.make(seed=81, B=3, lengths=[130, 0, 75], hq=2, hv=4, dk=128, dv=128, act="f16",
                        rule=rule, state="random", state_std=0.3, **extra)
    pb = workloads.make(seed=82, B=2, lengths=[64, 257], hq=1, hv=2, dk=128, dv=128, act="f16",
                        rule=rule, state="random", state_std=0.3, **extra)
    oa, fa, da = run(pa, path="chunked")
    ob, fb, db = run(pb, path="chunked")
    oa2, fa2 = _noalloc_like(pa, da, oa, fa, rule)
    ob2, fb2 = _noalloc_like(pb, db, ob, fb, rule)
    torch.cuda.synchronize()
    for x1, x2 in ((oa, oa2), (fa, fa2), (ob, ob2), (fb, fb2)):
        assert torch.equal(x1.nan_to_num(7.0), x2.nan_to_num(7.0))
    ref_o, ref_fin, _ = oracle.run_problem(pa)
    covered = ~np.isnan(ref_o)
    assert rel_err(o_flat(oa2, pa)[covered], ref_o[covered]) <= 5e-3
    assert rel_err(fa2.double().cpu().numpy(), ref_fin) <= 5e-3


@pytest.mark.gpu
def test_full_size_ragged_prefill_fits_the_scratch():
    """The ragged prefill configuration (16384 tokens, Hv = 32) needs about
    765 MB of workspace: it runs on the static scratch."""
    import workloads
    from gpu_helpers import run
    p = workloads.ragged_prefill()
    o1, f1, d = run(p, path="chunked")
    o2 = torch.full_like(o1, float("nan"))
    f2 = torch.empty_like(f1)
    prob = api.make_problem(q=d["q"], k=d["k"], v=d["v"], o=o2, final_state=f2, rule=p["rule"],
                            decay=d.get("decay"), beta=d.get("beta"), gate_bias=d.get("gate_bias"),
                            gate_scale=d.get("gate_scale"), cu_seqlens=d.get("cu_seqlens"),
                            initial_state=d.get("initial_state"), batch=p["batch"],
                            l2norm_k=p.get("l2norm_k", False), beta_sigmoid=p.get("beta_sigmoid", False))
    need = api.gdn_chunked_prefill_workspace_size(prob)
    assert 0 < need <= SCRATCH
    api.gdn_chunked_prefill_noalloc(prob)
    torch.cuda.synchronize()
    assert torch.equal(o1.nan_to_num(7.0), o2.nan_to_num(7.0)) and torch.equal(f1, f2)

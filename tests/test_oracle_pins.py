"""Pins the CPU oracle to facts fixed by the pages and by mathematics.

None of these re-run the oracle's own loop: each compares it with a different
computation (the second algebraic form printed on the Ascend page, dense
transition-matrix products, exact rational arithmetic, closed forms of the
linear and gated rules) or with an invariant the recurrence must satisfy.
"""
import math
from fractions import Fraction

import numpy as np
import torch
import pytest

import oracle
import workloads


def _np(x):
    return None if x is None else np.asarray(x.double().numpy() if hasattr(x, "double") else x,
                                              dtype=np.float64)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


# --------------------------------------------------------------------------
# 1. "aclnnRecurrentGatedDeltaRule", Formula: the product form
#    S_t = S_{t-1} (alpha_t Diag(alpha_kt) (I - beta_t k_t k_t^T)) + beta_t v_t k_t^T
#    must equal the oracle's decay -> retrieve -> write loop.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("per_key", [False, True])
def test_product_form_equals_oracle(per_key):
    rng = np.random.default_rng(11)
    T, dk, dv = 9, 5, 4
    q = rng.standard_normal((T, 1, dk))
    k = _unit(rng.standard_normal((T, 1, dk)))
    v = rng.standard_normal((T, 1, dv))
    g = -rng.random((T, 1, dk) if per_key else (T, 1)) * 0.7
    beta = rng.random((T, 1))
    S0 = rng.standard_normal((1, 1, dv, dk)) * 0.3
    o, fin, _ = oracle.gdn(q, k, v, rule="gated_delta", decay=g, beta=beta, initial_state=S0,
                           decay_per_key=per_key, scale=0.7, cu_seqlens=[0, T])
    S = S0[0, 0].copy()
    for t in range(T):
        a = np.diag(np.exp(g[t, 0]) if per_key else np.full(dk, np.exp(g[t, 0])))
        kt = k[t, 0][:, None]
        S = S @ (a @ (np.eye(dk) - beta[t, 0] * kt @ kt.T)) + beta[t, 0] * v[t, 0][:, None] @ kt.T
        np.testing.assert_allclose(o[t, 0], 0.7 * S @ q[t, 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(fin[0, 0], S, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# 2. Exact recall: g = 0, beta = 1, unit keys  =>  S_t k_t = v_t.  Reading
#    with q_t = k_t gives o_t = scale * v_t (and it holds for any decay too).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("rule", ["delta", "gated_delta"])
def test_exact_recall(rule):
    rng = np.random.default_rng(12)
    T, dk, dv = 12, 8, 6
    k = rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    S0 = rng.standard_normal((1, 1, dv, dk))
    decay = -rng.random((T, 1)) * 2 if rule == "gated_delta" else None
    o, _, _ = oracle.gdn(k, k, v, rule=rule, decay=decay, beta=np.ones((T, 1)),
                         initial_state=S0, l2norm_q=True, l2norm_k=True, scale=0.5)
    np.testing.assert_allclose(o[:, 0], 0.5 * v[:, 0], rtol=1e-11, atol=1e-11)


# --------------------------------------------------------------------------
# 3. beta = 0 and g = 0: the state never changes and o_t = scale * S_0 q_t.
# --------------------------------------------------------------------------
def test_beta_zero_g_zero_is_identity():
    rng = np.random.default_rng(13)
    T, dk, dv = 7, 6, 5
    q = rng.standard_normal((T, 1, dk))
    k = rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 2, dv))
    S0 = rng.standard_normal((1, 2, dv, dk))
    o, fin, _ = oracle.gdn(q, k, v, rule="gated_delta", decay=np.zeros((T, 2)),
                           beta=np.zeros((T, 2)), initial_state=S0, scale=1.0)
    assert np.array_equal(fin, S0)
    for h in range(2):
        np.testing.assert_allclose(o[:, h], q[:, 0] @ S0[0, h].T, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# 4. ONNX issue "Spec gap ... Gated DeltaNet-2", Proposed extension: GDN-2
#    with b_t = beta_t * 1 recovers v1.  Option A's write term carries no beta,
#    so the matching write gate w_t = beta_t * 1 is folded into v by the caller.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("per_key_decay", [False, True])
def test_gdn2_reduces_to_gated_delta(per_key_decay):
    rng = np.random.default_rng(14)
    T, hv, dk, dv = 10, 2, 6, 5
    q = rng.standard_normal((T, 1, dk))
    k = _unit(rng.standard_normal((T, 1, dk)))
    v = rng.standard_normal((T, hv, dv))
    g = -rng.random((T, hv))
    beta = rng.random((T, hv))
    S0 = rng.standard_normal((1, hv, dv, dk)) * 0.2
    o1, f1, _ = oracle.gdn(q, k, v, rule="gated_delta", decay=g, beta=beta, initial_state=S0)
    b_vec = np.repeat(beta[:, :, None], dk, axis=2)
    g2 = np.repeat(g[:, :, None], dk, axis=2) if per_key_decay else g
    o2, f2, _ = oracle.gdn(q, k, v * beta[:, :, None], rule="gdn2", decay=g2, beta=b_vec,
                           initial_state=S0, decay_per_key=per_key_decay)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(f2, f1, rtol=1e-12, atol=1e-12)


def test_gdn2_erase_acts_on_key_side():
    """GDN-2 proposal (A): with a one-hot erase gate only the selected key
    channel is retrieved: S_t = S' - (S' (b .* k)) k^T + v k^T, checked against
    dense matrices (I - k (b.*k)^T) form of the first display of that issue."""
    rng = np.random.default_rng(15)
    T, dk, dv = 6, 4, 3
    q = rng.standard_normal((T, 1, dk))
    k = rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    b = rng.random((T, 1, dk))
    g = -rng.random((T, 1, dk))
    S0 = rng.standard_normal((1, 1, dv, dk))
    o, fin, _ = oracle.gdn(q, k, v, rule="gdn2", decay=g, beta=b, initial_state=S0,
                           decay_per_key=True, scale=1.0)
    # Key-major form of the issue: S_K = (I - k (b.*k)^T) D S_K + k v^T,
    # S_K = M^T (dk x dv).
    SK = S0[0, 0].T.copy()
    for t in range(T):
        kt = k[t, 0][:, None]
        bk = (b[t, 0] * k[t, 0])[:, None]
        SK = (np.eye(dk) - kt @ bk.T) @ np.diag(np.exp(g[t, 0])) @ SK + kt @ v[t, 0][None, :]
        np.testing.assert_allclose(o[t, 0], SK.T @ q[t, 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(fin[0, 0], SK.T, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# 5. Gate closed forms ("com.microsoft.LinearAttentionGate", Description).
# --------------------------------------------------------------------------
def test_gate_closed_forms():
    h = 3
    a = np.zeros((2, h))
    d, b = oracle.gate(a, np.zeros(h), -np.ones(h), b=np.zeros((2, h)), want_beta=True)
    np.testing.assert_allclose(d, -math.log(2.0), rtol=0, atol=1e-16)
    assert np.all(b == 0.5)
    # decay_scale multiplies; dt_bias shifts the argument.
    d = oracle.gate(np.full((1, h), -1.5), np.full(h, 1.5), np.array([2.0, -3.0, 0.5]))
    np.testing.assert_allclose(d[0], np.array([2.0, -3.0, 0.5]) * math.log(2.0), rtol=1e-15)
    # softplus(x) - softplus(-x) = x, sigmoid(x) + sigmoid(-x) = 1, and the
    # large-argument asymptotes softplus(x) -> x, softplus(-x) -> e^-x.
    xs = np.linspace(-40, 40, 161).reshape(-1, 1)
    sp_p, sg_p = oracle.gate(xs, np.zeros(1), np.ones(1), b=xs, want_beta=True)
    sp_m, sg_m = oracle.gate(-xs, np.zeros(1), np.ones(1), b=-xs, want_beta=True)
    np.testing.assert_allclose(sp_p - sp_m, xs, rtol=1e-14, atol=1e-13)
    np.testing.assert_allclose(sg_p + sg_m, 1.0, rtol=0, atol=1e-15)
    big = oracle.gate(np.array([[50.0, -50.0]]), np.zeros(2), np.ones(2))
    np.testing.assert_allclose(big[0, 0], 50.0, rtol=1e-15)
    np.testing.assert_allclose(big[0, 1], math.exp(-50.0), rtol=1e-12)
    # Against the library routine on moderate arguments.
    for x in np.linspace(-20, 20, 41):
        d = oracle.gate(np.array([[x]]), np.zeros(1), np.ones(1))
        assert abs(d[0, 0] - math.log1p(math.exp(x))) <= 1e-14 * max(1.0, abs(x))
    # d/dx softplus = sigmoid (central difference).
    eps = 1e-6
    x0 = np.array([[-3.0, -0.2, 0.0, 1.7, 6.0]])
    up = oracle.gate(x0 + eps, np.zeros(5), np.ones(5))
    dn = oracle.gate(x0 - eps, np.zeros(5), np.ones(5))
    _, sg = oracle.gate(x0, np.zeros(5), np.ones(5), b=x0, want_beta=True)
    np.testing.assert_allclose((up - dn) / (2 * eps), sg, rtol=1e-8)


def test_raw_gate_arm_matches_gate_op():
    """The recurrence's raw arm (gatedDeltaUpdate) forms the same decay as the
    LinearAttentionGate op; sigmoid(0) = 1/2 on the beta side."""
    rng = np.random.default_rng(16)
    T, hv, dk, dv = 8, 2, 4, 3
    q, k = rng.standard_normal((T, 1, dk)), rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, hv, dv))
    a = rng.standard_normal((T, hv))
    bias = rng.uniform(-1, 1, hv)
    gscale = -np.exp(rng.uniform(0, 2, hv))
    g = oracle.gate(a, bias, gscale)
    o1, f1, _ = oracle.gdn(q, k, v, rule="gated_delta", decay=a, gate_bias=bias, gate_scale=gscale,
                           beta=np.zeros((T, hv)), beta_sigmoid=True)
    o2, f2, _ = oracle.gdn(q, k, v, rule="gated_delta", decay=g, beta=np.full((T, hv), 0.5))
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(f1, f2, rtol=1e-13, atol=1e-14)


# --------------------------------------------------------------------------
# 6. Linear and gated rules in closed (quadratic) form:
#    o_t = scale (e^{G_t} S_0 q_t + sum_{s<=t} e^{G_t - G_s} (k_s . q_t) v_s)
#    S_T = e^{G_T} S_0 + sum_s e^{G_T - G_s} v_s k_s^T,  G_t = sum_{j<=t} g_j.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("rule", ["linear", "gated"])
def test_linear_and_gated_quadratic_form(rule):
    rng = np.random.default_rng(17)
    T, dk, dv = 11, 5, 4
    q = rng.standard_normal((T, 1, dk))
    k = rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    S0 = rng.standard_normal((1, 1, dv, dk))
    g = -rng.random((T, 1)) if rule == "gated" else np.zeros((T, 1))
    o, fin, _ = oracle.gdn(q, k, v, rule=rule, decay=g if rule == "gated" else None,
                           initial_state=S0, scale=0.9)
    G = np.cumsum(g[:, 0])
    for t in range(T):
        ref = math.exp(G[t]) * S0[0, 0] @ q[t, 0]
        for s in range(t + 1):
            ref = ref + math.exp(G[t] - G[s]) * (k[s, 0] @ q[t, 0]) * v[s, 0]
        np.testing.assert_allclose(o[t, 0], 0.9 * ref, rtol=1e-12, atol=1e-12)
    S = math.exp(G[-1]) * S0[0, 0] + sum(math.exp(G[-1] - G[s]) * np.outer(v[s, 0], k[s, 0])
                                        for s in range(T))
    np.testing.assert_allclose(fin[0, 0], S, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# 7. Delta rules by dense transition matrices: S_T = S_0 P_1..T + sum_s B_s P_{s+1..T}
#    with P_t = alpha_t (I - beta_t k_t k_t^T), B_t = beta_t v_t k_t^T.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("rule", ["delta", "gated_delta"])
def test_delta_transition_products(rule):
    rng = np.random.default_rng(18)
    T, dk, dv = 8, 4, 3
    q = rng.standard_normal((T, 1, dk))
    k = rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    beta = rng.random((T, 1))
    g = -rng.random((T, 1)) if rule == "gated_delta" else np.zeros((T, 1))
    S0 = rng.standard_normal((1, 1, dv, dk))
    o, fin, _ = oracle.gdn(q, k, v, rule=rule, decay=g if rule == "gated_delta" else None,
                           beta=beta, initial_state=S0, scale=1.0)
    P = [math.exp(g[t, 0]) * (np.eye(dk) - beta[t, 0] * np.outer(k[t, 0], k[t, 0])) for t in range(T)]
    Bm = [beta[t, 0] * np.outer(v[t, 0], k[t, 0]) for t in range(T)]

    def prod(lo, hi):
        out = np.eye(dk)
        for t in range(lo, hi):
            out = out @ P[t]
        return out

    for t in range(T):
        St = S0[0, 0] @ prod(0, t + 1) + sum(Bm[s] @ prod(s + 1, t + 1) for s in range(t + 1))
        np.testing.assert_allclose(o[t, 0], St @ q[t, 0], rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(fin[0, 0], St, rtol=1e-11, atol=1e-11)


# --------------------------------------------------------------------------
# 8. Exact rational arithmetic on a 2x2 case: alpha = 1/2 exactly (g = -ln 2
#    through the gate op's closed form), beta = 1/2, unit keys (3/5, 4/5).
# --------------------------------------------------------------------------
def test_exact_rational_two_by_two():
    F = Fraction
    ks = [(F(3, 5), F(4, 5)), (F(0), F(1)), (F(-4, 5), F(3, 5))]
    vs = [(F(1), F(-2)), (F(3), F(1, 2)), (F(-1), F(0))]
    qs = [(F(1), F(0)), (F(2), F(-1)), (F(1, 2), F(1, 2))]
    S = [[F(1), F(0)], [F(0), F(1)]]
    alpha, beta = F(1, 2), F(1, 2)
    exp_o = []
    for kt, vt, qt in zip(ks, vs, qs):
        S = [[alpha * S[i][j] for j in range(2)] for i in range(2)]
        u = [S[i][0] * kt[0] + S[i][1] * kt[1] for i in range(2)]
        d = [beta * (vt[i] - u[i]) for i in range(2)]
        S = [[S[i][j] + d[i] * kt[j] for j in range(2)] for i in range(2)]
        exp_o.append([S[i][0] * qt[0] + S[i][1] * qt[1] for i in range(2)])
    g = math.log(0.5)
    k = np.array([[[float(a), float(b)]] for a, b in ks])
    v = np.array([[[float(a), float(b)]] for a, b in vs])
    q = np.array([[[float(a), float(b)]] for a, b in qs])
    o, fin, _ = oracle.gdn(q, k, v, rule="gated_delta", decay=np.full((3, 1), g),
                           beta=np.full((3, 1), 0.5), initial_state=np.eye(2)[None, None],
                           scale=1.0)
    np.testing.assert_allclose(o[:, 0], np.array(exp_o, dtype=float), rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(fin[0, 0], np.array(S, dtype=float), rtol=1e-15, atol=1e-15)


# --------------------------------------------------------------------------
# 9. Split / resume through the state (final_state -> initial_state).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("rule", ["linear", "gated", "delta", "gated_delta"])
def test_split_resume(rule):
    p = workloads.make(seed=19, B=1, cu_seqlens=[0, 20], hq=1, hv=2, dk=6, dv=5, act="f32",
                       rule=rule, state="random", state_std=0.3)
    o, fin, _ = oracle.run_problem(p)

    def part(t0, t1, init):
        sl = slice(t0, t1)
        return oracle.gdn(p["q"][sl], p["k"][sl], p["v"][sl], rule=rule,
                          decay=None if p["decay"] is None else p["decay"][sl],
                          beta=None if p["beta"] is None else p["beta"][sl],
                          gate_bias=p["gate_bias"], gate_scale=p["gate_scale"],
                          initial_state=init, l2norm_k=True, beta_sigmoid=p["beta_sigmoid"])

    oa, fa, _ = part(0, 7, p["initial_state"])
    ob, fb, _ = part(7, 20, fa)
    np.testing.assert_allclose(np.concatenate([oa, ob]), o, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(fb, fin, rtol=1e-13, atol=1e-14)


# --------------------------------------------------------------------------
# 10. Routing: clamped cu_seqlens, empty requests copy state through, slots.
#     ("com.microsoft.GatedDeltaNet" Inputs/Outputs tables; "gatedDeltaUpdate")
# --------------------------------------------------------------------------
def _small(seed, T, **kw):
    kw.setdefault("rule", "gated_delta")
    return workloads.make(seed=seed, B=kw.pop("B"), T=T, hq=1, hv=2, dk=4, dv=3, act="f32",
                          state="random", state_std=0.5, **kw)


def test_empty_request_copies_state_and_clamps():
    T = 6
    p = _small(20, T, B=4, cu_seqlens=[-5, 3, 3, 100, 1])
    o, fin, err = oracle.run_problem(p)
    S0 = _np(p["initial_state"])
    assert err == 0
    # request 1 = [3,3): empty -> state copied bit-exact; request 3 = [6, 1)
    # after the clamp: decreasing -> empty.
    assert np.array_equal(fin[1], S0[1]) and np.array_equal(fin[3], S0[3])
    # request 0 = [0,3) from the clamped -5; request 2 = [3,6) from the clamped 100.
    ref0 = oracle.gdn(p["q"][:3], p["k"][:3], p["v"][:3], decay=p["decay"][:3],
                      beta=p["beta"][:3], gate_bias=p["gate_bias"], gate_scale=p["gate_scale"],
                      initial_state=S0[0:1], l2norm_k=True, beta_sigmoid=True)
    ref2 = oracle.gdn(p["q"][3:], p["k"][3:], p["v"][3:], decay=p["decay"][3:],
                      beta=p["beta"][3:], gate_bias=p["gate_bias"], gate_scale=p["gate_scale"],
                      initial_state=S0[2:3], l2norm_k=True, beta_sigmoid=True)
    np.testing.assert_array_equal(o[:3], ref0[0])
    np.testing.assert_array_equal(o[3:], ref2[0])
    np.testing.assert_array_equal(fin[0], ref0[1][0])
    np.testing.assert_array_equal(fin[2], ref2[1][0])


def test_seq_lens_rows_equal_separate_requests():
    """Padded rank-4 rows bounded by seq_lens ("gatedDeltaUpdate"): request b
    is exactly the recurrence over the first clamp(seq_lens[b], 0, S) tokens of
    its row, run on its own; padding outputs stay NaN; an empty row copies its
    state through."""
    S, lens = 6, [6, 0, 2, 9, -1]
    p = workloads.make(seed=24, B=5, seq_len=S, seq_lens=lens, hq=1, hv=2, dk=4, dv=3, act="f32",
                       rule="gated_delta", state="random", state_std=0.5)
    o, fin, err = oracle.run_problem(p)
    S0 = _np(p["initial_state"])
    assert err == 0
    for b, n in enumerate(lens):
        n = min(max(n, 0), S)
        lo = b * S
        assert np.isnan(o[lo + n:lo + S]).all()
        if n == 0:
            assert np.array_equal(fin[b], S0[b])
            continue
        ref = oracle.gdn(p["q"][lo:lo + n], p["k"][lo:lo + n], p["v"][lo:lo + n],
                         decay=p["decay"][lo:lo + n], beta=p["beta"][lo:lo + n],
                         gate_bias=p["gate_bias"], gate_scale=p["gate_scale"],
                         initial_state=S0[b:b + 1], l2norm_k=True, beta_sigmoid=True)
        np.testing.assert_array_equal(o[lo:lo + n], ref[0])
        np.testing.assert_array_equal(fin[b], ref[1][0])
    with pytest.raises(ValueError):  # seq_lens bound the uniform layout only
        oracle.gdn(p["q"], p["k"], p["v"], decay=p["decay"], beta=p["beta"], gate_bias=p["gate_bias"],
                   gate_scale=p["gate_scale"], cu_seqlens=np.arange(6, dtype=np.int32) * S, batch=5,
                   seq_lens=np.asarray(lens, dtype=np.int32))


@pytest.mark.parametrize("rule", ["delta", "gated_delta"])
def test_shared_beta_equals_repeated_per_head_beta(rule):
    """beta with last dimension 1 (the LinearAttention schema's broadcast, per
    the GDN-2 issue) is the per-head form with the token's beta repeated over
    the value heads."""
    p = workloads.make(seed=25, B=2, lengths=[5, 4], hq=1, hv=3, dk=4, dv=3, act="f32", rule=rule,
                       state="random", state_std=0.5, beta_shared=True)
    assert tuple(p["beta"].shape) == (9,) and p["beta_shared"]
    o, fin, err = oracle.run_problem(p)
    q = dict(p)
    q["beta"] = p["beta"][:, None].repeat(1, 3)
    q["beta_shared"] = False
    o2, fin2, err2 = oracle.run_problem(q)
    assert err == err2 == 0
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(fin, fin2)
    # and a shared beta is not the same as the first head's beta everywhere else
    q["beta"] = p["beta"][:, None].repeat(1, 3) * torch.tensor([1.0, 0.5, 0.25])
    o3, _, _ = oracle.run_problem(q)
    assert not np.allclose(o[:, 1:], o3[:, 1:])


def test_uncovered_tokens_and_untouched_slots():
    p = _small(21, 8, B=2, cu_seqlens=[1, 4, 6], num_slots=5)
    p["slot_ids"] = np.array([3, 0], dtype=np.int32)
    o, fin, err = oracle.run_problem(p)
    S0 = _np(p["initial_state"])
    assert err == 0
    assert np.isnan(o[0]).all() and np.isnan(o[6:]).all()
    assert not np.isnan(o[1:6]).any()
    for r in (1, 2, 4):
        assert np.array_equal(fin[r], S0[r])
    assert not np.array_equal(fin[3], S0[3]) and not np.array_equal(fin[0], S0[0])


def test_bad_slot_sets_error_and_skips():
    p = _small(22, 6, B=3, cu_seqlens=[0, 2, 4, 6], num_slots=4)
    p["slot_ids"] = np.array([2, 7, -1], dtype=np.int32)
    o, fin, err = oracle.run_problem(p)
    assert err == oracle.ERR_BAD_SLOT
    assert np.isnan(o[2:]).all() and not np.isnan(o[:2]).any()
    S0 = _np(p["initial_state"])
    for r in (0, 1, 3):
        assert np.array_equal(fin[r], S0[r])


def test_slot_routing_equals_gathered_rows():
    p = _small(23, 9, B=3, cu_seqlens=[0, 2, 7, 9], num_slots=6)
    p["slot_ids"] = np.array([5, 1, 2], dtype=np.int32)
    o, fin, _ = oracle.run_problem(p)
    S0 = _np(p["initial_state"])
    q = dict(p)
    q["slot_ids"] = None
    q["initial_state"] = S0[[5, 1, 2]]
    q["num_slots"] = 3
    o2, fin2, _ = oracle.run_problem(q)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(fin[[5, 1, 2]], fin2)


# --------------------------------------------------------------------------
# 11. Grouped heads: value head h reads query/key head h * Hq / Hv.
# --------------------------------------------------------------------------
def test_grouped_heads_match_duplicated_heads():
    p = workloads.make(seed=24, B=2, cu_seqlens=[0, 5, 9], hq=2, hv=6, dk=4, dv=3, act="f32",
                       rule="gated_delta", state="random")
    o, fin, _ = oracle.run_problem(p)
    rep = dict(p)
    idx = [h * 2 // 6 for h in range(6)]
    assert idx == [0, 0, 0, 1, 1, 1]
    rep["q"] = p["q"][:, idx]
    rep["k"] = p["k"][:, idx]
    rep["hq"] = 6
    o2, fin2, _ = oracle.run_problem(rep)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(fin, fin2)


# --------------------------------------------------------------------------
# 12. Attribute semantics ("com.microsoft.GatedDeltaNet", Attributes).
# --------------------------------------------------------------------------
def test_scale_zero_selects_inverse_sqrt_dk():
    p = workloads.make(seed=25, B=1, cu_seqlens=[0, 6], hq=1, hv=1, dk=9, dv=3, act="f32")
    o0, _, _ = oracle.run_problem(p)
    p1 = dict(p, scale=1.0 / 3.0)
    o1, _, _ = oracle.run_problem(p1)
    np.testing.assert_allclose(o0, o1, rtol=1e-15)


def test_l2norm_flag_is_scale_invariant():
    p = workloads.make(seed=26, B=1, cu_seqlens=[0, 6], hq=1, hv=2, dk=5, dv=3, act="f32",
                       l2norm_q=True, l2norm_k=True)
    o0, f0, _ = oracle.run_problem(p)
    p1 = dict(p, q=p["q"] * 4.0, k=p["k"] * 0.25)
    o1, f1, _ = oracle.run_problem(p1)
    # The 1e-12 epsilon under the square root breaks exact invariance at the
    # 1e-12 relative level only.
    np.testing.assert_allclose(o0, o1, rtol=1e-9)
    np.testing.assert_allclose(f0, f1, rtol=1e-9)


def test_rule_degenerations():
    """linear == gated with g = 0; delta == gated_delta with g = 0."""
    base = dict(seed=27, B=1, cu_seqlens=[0, 7], hq=1, hv=2, dk=4, dv=3, act="f32",
                state="random", gate="log")
    for lo, hi in (("linear", "gated"), ("delta", "gated_delta")):
        a = workloads.make(rule=lo, **base)
        b = workloads.make(rule=hi, **base)
        b["decay"] = b["decay"] * 0.0
        b["initial_state"] = a["initial_state"]
        if lo == "delta":
            b["beta"] = a["beta"]
            b["beta_sigmoid"] = a["beta_sigmoid"]
        oa, fa, _ = oracle.run_problem(a)
        ob, fb, _ = oracle.run_problem(b)
        np.testing.assert_allclose(oa, ob, rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(fa, fb, rtol=1e-14, atol=1e-15)


def test_threads_do_not_change_results():
    p = workloads.make(seed=28, B=5, lengths=[3, 0, 4, 1, 2], hq=2, hv=4, dk=6, dv=5, act="f16",
                       state="random")
    o1, f1, _ = oracle.run_problem(p, threads=1)
    o4, f4, _ = oracle.run_problem(p, threads=4)
    np.testing.assert_array_equal(o1, o4)
    np.testing.assert_array_equal(f1, f4)


# --------------------------------------------------------------------------
# Per-key raw-gate arm ("gatedDeltaUpdate": gate_bias [HV, K] beside a
# [B, T, HV, K] gate, gate_scale [HV]): each key channel c of head h takes
# g = gate_scale[h] * softplus(raw + gate_bias[h, c]).  The log decays are
# formed here with the Python math library and fed to the oracle directly.
# A bias taken per head, per channel only, or a scale taken per channel fails.
# --------------------------------------------------------------------------
def test_per_key_raw_gate_arm():
    rng = np.random.default_rng(31)
    T, hv, dk, dv = 7, 2, 5, 3
    q = rng.standard_normal((T, 1, dk))
    k = _unit(rng.standard_normal((T, 1, dk)))
    v = rng.standard_normal((T, hv, dv))
    raw = rng.standard_normal((T, hv, dk)) * 2.0
    bias = rng.uniform(-2.0, 2.0, (hv, dk))
    gscale = -np.exp(rng.uniform(0.0, 2.0, hv))
    beta = rng.random((T, hv))
    S0 = rng.standard_normal((1, hv, dv, dk)) * 0.3
    g = np.empty((T, hv, dk))
    for t in range(T):
        for h in range(hv):
            for c in range(dk):
                g[t, h, c] = gscale[h] * math.log1p(math.exp(raw[t, h, c] + bias[h, c]))
    o1, f1, _ = oracle.gdn(q, k, v, rule="gated_delta", decay=raw, gate_bias=bias, gate_scale=gscale,
                           beta=beta, initial_state=S0, decay_per_key=True)
    o2, f2, _ = oracle.gdn(q, k, v, rule="gated_delta", decay=g, beta=beta, initial_state=S0,
                           decay_per_key=True)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(f1, f2, rtol=1e-13, atol=1e-14)


# --------------------------------------------------------------------------
# The GDN-2 erase gate through beta_activation: with BETA_SIGMOID the
# per-key beta logits x give b = 1 / (1 + e^-x) (GDN-2 issue: b_t in
# [0, 1]^{d_k}); b is formed here with the Python math library.
# --------------------------------------------------------------------------
def test_gdn2_erase_gate_sigmoid():
    rng = np.random.default_rng(32)
    T, hv, dk, dv = 6, 2, 4, 3
    q = rng.standard_normal((T, 1, dk))
    k = _unit(rng.standard_normal((T, 1, dk)))
    v = rng.standard_normal((T, hv, dv))
    x = rng.standard_normal((T, hv, dk)) * 3.0
    b = np.vectorize(lambda z: 1.0 / (1.0 + math.exp(-z)))(x)
    g = -rng.random((T, hv, dk))
    S0 = rng.standard_normal((1, hv, dv, dk)) * 0.3
    o1, f1, _ = oracle.gdn(q, k, v, rule="gdn2", decay=g, beta=x, beta_sigmoid=True, initial_state=S0,
                           decay_per_key=True)
    o2, f2, _ = oracle.gdn(q, k, v, rule="gdn2", decay=g, beta=b, initial_state=S0, decay_per_key=True)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(f1, f2, rtol=1e-13, atol=1e-14)


# --------------------------------------------------------------------------
# Key-major state ("gatedDeltaUpdate": the [B, HV, K, V] state decays by
# exp(g), takes the rank-1 update (beta k) (x) (v - S^T k) and emits
# o = (scale q)^T S).  That loop is written here in its own key-major form
# with numpy; the oracle run with key-major states must match it, and must
# equal the transpose of its value-major run exactly.
# --------------------------------------------------------------------------
def test_key_major_state_follows_the_clika_form():
    rng = np.random.default_rng(33)
    T, hq, hv, dk, dv, rows = 8, 1, 2, 5, 3, 4
    q = rng.standard_normal((T, hq, dk))
    k = _unit(rng.standard_normal((T, hq, dk)))
    v = rng.standard_normal((T, hv, dv))
    g = -rng.random((T, hv))
    beta = rng.random((T, hv))
    SK = rng.standard_normal((rows, hv, dk, dv)) * 0.3      # key-major slab
    cu = [0, 5, 8]
    slots = np.array([3, 1], dtype=np.int32)
    o, fin, err = oracle.gdn(q, k, v, rule="gated_delta", decay=g, beta=beta, initial_state=SK,
                             cu_seqlens=cu, slot_ids=slots, scale=0.6, state_kmajor=True)
    assert err == 0 and fin.shape == SK.shape
    want = SK.copy()
    for b in range(2):
        for h in range(hv):
            S = SK[slots[b], h].copy()                      # dk x dv
            for t in range(cu[b], cu[b + 1]):
                kt, qt = k[t, 0], q[t, 0]
                S = math.exp(g[t, h]) * S
                S = S + np.outer(beta[t, h] * kt, v[t, h] - S.T @ kt)
                np.testing.assert_allclose(o[t, h], (0.6 * qt) @ S, rtol=1e-12, atol=1e-12)
            want[slots[b], h] = S
    np.testing.assert_allclose(fin, want, rtol=1e-12, atol=1e-12)
    # the same run with value-major states gives the transposed states bit for bit
    o_v, fin_v, _ = oracle.gdn(q, k, v, rule="gated_delta", decay=g, beta=beta,
                               initial_state=np.ascontiguousarray(SK.transpose(0, 1, 3, 2)),
                               cu_seqlens=cu, slot_ids=slots, scale=0.6)
    assert np.array_equal(o_v, o)
    assert np.array_equal(fin_v.transpose(0, 1, 3, 2), fin)


# --------------------------------------------------------------------------
# GDN-2 proposal (B): the erase gate is an input of its own beside the scalar
# beta.  (1) b = beta * 1 gives gated_delta back ("old beta_t = b_t * 1 is the
# strict-generalization fallback").  (2) Against the issue's first display
# with the write term carrying beta and the write gate,
#   S_K = (I - k (b .* k)^T) D S_K + beta k (w .* v)^T,  written densely here.
# --------------------------------------------------------------------------
def test_gdn2_erase_gate_input_with_b_equal_beta_is_gated_delta():
    rng = np.random.default_rng(34)
    T, hv, dk, dv = 9, 2, 6, 4
    q = rng.standard_normal((T, 1, dk))
    k = _unit(rng.standard_normal((T, 1, dk)))
    v = rng.standard_normal((T, hv, dv))
    g = -rng.random((T, hv))
    x = rng.standard_normal((T, hv))
    beta = 1.0 / (1.0 + np.exp(-x))
    S0 = rng.standard_normal((1, hv, dv, dk)) * 0.3
    o1, f1, _ = oracle.gdn(q, k, v, rule="gated_delta", decay=g, beta=x, beta_sigmoid=True, initial_state=S0)
    b = np.repeat(beta[:, :, None], dk, axis=2)
    o2, f2, _ = oracle.gdn(q, k, v, rule="gdn2", decay=g, beta=x, beta_sigmoid=True, erase_gate=b,
                           initial_state=S0)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(f2, f1, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("shared", [False, True])
def test_gdn2_erase_gate_input_dense_form(shared):
    rng = np.random.default_rng(35)
    T, hv, dk, dv = 7, 2, 4, 3
    q = rng.standard_normal((T, 1, dk))
    k = rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, hv, dv))
    b = rng.random((T, hv, dk))
    w = rng.random((T, hv, dv))
    beta = rng.random((T,) if shared else (T, hv))
    g = -rng.random((T, hv, dk))
    S0 = rng.standard_normal((1, hv, dv, dk))
    o, fin, _ = oracle.gdn(q, k, v, rule="gdn2", decay=g, beta=beta, erase_gate=b, write_gate=w,
                           initial_state=S0, decay_per_key=True, scale=1.0, beta_shared=shared)
    for h in range(hv):
        SK = S0[0, h].T.copy()
        for t in range(T):
            bt = beta[t] if shared else beta[t, h]
            kt = k[t, 0][:, None]
            bk = (b[t, h] * k[t, 0])[:, None]
            SK = (np.eye(dk) - kt @ bk.T) @ np.diag(np.exp(g[t, h])) @ SK + bt * kt @ (w[t, h] * v[t, h])[None, :]
            np.testing.assert_allclose(o[t, h], SK.T @ q[t, 0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(fin[0, h], SK.T, rtol=1e-12, atol=1e-12)


def test_gdn2_write_gate_input_equals_folded():
    """Proposal (A) keeps the write gate outside the op (v <- w .* v by the
    caller); passed to the op it must give the same result, and proposal (B)
    with beta = 1 must equal proposal (A)."""
    rng = np.random.default_rng(36)
    T, hv, dk, dv = 8, 2, 5, 4
    q = rng.standard_normal((T, 1, dk))
    k = _unit(rng.standard_normal((T, 1, dk)))
    v = rng.standard_normal((T, hv, dv))
    w = rng.random((T, hv, dv))
    b = rng.random((T, hv, dk))
    g = -rng.random((T, hv, dk))
    S0 = rng.standard_normal((1, hv, dv, dk)) * 0.3
    o1, f1, _ = oracle.gdn(q, k, v * w, rule="gdn2", decay=g, beta=b, initial_state=S0, decay_per_key=True)
    o2, f2, _ = oracle.gdn(q, k, v, rule="gdn2", decay=g, beta=b, write_gate=w, initial_state=S0,
                           decay_per_key=True)
    np.testing.assert_allclose(o2, o1, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(f2, f1, rtol=1e-14, atol=1e-15)
    o3, f3, _ = oracle.gdn(q, k, v, rule="gdn2", decay=g, beta=np.ones((T, hv)), erase_gate=b, write_gate=w,
                           initial_state=S0, decay_per_key=True)
    np.testing.assert_allclose(o3, o1, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(f3, f1, rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("rule", ["linear", "gated_delta", "gdn2"])
def test_float_instantiation_tracks_the_double_build(rule):
    """The float instantiation of the oracle source (timed as a CPU baseline,
    never used for parity) computes the same recurrence: within fp32 rounding
    of the double build on a small random problem."""
    kw = dict(seed=7, B=3, lengths=[9, 0, 17], hq=2, hv=4, dk=16, dv=8, act="f32", rule=rule,
              state="random", state_std=0.3)
    if rule == "gdn2":
        kw.update(decay_per_key=True, gate_dtype="f32")
    p = workloads.make(**kw)
    o64, f64, e64 = oracle.run_problem(p)
    o32, f32, e32 = oracle.run_problem(p, real="f32")
    assert e64 == e32 == 0
    m = ~np.isnan(o64)
    assert np.array_equal(m, ~np.isnan(o32))
    assert np.abs(o32[m] - o64[m]).max() <= 1e-5 * np.abs(o64[m]).max()
    assert np.abs(f32 - f64).max() <= 1e-5 * np.abs(f64).max()

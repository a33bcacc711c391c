"""Checks, in float64 on the CPU, the chunk-parallel reformulation that the
CUDA chunked-prefill kernel implements, against the token-serial oracle.

The pages say only that a chunk-parallel prefill exists, that its per-chunk
system needs unit keys, and that the chunk size never changes the result
("com.microsoft.GatedDeltaNet": key input, chunk_size attribute).  The
per-chunk algebra used by the kernel is derived from the recurrence itself:
for a chunk with incoming state M0 and in-chunk log-decay cumulants G,

    A_rj = beta_r exp(G_r - G_j) (kappa_r . k_j)         (j < r)
    T    = (I + A)^-1                                   (unit lower triangular)
    U'   = T diag(beta) V,   W = T diag(beta e^G) Kappa
    Delta = U' - W M0^T
    O    = scale (diag(e^G) Q M0^T + P Delta),  P_rj = exp(G_r - G_j) (q_r . k_j), j <= r
    M_C  = e^{G_C} M0 + Delta^T diag(e^{G_C - G}) K

(kappa = k for the v1 rules, b .* k with beta = 1 for GDN-2; rules without
retrieval use Delta = V).  The same file checks the per-key-decay form of the
chunk step (block factorisation about reference tokens, running products on
the diagonal blocks, the affine chunk map the chain kernel applies) and the
decode kernel's token step with a lazy scalar decay factor.  These tests are
the derivations' checks: they are not the oracle and the oracle does not use
them.
"""
import numpy as np
import pytest

import oracle
import workloads


def _chunked(q, k, v, g, beta, kappa, M0, scale, C, retrieval):
    T, dk = k.shape
    M = M0.copy()
    out = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, C):
        sl = slice(c0, min(T, c0 + C))
        Q, K, V, X = q[sl], k[sl], v[sl], kappa[sl]
        G = np.cumsum(g[sl])
        bt = beta[sl]
        n = len(G)
        D = np.exp(G[:, None] - G[None, :])
        if retrieval:
            A = np.tril(bt[:, None] * D * (X @ K.T), -1)
            Tm = np.linalg.inv(np.eye(n) + A)
            U = Tm @ (bt[:, None] * V)
            W = Tm @ ((bt * np.exp(G))[:, None] * X)
            Delta = U - W @ M.T
        else:
            Delta = V
        P = np.tril(D * (Q @ K.T))
        out[sl] = scale * (np.exp(G)[:, None] * (Q @ M.T) + P @ Delta)
        M = np.exp(G[-1]) * M + Delta.T @ (np.exp(G[-1] - G)[:, None] * K)
    return out, M


@pytest.mark.parametrize("rule", ["linear", "gated", "delta", "gated_delta", "gdn2"])
@pytest.mark.parametrize("C", [1, 4, 16, 64])
def test_chunk_form_equals_token_loop(rule, C):
    T, dk, dv = 50, 8, 6
    p = workloads.make(seed=61, B=1, cu_seqlens=[0, T], hq=1, hv=1, dk=dk, dv=dv, act="f32",
                       rule=rule, gate="log", logdecay_range=(-3.0, 0.0), beta_mode="direct",
                       state="random", state_std=0.3, l2norm_k=False)
    k = p["k"].double().numpy()[:, 0]
    k = k / np.linalg.norm(k, axis=1, keepdims=True)
    p["k"] = p["k"].double().new_tensor(k[:, None, :]).float()
    k = p["k"].double().numpy()[:, 0]
    q = p["q"].double().numpy()[:, 0]
    v = p["v"].double().numpy()[:, 0]
    g = p["decay"].double().numpy()[:, 0] if p["decay"] is not None else np.zeros(T)
    if rule == "gdn2":
        b = p["beta"].double().numpy()[:, 0]
        kappa, beta = b * k, np.ones(T)
    elif p["beta"] is not None:
        kappa, beta = k, p["beta"].double().numpy()[:, 0]
    else:
        kappa, beta = k, np.ones(T)
    M0 = p["initial_state"].double().numpy()[0, 0]
    ref_o, ref_f, _ = oracle.run_problem(p)
    o, M = _chunked(q, k, v, g, beta, kappa, M0, 1 / np.sqrt(dk), C,
                    rule in ("delta", "gated_delta", "gdn2"))
    np.testing.assert_allclose(o, ref_o[:, 0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(M, ref_f[0, 0], rtol=1e-10, atol=1e-12)


def _chunked_perkey(q, k, v, g, beta, kappa, M0, scale, C, blk=16, retrieval=True):
    """The per-key-decay chunk step in the form the tensor-core prepare pass and
    the chain kernel compute it.  g is [T, dk] (one log decay per key channel),
    Gamma its in-chunk cumulants.  A and P: entries whose column lies in an
    earlier block of `blk` tokens are products of two scaled operands about the
    reference token rho = (first token of the row's block) - 1, both factors at
    most 1; entries inside a block come from a running product of per-token
    decays.  Then the affine chunk map
        S <- S + U^T Kt + S E,   O^T = U^T P^T + S Q'^T,
        E = Diag(e^{Gamma_C}) - I + Wn^T Kt,   Q' = Qh + P Wn,   Wn = -W.
    Without retrieval (the gated rule) there is no system: U = V and Wn = 0."""
    T, dk = k.shape
    S = M0.copy()
    out = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, C):
        sl = slice(c0, min(T, c0 + C))
        Q, K, V, X, bt = q[sl], k[sl], v[sl], kappa[sl], beta[sl]
        G = np.cumsum(g[sl], axis=0)  # [n, dk]
        alpha = np.exp(g[sl])
        n = len(G)
        A = np.zeros((n, n))
        P = np.zeros((n, n))
        for r in range(n):
            s = r // blk
            if s > 0:
                rho = blk * s - 1
                xr = X[r] * np.exp(G[r] - G[rho])
                qr = Q[r] * np.exp(G[r] - G[rho])
                for j in range(blk * s):
                    yj = K[j] * np.exp(G[rho] - G[j])
                    A[r, j] = bt[r] * xr @ yj
                    P[r, j] = qr @ yj
            e = np.ones(dk)
            for j in range(r, blk * s - 1, -1):  # down from the diagonal inside the block
                if j < r:
                    A[r, j] = bt[r] * np.sum(X[r] * K[j] * e)
                P[r, j] = np.sum(Q[r] * K[j] * e)
                e = e * alpha[j]
        if retrieval:
            Tm = np.linalg.inv(np.eye(n) + A)
            U = Tm @ (bt[:, None] * V)
            Wn = -Tm @ (bt[:, None] * (np.exp(G) * X))
        else:
            U, Wn = V, np.zeros((n, dk))
        Kt = np.exp(G[-1] - G) * K
        Qh = scale * np.exp(G) * Q
        E = np.diag(np.exp(G[-1])) - np.eye(dk) + Wn.T @ Kt
        Qp = Qh + scale * P @ Wn
        out[sl] = (U.T @ (scale * P).T + S @ Qp.T).T
        S = S + U.T @ Kt + S @ E
    return out, S


@pytest.mark.parametrize("rule", ["gated_delta", "gdn2", "gated"])
@pytest.mark.parametrize("C", [16, 64])
@pytest.mark.parametrize("lo", [-1.0, -6.0])
def test_per_key_chunk_form_equals_token_loop(rule, C, lo):
    """Per-key decay (GDN-2 issue; "gatedDeltaUpdate" per-key gate): the block
    factorisation and the affine chunk map equal the token loop, including
    strong decays whose in-chunk cumulants reach -380."""
    T, dk, dv = 150, 8, 6
    p = workloads.make(seed=62, B=1, cu_seqlens=[0, T], hq=1, hv=1, dk=dk, dv=dv, act="f32",
                       rule=rule, gate="log", logdecay_range=(lo, 0.0), decay_per_key=True,
                       beta_mode="direct", state="random", state_std=0.3, l2norm_k=False)
    k = p["k"].double().numpy()[:, 0]
    k = k / np.linalg.norm(k, axis=1, keepdims=True)
    p["k"] = p["k"].double().new_tensor(k[:, None, :]).float()
    k = p["k"].double().numpy()[:, 0]
    q = p["q"].double().numpy()[:, 0]
    v = p["v"].double().numpy()[:, 0]
    g = p["decay"].double().numpy()[:, 0]  # [T, dk]
    if rule == "gdn2":
        kappa, beta = p["beta"].double().numpy()[:, 0] * k, np.ones(T)
    elif rule == "gated":
        kappa, beta = k, np.zeros(T)
    else:
        kappa, beta = k, p["beta"].double().numpy()[:, 0]
    M0 = p["initial_state"].double().numpy()[0, 0]
    ref_o, ref_f, _ = oracle.run_problem(p)
    o, M = _chunked_perkey(q, k, v, g, beta, kappa, M0, 1 / np.sqrt(dk), C, retrieval=rule != "gated")
    np.testing.assert_allclose(o, ref_o[:, 0], rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(M, ref_f[0, 0], rtol=1e-9, atol=1e-11)


def _lazy_decay_loop(q, k, v, g, beta, kappa, M0, scale, retrieval, floor=1e-20):
    """The token step of the decode kernel with a scalar decay kept as a lazy
    factor, S = c * S~, so that each token touches the state once:
        c' = c alpha,  u = c' (S~ kappa),  d = beta (v - u)  (v without retrieval),
        o = scale (c' (S~ q) + d (k . q)),  S~ += (d / c') k^T,
    with c' folded into S~ before it underflows (c' < floor)."""
    S = M0.copy()
    c = 1.0
    out = np.zeros((len(k), v.shape[1]))
    for t in range(len(k)):
        cn = c * np.exp(g[t])
        u = cn * (S @ kappa[t])
        d = beta[t] * (v[t] - u) if retrieval else v[t]
        out[t] = scale * (cn * (S @ q[t]) + d * (k[t] @ q[t]))
        if cn < floor:
            S *= cn
            cn = 1.0
        S += np.outer(d / cn, k[t])
        c = cn
    return out, c * S


@pytest.mark.parametrize("rule", ["gated", "gated_delta", "gdn2"])
@pytest.mark.parametrize("lo", [-1.0, -30.0])
def test_lazy_decay_form_equals_token_loop(rule, lo):
    """The lazy-factor decode step equals the token loop, also when the decay
    is strong enough (log decays down to -30 per token) that the factor is
    folded back into the state several times."""
    T, dk, dv = 40, 8, 6
    p = workloads.make(seed=63, B=1, cu_seqlens=[0, T], hq=1, hv=1, dk=dk, dv=dv, act="f32",
                       rule=rule, gate="log", logdecay_range=(lo, 0.0), beta_mode="direct",
                       state="random", state_std=0.3, l2norm_k=False)
    k = p["k"].double().numpy()[:, 0]
    k = k / np.linalg.norm(k, axis=1, keepdims=True)
    p["k"] = p["k"].double().new_tensor(k[:, None, :]).float()
    k = p["k"].double().numpy()[:, 0]
    q = p["q"].double().numpy()[:, 0]
    v = p["v"].double().numpy()[:, 0]
    g = p["decay"].double().numpy()[:, 0]
    if rule == "gdn2":
        kappa, beta = p["beta"].double().numpy()[:, 0] * k, np.ones(T)
    elif rule == "gated_delta":
        kappa, beta = k, p["beta"].double().numpy()[:, 0]
    else:
        kappa, beta = k, np.ones(T)
    M0 = p["initial_state"].double().numpy()[0, 0]
    ref_o, ref_f, _ = oracle.run_problem(p)
    o, M = _lazy_decay_loop(q, k, v, g, beta, kappa, M0, 1 / np.sqrt(dk), rule != "gated")
    np.testing.assert_allclose(o, ref_o[:, 0], rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(M, ref_f[0, 0], rtol=1e-9, atol=1e-12)

"""Seeded synthetic inputs for the gated delta rule workloads.

This module only draws random numbers (torch CPU generators, so every machine
sees the same bits) and lays them out; it holds none of the recurrence's
arithmetic.  Both the CUDA parity tests and the CPU oracle take their inputs
from here.  Gate and beta activations are NOT applied here: the raw gate
projection, the raw beta logits and un-normalised keys are passed with the
flags that make the method itself apply softplus/sigmoid/L2-norm.

A problem is a plain dict:
    q, k            [T, Hq, dk] act dtype (rank-4 inputs are [B, S, Hq, dk])
    v               [T, Hv, dv] act dtype
    decay           raw gate projection or log-space decay, [T, Hv] or [T, Hv, dk]
    gate_bias       [Hv] or [Hv, dk] fp32, or None (log-space decay given)
    gate_scale      [Hv] fp32, the once-folded -exp(A_log), or None
    beta            [T, Hv] (or [T, Hv, dk] erase gate for gdn2), or None
    erase_gate      gdn2 with the erase gate as its own input: [T, Hv, dk] fp32
                    (beta is then the scalar [T, Hv] write rate), or None
    write_gate      gdn2 write gate passed to the op: [T, Hv, dv] fp32, or None
                    (folded into v by the caller, or absent)
    state_kmajor    states are [rows, Hv, dk, dv] instead of [rows, Hv, dv, dk]
    cu_seqlens      [B+1] int32 or None
    slot_ids        [B] int32 or None
    initial_state   [rows, Hv, dv, dk] fp32 or None (zeros)
    batch, seq_len (0 = packed rank-3), rule, scale, flags, act_dtype ('f16'/'f32')
"""
import torch

ACT = {"f16": torch.float16, "f32": torch.float32}


def _gen(seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def ragged_lengths(n, total, max_len, gen):
    """Integer lengths ~U[1, max_len], rescaled to sum to ``total``; the
    rounding residual goes to the longest request; every length is >= 1."""
    raw = torch.randint(1, max_len + 1, (n,), generator=gen).double()
    scaled = torch.clamp(torch.round(raw * total / raw.sum()), min=1).long()
    resid = total - int(scaled.sum())
    scaled[int(torch.argmax(scaled))] += resid
    assert int(scaled.sum()) == total and int(scaled.min()) >= 1
    return scaled


def cu_from_lengths(lengths):
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.as_tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    return cu


def make(*, seed, B, T=None, seq_len=0, lengths=None, cu_seqlens=None, hq, hv, dk, dv,
         act="f16", rule="gated_delta", gate="raw", decay_per_key=False,
         a_log_range=(0.0, 2.0), dt_bias_range=(-2.0, 2.0), gate_dtype=None,
         beta_dtype=None, logdecay_range=(-1.0, 0.0), beta_mode="sigmoid",
         state="zero", state_std=0.02, num_slots=None, slot_mode=None,
         write_gate=False, l2norm_q=False, l2norm_k=True, scale=0.0, qk_std=1.0, seq_lens=None,
         beta_shared=False, erase="beta", state_kmajor=False):
    """Draws one problem.  ``gate`` is 'raw' (raw projection + gate_bias +
    gate_scale), 'log' (log-space decay drawn U(logdecay_range)) or ignored
    for rules without decay.  ``beta_mode`` is 'sigmoid' (raw N(0,1) logits +
    BETA_SIGMOID flag) or 'direct' (beta drawn U(0,1), used as given).
    GDN-2 only: ``erase`` is 'beta' (the erase gate is the per-key beta) or
    'input' (a scalar beta as for gated_delta, and the erase gate
    sigmoid(N(0,1)) as its own input); ``write_gate`` is False, True / 'fold'
    (w = sigmoid(N(0,1)) multiplied into v here) or 'input' (w kept apart).
    ``state_kmajor`` draws the state key-major, [rows, Hv, dk, dv]."""
    gen = _gen(seed)
    dt = ACT[act]
    if seq_len:
        T = B * seq_len
    elif cu_seqlens is not None:
        cu_seqlens = torch.as_tensor(cu_seqlens, dtype=torch.int32)
        if T is None:
            T = int(cu_seqlens[-1])
    elif lengths is not None:
        cu_seqlens = cu_from_lengths(lengths)
        T = int(cu_seqlens[-1])
    assert T is not None
    p = {"batch": B, "seq_len": seq_len, "rule": rule, "scale": scale, "act_dtype": act,
         "hq": hq, "hv": hv, "dk": dk, "dv": dv, "total_tokens": T,
         "l2norm_q": l2norm_q, "l2norm_k": l2norm_k, "beta_sigmoid": False,
         "decay_per_key": False}
    p["q"] = (torch.randn(T, hq, dk, generator=gen) * qk_std).to(dt)
    p["k"] = (torch.randn(T, hq, dk, generator=gen) * qk_std).to(dt)
    v = torch.randn(T, hv, dv, generator=gen)
    p["write_gate"] = p["erase_gate"] = None
    p["state_kmajor"] = bool(state_kmajor)
    if write_gate:
        # GDN-2 write gate w ~ sigmoid(N(0,1)) on the value axis: folded into v
        # by the caller (a graph-level Mul, outside the op), or passed to the op
        w = torch.sigmoid(torch.randn(T, hv, dv, generator=gen))
        if write_gate == "input":
            p["write_gate"] = w.float()
        else:
            v = v * w
    p["v"] = v.to(dt)
    has_decay = rule in ("gated", "gated_delta", "gdn2")
    has_beta = rule in ("delta", "gated_delta", "gdn2")
    p["decay"] = p["gate_bias"] = p["gate_scale"] = p["beta"] = None
    if has_decay:
        shape = (T, hv, dk) if decay_per_key else (T, hv)
        pshape = (hv, dk) if decay_per_key else (hv,)
        p["decay_per_key"] = decay_per_key
        if gate == "raw":
            gd = ACT[gate_dtype] if gate_dtype else dt
            p["decay"] = torch.randn(*shape, generator=gen).to(gd)
            lo, hi = a_log_range
            a_log = lo + (hi - lo) * torch.rand(hv, generator=gen)
            p["gate_scale"] = (-torch.exp(a_log)).float()
            lo, hi = dt_bias_range
            p["gate_bias"] = (lo + (hi - lo) * torch.rand(*pshape, generator=gen)).float()
        elif gate == "log":
            lo, hi = logdecay_range
            p["decay"] = (lo + (hi - lo) * torch.rand(*shape, generator=gen)).float()
        else:
            raise ValueError(gate)
    if has_beta:
        per_key_beta = rule == "gdn2" and erase == "beta"
        bshape = (T, hv, dk) if per_key_beta else ((T,) if beta_shared else (T, hv))
        p["beta_shared"] = bool(beta_shared) and not per_key_beta
        bd = ACT[beta_dtype] if beta_dtype else torch.float32
        if beta_mode == "sigmoid":
            p["beta"] = torch.randn(*bshape, generator=gen).to(bd)
            p["beta_sigmoid"] = True
        else:
            p["beta"] = torch.rand(*bshape, generator=gen).to(bd)
        if rule == "gdn2" and erase == "input":
            p["erase_gate"] = torch.sigmoid(torch.randn(T, hv, dk, generator=gen)).float()
    p["cu_seqlens"] = cu_seqlens
    # padded-ragged rank-4 batch: request b uses the first seq_lens[b] tokens of its row
    p["seq_lens"] = torch.as_tensor(seq_lens, dtype=torch.int32) if seq_lens is not None else None
    rows = num_slots if num_slots else B
    p["num_slots"] = rows
    if slot_mode == "perm":
        p["slot_ids"] = torch.randperm(rows, generator=gen)[:B].to(torch.int32)
    else:
        p["slot_ids"] = None
    if state == "random":
        sshape = (rows, hv, dk, dv) if state_kmajor else (rows, hv, dv, dk)
        p["initial_state"] = torch.randn(*sshape, generator=gen) * state_std
    else:
        p["initial_state"] = None
    return p


# ---- the workloads the benchmark and the full-size tests run ------------------

def tiny_gated_delta(seed=1):
    """B=1, T=64, Hq=Hv=2, dk=dv=16, fp32; raw gate with A_log, dt_bias ~ U(-1,1);
    beta = sigmoid(N(0,1)); unit keys; zero state; scale = dk^-1/2."""
    return make(seed=seed, B=1, cu_seqlens=[0, 64], hq=2, hv=2, dk=16, dv=16, act="f32",
                rule="gated_delta", gate="raw", a_log_range=(-1.0, 1.0),
                dt_bias_range=(-1.0, 1.0), gate_dtype="f32")


def decode(L, seed=2, B=256, hq=16, hv=32, dk=128, dv=128, num_slots=1024):
    """256 requests of L tokens each (cu_seqlens = L * arange), fp16 q/k/v, an
    fp32 slab [1024, Hv, dv, dk] ~ N(0, 0.02) updated in place at distinct
    permuted slot ids; raw gate a, b ~ N(0,1) fp16, A_log ~ U(0,2),
    dt_bias ~ U(-2,2)."""
    cu = torch.arange(B + 1, dtype=torch.int32) * L
    return make(seed=seed, B=B, cu_seqlens=cu, hq=hq, hv=hv, dk=dk, dv=dv, act="f16",
                rule="gated_delta", gate="raw", beta_dtype="f16", state="random",
                num_slots=num_slots, slot_mode="perm")


def ragged_prefill(seed=3, n=8, total=16384, max_len=4096, hq=16, hv=32, dk=128, dv=128):
    """8 requests, lengths ~U[1,4096] rescaled to 16384 tokens, packed rank-3;
    g = -exp(U(0,2)) * softplus(N(0,1)) through the raw arm (dt_bias = 0);
    beta = sigmoid(N(0,1)); state ~ N(0, 0.02); final state returned."""
    gen = _gen(seed + 1000)
    lengths = ragged_lengths(n, total, max_len, gen)
    return make(seed=seed, B=n, lengths=lengths, hq=hq, hv=hv, dk=dk, dv=dv, act="f16",
                rule="gated_delta", gate="raw", gate_dtype="f32", dt_bias_range=(0.0, 0.0),
                state="random")


def long_prefill(rule, seed=4, B=4, S=8192, h=16, dk=128, dv=128):
    """B=4, S=8192, Hq=Hv=16, rank-4, fp16, config-2 distributions, zero state."""
    return make(seed=seed, B=B, seq_len=S, hq=h, hv=h, dk=dk, dv=dv, act="f16", rule=rule,
                gate="raw", beta_dtype="f16")


def gated_perkey(seed=6, B=2, S=4096, h=16, dk=128, dv=128, state="zero"):
    """The gated rule (no retrieval) with decay per key channel, GLA-style:
    the GDN-2 workload's per-key log decay -softplus(N(0,1)) (raw arm,
    gate_scale = -1, gate_bias = 0), B = 2, S = 4096, H = 16, fp16, fp32 gates."""
    return make(seed=seed, B=B, seq_len=S, hq=h, hv=h, dk=dk, dv=dv, act="f16", rule="gated", gate="raw",
                decay_per_key=True, gate_dtype="f32", a_log_range=(0.0, 0.0), dt_bias_range=(0.0, 0.0),
                state=state, state_std=0.02)


def gdn2(seed=5, B=2, S=4096, h=16, dk=128, dv=128, erase="beta", write_gate="fold"):
    """GDN-2: per-key log decay -softplus(N(0,1)) (raw arm, gate_scale = -1,
    gate_bias = 0), erase gate sigmoid(N(0,1)) per key channel, write gate
    sigmoid(N(0,1)) folded into v, unit keys, zero state.  ``erase='input'``
    passes the erase gate as its own input beside a scalar beta =
    sigmoid(N(0,1)); ``write_gate='input'`` passes w to the op."""
    return make(seed=seed, B=B, seq_len=S, hq=h, hv=h, dk=dk, dv=dv, act="f16", rule="gdn2",
                gate="raw", decay_per_key=True, gate_dtype="f32", a_log_range=(0.0, 0.0),
                dt_bias_range=(0.0, 0.0), write_gate=write_gate, erase=erase)


def token_ranges(p):
    """Per-request [t0, t1) after the cu_seqlens clamp (or the seq_lens bound
    of the padded rank-4 layout), as python ints (host bookkeeping for samplers
    and sentinel checks)."""
    T, B = p["total_tokens"], p["batch"]
    out = []
    cu = p.get("cu_seqlens")
    for b in range(B):
        if cu is not None:
            t0 = min(max(int(cu[b]), 0), T)
            t1 = min(max(int(cu[b + 1]), 0), T)
            t1 = max(t1, t0)
        else:
            L = T // B
            t0, t1 = b * L, (b + 1) * L
            if p.get("seq_lens") is not None:
                t1 = t0 + min(max(int(p["seq_lens"][b]), 0), L)
        out.append((t0, t1))
    return out

"""CPU oracle for the gated delta rule (TEST INFRASTRUCTURE ONLY).

The plain token-serial double-precision definition of the recurrence lives in
``gdn_oracle.c``; this module loads it through ctypes and converts arrays.
Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import it.  It shares no code with the CUDA library and the library never
calls it.

Inputs may be numpy arrays or CPU torch tensors of any float dtype; they are
converted exactly to float64 (fp16 and fp32 embed exactly).  Outputs come back
as float64 numpy arrays, unrounded; ``round_to`` rounds once (round to
nearest even) to an activation dtype.  ``real="f32"`` runs the float
instantiation of the same source instead (inputs rounded to float32): only the
benchmark's CPU-baseline leg uses it, to time it; every parity check uses the
double build.
"""
import ctypes
import os

import numpy as np

from . import build as _build

RULES = {"linear": 0, "gated": 1, "delta": 2, "gated_delta": 3, "gdn2": 4}
ERR_BAD_SLOT = 1

_dp = ctypes.POINTER(ctypes.c_double)
_fp = ctypes.POINTER(ctypes.c_float)
_ip = ctypes.POINTER(ctypes.c_int32)


def _problem_fields(creal, rp):
    return [
        ("batch", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
        ("hq", ctypes.c_int32), ("hv", ctypes.c_int32),
        ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
        ("rule", ctypes.c_int32),
        ("l2norm_q", ctypes.c_int32), ("l2norm_k", ctypes.c_int32),
        ("beta_sigmoid", ctypes.c_int32), ("decay_per_key", ctypes.c_int32),
        ("raw_gate", ctypes.c_int32), ("num_state_rows", ctypes.c_int32),
        ("threads", ctypes.c_int32),
        ("scale", creal),
        ("q", rp), ("k", rp), ("v", rp),
        ("decay", rp), ("gate_bias", rp), ("gate_scale", rp), ("beta", rp),
        ("cu_seqlens", _ip), ("slot_ids", _ip),
        ("initial_state", rp), ("final_state", rp), ("o", rp),
        ("error_word", _ip), ("seq_lens", _ip), ("beta_shared", ctypes.c_int32),
        ("state_kmajor", ctypes.c_int32), ("erase_gate", rp), ("write_gate", rp),
    ]


class _Problem(ctypes.Structure):
    _fields_ = _problem_fields(ctypes.c_double, _dp)


class _ProblemF32(ctypes.Structure):
    _fields_ = _problem_fields(ctypes.c_float, _fp)


# per arithmetic type: (numpy dtype, pointer type, problem struct)
_REAL = {"f64": (np.float64, _dp, _Problem), "f32": (np.float32, _fp, _ProblemF32)}
_libs = {}


def _load(real="f64"):
    if real not in _libs:
        _, rp, prob = _REAL[real]
        # GDN_ORACLE_LIB names a double build of a deliberately altered copy of
        # gdn_oracle.c: the planted-mistake test runs the pins against it
        alt = os.environ.get("GDN_ORACLE_LIB") if real == "f64" else None
        lib = ctypes.CDLL(alt or _build.build(real=real))
        lib.oracle_gdn.argtypes = [ctypes.POINTER(prob)]
        lib.oracle_gdn.restype = ctypes.c_int
        lib.oracle_gate.argtypes = [ctypes.c_int64, ctypes.c_int32, rp, rp, rp, rp, rp, rp]
        lib.oracle_gate.restype = ctypes.c_int
        _libs[real] = lib
    return _libs[real]


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor (CPU)
        x = x.detach().cpu()
        if str(x.dtype) in ("torch.float16", "torch.bfloat16", "torch.float32", "torch.float64"):
            x = x.double()
        x = x.numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a, typ):
    return None if a is None else a.ctypes.data_as(typ)


def gate(a, dt_bias, decay_scale, b=None, want_beta=False):
    """decay = decay_scale * softplus(a + dt_bias); beta = sigmoid(b).

    "com.microsoft.LinearAttentionGate", Description.  The last axis of ``a``
    is the head axis; leading axes are folded.
    """
    lib = _load()
    a64 = _f64(a)
    shape = a64.shape
    h = shape[-1]
    n = int(a64.size // h)
    bias = _f64(dt_bias).reshape(-1)
    dscale = _f64(decay_scale).reshape(-1)
    b64 = _f64(b) if b is not None else None
    decay = np.empty(shape, np.float64)
    beta = np.empty(shape, np.float64) if want_beta else None
    rc = lib.oracle_gate(n, h, _ptr(a64, _dp), _ptr(bias, _dp), _ptr(dscale, _dp),
                         _ptr(b64, _dp), _ptr(decay, _dp), _ptr(beta, _dp))
    if rc != 0:
        raise ValueError("oracle_gate rejected its arguments")
    return (decay, beta) if want_beta else decay


def gdn(q, k, v, *, rule="gated_delta", decay=None, beta=None, gate_bias=None,
        gate_scale=None, cu_seqlens=None, batch=None, slot_ids=None,
        initial_state=None, final_state=None, num_state_rows=None, scale=0.0,
        l2norm_q=False, l2norm_k=False, beta_sigmoid=False, decay_per_key=False,
        threads=1, seq_lens=None, beta_shared=False, state_kmajor=False, erase_gate=None,
        write_gate=None, real="f64"):
    """Runs the recurrence token by token in float64.

    q, k: [T, Hq, dk]; v: [T, Hv, dv] (rank-4 callers flatten [B, S] to T and
    pass batch=B).  Returns (o [T, Hv, dv], final_state [rows, Hv, dv, dk],
    error_word).  ``final_state`` (if given) is the buffer the update lands in
    (copied, so the caller's array is not modified); rows that no request
    names keep its values.  Output tokens outside every request are NaN.
    ``seq_lens`` ([batch], uniform layout only) shortens request b to the first
    seq_lens[b] tokens of its row.  ``beta_shared``: the scalar beta is [T],
    one per token for every value head.  ``state_kmajor``: states are
    [rows, Hv, dk, dv] ("gatedDeltaUpdate") instead of [rows, Hv, dv, dk].
    ``erase_gate`` ([T, Hv, dk], rule gdn2): the GDN-2 erase gate as its own
    input, beta then being the scalar write rate; ``write_gate`` ([T, Hv, dv],
    rule gdn2): the GDN-2 write gate, applied to v here.  ``real``: "f64" (the
    definition) or "f32" (the float instantiation, for timing only).
    """
    lib = _load(real)
    dt, rp, Prob = _REAL[real]

    def cv(x):
        x = _f64(x)
        return x if x is None or real == "f64" else np.ascontiguousarray(x.astype(dt))
    q64, k64, v64 = cv(q), cv(k), cv(v)
    T, hq, dk = q64.shape
    hv, dv = v64.shape[1], v64.shape[2]
    cu = _i32(cu_seqlens)
    slots = _i32(slot_ids)
    sl = _i32(seq_lens)
    if batch is None:
        batch = (len(cu) - 1) if cu is not None else 1
    init = cv(initial_state)
    if num_state_rows is None:
        if final_state is not None:
            num_state_rows = int(np.asarray(final_state.shape)[0])
        elif init is not None:
            num_state_rows = init.shape[0]
        else:
            num_state_rows = batch
    if final_state is not None:
        fin = cv(final_state).copy()
    elif init is not None:
        fin = init.copy()
    else:
        fin = np.zeros((num_state_rows, hv, dk, dv) if state_kmajor else (num_state_rows, hv, dv, dk), dt)
    o = np.full((T, hv, dv), np.nan, dt)
    err = np.zeros(1, np.int32)
    dec = cv(decay)
    bet = cv(beta)
    gb = cv(gate_bias)
    gs = cv(gate_scale)
    eg = cv(erase_gate)
    wg = cv(write_gate)
    raw = gb is not None or gs is not None
    prob = Prob(
        batch=batch, total_tokens=T, hq=hq, hv=hv, dk=dk, dv=dv, rule=RULES[rule],
        l2norm_q=int(l2norm_q), l2norm_k=int(l2norm_k), beta_sigmoid=int(beta_sigmoid),
        decay_per_key=int(decay_per_key), raw_gate=int(raw), num_state_rows=num_state_rows,
        threads=int(threads), scale=float(scale),
        q=_ptr(q64, rp), k=_ptr(k64, rp), v=_ptr(v64, rp),
        decay=_ptr(dec, rp), gate_bias=_ptr(gb, rp), gate_scale=_ptr(gs, rp),
        beta=_ptr(bet, rp), cu_seqlens=_ptr(cu, _ip), slot_ids=_ptr(slots, _ip),
        initial_state=_ptr(init, rp), final_state=_ptr(fin, rp), o=_ptr(o, rp),
        error_word=_ptr(err, _ip), seq_lens=_ptr(sl, _ip), beta_shared=int(beta_shared),
        state_kmajor=int(bool(state_kmajor)), erase_gate=_ptr(eg, rp), write_gate=_ptr(wg, rp),
    )
    rc = lib.oracle_gdn(ctypes.byref(prob))
    if rc != 0:
        raise ValueError("oracle_gdn rejected its arguments (rc=%d)" % rc)
    if real != "f64":
        o, fin = o.astype(np.float64), fin.astype(np.float64)
    return o, fin, int(err[0])


def torch_index(idx):
    import torch
    return torch.as_tensor(np.asarray(idx, dtype=np.int64))


def round_to(x, dtype):
    """Rounds float64 results once to an activation dtype ('f16' or 'f32')."""
    np_dtype = {"f16": np.float16, "f32": np.float32}[dtype]
    return np.asarray(x).astype(np_dtype).astype(np.float64)


def lib_path():
    return _build.LIB


__all__ = ["gate", "gdn", "run_problem", "round_to", "RULES", "ERR_BAD_SLOT", "lib_path"]
os.environ.setdefault("OMP_WAIT_POLICY", "PASSIVE")


def run_problem(p, threads=1, requests=None, real="f64"):
    """Runs the oracle on a problem dict (the layout ``workloads.make`` draws).

    ``requests`` optionally restricts the run to a subset of request indices
    (their tokens and state rows only); the other outputs stay NaN and the
    other state rows keep their initial values.  ``real`` as for ``gdn``.
    """
    q, k, v = p["q"], p["k"], p["v"]
    T = p["total_tokens"]
    q = q.reshape(T, p["hq"], p["dk"])
    k = k.reshape(T, p["hq"], p["dk"])
    v = v.reshape(T, p["hv"], p["dv"])
    cu = p.get("cu_seqlens")
    slots = p.get("slot_ids")
    batch = p["batch"]
    sl = p.get("seq_lens")
    if cu is None:
        L = T // batch
        cu_np = np.arange(batch + 1, dtype=np.int64) * L
    else:
        cu_np = np.asarray(cu.numpy() if hasattr(cu, "numpy") else cu, dtype=np.int64)
    ranges = []
    for b in range(batch):
        t0 = min(max(int(cu_np[b]), 0), T)
        t1 = max(min(max(int(cu_np[b + 1]), 0), T), t0)
        if sl is not None:
            t1 = t0 + min(max(int(sl[b]), 0), t1 - t0)
        ranges.append((t0, t1))
    if requests is not None:
        # Sub-problem: the chosen requests keep their own token ranges; their
        # state rows are gathered into a compact slab (row j = request j), so
        # the returned final state has one row per chosen request.
        req = list(requests)
        sub_cu = np.zeros(len(req) + 1, dtype=np.int64)
        rows = []
        T_, idx = 0, []
        for j, b in enumerate(req):
            t0, t1 = ranges[b]
            idx.extend(range(t0, t1))
            T_ += t1 - t0
            sub_cu[j + 1] = T_
            rows.append(int(slots[b]) if slots is not None else b)
        idx = np.asarray(idx, dtype=np.int64)

        def take(x):
            if x is None:
                return None
            if hasattr(x, "detach"):
                x = x.reshape((T,) + tuple(x.shape[1:]))
                return _f64(x[torch_index(idx)])
            xn = _f64(x)
            return xn.reshape((T,) + xn.shape[1:])[idx]

        init = p.get("initial_state")
        init_sub = None
        if init is not None:
            init_sub = _f64(init[torch_index(np.asarray(rows))] if hasattr(init, "detach")
                            else np.asarray(init)[rows])
        o_s, fin, err = gdn(take(q), take(k), take(v), rule=p["rule"], decay=take(p.get("decay")),
                            beta=take(p.get("beta")), gate_bias=p.get("gate_bias"),
                            gate_scale=p.get("gate_scale"), cu_seqlens=sub_cu, batch=len(req),
                            slot_ids=None, initial_state=init_sub, num_state_rows=len(req),
                            scale=p.get("scale", 0.0),
                            l2norm_q=p.get("l2norm_q", False), l2norm_k=p.get("l2norm_k", False),
                            beta_sigmoid=p.get("beta_sigmoid", False),
                            decay_per_key=p.get("decay_per_key", False), threads=threads,
                            beta_shared=p.get("beta_shared", False),
                            state_kmajor=p.get("state_kmajor", False),
                            erase_gate=take(p.get("erase_gate")), write_gate=take(p.get("write_gate")),
                            real=real)
        o = np.full((T, p["hv"], p["dv"]), np.nan)
        if len(idx):
            o[idx] = o_s
        return o, fin, err
    return gdn(q, k, v, rule=p["rule"], decay=p.get("decay"), beta=p.get("beta"),
               gate_bias=p.get("gate_bias"), gate_scale=p.get("gate_scale"),
               cu_seqlens=cu if cu is not None else None, batch=batch, slot_ids=slots,
               initial_state=p.get("initial_state"),
               num_state_rows=p.get("num_slots") or batch, scale=p.get("scale", 0.0),
               l2norm_q=p.get("l2norm_q", False), l2norm_k=p.get("l2norm_k", False),
               beta_sigmoid=p.get("beta_sigmoid", False),
               decay_per_key=p.get("decay_per_key", False), threads=threads, seq_lens=sl,
               beta_shared=p.get("beta_shared", False), state_kmajor=p.get("state_kmajor", False),
               erase_gate=p.get("erase_gate"), write_gate=p.get("write_gate"), real=real)

"""Helpers for the GPU parity tests: move a drawn problem to the device, run
one entry point through the C ABI, and compare with the oracle.

Error metric (per output tensor): max |x - ref| / max |ref| over the
elements compared.
"""
import numpy as np
import torch

from gated_delta_rule_gate_gb300 import api

DEV = "cuda"


def poison_uncovered(p):
    """Fills every token that no request covers (gaps between requests, the
    padding of seq_lens rows) with NaN in q, k, v and the gates: no result may
    depend on them."""
    import workloads
    T = p["total_tokens"]
    covered = np.zeros(T, dtype=bool)
    for t0, t1 in workloads.token_ranges(p):
        covered[t0:t1] = True
    idx = torch.as_tensor(np.nonzero(~covered)[0])
    for key in ("q", "k", "v", "decay", "beta", "erase_gate", "write_gate"):
        t = p.get(key)
        if t is not None and len(idx):
            t = t.clone()
            t.reshape((T,) + tuple(t.shape[1:]) if t.dim() > 1 else (T,))[idx] = float("nan")
            p[key] = t
    return p


def to_dev(p):
    d = dict(p)
    for key in ("q", "k", "v", "decay", "gate_bias", "gate_scale", "beta", "cu_seqlens",
                "slot_ids", "initial_state", "seq_lens", "erase_gate", "write_gate"):
        t = p.get(key)
        if t is not None:
            d[key] = torch.as_tensor(t).to(DEV).contiguous()
    return d


def rel_err(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    denom = np.max(np.abs(ref)) if ref.size else 0.0
    if ref.size == 0:
        return 0.0
    diff = np.max(np.abs(x - ref))
    return float(diff / denom) if denom > 0 else float(diff)


def shape_qkv(p, d):
    """Rank-4 problems pass [B, S, H, d] views; rank-3 pass [T, H, d]."""
    if p.get("seq_len"):
        B, S = p["batch"], p["seq_len"]
        return (d["q"].view(B, S, p["hq"], p["dk"]), d["k"].view(B, S, p["hq"], p["dk"]),
                d["v"].view(B, S, p["hv"], p["dv"]))
    return d["q"], d["k"], d["v"]


def run(p, path="recurrent", chunk=64, in_place=None, sentinel=float("nan"), error_word=None,
        stream=None, d=None, workspace_extra=None):
    """Runs the problem on the GPU.  Returns (o, final_state, d) with o and
    final_state on the device.  Output tokens not covered stay ``sentinel``.
    ``in_place``: final_state is the same tensor as initial_state (default: when
    slot_ids are present).  Otherwise final_state starts as ``sentinel``.
    ``workspace_extra`` (chunked path): the workspace is the least the call
    accepts plus this many bytes, instead of the single-pass size."""
    if d is None:
        d = to_dev(p)
    q, k, v = shape_qkv(p, d)
    o = torch.full(v.shape, sentinel, dtype=v.dtype, device=DEV)
    rows = p.get("num_slots") or p["batch"]
    if in_place is None:
        in_place = p.get("slot_ids") is not None
    init = d.get("initial_state")
    sshape = (rows, p["hv"], p["dk"], p["dv"]) if p.get("state_kmajor") else (rows, p["hv"], p["dv"], p["dk"])
    if in_place:
        if init is None:
            init = torch.zeros(*sshape, device=DEV)
        init = init.clone()
        fin = init
    else:
        fin = torch.full(sshape, sentinel, dtype=torch.float32, device=DEV)
    kw = dict(q=q, k=k, v=v, o=o, final_state=fin, rule=p["rule"], decay=d.get("decay"),
              beta=d.get("beta"), gate_bias=d.get("gate_bias"), gate_scale=d.get("gate_scale"),
              cu_seqlens=d.get("cu_seqlens"), slot_ids=d.get("slot_ids"), initial_state=init,
              seq_lens=d.get("seq_lens"), beta_shared=p.get("beta_shared", False),
              batch=p["batch"], scale=p.get("scale", 0.0), l2norm_q=p.get("l2norm_q", False),
              l2norm_k=p.get("l2norm_k", False), beta_sigmoid=p.get("beta_sigmoid", False),
              decay_per_key=p.get("decay_per_key", False), error_word=error_word,
              erase_gate=d.get("erase_gate"), write_gate=d.get("write_gate"),
              state_kmajor=p.get("state_kmajor", False))
    prob = api.make_problem(**kw)
    if path == "recurrent":
        api.gdn_recurrent_step(prob, stream=stream)
    elif workspace_extra is not None:
        n = api.gdn_chunked_prefill_workspace_size_min(prob, chunk) + workspace_extra
        ws = torch.empty(max(n, 1), dtype=torch.uint8, device=DEV)
        api.gdn_chunked_prefill(prob, chunk_size=chunk, workspace=ws, stream=stream)
    else:
        api.gdn_chunked_prefill(prob, chunk_size=chunk, stream=stream)
    return o, fin, d


def o_flat(o, p):
    return o.reshape(p["total_tokens"], p["hv"], p["dv"]).double().cpu().numpy()

"""Python binding of libgdn with the C ABI's names, over torch tensors.

PyTorch supplies device memory and the current stream; these functions only
read shapes, dtypes and pointers, fill the C structs of include/gdn.h and
call the library.  Nothing here computes any part of the recurrence.
"""
import ctypes

import torch

from . import _native as N

_DT = {torch.float32: N.DTYPE_F32, torch.float16: N.DTYPE_F16, torch.bfloat16: N.DTYPE_BF16}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype(t, what):
    if t.dtype not in _DT:
        raise TypeError("%s: unsupported dtype %s" % (what, t.dtype))
    return _DT[t.dtype]


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need_cuda(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("libgdn takes device tensors; got a tensor on %s" % t.device)
            if not t.is_contiguous():
                raise ValueError("libgdn takes contiguous tensors")


def make_problem(q, k, v, o, final_state, *, rule="gated_delta", decay=None, beta=None,
                 gate_bias=None, gate_scale=None, cu_seqlens=None, slot_ids=None,
                 initial_state=None, batch=None, scale=0.0, l2norm_q=False, l2norm_k=False,
                 beta_sigmoid=False, decay_per_key=False, error_word=None,
                 state_update_capacity=0, seq_lens=None, beta_shared=False, erase_gate=None,
                 write_gate=None, state_kmajor=False):
    """Builds the ``gdn_problem`` struct.  q/k are [T, Hq, dk] (rank-3, packed)
    or [B, S, Hq, dk] (rank-4); v/o follow with Hv, dv; states are
    [rows, Hv, dv, dk] fp32.  ``seq_lens`` ([B] int32, rank-4 only) bounds each
    row to its first seq_lens[b] tokens.  ``beta_shared``: beta is [T] (one
    per token for every value head).  GDN2: ``erase_gate`` ([T, Hv, dk] fp32)
    is the erase gate as its own input, beta then being the scalar write
    rate; ``write_gate`` ([T, Hv, dv] fp32) is multiplied into v by the
    kernels.  ``state_kmajor``: states are [rows, Hv, dk, dv].  Keeps
    references to the tensors alive on the returned struct."""
    _need_cuda(q, k, v, o, final_state, decay, beta, gate_bias, gate_scale, cu_seqlens,
               slot_ids, initial_state, error_word, seq_lens, erase_gate, write_gate)
    if q.dim() == 4:
        B, S, hq, dk = q.shape
        T, seq_len = B * S, S
        hv, dv = v.shape[2], v.shape[3]
    elif q.dim() == 3:
        T, hq, dk = q.shape
        hv, dv = v.shape[1], v.shape[2]
        seq_len = 0
        if batch is None:
            batch = (cu_seqlens.numel() - 1) if cu_seqlens is not None else 1
        B = batch
    else:
        raise ValueError("q must be rank 3 or 4")
    p = N.GdnProblem()
    p.batch, p.total_tokens, p.seq_len = int(B), int(T), int(seq_len)
    p.num_heads_q, p.num_heads_v, p.head_dim_k, p.head_dim_v = int(hq), int(hv), int(dk), int(dv)
    p.num_state_rows = int(final_state.shape[0]) if final_state is not None else 0
    p.act_dtype = _dtype(q, "q")
    for t, name in ((k, "k"), (v, "v"), (o, "o")):
        if t is not None and t.dtype != q.dtype:
            raise TypeError("%s must have the dtype of q" % name)
    p.decay_dtype = _dtype(decay, "decay") if decay is not None else N.DTYPE_F32
    p.beta_dtype = _dtype(beta, "beta") if beta is not None else N.DTYPE_F32
    p.rule = N.RULES[rule] if isinstance(rule, str) else int(rule)
    p.flags = ((N.FLAG_L2NORM_Q if l2norm_q else 0) | (N.FLAG_L2NORM_K if l2norm_k else 0) |
               (N.FLAG_BETA_SIGMOID if beta_sigmoid else 0) |
               (N.FLAG_DECAY_PER_KEY if decay_per_key else 0) | (N.FLAG_BETA_SHARED if beta_shared else 0) |
               (N.FLAG_STATE_KMAJOR if state_kmajor else 0))
    p.scale = float(scale)
    p.state_update_capacity = int(state_update_capacity)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("decay", decay),
                    ("gate_bias", gate_bias), ("gate_scale", gate_scale), ("beta", beta),
                    ("cu_seqlens", cu_seqlens), ("slot_ids", slot_ids),
                    ("initial_state", initial_state), ("final_state", final_state),
                    ("error_word", error_word), ("seq_lens", seq_lens), ("erase_gate", erase_gate),
                    ("write_gate", write_gate)):
        setattr(p, name, None if t is None else t.data_ptr())
    for t, name, dt in ((cu_seqlens, "cu_seqlens", torch.int32), (slot_ids, "slot_ids", torch.int32),
                        (seq_lens, "seq_lens", torch.int32),
                        (error_word, "error_word", torch.int32), (gate_bias, "gate_bias", torch.float32),
                        (gate_scale, "gate_scale", torch.float32),
                        (initial_state, "initial_state", torch.float32),
                        (final_state, "final_state", torch.float32), (erase_gate, "erase_gate", torch.float32),
                        (write_gate, "write_gate", torch.float32)):
        if t is not None and t.dtype != dt:
            raise TypeError("%s must be %s" % (name, dt))
    p._keep = (q, k, v, o, final_state, decay, beta, gate_bias, gate_scale, cu_seqlens, slot_ids,
               initial_state, error_word, seq_lens, erase_gate, write_gate)
    return p


def gdn_status_string(status):
    return N.status_string(status)


def gdn_gate(a, dt_bias, decay_scale, b=None, *, want_beta=False, decay_out=None, beta_out=None,
             stream=None):
    """decay = decay_scale * softplus(a + dt_bias); beta = sigmoid(b) if asked.
    Outputs take a's shape and dtype (allocated when not given)."""
    _need_cuda(a, dt_bias, decay_scale, b)
    if decay_out is None:
        decay_out = torch.empty_like(a)
    if want_beta and beta_out is None:
        beta_out = torch.empty_like(a)
    heads = a.shape[-1] if a.dim() > 0 else 1
    args = N.GdnGateArgs()
    args.n = a.numel() // max(heads, 1)
    args.heads = heads
    args.dtype = _dtype(a, "a")
    args.a, args.dt_bias, args.decay_scale = a.data_ptr(), dt_bias.data_ptr(), decay_scale.data_ptr()
    args.b = b.data_ptr() if b is not None else None
    args.decay_out = decay_out.data_ptr()
    args.beta_out = beta_out.data_ptr() if (want_beta or beta_out is not None) else None
    N.check(N.load().gdn_gate(ctypes.byref(args), _stream(stream)))
    return (decay_out, beta_out) if want_beta else decay_out


def gdn_recurrent_step(problem=None, *, stream=None, **kw):
    """Token-serial recurrence.  Pass a struct from make_problem(), or the
    make_problem() keyword arguments directly."""
    if problem is None:
        problem = make_problem(**kw)
    N.check(N.load().gdn_recurrent_step(ctypes.byref(problem), _stream(stream)))
    return problem


def gdn_chunked_prefill_workspace_size(problem, chunk_size=64):
    n = N.load().gdn_chunked_prefill_workspace_size(ctypes.byref(problem), int(chunk_size))
    if n == ctypes.c_size_t(-1).value:
        raise N.GdnError(N.GDN_ERR_UNSUPPORTED, N.last_error_message())
    return n


def gdn_chunked_prefill_workspace_size_min(problem, chunk_size=64):
    n = N.load().gdn_chunked_prefill_workspace_size_min(ctypes.byref(problem), int(chunk_size))
    if n == ctypes.c_size_t(-1).value:
        raise N.GdnError(N.GDN_ERR_UNSUPPORTED, N.last_error_message())
    return n


def gdn_chunked_prefill(problem=None, chunk_size=64, workspace=None, *, stream=None, **kw):
    """Chunk-parallel recurrence (same result within the tensor-core
    tolerance).  Allocates the workspace with torch when none is given."""
    if problem is None:
        problem = make_problem(**kw)
    lib = N.load()
    need = gdn_chunked_prefill_workspace_size(problem, chunk_size)
    if workspace is None and need > 0:
        dev = torch.device("cuda", torch.cuda.current_device())
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    N.check(lib.gdn_chunked_prefill(ctypes.byref(problem), int(chunk_size), ws_ptr, ws_bytes,
                                    _stream(stream)))
    problem._ws = workspace
    return problem


def gdn_chunked_prefill_noalloc(problem=None, chunk_size=64, *, stream=None, **kw):
    """gdn_chunked_prefill with the library's static per-device scratch
    instead of a workspace: no device memory is allocated around the call.
    Calls on one device must not overlap (they share the scratch); the first
    call on a device must not be inside a stream capture."""
    if problem is None:
        problem = make_problem(**kw)
    N.check(N.load().gdn_chunked_prefill_noalloc(ctypes.byref(problem), int(chunk_size), _stream(stream)))
    return problem

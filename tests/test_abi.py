"""C-ABI checks that need no GPU: the library loads, exports every function
include/gdn.h declares, and rejects bad arguments on the host before any
launch (so these calls never reach the device)."""
import ctypes
import os
import re

import pytest

from gated_delta_rule_gate_gb300 import _native as N

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(gdn_[a-z_0-9]+)\s*\(", src, re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for want in ("gdn_gate", "gdn_recurrent_step", "gdn_chunked_prefill",
                 "gdn_chunked_prefill_workspace_size", "gdn_status_string"):
        assert want in names


def test_library_exports_every_declared_symbol():
    lib = N.load()
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings():
    assert N.status_string(N.GDN_OK) == "ok"
    for s in range(1, 5):
        assert N.status_string(s) not in ("", "unknown status")
    assert N.status_string(99) == "unknown status"


FAKE = 0x100000  # a 256-byte aligned non-null address; never dereferenced by the host


def _problem(**over):
    p = N.GdnProblem()
    p.batch, p.total_tokens, p.seq_len = 2, 8, 0
    p.num_heads_q, p.num_heads_v, p.head_dim_k, p.head_dim_v = 2, 4, 16, 16
    p.num_state_rows = 0
    p.act_dtype, p.decay_dtype, p.beta_dtype = N.DTYPE_F16, N.DTYPE_F32, N.DTYPE_F32
    p.rule, p.flags, p.scale, p.state_update_capacity = N.RULES["gated_delta"], 0, 0.0, 0
    for f in ("q", "k", "v", "o", "decay", "beta", "final_state"):
        setattr(p, f, FAKE)
    for k, v in over.items():
        setattr(p, k, v)
    return p


def _call(p):
    return N.load().gdn_recurrent_step(ctypes.byref(p), None)


def _call_chunked(p, chunk=64, ws=None, nbytes=0):
    return N.load().gdn_chunked_prefill(ctypes.byref(p), chunk, ws, nbytes, None)


@pytest.mark.parametrize("over,status,msg", [
    (dict(num_heads_v=3), N.GDN_ERR_INVALID, "multiple"),
    (dict(num_heads_q=0), N.GDN_ERR_INVALID, "positive"),
    (dict(head_dim_k=0), N.GDN_ERR_INVALID, "positive"),
    (dict(head_dim_k=512), N.GDN_ERR_UNSUPPORTED, "256"),
    (dict(act_dtype=N.DTYPE_BF16), N.GDN_ERR_UNSUPPORTED, "bfloat16"),
    (dict(act_dtype=7), N.GDN_ERR_INVALID, "dtype"),
    (dict(rule=9), N.GDN_ERR_INVALID, "rule"),
    (dict(decay=None), N.GDN_ERR_INVALID, "needs decay"),
    (dict(beta=None), N.GDN_ERR_INVALID, "needs beta"),
    (dict(rule=N.RULES["linear"]), N.GDN_ERR_INVALID, "decay given"),
    (dict(rule=N.RULES["gated"]), N.GDN_ERR_INVALID, "beta given"),
    (dict(gate_bias=FAKE), N.GDN_ERR_INVALID, "together"),
    (dict(gate_scale=FAKE), N.GDN_ERR_INVALID, "together"),
    (dict(state_update_capacity=4), N.GDN_ERR_INVALID, "state_update_capacity"),
    (dict(seq_len=4, cu_seqlens=FAKE), N.GDN_ERR_INVALID, "rank-3"),
    (dict(seq_lens=FAKE), N.GDN_ERR_INVALID, "rank-4"),
    (dict(flags=N.FLAG_BETA_SHARED, rule=N.RULES["gdn2"]), N.GDN_ERR_INVALID, "BETA_SHARED"),
    (dict(seq_len=4, seq_lens=FAKE + 2), N.GDN_ERR_INVALID, "aligned"),
    (dict(seq_len=3), N.GDN_ERR_INVALID, "batch * seq_len"),
    (dict(total_tokens=7), N.GDN_ERR_INVALID, "multiple of batch"),
    (dict(final_state=None), N.GDN_ERR_INVALID, "final_state"),
    (dict(q=None), N.GDN_ERR_INVALID, "required"),
    (dict(q=FAKE + 1), N.GDN_ERR_INVALID, "aligned"),
    (dict(decay_dtype=N.DTYPE_BF16), N.GDN_ERR_UNSUPPORTED, "bfloat16"),
    (dict(act_dtype=N.DTYPE_F32, beta_dtype=N.DTYPE_F16), N.GDN_ERR_INVALID, "beta_dtype"),
    (dict(flags=0x100), N.GDN_ERR_INVALID, "flag"),
    (dict(rule=N.RULES["delta"], decay=None, flags=N.FLAG_DECAY_PER_KEY), N.GDN_ERR_INVALID,
     "PER_KEY"),
    (dict(num_state_rows=1), N.GDN_ERR_INVALID, "num_state_rows"),
    (dict(scale=float("inf")), N.GDN_ERR_INVALID, "finite"),
    (dict(erase_gate=FAKE), N.GDN_ERR_INVALID, "GDN2"),
    (dict(write_gate=FAKE), N.GDN_ERR_INVALID, "GDN2"),
    (dict(rule=N.RULES["gdn2"], erase_gate=FAKE + 2), N.GDN_ERR_INVALID, "aligned"),
    (dict(rule=N.RULES["gdn2"], write_gate=FAKE + 1), N.GDN_ERR_INVALID, "aligned"),
    (dict(flags=N.FLAG_STATE_KMAJOR << 1), N.GDN_ERR_INVALID, "flag"),
])
def test_recurrent_rejects(over, status, msg):
    p = _problem(**over)
    assert _call(p) == status
    assert msg.lower() in N.last_error_message().lower()
    # the chunked entry point applies the same contract first
    assert _call_chunked(p) == status


def test_chunked_rejects_unsupported_head_sizes():
    p = _problem(head_dim_k=12, head_dim_v=9)
    assert _call_chunked(p) == N.GDN_ERR_UNSUPPORTED
    assert N.load().gdn_chunked_prefill_workspace_size(ctypes.byref(p), 64) == ctypes.c_size_t(-1).value


def test_chunked_workspace_size():
    """The tensor-core path (dk = dv = 128, fp16) asks for a workspace: chunk
    offsets (B + 1 ints), a slot -> request table (one int per slot) and the
    request order (B ints), rounded up to 1 KiB; then one 88 KiB operand image
    per (chunk slot, value head), with T / 64 + B + 1 slots, for every rule.
    The other shapes need none."""
    lib = N.load()
    size = lambda p: lib.gdn_chunked_prefill_workspace_size(ctypes.byref(p), 64)
    B, T, hv = 4, 4 * 8192, 16
    slots = T // 64 + B + 1
    head = -(-(2 * B + 1 + slots) * 4 // 1024) * 1024
    images = slots * hv * 88 * 1024
    p = _problem(batch=B, total_tokens=T, num_heads_q=16, num_heads_v=hv, head_dim_k=128,
                 head_dim_v=128)
    assert size(p) == head + images
    p.rule, p.decay = N.RULES["delta"], None
    assert size(p) == head + images
    p.rule, p.beta = N.RULES["linear"], None
    assert size(p) == head + images
    p.rule, p.decay = N.RULES["gated"], FAKE
    assert size(p) == head + images
    assert size(_problem()) == 0  # dk = dv = 16 runs without a workspace
    # fp32 activations take the same path through fp16 copies of q, k, v kept in the workspace
    p = _problem(batch=B, total_tokens=T, num_heads_q=16, num_heads_v=hv, head_dim_k=128, head_dim_v=128,
                 act_dtype=N.DTYPE_F32)
    copy = lambda heads: -(-(T * heads * 128 * 2) // 256) * 256
    assert size(p) == head + images + 2 * copy(16) + copy(hv)
    # fp16 per-key gate rows (log decay; GDN-2's per-key beta) take fp32 copies [T, Hv, 128]
    gcopy = -(-(T * hv * 128 * 4) // 256) * 256
    p = _problem(batch=B, total_tokens=T, num_heads_q=16, num_heads_v=hv, head_dim_k=128, head_dim_v=128,
                 flags=N.FLAG_DECAY_PER_KEY, decay_dtype=N.DTYPE_F16, beta_dtype=N.DTYPE_F16)
    assert size(p) == head + images + gcopy
    p.rule = N.RULES["gdn2"]
    assert size(p) == head + images + 2 * gcopy


def test_chunked_rejects_a_small_workspace():
    p = _problem(batch=1, total_tokens=64, num_heads_q=1, num_heads_v=1, head_dim_k=128,
                 head_dim_v=128)
    need = N.load().gdn_chunked_prefill_workspace_size(ctypes.byref(p), 64)
    least = N.load().gdn_chunked_prefill_workspace_size_min(ctypes.byref(p), 64)
    assert need >= least > 0
    st = N.load().gdn_chunked_prefill(ctypes.byref(p), 64, ctypes.c_void_p(FAKE), least - 1, None)
    assert st == N.GDN_ERR_WORKSPACE
    st = N.load().gdn_chunked_prefill(ctypes.byref(p), 64, None, need, None)
    assert st == N.GDN_ERR_WORKSPACE
    st = N.load().gdn_chunked_prefill(ctypes.byref(p), 64, ctypes.c_void_p(FAKE + 16), need, None)
    assert st == N.GDN_ERR_WORKSPACE  # not 256-byte aligned


def test_gate_rejects():
    lib = N.load()
    a = N.GdnGateArgs()
    a.n, a.heads, a.dtype = 4, 3, N.DTYPE_F16
    a.a = a.dt_bias = a.decay_scale = a.decay_out = FAKE
    a.beta_out = FAKE  # beta requested without b
    assert lib.gdn_gate(ctypes.byref(a), None) == N.GDN_ERR_INVALID
    assert "without b" in N.last_error_message()
    a.beta_out = None
    a.dtype = N.DTYPE_BF16
    assert lib.gdn_gate(ctypes.byref(a), None) == N.GDN_ERR_UNSUPPORTED
    a.dtype = N.DTYPE_F16
    a.heads = 0
    assert lib.gdn_gate(ctypes.byref(a), None) == N.GDN_ERR_INVALID
    a.heads, a.n = 3, 0  # empty input: a no-op that launches nothing
    assert lib.gdn_gate(ctypes.byref(a), None) == N.GDN_OK
    assert lib.gdn_gate(None, None) == N.GDN_ERR_INVALID


def test_zero_batch_is_a_noop():
    p = _problem(batch=0, total_tokens=0)
    assert _call(p) == N.GDN_OK
    assert N.load().gdn_recurrent_step(None, None) == N.GDN_ERR_INVALID


def test_chunked_workspace_minimum():
    """The least workspace holds one chunk of every request (window ranges, a
    head and B * Hv images, plus any copies), whatever the request lengths;
    it never exceeds the single-pass size.  Below it the call is rejected with
    GDN_ERR_WORKSPACE."""
    lib = N.load()
    least = lambda p: lib.gdn_chunked_prefill_workspace_size_min(ctypes.byref(p), 64)
    full = lambda p: lib.gdn_chunked_prefill_workspace_size(ctypes.byref(p), 64)
    B, hv = 4, 16
    img = 88 * 1024
    for T in (4 * 8192, 4 * 65536):
        p = _problem(batch=B, total_tokens=T, num_heads_q=16, num_heads_v=hv, head_dim_k=128, head_dim_v=128)
        m = least(p)
        fixed = -(-(2 * B * 4) // 256) * 256 + (2 * B + 1) * 4 + 1023
        assert m == -(-(fixed + B * (hv * img + 4)) // 256) * 256
        assert m < full(p)
    p = _problem(batch=1, total_tokens=64, num_heads_q=1, num_heads_v=1, head_dim_k=128, head_dim_v=128)
    assert 0 < least(p) <= full(p)
    assert least(_problem()) == 0  # dk = dv = 16 runs without a workspace
    p = _problem(batch=B, total_tokens=4 * 8192, num_heads_q=16, num_heads_v=hv, head_dim_k=128, head_dim_v=128)
    st = lib.gdn_chunked_prefill(ctypes.byref(p), 64, ctypes.c_void_p(FAKE), least(p) - 256, None)
    assert st == N.GDN_ERR_WORKSPACE

"""GPU parity, through the C ABI, of two input forms on every kernel path:

* the key-major state layout ("gatedDeltaUpdate": state and slot slab
  [rows, Hv, dk, dv], GDN_FLAG_STATE_KMAJOR);
* the GDN-2 gates as inputs (ONNX GDN-2 issue: the erase gate as its own
  input beside a scalar beta, proposal B, and the write gate w passed to the
  op instead of folded into v).

Tolerances as in the other parity files: the token-serial path computes in
fp32 (state 1e-4, fp16 outputs 5e-3), the chunked path multiplies fp16
operands on the tensor cores (5e-3), all as max |x - ref| / max |ref|.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import DEV, o_flat, rel_err, run

pytestmark = pytest.mark.gpu

TOL_STATE = 1e-4
TOL_O = {"f32": 1e-4, "f16": 5e-3}
TOL_CHUNKED = 5e-3


def _cid(c):
    return "-".join("%s=%s" % (k, v) for k, v in sorted(c.items()))


def _check(p, o, fin, ref_o, ref_fin, tol_o, tol_s):
    og = o_flat(o, p)
    covered = ~np.isnan(ref_o)
    assert np.isnan(og[~covered]).all()
    e_o = rel_err(og[covered], ref_o[covered])
    e_s = rel_err(fin.double().cpu().numpy(), ref_fin)
    assert e_o <= tol_o and e_s <= tol_s, (e_o, e_s)


# ------------------------------------------------------------ key-major state
KM_RECURRENT = [
    dict(lengths=[1, 4, 0, 2, 3, 8, 1], dk=128, dv=128),                 # decode kernel
    dict(lengths=[1, 4, 0, 2, 3], dk=128, dv=128, rule="gdn2", decay_per_key=True, gate_dtype="f32"),
    dict(lengths=[1, 2, 12, 1], dk=128, dv=128, rule="linear"),          # decode kernel, restaged tokens
    dict(lengths=[120, 3, 77], dk=128, dv=128),                          # long-request kernel
    dict(lengths=[150, 40], dk=64, dv=96, rule="gated", act="f32"),      # long-request kernel, dv != dk
    dict(lengths=[3, 0, 5], dk=48, dv=24),                               # any-dk kernel
    dict(lengths=[2, 5, 1], dk=64, dv=64, rule="delta"),                 # any-dk kernel (short, dk 64)
]


@pytest.mark.parametrize("in_place", [True, False], ids=["slab", "separate"])
@pytest.mark.parametrize("case", KM_RECURRENT, ids=[_cid(c) for c in KM_RECURRENT])
def test_recurrent_key_major_state(case, in_place):
    kw = dict(seed=zlib.crc32(_cid(case).encode()) % 1000, B=len(case["lengths"]), hq=2, hv=4, act="f16",
              rule="gated_delta", state="random", state_std=0.3, num_slots=len(case["lengths"]) + 3,
              slot_mode="perm", state_kmajor=True)
    kw.update(case)
    p = workloads.make(**kw)
    ref_o, ref_fin, err = oracle.run_problem(p)
    assert err == 0
    o, fin, _ = run(p, in_place=in_place)
    if not in_place:  # rows no request names keep the sentinel
        ref_fin = ref_fin.copy()
        touched = set(int(s) for s in p["slot_ids"])
        for r in range(p["num_slots"]):
            if r not in touched:
                ref_fin[r] = np.nan
        fg = fin.double().cpu().numpy()
        assert all(np.isnan(fg[r]).all() for r in range(p["num_slots"]) if r not in touched)
        keep = sorted(touched)
        og = o_flat(o, p)
        covered = ~np.isnan(ref_o)
        assert rel_err(og[covered], ref_o[covered]) <= TOL_O[p["act_dtype"]]
        assert rel_err(fg[keep], ref_fin[keep]) <= TOL_STATE
        return
    _check(p, o, fin, ref_o, ref_fin, TOL_O[p["act_dtype"]], TOL_STATE)


KM_CHUNKED = [
    dict(rule="gated_delta"),                                              # tcgen05, chain split by rows
    dict(rule="linear"),
    dict(rule="gated"),
    dict(rule="delta", hq=8, hv=32, lengths=[70, 0, 130, 1, 64]),         # tcgen05, one CTA per chain
    dict(rule="gdn2", decay_per_key=True, gate_dtype="f32"),               # per-key prepare + chain
    dict(rule="gated_delta", dk=64, dv=64),                                # warp-level MMA kernel
    dict(rule="gated", decay_per_key=True, gate_dtype="f32"),              # per-key prepare, no retrieval
    dict(rule="gated", decay_per_key=True),                                # per-key, fp16 gate copies
    dict(rule="gated", decay_per_key=True, dk=64, dv=64),                  # token-serial fallback
]


@pytest.mark.parametrize("case", KM_CHUNKED, ids=[_cid(c) for c in KM_CHUNKED])
def test_chunked_key_major_state(case):
    kw = dict(seed=zlib.crc32(_cid(case).encode()) % 1000, B=5, lengths=[70, 0, 130, 1, 64], hq=1, hv=2,
              dk=128, dv=128, act="f16", state="random", state_std=0.3, num_slots=7, slot_mode="perm",
              state_kmajor=True)
    kw.update(case)
    kw["B"] = len(kw["lengths"])
    p = workloads.make(**kw)
    ref_o, ref_fin, err = oracle.run_problem(p)
    assert err == 0
    o, fin, _ = run(p, path="chunked")
    _check(p, o, fin, ref_o, ref_fin, TOL_CHUNKED, TOL_CHUNKED)
    # rows no request names are untouched, bit for bit
    touched = set(int(s) for s in p["slot_ids"])
    for r in range(7):
        if r not in touched:
            assert torch.equal(fin[r].cpu(), p["initial_state"][r])


def test_key_major_equals_transposed_value_major():
    """The same problem with the state stored either way: the key-major final
    state is the transpose of the value-major one (chunked path, within the
    tensor-core tolerance; outputs too)."""
    p = workloads.make(seed=91, B=3, lengths=[150, 9, 64], hq=2, hv=4, dk=128, dv=128, act="f16",
                       state="random", state_std=0.3)
    o1, f1, _ = run(p, path="chunked")
    pk = dict(p, state_kmajor=True, initial_state=p["initial_state"].transpose(2, 3).contiguous())
    o2, f2, _ = run(pk, path="chunked")
    assert rel_err(o_flat(o2, p), o_flat(o1, p)) <= TOL_CHUNKED
    assert rel_err(f2.transpose(2, 3).double().cpu().numpy(), f1.double().cpu().numpy()) <= TOL_CHUNKED


# ------------------------------------------------------------ GDN-2 gates as inputs
GATES_RECURRENT = [
    dict(lengths=[1, 4, 0, 2, 3], dk=128, dv=128),                          # decode kernel
    dict(lengths=[1, 4, 0, 2], dk=128, dv=128, beta_shared=True),
    dict(lengths=[1, 3, 2], dk=128, dv=128, act="f32", write_gate="fold"),  # erase input only
    dict(lengths=[2, 1, 3], dk=128, dv=128, erase="beta"),                  # write gate only
    dict(lengths=[1, 3], dk=128, dv=128, decay_per_key=False),              # scalar decay
    dict(lengths=[120, 3, 77], dk=128, dv=128),                             # long-request kernel
    dict(lengths=[3, 0, 5], dk=48, dv=24),                                  # any-dk kernel
    dict(lengths=[1, 2, 12, 1], dk=128, dv=128, state_kmajor=True),         # decode kernel, key-major
]


@pytest.mark.parametrize("case", GATES_RECURRENT, ids=[_cid(c) for c in GATES_RECURRENT])
def test_recurrent_gdn2_gates_as_inputs(case):
    kw = dict(seed=zlib.crc32(_cid(case).encode()) % 1000, B=len(case["lengths"]), hq=2, hv=4, act="f16",
              rule="gdn2", decay_per_key=True, gate_dtype="f32", erase="input", write_gate="input",
              state="random", state_std=0.3)
    kw.update(case)
    p = workloads.make(**kw)
    ref_o, ref_fin, err = oracle.run_problem(p)
    assert err == 0
    o, fin, _ = run(p)
    _check(p, o, fin, ref_o, ref_fin, TOL_O[p["act_dtype"]], TOL_STATE)


GATES_CHUNKED = [
    dict(),                                                                # per-key prepare + chain
    dict(beta_shared=True),
    dict(write_gate="fold"),
    dict(erase="beta"),
    dict(decay_per_key=False),                                             # scalar decay, same kernels
    dict(hq=8, hv=32, lengths=[70, 0, 130, 1, 64]),                        # one CTA per chain
    dict(dk=64, dv=64, decay_per_key=False),                               # warp-level MMA kernel
    dict(gate_dtype="f16"),                                                # per-key, fp16 gate copies
    dict(dk=64, dv=64, gate_dtype="f16"),                                  # token-serial fallback
]


@pytest.mark.parametrize("case", GATES_CHUNKED, ids=[_cid(c) or "base" for c in GATES_CHUNKED])
def test_chunked_gdn2_gates_as_inputs(case):
    kw = dict(seed=zlib.crc32(_cid(case).encode()) % 1000, B=5, lengths=[70, 0, 130, 1, 64], hq=1, hv=2,
              dk=128, dv=128, act="f16", rule="gdn2", decay_per_key=True, gate_dtype="f32", erase="input",
              write_gate="input", state="random", state_std=0.3)
    kw.update(case)
    kw["B"] = len(kw["lengths"])
    p = workloads.make(**kw)
    ref_o, ref_fin, err = oracle.run_problem(p)
    assert err == 0
    o, fin, _ = run(p, path="chunked")
    _check(p, o, fin, ref_o, ref_fin, TOL_CHUNKED, TOL_CHUNKED)


def test_chunked_write_gate_input_equals_folded():
    """The write gate passed to the op gives the result of folding it into v
    on the host (within the tensor-core tolerance: the folded v is rounded to
    fp16 once more)."""
    p = workloads.make(seed=92, B=2, lengths=[130, 70], hq=1, hv=2, dk=128, dv=128, act="f16", rule="gdn2",
                       decay_per_key=True, gate_dtype="f32", write_gate="input", state="random", state_std=0.3)
    o1, f1, _ = run(p, path="chunked")
    pf = dict(p, write_gate=None, v=(p["v"].float() * p["write_gate"]).half())
    o2, f2, _ = run(pf, path="chunked")
    assert rel_err(o_flat(o1, p), o_flat(o2, p)) <= TOL_CHUNKED
    assert rel_err(f1.double().cpu().numpy(), f2.double().cpu().numpy()) <= TOL_CHUNKED


# ------------------------------------------------------------ per-key decay range
@pytest.mark.parametrize("hi,flagged", [(0.0, False), (0.5, True)])
def test_chunked_per_key_decay_above_one_is_flagged(hi, flagged):
    """The per-key tensor-core path needs log decays <= 0: a direct log decay
    above 0 sets GDN_DEVERR_DECAY_RANGE (0x8) in the error word; decays in
    (0, 1] leave it clear and match the oracle."""
    p = workloads.make(seed=93, B=2, lengths=[100, 60], hq=1, hv=2, dk=128, dv=128, act="f16",
                       rule="gated_delta", decay_per_key=True, gate="log", logdecay_range=(-1.0, hi),
                       state="random", state_std=0.3)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, fin, _ = run(p, path="chunked", error_word=err)
    torch.cuda.synchronize()
    assert bool(int(err.item()) & 0x8) == flagged
    if not flagged:
        ref_o, ref_fin, _ = oracle.run_problem(p)
        _check(p, o, fin, ref_o, ref_fin, TOL_CHUNKED, TOL_CHUNKED)

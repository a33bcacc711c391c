"""GPU parity of gdn_recurrent_step and gdn_gate against the CPU oracle,
through the C ABI.

Tolerances (max |x - ref| / max |ref|): the recurrent path computes in fp32,
so the state and fp32 outputs must agree to 1e-4; fp16 outputs carry one
fp16 rounding (relative 2^-11 ~ 4.9e-4), so they are held to 5e-3.
Routing, untouched rows and sentinels are compared bit-exactly.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import workloads
from gated_delta_rule_gate_gb300 import api
from gpu_helpers import DEV, o_flat, poison_uncovered, rel_err, run, to_dev

pytestmark = pytest.mark.gpu

TOL_STATE = 1e-4
TOL_O = {"f32": 1e-4, "f16": 5e-3}


def _check(p, o, fin, ref_o, ref_fin, tol_o=None):
    act = p["act_dtype"]
    tol_o = tol_o or TOL_O[act]
    og = o_flat(o, p)
    covered = ~np.isnan(ref_o)
    # tokens outside every request keep the sentinel, bit for bit
    assert np.isnan(og[~covered]).all()
    assert rel_err(og[covered], ref_o[covered]) <= tol_o, rel_err(og[covered], ref_o[covered])
    fg = fin.double().cpu().numpy()
    assert rel_err(fg, ref_fin) <= TOL_STATE, rel_err(fg, ref_fin)


# ---------------------------------------------------------------- gate op
@pytest.mark.parametrize("act", ["f32", "f16"])
@pytest.mark.parametrize("shape", [(5,), (3, 7), (2, 5, 32), (1, 1023, 16)])
def test_gate_matches_oracle(act, shape):
    g = torch.Generator().manual_seed(41)
    dt = workloads.ACT[act]
    a = (torch.randn(*shape, generator=g) * 3).to(dt)
    b = (torch.randn(*shape, generator=g) * 3).to(dt)
    h = shape[-1]
    bias = torch.rand(h, generator=g) * 4 - 2
    scale = -torch.exp(torch.rand(h, generator=g) * 2)
    dec, bet = api.gdn_gate(a.to(DEV), bias.to(DEV), scale.to(DEV), b.to(DEV), want_beta=True)
    rd, rb = oracle.gate(a, bias, scale, b=b, want_beta=True)
    # fp32 math, one rounding on store: within a few ulps of the output type
    tol = 2e-6 if act == "f32" else 1e-3
    np.testing.assert_allclose(dec.double().cpu().numpy(), rd, rtol=tol, atol=1e-7)
    np.testing.assert_allclose(bet.double().cpu().numpy(), rb, rtol=tol, atol=1e-7)
    only = api.gdn_gate(a.to(DEV), bias.to(DEV), scale.to(DEV))
    assert torch.equal(only, dec)


# ---------------------------------------------------------------- sweeps
CASES = []
for dk, dv in [(16, 16), (32, 32), (64, 64), (128, 128), (256, 256), (12, 9), (128, 64), (48, 40)]:
    CASES.append(dict(dk=dk, dv=dv, hq=2, hv=4, rule="gated_delta", act="f16"))
for rule in ["linear", "gated", "delta", "gated_delta", "gdn2"]:
    for act in ["f32", "f16"]:
        CASES.append(dict(dk=128, dv=128, hq=1, hv=2, rule=rule, act=act))
        CASES.append(dict(dk=24, dv=20, hq=1, hv=3, rule=rule, act=act))
CASES += [
    dict(dk=128, dv=128, hq=2, hv=2, rule="gated_delta", act="f16", gate="log"),
    dict(dk=128, dv=128, hq=2, hv=2, rule="gated_delta", act="f16", gate_dtype="f32", beta_dtype="f16"),
    dict(dk=64, dv=64, hq=1, hv=2, rule="gated_delta", act="f16", decay_per_key=True),
    dict(dk=64, dv=32, hq=1, hv=2, rule="gated", act="f32", decay_per_key=True),
    dict(dk=40, dv=24, hq=1, hv=1, rule="gdn2", act="f16", decay_per_key=True, write_gate=True),
    dict(dk=128, dv=128, hq=1, hv=1, rule="gdn2", act="f16", decay_per_key=True, write_gate=True),
    dict(dk=128, dv=128, hq=2, hv=4, rule="gated_delta", act="f16", beta_mode="direct",
         l2norm_q=True),
    dict(dk=32, dv=32, hq=1, hv=1, rule="delta", act="f32", l2norm_k=False, qk_std=0.2),
]


def _case_id(c):
    return "-".join("%s=%s" % (k, v) for k, v in sorted(c.items()))


@pytest.mark.parametrize("case", CASES, ids=[_case_id(c) for c in CASES])
def test_recurrent_parity_sweep(case):
    c = dict(case)
    kw = dict(seed=zlib.crc32(_case_id(c).encode()) % 1000, B=4, lengths=[3, 0, 11, 8], state="random",
              state_std=0.5)
    kw.update(c)
    p = workloads.make(**kw)
    ref_o, ref_fin, err = oracle.run_problem(p)
    assert err == 0
    o, fin, _ = run(p)
    _check(p, o, fin, ref_o, ref_fin)


SMALL_BLOCK = []
for rule in ["linear", "gated", "delta", "gated_delta", "gdn2"]:
    for dk, dv in [(128, 128), (64, 40), (32, 64)]:
        SMALL_BLOCK.append(dict(rule=rule, dk=dk, dv=dv))


@pytest.mark.parametrize("case", SMALL_BLOCK, ids=[_case_id(c) for c in SMALL_BLOCK])
def test_decode_blocks_of_one_to_four_tokens(case):
    """Requests of 1..4 tokens through the decode schedule, every rule: each
    (request, head) pair is staged as one token block, its norms reduced
    together.  dv = 40 leaves inactive rows inside a slice pair; the slab is
    updated in place through permuted slots."""
    kw = dict(seed=zlib.crc32(_case_id(case).encode()) % 1000, B=7, lengths=[1, 2, 3, 4, 0, 4, 2],
              hq=1, hv=2, act="f16", state="random", state_std=0.5, num_slots=9, slot_mode="perm")
    kw.update(case)
    p = workloads.make(**kw)
    ref_o, ref_fin, err = oracle.run_problem(p)
    assert err == 0
    o, fin, _ = run(p, in_place=True)
    og = o_flat(o, p)
    assert rel_err(og, ref_o) <= TOL_O["f16"]
    slots = [int(s) for s in p["slot_ids"]]
    fg = fin[torch.tensor(slots, device=DEV)].double().cpu().numpy()
    assert rel_err(fg, ref_fin[slots]) <= TOL_STATE


@pytest.mark.parametrize("kmajor", [False, True], ids=["vmajor", "kmajor"])
@pytest.mark.parametrize("rule", ["gated", "gated_delta"])
def test_decode_strong_decay_folds_the_lazy_factor(rule, kmajor):
    """Per-token log decays in [-7, -5]: within a block of staged tokens the
    decode kernels' lazy decay factor (the state kept as c * S~) falls below
    1e-20 and is folded into the state mid-block.  Requests of 8 tokens (one
    block) and 20 (restaged in blocks of 8) match the oracle in both state
    layouts."""
    kw = dict(seed=71 + 2 * int(kmajor) + int(rule == "gated"), B=4, lengths=[8, 20, 3, 1], hq=1, hv=2,
              dk=128, dv=128, act="f16", rule=rule, gate="log", logdecay_range=(-7.0, -5.0),
              state="random", state_std=0.5, num_slots=6, slot_mode="perm", state_kmajor=kmajor)
    p = workloads.make(**kw)
    ref_o, ref_fin, err = oracle.run_problem(p)
    assert err == 0
    o, fin, _ = run(p, in_place=True)
    assert rel_err(o_flat(o, p), ref_o) <= TOL_O["f16"]
    slots = [int(s) for s in p["slot_ids"]]
    fg = fin[torch.tensor(slots, device=DEV)].double().cpu().numpy()
    assert rel_err(fg, ref_fin[slots]) <= TOL_STATE


@pytest.mark.parametrize("in_place", [False, True])
def test_slots_routing_and_untouched_rows(in_place):
    p = workloads.make(seed=51, B=5, lengths=[2, 1, 0, 4, 3], hq=4, hv=8, dk=128, dv=128,
                       act="f16", state="random", num_slots=11, slot_mode="perm")
    ref_o, ref_fin, _ = oracle.run_problem(p)
    o, fin, _ = run(p, in_place=in_place)
    slots = set(int(s) for s in p["slot_ids"])
    fg = fin.cpu()
    init = p["initial_state"]
    for r in range(11):
        if r in slots:
            assert rel_err(fg[r].double().numpy(), ref_fin[r]) <= TOL_STATE
        elif in_place:
            assert torch.equal(fg[r], init[r])  # untouched, bit for bit
        else:
            assert torch.isnan(fg[r]).all()  # never written
    # the empty request (b=2) copies its incoming state through bit-exactly
    s2 = int(p["slot_ids"][2])
    assert torch.equal(fg[s2], init[s2])
    _ = ref_o


def test_clamped_and_decreasing_cu_seqlens():
    T = 12
    p = workloads.make(seed=52, B=4, T=T, cu_seqlens=[-3, 5, 5, 40, 2], hq=1, hv=2, dk=64, dv=64,
                       act="f32", state="random")
    ref_o, ref_fin, _ = oracle.run_problem(p)
    o, fin, _ = run(p)
    _check(p, o, fin, ref_o, ref_fin)


def test_uncovered_tokens_keep_sentinel():
    p = workloads.make(seed=53, B=2, T=20, cu_seqlens=[3, 9, 14], hq=1, hv=1, dk=128, dv=128,
                       act="f16", state="random")
    ref_o, ref_fin, _ = oracle.run_problem(p)
    o, fin, _ = run(p)
    og = o_flat(o, p)
    assert np.isnan(og[:3]).all() and np.isnan(og[14:]).all()
    _check(p, o, fin, ref_o, ref_fin)


def test_zero_initial_state_and_uniform_packing():
    p = workloads.make(seed=54, B=3, T=15, hq=2, hv=2, dk=64, dv=64, act="f16")
    assert p["cu_seqlens"] is None
    ref_o, ref_fin, _ = oracle.run_problem(p)
    o, fin, _ = run(p)
    _check(p, o, fin, ref_o, ref_fin)


def test_rank4_layout():
    p = workloads.make(seed=55, B=2, seq_len=9, hq=2, hv=4, dk=128, dv=128, act="f16",
                       rule="gated_delta", state="random")
    ref_o, ref_fin, _ = oracle.run_problem(p)
    o, fin, _ = run(p)
    _check(p, o, fin, ref_o, ref_fin)


def test_long_request_many_token_blocks():
    p = workloads.make(seed=56, B=2, lengths=[300, 77], hq=1, hv=2, dk=128, dv=128, act="f16",
                       state="random")
    ref_o, ref_fin, _ = oracle.run_problem(p)
    o, fin, _ = run(p)
    _check(p, o, fin, ref_o, ref_fin)


def test_bad_slot_sets_error_word_and_skips():
    p = workloads.make(seed=57, B=3, lengths=[2, 2, 2], hq=1, hv=2, dk=128, dv=128, act="f16",
                       state="random", num_slots=4)
    p["slot_ids"] = torch.tensor([1, 9, -2], dtype=torch.int32)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, fin, _ = run(p, error_word=err)
    assert int(err.item()) & 1
    og = o_flat(o, p)
    assert np.isnan(og[2:]).all() and not np.isnan(og[:2]).any()
    fg = fin.cpu()
    for r in (0, 2, 3):
        assert torch.equal(fg[r], p["initial_state"][r])
    ref_o, ref_fin, rerr = oracle.run_problem(p)
    assert rerr == oracle.ERR_BAD_SLOT
    assert rel_err(fg[1].double().numpy(), ref_fin[1]) <= TOL_STATE


def test_deterministic_run_twice():
    p = workloads.make(seed=58, B=4, lengths=[4, 4, 4, 4], hq=2, hv=4, dk=128, dv=128, act="f16",
                       state="random")
    o1, f1, d = run(p)
    o2, f2, _ = run(p, d=d)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


def test_tiny_fp32_workload():
    p = workloads.tiny_gated_delta()
    ref_o, ref_fin, _ = oracle.run_problem(p)
    o, fin, _ = run(p)
    _check(p, o, fin, ref_o, ref_fin)


@pytest.mark.parametrize("kmajor", [False, True], ids=["vmajor", "kmajor"])
@pytest.mark.parametrize("L", [1, 4])
def test_decode_full_size(L, kmajor):
    """256 requests x 32 heads, dk = dv = 128, slab [1024, 32, 128, 128] in place,
    in the launch configuration the benchmark times: every request against the
    oracle, every untouched slab row bit for bit.  kmajor: the same slab
    stored key-major ([1024, 32, dk, dv], "gatedDeltaUpdate")."""
    p = workloads.decode(L)
    if kmajor:
        p = dict(p, state_kmajor=True,
                 initial_state=p["initial_state"].transpose(2, 3).contiguous())
    o, fin, d = run(p)
    torch.cuda.synchronize()
    # every request, its state row gathered into a compact slab (row j = request j)
    ref_o, ref_fin, err = oracle.run_problem(p, requests=range(p["batch"]), threads=16)
    assert err == 0
    og = o_flat(o, p)
    assert not np.isnan(og).any()
    assert rel_err(og, ref_o) <= TOL_O["f16"]
    slots = p["slot_ids"]
    rows = torch.as_tensor([int(x) for x in slots])
    fg = fin[rows.to(DEV)].double().cpu().numpy()
    assert rel_err(fg, ref_fin) <= TOL_STATE
    touched = set(int(x) for x in slots)
    untouched = torch.as_tensor([r for r in range(1024) if r not in touched])
    assert torch.equal(fin[untouched.to(DEV)].cpu(), p["initial_state"][untouched])


LONG_CASES = []
for rule in ["linear", "gated", "delta", "gated_delta", "gdn2"]:
    LONG_CASES.append(dict(rule=rule, act="f16", dk=128, dv=128, hq=1, hv=2))
LONG_CASES += [
    dict(rule="gated_delta", act="f32", dk=64, dv=64, hq=2, hv=4),
    dict(rule="gated_delta", act="f16", dk=128, dv=96, hq=1, hv=2, decay_per_key=True),
    dict(rule="gdn2", act="f16", dk=128, dv=128, hq=1, hv=1, decay_per_key=True, write_gate=True,
         gate_dtype="f32"),
    dict(rule="gdn2", act="f32", dk=32, dv=32, hq=1, hv=2, decay_per_key=True),
]


@pytest.mark.parametrize("case", LONG_CASES, ids=[_case_id(c) for c in LONG_CASES])
def test_recurrent_long_requests(case):
    """Requests averaging more than 32 tokens take the one-CTA-per-slice
    schedule with prefetched token blocks."""
    kw = dict(seed=zlib.crc32(_case_id(case).encode()) % 1000, B=3, lengths=[150, 0, 67],
              state="random", state_std=0.5, num_slots=5, slot_mode="perm")
    kw.update(case)
    p = workloads.make(**kw)
    ref_o, ref_fin, err = oracle.run_problem(p)
    assert err == 0
    o, fin, _ = run(p)
    _check(p, o, fin, ref_o, ref_fin)


@pytest.mark.parametrize("case", [
    dict(seq_len=4, seq_lens=[4, 1, 0, 3, 7], dk=128, dv=128),   # decode kernel
    dict(seq_len=150, seq_lens=[150, 0, 37, 400, 1], dk=128, dv=128),  # long-request kernel
    dict(seq_len=9, seq_lens=[2, 9, 0, 5, -3], dk=48, dv=24),     # any-dk kernel
], ids=["decode", "long", "generic"])
def test_seq_lens_padded_rows(case):
    """Rank-4 batch whose rows are bounded by seq_lens ("gatedDeltaUpdate"):
    each request takes the first clamp(seq_lens[b], 0, S) tokens of its row;
    padding tokens keep the sentinel; slots in place."""
    p = workloads.make(seed=43, B=5, hq=2, hv=4, act="f16", rule="gated_delta", state="random",
                       num_slots=8, slot_mode="perm", **case)
    p = poison_uncovered(p)  # NaN in every padding token
    ref_o, ref_fin, err = oracle.run_problem(p)
    assert err == 0
    o, fin, _ = run(p)
    _check(p, o, fin, ref_o, ref_fin)


@pytest.mark.parametrize("case", [
    dict(lengths=[1, 4, 0, 2], dk=128, dv=128),        # decode kernel
    dict(lengths=[120, 3, 77], dk=128, dv=128),        # long-request kernel
    dict(lengths=[3, 0, 5], dk=48, dv=24),             # any-dk kernel
], ids=["decode", "long", "generic"])
@pytest.mark.parametrize("rule", ["delta", "gated_delta"])
def test_shared_beta(case, rule):
    """beta [T]: one per token, broadcast over the value heads."""
    p = workloads.make(seed=44, B=len(case["lengths"]), hq=2, hv=4, act="f16", rule=rule,
                       state="random", beta_shared=True, **case)
    ref_o, ref_fin, err = oracle.run_problem(p)
    assert err == 0
    o, fin, _ = run(p)
    _check(p, o, fin, ref_o, ref_fin)

"""GPU parity of gdn_chunked_prefill against the CPU oracle, through the C ABI.

The chunked path multiplies fp16 operands on the tensor cores with fp32
accumulation and keeps the state in fp32, so outputs and final states are
held to 5e-3 of their max-norm (relative: max |x - ref| / max |ref|).
"""
import os
import zlib

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import DEV, o_flat, poison_uncovered, rel_err, run, to_dev

pytestmark = pytest.mark.gpu

TOL = 5e-3
THREADS = max(1, min(16, os.cpu_count() or 1))


def _check(p, o, fin, ref_o, ref_fin, rows=None):
    og = o_flat(o, p)
    covered = ~np.isnan(ref_o)
    assert np.isnan(og[~covered]).all()
    e_o = rel_err(og[covered], ref_o[covered])
    fg = fin.double().cpu().numpy()
    if rows is not None:
        fg = fg[rows]
    e_s = rel_err(fg, ref_fin)
    assert e_o <= TOL and e_s <= TOL, (e_o, e_s)
    return e_o, e_s


CASES = []
for rule in ["linear", "gated", "delta", "gated_delta", "gdn2"]:
    for act in ["f16", "f32"]:
        CASES.append(dict(rule=rule, act=act, dk=128, dv=128, hq=1, hv=2))
for dk, dv in [(16, 16), (32, 48), (64, 64), (64, 128), (128, 64), (128, 80)]:
    CASES.append(dict(rule="gated_delta", act="f16", dk=dk, dv=dv, hq=2, hv=4))
CASES += [
    dict(rule="gated_delta", act="f16", dk=128, dv=128, hq=2, hv=2, gate="log",
         logdecay_range=(-4.0, 0.0)),
    dict(rule="gated_delta", act="f16", dk=128, dv=128, hq=1, hv=1, beta_mode="direct",
         l2norm_q=True),
    dict(rule="gated_delta", act="f16", dk=64, dv=64, hq=1, hv=2, decay_per_key=True),
    dict(rule="gdn2", act="f16", dk=64, dv=64, hq=1, hv=1, decay_per_key=True, write_gate=True),
    # per-key decay on the tensor-core path (fp32 per-key gates, dk = dv = 128)
    dict(rule="gated_delta", act="f16", dk=128, dv=128, hq=1, hv=2, decay_per_key=True, gate_dtype="f32"),
    dict(rule="gdn2", act="f16", dk=128, dv=128, hq=2, hv=4, decay_per_key=True, gate_dtype="f32",
         write_gate=True),
    dict(rule="gdn2", act="f16", dk=128, dv=128, hq=1, hv=2, decay_per_key=True, gate="log",
         logdecay_range=(-6.0, 0.0), beta_mode="direct", l2norm_q=True),
    dict(rule="gated_delta", act="f16", dk=128, dv=128, hq=1, hv=2, decay_per_key=True, gate="log",
         logdecay_range=(-3.0, 0.0), l2norm_q=True),
    # the gated rule with per-key decay (no retrieval) on the per-key prepare pass
    dict(rule="gated", act="f16", dk=128, dv=128, hq=1, hv=1, decay_per_key=True, gate_dtype="f32"),
    dict(rule="gated", act="f16", dk=128, dv=128, hq=2, hv=4, decay_per_key=True, gate="log",
         logdecay_range=(-6.0, 0.0), l2norm_q=True),
    dict(rule="gated", act="f32", dk=128, dv=128, hq=1, hv=2, decay_per_key=True, gate_dtype="f32"),
    # per-key gates in fp16: the same path on fp32 copies of the gate rows
    dict(rule="gated_delta", act="f16", dk=128, dv=128, hq=1, hv=1, decay_per_key=True),
    dict(rule="gated", act="f16", dk=128, dv=128, hq=1, hv=1, decay_per_key=True),
    dict(rule="gdn2", act="f16", dk=128, dv=128, hq=1, hv=2, decay_per_key=True, write_gate=True),
    # per-key decay at other head sizes: the token-serial kernel
    dict(rule="gated", act="f16", dk=64, dv=64, hq=1, hv=1, decay_per_key=True),
]


def _cid(c):
    return "-".join("%s=%s" % (k, v) for k, v in sorted(c.items()))


@pytest.mark.parametrize("case", CASES, ids=[_cid(c) for c in CASES])
def test_chunked_parity_sweep(case):
    kw = dict(seed=zlib.crc32(_cid(case).encode()) % 1000, B=5, lengths=[70, 0, 130, 1, 64],
              state="random", state_std=0.3)
    kw.update(case)
    p = workloads.make(**kw)
    ref_o, ref_fin, err = oracle.run_problem(p)
    assert err == 0
    o, fin, _ = run(p, path="chunked")
    _check(p, o, fin, ref_o, ref_fin)


@pytest.mark.parametrize("chunk", [0, 16, 32, 64, 100, 1024])
def test_chunk_size_hint_never_changes_result(chunk):
    p = workloads.make(seed=71, B=2, lengths=[150, 77], hq=1, hv=2, dk=128, dv=128, act="f16",
                       state="random")
    o_ref, f_ref, d = run(p, path="chunked", chunk=64)
    o, f, _ = run(p, path="chunked", chunk=chunk, d=d)
    assert torch.equal(o.nan_to_num(7.0), o_ref.nan_to_num(7.0)) and torch.equal(f, f_ref)


@pytest.mark.parametrize("rule", ["linear", "gated", "delta", "gated_delta"])
def test_chunked_matches_recurrent(rule):
    p = workloads.make(seed=72, B=3, lengths=[200, 65, 9], hq=2, hv=4, dk=128, dv=128, act="f16",
                       rule=rule, state="random")
    o1, f1, d = run(p, path="chunked")
    o2, f2, _ = run(p, path="recurrent", d=d)
    assert rel_err(o_flat(o1, p), o_flat(o2, p)) <= TOL
    assert rel_err(f1.double().cpu().numpy(), f2.double().cpu().numpy()) <= TOL


def test_split_resume_through_state():
    p = workloads.make(seed=73, B=1, lengths=[300], hq=1, hv=2, dk=128, dv=128, act="f16",
                       state="random")
    o_all, f_all, d = run(p, path="chunked")
    a = dict(p, total_tokens=130, cu_seqlens=torch.tensor([0, 130], dtype=torch.int32))
    for key in ("q", "k", "v", "decay", "beta"):
        a[key] = p[key][:130]
    oa, fa, _ = run(a, path="chunked")
    bpart = dict(p, total_tokens=170, cu_seqlens=torch.tensor([0, 170], dtype=torch.int32),
                 initial_state=fa.cpu())
    for key in ("q", "k", "v", "decay", "beta"):
        bpart[key] = p[key][130:]
    ob, fb, _ = run(bpart, path="chunked")
    cat = torch.cat([oa, ob], 0)
    assert rel_err(cat.double().cpu().numpy(), o_all.double().cpu().numpy()) <= TOL
    assert rel_err(fb.double().cpu().numpy(), f_all.double().cpu().numpy()) <= TOL


def test_chunked_slots_and_empty_requests():
    p = workloads.make(seed=74, B=4, lengths=[90, 0, 40, 3], hq=2, hv=4, dk=128, dv=128, act="f16",
                       state="random", num_slots=9, slot_mode="perm")
    ref_o, ref_fin, _ = oracle.run_problem(p)
    o, fin, _ = run(p, path="chunked")
    _check(p, o, fin, ref_o, ref_fin)
    s1 = int(p["slot_ids"][1])
    assert torch.equal(fin[s1].cpu(), p["initial_state"][s1])
    touched = set(int(s) for s in p["slot_ids"])
    for r in range(9):
        if r not in touched:
            assert torch.equal(fin[r].cpu(), p["initial_state"][r])


def test_chunked_uncovered_tokens_and_clamping():
    # -4 clamps to 0, 300 to 200; the decreasing pair (300, 20) gives an empty
    # request.  (Decreasing entries that make clamped requests overlap are
    # left out: the pages do not say which request's output wins.)
    p = workloads.make(seed=75, B=4, T=200, cu_seqlens=[-4, 70, 70, 300, 20], hq=1, hv=2, dk=64,
                       dv=64, act="f16", state="random")
    ref_o, ref_fin, _ = oracle.run_problem(p)
    o, fin, _ = run(p, path="chunked")
    _check(p, o, fin, ref_o, ref_fin)
    assert torch.equal(fin[1].cpu(), p["initial_state"][1])
    assert torch.equal(fin[3].cpu(), p["initial_state"][3])


def test_chunked_bad_slot_sets_error_word():
    p = workloads.make(seed=76, B=2, lengths=[10, 10], hq=1, hv=2, dk=128, dv=128, act="f16",
                       state="random", num_slots=3)
    p["slot_ids"] = torch.tensor([2, 3], dtype=torch.int32)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, fin, _ = run(p, path="chunked", error_word=err)
    assert int(err.item()) & 1
    assert np.isnan(o_flat(o, p)[10:]).all()


def test_chunked_overlapping_requests_outgrow_the_workspace():
    """cu_seqlens [0, 640, 0, 640, 0, 640]: requests 0, 2 and 4 each cover all
    640 tokens (10 chunks), more than the T / 64 + B + 1 = 16 workspace slots
    that disjoint requests can need.  Request 0 runs; 2 and 4 are skipped
    with GDN_DEVERR_OVERLAP (0x4), their state rows left unwritten."""
    p = workloads.make(seed=78, B=5, T=640, cu_seqlens=[0, 640, 0, 640, 0, 640], hq=1, hv=1,
                       dk=128, dv=128, act="f16", state="random")
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, fin, _ = run(p, path="chunked", error_word=err)
    assert int(err.item()) & 4
    ref_o, ref_fin, _ = oracle.run_problem(p, requests=[0])
    assert rel_err(o_flat(o, p), ref_o) <= TOL
    fg = fin.double().cpu().numpy()
    assert rel_err(fg[[0]], ref_fin) <= TOL
    assert np.isnan(fg[2]).all() and np.isnan(fg[4]).all()
    for b in (1, 3):  # empty requests pass their state through
        assert torch.equal(fin[b].cpu(), p["initial_state"][b])


def test_chunked_tiny_fp32_workload():
    p = workloads.tiny_gated_delta()
    ref_o, ref_fin, _ = oracle.run_problem(p)
    o, fin, _ = run(p, path="chunked")
    _check(p, o, fin, ref_o, ref_fin)


def test_chunked_deterministic():
    p = workloads.make(seed=77, B=2, lengths=[100, 50], hq=1, hv=2, dk=128, dv=128, act="f16",
                       state="random")
    o1, f1, d = run(p, path="chunked")
    o2, f2, _ = run(p, path="chunked", d=d)
    assert torch.equal(o1.nan_to_num(3.0), o2.nan_to_num(3.0)) and torch.equal(f1, f2)


# ---------------------------------------------------------------- full sizes
def _full(p):
    """Runs a full-size workload in the launch configuration the benchmark
    times and checks every request (all tokens, all heads, every state row)
    against the oracle."""
    o, fin, d = run(p, path="chunked")
    torch.cuda.synchronize()
    ref_o, ref_fin, err = oracle.run_problem(p, threads=THREADS)
    assert err == 0
    og = o_flat(o, p)
    covered = ~np.isnan(ref_o)
    assert covered.all()
    e_o = rel_err(og, ref_o)
    e_s = rel_err(fin.double().cpu().numpy(), ref_fin)
    assert e_o <= TOL and e_s <= TOL, (e_o, e_s)
    assert not np.isnan(og).any()


def test_ragged_prefill_full_size():
    """8 ragged requests, 16384 tokens, Hv = 32: every request, including the
    middle ones whose chains the offsets kernel reorders (longest first)."""
    _full(workloads.ragged_prefill())


@pytest.mark.parametrize("rule", ["linear", "gated", "delta", "gated_delta"])
def test_long_prefill_full_size(rule):
    """B = 4, S = 8192, H = 16, rank-4: all four sequences."""
    _full(workloads.long_prefill(rule))


def test_gdn2_full_size():
    """GDN-2 extension, B = 2, S = 4096, H = 16, per-key decay and erase gate,
    write gate folded into v: both sequences."""
    _full(workloads.gdn2())


def test_gdn2_full_size_gates_as_inputs():
    """The same workload with the erase gate as its own input beside a scalar
    beta (GDN-2 issue, proposal B) and the write gate passed to the op rather
    than folded into v."""
    _full(workloads.gdn2(erase="input", write_gate="input"))


def test_gated_per_key_long():
    """The gated rule with decay per key channel (no retrieval) on the per-key
    prepare pass: B = 2, S = 4096, H = 16 with the GDN-2 workload's gate
    distribution, random incoming state; both sequences."""
    _full(workloads.gated_perkey(state="random"))


@pytest.mark.parametrize("rule,per_key", [("linear", False), ("gated", False), ("delta", False),
                                          ("gated_delta", False), ("gdn2", True), ("gated", True)])
def test_chunked_many_chains(rule, per_key):
    """160 (request, head) chains, more than the GPU has SMs: the chain kernel
    keeps one CTA per chain (fewer chains are split over two CTAs by value
    rows, which the other parity cases cover)."""
    kw = dict(seed=31, B=10, lengths=[70, 1, 64, 130, 5, 65, 0, 127, 33, 64], hq=8, hv=16, dk=128, dv=128,
              act="f16", rule=rule, state="random", state_std=0.3)
    if per_key:
        kw.update(decay_per_key=True, gate_dtype="f32", write_gate=rule == "gdn2")
    p = workloads.make(**kw)
    ref_o, ref_fin, err = oracle.run_problem(p)
    assert err == 0
    o, fin, _ = run(p, path="chunked")
    _check(p, o, fin, ref_o, ref_fin)


@pytest.mark.parametrize("case", [
    dict(rule="gated_delta"),
    dict(rule="linear"),
    dict(rule="gdn2", decay_per_key=True, gate_dtype="f32", write_gate=True),
    dict(rule="gated_delta", dk=64, dv=64),
    dict(rule="gated", decay_per_key=True, gate_dtype="f32"),
    dict(rule="gated", decay_per_key=True),
    dict(rule="gated", decay_per_key=True, dk=64, dv=64),
], ids=["tc-gated_delta", "tc-linear", "tc-perkey-gdn2", "mma", "tc-perkey-gated", "tc-perkey-f16-gates",
        "token-serial"])
def test_chunked_seq_lens_padded_rows(case):
    """Rank-4 batch whose rows are bounded by seq_lens ("gatedDeltaUpdate"):
    request b takes the first clamp(seq_lens[b], 0, S) tokens of its row, over
    every chunked path; padding tokens keep the sentinel."""
    kw = dict(seed=41, B=4, seq_len=100, seq_lens=[100, 0, 37, 250], hq=1, hv=2, dk=128, dv=128,
              act="f16", state="random", state_std=0.3)
    kw.update(case)
    p = poison_uncovered(workloads.make(**kw))  # NaN in every padding token
    ref_o, ref_fin, err = oracle.run_problem(p)
    assert err == 0
    o, fin, _ = run(p, path="chunked")
    _check(p, o, fin, ref_o, ref_fin)


@pytest.mark.parametrize("case", [dict(), dict(dk=64, dv=64),
                                  dict(decay_per_key=True, gate_dtype="f32")],
                         ids=["tc", "mma", "tc-perkey"])
@pytest.mark.parametrize("rule", ["delta", "gated_delta"])
def test_chunked_shared_beta(case, rule):
    """beta [T]: one per token, broadcast over the value heads, on every
    chunked path."""
    if rule == "delta" and case.get("decay_per_key"):
        pytest.skip("the delta rule has no decay")
    kw = dict(seed=45, B=3, lengths=[70, 0, 130], hq=1, hv=2, dk=128, dv=128, act="f16", rule=rule,
              state="random", state_std=0.3, beta_shared=True)
    kw.update(case)
    p = workloads.make(**kw)
    ref_o, ref_fin, err = oracle.run_problem(p)
    assert err == 0
    o, fin, _ = run(p, path="chunked")
    _check(p, o, fin, ref_o, ref_fin)


@pytest.mark.parametrize("case", [dict(rule="linear"), dict(rule="gated"), dict(rule="gated_delta"),
                                  dict(rule="gdn2", decay_per_key=True, gate_dtype="f32", write_gate=True),
                                  dict(rule="gated", dk=64, dv=64), dict(rule="gated_delta", act="f32"),
                                  dict(rule="gdn2", act="f32", decay_per_key=True, gate_dtype="f32"),
                                  dict(rule="gated", decay_per_key=True, gate_dtype="f32")],
                         ids=["tc-linear", "tc-gated", "tc-gated_delta", "tc-perkey-gdn2", "mma-gated",
                              "tc-f32-gated_delta", "tc-f32-perkey-gdn2", "tc-perkey-gated"])
def test_chunked_ignores_uncovered_tokens(case):
    """Tokens outside every request (before the first, between clamped
    requests, after the last) hold NaN in q, k, v and the gates: outputs and
    states match the oracle, and uncovered outputs keep the sentinel."""
    kw = dict(seed=46, B=3, T=260, cu_seqlens=[3, 70, 70, 200], hq=1, hv=2, dk=128, dv=128, act="f16",
              state="random", state_std=0.3)
    kw.update(case)
    p = poison_uncovered(workloads.make(**kw))
    ref_o, ref_fin, err = oracle.run_problem(p)
    assert err == 0
    o, fin, _ = run(p, path="chunked")
    _check(p, o, fin, ref_o, ref_fin)


@pytest.mark.parametrize("dk", [16, 128])
def test_chunked_widest_value_heads(dk):
    """dv = 256, the widest value head the chunked entry point takes (the
    warp-level MMA kernel), over several chunks and a ragged tail."""
    p = workloads.make(seed=51 + dk, B=3, lengths=[130, 0, 67], hq=1, hv=2, dk=dk, dv=256, act="f16",
                       rule="gated_delta", state="random", state_std=0.3)
    ref_o, ref_fin, err = oracle.run_problem(p, threads=THREADS)
    assert err == 0
    o, fin, _ = run(p, path="chunked")
    _check(p, o, fin, ref_o, ref_fin)


def test_chunked_more_requests_than_the_order_sort_takes():
    """2100 requests, past the 2048 the offsets kernel sorts longest first (it
    keeps index order above that): lengths 0..96 tokens, so the workspace holds
    T / 64 + B + 1 slots and every chain runs on its own CTA."""
    g = torch.Generator().manual_seed(52)
    lengths = torch.randint(0, 97, (2100,), generator=g).tolist()
    p = workloads.make(seed=52, B=len(lengths), lengths=lengths, hq=1, hv=1, dk=128, dv=128, act="f16",
                       rule="gated_delta", state="random", state_std=0.3)
    ref_o, ref_fin, err = oracle.run_problem(p, threads=THREADS)
    assert err == 0
    o, fin, _ = run(p, path="chunked")
    _check(p, o, fin, ref_o, ref_fin)


WINDOWED = [
    dict(rule="gated_delta"),
    dict(rule="linear"),
    dict(rule="gated"),
    dict(rule="delta", beta_shared=True),
    dict(rule="gdn2", decay_per_key=True, gate_dtype="f32", write_gate=True),
    dict(rule="gated", decay_per_key=True, gate_dtype="f32"),
    dict(rule="gated_delta", act="f32"),
    dict(rule="gated_delta", state_kmajor=True, num_slots=8, slot_mode="perm"),
]


@pytest.mark.parametrize("chunks", [1, 2])
@pytest.mark.parametrize("case", WINDOWED, ids=[_cid(c) for c in WINDOWED])
def test_chunked_windowed_workspace(case, chunks):
    """A workspace that holds ``chunks`` chunks of every request: the call runs
    in windows, each reading the fp32 state the last one left in final_state,
    so outputs and final state equal the single pass bit for bit (and the
    oracle within the tolerance).  Requests of 0, 1, 70, 130 and 200 tokens:
    some end in an early window and sit out the later ones."""
    kw = dict(seed=61, B=5, lengths=[70, 0, 130, 1, 200], hq=1, hv=2, dk=128, dv=128, act="f16",
              rule="gated_delta", state="random", state_std=0.3)
    kw.update(case)
    p = workloads.make(**kw)
    o1, f1, _ = run(p, path="chunked")
    per_chunk = p["batch"] * (p["hv"] * 88 * 1024 + 4)
    o2, f2, _ = run(p, path="chunked", workspace_extra=(chunks - 1) * per_chunk)
    torch.cuda.synchronize()
    assert torch.equal(torch.nan_to_num(o1, nan=7.0), torch.nan_to_num(o2, nan=7.0))
    assert torch.equal(torch.nan_to_num(f1, nan=7.0), torch.nan_to_num(f2, nan=7.0))
    ref_o, ref_fin, err = oracle.run_problem(p)
    assert err == 0
    _check(p, o2, f2, ref_o, ref_fin)


def test_ragged_prefill_full_size_windowed():
    """Config 3 (8 requests, 16384 tokens, Hv = 32) with a workspace of 16
    chunks per request (about 365 MB instead of 765 MB): four windows for the
    longest request; every request checked against the oracle."""
    p = workloads.ragged_prefill()
    per_chunk = p["batch"] * (p["hv"] * 88 * 1024 + 4)
    o, fin, _ = run(p, path="chunked", workspace_extra=15 * per_chunk)
    torch.cuda.synchronize()
    ref_o, ref_fin, err = oracle.run_problem(p, threads=THREADS)
    assert err == 0
    _check(p, o, fin, ref_o, ref_fin)


def test_chunked_windowed_seq_lens_rows():
    """Windows over the rank-4 layout with padded seq_lens rows (padding tokens
    NaN): bit-identical to the single pass, padding outputs untouched."""
    kw = dict(seed=62, B=4, seq_len=300, seq_lens=[300, 0, 37, 999], hq=1, hv=2, dk=128, dv=128,
              act="f16", rule="gated_delta", state="random", state_std=0.3)
    p = poison_uncovered(workloads.make(**kw))
    o1, f1, _ = run(p, path="chunked")
    o2, f2, _ = run(p, path="chunked", workspace_extra=0)  # one chunk per request per window
    torch.cuda.synchronize()
    assert torch.equal(torch.nan_to_num(o1, nan=7.0), torch.nan_to_num(o2, nan=7.0))
    assert torch.equal(f1, f2)
    ref_o, ref_fin, err = oracle.run_problem(p)
    assert err == 0
    _check(p, o2, f2, ref_o, ref_fin)

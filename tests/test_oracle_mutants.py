"""Planted mistakes in the oracle: every pin-checked oracle must fail its pins.

Each case copies ``oracle/gdn_oracle.c``, plants one plausible mistake in the
copy (a dropped term, a wrong sign or index, a transposed operand, a skipped
gate), builds it with the oracle's own flags and runs
``tests/test_oracle_pins.py`` against that build (``GDN_ORACLE_LIB``).  The pins
are independent of the oracle's arithmetic (closed forms, dense products,
brute force, the pages' formulas written out), so a mistake anywhere in the
recurrence, the gates or the routing must make at least one of them fail.  A
control build of the unaltered copy must pass them all.  CPU only: nothing
here touches the CUDA library.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gdn_oracle.c")

# (id, text in gdn_oracle.c, its replacement): each a mistake a reader could make
MUTANTS = [
    ("delta-sign", "delta[i] = beta * (vin[i] - u[i]);", "delta[i] = beta * (vin[i] + u[i]);"),
    ("delta-no-beta", "delta[i] = beta * (vin[i] - u[i]);", "delta[i] = vin[i] - u[i];"),
    ("no-readout-scale", "out[i] = scale * s;", "out[i] = s;"),
    ("decay-sign", "alpha[c] = exp(g);", "alpha[c] = exp(-g);"),
    ("grouped-heads-modulo", "(int32_t)((int64_t)h * hq / hv)", "(int32_t)(h % hq)"),
    ("per-key-bias-index", "p->gate_bias[(size_t)h * dk + c]", "p->gate_bias[c]"),
    ("per-head-bias-index", "softplus(raw + p->gate_bias[h])", "softplus(raw + p->gate_bias[0])"),
    ("gdn2-no-erase-sigmoid", "if (p->beta_sigmoid) bc = sigmoid(bc);", ""),
    ("gdn2-erase-gate-ignored", "kappa[c] = bc * kv[c];", "kappa[c] = kv[c];"),
    ("gdn2-write-gate-ignored",
     "const real w = p->write_gate ? p->write_gate[((size_t)t * hv + h) * dv + i] : 1.0;",
     "const real w = 1.0;"),
    ("gdn2-option-b-no-beta", "delta[i] = beta * (w * vin[i]) - u[i];", "delta[i] = (w * vin[i]) - u[i];"),
    ("write-with-query", "M[(size_t)i * dk + c] += delta[i] * kv[c];", "M[(size_t)i * dk + c] += delta[i] * qv[c];"),
    ("readout-with-key", "s += M[(size_t)i * dk + c] * qv[c];", "s += M[(size_t)i * dk + c] * kv[c];"),
    ("l2norm-no-sqrt", "real inv = 1.0 / sqrt(ss + 1e-12);", "real inv = 1.0 / (ss + 1e-12);"),
    ("kmajor-load-untransposed", "p->initial_state[state_off + (size_t)c * dv + i]",
     "p->initial_state[state_off + (size_t)i * dk + c]"),
    ("kmajor-store-untransposed", "p->final_state[state_off + (size_t)c * dv + i] = M[(size_t)i * dk + c];",
     "p->final_state[state_off + (size_t)i * dk + c] = M[(size_t)i * dk + c];"),
    ("seq-lens-ignored", "(p->seq_lens ? clamp_i32(p->seq_lens[b], 0, len) : len)", "len"),
    ("slots-ignored", "const int32_t row = p->slot_ids ? p->slot_ids[b] : b;", "const int32_t row = b;"),
    ("softplus-sign", "x + log1p(exp(-x))", "x - log1p(exp(-x))"),
    ("sigmoid-sign", "1.0 / (1.0 + exp(-x))", "1.0 / (1.0 + exp(x))"),
    ("gate-op-bias-sign", "softplus(a[e] + dt_bias[j])", "softplus(a[e] - dt_bias[j])"),
    ("beta-head-ignored",
     "real beta = p->beta[p->beta_shared ? (size_t)t : (size_t)t * hv + h];\n"
     "            if (p->beta_sigmoid) beta = sigmoid(beta);\n            memcpy",
     "real beta = p->beta[p->beta_shared ? (size_t)t : (size_t)t * hv];\n"
     "            if (p->beta_sigmoid) beta = sigmoid(beta);\n            memcpy"),
    ("default-scale-no-sqrt", "1.0 / sqrt((real)dk)", "1.0 / (real)dk"),
    ("query-norm-ignored", "if (p->l2norm_q) l2_normalise(qv, dk);", ""),
    ("per-key-decay-one-channel", "real raw = p->decay[((size_t)t * hv + h) * dk + c];",
     "real raw = p->decay[((size_t)t * hv + h) * dk];"),
    ("bad-slot-not-flagged", "*p->error_word |= ORACLE_ERR_BAD_SLOT;", "*p->error_word |= 0;"),
    ("beta-no-sigmoid",
     "real beta = p->beta[p->beta_shared ? (size_t)t : (size_t)t * hv + h];\n"
     "            if (p->beta_sigmoid) beta = sigmoid(beta);\n            memcpy",
     "real beta = p->beta[p->beta_shared ? (size_t)t : (size_t)t * hv + h];\n            memcpy"),
]

_DECAY = ("            for (int32_t i = 0; i < dv; ++i)\n"
          "                for (int32_t c = 0; c < dk; ++c) M[(size_t)i * dk + c] *= alpha[c];\n        }")
_WRITE = ("        for (int32_t i = 0; i < dv; ++i)\n"
          "            for (int32_t c = 0; c < dk; ++c) M[(size_t)i * dk + c] += delta[i] * kv[c];\n")
_READ = ("        real *out = p->o + ((size_t)t * hv + h) * dv;\n"
         "        for (int32_t i = 0; i < dv; ++i) {\n"
         "            real s = 0.0;\n"
         "            for (int32_t c = 0; c < dk; ++c) s += M[(size_t)i * dk + c] * qv[c];\n"
         "            out[i] = scale * s;\n"
         "        }\n")
# mistakes in the order of the steps: several edits each
MUTANTS_MULTI = [
    # the decay applied after the write (so the retrieval reads the undecayed state)
    ("decay-after-write", [(_DECAY, "        }"),
                           (_WRITE, _WRITE + "        if (rule_has_decay(p->rule))\n"
                                             "            for (int32_t i = 0; i < dv; ++i)\n"
                                             "                for (int32_t c = 0; c < dk; ++c)"
                                             " M[(size_t)i * dk + c] *= alpha[c];\n")]),
    # the readout taken from the state before this token's write
    ("readout-before-write", [(_WRITE + "\n" + _READ, _READ + _WRITE)]),
]


def _build(src_text, out_dir, name):
    if shutil.which("gcc") is None:
        pytest.skip("gcc is not available")
    c = os.path.join(out_dir, name + ".c")
    so = os.path.join(out_dir, "lib" + name + ".so")
    with open(c, "w") as fh:
        fh.write(src_text)
    # the flags of oracle/build.py (double build)
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-o", so, c, "-lm"],
                   check=True, capture_output=True)
    return so


def _run_pins(lib):
    env = dict(os.environ, GDN_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu",
                        # that test compares the double build with the unaltered float build,
                        # not with something independent of the oracle: it is no pin here
                        "-k", "not float_instantiation"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-1500:]


def test_every_planted_mistake_fails_a_pin(tmp_path):
    with open(SRC) as fh:
        text = fh.read()
    libs = {"control": _build(text, str(tmp_path), "control")}
    cases = [(name, [(old, new)]) for name, old, new in MUTANTS] + MUTANTS_MULTI
    for name, edits in cases:
        altered = text
        for old, new in edits:
            assert altered.count(old) == 1, "the text to alter must occur exactly once: " + name
            altered = altered.replace(old, new)
        libs[name] = _build(altered, str(tmp_path), name.replace("-", "_"))
    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        results = dict(zip(libs, ex.map(_run_pins, libs.values())))
    rc, out = results.pop("control")
    assert rc == 0, "the unaltered copy must pass every pin:\n" + out
    # exit code 1: a pin's assertion failed (not a crash or a collection error)
    survivors = {n: (rc, out) for n, (rc, out) in results.items() if rc != 1}
    assert not survivors, "planted mistakes no pin caught (or that broke the run): %s" % {
        n: (rc, out[-400:]) for n, (rc, out) in survivors.items()}

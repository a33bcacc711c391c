"""The pages' example calls (shapes only; the pages print no values)."""
import json
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_examples.json")


def _load():
    with open(GOLDEN) as f:
        return json.load(f)


def test_gated_delta_net_example_shapes():
    ex = _load()["gated_delta_net_example"]
    rng = np.random.default_rng(31)
    q = rng.standard_normal(ex["query"])
    k = rng.standard_normal(ex["key"])
    v = rng.standard_normal(ex["value"])
    o, fin, err = oracle.gdn(q, k, v, rule="gated_delta", decay=-rng.random(ex["decay"]),
                             beta=rng.random(ex["beta"]),
                             initial_state=rng.standard_normal(ex["initial_state"]),
                             l2norm_q=True, l2norm_k=True)
    assert list(o.shape) == ex["expected_output"]
    assert list(fin.shape) == ex["expected_final_state"]
    assert err == 0 and np.isfinite(o).all()


def test_linear_attention_gate_example_shapes():
    ex = _load()["linear_attention_gate_example"]
    rng = np.random.default_rng(32)
    d = oracle.gate(rng.standard_normal(ex["a"]), rng.standard_normal(ex["dt_bias"]),
                    -np.exp(rng.random(ex["decay_scale"])))
    assert list(d.shape) == ex["expected_decay"] and (d < 0).all()

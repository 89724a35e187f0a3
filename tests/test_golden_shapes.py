"""The oracle against the shape contracts printed on the pages
(tests/golden/shape_contracts.json, each entry cites its page and section)."""
import json
import os

import numpy as np

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden", "shape_contracts.json")


def _cases():
    with open(GOLD) as f:
        return {c["name"]: c for c in json.load(f)["cases"]}


def test_column_and_row_shapes():
    c = _cases()
    S, B, H, O = 6, 2, 16, 32
    p = c["column_output"]["p"]
    X = np.ones((S * B, H))
    W = np.ones((O, H))
    pre, A = oracle.column_fwd(X, oracle.shard_column_weight(W, p), None, "none")
    assert len(pre) == p and all(a.reshape(S, B, -1).shape == (S, B, O // p) for a in A)
    p = c["row_output"]["p"]
    I = 32
    Xs = [np.ones((S * B, I // p))] * p
    Ws = oracle.shard_row_weight(np.ones((O, I)), p)
    Y = oracle.row_fwd(Xs, Ws)
    assert Y.reshape(S, B, -1).shape == (S, B, O)


def test_sequence_parallel_shape():
    c = _cases()["sequence_parallel_shard"]
    S, B, H = 8, 2, 4
    shards = oracle.sp_split(np.zeros((S * B, H)), c["p"])
    assert all(s.reshape(-1, B, H).shape == (S // 4, B, H) for s in shards)


def test_mlp_pairing_widths():
    c = _cases()["mlp_pairing"]
    d, T = 16, c["p"]
    W1s = oracle.shard_column_weight(np.zeros((4 * d, d)), T)
    W2s = oracle.shard_row_weight(np.zeros((d, 4 * d)), T)
    assert all(w.shape == (4 * d // T, d) for w in W1s)
    assert all(w.shape == (d, 4 * d // T) for w in W2s)
    _, _, Y = oracle.mlp_fwd(np.zeros((3, d)), W1s, None, W2s, None, "gelu_tanh", False)
    assert Y.shape == (3, d)


def test_divide_example():
    c = _cases()["divide"]
    assert oracle.divide(c["output_size"], c["world_size"]) == c["per_partition"]
    W1s = oracle.shard_column_weight(np.zeros((c["output_size"], 8)), c["world_size"])
    assert W1s[0].shape == (c["per_partition"], 8)

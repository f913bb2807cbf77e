"""Pins of the oracle against the hand-worked examples in tests/golden/ (CPU only)."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _hex(s):
    return int(s, 16)


def _worked_inputs(g):
    c = g["config"]
    H = c["hidden"]
    ids = [np.array(r, np.int32).reshape(-1, c["top_k"]) for r in g["topk_ids"]]
    # Hidden rows: distinct bytes per token so a misplaced row shows.
    hidden = [np.arange(n * H * 2, dtype=np.uint16).astype(np.uint8).reshape(n, 2 * H) + 100 * s
              for s, n in enumerate(g["num_tokens"])]
    return c, ids, hidden


@pytest.mark.parametrize("masked", [False, True])
def test_worked_example_recv_ids(masked):
    g = _load("worked_example.json")
    c, ids, hidden = _worked_inputs(g)
    mask = 0b01 if masked else 0b11
    out = oracle.dispatch(c["ep_size"], c["num_experts"], c["top_k"], c["tokens_per_rank"],
                          g["num_tokens"], hidden, ids, mask_enabled=masked, active_rank_mask=mask)
    exp = g["expected_recv_ids_mask_rank0_only" if masked else "expected_recv_ids"]
    for d in range(c["ep_size"]):
        assert out.recv_ids[d].tolist() == exp[f"dest{d}"]


def test_worked_example_payload_rows():
    g = _load("worked_example.json")
    c, ids, hidden = _worked_inputs(g)
    T = c["tokens_per_rank"]
    out = oracle.dispatch(c["ep_size"], c["num_experts"], c["top_k"], T, g["num_tokens"], hidden, ids)
    exp = g["expected_recv_ids"]
    for d in range(c["ep_size"]):
        for r, row in enumerate(exp[f"dest{d}"]):
            s, t = divmod(r, T)
            if row[0] == -1:
                assert (out.recv_hidden[d][r] == oracle.SENTINEL_BYTE).all()
            else:
                np.testing.assert_array_equal(out.recv_hidden[d][r], hidden[s][t])


def test_worked_example_combine_cases():
    g = _load("worked_example.json")
    c, ids, _ = _worked_inputs(g)
    ep, T, H = c["ep_size"], c["tokens_per_rank"], c["hidden"]
    for case in g["combine_cases"]:
        s, t = case["token"]
        eo = [np.full((ep * T, H), 0x7FC1, np.uint16) for _ in range(ep)]  # NaN everywhere else
        eo[0][s * T + t] = _hex(case["eo_dest0"])
        eo[1][s * T + t] = _hex(case["eo_dest1"])
        masked = "mask" in case
        mask = sum(1 << r for r in case.get("mask", range(ep)))
        out = oracle.combine(ep, c["num_experts"], c["top_k"], H, T, g["num_tokens"], ids, eo,
                             mask_enabled=masked, active_rank_mask=mask)
        assert (out[s][t] == _hex(case["expected"])).all(), case["what"]


def test_combine_rounding_cases():
    g = _load("combine_rounding.json")
    c = g["config"]
    ep, T, H = c["ep_size"], c["tokens_per_rank"], c["hidden"]
    ids = [np.array([g["topk_ids"]], np.int32)] + [np.zeros((0, c["top_k"]), np.int32)] * (ep - 1)
    counts = [1] + [0] * (ep - 1)
    for case in g["cases"]:
        eo = [np.full((ep * T, H), _hex(v), np.uint16) for v in case["eo"]]
        out = oracle.combine(ep, c["num_experts"], c["top_k"], H, T, counts, ids, eo)
        assert int(out[0][0, 0]) == _hex(case["expected"]), case["what"]


def test_combine_rounding_cases_f16_f32():
    g = _load("combine_rounding_f16_f32.json")
    c = g["config"]
    ep, T, H = c["ep_size"], c["tokens_per_rank"], c["hidden"]
    ids = [np.array([g["topk_ids"]], np.int32)] + [np.zeros((0, c["top_k"]), np.int32)] * (ep - 1)
    counts = [1] + [0] * (ep - 1)
    for case in g["cases"]:
        npt = np.uint32 if case["dtype"] == "fp32" else np.uint16
        eo = [np.full((ep * T, H), _hex(v), npt) for v in case["eo"]]
        out = oracle.combine_typed(ep, c["num_experts"], c["top_k"], H, T, counts, ids, eo, case["dtype"])
        got = int(np.asarray(out[0]).view(npt)[0, 0])
        assert got == _hex(case["expected"]), case["what"]


def test_combine_typed_bf16_equals_combine():
    g = _load("combine_rounding.json")
    c = g["config"]
    ep, T, H = c["ep_size"], c["tokens_per_rank"], c["hidden"]
    ids = [np.array([g["topk_ids"]], np.int32)] + [np.zeros((0, c["top_k"]), np.int32)] * (ep - 1)
    counts = [1] + [0] * (ep - 1)
    for case in g["cases"]:
        eo = [np.full((ep * T, H), _hex(v), np.uint16) for v in case["eo"]]
        a = oracle.combine(ep, c["num_experts"], c["top_k"], H, T, counts, ids, eo)
        b = oracle.combine_typed(ep, c["num_experts"], c["top_k"], H, T, counts, ids, eo, "bf16")
        assert int(a[0][0, 0]) == int(b[0][0, 0]) == _hex(case["expected"])

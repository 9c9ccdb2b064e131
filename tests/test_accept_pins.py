"""Pins of the greedy-acceptance oracle: answers planted by construction,
numpy's argmax (a library routine) on random rows, tie and bad-input rules."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from speculative_decode_gateddeltanet_gb300.inputs import make_accept_case


@pytest.mark.parametrize("B,R,V,seed,dtype", [(6, 4, 64, 1, "bf16"), (16, 4, 4096, 2, "bf16"),
                                              (5, 1, 64, 3, "f32"), (32, 9, 512, 4, "f32")])
def test_oracle_finds_the_planted_answers(B, R, V, seed, dtype):
    case = make_accept_case(B, R, V, seed, dtype=dtype, inactive=B // 5)
    r = oracle.greedy_accept(case)
    n = case["n_rows"].numpy()
    assert r["status"] == 0
    assert np.array_equal(r["accept_len"], case["planted_accept"])
    for b in range(B):
        assert np.array_equal(r["target"][b, :n[b]], case["planted_target"][b, :n[b]])
        assert (r["target"][b, n[b]:] == -1).all()  # rows past n_rows untouched


def test_oracle_argmax_equals_numpy_first_maximum():
    rng = np.random.default_rng(7)
    logits = rng.integers(-3, 4, size=(4, 3, 40)).astype(np.float32)  # many ties
    case = {"logits": torch.from_numpy(logits), "drafts": torch.zeros((4, 2), dtype=torch.int32),
            "n_rows": torch.full((4,), 3, dtype=torch.int32)}
    r = oracle.greedy_accept(case)
    assert np.array_equal(r["target"], np.argmax(logits, axis=-1))


def test_accept_rule_on_explicit_cases():
    V = 8
    logits = np.zeros((3, 4, V), dtype=np.float32)
    tok = [[1, 2, 3, 4], [5, 5, 5, 5], [7, 0, 1, 2]]
    for b in range(3):
        for t in range(4):
            logits[b, t, tok[b][t]] = 1.0
    drafts = np.array([[1, 2, 3],    # all three drafts kept -> 3
                       [5, 4, 5],    # the second draft differs -> 1
                       [6, 0, 1]],   # the first draft differs -> 0
                      dtype=np.int32)
    case = {"logits": torch.from_numpy(logits), "drafts": torch.from_numpy(drafts),
            "n_rows": torch.tensor([4, 4, 4], dtype=torch.int32)}
    assert oracle.greedy_accept(case)["accept_len"].tolist() == [3, 1, 0]
    # n_rows caps the drafts considered; inactive and bad requests get 0
    case["n_rows"] = torch.tensor([2, 0, 9], dtype=torch.int32)
    r = oracle.greedy_accept(case)
    assert r["accept_len"].tolist() == [1, 0, 0] and r["status"] == oracle.BAD_NROWS

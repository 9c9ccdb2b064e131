"""Pins of the oracle's deferred commit (the previous step's accepted rows
committed inside the current step's verify) against one-row decode steps.

The deferred call for request b runs the previous step's rows 0..a_prev and
then the current rows from the slot; by the definition of the recurrence that
is one-token decode over the concatenated sequence, with the slot taken after
a_prev + 1 tokens [LightLLM #1330 "Qwen3.5 / Qwen3.5-MoE MTP speculative
decoding", Summary: the accept-count carry; FreeToken #844 "MTP drafts for
Qwen3.5 family + Flash-Next", Tests: verify and commit against stepwise
decode].  Compared bitwise: both sides run the same fp64 steps in the same
order.
"""
from __future__ import annotations

from dataclasses import replace

import numpy as np
import pytest

import oracle
from speculative_decode_gateddeltanet_gb300.inputs import LayerSpec, make_layer, make_step
from test_oracle_pins import chained_steps, f64


def spec(k, B=4, accept="uniform", inactive=0.0):
    return LayerSpec("deferred-pin", B=B, k=k, H_qk=2, H_v=4, d_k=8, d_v=8, dtype="f32", accept=accept,
                     pool="perm", inactive_frac=inactive)


def concatenated(prev, cur, b):
    """Request b's deferred block as one layer of single rows: the previous
    step's rows 0..a_prev, then the current rows."""
    ap, np_ = int(prev["accept_len"][b]), int(prev["n_rows"][b])
    keep = ap + 1 if np_ > 0 else 0
    n = int(cur["n_rows"][b])
    cat = dict(cur)
    for key in ("x", "g", "beta"):
        rows = np.concatenate([f64(prev[key])[:, :keep], f64(cur[key])[:, :n]], axis=1)
        cat[key] = rows
    cat["spec"] = replace(cur["spec"], k=keep + n - 1)
    return cat, keep, n


@pytest.mark.parametrize("kp,kc,seed", [(2, 2, 0), (3, 1, 1), (0, 4, 2), (5, 3, 3)])
def test_deferred_equals_decode_steps(kp, kc, seed):
    prev = make_layer(spec(kp, inactive=0.25), 100 + seed)
    cur = make_step(prev, spec(kc, inactive=0.25), 200 + seed)
    r = oracle.verify_deferred(cur, prev)
    assert r["status"] == 0
    touched = set()
    for b in range(cur["spec"].B):
        cat, keep, n = concatenated(prev, cur, b)
        s = int(cur["slot_ids"][b])
        if keep + n == 0:
            continue
        o_steps, _, _ = chained_steps(cat, keep + n, b)
        assert np.array_equal(r["o"][b, :n], o_steps[keep:]), f"request {b}: o != decode steps"
        assert np.isnan(r["o"][b, n:]).all()
        if keep:
            touched.add(s)
            _, S_c, cs_c = chained_steps(cat, keep, b)
            assert np.array_equal(r["ssm_state"][s], S_c), f"request {b}: state != {keep} steps"
            assert np.array_equal(r["conv_state"][s], cs_c), f"request {b}: conv != {keep} steps"
    for s in range(cur["spec"].pool_slots):
        if s not in touched:
            assert np.array_equal(r["ssm_state"][s], f64(cur["ssm_state"])[s])
            assert np.array_equal(r["conv_state"][s], f64(cur["conv_state"])[s])


def test_nothing_pending_is_a_verify():
    cur = make_layer(spec(3), 7)
    r = oracle.verify_deferred(cur, None)
    v = oracle.verify_commit(cur, commit=False)
    assert np.array_equal(r["o"], v["o"], equal_nan=True)
    assert np.array_equal(r["ssm_state"], f64(cur["ssm_state"]))


def test_a_sequence_of_deferred_steps_is_decode():
    """Three deferred steps and a final flush (no current rows) leave the
    slot where one-token decode over every accepted token leaves it."""
    layers = [make_layer(spec(2, B=2), 11)]
    for i, k in enumerate((3, 1)):
        layers.append(make_step(layers[-1], spec(k, B=2), 12 + i))
    pools = layers[0]
    prev = None
    for cur in layers:
        cur = dict(cur, conv_state=pools["conv_state"], ssm_state=pools["ssm_state"])
        pools = oracle.verify_deferred(cur, prev)
        prev = cur
    flush = dict(layers[-1], conv_state=pools["conv_state"], ssm_state=pools["ssm_state"])
    flush["n_rows"] = np.zeros(2, np.int32)
    end = oracle.verify_deferred(flush, prev)
    for b in range(2):
        xs, gs, bs = [], [], []
        for layer in layers:
            keep = int(layer["accept_len"][b]) + 1
            xs.append(f64(layer["x"])[:, :keep])
            gs.append(f64(layer["g"])[:, :keep])
            bs.append(f64(layer["beta"])[:, :keep])
        cat = dict(layers[0], x=np.concatenate(xs, 1), g=np.concatenate(gs, 1), beta=np.concatenate(bs, 1))
        steps = cat["x"].shape[1]
        cat["spec"] = replace(layers[0]["spec"], k=steps - 1)
        _, S, cs = chained_steps(cat, steps, b)
        s = int(layers[0]["slot_ids"][b])
        assert np.array_equal(end["ssm_state"][s], S)
        assert np.array_equal(end["conv_state"][s], cs)

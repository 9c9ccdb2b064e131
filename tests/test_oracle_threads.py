"""The oracle spread over host threads (the benchmark's all-core CPU baseline)
gives exactly the single-thread oracle's results: the same C routine on
disjoint requests, each writing only its own slots and output rows."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from speculative_decode_gateddeltanet_gb300.inputs import CONFIGS, TINY, LayerSpec, make_layer


@pytest.mark.parametrize("spec,threads", [
    (CONFIGS[TINY], 2),
    (LayerSpec("threads-qwen35-B5-k3", B=5, k=3, H_qk=16, H_v=32, d_k=128, d_v=128, accept="uniform",
               pool="double", inactive_frac=0.2), 3),
    (LayerSpec("threads-B7-k2", B=7, k=2, H_qk=2, H_v=4, d_k=16, d_v=32, pool="perm"), 16),
])
def test_threaded_oracle_equals_single_thread(spec, threads):
    layer = make_layer(spec, 17)
    one = oracle.verify_commit(layer)
    many = oracle.verify_commit_threads(layer, threads)
    assert many["threads"] == min(threads, spec.B)
    assert many["status"] == one["status"]
    assert np.array_equal(many["o"], one["o"], equal_nan=True)
    assert np.array_equal(many["ssm_state"], one["ssm_state"])
    assert np.array_equal(many["conv_state"], one["conv_state"])

"""Device-side greedy acceptance through the C ABI against the oracle
(bit-exact targets and accept lengths) and the planted answers, and the
accept lengths feeding a fused verify + commit with no host round trip."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_against_oracle
from speculative_decode_gateddeltanet_gb300.inputs import SWEEP, make_accept_case, make_layer, workload_layers

pytestmark = pytest.mark.gpu

# (B, R, V, dtype, inactive): the Qwen3.5 vocabulary at the verify shape, a
# one-row case, a ragged wide batch, fp32 logits
CASES = [(16, 4, 151936, "bf16", 0), (3, 1, 64, "f32", 0), (256, 9, 4096, "bf16", 26), (8, 3, 32000, "f32", 1)]


def run(case, device="cuda"):
    from speculative_decode_gateddeltanet_gb300 import gdn

    logits = case["logits"].to(device)
    drafts = case["drafts"].to(device)
    n_rows = case["n_rows"].to(device)
    B, R, _ = logits.shape
    target = torch.full((B, R), -1, dtype=torch.int32, device=device)
    acc = torch.full((B,), -7, dtype=torch.int32, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    gdn.greedy_accept(logits, drafts, n_rows, target, acc, status)
    torch.cuda.synchronize()
    return target.cpu().numpy(), acc.cpu().numpy(), int(status.item())


@pytest.mark.parametrize("B,R,V,dtype,inactive", CASES)
def test_greedy_accept_matches_oracle(B, R, V, dtype, inactive):
    case = make_accept_case(B, R, V, seed=B + R, dtype=dtype, inactive=inactive)
    target, acc, status = run(case)
    ref = oracle.greedy_accept(case)
    assert status == 0
    assert np.array_equal(acc, ref["accept_len"])
    assert np.array_equal(acc, case["planted_accept"])
    assert np.array_equal(target, ref["target"])  # rows past n_rows stay -1 on both sides


def test_greedy_accept_ties_and_random_rows():
    """Random small-integer logits (many equal maxima) against the oracle."""
    rng = np.random.default_rng(11)
    logits = torch.from_numpy(rng.integers(-2, 3, size=(9, 5, 256)).astype(np.float32))
    case = {"logits": logits.to(torch.bfloat16), "drafts": torch.from_numpy(rng.integers(0, 3, (9, 4), dtype=np.int32)),
            "n_rows": torch.from_numpy(rng.integers(0, 6, 9).astype(np.int32))}
    target, acc, status = run(case)
    ref = oracle.greedy_accept(case)
    assert status == 0 and np.array_equal(acc, ref["accept_len"]) and np.array_equal(target, ref["target"])


def test_device_accept_feeds_the_commit():
    """accept_len decided on the device goes straight into gdn_verify_commit."""
    from speculative_decode_gateddeltanet_gb300 import gdn

    ((spec, seed),) = workload_layers(SWEEP, batch=16)
    layer = make_layer(spec, seed)
    case = make_accept_case(spec.B, spec.R, 4096, seed=77)
    case["n_rows"] = layer["n_rows"].clone()
    # re-plant the drafts for these row counts so the accepted prefix varies
    planted = case["planted_target"]
    rng = np.random.default_rng(5)
    acc_want = np.array([rng.integers(0, int(n)) for n in layer["n_rows"]])
    drafts = case["drafts"].numpy().copy()
    for b in range(spec.B):
        for i in range(spec.R - 1):
            drafts[b, i] = planted[b, i] if i < acc_want[b] else (planted[b, i] + 1) % 4096
    case["drafts"] = torch.from_numpy(drafts)
    dev = gdn.DeviceLayer(layer, "cuda")
    logits, d_drafts = case["logits"].cuda(), case["drafts"].cuda()
    target = torch.empty((spec.B, spec.R), dtype=torch.int32, device="cuda")
    gdn.greedy_accept(logits, d_drafts, dev.n_rows, target, dev.accept_len, dev.status)
    gdn.gdn_verify_commit(dev.args())  # same stream, no host copy of accept_len
    torch.cuda.synchronize()
    assert np.array_equal(dev.accept_len.cpu().numpy(), acc_want)
    ref = oracle.verify_commit(dict(layer, accept_len=torch.from_numpy(acc_want.astype(np.int32))))
    check_against_oracle(dict(layer, accept_len=torch.from_numpy(acc_want.astype(np.int32))), dev, ref, commit=True)
    assert int(dev.status.item()) == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_nan_and_infinite_rows(dtype):
    """Rows with NaN logits against the oracle: NaN never wins, a row of only
    NaN gives token 0, a NaN at the planted maximum moves the choice to the
    largest remaining value; a row of only -inf gives token 0 (lowest index
    among equal values)."""
    case = make_accept_case(6, 3, 512, seed=21, dtype=dtype)
    case["n_rows"] = torch.full((6,), 3, dtype=torch.int32)
    lg = case["logits"].float()
    planted = case["planted_target"]
    lg[0, 0, :] = float("nan")                       # every logit NaN
    lg[1, 1, 0] = float("nan")                       # NaN at index 0
    lg[2, 0, int(planted[2, 0])] = float("nan")      # NaN where the maximum was planted
    lg[3, 2, ::2] = float("nan")                     # NaN at every even index
    lg[4, 1, :] = float("-inf")                      # every logit -inf
    lg[5, 0, :] = float("nan")
    lg[5, 0, 300] = float("-inf")                    # one -inf among NaN: it wins
    case["logits"] = lg.to(case["logits"].dtype)
    target, acc, status = run(case)
    ref = oracle.greedy_accept(case)
    assert status == 0
    assert np.array_equal(target, ref["target"]) and np.array_equal(acc, ref["accept_len"])
    assert target[0, 0] == 0 and target[4, 1] == 0 and target[5, 0] == 300
    assert target[2, 0] != planted[2, 0]


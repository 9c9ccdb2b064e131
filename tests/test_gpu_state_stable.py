"""GDN_FLAG_STATE_STABLE through the C ABI: with the caller's promise that
nothing still running on the stream writes a call's slots, slot_ids or
n_rows, each call fetches its state slices while the call before it drains.
Stacks of distinct layers launched back to back with the flag must match the
oracle under the stated tolerances and give the same bits as without it, in
every mode; a flagged call right after the device-side acceptance that
produces its accept_len must read the finished accept lengths."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import bits, check_against_oracle
from speculative_decode_gateddeltanet_gb300.inputs import (RAGGED, STACK, CONFIGS, make_accept_case,
                                                           make_layer, make_step, workload_layers)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _stack(n, snapshot=False):
    from speculative_decode_gateddeltanet_gb300 import gdn

    layers = [make_layer(spec, seed) for spec, seed in workload_layers(STACK, layers=n)]
    return layers, [gdn.DeviceLayer(layer, "cuda", snapshot=snapshot) for layer in layers]


def _run_stack(devs, mode, stable, stream):
    from speculative_decode_gateddeltanet_gb300 import gdn

    for d in devs:
        d.state_stable = stable
    args = [d.args() for d in devs]
    with torch.cuda.stream(stream):
        for a in args:
            if mode == "fused":
                gdn.gdn_verify_commit(a, stream)
            else:
                m = gdn.REPLAY if mode == "replay" else gdn.SNAPSHOT
                gdn.gdn_verify(a, m, stream)
                gdn.gdn_commit(a, m, stream)
    torch.cuda.synchronize()


@pytest.mark.parametrize("mode", ["fused", "replay", "snapshot"])
def test_flagged_stack_matches_oracle_and_unflagged_bits(mode):
    n = 8
    layers, flagged = _stack(n, snapshot=mode == "snapshot")
    _, plain = _stack(n, snapshot=mode == "snapshot")
    stream = torch.cuda.Stream()
    _run_stack(flagged, mode, True, stream)
    _run_stack(plain, mode, False, stream)
    for layer, f, p in zip(layers, flagged, plain):
        assert int(f.status.item()) == 0
        check_against_oracle(layer, f, oracle.verify_commit(layer), commit=True)
        assert torch.equal(bits(f.o), bits(p.o))
        assert torch.equal(bits(f.ssm_state), bits(p.ssm_state))
        assert torch.equal(bits(f.conv_state), bits(p.conv_state))


def test_flagged_ragged_layers_back_to_back():
    """Two B=256 ragged layers (requests of 2, 4 or 9 rows, 10 % inactive),
    the second flagged behind the first: 64 value heads, the one-buffer rows
    staging and a partial last round of items."""
    from dataclasses import replace

    from speculative_decode_gateddeltanet_gb300 import gdn

    base = CONFIGS[RAGGED]
    layers = [make_layer(replace(base, name=f"ragged-{i}"), 4100 + i) for i in range(2)]
    devs = [gdn.DeviceLayer(layer, "cuda") for layer in layers]
    _run_stack(devs, "fused", True, torch.cuda.Stream())
    for layer, d in zip(layers, devs):
        check_against_oracle(layer, d, oracle.verify_commit(layer), commit=True)


def test_flagged_deferred_stack():
    """Six layers in deferred form: every layer's first step (nothing
    pending), then every layer's second step, flagged, committing the first
    step's accepted rows from its carry."""
    from speculative_decode_gateddeltanet_gb300 import gdn

    specs = workload_layers(STACK, layers=6)
    firsts = [make_layer(spec, seed) for spec, seed in specs]
    seconds = [make_step(f, spec, seed + 50) for f, (spec, seed) in zip(firsts, specs)]
    stream = torch.cuda.Stream()
    d1s, d2s, a2s, prevs = [], [], [], []
    for first, second in zip(firsts, seconds):
        d1, d2 = gdn.DeviceLayer(first, "cuda"), gdn.DeviceLayer(second, "cuda")
        d1.conv_state, d1.ssm_state = d2.conv_state, d2.ssm_state  # one slot pool per layer
        a1 = d1.args()
        d1.carry = torch.empty(gdn.carry_bytes(a1) // 4, device="cuda")
        a1.carry = d1.carry.data_ptr()
        with torch.cuda.stream(stream):
            gdn.gdn_verify_deferred(a1, None, stream)
        d2.state_stable = True
        a2 = d2.args()
        d2.carry = torch.empty(gdn.carry_bytes(a2) // 4, device="cuda")
        a2.carry, a2.accept_len = d2.carry.data_ptr(), None
        d1s.append(d1)
        d2s.append(d2)
        a2s.append(a2)
        prevs.append(gdn.make_prev(x=d1.x, n_rows=d1.n_rows, accept_len=d1.accept_len, carry=d1.carry))
    with torch.cuda.stream(stream):
        for a2, pv in zip(a2s, prevs):
            gdn.gdn_verify_deferred(a2, pv, stream)
    torch.cuda.synchronize()
    for first, second, d2 in zip(firsts, seconds, d2s):
        assert int(d2.status.item()) == 0
        ref = oracle.verify_deferred(second, first)
        valid = np.zeros((second["spec"].B, second["spec"].R), bool)
        for b in range(second["spec"].B):
            valid[b, :int(second["n_rows"][b])] = True
        o = d2.o.double().cpu().numpy()
        err = float(np.abs(o[valid] - ref["o"][valid]).max() / np.abs(ref["o"][valid]).max())
        assert err <= 2e-3 and np.isnan(o[~valid]).all()
        S = d2.ssm_state.double().cpu().numpy()
        for b in range(second["spec"].B):
            s = int(second["slot_ids"][b])
            if int(first["n_rows"][b]) > 0:
                e = float(np.linalg.norm(S[s] - ref["ssm_state"][s]) / np.linalg.norm(ref["ssm_state"][s]))
                assert e <= 1e-3, f"slot {s}: {e:.3e}"
        ref_cs = torch.from_numpy(ref["conv_state"]).to(d2.conv_state.dtype)
        assert torch.equal(bits(d2.conv_state), bits(ref_cs))


@pytest.mark.parametrize("layers", [1, 4])
def test_flagged_call_after_device_acceptance(layers):
    """gdn_greedy_accept writes accept_len and, on the same stream, a flagged
    fused call per layer commits at it: the calls fetch their state early but
    read accept_len only once the acceptance kernels have finished."""
    from speculative_decode_gateddeltanet_gb300 import gdn

    specs = workload_layers(STACK, layers=layers)
    spec = specs[0][0]
    case = make_accept_case(spec.B, spec.R, 151936, seed=404)
    lays = [make_layer(s, seed) for s, seed in specs]
    for layer in lays:
        layer["n_rows"] = case["n_rows"].clone()
    devs = [gdn.DeviceLayer(layer, "cuda") for layer in lays]
    acc = torch.full((spec.B,), -1, dtype=torch.int32, device="cuda")
    target = torch.empty((spec.B, spec.R), dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    logits, drafts = case["logits"].cuda(), case["drafts"].cuda()
    args = []
    for d in devs:
        d.state_stable = True
        a = d.args()
        a.accept_len = acc.data_ptr()
        args.append(a)
    with torch.cuda.stream(stream):
        gdn.greedy_accept(logits, drafts, devs[0].n_rows, target, acc, stream=stream)
        for a in args:
            gdn.gdn_verify_commit(a, stream)
    torch.cuda.synchronize()
    want = case["planted_accept"]
    assert np.array_equal(acc.cpu().numpy(), want)
    for layer, d in zip(lays, devs):
        lay = dict(layer, accept_len=torch.from_numpy(want.astype(np.int32)))
        check_against_oracle(lay, d, oracle.verify_commit(lay), commit=True)
        assert int(d.status.item()) == 0

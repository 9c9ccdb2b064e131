"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bar: o within 2e-3 max relative error (max |o - o_ref| / max |o_ref| over the
call's valid rows), committed states within 1e-3 relative Frobenius error per
slot, committed conv windows, slot selection and untouched slots bit-exact,
rows outside n_rows untouched.  Plus GPU-internal checks: fused == verify +
replay commit == snapshot verify + copy commit bit for bit, and k+1 rows in one
call against k+1 one-row calls (windows bit for bit, o and state to fp32
rounding) [FreeToken #844, Tests].
"""
from __future__ import annotations

from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from gpu_util import (O_TOL, S_TOL, bits, check_against_oracle, committed_slots, o_error, run_gpu,
                      valid_rows)
from speculative_decode_gateddeltanet_gb300.inputs import (CONFIGS, RAGGED, SINGLE, STACK, SWEEP, SWEEP_B,
                                                           TINY, LayerSpec, make_layer, workload_layers)

pytestmark = pytest.mark.gpu
MODES = ["fused", "replay", "snapshot"]


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


_cache = {}


def cached(name, spec, seed):
    key = (name, seed)
    if key not in _cache:
        layer = make_layer(spec, seed)
        _cache[key] = (layer, oracle.verify_commit(layer))
    return _cache[key]


@pytest.mark.parametrize("mode", MODES)
def test_tiny_fp32(mode):
    (spec, seed), = workload_layers(TINY)
    layer, ref = cached(TINY, spec, seed)
    check_against_oracle(layer, run_gpu(layer, mode), ref, commit=True)


@pytest.mark.parametrize("mode", MODES)
def test_single_request(mode):
    (spec, seed), = workload_layers(SINGLE)
    layer, ref = cached(SINGLE, spec, seed)
    check_against_oracle(layer, run_gpu(layer, mode), ref, commit=True)


@pytest.mark.parametrize("B", SWEEP_B)
@pytest.mark.parametrize("mode", ["fused", "replay"])
def test_batch_sweep(B, mode):
    (spec, seed), = workload_layers(SWEEP, batch=B)
    layer, ref = cached(SWEEP, spec, seed)
    check_against_oracle(layer, run_gpu(layer, mode), ref, commit=True)


@pytest.mark.parametrize("B", [2, 8])
def test_batch_sweep_snapshot(B):
    (spec, seed), = workload_layers(SWEEP, batch=B)
    layer, ref = cached(SWEEP, spec, seed)
    check_against_oracle(layer, run_gpu(layer, "snapshot"), ref, commit=True)


@pytest.mark.parametrize("mode", MODES)
def test_ragged_B256(mode):
    (spec, seed), = workload_layers(RAGGED)
    layer, ref = cached(RAGGED, spec, seed)
    check_against_oracle(layer, run_gpu(layer, mode), ref, commit=True)


def test_stack_36_layers_back_to_back():
    """All 36 layers launched back to back on one stream, as the benchmark
    does, then each compared with the oracle."""
    from speculative_decode_gateddeltanet_gb300 import gdn

    layers, devs = [], []
    for spec, seed in workload_layers(STACK):
        layer = make_layer(spec, seed)
        layers.append(layer)
        devs.append(gdn.DeviceLayer(layer, "cuda"))
    for dev in devs:
        gdn.gdn_verify_commit(dev.args())
    torch.cuda.synchronize()
    for layer, dev in zip(layers, devs):
        check_against_oracle(layer, dev, oracle.verify_commit(layer), commit=True)
        assert int(dev.status.item()) == 0


@pytest.mark.parametrize("name", [SINGLE, RAGGED, TINY])
def test_modes_agree_bitwise(name):
    (spec, seed), = workload_layers(name)
    layer, _ = cached(name, spec, seed)
    runs = {m: run_gpu(layer, m) for m in MODES + ["verify"]}
    valid = torch.from_numpy(valid_rows(layer))
    ref = runs["fused"]
    for m, dev in runs.items():
        assert torch.equal(bits(dev.o[valid.cuda()]), bits(ref.o[valid.cuda()])), m
        if m != "verify":
            assert torch.equal(bits(dev.ssm_state), bits(ref.ssm_state)), m
            assert torch.equal(bits(dev.conv_state), bits(ref.conv_state)), m


def test_verify_only_leaves_slots_untouched():
    (spec, seed), = workload_layers(RAGGED)
    layer, ref = cached(RAGGED, spec, seed)
    for mode in ("verify", "verify_snapshot"):
        dev = run_gpu(layer, mode)
        check_against_oracle(layer, dev, ref, commit=False)


@pytest.mark.parametrize("name", [TINY, SINGLE])
def test_snapshot_rows_match_oracle(name):
    (spec, seed), = workload_layers(name)
    layer = make_layer(spec, seed)
    ref = oracle.verify_commit(layer, commit=False, snapshot=True)
    dev = run_gpu(layer, "verify_snapshot")
    sS = dev.scratch_S.double().cpu().numpy()
    scs = dev.scratch_cs.cpu()
    for b in range(spec.B):
        for t in range(int(layer["n_rows"][b])):
            r = ref["snap_S"][b, t]
            err = np.linalg.norm(sS[b, t] - r) / np.linalg.norm(r)
            assert err <= S_TOL, (b, t, err)
            want = torch.from_numpy(ref["snap_cs"][b, t]).to(scs.dtype)
            assert torch.equal(bits(scs[b, t]), bits(want)), (b, t)


def test_chained_single_rows_match_one_call():
    """k+1 one-row fused calls (accept 0 each) against one (k+1)-row call: the
    same decode steps, so the committed windows agree bit for bit and o and
    the state agree to fp32 rounding (the multi-row call takes each chunk's
    dot products on the chunk's starting state, one row at a time does not)."""
    from speculative_decode_gateddeltanet_gb300 import gdn

    (spec, seed), = workload_layers(SWEEP, batch=4)
    layer = make_layer(spec, seed)
    full_acc = layer["n_rows"] - 1
    multi = gdn.DeviceLayer(dict(layer, accept_len=full_acc), "cuda")
    gdn.gdn_verify_commit(multi.args())
    chain = gdn.DeviceLayer(layer, "cuda")
    o_chain = torch.full_like(multi.o, float("nan"))
    for t in range(spec.R):
        n_t = (chain.n_rows > t).int()
        o_t = torch.full((spec.B, 1, spec.H_v, spec.d_v), float("nan"), device="cuda")
        x_t = chain.x[:, t:t + 1].contiguous()
        g_t = chain.g[:, t:t + 1].contiguous()
        beta_t = chain.beta[:, t:t + 1].contiguous()
        work = torch.empty(chain.work.numel(), device="cuda")
        a = gdn.make_args(x=x_t, g=g_t, beta=beta_t, conv_w=chain.conv_w,
                          conv_state=chain.conv_state, ssm_state=chain.ssm_state,
                          slot_ids=chain.slot_ids, n_rows=n_t, accept_len=torch.zeros_like(n_t),
                          o=o_t, work=work, status=chain.status, H_qk=spec.H_qk)
        gdn.gdn_verify_commit(a)
        torch.cuda.synchronize()
        o_chain[:, t] = o_t[:, 0]
    valid = torch.from_numpy(valid_rows(layer)).cuda()
    diff = (o_chain[valid] - multi.o[valid]).abs().max() / multi.o[valid].abs().max()
    assert float(diff) <= 1e-5, float(diff)
    for s_ in committed_slots(dict(layer, accept_len=full_acc)):
        err = torch.linalg.norm(chain.ssm_state[s_] - multi.ssm_state[s_]) / torch.linalg.norm(multi.ssm_state[s_])
        assert float(err) <= 1e-5, (s_, float(err))
    assert torch.equal(bits(chain.conv_state), bits(multi.conv_state))


SHAPES = [
    LayerSpec("dk32", B=3, k=3, H_qk=4, H_v=8, d_k=32, d_v=32, pool="double"),
    LayerSpec("dk64", B=3, k=2, H_qk=2, H_v=8, d_k=64, d_v=64, pool="perm"),
    LayerSpec("dk16-dv32", B=3, k=4, H_qk=2, H_v=4, d_k=16, d_v=32, pool="perm"),
    LayerSpec("dk128-G1", B=2, k=3, H_qk=4, H_v=4, d_k=128, d_v=128, pool="perm"),
    LayerSpec("dk128-dv64", B=2, k=3, H_qk=2, H_v=8, d_k=128, d_v=64, pool="perm"),
    LayerSpec("k0-one-row", B=5, k=0, H_qk=2, H_v=4, d_k=128, d_v=128, pool="double"),
    LayerSpec("k15-max-rows", B=2, k=15, H_qk=2, H_v=4, d_k=128, d_v=128, pool="perm"),
    LayerSpec("f32-qwen-heads", B=2, k=3, H_qk=16, H_v=32, d_k=128, d_v=128, dtype="f32", pool="perm"),
]


@pytest.mark.parametrize("spec", SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("mode", MODES)
def test_shapes(spec, mode):
    layer = make_layer(spec, 77)
    check_against_oracle(layer, run_gpu(layer, mode), oracle.verify_commit(layer), commit=True)


@pytest.mark.parametrize("which", ["none", "all"])
def test_accept_extremes(which):
    spec = LayerSpec("acc", B=4, k=3, H_qk=16, H_v=32, d_k=128, d_v=128, pool="double")
    layer = make_layer(spec, 11)
    layer["accept_len"] = torch.zeros(4, dtype=torch.int32) if which == "none" else layer["n_rows"] - 1
    for mode in MODES:
        check_against_oracle(layer, run_gpu(layer, mode), oracle.verify_commit(layer), commit=True)


def test_inactive_and_bad_requests_flagged_and_skipped():
    from speculative_decode_gateddeltanet_gb300 import gdn

    spec = LayerSpec("bad", B=6, k=2, H_qk=2, H_v=4, d_k=128, d_v=128, pool="double")
    layer = make_layer(spec, 3)
    P = spec.pool_slots
    layer["n_rows"] = torch.tensor([3, 0, 3, 3, 5, 3], dtype=torch.int32)      # 1 inactive, 4 bad n
    layer["slot_ids"] = torch.tensor([0, 1, P, 3, 4, 5], dtype=torch.int32)    # 2 bad slot
    layer["accept_len"] = torch.tensor([1, 0, 0, 3, 0, 2], dtype=torch.int32)  # 3 bad accept
    ref = oracle.verify_commit(layer)
    assert ref["status"] == 7
    for mode, want in (("fused", 7), ("replay", 7), ("snapshot", 7), ("verify", 3)):
        dev = run_gpu(layer, mode)
        assert int(dev.status.item()) == want, mode
        check_against_oracle(layer, dev, ref, commit=mode != "verify")
    # all requests inactive: nothing written at all
    layer["n_rows"] = torch.zeros(6, dtype=torch.int32)
    dev = run_gpu(layer, "fused")
    assert torch.isnan(dev.o).all() and int(dev.status.item()) == 0
    assert torch.equal(bits(dev.ssm_state), bits(layer["ssm_state"]))


def test_calls_repeat_on_the_same_buffers():
    """Three fused calls in a row on the same buffers (state, windows and work
    reused): the third call's state equals the oracle run three times."""
    from speculative_decode_gateddeltanet_gb300 import gdn

    (spec, seed), = workload_layers(SWEEP, batch=16)
    layer = make_layer(spec, seed)
    dev = gdn.DeviceLayer(layer, "cuda")
    cur = dict(layer)
    for _ in range(3):
        gdn.gdn_verify_commit(dev.args())
        torch.cuda.synchronize()
        r = oracle.verify_commit(cur)
        cur = dict(cur, ssm_state=torch.from_numpy(r["ssm_state"]).float(),
                   conv_state=torch.from_numpy(r["conv_state"]).to(torch.bfloat16))
    for s in committed_slots(layer):
        err = torch.linalg.norm(dev.ssm_state[s].double().cpu() - cur["ssm_state"][s].double()) / \
            torch.linalg.norm(cur["ssm_state"][s].double())
        assert float(err) <= S_TOL
    assert torch.equal(bits(dev.conv_state), bits(cur["conv_state"]))


def test_guard_bands_untouched():
    """o and the state pool sit inside larger buffers; the bytes around them
    must not change."""
    from speculative_decode_gateddeltanet_gb300 import gdn

    (spec, seed), = workload_layers(SWEEP, batch=4)
    layer = make_layer(spec, seed)
    dev = gdn.DeviceLayer(layer, "cuda")
    G = 4096
    o_buf = torch.full((G + dev.o.numel() + G,), -7.0, device="cuda")
    s_buf = torch.full((G + dev.ssm_state.numel() + G,), -9.0, device="cuda")
    o = o_buf[G:G + dev.o.numel()].view_as(dev.o)
    o.fill_(float("nan"))
    S = s_buf[G:G + dev.ssm_state.numel()].view_as(dev.ssm_state)
    S.copy_(dev.ssm_state)
    a = gdn.make_args(x=dev.x, g=dev.g, beta=dev.beta, conv_w=dev.conv_w, conv_state=dev.conv_state,
                      ssm_state=S, slot_ids=dev.slot_ids, n_rows=dev.n_rows, accept_len=dev.accept_len,
                      o=o, work=dev.work, status=dev.status, H_qk=spec.H_qk)
    gdn.gdn_verify_commit(a)
    torch.cuda.synchronize()
    assert bool((o_buf[:G] == -7.0).all()) and bool((o_buf[-G:] == -7.0).all())
    assert bool((s_buf[:G] == -9.0).all()) and bool((s_buf[-G:] == -9.0).all())
    ref = oracle.verify_commit(layer)
    assert o_error(o.double().cpu().numpy(), ref["o"], valid_rows(layer)) <= O_TOL


RAW_CASES = [(TINY, None, "fused"), (SINGLE, None, "fused"), (SWEEP, 16, "fused"), (SWEEP, 4, "replay"),
             (RAGGED, None, "fused"), (TINY, None, "snapshot")]


@pytest.mark.parametrize("name,batch,mode", RAW_CASES, ids=lambda c: str(c))
def test_raw_gating_matches_oracle(name, batch, mode):
    """The prologue forms g = -exp(A_log) softplus(a) and beta = sigmoid(b)
    from the raw projections (GDN_FLAG_RAW_GATING); the oracle forms them in
    fp64 from the same fp32 inputs."""
    ((spec, seed),) = workload_layers(name, batch=batch)
    layer = make_layer(spec, seed)
    ref = oracle.verify_commit(layer, commit=True, raw_gating=True)
    dev = run_gpu(layer, mode, raw_gating=True)
    check_against_oracle(layer, dev, ref, commit=True)
    assert int(dev.status.item()) == 0


DEGENERATE = {
    "no_write": (0.0, 0.0),        # g = 0, beta = 0: the state is only read (S unchanged, o = scale S0 q)
    "exact_write": (0.0, 1.0),     # g = 0, beta = 1: each row overwrites S k = v
    "full_decay": (-200.0, 1.0),   # exp(g) = 0 in fp32: each row leaves S = v k^T
}


@pytest.mark.parametrize("case", sorted(DEGENERATE))
@pytest.mark.parametrize("mode", MODES)
def test_degenerate_gating(case, mode):
    """The recurrence's special cases through the whole CUDA path: no write,
    exact write and full decay (decay products underflowing to zero inside
    a chunk), against the oracle; with no write the committed state equals
    the input state bit for bit."""
    g_val, b_val = DEGENERATE[case]
    spec = LayerSpec("degenerate", B=4, k=3, H_qk=16, H_v=32, d_k=128, d_v=128, pool="perm")
    layer = make_layer(spec, 77)
    layer["g"] = torch.full_like(layer["g"], g_val)
    layer["beta"] = torch.full_like(layer["beta"], b_val)
    dev = run_gpu(layer, mode)
    check_against_oracle(layer, dev, oracle.verify_commit(layer), commit=True)
    assert int(dev.status.item()) == 0
    if case == "no_write":
        assert torch.equal(bits(dev.ssm_state), bits(layer["ssm_state"]))

"""GPU parity of the deferred commit (``gdn_verify_deferred``): step s's call
commits step s-1's accepted rows and verifies step s's rows in one pass over
the state [LightLLM #1330 "Qwen3.5 / Qwen3.5-MoE MTP speculative decoding",
Summary: the accept-count carry; lmdeploy #5006 "speculative decoding for
TurboMind", Verification path: verify-and-commit mode].

Against the oracle's definition (a replay commit of the previous step, then a
verify of the current one): o of the current rows within 2e-3, committed
states within 1e-3 relative Frobenius error, conv windows and untouched slots
bit-exact; against the fused form over a sequence of steps; and bad pending
data flagged and skipped.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import O_TOL, S_TOL, bits
from speculative_decode_gateddeltanet_gb300.inputs import LayerSpec, make_layer, make_step

pytestmark = pytest.mark.gpu

QWEN = dict(H_qk=16, H_v=32, d_k=128, d_v=128)


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_deferred(cur, prev, raw_gating=False):
    """Two deferred calls on the GPU sharing one slot pool: the previous
    step's (nothing pending; it writes its carry), then the current step's,
    which commits the previous step's accepted rows from that carry.  Returns
    (DeviceLayer of the current call, DeviceLayer of the previous call)."""
    from speculative_decode_gateddeltanet_gb300 import gdn

    dev = gdn.DeviceLayer(cur, "cuda", raw_gating=raw_gating)
    pd, pdev = None, None
    if prev is not None:
        pdev = gdn.DeviceLayer(prev, "cuda", raw_gating=raw_gating)
        pdev.conv_state, pdev.ssm_state = dev.conv_state, dev.ssm_state  # one pool
        a1 = pdev.args()
        pdev.carry = torch.empty(gdn.carry_bytes(a1) // 4, device="cuda")
        a1.carry = pdev.carry.data_ptr()
        gdn.gdn_verify_deferred(a1, None)
        pd = gdn.make_prev(x=pdev.x, n_rows=pdev.n_rows, accept_len=pdev.accept_len, carry=pdev.carry)
    a = dev.args()
    dev.carry = torch.empty(gdn.carry_bytes(a) // 4, device="cuda")
    a.carry = dev.carry.data_ptr()
    a.accept_len = None  # never read by the deferred call
    gdn.gdn_verify_deferred(a, pd)
    torch.cuda.synchronize()
    return dev, pdev


def valid_current(cur, prev):
    spec = cur["spec"]
    Rp = prev["spec"].R if prev is not None else 0
    v = np.zeros((spec.B, spec.R), bool)
    commits = set()
    for b in range(spec.B):
        n, s = int(cur["n_rows"][b]), int(cur["slot_ids"][b])
        np_ = int(prev["n_rows"][b]) if prev is not None else 0
        ap = int(prev["accept_len"][b]) if prev is not None else -1
        if not (0 <= n <= spec.R and 0 <= np_ <= Rp and 0 <= s < spec.pool_slots):
            continue
        if np_ > 0 and not 0 <= ap < np_:
            continue
        v[b, :n] = True
        if np_ > 0:
            commits.add(s)
    return v, commits


def check(cur, prev, dev, ref):
    valid, commits = valid_current(cur, prev)
    o = dev.o.double().cpu().numpy()
    if valid.any():
        err = float(np.abs(o[valid] - ref["o"][valid]).max() / np.abs(ref["o"][valid]).max())
        assert err <= O_TOL, f"o max relative error {err:.3e}"
    assert np.isnan(o[~valid]).all(), "rows outside the current valid rows were written"
    S, cs = dev.ssm_state.cpu(), dev.conv_state.cpu()
    for s in range(cur["spec"].pool_slots):
        if s in commits:
            ref_S = ref["ssm_state"][s]
            e = float(np.linalg.norm(S[s].double().numpy() - ref_S) / np.linalg.norm(ref_S))
            assert e <= S_TOL, f"slot {s}: state error {e:.3e}"
            assert torch.equal(bits(cs[s]), bits(torch.from_numpy(ref["conv_state"][s]).to(cs.dtype))), s
        else:
            assert torch.equal(bits(S[s]), bits(cur["ssm_state"][s])), f"slot {s} state touched"
            assert torch.equal(bits(cs[s]), bits(cur["conv_state"][s])), f"slot {s} conv touched"


def spec_of(B, k, dtype="bf16", shape=QWEN, **kw):
    return LayerSpec("deferred", B=B, k=k, dtype=dtype, pool="perm", **shape, **kw)


TINY_SHAPE = dict(H_qk=2, H_v=4, d_k=16, d_v=16)
CASES = [
    ("tiny-f32", spec_of(2, 2, "f32", TINY_SHAPE), spec_of(2, 2, "f32", TINY_SHAPE)),
    ("B1-k3", spec_of(1, 3), spec_of(1, 3)),
    ("B16-k3", spec_of(16, 3), spec_of(16, 3)),
    ("B4-k0-then-k3", spec_of(4, 0), spec_of(4, 3)),
    ("B8-k5-then-k1-inactive", spec_of(8, 5, inactive_frac=0.25), spec_of(8, 1, inactive_frac=0.25)),
    ("B64-ragged", spec_of(64, 8, k_choices=(1, 3, 8), inactive_frac=0.1),
     spec_of(64, 3, k_choices=(1, 3), inactive_frac=0.1)),
    ("d_k64", spec_of(4, 2, shape=dict(H_qk=4, H_v=8, d_k=64, d_v=64)),
     spec_of(4, 3, shape=dict(H_qk=4, H_v=8, d_k=64, d_v=64))),
    ("d_k32-16-rows-both", spec_of(4, 15, shape=dict(H_qk=2, H_v=4, d_k=32, d_v=64)),
     spec_of(4, 15, shape=dict(H_qk=2, H_v=4, d_k=32, d_v=64))),
    ("d_k16-f32-k7-then-k0", spec_of(3, 7, "f32", TINY_SHAPE), spec_of(3, 0, "f32", TINY_SHAPE)),
]


@pytest.mark.parametrize("name,ps,cs", CASES, ids=[c[0] for c in CASES])
def test_deferred_matches_oracle(name, ps, cs):
    prev = make_layer(ps, 500 + len(name))
    cur = make_step(prev, cs, 600 + len(name))
    ref = oracle.verify_deferred(cur, prev)
    dev, pdev = run_deferred(cur, prev)
    assert int(dev.status.item()) == ref["status"] == 0
    check(cur, prev, dev, ref)
    # the first call, with nothing pending, is a verify of the previous step's rows
    first = oracle.verify_commit(prev, commit=False)
    valid, _ = valid_current(prev, None)
    o1 = pdev.o.double().cpu().numpy()
    err = float(np.abs(o1[valid] - first["o"][valid]).max() / np.abs(first["o"][valid]).max())
    assert err <= O_TOL and int(pdev.status.item()) == 0


def test_deferred_raw_gating():
    prev = make_layer(spec_of(16, 3), 71)
    cur = make_step(prev, spec_of(16, 3), 72)
    ref = oracle.verify_deferred(cur, prev, raw_gating=True)
    dev, _ = run_deferred(cur, prev, raw_gating=True)
    assert int(dev.status.item()) == 0
    check(cur, prev, dev, ref)


def test_nothing_pending_equals_verify_bitwise():
    from gpu_util import run_gpu

    cur = make_layer(spec_of(16, 3), 81)
    dev, _ = run_deferred(cur, None)
    ver = run_gpu(cur, "verify")
    assert torch.equal(bits(dev.o), bits(ver.o))
    assert torch.equal(bits(dev.ssm_state), bits(cur["ssm_state"]))
    check(cur, None, dev, oracle.verify_deferred(cur, None))


def test_sequence_of_deferred_steps_matches_fused_steps():
    """Four decode steps in deferred form plus a flush, on the same device
    pools, each call committing the one before from its carry, against the
    oracle running each step as a fused verify+commit: every step's o and the
    final pools."""
    from speculative_decode_gateddeltanet_gb300 import gdn

    steps = [make_layer(spec_of(8, 3, inactive_frac=0.125), 90)]
    for i, k in enumerate((2, 3, 1)):
        steps.append(make_step(steps[-1], spec_of(8, k, inactive_frac=0.125), 91 + i))
    B = 8
    first = steps[0]
    conv_state = first["conv_state"].cuda().contiguous()
    ssm_state = first["ssm_state"].cuda().contiguous()
    conv_w = first["conv_w"].cuda().contiguous()
    slots = first["slot_ids"].cuda().contiguous()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_pools = dict(first)
    prev_t = None
    for i, layer in enumerate(steps + [None]):
        flush = layer is None
        if flush:  # no current rows: only the last step's commit
            layer = dict(steps[-1], n_rows=torch.zeros(B, dtype=torch.int32))
        cur_t = {k: layer[k].cuda().contiguous() for k in ("x", "g", "beta", "n_rows", "accept_len")}
        o = torch.full((B, layer["spec"].R, 32, 128), float("nan"), device="cuda")
        a = gdn.make_args(x=cur_t["x"], g=cur_t["g"], beta=cur_t["beta"], conv_w=conv_w,
                          conv_state=conv_state, ssm_state=ssm_state, slot_ids=slots,
                          n_rows=cur_t["n_rows"], o=o, status=status, H_qk=16)
        cur_t["carry"] = torch.empty(gdn.carry_bytes(a) // 4, device="cuda")
        a.carry = cur_t["carry"].data_ptr()
        work = torch.empty(gdn.work_bytes(a) // 4, device="cuda")
        a.work = work.data_ptr()
        pd = None if prev_t is None else gdn.make_prev(x=prev_t["x"], n_rows=prev_t["n_rows"],
                                                       accept_len=prev_t["accept_len"], carry=prev_t["carry"])
        gdn.gdn_verify_deferred(a, pd)
        torch.cuda.synchronize()
        if not flush:  # the oracle's fused step i: o from the committed pools, then the commit
            r = oracle.verify_commit(dict(layer, conv_state=ref_pools["conv_state"],
                                          ssm_state=ref_pools["ssm_state"]))
            valid = np.zeros((B, layer["spec"].R), bool)
            for b in range(B):
                valid[b, :int(layer["n_rows"][b])] = True
            og = o.double().cpu().numpy()
            err = float(np.abs(og[valid] - r["o"][valid]).max() / np.abs(r["o"][valid]).max())
            assert err <= O_TOL, f"step {i}: o error {err:.3e}"
            assert np.isnan(og[~valid]).all()
            ref_pools = {"conv_state": r["conv_state"], "ssm_state": r["ssm_state"]}
        prev_t = cur_t
    assert int(status.item()) == 0
    S = ssm_state.double().cpu().numpy()
    for s in range(first["spec"].pool_slots):
        e = float(np.linalg.norm(S[s] - ref_pools["ssm_state"][s]) / np.linalg.norm(ref_pools["ssm_state"][s]))
        assert e <= 4 * S_TOL, f"slot {s}: state error {e:.3e} after four steps"
    ref_cs = torch.from_numpy(ref_pools["conv_state"]).to(torch.bfloat16)
    assert torch.equal(bits(conv_state), bits(ref_cs))


def test_bad_pending_data_flagged_and_skipped():
    prev = make_layer(spec_of(6, 2), 31)
    cur = make_step(prev, spec_of(6, 2), 32)
    prev["n_rows"] = torch.tensor([3, 3, 3, 5, 0, 2], dtype=torch.int32)     # 3: pending n_rows > R
    prev["accept_len"] = torch.tensor([1, 3, 0, 0, 0, 1], dtype=torch.int32)  # 1: accept >= n_rows
    cur["n_rows"] = torch.tensor([3, 3, 4, 3, 0, 0], dtype=torch.int32)      # 2: current n_rows > R
    # 4: nothing pending, nothing current; 5: commit only (no current rows)
    good = [0, 5]
    ref = oracle.verify_deferred(cur, prev, requests=good)
    dev, _ = run_deferred(cur, prev)
    from speculative_decode_gateddeltanet_gb300 import gdn

    assert int(dev.status.item()) == gdn.STATUS_BAD_ACCEPT | gdn.STATUS_BAD_NROWS
    check(cur, prev, dev, ref)

"""Helpers for the GPU parity tests: run a layer call through the C ABI and
compare it with the oracle under the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle

O_TOL = 2e-3   # max |o - o_ref| / max |o_ref| over the valid rows of a call
S_TOL = 1e-3   # ||S - S_ref||_F / ||S_ref||_F per committed slot


def run_gpu(layer: dict, mode: str, device="cuda", **kw):
    """mode: fused | replay | snapshot | verify | verify_snapshot.  Returns the
    DeviceLayer after the call(s), synchronised."""
    from speculative_decode_gateddeltanet_gb300 import gdn

    snap = mode in ("snapshot", "verify_snapshot")
    dev = gdn.DeviceLayer(layer, device, snapshot=snap, **kw)
    a = dev.args()
    if mode == "fused":
        gdn.gdn_verify_commit(a)
    elif mode == "replay":
        gdn.gdn_verify(a, gdn.REPLAY)
        gdn.gdn_commit(a, gdn.REPLAY)
    elif mode == "snapshot":
        gdn.gdn_verify(a, gdn.SNAPSHOT)
        gdn.gdn_commit(a, gdn.SNAPSHOT)
    elif mode == "verify":
        gdn.gdn_verify(a, gdn.REPLAY)
    elif mode == "verify_snapshot":
        gdn.gdn_verify(a, gdn.SNAPSHOT)
    else:
        raise ValueError(mode)
    torch.cuda.synchronize()
    return dev


def bits(t: torch.Tensor) -> torch.Tensor:
    t = t.detach().cpu()
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def valid_rows(layer) -> np.ndarray:
    spec = layer["spec"]
    v = np.zeros((spec.B, spec.R), bool)
    for b in range(spec.B):
        n = int(layer["n_rows"][b])
        if 0 < n <= spec.R and 0 <= int(layer["slot_ids"][b]) < spec.pool_slots:
            v[b, :n] = True
    return v


def committed_slots(layer) -> set[int]:
    spec = layer["spec"]
    out = set()
    for b in range(spec.B):
        n, s, a = int(layer["n_rows"][b]), int(layer["slot_ids"][b]), int(layer["accept_len"][b])
        if 0 < n <= spec.R and 0 <= s < spec.pool_slots and 0 <= a < n:
            out.add(s)
    return out


def o_error(o_gpu: np.ndarray, o_ref: np.ndarray, valid: np.ndarray) -> float:
    ref = o_ref[valid]
    return float(np.abs(o_gpu[valid] - ref).max() / np.abs(ref).max())


def o_error_per_head(o_gpu: np.ndarray, o_ref: np.ndarray, valid: np.ndarray) -> float:
    """Worst, over the valid (request, row, value head) triples, of
    max |o - o_ref| / max |o_ref| within that head's d_v outputs: the margin
    a single small head has, beside the whole-call figure the bar is stated
    on.  Heads whose reference is exactly zero are skipped."""
    ref = o_ref[valid]  # [n][H_v][d_v]
    den = np.abs(ref).max(axis=-1)
    num = np.abs(o_gpu[valid] - ref).max(axis=-1)
    ok = den > 0
    return float((num[ok] / den[ok]).max()) if ok.any() else 0.0


def check_against_oracle(layer: dict, dev, ref: dict, *, commit: bool, check_o: bool = True):
    """o within O_TOL on valid rows and untouched (NaN) elsewhere; committed
    slots within S_TOL and their conv window bit-exact; every other slot
    bitwise unchanged.  Returns (o_err, worst_state_err)."""
    valid = valid_rows(layer)
    o = dev.o.double().cpu().numpy()
    o_err = 0.0
    if check_o:
        o_err = o_error(o, ref["o"], valid)
        head_err = o_error_per_head(o, ref["o"], valid)
        print(f"[parity] {layer['spec'].name}: o error {o_err:.2e} of the call's max |o|; "
              f"worst single (request, row, head) {head_err:.2e} of its own max |o|")
        assert o_err <= O_TOL, f"o max relative error {o_err:.3e}"
        assert np.isnan(o[~valid]).all(), "rows outside the valid set were written"
    S_gpu = dev.ssm_state.cpu()
    cs_gpu = dev.conv_state.cpu()
    S_in, cs_in = layer["ssm_state"], layer["conv_state"]
    slots = committed_slots(layer) if commit else set()
    worst = 0.0
    for s in range(layer["spec"].pool_slots):
        if s in slots:
            ref_S = ref["ssm_state"][s]
            err = float(np.linalg.norm(S_gpu[s].double().numpy() - ref_S) / np.linalg.norm(ref_S))
            worst = max(worst, err)
            assert err <= S_TOL, f"slot {s}: state relative Frobenius error {err:.3e}"
            ref_cs = torch.from_numpy(ref["conv_state"][s]).to(cs_gpu.dtype)
            assert torch.equal(bits(cs_gpu[s]), bits(ref_cs)), f"slot {s}: committed conv window differs"
        else:
            assert torch.equal(bits(S_gpu[s]), bits(S_in[s])), f"slot {s}: state touched"
            assert torch.equal(bits(cs_gpu[s]), bits(cs_in[s])), f"slot {s}: conv state touched"
    return o_err, worst


def oracle_ref(layer, commit=True, **kw):
    return oracle.verify_commit(layer, commit=commit, **kw)

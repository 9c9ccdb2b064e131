"""CPU oracle for GatedDeltaNet speculative verify + commit.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg may call it; the product path never does.  The arithmetic
lives in ``gdn_oracle.c`` (plain C, fp64); this module only marshals arrays
into it with ctypes.  It imports nothing from the CUDA library's package.

Parity status of each part (what pins it) is listed in the tests'
``test_oracle_pins.py`` docstrings.  Every function here is pinned by at
least one invariant, closed form or brute-force case; the value-head to
q/k-head mapping is a shared convention and is pinned only by the
one-hot test that fixes which q/k head each value head reads.
"""
from __future__ import annotations

import ctypes
import time

import numpy as np

from . import build as _build

BAD_SLOT, BAD_NROWS, BAD_ACCEPT = 1, 2, 4
MUTATIONS = {
    "conv_commit_early": 1,
    "commit_a_rows": 2,
    "verify_writes_live": 3,
    "taps_reversed": 4,
    "gqa_modulo": 5,
    "o_before_update": 6,
    "no_k_norm": 7,
    "no_scale": 8,
    "decay_after": 9,
    "no_beta": 10,
    "no_silu": 11,
}
DEFAULT_EPS = 1e-6


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("B", "R", "H_qk", "H_v", "d_k", "d_v", "W", "P")] + [
        ("scale", ctypes.c_double),
        ("l2_eps", ctypes.c_double),
    ]


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(str(_build.build()))
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int)
        lib.oracle_gdn_verify_commit.argtypes = [
            ctypes.POINTER(_Dims), dp, dp, dp, dp, dp, dp, ip, ip, ip, dp, dp, dp, ctypes.c_int]
        lib.oracle_gdn_verify_commit.restype = ctypes.c_int
        lib.oracle_gdn_gating.argtypes = [ctypes.c_long, ctypes.c_int, dp, dp, dp, dp, dp]
        lib.oracle_gdn_gating.restype = None
        lib.oracle_greedy_accept.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_long, dp, ip, ip, ip, ip]
        lib.oracle_greedy_accept.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # torch tensor: widen exactly (bf16/fp32 -> fp64)
        import torch
        a = a.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a, ty):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ty))


def gating(a, b, A_log):
    """g = -exp(A_log) softplus(a), beta = sigmoid(b) per row and value head
    (fp64, ``oracle_gdn_gating``); a, b are [..][H_v], A_log is [H_v]."""
    a64, b64 = _f64(a), _f64(b)
    shape = a64.shape
    hv = shape[-1]
    n = a64.size // hv
    g = np.empty(shape)
    beta = np.empty(shape)
    dp = ctypes.c_double
    _load().oracle_gdn_gating(n, hv, _ptr(_f64(A_log), dp), _ptr(a64, dp), _ptr(b64, dp),
                              _ptr(g, dp), _ptr(beta, dp))
    return g, beta


def verify_commit(layer: dict, *, commit: bool = True, snapshot: bool = False,
                  accept_len=None, scale: float | None = None, l2_eps: float = DEFAULT_EPS,
                  mutation: int | str = 0, requests=None, raw_gating: bool = False) -> dict:
    """Run the oracle on one layer call (the dict ``inputs.make_layer`` returns).

    commit=False is a verify-only call (slots untouched).  ``requests``
    restricts the call to a subset of request indices (for sampled checks at
    full size); the other requests are treated as inactive.  raw_gating=True
    forms g and beta from the layer's raw projections a_raw, b_raw and A_log.  Returns fp64
    numpy arrays: o [B][R][H_v][d_v] (NaN where not produced), the slot pools
    after the call, the status bits, and with snapshot=True the per-row
    states and conv windows."""
    spec = layer["spec"]
    B, R, C, W = spec.B, spec.R, spec.C, spec.W
    dims = _Dims(B, R, spec.H_qk, spec.H_v, spec.d_k, spec.d_v, W, spec.pool_slots,
                 spec.d_k ** -0.5 if scale is None else scale, l2_eps)
    x, g, beta = _f64(layer["x"]), _f64(layer["g"]), _f64(layer["beta"])
    if raw_gating:  # the layer's raw gating projections instead of g and beta
        g, beta = gating(layer["a_raw"], layer["b_raw"], layer["A_log"])
    conv_w = _f64(layer["conv_w"])
    conv_state = _f64(layer["conv_state"]).copy()
    ssm_state = _f64(layer["ssm_state"]).copy()
    slots = _i32(layer["slot_ids"])
    n_rows = _i32(layer["n_rows"]).copy()
    if requests is not None:
        keep = np.zeros(B, dtype=bool)
        keep[np.asarray(list(requests), dtype=np.int64)] = True
        n_rows[~keep] = 0
    acc = _i32(layer["accept_len"] if accept_len is None else accept_len) if commit else None
    o = np.full((B, R, spec.H_v, spec.d_v), np.nan)
    snap_S = np.full((B, R) + ssm_state.shape[1:], np.nan) if snapshot else None
    snap_cs = np.full((B, R, C, W - 1), np.nan) if snapshot else None
    mut = MUTATIONS[mutation] if isinstance(mutation, str) else int(mutation)
    dp, ip = ctypes.c_double, ctypes.c_int
    t0 = time.perf_counter()
    status = _load().oracle_gdn_verify_commit(
        ctypes.byref(dims), _ptr(x, dp), _ptr(g, dp), _ptr(beta, dp), _ptr(conv_w, dp),
        _ptr(conv_state, dp), _ptr(ssm_state, dp), _ptr(slots, ip), _ptr(n_rows, ip),
        _ptr(acc, ip), _ptr(o, dp), _ptr(snap_S, dp), _ptr(snap_cs, dp), mut)
    seconds = time.perf_counter() - t0
    out = {"o": o, "ssm_state": ssm_state, "conv_state": conv_state, "status": int(status),
           "seconds": seconds}
    if snapshot:
        out["snap_S"], out["snap_cs"] = snap_S, snap_cs
    return out


def verify_commit_threads(layer: dict, threads: int, *, scale: float | None = None,
                          l2_eps: float = DEFAULT_EPS) -> dict:
    """``verify_commit`` (fused verify + commit) with the requests spread over
    ``threads`` host threads: thread i runs the same C routine on requests
    b = i, i + threads, ... with the others masked inactive.  Requests touch
    disjoint slots and output rows, and the routine keeps no state between
    calls, so the threads share the arrays and the result equals
    ``verify_commit``'s exactly.  ctypes releases the interpreter lock during
    each C call, so the threads run in parallel.  ``seconds`` is the wall time
    of the parallel region (marshalling excluded, as in ``verify_commit``)."""
    from concurrent.futures import ThreadPoolExecutor

    spec = layer["spec"]
    B, R, C, W = spec.B, spec.R, spec.C, spec.W
    dims = _Dims(B, R, spec.H_qk, spec.H_v, spec.d_k, spec.d_v, W, spec.pool_slots,
                 spec.d_k ** -0.5 if scale is None else scale, l2_eps)
    x, g, beta = _f64(layer["x"]), _f64(layer["g"]), _f64(layer["beta"])
    conv_w = _f64(layer["conv_w"])
    conv_state = _f64(layer["conv_state"]).copy()
    ssm_state = _f64(layer["ssm_state"]).copy()
    slots = _i32(layer["slot_ids"])
    n_all = _i32(layer["n_rows"])
    acc = _i32(layer["accept_len"])
    o = np.full((B, R, spec.H_v, spec.d_v), np.nan)
    threads = max(1, min(int(threads), B))
    masks = []
    for i in range(threads):
        n = np.zeros_like(n_all)
        n[i::threads] = n_all[i::threads]
        masks.append(n)
    lib = _load()
    dp, ip = ctypes.c_double, ctypes.c_int

    def run(n):
        return lib.oracle_gdn_verify_commit(
            ctypes.byref(dims), _ptr(x, dp), _ptr(g, dp), _ptr(beta, dp), _ptr(conv_w, dp),
            _ptr(conv_state, dp), _ptr(ssm_state, dp), _ptr(slots, ip), _ptr(n, ip),
            _ptr(acc, ip), _ptr(o, dp), None, None, 0)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        t0 = time.perf_counter()
        statuses = list(ex.map(run, masks))
        seconds = time.perf_counter() - t0
    status = 0
    for st in statuses:
        status |= int(st)
    return {"o": o, "ssm_state": ssm_state, "conv_state": conv_state, "status": status,
            "seconds": seconds, "threads": threads}


def verify_deferred(cur: dict, prev: dict | None = None, *, requests=None, scale: float | None = None,
                    l2_eps: float = DEFAULT_EPS, raw_gating: bool = False) -> dict:
    """Deferred commit on the CPU, by its definition: the previous step's rows
    0..accept_len are committed (a commit of ``prev`` that replays them from
    the slots), then the current rows are verified from the committed slots.

    ``cur`` holds the current step's rows and the weights, slot ids and slot
    pools as they stand before the previous step's commit; ``prev`` (None =
    nothing pending) holds the previous step's x, g, beta (a_raw, b_raw),
    n_rows and accept_len, its own spec giving its rows per request.  Both
    oracle calls run over ``requests`` only.  Returns o of the current rows,
    the pools after the call and the OR of both calls' status bits."""
    pools, status, seconds = cur, 0, 0.0
    if prev is not None:
        step = dict(prev)
        for key in ("conv_w", "conv_state", "ssm_state", "slot_ids", "A_log"):
            step[key] = cur[key]
        r1 = verify_commit(step, commit=True, requests=requests, scale=scale, l2_eps=l2_eps,
                           raw_gating=raw_gating)
        pools = dict(cur, conv_state=r1["conv_state"], ssm_state=r1["ssm_state"])
        status, seconds = r1["status"], r1["seconds"]
    r2 = verify_commit(pools, commit=False, requests=requests, scale=scale, l2_eps=l2_eps,
                       raw_gating=raw_gating)
    return {"o": r2["o"], "ssm_state": r2["ssm_state"], "conv_state": r2["conv_state"],
            "status": status | r2["status"], "seconds": seconds + r2["seconds"]}


def greedy_accept(case: dict) -> dict:
    """Greedy acceptance on the CPU (``oracle_greedy_accept``) for the dict
    ``inputs.make_accept_case`` returns: target [B][R] (-1 where no row) and
    accept_len [B]."""
    logits = _f64(case["logits"])
    B, R, V = logits.shape
    drafts = _i32(case["drafts"]) if R > 1 else np.zeros((B, 1), dtype=np.int32)
    n_rows = _i32(case["n_rows"])
    target = np.full((B, R), -1, dtype=np.int32)
    acc = np.zeros(B, dtype=np.int32)
    ip = ctypes.c_int
    status = _load().oracle_greedy_accept(B, R, V, _ptr(logits, ctypes.c_double), _ptr(drafts, ip),
                                          _ptr(n_rows, ip), _ptr(target, ip), _ptr(acc, ip))
    return {"target": target, "accept_len": acc, "status": int(status)}

"""Seeded synthetic inputs for one GatedDeltaNet verify/commit layer call.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests.  It draws random numbers and casts them to the storage dtypes;
it holds none of the method's arithmetic (no convolution, normalisation or
delta-rule step).  The only arithmetic here is the input recipe itself:
the per-head log-decay ``g = -exp(A_log) * softplus(x)`` and ``beta =
sigmoid(z)`` that a Qwen3.5-style gated delta layer feeds its recurrence.

Random draws use numpy's PCG64 generator so that a seed gives the same
numbers on x86 and on Arm; casts to bf16 round to nearest-even via torch.

Shapes (all row-major):
  x          [B][R][C]            pre-conv mixed q|k|v rows, C = 2*H_qk*d_k + H_v*d_v
  g, beta    [B][R][H_v]  fp32    log-decay (<= 0) and write strength in (0, 1)
  conv_w     [C][W]               depthwise causal conv taps, tap W-1 hits the newest row
  conv_state [P][C][W-1]          committed conv window per slot, oldest column first
  ssm_state  [P][H_v][d_v][d_k]   fp32 committed delta-rule state per slot
  slot_ids   [B] int32            request -> slot
  n_rows     [B] int32            valid rows (k_b + 1), 0 = inactive request
  accept_len [B] int32            accepted drafts a_b in 0..k_b (commit a_b + 1 rows)
  a_raw, b_raw [B][R][H_v] fp32   the raw projections x and z above (for raw-gating calls)
  A_log      [H_v] fp32           the per-head decay parameter above
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch

__all__ = ["LayerSpec", "make_layer", "make_step", "CONFIGS", "workload_layers", "spec_bytes", "deferred_bytes"]


@dataclass(frozen=True)
class LayerSpec:
    """One layer call's shape and input recipe."""

    name: str
    B: int
    k: int                      # drafts per request (rows = k + 1); k_max when ragged
    H_qk: int
    H_v: int
    d_k: int
    d_v: int
    W: int = 4
    dtype: str = "bf16"         # storage type of x, conv_w, conv_state: "bf16" | "f32"
    accept: str = "uniform"     # "uniform" | "binom:<n>:<p>" | "fixed:<a0>,<a1>,..."
    pool: str = "perm"          # "identity" | "perm" | "double"
    k_choices: tuple = ()       # ragged: per-request k drawn uniformly from these
    inactive_frac: float = 0.0  # fraction of requests masked out (n_rows = 0)
    s_std: float = 0.02         # std of the initial SSM state

    @property
    def R(self) -> int:
        return self.k + 1

    @property
    def C(self) -> int:
        return 2 * self.H_qk * self.d_k + self.H_v * self.d_v

    @property
    def pool_slots(self) -> int:
        return 2 * self.B if self.pool == "double" else self.B

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4


def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def _store(a: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def make_layer(spec: LayerSpec, seed: int) -> dict:
    """Draw one layer call's inputs on the CPU.  Same seed -> same tensors."""
    rng = np.random.Generator(np.random.PCG64(seed))
    B, R, C, W = spec.B, spec.R, spec.C, spec.W
    H_v, d_v, d_k, P = spec.H_v, spec.d_v, spec.d_k, spec.pool_slots

    x = _normal(rng, (B, R, C), 1.0)
    conv_w = _normal(rng, (C, W), 0.5)
    conv_state = _normal(rng, (P, C, W - 1), 1.0)
    ssm_state = _normal(rng, (P, H_v, d_v, d_k), spec.s_std)

    # gating recipe of a Qwen3.5-style GDN layer: g = -exp(A_log) * softplus(x)
    a_log = rng.uniform(0.0, math.log(16.0), size=(H_v,))
    gx = rng.standard_normal(size=(B, R, H_v))
    g = -np.exp(a_log)[None, None, :] * np.logaddexp(0.0, gx)
    bz = rng.standard_normal(size=(B, R, H_v))
    beta = 1.0 / (1.0 + np.exp(-bz))

    if spec.k_choices:
        ks = rng.choice(np.asarray(spec.k_choices), size=B)
        assert ks.max() <= spec.k
    else:
        ks = np.full(B, spec.k)
    n_rows = (ks + 1).astype(np.int64)

    if spec.accept.startswith("fixed:"):
        acc = np.asarray([int(v) for v in spec.accept[6:].split(",")], dtype=np.int64)
        assert acc.shape == (B,)
    elif spec.accept.startswith("binom:"):
        _, nn, p = spec.accept.split(":")
        acc = np.minimum(rng.binomial(int(nn), float(p), size=B), ks)
    elif spec.accept == "uniform":
        acc = rng.integers(0, ks + 1)
    else:
        raise ValueError(spec.accept)

    if spec.pool == "identity":
        slots = np.arange(B)
    elif spec.pool == "perm":
        slots = rng.permutation(B)
    elif spec.pool == "double":
        slots = rng.choice(2 * B, size=B, replace=False)
    else:
        raise ValueError(spec.pool)

    n_inactive = int(round(spec.inactive_frac * B))
    if n_inactive:
        off = rng.choice(B, size=n_inactive, replace=False)
        n_rows[off] = 0
        acc[off] = 0

    return {
        "spec": spec,
        "seed": seed,
        "x": _store(x, spec.dtype),
        "conv_w": _store(conv_w, spec.dtype),
        "conv_state": _store(conv_state, spec.dtype),
        "ssm_state": torch.from_numpy(ssm_state),
        "g": torch.from_numpy(g.astype(np.float32)),
        "beta": torch.from_numpy(beta.astype(np.float32)),
        # the raw gating projections g and beta come from (for callers that
        # pass them with the raw-gating flag)
        "a_raw": torch.from_numpy(gx.astype(np.float32)),
        "b_raw": torch.from_numpy(bz.astype(np.float32)),
        "A_log": torch.from_numpy(a_log.astype(np.float32)),
        "slot_ids": torch.from_numpy(slots.astype(np.int32)),
        "n_rows": torch.from_numpy(n_rows.astype(np.int32)),
        "accept_len": torch.from_numpy(acc.astype(np.int32)),
    }


def make_step(prev: dict, spec: LayerSpec, seed: int) -> dict:
    """The same layer's inputs at the next decode step: fresh rows, gating,
    row counts and accept counts drawn as ``make_layer`` draws them (spec may
    change k, not B, the head shapes, dtype or pool), with prev's weights,
    A_log, slot ids and slot pools carried over."""
    p = prev["spec"]
    assert (spec.B, spec.H_qk, spec.H_v, spec.d_k, spec.d_v, spec.W, spec.dtype, spec.pool_slots) == \
        (p.B, p.H_qk, p.H_v, p.d_k, p.d_v, p.W, p.dtype, p.pool_slots)
    step = make_layer(spec, seed)
    for key in ("conv_w", "conv_state", "ssm_state", "slot_ids", "A_log"):
        step[key] = prev[key]
    return step


_QWEN = dict(H_qk=16, H_v=32, d_k=128, d_v=128)

#: The workloads, by name.  The batch sweep and the 36-layer stack expand into
#: individual layer calls through ``workload_layers``.
TINY = "tiny-fp32"
SINGLE = "qwen35-B1-k3"
SWEEP = "qwen35-sweep-k2"
STACK = "qwen35-36L-B16-k3"
RAGGED = "ragged-B256-k1_3_8"

CONFIGS = {
    TINY: LayerSpec(TINY, B=2, k=2, H_qk=2, H_v=4, d_k=16, d_v=16, dtype="f32",
                    accept="fixed:0,2", pool="identity"),
    SINGLE: LayerSpec(SINGLE, B=1, k=3, accept="uniform", pool="identity", **_QWEN),
    SWEEP: LayerSpec(SWEEP, B=16, k=2, accept="binom:2:0.72", pool="double", **_QWEN),
    STACK: LayerSpec(STACK, B=16, k=3, accept="uniform", pool="perm", **_QWEN),
    RAGGED: LayerSpec(RAGGED, B=256, k=8, H_qk=16, H_v=64, d_k=128, d_v=128,
                      accept="uniform", pool="perm", k_choices=(1, 3, 8), inactive_frac=0.1),
}

SWEEP_B = (1, 2, 4, 8, 16, 32, 64)
STACK_LAYERS = 36
_SEED_BASE = {TINY: 0, SINGLE: 1000, SWEEP: 2000, STACK: 3000, RAGGED: 4000}


def workload_layers(name: str, batch: int | None = None, layers: int | None = None):
    """(spec, seed) pairs of one workload's layer calls.

    Seeds: tiny 0, single-request 1000, batch sweep 2000 + B (one layer per
    batch size), stack 3000 + layer index, ragged 4000."""
    base, seed0 = CONFIGS[name], _SEED_BASE[name]
    if name == SWEEP:
        bs = SWEEP_B if batch is None else (batch,)
        return [(replace(base, B=b, name=f"qwen35-B{b}-k2"), seed0 + b) for b in bs]
    if name == STACK:
        n = STACK_LAYERS if layers is None else layers
        return [(base, seed0 + layer) for layer in range(n)]
    return [(base, seed0)]


def spec_bytes(spec: LayerSpec, n_rows) -> int:
    """Fused-minimum algorithmic bytes of one verify+commit call.

    Per active request (n valid rows): SSM state read + write, conv state
    read + write, n rows of x, n rows of g and beta, n rows of o; plus the
    conv weights once per call."""
    s = 2 * spec.H_v * spec.d_v * spec.d_k * 4
    cs = 2 * spec.C * (spec.W - 1) * spec.elem_bytes
    per_row = spec.C * spec.elem_bytes + spec.H_v * 8 + spec.H_v * spec.d_v * 4
    total = spec.C * spec.W * spec.elem_bytes
    for n in (int(v) for v in n_rows):
        if n > 0:
            total += s + cs + n * per_row
    return total


def deferred_bytes(spec: LayerSpec, n_rows, n_prev, acc_prev) -> int:
    """Algorithmic bytes of one deferred-commit call: ``spec_bytes``'s terms
    for every request with current or pending rows; for a request with
    pending rows, those rows' x (acc_prev + 1 rows, for the conv window) and
    their carry (per row: H_v d_v update values, H_qk d_k of k^, H_v decays)
    read; and the carry of the current rows written."""
    s = 2 * spec.H_v * spec.d_v * spec.d_k * 4
    cs = 2 * spec.C * (spec.W - 1) * spec.elem_bytes
    per_row = spec.C * spec.elem_bytes + spec.H_v * 8 + spec.H_v * spec.d_v * 4
    carry_row = (spec.H_v * spec.d_v + spec.H_qk * spec.d_k + spec.H_v) * 4
    total = spec.C * spec.W * spec.elem_bytes
    for n, np_, a in zip((int(v) for v in n_rows), (int(v) for v in n_prev), (int(v) for v in acc_prev)):
        if n > 0 or np_ > 0:
            total += s + cs + max(n, 0) * (per_row + carry_row)
        if np_ > 0:
            total += (a + 1) * (spec.C * spec.elem_bytes + carry_row)
    return total


def make_accept_case(B: int, R: int, V: int, seed: int, dtype: str = "bf16", inactive: int = 0,
                     ties: bool = True) -> dict:
    """Target logits and drafts of one greedy-acceptance call, with the
    answers planted by construction rather than computed.

    Logits are N(0, 1) clipped to [-6, 6]; each valid row gets one planted
    token at +8, so that token is the row's largest value (with ``ties``,
    some rows also get a second +8 at a higher index, which must lose to the
    lower one).  Request b accepts a_b ~ U{0..k_b} drafts: drafts up to a_b
    copy the planted tokens of the rows before them, the next one differs.
    Returns logits, drafts [B][R-1], n_rows, and the planted target and
    accept_len."""
    rng = np.random.Generator(np.random.PCG64(seed))
    logits = np.clip(rng.standard_normal((B, R, V)), -6.0, 6.0)
    n_rows = rng.integers(1, R + 1, size=B)
    if inactive:
        n_rows[rng.choice(B, size=inactive, replace=False)] = 0
    planted = rng.integers(0, V - 1, size=(B, R))
    for b in range(B):
        for t in range(R):
            logits[b, t, planted[b, t]] = 8.0
            if ties and (b + t) % 3 == 0:
                logits[b, t, rng.integers(planted[b, t] + 1, V)] = 8.0  # a later equal maximum
    acc = np.array([rng.integers(0, max(int(n), 1)) if n > 0 else 0 for n in n_rows])
    drafts = rng.integers(0, V, size=(B, max(R - 1, 1)))
    for b in range(B):
        for i in range(R - 1):
            if i < acc[b]:
                drafts[b, i] = planted[b, i]
            elif i == acc[b]:
                drafts[b, i] = (planted[b, i] + 1) % V
    store = torch.bfloat16 if dtype == "bf16" else torch.float32
    return {
        "logits": torch.from_numpy(logits.astype(np.float32)).to(store),
        "drafts": torch.from_numpy(drafts[:, :max(R - 1, 1)].astype(np.int32)),
        "n_rows": torch.from_numpy(n_rows.astype(np.int32)),
        "planted_target": planted.astype(np.int32),
        "planted_accept": acc.astype(np.int32),
    }

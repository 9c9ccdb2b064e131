"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself through the same code path:
each pin is an invariant the pages state, a closed form computed by a second
algorithm (library conv1d + explicit transition-matrix products), or a
special case with a known answer.  ``test_every_mutation_is_caught`` plants
each deliberate mistake the oracle can switch on and checks that at least one
pin fails on it.

Pinned:
  * verify == k+1 sequential decode steps; commit(a) == a+1 steps
    [FreeToken #844, Tests: test_verify_commit_matches_stepwise_decode]
  * verify-only leaves the slots bitwise untouched [FreeToken #828, Design]
  * conv window: tap W-1 on the newest row, committed window = last W-1 entries
    of [history | accepted rows] [FreeToken #844, Flash-Next target verify;
    Tests: a mutation that shifts the committed window by one column]
  * the delta rule, decay, write strength, scale, L2 norm, SiLU: closed form
    and special cases (beta=0 pure decay, beta=1 exact write S k = v,
    orthonormal keys keep every written value)
  * value head h reads q/k head h // (H_v / H_qk): one-hot q per q/k head.
  * the raw gating g = -exp(A_log) softplus(a), beta = sigmoid(b): torch's own
    softplus and sigmoid (library routines), including tails where the naive
    forms overflow.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from speculative_decode_gateddeltanet_gb300.inputs import CONFIGS, TINY, LayerSpec, make_layer


# ----------------------------------------------------------------- helpers
def tiny_layer(seed=0, **over):
    spec = over.pop("spec", CONFIGS[TINY])
    layer = make_layer(spec, seed)
    for k, v in over.items():
        layer[k] = v
    return layer


def small_spec(B=2, k=3, H_qk=1, H_v=2, d=4, W=4):
    return LayerSpec("pin", B=B, k=k, H_qk=H_qk, H_v=H_v, d_k=d, d_v=d, W=W, dtype="f32",
                     accept="uniform", pool="identity")


def f64(t):
    return t.detach().double().numpy() if hasattr(t, "detach") else np.asarray(t, np.float64)


def qkv_by_library(layer, l2_eps):
    """q, k, v for every (b, t) by a second route: torch conv1d over the staged
    [conv_state | x] sequence, torch SiLU, numpy L2 norm.  [B][R] lists."""
    spec = layer["spec"]
    C, W, Hq, dk = spec.C, spec.W, spec.H_qk, spec.d_k
    x, cs, w = f64(layer["x"]), f64(layer["conv_state"]), f64(layer["conv_w"])
    out = []
    for b in range(spec.B):
        s = int(layer["slot_ids"][b])
        n = int(layer["n_rows"][b])
        seq = np.concatenate([cs[s], x[b, :n].T], axis=1)  # [C][W-1+n]
        y = torch.nn.functional.conv1d(torch.from_numpy(seq)[None], torch.from_numpy(w)[:, None, :],
                                       groups=C)[0]
        y = torch.nn.functional.silu(y).numpy().T  # [n][C]
        rows = []
        for t in range(n):
            q = y[t, :Hq * dk].reshape(Hq, dk)
            k = y[t, Hq * dk:2 * Hq * dk].reshape(Hq, dk)
            v = y[t, 2 * Hq * dk:].reshape(spec.H_v, spec.d_v)
            q = q / np.sqrt((q * q).sum(-1, keepdims=True) + l2_eps)
            k = k / np.sqrt((k * k).sum(-1, keepdims=True) + l2_eps)
            rows.append((q, k, v))
        out.append(rows)
    return out


def closed_form(layer, l2_eps=oracle.DEFAULT_EPS, scale=None):
    """States and outputs by the transition-matrix form, unrolled:
    S_t = S_0 A_1..A_t + sum_s beta_s v_s k_s^T A_{s+1}..A_t,
    A_t = alpha_t (I - beta_t k_t k_t^T),  o_t = scale S_t q_t."""
    spec = layer["spec"]
    G = spec.H_v // spec.H_qk
    scale = spec.d_k ** -0.5 if scale is None else scale
    g, beta, S0 = f64(layer["g"]), f64(layer["beta"]), f64(layer["ssm_state"])
    qkv = qkv_by_library(layer, l2_eps)
    I = np.eye(spec.d_k)
    states, outs = {}, {}
    for b in range(spec.B):
        s = int(layer["slot_ids"][b])
        n = int(layer["n_rows"][b])
        for h in range(spec.H_v):
            hq = h // G
            A = [np.exp(g[b, t, h]) * (I - beta[b, t, h] * np.outer(qkv[b][t][1][hq], qkv[b][t][1][hq]))
                 for t in range(n)]

            def prod(i, j):  # A_i ... A_j (identity if empty)
                P = I.copy()
                for m in range(i, j + 1):
                    P = P @ A[m]
                return P

            for t in range(n):
                St = S0[s, h] @ prod(0, t)
                for u in range(t + 1):
                    k_u = qkv[b][u][1][hq]
                    St = St + beta[b, u, h] * np.outer(qkv[b][u][2][h], k_u) @ prod(u + 1, t)
                states[(b, t, h)] = St
                outs[(b, t, h)] = scale * St @ qkv[b][t][0][hq]
    return states, outs


def chained_steps(layer, n_steps, b, mutation=0, l2_eps=oracle.DEFAULT_EPS):
    """Run request b as n_steps one-row verify+commit calls (a = 0 each): the
    single-token decode steps.  Returns per-step o and the final slot pools."""
    spec = layer["spec"]
    one = LayerSpec("step", B=1, k=0, H_qk=spec.H_qk, H_v=spec.H_v, d_k=spec.d_k, d_v=spec.d_v,
                    W=spec.W, dtype=spec.dtype, pool="identity")
    s = int(layer["slot_ids"][b])
    cs = f64(layer["conv_state"])[s:s + 1].copy()
    S = f64(layer["ssm_state"])[s:s + 1].copy()
    os_ = []
    for t in range(n_steps):
        step = {"spec": one, "x": f64(layer["x"])[b:b + 1, t:t + 1], "g": f64(layer["g"])[b:b + 1, t:t + 1],
                "beta": f64(layer["beta"])[b:b + 1, t:t + 1], "conv_w": f64(layer["conv_w"]),
                "conv_state": cs, "ssm_state": S, "slot_ids": np.zeros(1, np.int32),
                "n_rows": np.ones(1, np.int32), "accept_len": np.zeros(1, np.int32)}
        r = oracle.verify_commit(step, mutation=mutation, l2_eps=l2_eps)
        os_.append(r["o"][0, 0])
        cs, S = r["conv_state"], r["ssm_state"]
    return np.stack(os_), S[0], cs[0]


# -------------------------------------------------------------------- pins
def pin_stepwise(mutation=0):
    """verify over k+1 rows == k+1 decode steps (o bitwise); commit at every a
    == a+1 decode steps (state and conv window bitwise)."""
    layer = tiny_layer()
    spec = layer["spec"]
    full = oracle.verify_commit(layer, commit=False, mutation=mutation)
    for b in range(spec.B):
        n = int(layer["n_rows"][b])
        o_steps, _, _ = chained_steps(layer, n, b, mutation)
        assert np.array_equal(full["o"][b, :n], o_steps), "verify rows != decode steps"
        s = int(layer["slot_ids"][b])
        for a in range(n):
            acc = layer["accept_len"].clone()
            acc[b] = a
            com = oracle.verify_commit(layer, accept_len=acc, mutation=mutation)
            _, S_a, cs_a = chained_steps(layer, a + 1, b, mutation)
            assert np.array_equal(com["ssm_state"][s], S_a), f"commit(a={a}) state != {a + 1} steps"
            assert np.array_equal(com["conv_state"][s], cs_a), f"commit(a={a}) conv != {a + 1} steps"


def pin_verify_read_only(mutation=0):
    layer = tiny_layer()
    r = oracle.verify_commit(layer, commit=False, mutation=mutation)
    assert np.array_equal(r["ssm_state"], f64(layer["ssm_state"]))
    assert np.array_equal(r["conv_state"], f64(layer["conv_state"]))


def pin_closed_form(mutation=0):
    """Rank-1 recurrence == unrolled transition-matrix products (1e-12)."""
    cases = [tiny_layer()]
    for i, d in enumerate((2, 3, 4)):
        spec = small_spec(d=d, k=3 + i, H_qk=1 + (d == 4), H_v=2 + 2 * (d == 4))
        cases.append(make_layer(spec, 100 + d))
    for layer in cases:
        spec = layer["spec"]
        r = oracle.verify_commit(layer, commit=False, mutation=mutation)
        states, outs = closed_form(layer)
        ref_scale = max(abs(v).max() for v in outs.values())
        for (b, t, h), ov in outs.items():
            assert np.allclose(r["o"][b, t, h], ov, rtol=0, atol=1e-12 * ref_scale), (b, t, h)
        # committed state at each request's accept_len
        c = oracle.verify_commit(layer, mutation=mutation)
        for b in range(spec.B):
            s, a = int(layer["slot_ids"][b]), int(layer["accept_len"][b])
            for h in range(spec.H_v):
                ref = states[(b, a, h)]
                assert np.allclose(c["ssm_state"][s, h], ref, rtol=0, atol=1e-12 * abs(ref).max())


def _one_hot_layer(d=8, H_qk=2, H_v=4, n=4, tap=3, g0=True, beta1=True, seed=5):
    """Conv taps = e_tap; q and k channels one-hot so that after SiLU and L2 norm
    q_t = k_t = e_{p(t, hq)} with p(t, hq) = (t + 2*hq) mod d (orthonormal
    across rows when n <= d).  v, conv history random."""
    spec = LayerSpec("onehot", B=1, k=n - 1, H_qk=H_qk, H_v=H_v, d_k=d, d_v=d, dtype="f32",
                     pool="identity")
    layer = make_layer(spec, seed)
    C, W = spec.C, spec.W
    w = np.zeros((C, W), np.float32)
    w[:, tap] = 1.0
    x = f64(layer["x"]).astype(np.float32)
    cs = f64(layer["conv_state"]).astype(np.float32)
    qk = slice(0, 2 * H_qk * d)
    x[:, :, qk] = 0.0
    cs[:, qk, :] = 0.0
    seq_len = W - 1 + n
    for m in range(seq_len):  # one-hot at every staged position the tap can hit
        t = m - tap
        for hq in range(H_qk):
            p = (t + 2 * hq) % d
            for base in (0, H_qk * d):
                if m < W - 1:
                    cs[0, base + hq * d + p, m] = 4.0
                else:
                    x[0, m - (W - 1), base + hq * d + p] = 4.0
    layer["conv_w"] = torch.from_numpy(w)
    layer["x"] = torch.from_numpy(x)
    layer["conv_state"] = torch.from_numpy(cs)
    if g0:
        layer["g"] = torch.zeros_like(layer["g"])
    if beta1:
        layer["beta"] = torch.ones_like(layer["beta"])
    return layer


def pin_exact_write_and_taps(mutation=0):
    """g=0, beta=1, orthonormal keys: S_t k_j = v_j for all j <= t, and
    o_t = scale * v_t (q_t = k_t).  v_t must be SiLU of the staged entry the
    tap selects: tap j at row t reads entry t+j of [history | rows]."""
    for tap in range(4):
        layer = _one_hot_layer(tap=tap)
        spec = layer["spec"]
        d, G, W = spec.d_k, spec.H_v // spec.H_qk, spec.W
        x, cs = f64(layer["x"]), f64(layer["conv_state"])
        C = spec.C
        seq = np.concatenate([cs[0], x[0].T], axis=1)  # [C][W-1+n]
        voff = 2 * spec.H_qk * d
        for a in range(spec.R):
            acc = torch.tensor([a], dtype=torch.int32)
            r = oracle.verify_commit(layer, accept_len=acc, l2_eps=0.0, mutation=mutation)
            S = r["ssm_state"][0]
            for h in range(spec.H_v):
                hq = h // G
                for t in range(a + 1):
                    p = (t + 2 * hq) % d
                    v_t = torch.nn.functional.silu(torch.from_numpy(seq[voff + h * d: voff + (h + 1) * d,
                                                                        t + tap])).numpy()
                    assert np.allclose(S[h][:, p], v_t, rtol=0, atol=1e-12), (tap, a, h, t)
                    assert np.allclose(r["o"][0, t, h], d ** -0.5 * v_t, rtol=0, atol=1e-12)
            # committed conv window: last W-1 staged entries after row a
            assert np.array_equal(r["conv_state"][0], seq[:, a + 1:a + W])
            assert C == seq.shape[0]


def pin_pure_decay(mutation=0):
    """beta = 0: the state only decays, S_a = exp(sum_{t<=a} g_t) S_0."""
    layer = tiny_layer()
    layer["beta"] = torch.zeros_like(layer["beta"])
    spec = layer["spec"]
    r = oracle.verify_commit(layer, mutation=mutation)
    g, S0 = f64(layer["g"]), f64(layer["ssm_state"])
    for b in range(spec.B):
        s, a = int(layer["slot_ids"][b]), int(layer["accept_len"][b])
        for h in range(spec.H_v):
            ref = np.exp(g[b, :a + 1, h].sum()) * S0[s, h]
            assert np.allclose(r["ssm_state"][s, h], ref, rtol=1e-13, atol=0)


def pin_identity_step(mutation=0):
    """g = 0, beta = 0: S unchanged bitwise, o_t = scale * S_0 q_t."""
    layer = tiny_layer()
    layer["g"] = torch.zeros_like(layer["g"])
    layer["beta"] = torch.zeros_like(layer["beta"])
    r = oracle.verify_commit(layer, mutation=mutation)
    assert np.array_equal(r["ssm_state"], f64(layer["ssm_state"]))
    spec = layer["spec"]
    qkv = qkv_by_library(layer, oracle.DEFAULT_EPS)
    S0 = f64(layer["ssm_state"])
    G = spec.H_v // spec.H_qk
    for b in range(spec.B):
        s = int(layer["slot_ids"][b])
        for t in range(int(layer["n_rows"][b])):
            for h in range(spec.H_v):
                ref = spec.d_k ** -0.5 * S0[s, h] @ qkv[b][t][0][h // G]
                assert np.allclose(r["o"][b, t, h], ref, rtol=0, atol=1e-13)


def pin_head_mapping(mutation=0):
    """One-hot q per q/k head, beta = 0, g = 0: o[h] = scale * S_0[h][:, p(hq)]
    picks the column of q/k head h // G."""
    layer = _one_hot_layer(tap=3, beta1=False, H_qk=2, H_v=4)
    layer["beta"] = torch.zeros_like(layer["beta"])
    spec = layer["spec"]
    d, G = spec.d_k, spec.H_v // spec.H_qk
    r = oracle.verify_commit(layer, commit=False, l2_eps=0.0, mutation=mutation)
    S0 = f64(layer["ssm_state"])[0]
    for t in range(spec.R):
        for h in range(spec.H_v):
            p = (t + 2 * (h // G)) % d
            assert np.allclose(r["o"][0, t, h], d ** -0.5 * S0[h][:, p], rtol=1e-14, atol=0)


def pin_status_and_masking(mutation=0):
    """Inactive requests produce nothing; a bad slot or row count skips the
    request with a status bit; a bad accept_len keeps o but skips the commit."""
    layer = tiny_layer()
    spec = layer["spec"]
    base = oracle.verify_commit(layer, mutation=mutation)
    m = dict(layer)
    m["n_rows"] = torch.tensor([0, 3], dtype=torch.int32)
    r = oracle.verify_commit(m, mutation=mutation)
    assert np.isnan(r["o"][0]).all() and r["status"] == 0
    assert np.array_equal(r["ssm_state"][0], f64(layer["ssm_state"])[0])
    assert np.array_equal(r["o"][1], base["o"][1])
    m["n_rows"] = torch.tensor([3, 3], dtype=torch.int32)
    m["slot_ids"] = torch.tensor([0, spec.pool_slots], dtype=torch.int32)
    r = oracle.verify_commit(m, mutation=mutation)
    assert r["status"] == oracle.BAD_SLOT and np.isnan(r["o"][1]).all()
    m["slot_ids"] = layer["slot_ids"]
    m["n_rows"] = torch.tensor([3, spec.R + 1], dtype=torch.int32)
    r = oracle.verify_commit(m, mutation=mutation)
    assert r["status"] == oracle.BAD_NROWS
    m["n_rows"] = layer["n_rows"]
    r = oracle.verify_commit(m, accept_len=torch.tensor([0, 3], dtype=torch.int32), mutation=mutation)
    assert r["status"] == oracle.BAD_ACCEPT
    assert np.array_equal(r["o"][1], base["o"][1])
    assert np.array_equal(r["ssm_state"][1], f64(layer["ssm_state"])[1])


def pin_snapshots(mutation=0):
    """The per-row snapshot at row t equals what a commit at a = t writes."""
    layer = tiny_layer()
    spec = layer["spec"]
    snap = oracle.verify_commit(layer, commit=False, snapshot=True, mutation=mutation)
    for b in range(spec.B):
        s = int(layer["slot_ids"][b])
        for t in range(int(layer["n_rows"][b])):
            acc = layer["accept_len"].clone()
            acc[b] = t
            c = oracle.verify_commit(layer, accept_len=acc, mutation=mutation)
            assert np.array_equal(snap["snap_S"][b, t], c["ssm_state"][s])
            assert np.array_equal(snap["snap_cs"][b, t], c["conv_state"][s])


PINS = [pin_stepwise, pin_verify_read_only, pin_closed_form, pin_exact_write_and_taps,
        pin_pure_decay, pin_identity_step, pin_head_mapping, pin_status_and_masking, pin_snapshots]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(0)


@pytest.mark.parametrize("mutation", sorted(oracle.MUTATIONS))
def test_every_mutation_is_caught(mutation):
    failed = []
    for pin in PINS:
        try:
            pin(oracle.MUTATIONS[mutation])
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin catches mutation {mutation}"


# ------------------------------------------------------------ raw gating
def test_raw_gating_matches_library_softplus_and_sigmoid():
    """oracle.gating against torch.nn.functional.softplus / torch.sigmoid in
    fp64, with values pushed into both tails; and a raw-gating call equals a
    call given torch's g and beta."""
    layer = tiny_layer(seed=5)
    a = layer["a_raw"].double().clone()
    b = layer["b_raw"].double().clone()
    a[0, 0, 0], a[0, 1, 0], a[1, 0, 1] = 80.0, -80.0, 1e-9
    b[0, 0, 1], b[0, 1, 1], b[1, 0, 0] = 60.0, -60.0, 0.0
    A_log = layer["A_log"].double()
    g_ref = -torch.exp(A_log) * torch.nn.functional.softplus(a, threshold=1000.0)
    beta_ref = torch.sigmoid(b)
    g, beta = oracle.gating(a, b, A_log)
    np.testing.assert_allclose(g, g_ref.numpy(), rtol=1e-14, atol=1e-300)
    np.testing.assert_allclose(beta, beta_ref.numpy(), rtol=1e-14, atol=1e-300)
    assert beta[0, 1, 1] > 0.0 and beta[0, 0, 1] <= 1.0 and np.all(g <= 0.0)

    raw = oracle.verify_commit(dict(layer, a_raw=a, b_raw=b), raw_gating=True)
    given = oracle.verify_commit(dict(layer, g=g_ref, beta=beta_ref))
    valid = ~np.isnan(given["o"])
    np.testing.assert_allclose(raw["o"][valid], given["o"][valid], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(raw["ssm_state"], given["ssm_state"], rtol=1e-13, atol=1e-15)
    assert np.array_equal(raw["conv_state"], given["conv_state"])


def test_raw_gating_tails_reduce_to_the_special_cases():
    """a -> -inf gives g = 0 (no decay) and b -> +inf gives beta = 1, so the
    raw call reduces to the exact-write case S k = v of the precomputed one."""
    layer = tiny_layer(seed=6)
    big = torch.full_like(layer["a_raw"], 1e4)
    raw = oracle.verify_commit(dict(layer, a_raw=-big, b_raw=big), raw_gating=True)
    given = oracle.verify_commit(dict(layer, g=torch.zeros_like(big), beta=torch.ones_like(big)))
    valid = ~np.isnan(given["o"])
    assert np.array_equal(raw["o"][valid], given["o"][valid])
    assert np.array_equal(raw["ssm_state"], given["ssm_state"])

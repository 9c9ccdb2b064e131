"""CUDA-graph capture of whole verify/commit sequences through the C ABI: the
library allocates nothing and never synchronises, so a captured multi-layer
step replays to the same bits as the same calls launched eagerly (the
pages' capture-safe verify with no device-to-host sync), and the replayed
results match the oracle run on the same sequence of calls under the stated
tolerances."""
from __future__ import annotations

import pytest
import torch

import oracle
from gpu_util import bits, check_against_oracle
from speculative_decode_gateddeltanet_gb300.inputs import STACK, SWEEP, make_layer, workload_layers

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _layers(name, **kw):
    return [make_layer(spec, seed) for spec, seed in workload_layers(name, **kw)]


def _reset(devs, layers):
    for d, layer in zip(devs, layers):
        for k in d.KEYS:
            getattr(d, k).copy_(layer[k])
        d.o.fill_(float("nan"))
        d.status.zero_()


def _same(a, b):
    for x, y in zip(a, b):
        assert torch.equal(bits(x.o), bits(y.o))
        assert torch.equal(bits(x.ssm_state), bits(y.ssm_state))
        assert torch.equal(bits(x.conv_state), bits(y.conv_state))
        assert int(x.status.item()) == int(y.status.item()) == 0


@pytest.mark.parametrize("mode,stable", [("fused", False), ("replay", False), ("fused", True), ("replay", True)])
def test_captured_stack_replays_to_eager_bits(mode, stable):
    """Six stack layers captured as one graph (optionally with
    GDN_FLAG_STATE_STABLE, as the benchmark runs them), replayed twice from
    the same buffers: eager bits each time, and the oracle's results."""
    from speculative_decode_gateddeltanet_gb300 import gdn

    layers = _layers(STACK, layers=6)
    eager = [gdn.DeviceLayer(layer, "cuda") for layer in layers]
    graphed = [gdn.DeviceLayer(layer, "cuda") for layer in layers]
    for d in eager + graphed:
        d.state_stable = stable
    stream = torch.cuda.Stream()

    def step(devs, args):
        for a in args:
            if mode == "fused":
                gdn.gdn_verify_commit(a, stream)
            else:
                gdn.gdn_verify(a, gdn.REPLAY, stream)
                gdn.gdn_commit(a, gdn.REPLAY, stream)

    eargs = [d.args() for d in eager]
    with torch.cuda.stream(stream):
        step(eager, eargs)
    torch.cuda.synchronize()

    gargs = [d.args() for d in graphed]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step(graphed, gargs)
    torch.cuda.synchronize()
    # capture records the launches without running them
    assert all(torch.isnan(d.o).all() for d in graphed)
    assert all(torch.equal(d.ssm_state.cpu(), layer["ssm_state"]) for d, layer in zip(graphed, layers))

    for _ in range(2):  # replay from the same starting buffers twice
        _reset(graphed, layers)
        g.replay()
        torch.cuda.synchronize()
        _same(eager, graphed)
    for layer, d in zip(layers, graphed):
        check_against_oracle(layer, d, oracle.verify_commit(layer), commit=True)


def test_captured_step_sequence_matches_eager_steps():
    """Three decode steps of one layer: the captured step replayed three
    times equals three eager steps (each commit feeds the next verify)."""
    from speculative_decode_gateddeltanet_gb300 import gdn

    (layer,) = _layers(SWEEP, batch=8)
    eager = gdn.DeviceLayer(layer, "cuda")
    graphed = gdn.DeviceLayer(layer, "cuda")
    stream = torch.cuda.Stream()
    ea, ga = eager.args(), graphed.args()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        gdn.gdn_verify_commit(ea, stream)  # the library's per-kernel setup runs outside the capture
    torch.cuda.synchronize()
    _reset([eager], [layer])
    with torch.cuda.graph(g, stream=stream):
        gdn.gdn_verify_commit(ga, stream)
    for _ in range(3):
        with torch.cuda.stream(stream):
            gdn.gdn_verify_commit(ea, stream)
        g.replay()
    torch.cuda.synchronize()
    _same([eager], [graphed])
    # the oracle's three steps, each starting from the pools the step before committed
    pools = {"conv_state": layer["conv_state"], "ssm_state": layer["ssm_state"]}
    for _ in range(3):
        ref = oracle.verify_commit(dict(layer, **pools))
        pools = {"conv_state": torch.from_numpy(ref["conv_state"]).to(layer["conv_state"].dtype),
                 "ssm_state": torch.from_numpy(ref["ssm_state"])}  # the oracle's chain stays in fp64
    check_against_oracle(layer, graphed, ref, commit=True)


def test_captured_deferred_steps_match_eager():
    """Two deferred steps of one layer: the first (nothing pending) writes its
    carry, the second commits the first's accepted rows from that carry and
    writes its own.  The pair captured as one graph and replayed equals the
    same calls launched eagerly, bit for bit: o, both carries and the pools."""
    from speculative_decode_gateddeltanet_gb300 import gdn
    from speculative_decode_gateddeltanet_gb300.inputs import make_step

    (first,) = _layers(STACK, layers=1)
    second = make_step(first, first["spec"], 3100)
    stream = torch.cuda.Stream()

    def build():
        d1 = gdn.DeviceLayer(first, "cuda")
        d2 = gdn.DeviceLayer(second, "cuda")
        d2.conv_state, d2.ssm_state = d1.conv_state, d1.ssm_state  # one slot pool
        a1, a2 = d1.args(), d2.args()
        d1.carry = torch.zeros(gdn.carry_bytes(a1) // 4, device="cuda")
        d2.carry = torch.zeros(gdn.carry_bytes(a2) // 4, device="cuda")
        a1.carry, a2.carry = d1.carry.data_ptr(), d2.carry.data_ptr()
        prev = gdn.make_prev(x=d1.x, n_rows=d1.n_rows, accept_len=d1.accept_len, carry=d1.carry)
        return d1, d2, a1, a2, prev

    def step(a1, a2, prev):
        gdn.gdn_verify_deferred(a1, None, stream)
        gdn.gdn_verify_deferred(a2, prev, stream)

    e1, e2, ea1, ea2, eprev = build()
    with torch.cuda.stream(stream):
        step(ea1, ea2, eprev)
    torch.cuda.synchronize()
    g1, g2, ga1, ga2, gprev = build()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step(ga1, ga2, gprev)
    g.replay()
    torch.cuda.synchronize()
    for x, y in ((e1, g1), (e2, g2)):
        assert torch.equal(bits(x.o), bits(y.o))
        assert torch.equal(bits(x.carry), bits(y.carry))
        assert int(x.status.item()) == int(y.status.item()) == 0
    assert torch.equal(bits(e2.ssm_state), bits(g2.ssm_state))
    assert torch.equal(bits(e2.conv_state), bits(g2.conv_state))

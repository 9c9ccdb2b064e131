"""CUDA-graph capture of whole verify/commit sequences through the C ABI: the
library allocates nothing and never synchronises, so a captured multi-layer
step replays to the same bits as the same calls launched eagerly (the
pages' capture-safe verify with no device-to-host sync)."""
from __future__ import annotations

import pytest
import torch

from gpu_util import bits
from speculative_decode_gateddeltanet_gb300.inputs import STACK, SWEEP, make_layer, workload_layers

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("mode", ["fused", "replay"])
def test_captured_stack_replays_to_eager_bits(mode):
    from speculative_decode_gateddeltanet_gb300 import gdn

    layers = _layers(STACK, layers=6)
    eager = [gdn.DeviceLayer(layer, "cuda") for layer in layers]
    graphed = [gdn.DeviceLayer(layer, "cuda") for layer in layers]
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

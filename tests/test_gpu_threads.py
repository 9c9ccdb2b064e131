"""Calls from several host threads at once, each on its own stream.

The library's host side caches per-shape launch choices (rows staging, item
geometry, resident-CTA counts) and sets each kernel's attributes once per
device.  Four threads run calls of four shapes that make different choices
(4-row and 9-row requests at d_k = 128, d_k = 64, and a batch large enough for
64-row items), many times over, concurrently; every call must leave the
oracle's results.
"""
from __future__ import annotations

import threading

import pytest
import torch

import oracle
from gpu_util import check_against_oracle
from speculative_decode_gateddeltanet_gb300.inputs import LayerSpec, make_layer

pytestmark = pytest.mark.gpu

SPECS = [
    LayerSpec("thr-k3", B=2, k=3, H_qk=2, H_v=4, d_k=128, d_v=128, pool="perm"),
    LayerSpec("thr-k8", B=3, k=8, H_qk=2, H_v=4, d_k=128, d_v=128, pool="double"),
    LayerSpec("thr-dk64", B=3, k=2, H_qk=2, H_v=8, d_k=64, d_v=64, pool="perm"),
    LayerSpec("thr-wide", B=20, k=5, H_qk=16, H_v=32, d_k=128, d_v=128, pool="perm"),
]


def test_concurrent_calls_from_host_threads(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gdn = cuda_lib
    layers = [make_layer(s, 71 + i) for i, s in enumerate(SPECS)]
    refs = [oracle.verify_commit(layer) for layer in layers]
    devs = [gdn.DeviceLayer(layer, "cuda") for layer in layers]
    pristine = [(d.ssm_state.clone(), d.conv_state.clone()) for d in devs]
    torch.cuda.synchronize()
    errors = []
    start = threading.Barrier(len(SPECS))

    def worker(i):
        try:
            d = devs[i]
            stream = torch.cuda.Stream()
            a = d.args()
            start.wait()
            for _ in range(25):
                with torch.cuda.stream(stream):
                    d.ssm_state.copy_(pristine[i][0])
                    d.conv_state.copy_(pristine[i][1])
                gdn.gdn_verify_commit(a, stream.cuda_stream)
            stream.synchronize()
        except Exception as e:  # reported by the main thread
            errors.append((SPECS[i].name, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(SPECS))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for layer, d, ref in zip(layers, devs, refs):
        assert int(d.status.item()) == 0, layer["spec"].name
        check_against_oracle(layer, d, ref, commit=True)

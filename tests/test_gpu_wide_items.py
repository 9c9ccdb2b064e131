"""The rows kernel's two item geometries at d_k = 128.

An item is a slice of one value head's state: 32 rows run by two warps, or
64 rows run by four (the wide geometry).  The choice changes which CTA and
warp runs a state row, not the row's arithmetic: each row's dot products are
reduced over the same 8 lanes in the same order and its recurrence and update
are the same instructions.  So a call forced to either geometry through the
test-only build must write the same o, state and conv windows bit for bit,
and both must match the oracle.  The choice by shape: 64-row items for calls
of more than 4 rows per request whose 64-row items outnumber the two-warp
kernel's resident CTAs, 32 otherwise and for every deferred call.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import oracle
from gpu_util import bits, check_against_oracle, valid_rows
from speculative_decode_gateddeltanet_gb300.inputs import LayerSpec, make_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hooks(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decode_gateddeltanet_gb300 import build as pkg_build

    lib = ctypes.CDLL(str(pkg_build.build_test_hooks()))
    A = ctypes.POINTER(cuda_lib.GdnArgs)
    for name, args in (("gdn_verify", [A, ctypes.c_int, ctypes.c_void_p]),
                       ("gdn_commit", [A, ctypes.c_int, ctypes.c_void_p]),
                       ("gdn_verify_commit", [A, ctypes.c_void_p]),
                       ("gdn_verify_deferred", [A, ctypes.POINTER(cuda_lib.GdnPrevRows), ctypes.c_void_p]),
                       ("gdn_test_force_item_rows", [ctypes.c_int]),
                       ("gdn_test_last_item_rows", [])):
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    yield lib
    lib.gdn_test_force_item_rows(0)


def run(hooks, gdn, layer, mode, rows_per_item):
    """One call (or verify + commit pair) through the test-only build with the
    item geometry forced; returns the DeviceLayer and the rows per item of the
    rows kernel's calls (the snapshot commit is a plain copy and has none)."""
    assert hooks.gdn_test_force_item_rows(rows_per_item) == 0
    snap = mode == "snapshot"
    dev = gdn.DeviceLayer(layer, "cuda", snapshot=snap)
    a = ctypes.byref(dev.args())
    if mode == "fused":
        assert hooks.gdn_verify_commit(a, None) == 0
        rows = hooks.gdn_test_last_item_rows()
    elif mode == "replay":
        assert hooks.gdn_verify(a, gdn.REPLAY, None) == 0
        rows = hooks.gdn_test_last_item_rows()
        assert hooks.gdn_commit(a, gdn.REPLAY, None) == 0
        assert hooks.gdn_test_last_item_rows() == rows
    else:
        assert hooks.gdn_verify(a, gdn.SNAPSHOT, None) == 0
        rows = hooks.gdn_test_last_item_rows()
        assert hooks.gdn_commit(a, gdn.SNAPSHOT, None) == 0
    torch.cuda.synchronize()
    return dev, rows


# d_k = 128 shapes: d_v of one, two and four 64-row items; 1 to 16 rows per
# request (k = 0 .. 15); GQA groups of 1, 2 and 4; ragged row counts
SHAPES = [
    LayerSpec("w-dv64-k5", B=3, k=5, H_qk=2, H_v=8, d_k=128, d_v=64, pool="perm"),
    LayerSpec("w-dv128-k8-ragged", B=6, k=8, H_qk=2, H_v=4, d_k=128, d_v=128, k_choices=(1, 3, 8),
              inactive_frac=0.2, pool="double"),
    LayerSpec("w-dv256-k3-G1", B=2, k=3, H_qk=4, H_v=4, d_k=128, d_v=256, pool="perm"),
    LayerSpec("w-dv128-k15", B=2, k=15, H_qk=2, H_v=8, d_k=128, d_v=128, pool="perm"),
    LayerSpec("w-dv128-k0", B=4, k=0, H_qk=2, H_v=4, d_k=128, d_v=128, pool="double"),
    LayerSpec("w-qwen-heads-k5", B=2, k=5, H_qk=16, H_v=32, d_k=128, d_v=128, pool="perm"),
]


@pytest.mark.parametrize("spec", SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("mode", ["fused", "replay", "snapshot"])
def test_wide_items_match_two_warp_items_bitwise_and_the_oracle(hooks, cuda_lib, spec, mode):
    layer = make_layer(spec, 91)
    wide, r64 = run(hooks, cuda_lib, layer, mode, 64)
    narrow, r32 = run(hooks, cuda_lib, layer, mode, 32)
    assert (r64, r32) == (64, 32)
    valid = torch.from_numpy(valid_rows(layer)).cuda()
    assert torch.equal(bits(wide.o[valid]), bits(narrow.o[valid]))
    assert torch.equal(bits(wide.ssm_state), bits(narrow.ssm_state))
    assert torch.equal(bits(wide.conv_state), bits(narrow.conv_state))
    assert int(wide.status.item()) == int(narrow.status.item())
    check_against_oracle(layer, wide, oracle.verify_commit(layer), commit=True)


def test_wide_geometry_applies_only_where_it_can(hooks, cuda_lib):
    """Forcing 64 rows per item leaves d_v = 32 or 96 (not a multiple of 64)
    and d_k below 128 on their own geometry; the results still match the
    oracle."""
    for spec, want in ((LayerSpec("w-dv96", B=2, k=5, H_qk=2, H_v=4, d_k=128, d_v=96, pool="perm"), 32),
                       (LayerSpec("w-dv32", B=2, k=5, H_qk=2, H_v=4, d_k=128, d_v=32, pool="perm"), 32),
                       (LayerSpec("w-dk64", B=2, k=5, H_qk=2, H_v=4, d_k=64, d_v=64, pool="perm"), 32)):
        layer = make_layer(spec, 92)
        dev, rows = run(hooks, cuda_lib, layer, "fused", 64)
        assert rows == want, spec.name
        check_against_oracle(layer, dev, oracle.verify_commit(layer), commit=True)


def _choice(hooks, gdn, spec, deferred=False):
    assert hooks.gdn_test_force_item_rows(0) == 0
    layer = make_layer(spec, 93)
    dev = gdn.DeviceLayer(layer, "cuda")
    a = dev.args()
    if deferred:
        dev.carry = torch.empty(gdn.carry_bytes(a) // 4, device="cuda")
        a.carry = dev.carry.data_ptr()
        a.accept_len = None
        assert hooks.gdn_verify_deferred(ctypes.byref(a), None, None) == 0
    else:
        assert hooks.gdn_verify_commit(ctypes.byref(a), None) == 0
    torch.cuda.synchronize()
    assert int(dev.status.item()) == 0
    return hooks.gdn_test_last_item_rows()


def test_geometry_chosen_by_shape(hooks, cuda_lib):
    slots = 8 * torch.cuda.get_device_properties(0).multi_processor_count  # two-warp CTAs resident
    heads = dict(H_qk=16, H_v=32, d_k=128, d_v=128, pool="perm")
    B_fill = -(-slots // 64)  # 64-row items (2 per head) that reach the resident-CTA count
    # more than 4 rows per request and enough 64-row items: wide
    assert _choice(hooks, cuda_lib, LayerSpec("c-wide", B=B_fill, k=5, **heads)) == 64
    # one request fewer: two-warp
    assert _choice(hooks, cuda_lib, LayerSpec("c-few", B=B_fill - 1, k=5, **heads)) == 32
    # 4 rows per request (the k = 3 stack): two-warp
    assert _choice(hooks, cuda_lib, LayerSpec("c-k3", B=B_fill, k=3, **heads)) == 32
    # deferred calls keep the two-warp geometry (their carry is laid out by it)
    assert _choice(hooks, cuda_lib, LayerSpec("c-def", B=B_fill, k=5, **heads), deferred=True) == 32

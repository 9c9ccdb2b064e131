"""The debug/test build's check that active requests name distinct slots.

Two active requests on one slot make the call's results undefined (both would
read and write the same state).  The regular build spends nothing on this;
the test-only build (GDN_TEST_HOOKS) compares, in each request's first
prologue block, its slot with every other active request's and sets
GDN_STATUS_DUPLICATE_SLOT.  Inactive requests (n_rows = 0) may share a slot.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

from speculative_decode_gateddeltanet_gb300.inputs import LayerSpec, make_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hooks(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decode_gateddeltanet_gb300 import build as pkg_build

    lib = ctypes.CDLL(str(pkg_build.build_test_hooks()))
    lib.gdn_verify_commit.argtypes = [ctypes.POINTER(cuda_lib.GdnArgs), ctypes.c_void_p]
    lib.gdn_verify_commit.restype = ctypes.c_int
    lib.gdn_verify.argtypes = [ctypes.POINTER(cuda_lib.GdnArgs), ctypes.c_int, ctypes.c_void_p]
    lib.gdn_verify.restype = ctypes.c_int
    return lib


SPEC = LayerSpec("dup-B5-k3", B=5, k=3, H_qk=2, H_v=4, d_k=64, d_v=64, pool="double")


def _status(hooks, gdn, slot_ids, n_rows, verify_only=False):
    layer = make_layer(SPEC, 81)
    dev = gdn.DeviceLayer(layer, "cuda")
    dev.slot_ids.copy_(torch.tensor(slot_ids, dtype=torch.int32))
    dev.n_rows.copy_(torch.tensor(n_rows, dtype=torch.int32))
    a = ctypes.byref(dev.args())
    rc = hooks.gdn_verify(a, gdn.REPLAY, None) if verify_only else hooks.gdn_verify_commit(a, None)
    assert rc == 0
    torch.cuda.synchronize()
    return int(dev.status.item())


def test_duplicate_active_slots_are_reported(hooks, cuda_lib):
    gdn = cuda_lib
    assert _status(hooks, gdn, [0, 1, 2, 3, 4], [4, 4, 4, 4, 4]) == 0
    assert _status(hooks, gdn, [0, 1, 1, 3, 4], [4, 4, 4, 4, 4]) & gdn.STATUS_DUPLICATE_SLOT
    assert _status(hooks, gdn, [7, 1, 2, 3, 7], [4, 2, 4, 4, 1], verify_only=True) & gdn.STATUS_DUPLICATE_SLOT


def test_inactive_requests_may_share_a_slot(hooks, cuda_lib):
    gdn = cuda_lib
    # request 2 is inactive (n_rows = 0), so its slot clashes with nobody
    assert _status(hooks, gdn, [0, 1, 1, 3, 4], [4, 4, 0, 4, 4]) == 0

"""The prologue's slot guess, made to miss on the GPU.

For requests of at most 4 rows the prologue loads the conv window of the slot
it reads before its dependency wait, together with the request data, and
loads the window again when the request's slot (read after the wait) turns
out to differ.  A test-only kernel ahead of the call (GDN_TEST_HOOKS build)
releases the call's grids at once and only rewrites slot_ids some
milliseconds later, so every prologue block reads the old slots as its guess
and must take the reload.  The results must still be those of the new slots.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import oracle
from gpu_util import check_against_oracle
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
    lib.gdn_commit.argtypes = [ctypes.POINTER(cuda_lib.GdnArgs), ctypes.c_int, ctypes.c_void_p]
    lib.gdn_commit.restype = ctypes.c_int
    lib.gdn_test_late_write.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_ulonglong,
                                        ctypes.c_void_p]
    lib.gdn_test_late_write.restype = ctypes.c_int
    lib.gdn_test_guess_misses.argtypes = [ctypes.c_int]
    lib.gdn_test_guess_misses.restype = ctypes.c_longlong
    return lib


SPEC = LayerSpec("guess-B4-k3", B=4, k=3, H_qk=2, H_v=4, d_k=128, d_v=128, pool="double")


@pytest.mark.parametrize("mode", ["fused", "replay"])
def test_missed_slot_guess_reloads_the_window(hooks, cuda_lib, mode):
    gdn = cuda_lib
    layer = make_layer(SPEC, 61)
    # a first call of the same shape, so the one under test launches right
    # behind the writer (no first-call host setup in between)
    warm = gdn.DeviceLayer(layer, "cuda")
    assert hooks.gdn_verify_commit(ctypes.byref(warm.args()), None) == 0
    assert hooks.gdn_verify(ctypes.byref(warm.args()), gdn.REPLAY, None) == 0
    assert hooks.gdn_commit(ctypes.byref(warm.args()), gdn.REPLAY, None) == 0
    dev = gdn.DeviceLayer(layer, "cuda")
    right = dev.slot_ids.clone()
    wrong = (right + SPEC.B) % SPEC.pool_slots  # other valid slots of the pool
    assert not torch.equal(wrong, right)
    dev.slot_ids.copy_(wrong)
    torch.cuda.synchronize()
    assert hooks.gdn_test_guess_misses(1) >= 0  # cleared
    stream = torch.cuda.current_stream().cuda_stream
    a = ctypes.byref(dev.args())
    # the writer releases the call at once and rewrites slot_ids 10 ms later (the call is
    # launched within microseconds, so its prologue reads the old slots whatever the host load)
    assert hooks.gdn_test_late_write(dev.slot_ids.data_ptr(), right.data_ptr(), SPEC.B, 10_000_000, stream) == 0
    if mode == "fused":
        assert hooks.gdn_verify_commit(a, stream) == 0
    else:
        assert hooks.gdn_verify(a, gdn.REPLAY, stream) == 0
        assert hooks.gdn_commit(a, gdn.REPLAY, stream) == 0
    torch.cuda.synchronize()
    misses = hooks.gdn_test_guess_misses(1)
    # every prologue block (H_qk q/k blocks + 1 v block per request) of the
    # first call read the old slot before the writer had run
    assert misses >= SPEC.B * (SPEC.H_qk + 1), misses
    assert torch.equal(dev.slot_ids, right)
    assert int(dev.status.item()) == 0
    check_against_oracle(layer, dev, oracle.verify_commit(layer), commit=True)
